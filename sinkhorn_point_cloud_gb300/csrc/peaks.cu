// peaks.cu -- throughput probes for the roofline denominators of the fp32
// paths: MUFU ex2, scalar FFMA and packed f32x2 FMA, in operations per SM per
// clock.  Built as a separate small library (libsotpeaks.so) used only by the
// benchmark; not part of the solver ABI.
//
// One CTA of 1024 threads per SM (grid = SM count, so the block scheduler
// places exactly one per SM); each thread runs 8 independent dependency chains
// for `iters` rounds and every CTA times itself with clock64 (SM cycles), so
// per-SM throughput = the CTA's operations / its cycles.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace {

template <int KIND>
__global__ void __launch_bounds__(1024) probe_kernel(int iters, float seed, float* sink, long long* cycles) {
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = seed + 0.001f * (threadIdx.x + k);
    float2 w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = make_float2(v[k], v[k] + 0.5f);
    const float2 a2 = make_float2(0.999f, 0.998f), b2 = make_float2(1e-3f, 2e-3f);
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (KIND == 0) v[k] = ex2f(v[k]);
            if (KIND == 1) v[k] = fmaf(v[k], 0.999f, 1e-3f);
            if (KIND == 2) w[k] = ffma2(w[k], a2, b2);
        }
    }
    __syncthreads();
    const long long t1 = clock64();
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) acc += v[k] + w[k].x + w[k].y;
    if (acc == 1234.5f) sink[threadIdx.x] = acc;  // keeps the chains alive
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

}  // namespace

extern "C" {

// kind: 0 = ex2 (MUFU), 1 = FFMA, 2 = packed f32x2 FMA (counts 2 lanes per instruction).
// Returns lane-operations per SM per clock in *rate_host; negative status on error.
int sotpeaks_measure(int kind, double* rate_host) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -5;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int threads = 1024, iters = 2048;
    const int blocks = sms;
    float* sink = nullptr;
    long long* cyc = nullptr;
    if (cudaMalloc(&sink, threads * sizeof(float)) != cudaSuccess) return -7;
    if (cudaMalloc(&cyc, blocks * sizeof(long long)) != cudaSuccess) { cudaFree(sink); return -7; }
    for (int rep = 0; rep < 2; ++rep) {  // first launch warms up
        if (kind == 0) probe_kernel<0><<<blocks, threads>>>(iters, -0.5f, sink, cyc);
        else if (kind == 1) probe_kernel<1><<<blocks, threads>>>(iters, 0.5f, sink, cyc);
        else probe_kernel<2><<<blocks, threads>>>(iters, 0.5f, sink, cyc);
    }
    cudaError_t e = cudaDeviceSynchronize();
    long long* h = new long long[blocks];
    if (e == cudaSuccess) e = cudaMemcpy(h, cyc, blocks * sizeof(long long), cudaMemcpyDeviceToHost);
    double mean = 0.0;
    for (int i = 0; i < blocks; ++i) mean += (double)h[i];
    mean /= blocks;
    delete[] h;
    cudaFree(sink);
    cudaFree(cyc);
    if (e != cudaSuccess) return -5;
    const double ops_per_block = (double)threads * iters * 8 * (kind == 2 ? 2 : 1);
    *rate_host = ops_per_block / mean;
    return 0;
}

}  // extern "C"
