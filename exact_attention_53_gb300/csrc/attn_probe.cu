// Throughput probe for the secondary ceiling of the softmax: ex2.approx (the
// MUFU pipe).  Each thread runs 8 independent chains so the pipe, not the
// dependency latency, limits the rate.  Declared in include/attn_probe.h.
#include <cuda_runtime.h>

#pragma GCC visibility push(default)    // the C ABI is the library's only export
#include "attn_probe.h"
#pragma GCC visibility pop
#include "sm100.cuh"

namespace {

__global__ void __launch_bounds__(256) ex2_rate_kernel(float* out, int iters, float seed) {
    using attn::sm100::ex2_approx;
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = seed * static_cast<float>(threadIdx.x + i) * 1e-6f - 0.5f;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = ex2_approx(x[i]) - 1.5f;   // stays in (-1.5, 0.5)
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += x[i];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

extern "C" int attn_probe_ex2(float* out, int blocks, int iters, struct CUstream_st* stream) {
    if (!out || blocks < 1 || iters < 1) return 1;
    ex2_rate_kernel<<<blocks, 256, 0, stream>>>(out, iters, 1.0f);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
