// Host-side launch contract between the C-ABI layer (attn_api.cu) and the
// per-(head_dim, dtype, causal) kernel instantiations (attn_inst.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace attn {

struct FwdArgs {
    CUtensorMap tm_q;       // [B·H, S_q, d] rows of Q, box 64 × 128
    CUtensorMap tm_k;       // [B·H, S_k, d] rows of K, box 64 × 128
    CUtensorMap tm_v;       // [B·H, S_k, d] rows of V, box 64 × 128
    void* o;                // [B, H, S_q, d], same dtype as Q
    float* lse;             // [B, H, S_q] fp32, natural log
    int32_t S_q;
    int32_t S_k;
    int32_t BH;             // B·H
    float scale_log2;       // scale · log2(e), >= 0
    unsigned int* status;   // device status word (bit set on a wait that ran out)
};

// Rows per query tile and keys per key/value tile, fixed for every head_dim.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;

// Query tiles per CTA: two (ping-pong between two softmax warpgroups) for
// d <= 128; one for d = 256, where two 256-column O accumulators would fill
// tensor memory.
__host__ __device__ constexpr int q_tiles_per_cta(int d) { return d == 256 ? 1 : 2; }

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_attn_fwd(const FwdArgs& args, cudaStream_t stream);

}  // namespace attn
