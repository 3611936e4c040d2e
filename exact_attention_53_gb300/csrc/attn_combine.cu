// Merge of split-KV partial results.
//
// The forward kernel's split mode cuts the keys of each (head, query block)
// into n_split ranges and writes, per range s and query row i, the normalised
// partial output O_s,i = Σ_{j∈s} p_ij v_j / Σ_{j∈s} p_ij (fp32) and the range's
// log-sum-exp LSE_s,i = ln Σ_{j∈s} exp(S_ij).  The LSE output of the forward
// (oxicuda-dnn 0.1.8, src/attn/flash_attn/hopper.rs, FlashAttention3Plan::
// generate_forward, the final "write O and LSE" step) is exactly what makes the
// ranges mergeable:
//
//     LSE_i = ln Σ_s exp(LSE_s,i)
//     O_i   = Σ_s exp(LSE_s,i − LSE_i) · O_s,i
//
// One warp per query row; lane l owns d/32 consecutive columns, so every load
// and store of a warp covers one contiguous row segment.  O is written in the
// caller's layout (batch, head and row strides), LSE densely.  The pass is bound by
// reading the partials once (n_split · (d + 1) · 4 bytes per row).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_launch.h"

namespace attn {
namespace {

template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* __restrict__ o_part,
                                                           const float* __restrict__ lse_part,
                                                           void* __restrict__ o,
                                                           float* __restrict__ lse, int n_split,
                                                           long long rows, int H, int S_q,
                                                           RowLayout o_lay) {
    constexpr int PER_LANE = D / 32;          // 2, 4 or 8 columns
    // Launched as a programmatic dependent of the range kernel: wait until
    // that grid has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;

    // Weights, lane-parallel over ranges (32 per pass): the largest partial LSE
    // first, so every weight exp(LSE_s − m) is at most 1.
    float m = -INFINITY;
    for (int s = lane; s < n_split; s += 32) m = fmaxf(m, lse_part[s * rows + row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));

    float acc[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) acc[i] = 0.f;
    float wsum = 0.f;
    const size_t col = static_cast<size_t>(lane) * PER_LANE;
    for (int s0 = 0; s0 < n_split; s0 += 32) {
        const int s_lane = s0 + lane;
        const float w_lane = s_lane < n_split ? expf(lse_part[s_lane * rows + row] - m) : 0.f;
        wsum += w_lane;
        const int cnt = min(32, n_split - s0);
        // The ranges' partial rows are independent loads: unrolled so several are
        // in flight at once.
#pragma unroll 4
        for (int j = 0; j < cnt; ++j) {
            const float w = __shfl_sync(0xffffffffu, w_lane, j);
            const float* src = o_part + (static_cast<size_t>(s0 + j) * rows + row) * D + col;
            if constexpr (PER_LANE == 2) {
                const float2 x = *reinterpret_cast<const float2*>(src);
                acc[0] = fmaf(w, x.x, acc[0]);
                acc[1] = fmaf(w, x.y, acc[1]);
            } else {
#pragma unroll
                for (int i = 0; i < PER_LANE; i += 4) {
                    const float4 x = *reinterpret_cast<const float4*>(src + i);
                    acc[i] = fmaf(w, x.x, acc[i]);
                    acc[i + 1] = fmaf(w, x.y, acc[i + 1]);
                    acc[i + 2] = fmaf(w, x.z, acc[i + 2]);
                    acc[i + 3] = fmaf(w, x.w, acc[i + 3]);
                }
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
    // wsum >= 1 (the largest range contributes exp(0)).
    const float inv = 1.f / wsum;
    uint32_t packed[PER_LANE / 2];
#pragma unroll
    for (int i = 0; i < PER_LANE / 2; ++i) {
        const float a = acc[2 * i] * inv, b = acc[2 * i + 1] * inv;
        if (BF16) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
            packed[i] = *reinterpret_cast<const uint32_t*>(&h);
        } else {
            const __half2 h = __floats2half2_rn(a, b);
            packed[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
    }
    const long long bh = row / S_q, q = row - bh * S_q;
    const long long b = bh / H, h = bh - b * H;
    uint16_t* dst = static_cast<uint16_t*>(o) +
                    static_cast<size_t>(b * o_lay.batch + h * o_lay.head + q * o_lay.row) + col;
    if constexpr (PER_LANE == 2) {
        *reinterpret_cast<uint32_t*>(dst) = packed[0];
    } else if constexpr (PER_LANE == 4) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
    } else {
        *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
    if (lane == 0) lse[row] = m + logf(wsum);
}

template <int D>
cudaError_t launch_d(const float* o_part, const float* lse_part, void* o, float* lse, int n_split,
                     long long rows, bool bf16, int H, int S_q, const RowLayout& o_lay,
                     cudaStream_t stream) {
    const long long blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // Programmatic stream serialisation: the launch is set up while the range
    // kernel is still running; the kernel's griddepcontrol.wait orders the reads.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (bf16)
        return cudaLaunchKernelEx(&cfg, attn_combine_kernel<D, true>, o_part, lse_part, o, lse,
                                  n_split, rows, H, S_q, o_lay);
    return cudaLaunchKernelEx(&cfg, attn_combine_kernel<D, false>, o_part, lse_part, o, lse,
                              n_split, rows, H, S_q, o_lay);
}

}  // namespace

cudaError_t launch_attn_combine(const float* o_part, const float* lse_part, void* o, float* lse,
                                int n_split, long long rows, int d, bool bf16, int H, int S_q,
                                const RowLayout& o_lay, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    switch (d) {
        case 64:
            return launch_d<64>(o_part, lse_part, o, lse, n_split, rows, bf16, H, S_q, o_lay, stream);
        case 128:
            return launch_d<128>(o_part, lse_part, o, lse, n_split, rows, bf16, H, S_q, o_lay, stream);
        case 256:
            return launch_d<256>(o_part, lse_part, o, lse, n_split, rows, bf16, H, S_q, o_lay, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
