// Host-side launch contract between the C-ABI layer (attn_api.cu) and the
// per-(head_dim, dtype, causal) kernel instantiations (attn_inst.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

namespace attn {

namespace sm100 {
struct DeviceWords;     // per-GPU status and abort words (sm100.cuh)
}
using sm100::DeviceWords;

// Every kernel launch with bounded waits gets a launch number, unique per
// device, and a time budget after which each of its CTAs gives up (sm100.cuh,
// Guard).

struct FwdArgs {
    // 4-D maps (d, S, heads, B) with the tensors' own row, head and batch
    // strides; box 64 columns × 128 rows × 1 × 1.
    CUtensorMap tm_q;       // Q: (d, S_q, H, B)
    CUtensorMap tm_k;       // K: (d, S_k, H_kv, B)
    CUtensorMap tm_v;       // V: (d, S_k, H_kv, B)
    CUtensorMap tm_o;       // O: (d, S_q, H, B), stores
    void* o;                // [B, H, S_q, d], same dtype as Q
    float* lse;             // [B, H, S_q] fp32, natural log
    int32_t S_q;
    int32_t S_k;
    int32_t BH;             // B·H
    int32_t H;              // query heads
    int32_t kv_group;       // query heads per key/value head (H / H_kv)
    int32_t causal_off;     // causal: key j is visible to query i iff j <= i + causal_off
    float scale_log2;       // scale · log2(e), either sign
    int32_t num_sms;        // SMs of the device (split-KV range planning)
    int32_t device;         // CUDA device ordinal the launch runs on (< 64)
    // split-KV only (launch_attn_fwd<..., SPLIT = true>)
    int32_t n_split;        // key ranges per (head, query block)
    int32_t kv_per_split;   // key tiles per range
    float* o_part;          // [n_split, B·H, S_q, d] fp32: O/l of each range
    float* lse_part;        // [n_split, B·H, S_q] fp32: LSE of each range
    int32_t pack;           // query heads per unit's query tile (1, or H / H_kv when packed)
    DeviceWords* words;     // device status word (bit set on a wait that ran out) and abort word
    unsigned long long launch;      // launch number of the forward kernel
    unsigned long long budget_ns;   // deadline of each CTA, from its start
};

// Run `setup` (a kernel's shared-memory opt-in and resource check) on the
// first launch of that kernel on `device` only; `done` holds one bit per
// device.  Returns setup's error, and keeps trying until it succeeds.
template <typename F>
cudaError_t configure_once(std::atomic<uint64_t>& done, int device, F&& setup) {
    const uint64_t bit = uint64_t(1) << device;
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    const cudaError_t e = setup();
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Element strides of a [B, heads, S, d] tensor (d contiguous).
struct RowLayout {
    long long batch, head, row;
};

// Rows per query tile and keys per key/value tile, fixed for every head_dim.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;

// Query tiles per CTA: two (ping-pong between two softmax warpgroups) for
// d <= 128; one for d = 256, where two 256-column O accumulators would fill
// tensor memory.
__host__ __device__ constexpr int q_tiles_per_cta(int d) { return d == 256 ? 1 : 2; }

// Static plan of one kernel instantiation: tiles, warp roles, shared and
// tensor memory.  Shared by the kernel and the host (attn_fwd_plan).
// TILES_: query tiles per work unit (q_tiles_per_cta(D) for the one-pass
// forward; 1 for split-KV, whose units are short and must not wait on a
// second query tile that short queries leave empty).
template <int D, int TILES_ = q_tiles_per_cta(D)>
struct FwdTile {
    static constexpr int BM = kBlockM;
    static constexpr int BN = kBlockN;
    static constexpr int TILES = TILES_;
    static constexpr int CHUNKS = D / 64;                 // 128-byte swizzle atoms along d
    static constexpr int ATOM_ROWS_BYTES = 128;           // one row of one atom
    static constexpr int Q_CHUNK_BYTES = BM * ATOM_ROWS_BYTES;
    static constexpr int KV_CHUNK_BYTES = BN * ATOM_ROWS_BYTES;
    static constexpr int Q_TILE_BYTES = BM * D * 2;
    static constexpr int KV_TILE_BYTES = BN * D * 2;
    static constexpr int NS = D == 64 ? 8 : (D == 128 ? 4 : 2);
    // O leaves through a staging buffer of up to two 64-column chunks (TMA
    // store boxes), in STAGE_ROUNDS rounds per query tile.
    static constexpr int STAGE_CHUNKS = CHUNKS < 2 ? CHUNKS : 2;
    static constexpr int STAGE_ROUNDS = CHUNKS / STAGE_CHUNKS;
    static constexpr int STAGE_BYTES = STAGE_CHUNKS * Q_CHUNK_BYTES;
    static constexpr int TILE_BYTES = TILES * Q_TILE_BYTES + NS * KV_TILE_BYTES + STAGE_BYTES;
    // Work-queue answers (cluster launch control) in flight: unit ids this CTA
    // has claimed ahead of the ones it is working on.
    static constexpr int CLC_SLOTS = 4;
    static constexpr int NUM_BARS = 2 + 2 * NS + 2 + 2 + 2 + 1 + 2 + 1 + 2 * CLC_SLOTS;
    static constexpr int SMEM_BYTES = 1024 + TILE_BYTES + CLC_SLOTS * 16 + NUM_BARS * 8 + 16;
    static constexpr int SOFTMAX_WARPS = 4 * TILES;
    static constexpr int PRODUCER_WARP = SOFTMAX_WARPS;       // first warp of the aux warpgroup
    static constexpr int MMA_WARP = SOFTMAX_WARPS + 1;
    static constexpr int STORE_WARP = SOFTMAX_WARPS + 2;      // O stores (not in split-KV)
    static constexpr int THREADS = 32 * (SOFTMAX_WARPS + 4);  // + one aux warpgroup
    // Register split (TILES == 2): 12 warps put 3 on each SM sub-partition, so
    // the launch gets 168 registers a thread (16384 / 3 warps / 32, rounded to
    // 8).  The aux warpgroup gives most of its share to the softmax ones:
    // 2·216 + 72 = 3·168 (72 is the least the aux roles need without spills).
    static constexpr int LAUNCH_REGS = 168;
    static constexpr int SOFTMAX_REGS = 216;
    static constexpr int AUX_REGS = 72;
    static_assert(TILES == 1 || 2 * SOFTMAX_REGS + AUX_REGS <= 3 * LAUNCH_REGS, "register split");
    // tensor memory columns: S buffers 0 and 1, then one O accumulator per tile
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_STRIDE = 128;             // S buffer b at column b * 128
    static constexpr uint32_t P_OFF = 64;                 // P (16-bit, packed) over S cols 64..127
    static constexpr uint32_t O_COL = 256;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(O_COL + TILES * D <= TMEM_COLS, "tensor memory budget");
};

// The tile plan a kernel instantiation runs with.
template <int D, bool SPLIT>
using KernelTile = FwdTile<D, SPLIT ? 1 : q_tiles_per_cta(D)>;

template <int D, bool BF16, bool CAUSAL, bool SPLIT>
cudaError_t launch_attn_fwd(const FwdArgs& args, cudaStream_t stream);

// Merge n_split partial results: LSE = ln Σ_s exp(LSE_s), O = Σ_s exp(LSE_s − LSE)·O_s,
// written as the output dtype into o (element strides o_lay over [B, H, S_q, d])
// and as fp32 into the dense lse.  rows = B·H·S_q.
cudaError_t launch_attn_combine(const float* o_part, const float* lse_part, void* o, float* lse,
                                int n_split, long long rows, int d, bool bf16, int H, int S_q,
                                const RowLayout& o_lay, cudaStream_t stream);

// Backward launch contract (attn_bwd.cuh).  The dK/dV kernel keeps 128-row K
// and V tiles and streams 64-row Q and dO steps (d = 256: two passes, dV and
// dK, attn_bwd_wide.cuh); the dQ kernel keeps 128-row Q and dO tiles and
// streams 128-row K and V steps (64-row at d = 256).
struct BwdArgs {
    // 4-D maps (d, S, heads, B) in each tensor's own layout
    CUtensorMap tm_k_fixed, tm_v_fixed;   // K, V: (d, S_k, H_kv, B), box 64 × 128
    CUtensorMap tm_q_step, tm_do_step;    // Q, dO: (d, S_q, H, B), box 64 × 64
    CUtensorMap tm_q_fixed, tm_do_fixed;  // Q, dO: (d, S_q, H, B), box 64 × 128
    CUtensorMap tm_k_step, tm_v_step;     // K, V: box 64 × 64 (d = 256 only: the dQ kernel's steps)
    CUtensorMap tm_dk_out, tm_dv_out;     // dK, dV: (d, S_k, H_kv, B), box 64 × 32, stores (d <= 128)
    const void* o;                        // forward output [B, H, S_q, d]
    const void* dout;                     // dO [B, H, S_q, d]
    const float* lse;                     // forward LSE [B, H, S_q], natural log
    float* lse2;                          // workspace [B·H, S_pad]: LSE·log2(e)
    float* delta;                         // workspace [B·H, S_pad]: rowsum(dO ∘ O)
    void* dq;
    void* dk;
    void* dv;
    RowLayout o_lay, do_lay, dq_lay, dk_lay, dv_lay;
    int32_t S_q, S_k, BH, S_pad;          // S_pad = S_q rounded up to 128
    int32_t H;                            // query heads
    int32_t kv_group;                     // query heads per key/value head
    int32_t causal_off;                   // key j visible to query i iff j <= i + causal_off
    float scale, scale_log2;
    int32_t num_sms;
    int32_t device;                       // CUDA device ordinal (< 64)
    DeviceWords* words;
    // Launch numbers of the key-side kernel (the dV pass at d = 256), of the
    // dK pass (d = 256) and of the dQ kernel, and the CTAs' time budget.
    unsigned long long launch_dkdv, launch_key2, launch_dq, budget_ns;
    // When set, the dQ kernel runs on aux_stream, concurrently with the dK/dV
    // kernel on the caller's stream (they read the same inputs and write
    // disjoint outputs): ev_fork orders it after the prep kernel, ev_join
    // brings the caller's stream back after it.  The caller holds a lock that
    // serialises use of these three.
    cudaStream_t aux_stream;
    cudaEvent_t ev_fork, ev_join;
};

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_attn_bwd(const BwdArgs& args, cudaStream_t stream);

#ifdef ATTN_DEBUG_FAULTS
// Debug builds only (never the release library): the forward's producer, and
// the backward's dK/dV producer, load nothing for this work unit and stop, so
// the unit's consumers wait until their limit runs out.  -1: no unit skipped.
__device__ int g_attn_debug_skip_unit = -1;
#endif

// Device address of the built-in split-KV scratch (ATTN_NOALLOC_SCRATCH_BYTES
// bytes, 256-byte aligned) on the current device.
cudaError_t noalloc_scratch_address(void** ptr);

}  // namespace attn
