// Attention backward on sm_103a: tcgen05 MMAs with TMEM accumulators, TMA
// loads into shared-memory rings, mbarrier handoffs, persistent CTAs.
//
// The steps are those of the page's backward (oxicuda-dnn 0.1.8,
// src/attn/flash_attn/hopper.rs, doc comment of generate_backward): recompute
// P from the forward's log-sum-exp, then dV = Pᵀ·dO, dP = dO·Vᵀ,
// dS = P ∘ (dP − D) with D_i = rowsum(dO ∘ O), dQ = dS·K, dK = dSᵀ·Q (dQ and
// dK times the softmax scale).  Three kernels:
//
//   attn_bwd_prep_kernel   D_i = Σ_c dO_ic·O_ic and LSE_i·log2(e), one row
//                          per warp, into a workspace padded to whole tiles
//                          (padding rows: D = 0, LSE = +inf, so P = 0 there);
//   attn_bwd_dkdv_kernel   one unit = (head, 128 keys): loops over 64-row
//                          query steps, Sᵀ = K·Qᵀ and dPᵀ = V·dOᵀ into TMEM,
//                          Pᵀ and dSᵀ formed by four softmax warps (one key
//                          row per thread), dV += Pᵀ·dO and dK += dSᵀ·Q with
//                          Pᵀ / dSᵀ read from TMEM;
//   attn_bwd_dq_kernel     one unit = (head, 128 queries): loops over 128-key
//                          steps, S = Q·Kᵀ and dP = dO·Vᵀ, dS by the softmax
//                          warps (one query row per thread), dQ += dS·K.
//
// In both main kernels four epilogue warps read the finished accumulators of
// a unit out of TMEM, release them (the next unit's first accumulating MMA
// waits for that) and store them while the next unit's steps run; the dK/dV
// kernel stages them in shared memory for TMA tensor stores.
//
// dQ gets its own pass (it recomputes S and dP) instead of the page's f32
// atomics, so every result is deterministic: no two CTAs ever add into the
// same output.  Tensor memory holds two S buffers, two dP buffers and the
// accumulators (dV and dK: 2·d columns; dQ: d), so this file's dK/dV kernel
// takes head_dim 64 or 128 (256: attn_bwd_wide.cuh).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "attn_launch.h"
#include "sm100.cuh"

namespace attn {

// Status bits of the backward kernels (shared word with the forward).
constexpr unsigned int kStatusBwdProducer = 1u << 5;
constexpr unsigned int kStatusBwdMma = 1u << 6;
constexpr unsigned int kStatusBwdSoftmax = 1u << 7;
constexpr unsigned int kStatusBwdDrain = 1u << 8;
constexpr unsigned int kStatusBwdEpilogue = 1u << 10;

template <int D>
struct BwdTile {
    static_assert(D == 64 || D == 128, "the backward is built for head_dim 64 and 128");
    static constexpr int BU = 128;                    // rows of the unit's fixed operands
    static constexpr int BS = 64;                     // rows per step
    static constexpr int CHUNKS = D / 64;             // 128-byte swizzle atoms along d
    static constexpr int BIG_CHUNK = BU * 128;        // one atom column of a 128-row tile
    static constexpr int SMALL_CHUNK = BS * 128;      // of a 64-row tile
    static constexpr int BIG_TILE = BU * D * 2;
    static constexpr int SMALL_TILE = BS * D * 2;
    static constexpr int NS = D == 64 ? 8 : 4;        // ring slots, two 64-row tiles each
    static constexpr int SLOT_BYTES = 2 * SMALL_TILE;
    static constexpr int STAT_FLOATS = 2 * BS;        // per slot: LSE·log2e and D of 64 rows
    static constexpr int CLC_SLOTS = 4;               // work-queue answers in flight
    static constexpr int NUM_BARS = 2 + 2 * NS + 2 + 2 + 1 + 2 + 1 + 2 * CLC_SLOTS;
    // Output staging: each epilogue warp stages 64 columns of its 32 key rows
    // in the 128-byte swizzled layout (4 KB) and stores them with one TMA
    // tensor store.
    static constexpr int STG_WARP = 32 * 128;
    static constexpr int STG_OFF = 2 * BIG_TILE + NS * SLOT_BYTES + NS * STAT_FLOATS * 4;
    static constexpr int TILE_BYTES = STG_OFF + 4 * STG_WARP;
    static constexpr int SMEM_BYTES = 1024 + TILE_BYTES + CLC_SLOTS * 16 + NUM_BARS * 8 + 16;
    static constexpr int THREADS = 384;     // softmax warps 0-3, epilogue 4-7, producer, MMA, 2 idle
    static constexpr int EPI_WARP = 4;      // first epilogue warp (warp % 4 = its lane quarter)
    static constexpr int PRODUCER_WARP = 8;
    static constexpr int MMA_WARP = 9;
    // Register split: the launch grants LAUNCH_REGS a thread (65536 over 12
    // warps, rounded down to a multiple of 8); the softmax and epilogue
    // warpgroups grow to their budgets, the aux warpgroup (producer, MMA and
    // two idle warps) shrinks to its own.  The sum is 3·LAUNCH_REGS.
    static constexpr int LAUNCH_REGS = 168;
    static constexpr int SOFTMAX_REGS = 200;
    static constexpr int EPI_REGS = 152;
    static constexpr int AUX_REGS = 152;
    static_assert(SOFTMAX_REGS + EPI_REGS + AUX_REGS <= 3 * LAUNCH_REGS, "register split");
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 0;              // S buffer b at column 64·b (fp32)
    static constexpr uint32_t DP_COL = 128;           // dP buffer b at 128 + 64·b
    static constexpr uint32_t PK_OFF = 32;            // packed 16-bit results over cols 32..63
    static constexpr uint32_t ACC_COL = 256;          // accumulators: 256 (+ D)
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(ACC_COL + 2 * D <= TMEM_COLS, "tensor memory budget");
};

// Unit L -> (head, tile).  Full attention: a head's tiles are adjacent, so the
// units in flight share that head's step operands in L2.  Causal: heads in
// groups of head_group, heaviest tiles of the group first (HEAVY_LOW: tile 0
// is the heaviest, as for key tiles; otherwise the last tile is).
template <bool CAUSAL, bool HEAVY_LOW>
__device__ __forceinline__ void bwd_unit_coords(int L, int BH, int n_tiles, int head_group,
                                                int& bh, int& tile) {
    if (CAUSAL) {
        const int per_group = head_group * n_tiles;
        const int g = L / per_group;
        const int r = L - g * per_group;
        const int g0 = g * head_group;
        const int gsz = min(head_group, BH - g0);
        const int ti = r / gsz;
        bh = g0 + (r - ti * gsz);
        tile = HEAVY_LOW ? ti : n_tiles - 1 - ti;
    } else {
        bh = L / n_tiles;
        tile = L - bh * n_tiles;
    }
}

// Softmax-side work of one step for one row: P = 2^(s·scale·log2e − L) (0
// where masked), dS = P·(dP − Dv); packs dS (and P when WANT_P) as 16-bit
// pairs.  Per column c: lse2[c], dd[c] (COLUMN_STATS: one value per column,
// read from shared memory; else the row's own, broadcast).  keep(c) tells
// whether column c is visible.  Two columns at a time on the packed fp32 pipe.
template <bool MASKED, bool BF16, bool WANT_P, bool COLUMN_STATS, typename Keep>
__device__ __forceinline__ void grad_pack64(const uint32_t (&s)[64], const uint32_t (&dp)[64],
                                            const float* lse2, const float* dd, float row_lse2,
                                            float row_dd, float scale_log2, Keep keep,
                                            uint32_t (&pk_p)[32], uint32_t (&pk_ds)[32]) {
    using namespace sm100;
    const float2 sl2 = make_float2(scale_log2, scale_log2);
    const float2 row_nl = make_float2(-row_lse2, -row_lse2);
    const float2 row_nd = make_float2(-row_dd, -row_dd);
#pragma unroll
    for (int c = 0; c < 64; c += 4) {
        float2 nl[2], nd[2];
        if (COLUMN_STATS) {
            const float4 l4 = *reinterpret_cast<const float4*>(lse2 + c);
            const float4 d4 = *reinterpret_cast<const float4*>(dd + c);
            nl[0] = make_float2(-l4.x, -l4.y);
            nl[1] = make_float2(-l4.z, -l4.w);
            nd[0] = make_float2(-d4.x, -d4.y);
            nd[1] = make_float2(-d4.z, -d4.w);
        } else {
            nl[0] = nl[1] = row_nl;
            nd[0] = nd[1] = row_nd;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int cc = c + 2 * i;
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[cc]), __uint_as_float(s[cc + 1])),
                                        sl2, nl[i]);
            float p0 = ex2_approx(x.x);
            float p1 = ex2_approx(x.y);
            if (MASKED) {
                p0 = keep(cc) ? p0 : 0.f;
                p1 = keep(cc + 1) ? p1 : 0.f;
            }
            const float2 t = __fadd2_rn(make_float2(__uint_as_float(dp[cc]), __uint_as_float(dp[cc + 1])),
                                        nd[i]);
            const float2 g = __fmul2_rn(make_float2(p0, p1), t);
            if (WANT_P) pk_p[cc / 2] = BF16 ? pack_bf16(p0, p1) : pack_f16(p0, p1);
            pk_ds[cc / 2] = BF16 ? pack_bf16(g.x, g.y) : pack_f16(g.x, g.y);
        }
    }
}

// Store one row of an fp32 TMEM accumulator (D columns at `taddr`) times
// `mul` as 16-bit values to `dst` (D contiguous elements).
template <int D, bool BF16>
__device__ __forceinline__ void store_row_from_tmem(uint32_t taddr, float mul, void* dst,
                                                    bool store) {
    using namespace sm100;
    uint4* out = reinterpret_cast<uint4*>(dst);
#pragma unroll 1
    for (int cc = 0; cc < D; cc += 32) {
        uint32_t r[32];
        tmem_ld32(taddr + cc, r);
        if (store) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float a = __uint_as_float(r[8 * i + 2 * k]) * mul;
                    const float b = __uint_as_float(r[8 * i + 2 * k + 1]) * mul;
                    w[k] = BF16 ? pack_bf16(a, b) : pack_f16(a, b);
                }
                out[cc / 8 + i] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
}

// One row of an fp32 TMEM accumulator (D columns at `taddr`) times `mul`,
// packed as 16-bit pairs into out[D/2]: CH-column loads (64 or 32; fewer
// registers in flight), one wait each.
template <int D, bool BF16, int CH = 64>
__device__ __forceinline__ void read_acc_packed(uint32_t taddr, float mul, uint32_t (&out)[D / 2]) {
    using namespace sm100;
    static_assert(CH == 64 || CH == 32, "64- or 32-column loads");
#pragma unroll
    for (int c = 0; c < D; c += CH) {
        uint32_t r[CH];
        if constexpr (CH == 64) tmem_ld64(taddr + c, r);
        else tmem_ld32(taddr + c, r);
#pragma unroll
        for (int i = 0; i < CH / 2; ++i) {
            const float a = __uint_as_float(r[2 * i]) * mul;
            const float b = __uint_as_float(r[2 * i + 1]) * mul;
            out[c / 2 + i] = BF16 ? pack_bf16(a, b) : pack_f16(a, b);
        }
    }
}

// One warp stores 64 columns of its 32 rows: each lane's 32 packed words
// (w[0..31], its row) go to the warp's 4 KB staging tile in the 128-byte
// swizzled layout (1024-byte aligned), then lane 0 stores the tile with one
// TMA tensor store at (col, row0, head, batch); rows past the tensor's extent
// are not written.  Lane 0 first waits until its previous store has finished
// reading the tile.
__device__ __forceinline__ void store_tile_64(const uint32_t* w, uint8_t* tile, int lane,
                                              const CUtensorMap* map, int col, int row0,
                                              int head, int batch) {
    using namespace sm100;
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
    uint8_t* row = tile + lane * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(row + ((c ^ (lane & 7)) << 4)) =
            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_4d(map, tile, col, row0, head, batch);
        bulk_commit_group();
    }
}

// Store D packed 16-bit values (D/2 words) to `dst` as 16-byte pieces.
template <int D>
__device__ __forceinline__ void store_packed_row(const uint32_t (&w)[D / 2], void* dst) {
    uint4* out = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < D / 8; ++i) out[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
}

// ============================================================== prep
// delta[bh, i] = Σ_c dO[b,h,i,c]·O[b,h,i,c]; lse2[bh, i] = LSE[bh,i]·log2(e);
// for i in [S_q, S_pad): delta = 0, lse2 = +inf.  Each lane loads 16 bytes of
// a row of O and of dO; a warp covers PREP_ROWS rows with all its loads
// issued before the first is used, then reduces each row across its lanes.
constexpr int kPrepIters = 4;

template <int D>
constexpr int prep_rows_per_warp() { return (32 / (D / 8)) * kPrepIters; }

__device__ __forceinline__ float dot8(uint4 a, uint4 b, bool bf16, float acc) {
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        float a0, a1, b0, b1;
        if (bf16) {
            a0 = __uint_as_float(aw[w] << 16); a1 = __uint_as_float(aw[w] & 0xffff0000u);
            b0 = __uint_as_float(bw[w] << 16); b1 = __uint_as_float(bw[w] & 0xffff0000u);
        } else {
            const float2 af = __half22float2(*reinterpret_cast<const __half2*>(&aw[w]));
            const float2 bf = __half22float2(*reinterpret_cast<const __half2*>(&bw[w]));
            a0 = af.x; a1 = af.y; b0 = bf.x; b1 = bf.y;
        }
        acc = fmaf(a0, b0, acc);
        acc = fmaf(a1, b1, acc);
    }
    return acc;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const uint16_t* __restrict__ o,
                                                            const uint16_t* __restrict__ dout,
                                                            const float* __restrict__ lse,
                                                            float* __restrict__ lse2,
                                                            float* __restrict__ delta, int S_q,
                                                            int S_pad, long long rows_pad, int H,
                                                            RowLayout o_lay, RowLayout do_lay) {
    constexpr int LPR = D / 8;                        // lanes per row, 8 elements each
    constexpr int RPI = 32 / LPR;                     // rows per load instruction
    const long long warp_id = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR;
    const int col = (lane % LPR) * 8;
    uint4 ov[kPrepIters], dv[kPrepIters];
    long long rr[kPrepIters];
    int ii[kPrepIters];
    long long bb[kPrepIters];
#pragma unroll
    for (int it = 0; it < kPrepIters; ++it) {
        const long long r = warp_id * (RPI * kPrepIters) + it * RPI + sub;
        rr[it] = r;
        ov[it] = make_uint4(0, 0, 0, 0);
        dv[it] = make_uint4(0, 0, 0, 0);
        const long long bh = r / S_pad;
        const int i = static_cast<int>(r - bh * S_pad);
        ii[it] = i;
        bb[it] = bh;
        if (r < rows_pad && i < S_q) {
            const long long b_ = bh / H, h_ = bh - b_ * H;
            ov[it] = *reinterpret_cast<const uint4*>(
                o + (b_ * o_lay.batch + h_ * o_lay.head + i * o_lay.row + col));
            dv[it] = *reinterpret_cast<const uint4*>(
                dout + (b_ * do_lay.batch + h_ * do_lay.head + i * do_lay.row + col));
        }
    }
#pragma unroll
    for (int it = 0; it < kPrepIters; ++it) {
        float acc = dot8(ov[it], dv[it], BF16, 0.f);
#pragma unroll
        for (int sh = LPR / 2; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
        if (lane % LPR == 0 && rr[it] < rows_pad) {
            if (ii[it] < S_q) {
                delta[rr[it]] = acc;
                lse2[rr[it]] = lse[static_cast<size_t>(bb[it]) * S_q + ii[it]] * 1.4426950408889634f;
            } else {
                delta[rr[it]] = 0.f;
                lse2[rr[it]] = __int_as_float(0x7f800000);
            }
        }
    }
}

// The warpgroup register split assumes the launch grants `regs` a thread;
// refuse to launch a build where it does not (setmaxnreg would stall).
template <typename K>
cudaError_t check_launch_regs(K kernel, int regs) {
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    return fa.numRegs == regs ? cudaSuccess : cudaErrorInvalidConfiguration;
}

// ============================================================== dK, dV
template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(BwdTile<D>::THREADS, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_k,    // box 64 × 128
                         const __grid_constant__ CUtensorMap tm_v,    // box 64 × 128
                         const __grid_constant__ CUtensorMap tm_q,    // box 64 × 64
                         const __grid_constant__ CUtensorMap tm_do,   // box 64 × 64
                         const __grid_constant__ CUtensorMap tm_dv,   // box 64 × 32, stores
                         const __grid_constant__ CUtensorMap tm_dk,   // box 64 × 32, stores
                         const float* __restrict__ lse2, const float* __restrict__ delta,
                         int S_q, int S_k, int BHkv, int H, int kv_group,
                         int S_pad, int head_group, int causal_off, float scale,
                         float scale_log2, DeviceWords* __restrict__ words,
                         unsigned long long launch, unsigned long long budget_ns) {
    using T = BwdTile<D>;
    using namespace sm100;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* sK = smem;
    uint8_t* sV = sK + T::BIG_TILE;
    uint8_t* sRing = sV + T::BIG_TILE;                // slot s: Q at s·SLOT, dO at +SMALL_TILE
    float* sStat = reinterpret_cast<float*>(sRing + T::NS * T::SLOT_BYTES);
    uint8_t* clc_resp = smem + T::TILE_BYTES;         // [CLC_SLOTS] 16-byte answers
    uint64_t* bars = reinterpret_cast<uint64_t*>(clc_resp + T::CLC_SLOTS * 16);
    uint64_t* kv_full = bars;
    uint64_t* kv_empty = kv_full + 1;
    uint64_t* slot_full = kv_empty + 1;
    uint64_t* slot_empty = slot_full + T::NS;
    uint64_t* s_full = slot_empty + T::NS;    // [2] Sᵀ and dPᵀ of buffer b computed
    uint64_t* p_full = s_full + 2;            // [2] Pᵀ and dSᵀ of buffer b written (per warp)
    uint64_t* acc_done = p_full + 2;          // dV and dK of the unit complete
    uint64_t* acc_free = acc_done + 1;        // [2] dV, dK read out (per epilogue warp)
    uint64_t* drain = acc_free + 2;
    uint64_t* clc_full = drain + 1;           // [CLC_SLOTS] work-queue answer landed
    uint64_t* clc_empty = clc_full + T::CLC_SLOTS;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(clc_empty + T::CLC_SLOTS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    unsigned int* status = &words->status;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_kt = (S_k + T::BU - 1) / T::BU;
    const int n_qs = (S_q + T::BS - 1) / T::BS;
    const int n_units = BHkv * n_kt;
    const int H_kv = H / kv_group;
    // A unit is (batch, key/value head, key tile); its steps run over the
    // kv_group query heads that read this head, each over its query tiles.
    // Causal: query rows that see none of the tile's keys are skipped.
    auto unit_info = [&](int L, int& b, int& hk, int& kt, int& q_begin, int& n) {
        int bhk;
        bwd_unit_coords<CAUSAL, true>(L, BHkv, n_kt, head_group, bhk, kt);
        b = bhk / H_kv;
        hk = bhk - b * H_kv;
        q_begin = CAUSAL ? min(n_qs, max(0, kt * T::BU - causal_off) / T::BS) : 0;
        n = (n_qs - q_begin) * kv_group;
    };
    // Steps of a unit visit query tiles q_begin .. n_qs-1 of each query head of
    // the group in turn; advance (h, qi) to the next step.
    auto next_step = [&](int q_begin, int& h, int& qi) {
        if (++qi == n_qs) {
            qi = q_begin;
            ++h;
        }
    };
    // Full attention: units come from the hardware work queue (one CTA per
    // unit in the grid; see WorkQueue), the producer claiming the next one
    // after each unit's loads.  Causal: a persistent grid takes the units in
    // rounds of gridDim.x, in serpentine order (CTA c takes position c of even
    // rounds and gridDim.x-1-c of odd ones).  unit_at returns 1 with the unit
    // in L, 2 when this CTA has no unit in round r, 0 when it is done, -1 when
    // a wait gave up.  The four softmax warps and the MMA warp consume queue
    // answers.
    const WorkQueue<T::CLC_SLOTS> queue{clc_resp, clc_full, clc_empty};
    auto unit_at = [&](int r, int& L, bool consumer, unsigned int code) -> int {
        if (!CAUSAL) return queue.unit(r, L, consumer, abort_flag, status, code);
        const int G = static_cast<int>(gridDim.x);
        const int c = static_cast<int>(blockIdx.x);
        if (static_cast<long long>(r) * G >= n_units) return 0;
        L = r * G + ((r & 1) ? (G - 1 - c) : c);
        return L < n_units ? 1 : 2;
    };

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        mbar_init(kv_empty, 1);
        for (int s = 0; s < T::NS; ++s) {
            mbar_init(&slot_full[s], 1);
            mbar_init(&slot_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], 4);
        }
        mbar_init(acc_done, 1);
        mbar_init(&acc_free[0], 4);
        mbar_init(&acc_free[1], 4);
        mbar_init(drain, 1);
        for (int s = 0; s < T::CLC_SLOTS; ++s) {
            mbar_init(&clc_full[s], 1);
            mbar_init(&clc_empty[s], 9);         // softmax and epilogue warps, the MMA warp
        }
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, T::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Each role below ends in its own copy of the teardown, so no code runs
    // under two register budgets.
    auto teardown = [&]() {
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            tc_fence_after();
            tmem_dealloc(tmem, T::TMEM_COLS);
            if (lane == 0) publish_abort(abort_flag, words, launch);
        }
    };

    if (warp >= T::PRODUCER_WARP) {
      regs_set<T::AUX_REGS, T::LAUNCH_REGS>();
      if (warp == T::PRODUCER_WARP) {
        // ------------------------------------------------------------ TMA producer
        const bool leader = elect_one();
        if (leader) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_do);
        }
        __syncwarp();
        LaunchWatch watch(words, launch, budget_ns);
        bool ok = true;
        int idx = 0;      // ring position, across units
        int uk = 0;       // units with work started by this CTA
        int claims = 0;   // work-queue requests issued (full attention)
        auto claim_next = [&]() {
            if (!CAUSAL) ok = queue.claim(claims, leader, abort_flag, status, kStatusBwdProducer);
        };
        for (int r = 0; ok; ++r) {
            if (watch.stop(abort_flag, status)) break;
            int L = 0;
            const int got = unit_at(r, L, false, kStatusBwdProducer);
            if (got < 0) ok = false;
            if (got <= 0) break;
            if (got == 2) continue;
            int b, hk, kt, q_begin, n;
            unit_info(L, b, hk, kt, q_begin, n);
#ifdef ATTN_DEBUG_FAULTS
            // Debug builds only: load nothing for the chosen unit and stop, so
            // its consumers' waits run out.
            if (L == g_attn_debug_skip_unit) break;
#endif
            if (n == 0) {
                claim_next();
                continue;
            }
            ok = mbar_wait(kv_empty, (uk & 1) ^ 1, abort_flag, status, kStatusBwdProducer);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ++uk;
            if (leader) {
                mbar_arrive_expect_tx(kv_full, 2 * T::BIG_TILE);
#pragma unroll
                for (int c = 0; c < T::CHUNKS; ++c) {
                    tma_load_4d(sK + c * T::BIG_CHUNK, &tm_k, kv_full, c * 64, kt * T::BU, hk, b);
                    tma_load_4d(sV + c * T::BIG_CHUNK, &tm_v, kv_full, c * 64, kt * T::BU, hk, b);
                }
            }
            __syncwarp();
            int h = hk * kv_group, qi = q_begin;
            for (int t = 0; t < n && ok; ++t, next_step(q_begin, h, qi)) {
                if ((idx & 7) == 0 && watch.stop(abort_flag, status)) {
                    ok = false;
                    break;
                }
                const int slot = idx % T::NS;
                ok = mbar_wait(&slot_empty[slot], ((idx / T::NS) & 1) ^ 1, abort_flag, status,
                               kStatusBwdProducer);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                if (leader) {
                    const int q0 = qi * T::BS;
                    uint8_t* dst = sRing + slot * T::SLOT_BYTES;
                    float* st = sStat + slot * T::STAT_FLOATS;
                    const size_t soff = (static_cast<size_t>(b) * H + h) * S_pad + q0;
                    mbar_arrive_expect_tx(&slot_full[slot], T::SLOT_BYTES + T::STAT_FLOATS * 4);
#pragma unroll
                    for (int c = 0; c < T::CHUNKS; ++c) {
                        tma_load_4d(dst + c * T::SMALL_CHUNK, &tm_q, &slot_full[slot], c * 64, q0,
                                    h, b);
                        tma_load_4d(dst + T::SMALL_TILE + c * T::SMALL_CHUNK, &tm_do,
                                    &slot_full[slot], c * 64, q0, h, b);
                    }
                    bulk_load(st, lse2 + soff, T::BS * 4, &slot_full[slot]);
                    bulk_load(st + T::BS, delta + soff, T::BS * 4, &slot_full[slot]);
                }
                __syncwarp();
                ++idx;
            }
            if (!ok) break;
            if (uk == 1 && watch.launch_gave_up(abort_flag)) break;
            claim_next();    // the next unit, once this one's loads are all issued
        }
        if (*abort_flag && leader) {
            // Let every copy this CTA started land before it exits.
            const uint64_t t0 = global_timer_ns();
            for (int i = max(0, idx - T::NS); i < idx; ++i) {
                const uint32_t a = smem_u32(&slot_full[i % T::NS]);
                while (!mbar_try_wait(a, (i / T::NS) & 1)) {
                    if (global_timer_ns() - t0 > kWaitLimitNs) {
                        atomicOr(status, kStatusBwdDrain);
                        break;
                    }
                }
            }
            if (uk > 0) {
                const uint32_t a = smem_u32(kv_full);
                while (!mbar_try_wait(a, static_cast<uint32_t>(uk - 1) & 1u)) {
                    if (global_timer_ns() - t0 > kWaitLimitNs) {
                        atomicOr(status, kStatusBwdDrain);
                        break;
                    }
                }
            }
            queue.drain(claims, status, kStatusBwdDrain);
        }
        __syncwarp();
      } else if (warp == T::MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t id_s = idesc_f16(128, T::BS, BF16, false, false);
        constexpr uint32_t id_acc = idesc_f16(128, D, BF16, false, true);
        const uint64_t k_desc = sdesc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t v_desc = sdesc_sw128(smem_u32(sV), 16, 1024);
        const uint64_t rk_desc = sdesc_sw128(smem_u32(sRing), 16, 1024);            // K-major
        const uint64_t rm_desc = sdesc_sw128(smem_u32(sRing), T::SMALL_CHUNK, 1024); // MN-major
        const uint32_t k_lo = static_cast<uint32_t>(k_desc), k_hi = static_cast<uint32_t>(k_desc >> 32);
        const uint32_t v_lo = static_cast<uint32_t>(v_desc), v_hi = static_cast<uint32_t>(v_desc >> 32);
        const uint32_t rk_lo = static_cast<uint32_t>(rk_desc), rk_hi = static_cast<uint32_t>(rk_desc >> 32);
        const uint32_t rm_lo = static_cast<uint32_t>(rm_desc), rm_hi = static_cast<uint32_t>(rm_desc >> 32);
        bool ok = true;
        int acq = 0;                 // ring position, across units
        uint32_t gs = 0;             // steps issued, across units (S/dP buffer = gs & 1)
        int uk = 0;
        auto acquire = [&](int& slot) {
            if (!ok) return;
            slot = acq % T::NS;
            ok = mbar_wait(&slot_full[slot], (acq / T::NS) & 1, abort_flag, status, kStatusBwdMma);
            ok = __all_sync(0xffffffffu, ok);
            ++acq;
            tc_fence_after();
        };
        // Sᵀ_b = K·Q_slotᵀ and dPᵀ_b = V·dO_slotᵀ: M = 128 keys, N = 64 queries, K = D
        auto mma_s = [&](int slot, int b) {
            const uint32_t qoff = (slot * T::SLOT_BYTES) >> 4;
            const uint32_t dooff = (slot * T::SLOT_BYTES + T::SMALL_TILE) >> 4;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t ao = ((kk >> 2) * T::BIG_CHUNK + (kk & 3) * 32) >> 4;
                const uint32_t bo = ((kk >> 2) * T::SMALL_CHUNK + (kk & 3) * 32) >> 4;
                mma_ss_warp(tmem + T::S_COL + b * 64, k_lo + ao, k_hi, rk_lo + qoff + bo, rk_hi,
                            id_s, kk > 0 ? 1u : 0u);
                mma_ss_warp(tmem + T::DP_COL + b * 64, v_lo + ao, v_hi, rk_lo + dooff + bo, rk_hi,
                            id_s, kk > 0 ? 1u : 0u);
            }
        };
        // dV += Pᵀ_b·dO_slot (g = 0) and dK += dSᵀ_b·Q_slot (g = 1): M = 128
        // keys, N = D, K = 64 queries.  mask bit g selects the products; with
        // both, the two accumulators' MMAs alternate.
        auto mma_acc = [&](int slot, int b, bool acc, int mask) {
            const uint32_t qoff = (slot * T::SLOT_BYTES) >> 4;
            const uint32_t dooff = (slot * T::SLOT_BYTES + T::SMALL_TILE) >> 4;
#pragma unroll
            for (int kk = 0; kk < T::BS / 16; ++kk) {
                const uint32_t bo = (kk * 16 * 128) >> 4;
                if (mask & 1)
                    mma_ts_warp(tmem + T::ACC_COL, tmem + T::S_COL + b * 64 + T::PK_OFF + kk * 8,
                                rm_lo + dooff + bo, rm_hi, id_acc, (acc || kk > 0) ? 1u : 0u);
                if (mask & 2)
                    mma_ts_warp(tmem + T::ACC_COL + D,
                                tmem + T::DP_COL + b * 64 + T::PK_OFF + kk * 8, rm_lo + qoff + bo,
                                rm_hi, id_acc, (acc || kk > 0) ? 1u : 0u);
            }
        };
        uint32_t pc0 = 0, pc1 = 0;
        for (int r = 0; ok; ++r) {
            int L = 0;
            const int got = unit_at(r, L, true, kStatusBwdMma);
            if (got < 0) ok = false;
            if (got <= 0) break;
            if (got == 2) continue;
            int b, hk, kt, q_begin, n;
            unit_info(L, b, hk, kt, q_begin, n);
            if (n == 0) continue;
            ok = mbar_wait(kv_full, uk & 1, abort_flag, status, kStatusBwdMma);
            ok = __all_sync(0xffffffffu, ok);
            ++uk;
            tc_fence_after();
            if (!ok) break;
            int sl = 0;
            acquire(sl);
            if (!ok) break;
            mma_s(sl, gs & 1);
            tc_commit_warp(&s_full[gs & 1]);
            int sl_next = 0;
            if (n > 1) {
                acquire(sl_next);
                if (!ok) break;
                mma_s(sl_next, (gs + 1) & 1);
                tc_commit_warp(&s_full[(gs + 1) & 1]);
            }
            if (n <= 2) tc_commit_warp(kv_empty);          // K and V no longer needed
            int cur = sl, nxt = sl_next;
            for (int t = 0; t < n && ok; ++t) {
                const int b = static_cast<int>((gs + t) & 1);
                ok = mbar_wait(&p_full[b], (b ? pc1 : pc0) & 1, abort_flag, status, kStatusBwdMma);
                ok = __all_sync(0xffffffffu, ok);
                if (b) ++pc1; else ++pc0;
                tc_fence_after();
                if (!ok) break;
                if (t == 0 && uk > 1) {
                    // A unit's first dV (dK) MMA overwrites that accumulator:
                    // the epilogue warps must have read out the previous unit's.
                    for (int g = 0; g < 2 && ok; ++g) {
                        ok = mbar_wait(&acc_free[g], (uk - 2) & 1, abort_flag, status,
                                       kStatusBwdMma);
                        ok = __all_sync(0xffffffffu, ok);
                        tc_fence_after();
                        if (ok) mma_acc(cur, b, false, 1 << g);
                    }
                    if (!ok) break;
                } else {
                    mma_acc(cur, b, t > 0, 3);
                }
                tc_commit_warp(&slot_empty[cur]);
                int nn = 0;
                if (t + 2 < n) {
                    acquire(nn);
                    if (!ok) break;
                    mma_s(nn, b);
                    tc_commit_warp(&s_full[b]);
                    if (t + 3 == n) tc_commit_warp(kv_empty);
                }
                cur = nxt;
                nxt = nn;
            }
            if (!ok) break;
            tc_commit_warp(acc_done);
            gs += static_cast<uint32_t>(n);
        }
        tc_commit_warp(drain);
        const uint32_t a = smem_u32(drain);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(a, 0)) {
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                if (elect_one()) {
                    *abort_flag = 1;
                    atomicOr(status, kStatusBwdDrain);
                }
                break;
            }
        }
        __syncwarp();
      }
      teardown();
    } else if (warp >= T::EPI_WARP) {
        regs_set<T::EPI_REGS, T::LAUNCH_REGS>();
        // ------------------------------------------------------------ epilogue warps
        // Read dV out of tensor memory as packed 16-bit rows (one key row per
        // thread), release it to the next unit and store it, then the same
        // for dK: 64 columns of the warp's 32 rows at a time, through its
        // staging tile.
        const int quarter = warp & 3;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        uint8_t* tile = smem + T::STG_OFF + quarter * T::STG_WARP;
        bool ok = true;
        int ue = 0;
        for (int r = 0; ok; ++r) {
            int L = 0;
            const int got = unit_at(r, L, true, kStatusBwdEpilogue);
            if (got < 0) ok = false;
            if (got <= 0) break;
            if (got == 2) continue;
            int b, hk, kt, q_begin, n;
            unit_info(L, b, hk, kt, q_begin, n);
            const int row0 = kt * T::BU + quarter * 32;
            // Keys no query sees (n = 0) get zero gradients.
            uint32_t wv[D / 2], wk[D / 2];
            if (n > 0) {
                ok = mbar_wait_idle(acc_done, ue & 1, abort_flag, status, kStatusBwdEpilogue);
                ok = __all_sync(0xffffffffu, ok);
                ++ue;
                if (!ok) break;
                tc_fence_after();
                read_acc_packed<D, BF16>(lane_base + T::ACC_COL, 1.f, wv);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_free[0]);
            } else {
#pragma unroll
                for (int i = 0; i < D / 2; ++i) wv[i] = 0u;
            }
#pragma unroll
            for (int c = 0; c < D; c += 64)
                store_tile_64(wv + c / 2, tile, lane, &tm_dv, c, row0, hk, b);
            if (n > 0) {
                read_acc_packed<D, BF16>(lane_base + T::ACC_COL + D, scale, wk);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_free[1]);
            } else {
#pragma unroll
                for (int i = 0; i < D / 2; ++i) wk[i] = 0u;
            }
#pragma unroll
            for (int c = 0; c < D; c += 64)
                store_tile_64(wk + c / 2, tile, lane, &tm_dk, c, row0, hk, b);
        }
        bulk_wait_all();       // every tile store has landed before the CTA exits
        teardown();
    } else {
        // ------------------------------------------------------------ softmax warps
        regs_set<T::SOFTMAX_REGS, T::LAUNCH_REGS>();
        const int row = warp * 32 + lane;              // key row within the tile
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        bool ok = true;
        uint32_t gs = 0;
        for (int r = 0; ok; ++r) {
            int L = 0;
            const int got = unit_at(r, L, true, kStatusBwdSoftmax);
            if (got < 0) ok = false;
            if (got <= 0) break;
            if (got == 2) continue;
            int b, hk, kt, q_begin, n;
            unit_info(L, b, hk, kt, q_begin, n);
            const int key = kt * T::BU + row;
            int h = hk * kv_group, qi = q_begin;
            for (int t = 0; t < n; ++t, next_step(q_begin, h, qi)) {
                const uint32_t s = gs + static_cast<uint32_t>(t);
                const int buf = static_cast<int>(s & 1);
                const int slot = static_cast<int>(s % T::NS);
                ok = mbar_wait(&s_full[buf], (s >> 1) & 1, abort_flag, status, kStatusBwdSoftmax);
                if (ok) ok = mbar_wait(&slot_full[slot], (s / T::NS) & 1, abort_flag, status,
                                       kStatusBwdSoftmax);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                uint32_t sv[64], dpv[64];
                tmem_ld64(lane_base + T::S_COL + buf * 64, sv);
                tmem_ld64(lane_base + T::DP_COL + buf * 64, dpv);
                const float* st = sStat + slot * T::STAT_FLOATS;
                const int q0 = qi * T::BS;
                // key > query + causal_off is masked; only steps that reach below the
                // diagonal need it
                const bool masked = CAUSAL && q0 + causal_off < kt * T::BU + T::BU - 1;
                uint32_t pk_p[32], pk_ds[32];
                if (masked) {
                    const int lim = key - q0 - causal_off;     // visible iff c >= lim
                    grad_pack64<true, BF16, true, true>(sv, dpv, st, st + T::BS, 0.f, 0.f,
                                                        scale_log2,
                                                        [&](int c) { return c >= lim; }, pk_p, pk_ds);
                } else {
                    grad_pack64<false, BF16, true, true>(sv, dpv, st, st + T::BS, 0.f, 0.f,
                                                         scale_log2, [](int) { return true; },
                                                         pk_p, pk_ds);
                }
                tmem_st32(lane_base + T::S_COL + buf * 64 + T::PK_OFF, pk_p);
                tmem_st32(lane_base + T::DP_COL + buf * 64 + T::PK_OFF, pk_ds);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[buf]);
            }
            if (!ok) break;
            gs += static_cast<uint32_t>(n);
        }
        teardown();
    }
}

// ============================================================== dQ
// 128-key steps for d <= 128, so every Q·Kᵀ / dO·Vᵀ MMA has N = 128; 64-key
// steps for d = 256, where the fixed Q and dO tiles take 128 KB of shared
// memory.  Tensor memory: S in two buffers (columns 0 and BS; dS overwrites
// the first BS/2 columns of its own buffer as packed 16-bit pairs), one dP
// buffer (2·BS) that the softmax warps release as soon as they have read it,
// and dQ.  K and V arrive through separate shared-memory rings.
template <int D>
struct DqTile {
    static_assert(D == 64 || D == 128 || D == 256, "head_dim 64, 128 or 256");
    static constexpr int BU = 128;                    // query rows per unit
    static constexpr int BS = D == 256 ? 64 : 128;    // keys per step
    static constexpr int CHUNKS = D / 64;
    static constexpr int FIX_CHUNK = BU * 128;        // one atom column of the 128-row Q / dO
    static constexpr int FIX_TILE = BU * D * 2;
    static constexpr int KV_CHUNK = BS * 128;         // of a K / V step
    static constexpr int KV_TILE = BS * D * 2;
    // K and V stream through rings of their own: V of a step is free once its
    // dP MMA is done, K only after the step's dQ MMA.
    static constexpr int KS = D == 64 ? 5 : (D == 128 ? 3 : 2);   // K ring slots
    static constexpr int VS = D == 64 ? 4 : (D == 128 ? 2 : 1);   // V ring slots
    static constexpr int CLC_SLOTS = 4;               // work-queue answers in flight
    static constexpr int NUM_BARS = 2 + 2 * KS + 2 * VS + 2 + 1 + 2 + 1 + 1 + 1 + 2 * CLC_SLOTS;
    static constexpr int TILE_BYTES = 2 * FIX_TILE + (KS + VS) * KV_TILE;
    static constexpr int SMEM_BYTES = 1024 + TILE_BYTES + CLC_SLOTS * 16 + NUM_BARS * 8 + 16;
    static constexpr int THREADS = 384;     // softmax warps 0-3, epilogue 4-7, producer, MMA, 2 idle
    static constexpr int EPI_WARP = 4;      // first epilogue warp (warp % 4 = its lane quarter)
    static constexpr int PRODUCER_WARP = 8;
    static constexpr int MMA_WARP = 9;
    // Register split: the launch grants LAUNCH_REGS a thread (65536 over 12
    // warps, rounded down to a multiple of 8); the softmax and epilogue
    // warpgroups grow to their budgets, the aux warpgroup (producer, MMA and
    // two idle warps) shrinks to its own.  The sum is 3·LAUNCH_REGS.
    static constexpr int LAUNCH_REGS = 168;
    static constexpr int SOFTMAX_REGS = 176;
    static constexpr int EPI_REGS = 192;
    static constexpr int AUX_REGS = 136;
    static_assert(SOFTMAX_REGS + EPI_REGS + AUX_REGS <= 3 * LAUNCH_REGS, "register split");
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 0;              // S buffer b at BS·b
    static constexpr uint32_t DP_COL = 2 * BS;
    static constexpr uint32_t ACC_COL = D == 256 ? 256 : 384;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(DP_COL + BS <= ACC_COL && ACC_COL + D <= TMEM_COLS, "tensor memory budget");
};

template <int D, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(DqTile<D>::THREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,    // box 64 × 128
                       const __grid_constant__ CUtensorMap tm_do,   // box 64 × 128
                       const __grid_constant__ CUtensorMap tm_k,    // box 64 × 128
                       const __grid_constant__ CUtensorMap tm_v,    // box 64 × 128
                       const float* __restrict__ lse2, const float* __restrict__ delta,
                       uint16_t* __restrict__ dq, RowLayout dq_lay, int S_q, int S_k, int BH,
                       int H, int kv_group, int S_pad, int head_group, int causal_off,
                       float scale, float scale_log2, DeviceWords* __restrict__ words,
                       unsigned long long launch, unsigned long long budget_ns) {
    using T = DqTile<D>;
    using namespace sm100;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* sQ = smem;
    uint8_t* sdO = sQ + T::FIX_TILE;
    uint8_t* sKr = sdO + T::FIX_TILE;                  // K ring
    uint8_t* sVr = sKr + T::KS * T::KV_TILE;           // V ring
    uint8_t* clc_resp = smem + T::TILE_BYTES;          // [CLC_SLOTS] 16-byte answers
    uint64_t* bars = reinterpret_cast<uint64_t*>(clc_resp + T::CLC_SLOTS * 16);
    uint64_t* q_full = bars;
    uint64_t* q_empty = q_full + 1;
    uint64_t* k_full = q_empty + 1;
    uint64_t* k_empty = k_full + T::KS;
    uint64_t* v_full = k_empty + T::KS;
    uint64_t* v_empty = v_full + T::VS;
    uint64_t* s_full = v_empty + T::VS;      // [2] S_b and the dP of that step computed
    uint64_t* dp_free = s_full + 2;          // the dP buffer has been read (per warp)
    uint64_t* p_full = dp_free + 1;          // [2] dS written over S_b (per warp)
    uint64_t* acc_done = p_full + 2;
    uint64_t* acc_free = acc_done + 1;       // dQ read out (per epilogue warp)
    uint64_t* drain = acc_free + 1;
    uint64_t* clc_full = drain + 1;          // [CLC_SLOTS] work-queue answer landed
    uint64_t* clc_empty = clc_full + T::CLC_SLOTS;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(clc_empty + T::CLC_SLOTS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    unsigned int* status = &words->status;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n_qt = (S_q + T::BU - 1) / T::BU;
    const int n_ks = (S_k + T::BS - 1) / T::BS;
    const int n_units = BH * n_qt;
    auto unit_info = [&](int L, int& bh, int& qt, int& n) {
        bwd_unit_coords<CAUSAL, false>(L, BH, n_qt, head_group, bh, qt);
        n = n_ks;
        if (CAUSAL) {
            const int last_key = min(qt * T::BU + T::BU, S_q) - 1 + causal_off;
            n = min(n_ks, last_key / T::BS + 1);
        }
    };
    // Full attention: units come from the hardware work queue (one CTA per
    // unit in the grid; see WorkQueue), the producer claiming the next one
    // after each unit's loads.  Causal: a persistent grid takes the units in
    // rounds of gridDim.x, in serpentine order (CTA c takes position c of even
    // rounds and gridDim.x-1-c of odd ones).  unit_at returns 1 with the unit
    // in L, 2 when this CTA has no unit in round r, 0 when it is done, -1 when
    // a wait gave up.  The four softmax warps and the MMA warp consume queue
    // answers.
    const WorkQueue<T::CLC_SLOTS> queue{clc_resp, clc_full, clc_empty};
    auto unit_at = [&](int r, int& L, bool consumer, unsigned int code) -> int {
        if (!CAUSAL) return queue.unit(r, L, consumer, abort_flag, status, code);
        const int G = static_cast<int>(gridDim.x);
        const int c = static_cast<int>(blockIdx.x);
        if (static_cast<long long>(r) * G >= n_units) return 0;
        L = r * G + ((r & 1) ? (G - 1 - c) : c);
        return L < n_units ? 1 : 2;
    };

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < T::KS; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < T::VS; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], 4);
        }
        mbar_init(dp_free, 4);
        mbar_init(acc_done, 1);
        mbar_init(acc_free, 4);
        mbar_init(drain, 1);
        for (int s = 0; s < T::CLC_SLOTS; ++s) {
            mbar_init(&clc_full[s], 1);
            mbar_init(&clc_empty[s], 9);         // softmax and epilogue warps, the MMA warp
        }
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, T::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Each role below ends in its own copy of the teardown, so no code runs
    // under two register budgets.
    auto teardown = [&]() {
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            tc_fence_after();
            tmem_dealloc(tmem, T::TMEM_COLS);
            if (lane == 0) publish_abort(abort_flag, words, launch);
        }
    };

    if (warp >= T::PRODUCER_WARP) {
      regs_set<T::AUX_REGS, T::LAUNCH_REGS>();
      if (warp == T::PRODUCER_WARP) {
        const bool leader = elect_one();
        if (leader) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_do);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
        }
        __syncwarp();
        LaunchWatch watch(words, launch, budget_ns);
        bool ok = true;
        int kidx = 0, vidx = 0;
        int uq = 0;
        // One tile into ring slot idx % SLOTS once its previous use is released.
        auto load = [&](const CUtensorMap* map, uint8_t* ring, uint64_t* full, uint64_t* empty,
                        int slots, int& idx, int row, int hk, int b) {
            if (!ok) return;
            if ((idx & 7) == 0 && watch.stop(abort_flag, status)) {
                ok = false;
                return;
            }
            const int slot = idx % slots;
            ok = mbar_wait(&empty[slot], ((idx / slots) & 1) ^ 1, abort_flag, status,
                           kStatusBwdProducer);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) return;
            if (leader) {
                mbar_arrive_expect_tx(&full[slot], T::KV_TILE);
#pragma unroll
                for (int c = 0; c < T::CHUNKS; ++c)
                    tma_load_4d(ring + slot * T::KV_TILE + c * T::KV_CHUNK, map, &full[slot], c * 64,
                                row, hk, b);
            }
            __syncwarp();
            ++idx;
        };
        int claims = 0;   // work-queue requests issued (full attention)
        for (int r = 0; ok; ++r) {
            if (watch.stop(abort_flag, status)) break;
            int L = 0;
            const int got = unit_at(r, L, false, kStatusBwdProducer);
            if (got < 0) ok = false;
            if (got <= 0) break;
            if (got == 2) continue;
            int bh, qt, n;
            unit_info(L, bh, qt, n);
            const int b = bh / H, h = bh - b * H, hk = h / kv_group;
            ok = mbar_wait(q_empty, (uq & 1) ^ 1, abort_flag, status, kStatusBwdProducer);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ++uq;
            if (leader) {
                mbar_arrive_expect_tx(q_full, 2 * T::FIX_TILE);
#pragma unroll
                for (int c = 0; c < T::CHUNKS; ++c) {
                    tma_load_4d(sQ + c * T::FIX_CHUNK, &tm_q, q_full, c * 64, qt * T::BU, h, b);
                    tma_load_4d(sdO + c * T::FIX_CHUNK, &tm_do, q_full, c * 64, qt * T::BU, h, b);
                }
            }
            __syncwarp();
            for (int t = 0; t < n && ok; ++t) {
                load(&tm_k, sKr, k_full, k_empty, T::KS, kidx, t * T::BS, hk, b);
                load(&tm_v, sVr, v_full, v_empty, T::VS, vidx, t * T::BS, hk, b);
            }
            if (!ok) break;
            if (uq == 1 && watch.launch_gave_up(abort_flag)) break;
            // the next unit, once this one's loads are all issued
            if (!CAUSAL) ok = queue.claim(claims, leader, abort_flag, status, kStatusBwdProducer);
        }
        if (*abort_flag && leader) {
            const uint64_t t0 = global_timer_ns();
            auto drain_ring = [&](uint64_t* full, int slots, int idx) {
                for (int i = max(0, idx - slots); i < idx; ++i) {
                    const uint32_t a = smem_u32(&full[i % slots]);
                    while (!mbar_try_wait(a, (i / slots) & 1)) {
                        if (global_timer_ns() - t0 > kWaitLimitNs) {
                            atomicOr(status, kStatusBwdDrain);
                            break;
                        }
                    }
                }
            };
            drain_ring(k_full, T::KS, kidx);
            drain_ring(v_full, T::VS, vidx);
            if (uq > 0) {
                const uint32_t a = smem_u32(q_full);
                while (!mbar_try_wait(a, static_cast<uint32_t>(uq - 1) & 1u)) {
                    if (global_timer_ns() - t0 > kWaitLimitNs) {
                        atomicOr(status, kStatusBwdDrain);
                        break;
                    }
                }
            }
            queue.drain(claims, status, kStatusBwdDrain);
        }
        __syncwarp();
      } else if (warp == T::MMA_WARP) {
        constexpr uint32_t id_s = idesc_f16(128, T::BS, BF16, false, false);
        constexpr uint32_t id_acc = idesc_f16(128, D, BF16, false, true);
        const uint64_t q_desc = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t do_desc = sdesc_sw128(smem_u32(sdO), 16, 1024);
        const uint64_t kk_desc = sdesc_sw128(smem_u32(sKr), 16, 1024);          // K as K-major B
        const uint64_t km_desc = sdesc_sw128(smem_u32(sKr), T::KV_CHUNK, 1024); // K as MN-major B
        const uint64_t vk_desc = sdesc_sw128(smem_u32(sVr), 16, 1024);
        const uint32_t q_lo = static_cast<uint32_t>(q_desc), q_hi = static_cast<uint32_t>(q_desc >> 32);
        const uint32_t do_lo = static_cast<uint32_t>(do_desc), do_hi = static_cast<uint32_t>(do_desc >> 32);
        const uint32_t kk_lo = static_cast<uint32_t>(kk_desc), kk_hi = static_cast<uint32_t>(kk_desc >> 32);
        const uint32_t km_lo = static_cast<uint32_t>(km_desc), km_hi = static_cast<uint32_t>(km_desc >> 32);
        const uint32_t vk_lo = static_cast<uint32_t>(vk_desc), vk_hi = static_cast<uint32_t>(vk_desc >> 32);
        bool ok = true;
        int kacq = 0, vacq = 0;
        uint32_t gs = 0;              // steps of all units so far (S buffer = step & 1)
        int uq = 0;
        uint32_t dpf = 0;             // dp_free phases consumed
        uint32_t pc0 = 0, pc1 = 0;
        auto acquire = [&](uint64_t* full, int slots, int& acq, int& slot) {
            if (!ok) return;
            slot = acq % slots;
            ok = mbar_wait(&full[slot], (acq / slots) & 1, abort_flag, status, kStatusBwdMma);
            ok = __all_sync(0xffffffffu, ok);
            ++acq;
            tc_fence_after();
        };
        // S_b = Q·K_slotᵀ: M = 128 queries, N = 128 keys, K = D
        auto mma_s = [&](int slot, int b) {
            const uint32_t koff = (slot * T::KV_TILE) >> 4;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t o = ((kk >> 2) * T::FIX_CHUNK + (kk & 3) * 32) >> 4;
                const uint32_t ok_ = ((kk >> 2) * T::KV_CHUNK + (kk & 3) * 32) >> 4;
                mma_ss_warp(tmem + T::S_COL + b * T::BS, q_lo + o, q_hi, kk_lo + koff + ok_, kk_hi,
                            id_s, kk > 0 ? 1u : 0u);
            }
        };
        // dP = dO·V_slotᵀ
        auto mma_dp = [&](int slot) {
            const uint32_t voff = (slot * T::KV_TILE) >> 4;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t o = ((kk >> 2) * T::FIX_CHUNK + (kk & 3) * 32) >> 4;
                const uint32_t ov = ((kk >> 2) * T::KV_CHUNK + (kk & 3) * 32) >> 4;
                mma_ss_warp(tmem + T::DP_COL, do_lo + o, do_hi, vk_lo + voff + ov, vk_hi, id_s,
                            kk > 0 ? 1u : 0u);
            }
        };
        // dQ += dS_b·K_slot: M = 128 queries, N = D, K = 128 keys (dS packed in cols 0..63 of S_b)
        auto mma_acc = [&](int slot, int b, bool acc) {
            const uint32_t koff = (slot * T::KV_TILE) >> 4;
#pragma unroll
            for (int kk = 0; kk < T::BS / 16; ++kk) {
                const uint32_t bo = (kk * 16 * 128) >> 4;
                mma_ts_warp(tmem + T::ACC_COL, tmem + T::S_COL + b * T::BS + kk * 8,
                            km_lo + koff + bo, km_hi, id_acc, (acc || kk > 0) ? 1u : 0u);
            }
        };
        auto wait_dp_free = [&]() {
            if (!ok) return;
            ok = mbar_wait(dp_free, dpf & 1, abort_flag, status, kStatusBwdMma);
            ok = __all_sync(0xffffffffu, ok);
            ++dpf;
            tc_fence_after();
        };
        // The dP buffer is free for the first step of a unit once the previous
        // unit's last step has released it (dpf counts releases; gs counts steps).
        for (int r = 0; ok; ++r) {
            int L = 0;
            const int got = unit_at(r, L, true, kStatusBwdMma);
            if (got < 0) ok = false;
            if (got <= 0) break;
            if (got == 2) continue;
            int bh, qt, n;
            unit_info(L, bh, qt, n);
            ok = mbar_wait(q_full, uq & 1, abort_flag, status, kStatusBwdMma);
            ok = __all_sync(0xffffffffu, ok);
            ++uq;
            tc_fence_after();
            if (!ok) break;
            int cur = 0, nxt = 0, vs = 0;
            acquire(k_full, T::KS, kacq, cur);
            if (!ok) break;
            mma_s(cur, gs & 1);
            if (gs > 0) wait_dp_free();                    // previous step's dP read
            acquire(v_full, T::VS, vacq, vs);
            if (!ok) break;
            mma_dp(vs);
            tc_commit_warp(&v_empty[vs]);
            tc_commit_warp(&s_full[gs & 1]);
            if (n > 1) {
                acquire(k_full, T::KS, kacq, nxt);
                if (!ok) break;
                mma_s(nxt, (gs + 1) & 1);
            }
            for (int t = 0; t < n && ok; ++t) {
                const int b = static_cast<int>((gs + t) & 1);
                if (t + 1 < n) {
                    // dP of the next step once the softmax warps have read this one's
                    wait_dp_free();
                    acquire(v_full, T::VS, vacq, vs);
                    if (!ok) break;
                    mma_dp(vs);
                    tc_commit_warp(&v_empty[vs]);
                    tc_commit_warp(&s_full[b ^ 1]);
                    if (t + 2 == n) tc_commit_warp(q_empty);   // last use of Q and dO issued
                } else if (n == 1) {
                    tc_commit_warp(q_empty);
                }
                ok = mbar_wait(&p_full[b], (b ? pc1 : pc0) & 1, abort_flag, status, kStatusBwdMma);
                // the unit's first dQ MMA overwrites the accumulator: the
                // epilogue warps must have read out the previous unit's
                if (ok && t == 0 && uq > 1)
                    ok = mbar_wait(acc_free, (uq - 2) & 1, abort_flag, status, kStatusBwdMma);
                ok = __all_sync(0xffffffffu, ok);
                if (b) ++pc1; else ++pc0;
                tc_fence_after();
                if (!ok) break;
                mma_acc(cur, b, t > 0);
                tc_commit_warp(&k_empty[cur]);
                int nn = 0;
                if (t + 2 < n) {
                    acquire(k_full, T::KS, kacq, nn);
                    if (!ok) break;
                    mma_s(nn, b);
                }
                cur = nxt;
                nxt = nn;
            }
            if (!ok) break;
            tc_commit_warp(acc_done);
            gs += static_cast<uint32_t>(n);
        }
        tc_commit_warp(drain);
        const uint32_t a = smem_u32(drain);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(a, 0)) {
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                if (elect_one()) {
                    *abort_flag = 1;
                    atomicOr(status, kStatusBwdDrain);
                }
                break;
            }
        }
        __syncwarp();
      }
      teardown();
    } else if (warp >= T::EPI_WARP) {
        regs_set<T::EPI_REGS, T::LAUNCH_REGS>();
        // Epilogue warps: read dQ out of tensor memory as packed 16-bit rows,
        // release the accumulator to the next unit, then store (one query row
        // per thread).
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        bool ok = true;
        int ue = 0;
        for (int r = 0; ok; ++r) {
            int L = 0;
            const int got = unit_at(r, L, true, kStatusBwdEpilogue);
            if (got < 0) ok = false;
            if (got <= 0) break;
            if (got == 2) continue;
            int bh, qt, n;
            unit_info(L, bh, qt, n);
            const int q_idx = qt * T::BU + row;
            ok = mbar_wait_idle(acc_done, ue & 1, abort_flag, status, kStatusBwdEpilogue);
            ok = __all_sync(0xffffffffu, ok);
            ++ue;
            if (!ok) break;
            tc_fence_after();
            uint32_t pq[D / 2];
            read_acc_packed<D, BF16>(lane_base + T::ACC_COL, scale, pq);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free);
            const int b = bh / H, h = bh - b * H;
            if (q_idx < S_q)
                store_packed_row<D>(pq, dq + static_cast<size_t>(b * dq_lay.batch + h * dq_lay.head +
                                                                 static_cast<long long>(q_idx) *
                                                                     dq_lay.row));
        }
        teardown();
    } else {
        regs_set<T::SOFTMAX_REGS, T::LAUNCH_REGS>();
        const int row = warp * 32 + lane;                // query row within the tile
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        bool ok = true;
        uint32_t gs = 0;
        for (int r = 0; ok; ++r) {
            int L = 0;
            const int got = unit_at(r, L, true, kStatusBwdSoftmax);
            if (got < 0) ok = false;
            if (got <= 0) break;
            if (got == 2) continue;
            int bh, qt, n;
            unit_info(L, bh, qt, n);
            const int q_idx = qt * T::BU + row;
            const float row_lse2 = lse2[static_cast<size_t>(bh) * S_pad + q_idx];
            const float row_dd = delta[static_cast<size_t>(bh) * S_pad + q_idx];
            const int row_begin = qt * T::BU;
            for (int t = 0; t < n; ++t) {
                const uint32_t s = gs + static_cast<uint32_t>(t);
                const int b = static_cast<int>(s & 1);
                ok = mbar_wait(&s_full[b], (s >> 1) & 1, abort_flag, status, kStatusBwdSoftmax);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const int kv0 = t * T::BS;
                const bool masked =
                    (CAUSAL && kv0 + T::BS - 1 > row_begin + causal_off) || (kv0 + T::BS > S_k);
                const int lim =
                    masked ? min(S_k, CAUSAL ? q_idx + 1 + causal_off : S_k) - kv0 : T::BS;
                const uint32_t sb = lane_base + T::S_COL + b * T::BS;
                // Halves of 64 keys (two for 128-key steps); dS of half h goes to
                // columns 32h..32h+31 of S_b, which have been read by then.
#pragma unroll 1
                for (int h = 0; h < T::BS / 64; ++h) {
                    uint32_t sv[64], dpv[64];
                    tmem_ld64(sb + h * 64, sv);
                    tmem_ld64(lane_base + T::DP_COL + h * 64, dpv);
                    if (h == T::BS / 64 - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(dp_free);
                    }
                    uint32_t pk_p[32], pk_ds[32];
                    const int hl = lim - h * 64;
                    if (masked) {
                        grad_pack64<true, BF16, false, false>(sv, dpv, nullptr, nullptr, row_lse2,
                                                              row_dd, scale_log2,
                                                              [&](int c) { return c < hl; }, pk_p,
                                                              pk_ds);
                    } else {
                        grad_pack64<false, BF16, false, false>(sv, dpv, nullptr, nullptr,
                                                               row_lse2, row_dd, scale_log2,
                                                               [](int) { return true; }, pk_p,
                                                               pk_ds);
                    }
                    tmem_st32(sb + h * 32, pk_ds);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[b]);
            }
            if (!ok) break;
            gs += static_cast<uint32_t>(n);
        }
        teardown();
    }
}

}  // namespace attn

#include "attn_bwd_wide.cuh"

namespace attn {

// ============================================================== launch
// The key-side kernels of one backward call: attn_bwd_dkdv_kernel for
// d <= 128; the two passes of attn_bwd_wide_kernel (dV, then dK) for d = 256.
template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_key_side(const BwdArgs& a, cudaStream_t stream, long long op_bytes,
                            long long group_bytes) {
    cudaError_t err;
    const int bh_kv = a.BH / a.kv_group;
    const int hg_kv = static_cast<int>(
        std::max<long long>(1, group_bytes / (op_bytes * a.S_q * a.kv_group)));
    if constexpr (D != 256) {
        using T = BwdTile<D>;
        auto kdkdv = attn_bwd_dkdv_kernel<D, BF16, CAUSAL>;
        static std::atomic<uint64_t> configured_dkdv{0};
        err = configure_once(configured_dkdv, a.device, [&]() {
            const cudaError_t e = cudaFuncSetAttribute(
                kdkdv, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
            return e != cudaSuccess ? e : check_launch_regs(kdkdv, T::LAUNCH_REGS);
        });
        if (err != cudaSuccess) return err;
        const int n_kt = (a.S_k + T::BU - 1) / T::BU;
        const long long units_kv = static_cast<long long>(bh_kv) * n_kt;
        if (units_kv > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        // Full attention: one CTA per unit (the work queue hands the units out);
        // causal: one persistent CTA per SM.
        kdkdv<<<static_cast<int>(CAUSAL ? std::min<long long>(units_kv, a.num_sms) : units_kv),
                T::THREADS, T::SMEM_BYTES,
                stream>>>(a.tm_k_fixed, a.tm_v_fixed, a.tm_q_step, a.tm_do_step, a.tm_dv_out,
                          a.tm_dk_out, a.lse2, a.delta, a.S_q, a.S_k, bh_kv, a.H, a.kv_group,
                          a.S_pad, hg_kv,
                          a.causal_off, a.scale, a.scale_log2, a.words, a.launch_dkdv,
                          a.budget_ns);
        return cudaGetLastError();
    } else {
        auto kdv = attn_bwd_wide_kernel<BF16, CAUSAL, kPassDV>;
        auto kdk = attn_bwd_wide_kernel<BF16, CAUSAL, kPassDK>;
        using TV = BwdWideTile<kPassDV>;
        using TK = BwdWideTile<kPassDK>;
        static std::atomic<uint64_t> configured_wide{0};
        err = configure_once(configured_wide, a.device, [&]() {
            cudaError_t e = cudaFuncSetAttribute(kdv, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 TV::SMEM_BYTES);
            if (e != cudaSuccess) return e;
            return cudaFuncSetAttribute(kdk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        TK::SMEM_BYTES);
        });
        if (err != cudaSuccess) return err;
        const int n_kt = (a.S_k + TV::BU - 1) / TV::BU;
        const long long units_kv = static_cast<long long>(bh_kv) * n_kt;
        if (units_kv > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        const int grid =
            static_cast<int>(CAUSAL ? std::min<long long>(units_kv, a.num_sms) : units_kv);
        kdv<<<grid, TV::THREADS, TV::SMEM_BYTES, stream>>>(
            a.tm_k_fixed, a.tm_v_fixed, a.tm_q_step, a.tm_do_step, a.lse2, a.delta,
            static_cast<uint16_t*>(a.dv), a.dv_lay, a.S_q, a.S_k, bh_kv, a.H, a.kv_group, a.S_pad,
            hg_kv, a.causal_off, 1.f, a.scale_log2, a.words, a.launch_dkdv, a.budget_ns);
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
        kdk<<<grid, TK::THREADS, TK::SMEM_BYTES, stream>>>(
            a.tm_k_fixed, a.tm_v_fixed, a.tm_q_step, a.tm_do_step, a.lse2, a.delta,
            static_cast<uint16_t*>(a.dk), a.dk_lay, a.S_q, a.S_k, bh_kv, a.H, a.kv_group, a.S_pad,
            hg_kv, a.causal_off, a.scale, a.scale_log2, a.words, a.launch_key2, a.budget_ns);
        return cudaGetLastError();
    }
}

template <int D, bool BF16, bool CAUSAL>
cudaError_t launch_attn_bwd(const BwdArgs& a, cudaStream_t stream) {
    // D and LSE·log2e into the padded workspace.
    const long long rows_pad = static_cast<long long>(a.BH) * a.S_pad;
    const long long rows_per_block = 8LL * prep_rows_per_warp<D>();
    const long long pblocks = (rows_pad + rows_per_block - 1) / rows_per_block;
    if (pblocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    attn_bwd_prep_kernel<D, BF16><<<static_cast<unsigned>(pblocks), 256, 0, stream>>>(
        static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dout), a.lse, a.lse2,
        a.delta, a.S_q, a.S_pad, rows_pad, a.H, a.o_lay, a.do_lay);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;

    // dQ and dK/dV only read what prep wrote: with a helper stream, the dQ
    // kernel forks off here and its CTAs take the SMs that the dK/dV kernel's
    // last units leave idle.
    cudaStream_t dq_stream = stream;
    if (a.aux_stream) {
        err = cudaEventRecord(a.ev_fork, stream);
        if (err == cudaSuccess) err = cudaStreamWaitEvent(a.aux_stream, a.ev_fork, 0);
        if (err != cudaSuccess) return err;
        dq_stream = a.aux_stream;
    }
    const long long op_bytes = 2LL * D * 2;   // per row of one head: two operands
    const long long group_bytes = 48LL << 20;

    err = launch_key_side<D, BF16, CAUSAL>(a, stream, op_bytes, group_bytes);
    if (err != cudaSuccess) return err;

    using TQ = DqTile<D>;
    auto kdq = attn_bwd_dq_kernel<D, BF16, CAUSAL>;
    static std::atomic<uint64_t> configured_dq{0};
    err = configure_once(configured_dq, a.device, [&]() {
        const cudaError_t e =
            cudaFuncSetAttribute(kdq, cudaFuncAttributeMaxDynamicSharedMemorySize, TQ::SMEM_BYTES);
        return e != cudaSuccess ? e : check_launch_regs(kdq, TQ::LAUNCH_REGS);
    });
    if (err != cudaSuccess) return err;
    const int n_qt = (a.S_q + TQ::BU - 1) / TQ::BU;
    const long long units_q = static_cast<long long>(a.BH) * n_qt;
    if (units_q > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int hg_q = static_cast<int>(std::max<long long>(1, group_bytes / (op_bytes * a.S_k)));
    kdq<<<static_cast<int>(CAUSAL ? std::min<long long>(units_q, a.num_sms) : units_q), TQ::THREADS,
          TQ::SMEM_BYTES,
          dq_stream>>>(a.tm_q_fixed, a.tm_do_fixed, D == 256 ? a.tm_k_step : a.tm_k_fixed,
                       D == 256 ? a.tm_v_step : a.tm_v_fixed, a.lse2, a.delta,
                    static_cast<uint16_t*>(a.dq), a.dq_lay, a.S_q, a.S_k, a.BH, a.H, a.kv_group,
                    a.S_pad, hg_q, a.causal_off, a.scale, a.scale_log2, a.words, a.launch_dq,
                    a.budget_ns);
    err = cudaGetLastError();
    if (err != cudaSuccess || !a.aux_stream) return err;
    err = cudaEventRecord(a.ev_join, a.aux_stream);
    if (err != cudaSuccess) return err;
    return cudaStreamWaitEvent(stream, a.ev_join, 0);
}

}  // namespace attn
