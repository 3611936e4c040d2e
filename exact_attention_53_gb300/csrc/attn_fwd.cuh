// Exact scaled-dot-product attention forward for sm_103a.
//
// What it computes (oxicuda-dnn 0.1.8 hopper.rs, doc comment of
// FlashAttention3Plan::generate_forward): per key/value tile, S = Q·Kᵀ, an
// online softmax with a running row maximum m and row sum l, causal masking of
// future keys, O_acc += P·V, and after the last tile O = O_acc / l together
// with the log-sum-exp m + log l.  The S_q × S_k score matrix never leaves the
// SM.
//
// How it maps onto Blackwell:
//   * A work unit is one (batch·head, query block); a query block is two
//     128-row query tiles for d = 64/128, one tile for d = 256.  One CTA runs
//     per SM and takes units from the hardware work queue (below).
//   * Warp roles: 4 softmax warps per query tile (one row per thread, the
//     warp's TMEM lane quarter), one TMA producer warp, one MMA-issuing warp
//     and one warp that issues the TMA stores of O.
//   * K and V tiles (128 keys × d, 128-byte swizzled) stream through an
//     NS-slot shared-memory ring, handed over with full/empty mbarriers.
//   * S = Q·Kᵀ and O += P·V are tcgen05.mma (M = 128, fp32 accumulate) into
//     tensor memory.  Softmax reads S with tcgen05.ld, writes P (fp16/bf16)
//     back over the upper half of the S columns with tcgen05.st, and the PV
//     MMA takes P straight from tensor memory.
//   * The running maximum used for exponentiation is only raised when a
//     tile's row sum of exponentials exceeds rescale_sum<BF16>() (2^20 for
//     bf16, 2^15 for fp16), i.e. when the scores have outgrown the maximum by
//     enough to matter for the range of the 16-bit P or of fp32; O and l
//     always share the same (possibly stale) maximum, so O / l and the
//     log-sum-exp are unchanged.  This skips almost all O rescales and the
//     per-element maximum tracking, without approximating anything.
//   * Causal: key tiles entirely above the diagonal are never loaded or
//     computed; only tiles that straddle it (or the ragged end of the keys)
//     take the masked path.  Query blocks are issued heaviest first.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "attn_launch.h"
#include "sm100.cuh"

namespace attn {

// Status bits written when a bounded wait runs out.
enum : unsigned int {
    kStatusProducer = 1u,
    kStatusMma = 2u,
    kStatusSoftmax = 4u,
    kStatusEpilogue = 8u,
    kStatusDrain = 16u,
};

// Largest row sum of one tile's exponentials that is kept without raising the
// running maximum.  Every p of the tile is at most that sum, and P goes to the
// P·V product as a 16-bit value: bf16 has fp32's exponent range, so 2^20 only
// keeps the fp32 sums well inside range; fp16 overflows above 65504, so its
// bound is 2^15 (a larger p would round to +inf in the packed P).
template <bool BF16>
__host__ __device__ constexpr float rescale_sum() {
    return BF16 ? 1048576.0f : 32768.0f;
}
constexpr float kLn2 = 0.693147180559945309f;



// Number of key tiles query tile t of a block starting at row q0 visits.
template <bool CAUSAL>
__device__ __forceinline__ int kv_tiles_for(int row_begin, int S_q, int S_k, int causal_off) {
    if (row_begin >= S_q) return 0;
    int n = (S_k + kBlockN - 1) / kBlockN;
    if (CAUSAL) {
        const int last_key = min(row_begin + kBlockM, S_q) - 1 + causal_off;
        n = min(n, last_key / kBlockN + 1);
    }
    return n;
}

// Row maximum of one 128-score row: 8 independent chains of 3-input maxima.
// MASKED: scores at c >= lim are excluded (they become −∞).  The masked and
// unmasked forms are separate instantiations so the unmasked path carries no
// per-element compare/select.
template <bool MASKED>
__device__ __forceinline__ float row_max128(float (&s)[128], int lim) {
    using namespace sm100;
    if (MASKED) {
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = c < lim ? s[c] : -INFINITY;
    }
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = fmaxf(s[2 * i], s[2 * i + 1]);
#pragma unroll
    for (int c = 16; c < 128; c += 16)
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = fmax3(a[i], s[c + i], s[c + 8 + i]);
    return fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
}

// p = 2^(s·scale_log2 − m) for one row, packed to 16-bit pairs in `pk`;
// returns Σ p (fp32).  Two lanes at a time on the packed fp32 pipe.
// MASKED: p = 0 for c >= lim.
template <bool MASKED, bool BF16>
__device__ __forceinline__ float exp_pack128(const float (&s)[128], int lim, float scale_log2,
                                             float neg_m, uint32_t (&pk)[64]) {
    using namespace sm100;
    const float2 sl2 = make_float2(scale_log2, scale_log2);
    const float2 nm = make_float2(neg_m, neg_m);
    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                     make_float2(0.f, 0.f)};
#pragma unroll
    for (int c = 0; c < 128; c += 2) {
        const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), sl2, nm);
        float p0 = ex2_approx(x.x);
        float p1 = ex2_approx(x.y);
        if (MASKED) {
            p0 = c < lim ? p0 : 0.f;
            p1 = c + 1 < lim ? p1 : 0.f;
        }
        acc[(c >> 1) & 3] = __fadd2_rn(acc[(c >> 1) & 3], make_float2(p0, p1));
        pk[c >> 1] = BF16 ? pack_bf16(p0, p1) : pack_f16(p0, p1);
    }
    const float2 a01 = __fadd2_rn(acc[0], acc[1]);
    const float2 a23 = __fadd2_rn(acc[2], acc[3]);
    const float2 t = __fadd2_rn(a01, a23);
    return t.x + t.y;
}

// Work unit L (one (batch·head, query block)) -> head and first query row.
// Full attention: the query blocks of one head are adjacent, so the units in
// flight at a time share a few heads' K/V in L2.  Causal: heads go in groups
// of `head_group` (sized so a group's K/V fits in L2) and within a group the
// heaviest query blocks of all its heads go first, which keeps the tail short.
template <bool CAUSAL, int ROWS_PER_UNIT>
__device__ __forceinline__ void unit_coords(int L, int BH, int n_qblk, int head_group, int& bh,
                                            int& q0) {
    int qblk;
    if (CAUSAL) {
        const int per_group = head_group * n_qblk;
        const int g = L / per_group;
        const int r = L - g * per_group;
        const int g0 = g * head_group;
        const int gsz = min(head_group, BH - g0);
        const int qi = r / gsz;
        bh = g0 + (r - qi * gsz);
        qblk = n_qblk - 1 - qi;
    } else {
        bh = L / n_qblk;
        qblk = L - bh * n_qblk;
    }
    q0 = qblk * ROWS_PER_UNIT;
}

// Persistent kernel over a hardware work queue.  The grid has one CTA per
// work unit, but only about one per SM ever starts: a running CTA does its own
// unit (blockIdx.x), then claims further units by cancelling CTAs that have
// not started yet (cluster launch control) and doing their work, until none
// is left.  Units are numbered heaviest first, so this is longest-first list
// scheduling with no counter in global memory.  Every mbarrier phase and the
// K/V ring position carry over from one unit to the next, so the next unit's
// Q load and first Q·Kᵀ overlap the current unit's last P·V and epilogue.
template <int D, bool BF16, bool CAUSAL, bool SPLIT>
__global__ void __launch_bounds__(KernelTile<D, SPLIT>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o,
                    float* __restrict__ lse_ptr, int S_q, int S_k, int BH, int n_qblk,
                    int head_group, float scale_log2_signed, DeviceWords* __restrict__ words,
                    unsigned long long launch, unsigned long long budget_ns,
                    int n_split, int kv_per_split, float* __restrict__ o_part,
                    float* __restrict__ lse_part, int H, int kv_group, int causal_off,
                    int pack) {
    using T = KernelTile<D, SPLIT>;
    using namespace sm100;
    constexpr int ROWS = T::BM * T::TILES;                 // query rows per unit

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* sQ = smem;
    uint8_t* sKV = sQ + T::TILES * T::Q_TILE_BYTES;
    uint8_t* sO = sKV + T::NS * T::KV_TILE_BYTES;           // O staging for TMA stores
    uint8_t* clc_resp = smem + T::TILE_BYTES;               // [CLC_SLOTS] 16-byte answers
    uint64_t* bars = reinterpret_cast<uint64_t*>(clc_resp + T::CLC_SLOTS * 16);
    uint64_t* q_full = bars;                 // Q of the current unit landed
    uint64_t* q_empty = q_full + 1;          // last Q·Kᵀ of the unit finished
    uint64_t* kv_full = q_empty + 1;
    uint64_t* kv_empty = kv_full + T::NS;
    uint64_t* s_full = kv_empty + T::NS;     // [2] S buffer b written
    uint64_t* p_full = s_full + 2;           // [2] P in buffer b written (+ O rescaled), per warp
    uint64_t* o_done = p_full + 2;           // [2] last P·V of tile t (TILES == 1: every P·V)
    uint64_t* drain = o_done + 2;            // every MMA of the CTA finished
    uint64_t* epi_bar = drain + 1;           // [2] O rows of tile t staged, per warp
    uint64_t* stage_free = epi_bar + 2;      // staging buffer read by its TMA store
    uint64_t* clc_full = stage_free + 1;     // [CLC_SLOTS] work-queue answer landed
    uint64_t* clc_empty = clc_full + T::CLC_SLOTS;  // [CLC_SLOTS] answer read by every consumer
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(clc_empty + T::CLC_SLOTS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    unsigned int* status = &words->status;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // The softmax folds the scale into its exponent and its running maximum,
    // which needs a non-negative factor.  A negative scale is applied as
    // |scale| on S = (−Q)·Kᵀ: the Q·Kᵀ MMA negates its A operand, an exact
    // sign flip, so max_j(scale·s_ij) is the maximum of the scores it writes.
    const bool neg_scale = scale_log2_signed < 0.f;
    const float scale_log2 = fabsf(scale_log2_signed);
    // SPLIT: every (head, query block) is cut into n_split work units along the
    // keys (kv_per_split key tiles each); each writes O/l in fp32 and its own
    // log-sum-exp to o_part / lse_part for attn_combine to merge.  With
    // pack > 1 (split only) a unit's query tile holds the S_q rows of all
    // `pack` query heads that share one key/value head (pack·S_q <= 128 rows),
    // so each K/V tile is read and multiplied once for the whole group.
    const bool packed = SPLIT && pack > 1;
    const int units_bh = packed ? BH / pack : BH;
    // Unit L -> unit head (query head, or key/value head when packed), first
    // query row, key tiles of each query tile, first key tile, split.
    auto unit_info = [&](int L, int& bh, int& q0, int& n0, int& n1, int& kb, int& sp) {
        sp = SPLIT ? L % n_split : 0;
        unit_coords<CAUSAL, ROWS>(SPLIT ? L / n_split : L, units_bh, n_qblk, head_group, bh, q0);
        n0 = kv_tiles_for<CAUSAL>(q0, S_q, S_k, causal_off);
        n1 = T::TILES == 2 ? kv_tiles_for<CAUSAL>(q0 + T::BM, S_q, S_k, causal_off) : 0;
        kb = 0;
        if (SPLIT) {
            kb = sp * kv_per_split;
            n0 = max(0, min(n0, kb + kv_per_split) - kb);
            n1 = max(0, min(n1, kb + kv_per_split) - kb);
        }
    };
    // (b·H + h) -> batch, query head and the key/value head it reads (heads
    // are grouped kv_group to one key/value head).
    auto heads_of = [&](int bh, int& b, int& h, int& hk) {
        if (packed) {                        // bh counts key/value heads; h = first query head
            const int H_kv = H / kv_group;
            b = bh / H_kv;
            hk = bh - b * H_kv;
            h = hk * kv_group;
        } else {
            b = bh / H;
            h = bh - b * H;
            hk = h / kv_group;
        }
    };
    // Units of this CTA: its own, then those the producer warp claims from
    // the hardware work queue.  Consumers (the softmax, MMA and, without
    // SPLIT, store warps) free each answer's slot once read.
    constexpr int CLC_CONSUMERS = T::SOFTMAX_WARPS + (SPLIT ? 1 : 2);
    constexpr int STORE_WARP = T::STORE_WARP;
    const WorkQueue<T::CLC_SLOTS> queue{clc_resp, clc_full, clc_empty};
    auto unit_at = [&](int r, int& L, unsigned int bit, bool consumer) -> int {
        return queue.unit(r, L, consumer, abort_flag, status, bit);
    };

    if (packed) {
        // Rows past pack·S_q of the query tile are never loaded; keep them zero
        // so their (unstored) scores stay finite.
        uint4* zq = reinterpret_cast<uint4*>(sQ);
        for (int i = threadIdx.x; i < T::TILES * T::Q_TILE_BYTES / 16; i += blockDim.x)
            zq[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < T::NS; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], 4);           // one arrival per softmax warp
            mbar_init(&o_done[b], 1);
            mbar_init(&epi_bar[b], 4);
        }
        mbar_init(drain, 1);
        mbar_init(stage_free, 1);
        for (int s = 0; s < T::CLC_SLOTS; ++s) {
            mbar_init(&clc_full[s], 1);
            mbar_init(&clc_empty[s], CLC_CONSUMERS);
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

    // Each branch below ends in its own copy of the teardown, so no code runs
    // under two different register budgets.
    auto teardown = [&]() {
        tc_fence_before();
        __syncthreads();
        if (warp == 0) {
            tc_fence_after();
            tmem_dealloc(tmem, T::TMEM_COLS);
            if (lane == 0) publish_abort(abort_flag, words, launch);
        }
    };

    if (warp >= T::SOFTMAX_WARPS) {
      if (T::TILES == 2) regs_shrink<T::AUX_REGS>();
      // Both aux roles run warp-uniform loops (waits on every lane); only the
      // TMA / MMA / commit instructions themselves are issued by one lane.
      if (warp == T::PRODUCER_WARP) {
        // ------------------------------------------------------------ TMA producer
        const bool leader = elect_one();
        if (leader) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_o);
        }
        __syncwarp();
        LaunchWatch watch(words, launch, budget_ns);
        int idx = 0;                          // K/V ring position, across units
        int uq = 0;                           // units started by this CTA
        int q_loads = 0;                      // Q loads issued
        bool ok = true;
        auto issue = [&](const CUtensorMap* map, int j, int hk, int b) {
            if (!ok) return;
            if ((idx & 7) == 0 && watch.stop(abort_flag, status)) {
                ok = false;
                return;
            }
            const int slot = idx % T::NS;
            ok = mbar_wait(&kv_empty[slot], ((idx / T::NS) & 1) ^ 1, abort_flag, status, kStatusProducer);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) return;
            if (leader) {
                mbar_arrive_expect_tx(&kv_full[slot], T::KV_TILE_BYTES);
                uint8_t* dst = sKV + slot * T::KV_TILE_BYTES;
#pragma unroll
                for (int c = 0; c < T::CHUNKS; ++c)
                    tma_load_4d(dst + c * T::KV_CHUNK_BYTES, map, &kv_full[slot], c * 64,
                                j * T::BN, hk, b);
            }
            __syncwarp();
            ++idx;
        };
        int claims = 0;                       // work-queue requests issued
        for (int r = 0; ok; ++r) {
            if (watch.stop(abort_flag, status)) break;
            int L = 0;
            const int got = unit_at(r, L, kStatusProducer, false);
            if (got < 0) ok = false;
            if (got <= 0) break;
            int bh, q0, n0, n1, kb, sp, b, h, hk;
            unit_info(L, bh, q0, n0, n1, kb, sp);
            heads_of(bh, b, h, hk);
#ifdef ATTN_DEBUG_FAULTS
            // Debug builds only: load nothing for the chosen unit and stop, so
            // its consumers' waits run out.
            if (L == g_attn_debug_skip_unit) break;
#endif
            const int n_max = max(n0, n1);
            const int uq_now = uq++;
            // Q of this unit once the previous unit's last Q·Kᵀ is done.
            ok = mbar_wait(q_empty, (uq_now & 1) ^ 1, abort_flag, status, kStatusProducer);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            if (leader) {
                if (packed) {
                    // one box of S_q rows × pack heads per 64-column chunk
                    mbar_arrive_expect_tx(q_full, T::CHUNKS * S_q * pack * 128);
                    for (int c = 0; c < T::CHUNKS; ++c)
                        tma_load_4d(sQ + c * T::Q_CHUNK_BYTES, &tm_q, q_full, c * 64, 0, h, b);
                } else {
                    mbar_arrive_expect_tx(q_full, T::TILES * T::Q_TILE_BYTES);
                    for (int t = 0; t < T::TILES; ++t)
                        for (int c = 0; c < T::CHUNKS; ++c)
                            tma_load_4d(sQ + (t * T::CHUNKS + c) * T::Q_CHUNK_BYTES, &tm_q,
                                        q_full, c * 64, q0 + t * T::BM, h, b);
                }
            }
            __syncwarp();
            ++q_loads;
            // K/V in the MMA warp's consumption order.
            if (T::TILES == 2) {
                for (int j = 0; j < n_max && ok; ++j) {
                    issue(&tm_k, kb + j, hk, b);
                    issue(&tm_v, kb + j, hk, b);
                }
            } else {
                issue(&tm_k, kb, hk, b);
                if (n_max > 1) issue(&tm_k, kb + 1, hk, b);
                for (int j = 0; j < n_max && ok; ++j) {
                    issue(&tm_v, kb + j, hk, b);
                    if (j + 2 < n_max) issue(&tm_k, kb + j + 2, hk, b);
                }
            }
            if (!ok) break;
            if (r == 0 && watch.launch_gave_up(abort_flag)) break;
            // Claim the next unit only now, with this unit's last loads in the
            // ring: a unit claimed earlier would wait behind this whole unit
            // while idle CTAs find the queue empty.
            ok = queue.claim(claims, leader, abort_flag, status, kStatusProducer);
        }
        if (*abort_flag && leader) {
            // Let every copy this CTA started land before it exits.
            const uint64_t t0 = global_timer_ns();
            for (int i = max(0, idx - T::NS); i < idx; ++i)
                drain_wait(&kv_full[i % T::NS], (i / T::NS) & 1, t0, status, kStatusDrain);
            if (q_loads > 0)
                drain_wait(q_full, static_cast<uint32_t>(q_loads - 1) & 1u, t0, status, kStatusDrain);
            queue.drain(claims, status, kStatusDrain);   // and the last work-queue answer
        }
        __syncwarp();
      } else if (warp == T::MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t id_s =
            idesc_f16(128, T::BN, BF16, false, false) | (neg_scale ? kIdescNegateA : 0u);
        constexpr uint32_t id_o = idesc_f16(128, D, BF16, false, true);
        const uint32_t q_base = smem_u32(sQ);
        const uint32_t kv_base = smem_u32(sKV);
        bool ok = true;
        int acq = 0;                          // K/V ring position, across units
        uint32_t pc0 = 0, pc1 = 0;            // P handoffs consumed per buffer
        int uq = 0;
        auto acquire = [&](int& slot) {
            if (!ok) return;
            slot = acq % T::NS;
            ok = mbar_wait(&kv_full[slot], (acq / T::NS) & 1, abort_flag, status, kStatusMma);
            ok = __all_sync(0xffffffffu, ok);
            ++acq;
            tc_fence_after();
        };
        auto wait_p = [&](int b) {
            if (!ok) return;
            ok = mbar_wait(&p_full[b], (b ? pc1 : pc0) & 1, abort_flag, status, kStatusMma);
            ok = __all_sync(0xffffffffu, ok);
            if (b) ++pc1; else ++pc0;
            tc_fence_after();
        };
        // Descriptors are built once; a K step moves the start address, which
        // lives in the low 14 bits of the low word (addr >> 4, < 2^14 for any
        // shared-memory address), so stepping is a 32-bit add without carries.
        const uint64_t qk_desc = sdesc_sw128(q_base, 16, 1024);
        const uint64_t kk_desc = sdesc_sw128(kv_base, 16, 1024);
        const uint64_t v_desc = sdesc_sw128(kv_base, T::KV_CHUNK_BYTES, 1024);
        const uint32_t q_lo = static_cast<uint32_t>(qk_desc);
        const uint32_t q_hi = static_cast<uint32_t>(qk_desc >> 32);
        const uint32_t k_lo = static_cast<uint32_t>(kk_desc);
        const uint32_t k_hi = static_cast<uint32_t>(kk_desc >> 32);
        const uint32_t v_lo = static_cast<uint32_t>(v_desc);
        const uint32_t v_hi = static_cast<uint32_t>(v_desc >> 32);
        // S_b = Q_t · K(slot)ᵀ : M = 128, N = BN, K = D in steps of 16
        auto mma_qk = [&](int t, int slot, int b) {
            const uint32_t qa = q_lo + ((t * T::Q_TILE_BYTES) >> 4);
            const uint32_t ka = k_lo + ((slot * T::KV_TILE_BYTES) >> 4);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * T::Q_CHUNK_BYTES + (kk & 3) * 32) >> 4;
                const uint32_t koff = ((kk >> 2) * T::KV_CHUNK_BYTES + (kk & 3) * 32) >> 4;
                mma_ss_warp(tmem + b * T::S_STRIDE, qa + off, q_hi, ka + koff, k_hi, id_s,
                            kk > 0 ? 1u : 0u);
            }
        };
        // O_t (+)= P_b · V(slot) : M = 128, N = D, K = BN in steps of 16
        auto mma_pv = [&](int t, int slot, int b, bool acc) {
            const uint32_t va = v_lo + ((slot * T::KV_TILE_BYTES) >> 4);
            const uint32_t pa = tmem + b * T::S_STRIDE + T::P_OFF;
            const uint32_t oa = tmem + T::O_COL + t * D;
#pragma unroll
            for (int kk = 0; kk < T::BN / 16; ++kk) {
                mma_ts_warp(oa, pa + kk * 8, va + ((kk * 16 * 128) >> 4), v_hi, id_o,
                            (acc || kk > 0) ? 1u : 0u);
            }
        };
        int gs = 0;                           // TILES == 1: S/PV steps across units
        for (int r = 0; ok; ++r) {
            int L = 0;
            const int got = unit_at(r, L, kStatusMma, true);
            if (got < 0) ok = false;
            if (got <= 0) break;
            int bh, q0, n0, n1, kb, sp;
            unit_info(L, bh, q0, n0, n1, kb, sp);
            const int n_max = max(n0, n1);
            ok = mbar_wait(q_full, uq & 1, abort_flag, status, kStatusMma);
            ++uq;
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            if (!ok) break;
            if (T::TILES == 2) {
                int kslot = 0, vslot = 0;
                acquire(kslot);
                if (!ok) break;
                if (n0 > 0) { mma_qk(0, kslot, 0); tc_commit_warp(&s_full[0]); }
                if (n1 > 0) { mma_qk(1, kslot, 1); tc_commit_warp(&s_full[1]); }
                tc_commit_warp(&kv_empty[kslot]);
                if (n_max == 1) tc_commit_warp(q_empty);
                for (int j = 0; j < n_max && ok; ++j) {
                    const bool has_next = j + 1 < n_max;
                    acquire(vslot);
                    if (j < n0) {
                        wait_p(0);
                        if (!ok) break;
                        mma_pv(0, vslot, 0, j > 0);
                        if (j == n0 - 1) tc_commit_warp(&o_done[0]);
                    }
                    if (has_next) acquire(kslot);
                    if (!ok) break;
                    if (j + 1 < n0) { mma_qk(0, kslot, 0); tc_commit_warp(&s_full[0]); }
                    if (j < n1) {
                        wait_p(1);
                        if (!ok) break;
                        mma_pv(1, vslot, 1, j > 0);
                        if (j == n1 - 1) tc_commit_warp(&o_done[1]);
                    }
                    tc_commit_warp(&kv_empty[vslot]);
                    if (j + 1 < n1) { mma_qk(1, kslot, 1); tc_commit_warp(&s_full[1]); }
                    if (has_next) tc_commit_warp(&kv_empty[kslot]);
                    if (j + 2 == n_max) tc_commit_warp(q_empty);   // last Q·Kᵀ issued
                }
            } else {
                const int n = n0;
                int slot = 0;
                acquire(slot);
                if (!ok) break;
                mma_qk(0, slot, gs & 1);
                tc_commit_warp(&s_full[gs & 1]);
                tc_commit_warp(&kv_empty[slot]);
                if (n > 1) {
                    acquire(slot);
                    if (!ok) break;
                    mma_qk(0, slot, (gs + 1) & 1);
                    tc_commit_warp(&s_full[(gs + 1) & 1]);
                    tc_commit_warp(&kv_empty[slot]);
                }
                if (n <= 2) tc_commit_warp(q_empty);
                for (int j = 0; j < n && ok; ++j) {
                    const int b = (gs + j) & 1;
                    int vslot = 0;
                    acquire(vslot);
                    wait_p(b);
                    if (!ok) break;
                    mma_pv(0, vslot, b, j > 0);
                    tc_commit_warp(&o_done[0]);
                    tc_commit_warp(&kv_empty[vslot]);
                    if (j + 2 < n) {
                        acquire(slot);
                        if (!ok) break;
                        mma_qk(0, slot, b);
                        tc_commit_warp(&s_full[b]);
                        tc_commit_warp(&kv_empty[slot]);
                        if (j + 3 == n) tc_commit_warp(q_empty);
                    }
                }
                gs += n;
            }
        }
        // Every MMA of this CTA has finished once `drain` flips.
        tc_commit_warp(drain);
        const uint32_t a = smem_u32(drain);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(a, 0)) {
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                if (elect_one()) {
                    *abort_flag = 1;
                    atomicOr(status, kStatusDrain);
                }
                break;
            }
        }
        __syncwarp();
      } else if (warp == STORE_WARP && !SPLIT) {
        // ------------------------------------------------------------ O stores
        // Stores each staged round of O with TMA and frees the staging buffer
        // once the copy has read it, so the softmax warps never wait on a store.
        bool ok = true;
        uint32_t ph[2] = {0, 0};
        bool stored = false;
        for (int r = 0; ok; ++r) {
            int L = 0;
            const int got = unit_at(r, L, kStatusEpilogue, true);
            if (got < 0) ok = false;
            if (got <= 0) break;
            int bh, q0, n0, n1, kb, sp;
            unit_info(L, bh, q0, n0, n1, kb, sp);
            for (int t = 0; t < T::TILES && ok; ++t) {
                if ((t == 0 ? n0 : n1) <= 0) continue;
                for (int rr = 0; rr < T::STAGE_ROUNDS; ++rr) {
                    ok = mbar_wait(&epi_bar[t], ph[t] & 1, abort_flag, status, kStatusEpilogue);
                    ok = __all_sync(0xffffffffu, ok);
                    ++ph[t];
                    if (!ok) break;
                    if (elect_one()) {
                        for (int c = 0; c < T::STAGE_CHUNKS; ++c)
                            tma_store_4d(&tm_o, sO + c * T::Q_CHUNK_BYTES,
                                         (rr * T::STAGE_CHUNKS + c) * 64, q0 + t * T::BM, bh % H,
                                         bh / H);
                        bulk_commit_group();
                        bulk_wait_read_all();
                        mbar_arrive(stage_free);
                        stored = true;
                    }
                    __syncwarp();
                }
            }
        }
        if (stored) bulk_wait_all();
        __syncwarp();
      }
      teardown();
    } else {
        if (T::TILES == 2) regs_grow<T::SOFTMAX_REGS>();
        // ------------------------------------------------------------ softmax warps
        const int t = T::TILES == 2 ? (warp >> 2) : 0;
        const int wq = warp & 3;                      // TMEM lane quarter of this warp
        const int row = wq * 32 + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
        bool ok = true;
        uint32_t sc = 0;                              // S tiles consumed by this warpgroup
        uint32_t oc = 0;                              // o_done phases consumed
        uint32_t round = 0;                           // staging rounds of the whole CTA

        for (int r = 0; ok; ++r) {
            int L = 0;
            const int got = unit_at(r, L, kStatusSoftmax, true);
            if (got < 0) ok = false;
            if (got <= 0) break;
            int bh, q0, n0, n1, kb, sp;
            unit_info(L, bh, q0, n0, n1, kb, sp);
            const int n = t == 0 ? n0 : n1;
            const int row_begin = q0 + t * T::BM;
            const int q_idx = row_begin + row;
            float m = -INFINITY;                      // running max, log2 units (scale folded)
            float l = 0.f;                            // running sum of exp2(x - m)

            for (int j = 0; j < n; ++j) {
                // TILES == 2: S buffer t, one S per step.  TILES == 1: the two
                // buffers alternate; sc counts steps across units.
                const int b = T::TILES == 2 ? t : static_cast<int>(sc & 1);
                const uint32_t parity = T::TILES == 2 ? (sc & 1) : ((sc >> 1) & 1);
                ok = mbar_wait(&s_full[b], parity, abort_flag, status, kStatusSoftmax);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                ++sc;

                uint32_t sa[64], sb[64];
                tmem_ld64x2(lane_base + b * T::S_STRIDE, lane_base + b * T::S_STRIDE + 64, sa, sb);
                float s[128];
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    s[c] = __uint_as_float(sa[c]);
                    s[64 + c] = __uint_as_float(sb[c]);
                }

                const int kv0 = (kb + j) * T::BN;
                const bool masked =
                    (CAUSAL && kv0 + T::BN - 1 > row_begin + causal_off) || (kv0 + T::BN > S_k);
                // keys kv0 + c with c < lim are visible to this row
                const int lim =
                    masked ? max(0, min(S_k, CAUSAL ? q_idx + 1 + causal_off : S_k) - kv0) : T::BN;

                uint32_t pk[64];
                bool rescale = false;
                float alpha = 1.f;
                if (m == -INFINITY) {
                    // First visible tile of this row: the maximum has to come first.
                    const float mx = masked ? row_max128<true>(s, lim) : row_max128<false>(s, lim);
                    m = (mx == -INFINITY) ? -INFINITY : mx * scale_log2;
                    const float neg_m = (m == -INFINITY) ? 0.f : -m;
                    l = masked ? exp_pack128<true, BF16>(s, lim, scale_log2, neg_m, pk)
                               : exp_pack128<false, BF16>(s, lim, scale_log2, neg_m, pk);
                } else {
                    // Exponentiate against the running maximum.  A row whose sum of
                    // exponentials exceeds rescale_sum (its scores outgrew the
                    // maximum; rare) re-reads its scores from TMEM (P has not been
                    // written over them yet) and is redone against its new maximum.
                    // Either way O and l share one maximum, so the result is exact.
                    float lsum = masked
                        ? exp_pack128<true, BF16>(s, lim, scale_log2, -m, pk)
                        : exp_pack128<false, BF16>(s, lim, scale_log2, -m, pk);
                    const bool grow = !(lsum <= rescale_sum<BF16>());   // also catches inf and NaN
                    if (__any_sync(0xffffffffu, grow)) {
                        uint32_t ra[64], rb[64];
                        tmem_ld64x2(lane_base + b * T::S_STRIDE, lane_base + b * T::S_STRIDE + 64,
                                    ra, rb);
                        if (grow) {
#pragma unroll
                            for (int c = 0; c < 64; ++c) {
                                s[c] = __uint_as_float(ra[c]);
                                s[64 + c] = __uint_as_float(rb[c]);
                            }
                            const float mx = masked ? row_max128<true>(s, lim) : row_max128<false>(s, lim);
                            const float m_new = fmaxf(m, mx * scale_log2);
                            alpha = ex2_approx(m - m_new);
                            m = m_new;
                            l *= alpha;
                            rescale = true;
                            lsum = masked
                                ? exp_pack128<true, BF16>(s, lim, scale_log2, -m, pk)
                                : exp_pack128<false, BF16>(s, lim, scale_log2, -m, pk);
                        }
                    }
                    l += lsum;
                }

                tmem_st32(lane_base + b * T::S_STRIDE + T::P_OFF, pk);
                tmem_st32(lane_base + b * T::S_STRIDE + T::P_OFF + 32, pk + 32);

                if (T::TILES == 1 && j > 0) {
                    // O holds PV up to key tile j-1 only once that MMA has finished.
                    ok = mbar_wait(&o_done[0], oc & 1, abort_flag, status, kStatusSoftmax);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    ++oc;
                    tc_fence_after();
                }
                if (__any_sync(0xffffffffu, rescale)) {
                    const uint32_t o_base = lane_base + T::O_COL + t * D;
#pragma unroll 1
                    for (int cc = 0; cc < D; cc += 32) {
                        uint32_t r[32];
                        tmem_ld32(o_base + cc, r);
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st32(o_base + cc, r);
                    }
                }
                // Each lane's TMEM stores are complete (wait::st) and fenced; after the
                // warp converges one lane publishes them for the whole warp.
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[b]);
            }
            if (!ok) break;

            // ---------------------------------------------------------- epilogue
            if (SPLIT) {
                // Partial result of this key range: O/l in fp32 and its LSE.
                if (n > 0) {
                    ok = mbar_wait(&o_done[t], oc & 1, abort_flag, status, kStatusEpilogue);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    ++oc;
                    tc_fence_after();
                    const float inv_l = 1.f / l;
                    bool store = q_idx < S_q;
                    size_t prow = (static_cast<size_t>(sp) * BH + bh) * S_q + q_idx;
                    if (packed) {
                        // row = (query head within the group) · S_q + query
                        int b_, h_, hk_;
                        heads_of(bh, b_, h_, hk_);
                        const int hl = row / S_q;
                        store = row < S_q * pack;
                        prow = (static_cast<size_t>(sp) * BH + static_cast<size_t>(b_) * H + h_ + hl) *
                                   S_q + (row - hl * S_q);
                    }
                    float4* dst = reinterpret_cast<float4*>(o_part + prow * D);
                    const uint32_t o_base = lane_base + T::O_COL + t * D;
#pragma unroll 1
                    for (int cc = 0; cc < D; cc += 32) {
                        uint32_t v[32];
                        tmem_ld32(o_base + cc, v);
                        if (store) {
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                dst[cc / 4 + i] = make_float4(__uint_as_float(v[4 * i]) * inv_l,
                                                              __uint_as_float(v[4 * i + 1]) * inv_l,
                                                              __uint_as_float(v[4 * i + 2]) * inv_l,
                                                              __uint_as_float(v[4 * i + 3]) * inv_l);
                        }
                    }
                    if (store) lse_part[prow] = (m + log2f(l)) * kLn2;
                }
                continue;
            }
            // Rounds of the staging buffer run in a fixed order over the CTA:
            // tile 0's then tile 1's, unit after unit.
            const uint32_t rounds_t0 = n0 > 0 ? T::STAGE_ROUNDS : 0;
            const uint32_t rounds_t1 = (T::TILES == 2 && n1 > 0) ? T::STAGE_ROUNDS : 0;
            if (n > 0) {
                const uint32_t parity = T::TILES == 2 ? (oc & 1) : (oc & 1);
                ok = mbar_wait(&o_done[t], parity, abort_flag, status, kStatusEpilogue);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                ++oc;
                tc_fence_after();
                const float inv_l = 1.f / l;
                const uint32_t o_base = lane_base + T::O_COL + t * D;
                uint32_t r_idx = round + (t == 1 ? rounds_t0 : 0);
                for (int rr = 0; rr < T::STAGE_ROUNDS; ++rr, ++r_idx) {
                    // The staging buffer is free once the previous round's TMA store
                    // has read it.
                    if (r_idx > 0) {
                        ok = mbar_wait(stage_free, (r_idx - 1) & 1, abort_flag, status,
                                       kStatusEpilogue);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                    }
#pragma unroll 1
                    for (int cc = 0; cc < T::STAGE_CHUNKS * 64; cc += 32) {
                        uint32_t r[32];
                        tmem_ld32(o_base + rr * T::STAGE_CHUNKS * 64 + cc, r);
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float a = __uint_as_float(r[2 * i]) * inv_l;
                            const float c = __uint_as_float(r[2 * i + 1]) * inv_l;
                            w[i] = BF16 ? pack_bf16(a, c) : pack_f16(a, c);
                        }
                        uint8_t* rowp = sO + (cc / 64) * T::Q_CHUNK_BYTES + row * 128;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int unit = ((cc & 63) / 8) + i;      // 16-byte unit in the row
                            *reinterpret_cast<uint4*>(rowp + ((unit ^ (row & 7)) * 16)) =
                                make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                        }
                    }
                    // Every warp publishes its rows; the store warp issues the round's
                    // TMA store once all four have.
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&epi_bar[t]);
                    if (!ok) break;
                }
                if (!ok) break;
                if (q_idx < S_q)
                    lse_ptr[static_cast<size_t>(bh) * S_q + q_idx] = (m + log2f(l)) * kLn2;
            }
            round += rounds_t0 + rounds_t1;
        }
        teardown();
    }
}

template <int D, bool BF16, bool CAUSAL, bool SPLIT>
cudaError_t launch_attn_fwd(const FwdArgs& a, cudaStream_t stream) {
    using T = KernelTile<D, SPLIT>;
    static_assert(!(SPLIT && CAUSAL), "split-KV is built for full attention only");
    auto kernel = attn_fwd_kernel<D, BF16, CAUSAL, SPLIT>;
    static std::atomic<uint64_t> configured{0};
    cudaError_t err = configure_once(configured, a.device, [&]() {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             T::SMEM_BYTES);
        if (e != cudaSuccess || T::TILES != 2) return e;
        // The warpgroup register split assumes the launch grants LAUNCH_REGS a
        // thread; refuse to launch a build where it does not (it would stall).
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return e;
        return fa.numRegs == T::LAUNCH_REGS ? cudaSuccess : cudaErrorInvalidConfiguration;
    });
    if (err != cudaSuccess) return err;
    int head_group = 1;
    if (CAUSAL) {
        const long long kv_head_bytes = 2LL * a.S_k * D * 2;
        const long long budget = 48LL << 20;
        head_group = static_cast<int>(std::max(1LL, std::min<long long>(a.BH, budget / kv_head_bytes)));
    }
    const int rows_per_cta = T::BM * T::TILES;
    const int n_qblk = (a.S_q + rows_per_cta - 1) / rows_per_cta;
    const int n_split = SPLIT ? a.n_split : 1;
    const int pack = SPLIT ? a.pack : 1;
    const long long units = static_cast<long long>(a.BH / pack) * n_qblk * n_split;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // One CTA per unit; each takes the whole of tensor memory and most of shared
    // memory, so one runs per SM and the running ones cancel and take over the rest.
    const int grid = static_cast<int>(units);
    kernel<<<grid, T::THREADS, T::SMEM_BYTES, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.lse, a.S_q,
                                                         a.S_k, a.BH, n_qblk, head_group,
                                                         a.scale_log2, a.words, a.launch,
                                                         a.budget_ns, n_split,
                                                         a.kv_per_split, a.o_part, a.lse_part, a.H,
                                                         a.kv_group, a.causal_off, pack);
    return cudaGetLastError();
}

}  // namespace attn
