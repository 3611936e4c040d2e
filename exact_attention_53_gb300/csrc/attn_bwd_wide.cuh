// Key-side backward for head_dim 256 (dV and dK), in two passes.
//
// The steps are those of the page's backward (oxicuda-dnn 0.1.8 hopper.rs,
// doc comment of generate_backward), as in attn_bwd.cuh: P recomputed from the
// forward's log-sum-exp, dV = Pᵀ·dO, dP = dO·Vᵀ, dS = P ∘ (dP − D),
// dK = dSᵀ·Q (times the scale).  At d = 256 the two accumulators dV and dK of a
// 128-key unit take 2 × 256 columns, all of tensor memory, and leave none for
// Sᵀ and dPᵀ; so each accumulator gets a pass of its own over the same units
// and steps, each recomputing Sᵀ = K·Qᵀ:
//
//   PASS_DV  K fixed; per 64-query step Sᵀ, Pᵀ by the softmax warps,
//            dV += Pᵀ·dO                              (tensor memory: Sᵀ[2], dV)
//   PASS_DK  K and V fixed; per step Sᵀ and dPᵀ = V·dOᵀ, dSᵀ by the softmax
//            warps, dK += dSᵀ·Q                        (Sᵀ[2], dPᵀ[2], dK)
//
// Q and dO stream through rings of their own (32 KB a 64-row step each): a dO
// slot is free as soon as the MMA that last reads it is done, a Q slot (which
// also carries the step's LSE·log2e and D rows) once the softmax warps have read
// those and the accumulating MMA is done.  Units, their order, causal
// skipping, grouped key/value heads, bounded waits and the launch watch are
// those of attn_bwd_dkdv_kernel.
#pragma once

namespace attn {

enum : int { kPassDV = 0, kPassDK = 1 };

template <int PASS>
struct BwdWideTile {
    static constexpr int D = 256;
    static constexpr int BU = 128;                    // keys per unit
    static constexpr int BS = 64;                     // query rows per step
    static constexpr int CHUNKS = D / 64;             // 128-byte swizzle atoms along d
    static constexpr int BIG_CHUNK = BU * 128;        // one atom column of a 128-row tile
    static constexpr int SMALL_CHUNK = BS * 128;      // of a 64-row tile
    static constexpr int BIG_TILE = BU * D * 2;       // 64 KB
    static constexpr int SMALL_TILE = BS * D * 2;     // 32 KB
    static constexpr int FIXED = PASS == kPassDK ? 2 : 1;        // K (and V)
    // Q ring slots: a Q slot is held from its step's Sᵀ (issued two steps
    // ahead) until the softmax warps have read its statistics, so with two
    // slots every Sᵀ waited for its Q to arrive; the dV pass has room for a
    // third (dV pass at B=2, H=8, S=8192: 1.40 → 0.84 ms), the dK pass (K and
    // V fixed) not.
    static constexpr int NQ = PASS == kPassDK ? 2 : 3;
    static constexpr int NO = PASS == kPassDK ? 1 : 2;           // dO ring slots
    static constexpr int STAT_FLOATS = 2 * BS;        // per Q slot: LSE·log2e and D of 64 rows
    static constexpr int CLC_SLOTS = 4;
    static constexpr int NUM_BARS = 2 + 2 * NQ + 2 * NO + 2 + 2 + 1 + 1 + 2 * CLC_SLOTS;
    static constexpr int TILE_BYTES =
        FIXED * BIG_TILE + (NQ + NO) * SMALL_TILE + NQ * STAT_FLOATS * 4;
    static constexpr int SMEM_BYTES = 1024 + TILE_BYTES + CLC_SLOTS * 16 + NUM_BARS * 8 + 16;
    static constexpr int THREADS = 192;               // 4 softmax warps, producer, MMA
    static constexpr int PRODUCER_WARP = 4;
    static constexpr int MMA_WARP = 5;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 0;              // Sᵀ buffer b at 64·b (fp32)
    static constexpr uint32_t DP_COL = 128;           // dPᵀ buffer b at 128 + 64·b (PASS_DK)
    static constexpr uint32_t PK_OFF = 32;            // packed 16-bit Pᵀ / dSᵀ over cols 32..63
    static constexpr uint32_t ACC_COL = 256;          // dV or dK: 256 columns
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(ACC_COL + D <= TMEM_COLS, "tensor memory budget");
};

// p = 2^(s·scale·log2e − LSE₂[c]) for 64 columns (0 where masked), packed as
// 16-bit pairs; LSE₂ per column from shared memory.
template <bool MASKED, bool BF16, typename Keep>
__device__ __forceinline__ void prob_pack64(const uint32_t (&s)[64], const float* lse2,
                                            float scale_log2, Keep keep, uint32_t (&pk)[32]) {
    using namespace sm100;
    const float2 sl2 = make_float2(scale_log2, scale_log2);
#pragma unroll
    for (int c = 0; c < 64; c += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(lse2 + c);
        const float2 nl[2] = {make_float2(-l4.x, -l4.y), make_float2(-l4.z, -l4.w)};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int cc = c + 2 * i;
            const float2 x = __ffma2_rn(
                make_float2(__uint_as_float(s[cc]), __uint_as_float(s[cc + 1])), sl2, nl[i]);
            float p0 = ex2_approx(x.x);
            float p1 = ex2_approx(x.y);
            if (MASKED) {
                p0 = keep(cc) ? p0 : 0.f;
                p1 = keep(cc + 1) ? p1 : 0.f;
            }
            pk[cc / 2] = BF16 ? pack_bf16(p0, p1) : pack_f16(p0, p1);
        }
    }
}

template <bool BF16, bool CAUSAL, int PASS>
__global__ void __launch_bounds__(BwdWideTile<PASS>::THREADS, 1)
    attn_bwd_wide_kernel(const __grid_constant__ CUtensorMap tm_k,    // box 64 × 128
                         const __grid_constant__ CUtensorMap tm_v,    // box 64 × 128 (PASS_DK)
                         const __grid_constant__ CUtensorMap tm_q,    // box 64 × 64
                         const __grid_constant__ CUtensorMap tm_do,   // box 64 × 64
                         const float* __restrict__ lse2, const float* __restrict__ delta,
                         uint16_t* __restrict__ out, RowLayout out_lay, int S_q, int S_k,
                         int BHkv, int H, int kv_group, int S_pad, int head_group,
                         int causal_off, float out_scale, float scale_log2,
                         DeviceWords* __restrict__ words, unsigned long long launch,
                         unsigned long long budget_ns) {
    using T = BwdWideTile<PASS>;
    constexpr int D = T::D;
    constexpr bool DK = PASS == kPassDK;
    using namespace sm100;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t* sK = smem;
    uint8_t* sV = sK + T::BIG_TILE;                   // PASS_DK only
    uint8_t* sQ = sK + T::FIXED * T::BIG_TILE;        // Q ring
    uint8_t* sO = sQ + T::NQ * T::SMALL_TILE;         // dO ring
    float* sStat = reinterpret_cast<float*>(sO + T::NO * T::SMALL_TILE);
    uint8_t* clc_resp = smem + T::TILE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(clc_resp + T::CLC_SLOTS * 16);
    uint64_t* kv_full = bars;                 // fixed K (and V) of the unit landed
    uint64_t* kv_empty = kv_full + 1;         // last MMA reading them finished
    uint64_t* q_full = kv_empty + 1;          // [NQ]
    uint64_t* q_empty = q_full + T::NQ;       // [NQ]
    uint64_t* o_full = q_empty + T::NQ;       // [NO]
    uint64_t* o_empty = o_full + T::NO;       // [NO]
    uint64_t* s_full = o_empty + T::NO;       // [2] Sᵀ (and dPᵀ) of buffer b computed
    uint64_t* p_full = s_full + 2;            // [2] Pᵀ or dSᵀ of buffer b written (per warp)
    uint64_t* acc_done = p_full + 2;
    uint64_t* drain = acc_done + 1;
    uint64_t* clc_full = drain + 1;
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
    auto unit_info = [&](int L, int& b, int& hk, int& kt, int& q_begin, int& n) {
        int bhk;
        bwd_unit_coords<CAUSAL, true>(L, BHkv, n_kt, head_group, bhk, kt);
        b = bhk / H_kv;
        hk = bhk - b * H_kv;
        q_begin = CAUSAL ? min(n_qs, max(0, kt * T::BU - causal_off) / T::BS) : 0;
        n = (n_qs - q_begin) * kv_group;
    };
    auto next_step = [&](int q_begin, int& h, int& qi) {
        if (++qi == n_qs) {
            qi = q_begin;
            ++h;
        }
    };
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
        for (int s = 0; s < T::NQ; ++s) {
            mbar_init(&q_full[s], 1);
            mbar_init(&q_empty[s], 1);
        }
        for (int s = 0; s < T::NO; ++s) {
            mbar_init(&o_full[s], 1);
            mbar_init(&o_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], 4);
        }
        mbar_init(acc_done, 1);
        mbar_init(drain, 1);
        for (int s = 0; s < T::CLC_SLOTS; ++s) {
            mbar_init(&clc_full[s], 1);
            mbar_init(&clc_empty[s], 5);         // softmax warps 0-3 and the MMA warp
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

    if (warp == T::PRODUCER_WARP) {
        // ------------------------------------------------------------ TMA producer
        const bool leader = elect_one();
        if (leader) {
            tma_prefetch_desc(&tm_k);
            if (DK) tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_do);
        }
        __syncwarp();
        LaunchWatch watch(words, launch, budget_ns);
        bool ok = true;
        int qidx = 0, oidx = 0;   // ring positions, across units
        int uk = 0;               // units with work started by this CTA
        int claims = 0;
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
            if (n == 0) {
                claim_next();
                continue;
            }
            ok = mbar_wait(kv_empty, (uk & 1) ^ 1, abort_flag, status, kStatusBwdProducer);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ++uk;
            if (leader) {
                mbar_arrive_expect_tx(kv_full, T::FIXED * T::BIG_TILE);
#pragma unroll
                for (int c = 0; c < T::CHUNKS; ++c) {
                    tma_load_4d(sK + c * T::BIG_CHUNK, &tm_k, kv_full, c * 64, kt * T::BU, hk, b);
                    if (DK)
                        tma_load_4d(sV + c * T::BIG_CHUNK, &tm_v, kv_full, c * 64, kt * T::BU,
                                    hk, b);
                }
            }
            __syncwarp();
            int h = hk * kv_group, qi = q_begin;
            for (int t = 0; t < n && ok; ++t, next_step(q_begin, h, qi)) {
                if ((qidx & 7) == 0 && watch.stop(abort_flag, status)) {
                    ok = false;
                    break;
                }
                const int q0 = qi * T::BS;
                // Q and the step's LSE·log2e and D rows
                const int qs = qidx % T::NQ;
                ok = mbar_wait(&q_empty[qs], ((qidx / T::NQ) & 1) ^ 1, abort_flag, status,
                               kStatusBwdProducer);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                if (leader) {
                    float* st = sStat + qs * T::STAT_FLOATS;
                    const size_t soff = (static_cast<size_t>(b) * H + h) * S_pad + q0;
                    mbar_arrive_expect_tx(&q_full[qs], T::SMALL_TILE + T::STAT_FLOATS * 4);
#pragma unroll
                    for (int c = 0; c < T::CHUNKS; ++c)
                        tma_load_4d(sQ + qs * T::SMALL_TILE + c * T::SMALL_CHUNK, &tm_q,
                                    &q_full[qs], c * 64, q0, h, b);
                    bulk_load(st, lse2 + soff, T::BS * 4, &q_full[qs]);
                    bulk_load(st + T::BS, delta + soff, T::BS * 4, &q_full[qs]);
                }
                __syncwarp();
                ++qidx;
                // dO
                const int os = oidx % T::NO;
                ok = mbar_wait(&o_empty[os], ((oidx / T::NO) & 1) ^ 1, abort_flag, status,
                               kStatusBwdProducer);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                if (leader) {
                    mbar_arrive_expect_tx(&o_full[os], T::SMALL_TILE);
#pragma unroll
                    for (int c = 0; c < T::CHUNKS; ++c)
                        tma_load_4d(sO + os * T::SMALL_TILE + c * T::SMALL_CHUNK, &tm_do,
                                    &o_full[os], c * 64, q0, h, b);
                }
                __syncwarp();
                ++oidx;
            }
            if (!ok) break;
            if (uk == 1 && watch.launch_gave_up(abort_flag)) break;
            claim_next();
        }
        if (*abort_flag && leader) {
            // Let every copy this CTA started land before it exits.
            const uint64_t t0 = global_timer_ns();
            for (int i = max(0, qidx - T::NQ); i < qidx; ++i)
                drain_wait(&q_full[i % T::NQ], (i / T::NQ) & 1, t0, status, kStatusBwdDrain);
            for (int i = max(0, oidx - T::NO); i < oidx; ++i)
                drain_wait(&o_full[i % T::NO], (i / T::NO) & 1, t0, status, kStatusBwdDrain);
            if (uk > 0)
                drain_wait(kv_full, static_cast<uint32_t>(uk - 1) & 1u, t0, status,
                           kStatusBwdDrain);
            queue.drain(claims, status, kStatusBwdDrain);
        }
        __syncwarp();
    } else if (warp == T::MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t id_s = idesc_f16(128, T::BS, BF16, false, false);
        constexpr uint32_t id_acc = idesc_f16(128, D, BF16, false, true);
        const uint64_t k_desc = sdesc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t v_desc = sdesc_sw128(smem_u32(sV), 16, 1024);
        const uint64_t qk_desc = sdesc_sw128(smem_u32(sQ), 16, 1024);            // Q, K-major
        const uint64_t qm_desc = sdesc_sw128(smem_u32(sQ), T::SMALL_CHUNK, 1024); // Q, MN-major
        const uint64_t ok_desc = sdesc_sw128(smem_u32(sO), 16, 1024);            // dO, K-major
        const uint64_t om_desc = sdesc_sw128(smem_u32(sO), T::SMALL_CHUNK, 1024); // dO, MN-major
        const uint32_t k_lo = static_cast<uint32_t>(k_desc), k_hi = static_cast<uint32_t>(k_desc >> 32);
        const uint32_t v_lo = static_cast<uint32_t>(v_desc), v_hi = static_cast<uint32_t>(v_desc >> 32);
        const uint32_t qk_lo = static_cast<uint32_t>(qk_desc), qk_hi = static_cast<uint32_t>(qk_desc >> 32);
        const uint32_t qm_lo = static_cast<uint32_t>(qm_desc), qm_hi = static_cast<uint32_t>(qm_desc >> 32);
        const uint32_t ok_lo = static_cast<uint32_t>(ok_desc), ok_hi = static_cast<uint32_t>(ok_desc >> 32);
        const uint32_t om_lo = static_cast<uint32_t>(om_desc), om_hi = static_cast<uint32_t>(om_desc >> 32);
        bool ok = true;
        int qacq = 0, oacq = 0;      // ring positions, across units
        uint32_t gs = 0;             // steps issued, across units (S/dP buffer = step & 1)
        int uk = 0;
        auto acquire = [&](uint64_t* full, int slots, int& acq, int& slot) {
            if (!ok) return;
            slot = acq % slots;
            ok = mbar_wait(&full[slot], (acq / slots) & 1, abort_flag, status, kStatusBwdMma);
            ok = __all_sync(0xffffffffu, ok);
            ++acq;
            tc_fence_after();
        };
        // Sᵀ_b = K·Q_qsᵀ (and dPᵀ_b = V·dO_osᵀ): M = 128 keys, N = 64 queries, K = 256
        auto mma_s = [&](int qs, int os, int b) {
            const uint32_t qoff = (qs * T::SMALL_TILE) >> 4;
            const uint32_t ooff = (os * T::SMALL_TILE) >> 4;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t ao = ((kk >> 2) * T::BIG_CHUNK + (kk & 3) * 32) >> 4;
                const uint32_t bo = ((kk >> 2) * T::SMALL_CHUNK + (kk & 3) * 32) >> 4;
                mma_ss_warp(tmem + T::S_COL + b * 64, k_lo + ao, k_hi, qk_lo + qoff + bo, qk_hi,
                            id_s, kk > 0 ? 1u : 0u);
                if (DK)
                    mma_ss_warp(tmem + T::DP_COL + b * 64, v_lo + ao, v_hi, ok_lo + ooff + bo,
                                ok_hi, id_s, kk > 0 ? 1u : 0u);
            }
        };
        // dV += Pᵀ_b·dO_os, or dK += dSᵀ_b·Q_qs: M = 128 keys, N = 256, K = 64 queries
        auto mma_acc = [&](int qs, int os, int b, bool acc) {
            const uint32_t a_col = DK ? T::DP_COL + b * 64 + T::PK_OFF : T::S_COL + b * 64 + T::PK_OFF;
            const uint32_t m_lo = DK ? qm_lo + ((qs * T::SMALL_TILE) >> 4)
                                     : om_lo + ((os * T::SMALL_TILE) >> 4);
            const uint32_t m_hi = DK ? qm_hi : om_hi;
#pragma unroll
            for (int kk = 0; kk < T::BS / 16; ++kk) {
                const uint32_t bo = (kk * 16 * 128) >> 4;
                mma_ts_warp(tmem + T::ACC_COL, tmem + a_col + kk * 8, m_lo + bo, m_hi, id_acc,
                            (acc || kk > 0) ? 1u : 0u);
            }
        };
        // Issue step s's Sᵀ (and dPᵀ) into buffer b; returns its ring slots.
        auto issue_s = [&](int b, int& qs, int& os) {
            acquire(q_full, T::NQ, qacq, qs);
            if (DK) acquire(o_full, T::NO, oacq, os);
            if (!ok) return;
            mma_s(qs, os, b);
            tc_commit_warp(&s_full[b]);
            if (DK) tc_commit_warp(&o_empty[os]);     // dO read by dPᵀ only
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
            int qs_cur = 0, os_cur = 0, qs_nxt = 0, os_nxt = 0;
            issue_s(gs & 1, qs_cur, os_cur);
            if (!ok) break;
            if (n > 1) {
                issue_s((gs + 1) & 1, qs_nxt, os_nxt);
                if (!ok) break;
            }
            if (n <= 2) tc_commit_warp(kv_empty);          // K (and V) no longer needed
            for (int t = 0; t < n && ok; ++t) {
                const int bb = static_cast<int>((gs + t) & 1);
                ok = mbar_wait(&p_full[bb], (bb ? pc1 : pc0) & 1, abort_flag, status,
                               kStatusBwdMma);
                ok = __all_sync(0xffffffffu, ok);
                if (bb) ++pc1; else ++pc0;
                tc_fence_after();
                if (!ok) break;
                if (!DK) {
                    // dV reads dO of this step: its slot comes now (in step order)
                    acquire(o_full, T::NO, oacq, os_cur);
                    if (!ok) break;
                }
                mma_acc(qs_cur, os_cur, bb, t > 0);
                tc_commit_warp(&q_empty[qs_cur]);          // Q and its statistics done
                if (!DK) tc_commit_warp(&o_empty[os_cur]);
                int qs_nn = 0, os_nn = 0;
                if (t + 2 < n) {
                    issue_s(bb, qs_nn, os_nn);
                    if (!ok) break;
                    if (t + 3 == n) tc_commit_warp(kv_empty);
                }
                qs_cur = qs_nxt;
                os_cur = os_nxt;
                qs_nxt = qs_nn;
                os_nxt = os_nn;
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
    } else if (warp < 4) {
        // ------------------------------------------------------------ softmax warps
        const int row = warp * 32 + lane;              // key row within the tile
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        bool ok = true;
        uint32_t gs = 0;
        int uk = 0;
        for (int r = 0; ok; ++r) {
            int L = 0;
            const int got = unit_at(r, L, true, kStatusBwdSoftmax);
            if (got < 0) ok = false;
            if (got <= 0) break;
            if (got == 2) continue;
            int b, hk, kt, q_begin, n;
            unit_info(L, b, hk, kt, q_begin, n);
            const int key = kt * T::BU + row;
            uint16_t* out_row = out + static_cast<size_t>(b * out_lay.batch + hk * out_lay.head +
                                                          static_cast<long long>(key) * out_lay.row);
            if (n == 0) {
                // No query sees these keys: their gradients are zero.
                if (key < S_k) {
                    uint4* pa = reinterpret_cast<uint4*>(out_row);
                    for (int i = 0; i < D / 8; ++i) pa[i] = make_uint4(0, 0, 0, 0);
                }
                continue;
            }
            int h = hk * kv_group, qi = q_begin;
            for (int t = 0; t < n; ++t, next_step(q_begin, h, qi)) {
                const uint32_t s = gs + static_cast<uint32_t>(t);
                const int buf = static_cast<int>(s & 1);
                const int qs = static_cast<int>(s % T::NQ);
                ok = mbar_wait(&s_full[buf], (s >> 1) & 1, abort_flag, status, kStatusBwdSoftmax);
                if (ok) ok = mbar_wait(&q_full[qs], (s / T::NQ) & 1, abort_flag, status,
                                       kStatusBwdSoftmax);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const float* st = sStat + qs * T::STAT_FLOATS;
                const int q0 = qi * T::BS;
                // key > query + causal_off is masked; only steps that reach below the
                // diagonal need it
                const bool masked = CAUSAL && q0 + causal_off < kt * T::BU + T::BU - 1;
                const int lim = key - q0 - causal_off;     // visible iff c >= lim
                uint32_t sv[64];
                tmem_ld64(lane_base + T::S_COL + buf * 64, sv);
                if (DK) {
                    uint32_t dpv[64], pk_p[32], pk_ds[32];
                    tmem_ld64(lane_base + T::DP_COL + buf * 64, dpv);
                    if (masked)
                        grad_pack64<true, BF16, false, true>(sv, dpv, st, st + T::BS, 0.f, 0.f,
                                                             scale_log2,
                                                             [&](int c) { return c >= lim; },
                                                             pk_p, pk_ds);
                    else
                        grad_pack64<false, BF16, false, true>(sv, dpv, st, st + T::BS, 0.f, 0.f,
                                                              scale_log2, [](int) { return true; },
                                                              pk_p, pk_ds);
                    tmem_st32(lane_base + T::DP_COL + buf * 64 + T::PK_OFF, pk_ds);
                } else {
                    uint32_t pk_p[32];
                    if (masked)
                        prob_pack64<true, BF16>(sv, st, scale_log2,
                                                [&](int c) { return c >= lim; }, pk_p);
                    else
                        prob_pack64<false, BF16>(sv, st, scale_log2, [](int) { return true; },
                                                 pk_p);
                    tmem_st32(lane_base + T::S_COL + buf * 64 + T::PK_OFF, pk_p);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[buf]);
            }
            if (!ok) break;
            gs += static_cast<uint32_t>(n);
            ok = mbar_wait(acc_done, uk & 1, abort_flag, status, kStatusBwdSoftmax);
            ok = __all_sync(0xffffffffu, ok);
            ++uk;
            if (!ok) break;
            tc_fence_after();
            store_row_from_tmem<D, BF16>(lane_base + T::ACC_COL, out_scale, out_row, key < S_k);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, T::TMEM_COLS);
        if (lane == 0) publish_abort(abort_flag, words, launch);
    }
}

}  // namespace attn
