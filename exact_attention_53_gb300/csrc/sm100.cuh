// Blackwell (sm_100 family, built for sm_103a) primitives as inline PTX:
// mbarriers with bounded waits, TMA tensor loads, tcgen05 tensor-memory
// allocation, MMA issue, commit, and TMEM <-> register moves.
//
// Every wait here is bounded by a wall-clock limit read from %globaltimer, and
// every launch by a deadline and a launch-wide stop (LaunchWatch).  A wait that
// runs out records a code in the device status word, stops its CTA and returns
// false, so the kernel can drain and return instead of spinning forever.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace attn {
namespace sm100 {

// ---------------------------------------------------------------- addressing
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Upper bound on one wait.  Real waits in this library last microseconds.  A
// debug build (ATTN_DEBUG_FAULTS, never the release library) waits 1 ms so
// that a test can make a wait run out quickly.
#ifdef ATTN_DEBUG_FAULTS
constexpr uint64_t kWaitLimitNs = 1000000ull;
#else
constexpr uint64_t kWaitLimitNs = 2000000000ull;
#endif
// How often a CTA's producer looks whether another CTA of its launch gave up.
constexpr uint64_t kPeerCheckNs = 50000ull;

// Status bit recorded when a CTA passes its launch's deadline.
constexpr unsigned int kStatusDeadline = 1u << 9;

// Per-GPU words in global memory, shared by every launch of the library:
// the status bits of waits that ran out (read and cleared by the host), and
// the number of the last launch that gave up.
struct DeviceWords {
    unsigned int status;
    unsigned int reserved;
    unsigned long long abort_launch;
};

// Wait for the phase of parity `parity` to complete.  Returns false (after
// recording `code` in *status and raising the CTA's abort flag) when the
// limit runs out, or at once when this CTA has been stopped.  The spin and its
// exit path are kept to the fewest instructions: the wait is inlined at every
// handoff of every role, and extra code here (even on the exit path) was
// measured to slow the kernels by a few percent.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag, unsigned int* status,
                                          unsigned int code) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(a, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(status, code);
            return false;
        }
    }
}

// mbar_wait for a role that idles for a long time (a whole work unit) and is
// not on the critical path: it first polls with a kIdleSleepNs sleep between
// tries (at most kIdleTries of them, about a millisecond), leaving its issue
// slots to the warps of the same SM sub-partition that do the unit's work
// (polling without the sleep slowed those warps measurably), then waits as
// mbar_wait does, with the same limit and abort behaviour.
constexpr unsigned int kIdleSleepNs = 128;
constexpr int kIdleTries = 4096;

__device__ __forceinline__ bool mbar_wait_idle(uint64_t* bar, uint32_t parity,
                                               volatile int* abort_flag, unsigned int* status,
                                               unsigned int code) {
    const uint32_t a = smem_u32(bar);
    for (int i = 0; i < kIdleTries && !mbar_try_wait(a, parity); ++i) __nanosleep(kIdleSleepNs);
    return mbar_wait(bar, parity, abort_flag, status, code);
}

// Launch-wide bounds, kept in registers by each CTA's TMA producer warp (the
// one role that runs ahead of the others and is never on the critical path).
// Together with the bounded waits they make every launch end in bounded time:
//   * one wait gives up after kWaitLimitNs (mbar_wait), raising the CTA's
//     abort flag, so every other role of the CTA leaves at its next wait;
//   * the producer checks at every eighth load it issues and at every work
//     unit that the CTA has not run past its deadline (its start plus a budget the host
//     derives from the launch's work, far above its real duration), and stops
//     the CTA if it has;
//   * a CTA that gave up records its launch number in words->abort_launch on
//     its way out (publish_abort); producers read it once their first unit's
//     loads are issued and every kPeerCheckNs after that, so the launch's
//     other CTAs stop too.
// Every role's step loop waits on a barrier that the producer (directly or
// through the MMA warp) completes once per step, so a role that ran past its
// partners (a wrong trip count) blocks within a ring's depth of steps and
// leaves there; the producer itself is bounded by the deadline.
struct LaunchWatch {
    const DeviceWords* words;
    unsigned long long launch;        // this launch's number (host counter, per device)
    uint64_t deadline;                // %globaltimer value after which the CTA gives up
    uint64_t next_peer;               // when to read words->abort_launch next

    __device__ __forceinline__ LaunchWatch(const DeviceWords* w, unsigned long long launch_no,
                                           unsigned long long budget_ns)
        : words(w), launch(launch_no) {
        const uint64_t now = global_timer_ns();
        deadline = now + budget_ns;
        next_peer = now + kPeerCheckNs;
    }

    // Read the abort word now (the producer calls this once its first unit's
    // loads are in flight, so the read's latency hides behind them): a CTA
    // that starts after its launch gave up stops here.
    __device__ __forceinline__ bool launch_gave_up(volatile int* abort_flag) {
        int s = *reinterpret_cast<const volatile unsigned long long*>(&words->abort_launch) ==
                launch;
        s = __shfl_sync(0xffffffffu, s, 0);
        if (s && (threadIdx.x & 31) == 0) *abort_flag = 1;
        return s != 0;
    }

    // True once the CTA must stop: it already has, it passed its deadline
    // (status bit kStatusDeadline), or another CTA of the launch gave up.
    // Warp-uniform: lane 0 decides.
    __device__ __forceinline__ bool stop(volatile int* abort_flag, unsigned int* status) {
        int s = *abort_flag;
        if (!s) {
            const uint64_t now = global_timer_ns();
            if (now > deadline) {
                if ((threadIdx.x & 31) == 0) {
                    *abort_flag = 1;
                    atomicOr(status, kStatusDeadline);
                }
                s = 1;
            } else if (now >= next_peer) {
                s = *reinterpret_cast<const volatile unsigned long long*>(&words->abort_launch) ==
                    launch;
                if (s && (threadIdx.x & 31) == 0) *abort_flag = 1;
                next_peer = now + kPeerCheckNs;
            }
        }
        return __shfl_sync(0xffffffffu, s, 0) != 0;
    }
};

// On a CTA's way out: if it gave up, tell the launch's other CTAs.
__device__ __forceinline__ void publish_abort(volatile int* abort_flag, DeviceWords* words,
                                              unsigned long long launch) {
    if (*abort_flag) atomicMax(&words->abort_launch, launch);
}

// After this CTA gave up: wait (bounded) for the phase of parity `parity` of
// `bar` to complete, e.g. for a copy in flight to land before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t t0,
                                           unsigned int* status, unsigned int code) {
    const uint32_t a = smem_u32(bar);
    while (!mbar_try_wait(a, parity)) {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, code);
            break;
        }
    }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 4-D tiled load of one box into shared memory, coordinates (innermost, row,
// head, batch); completion is counted in bytes on `bar`.  Rows past the
// tensor's extent are filled with zeros and still counted.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1, int32_t c2, int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
        "r"(c3)
        : "memory");
}

// 4-D tiled store of one box from shared memory (rows past the tensor's extent
// are not written), tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int32_t c0,
                                             int32_t c1, int32_t c2, int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// 1-D bulk copy global -> shared of `bytes` (a multiple of 16; both addresses
// 16-byte aligned), completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every bulk group this thread committed has finished reading its
// shared-memory source (the source may then be overwritten).
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until every bulk group this thread committed has finished writing.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA, tensor core).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- cluster launch control
// Ask the hardware to cancel one CTA of this grid that has not started yet.
// The 16-byte answer lands at `resp` (16-byte aligned shared memory) and
// completes 16 transaction bytes on `bar`, which the caller has armed with
// mbar_arrive_expect_tx(bar, 16).  A CTA that wins a cancellation does that
// CTA's work itself: a hardware work queue for persistent kernels.
__device__ __forceinline__ void clc_try_cancel(uint32_t resp, uint64_t* bar) {
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 "
        "[%0], [%1];" ::"r"(resp),
        "r"(smem_u32(bar))
        : "memory");
}

// Decode an answer: true and the cancelled CTA's blockIdx.x if the request
// won a CTA; false once no CTA was left to cancel.
__device__ __forceinline__ bool clc_query(uint32_t resp, int& ctaid_x) {
    uint32_t won;
    uint32_t x = 0;
    asm volatile(
        "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t"
        "ld.shared.b128 r, [%2];\n\t"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
        : "=r"(won), "+r"(x)
        : "r"(resp)
        : "memory");
    ctaid_x = static_cast<int>(x);
    return won != 0;
}

// A CTA's sequence of work units over a grid with one CTA per unit.  Unit 0
// is the CTA's own (blockIdx.x); unit r >= 1 is the answer to claim r-1,
// which lands in slot (r-1) % SLOTS of `resp` (16 bytes a slot) and completes
// full[slot].  Every consumer warp arrives once on empty[slot] after reading
// it; the claiming warp reuses a slot only after that.  At most one claim is
// in flight, and none is made once one has come back empty.
template <int SLOTS>
struct WorkQueue {
    uint8_t* resp;
    uint64_t* full;
    uint64_t* empty;

    // Unit r: 1 with the unit in L, 0 when the queue is empty, -1 when the
    // wait gave up.  Warp-uniform.
    __device__ __forceinline__ int unit(int r, int& L, bool consumer, volatile int* abort_flag,
                                        unsigned int* status, unsigned int code) const {
        if (r == 0) {
            L = static_cast<int>(blockIdx.x);
            return 1;
        }
        const int i = r - 1;
        const int slot = i % SLOTS;
        bool got = mbar_wait(&full[slot], (i / SLOTS) & 1, abort_flag, status, code);
        got = __all_sync(0xffffffffu, got);
        if (!got) return -1;
        int x = 0;
        const bool won = clc_query(smem_u32(resp + slot * 16), x);
        if (consumer) {
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(&empty[slot]);
        }
        L = x;
        return won ? 1 : 0;
    }

    // Claim the next unit (claim number `claims`, then incremented); the
    // calling warp's `leader` lane issues it.  False when the wait gave up.
    __device__ __forceinline__ bool claim(int& claims, bool leader, volatile int* abort_flag,
                                          unsigned int* status, unsigned int code) const {
        const int slot = claims % SLOTS;
        bool ok = mbar_wait(&empty[slot], ((claims / SLOTS) & 1) ^ 1, abort_flag, status, code);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) return false;
        if (leader) {
            fence_proxy_async_smem();           // earlier reads of the slot come first
            mbar_arrive_expect_tx(&full[slot], 16);
            clc_try_cancel(smem_u32(resp + slot * 16), &full[slot]);
        }
        __syncwarp();
        ++claims;
        return true;
    }

    // After an abort: wait (bounded) for the last claim's answer to land.
    __device__ __forceinline__ void drain(int claims, unsigned int* status,
                                          unsigned int code) const {
        if (claims == 0) return;
        const int i = claims - 1;
        drain_wait(&full[i % SLOTS], (i / SLOTS) & 1, global_timer_ns(), status, code);
    }
};

// Barrier over `count` threads (a multiple of 32) on hardware barrier `id`.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Warp-collective forms: every lane of the (converged) warp executes them with
// the same operands, and one elected lane issues the instruction.  Keeping the
// issuing loop warp-uniform lets the compiler keep descriptors and addresses
// in uniform registers; issuing from a divergent single lane instead costs
// about a hundred cycles per MMA.  elect.sync picks the same leader every
// time, so MMAs and the commit that tracks them come from one thread.
__device__ __forceinline__ void mma_ss_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\t"
        "elect.sync r|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\t"
        "elect.sync r|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Same, with the two 64-bit smem descriptors passed as (low, high) 32-bit
// halves: callers step along K by adding to the low half only.
__device__ __forceinline__ void mma_ss_warp(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi,
                                            uint32_t b_lo, uint32_t b_hi, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\t.reg .b64 da, db;\n\t"
        "mov.b64 da, {%1, %2};\n\t"
        "mov.b64 db, {%3, %4};\n\t"
        "elect.sync r|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                            uint32_t b_hi, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\t.reg .b64 db;\n\t"
        "mov.b64 db, {%2, %3};\n\t"
        "elect.sync r|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit_warp(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\t"
        "elect.sync r|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .b32 r;\n\t"
        "elect.sync r|e, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, e;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// Shared-memory matrix descriptor, 128-byte swizzle (the layout TMA writes
// with CU_TENSOR_MAP_SWIZZLE_128B into 1024-byte aligned tiles).
//   bits  0-13 start address >> 4
//   bits 16-29 leading-dimension byte offset >> 4
//   bits 32-45 stride-dimension byte offset >> 4
//   bits 46-47 descriptor version (1 on sm_100 family)
//   bits 61-63 layout: 2 = 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// Instruction descriptor for kind::f16 with an fp32 accumulator.
//   bits 4-5 D type (1 = f32); 7-9 A type, 10-12 B type (0 = f16, 1 = bf16);
//   13 / 14 negate A / B; 15 / 16 A / B major (0 = K-major, 1 = MN-major);
//   17-22 N >> 3; 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool a_mn_major,
                                                 bool b_mn_major) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// OR-ed into an instruction descriptor: the MMA uses −A in place of A (an
// exact sign flip of every A element).
constexpr uint32_t kIdescNegateA = 1u << 13;

// ---------------------------------------------------------------- TMEM <-> registers
// 32x32b shape: thread i of the warp gets lane (base lane + i); .xN gives N
// consecutive 32-bit columns.  The wait is folded into the same asm statement
// so no value is read before it has landed.
#define ATTN_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
    "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define ATTN_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
    "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : ATTN_R8(0), ATTN_R8(8), ATTN_R8(16), ATTN_R8(24)
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
        "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : ATTN_R8(0), ATTN_R8(8), ATTN_R8(16), ATTN_R8(24), ATTN_R8(32), ATTN_R8(40),
          ATTN_R8(48), ATTN_R8(56)
        : "r"(taddr)
        : "memory");
}

// Two 64-column loads in flight together, one wait for both.
#define ATTN_Q8(i) "=r"(q[i]), "=r"(q[i + 1]), "=r"(q[i + 2]), "=r"(q[i + 3]), \
    "=r"(q[i + 4]), "=r"(q[i + 5]), "=r"(q[i + 6]), "=r"(q[i + 7])
__device__ __forceinline__ void tmem_ld64x2(uint32_t taddr_a, uint32_t taddr_b, uint32_t (&r)[64],
                                            uint32_t (&q)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
        "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%128];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
        "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,"
        "%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
        "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%129];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : ATTN_R8(0), ATTN_R8(8), ATTN_R8(16), ATTN_R8(24), ATTN_R8(32), ATTN_R8(40),
          ATTN_R8(48), ATTN_R8(56), ATTN_Q8(0), ATTN_Q8(8), ATTN_Q8(16), ATTN_Q8(24), ATTN_Q8(32),
          ATTN_Q8(40), ATTN_Q8(48), ATTN_Q8(56)
        : "r"(taddr_a), "r"(taddr_b)
        : "memory");
}
#undef ATTN_Q8

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        ATTN_W8(0), ATTN_W8(8), ATTN_W8(16), ATTN_W8(24)
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#undef ATTN_R8
#undef ATTN_W8

// ---------------------------------------------------------------- registers
// Per-warpgroup register budget changes (all 128 threads of the warpgroup
// execute the same instruction).  The sum over warpgroups must not exceed the
// registers the CTA was launched with.
template <int N>
__device__ __forceinline__ void regs_grow() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_shrink() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
// Move a warpgroup from the launch's LAUNCH registers a thread to N: grow
// when N is larger, shrink when smaller, nothing when equal (setmaxnreg.inc
// must not lower the count, nor .dec raise it).
template <int N, int LAUNCH>
__device__ __forceinline__ void regs_set() {
    static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg takes 24..256 in steps of 8");
    if constexpr (N > LAUNCH) regs_grow<N>();
    else if constexpr (N < LAUNCH) regs_shrink<N>();
}

// ---------------------------------------------------------------- math
// Three-input maximum (one instruction on sm_100 family).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two floats to a bf16x2 / f16x2 word, round-to-nearest-even; `lo` lands in
// the low 16 bits (the lower-addressed element).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace sm100
}  // namespace attn
