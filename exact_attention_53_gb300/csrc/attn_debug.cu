// Debug build of the attention forward and backward for failure-detection
// tests (libattn_debug.so, declared in include/attn_debug.h).
//
// The same kernel source as the release library, compiled with
// ATTN_DEBUG_FAULTS: every bounded wait gives up after 1 ms instead of 2 s, and
// the producer warp (the forward's, or the backward dK/dV kernel's) can be
// told to load nothing for one work unit and stop, so the unit's consumers
// wait on barriers that nothing will complete; the caller also sets the CTAs'
// time budget, so a test can make the launch pass its deadline.  Nothing faults or hangs: the waits run out or the deadline
// passes, the CTA records it in its own status word, stops the launch's other
// CTAs, frees tensor memory and returns.
// The release library (libattn.so) is built without this flag and has neither
// the short limit nor the skip.
#define ATTN_DEBUG_FAULTS 1

#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

// Built with -fvisibility=hidden: only the two entry points below are
// exported.  Everything else (the kernel's host stub, the per-kernel set-up
// flags of its launcher) stays private to this library, so a process that
// also loads libattn.so never mixes the two builds' code or state.
#pragma GCC visibility push(default)
#include "attn_debug.h"
#pragma GCC visibility pop
#include "attn_bwd.cuh"
#include "attn_fwd.cuh"

namespace {

__device__ attn::DeviceWords g_debug_words;
std::atomic<unsigned long long> g_debug_launches{0};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Dense [B, H, S, 64] bf16 as a 4-D map (d, S, H, B), box 64 × `rows` rows, 128-byte swizzle.
bool encode(CUtensorMap* map, const void* base, int64_t B, int64_t H, int64_t S,
            uint32_t rows = 128) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t strides[3] = {64 * 2, static_cast<cuuint64_t>(S * 64 * 2),
                             static_cast<cuuint64_t>(H * S * 64 * 2)};
    cuuint32_t box[4] = {64, rows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

int attn_debug_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                   int64_t H, int64_t S, float scale, int skip_unit, uint64_t budget_ns,
                   struct CUstream_st* stream) {
    if (!q || !k || !v || !o || !lse || B < 1 || H < 1 || S < 1 || B * H > (1 << 20) ||
        S > (1 << 16))
        return static_cast<int>(cudaErrorInvalidValue);
    void* words = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&words, g_debug_words);
    if (e != cudaSuccess) return static_cast<int>(e);
    e = cudaMemcpyToSymbolAsync(attn::g_attn_debug_skip_unit, &skip_unit, sizeof(int), 0,
                                cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return static_cast<int>(e);
    attn::FwdArgs a{};
    if (!encode(&a.tm_q, q, B, H, S) || !encode(&a.tm_k, k, B, H, S) ||
        !encode(&a.tm_v, v, B, H, S) || !encode(&a.tm_o, o, B, H, S))
        return static_cast<int>(cudaErrorInvalidValue);
    a.o = o;
    a.lse = lse;
    a.S_q = a.S_k = static_cast<int32_t>(S);
    a.BH = static_cast<int32_t>(B * H);
    a.H = static_cast<int32_t>(H);
    a.kv_group = 1;
    a.causal_off = 0;
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    a.n_split = 1;
    a.pack = 1;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
    a.device = dev;
    a.words = static_cast<attn::DeviceWords*>(words);
    a.launch = ++g_debug_launches;
    a.budget_ns = budget_ns ? budget_ns : 5000000000ull;
    return static_cast<int>(attn::launch_attn_fwd<64, true, false, false>(a, stream));
}

int attn_debug_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, float* workspace, int64_t B,
                   int64_t H, int64_t S, float scale, int skip_unit, uint64_t budget_ns,
                   struct CUstream_st* stream) {
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace || B < 1 ||
        H < 1 || S < 1 || B * H > (1 << 20) || S > (1 << 16))
        return static_cast<int>(cudaErrorInvalidValue);
    void* words = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&words, g_debug_words);
    if (e != cudaSuccess) return static_cast<int>(e);
    e = cudaMemcpyToSymbolAsync(attn::g_attn_debug_skip_unit, &skip_unit, sizeof(int), 0,
                                cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return static_cast<int>(e);
    attn::BwdArgs g{};
    if (!encode(&g.tm_k_fixed, k, B, H, S) || !encode(&g.tm_v_fixed, v, B, H, S) ||
        !encode(&g.tm_q_step, q, B, H, S, 64) || !encode(&g.tm_do_step, dout, B, H, S, 64) ||
        !encode(&g.tm_q_fixed, q, B, H, S) || !encode(&g.tm_do_fixed, dout, B, H, S) ||
        !encode(&g.tm_dk_out, dk, B, H, S, 32) || !encode(&g.tm_dv_out, dv, B, H, S, 32))
        return static_cast<int>(cudaErrorInvalidValue);
    const int64_t s_pad = (S + 127) / 128 * 128;
    const attn::RowLayout lay{H * S * 64, S * 64, 64};
    g.o = o;
    g.dout = dout;
    g.lse = lse;
    g.lse2 = workspace;
    g.delta = workspace + B * H * s_pad;
    g.dq = dq;
    g.dk = dk;
    g.dv = dv;
    g.o_lay = g.do_lay = g.dq_lay = g.dk_lay = g.dv_lay = lay;
    g.S_q = g.S_k = static_cast<int32_t>(S);
    g.BH = static_cast<int32_t>(B * H);
    g.S_pad = static_cast<int32_t>(s_pad);
    g.H = static_cast<int32_t>(H);
    g.kv_group = 1;
    g.causal_off = 0;
    g.scale = scale;
    g.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    if (dev < 0 || dev >= 64) return static_cast<int>(cudaErrorInvalidDevice);
    e = cudaDeviceGetAttribute(&g.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return static_cast<int>(e);
    g.device = dev;
    g.words = static_cast<attn::DeviceWords*>(words);
    g.launch_dkdv = ++g_debug_launches;
    g.launch_key2 = ++g_debug_launches;
    g.launch_dq = ++g_debug_launches;
    g.budget_ns = budget_ns ? budget_ns : 5000000000ull;
    g.aux_stream = nullptr;                    // the dQ kernel runs on `stream` too
    return static_cast<int>(attn::launch_attn_bwd<64, true, false>(g, stream));
}

int attn_debug_status(unsigned int* status, struct CUstream_st* stream) {
    if (!status) return static_cast<int>(cudaErrorInvalidValue);
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return static_cast<int>(e);
    attn::DeviceWords w{};
    e = cudaMemcpyFromSymbol(&w, g_debug_words, sizeof(w));
    if (e != cudaSuccess) return static_cast<int>(e);
    *status = w.status;
    const attn::DeviceWords zero{};
    return static_cast<int>(cudaMemcpyToSymbol(g_debug_words, &zero, sizeof(zero)));
}

}  // extern "C"
