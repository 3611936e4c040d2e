// C ABI of libattn.so: argument validation, TMA descriptor encoding, kernel
// selection and launch.  Declared in include/attn.h.
//
// Validation mirrors the page's validate_config (oxicuda-dnn 0.1.8 hopper.rs):
// head_dim must be one of SUPPORTED_HEAD_DIMS, the element type f16 or bf16,
// and every failure names the offending field.  Problem sizes, pointers and the
// scale are checked here as well, because the library takes raw pointers.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#pragma GCC visibility push(default)    // the C ABI is the library's only export
#include "attn.h"
#pragma GCC visibility pop
#include "attn_launch.h"
#include "sm100.cuh"

namespace {

constexpr int kVersion = 10000;  // 1.0.0
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxSeq = int64_t(1) << 22;

thread_local char g_msg[512] = "";

attn_status_t fail(attn_status_t s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return s;
}

attn_status_t ok() {
    g_msg[0] = '\0';
    return ATTN_OK;
}

// Status bits (bit per role) set by a kernel whose bounded wait ran out, and
// the number of the last launch that gave up.
__device__ attn::DeviceWords g_attn_words;

std::atomic<int> g_device_checked[kMaxDevices];          // 0 unknown, 1 ok, 2 unsupported
std::atomic<attn::DeviceWords*> g_words_ptr[kMaxDevices];
std::atomic<unsigned long long> g_launches[kMaxDevices];  // kernel launches numbered per device
std::atomic<int> g_num_sms[kMaxDevices];
std::atomic<void*> g_noalloc_scratch[kMaxDevices];       // attn_fwd_splitkv_noalloc's scratch

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

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool aligned(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// Element strides of a [B, heads, S, d] view; the d elements of a row are contiguous.
using Layout = attn_layout_t;

Layout dense_layout(int64_t heads, int64_t S, int64_t d) { return {heads * S * d, S * d, d}; }

// Bytes from the first to one past the last element of a [B, heads, S, d] view.
size_t span_bytes(const Layout& l, int64_t B, int64_t heads, int64_t S, int64_t d) {
    return static_cast<size_t>((B - 1) * l.batch + (heads - 1) * l.head + (S - 1) * l.row + d) * 2;
}

struct Problem {
    int64_t B, H, S_q, S_k, d;
    int64_t H_kv = 0;            // key/value heads (H for plain multi-head attention)
    bool causal;
    int64_t causal_off = 0;      // key j visible to query i iff j <= i + causal_off
    int64_t pack = 1;            // split-KV: query heads sharing one query tile
    float scale;
    attn_dtype_t dtype;
    Layout lq, lk, lv, lo;
    size_t q_bytes, kv_bytes, o_bytes, lse_bytes;   // spans of q, k (= v), o, lse
    size_t v_bytes;
};

attn_status_t validate_sizes(Problem& p, int64_t B, int64_t H, int64_t S_q, int64_t S_k,
                             int64_t d, int causal, float scale, attn_dtype_t dtype) {
    if (B < 1) return fail(ATTN_ERR_INVALID_ARG, "B must be >= 1, got %lld", (long long)B);
    if (H < 1) return fail(ATTN_ERR_INVALID_ARG, "H must be >= 1, got %lld", (long long)H);
    if (S_q < 1) return fail(ATTN_ERR_INVALID_ARG, "S_q must be >= 1, got %lld", (long long)S_q);
    if (S_k < 1) return fail(ATTN_ERR_INVALID_ARG, "S_k must be >= 1, got %lld", (long long)S_k);
    if (d < 1) return fail(ATTN_ERR_INVALID_ARG, "d must be >= 1, got %lld", (long long)d);
    if (d != 64 && d != 128 && d != 256)
        return fail(ATTN_ERR_UNSUPPORTED, "head_dim d=%lld not supported; must be one of [64, 128, 256]",
                    (long long)d);
    if (dtype != ATTN_DTYPE_F16 && dtype != ATTN_DTYPE_BF16)
        return fail(ATTN_ERR_UNSUPPORTED, "dtype must be ATTN_DTYPE_F16 (0) or ATTN_DTYPE_BF16 (1), got %d",
                    (int)dtype);
    if (causal != 0 && causal != 1)
        return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1, got %d", causal);
    if (!std::isfinite(scale))
        return fail(ATTN_ERR_INVALID_ARG, "scale must be finite");
    if (B * H > INT32_MAX || B > INT32_MAX || H > INT32_MAX)
        return fail(ATTN_ERR_INVALID_ARG, "B*H = %lld exceeds 2^31-1", (long long)(B * H));
    if (S_q > kMaxSeq) return fail(ATTN_ERR_INVALID_ARG, "S_q=%lld exceeds 2^22", (long long)S_q);
    if (S_k > kMaxSeq) return fail(ATTN_ERR_INVALID_ARG, "S_k=%lld exceeds 2^22", (long long)S_k);
    p.B = B; p.H = H; p.S_q = S_q; p.S_k = S_k; p.d = d;
    p.H_kv = H;
    p.causal = causal != 0;
    p.causal_off = 0;
    p.scale = scale;
    p.dtype = dtype;
    p.lq = p.lo = dense_layout(H, S_q, d);
    p.lk = p.lv = dense_layout(H, S_k, d);
    const size_t bh = static_cast<size_t>(B * H);
    p.q_bytes = bh * static_cast<size_t>(S_q) * static_cast<size_t>(d) * 2;
    p.kv_bytes = bh * static_cast<size_t>(S_k) * static_cast<size_t>(d) * 2;
    p.v_bytes = p.kv_bytes;
    p.o_bytes = p.q_bytes;
    p.lse_bytes = bh * static_cast<size_t>(S_q) * 4;
    return ATTN_OK;
}

// A [B, heads, S, d] view whose elements are all distinct: sorted by stride,
// each dimension must step past everything the smaller ones span.
bool layout_injective(const Layout& l, int64_t B, int64_t heads, int64_t S, int64_t d) {
    struct Dim { int64_t stride, extent; };
    Dim dims[3] = {{l.row, S}, {l.head, heads}, {l.batch, B}};
    std::sort(dims, dims + 3, [](const Dim& a, const Dim& b) { return a.stride < b.stride; });
    int64_t reach = d;                    // elements spanned by the smaller dimensions
    for (const Dim& x : dims) {
        if (x.extent <= 1) continue;
        if (x.stride < reach) return false;
        reach = x.stride * (x.extent - 1) + reach;
    }
    return true;
}

attn_status_t check_layout(const Layout& l, const char* name, int64_t d) {
    const int64_t s[3] = {l.batch, l.head, l.row};
    const char* nm[3] = {"batch", "head", "row"};
    for (int i = 0; i < 3; ++i) {
        if (s[i] < 1 || s[i] % 8 != 0 || s[i] > (int64_t(1) << 39))
            return fail(ATTN_ERR_INVALID_ARG,
                        "%s %s stride %lld must be a positive multiple of 8 elements (16 bytes) below 2^39",
                        name, nm[i], (long long)s[i]);
    }
    if (l.row < d)
        return fail(ATTN_ERR_INVALID_ARG, "%s row stride %lld is below d=%lld", name, (long long)l.row,
                    (long long)d);
    return ATTN_OK;
}

// Sizes, heads, mask and the q, k, v, o layouts shared by the general forward
// and backward entry points.
attn_status_t validate_common(Problem& p, int64_t B, int64_t H, int64_t H_kv, int64_t S_q,
                              int64_t S_k, int64_t d, int mask, float scale, attn_dtype_t dtype,
                              const Layout& lq, const Layout& lk, const Layout& lv,
                              const Layout& lo) {
    if (mask < 0 || mask > 2)
        return fail(ATTN_ERR_INVALID_ARG, "mask must be 0, 1 or 2, got %d", mask);
    attn_status_t s = validate_sizes(p, B, H, S_q, S_k, d, mask != 0 ? 1 : 0, scale, dtype);
    if (s != ATTN_OK) return s;
    if (H_kv < 1 || H_kv > H || H % H_kv != 0)
        return fail(ATTN_ERR_INVALID_ARG, "H_kv=%lld must divide H=%lld", (long long)H_kv,
                    (long long)H);
    if (mask == 2 && S_q > S_k)
        return fail(ATTN_ERR_UNSUPPORTED,
                    "bottom-right causal mask needs S_q <= S_k (got S_q=%lld, S_k=%lld): earlier "
                    "queries would see no key",
                    (long long)S_q, (long long)S_k);
    if ((s = check_layout(lq, "q", d)) != ATTN_OK) return s;
    if ((s = check_layout(lk, "k", d)) != ATTN_OK) return s;
    if ((s = check_layout(lv, "v", d)) != ATTN_OK) return s;
    if ((s = check_layout(lo, "o", d)) != ATTN_OK) return s;
    p.H_kv = H_kv;
    p.causal_off = mask == 2 ? S_k - S_q : 0;
    p.lq = lq;
    p.lk = lk;
    p.lv = lv;
    p.lo = lo;
    p.q_bytes = span_bytes(p.lq, p.B, p.H, p.S_q, p.d);
    p.kv_bytes = span_bytes(p.lk, p.B, p.H_kv, p.S_k, p.d);
    p.v_bytes = span_bytes(p.lv, p.B, p.H_kv, p.S_k, p.d);
    p.o_bytes = span_bytes(p.lo, p.B, p.H, p.S_q, p.d);
    return ATTN_OK;
}

attn_status_t validate_general(Problem& p, const attn_fwd_params_t* a) {
    if (!a) return fail(ATTN_ERR_INVALID_ARG, "params is null");
    attn_status_t s = validate_common(p, a->B, a->H, a->H_kv, a->S_q, a->S_k, a->d, a->mask,
                                      a->scale, a->dtype, a->q_layout, a->k_layout, a->v_layout,
                                      a->o_layout);
    if (s != ATTN_OK) return s;
    if (!layout_injective(p.lo, p.B, p.H, p.S_q, p.d))
        return fail(ATTN_ERR_INVALID_ARG, "o layout maps two elements to one address");
    return ATTN_OK;
}

attn_status_t validate_device_ptrs(const Problem& p, const void* q, const void* k, const void* v,
                                   const void* o, const void* lse) {
    if (!q) return fail(ATTN_ERR_INVALID_ARG, "q is null");
    if (!k) return fail(ATTN_ERR_INVALID_ARG, "k is null");
    if (!v) return fail(ATTN_ERR_INVALID_ARG, "v is null");
    if (!o) return fail(ATTN_ERR_INVALID_ARG, "o is null");
    if (!lse) return fail(ATTN_ERR_INVALID_ARG, "lse is null");
    if (!aligned(q, 16)) return fail(ATTN_ERR_INVALID_ARG, "q is not 16-byte aligned");
    if (!aligned(k, 16)) return fail(ATTN_ERR_INVALID_ARG, "k is not 16-byte aligned");
    if (!aligned(v, 16)) return fail(ATTN_ERR_INVALID_ARG, "v is not 16-byte aligned");
    if (!aligned(o, 16)) return fail(ATTN_ERR_INVALID_ARG, "o is not 16-byte aligned");
    if (!aligned(lse, 4)) return fail(ATTN_ERR_INVALID_ARG, "lse is not 4-byte aligned");
    if (overlaps(o, p.o_bytes, q, p.q_bytes)) return fail(ATTN_ERR_INVALID_ARG, "o overlaps q");
    if (overlaps(o, p.o_bytes, k, p.kv_bytes)) return fail(ATTN_ERR_INVALID_ARG, "o overlaps k");
    if (overlaps(o, p.o_bytes, v, p.v_bytes)) return fail(ATTN_ERR_INVALID_ARG, "o overlaps v");
    if (overlaps(lse, p.lse_bytes, q, p.q_bytes)) return fail(ATTN_ERR_INVALID_ARG, "lse overlaps q");
    if (overlaps(lse, p.lse_bytes, k, p.kv_bytes)) return fail(ATTN_ERR_INVALID_ARG, "lse overlaps k");
    if (overlaps(lse, p.lse_bytes, v, p.v_bytes)) return fail(ATTN_ERR_INVALID_ARG, "lse overlaps v");
    if (overlaps(lse, p.lse_bytes, o, p.o_bytes)) return fail(ATTN_ERR_INVALID_ARG, "lse overlaps o");
    return ATTN_OK;
}

// The kernels are built for sm_103a only; check the current device once.
attn_status_t check_device(int* dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_UNSUPPORTED, "device ordinal %d", dev);
    int state = g_device_checked[dev].load(std::memory_order_acquire);
    if (state == 0) {
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        g_num_sms[dev].store(sms);
        state = (major == 10 && minor == 3) ? 1 : 2;
        g_device_checked[dev].store(state, std::memory_order_release);
        if (state == 1) {
            void* sp = nullptr;
            e = cudaGetSymbolAddress(&sp, g_attn_words);
            if (e != cudaSuccess) {
                g_device_checked[dev].store(0);
                return fail(ATTN_ERR_CUDA, "cudaGetSymbolAddress(status): %s", cudaGetErrorString(e));
            }
            g_words_ptr[dev].store(static_cast<attn::DeviceWords*>(sp));
        }
    }
    if (state != 1)
        return fail(ATTN_ERR_UNSUPPORTED, "device %d is not an sm_103 GPU; this library is built for sm_103a only", dev);
    *dev_out = dev;
    return ATTN_OK;
}

// A fresh launch number on device dev (never 0, which the abort word holds
// when no launch has given up).
unsigned long long next_launch(int dev) { return g_launches[dev].fetch_add(1) + 1; }

// Time budget of each CTA of a launch doing `flops` of work: 5 s plus the
// time the work would take at 10 TFLOP/s, two orders of magnitude below what
// the kernels sustain, so only a CTA that has stopped making progress meets it.
unsigned long long budget_ns(double flops) {
    const double ns = 5e9 + flops / 1e4;
    return ns > 1e18 ? 1000000000000000000ull : static_cast<unsigned long long>(ns);
}

// Recently encoded tensor maps of this host thread.  A map is a function of
// its encoding inputs alone (address, sizes, strides, box, element type), so a
// repeated call on the same buffers reuses it instead of encoding it again.
struct MapKey {
    const void* base;
    uint64_t dims[4];
    uint64_t strides[3];
    uint32_t box[4];
    int32_t dtype;
    int32_t pad;
};

struct MapCache {
    static constexpr int kEntries = 16;
    MapKey key[kEntries];
    CUtensorMap map[kEntries];
    int used = 0, next = 0;
};

thread_local MapCache t_maps;

// A [B, heads, S, d] view as a 4-D map (d, S, heads, B) with its own strides;
// box 64 columns × box_rows rows of one head.
attn_status_t encode_4d(CUtensorMap* map, const void* base, const Problem& p, int64_t S,
                        int64_t heads, const Layout& l, uint32_t box_rows, const char* name,
                        uint32_t box_heads = 1) {
    MapKey key;
    std::memset(&key, 0, sizeof(key));
    key.base = base;
    key.dims[0] = static_cast<uint64_t>(p.d);
    key.dims[1] = static_cast<uint64_t>(S);
    key.dims[2] = static_cast<uint64_t>(heads);
    key.dims[3] = static_cast<uint64_t>(p.B);
    key.strides[0] = static_cast<uint64_t>(l.row * 2);
    key.strides[1] = static_cast<uint64_t>(l.head * 2);
    key.strides[2] = static_cast<uint64_t>(l.batch * 2);
    key.box[0] = 64;
    key.box[1] = box_rows;
    key.box[2] = box_heads;
    key.box[3] = 1;
    key.dtype = static_cast<int32_t>(p.dtype);
    MapCache& c = t_maps;
    for (int i = 0; i < c.used; ++i) {
        if (std::memcmp(&c.key[i], &key, sizeof(key)) == 0) {
            *map = c.map[i];
            return ATTN_OK;
        }
    }
    auto fn = encode_fn();
    if (!fn) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    cuuint64_t dims[4] = {key.dims[0], key.dims[1], key.dims[2], key.dims[3]};
    cuuint64_t strides[3] = {key.strides[0], key.strides[1], key.strides[2]};
    cuuint32_t box[4] = {key.box[0], key.box[1], key.box[2], key.box[3]};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map,
                    p.dtype == ATTN_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    4, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ATTN_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", name, (int)r);
    const int slot = c.used < MapCache::kEntries ? c.used++ : c.next;
    if (slot == c.next) c.next = (c.next + 1) % MapCache::kEntries;
    c.key[slot] = key;
    c.map[slot] = *map;
    return ATTN_OK;
}

template <int D>
void fill_plan_d(const Problem& p, attn_plan_t* out) {
    using T = attn::FwdTile<D>;
    out->block_m = T::BM;
    out->block_n = T::BN;
    out->q_tiles = (p.S_q + T::BM - 1) / T::BM;
    out->kv_tiles = (p.S_k + T::BN - 1) / T::BN;
    out->q_tiles_per_cta = T::TILES;
    out->bh = p.B * p.H;
    out->units = out->bh * ((out->q_tiles + T::TILES - 1) / T::TILES);
    out->threads = T::THREADS;
    out->smem_bytes = T::SMEM_BYTES;
    out->tmem_cols = static_cast<int32_t>(T::TMEM_COLS);
    out->kv_stages = T::NS;
}

void fill_plan(const Problem& p, attn_plan_t* out) {
    if (p.d == 64) fill_plan_d<64>(p, out);
    else if (p.d == 128) fill_plan_d<128>(p, out);
    else fill_plan_d<256>(p, out);
}

using LaunchFn = cudaError_t (*)(const attn::FwdArgs&, cudaStream_t);

LaunchFn pick(int64_t d, bool bf16, bool causal) {
#define ATTN_PICK(D)                                                                   \
    if (d == D) {                                                                      \
        if (bf16) return causal ? attn::launch_attn_fwd<D, true, true, false>          \
                                : attn::launch_attn_fwd<D, true, false, false>;        \
        return causal ? attn::launch_attn_fwd<D, false, true, false>                   \
                      : attn::launch_attn_fwd<D, false, false, false>;                 \
    }
    ATTN_PICK(64)
    ATTN_PICK(128)
    ATTN_PICK(256)
#undef ATTN_PICK
    return nullptr;
}

LaunchFn pick_split(int64_t d, bool bf16) {
    if (d == 64) return bf16 ? attn::launch_attn_fwd<64, true, false, true>
                             : attn::launch_attn_fwd<64, false, false, true>;
    if (d == 128) return bf16 ? attn::launch_attn_fwd<128, true, false, true>
                              : attn::launch_attn_fwd<128, false, false, true>;
    if (d == 256) return bf16 ? attn::launch_attn_fwd<256, true, false, true>
                              : attn::launch_attn_fwd<256, false, false, true>;
    return nullptr;
}

// Maps, sizes and device words shared by every launch of problem p.
attn_status_t fill_args(attn::FwdArgs& a, const Problem& p, int dev, const void* q, const void* k,
                        const void* v, void* o, float* lse) {
    attn_status_t s;
    const uint32_t rows = attn::kBlockM;
    if ((s = encode_4d(&a.tm_q, q, p, p.S_q, p.H, p.lq, rows, "q")) != ATTN_OK) return s;
    if ((s = encode_4d(&a.tm_k, k, p, p.S_k, p.H_kv, p.lk, rows, "k")) != ATTN_OK) return s;
    if ((s = encode_4d(&a.tm_v, v, p, p.S_k, p.H_kv, p.lv, rows, "v")) != ATTN_OK) return s;
    if ((s = encode_4d(&a.tm_o, o, p, p.S_q, p.H, p.lo, rows, "o")) != ATTN_OK) return s;
    a.o = o;
    a.lse = lse;
    a.S_q = static_cast<int32_t>(p.S_q);
    a.S_k = static_cast<int32_t>(p.S_k);
    a.BH = static_cast<int32_t>(p.B * p.H);
    a.H = static_cast<int32_t>(p.H);
    a.kv_group = static_cast<int32_t>(p.H / p.H_kv);
    a.causal_off = static_cast<int32_t>(p.causal_off);
    a.scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
    a.words = g_words_ptr[dev].load();
    a.launch = next_launch(dev);
    a.budget_ns = budget_ns(4.0 * double(p.B) * double(p.H) * double(p.S_q) * double(p.S_k) *
                            double(p.d));
    a.num_sms = g_num_sms[dev].load();
    a.device = dev;
    a.n_split = 1;
    a.kv_per_split = 0;
    a.o_part = nullptr;
    a.lse_part = nullptr;
    a.pack = 1;
    return ATTN_OK;
}

attn_status_t launch_checked(const Problem& p, const void* q, const void* k, const void* v,
                             void* o, float* lse, cudaStream_t stream) {
    int dev = 0;
    attn_status_t s = check_device(&dev);
    if (s != ATTN_OK) return s;
    attn::FwdArgs a;
    if ((s = fill_args(a, p, dev, q, k, v, o, lse)) != ATTN_OK) return s;
    LaunchFn fn = pick(p.d, p.dtype == ATTN_DTYPE_BF16, p.causal);
    if (!fn) return fail(ATTN_ERR_UNSUPPORTED, "no kernel for d=%lld", (long long)p.d);
    cudaError_t e = fn(a, stream);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    return ok();
}

// ---------------------------------------------------------------- split-KV
struct SplitPlan {
    int64_t n_split;         // key ranges actually used (no range is empty)
    int64_t kv_per_split;    // key tiles per range (the last may have fewer)
    int64_t workspace_bytes; // 0 when n_split == 1 (the plain kernel runs)
};

// Split-KV units hold one 128-row query tile each.
int64_t split_query_blocks(const Problem& p) { return (p.S_q + attn::kBlockM - 1) / attn::kBlockM; }

// Requested (or, for 0, chosen) range count -> ranges, tiles per range, bytes.
// Auto: the count whose persistent schedule (waves of num_sms units, a unit
// costing its key tiles plus about one tile of setup) finishes first; ties go
// to fewer ranges, which also keeps the merge pass small.
attn_status_t split_plan(const Problem& p, int64_t n_req, int num_sms, SplitPlan* out) {
    const int64_t n_kv = (p.S_k + attn::kBlockN - 1) / attn::kBlockN;
    const int64_t base = p.pack > 1 ? p.B * p.H_kv : p.B * p.H * split_query_blocks(p);
    int64_t n = 1;
    if (n_req > 0) {
        n = std::min(n_req, n_kv);
    } else {
        double best = 0;
        const int64_t cap = std::min<int64_t>(n_kv, 1024);
        for (int64_t c = 1; c <= cap; ++c) {
            const int64_t per = (n_kv + c - 1) / c;
            const int64_t used = (n_kv + per - 1) / per;
            const int64_t waves = (base * used + num_sms - 1) / num_sms;
            const double cost = double(waves) * double(per + 1);
            if (c == 1 || cost < best) {
                best = cost;
                n = used;
            }
        }
    }
    const int64_t per = (n_kv + n - 1) / n;
    n = (n_kv + per - 1) / per;
    if (base * n > INT32_MAX)
        return fail(ATTN_ERR_INVALID_ARG, "n_split=%lld gives %lld work units, above 2^31-1",
                    (long long)n, (long long)(base * n));
    if (n > 1 && double(n) * double(p.B * p.H) * double(p.S_q) * double(p.d + 1) * 4.0 > 0x1p60)
        return fail(ATTN_ERR_INVALID_ARG, "n_split=%lld needs a workspace above 2^60 bytes",
                    (long long)n);
    out->n_split = n;
    out->kv_per_split = per;
    // One range runs the one-pass kernel without a workspace, except for
    // packed head groups, which only the split kernel computes.
    out->workspace_bytes = (n > 1 || p.pack > 1)
                               ? n * p.B * p.H * p.S_q * (p.d + 1) * int64_t(sizeof(float))
                               : 0;
    return ATTN_OK;
}

attn_status_t resolve_split(const Problem& p, int64_t n_split, SplitPlan* sp) {
    if (n_split < 0)
        return fail(ATTN_ERR_INVALID_ARG, "n_split must be >= 0 (0 = automatic), got %lld",
                    (long long)n_split);
    int sms = 0;
    if (n_split == 0) {
        int dev = 0;
        attn_status_t s = check_device(&dev);
        if (s != ATTN_OK) return s;
        sms = g_num_sms[dev].load();
    }
    return split_plan(p, n_split, sms, sp);
}

// Split-KV over general layouts: full attention (a bottom-right mask with one
// query row is the same thing); grouped heads pack into one query tile when
// their S_q rows fit in 128.
attn_status_t validate_split_general(Problem& p, const attn_fwd_params_t* a) {
    attn_status_t s = validate_general(p, a);
    if (s != ATTN_OK) return s;
    const bool full = a->mask == 0 || (a->mask == 2 && a->S_q == 1);
    if (!full)
        return fail(ATTN_ERR_UNSUPPORTED,
                    "split-KV computes full attention (mask 0, or the bottom-right mask with S_q = 1)");
    p.causal = false;
    p.causal_off = 0;
    const int64_t group = p.H / p.H_kv;
    p.pack = (group > 1 && p.S_q * group <= attn::kBlockM) ? group : 1;
    return ATTN_OK;
}

// ---------------------------------------------------------------- backward
using BwdLaunchFn = cudaError_t (*)(const attn::BwdArgs&, cudaStream_t);

BwdLaunchFn pick_bwd(int64_t d, bool bf16, bool causal) {
#define ATTN_PICK_BWD(D)                                                              \
    if (d == D) {                                                                     \
        if (bf16) return causal ? attn::launch_attn_bwd<D, true, true>                \
                                : attn::launch_attn_bwd<D, true, false>;              \
        return causal ? attn::launch_attn_bwd<D, false, true>                         \
                      : attn::launch_attn_bwd<D, false, false>;                       \
    }
    ATTN_PICK_BWD(64)
    ATTN_PICK_BWD(128)
    ATTN_PICK_BWD(256)
#undef ATTN_PICK_BWD
    return nullptr;
}

int64_t bwd_s_pad(const Problem& p) { return (p.S_q + 127) / 128 * 128; }

int64_t bwd_workspace_bytes(const Problem& p) { return 2 * p.B * p.H * bwd_s_pad(p) * 4; }

attn_status_t validate_bwd_head_dim(const Problem& p) {
    if (p.d != 64 && p.d != 128 && p.d != 256)
        return fail(ATTN_ERR_UNSUPPORTED,
                    "head_dim d=%lld not supported by the backward; must be one of [64, 128, 256]",
                    (long long)p.d);
    return ATTN_OK;
}

// Helper streams and events of the host-buffer entry point, created on a
// device's first attn_fwd_host call and kept for the life of the process.
struct HostPipe {
    static constexpr int kChunks = 8;
    // Chunk sizes in proportion to these weights (when there are at least
    // kWeightSum heads): the first and last chunks are a third of the others,
    // so the pipeline fills (first upload, nothing to overlap it) and drains
    // (last forward and download) sooner.  Measured with B=2, H=32, S=4096,
    // d=128: 1.186 ms per call against 1.227 ms with equal chunks; 10 or 12
    // chunks were slower.
    static constexpr int kWeight[kChunks] = {1, 3, 3, 3, 3, 3, 3, 1};
    static constexpr int kWeightSum = 20;
    std::mutex mu;
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, out_done = nullptr;
    cudaEvent_t in_done[kChunks] = {}, comp_done[kChunks] = {};
};
HostPipe g_pipes[kMaxDevices];

attn_status_t host_pipe(int dev, HostPipe** out) {
    HostPipe& pp = g_pipes[dev];
    std::lock_guard<std::mutex> lock(pp.mu);
    if (!pp.ready) {
        cudaError_t e = cudaStreamCreateWithFlags(&pp.in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&pp.out, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&pp.start, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&pp.out_done, cudaEventDisableTiming);
        for (int i = 0; i < HostPipe::kChunks && e == cudaSuccess; ++i) {
            e = cudaEventCreateWithFlags(&pp.in_done[i], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&pp.comp_done[i], cudaEventDisableTiming);
        }
        if (e != cudaSuccess)
            return fail(ATTN_ERR_CUDA, "creating the copy streams: %s", cudaGetErrorString(e));
        pp.ready = true;
    }
    *out = &pp;
    return ATTN_OK;
}

// One helper stream per device for the backward's dQ kernel (see BwdArgs).
struct BwdFork {
    std::mutex mu;
    bool ready = false;
    cudaStream_t aux = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
BwdFork g_bwd_fork[kMaxDevices];

attn_status_t bwd_fork(int dev, BwdFork** out) {
    BwdFork& f = g_bwd_fork[dev];
    std::lock_guard<std::mutex> lock(f.mu);
    if (!f.ready) {
        cudaError_t e = cudaStreamCreateWithFlags(&f.aux, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&f.fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&f.join, cudaEventDisableTiming);
        if (e != cudaSuccess)
            return fail(ATTN_ERR_CUDA, "creating the backward helper stream: %s",
                        cudaGetErrorString(e));
        f.ready = true;
    }
    *out = &f;
    return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t d, int causal,
                       float scale, attn_dtype_t dtype, struct CUstream_st* stream) {
    Problem p;
    attn_status_t s = validate_sizes(p, B, H, S_q, S_k, d, causal, scale, dtype);
    if (s != ATTN_OK) return s;
    if ((s = validate_device_ptrs(p, q, k, v, o, lse)) != ATTN_OK) return s;
    return launch_checked(p, q, k, v, o, lse, stream);
}

attn_status_t attn_fwd_general(const attn_fwd_params_t* params, struct CUstream_st* stream) {
    Problem p;
    attn_status_t s = validate_general(p, params);
    if (s != ATTN_OK) return s;
    if ((s = validate_device_ptrs(p, params->q, params->k, params->v, params->o, params->lse)) != ATTN_OK)
        return s;
    return launch_checked(p, params->q, params->k, params->v, params->o, params->lse, stream);
}

attn_status_t attn_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                            void* o_host, float* lse_host, void* q_dev, void* k_dev, void* v_dev,
                            void* o_dev, float* lse_dev, int64_t B, int64_t H, int64_t S_q,
                            int64_t S_k, int64_t d, int causal, float scale, attn_dtype_t dtype,
                            struct CUstream_st* stream) {
    Problem p;
    attn_status_t s = validate_sizes(p, B, H, S_q, S_k, d, causal, scale, dtype);
    if (s != ATTN_OK) return s;
    if (!q_host) return fail(ATTN_ERR_INVALID_ARG, "q_host is null");
    if (!k_host) return fail(ATTN_ERR_INVALID_ARG, "k_host is null");
    if (!v_host) return fail(ATTN_ERR_INVALID_ARG, "v_host is null");
    if (!o_host) return fail(ATTN_ERR_INVALID_ARG, "o_host is null");
    if (!lse_host) return fail(ATTN_ERR_INVALID_ARG, "lse_host is null");
    if ((s = validate_device_ptrs(p, q_dev, k_dev, v_dev, o_dev, lse_dev)) != ATTN_OK) return s;
    if (overlaps(q_dev, p.q_bytes, k_dev, p.kv_bytes) || overlaps(q_dev, p.q_bytes, v_dev, p.kv_bytes) ||
        overlaps(k_dev, p.kv_bytes, v_dev, p.kv_bytes))
        return fail(ATTN_ERR_INVALID_ARG, "q_dev, k_dev and v_dev must not overlap (they are copy targets)");
    int dev = 0;
    if ((s = check_device(&dev)) != ATTN_OK) return s;
    HostPipe* pipe = nullptr;
    if ((s = host_pipe(dev, &pipe)) != ATTN_OK) return s;
    std::lock_guard<std::mutex> lock(pipe->mu);

    // Heads are independent problems, so the call is cut into chunks of
    // consecutive (b, h): chunk c's upload (helper stream `in`), its forward
    // (the caller's stream) and its download (helper stream `out`) overlap
    // with those of its neighbours.  Dense layouts keep each chunk contiguous.
    const int64_t BH = B * H;
    const size_t total = p.q_bytes + 2 * p.kv_bytes + p.o_bytes;
    const int64_t chunks = total < (size_t(32) << 20) ? 1 : std::min<int64_t>(HostPipe::kChunks, BH);
    const bool weighted = chunks == HostPipe::kChunks && BH >= HostPipe::kWeightSum;
    auto bound = [&](int64_t c) -> int64_t {      // first (b, h) of chunk c
        if (!weighted) return BH * c / chunks;
        int64_t w = 0;
        for (int64_t i = 0; i < c; ++i) w += HostPipe::kWeight[i];
        return BH * w / HostPipe::kWeightSum;
    };
    const size_t q_head = static_cast<size_t>(S_q * d * 2), kv_head = static_cast<size_t>(S_k * d * 2);
    const size_t l_head = static_cast<size_t>(S_q * 4);
    cudaError_t e;
    auto cuda_fail = [&](const char* what) {
        return fail(ATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    };
    // The helper streams start after everything already queued on `stream`.
    if ((e = cudaEventRecord(pipe->start, stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(pipe->in, pipe->start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(pipe->out, pipe->start, 0)) != cudaSuccess)
        return cuda_fail("ordering the copy streams");
    for (int64_t c = 0; c < chunks; ++c) {
        const int64_t h0 = bound(c), h1 = bound(c + 1);
        const size_t n = static_cast<size_t>(h1 - h0);
        auto at = [&](const void* base, size_t per_head) {
            return static_cast<const char*>(base) + static_cast<size_t>(h0) * per_head;
        };
        if ((e = cudaMemcpyAsync(const_cast<char*>(at(q_dev, q_head)), at(q_host, q_head), n * q_head,
                                 cudaMemcpyHostToDevice, pipe->in)) != cudaSuccess ||
            (e = cudaMemcpyAsync(const_cast<char*>(at(k_dev, kv_head)), at(k_host, kv_head), n * kv_head,
                                 cudaMemcpyHostToDevice, pipe->in)) != cudaSuccess ||
            (e = cudaMemcpyAsync(const_cast<char*>(at(v_dev, kv_head)), at(v_host, kv_head), n * kv_head,
                                 cudaMemcpyHostToDevice, pipe->in)) != cudaSuccess ||
            (e = cudaEventRecord(pipe->in_done[c], pipe->in)) != cudaSuccess)
            return cuda_fail("host-to-device copy");
    }
    for (int64_t c = 0; c < chunks; ++c) {
        const int64_t h0 = bound(c), h1 = bound(c + 1);
        const size_t n = static_cast<size_t>(h1 - h0);
        auto at = [&](const void* base, size_t per_head) {
            return const_cast<char*>(static_cast<const char*>(base) + static_cast<size_t>(h0) * per_head);
        };
        Problem pc;
        if ((s = validate_sizes(pc, 1, h1 - h0, S_q, S_k, d, causal, scale, dtype)) != ATTN_OK) return s;
        if ((e = cudaStreamWaitEvent(stream, pipe->in_done[c], 0)) != cudaSuccess)
            return cuda_fail("ordering the forward");
        if ((s = launch_checked(pc, at(q_dev, q_head), at(k_dev, kv_head), at(v_dev, kv_head),
                                at(o_dev, q_head), reinterpret_cast<float*>(at(lse_dev, l_head)),
                                stream)) != ATTN_OK)
            return s;
        if ((e = cudaEventRecord(pipe->comp_done[c], stream)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(pipe->out, pipe->comp_done[c], 0)) != cudaSuccess)
            return cuda_fail("ordering the download");
        if ((e = cudaMemcpyAsync(at(o_host, q_head), at(o_dev, q_head), n * q_head,
                                 cudaMemcpyDeviceToHost, pipe->out)) != cudaSuccess ||
            (e = cudaMemcpyAsync(at(lse_host, l_head), at(lse_dev, l_head), n * l_head,
                                 cudaMemcpyDeviceToHost, pipe->out)) != cudaSuccess)
            return cuda_fail("device-to-host copy");
    }
    // `stream` reaches this point only once every download has finished.
    if ((e = cudaEventRecord(pipe->out_done, pipe->out)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(stream, pipe->out_done, 0)) != cudaSuccess)
        return cuda_fail("joining the copy streams");
    return ok();
}

attn_status_t attn_fwd_plan(int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t d, int causal,
                            attn_dtype_t dtype, attn_plan_t* plan) {
    if (!plan) return fail(ATTN_ERR_INVALID_ARG, "plan is null");
    Problem p;
    attn_status_t s = validate_sizes(p, B, H, S_q, S_k, d, causal, 1.0f, dtype);
    if (s != ATTN_OK) return s;
    fill_plan(p, plan);
    return ok();
}

attn_status_t attn_fwd_splitkv_plan(int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t d,
                                    attn_dtype_t dtype, int64_t n_split, int64_t* n_split_used,
                                    int64_t* workspace_bytes) {
    if (!n_split_used) return fail(ATTN_ERR_INVALID_ARG, "n_split_used is null");
    if (!workspace_bytes) return fail(ATTN_ERR_INVALID_ARG, "workspace_bytes is null");
    Problem p;
    attn_status_t s = validate_sizes(p, B, H, S_q, S_k, d, 0, 1.0f, dtype);
    if (s != ATTN_OK) return s;
    SplitPlan sp;
    if ((s = resolve_split(p, n_split, &sp)) != ATTN_OK) return s;
    *n_split_used = sp.n_split;
    *workspace_bytes = sp.workspace_bytes;
    return ok();
}

attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                               int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t d,
                               float scale, attn_dtype_t dtype, int64_t n_split, void* workspace,
                               int64_t workspace_bytes, struct CUstream_st* stream) {
    Problem p;
    attn_status_t s = validate_sizes(p, B, H, S_q, S_k, d, 0, scale, dtype);
    if (s != ATTN_OK) return s;
    if ((s = validate_device_ptrs(p, q, k, v, o, lse)) != ATTN_OK) return s;
    SplitPlan sp;
    if ((s = resolve_split(p, n_split, &sp)) != ATTN_OK) return s;
    if (sp.n_split == 1) return launch_checked(p, q, k, v, o, lse, stream);
    if (!workspace) return fail(ATTN_ERR_INVALID_ARG, "workspace is null");
    if (!aligned(workspace, 16)) return fail(ATTN_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
    if (workspace_bytes < sp.workspace_bytes)
        return fail(ATTN_ERR_INVALID_ARG, "workspace_bytes=%lld is below the %lld bytes %lld ranges need",
                    (long long)workspace_bytes, (long long)sp.workspace_bytes, (long long)sp.n_split);
    const size_t wb = static_cast<size_t>(sp.workspace_bytes);
    if (overlaps(workspace, wb, q, p.q_bytes)) return fail(ATTN_ERR_INVALID_ARG, "workspace overlaps q");
    if (overlaps(workspace, wb, k, p.kv_bytes)) return fail(ATTN_ERR_INVALID_ARG, "workspace overlaps k");
    if (overlaps(workspace, wb, v, p.kv_bytes)) return fail(ATTN_ERR_INVALID_ARG, "workspace overlaps v");
    if (overlaps(workspace, wb, o, p.o_bytes)) return fail(ATTN_ERR_INVALID_ARG, "workspace overlaps o");
    if (overlaps(workspace, wb, lse, p.lse_bytes)) return fail(ATTN_ERR_INVALID_ARG, "workspace overlaps lse");
    int dev = 0;
    if ((s = check_device(&dev)) != ATTN_OK) return s;
    attn::FwdArgs a;
    if ((s = fill_args(a, p, dev, q, k, v, o, lse)) != ATTN_OK) return s;
    const int64_t rows = p.B * p.H * p.S_q;
    a.n_split = static_cast<int32_t>(sp.n_split);
    a.kv_per_split = static_cast<int32_t>(sp.kv_per_split);
    a.o_part = static_cast<float*>(workspace);
    a.lse_part = a.o_part + sp.n_split * rows * p.d;
    LaunchFn fn = pick_split(p.d, p.dtype == ATTN_DTYPE_BF16);
    if (!fn) return fail(ATTN_ERR_UNSUPPORTED, "no kernel for d=%lld", (long long)p.d);
    cudaError_t e = fn(a, stream);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    e = attn::launch_attn_combine(a.o_part, a.lse_part, o, lse, a.n_split, rows,
                                  static_cast<int>(p.d), p.dtype == ATTN_DTYPE_BF16,
                                  static_cast<int>(p.H), static_cast<int>(p.S_q),
                                  attn::RowLayout{p.lo.batch, p.lo.head, p.lo.row}, stream);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "combine launch: %s", cudaGetErrorString(e));
    return ok();
}

attn_status_t attn_fwd_splitkv_general_plan(const attn_fwd_params_t* params, int64_t n_split,
                                            int64_t* n_split_used, int64_t* workspace_bytes) {
    if (!n_split_used) return fail(ATTN_ERR_INVALID_ARG, "n_split_used is null");
    if (!workspace_bytes) return fail(ATTN_ERR_INVALID_ARG, "workspace_bytes is null");
    Problem p;
    attn_status_t s = validate_split_general(p, params);
    if (s != ATTN_OK) return s;
    SplitPlan sp;
    if ((s = resolve_split(p, n_split, &sp)) != ATTN_OK) return s;
    *n_split_used = sp.n_split;
    *workspace_bytes = sp.workspace_bytes;
    return ok();
}

attn_status_t attn_fwd_splitkv_general(const attn_fwd_params_t* params, int64_t n_split,
                                       void* workspace, int64_t workspace_bytes,
                                       struct CUstream_st* stream) {
    Problem p;
    attn_status_t s = validate_split_general(p, params);
    if (s != ATTN_OK) return s;
    const void *q = params->q, *k = params->k, *v = params->v;
    void* o = params->o;
    float* lse = params->lse;
    if ((s = validate_device_ptrs(p, q, k, v, o, lse)) != ATTN_OK) return s;
    SplitPlan sp;
    if ((s = resolve_split(p, n_split, &sp)) != ATTN_OK) return s;
    if (sp.workspace_bytes == 0) return launch_checked(p, q, k, v, o, lse, stream);
    if (!workspace) return fail(ATTN_ERR_INVALID_ARG, "workspace is null");
    if (!aligned(workspace, 16)) return fail(ATTN_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
    if (workspace_bytes < sp.workspace_bytes)
        return fail(ATTN_ERR_INVALID_ARG, "workspace_bytes=%lld is below the %lld bytes %lld ranges need",
                    (long long)workspace_bytes, (long long)sp.workspace_bytes, (long long)sp.n_split);
    const size_t wb = static_cast<size_t>(sp.workspace_bytes);
    if (overlaps(workspace, wb, q, p.q_bytes)) return fail(ATTN_ERR_INVALID_ARG, "workspace overlaps q");
    if (overlaps(workspace, wb, k, p.kv_bytes)) return fail(ATTN_ERR_INVALID_ARG, "workspace overlaps k");
    if (overlaps(workspace, wb, v, p.v_bytes)) return fail(ATTN_ERR_INVALID_ARG, "workspace overlaps v");
    if (overlaps(workspace, wb, o, p.o_bytes)) return fail(ATTN_ERR_INVALID_ARG, "workspace overlaps o");
    if (overlaps(workspace, wb, lse, p.lse_bytes)) return fail(ATTN_ERR_INVALID_ARG, "workspace overlaps lse");
    int dev = 0;
    if ((s = check_device(&dev)) != ATTN_OK) return s;
    attn::FwdArgs a;
    if ((s = fill_args(a, p, dev, q, k, v, o, lse)) != ATTN_OK) return s;
    if (p.pack > 1) {
        // one box = the S_q rows of the pack query heads of a key/value head
        if ((s = encode_4d(&a.tm_q, q, p, p.S_q, p.H, p.lq, static_cast<uint32_t>(p.S_q), "q",
                           static_cast<uint32_t>(p.pack))) != ATTN_OK)
            return s;
        a.pack = static_cast<int32_t>(p.pack);
    }
    const int64_t rows = p.B * p.H * p.S_q;
    a.n_split = static_cast<int32_t>(sp.n_split);
    a.kv_per_split = static_cast<int32_t>(sp.kv_per_split);
    a.o_part = static_cast<float*>(workspace);
    a.lse_part = a.o_part + sp.n_split * rows * p.d;
    LaunchFn fn = pick_split(p.d, p.dtype == ATTN_DTYPE_BF16);
    if (!fn) return fail(ATTN_ERR_UNSUPPORTED, "no kernel for d=%lld", (long long)p.d);
    cudaError_t e = fn(a, stream);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    e = attn::launch_attn_combine(a.o_part, a.lse_part, o, lse, a.n_split, rows,
                                  static_cast<int>(p.d), p.dtype == ATTN_DTYPE_BF16,
                                  static_cast<int>(p.H), static_cast<int>(p.S_q),
                                  attn::RowLayout{p.lo.batch, p.lo.head, p.lo.row}, stream);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "combine launch: %s", cudaGetErrorString(e));
    return ok();
}

attn_status_t attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o,
                                       float* lse, int64_t B, int64_t H, int64_t S_q, int64_t S_k,
                                       int64_t d, float scale, attn_dtype_t dtype, int64_t n_split,
                                       struct CUstream_st* stream) {
    Problem p;
    attn_status_t s = validate_sizes(p, B, H, S_q, S_k, d, 0, scale, dtype);
    if (s != ATTN_OK) return s;
    if ((s = validate_device_ptrs(p, q, k, v, o, lse)) != ATTN_OK) return s;
    SplitPlan sp;
    if ((s = resolve_split(p, n_split, &sp)) != ATTN_OK) return s;
    if (sp.workspace_bytes > int64_t(ATTN_NOALLOC_SCRATCH_BYTES))
        return fail(ATTN_ERR_INVALID_ARG,
                    "%lld ranges need %lld bytes of scratch, above the built-in %lld bytes; "
                    "use a smaller n_split or attn_fwd_splitkv with a workspace",
                    (long long)sp.n_split, (long long)sp.workspace_bytes,
                    (long long)ATTN_NOALLOC_SCRATCH_BYTES);
    if (sp.n_split == 1) return launch_checked(p, q, k, v, o, lse, stream);
    int dev = 0;
    if ((s = check_device(&dev)) != ATTN_OK) return s;
    // The scratch's address on this device, looked up once with it current.
    void* scratch = g_noalloc_scratch[dev].load(std::memory_order_acquire);
    if (!scratch) {
        cudaError_t e = attn::noalloc_scratch_address(&scratch);
        if (e != cudaSuccess || !scratch)
            return fail(ATTN_ERR_CUDA, "cudaGetSymbolAddress(split-KV scratch): %s",
                        cudaGetErrorString(e));
        g_noalloc_scratch[dev].store(scratch, std::memory_order_release);
    }
    attn::FwdArgs a;
    if ((s = fill_args(a, p, dev, q, k, v, o, lse)) != ATTN_OK) return s;
    const int64_t rows = p.B * p.H * p.S_q;
    a.n_split = static_cast<int32_t>(sp.n_split);
    a.kv_per_split = static_cast<int32_t>(sp.kv_per_split);
    a.o_part = static_cast<float*>(scratch);
    a.lse_part = a.o_part + sp.n_split * rows * p.d;
    LaunchFn fn = pick_split(p.d, p.dtype == ATTN_DTYPE_BF16);
    if (!fn) return fail(ATTN_ERR_UNSUPPORTED, "no kernel for d=%lld", (long long)p.d);
    cudaError_t e = fn(a, stream);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    e = attn::launch_attn_combine(a.o_part, a.lse_part, o, lse, a.n_split, rows,
                                  static_cast<int>(p.d), p.dtype == ATTN_DTYPE_BF16,
                                  static_cast<int>(p.H), static_cast<int>(p.S_q),
                                  attn::RowLayout{p.lo.batch, p.lo.head, p.lo.row}, stream);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "combine launch: %s", cudaGetErrorString(e));
    return ok();
}

attn_status_t attn_bwd_workspace_size(int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t d,
                                      attn_dtype_t dtype, int64_t* workspace_bytes) {
    if (!workspace_bytes) return fail(ATTN_ERR_INVALID_ARG, "workspace_bytes is null");
    Problem p;
    attn_status_t s = validate_sizes(p, B, H, S_q, S_k, d, 0, 1.0f, dtype);
    if (s != ATTN_OK) return s;
    if ((s = validate_bwd_head_dim(p)) != ATTN_OK) return s;
    *workspace_bytes = bwd_workspace_bytes(p);
    return ok();
}

attn_status_t attn_bwd_general(const attn_bwd_params_t* a, struct CUstream_st* stream) {
    if (!a) return fail(ATTN_ERR_INVALID_ARG, "params is null");
    Problem p;
    attn_status_t s = validate_common(p, a->B, a->H, a->H_kv, a->S_q, a->S_k, a->d, a->mask,
                                      a->scale, a->dtype, a->q_layout, a->k_layout, a->v_layout,
                                      a->o_layout);
    if (s != ATTN_OK) return s;
    if ((s = validate_bwd_head_dim(p)) != ATTN_OK) return s;
    if ((s = check_layout(a->do_layout, "dout", p.d)) != ATTN_OK) return s;
    if ((s = check_layout(a->dq_layout, "dq", p.d)) != ATTN_OK) return s;
    if ((s = check_layout(a->dk_layout, "dk", p.d)) != ATTN_OK) return s;
    if ((s = check_layout(a->dv_layout, "dv", p.d)) != ATTN_OK) return s;
    if (!layout_injective(a->dq_layout, p.B, p.H, p.S_q, p.d))
        return fail(ATTN_ERR_INVALID_ARG, "dq layout maps two elements to one address");
    if (!layout_injective(a->dk_layout, p.B, p.H_kv, p.S_k, p.d))
        return fail(ATTN_ERR_INVALID_ARG, "dk layout maps two elements to one address");
    if (!layout_injective(a->dv_layout, p.B, p.H_kv, p.S_k, p.d))
        return fail(ATTN_ERR_INVALID_ARG, "dv layout maps two elements to one address");
    struct Buf {
        const void* ptr;
        size_t bytes;
        size_t align;
        const char* name;
        bool written;
    };
    const size_t wb = static_cast<size_t>(bwd_workspace_bytes(p));
    const Buf bufs[] = {
        {a->q, p.q_bytes, 16, "q", false},
        {a->k, p.kv_bytes, 16, "k", false},
        {a->v, p.v_bytes, 16, "v", false},
        {a->o, p.o_bytes, 16, "o", false},
        {a->lse, p.lse_bytes, 4, "lse", false},
        {a->dout, span_bytes(a->do_layout, p.B, p.H, p.S_q, p.d), 16, "dout", false},
        {a->dq, span_bytes(a->dq_layout, p.B, p.H, p.S_q, p.d), 16, "dq", true},
        {a->dk, span_bytes(a->dk_layout, p.B, p.H_kv, p.S_k, p.d), 16, "dk", true},
        {a->dv, span_bytes(a->dv_layout, p.B, p.H_kv, p.S_k, p.d), 16, "dv", true},
        {a->workspace, wb, 16, "workspace", true},
    };
    for (const Buf& b : bufs) {
        if (!b.ptr) return fail(ATTN_ERR_INVALID_ARG, "%s is null", b.name);
        if (!aligned(b.ptr, b.align))
            return fail(ATTN_ERR_INVALID_ARG, "%s is not %zu-byte aligned", b.name, b.align);
    }
    if (a->workspace_bytes < static_cast<int64_t>(wb))
        return fail(ATTN_ERR_INVALID_ARG, "workspace_bytes=%lld is below the %lld bytes needed",
                    (long long)a->workspace_bytes, (long long)wb);
    // Every written buffer must be disjoint from every other buffer.
    for (const Buf& w : bufs) {
        if (!w.written) continue;
        for (const Buf& x : bufs) {
            if (&x == &w) continue;
            if (overlaps(w.ptr, w.bytes, x.ptr, x.bytes))
                return fail(ATTN_ERR_INVALID_ARG, "%s overlaps %s", w.name, x.name);
        }
    }
    int dev = 0;
    if ((s = check_device(&dev)) != ATTN_OK) return s;
    attn::BwdArgs g;
    if ((s = encode_4d(&g.tm_k_fixed, a->k, p, p.S_k, p.H_kv, p.lk, 128, "k")) != ATTN_OK) return s;
    if ((s = encode_4d(&g.tm_v_fixed, a->v, p, p.S_k, p.H_kv, p.lv, 128, "v")) != ATTN_OK) return s;
    if ((s = encode_4d(&g.tm_q_step, a->q, p, p.S_q, p.H, p.lq, 64, "q")) != ATTN_OK) return s;
    if ((s = encode_4d(&g.tm_do_step, a->dout, p, p.S_q, p.H, a->do_layout, 64, "dout")) != ATTN_OK)
        return s;
    if ((s = encode_4d(&g.tm_q_fixed, a->q, p, p.S_q, p.H, p.lq, 128, "q")) != ATTN_OK) return s;
    if ((s = encode_4d(&g.tm_do_fixed, a->dout, p, p.S_q, p.H, a->do_layout, 128, "dout")) != ATTN_OK)
        return s;
    if (p.d == 256) {
        if ((s = encode_4d(&g.tm_k_step, a->k, p, p.S_k, p.H_kv, p.lk, 64, "k")) != ATTN_OK) return s;
        if ((s = encode_4d(&g.tm_v_step, a->v, p, p.S_k, p.H_kv, p.lv, 64, "v")) != ATTN_OK) return s;
    } else {
        if ((s = encode_4d(&g.tm_dk_out, a->dk, p, p.S_k, p.H_kv, a->dk_layout, 32, "dk")) != ATTN_OK)
            return s;
        if ((s = encode_4d(&g.tm_dv_out, a->dv, p, p.S_k, p.H_kv, a->dv_layout, 32, "dv")) != ATTN_OK)
            return s;
    }
    auto rl = [](const attn_layout_t& l) { return attn::RowLayout{l.batch, l.head, l.row}; };
    const int64_t s_pad = bwd_s_pad(p);
    g.o = a->o;
    g.dout = a->dout;
    g.lse = a->lse;
    g.lse2 = static_cast<float*>(a->workspace);
    g.delta = g.lse2 + p.B * p.H * s_pad;
    g.dq = a->dq;
    g.dk = a->dk;
    g.dv = a->dv;
    g.o_lay = rl(p.lo);
    g.do_lay = rl(a->do_layout);
    g.dq_lay = rl(a->dq_layout);
    g.dk_lay = rl(a->dk_layout);
    g.dv_lay = rl(a->dv_layout);
    g.S_q = static_cast<int32_t>(p.S_q);
    g.S_k = static_cast<int32_t>(p.S_k);
    g.BH = static_cast<int32_t>(p.B * p.H);
    g.S_pad = static_cast<int32_t>(s_pad);
    g.H = static_cast<int32_t>(p.H);
    g.kv_group = static_cast<int32_t>(p.H / p.H_kv);
    g.causal_off = static_cast<int32_t>(p.causal_off);
    g.scale = p.scale;
    g.scale_log2 = static_cast<float>(static_cast<double>(p.scale) * 1.4426950408889634);
    g.num_sms = g_num_sms[dev].load();
    g.device = dev;
    g.words = g_words_ptr[dev].load();
    g.launch_dkdv = next_launch(dev);
    g.launch_key2 = next_launch(dev);
    g.launch_dq = next_launch(dev);
    // seven S_q×S_k×d products of 2 flops per element between the kernels
    // (eight at d = 256)
    g.budget_ns = budget_ns(16.0 * double(p.B) * double(p.H) * double(p.S_q) * double(p.S_k) *
                            double(p.d));
    BwdLaunchFn fn = pick_bwd(p.d, p.dtype == ATTN_DTYPE_BF16, p.causal);
    if (!fn) return fail(ATTN_ERR_UNSUPPORTED, "no backward kernel for d=%lld", (long long)p.d);
    BwdFork* fork = nullptr;
    if ((s = bwd_fork(dev, &fork)) != ATTN_OK) return s;
    g.aux_stream = fork->aux;
    g.ev_fork = fork->fork;
    g.ev_join = fork->join;
    cudaError_t e;
    {
        std::lock_guard<std::mutex> lock(fork->mu);
        e = fn(g, stream);
    }
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "backward launch: %s", cudaGetErrorString(e));
    return ok();
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv,
                       int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t d, int causal,
                       float scale, attn_dtype_t dtype, void* workspace, int64_t workspace_bytes,
                       struct CUstream_st* stream) {
    if (causal != 0 && causal != 1)
        return fail(ATTN_ERR_INVALID_ARG, "causal must be 0 or 1, got %d", causal);
    const attn_layout_t lq = dense_layout(H, S_q, d), lk = dense_layout(H, S_k, d);
    attn_bwd_params_t a;
    a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse; a.dout = dout;
    a.dq = dq; a.dk = dk; a.dv = dv;
    a.B = B; a.H = H; a.H_kv = H; a.S_q = S_q; a.S_k = S_k; a.d = d;
    a.q_layout = lq; a.k_layout = lk; a.v_layout = lk; a.o_layout = lq;
    a.do_layout = lq; a.dq_layout = lq; a.dk_layout = lk; a.dv_layout = lk;
    a.mask = causal;
    a.scale = scale;
    a.dtype = dtype;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    return attn_bwd_general(&a, stream);
}

const char* attn_last_error(void) { return g_msg; }

attn_status_t attn_get_device_status(struct CUstream_st* stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
    int dev = 0;
    attn_status_t s = check_device(&dev);
    if (s != ATTN_OK) return s;
    attn::DeviceWords w{};
    e = cudaMemcpyFromSymbol(&w, g_attn_words, sizeof(w));
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "reading status: %s", cudaGetErrorString(e));
    const unsigned int v = w.status;
    if (v == 0 && w.abort_launch == 0) return ok();
    const attn::DeviceWords zero{};
    e = cudaMemcpyToSymbol(g_attn_words, &zero, sizeof(zero));
    if (e != cudaSuccess) return fail(ATTN_ERR_CUDA, "clearing status: %s", cudaGetErrorString(e));
    return fail(ATTN_ERR_TIMEOUT, "a bounded wait ran out in:%s%s%s%s%s%s%s%s%s%s%s",
                (v & 1u) ? " producer" : "", (v & 2u) ? " mma" : "", (v & 4u) ? " softmax" : "",
                (v & 8u) ? " epilogue" : "", (v & 16u) ? " drain" : "",
                (v & 32u) ? " bwd-producer" : "", (v & 64u) ? " bwd-mma" : "",
                (v & 128u) ? " bwd-softmax" : "", (v & 256u) ? " bwd-drain" : "",
                (v & 1024u) ? " bwd-epilogue" : "",
                (v & attn::sm100::kStatusDeadline) ? " (launch deadline passed)" : "");
}

int attn_version(void) { return kVersion; }

}  // extern "C"
