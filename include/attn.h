/*
 * attn.h — C ABI of the GB300 (sm_103a) exact attention forward library
 * (libattn.so).
 *
 * The operation (oxicuda-dnn 0.1.8, src/attn/flash_attn/hopper.rs, doc comment
 * of FlashAttention3Plan::generate_forward, and the kernel parameter list
 * built there):
 *
 *     S      = scale · Q · Kᵀ                 per (b, h), S_q × S_k
 *     S[i,j] = −∞ for j > i                   when causal (top-left aligned)
 *     O      = softmax_rows(S) · V
 *     LSE_i  = ln Σ_j exp(S[i,j])             natural log, scale included
 *
 * computed tile by tile with an online softmax, so the S_q × S_k matrix never
 * reaches device memory.
 *
 * Layout.  Q is [B, H, S_q, d]; K and V are [B, H, S_k, d]; O is [B, H, S_q, d];
 * all dense row-major (d contiguous) in the element type `dtype`.  LSE is
 * [B, H, S_q] fp32.  d ∈ {64, 128, 256} (SUPPORTED_HEAD_DIMS on the page).
 *
 * Ownership.  The caller owns every buffer.  The library allocates no device
 * memory (split-KV partials go to a caller workspace or to a static array
 * built into the library), keeps no pointer after a call returns, and
 * enqueues all device work on `stream` (NULL = the legacy default stream;
 * attn_fwd_host also uses two helper streams of its own, attn_bwd one, each
 * forked from and joined back to `stream`); calls return before
 * the work completes.  Forward kernels hand out their work units through the
 * GPU's own work queue (one CTA per unit; running CTAs cancel and take over
 * CTAs that have not started), so they keep no counter in device memory and
 * calls on different streams may run concurrently without coordination.
 *
 * Errors.  Argument checks happen on the host before anything is enqueued and
 * return a status; attn_last_error() then describes the offending argument
 * by name (as the page's validate_config does).
 *
 * Bounded execution.  No kernel of this library can hang its stream.  Every
 * wait inside a kernel gives up after 2 s; every CTA gives up once it has run
 * longer than a budget the host derives from the launch's work (5 s plus the
 * time the work would take at 10 TFLOP/s), checked in its waits and at the
 * head of each of its loops; and a CTA that gives up stops the rest of its
 * launch (CTAs that start later leave at once, running ones at their next
 * wait that lasts over 0.1 ms).  Such a launch returns early with its outputs
 * incomplete, and the next attn_get_device_status() reports ATTN_ERR_TIMEOUT.
 */
#ifndef ATTN_GB300_ATTN_H_
#define ATTN_GB300_ATTN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st*` */

typedef enum {
    ATTN_DTYPE_F16 = 0,
    ATTN_DTYPE_BF16 = 1
} attn_dtype_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* null or misaligned pointer, size < 1, overlap, non-finite scale, size too large */
    ATTN_ERR_UNSUPPORTED = 2, /* head_dim not in {64,128,256}, dtype not f16/bf16, no sm_103 device */
    ATTN_ERR_CUDA = 3,        /* a CUDA runtime or driver call failed (message has the CUDA error) */
    ATTN_ERR_TIMEOUT = 4      /* a kernel's bounded internal wait ran out (reported by attn_get_device_status) */
} attn_status_t;

/*
 * attn_plan_t — how attn_fwd would launch a problem (see attn_fwd_plan).
 * The page's plan object (FlashAttention3Plan::launch_params and
 * ::shared_memory_bytes) reports the same kind of figures for its design.
 */
typedef struct {
    int64_t block_m;          /* query rows per tile (128) */
    int64_t block_n;          /* keys per key/value tile (128) */
    int64_t q_tiles;          /* ceil(S_q / block_m): query tiles per (b, h) */
    int64_t kv_tiles;         /* ceil(S_k / block_n): key tiles per (b, h) */
    int64_t q_tiles_per_cta;  /* 2 for d <= 128 (ping-pong), 1 for d = 256 */
    int64_t bh;               /* B·H */
    int64_t units;            /* work units, bh · ceil(q_tiles / q_tiles_per_cta); the launch
                                 has one CTA per unit, of which about one per SM runs and
                                 takes the rest over through the GPU's work queue */
    int32_t threads;          /* threads per CTA */
    int32_t smem_bytes;       /* dynamic shared memory per CTA */
    int32_t tmem_cols;        /* tensor-memory columns allocated per CTA */
    int32_t kv_stages;        /* slots in the K/V shared-memory ring */
} attn_plan_t;

/*
 * attn_fwd_plan — fill *plan with the launch attn_fwd would use for these
 * sizes.  Host-only: validates the same size/dtype/scale-free arguments as
 * attn_fwd (same statuses and messages) and touches no device.  plan must
 * be non-null.
 */
attn_status_t attn_fwd_plan(int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t d, int causal,
                            attn_dtype_t dtype, attn_plan_t* plan);

/*
 * attn_fwd — enqueue the attention forward on `stream`.
 *
 *   q, k, v  device pointers, 16-byte aligned, element type `dtype`:
 *            q [B,H,S_q,d], k and v [B,H,S_k,d]
 *   o        device pointer, 16-byte aligned, [B,H,S_q,d] in `dtype`; written
 *   lse      device pointer, 4-byte aligned, [B,H,S_q] fp32; written
 *   B, H     batch and heads, >= 1, B·H <= 2^31 − 1
 *   S_q, S_k query and key lengths, 1 .. 2^22 (need not be tile multiples)
 *   d        head dimension: 64, 128 or 256
 *   causal   0 or 1; 1 masks key j for query i when j > i (top-left)
 *   scale    multiplier of Q·Kᵀ, any finite value (1/sqrt(d) is the usual;
 *            0 gives uniform weights, a negative scale favours the keys least
 *            aligned with the query)
 *   stream   CUDA stream
 *
 * o and lse must not overlap q, k, v or each other.  Returns ATTN_OK once the
 * kernel is enqueued.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t d, int causal,
                       float scale, attn_dtype_t dtype, struct CUstream_st* stream);

/*
 * General layouts (the page's kernel takes per-tensor batch and head strides:
 * stride_qb, stride_qh, stride_kb, ...).  An attn_layout_t gives, in
 * elements, the distance between consecutive batch entries, heads and
 * sequence positions of one tensor; the d elements of a position are
 * contiguous.  The dense [B, H, S, d] layout is {H·S·d, S·d, d}; a
 * [B, S, H, d] tensor is {S·H·d, d, H·d}; q, k and v may be views into one
 * packed [B, S, 3, H, d] allocation.
 */
typedef struct {
    int64_t batch, head, row;
} attn_layout_t;

typedef enum {
    ATTN_MASK_NONE = 0,
    ATTN_MASK_CAUSAL = 1,              /* key j visible to query i iff j <= i (top-left) */
    ATTN_MASK_CAUSAL_BOTTOM_RIGHT = 2  /* iff j <= i + S_k - S_q; needs S_q <= S_k */
} attn_mask_t;

typedef struct {
    const void* q;            /* [B, H, S_q, d] in q_layout */
    const void* k;            /* [B, H_kv, S_k, d] in k_layout */
    const void* v;            /* [B, H_kv, S_k, d] in v_layout */
    void* o;                  /* [B, H, S_q, d] in o_layout; written */
    float* lse;               /* [B, H, S_q] fp32, dense; written */
    int64_t B, H, H_kv, S_q, S_k, d;
    attn_layout_t q_layout, k_layout, v_layout, o_layout;
    int mask;                 /* attn_mask_t */
    float scale;
    attn_dtype_t dtype;
} attn_fwd_params_t;

/*
 * attn_fwd_general — attn_fwd over general layouts, grouped key/value heads
 * and a choice of causal alignment.
 *
 *   H_kv      key/value heads, dividing H: query head h reads key/value head
 *             h / (H / H_kv) (H_kv = H is plain multi-head attention).  The
 *             page has only H = H_kv; this generalisation changes which K/V
 *             a head reads, not the arithmetic.
 *   layouts   every stride a positive multiple of 8 elements (16 bytes, the
 *             tensor-map rule), row stride >= d; o's layout must not map two
 *             elements to one address.  Pointers 16-byte aligned (lse 4).
 *   mask      ATTN_MASK_NONE / _CAUSAL / _CAUSAL_BOTTOM_RIGHT (S_q <= S_k,
 *             else ATTN_ERR_UNSUPPORTED).
 *
 * o and lse must not overlap each other or the byte ranges q, k and v span
 * (inputs may overlap each other).  Errors as attn_fwd.
 */
attn_status_t attn_fwd_general(const attn_fwd_params_t* params, struct CUstream_st* stream);

/*
 * attn_fwd_splitkv_general_plan / attn_fwd_splitkv_general — the split-KV
 * forward (attn_fwd_splitkv) over general layouts and grouped key/value
 * heads.  `params` as attn_fwd_general with mask ATTN_MASK_NONE (or
 * ATTN_MASK_CAUSAL_BOTTOM_RIGHT with S_q = 1, which is the same); n_split,
 * workspace and its rules as attn_fwd_splitkv (the workspace size is the
 * same for the same B, H, S_q, d).  When H_kv < H and S_q·(H / H_kv) <= 128
 * the query rows of all heads that share a key/value head are computed in
 * one tile, so each key/value tile is read and multiplied once per group
 * (decoding with grouped-query attention); such packed groups always take
 * the split path, so their workspace is needed even for one range.
 */
attn_status_t attn_fwd_splitkv_general_plan(const attn_fwd_params_t* params, int64_t n_split,
                                            int64_t* n_split_used, int64_t* workspace_bytes);
attn_status_t attn_fwd_splitkv_general(const attn_fwd_params_t* params, int64_t n_split,
                                       void* workspace, int64_t workspace_bytes,
                                       struct CUstream_st* stream);

/*
 * attn_fwd_host — the same forward, for inputs and outputs in HOST memory.
 *
 * Copies q_host, k_host, v_host into the caller's device buffers q_dev,
 * k_dev, v_dev, runs attn_fwd on them into o_dev, lse_dev, and copies o_dev,
 * lse_dev back into o_host, lse_host.  Heads are independent, so problems
 * above 32 MB are cut into up to eight chunks of consecutive (b, h) whose
 * uploads, forwards and downloads overlap: the copies run on two helper
 * streams that the library creates on a device's first call (with a few
 * events; no memory is allocated) and orders after the work already on
 * `stream`; the forwards run on `stream`, which reaches the end of this call
 * only when every download has finished.  Host buffers should be page-locked
 * for the copies to be asynchronous.  Shapes, alignment and argument rules
 * are those of attn_fwd (device buffers as there; host buffers non-null).
 * Calls on one device are enqueued one at a time (a host lock); the results
 * are in o_host / lse_host once `stream` has reached this point.
 */
attn_status_t attn_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                            void* o_host, float* lse_host, void* q_dev, void* k_dev, void* v_dev,
                            void* o_dev, float* lse_dev, int64_t B, int64_t H, int64_t S_q,
                            int64_t S_k, int64_t d, int causal, float scale, attn_dtype_t dtype,
                            struct CUstream_st* stream);

/*
 * Split-KV forward (full attention, short S_q against long S_k).
 *
 * The same O and LSE as attn_fwd with causal = 0, computed with the keys of
 * every (b, h, query block) cut into n_split ranges of whole 128-key tiles so
 * that enough work units exist to fill the GPU when B·H·ceil(S_q/256) is small
 * (decoding).  Each range writes its normalised partial output O_s (fp32) and
 * its log-sum-exp LSE_s to the caller's workspace; a second kernel merges them
 * with LSE = ln Σ_s exp(LSE_s), O = Σ_s exp(LSE_s − LSE)·O_s.  The merge uses
 * only the LSE output the page's forward defines (oxicuda-dnn 0.1.8,
 * src/attn/flash_attn/hopper.rs, FlashAttention3Plan::generate_forward, final
 * step); the page itself has no split-KV scheme.  Rounding differs from
 * attn_fwd (the partial outputs are rounded to fp32, not to the output
 * dtype), within the same tolerance of the exact result.
 *
 * attn_fwd_splitkv_plan — ranges and workspace size for these sizes.
 *   n_split          0 = automatic: the count whose schedule over the current
 *                    device's SMs finishes first (queries the device); >= 1 =
 *                    that many ranges, capped at ceil(S_k/128) and reduced
 *                    so that no range is empty
 *   *n_split_used    ranges attn_fwd_splitkv will use (1 = the plain kernel
 *                    runs and no workspace is needed)
 *   *workspace_bytes n_split_used · B·H·S_q · (d + 1) · 4, or 0 when
 *                    n_split_used is 1
 * Validates like attn_fwd; n_split < 0 and null outputs are
 * ATTN_ERR_INVALID_ARG.  Only n_split = 0 touches the device.
 */
attn_status_t attn_fwd_splitkv_plan(int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t d,
                                    attn_dtype_t dtype, int64_t n_split, int64_t* n_split_used,
                                    int64_t* workspace_bytes);

/*
 * attn_fwd_splitkv — enqueue the split-KV forward on `stream`.
 *
 *   q, k, v, o, lse, B, H, S_q, S_k, d, scale, dtype, stream  as attn_fwd
 *                    (no causal argument: full attention only)
 *   n_split          as attn_fwd_splitkv_plan (the same device must be
 *                    current for n_split = 0, so both pick the same count)
 *   workspace        device pointer, 16-byte aligned, at least the
 *                    workspace_bytes attn_fwd_splitkv_plan reports; may be
 *                    null when that is 0.  Owned by the caller; written
 *                    before it is read on every call (nothing needs clearing),
 *                    must not overlap q, k, v, o or lse, and must not be used
 *                    by another call in flight at the same time
 *   workspace_bytes  size of `workspace` in bytes
 *
 * Launches two kernels (ranges, then merge) in order on `stream`, or the
 * attn_fwd kernel alone when one range is used.
 */
attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                               int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t d,
                               float scale, attn_dtype_t dtype, int64_t n_split, void* workspace,
                               int64_t workspace_bytes, struct CUstream_st* stream);

/*
 * Backward pass (oxicuda-dnn 0.1.8, src/attn/flash_attn/hopper.rs, doc comment
 * of FlashAttention3Plan::generate_backward, and its parameter list q, k, v,
 * o, do, lse, di, dq, dk, dv, sm_scale): with P recomputed from the saved LSE,
 *
 *     dV = Pᵀ·dO      dP = dO·Vᵀ      dS = P ∘ (dP − D),  D_i = Σ_c dO_ic·O_ic
 *     dQ = scale·dS·K                 dK = scale·dSᵀ·Q
 *
 * (the gradients of Σ O ∘ dO for the forward above; the scale follows from the
 * chain rule through scale·Q·Kᵀ).  dQ is produced by its own pass, not by
 * atomic adds, so results are deterministic.  head_dim 64, 128 or 256 (at
 * 256 the key side runs as two passes, dV then dK, each recomputing Sᵀ).
 *
 * attn_bwd_workspace_size — bytes of workspace attn_bwd needs:
 * 2 · B·H · S_pad · 4 with S_pad = S_q rounded up to a multiple of 128 (the
 * page's di vector and the LSE in base 2, padded to whole tiles).  Validates
 * like attn_fwd; touches no device.
 */
attn_status_t attn_bwd_workspace_size(int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t d,
                                      attn_dtype_t dtype, int64_t* workspace_bytes);

/*
 * attn_bwd — enqueue the backward on `stream`: a prep kernel, then the dK/dV
 * kernel (d = 256: a dV and a dK kernel) on `stream` and the dQ kernel, at the
 * same time, on a helper stream
 * that the library creates for the device on its first backward call (forked
 * from `stream` after the prep kernel and joined back before the call's end,
 * so `stream` sees one ordered operation).  A stream capture of `stream`
 * takes the helper stream in with it; keep other captures of attn_bwd on the
 * same device from overlapping it in time.
 *
 *   q, k, v    the forward's inputs (layouts as attn_fwd), device, 16-byte aligned
 *   o, lse     the forward's outputs for the same q, k, v, causal and scale
 *              (o 16-byte aligned, lse 4-byte aligned)
 *   dout       dO, the gradient of the loss with respect to o, [B,H,S_q,d]
 *   dq, dk, dv outputs, [B,H,S_q,d], [B,H,S_k,d], [B,H,S_k,d] in `dtype`,
 *              16-byte aligned; every element is written (key rows that no
 *              query sees get zeros)
 *   B .. dtype as attn_fwd
 *   workspace  device, 16-byte aligned, at least attn_bwd_workspace_size
 *              bytes; written before it is read (nothing needs clearing);
 *              calls in flight at the same time need separate workspaces
 *
 * dq, dk, dv and workspace must not overlap each other or any input.
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv,
                       int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t d, int causal,
                       float scale, attn_dtype_t dtype, void* workspace, int64_t workspace_bytes,
                       struct CUstream_st* stream);

/*
 * attn_bwd_general — attn_bwd over general layouts, grouped key/value heads
 * and a choice of causal alignment (the same rules as attn_fwd_general).  dk
 * and dv are the gradients of the H_kv key/value heads: each sums the
 * contributions of the H / H_kv query heads that read it.  Every output
 * layout must map distinct elements to distinct addresses; outputs and the
 * workspace must not overlap anything.  The workspace size is the one
 * attn_bwd_workspace_size reports for (B, H, S_q, S_k, d).
 */
typedef struct {
    const void* q;
    const void* k;
    const void* v;
    const void* o;            /* the forward's output for these inputs */
    const float* lse;         /* the forward's LSE, dense [B, H, S_q] */
    const void* dout;         /* dO, [B, H, S_q, d] in do_layout */
    void* dq;                 /* [B, H, S_q, d] in dq_layout; written */
    void* dk;                 /* [B, H_kv, S_k, d] in dk_layout; written */
    void* dv;                 /* [B, H_kv, S_k, d] in dv_layout; written */
    int64_t B, H, H_kv, S_q, S_k, d;
    attn_layout_t q_layout, k_layout, v_layout, o_layout, do_layout, dq_layout, dk_layout,
        dv_layout;
    int mask;                 /* attn_mask_t */
    float scale;
    attn_dtype_t dtype;
    void* workspace;
    int64_t workspace_bytes;
} attn_bwd_params_t;

attn_status_t attn_bwd_general(const attn_bwd_params_t* params, struct CUstream_st* stream);

/*
 * attn_fwd_splitkv_noalloc — attn_fwd_splitkv without a caller workspace and
 * without allocating anything.
 *
 * The page has no counterpart to this entry point: it is a library service.
 * It is for callers that cannot allocate device memory on the call path:
 * code that runs under a fixed, pre-reserved memory budget, or that holds no
 * device allocator of its own (a plain C caller), or that must not call
 * cudaMalloc/cudaFree between launches because cudaFree synchronises the
 * device and either call can fail at run time.  Instead of a workspace the
 * partial results go to a scratch array built into the library: a static
 * device array of ATTN_NOALLOC_SCRATCH_BYTES (16 MiB) on each device, whose
 * address is looked up once per device.
 *
 *   q, k, v, o, lse, B, H, S_q, S_k, d, scale, dtype, n_split, stream
 *                    as attn_fwd_splitkv
 *
 * Sizes whose plan (attn_fwd_splitkv_plan with the same arguments) needs
 * more than ATTN_NOALLOC_SCRATCH_BYTES of workspace are rejected with
 * ATTN_ERR_INVALID_ARG before anything is enqueued; choose a smaller n_split
 * or use attn_fwd_splitkv.  A plan of one range needs no scratch.
 *
 * First call on a device: it looks up the scratch's device address (a CUDA
 * runtime call, cudaGetSymbolAddress, which may load the array's module) with
 * that device current.  Make that first call before any stream capture
 * starts; later calls on the device make no such lookup.
 *
 * Nothing in the scratch needs to start at zero: every call writes the
 * partial results it reads.  The scratch is shared by every call on the
 * device, so two calls whose work overlaps in time (different streams, or
 * different host threads without ordering between their streams) race on it
 * and may return wrong results; order them (one stream, or events).
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (16 * 1024 * 1024)

attn_status_t attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o,
                                       float* lse, int64_t B, int64_t H, int64_t S_q, int64_t S_k,
                                       int64_t d, float scale, attn_dtype_t dtype, int64_t n_split,
                                       struct CUstream_st* stream);

/*
 * attn_last_error — message for the last non-OK status returned on this host
 * thread ("" if none).  The string stays valid until the next call on this
 * thread.
 */
const char* attn_last_error(void);

/*
 * attn_get_device_status — synchronise `stream`, then read and clear the
 * current device's status words (shared by the forward and backward kernels).
 * ATTN_OK if every kernel since the last read finished its waits;
 * ATTN_ERR_TIMEOUT if one gave up (the message names the roles, and says when
 * a CTA passed its launch's deadline); ATTN_ERR_CUDA if the synchronisation
 * itself failed.  A launch captured in a CUDA graph keeps its launch number,
 * so after a replay that gave up, later replays of the same graph stop at
 * once until this call clears the words.
 */
attn_status_t attn_get_device_status(struct CUstream_st* stream);

/* attn_version — library version, major·10000 + minor·100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H_ */
