/*
 * attn_debug.h — failure-detection hooks of libattn_debug.so, a debug build of
 * the attention forward and backward kernels.  Not part of the attention
 * operation, and not exported by the release library libattn.so.
 *
 * libattn_debug.so compiles the release kernel source with its bounded waits
 * shortened from 2 s to 1 ms and with one hook: the TMA producer warp (the
 * forward's, or the backward dK/dV kernel's) can be told to issue no load for
 * one work unit and stop.  The consumers of that
 * unit then wait on barriers nothing completes, their waits run out, the CTA
 * records which roles gave up, tells the launch's other CTAs to stop, frees its
 * tensor memory and returns; the GPU context stays usable.  The CTAs' time
 * budget is an argument too, so a launch can be made to pass its deadline.
 * Tests use it to check that both are reported and that neither hangs.
 *
 * attn_debug_fwd — enqueue one full-attention forward on `stream` over dense
 *   bf16 q, k, v, o [B, H, S, 64] (device, 16-byte aligned) and fp32 lse
 *   [B, H, S], scaled by `scale`.  skip_unit: the work unit (one head and 256
 *   query rows, numbered head-major) whose loads the producer skips, or -1 for
 *   none (then the call computes the forward like attn_fwd).  budget_ns: each
 *   CTA's time budget, after which its producer stops it and the launch (0: 5 s,
 *   far above any real duration).  Returns 0, or a cudaError_t value (1 for
 *   bad arguments).
 * attn_debug_bwd — enqueue one full-attention backward on `stream` (the prep,
 *   dK/dV and dQ kernels, one after the other) over dense bf16 q, k, v, o,
 *   dout, dq, dk, dv [B, H, S, 64] (device, 16-byte aligned), fp32 lse
 *   [B, H, S] from the forward, and a device workspace of 2·B·H·S_pad floats
 *   (S_pad = S rounded up to 128).  skip_unit: the dK/dV kernel's work unit
 *   (one head and 128 keys, numbered head-major) whose loads its producer
 *   skips, or -1 for none (then the call computes the backward like
 *   attn_bwd).  budget_ns: as for attn_debug_fwd.  Returns 0, or a
 *   cudaError_t value (1 for bad arguments).
 * attn_debug_status — synchronise `stream`, write the debug library's status
 *   word (forward roles — bit 1: producer, 2: MMA, 4: softmax, 8: epilogue,
 *   16: drain; backward roles — 32: producer, 64: MMA, 128: softmax, 256:
 *   drain, 1024: epilogue; 512: deadline; 0 when no wait ran out) to *status
 *   and clear it.  Returns 0 or a cudaError_t value.
 */
#ifndef ATTN_GB300_ATTN_DEBUG_H_
#define ATTN_GB300_ATTN_DEBUG_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;

int attn_debug_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                   int64_t H, int64_t S, float scale, int skip_unit, uint64_t budget_ns,
                   struct CUstream_st* stream);
int attn_debug_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, void* dq, void* dk, void* dv, float* workspace, int64_t B,
                   int64_t H, int64_t S, float scale, int skip_unit, uint64_t budget_ns,
                   struct CUstream_st* stream);
int attn_debug_status(unsigned int* status, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_DEBUG_H_ */
