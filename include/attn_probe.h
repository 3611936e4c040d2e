/*
 * attn_probe.h — measurement helper exported by libattn.so (not part of the
 * attention operation).
 *
 * attn_probe_ex2 — enqueue `blocks` blocks of 256 threads, each thread
 * evaluating 8 × `iters` ex2.approx.f32 in 8 independent chains, and write one
 * float per thread to `out` (device, blocks·256 floats).  Timing it gives the
 * exp2 throughput of the MUFU pipe, the secondary ceiling of the softmax.
 * Returns 0, 1 for bad arguments, 3 if the launch failed.
 */
#ifndef ATTN_GB300_ATTN_PROBE_H_
#define ATTN_GB300_ATTN_PROBE_H_

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;

int attn_probe_ex2(float* out, int blocks, int iters, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_PROBE_H_ */
