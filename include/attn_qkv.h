/*
 * attn_qkv.h -- C ABI of the fused QKV producer on GB300 (sm_103a): the launch
 * that makes the attention forward's inputs (attn_fwd.h) in their layouts.
 *
 * On the page ".../Coppelius/Build/Graph.alpha" a layer's attention inputs
 * come from the QKV product of the normed activations with the QKV matrix,
 * then a "qk-rope" launch (rotary embedding of the query and key heads with
 * the cosine and sine tables) and a "value-transpose" launch.  Here one kernel
 * does all three: the product runs on the tensor cores and its epilogue
 * rotates, rounds and writes Q, K and V^T directly.  For token t:
 *
 *   y[t][n] = sum_i X[t][i] W[n][i]                n < (heads + 2 kv_heads) * 64
 *
 * parts in the order Q (heads * 64 outputs), K (kv_heads * 64), V
 * (kv_heads * 64), head h of a part at its outputs h*64 .. h*64 + 63.  Query
 * and key heads are rotated pair by pair, pair p being elements (2p, 2p + 1):
 * with c = cosines[t][p], s = sines[t][p], (a, b) -> (a c - b s, a s + b c).
 * The product and the rotation are binary32; each output is rounded once to
 * binary16 (round to nearest even).
 *
 * Layouts (row-major):
 *   x        binary16 [T][width]                      (the normed activations)
 *   w        binary16 [(heads + 2 kv_heads) * 64][width]  (output-major)
 *   cosines  binary32 [T][32]    sines  binary32 [T][32]  (the rotary tables)
 *   q        binary16 [heads][T][64]                  -- output
 *   k        binary16 [kv_heads][T][64]               -- output
 *   vT       binary16 [kv_heads][64][T]               -- output
 *
 * Ownership: the caller owns every buffer; the library allocates a 4-byte
 * status word per device on first use.  Errors: an attn_status (attn_fwd.h);
 * argument errors are detected on the host before anything is launched.
 */
#ifndef ATTN_QKV_H
#define ATTN_QKV_H

#include <stddef.h>

#include "attn_fwd.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_qkv_rope -- the fused QKV producer on device buffers.
 *
 * x, w, cosines, sines, q, k, vT: device pointers, 16-byte aligned, layouts
 *   above.
 * T: tokens; T > 0 and T % 64 == 0 (the attention's admission).
 * width: the input width; width > 0 and width % 64 == 0.
 * heads, kv_heads: heads > 0, kv_heads > 0, heads % kv_heads == 0,
 *   heads <= 65535, and heads * 64 * T * 4 <= 2^32 - 1.
 * stream: the stream to run on.
 *
 * Returns ATTN_OK once the kernel is queued; ATTN_EINVAL, ATTN_EALIGN or
 * ATTN_EOVERLAP (an output overlaps an input or another output) before
 * anything is queued; ATTN_EDEVICE without a suitable device; ATTN_ELAUNCH
 * if the runtime rejects the launch.  Every element of q, k and vT is
 * written.  A wait inside the kernel that gives up after 1 s is reported by
 * attn_qkv_last_device_status.
 */
int attn_qkv_rope(const void *x, const void *w, const float *cosines, const float *sines,
                  void *q, void *k, void *vT, int T, int width, int heads, int kv_heads,
                  cudaStream_t stream);

/*
 * attn_qkv_last_device_status -- synchronises `stream`, then returns and
 * clears the current device's status word of this kernel: ATTN_OK, or
 * ATTN_ETIMEOUT if a wait gave up since the last call.  ATTN_ELAUNCH if the
 * synchronisation reports a CUDA error.
 */
int attn_qkv_last_device_status(cudaStream_t stream);

/*
 * attn_qkv_test_inject_stall -- test hook for the producer's failure detection.
 *
 * The source pages have no counterpart of this entry point.  It makes the
 * next attn_qkv_rope call's first CTA skip the X half of its first shared-
 * memory stage.  The MMA warp's wait on that stage runs out after 1 s: the CTA
 * records a timeout, lets the copies it issued land, frees its tensor memory
 * and exits; the other CTAs run as usual (so that call's outputs are not
 * valid); attn_qkv_last_device_status then returns ATTN_ETIMEOUT, and later
 * calls run normally.  Always returns ATTN_OK.
 */
int attn_qkv_test_inject_stall(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_QKV_H */
