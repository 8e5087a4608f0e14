/*
 * attn_bwd.h -- C ABI of the GB300 (sm_103a) backward pass of the causal
 * grouped-query attention whose forward attn_fwd.h declares.
 *
 * The operation is the backward statement of the page
 * "Realization/Nvidia/SM86/StreamingAttentionSM86.alpha" (the comment that
 * opens its backward pass, before the query launch).  With the forward's
 * output O and base-2 log-sum-exp L, for query head h (K/V head
 * g = floor(h / (heads / kv_heads))), query row i and key j <= i:
 *
 *   P_ij  = 2^(c * sum_e Q[h][i][e] K[g][j][e] - L[h][i])    (0 for j > i)
 *   dP_ij = sum_e dO[i][h*64 + e] V^T[g][e][j]
 *   D_i   = sum_e dO[i][h*64 + e] O[i][h*64 + e]
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ[h][i][e]  = s sum_j dS_ij K[g][j][e]
 *   dK[g][j][e]  = s sum over the group's heads h and rows i of dS_ij Q[h][i][e]
 *   dVT[g][e][j] = sum over the group's heads h and rows i of P_ij dO[i][h*64 + e]
 *
 * with s the natural score scale (1/8 for head width 64; c = s / ln 2 is the
 * forward's).  As on that page P and dS are rounded to binary16 for their
 * products and every sum is binary32.  The page writes one dK / dV^T plane per
 * query head and sums each group's planes in a separate reduce launch; here
 * the key kernel walks the whole group, so the sum happens in its accumulator
 * and the results land directly in the compact K/V layout.
 *
 * Layouts (row-major; the forward's, plus dO in O's token-major layout):
 *   q    binary16 [heads][T][64]         k   binary16 [kv_heads][T][64]
 *   vT   binary16 [kv_heads][64][T]      o   binary16 [T][heads*64]  (forward's O)
 *   lse  binary32 [heads][T]             dO  binary16 [T][heads*64]
 *   dq   binary32 [heads][T][64]                 -- output
 *   dk   binary32 [kv_heads][T][64]              -- output
 *   dvT  binary32 [kv_heads][64][T]              -- output
 *
 * Ownership: the caller owns every buffer, including `workspace`, where the
 * call keeps the row terms D (binary32 [heads][T]) between its launches and,
 * for short problems, partial dK and dV^T planes (below).  The library
 * allocates a 4-byte status word per device on first use and never frees it;
 * nothing is allocated per call.
 *
 * Short problems: the key launch has one unit per (K/V head, 128-key tile),
 * each walking every query head of its group over every later query tile.
 * When that gives fewer than 128 units, a group of two or more heads and a
 * longest walk of at least 16 steps (group * ceil(T / 128)), each pair's steps
 * are shared out over S = min(group, ceil(256 / units), 8) units that write
 * partial sums into the workspace, and a third launch adds the S planes in a
 * fixed order (so results stay deterministic, and differ from the unsplit sum
 * only by the order of the binary32 additions).  S depends on the shape only.
 *
 * Errors: every entry point returns an attn_status (attn_fwd.h).  Argument
 * errors are detected on the host before anything is launched.  The launches
 * (the query kernel, the key kernel, and for short problems the sum of the
 * partial planes) are asynchronous and ordered on `stream`.
 */
#ifndef ATTN_BWD_H
#define ATTN_BWD_H

#include <stddef.h>

#include "attn_fwd.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_bwd_workspace_bytes -- device bytes attn_bwd needs as `workspace` for
 * the given shape, or 0 if the shape is not admitted: heads * T * 4 rounded up
 * to 256 bytes, plus, for the short problems whose key launch is split (above),
 * two arrays of S partial planes of kv_heads * T * 64 binary32 values, each
 * rounded up to 256 bytes.
 */
size_t attn_bwd_workspace_bytes(int T, int heads, int kv_heads);

/*
 * attn_bwd -- the backward pass on device buffers.
 *
 * q, k, vT, o, lse, dO: device pointers, 16-byte aligned, layouts above; o and
 *   lse are what attn_fwd wrote for q, k, vT and c.
 * dq, dk, dvT: device pointers, 16-byte aligned; every element is written.
 * T, heads, kv_heads: as attn_fwd (T > 0, T % 64 == 0, heads % kv_heads == 0,
 *   heads <= 65535, heads * 64 * T * 4 <= 2^32 - 1).
 * c: the forward's scale (finite, > 0); s: the natural scale (finite, > 0).
 * workspace: device buffer of at least attn_bwd_workspace_bytes bytes,
 *   256-byte aligned; its contents on entry do not matter.
 * stream: the stream to run on.
 *
 * Returns ATTN_OK once the launches are queued; ATTN_EINVAL (a size, a scale,
 * a NULL pointer or a short workspace), ATTN_EALIGN or ATTN_EOVERLAP (an
 * output or the workspace overlaps an input or another output) before
 * anything is queued; ATTN_EDEVICE without a suitable device; ATTN_ELAUNCH if
 * the runtime rejects a launch.  A wait inside the kernels that gives up
 * after 1 s is reported by attn_bwd_last_device_status.
 */
int attn_bwd(const void *q, const void *k, const void *vT, const void *o,
             const float *lse, const void *dO, float *dq, float *dk, float *dvT,
             int T, int heads, int kv_heads, float c, float s,
             void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * attn_bwd_last_device_status -- synchronises `stream`, then returns and
 * clears the current device's backward status word: ATTN_OK, or ATTN_ETIMEOUT
 * if a wait inside a backward kernel gave up since the last call (the
 * outputs of that call are then not valid).  ATTN_ELAUNCH if the
 * synchronisation reports a CUDA error.
 */
int attn_bwd_last_device_status(cudaStream_t stream);

/*
 * attn_bwd_test_inject_stall -- test hook for the backward's failure detection.
 *
 * The source pages have no counterpart of this entry point.  It makes the
 * next attn_bwd call's query launch skip the first K/V copy of its first CTA.
 * The wait on that copy runs out after 1 s: the CTA records a timeout, drains
 * what it issued, frees its tensor memory and exits; the key launch runs as
 * usual (on that CTA's missing row terms, so the call's outputs are not
 * valid); attn_bwd_last_device_status then returns ATTN_ETIMEOUT, and later
 * calls run normally.  Always returns ATTN_OK.
 */
int attn_bwd_test_inject_stall(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_BWD_H */
