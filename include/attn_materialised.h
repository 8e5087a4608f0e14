/*
 * attn_materialised.h -- C ABI of the materialised causal grouped-query
 * attention forward on GB300 (sm_103a): the prior design the page
 * "Realization/Nvidia/SM86/StreamingAttentionSM86.alpha" replaces, kept as a
 * second workload to cross-check the streaming forward.
 *
 * It computes what attn_fwd computes (attn_fwd.h), in three launches through
 * planes in the caller's workspace, as the page ".../Coppelius/Build/Graph.alpha"
 * lays out its attention before the streaming kernels (a binary32 scores plane
 * of heads x T x T, a "softmax-forward" launch writing binary16 probabilities,
 * then their product with V):
 *
 *   1. S[h][i][j] = sum_e Q[h][i][e] K[g][j][e]        binary32, key tiles j <= i's tile
 *   2. per row: t = S c, m = max_{j<=i} t, l = sum_{j<=i} 2^(t - m),
 *      P[h][i][j] = 2^(t_j - m) / l rounded to binary16 (0 for j > i),
 *      LSE[h][i] = m + log2 l
 *   3. O[i][h*64 + e] = sum_j P[h][i][j] V^T[g][e][j]    rounded to binary16
 *
 * Here the probabilities are normalised before the binary16 rounding (the
 * materialised path rounds its probabilities); the streaming forward rounds
 * 2^(t - m) and divides by l at the end.  Both stay within the tolerance of
 * the exact definition.
 *
 * Layouts: q, k, vT, o, lse as attn_fwd.  Workspace: the scores plane
 * (binary32 [heads][T][T]) then the probability plane (binary16
 * [heads][T][T]), 256-byte aligned; only the causal tiles are written and
 * read.  Ownership: the caller owns every buffer; the library allocates a
 * 4-byte status word per device on first use.
 *
 * Errors: every entry point returns an attn_status (attn_fwd.h); argument
 * errors are detected on the host before anything is launched.
 */
#ifndef ATTN_MATERIALISED_H
#define ATTN_MATERIALISED_H

#include <stddef.h>

#include "attn_fwd.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * attn_materialised_workspace_bytes -- device bytes of the two planes
 * (heads * T * T * 6, the scores plane rounded up to 256 bytes), or 0 if the
 * shape is not admitted.
 */
size_t attn_materialised_workspace_bytes(int T, int heads, int kv_heads);

/*
 * attn_fwd_materialised -- the forward pass through materialised planes.
 *
 * q, k, vT, o, lse: device pointers, 16-byte aligned, layouts as attn_fwd.
 * T, heads, kv_heads, c: as attn_fwd (the same admission), and T <= 16384 (the
 *   planes grow as heads * T^2).
 * workspace: device buffer of at least attn_materialised_workspace_bytes
 *   bytes, 256-byte aligned; its contents on entry do not matter.
 * stream: the stream to run on.
 *
 * Returns ATTN_OK once the three launches are queued; ATTN_EINVAL (a size, the
 * scale, a NULL pointer or a short workspace), ATTN_EALIGN or ATTN_EOVERLAP
 * (an output or the workspace overlaps an input or another output) before
 * anything is queued; ATTN_EDEVICE without a suitable device; ATTN_ELAUNCH if
 * the runtime rejects a launch.  Every element of o and lse is written.  A
 * wait inside a kernel that gives up after 1 s is reported by
 * attn_materialised_last_device_status.
 */
int attn_fwd_materialised(const void *q, const void *k, const void *vT, void *o, float *lse,
                          int T, int heads, int kv_heads, float c,
                          void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * attn_materialised_last_device_status -- synchronises `stream`, then returns
 * and clears the current device's status word of these kernels: ATTN_OK, or
 * ATTN_ETIMEOUT if a wait gave up since the last call.  ATTN_ELAUNCH if the
 * synchronisation reports a CUDA error.
 */
int attn_materialised_last_device_status(cudaStream_t stream);

/*
 * attn_materialised_test_inject_stall -- test hook for the materialised
 * path's failure detection.
 *
 * The source pages have no counterpart of this entry point.  It makes the
 * next attn_fwd_materialised call's scores launch skip the K-tile copy of its
 * first block.  That block's wait runs out after 1 s: it records a timeout,
 * stores nothing, waits (bounded) for its other copy, frees its tensor memory
 * and exits; the other blocks and the two later launches run as usual (on a
 * scores tile that was not written, so that call's outputs are not valid);
 * attn_materialised_last_device_status then returns ATTN_ETIMEOUT, and later
 * calls run normally.  Always returns ATTN_OK.
 */
int attn_materialised_test_inject_stall(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_MATERIALISED_H */
