/*
 * attn_fwd.h -- C ABI of the GB300 (sm_103a) causal grouped-query attention
 * forward pass, computed as a streaming normalised sum.
 *
 * The operation is the one stated in the header comment of the page
 * "Realization/Nvidia/SM86/StreamingAttentionSM86.alpha": for every query
 * head h (reading compact K/V head g = floor(h / (heads / kv_heads)), the
 * page's grid mapping "head = kvHead * groups + z") and every query row i,
 *
 *   t_ij = c * sum_e Q[h][i][e] K[g][j][e]      for keys j <= i (causal, diagonal kept)
 *   O[i][h*64 + e] = sum_j 2^(t_ij - m_i) V^T[g][e][j] / l_i
 *   LSE[h][i]      = m_i + log2 l_i             (base 2)
 *
 * with m_i = max_j t_ij and l_i = sum_j 2^(t_ij - m_i).  c is the binary32
 * nearest scale / ln 2 (for head width 64, scale = 1/8).  As on that page,
 * the weights 2^(t - m) are rounded to binary16 only for their product with
 * V; the running maximum, the running sum and the weighted sum stay binary32.
 *
 * Layouts (all row-major, the page's argument block "pointers to Q, K, V^T,
 * O and L, then c"):
 *   q    binary16 [heads][T][64]
 *   k    binary16 [kv_heads][T][64]
 *   vT   binary16 [kv_heads][64][T]    (V transposed per K/V head)
 *   o    binary16 [T][heads*64]        (token-major, heads merged)  -- output
 *   lse  binary32 [heads][T]           (base-2 log-sum-exp)          -- output
 *
 * Ownership: the caller owns every buffer.  The library keeps, per device, a
 * 384-byte scratch block it allocates on first use and never frees (a status
 * word and 32 slots of work counters the kernel's dynamic tile scheduler
 * uses, one slot per launch in rotation); it allocates nothing per call.
 * More than 32 launches in flight on the GPU at once would share a slot.
 *
 * Errors: every entry point returns an attn_status.  Argument errors are
 * detected on the host before anything is launched.  The launches are
 * asynchronous and ordered on `stream` like a kernel launch.
 */
#ifndef ATTN_FWD_H
#define ATTN_FWD_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's stream handle (NULL = the legacy default stream). */
typedef struct CUstream_st *cudaStream_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_EINVAL = -1,   /* a size or the scale is outside what the operation admits */
    ATTN_EALIGN = -2,   /* a pointer is not 16-byte aligned */
    ATTN_EOVERLAP = -3, /* an output overlaps an input or the other output */
    ATTN_ELAUNCH = -4,  /* the CUDA runtime refused a copy, the set-up or the launch */
    ATTN_EDEVICE = -5,  /* no current CUDA device, or it is not an sm_103 (GB300) part */
    ATTN_ETIMEOUT = -6  /* a kernel wait gave up after 1 s (reported by attn_last_device_status) */
} attn_status;

/* Largest number of query heads admitted (the page's limit of 65535). */
#define ATTN_MAX_HEADS 65535
/* Head width: the only one the page defines. */
#define ATTN_HEAD_DIM 64

/*
 * attn_fwd -- the forward pass on device buffers.
 *
 * q, k, vT, o, lse: device pointers, 16-byte aligned, layouts above.
 * T: sequence length; T > 0 and T % 64 == 0.
 * heads, kv_heads: heads > 0, kv_heads > 0, heads % kv_heads == 0,
 *   heads <= 65535, and heads * 64 * T * 4 <= 2^32 - 1 (the page's admission
 *   predicate for the forward program).
 * c: finite and > 0.
 * stream: the stream to run on.
 *
 * Returns ATTN_OK once the kernel is queued; ATTN_EINVAL / ATTN_EALIGN /
 * ATTN_EOVERLAP before anything is queued if an argument is bad;
 * ATTN_EDEVICE without a suitable device; ATTN_ELAUNCH if the runtime
 * rejects the launch.  Every element of o and lse is written.
 */
int attn_fwd(const void *q, const void *k, const void *vT, void *o, float *lse,
             int T, int heads, int kv_heads, float c, cudaStream_t stream);

/*
 * attn_fwd_workspace_bytes -- device bytes attn_fwd_host needs for the given
 * shape (Q, K, V^T, O and LSE packed at 256-byte boundaries), or 0 if the
 * shape is not admitted.
 */
size_t attn_fwd_workspace_bytes(int T, int heads, int kv_heads);

/*
 * attn_fwd_host -- the forward pass on HOST buffers (same layouts as
 * attn_fwd).  The problem is cut into up to four groups of K/V heads (with
 * their query heads); for each group the call queues the copies of its q, k,
 * vT slices into `workspace` (a device buffer of at least
 * attn_fwd_workspace_bytes bytes, 256-byte aligned, owned by the caller), the
 * kernel on `stream`, and the copies of its O columns and LSE rows back into
 * o and lse.  The copies in and out run on two streams the library creates
 * once per device, ordered by events after the work already queued on
 * `stream`, so both directions overlap the compute; `stream` completes only
 * after the last copy out.  Host buffers should be page-locked for the copies
 * to be asynchronous; the caller synchronises `stream` before reading o and
 * lse.  Calls from several host threads are serialised while they queue.
 * Errors as attn_fwd; ATTN_EINVAL also if workspace_bytes is too small.
 */
int attn_fwd_host(const void *q, const void *k, const void *vT, void *o, float *lse,
                  int T, int heads, int kv_heads, float c,
                  void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * attn_last_device_status -- synchronises `stream`, then returns and clears
 * the current device's status word: ATTN_OK, or ATTN_ETIMEOUT if a wait
 * inside a kernel gave up since the last call (the kernel then wrote no
 * trustworthy output and exited cleanly).  ATTN_ELAUNCH if the synchronisation
 * itself reports a CUDA error.
 */
int attn_last_device_status(cudaStream_t stream);

/*
 * attn_fwd_noalloc -- attn_fwd for callers that cannot allocate device memory.
 *
 * The source pages have no counterpart of this entry point; it exists for
 * callers such as runtimes that plan every device byte ahead of time and
 * forbid allocation once running, processes held to a fixed device-memory
 * quota, and latency-critical loops that cannot afford cudaMalloc's implicit
 * device synchronisation.  attn_fwd allocates a scratch block per device on
 * its first call; this variant instead keeps the kernel's scratch (a status
 * word and 16 slots of work counters for the tile scheduler) in a fixed
 * 256-byte array compiled into the library, so it calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 * Arguments, layouts, admission checks and results are those of attn_fwd.
 * status: NULL, or a pointer to device, managed or page-locked host memory
 *   that receives (ordered on `stream`) the kernel's status word: 0 if every
 *   wait inside the kernel completed, non-zero if one gave up (then o and lse
 *   are not valid).  A pointer to pageable host memory returns ATTN_EINVAL.
 *
 * The scratch this kernel needs does not depend on the shape: it fills the
 * whole 256-byte array (the status word at word 0, words 1-31 unused, the 16
 * counter slots of two words at words 32-63), checked when the library is
 * compiled.
 * The first call on each device looks up the array's device address and
 * sets the kernel's shared-memory attribute: make that first call before any
 * stream capture.  Each call clears the status word and its counter slot
 * (they keep the previous call's values until then).  Every call on every
 * stream shares the one array: calls that overlap on the GPU race on the
 * status word, and on a counter slot when more than 16 are in flight.
 */
int attn_fwd_noalloc(const void *q, const void *k, const void *vT, void *o, float *lse,
                     int T, int heads, int kv_heads, float c, int *status,
                     cudaStream_t stream);

/*
 * attn_test_inject_stall -- test hook for the kernel's failure detection.
 *
 * The source pages have no counterpart of this entry point.  It makes the
 * next attn_fwd launch in this process skip the Q-tile copy of its work unit
 * 0 (the heaviest, whichever CTA takes it).  The wait on the missing tile
 * then runs out after 1 s: the CTA
 * records a timeout, drains the copies and MMAs it issued, frees its tensor
 * memory and exits; attn_last_device_status then returns ATTN_ETIMEOUT (and
 * clears the status word and the scheduler's counters), and later launches
 * run normally.  Always returns ATTN_OK.  Only attn_fwd consumes the hook.
 */
int attn_test_inject_stall(void);

/*
 * attn_test_set_split_mode -- test hook choosing the forward kernel's mode.
 *
 * The source pages have no counterpart of this entry point.  attn_fwd (and
 * attn_fwd_host, attn_fwd_noalloc) run short problems -- fewer 256-row units
 * (heads * ceil(T / 256)) than the device has SMs -- in a split mode: a work
 * unit is 128 query rows whose key tiles are shared out between the kernel's
 * two softmax warpgroups, and the two partial results of every row are merged
 * at the end.  Longer problems run in the normal mode (256-row units, both
 * warpgroups over all key tiles of their own 128 rows).  Both modes compute
 * the same quantities.  mode: -1 chooses by size (the default), 0 forces the
 * normal mode, 1 the split mode, for every later call in this process.
 * Returns ATTN_OK, or ATTN_EINVAL for any other mode.
 */
int attn_test_set_split_mode(int mode);

/* A static, human-readable name for a status code. */
const char *attn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_H */
