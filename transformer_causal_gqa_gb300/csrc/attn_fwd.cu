// attn_fwd.cu -- causal grouped-query attention forward for GB300 (sm_103a),
// computed as a streaming normalised sum, behind the C ABI of attn_fwd.h.
//
// What it computes is the forward pass described in the header comment of
// "Realization/Nvidia/SM86/StreamingAttentionSM86.alpha": scores in base-2
// units t = S c, a running row maximum m, running sum l and running weighted
// sum O folded tile by tile (a new maximum m' scales the old l and O by
// 2^(m - m')), the weights 2^(t - m) rounded to binary16 only for their
// product with V, O / l written binary16 token-major and m + log2 l written
// binary32 per head.  Only the tiles up to and including the diagonal one are
// visited, and only the diagonal tile is masked (key column > query row).
//
// How (GB300-first, not the page's SM86 register-fragment design):
//   * a persistent grid, one CTA per SM, takes work units of 256 query rows
//     of one head (two 128-row subtiles sharing every K/V^T tile) from a
//     global counter, heaviest (latest) row blocks first;
//   * one warp issues TMA loads: Q subtiles and a ring of 16 KiB K and V^T
//     tiles (128 keys x 64), 128-byte swizzled, signalled by mbarriers;
//   * three warps issue tcgen05 MMAs: one issues S = Q K^T (M=128, N=128,
//     K=64) into tensor memory for both subtiles, in whichever order their S
//     buffers free up; one per subtile issues O += P V (M=128, N=64, K=128)
//     with P read from its own tensor-memory columns;
//   * two softmax warpgroups, one per subtile, one thread per query row:
//     tcgen05.ld the row's 128 scores, mask, row maximum, exp2, row sum,
//     round P to binary16 and tcgen05.st it; rescale O in tensor memory when
//     the row's reference maximum moves; at the end normalise and store O and
//     the LSE.
//   The subtiles are not kept in step: each one's softmax overlaps the other's
//   MMAs and exp2 phase.
//
//   The reference maximum m a row's weights are taken against moves only when
//   a tile's maximum exceeds it by more than kMaxSlack (8 in base-2 units), so
//   the weights 2^(t - m) stay below 2^8 (well inside binary16) and O is
//   rescaled only on such a jump instead of on every rise.  The folded sums
//   are those of the page's recurrence with another choice of m; O / l and
//   m + log2 l do not depend on that choice.
//
// Short problems (fewer 256-row units than SMs) run in a split mode instead: a
// unit is 128 query rows, subtile 0 takes the first half of its key tiles and
// subtile 1 the second half (with the diagonal), both against the same Q tile,
// and at the end subtile 1 merges the two partial (m, l, O) of each row --
// the page's merge rule applied across the two halves -- and writes O / l and
// m + log2 l.  The longest chain of key tiles is then half as long.
//
// Every wait on an mbarrier is bounded in time; on expiry the CTA records
// ATTN_ETIMEOUT in a device status word, drains what it has in flight, frees
// its tensor memory and exits.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn_fwd.h"
#include "sm103_ptx.cuh"

namespace {

using namespace sm103;

constexpr int kHeadDim = 64;
constexpr int kBlockM = 128;              // query rows per subtile = TMEM lanes
constexpr int kUnitRows = 2 * kBlockM;    // query rows per work unit
constexpr int kBlockN = 128;              // keys per K / V^T tile
constexpr int kStages = 6;                // K / V^T ring slots
constexpr uint32_t kTileBytes = kBlockN * kHeadDim * 2;  // 16 KiB: a K tile, a V^T tile, a Q subtile
constexpr int kThreads = 384;             // 8 softmax warps, 3 MMA-issuing warps, TMA warp
constexpr int kSWarp = 8;                 // issues S = Q K^T for both subtiles
constexpr int kPvWarp0 = 9;               // issues O_s += P_s V for subtile s = warp - kPvWarp0
constexpr int kLoadWarp = 11;
constexpr int kConsumerWarps = 11;        // every warp but the TMA warp reads the unit queue
constexpr int kUnitSlots = 4;             // unit queue depth
static_assert(kStages % 2 == 0, "K tiles must land in even ring slots, V^T tiles in odd ones");
constexpr uint32_t kTmemCols = 512;
// tensor-memory columns: S of subtile s at 128 s, O at 256 + 64 s, P (binary16
// pairs) at 384 + 64 s -- all 512 columns
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr uint32_t kColP = 384;

// barrier indices
constexpr int kBarQFull = 0;                    // + Q buffer (2)
constexpr int kBarQEmpty = 2;                   // + Q buffer
constexpr int kBarKvFull = 4;                   // + ring slot
constexpr int kBarKvEmpty = kBarKvFull + kStages;
constexpr int kBarSFull = kBarKvEmpty + kStages;  // + subtile: S_s computed
constexpr int kBarSFree = kBarSFull + 2;        // + subtile: S_s read into registers
constexpr int kBarPFull = kBarSFree + 2;        // + subtile: P_s written, O_s rescaled
constexpr int kBarPvDone = kBarPFull + 2;       // + subtile: O_s += P_s V complete
constexpr int kBarUnitFull = kBarPvDone + 2;    // + queue slot: a unit id published
constexpr int kBarUnitEmpty = kBarUnitFull + kUnitSlots;  // + queue slot: read by every consumer
constexpr int kBarDrain = kBarUnitEmpty + kUnitSlots;     // + MMA warp (0..2): its own drain on abort
constexpr int kBarMergeReady = kBarDrain + 3;   // split mode: subtile 0's partial (m, l, O) is ready
constexpr int kBarMergeDone = kBarMergeReady + 1;  // split mode: subtile 1 has read it
constexpr int kNumBars = kBarMergeDone + 1;

// dynamic shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t kOffQ = 0;                               // 2 buffers x 2 subtiles
constexpr uint32_t kOffRing = 4 * kTileBytes;
constexpr uint32_t kOffBar = kOffRing + kStages * kTileBytes;
constexpr uint32_t kOffUnits = kOffBar + kNumBars * 8;
constexpr uint32_t kOffTmemPtr = kOffUnits + kUnitSlots * 4;
constexpr uint32_t kOffAbort = kOffTmemPtr + 4;
constexpr uint32_t kOffMerge = (kOffAbort + 4 + 15) & ~15u;   // split mode: m and l of 128 rows
constexpr uint32_t kSmemUsed = kOffMerge + 2 * kBlockM * 4;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for aligning the base

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s: far beyond any legitimate wait
constexpr float kMaxSlack = 8.f;  // a row's reference maximum moves only on a larger jump

// Device scratch the kernel uses beyond its inputs and outputs: a status
// word, and a ring of work-counter slots (next unit, finished CTAs), one slot
// per launch so that launches overlapping on different streams do not share one.
constexpr int kScratchStatus = 0;
constexpr int kScratchSched = 32;         // first counter slot (2 ints per slot)

struct Params {
  int T;
  int heads;
  int group;          // query heads per K/V head
  int row_blocks;     // ceil(T / 256), or ceil(T / 128) in split mode
  int units;          // heads * row_blocks
  float c;
  __half *o;
  float *lse;
  int *status;
  int *sched;         // this launch's counter slot: [0] next unit, [1] CTAs done
};

struct Unit {
  int h, g, b;        // query head, K/V head, row block
  int row0;           // first query row
  int n0, n1;         // key tiles visited by subtile 0 and subtile 1
  // split mode only:
  int k1;             // key tile of subtile 1's first step (n0)
  int diag0, diag1;   // step of each subtile that meets the diagonal (-1: none)
  int ring;           // ring positions the unit's K and V^T tiles take
};

// Unit u in order of decreasing cost: the latest row blocks (most key tiles) first.
// Normal mode: 256 rows, subtile s holds rows 128 s .. +127 and visits tiles 0 ..
// its diagonal; both read every K, V^T tile.  Split mode: 128 rows read by both
// subtiles; of the n key tiles 0 .. diagonal, subtile 0 visits the first n / 2
// and subtile 1 the rest; each tile is read by one subtile.
template <bool kSplit>
__device__ __forceinline__ Unit decode_unit(int u, const Params &p) {
  Unit w;
  const int rb = u / p.heads;
  w.h = u - rb * p.heads;
  w.b = p.row_blocks - 1 - rb;
  w.g = w.h / p.group;
  if (!kSplit) {
    w.row0 = w.b * kUnitRows;
    const int end = min(p.T, w.row0 + kUnitRows);
    w.n0 = 2 * w.b + 1;                   // subtile 0: tiles 0 .. its diagonal 2b
    w.n1 = (end + kBlockN - 1) / kBlockN; // subtile 1: through 2b+1, or 2b when it holds no row < T
    // k1, diag0, diag1 and ring serve the split mode only (the normal mode
    // uses 0, 2b, 2b+1 and 2 n1 directly)
    w.k1 = w.diag0 = w.diag1 = w.ring = 0;
  } else {
    w.row0 = w.b * kBlockM;
    const int n = w.b + 1;
    w.n0 = n / 2;
    w.n1 = n - w.n0;
    w.k1 = w.n0;
    w.diag0 = -1;
    w.diag1 = w.n1 - 1;
    w.ring = 2 * n;
  }
  return w;
}

// Place of step j of subtile s among the unit's K, V^T tile pairs in the ring:
// normal mode, pair j (shared by both subtiles); split mode, the two subtiles'
// steps alternate while both have steps left, then subtile 1's remaining ones.
template <bool kSplit>
__device__ __forceinline__ int pair_of(const Unit &w, int s, int j) {
  if (!kSplit) return j;
  return j < w.n0 ? 2 * j + s : w.n0 + j;
}

struct Sync {
  uint32_t bar0;              // smem address of barrier 0
  volatile int *abort_flag;   // smem
  volatile int *units;        // smem unit queue
  int *status;                // global
  __device__ __forceinline__ uint32_t bar(int i) const { return bar0 + 8u * i; }

  // Bounded wait: false if the CTA is aborting or the wait ran out of time.
  __device__ bool wait(int i, uint32_t parity, int where) const {
    const uint32_t b = bar(i);
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait(b, parity)) return true;
      if ((it & 63u) == 0) {
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          *abort_flag = 1;
          atomicCAS(status, 0, where);
          return false;
        }
      }
    }
  }

  // Bounded wait taken by a whole warp: every lane gets the same answer.
  __device__ bool wait_warp(int i, uint32_t parity, int where) const {
    const bool ok = wait(i, parity, where);
    return __all_sync(0xffffffffu, ok);
  }

  // While aborting: wait for this thread's own copies or MMAs in flight,
  // bounded in time only.
  __device__ void drain_wait(int i, uint32_t parity) const {
    const uint32_t b = bar(i);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(b, parity))
      if (globaltimer_ns() - t0 > kWaitLimitNs) break;
  }

  // The k-th unit this CTA works on, read by a whole consumer warp from the
  // queue the TMA warp fills: a unit id, -1 when the work is exhausted, -2 if
  // the CTA is aborting.
  __device__ int next_unit(int k) const {
    const int slot = k % kUnitSlots;
    if (!wait_warp(kBarUnitFull + slot, (k / kUnitSlots) & 1, 30)) return -2;
    const int u = units[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar(kBarUnitEmpty + slot));
    return u;
  }
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (d0, d1) = (a0 * b + c, a1 * b + c), two IEEE fmas in one instruction.
__device__ __forceinline__ void fma2(float &d0, float &d1, float a0, float a1, float b, float c) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %4};\n\t"
      "mov.b64 rc, {%5, %5};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

// (s0, s1) += (a0, a1), two IEEE adds in one instruction.
__device__ __forceinline__ void add2(float &s0, float &s1, float a0, float a1) {
  asm("{\n\t.reg .b64 ra, rs;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rs, {%0, %1};\n\t"
      "add.f32x2 rs, rs, ra;\n\t"
      "mov.b64 {%0, %1}, rs;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "f"(a0), "f"(a1));
}

// (d0, d1) = (a0 * b, a1 * b), two IEEE multiplies in one instruction.
__device__ __forceinline__ void mul2(float &d0, float &d1, float b) {
  asm("{\n\t.reg .b64 ra, rb;\n\t"
      "mov.b64 ra, {%0, %1};\n\t"
      "mov.b64 rb, {%2, %2};\n\t"
      "mul.f32x2 ra, ra, rb;\n\t"
      "mov.b64 {%0, %1}, ra;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(b));
}

// ----------------------------------------------------------------------------
// TMA warp (one lane): takes units from the global work counter and publishes
// them to the CTA's unit queue; for each, loads the two Q subtiles into the
// unit's Q buffer, then K(j), V^T(j) for j = 0 .. n1-1 through the ring.
// kStallHook (test builds of the launch only): the Q tile of work unit 0 (whichever CTA
// claims it) is never loaded.  Both subtiles need it in either mode, so their S issue
// waits until it runs out.
template <bool kStallHook, bool kSplit>
__device__ void load_role(const CUtensorMap *tmQ, const CUtensorMap *tmK, const CUtensorMap *tmV,
                          const Params &p, const Sync &sy, uint32_t smem) {
  uint32_t pos = 0;         // running ring position (K and V^T tiles alternate)
  uint32_t pos_issued = 0;  // ring positions whose copy has been issued
  uint32_t q_issued = 0;    // Q loads issued
  for (int k = 0;; ++k) {
    const int slot = k % kUnitSlots;
    if (!sy.wait(kBarUnitEmpty + slot, ((k / kUnitSlots) & 1) ^ 1, 1)) goto drain;
    int u = atomicAdd(&p.sched[0], 1);
    if (u >= p.units) u = -1;
    sy.units[slot] = u;
    mbar_arrive(sy.bar(kBarUnitFull + slot));
    if (u < 0) break;
    const Unit w = decode_unit<kSplit>(u, p);
    const int qb = k & 1;
    if (!sy.wait(kBarQEmpty + qb, ((k >> 1) & 1) ^ 1, 1)) goto drain;
    ++q_issued;
    const uint32_t qdst = smem + kOffQ + qb * 2 * kTileBytes;
    if (!(kStallHook && u == 0)) {  // test hook: this Q tile never arrives
      // split mode: one Q tile, read by both subtiles
      mbar_arrive_expect_tx(sy.bar(kBarQFull + qb), (kSplit ? 1 : 2) * kTileBytes);
      tma_load_3d(qdst, tmQ, sy.bar(kBarQFull + qb), 0, w.row0, w.h);
      if (!kSplit)
        tma_load_3d(qdst + kTileBytes, tmQ, sy.bar(kBarQFull + qb), 0, w.row0 + kBlockM, w.h);
    }
    for (int jp = 0; jp < (kSplit ? w.ring / 2 : w.n1); ++jp) {
      // the key tile of pair jp
      int j = jp;
      if (kSplit) j = jp < 2 * w.n0 ? (jp & 1 ? w.k1 : 0) + (jp >> 1) : jp;
      for (int kv = 0; kv < 2; ++kv, ++pos) {
        const uint32_t rs = pos % kStages;
        if (!sy.wait(kBarKvEmpty + rs, ((pos / kStages) & 1) ^ 1, 2)) goto drain;
        const uint32_t dst = smem + kOffRing + rs * kTileBytes;
        const uint32_t full = sy.bar(kBarKvFull + rs);
        pos_issued = pos + 1;
        mbar_arrive_expect_tx(full, kTileBytes);
        if (kv == 0) {
          tma_load_3d(dst, tmK, full, 0, j * kBlockN, w.g);
        } else {
          tma_load_3d(dst, tmV, full, j * kBlockN, 0, w.g);
          tma_load_3d(dst + kTileBytes / 2, tmV, full, j * kBlockN + kBlockN / 2, 0, w.g);
        }
      }
    }
  }
  // This CTA takes no more units.  The last CTA to get here resets the
  // launch's counter slot for the next launch that uses it.
  if (atomicAdd(&p.sched[1], 1) == (int)gridDim.x - 1) {
    atomicExch(&p.sched[0], 0);
    atomicExch(&p.sched[1], 0);
  }
  return;
drain:
  // Aborting: let the copies already issued land before the CTA exits.
  for (uint32_t i = 0; i < kStages && i < pos_issued; ++i) {
    const uint32_t q = pos_issued - 1 - i;
    sy.drain_wait(kBarKvFull + q % kStages, (q / kStages) & 1);
  }
  for (uint32_t i = 0; i < 2 && i < q_issued; ++i) {
    const uint32_t q = q_issued - 1 - i;
    sy.drain_wait(kBarQFull + (q & 1), (q >> 1) & 1);
  }
}

// ----------------------------------------------------------------------------
// The tensor pipe takes a new tcgen05.mma from a given warp only every ~100
// cycles, so three warps issue concurrently: one for S = Q K^T (both
// subtiles, 4 MMAs of N = 128 per tile each) and one per subtile for
// O += P V (8 MMAs of N = 64 per tile, A = P read from tensor memory).
// Each accumulation chain is issued by a single warp, so it stays ordered.

// S issuer: S_s(j) as soon as the softmax has pulled S_s(j-1) into registers.
// The two subtiles are served in whichever order their S buffers free up
// (subtile 1 is tested first), not strictly in turn.  Issued strictly in turn,
// both subtiles' S became ready together and their softmax warpgroups ran in
// lockstep, meeting on the SFU; served this way, one pick every ~1000 cycles
// keeps them about half a tile apart.
template <bool kSplit>
__device__ void s_role(const Params &p, const Sync &sy, uint32_t smem, uint32_t tmem) {
  constexpr uint32_t idS = idesc_f16_f32(kBlockM, kBlockN);
  uint32_t pos = 0;
  uint32_t s_issued0 = 0, s_issued1 = 0;  // S MMAs issued per subtile (S-free is an "empty" barrier)
  for (int k = 0;; ++k) {
    const int u = sy.next_unit(k);
    if (u == -1) return;
    if (u < 0) goto drain;
    {
      const Unit w = decode_unit<kSplit>(u, p);
      const int qb = k & 1;
      if (!sy.wait_warp(kBarQFull + qb, (k >> 1) & 1, 11)) goto drain;
      tc_fence_after();
      const int n0 = w.n0, n1 = w.n1;
      int j0 = 0, j1 = 0;
      uint64_t t0 = 0;
      uint32_t spins = 0;
      while (j0 < n0 || j1 < n1) {
        // subtile 1 first, then subtile 0 (subtile 1 settles a little ahead)
        const int first = 1;
        int pick = -1;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int s = first ^ c;
          const int js = s ? j1 : j0;
          if (js >= (s ? n1 : n0)) continue;
          const uint32_t kpos = pos + 2 * pair_of<kSplit>(w, s, js);
          const uint32_t sfree_parity = ((s ? s_issued1 : s_issued0) & 1) ^ 1;
          const bool ready = mbar_test_wait(sy.bar(kBarSFree + s), sfree_parity) &&
                             mbar_test_wait(sy.bar(kBarKvFull + kpos % kStages), (kpos / kStages) & 1);
          if (__all_sync(0xffffffffu, ready)) { pick = s; break; }
        }
        if (pick < 0) {
          if (spins == 0) t0 = globaltimer_ns();
          if ((++spins & 63u) == 0) {
            if (*sy.abort_flag) goto drain;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
              *sy.abort_flag = 1;
              atomicCAS(sy.status, 0, 13);
              goto drain;
            }
          }
          continue;
        }
        spins = 0;
        tc_fence_after();
        const int s = pick;
        const int j = s ? j1 : j0;
        const uint32_t kslot = (pos + 2 * pair_of<kSplit>(w, s, j)) % kStages;
        const uint32_t kbase = smem + kOffRing + kslot * kTileBytes;
        const uint32_t qbase = smem + kOffQ + (qb * 2 + (kSplit ? 0 : s)) * kTileBytes;
        // the four MMAs of S_s(j) under one election (issued back to back)
        mma_ss_k64(tmem + kColS + 128u * s, sw128_desc(qbase), sw128_desc(kbase), idS);
        mma_commit(sy.bar(kBarSFull + s));
        if (s) { ++s_issued1; j1 = j + 1; } else { ++s_issued0; j0 = j + 1; }
        // K(j) is released once every subtile that reads it has its S issued
        // (split mode: it has one reader)
        const bool other_done = kSplit || (s ? (j0 > j || j >= n0) : (j1 > j || j >= n1));
        if (other_done) mma_commit(sy.bar(kBarKvEmpty + kslot));
      }
      mma_commit(sy.bar(kBarQEmpty + qb));  // every S of this unit issued
      pos += kSplit ? w.ring : 2 * w.n1;
    }
  }
drain:
  mma_commit(sy.bar(kBarDrain + 0));
  sy.drain_wait(kBarDrain + 0, 0);
}

// P V issuer for subtile s: O_s += P_s(j) V(j) once the softmax has written P_s(j).
// It releases every V^T tile of the unit (the barrier counts both subtiles'
// issuers), including the one subtile 0 does not read when n1 > n0.
template <bool kSplit>
__device__ void pv_role(int s, const Params &p, const Sync &sy, uint32_t smem, uint32_t tmem) {
  constexpr uint32_t idPV = idesc_f16_f32(kBlockM, kHeadDim);
  uint32_t pos = 0;
  uint32_t pphase = 0;
  for (int k = 0;; ++k) {
    const int u = sy.next_unit(k);
    if (u == -1) return;
    if (u < 0) goto drain;
    const Unit w = decode_unit<kSplit>(u, p);
    const int n = s ? w.n1 : w.n0;
    for (int j = 0; j < n; ++j) {
      const uint32_t vpos = pos + 2 * pair_of<kSplit>(w, s, j) + 1;
      const uint32_t vslot = vpos % kStages;
      if (!sy.wait_warp(kBarPFull + s, pphase, 14)) goto drain;
      pphase ^= 1;
      if (!sy.wait_warp(kBarKvFull + vslot, (vpos / kStages) & 1, 10)) goto drain;
      tc_fence_after();
      const uint32_t vbase = smem + kOffRing + vslot * kTileBytes;
      const uint32_t pcol = tmem + kColP + 64u * s;
#pragma unroll
      for (int kk = 0; kk < kBlockN / 16; ++kk) {
        const uint64_t bdesc = sw128_desc(vbase + (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32);
        mma_ts(tmem + kColO + 64u * s, pcol + 8u * kk, bdesc, idPV, (j > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(sy.bar(kBarPvDone + s));
      mma_commit(sy.bar(kBarKvEmpty + vslot));
      // a V^T tile the other subtile does not read (every tile in split mode): this
      // issuer releases it for both, after its own wait on the tile, so the arrival
      // cannot land in the slot's previous phase
      if (kSplit || j >= w.n0) mma_commit(sy.bar(kBarKvEmpty + vslot));
    }
    pos += kSplit ? w.ring : 2 * w.n1;
  }
drain:
  mma_commit(sy.bar(kBarDrain + 1 + s));
  sy.drain_wait(kBarDrain + 1 + s, 0);
}

// ----------------------------------------------------------------------------
// Softmax warpgroup for subtile s: thread r owns query row r (TMEM lane r).
template <bool kSplit>
__device__ void softmax_role(int s, const Params &p, const Sync &sy, uint32_t tmem,
                             float *merge_ml) {
  const int r = threadIdx.x & 127;
  const bool leader = (threadIdx.x & 31) == 0;
  const uint32_t lane_base = (uint32_t)((threadIdx.x & 96)) << 16;  // warp's 32-lane slice
  const uint32_t tS = tmem + lane_base + kColS + 128u * s;
  const uint32_t tO = tmem + lane_base + kColO + 64u * s;
  const uint32_t tP = tmem + lane_base + kColP + 64u * s;
  const float c = p.c;
  uint32_t sphase = 0, pvphase = 0;
  for (int k = 0;; ++k) {
    const int u = sy.next_unit(k);
    if (u < 0) return;
    const Unit w = decode_unit<kSplit>(u, p);
    const int n = s ? w.n1 : w.n0;
    const int diag = kSplit ? (s ? w.diag1 : w.diag0) : 2 * w.b + s;
    float m_run = -INFINITY, l_run = 0.f;
    // S_s(j+1) is tested (without blocking) right after P_s(j) is handed over; when
    // it was already complete the next tile skips its wait.  Each barrier test
    // costs a shared-memory round trip in the running kernel, and this one overlaps
    // the loop's turn instead of sitting in front of the next tile.
    bool s_seen = false;
    for (int j = 0; j < n; ++j) {
      if (!__all_sync(0xffffffffu, s_seen) && !sy.wait_warp(kBarSFull + s, sphase, 20 + s)) return;
      sphase ^= 1;
      tc_fence_after();
      uint32_t sr[128];
      tmem_ld_x128(tS, sr);
      // S_s is in registers: the tensor pipe may overwrite it with S_s(j+1)
      tc_fence_before();
      __syncwarp();
      if (leader) mbar_arrive(sy.bar(kBarSFree + s));
      float sv[128];
#pragma unroll
      for (int col = 0; col < kBlockN; ++col) sv[col] = __uint_as_float(sr[col]);
      if (j == diag) {
#pragma unroll
        for (int col = 0; col < kBlockN; ++col)
          if (col > r) sv[col] = -INFINITY;
      }
      // row maximum: eight independent chains of 3-input max
      float mx8[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) mx8[a] = fmaxf(sv[a], sv[8 + a]);
#pragma unroll
      for (int col = 16; col < kBlockN; col += 16)
#pragma unroll
        for (int a = 0; a < 8; ++a) mx8[a] = max3(mx8[a], sv[col + a], sv[col + 8 + a]);
      const float mx = max3(max3(mx8[0], mx8[1], mx8[2]), max3(mx8[3], mx8[4], mx8[5]),
                            fmaxf(mx8[6], mx8[7]));
      // the reference maximum moves only when this tile exceeds it by more than
      // kMaxSlack (always on the first tile, where m_run = -inf)
      const float mt = mx * c;
      const float m_new = (mt > m_run + kMaxSlack) ? mt : m_run;
      const float alpha = (m_new == m_run) ? 1.f : ex2(m_run - m_new);
      const float neg = -m_new;
      // P = 2^(S c - m'), in three dense passes so the SFU sees 128 back-to-back
      // exp2: paired fmas, then exp2, then paired row sums and binary16 packing
#pragma unroll
      for (int i = 0; i < 64; ++i) fma2(sv[2 * i], sv[2 * i + 1], sv[2 * i], sv[2 * i + 1], c, neg);
#pragma unroll
      for (int i = 0; i < 128; ++i) sv[i] = ex2(sv[i]);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t pk[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        add2(acc[2 * (i & 3)], acc[2 * (i & 3) + 1], sv[2 * i], sv[2 * i + 1]);
        pk[i] = pack_half2(sv[2 * i], sv[2 * i + 1]);
      }
      const float sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
      l_run = l_run * alpha + sum;
      if (j > 0) {
        // P_s(j-1) V(j-1) must be complete before O_s is rescaled and P_s is overwritten
        if (!sy.wait_warp(kBarPvDone + s, pvphase, 24 + s)) return;
        pvphase ^= 1;
        tc_fence_after();
        // the reference maximum moved for some row of this warp: O *= 2^(m - m') (alpha = 1 elsewhere)
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          uint32_t orow[64];
          tmem_ld_x64(tO, orow);
          float of[64];
#pragma unroll
          for (int i = 0; i < 64; ++i) of[i] = __uint_as_float(orow[i]);
#pragma unroll
          for (int i = 0; i < 64; i += 2) mul2(of[i], of[i + 1], alpha);
#pragma unroll
          for (int i = 0; i < 64; ++i) orow[i] = __float_as_uint(of[i]);
          tmem_st_x64_async(tO, orow);
        }
      }
      tmem_st_x64_async(tP, pk);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (leader) mbar_arrive(sy.bar(kBarPFull + s));
      m_run = m_new;
      s_seen = j + 1 < n && mbar_test_wait(sy.bar(kBarSFull + s), sphase);
    }
    // epilogue: O / l and m + log2 l once the last P V is done
    if (!kSplit || n > 0) {
      if (!sy.wait_warp(kBarPvDone + s, pvphase, 22 + s)) return;
      pvphase ^= 1;
      tc_fence_after();
    }
    if (kSplit && s == 0) {
      // split mode: hand this half's m and l to subtile 1, which merges the two
      // halves of every row (its O is read from tensor memory by subtile 1's warps
      // on the same lanes), and wait until it has done so before O is reused
      merge_ml[r] = m_run;
      merge_ml[kBlockM + r] = l_run;
      tc_fence_before();
      __syncwarp();
      if (leader) mbar_arrive(sy.bar(kBarMergeReady));
      if (!sy.wait_warp(kBarMergeDone, k & 1, 26)) return;
      tc_fence_after();
      continue;
    }
    uint32_t orow[64];
    tmem_ld_x64(tO, orow);
    if (kSplit) {
      // merge with subtile 0's half: m = max(m0, m1), each half scaled by 2^(m_h - m)
      if (!sy.wait_warp(kBarMergeReady, k & 1, 27)) return;
      tc_fence_after();
      const float m0 = merge_ml[r], l0 = merge_ml[kBlockM + r];
      const float m = fmaxf(m0, m_run);
      const float a0 = l0 > 0.f ? ex2(m0 - m) : 0.f;
      const float a1 = ex2(m_run - m);
      if (__any_sync(0xffffffffu, l0 > 0.f)) {
        uint32_t o0[64];
        tmem_ld_x64(tmem + lane_base + kColO, o0);
#pragma unroll
        for (int i = 0; i < 64; ++i)
          orow[i] = __float_as_uint(fmaf(__uint_as_float(o0[i]), a0, __uint_as_float(orow[i]) * a1));
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) orow[i] = __float_as_uint(__uint_as_float(orow[i]) * a1);
      }
      l_run = l0 * a0 + l_run * a1;
      m_run = m;
      tc_fence_before();
      __syncwarp();
      if (leader) mbar_arrive(sy.bar(kBarMergeDone));
    }
    const int row = w.row0 + (kSplit ? 0 : s * kBlockM) + r;
    if (row < p.T) {
      const float inv = 1.f / l_run;
      uint4 *dst = reinterpret_cast<uint4 *>(p.o + ((size_t)row * p.heads + w.h) * kHeadDim);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint4 v;
        v.x = pack_half2(__uint_as_float(orow[8 * i + 0]) * inv, __uint_as_float(orow[8 * i + 1]) * inv);
        v.y = pack_half2(__uint_as_float(orow[8 * i + 2]) * inv, __uint_as_float(orow[8 * i + 3]) * inv);
        v.z = pack_half2(__uint_as_float(orow[8 * i + 4]) * inv, __uint_as_float(orow[8 * i + 5]) * inv);
        v.w = pack_half2(__uint_as_float(orow[8 * i + 6]) * inv, __uint_as_float(orow[8 * i + 7]) * inv);
        dst[i] = v;
      }
      p.lse[(size_t)w.h * p.T + row] = m_run + log2f(l_run);
    }
    tc_fence_before();  // O's reads are ordered before the next unit's first P V
  }
}

template <bool kStallHook, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t smem = (raw + 1023u) & ~1023u;
  uint8_t *smem_gen = smem_raw + (smem - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  Sync sy;
  sy.bar0 = smem + kOffBar;
  sy.abort_flag = reinterpret_cast<volatile int *>(smem_gen + kOffAbort);
  sy.units = reinterpret_cast<volatile int *>(smem_gen + kOffUnits);
  sy.status = p.status;

  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int b = 0; b < 2; ++b) {
      mbar_init(sy.bar(kBarQFull + b), 1);
      mbar_init(sy.bar(kBarQEmpty + b), 1);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(sy.bar(kBarKvFull + i), 1);
      // K slots are released by the S issuer, V^T slots by both P V issuers
      mbar_init(sy.bar(kBarKvEmpty + i), (i % 2 == 0) ? 1 : 2);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(sy.bar(kBarSFull + s), 1);
      mbar_init(sy.bar(kBarSFree + s), kBlockM / 32);  // one arrival per softmax warp
      mbar_init(sy.bar(kBarPFull + s), kBlockM / 32);
      mbar_init(sy.bar(kBarPvDone + s), 1);
    }
    for (int i = 0; i < kUnitSlots; ++i) {
      mbar_init(sy.bar(kBarUnitFull + i), 1);
      mbar_init(sy.bar(kBarUnitEmpty + i), kConsumerWarps);
    }
    for (int i = 0; i < 3; ++i) mbar_init(sy.bar(kBarDrain + i), 1);
    mbar_init(sy.bar(kBarMergeReady), kBlockM / 32);   // subtile 0's softmax warps
    mbar_init(sy.bar(kBarMergeDone), kBlockM / 32);    // subtile 1's softmax warps
    *sy.abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kSWarp) {
    tmem_alloc(smem + kOffTmemPtr, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem_gen + kOffTmemPtr);

  if (warp < 8) {
    // warps 0-3 take subtile 1 (the one a unit's last tile belongs to), warps 4-7 subtile 0
    softmax_role<kSplit>(1 - (warp >> 2), p, sy, tmem,
                         reinterpret_cast<float *>(smem_gen + kOffMerge));
  } else if (warp == kSWarp) {
    s_role<kSplit>(p, sy, smem, tmem);
  } else if (warp == kPvWarp0 || warp == kPvWarp0 + 1) {
    pv_role<kSplit>(warp - kPvWarp0, p, sy, smem, tmem);
  } else if (warp == kLoadWarp) {
    if (lane == 0) load_role<kStallHook, kSplit>(&tmQ, &tmK, &tmV, p, sy, smem);
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kSWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ============================================================================
// host side

constexpr int kSchedSlots = 32;           // counter slots in attn_fwd's scratch
constexpr int kScratchInts = kScratchSched + 2 * kSchedSlots;

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int *scratch = nullptr;     // kScratchInts ints: status word, then the counter slots
  unsigned calls = 0;         // launches so far; picks the counter slot
};

std::mutex g_mutex;
// test hook: launches left to stall, and their wait bound
int g_stall_launches = 0;
DeviceState g_dev[64];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool set_smem_attributes() {
  return cudaFuncSetAttribute(attn_fwd_kernel<false, false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) == cudaSuccess &&
         cudaFuncSetAttribute(attn_fwd_kernel<false, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) == cudaSuccess &&
         cudaFuncSetAttribute(attn_fwd_kernel<true, false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) == cudaSuccess &&
         cudaFuncSetAttribute(attn_fwd_kernel<true, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) == cudaSuccess;
}

// test hook: -1 chooses the mode by size (split when fewer 256-row units than SMs),
// 0 and 1 force the normal and the split mode
int g_split_mode = -1;

// Split mode for problems with fewer 256-row units than SMs: the longest chain
// of key tiles is then what bounds the call, and splitting each unit's key
// tiles between the two subtiles halves it.
bool use_split(int T, int heads, int sms) {
  int mode;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    mode = g_split_mode;
  }
  if (mode >= 0) return mode == 1;
  return (long long)heads * ((T + kUnitRows - 1) / kUnitRows) < sms;
}

template <bool kStallHook>
void launch_kernel(bool split, int grid, cudaStream_t stream, const CUtensorMap *tm, const Params &p) {
  if (split)
    attn_fwd_kernel<kStallHook, true><<<grid, kThreads, kSmemBytes, stream>>>(tm[0], tm[1], tm[2], p);
  else
    attn_fwd_kernel<kStallHook, false><<<grid, kThreads, kSmemBytes, stream>>>(tm[0], tm[1], tm[2], p);
}

int device_state(DeviceState **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return ATTN_EDEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState &st = g_dev[dev];
  if (!st.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return ATTN_EDEVICE;
    if (prop.major != 10 || prop.minor != 3) return ATTN_EDEVICE;
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void *fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return ATTN_ELAUNCH;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (!set_smem_attributes()) return ATTN_ELAUNCH;
    if (cudaMalloc(&st.scratch, kScratchInts * sizeof(int)) != cudaSuccess) return ATTN_ELAUNCH;
    if (cudaMemset(st.scratch, 0, kScratchInts * sizeof(int)) != cudaSuccess) return ATTN_ELAUNCH;
    st.sms = prop.multiProcessorCount;
    st.ready = true;
  }
  *out = &st;
  return ATTN_OK;
}

bool encode_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1) {
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// The page's admission predicate for the forward program, plus c.
int check_shape(int T, int heads, int kv_heads, float c) {
  if (T <= 0 || heads <= 0 || kv_heads <= 0) return ATTN_EINVAL;
  if (T % 64 != 0) return ATTN_EINVAL;
  if (heads % kv_heads != 0) return ATTN_EINVAL;
  if (heads > ATTN_MAX_HEADS) return ATTN_EINVAL;
  if ((uint64_t)heads * 64u * (uint64_t)T * 4u > 0xFFFFFFFFull) return ATTN_EINVAL;
  if (!std::isfinite(c) || !(c > 0.f)) return ATTN_EINVAL;
  return ATTN_OK;
}

struct Sizes {
  size_t q, kv, o, lse;
};
Sizes sizes_of(int T, int heads, int kv_heads) {
  Sizes z;
  z.q = (size_t)heads * T * kHeadDim * 2;
  z.kv = (size_t)kv_heads * T * kHeadDim * 2;
  z.o = z.q;
  z.lse = (size_t)heads * T * 4;
  return z;
}

int check_args(const void *q, const void *k, const void *vT, const void *o, const void *lse, int T,
               int heads, int kv_heads, float c) {
  const int rc = check_shape(T, heads, kv_heads, c);
  if (rc) return rc;
  if (!q || !k || !vT || !o || !lse) return ATTN_EINVAL;
  for (const void *ptr : {q, k, vT, o, lse})
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return ATTN_EALIGN;
  const Sizes z = sizes_of(T, heads, kv_heads);
  if (overlaps(o, z.o, lse, z.lse)) return ATTN_EOVERLAP;
  for (const void *out : {o, lse}) {
    const size_t n = out == o ? z.o : z.lse;
    if (overlaps(out, n, q, z.q) || overlaps(out, n, k, z.kv) || overlaps(out, n, vT, z.kv))
      return ATTN_EOVERLAP;
  }
  return ATTN_OK;
}

// Encodes the three tensor maps and fills the kernel parameters (all but the scratch).
bool prepare(const void *q, const void *k, const void *vT, void *o, float *lse, int T, int heads,
             int kv_heads, float c, bool split, CUtensorMap *tm, Params *p) {
  const uint64_t rowb = kHeadDim * 2;
  if (!encode_3d(&tm[0], q, kHeadDim, T, heads, rowb, rowb * T, kHeadDim, kBlockM) ||
      !encode_3d(&tm[1], k, kHeadDim, T, kv_heads, rowb, rowb * T, kHeadDim, kBlockN) ||
      !encode_3d(&tm[2], vT, T, kHeadDim, kv_heads, (uint64_t)T * 2, (uint64_t)T * 2 * kHeadDim,
                 kBlockN / 2, kHeadDim))
    return false;
  p->T = T;
  p->heads = heads;
  p->group = heads / kv_heads;
  p->row_blocks = split ? (T + kBlockM - 1) / kBlockM : (T + kUnitRows - 1) / kUnitRows;
  p->units = heads * p->row_blocks;
  p->c = c;
  p->o = static_cast<__half *>(o);
  p->lse = lse;
  return true;
}

}  // namespace

extern "C" int attn_fwd(const void *q, const void *k, const void *vT, void *o, float *lse, int T,
                        int heads, int kv_heads, float c, cudaStream_t stream) {
  int rc = check_args(q, k, vT, o, lse, T, heads, kv_heads, c);
  if (rc) return rc;
  DeviceState *st = nullptr;
  if ((rc = device_state(&st))) return rc;
  CUtensorMap tm[3];
  Params p;
  const bool split = use_split(T, heads, st->sms);
  if (!prepare(q, k, vT, o, lse, T, heads, kv_heads, c, split, tm, &p)) return ATTN_ELAUNCH;
  unsigned slot;
  bool stall = false;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    slot = st->calls++ % kSchedSlots;
    if (g_stall_launches > 0) {
      --g_stall_launches;
      stall = true;
    }
  }
  p.status = st->scratch + kScratchStatus;
  p.sched = st->scratch + kScratchSched + 2 * slot;
  const int grid = p.units < st->sms ? p.units : st->sms;
  if (stall)
    launch_kernel<true>(split, grid, stream, tm, p);
  else
    launch_kernel<false>(split, grid, stream, tm, p);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
  return ATTN_OK;
}

extern "C" size_t attn_fwd_workspace_bytes(int T, int heads, int kv_heads) {
  if (check_shape(T, heads, kv_heads, 1.f)) return 0;
  const Sizes z = sizes_of(T, heads, kv_heads);
  auto up = [](size_t n) { return (n + 255) & ~(size_t)255; };
  return up(z.q) + 2 * up(z.kv) + up(z.o) + up(z.lse);
}

namespace {
// attn_fwd_host's pipeline: the problem is cut into up to kHostChunks groups of
// K/V heads; chunk c's inputs are copied in on one stream while the kernel runs
// on chunk c - 1 on the caller's stream and chunk c - 2's outputs are copied out
// on a third, so the transfers in both directions overlap the compute.
constexpr int kHostChunks = 4;
struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t in_done[kHostChunks] = {}, comp_done[kHostChunks] = {};
};
std::mutex g_pipe_mutex;
HostPipe g_pipe[64];

int host_pipe(HostPipe **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return ATTN_EDEVICE;
  }
  HostPipe &hp = g_pipe[dev];
  if (!hp.ready) {
    bool ok = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < kHostChunks; ++i)
      ok = cudaEventCreateWithFlags(&hp.in_done[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&hp.comp_done[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      return ATTN_ELAUNCH;
    }
    hp.ready = true;
  }
  *out = &hp;
  return ATTN_OK;
}
}  // namespace

extern "C" int attn_fwd_host(const void *q, const void *k, const void *vT, void *o, float *lse,
                             int T, int heads, int kv_heads, float c, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_shape(T, heads, kv_heads, c);
  if (rc) return rc;
  if (!q || !k || !vT || !o || !lse || !workspace) return ATTN_EINVAL;
  if (workspace_bytes < attn_fwd_workspace_bytes(T, heads, kv_heads)) return ATTN_EINVAL;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_EALIGN;
  DeviceState *st = nullptr;
  if ((rc = device_state(&st))) return rc;   // before the pipeline: reports a missing device
  const Sizes z = sizes_of(T, heads, kv_heads);
  auto up = [](size_t n) { return (n + 255) & ~(size_t)255; };
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  uint8_t *dq = ws, *dk = dq + up(z.q), *dv = dk + up(z.kv), *dout = dv + up(z.kv),
          *dlse = dout + up(z.o);
  std::lock_guard<std::mutex> lock(g_pipe_mutex);   // one call's events at a time
  HostPipe *hp = nullptr;
  if ((rc = host_pipe(&hp))) return rc;
  const int group = heads / kv_heads;
  const int chunks = kv_heads < kHostChunks ? kv_heads : kHostChunks;
  const size_t head_bytes = (size_t)T * kHeadDim * 2;   // one head of Q, K or V^T
  bool ok = cudaEventRecord(hp->start, stream) == cudaSuccess &&
            cudaStreamWaitEvent(hp->in, hp->start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(hp->out, hp->start, 0) == cudaSuccess;
  size_t o_off = 0;   // chunk c's O, [T][its heads x 64], lies whole in the device O region
  for (int ch = 0; ok && ch < chunks; ++ch) {
    const int g0 = (int)((long long)kv_heads * ch / chunks);
    const int g1 = (int)((long long)kv_heads * (ch + 1) / chunks);
    const int h0 = g0 * group, hc = (g1 - g0) * group;
    const uint8_t *hq = static_cast<const uint8_t *>(q) + (size_t)h0 * head_bytes;
    const uint8_t *hk = static_cast<const uint8_t *>(k) + (size_t)g0 * head_bytes;
    const uint8_t *hv = static_cast<const uint8_t *>(vT) + (size_t)g0 * head_bytes;
    uint8_t *cq = dq + (size_t)h0 * head_bytes, *ck = dk + (size_t)g0 * head_bytes,
            *cv = dv + (size_t)g0 * head_bytes, *co = dout + o_off;
    float *clse = reinterpret_cast<float *>(dlse) + (size_t)h0 * T;
    ok = cudaMemcpyAsync(cq, hq, (size_t)hc * head_bytes, cudaMemcpyHostToDevice, hp->in) ==
             cudaSuccess &&
         cudaMemcpyAsync(ck, hk, (size_t)(g1 - g0) * head_bytes, cudaMemcpyHostToDevice, hp->in) ==
             cudaSuccess &&
         cudaMemcpyAsync(cv, hv, (size_t)(g1 - g0) * head_bytes, cudaMemcpyHostToDevice, hp->in) ==
             cudaSuccess &&
         cudaEventRecord(hp->in_done[ch], hp->in) == cudaSuccess &&
         cudaStreamWaitEvent(stream, hp->in_done[ch], 0) == cudaSuccess;
    if (!ok) break;
    if ((rc = attn_fwd(cq, ck, cv, co, clse, T, hc, g1 - g0, c, stream))) return rc;
    // O's chunk is a column block of the host's [T][heads x 64]: a 2-D copy
    ok = cudaEventRecord(hp->comp_done[ch], stream) == cudaSuccess &&
         cudaStreamWaitEvent(hp->out, hp->comp_done[ch], 0) == cudaSuccess &&
         cudaMemcpy2DAsync(static_cast<uint8_t *>(o) + (size_t)h0 * kHeadDim * 2,
                           (size_t)heads * kHeadDim * 2, co, (size_t)hc * kHeadDim * 2,
                           (size_t)hc * kHeadDim * 2, T, cudaMemcpyDeviceToHost, hp->out) ==
             cudaSuccess &&
         cudaMemcpyAsync(lse + (size_t)h0 * T, clse, (size_t)hc * T * 4, cudaMemcpyDeviceToHost,
                         hp->out) == cudaSuccess;
    o_off += (size_t)hc * head_bytes;
  }
  // the caller's stream completes only after the last copy out
  ok = ok && cudaEventRecord(hp->done, hp->out) == cudaSuccess &&
       cudaStreamWaitEvent(stream, hp->done, 0) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return ATTN_ELAUNCH;
  }
  return ATTN_OK;
}

extern "C" int attn_last_device_status(cudaStream_t stream) {
  DeviceState *st = nullptr;
  int rc = device_state(&st);
  if (rc) return rc;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ELAUNCH;
  int word = 0;
  if (cudaMemcpy(&word, st->scratch + kScratchStatus, sizeof(int), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return ATTN_ELAUNCH;
  // an aborted launch may also have left its work counters set: clear them all
  if (word != 0 && cudaMemset(st->scratch, 0, kScratchInts * sizeof(int)) != cudaSuccess)
    return ATTN_ELAUNCH;
  return word ? ATTN_ETIMEOUT : ATTN_OK;
}

// ============================================================================
// attn_fwd_noalloc: the same kernel with its scratch (the status word) in a
// fixed array compiled into this library instead of a cudaMalloc'd word.

// 256 bytes (64 words), held by every GPU that loads this library until the
// process exits: the status word at [0], words [1, 32) unused, and 16
// work-counter slots of two words at [32, 64).  Host code must not use this
// name as a device address: it gets the address from cudaGetSymbolAddress.
constexpr int kNoAllocSchedSlots = 16;
constexpr int kNoAllocScratchInts = kScratchSched + 2 * kNoAllocSchedSlots;
static __device__ __align__(256) int g_noalloc_scratch[64];
static_assert(kNoAllocScratchInts * sizeof(int) <= sizeof(g_noalloc_scratch),
              "the kernel's scratch must fit the fixed array");

namespace {

struct NoAllocState {
  bool ready = false;
  int sms = 0;
  int *scratch = nullptr;  // device address of g_noalloc_scratch on this device
  unsigned calls = 0;      // launches so far; picks the counter slot
};
NoAllocState g_noalloc[64];

// Once per device, with that device current: checks the device, sets the
// kernel's shared-memory attribute and looks up the array's device address.
int noalloc_state(NoAllocState **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return ATTN_EDEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  NoAllocState &st = g_noalloc[dev];
  if (!st.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return ATTN_EDEVICE;
    if (prop.major != 10 || prop.minor != 3) return ATTN_EDEVICE;
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void *fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return ATTN_ELAUNCH;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (!set_smem_attributes()) return ATTN_ELAUNCH;
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return ATTN_ELAUNCH;
    }
    st.scratch = static_cast<int *>(ptr);
    st.sms = prop.multiProcessorCount;
    st.ready = true;
  }
  *out = &st;
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_fwd_noalloc(const void *q, const void *k, const void *vT, void *o, float *lse,
                                int T, int heads, int kv_heads, float c, int *status,
                                cudaStream_t stream) {
  int rc = check_args(q, k, vT, o, lse, T, heads, kv_heads, c);
  if (rc) return rc;
  if (status) {
    // the status copy is stream-ordered: pageable host memory would make it
    // synchronous (and it cannot be captured), so only device, managed or
    // page-locked host memory is accepted
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, status) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_EINVAL;
    }
    if (attr.type == cudaMemoryTypeUnregistered) return ATTN_EINVAL;
  }
  NoAllocState *st = nullptr;
  if ((rc = noalloc_state(&st))) return rc;
  CUtensorMap tm[3];
  Params p;
  const bool split = use_split(T, heads, st->sms);
  if (!prepare(q, k, vT, o, lse, T, heads, kv_heads, c, split, tm, &p)) return ATTN_ELAUNCH;
  unsigned slot;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    slot = st->calls++ % kNoAllocSchedSlots;
  }
  p.status = st->scratch + kScratchStatus;
  p.sched = st->scratch + kScratchSched + 2 * slot;
  // the array keeps the previous call's contents: the kernel only ever sets the
  // status word from 0, and counts units from a zeroed counter slot
  if (cudaMemsetAsync(p.status, 0, sizeof(int), stream) != cudaSuccess ||
      cudaMemsetAsync(p.sched, 0, 2 * sizeof(int), stream) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ELAUNCH;
  }
  const int grid = p.units < st->sms ? p.units : st->sms;
  launch_kernel<false>(split, grid, stream, tm, p);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
  if (status && cudaMemcpyAsync(status, p.status, sizeof(int), cudaMemcpyDefault, stream) !=
                    cudaSuccess) {
    cudaGetLastError();
    return ATTN_ELAUNCH;
  }
  return ATTN_OK;
}

extern "C" int attn_test_set_split_mode(int mode) {
  if (mode < -1 || mode > 1) return ATTN_EINVAL;
  std::lock_guard<std::mutex> lock(g_mutex);
  g_split_mode = mode;
  return ATTN_OK;
}

extern "C" int attn_test_inject_stall(void) {
  std::lock_guard<std::mutex> lock(g_mutex);
  g_stall_launches = 1;
  return ATTN_OK;
}

extern "C" const char *attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_EINVAL: return "invalid argument (shape, scale or null pointer)";
    case ATTN_EALIGN: return "pointer not 16-byte aligned";
    case ATTN_EOVERLAP: return "an output overlaps an input or the other output";
    case ATTN_ELAUNCH: return "CUDA runtime refused a copy, the set-up or the launch";
    case ATTN_EDEVICE: return "no sm_103 (GB300) CUDA device is current";
    case ATTN_ETIMEOUT: return "a kernel wait timed out; outputs are not valid";
    default: return "unknown status";
  }
}
