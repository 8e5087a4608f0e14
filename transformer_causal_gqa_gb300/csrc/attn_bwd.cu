// attn_bwd.cu -- backward pass of the causal grouped-query attention for GB300
// (sm_103a), behind the C ABI of attn_bwd.h.
//
// What it computes is the backward statement of the page
// "Realization/Nvidia/SM86/StreamingAttentionSM86.alpha": with the forward's
// output O and base-2 log-sum-exp L, P = 2^(S c - L) is recomputed tile by
// tile; dP = dO V^T; the row term D = rowsum(dO O); dS = P (dP - D); then
// dQ = s dS K, dK = s dS^T Q and dV = P^T dO, s the natural score scale, and
// dK, dV are summed over the query heads that share a K/V head.  P and dS are
// rounded to binary16 for their products; every sum stays binary32.
//
// GB300 realisation: two persistent warp-specialised kernels (one TMA warp,
// tcgen05 MMA issuer warps, four compute warps with one thread per
// tensor-memory lane).  The query launch makes D and dQ per (query head,
// 128-row tile); the key launch makes dK and dV per (K/V head, 128-key tile)
// and runs over every query head of the group in turn, so the group sum
// happens in the tensor-memory accumulator instead of a separate reduce pass.
// Products whose B operand would run along the wrong dimension read
// transposed copies (V, K^T, Q^T, dO^T) that a transpose kernel writes into
// the caller's workspace first, so every MMA operand is K-major.  Every wait
// is bounded (1 s), as in the forward.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_bwd.h"
#include "sm103_ptx.cuh"

namespace {

using namespace sm103;

constexpr int kD = 64;                            // head width
constexpr int kTile = 128;                        // query rows / keys per tile (= TMEM lanes)
constexpr uint32_t kTileBytes = kTile * kD * 2;   // one binary16 tile: 16 KiB
constexpr uint32_t kHalfTileBytes = kTileBytes / 2;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kThreads = 256;                     // 8 warps
constexpr uint32_t kTmemCols = 512;

// ---------------------------------------------------------------------------- shared pieces
struct Sync {
  uint32_t bar0;
  volatile int *abort_flag;
  int *status;
  __device__ __forceinline__ uint32_t bar(int i) const { return bar0 + 8u * i; }
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
  __device__ bool wait_warp(int i, uint32_t parity, int where) const {
    const bool ok = wait(i, parity, where);
    return __all_sync(0xffffffffu, ok);
  }
  __device__ void drain_wait(int i, uint32_t parity) const {
    const uint32_t b = bar(i);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(b, parity))
      if (globaltimer_ns() - t0 > kWaitLimitNs) break;
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

// 1-D bulk copy global -> shared, counted in bytes on `bar` (size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

struct BwdParams {
  int T, heads, kv_heads, group;
  int q_tiles;        // ceil(T / 128)
  float c, s;
  const float *lse;   // [H][T]
  const __half *o;    // [T][H*64]
  const __half *dO;   // [T][H*64]
  float *D;           // [H][T] row terms (query launch writes, key launch reads)
  float *dq;          // [H][T][64]
  float *dk;          // [G][T][64]
  float *dvT;         // [G][64][T]
  int *status;
};

// k-th unit of this CTA (static, serpentine over the grid; units are numbered
// heaviest first); -1 when done.
__device__ __forceinline__ int unit_of(int k, int units) {
  const int G = gridDim.x;
  const int slot = (k & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x;
  const int u = k * G + slot;
  return u < units ? u : -1;
}

// ============================================================================ query launch
// Unit = (query head h, 128-row query tile qt), latest (heaviest) tiles first;
// key tiles 0 .. qt.  Tensor memory: S at 0, dP at 128 (fp32, 128 columns
// each), dS at 256 (binary16 pairs, 64 columns), dQ at 320 (fp32, 64 columns).
namespace qlaunch {
constexpr int kStages = 3;                       // ring of {K, V, K^T} tiles
constexpr uint32_t kStageBytes = 3 * kTileBytes;
constexpr uint32_t kOffQ = 0;                    // Q tile, dO tile
constexpr uint32_t kOffRing = 2 * kTileBytes;
constexpr uint32_t kOffBar = kOffRing + kStages * kStageBytes;
constexpr int kBarQFull = 0, kBarQEmpty = 1;
constexpr int kBarKvFull = 2, kBarKvEmpty = 2 + kStages;
constexpr int kBarSFull = 2 + 2 * kStages, kBarSFree = kBarSFull + 1;
constexpr int kBarDsFull = kBarSFree + 1, kBarDqDone = kBarDsFull + 1;
constexpr int kBarDrain = kBarDqDone + 1;        // + issuer warp (0, 1)
constexpr int kNumBars = kBarDrain + 2;
constexpr uint32_t kOffTmemPtr = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemPtr + 4;
constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;
constexpr uint32_t kColS = 0, kColDP = 128, kColDS = 256, kColDQ = 320;
constexpr int kWarpSdp = 4, kWarpDq = 5, kWarpLoad = 6;

struct Unit {
  int h, g, qt, nk;   // nk: key tiles 0 .. qt (the diagonal)
};
__device__ __forceinline__ Unit decode(int u, const BwdParams &p) {
  Unit w;
  const int r = u / p.heads;
  w.h = u - r * p.heads;
  w.qt = p.q_tiles - 1 - r;
  w.g = w.h / p.group;
  w.nk = w.qt + 1;
  return w;
}

__device__ void load_role(const CUtensorMap *tmQ, const CUtensorMap *tmDO, const CUtensorMap *tmK,
                          const CUtensorMap *tmV, const CUtensorMap *tmKT, const BwdParams &p,
                          const Sync &sy, uint32_t smem) {
  const int units = p.heads * p.q_tiles;
  uint32_t pos = 0, pos_issued = 0, q_issued = 0;
  int k = 0;
  for (int u = unit_of(0, units); u >= 0; u = unit_of(++k, units)) {
    const Unit w = decode(u, p);
    if (!sy.wait(kBarQEmpty, (k & 1) ^ 1, 101)) goto drain;
    ++q_issued;
    mbar_arrive_expect_tx(sy.bar(kBarQFull), 2 * kTileBytes);
    tma_load_3d(smem + kOffQ, tmQ, sy.bar(kBarQFull), 0, w.qt * kTile, w.h);
    tma_load_3d(smem + kOffQ + kTileBytes, tmDO, sy.bar(kBarQFull), w.h * kD, w.qt * kTile, 0);
    for (int j = 0; j < w.nk; ++j, ++pos) {
      const uint32_t st = pos % kStages;
      if (!sy.wait(kBarKvEmpty + st, ((pos / kStages) & 1) ^ 1, 102)) goto drain;
      const uint32_t dst = smem + kOffRing + st * kStageBytes;
      const uint32_t full = sy.bar(kBarKvFull + st);
      mbar_arrive_expect_tx(full, kStageBytes);
      pos_issued = pos + 1;
      tma_load_3d(dst, tmK, full, 0, j * kTile, w.g);
      tma_load_3d(dst + kTileBytes, tmV, full, 0, j * kTile, w.g);
      tma_load_3d(dst + 2 * kTileBytes, tmKT, full, j * kTile, 0, w.g);
      tma_load_3d(dst + 2 * kTileBytes + kHalfTileBytes, tmKT, full, j * kTile + kTile / 2, 0, w.g);
    }
  }
  return;
drain:
  for (uint32_t i = 0; i < kStages && i < pos_issued; ++i) {
    const uint32_t q = pos_issued - 1 - i;
    sy.drain_wait(kBarKvFull + q % kStages, (q / kStages) & 1);
  }
  if (q_issued > 0) sy.drain_wait(kBarQFull, (q_issued - 1) & 1);
}

// S = Q K^T and dP = dO V^T for every key tile, once the compute warps have
// pulled the previous pair into registers.
__device__ void sdp_role(const BwdParams &p, const Sync &sy, uint32_t smem, uint32_t tmem) {
  constexpr uint32_t id = idesc_f16_f32(kTile, kTile);
  const int units = p.heads * p.q_tiles;
  uint32_t pos = 0, issued = 0;
  int k = 0;
  for (int u = unit_of(0, units); u >= 0; u = unit_of(++k, units)) {
    const Unit w = decode(u, p);
    if (!sy.wait_warp(kBarQFull, k & 1, 111)) goto drain;
    tc_fence_after();
    for (int j = 0; j < w.nk; ++j, ++pos) {
      const uint32_t st = pos % kStages;
      if (!sy.wait_warp(kBarKvFull + st, (pos / kStages) & 1, 112)) goto drain;
      if (!sy.wait_warp(kBarSFree, (issued & 1) ^ 1, 113)) goto drain;
      ++issued;
      tc_fence_after();
      const uint32_t kb = smem + kOffRing + st * kStageBytes;
#pragma unroll
      for (int e = 0; e < kD / 16; ++e)
        mma_ss(tmem + kColS, sw128_desc(smem + kOffQ + e * 32), sw128_desc(kb + e * 32), id,
               e > 0 ? 1u : 0u);
#pragma unroll
      for (int e = 0; e < kD / 16; ++e)
        mma_ss(tmem + kColDP, sw128_desc(smem + kOffQ + kTileBytes + e * 32),
               sw128_desc(kb + kTileBytes + e * 32), id, e > 0 ? 1u : 0u);
      mma_commit(sy.bar(kBarSFull));
      mma_commit(sy.bar(kBarKvEmpty + st));
    }
    mma_commit(sy.bar(kBarQEmpty));
  }
  return;
drain:
  mma_commit(sy.bar(kBarDrain + 0));
  sy.drain_wait(kBarDrain + 0, 0);
}

// dQ += dS K (A = dS from tensor memory, B = K^T, K-major over keys).
__device__ void dq_role(const BwdParams &p, const Sync &sy, uint32_t smem, uint32_t tmem) {
  constexpr uint32_t id = idesc_f16_f32(kTile, kD);
  const int units = p.heads * p.q_tiles;
  uint32_t pos = 0, dphase = 0;
  int k = 0;
  for (int u = unit_of(0, units); u >= 0; u = unit_of(++k, units)) {
    const Unit w = decode(u, p);
    for (int j = 0; j < w.nk; ++j, ++pos) {
      const uint32_t st = pos % kStages;
      if (!sy.wait_warp(kBarDsFull, dphase, 121)) goto drain;
      dphase ^= 1;
      if (!sy.wait_warp(kBarKvFull + st, (pos / kStages) & 1, 122)) goto drain;
      tc_fence_after();
      const uint32_t ktb = smem + kOffRing + st * kStageBytes + 2 * kTileBytes;
#pragma unroll
      for (int e = 0; e < kTile / 16; ++e)
        mma_ts(tmem + kColDQ, tmem + kColDS + 8u * e,
               sw128_desc(ktb + (e >> 2) * kHalfTileBytes + (e & 3) * 32), id,
               (j > 0 || e > 0) ? 1u : 0u);
      mma_commit(sy.bar(kBarDqDone));
      mma_commit(sy.bar(kBarKvEmpty + st));
    }
  }
  return;
drain:
  mma_commit(sy.bar(kBarDrain + 1));
  sy.drain_wait(kBarDrain + 1, 0);
}

// Compute warps: thread r owns query row r of the tile (tensor-memory lane r).
__device__ void compute_role(const BwdParams &p, const Sync &sy, uint32_t tmem) {
  const int r = threadIdx.x & 127;
  const bool leader = (threadIdx.x & 31) == 0;
  const uint32_t lane_base = (uint32_t)(threadIdx.x & 96) << 16;
  const float c = p.c;
  const int units = p.heads * p.q_tiles;
  uint32_t sphase = 0, dqphase = 0;
  int k = 0;
  for (int u = unit_of(0, units); u >= 0; u = unit_of(++k, units)) {
    const Unit w = decode(u, p);
    const int row = w.qt * kTile + r;
    const bool valid = row < p.T;
    // the row term D = rowsum(dO O) and the forward's L for this row
    float L = 0.f, D = 0.f;
    if (valid) {
      const size_t at = ((size_t)row * p.heads + w.h) * kD;
      const uint4 *go = reinterpret_cast<const uint4 *>(p.dO + at);
      const uint4 *oo = reinterpret_cast<const uint4 *>(p.o + at);
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 a = go[i], b = oo[i];
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float2 fa = __half22float2(*reinterpret_cast<const __half2 *>(&av[t]));
          const float2 fb = __half22float2(*reinterpret_cast<const __half2 *>(&bv[t]));
          acc0 = fmaf(fa.x, fb.x, acc0);
          acc1 = fmaf(fa.y, fb.y, acc1);
        }
      }
      D = acc0 + acc1;
      L = p.lse[(size_t)w.h * p.T + row];
      p.D[(size_t)w.h * p.T + row] = D;
    }
    const float negL = -L;
    for (int j = 0; j < w.nk; ++j) {
      if (!sy.wait_warp(kBarSFull, sphase, 131)) return;
      sphase ^= 1;
      tc_fence_after();
      uint32_t pk[64];   // dS row: columns 2m, 2m+1 in pk[m]
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t sr[32], dr[32];
        tmem_ld_x32(tmem + lane_base + kColS + 32u * c4, sr);
        tmem_ld_x32(tmem + lane_base + kColDP + 32u * c4, dr);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int col = 32 * c4 + 2 * i;
          float p0 = ex2(fmaf(__uint_as_float(sr[2 * i]), c, negL));
          float p1 = ex2(fmaf(__uint_as_float(sr[2 * i + 1]), c, negL));
          if (j == w.qt) {            // diagonal tile: keys after the row get P = 0
            if (col > r) p0 = 0.f;
            if (col + 1 > r) p1 = 0.f;
          }
          const float ds0 = p0 * (__uint_as_float(dr[2 * i]) - D);
          const float ds1 = p1 * (__uint_as_float(dr[2 * i + 1]) - D);
          pk[16 * c4 + i] = pack_half2(ds0, ds1);
        }
      }
      // S and dP are in registers: the next pair may be computed over them
      tc_fence_before();
      __syncwarp();
      if (leader) mbar_arrive(sy.bar(kBarSFree));
      if (j > 0) {   // dS(j-1) K must be complete before dS is overwritten
        if (!sy.wait_warp(kBarDqDone, dqphase, 132)) return;
        dqphase ^= 1;
        tc_fence_after();
      }
      tmem_st_x64(tmem + lane_base + kColDS, pk);
      tc_fence_before();
      __syncwarp();
      if (leader) mbar_arrive(sy.bar(kBarDsFull));
    }
    // epilogue: dQ = s (sum) once the last product is done
    if (!sy.wait_warp(kBarDqDone, dqphase, 133)) return;
    dqphase ^= 1;
    tc_fence_after();
    uint32_t qr[64];
    tmem_ld_x64(tmem + lane_base + kColDQ, qr);
    if (valid) {
      float4 *dst = reinterpret_cast<float4 *>(p.dq + ((size_t)w.h * p.T + row) * kD);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        dst[i] = make_float4(__uint_as_float(qr[4 * i]) * p.s, __uint_as_float(qr[4 * i + 1]) * p.s,
                             __uint_as_float(qr[4 * i + 2]) * p.s, __uint_as_float(qr[4 * i + 3]) * p.s);
    }
    tc_fence_before();
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    query_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                 const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmKT, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t smem = (raw + 1023u) & ~1023u;
  uint8_t *smem_gen = smem_raw + (smem - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Sync sy;
  sy.bar0 = smem + kOffBar;
  sy.abort_flag = reinterpret_cast<volatile int *>(smem_gen + kOffAbort);
  sy.status = p.status;
  if (warp == kWarpLoad && lane == 0) {
    mbar_init(sy.bar(kBarQFull), 1);
    mbar_init(sy.bar(kBarQEmpty), 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(sy.bar(kBarKvFull + i), 1);
      mbar_init(sy.bar(kBarKvEmpty + i), 2);   // S/dP issuer and dQ issuer
    }
    mbar_init(sy.bar(kBarSFull), 1);
    mbar_init(sy.bar(kBarSFree), 4);
    mbar_init(sy.bar(kBarDsFull), 4);
    mbar_init(sy.bar(kBarDqDone), 1);
    mbar_init(sy.bar(kBarDrain + 0), 1);
    mbar_init(sy.bar(kBarDrain + 1), 1);
    *sy.abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kWarpSdp) {
    tmem_alloc(smem + kOffTmemPtr, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem_gen + kOffTmemPtr);
  if (warp < 4) {
    compute_role(p, sy, tmem);
  } else if (warp == kWarpSdp) {
    sdp_role(p, sy, smem, tmem);
  } else if (warp == kWarpDq) {
    dq_role(p, sy, smem, tmem);
  } else if (warp == kWarpLoad) {
    if (lane == 0) load_role(&tmQ, &tmDO, &tmK, &tmV, &tmKT, p, sy, smem);
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpSdp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}
}  // namespace qlaunch

// ============================================================================ key launch
// Unit = (K/V head g, 128-key tile kt), earliest (heaviest) tiles first.  A
// unit steps through every query head z of the group and, for each, the
// query tiles kt .. q_tiles-1, accumulating dK and dV over all of them.
// Tensor memory: S^T at 0, dP^T at 128 (fp32), P^T at 256, dS^T at 320
// (binary16 pairs), dV at 384, dK at 448 (fp32).
namespace klaunch {
constexpr int kStages = 2;   // ring of {Q, dO, Q^T, dO^T tiles, L, D}
constexpr uint32_t kStageBytes = 4 * kTileBytes + 2 * kTile * 4;
constexpr uint32_t kOffK = 0;                    // K tile, V tile
constexpr uint32_t kOffRing = 2 * kTileBytes;
constexpr uint32_t kOffBar = kOffRing + kStages * kStageBytes;
constexpr int kBarKvFull = 0, kBarKvEmpty = 1;
constexpr int kBarQFull = 2, kBarQEmpty = 2 + kStages;
constexpr int kBarSFull = 2 + 2 * kStages, kBarSFree = kBarSFull + 1;
constexpr int kBarPFull = kBarSFree + 1, kBarDvDone = kBarPFull + 1, kBarDkDone = kBarDvDone + 1;
constexpr int kBarDrain = kBarDkDone + 1;        // + issuer warp (0..2)
constexpr int kNumBars = kBarDrain + 3;
constexpr uint32_t kOffTmemPtr = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemPtr + 4;
constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;
constexpr uint32_t kColS = 0, kColDP = 128, kColP = 256, kColDS = 320, kColDV = 384, kColDK = 448;
constexpr int kWarpSdp = 4, kWarpDv = 5, kWarpDk = 6, kWarpLoad = 7;
// offsets inside a stage
constexpr uint32_t kSQ = 0, kSDO = kTileBytes, kSQT = 2 * kTileBytes, kSDOT = 3 * kTileBytes;
constexpr uint32_t kSL = 4 * kTileBytes, kSDd = kSL + kTile * 4;

struct Unit {
  int g, kt, nq, steps;   // query tiles kt .. kt + nq - 1 for each of the group's heads
};
__device__ __forceinline__ Unit decode(int u, const BwdParams &p) {
  Unit w;
  const int r = u / p.kv_heads;
  w.g = u - r * p.kv_heads;
  w.kt = r;                      // earliest key tiles see the most query tiles
  w.nq = p.q_tiles - w.kt;
  w.steps = p.group * w.nq;
  return w;
}
// step i of a unit: query head and query tile
__device__ __forceinline__ void step_of(const Unit &w, int i, const BwdParams &p, int &h, int &qt) {
  const int z = i / w.nq;
  h = w.g * p.group + z;
  qt = w.kt + (i - z * w.nq);
}

__device__ void load_role(const CUtensorMap *tmK, const CUtensorMap *tmV, const CUtensorMap *tmQ,
                          const CUtensorMap *tmDO, const CUtensorMap *tmQT,
                          const CUtensorMap *tmDOT, const BwdParams &p, const Sync &sy,
                          uint32_t smem) {
  const int units = p.kv_heads * p.q_tiles;
  uint32_t pos = 0, pos_issued = 0, kv_issued = 0;
  int k = 0;
  for (int u = unit_of(0, units); u >= 0; u = unit_of(++k, units)) {
    const Unit w = decode(u, p);
    if (!sy.wait(kBarKvEmpty, (k & 1) ^ 1, 201)) goto drain;
    ++kv_issued;
    mbar_arrive_expect_tx(sy.bar(kBarKvFull), 2 * kTileBytes);
    tma_load_3d(smem + kOffK, tmK, sy.bar(kBarKvFull), 0, w.kt * kTile, w.g);
    tma_load_3d(smem + kOffK + kTileBytes, tmV, sy.bar(kBarKvFull), 0, w.kt * kTile, w.g);
    for (int i = 0; i < w.steps; ++i, ++pos) {
      int h, qt;
      step_of(w, i, p, h, qt);
      const uint32_t st = pos % kStages;
      if (!sy.wait(kBarQEmpty + st, ((pos / kStages) & 1) ^ 1, 202)) goto drain;
      const uint32_t dst = smem + kOffRing + st * kStageBytes;
      const uint32_t full = sy.bar(kBarQFull + st);
      const int rows = min(kTile, p.T - qt * kTile);      // query rows that exist (64 or 128)
      mbar_arrive_expect_tx(full, 4 * kTileBytes + 2 * rows * 4);
      pos_issued = pos + 1;
      tma_load_3d(dst + kSQ, tmQ, full, 0, qt * kTile, h);
      tma_load_3d(dst + kSDO, tmDO, full, h * kD, qt * kTile, 0);
      tma_load_3d(dst + kSQT, tmQT, full, qt * kTile, 0, h);
      tma_load_3d(dst + kSQT + kHalfTileBytes, tmQT, full, qt * kTile + kTile / 2, 0, h);
      tma_load_3d(dst + kSDOT, tmDOT, full, qt * kTile, 0, h);
      tma_load_3d(dst + kSDOT + kHalfTileBytes, tmDOT, full, qt * kTile + kTile / 2, 0, h);
      bulk_load(dst + kSL, p.lse + (size_t)h * p.T + qt * kTile, rows * 4, full);
      bulk_load(dst + kSDd, p.D + (size_t)h * p.T + qt * kTile, rows * 4, full);
    }
  }
  return;
drain:
  for (uint32_t i = 0; i < kStages && i < pos_issued; ++i) {
    const uint32_t q = pos_issued - 1 - i;
    sy.drain_wait(kBarQFull + q % kStages, (q / kStages) & 1);
  }
  if (kv_issued > 0) sy.drain_wait(kBarKvFull, (kv_issued - 1) & 1);
}

// S^T = K Q^T and dP^T = V dO^T per step.
__device__ void sdp_role(const BwdParams &p, const Sync &sy, uint32_t smem, uint32_t tmem) {
  constexpr uint32_t id = idesc_f16_f32(kTile, kTile);
  const int units = p.kv_heads * p.q_tiles;
  uint32_t pos = 0, issued = 0;
  int k = 0;
  for (int u = unit_of(0, units); u >= 0; u = unit_of(++k, units)) {
    const Unit w = decode(u, p);
    if (!sy.wait_warp(kBarKvFull, k & 1, 211)) goto drain;
    tc_fence_after();
    for (int i = 0; i < w.steps; ++i, ++pos) {
      const uint32_t st = pos % kStages;
      if (!sy.wait_warp(kBarQFull + st, (pos / kStages) & 1, 212)) goto drain;
      if (!sy.wait_warp(kBarSFree, (issued & 1) ^ 1, 213)) goto drain;
      ++issued;
      tc_fence_after();
      const uint32_t sb = smem + kOffRing + st * kStageBytes;
#pragma unroll
      for (int e = 0; e < kD / 16; ++e)
        mma_ss(tmem + kColS, sw128_desc(smem + kOffK + e * 32), sw128_desc(sb + kSQ + e * 32), id,
               e > 0 ? 1u : 0u);
#pragma unroll
      for (int e = 0; e < kD / 16; ++e)
        mma_ss(tmem + kColDP, sw128_desc(smem + kOffK + kTileBytes + e * 32),
               sw128_desc(sb + kSDO + e * 32), id, e > 0 ? 1u : 0u);
      mma_commit(sy.bar(kBarSFull));
      mma_commit(sy.bar(kBarQEmpty + st));
    }
    mma_commit(sy.bar(kBarKvEmpty));
  }
  return;
drain:
  mma_commit(sy.bar(kBarDrain + 0));
  sy.drain_wait(kBarDrain + 0, 0);
}

// dV += P^T dO (B = dO^T) when which == 0, dK += dS^T Q (B = Q^T) when which == 1.
__device__ void acc_role(int which, const BwdParams &p, const Sync &sy, uint32_t smem,
                         uint32_t tmem) {
  constexpr uint32_t id = idesc_f16_f32(kTile, kD);
  const int units = p.kv_heads * p.q_tiles;
  const uint32_t a_col = which ? kColDS : kColP;
  const uint32_t d_col = which ? kColDK : kColDV;
  const uint32_t b_off = which ? kSQT : kSDOT;
  const int done_bar = which ? kBarDkDone : kBarDvDone;
  uint32_t pos = 0, pphase = 0;
  int k = 0;
  for (int u = unit_of(0, units); u >= 0; u = unit_of(++k, units)) {
    const Unit w = decode(u, p);
    for (int i = 0; i < w.steps; ++i, ++pos) {
      const uint32_t st = pos % kStages;
      if (!sy.wait_warp(kBarPFull, pphase, 221 + which)) goto drain;
      pphase ^= 1;
      if (!sy.wait_warp(kBarQFull + st, (pos / kStages) & 1, 223 + which)) goto drain;
      tc_fence_after();
      const uint32_t bb = smem + kOffRing + st * kStageBytes + b_off;
#pragma unroll
      for (int e = 0; e < kTile / 16; ++e)
        mma_ts(tmem + d_col, tmem + a_col + 8u * e,
               sw128_desc(bb + (e >> 2) * kHalfTileBytes + (e & 3) * 32), id,
               (i > 0 || e > 0) ? 1u : 0u);
      mma_commit(sy.bar(done_bar));
      mma_commit(sy.bar(kBarQEmpty + st));
    }
  }
  return;
drain:
  mma_commit(sy.bar(kBarDrain + 1 + which));
  sy.drain_wait(kBarDrain + 1 + which, 0);
}

// Compute warps: thread r owns key row r of the tile (tensor-memory lane r);
// columns are the step's 128 queries, whose L and D come from shared memory.
__device__ void compute_role(const BwdParams &p, const Sync &sy, const uint8_t *smem_gen,
                             uint32_t tmem) {
  const int r = threadIdx.x & 127;
  const bool leader = (threadIdx.x & 31) == 0;
  const uint32_t lane_base = (uint32_t)(threadIdx.x & 96) << 16;
  const float c = p.c;
  const int units = p.kv_heads * p.q_tiles;
  uint32_t pos = 0, sphase = 0, dvphase = 0, dkphase = 0;
  int k = 0;
  for (int u = unit_of(0, units); u >= 0; u = unit_of(++k, units)) {
    const Unit w = decode(u, p);
    const int key = w.kt * kTile + r;
    for (int i = 0; i < w.steps; ++i, ++pos) {
      int h, qt;
      step_of(w, i, p, h, qt);
      const uint32_t st = pos % kStages;
      // the stage's copies (L and D among them) are visible to this thread once it
      // has seen the stage's barrier complete
      if (!sy.wait_warp(kBarQFull + st, (pos / kStages) & 1, 230)) return;
      if (!sy.wait_warp(kBarSFull, sphase, 231)) return;
      sphase ^= 1;
      tc_fence_after();
      const float *Ls = reinterpret_cast<const float *>(smem_gen + kOffRing + st * kStageBytes + kSL);
      const float *Ds = reinterpret_cast<const float *>(smem_gen + kOffRing + st * kStageBytes + kSDd);
      const int first = qt * kTile - key;                // query index of column 0, minus the key
      const int qlimit = min(kTile, p.T - qt * kTile);   // columns that are real queries
      uint32_t pp[64], pd[64];   // P^T and dS^T rows: columns 2m, 2m+1 in [m]
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t sr[32], dr[32];
        tmem_ld_x32(tmem + lane_base + kColS + 32u * c4, sr);
        tmem_ld_x32(tmem + lane_base + kColDP + 32u * c4, dr);
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const int col = 32 * c4 + 4 * i4;
          const float4 L4 = *reinterpret_cast<const float4 *>(Ls + col);
          const float4 D4 = *reinterpret_cast<const float4 *>(Ds + col);
          const float Lv[4] = {L4.x, L4.y, L4.z, L4.w}, Dv[4] = {D4.x, D4.y, D4.z, D4.w};
          float pv[4], dv[4];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            // causal: query (qt*128 + col + t) sees this key when it is not earlier;
            // columns past the sequence end are not queries (their L, D are stale)
            const bool live = (first + col + t >= 0) && (col + t < qlimit);
            const float pr = ex2(fmaf(__uint_as_float(sr[4 * i4 + t]), c, -Lv[t]));
            pv[t] = live ? pr : 0.f;
            dv[t] = live ? pr * (__uint_as_float(dr[4 * i4 + t]) - Dv[t]) : 0.f;
          }
          pp[16 * c4 + 2 * i4] = pack_half2(pv[0], pv[1]);
          pp[16 * c4 + 2 * i4 + 1] = pack_half2(pv[2], pv[3]);
          pd[16 * c4 + 2 * i4] = pack_half2(dv[0], dv[1]);
          pd[16 * c4 + 2 * i4 + 1] = pack_half2(dv[2], dv[3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (leader) mbar_arrive(sy.bar(kBarSFree));
      if (i > 0) {   // the previous step's products must be done before P^T, dS^T are overwritten
        if (!sy.wait_warp(kBarDvDone, dvphase, 232)) return;
        dvphase ^= 1;
        if (!sy.wait_warp(kBarDkDone, dkphase, 233)) return;
        dkphase ^= 1;
        tc_fence_after();
      }
      tmem_st_x64(tmem + lane_base + kColP, pp);
      tmem_st_x64(tmem + lane_base + kColDS, pd);
      tc_fence_before();
      __syncwarp();
      if (leader) mbar_arrive(sy.bar(kBarPFull));
    }
    // epilogue: dV^T and s dK for this key row
    if (!sy.wait_warp(kBarDvDone, dvphase, 234)) return;
    dvphase ^= 1;
    if (!sy.wait_warp(kBarDkDone, dkphase, 235)) return;
    dkphase ^= 1;
    tc_fence_after();
    {
      uint32_t vr[64];
      tmem_ld_x64(tmem + lane_base + kColDV, vr);
      if (key < p.T) {
        float *dvt = p.dvT + (size_t)w.g * kD * p.T + key;
#pragma unroll
        for (int e = 0; e < kD; ++e) dvt[(size_t)e * p.T] = __uint_as_float(vr[e]);
      }
    }
    {
      uint32_t kr[64];
      tmem_ld_x64(tmem + lane_base + kColDK, kr);
      if (key < p.T) {
        float4 *dk = reinterpret_cast<float4 *>(p.dk + ((size_t)w.g * p.T + key) * kD);
#pragma unroll
        for (int e = 0; e < 16; ++e)
          dk[e] = make_float4(__uint_as_float(kr[4 * e]) * p.s, __uint_as_float(kr[4 * e + 1]) * p.s,
                              __uint_as_float(kr[4 * e + 2]) * p.s, __uint_as_float(kr[4 * e + 3]) * p.s);
      }
    }
    tc_fence_before();
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    key_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ CUtensorMap tmQT, const __grid_constant__ CUtensorMap tmDOT,
               const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t smem = (raw + 1023u) & ~1023u;
  uint8_t *smem_gen = smem_raw + (smem - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Sync sy;
  sy.bar0 = smem + kOffBar;
  sy.abort_flag = reinterpret_cast<volatile int *>(smem_gen + kOffAbort);
  sy.status = p.status;
  if (warp == kWarpLoad && lane == 0) {
    mbar_init(sy.bar(kBarKvFull), 1);
    mbar_init(sy.bar(kBarKvEmpty), 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(sy.bar(kBarQFull + i), 1);
      mbar_init(sy.bar(kBarQEmpty + i), 3);   // S^T/dP^T, dV and dK issuers
    }
    mbar_init(sy.bar(kBarSFull), 1);
    mbar_init(sy.bar(kBarSFree), 4);
    mbar_init(sy.bar(kBarPFull), 4);
    mbar_init(sy.bar(kBarDvDone), 1);
    mbar_init(sy.bar(kBarDkDone), 1);
    for (int i = 0; i < 3; ++i) mbar_init(sy.bar(kBarDrain + i), 1);
    *sy.abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kWarpSdp) {
    tmem_alloc(smem + kOffTmemPtr, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem_gen + kOffTmemPtr);
  if (warp < 4) {
    compute_role(p, sy, smem_gen, tmem);
  } else if (warp == kWarpSdp) {
    sdp_role(p, sy, smem, tmem);
  } else if (warp == kWarpDv || warp == kWarpDk) {
    acc_role(warp - kWarpDv, p, sy, smem, tmem);
  } else if (warp == kWarpLoad) {
    if (lane == 0) load_role(&tmK, &tmV, &tmQ, &tmDO, &tmQT, &tmDOT, p, sy, smem);
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpSdp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}
}  // namespace klaunch

// ============================================================================ transposes
// dst[b][col][row] = src[b][row][col] for a batch of binary16 matrices whose
// rows and columns are multiples of 64, through 64 x 64 shared-memory tiles.
__global__ void __launch_bounds__(256) transpose_kernel(const __half *src, __half *dst, int rows,
                                                        int cols, long long src_ld,
                                                        long long src_batch, long long dst_ld,
                                                        long long dst_batch) {
  __shared__ __half tile[64][66];
  const int c0 = blockIdx.x * 64, r0 = blockIdx.y * 64, b = blockIdx.z;
  if (c0 + 64 > cols || r0 + 64 > rows) return;
  const __half *s = src + b * src_batch;
  __half *d = dst + b * dst_batch;
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int rr = i >> 6, cc = i & 63;
    tile[rr][cc] = s[(long long)(r0 + rr) * src_ld + c0 + cc];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int cc = i >> 6, rr = i & 63;
    d[(long long)(c0 + cc) * dst_ld + r0 + rr] = tile[rr][cc];
  }
}

// ============================================================================ host side
struct BwdState {
  bool ready = false;
  int sms = 0;
  int *status = nullptr;
};
std::mutex g_bwd_mutex;
BwdState g_bwd[64];
PFN_cuTensorMapEncodeTiled_v12000 g_bwd_encode = nullptr;

int bwd_state(BwdState **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return ATTN_EDEVICE;
  }
  std::lock_guard<std::mutex> lock(g_bwd_mutex);
  BwdState &st = g_bwd[dev];
  if (!st.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return ATTN_EDEVICE;
    if (prop.major != 10 || prop.minor != 3) return ATTN_EDEVICE;
    if (!g_bwd_encode) {
      cudaDriverEntryPointQueryResult q;
      void *fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return ATTN_ELAUNCH;
      g_bwd_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (cudaFuncSetAttribute(qlaunch::query_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)qlaunch::kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(klaunch::key_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)klaunch::kSmemBytes) != cudaSuccess)
      return ATTN_ELAUNCH;
    if (cudaMalloc(&st.status, sizeof(int)) != cudaSuccess) return ATTN_ELAUNCH;
    if (cudaMemset(st.status, 0, sizeof(int)) != cudaSuccess) return ATTN_ELAUNCH;
    st.sms = prop.multiProcessorCount;
    st.ready = true;
  }
  *out = &st;
  return ATTN_OK;
}

bool encode_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1) {
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1, stride2};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_bwd_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t up256(size_t n) { return (n + 255) & ~(size_t)255; }

// Workspace layout: V, K^T (per K/V head), Q^T, dO^T (per query head), all
// binary16, then D (binary32 [heads][T]); each part starts on 256 bytes.
struct BwdWorkspace {
  size_t v, kt, qt, dot, d, total;
};
BwdWorkspace bwd_layout(int T, int heads, int kv_heads) {
  BwdWorkspace w;
  const size_t kvb = (size_t)kv_heads * T * kD * 2, hb = (size_t)heads * T * kD * 2;
  w.v = 0;
  w.kt = w.v + up256(kvb);
  w.qt = w.kt + up256(kvb);
  w.dot = w.qt + up256(hb);
  w.d = w.dot + up256(hb);
  w.total = w.d + up256((size_t)heads * T * 4);
  return w;
}

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

int check_bwd_shape(int T, int heads, int kv_heads, float c, float s) {
  if (T <= 0 || heads <= 0 || kv_heads <= 0) return ATTN_EINVAL;
  if (T % 64 != 0) return ATTN_EINVAL;
  if (heads % kv_heads != 0) return ATTN_EINVAL;
  if (heads > ATTN_MAX_HEADS) return ATTN_EINVAL;
  if ((uint64_t)heads * 64u * (uint64_t)T * 4u > 0xFFFFFFFFull) return ATTN_EINVAL;
  if (!std::isfinite(c) || !(c > 0.f) || !std::isfinite(s) || !(s > 0.f)) return ATTN_EINVAL;
  return ATTN_OK;
}

}  // namespace

extern "C" size_t attn_bwd_workspace_bytes(int T, int heads, int kv_heads) {
  if (check_bwd_shape(T, heads, kv_heads, 1.f, 1.f)) return 0;
  return bwd_layout(T, heads, kv_heads).total;
}

extern "C" int attn_bwd(const void *q, const void *k, const void *vT, const void *o,
                        const float *lse, const void *dO, float *dq, float *dk, float *dvT,
                        int T, int heads, int kv_heads, float c, float s, void *workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_bwd_shape(T, heads, kv_heads, c, s);
  if (rc) return rc;
  const void *ins[] = {q, k, vT, o, lse, dO};
  void *outs[] = {dq, dk, dvT, workspace};
  for (const void *ptr : ins)
    if (!ptr) return ATTN_EINVAL;
  for (const void *ptr : outs)
    if (!ptr) return ATTN_EINVAL;
  for (const void *ptr : ins)
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return ATTN_EALIGN;
  for (const void *ptr : outs)
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return ATTN_EALIGN;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_EALIGN;
  const BwdWorkspace ws = bwd_layout(T, heads, kv_heads);
  if (workspace_bytes < ws.total) return ATTN_EINVAL;
  const size_t hq = (size_t)heads * T * kD, kvn = (size_t)kv_heads * T * kD;
  const size_t in_sizes[] = {hq * 2, kvn * 2, kvn * 2, hq * 2, (size_t)heads * T * 4, hq * 2};
  const size_t out_sizes[] = {hq * 4, kvn * 4, kvn * 4, ws.total};
  for (int a = 0; a < 4; ++a) {
    for (int b = 0; b < 6; ++b)
      if (ranges_overlap(outs[a], out_sizes[a], ins[b], in_sizes[b])) return ATTN_EOVERLAP;
    for (int b = a + 1; b < 4; ++b)
      if (ranges_overlap(outs[a], out_sizes[a], outs[b], out_sizes[b])) return ATTN_EOVERLAP;
  }
  BwdState *st = nullptr;
  if ((rc = bwd_state(&st))) return rc;

  uint8_t *wsb = static_cast<uint8_t *>(workspace);
  __half *Vh = reinterpret_cast<__half *>(wsb + ws.v);
  __half *KTh = reinterpret_cast<__half *>(wsb + ws.kt);
  __half *QTh = reinterpret_cast<__half *>(wsb + ws.qt);
  __half *DOTh = reinterpret_cast<__half *>(wsb + ws.dot);
  float *Dw = reinterpret_cast<float *>(wsb + ws.d);

  // transposed copies, so every MMA operand is K-major
  const dim3 tb(256);
  transpose_kernel<<<dim3(T / 64, 1, kv_heads), tb, 0, stream>>>(
      static_cast<const __half *>(vT), Vh, kD, T, T, (long long)kD * T, kD, (long long)T * kD);
  transpose_kernel<<<dim3(1, T / 64, kv_heads), tb, 0, stream>>>(
      static_cast<const __half *>(k), KTh, T, kD, kD, (long long)T * kD, T, (long long)kD * T);
  transpose_kernel<<<dim3(1, T / 64, heads), tb, 0, stream>>>(
      static_cast<const __half *>(q), QTh, T, kD, kD, (long long)T * kD, T, (long long)kD * T);
  transpose_kernel<<<dim3(1, T / 64, heads), tb, 0, stream>>>(
      static_cast<const __half *>(dO), DOTh, T, kD, (long long)heads * kD, kD, T,
      (long long)kD * T);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;

  const uint64_t rowb = kD * 2, trow = (uint64_t)T * 2;
  CUtensorMap tmQ, tmK, tmV, tmKT, tmQT, tmDOT, tmDO;
  if (!encode_3d(&tmQ, q, kD, T, heads, rowb, rowb * T, kD, kTile) ||
      !encode_3d(&tmK, k, kD, T, kv_heads, rowb, rowb * T, kD, kTile) ||
      !encode_3d(&tmV, Vh, kD, T, kv_heads, rowb, rowb * T, kD, kTile) ||
      !encode_3d(&tmKT, KTh, T, kD, kv_heads, trow, trow * kD, kTile / 2, kD) ||
      !encode_3d(&tmQT, QTh, T, kD, heads, trow, trow * kD, kTile / 2, kD) ||
      !encode_3d(&tmDOT, DOTh, T, kD, heads, trow, trow * kD, kTile / 2, kD) ||
      !encode_3d(&tmDO, dO, (uint64_t)heads * kD, T, 1, (uint64_t)heads * kD * 2,
                 (uint64_t)heads * kD * 2 * T, kD, kTile))
    return ATTN_ELAUNCH;

  BwdParams p;
  p.T = T;
  p.heads = heads;
  p.kv_heads = kv_heads;
  p.group = heads / kv_heads;
  p.q_tiles = (T + kTile - 1) / kTile;
  p.c = c;
  p.s = s;
  p.lse = lse;
  p.o = static_cast<const __half *>(o);
  p.dO = static_cast<const __half *>(dO);
  p.D = Dw;
  p.dq = dq;
  p.dk = dk;
  p.dvT = dvT;
  p.status = st->status;
  const int qunits = heads * p.q_tiles, kunits = kv_heads * p.q_tiles;
  qlaunch::query_kernel<<<qunits < st->sms ? qunits : st->sms, kThreads, qlaunch::kSmemBytes,
                          stream>>>(tmQ, tmDO, tmK, tmV, tmKT, p);
  klaunch::key_kernel<<<kunits < st->sms ? kunits : st->sms, kThreads, klaunch::kSmemBytes,
                        stream>>>(tmK, tmV, tmQ, tmDO, tmQT, tmDOT, p);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
  return ATTN_OK;
}

extern "C" int attn_bwd_last_device_status(cudaStream_t stream) {
  BwdState *st = nullptr;
  int rc = bwd_state(&st);
  if (rc) return rc;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ELAUNCH;
  int word = 0;
  if (cudaMemcpy(&word, st->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ELAUNCH;
  if (word != 0 && cudaMemset(st->status, 0, sizeof(int)) != cudaSuccess) return ATTN_ELAUNCH;
  return word ? ATTN_ETIMEOUT : ATTN_OK;
}
