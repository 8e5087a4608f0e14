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
// tcgen05 MMA issuer warps, eight compute warps, one tile row per thread and
// half the tile's columns per warpgroup).  The query launch makes D and dQ
// per (query head, 128-row tile); the key launch makes dK and dV per (K/V
// head, 128-key tile) and runs over every query head of the group in turn, so
// the group sum happens in the tensor-memory accumulator instead of a
// separate reduce pass.  Operands are read where they lie: a product whose
// operand runs along the other dimension (V^T for dP, K for dQ, Q and dO for
// dK and dV) reads its tile MN-major, so nothing is transposed in memory.
// Every wait is bounded (1 s), as in the forward.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
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
  // Two waits taken together: both barriers are tested back to back, so a pair
  // that is already complete costs one round trip instead of two.
  __device__ bool wait2_warp(int i, uint32_t pi, int wi, int j, uint32_t pj, int wj) const {
    const bool a = mbar_test_wait(bar(i), pi);
    const bool b = mbar_test_wait(bar(j), pj);
    if (__all_sync(0xffffffffu, a && b)) return true;
    return wait_warp(i, pi, wi) && wait_warp(j, pj, wj);
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

// Paired IEEE binary32 arithmetic, one f32x2 instruction each:
// (d0, d1) = (a0 b + c0, a1 b + c1)
__device__ __forceinline__ void fma2(float &d0, float &d1, float a0, float a1, float b, float c0, float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %4};\n\t"
      "mov.b64 rc, {%5, %6};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c0), "f"(c1));
}
// (d0, d1) = (p0 (q0 - r0), p1 (q1 - r1))
__device__ __forceinline__ void mulsub2(float &d0, float &d1, float p0, float p1, float q0, float q1,
                                        float r0, float r1) {
  asm("{\n\t.reg .b64 rp, rq, rr, rd;\n\t"
      "mov.b64 rp, {%2, %3};\n\t"
      "mov.b64 rq, {%4, %5};\n\t"
      "mov.b64 rr, {%6, %7};\n\t"
      "sub.f32x2 rd, rq, rr;\n\t"
      "mul.f32x2 rd, rp, rd;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(p0), "f"(p1), "f"(q0), "f"(q1), "f"(r0), "f"(r1));
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
  // Short problems: each key-launch unit's steps are shared out over `splits`
  // units, each writing its partial dK (already times s) and dV^T into plane
  // `split` of these workspace arrays, [splits][G][T][64] and [splits][G][64][T];
  // a reduce launch sums the planes.  splits == 1: written to dk, dvT directly.
  int splits;
  float *dk_part;
  float *dv_part;
  int *status;
  int stall;          // test hook: CTA 0 of the query launch never loads its first K/V stage
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
// key tiles 0 .. qt.  Eight compute warps: warp w serves tensor-memory lanes
// 32 (w % 4) .. +31 (one query row per thread) and key columns 64 (w / 4) ..
// +63 of each tile.  A step loads its S and dP rows with one wait, releases
// both at once (so the next pair is formed while this one is processed), and
// forms P and dS in one pass.  Tensor memory: S at 0, dP at 128 (fp32), dS in
// two buffers at 256 and 320 (binary16 pairs, so a step need not wait for the
// previous dQ product), dQ at 384 (fp32, 64 columns).  The unit's O tile comes
// with its Q and dO tiles, so the row term D is formed from shared memory.
namespace qlaunch {
constexpr int kStages = 4;                       // ring of {K tile, V^T tile}
constexpr uint32_t kStageBytes = 2 * kTileBytes;
constexpr uint32_t kOffQ = 0;                    // Q tile, dO tile, O tile
constexpr uint32_t kOffRing = 3 * kTileBytes;
constexpr uint32_t kOffBar = kOffRing + kStages * kStageBytes;
constexpr int kBarQFull = 0, kBarQEmpty = 1;
constexpr int kBarKvFull = 2, kBarKvEmpty = 2 + kStages;
constexpr int kBarSdFull = 2 + 2 * kStages, kBarSdFree = kBarSdFull + 1;
constexpr int kBarDsFull = kBarSdFree + 1, kBarDqDone = kBarDsFull + 2;   // two each
constexpr int kBarDrain = kBarDqDone + 2;        // + issuer warp (0, 1)
constexpr int kNumBars = kBarDrain + 2;
constexpr uint32_t kOffTmemPtr = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemPtr + 4;
constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;
constexpr uint32_t kColS = 0, kColDP = 128, kColDS = 256, kColDQ = 384;
constexpr int kComputeWarps = 8;
constexpr int kWarpSdp = 8, kWarpDq = 9, kWarpLoad = 10;
constexpr int kThreads = 32 * 11;

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
__device__ void load_role(const CUtensorMap *tmQ, const CUtensorMap *tmDO, const CUtensorMap *tmO,
                          const CUtensorMap *tmK, const CUtensorMap *tmVT, const BwdParams &p,
                          const Sync &sy, uint32_t smem) {
  const int units = p.heads * p.q_tiles;
  uint32_t pos = 0, pos_issued = 0, q_issued = 0;
  int k = 0;
  for (int u = unit_of(0, units); u >= 0; u = unit_of(++k, units)) {
    const Unit w = decode(u, p);
    if (!sy.wait(kBarQEmpty, (k & 1) ^ 1, 101)) goto drain;
    ++q_issued;
    mbar_arrive_expect_tx(sy.bar(kBarQFull), 3 * kTileBytes);
    tma_load_3d(smem + kOffQ, tmQ, sy.bar(kBarQFull), 0, w.qt * kTile, w.h);
    tma_load_3d(smem + kOffQ + kTileBytes, tmDO, sy.bar(kBarQFull), w.h * kD, w.qt * kTile, 0);
    tma_load_3d(smem + kOffQ + 2 * kTileBytes, tmO, sy.bar(kBarQFull), w.h * kD, w.qt * kTile, 0);
    for (int j = 0; j < w.nk; ++j, ++pos) {
      const uint32_t st = pos % kStages;
      if (!sy.wait(kBarKvEmpty + st, ((pos / kStages) & 1) ^ 1, 102)) goto drain;
      const uint32_t dst = smem + kOffRing + st * kStageBytes;
      const uint32_t full = sy.bar(kBarKvFull + st);
      mbar_arrive_expect_tx(full, kStageBytes);
      pos_issued = pos + 1;
      if (p.stall && blockIdx.x == 0 && pos == 0) continue;   // this stage never lands
      tma_load_3d(dst, tmK, full, 0, j * kTile, w.g);
      tma_load_3d(dst + kTileBytes, tmVT, full, j * kTile, 0, w.g);
      tma_load_3d(dst + kTileBytes + kHalfTileBytes, tmVT, full, j * kTile + kTile / 2, 0, w.g);
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

// S = Q K^T and dP = dO V^T for one key tile, once the compute warps have
// pulled the previous pair into registers; one commit for both.
__device__ void sdp_role(const BwdParams &p, const Sync &sy, uint32_t smem, uint32_t tmem) {
  constexpr uint32_t idS = idesc_f16_f32(kTile, kTile);
  constexpr uint32_t idDP = idesc_f16_f32_mn(kTile, kTile, false, true);
  const int units = p.heads * p.q_tiles;
  uint32_t pos = 0;
  int k = 0;
  for (int u = unit_of(0, units); u >= 0; u = unit_of(++k, units)) {
    const Unit w = decode(u, p);
    if (!sy.wait_warp(kBarQFull, k & 1, 111)) goto drain;
    tc_fence_after();
    for (int j = 0; j < w.nk; ++j, ++pos) {
      const uint32_t st = pos % kStages;
      if (!sy.wait2_warp(kBarKvFull + st, (pos / kStages) & 1, 112, kBarSdFree, (pos & 1) ^ 1, 113)) goto drain;
      tc_fence_after();
      const uint32_t kb = smem + kOffRing + st * kStageBytes;
#pragma unroll
      for (int e = 0; e < kD / 16; ++e)
        mma_ss(tmem + kColS, sw128_desc(smem + kOffQ + e * 32), sw128_desc(kb + e * 32), idS,
               e > 0 ? 1u : 0u);
#pragma unroll
      for (int e = 0; e < kD / 16; ++e)
        mma_ss(tmem + kColDP, sw128_desc(smem + kOffQ + kTileBytes + e * 32),
               sw128_mn_desc(kb + kTileBytes + e * 2048, kHalfTileBytes), idDP, e > 0 ? 1u : 0u);
      mma_commit(sy.bar(kBarSdFull));
      mma_commit(sy.bar(kBarKvEmpty + st));
    }
    mma_commit(sy.bar(kBarQEmpty));
  }
  return;
drain:
  mma_commit(sy.bar(kBarDrain + 0));
  sy.drain_wait(kBarDrain + 0, 0);
}

// dQ += dS K (A = dS from one of two tensor-memory buffers; B MN-major from the K tile).
__device__ void dq_role(const BwdParams &p, const Sync &sy, uint32_t smem, uint32_t tmem) {
  constexpr uint32_t id = idesc_f16_f32_mn(kTile, kD, false, true);
  const int units = p.heads * p.q_tiles;
  uint32_t pos = 0;
  int k = 0;
  for (int u = unit_of(0, units); u >= 0; u = unit_of(++k, units)) {
    const Unit w = decode(u, p);
    for (int j = 0; j < w.nk; ++j, ++pos) {
      const uint32_t st = pos % kStages, b = pos & 1;
      if (!sy.wait2_warp(kBarDsFull + b, (pos >> 1) & 1, 121, kBarKvFull + st, (pos / kStages) & 1, 122)) goto drain;
      tc_fence_after();
      const uint32_t kb = smem + kOffRing + st * kStageBytes;
#pragma unroll
      for (int e = 0; e < kTile / 16; ++e)
        mma_ts(tmem + kColDQ, tmem + kColDS + 64u * b + 8u * e,
               sw128_mn_desc(kb + e * 2048, kHalfTileBytes), id, (j > 0 || e > 0) ? 1u : 0u);
      mma_commit(sy.bar(kBarDqDone + b));
      mma_commit(sy.bar(kBarKvEmpty + st));
    }
  }
  return;
drain:
  mma_commit(sy.bar(kBarDrain + 1));
  sy.drain_wait(kBarDrain + 1, 0);
}

__device__ void compute_role(const BwdParams &p, const Sync &sy, const uint8_t *smem_gen,
                             uint32_t tmem) {
  const int warp = threadIdx.x >> 5;
  const int r = 32 * (warp & 3) + (threadIdx.x & 31);   // tile row (tensor-memory lane)
  const int half = warp >> 2;                            // key columns 64 half .. +63
  const int col0 = 64 * half;
  const bool leader = (threadIdx.x & 31) == 0;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
  const float c = p.c;
  const int units = p.heads * p.q_tiles;
  uint32_t pos = 0;
  int k = 0;
  for (int u = unit_of(0, units); u >= 0; u = unit_of(++k, units)) {
    const Unit w = decode(u, p);
    const int row = w.qt * kTile + r;
    const bool valid = row < p.T;
    // the row term D = rowsum(dO O), from the unit's dO and O tiles in shared memory
    // (128-byte swizzled rows: chunk i of row r at i ^ (r mod 8)), and the forward's L
    if (!sy.wait_warp(kBarQFull, k & 1, 135)) return;
    float L = 0.f, D = 0.f;
    if (valid) {
      const uint8_t *rdo = smem_gen + kOffQ + kTileBytes + r * 128;
      const uint8_t *ro = smem_gen + kOffQ + 2 * kTileBytes + r * 128;
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 a = *reinterpret_cast<const uint4 *>(rdo + ((i ^ (r & 7)) << 4));
        const uint4 b = *reinterpret_cast<const uint4 *>(ro + ((i ^ (r & 7)) << 4));
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
      if (half == 0) p.D[(size_t)w.h * p.T + row] = D;
    }
    // the Q buffer (with dO and O) may be refilled once the products and these reads are done
    __syncwarp();
    if (leader) mbar_arrive(sy.bar(kBarQEmpty));
    const float negL = -L;
    for (int j = 0; j < w.nk; ++j, ++pos) {
      const uint32_t b = pos & 1;
      if (!sy.wait_warp(kBarSdFull, pos & 1, 131)) return;
      tc_fence_after();
      uint32_t sr[64], dr[64];
      tmem_ld_2x64(tmem + lane_base + kColS + col0, tmem + lane_base + kColDP + col0, sr, dr);
      tc_fence_before();
      __syncwarp();
      if (leader) mbar_arrive(sy.bar(kBarSdFree));
      // P = 2^(S c - L) and dS = P (dP - D) in one pass, packed to binary16 pairs
      // (key columns col0 + 2m, +1 in pk[m]); on the diagonal tile keys after the
      // row get P = 0
      uint32_t pk[32];
      if (j == w.qt) {
        const int lim = r - col0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float x0, x1, g0, g1;
          fma2(x0, x1, __uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]), c, negL, negL);
          float p0 = ex2(x0), p1 = ex2(x1);
          if (2 * i > lim) p0 = 0.f;
          if (2 * i + 1 > lim) p1 = 0.f;
          mulsub2(g0, g1, p0, p1, __uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1]), D, D);
          pk[i] = pack_half2(g0, g1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float x0, x1, g0, g1;
          fma2(x0, x1, __uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]), c, negL, negL);
          const float p0 = ex2(x0), p1 = ex2(x1);
          mulsub2(g0, g1, p0, p1, __uint_as_float(dr[2 * i]), __uint_as_float(dr[2 * i + 1]), D, D);
          pk[i] = pack_half2(g0, g1);
        }
      }
      if (pos >= 2) {   // the product that read this dS buffer two steps ago must be complete
        if (!sy.wait_warp(kBarDqDone + b, ((pos >> 1) & 1) ^ 1, 133)) return;
        tc_fence_after();
      }
      tmem_st_x32(tmem + lane_base + kColDS + 64u * b + 32u * half, pk);
      tc_fence_before();
      __syncwarp();
      if (leader) mbar_arrive(sy.bar(kBarDsFull + b));
    }
    // epilogue: dQ = s (sum) once the last product is done; each half writes 32 columns
    if (!sy.wait_warp(kBarDqDone + ((pos - 1) & 1), ((pos - 1) >> 1) & 1, 134)) return;
    tc_fence_after();
    uint32_t qr[32];
    tmem_ld_x32(tmem + lane_base + kColDQ + 32u * half, qr);
    if (valid) {
      float4 *dst = reinterpret_cast<float4 *>(p.dq + ((size_t)w.h * p.T + row) * kD + 32 * half);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dst[i] = make_float4(__uint_as_float(qr[4 * i]) * p.s, __uint_as_float(qr[4 * i + 1]) * p.s,
                             __uint_as_float(qr[4 * i + 2]) * p.s, __uint_as_float(qr[4 * i + 3]) * p.s);
    }
    tc_fence_before();
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    query_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                 const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmVT, const BwdParams p) {
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
    mbar_init(sy.bar(kBarQEmpty), 1 + kComputeWarps);   // the S/dP issuer's commit, the row-term reads
    for (int i = 0; i < kStages; ++i) {
      mbar_init(sy.bar(kBarKvFull + i), 1);
      mbar_init(sy.bar(kBarKvEmpty + i), 2);   // S/dP issuer and dQ issuer
    }
    mbar_init(sy.bar(kBarSdFull), 1);
    mbar_init(sy.bar(kBarSdFree), kComputeWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(sy.bar(kBarDsFull + i), kComputeWarps);
      mbar_init(sy.bar(kBarDqDone + i), 1);
    }
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
  if (warp < kComputeWarps) {
    compute_role(p, sy, smem_gen, tmem);
  } else if (warp == kWarpSdp) {
    sdp_role(p, sy, smem, tmem);
  } else if (warp == kWarpDq) {
    dq_role(p, sy, smem, tmem);
  } else if (warp == kWarpLoad) {
    if (lane == 0) load_role(&tmQ, &tmDO, &tmO, &tmK, &tmVT, p, sy, smem);
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
// Eight compute warps: warp w serves lanes 32 (w % 4) .. +31 (one key per
// thread) and query columns 64 (w / 4) .. +63; as in the query launch, S^T
// and dP^T arrive and are released together, while P^T and dS^T go to the
// dV and dK products one column half at a time.  Tensor memory: S^T at 0,
// dP^T at 128 (fp32), P^T at 256, dS^T at 320 (binary16 pairs), dV at 384,
// dK at 448 (fp32).
namespace klaunch {
constexpr int kStages = 5;   // ring of {Q tile, dO tile, L, D}
constexpr uint32_t kStageBytes = 2 * kTileBytes + 1024;   // L and D: 512 bytes each
constexpr uint32_t kOffK = 0;                              // K tile, V^T tile
constexpr uint32_t kOffRing = 2 * kTileBytes;
constexpr uint32_t kOffBar = kOffRing + kStages * kStageBytes;
constexpr int kBarKvFull = 0, kBarKvEmpty = 1;
constexpr int kBarQFull = 2, kBarQEmpty = 2 + kStages;
constexpr int kBarSFull = 2 + 2 * kStages, kBarSFree = kBarSFull + 1;   // S^T and dP^T together
// per query-column half h: P^T, dS^T written (PFull + h), dV and dK products of it done (Done + h)
constexpr int kBarPFull = kBarSFree + 1, kBarDone = kBarPFull + 2;
constexpr int kBarDrain = kBarDone + 2;          // + issuer warp (0..2)
constexpr int kNumBars = kBarDrain + 3;
constexpr uint32_t kOffTmemPtr = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemPtr + 4;
constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;
constexpr uint32_t kColS = 0, kColDP = 128, kColP = 256, kColDS = 320, kColDV = 384, kColDK = 448;
constexpr int kComputeWarps = 8;
constexpr int kWarpSdp = 8, kWarpDv = 9, kWarpDk = 10, kWarpLoad = 11;
constexpr int kThreads = 32 * 12;
// offsets inside a stage
constexpr uint32_t kSQ = 0, kSDO = kTileBytes, kSL = 2 * kTileBytes, kSDd = kSL + kTile * 4;

struct Unit {
  int g, kt, nq;    // query tiles kt .. kt + nq - 1 for each of the group's heads
  int split;        // which share of the (K/V head, key tile) pair's steps
  int first, steps; // this unit's steps: first .. first + steps - 1 of the pair's
};
__device__ __forceinline__ int key_units(const BwdParams &p) {
  return p.kv_heads * p.q_tiles * p.splits;
}
__device__ __forceinline__ Unit decode(int u, const BwdParams &p) {
  Unit w;
  const int per_tile = p.kv_heads * p.splits;
  const int r = u / per_tile;
  const int rem = u - r * per_tile;
  w.g = rem / p.splits;
  w.split = rem - w.g * p.splits;
  w.kt = r;                      // earliest key tiles see the most query tiles
  w.nq = p.q_tiles - w.kt;
  const int total = p.group * w.nq;
  w.first = (int)((long long)total * w.split / p.splits);
  w.steps = (int)((long long)total * (w.split + 1) / p.splits) - w.first;
  return w;
}
// step i of a unit: query head and query tile
__device__ __forceinline__ void step_of(const Unit &w, int i, const BwdParams &p, int &h, int &qt) {
  const int j = w.first + i;
  const int z = j / w.nq;
  h = w.g * p.group + z;
  qt = w.kt + (j - z * w.nq);
}

__device__ void load_role(const CUtensorMap *tmK, const CUtensorMap *tmVT, const CUtensorMap *tmQ,
                          const CUtensorMap *tmDO, const BwdParams &p, const Sync &sy,
                          uint32_t smem) {
  const int units = key_units(p);
  uint32_t pos = 0, pos_issued = 0, kv_issued = 0;
  int k = 0;
  for (int u = unit_of(0, units); u >= 0; u = unit_of(++k, units)) {
    const Unit w = decode(u, p);
    if (!sy.wait(kBarKvEmpty, (k & 1) ^ 1, 201)) goto drain;
    ++kv_issued;
    mbar_arrive_expect_tx(sy.bar(kBarKvFull), 2 * kTileBytes);
    tma_load_3d(smem + kOffK, tmK, sy.bar(kBarKvFull), 0, w.kt * kTile, w.g);
    tma_load_3d(smem + kOffK + kTileBytes, tmVT, sy.bar(kBarKvFull), w.kt * kTile, 0, w.g);
    tma_load_3d(smem + kOffK + kTileBytes + kHalfTileBytes, tmVT, sy.bar(kBarKvFull),
                w.kt * kTile + kTile / 2, 0, w.g);
    for (int i = 0; i < w.steps; ++i, ++pos) {
      int h, qt;
      step_of(w, i, p, h, qt);
      const uint32_t st = pos % kStages;
      if (!sy.wait(kBarQEmpty + st, ((pos / kStages) & 1) ^ 1, 202)) goto drain;
      const uint32_t dst = smem + kOffRing + st * kStageBytes;
      const uint32_t full = sy.bar(kBarQFull + st);
      const int rows = min(kTile, p.T - qt * kTile);      // query rows that exist (64 or 128)
      mbar_arrive_expect_tx(full, 2 * kTileBytes + 2 * rows * 4);
      pos_issued = pos + 1;
      tma_load_3d(dst + kSQ, tmQ, full, 0, qt * kTile, h);
      tma_load_3d(dst + kSDO, tmDO, full, h * kD, qt * kTile, 0);
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

// S^T = K Q^T (both K-major) and dP^T = V dO^T (A read MN-major from the V^T tile).
__device__ void sdp_role(const BwdParams &p, const Sync &sy, uint32_t smem, uint32_t tmem) {
  constexpr uint32_t idS = idesc_f16_f32(kTile, kTile);
  constexpr uint32_t idDP = idesc_f16_f32_mn(kTile, kTile, true, false);
  const int units = key_units(p);
  uint32_t pos = 0;
  int k = 0;
  for (int u = unit_of(0, units); u >= 0; u = unit_of(++k, units)) {
    const Unit w = decode(u, p);
    if (!sy.wait_warp(kBarKvFull, k & 1, 211)) goto drain;
    tc_fence_after();
    for (int i = 0; i < w.steps; ++i, ++pos) {
      const uint32_t st = pos % kStages;
      if (!sy.wait2_warp(kBarQFull + st, (pos / kStages) & 1, 212, kBarSFree, (pos & 1) ^ 1, 213)) goto drain;
      tc_fence_after();
      const uint32_t sb = smem + kOffRing + st * kStageBytes;
#pragma unroll
      for (int e = 0; e < kD / 16; ++e)
        mma_ss(tmem + kColS, sw128_desc(smem + kOffK + e * 32), sw128_desc(sb + kSQ + e * 32), idS,
               e > 0 ? 1u : 0u);
#pragma unroll
      for (int e = 0; e < kD / 16; ++e)
        mma_ss(tmem + kColDP, sw128_mn_desc(smem + kOffK + kTileBytes + e * 2048, kHalfTileBytes),
               sw128_desc(sb + kSDO + e * 32), idDP, e > 0 ? 1u : 0u);
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

// dV += P^T dO (B = dO tile) when which == 0, dK += dS^T Q (B = Q tile) when
// which == 1; B is read MN-major from the tile.  The products run over the step's
// two halves of query columns (K = 64 each), each as soon as the compute warps of
// that half have written it, and each half's completion is signalled on its own
// barrier: a half's next P^T, dS^T wait only for the products that read its own.
__device__ void acc_role(int which, const BwdParams &p, const Sync &sy, uint32_t smem,
                         uint32_t tmem) {
  constexpr uint32_t id = idesc_f16_f32_mn(kTile, kD, false, true);
  const int units = key_units(p);
  const uint32_t a_col = which ? kColDS : kColP;
  const uint32_t d_col = which ? kColDK : kColDV;
  const uint32_t b_off = which ? kSQ : kSDO;
  uint32_t pos = 0;
  int k = 0;
  for (int u = unit_of(0, units); u >= 0; u = unit_of(++k, units)) {
    const Unit w = decode(u, p);
    for (int i = 0; i < w.steps; ++i, ++pos) {
      const uint32_t st = pos % kStages;
      const uint32_t bb = smem + kOffRing + st * kStageBytes + b_off;
      // each half of the query columns as soon as its P^T, dS^T are written
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        if (hh == 0) {
          if (!sy.wait2_warp(kBarPFull, pos & 1, 221 + which, kBarQFull + st, (pos / kStages) & 1, 223 + which)) goto drain;
        } else if (!sy.wait_warp(kBarPFull + 1, pos & 1, 225 + which)) {
          goto drain;
        }
        tc_fence_after();
#pragma unroll
        for (int e = 4 * hh; e < 4 * hh + 4; ++e)
          mma_ts(tmem + d_col, tmem + a_col + 8u * e, sw128_mn_desc(bb + e * 2048, kHalfTileBytes),
                 id, (i > 0 || e > 0) ? 1u : 0u);
        mma_commit(sy.bar(kBarDone + hh));
      }
      mma_commit(sy.bar(kBarQEmpty + st));
    }
  }
  return;
drain:
  mma_commit(sy.bar(kBarDrain + 1 + which));
  sy.drain_wait(kBarDrain + 1 + which, 0);
}

// One key row's step over the thread's 64 query columns: P^T = 2^(S^T c - L)
// and dS^T = P^T (dP^T - D), packed to binary16 pairs (query columns 2m,
// 2m+1 in [m]).  With kMasked, column t is kept only when lo <= t < hi.
// Three passes (the exponents, then the 64 exp2 back to back, then dS^T and
// the packing) keep the SFU fed while the other pipes work on the neighbours.
template <bool kMasked>
__device__ __forceinline__ void key_step(const uint32_t (&sr)[64], const uint32_t (&dr)[64],
                                         const float *Ls, const float *Ds, float c, int lo, int hi,
                                         uint32_t (&pp)[32], uint32_t (&pd)[32]) {
  float pf[64];
#pragma unroll
  for (int t4 = 0; t4 < 16; ++t4) {
    const float4 L4 = *reinterpret_cast<const float4 *>(Ls + 4 * t4);
    fma2(pf[4 * t4], pf[4 * t4 + 1], __uint_as_float(sr[4 * t4]), __uint_as_float(sr[4 * t4 + 1]), c, -L4.x, -L4.y);
    fma2(pf[4 * t4 + 2], pf[4 * t4 + 3], __uint_as_float(sr[4 * t4 + 2]), __uint_as_float(sr[4 * t4 + 3]), c, -L4.z, -L4.w);
  }
#pragma unroll
  for (int t = 0; t < 64; ++t) pf[t] = ex2(pf[t]);
#pragma unroll
  for (int t4 = 0; t4 < 16; ++t4) {
    const float4 D4 = *reinterpret_cast<const float4 *>(Ds + 4 * t4);
    const float Dv[4] = {D4.x, D4.y, D4.z, D4.w};
    float pv[4], dv[4];
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      const int t = 4 * t4 + e;
      float g0, g1;
      mulsub2(g0, g1, pf[t], pf[t + 1], __uint_as_float(dr[t]), __uint_as_float(dr[t + 1]), Dv[e], Dv[e + 1]);
      const bool live0 = !kMasked || (t >= lo && t < hi);
      const bool live1 = !kMasked || (t + 1 >= lo && t + 1 < hi);
      pv[e] = live0 ? pf[t] : 0.f;
      dv[e] = live0 ? g0 : 0.f;
      pv[e + 1] = live1 ? pf[t + 1] : 0.f;
      dv[e + 1] = live1 ? g1 : 0.f;
    }
    pp[2 * t4] = pack_half2(pv[0], pv[1]);
    pp[2 * t4 + 1] = pack_half2(pv[2], pv[3]);
    pd[2 * t4] = pack_half2(dv[0], dv[1]);
    pd[2 * t4 + 1] = pack_half2(dv[2], dv[3]);
  }
}

__device__ void compute_role(const BwdParams &p, const Sync &sy, const uint8_t *smem_gen,
                             uint32_t tmem) {
  const int warp = threadIdx.x >> 5;
  const int r = 32 * (warp & 3) + (threadIdx.x & 31);   // key row of the tile (lane)
  const int half = warp >> 2;                            // query columns 64 half .. +63
  const int col0 = 64 * half;
  const bool leader = (threadIdx.x & 31) == 0;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
  const float c = p.c;
  const int units = key_units(p);
  uint32_t pos = 0;
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
      if (!sy.wait2_warp(kBarQFull + st, (pos / kStages) & 1, 230, kBarSFull, pos & 1, 231)) return;
      tc_fence_after();
      uint32_t sr[64], dr[64];
      tmem_ld_2x64(tmem + lane_base + kColS + col0, tmem + lane_base + kColDP + col0, sr, dr);
      tc_fence_before();
      __syncwarp();
      if (leader) mbar_arrive(sy.bar(kBarSFree));
      const float *Ls =
          reinterpret_cast<const float *>(smem_gen + kOffRing + st * kStageBytes + kSL) + col0;
      const float *Ds =
          reinterpret_cast<const float *>(smem_gen + kOffRing + st * kStageBytes + kSDd) + col0;
      // column t is query qt*128 + col0 + t: it sees this key when it is not earlier,
      // and exists when it is before the sequence end; only the diagonal tile and a
      // ragged last tile need the test
      const bool masked = qt == w.kt || qt * kTile + kTile > p.T;
      const int lo = key - (qt * kTile + col0);
      const int hi = min(kTile, p.T - qt * kTile) - col0;
      uint32_t pp[32], pd[32];
      if (masked)
        key_step<true>(sr, dr, Ls, Ds, c, lo, hi, pp, pd);
      else
        key_step<false>(sr, dr, Ls, Ds, c, lo, hi, pp, pd);
      if (i > 0) {   // the previous step's products of this half must be done before its P^T, dS^T are overwritten
        if (!sy.wait_warp(kBarDone + half, (pos - 1) & 1, 233)) return;
        tc_fence_after();
      }
      tmem_st_2x32(tmem + lane_base + kColP + 32u * half, tmem + lane_base + kColDS + 32u * half, pp, pd);
      tc_fence_before();
      __syncwarp();
      if (leader) mbar_arrive(sy.bar(kBarPFull + half));
    }
    // epilogue: the first half writes dV^T, the second s dK, for this key row (into
    // the unit's partial planes when the pair's steps are shared out; a share with
    // no steps writes zeros)
    uint32_t ar[64];
    if (w.steps > 0) {
      if (!sy.wait2_warp(kBarDone, (pos - 1) & 1, 235, kBarDone + 1, (pos - 1) & 1, 236)) return;
      tc_fence_after();
      tmem_ld_x64(tmem + lane_base + (half ? kColDK : kColDV), ar);
    } else {
#pragma unroll
      for (int e = 0; e < kD; ++e) ar[e] = 0u;
    }
    if (key < p.T) {
      const size_t plane = (size_t)p.kv_heads * p.T * kD;
      float *dv_base = p.splits > 1 ? p.dv_part + plane * w.split : p.dvT;
      float *dk_base = p.splits > 1 ? p.dk_part + plane * w.split : p.dk;
      if (half == 0) {
        float *dvt = dv_base + (size_t)w.g * kD * p.T + key;
#pragma unroll
        for (int e = 0; e < kD; ++e) dvt[(size_t)e * p.T] = __uint_as_float(ar[e]);
      } else {
        float4 *dk = reinterpret_cast<float4 *>(dk_base + ((size_t)w.g * p.T + key) * kD);
#pragma unroll
        for (int e = 0; e < 16; ++e)
          dk[e] = make_float4(__uint_as_float(ar[4 * e]) * p.s, __uint_as_float(ar[4 * e + 1]) * p.s,
                              __uint_as_float(ar[4 * e + 2]) * p.s, __uint_as_float(ar[4 * e + 3]) * p.s);
      }
    }
    tc_fence_before();
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    key_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmVT,
               const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
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
    mbar_init(sy.bar(kBarSFree), kComputeWarps);
    for (int h = 0; h < 2; ++h) {
      mbar_init(sy.bar(kBarPFull + h), kComputeWarps / 2);
      mbar_init(sy.bar(kBarDone + h), 2);   // the dV and the dK issuer
    }
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
  if (warp < kComputeWarps) {
    compute_role(p, sy, smem_gen, tmem);
  } else if (warp == kWarpSdp) {
    sdp_role(p, sy, smem, tmem);
  } else if (warp == kWarpDv || warp == kWarpDk) {
    acc_role(warp - kWarpDv, p, sy, smem, tmem);
  } else if (warp == kWarpLoad) {
    if (lane == 0) load_role(&tmK, &tmVT, &tmQ, &tmDO, p, sy, smem);
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

// The sum over the key launch's partial planes (short problems only): out[x] =
// sum over i of part[i n + x], in order i = 0, 1, ... (deterministic), for dK and
// dV^T at once.  n is a multiple of 4 (whole 64-wide rows).
__global__ void __launch_bounds__(256) reduce_splits_kernel(const float *dk_part, const float *dv_part,
                                                            float *dk, float *dvT, size_t n,
                                                            int splits) {
  const size_t n4 = n / 4;
  for (size_t x = (size_t)blockIdx.x * blockDim.x + threadIdx.x; x < 2 * n4;
       x += (size_t)gridDim.x * blockDim.x) {
    const bool second = x >= n4;
    const size_t y = second ? x - n4 : x;
    const float4 *src = reinterpret_cast<const float4 *>(second ? dv_part : dk_part) + y;
    float4 acc = src[0];
    for (int i = 1; i < splits; ++i) {
      const float4 v = src[(size_t)i * n4];
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    reinterpret_cast<float4 *>(second ? dvT : dk)[y] = acc;
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
std::atomic<int> g_bwd_stall{0};   // test hook: the next attn_bwd call stalls one CTA
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

// Short problems share each (K/V head, key tile) pair's steps out over several
// key-launch units.  With fewer than 128 units, the key launch's longest unit --
// a whole group of query heads over every later query tile, group * q_tiles
// steps -- bounds the call; the query launch's longest is q_tiles steps.  So a
// group of two or more heads whose chain is at least 16 steps gets
// S = min(group, ceil(256 / units), 8) shares (at least one step each), and a
// reduce launch adds them.  A function of the shape alone, so the workspace
// size is too.
int key_splits(int T, int heads, int kv_heads) {
  const int q_tiles = (T + kTile - 1) / kTile;
  const int group = heads / kv_heads;
  const long long units = (long long)kv_heads * q_tiles;
  if (units >= 128 || group < 2 || (long long)group * q_tiles < 16) return 1;
  long long s = (256 + units - 1) / units;
  if (s > group) s = group;
  return (int)(s < 8 ? s : 8);
}

// Workspace: the row terms D (binary32 [heads][T]) the query launch writes
// for the key launch; with split key units, their partial dK and dV^T planes.
size_t bwd_workspace(int T, int heads, int kv_heads) {
  const int sp = key_splits(T, heads, kv_heads);
  const size_t plane = (size_t)kv_heads * T * kD * 4;
  return up256((size_t)heads * T * 4) + (sp > 1 ? 2 * up256(plane * sp) : 0);
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
  return bwd_workspace(T, heads, kv_heads);
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
  const size_t ws_bytes = bwd_workspace(T, heads, kv_heads);
  if (workspace_bytes < ws_bytes) return ATTN_EINVAL;
  const size_t hq = (size_t)heads * T * kD, kvn = (size_t)kv_heads * T * kD;
  const size_t in_sizes[] = {hq * 2, kvn * 2, kvn * 2, hq * 2, (size_t)heads * T * 4, hq * 2};
  const size_t out_sizes[] = {hq * 4, kvn * 4, kvn * 4, ws_bytes};
  for (int a = 0; a < 4; ++a) {
    for (int b = 0; b < 6; ++b)
      if (ranges_overlap(outs[a], out_sizes[a], ins[b], in_sizes[b])) return ATTN_EOVERLAP;
    for (int b = a + 1; b < 4; ++b)
      if (ranges_overlap(outs[a], out_sizes[a], outs[b], out_sizes[b])) return ATTN_EOVERLAP;
  }
  BwdState *st = nullptr;
  if ((rc = bwd_state(&st))) return rc;

  const uint64_t rowb = kD * 2, trow = (uint64_t)T * 2;
  CUtensorMap tmQ, tmK, tmVT, tmDO, tmO;
  if (!encode_3d(&tmQ, q, kD, T, heads, rowb, rowb * T, kD, kTile) ||
      !encode_3d(&tmK, k, kD, T, kv_heads, rowb, rowb * T, kD, kTile) ||
      !encode_3d(&tmVT, vT, T, kD, kv_heads, trow, trow * kD, kTile / 2, kD) ||
      !encode_3d(&tmDO, dO, (uint64_t)heads * kD, T, 1, (uint64_t)heads * kD * 2,
                 (uint64_t)heads * kD * 2 * T, kD, kTile) ||
      !encode_3d(&tmO, o, (uint64_t)heads * kD, T, 1, (uint64_t)heads * kD * 2,
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
  p.D = static_cast<float *>(workspace);
  p.dq = dq;
  p.dk = dk;
  p.dvT = dvT;
  p.splits = key_splits(T, heads, kv_heads);
  {
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t plane = (size_t)kv_heads * T * kD * 4;
    p.dk_part = reinterpret_cast<float *>(ws + up256((size_t)heads * T * 4));
    p.dv_part = reinterpret_cast<float *>(ws + up256((size_t)heads * T * 4) + up256(plane * p.splits));
  }
  p.status = st->status;
  p.stall = g_bwd_stall.exchange(0);
  const int qunits = heads * p.q_tiles, kunits = kv_heads * p.q_tiles * p.splits;
  qlaunch::query_kernel<<<qunits < st->sms ? qunits : st->sms, qlaunch::kThreads,
                          qlaunch::kSmemBytes, stream>>>(tmQ, tmDO, tmO, tmK, tmVT, p);
  klaunch::key_kernel<<<kunits < st->sms ? kunits : st->sms, klaunch::kThreads,
                        klaunch::kSmemBytes, stream>>>(tmK, tmVT, tmQ, tmDO, p);
  if (p.splits > 1) {
    const size_t n = (size_t)kv_heads * T * kD;
    const size_t blocks = (2 * n / 4 + 255) / 256;
    reduce_splits_kernel<<<(unsigned)(blocks < 4u * (size_t)st->sms ? blocks : 4u * (size_t)st->sms),
                           256, 0, stream>>>(p.dk_part, p.dv_part, dk, dvT, n, p.splits);
  }
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

extern "C" int attn_bwd_test_inject_stall(void) {
  g_bwd_stall.store(1);
  return ATTN_OK;
}
