// attn_materialised.cu -- the materialised causal grouped-query attention
// forward for GB300 (sm_103a), behind attn_materialised.h.
//
// The prior design that the page "Realization/Nvidia/SM86/StreamingAttentionSM86.alpha"
// replaces, laid out as the page ".../Coppelius/Build/Graph.alpha" lays out its
// attention planes (a binary32 scores plane of heads x T x T, a "softmax-forward"
// launch writing binary16 probabilities, then their product with V).  Three
// launches:
//   scores_kernel   S = Q K^T per (head, query tile, key tile <= diagonal): TMA
//                   loads, four tcgen05 MMAs into tensor memory, the binary32
//                   tile staged in shared memory and written by TMA stores;
//   softmax_kernel  one warp per row: t = S c, an online row maximum and sum in
//                   one pass, then normalised binary16 probabilities and the
//                   base-2 LSE;
//   pv_kernel       O = P V per (head, query tile): a two-stage TMA ring of P and
//                   V^T tiles, tcgen05 MMAs, binary16 O token-major.
// Every wait is bounded (1 s); a timeout is recorded in a status word.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <atomic>
#include <mutex>

#include "attn_materialised.h"
#include "sm103_ptx.cuh"

namespace {

using namespace sm103;

constexpr int kD = 64;
constexpr int kTile = 128;
constexpr uint32_t kTileBytes = kTile * kD * 2;   // 16 KiB
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kMaxT = 16384;                      // admission: the planes grow as T^2

struct MatParams {
  int T, heads, kv_heads, group, q_tiles;
  float c;
  float *S;        // [H][T][T] binary32
  __half *P;       // [H][T][T] binary16
  __half *o;       // [T][H*64]
  float *lse;      // [H][T]
  int *status;
  int stall;       // test hook: the scores kernel's first block never loads its K tile
};

// Bounded wait on an mbarrier phase; records `where` in the status word on expiry.
__device__ bool wait_bounded(uint32_t bar, uint32_t parity, int *status, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(status, 0, where);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------- scores
// Block (kt, qt) of head h: grid.x enumerates the causal tiles (qt, kt <= qt).
// Shared memory: the Q and K tiles, then -- over them, once the MMAs that read
// them are complete -- the binary32 result staged as four 32-column boxes of
// 128 rows (128-byte swizzle) for the TMA store.  64 KiB per CTA lets three
// CTAs share an SM (3 x 128 tensor-memory columns), so one CTA's store overlaps
// another's loads and products.
constexpr uint32_t kStageOff = 0;
constexpr uint32_t kBoxBytes = kTile * 32 * 4;       // 16 KiB
constexpr uint32_t kScoresBarOff = kStageOff + 4 * kBoxBytes;
constexpr uint32_t kScoresSmem = kScoresBarOff + 64 + 1024;

__global__ void __launch_bounds__(128) scores_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                     const __grid_constant__ CUtensorMap tmK,
                                                     const __grid_constant__ CUtensorMap tmS,
                                                     const MatParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t smem = (raw + 1023u) & ~1023u;
  uint8_t *smem_gen = smem_raw + (smem - raw);
  const uint32_t bar_full = smem + kScoresBarOff, bar_done = bar_full + 8;
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem_gen + kScoresBarOff + 16);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_gen + kScoresBarOff + 20);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int rem = blockIdx.x;
  int qt = (int)((sqrtf(8.f * (float)rem + 1.f) - 1.f) * 0.5f);
  while ((qt + 1) * (qt + 2) / 2 <= rem) ++qt;
  while (qt * (qt + 1) / 2 > rem) --qt;
  const int kt = rem - qt * (qt + 1) / 2;
  const int g = h / p.group;

  if (threadIdx.x == 0) {
    mbar_init(bar_full, 1);
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    mbar_fence_init();
    mbar_arrive_expect_tx(bar_full, 2 * kTileBytes);
    tma_load_3d(smem, &tmQ, bar_full, 0, qt * kTile, h);
    if (!(p.stall && blockIdx.x == 0 && blockIdx.y == 0))   // test hook: this K tile never lands
      tma_load_3d(smem + kTileBytes, &tmK, bar_full, 0, kt * kTile, g);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 1) {
    const bool ok = __all_sync(0xffffffffu, wait_bounded(bar_full, 0, p.status, 301));
    if (ok) {
      tc_fence_after();
      constexpr uint32_t id = idesc_f16_f32(kTile, kTile);
#pragma unroll
      for (int e = 0; e < kD / 16; ++e)
        mma_ss(tmem, sw128_desc(smem + e * 32), sw128_desc(smem + kTileBytes + e * 32), id,
               e > 0 ? 1u : 0u);
    } else if (lane == 0) {
      *abort_flag = 1;
    }
    mma_commit(bar_done);
  }
  const bool ok = __all_sync(0xffffffffu, wait_bounded(bar_done, 0, p.status, 302));
  if (!ok && lane == 0) *abort_flag = 1;
  tc_fence_after();
  uint32_t sr[128];
  tmem_ld_x128(tmem + ((uint32_t)(32 * warp) << 16), sr);
  // row r's 32-column slice b goes to box b, row r: its eight 16-byte chunks
  // permuted by the 128-byte swizzle (chunk c at c ^ (r mod 8))
  const int r = 32 * warp + lane;
#pragma unroll
  for (int b = 0; b < 4; ++b)
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      const uint32_t addr = smem + kStageOff + b * kBoxBytes + r * 128 + ((cc ^ (r & 7)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                   "r"(sr[32 * b + 4 * cc]), "r"(sr[32 * b + 4 * cc + 1]),
                   "r"(sr[32 * b + 4 * cc + 2]), "r"(sr[32 * b + 4 * cc + 3])
                   : "memory");
    }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!*abort_flag) {
      // rows past T are clipped by the copy; a 64-key last tile stores two boxes
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if (kt * kTile + 32 * b < p.T)
          tma_store_3d(&tmS, smem + kStageOff + b * kBoxBytes, kt * kTile + 32 * b, qt * kTile, h);
      tma_store_commit_wait();
    } else {
      // let a copy that is still in flight land before the shared memory is released
      // (the values staged over it are discarded)
      wait_bounded(bar_full, 0, p.status, 303);
    }
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// ---------------------------------------------------------------------------- softmax
// One warp per (row i, head h), eight rows per CTA.  Pass 1 streams the row's
// causal scores once (a float4 per lane per step), keeping per lane a running
// maximum m of t = S c and a sum l = sum 2^(t - m) rescaled whenever m rises;
// the lanes' pairs are then merged.  Pass 2 reads the scores again and writes
// the normalised binary16 probabilities, zero-filled to the end of the
// diagonal tile.  The rows in flight (up to 32 KiB each) outgrow L2 at large T,
// so pass 2 walks the row backwards (its end, read last, is the likeliest to
// be in L2) and marks its loads and the probability stores evict-first: a
// score is not read a third time, and those lines give way to the rows still
// waiting for their second read.  (Holding the row in registers instead, over
// four warps, measured slower: it halves the rows in flight per SM.)
__device__ __forceinline__ float rescale(float m_old, float m_new) {
  return m_old == -INFINITY ? 0.f : ex2(m_old - m_new);
}

// 16-byte load and 8-byte store with an L2 eviction policy from createpolicy.
__device__ __forceinline__ float4 ld_policy(const float *ptr, uint64_t pol) {
  float4 v;
  asm("ld.global.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
      : "l"(ptr), "l"(pol));
  return v;
}
__device__ __forceinline__ void st_policy(void *ptr, uint2 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.b32 [%0], {%1, %2}, %3;" ::"l"(ptr), "r"(v.x), "r"(v.y),
               "l"(pol)
               : "memory");
}

__global__ void __launch_bounds__(256) softmax_kernel(const MatParams p) {
  uint64_t evict_first;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(evict_first));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * 8 + warp, h = blockIdx.y;
  if (i >= p.T) return;
  const float *srow = p.S + ((size_t)h * p.T + i) * p.T;
  __half *prow = p.P + ((size_t)h * p.T + i) * p.T;
  const int n = i + 1;                                   // keys 0 .. i
  const int end = min(p.T, (i / kTile + 1) * kTile);     // the diagonal tile's end
  const float c = p.c;
  float m = -INFINITY, l = 0.f;
#pragma unroll 4
  for (int j0 = 4 * lane; j0 < n; j0 += 128) {
    const float4 a = *reinterpret_cast<const float4 *>(srow + j0);
    float t[4] = {a.x * c, a.y * c, a.z * c, a.w * c};
#pragma unroll
    for (int e = 1; e < 4; ++e)
      if (j0 + e >= n) t[e] = -INFINITY;
    const float m_new = fmaxf(m, fmaxf(fmaxf(t[0], t[1]), fmaxf(t[2], t[3])));
    l = l * rescale(m, m_new) + ((ex2(t[0] - m_new) + ex2(t[1] - m_new)) +
                                 (ex2(t[2] - m_new) + ex2(t[3] - m_new)));
    m = m_new;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
    const float m_new = fmaxf(m, m2);
    l = l * rescale(m, m_new) + l2 * rescale(m2, m_new);
    m = m_new;
  }
  const float inv = 1.f / l;
  if (lane == 0) p.lse[(size_t)h * p.T + i] = m + log2f(l);
  const int nsteps = (end + 127) / 128;
#pragma unroll 4
  for (int st = nsteps - 1; st >= 0; --st) {
    const int j0 = 128 * st + 4 * lane;
    if (j0 >= end) continue;
    float q[4] = {0.f, 0.f, 0.f, 0.f};
    if (j0 < n) {
      const float4 a = ld_policy(srow + j0, evict_first);
      const float t[4] = {a.x * c, a.y * c, a.z * c, a.w * c};
#pragma unroll
      for (int e = 0; e < 4; ++e) q[e] = j0 + e < n ? ex2(t[e] - m) * inv : 0.f;
    }
    __half2 lo = __floats2half2_rn(q[0], q[1]), hi = __floats2half2_rn(q[2], q[3]);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t *>(&lo);
    v.y = *reinterpret_cast<uint32_t *>(&hi);
    st_policy(prow + j0, v, evict_first);
  }
}

// ---------------------------------------------------------------------------- P V
// One CTA of 128 threads per (query tile qt, head h); key tiles 0 .. qt through
// a two-stage ring of {P tile (two 64-key boxes), V^T tile (two 64-key boxes)}.
constexpr uint32_t kPvStage = 2 * kTileBytes + kTileBytes;   // 48 KiB
constexpr uint32_t kPvSmem = 2 * kPvStage + 64 + 1024;

__global__ void __launch_bounds__(128) pv_kernel(const __grid_constant__ CUtensorMap tmP,
                                                 const __grid_constant__ CUtensorMap tmVT,
                                                 const MatParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t smem = (raw + 1023u) & ~1023u;
  uint8_t *smem_gen = smem_raw + (smem - raw);
  const uint32_t bars = smem + 2 * kPvStage;   // full[2], empty[2], done
  volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem_gen + 2 * kPvStage + 40);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_gen + 2 * kPvStage + 44);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y, g = h / p.group;
  const int nk = qt + 1;
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 16u + 8u * s; };
  const uint32_t done = bars + 32u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(const_cast<uint32_t *>(tmem_slot)), 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {   // producer
      int issued = 0;
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt & 1;
        if (kt >= 2 && !wait_bounded(empty(s), ((kt >> 1) - 1) & 1, p.status, 311)) {
          *abort_flag = 1;
          break;
        }
        const uint32_t dst = smem + s * kPvStage;
        mbar_arrive_expect_tx(full(s), kPvStage);
        tma_load_3d(dst, &tmP, full(s), kt * kTile, qt * kTile, h);
        tma_load_3d(dst + kTileBytes, &tmP, full(s), kt * kTile + 64, qt * kTile, h);
        tma_load_3d(dst + 2 * kTileBytes, &tmVT, full(s), kt * kTile, 0, g);
        tma_load_3d(dst + 2 * kTileBytes + kTileBytes / 2, &tmVT, full(s), kt * kTile + 64, 0, g);
        issued = kt + 1;
      }
      // on an early stop, let the copies in flight land before the CTA exits
      if (*abort_flag)
        for (int kt = issued - 2 < 0 ? 0 : issued - 2; kt < issued; ++kt)
          wait_bounded(full(kt & 1), (kt >> 1) & 1, p.status, 312);
    }
    __syncwarp();
  } else if (warp == 1) {   // MMA issuer
    constexpr uint32_t id = idesc_f16_f32(kTile, kD);
    bool ok = true;
    for (int kt = 0; kt < nk && ok; ++kt) {
      const int s = kt & 1;
      ok = __all_sync(0xffffffffu, wait_bounded(full(s), (kt >> 1) & 1, p.status, 313));
      if (!ok) break;
      tc_fence_after();
      const uint32_t base = smem + s * kPvStage;
#pragma unroll
      for (int e = 0; e < kTile / 16; ++e)
        mma_ss(tmem, sw128_desc(base + (e >> 2) * kTileBytes + (e & 3) * 32),
               sw128_desc(base + 2 * kTileBytes + (e >> 2) * (kTileBytes / 2) + (e & 3) * 32), id,
               (kt > 0 || e > 0) ? 1u : 0u);
      mma_commit(empty(s));
    }
    if (!ok && lane == 0) *abort_flag = 1;
    mma_commit(done);
  }
  const bool ok = __all_sync(0xffffffffu, wait_bounded(done, 0, p.status, 314));
  if (!ok && lane == 0) *abort_flag = 1;
  tc_fence_after();
  uint32_t orow[64];
  tmem_ld_x64(tmem + ((uint32_t)(32 * warp) << 16), orow);
  tc_fence_before();
  __syncthreads();
  if (!*abort_flag) {
    const int row = qt * kTile + 32 * warp + lane;
    if (row < p.T) {
      uint4 *dst = reinterpret_cast<uint4 *>(p.o + ((size_t)row * p.heads + h) * kD);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint4 v;
        __half2 a = __floats2half2_rn(__uint_as_float(orow[8 * i]), __uint_as_float(orow[8 * i + 1]));
        __half2 b = __floats2half2_rn(__uint_as_float(orow[8 * i + 2]), __uint_as_float(orow[8 * i + 3]));
        __half2 cc = __floats2half2_rn(__uint_as_float(orow[8 * i + 4]), __uint_as_float(orow[8 * i + 5]));
        __half2 d = __floats2half2_rn(__uint_as_float(orow[8 * i + 6]), __uint_as_float(orow[8 * i + 7]));
        v.x = *reinterpret_cast<uint32_t *>(&a);
        v.y = *reinterpret_cast<uint32_t *>(&b);
        v.z = *reinterpret_cast<uint32_t *>(&cc);
        v.w = *reinterpret_cast<uint32_t *>(&d);
        dst[i] = v;
      }
    }
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// ---------------------------------------------------------------------------- host side
struct MatState {
  bool ready = false;
  int *status = nullptr;
};
std::mutex g_mat_mutex;
MatState g_mat[64];
std::atomic<int> g_mat_stall{0};   // test hook: the next attn_fwd_materialised call stalls one block
PFN_cuTensorMapEncodeTiled_v12000 g_mat_encode = nullptr;

int mat_state(MatState **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return ATTN_EDEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mat_mutex);
  MatState &st = g_mat[dev];
  if (!st.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return ATTN_EDEVICE;
    if (prop.major != 10 || prop.minor != 3) return ATTN_EDEVICE;
    if (!g_mat_encode) {
      cudaDriverEntryPointQueryResult q;
      void *fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return ATTN_ELAUNCH;
      g_mat_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (cudaFuncSetAttribute(scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kScoresSmem) != cudaSuccess ||
        cudaFuncSetAttribute(pv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kPvSmem) != cudaSuccess)
      return ATTN_ELAUNCH;
    if (cudaMalloc(&st.status, sizeof(int)) != cudaSuccess) return ATTN_ELAUNCH;
    if (cudaMemset(st.status, 0, sizeof(int)) != cudaSuccess) return ATTN_ELAUNCH;
    st.ready = true;
  }
  *out = &st;
  return ATTN_OK;
}

bool encode_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1,
               CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_FLOAT16) {
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1, stride2};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_mat_encode(m, dtype, 3, const_cast<void *>(base), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

int check_mat_shape(int T, int heads, int kv_heads, float c) {
  if (T <= 0 || heads <= 0 || kv_heads <= 0) return ATTN_EINVAL;
  if (T % 64 != 0 || T > kMaxT) return ATTN_EINVAL;
  if (heads % kv_heads != 0) return ATTN_EINVAL;
  if (heads > ATTN_MAX_HEADS) return ATTN_EINVAL;
  if ((uint64_t)heads * 64u * (uint64_t)T * 4u > 0xFFFFFFFFull) return ATTN_EINVAL;
  if (!std::isfinite(c) || !(c > 0.f)) return ATTN_EINVAL;
  return ATTN_OK;
}

size_t scores_bytes(int T, int heads) {
  return ((size_t)heads * T * T * 4 + 255) & ~(size_t)255;
}

}  // namespace

extern "C" size_t attn_materialised_workspace_bytes(int T, int heads, int kv_heads) {
  if (check_mat_shape(T, heads, kv_heads, 1.f)) return 0;
  return scores_bytes(T, heads) + (size_t)heads * T * T * 2;
}

extern "C" int attn_fwd_materialised(const void *q, const void *k, const void *vT, void *o,
                                     float *lse, int T, int heads, int kv_heads, float c,
                                     void *workspace, size_t workspace_bytes,
                                     cudaStream_t stream) {
  int rc = check_mat_shape(T, heads, kv_heads, c);
  if (rc) return rc;
  const void *ins[] = {q, k, vT};
  void *outs[] = {o, lse, workspace};
  for (const void *ptr : ins)
    if (!ptr) return ATTN_EINVAL;
  for (const void *ptr : outs)
    if (!ptr) return ATTN_EINVAL;
  for (const void *ptr : ins)
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return ATTN_EALIGN;
  for (const void *ptr : outs)
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return ATTN_EALIGN;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_EALIGN;
  const size_t ws = attn_materialised_workspace_bytes(T, heads, kv_heads);
  if (workspace_bytes < ws) return ATTN_EINVAL;
  const size_t hq = (size_t)heads * T * kD * 2, kvb = (size_t)kv_heads * T * kD * 2;
  const size_t in_sizes[] = {hq, kvb, kvb};
  const size_t out_sizes[] = {hq, (size_t)heads * T * 4, ws};
  for (int a = 0; a < 3; ++a) {
    for (int b = 0; b < 3; ++b)
      if (ranges_overlap(outs[a], out_sizes[a], ins[b], in_sizes[b])) return ATTN_EOVERLAP;
    for (int b = a + 1; b < 3; ++b)
      if (ranges_overlap(outs[a], out_sizes[a], outs[b], out_sizes[b])) return ATTN_EOVERLAP;
  }
  MatState *st = nullptr;
  if ((rc = mat_state(&st))) return rc;

  MatParams p;
  p.T = T;
  p.heads = heads;
  p.kv_heads = kv_heads;
  p.group = heads / kv_heads;
  p.q_tiles = (T + kTile - 1) / kTile;
  p.c = c;
  p.S = static_cast<float *>(workspace);
  p.P = reinterpret_cast<__half *>(static_cast<uint8_t *>(workspace) + scores_bytes(T, heads));
  p.o = static_cast<__half *>(o);
  p.lse = lse;
  p.status = st->status;
  p.stall = g_mat_stall.exchange(0);

  const uint64_t rowb = kD * 2, trow = (uint64_t)T * 2;
  CUtensorMap tmQ, tmK, tmP, tmVT, tmS;
  if (!encode_3d(&tmQ, q, kD, T, heads, rowb, rowb * T, kD, kTile) ||
      !encode_3d(&tmS, p.S, T, T, heads, (uint64_t)T * 4, (uint64_t)T * T * 4, 32, kTile,
                 CU_TENSOR_MAP_DATA_TYPE_FLOAT32) ||
      !encode_3d(&tmK, k, kD, T, kv_heads, rowb, rowb * T, kD, kTile) ||
      !encode_3d(&tmP, p.P, T, T, heads, trow, trow * T, 64, kTile) ||
      !encode_3d(&tmVT, vT, T, kD, kv_heads, trow, trow * kD, 64, kD))
    return ATTN_ELAUNCH;

  const int tri = p.q_tiles * (p.q_tiles + 1) / 2;
  scores_kernel<<<dim3(tri, heads), 128, kScoresSmem, stream>>>(tmQ, tmK, tmS, p);
  softmax_kernel<<<dim3((T + 7) / 8, heads), 256, 0, stream>>>(p);
  pv_kernel<<<dim3(p.q_tiles, heads), 128, kPvSmem, stream>>>(tmP, tmVT, p);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
  return ATTN_OK;
}

extern "C" int attn_materialised_last_device_status(cudaStream_t stream) {
  MatState *st = nullptr;
  int rc = mat_state(&st);
  if (rc) return rc;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ELAUNCH;
  int word = 0;
  if (cudaMemcpy(&word, st->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ELAUNCH;
  if (word != 0 && cudaMemset(st->status, 0, sizeof(int)) != cudaSuccess) return ATTN_ELAUNCH;
  return word ? ATTN_ETIMEOUT : ATTN_OK;
}

extern "C" int attn_materialised_test_inject_stall(void) {
  g_mat_stall.store(1);
  return ATTN_OK;
}
