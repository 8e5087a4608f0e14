// attn_qkv.cu -- the fused QKV producer for GB300 (sm_103a), behind attn_qkv.h:
// the QKV product of the normed activations with the QKV matrix on the tensor
// cores, with the rotary embedding of the query and key heads and the value
// transpose done in the product's epilogue (the page ".../Coppelius/Build/Graph.alpha"
// runs these as the QKV product, then "qk-rope", then "value-transpose").
//
// A persistent grid (one CTA per SM) walks the output tiles in pairs: tokens
// 256 m' .. +255 (two 128-token tiles, taken by CTAs 2i and 2i + 1) x outputs
// 192 n .. +191 (three heads; 1024 tiles fill seven waves of 152 SMs to 96 %,
// where four-head tiles filled six to 84 %).  The two CTAs of a pair read the
// same W slice at about the same time, so the second read is served by L2.  In
// each CTA warp 0 (one lane) streams 64-wide slices of its X tile and of the W
// slice through a five-stage TMA ring, with plain loads into its own shared
// memory; warp 1 issues the tcgen05 MMAs (M = 128, N = 192, K = 16) into one of
// two tensor-memory accumulators and releases each stage once they have read it;
// warps 2-5 (one token per thread) take a finished accumulator, rotate the
// query and key heads' pairs in binary32, round to binary16 and write Q and K
// rows and V^T columns, while the next tile accumulates in the other buffer.
// Every wait is bounded (1 s); a timeout is recorded in a status word.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <atomic>
#include <mutex>

#include "attn_qkv.h"
#include "sm103_ptx.cuh"

namespace {

using namespace sm103;

constexpr int kD = 64;                      // head width
constexpr int kBM = 128;                    // tokens per tile (= TMEM lanes)
constexpr int kBN = 192;                    // outputs per tile: three heads
constexpr int kBK = 64;                     // width slice per stage (one 128-byte swizzle row)
constexpr int kStages = 5;
constexpr uint32_t kABytes = kBM * kBK * 2;   // 16 KiB
constexpr uint32_t kBBytes = kBN * kBK * 2;   // 24 KiB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kOffBar = kStages * kStageBytes;
constexpr int kBarFull = 0, kBarEmpty = kStages, kBarAccFull = 2 * kStages,
              kBarAccFree = kBarAccFull + 2, kBarDrain = kBarAccFree + 2;
constexpr int kNumBars = kBarDrain + 1;
constexpr uint32_t kOffTmemPtr = kOffBar + kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemPtr + 4;
constexpr uint32_t kSmemBytes = kOffAbort + 4 + 1024;
constexpr int kThreads = 32 * 6;
constexpr int kEpiWarps = 4;
constexpr uint64_t kWaitLimitNs = 1000000000ull;


struct QkvParams {
  int T, width, heads, kv_heads, n_out, m_tiles, n_tiles, k_slices;
  const float *cosines, *sines;
  __half *q, *k, *vT;
  int *status;
  int stall;          // test hook: CTA 0 never loads the X half of its first stage
};

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
    return __all_sync(0xffffffffu, wait(i, parity, where));
  }
  __device__ void drain_wait(int i, uint32_t parity) const {
    const uint32_t b = bar(i);
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(b, parity))
      if (globaltimer_ns() - t0 > kWaitLimitNs) break;
  }
};

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ void load_role(const CUtensorMap *tmX, const CUtensorMap *tmW, const QkvParams &p,
                          const Sync &sy, uint32_t smem) {
  const int pairs = (p.m_tiles + 1) / 2 * p.n_tiles;
  const int rank = (int)(blockIdx.x & 1);
  uint32_t it = 0, issued = 0;
  for (int tp = blockIdx.x / 2; tp < pairs; tp += gridDim.x / 2) {
    const int m = 2 * (tp / p.n_tiles) + rank, n = tp % p.n_tiles;
    for (int kc = 0; kc < p.k_slices; ++kc, ++it) {
      const uint32_t s = it % kStages;
      if (!sy.wait(kBarEmpty + s, ((it / kStages) & 1) ^ 1, 401)) goto drain;
      const uint32_t dst = smem + s * kStageBytes;
      mbar_arrive_expect_tx(sy.bar(kBarFull + s), kStageBytes);
      issued = it + 1;
      if (!(p.stall && blockIdx.x == 0 && it == 0))   // test hook: this X slice never lands
        tma_load_3d(dst, tmX, sy.bar(kBarFull + s), kc * kBK, m * kBM, 0);
      tma_load_3d(dst + kABytes, tmW, sy.bar(kBarFull + s), kc * kBK, n * kBN, 0);
    }
  }
  return;
drain:
  for (uint32_t i = 0; i < kStages && i < issued; ++i) {
    const uint32_t j = issued - 1 - i;
    sy.drain_wait(kBarFull + j % kStages, (j / kStages) & 1);
  }
}

__device__ void mma_role(const QkvParams &p, const Sync &sy, uint32_t smem, uint32_t tmem) {
  constexpr uint32_t id = idesc_f16_f32(kBM, kBN);
  const int pairs = (p.m_tiles + 1) / 2 * p.n_tiles;
  uint32_t it = 0, lt = 0;
  for (int tp = blockIdx.x / 2; tp < pairs; tp += gridDim.x / 2, ++lt) {
    const uint32_t b = lt & 1;
    if (!sy.wait_warp(kBarAccFree + b, ((lt >> 1) & 1) ^ 1, 411)) goto drain;
    tc_fence_after();
    for (int kc = 0; kc < p.k_slices; ++kc, ++it) {
      const uint32_t s = it % kStages;
      if (!sy.wait_warp(kBarFull + s, (it / kStages) & 1, 412)) goto drain;
      tc_fence_after();
      const uint32_t base = smem + s * kStageBytes;
#pragma unroll
      for (int e = 0; e < kBK / 16; ++e)
        mma_ss(tmem + kBN * b, sw128_desc(base + e * 32), sw128_desc(base + kABytes + e * 32), id,
               (kc > 0 || e > 0) ? 1u : 0u);
      mma_commit(sy.bar(kBarEmpty + s));
    }
    mma_commit(sy.bar(kBarAccFull + b));
  }
  return;
drain:
  mma_commit(sy.bar(kBarDrain));
  sy.drain_wait(kBarDrain, 0);
}

// Warps 2-5: thread = token row of the tile (tensor-memory lane 32 (warp % 4) + lane).
__device__ void epilogue_role(const QkvParams &p, const Sync &sy, uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = 32 * (warp & 3) + lane;
  const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
  const int pairs = (p.m_tiles + 1) / 2 * p.n_tiles;
  const int heads_all = p.heads + 2 * p.kv_heads;
  const int rank = (int)(blockIdx.x & 1);
  uint32_t lt = 0;
  for (int tp = blockIdx.x / 2; tp < pairs; tp += gridDim.x / 2, ++lt) {
    const int m = 2 * (tp / p.n_tiles) + rank, n = tp % p.n_tiles;
    const uint32_t b = lt & 1;
    const int tok = m * kBM + r;
    const bool valid = tok < p.T;
    // this token's rotary row (the tables are [T][32])
    float cs[kD / 2], sn[kD / 2];
    if (valid) {
      const float4 *c4 = reinterpret_cast<const float4 *>(p.cosines + (size_t)tok * (kD / 2));
      const float4 *s4 = reinterpret_cast<const float4 *>(p.sines + (size_t)tok * (kD / 2));
#pragma unroll
      for (int i = 0; i < kD / 8; ++i) {
        const float4 a = c4[i], z = s4[i];
        cs[4 * i] = a.x, cs[4 * i + 1] = a.y, cs[4 * i + 2] = a.z, cs[4 * i + 3] = a.w;
        sn[4 * i] = z.x, sn[4 * i + 1] = z.y, sn[4 * i + 2] = z.z, sn[4 * i + 3] = z.w;
      }
    }
    if (!sy.wait_warp(kBarAccFull + b, (lt >> 1) & 1, 421)) return;
    tc_fence_after();
#pragma unroll 1
    for (int hh = 0; hh < kBN / kD; ++hh) {
      const int gh = n * (kBN / kD) + hh;   // head across the three parts
      if (gh >= heads_all) break;
      uint32_t acc[64];
      tmem_ld_x64(tmem + lane_base + kBN * b + kD * hh, acc);
      if (!valid) continue;
      if (gh < p.heads + p.kv_heads) {
        // query or key head: rotate each pair, round, write the 128-byte row
        __half *dst = gh < p.heads ? p.q + ((size_t)gh * p.T + tok) * kD
                                   : p.k + ((size_t)(gh - p.heads) * p.T + tok) * kD;
        uint32_t o[32];
#pragma unroll
        for (int pr = 0; pr < kD / 2; ++pr) {
          const float a = __uint_as_float(acc[2 * pr]), bb = __uint_as_float(acc[2 * pr + 1]);
          o[pr] = pack_half2(fmaf(a, cs[pr], -bb * sn[pr]), fmaf(a, sn[pr], bb * cs[pr]));
        }
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int i = 0; i < 8; ++i) d4[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
      } else {
        // value head: column tok of V^T (consecutive lanes write consecutive tokens)
        __half *dst = p.vT + (size_t)(gh - p.heads - p.kv_heads) * kD * p.T + tok;
#pragma unroll
        for (int e = 0; e < kD; ++e) dst[(size_t)e * p.T] = __float2half_rn(__uint_as_float(acc[e]));
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sy.bar(kBarAccFree + b));
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    qkv_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
               const QkvParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t smem = (raw + 1023u) & ~1023u;
  uint8_t *smem_gen = smem_raw + (smem - raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Sync sy;
  sy.bar0 = smem + kOffBar;
  sy.abort_flag = reinterpret_cast<volatile int *>(smem_gen + kOffAbort);
  sy.status = p.status;
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(sy.bar(kBarFull + i), 1);
      mbar_init(sy.bar(kBarEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sy.bar(kBarAccFull + i), 1);
      mbar_init(sy.bar(kBarAccFree + i), kEpiWarps);
    }
    mbar_init(sy.bar(kBarDrain), 1);
    *sy.abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(smem + kOffTmemPtr, 512);   // two accumulators of kBN columns
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem_gen + kOffTmemPtr);
  if (warp == 0) {
    if (lane == 0) load_role(&tmX, &tmW, p, sy, smem);
    __syncwarp();
  } else if (warp == 1) {
    mma_role(p, sy, smem, tmem);
  } else {
    epilogue_role(p, sy, tmem);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------- host side
struct QkvState {
  bool ready = false;
  int sms = 0;
  int *status = nullptr;
};
std::mutex g_qkv_mutex;
QkvState g_qkv[64];
std::atomic<int> g_qkv_stall{0};   // test hook: the next attn_qkv_rope call stalls one CTA
PFN_cuTensorMapEncodeTiled_v12000 g_qkv_encode = nullptr;

int qkv_state(QkvState **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return ATTN_EDEVICE;
  }
  std::lock_guard<std::mutex> lock(g_qkv_mutex);
  QkvState &st = g_qkv[dev];
  if (!st.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return ATTN_EDEVICE;
    if (prop.major != 10 || prop.minor != 3) return ATTN_EDEVICE;
    if (!g_qkv_encode) {
      cudaDriverEntryPointQueryResult q;
      void *fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return ATTN_ELAUNCH;
      g_qkv_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (cudaFuncSetAttribute(qkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
      return ATTN_ELAUNCH;
    if (cudaMalloc(&st.status, sizeof(int)) != cudaSuccess) return ATTN_ELAUNCH;
    if (cudaMemset(st.status, 0, sizeof(int)) != cudaSuccess) return ATTN_ELAUNCH;
    st.sms = prop.multiProcessorCount;
    st.ready = true;
  }
  *out = &st;
  return ATTN_OK;
}

// A 2-D binary16 matrix [rows][cols] (cols contiguous), 128-byte swizzle, box
// of 64 columns x box_rows rows.
bool encode_rows(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  cuuint64_t dims[3] = {cols, rows, 1};
  cuuint64_t strides[2] = {cols * 2, cols * 2 * rows};
  cuuint32_t box[3] = {(cuuint32_t)kBK, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_qkv_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

extern "C" int attn_qkv_rope(const void *x, const void *w, const float *cosines,
                             const float *sines, void *q, void *k, void *vT, int T, int width,
                             int heads, int kv_heads, cudaStream_t stream) {
  if (T <= 0 || T % 64 != 0 || width <= 0 || width % kBK != 0) return ATTN_EINVAL;
  if (heads <= 0 || kv_heads <= 0 || heads % kv_heads != 0 || heads > ATTN_MAX_HEADS)
    return ATTN_EINVAL;
  if ((uint64_t)heads * 64u * (uint64_t)T * 4u > 0xFFFFFFFFull) return ATTN_EINVAL;
  const void *ins[] = {x, w, cosines, sines};
  void *outs[] = {q, k, vT};
  for (const void *ptr : ins)
    if (!ptr) return ATTN_EINVAL;
  for (const void *ptr : outs)
    if (!ptr) return ATTN_EINVAL;
  for (const void *ptr : ins)
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return ATTN_EALIGN;
  for (const void *ptr : outs)
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return ATTN_EALIGN;
  const int n_out = (heads + 2 * kv_heads) * kD;
  const size_t in_sizes[] = {(size_t)T * width * 2, (size_t)n_out * width * 2,
                             (size_t)T * (kD / 2) * 4, (size_t)T * (kD / 2) * 4};
  const size_t out_sizes[] = {(size_t)heads * T * kD * 2, (size_t)kv_heads * T * kD * 2,
                              (size_t)kv_heads * T * kD * 2};
  for (int a = 0; a < 3; ++a) {
    for (int b = 0; b < 4; ++b)
      if (ranges_overlap(outs[a], out_sizes[a], ins[b], in_sizes[b])) return ATTN_EOVERLAP;
    for (int b = a + 1; b < 3; ++b)
      if (ranges_overlap(outs[a], out_sizes[a], outs[b], out_sizes[b])) return ATTN_EOVERLAP;
  }
  QkvState *st = nullptr;
  int rc = qkv_state(&st);
  if (rc) return rc;
  CUtensorMap tmX, tmW;
  if (!encode_rows(&tmX, x, width, T, kBM) || !encode_rows(&tmW, w, width, n_out, kBN))
    return ATTN_ELAUNCH;
  QkvParams p;
  p.T = T;
  p.width = width;
  p.heads = heads;
  p.kv_heads = kv_heads;
  p.n_out = n_out;
  p.m_tiles = (T + kBM - 1) / kBM;
  p.n_tiles = (n_out + kBN - 1) / kBN;
  p.k_slices = width / kBK;
  p.cosines = cosines;
  p.sines = sines;
  p.q = static_cast<__half *>(q);
  p.k = static_cast<__half *>(k);
  p.vT = static_cast<__half *>(vT);
  p.status = st->status;
  p.stall = g_qkv_stall.exchange(0);
  const int pairs = (p.m_tiles + 1) / 2 * p.n_tiles;
  // an even grid: CTAs 2i and 2i + 1 take the two token tiles of a pair
  const int slots = st->sms / 2;
  const int grid = 2 * (pairs < slots ? pairs : slots);
  qkv_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tmX, tmW, p);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
  return ATTN_OK;
}

extern "C" int attn_qkv_last_device_status(cudaStream_t stream) {
  QkvState *st = nullptr;
  int rc = qkv_state(&st);
  if (rc) return rc;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ELAUNCH;
  int word = 0;
  if (cudaMemcpy(&word, st->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ELAUNCH;
  if (word != 0 && cudaMemset(st->status, 0, sizeof(int)) != cudaSuccess) return ATTN_ELAUNCH;
  return word ? ATTN_ETIMEOUT : ATTN_OK;
}

extern "C" int attn_qkv_test_inject_stall(void) {
  g_qkv_stall.store(1);
  return ATTN_OK;
}
