// Grouped bf16 GEMMs on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators, TMA-fed shared-memory ring), persistent and warp-specialised:
//   warps 0-3  epilogue (TMEM -> registers -> global), one TMEM lane per row
//   warp 4     TMA producer (one elected lane)
//   warp 5     MMA issuer (one elected lane); owns the TMEM allocation
// Two TMEM accumulators let the epilogue of tile i overlap the MMAs of i+1.
//
// gate/up:  for the rows of group e:  G = A Wg_e^T, U = A Wu_e^T  (bf16; one
//           UMMA with N = 256: Wg rows n0..n0+127 stacked over Wu rows
//           n0..n0+127), epilogue h = SiLU(G) ⊙ U -> fp16.  G and U stay in TMEM.
//           (MiniMind lesson 13 "FFN 与 MoE" §0/§1.2 equations; minimind3.com
//           chapter 4 §4.2.)  h is stored in fp16 (11-bit significand): bf16
//           storage of h alone added ~0.005 RMS-relative max error on top of
//           the unavoidable bf16 rounding of y.
// down:     Y = h Wd_e^T (fp16 x fp16, Wd converted from bf16 exactly); the
//           epilogue scales each row by its routing weight alpha and writes /
//           accumulates it into y at the row's token (lesson 13 step 5:
//           expert output times weight, index_add_ into y).
#include <mutex>
#include <map>
#include <tuple>

#include "mm_kernels.cuh"

namespace mm {

// ------------------------------------------------------------------ geometry
constexpr int kUpStages = 4;
constexpr int kUpAStage = kTcBM * kTcBK * 2;             // 16 KiB
constexpr int kUpBStage = 2 * kUpBN * kTcBK * 2;         // 32 KiB (g rows | u rows)
constexpr int kUpAccStride = 256;                        // TMEM columns per accumulator
constexpr int kUpSmem = kUpStages * (kUpAStage + kUpBStage) + 2048;

constexpr int kDnStages = 5;
constexpr int kDnAStage = kTcBM * kTcBK * 2;             // 16 KiB
constexpr int kDnBStage = kDownBN * kTcBK * 2;           // 24 KiB
constexpr int kDnAccStride = 256;
constexpr int kDnSmem = kDnStages * (kDnAStage + kDnBStage) + 2048;

constexpr uint32_t kTmemCols = 512;
static_assert(kUpSmem <= 232448 && kDnSmem <= 232448, "shared memory budget");

template <int MAXE>
struct UpParams {
  CUtensorMap a;
  CUtensorMap wg[MAXE];
  CUtensorMap wu[MAXE];
};
template <int MAXE>
struct DownParams {
  CUtensorMap a;
  CUtensorMap wd[MAXE];
};

struct TileInfo {
  int g, w, row0, rows, n0;   // group, weight index, first row, valid rows, first column
};

// Tile t of the grouped problem: groups in order, within a group m-blocks of
// 128 rows, n-blocks fastest.  Binary search over the groups' first tiles.
__device__ __forceinline__ TileInfo decode_tile(int t, const int* s_off, const int* s_tstart, int G,
                                                int n_weights, int n_tiles, int BN) {
  int lo = 0, hi = G - 1;            // last group with s_tstart[g] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_tstart[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int g = lo;
  const int local = t - s_tstart[g];
  const int mb = local / n_tiles, nb = local - mb * n_tiles;
  TileInfo ti;
  ti.g = g;
  ti.w = g % n_weights;
  ti.row0 = s_off[g] + mb * kTcBM;
  ti.rows = min(kTcBM, s_off[g + 1] - ti.row0);
  ti.n0 = nb * BN;
  return ti;
}

__device__ __forceinline__ void build_schedule(const GroupRows& gr, int n_tiles, int* s_off,
                                               int* s_tstart) {
  int run = 0;
  for (int g = 0; g < gr.G; ++g) {
    const int o0 = gr.offsets ? gr.offsets[g] : 0;
    const int o1 = gr.offsets ? gr.offsets[g + 1] : gr.dense_rows;
    s_off[g] = o0;
    s_tstart[g] = run;
    run += ((o1 - o0 + kTcBM - 1) / kTcBM) * n_tiles;
  }
  s_off[gr.G] = gr.offsets ? gr.offsets[gr.G] : gr.dense_rows;
  s_tstart[gr.G] = run;
}

__device__ __forceinline__ uint8_t* align1024(unsigned char* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Warp-uniform bounded wait: every lane waits, then the warp agrees.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          WsHeader* hdr, unsigned where) {
  const bool ok = mbar_wait(bar, parity, abort, hdr, where);
  return __all_sync(0xffffffffu, ok);
}

// =============================================================== gate / up
template <int MAXE>
__global__ void __launch_bounds__(kTcThreads, 1)
gateup_tc_kernel(const __grid_constant__ UpParams<MAXE> P, const GroupRows g, const int H,
                 const int I, __half* __restrict__ hout, WsHeader* hdr) {
  extern __shared__ unsigned char smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kUpStages * kUpAStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kUpStages * kUpBStage);
  uint64_t* full = bars;
  uint64_t* empty = bars + kUpStages;
  uint64_t* tfull = bars + 2 * kUpStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drained = tempty + 2;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_off[kMaxGroups + 1], s_tstart[kMaxGroups + 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = (I + kUpBN - 1) / kUpBN;
  const int nkb = (H + kTcBK - 1) / kTcBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kUpStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4 * 32);
    }
    mbar_init(drained, 1);
    fence_mbar_init();
    s_abort = 0;
    build_schedule(g, n_tiles, s_off, s_tstart);
  }
  if (warp == 4 && lane == 0) tma_prefetch_desc(&P.a);
  if (warp == 5) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int total = s_tstart[g.G];
  volatile int* abort = &s_abort;

  if (warp == 4) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileInfo ti = decode_tile(tile, s_off, s_tstart, g.G, g.n_weights, n_tiles, kUpBN);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kUpStages;
          const uint32_t ph = (it / kUpStages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort, hdr, 1)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], kUpAStage + kUpBStage);
          tma_load_2d(sA + s * kUpAStage, &P.a, &full[s], kb * kTcBK, ti.row0);
          tma_load_2d(sB + s * kUpBStage, &P.wg[ti.w], &full[s], kb * kTcBK, ti.n0);
          tma_load_2d(sB + s * kUpBStage + kUpBStage / 2, &P.wu[ti.w], &full[s], kb * kTcBK,
                      ti.n0);
        }
      }
      if (!ok) {
        // let copies already in flight land before the CTA exits
        for (int j = 0; j < kUpStages; ++j) {
          const int i2 = it - 1 - j;
          if (i2 < 0) break;
          mbar_wait(&full[i2 % kUpStages], (i2 / kUpStages) & 1, nullptr, hdr, 2);
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTcBM, 2 * kUpBN);
      int it = 0, local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t aph = (local >> 1) & 1;
        if (!mbar_wait(&tempty[acc], aph ^ 1, abort, hdr, 3)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + acc * kUpAccStride;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kUpStages;
          const uint32_t ph = (it / kUpStages) & 1;
          if (!mbar_wait(&full[s], ph, abort, hdr, 4)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * kUpAStage);
          const uint32_t b0 = smem_u32(sB + s * kUpBStage);
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk)
            umma_bf16(d, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), idesc,
                      (kb > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
      }
      // all issued MMAs must finish before TMEM is released
      umma_commit(drained);
      mbar_wait(drained, 0, nullptr, hdr, 5);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue (warps 0-3)
    const int row = warp * 32 + lane;
    int local = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
      const TileInfo ti = decode_tile(tile, s_off, s_tstart, g.G, g.n_weights, n_tiles, kUpBN);
      const int acc = local & 1;
      const uint32_t aph = (local >> 1) & 1;
      if (!warp_wait(&tfull[acc], aph, abort, hdr, 6)) break;
      tc_fence_after();
      const uint32_t tb = tmem + (static_cast<uint32_t>(warp * 32) << 16) + acc * kUpAccStride;
      const bool valid = row < ti.rows;
      __half* dst = hout + static_cast<int64_t>(ti.row0 + (valid ? row : 0)) * I + ti.n0;
#pragma unroll 1
      for (int c = 0; c < kUpBN / 32; ++c) {
        uint32_t gr[32], ur[32];
        tmem_ld_32x32b_x32(tb + c * 32, gr);
        tmem_ld_32x32b_x32(tb + kUpBN + c * 32, ur);
        tmem_ld_wait();
        if (valid && ti.n0 + c * 32 < I) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float g0 = __uint_as_float(gr[2 * j]), g1 = __uint_as_float(gr[2 * j + 1]);
            const float u0 = __uint_as_float(ur[2 * j]), u1 = __uint_as_float(ur[2 * j + 1]);
            const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
            const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
            pk[j] = pack_f16x2(h0, h1);
          }
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

// =============================================================== down
template <int MAXE>
__global__ void __launch_bounds__(kTcThreads, 1)
down_tc_kernel(const __grid_constant__ DownParams<MAXE> P, const GroupRows g, const int H,
               const int I, const DownEpilogue ep, WsHeader* hdr) {
  extern __shared__ unsigned char smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kDnStages * kDnAStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kDnStages * kDnBStage);
  uint64_t* full = bars;
  uint64_t* empty = bars + kDnStages;
  uint64_t* tfull = bars + 2 * kDnStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drained = tempty + 2;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_off[kMaxGroups + 1], s_tstart[kMaxGroups + 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = (H + kDownBN - 1) / kDownBN;
  const int nkb = (I + kTcBK - 1) / kTcBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDnStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4 * 32);
    }
    mbar_init(drained, 1);
    fence_mbar_init();
    s_abort = 0;
    build_schedule(g, n_tiles, s_off, s_tstart);
  }
  if (warp == 4 && lane == 0) tma_prefetch_desc(&P.a);
  if (warp == 5) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int total = s_tstart[g.G];
  volatile int* abort = &s_abort;

  if (warp == 4) {
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const TileInfo ti = decode_tile(tile, s_off, s_tstart, g.G, g.n_weights, n_tiles, kDownBN);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kDnStages;
          const uint32_t ph = (it / kDnStages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort, hdr, 11)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], kDnAStage + kDnBStage);
          tma_load_2d(sA + s * kDnAStage, &P.a, &full[s], kb * kTcBK, ti.row0);
          tma_load_2d(sB + s * kDnBStage, &P.wd[ti.w], &full[s], kb * kTcBK, ti.n0);
        }
      }
      if (!ok) {
        for (int j = 0; j < kDnStages; ++j) {
          const int i2 = it - 1 - j;
          if (i2 < 0) break;
          mbar_wait(&full[i2 % kDnStages], (i2 / kDnStages) & 1, nullptr, hdr, 12);
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(kTcBM, kDownBN);
      int it = 0, local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t aph = (local >> 1) & 1;
        if (!mbar_wait(&tempty[acc], aph ^ 1, abort, hdr, 13)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + acc * kDnAccStride;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kDnStages;
          const uint32_t ph = (it / kDnStages) & 1;
          if (!mbar_wait(&full[s], ph, abort, hdr, 14)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * kDnAStage);
          const uint32_t b0 = smem_u32(sB + s * kDnBStage);
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk)
            umma_bf16(d, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), idesc,
                      (kb > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
      }
      umma_commit(drained);
      mbar_wait(drained, 0, nullptr, hdr, 15);
    }
    __syncwarp();
  } else {
    const int row = warp * 32 + lane;
    int local = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local) {
      const TileInfo ti = decode_tile(tile, s_off, s_tstart, g.G, g.n_weights, n_tiles, kDownBN);
      const int acc = local & 1;
      const uint32_t aph = (local >> 1) & 1;
      // per-row routing info is read before the accumulator is ready
      const bool valid = row < ti.rows;
      int64_t tok = 0;
      float alpha = 1.0f;
      if (valid) {
        const int pos = ti.row0 + row;
        if (ep.perm != nullptr) {
          const int a = ep.perm[pos];
          alpha = ep.topk_w != nullptr ? ep.topk_w[a] : 1.0f;
          tok = a / ep.k;
        } else {
          tok = pos;
        }
      }
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(ep.y) + tok * H + ti.n0;
      float* acc32 = ep.acc32 + tok * H + ti.n0;
      if (!warp_wait(&tfull[acc], aph, abort, hdr, 16)) break;
      tc_fence_after();
      const uint32_t tb = tmem + (static_cast<uint32_t>(warp * 32) << 16) + acc * kDnAccStride;
#pragma unroll 1
      for (int c = 0; c < kDownBN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tb + c * 32, r);
        tmem_ld_wait();
        if (valid && ti.n0 + c * 32 < H) {
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = alpha * __uint_as_float(r[j]);
          float4* a4 = reinterpret_cast<float4*>(acc32 + c * 32);
          if (ep.mode == kCombineFirst) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              a4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          } else {
            if (ep.mode != kCombineStore) {
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const float4 o = a4[q];
                v[4 * q] += o.x; v[4 * q + 1] += o.y; v[4 * q + 2] += o.z; v[4 * q + 3] += o.w;
              }
            }
            if (ep.mode == kCombineAccum) {
#pragma unroll
              for (int q = 0; q < 8; ++q)
                a4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            } else {
              uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
              for (int q = 0; q < 4; ++q)
                d4[q] = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]),
                                   pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                                   pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                                   pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

// =============================================================== host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 16-bit row-major [outer, inner] matrix (bf16 or fp16), box = 64 (inner) x
// box_rows (outer), 128-byte swizzle, zero fill outside the matrix.  Cached by
// (ptr, shape, box, type).
static bool make_map_16(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t outer,
                        uint32_t box_rows, bool is_f16) {
  using Key = std::tuple<uintptr_t, uint64_t, uint64_t, uint32_t, bool>;
  static std::mutex mu;
  static std::map<Key, CUtensorMap> cache;
  const Key key{reinterpret_cast<uintptr_t>(ptr), inner, outer, box_rows, is_f16};
  std::lock_guard<std::mutex> lock(mu);
  auto itc = cache.find(key);
  if (itc != cache.end()) {
    *out = itc->second;
    return true;
  }
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kTcBK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(out, is_f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         2, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (cache.size() > 4096) cache.clear();
  cache.emplace(key, *out);
  return true;
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

static int grid_for(int64_t a_rows, const GroupRows& g, int n_tiles) {
  int64_t tiles;
  if (g.offsets == nullptr)
    tiles = ((g.dense_rows + kTcBM - 1) / kTcBM) * static_cast<int64_t>(n_tiles);
  else
    tiles = ((a_rows + kTcBM - 1) / kTcBM + g.G) * static_cast<int64_t>(n_tiles);
  const int sms = num_sms();
  return static_cast<int>(tiles < sms ? (tiles > 0 ? tiles : 1) : sms);
}

template <int MAXE>
static cudaError_t gateup_impl(const void* A, int64_t a_rows, int H, int I, const GroupRows& g,
                               const void* const* Wg, const void* const* Wu, void* h_out,
                               WsHeader* hdr, cudaStream_t st) {
  UpParams<MAXE> p;
  memset(&p, 0, sizeof(p));
  if (!make_map_16(&p.a, A, H, a_rows, kTcBM, false)) return cudaErrorInvalidValue;
  for (int e = 0; e < g.n_weights; ++e) {
    if (!make_map_16(&p.wg[e], Wg[e], H, I, kUpBN, false)) return cudaErrorInvalidValue;
    if (!make_map_16(&p.wu[e], Wu[e], H, I, kUpBN, false)) return cudaErrorInvalidValue;
  }
  auto fn = gateup_tc_kernel<MAXE>;
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kUpSmem);
  if (err != cudaSuccess) return err;
  const int n_tiles = (I + kUpBN - 1) / kUpBN;
  fn<<<grid_for(a_rows, g, n_tiles), kTcThreads, kUpSmem, st>>>(
      p, g, H, I, static_cast<__half*>(h_out), hdr);
  return cudaGetLastError();
}

template <int MAXE>
static cudaError_t down_impl(const void* h, int64_t a_rows, int H, int I, const GroupRows& g,
                             const void* const* Wd, const DownEpilogue& ep, WsHeader* hdr,
                             cudaStream_t st) {
  DownParams<MAXE> p;
  memset(&p, 0, sizeof(p));
  if (!make_map_16(&p.a, h, I, a_rows, kTcBM, true)) return cudaErrorInvalidValue;
  for (int e = 0; e < g.n_weights; ++e)
    if (!make_map_16(&p.wd[e], Wd[e], I, H, kDownBN, true)) return cudaErrorInvalidValue;
  auto fn = down_tc_kernel<MAXE>;
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kDnSmem);
  if (err != cudaSuccess) return err;
  const int n_tiles = (H + kDownBN - 1) / kDownBN;
  fn<<<grid_for(a_rows, g, n_tiles), kTcThreads, kDnSmem, st>>>(p, g, H, I, ep, hdr);
  return cudaGetLastError();
}

cudaError_t launch_gateup_tc(const void* A, int64_t a_rows, int H, int I, const GroupRows& g,
                             const void* const* Wg, const void* const* Wu, void* h_out,
                             WsHeader* hdr, cudaStream_t st) {
  if (g.n_weights <= 8) return gateup_impl<8>(A, a_rows, H, I, g, Wg, Wu, h_out, hdr, st);
  return gateup_impl<MM_MAX_EXPERTS>(A, a_rows, H, I, g, Wg, Wu, h_out, hdr, st);
}

cudaError_t launch_down_tc(const void* h, int64_t a_rows, int H, int I, const GroupRows& g,
                           const void* const* Wd, const DownEpilogue& ep, WsHeader* hdr,
                           cudaStream_t st) {
  if (g.n_weights <= 8) return down_impl<8>(h, a_rows, H, I, g, Wd, ep, hdr, st);
  return down_impl<MM_MAX_EXPERTS>(h, a_rows, H, I, g, Wd, ep, hdr, st);
}

}  // namespace mm
