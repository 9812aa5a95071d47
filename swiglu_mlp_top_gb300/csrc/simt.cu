// CUDA-core (fp32 FMA) grouped FFN kernels.  They carry the fp32 workloads,
// where the tensor cores' TF32 rounding (about 2^-11 per input) would exceed
// the fp32 tolerance, and serve as an independent second GPU path for bf16.
// Same grouped layout as the tensor-core kernels: rows of A are grouped by
// expert (offsets), and tiles never straddle two groups.
//
// gate/up: h = SiLU(A Wg_e^T) ⊙ (A Wu_e^T)    (MiniMind lesson 13 §0/§1.2)
// down:    y[token] (+)= alpha * (h Wd_e^T)    (lesson 13 step 5)
#include "mm_kernels.cuh"

namespace mm {

constexpr int kSimtBM = 32, kSimtBN = 32, kSimtBK = 32, kSimtThreads = 256;

template <typename T>
__device__ __forceinline__ float ld_f32(const T* p);
template <>
__device__ __forceinline__ float ld_f32<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <>
__device__ __forceinline__ float ld_f32<__half>(const __half* p) { return __half2float(*p); }
template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

struct SimtTile {
  int g, w, row0, rows, n0;
};

__device__ __forceinline__ void simt_schedule(const GroupRows& g, int n_tiles, int* s_off,
                                              int* s_tstart) {
  if (threadIdx.x == 0) {
    int run = 0;
    for (int q = 0; q < g.G; ++q) {
      const int o0 = g.offsets ? g.offsets[q] : 0;
      const int o1 = g.offsets ? g.offsets[q + 1] : g.dense_rows;
      s_off[q] = o0;
      s_tstart[q] = run;
      run += ((o1 - o0 + kSimtBM - 1) / kSimtBM) * n_tiles;
    }
    s_off[g.G] = g.offsets ? g.offsets[g.G] : g.dense_rows;
    s_tstart[g.G] = run;
  }
  __syncthreads();
}

__device__ __forceinline__ SimtTile simt_tile(int t, const int* s_off, const int* s_tstart, int G,
                                              int n_weights, int n_tiles) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_tstart[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int q = lo;
  const int local = t - s_tstart[q];
  const int mb = local / n_tiles;
  SimtTile st;
  st.g = q;
  st.w = q % n_weights;
  st.row0 = s_off[q] + mb * kSimtBM;
  st.rows = min(kSimtBM, s_off[q + 1] - st.row0);
  st.n0 = (local - mb * n_tiles) * kSimtBN;
  return st;
}

template <typename T, typename Th>
__global__ void __launch_bounds__(kSimtThreads)
gateup_simt_kernel(const T* __restrict__ A, const GroupRows g, const PtrArray wg, const PtrArray wu,
                   int H, int I, Th* __restrict__ hout) {
  __shared__ int s_off[kMaxGroups + 1], s_tstart[kMaxGroups + 1];
  __shared__ float As[kSimtBM][kSimtBK + 1];
  __shared__ float Gs[kSimtBN][kSimtBK + 1];
  __shared__ float Us[kSimtBN][kSimtBK + 1];
  const int n_tiles = (I + kSimtBN - 1) / kSimtBN;
  simt_schedule(g, n_tiles, s_off, s_tstart);
  const int total = s_tstart[g.G];
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;

  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    const SimtTile ti = simt_tile(tile, s_off, s_tstart, g.G, g.n_weights, n_tiles);
    const T* Wg = static_cast<const T*>(wg.p[ti.w]);
    const T* Wu = static_cast<const T*>(wu.p[ti.w]);
    float ag[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, au[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    for (int k0 = 0; k0 < H; k0 += kSimtBK) {
      for (int i = tid; i < kSimtBM * kSimtBK; i += kSimtThreads) {
        const int r = i / kSimtBK, c = i % kSimtBK;
        const bool okk = k0 + c < H;
        As[r][c] = (r < ti.rows && okk) ? ld_f32(A + static_cast<int64_t>(ti.row0 + r) * H + k0 + c) : 0.f;
        const bool okn = ti.n0 + r < I;
        Gs[r][c] = (okn && okk) ? ld_f32(Wg + static_cast<int64_t>(ti.n0 + r) * H + k0 + c) : 0.f;
        Us[r][c] = (okn && okk) ? ld_f32(Wu + static_cast<int64_t>(ti.n0 + r) * H + k0 + c) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < kSimtBK; ++kk) {
        const float a0 = As[2 * ty][kk], a1 = As[2 * ty + 1][kk];
        const float g0 = Gs[2 * tx][kk], g1 = Gs[2 * tx + 1][kk];
        const float u0 = Us[2 * tx][kk], u1 = Us[2 * tx + 1][kk];
        ag[0][0] = fmaf(a0, g0, ag[0][0]); ag[0][1] = fmaf(a0, g1, ag[0][1]);
        ag[1][0] = fmaf(a1, g0, ag[1][0]); ag[1][1] = fmaf(a1, g1, ag[1][1]);
        au[0][0] = fmaf(a0, u0, au[0][0]); au[0][1] = fmaf(a0, u1, au[0][1]);
        au[1][0] = fmaf(a1, u0, au[1][0]); au[1][1] = fmaf(a1, u1, au[1][1]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = 2 * ty + i;
      if (r >= ti.rows) continue;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = ti.n0 + 2 * tx + j;
        if (c < I)
          hout[static_cast<int64_t>(ti.row0 + r) * I + c] = from_f32<Th>(silu_f32(ag[i][j]) * au[i][j]);
      }
    }
  }
}

template <typename T, typename Th>
__global__ void __launch_bounds__(kSimtThreads)
down_simt_kernel(const Th* __restrict__ Hm, const GroupRows g, const PtrArray wd, int H, int I,
                 const DownEpilogue ep) {
  __shared__ int s_off[kMaxGroups + 1], s_tstart[kMaxGroups + 1];
  __shared__ float As[kSimtBM][kSimtBK + 1];
  __shared__ float Ds[kSimtBN][kSimtBK + 1];
  const int n_tiles = (H + kSimtBN - 1) / kSimtBN;
  simt_schedule(g, n_tiles, s_off, s_tstart);
  const int total = s_tstart[g.G];
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  T* y = static_cast<T*>(ep.y);

  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    const SimtTile ti = simt_tile(tile, s_off, s_tstart, g.G, g.n_weights, n_tiles);
    const T* Wd = static_cast<const T*>(wd.p[ti.w]);
    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    for (int k0 = 0; k0 < I; k0 += kSimtBK) {
      for (int i = tid; i < kSimtBM * kSimtBK; i += kSimtThreads) {
        const int r = i / kSimtBK, c = i % kSimtBK;
        const bool okk = k0 + c < I;
        As[r][c] = (r < ti.rows && okk) ? ld_f32(Hm + static_cast<int64_t>(ti.row0 + r) * I + k0 + c) : 0.f;
        Ds[r][c] = (ti.n0 + r < H && okk) ? ld_f32(Wd + static_cast<int64_t>(ti.n0 + r) * I + k0 + c) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < kSimtBK; ++kk) {
        const float a0 = As[2 * ty][kk], a1 = As[2 * ty + 1][kk];
        const float d0 = Ds[2 * tx][kk], d1 = Ds[2 * tx + 1][kk];
        acc[0][0] = fmaf(a0, d0, acc[0][0]); acc[0][1] = fmaf(a0, d1, acc[0][1]);
        acc[1][0] = fmaf(a1, d0, acc[1][0]); acc[1][1] = fmaf(a1, d1, acc[1][1]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = 2 * ty + i;
      if (r >= ti.rows) continue;
      const int pos = ti.row0 + r;
      int64_t tok = pos;
      float alpha = 1.0f;
      if (ep.perm != nullptr) {
        const int a = ep.perm[pos];
        alpha = ep.topk_w != nullptr ? ep.topk_w[a] : 1.0f;
        tok = a / ep.k;
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int c = ti.n0 + 2 * tx + j;
        if (c >= H) continue;
        float v = alpha * acc[i][j];
        const int64_t o = tok * H + c;
        if (ep.mode == kCombineFirst) {
          ep.acc32[o] = v;
          continue;
        }
        if (ep.mode != kCombineStore) v += ep.acc32[o];
        if (ep.mode == kCombineAccum) {
          ep.acc32[o] = v;
        } else {
          if (ep.resid != nullptr) v += ld_f32(static_cast<const T*>(ep.resid) + o);
          y[o] = from_f32<T>(v);
        }
      }
    }
  }
}

static int simt_grid(int64_t a_rows, const GroupRows& g, int n_tiles) {
  int64_t tiles = (g.offsets == nullptr)
                      ? ((g.dense_rows + kSimtBM - 1) / kSimtBM) * static_cast<int64_t>(n_tiles)
                      : ((a_rows + kSimtBM - 1) / kSimtBM + g.G) * static_cast<int64_t>(n_tiles);
  const int64_t cap = 8LL * num_sms();
  if (tiles > cap) tiles = cap;
  return static_cast<int>(tiles > 0 ? tiles : 1);
}

cudaError_t launch_gateup_simt(int dtype, const void* A, int64_t a_rows, int H, int I,
                               const GroupRows& g, const void* const* Wg, const void* const* Wu,
                               void* h_out, cudaStream_t st) {
  PtrArray pg, pu;
  for (int e = 0; e < g.n_weights; ++e) {
    pg.p[e] = Wg[e];
    pu.p[e] = Wu[e];
  }
  const int grid = simt_grid(a_rows, g, (I + kSimtBN - 1) / kSimtBN);
  if (dtype == kDtypeBF16)
    gateup_simt_kernel<__nv_bfloat16, __half><<<grid, kSimtThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(A), g, pg, pu, H, I, static_cast<__half*>(h_out));
  else
    gateup_simt_kernel<float, float><<<grid, kSimtThreads, 0, st>>>(
        static_cast<const float*>(A), g, pg, pu, H, I, static_cast<float*>(h_out));
  return cudaGetLastError();
}

cudaError_t launch_down_simt(int dtype, const void* h, int64_t a_rows, int H, int I,
                             const GroupRows& g, const void* const* Wd, const DownEpilogue& ep,
                             cudaStream_t st) {
  PtrArray pd;
  for (int e = 0; e < g.n_weights; ++e) pd.p[e] = Wd[e];
  const int grid = simt_grid(a_rows, g, (H + kSimtBN - 1) / kSimtBN);
  if (dtype == kDtypeBF16)
    down_simt_kernel<__nv_bfloat16, __half><<<grid, kSimtThreads, 0, st>>>(
        static_cast<const __half*>(h), g, pd, H, I, ep);
  else
    down_simt_kernel<float, float><<<grid, kSimtThreads, 0, st>>>(static_cast<const float*>(h), g,
                                                                   pd, H, I, ep);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ watchdog
// One thread waits on an mbarrier that nothing arrives on; the bounded wait
// gives up after limit_us, records MM_ERR_TIMEOUT and the kernel returns.
__global__ void watchdog_selftest_kernel(WsHeader* hdr, uint32_t limit_us) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  const uint32_t addr = smem_u32(&bar);
  const unsigned long long t0 = globaltimer_ns();
  const unsigned long long limit = static_cast<unsigned long long>(limit_us) * 1000ull;
  uint32_t n = 0;
  while (!mbar_try_wait(addr, 0)) {
    if (globaltimer_ns() - t0 > limit || ++n > (1u << 30)) {
      report_timeout(hdr, 99);
      return;
    }
  }
}

cudaError_t launch_watchdog_selftest(WsHeader* hdr, uint32_t limit_us, cudaStream_t st) {
  watchdog_selftest_kernel<<<1, 32, 0, st>>>(hdr, limit_us);
  return cudaGetLastError();
}

}  // namespace mm
