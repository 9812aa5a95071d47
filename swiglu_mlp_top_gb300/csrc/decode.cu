// Decode-sized forward (T <= kDecodeMaxT tokens): weight-streaming kernels
// on the CUDA cores.  Each weight row is read from HBM exactly once with
// coalesced 16-byte loads and kept in registers while every token that needs
// it is applied, so the time is the weights' HBM traffic.  For the MoE only
// the experts some token selected are read.
//
//   gate/up:  h[a, i] = SiLU(Wg_e[i] . x_t) * (Wu_e[i] . x_t)   for every
//             assignment a = (t, s) with expert e     (lesson 13 §0/§1.2)
//   down:     y[t, j] = sum_s alpha_{t,s} * (Wd_{e_s}[j] . h[t, s])  in slot
//             order, fp32, rounded once (lesson 13 §0 MoE equation, step 5)
#include "mm_kernels.cuh"

namespace mm {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;

// 8 consecutive elements of a row, kept packed in registers.
template <typename T> struct Pack8;
template <> struct Pack8<__nv_bfloat16> { uint4 r; };
template <> struct Pack8<float> { uint4 r0, r1; };

__device__ __forceinline__ void ld_pack(const __nv_bfloat16* p, Pack8<__nv_bfloat16>& v) {
  v.r = __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void ld_pack(const float* p, Pack8<float>& v) {
  v.r0 = __ldg(reinterpret_cast<const uint4*>(p));
  v.r1 = __ldg(reinterpret_cast<const uint4*>(p) + 1);
}
__device__ __forceinline__ void unpack(const Pack8<__nv_bfloat16>& v, float (&f)[8]) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v.r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 q = __bfloat1622float2(b[i]);
    f[2 * i] = q.x;
    f[2 * i + 1] = q.y;
  }
}
__device__ __forceinline__ void unpack(const Pack8<float>& v, float (&f)[8]) {
  f[0] = __uint_as_float(v.r0.x); f[1] = __uint_as_float(v.r0.y);
  f[2] = __uint_as_float(v.r0.z); f[3] = __uint_as_float(v.r0.w);
  f[4] = __uint_as_float(v.r1.x); f[5] = __uint_as_float(v.r1.y);
  f[6] = __uint_as_float(v.r1.z); f[7] = __uint_as_float(v.r1.w);
}

template <typename T>
__device__ __forceinline__ void load8f(const T* p, float (&v)[8]);
template <>
__device__ __forceinline__ void load8f<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(b[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
template <>
__device__ __forceinline__ void load8f<float>(const float* p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The experts that some assignment selected, in ascending order (dense: one
// "expert" 0 with every token).  Written by thread 0 into shared memory.
struct Touched {
  int n;
  int e[MM_MAX_EXPERTS];
};

__device__ __forceinline__ void find_touched(const int32_t* topk_idx, int nA, int E, Touched* t) {
  if (threadIdx.x == 0) {
    uint64_t m = 0;
    if (topk_idx == nullptr) {
      m = 1;
    } else {
      for (int a = 0; a < nA; ++a) m |= 1ull << topk_idx[a];
    }
    int n = 0;
    for (int e = 0; e < E; ++e)
      if ((m >> e) & 1ull) t->e[n++] = e;
    t->n = n;
  }
  __syncthreads();
}

// ---------------------------------------------------------------- gate/up
// Work item = (touched expert, block of kDecWarps rows); warp w owns row
// i = block*kDecWarps + w and holds its Wg / Wu row slices in registers.
template <typename Tin, int MAXC>
__global__ void __launch_bounds__(kDecThreads)
stream_gateup_kernel(const Tin* __restrict__ x, const PtrArray wg, const PtrArray wu,
                     const int32_t* __restrict__ topk_idx, int T, int H, int I, int E, int k,
                     float* __restrict__ hdec) {
  __shared__ Touched tch;
  const int nA = (topk_idx != nullptr) ? T * k : T;
  find_touched(topk_idx, nA, E, &tch);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nch = H / 8;
  const int blocks = (I + kDecWarps - 1) / kDecWarps;
  const int items = tch.n * blocks;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int e = tch.e[item / blocks];
    const int i = (item % blocks) * kDecWarps + warp;
    if (i >= I) continue;                                  // warp-uniform
    const Tin* g_row = static_cast<const Tin*>(wg.p[e]) + static_cast<int64_t>(i) * H;
    const Tin* u_row = static_cast<const Tin*>(wu.p[e]) + static_cast<int64_t>(i) * H;
    Pack8<Tin> gw[MAXC], uw[MAXC];
#pragma unroll
    for (int c = 0; c < MAXC; ++c) {
      const int ch = lane + 32 * c;
      if (ch < nch) {
        ld_pack(g_row + ch * 8, gw[c]);
        ld_pack(u_row + ch * 8, uw[c]);
      }
    }
    for (int a = 0; a < nA; ++a) {
      if (topk_idx != nullptr && topk_idx[a] != e) continue;   // uniform: same a for the warp
      const int t = (topk_idx != nullptr) ? a / k : a;
      const Tin* xr = x + static_cast<int64_t>(t) * H;
      float g = 0.f, u = 0.f;
#pragma unroll
      for (int c = 0; c < MAXC; ++c) {
        const int ch = lane + 32 * c;
        if (ch < nch) {
          float xv[8], gf[8], uf[8];
          load8f(xr + ch * 8, xv);
          unpack(gw[c], gf);
          unpack(uw[c], uf);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            g = fmaf(gf[q], xv[q], g);
            u = fmaf(uf[q], xv[q], u);
          }
        }
      }
      g = warp_allsum(g);
      u = warp_allsum(u);
      if (lane == 0) hdec[static_cast<int64_t>(a) * I + i] = silu_f32(g) * u;
    }
  }
}

// ---------------------------------------------------------------- down + combine
// Work item = block of kRowsPerItem output rows j.  For every (touched
// expert, row) pair a warp streams Wd_e[j, :] once and forms the dot products
// with the h rows of that expert's assignments; the block then sums each
// token's slots in order.
constexpr int kRowsPerItem = 4;

template <typename Tout, int MAXC>
__global__ void __launch_bounds__(kDecThreads)
stream_down_kernel(const float* __restrict__ hdec, const PtrArray wd,
                   const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w, int T,
                   int H, int I, int E, int k, Tout* __restrict__ y) {
  __shared__ Touched tch;
  __shared__ float part[kDecodeMaxT * MM_MAX_TOPK][kRowsPerItem];
  const int nA = (topk_idx != nullptr) ? T * k : T;
  find_touched(topk_idx, nA, E, &tch);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nch = I / 8;
  const int items = (H + kRowsPerItem - 1) / kRowsPerItem;
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    const int j0 = item * kRowsPerItem;
    const int pairs = tch.n * kRowsPerItem;
    for (int pr = warp; pr < pairs; pr += kDecWarps) {
      const int e = tch.e[pr / kRowsPerItem];
      const int jl = pr % kRowsPerItem;
      const int j = j0 + jl;
      if (j >= H) continue;
      const Tout* d_row = static_cast<const Tout*>(wd.p[e]) + static_cast<int64_t>(j) * I;
      Pack8<Tout> dw[MAXC];
#pragma unroll
      for (int c = 0; c < MAXC; ++c) {
        const int ch = lane + 32 * c;
        if (ch < nch) ld_pack(d_row + ch * 8, dw[c]);
      }
      for (int a = 0; a < nA; ++a) {
        if (topk_idx != nullptr && topk_idx[a] != e) continue;
        const float* hr = hdec + static_cast<int64_t>(a) * I;
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < MAXC; ++c) {
          const int ch = lane + 32 * c;
          if (ch < nch) {
            float hv[8], df[8];
            load8f(hr + ch * 8, hv);
            unpack(dw[c], df);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc = fmaf(df[q], hv[q], acc);
          }
        }
        acc = warp_allsum(acc);
        if (lane == 0) part[a][jl] = acc;
      }
    }
    __syncthreads();
    const int ntok_rows = T * kRowsPerItem;
    for (int q = threadIdx.x; q < ntok_rows; q += blockDim.x) {
      const int t = q / kRowsPerItem, jl = q % kRowsPerItem;
      const int j = j0 + jl;
      if (j >= H) continue;
      float v;
      if (topk_idx == nullptr) {
        v = part[t][jl];
      } else {
        v = 0.f;
        for (int s = 0; s < k; ++s) v += topk_w[t * k + s] * part[t * k + s][jl];
      }
      y[static_cast<int64_t>(t) * H + j] = static_cast<Tout>(v);
    }
    __syncthreads();
  }
}

static int decode_grid(int items) {
  const int cap = 2 * num_sms();
  return items < cap ? (items > 0 ? items : 1) : cap;
}

// Chunks of 8 elements per lane for a reduction length K: ceil(K / 256),
// rounded up to an instantiated size.
static int chunks_for(int K) {
  const int c = (K + 255) / 256;
  return c <= 1 ? 1 : c <= 2 ? 2 : c <= 4 ? 4 : c <= 8 ? 8 : c <= 12 ? 12 : 16;
}

template <typename Tx>
static cudaError_t launch_stream_t(const void* x, const PtrArray& pg, const PtrArray& pu,
                                   const PtrArray& pd, const int32_t* topk_idx,
                                   const float* topk_w, int T, int H, int I, int nw, int k,
                                   float* hdec, void* y, cudaStream_t st) {
  const int g1 = decode_grid(nw * ((I + kDecWarps - 1) / kDecWarps));
  const int g2 = decode_grid((H + kRowsPerItem - 1) / kRowsPerItem);
#define MM_GU(C)                                                                              \
  stream_gateup_kernel<Tx, C><<<g1, kDecThreads, 0, st>>>(static_cast<const Tx*>(x), pg, pu,    \
                                                         topk_idx, T, H, I, nw, k, hdec)
  switch (chunks_for(H)) {
    case 1: MM_GU(1); break;
    case 2: MM_GU(2); break;
    case 4: MM_GU(4); break;
    case 8: MM_GU(8); break;
    case 12: MM_GU(12); break;
    default: MM_GU(16); break;
  }
#undef MM_GU
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
#define MM_DN(C)                                                                              \
  stream_down_kernel<Tx, C><<<g2, kDecThreads, 0, st>>>(hdec, pd, topk_idx, topk_w, T, H, I,   \
                                                       nw, k, static_cast<Tx*>(y))
  switch (chunks_for(I)) {
    case 1: MM_DN(1); break;
    case 2: MM_DN(2); break;
    case 4: MM_DN(4); break;
    case 8: MM_DN(8); break;
    case 12: MM_DN(12); break;
    default: MM_DN(16); break;
  }
#undef MM_DN
  return cudaGetLastError();
}

cudaError_t launch_stream_ffn(int dtype, const void* x, const void* const* Wg,
                              const void* const* Wu, const void* const* Wd,
                              const int32_t* topk_idx, const float* topk_w, int T, int H, int I,
                              int E, int k, float* hdec, void* y, cudaStream_t st) {
  PtrArray pg, pu, pd;
  const int nw = (topk_idx != nullptr) ? E : 1;
  for (int e = 0; e < nw; ++e) {
    pg.p[e] = Wg[e];
    pu.p[e] = Wu[e];
    pd.p[e] = Wd[e];
  }
  if (dtype == kDtypeBF16)
    return launch_stream_t<__nv_bfloat16>(x, pg, pu, pd, topk_idx, topk_w, T, H, I, nw, k, hdec,
                                          y, st);
  return launch_stream_t<float>(x, pg, pu, pd, topk_idx, topk_w, T, H, I, nw, k, hdec, y, st);
}

}  // namespace mm
