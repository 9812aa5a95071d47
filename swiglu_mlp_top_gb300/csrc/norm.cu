// RMSNorm prologue of the MiniMind block (lesson 13 "FFN 与 MoE" §3 step 2:
// hidden_states + mlp(post_attention_layernorm(hidden_states)); the pages
// name the norm an RMSNorm: x / sqrt(mean_h x_h^2 + eps) * w).
//   - norm_fold_router: the router weights with w folded in, split into two
//     bf16 halves whose sum is w_h * Wr[e][h] exactly (the product of two
//     bf16 has at most 16 significant bits: hi keeps the top 8, lo the rest),
//     so that the tensor-core router's products x_h * hi + x_h * lo are exact;
//   - rms_norm_rows: x_n = x * inv_rms * w in x's dtype, and inv_rms per token,
//     for the paths that read the normalised rows from memory (dense FFN).
#include <cstring>

#include "mm_kernels.cuh"

namespace mm {

// Both kernels are programmatic dependents (pdl_enter): they wait for the
// previous kernel (which may still read their output, or write their input),
// then let the next one launch at once; it waits for them before reading.

__global__ void norm_fold_router_kernel(const __nv_bfloat16* __restrict__ Wr,
                                        const __nv_bfloat16* __restrict__ w, int E, int H,
                                        __nv_bfloat16* __restrict__ wr_hl) {
  pdl_enter();
  const int64_t n = static_cast<int64_t>(E) * H;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float p = __bfloat162float(Wr[i]) * __bfloat162float(w[i % H]);   // exact
    const __nv_bfloat16 hi = __float2bfloat16_rn(p);
    const __nv_bfloat16 lo = __float2bfloat16_rn(p - __bfloat162float(hi));  // exact remainder
    wr_hl[i] = hi;
    wr_hl[n + i] = lo;
  }
}

// 16-byte vectors of 8 bf16 / 4 fp32 as fp32 values, and back.
template <typename T> struct Vec16;
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int kN = 8;
  __device__ static void load(const void* p, float (&v)[8]) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(w[j] << 16);
      v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  }
  __device__ static void store(void* p, const float (&v)[8]) {
    *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                              pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
  }
};
template <> struct Vec16<float> {
  static constexpr int kN = 4;
  __device__ static void load(const void* p, float (&v)[4]) {
    const float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  __device__ static void store(void* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};

// One warp per row, 16-byte vectors: the sum of squares in fp32 (lane
// partial sums, a fixed tree), then the row times inv_rms * w (the row is
// read again from L1 / L2).
template <typename T>
__global__ void rms_norm_rows_kernel(const T* __restrict__ x, const T* __restrict__ w, float eps,
                                     int64_t n_rows, int H, T* __restrict__ xn,
                                     float* __restrict__ inv_rms) {
  using V = Vec16<T>;
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= n_rows) return;
  const T* xr = x + row * H;
  const int nv = H / V::kN;
  // the lane's first kCache vectors stay in registers between the two passes
  constexpr int kCache = 8;
  float cache[kCache][V::kN];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kCache; ++i) {
    const int c = lane + 32 * i;
    if (c < nv) {
      V::load(xr + c * V::kN, cache[i]);
#pragma unroll
      for (int j = 0; j < V::kN; ++j) ss = fmaf(cache[i][j], cache[i][j], ss);
    }
  }
  for (int c = lane + 32 * kCache; c < nv; c += 32) {
    float v[V::kN];
    V::load(xr + c * V::kN, v);
#pragma unroll
    for (int j = 0; j < V::kN; ++j) ss = fmaf(v[j], v[j], ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float s = 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
  if (lane == 0 && inv_rms != nullptr) inv_rms[row] = s;
  T* out = xn + row * H;
#pragma unroll
  for (int i = 0; i < kCache; ++i) {
    const int c = lane + 32 * i;
    if (c < nv) {
      float g[V::kN];
      V::load(w + c * V::kN, g);
#pragma unroll
      for (int j = 0; j < V::kN; ++j) cache[i][j] = cache[i][j] * s * g[j];
      V::store(out + c * V::kN, cache[i]);
    }
  }
  for (int c = lane + 32 * kCache; c < nv; c += 32) {
    float v[V::kN], g[V::kN];
    V::load(xr + c * V::kN, v);
    V::load(w + c * V::kN, g);
#pragma unroll
    for (int j = 0; j < V::kN; ++j) v[j] = v[j] * s * g[j];
    V::store(out + c * V::kN, v);
  }
}

template <typename Kern, typename... Args>
static cudaError_t launch_dependent(Kern fn, int grid, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, args...);
}

cudaError_t launch_norm_fold_router(const void* Wr, const void* w, int E, int H, void* wr_hl,
                                    cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(E) * H;
  const int grid = static_cast<int>((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
  return launch_dependent(norm_fold_router_kernel, grid, st, static_cast<const __nv_bfloat16*>(Wr),
                          static_cast<const __nv_bfloat16*>(w), E, H,
                          static_cast<__nv_bfloat16*>(wr_hl));
}

cudaError_t launch_rms_norm_rows(int dtype, const void* x, const void* w, float eps, int64_t T,
                                 int H, void* xn, float* inv_rms, cudaStream_t st) {
  const int grid = static_cast<int>((T + 7) / 8);
  if (dtype == kDtypeBF16)
    return launch_dependent(rms_norm_rows_kernel<__nv_bfloat16>, grid, st,
                            static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w),
                            eps, T, H, static_cast<__nv_bfloat16*>(xn), inv_rms);
  return launch_dependent(rms_norm_rows_kernel<float>, grid, st, static_cast<const float*>(x),
                          static_cast<const float*>(w), eps, T, H, static_cast<float*>(xn), inv_rms);
}

}  // namespace mm
