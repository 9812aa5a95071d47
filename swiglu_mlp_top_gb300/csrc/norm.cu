// RMSNorm prologue of the MiniMind block (lesson 13 "FFN 与 MoE" §3 step 2:
// hidden_states + mlp(post_attention_layernorm(hidden_states)); the pages
// name the norm an RMSNorm: x / sqrt(mean_h x_h^2 + eps) * w).
//   - norm_fold_router: the router weights with w folded in, split into two
//     bf16 halves whose sum is w_h * Wr[e][h] exactly (the product of two
//     bf16 has at most 16 significant bits: hi keeps the top 8, lo the rest),
//     so that the tensor-core router's products x_h * hi + x_h * lo are exact;
//   - rms_norm_rows: x_n = x * inv_rms * w in x's dtype, and inv_rms per token,
//     for the paths that read the normalised rows from memory (dense FFN).
#include "mm_kernels.cuh"

namespace mm {

__global__ void norm_fold_router_kernel(const __nv_bfloat16* __restrict__ Wr,
                                        const __nv_bfloat16* __restrict__ w, int E, int H,
                                        __nv_bfloat16* __restrict__ wr_hl) {
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

// One warp per row: sum of squares in fp32 (lane-strided, fixed tree), then
// the row times inv_rms * w.
template <typename T>
__global__ void rms_norm_rows_kernel(const T* __restrict__ x, const T* __restrict__ w, float eps,
                                     int64_t n_rows, int H, T* __restrict__ xn,
                                     float* __restrict__ inv_rms) {
  const int lane = threadIdx.x & 31;
  const int64_t row = blockIdx.x * static_cast<int64_t>(blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= n_rows) return;
  const T* xr = x + row * H;
  float ss = 0.f;
  for (int h = lane; h < H; h += 32) {
    const float v = static_cast<float>(xr[h]);
    ss = fmaf(v, v, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float s = 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
  if (lane == 0 && inv_rms != nullptr) inv_rms[row] = s;
  T* out = xn + row * H;
  for (int h = lane; h < H; h += 32) out[h] = static_cast<T>(static_cast<float>(xr[h]) * s * static_cast<float>(w[h]));
}

cudaError_t launch_norm_fold_router(const void* Wr, const void* w, int E, int H, void* wr_hl,
                                    cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(E) * H;
  const int grid = static_cast<int>((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
  norm_fold_router_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(Wr),
                                                static_cast<const __nv_bfloat16*>(w), E, H,
                                                static_cast<__nv_bfloat16*>(wr_hl));
  return cudaGetLastError();
}

cudaError_t launch_rms_norm_rows(int dtype, const void* x, const void* w, float eps, int64_t T,
                                 int H, void* xn, float* inv_rms, cudaStream_t st) {
  const int grid = static_cast<int>((T + 7) / 8);
  if (dtype == kDtypeBF16)
    rms_norm_rows_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w), eps, T, H,
        static_cast<__nv_bfloat16*>(xn), inv_rms);
  else
    rms_norm_rows_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(x),
                                                     static_cast<const float*>(w), eps, T, H,
                                                     static_cast<float*>(xn), inv_rms);
  return cudaGetLastError();
}

}  // namespace mm
