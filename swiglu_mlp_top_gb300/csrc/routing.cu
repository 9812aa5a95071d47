// Router (logits, softmax, top-k, renormalisation, aux partials), the
// dispatch of tokens into expert-contiguous rows, the aux-loss finalisation
// and the ordered combine used when k >= 3.
//
// Follows MiniMind lesson 13 "FFN 与 MoE" §1.5 (router equations), §1.6 and
// step 6 (aux loss), step 4-5 (top-k, renormalisation, per-expert dispatch
// and index_add_ into y), and minimind3.com chapter 4 §4.3-§4.4.
#include "mm_kernels.cuh"

namespace mm {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <typename Tin>
__device__ __forceinline__ void load_vec8(const Tin* p, float (&v)[8]);

template <>
__device__ __forceinline__ void load_vec8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
  uint4 raw = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

template <>
__device__ __forceinline__ void load_vec8<float>(const float* p, float (&v)[8]) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// ---------------------------------------------------------------------------
// Router: one warp per token, kRouteTokensPerBlock tokens per block.
//   r_e = sum_h x[t,h] Wr[e,h] (+ bias_e)      fp32, lanes split h, xor-tree sum
//   p = softmax(r)                              fp32, max subtracted
//   S = k largest p, ties -> lower index        sequential selection
//   alpha_s = p_S[s] / (sum_S p + 1e-20)
// Per-block partials of count_e and sum_t p_{t,e} are reduced in a fixed
// order (token order within a warp, then warp order) so results do not
// depend on scheduling.
// ---------------------------------------------------------------------------
template <typename Tin, int MAXE>
__global__ void __launch_bounds__(kRouteThreads)
router_kernel(const Tin* __restrict__ x, const Tin* __restrict__ Wr, const float* __restrict__ bias,
              int64_t T, int H, int E, int k, int32_t* __restrict__ topk_idx,
              float* __restrict__ topk_w, int32_t* __restrict__ blk_cnt,
              float* __restrict__ blk_prob) {
  extern __shared__ __align__(16) unsigned char route_smem[];
  float* w_s = reinterpret_cast<float*>(route_smem);                 // [E][H]
  __shared__ float red_p[kRouteThreads / 32][MAXE];
  __shared__ int red_c[kRouteThreads / 32][MAXE];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < E * H; i += blockDim.x) w_s[i] = to_f32(Wr[i]);
  __syncthreads();

  constexpr int kWarps = kRouteThreads / 32;
  constexpr int kPerWarp = kRouteTokensPerBlock / kWarps;
  // lane e keeps the running sums of expert e (and e + 32 when E > 32)
  float psum0 = 0.f, psum1 = 0.f;
  int cnt0 = 0, cnt1 = 0;

  for (int j = 0; j < kPerWarp; ++j) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kRouteTokensPerBlock + warp * kPerWarp + j;
    if (t >= T) break;   // uniform across the warp
    float acc[MAXE];
#pragma unroll
    for (int e = 0; e < MAXE; ++e) acc[e] = 0.f;
    const Tin* xr = x + t * H;
    for (int h = lane * 8; h < H; h += 256) {
      float xv[8];
      load_vec8(xr + h, xv);
#pragma unroll
      for (int e = 0; e < MAXE; ++e) {
        if (e < E) {
          const float* w = w_s + e * H + h;
          float s = acc[e];
#pragma unroll
          for (int i = 0; i < 8; ++i) s = fmaf(xv[i], w[i], s);
          acc[e] = s;
        }
      }
    }
    float r[MAXE];
    float m = -INFINITY;
#pragma unroll
    for (int e = 0; e < MAXE; ++e) {
      if (e < E) {
        r[e] = warp_sum(acc[e]) + (bias != nullptr ? bias[e] : 0.f);
        m = fmaxf(m, r[e]);
      }
    }
    float z = 0.f;
#pragma unroll
    for (int e = 0; e < MAXE; ++e) {
      if (e < E) {
        r[e] = expf(r[e] - m);
        z += r[e];
      }
    }
    float p[MAXE];
#pragma unroll
    for (int e = 0; e < MAXE; ++e) p[e] = (e < E) ? r[e] / z : 0.f;

    // top-k by repeated selection; strict '>' keeps the lowest index on ties.
    // Pass 1 finds the set and sum_S p; pass 2 repeats the same selection and
    // writes the slots with alpha = p / (sum_S p + 1e-20).
    uint64_t chosen = 0;
    float sel_sum = 0.f;
    for (int pass = 0; pass < 2; ++pass) {
      uint64_t taken = 0;
      for (int s = 0; s < k; ++s) {
        int best = -1;
        float bp = 0.f;
#pragma unroll
        for (int e = 0; e < MAXE; ++e) {
          if (e < E && !((taken >> e) & 1ull) && (best < 0 || p[e] > bp)) {
            best = e;
            bp = p[e];
          }
        }
        taken |= 1ull << best;
        if (pass == 0) {
          sel_sum += bp;
        } else if (lane == 0) {
          topk_idx[t * k + s] = best;
          topk_w[t * k + s] = bp / (sel_sum + 1e-20f);
        }
      }
      chosen = taken;
    }
#pragma unroll
    for (int e = 0; e < MAXE; ++e) {
      if (e < E) {
        if (e == lane) {
          psum0 += p[e];
          cnt0 += static_cast<int>((chosen >> e) & 1ull);
        } else if (e == lane + 32) {
          psum1 += p[e];
          cnt1 += static_cast<int>((chosen >> e) & 1ull);
        }
      }
    }
  }
  if (lane < E && lane < MAXE) {
    red_p[warp][lane] = psum0;
    red_c[warp][lane] = cnt0;
  }
  if (lane + 32 < E && lane + 32 < MAXE) {
    red_p[warp][lane + 32] = psum1;
    red_c[warp][lane + 32] = cnt1;
  }
  __syncthreads();
  if (tid < E) {
    float ps = 0.f;
    int c = 0;
    for (int w = 0; w < kWarps; ++w) {
      ps += red_p[w][tid];
      c += red_c[w][tid];
    }
    blk_prob[static_cast<int64_t>(blockIdx.x) * E + tid] = ps;
    blk_cnt[static_cast<int64_t>(blockIdx.x) * E + tid] = c;
  }
}

// ---------------------------------------------------------------------------
// Finalisation shared by dispatch (block 0) and the route-only path:
//   count_e = sum_b blk_cnt[b][e];  P_e = sum_b blk_prob[b][e]  (block order, fp64)
//   offsets = exclusive scan of count;  aux = E*coef*sum_e (count_e/T)(P_e/T)
// Runs in one block with >= E threads.
// ---------------------------------------------------------------------------
__device__ void finalize_aux(int E, int nblk, int64_t T, float coef,
                             const int32_t* __restrict__ blk_cnt,
                             const float* __restrict__ blk_prob, int32_t* offsets,
                             int32_t* counts, float* aux_loss, int32_t* counts_out) {
  __shared__ double s_term[MM_MAX_EXPERTS];
  __shared__ int s_cnt[MM_MAX_EXPERTS];
  const int tid = threadIdx.x;
  if (tid < E) {
    int c = 0;
    double P = 0.0;
    for (int b = 0; b < nblk; ++b) {
      c += blk_cnt[static_cast<int64_t>(b) * E + tid];
      P += static_cast<double>(blk_prob[static_cast<int64_t>(b) * E + tid]);
    }
    s_cnt[tid] = c;
    s_term[tid] = (static_cast<double>(c) / static_cast<double>(T)) * (P / static_cast<double>(T));
    if (counts != nullptr) counts[tid] = c;
    if (counts_out != nullptr) counts_out[tid] = c;
  }
  __syncthreads();
  if (tid == 0) {
    double acc = 0.0;
    int run = 0;
    for (int e = 0; e < E; ++e) {
      acc += s_term[e];
      if (offsets != nullptr) offsets[e] = run;
      run += s_cnt[e];
    }
    if (offsets != nullptr) offsets[E] = run;
    if (aux_loss != nullptr)
      *aux_loss = static_cast<float>(static_cast<double>(E) * static_cast<double>(coef) * acc);
  }
  __syncthreads();
}

__global__ void route_finalize_kernel(int E, int nblk, int64_t T, float coef,
                                      const int32_t* __restrict__ blk_cnt,
                                      const float* __restrict__ blk_prob, int32_t* offsets,
                                      int32_t* counts, float* aux_loss, int32_t* counts_out) {
  finalize_aux(E, nblk, T, coef, blk_cnt, blk_prob, offsets, counts, aux_loss, counts_out);
}

// ---------------------------------------------------------------------------
// Dispatch: block b owns the same tokens as router block b.  Each assignment
// (t, s) with expert e = topk_idx[t,s] gets the row
//   pos = offsets[e] + #(assignments to e in blocks < b) + rank within block,
// where the rank follows token order (a token meets an expert at most once),
// so every expert's rows are in ascending token order.  perm[pos] = t*k + s,
// and x[t] is copied to Xp[pos].  Optionally zeroes y[t] (for the k = 2
// accumulation).  Block 0 also writes offsets, counts and the aux loss.
// ---------------------------------------------------------------------------
template <typename Tin>
__global__ void __launch_bounds__(kRouteThreads)
dispatch_kernel(const Tin* __restrict__ x, int64_t T, int H, int E, int k, float coef, int nblk,
                const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ blk_cnt,
                const float* __restrict__ blk_prob, int32_t* __restrict__ offsets,
                int32_t* __restrict__ counts, float* __restrict__ aux_loss,
                int32_t* __restrict__ perm, Tin* __restrict__ Xp, Tin* __restrict__ y_zero) {
  constexpr int kWarps = kRouteThreads / 32;
  __shared__ int s_base[MM_MAX_EXPERTS];
  __shared__ int s_tot[MM_MAX_EXPERTS];
  __shared__ int s_pre[MM_MAX_EXPERTS];
  __shared__ int s_wcnt[kWarps][MM_MAX_EXPERTS];
  __shared__ int s_pos[kRouteTokensPerBlock * MM_MAX_EXPERTS];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  if (b == 0) finalize_aux(E, nblk, T, coef, blk_cnt, blk_prob, offsets, counts, aux_loss, nullptr);

  if (tid < E) {
    int tot = 0, pre = 0;
    for (int bb = 0; bb < nblk; ++bb) {
      const int c = blk_cnt[static_cast<int64_t>(bb) * E + tid];
      tot += c;
      if (bb < b) pre += c;
    }
    s_tot[tid] = tot;
    s_pre[tid] = pre;
  }
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < E; ++e) {
      s_base[e] = run + s_pre[e];
      run += s_tot[e];
    }
  }
  __syncthreads();

  const int64_t tok0 = static_cast<int64_t>(b) * kRouteTokensPerBlock;
  const int ntok = static_cast<int>((T - tok0) < kRouteTokensPerBlock ? (T - tok0) : kRouteTokensPerBlock);
  const int nA = ntok * k;
  for (int c0 = 0; c0 < nA; c0 += kRouteThreads) {
    for (int i = tid; i < kWarps * E; i += kRouteThreads) (&s_wcnt[0][0])[(i / E) * MM_MAX_EXPERTS + (i % E)] = 0;
    __syncthreads();
    const int a = c0 + tid;
    const bool valid = a < nA;
    const int e = valid ? topk_idx[tok0 * k + a] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (valid && lane == __ffs(peers) - 1) s_wcnt[warp][e] = __popc(peers);
    __syncthreads();
    if (valid) {
      int pre = 0;
      for (int w = 0; w < warp; ++w) pre += s_wcnt[w][e];
      const int pos = s_base[e] + pre + rank;
      perm[pos] = static_cast<int32_t>(tok0 * k + a);
      s_pos[a] = pos;
    }
    __syncthreads();
    if (tid < E) {
      int add = 0;
      for (int w = 0; w < kWarps; ++w) add += s_wcnt[w][tid];
      s_base[tid] += add;
    }
    __syncthreads();
  }

  // copy rows: one warp per assignment, 16-byte vectors
  constexpr int kVec = 16 / sizeof(Tin);
  const int nv = H / kVec;
  for (int a = warp; a < nA; a += kWarps) {
    const int64_t t = tok0 + a / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
    uint4* dst = reinterpret_cast<uint4*>(Xp + static_cast<int64_t>(s_pos[a]) * H);
    for (int v = lane; v < nv; v += 32) dst[v] = src[v];
  }
  if (y_zero != nullptr) {
    const uint4 zero = make_uint4(0, 0, 0, 0);
    for (int tl = warp; tl < ntok; tl += kWarps) {
      uint4* dst = reinterpret_cast<uint4*>(y_zero + (tok0 + tl) * H);
      for (int v = lane; v < nv; v += 32) dst[v] = zero;
    }
  }
}

// ---------------------------------------------------------------------------
// Ordered combine for k >= 3: y[t] = 0; for the slots of t in ascending
// expert index: y[t] = round_to_dtype(y[t] + contribution) — the pages'
// index_add_ into y, expert by expert.
// ---------------------------------------------------------------------------
template <typename Tout>
__global__ void combine_ordered_kernel(const Tout* __restrict__ slots, const int32_t* __restrict__ topk_idx,
                                       int64_t T, int H, int k, Tout* __restrict__ y) {
  const int64_t t = blockIdx.x;
  if (t >= T) return;
  __shared__ int order[MM_MAX_EXPERTS];
  if (threadIdx.x == 0) {
    // selection sort of the k slots by expert index (k <= 64)
    uint64_t used = 0;
    for (int i = 0; i < k; ++i) {
      int best = -1, be = 0;
      for (int s = 0; s < k; ++s) {
        const int e = topk_idx[t * k + s];
        if (!((used >> s) & 1ull) && (best < 0 || e < be)) {
          best = s;
          be = e;
        }
      }
      used |= 1ull << best;
      order[i] = best;
    }
  }
  __syncthreads();
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    Tout acc = static_cast<Tout>(0.f);
    for (int i = 0; i < k; ++i) {
      const Tout c = slots[(t * k + order[i]) * H + h];
      acc = static_cast<Tout>(to_f32(acc) + to_f32(c));
    }
    y[t * H + h] = acc;
  }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
template <typename Tin>
static cudaError_t launch_router_t(const void* x, const void* Wr, const float* bias, int64_t T, int H,
                                   int E, int k, int32_t* topk_idx, float* topk_w, int32_t* blk_cnt,
                                   float* blk_prob, cudaStream_t st) {
  const int nblk = static_cast<int>((T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock);
  const size_t smem = static_cast<size_t>(E) * H * sizeof(float);
#define MM_ROUTER_CASE(ME)                                                                     \
  {                                                                                            \
    auto fn = router_kernel<Tin, ME>;                                                          \
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,   \
                                           static_cast<int>(smem));                            \
    if (err != cudaSuccess) return err;                                                        \
    fn<<<nblk, kRouteThreads, smem, st>>>(static_cast<const Tin*>(x),                          \
                                          static_cast<const Tin*>(Wr), bias, T, H, E, k,        \
                                          topk_idx, topk_w, blk_cnt, blk_prob);                \
    return cudaGetLastError();                                                                 \
  }
  if (E <= 8) MM_ROUTER_CASE(8)
  if (E <= 16) MM_ROUTER_CASE(16)
  if (E <= 32) MM_ROUTER_CASE(32)
  MM_ROUTER_CASE(64)
#undef MM_ROUTER_CASE
}

cudaError_t launch_router(int dtype, const void* x, const void* Wr, const float* bias, int64_t T,
                          int H, int E, int k, int32_t* topk_idx, float* topk_w, int32_t* blk_cnt,
                          float* blk_prob, cudaStream_t st) {
  if (dtype == kDtypeBF16)
    return launch_router_t<__nv_bfloat16>(x, Wr, bias, T, H, E, k, topk_idx, topk_w, blk_cnt,
                                          blk_prob, st);
  return launch_router_t<float>(x, Wr, bias, T, H, E, k, topk_idx, topk_w, blk_cnt, blk_prob, st);
}

cudaError_t launch_route_finalize(int E, int nblk, int64_t T, float coef, const int32_t* blk_cnt,
                                  const float* blk_prob, int32_t* offsets, int32_t* counts,
                                  float* aux_loss, int32_t* counts_out, cudaStream_t st) {
  route_finalize_kernel<<<1, 64, 0, st>>>(E, nblk, T, coef, blk_cnt, blk_prob, offsets, counts,
                                          aux_loss, counts_out);
  return cudaGetLastError();
}

cudaError_t launch_dispatch(int dtype, const void* x, int64_t T, int H, int E, int k, float coef,
                            const int32_t* topk_idx, const int32_t* blk_cnt, const float* blk_prob,
                            int32_t* offsets, int32_t* counts, float* aux_loss, int32_t* perm,
                            void* Xp, void* y_zero, cudaStream_t st) {
  const int nblk = static_cast<int>((T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock);
  if (dtype == kDtypeBF16) {
    dispatch_kernel<__nv_bfloat16><<<nblk, kRouteThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), T, H, E, k, coef, nblk, topk_idx, blk_cnt, blk_prob,
        offsets, counts, aux_loss, perm, static_cast<__nv_bfloat16*>(Xp),
        static_cast<__nv_bfloat16*>(y_zero));
  } else {
    dispatch_kernel<float><<<nblk, kRouteThreads, 0, st>>>(
        static_cast<const float*>(x), T, H, E, k, coef, nblk, topk_idx, blk_cnt, blk_prob, offsets,
        counts, aux_loss, perm, static_cast<float*>(Xp), static_cast<float*>(y_zero));
  }
  return cudaGetLastError();
}

cudaError_t launch_combine_ordered(int dtype, const void* slots, const int32_t* topk_idx, int64_t T,
                                   int H, int k, void* y, cudaStream_t st) {
  if (dtype == kDtypeBF16) {
    combine_ordered_kernel<__nv_bfloat16><<<static_cast<unsigned>(T), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(slots), topk_idx, T, H, k, static_cast<__nv_bfloat16*>(y));
  } else {
    combine_ordered_kernel<float><<<static_cast<unsigned>(T), 256, 0, st>>>(
        static_cast<const float*>(slots), topk_idx, T, H, k, static_cast<float*>(y));
  }
  return cudaGetLastError();
}

}  // namespace mm
