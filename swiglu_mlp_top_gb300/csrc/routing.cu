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
// Router ([L13] §1.5 equations; chapter 4 §4.3 steps 1-2).  A warp routes
// TPW = 32 / EP tokens per pass (EP = E rounded up to 8, 16, 32 or 64):
//   r_{t,e} = sum_h x[t,h] Wr[e,h] (+ bias_e)   fp32; lanes split h into
//             8-element chunks and hold TPW x EP partial sums, which a
//             butterfly reduce-scatter (5 shuffle rounds) leaves as one
//             (token, expert) logit per lane;
//   p = softmax(r)                              fp32, max subtracted, within
//                                               the token's lane group;
//   S = k largest p, equal p -> lower index     k group-wide arg-max rounds;
//   alpha_s = p_S[s] / (sum_S p + 1e-20).
// Per block it also records, for every (slot s, expert e) group g = s*E + e,
// how many of its tokens chose e in slot s (blk_cnt[b][g]), and sum_t p_{t,e}
// over its tokens (blk_prob[b][e]); every sum runs in a fixed order.
// ---------------------------------------------------------------------------
template <typename Tin, int EP>
__global__ void __launch_bounds__(kRouteThreads)
router_kernel(const Tin* __restrict__ x, const Tin* __restrict__ Wr, const float* __restrict__ bias,
              int64_t T, int H, int E, int k, int32_t* __restrict__ topk_idx,
              float* __restrict__ topk_w, int32_t* __restrict__ blk_cnt,
              float* __restrict__ blk_prob) {
  constexpr int R = (EP > 32) ? EP / 32 : 1;      // values per lane after the reduction
  constexpr int NV = 32 * R;                       // partial sums per lane
  constexpr int TPW = NV / EP;                     // tokens per pass
  constexpr int GL = (EP < 32) ? EP : 32;          // lanes per token group
  constexpr int kWarps = kRouteThreads / 32;
  constexpr int kPerWarp = kRouteTokensPerBlock / kWarps;
  static_assert(kPerWarp % TPW == 0, "passes cover a warp's tokens");

  extern __shared__ float4 route_smem4[];
  const int nch = H / 8;                           // 8-element chunks per row
  float4* w_lo = route_smem4;                      // [E][nch] elements 0..3 of each chunk
  float4* w_hi = route_smem4 + E * nch;            // [E][nch] elements 4..7
  int* s_gcnt = reinterpret_cast<int*>(route_smem4 + 2 * E * nch);   // [k*E]
  __shared__ float red_p[kWarps][EP];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = k * E;
  for (int i = tid; i < E * nch; i += blockDim.x) {
    const int e = i / nch, c = i - e * nch;
    float v[8];
    load_vec8(Wr + static_cast<int64_t>(e) * H + c * 8, v);
    w_lo[i] = make_float4(v[0], v[1], v[2], v[3]);
    w_hi[i] = make_float4(v[4], v[5], v[6], v[7]);
  }
  for (int i = tid; i < G; i += blockDim.x) s_gcnt[i] = 0;
  __syncthreads();

  // (token, expert) pairs this lane owns after the reduction
  int e_of[R];
  const int t_loc = (R == 1) ? lane / EP : 0;
  const int gbase = t_loc * GL;
#pragma unroll
  for (int j = 0; j < R; ++j) e_of[j] = (R == 1) ? (lane % EP) : (lane + 32 * j);
  float bias_v[R];
#pragma unroll
  for (int j = 0; j < R; ++j) bias_v[j] = (bias != nullptr && e_of[j] < E) ? bias[e_of[j]] : 0.f;
  float psum[R];
#pragma unroll
  for (int j = 0; j < R; ++j) psum[j] = 0.f;

  for (int pass = 0; pass < kPerWarp / TPW; ++pass) {
    const int64_t tbase = static_cast<int64_t>(blockIdx.x) * kRouteTokensPerBlock +
                          warp * kPerWarp + pass * TPW;
    if (tbase >= T) break;   // uniform across the warp
    float v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = 0.f;
    for (int c = lane; c < nch; c += 32) {
      float xv[TPW][8];
#pragma unroll
      for (int t = 0; t < TPW; ++t) {
        if (tbase + t < T) {
          load_vec8(x + (tbase + t) * H + c * 8, xv[t]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) xv[t][i] = 0.f;
        }
      }
#pragma unroll
      for (int e = 0; e < EP; ++e) {
        if (e < E) {
          const float4 a = w_lo[e * nch + c], b = w_hi[e * nch + c];
#pragma unroll
          for (int t = 0; t < TPW; ++t) {
            float s = v[t * EP + e];
            s = fmaf(xv[t][0], a.x, s); s = fmaf(xv[t][1], a.y, s);
            s = fmaf(xv[t][2], a.z, s); s = fmaf(xv[t][3], a.w, s);
            s = fmaf(xv[t][4], b.x, s); s = fmaf(xv[t][5], b.y, s);
            s = fmaf(xv[t][6], b.z, s); s = fmaf(xv[t][7], b.w, s);
            v[t * EP + e] = s;
          }
        }
      }
    }
    // butterfly reduce-scatter: after the round with offset o a lane keeps the
    // half of its values whose index bit o matches its own lane bit; at the
    // end lane L holds the full sums of pairs L + 32 j
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int j = 0; j < R; ++j) {
#pragma unroll
        for (int i = 0; i < o; ++i) {
          const float lo = v[j * 32 + i], hi = v[j * 32 + i + o];
          const float send = up ? lo : hi;
          const float keep = up ? hi : lo;
          v[j * 32 + i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
    }
    const int64_t tok = tbase + t_loc;
    const bool valid = tok < T;
    float r[R];
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      r[j] = (e_of[j] < E) ? v[j * 32] + bias_v[j] : -INFINITY;
      m = fmaxf(m, r[j]);
    }
#pragma unroll
    for (int o = GL / 2; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      r[j] = (e_of[j] < E) ? expf(r[j] - m) : 0.f;
      z += r[j];
    }
#pragma unroll
    for (int o = GL / 2; o >= 1; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    float p[R];
#pragma unroll
    for (int j = 0; j < R; ++j) p[j] = r[j] / z;

    // top-k: k rounds of a group-wide arg-max over (p desc, index asc)
    float sel_p[MM_MAX_TOPK];
    int sel_e[MM_MAX_TOPK];
    unsigned taken = 0;
    float sel_sum = 0.f;
#pragma unroll
    for (int s = 0; s < MM_MAX_TOPK; ++s) {
      sel_p[s] = 0.f;
      sel_e[s] = 0;
      if (s < k) {
        float bp = -1.f;
        int be = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < R; ++j) {
          if (!((taken >> j) & 1u) && e_of[j] < E && (p[j] > bp || (p[j] == bp && e_of[j] < be))) {
            bp = p[j];
            be = e_of[j];
          }
        }
#pragma unroll
        for (int o = GL / 2; o >= 1; o >>= 1) {
          const float op = __shfl_xor_sync(0xffffffffu, bp, o);
          const int oe = __shfl_xor_sync(0xffffffffu, be, o);
          if (op > bp || (op == bp && oe < be)) {
            bp = op;
            be = oe;
          }
        }
        sel_p[s] = bp;
        sel_e[s] = be;
        sel_sum += bp;
#pragma unroll
        for (int j = 0; j < R; ++j)
          if (e_of[j] == be) taken |= 1u << j;
      }
    }
    const int slot = lane - gbase;
    if (valid && slot < k) {
      int we = 0;
      float wp = 0.f;
#pragma unroll
      for (int s = 0; s < MM_MAX_TOPK; ++s)
        if (s == slot) {
          we = sel_e[s];
          wp = sel_p[s];
        }
      topk_idx[tok * k + slot] = we;
      topk_w[tok * k + slot] = wp / (sel_sum + 1e-20f);
      atomicAdd(&s_gcnt[slot * E + we], 1);
    }
#pragma unroll
    for (int j = 0; j < R; ++j)
      if (valid) psum[j] += p[j];
  }
  // sum the token groups of the warp (lanes with the same expert), fixed order
#pragma unroll
  for (int o = GL; o < 32; o <<= 1) {
#pragma unroll
    for (int j = 0; j < R; ++j) psum[j] += __shfl_xor_sync(0xffffffffu, psum[j], o);
  }
  if (lane < GL) {
#pragma unroll
    for (int j = 0; j < R; ++j)
      if (e_of[j] < EP) red_p[warp][e_of[j]] = psum[j];
  }
  __syncthreads();
  if (tid < E) {
    float ps = 0.f;
    for (int w = 0; w < kWarps; ++w) ps += red_p[w][tid];
    blk_prob[static_cast<int64_t>(blockIdx.x) * E + tid] = ps;
  }
  for (int g = tid; g < G; g += blockDim.x)
    blk_cnt[static_cast<int64_t>(blockIdx.x) * G + g] = s_gcnt[g];
}

// ---------------------------------------------------------------------------
// Scan (one block): for every group g = s*E + e
//   blk_base[b][g] = sum_{b' < b} blk_cnt[b'][g]    (a lane owns a run of blocks)
//   tot[g] = sum_b blk_cnt[b][g];  offsets = exclusive scan of tot over g
// and the aux loss ([L13] §1.6; chapter 4 §4.4):
//   count_e = sum_s tot[s*E + e];  P_e = sum_b blk_prob[b][e]  (fixed order)
//   aux = E * coef * sum_e (count_e / T) * (P_e / T)
// Rows of the dispatched matrix are thus ordered by slot, then expert, then
// token.  offsets / blk_base may be null (route-only call).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kScanThreads)
route_scan_kernel(int E, int k, int nblk, int64_t T, float coef,
                  const int32_t* __restrict__ blk_cnt, const float* __restrict__ blk_prob,
                  int32_t* __restrict__ blk_base, int32_t* __restrict__ offsets,
                  int32_t* __restrict__ counts, float* __restrict__ aux_loss) {
  __shared__ int s_tot[kMaxGroups];
  __shared__ float s_P[MM_MAX_EXPERTS];
  __shared__ int s_cnt[MM_MAX_EXPERTS];
  const int G = k * E;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kScanThreads / 32;
  const int per = (nblk + 31) / 32;

  for (int g = warp; g < G; g += kWarps) {
    const int b0 = lane * per;
    const int b1 = min(nblk, b0 + per);
    int sum = 0;
#pragma unroll 8
    for (int b = b0; b < b1; ++b) sum += blk_cnt[static_cast<int64_t>(b) * G + g];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (blk_base != nullptr) {
      int run = incl - sum;
      for (int b = b0; b < b1; ++b) {
        const int64_t i = static_cast<int64_t>(b) * G + g;
        blk_base[i] = run;
        run += blk_cnt[i];
      }
    }
    const int tot = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) s_tot[g] = tot;
  }
  for (int e = warp; e < E; e += kWarps) {
    // lane-strided partial sums, then a fixed xor-tree: the order depends only on nblk
    float P = 0.f;
#pragma unroll 8
    for (int b = lane; b < nblk; b += 32) P += blk_prob[static_cast<int64_t>(b) * E + e];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) P += __shfl_xor_sync(0xffffffffu, P, o);
    if (lane == 0) s_P[e] = P;
  }
  __syncthreads();
  if (threadIdx.x < E) {
    int c = 0;
    for (int s = 0; s < k; ++s) c += s_tot[s * E + threadIdx.x];
    s_cnt[threadIdx.x] = c;
    if (counts != nullptr) counts[threadIdx.x] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (offsets != nullptr) {
      int run = 0;
      for (int g = 0; g < G; ++g) {
        offsets[g] = run;
        run += s_tot[g];
      }
      offsets[G] = run;
    }
    // E*coef*sum_e (count_e/T)(P_e/T) = (E*coef/T^2) * sum_e count_e * P_e
    float acc = 0.f;
    for (int e = 0; e < E; ++e) acc = fmaf(static_cast<float>(s_cnt[e]), s_P[e], acc);
    const float invT = 1.0f / static_cast<float>(T);
    if (aux_loss != nullptr) *aux_loss = static_cast<float>(E) * coef * acc * invT * invT;
  }
}

// ---------------------------------------------------------------------------
// Dispatch: block b owns the same tokens as router block b.  Assignment
// (t, s) with expert e goes to group g = s*E + e and gets the row
//   pos = offsets[g] + blk_base[b][g] + rank of t among the block's tokens
//         that chose e in slot s (token order),
// so every group's rows are in ascending token order.  perm[pos] = t*k + s,
// and x[t] is copied to Xp[pos].
// ---------------------------------------------------------------------------
template <typename Tin>
__global__ void __launch_bounds__(kRouteThreads)
dispatch_kernel(const Tin* __restrict__ x, int64_t T, int H, int E, int k,
                const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ blk_base,
                const int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                Tin* __restrict__ Xp) {
  __shared__ int s_w0cnt[MM_MAX_EXPERTS];   // per-expert count in warp 0 (tokens 0..31)
  __shared__ int s_pos[kRouteTokensPerBlock * MM_MAX_EXPERTS];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  const int G = k * E;
  const int64_t tok0 = static_cast<int64_t>(b) * kRouteTokensPerBlock;
  const int ntok = static_cast<int>((T - tok0) < kRouteTokensPerBlock ? (T - tok0) : kRouteTokensPerBlock);
  static_assert(kRouteTokensPerBlock == 64, "two ranking warps cover one slot of a block");

  for (int s = 0; s < k; ++s) {
    for (int i = tid; i < E; i += kRouteThreads) s_w0cnt[i] = 0;
    __syncthreads();
    int e = -1, rank = 0;
    if (warp < 2) {
      const int tl = warp * 32 + lane;
      e = (tl < ntok) ? topk_idx[(tok0 + tl) * k + s] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      rank = __popc(peers & ((1u << lane) - 1u));
      if (warp == 0 && e >= 0 && lane == __ffs(peers) - 1) s_w0cnt[e] = __popc(peers);
    }
    __syncthreads();
    if (warp < 2 && e >= 0) {
      const int tl = warp * 32 + lane;
      const int g = s * E + e;
      const int pos = offsets[g] + blk_base[static_cast<int64_t>(b) * G + g] +
                      (warp == 1 ? s_w0cnt[e] : 0) + rank;
      perm[pos] = static_cast<int32_t>((tok0 + tl) * k + s);
      s_pos[tl * k + s] = pos;
    }
    __syncthreads();
  }

  // copy rows: a flat loop over (assignment, 16-byte vector) pairs
  constexpr int kVec = 16 / sizeof(Tin);
  const int nv = H / kVec;
  const int total = ntok * k * nv;
  const uint4* src = reinterpret_cast<const uint4*>(x + tok0 * H);
  uint4* dst = reinterpret_cast<uint4*>(Xp);
#pragma unroll 4
  for (int i = tid; i < total; i += kRouteThreads) {
    const int a = i / nv;
    const int v = i - a * nv;
    dst[static_cast<int64_t>(s_pos[a]) * nv + v] = src[(a / k) * nv + v];
  }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
size_t router_smem_bytes(int H, int E, int k) {
  return static_cast<size_t>(E) * H * sizeof(float) + static_cast<size_t>(k) * E * sizeof(int);
}

template <typename Tin>
static cudaError_t launch_router_t(const void* x, const void* Wr, const float* bias, int64_t T, int H,
                                   int E, int k, int32_t* topk_idx, float* topk_w, int32_t* blk_cnt,
                                   float* blk_prob, cudaStream_t st) {
  const int nblk = static_cast<int>((T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock);
  const size_t smem = router_smem_bytes(H, E, k);
#define MM_ROUTER_CASE(EPAD)                                                                   \
  {                                                                                            \
    auto fn = router_kernel<Tin, EPAD>;                                                        \
    cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), smem);             \
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

cudaError_t launch_route_scan(int E, int k, int64_t T, float coef, const int32_t* blk_cnt,
                              const float* blk_prob, int32_t* blk_base, int32_t* offsets,
                              int32_t* counts, float* aux_loss, cudaStream_t st) {
  const int nblk = static_cast<int>((T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock);
  route_scan_kernel<<<1, kScanThreads, 0, st>>>(E, k, nblk, T, coef, blk_cnt, blk_prob, blk_base,
                                                offsets, counts, aux_loss);
  return cudaGetLastError();
}

cudaError_t launch_dispatch(int dtype, const void* x, int64_t T, int H, int E, int k,
                            const int32_t* topk_idx, const int32_t* blk_base,
                            const int32_t* offsets, int32_t* perm, void* Xp, cudaStream_t st) {
  const int nblk = static_cast<int>((T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock);
  if (dtype == kDtypeBF16) {
    dispatch_kernel<__nv_bfloat16><<<nblk, kRouteThreads, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), T, H, E, k, topk_idx, blk_base, offsets, perm,
        static_cast<__nv_bfloat16*>(Xp));
  } else {
    dispatch_kernel<float><<<nblk, kRouteThreads, 0, st>>>(
        static_cast<const float*>(x), T, H, E, k, topk_idx, blk_base, offsets, perm,
        static_cast<float*>(Xp));
  }
  return cudaGetLastError();
}

}  // namespace mm
