// Router (logits, softmax, top-k, renormalisation, aux partials), the
// dispatch of tokens into expert-contiguous rows, the aux-loss finalisation
// and the ordered combine used when k >= 3.
//
// Follows MiniMind lesson 13 "FFN 与 MoE" §1.5 (router equations), §1.6 and
// step 6 (aux loss), step 4-5 (top-k, renormalisation, per-expert dispatch
// and index_add_ into y), and minimind3.com chapter 4 §4.3-§4.4.
#include <algorithm>
#include <cstring>
#include <mutex>

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

// 8 consecutive elements as four packed fp32 pairs (element 2i in the low word).
template <typename Tin>
__device__ __forceinline__ void load_pairs8(const Tin* p, u64 (&q)[4]);
template <>
__device__ __forceinline__ void load_pairs8<__nv_bfloat16>(const __nv_bfloat16* p, u64 (&q)[4]) {
  const uint4 raw = *reinterpret_cast<const uint4*>(p);
  q[0] = bf2(raw.x); q[1] = bf2(raw.y); q[2] = bf2(raw.z); q[3] = bf2(raw.w);
}
template <>
__device__ __forceinline__ void load_pairs8<float>(const float* p, u64 (&q)[4]) {
  const ulonglong2 a = *reinterpret_cast<const ulonglong2*>(p);
  const ulonglong2 b = *reinterpret_cast<const ulonglong2*>(p + 4);
  q[0] = a.x; q[1] = a.y; q[2] = b.x; q[3] = b.y;
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
__device__ void scan_block(int E, int k, int nblk, int64_t T, const RouteExtras& X,
                           const int32_t* __restrict__ blk_cnt, const float* __restrict__ blk_prob);

// z-loss = z_coef * (1/T) * sum_t lse_t^2 from the router blocks' sums of
// lse^2, by one warp: lane-strided partial sums over the blocks, then a
// fixed xor tree (the order depends only on nblk).
__device__ __forceinline__ void finalize_z_loss(const RouterVariant& rv, int nblk, int64_t T,
                                                int lane) {
  float zs = 0.f;
#pragma unroll 8
  for (int b = lane; b < nblk; b += 32) zs += __ldcg(rv.blk_z + b);
  zs = warp_sum(zs);
  if (lane == 0) *rv.z_loss = rv.z_coef * zs / static_cast<float>(T);
}

template <typename Tin, int EP>
__global__ void __launch_bounds__(kRouteThreads)
router_kernel(const Tin* __restrict__ x, const Tin* __restrict__ Wr, const float* __restrict__ bias,
              int64_t T, int H, int E, int k, int32_t* __restrict__ topk_idx,
              float* __restrict__ topk_w, int32_t* __restrict__ blk_cnt,
              float* __restrict__ blk_prob, const RouteExtras X) {

  constexpr int R = (EP > 32) ? EP / 32 : 1;      // values per lane after the reduction
  constexpr int NV = 32 * R;                       // partial sums per lane
  constexpr int TPW = NV / EP;                     // tokens per pass
  constexpr int GL = (EP < 32) ? EP : 32;          // lanes per token group
  constexpr int kWarps = kRouteThreads / 32;
  constexpr int kPerWarp = kRouteTokensPerBlock / kWarps;
  static_assert(kPerWarp % TPW == 0, "passes cover a warp's tokens");

  // the dispatch kernel may launch as soon as router blocks start to leave
  // (it waits for this grid before reading the routing results)
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int rblk = blockIdx.x;                     // router block: tokens [64 rblk, +64)
  const int nblk = static_cast<int>((T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock);

  extern __shared__ float4 route_smem4[];
  const int nch = H / 8;                           // 8-element chunks per row
  // Wr [E][H] as stored, then the group counters; x rows at X.x_off
  Tin* wsm = reinterpret_cast<Tin*>(route_smem4);
  int* s_gcnt = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(route_smem4) +
                                       static_cast<size_t>(E) * H * sizeof(Tin));   // [k*E]
  __shared__ float red_p[kWarps][EP];
  __shared__ float red_z[kWarps];
  __shared__ __align__(8) uint64_t xbar;
  __shared__ int s_last;
  const RouterVariant& rv = X.rv;
  const Tin* norm_w = static_cast<const Tin*>(X.norm.w);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = k * E;
  // Wr and (when X.stage_x) this block's x rows come into shared memory by
  // bulk copies
  const int64_t t0 = static_cast<int64_t>(rblk) * kRouteTokensPerBlock;
  const int ntok = static_cast<int>(T - t0 < kRouteTokensPerBlock ? T - t0 : kRouteTokensPerBlock);
  const Tin* xsrc = x + t0 * H;                    // row t of the block at xsrc + t * H
  Tin* xs = reinterpret_cast<Tin*>(reinterpret_cast<unsigned char*>(route_smem4) + X.x_off);
  if (tid == 0) {
    mbar_init(&xbar, 1);
    fence_mbar_init();
    const uint32_t wbytes = static_cast<uint32_t>(E) * H * sizeof(Tin);
    const uint32_t xbytes = X.stage_x ? static_cast<uint32_t>(ntok) * H * sizeof(Tin) : 0u;
    mbar_arrive_expect_tx(&xbar, wbytes + xbytes);
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(wsm)), "l"(Wr), "r"(wbytes), "r"(smem_u32(&xbar))
        : "memory");
    if (xbytes)
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
          ::"r"(smem_u32(xs)), "l"(xsrc), "r"(xbytes), "r"(smem_u32(&xbar))
          : "memory");
  }
  if (X.stage_x) xsrc = xs;

  for (int i = tid; i < G; i += blockDim.x) s_gcnt[i] = 0;
  __syncthreads();
  if (!__syncthreads_and(mbar_wait(&xbar, 0, nullptr, X.hdr, 60))) return;

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
  float zsum = 0.f;                                // lse^2 of the lane group's tokens (slot-0 lane)

  for (int pass = 0; pass < kPerWarp / TPW; ++pass) {
    const int lbase = warp * kPerWarp + pass * TPW;      // token within the block
    const int64_t tbase = t0 + lbase;
    if (tbase >= T) break;   // uniform across the warp
    // packed fp32 partial sums (even / odd elements), folded before the reduction
    u64 acc[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) acc[i] = 0ull;
    u64 ss2[TPW];                                  // block norm: sums of x^2 per token
#pragma unroll
    for (int t = 0; t < TPW; ++t) ss2[t] = 0ull;
    for (int c = lane; c < nch; c += 32) {
      u64 xv[TPW][4];
#pragma unroll
      for (int t = 0; t < TPW; ++t) {
        if (tbase + t < T) {
          load_pairs8(xsrc + static_cast<int64_t>(lbase + t) * H + c * 8, xv[t]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) xv[t][i] = 0ull;
        }
      }
      if (norm_w != nullptr) {
        // x_h^2 for the norm, then x_h * w_h (exact in fp32 for bf16)
        u64 wv[4];
        load_pairs8(norm_w + c * 8, wv);
#pragma unroll
        for (int t = 0; t < TPW; ++t)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            ss2[t] = ffma2(xv[t][q], xv[t][q], ss2[t]);
            xv[t][q] = ffma2(xv[t][q], wv[q], 0ull);
          }
      }
#pragma unroll
      for (int e = 0; e < EP; ++e) {
        if (e < E) {
          u64 wv[4];
          load_pairs8(wsm + static_cast<int64_t>(e) * H + c * 8, wv);
#pragma unroll
          for (int t = 0; t < TPW; ++t) {
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[t * EP + e] = ffma2(xv[t][q], wv[q], acc[t * EP + e]);
          }
        }
      }
    }
    float v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = hsum2(acc[i]);
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
    float inv = 1.0f;
    if (norm_w != nullptr) {
      // this lane's token: its sum of squares over all lanes, in a fixed order
      float ssv = 0.f;
#pragma unroll
      for (int t = 0; t < TPW; ++t) {
        const float w = warp_sum(hsum2(ss2[t]));
        if (t == t_loc) ssv = w;
      }
      inv = 1.0f / sqrtf(ssv / static_cast<float>(H) + X.norm.eps);
      if (valid && lane == gbase) X.norm.inv_rms[tok] = inv;
    }
    float r[R];
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      r[j] = (e_of[j] < E) ? inv * v[j * 32] + bias_v[j] : -INFINITY;
      if (rv.noise != nullptr && valid && e_of[j] < E) r[j] += rv.noise[tok * E + e_of[j]];
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
    const float lse = m + logf(z);
    if (valid) {
      if (rv.probs != nullptr) {
#pragma unroll
        for (int j = 0; j < R; ++j)
          if (e_of[j] < E) rv.probs[tok * E + e_of[j]] = p[j];
      }
      if (lane == gbase) {
        if (rv.lse != nullptr) rv.lse[tok] = lse;
        zsum = fmaf(lse, lse, zsum);
      }
    }

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
  zsum = warp_sum(zsum);
  if (lane == 0) red_z[warp] = zsum;
  __syncthreads();
  if (tid < E) {
    float ps = 0.f;
    for (int w = 0; w < kWarps; ++w) ps += red_p[w][tid];
    blk_prob[static_cast<int64_t>(rblk) * E + tid] = ps;
  }
  if (tid == 0 && rv.blk_z != nullptr) {
    float zs = 0.f;
    for (int w = 0; w < kWarps; ++w) zs += red_z[w];
    rv.blk_z[rblk] = zs;
  }
  for (int g = tid; g < G; g += blockDim.x)
    blk_cnt[static_cast<int64_t>(rblk) * G + g] = s_gcnt[g];

  // route-only calls: the router block that finishes last runs the scan
  // (partials, fence, count: whoever brings the count to nblk sees every
  // block's partials); it resets the counter for the next launch.  The MoE
  // forward leaves this to the dispatch kernel.
  if (!X.do_scan) return;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&X.hdr->route_done, 1u) == static_cast<unsigned>(nblk - 1));
  __syncthreads();
  if (s_last) {
    __threadfence();
    scan_block(E, k, nblk, T, X, blk_cnt, blk_prob);
    if (tid == 0) X.hdr->route_done = 0u;
  }
}


// ---------------------------------------------------------------------------
// Scan, run by the router block that finishes last: for every group
// g = s*E + e
//   blk_base[b][g] = sum_{b' < b} blk_cnt[b'][g]    (a lane owns a run of blocks)
//   tot[g] = sum_b blk_cnt[b][g];  offsets = exclusive scan of tot over g
// and the aux loss ([L13] §1.6; chapter 4 §4.4):
//   count_e = sum_s tot[s*E + e];  P_e = sum_b blk_prob[b][e]  (fixed order)
//   aux = E * coef * sum_e (count_e / T) * (P_e / T)
// Rows of the dispatched matrix are thus ordered by slot, then expert, then
// token.  offsets / blk_base may be null (route-only call).  The other
// blocks' partials are read through L2 (ld.global.cg).
// ---------------------------------------------------------------------------
__device__ void scan_block(int E, int k, int nblk, int64_t T, const RouteExtras& X,
                           const int32_t* __restrict__ blk_cnt, const float* __restrict__ blk_prob) {
  __shared__ int s_tot[kMaxGroups];
  __shared__ float s_P[MM_MAX_EXPERTS];
  __shared__ int s_cnt[MM_MAX_EXPERTS];
  const int G = k * E;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kRouteThreads / 32;
  const int per = (nblk + 31) / 32;

  for (int g = warp; g < G; g += kWarps) {
    const int b0 = lane * per;
    const int b1 = min(nblk, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; b += 8) {
      int c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        c[j] = (b + j < b1) ? __ldcg(blk_cnt + static_cast<int64_t>(b + j) * G + g) : 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) sum += c[j];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (X.blk_base != nullptr) {
      // every count of a run of 8 is requested before the running sum uses it
      int run = incl - sum;
      for (int b = b0; b < b1; b += 8) {
        int c[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          c[j] = (b + j < b1) ? __ldcg(blk_cnt + static_cast<int64_t>(b + j) * G + g) : 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (b + j < b1) X.blk_base[static_cast<int64_t>(b + j) * G + g] = run;
          run += c[j];
        }
      }
    }
    const int tot = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) s_tot[g] = tot;
  }
  for (int e = warp; e < E; e += kWarps) {
    // lane-strided partial sums, then a fixed xor-tree: the order depends only on nblk
    float P = 0.f;
#pragma unroll 8
    for (int b = lane; b < nblk; b += 32) P += __ldcg(blk_prob + static_cast<int64_t>(b) * E + e);
    P = warp_sum(P);
    if (lane == 0) s_P[e] = P;
  }
  __syncthreads();
  if (threadIdx.x < E) {
    int c = 0;
    for (int s = 0; s < k; ++s) c += s_tot[s * E + threadIdx.x];
    s_cnt[threadIdx.x] = c;
    if (X.counts != nullptr) X.counts[threadIdx.x] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (X.offsets != nullptr) {
      int run = 0;
      for (int g = 0; g < G; ++g) {
        X.offsets[g] = run;
        run += s_tot[g];
      }
      X.offsets[G] = run;
    }
    // E*coef*sum_e (count_e/T)(P_e/T) = (E*coef/T^2) * sum_e count_e * P_e
    float acc = 0.f;
    for (int e = 0; e < E; ++e) acc = fmaf(static_cast<float>(s_cnt[e]), s_P[e], acc);
    const float invT = 1.0f / static_cast<float>(T);
    if (X.aux_loss != nullptr) *X.aux_loss = static_cast<float>(E) * X.coef * acc * invT * invT;
  }
  if (warp == kWarps - 1 && X.rv.z_loss != nullptr)
    finalize_z_loss(X.rv, nblk, T, lane);
}


// Group totals s_tot[g] over the nblk router blocks' counts, the rows of
// each group in router blocks [0, b) (s_base[g]), and the exclusive scan of
// the totals (s_off[0..G]).  Warp w sums a run of router blocks, lane g its
// group (all counts of the run requested at once), then the warps' partial
// sums are added in warp order.  All kRouteThreads threads take part; the
// counts are read through L2 (another block of the grid may have written
// them).
__device__ void group_offsets(const int32_t* __restrict__ blk_cnt, int nblk, int G, int b,
                              int* s_tot, int* s_base, int* s_off, int (*s_part)[32][2]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kRouteThreads / 32;
  {
    const int per = (nblk + kWarps - 1) / kWarps;
    const int b0 = warp * per, b1 = min(nblk, b0 + per);
    for (int g0 = 0; g0 < G; g0 += 32) {
      const int g = g0 + lane;
      int all = 0, before = 0;
      if (g < G) {
        for (int bb = b0; bb < b1; bb += 32) {
          int c[32];                         // one round of requests for a run of 32 blocks
#pragma unroll
          for (int j = 0; j < 32; ++j)
            c[j] = (bb + j < b1) ? __ldcg(blk_cnt + static_cast<int64_t>(bb + j) * G + g) : 0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            all += c[j];
            before += (bb + j < b) ? c[j] : 0;
          }
        }
      }
      __syncthreads();                       // s_part of the previous round is read
      if (g < G) {
        s_part[warp][lane][0] = all;
        s_part[warp][lane][1] = before;
      }
      __syncthreads();
      if (tid < 32 && g0 + tid < G) {
        int a = 0, bf = 0;
        for (int w = 0; w < kWarps; ++w) {
          a += s_part[w][tid][0];
          bf += s_part[w][tid][1];
        }
        s_tot[g0 + tid] = a;
        s_base[g0 + tid] = bf;
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive scan of the group totals: a lane owns a run of groups
    const int gper = (G + 31) / 32;
    const int g0 = lane * gper, g1 = min(G, g0 + gper);
    int sum = 0;
    for (int g = g0; g < g1; ++g) sum += s_tot[g];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int run = incl - sum;
    for (int g = g0; g < g1; ++g) {
      s_off[g] = run;
      run += s_tot[g];
    }
    if (lane == 31) s_off[G] = incl;
  }
  __syncthreads();
}

// What one block of the dispatch writes for the whole call: the group
// offsets, the expert counts, the aux loss ([L13] §1.6; chapter 4 §4.4:
// aux = E*coef*sum_e (count_e/T)(P_e/T), P_e = sum_b blk_prob[b][e] by warp
// e % 8 as lane-strided partial sums over the router blocks and a fixed xor
// tree, then one thread adds count_e * P_e in expert order) and the z-loss.
// All kRouteThreads threads of that block take part.
__device__ void write_route_totals(const DispatchOut& D, const int* s_tot, const int* s_off, int G,
                                   int E, int k, int nblk, const float* __restrict__ blk_prob,
                                   int64_t T) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kRouteThreads / 32;
  for (int g = tid; g <= G; g += kRouteThreads) D.offsets[g] = s_off[g];
  for (int e = tid; e < E; e += kRouteThreads) {
    int c = 0;
    for (int s = 0; s < k; ++s) c += s_tot[s * E + e];
    if (D.counts != nullptr) D.counts[e] = c;
  }
  __shared__ float s_P[MM_MAX_EXPERTS];
  for (int e = warp; e < E; e += kWarps) {
    float P = 0.f;
#pragma unroll 8
    for (int bb = lane; bb < nblk; bb += 32) P += __ldcg(blk_prob + static_cast<int64_t>(bb) * E + e);
    P = warp_sum(P);
    if (lane == 0) s_P[e] = P;
  }
  __syncthreads();
  if (tid == 0) {
    float acc = 0.f;
    for (int e = 0; e < E; ++e) {
      int c = 0;
      for (int s = 0; s < k; ++s) c += s_tot[s * E + e];
      acc = fmaf(static_cast<float>(c), s_P[e], acc);
    }
    const float invT = 1.0f / static_cast<float>(T);
    *D.aux_loss = static_cast<float>(E) * D.coef * acc * invT * invT;
  }
  if (warp == kWarps - 1 && D.rv.z_loss != nullptr) finalize_z_loss(D.rv, nblk, T, lane);
}

// write_route_totals for the last four warps of a block alone (their own
// named barrier), so that the block's other warps can go on meanwhile; the
// same arithmetic in the same order.
__device__ void write_route_totals_w4(const DispatchOut& D, const int* s_tot, const int* s_off,
                                      int G, int E, int k, int nblk,
                                      const float* __restrict__ blk_prob, int64_t T) {
  const int t4 = threadIdx.x - (blockDim.x - 128), lane = threadIdx.x & 31, wi = t4 >> 5;
  for (int g = t4; g <= G; g += 128) D.offsets[g] = s_off[g];
  for (int e = t4; e < E; e += 128) {
    int c = 0;
    for (int s = 0; s < k; ++s) c += s_tot[s * E + e];
    if (D.counts != nullptr) D.counts[e] = c;
  }
  __shared__ float s_P4[MM_MAX_EXPERTS];
  for (int e = wi; e < E; e += 4) {
    float P = 0.f;
#pragma unroll 8
    for (int bb = lane; bb < nblk; bb += 32) P += __ldcg(blk_prob + static_cast<int64_t>(bb) * E + e);
    P = warp_sum(P);
    if (lane == 0) s_P4[e] = P;
  }
  asm volatile("bar.sync 1, 128;" ::: "memory");
  if (t4 == 0) {
    float acc = 0.f;
    for (int e = 0; e < E; ++e) {
      int c = 0;
      for (int s = 0; s < k; ++s) c += s_tot[s * E + e];
      acc = fmaf(static_cast<float>(c), s_P4[e], acc);
    }
    const float invT = 1.0f / static_cast<float>(T);
    *D.aux_loss = static_cast<float>(E) * D.coef * acc * invT * invT;
  }
  if (wi == 3 && D.rv.z_loss != nullptr) finalize_z_loss(D.rv, nblk, T, lane);
}

// ---------------------------------------------------------------------------
// Dispatch: block b owns the same tokens as router block b.  From the
// router's per-block counts it derives, for every (slot s, expert e) group
// g = s*E + e, the rows before its own block (base) and the group totals;
// block 0 also writes the group offsets, the expert counts and the aux loss
// ([L13] §1.6; chapter 4 §4.4: aux = E*coef*sum_e (count_e/T)(P_e/T), with
// P_e = sum_b blk_prob[b][e] in a fixed order).  Assignment (t, s) with
// expert e gets the row
//   pos = offset[g] + base[g] + rank of t among the block's tokens that chose
//         e in slot s (token order),
// so every group's rows are in ascending token order; perm[pos] = t*k + s and
// x[t] is copied to Xp[pos] — staged in shared memory by one bulk copy and
// written back by one bulk copy per row when the block's rows fit.
// ---------------------------------------------------------------------------
template <typename Tin>
__global__ void __launch_bounds__(kRouteThreads)
dispatch_kernel(const Tin* __restrict__ x, int64_t T, int H, int E, int k,
                const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ blk_cnt,
                const float* __restrict__ blk_prob, const DispatchOut D,
                int32_t* __restrict__ perm, Tin* __restrict__ Xp, int stage_x) {
  extern __shared__ __align__(128) unsigned char disp_smem[];
  __shared__ int s_w0cnt[MM_MAX_EXPERTS];   // per-expert count in warp 0 (tokens 0..31)
  __shared__ int s_pos[kRouteTokensPerBlock * MM_MAX_TOPK];
  __shared__ int s_base[kMaxGroups], s_tot[kMaxGroups], s_off[kMaxGroups + 1];
  __shared__ int s_part[kRouteThreads / 32][32][2];
  __shared__ __align__(8) uint64_t xbar;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kRouteThreads / 32;
  const int b = blockIdx.x;
  const int nblk = gridDim.x;
  const int G = k * E;
  const int64_t tok0 = static_cast<int64_t>(b) * kRouteTokensPerBlock;
  const int ntok = static_cast<int>((T - tok0) < kRouteTokensPerBlock ? (T - tok0) : kRouteTokensPerBlock);
  static_assert(kRouteTokensPerBlock == 64, "two ranking warps cover one slot of a block");
  Tin* xs = reinterpret_cast<Tin*>(disp_smem);
  const uint32_t rowb = static_cast<uint32_t>(H) * sizeof(Tin);

  if (tid == 0 && stage_x) {
    mbar_init(&xbar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&xbar, static_cast<uint32_t>(ntok) * rowb);
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(xs)), "l"(x + tok0 * H), "r"(static_cast<uint32_t>(ntok) * rowb),
        "r"(smem_u32(&xbar))
        : "memory");
  }

  // the routing results come from the router grid, launched just before
  // (x is the caller's input and may be read at once)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // this block's selections, requested together with the counts below
  __shared__ int s_sel[kRouteTokensPerBlock * MM_MAX_TOPK];
  for (int a = tid; a < ntok * k; a += kRouteThreads) s_sel[a] = topk_idx[tok0 * k + a];

  group_offsets(blk_cnt, nblk, G, b, s_tot, s_base, s_off, s_part);
  if (b == 0) write_route_totals(D, s_tot, s_off, G, E, k, nblk, blk_prob, T);
  for (int s = 0; s < k; ++s) {
    for (int i = tid; i < E; i += kRouteThreads) s_w0cnt[i] = 0;
    __syncthreads();
    int e = -1, rank = 0;
    if (warp < 2) {
      const int tl = warp * 32 + lane;
      e = (tl < ntok) ? s_sel[tl * k + s] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      rank = __popc(peers & ((1u << lane) - 1u));
      if (warp == 0 && e >= 0 && lane == __ffs(peers) - 1) s_w0cnt[e] = __popc(peers);
    }
    __syncthreads();
    if (warp < 2 && e >= 0) {
      const int tl = warp * 32 + lane;
      const int g = s * E + e;
      const int pos = s_off[g] + s_base[g] + (warp == 1 ? s_w0cnt[e] : 0) + rank;
      perm[pos] = static_cast<int32_t>((tok0 + tl) * k + s);
      s_pos[tl * k + s] = pos;
    }
    __syncthreads();
  }

  const int na = ntok * k;
  const Tin* norm_w = static_cast<const Tin*>(D.norm.w);
  if (Xp == nullptr) return;                   // permute-free: the GEMM gathers x rows itself
  if (stage_x) {
    // one bulk copy per assignment row, shared -> global
    if (!__syncthreads_and(mbar_wait(&xbar, 0, nullptr, D.hdr, 61))) return;
    if (norm_w != nullptr) {
      // block norm: the staged rows become x * inv_rms * w in place, by
      // 8-element chunks (a warp per row at a time)
      const int nch = H / 8;
      for (int tl = warp; tl < ntok; tl += kWarps) {
        const float inv = D.norm.inv_rms[tok0 + tl];
        Tin* row = xs + static_cast<int64_t>(tl) * H;
        for (int c = lane; c < nch; c += 32) {
          float v[8];
          load_vec8(row + c * 8, v);
          float g[8];
          load_vec8(norm_w + c * 8, g);
#pragma unroll
          for (int j = 0; j < 8; ++j) row[c * 8 + j] = static_cast<Tin>(v[j] * inv * g[j]);
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
    }
    if (tid < na) {
      for (int a = tid; a < na; a += kRouteThreads)
        bulk_store(Xp + static_cast<int64_t>(s_pos[a]) * H, xs + static_cast<int64_t>(a / k) * H, rowb);
      bulk_commit();
      bulk_wait_all();
    }
  } else {
    // a warp per row, 16-byte vectors
    constexpr int kVec = 16 / sizeof(Tin);
    const int nv = H / kVec;
    for (int a = warp; a < na; a += kWarps) {
      if (norm_w != nullptr) {
        const Tin* src = x + (tok0 + a / k) * H;
        Tin* dst = Xp + static_cast<int64_t>(s_pos[a]) * H;
        const float inv = D.norm.inv_rms[tok0 + a / k];
        for (int h = lane; h < H; h += 32)
          dst[h] = static_cast<Tin>(to_f32(src[h]) * inv * to_f32(norm_w[h]));
        continue;
      }
      const uint4* src = reinterpret_cast<const uint4*>(x + (tok0 + a / k) * H);
      uint4* dst = reinterpret_cast<uint4*>(Xp + static_cast<int64_t>(s_pos[a]) * H);
#pragma unroll 4
      for (int v = lane; v < nv; v += 32) dst[v] = src[v];
    }
  }
}


// ---------------------------------------------------------------------------
// Router on the tensor cores (bf16, E <= 64): the same outputs as
// router_kernel for one 64-token block per CTA.  L = x Wr^T by tcgen05 (x
// rows as the M operand: 128 rows are read from each x tile, rows past the
// block's 64 land in TMEM lanes that are never read; Wr padded to EP rows as
// N), the x and Wr k-blocks fetched as 3-D TMA boxes of nkb k-blocks through
// a two-stage ring.  Warps 0 and 1 (TMEM lanes 0-63: one token per thread)
// then take softmax, top-k, alpha, the block's group counts and
// probability sums (fixed-order reductions) exactly as router_kernel does.
// ---------------------------------------------------------------------------
// One token's routing from its logits p[0..E) (fp32, as accumulated):
// p += bias (+ noise); p = softmax(p) (max subtracted); lse = logsumexp of
// the biased logits; top-k by k arg-max passes in expert order with a strict
// comparison (equal p -> the lower index first); sel_sum = sum of the k
// selected p.  The tensor-core router and the fused router + dispatch share
// it, so both take the same decisions bit for bit.
template <int EP>
__device__ __forceinline__ void route_token(float (&p)[EP], int E, int k, const float* s_bias,
                                            const float* nz, float& lse,
                                            int (&sel_e)[MM_MAX_TOPK],
                                            float (&sel_p)[MM_MAX_TOPK], float& sel_sum) {
  // loops over the E experts only (E is uniform; the padded columns past
  // E are never read)
  float m = -INFINITY;
#pragma unroll
  for (int e = 0; e < EP; ++e) {
    if (e >= E) break;
    p[e] += s_bias[e];
    if (nz != nullptr) p[e] += nz[e];
    m = fmaxf(m, p[e]);
  }
  float z = 0.f;
#pragma unroll
  for (int e = 0; e < EP; ++e) {
    if (e >= E) break;
    p[e] = expf(p[e] - m);
    z += p[e];
  }
#pragma unroll
  for (int e = 0; e < EP; ++e) {
    if (e >= E) break;
    p[e] = p[e] / z;
  }
  lse = m + logf(z);
  uint64_t taken = 0;
  sel_sum = 0.f;
#pragma unroll
  for (int sl = 0; sl < MM_MAX_TOPK; ++sl) {
    sel_e[sl] = 0;
    sel_p[sl] = 0.f;
    if (sl < k) {
      float bp = -1.f;
      int be = 0;
#pragma unroll
      for (int e = 0; e < EP; ++e) {
        if (e >= E) break;
        if (!((taken >> e) & 1ull) && p[e] > bp) {
          bp = p[e];
          be = e;
        }
      }
      taken |= 1ull << be;
      sel_sum += bp;
      sel_e[sl] = be;
      sel_p[sl] = bp;
    }
  }
}

// Block norm, tensor-core routers: columns [0, E) of the accumulator row
// hold x . hi, columns [E, 2E) x . lo; the logits are inv_rms * (hi + lo).
// The remainders are loaded from TMEM at column E (a runtime column address)
// so that every register index is a compile-time one.  The loads touch
// columns below E + 16 * ceil(E / 16), inside the callers' allocations (64
// columns with E <= 32; 32 columns with E <= 8).  Warp-collective.
template <int EP>
__device__ __forceinline__ void norm_logits(float (&p)[EP], uint32_t trow, int E, float inv_rms) {
  float lo[EP];
#pragma unroll
  for (int c0 = 0; c0 < EP; c0 += 16) {
    if (c0 >= E) {
#pragma unroll
      for (int j = 0; j < 16; ++j) lo[c0 + j] = 0.f;
      continue;
    }
    uint32_t r[16];
    tmem_ld_32x32b_x16(trow + static_cast<uint32_t>(E + c0), r);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 16; ++j) lo[c0 + j] = __uint_as_float(r[j]);
  }
#pragma unroll
  for (int e = 0; e < EP; ++e)
    if (e < E) p[e] = inv_rms * (p[e] + lo[e]);
}

constexpr int kRtStages = 2;
struct RtMaps {
  CUtensorMap x;                 // x as (64, T, H / 64), box 64 x 64 x nkb
  CUtensorMap wr;                // Wr as (64, E, H / 64), box 64 x EP x nkb (rows >= E read as 0)
};

template <int EP>
__global__ void __launch_bounds__(kRouteThreads)
router_tc_kernel(const __grid_constant__ RtMaps M, int64_t T, int H, int E, int k,
                 const float* __restrict__ bias, int32_t* __restrict__ topk_idx,
                 float* __restrict__ topk_w, int32_t* __restrict__ blk_cnt,
                 float* __restrict__ blk_prob, const RouteExtras X, int nkb, uint32_t stage_bytes) {
  // the dispatch kernel may launch as soon as router blocks start to leave
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ unsigned char rt_raw[];
  uint8_t* smem = align1024(rt_raw);
  __shared__ __align__(8) uint64_t full[kRtStages], empty[kRtStages], lbar, drained;
  __shared__ uint32_t s_tmem;
  __shared__ int s_gcnt[kMaxGroups];
  __shared__ float s_red[2][EP];
  __shared__ float s_redz[2];
  __shared__ float s_bias[EP];
  __shared__ float s_inv[kRouteTokensPerBlock];
  __shared__ int s_last;
  const RouterVariant& rv = X.rv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rblk = blockIdx.x;
  const int nblk = static_cast<int>((T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock);
  const int64_t t0 = static_cast<int64_t>(rblk) * kRouteTokensPerBlock;
  const int ntok = static_cast<int>(T - t0 < kRouteTokensPerBlock ? T - t0 : kRouteTokensPerBlock);
  const int G = k * E;
  const int nst = (H / 64) / nkb;
  constexpr uint32_t kXTile = 64 * 128;          // 64 rows x one k-block
  constexpr uint32_t kWTile = EP * 128;
  WsHeader* hdr = X.hdr;

  if (tid == 0) {
    for (int q = 0; q < kRtStages; ++q) {
      mbar_init(&full[q], 1);
      mbar_init(&empty[q], 1);
    }
    mbar_init(&lbar, 1);
    mbar_init(&drained, 1);
    fence_mbar_init();
  }
  for (int g = tid; g < G; g += kRouteThreads) s_gcnt[g] = 0;
  if (warp == 1) {
    tmem_alloc(&s_tmem, 64);
    tmem_relinquish();
  }
  // launched as a programmatic dependent: the set-up above overlaps the
  // previous kernel of the stream, whose outputs (x, Wr, the bias, or the
  // buffers written here) are touched only once it has finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid < EP) s_bias[tid] = (bias != nullptr && tid < E) ? bias[tid] : 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  bool ok = true;

  if (tid == 0) {
    // producer: stage q = nkb x tiles, then nkb Wr tiles
    for (int q = 0; ok && q < nst; ++q) {
      const int sl = q % kRtStages;
      if (!mbar_wait(&empty[sl], ((q / kRtStages) & 1) ^ 1, nullptr, hdr, 62)) { ok = false; break; }
      uint8_t* st = smem + sl * stage_bytes;
      mbar_arrive_expect_tx(&full[sl], static_cast<uint32_t>(nkb) * (kXTile + kWTile));
      tma_load_3d(st, &M.x, &full[sl], 0, static_cast<int32_t>(t0), q * nkb);
      tma_load_3d(st + nkb * kXTile, &M.wr, &full[sl], 0, 0, q * nkb);
    }
  }
  if (tid == 32) {
    // MMA issuer: L[t, e] += x_t . Wr_e over the k-blocks
    const uint32_t idesc = idesc_bf16_f32(128, EP);
    for (int q = 0; ok && q < nst; ++q) {
      const int sl = q % kRtStages;
      if (!mbar_wait(&full[sl], (q / kRtStages) & 1, nullptr, hdr, 63)) { ok = false; break; }
      tc_fence_after();
      const uint8_t* st = smem + sl * stage_bytes;
      for (int kl = 0; kl < nkb; ++kl) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem, smem_desc_sw128(smem_u32(st + kl * kXTile + kk * 32)),
                    smem_desc_sw128(smem_u32(st + nkb * kXTile + kl * kWTile + kk * 32)), idesc,
                    (q | kl | kk) ? 1u : 0u);
      }
      umma_commit(&empty[sl]);
    }
    if (ok) umma_commit(&lbar);
  }
  // block RMSNorm: the other warps take each token's 1 / rms from its row of
  // x while the MMAs run (warp w' = warp - 2 takes tokens w', w' + 6, ...;
  // lanes over 16-byte vectors, a fixed tree)
  const bool norm = X.norm.w != nullptr;
  if (norm) {
    if (warp >= 2) {
      for (int t = warp - 2; t < ntok; t += kRouteThreads / 32 - 2) {
        const uint4* row = reinterpret_cast<const uint4*>(X.xrow) + (t0 + t) * (H / 8);
        float ss = 0.f;
        for (int v = lane; v < H / 8; v += 32) {
          const uint4 q = row[v];
          const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float a = __uint_as_float(w4[j] << 16), b = __uint_as_float(w4[j] & 0xffff0000u);
            ss = fmaf(a, a, ss);
            ss = fmaf(b, b, ss);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) {
          const float sv = 1.0f / sqrtf(ss / static_cast<float>(H) + X.norm.eps);
          s_inv[t] = sv;
          X.norm.inv_rms[t0 + t] = sv;
        }
      }
    }
    __syncthreads();
  }
  if (warp < 2) {
    const int t = warp * 32 + lane;              // TMEM lane = token of the block
    const bool valid = t < ntok;
    ok = warp_wait(&lbar, 0, nullptr, hdr, 64) && ok;
    tc_fence_after();
    float p[EP];
    if (ok) {
#pragma unroll
      for (int c0 = 0; c0 < EP; c0 += 16) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) p[c0 + j] = __uint_as_float(r[j]);
      }
      if (norm) {
        // logits = inv_rms * (x . hi + x . lo); columns E.. hold the remainders
        const float sv = valid ? s_inv[t] : 0.f;
        norm_logits<EP>(p, tmem + (static_cast<uint32_t>(warp * 32) << 16), E, sv);
      }
      const float* nz = (rv.noise != nullptr && valid) ? rv.noise + (t0 + t) * E : nullptr;
      float lse, sel_sum;
      int sel_e[MM_MAX_TOPK];
      float sel_p[MM_MAX_TOPK];
      route_token<EP>(p, E, k, s_bias, nz, lse, sel_e, sel_p, sel_sum);
      if (valid) {
        if (rv.probs != nullptr) {
          float* pr = rv.probs + (t0 + t) * E;
#pragma unroll
          for (int e = 0; e < EP; ++e) {
            if (e >= E) break;
            pr[e] = p[e];
          }
        }
        if (rv.lse != nullptr) rv.lse[t0 + t] = lse;
      }
      {
        float v = valid ? lse * lse : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) s_redz[warp] = v;
      }
      if (valid) {
        const float inv = sel_sum + 1e-20f;
#pragma unroll
        for (int sl = 0; sl < MM_MAX_TOPK; ++sl) {
          if (sl < k) {
            topk_idx[(t0 + t) * k + sl] = sel_e[sl];
            topk_w[(t0 + t) * k + sl] = sel_p[sl] / inv;
            atomicAdd(&s_gcnt[sl * E + sel_e[sl]], 1);
          }
        }
      }
      // the block's probability sums per expert: fixed butterfly order
#pragma unroll
      for (int e = 0; e < EP; ++e) {
        if (e >= E) break;
        float v = valid ? p[e] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) s_red[warp][e] = v;
      }
    }
  }
  ok = __syncthreads_and(ok);
  if (ok) {
    if (tid < E) blk_prob[static_cast<int64_t>(rblk) * E + tid] = s_red[0][tid] + s_red[1][tid];
    if (tid == 0 && rv.blk_z != nullptr) rv.blk_z[rblk] = s_redz[0] + s_redz[1];
    for (int g = tid; g < G; g += kRouteThreads) blk_cnt[static_cast<int64_t>(rblk) * G + g] = s_gcnt[g];
  }
  if (tid == 32) {
    umma_commit(&drained);                       // every issued UMMA has finished
    mbar_wait(&drained, 0, nullptr, hdr, 65);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 64);
  // route-only calls: as router_kernel
  if (!X.do_scan || !ok) return;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&X.hdr->route_done, 1u) == static_cast<unsigned>(nblk - 1));
  __syncthreads();
  if (s_last) {
    __threadfence();
    scan_block(E, k, nblk, T, X, blk_cnt, blk_prob);
    if (tid == 0) X.hdr->route_done = 0u;
  }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
size_t router_smem_bytes(int H, int E, int k) {
  return static_cast<size_t>(E) * H * sizeof(float) + static_cast<size_t>(k) * E * sizeof(int);
}

// Router grid: one block per 64 tokens.  x is staged in shared memory when the block's rows and Wr
// fit in 110 KiB together (two blocks per SM).
template <typename Tin>
static cudaError_t launch_router_t(const void* x, const void* Wr, const float* bias, int64_t T, int H,
                                   int E, int k, int32_t* topk_idx, float* topk_w, int32_t* blk_cnt,
                                   float* blk_prob, RouteExtras X, cudaStream_t st) {
  const int nblk = static_cast<int>((T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock);
  size_t smem = static_cast<size_t>(E) * H * sizeof(Tin) + static_cast<size_t>(k) * E * sizeof(int);
  X.x_off = static_cast<uint32_t>((smem + 127) & ~size_t(127));
  const size_t xbytes = static_cast<size_t>(kRouteTokensPerBlock) * H * sizeof(Tin);
  X.stage_x = X.x_off + xbytes <= 110 * 1024 ? 1 : 0;
  if (X.stage_x) smem = X.x_off + xbytes;
#define MM_ROUTER_CASE(EPAD)                                                                   \
  {                                                                                            \
    auto fn = router_kernel<Tin, EPAD>;                                                        \
    cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), smem);             \
    if (err != cudaSuccess) return err;                                                        \
    fn<<<nblk, kRouteThreads, smem, st>>>(static_cast<const Tin*>(x),               \
                                                     static_cast<const Tin*>(Wr), bias, T, H,   \
                                                     E, k, topk_idx, topk_w, blk_cnt,          \
                                                     blk_prob, X);                             \
    return cudaGetLastError();                                                                 \
  }
  if (E <= 8) MM_ROUTER_CASE(8)
  if (E <= 16) MM_ROUTER_CASE(16)
  if (E <= 32) MM_ROUTER_CASE(32)
  MM_ROUTER_CASE(64)
#undef MM_ROUTER_CASE
}

// Tensor-core router for bf16 (H a multiple of 64, E <= 64): nkb k-blocks
// per stage (the most, up to 4, that divide H / 64).
template <int EP>
static cudaError_t launch_router_tc(const void* x, const void* Wr, const float* bias, int64_t T,
                                    int H, int E, int k, int32_t* topk_idx, float* topk_w,
                                    int32_t* blk_cnt, float* blk_prob, const RouteExtras& X,
                                    cudaStream_t st) {
  const int KB = H / 64;
  int nkb = 4;
  while (KB % nkb != 0) --nkb;
  const size_t xt = 64 * 128, wt = static_cast<size_t>(EP) * 128;
  // the A read of a stage's last x tile spans 128 rows
  size_t stage = std::max(nkb * (xt + wt), (nkb - 1) * xt + 2 * xt);
  stage = (stage + 1023) / 1024 * 1024;
  const size_t smem = kRtStages * stage + 1024;
  static RtMaps m;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  const uint64_t sx[2] = {static_cast<uint64_t>(H) * 2, 128};
  const uint64_t dx[3] = {64, static_cast<uint64_t>(T), static_cast<uint64_t>(KB)};
  const uint32_t bx[3] = {64, static_cast<uint32_t>(kRouteTokensPerBlock), static_cast<uint32_t>(nkb)};
  if (!make_map_3d(&m.x, x, dx, sx, bx)) return cudaErrorInvalidValue;
  // with the block norm, the B operand is w * Wr as 2E rows (high parts, remainders)
  const bool norm = X.norm.w != nullptr;
  const uint64_t dw[3] = {64, static_cast<uint64_t>(norm ? 2 * E : E), static_cast<uint64_t>(KB)};
  const uint32_t bw[3] = {64, static_cast<uint32_t>(EP), static_cast<uint32_t>(nkb)};
  if (!make_map_3d(&m.wr, norm ? X.norm.wr_hl : Wr, dw, sx, bw)) return cudaErrorInvalidValue;
  auto fn = router_tc_kernel<EP>;
  cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), smem);
  if (err != cudaSuccess) return err;
  const int nblk = static_cast<int>((T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock);
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(nblk);
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, m, T, H, E, k, bias, topk_idx, topk_w, blk_cnt, blk_prob, X,
                            nkb, static_cast<uint32_t>(stage));
}

// ---------------------------------------------------------------------------
// Router and dispatch in one kernel, so that x is read from HBM once per
// call (bf16; H a multiple of 64 up to 768; E, or 2E with the block norm,
// up to 16; k up to 4; every block resident at once: T <= TB x the SMs).
// Block b routes tokens [TB b, +TB), TB = 128 or 64 (64 when that still
// keeps every block resident: twice the SMs for T <= 64 x the SMs): router
// blocks TB/64 b .. of the two-kernel path, whose per-block partials
// (counts, probability sums, lse^2 sums) it writes unchanged, so that every
// output is the same bit for bit.  Its x rows stay in shared memory for the
// whole call: all H / 64 k-blocks as 128-byte-swizzled tiles, the A operand
// of the logits' UMMA (M = 128, N = 16, fp32 in TMEM; with TB = 64 the MMA's
// rows 64-127 read the next tile's rows, whose results in TMEM lanes 64-127
// no thread uses) and, after one grid barrier that
// publishes every block's group counts, the source of its rows of Xp.
// Past the barrier each block derives the group offsets and its bases as
// the dispatch kernel does, writes perm and its Xp rows (x * inv_rms * w
// with the block norm), and block 0 the offsets, counts, aux loss and
// z-loss.  The next kernel of the stream is released only after the
// barrier, when every block of this grid already holds its SM.
// Warp roles: warps 0-3 route (thread = token = TMEM lane); warp 4 lane 0
// issues the TMA loads, warp 5 lane 0 the UMMAs; all 8 warps take the norm's
// sums of squares and the row copies.
// ---------------------------------------------------------------------------
constexpr int kRdTokens = 128;                   // tokens per block, at most
constexpr int kRdThreads = 512;                  // 16 warps: the row copies want many
constexpr int kRdEP = 16;                        // UMMA N: E (2E with the norm) padded
constexpr int kRdMaxKb = 12;                     // H <= 768
constexpr int kRdMaxK = 4;
constexpr int kRdMaxG = kRdEP * kRdMaxK;
constexpr uint32_t kRdWTile = kRdEP * 128;

// Dynamic shared memory of a block of TB tokens: the x tiles, the router
// weight tiles, alignment, and for TB < 128 room for the UMMA's rows past
// the last x tile (it reads 128 rows from each tile's start).
constexpr size_t rd_smem_bytes(int TB, int KB) {
  return static_cast<size_t>(KB) * (static_cast<size_t>(TB) * 128 + kRdWTile) +
         static_cast<size_t>(kRdTokens - TB) * 128 + 1024;
}

struct RdMaps {
  CUtensorMap x;                 // x as (64, T, H / 64), box 64 x TB x nkb (rows >= T read as 0)
  CUtensorMap wr;                // Wr (or the norm's halves) as (64, En, H / 64), box 64 x 16 x nkb
};

template <int TB>
__global__ void __launch_bounds__(kRdThreads, 1)
route_dispatch_kernel(const __grid_constant__ RdMaps M, int64_t T, int H, int E, int k,
                      const float* __restrict__ bias, int32_t* __restrict__ topk_idx,
                      float* __restrict__ topk_w, int32_t* __restrict__ blk_cnt,
                      float* __restrict__ blk_prob, const DispatchOut D,
                      int32_t* __restrict__ perm, __nv_bfloat16* __restrict__ Xp, int nkb) {
  constexpr int EP = kRdEP;
  static_assert(TB == 64 || TB == 128, "tokens per block");
  constexpr int kRB = TB / kRouteTokensPerBlock;         // router blocks per block
  constexpr uint32_t kRdXTile = TB * 128;                // TB rows x one k-block
  extern __shared__ unsigned char rd_raw[];
  uint8_t* smem = align1024(rd_raw);
  const int KB = H / 64;
  const int nst = KB / nkb;
  uint8_t* sx = smem;                            // [KB][TB rows][128 B]
  uint8_t* sw = smem + KB * kRdXTile;            // [KB][16 rows][128 B]
  __shared__ __align__(8) uint64_t full[kRdMaxKb], lbar, drained;
  __shared__ uint32_t s_tmem;
  __shared__ int s_gcnt[kRB][kRdMaxG];           // per router block of 64 tokens
  __shared__ float s_red[4][EP];
  __shared__ float s_redz[4];
  __shared__ float s_bias[EP];
  __shared__ float s_inv[TB];
  __shared__ int s_wcnt[4][EP];
  __shared__ int s_pos[TB * kRdMaxK];
  __shared__ int s_tot[kRdMaxG], s_base[kRdMaxG], s_off[kRdMaxG + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kRdThreads / 32;
  const int b = blockIdx.x;
  const int64_t t0 = static_cast<int64_t>(b) * TB;
  const int ntok = static_cast<int>(T - t0 < TB ? T - t0 : TB);
  const int nrb = static_cast<int>((T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock);
  const int rb0 = kRB * b;                       // this block's first router block
  const int G = k * E;
  WsHeader* hdr = D.hdr;
  const RouterVariant& rv = D.rv;
  const __nv_bfloat16* norm_w = static_cast<const __nv_bfloat16*>(D.norm.w);

  if (tid == 0) {
    for (int q = 0; q < nst; ++q) mbar_init(&full[q], 1);
    mbar_init(&lbar, 1);
    mbar_init(&drained, 1);
    fence_mbar_init();
  }
  for (int g = tid; g < kRB * kRdMaxG; g += kRdThreads) (&s_gcnt[0][0])[g] = 0;
  if (warp == 4) {
    tmem_alloc(&s_tmem, 32);
    tmem_relinquish();
  }
  // launched as a programmatic dependent: x, Wr and the outputs belong to
  // the previous kernel until it has finished
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid < EP) s_bias[tid] = (bias != nullptr && tid < E) ? bias[tid] : 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  bool ok = true;

  if (tid == 4 * 32) {
    // producer: every stage at once (nkb k-blocks of x and of Wr each); no slot is reused
    for (int q = 0; q < nst; ++q) {
      mbar_arrive_expect_tx(&full[q], static_cast<uint32_t>(nkb) * (kRdXTile + kRdWTile));
      tma_load_3d(sx + q * nkb * kRdXTile, &M.x, &full[q], 0, static_cast<int32_t>(t0), q * nkb);
      tma_load_3d(sw + q * nkb * kRdWTile, &M.wr, &full[q], 0, 0, q * nkb);
    }
  }
  if (tid == 5 * 32) {
    // MMA issuer: L[t, e] = sum over the k-blocks of x_t . Wr_e
    const uint32_t idesc = idesc_bf16_f32(128, EP);
    bool mok = true;
    for (int q = 0; q < nst && mok; ++q) {
      if (!mbar_wait(&full[q], 0, nullptr, hdr, 66)) {
        mok = false;
        break;
      }
      tc_fence_after();
      for (int kl = 0; kl < nkb; ++kl) {
        const int kb = q * nkb + kl;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem, smem_desc_sw128(smem_u32(sx + kb * kRdXTile + kk * 32)),
                    smem_desc_sw128(smem_u32(sw + kb * kRdWTile + kk * 32)), idesc,
                    (kb | kk) ? 1u : 0u);
      }
    }
    if (mok) umma_commit(&lbar);
  }
  if (norm_w != nullptr) {
    // block RMSNorm: each token's 1 / rms from its staged row (warp w takes
    // tokens w, w + 8, ...; lanes over 16-byte vectors in row order, then a
    // fixed xor tree: the tensor-core router's order)
    bool landed = true;
    for (int q = 0; q < nst; ++q) landed = warp_wait(&full[q], 0, nullptr, hdr, 67) && landed;
    if (landed) {
      for (int t = warp; t < ntok; t += kWarps) {
        float ss = 0.f;
        for (int v = lane; v < H / 8; v += 32) {
          const uint4 qv = *reinterpret_cast<const uint4*>(
              sx + (v >> 3) * kRdXTile + t * 128 + (((v & 7) ^ (t & 7)) << 4));
          const uint32_t w4[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float a = __uint_as_float(w4[j] << 16), c = __uint_as_float(w4[j] & 0xffff0000u);
            ss = fmaf(a, a, ss);
            ss = fmaf(c, c, ss);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) {
          const float sv = 1.0f / sqrtf(ss / static_cast<float>(H) + D.norm.eps);
          s_inv[t] = sv;
          D.norm.inv_rms[t0 + t] = sv;
        }
      }
    }
    ok = ok && landed;
    __syncthreads();
  }

  // ---- routing: warps 0-3, thread = token (TMEM lane)
  int sel_e[MM_MAX_TOPK];
  int rk[kRdMaxK];
  const int t = tid;
  const bool valid = warp < 4 && t < ntok;
  if (warp < 4) {
    ok = warp_wait(&lbar, 0, nullptr, hdr, 68) && ok;
    tc_fence_after();
    float p[EP];
    float lse = 0.f, sel_sum = 0.f;
    float sel_p[MM_MAX_TOPK];
    if (ok) {
      uint32_t r[16];
      tmem_ld_32x32b_x16(tmem + (static_cast<uint32_t>(warp * 32) << 16), r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) p[j] = __uint_as_float(r[j]);
      if (norm_w != nullptr) {
        // logits = inv_rms * (x . hi + x . lo); columns E.. hold the remainders
        const float sv = valid ? s_inv[t] : 0.f;
        norm_logits<EP>(p, tmem + (static_cast<uint32_t>(warp * 32) << 16), E, sv);
      }
      const float* nz = (rv.noise != nullptr && valid) ? rv.noise + (t0 + t) * E : nullptr;
      route_token<EP>(p, E, k, s_bias, nz, lse, sel_e, sel_p, sel_sum);
    } else {
#pragma unroll
      for (int e = 0; e < EP; ++e) p[e] = 0.f;
#pragma unroll
      for (int sl = 0; sl < MM_MAX_TOPK; ++sl) sel_e[sl] = 0;
    }
    if (valid && ok) {
      if (rv.probs != nullptr) {
        float* pr = rv.probs + (t0 + t) * E;
#pragma unroll
        for (int e = 0; e < EP; ++e) {
          if (e >= E) break;
          pr[e] = p[e];
        }
      }
      if (rv.lse != nullptr) rv.lse[t0 + t] = lse;
      const float inv = sel_sum + 1e-20f;
#pragma unroll
      for (int sl = 0; sl < MM_MAX_TOPK; ++sl) {
        if (sl < k) {
          topk_idx[(t0 + t) * k + sl] = sel_e[sl];
          topk_w[(t0 + t) * k + sl] = sel_p[sl] / inv;
        }
      }
    }
    {
      float v = (valid && ok) ? lse * lse : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) s_redz[warp] = v;
    }
    // the router block's probability sums per expert: fixed butterfly order
#pragma unroll
    for (int e = 0; e < EP; ++e) {
      if (e >= E) break;
      float v = (valid && ok) ? p[e] : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) s_red[warp][e] = v;
    }
  }
  // rank of each assignment among the block's tokens that chose the same
  // expert in the same slot, in token order, and from the same matches the
  // router blocks' group counts (warps 0-1: router block rb0, warps 2-3:
  // rb0 + 1 when TB = 128)
#pragma unroll
  for (int sl = 0; sl < kRdMaxK; ++sl) {
    if (sl >= k) break;
    int e = -1, rank = 0;
    unsigned peers = 0;
    if (warp < 4) {
      e = valid ? sel_e[sl] : -1;
      peers = __match_any_sync(0xffffffffu, e);
      rank = __popc(peers & ((1u << lane) - 1u));
    }
    for (int i = tid; i < 4 * EP; i += kRdThreads) (&s_wcnt[0][0])[i] = 0;
    __syncthreads();
    if (warp < 4 && e >= 0 && lane == __ffs(peers) - 1) s_wcnt[warp][e] = __popc(peers);
    __syncthreads();
    if (warp < 4 && e >= 0) {
      for (int w = 0; w < warp; ++w) rank += s_wcnt[w][e];
      rk[sl] = rank;
    }
    if (tid < kRB * E) {
      const int i = tid / E, ee = tid - i * E;
      s_gcnt[i][sl * E + ee] = s_wcnt[2 * i][ee] + s_wcnt[2 * i + 1][ee];
    }
    __syncthreads();
  }
  ok = __syncthreads_and(ok) != 0;
  // the router blocks' partials, as the tensor-core router writes them (warp
  // 0; the grid barrier's __syncthreads and release by thread 0 publish them)
  if (ok && warp == 0) {
    for (int i = 0; i < kRB; ++i) {
      const int rb = rb0 + i;
      if (rb >= nrb) break;
      if (lane < E) blk_prob[static_cast<int64_t>(rb) * E + lane] = s_red[2 * i][lane] + s_red[2 * i + 1][lane];
      if (lane == 0 && rv.blk_z != nullptr) rv.blk_z[rb] = s_redz[2 * i] + s_redz[2 * i + 1];
      for (int g = lane; g < G; g += 32) blk_cnt[static_cast<int64_t>(rb) * G + g] = s_gcnt[i][g];
    }
  }
  unsigned ticket = 0;
  ok = grid_barrier(hdr, 69, 1, &ticket) && ok;
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (ok) {
    // group totals and this block's bases: thread (slice j, group g) adds the
    // counts of router blocks j, j + S, ... (all requested at once), then the
    // slices meet in shared memory (integer sums: exact in any order)
    for (int g = tid; g < G; g += kRdThreads) {
      s_tot[g] = 0;
      s_base[g] = 0;
    }
    __syncthreads();
    {
      const int S = kRdThreads / G;                // G <= 64: at least 8 slices
      const int g = tid % G, j = tid / G;
      if (j < S) {
        int all = 0, before = 0;
        for (int rb = j; rb < nrb; rb += 8 * S) {
          int c[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int r = rb + u * S;
            c[u] = r < nrb ? __ldcg(blk_cnt + static_cast<int64_t>(r) * G + g) : 0;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            all += c[u];
            before += (rb + u * S < rb0) ? c[u] : 0;
          }
        }
        atomicAdd(&s_tot[g], all);
        atomicAdd(&s_base[g], before);
      }
    }
    __syncthreads();
    if (warp == 0) {
      // exclusive scan of the group totals, two groups a lane (G <= 64)
      const int g0 = 2 * lane;
      const int c0 = g0 < G ? s_tot[g0] : 0, c1 = g0 + 1 < G ? s_tot[g0 + 1] : 0;
      int incl = c0 + c1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      const int ex = incl - c0 - c1;
      if (g0 < G) s_off[g0] = ex;
      if (g0 + 1 < G) s_off[g0 + 1] = ex + c0;
      if (lane == 31) s_off[G] = incl;
    }
    __syncthreads();
    const bool totals = b == 0;
    if (valid) {
#pragma unroll
      for (int sl = 0; sl < kRdMaxK; ++sl) {
        if (sl >= k) break;
        const int g = sl * E + sel_e[sl];
        const int pos = s_off[g] + s_base[g] + rk[sl];
        s_pos[t * k + sl] = pos;
        perm[pos] = static_cast<int32_t>((t0 + t) * k + sl);
      }
    }
    __syncthreads();
    if (totals && warp >= kWarps - 4) {
      // block 0: warps 12-15 write the call's totals while warps 0-11 copy its rows
      write_route_totals_w4(D, s_tot, s_off, G, E, k, nrb, blk_prob, T);
    } else if (Xp != nullptr) {
      // the staged rows, un-swizzled: a warp per assignment row, lane l on
      // 16-byte chunks l, l + 32, ... (k-block (l >> 3) + 4 j, chunk l & 7),
      // two rows in flight per warp (block 0: warps 0-11)
      const int na = ntok * k;
      const int nv = H / 8;
      const uint32_t lane_off = static_cast<uint32_t>(lane >> 3) * kRdXTile;
      const int lq = lane & 7;
      const int nw = totals ? kWarps - 4 : kWarps;   // copying warps
      const int cw = warp;
      constexpr int kCh = kRdMaxKb * 64 / 8 / 32;     // 16-byte chunks per lane and row, at most
      for (int a0 = cw; a0 < na; a0 += 2 * nw) {
        // two rows: every chunk requested before any is stored
        uint4 q[2][kCh];
        int64_t drow[2];
        int trow[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int a = a0 + r * nw;
          trow[r] = a < na ? a / k : -1;
          drow[r] = a < na ? static_cast<int64_t>(s_pos[a]) * H : 0;
          if (a >= na) continue;
          const int tt = trow[r];
          const uint8_t* src = sx + lane_off + tt * 128 + ((lq ^ (tt & 7)) << 4);
#pragma unroll
          for (int c = 0; c < kCh; ++c)
            if (lane + 32 * c < nv) q[r][c] = *reinterpret_cast<const uint4*>(src + 4 * c * kRdXTile);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          if (trow[r] < 0) continue;
          __nv_bfloat16* dst = Xp + drow[r] + lane * 8;
          const float inv = norm_w != nullptr ? s_inv[trow[r]] : 1.f;
#pragma unroll
          for (int c = 0; c < kCh; ++c) {
            const int v = lane + 32 * c;                // this lane's chunk
            if (v >= nv) continue;
            uint4 qv = q[r][c];
            if (norm_w != nullptr) {
              float xv[8], g8[8];
              const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&qv);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float2 f = __bfloat1622float2(h2[j]);
                xv[2 * j] = f.x;
                xv[2 * j + 1] = f.y;
              }
              load_vec8(norm_w + v * 8, g8);
              __nv_bfloat16 o8[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) o8[j] = static_cast<__nv_bfloat16>(xv[j] * inv * g8[j]);
              qv = *reinterpret_cast<const uint4*>(o8);
            }
            *reinterpret_cast<uint4*>(dst + 32 * c * 8) = qv;
          }
        }
      }
    }
  }
  if (tid == 5 * 32) {
    umma_commit(&drained);                       // every issued UMMA has finished
    mbar_wait(&drained, 0, nullptr, hdr, 70);
  }
  if (tid == 4 * 32)                             // every copy into shared memory has landed
    for (int q = 0; q < nst; ++q) mbar_wait(&full[q], 0, nullptr, hdr, 71);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, 32);
  if (tid == 0) grid_barrier_reset(hdr, ticket);
}

// Blocks of TB tokens that can be resident at once (one per SM), per H.
template <int TB>
static int64_t rd_max_blocks(int H) {
  static int64_t max_blocks[kRdMaxKb + 1];
  static bool known[kRdMaxKb + 1];
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  const int KB = H / 64;
  if (!known[KB]) {
    const size_t smem = rd_smem_bytes(TB, KB);
    auto fn = route_dispatch_kernel<TB>;
    int per_sm = 0;
    if (ensure_dynamic_smem(reinterpret_cast<const void*>(fn), smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kRdThreads, smem) != cudaSuccess) {
      (void)cudaGetLastError();
      per_sm = 0;
    }
    max_blocks[KB] = static_cast<int64_t>(per_sm) * num_sms();
    known[KB] = true;
  }
  return max_blocks[KB];
}

// Tokens per block of the fused router + dispatch for this call: 64 while
// every block of 64 still fits on the GPU at once, else 128; 0 if neither.
static int rd_tokens_per_block(int64_t T, int H) {
  if ((T + 63) / 64 <= rd_max_blocks<64>(H)) return 64;
  if ((T + 127) / 128 <= rd_max_blocks<128>(H)) return 128;
  return 0;
}

// Whether the fused router + dispatch takes this call: bf16, the shapes it
// is built for, 16-byte aligned x and router weights, and every block
// resident at once (one per SM).
bool route_dispatch_ok(int dtype, const void* x, const void* Wr, int64_t T, int H, int E, int k,
                       const DispatchOut& D) {
  const bool norm = D.norm.w != nullptr;
  const int En = norm ? 2 * E : E;
  const void* wr = norm ? D.norm.wr_hl : Wr;
  if (dtype != kDtypeBF16 || H % 64 != 0 || H / 64 > kRdMaxKb || En > kRdEP || k > kRdMaxK ||
      T < 1 || (reinterpret_cast<uintptr_t>(x) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(wr) & 15u) != 0 || D.hdr == nullptr)
    return false;
  return rd_tokens_per_block(T, H) > 0;
}

// Launch of the fused router + dispatch; route_dispatch_ok() must hold.
cudaError_t launch_route_dispatch(int dtype, const void* x, const void* Wr, const float* bias,
                                  int64_t T, int H, int E, int k, int32_t* topk_idx, float* topk_w,
                                  int32_t* blk_cnt, float* blk_prob, const DispatchOut& D,
                                  int32_t* perm, void* Xp, cudaStream_t st) {
  (void)dtype;
  const bool norm = D.norm.w != nullptr;
  const int En = norm ? 2 * E : E;
  const void* wr = norm ? D.norm.wr_hl : Wr;
  const int KB = H / 64;
  const int TB = rd_tokens_per_block(T, H);
  if (TB == 0) return cudaErrorInvalidValue;
  int nkb = 4;
  while (KB % nkb != 0) --nkb;
  const size_t smem = rd_smem_bytes(TB, KB);
  auto fn = TB == 64 ? route_dispatch_kernel<64> : route_dispatch_kernel<128>;
  const int64_t nblk = (T + TB - 1) / TB;
  RdMaps m;
  const uint64_t sx[2] = {static_cast<uint64_t>(H) * 2, 128};
  const uint64_t dx[3] = {64, static_cast<uint64_t>(T), static_cast<uint64_t>(KB)};
  const uint32_t bx[3] = {64, static_cast<uint32_t>(TB), static_cast<uint32_t>(nkb)};
  if (!make_map_3d(&m.x, x, dx, sx, bx)) return cudaErrorInvalidValue;
  const uint64_t dw[3] = {64, static_cast<uint64_t>(En), static_cast<uint64_t>(KB)};
  const uint32_t bw[3] = {64, static_cast<uint32_t>(kRdEP), static_cast<uint32_t>(nkb)};
  if (!make_map_3d(&m.wr, wr, dw, sx, bw)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(static_cast<unsigned>(nblk));
  cfg.blockDim = dim3(kRdThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, m, T, H, E, k, bias, topk_idx, topk_w, blk_cnt, blk_prob, D,
                            perm, static_cast<__nv_bfloat16*>(Xp), nkb);
}

cudaError_t launch_router(int dtype, const void* x, const void* Wr, const float* bias, int64_t T,
                          int H, int E, int k, int32_t* topk_idx, float* topk_w, int32_t* blk_cnt,
                          float* blk_prob, const RouteOut& out, WsHeader* hdr, cudaStream_t st) {
  RouteExtras X;
  memset(&X, 0, sizeof(X));
  X.blk_base = out.blk_base;
  X.offsets = out.offsets;
  X.counts = out.counts;
  X.aux_loss = out.aux_loss;
  X.coef = out.coef;
  X.do_scan = out.do_scan;
  X.hdr = hdr;
  X.rv = out.rv;
  X.norm = out.norm;
  X.xrow = x;
  // the block norm doubles the router's N (high parts and remainders)
  const int En = X.norm.w != nullptr ? 2 * E : E;
  const bool tc_ok = dtype == kDtypeBF16 && H % 64 == 0 && En <= 64 &&
                     (reinterpret_cast<uintptr_t>(x) & 15u) == 0 && (reinterpret_cast<uintptr_t>(Wr) & 15u) == 0;
  if (tc_ok) {
    if (En <= 16)
      return launch_router_tc<16>(x, Wr, bias, T, H, E, k, topk_idx, topk_w, blk_cnt, blk_prob, X, st);
    if (En <= 32)
      return launch_router_tc<32>(x, Wr, bias, T, H, E, k, topk_idx, topk_w, blk_cnt, blk_prob, X, st);
    return launch_router_tc<64>(x, Wr, bias, T, H, E, k, topk_idx, topk_w, blk_cnt, blk_prob, X, st);
  }
  if (dtype == kDtypeBF16)
    return launch_router_t<__nv_bfloat16>(x, Wr, bias, T, H, E, k, topk_idx, topk_w, blk_cnt,
                                          blk_prob, X, st);
  return launch_router_t<float>(x, Wr, bias, T, H, E, k, topk_idx, topk_w, blk_cnt, blk_prob, X,
                                st);
}

// Launch with programmatic stream serialisation: the dispatch blocks may
// start while the router grid finishes (they wait for it before reading its
// results).
template <typename Tin>
static cudaError_t launch_dispatch_t(const Tin* x, int64_t T, int H, int E, int k,
                                     const int32_t* topk_idx, const int32_t* blk_cnt,
                                     const float* blk_prob, const DispatchOut& D, int32_t* perm,
                                     Tin* Xp, cudaStream_t st) {
  const int nblk = static_cast<int>((T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock);
  const size_t smem = static_cast<size_t>(kRouteTokensPerBlock) * H * sizeof(Tin);
  const int stage = (Xp != nullptr && smem <= 110 * 1024) ? 1 : 0;   // no rows to copy: no staging
  auto fn = dispatch_kernel<Tin>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), stage ? smem : 0);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(nblk);
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = stage ? smem : 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, x, T, H, E, k, topk_idx, blk_cnt, blk_prob, D, perm, Xp,
                            stage);
}

cudaError_t launch_dispatch(int dtype, const void* x, int64_t T, int H, int E, int k,
                            const int32_t* topk_idx, const int32_t* blk_cnt, const float* blk_prob,
                            const DispatchOut& D, int32_t* perm, void* Xp, cudaStream_t st) {
  if (dtype == kDtypeBF16)
    return launch_dispatch_t(static_cast<const __nv_bfloat16*>(x), T, H, E, k, topk_idx, blk_cnt,
                             blk_prob, D, perm, static_cast<__nv_bfloat16*>(Xp), st);
  return launch_dispatch_t(static_cast<const float*>(x), T, H, E, k, topk_idx, blk_cnt, blk_prob,
                           D, perm, static_cast<float*>(Xp), st);
}

}  // namespace mm
