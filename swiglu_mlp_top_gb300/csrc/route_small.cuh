// Routing of a handful of tokens (T <= MAXT) inside one CTA, shared by
// the two streaming kernels: per-token softmax and top-k on one warp each,
// then one warp groups the assignments by expert.  Every CTA of a grid runs
// the same code on the same logits, so all CTAs reach the same tables.
// (MiniMind lesson 13 "FFN 与 MoE" §1.5; minimind3.com chapter 4 §4.3.)
#pragma once

#include "mm_kernels.cuh"

namespace mm {

template <int MAXT>
struct SmallRoute {
  int nA;                                   // assignments (MoE: T*k, dense: T)
  int n_touched;
  int touched[MM_MAX_EXPERTS];              // ascending expert ids
  int slot_of[MM_MAX_EXPERTS];              // expert -> position in touched[] (or -1)
  int cnt[MM_MAX_EXPERTS];                  // assignments per expert
  int e_start[MM_MAX_EXPERTS + 1];          // expert e's assignments: by_e[e_start[e] ..]
  int sel_e[MAXT * MM_MAX_TOPK];     // expert of assignment a = t*k + s
  float sel_a[MAXT * MM_MAX_TOPK];   // its alpha
  int rank[MAXT * MM_MAX_TOPK];      // its place among its expert's assignments
  int by_e[MAXT * MM_MAX_TOPK];      // assignments grouped by expert, in token order
  float prob[MAXT][MM_MAX_EXPERTS + 1];  // logits, then probabilities (row padded)
  float lse[MAXT];                       // logsumexp of each token's logits
};

__device__ __forceinline__ float warp_allsum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per token (t = first_warp, first_warp + nwarps, ...): R.prob[t][:]
// holds the logits on entry and the probabilities on exit.  Lane l holds
// experts l and l + 32 in registers; the logits get the bias and, if given,
// the router noise of the token; the maximum and the sum of the
// exponentials are warp reductions (softmax with the maximum subtracted),
// and each of the k selections is a warp arg-max (larger probability, else
// lower expert index); alpha = p / (sum_S p + 1e-20).  R.lse[t] receives
// the logsumexp of the token's logits, m + log(sum).
template <int MAXT>
__device__ __forceinline__ void route_softmax_topk_warp(SmallRoute<MAXT>& R, int T, int E, int k,
                                                        const float* bias, int first_warp,
                                                        int nwarps, int lane,
                                                        const float* noise = nullptr) {
  for (int t = first_warp; t < T; t += nwarps) {
    float* row = R.prob[t];
    const bool v0 = lane < E, v1 = lane + 32 < E;
    float r0 = v0 ? row[lane] + bias[lane] : -INFINITY;
    float r1 = v1 ? row[lane + 32] + bias[lane + 32] : -INFINITY;
    if (noise != nullptr) {
      if (v0) r0 += noise[t * E + lane];
      if (v1) r1 += noise[t * E + lane + 32];
    }
    float m = fmaxf(r0, r1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float x0 = v0 ? __expf(r0 - m) : 0.f;
    const float x1 = v1 ? __expf(r1 - m) : 0.f;
    const float zsum = warp_allsum_f(x0 + x1);
    const float rz = 1.0f / zsum;
    if (lane == 0) R.lse[t] = m + logf(zsum);
    const float p0 = x0 * rz, p1 = x1 * rz;
    if (v0) row[lane] = p0;
    if (v1) row[lane + 32] = p1;
    bool took0 = false, took1 = false;
    float sel_sum = 0.f;
    for (int s = 0; s < k; ++s) {
      // this lane's best unselected expert (the lower index on a tie)
      float bp = -1.f;
      int be = 2 * MM_MAX_EXPERTS;
      if (v0 && !took0) { bp = p0; be = lane; }
      if (v1 && !took1 && p1 > bp) { bp = p1; be = lane + 32; }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float op = __shfl_xor_sync(0xffffffffu, bp, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (op > bp || (op == bp && oe < be)) { bp = op; be = oe; }
      }
      took0 = took0 || be == lane;
      took1 = took1 || be == lane + 32;
      sel_sum += bp;
      if (lane == 0) {
        R.sel_e[t * k + s] = be;
        R.sel_a[t * k + s] = bp;
      }
    }
    __syncwarp();
    const float inv = sel_sum + 1e-20f;
    if (lane < k) R.sel_a[t * k + lane] = R.sel_a[t * k + lane] / inv;
    __syncwarp();
  }
}

// One warp: per-expert counts, their prefix, the touched experts in
// ascending order and the assignments grouped by expert (token order kept).
template <int MAXT>
__device__ __forceinline__ void route_group(SmallRoute<MAXT>& R, int nA, int E, int lane) {
  for (int e = lane; e < E; e += 32) R.cnt[e] = 0;
  __syncwarp();
  for (int base = 0; base < nA; base += 32) {
    const int a = base + lane;
    const bool valid = a < nA;
    const int e = valid ? R.sel_e[a] : MM_MAX_EXPERTS + lane;   // idle lanes match no one
    const unsigned mask = __match_any_sync(0xffffffffu, e);
    const unsigned below = mask & ((1u << lane) - 1u);
    const int prior = valid ? R.cnt[e] : 0;
    __syncwarp();
    if (valid) {
      R.rank[a] = prior + __popc(below);
      if (below == 0u) R.cnt[e] = prior + __popc(mask);
    }
    __syncwarp();
  }
  const unsigned lt = (1u << lane) - 1u;
  const int c0 = lane < E ? R.cnt[lane] : 0;
  const int c1 = lane + 32 < E ? R.cnt[lane + 32] : 0;
  int s0 = c0, s1 = c1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n0 = __shfl_up_sync(0xffffffffu, s0, o);
    const int n1 = __shfl_up_sync(0xffffffffu, s1, o);
    if (lane >= o) { s0 += n0; s1 += n1; }
  }
  const int tot0 = __shfl_sync(0xffffffffu, s0, 31);
  if (lane < E) R.e_start[lane] = s0 - c0;
  if (lane + 32 < E) R.e_start[lane + 32] = tot0 + s1 - c1;
  const unsigned b0 = __ballot_sync(0xffffffffu, c0 > 0);
  const unsigned b1 = __ballot_sync(0xffffffffu, c1 > 0);
  const int p0 = __popc(b0 & lt), p1 = __popc(b0) + __popc(b1 & lt);
  if (lane < E) R.slot_of[lane] = c0 > 0 ? p0 : -1;
  if (lane + 32 < E) R.slot_of[lane + 32] = c1 > 0 ? p1 : -1;
  if (c0 > 0) R.touched[p0] = lane;
  if (c1 > 0) R.touched[p1] = lane + 32;
  if (lane == 0) {
    R.n_touched = __popc(b0) + __popc(b1);
    R.nA = nA;
    R.e_start[E] = nA;
  }
  __syncwarp();
  for (int a = lane; a < nA; a += 32) R.by_e[R.e_start[R.sel_e[a]] + R.rank[a]] = a;
}

// Dense FFN: one weight set, every token, alpha 1.
template <int MAXT>
__device__ __forceinline__ void route_dense(SmallRoute<MAXT>& R, int T, int tid) {
  if (tid < T) {
    R.sel_e[tid] = 0;
    R.sel_a[tid] = 1.0f;
    R.by_e[tid] = tid;
  }
  if (tid == 0) {
    R.nA = T;
    R.n_touched = 1;
    R.touched[0] = 0;
    R.slot_of[0] = 0;
    R.cnt[0] = T;
    R.e_start[0] = 0;
    R.e_start[1] = T;
  }
}

// Block 0's routing outputs: topk_idx, topk_w and
// aux = E * coef * sum_e (count_e / T)(P_e / T)  (lesson 13 §1.6), by one warp;
// with a router variant also the probabilities, lse and
// z-loss = z_coef * (1/T) sum_t lse_t^2 (fixed summation order).
template <int MAXT>
__device__ __forceinline__ void route_outputs(const SmallRoute<MAXT>& R, int T, int E, float coef,
                                              int32_t* topk_idx, float* topk_w, float* aux_loss,
                                              int tid, int nthreads, int aux_warp,
                                              const RouterVariant* rv = nullptr) {
  for (int a = tid; a < R.nA; a += nthreads) {
    topk_idx[a] = R.sel_e[a];
    topk_w[a] = R.sel_a[a];
  }
  if (rv != nullptr) {
    if (rv->probs != nullptr)
      for (int i = tid; i < T * E; i += nthreads) rv->probs[i] = R.prob[i / E][i % E];
    if (rv->lse != nullptr)
      for (int t = tid; t < T; t += nthreads) rv->lse[t] = R.lse[t];
    if (rv->z_loss != nullptr && (tid >> 5) == aux_warp) {
      const int lane = tid & 31;
      float zs = 0.f;
      for (int t = lane; t < T; t += 32) zs = fmaf(R.lse[t], R.lse[t], zs);
      zs = warp_allsum_f(zs);
      if (lane == 0) *rv->z_loss = rv->z_coef * zs / static_cast<float>(T);
    }
  }
  if ((tid >> 5) == aux_warp) {
    const int lane = tid & 31;
    float acc = 0.f;
    for (int e = lane; e < E; e += 32) {
      float Pe = 0.f;
      for (int t = 0; t < T; ++t) Pe += R.prob[t][e];
      acc = fmaf(static_cast<float>(R.cnt[e]), Pe, acc);
    }
    acc = warp_allsum_f(acc);
    const float invT = 1.0f / static_cast<float>(T);
    if (lane == 0) *aux_loss = static_cast<float>(E) * coef * acc * invT * invT;
  }
}

}  // namespace mm
