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
};

__device__ __forceinline__ float warp_allsum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One thread per token t (t = first, first + stride, ...): R.prob[t][:]
// holds the logits on entry and the probabilities on exit.  Softmax with the
// maximum subtracted (fast exponential, one reciprocal); then k arg-max passes in expert order with a strict
// comparison, so that of equal probabilities the lower expert index is taken
// first; alpha = p / (sum_S p + 1e-20).
template <int MAXT>
__device__ __forceinline__ void route_softmax_topk(SmallRoute<MAXT>& R, int T, int E, int k,
                                                   const float* bias, int first, int stride) {
  for (int t = first; t < T; t += stride) {
    float* row = R.prob[t];
    float m = -INFINITY;
    for (int e = 0; e < E; ++e) {
      const float r = row[e] + bias[e];
      row[e] = r;
      m = fmaxf(m, r);
    }
    float z = 0.f;
    for (int e = 0; e < E; ++e) {
      const float x = __expf(row[e] - m);
      row[e] = x;
      z += x;
    }
    const float rz = 1.0f / z;
    for (int e = 0; e < E; ++e) row[e] *= rz;
    uint64_t taken = 0;
    float sel_sum = 0.f;
    for (int s = 0; s < k; ++s) {
      float bp = -1.f;
      int be = 0;
      for (int e = 0; e < E; ++e) {
        const float p = row[e];
        if (!((taken >> e) & 1ull) && p > bp) { bp = p; be = e; }
      }
      taken |= 1ull << be;
      sel_sum += bp;
      R.sel_e[t * k + s] = be;
      R.sel_a[t * k + s] = bp;
    }
    const float inv = sel_sum + 1e-20f;
    for (int s = 0; s < k; ++s) R.sel_a[t * k + s] = R.sel_a[t * k + s] / inv;
  }
}

// The same on one warp per token (t = first_warp, first_warp + nwarps, ...):
// lane l holds experts l and l + 32 in registers; the maximum and the sum of
// the exponentials are warp reductions, and each of the k selections is a
// warp arg-max (larger probability, else lower expert index).  Latency-bound
// calls (a few tokens) take this form; the sum runs in a different order from
// route_softmax_topk's, so probabilities can differ in their last bits.
template <int MAXT>
__device__ __forceinline__ void route_softmax_topk_warp(SmallRoute<MAXT>& R, int T, int E, int k,
                                                        const float* bias, int first_warp,
                                                        int nwarps, int lane) {
  for (int t = first_warp; t < T; t += nwarps) {
    float* row = R.prob[t];
    const bool v0 = lane < E, v1 = lane + 32 < E;
    const float r0 = v0 ? row[lane] + bias[lane] : -INFINITY;
    const float r1 = v1 ? row[lane + 32] + bias[lane + 32] : -INFINITY;
    float m = fmaxf(r0, r1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float x0 = v0 ? __expf(r0 - m) : 0.f;
    const float x1 = v1 ? __expf(r1 - m) : 0.f;
    const float rz = 1.0f / warp_allsum_f(x0 + x1);
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
// aux = E * coef * sum_e (count_e / T)(P_e / T)  (lesson 13 §1.6), by one warp.
template <int MAXT>
__device__ __forceinline__ void route_outputs(const SmallRoute<MAXT>& R, int T, int E, float coef,
                                              int32_t* topk_idx, float* topk_w, float* aux_loss,
                                              int tid, int nthreads, int aux_warp) {
  for (int a = tid; a < R.nA; a += nthreads) {
    topk_idx[a] = R.sel_e[a];
    topk_w[a] = R.sel_a[a];
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
