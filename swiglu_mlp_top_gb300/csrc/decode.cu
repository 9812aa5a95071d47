// Decode-sized forward (T <= kDecodeMaxT tokens, bf16): one cooperative
// weight-streaming kernel on the CUDA cores.  Every weight row is read from
// HBM once, by the bulk-copy engine into shared memory; for the MoE only the
// experts some token selected are read.
//
//   route (MoE)  logits, softmax, top-k, alpha (lesson 13 §1.5, chapter 4
//                §4.3): small at this size, so every CTA computes it for all
//                T tokens with the same code and order, and all CTAs agree;
//                block 0 writes topk_idx, topk_w and the aux loss (lesson 13 §1.6)
//   gate/up      h[a, i] = SiLU(Wg_e[i] . x_t) * (Wu_e[i] . x_t) for every
//                assignment a = (t, s) of expert e, fp32  (lesson 13 §0/§1.2)
//   grid barrier (h complete)
//   down         y[t, j] = sum_s alpha_{t,s} (Wd_{e_s}[j] . h[t, s]) in slot
//                order, fp32, rounded once       (lesson 13 §0 MoE equation)
//
// Each CTA issues the bulk copies of its first gate/up slices and of its
// first Wd rows as soon as it knows the touched experts (dense: at entry), so
// the down weights are in shared memory by the time the barrier opens.  The
// products use packed fp32 FMA (two lanes of fp32 per instruction) on
// operands widened from bf16; every dot product accumulates in fp32.
#include "route_small.cuh"

namespace mm {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kUpRows = kDecWarps;          // Wg / Wu rows per gate/up unit (one per warp)
constexpr int kDnRows = 4;                  // output columns (Wd rows) per down unit
constexpr int kMaxRing = 6;                 // gate/up stages
constexpr int kMaxWdSlots = 4;              // Wd buffers
constexpr int kMaxHRows = 32;               // h rows staged at once
constexpr size_t kDecSmemBudget = 200 * 1024;
constexpr size_t kDecSmemTwoPerSm = 100 * 1024;

// Shared-memory plan, chosen on the host.  Phase 1 holds x (fp32) at offset 0
// and the gate/up ring after it (Wr sits at the ring's start during the
// routing); phase 2 reuses offset 0 for the staged h rows.  The Wd buffers
// live above both, since they fill during phase 1.
struct DecPlan {
  int ring, wd_slots, h_rows, per_sm;
  uint32_t ring_off, wd_off, total;
};

struct DecodeArgs {
  const void* x;            // [T, H] bf16
  const void* Wr;           // [E, H] bf16, or nullptr (dense)
  const float* bias;        // [E] or nullptr
  PtrArray wg, wu, wd;      // per expert
  int T, H, I, E, k;
  float coef;
  int32_t* topk_idx;        // written by block 0 (MoE)
  float* topk_w;
  float* aux_loss;
  float* h;                 // [T*k, I] fp32 scratch (dense: [T, I])
  void* y;                  // [T, H] bf16
  WsHeader* hdr;
  DecPlan plan;
  RouterVariant rv;         // router noise, z-loss, saved statistics (MoE)
};


// 1-D bulk copy global -> this CTA's shared memory, completion on `bar`.
__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// The same with an L2 cache policy (the streamed weights: evict first).
__device__ __forceinline__ void bulk_load_hint(void* sdst, const void* gsrc, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// One gate/up row i of expert e for m <= NT assignments (list): the lanes
// split H in chunks of 8, the row's Wg and Wu chunks are widened once and
// applied to every token's fp32 x chunk.
template <int NT>
__device__ __forceinline__ void gateup_row(const __nv_bfloat16* grow, const __nv_bfloat16* urow,
                                           const float* xs, const int* list, int m, int kk, int H,
                                           int I, int i, float* hout, int lane) {
  const float* xr[NT];
#pragma unroll
  for (int tt = 0; tt < NT; ++tt) xr[tt] = xs + static_cast<size_t>(list[tt < m ? tt : m - 1] / kk) * H;
  u64 ga[NT], ua[NT];
#pragma unroll
  for (int tt = 0; tt < NT; ++tt) ga[tt] = ua[tt] = 0ull;
  for (int c = lane; c < H / 8; c += 32) {
    const uint4 gw = *reinterpret_cast<const uint4*>(grow + c * 8);
    const uint4 uw = *reinterpret_cast<const uint4*>(urow + c * 8);
    const u64 g0 = bf2(gw.x), g1 = bf2(gw.y), g2 = bf2(gw.z), g3 = bf2(gw.w);
    const u64 u0 = bf2(uw.x), u1 = bf2(uw.y), u2 = bf2(uw.z), u3 = bf2(uw.w);
#pragma unroll
    for (int tt = 0; tt < NT; ++tt) {
      const ulonglong2 xa = *reinterpret_cast<const ulonglong2*>(xr[tt] + c * 8);
      const ulonglong2 xb = *reinterpret_cast<const ulonglong2*>(xr[tt] + c * 8 + 4);
      ga[tt] = ffma2(g0, xa.x, ga[tt]);
      ua[tt] = ffma2(u0, xa.x, ua[tt]);
      ga[tt] = ffma2(g1, xa.y, ga[tt]);
      ua[tt] = ffma2(u1, xa.y, ua[tt]);
      ga[tt] = ffma2(g2, xb.x, ga[tt]);
      ua[tt] = ffma2(u2, xb.x, ua[tt]);
      ga[tt] = ffma2(g3, xb.y, ga[tt]);
      ua[tt] = ffma2(u3, xb.y, ua[tt]);
    }
  }
  float v[2 * NT];
#pragma unroll
  for (int tt = 0; tt < NT; ++tt) {
    v[2 * tt] = hsum2(ga[tt]);
    v[2 * tt + 1] = hsum2(ua[tt]);
  }
  const float r = reduce_scatter<2 * NT>(v, lane);   // value 2t = g_t, 2t + 1 = u_t
  constexpr int span = 32 / (2 * NT);                // lanes holding one value
  const float u = __shfl_down_sync(0xffffffffu, r, span);
  if (lane % (2 * span) == 0) {
    const int tt = lane / (2 * span);
    if (tt < m) hout[static_cast<size_t>(list[tt]) * I + i] = silu_f32(r) * u;
  }
}

// One Wd row (output column j) against m <= NA staged h rows; the result for
// staged row sbase + q goes to part[ids[q]][jl].
template <int NA>
__device__ __forceinline__ void down_row(const __nv_bfloat16* wrow, const float* hst, int sbase,
                                         const int* ids, int m, int I, int jl,
                                         float (*part)[kDnRows], int lane) {
  const float* hr[NA];
#pragma unroll
  for (int q = 0; q < NA; ++q) hr[q] = hst + static_cast<size_t>(sbase + (q < m ? q : m - 1)) * I;
  // two 8-element chunks per step into two accumulator sets, so that the
  // loads of one overlap the products of the other (fixed order: the sets are
  // added at the end)
  u64 acc[2][NA];
#pragma unroll
  for (int q = 0; q < NA; ++q) acc[0][q] = acc[1][q] = 0ull;
  for (int c0 = lane; c0 < I / 8; c0 += 64) {
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int c = c0 + 32 * h2;
      if (c >= I / 8) break;
      const uint4 w = *reinterpret_cast<const uint4*>(wrow + c * 8);
      const u64 w0 = bf2(w.x), w1 = bf2(w.y), w2 = bf2(w.z), w3 = bf2(w.w);
#pragma unroll
      for (int q = 0; q < NA; ++q) {
        const ulonglong2 ha = *reinterpret_cast<const ulonglong2*>(hr[q] + c * 8);
        const ulonglong2 hb = *reinterpret_cast<const ulonglong2*>(hr[q] + c * 8 + 4);
        acc[h2][q] = ffma2(w0, ha.x, acc[h2][q]);
        acc[h2][q] = ffma2(w1, ha.y, acc[h2][q]);
        acc[h2][q] = ffma2(w2, hb.x, acc[h2][q]);
        acc[h2][q] = ffma2(w3, hb.y, acc[h2][q]);
      }
    }
  }
  float v[NA];
#pragma unroll
  for (int q = 0; q < NA; ++q) v[q] = hsum2(acc[0][q]) + hsum2(acc[1][q]);
  const float r = reduce_scatter<NA>(v, lane);
  constexpr int span = 32 / NA;
  if (lane % span == 0) {
    const int q = lane / span;
    if (q < m) part[ids[q]][jl] = r;
  }
}

// MoE routing of all T tokens.  Logits: (token, expert) pairs, four per warp
// at a time, lanes split H, fp32; then softmax / top-k (one warp per token)
// and the grouping by expert (route_small.cuh).
__device__ void decode_route(const DecodeArgs& A, const float* xs, const __nv_bfloat16* Wr,
                             const float* bias, SmallRoute<kDecodeMaxT>& R) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int E = A.E, k = A.k, H = A.H;
  const int pairs = A.T * E;
  for (int p0 = warp * 4; p0 < pairs; p0 += kDecWarps * 4) {
    const float* xr[4];
    const __nv_bfloat16* wr[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int p = min(p0 + q, pairs - 1);
      const int t = p / E;
      xr[q] = xs + static_cast<size_t>(t) * H;
      wr[q] = Wr + static_cast<size_t>(p - t * E) * H;
    }
    u64 acc[4] = {0ull, 0ull, 0ull, 0ull};
    for (int c = lane; c < H / 8; c += 32) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 w = *reinterpret_cast<const uint4*>(wr[q] + c * 8);
        const ulonglong2 xa = *reinterpret_cast<const ulonglong2*>(xr[q] + c * 8);
        const ulonglong2 xb = *reinterpret_cast<const ulonglong2*>(xr[q] + c * 8 + 4);
        acc[q] = ffma2(bf2(w.x), xa.x, acc[q]);
        acc[q] = ffma2(bf2(w.y), xa.y, acc[q]);
        acc[q] = ffma2(bf2(w.z), xb.x, acc[q]);
        acc[q] = ffma2(bf2(w.w), xb.y, acc[q]);
      }
    }
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = hsum2(acc[q]);
    const float r = reduce_scatter<4>(v, lane);
    if ((lane & 7) == 0) {
      const int p = p0 + (lane >> 3);
      if (p < pairs) R.prob[p / E][p % E] = r;
    }
  }
  __syncthreads();
  route_softmax_topk_warp(R, A.T, E, k, bias, warp, kDecWarps, lane, A.rv.noise);
  __syncthreads();
  if (warp == 0) route_group(R, A.T * k, E, lane);
  __syncthreads();
}

__global__ void __launch_bounds__(kDecThreads)
decode_ffn_kernel(const DecodeArgs A) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ SmallRoute<kDecodeMaxT> R;
  __shared__ __align__(8) uint64_t bar[kMaxRing + kMaxWdSlots + 1];
  __shared__ float part[kDecodeMaxT * MM_MAX_TOPK][kDnRows];
  __shared__ float s_bias[MM_MAX_EXPERTS];
  const DecPlan& P = A.plan;
  const int H = A.H, I = A.I;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x;
  const bool moe = A.Wr != nullptr;
  const int kk = moe ? A.k : 1;
  float* xs = reinterpret_cast<float*>(dsm);
  unsigned char* ring = dsm + P.ring_off;
  unsigned char* wdbuf = dsm + P.wd_off;
  float* hst = reinterpret_cast<float*>(dsm);
  uint64_t* ring_bar = bar;
  uint64_t* wd_bar = bar + kMaxRing;
  uint64_t* h_bar = bar + kMaxRing + kMaxWdSlots;
  const size_t slice = static_cast<size_t>(kUpRows) * H * 2;   // one of Wg / Wu
  const size_t stage = 2 * slice;
  const size_t slot = static_cast<size_t>(kDnRows) * I * 2;
  const int slices = I / kUpRows;
  const int dn_units = H / kDnRows;
  const int my_dn = blockIdx.x < dn_units ? (dn_units - blockIdx.x + G - 1) / G : 0;

  // copies issued (thread 0) and consumed (every thread)
  int up_issued = 0, wd_issued = 0, h_issued = 0;
  int up_used = 0, wd_used = 0, h_used = 0;
  int n_touched = 1, my_up = 0, my_wd = 0;

  const uint64_t pol = l2_evict_first_policy();     // weights: read once per launch
  auto issue_up = [&](int it) {
    const int u = blockIdx.x + it * G;
    const int e = moe ? R.touched[u / slices] : 0;
    const int r0 = (u % slices) * kUpRows;
    const uint32_t bytes = static_cast<uint32_t>(slice);
    unsigned char* dst = ring + (it % P.ring) * stage;
    uint64_t* b = &ring_bar[it % P.ring];
    mbar_arrive_expect_tx(b, 2 * bytes);
    bulk_load_hint(dst, static_cast<const __nv_bfloat16*>(A.wg.p[e]) + static_cast<size_t>(r0) * H,
                   bytes, b, pol);
    bulk_load_hint(dst + slice, static_cast<const __nv_bfloat16*>(A.wu.p[e]) + static_cast<size_t>(r0) * H,
                   bytes, b, pol);
    ++up_issued;
  };
  auto issue_wd = [&](int q) {
    const int r = q / n_touched, ti = q - r * n_touched;
    const int du = blockIdx.x + r * G;
    const int e = moe ? R.touched[ti] : 0;
    uint64_t* b = &wd_bar[q % P.wd_slots];
    mbar_arrive_expect_tx(b, static_cast<uint32_t>(slot));
    bulk_load_hint(wdbuf + (q % P.wd_slots) * slot,
                   static_cast<const __nv_bfloat16*>(A.wd.p[e]) + static_cast<size_t>(du) * kDnRows * I,
                   static_cast<uint32_t>(slot), b, pol);
    ++wd_issued;
  };
  auto issue_first = [&]() {
    for (int it = 0; it < P.ring && it < my_up; ++it) issue_up(it);
    for (int q = 0; q < P.wd_slots && q < my_wd; ++q) issue_wd(q);
  };

  if (tid == 0) {
    for (int q = 0; q < kMaxRing + kMaxWdSlots + 1; ++q) mbar_init(&bar[q], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (!moe) {                                 // dense: the weights needed are known now
    my_up = blockIdx.x < slices ? (slices - blockIdx.x + G - 1) / G : 0;
    my_wd = my_dn;
    if (tid == 0) issue_first();
  }
  {
    // x as fp32; Wr (bf16) at the ring's start when it fits; logit bias
    const bool wr_smem = moe && static_cast<size_t>(A.E) * H * 2 <= P.ring * stage;
    const int nx = A.T * H / 8;
    const int nw = wr_smem ? A.E * H / 8 : 0;
    for (int i = tid; i < nx + nw; i += kDecThreads) {
      if (i < nx) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(A.x) + i);
        ulonglong2 lo, hi;
        lo.x = bf2(w.x); lo.y = bf2(w.y); hi.x = bf2(w.z); hi.y = bf2(w.w);
        reinterpret_cast<ulonglong2*>(xs)[2 * i] = lo;
        reinterpret_cast<ulonglong2*>(xs)[2 * i + 1] = hi;
      } else {
        reinterpret_cast<uint4*>(ring)[i - nx] = __ldg(reinterpret_cast<const uint4*>(A.Wr) + (i - nx));
      }
    }
    if (tid < MM_MAX_EXPERTS) s_bias[tid] = (moe && A.bias != nullptr && tid < A.E) ? A.bias[tid] : 0.f;
    __syncthreads();
    if (moe) {
      decode_route(A, xs, wr_smem ? reinterpret_cast<const __nv_bfloat16*>(ring)
                                  : static_cast<const __nv_bfloat16*>(A.Wr), s_bias, R);
    } else {
      route_dense(R, A.T, tid);
      __syncthreads();
    }
  }
  if (moe) {
    n_touched = R.n_touched;
    const int up_units = n_touched * slices;
    my_up = blockIdx.x < up_units ? (up_units - blockIdx.x + G - 1) / G : 0;
    my_wd = my_dn * n_touched;
    if (blockIdx.x == 0)
      route_outputs(R, A.T, A.E, A.coef, A.topk_idx, A.topk_w, A.aux_loss, tid, kDecThreads, 1,
                    &A.rv);
    __syncthreads();                          // Wr in the ring is no longer read
    if (tid == 0) {
      fence_proxy_async_smem();
      issue_first();
    }
  }

  // ---- gate/up: this CTA's units blockIdx.x + it*G; warp w owns row w
  bool ok = true;
  for (int it = 0; ok && it < my_up; ++it) {
    const int s = it % P.ring;
    ok = __syncthreads_and(mbar_wait(&ring_bar[s], (it / P.ring) & 1, nullptr, A.hdr, 20));
    if (!ok) break;
    up_used = it + 1;
    const int u = blockIdx.x + it * G;
    const int e = moe ? R.touched[u / slices] : 0;
    const int i = (u % slices) * kUpRows + warp;
    const __nv_bfloat16* grow = reinterpret_cast<const __nv_bfloat16*>(ring + s * stage) + warp * H;
    const __nv_bfloat16* urow = grow + kUpRows * H;
    const int* list = R.by_e + R.e_start[e];  // the assignments of expert e, in order
    const int n = R.e_start[e + 1] - R.e_start[e];
    for (int g0 = 0; g0 < n; g0 += 8) {
      const int m = min(8, n - g0);
      if (m == 1)
        gateup_row<1>(grow, urow, xs, list + g0, m, kk, H, I, i, A.h, lane);
      else if (m == 2)
        gateup_row<2>(grow, urow, xs, list + g0, m, kk, H, I, i, A.h, lane);
      else if (m <= 4)
        gateup_row<4>(grow, urow, xs, list + g0, m, kk, H, I, i, A.h, lane);
      else
        gateup_row<8>(grow, urow, xs, list + g0, m, kk, H, I, i, A.h, lane);
    }
    __syncthreads();                          // stage s is no longer read
    if (tid == 0 && it + P.ring < my_up) {
      fence_proxy_async_smem();
      issue_up(it + P.ring);
    }
  }

  // ---- every h row written before any CTA reads it
  unsigned ticket = 0xffffffffu;
  if (ok) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    ok = grid_barrier(A.hdr, 24, 1, &ticket);
  }

  // ---- down: unit = kDnRows output columns, every touched expert
  const int nA = R.nA;
  const bool h_once = nA <= P.h_rows;         // one stage serves every unit
  for (int r = 0; ok && r < my_dn; ++r) {
    const int j0 = (blockIdx.x + r * G) * kDnRows;
    int ti = 0;
    __syncthreads();                          // part[] of the previous unit is read
    for (int q0 = 0; ok && q0 < nA; q0 += P.h_rows) {
      const int q1 = min(nA, q0 + P.h_rows);
      if (!(h_once && r > 0)) {
        __syncthreads();                      // the previous stage is no longer read
        if (tid == 0) {
          fence_proxy_async_smem();
          asm volatile("fence.proxy.async.global;" ::: "memory");
          mbar_arrive_expect_tx(h_bar, static_cast<uint32_t>(q1 - q0) * I * 4);
          for (int q = q0; q < q1; ++q)
            bulk_load(hst + static_cast<size_t>(q - q0) * I, A.h + static_cast<size_t>(R.by_e[q]) * I,
                      static_cast<uint32_t>(I) * 4, h_bar);
          ++h_issued;
        }
        ok = __syncthreads_and(mbar_wait(h_bar, h_used & 1, nullptr, A.hdr, 21));
        if (!ok) break;
        ++h_used;
      }
      while (ti < n_touched) {
        const int e = R.touched[ti];
        if (R.e_start[e] >= q1) break;        // its rows come with a later stage
        const int ea = max(R.e_start[e], q0), eb = min(R.e_start[e + 1], q1);
        const int q = r * n_touched + ti;     // Wd copy index
        const int b = q % P.wd_slots;
        if (q >= wd_used) {
          ok = __syncthreads_and(mbar_wait(&wd_bar[b], (q / P.wd_slots) & 1, nullptr, A.hdr, 22));
          if (!ok) break;
          wd_used = q + 1;
        }
        // warp w: column w % kDnRows; the expert's staged rows four at a
        // time, round-robin over the warps of that column
        constexpr int kWarpsPerCol = kDecWarps / kDnRows;
        const int jl = warp % kDnRows;
        const __nv_bfloat16* wrow = reinterpret_cast<const __nv_bfloat16*>(wdbuf + b * slot) + jl * I;
        for (int g0 = ea + (warp / kDnRows) * 4; g0 < eb; g0 += 4 * kWarpsPerCol) {
          const int m = min(4, eb - g0);
          if (m == 1)
            down_row<1>(wrow, hst, g0 - q0, R.by_e + g0, m, I, jl, part, lane);
          else if (m == 2)
            down_row<2>(wrow, hst, g0 - q0, R.by_e + g0, m, I, jl, part, lane);
          else
            down_row<4>(wrow, hst, g0 - q0, R.by_e + g0, m, I, jl, part, lane);
        }
        if (R.e_start[e + 1] > q1) break;     // e continues in the next stage
        __syncthreads();                      // e is done: its buffer takes a later copy
        if (tid == 0 && q + P.wd_slots < my_wd) {
          fence_proxy_async_smem();
          issue_wd(q + P.wd_slots);
        }
        ++ti;
      }
    }
    __syncthreads();
    if (!ok) break;
    for (int q = tid; q < A.T * kDnRows; q += kDecThreads) {
      const int t = q / kDnRows, jl = q % kDnRows;
      float v = 0.f;
      for (int s = 0; s < kk; ++s) v = fmaf(R.sel_a[t * kk + s], part[t * kk + s][jl], v);
      static_cast<__nv_bfloat16*>(A.y)[static_cast<size_t>(t) * H + j0 + jl] = __float2bfloat16_rn(v);
    }
  }
  if (tid == 0) {
    // copies still in flight (a unit not reached after a failed wait) land
    // before the CTA exits
    for (int it = up_used; it < up_issued; ++it)
      mbar_wait(&ring_bar[it % P.ring], (it / P.ring) & 1, nullptr, nullptr, 25);
    for (int q = wd_used; q < wd_issued; ++q)
      mbar_wait(&wd_bar[q % P.wd_slots], (q / P.wd_slots) & 1, nullptr, nullptr, 25);
    if (h_issued > h_used) mbar_wait(h_bar, h_used & 1, nullptr, nullptr, 25);
    grid_barrier_reset(A.hdr, ticket);
  }
}

namespace {

size_t round128(size_t v) { return (v + 127) & ~size_t(127); }

// Shared-memory plan: as many gate/up stages and Wd buffers as fit; two CTAs
// per SM when the smallest plan leaves room for a second one.
DecPlan decode_plan(int T, int H, int I, int nA) {
  const size_t x = round128(static_cast<size_t>(T) * H * 4);
  const size_t stage = 2 * static_cast<size_t>(kUpRows) * H * 2;
  const size_t slot = static_cast<size_t>(kDnRows) * I * 2;
  const size_t hrow = static_cast<size_t>(I) * 4;
  auto layout = [&](DecPlan& p) {
    p.ring_off = static_cast<uint32_t>(x);
    const size_t a = x + p.ring * stage;
    const size_t b = static_cast<size_t>(p.h_rows) * hrow;
    p.wd_off = static_cast<uint32_t>(round128(a > b ? a : b));
    return static_cast<size_t>(p.wd_off) + p.wd_slots * slot;
  };
  DecPlan p;
  p.ring = 2;
  p.wd_slots = 2;
  p.h_rows = nA < kMaxHRows ? nA : kMaxHRows;
  p.per_sm = 1;
  while (p.h_rows > 1 && layout(p) > kDecSmemBudget) --p.h_rows;
  size_t total = layout(p);
  if (total > kDecSmemBudget) {
    p.total = 0;                              // does not fit
    return p;
  }
  if (total <= kDecSmemTwoPerSm) {
    p.per_sm = 2;
  } else {
    // grow the gate/up ring and the Wd buffers in turn while they fit
    const int order[6][2] = {{3, 2}, {3, 3}, {4, 3}, {4, 4}, {5, 4}, {6, 4}};
    for (const auto& o : order) {
      DecPlan q = p;
      q.ring = o[0];
      q.wd_slots = o[1];
      if (layout(q) <= kDecSmemBudget) p = q;
    }
    total = layout(p);
  }
  p.total = static_cast<uint32_t>(total);
  return p;
}

}  // namespace

size_t decode_smem_bytes(int T, int H, int I, int E, int k) {
  const DecPlan p = decode_plan(T, H, I, T * (E > 1 ? k : 1));
  return p.total == 0 ? ~size_t(0) : p.total;
}

cudaError_t launch_decode_ffn(const void* x, const void* Wr, const float* bias,
                              const void* const* Wg, const void* const* Wu, const void* const* Wd,
                              int T, int H, int I, int E, int k, float coef, int32_t* topk_idx,
                              float* topk_w, float* aux_loss, void* hbuf, void* y, WsHeader* hdr,
                              cudaStream_t st, const RouterVariant* rv) {
  DecodeArgs A;
  memset(&A, 0, sizeof(A));
  if (rv != nullptr) A.rv = *rv;
  A.x = x;
  A.Wr = Wr;
  A.bias = bias;
  const int nw = (Wr != nullptr) ? E : 1;
  for (int e = 0; e < nw; ++e) {
    A.wg.p[e] = Wg[e];
    A.wu.p[e] = Wu[e];
    A.wd.p[e] = Wd[e];
  }
  A.T = T; A.H = H; A.I = I; A.E = nw; A.k = (Wr != nullptr) ? k : 1; A.coef = coef;
  A.topk_idx = topk_idx; A.topk_w = topk_w; A.aux_loss = aux_loss;
  A.h = static_cast<float*>(hbuf); A.y = y; A.hdr = hdr;
  A.plan = decode_plan(T, H, I, T * A.k);
  if (A.plan.total == 0) return cudaErrorInvalidValue;
  const size_t smem = A.plan.total;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(decode_ffn_kernel), smem);
  if (e != cudaSuccess) return e;
  // every CTA must be resident (grid barrier)
  int fit = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, decode_ffn_kernel, kDecThreads, smem);
  if (e != cudaSuccess) return e;
  if (fit < 1) return cudaErrorInvalidConfiguration;
  const int grid = num_sms() * (fit < A.plan.per_sm ? fit : A.plan.per_sm);
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_ffn_kernel, A);
}

}  // namespace mm
