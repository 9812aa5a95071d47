// Backward pass of the MoE layer outside the GEMMs: the dispatch of the
// assignments into expert groups, and the router backward.
//
// The router gradient follows p-chao.com "MiniMind 学习笔记 08" §7 (the
// selection has no gradient; the router learns through the selected
// weights) and chapter 4 §4.4 of minimind3.com (in aux, the load f_e is not
// differentiable, the mean probability P_e is):
//   alpha_s = p_{S_s} / Z, Z = sum_S p + 1e-20
//       dp_{S_s} += (dalpha_s - sum_j dalpha_j alpha_j) / Z
//   aux = E coef sum_e (count_e / T)(sum_t p_{t,e} / T)
//       dp_{t,e} += d_aux E coef count_e / T^2
//   softmax:  dr_e = p_e (dp_e - sum_j p_j dp_j)
//   z-loss = z_coef / T sum_t lse_t^2:  dr_e += d_z 2 z_coef lse_t p_e / T
//   dx_t = sum_s dx_{t,s} (slot order) + sum_e dr_e Wr_e;  dWr = dr^T x;  d_bias = sum_t dr_t
// Every sum runs in a fixed order; the results are deterministic.
#include <algorithm>
#include <cstring>

#include "mm_kernels.cuh"

namespace mm {

constexpr int kBwdTok = 64;           // tokens per block (count, dispatch, router backward)
constexpr int kBwdThreads = 256;

__device__ __forceinline__ float bw_warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Per block of 64 tokens: assignments per expert.
__global__ void __launch_bounds__(kBwdThreads)
bwd_count_kernel(const int32_t* __restrict__ topk_idx, int64_t T, int E, int k,
                 int32_t* __restrict__ blk_cnt) {
  pdl_enter();
  __shared__ int cnt[MM_MAX_EXPERTS];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kBwdTok;
  const int na = static_cast<int>(T - t0 < kBwdTok ? T - t0 : kBwdTok) * k;
  for (int a = threadIdx.x; a < na; a += blockDim.x) atomicAdd(&cnt[topk_idx[t0 * k + a]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) blk_cnt[static_cast<int64_t>(blockIdx.x) * E + e] = cnt[e];
}

// Block b owns the assignments of tokens [64 b, 64 b + 64).  From every
// block's counts it derives the expert totals, the padded group offsets
// (each group starts on a multiple of kBwAlign rows) and its own base in
// each group; an assignment's row is offset[e] + base[e] + its rank among
// the block's assignments to e in (token, slot) order.  It writes perm /
// pos and copies the x and dy rows; block 0 also writes offsets and counts
// and zeroes the padding rows.
template <typename Tin>
__global__ void __launch_bounds__(kBwdThreads)
bwd_dispatch_kernel(const Tin* __restrict__ x, const Tin* __restrict__ dy,
                    const int32_t* __restrict__ topk_idx, int64_t T, int H, int E, int k,
                    const int32_t* __restrict__ blk_cnt, BwdDispatchOut o, int stage) {
  pdl_enter();
  __shared__ int s_tot[MM_MAX_EXPERTS], s_base[MM_MAX_EXPERTS], s_off[MM_MAX_EXPERTS + 1];
  __shared__ int s_run[MM_MAX_EXPERTS];
  __shared__ int s_pos[kBwdTok * MM_MAX_TOPK];
  __shared__ __align__(8) uint64_t rowbar;
  extern __shared__ __align__(128) unsigned char bwd_rows[];   // stage: x rows, then dy rows
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x, nblk = gridDim.x;
  const int64_t t0 = static_cast<int64_t>(b) * kBwdTok;
  const int ntok = static_cast<int>(T - t0 < kBwdTok ? T - t0 : kBwdTok);
  const int na = ntok * k;
  const uint32_t rowb = static_cast<uint32_t>(H) * sizeof(Tin);
  Tin* xs = reinterpret_cast<Tin*>(bwd_rows);
  Tin* ds = xs + static_cast<int64_t>(kBwdTok) * H;
  if (stage && tid == 0) {
    // the block's x and dy rows, one bulk copy each, while the ranks are worked out
    mbar_init(&rowbar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&rowbar, 2u * static_cast<uint32_t>(ntok) * rowb);
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(xs)), "l"(x + t0 * H), "r"(static_cast<uint32_t>(ntok) * rowb),
        "r"(smem_u32(&rowbar))
        : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(ds)), "l"(dy + t0 * H), "r"(static_cast<uint32_t>(ntok) * rowb),
        "r"(smem_u32(&rowbar))
        : "memory");
  }
  // totals and this block's base per expert: warp w takes experts w, w + 8,
  // ...; its lanes split the blocks (all loads in flight together) and a
  // warp reduction adds them (integers: any order gives the same sums)
  for (int e = warp; e < E; e += kBwdThreads / 32) {
    int all = 0, before = 0;
    for (int bb = lane; bb < nblk; bb += 32) {
      const int c = blk_cnt[static_cast<int64_t>(bb) * E + e];
      all += c;
      before += bb < b ? c : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      all += __shfl_xor_sync(0xffffffffu, all, o);
      before += __shfl_xor_sync(0xffffffffu, before, o);
    }
    if (lane == 0) {
      s_tot[e] = all;
      s_base[e] = before;
      s_run[e] = 0;
    }
  }
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < E; ++e) {
      s_off[e] = run;
      run += (s_tot[e] + kBwAlign - 1) / kBwAlign * kBwAlign;
    }
    s_off[E] = run;
  }
  __syncthreads();
  // ranks: warp 0 walks the block's assignments 32 at a time in order
  if (warp == 0) {
    for (int base = 0; base < na; base += 32) {
      const int a = base + lane;
      const bool valid = a < na;
      const int e = valid ? topk_idx[t0 * k + a] : MM_MAX_EXPERTS + lane;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const unsigned below = peers & ((1u << lane) - 1u);
      const int prior = valid ? s_run[e] : 0;
      __syncwarp();
      if (valid) {
        s_pos[a] = s_off[e] + s_base[e] + prior + __popc(below);
        if (below == 0u) s_run[e] = prior + __popc(peers);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  for (int a = tid; a < na; a += blockDim.x) {
    o.perm[s_pos[a]] = static_cast<int32_t>(t0 * k + a);
    o.pos[t0 * k + a] = s_pos[a];
  }
  constexpr int kVec = 16 / sizeof(Tin);
  const int nv = H / kVec;
  if (stage) {
    // rows: two bulk copies per assignment (x, dy), shared -> global
    const bool landed = __syncthreads_and(mbar_wait(&rowbar, 0, nullptr, o.hdr, 90));
    if (landed && tid < na) {
      for (int a = tid; a < na; a += kBwdThreads) {
        const int64_t d = static_cast<int64_t>(s_pos[a]) * H;
        bulk_store(static_cast<Tin*>(o.xp) + d, xs + static_cast<int64_t>(a / k) * H, rowb);
        bulk_store(static_cast<Tin*>(o.dyp) + d, ds + static_cast<int64_t>(a / k) * H, rowb);
      }
      bulk_commit();
      bulk_wait_all();
    }
  } else {
    // rows: one flat loop over (assignment, 16-byte vector) items, four in
    // flight per thread
    const int items = na * nv;
#pragma unroll 4
    for (int i = tid; i < items; i += kBwdThreads) {
      const int a = i / nv, v = i - a * nv;
      const int64_t t = t0 + a / k;
      const int64_t d = static_cast<int64_t>(s_pos[a]) * nv + v;
      reinterpret_cast<uint4*>(o.xp)[d] = reinterpret_cast<const uint4*>(x)[t * nv + v];
      reinterpret_cast<uint4*>(o.dyp)[d] = reinterpret_cast<const uint4*>(dy)[t * nv + v];
    }
  }
  if (b == 0) {
    for (int e = tid; e <= E; e += blockDim.x) o.offsets[e] = s_off[e];
    for (int e = tid; e < E; e += blockDim.x) o.counts[e] = s_tot[e];
    // padding rows of every group: zero x and dy rows, perm -1
    for (int e = 0; e < E; ++e) {
      const int p0 = s_off[e] + s_tot[e], p1 = s_off[e + 1];
      for (int r = p0 + warp; r < p1; r += kBwdThreads / 32) {
        if (lane == 0) o.perm[r] = -1;
        uint4* dx4 = reinterpret_cast<uint4*>(static_cast<Tin*>(o.xp) + static_cast<int64_t>(r) * H);
        uint4* dd4 = reinterpret_cast<uint4*>(static_cast<Tin*>(o.dyp) + static_cast<int64_t>(r) * H);
        for (int v = lane; v < nv; v += 32) {
          dx4[v] = make_uint4(0u, 0u, 0u, 0u);
          dd4[v] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
  }
}

// Four consecutive bf16 (8-byte aligned) as fp32, and back.
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  v[0] = __uint_as_float(raw.x << 16);
  v[1] = __uint_as_float(raw.x & 0xffff0000u);
  v[2] = __uint_as_float(raw.y << 16);
  v[3] = __uint_as_float(raw.y & 0xffff0000u);
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, const float4& a) {
  *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
}

// Router backward over blocks of 8 tokens (one warp per token: lane l holds
// experts l and l + 32): dr [T, E] and dx [T, H] (the k per-assignment rows
// in slot order plus dr Wr, by all the block's threads).  Small blocks keep
// many tokens in flight: each step is a short chain of dependent loads.
constexpr int kRbTok = 8;

template <typename Tin>
__global__ void __launch_bounds__(kBwdThreads)
router_bwd_kernel(const Tin* __restrict__ Wr, int64_t T, int H, int E, int k, const RouterBwd rb) {
  pdl_enter();
  __shared__ float s_dr[kRbTok * MM_MAX_EXPERTS];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kRbTok;
  const int ntok = static_cast<int>(T - t0 < kRbTok ? T - t0 : kRbTok);
  const float invT = 1.0f / static_cast<float>(T);
  const bool v0 = lane < E, v1 = lane + 32 < E;
  if (warp < ntok) {
    const int tl = warp;
    const int64_t t = t0 + tl;
    const float aux0 = v0 ? rb.d_aux * static_cast<float>(E) * rb.coef * static_cast<float>(rb.counts[lane]) * invT * invT : 0.f;
    const float aux1 = v1 ? rb.d_aux * static_cast<float>(E) * rb.coef * static_cast<float>(rb.counts[lane + 32]) * invT * invT : 0.f;
    const float p0 = v0 ? rb.probs[t * E + lane] : 0.f;
    const float p1 = v1 ? rb.probs[t * E + lane + 32] : 0.f;
    float dp0 = aux0, dp1 = aux1;
    // dalpha_s = sum of the row's partials (lane-strided, then a fixed tree)
    float Z = 0.f, c = 0.f;
    float da[MM_MAX_TOPK];
    int sel[MM_MAX_TOPK];
#pragma unroll
    for (int s = 0; s < MM_MAX_TOPK; ++s) {
      da[s] = 0.f;
      sel[s] = 0;
      if (s < k) {
        const float* part = rb.dalpha_part + static_cast<int64_t>(rb.pos[t * k + s]) * rb.n_parts;
        float v = 0.f;
        for (int j = lane; j < rb.n_parts; j += 32) v += part[j];
        da[s] = bw_warp_sum(v);
        sel[s] = rb.topk_idx[t * k + s];
        Z += __shfl_sync(0xffffffffu, sel[s] < 32 ? p0 : p1, sel[s] & 31);
        c = fmaf(da[s], rb.topk_w[t * k + s], c);
      }
    }
    Z += 1e-20f;
#pragma unroll
    for (int s = 0; s < MM_MAX_TOPK; ++s) {
      if (s < k) {
        const float g = (da[s] - c) / Z;
        if (sel[s] == lane) dp0 += g;
        if (sel[s] == lane + 32) dp1 += g;
      }
    }
    const float S = bw_warp_sum(p0 * dp0 + p1 * dp1);
    float dr0 = p0 * (dp0 - S), dr1 = p1 * (dp1 - S);
    if (rb.lse != nullptr) {
      const float zf = rb.d_z * 2.0f * rb.z_coef * rb.lse[t] * invT;
      dr0 = fmaf(zf, p0, dr0);
      dr1 = fmaf(zf, p1, dr1);
    }
    if (v0) { rb.dr[t * E + lane] = dr0; s_dr[tl * E + lane] = dr0; }
    if (v1) { rb.dr[t * E + lane + 32] = dr1; s_dr[tl * E + lane + 32] = dr1; }
  }
  __syncthreads();
  // dx_t = sum_s dxp[pos(t, s)] (slot order) + sum_e dr_e Wr_e
  const int nc4 = H / 4;
  for (int i = tid; i < ntok * nc4; i += blockDim.x) {
    const int tl = i / nc4, h = 4 * (i - tl * nc4);
    const int64_t t = t0 + tl;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < k; ++s) {
      const uint2 v = *reinterpret_cast<const uint2*>(rb.dxp + static_cast<int64_t>(rb.pos[t * k + s]) * H + h);
      const float2 a = f16x2_to_f32x2(v.x), b = f16x2_to_f32x2(v.y);
      acc.x += a.x; acc.y += a.y; acc.z += b.x; acc.w += b.y;
    }
    for (int e = 0; e < E; ++e) {
      const float d = s_dr[tl * E + e];
      float w[4];
      load4(Wr + static_cast<int64_t>(e) * H + h, w);
      acc.x = fmaf(d, w[0], acc.x);
      acc.y = fmaf(d, w[1], acc.y);
      acc.z = fmaf(d, w[2], acc.z);
      acc.w = fmaf(d, w[3], acc.w);
    }
    store4(static_cast<Tin*>(rb.dx) + t * H + h, acc);
  }
}

// Per block of 64 tokens, the partials of dWr = dr^T x (element (e, h) =
// sum_t dr[t][e] x[t][h] in token order; a thread holds 4 columns x 8
// experts, so each x element is read once per 8 experts) and of
// d_bias = sum_t dr_t.
template <typename Tin>
__global__ void __launch_bounds__(kBwdThreads)
router_dwr_kernel(const Tin* __restrict__ x, int64_t T, int H, int E, const RouterBwd rb) {
  pdl_enter();
  extern __shared__ float s_dr[];              // [64][E]
  const int tid = threadIdx.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kBwdTok;
  const int ntok = static_cast<int>(T - t0 < kBwdTok ? T - t0 : kBwdTok);
  for (int i = tid; i < ntok * E; i += blockDim.x) s_dr[i] = rb.dr[t0 * E + i];
  __syncthreads();
  const int nc4 = H / 4, nec = (E + 7) / 8;
  for (int item = tid; item < nc4 * nec; item += blockDim.x) {
    const int c4 = item % nc4, e0 = (item / nc4) * 8;
    float acc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[j][q] = 0.f;
#pragma unroll 8
    for (int tl = 0; tl < ntok; ++tl) {
      float xv[4];
      load4(x + (t0 + tl) * H + 4 * c4, xv);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float d = (e0 + j < E) ? s_dr[tl * E + e0 + j] : 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[j][q] = fmaf(d, xv[q], acc[j][q]);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (e0 + j < E)
        *reinterpret_cast<float4*>(rb.dwr_part + (static_cast<int64_t>(blockIdx.x) * E + e0 + j) * H + 4 * c4) =
            make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
  }
  for (int e = tid; e < E; e += blockDim.x) {
    float acc = 0.f;
    for (int tl = 0; tl < ntok; ++tl) acc += s_dr[tl * E + e];
    rb.dbias_part[static_cast<int64_t>(blockIdx.x) * E + e] = acc;
  }
}

// dWr[e][h] = sum_b dwr_part[b][e][h] and d_bias[e] = sum_b dbias_part[b][e].
// A block takes 64 outputs; its 4 thread rows split the blocks b into four
// contiguous quarters, each summed with 4 independent accumulators (loads in
// flight together), then the quarters are added in order: a fixed order
// that depends only on nblk.
constexpr int kRedCols = 64;
__global__ void __launch_bounds__(256)
router_bwd_reduce_kernel(const float* __restrict__ dwr_part, const float* __restrict__ dbias_part,
                         int nblk, int E, int H, float* __restrict__ dWr, float* __restrict__ d_bias) {
  pdl_enter();
  __shared__ float part[4][kRedCols];
  const int64_t n = static_cast<int64_t>(E) * H;
  const int col = threadIdx.x % kRedCols, q = threadIdx.x / kRedCols;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kRedCols + col;
  const bool is_w = i < n;
  const bool is_b = !is_w && i < n + E && d_bias != nullptr;
  const float* src = is_w ? dwr_part + i : dbias_part + (i - n);
  const int64_t stride = is_w ? n : E;
  const int b0 = nblk * q / 4, b1 = nblk * (q + 1) / 4;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  if (is_w || is_b) {
    int b = b0;
    for (; b + 4 <= b1; b += 4) {
      a0 += src[(b + 0) * stride];
      a1 += src[(b + 1) * stride];
      a2 += src[(b + 2) * stride];
      a3 += src[(b + 3) * stride];
    }
    for (; b < b1; ++b) a0 += src[b * stride];
  }
  part[q][col] = (a0 + a1) + (a2 + a3);
  __syncthreads();
  if (q == 0 && (is_w || is_b)) {
    const float v = ((part[0][col] + part[1][col]) + part[2][col]) + part[3][col];
    if (is_w) dWr[i] = v; else d_bias[i - n] = v;
  }
}

// ---------------------------------------------------------------- launchers
static int bwd_blocks(int64_t T) { return static_cast<int>((T + kBwdTok - 1) / kBwdTok); }

cudaError_t launch_bwd_count(const int32_t* topk_idx, int64_t T, int E, int k, int32_t* blk_cnt,
                             cudaStream_t st) {
  return launch_dependent_kernel(bwd_count_kernel, dim3(bwd_blocks(T)), dim3(kBwdThreads), 0, st,
                                 topk_idx, T, E, k, blk_cnt);
}

cudaError_t launch_bwd_dispatch(const void* x, const void* dy, const int32_t* topk_idx, int64_t T,
                                int H, int E, int k, const int32_t* blk_cnt,
                                const BwdDispatchOut& o, cudaStream_t st) {
  if (H % 8 != 0) return cudaErrorInvalidValue;
  // the block's x and dy rows staged in shared memory when they fit (bulk
  // copies in and out), else 16-byte loads and stores
  const size_t rows = 2 * static_cast<size_t>(kBwdTok) * H * sizeof(__nv_bfloat16);
  const int stage = rows <= 200 * 1024 && o.hdr != nullptr ? 1 : 0;
  const size_t smem = stage ? rows : 0;
  auto fn = bwd_dispatch_kernel<__nv_bfloat16>;
  if (stage) {
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), smem);
    if (e != cudaSuccess) return e;
  }
  return launch_dependent_kernel(fn, dim3(bwd_blocks(T)), dim3(kBwdThreads), smem, st,
                                 static_cast<const __nv_bfloat16*>(x),
                                 static_cast<const __nv_bfloat16*>(dy), topk_idx, T, H, E, k,
                                 blk_cnt, o, stage);
}

cudaError_t launch_router_bwd(const void* x, const void* Wr, int64_t T, int H, int E, int k,
                              const RouterBwd& rb, cudaStream_t st) {
  if (H % 4 != 0) return cudaErrorInvalidValue;
  const int grid = static_cast<int>((T + kRbTok - 1) / kRbTok);
  cudaError_t e = launch_dependent_kernel(router_bwd_kernel<__nv_bfloat16>, dim3(grid),
                                          dim3(kBwdThreads), 0, st,
                                          static_cast<const __nv_bfloat16*>(Wr), T, H, E, k, rb);
  if (e != cudaSuccess) return e;
  const size_t smem = static_cast<size_t>(kBwdTok) * E * sizeof(float);
  return launch_dependent_kernel(router_dwr_kernel<__nv_bfloat16>, dim3(bwd_blocks(T)),
                                 dim3(kBwdThreads), smem, st,
                                 static_cast<const __nv_bfloat16*>(x), T, H, E, rb);
}

cudaError_t launch_router_bwd_reduce(const float* dwr_part, const float* dbias_part, int nblk,
                                     int E, int H, float* dWr, float* d_bias, cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(E) * H + E;
  const int grid = static_cast<int>((n + kRedCols - 1) / kRedCols);
  return launch_dependent_kernel(router_bwd_reduce_kernel, dim3(grid), dim3(256), 0, st, dwr_part,
                                 dbias_part, nblk, E, H, dWr, d_bias);
}

}  // namespace mm
