// Decode-sized forward (T <= kDecodeMaxT tokens, bf16): one cooperative
// weight-streaming kernel on the CUDA cores.  Every weight row is read from
// HBM once, by the bulk-copy engine into shared memory; for the MoE only the
// experts some token selected are read.
//
//   route (MoE)  logits, softmax, top-k, alpha (lesson 13 §1.5, chapter 4
//                §4.3): cheap at this size, so every CTA computes it for all
//                T tokens with the same code and order, and all CTAs agree;
//                block 0 writes topk_idx, topk_w and the aux loss (lesson 13 §1.6)
//   gate/up      h[a, i] = SiLU(Wg_e[i] . x_t) * (Wu_e[i] . x_t) for every
//                assignment a = (t, s) of expert e, fp16   (lesson 13 §0/§1.2)
//   grid barrier (h complete)
//   down         y[t, j] = sum_s alpha_{t,s} (Wd_{e_s}[j] . h[t, s]) in slot
//                order, fp32, rounded once       (lesson 13 §0 MoE equation)
//
// Each CTA issues the bulk copies of its first gate/up slice and of its first
// Wd rows as soon as it knows the touched experts, so the down weights are
// already in shared memory when the barrier opens.
#include "mm_kernels.cuh"

namespace mm {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kUpRows = kDecWarps;          // Wg / Wu rows per gate/up slice (1 per warp)
constexpr int kDnRows = 4;                  // output rows per down unit
constexpr int kTokGroup = 8;                // tokens whose sums a lane keeps at once
constexpr int kHStage = 16;                 // h rows (assignments) staged at once
constexpr size_t kWrSmemMax = 32 * 1024;    // Wr staged in shared memory up to this size

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
  __half* h;                // [T*k, I] fp16 scratch (dense: [T, I])
  void* y;                  // [T, H] bf16
  WsHeader* hdr;
};

// Routing tables shared by the CTA.
struct DecRoute {
  int nA;                                   // assignments (MoE: T*k, dense: T)
  int n_touched;
  int touched[MM_MAX_EXPERTS];              // ascending expert ids
  int sel_e[kDecodeMaxT * MM_MAX_TOPK];     // expert of assignment a = t*k + s
  float sel_a[kDecodeMaxT * MM_MAX_TOPK];   // its alpha
  float prob[kDecodeMaxT][MM_MAX_EXPERTS];  // logits, then probabilities
  int by_e[kDecodeMaxT * MM_MAX_TOPK];      // assignments grouped by expert, in order
  int e_start[MM_MAX_EXPERTS + 1];          // expert e's assignments: by_e[e_start[e] ..]
};

__device__ __forceinline__ void cvt8(const uint4& raw, float (&f)[8]) {
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 q = __bfloat1622float2(b[i]);
    f[2 * i] = q.x;
    f[2 * i + 1] = q.y;
  }
}
__device__ __forceinline__ void cvt8h(const uint4& raw, float (&f)[8]) {
  const __half2* b = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 q = __half22float2(b[i]);
    f[2 * i] = q.x;
    f[2 * i + 1] = q.y;
  }
}

__device__ __forceinline__ float warp_allsum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 1-D bulk copy global -> this CTA's shared memory, completion on `bar`.
__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__host__ __device__ inline size_t round128(size_t v) { return (v + 127) & ~size_t(127); }
__host__ __device__ inline size_t wr_bytes(int E, int H) { return static_cast<size_t>(E) * H * 2; }

// Shared-memory layout: x | gate/up ring (2 x (Wg, Wu) slices) | Wd slots (2) |
// h stage (also holds Wr during the routing).
struct DecLayout {
  size_t ring, wd, hst, total;
};
__host__ __device__ inline DecLayout dec_layout(int T, int H, int I, int E, int nA) {
  DecLayout L;
  L.ring = round128(static_cast<size_t>(T) * H * 2);
  L.wd = L.ring + round128(2 * 2 * static_cast<size_t>(kUpRows) * H * 2);
  L.hst = L.wd + round128(2 * static_cast<size_t>(kDnRows) * I * 2);
  const size_t hs = static_cast<size_t>(nA < kHStage ? nA : kHStage) * I * 2;
  const size_t wr = wr_bytes(E, H) <= kWrSmemMax ? wr_bytes(E, H) : 0;
  L.total = L.hst + round128(hs > wr ? hs : wr);
  return L;
}

// Routing of all T tokens.  Logits: (token, expert) pairs spread over the
// warps, four at a time with independent sums (lanes split H, xor-tree sum),
// fp32.  Then warp t, lane e: softmax over the experts with the maximum
// subtracted, and k arg-max rounds over (p desc, index asc) — equal
// probabilities go to the lower index; alpha = p / (sum_S p + 1e-20).
__device__ void decode_route(const DecodeArgs& A, const __nv_bfloat16* xs,
                             const __nv_bfloat16* wrs, DecRoute& R) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nch = A.H / 8;
  if (A.Wr == nullptr) {                      // dense: one weight set, every token
    if (threadIdx.x < A.T) {
      R.sel_e[threadIdx.x] = 0;
      R.sel_a[threadIdx.x] = 1.0f;
      R.by_e[threadIdx.x] = threadIdx.x;
    }
    if (threadIdx.x == 0) {
      R.nA = A.T;
      R.n_touched = 1;
      R.touched[0] = 0;
      R.e_start[0] = 0;
      R.e_start[1] = A.T;
    }
    __syncthreads();
    return;
  }
  const __nv_bfloat16* Wr = wrs != nullptr ? wrs : static_cast<const __nv_bfloat16*>(A.Wr);
  const int E = A.E, k = A.k;
  const int pairs = A.T * E;
  for (int p0 = warp * 4; p0 < pairs; p0 += kDecWarps * 4) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c = lane; c < nch; c += 32) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int p = p0 + q;
        if (p < pairs) {
          const int t = p / E, e = p - t * E;
          float xv[8], wv[8];
          cvt8(*reinterpret_cast<const uint4*>(xs + t * A.H + c * 8), xv);
          cvt8(*reinterpret_cast<const uint4*>(Wr + static_cast<int64_t>(e) * A.H + c * 8), wv);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[q] = fmaf(xv[j], wv[j], acc[q]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = warp_allsum(acc[q]);
    if (lane < 4 && p0 + lane < pairs) {
      float v = acc[0];
#pragma unroll
      for (int q = 1; q < 4; ++q)
        if (lane == q) v = acc[q];
      const int p = p0 + lane;
      R.prob[p / E][p % E] = v;
    }
  }
  __syncthreads();
  for (int t = warp; t < A.T; t += kDecWarps) {
    // lane holds experts lane and lane + 32
    float r0 = -INFINITY, r1 = -INFINITY;
    if (lane < E) r0 = R.prob[t][lane] + (A.bias != nullptr ? A.bias[lane] : 0.f);
    if (lane + 32 < E) r1 = R.prob[t][lane + 32] + (A.bias != nullptr ? A.bias[lane + 32] : 0.f);
    float m = fmaxf(r0, r1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float x0 = (lane < E) ? expf(r0 - m) : 0.f;
    const float x1 = (lane + 32 < E) ? expf(r1 - m) : 0.f;
    const float z = warp_allsum(x0 + x1);
    const float p0 = x0 / z, p1 = x1 / z;
    if (lane < E) R.prob[t][lane] = p0;
    if (lane + 32 < E) R.prob[t][lane + 32] = p1;
    bool taken0 = lane >= E, taken1 = lane + 32 >= E;
    float sel_sum = 0.f;
    for (int s = 0; s < k; ++s) {
      float bp = -1.f;
      int be = 0x7fffffff;
      if (!taken0) { bp = p0; be = lane; }
      if (!taken1 && (p1 > bp)) { bp = p1; be = lane + 32; }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float op = __shfl_xor_sync(0xffffffffu, bp, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (op > bp || (op == bp && oe < be)) { bp = op; be = oe; }
      }
      if (be == lane) taken0 = true;
      if (be == lane + 32) taken1 = true;
      sel_sum += bp;
      if (lane == 0) {
        R.sel_e[t * k + s] = be;
        R.sel_a[t * k + s] = bp;
      }
    }
    __syncwarp();
    if (lane < k) R.sel_a[t * k + lane] = R.sel_a[t * k + lane] / (sel_sum + 1e-20f);
  }
  __syncthreads();
  // per-expert counts, their prefix, and each assignment's place (order kept)
  const int nA = A.T * k;
  if (threadIdx.x < E) {
    int c = 0;
    for (int a = 0; a < nA; ++a) c += (R.sel_e[a] == static_cast<int>(threadIdx.x));
    R.e_start[threadIdx.x + 1] = c;                 // count for now
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    R.nA = nA;
    R.e_start[0] = 0;
    int n = 0;
    for (int e = 0; e < E; ++e) {
      if (R.e_start[e + 1] > 0) R.touched[n++] = e;
      R.e_start[e + 1] += R.e_start[e];
    }
    R.n_touched = n;
  }
  __syncthreads();
  if (threadIdx.x < nA) {
    const int a = threadIdx.x, e = R.sel_e[a];
    int rank = 0;
    for (int b = 0; b < a; ++b) rank += (R.sel_e[b] == e);
    R.by_e[R.e_start[e] + rank] = a;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kDecThreads)
decode_ffn_kernel(const DecodeArgs A) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ DecRoute R;
  __shared__ __align__(8) uint64_t bar[5];     // ring 0, ring 1, Wd slot 0, Wd slot 1, h stage
  __shared__ float part[kDecodeMaxT * MM_MAX_TOPK][kDnRows];
  const int H = A.H, I = A.I;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nA_max = (A.Wr != nullptr) ? A.T * A.k : A.T;
  const DecLayout Ly = dec_layout(A.T, H, I, A.E, nA_max);
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(dsm);
  unsigned char* ring = dsm + Ly.ring;
  unsigned char* wdbuf = dsm + Ly.wd;
  __half* hst = reinterpret_cast<__half*>(dsm + Ly.hst);
  __nv_bfloat16* wrs = (A.Wr != nullptr && wr_bytes(A.E, H) <= kWrSmemMax)
                           ? reinterpret_cast<__nv_bfloat16*>(hst) : nullptr;
  const size_t slice_bytes = static_cast<size_t>(kUpRows) * H * 2;   // one of Wg / Wu
  const size_t slot_bytes = static_cast<size_t>(kDnRows) * I * 2;
  uint32_t phase[5] = {0, 0, 0, 0, 0};
  bool inflight[5] = {false, false, false, false, false};           // thread 0 issues

  if (threadIdx.x == 0) {
    for (int q = 0; q < 5; ++q) mbar_init(&bar[q], 1);
    fence_mbar_init();
  }
  {
    const int nx = A.T * H / 8;
    const int nw = (wrs != nullptr) ? A.E * H / 8 : 0;
    for (int i = threadIdx.x; i < nx + nw; i += blockDim.x) {
      if (i < nx)
        reinterpret_cast<uint4*>(xs)[i] = __ldg(reinterpret_cast<const uint4*>(A.x) + i);
      else
        reinterpret_cast<uint4*>(wrs)[i - nx] = __ldg(reinterpret_cast<const uint4*>(A.Wr) + (i - nx));
    }
  }
  __syncthreads();
  decode_route(A, xs, wrs, R);

  if (blockIdx.x == 0 && A.Wr != nullptr) {
    for (int a = threadIdx.x; a < R.nA; a += blockDim.x) {
      A.topk_idx[a] = R.sel_e[a];
      A.topk_w[a] = R.sel_a[a];
    }
    if (warp == 0) {
      // aux = E*coef*sum_e (count_e/T)(P_e/T): lane e sums its expert
      float acc = 0.f;
      for (int e = lane; e < A.E; e += 32) {
        float P = 0.f;
        for (int t = 0; t < A.T; ++t) P += R.prob[t][e];
        acc = fmaf(static_cast<float>(R.e_start[e + 1] - R.e_start[e]), P, acc);
      }
      acc = warp_allsum(acc);
      const float invT = 1.0f / static_cast<float>(A.T);
      if (lane == 0) *A.aux_loss = static_cast<float>(A.E) * A.coef * acc * invT * invT;
    }
  }

  // ---- work lists
  const int slices = (I + kUpRows - 1) / kUpRows;
  const int up_units = R.n_touched * slices;
  const int dn_units = (H + kDnRows - 1) / kDnRows;
  auto issue_up = [&](int unit, int b) {
    fence_proxy_async_smem();
    const int e = R.touched[unit / slices];
    const int r0 = (unit % slices) * kUpRows;
    const int rows = min(kUpRows, I - r0);
    const uint32_t bytes = static_cast<uint32_t>(rows) * H * 2;
    unsigned char* dst = ring + b * 2 * slice_bytes;
    mbar_arrive_expect_tx(&bar[b], 2 * bytes);
    bulk_load(dst, static_cast<const __nv_bfloat16*>(A.wg.p[e]) + static_cast<int64_t>(r0) * H,
              bytes, &bar[b]);
    bulk_load(dst + slice_bytes,
              static_cast<const __nv_bfloat16*>(A.wu.p[e]) + static_cast<int64_t>(r0) * H, bytes,
              &bar[b]);
  };
  auto issue_wd = [&](int unit, int ti, int b) {
    fence_proxy_async_smem();
    const int j0 = unit * kDnRows;
    const int rows = min(kDnRows, H - j0);
    const int e = R.touched[ti];
    const uint32_t bytes = static_cast<uint32_t>(rows) * I * 2;
    mbar_arrive_expect_tx(&bar[2 + b], bytes);
    bulk_load(wdbuf + b * slot_bytes,
              static_cast<const __nv_bfloat16*>(A.wd.p[e]) + static_cast<int64_t>(j0) * I, bytes,
              &bar[2 + b]);
  };
  __syncthreads();                             // Wr in the h stage is no longer read
  if (threadIdx.x == 0) {
    if (blockIdx.x < up_units) {
      issue_up(blockIdx.x, 0);
      inflight[0] = true;
    }
    if (blockIdx.x < dn_units) {               // the first down unit's first two experts
      for (int q = 0; q < 2 && q < R.n_touched; ++q) {
        issue_wd(blockIdx.x, q, q);
        inflight[2 + q] = true;
      }
    }
  }

  // ---- gate/up: units blockIdx.x, + gridDim.x, ...; warp w owns row w
  bool ok = true;
  for (int it = 0, u = blockIdx.x; ok && u < up_units; u += gridDim.x, ++it) {
    const int b = it & 1;
    const int nxt = u + static_cast<int>(gridDim.x);
    __syncthreads();                           // buffer b^1 is no longer being read
    if (threadIdx.x == 0 && nxt < up_units) {
      issue_up(nxt, b ^ 1);
      inflight[b ^ 1] = true;
    }
    ok = __syncthreads_and(mbar_wait(&bar[b], phase[b], nullptr, A.hdr, 20));
    if (!ok) break;
    phase[b] ^= 1;
    inflight[b] = false;
    const int e = R.touched[u / slices];
    const int i = (u % slices) * kUpRows + warp;
    if (i >= I) continue;
    const __nv_bfloat16* grow = reinterpret_cast<const __nv_bfloat16*>(ring + b * 2 * slice_bytes) + warp * H;
    const __nv_bfloat16* urow = grow + kUpRows * H;
    const int* list = R.by_e + R.e_start[e];   // the assignments of expert e, in order
    const int n = R.e_start[e + 1] - R.e_start[e];
    for (int g0 = 0; g0 < n; g0 += kTokGroup) {
      // 2*kTokGroup independent partial sums: g_t and u_t of up to 8 tokens
      float v[2 * kTokGroup];
#pragma unroll
      for (int q = 0; q < 2 * kTokGroup; ++q) v[q] = 0.f;
      for (int c = lane; c < H / 8; c += 32) {
        float gv[8], uv[8];
        cvt8(*reinterpret_cast<const uint4*>(grow + c * 8), gv);
        cvt8(*reinterpret_cast<const uint4*>(urow + c * 8), uv);
#pragma unroll
        for (int tt = 0; tt < kTokGroup; ++tt) {
          if (g0 + tt < n) {
            const int a = list[g0 + tt];
            const int t = (A.Wr != nullptr) ? a / A.k : a;
            float xv[8];
            cvt8(*reinterpret_cast<const uint4*>(xs + t * H + c * 8), xv);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              v[2 * tt] = fmaf(gv[q], xv[q], v[2 * tt]);
              v[2 * tt + 1] = fmaf(uv[q], xv[q], v[2 * tt + 1]);
            }
          }
        }
      }
      // butterfly reduce-scatter of the 16 sums: lane L ends with the full
      // sum of value L >> 1 (value 2t = g_t, 2t + 1 = u_t)
#pragma unroll
      for (int o = 16; o >= 2; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int q = 0; q < o / 2; ++q) {
          const float lo = v[q], hi = v[q + o / 2];
          v[q] = (up ? hi : lo) + __shfl_xor_sync(0xffffffffu, up ? lo : hi, o);
        }
      }
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
      const float u_val = __shfl_down_sync(0xffffffffu, v[0], 2);   // lane L+2 holds u_t
      const int tt = lane >> 2;
      if ((lane & 3) == 0 && g0 + tt < n)
        A.h[static_cast<int64_t>(list[g0 + tt]) * I + i] = __float2half_rn(silu_f32(v[0]) * u_val);
    }
  }

  // ---- every h row written before any CTA reads it
  if (ok) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    ok = grid_barrier(A.hdr, 24);
  }

  // ---- down: unit = kDnRows output rows, every touched expert
  const int kk = (A.Wr != nullptr) ? A.k : 1;
  for (int du = blockIdx.x, round = 0; ok && du < dn_units; du += gridDim.x, ++round) {
    const int j0 = du * kDnRows;
    const int rows = min(kDnRows, H - j0);
    if (round > 0 && threadIdx.x == 0) {       // later units: fetch their first two experts now
      for (int q = 0; q < 2 && q < R.n_touched; ++q) {
        issue_wd(du, q, q);
        inflight[2 + q] = true;
      }
    }
    bool waited[2] = {false, false};
    int ti = 0;
    for (int q0 = 0; ok && q0 < R.nA;) {
      const int q1 = min(R.nA, q0 + kHStage);
      __syncthreads();                         // the previous stage is no longer read
      if (threadIdx.x == 0) {
        fence_proxy_async_smem();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        mbar_arrive_expect_tx(&bar[4], static_cast<uint32_t>(q1 - q0) * I * 2);
        for (int q = q0; q < q1; ++q)
          bulk_load(hst + static_cast<size_t>(q - q0) * I, A.h + static_cast<int64_t>(R.by_e[q]) * I,
                    static_cast<uint32_t>(I) * 2, &bar[4]);
        inflight[4] = true;
      }
      ok = __syncthreads_and(mbar_wait(&bar[4], phase[4], nullptr, A.hdr, 21));
      if (!ok) break;
      phase[4] ^= 1;
      inflight[4] = false;
      while (ti < R.n_touched) {
        const int e = R.touched[ti];
        if (R.e_start[e] >= q1) break;         // its rows come with a later stage
        const int ea = max(R.e_start[e], q0), eb = min(R.e_start[e + 1], q1);
        const int b = ti & 1;
        if (!waited[b]) {
          ok = __syncthreads_and(mbar_wait(&bar[2 + b], phase[2 + b], nullptr, A.hdr, 22));
          if (!ok) break;
          waited[b] = true;
        }
        const __nv_bfloat16* ws = reinterpret_cast<const __nv_bfloat16*>(wdbuf + b * slot_bytes);
        // warp w: row w % kDnRows; the expert's assignments in this stage four
        // at a time, round-robin over the warps of that row
        constexpr int kWarpsPerRow = kDecWarps / kDnRows;
        const int jl = warp % kDnRows;
        if (jl < rows) {
          for (int g0 = ea + (warp / kDnRows) * 4; g0 < eb; g0 += 4 * kWarpsPerRow) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int c = lane; c < I / 8; c += 32) {
              float wv[8];
              cvt8(*reinterpret_cast<const uint4*>(ws + jl * I + c * 8), wv);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                if (g0 + q < eb) {
                  float hv[8];
                  cvt8h(*reinterpret_cast<const uint4*>(hst + static_cast<size_t>(g0 + q - q0) * I + c * 8), hv);
#pragma unroll
                  for (int j = 0; j < 8; ++j) acc[q] = fmaf(wv[j], hv[j], acc[q]);
                }
              }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] = warp_allsum(acc[q]);
            if (lane < 4 && g0 + lane < eb) {
              float val = acc[0];
#pragma unroll
              for (int q = 1; q < 4; ++q)
                if (lane == q) val = acc[q];
              part[R.by_e[g0 + lane]][jl] = val;
            }
          }
        }
        if (R.e_start[e + 1] > q1) break;      // e continues in the next stage
        __syncthreads();                       // e is done: its slot takes the expert after next
        phase[2 + b] ^= 1;
        waited[b] = false;
        if (threadIdx.x == 0) {
          inflight[2 + b] = false;
          if (ti + 2 < R.n_touched) {
            issue_wd(du, ti + 2, b);
            inflight[2 + b] = true;
          }
        }
        ++ti;
      }
      q0 = q1;
    }
    __syncthreads();
    if (!ok) break;
    for (int q = threadIdx.x; q < A.T * rows; q += blockDim.x) {
      const int t = q / rows, jl = q % rows;
      float v = 0.f;
      for (int s = 0; s < kk; ++s) v += R.sel_a[t * kk + s] * part[t * kk + s][jl];
      static_cast<__nv_bfloat16*>(A.y)[static_cast<int64_t>(t) * H + j0 + jl] = __float2bfloat16_rn(v);
    }
  }
  // let copies still in flight (a unit this CTA did not reach, or a failed
  // wait) land before the CTA exits
  if (threadIdx.x == 0)
    for (int q = 0; q < 5; ++q)
      if (inflight[q]) mbar_wait(&bar[q], phase[q], nullptr, nullptr, 25);
}

size_t decode_smem_bytes(int T, int H, int I, int E, int k) {
  return dec_layout(T, H, I, E, T * k).total;
}

cudaError_t launch_decode_ffn(const void* x, const void* Wr, const float* bias,
                              const void* const* Wg, const void* const* Wu, const void* const* Wd,
                              int T, int H, int I, int E, int k, float coef, int32_t* topk_idx,
                              float* topk_w, float* aux_loss, void* hbuf, void* y, WsHeader* hdr,
                              cudaStream_t st) {
  DecodeArgs A;
  memset(&A, 0, sizeof(A));
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
  A.h = static_cast<__half*>(hbuf); A.y = y; A.hdr = hdr;
  const size_t smem = dec_layout(T, H, I, nw, T * A.k).total;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(decode_ffn_kernel), smem);
  if (e != cudaSuccess) return e;
  // every CTA must be resident (grid barrier): as many as fit, at most two per SM
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_ffn_kernel, kDecThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int grid = num_sms() * (per_sm < 2 ? per_sm : 2);
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
