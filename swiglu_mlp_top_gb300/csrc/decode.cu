// Decode-sized forward (T <= kDecodeMaxT tokens): weight streaming on the
// CUDA cores in two kernels.  Every weight row is read from HBM once, by the
// bulk-copy engine into shared memory, while the previous slice is in use;
// for the MoE only the experts some token selected are read.
//
//   A  route (MoE) + gate/up:  h[a, i] = SiLU(Wg_e[i] . x_t) * (Wu_e[i] . x_t)
//      for every assignment a = (t, s) of expert e, stored in fp16
//                                                          (lesson 13 §0/§1.2)
//   B  route (MoE) + down + combine:
//      y[t, j] = sum_s alpha_{t,s} (Wd_{e_s}[j] . h[t, s])  in slot order, fp32,
//      rounded once                             (lesson 13 §0 MoE equation, step 5)
//
// The routing (logits, softmax, top-k, alpha; lesson 13 §1.5, chapter 4 §4.3)
// is cheap at this size, so every CTA computes it for all T tokens with the
// same code and order, and all CTAs agree on it; block 0 of kernel A writes
// topk_idx, topk_w and the aux loss (lesson 13 §1.6).  Kernel B is launched as
// a programmatic dependent of A: it routes and starts streaming its Wd rows
// while A runs, and waits for A's h only before staging it.
#include "mm_kernels.cuh"

namespace mm {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kUpRows = kDecWarps;          // Wg / Wu rows per gate/up slice (1 per warp)
constexpr int kDnRows = 4;                  // output rows per down unit
constexpr int kTokGroup = 8;                // tokens whose sums a lane keeps at once
constexpr int kHStage = 16;                 // h rows (assignments) staged at once in kernel B

struct DecodeArgs {
  const void* x;            // [T, H] bf16
  const void* Wr;           // [E, H] bf16, or nullptr (dense)
  const float* bias;        // [E] or nullptr
  PtrArray wg, wu, wd;      // per expert
  int T, H, I, E, k;
  float coef;
  int32_t* topk_idx;        // written by block 0 of kernel A (MoE)
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

// x [T, H] and (MoE, when it fits) Wr [E, H] into shared memory.
__device__ __forceinline__ void load_inputs(const DecodeArgs& A, __nv_bfloat16* xs,
                                            __nv_bfloat16* wrs) {
  const int nx = A.T * A.H / 8;
  const int nw = (A.Wr != nullptr && wrs != nullptr) ? A.E * A.H / 8 : 0;
  for (int i = threadIdx.x; i < nx + nw; i += blockDim.x) {
    if (i < nx)
      reinterpret_cast<uint4*>(xs)[i] = __ldg(reinterpret_cast<const uint4*>(A.x) + i);
    else
      reinterpret_cast<uint4*>(wrs)[i - nx] = __ldg(reinterpret_cast<const uint4*>(A.Wr) + (i - nx));
  }
}

// Routing of all T tokens.  Logits: (token, expert) pairs are spread over
// the warps, four at a time with independent sums (lanes split H, xor-tree
// sum), fp32.  Then per token (one thread each): softmax with the maximum
// subtracted, k sequential selections with strict '>' (equal probabilities ->
// lower index), alpha = p / (sum_S p + 1e-20).  Dense: one weight set, every
// token with alpha 1.  Wr is read from `wrs` (shared) or global when null.
__device__ void decode_route(const DecodeArgs& A, const __nv_bfloat16* xs,
                             const __nv_bfloat16* wrs, DecRoute& R) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nch = A.H / 8;
  if (A.Wr == nullptr) {
    if (threadIdx.x == 0) {
      R.nA = A.T;
      R.n_touched = 1;
      R.touched[0] = 0;
      for (int t = 0; t < A.T; ++t) {
        R.sel_e[t] = 0;
        R.sel_a[t] = 1.0f;
        R.by_e[t] = t;
      }
      R.e_start[0] = 0;
      R.e_start[1] = A.T;
    }
    __syncthreads();
    return;
  }
  const __nv_bfloat16* Wr = wrs != nullptr ? wrs : static_cast<const __nv_bfloat16*>(A.Wr);
  const int pairs = A.T * A.E;
  for (int p0 = warp * 4; p0 < pairs; p0 += kDecWarps * 4) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c = lane; c < nch; c += 32) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int p = p0 + q;
        if (p < pairs) {
          const int t = p / A.E, e = p - t * A.E;
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
      const int t = p / A.E, e = p - t * A.E;
      R.prob[t][e] = v + (A.bias != nullptr ? A.bias[e] : 0.f);
    }
  }
  __syncthreads();
  if (threadIdx.x < A.T) {
    const int t = threadIdx.x;
    float m = -INFINITY;
    for (int e = 0; e < A.E; ++e) m = fmaxf(m, R.prob[t][e]);
    float z = 0.f;
    for (int e = 0; e < A.E; ++e) {
      const float v = expf(R.prob[t][e] - m);
      R.prob[t][e] = v;
      z += v;
    }
    for (int e = 0; e < A.E; ++e) R.prob[t][e] = R.prob[t][e] / z;
    uint64_t taken = 0;
    float sum = 0.f;
    for (int s = 0; s < A.k; ++s) {
      int best = -1;
      float bp = 0.f;
      for (int e = 0; e < A.E; ++e) {
        const float p = R.prob[t][e];
        if (!((taken >> e) & 1ull) && (best < 0 || p > bp)) {
          best = e;
          bp = p;
        }
      }
      taken |= 1ull << best;
      R.sel_e[t * A.k + s] = best;
      R.sel_a[t * A.k + s] = bp;
      sum += bp;
    }
    for (int s = 0; s < A.k; ++s) R.sel_a[t * A.k + s] = R.sel_a[t * A.k + s] / (sum + 1e-20f);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    R.nA = A.T * A.k;
    uint64_t m = 0;
    for (int a = 0; a < R.nA; ++a) m |= 1ull << R.sel_e[a];
    int n = 0;
    for (int e = 0; e < A.E; ++e)
      if ((m >> e) & 1ull) R.touched[n++] = e;
    R.n_touched = n;
    int q = 0;
    for (int e = 0; e < A.E; ++e) {
      R.e_start[e] = q;
      for (int a = 0; a < R.nA; ++a)
        if (R.sel_e[a] == e) R.by_e[q++] = a;
    }
    R.e_start[A.E] = q;
  }
  __syncthreads();
}

__host__ __device__ inline size_t round128(size_t v) { return (v + 127) & ~size_t(127); }
__host__ __device__ inline size_t wr_bytes(int E, int H) { return static_cast<size_t>(E) * H * 2; }
constexpr size_t kWrSmemMax = 32 * 1024;    // Wr staged in shared memory up to this size

// ---------------------------------------------------------------- kernel A
// Work unit = (touched expert, slice of kUpRows rows of Wg / Wu).  The CTA
// walks its units with two shared-memory buffers: the bulk copy of its next
// unit is in flight while the current one is computed.  Warp w owns row w of
// the slice; lanes split H into 8-element chunks and keep the partial sums of
// up to kTokGroup tokens apart.
__host__ __device__ inline size_t smem_a_bytes(int T, int H, int E) {
  const size_t bufs = 2 * 2 * static_cast<size_t>(kUpRows) * H * 2;
  const size_t wr = wr_bytes(E, H) <= kWrSmemMax ? wr_bytes(E, H) : 0;
  return round128(static_cast<size_t>(T) * H * 2) + (bufs > wr ? bufs : wr);
}

__global__ void __launch_bounds__(kDecThreads)
decode_gateup_kernel(const DecodeArgs A) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ DecRoute R;
  __shared__ __align__(8) uint64_t bar[2];
  const int H = A.H, I = A.I;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t slice_bytes = static_cast<size_t>(kUpRows) * H * 2;   // one of Wg / Wu
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(dsm);
  unsigned char* buf = dsm + round128(static_cast<size_t>(A.T) * H * 2);
  __nv_bfloat16* wrs = (A.Wr != nullptr && wr_bytes(A.E, H) <= kWrSmemMax)
                           ? reinterpret_cast<__nv_bfloat16*>(buf) : nullptr;   // before the ring

  // the dependent grid (kernel B) may start its own prologue now
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  load_inputs(A, xs, wrs);
  __syncthreads();
  decode_route(A, xs, wrs, R);

  if (blockIdx.x == 0 && A.Wr != nullptr) {
    // routing outputs and aux = E*coef*sum_e (count_e/T)(P_e/T)
    for (int a = threadIdx.x; a < R.nA; a += blockDim.x) {
      A.topk_idx[a] = R.sel_e[a];
      A.topk_w[a] = R.sel_a[a];
    }
    if (threadIdx.x == 0) {
      float acc = 0.f;
      for (int e = 0; e < A.E; ++e) {
        float P = 0.f;
        for (int t = 0; t < A.T; ++t) P += R.prob[t][e];
        acc = fmaf(static_cast<float>(R.e_start[e + 1] - R.e_start[e]), P, acc);
      }
      const float invT = 1.0f / static_cast<float>(A.T);
      *A.aux_loss = static_cast<float>(A.E) * A.coef * acc * invT * invT;
    }
  }

  const int slices = (I + kUpRows - 1) / kUpRows;
  const int units = R.n_touched * slices;
  auto issue = [&](int unit, int b) {
    fence_proxy_async_smem();                  // earlier generic reads of this buffer come first
    const int e = R.touched[unit / slices];
    const int r0 = (unit % slices) * kUpRows;
    const int rows = min(kUpRows, I - r0);
    const uint32_t bytes = static_cast<uint32_t>(rows) * H * 2;
    unsigned char* dst = buf + b * 2 * slice_bytes;
    mbar_arrive_expect_tx(&bar[b], 2 * bytes);
    bulk_load(dst, static_cast<const __nv_bfloat16*>(A.wg.p[e]) + static_cast<int64_t>(r0) * H,
              bytes, &bar[b]);
    bulk_load(dst + slice_bytes,
              static_cast<const __nv_bfloat16*>(A.wu.p[e]) + static_cast<int64_t>(r0) * H, bytes,
              &bar[b]);
  };
  int u = blockIdx.x;
  bool inflight[2] = {false, false};           // tracked by thread 0, which issues
  __syncthreads();                             // Wr in `buf` is no longer read
  if (threadIdx.x == 0 && u < units) {
    issue(u, 0);
    inflight[0] = true;
  }
  uint32_t phase[2] = {0, 0};
  for (int it = 0; u < units; u += gridDim.x, ++it) {
    const int b = it & 1;
    const int nxt = u + static_cast<int>(gridDim.x);
    __syncthreads();                           // buffer b^1 is no longer being read
    if (threadIdx.x == 0 && nxt < units) {
      issue(nxt, b ^ 1);
      inflight[b ^ 1] = true;
    }
    const bool ok = mbar_wait(&bar[b], phase[b], nullptr, A.hdr, 20);
    if (!__syncthreads_and(ok)) break;
    phase[b] ^= 1;
    inflight[b] = false;
    const int e = R.touched[u / slices];
    const int r0 = (u % slices) * kUpRows;
    const __nv_bfloat16* gsl = reinterpret_cast<const __nv_bfloat16*>(buf + b * 2 * slice_bytes);
    const __nv_bfloat16* usl = gsl + kUpRows * H;
    const int row = warp;                      // one row of Wg and Wu per warp
    const int i = r0 + row;
    if (i >= I) continue;
    const int* list = R.by_e + R.e_start[e];   // the assignments of expert e, in order
    const int n = R.e_start[e + 1] - R.e_start[e];
    for (int g0 = 0; g0 < n; g0 += kTokGroup) {
      // 2*kTokGroup independent partial sums: g_t and u_t of up to 8 tokens
      float v[2 * kTokGroup];
#pragma unroll
      for (int q = 0; q < 2 * kTokGroup; ++q) v[q] = 0.f;
      for (int c = lane; c < H / 8; c += 32) {
        float gv[8], uv[8];
        cvt8(*reinterpret_cast<const uint4*>(gsl + row * H + c * 8), gv);
        cvt8(*reinterpret_cast<const uint4*>(usl + row * H + c * 8), uv);
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
  // after a wait gave up, let copies still in flight land before exiting
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b)
      if (inflight[b]) mbar_wait(&bar[b], phase[b], nullptr, nullptr, 22);
  }
}

// ---------------------------------------------------------------- kernel B
// Unit = kDnRows output rows j.  For each touched expert the CTA bulk-copies
// Wd_e[j0 : j0 + kDnRows, :] into a double-buffered slot (the first copy is
// issued before waiting for kernel A).  After the wait it bulk-copies the h
// rows of up to kHStage assignments (grouped by expert) into shared memory
// and forms each (row, assignment) dot product from shared memory; the block
// then sums each token's slots in order and rounds once.
__host__ __device__ inline size_t smem_b_bytes(int T, int H, int I, int E) {
  const size_t wd = 2 * static_cast<size_t>(kDnRows) * I * 2;
  const size_t hs = static_cast<size_t>(kHStage) * I * 2;
  const size_t wr = wr_bytes(E, H) <= kWrSmemMax ? wr_bytes(E, H) : 0;
  return round128(static_cast<size_t>(T) * H * 2) + round128(wd) + (hs > wr ? hs : wr);
}

__global__ void __launch_bounds__(kDecThreads)
decode_down_kernel(const DecodeArgs A) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ DecRoute R;
  __shared__ __align__(8) uint64_t bar[3];     // Wd slot 0, Wd slot 1, h stage
  __shared__ float part[kDecodeMaxT * MM_MAX_TOPK][kDnRows];
  const int H = A.H, I = A.I;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(dsm);
  unsigned char* wdbuf = dsm + round128(static_cast<size_t>(A.T) * H * 2);
  const size_t slot_bytes = static_cast<size_t>(kDnRows) * I * 2;
  __half* hst = reinterpret_cast<__half*>(wdbuf + round128(2 * slot_bytes));
  __nv_bfloat16* wrs = (A.Wr != nullptr && wr_bytes(A.E, H) <= kWrSmemMax)
                           ? reinterpret_cast<__nv_bfloat16*>(hst) : nullptr;   // before h

  if (threadIdx.x == 0) {
    for (int q = 0; q < 3; ++q) mbar_init(&bar[q], 1);
    fence_mbar_init();
  }
  load_inputs(A, xs, wrs);
  __syncthreads();
  decode_route(A, xs, wrs, R);

  const int units = (H + kDnRows - 1) / kDnRows;
  const int unit = blockIdx.x;
  const bool active = unit < units;            // uniform across the block
  const int j0 = unit * kDnRows;
  const int rows = active ? min(kDnRows, H - j0) : 0;
  auto issue_wd = [&](int ti, int b) {
    fence_proxy_async_smem();                  // earlier generic reads of this slot come first
    const int e = R.touched[ti];
    const uint32_t bytes = static_cast<uint32_t>(rows) * I * 2;
    mbar_arrive_expect_tx(&bar[b], bytes);
    bulk_load(wdbuf + b * slot_bytes,
              static_cast<const __nv_bfloat16*>(A.wd.p[e]) + static_cast<int64_t>(j0) * I, bytes,
              &bar[b]);
  };
  bool inflight[3] = {false, false, false};    // tracked by thread 0, which issues
  if (threadIdx.x == 0 && active) {
    for (int q = 0; q < 2 && q < R.n_touched; ++q) {
      issue_wd(q, q);
      inflight[q] = true;
    }
  }

  // h comes from kernel A: wait for that grid (and its memory) before staging it
  asm volatile("griddepcontrol.wait;" ::: "memory");

  uint32_t phase[3] = {0, 0, 0};
  bool waited[2] = {false, false};
  bool ok = active;
  int ti = 0;                                  // current touched expert
  for (int q0 = 0; ok && q0 < R.nA;) {
    const int q1 = min(R.nA, q0 + kHStage);
    __syncthreads();                           // the previous stage is no longer read
    if (threadIdx.x == 0) {
      fence_proxy_async_smem();                // earlier generic reads of the stage come first
      mbar_arrive_expect_tx(&bar[2], static_cast<uint32_t>(q1 - q0) * I * 2);
      for (int q = q0; q < q1; ++q)
        bulk_load(hst + static_cast<size_t>(q - q0) * I, A.h + static_cast<int64_t>(R.by_e[q]) * I,
                  static_cast<uint32_t>(I) * 2, &bar[2]);
      inflight[2] = true;
    }
    ok = __syncthreads_and(mbar_wait(&bar[2], phase[2], nullptr, A.hdr, 21));
    if (!ok) break;
    phase[2] ^= 1;
    inflight[2] = false;
    // the touched experts with assignments in [q0, q1), in order
    while (ti < R.n_touched) {
      const int e = R.touched[ti];
      if (R.e_start[e] >= q1) break;           // its rows come with a later stage
      const int ea = max(R.e_start[e], q0), eb = min(R.e_start[e + 1], q1);
      const int b = ti & 1;
      if (!waited[b]) {
        ok = __syncthreads_and(mbar_wait(&bar[b], phase[b], nullptr, A.hdr, 22));
        if (!ok) break;
        waited[b] = true;
      }
      const __nv_bfloat16* ws = reinterpret_cast<const __nv_bfloat16*>(wdbuf + b * slot_bytes);
      // warp w: row w % kDnRows; the assignments of e in this stage, four at a
      // time, round-robin over the kDecWarps / kDnRows warps of that row
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
      if (R.e_start[e + 1] > q1) break;        // e continues in the next stage
      // e is done: its slot takes the expert after next
      __syncthreads();
      phase[b] ^= 1;
      waited[b] = false;
      if (threadIdx.x == 0) {
        inflight[b] = false;
        if (ti + 2 < R.n_touched) {
          issue_wd(ti + 2, b);
          inflight[b] = true;
        }
      }
      ++ti;
    }
    q0 = q1;
  }
  __syncthreads();
  if (!ok) {
    if (threadIdx.x == 0)
      for (int q = 0; q < 3; ++q)
        if (inflight[q]) mbar_wait(&bar[q], phase[q], nullptr, nullptr, 23);
    return;
  }
  const int kk = (A.Wr != nullptr) ? A.k : 1;
  for (int q = threadIdx.x; q < A.T * rows; q += blockDim.x) {
    const int t = q / rows, jl = q % rows;
    float v = 0.f;
    for (int s = 0; s < kk; ++s) v += R.sel_a[t * kk + s] * part[t * kk + s][jl];
    static_cast<__nv_bfloat16*>(A.y)[static_cast<int64_t>(t) * H + j0 + jl] = __float2bfloat16_rn(v);
  }
}

size_t decode_smem_bytes(int T, int H, int I) {
  const size_t a = smem_a_bytes(T, H, MM_MAX_EXPERTS);
  const size_t b = smem_b_bytes(T, H, I, MM_MAX_EXPERTS);
  return a > b ? a : b;
}

cudaError_t launch_decode_ffn(const void* x, const void* Wr, const float* bias,
                              const void* const* Wg, const void* const* Wu, const void* const* Wd,
                              int T, int H, int I, int E, int k, float coef, int32_t* topk_idx,
                              float* topk_w, float* aux_loss, float* hbuf, void* y, WsHeader* hdr,
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
  A.h = reinterpret_cast<__half*>(hbuf); A.y = y; A.hdr = hdr;
  const size_t sa = smem_a_bytes(T, H, nw), sb = smem_b_bytes(T, H, I, nw);
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(decode_gateup_kernel), sa);
  if (e != cudaSuccess) return e;
  e = ensure_dynamic_smem(reinterpret_cast<const void*>(decode_down_kernel), sb);
  if (e != cudaSuccess) return e;
  const int gridA = 2 * num_sms();
  decode_gateup_kernel<<<gridA, kDecThreads, sa, st>>>(A);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // kernel B as a programmatic dependent of A: its prologue overlaps A
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((H + kDnRows - 1) / kDnRows);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = sb;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_down_kernel, A);
}

}  // namespace mm
