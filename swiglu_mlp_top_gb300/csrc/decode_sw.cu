// Dense SwiGLU FFN for up to 128 tokens on the 5th-generation tensor cores,
// with the operands swapped against decode_tc.cu: the tokens are the UMMA M
// operand (TMEM lane = token; rows past T are never stored), the weights the
// N operand.  A unit is R rows of I (R = 32 up to 64 tokens, else 64), so a
// dense FFN has 76 or 38 units at I = 2432 where decode_tc.cu's 128-row M
// tiles give it only 19.
//
// Per unit (MiniMind lesson 13 §0 / §1.2; minimind3.com chapter 4 §4.2):
//   gate/up   G, U [T x R] = x [T x H] . Wg/Wu[R rows, H]^T, K = H in
//             stages of nkb 64-wide k-blocks of x, Wg and Wu, each fetched by
//             one 3-D TMA box (a box of 8 KiB moves ~30 GB/s per SM, one of
//             32 KiB ~95 GB/s); TMEM, N = R each
//   epilogue  h = SiLU(G) * U, split into a bf16 high part and a bf16
//             remainder, written as two 128-row A tiles (128-byte swizzle)
//   down      y_u [T x H] = h . Wd[:, unit's R columns]^T, N = 128 output
//             columns per MMA, two 128-column blocks of y per TMEM pass and
//             per box of Wd; two TMEM buffers, so that the epilogue drains
//             one pass while the next accumulates
//   partial   y_u (fp32, tokens < T) to global memory, 4-column groups in
//             token order so that the lanes of a store write one run
// then one grid barrier and every CTA adds a share of the unit partials in
// unit order (deterministic) and rounds y to bf16 once.
//
// Warp roles (320 threads): warp 0 lane 0 issues TMA, warp 1 lane 0 issues
// UMMA and owns TMEM, warps 2-9 are the epilogue (TMEM lane quadrant
// warp % 4, column half (warp - 2) / 4).  Every wait is bounded.
#include <mutex>

#include "mm_kernels.cuh"

namespace mm {

constexpr int kSwThreads = 320;

constexpr int kSwMaxStages = 8;
// Unit geometry for R rows of I per unit (R = 32 or 64): h and Wd tiles are
// K-major with K = R, rows of 2R bytes, 128-byte swizzle for R = 64 and
// 64-byte swizzle for R = 32.
template <int R>
struct SwUnit {
  static_assert(R == 32 || R == 64, "unit rows");
  static constexpr int kWTile = R * 128;         // one k-block of the unit's Wg (or Wu) rows
  static constexpr int kHRow = R * 2;
  static constexpr int kDTile = 128 * kHRow;     // 128 rows of h, or 128 rows of Wd x R
  static constexpr int kKSteps = R / 16;         // UMMA k-steps of the down product
  __device__ static __forceinline__ uint64_t desc(uint32_t saddr) {
    return R == 64 ? smem_desc_sw128(saddr) : smem_desc_sw64(saddr);
  }
};
constexpr uint32_t kSwTmemCols = 512;
constexpr uint32_t kSwColG = 0, kSwColU = 64;    // gate/up accumulators
constexpr uint32_t kSwBufCols = 256;             // y: two buffers of two 128-column blocks
constexpr int kSwPassBlocks = 2;                 // (G and U use buffer 0 before the first pass)
constexpr int kSwEpiWarps = 8;
constexpr int kSwMaxCtas = 160;
constexpr int kSwMaxSlices = 16;                 // final sum: threads per output quad at most
constexpr int kSwSumChunk = 16;                  // final sum: partials requested at once
constexpr size_t kSwSmemBudget = 200 * 1024;

struct SwMaps {
  CUtensorMap x;                  // x as (64, T, H / 64), box 64 x Np x nkb (rows >= T read as 0)
  CUtensorMap wg, wu;             // [I, H] as (64, I, H / 64), box 64 x R x nkb
  CUtensorMap wd;                 // [H, I] as (I, 128, H / 128), box R x 128 x 2
};

struct SwArgs {
  int T, Np, H, I, n_units, stages;
  int nkb;                        // k-blocks per gate/up stage
  uint32_t stage_bytes;           // nkb x tiles + nkb Wg tiles + nkb Wu tiles, or three Wd tiles
  uint32_t xtile;                 // Np * 128 bytes
  uint32_t h_off;                 // two h tiles (high part, remainder), 256 R bytes each
  float* pd;                      // [n_units][H / 4][T][4] fp32 partials
  void* y;                        // [T, H] bf16
  WsHeader* hdr;
  int pdl;                        // launched as a programmatic dependent (see the kernel)
};

__device__ __forceinline__ float sw_swiglu(float g, float u) {
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

template <int R>
__global__ void __launch_bounds__(kSwThreads, 1)
decode_sw_kernel(const __grid_constant__ SwMaps M, const SwArgs A) {
  using U = SwUnit<R>;
  constexpr int kSwRows = R;
  constexpr int kSwWTile = U::kWTile;
  constexpr int kSwHRow = U::kHRow;
  constexpr int kSwDTile = U::kDTile;
  constexpr int kSwKSteps = U::kKSteps;
  extern __shared__ unsigned char smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* ring = smem;
  uint8_t* hhi = smem + A.h_off;
  uint8_t* hlo = hhi + kSwDTile;
  __shared__ __align__(8) uint64_t full[kSwMaxStages], empty[kSwMaxStages];
  __shared__ __align__(8) uint64_t tfull, tempty, hfull, hempty, yfull[2], yempty[2], drained;
  __shared__ uint32_t s_tmem;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int T = A.T, H = A.H, S = A.stages;
  const uint32_t SB = A.stage_bytes;
  const int KB_H = H / 64, MB_H = H / 128;
  const int n_pass = (MB_H + kSwPassBlocks - 1) / kSwPassBlocks;
  WsHeader* hdr = A.hdr;
  const bool epi = warp >= 2;
  const int quad = warp & 3;
  const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;

  if (tid == 0) {
    for (int s = 0; s < kSwMaxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull, 1);
    mbar_init(&tempty, kSwEpiWarps);
    mbar_init(&hfull, kSwEpiWarps);
    mbar_init(&hempty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&yfull[b], 1);
      mbar_init(&yempty[b], kSwEpiWarps);
    }
    mbar_init(&drained, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, kSwTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  int p_it = 0, m_it = 0;
  bool ok = true;
  auto acquire = [&](int& s) -> bool {
    s = p_it % S;
    return mbar_wait(&empty[s], ((p_it / S) & 1) ^ 1, nullptr, hdr, 60);
  };
  auto consume = [&](int& s) -> bool {
    s = m_it % S;
    const bool r = mbar_wait(&full[s], (m_it / S) & 1, nullptr, hdr, 61);
    tc_fence_after();
    return r;
  };
  auto sdesc = [&](const uint8_t* p) { return smem_desc_sw128(smem_u32(p)); };

  const int nkb = A.nkb;
  const uint32_t xpart = static_cast<uint32_t>(nkb) * A.xtile;       // x tiles of a stage
  const uint32_t wpart = static_cast<uint32_t>(nkb) * kSwWTile;       // Wg (or Wu) tiles of a stage
  if (tid == 0) {
    // gate/up stage = nkb x tiles, nkb Wg tiles, nkb Wu tiles.  An x tile is
    // the A operand: 128 rows are read, and the tiles behind it fill rows
    // >= Np, whose products land in TMEM lanes that are never read.  A down
    // stage = the three Wd tiles of one TMEM pass (blocks past H read as 0).
    //
    // As a programmatic dependent of the previous call, the weights of the
    // first S stages are requested before griddepcontrol.wait (they need
    // nothing from the previous kernel); the x tiles of those stages wait for
    // it, and are requested before any stage is reused.
    const uint64_t pol = l2_evict_first_policy();
    bool waited = !A.pdl;
    int n_def = 0, def_s[kSwMaxStages], def_kb[kSwMaxStages];
    auto flush = [&]() {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      waited = true;
      for (int i = 0; i < n_def; ++i)
        tma_load_3d(ring + def_s[i] * SB, &M.x, &full[def_s[i]], 0, 0, def_kb[i]);
      n_def = 0;
    };
    for (int u = cta; ok && u < A.n_units; u += G) {
      for (int kb0 = 0; kb0 < KB_H; kb0 += nkb) {
        if (!waited && p_it >= S) flush();
        int s;
        if (!acquire(s)) { ok = false; break; }
        uint8_t* st = ring + s * SB;
        mbar_arrive_expect_tx(&full[s], xpart + 2 * wpart);
        if (waited) {
          tma_load_3d(st, &M.x, &full[s], 0, 0, kb0);
        } else {
          def_s[n_def] = s;
          def_kb[n_def] = kb0;
          ++n_def;
        }
        tma_load_3d_hint(st + xpart, &M.wg, &full[s], 0, u * kSwRows, kb0, pol);
        tma_load_3d_hint(st + xpart + wpart, &M.wu, &full[s], 0, u * kSwRows, kb0, pol);
        ++p_it;
      }
      for (int p = 0; ok && p < n_pass; ++p) {
        if (!waited && p_it >= S) flush();
        int s;
        if (!acquire(s)) { ok = false; break; }
        mbar_arrive_expect_tx(&full[s], kSwPassBlocks * kSwDTile);
        tma_load_3d_hint(ring + s * SB, &M.wd, &full[s], u * kSwRows, 0, p * kSwPassBlocks, pol);
        ++p_it;
      }
    }
    if (!waited) flush();
  }
  if (tid == 32) {
    const uint32_t idesc_gu = idesc_bf16_f32(128, kSwRows);
    const uint32_t idesc_dn = idesc_bf16_f32(128, 128);
    int j = 0, uses[2] = {0, 0};
    for (int u = cta; ok && u < A.n_units; u += G, ++j) {
      // G, U occupy the first columns of y buffer 0: its last pass must be drained
      if (uses[0] > 0 && !mbar_wait(&yempty[0], (uses[0] - 1) & 1, nullptr, hdr, 62)) { ok = false; break; }
      if (!mbar_wait(&tempty, (j & 1) ^ 1, nullptr, hdr, 62)) { ok = false; break; }
      tc_fence_after();
      for (int kb0 = 0; kb0 < KB_H; kb0 += nkb) {
        int s;
        if (!consume(s)) { ok = false; break; }
        const uint8_t* st = ring + s * SB;
#pragma unroll 1
        for (int kl = 0; kl < nkb; ++kl) {
          const uint8_t* xa = st + kl * A.xtile;
          const uint8_t* wg = st + xpart + kl * kSwWTile;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = sdesc(xa + kk * 32);
            const uint32_t acc = (kb0 + kl || kk) ? 1u : 0u;
            umma_bf16(tmem + kSwColG, a, sdesc(wg + kk * 32), idesc_gu, acc);
            umma_bf16(tmem + kSwColU, a, sdesc(wg + wpart + kk * 32), idesc_gu, acc);
          }
        }
        umma_commit(&empty[s]);
        ++m_it;
      }
      if (!ok) break;
      umma_commit(&tfull);
      if (!mbar_wait(&hfull, j & 1, nullptr, hdr, 63)) { ok = false; break; }
      tc_fence_after();
      for (int p = 0; ok && p < n_pass; ++p) {
        const int b = p & 1;              // TMEM buffer of this pass
        if (!mbar_wait(&yempty[b], (uses[b] & 1) ^ 1, nullptr, hdr, 64)) { ok = false; break; }
        tc_fence_after();
        const int nblk = MB_H - p * kSwPassBlocks < kSwPassBlocks ? MB_H - p * kSwPassBlocks : kSwPassBlocks;
        int s;
        if (!consume(s)) { ok = false; break; }
        const uint8_t* st = ring + s * SB;
        for (int q = 0; q < nblk; ++q) {
          const uint32_t d = tmem + b * kSwBufCols + q * 128;
          const uint8_t* wd = st + q * kSwDTile;
#pragma unroll
          for (int kk = 0; kk < kSwKSteps; ++kk)
            umma_bf16(d, U::desc(smem_u32(hhi + kk * 32)), U::desc(smem_u32(wd + kk * 32)), idesc_dn,
                      kk ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < kSwKSteps; ++kk)
            umma_bf16(d, U::desc(smem_u32(hlo + kk * 32)), U::desc(smem_u32(wd + kk * 32)), idesc_dn, 1u);
        }
        umma_commit(&empty[s]);
        ++m_it;
        umma_commit(&yfull[b]);
        ++uses[b];
      }
      if (!ok) break;
      umma_commit(&hempty);
    }
  }
  if (epi) {
    // warp (quad, half): tokens 32 quad .. 32 quad + 31, half of the columns;
    // a quad with no token below T has nothing to compute or store
    const int half = (warp - 2) >> 2;
    const int t = quad * 32 + lane;            // TMEM lane = token
    const bool quad_live = quad * 32 < T, live = t < T;
    // the partials of y go to the workspace the previous call also used
    if (A.pdl) asm volatile("griddepcontrol.wait;" ::: "memory");
    int j = 0, uses[2] = {0, 0};
    for (int u = cta; ok && u < A.n_units; u += G, ++j) {
      if (!warp_wait(&tfull, j & 1, nullptr, hdr, 65)) { ok = false; break; }
      if (j > 0 && !warp_wait(&hempty, (j - 1) & 1, nullptr, hdr, 66)) { ok = false; break; }
      tc_fence_after();
      // row t of the two h tiles: R values in 16-byte chunks, chunk c stored
      // at chunk position c ^ (t % 8) (128-byte rows) or c ^ ((t / 2) % 4)
      // (64-byte rows); this warp writes the chunks of columns
      // half * R / 2 .. (half + 1) * R / 2
      if (quad_live) {
#pragma unroll 1
        for (int c0 = half * (kSwRows / 2); c0 < (half + 1) * (kSwRows / 2); c0 += 16) {
          uint32_t gr[16], ur[16];
          tmem_ld_32x32b_x16(tmem + lane_base + kSwColG + c0, gr);
          tmem_ld_32x32b_x16(tmem + lane_base + kSwColU + c0, ur);
          tmem_ld_wait();
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int i0 = hc * 8 + 2 * q;
              const float v0 = sw_swiglu(__uint_as_float(gr[i0]), __uint_as_float(ur[i0]));
              const float v1 = sw_swiglu(__uint_as_float(gr[i0 + 1]), __uint_as_float(ur[i0 + 1]));
              const __nv_bfloat16 h0 = __float2bfloat16_rn(v0), h1 = __float2bfloat16_rn(v1);
              hi[q] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
                      (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
              lo[q] = pack_bf16x2(v0 - __bfloat162float(h0), v1 - __bfloat162float(h1));
            }
            const int chunk = (c0 >> 3) + hc;
            const int pos = kSwRows == 64 ? (chunk ^ (t & 7)) : (chunk ^ ((t >> 1) & 3));
            const uint32_t off = static_cast<uint32_t>(t) * kSwHRow + (pos << 4);
            *reinterpret_cast<uint4*>(hhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(hlo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&hfull);
        mbar_arrive(&tempty);
      }
      // this unit's partial of y, one TMEM pass at a time, stored as 4-column
      // groups g = column / 4 in token order, pd[u][g][t][4]: the lanes
      // (tokens) of one store write one contiguous run
      float4* pu = reinterpret_cast<float4*>(A.pd) + static_cast<size_t>(u) * T * (H / 4) + t;
      for (int p = 0; ok && p < n_pass; ++p) {
        const int b = p & 1;
        if (!warp_wait(&yfull[b], uses[b] & 1, nullptr, hdr, 67)) { ok = false; break; }
        tc_fence_after();
        const int nblk = MB_H - p * kSwPassBlocks < kSwPassBlocks ? MB_H - p * kSwPassBlocks : kSwPassBlocks;
        if (quad_live) {
#pragma unroll 1
          for (int q = 0; q < nblk; ++q) {
            const int col0 = q * 128 + half * 64;          // this warp's 64 columns of block q
            uint32_t r0[32], r1[32];
            tmem_ld_32x32b_x32(tmem + lane_base + b * kSwBufCols + col0, r0);
            tmem_ld_32x32b_x32(tmem + lane_base + b * kSwBufCols + col0 + 32, r1);
            tmem_ld_wait();
            if (live) {
              const int g0 = ((p * kSwPassBlocks + q) * 128 + half * 64) / 4;
#pragma unroll
              for (int w = 0; w < 8; ++w)
                pu[static_cast<size_t>(g0 + w) * T] =
                    make_float4(__uint_as_float(r0[4 * w]), __uint_as_float(r0[4 * w + 1]),
                                __uint_as_float(r0[4 * w + 2]), __uint_as_float(r0[4 * w + 3]));
#pragma unroll
              for (int w = 0; w < 8; ++w)
                pu[static_cast<size_t>(g0 + 8 + w) * T] =
                    make_float4(__uint_as_float(r1[4 * w]), __uint_as_float(r1[4 * w + 1]),
                                __uint_as_float(r1[4 * w + 2]), __uint_as_float(r1[4 * w + 3]));
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&yempty[b]);
        ++uses[b];
      }
    }
  }
  tc_fence_before();
  ok = __syncthreads_and(ok);
  tc_fence_after();

  // y = the unit partials added in unit order; each CTA takes a contiguous
  // range of quads q = g * T + t (columns 4g .. 4g + 3 of token t), up to
  // kSwMaxSlices threads share a quad
  unsigned ticket = 0xffffffffu;
  // the barrier's counters are the previous call's too: every thread has
  // waited for that kernel (the producer and epilogue above; the rest here)
  if (A.pdl) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (ok) ok = grid_barrier(hdr, 68, 1, &ticket);
  // every CTA of this grid is resident once it passes the barrier: only now
  // may the next kernel start taking the SMs that this one leaves
  if (A.pdl && threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (ok) {
    const int Gp = A.n_units;
    const int nq_all = T * H / 4;
    const int q0 = static_cast<int>(static_cast<long long>(cta) * nq_all / G);
    const int nq = static_cast<int>(static_cast<long long>(cta + 1) * nq_all / G) - q0;
    if (nq > 0) {
      int ns = kSwThreads / nq;
      ns = ns < 1 ? 1 : (ns > kSwMaxSlices ? kSwMaxSlices : ns);
      ns = ns > Gp ? Gp : ns;
      float4* red = reinterpret_cast<float4*>(ring);
      const float4* pd4 = reinterpret_cast<const float4*>(A.pd) + q0;
      for (int w = tid; w < nq * ns; w += kSwThreads) {
        const int sl = w / nq, qi = w - sl * nq;
        const int c0 = sl * Gp / ns, c1 = (sl + 1) * Gp / ns;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int cb = c0; cb < c1; cb += kSwSumChunk) {
          float4 part[kSwSumChunk];
#pragma unroll
          for (int w2 = 0; w2 < kSwSumChunk; ++w2)
            part[w2] = cb + w2 < c1 ? __ldcg(pd4 + static_cast<size_t>(cb + w2) * nq_all + qi)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int w2 = 0; w2 < kSwSumChunk; ++w2) {
            v.x += part[w2].x; v.y += part[w2].y; v.z += part[w2].z; v.w += part[w2].w;
          }
        }
        red[w] = v;
      }
      __syncthreads();
      for (int qi = tid; qi < nq; qi += kSwThreads) {
        float4 v = red[qi];
        for (int sl = 1; sl < ns; ++sl) {
          const float4 o = red[sl * nq + qi];
          v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
        }
        uint2 pk;
        pk.x = pack_bf16x2(v.x, v.y);
        pk.y = pack_bf16x2(v.z, v.w);
        const int q = q0 + qi, g = q / T, t = q - g * T;
        reinterpret_cast<uint2*>(A.y)[static_cast<size_t>(t) * (H / 4) + g] = pk;
      }
    }
  }

  if (tid == 32) {
    umma_commit(&drained);              // every issued UMMA has finished
    mbar_wait(&drained, 0, nullptr, hdr, 69);
  }
  if (tid == 0 && !ok) {
    for (int j = 0; j < S && j < p_it; ++j) {   // copies in flight land before exit
      const int q = p_it - 1 - j;
      mbar_wait(&full[q % S], (q / S) & 1, nullptr, nullptr, 70);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kSwTmemCols);
  if (tid == 0) grid_barrier_reset(hdr, ticket);
}

// =============================================================== host side
namespace {

struct SwLayout {
  int R, Np, stages, n_units, nkb;
  size_t xtile, stage, h_off, smem, pd;
};

inline size_t sw_round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool sw_layout(int T, int H, int I, SwLayout& L) {
  if (T < 1 || T > kDecodeSwMaxT || H % 128 != 0 || I % 64 != 0) return false;
  L.Np = (T + 15) / 16 * 16;
  // 32-row units: twice the streaming CTAs; 64-row units: half the partials
  // of y, which pays from about 100 tokens (measured: T = 16 / 64 / 100 took
  // 14.7 / 17.2 / 21.2 us with 32 rows, 15.6 / 17.7 / 20.6 with 64)
  L.R = L.Np <= 64 ? 32 : 64;
  const int kSwWTile = L.R * 128;
  const int kSwDTile = 128 * L.R * 2;
  L.n_units = I / L.R;
  L.xtile = static_cast<size_t>(L.Np) * 128;
  // the most k-blocks per gate/up stage (larger TMA boxes stream faster)
  // that leave three stages (else two); a stage also holds one pass of Wd
  const size_t h = 2 * static_cast<size_t>(kSwDTile);
  const int KB_H = H / 64;
  L.nkb = 0;
  for (int min_stages = 3; min_stages >= 2 && L.nkb == 0; --min_stages) {
    for (int nkb = 4; nkb >= 1 && L.nkb == 0; --nkb) {
      if (KB_H % nkb != 0 || (min_stages == 3 && nkb == 1)) continue;
      const size_t st = sw_round_up(std::max(nkb * (L.xtile + 2 * kSwWTile),
                                             static_cast<size_t>(kSwPassBlocks) * kSwDTile), 1024);
      if (kSwSmemBudget >= 1024 + h + static_cast<size_t>(min_stages) * st) {
        L.nkb = nkb;
        L.stage = st;
      }
    }
  }
  if (L.nkb == 0) return false;
  L.stages = static_cast<int>((kSwSmemBudget - 1024 - h) / L.stage);
  if (L.stages > kSwMaxStages) L.stages = kSwMaxStages;
  L.h_off = static_cast<size_t>(L.stages) * L.stage;
  L.smem = L.h_off + h + 1024;
  L.pd = sw_round_up(static_cast<size_t>(L.n_units) * T * H * 4, 256);
  return true;
}

}  // namespace

size_t decode_sw_bytes(int T, int H, int I) {
  SwLayout L;
  return sw_layout(T, H, I, L) ? L.pd : 0;
}

cudaError_t launch_decode_sw(const void* x, const void* Wg, const void* Wu, const void* Wd, int T,
                             int H, int I, void* scratch, void* y, WsHeader* hdr, cudaStream_t st) {
  SwLayout L;
  if (!sw_layout(T, H, I, L)) return cudaErrorInvalidValue;
  static SwMaps m;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  {
    // k-block views: element (e, row, kb) of a [rows, H] matrix at row * H + kb * 64 + e
    const uint64_t sx[2] = {static_cast<uint64_t>(H) * 2, 128};
    const uint64_t dx[3] = {64, static_cast<uint64_t>(T), static_cast<uint64_t>(H / 64)};
    const uint32_t bx[3] = {64, static_cast<uint32_t>(L.Np), static_cast<uint32_t>(L.nkb)};
    if (!make_map_3d(&m.x, x, dx, sx, bx)) return cudaErrorInvalidValue;
    const uint64_t dw[3] = {64, static_cast<uint64_t>(I), static_cast<uint64_t>(H / 64)};
    const uint32_t bw[3] = {64, static_cast<uint32_t>(L.R), static_cast<uint32_t>(L.nkb)};
    if (!make_map_3d(&m.wg, Wg, dw, sx, bw)) return cudaErrorInvalidValue;
    if (!make_map_3d(&m.wu, Wu, dw, sx, bw)) return cudaErrorInvalidValue;
    // Wd [H, I] as (i, row within a 128-row block, block)
    const uint64_t sd[2] = {static_cast<uint64_t>(I) * 2, static_cast<uint64_t>(I) * 2 * 128};
    const uint64_t dd[3] = {static_cast<uint64_t>(I), 128, static_cast<uint64_t>(H / 128)};
    const uint32_t bd[3] = {static_cast<uint32_t>(L.R), 128, static_cast<uint32_t>(kSwPassBlocks)};
    if (!make_map_3d(&m.wd, Wd, dd, sd, bd, false,
                     L.R == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  }
  SwArgs A;
  memset(&A, 0, sizeof(A));
  A.T = T; A.Np = L.Np; A.H = H; A.I = I; A.n_units = L.n_units; A.stages = L.stages;
  A.nkb = L.nkb;
  A.stage_bytes = static_cast<uint32_t>(L.stage);
  A.xtile = static_cast<uint32_t>(L.xtile);
  A.h_off = static_cast<uint32_t>(L.h_off);
  A.pd = static_cast<float*>(scratch);
  A.y = y;
  A.hdr = hdr;
  auto fn = L.R == 64 ? decode_sw_kernel<64> : decode_sw_kernel<32>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), L.smem);
  if (e != cudaSuccess) return e;
  int fit = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, fn, kSwThreads, L.smem);
  if (e != cudaSuccess) return e;
  if (fit < 1) return cudaErrorInvalidConfiguration;
  int grid = num_sms();
  if (grid > kSwMaxCtas) grid = kSwMaxCtas;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSwThreads);
  cfg.dynamicSmemBytes = L.smem;
  cfg.stream = st;
  // One wave (grid <= SMs x resident CTAs), launched as a programmatic
  // dependent of the previous kernel: its CTAs start as that kernel's CTAs
  // leave the SMs, and every one of them becomes resident once that kernel
  // ends (no kernel waits for a later one), so the grid barrier needs no
  // cooperative launch.  Its successor starts only after this grid's barrier.
  A.pdl = 1;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, m, A);
}

}  // namespace mm
