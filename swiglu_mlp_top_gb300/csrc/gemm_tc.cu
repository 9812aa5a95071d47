// Grouped GEMMs on the 5th-generation tensor cores: tcgen05 UMMA over a CTA
// pair (cta_group::2, M = 256: each CTA of the cluster owns 128 rows of A and
// half of the N columns of B in its shared memory), fp32 accumulators in
// TMEM, operands staged by TMA into a 6-deep shared-memory ring.  Persistent
// and warp-specialised, in each CTA of the pair:
//   warps 0-3  epilogue (TMEM -> registers -> global), one TMEM lane per row
//   warp 4     TMA producer (one elected lane) for this CTA's A and B halves
//   warp 5     (even CTA only) MMA issuer; both CTAs' warp 5 allocate TMEM
// Two TMEM accumulators let the epilogue of tile i overlap the MMAs of i+1.
// Splitting B across the pair halves the shared-memory traffic per SM, which
// a single-CTA M = 128 tile saturates before the tensor pipe.
//
// gate/up:  for the rows of group g:  G = A Wg^T, U = A Wu^T  (bf16; N = 256:
//           the even CTA stages Wg rows n0..n0+127, the odd CTA the same Wu
//           rows), epilogue h = SiLU(G) ⊙ U -> fp16.  G and U stay in TMEM.
//           (MiniMind lesson 13 "FFN 与 MoE" §0/§1.2 equations; minimind3.com
//           chapter 4 §4.2.)  h is stored in fp16 (11-bit significand): bf16
//           storage of h alone added ~0.005 RMS-relative max error on top of
//           the unavoidable bf16 rounding of y.
// down:     Y = h Wd^T (fp16 x fp16, Wd converted from bf16 exactly; N = 256,
//           128 columns of Wd rows per CTA); the epilogue scales each row by
//           its routing weight alpha and stores / accumulates it at the row's
//           token (lesson 13 step 5: expert output times weight, index_add_).
#include <mutex>
#include <map>
#include <tuple>

#include "mm_kernels.cuh"

namespace mm {

// ------------------------------------------------------------------ geometry
constexpr int kOpUp = 0, kOpDown = 1;
// The gate/up GEMM run again in the backward pass: same operands and tiles,
// an epilogue that differentiates the SwiGLU (UpBwd) instead of storing h.
constexpr int kOpUpBwd = 2;
// Smallest magnitude that rounds to infinity in fp16 (65504 + half an ulp).
constexpr float kF16Overflow = 65520.0f;
constexpr int kPairM = 2 * kTcBM;                        // rows per tile pair
constexpr int kN = 256;                                  // UMMA N (both ops)
// The operand ring holds six k-blocks of A and B (16 KiB each per CTA),
// grouped into stages of kKb k-blocks fetched by one 3-D TMA box each:
// gate/up measured 163 us with stages of two k-blocks against 170 with one,
// the down GEMM 61 against 60, so each takes its own.
constexpr int kATile = kTcBM * kTcBK * 2;                // 16 KiB: 128 rows x one k-block
constexpr int kBTile = (kN / 2) * kTcBK * 2;             // 16 KiB: this CTA's half of N x one k-block
constexpr int kRingKb = 6;                               // k-blocks in the ring
constexpr int kAccStride = 256;                          // TMEM columns per accumulator
// Epilogue: 8 warps; warp w reads TMEM lanes 32*(w%4).. (its rows) and
// handles half w/4 of the tile's columns, through a 2 KiB staging tile per
// warp: gate/up stages each 32-row x 32-column fp16 piece in the
// 64-byte-swizzled layout of a TMA box and writes it with one tensor store;
// down transposes 32-row x 16-column fp32 pieces through it.
constexpr int kEpiWarps = 8;
constexpr int kStageEpi = kEpiWarps * 32 * 64;           // 16 KiB
constexpr int kWarpProducer = kEpiWarps, kWarpMma = kEpiWarps + 1;
constexpr int kThreads = 32 * (kEpiWarps + 2);
constexpr int kSmem = kRingKb * (kATile + kBTile) + kStageEpi + 2048;
// Wide down tile (N = 384 as two MMAs of N = 192, one 384-column
// accumulator): taken when it makes every tile pair fit in one wave.  Each
// CTA stages 192 rows of Wd per k-block (two boxes of 96), so the ring holds
// five k-blocks.
constexpr int kNWide = 384;
constexpr int kRingKbWide = 5;
constexpr int kSmemWide = kRingKbWide * (kATile + (kNWide / 2) * kTcBK * 2) + kStageEpi + 2048;
static_assert(kSmemWide <= 232448 - 8192, "shared memory budget (wide down tile)");
constexpr uint32_t kTmemCols = 512;
static_assert(kSmem <= 232448, "shared memory budget");

// Per op: output columns per tile, k-blocks per TMA stage, k-blocks in the
// ring, epilogue staging bytes.  The backward gate/up stages three 2 KiB
// pieces per warp (dG, dU, alpha h; one tensor store each), paid for with a
// ring of five k-blocks.
template <int OP> struct OpTraits;
template <> struct OpTraits<kOpUp> {
  static constexpr int kOutCols = kN / 2, kKb = 2, kRing = kRingKb, kStage = kStageEpi;
};
template <> struct OpTraits<kOpUpBwd> {
  static constexpr int kOutCols = kN / 2, kKb = 1, kRing = 5, kStage = 3 * kStageEpi;
};
template <> struct OpTraits<kOpDown> {
  static constexpr int kOutCols = kN, kKb = 1, kRing = kRingKb, kStage = kStageEpi;
};
template <int OP>
constexpr int kSmemOf = OpTraits<OP>::kRing * (kATile + kBTile) + OpTraits<OP>::kStage + 2048;
static_assert(kSmemOf<kOpUpBwd> <= 232448, "shared memory budget (backward gate/up)");

template <int MAXW>
struct TcParams {
  CUtensorMap out;          // gate/up: h [a_rows, I] fp16; down of a dense FFN: y [a_rows, H]
                            // bf16; box 32 x 32, 64-byte swizzle (TMA stores)
  CUtensorMap a;            // A [a_rows, K]
  CUtensorMap b0[MAXW];     // gate/up: Wg; down: fp16 Wd  (box rows = N/2)
  CUtensorMap b1[MAXW];     // gate/up: Wu; down: unused
  CUtensorMap ag;           // gate/up gathering rows: x [T, K], box 64 x 1 row
  CUtensorMap out2;         // backward gate/up: alpha h [a_rows, I] bf16 (out: dG|dU [a_rows, 2I])
};

struct TileInfo {
  int g, w, row0, rows, n0;   // group, weight index, this CTA's first row / valid rows, column
};

// Tile-pair t of the grouped problem: groups in order, within a group
// m-blocks of 256 rows, n-blocks fastest.  Binary search over the groups'
// first tiles.  The CTA of rank r takes rows [row0 + 128 r, +128).
__device__ __forceinline__ TileInfo decode_tile(int t, const int* s_off, const int* s_tstart, int G,
                                                int n_weights, int n_tiles, int out_cols,
                                                int rank) {
  int lo = 0, hi = G - 1;            // last group with s_tstart[g] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_tstart[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int g = lo;
  const int local = t - s_tstart[g];
  const int mb = local / n_tiles, nb = local - mb * n_tiles;
  TileInfo ti;
  ti.g = g;
  ti.w = g % n_weights;
  ti.row0 = s_off[g] + mb * kPairM + rank * kTcBM;
  ti.rows = min(kTcBM, s_off[g + 1] - ti.row0);   // may be <= 0 for the odd CTA
  ti.n0 = nb * out_cols;
  return ti;
}

__device__ __forceinline__ void build_schedule(const GroupRows& gr, int n_tiles, int* s_off,
                                               int* s_tstart) {
  int run = 0;
  for (int g = 0; g < gr.G; ++g) {
    const int o0 = gr.offsets ? gr.offsets[g] : 0;
    const int o1 = gr.offsets ? gr.offsets[g + 1] : gr.dense_rows;
    s_off[g] = o0;
    s_tstart[g] = run;
    run += ((o1 - o0 + kPairM - 1) / kPairM) * n_tiles;
  }
  s_off[gr.G] = gr.offsets ? gr.offsets[gr.G] : gr.dense_rows;
  s_tstart[gr.G] = run;
}

// ---------------------------------------------------------------- epilogues
// gate/up: 64 h columns (half `half` of the tile's 128) of one row:
// h = SiLU(g) * u, fp16, as two 32-column pieces.  A warp whose 32 rows are
// all in the group writes each piece with one TMA tensor store from its
// swizzled staging tile; a warp holding a group's ragged end stores its
// valid rows directly (the rows past the end belong to the next group).
// Returns true when some value of the lane's pieces is not representable in
// fp16 (|h| >= 65520 rounds to infinity; a NaN or an infinite g or u).
// One lane's row of a 32-row x 32-column 16-bit piece into a staging tile in
// the 64-byte-swizzled layout of a TMA box: 64-byte rows, 16-byte chunk q of
// row r at chunk q ^ ((r >> 1) & 3).
__device__ __forceinline__ void stage_row64(uint8_t* tile, int lane, const uint32_t* pk) {
  uint8_t* r64 = tile + lane * 64;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(r64 + ((q ^ ((lane >> 1) & 3)) << 4)) =
        make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
}

__device__ __forceinline__ bool epilogue_up(uint32_t tb, const TileInfo& ti, int I, __half* hout,
                                            int row, int half, uint8_t* wstage,
                                            const CUtensorMap* hmap) {
  const int lane = row & 31;
  // |h| as packed fp16 pairs, max over the lane's values (NaN wins): a half
  // with an all-ones exponent (inf or NaN) is a value fp16 cannot hold
  uint32_t hmax = 0u;
  const bool valid = row < ti.rows;
  const bool full_warp = (row | 31) < ti.rows;   // warp-uniform
  const int col0 = ti.n0 + half * 64;
  __half* dst = hout + static_cast<int64_t>(ti.row0 + (valid ? row : 0)) * I + col0;
#pragma unroll 1
  for (int c = 0; c < 2; ++c) {
    const int tcol = half * 64 + c * 32;         // TMEM column of g; u is kN/2 further
    uint32_t gr[32], ur[32];
    tmem_ld_32x32b_x32(tb + tcol, gr);
    tmem_ld_32x32b_x32(tb + kN / 2 + tcol, ur);
    tmem_ld_wait();
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float g0 = __uint_as_float(gr[2 * j]), g1 = __uint_as_float(gr[2 * j + 1]);
      const float u0 = __uint_as_float(ur[2 * j]), u1 = __uint_as_float(ur[2 * j + 1]);
      const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
      const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
      pk[j] = pack_f16x2(h0, h1);
      hmax = hmax2_nan_abs(hmax, pk[j]);
    }
    if (col0 + c * 32 >= I) continue;            // piece past the last column
    if (full_warp) {
      if (lane == 0) bulk_wait_read();             // previous store has read the tile
      __syncwarp();
      stage_row64(wstage, lane, pk);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(hmap, wstage, col0 + c * 32, ti.row0 + (row & ~31));
        bulk_commit();
      }
    } else if (valid) {
      uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
      for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    }
  }
  const bool out_of_range = (hmax & 0x7c00u) == 0x7c00u || (hmax & 0x7c000000u) == 0x7c000000u;
  return out_of_range && valid;
}

// gate/up of the backward: the warp's 32 rows x 64 columns (half `half` of
// the tile's 128) of g and u from TMEM; per element, with s = sigmoid(g):
//   h = g s u;  dalpha += h * dhu;  dh = alpha dhu;  dU = dh g s;
//   dG = dh u s (1 + g (1 - s))
// (the chain rule through lesson 13 §0's h = SiLU(g) ⊙ u).  dG, dU and
// alpha h go out as bf16 in 32-column pieces: a warp whose 32 rows are all
// in the group stages the three pieces and writes each with one TMA tensor
// store (dG and dU through the [rows, 2I] map, alpha h through its own); a
// warp holding a group's ragged end stores its valid rows directly.  The
// row's dalpha partial over these 64 columns goes to
// dalpha_part[row][2 nb + half].  Every lane takes part in the TMEM loads
// (warp-collective); only the rows of the group (`valid`) read dhu and store.
__device__ __forceinline__ void epilogue_up_bwd(uint32_t tb, const TileInfo& ti, int I, int row,
                                                int half, const UpBwd& ub, uint8_t* wstage,
                                                const CUtensorMap* gumap,
                                                const CUtensorMap* hmap) {
  const int lane = row & 31;
  const bool valid = row < ti.rows;              // else: past the group, the next group's row
  const bool full_warp = (row | 31) < ti.rows;   // warp-uniform
  const int64_t r = ti.row0 + (valid ? row : 0);
  float alpha = 1.0f;
  if (valid && ub.perm != nullptr) {
    const int a = ub.perm[r];
    alpha = a >= 0 ? ub.topk_w[a] : 0.0f;        // padding rows: zero gradient
  }
  const int col0 = ti.n0 + half * 64;
  float dpart = 0.f;
#pragma unroll 1
  for (int c = 0; c < 2; ++c) {
    const int col = col0 + c * 32;
    const int tcol = half * 64 + c * 32;         // TMEM column of g; u is kN/2 further
    uint32_t gr[32], ur[32];
    tmem_ld_32x32b_x32(tb + tcol, gr);
    tmem_ld_32x32b_x32(tb + kN / 2 + tcol, ur);
    tmem_ld_wait();
    if (col >= I) continue;                      // warp-uniform
    float dv[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) dv[q] = 0.f;
    if (valid) {
      const uint4* dsrc = reinterpret_cast<const uint4*>(ub.dhu + r * I + col);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = dsrc[q];
        const float2 f0 = f16x2_to_f32x2(v.x), f1 = f16x2_to_f32x2(v.y);
        const float2 f2 = f16x2_to_f32x2(v.z), f3 = f16x2_to_f32x2(v.w);
        dv[8 * q] = f0.x; dv[8 * q + 1] = f0.y; dv[8 * q + 2] = f1.x; dv[8 * q + 3] = f1.y;
        dv[8 * q + 4] = f2.x; dv[8 * q + 5] = f2.y; dv[8 * q + 6] = f3.x; dv[8 * q + 7] = f3.y;
      }
    }
    uint32_t pg[16], pu[16], ph[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float o_g[2], o_u[2], o_h[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float g = __uint_as_float(gr[2 * j + e]);
        const float u = __uint_as_float(ur[2 * j + e]);
        const float d = dv[2 * j + e];
        const float sg = __fdividef(1.0f, 1.0f + __expf(-g));   // 0 once exp(-g) > 2^126
        const float silu = g * sg;
        const float h = silu * u;
        dpart = fmaf(h, d, dpart);
        const float dh = alpha * d;
        o_u[e] = dh * silu;
        o_g[e] = dh * u * (sg * (1.0f + g * (1.0f - sg)));
        o_h[e] = alpha * h;
      }
      pg[j] = pack_bf16x2(o_g[0], o_g[1]);
      pu[j] = pack_bf16x2(o_u[0], o_u[1]);
      ph[j] = pack_bf16x2(o_h[0], o_h[1]);
    }
    if (full_warp) {
      if (lane == 0) bulk_wait_read();           // the previous pieces' stores have read them
      __syncwarp();
      stage_row64(wstage, lane, pg);
      stage_row64(wstage + 2048, lane, pu);
      stage_row64(wstage + 4096, lane, ph);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int rb = ti.row0 + (row & ~31);
        tma_store_2d(gumap, wstage, col, rb);
        tma_store_2d(gumap, wstage + 2048, I + col, rb);
        tma_store_2d(hmap, wstage + 4096, col, rb);
        bulk_commit();
      }
    } else if (valid) {
      uint4* dg = reinterpret_cast<uint4*>(ub.dgu + r * (2 * static_cast<int64_t>(I)) + col);
      uint4* du = reinterpret_cast<uint4*>(ub.dgu + r * (2 * static_cast<int64_t>(I)) + I + col);
      uint4* dh4 = reinterpret_cast<uint4*>(ub.ha + r * I + col);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        dg[q] = make_uint4(pg[4 * q], pg[4 * q + 1], pg[4 * q + 2], pg[4 * q + 3]);
        du[q] = make_uint4(pu[4 * q], pu[4 * q + 1], pu[4 * q + 2], pu[4 * q + 3]);
        dh4[q] = make_uint4(ph[4 * q], ph[4 * q + 1], ph[4 * q + 2], ph[4 * q + 3]);
      }
    }
  }
  if (valid && ub.dalpha_part != nullptr)
    ub.dalpha_part[r * ub.n_parts + (ti.n0 / (kN / 2)) * 2 + half] = dpart;
}

// down: 128 y columns (half `half` of the tile's 256) of the warp's 32 rows,
// scaled by each row's alpha: Store -> y (x's dtype); First -> acc32 = v;
// Accum -> acc32 += v; Last -> y = round(acc32 + v).  The rows are tokens
// scattered over y / acc32, so a thread-per-row store would touch 32 lines
// per instruction.  Instead each 16-column piece goes TMEM -> registers
// (thread = row) -> the warp's 64-byte-row staging tile -> back out with
// lane l on row 8i + l/4, columns 4(l%4)..+3: every global access of the
// warp then covers 8 rows x 64 contiguous bytes.  The running sum is
// requested two pieces ahead of its use.
struct DownRow {
  int64_t tok;
  float alpha;
  bool valid;
};

__device__ __forceinline__ DownRow down_row_info(const TileInfo& ti, const DownEpilogue& ep,
                                                 int row) {
  DownRow d{0, 1.0f, row < ti.rows};
  if (d.valid) {
    const int pos = ti.row0 + row;
    if (ep.perm != nullptr) {
      const int a = ep.perm[pos];
      d.alpha = ep.topk_w != nullptr ? ep.topk_w[a] : 1.0f;
      d.tok = a / ep.k;
    } else {
      d.tok = pos;
    }
  }
  return d;
}

__device__ __forceinline__ bool down_reads_sum(const DownEpilogue& ep) {
  return ep.mode == kCombineAccum || ep.mode == kCombineLast;
}

constexpr int kDnPiece = 16;                    // columns per staged piece

// Rows this lane serves in the transposed phase: 8i + lane/4, i = 0..3.
struct DownLanes {
  int64_t off[4];     // element offset of the row's first column of the tile half
  uint32_t valid;     // bit i: row 8i + lane/4 holds an assignment
};

__device__ __forceinline__ DownLanes down_lanes(const DownRow& d, const TileInfo& ti, int H,
                                                int half, int lane, int hc) {
  DownLanes L;
  const uint32_t vmask = __ballot_sync(0xffffffffu, d.valid);
  const int col0 = ti.n0 + half * hc;
  L.valid = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + (lane >> 2);
    const long long tok = __shfl_sync(0xffffffffu, static_cast<long long>(d.tok), r);
    L.off[i] = tok * H + col0 + 4 * (lane & 3);
    L.valid |= ((vmask >> r) & 1u) << i;
  }
  return L;
}

// the running sum at piece c for the lane's four rows, if the mode reads it
__device__ __forceinline__ void down_prefetch(const DownLanes& L, const DownEpilogue& ep, int c,
                                              float4 (&pre)[4]) {
  if (!down_reads_sum(ep)) return;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if ((L.valid >> i) & 1u)
      pre[i] = __ldcg(reinterpret_cast<const float4*>(ep.acc32 + L.off[i] + c * kDnPiece));
}

// down, dense FFN (rows are tokens in order, alpha = 1, plain store) and a
// warp whose 32 rows are all in the problem: 32-column pieces of bf16 y go
// through the warp's 64-byte-swizzled staging tile and out with one tensor
// store each, like h in the gate/up epilogue.
template <int HC>
__device__ __forceinline__ void epilogue_down_dense(uint32_t tb, const TileInfo& ti, int H,
                                                    int half, int lane, int row_base,
                                                    uint8_t* wstage, const CUtensorMap* ymap,
                                                    const __nv_bfloat16* resid) {
  const int col0 = ti.n0 + half * HC;
#pragma unroll 1
  for (int c = 0; c < HC / 32; ++c) {
    if (col0 + c * 32 >= H) break;               // warp-uniform: past the last column
    uint32_t r0[16], r1[16];
    tmem_ld_32x32b_x16(tb + half * HC + c * 32, r0);
    tmem_ld_32x32b_x16(tb + half * HC + c * 32 + 16, r1);
    tmem_ld_wait();
    if (resid != nullptr) {
      // the block's residual x[row, 32 columns], added before the one rounding
      const uint4* xr = reinterpret_cast<const uint4*>(
          resid + static_cast<int64_t>(row_base + lane) * H + col0 + c * 32);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = xr[q];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t* dst = q < 2 ? r0 : r1;
        const int b = (q & 1) * 8;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          dst[b + 2 * j] = __float_as_uint(__uint_as_float(dst[b + 2 * j]) + __uint_as_float(w[j] << 16));
          dst[b + 2 * j + 1] =
              __float_as_uint(__uint_as_float(dst[b + 2 * j + 1]) + __uint_as_float(w[j] & 0xffff0000u));
        }
      }
    }
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      pk[j] = pack_bf16x2(__uint_as_float(r0[2 * j]), __uint_as_float(r0[2 * j + 1]));
      pk[8 + j] = pack_bf16x2(__uint_as_float(r1[2 * j]), __uint_as_float(r1[2 * j + 1]));
    }
    if (lane == 0) bulk_wait_read();             // the previous store has read the tile
    __syncwarp();
    // 64-byte rows, 16-byte chunk q of row r at chunk q ^ ((r >> 1) & 3)
    uint8_t* r64 = wstage + lane * 64;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(r64 + ((q ^ ((lane >> 1) & 3)) << 4)) =
          make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(ymap, wstage, col0 + c * 32, row_base);
      bulk_commit();
    }
  }
}

template <int HC>
__device__ __forceinline__ void epilogue_down(uint32_t tb, const DownRow& d, const DownLanes& L,
                                              const TileInfo& ti, int H, const DownEpilogue& ep,
                                              int half, int lane, uint8_t* wstage,
                                              float4 (&pre)[4], float4 (&pre2)[4]) {
  const int col0 = ti.n0 + half * HC;
  constexpr int kPieces = HC / kDnPiece;
  const uint32_t st0 = smem_u32(wstage);
  const uint64_t keep = l2_evict_last_policy();
  if (lane == 0) bulk_wait_read();               // a dense tile's tensor stores used the tile
  __syncwarp();
#pragma unroll 1
  for (int c = 0; c < kPieces; ++c) {
    if (col0 + c * kDnPiece >= H) break;         // warp-uniform: past the last column
    uint32_t r[16];
    tmem_ld_32x32b_x16(tb + half * HC + c * kDnPiece, r);
    float4 nxt[4];
    if (c + 2 < kPieces && col0 + (c + 2) * kDnPiece < H) down_prefetch(L, ep, c + 2, nxt);
    tmem_ld_wait();
    __syncwarp();                                // the previous piece has been read back
    // row `lane`: 64 bytes, 16-byte chunk q at q ^ ((lane >> 1) & 3)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t a = st0 + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4);
      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                   "f"(d.alpha * __uint_as_float(r[4 * q])), "f"(d.alpha * __uint_as_float(r[4 * q + 1])),
                   "f"(d.alpha * __uint_as_float(r[4 * q + 2])), "f"(d.alpha * __uint_as_float(r[4 * q + 3]))
                   : "memory");
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = 8 * i + (lane >> 2);
      const uint32_t a = st0 + row * 64 + (((lane & 3) ^ ((row >> 1) & 3)) << 4);
      float4 v;
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a) : "memory");
      if (!((L.valid >> i) & 1u)) continue;
      if (down_reads_sum(ep)) {
        v.x += pre[i].x; v.y += pre[i].y; v.z += pre[i].z; v.w += pre[i].w;
      }
      const int64_t o = L.off[i] + c * kDnPiece;
      if (ep.mode == kCombineFirst || ep.mode == kCombineAccum) {
        // the next slot's launch reads it back: keep it in L2 if it can
        st_f32x4_hint(ep.acc32 + o, v, keep);
      } else {
        if (ep.resid != nullptr) {       // the block's residual, before the one rounding
          const uint2 xr = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(ep.resid) + o);
          v.x += __uint_as_float(xr.x << 16);
          v.y += __uint_as_float(xr.x & 0xffff0000u);
          v.z += __uint_as_float(xr.y << 16);
          v.w += __uint_as_float(xr.y & 0xffff0000u);
        }
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(ep.y) + o) =
            make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      pre[i] = pre2[i];
      pre2[i] = nxt[i];
    }
  }
}

// down, y stored straight from the accumulator (mode Store, no residual:
// top-1 MoE, or a dense warp holding a ragged end): y = round(alpha v), so
// each 32-column piece is scaled and packed to bf16 before the transpose
// (64-byte rows in the staging tile, chunk q of row r at q ^ ((r >> 1) & 3))
// and lane l writes 8 columns (16 bytes) of row 8i + l/4: every warp store
// covers 8 rows x 64 contiguous bytes, with half the store instructions of
// the fp32 transpose above.  Same arithmetic, same bits.
template <int HC>
__device__ __forceinline__ void epilogue_down_store16(uint32_t tb, const DownRow& d,
                                                      const DownLanes& L, const TileInfo& ti,
                                                      int H, const DownEpilogue& ep, int half,
                                                      int lane, uint8_t* wstage) {
  const int col0 = ti.n0 + half * HC;
  const uint32_t st0 = smem_u32(wstage);
  if (lane == 0) bulk_wait_read();               // a dense tile's tensor stores used the tile
  __syncwarp();
  __nv_bfloat16* y = static_cast<__nv_bfloat16*>(ep.y);
#pragma unroll 1
  for (int c = 0; c < HC / 32; ++c) {
    if (col0 + c * 32 >= H) break;               // warp-uniform: past the last column
    uint32_t r[32];
    tmem_ld_32x32b_x32(tb + half * HC + c * 32, r);
    tmem_ld_wait();
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      pk[j] = pack_bf16x2(d.alpha * __uint_as_float(r[2 * j]), d.alpha * __uint_as_float(r[2 * j + 1]));
    __syncwarp();                                // the previous piece has been read back
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t a = st0 + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(pk[4 * q]),
                   "r"(pk[4 * q + 1]), "r"(pk[4 * q + 2]), "r"(pk[4 * q + 3])
                   : "memory");
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = 8 * i + (lane >> 2);
      const uint32_t a = st0 + row * 64 + (((lane & 3) ^ ((row >> 1) & 3)) << 4);
      uint4 v;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
      if (!((L.valid >> i) & 1u)) continue;
      // L.off: the row's first column plus 4 (lane & 3); here 8 (lane & 3)
      *reinterpret_cast<uint4*>(y + L.off[i] + 4 * (lane & 3) + c * 32) = v;
    }
  }
}

// --------------------------------------------------------- fp16 copy of Wd
// The copy works in batches of four 16-byte vectors per epilogue thread
// (16 KiB per CTA): vectors v + t + j * 256 of one index space over the
// matrices, below v1.  A tile's first batch is requested before the
// epilogue waits for the tile's accumulator and written after its epilogue,
// so the load latency hides behind the wait; the bf16 weights are read once
// (evict-first), the fp16 copy stays in L2 for the down GEMM.
constexpr int kCvStride = kEpiWarps * 32;
constexpr int kCvBatch = 4 * kCvStride;

__device__ __forceinline__ void cv_load(const WdConvert& cv, int64_t v, int64_t v1, int t,
                                        uint4 (&raw)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int64_t u = v + t + j * kCvStride;
    if (u < v1) {
      const int64_t m = u / cv.nvec;
      raw[j] = __ldcs(static_cast<const uint4*>(cv.src.p[m]) + (u - m * cv.nvec));
    }
  }
}

__device__ __forceinline__ bool cv_store(const WdConvert& cv, int64_t v, int64_t v1, int t,
                                         const uint4 (&raw)[4]) {
  uint4* dst = reinterpret_cast<uint4*>(cv.dst);
  bool out_of_range = false;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int64_t u = v + t + j * kCvStride;
    if (u < v1) {
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw[j]);
      uint4 out;
      uint32_t* o = reinterpret_cast<uint32_t*>(&out);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(b[q]);
        o[q] = pack_f16x2(f.x, f.y);
        out_of_range |= !(fabsf(f.x) < kF16Overflow) | !(fabsf(f.y) < kF16Overflow);
      }
      __stcg(dst + u, out);
    }
  }
  return out_of_range;
}

// the batches of [v0, v1) from v onwards, one after the other
__device__ __forceinline__ bool cv_rest(const WdConvert& cv, int64_t v, int64_t v1, int t) {
  bool out_of_range = false;
#pragma unroll 1
  for (; v < v1; v += kCvBatch) {
    uint4 raw[4];
    cv_load(cv, v, v1, t, raw);
    out_of_range |= cv_store(cv, v, v1, t, raw);
  }
  return out_of_range;
}


// =============================================================== kernel
// K = contraction length (H for gate/up, I for down); NCOLS = output width
// (I for gate/up, H for down).  NW = N of a down tile pair: 256 (two TMEM
// accumulators), or kNWide (one accumulator; tiles that fit one wave).
template <int OP, int MAXW, int NW = kN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ TcParams<MAXW> P, const GroupRows g, const int K,
                    const int NCOLS, __half* __restrict__ hout, const DownEpilogue ep,
                    const WdConvert cv, WsHeader* hdr, const int dep_mainloop, const UpBwd ub,
                    const RowGather gat) {
  static_assert(NW == kN || (OP == kOpDown && NW == kNWide), "tile width");
  constexpr bool kWide = NW == kNWide;
  constexpr bool kUpLike = OP != kOpDown;       // gate/up tiles (forward or backward)
  constexpr int kOutCols = kUpLike ? OpTraits<OP>::kOutCols : NW;
  constexpr int kHC = NW / 2;                     // down: columns per epilogue warp half
  extern __shared__ unsigned char smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  constexpr int kKbStage = OpTraits<OP>::kKb;
  constexpr int kStages = (kWide ? kRingKbWide : OpTraits<OP>::kRing) / kKbStage;
  constexpr int kAStage = kKbStage * kATile;
  constexpr int kBTileK = (kUpLike ? kN / 2 : NW / 2) * kTcBK * 2;   // B rows of this CTA, one k-block
  constexpr int kBStage = kKbStage * kBTileK;
  uint8_t* sB = smem + kStages * kAStage;
  uint8_t* sEpi = sB + kStages * kBStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + OpTraits<OP>::kStage);
  uint64_t* full = bars;                  // [kStages] even CTA: both CTAs' bytes
  uint64_t* empty = bars + kStages;       // [kStages] each CTA: released by the pair's MMAs
  uint64_t* tfull = bars + 2 * kStages;   // [2] each CTA: accumulator ready
  uint64_t* tempty = tfull + 2;           // [2] even CTA: both CTAs' epilogues done
  uint64_t* drained = tempty + 2;         // even CTA: all MMAs finished
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_off[kMaxGroups + 1], s_tstart[kMaxGroups + 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
  const int n_tiles = (NCOLS + kOutCols - 1) / kOutCols;
  const int nkb = (K + kTcBK - 1) / kTcBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * kEpiWarps);   // one arrival per epilogue warp of both CTAs
    }
    mbar_init(drained, 1);
    fence_mbar_init();
    s_abort = 0;
    // The group offsets of a grouped problem are written by the previous
    // kernel (the dispatch), which lets this one launch before it writes
    // them: with dep_mainloop the schedule is built only once that kernel
    // has completed.  (The barrier set-up above still overlaps it.)
    if (dep_mainloop && g.offsets != nullptr) asm volatile("griddepcontrol.wait;" ::: "memory");
    build_schedule(g, n_tiles, s_off, s_tstart);
  }
  if (warp == kWarpProducer && lane == 0) tma_prefetch_desc(gat.perm != nullptr ? &P.ag : &P.a);
  if (warp == kWarpMma) {
    tmem_alloc_cta2(&s_tmem, kTmemCols);
    tmem_relinquish_cta2();
  }
  tc_fence_before();
  cluster_sync();            // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int total = s_tstart[g.G];
  volatile int* abort = &s_abort;

  // Programmatic dependent launch: with dep_mainloop the operands come from
  // the previous kernel, so the producer waits for it before the first load
  // and only then lets the next kernel launch (which may then rely on this
  // kernel's inputs being complete); otherwise the next kernel may launch at
  // once.  griddepcontrol is a no-op for a launch without the attribute.
  if (!dep_mainloop && threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == kWarpProducer && OP == kOpUp && gat.perm != nullptr) {
    // ------------------------------------------------ TMA producer, A rows gathered
    // Lane l gathers rows 4l .. 4l + 3 of the CTA's 128 (x rows of their
    // tokens; rows past the problem read row 0, their results are never
    // stored); lane 0 waits for the stage and loads B.  Both k-blocks of a
    // stage are always requested (columns past K read as zero), so every
    // stage carries the same bytes.
    if (dep_mainloop) {
      if (lane == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
      __syncwarp();
      if (lane == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    int it = 0;
    bool ok = true;
    for (int tile = cluster; ok && tile < total; tile += n_clusters) {
      const TileInfo ti = decode_tile(tile, s_off, s_tstart, g.G, g.n_weights, n_tiles, kOutCols,
                                      static_cast<int>(rank));
      int tok[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = ti.row0 + 4 * lane + j;
        tok[j] = r < gat.n_rows ? gat.perm[r] / gat.k : 0;
      }
      const CUtensorMap* bmap = rank == 1 ? &P.b1[ti.w] : &P.b0[ti.w];
      for (int kb = 0; kb < nkb; kb += kKbStage, ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        bool w_ok = true;
        if (lane == 0) w_ok = mbar_wait(&empty[s], ph ^ 1, abort, hdr, 1);
        if (!__shfl_sync(0xffffffffu, w_ok ? 1 : 0, 0)) { ok = false; break; }
        const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
        if (lane == 0) {
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * (kAStage + kBStage));
          tma_load_3d_cta2(sB + s * kBStage, bmap, fb, 0, ti.n0, kb);
        }
#pragma unroll
        for (int kl = 0; kl < kKbStage; ++kl)
          tma_gather4_cta2(sA + s * kAStage + kl * kATile + lane * 4 * 128, &P.ag, fb,
                           (kb + kl) * kTcBK, tok[0], tok[1], tok[2], tok[3]);
      }
    }
    if (!ok && rank == 0 && lane == 0) {
      for (int j = 0; j < kStages; ++j) {
        const int i2 = it - 1 - j;
        if (i2 < 0) break;
        mbar_wait(&full[i2 % kStages], (i2 / kStages) & 1, nullptr, hdr, 2);
      }
    }
    __syncwarp();
  } else if (warp == kWarpProducer) {
    // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      if (dep_mainloop) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      }
      int it = 0;
      bool ok = true;
      for (int tile = cluster; ok && tile < total; tile += n_clusters) {
        const TileInfo ti = decode_tile(tile, s_off, s_tstart, g.G, g.n_weights, n_tiles,
                                        kOutCols, static_cast<int>(rank));
        const CUtensorMap* bmap = (kUpLike && rank == 1) ? &P.b1[ti.w] : &P.b0[ti.w];
        // wide tile: this CTA's B rows are two boxes of 96, Wd rows
        // n0 + 96 rank .. and n0 + 192 + 96 rank .., so that the first MMA
        // (N = 192) yields y columns n0 .. n0 + 191 and the second the rest
        const int bcoord = kUpLike ? ti.n0
                                         : ti.n0 + static_cast<int>(rank) * (kWide ? kHC / 2 : kHC);
        for (int kb = 0; kb < nkb; kb += kKbStage, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort, hdr, 1)) { ok = false; break; }
          const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * (kAStage + kBStage));
          tma_load_3d_cta2(sA + s * kAStage, &P.a, fb, 0, ti.row0, kb);
          tma_load_3d_cta2(sB + s * kBStage, bmap, fb, 0, bcoord, kb);
          if constexpr (kWide)
            tma_load_3d_cta2(sB + s * kBStage + kBStage / 2, bmap, fb, 0, bcoord + NW / 2, kb);
        }
      }
      if (!ok && rank == 0) {
        // let copies already in flight land before the pair exits
        for (int j = 0; j < kStages; ++j) {
          const int i2 = it - 1 - j;
          if (i2 < 0) break;
          mbar_wait(&full[i2 % kStages], (i2 / kStages) & 1, nullptr, hdr, 2);
        }
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------ MMA issuer (even CTA)
    if (rank == 0 && lane == 0) {
      constexpr uint32_t idesc = kUpLike ? idesc_bf16_f32(kPairM, kN)
                                 : idesc_f16_f32(kPairM, kWide ? NW / 2 : NW);
      int it = 0, local = 0;
      bool ok = true;
      for (int tile = cluster; ok && tile < total; tile += n_clusters, ++local) {
        // wide tiles: one accumulator, so tile i + 1 waits for tile i's epilogue
        const int acc = kWide ? 0 : (local & 1);
        const uint32_t aph = kWide ? (local & 1) : ((local >> 1) & 1);
        if (!mbar_wait(&tempty[acc], aph ^ 1, abort, hdr, 3)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + acc * kAccStride;
        for (int kb = 0; kb < nkb; kb += kKbStage, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!mbar_wait(&full[s], ph, abort, hdr, 4)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kl = 0; kl < kKbStage; ++kl) {
            if (kb + kl >= nkb) break;               // a box past K was zero-filled
            const uint32_t a0 = smem_u32(sA + s * kAStage + kl * kATile);
            const uint32_t b0 = smem_u32(sB + s * kBStage + kl * kBTileK);
#pragma unroll
            for (int kk = 0; kk < kTcBK / 16; ++kk) {
              const uint32_t accf = (kb + kl > 0 || kk > 0) ? 1u : 0u;
              umma_f16_cta2(d, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), idesc, accf);
              if constexpr (kWide)   // the second box: accumulator columns 192 .. 383
                umma_f16_cta2(d + NW / 2, smem_desc_sw128(a0 + kk * 32),
                              smem_desc_sw128(b0 + kBStage / 2 + kk * 32), idesc, accf);
            }
          }
          umma_commit_cta2_mc(&empty[s], 0x3);
        }
        if (!ok) break;
        umma_commit_cta2_mc(&tfull[acc], 0x3);
      }
      // all issued MMAs must finish before TMEM is released
      umma_commit_cta2_mc(drained, 0x1);
      mbar_wait(drained, 0, nullptr, hdr, 5);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue (warps 0-7, both CTAs)
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;
    uint8_t* wstage = sEpi + warp * (OpTraits<OP>::kStage / kEpiWarps);   // this warp's staging
    const uint32_t te0 = mapa_shared(smem_u32(&tempty[0]), 0);
    const uint32_t te1 = mapa_shared(smem_u32(&tempty[1]), 0);
    // the running fp32 sum is the previous kernel's output
    if (OP == kOpDown && (ep.mode == kCombineAccum || ep.mode == kCombineLast))
      asm volatile("griddepcontrol.wait;" ::: "memory");
    // gate/up: this CTA's share of the fp16 Wd copy, one piece before each
    // of its tiles (all of it if it has none).  The previous kernel (and so
    // any earlier reader of the copy) has finished first.
    int64_t cv0 = 0, cv1 = 0;
    int n_local = 0;
    bool range_bad = false;     // gate/up: an h or Wd value beyond the fp16 range
    if (OP == kOpUp && cv.n_mat > 0) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      const int64_t nv = cv.nvec * cv.n_mat;
      cv0 = nv * blockIdx.x / gridDim.x;
      cv1 = nv * (blockIdx.x + 1) / gridDim.x;
      n_local = cluster < total ? (total - cluster + n_clusters - 1) / n_clusters : 0;
      if (n_local == 0) range_bad |= cv_rest(cv, cv0, cv1, threadIdx.x);
    }
    int local = 0;
    for (int tile = cluster; tile < total; tile += n_clusters, ++local) {
      const TileInfo ti = decode_tile(tile, s_off, s_tstart, g.G, g.n_weights, n_tiles, kOutCols,
                                      static_cast<int>(rank));
      const int acc = kWide ? 0 : (local & 1);
      const uint32_t aph = kWide ? (local & 1) : ((local >> 1) & 1);
      DownRow dr{0, 1.0f, false};
      DownLanes dl;
      float4 pre[4], pre2[4];
      if constexpr (OP == kOpDown) {
        // independent of the MMAs: requested while they run
        dr = down_row_info(ti, ep, row);
        // the running sum of this row's 128 columns: pulled into L2 while the
        // MMAs run, so the epilogue's reads of it do not wait on DRAM
        if (down_reads_sum(ep) && dr.valid && ti.n0 + half * kHC < NCOLS) {
          const float* a = ep.acc32 + dr.tok * NCOLS + ti.n0 + half * kHC;
#pragma unroll
          for (int j = 0; j < kHC / 32; ++j)
            if (ti.n0 + half * kHC + j * 32 < NCOLS)
              asm volatile("prefetch.global.L2 [%0];" ::"l"(a + j * 32) : "memory");
        }
        // the block's residual rows: pulled into L2 while the MMAs run
        if (ep.resid != nullptr && dr.valid && ti.n0 + half * kHC < NCOLS &&
            (ep.mode == kCombineStore || ep.mode == kCombineLast)) {
          const __nv_bfloat16* a = static_cast<const __nv_bfloat16*>(ep.resid) + dr.tok * NCOLS +
                                   ti.n0 + half * kHC;
#pragma unroll
          for (int j = 0; j < kHC / 64; ++j)
            if (ti.n0 + half * kHC + j * 64 < NCOLS)
              asm volatile("prefetch.global.L2 [%0];" ::"l"(a + j * 64) : "memory");
        }
        dl = down_lanes(dr, ti, NCOLS, half, lane, kHC);
        if (ti.n0 + half * kHC < NCOLS) down_prefetch(dl, ep, 0, pre);
        if (ti.n0 + half * kHC + kDnPiece < NCOLS) down_prefetch(dl, ep, 1, pre2);
      }
      int64_t ca = 0, cb = 0;           // this tile's piece of the Wd copy
      uint4 craw[4];
      if (OP == kOpUp && n_local > 0) {
        ca = cv0 + (cv1 - cv0) * local / n_local;
        cb = cv0 + (cv1 - cv0) * (local + 1) / n_local;
        cv_load(cv, ca, cb, threadIdx.x, craw);
      }
      if constexpr (OP == kOpUpBwd) {
        // this row's 64 dh columns (fp16): pulled into L2 while the MMAs run
        if (row < ti.rows && ti.n0 + half * 64 < NCOLS) {
          const __half* a = ub.dhu + (ti.row0 + row) * NCOLS + ti.n0 + half * 64;
          asm volatile("prefetch.global.L2 [%0];" ::"l"(a) : "memory");   // 128 bytes: 64 columns
        }
      }
      if (!warp_wait(&tfull[acc], aph, abort, hdr, 6)) break;
      tc_fence_after();
      const uint32_t tb = tmem + (static_cast<uint32_t>(quad * 32) << 16) + acc * kAccStride;
      if constexpr (OP == kOpUp)
        range_bad |= epilogue_up(tb, ti, NCOLS, hout, row, half, wstage, &P.out);
      else if constexpr (OP == kOpUpBwd)
        epilogue_up_bwd(tb, ti, NCOLS, row, half, ub, wstage, &P.out, &P.out2);
      else if (ep.perm == nullptr && ep.mode == kCombineStore && (row | 31) < ti.rows)
        epilogue_down_dense<kHC>(tb, ti, NCOLS, half, lane, ti.row0 + (row & ~31), wstage, &P.out,
                                 static_cast<const __nv_bfloat16*>(ep.resid));
      else if (ep.mode == kCombineStore && ep.resid == nullptr && (NCOLS & 31) == 0)
        epilogue_down_store16<kHC>(tb, dr, dl, ti, NCOLS, ep, half, lane, wstage);
      else
        epilogue_down<kHC>(tb, dr, dl, ti, NCOLS, ep, half, lane, wstage, pre, pre2);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? te1 : te0);
      if (OP == kOpUp && ca < cb) {
        range_bad |= cv_store(cv, ca, cb, threadIdx.x, craw);
        range_bad |= cv_rest(cv, ca + kCvBatch, cb, threadIdx.x);
      }
    }
    if constexpr (OP == kOpUp) report_range(hdr, range_bad, 100);
    bulk_wait_all();   // this warp's tensor stores have landed
  }

  tc_fence_before();
  cluster_sync();            // no CTA leaves while its peer may still signal it
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc_cta2(tmem, kTmemCols);
}

// =============================================================== host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 16-bit row-major [outer, inner] matrix (bf16 or fp16), box = box_inner
// (inner) x box_rows (outer), zero fill outside the matrix.  Cached by
// (ptr, shape, box, type, swizzle).
bool make_map_16(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t outer,
                 uint32_t box_rows, bool is_f16, uint32_t box_inner, CUtensorMapSwizzle swz) {
  using Key = std::tuple<uintptr_t, uint64_t, uint64_t, uint32_t, bool, uint32_t, int>;
  static std::mutex mu;
  static std::map<Key, CUtensorMap> cache;
  const Key key{reinterpret_cast<uintptr_t>(ptr), inner, outer, box_rows, is_f16, box_inner,
                static_cast<int>(swz)};
  std::lock_guard<std::mutex> lock(mu);
  auto itc = cache.find(key);
  if (itc != cache.end()) {
    *out = itc->second;
    return true;
  }
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(out, is_f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         2, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (cache.size() > 4096) cache.clear();
  cache.emplace(key, *out);
  return true;
}

bool make_map_2d(CUtensorMap* out, const void* ptr, bool fp32, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz) {
  using Key = std::tuple<uintptr_t, bool, uint64_t, uint64_t, uint64_t, uint32_t, uint32_t, int>;
  static std::mutex mu;
  static std::map<Key, CUtensorMap> cache;
  const Key key{reinterpret_cast<uintptr_t>(ptr), fp32, inner, outer, row_bytes, box_inner,
                box_rows, static_cast<int>(swz)};
  std::lock_guard<std::mutex> lock(mu);
  auto itc = cache.find(key);
  if (itc != cache.end()) {
    *out = itc->second;
    return true;
  }
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(out, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         2, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (cache.size() > 4096) cache.clear();
  cache.emplace(key, *out);
  return true;
}

bool make_map_3d(CUtensorMap* out, const void* ptr, const uint64_t dims[3],
                 const uint64_t strides[2], const uint32_t box[3], bool is_f16,
                 CUtensorMapSwizzle swz) {
  using Key = std::tuple<uintptr_t, uint64_t, uint64_t, uint64_t, uint64_t, uint64_t, uint32_t,
                         uint32_t, uint32_t, bool, int>;
  static std::mutex mu;
  static std::map<Key, CUtensorMap> cache;
  const Key key{reinterpret_cast<uintptr_t>(ptr), dims[0], dims[1], dims[2], strides[0],
                strides[1], box[0], box[1], box[2], is_f16, static_cast<int>(swz)};
  std::lock_guard<std::mutex> lock(mu);
  auto itc = cache.find(key);
  if (itc != cache.end()) {
    *out = itc->second;
    return true;
  }
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides[0], strides[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(out, is_f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         3, const_cast<void*>(ptr), d, st, bx,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (cache.size() > 4096) cache.clear();
  cache.emplace(key, *out);
  return true;
}

int num_sms() {
  constexpr int kMaxDev = 64;
  static int cached[kMaxDev] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < kMaxDev && cached[dev] > 0) return cached[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  n = n > 0 ? n : 1;
  if (dev >= 0 && dev < kMaxDev) cached[dev] = n;
  return n;
}

cudaError_t ensure_dynamic_smem(const void* fn, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> done;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find({dev, fn});
  if (it != done.end() && it->second >= bytes) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) done[{dev, fn}] = bytes;
  return e;
}

// Launch with programmatic stream serialisation (the kernel may start while
// the previous kernel of the stream finishes; see griddepcontrol in it).
template <typename Kern, typename... Args>
static cudaError_t launch_pdl(Kern fn, int grid, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, args...);
}

// Operand map of a 16-bit row-major [rows, K] matrix (K a multiple of 64) as
// (64 elements, rows, K / 64): box 64 x box_rows x kb, i.e. kb consecutive
// 128-byte-swizzled k-block tiles per TMA.
static bool kblock_map(CUtensorMap* out, const void* ptr, int K, int64_t rows, int box_rows,
                       bool is_f16, int kb) {
  const uint64_t dims[3] = {64, static_cast<uint64_t>(rows), static_cast<uint64_t>(K / 64)};
  const uint64_t strides[2] = {static_cast<uint64_t>(K) * 2, 128};
  const uint32_t box[3] = {64, static_cast<uint32_t>(box_rows), static_cast<uint32_t>(kb)};
  return make_map_3d(out, ptr, dims, strides, box, is_f16);
}

// Upper bound on the tile pairs of a grouped problem with n_tiles column
// tiles (the group sizes are only known on the device).
static int64_t tiles_bound(int64_t a_rows, const GroupRows& g, int n_tiles) {
  if (g.offsets == nullptr)
    return ((g.dense_rows + kPairM - 1) / kPairM) * static_cast<int64_t>(n_tiles);
  return ((a_rows + kPairM - 1) / kPairM + g.G) * static_cast<int64_t>(n_tiles);
}

// Number of CTA pairs: one per tile pair, at most one per co-resident pair.
static int clusters_for(int64_t a_rows, const GroupRows& g, int n_tiles) {
  const int64_t tiles = tiles_bound(a_rows, g, n_tiles);
  const int pairs = num_sms() / 2;
  return static_cast<int>(tiles < pairs ? (tiles > 0 ? tiles : 1) : pairs);
}

template <int MAXW>
static cudaError_t gateup_impl(const void* A, int64_t a_rows, int H, int I, const GroupRows& g,
                               const void* const* Wg, const void* const* Wu, void* h_out,
                               const WdConvert& cv, WsHeader* hdr, cudaStream_t st,
                               const RowGather& gat, int64_t x_rows) {
  TcParams<MAXW> p;
  memset(&p, 0, sizeof(p));
  if (!make_map_16(&p.out, h_out, I, a_rows, 32, true, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  constexpr int kb = OpTraits<kOpUp>::kKb;
  if (gat.perm != nullptr) {
    // A = x [x_rows, H] gathered one row per box row
    if (!make_map_16(&p.ag, A, H, x_rows, 1, false, kTcBK, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else if (!kblock_map(&p.a, A, H, a_rows, kTcBM, false, kb)) {
    return cudaErrorInvalidValue;
  }
  for (int e = 0; e < g.n_weights; ++e) {
    if (!kblock_map(&p.b0[e], Wg[e], H, I, kN / 2, false, kb)) return cudaErrorInvalidValue;
    if (!kblock_map(&p.b1[e], Wu[e], H, I, kN / 2, false, kb)) return cudaErrorInvalidValue;
  }
  auto fn = grouped_gemm_kernel<kOpUp, MAXW>;
  cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), kSmem);
  if (err != cudaSuccess) return err;
  const int n_tiles = (I + kN / 2 - 1) / (kN / 2);
  DownEpilogue none{};
  return launch_pdl(fn, 2 * clusters_for(a_rows, g, n_tiles), kSmem, st, p, g, H, I,
                    static_cast<__half*>(h_out), none, cv, hdr, 1, UpBwd{}, gat);
}

template <int MAXW>
static cudaError_t gateup_bwd_impl(const void* A, int64_t a_rows, int H, int I, const GroupRows& g,
                                   const void* const* Wg, const void* const* Wu, const UpBwd& ub,
                                   WsHeader* hdr, cudaStream_t st) {
  TcParams<MAXW> p;
  memset(&p, 0, sizeof(p));
  constexpr int kb = OpTraits<kOpUpBwd>::kKb;
  if (!kblock_map(&p.a, A, H, a_rows, kTcBM, false, kb)) return cudaErrorInvalidValue;
  // outputs: dG | dU [a_rows, 2I] and alpha h [a_rows, I], 32 x 32 store boxes
  if (!make_map_16(&p.out, ub.dgu, 2 * static_cast<uint64_t>(I), a_rows, 32, false, 32,
                   CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map_16(&p.out2, ub.ha, I, a_rows, 32, false, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  for (int e = 0; e < g.n_weights; ++e) {
    if (!kblock_map(&p.b0[e], Wg[e], H, I, kN / 2, false, kb)) return cudaErrorInvalidValue;
    if (!kblock_map(&p.b1[e], Wu[e], H, I, kN / 2, false, kb)) return cudaErrorInvalidValue;
  }
  auto fn = grouped_gemm_kernel<kOpUpBwd, MAXW>;
  cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), kSmemOf<kOpUpBwd>);
  if (err != cudaSuccess) return err;
  const int n_tiles = (I + kN / 2 - 1) / (kN / 2);
  DownEpilogue none{};
  WdConvert no_cv{};
  return launch_pdl(fn, 2 * clusters_for(a_rows, g, n_tiles), kSmemOf<kOpUpBwd>, st, p, g, H, I,
                    static_cast<__half*>(nullptr), none, no_cv, hdr, 1, ub, RowGather{});
}

cudaError_t launch_gateup_bwd_tc(const void* A, int64_t a_rows, int H, int I, const GroupRows& g,
                                 const void* const* Wg, const void* const* Wu, const UpBwd& ub,
                                 WsHeader* hdr, cudaStream_t st) {
  if (I % 64 != 0) return cudaErrorInvalidValue;
  if (g.n_weights <= 8) return gateup_bwd_impl<8>(A, a_rows, H, I, g, Wg, Wu, ub, hdr, st);
  return gateup_bwd_impl<MM_MAX_EXPERTS>(A, a_rows, H, I, g, Wg, Wu, ub, hdr, st);
}

template <int MAXW>
static cudaError_t down_impl(const void* h, int64_t a_rows, int H, int I, const GroupRows& g,
                             const void* const* Wd, const DownEpilogue& ep, WsHeader* hdr,
                             cudaStream_t st) {
  // 384-wide tiles where they put every tile pair in one wave and 256-wide
  // ones do not (e.g. 8192 top-1 rows over 4 experts at H = 768: ~100 tile
  // pairs in two waves against ~70 in one)
  const int pairs = num_sms() / 2;
  const bool wide = tiles_bound(a_rows, g, (H + kNWide - 1) / kNWide) <= pairs &&
                    tiles_bound(a_rows, g, (H + kN - 1) / kN) > pairs;
  const int nw = wide ? kNWide : kN;
  TcParams<MAXW> p;
  memset(&p, 0, sizeof(p));
  constexpr int kb = OpTraits<kOpDown>::kKb;
  if (!kblock_map(&p.a, h, I, a_rows, kTcBM, true, kb)) return cudaErrorInvalidValue;
  for (int e = 0; e < g.n_weights; ++e)
    if (!kblock_map(&p.b0[e], Wd[e], I, H, wide ? kNWide / 4 : kN / 2, true, kb))
      return cudaErrorInvalidValue;
  // dense FFN: y is written with tensor stores (32 x 32 boxes, 64-byte swizzle)
  if (ep.perm == nullptr && ep.mode == kCombineStore &&
      !make_map_16(&p.out, ep.y, H, a_rows, 32, false, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  auto fn = wide ? grouped_gemm_kernel<kOpDown, MAXW, kNWide> : grouped_gemm_kernel<kOpDown, MAXW>;
  const size_t smem = wide ? kSmemWide : kSmem;
  cudaError_t err = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), smem);
  if (err != cudaSuccess) return err;
  const int n_tiles = (H + nw - 1) / nw;
  // a later slot's operands (h, fp16 Wd) were complete before the previous
  // slot's launch let it start: only its epilogue waits (for the fp32 sum)
  const int dep = (ep.mode == kCombineAccum || ep.mode == kCombineLast) ? 0 : 1;
  WdConvert no_cv{};
  return launch_pdl(fn, 2 * clusters_for(a_rows, g, n_tiles), smem, st, p, g, I, H,
                    static_cast<__half*>(nullptr), ep, no_cv, hdr, dep, UpBwd{}, RowGather{});
}

cudaError_t launch_gateup_tc(const void* A, int64_t a_rows, int H, int I, const GroupRows& g,
                             const void* const* Wg, const void* const* Wu, void* h_out,
                             const void* const* wd_src, int n_wd, void* wd16, WsHeader* hdr,
                             cudaStream_t st, const RowGather* gather) {
  const RowGather gat = gather ? *gather : RowGather{};
  // gathering: A is x [T, H] with T = a_rows / k rows
  const int64_t x_rows = gather ? a_rows / gather->k : a_rows;
  WdConvert cv{};
  if (n_wd > 0) {
    if (n_wd > MM_MAX_EXPERTS || (static_cast<int64_t>(H) * I) % 8 != 0 || wd16 == nullptr)
      return cudaErrorInvalidValue;
    for (int m = 0; m < n_wd; ++m) cv.src.p[m] = wd_src[m];
    cv.dst = static_cast<__half*>(wd16);
    cv.nvec = static_cast<int64_t>(H) * I / 8;
    cv.n_mat = n_wd;
  }
  if (g.n_weights <= 8) return gateup_impl<8>(A, a_rows, H, I, g, Wg, Wu, h_out, cv, hdr, st, gat, x_rows);
  return gateup_impl<MM_MAX_EXPERTS>(A, a_rows, H, I, g, Wg, Wu, h_out, cv, hdr, st, gat, x_rows);
}

cudaError_t launch_down_tc(const void* h, int64_t a_rows, int H, int I, const GroupRows& g,
                           const void* const* Wd, const DownEpilogue& ep, WsHeader* hdr,
                           cudaStream_t st) {
  if (g.n_weights <= 8) return down_impl<8>(h, a_rows, H, I, g, Wd, ep, hdr, st);
  return down_impl<MM_MAX_EXPERTS>(h, a_rows, H, I, g, Wd, ep, hdr, st);
}

}  // namespace mm
