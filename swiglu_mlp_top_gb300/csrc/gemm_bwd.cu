// Tensor-core GEMMs of the backward pass: C = A B^T over bf16 operands with
// fp32 accumulation, where an operand may be stored MN-major (its M or N
// index contiguous in memory), as the backward's contractions need:
//   dh  = dy Wd          B = Wd [H, I] read with N = I contiguous
//   dx  = dG Wg + dU Wu  B = Wg, Wu [I, H] read with N = H contiguous
//   dWd = dy^T (alpha h), dWg = dG^T x, dWu = dU^T x
//                        A and B both MN-major, K = the tokens (rows)
// (MiniMind lesson 13 "FFN 与 MoE" §0 / §1.2 equations, differentiated; the
// router part lives in backward.cu.)
//
// Same machinery as the forward GEMM (gemm_tc.cu): CTA pairs running
// tcgen05.mma.cta_group::2 with M = 256 (128 rows of A per CTA) and N = 256
// (each CTA stages half of B), operands brought by TMA into a 6-stage ring
// of 128-byte-swizzled tiles, two 256-column TMEM accumulators so that the
// epilogue of one tile overlaps the MMAs of the next, warp roles: 8 epilogue
// warps, 1 TMA producer, 1 MMA issuer (even CTA).
//
// An MN-major tile of 128 (M or N) x 64 (K) is one 3-D TMA box of the
// matrix viewed as (64 columns, rows, column blocks of 64): box 64 x 64 x 2,
// landing as two 8 KiB halves, each 64 K-rows of 128 bytes in 1024-byte
// swizzle atoms of 8 rows (one 16 KiB request; two 8 KiB requests per tile
// left the GEMM waiting on the TMA).
// Its UMMA descriptor: leading byte offset = 8192 (the next 64 elements
// along M / N, i.e. the second box), stride byte offset = 1024 (the next 8
// K-rows); one MMA of K = 16 starts 16 K-rows (2048 bytes) further.
//
// Schedules:
//   kSchedRows  tiles over (group, 256-row block of the group's rows, N
//               block): the dgrad GEMMs, A [rows, K] K-major, one weight
//               matrix per group (two for dx: Wg for the first half of K,
//               Wu for the second); output rows = A rows, in fp32, bf16 or
//               fp16 (dh and the per-assignment dx rows; range-checked).
//   kSchedKGrp  tiles over (problem, M block, N block); a problem is one
//               weight gradient, whose K runs over the rows of its group
//               [koff[g], koff[g+1]) (64-row aligned, padding rows zero);
//               problems in descending K, tiles dealt in snake rounds.
#include <cstring>

#include "mm_kernels.cuh"

namespace mm {

constexpr int kBwStages = 6;
constexpr int kBwTile = 128 * 64 * 2;                 // 16 KiB: 128 rows x one 64-wide k-block
constexpr int kBwEpiWarps = 8;
constexpr int kBwThreads = 32 * (kBwEpiWarps + 2);
constexpr int kBwWarpProducer = kBwEpiWarps, kBwWarpMma = kBwEpiWarps + 1;
// Epilogue staging: one 32-row x 32-column piece per warp (4 KiB of fp32).
constexpr int kBwStage = 32 * 128;
// + 1024 bytes of alignment slack and 256 of barriers
constexpr int kBwSmem = kBwStages * 2 * kBwTile + kBwEpiWarps * kBwStage + 1024 + 256;
// with the static arrays (s_off, s_tstart, s_tmem, s_abort) within the 227 KiB of a block
static_assert(kBwSmem + 8 * (kBwMaxGroups + 1) + kBwMaxGroups + 16 <= 232448, "shared memory budget");

// UMMA descriptor of an MN-major 128 x 64 tile stored as two 64 x 64
// 128-byte-swizzled TMA boxes (see the file comment).
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
  d |= static_cast<uint64_t>(8192u >> 4) << 16;            // leading byte offset: next 64 along M/N
  d |= static_cast<uint64_t>(1024u >> 4) << 32;            // stride byte offset: next 8 K-rows
  d |= static_cast<uint64_t>(1u) << 46;                    // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                    // 128-byte swizzle
  return d;
}

struct BwTile {
  int p, g, row0, rows, m0, n0, kb0, nkb;   // problem / group, rows or M block, N block, K range
};

__device__ __forceinline__ int find_last_le(const int* starts, int n, int t) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (starts[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int SCHED>
// Tile t: rows schedule in group order; K-grouped in the order s_pord gives
// the problems (descending K), s_tstart holding the first tile of each in
// that order.
__device__ __forceinline__ BwTile bw_decode(int t, const BwParams& P, const int* s_off,
                                            const int* s_tstart, const uint8_t* s_pord,
                                            int n_tiles_n, int rank) {
  BwTile ti;
  if constexpr (SCHED == kSchedRows) {
    const int g = find_last_le(s_tstart, P.G, t);
    const int local = t - s_tstart[g];
    const int mb = local / n_tiles_n, nb = local - mb * n_tiles_n;
    ti.p = g;
    ti.g = g;
    ti.row0 = s_off[g] + mb * 256 + rank * 128;
    ti.rows = min(128, s_off[g + 1] - ti.row0);
    ti.m0 = 0;
    ti.n0 = nb * 256;
    ti.kb0 = 0;
    ti.nkb = P.K / 64;
  } else {
    const int i = find_last_le(s_tstart, P.G, t);
    const int p = s_pord[i];
    const BwProblem& pr = P.prob[p];
    const int ntn = (pr.N + 255) / 256;
    const int local = t - s_tstart[i];
    const int mb = local / ntn, nb = local - mb * ntn;
    ti.p = p;
    ti.g = pr.grp;
    ti.m0 = mb * 256 + rank * 128;
    ti.rows = min(128, pr.M - ti.m0);
    ti.row0 = ti.m0;
    ti.n0 = nb * 256;
    const int k0 = s_off[pr.grp], k1 = s_off[pr.grp + 1];
    ti.kb0 = k0 / 64;
    ti.nkb = (k1 - k0 + 63) / 64;
  }
  return ti;
}

// The j-th tile of CTA pair c of nc.  Rows schedule: a plain stride (its
// tiles cost the same).  K-grouped: a tile costs its problem's K, which
// follows the experts' loads (a skewed top-2 call has one expert with ~8x
// the rows of another), so the tiles, problems in descending K, go out in
// rounds of nc, alternately forwards and backwards: the pairs that took a
// round's longest tiles take the next round's shortest.  (Modelled on the
// top-2 skewed call's counts, the busiest pair's k-blocks drop from 785 to
// 710, against a mean of 611.)
template <int SCHED>
__device__ __forceinline__ int bw_tile_index(int j, int c, int nc) {
  if constexpr (SCHED == kSchedKGrp) return j * nc + ((j & 1) ? nc - 1 - c : c);
  return j * nc + c;
}

template <int SCHED>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kBwThreads, 1)
bw_gemm_kernel(const __grid_constant__ BwParams P, WsHeader* hdr) {
  extern __shared__ unsigned char smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kBwStages * kBwTile;
  uint8_t* sEpi = sB + kBwStages * kBwTile;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + kBwEpiWarps * kBwStage);
  uint64_t* full = bars;                   // [kBwStages] even CTA: both CTAs' bytes
  uint64_t* empty = bars + kBwStages;      // [kBwStages] each CTA: released by the pair's MMAs
  uint64_t* tfull = bars + 2 * kBwStages;  // [2] each CTA: accumulator ready
  uint64_t* tempty = tfull + 2;            // [2] even CTA: both CTAs' epilogues done
  uint64_t* drained = tempty + 2;          // even CTA: all MMAs finished
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_off[kBwMaxGroups + 1], s_tstart[kBwMaxGroups + 1];
  __shared__ uint8_t s_pord[kBwMaxGroups];        // K-grouped: problems by descending K

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
  const int n_tiles_n = (P.N + 255) / 256;      // kSchedRows only

  if (threadIdx.x == 0) {
    for (int s = 0; s < kBwStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * kBwEpiWarps);
    }
    mbar_init(drained, 1);
    fence_mbar_init();
    s_abort = 0;
    // a programmatic dependent: the offsets and operands are the previous
    // kernel's output (every role reads them only after the cluster barrier
    // below, which follows this wait)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // group rows (rows schedule) or K ranges (K-grouped), from the device
    // offsets, or one dense range [0, dense_rows)
    const int ngrp = SCHED == kSchedRows ? P.G : P.n_groups;
    for (int g = 0; g <= ngrp; ++g)
      s_off[g] = P.offsets ? P.offsets[g] : (g == 0 ? 0 : P.dense_rows);
    int run = 0;
    for (int q = 0; q < P.G; ++q) {
      s_tstart[q] = run;
      if constexpr (SCHED == kSchedRows) {
        run += ((s_off[q + 1] - s_off[q] + 255) / 256) * n_tiles_n;
      } else {
        run += ((P.prob[q].M + 255) / 256) * ((P.prob[q].N + 255) / 256);
      }
    }
    s_tstart[P.G] = run;
  }
  if (warp == kBwWarpMma) {
    tmem_alloc_cta2(&s_tmem, 512);
    tmem_relinquish_cta2();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if constexpr (SCHED == kSchedKGrp) {
    // problems in descending K (ties in index order), each thread placing
    // one problem by counting those before it; then their first tiles
    const int q = threadIdx.x;
    if (q < P.G) {
      const int gq = P.prob[q].grp;
      const int kq = (s_off[gq + 1] - s_off[gq] + 63) / 64;
      int pos = 0;
      for (int o = 0; o < P.G; ++o) {
        const int go = P.prob[o].grp;
        const int ko = (s_off[go + 1] - s_off[go] + 63) / 64;
        pos += (ko > kq || (ko == kq && o < q)) ? 1 : 0;
      }
      s_pord[pos] = static_cast<uint8_t>(q);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int run = 0;
      for (int i = 0; i < P.G; ++i) {
        const BwProblem& pr = P.prob[s_pord[i]];
        s_tstart[i] = run;
        run += ((pr.M + 255) / 256) * ((pr.N + 255) / 256);
      }
      s_tstart[P.G] = run;
    }
    __syncthreads();
  }
  const uint32_t tmem = s_tmem;
  const int total = s_tstart[P.G];
  volatile int* abort = &s_abort;

  if (warp == kBwWarpProducer) {
    // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int j = 0; ok && j * n_clusters < total; ++j) {
        const int tile = bw_tile_index<SCHED>(j, cluster, n_clusters);
        if (tile >= total) continue;               // the last round's missing tiles
        const BwTile ti = bw_decode<SCHED>(tile, P, s_off, s_tstart, s_pord, n_tiles_n,
                                           static_cast<int>(rank));
        for (int kb = 0; kb < ti.nkb; ++kb, ++it) {
          const int s = it % kBwStages;
          const uint32_t ph = (it / kBwStages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort, hdr, 81)) { ok = false; break; }
          const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 4 * kBwTile);
          uint8_t* a_dst = sA + s * kBwTile;
          uint8_t* b_dst = sB + s * kBwTile;
          // this CTA's half of N: columns n0 + 128 rank ..
          const int ncol = ti.n0 + 128 * static_cast<int>(rank);
          if constexpr (SCHED == kSchedRows) {
            // A: K-major rows of this CTA; B: MN-major, the low or high weight matrix
            tma_load_2d_cta2(a_dst, &P.a[0], fb, kb * 64, ti.row0);
            const bool hi = kb >= P.kb_split;
            const CUtensorMap* bm = hi ? &P.b_hi[ti.g] : &P.b_lo[ti.g];
            const int kk = (hi ? kb - P.kb_split : kb) * 64;
            tma_load_3d_cta2(b_dst, bm, fb, 0, kk, ncol / 64);
          } else {
            // A and B both MN-major: K rows kb0 + kb of the group
            const BwProblem& pr = P.prob[ti.p];
            const int krow = (ti.kb0 + kb) * 64;
            const int mcol = pr.a_col0 + ti.m0;
            tma_load_3d_cta2(a_dst, &P.a[pr.a_map], fb, 0, krow, mcol / 64);
            tma_load_3d_cta2(b_dst, &P.b_lo[pr.b_map], fb, 0, krow, ncol / 64);
          }
        }
      }
      if (!ok && rank == 0) {
        for (int j = 0; j < kBwStages; ++j) {
          const int i2 = it - 1 - j;
          if (i2 < 0) break;
          mbar_wait(&full[i2 % kBwStages], (i2 / kBwStages) & 1, nullptr, hdr, 82);
        }
      }
    }
    __syncwarp();
  } else if (warp == kBwWarpMma) {
    // ------------------------------------------------ MMA issuer (even CTA)
    if (rank == 0 && lane == 0) {
      constexpr uint32_t kAMn = SCHED == kSchedKGrp ? 1u : 0u;
      constexpr uint32_t idesc = idesc_bf16_f32(256, 256) | (kAMn << 15) | (1u << 16);
      int it = 0, used = 0;
      bool ok = true;
      for (int j = 0; ok && j * n_clusters < total; ++j) {
        const int tile = bw_tile_index<SCHED>(j, cluster, n_clusters);
        if (tile >= total) continue;
        const BwTile ti = bw_decode<SCHED>(tile, P, s_off, s_tstart, s_pord, n_tiles_n, 0);
        if (ti.nkb == 0) continue;                 // the epilogue writes zeros for it
        const int acc = used & 1;
        const uint32_t aph = (used >> 1) & 1;
        ++used;
        if (!mbar_wait(&tempty[acc], aph ^ 1, abort, hdr, 83)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + acc * 256;
        for (int kb = 0; kb < ti.nkb; ++kb, ++it) {
          const int s = it % kBwStages;
          const uint32_t ph = (it / kBwStages) & 1;
          if (!mbar_wait(&full[s], ph, abort, hdr, 84)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + s * kBwTile);
          const uint32_t b0 = smem_u32(sB + s * kBwTile);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = kAMn ? smem_desc_sw128_mn(a0 + kk * 2048) : smem_desc_sw128(a0 + kk * 32);
            umma_f16_cta2(d, ad, smem_desc_sw128_mn(b0 + kk * 2048), idesc, (kb | kk) ? 1u : 0u);
          }
          umma_commit_cta2_mc(&empty[s], 0x3);
        }
        if (!ok) break;
        umma_commit_cta2_mc(&tfull[acc], 0x3);
      }
      umma_commit_cta2_mc(drained, 0x1);
      mbar_wait(drained, 0, nullptr, hdr, 85);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ epilogue (warps 0-7, both CTAs)
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;
    uint8_t* wstage = sEpi + warp * kBwStage;     // this warp's staging piece
    const uint32_t te0 = mapa_shared(smem_u32(&tempty[0]), 0);
    const uint32_t te1 = mapa_shared(smem_u32(&tempty[1]), 0);
    int used = 0;
    uint32_t hmax = 0u;     // fp16 output: max |value| of the lane's rows, as packed halves
    for (int j = 0; j * n_clusters < total; ++j) {
      const int tile = bw_tile_index<SCHED>(j, cluster, n_clusters);
      if (tile >= total) continue;
      const BwTile ti = bw_decode<SCHED>(tile, P, s_off, s_tstart, s_pord, n_tiles_n,
                                         static_cast<int>(rank));
      // output row / columns / leading dimension of this tile
      float* out32 = nullptr;
      uint16_t* out16 = nullptr;                 // bf16 or fp16 (P.out_type)
      int64_t ldo;
      int ncols;
      if constexpr (SCHED == kSchedRows) {
        ldo = P.ldo;
        ncols = P.N;
        if (P.out_type != kBwOutF32) out16 = static_cast<uint16_t*>(P.out); else out32 = static_cast<float*>(P.out);
      } else {
        ldo = P.prob[ti.p].N;
        ncols = P.prob[ti.p].N;
        out32 = P.prob[ti.p].out;
      }
      const bool valid = row < ti.rows;
      // rows schedule: all 32 rows of the warp in the group, so its pieces
      // go out as tensor stores (the rows past a group are the next group's)
      const bool tma_piece = SCHED == kSchedRows && P.out_tma && (row | 31) < ti.rows;
      const int64_t orow = static_cast<int64_t>(ti.row0 + row);
      if (ti.nkb == 0) {
        // empty K range (an expert no token chose): the gradient is zero
        if (valid && out32 != nullptr)
          for (int c = half * 128; c < half * 128 + 128; c += 4)
            if (ti.n0 + c < ncols)
              *reinterpret_cast<float4*>(out32 + orow * ldo + ti.n0 + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        continue;
      }
      const int acc = used & 1;
      const uint32_t aph = (used >> 1) & 1;
      ++used;
      if (!warp_wait(&tfull[acc], aph, abort, hdr, 86)) break;
      tc_fence_after();
      const uint32_t tb = tmem + (static_cast<uint32_t>(quad * 32) << 16) + acc * 256 + half * 128;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const int col = ti.n0 + half * 128 + c * 32;
        uint32_t r[32];
        tmem_ld_32x32b_x32(tb + c * 32, r);     // every lane (warp-collective)
        tmem_ld_wait();
        if (col >= ncols) continue;              // warp-uniform
        // 16-bit output: the row's 32 values as 16 packed pairs
        uint32_t pk[16];
        if (out16 != nullptr) {
          if (P.out_type == kBwOutF16) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              pk[j] = pack_f16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
              if (valid) hmax = hmax2_nan_abs(hmax, pk[j]);   // rows past the group do not count
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              pk[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
          }
        }
        if (tma_piece) {
          // through the swizzled staging piece: fp32 in 128-byte rows (chunk q
          // of row r at q ^ (r & 7)), 16-bit in 64-byte rows (q ^ ((r >> 1) & 3))
          if (lane == 0) bulk_wait_read();       // the previous piece's store has read it
          __syncwarp();
          if (out16 != nullptr) {
            uint8_t* r64 = wstage + lane * 64;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4*>(r64 + ((q ^ ((lane >> 1) & 3)) << 4)) =
                  make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          } else {
            uint8_t* r128 = wstage + lane * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<uint4*>(r128 + ((q ^ (lane & 7)) << 4)) =
                  make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&P.o, wstage, col, ti.row0 + (row & ~31));
            bulk_commit();
          }
        } else if (!valid) {
          // rows past the group / matrix: nothing to store
        } else if (out16 != nullptr) {
          uint4* d4 = reinterpret_cast<uint4*>(out16 + orow * ldo + col);
#pragma unroll
          for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        } else {
          float4* d4 = reinterpret_cast<float4*>(out32 + orow * ldo + col);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            d4[q] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc ? te1 : te0);
    }
    if constexpr (SCHED == kSchedRows)
      if (P.out_type == kBwOutF16) report_range(hdr, f16x2_out_of_range(hmax), 101);
    bulk_wait_all();   // this warp's tensor stores have landed
  }

  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == kBwWarpMma) tmem_dealloc_cta2(tmem, 512);
}

// =============================================================== host side
// MN-major tiles of a bf16 row-major [rows, cols] matrix (cols a multiple of
// 64): the matrix as (64 columns, rows, cols / 64 column blocks), box 64 x 64
// x 2 (two column blocks of 64 K-rows), 128-byte swizzle; zero fill past
// the matrix.
static bool box64(CUtensorMap* m, const void* ptr, int64_t cols, int64_t rows) {
  const uint64_t dims[3] = {64, static_cast<uint64_t>(rows), static_cast<uint64_t>(cols / 64)};
  const uint64_t strides[2] = {static_cast<uint64_t>(cols) * 2, 128};
  const uint32_t box[3] = {64, 64, 2};
  return make_map_3d(m, ptr, dims, strides, box);
}

static int bw_clusters(int64_t tiles) {
  const int pairs = num_sms() / 2;
  return static_cast<int>(tiles < pairs ? (tiles > 0 ? tiles : 1) : pairs);
}

template <int SCHED>
static cudaError_t bw_launch(const BwParams& p, int64_t tiles_bound, WsHeader* hdr, cudaStream_t st) {
  auto fn = bw_gemm_kernel<SCHED>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), kBwSmem);
  if (e != cudaSuccess) return e;
  return launch_dependent_kernel(fn, dim3(2 * bw_clusters(tiles_bound)), dim3(kBwThreads), kBwSmem,
                                 st, p, hdr);
}

cudaError_t launch_bw_dgrad(const void* A, int64_t a_rows, int K, const int32_t* offsets, int G,
                            int dense_rows, const void* const* b_lo, const void* const* b_hi,
                            int kb_split, int N, void* out, int64_t ldo, int out_type,
                            WsHeader* hdr, cudaStream_t st) {
  if (G < 1 || G > kBwMaxGroups || K % 64 != 0 || N % 64 != 0) return cudaErrorInvalidValue;
  BwParams p;
  memset(&p, 0, sizeof(p));
  // A [a_rows, K] K-major: box 64 (K) x 128 rows
  if (!make_map_16(&p.a[0], A, static_cast<uint64_t>(K), static_cast<uint64_t>(a_rows), 128, false,
                   64, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // B (per group) [K rows, N cols] MN-major; b_hi covers the k-blocks from kb_split on
  const int klo = kb_split * 64, khi = K - klo;
  for (int g = 0; g < G; ++g) {
    if (!box64(&p.b_lo[g], b_lo[g], N, klo)) return cudaErrorInvalidValue;
    if (khi > 0 && !box64(&p.b_hi[g], b_hi[g], N, khi)) return cudaErrorInvalidValue;
  }
  p.offsets = offsets;
  p.G = G;
  p.dense_rows = dense_rows;
  p.K = K;
  p.N = N;
  p.kb_split = khi > 0 ? kb_split : K / 64;
  p.out = out;
  p.ldo = ldo;
  p.out_type = out_type;
  // full 32-row pieces as TMA stores, where the output's address and pitch allow
  const int esz = out_type == kBwOutF32 ? 4 : 2;
  const bool aligned = reinterpret_cast<uintptr_t>(out) % 16 == 0 && (ldo * esz) % 16 == 0;
  if (out_type == kBwOutF16)
    p.out_tma = (aligned && ldo == N &&
                 make_map_16(&p.o, out, static_cast<uint64_t>(N), static_cast<uint64_t>(a_rows), 32,
                             true, 32, CU_TENSOR_MAP_SWIZZLE_64B)) ? 1 : 0;
  else
    p.out_tma = (aligned &&
                 make_map_2d(&p.o, out, out_type == kBwOutF32, static_cast<uint64_t>(N),
                             static_cast<uint64_t>(a_rows), static_cast<uint64_t>(ldo) * esz, 32, 32,
                             out_type == kBwOutF32 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                   : CU_TENSOR_MAP_SWIZZLE_64B)) ? 1 : 0;
  const int64_t ntn = (N + 255) / 256;
  const int64_t tiles = offsets ? ((a_rows + 255) / 256 + G) * ntn : ((dense_rows + 255) / 256) * ntn;
  return bw_launch<kSchedRows>(p, tiles, hdr, st);
}

cudaError_t launch_bw_wgrad(const void* const* a_mats, const int64_t* a_cols, int n_a,
                            const void* const* b_mats, const int64_t* b_cols, int n_b,
                            int64_t k_rows, const BwProblem* probs, int n_probs,
                            const int32_t* offsets, int n_groups, int dense_rows, WsHeader* hdr,
                            cudaStream_t st) {
  if (n_probs < 1 || n_probs > kBwMaxGroups || n_a > kBwMaxMaps || n_b > kBwMaxMaps)
    return cudaErrorInvalidValue;
  BwParams p;
  memset(&p, 0, sizeof(p));
  for (int i = 0; i < n_a; ++i)
    if (!box64(&p.a[i], a_mats[i], a_cols[i], k_rows)) return cudaErrorInvalidValue;
  for (int i = 0; i < n_b; ++i)
    if (!box64(&p.b_lo[i], b_mats[i], b_cols[i], k_rows)) return cudaErrorInvalidValue;
  int64_t tiles = 0;
  for (int q = 0; q < n_probs; ++q) {
    if (probs[q].M % 64 != 0 || probs[q].N % 64 != 0) return cudaErrorInvalidValue;
    p.prob[q] = probs[q];
    tiles += static_cast<int64_t>((probs[q].M + 255) / 256) * ((probs[q].N + 255) / 256);
  }
  p.G = n_probs;
  p.n_groups = n_groups;
  p.offsets = offsets;
  p.dense_rows = dense_rows;
  return bw_launch<kSchedKGrp>(p, tiles, hdr, st);
}

}  // namespace mm
