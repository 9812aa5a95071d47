// Decode-sized forward on the 5th-generation tensor cores (T <= 64 tokens,
// bf16): one cooperative kernel that streams every needed weight row once.
// The weights are the UMMA M operand (tiles of 128 rows x 64 k, TMA-fed,
// 128-byte swizzle); the T tokens, padded to Np = 16·ceil(T/16) with zero
// rows, are the N operand; fp32 accumulators live in TMEM.
//
//   1  x (all Np rows) -> shared memory once.  MoE: router logits
//      L = x Wr^T on the tensor core (x rows as M, experts as N); then
//      softmax / top-k / alpha per token and the grouping by expert
//      (route_small.cuh; lesson 13 §1.5, chapter 4 §4.3).  Block 0 writes
//      topk_idx, topk_w and the aux loss (lesson 13 §1.6).
//   2  gate/up units (touched expert e, 128 rows of I, k-range):
//      G = Wg_e x^T, U = Wu_e x^T.  With one k-range per unit the epilogue
//      forms h = SiLU(G) ⊙ U (lesson 13 §0/§1.2) directly; otherwise it
//      writes fp32 partial G, U and, after a grid barrier, every CTA reduces
//      a share of them in k-range order.  Either way the result is stored as
//      Hp_e[t, i] = alpha_{t,e} h_{t,e}[i] (0 for tokens not routed to e), split
//      into a bf16 high part and a bf16 remainder: the down product then runs
//      on bf16 operands with ~16 significant bits of h.
//   3  grid barrier; down: y^T = sum_e Wd_e Hp_e^T.  The (output m-block,
//      expert, k-block) tiles are cut into one contiguous range per CTA; each
//      CTA accumulates its range in TMEM and writes one fp32 partial per
//      output m-block it touches.  The Wd tiles of a CTA's first tiles are
//      requested before the barrier, since they do not depend on h.
//   4  grid barrier; every CTA adds a share of the partials in CTA order and
//      rounds y to bf16 once (deterministic; the weighted sum over the
//      selected experts is part of the fp32 accumulation).
//
// Fused variant (many (expert, I-block) units, y^T for all H rows fits in
// TMEM beside the gate/up accumulators): each unit also streams its 128
// columns of Wd_e and multiplies them by its own h, kept in shared memory as
// the B operand; a CTA's units accumulate y^T in TMEM, the CTA writes one
// fp32 partial of y, and after a single grid barrier the partials are added in
// CTA order.  h never reaches global memory.  MoE calls stream speculatively:
// every expert's units start at once, the router runs on stages the ring
// then skips and the epilogue warps route meanwhile; once the routing is
// published, units of experts no token selected stop (the producer records
// how many of their stages it issued, the MMA issuer releases exactly those).
//
// Warp roles (320 threads): warp 0 lane 0 issues TMA, warp 1 lane 0 issues
// UMMA and owns TMEM, warps 2-9 are the epilogue (TMEM lane quadrant
// warp % 4, token-column half (warp - 2) / 4).  All waits are bounded.
#include <algorithm>
#include <mutex>

#include "route_small.cuh"

namespace mm {

constexpr int kDtThreads = 320;
constexpr int kDtEpiWarps = 8;
constexpr int kDtMaxStages = 4;
constexpr int kDtTileA = 128 * 64 * 2;          // 16 KiB: 128 weight rows x 64 k
constexpr uint32_t kDtTmemCols = 512;
constexpr uint32_t kDtColGU = 0;                // two (G, U) buffers, 2 * Np columns each
constexpr uint32_t kDtColD = 256;               // down accumulator
constexpr uint32_t kDtColL = 384;               // router logits (speculative: the last Epad columns)
constexpr int kDtMaxSeg = 2;                    // output m-blocks per CTA range
constexpr int kDtMaxCtas = 160;                 // grid cap (152 SMs on GB300)
constexpr int kDtMaxMB = 64;                    // output m-blocks (H <= 8192)
constexpr int kDtMaxSplit = 4;                  // k-ranges per gate/up block at most
constexpr int kDtReduceChunk = 32;              // partials requested at once in the final sum
constexpr size_t kDtSmemBudget = 196 * 1024;   // dynamic; static use is ~27 KiB
constexpr int kDtFusedMinUnits = 64;            // fused variant: (expert, I-block) units at least
constexpr int kDtMaxLocalUnits = 64;            // speculative: units per CTA at most (cut table)
constexpr int kDtMaxSlices = 16;                // fused: partial sums per output quad at most
constexpr int kDtSumChunk = 16;                 // fused: partials requested at once

template <int MAXW>
struct DtMaps {
  CUtensorMap x;                  // x [T, H], box 64 x Np (rows >= T read as 0)
  CUtensorMap wr;                 // Wr [E, H], box 64 x Epad
  CUtensorMap hp;                 // Hp [nt_max * 2 * Np, I], box 64 x Np (loads, 128-byte swizzle)
  CUtensorMap hps;                // the same matrix, box 128 x Np, no swizzle (stores)
  CUtensorMap wg[MAXW], wu[MAXW]; // [I, H], box 64 x 128
  CUtensorMap wd[MAXW];           // [H, I], box 64 x 128
};

struct DtArgs {
  int T, Np, H, I, E, k;          // E = k = 1 for the dense FFN
  int moe;
  float coef;
  const float* bias;
  int32_t* topk_idx;
  float* topk_w;
  float* aux_loss;
  __nv_bfloat16* hp;              // [nt_max][2][Np][I]
  float* pgu;                     // [units][2][Np][128]   (split gate/up only)
  float* pd;                      // [grid][kDtMaxSeg][Np][128]
  void* y;                        // [T, H] bf16
  WsHeader* hdr;
  int stages;
  int gu_bufs;                    // fused: (G, U) TMEM buffers (1 or 2)
  int spec;                       // fused MoE: every expert streamed from the start, routed meanwhile
  int router_stages;              // ring stages the router's x and Wr tiles cover
  int Epad;                       // experts padded to a multiple of 16 (router N)
  uint32_t stage_bytes;           // 32 KiB of weight tiles + one x tile
  uint32_t hstage_off;            // Hp staging tile [2][Np][128] bf16 (epilogue -> TMA store)
  uint32_t alpha_off;             // alpha table [nt_max][Np] fp32
  RouterVariant rv;               // router noise, z-loss, saved statistics (MoE)
};

// Work plan derived from the routing; identical in every thread of the grid.
struct DtPlan {
  int nt, MB_I, MB_H, KB_H, KB_I;
  int s_up, n_units;              // gate/up: blocks * k-ranges
  int F;                          // down tiles: MB_H * nt * KB_I (F * grid < 2^31)
  int per_mb;                     // down tiles per output m-block
};

__device__ __forceinline__ int dt_range_start(int c, int F, int G) { return c * F / G; }
// CTA whose down range holds tile f (the largest c with start(c) <= f).
__device__ __forceinline__ int dt_cta_of(int f, int F, int G) { return ((f + 1) * G - 1) / F; }

// SiLU(g) * u with the fast exponential and division (for g -> -inf the
// divisor overflows to inf and the quotient is 0).
__device__ __forceinline__ float swiglu_fast(float g, float u) {
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

constexpr int kDtEpiLeader = 64;                // warp 2, lane 0
// Barrier among the eight epilogue warps only (named barrier 1), plain and
// with an AND of one predicate over the 256 threads.
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDtEpiWarps * 32) : "memory");
}
__device__ __forceinline__ bool epi_sync_and(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\t"
      "setp.ne.u32 a, %1, 0;\n\t"
      "bar.red.and.pred b, 1, %2, a;\n\t"
      "selp.u32 %0, 1, 0, b;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(p)), "n"(kDtEpiWarps * 32)
      : "memory");
  return r != 0;
}



// kFused: every unit (expert, 128 rows of I) also runs its share of the
// down product in the same CTA, from h kept in shared memory; each CTA
// writes one fp32 partial of y and the partials are added after one grid
// barrier.  Otherwise h goes through global memory (split-K gate/up, down
// ranges over output m-blocks, two or three grid barriers).
template <int MAXW, bool kFused>
__global__ void __launch_bounds__(kDtThreads, 1)
decode_tc_kernel(const __grid_constant__ DtMaps<MAXW> M, const DtArgs A) {
  extern __shared__ unsigned char smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* ring = smem;                                     // [stages][A.stage_bytes]
  float* alpha = reinterpret_cast<float*>(smem + A.alpha_off);
  __nv_bfloat16* hstage = reinterpret_cast<__nv_bfloat16*>(smem + A.hstage_off);
  __shared__ SmallRoute<kDecodeTcMaxT> R;
  __shared__ __align__(8) uint64_t full[kDtMaxStages], empty[kDtMaxStages];
  __shared__ __align__(8) uint64_t wbar, lbar, tfull[2], tempty[2], dfull, dempty, drained;
  __shared__ __align__(8) uint64_t hfull, hempty;      // fused: h tiles written / read
  // speculative streaming: the routing once known (flag, selected experts)
  // and, per local unit, the stages the producer issued before it dropped
  // the unit of an unselected expert (-1: not dropped)
  __shared__ volatile int s_routed;
  __shared__ volatile unsigned long long s_selected;
  __shared__ volatile int s_cut[kDtMaxLocalUnits];
  __shared__ uint32_t s_tmem;
  __shared__ float s_bias[MM_MAX_EXPERTS];
  __shared__ int s_first_mb[kDtMaxCtas];        // first output m-block of each CTA's range (-1: empty)
  __shared__ int s_c0[kDtMaxMB], s_c1[kDtMaxMB]; // CTAs whose ranges meet output m-block mb

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int T = A.T, Np = A.Np, H = A.H, I = A.I, S = A.stages;
  const uint32_t SB = A.stage_bytes;
  const uint32_t xtile = static_cast<uint32_t>(Np) * 128;  // bytes of one x / Hp tile
  const uint32_t idesc = idesc_bf16_f32(128, Np);
  const bool moe = A.moe != 0;
  WsHeader* hdr = A.hdr;
  // epilogue warps 2..9: TMEM lane quadrant warp % 4, column half (warp - 2) / 4
  const bool epi = warp >= 2;
  const int quad = warp & 3, half = (warp - 2) >> 2;
  const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;

  if (tid == 0) {
    for (int s = 0; s < kDtMaxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&wbar, 1);
    mbar_init(&lbar, 1);
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kDtEpiWarps);
    }
    mbar_init(&dfull, 1);
    mbar_init(&dempty, kDtEpiWarps);
    mbar_init(&drained, 1);
    mbar_init(&hfull, kDtEpiWarps);
    mbar_init(&hempty, 1);
    fence_mbar_init();
    s_routed = 0;
    s_selected = 0ull;
    for (int q = 0; q < kDtMaxLocalUnits; ++q) s_cut[q] = -1;
  }
  if (tid < MM_MAX_EXPERTS) s_bias[tid] = (moe && A.bias != nullptr && tid < A.E) ? A.bias[tid] : 0.f;
  if (warp == 1) {
    tmem_alloc(&s_tmem, kDtTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  // role state: stage uses issued (producer) / consumed (MMA)
  int p_it = 0, m_it = 0;
  bool ok = true;
  auto acquire = [&](int& s) -> bool {      // producer: next ring stage, once it is empty
    s = p_it % S;
    return mbar_wait(&empty[s], ((p_it / S) & 1) ^ 1, nullptr, hdr, 40);
  };
  auto consume = [&](int& s) -> bool {      // MMA: next ring stage, once it is full
    s = m_it % S;
    const bool r = mbar_wait(&full[s], (m_it / S) & 1, nullptr, hdr, 41);
    tc_fence_after();
    return r;
  };
  auto sdesc = [&](const uint8_t* p) { return smem_desc_sw128(smem_u32(p)); };
  const uint64_t pol = l2_evict_first_policy();     // weights: read once per launch

  // ------------------------------------------------------------ 1: router (MoE)
  // L[t, e] = x_t . Wr_e.  All k-blocks are requested at once into the ring
  // region (its stages are first used after the routing): the x tiles
  // (A operand: 128 rows are read from each, rows >= Np are ignored), then
  // the Wr tiles (B operand, N = Epad).
  const int KB_H = H / 64;
  const uint32_t wtile = static_cast<uint32_t>(A.Epad) * 128;
  uint8_t* rx = ring;
  uint8_t* rw = ring + KB_H * xtile;
  // speculative (fused MoE only): the router runs inside the unit phase, its
  // logits in the last Epad TMEM columns.  Those may be y^T's last columns:
  // the first down MMA of the CTA waits for h, which the epilogue writes only
  // after it has read the logits and routed.
  const bool spec = kFused && A.spec != 0;
  const uint32_t colL = spec ? kDtTmemCols - static_cast<uint32_t>(A.Epad) : kDtColL;
  auto router_issue = [&]() {               // thread 0
    mbar_arrive_expect_tx(&wbar, KB_H * (xtile + wtile));
    for (int kb = 0; kb < KB_H; ++kb) {
      tma_load_2d(rx + kb * xtile, &M.x, &wbar, kb * 64, 0);
      tma_load_2d(rw + kb * wtile, &M.wr, &wbar, kb * 64, 0);
    }
  };
  auto router_mma = [&]() -> bool {         // thread 32
    if (!mbar_wait(&wbar, 0, nullptr, hdr, 42)) return false;
    tc_fence_after();
    const uint32_t idesc_r = idesc_bf16_f32(128, A.Epad);
    for (int kb = 0; kb < KB_H; ++kb) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        umma_bf16(tmem + colL, sdesc(rx + kb * xtile + kk * 32), sdesc(rw + kb * wtile + kk * 32),
                  idesc_r, (kb | kk) ? 1u : 0u);
    }
    umma_commit(&lbar);
    return true;
  };
  auto router_read = [&]() -> bool {        // epilogue warps of column half 0 (TMEM lane = token)
    const bool r = warp_wait(&lbar, 0, nullptr, hdr, 43);
    tc_fence_after();
    const int t = quad * 32 + lane;
#pragma unroll 1
    for (int c0 = 0; r && c0 < A.Epad; c0 += 8) {
      uint32_t v[8];
      tmem_ld_32x32b_x8(tmem + lane_base + colL + c0, v);
      tmem_ld_wait();
      if (t < T) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (c0 + j < A.E) R.prob[t][c0 + j] = __uint_as_float(v[j]);
      }
    }
    return r;
  };
  if (moe && !spec) {
    if (tid == 0) router_issue();
    if (tid == 32) ok = router_mma();
    if (epi && half == 0) ok = router_read();
  }
  tc_fence_before();
  ok = __syncthreads_and(ok);
  tc_fence_after();

  // ------------------------------------------------------------ routing
  if (ok && !spec) {
    if (moe) {
      route_softmax_topk_warp(R, T, A.E, A.k, s_bias, warp, kDtThreads / 32, lane, A.rv.noise);
      __syncthreads();
      if (warp == 0) route_group(R, T * A.k, A.E, lane);
    } else {
      route_dense(R, T, tid);
    }
    __syncthreads();
    for (int q = tid; q < R.n_touched * Np; q += kDtThreads) alpha[q] = 0.f;
    __syncthreads();
    for (int a = tid; a < R.nA; a += kDtThreads) {
      const int t = moe ? a / A.k : a;
      alpha[R.slot_of[R.sel_e[a]] * Np + t] = R.sel_a[a];
    }
    if (moe && cta == 0)
      route_outputs(R, T, A.E, A.coef, A.topk_idx, A.topk_w, A.aux_loss, tid, kDtThreads, 2,
                    &A.rv);
    __syncthreads();
  }

  unsigned ticket = 0xffffffffu;
  if constexpr (kFused) {
    // ---------------------------------------------------------- 2+3: units
    // unit u = (touched expert ti, I-block mb): stages of Wg|Wu|x tiles
    // (gate/up, K = H), then stages of two Wd tiles (output m-block mbd,
    // K = the unit's 128 values of I).  h = SiLU(G) * U * alpha goes from
    // TMEM into four shared tiles (bf16 high part and remainder, two k-halves;
    // Np rows x 128 bytes, 128-byte swizzle): the B operand of the down MMAs,
    // which accumulate y^T for all H rows in TMEM across the CTA's units.
    // speculative: every expert is a unit (alpha indexed by expert); the
    // router's tiles take the first A.router_stages ring stages, whose first
    // use is completed by hand (full: a plain arrival; empty: a commit after
    // the router MMAs), so that the ring then runs as if they had been used
    const int nt = spec ? A.E : ((ok && R.n_touched > 0) ? R.n_touched : 1);
    const int MB_I = (I + 127) / 128, MB_H = H / 128;
    const int n_units = nt * MB_I;
    const int nb = A.gu_bufs;
    const uint32_t colD = 2u * static_cast<uint32_t>(Np * nb);
    uint8_t* hs = reinterpret_cast<uint8_t*>(hstage);      // tile (part, k-half) at (2 part + kh) * xtile
    // speculative: expert e's units are dropped once the routing is known
    // and no token selected e
    auto dropped = [&](int e) -> bool {
      if (!s_routed) return false;
      __threadfence_block();
      return ((s_selected >> e) & 1ull) == 0ull;
    };
    auto wait_routed = [&]() -> bool {
      const unsigned long long t0 = globaltimer_ns();
      for (uint32_t n = 0; !s_routed; ++n)
        if ((n & 63u) == 63u && (globaltimer_ns() - t0 > kWaitLimitNs || n > (1u << 30))) {
          report_timeout(hdr, 56);
          return false;
        }
      __threadfence_block();
      return true;
    };
    // MMA: stage q of local unit j, once it is full (1), or 0 when the
    // producer dropped the unit before issuing it; -1 on time-out
    auto take = [&](int j, int q, int& s) -> int {
      s = m_it % S;
      const uint32_t addr = smem_u32(&full[s]), par = (m_it / S) & 1;
      const unsigned long long t0 = globaltimer_ns();
      for (uint32_t n = 0;; ++n) {
        if (mbar_try_wait(addr, par)) {
          tc_fence_after();
          return 1;
        }
        const int c = s_cut[j];
        if (c >= 0 && q >= c) return 0;
        if ((n & 63u) == 63u && (globaltimer_ns() - t0 > kWaitLimitNs || n > (1u << 30))) {
          report_timeout(hdr, 55);
          return -1;
        }
      }
    };
    if (ok) {
      if (tid == 0) {
        if (spec) {
          router_issue();
          for (int q = 0; q < A.router_stages; ++q) mbar_arrive(&full[q]);
          p_it = A.router_stages;
        }
        int j = 0;
        for (int u = cta; ok && u < n_units; u += G, ++j) {
          const int ti = u / MB_I, mb = u - ti * MB_I, e = spec ? ti : R.touched[ti];
          for (int q = 0; q < KB_H + MB_H; ++q) {
            if (spec && dropped(e)) {                 // stop; the MMA consumes what was issued
              s_cut[j] = q;
              break;
            }
            int s;
            if (!acquire(s)) { ok = false; break; }
            uint8_t* st = ring + s * SB;
            if (q < KB_H) {
              mbar_arrive_expect_tx(&full[s], 2 * kDtTileA + xtile);
              tma_load_2d_hint(st, &M.wg[e], &full[s], q * 64, mb * 128, pol);
              tma_load_2d_hint(st + kDtTileA, &M.wu[e], &full[s], q * 64, mb * 128, pol);
              tma_load_2d(st + 2 * kDtTileA, &M.x, &full[s], q * 64, 0);
            } else {
              const int mbd = q - KB_H;
              mbar_arrive_expect_tx(&full[s], 2 * kDtTileA);
              tma_load_2d_hint(st, &M.wd[e], &full[s], mb * 128, mbd * 128, pol);
              tma_load_2d_hint(st + kDtTileA, &M.wd[e], &full[s], mb * 128 + 64, mbd * 128, pol);
            }
            ++p_it;
          }
        }
      }
      if (tid == 32) {
        if (spec) {
          ok = router_mma();
          for (int q = 0; q < A.router_stages; ++q) umma_commit(&empty[q]);
          m_it = A.router_stages;
        }
        // j: local unit; jj: units kept (their (G, U), h and y^T protocol)
        int j = 0, jj = 0;
        for (int u = cta; ok && u < n_units; u += G, ++j) {
          const int ti = u / MB_I, e = spec ? ti : 0;
          const int acc = nb == 2 ? (jj & 1) : 0, use = nb == 2 ? (jj >> 1) : jj;
          if (!mbar_wait(&tempty[acc], (use & 1) ^ 1, nullptr, hdr, 44)) { ok = false; break; }
          tc_fence_after();
          const uint32_t dg = tmem + kDtColGU + acc * 2 * Np, du = dg + Np;
          int q = 0;
          for (; q < KB_H; ++q) {
            int s;
            const int r = take(j, q, s);
            if (r <= 0) { ok = r == 0; break; }
            const uint8_t* st = ring + s * SB;
            const uint8_t* b = st + 2 * kDtTileA;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16(dg, sdesc(st + kk * 32), sdesc(b + kk * 32), idesc, (q || kk) ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16(du, sdesc(st + kDtTileA + kk * 32), sdesc(b + kk * 32), idesc, (q || kk) ? 1u : 0u);
            umma_commit(&empty[s]);
            ++m_it;
          }
          if (!ok) break;
          // keep the unit?  (speculative: once the routing is known)
          if (spec && !wait_routed()) { ok = false; break; }
          if (spec && dropped(e)) {
            // release the unit's remaining issued stages without using them
            for (; q < KB_H + MB_H; ++q) {
              int s;
              const int r = take(j, q, s);
              if (r <= 0) { ok = r == 0; break; }
              umma_commit(&empty[s]);
              ++m_it;
            }
            if (!ok) break;
            continue;
          }
          umma_commit(&tfull[acc]);
          if (!mbar_wait(&hfull, jj & 1, nullptr, hdr, 53)) { ok = false; break; }
          tc_fence_after();
          for (int mbd = 0; mbd < MB_H; ++mbd) {
            int s;
            if (!consume(s)) { ok = false; break; }
            const uint8_t* st = ring + s * SB;
            const uint32_t d = tmem + colD + mbd * Np;
#pragma unroll 1
            for (int h4 = 0; h4 < 4; ++h4) {        // (k-half, part) = (h4 >> 1, h4 & 1)
              const uint8_t* a = st + (h4 >> 1) * kDtTileA;
              const uint8_t* b = hs + (2 * (h4 & 1) + (h4 >> 1)) * xtile;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_bf16(d, sdesc(a + kk * 32), sdesc(b + kk * 32), idesc, (jj || h4 || kk) ? 1u : 0u);
            }
            umma_commit(&empty[s]);
            ++m_it;
          }
          if (!ok) break;
          umma_commit(&hempty);
          ++jj;
        }
        if (ok && jj > 0) umma_commit(&dfull);
      }
      if (epi) {
        const int rl = quad * 32 + lane;
        const int cbeg = half * (Np / 2), cend = cbeg + Np / 2;   // this warp's token columns
        // element (t, rl) of the h tiles: k-half rl / 64, column rl % 64 of
        // row t, 16-byte chunks swizzled by t % 8
        const int col = rl & 63;
        uint8_t* hhi = hs + (rl >> 6) * xtile;
        uint8_t* hlo = hhi + 2 * xtile;
        if (spec) {
          // routing on the epilogue warps (named barrier 1) while the weights stream
          bool r = true;
          if (half == 0) r = router_read();
          ok = epi_sync_and(r);
          if (ok) {
            const int etid = tid - 64, en = kDtEpiWarps * 32;
            route_softmax_topk_warp(R, T, A.E, A.k, s_bias, etid >> 5, en >> 5, lane, A.rv.noise);
            for (int q = etid; q < A.E * Np; q += en) alpha[q] = 0.f;
            epi_sync();
            if (warp == 2) route_group(R, T * A.k, A.E, lane);
            for (int a = etid; a < T * A.k; a += en) alpha[R.sel_e[a] * Np + a / A.k] = R.sel_a[a];
            epi_sync();
            if (etid == 0) {
              // publish the routing to the producer and the MMA issuer
              unsigned long long sel = 0ull;
              for (int e = 0; e < A.E; ++e)
                if (R.slot_of[e] >= 0) sel |= 1ull << e;
              s_selected = sel;
              __threadfence_block();
              s_routed = 1;
            }
            if (cta == 0)
              route_outputs(R, T, A.E, A.coef, A.topk_idx, A.topk_w, A.aux_loss, etid, en, 0, &A.rv);
          }
        }
        int jj = 0;                                   // units kept
        for (int u = cta; ok && u < n_units; u += G) {
          const int ti = u / MB_I;
          if (spec && R.slot_of[ti] < 0) continue;    // unselected expert: dropped
          const int acc = nb == 2 ? (jj & 1) : 0, use = nb == 2 ? (jj >> 1) : jj;
          if (!warp_wait(&tfull[acc], use & 1, nullptr, hdr, 45)) { ok = false; break; }
          if (jj > 0 && !warp_wait(&hempty, (jj - 1) & 1, nullptr, hdr, 54)) { ok = false; break; }
          tc_fence_after();
          const uint32_t tg = tmem + lane_base + kDtColGU + acc * 2 * Np;
#pragma unroll 1
          for (int c0 = cbeg; c0 < cend; c0 += 8) {
            uint32_t gr[8], ur[8];
            tmem_ld_32x32b_x8(tg + c0, gr);
            tmem_ld_32x32b_x8(tg + Np + c0, ur);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const int t = c0 + jj;
              const float v = swiglu_fast(__uint_as_float(gr[jj]), __uint_as_float(ur[jj])) *
                              alpha[ti * Np + t];
              const __nv_bfloat16 hi = __float2bfloat16_rn(v);
              const int off = t * 128 + ((((col >> 3) ^ (t & 7)) << 4) | ((col & 7) << 1));
              *reinterpret_cast<__nv_bfloat16*>(hhi + off) = hi;
              *reinterpret_cast<__nv_bfloat16*>(hlo + off) = __float2bfloat16_rn(v - __bfloat162float(hi));
            }
          }
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&hfull);
            mbar_arrive(&tempty[acc]);
          }
          ++jj;
        }
        // the CTA's partial of y: pd[cta][t][row], tokens t < T only (zeros
        // when every unit of the CTA was dropped)
        if (ok && jj == 0 && cta < n_units) {
          float* pdst = A.pd + static_cast<size_t>(cta) * T * H + rl;
          for (int c0 = cbeg; c0 < cend && c0 < T; ++c0)
            for (int mbd = 0; mbd < MB_H; ++mbd) pdst[static_cast<size_t>(c0) * H + mbd * 128] = 0.f;
        }
        if (ok && jj > 0) {
          if (!warp_wait(&dfull, 0, nullptr, hdr, 49)) {
            ok = false;
          } else {
            tc_fence_after();
            float* pdst = A.pd + static_cast<size_t>(cta) * T * H + rl;
            const int cstop = cend < T ? cend : T;
            // four output m-blocks per TMEM wait
#pragma unroll 1
            for (int c0 = cbeg; c0 < cstop; c0 += 8) {
#pragma unroll 1
              for (int m0 = 0; m0 < MB_H; m0 += 4) {
                uint32_t r[4][8];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  if (m0 + q < MB_H) tmem_ld_32x32b_x8(tmem + lane_base + colD + (m0 + q) * Np + c0, r[q]);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  if (m0 + q >= MB_H) break;
#pragma unroll
                  for (int jj = 0; jj < 8; ++jj)
                    if (c0 + jj < T)
                      pdst[static_cast<size_t>(c0 + jj) * H + (m0 + q) * 128] = __uint_as_float(r[q][jj]);
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      ok = __syncthreads_and(ok);
      tc_fence_after();
    }

    // ---------------------------------------------------------- 4: y
    // y = the partials of CTAs 0 .. Gp-1 added in CTA order.  Each CTA takes
    // a contiguous range of 4-element quads of y; up to kDtMaxSlices threads
    // share a quad (contiguous CTA slices), their sums added in slice order.
    if (ok) ok = grid_barrier(hdr, 50, 1, &ticket);
    if (ok) {
      const int Gp = n_units < G ? n_units : G;
      const int nq_all = T * H / 4;
      const int q0 = static_cast<int>(static_cast<long long>(cta) * nq_all / G);
      const int nq = static_cast<int>(static_cast<long long>(cta + 1) * nq_all / G) - q0;
      if (nq > 0) {
        int ns = kDtThreads / nq;
        ns = ns < 1 ? 1 : (ns > kDtMaxSlices ? kDtMaxSlices : ns);
        ns = ns > Gp ? Gp : ns;
        float4* red = reinterpret_cast<float4*>(ring);        // [ns][nq]; the ring is idle now
        const float4* pd4 = reinterpret_cast<const float4*>(A.pd) + q0;
        for (int w = tid; w < nq * ns; w += kDtThreads) {
          const int sl = w / nq, qi = w - sl * nq;
          const int c0 = sl * Gp / ns, c1 = (sl + 1) * Gp / ns;
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int cb = c0; cb < c1; cb += kDtSumChunk) {
            float4 part[kDtSumChunk];
#pragma unroll
            for (int w2 = 0; w2 < kDtSumChunk; ++w2)
              part[w2] = cb + w2 < c1 ? __ldcg(pd4 + static_cast<size_t>(cb + w2) * nq_all + qi)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w2 = 0; w2 < kDtSumChunk; ++w2) {
              v.x += part[w2].x; v.y += part[w2].y; v.z += part[w2].z; v.w += part[w2].w;
            }
          }
          red[w] = v;
        }
        __syncthreads();
        for (int qi = tid; qi < nq; qi += kDtThreads) {
          float4 v = red[qi];
          for (int sl = 1; sl < ns; ++sl) {
            const float4 o = red[sl * nq + qi];
            v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
          }
          const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
          uint2 pk;
          pk.x = *reinterpret_cast<const uint32_t*>(&lo);
          pk.y = *reinterpret_cast<const uint32_t*>(&hi);
          reinterpret_cast<uint2*>(A.y)[q0 + qi] = pk;
        }
      }
    }
  } else {
    DtPlan P;
    P.nt = (ok && R.n_touched > 0) ? R.n_touched : 1;
    P.MB_I = (I + 127) / 128;
    P.MB_H = H / 128;
    P.KB_H = KB_H;
    P.KB_I = I / 64;
    {
      // split K when fewer than half the CTAs would stream (ranges of at
      // least 3 k-blocks), else only for long rows (ranges of at least 12
      // k-blocks): a shorter stream finishes sooner than the extra grid
      // barrier and the partial sums cost
      const int blocks = P.nt * P.MB_I;
      const int kmin = blocks * 2 <= G ? 3 : 12;
      const int max_split = P.KB_H / kmin < 1 ? 1 : (P.KB_H / kmin > kDtMaxSplit ? kDtMaxSplit : P.KB_H / kmin);
      int s_up = (G + blocks - 1) / blocks;
      s_up = s_up < 1 ? 1 : (s_up > max_split ? max_split : s_up);
      P.s_up = s_up;
      P.n_units = blocks * s_up;
    }
    P.per_mb = P.nt * P.KB_I;
    P.F = P.MB_H * P.per_mb;
    // the down tiles go to the first Gd CTAs, at least three per CTA
    const int Gd = (P.F + 2) / 3 < G ? (P.F + 2) / 3 : G;
    const int r0 = cta < Gd ? dt_range_start(cta, P.F, Gd) : P.F;
    const int r1 = cta < Gd ? dt_range_start(cta + 1, P.F, Gd) : P.F;
    const int my_down = r1 - r0;
    const int n_pre = my_down < S ? my_down : S;     // Wd tiles requested before the barrier
    int pre_it0 = 0;                                 // producer: stage use of the first of them
    // contributors of every output m-block, for the final reduction
    for (int c = tid; c < Gd; c += kDtThreads) {
      const int s0 = dt_range_start(c, P.F, Gd);
      s_first_mb[c] = dt_range_start(c + 1, P.F, Gd) > s0 ? s0 / P.per_mb : -1;
    }
    for (int mb = tid; mb < P.MB_H; mb += kDtThreads) {
      s_c0[mb] = dt_cta_of(mb * P.per_mb, P.F, Gd);
      s_c1[mb] = dt_cta_of(mb * P.per_mb + P.per_mb - 1, P.F, Gd);
    }

    // unit u -> (touched index, m-block, k-block range)
    auto unit_of = [&](int u, int& ti, int& mb, int& kb0, int& kb1) {
      const int blk = u / P.s_up, kr = u - blk * P.s_up;
      ti = blk / P.MB_I;
      mb = blk - ti * P.MB_I;
      kb0 = kr * P.KB_H / P.s_up;
      kb1 = (kr + 1) * P.KB_H / P.s_up;
    };
    auto tile_of = [&](int f, int& mbd, int& ti, int& kb) {
      mbd = f / P.per_mb;
      const int rem = f - mbd * P.per_mb;
      ti = rem / P.KB_I;
      kb = rem - ti * P.KB_I;
    };

    // ------------------------------------------------------------ 2: gate/up
    // stage = Wg tile at 0, Wu tile at 16 KiB, x tile (B, N = Np) at 32 KiB
    if (ok) {
      if (tid == 0) {
        for (int u = cta; ok && u < P.n_units; u += G) {
          int ti, mb, kb0, kb1;
          unit_of(u, ti, mb, kb0, kb1);
          const int e = R.touched[ti];
          for (int kb = kb0; kb < kb1; ++kb) {
            int s;
            if (!acquire(s)) { ok = false; break; }
            uint8_t* st = ring + s * SB;
            mbar_arrive_expect_tx(&full[s], 2 * kDtTileA + xtile);
            tma_load_2d_hint(st, &M.wg[e], &full[s], kb * 64, mb * 128, pol);
            tma_load_2d_hint(st + kDtTileA, &M.wu[e], &full[s], kb * 64, mb * 128, pol);
            tma_load_2d(st + 2 * kDtTileA, &M.x, &full[s], kb * 64, 0);
            ++p_it;
          }
        }
        pre_it0 = p_it;
        for (int j = 0; ok && j < n_pre; ++j) {
          int mbd, ti, kb, s;
          tile_of(r0 + j, mbd, ti, kb);
          if (!acquire(s)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], kDtTileA + 2 * xtile);   // the Hp tiles follow later
          tma_load_2d_hint(ring + s * SB, &M.wd[R.touched[ti]], &full[s], kb * 64, mbd * 128, pol);
          ++p_it;
        }
      }
      if (tid == 32) {
        int local = 0;
        for (int u = cta; ok && u < P.n_units; u += G, ++local) {
          int ti, mb, kb0, kb1;
          unit_of(u, ti, mb, kb0, kb1);
          const int acc = local & 1;
          if (!mbar_wait(&tempty[acc], ((local >> 1) & 1) ^ 1, nullptr, hdr, 44)) { ok = false; break; }
          tc_fence_after();
          const uint32_t dg = tmem + kDtColGU + acc * 2 * Np, du = dg + Np;
          for (int kb = kb0; kb < kb1; ++kb) {
            int s;
            if (!consume(s)) { ok = false; break; }
            const uint8_t* st = ring + s * SB;
            const uint8_t* b = st + 2 * kDtTileA;
  #pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16(dg, sdesc(st + kk * 32), sdesc(b + kk * 32), idesc, (kb > kb0 || kk) ? 1u : 0u);
  #pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16(du, sdesc(st + kDtTileA + kk * 32), sdesc(b + kk * 32), idesc,
                        (kb > kb0 || kk) ? 1u : 0u);
            umma_commit(&empty[s]);
            ++m_it;
          }
          if (!ok) break;
          umma_commit(&tfull[acc]);
        }
      }
      if (epi) {
        const int rl = quad * 32 + lane;
        const int cbeg = half * (Np / 2), cend = cbeg + Np / 2;   // this warp's token columns
        int local = 0;
        for (int u = cta; ok && u < P.n_units; u += G, ++local) {
          int ti, mb, kb0, kb1;
          unit_of(u, ti, mb, kb0, kb1);
          const int acc = local & 1;
          // all epilogue warps leave together (they meet at named barriers below)
          if (!epi_sync_and(warp_wait(&tfull[acc], (local >> 1) & 1, nullptr, hdr, 45))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tg = tmem + lane_base + kDtColGU + acc * 2 * Np;
          // compact loops: this code runs once per launch and unit, so its
          // size (instruction fetch) matters more than its unrolling
          if (P.s_up == 1) {
            // h through a shared tile [part][t][row] and two TMA stores (rows
            // past I are clipped by the store)
            if (tid == kDtEpiLeader) bulk_wait_read();   // the previous unit's stores read it
            epi_sync();
  #pragma unroll 1
            for (int c0 = cbeg; c0 < cend; c0 += 8) {
              uint32_t gr[8], ur[8];
              tmem_ld_32x32b_x8(tg + c0, gr);
              tmem_ld_32x32b_x8(tg + Np + c0, ur);
              tmem_ld_wait();
  #pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int t = c0 + j;
                const float v = swiglu_fast(__uint_as_float(gr[j]), __uint_as_float(ur[j])) *
                                alpha[ti * Np + t];
                const __nv_bfloat16 hi = __float2bfloat16_rn(v);
                hstage[t * 128 + rl] = hi;
                hstage[(Np + t) * 128 + rl] = __float2bfloat16_rn(v - __bfloat162float(hi));
              }
            }
            fence_proxy_async_smem();
            epi_sync();
            if (tid == kDtEpiLeader) {
              tma_store_2d(&M.hps, hstage, mb * 128, (ti * 2) * Np);
              tma_store_2d(&M.hps, hstage + Np * 128, mb * 128, (ti * 2 + 1) * Np);
              bulk_commit();
            }
          } else {
            float* pg = A.pgu + static_cast<size_t>(u) * 2 * Np * 128;
  #pragma unroll 1
            for (int c0 = cbeg; c0 < cend; c0 += 8) {
              uint32_t gr[8], ur[8];
              tmem_ld_32x32b_x8(tg + c0, gr);
              tmem_ld_32x32b_x8(tg + Np + c0, ur);
              tmem_ld_wait();
  #pragma unroll
              for (int j = 0; j < 8; ++j) {
                pg[static_cast<size_t>(c0 + j) * 128 + rl] = __uint_as_float(gr[j]);
                pg[static_cast<size_t>(Np + c0 + j) * 128 + rl] = __uint_as_float(ur[j]);
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);
        }
        if (tid == kDtEpiLeader) bulk_wait_all();   // h has reached global memory
      }
      ok = __syncthreads_and(ok);
    }

    // ------------------------------------------------------------ h complete
    unsigned round = 1;
    if (ok) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      ok = grid_barrier(hdr, 46, round++, nullptr);
    }
    if (ok && P.s_up > 1) {
      // add the k-range partials of G and U in order (zeros past s_up change
      // nothing), then as the direct path
      const int blocks = P.nt * P.MB_I;
      const int per_blk = Np * 128;
      const int total = blocks * per_blk;
      const int stride = G * kDtThreads;
      for (int q0 = cta * kDtThreads + tid; q0 < total; q0 += 2 * stride) {
        // every partial of two elements is requested before any is added
        float pgv[2][kDtMaxSplit], puv[2][kDtMaxSplit];
  #pragma unroll
        for (int w = 0; w < 2; ++w) {
          const int q = q0 + w * stride;
          const int blk = q / per_blk, rem = q - blk * per_blk;
          const float* pg = A.pgu + static_cast<size_t>(blk * P.s_up) * 2 * per_blk + rem;
  #pragma unroll
          for (int kr = 0; kr < kDtMaxSplit; ++kr) {
            const bool live = q < total && kr < P.s_up;
            pgv[w][kr] = live ? pg[static_cast<size_t>(kr) * 2 * per_blk] : 0.f;
            puv[w][kr] = live ? pg[static_cast<size_t>(kr) * 2 * per_blk + per_blk] : 0.f;
          }
        }
  #pragma unroll
        for (int w = 0; w < 2; ++w) {
          const int q = q0 + w * stride;
          if (q >= total) break;
          float g = 0.f, uu = 0.f;
  #pragma unroll
          for (int kr = 0; kr < kDtMaxSplit; ++kr) {
            g += pgv[w][kr];
            uu += puv[w][kr];
          }
          const int blk = q / per_blk, rem = q - blk * per_blk;
          const int t = rem >> 7, rl = rem & 127;
          const int ti = blk / P.MB_I, mb = blk - ti * P.MB_I;
          const int i = mb * 128 + rl;
          if (i >= I) continue;
          const float v = swiglu_fast(g, uu) * alpha[ti * Np + t];
          const __nv_bfloat16 hi = __float2bfloat16_rn(v);
          const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
          A.hp[(static_cast<size_t>(ti * 2) * Np + t) * I + i] = hi;
          A.hp[(static_cast<size_t>(ti * 2 + 1) * Np + t) * I + i] = lo;
        }
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");
      ok = grid_barrier(hdr, 47, round++, nullptr);
    }

    // ------------------------------------------------------------ 3: down
    // stage = Wd tile at 0, Hp high part at 16 KiB, Hp remainder after it
    if (ok) {
      if (tid == 0) {
        asm volatile("fence.proxy.async.global;" ::: "memory");
        for (int j = 0; ok && j < my_down; ++j) {
          int mbd, ti, kb, s;
          tile_of(r0 + j, mbd, ti, kb);
          if (j < n_pre) {
            s = (pre_it0 + j) % S;                  // Wd already requested, bytes armed
          } else {
            if (!acquire(s)) { ok = false; break; }
            mbar_arrive_expect_tx(&full[s], kDtTileA + 2 * xtile);
            tma_load_2d_hint(ring + s * SB, &M.wd[R.touched[ti]], &full[s], kb * 64, mbd * 128, pol);
            ++p_it;
          }
          uint8_t* b = ring + s * SB + kDtTileA;
          tma_load_2d(b, &M.hp, &full[s], kb * 64, (ti * 2) * Np);
          tma_load_2d(b + xtile, &M.hp, &full[s], kb * 64, (ti * 2 + 1) * Np);
        }
      }
      if (tid == 32) {
        int seg = -1, prev = -1;
        bool first = true;
        for (int j = 0; ok && j < my_down; ++j) {
          int mbd, ti, kb, s;
          tile_of(r0 + j, mbd, ti, kb);
          if (mbd != prev) {
            if (seg >= 0) umma_commit(&dfull);
            ++seg;
            prev = mbd;
            if (!mbar_wait(&dempty, (seg & 1) ^ 1, nullptr, hdr, 48)) { ok = false; break; }
            tc_fence_after();
            first = true;
          }
          if (!consume(s)) { ok = false; break; }
          const uint8_t* a = ring + s * SB;
          const uint8_t* b = a + kDtTileA;
  #pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem + kDtColD, sdesc(a + kk * 32), sdesc(b + kk * 32), idesc,
                      (!first || kk) ? 1u : 0u);
  #pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem + kDtColD, sdesc(a + kk * 32), sdesc(b + xtile + kk * 32), idesc, 1u);
          first = false;
          umma_commit(&empty[s]);
          ++m_it;
        }
        if (ok && seg >= 0) umma_commit(&dfull);
      }
      if (epi) {
        const int rl = quad * 32 + lane;
        const int cbeg = half * (Np / 2), cend = cbeg + Np / 2;
        const int n_seg = my_down > 0 ? (r1 - 1) / P.per_mb - r0 / P.per_mb + 1 : 0;
        for (int seg = 0; ok && seg < n_seg; ++seg) {
          if (!warp_wait(&dfull, seg & 1, nullptr, hdr, 49)) { ok = false; break; }
          tc_fence_after();
          float* pdst = A.pd + (static_cast<size_t>(cta) * kDtMaxSeg + seg) * Np * 128;
  #pragma unroll 1
          for (int c0 = cbeg; c0 < cend; c0 += 8) {
            uint32_t r[8];
            tmem_ld_32x32b_x8(tmem + lane_base + kDtColD + c0, r);
            tmem_ld_wait();
  #pragma unroll
            for (int j = 0; j < 8; ++j) pdst[static_cast<size_t>(c0 + j) * 128 + rl] = __uint_as_float(r[j]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&dempty);
        }
      }
      ok = __syncthreads_and(ok);
    }

    // ------------------------------------------------------------ 4: y
    if (ok) ok = grid_barrier(hdr, 50, round, &ticket);
    if (ok) {
      const int total = T * H;
      for (int q = cta * kDtThreads + tid; q < total; q += G * kDtThreads) {
        const int t = q / H, j = q - t * H;
        const int mbd = j >> 7, rl = j & 127;
        float v = 0.f;
        for (int cb = s_c0[mbd]; cb <= s_c1[mbd]; cb += kDtReduceChunk) {
          float part[kDtReduceChunk];
  #pragma unroll
          for (int w = 0; w < kDtReduceChunk; ++w) {
            const int c = cb + w;
            const int fm = c <= s_c1[mbd] ? s_first_mb[c] : -1;   // -1: past the end or empty range
            part[w] = fm >= 0 ? A.pd[((static_cast<size_t>(c) * kDtMaxSeg + (mbd - fm)) * Np + t) * 128 + rl]
                              : 0.f;
          }
  #pragma unroll
          for (int w = 0; w < kDtReduceChunk; ++w) v += part[w];
        }
        static_cast<__nv_bfloat16*>(A.y)[q] = __float2bfloat16_rn(v);
      }
    }

  }

  // ------------------------------------------------------------ teardown
  if (tid == 32) {
    // every issued UMMA has finished before TMEM is released
    umma_commit(&drained);
    mbar_wait(&drained, 0, nullptr, hdr, 51);
  }
  if (tid == 0 && !ok) {
    // copies still in flight land before the CTA exits (bounded)
    for (int j = 0; j < S && j < p_it; ++j) {
      const int q = p_it - 1 - j;
      mbar_wait(&full[q % S], (q / S) & 1, nullptr, nullptr, 52);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kDtTmemCols);
  if (tid == 0) grid_barrier_reset(hdr, ticket);
}

// =============================================================== host side
namespace {

struct DtLayout {
  int Np, Epad, nt_max, stages;
  int fused, gu_bufs;                   // down product per unit in the same CTA
  int spec, router_stages;              // fused MoE streaming every expert before the routing
  size_t stage, alpha_off, hstage_off, smem;   // shared memory
  size_t hp, pgu, pd, total;            // workspace (after the header)
};

inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool dt_layout(int T, int H, int I, int E, int k, DtLayout& L) {
  if (T < 1 || T > kDecodeTcMaxT || H % 128 != 0 || I % 64 != 0) return false;
  if (E > 1 && (E > MM_MAX_EXPERTS || k < 1 || k > MM_MAX_TOPK || k > E)) return false;
  L.Np = (T + 15) / 16 * 16;
  L.Epad = (E + 15) / 16 * 16;
  // MoE: the alpha table has a row per expert (speculative streaming indexes
  // it by expert), h at most one per expert
  L.nt_max = E > 1 ? E : 1;
  // a stage holds two 16 KiB weight tiles and one x tile (gate/up), or the
  // x and Wr tiles (router), or a Wd tile and the two Hp tiles (down)
  L.stage = round_up(2 * static_cast<size_t>(kDtTileA) + static_cast<size_t>(L.Np) * 128, 1024);
  const size_t alpha = round_up(static_cast<size_t>(L.nt_max) * L.Np * 4, 1024);
  const size_t hstage = static_cast<size_t>(2) * L.Np * 128 * 2;
  if (kDtSmemBudget < 1024 + alpha + hstage + 2 * L.stage) return false;
  L.stages = static_cast<int>((kDtSmemBudget - 1024 - alpha - hstage) / L.stage);
  if (L.stages > kDtMaxStages) L.stages = kDtMaxStages;
  L.alpha_off = static_cast<size_t>(L.stages) * L.stage;
  L.hstage_off = L.alpha_off + alpha;
  L.smem = L.hstage_off + hstage + 1024;             // 1 KiB: alignment slack
  const int G = kDtMaxCtas;
  const int blocks = L.nt_max * ((I + 127) / 128);
  // fused: the (G, U) accumulators and y^T for all H rows fit in TMEM, and
  // there are units enough to keep most SMs streaming (a fused unit cannot be
  // split along K; the dense FFN at H = 768 has only I / 128 of them)
  const int MB_H = H / 128;
  L.fused = ((MB_H + 2) * L.Np <= static_cast<int>(kDtTmemCols) && blocks >= kDtFusedMinUnits) ? 1 : 0;
  L.gu_bufs = (MB_H + 4) * L.Np <= static_cast<int>(kDtTmemCols) ? 2 : 1;
  const int units = blocks + G;                      // blocks * ceil(G / blocks) < blocks + G
  if (H / 128 > G || H / 128 > kDtMaxMB) return false;
  L.spec = 0;
  L.router_stages = 0;
  {
    // MoE router: all x tiles, then all Wr tiles, in the ring region; the A
    // read of the last x tile spans 128 rows
    const size_t xt = static_cast<size_t>(L.Np) * 128, wt = static_cast<size_t>(L.Epad) * 128;
    const size_t kbh = static_cast<size_t>(H / 64);
    const size_t need = std::max(kbh * (xt + wt), (kbh - 1) * xt + kDtTileA);
    if (E > 1 && need > static_cast<size_t>(L.stages) * L.stage) return false;
    // speculative streaming (fused MoE): every expert's units stream from
    // the start while the router and the routing run, and the units of the
    // experts no token selected are dropped once the routing is known; the
    // router's stages must leave one free, and the gate/up columns of TMEM
    // must stay clear of the router's logits (the last Epad columns)
    L.router_stages = static_cast<int>((need + L.stage - 1) / L.stage);
    if (L.fused && E > 1 && L.router_stages < L.stages &&
        2 * L.Np * L.gu_bufs + L.Epad <= static_cast<int>(kDtTmemCols))
      L.spec = 1;
  }
  {
    const long long F = static_cast<long long>(H / 128) * L.nt_max * (I / 64);
    if ((F + 1) * G >= (1ll << 31)) return false;    // down-range arithmetic in 32 bits
  }
  if (L.fused) {
    L.hp = 0;
    L.pgu = 0;
    L.pd = round_up(static_cast<size_t>(G) * T * H * 4, 256);   // one partial of y per CTA
  } else {
    L.hp = round_up(static_cast<size_t>(L.nt_max) * 2 * L.Np * I * 2, 256);
    L.pgu = round_up(static_cast<size_t>(units) * 2 * L.Np * 128 * 4, 256);
    L.pd = round_up(static_cast<size_t>(G) * kDtMaxSeg * L.Np * 128 * 4, 256);
  }
  L.total = L.hp + L.pgu + L.pd;
  return true;
}

template <int MAXW>
cudaError_t decode_tc_impl(const DtLayout& L, const void* x, const void* Wr,
                           const void* const* Wg, const void* const* Wu, const void* const* Wd,
                           DtArgs& A, cudaStream_t st) {
  static DtMaps<MAXW> m;                 // host staging, copied into the launch
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  const int T = A.T, H = A.H, I = A.I, nw = A.moe ? A.E : 1;
  if (!make_map_16(&m.x, x, H, T, L.Np, false)) return cudaErrorInvalidValue;
  if (A.moe && !make_map_16(&m.wr, Wr, H, A.E, L.Epad, false)) return cudaErrorInvalidValue;
  if (!L.fused) {
    if (!make_map_16(&m.hp, A.hp, I, static_cast<uint64_t>(L.nt_max) * 2 * L.Np, L.Np, false))
      return cudaErrorInvalidValue;
    if (!make_map_16(&m.hps, A.hp, I, static_cast<uint64_t>(L.nt_max) * 2 * L.Np, L.Np, false, 128,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  for (int e = 0; e < nw; ++e) {
    if (!make_map_16(&m.wg[e], Wg[e], H, I, 128, false)) return cudaErrorInvalidValue;
    if (!make_map_16(&m.wu[e], Wu[e], H, I, 128, false)) return cudaErrorInvalidValue;
    if (!make_map_16(&m.wd[e], Wd[e], I, H, 128, false)) return cudaErrorInvalidValue;
  }
  auto fn = L.fused ? decode_tc_kernel<MAXW, true> : decode_tc_kernel<MAXW, false>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(fn), L.smem);
  if (e != cudaSuccess) return e;
  int fit = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, fn, kDtThreads, L.smem);
  if (e != cudaSuccess) return e;
  if (fit < 1) return cudaErrorInvalidConfiguration;
  int grid = num_sms();
  if (grid > kDtMaxCtas) grid = kDtMaxCtas;
  // the speculative cut table holds kDtMaxLocalUnits units per CTA
  if (A.spec && (A.E * ((I + 127) / 128) + grid - 1) / grid > kDtMaxLocalUnits) A.spec = 0;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDtThreads);
  cfg.dynamicSmemBytes = L.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, m, A);
}

}  // namespace

size_t decode_tc_bytes(int T, int H, int I, int E, int k) {
  DtLayout L;
  return dt_layout(T, H, I, E, k, L) ? L.total : 0;
}

cudaError_t launch_decode_tc(const void* x, const void* Wr, const float* bias,
                             const void* const* Wg, const void* const* Wu, const void* const* Wd,
                             int T, int H, int I, int E, int k, float coef, int32_t* topk_idx,
                             float* topk_w, float* aux_loss, void* scratch, void* y,
                             WsHeader* hdr, cudaStream_t st, const RouterVariant* rv) {
  const bool moe = Wr != nullptr;
  DtLayout L;
  if (!dt_layout(T, H, I, moe ? E : 1, moe ? k : 1, L)) return cudaErrorInvalidValue;
  DtArgs A;
  memset(&A, 0, sizeof(A));
  if (rv != nullptr && moe) A.rv = *rv;
  A.T = T; A.Np = L.Np; A.H = H; A.I = I;
  A.E = moe ? E : 1; A.k = moe ? k : 1; A.moe = moe ? 1 : 0; A.coef = coef; A.bias = bias;
  A.topk_idx = topk_idx; A.topk_w = topk_w; A.aux_loss = aux_loss;
  char* base = static_cast<char*>(scratch);
  A.hp = reinterpret_cast<__nv_bfloat16*>(base);
  A.pgu = reinterpret_cast<float*>(base + L.hp);
  A.pd = reinterpret_cast<float*>(base + L.hp + L.pgu);
  A.y = y; A.hdr = hdr;
  A.stages = L.stages;
  A.gu_bufs = L.gu_bufs;
  A.spec = L.spec;
  A.router_stages = L.router_stages;
  A.Epad = L.Epad;
  A.stage_bytes = static_cast<uint32_t>(L.stage);
  A.hstage_off = static_cast<uint32_t>(L.hstage_off);
  A.alpha_off = static_cast<uint32_t>(L.alpha_off);
  if (A.E <= 8) return decode_tc_impl<8>(L, x, Wr, Wg, Wu, Wd, A, st);
  return decode_tc_impl<MM_MAX_EXPERTS>(L, x, Wr, Wg, Wu, Wd, A, st);
}

}  // namespace mm
