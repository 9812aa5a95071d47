// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstring>

#include "../../include/mm.h"
#include "mm_device.cuh"

namespace mm {

constexpr int kDtypeF32 = MM_DTYPE_F32;
constexpr int kDtypeBF16 = MM_DTYPE_BF16;

// Router / dispatch geometry.
constexpr int kRouteThreads = 256;          // 8 warps
constexpr int kRouteTokensPerBlock = 64;    // 8 tokens per warp
constexpr int kScanThreads = 512;
constexpr int kMaxGroups = MM_MAX_EXPERTS * MM_MAX_TOPK;     // (slot, expert) groups

// Decode-sized calls stream each weight row once: on the CUDA cores for
// T <= kDecodeMaxT, on the tensor cores (decode_tc.cu) for T <= kDecodeTcMaxT.
constexpr int kDecodeMaxT = 16;
constexpr int kDecodeTcMaxT = 64;
constexpr int kDecodeSwMaxT = 128;          // dense FFN with the tokens as the M operand

// Per-expert device pointers passed by value to a kernel.
struct PtrArray {
  const void* p[MM_MAX_EXPERTS];
};

// Tensor-core GEMM geometry (tcgen05 over a CTA pair; the rest in gemm_tc.cu).
constexpr int kTcBM = 128;                  // rows per CTA (TMEM lanes)
constexpr int kTcBK = 64;                   // K per stage: one 128-byte swizzle row of 16-bit data

// How the down-projection epilogue writes its rows.  With k >= 2 the
// contributions of a token are summed in fp32 in slot order, one slot per
// launch (phase): the first phase stores, middle phases add, the last phase
// adds and rounds once to y's dtype.  No atomics; the result is deterministic.
enum CombineMode : int {
  kCombineStore = 0,    // y[token] = alpha * acc                   (dense, k = 1)
  kCombineFirst = 1,    // acc32[token] = alpha * acc                (slot 0 of k >= 2)
  kCombineAccum = 2,    // acc32[token] += alpha * acc               (slots 1 .. k-2)
  kCombineLast = 3      // y[token] = round(acc32[token] + alpha * acc)   (slot k-1)
};

// Description of the row groups of a grouped GEMM: group g owns rows
// [offsets[g], offsets[g+1]) of A and uses weight matrix g % n_weights.
struct GroupRows {
  const int32_t* offsets;   // device [G+1], or nullptr: one group of dense_rows rows
  int G;
  int dense_rows;
  int n_weights;
};

// Epilogue inputs of the down projection.
struct DownEpilogue {
  void* y;                  // [T, H], x's dtype
  float* acc32;             // [T, H] fp32 running sum (k >= 2), may alias y for fp32
  const int32_t* perm;      // row -> t*k + s, or nullptr (row == token, alpha = 1)
  const float* topk_w;      // [T*k] alpha, or nullptr (alpha = 1)
  int k;
  int mode;                 // CombineMode
  const void* resid;        // [T, H] x's dtype, added to y at the final store
                            // (the block's residual), or nullptr
};

// fp16 copy of the down matrices, made by the epilogue warps of the gate/up
// GEMM while its tensor pipe runs (HBM is mostly idle then): n_mat bf16
// matrices of nvec 16-byte vectors each -> dst [n_mat][8 * nvec] fp16.
// The conversion is exact for |w| >= 2^-14 (smaller magnitudes become fp16
// subnormals, error <= 2^-25).  n_mat = 0: nothing to convert.
struct WdConvert {
  PtrArray src;
  __half* dst;
  int64_t nvec;
  int n_mat;
};

// Router variants and saved router statistics, all optional (null / 0:
// off).  noise: router noise, added to each token's logits after the bias;
// z-loss = z_coef * (1/T) sum_t lse_t^2 with lse_t the logsumexp of the
// token's logits; probs / lse: the softmax probabilities [T, E] and lse [T]
// as computed, for a backward pass.  blk_z is workspace: per router block,
// the sum of its tokens' lse^2, added in a fixed order by the finaliser.
struct RouterVariant {
  const float* noise;    // [T, E] fp32
  float z_coef;
  float* z_loss;         // fp32 scalar
  float* probs;          // [T, E] fp32
  float* lse;            // [T] fp32
  float* blk_z;          // [nblk] fp32 (prefill router)
};

// RMSNorm prologue of the MiniMind block (lesson 13 §3 step 2: hidden +
// mlp(post_attention_layernorm(hidden))), x_n = x / sqrt(mean x^2 + eps) * w.
// The router takes it at full precision: logits = inv_rms * x . (w * Wr),
// with w * Wr as the tensor core's two exact bf16 halves (wr_hl rows [0, E):
// high part, [E, 2E): remainder), or w folded into x on the CUDA cores; it
// stores each token's inv_rms for the dispatch, which writes the rows x_n.
struct BlockNorm {
  const void* w;          // [H] x's dtype; null: no norm
  float eps;
  float* inv_rms;         // [T] fp32 out (router) / in (dispatch)
  const void* wr_hl;      // bf16 [2E, H] (tensor-core router)
};

// Router grid (routing.cu): per 64-token block logits, softmax, top-k, alpha
// and partial counts / probability sums; with do_scan the block that
// finishes last runs the scan (counts, aux loss; its counter lives in the
// workspace header).
struct RouteOut {
  int32_t* blk_base;     // [nblk, k*E] or null
  int32_t* offsets;      // [k*E + 1] or null
  int32_t* counts;       // [E] or null
  float* aux_loss;       // scalar or null
  float coef;
  int do_scan;           // 0: the dispatch kernel derives bases, offsets, counts, aux
  RouterVariant rv;
  BlockNorm norm;
};
struct RouteExtras {
  int32_t* blk_base;
  int32_t* offsets;
  int32_t* counts;
  float* aux_loss;
  float coef;
  WsHeader* hdr;
  int stage_x;           // x rows staged in shared memory at byte x_off
  uint32_t x_off;
  int do_scan;
  RouterVariant rv;
  BlockNorm norm;
  const void* xrow;      // x in global memory (the norm's sums of squares)
};
cudaError_t launch_router(int dtype, const void* x, const void* Wr, const float* bias, int64_t T,
                          int H, int E, int k, int32_t* topk_idx, float* topk_w, int32_t* blk_cnt,
                          float* blk_prob, const RouteOut& out, WsHeader* hdr, cudaStream_t st);
size_t router_smem_bytes(int H, int E, int k);
// Dispatch (routing.cu): group bases, offsets, expert counts and the aux
// loss from the router's per-block partials, then the token permute.
struct DispatchOut {
  int32_t* offsets;      // [k*E + 1]
  int32_t* counts;       // [E] or null
  float* aux_loss;
  float coef;
  WsHeader* hdr;
  RouterVariant rv;      // block 0 finalises the z-loss from rv.blk_z
  BlockNorm norm;        // w != null: the rows written are x * inv_rms * w
};
cudaError_t launch_dispatch(int dtype, const void* x, int64_t T, int H, int E, int k,
                            const int32_t* topk_idx, const int32_t* blk_cnt, const float* blk_prob,
                            const DispatchOut& D, int32_t* perm, void* Xp, cudaStream_t st);

// Router and dispatch fused into one kernel (routing.cu): the same outputs
// as launch_router followed by launch_dispatch, with x read once.  Taken
// where route_dispatch_ok() holds (shapes, alignment, every block resident);
// otherwise the two kernels run.
bool route_dispatch_ok(int dtype, const void* x, const void* Wr, int64_t T, int H, int E, int k,
                       const DispatchOut& D);
cudaError_t launch_route_dispatch(int dtype, const void* x, const void* Wr, const float* bias,
                                  int64_t T, int H, int E, int k, int32_t* topk_idx, float* topk_w,
                                  int32_t* blk_cnt, float* blk_prob, const DispatchOut& D,
                                  int32_t* perm, void* Xp, cudaStream_t st);

// Permute-free gate/up: row r of the grouped problem is x row perm[r] / k
// (gathered by TMA, four rows per request) instead of a copied row of Xp.
struct RowGather {
  const int32_t* perm;      // [n_rows] row -> assignment t*k + s, or null: A rows as stored
  int k;
  int n_rows;               // rows of the grouped problem (T*k)
};

// Tensor-core grouped GEMMs.  A is [rows, K] row-major; each group multiplies
// its rows by its own weight matrices.  gate/up: bf16 A and weights, fp16 h
// out.  down: fp16 h and fp16 Wd.
// wd_src / n_wd: the down matrices to copy to fp16 at wd16 (n_wd = 0: none).
cudaError_t launch_gateup_tc(const void* A, int64_t a_rows, int H, int I, const GroupRows& g,
                             const void* const* Wg, const void* const* Wu, void* h_out,
                             const void* const* wd_src, int n_wd, void* wd16, WsHeader* hdr,
                             cudaStream_t st, const RowGather* gather = nullptr);
cudaError_t launch_down_tc(const void* h, int64_t a_rows, int H, int I, const GroupRows& g,
                           const void* const* Wd, const DownEpilogue& ep, WsHeader* hdr,
                           cudaStream_t st);

// CUDA-core (fp32 FMA) grouped kernels, any dtype.
cudaError_t launch_gateup_simt(int dtype, const void* A, int64_t a_rows, int H, int I,
                               const GroupRows& g, const void* const* Wg, const void* const* Wu,
                               void* h_out, cudaStream_t st);
cudaError_t launch_down_simt(int dtype, const void* h, int64_t a_rows, int H, int I,
                             const GroupRows& g, const void* const* Wd, const DownEpilogue& ep,
                             cudaStream_t st);

// Decode-sized forward on the CUDA cores (T <= kDecodeMaxT, bf16): one
// cooperative kernel routes (MoE: Wr != nullptr), writes the fp32 h [T*k, I]
// (dense: [T, I]) into hbuf, meets every other CTA at a grid barrier kept in
// the workspace header, and forms y.  Block 0 writes topk_idx / topk_w /
// aux_loss (MoE).  decode_smem_bytes is its dynamic shared memory (dense: E = k = 1).
size_t decode_smem_bytes(int T, int H, int I, int E, int k);
cudaError_t launch_decode_ffn(const void* x, const void* Wr, const float* bias,
                              const void* const* Wg, const void* const* Wu, const void* const* Wd,
                              int T, int H, int I, int E, int k, float coef, int32_t* topk_idx,
                              float* topk_w, float* aux_loss, void* hbuf, void* y, WsHeader* hdr,
                              cudaStream_t st, const RouterVariant* rv = nullptr);

// Decode-sized forward on the tensor cores (T <= kDecodeTcMaxT, bf16): one
// cooperative kernel; weights are the UMMA M operand (128 rows per tile), the
// T tokens (padded to a multiple of 16) the N operand.  decode_tc_bytes is
// its workspace after the 256-byte header (0: shape not supported).
size_t decode_tc_bytes(int T, int H, int I, int E, int k);
cudaError_t launch_decode_tc(const void* x, const void* Wr, const float* bias,
                             const void* const* Wg, const void* const* Wu, const void* const* Wd,
                             int T, int H, int I, int E, int k, float coef, int32_t* topk_idx,
                             float* topk_w, float* aux_loss, void* scratch, void* y,
                             WsHeader* hdr, cudaStream_t st, const RouterVariant* rv = nullptr);

// Dense FFN on the tensor cores with the tokens as the M operand (T <=
// kDecodeSwMaxT, bf16; decode_sw.cu): one cooperative kernel, units of 64
// rows of I each run gate/up, SwiGLU and their share of the down product,
// unit partials of y added after one grid barrier.  decode_sw_bytes is its
// workspace after the 256-byte header (0: shape not supported).
size_t decode_sw_bytes(int T, int H, int I);
cudaError_t launch_decode_sw(const void* x, const void* Wg, const void* Wu, const void* Wd, int T,
                             int H, int I, void* scratch, void* y, WsHeader* hdr, cudaStream_t st);

cudaError_t launch_watchdog_selftest(WsHeader* hdr, uint32_t limit_us, cudaStream_t st);

// fp16 copy of a bf16 down-projection matrix of n elements (n a multiple of
// 8, 16-byte aligned); out-of-range values set MM_ERR_RANGE in hdr (nullable).
cudaError_t launch_prepare_wd16(const void* Wd, void* Wd16, int64_t n, WsHeader* hdr,
                                cudaStream_t st);

// Block prologue helpers (norm.cu): the router weights with the norm weight
// folded in, as exact bf16 halves (hi = bf16(w * Wr), lo = w * Wr - hi), and
// the normalised rows x_n = x * inv_rms * w (x's dtype) with inv_rms [T].
cudaError_t launch_norm_fold_router(const void* Wr, const void* w, int E, int H, void* wr_hl,
                                    cudaStream_t st);
cudaError_t launch_rms_norm_rows(int dtype, const void* x, const void* w, float eps, int64_t T,
                                 int H, void* xn, float* inv_rms, cudaStream_t st);

// ----------------------------------------------------------- backward pass
// Tensor-core GEMMs of the backward (gemm_bwd.cu).  kSchedRows: row groups
// of a K-major A (dgrad: dh = dy Wd, dx = [dG | dU] [Wg; Wu]); kSchedKGrp:
// weight gradients whose K runs over a group's rows (A and B MN-major).
constexpr int kSchedRows = 0, kSchedKGrp = 1;
constexpr int kBwMaxMaps = 2;                            // A matrices of the K-grouped GEMM
constexpr int kBwMaxGroups = 3 * MM_MAX_EXPERTS;         // problems (K-grouped) / groups (rows)

// One weight gradient: out [M, N] fp32 = A[:, a_col0 .. a_col0 + M)^T B over
// the rows of group grp; A = a_map-th A matrix, B = b_map-th B matrix.
struct BwProblem {
  float* out;
  int M, N;
  int grp;
  int a_map, b_map;
  int a_col0;
};

struct BwParams {
  CUtensorMap a[kBwMaxMaps];            // rows: A [rows, K] (box 64 x 128); K-grouped: A matrices (64 x 64)
  CUtensorMap b_lo[MM_MAX_EXPERTS];     // rows: per group, B for k-blocks < kb_split; K-grouped: B matrices
  CUtensorMap b_hi[MM_MAX_EXPERTS];     // rows: per group, B for k-blocks >= kb_split
  BwProblem prob[kBwMaxGroups];         // K-grouped problems
  const int32_t* offsets;               // group row offsets [G+1] (rows) / [n_groups+1], or null
  int G;                                // groups (rows) / problems (K-grouped)
  int n_groups;                         // K-grouped: groups of rows
  int dense_rows;                       // offsets == null: one group [0, dense_rows)
  int K, N, kb_split;                   // rows schedule
  void* out;                            // rows schedule: [rows, ldo]
  int64_t ldo;
  int out_type;                         // rows schedule: kBwOutF32 / kBwOutBF16 / kBwOutF16
  int out_tma;                          // rows schedule: full 32-row pieces go out through o
  CUtensorMap o;                        // rows schedule: out as 32 x 32 store boxes
};

// Output element type of a rows-schedule GEMM.  fp16 output (dh, read only
// by the SwiGLU-backward epilogue) is checked against the fp16 range: a value
// that rounds to infinity (or a NaN) records MM_ERR_RANGE in the header.
constexpr int kBwOutF32 = 0, kBwOutBF16 = 1, kBwOutF16 = 2;
cudaError_t launch_bw_dgrad(const void* A, int64_t a_rows, int K, const int32_t* offsets, int G,
                            int dense_rows, const void* const* b_lo, const void* const* b_hi,
                            int kb_split, int N, void* out, int64_t ldo, int out_type,
                            WsHeader* hdr, cudaStream_t st);
cudaError_t launch_bw_wgrad(const void* const* a_mats, const int64_t* a_cols, int n_a,
                            const void* const* b_mats, const int64_t* b_cols, int n_b,
                            int64_t k_rows, const BwProblem* probs, int n_probs,
                            const int32_t* offsets, int n_groups, int dense_rows, WsHeader* hdr,
                            cudaStream_t st);

// Epilogue of the gate/up GEMM run again in the backward (recomputing g and
// u): with dhu = dy Wd (unscaled by alpha) of the row, alpha of the row,
//   h = SiLU(g) u;  dalpha partial = sum over the tile's columns of h * dhu;
//   dh = alpha dhu;  dU = dh SiLU(g);  dG = dh u SiLU'(g);  out: dG | dU, alpha h.
struct UpBwd {
  const __half* dhu;          // [rows, I] fp16 (not an MMA operand: 11 significant bits)
  const int32_t* perm;        // row -> assignment t*k + s, -1 for padding; null: alpha = 1
  const float* topk_w;        // [T*k] alpha
  __nv_bfloat16* dgu;         // [rows, 2I]: dG in columns [0, I), dU in [I, 2I)
  __nv_bfloat16* ha;          // [rows, I]: alpha * h
  float* dalpha_part;         // [rows, n_parts] or null
  int n_parts;                // 2 * ceil(I / 128)
};
// Launch as a programmatic dependent of the stream's previous kernel (the
// kernel's set-up and the launch itself overlap that kernel's tail; the
// kernel waits for it with griddepcontrol.wait before touching its data).
template <typename Kern, typename... Args>
inline cudaError_t launch_dependent_kernel(Kern fn, dim3 grid, dim3 block, size_t smem,
                                           cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, args...);
}

cudaError_t launch_gateup_bwd_tc(const void* A, int64_t a_rows, int H, int I, const GroupRows& g,
                                 const void* const* Wg, const void* const* Wu, const UpBwd& ub,
                                 WsHeader* hdr, cudaStream_t st);

// Backward dispatch and router backward (backward.cu).  Rows of the backward
// are grouped by expert (token order, then slot), each group starting on a
// multiple of 64 rows; padding rows are zero in Xp and dYp and have perm -1.
constexpr int kBwAlign = 64;
cudaError_t launch_bwd_count(const int32_t* topk_idx, int64_t T, int E, int k, int32_t* blk_cnt,
                             cudaStream_t st);
struct BwdDispatchOut {
  int32_t* offsets;           // [E + 1] padded group offsets
  int32_t* counts;            // [E] assignments per expert
  int32_t* perm;              // [rows_pad] row -> assignment, -1 padding
  int32_t* pos;               // [T*k] assignment -> row
  void* xp;                   // [rows_pad, H] x rows
  void* dyp;                  // [rows_pad, H] dy rows
  WsHeader* hdr;              // watchdog (the staged copy's bounded wait)
};
cudaError_t launch_bwd_dispatch(const void* x, const void* dy, const int32_t* topk_idx, int64_t T,
                                int H, int E, int k, const int32_t* blk_cnt,
                                const BwdDispatchOut& o, cudaStream_t st);
struct RouterBwd {
  const int32_t* topk_idx;    // [T, k]
  const float* topk_w;        // [T, k] alpha
  const float* probs;         // [T, E]
  const float* lse;           // [T] or null (z term off)
  const int32_t* counts;      // [E]
  const int32_t* pos;         // [T*k]
  const float* dalpha_part;   // [rows_pad, n_parts]
  int n_parts;
  const __half* dxp;          // [rows_pad, H] fp16 per-assignment dx (range-checked when written)
  float coef, d_aux, z_coef, d_z;
  float* dr;                  // [T, E] out: dL/dlogits
  void* dx;                   // [T, H] out, x's dtype
  float* dwr_part;            // [nblk, E, H] out
  float* dbias_part;          // [nblk, E] out
};
cudaError_t launch_router_bwd(const void* x, const void* Wr, int64_t T, int H, int E, int k,
                              const RouterBwd& rb, cudaStream_t st);
cudaError_t launch_router_bwd_reduce(const float* dwr_part, const float* dbias_part, int nblk,
                                     int E, int H, float* dWr, float* d_bias, cudaStream_t st);

// Workspace of the path that `path` (AUTO: the automatic choice) resolves to
// for a dense call of this shape; 0 when that path does not take it.
size_t dense_workspace_for_path(int64_t T, int H, int I, int dtype, int path);

// TMA tensor map of a 16-bit row-major [outer, inner] matrix, box box_inner x
// box_rows, zero fill outside; cached by (pointer, shape, box, type, swizzle).
bool make_map_16(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t outer,
                 uint32_t box_rows, bool is_f16, uint32_t box_inner = kTcBK,
                 CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B);

// TMA tensor map of a 16-bit tensor (bf16, or fp16) viewed in three dimensions (element
// strides 1, strides[0], strides[1] bytes), box box[0] x box[1] x box[2],
// 2-D map of a row-major matrix of fp32 or bf16 elements with an explicit
// row pitch (bytes, a multiple of 16), for TMA tensor stores; cached like
// make_map_16.
bool make_map_2d(CUtensorMap* out, const void* ptr, bool fp32, uint64_t inner, uint64_t outer,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz);
// 128-byte swizzle unless given, zero fill outside; cached like make_map_16.
bool make_map_3d(CUtensorMap* out, const void* ptr, const uint64_t dims[3],
                 const uint64_t strides[2], const uint32_t box[3], bool is_f16 = false,
                 CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B);

int num_sms();   // of the current device, looked up once per device

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) for `fn`, skipped when an
// equal or larger value was already set on the current device (so that calls
// made during stream capture issue no attribute changes after the first).
cudaError_t ensure_dynamic_smem(const void* fn, size_t bytes);

}  // namespace mm
