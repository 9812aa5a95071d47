// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

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
};
cudaError_t launch_dispatch(int dtype, const void* x, int64_t T, int H, int E, int k,
                            const int32_t* topk_idx, const int32_t* blk_cnt, const float* blk_prob,
                            const DispatchOut& D, int32_t* perm, void* Xp, cudaStream_t st);

// Tensor-core grouped GEMMs.  A is [rows, K] row-major; each group multiplies
// its rows by its own weight matrices.  gate/up: bf16 A and weights, fp16 h
// out.  down: fp16 h and fp16 Wd.
// wd_src / n_wd: the down matrices to copy to fp16 at wd16 (n_wd = 0: none).
cudaError_t launch_gateup_tc(const void* A, int64_t a_rows, int H, int I, const GroupRows& g,
                             const void* const* Wg, const void* const* Wu, void* h_out,
                             const void* const* wd_src, int n_wd, void* wd16, WsHeader* hdr,
                             cudaStream_t st);
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
