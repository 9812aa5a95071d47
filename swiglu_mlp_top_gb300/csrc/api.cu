// C ABI (include/mm.h): argument checks, workspace layout, kernel sequencing.
// Every entry point only enqueues work on the caller's stream.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "mm_kernels.cuh"

namespace mm {
namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t elem_bytes(int dtype) { return dtype == kDtypeBF16 ? 2 : 4; }
inline int route_blocks(int64_t T) {
  return static_cast<int>((T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock);
}

thread_local char g_last_error[256] = "";

int cuda_fail(cudaError_t e, const char* what) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s", what, cudaGetErrorString(e));
  return MM_ERR_CUDA;
}

// ----------------------------------------------------------------- layouts
struct MoeLayout {
  size_t offsets, counts, blk_cnt, blk_prob, blk_z, inv_rms, wr_hl, perm, xp, h, acc32, wd16, total;
};

// h is stored in fp16 for bf16 inputs (see gemm_tc.cu) and in fp32 for fp32.
inline size_t h_bytes(int dtype) { return dtype == kDtypeBF16 ? 2 : 4; }

// Workspace of the MoE forward: routing tables, the dispatched rows Xp
// ([T*k, H], grouped by slot, then expert, then token), h ([T*k, I]) and,
// for bf16, the fp32 running sum of y ([T, H], k >= 2) and fp16 copies of the
// E down-projection matrices.
MoeLayout moe_layout(int64_t T, int H, int I, int E, int k, int dtype, bool with_xp = true) {
  MoeLayout L;
  const size_t es = elem_bytes(dtype);
  const size_t nblk = static_cast<size_t>(route_blocks(T));
  const size_t rows = static_cast<size_t>(T) * static_cast<size_t>(k);
  const size_t G = static_cast<size_t>(k) * E;
  size_t off = sizeof(WsHeader);
  L.offsets = off;  off += align_up(4 * (G + 1));
  L.counts = off;   off += align_up(4 * static_cast<size_t>(E));
  L.blk_cnt = off;  off += align_up(4 * nblk * G);
  L.blk_prob = off; off += align_up(4 * nblk * E);
  L.blk_z = off;    off += align_up(4 * nblk);
  L.inv_rms = off;  off += align_up(4 * static_cast<size_t>(T));            // block norm
  L.wr_hl = off;    off += align_up(4 * static_cast<size_t>(E) * H);        // block norm, bf16 [2E, H]
  L.perm = off;     off += align_up(4 * rows);
  L.xp = off;       if (with_xp) off += align_up(es * rows * H);   // not with the gathering gate/up
  L.h = off;        off += align_up(h_bytes(dtype) * rows * I);
  L.acc32 = off;    if (k >= 2 && dtype == kDtypeBF16) off += align_up(4 * static_cast<size_t>(T) * H);
  // bf16: fp16 copy of the E down matrices
  L.wd16 = off;
  if (dtype == kDtypeBF16) off += align_up(2 * static_cast<size_t>(E) * H * I);
  L.total = off;
  return L;
}

struct RouteLayout {
  size_t blk_cnt, blk_prob, blk_z, total;
};
RouteLayout route_layout(int64_t T, int E, int k) {
  RouteLayout L;
  const size_t nblk = static_cast<size_t>(route_blocks(T));
  size_t off = sizeof(WsHeader);
  L.blk_cnt = off;  off += align_up(4 * nblk * static_cast<size_t>(k) * E);
  L.blk_prob = off; off += align_up(4 * nblk * E);
  L.blk_z = off;    off += align_up(4 * nblk);
  L.total = off;
  return L;
}

// Backward of the dense FFN (bf16): dh = dy Wd [T, I] (fp16: only the
// SwiGLU-backward epilogue reads it, no MMA), dG | dU [T, 2I] and h [T, I]
// (bf16: operands of the tensor-core GEMMs).
struct DenseBwdLayout {
  size_t dh, dgu, h, total;
};
DenseBwdLayout dense_bwd_layout(int64_t T, int I) {
  DenseBwdLayout L;
  const size_t ti = static_cast<size_t>(T) * I;
  size_t off = sizeof(WsHeader);
  L.dh = off;  off += align_up(2 * ti);
  L.dgu = off; off += align_up(4 * ti);
  L.h = off;   off += align_up(2 * ti);
  L.total = off;
  return L;
}

// Backward of the MoE layer (bf16).  Rows are the T*k assignments grouped by
// expert, each group padded to a multiple of kBwAlign rows: at most
// T*k + E*(kBwAlign - 1) rows.
struct MoeBwdLayout {
  int64_t rows;                    // row capacity of the padded buffers
  int n_parts;                     // dalpha partials per row
  size_t blk_cnt, offsets, counts, pos, perm, xp, dyp, dhu, dgu, ha, dpart, dxp, dr, dwr_part,
      dbias_part, total;
};
MoeBwdLayout moe_bwd_layout(int64_t T, int H, int I, int E, int k) {
  MoeBwdLayout L;
  const size_t nblk = static_cast<size_t>(route_blocks(T));
  L.rows = T * k + static_cast<int64_t>(E) * (kBwAlign - 1);
  L.n_parts = 2 * ((I + 127) / 128);
  const size_t R = static_cast<size_t>(L.rows);
  size_t off = sizeof(WsHeader);
  L.blk_cnt = off;    off += align_up(4 * nblk * E);
  L.offsets = off;    off += align_up(4 * (static_cast<size_t>(E) + 1));
  L.counts = off;     off += align_up(4 * static_cast<size_t>(E));
  L.pos = off;        off += align_up(4 * static_cast<size_t>(T) * k);
  L.perm = off;       off += align_up(4 * R);
  L.xp = off;         off += align_up(2 * R * H);
  L.dyp = off;        off += align_up(2 * R * H);
  L.dhu = off;        off += align_up(2 * R * I);
  L.dgu = off;        off += align_up(4 * R * I);
  L.ha = off;         off += align_up(2 * R * I);
  L.dpart = off;      off += align_up(4 * R * L.n_parts);
  L.dxp = off;        off += align_up(2 * R * H);
  L.dr = off;         off += align_up(4 * static_cast<size_t>(T) * E);
  L.dwr_part = off;   off += align_up(4 * nblk * E * H);
  L.dbias_part = off; off += align_up(4 * nblk * E);
  L.total = off;
  return L;
}

// Dense workspace of the tensor-core and SIMT paths: h [T, I], then (bf16)
// the fp16 copy of Wd.
size_t dense_h_bytes(int64_t T, int I, int dtype) {
  return align_up(h_bytes(dtype) * static_cast<size_t>(T) * I);
}
size_t dense_tensor_ws_bytes(int64_t T, int H, int I, int dtype) {
  return sizeof(WsHeader) + dense_h_bytes(T, I, dtype) +
         (dtype == kDtypeBF16 ? align_up(2 * static_cast<size_t>(H) * I) : 0);
}

// The dense block (x + FFN(RMSNorm(x))): the tensor-core / SIMT workspace,
// then the normalised rows x_n [T, H] and inv_rms [T].
size_t dense_block_ws_bytes(int64_t T, int H, int I, int dtype) {
  return dense_tensor_ws_bytes(T, H, I, dtype) + align_up(elem_bytes(dtype) * static_cast<size_t>(T) * H) +
         align_up(4 * static_cast<size_t>(T));
}

bool valid_dtype(int dtype) { return dtype == kDtypeF32 || dtype == kDtypeBF16; }

// bf16 tensor-core / streaming kernels tile K and N by 64
bool tensor_shape_ok(int H, int I) { return H % 64 == 0 && I % 64 == 0; }

// Scratch (after the header) of the two weight-streaming kernels; 0 when the
// shape is outside the kernel's limits.  E = k = 1 for the dense FFN.
size_t stream_simt_bytes(int64_t T, int H, int I, int E, int k, int dtype) {
  if (dtype != kDtypeBF16 || T < 1 || T > kDecodeMaxT) return 0;
  if (decode_smem_bytes(static_cast<int>(T), H, I, E, k) > 200 * 1024) return 0;
  return align_up(4 * static_cast<size_t>(T) * k * I);    // fp32 h
}
size_t stream_tc_bytes(int64_t T, int H, int I, int E, int k, int dtype) {
  if (dtype != kDtypeBF16 || T < 1 || T > kDecodeTcMaxT) return 0;
  return decode_tc_bytes(static_cast<int>(T), H, I, E, k);
}
// The dense FFN streams on the tensor cores with the tokens as the M operand
// (decode_sw.cu, up to kDecodeSwMaxT tokens) where that kernel takes the
// shape, else with the weights as the M operand (decode_tc.cu).
size_t dense_stream_tc_bytes(int64_t T, int H, int I, int dtype) {
  if (dtype != kDtypeBF16 || T < 1 || T > kDecodeSwMaxT) return 0;
  const size_t sw = decode_sw_bytes(static_cast<int>(T), H, I);
  return sw ? sw : stream_tc_bytes(T, H, I, 1, 1, dtype);
}

// Workspace of one path (0: the path does not take this shape), and the
// workspace that serves every path valid for the shape.
size_t dense_path_bytes(int64_t T, int H, int I, int dtype, int p) {
  size_t b = 0;
  switch (p) {
    case MM_PATH_STREAM: b = stream_simt_bytes(T, H, I, 1, 1, dtype); break;
    case MM_PATH_STREAM_TC: b = dense_stream_tc_bytes(T, H, I, dtype); break;
    default: return dense_tensor_ws_bytes(T, H, I, dtype);
  }
  return b ? sizeof(WsHeader) + b : 0;
}
size_t dense_ws_bytes(int64_t T, int H, int I, int dtype) {
  size_t need = dense_tensor_ws_bytes(T, H, I, dtype);
  need = std::max(need, dense_path_bytes(T, H, I, dtype, MM_PATH_STREAM));
  need = std::max(need, dense_path_bytes(T, H, I, dtype, MM_PATH_STREAM_TC));
  return need;
}
size_t moe_path_bytes(int64_t T, int H, int I, int E, int k, int dtype, int p) {
  size_t b = 0;
  switch (p) {
    case MM_PATH_STREAM: b = stream_simt_bytes(T, H, I, E, k, dtype); break;
    case MM_PATH_STREAM_TC: b = stream_tc_bytes(T, H, I, E, k, dtype); break;
    case MM_PATH_TENSOR_GATHER: return moe_layout(T, H, I, E, k, dtype, false).total;
    default: return moe_layout(T, H, I, E, k, dtype).total;
  }
  return b ? sizeof(WsHeader) + b : 0;
}
size_t moe_ws_bytes(int64_t T, int H, int I, int E, int k, int dtype) {
  size_t need = moe_layout(T, H, I, E, k, dtype).total;
  need = std::max(need, moe_path_bytes(T, H, I, E, k, dtype, MM_PATH_STREAM));
  need = std::max(need, moe_path_bytes(T, H, I, E, k, dtype, MM_PATH_STREAM_TC));
  return need;
}

// AUTO: fp32 -> CUDA-core kernels.  bf16 -> weight streaming for decode-sized
// T (every weight row read once): on the CUDA cores for the smallest T (up to
// 4 tokens dense, 2 tokens MoE: their cost grows with the tokens and the
// touched experts), on the tensor cores up to kDecodeSwMaxT tokens (dense) or
// kDecodeTcMaxT (MoE) (a fixed cost of one to three grid barriers and the
// partial sums); tensor-core GEMMs beyond.
inline int64_t stream_simt_auto_max_t(int E) { return E == 1 ? 4 : 2; }
int resolve_path(int path, int dtype, int64_t T, int H, int I, int E, int k, bool dense) {
  if (path != MM_PATH_AUTO) return path;
  if (dtype == kDtypeF32) return MM_PATH_SIMT;
  if (T <= stream_simt_auto_max_t(E) && stream_simt_bytes(T, H, I, E, k, dtype) > 0)
    return MM_PATH_STREAM;
  if (dense ? dense_stream_tc_bytes(T, H, I, dtype) > 0 : stream_tc_bytes(T, H, I, E, k, dtype) > 0)
    return MM_PATH_STREAM_TC;
  if (stream_simt_bytes(T, H, I, E, k, dtype) > 0) return MM_PATH_STREAM;
  return MM_PATH_TENSOR;
}

}  // namespace

// Workspace of the path that AUTO (or `path`) resolves to for a dense call; 0
// when that path does not take the shape.  Used by the no-allocation entry.
size_t dense_workspace_for_path(int64_t T, int H, int I, int dtype, int path) {
  if (T < 1 || H < 1 || I < 1 || !valid_dtype(dtype)) return 0;
  return dense_path_bytes(T, H, I, dtype, resolve_path(path, dtype, T, H, I, 1, 1, true));
}

namespace {

inline char* ws_at(void* ws, size_t off) { return static_cast<char*>(ws) + off; }
inline float* f32_at(void* ws, size_t off) { return reinterpret_cast<float*>(ws_at(ws, off)); }

// ----------------------------------------------------------- measurement hooks
std::atomic<uint64_t> g_launches{0};

struct Profiler {
  std::mutex mu;
  int kernel = 0;
  int max = 0;
  int used = 0;
  std::vector<cudaEvent_t> start, stop;
};
Profiler g_prof;

// Runs `launch` (which enqueues one kernel on `st`), bracketed by timing
// events when that kernel is being profiled.
template <class F>
cudaError_t counted_launch(int kernel, cudaStream_t st, F&& launch) {
  cudaEvent_t a = nullptr, b = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_prof.mu);
    if (g_prof.kernel == kernel && g_prof.used < g_prof.max) {
      const int i = g_prof.used;
      if (i >= static_cast<int>(g_prof.start.size())) {
        cudaEvent_t e0, e1;
        if (cudaEventCreate(&e0) == cudaSuccess && cudaEventCreate(&e1) == cudaSuccess) {
          g_prof.start.push_back(e0);
          g_prof.stop.push_back(e1);
        }
      }
      if (i < static_cast<int>(g_prof.start.size())) {
        a = g_prof.start[i];
        b = g_prof.stop[i];
        ++g_prof.used;
      }
    }
  }
  if (a) cudaEventRecord(a, st);
  cudaError_t e = launch();
  if (b) cudaEventRecord(b, st);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return e;
}

}  // namespace
}  // namespace mm

using namespace mm;

extern "C" {

const char* mm_status_string(int status) {
  switch (status) {
    case MM_OK: return "MM_OK";
    case MM_ERR_INVALID_ARG: return "MM_ERR_INVALID_ARG";
    case MM_ERR_UNSUPPORTED: return "MM_ERR_UNSUPPORTED";
    case MM_ERR_WORKSPACE: return "MM_ERR_WORKSPACE";
    case MM_ERR_CUDA: return "MM_ERR_CUDA";
    case MM_ERR_TIMEOUT: return "MM_ERR_TIMEOUT";
    case MM_ERR_RANGE: return "MM_ERR_RANGE";
    default: return "MM_ERR_UNKNOWN";
  }
}

int mm_version(void) { return 100; }

const char* mm_last_error(void) { return g_last_error; }

size_t mm_swiglu_ffn_workspace_bytes(int64_t T, int H, int I, int dtype) {
  if (T < 0 || H < 1 || I < 1 || !valid_dtype(dtype)) return 0;
  return dense_ws_bytes(T, H, I, dtype);
}

static int swiglu_ffn_impl(const void* x, const void* Wg, const void* Wu, const void* Wd,
                           const void* Wd16, void* y, int64_t T, int H, int I, int dtype,
                           void* workspace, size_t workspace_bytes, void* stream, int path);

int mm_swiglu_ffn_ex(const void* x, const void* Wg, const void* Wu, const void* Wd, void* y,
                     int64_t T, int H, int I, int dtype, void* workspace, size_t workspace_bytes,
                     void* stream, int path) {
  return swiglu_ffn_impl(x, Wg, Wu, Wd, nullptr, y, T, H, I, dtype, workspace, workspace_bytes,
                         stream, path);
}

int mm_swiglu_ffn_prepared(const void* x, const void* Wg, const void* Wu, const void* Wd,
                           const void* Wd16, void* y, int64_t T, int H, int I, int dtype,
                           void* workspace, size_t workspace_bytes, void* stream, int path) {
  if (Wd16 != nullptr && !aligned16(Wd16)) return MM_ERR_INVALID_ARG;
  return swiglu_ffn_impl(x, Wg, Wu, Wd, Wd16, y, T, H, I, dtype, workspace, workspace_bytes,
                         stream, path);
}

static int swiglu_ffn_impl(const void* x, const void* Wg, const void* Wu, const void* Wd,
                           const void* Wd16, void* y, int64_t T, int H, int I, int dtype,
                           void* workspace, size_t workspace_bytes, void* stream, int path) {
  if (!valid_dtype(dtype) || T < 0 || H < 1 || I < 1) return MM_ERR_INVALID_ARG;
  if (H % 8 != 0 || I % 8 != 0) return MM_ERR_UNSUPPORTED;
  if (T > (int64_t{1} << 30)) return MM_ERR_UNSUPPORTED;
  if (path < MM_PATH_AUTO || path > MM_PATH_TENSOR_GATHER) return MM_ERR_INVALID_ARG;
  if (path == MM_PATH_TENSOR_GATHER) path = MM_PATH_TENSOR;   // nothing to gather in a dense FFN
  if (T == 0) return MM_OK;
  if (!x || !Wg || !Wu || !Wd || !y) return MM_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd) || !aligned16(y))
    return MM_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return MM_ERR_WORKSPACE;
  const int p = resolve_path(path, dtype, T, H, I, 1, 1, true);
  if (p == MM_PATH_TENSOR && (dtype != kDtypeBF16 || !tensor_shape_ok(H, I)))
    return MM_ERR_UNSUPPORTED;
  const size_t need = dense_path_bytes(T, H, I, dtype, p);
  if (need == 0) return MM_ERR_UNSUPPORTED;
  if (workspace_bytes < need) return MM_ERR_WORKSPACE;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(workspace);
  void* h = ws_at(workspace, sizeof(WsHeader));
  if (p == MM_PATH_STREAM || p == MM_PATH_STREAM_TC) {
    // scratch (fp32 h, or the tensor-core kernel's buffers) after the header
    const void* wg1[1] = {Wg};
    const void* wu1[1] = {Wu};
    const void* wd1[1] = {Wd};
    cudaError_t e = counted_launch(MM_KERNEL_DECODE, st, [&] {
      if (p == MM_PATH_STREAM)
        return launch_decode_ffn(x, nullptr, nullptr, wg1, wu1, wd1, static_cast<int>(T), H, I, 1,
                                 1, 0.f, nullptr, nullptr, nullptr, h, y, hdr, st);
      if (decode_sw_bytes(static_cast<int>(T), H, I) > 0)
        return launch_decode_sw(x, Wg, Wu, Wd, static_cast<int>(T), H, I, h, y, hdr, st);
      return launch_decode_tc(x, nullptr, nullptr, wg1, wu1, wd1, static_cast<int>(T), H, I, 1, 1,
                              0.f, nullptr, nullptr, nullptr, h, y, hdr, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "stream ffn");
    return MM_OK;
  }
  GroupRows g{nullptr, 1, static_cast<int>(T), 1};
  DownEpilogue ep{y, nullptr, nullptr, nullptr, 1, kCombineStore};
  const void* wg[1] = {Wg};
  const void* wu[1] = {Wu};
  const void* wd[1] = {Wd};
  cudaError_t e;
  if (p == MM_PATH_TENSOR) {
    // the gate/up kernel also makes the fp16 copy of Wd that the down GEMM
    // reads, unless the caller prepared one
    void* wd16 = ws_at(workspace, sizeof(WsHeader) + dense_h_bytes(T, I, dtype));
    const void* wd16p[1] = {Wd16 != nullptr ? Wd16 : wd16};
    e = counted_launch(MM_KERNEL_GATEUP, st, [&] {
      return launch_gateup_tc(x, T, H, I, g, wg, wu, h, wd, Wd16 != nullptr ? 0 : 1, wd16, hdr, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "gateup_tc");
    e = counted_launch(MM_KERNEL_DOWN, st, [&] { return launch_down_tc(h, T, H, I, g, wd16p, ep, hdr, st); });
    if (e != cudaSuccess) return cuda_fail(e, "down_tc");
  } else {
    e = counted_launch(MM_KERNEL_GATEUP, st, [&] { return launch_gateup_simt(dtype, x, T, H, I, g, wg, wu, h, st); });
    if (e != cudaSuccess) return cuda_fail(e, "gateup_simt");
    e = counted_launch(MM_KERNEL_DOWN, st, [&] { return launch_down_simt(dtype, h, T, H, I, g, wd, ep, st); });
    if (e != cudaSuccess) return cuda_fail(e, "down_simt");
  }
  return MM_OK;
}

int mm_swiglu_ffn(const void* x, const void* Wg, const void* Wu, const void* Wd, void* y,
                  int64_t T, int H, int I, int dtype, void* workspace, size_t workspace_bytes,
                  void* stream) {
  return mm_swiglu_ffn_ex(x, Wg, Wu, Wd, y, T, H, I, dtype, workspace, workspace_bytes, stream,
                          MM_PATH_AUTO);
}

size_t mm_moe_workspace_bytes_for_path(int64_t T, int H, int I, int E, int k, int dtype,
                                       int path) {
  if (T < 1 || H < 1 || I < 1 || E < 1 || E > MM_MAX_EXPERTS || k < 1 || k > E ||
      k > MM_MAX_TOPK || !valid_dtype(dtype) || path < MM_PATH_AUTO || path > MM_PATH_TENSOR_GATHER)
    return 0;
  if (path == MM_PATH_AUTO) return moe_ws_bytes(T, H, I, E, k, dtype);
  return moe_path_bytes(T, H, I, E, k, dtype, path);
}

size_t mm_moe_workspace_bytes(int64_t T, int H, int I, int E, int k, int dtype) {
  if (T < 1 || H < 1 || I < 1 || E < 1 || E > MM_MAX_EXPERTS || k < 1 || k > E ||
      !valid_dtype(dtype))
    return 0;
  if (k > MM_MAX_TOPK) return 0;
  return moe_ws_bytes(T, H, I, E, k, dtype);
}

static int check_route_args(const void* x, const void* Wr, int64_t T, int H, int E, int k,
                            int dtype, const float* logit_bias, const int32_t* topk_idx,
                            const float* topk_w, const float* aux_loss) {
  if (!valid_dtype(dtype) || T < 1 || H < 1 || E < 1 || k < 1 || k > E) return MM_ERR_INVALID_ARG;
  if (E > MM_MAX_EXPERTS || k > MM_MAX_TOPK) return MM_ERR_UNSUPPORTED;
  if (H % 8 != 0) return MM_ERR_UNSUPPORTED;
  if (router_smem_bytes(H, E, k) > 200 * 1024) return MM_ERR_UNSUPPORTED;
  if (T > (int64_t{1} << 30) / k) return MM_ERR_UNSUPPORTED;
  if (!x || !Wr || !topk_idx || !topk_w || !aux_loss) return MM_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(Wr)) return MM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(topk_idx) & 3u) || (reinterpret_cast<uintptr_t>(topk_w) & 3u) ||
      (reinterpret_cast<uintptr_t>(aux_loss) & 3u))
    return MM_ERR_INVALID_ARG;
  if (logit_bias && (reinterpret_cast<uintptr_t>(logit_bias) & 3u)) return MM_ERR_INVALID_ARG;
  return MM_OK;
}

// Router variants of an options struct as the kernels take them (the
// per-block z sums live in the workspace at blk_z).
static int router_variant(const mm_moe_options* o, void* blk_z, RouterVariant* rv) {
  memset(rv, 0, sizeof(*rv));
  if (o == nullptr) return MM_OK;
  auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!a4(o->logit_noise) || !a4(o->z_loss) || !a4(o->router_probs) || !a4(o->router_lse))
    return MM_ERR_INVALID_ARG;
  rv->noise = o->logit_noise;
  rv->z_coef = o->z_coef;
  rv->z_loss = o->z_loss;
  rv->probs = o->router_probs;
  rv->lse = o->router_lse;
  rv->blk_z = o->z_loss != nullptr ? static_cast<float*>(blk_z) : nullptr;
  return MM_OK;
}

static int moe_forward_impl(const void* x, const void* Wr, const void* const* Wg,
                            const void* const* Wu, const void* const* Wd, int64_t T, int H, int I,
                            int E, int k, float coef, int dtype, const float* logit_bias, void* y,
                            int32_t* topk_idx, float* topk_w, float* aux_loss, void* workspace,
                            size_t workspace_bytes, void* stream, const mm_moe_options* opts) {
  int path = opts ? opts->path : MM_PATH_AUTO;
  const void* norm_w = opts ? opts->norm_weight : nullptr;
  const bool resid = opts && opts->residual;
  int rc = check_route_args(x, Wr, T, H, E, k, dtype, logit_bias, topk_idx, topk_w, aux_loss);
  if (rc != MM_OK) return rc;
  if (norm_w != nullptr || resid) {
    // the block prologue / epilogue live in the router, dispatch and down
    // kernels: the tensor-core or CUDA-core GEMM paths, not the streaming ones
    if (path == MM_PATH_STREAM || path == MM_PATH_STREAM_TC) return MM_ERR_UNSUPPORTED;
    if (path == MM_PATH_AUTO) path = dtype == kDtypeBF16 ? MM_PATH_TENSOR : MM_PATH_SIMT;
    if (norm_w != nullptr && (!aligned16(norm_w) || !(opts->norm_eps >= 0.f))) return MM_ERR_INVALID_ARG;
    if (resid && y == x) return MM_ERR_INVALID_ARG;   // x is read as the residual while y is written
  }
  if (I < 1) return MM_ERR_INVALID_ARG;
  if (I % 8 != 0) return MM_ERR_UNSUPPORTED;
  if (path < MM_PATH_AUTO || path > MM_PATH_TENSOR_GATHER) return MM_ERR_INVALID_ARG;
  // gathering x rows needs them as the layer's input: with the block norm the
  // dispatch writes normalised rows instead
  bool gather = path == MM_PATH_TENSOR_GATHER;
  if (gather) {
    if (dtype != kDtypeBF16) return MM_ERR_UNSUPPORTED;
    path = MM_PATH_TENSOR;
    if (norm_w != nullptr) gather = false;
  }
  if (!Wg || !Wu || !Wd || !y || !aligned16(y)) return MM_ERR_INVALID_ARG;
  for (int e = 0; e < E; ++e) {
    if (!Wg[e] || !Wu[e] || !Wd[e]) return MM_ERR_INVALID_ARG;
    if (!aligned16(Wg[e]) || !aligned16(Wu[e]) || !aligned16(Wd[e])) return MM_ERR_INVALID_ARG;
  }
  if (!workspace || !aligned16(workspace)) return MM_ERR_WORKSPACE;
  const int p = resolve_path(path, dtype, T, H, I, E, k, false);
  if (p == MM_PATH_TENSOR && (dtype != kDtypeBF16 || !tensor_shape_ok(H, I)))
    return MM_ERR_UNSUPPORTED;
  const size_t need = moe_path_bytes(T, H, I, E, k, dtype, gather ? MM_PATH_TENSOR_GATHER : p);
  if (need == 0) return MM_ERR_UNSUPPORTED;
  if (workspace_bytes < need) return MM_ERR_WORKSPACE;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(workspace);
  if (p == MM_PATH_STREAM || p == MM_PATH_STREAM_TC) {
    // decode-sized: routing, experts and combine in one streaming kernel,
    // with its scratch after the header
    void* scratch = ws_at(workspace, sizeof(WsHeader));
    RouterVariant rv;
    rc = router_variant(opts, nullptr, &rv);
    if (rc != MM_OK) return rc;
    cudaError_t e = counted_launch(MM_KERNEL_DECODE, st, [&] {
      if (p == MM_PATH_STREAM)
        return launch_decode_ffn(x, Wr, logit_bias, Wg, Wu, Wd, static_cast<int>(T), H, I, E, k,
                                 coef, topk_idx, topk_w, aux_loss, scratch, y, hdr, st, &rv);
      return launch_decode_tc(x, Wr, logit_bias, Wg, Wu, Wd, static_cast<int>(T), H, I, E, k,
                              coef, topk_idx, topk_w, aux_loss, scratch, y, hdr, st, &rv);
    });
    if (e != cudaSuccess) return cuda_fail(e, "decode ffn");
    return MM_OK;
  }
  const MoeLayout L = moe_layout(T, H, I, E, k, dtype, !gather);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws_at(workspace, L.offsets));
  int32_t* counts = reinterpret_cast<int32_t*>(ws_at(workspace, L.counts));
  int32_t* blk_cnt = reinterpret_cast<int32_t*>(ws_at(workspace, L.blk_cnt));
  float* blk_prob = reinterpret_cast<float*>(ws_at(workspace, L.blk_prob));
  int32_t* perm = reinterpret_cast<int32_t*>(ws_at(workspace, L.perm));
  void* xp = ws_at(workspace, L.xp);
  void* h = ws_at(workspace, L.h);
  float* acc32 = (dtype == kDtypeF32) ? static_cast<float*>(y)
                                      : reinterpret_cast<float*>(ws_at(workspace, L.acc32));

  const int64_t rows = T * k;
  const void* wd16p[MM_MAX_EXPERTS];
  char* wd16 = ws_at(workspace, L.wd16);
  const void* const* prep = opts ? opts->wd_f16 : nullptr;   // prepared fp16 down weights
  if (prep != nullptr)
    for (int q = 0; q < E; ++q)
      if (prep[q] == nullptr || !aligned16(prep[q])) return MM_ERR_INVALID_ARG;
  if (p == MM_PATH_TENSOR)
    for (int q = 0; q < E; ++q)
      wd16p[q] = prep != nullptr ? prep[q] : wd16 + static_cast<size_t>(q) * H * I * 2;
  RouterVariant rv;
  rc = router_variant(opts, ws_at(workspace, L.blk_z), &rv);
  if (rc != MM_OK) return rc;
  BlockNorm nrm{norm_w, norm_w ? opts->norm_eps : 0.f, f32_at(workspace, L.inv_rms),
                ws_at(workspace, L.wr_hl)};
  if (norm_w != nullptr && dtype == kDtypeBF16) {
    // w folded into the router weights (exact bf16 halves) for the tensor-core router
    cudaError_t e0 = counted_launch(MM_KERNEL_ROUTER, st, [&] {
      return launch_norm_fold_router(Wr, norm_w, E, H, ws_at(workspace, L.wr_hl), st);
    });
    if (e0 != cudaSuccess) return cuda_fail(e0, "norm fold");
  }
  const RouteOut ro{nullptr, nullptr, nullptr, nullptr, coef, 0, rv, nrm};
  const DispatchOut dout{offsets, counts, aux_loss, coef, hdr, rv, nrm};
  // router and permute in one kernel where every block fits on the GPU at once
  // (x read once); otherwise the router grid, then the dispatch grid
  cudaError_t e;
  const bool separate = opts != nullptr && opts->separate_routing != 0;
  if (!separate && route_dispatch_ok(dtype, x, Wr, T, H, E, k, dout)) {
    e = counted_launch(MM_KERNEL_ROUTER, st, [&] {
      return launch_route_dispatch(dtype, x, Wr, logit_bias, T, H, E, k, topk_idx, topk_w,
                                   blk_cnt, blk_prob, dout, perm, gather ? nullptr : xp, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "router + dispatch");
  } else {
    e = counted_launch(MM_KERNEL_ROUTER, st, [&] {
      return launch_router(dtype, x, Wr, logit_bias, T, H, E, k, topk_idx, topk_w, blk_cnt,
                           blk_prob, ro, hdr, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "router");
    e = counted_launch(MM_KERNEL_DISPATCH, st, [&] {
      return launch_dispatch(dtype, x, T, H, E, k, topk_idx, blk_cnt, blk_prob, dout, perm,
                             gather ? nullptr : xp, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "dispatch");
  }

  // gate/up over all k*E (slot, expert) groups at once; on the tensor path
  // the same kernel makes the fp16 copy of Wd that the down GEMM reads, with
  // its epilogue warps while the tensor pipe runs (HBM is mostly idle then)
  GroupRows gu{offsets, k * E, 0, E};
  const RowGather rg{perm, k, static_cast<int>(rows)};
  if (p == MM_PATH_TENSOR)
    e = counted_launch(MM_KERNEL_GATEUP, st, [&] {
      return launch_gateup_tc(gather ? x : xp, rows, H, I, gu, Wg, Wu, h, Wd,
                              prep != nullptr ? 0 : E, wd16, hdr, st, gather ? &rg : nullptr);
    });
  else
    e = counted_launch(MM_KERNEL_GATEUP, st, [&] {
      return launch_gateup_simt(dtype, xp, rows, H, I, gu, Wg, Wu, h, st);
    });
  if (e != cudaSuccess) return cuda_fail(e, "gateup");
  // down: one phase per slot; the k contributions of a token are summed in
  // fp32 in slot order and rounded once
  for (int s = 0; s < k; ++s) {
    GroupRows gd{offsets + static_cast<size_t>(s) * E, E, 0, E};
    DownEpilogue ep{y, acc32, perm, topk_w, k,
                    k == 1 ? kCombineStore
                           : (s == 0 ? kCombineFirst : (s == k - 1 ? kCombineLast : kCombineAccum)),
                    resid ? x : nullptr};
    if (p == MM_PATH_TENSOR)
      e = counted_launch(MM_KERNEL_DOWN, st, [&] {
        return launch_down_tc(h, rows, H, I, gd, wd16p, ep, hdr, st);
      });
    else
      e = counted_launch(MM_KERNEL_DOWN, st, [&] {
        return launch_down_simt(dtype, h, rows, H, I, gd, Wd, ep, st);
      });
    if (e != cudaSuccess) return cuda_fail(e, "down");
  }
  return MM_OK;
}

int mm_moe_forward_ex(const void* x, const void* Wr, const void* const* Wg,
                      const void* const* Wu, const void* const* Wd, int64_t T, int H, int I, int E,
                      int k, float coef, int dtype, const float* logit_bias, void* y,
                      int32_t* topk_idx, float* topk_w, float* aux_loss, void* workspace,
                      size_t workspace_bytes, void* stream, int path) {
  mm_moe_options o;
  memset(&o, 0, sizeof(o));
  o.path = path;
  return moe_forward_impl(x, Wr, Wg, Wu, Wd, T, H, I, E, k, coef, dtype, logit_bias, y, topk_idx,
                          topk_w, aux_loss, workspace, workspace_bytes, stream, &o);
}

int mm_moe_forward_opts(const void* x, const void* Wr, const void* const* Wg,
                        const void* const* Wu, const void* const* Wd, int64_t T, int H, int I,
                        int E, int k, float coef, int dtype, const float* logit_bias, void* y,
                        int32_t* topk_idx, float* topk_w, float* aux_loss, void* workspace,
                        size_t workspace_bytes, void* stream, const mm_moe_options* opts) {
  return moe_forward_impl(x, Wr, Wg, Wu, Wd, T, H, I, E, k, coef, dtype, logit_bias, y, topk_idx,
                          topk_w, aux_loss, workspace, workspace_bytes, stream, opts);
}

int mm_moe_forward(const void* x, const void* Wr, const void* const* Wg, const void* const* Wu,
                   const void* const* Wd, int64_t T, int H, int I, int E, int k, float coef,
                   int dtype, const float* logit_bias, void* y, int32_t* topk_idx, float* topk_w,
                   float* aux_loss, void* workspace, size_t workspace_bytes, void* stream) {
  return mm_moe_forward_ex(x, Wr, Wg, Wu, Wd, T, H, I, E, k, coef, dtype, logit_bias, y, topk_idx,
                           topk_w, aux_loss, workspace, workspace_bytes, stream, MM_PATH_AUTO);
}

size_t mm_moe_route_workspace_bytes(int64_t T, int E, int k) {
  if (T < 1 || E < 1 || E > MM_MAX_EXPERTS || k < 1 || k > E || k > MM_MAX_TOPK) return 0;
  return route_layout(T, E, k).total;
}

int mm_moe_route(const void* x, const void* Wr, int64_t T, int H, int E, int k, float coef,
                 int dtype, const float* logit_bias, int32_t* topk_idx, float* topk_w,
                 float* aux_loss, int32_t* expert_counts, void* workspace, size_t workspace_bytes,
                 void* stream) {
  return mm_moe_route_opts(x, Wr, T, H, E, k, coef, dtype, logit_bias, topk_idx, topk_w, aux_loss,
                           expert_counts, workspace, workspace_bytes, stream, nullptr);
}

int mm_moe_route_opts(const void* x, const void* Wr, int64_t T, int H, int E, int k, float coef,
                      int dtype, const float* logit_bias, int32_t* topk_idx, float* topk_w,
                      float* aux_loss, int32_t* expert_counts, void* workspace,
                      size_t workspace_bytes, void* stream, const mm_moe_options* opts) {
  int rc = check_route_args(x, Wr, T, H, E, k, dtype, logit_bias, topk_idx, topk_w, aux_loss);
  if (rc != MM_OK) return rc;
  if (expert_counts && (reinterpret_cast<uintptr_t>(expert_counts) & 3u)) return MM_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return MM_ERR_WORKSPACE;
  const RouteLayout L = route_layout(T, E, k);
  if (workspace_bytes < L.total) return MM_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* blk_cnt = reinterpret_cast<int32_t*>(ws_at(workspace, L.blk_cnt));
  float* blk_prob = reinterpret_cast<float*>(ws_at(workspace, L.blk_prob));
  WsHeader* hdr = reinterpret_cast<WsHeader*>(workspace);
  RouterVariant rv;
  rc = router_variant(opts, ws_at(workspace, L.blk_z), &rv);
  if (rc != MM_OK) return rc;
  const RouteOut ro{nullptr, nullptr, expert_counts, aux_loss, coef, 1, rv, BlockNorm{}};
  cudaError_t e = counted_launch(MM_KERNEL_ROUTER, st, [&] {
    return launch_router(dtype, x, Wr, logit_bias, T, H, E, k, topk_idx, topk_w, blk_cnt, blk_prob,
                         ro, hdr, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "router");
  return MM_OK;
}

// ------------------------------------------------------------------ prepared weights
int mm_prepare_down_weights(const void* Wd, void* Wd16, int H, int I, void* status_ws,
                            void* stream) {
  if (!Wd || !Wd16 || H < 1 || I < 1) return MM_ERR_INVALID_ARG;
  if (!aligned16(Wd) || !aligned16(Wd16) || (status_ws && !aligned16(status_ws)))
    return MM_ERR_INVALID_ARG;
  const int64_t n = static_cast<int64_t>(H) * I;
  if (n % 8 != 0) return MM_ERR_UNSUPPORTED;
  cudaError_t e = launch_prepare_wd16(Wd, Wd16, n, static_cast<WsHeader*>(status_ws),
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prepare Wd");
  return MM_OK;
}

// ------------------------------------------------------------------ dense block
size_t mm_swiglu_ffn_block_workspace_bytes(int64_t T, int H, int I, int dtype) {
  if (T < 0 || H < 1 || I < 1 || !valid_dtype(dtype)) return 0;
  return dense_block_ws_bytes(T, H, I, dtype);
}

int mm_swiglu_ffn_block(const void* x, const void* norm_w, float norm_eps, const void* Wg,
                        const void* Wu, const void* Wd, void* y, int64_t T, int H, int I,
                        int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_dtype(dtype) || T < 0 || H < 1 || I < 1 || !(norm_eps >= 0.f)) return MM_ERR_INVALID_ARG;
  if (H % 8 != 0 || I % 8 != 0) return MM_ERR_UNSUPPORTED;
  if (dtype == kDtypeBF16 && !tensor_shape_ok(H, I)) return MM_ERR_UNSUPPORTED;
  if (T > (int64_t{1} << 30)) return MM_ERR_UNSUPPORTED;
  if (T == 0) return MM_OK;
  if (!x || !norm_w || !Wg || !Wu || !Wd || !y) return MM_ERR_INVALID_ARG;
  const void* ptrs[] = {x, norm_w, Wg, Wu, Wd, y};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MM_ERR_INVALID_ARG;
  if (y == x) return MM_ERR_INVALID_ARG;            // the residual is read while y is written
  if (!workspace || !aligned16(workspace)) return MM_ERR_WORKSPACE;
  const size_t need = dense_block_ws_bytes(T, H, I, dtype);
  if (workspace_bytes < need) return MM_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(workspace);
  const size_t base = dense_tensor_ws_bytes(T, H, I, dtype);
  void* xn = ws_at(workspace, base);
  float* inv = f32_at(workspace, base + align_up(elem_bytes(dtype) * static_cast<size_t>(T) * H));
  // prologue: the normalised rows (the GEMMs read their A operand by TMA)
  cudaError_t e = counted_launch(MM_KERNEL_DISPATCH, st, [&] {
    return launch_rms_norm_rows(dtype, x, norm_w, norm_eps, T, H, xn, inv, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "rms norm");
  void* h = ws_at(workspace, sizeof(WsHeader));
  GroupRows g{nullptr, 1, static_cast<int>(T), 1};
  DownEpilogue ep{y, nullptr, nullptr, nullptr, 1, kCombineStore, x};   // + the residual
  const void* wg[1] = {Wg};
  const void* wu[1] = {Wu};
  const void* wd[1] = {Wd};
  if (dtype == kDtypeBF16) {
    void* wd16 = ws_at(workspace, sizeof(WsHeader) + dense_h_bytes(T, I, dtype));
    const void* wd16p[1] = {wd16};
    e = counted_launch(MM_KERNEL_GATEUP, st, [&] {
      return launch_gateup_tc(xn, T, H, I, g, wg, wu, h, wd, 1, wd16, hdr, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "gateup_tc");
    e = counted_launch(MM_KERNEL_DOWN, st, [&] { return launch_down_tc(h, T, H, I, g, wd16p, ep, hdr, st); });
    if (e != cudaSuccess) return cuda_fail(e, "down_tc");
  } else {
    e = counted_launch(MM_KERNEL_GATEUP, st, [&] { return launch_gateup_simt(dtype, xn, T, H, I, g, wg, wu, h, st); });
    if (e != cudaSuccess) return cuda_fail(e, "gateup_simt");
    e = counted_launch(MM_KERNEL_DOWN, st, [&] { return launch_down_simt(dtype, h, T, H, I, g, wd, ep, st); });
    if (e != cudaSuccess) return cuda_fail(e, "down_simt");
  }
  return MM_OK;
}

// ------------------------------------------------------------------ backward
size_t mm_swiglu_ffn_backward_workspace_bytes(int64_t T, int H, int I, int dtype) {
  if (T < 0 || H < 1 || I < 1 || dtype != kDtypeBF16) return 0;
  return dense_bwd_layout(T, I).total;
}

static bool bwd_shape_ok(int H, int I) { return H % 64 == 0 && I % 64 == 0; }

int mm_swiglu_ffn_backward(const void* x, const void* Wg, const void* Wu, const void* Wd,
                           const void* dy, int64_t T, int H, int I, int dtype, void* dx,
                           float* dWg, float* dWu, float* dWd, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (!valid_dtype(dtype) || T < 0 || H < 1 || I < 1) return MM_ERR_INVALID_ARG;
  if (dtype != kDtypeBF16 || !bwd_shape_ok(H, I)) return MM_ERR_UNSUPPORTED;
  if (T > (int64_t{1} << 30)) return MM_ERR_UNSUPPORTED;
  if (!x || !Wg || !Wu || !Wd || !dy || !dx || !dWg || !dWu || !dWd) return MM_ERR_INVALID_ARG;
  const void* ptrs[] = {x, Wg, Wu, Wd, dy, dx, dWg, dWu, dWd};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MM_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return MM_ERR_WORKSPACE;
  const DenseBwdLayout L = dense_bwd_layout(T, I);
  if (workspace_bytes < L.total) return MM_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(workspace);
  if (T == 0) {
    // no tokens: the weight gradients are zero
    const size_t wb = 4 * static_cast<size_t>(H) * I;
    for (float* q : {dWg, dWu, dWd}) {
      cudaError_t e = cudaMemsetAsync(q, 0, wb, st);
      if (e != cudaSuccess) return cuda_fail(e, "zero dW");
    }
    return MM_OK;
  }
  void* dh = ws_at(workspace, L.dh);
  void* dgu = ws_at(workspace, L.dgu);
  void* h = ws_at(workspace, L.h);
  const int Ti = static_cast<int>(T);
  // dh = dy Wd
  const void* wd1[1] = {Wd};
  cudaError_t e = counted_launch(MM_KERNEL_BWD_DGRAD, st, [&] {
    return launch_bw_dgrad(dy, T, H, nullptr, 1, Ti, wd1, wd1, H / 64, I, dh, I, kBwOutF16, hdr, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "bwd dh");
  // g, u again; dG, dU, h
  const void* wg1[1] = {Wg};
  const void* wu1[1] = {Wu};
  UpBwd ub{static_cast<const __half*>(dh), nullptr, nullptr,
           static_cast<__nv_bfloat16*>(dgu), static_cast<__nv_bfloat16*>(h), nullptr, 0};
  GroupRows gr{nullptr, 1, Ti, 1};
  e = counted_launch(MM_KERNEL_BWD_SWIGLU, st, [&] {
    return launch_gateup_bwd_tc(x, T, H, I, gr, wg1, wu1, ub, hdr, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "bwd swiglu");
  // dx = dG Wg + dU Wu
  e = counted_launch(MM_KERNEL_BWD_DGRAD, st, [&] {
    return launch_bw_dgrad(dgu, T, 2 * I, nullptr, 1, Ti, wg1, wu1, I / 64, H, dx, H, kBwOutBF16, hdr, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "bwd dx");
  // dWd = dy^T h, dWg = dG^T x, dWu = dU^T x
  const void* am[2] = {dy, dgu};
  const int64_t ac[2] = {H, 2 * static_cast<int64_t>(I)};
  const void* bm[2] = {h, x};
  const int64_t bc[2] = {I, H};
  const BwProblem pr[3] = {{dWd, H, I, 0, 0, 0, 0}, {dWg, I, H, 0, 1, 1, 0}, {dWu, I, H, 0, 1, 1, I}};
  e = counted_launch(MM_KERNEL_BWD_WGRAD, st, [&] {
    return launch_bw_wgrad(am, ac, 2, bm, bc, 2, T, pr, 3, nullptr, 1, Ti, hdr, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "bwd wgrad");
  return MM_OK;
}

size_t mm_moe_backward_workspace_bytes(int64_t T, int H, int I, int E, int k, int dtype) {
  if (T < 1 || H < 1 || I < 1 || E < 1 || E > MM_MAX_EXPERTS || k < 1 || k > E ||
      k > MM_MAX_TOPK || dtype != kDtypeBF16)
    return 0;
  return moe_bwd_layout(T, H, I, E, k).total;
}

int mm_moe_backward(const void* x, const void* Wr, const void* const* Wg, const void* const* Wu,
                    const void* const* Wd, int64_t T, int H, int I, int E, int k, float coef,
                    int dtype, const int32_t* topk_idx, const float* topk_w,
                    const float* router_probs, const float* router_lse, const void* dy,
                    float d_aux, float z_coef, float d_z, void* dx, float* dWr,
                    float* const* dWg, float* const* dWu, float* const* dWd, float* d_bias,
                    void* workspace, size_t workspace_bytes, void* stream) {
  if (!valid_dtype(dtype) || T < 1 || H < 1 || I < 1 || E < 1 || k < 1 || k > E)
    return MM_ERR_INVALID_ARG;
  if (E > MM_MAX_EXPERTS || k > MM_MAX_TOPK) return MM_ERR_UNSUPPORTED;
  if (dtype != kDtypeBF16 || !bwd_shape_ok(H, I)) return MM_ERR_UNSUPPORTED;
  if (T > (int64_t{1} << 30) / k) return MM_ERR_UNSUPPORTED;
  if (!x || !Wr || !Wg || !Wu || !Wd || !topk_idx || !topk_w || !router_probs || !dy || !dx ||
      !dWr || !dWg || !dWu || !dWd)
    return MM_ERR_INVALID_ARG;
  if (z_coef != 0.f && d_z != 0.f && router_lse == nullptr) return MM_ERR_INVALID_ARG;
  const void* ptrs[] = {x, Wr, dy, dx, dWr};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MM_ERR_INVALID_ARG;
  for (int e = 0; e < E; ++e) {
    const void* w[] = {Wg[e], Wu[e], Wd[e], dWg[e], dWu[e], dWd[e]};
    for (const void* q : w)
      if (!q || !aligned16(q)) return MM_ERR_INVALID_ARG;
  }
  auto a4 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 3u) == 0; };
  if (!a4(topk_idx) || !a4(topk_w) || !a4(router_probs) || !a4(router_lse) || !a4(d_bias))
    return MM_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace)) return MM_ERR_WORKSPACE;
  const MoeBwdLayout L = moe_bwd_layout(T, H, I, E, k);
  if (workspace_bytes < L.total) return MM_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(workspace);
  auto i32 = [&](size_t off) { return reinterpret_cast<int32_t*>(ws_at(workspace, off)); };
  auto f32 = [&](size_t off) { return reinterpret_cast<float*>(ws_at(workspace, off)); };
  int32_t* offsets = i32(L.offsets);
  void* xp = ws_at(workspace, L.xp);
  void* dyp = ws_at(workspace, L.dyp);
  void* dhu = ws_at(workspace, L.dhu);
  void* dgu = ws_at(workspace, L.dgu);
  void* ha = ws_at(workspace, L.ha);
  const int nblk = route_blocks(T);
  const int64_t R = L.rows;

  // 1. group the assignments by expert (padded), gather x and dy rows
  cudaError_t e = counted_launch(MM_KERNEL_BWD_ROUTER, st, [&] {
    return launch_bwd_count(topk_idx, T, E, k, i32(L.blk_cnt), st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "bwd count");
  const BwdDispatchOut dout{offsets, i32(L.counts), i32(L.perm), i32(L.pos), xp, dyp, hdr};
  e = counted_launch(MM_KERNEL_BWD_ROUTER, st, [&] {
    return launch_bwd_dispatch(x, dy, topk_idx, T, H, E, k, i32(L.blk_cnt), dout, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "bwd dispatch");
  // 2. dhu = dy Wd_e (unscaled by alpha), per expert group
  e = counted_launch(MM_KERNEL_BWD_DGRAD, st, [&] {
    return launch_bw_dgrad(dyp, R, H, offsets, E, 0, Wd, Wd, H / 64, I, dhu, I, kBwOutF16, hdr, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "bwd dhu");
  // 3. g, u again: dG, dU, alpha h, dalpha partials
  const UpBwd ub{static_cast<const __half*>(dhu), i32(L.perm), topk_w,
                 static_cast<__nv_bfloat16*>(dgu), static_cast<__nv_bfloat16*>(ha), f32(L.dpart),
                 L.n_parts};
  const GroupRows gr{offsets, E, 0, E};
  e = counted_launch(MM_KERNEL_BWD_SWIGLU, st, [&] {
    return launch_gateup_bwd_tc(xp, R, H, I, gr, Wg, Wu, ub, hdr, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "bwd swiglu");
  // 4. per-assignment dx rows (fp16, range-checked) = dG Wg_e + dU Wu_e
  e = counted_launch(MM_KERNEL_BWD_DGRAD, st, [&] {
    return launch_bw_dgrad(dgu, R, 2 * I, offsets, E, 0, Wg, Wu, I / 64, H, ws_at(workspace, L.dxp), H,
                           kBwOutF16, hdr, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "bwd dxp");
  // 5. weight gradients over each expert's rows
  const void* am[2] = {dyp, dgu};
  const int64_t ac[2] = {H, 2 * static_cast<int64_t>(I)};
  const void* bm[2] = {ha, xp};
  const int64_t bc[2] = {I, H};
  BwProblem pr[kBwMaxGroups];
  for (int q = 0; q < E; ++q) {
    pr[3 * q + 0] = BwProblem{dWd[q], H, I, q, 0, 0, 0};
    pr[3 * q + 1] = BwProblem{dWg[q], I, H, q, 1, 1, 0};
    pr[3 * q + 2] = BwProblem{dWu[q], I, H, q, 1, 1, I};
  }
  e = counted_launch(MM_KERNEL_BWD_WGRAD, st, [&] {
    return launch_bw_wgrad(am, ac, 2, bm, bc, 2, R, pr, 3 * E, offsets, E, 0, hdr, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "bwd wgrad");
  // 6. router: dr, dx (slot-ordered sum + dr Wr), dWr / d_bias partials, then their sums
  const RouterBwd rb{topk_idx, topk_w, router_probs, (z_coef != 0.f && d_z != 0.f) ? router_lse : nullptr,
                     i32(L.counts), i32(L.pos), f32(L.dpart), L.n_parts,
                     reinterpret_cast<const __half*>(ws_at(workspace, L.dxp)), coef, d_aux,
                     z_coef, d_z, f32(L.dr), dx, f32(L.dwr_part), f32(L.dbias_part)};
  e = counted_launch(MM_KERNEL_BWD_ROUTER, st, [&] {
    return launch_router_bwd(x, Wr, T, H, E, k, rb, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "bwd router");
  e = counted_launch(MM_KERNEL_BWD_ROUTER, st, [&] {
    return launch_router_bwd_reduce(f32(L.dwr_part), f32(L.dbias_part), nblk, E, H, dWr, d_bias, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "bwd router reduce");
  return MM_OK;
}

uint64_t mm_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int mm_profile_start(int kernel_id, int max_launches) {
  switch (kernel_id) {
    case MM_KERNEL_ROUTER: case MM_KERNEL_DISPATCH: case MM_KERNEL_GATEUP: case MM_KERNEL_DOWN:
    case MM_KERNEL_DECODE: case MM_KERNEL_BWD_DGRAD: case MM_KERNEL_BWD_SWIGLU:
    case MM_KERNEL_BWD_WGRAD: case MM_KERNEL_BWD_ROUTER: break;
    default: return MM_ERR_INVALID_ARG;
  }
  if (max_launches < 1 || max_launches > 100000) return MM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_prof.mu);
  g_prof.kernel = kernel_id;
  g_prof.max = max_launches;
  g_prof.used = 0;
  return MM_OK;
}

int mm_profile_stop(double* total_ms, int* launches) {
  std::lock_guard<std::mutex> lock(g_prof.mu);
  double sum = 0.0;
  int n = g_prof.used;
  for (int i = 0; i < n; ++i) {
    cudaError_t e = cudaEventSynchronize(g_prof.stop[i]);
    if (e != cudaSuccess) return cuda_fail(e, "profile sync");
    float ms = 0.f;
    e = cudaEventElapsedTime(&ms, g_prof.start[i], g_prof.stop[i]);
    if (e != cudaSuccess) return cuda_fail(e, "profile elapsed");
    sum += ms;
  }
  g_prof.kernel = 0;
  g_prof.used = 0;
  if (total_ms) *total_ms = sum;
  if (launches) *launches = n;
  return MM_OK;
}

int mm_check_status(void* workspace, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream");
  if (workspace == nullptr) return MM_OK;
  unsigned int word = 0;
  e = cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (word != 0) {
    e = cudaMemset(workspace, 0, sizeof(WsHeader));
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
    return static_cast<int>(word);
  }
  return MM_OK;
}

int mm_watchdog_selftest(void* workspace, size_t workspace_bytes, uint32_t limit_us, void* stream) {
  if (!workspace || workspace_bytes < sizeof(WsHeader) || !aligned16(workspace))
    return MM_ERR_WORKSPACE;
  if (limit_us < 1 || limit_us > 10000000u) return MM_ERR_INVALID_ARG;
  cudaError_t e = launch_watchdog_selftest(reinterpret_cast<WsHeader*>(workspace), limit_us,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "watchdog_selftest");
  return MM_OK;
}

}  // extern "C"
