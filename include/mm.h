/*
 * mm.h — C ABI of the GB300 (sm_103a) SwiGLU FFN and top-k MoE forward.
 *
 * The operations follow the MiniMind pages on the FFN / MoE sub-layer:
 *   [L13] MiniMind course, lesson 13 "FFN 与 MoE" (course/13_ffn_and_moe.md),
 *         §0 / §1.2 (SwiGLU equations), §1.5 (router, softmax, top-k, alpha),
 *         §1.6 (load-balancing aux loss), §3 steps 3-6 (module forward).
 *   [CH4] minimind3.com, chapter 4 "前馈网络 MLP & MoE", §4.2 (SwiGLU),
 *         §4.3 (MoE routing, renormalisation, dispatch), §4.4 (aux loss).
 *
 * Conventions shared by every entry point:
 *   - All tensors are dense, row-major, in DEVICE memory owned by the caller,
 *     and 16-byte aligned.  Weights use the nn.Linear layout [out, in]:
 *       Wg, Wu: [I, H]   Wd: [H, I]   Wr: [E, H]   x, y: [T, H].
 *   - dtype selects the element type of x, the weights and y:
 *       MM_DTYPE_BF16 — bf16 storage, fp32 accumulation (tcgen05 tensor
 *                       cores; for T <= 128 (dense FFN) or T <= 64 (MoE)
 *                       one weight-streaming kernel that reads every
 *                       needed weight row once);
 *       MM_DTYPE_F32  — fp32 storage and fp32 SIMT arithmetic (no TF32).
 *     Router logits, probabilities, alpha and the aux loss are always fp32.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call only enqueues work on that stream and returns; none synchronises
 *     the host except mm_check_status().  No call allocates device memory:
 *     scratch lives in the caller's `workspace`, whose size the matching
 *     *_workspace_bytes() function returns.  The one exception is a fixed
 *     array of MM_NOALLOC_SCRATCH_BYTES that the library's module reserves
 *     on every GPU where it is loaded (used only by mm_swiglu_ffn_noalloc).
 *     Calls that share a workspace must be ordered on one stream.  The first 256 bytes of a
 *     workspace hold device-side state (the watchdog word and the counter of
 *     the streaming kernel's grid barrier): zero them once before the
 *     workspace's first use (cudaMemset).  Every call leaves them consistent,
 *     and mm_check_status() zeroes them again after it reports a timeout.
 *   - Argument errors are reported synchronously as a non-zero mm_status
 *     with nothing enqueued.  Device-side watchdog failures (a pipeline wait
 *     that exceeded its time limit) are recorded in the workspace and
 *     reported by mm_check_status().
 *   - The library keeps only a host-side cache of TMA tensor maps keyed by
 *     (device pointer, shape); it is safe to call from one host thread at a
 *     time per process.
 */
#ifndef MM_H_
#define MM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MM_OK = 0,
  MM_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, k > E, ... */
  MM_ERR_UNSUPPORTED = 2,   /* valid but outside this build's limits          */
  MM_ERR_WORKSPACE = 3,     /* workspace null or smaller than required        */
  MM_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed              */
  MM_ERR_TIMEOUT = 5,       /* a device pipeline wait hit its time limit      */
  MM_ERR_RANGE = 6          /* bf16 tensor-core paths: a value of h, or of Wd
                               (forward), or of dh = dy Wd (backward), is
                               beyond the fp16 range (|v| >= 65520) of its
                               intermediate copy; the results may hold
                               inf/NaN.  Recorded on the device, reported by
                               mm_check_status()                              */
} mm_status;

typedef enum { MM_DTYPE_F32 = 0, MM_DTYPE_BF16 = 1 } mm_dtype;

/* Which kernels carry the FFN part of a call (the *_ex entry points). */
typedef enum {
  MM_PATH_AUTO = 0,    /* bf16: streaming up to 128 (dense) / 64 (MoE) tokens, tensor-core GEMMs beyond; f32: SIMT */
  MM_PATH_TENSOR = 1,  /* bf16 only: grouped tcgen05/TMEM GEMMs fed by TMA          */
  MM_PATH_STREAM = 2,  /* bf16 only, T <= 16: weight streaming on the CUDA cores       */
  MM_PATH_SIMT = 3,    /* any dtype: plain fp32-FMA CUDA-core kernels                */
  MM_PATH_STREAM_TC = 4, /* bf16 only, T <= 128 dense / 64 MoE: weight streaming on the tensor cores */
  MM_PATH_TENSOR_GATHER = 5 /* bf16 MoE only: as MM_PATH_TENSOR, but the gate/up GEMM gathers x
                               rows by token index (TMA gather4) and no permuted copy of x
                               is made (a dense FFN call takes MM_PATH_TENSOR) */
} mm_path;

/* Limits of this build. */
#define MM_MAX_EXPERTS 64
#define MM_MAX_TOPK 8

/* Human-readable name of an mm_status value (static string). */
const char* mm_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int mm_version(void);

/* Text of the last CUDA failure reported as MM_ERR_CUDA on this host thread
 * (static thread-local storage; empty if none). */
const char* mm_last_error(void);

/* ------------------------------------------------------------------------
 * Dense SwiGLU FFN   ([L13] §0 / §1.2; [CH4] §4.2)
 *
 *   u = Wu x,  g = Wg x,  h = SiLU(g) ⊙ u,  y = Wd h,  SiLU(z) = z·sigmoid(z)
 *
 * x [T,H], Wg/Wu [I,H], Wd [H,I] in; y [T,H] out (overwritten).  g and u
 * never reach memory; h ([T,I]) lives in the workspace, in fp16 on the bf16
 * tensor-core path (with Wd converted to fp16) and fp32 for fp32 inputs.  A
 * value of h or Wd at or beyond the fp16 range (|v| >= 65520) is recorded
 * on the device and reported by mm_check_status() as MM_ERR_RANGE (the
 * weight-streaming paths keep h in fp32 or as a bf16 pair and need no check).
 * Limits: T >= 0 (T = 0 enqueues nothing); H, I >= 1; bf16 tensor and
 * streaming paths need H and I to be multiples of 64.
 * ---------------------------------------------------------------------- */
size_t mm_swiglu_ffn_workspace_bytes(int64_t T, int H, int I, int dtype);

int mm_swiglu_ffn(const void* x, const void* Wg, const void* Wu, const void* Wd,
                  void* y, int64_t T, int H, int I, int dtype,
                  void* workspace, size_t workspace_bytes, void* stream);

int mm_swiglu_ffn_ex(const void* x, const void* Wg, const void* Wu, const void* Wd,
                     void* y, int64_t T, int H, int I, int dtype,
                     void* workspace, size_t workspace_bytes, void* stream, int path);

/* Dense FFN in its MiniMind block ([L13] §3 step 2):
 *   y = x + FFN(RMSNorm(x)),  RMSNorm(x) = x / sqrt(mean_h x_h^2 + norm_eps) * w
 * norm_w [H] in x's dtype.  The normalised rows are written once (x's dtype)
 * for the GEMMs; the residual is added in the down GEMM's epilogue before y's
 * one rounding.  bf16: tensor cores; fp32: CUDA cores.  y must not alias x. */
size_t mm_swiglu_ffn_block_workspace_bytes(int64_t T, int H, int I, int dtype);

int mm_swiglu_ffn_block(const void* x, const void* norm_w, float norm_eps,
                        const void* Wg, const void* Wu, const void* Wd,
                        void* y, int64_t T, int H, int I, int dtype,
                        void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Prepared down weights
 *
 * The pages have no counterpart: the bf16 tensor-core prefill path keeps h
 * in fp16 (precision, see the dense FFN above), so it multiplies h by an fp16
 * copy of Wd, which both forwards otherwise make inside every call.  A caller
 * whose weights change less often than it runs the layer converts once:
 *   Wd16 [H, I] fp16 = Wd [H, I] bf16, exact for |w| >= 2^-14 (smaller
 *   magnitudes become fp16 subnormals, absolute error <= 2^-25).
 * A value at or beyond the fp16 range (|w| >= 65520) is recorded as
 * MM_ERR_RANGE in `status_ws` (a workspace of >= 256 bytes read by
 * mm_check_status; nullable: no report).  Asynchronous on `stream`.
 * H * I must be a multiple of 8; pointers 16-byte aligned.
 * ---------------------------------------------------------------------- */
int mm_prepare_down_weights(const void* Wd, void* Wd16, int H, int I, void* status_ws,
                            void* stream);

/* mm_swiglu_ffn_ex with prepared down weights: Wd16 (nullable) is used by the
 * tensor-core path in place of the in-call fp16 copy of Wd. */
int mm_swiglu_ffn_prepared(const void* x, const void* Wg, const void* Wu, const void* Wd,
                           const void* Wd16, void* y, int64_t T, int H, int I, int dtype,
                           void* workspace, size_t workspace_bytes, void* stream, int path);

/* ------------------------------------------------------------------------
 * Dense SwiGLU FFN without caller-provided scratch
 *
 * The pages describe no counterpart of this entry point; it exists for
 * callers that cannot allocate device memory when they run the FFN: code
 * that enqueues work while a CUDA graph is being captured in a mode that
 * forbids cudaMalloc, plug-ins of inference runtimes whose enqueue step
 * must not allocate, and real-time loops that cannot afford the implicit
 * device synchronisation of cudaMalloc / cudaFree.
 *
 * Same arguments and result as mm_swiglu_ffn, minus the workspace: its
 * scratch is a fixed array of MM_NOALLOC_SCRATCH_BYTES bytes of device
 * memory that belongs to this library.  The CUDA runtime reserves it on
 * every GPU where the library is loaded and keeps it until the process
 * exits.  The call allocates nothing.
 *
 *   - Size limit: the call needs mm_swiglu_ffn_workspace_bytes(T, H, I,
 *     dtype) <= MM_NOALLOC_SCRATCH_BYTES.  Anything larger returns
 *     MM_ERR_UNSUPPORTED with nothing enqueued.  For example, with H = 768,
 *     I = 2432 and bf16 this means T <= 2681.
 *   - The first call on each device looks up the array's device address,
 *     with that device current.  Make that first call before any stream
 *     capture starts.
 *   - All calls share the one array, and it keeps the last call's contents.
 *     Calls that overlap on the GPU therefore race: order them on one
 *     stream, or finish one before starting the next.
 *   - Each call first zeroes the array's 256-byte state header on `stream`
 *     (grid-barrier counters and the watchdog word), so a call whose
 *     pipeline wait gave up leaves no state behind for the next one.  That
 *     watchdog word is not readable through mm_check_status: a timed-out
 *     call is not reported.  Stream errors are still reported by the CUDA
 *     runtime.
 * ---------------------------------------------------------------------- */
#define MM_NOALLOC_SCRATCH_BYTES (16u << 20)

int mm_swiglu_ffn_noalloc(const void* x, const void* Wg, const void* Wu, const void* Wd,
                          void* y, int64_t T, int H, int I, int dtype, void* stream);

/* ------------------------------------------------------------------------
 * Top-k MoE forward   ([L13] §1.5, §1.6, §3 steps 4-6; [CH4] §4.3, §4.4)
 *
 *   r = Wr x (+ logit_bias);  p = softmax(r)            (fp32)
 *   S = TopK(p, k): descending p, equal p -> lower expert index first
 *   alpha_e = p_e / (sum_{j in S} p_j + 1e-20)
 *   y = sum_{e in S} alpha_e · SwiGLU_e(x)   — the k terms are added in fp32
 *       and rounded once to y's dtype, in a fixed order per path (results are
 *       deterministic; the pages' index_add_ into y rounds every term, which
 *       costs accuracy)
 *   count_e = #{(t,s): S_t[s] = e},  P_e = sum_t p_{t,e}
 *   aux_loss = E · coef · sum_e (count_e / T) · (P_e / T)
 *
 * Arguments:
 *   x [T,H], Wr [E,H]                 device, dtype
 *   Wg, Wu, Wd                        HOST arrays of E device pointers, one
 *                                     [I,H] / [I,H] / [H,I] matrix per expert
 *   logit_bias                        device fp32 [E], or NULL (no bias: the
 *                                     pages' router exactly)
 *   y [T,H]                           device, dtype, overwritten
 *   topk_idx [T,k]                    device int32, slots in descending p
 *   topk_w [T,k]                      device fp32, alpha of each slot
 *   aux_loss                          device fp32 scalar (coef = 0 gives 0)
 * Limits: T >= 1; 1 <= E <= MM_MAX_EXPERTS; 1 <= k <= min(E, MM_MAX_TOPK);
 * H a multiple of 8 and (E*H + k*E)*4 <= 200 KiB.
 * ---------------------------------------------------------------------- */
size_t mm_moe_workspace_bytes(int64_t T, int H, int I, int E, int k, int dtype);
/* The workspace one path needs (0: the path does not take the shape); the
 * gathering path (MM_PATH_TENSOR_GATHER) needs no T*k*H permuted copy of x. */
size_t mm_moe_workspace_bytes_for_path(int64_t T, int H, int I, int E, int k, int dtype,
                                       int path);

int mm_moe_forward(const void* x, const void* Wr,
                   const void* const* Wg, const void* const* Wu, const void* const* Wd,
                   int64_t T, int H, int I, int E, int k, float coef, int dtype,
                   const float* logit_bias,
                   void* y, int32_t* topk_idx, float* topk_w, float* aux_loss,
                   void* workspace, size_t workspace_bytes, void* stream);

int mm_moe_forward_ex(const void* x, const void* Wr,
                      const void* const* Wg, const void* const* Wu, const void* const* Wd,
                      int64_t T, int H, int I, int E, int k, float coef, int dtype,
                      const float* logit_bias,
                      void* y, int32_t* topk_idx, float* topk_w, float* aux_loss,
                      void* workspace, size_t workspace_bytes, void* stream, int path);

/* ------------------------------------------------------------------------
 * Router variants and saved router statistics   (p-chao.com "MiniMind 学习笔记
 * 08：FeedForward 与 MoE" §10, table of large-scale MoE mechanisms: "router
 * noise" and "z-loss"; §7: the router gradient flows through topk_weight)
 *
 * The table names the two mechanisms without formulas; this build reads
 * them as:
 *   router noise:  r_{t,e} = W_router x_t + logit_bias_e + noise_{t,e}, with
 *                  the caller's draws noise [T, E] (scale included); the
 *                  noisy logits feed softmax, top-k, alpha and aux;
 *   z-loss:        z_loss = z_coef * (1/T) * sum_t lse_t^2,
 *                  lse_t = log sum_e exp(r_{t,e}).
 * router_probs / router_lse return p [T, E] and lse [T] as computed, the
 * statistics a backward pass needs.
 *
 * Every pointer is nullable (NULL: off / not written); an options struct of
 * zeros is the plain mm_moe_forward_ex with path AUTO.  Every path (tensor,
 * streaming, SIMT) takes every option.  Pointers must be 4-byte aligned.
 * ---------------------------------------------------------------------- */
typedef struct {
  int path;                   /* mm_path of the FFN part (MM_PATH_AUTO = 0)        */
  const float* logit_noise;   /* device fp32 [T, E]: router noise, or NULL         */
  float z_coef;               /* z-loss coefficient                                */
  float* z_loss;              /* device fp32 scalar out, or NULL (not computed)    */
  float* router_probs;        /* device fp32 [T, E] out: softmax p, or NULL        */
  float* router_lse;          /* device fp32 [T] out: logsumexp of the logits, or NULL */
  /* MiniMind block ([L13] §3 step 2: hidden + mlp(post_attention_layernorm(hidden))):
   * with norm_weight, the layer's input is x_n = x / sqrt(mean_h x_h^2 + norm_eps) * w
   * (RMSNorm; the router takes it at full precision, the experts rounded to x's
   * dtype); with residual != 0, y = x + MoE(...).  Either one runs the call on the
   * tensor-core (bf16) or CUDA-core GEMMs; the streaming paths return
   * MM_ERR_UNSUPPORTED.  y must not alias x. */
  const void* norm_weight;    /* device [H], x's dtype, or NULL                    */
  float norm_eps;
  int residual;
  /* Prepared down weights (mm_prepare_down_weights): a HOST array of E device
   * pointers to fp16 [H, I] copies of Wd[e], or NULL.  The bf16 tensor-core
   * path then multiplies by them instead of making the fp16 copy inside the
   * call; the other paths read Wd. */
  const void* const* wd_f16;
  /* Router and permute (prefill tensor-core path): 0 runs them as one kernel
   * where all of its blocks fit on the GPU at once (bf16, H <= 768, E <= 16
   * (8 with norm_weight), k <= 4, T <= 128 x the SMs), so that x is read once;
   * its blocks wait for one another at one grid-wide barrier (bounded: after
   * 1 s the call fails with MM_ERR_TIMEOUT), so it assumes no kernel of
   * another stream holds SMs meanwhile.  1 always runs the router and the
   * permute as two kernels with no grid-wide wait.  The results are the same
   * bit for bit. */
  int separate_routing;
} mm_moe_options;

int mm_moe_forward_opts(const void* x, const void* Wr,
                        const void* const* Wg, const void* const* Wu, const void* const* Wd,
                        int64_t T, int H, int I, int E, int k, float coef, int dtype,
                        const float* logit_bias,
                        void* y, int32_t* topk_idx, float* topk_w, float* aux_loss,
                        void* workspace, size_t workspace_bytes, void* stream,
                        const mm_moe_options* opts);

/* Router half of the MoE forward only (logits, softmax, top-k, alpha, aux):
 * same arguments and meaning as mm_moe_forward without the experts and y.
 * expert_counts (device int32 [E], nullable) receives count_e. */
size_t mm_moe_route_workspace_bytes(int64_t T, int E, int k);

int mm_moe_route(const void* x, const void* Wr, int64_t T, int H, int E, int k,
                 float coef, int dtype, const float* logit_bias,
                 int32_t* topk_idx, float* topk_w, float* aux_loss,
                 int32_t* expert_counts,
                 void* workspace, size_t workspace_bytes, void* stream);

/* The same with router variants (opts->path is ignored). */
int mm_moe_route_opts(const void* x, const void* Wr, int64_t T, int H, int E, int k,
                      float coef, int dtype, const float* logit_bias,
                      int32_t* topk_idx, float* topk_w, float* aux_loss,
                      int32_t* expert_counts,
                      void* workspace, size_t workspace_bytes, void* stream,
                      const mm_moe_options* opts);

/* ------------------------------------------------------------------------
 * Backward pass   (training objective L_train = L_lm + L_aux, [L13] step 8;
 * the router's gradient flows only through the selected weights alpha,
 * p-chao.com "MiniMind 学习笔记 08" §7; in aux only P_e carries gradient,
 * [CH4] §4.4)
 *
 * bf16 only, on the tensor cores; H and I multiples of 64.  Inputs and
 * outputs are device memory; every gradient is OVERWRITTEN (not added to).
 * The intermediate dh = dy Wd is kept in the workspace in fp16 (11
 * significant bits); a value beyond the fp16 range is reported by
 * mm_check_status() as MM_ERR_RANGE.
 *
 * Dense FFN: for dy = dL/dy [T, H] (bf16),
 *   dx [T, H] (bf16) and dWg, dWu [I, H], dWd [H, I] (fp32) with
 *   dWd = dy^T h, dh = dy Wd, dU = dh SiLU(g), dG = dh u SiLU'(g),
 *   dx = dG Wg + dU Wu, dWg = dG^T x, dWu = dU^T x  (g and u recomputed).
 * T = 0 zeroes the weight gradients.
 * ---------------------------------------------------------------------- */
size_t mm_swiglu_ffn_backward_workspace_bytes(int64_t T, int H, int I, int dtype);

int mm_swiglu_ffn_backward(const void* x, const void* Wg, const void* Wu, const void* Wd,
                           const void* dy, int64_t T, int H, int I, int dtype,
                           void* dx, float* dWg, float* dWu, float* dWd,
                           void* workspace, size_t workspace_bytes, void* stream);

/* MoE layer: gradients of L = <dy, y> + d_aux * aux_loss + d_z * z_loss
 * (d_aux = d_z = 1 for L_lm + L_aux + L_z), given the forward's saved routing:
 * topk_idx, topk_w (alpha) and router_probs [T, E] from mm_moe_forward_opts
 * (router_lse [T] too when z_coef and d_z are non-zero, else nullable).
 * The router noise and logit bias of the forward are already inside those
 * probabilities.  Outputs:
 *   dx [T, H] (bf16), dWr [E, H] (fp32), dWg[e], dWu[e] [I, H] and dWd[e]
 *   [H, I] (HOST arrays of E device fp32 pointers; an expert no token chose
 *   gets zeros), d_bias [E] (fp32, nullable): the gradient of the logit bias
 *   as a parameter (= sum_t dL/dlogits).
 * Deterministic: every sum runs in a fixed order.
 * ---------------------------------------------------------------------- */
size_t mm_moe_backward_workspace_bytes(int64_t T, int H, int I, int E, int k, int dtype);

int mm_moe_backward(const void* x, const void* Wr,
                    const void* const* Wg, const void* const* Wu, const void* const* Wd,
                    int64_t T, int H, int I, int E, int k, float coef, int dtype,
                    const int32_t* topk_idx, const float* topk_w,
                    const float* router_probs, const float* router_lse,
                    const void* dy, float d_aux, float z_coef, float d_z,
                    void* dx, float* dWr, float* const* dWg, float* const* dWu,
                    float* const* dWd, float* d_bias,
                    void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Status
 * ---------------------------------------------------------------------- */
/* Synchronises `stream`, reads and clears the device status word kept at
 * the start of `workspace` (any workspace used by the calls above), and
 * returns MM_ERR_TIMEOUT if a kernel gave up on a pipeline wait since the
 * last check, MM_ERR_RANGE if an fp16 intermediate overflowed (the first
 * failure recorded wins), MM_ERR_CUDA if the stream reported an error, else
 * MM_OK. */
int mm_check_status(void* workspace, void* stream);

/* Self-test of the watchdog: launches one block that waits on a barrier no
 * one arrives on, with the given limit in microseconds (1 .. 10,000,000).
 * The wait gives up, records MM_ERR_TIMEOUT in `workspace` (>= 256 bytes)
 * and the kernel returns normally; mm_check_status() then reports it. */
int mm_watchdog_selftest(void* workspace, size_t workspace_bytes,
                         uint32_t limit_us, void* stream);

/* ------------------------------------------------------------------------
 * Measurement hooks (host-side only; they add no work to the kernels)
 * ---------------------------------------------------------------------- */
typedef enum {
  MM_KERNEL_ROUTER = 1,     /* logits/softmax/top-k/alpha/aux partials      */
  MM_KERNEL_DISPATCH = 3,   /* aux finalisation, group offsets, token permute */
  MM_KERNEL_GATEUP = 4,     /* gate/up GEMM with the SwiGLU epilogue        */
  MM_KERNEL_DOWN = 5,       /* down GEMM with the alpha-scaled combine      */
  MM_KERNEL_DECODE = 7,     /* decode-sized weight-streaming kernel (whole call) */
  MM_KERNEL_BWD_DGRAD = 8,  /* backward: dh = dy Wd and dx = dG Wg + dU Wu GEMMs */
  MM_KERNEL_BWD_SWIGLU = 9, /* backward: gate/up recomputed, SwiGLU derivative */
  MM_KERNEL_BWD_WGRAD = 10, /* backward: weight-gradient GEMMs                */
  MM_KERNEL_BWD_ROUTER = 11 /* backward: dispatch, router gradient, dx combine */
} mm_kernel_id;

/* Number of kernels this library has enqueued since it was loaded. */
uint64_t mm_launch_count(void);

/* Start timing every launch of one kernel (mm_kernel_id) with a pair of CUDA
 * events recorded on the launching stream around it, for at most
 * max_launches launches (1 .. 100000).  The events are created by the
 * library.  Returns MM_ERR_INVALID_ARG for a bad id or count. */
int mm_profile_start(int kernel_id, int max_launches);

/* Stop timing: waits for the last recorded event, returns the summed
 * duration in milliseconds and the number of launches timed. */
int mm_profile_stop(double* total_ms, int* launches);

#ifdef __cplusplus
}
#endif

#endif /* MM_H_ */
