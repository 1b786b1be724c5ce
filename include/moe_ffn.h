/*
 * moe_ffn.h - C ABI of a single-GPU (sm_103a) forward pass of a routed
 * Mixture-of-Experts FFN layer.
 *
 * The layer computes, for every token t with hidden row x_t,
 *
 *     y_t = F_s(x_t) + sum_{e in I_t} g_{t,e} F_e(x_t),   |I_t| = k,
 *     F(x) = (SiLU(x W1[:, :I]) * x W1[:, I:]) W2,
 *
 * the MoE output equation of "Megatron-LM 的 MoE 并行：以 DeepSeek-V4 为例"
 * (section 模型与入口) with the expert FFN, dispatch and combine of the
 * "mega_moe" operator page (section 计算公式: EP Dispatch, Expert Compute,
 * Token Combine).  I_t and g come from the router of the same Megatron page
 * (section 路由与负载 / 路由张量) or from a token-id hash table (section
 * 路由与负载 / Hash 路由).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library never allocates: scratch space is the caller's workspace, sized
 *     by moe_workspace_size() and prepared once by moe_workspace_init().
 *   - bf16 tensors are passed as uint16_t bit patterns, row-major, dense.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Host-checkable errors are returned before anything is
 *     launched.  Data errors found on the device (an expert id outside
 *     [0, E), a token id outside [0, V), a pipeline wait that timed out) are
 *     recorded in the workspace's status word; the offending assignment is
 *     skipped and moe_sync_status() reports the error.
 *   - Device pointers must be 16-byte aligned.  H and I must be multiples of
 *     64; for the router, E must be a multiple of 8.
 *   - One workspace serves one stream at a time: calls that overlap on the
 *     GPU and share a workspace race.
 */
#ifndef MOE_FFN_H
#define MOE_FFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer    */
  MOE_ERR_UNSUPPORTED = 2,   /* shape outside what the kernels implement      */
  MOE_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required    */
  MOE_ERR_BAD_EXPERT_ID = 4, /* device: an expert id outside [0, E)           */
  MOE_ERR_BAD_TOKEN_ID = 5,  /* device: a hash token id outside [0, V)        */
  MOE_ERR_TIMEOUT = 6,       /* device: a pipeline wait ran out of time       */
  MOE_ERR_CUDA = 7,          /* a CUDA runtime call failed                    */
  MOE_ERR_BOUNDS = 8         /* device, debug build only: an index read from
                                data was outside the array it indexes (the
                                access was skipped)                          */
} moe_status;

/* Affinity a = score(l) of a router logit l. */
typedef enum moe_score_fn {
  MOE_SCORE_SIGMOID = 0,       /* a = 1 / (1 + exp(-l))                            */
  MOE_SCORE_SQRT_SOFTPLUS = 1, /* a = sqrt(log(1 + exp(l))): the DeepSeek-V4 rule
                                  of the Megatron page, section 路由张量          */
  MOE_SCORE_SOFTMAX = 2        /* a = softmax over experts: the gate of
                                  "Megatron 分布式训练全维度并行技术文档", 4.2    */
} moe_score_fn;

typedef struct moe_params {
  int32_t T;          /* tokens (rows of X); 0 is allowed and does nothing     */
  int32_t H;          /* hidden size, multiple of 64                          */
  int32_t E;          /* routed experts, 1..4096                               */
  int32_t k;          /* experts per token, 1..min(E, 16)                      */
  int32_t I;          /* expert intermediate size, multiple of 64             */
  int32_t has_shared; /* 1: add one shared expert (Ws1, Ws2) with weight 1    */
  int32_t score_fn;   /* moe_score_fn                                          */
  float alpha;        /* gate scale                                            */
  int32_t renorm;     /* 1: g = alpha * a / sum_{selected} a;  0: g = alpha * a */
} moe_params;

/* Bytes of workspace the calls below need for these parameters. */
size_t moe_workspace_size(const moe_params* p);

/* Zero the workspace's status header.  Call once before the first use of a
 * workspace (and it may be called again at any time between calls). */
moe_status moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Router (Megatron page, section 路由与负载 / 路由张量; softmax gate of the
 * parallelism page, section 4.2):
 *   l = X Wg;  a = score_fn(l);  I_t = TopK_k(a + bias), listed by descending
 *   selection score, equal scores to the lower expert id;  G[t, j] = alpha *
 *   a[t, E_ids[t, j]] / sum_j a[t, E_ids[t, j]] (renorm = 1) or alpha * a.
 * The softmax rule selects on a alone and takes no bias.
 * Hash routing (section 路由与负载 / Hash 路由): when token_ids != NULL the ids
 * are E_ids[t, :] = tid2eid[token_ids[t], :] (table order) and the gates use
 * the same formula at those ids; bias must then be NULL.
 *   X        [T, H]  bf16      token rows
 *   Wg       [H, E]  bf16      gating linear (row-major: E contiguous)
 *   bias     [E]     fp32      selection-only expert bias, or NULL
 *   token_ids[T]     int32     hash mode only, else NULL
 *   tid2eid  [V, k]  int32     hash mode only, else NULL
 *   E_ids    [T, k]  int32     out
 *   G        [T, k]  fp32      out
 * A token whose top-k selection is too close to call in float32 is re-decided
 * with float64 logits, so the ids equal those of an exact evaluation except at
 * exact ties. */
moe_status moe_route(const moe_params* p, const uint16_t* X, const uint16_t* Wg,
                     const float* bias, const int32_t* token_ids, const int32_t* tid2eid,
                     int32_t V, int32_t* E_ids, float* G, void* ws, size_t ws_bytes,
                     void* stream);

/* The router's float32 logits alone, l = X Wg, into logits [T, E] fp32. */
moe_status moe_route_logits(const moe_params* p, const uint16_t* X, const uint16_t* Wg,
                            float* logits, void* ws, size_t ws_bytes, void* stream);

/* Dispatch ("mega_moe" page, section EP Dispatch; Megatron page, section
 * AlltoAll 的前向 / 计数与重排):
 *   counts [E]      int32 out   assignments per expert (ids outside [0,E) dropped)
 *   offsets[E + 1]  int32 out   exclusive prefix sum of counts
 *   perm   [T * k]  int32 out   perm[p] = flat assignment index t*k + j at expert
 *                               block row p, ascending inside each block; entries
 *                               past offsets[E] are left untouched. */
moe_status moe_dispatch(const moe_params* p, const int32_t* E_ids, int32_t* counts,
                        int32_t* offsets, int32_t* perm, void* ws, size_t ws_bytes,
                        void* stream);

/* Layer forward ("mega_moe" page, section 计算公式, plus the shared expert of
 * the Megatron page's MoE output equation):
 *   X    [T, H]      bf16   token rows
 *   E_ids[T, k]      int32  expert ids (from moe_route or the caller)
 *   G    [T, k]      fp32   gates
 *   W1   [E, H, 2I]  bf16   Linear1; columns [0, I) gate, [I, 2I) up
 *   W2   [E, I, H]   bf16   Linear2
 *   Ws1  [H, 2I], Ws2 [I, H]  bf16 shared expert (has_shared = 1), else NULL
 *   Y    [T, H]      bf16   out
 * Precision: float32 accumulation in both GEMMs and in the combine; the SwiGLU
 * rows are kept in bf16 (round to nearest even) between the GEMMs, each
 * expert's output rows in float32, and Y is rounded to bf16 once at the end.
 * With k = 1 and no shared expert the combine is done by Linear2's epilogue:
 * each float32 row times its gate is rounded once into Y (the expert rows are
 * not kept), and tokens whose id was dropped get zero rows, as in the combine.
 * Every step (dispatch, Linear1 with SwiGLU, Linear2, combine) runs in this
 * library's kernels, with no host synchronisation: sizes come from device
 * memory, so a call (with moe_route before it) can be captured in a CUDA graph
 * and replayed. */
moe_status moe_forward(const moe_params* p, const uint16_t* X, const int32_t* E_ids,
                       const float* G, const uint16_t* W1, const uint16_t* W2,
                       const uint16_t* Ws1, const uint16_t* Ws2, uint16_t* Y, void* ws,
                       size_t ws_bytes, void* stream);

/* Dispatch for callers that cannot provide a workspace.  There is no
 * counterpart of this call in the pages: it exists because some callers may not
 * allocate device memory where they route tokens (their device memory is held
 * by another allocator, or a cudaMalloc/cudaFree, which can synchronise the
 * device, is not acceptable on their path).  Same results as moe_dispatch
 * (counts [E], offsets [E + 1], perm [T * k], all caller-owned device memory),
 * but the scratch is a fixed array inside the library (about 1.2 MB, held on
 * every GPU that loads the library until the process exits).
 * Limits: T * k <= 262144 and E <= 512, else MOE_ERR_UNSUPPORTED before any
 * device work.  The call allocates nothing.  Its first call in each CUDA
 * context (on each device, and again after a device reset) looks up the
 * array's device address (cudaGetSymbolAddress); make that first call before
 * any stream capture.  All calls share the array: calls that overlap on the
 * GPU race, so serialise them.  Ids outside [0, E) are dropped and there is no
 * status word: a caller sees them only as offsets[E] < T * k. */
moe_status moe_dispatch_noalloc(const moe_params* p, const int32_t* E_ids, int32_t* counts,
                                int32_t* offsets, int32_t* perm, void* stream);

/* moe_forward, recording caller-created CUDA events (cudaEvent_t, NULL entries
 * skipped) on `stream` at the stage boundaries, for measurement:
 *   stage_events[0] before dispatch      [1] after dispatch
 *   stage_events[2] after Linear1+SwiGLU [3] after Linear2   [4] after combine
 * stage_events itself may be NULL (then this is moe_forward). */
moe_status moe_forward_timed(const moe_params* p, const uint16_t* X, const int32_t* E_ids,
                             const float* G, const uint16_t* W1, const uint16_t* W2,
                             const uint16_t* Ws1, const uint16_t* Ws2, uint16_t* Y, void* ws,
                             size_t ws_bytes, void* stream, void* const* stage_events);

/* Bytes of workspace moe_forward_a8w8 needs for these parameters. */
size_t moe_workspace_size_a8w8(const moe_params* p);

/* Layer forward in the A8W8-INT form of the "mega_moe" page (section 计算过程,
 * A8W8 scenario), no shared expert (has_shared must be 0):
 *   each token row is quantised, s^X_t = max|x_t| / 127, q_t = round(x_t / s^X_t)
 *   (nearest integer, halves away from zero; float32);
 *   per expert: C = Q_e W1q[e]^T (int32), H = (C * S1[e]) * s^X,
 *   A = SiLU(H[:, :I]) * H[:, I:], each row of A re-quantised the same way
 *   (s^A, A8), D = A8 W2q[e]^T (int32), Y_e = (D * S2[e]) * s^A kept in bf16;
 *   y_t = sum_j G[t, j] Y[row(t, j)] (fp32 sum, bf16 out).
 *   The weights keep the operator's layout, one row per output channel with
 *   K contiguous (rows 0..I-1 of W1q are the SiLU branch):
 *   W1q [E, 2I, H] int8, S1 [E, 2I] fp32 (per output channel)
 *   W2q [E, H, I]  int8, S2 [E, H]  fp32
 *   X [T, H] bf16, E_ids [T, k], G [T, k] fp32, Y [T, H] bf16 out.
 * H and I must be multiples of 64 (MOE_ERR_UNSUPPORTED otherwise).
 * The int8 products run on the fp16 tensor-core path (GB300's int8 tensor rate
 * is far lower): codes are exact in fp16 and the fp32 accumulator holds each
 * int32 sum exactly while every partial sum stays below 2^24 in magnitude
 * (always true for K * 127 * 127 < 2^24, i.e. K <= 1040; beyond that, true
 * unless the codes of a row and a column agree in sign at full scale).
 * stage_events: NULL, or 5 caller-created cudaEvent_t recorded at: start,
 * after dispatch and token quantisation, after Linear1, after the
 * re-quantisation and Linear2, after combine. */
moe_status moe_forward_a8w8(const moe_params* p, const uint16_t* X, const int32_t* E_ids,
                            const float* G, const int8_t* W1q, const float* S1,
                            const int8_t* W2q, const float* S2, uint16_t* Y, void* ws,
                            size_t ws_bytes, void* stream, void* const* stage_events);

/* Bytes of workspace moe_forward_train and moe_backward need (the forward's
 * workspace plus the tensors the backward keeps or builds). */
size_t moe_workspace_size_train(const moe_params* p);

/* moe_forward that also keeps, in the workspace, what moe_backward needs: the
 * routing permutation, the Linear1 pre-activations (bf16), the SwiGLU output
 * and the expert output rows.  Same arguments and results as moe_forward;
 * the workspace must hold moe_workspace_size_train(p) bytes. */
moe_status moe_forward_train(const moe_params* p, const uint16_t* X, const int32_t* E_ids,
                             const float* G, const uint16_t* W1, const uint16_t* W2,
                             const uint16_t* Ws1, const uint16_t* Ws2, uint16_t* Y, void* ws,
                             size_t ws_bytes, void* stream);

/* Backward of the layer for the upstream gradient dY [T, H] (bf16), after
 * moe_forward_train on the same workspace, inputs and routing.  The top-k ids
 * are constants; the selected experts' gates and affinities carry gradient to
 * the router ("Megatron-LM 的 MoE 并行：以 DeepSeek-V4 为例", section 反向的通信;
 * the parallelism page's section 4.7, 反向流程):
 *   dG[t, j]  = <dY_t, Y_e(x_t)>                       (mixing-weight gradient)
 *   expert e: dYp = g dY (rows of e), dA = dYp W2[e]^T, dHg = dA * Hu * SiLU'(Hg),
 *             dHu = dA * SiLU(Hg), dW2[e] = A^T dYp, dW1[e] = X_e^T dH,
 *             dX_e = dH W1[e]^T;  the shared expert likewise with g = 1;
 *   router:   dL/da from dG through the gate rule, dL/dl through the affinity,
 *             dWg = X^T dl, and dX gets dl Wg^T;
 *   dX_t = sum over the token's assignments of dX_e + shared + router parts.
 * Outputs: dX [T, H] bf16; dWg [H, E], dW1 [E, H, 2I], dW2 [E, I, H], dWs1
 * [H, 2I], dWs2 [I, H] fp32 (overwritten, not accumulated); dG [T, k] fp32
 * or NULL.  E_ids and G as given to the forward (top-k or hash routing).  The
 * products run on bf16 tensor cores with fp32 accumulation; dY, the gate-
 * scaled rows, the pre-activations and their gradient and the logit
 * gradient are bf16.  E must be a multiple of 8.  stage_events: NULL or 5
 * cudaEvent_t recorded at: start, after the un-permute backward, after the
 * two input-gradient GEMMs, after the weight gradients, at the end. */
moe_status moe_backward(const moe_params* p, const uint16_t* X, const uint16_t* Wg,
                        const int32_t* E_ids, const float* G, const uint16_t* W1,
                        const uint16_t* W2, const uint16_t* Ws1, const uint16_t* Ws2,
                        const uint16_t* dY, uint16_t* dX, float* dWg, float* dW1, float* dW2,
                        float* dWs1, float* dWs2, float* dG, void* ws, size_t ws_bytes,
                        void* stream, void* const* stage_events);

/* Element formats of the MX forms ("mega_moe" page, section 约束说明:
 * dispatch_quant_out_dtype FLOAT8_E4M3FN, FLOAT8_E5M2 or FLOAT4_E2M1, group
 * size 32, FLOAT8_E8M0 scales).  The values are also the tensor cores'
 * format codes.  E2M1 codes are stored two per byte, the even element in the
 * low nibble, so an E2M1 tensor [rows, cols] occupies [rows, cols / 2] bytes. */
typedef enum moe_mx_format {
  MOE_MX_E4M3 = 0, /* 1 sign, 4 exponent (bias 7), 3 mantissa bits; max 448   */
  MOE_MX_E5M2 = 1, /* 1 sign, 5 exponent (bias 15), 2 mantissa bits; max 57344 */
  MOE_MX_E2M1 = 5  /* 1 sign, 2 exponent (bias 1), 1 mantissa bit; max 6      */
} moe_mx_format;

/* Q_MX of bf16 rows, the MX quantisation of the "mega_moe" page (section
 * 计算过程, MXFP scenario): for each group of 32 consecutive values v of a
 * row, the shared exponent e = floor(log2 max|v|) - emax (emax 8 for E4M3,
 * 15 for E5M2, 2 for E2M1; clamped below at -127, and -127 for a group of zeros) is
 * stored as the E8M0 code e + 127, and each element as the FP8 code of
 * v / 2^e rounded to nearest, ties to even, saturating at the largest finite
 * value.  (The pages name the operation; these details follow the OCP
 * Microscaling formats definition.)  Use it to prepare MX weights from bf16
 * ones, or to inspect the token quantisation of moe_forward_mx.
 *   X [rows, cols] bf16 (16-byte aligned), cols a multiple of 32;
 *   Q [rows, cols] codes out ([rows, cols / 2] for E2M1; 16-byte aligned);
 *   S [rows, cols / 32] out.
 * Asynchronous on `stream`; errors are host-checked only. */
moe_status moe_quantize_mx(int32_t fmt, const uint16_t* X, int32_t rows, int32_t cols,
                           uint8_t* Q, uint8_t* S, void* stream);

/* Bytes of workspace moe_forward_mx needs for these parameters. */
size_t moe_workspace_size_mx(const moe_params* p);

/* Layer forward in the MX forms of the "mega_moe" page (section 计算过程,
 * MXFP scenario; section 约束说明: A8W8-FP, A8W4-FP, A4W4-FP), no shared expert
 * (has_shared must be 0), combine unquantised.  fmt is the activations'
 * element format, wfmt the weights': (E4M3, E4M3), (E5M2, E5M2) (A8W8-FP),
 * (E4M3 or E5M2, E2M1) (A8W4-FP), (E2M1, E2M1) (A4W4-FP); other pairs give
 * MOE_ERR_UNSUPPORTED:
 *   (Xq, SX) = Q_MX(X) per token row (see moe_quantize_mx);
 *   per expert e with rows R_e: Z = DQ(Xq[R_e]) DQ(W1[e])^T [n_e, 2I];
 *   U = Z[:, :I] * sigmoid(Z[:, :I]) * Z[:, I:]; (Uq, SU) = Q_MX(U);
 *   O = DQ(Uq) DQ(W2[e])^T [n_e, H], kept in bf16;
 *   y_t = sum_j G[t, j] O[row(t, j)] (fp32 sum, bf16 out).
 * DQ multiplies each code by its group's scale 2^(code - 127).
 *   W1 [E, 2I, H] codes (H contiguous; E2M1 packed: [E, 2I, H / 2] bytes;
 *      the first I rows are the SiLU branch), S1 [E, 2I, H / 32] E8M0 codes:
 *      the pages' weight1 and weightScales1 [E, 2I, H / 64, 2] read as one
 *      group per 32 of H;
 *   W2 [E, H, I] codes (E2M1: [E, H, I / 2] bytes), S2 [E, H, I / 32];
 *   X [T, H] bf16, E_ids [T, k], G [T, k] fp32, Y [T, H] bf16 out.
 * H and I must be multiples of 128 (MOE_ERR_UNSUPPORTED otherwise); S1 and
 * S2 must be 4-byte aligned, the other pointers 16-byte aligned (scales at
 * 16-byte aligned addresses whose rows are 16-byte multiples, H and I
 * multiples of 512, are read in wider chunks).  The products run on the
 * block-scaled tensor cores with fp32 accumulation: kind::mxf8f6f4, or
 * kind::mxf4 on packed tiles for E2M1 x E2M1 when H and I are multiples of
 * 256.
 * stage_events: NULL, or 5 caller-created cudaEvent_t recorded at: start,
 * after dispatch and token quantisation, after Linear1 (+ SwiGLU and
 * re-quantisation), after Linear2, after combine. */
moe_status moe_forward_mx(const moe_params* p, int32_t fmt, int32_t wfmt, const uint16_t* X,
                          const int32_t* E_ids, const float* G, const uint8_t* W1,
                          const uint8_t* S1, const uint8_t* W2, const uint8_t* S2, uint16_t* Y,
                          void* ws, size_t ws_bytes, void* stream, void* const* stage_events);

/* Synchronise `stream`, read the workspace's device status word, clear it and
 * return the most serious error recorded since the last call, in the order
 * TIMEOUT, BAD_TOKEN_ID, BAD_EXPERT_ID (MOE_OK if none).  A bad hash token
 * gives its token ids -1 and gates 0; moe_forward then drops those
 * assignments and records BAD_EXPERT_ID as well. */
moe_status moe_sync_status(void* ws, size_t ws_bytes, void* stream);

/* Self-test of the device-side wait limit: launches one kernel that waits on
 * an mbarrier nothing arrives on.  The wait gives up after limit_us
 * microseconds (1..1000000) and records MOE_ERR_TIMEOUT in the workspace
 * status word, which moe_sync_status() then returns.  The GPU context stays
 * usable.  The same bounded wait guards every pipeline wait of the GEMMs. */
moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, uint32_t limit_us, void* stream);

/* Self-test of the debug build's bounds checks (the library compiled with
 * MOE_DEBUG_BOUNDS, which checks every index the kernels read from data
 * against the extent of the array it indexes and skips a bad access instead
 * of trapping).  Launches one kernel that writes element `index` of a 32-int
 * array at byte 128 of the workspace's status header through such a check:
 * an index outside [0, 32) is skipped and recorded, and the next
 * moe_sync_status() returns MOE_ERR_BOUNDS.  The release library checks
 * nothing and returns MOE_ERR_UNSUPPORTED without launching.  Not a part of
 * the layer: it has no counterpart on the pages. */
moe_status moe_selftest_bounds(void* ws, size_t ws_bytes, int64_t index, void* stream);

/* Static text for a status code. */
const char* moe_status_string(moe_status s);

/* Version of this ABI (incremented on any incompatible change). */
int32_t moe_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H */
