/*
 * gpt2_ops.h — kernel-level C ABI: each step of the GPT-2 training step as
 * its own call, for per-kernel parity tests and roofline measurement.
 *
 * The layers and their backward formulas are those of "llm.c: GPT-2 training
 * in plain C, with every gradient written by hand", §2 How the code works
 * (encoder, layernorm, matmul, attention, gelu, residual, softmax and
 * crossentropy, each with a hand-written backward; attention's causal loop
 * t2 <= t), with the fusions of "llm.c's Origin and the Future of LLM
 * Compilers", [13:50] Avengers Assemble (residual add fused into LayerNorm,
 * softmax and cross-entropy fused in the classifier, AdamW as one fused
 * update, deterministic encoder backward without atomics).
 *
 * Conventions
 *   - dtype selects the activation element type: GPT2_PRECISION_FP32 (float)
 *     or GPT2_PRECISION_BF16 (__nv_bfloat16).  Statistics (mean, rstd, LSE,
 *     losses) and parameter gradients are always float.
 *   - Every pointer except `*_host` is a device pointer owned by the caller;
 *     rows are contiguous and row-major unless a leading dimension is given.
 *     Vector kernels need 16-byte aligned rows (C multiple of 4 floats or 8
 *     bf16 values).
 *   - `scratch` is caller-owned device memory of at least the size the
 *     matching *_scratch_bytes() call returns; it is overwritten.
 *   - `stream` is a cudaStream_t; calls only enqueue work.
 *   - Returns GPT2_OK or GPT2_ERR_INVALID_ARG (bad shape/dtype/scratch) or
 *     GPT2_ERR_CUDA (launch failure).  Kernels that check ranges OR a bit into
 *     *flags_dev (1 token, 2 target, 4 timeout) instead of faulting.
 */
#ifndef GPT2_B300_OPS_H
#define GPT2_B300_OPS_H

#include <stddef.h>
#include <stdint.h>

#include "gpt2.h"

#ifdef __cplusplus
extern "C" {
#endif

/* out[b,t,:] = wte[tok[b,t]] + wpe[t]   (out: [B*T][C], wte: [V..][C], wpe: [>=T][C]) */
int gpt2_op_encoder_forward(int dtype, void* out, const int32_t* tokens, const void* wte, const void* wpe,
                            int B, int T, int C, int V, int* flags_dev, void* stream);

/* dwpe[t] += sum_b dres[b,t];  dwte[v] += sum of dres rows with token v, in a
 * fixed order (deterministic).  dres: float [B*T][C]; dwte: [V][C].  With
 * B*T <= 16384 the positions are grouped by a radix sort on the token and
 * each token's sum is taken over fixed chunks of the sorted positions (chunk
 * partials added in chunk order); otherwise a bitonic sort and one sum per
 * token in position order.  A position whose token is outside [0, V) adds
 * nothing to dwte (its dwpe term still counts) and ORs 1 into *flags_dev
 * (flags_dev may be NULL).  1 <= V <= 65535.
 * scratch: gpt2_op_encoder_backward_scratch_bytes(B, T, C) bytes. */
size_t gpt2_op_encoder_backward_scratch_bytes(int B, int T, int C);
int gpt2_op_encoder_backward(float* dwte, float* dwpe, const float* dres, const int32_t* tokens, int B, int T,
                             int C, int V, int* flags_dev, void* scratch, size_t scratch_bytes, void* stream);

/* The same encoder backward without a scratch argument, for callers that
 * cannot allocate device memory: code running inside a host program that owns
 * all device memory (a framework's caching allocator or a fixed, pre-planned
 * budget) and code on latency-critical paths where cudaMalloc's implicit
 * synchronisation is not acceptable.  (The llm.c pages have no counterpart of
 * this call.)  Its scratch is a library-owned device array of
 * GPT2_NOALLOC_MAX_TOKENS 32-bit keys (128 KiB), held on every GPU that loads
 * the library until the process exits; the call itself allocates nothing.
 * The first call on a device looks up the array's device address on that
 * device, so make that first call before capturing any stream on it.  Calls
 * share the array: calls that overlap on the GPU race, and each call rewrites
 * every key slot it reads, so no state carries over between calls.
 * Tokens are range-checked as in gpt2_op_encoder_backward (V, flags_dev).
 * Returns GPT2_ERR_BUFFER_TOO_SMALL when B*T exceeds GPT2_NOALLOC_MAX_TOKENS,
 * GPT2_ERR_INVALID_ARG for bad pointers, C % 4 != 0 or V outside [1, 65535],
 * GPT2_ERR_CUDA if the array's address cannot be obtained or a launch fails. */
#define GPT2_NOALLOC_MAX_TOKENS 32768
int gpt2_op_encoder_backward_noalloc(float* dwte, float* dwpe, const float* dres, const int32_t* tokens, int B,
                                     int T, int C, int V, int* flags_dev, void* stream);

/* r = a + b (b may be NULL: r = a, resid_out unused); y = (r - mean)*rstd*w + bias,
 * rstd = 1/sqrt(biased var + 1e-5); rows x C. */
int gpt2_op_residual_layernorm_forward(int dtype, void* resid_out, void* y, float* mean, float* rstd,
                                       const void* a, const void* b, const void* w, const void* bias, int rows,
                                       int C, void* stream);

/* dres = (accumulate ? dres : 0) + dx with dx = rstd*(dnorm - mean(dnorm) - xhat*mean(dnorm*xhat)),
 * dnorm = dy*w; dres_c (optional) receives dres in dtype.  If dw and db are given:
 * dw += sum dy*xhat, db += sum dy, and (if dres_sum is given) dres_sum += the column
 * sums of the new dres, which is the bias gradient of the projection whose output
 * gradient dres is.  The sums go through per-chunk partials in scratch and are added
 * in a fixed order (deterministic). */
size_t gpt2_op_layernorm_backward_scratch_bytes(int rows, int C);
int gpt2_op_layernorm_backward(int dtype, float* dres, void* dres_c, const void* dy, const void* x,
                               const float* mean, const float* rstd, const void* w, float* dw, float* db,
                               float* dres_sum, int rows, int C, int accumulate, void* scratch,
                               size_t scratch_bytes, void* stream);

/* The LayerNorm backward as the training step runs it: the residual gradient
 * passed from one layer to the next in the activation dtype (bf16 in the bf16
 * step, float in the fp32 step) instead of an fp32 accumulator plus a copy.
 * dres_out = (dres_in ? dres_in : 0) + dx, both [rows][C] in dtype (dres_in
 * NULL: no incoming gradient; dres_in == dres_out: in place); dres_f32
 * (optional) receives the new value in float, before rounding to dtype
 * (dres_out may then be NULL).  dw, db, dres_sum and scratch as for
 * gpt2_op_layernorm_backward, dres_sum taking the column sums of the new value
 * before rounding.  Pointers 16-byte aligned. */
int gpt2_op_layernorm_backward_rg(int dtype, void* dres_out, const void* dres_in, float* dres_f32, const void* dy,
                                  const void* x, const float* mean, const float* rstd, const void* w, float* dw,
                                  float* db, float* dres_sum, int rows, int C, void* scratch, size_t scratch_bytes,
                                  void* stream);

/* D(m,n) = sum_k A(m,k) B(n,k) then an epilogue:
 *   A(m,k) = a_kmajor ? A[m*lda+k] : A[k*lda+m];  B(n,k) = b_kmajor ? B[n*ldb+k] : B[k*ldb+n]
 *   epilogue 0: D = acc (+bias[n])          1: aux = acc + bias[n], D = GELU_tanh(aux)
 *            2: D = acc * GELU_tanh'(aux)   3: D (float) += acc
 * path: 0 = best available, 1 = SIMT kernel, 2 = tensor-core (tcgen05) kernel only
 * (GPT2_ERR_INVALID_ARG if the shape/layout is outside what it handles).
 * workspace (optional, tensor-core path, epilogue 3): device memory of at least
 * gpt2_op_matmul_workspace_bytes(M, N, K, 3) bytes, 16-byte aligned, overwritten.
 * With it the kernel may split K across CTAs: each split stores its partial
 * product in the workspace and a second kernel adds the partials into D in
 * split order, so the result is deterministic.  Calls that share one workspace
 * must not overlap on the GPU.  Without it (NULL) there is no split. */
size_t gpt2_op_matmul_workspace_bytes(int M, int N, int K, int epilogue);
int gpt2_op_matmul(int dtype, const void* A, long long lda, int a_kmajor, const void* B, long long ldb,
                   int b_kmajor, int M, int N, int K, void* D, long long ldd, const void* bias, void* aux,
                   long long ldaux, int epilogue, int path, int* flags_dev, void* workspace,
                   size_t workspace_bytes, void* stream);
/* `batch` independent products of the same shape in one launch: item z uses
 * A + z*sA, B + z*sB, D + z*sD and aux + z*sAux (strides in elements of each
 * array's type; multiples of 16 bytes on the tensor-core path), with the
 * layouts and epilogues of gpt2_op_matmul but no bias and no K split.  Each
 * item's output tile is written by exactly one CTA, so epilogue 3 (D +=) stays
 * deterministic.  The weight-gradient products of all layers of a model, taken
 * together after the backward pass, are the intended use. */
int gpt2_op_matmul_batched(int dtype, int batch, const void* A, long long lda, long long sA, int a_kmajor,
                           const void* B, long long ldb, long long sB, int b_kmajor, int M, int N, int K, void* D,
                           long long ldd, long long sD, void* aux, long long ldaux, long long sAux, int epilogue,
                           int path, int* flags_dev, void* stream);

/* The attention-projection input gradient with the attention backward's
 * D = rowsum(dO * O) taken in its epilogue (bf16, tensor-core path only):
 * dX[M][K] = dY[M][N] . W[N][K] (dY row-major [M][ldy], W row-major [N][ldw],
 * dX row-major [M][ldx]), and for every row m = b*T + t and head h (64
 * columns of dX): D[(b*H + h)*T + t] = sum of dX[m][c] * O[m][c] over the
 * head's columns, with dX as stored in bf16 and O [M][ldo] the attention
 * output.  K must be 64*H and M a multiple of T.  The result feeds
 * gpt2_op_attention_backward's D.  flags_dev: a bounded wait that runs out
 * ORs 4 into it. */
int gpt2_op_matmul_rowdot(const void* dY, long long ldy, const void* W, long long ldw, int M, int N, int K, void* dX,
                          long long ldx, const void* O, long long ldo, float* D, int T, int H, int* flags_dev,
                          void* stream);

/* The LayerNorm in front of a product folded into it (the pages' fused
 * LayerNorm -> matmul, "llm.c's Origin and the Future of LLM Compilers",
 * [13:50] Avengers Assemble).  Since LN(r) = (r - mean) rstd gamma + beta per
 * row, LN(r) W^T + b = rstd (r W'^T - mean s) + c with W' = W diag(gamma),
 * s[n] = sum_k W'[n][k], c[n] = b[n] + sum_k beta[k] W[n][k]: the product runs
 * on the LayerNorm's input r itself and its epilogue applies the row's
 * statistics, so no normalised copy of r is written or read.
 *   gpt2_op_lnfold_weights: Wf (bf16 [N][K]) = W diag(gamma) rounded, s[n] the
 *     sum of Wf's row as stored, c[n] = bias[n] + sum_k beta[k] W[n][k] (fp32),
 *     for `items` stacked weights (item z: W + z*N*K, gamma/beta + z*K,
 *     bias + z*N, outputs likewise); W, gamma, beta fp32; bias may be NULL.
 *     K % 8 == 0, pointers 16-byte aligned.
 *   gpt2_op_matmul_lnfold: D[m][n] = rstd[m] (sum_k R[m][k] Wf[n][k] -
 *     mean[m] s[n]) + c[n] stored bf16 (R [M][ldr] the LayerNorm input, bf16;
 *     mean/rstd its row statistics); with aux non-NULL the GELU form: aux =
 *     that value (bf16), D = GELU(aux).  Tensor cores only: INVALID_ARG when
 *     the shape is outside what they handle (N % 8, 16-byte aligned rows).
 *     flags_dev: a bounded wait that runs out ORs 4 into it. */
int gpt2_op_lnfold_weights(void* Wf, float* s, float* c, const float* W, const float* gamma, const float* beta,
                           const float* bias, int items, int N, int K, void* stream);
int gpt2_op_matmul_lnfold(const void* R, long long ldr, const float* mean, const float* rstd, const void* Wf,
                          long long ldw, const float* s, const float* c, int M, int N, int K, void* D, long long ldd,
                          void* aux, long long ldaux, int* flags_dev, void* stream);

/* Causal multi-head attention over qkv [B*T][3C] (columns Q | K | V, head h uses
 * columns h*hd..h*hd+hd-1 of each); out [B*T][C]; lse [B][H][T] = log sum exp of
 * the scaled scores q.k/sqrt(hd) over t2 <= t (the attention layer and its
 * causal loop in "llm.c: GPT-2 training in plain C, with every gradient written
 * by hand", §2 How the code works).
 * path: 0 = best available, 1 = SIMT kernels, 2 = tensor-core (tcgen05) kernels
 * only.  The tensor-core kernels need dtype bf16, hd = 64, T % 128 == 0, 16-byte
 * aligned pointers and flags_dev (a bounded wait that runs out ORs 4 into it);
 * path 2 outside that returns GPT2_ERR_INVALID_ARG. */
int gpt2_op_attention_forward(int dtype, void* out, float* lse, const void* qkv, int B, int T, int C, int H,
                              int path, int* flags_dev, void* stream);
/* dqkv [B*T][3C] from dout [B*T][C] with P recomputed from lse:
 * D = rowsum(dO*O), dS = P*(dO.V^T - D), dQ = dS K/sqrt(hd), dK = dS^T Q/sqrt(hd),
 * dV = P^T dO.  scratch (16-byte aligned) receives D as float [B][H][T] at its
 * start and, when T % 128 == 0, the bf16 dS blocks of the causal triangle that
 * the tensor-core dK/dV kernel hands to its dQ kernel (B*H*n(n+1)/2 blocks of
 * 32 KB, n = T/128) after it; no atomics, so the result is deterministic.
 * path and flags_dev as for the forward. */
size_t gpt2_op_attention_backward_scratch_bytes(int B, int T, int H);
int gpt2_op_attention_backward(int dtype, void* dqkv, const void* dout, const void* qkv, const void* out,
                               const float* lse, int B, int T, int C, int H, int path, int* flags_dev,
                               void* scratch, size_t scratch_bytes, void* stream);

/* Per row of logits [rows][Vp]: losses[r] = logsumexp(z[0:V]) - z[target];
 * write_grad: z[v] = (softmax(z[0:V])[v] - [v == target]) * dloss in place, pads 0. */
int gpt2_op_softmax_crossentropy(int dtype, void* logits, float* losses, const int32_t* targets, int rows, int V,
                                 int Vp, float dloss, int write_grad, int* flags_dev, void* stream);

/* The classifier's fused form (bf16, tensor cores): D[M][N] = A[M][K] . B[N][K]^T
 * stored as bf16 (both operands K-major), and, per row and column tile n of
 * gpt2_op_logit_stats_tiles(N), the statistics of the stored values of the
 * columns < stats_cols: stats[(row * tiles + n) * 2] = their maximum m,
 * stats[... + 1] = sum of exp(value - m) (m = -inf, sum 0 for a tile without
 * such columns).  stats: M * tiles * 2 floats, 8-byte aligned, caller-owned.
 * gpt2_op_softmax_crossentropy_stats then gives the same losses and dlogits as
 * gpt2_op_softmax_crossentropy (write_grad = 1) from D and those statistics,
 * reading each row once: the row's log-sum-exp is M + ln S with M = max_n m_n,
 * S = sum_n s_n exp(m_n - M).  Both need flags_dev (bounded waits report
 * FLAG_TIMEOUT, a target outside [0, V) FLAG_TARGET_RANGE); INVALID_ARG when the
 * shape or alignment is not supported (N % 8, 16-byte aligned pointers). */
int gpt2_op_logit_stats_tiles(int N);
int gpt2_op_matmul_logit_stats(const void* A, long long lda, const void* B, long long ldb, int M, int N, int K,
                               void* D, long long ldd, float* stats, int stats_cols, int* flags_dev, void* stream);
int gpt2_op_softmax_crossentropy_stats(void* logits, float* losses, const int32_t* targets, const float* stats,
                                       int rows, int V, int Vp, float dloss, int* flags_dev, void* stream);

/* AdamW on n floats (n % 4 == 0), bias-corrected at step t >= 1, decay wd;
 * p_bf16 (optional) receives the updated parameters rounded to bf16;
 * gscale_dev (optional, one device float): every gradient is multiplied by it
 * first (the clip factor gpt2_op_grad_norm leaves in out2_dev[1]). */
int gpt2_op_adamw(float* p, const float* g, float* m, float* v, void* p_bf16, long long n, float lr, float b1,
                  float b2, float eps, float wd, int t, const float* gscale_dev, void* stream);

/* Global gradient norm and clip factor (the llm.c tour's global_norm component;
 * the pages give no formula, the plainest reading is taken):
 * out2_dev[0] = sqrt(sum_i g_i^2), out2_dev[1] = min(1, max_norm / (norm + 1e-6)).
 * g 16-byte aligned, n > 0, max_norm > 0; scratch of gpt2_op_grad_norm_scratch_bytes()
 * bytes.  The sum runs over fixed chunks in a fixed order: deterministic. */
size_t gpt2_op_grad_norm_scratch_bytes(void);
int gpt2_op_grad_norm(const float* g, long long n, float max_norm, float* out2_dev, void* scratch,
                      size_t scratch_bytes, void* stream);

/* tanh-form GELU forward / backward (dinp = dout * GELU'(inp)) over n elements. */
int gpt2_op_gelu_forward(int dtype, void* out, const void* in, long long n, void* stream);
int gpt2_op_gelu_backward(int dtype, void* dinp, const void* inp, const void* dout, long long n, void* stream);

/* out[c] += sum_r X[r*ldx + c] (deterministic order); cols and ldx multiples of
 * 4 floats / 8 bf16, X 16-byte aligned. */
size_t gpt2_op_colsum_scratch_bytes(int rows, int cols);
int gpt2_op_colsum(int dtype, float* out, const void* X, int rows, int cols, long long ldx, void* scratch,
                   size_t scratch_bytes, void* stream);

/* Check of the failure path of the tensor-core kernels' bounded waits (the
 * llm.c tour's detail graph keeps long runs observable with an outlier
 * detector; here a kernel that stops making progress must report it instead
 * of hanging the GPU).  Launches one CTA that allocates tensor memory and
 * waits on an mbarrier that nothing signals: one warp gives up after limit_us
 * microseconds (1 .. 1000000) and raises the CTA's abort flag, the other warp
 * (on the kernels' default limit) stops on that flag, the tensor memory is
 * freed and FLAG_TIMEOUT (4) is ORed into *flags_dev -- the path every
 * GEMM and attention kernel takes when a wait runs out.  Synchronises the
 * stream and returns GPT2_ERR_TIMEOUT when the flag is set (the expected
 * outcome), GPT2_OK if not, GPT2_ERR_INVALID_ARG for a bad limit, a NULL
 * flags_dev or no tensor-core device, GPT2_ERR_CUDA if the launch fails.
 * The device stays usable afterwards. */
int gpt2_op_wait_probe(int limit_us, int* flags_dev, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* GPT2_B300_OPS_H */
