// Kernel-level C ABI (include/gpt2_ops.h): argument checks and dispatch on
// the activation dtype; all work is in the kernels of kernels_simt.cu and
// gemm_tc.cu.
#include <cmath>

#include "../../include/gpt2_ops.h"
#include "kernels.cuh"

#define ST(s) ((cudaStream_t)(s))
static inline int rc_of(cudaError_t e) {
  return e == cudaSuccess ? GPT2_OK : (e == cudaErrorInvalidValue || e == cudaErrorNotSupported ? GPT2_ERR_INVALID_ARG : GPT2_ERR_CUDA);
}
static inline bool bad_dtype(int d) { return d != GPT2_PRECISION_FP32 && d != GPT2_PRECISION_BF16; }
static inline bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

extern "C" {

int gpt2_op_encoder_forward(int dtype, void* out, const int32_t* tokens, const void* wte, const void* wpe, int B,
                            int T, int C, int V, int* flags_dev, void* stream) {
  if (bad_dtype(dtype) || !out || !tokens || !wte || !wpe || !flags_dev || B <= 0 || T <= 0 || V <= 0) return GPT2_ERR_INVALID_ARG;
  if (C <= 0 || C % (dtype ? 8 : 4) || !aligned16(out) || !aligned16(wte) || !aligned16(wpe)) return GPT2_ERR_INVALID_ARG;
  if (dtype == GPT2_PRECISION_BF16)
    return rc_of(encoder_forward<bf16>((bf16*)out, tokens, (const bf16*)wte, (const bf16*)wpe, B, T, C, V, flags_dev, ST(stream)));
  return rc_of(encoder_forward<float>((float*)out, tokens, (const float*)wte, (const float*)wpe, B, T, C, V, flags_dev, ST(stream)));
}

size_t gpt2_op_encoder_backward_scratch_bytes(int B, int T, int C) {
  if (B <= 0 || T <= 0 || (long long)B * T > 32768) return 0;
  if (C > 0 && encoder_backward_fast_supported(B * T, C)) return encoder_backward_fast_scratch_bytes(B * T, C);
  return encoder_backward_scratch_bytes(B * T);
}

int gpt2_op_encoder_backward(float* dwte, float* dwpe, const float* dres, const int32_t* tokens, int B, int T, int C,
                             int V, int* flags_dev, void* scratch, size_t scratch_bytes, void* stream) {
  if (!dwte || !dwpe || !dres || !tokens || !scratch || B <= 0 || T <= 0 || C <= 0 || C % 4) return GPT2_ERR_INVALID_ARG;
  if (V <= 0 || V > 65535) return GPT2_ERR_INVALID_ARG;
  if ((long long)B * T > 32768 || scratch_bytes < gpt2_op_encoder_backward_scratch_bytes(B, T, C)) return GPT2_ERR_INVALID_ARG;
  if (encoder_backward_fast_supported(B * T, C))
    return rc_of(encoder_backward_fast(dwte, dwpe, dres, tokens, B, T, C, V, flags_dev, scratch, ST(stream)));
  return rc_of(encoder_backward(dwte, dwpe, dres, tokens, B, T, C, V, flags_dev, (uint32_t*)scratch, ST(stream)));
}

int gpt2_op_residual_layernorm_forward(int dtype, void* resid_out, void* y, float* mean, float* rstd, const void* a,
                                       const void* b, const void* w, const void* bias, int rows, int C, void* stream) {
  if (bad_dtype(dtype) || !y || !mean || !rstd || !a || !w || !bias || rows <= 0 || C <= 0) return GPT2_ERR_INVALID_ARG;
  if (C % (dtype ? 8 : 4) || C > 2048 || (b && !resid_out)) return GPT2_ERR_INVALID_ARG;
  if (dtype == GPT2_PRECISION_BF16)
    return rc_of(residual_layernorm_forward<bf16>((bf16*)resid_out, (bf16*)y, mean, rstd, (const bf16*)a, (const bf16*)b,
                                                  (const bf16*)w, (const bf16*)bias, rows, C, ST(stream)));
  return rc_of(residual_layernorm_forward<float>((float*)resid_out, (float*)y, mean, rstd, (const float*)a,
                                                 (const float*)b, (const float*)w, (const float*)bias, rows, C, ST(stream)));
}

size_t gpt2_op_layernorm_backward_scratch_bytes(int rows, int C) {
  if (rows <= 0 || C <= 0) return 0;
  return ln_backward_partial_floats(rows, C) * sizeof(float);
}

int gpt2_op_layernorm_backward(int dtype, float* dres, void* dres_c, const void* dy, const void* x, const float* mean,
                               const float* rstd, const void* w, float* dw, float* db, float* dres_sum, int rows,
                               int C, int accumulate, void* scratch, size_t scratch_bytes, void* stream) {
  if (bad_dtype(dtype) || !dres || !dy || !x || !mean || !rstd || !w || rows <= 0 || C <= 0) return GPT2_ERR_INVALID_ARG;
  if (C % (dtype ? 8 : 4) || C > 2048) return GPT2_ERR_INVALID_ARG;
  const bool sums = dw || db || dres_sum;
  if (sums && (!dw || !db || !scratch || scratch_bytes < gpt2_op_layernorm_backward_scratch_bytes(rows, C)))
    return GPT2_ERR_INVALID_ARG;
  float* part = sums ? (float*)scratch : nullptr;
  if (dtype == GPT2_PRECISION_BF16)
    return rc_of(layernorm_backward<bf16>(dres, (bf16*)dres_c, (const bf16*)dy, (const bf16*)x, mean, rstd,
                                          (const bf16*)w, rows, C, accumulate, dw, db, dres_sum, part, ST(stream)));
  return rc_of(layernorm_backward<float>(dres, (float*)dres_c, (const float*)dy, (const float*)x, mean, rstd,
                                         (const float*)w, rows, C, accumulate, dw, db, dres_sum, part, ST(stream)));
}

int gpt2_op_layernorm_backward_rg(int dtype, void* dres_out, const void* dres_in, float* dres_f32, const void* dy,
                                  const void* x, const float* mean, const float* rstd, const void* w, float* dw,
                                  float* db, float* dres_sum, int rows, int C, void* scratch, size_t scratch_bytes,
                                  void* stream) {
  if (bad_dtype(dtype) || (!dres_out && !dres_f32) || !dy || !x || !mean || !rstd || !w || rows <= 0 || C <= 0)
    return GPT2_ERR_INVALID_ARG;
  if (C % (dtype ? 8 : 4) || C > 2048) return GPT2_ERR_INVALID_ARG;
  for (const void* q : {(const void*)dres_out, dres_in, (const void*)dres_f32, dy, x, w})
    if (!aligned16(q)) return GPT2_ERR_INVALID_ARG;
  const bool sums = dw || db || dres_sum;
  if (sums && (!dw || !db || !scratch || scratch_bytes < gpt2_op_layernorm_backward_scratch_bytes(rows, C)))
    return GPT2_ERR_INVALID_ARG;
  float* part = sums ? (float*)scratch : nullptr;
  if (dtype == GPT2_PRECISION_BF16)
    return rc_of(layernorm_backward_rg<bf16, bf16>((bf16*)dres_out, (const bf16*)dres_in, nullptr, dres_f32,
                                                   (const bf16*)dy, (const bf16*)x, mean, rstd, (const bf16*)w, rows,
                                                   C, dw, db, dres_sum, part, ST(stream)));
  return rc_of(layernorm_backward_rg<float, float>((float*)dres_out, (const float*)dres_in, nullptr, dres_f32,
                                                   (const float*)dy, (const float*)x, mean, rstd, (const float*)w,
                                                   rows, C, dw, db, dres_sum, part, ST(stream)));
}

int gpt2_op_lnfold_weights(void* Wf, float* s, float* c, const float* W, const float* gamma, const float* beta,
                           const float* bias, int items, int N, int K, void* stream) {
  if (!Wf || !s || !c || !W || !gamma || !beta || items <= 0 || N <= 0 || K <= 0 || K % 8) return GPT2_ERR_INVALID_ARG;
  for (const void* q : {(const void*)Wf, (const void*)W, (const void*)gamma, (const void*)beta})
    if (!aligned16(q)) return GPT2_ERR_INVALID_ARG;
  return rc_of(lnfold_weights((bf16*)Wf, s, c, W, gamma, beta, bias, items, N, K, ST(stream)));
}

int gpt2_op_matmul_lnfold(const void* R, long long ldr, const float* mean, const float* rstd, const void* Wf,
                          long long ldw, const float* s, const float* c, int M, int N, int K, void* D, long long ldd,
                          void* aux, long long ldaux, int* flags_dev, void* stream) {
  if (!R || !mean || !rstd || !Wf || !s || !c || !D || !flags_dev || M <= 0 || N <= 0 || K <= 0)
    return GPT2_ERR_INVALID_ARG;
  GemmArgs a{R, ldr, 1, Wf, ldw, 1, M, N, K, D, ldd, nullptr, aux, ldaux, aux ? EPI_GELU : EPI_STORE};
  a.ln_mean = mean;
  a.ln_rstd = rstd;
  a.ln_s = s;
  a.ln_c = c;
  if (!gemm_tc_supported(a)) return GPT2_ERR_INVALID_ARG;
  return rc_of(gemm_tc(a, flags_dev, ST(stream)));
}

size_t gpt2_op_matmul_workspace_bytes(int M, int N, int K, int epilogue) {
  if (M <= 0 || N <= 0 || K <= 0 || epilogue != EPI_ACC_F32) return 0;
  return gemm_tc_workspace_floats(M, N, K, GPT2_NOMINAL_SMS) * sizeof(float);
}

int gpt2_op_matmul(int dtype, const void* A, long long lda, int a_kmajor, const void* B, long long ldb, int b_kmajor,
                   int M, int N, int K, void* D, long long ldd, const void* bias, void* aux, long long ldaux,
                   int epilogue, int path, int* flags_dev, void* workspace, size_t workspace_bytes,
                   void* stream) {
  if (bad_dtype(dtype) || !A || !B || !D || M <= 0 || N <= 0 || K <= 0 || epilogue < 0 || epilogue > 3) return GPT2_ERR_INVALID_ARG;
  if ((epilogue == EPI_GELU || epilogue == EPI_GELU_BWD) && !aux) return GPT2_ERR_INVALID_ARG;
  if (workspace && ((uintptr_t)workspace & 15)) return GPT2_ERR_INVALID_ARG;
  GemmArgs a{A, lda, a_kmajor, B, ldb, b_kmajor, M, N, K, D, ldd, bias, aux, ldaux, epilogue,
             (float*)workspace, workspace ? workspace_bytes / sizeof(float) : 0};
  // path 0 with at most 32 rows: the few-row SIMT kernel (as the decode step uses)
  if (path == 0 && (dtype == GPT2_PRECISION_BF16 ? gemm_skinny_supported<bf16>(a) : gemm_skinny_supported<float>(a)))
    return rc_of(dtype == GPT2_PRECISION_BF16 ? gemm_skinny<bf16>(a, ST(stream)) : gemm_skinny<float>(a, ST(stream)));
  // (path 0 takes the tensor cores only with flags_dev, which their bounded waits report into)
  if (path == 2 || (path == 0 && dtype == GPT2_PRECISION_BF16 && flags_dev && gemm_tc_supported(a))) {
    if (dtype != GPT2_PRECISION_BF16 || !flags_dev || !gemm_tc_supported(a)) return GPT2_ERR_INVALID_ARG;
    return rc_of(gemm_tc(a, flags_dev, ST(stream)));
  }
  if (dtype == GPT2_PRECISION_BF16) return rc_of(gemm_simt<bf16>(a, ST(stream)));
  return rc_of(gemm_simt<float>(a, ST(stream)));
}

int gpt2_op_matmul_batched(int dtype, int batch, const void* A, long long lda, long long sA, int a_kmajor,
                           const void* B, long long ldb, long long sB, int b_kmajor, int M, int N, int K, void* D,
                           long long ldd, long long sD, void* aux, long long ldaux, long long sAux, int epilogue,
                           int path, int* flags_dev, void* stream) {
  if (bad_dtype(dtype) || batch <= 0 || !A || !B || !D || M <= 0 || N <= 0 || K <= 0 || epilogue < 0 || epilogue > 3)
    return GPT2_ERR_INVALID_ARG;
  if ((epilogue == EPI_GELU || epilogue == EPI_GELU_BWD) && !aux) return GPT2_ERR_INVALID_ARG;
  if (sA < 0 || sB < 0 || sD < 0 || sAux < 0 || path < 0 || path > 2) return GPT2_ERR_INVALID_ARG;
  GemmArgs a{A, lda, a_kmajor, B, ldb, b_kmajor, M, N, K, D, ldd, nullptr, aux, ldaux, epilogue,
             nullptr, 0, batch, sA, sB, sD, sAux};
  if (path == 2 || (path == 0 && dtype == GPT2_PRECISION_BF16 && gemm_tc_supported(a))) {
    if (dtype != GPT2_PRECISION_BF16 || !flags_dev || !gemm_tc_supported(a)) return GPT2_ERR_INVALID_ARG;
    return rc_of(gemm_tc(a, flags_dev, ST(stream)));
  }
  if (dtype == GPT2_PRECISION_BF16) return rc_of(gemm_simt<bf16>(a, ST(stream)));
  return rc_of(gemm_simt<float>(a, ST(stream)));
}

int gpt2_op_matmul_rowdot(const void* dY, long long ldy, const void* W, long long ldw, int M, int N, int K, void* dX,
                          long long ldx, const void* O, long long ldo, float* D, int T, int H, int* flags_dev,
                          void* stream) {
  if (!dY || !W || !dX || !O || !D || !flags_dev || M <= 0 || N <= 0 || K <= 0 || T <= 0 || H <= 0)
    return GPT2_ERR_INVALID_ARG;
  GemmArgs a{dY, ldy, 1, W, ldw, 0, M, K, N, dX, ldx, nullptr, const_cast<void*>(O), ldo, EPI_ROWDOT,
             nullptr, 0, 1, 0, 0, 0, 0, D, T, H};
  if (!gemm_tc_supported(a)) return GPT2_ERR_INVALID_ARG;
  return rc_of(gemm_tc(a, flags_dev, ST(stream)));
}

int gpt2_op_logit_stats_tiles(int N) { return N > 0 ? gemm_tc_stats_tiles(N) : 0; }

int gpt2_op_matmul_logit_stats(const void* A, long long lda, const void* B, long long ldb, int M, int N, int K,
                               void* D, long long ldd, float* stats, int stats_cols, int* flags_dev, void* stream) {
  if (!A || !B || !D || !stats || !flags_dev || M <= 0 || N <= 0 || K <= 0 || stats_cols <= 0 ||
      ((uintptr_t)stats & 7))
    return GPT2_ERR_INVALID_ARG;
  GemmArgs a{A, lda, 1, B, ldb, 1, M, N, K, D, ldd, nullptr, nullptr, 0, EPI_STORE};
  a.rowstats = stats;
  a.stats_cols = stats_cols;
  if (!gemm_tc_supported(a)) return GPT2_ERR_INVALID_ARG;
  return rc_of(gemm_tc(a, flags_dev, ST(stream)));
}

int gpt2_op_softmax_crossentropy_stats(void* logits, float* losses, const int32_t* targets, const float* stats,
                                       int rows, int V, int Vp, float dloss, int* flags_dev, void* stream) {
  if (!logits || !losses || !targets || !stats || !flags_dev || rows <= 0 || V <= 0 || Vp < V) return GPT2_ERR_INVALID_ARG;
  return rc_of(softmax_ce_from_stats((bf16*)logits, losses, targets, stats, gemm_tc_stats_tiles(Vp), rows, V, Vp,
                                     dloss, flags_dev, ST(stream)));
}

int gpt2_op_attention_forward(int dtype, void* out, float* lse, const void* qkv, int B, int T, int C, int H, int path,
                              int* flags_dev, void* stream) {
  if (bad_dtype(dtype) || !out || !lse || !qkv || B <= 0 || T <= 0 || C <= 0 || H <= 0 || C % H) return GPT2_ERR_INVALID_ARG;
  if (path < 0 || path > 2) return GPT2_ERR_INVALID_ARG;
  const bool tc = dtype == GPT2_PRECISION_BF16 && flags_dev && attention_tc_supported(B, T, C, H);
  if (path == 2 && !tc) return GPT2_ERR_INVALID_ARG;
  if (tc && path != 1)
    return rc_of(attention_forward_tc((bf16*)out, lse, (const bf16*)qkv, B, T, C, H, flags_dev, ST(stream)));
  if (dtype == GPT2_PRECISION_BF16)
    return rc_of(attention_forward_simt<bf16>((bf16*)out, lse, (const bf16*)qkv, B, T, C, H, ST(stream)));
  return rc_of(attention_forward_simt<float>((float*)out, lse, (const float*)qkv, B, T, C, H, ST(stream)));
}

// D [B][H][T] fp32, padded to 1 KB, then (T % 128 == 0) the dS block buffer
// of the tensor-core backward
static size_t attn_d_bytes(int B, int T, int H) { return ((size_t)B * T * H * sizeof(float) + 1023) & ~(size_t)1023; }
size_t gpt2_op_attention_backward_scratch_bytes(int B, int T, int H) {
  if (B <= 0 || T <= 0 || H <= 0) return 0;
  return attn_d_bytes(B, T, H) + attention_tc_ds_bytes(B, T, H);
}

int gpt2_op_attention_backward(int dtype, void* dqkv, const void* dout, const void* qkv, const void* out,
                               const float* lse, int B, int T, int C, int H, int path, int* flags_dev, void* scratch,
                               size_t scratch_bytes, void* stream) {
  if (bad_dtype(dtype) || !dqkv || !dout || !qkv || !out || !lse || !scratch || B <= 0 || T <= 0 || C <= 0 || H <= 0 ||
      C % H)
    return GPT2_ERR_INVALID_ARG;
  if (path < 0 || path > 2) return GPT2_ERR_INVALID_ARG;
  if (scratch_bytes < gpt2_op_attention_backward_scratch_bytes(B, T, H)) return GPT2_ERR_INVALID_ARG;
  const bool tc = dtype == GPT2_PRECISION_BF16 && flags_dev && attention_tc_supported(B, T, C, H);
  if (path == 2 && !tc) return GPT2_ERR_INVALID_ARG;
  if (tc && path != 1)
    return rc_of(attention_backward_tc((bf16*)dqkv, (float*)scratch, (uint8_t*)scratch + attn_d_bytes(B, T, H),
                                       (const bf16*)dout, (const bf16*)qkv, (const bf16*)out, lse, B, T, C, H,
                                       flags_dev, ST(stream)));
  if (dtype == GPT2_PRECISION_BF16)
    return rc_of(attention_backward_simt<bf16>((bf16*)dqkv, (float*)scratch, (const bf16*)dout, (const bf16*)qkv,
                                               (const bf16*)out, lse, B, T, C, H, ST(stream)));
  return rc_of(attention_backward_simt<float>((float*)dqkv, (float*)scratch, (const float*)dout, (const float*)qkv,
                                              (const float*)out, lse, B, T, C, H, ST(stream)));
}

int gpt2_op_softmax_crossentropy(int dtype, void* logits, float* losses, const int32_t* targets, int rows, int V,
                                 int Vp, float dloss, int write_grad, int* flags_dev, void* stream) {
  if (bad_dtype(dtype) || !logits || !losses || !targets || !flags_dev || rows <= 0 || V <= 0 || Vp < V) return GPT2_ERR_INVALID_ARG;
  if (Vp % (dtype ? 8 : 4)) return GPT2_ERR_INVALID_ARG;
  if (dtype == GPT2_PRECISION_BF16)
    return rc_of(softmax_ce<bf16>((bf16*)logits, losses, targets, rows, V, Vp, dloss, write_grad, flags_dev, ST(stream)));
  return rc_of(softmax_ce<float>((float*)logits, losses, targets, rows, V, Vp, dloss, write_grad, flags_dev, ST(stream)));
}

int gpt2_op_adamw(float* p, const float* g, float* m, float* v, void* p_bf16, long long n, float lr, float b1,
                  float b2, float eps, float wd, int t, const float* gscale_dev, void* stream) {
  if (!p || !g || !m || !v || n <= 0 || n % 4 || t < 1) return GPT2_ERR_INVALID_ARG;
  AdamSegments seg{};
  seg.n = 1;
  seg.off[0] = 0;
  seg.off[1] = n;
  seg.wd[0] = wd;
  float bc1 = (float)(1.0 - std::pow((double)b1, (double)t));
  float bc2 = (float)(1.0 - std::pow((double)b2, (double)t));
  return rc_of(adamw(p, g, m, v, (bf16*)p_bf16, n, lr, b1, b2, eps, bc1, bc2, seg, gscale_dev, ST(stream)));
}

size_t gpt2_op_grad_norm_scratch_bytes(void) { return grad_norm_scratch_floats() * sizeof(float); }

int gpt2_op_grad_norm(const float* g, long long n, float max_norm, float* out2_dev, void* scratch,
                      size_t scratch_bytes, void* stream) {
  if (!g || !out2_dev || !scratch || n <= 0 || !(max_norm > 0.f) || !aligned16(g)) return GPT2_ERR_INVALID_ARG;
  if (scratch_bytes < gpt2_op_grad_norm_scratch_bytes()) return GPT2_ERR_INVALID_ARG;
  return rc_of(grad_norm(g, n, max_norm, out2_dev, (float*)scratch, ST(stream)));
}

int gpt2_op_gelu_forward(int dtype, void* out, const void* in, long long n, void* stream) {
  if (bad_dtype(dtype) || !out || !in || n <= 0) return GPT2_ERR_INVALID_ARG;
  if (dtype == GPT2_PRECISION_BF16) return rc_of(gelu_forward<bf16>((bf16*)out, (const bf16*)in, n, ST(stream)));
  return rc_of(gelu_forward<float>((float*)out, (const float*)in, n, ST(stream)));
}

int gpt2_op_gelu_backward(int dtype, void* dinp, const void* inp, const void* dout, long long n, void* stream) {
  if (bad_dtype(dtype) || !dinp || !inp || !dout || n <= 0) return GPT2_ERR_INVALID_ARG;
  if (dtype == GPT2_PRECISION_BF16)
    return rc_of(gelu_backward<bf16>((bf16*)dinp, (const bf16*)inp, (const bf16*)dout, n, ST(stream)));
  return rc_of(gelu_backward<float>((float*)dinp, (const float*)inp, (const float*)dout, n, ST(stream)));
}

size_t gpt2_op_colsum_scratch_bytes(int rows, int cols) {
  if (rows <= 0 || cols <= 0) return 0;
  return colsum_partial_floats(rows, cols) * sizeof(float);
}

int gpt2_op_colsum(int dtype, float* out, const void* X, int rows, int cols, long long ldx, void* scratch,
                   size_t scratch_bytes, void* stream) {
  if (bad_dtype(dtype) || !out || !X || !scratch || rows <= 0 || cols <= 0 || ldx < cols) return GPT2_ERR_INVALID_ARG;
  if (scratch_bytes < gpt2_op_colsum_scratch_bytes(rows, cols)) return GPT2_ERR_INVALID_ARG;
  if (cols % (dtype ? 8 : 4) || ldx % (dtype ? 8 : 4) || !aligned16(X)) return GPT2_ERR_INVALID_ARG;
  if (dtype == GPT2_PRECISION_BF16)
    return rc_of(colsum<bf16>(out, (const bf16*)X, rows, cols, ldx, (float*)scratch, ST(stream)));
  return rc_of(colsum<float>(out, (const float*)X, rows, cols, ldx, (float*)scratch, ST(stream)));
}

}  // extern "C"
