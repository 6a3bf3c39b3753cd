// Launchers of every kernel on the training step, shared by the model driver
// and the per-operation C ABI.  All launchers enqueue on `st` and return the
// launch status; none allocates memory — scratch comes from the caller.
#pragma once
#include "common.cuh"

#define GPT2_MAX_SEGS 16

// ---- GEMM ------------------------------------------------------------------
// D(m, n) = sum_k A(m, k) * B(n, k) followed by an epilogue.
//   A(m,k) = a_kmajor ? A[m*lda + k] : A[k*lda + m]
//   B(n,k) = b_kmajor ? B[n*ldb + k] : B[k*ldb + n]
enum GemmEpi : int {
  EPI_STORE = 0,     // D[m,n] = acc (+ bias[n])                       (type T)
  EPI_GELU = 1,      // aux[m,n] = acc + bias[n]; D[m,n] = GELU(aux)   (type T)
  EPI_GELU_BWD = 2,  // D[m,n] = acc * GELU'(aux[m,n])                 (type T)
  EPI_ACC_F32 = 3,   // D[m,n] += acc                                  (float)
  // D[m,n] = acc (type T), and for every row m = b*dT + t and 64-column
  // head h: dvec[(b*dH + h)*dT + t] = sum over the head's columns of
  // D[m,n] * aux[m,n] (D as stored), the attention backward's rowsum(dO * O)
  EPI_ROWDOT = 4,
};
struct GemmArgs {
  const void* A; long long lda; int a_kmajor;
  const void* B; long long ldb; int b_kmajor;
  int M, N, K;
  void* D; long long ldd;
  const void* bias;          // [N] of type T or nullptr
  void* aux; long long ldaux;
  int epi;
  // optional fp32 workspace: lets the tensor-core path split K of an
  // EPI_ACC_F32 product across CTAs (partials added in split order afterwards)
  float* ws; size_t ws_floats;
  // batch > 1: that many independent products, item z reading A + z*sA,
  // B + z*sB (and aux + z*sAux) and writing D + z*sD (element strides); no
  // bias, no K split
  int batch; long long sA, sB, sD, sAux;
  float* dvec; int dT, dH;  // EPI_ROWDOT only
  int acc_store;            // EPI_ACC_F32: D = acc instead of D += acc (the first writer of a fresh gradient)
  // EPI_STORE on the tensor-core path (optional): per row and column tile n
  // (gemm_tc_stats_tiles(N) tiles), the statistics of the stored (bf16)
  // values of the columns < stats_cols: m = their maximum, s = the sum of
  // exp(value - m), at rowstats[(row * tiles + n) * 2 + {0, 1}]
  float* rowstats; int stats_cols;
  // EPI_STORE / EPI_GELU on the tensor-core path (optional, no bias): the
  // LayerNorm of A folded into the product.  A is the LayerNorm's input r,
  // B the weight with the LayerNorm gain folded in (W' = W diag(gamma)); the
  // epilogue takes acc = r . W'^T to ln_rstd[m] * (acc - ln_mean[m] * ln_s[n]) +
  // ln_c[n], which is LN(r) . W^T + b with ln_s[n] = sum_k W'[n][k] and
  // ln_c[n] = b[n] + sum_k beta[k] W[n][k] (see lnfold_weights)
  const float* ln_mean; const float* ln_rstd; const float* ln_s; const float* ln_c;
};
// The folded weights of lnfold GEMMs, for `items` stacked weights of N x K:
// Wf = bf16(W diag(gamma)) (row-major [N][K]), s[n] = sum_k of Wf[n][k] as
// stored, c[n] = bias[n] + sum_k beta[k] W[n][k]; item z reads W + z*N*K,
// gamma/beta + z*K, bias + z*N and writes Wf + z*N*K, s/c + z*N.  K % 8 == 0.
// out_rows (default N): rows between items in Wf, s and c (items interleaved
// with other weights' rows)
cudaError_t lnfold_weights(bf16* Wf, float* s, float* c, const float* W, const float* gamma, const float* beta,
                           const float* bias, int items, int N, int K, cudaStream_t st, long long out_rows = 0);
template <typename T> cudaError_t gemm_simt(const GemmArgs& a, cudaStream_t st);
// two EPI_ACC_F32 products with the same N, K and operand majors as one launch
// (the weight gradients of two weight types), or two launches when that does not pay
cudaError_t gemm_tc_grouped(const GemmArgs& a, const GemmArgs& b, int* flags, cudaStream_t st);
int gemm_tc_stats_tiles(int N);  // column tiles of an N-wide tensor-core product
// softmax + cross-entropy of bf16 logit rows from the per-tile statistics of
// the classifier product (see GemmArgs::rowstats): loss and dlogits in place
cudaError_t softmax_ce_from_stats(bf16* logits, float* losses, const int* targets, const float* rowstats, int tiles,
                                  int rows, int V, int Vp, float dloss, int* flags, cudaStream_t st);
// products with at most 32 rows (one position per sequence when decoding):
// both operands K-major, EPI_STORE or EPI_GELU, A small enough for shared memory
template <typename T> bool gemm_skinny_supported(const GemmArgs& a);
template <typename T> cudaError_t gemm_skinny(const GemmArgs& a, cudaStream_t st);
// tcgen05/TMA tensor-core path (bf16 operands); returns cudaErrorNotSupported
// when the shape or layout is outside what the kernel handles.
cudaError_t gemm_tc(const GemmArgs& a, int* flags, cudaStream_t st);
// workspace floats a split-K weight-gradient product of this shape uses on a
// GPU with `sms` SMs (0: no split)
size_t gemm_tc_workspace_floats(int M, int N, int K, int sms);
#define GPT2_NOMINAL_SMS 148
bool gemm_tc_supported(const GemmArgs& a);

// ---- bandwidth kernels ---------------------------------------------------
template <typename T>
cudaError_t encoder_forward(T* out, const int* tok, const T* wte, const T* wpe, int B, int T_, int C,
                            int V, int* flags, cudaStream_t st);
// dwte/dwpe += scatter of dres (fp32 [B*T][C]); keys: pow2(B*T) uint32 keys of
// scratch (accumulate_wpe = 0: dwpe is overwritten instead of added to).
// Positions whose token is outside [0, V) (V <= 65535) add nothing to dwte and
// OR FLAG_TOKEN_RANGE into *flags (flags may be null).
cudaError_t encoder_backward(float* dwte, float* dwpe, const float* dres, const int* tok, int B, int T_,
                             int C, int V, int* flags, uint32_t* keys, cudaStream_t st, int accumulate_wpe = 1);
size_t encoder_backward_scratch_bytes(int BT);
// the same with a larger scratch (BT <= 16384): radix-sorted keys and
// fixed-size chunks of the per-token sums, so no CTA waits on a long run
bool encoder_backward_fast_supported(int BT, int C);
size_t encoder_backward_fast_scratch_bytes(int BT, int C);
cudaError_t encoder_backward_fast(float* dwte, float* dwpe, const float* dres, const int* tok, int B, int T_, int C,
                                  int V, int* flags, void* scratch, cudaStream_t st, int accumulate_wpe = 1);

template <typename T>
cudaError_t residual_layernorm_forward(T* resid_out, T* y, float* mean, float* rstd, const T* a,
                                       const T* b, const T* w, const T* bias, int rows, int C,
                                       cudaStream_t st);
// dres = (accumulate ? dres : 0) + LN backward(dy); dres_c (optional) = T copy.
// With dw, db (and optionally dres_sum): dw += sum_rows dy*xhat, db += sum_rows dy,
// dres_sum += sum_rows of the new dres, through deterministic per-chunk partials
// (partial: ln_backward_partial_floats(rows, C) floats of scratch).
template <typename T>
cudaError_t layernorm_backward(float* dres, T* dres_c, const T* dy, const T* x, const float* mean,
                               const float* rstd, const T* w, int rows, int C, int accumulate, float* dw,
                               float* db, float* dres_sum, float* partial, cudaStream_t st,
                               int* deferred_chunks = nullptr);
// The same with the residual gradient passed along in its own type RT (the
// activation type in the training step, float in fp32 mode):
//   rout = (rin ? rin : 0) + dx; rcopy (T) and rf32 (float) optional copies of
//   the new value (before rounding to RT); rout may be null when rf32 is given;
//   rin may equal rout.  RT = bf16 only with T = bf16.
template <typename T, typename RT>
cudaError_t layernorm_backward_rg(RT* rout, const RT* rin, T* rcopy, float* rf32, const T* dy, const T* x,
                                  const float* mean, const float* rstd, const T* w, int rows, int C, float* dw,
                                  float* db, float* dres_sum, float* partial, cudaStream_t st,
                                  int* deferred_chunks = nullptr);
// With deferred_chunks, layernorm_backward only writes its per-chunk partial
// sums (partial[chunk][3][C]) and stores the chunk count there; the sums are
// added later by reduce_partials, possibly for several calls at once:
// out_o[z*sOut + c] += sum_k partial[z*sPart + (k*nout + o)*C + c] (sPart = 0:
// nchunks*nout*C), chunks in a fixed order.
cudaError_t reduce_partials(float* out0, float* out1, float* out2, const float* partial, int nchunks, int C,
                            int nout, cudaStream_t st, int nbatch = 1, long long sOut = 0, long long sPart = 0,
                            int accumulate = 1);
size_t ln_backward_partial_floats(int rows, int C);
// out[c] += sum_rows X[r*ldx + c]; partial: colsum_partial_floats(rows, cols) floats.
// nbatch > 1: the same for items z = 0..nbatch-1 at out + z*sOut, X + z*sX
// (partial: nbatch times as many floats), in one pair of launches.
template <typename T>
cudaError_t colsum(float* out, const T* X, int rows, int cols, long long ldx, float* partial, cudaStream_t st,
                   int nbatch = 1, long long sOut = 0, long long sX = 0, int accumulate = 1);
size_t colsum_partial_floats(int rows, int cols);
int reduce_chunks(int rows);  // number of row chunks the reductions use

template <typename T>
cudaError_t attention_forward_simt(T* out, float* lse, const T* qkv, int B, int T_, int C, int H,
                                   cudaStream_t st);
template <typename T>
cudaError_t attention_backward_simt(T* dqkv, float* Dbuf, const T* dout, const T* qkv, const T* out,
                                    const float* lse, int B, int T_, int C, int H, cudaStream_t st);

// tcgen05 flash attention (bf16, head size 64, T % 128 == 0).  The backward
// writes D = rowsum(dO * O) into Dbuf [B][H][T] and passes the bf16 dS blocks
// of the causal triangle from its dK/dV kernel to its dQ kernel through dS
// (attention_tc_ds_bytes(B, T, H) bytes, 16-byte aligned; 0 when T % 128).
bool attention_tc_supported(int B, int T, int C, int H);
size_t attention_tc_ds_bytes(int B, int T, int H);
cudaError_t attention_forward_tc(bf16* out, float* lse, const bf16* qkv, int B, int T, int C, int H, int* flags,
                                 cudaStream_t st);
// (d_ready: Dbuf already holds D, e.g. from the EPI_ROWDOT epilogue of the
// GEMM that produced dout)
cudaError_t attention_backward_tc(bf16* dqkv, float* Dbuf, void* dS, const bf16* dout, const bf16* qkv,
                                  const bf16* out, const float* lse, int B, int T, int C, int H, int* flags,
                                  cudaStream_t st, bool d_ready = false);

template <typename T>
cudaError_t softmax_ce(T* logits, float* losses, const int* targets, int rows, int V, int Vp,
                       float dloss, int write_grad, int* flags, cudaStream_t st);
cudaError_t mean_loss(float* loss, const float* losses, int n, cudaStream_t st);

struct AdamSegments {
  int n;
  long long off[GPT2_MAX_SEGS + 1];
  float wd[GPT2_MAX_SEGS];
};
// gscale (optional, device): every gradient is multiplied by *gscale first
cudaError_t adamw(float* p, const float* g, float* m, float* v, bf16* pc, long long n, float lr,
                  float b1, float b2, float eps, float bc1, float bc2, const AdamSegments& seg,
                  const float* gscale, cudaStream_t st);
// out2[0] = ||g||_2, out2[1] = min(1, max_norm / (norm + 1e-6)); partial:
// grad_norm_scratch_floats() floats of scratch; deterministic
cudaError_t grad_norm(const float* g, long long n, float max_norm, float* out2, float* partial, cudaStream_t st);
size_t grad_norm_scratch_floats();
cudaError_t convert_f32_bf16(bf16* out, const float* in, long long n, cudaStream_t st);

template <typename T>
cudaError_t gelu_forward(T* out, const T* in, long long n, cudaStream_t st);
// inference with a KV cache (the cache: qkv [B*Tmax][3C], row b*Tmax + t =
// position t of sequence b): attention of position pos of every sequence over
// keys 0..pos -> out [B][C]; and the sampler over the first V logits of each
// row (temperature 0: argmax, lowest index on ties; else inverse CDF of
// softmax(z / temperature) at coins[row]) -> out_tok [rows]
template <typename T>
cudaError_t decode_attention(T* out, const T* qkv, int B, int Tmax, int pos, int C, int H, cudaStream_t st);
template <typename T>
cudaError_t sample_tokens(int* out_tok, const T* logits, long long ld, int rows, int V, float temperature,
                          const float* coins, cudaStream_t st);
// y = (r - mean) * rstd * w + bias per row (the LayerNorm forward's last step
// on a stored residual row and its stored statistics), rows x C
template <typename T>
cudaError_t layernorm_apply(T* y, const T* r, const float* mean, const float* rstd, const T* w, const T* bias,
                            int rows, int C, cudaStream_t st);
template <typename T>
cudaError_t gelu_backward(T* dinp, const T* inp, const T* dout, long long n, cudaStream_t st);
// One decoding position through every transformer block in one cooperative
// launch (bf16): w = the [L]-stacked bf16 weights ln1w, ln1b, qkvw, qkvb, apw,
// apb, ln2w, ln2b, fcw, fcb, fpw, fpb; qkv the KV cache ([L][B*Tmax][3C]);
// x0 [B][C] holds the embedded rows on entry and the last block's residual on
// return; x1 [B][C], att [B][C], h [B][4C] scratch; bar 4 bytes (zeroed
// here).  A grid barrier that waits too long raises FLAG_TIMEOUT in flags.
bool decode_layers_supported(int B, int C, int H, int Tmax);
cudaError_t decode_layers(const bf16* const* w, bf16* qkv, bf16* x0, bf16* x1, bf16* att, bf16* h, unsigned* bar,
                          int* flags, int L, int B, int C, int H, int Tmax, int pos, cudaStream_t st);
