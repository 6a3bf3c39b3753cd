// The GPT-2 training step behind the C ABI of include/gpt2.h.
//
// gpt2_forward / gpt2_backward / gpt2_adamw_step enqueue the layer kernels in
// the order of "llm.c: GPT-2 training in plain C, with every gradient written
// by hand", §2 How the code works: encoder, then per block
// layernorm -> qkv matmul -> attention -> attention projection -> residual ->
// layernorm -> fc matmul -> GELU -> fc projection -> residual, final
// layernorm, tied classifier, softmax + cross-entropy; the backward runs the
// same list in reverse.  Every residual add is fused into the next LayerNorm
// and the classifier's softmax/cross-entropy backward is fused into its
// forward ("llm.c's Origin and the Future of LLM Compilers", [13:50]).
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "kernels.cuh"
#include "model_layout.h"

extern void gpt2_count_launches(int n);
extern unsigned long long gpt2_total_launches();

struct gpt2 {
  gpt2_config cfg;
  // inference: positions 0..cache_len-1 of every sequence are in the KV cache
  // (the qkv activations); the last logits are B rows ld elements apart
  int cache_len = 0;
  size_t last_logits = 0;  // byte offset in the buffer
  long long last_ld = 0;
  ParamLayout pl;
  BufferLayout bl;
  char* base = nullptr;
  cudaStream_t st = nullptr;
  int BT = 0;
  bool have_targets = false;   // last forward computed loss + dlogits
  bool logits_valid = false;   // last forward kept the logits
  bool loss_valid = false;
  const int32_t* fwd_tokens = nullptr;
  bool clip_pending = false;   // gpt2_clip_grad_norm ran since the last AdamW step
  // captured zero_grad + forward + backward (gpt2_graph_step), for these token pointers
  cudaGraphExec_t gexec = nullptr;
  const int32_t* g_tok = nullptr;
  const int32_t* g_tgt = nullptr;
  unsigned long long g_launches = 0;  // kernels in the captured graph
  std::string err;
  // GEMM event trace (roofline measurement)
  bool prof_on = false;
  std::vector<cudaEvent_t> prof_ev;  // pairs
  std::vector<double> prof_flops;
  size_t prof_n = 0;
  template <typename P> P* at(size_t off) const { return reinterpret_cast<P*>(base + off); }
};

static std::string g_create_err;

#define FAIL(m, code, ...)                                          \
  do {                                                              \
    char _b[512];                                                   \
    snprintf(_b, sizeof _b, __VA_ARGS__);                           \
    if (m) (m)->err = _b; else g_create_err = _b;                   \
    return code;                                                    \
  } while (0)
#define CK(m, call)                                                                       \
  do {                                                                                    \
    cudaError_t _e = (call);                                                              \
    if (_e != cudaSuccess)                                                                \
      FAIL(m, GPT2_ERR_CUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(_e), __FILE__, __LINE__); \
  } while (0)

// --------------------------------------------------------------------------
// config validation and the planner
// --------------------------------------------------------------------------
int validate_config(const gpt2_config& c, const char** why) {
  *why = "";
  if (c.L <= 0 || c.C <= 0 || c.H <= 0 || c.max_T <= 0 || c.V <= 0 || c.Vp <= 0 || c.B <= 0 || c.T <= 0)
    return *why = "all sizes must be positive", GPT2_ERR_INVALID_CONFIG;
  if (c.C % c.H) return *why = "C must be a multiple of H", GPT2_ERR_INVALID_CONFIG;
  if (c.Vp < c.V) return *why = "Vp must be >= V", GPT2_ERR_INVALID_CONFIG;
  if (c.T > c.max_T) return *why = "T must be <= max_T", GPT2_ERR_INVALID_CONFIG;
  if (c.C > 2048) return *why = "C must be <= 2048", GPT2_ERR_INVALID_CONFIG;
  if (c.V > 65535) return *why = "V must be <= 65535", GPT2_ERR_INVALID_CONFIG;
  if ((long long)c.B * c.T > 32768) return *why = "B*T must be <= 32768", GPT2_ERR_INVALID_CONFIG;
  int hd = c.C / c.H;
  if (c.precision == GPT2_PRECISION_FP32) {
    if (c.C % 4 || c.Vp % 4) return *why = "fp32 mode needs C % 4 == 0 and Vp % 4 == 0", GPT2_ERR_INVALID_CONFIG;
    if (hd > 128) return *why = "head size must be <= 128", GPT2_ERR_INVALID_CONFIG;
  } else if (c.precision == GPT2_PRECISION_BF16) {
    if (c.C % 64) return *why = "bf16 mode needs C % 64 == 0", GPT2_ERR_INVALID_CONFIG;
    if (hd != 64) return *why = "bf16 mode needs head size 64", GPT2_ERR_INVALID_CONFIG;
    if (c.T % 128) return *why = "bf16 mode needs T % 128 == 0", GPT2_ERR_INVALID_CONFIG;
    if (((long long)c.B * c.T) % 128) return *why = "bf16 mode needs B*T % 128 == 0", GPT2_ERR_INVALID_CONFIG;
    if (c.Vp % 128) return *why = "bf16 mode needs Vp % 128 == 0", GPT2_ERR_INVALID_CONFIG;
  } else {
    return *why = "precision must be GPT2_PRECISION_FP32 or GPT2_PRECISION_BF16", GPT2_ERR_INVALID_CONFIG;
  }
  if (c.recompute < 0 || c.recompute > 2) return *why = "recompute must be 0, 1 or 2", GPT2_ERR_INVALID_CONFIG;
  if (c.ln_fold < 0 || c.ln_fold > 1) return *why = "ln_fold must be 0 or 1", GPT2_ERR_INVALID_CONFIG;
  if (c.ln_fold && (c.precision != GPT2_PRECISION_BF16 || c.recompute != 2))
    return *why = "ln_fold needs bf16 precision and recompute 2", GPT2_ERR_INVALID_CONFIG;
  return GPT2_OK;
}

BufferLayout buffer_layout(const gpt2_config& c) {
  BufferLayout b{};
  ParamLayout pl = param_layout(c);
  size_t es = c.precision == GPT2_PRECISION_BF16 ? 2 : 4;  // activation element size
  size_t L = c.L, C = c.C, BT = (size_t)c.B * c.T;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t r = o;
    o += (bytes + 255) & ~(size_t)255;
    return r;
  };
  b.params = take(pl.total * 4);
  b.grads = take(pl.total * 4);
  b.m = take(pl.total * 4);
  b.v = take(pl.total * 4);
  b.pbf = c.precision == GPT2_PRECISION_BF16 ? take(pl.total * 2) : 0;
  // recompute 2 keeps one LayerNorm output, 1 and 2 keep one GELU output and
  // one layer's output gradients (the weight gradients then run in the layer loop)
  const size_t n_ln = c.recompute >= 2 ? 1 : 2 * L + 1, n_gelu = c.recompute >= 1 ? 1 : L;
  const size_t n_dlayer = c.recompute >= 1 ? 1 : L;
  b.resid = take((2 * L + 1) * BT * C * es);
  b.ln = take(n_ln * BT * C * es);
  b.ln_mean = take((2 * L + 1) * BT * 4);
  b.ln_rstd = take((2 * L + 1) * BT * 4);
  b.qkv = take(L * BT * 3 * C * es);
  b.atty = take(L * BT * C * es);
  b.lse = take(L * BT * c.H * 4);
  b.fch = take(L * BT * 4 * C * es);
  b.fchg = take(n_gelu * BT * 4 * C * es);
  b.proj = take(BT * C * es);
  b.logits = take(BT * (size_t)c.Vp * es);
  // per row and 256-column tile of the logits, (max, sum of exp) from the
  // classifier product's epilogue (bf16 mode), read by the softmax
  b.lstats = c.precision == GPT2_PRECISION_BF16 ? take(BT * (size_t)gemm_tc_stats_tiles(c.Vp) * 2 * 4) : 0;
  b.losses = take(BT * 4);
  b.loss = take(256);
  b.dres = take(BT * C * 4);
  // output gradients every layer keeps until the weight gradients of all
  // layers are taken together after the backward pass: the residual gradient
  // entering the fc projection and the attention projection ([L][2][BT][C]),
  // the fc output gradient ([L][BT][4C]) and the qkv gradient ([L][BT][3C])
  b.dresc = take(n_dlayer * 2 * BT * C * es);
  b.dfch = take(n_dlayer * BT * 4 * C * es);
  b.dqkv = take(n_dlayer * BT * 3 * C * es);
  b.dsmall = take(BT * C * es);
  b.attD = take(BT * c.H * 4);
  // dS blocks of the tensor-core attention backward (by shape alone, so the
  // size does not depend on the machine the layout is computed on)
  b.attS = c.precision == GPT2_PRECISION_BF16 && c.C == 64 * c.H ? take(attention_tc_ds_bytes(c.B, c.T, c.H)) : 0;
  // the parameter-sum partials of all 2L+1 LayerNorm backwards (reduced
  // together after the layer loop), later the column-sum partials of all
  // layers' fc output gradients
  // (with recompute the per-layer column sums use the space after the LayerNorm slots)
  const size_t ln_part = (2 * L + 1) * ln_backward_partial_floats((int)BT, (int)C);
  const size_t cs_part = n_dlayer * colsum_partial_floats((int)BT, 4 * (int)C);
  b.partial = take((c.recompute >= 1 ? ln_part + cs_part : std::max(ln_part, cs_part)) * sizeof(float));
  b.keys = take(std::max(encoder_backward_scratch_bytes((int)BT), encoder_backward_fast_scratch_bytes((int)BT, (int)C)));
  // split-K workspace of the classifier weight gradient (bf16 mode)
  b.ws_floats = 0;
  if (c.precision == GPT2_PRECISION_BF16) {
    const int iBT = (int)BT, iC = (int)C;
    // (without recompute the per-layer weight gradients run batched over the
    // layers, unsplit; with it they run one layer at a time and may split K)
    b.ws_floats = gemm_tc_workspace_floats(c.Vp, iC, iBT, GPT2_NOMINAL_SMS);
    if (c.recompute >= 1) {
      const int shapes[4][2] = {{iC, 4 * iC}, {4 * iC, iC}, {iC, iC}, {3 * iC, iC}};
      for (auto& sh : shapes)
        b.ws_floats = std::max(b.ws_floats, gemm_tc_workspace_floats(sh[0], sh[1], iBT, GPT2_NOMINAL_SMS));
    }
  }
  b.ws = take(std::max<size_t>(b.ws_floats, 1) * sizeof(float));
  b.gnorm = take((2 + grad_norm_scratch_floats()) * sizeof(float));  // norm, clip factor, chunk sums
  b.flags = take(256);
  b.tok = take(BT * 4);
  b.tgt = take(BT * 4);
  // inference with a KV cache, one new position per sequence: residual
  // ping-pong, LayerNorm output, attention output, projection output (B x C
  // each), fc pre-activation and GELU (B x 4C), logits (B x Vp), stats (2 x B fp32)
  b.dec = take(((5 + 8) * (size_t)c.B * C + (size_t)c.B * c.Vp) * es + 2 * (size_t)c.B * 4);
  // ln_fold: per layer the qkv (3C rows) then the fc (4C rows) weight with
  // the LayerNorm gain folded in, and their column sums s, c
  b.wfold = c.ln_fold ? take(L * 7 * C * C * 2) : 0;
  b.fold_s = c.ln_fold ? take(L * 7 * C * 4) : 0;
  b.fold_c = c.ln_fold ? take(L * 7 * C * 4) : 0;
  b.decbar = take(256);
  b.total = o;
  return b;
}

// --------------------------------------------------------------------------
// typed views and the step
// --------------------------------------------------------------------------
template <typename T>
struct Step {
  gpt2* m;
  const gpt2_config& c;
  size_t BT, C, L;
  explicit Step(gpt2* mm) : m(mm), c(mm->cfg), BT((size_t)mm->BT), C(mm->cfg.C), L(mm->cfg.L) {}

  // compute copy of a parameter tensor (bf16 copy in bf16 mode, master fp32 otherwise)
  const T* W(int t, size_t layer = 0, size_t per_layer = 0) const {
    size_t e = m->pl.off[t] + layer * per_layer;
    if (c.precision == GPT2_PRECISION_BF16) return m->at<T>(m->bl.pbf) + e;
    return m->at<T>(m->bl.params) + e;
  }
  float* G(int t, size_t layer = 0, size_t per_layer = 0) const {
    return m->at<float>(m->bl.grads) + m->pl.off[t] + layer * per_layer;
  }
  T* resid(size_t i) const { return m->at<T>(m->bl.resid) + i * BT * C; }
  // LayerNorm output i (one buffer for all i under recompute 2)
  T* ln(size_t i) const { return m->at<T>(m->bl.ln) + (c.recompute >= 2 ? 0 : i) * BT * C; }
  float* mean(size_t i) const { return m->at<float>(m->bl.ln_mean) + i * BT; }
  float* rstd(size_t i) const { return m->at<float>(m->bl.ln_rstd) + i * BT; }
  T* qkv(size_t l) const { return m->at<T>(m->bl.qkv) + l * BT * 3 * C; }
  T* atty(size_t l) const { return m->at<T>(m->bl.atty) + l * BT * C; }
  float* lse(size_t l) const { return m->at<float>(m->bl.lse) + l * BT * c.H; }
  T* fch(size_t l) const { return m->at<T>(m->bl.fch) + l * BT * 4 * C; }
  T* fchg(size_t l) const { return m->at<T>(m->bl.fchg) + (c.recompute >= 1 ? 0 : l) * BT * 4 * C; }
  T* proj() const { return m->at<T>(m->bl.proj); }
  T* logits() const { return m->at<T>(m->bl.logits); }
  float* losses() const { return m->at<float>(m->bl.losses); }
  float* dres() const { return m->at<float>(m->bl.dres); }
  // operand copy of dres for the GEMMs (== dres in fp32 mode)
  // copy of the residual gradient that enters layer l's fc projection (k = 0)
  // or attention projection (k = 1)
  // (one layer's worth under recompute >= 1)
  size_t dl(size_t l) const { return c.recompute >= 1 ? 0 : l; }
  T* dresc(size_t l, int k) const { return m->at<T>(m->bl.dresc) + (2 * dl(l) + k) * BT * C; }
  T* dfch(size_t l) const { return m->at<T>(m->bl.dfch) + dl(l) * BT * 4 * C; }
  T* dqkv(size_t l) const { return m->at<T>(m->bl.dqkv) + dl(l) * BT * 3 * C; }
  // recompute: LayerNorm output i from the stored residual stream and statistics
  // (the forward's arithmetic on the same stored values: the same bits)
  cudaError_t ln_recompute(size_t i, const T* w, const T* b) {
    if (c.recompute < 2) return cudaSuccess;
    return layernorm_apply<T>(ln(i), resid(i), mean(i), rstd(i), w, b, m->BT, c.C, m->st);
  }
  // recompute: GELU of layer l's fc pre-activation
  cudaError_t gelu_recompute(size_t l) {
    if (c.recompute < 1) return cudaSuccess;
    return gelu_forward<T>(fchg(l), fch(l), (long long)m->BT * 4 * c.C, m->st);
  }
  T* dsmall() const { return m->at<T>(m->bl.dsmall); }
  // one-position inference scratch: k-th B x C slab (0, 1: residual, 2: LN out,
  // 3: attention out, 4: projection out), fc pre-activation / GELU (B x 4C),
  // logits (B x Vp), then the LayerNorm statistics
  T* dec(int k) const { return m->at<T>(m->bl.dec) + (size_t)k * c.B * C; }
  T* dec_fch() const { return dec(5); }
  T* dec_fchg() const { return dec(9); }
  T* dec_logits() const { return dec(13); }
  float* dec_stats() const { return reinterpret_cast<float*>(dec_logits() + (size_t)c.B * c.Vp); }
  int* flags() const { return m->at<int>(m->bl.flags); }

  // which kernel takes a product: 0 few-row, 1 tensor cores, 2 SIMT.  A few
  // rows (decoding) go to the few-row kernel, except for very wide products
  // (the classifier), which have enough tiles for the tensor cores
  int gemm_path(const GemmArgs& a) const {
    const bool tc_ok = c.precision == GPT2_PRECISION_BF16 && gemm_tc_supported(a);
    if (gemm_skinny_supported<T>(a) && !(tc_ok && a.N >= 16384)) return 0;
    return tc_ok ? 1 : 2;
  }
  cudaError_t gemm(GemmArgs a) {
    bool rec = m->prof_on && m->prof_n < m->prof_flops.size();
    if (rec) cudaEventRecord(m->prof_ev[2 * m->prof_n], m->st);
    cudaError_t e;
    const int path = gemm_path(a);
    if (path == 0) e = gemm_skinny<T>(a, m->st);
    else if (path == 1) e = gemm_tc(a, flags(), m->st);
    else e = gemm_simt<T>(a, m->st);
    if (rec) {
      cudaEventRecord(m->prof_ev[2 * m->prof_n + 1], m->st);
      m->prof_flops[m->prof_n++] = 2.0 * a.M * a.N * (double)a.K * (a.batch > 1 ? a.batch : 1);
    }
    return e;
  }
  // fp32 master copy of a parameter tensor
  const float* P(int t) const { return m->at<float>(m->bl.params) + m->pl.off[t]; }
  // ln_fold: layer l's folded qkv (k = 0) or fc (k = 1) weight and its sums
  size_t fold_row(size_t l, int k) const { return l * 7 * C + (k ? 3 * C : 0); }
  bf16* wfold(size_t l, int k) const { return m->at<bf16>(m->bl.wfold) + fold_row(l, k) * C; }
  float* fold_s(size_t l, int k) const { return m->at<float>(m->bl.fold_s) + fold_row(l, k); }
  float* fold_c(size_t l, int k) const { return m->at<float>(m->bl.fold_c) + fold_row(l, k); }
  // out[BT][N] = LayerNorm i (of resid(i)) . W^T + b with the LayerNorm folded
  // into the product (layer l's qkv for k = 0, fc with GELU for k = 1)
  cudaError_t linear_fwd_folded(T* out, size_t i, size_t l, int k, int N, T* aux) {
    GemmArgs a{resid(i), (long long)C, 1, wfold(l, k), (long long)C, 1, m->BT, N, (int)C, out, N, nullptr, aux, N,
               aux ? EPI_GELU : EPI_STORE};
    a.ln_mean = mean(i);
    a.ln_rstd = rstd(i);
    a.ln_s = fold_s(l, k);
    a.ln_c = fold_c(l, k);
    return gemm(a);
  }
  // out[M][N] = X[M][K] . W[N][K]^T (+ bias), optionally with GELU (aux = pre-activation)
  cudaError_t linear_fwd(T* out, const T* X, const T* Wt, const T* bias, int M, int N, int K, T* aux = nullptr) {
    GemmArgs a{X, K, 1, Wt, K, 1, M, N, K, out, N, bias, aux, N, aux ? EPI_GELU : EPI_STORE};
    return gemm(a);
  }
  // dX[M][K] = dY[M][N] . W[N][K]  (optionally times GELU'(aux))
  cudaError_t linear_dgrad(T* dX, const T* dY, const T* Wt, int M, int N, int K, const T* aux = nullptr) {
    GemmArgs a{dY, N, 1, Wt, K, 0, M, K, N, dX, K, nullptr, (void*)aux, K, aux ? EPI_GELU_BWD : EPI_STORE};
    return gemm(a);
  }
  // dW[N][K] += dY[M][N]^T . X[M][K]
  cudaError_t linear_wgrad(float* dW, const T* dY, const T* X, int M, int N, int K) {
    GemmArgs a{dY, N, 0, X, K, 0, N, K, M, dW, K, nullptr, nullptr, 0, EPI_ACC_F32,
               m->at<float>(m->bl.ws), m->bl.ws_floats};
    a.acc_store = fresh;
    return gemm(a);
  }
  // the same for every layer at once: item l reads dY + l*sY and X + l*sX and
  // adds into dW + l*N*K (the [L]-stacked gradient of one weight type)
  cudaError_t linear_wgrad_layers(float* dW, const T* dY, long long sY, const T* X, long long sX, int M, int N,
                                  int K) {
    GemmArgs a{dY, N, 0, X, K, 0, N, K, M, dW, K, nullptr, nullptr, 0, EPI_ACC_F32, nullptr, 0,
               (int)c.L, sY, sX, (long long)N * K, 0};
    a.acc_store = fresh;
    return gemm(a);
  }

  // two weight types' gradients for every layer (the same input width K and
  // rows M = B*T), as one tensor-core launch when that fills the last wave better
  cudaError_t linear_wgrad_layers_pair(float* dW1, const T* dY1, long long sY1, const T* X1, long long sX1, int N1,
                                       float* dW2, const T* dY2, long long sY2, const T* X2, long long sX2, int N2,
                                       int M, int K) {
    GemmArgs a{dY1, N1, 0, X1, K, 0, N1, K, M, dW1, K, nullptr, nullptr, 0, EPI_ACC_F32, nullptr, 0,
               (int)c.L, sY1, sX1, (long long)N1 * K, 0};
    GemmArgs b{dY2, N2, 0, X2, K, 0, N2, K, M, dW2, K, nullptr, nullptr, 0, EPI_ACC_F32, nullptr, 0,
               (int)c.L, sY2, sX2, (long long)N2 * K, 0};
    a.acc_store = b.acc_store = fresh;
    if (gemm_path(a) != 1 || gemm_path(b) != 1) {
      cudaError_t e = gemm(a);
      return e != cudaSuccess ? e : gemm(b);
    }
    const bool rec = m->prof_on && m->prof_n < m->prof_flops.size();
    if (rec) cudaEventRecord(m->prof_ev[2 * m->prof_n], m->st);
    cudaError_t e = gemm_tc_grouped(a, b, flags(), m->st);
    if (rec) {
      cudaEventRecord(m->prof_ev[2 * m->prof_n + 1], m->st);
      m->prof_flops[m->prof_n++] = 2.0 * (double)(N1 + N2) * K * (double)M * c.L;
    }
    return e;
  }

  // causal attention: tcgen05 flash kernels in bf16 mode, SIMT kernels in fp32 mode
  bool attention_on_tc() const {
    return c.precision == GPT2_PRECISION_BF16 && attention_tc_supported(c.B, c.T, c.C, c.H);
  }
  cudaError_t attention_fwd(T* out, float* lse_, const T* qkv_) {
    if (attention_on_tc())
      return attention_forward_tc((bf16*)out, lse_, (const bf16*)qkv_, c.B, c.T, c.C, c.H, flags(), m->st);
    return attention_forward_simt<T>(out, lse_, qkv_, c.B, c.T, c.C, c.H, m->st);
  }
  // attention-projection input gradient; on the tensor-core path its epilogue
  // also takes the attention backward's D = rowsum(dO * O) (returns whether it did)
  cudaError_t attproj_dgrad(T* dX, const T* dY, const T* Wt, const T* O, bool* d_ready) {
    const int M = m->BT, N = c.C, K = c.C;
    *d_ready = false;
    if (attention_on_tc()) {
      GemmArgs a{dY, N, 1, Wt, K, 0, M, K, N, dX, K, nullptr, (void*)O, K, EPI_ROWDOT, nullptr, 0,
                 1, 0, 0, 0, 0, m->at<float>(m->bl.attD), c.T, c.H};
      if (gemm_tc_supported(a)) {
        *d_ready = true;
        return gemm(a);
      }
    }
    return linear_dgrad(dX, dY, Wt, M, N, K);
  }
  cudaError_t attention_bwd(T* dqkv, const T* dout, const T* qkv_, const T* out, const float* lse_,
                            bool d_ready = false) {
    float* Dbuf = m->at<float>(m->bl.attD);
    if (attention_on_tc())
      return attention_backward_tc((bf16*)dqkv, Dbuf, m->at<uint8_t>(m->bl.attS), (const bf16*)dout,
                                   (const bf16*)qkv_, (const bf16*)out, lse_, c.B, c.T, c.C, c.H, flags(), m->st,
                                   d_ready);
    return attention_backward_simt<T>(dqkv, Dbuf, dout, qkv_, out, lse_, c.B, c.T, c.C, c.H, m->st);
  }

  int forward(const int32_t* tok, const int32_t* tgt) {
    cudaStream_t st = m->st;
    int B = c.B, T_ = c.T, Ci = c.C, Li = c.L, BTi = m->BT;
    size_t CC = C * C;
    CK(m, encoder_forward<T>(resid(0), tok, W(GPT2_WTE), W(GPT2_WPE), B, T_, Ci, c.V, flags(), st));
    const bool fold = c.ln_fold != 0;
    if (fold) {  // this step's weights with the LayerNorm gains folded in
      CK(m, lnfold_weights(wfold(0, 0), fold_s(0, 0), fold_c(0, 0), P(GPT2_QKVW), P(GPT2_LN1W), P(GPT2_LN1B),
                           P(GPT2_QKVB), Li, 3 * Ci, Ci, st, 7 * C));
      CK(m, lnfold_weights(wfold(0, 1), fold_s(0, 1), fold_c(0, 1), P(GPT2_FCW), P(GPT2_LN2W), P(GPT2_LN2B),
                           P(GPT2_FCB), Li, 4 * Ci, Ci, st, 7 * C));
    }
    for (int l = 0; l < Li; l++) {
      // with the fold only the residual stream and the statistics are written
      if (l == 0)
        CK(m, residual_layernorm_forward<T>(nullptr, fold ? nullptr : ln(0), mean(0), rstd(0), resid(0), nullptr,
                                            W(GPT2_LN1W, l, C), W(GPT2_LN1B, l, C), BTi, Ci, st));
      else
        CK(m, residual_layernorm_forward<T>(resid(2 * l), fold ? nullptr : ln(2 * l), mean(2 * l), rstd(2 * l),
                                            resid(2 * l - 1), proj(), W(GPT2_LN1W, l, C), W(GPT2_LN1B, l, C), BTi,
                                            Ci, st));
      if (fold) CK(m, linear_fwd_folded(qkv(l), 2 * l, l, 0, 3 * Ci, nullptr));
      else CK(m, linear_fwd(qkv(l), ln(2 * l), W(GPT2_QKVW, l, 3 * CC), W(GPT2_QKVB, l, 3 * C), BTi, 3 * Ci, Ci));
      CK(m, attention_fwd(atty(l), lse(l), qkv(l)));
      CK(m, linear_fwd(proj(), atty(l), W(GPT2_ATTPROJW, l, CC), W(GPT2_ATTPROJB, l, C), BTi, Ci, Ci));
      CK(m, residual_layernorm_forward<T>(resid(2 * l + 1), fold ? nullptr : ln(2 * l + 1), mean(2 * l + 1),
                                          rstd(2 * l + 1), resid(2 * l), proj(), W(GPT2_LN2W, l, C), W(GPT2_LN2B, l, C),
                                          BTi, Ci, st));
      if (fold) CK(m, linear_fwd_folded(fchg(l), 2 * l + 1, l, 1, 4 * Ci, fch(l)));
      else
        CK(m, linear_fwd(fchg(l), ln(2 * l + 1), W(GPT2_FCW, l, 4 * CC), W(GPT2_FCB, l, 4 * C), BTi, 4 * Ci, Ci,
                         fch(l)));
      CK(m, linear_fwd(proj(), fchg(l), W(GPT2_FCPROJW, l, 4 * CC), W(GPT2_FCPROJB, l, C), BTi, Ci, 4 * Ci));
    }
    size_t f = 2 * L;
    CK(m, residual_layernorm_forward<T>(resid(f), ln(f), mean(f), rstd(f), resid(f - 1), proj(), W(GPT2_LNFW),
                                        W(GPT2_LNFB), BTi, Ci, st));
    // with targets on the tensor cores, the classifier's epilogue also takes
    // each row's (max, sum of exp) per column tile, so the softmax reads the
    // logits once
    GemmArgs cls{ln(f), Ci, 1, W(GPT2_WTE), Ci, 1, BTi, c.Vp, Ci, logits(), c.Vp, nullptr, nullptr, c.Vp, EPI_STORE};
    if (tgt && m->bl.lstats) {
      cls.rowstats = m->at<float>(m->bl.lstats);
      cls.stats_cols = c.V;
      if (gemm_path(cls) != 1) cls.rowstats = nullptr;
    }
    CK(m, gemm(cls));
    if (tgt) {
      if (cls.rowstats)
        CK(m, softmax_ce_from_stats((bf16*)logits(), losses(), tgt, cls.rowstats, gemm_tc_stats_tiles(c.Vp), BTi, c.V,
                                    c.Vp, 1.0f / (float)BTi, flags(), st));
      else CK(m, softmax_ce<T>(logits(), losses(), tgt, BTi, c.V, c.Vp, 1.0f / (float)BTi, 1, flags(), st));
      CK(m, mean_loss(m->at<float>(m->bl.loss), losses(), BTi, st));
    }
    return GPT2_OK;
  }

  // One new position `pos` for every sequence, reading keys and values 0..pos
  // from the KV cache and writing this position's q | k | v into it: the
  // forward of one token per sequence (tok [B]), logits into dec_logits().
  int decode(const int32_t* tok, int pos) {
    cudaStream_t st = m->st;
    const int Bi = c.B, Ci = c.C, Li = c.L;
    const size_t CC = C * C;
    T* x[2] = {dec(0), dec(1)};
    T *lnb = dec(2), *att = dec(3), *prj = dec(4), *fh = dec_fch(), *fg = dec_fchg();
    float *mu = dec_stats(), *rs = dec_stats() + Bi;
    // x = wte[tok] + wpe[pos]: the encoder with one position, its wpe row pos
    CK(m, encoder_forward<T>(x[0], tok, W(GPT2_WTE), W(GPT2_WPE) + (size_t)pos * C, Bi, 1, Ci, c.V, flags(), st));
    if constexpr (sizeof(T) == 2) {
      if (decode_layers_supported(Bi, Ci, c.H, c.T)) {
        // every block in one cooperative launch; the residual comes back in x[0]
        const bf16* w[12] = {W(GPT2_LN1W), W(GPT2_LN1B), W(GPT2_QKVW), W(GPT2_QKVB), W(GPT2_ATTPROJW),
                             W(GPT2_ATTPROJB), W(GPT2_LN2W), W(GPT2_LN2B), W(GPT2_FCW), W(GPT2_FCB),
                             W(GPT2_FCPROJW), W(GPT2_FCPROJB)};
        CK(m, decode_layers(w, qkv(0), x[0], x[1], att, fg, m->at<unsigned>(m->bl.decbar), flags(), Li, Bi, Ci, c.H,
                            c.T, pos, st));
        CK(m, residual_layernorm_forward<T>(nullptr, lnb, mu, rs, x[0], nullptr, W(GPT2_LNFW), W(GPT2_LNFB), Bi, Ci,
                                            st));
        CK(m, linear_fwd(dec_logits(), lnb, W(GPT2_WTE), nullptr, Bi, c.Vp, Ci));
        return GPT2_OK;
      }
    }
    int cur = 0;
    for (int l = 0; l < Li; l++) {
      if (l == 0) {
        CK(m, residual_layernorm_forward<T>(nullptr, lnb, mu, rs, x[0], nullptr, W(GPT2_LN1W, l, C),
                                            W(GPT2_LN1B, l, C), Bi, Ci, st));
      } else {
        CK(m, residual_layernorm_forward<T>(x[cur ^ 1], lnb, mu, rs, x[cur], prj, W(GPT2_LN1W, l, C),
                                            W(GPT2_LN1B, l, C), Bi, Ci, st));
        cur ^= 1;
      }
      // q | k | v of position pos straight into cache rows b*T + pos
      GemmArgs a{lnb, (long long)C, 1, W(GPT2_QKVW, l, 3 * CC), (long long)C, 1, Bi, 3 * Ci, Ci,
                 qkv(l) + (size_t)pos * 3 * C, (long long)c.T * 3 * Ci, W(GPT2_QKVB, l, 3 * C), nullptr, 0, EPI_STORE};
      CK(m, gemm(a));
      CK(m, decode_attention<T>(att, qkv(l), Bi, c.T, pos, Ci, c.H, st));
      CK(m, linear_fwd(prj, att, W(GPT2_ATTPROJW, l, CC), W(GPT2_ATTPROJB, l, C), Bi, Ci, Ci));
      CK(m, residual_layernorm_forward<T>(x[cur ^ 1], lnb, mu, rs, x[cur], prj, W(GPT2_LN2W, l, C),
                                          W(GPT2_LN2B, l, C), Bi, Ci, st));
      cur ^= 1;
      CK(m, linear_fwd(fg, lnb, W(GPT2_FCW, l, 4 * CC), W(GPT2_FCB, l, 4 * C), Bi, 4 * Ci, Ci, fh));
      CK(m, linear_fwd(prj, fg, W(GPT2_FCPROJW, l, 4 * CC), W(GPT2_FCPROJB, l, C), Bi, Ci, 4 * Ci));
    }
    CK(m, residual_layernorm_forward<T>(x[cur ^ 1], lnb, mu, rs, x[cur], prj, W(GPT2_LNFW), W(GPT2_LNFB), Bi, Ci, st));
    CK(m, linear_fwd(dec_logits(), lnb, W(GPT2_WTE), nullptr, Bi, c.Vp, Ci));
    return GPT2_OK;
  }

  // fresh: the gradient buffer holds garbage and every gradient's first
  // writer stores instead of adding (the graph step's backward, with no zero_grad)
  int fresh = 0;
  int backward(const int32_t* tok, bool fresh_grads = false) {
    fresh = fresh_grads ? 1 : 0;
    const int acc = fresh ? 0 : 1;
    cudaStream_t st = m->st;
    int Ci = c.C, Li = c.L, BTi = m->BT;
    size_t CC = C * C;
    float* part = m->at<float>(m->bl.partial);
    size_t f = 2 * L;
    // recompute >= 1: weight gradients inside the layer loop, from one layer's
    // recomputed GELU / LayerNorm outputs; else batched after the loop
    const bool perlayer = c.recompute >= 1;
    // every LayerNorm backward leaves its parameter-sum partials in its own
    // slot (LN1 of layer l: 2l, LN2: 2l+1, final: 2L); they are reduced after
    // the loop.  Per-layer column sums use the space after the slots.
    const size_t lnslot = ln_backward_partial_floats(BTi, Ci);
    float* cpart = part + (2 * L + 1) * lnslot;
    int nch = 0;
    // classifier (tied wte): dlnf = dlogits . wte ; dwte += dlogits^T . lnf
    CK(m, linear_dgrad(dsmall(), logits(), W(GPT2_WTE), BTi, c.Vp, Ci));
    CK(m, ln_recompute(f, W(GPT2_LNFW), W(GPT2_LNFB)));
    CK(m, linear_wgrad(G(GPT2_WTE), logits(), ln(f), BTi, c.Vp, Ci));
    // The residual gradient runs backwards through the LayerNorm backwards in
    // the activation type, from one kept slot to the next: dresc(l, 0) enters
    // layer l's fc projection, dresc(l, 1) its attention projection; the
    // last one (into the embeddings) is written in fp32 to dres().
    // final LayerNorm; the column sums of the resulting residual gradient are
    // the bias gradient of the last fc projection (whose output gradient it is)
    CK(m, (layernorm_backward_rg<T, T>(dresc(L - 1, 0), nullptr, nullptr, nullptr, dsmall(), resid(f), mean(f), rstd(f),
                                      W(GPT2_LNFW), BTi, Ci, G(GPT2_LNFW), G(GPT2_LNFB), G(GPT2_FCPROJB, L - 1, C),
                                      part + 2 * L * lnslot, st, &nch)));
    for (int l = Li - 1; l >= 0; l--) {
      // fc projection (+ GELU backward fused into its input-gradient GEMM)
      CK(m, linear_dgrad(dfch(l), dresc(l, 0), W(GPT2_FCPROJW, l, 4 * CC), BTi, Ci, 4 * Ci, fch(l)));
      if (perlayer) {
        CK(m, gelu_recompute(l));
        CK(m, linear_wgrad(G(GPT2_FCPROJW, l, 4 * CC), dresc(l, 0), fchg(l), BTi, Ci, 4 * Ci));
      }
      // fc
      CK(m, linear_dgrad(dsmall(), dfch(l), W(GPT2_FCW, l, 4 * CC), BTi, 4 * Ci, Ci));
      if (perlayer) {
        CK(m, ln_recompute(2 * l + 1, W(GPT2_LN2W, l, C), W(GPT2_LN2B, l, C)));
        CK(m, linear_wgrad(G(GPT2_FCW, l, 4 * CC), dfch(l), ln(2 * l + 1), BTi, 4 * Ci, Ci));
        CK(m, colsum<T>(G(GPT2_FCB, l, 4 * C), dfch(l), BTi, 4 * Ci, 4 * Ci, cpart, st, 1, 0, 0, acc));
      }
      // LN2 (+ residual gradient; its column sums give the attention-projection bias gradient)
      CK(m, (layernorm_backward_rg<T, T>(dresc(l, 1), dresc(l, 0), nullptr, nullptr, dsmall(), resid(2 * l + 1),
                                        mean(2 * l + 1), rstd(2 * l + 1), W(GPT2_LN2W, l, C), BTi, Ci,
                                        G(GPT2_LN2W, l, C), G(GPT2_LN2B, l, C), G(GPT2_ATTPROJB, l, C),
                                        part + (2 * l + 1) * lnslot, st, &nch)));
      // attention projection (its epilogue also forms the attention backward's D)
      bool d_ready = false;
      CK(m, attproj_dgrad(dsmall(), dresc(l, 1), W(GPT2_ATTPROJW, l, CC), atty(l), &d_ready));
      if (perlayer) CK(m, linear_wgrad(G(GPT2_ATTPROJW, l, CC), dresc(l, 1), atty(l), BTi, Ci, Ci));
      // attention
      CK(m, attention_bwd(dqkv(l), dsmall(), qkv(l), atty(l), lse(l), d_ready));
      // qkv
      CK(m, linear_dgrad(dsmall(), dqkv(l), W(GPT2_QKVW, l, 3 * CC), BTi, 3 * Ci, Ci));
      if (perlayer) {
        CK(m, ln_recompute(2 * l, W(GPT2_LN1W, l, C), W(GPT2_LN1B, l, C)));
        CK(m, linear_wgrad(G(GPT2_QKVW, l, 3 * CC), dqkv(l), ln(2 * l), BTi, 3 * Ci, Ci));
        CK(m, colsum<T>(G(GPT2_QKVB, l, 3 * C), dqkv(l), BTi, 3 * Ci, 3 * Ci, cpart, st, 1, 0, 0, acc));
      }
      // LN1 (+ residual gradient; its column sums give the previous block's fc-projection bias gradient)
      CK(m, (layernorm_backward_rg<T, T>(l > 0 ? dresc(l - 1, 0) : nullptr, dresc(l, 1), nullptr,
                                        l > 0 ? nullptr : dres(), dsmall(), resid(2 * l), mean(2 * l), rstd(2 * l),
                                        W(GPT2_LN1W, l, C), BTi, Ci, G(GPT2_LN1W, l, C), G(GPT2_LN1B, l, C),
                                        l > 0 ? G(GPT2_FCPROJB, l - 1, C) : nullptr, part + 2 * l * lnslot, st, &nch)));
    }
    // LayerNorm weight / bias sums and the projection biases they give, for
    // all layers: final LN, every LN2 (one batched launch), LN1 of layers
    // 1..L-1 (one batched launch), LN1 of layer 0
    const long long sl = (long long)lnslot;
    CK(m, reduce_partials(G(GPT2_LNFW), G(GPT2_LNFB), G(GPT2_FCPROJB, L - 1, C), part + 2 * L * lnslot, nch, Ci, 3, st,
                          1, 0, 0, acc));
    CK(m, reduce_partials(G(GPT2_LN2W), G(GPT2_LN2B), G(GPT2_ATTPROJB), part + lnslot, nch, Ci, 3, st, Li, Ci, 2 * sl,
                          acc));
    if (Li > 1)
      CK(m, reduce_partials(G(GPT2_LN1W, 1, C), G(GPT2_LN1B, 1, C), G(GPT2_FCPROJB), part + 2 * lnslot, nch, Ci, 3, st,
                            Li - 1, Ci, 2 * sl, acc));
    CK(m, reduce_partials(G(GPT2_LN1W), G(GPT2_LN1B), nullptr, part, nch, Ci, 3, st, 1, 0, 0, acc));
    if (!perlayer) {
      // weight gradients of every layer, one batched product per weight type
      const long long sBT = (long long)BTi * Ci;
      CK(m, linear_wgrad_layers(G(GPT2_FCPROJW), dresc(0, 0), 2 * sBT, fchg(0), 4 * sBT, BTi, Ci, 4 * Ci));
      CK(m, linear_wgrad_layers(G(GPT2_FCW), dfch(0), 4 * sBT, ln(1), 2 * sBT, BTi, 4 * Ci, Ci));
      // attention projection and qkv together: 108 + 324 pair tiles at 124M share one last wave
      CK(m, linear_wgrad_layers_pair(G(GPT2_ATTPROJW), dresc(0, 1), 2 * sBT, atty(0), sBT, Ci, G(GPT2_QKVW), dqkv(0),
                                     3 * sBT, ln(0), 2 * sBT, 3 * Ci, BTi, Ci));
      // bias gradients of the fc and qkv layers of every layer: column sums of their output gradients
      CK(m, colsum<T>(G(GPT2_FCB), dfch(0), BTi, 4 * Ci, 4 * Ci, part, st, Li, 4 * Ci, 4 * sBT, acc));
      CK(m, colsum<T>(G(GPT2_QKVB), dqkv(0), BTi, 3 * Ci, 3 * Ci, part, st, Li, 3 * Ci, 3 * sBT, acc));
    }
    if (encoder_backward_fast_supported(BTi, Ci))
      CK(m, encoder_backward_fast(G(GPT2_WTE), G(GPT2_WPE), dres(), tok, c.B, c.T, Ci, c.V, flags(),
                                  m->at<uint32_t>(m->bl.keys), st, acc));
    else
      CK(m, encoder_backward(G(GPT2_WTE), G(GPT2_WPE), dres(), tok, c.B, c.T, Ci, c.V, flags(),
                             m->at<uint32_t>(m->bl.keys), st, acc));
    return GPT2_OK;
  }
};

static int check_flags(gpt2* m) {
  int h[4] = {0, 0, 0, 0};
  CK(m, cudaMemcpyAsync(h, m->at<int>(m->bl.flags), sizeof h, cudaMemcpyDeviceToHost, m->st));
  CK(m, cudaStreamSynchronize(m->st));
  if (h[0]) {
    CK(m, cudaMemsetAsync(m->at<int>(m->bl.flags), 0, sizeof h, m->st));
    CK(m, cudaStreamSynchronize(m->st));
    if (h[0] & FLAG_TIMEOUT) FAIL(m, GPT2_ERR_TIMEOUT, "a kernel's bounded wait ran out (flags=0x%x)", h[0]);
    if (h[0] & FLAG_TOKEN_RANGE) FAIL(m, GPT2_ERR_TOKEN_RANGE, "a token id is outside [0, V)");
    if (h[0] & FLAG_TARGET_RANGE) FAIL(m, GPT2_ERR_TOKEN_RANGE, "a target id is outside [0, V)");
  }
  return GPT2_OK;
}

// --------------------------------------------------------------------------
// C ABI
// --------------------------------------------------------------------------
extern "C" {

size_t gpt2_num_parameters(const gpt2_config* cfg) {
  const char* why;
  if (!cfg || validate_config(*cfg, &why) != GPT2_OK) return 0;
  return param_layout(*cfg).total;
}

size_t gpt2_tensor_numel(const gpt2_config* cfg, int tensor) {
  const char* why;
  if (!cfg || tensor < 0 || tensor >= GPT2_NUM_TENSORS || validate_config(*cfg, &why) != GPT2_OK) return 0;
  return param_layout(*cfg).numel[tensor];
}

size_t gpt2_required_bytes(const gpt2_config* cfg) {
  const char* why;
  if (!cfg || validate_config(*cfg, &why) != GPT2_OK) return 0;
  return buffer_layout(*cfg).total;
}

int gpt2_init_params_host(const gpt2_config* cfg, uint64_t seed, float* host_out) {
  const char* why;
  if (!cfg || !host_out) FAIL((gpt2*)nullptr, GPT2_ERR_INVALID_ARG, "NULL argument");
  int rc = validate_config(*cfg, &why);
  if (rc) FAIL((gpt2*)nullptr, rc, "invalid config: %s", why);
  init_params_host(*cfg, seed, host_out);
  return GPT2_OK;
}

int gpt2_create(const gpt2_config* cfg, uint64_t seed, void* dev_buf, size_t bytes, void* cuda_stream, gpt2** out) {
  const char* why;
  if (out) *out = nullptr;
  if (!cfg || !dev_buf || !out) FAIL((gpt2*)nullptr, GPT2_ERR_INVALID_ARG, "NULL argument");
  int rc = validate_config(*cfg, &why);
  if (rc) FAIL((gpt2*)nullptr, rc, "invalid config: %s", why);
  BufferLayout bl = buffer_layout(*cfg);
  if (bytes < bl.total)
    FAIL((gpt2*)nullptr, GPT2_ERR_BUFFER_TOO_SMALL, "buffer has %zu bytes, the model needs %zu", bytes, bl.total);
  if ((uintptr_t)dev_buf % 256) FAIL((gpt2*)nullptr, GPT2_ERR_INVALID_ARG, "dev_buf must be 256-byte aligned");
  gpt2* m = new gpt2();
  m->cfg = *cfg;
  m->pl = param_layout(*cfg);
  m->bl = bl;
  m->base = (char*)dev_buf;
  m->st = (cudaStream_t)cuda_stream;
  m->BT = cfg->B * cfg->T;
  std::vector<float> host(m->pl.total);
  init_params_host(*cfg, seed, host.data());
  cudaError_t e = cudaMemsetAsync(m->base, 0, bl.total, m->st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(m->at<float>(bl.params), host.data(), m->pl.total * 4, cudaMemcpyHostToDevice, m->st);
  if (e == cudaSuccess && cfg->precision == GPT2_PRECISION_BF16)
    e = convert_f32_bf16(m->at<bf16>(bl.pbf), m->at<float>(bl.params), (long long)m->pl.total, m->st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(m->st);
  if (e != cudaSuccess) {
    g_create_err = std::string("gpt2_create: ") + cudaGetErrorString(e);
    delete m;
    return GPT2_ERR_CUDA;
  }
  gpt2_count_launches(cfg->precision == GPT2_PRECISION_BF16 ? 1 : 0);
  *out = m;
  return GPT2_OK;
}

int gpt2_forward(gpt2* m, const int32_t* tokens_dev, const int32_t* targets_dev, float* loss_host) {
  if (!m) return GPT2_ERR_INVALID_ARG;
  if (!tokens_dev) FAIL(m, GPT2_ERR_INVALID_ARG, "tokens_dev is NULL");
  if (loss_host && !targets_dev) FAIL(m, GPT2_ERR_INVALID_ARG, "loss_host needs targets_dev");
  int rc = m->cfg.precision == GPT2_PRECISION_BF16 ? Step<bf16>(m).forward(tokens_dev, targets_dev)
                                                   : Step<float>(m).forward(tokens_dev, targets_dev);
  m->have_targets = rc == GPT2_OK && targets_dev != nullptr;
  m->logits_valid = rc == GPT2_OK && targets_dev == nullptr;
  m->loss_valid = m->have_targets;
  m->fwd_tokens = tokens_dev;
  m->cache_len = 0;  // the qkv activations (the inference cache) now hold this batch
  if (rc) return rc;
  if (loss_host) return gpt2_get_loss(m, loss_host);
  return GPT2_OK;
}

int gpt2_infer_prefill(gpt2* m, const int32_t* tokens_dev, int n) {
  if (!m) return GPT2_ERR_INVALID_ARG;
  if (!tokens_dev) FAIL(m, GPT2_ERR_INVALID_ARG, "tokens_dev is NULL");
  if (n < 1 || n > m->cfg.T) FAIL(m, GPT2_ERR_INVALID_ARG, "prefill length %d outside 1..T=%d", n, m->cfg.T);
  int rc = gpt2_forward(m, tokens_dev, nullptr, nullptr);
  m->cache_len = 0;
  if (rc) return rc;
  const size_t es = m->cfg.precision == GPT2_PRECISION_BF16 ? 2 : 4;
  m->cache_len = n;
  m->last_logits = m->bl.logits + (size_t)(n - 1) * m->cfg.Vp * es;  // rows b*T + n-1
  m->last_ld = (long long)m->cfg.T * m->cfg.Vp;
  return GPT2_OK;
}

int gpt2_infer_step(gpt2* m, const int32_t* tokens_dev, int pos) {
  if (!m) return GPT2_ERR_INVALID_ARG;
  if (!tokens_dev) FAIL(m, GPT2_ERR_INVALID_ARG, "tokens_dev is NULL");
  if (m->cache_len < 1) FAIL(m, GPT2_ERR_BAD_ORDER, "gpt2_infer_step needs gpt2_infer_prefill first");
  if (pos != m->cache_len || pos >= m->cfg.T)
    FAIL(m, GPT2_ERR_INVALID_ARG, "position %d: the cache holds %d positions of at most T=%d", pos, m->cache_len,
         m->cfg.T);
  int rc = m->cfg.precision == GPT2_PRECISION_BF16 ? Step<bf16>(m).decode(tokens_dev, pos)
                                                   : Step<float>(m).decode(tokens_dev, pos);
  m->have_targets = m->logits_valid = m->loss_valid = false;  // the training activations are overwritten
  if (rc) {
    m->cache_len = 0;
    return rc;
  }
  m->cache_len = pos + 1;
  m->last_logits = m->bl.dec + ((5 + 8) * (size_t)m->cfg.B * m->cfg.C) *
                                   (m->cfg.precision == GPT2_PRECISION_BF16 ? 2 : 4);
  m->last_ld = m->cfg.Vp;
  return GPT2_OK;
}

int gpt2_sample(gpt2* m, float temperature, const float* coins_dev, int32_t* out_tokens_dev) {
  if (!m) return GPT2_ERR_INVALID_ARG;
  if (!out_tokens_dev || (temperature > 0.f && !coins_dev) || !(temperature >= 0.f))
    FAIL(m, GPT2_ERR_INVALID_ARG, "sampling needs out_tokens_dev, a temperature >= 0 and coins_dev when it is > 0");
  if (m->cache_len < 1) FAIL(m, GPT2_ERR_BAD_ORDER, "gpt2_sample needs gpt2_infer_prefill or gpt2_infer_step first");
  if (m->cfg.precision == GPT2_PRECISION_BF16)
    CK(m, sample_tokens<bf16>((int*)out_tokens_dev, m->at<bf16>(m->last_logits), m->last_ld, m->cfg.B, m->cfg.V,
                              temperature, coins_dev, m->st));
  else
    CK(m, sample_tokens<float>((int*)out_tokens_dev, m->at<float>(m->last_logits), m->last_ld, m->cfg.B, m->cfg.V,
                               temperature, coins_dev, m->st));
  return GPT2_OK;
}

int gpt2_get_infer_logits(gpt2* m, float* host) {
  if (!m || !host) return GPT2_ERR_INVALID_ARG;
  if (m->cache_len < 1) FAIL(m, GPT2_ERR_BAD_ORDER, "no inference logits yet");
  int rc = check_flags(m);
  if (rc) return rc;
  const size_t Vp = m->cfg.Vp;
  if (m->cfg.precision == GPT2_PRECISION_BF16) {
    std::vector<uint16_t> tmp((size_t)m->cfg.B * Vp);
    CK(m, cudaMemcpy2DAsync(tmp.data(), Vp * 2, m->base + m->last_logits, (size_t)m->last_ld * 2, Vp * 2, m->cfg.B,
                            cudaMemcpyDeviceToHost, m->st));
    CK(m, cudaStreamSynchronize(m->st));
    for (size_t i = 0; i < tmp.size(); i++) {
      uint32_t u = (uint32_t)tmp[i] << 16;
      memcpy(&host[i], &u, 4);
    }
  } else {
    CK(m, cudaMemcpy2DAsync(host, Vp * 4, m->base + m->last_logits, (size_t)m->last_ld * 4, Vp * 4, m->cfg.B,
                            cudaMemcpyDeviceToHost, m->st));
    CK(m, cudaStreamSynchronize(m->st));
  }
  return GPT2_OK;
}

int gpt2_backward(gpt2* m) {
  if (!m) return GPT2_ERR_INVALID_ARG;
  if (!m->have_targets) FAIL(m, GPT2_ERR_BAD_ORDER, "gpt2_backward needs a gpt2_forward with targets first");
  int rc = m->cfg.precision == GPT2_PRECISION_BF16 ? Step<bf16>(m).backward(m->fwd_tokens)
                                                   : Step<float>(m).backward(m->fwd_tokens);
  m->have_targets = false;  // dlogits consumed
  return rc;
}

int gpt2_zero_grad(gpt2* m) {
  if (!m) return GPT2_ERR_INVALID_ARG;
  CK(m, cudaMemsetAsync(m->at<float>(m->bl.grads), 0, m->pl.total * 4, m->st));
  return GPT2_OK;
}

int gpt2_adamw_step(gpt2* m, float lr, float b1, float b2, float eps, float wd, int t) {
  if (!m) return GPT2_ERR_INVALID_ARG;
  if (t < 1) FAIL(m, GPT2_ERR_INVALID_ARG, "AdamW step t must be >= 1");
  AdamSegments seg{};
  seg.n = GPT2_NUM_TENSORS;
  for (int i = 0; i <= GPT2_NUM_TENSORS; i++) seg.off[i] = (long long)m->pl.off[i];
  for (int i = 0; i < GPT2_NUM_TENSORS; i++) {
    bool decay = i == GPT2_WTE || i == GPT2_WPE || i == GPT2_QKVW || i == GPT2_ATTPROJW || i == GPT2_FCW ||
                 i == GPT2_FCPROJW;
    seg.wd[i] = decay ? wd : 0.f;
  }
  float bc1 = (float)(1.0 - std::pow((double)b1, (double)t));
  float bc2 = (float)(1.0 - std::pow((double)b2, (double)t));
  bf16* pc = m->cfg.precision == GPT2_PRECISION_BF16 ? m->at<bf16>(m->bl.pbf) : nullptr;
  const float* gscale = m->clip_pending ? m->at<float>(m->bl.gnorm) + 1 : nullptr;
  m->clip_pending = false;
  CK(m, adamw(m->at<float>(m->bl.params), m->at<float>(m->bl.grads), m->at<float>(m->bl.m), m->at<float>(m->bl.v),
              pc, (long long)m->pl.total, lr, b1, b2, eps, bc1, bc2, seg, gscale, m->st));
  return GPT2_OK;
}

int gpt2_clip_grad_norm(gpt2* m, float max_norm) {
  if (!m) return GPT2_ERR_INVALID_ARG;
  if (!(max_norm > 0.f)) FAIL(m, GPT2_ERR_INVALID_ARG, "max_norm must be > 0");
  float* gn = m->at<float>(m->bl.gnorm);
  CK(m, grad_norm(m->at<float>(m->bl.grads), (long long)m->pl.total, max_norm, gn, gn + 2, m->st));
  m->clip_pending = true;
  return GPT2_OK;
}

int gpt2_get_grad_norm(gpt2* m, float* norm_host) {
  if (!m || !norm_host) return GPT2_ERR_INVALID_ARG;
  CK(m, cudaMemcpyAsync(norm_host, m->at<float>(m->bl.gnorm), sizeof(float), cudaMemcpyDeviceToHost, m->st));
  CK(m, cudaStreamSynchronize(m->st));
  return GPT2_OK;
}

float gpt2_lr_schedule(float max_lr, float final_frac, int warmup, int total, int step) {
  if (step < warmup) return max_lr * (float)(step + 1) / (float)warmup;
  const double min_lr = (double)final_frac * max_lr;
  if (step >= total) return (float)min_lr;
  const double ratio = (double)(step - warmup) / (double)(total - warmup);
  return (float)(min_lr + 0.5 * (1.0 + std::cos(3.141592653589793 * ratio)) * ((double)max_lr - min_lr));
}

int gpt2_step_host(gpt2* m, const int32_t* tokens_host, const int32_t* targets_host, float lr, float b1, float b2,
                   float eps, float wd, int t, float* loss_host) {
  if (!m) return GPT2_ERR_INVALID_ARG;
  if (!tokens_host || !targets_host || !loss_host) FAIL(m, GPT2_ERR_INVALID_ARG, "NULL host pointer");
  size_t nb = (size_t)m->BT * 4;
  int32_t* tok = m->at<int32_t>(m->bl.tok);
  int32_t* tgt = m->at<int32_t>(m->bl.tgt);
  CK(m, cudaMemcpyAsync(tok, tokens_host, nb, cudaMemcpyHostToDevice, m->st));
  CK(m, cudaMemcpyAsync(tgt, targets_host, nb, cudaMemcpyHostToDevice, m->st));
  int rc;
  if (m->st) {  // the model's own token buffers never move: replay one captured graph
    rc = gpt2_graph_step(m, tok, tgt);
  } else {
    rc = gpt2_zero_grad(m);
    if (!rc) rc = gpt2_forward(m, tok, tgt, nullptr);
    if (!rc) rc = gpt2_backward(m);
  }
  if (!rc) rc = gpt2_adamw_step(m, lr, b1, b2, eps, wd, t);
  if (!rc) rc = gpt2_get_loss(m, loss_host);
  return rc;
}

int gpt2_graph_step(gpt2* m, const int32_t* tokens_dev, const int32_t* targets_dev) {
  if (m) m->cache_len = 0;
  if (!m) return GPT2_ERR_INVALID_ARG;
  if (!tokens_dev || !targets_dev) FAIL(m, GPT2_ERR_INVALID_ARG, "tokens_dev and targets_dev are required");
  if (!m->st) FAIL(m, GPT2_ERR_INVALID_ARG, "graph capture needs a created stream, not the legacy default one");
  if (!m->gexec || m->g_tok != tokens_dev || m->g_tgt != targets_dev) {
    if (m->gexec) {
      cudaGraphExecDestroy(m->gexec);
      m->gexec = nullptr;
    }
    const unsigned long long l0 = gpt2_total_launches();
    const bool prof = m->prof_on;
    m->prof_on = false;  // no event records inside the graph
    CK(m, cudaStreamBeginCapture(m->st, cudaStreamCaptureModeThreadLocal));
    // zero_grad + forward + backward, the backward writing fresh gradients
    // (every gradient's first writer stores), so no memset of the buffer runs
    int rc = gpt2_forward(m, tokens_dev, targets_dev, nullptr);
    if (!rc) {
      rc = m->cfg.precision == GPT2_PRECISION_BF16 ? Step<bf16>(m).backward(m->fwd_tokens, true)
                                                   : Step<float>(m).backward(m->fwd_tokens, true);
      m->have_targets = false;
    }
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(m->st, &graph);
    m->prof_on = prof;
    if (rc) {
      if (graph) cudaGraphDestroy(graph);
      return rc;
    }
    if (e != cudaSuccess) FAIL(m, GPT2_ERR_CUDA, "stream capture failed: %s", cudaGetErrorString(e));
    e = cudaGraphInstantiate(&m->gexec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
      m->gexec = nullptr;
      FAIL(m, GPT2_ERR_CUDA, "graph instantiation failed: %s", cudaGetErrorString(e));
    }
    // the capture counted its launches once; replays count them again below
    m->g_launches = gpt2_total_launches() - l0;
    gpt2_count_launches(-(int)m->g_launches);
    m->g_tok = tokens_dev;
    m->g_tgt = targets_dev;
  }
  CK(m, cudaGraphLaunch(m->gexec, m->st));
  gpt2_count_launches((int)m->g_launches);
  m->have_targets = false;  // the backward in the graph consumed dlogits
  m->logits_valid = false;
  m->loss_valid = true;
  m->fwd_tokens = tokens_dev;
  return GPT2_OK;
}

int gpt2_get_loss(gpt2* m, float* loss_host) {
  if (!m || !loss_host) return GPT2_ERR_INVALID_ARG;
  if (!m->loss_valid) FAIL(m, GPT2_ERR_BAD_ORDER, "no forward with targets has run");
  CK(m, cudaMemcpyAsync(loss_host, m->at<float>(m->bl.loss), 4, cudaMemcpyDeviceToHost, m->st));
  int rc = check_flags(m);
  if (rc) return rc;
  if (!std::isfinite(*loss_host)) FAIL(m, GPT2_ERR_NAN, "loss is not finite (%f)", *loss_host);
  return GPT2_OK;
}

int gpt2_get_params(gpt2* m, int tensor, float* host) {
  if (!m || !host || tensor < 0 || tensor >= GPT2_NUM_TENSORS) return GPT2_ERR_INVALID_ARG;
  CK(m, cudaMemcpyAsync(host, m->at<float>(m->bl.params) + m->pl.off[tensor], m->pl.numel[tensor] * 4,
                        cudaMemcpyDeviceToHost, m->st));
  CK(m, cudaStreamSynchronize(m->st));
  return GPT2_OK;
}

int gpt2_set_params(gpt2* m, int tensor, const float* host) {
  if (!m || !host || tensor < 0 || tensor >= GPT2_NUM_TENSORS) return GPT2_ERR_INVALID_ARG;
  float* dst = m->at<float>(m->bl.params) + m->pl.off[tensor];
  CK(m, cudaMemcpyAsync(dst, host, m->pl.numel[tensor] * 4, cudaMemcpyHostToDevice, m->st));
  if (m->cfg.precision == GPT2_PRECISION_BF16) {
    CK(m, convert_f32_bf16(m->at<bf16>(m->bl.pbf) + m->pl.off[tensor], dst, (long long)m->pl.numel[tensor], m->st));
    gpt2_count_launches(1);
  }
  CK(m, cudaStreamSynchronize(m->st));
  return GPT2_OK;
}

int gpt2_get_grads(gpt2* m, int tensor, float* host) {
  if (!m || !host || tensor < 0 || tensor >= GPT2_NUM_TENSORS) return GPT2_ERR_INVALID_ARG;
  CK(m, cudaMemcpyAsync(host, m->at<float>(m->bl.grads) + m->pl.off[tensor], m->pl.numel[tensor] * 4,
                        cudaMemcpyDeviceToHost, m->st));
  CK(m, cudaStreamSynchronize(m->st));
  return GPT2_OK;
}

static int copy_act_to_host(gpt2* m, size_t off, size_t n, float* host) {
  if (m->cfg.precision == GPT2_PRECISION_BF16) {
    std::vector<uint16_t> tmp(n);
    CK(m, cudaMemcpyAsync(tmp.data(), m->base + off, n * 2, cudaMemcpyDeviceToHost, m->st));
    CK(m, cudaStreamSynchronize(m->st));
    for (size_t i = 0; i < n; i++) {
      uint32_t u = (uint32_t)tmp[i] << 16;
      memcpy(&host[i], &u, 4);
    }
  } else {
    CK(m, cudaMemcpyAsync(host, m->base + off, n * 4, cudaMemcpyDeviceToHost, m->st));
    CK(m, cudaStreamSynchronize(m->st));
  }
  return GPT2_OK;
}

int gpt2_get_logits(gpt2* m, float* host) {
  if (!m || !host) return GPT2_ERR_INVALID_ARG;
  if (!m->logits_valid) FAIL(m, GPT2_ERR_BAD_ORDER, "logits are kept only by a forward without targets");
  int rc = copy_act_to_host(m, m->bl.logits, (size_t)m->BT * m->cfg.Vp, host);
  return rc ? rc : check_flags(m);
}

int gpt2_get_losses(gpt2* m, float* host) {
  if (!m || !host) return GPT2_ERR_INVALID_ARG;
  if (!m->loss_valid) FAIL(m, GPT2_ERR_BAD_ORDER, "no forward with targets has run");
  CK(m, cudaMemcpyAsync(host, m->at<float>(m->bl.losses), (size_t)m->BT * 4, cudaMemcpyDeviceToHost, m->st));
  return check_flags(m);
}

int gpt2_sync(gpt2* m) {
  if (!m) return GPT2_ERR_INVALID_ARG;
  return check_flags(m);
}

uint64_t gpt2_launch_count(gpt2* m) {
  (void)m;
  return (uint64_t)gpt2_total_launches();
}

const char* gpt2_last_error(gpt2* m) { return m ? m->err.c_str() : g_create_err.c_str(); }

int gpt2_profile_gemm(gpt2* m, int enable) {
  if (!m) return GPT2_ERR_INVALID_ARG;
  if (enable && m->prof_ev.empty()) {
    const size_t n = 8192;
    m->prof_ev.resize(2 * n);
    for (auto& e : m->prof_ev) CK(m, cudaEventCreate(&e));
    m->prof_flops.assign(n, 0.0);
  }
  m->prof_on = enable != 0;
  return GPT2_OK;
}

int gpt2_profile_read(gpt2* m, double* ms_total, uint64_t* launches, double* flops_total) {
  if (!m || !ms_total || !launches || !flops_total) return GPT2_ERR_INVALID_ARG;
  CK(m, cudaStreamSynchronize(m->st));
  double ms = 0, fl = 0;
  for (size_t i = 0; i < m->prof_n; i++) {
    float t = 0.f;
    CK(m, cudaEventElapsedTime(&t, m->prof_ev[2 * i], m->prof_ev[2 * i + 1]));
    ms += t;
    fl += m->prof_flops[i];
  }
  *ms_total = ms;
  *launches = m->prof_n;
  *flops_total = fl;
  m->prof_n = 0;
  return GPT2_OK;
}

void gpt2_destroy(gpt2* m) {
  if (!m) return;
  if (m->gexec) cudaGraphExecDestroy(m->gexec);
  for (auto& e : m->prof_ev) cudaEventDestroy(e);
  delete m;
}

}  // extern "C"
