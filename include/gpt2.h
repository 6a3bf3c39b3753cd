/*
 * gpt2.h — C ABI of a B300-native (sm_103a) GPT-2 training step on one GPU.
 *
 * The operation is the one the llm.c pages describe: gpt2_forward (token and
 * position embedding, pre-LN blocks, tied classifier, softmax cross-entropy),
 * gpt2_backward (each layer's hand-derived backward, run in reverse), and the
 * AdamW update over one pre-planned contiguous buffer.  Sources:
 *   - "llm.c: GPT-2 training in plain C, with every gradient written by hand",
 *     §2 How the code works (layer list, backward in reverse, one memory block)
 *   - "llm.c's Origin and the Future of LLM Compilers" (CUDA MODE talk),
 *     [3:47] Pure C (all memory planned and allocated once) and
 *     [13:50] Avengers Assemble (mixed precision, fused kernels, determinism).
 *
 * Conventions for every call below
 *   - Return value: GPT2_OK (0) or a negative GPT2_ERR_* code; the message of
 *     the last failure on a handle is available from gpt2_last_error().
 *   - Device pointers are plain CUDA device addresses in the current device's
 *     context; the caller owns all memory passed in.  The library never calls
 *     cudaMalloc/cudaFree: the model lives in ONE caller-provided device buffer
 *     of gpt2_required_bytes() bytes.
 *   - Work is enqueued on the caller's CUDA stream (a cudaStream_t passed as
 *     void*, NULL = legacy default stream).  Calls return without waiting,
 *     except where a host pointer receives a result (loss_host, gpt2_get_*),
 *     which synchronises that stream.
 *   - Weights are stored [out_features][in_features] (K contiguous); token and
 *     target arrays are int32 [B][T] row-major on the device.
 */
#ifndef GPT2_B300_H
#define GPT2_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
#define GPT2_OK                    0
#define GPT2_ERR_INVALID_CONFIG   -1  /* shape/precision not supported        */
#define GPT2_ERR_BUFFER_TOO_SMALL -2  /* dev_buf smaller than required bytes  */
#define GPT2_ERR_BAD_ORDER        -3  /* e.g. backward without a prior forward */
#define GPT2_ERR_TOKEN_RANGE      -4  /* a token or target outside [0, V)      */
#define GPT2_ERR_CUDA             -5  /* a CUDA runtime call failed            */
#define GPT2_ERR_NAN              -6  /* the loss is not finite                */
#define GPT2_ERR_INVALID_ARG      -7  /* NULL handle/pointer, bad tensor id    */
#define GPT2_ERR_TIMEOUT          -8  /* a kernel's bounded wait ran out       */

#define GPT2_PRECISION_FP32 0  /* fp32 activations and SIMT kernels (exact checks) */
#define GPT2_PRECISION_BF16 1  /* bf16 activations/weights, fp32 master, tensor cores */

/* Canonical parameter tensor ids (the order of the one parameter buffer). */
enum {
  GPT2_WTE = 0, GPT2_WPE, GPT2_LN1W, GPT2_LN1B, GPT2_QKVW, GPT2_QKVB,
  GPT2_ATTPROJW, GPT2_ATTPROJB, GPT2_LN2W, GPT2_LN2B, GPT2_FCW, GPT2_FCB,
  GPT2_FCPROJW, GPT2_FCPROJB, GPT2_LNFW, GPT2_LNFB, GPT2_NUM_TENSORS
};

/* Model and batch shape.  L layers, C channels, H heads (hd = C/H), max_T
 * positions in wpe, V real vocabulary entries, Vp >= V padded rows of wte
 * (logit columns V..Vp-1 are masked out of the softmax), batch B x T tokens.
 * Precision GPT2_PRECISION_BF16 needs C % 64 == 0, hd == 64, T % 128 == 0,
 * (B*T) % 128 == 0, Vp % 128 == 0; GPT2_PRECISION_FP32 needs C % 4 == 0 and
 * hd <= 128.  Both need C <= 2048, T <= max_T, B*T <= 32768, V <= 65535. */
/* recompute: 0 keeps every activation the backward reads (fastest); 1 keeps
 * only the fc pre-activation and recomputes GELU of it in the backward; 2
 * also recomputes every LayerNorm output from the stored residual stream and
 * statistics (the pages' activation-recompute option, "llm.c's Origin and the
 * Future of LLM Compilers" [13:50]).  With recompute > 0 the weight gradients
 * run inside the layer loop and only one layer's GELU / LayerNorm outputs and
 * output gradients are held at a time, which shrinks the buffer; the forward
 * results and the gradients are those of recompute 0. */
/* ln_fold (bf16 with recompute 2 only): the LayerNorms in front of the qkv
 * and fc products are folded into those products (the pages' fused LayerNorm
 * -> matmul, [13:50]): each step first forms W diag(gamma) (bf16) and the two
 * per-output-column sums the fold needs, the LayerNorm kernels then write
 * only the residual stream and its statistics, and the qkv and fc products
 * run on the residual stream and normalise in their epilogue
 * (gpt2_op_matmul_lnfold).  With recompute 2 the backward rebuilds the
 * LayerNorm outputs it needs anyway, so no normalised activation is written
 * in the forward.  0 = off. */
typedef struct {
  int L, C, H, max_T, V, Vp, B, T;
  int precision;
  int recompute;
  int ln_fold;
} gpt2_config;

typedef struct gpt2 gpt2;  /* opaque handle; host memory owned by the library */

/* Number of parameters (sum of all canonical tensors). 0 on a bad config. */
size_t gpt2_num_parameters(const gpt2_config* cfg);
/* Element count of one canonical tensor, 0 on a bad id or config. */
size_t gpt2_tensor_numel(const gpt2_config* cfg, int tensor);
/* Exact byte size of the single device buffer the model needs (parameters,
 * grads, AdamW moments, bf16 weight copy, activations, scratch). 0 on a bad
 * config. */
size_t gpt2_required_bytes(const gpt2_config* cfg);

/* Host-only: write the seeded initial parameters (canonical order, fp32,
 * gpt2_num_parameters() floats) to host_out.  The generator is SplitMix64
 * used as a counter-based stream (element i draws outputs 2i and 2i+1) and
 * Box-Muller in double; weights N(0, 0.02), residual projections
 * N(0, 0.02/sqrt(2L)), wte pad rows 0, LayerNorm gains 1, biases 0. */
int gpt2_init_params_host(const gpt2_config* cfg, uint64_t seed, float* host_out);

/* Create a model inside dev_buf (>= gpt2_required_bytes) and initialise its
 * parameters from seed (as gpt2_init_params_host), zero grads and moments.
 * stream: the cudaStream_t all later calls enqueue on.  *out receives the
 * handle; on failure *out is NULL and the code says why. */
int gpt2_create(const gpt2_config* cfg, uint64_t seed, void* dev_buf, size_t bytes,
                void* cuda_stream, gpt2** out);

/* Forward pass over tokens_dev [B][T].  With targets_dev non-NULL it also
 * computes per-position cross-entropy, the mean loss, and writes dlogits =
 * (softmax - onehot)/(B*T) in place of the logits (ready for gpt2_backward);
 * with targets_dev NULL the logits are kept (gpt2_get_logits).  loss_host
 * non-NULL: synchronise, check the range flags and store the mean loss. */
int gpt2_forward(gpt2* m, const int32_t* tokens_dev, const int32_t* targets_dev, float* loss_host);

/* Backward pass; needs a forward with targets since the last backward.
 * Parameter gradients ACCUMULATE (+=) into the grad buffer. */
int gpt2_backward(gpt2* m);

/* Zero the parameter-gradient buffer. */
int gpt2_zero_grad(gpt2* m);

/* AdamW over the whole parameter buffer, t >= 1 the step number:
 * m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2; p -= lr (m/(1-b1^t)) /
 * (sqrt(v/(1-b2^t)) + eps) + lr wd p, with wd applied to the 2-D tensors
 * (wte, wpe, qkvw, attprojw, fcw, fcprojw) only.  Refreshes the bf16 copy. */
int gpt2_adamw_step(gpt2* m, float lr, float b1, float b2, float eps, float wd, int t);

/* Forward (with targets) + backward as ONE captured CUDA graph, the backward
 * writing fresh gradients: the first writer of every gradient stores instead
 * of adding, so no zero_grad memset runs and the previous gradients are
 * overwritten.  The first call captures the launches on the model's stream
 * for these token/target device pointers and instantiates the graph; later
 * calls with the same pointers replay it (one launch; the step's ~200
 * kernels run without host gaps).  New pointers recapture.  The contents of
 * the token arrays are read at replay time.  Needs a created (non-default)
 * stream; run AdamW (and clipping) after it as usual.  Equivalent to
 * gpt2_zero_grad; gpt2_forward(tokens, targets, NULL); gpt2_backward, up to
 * the sign of zero gradients (0 + x and x differ only there). */
int gpt2_graph_step(gpt2* m, const int32_t* tokens_dev, const int32_t* targets_dev);

/* Gradient-norm clipping, the step before AdamW (the llm.c tour names a
 * global_norm component and LR warmup/decay schedulers; no formulas are given,
 * the plainest readings are taken).  gpt2_clip_grad_norm enqueues the global L2
 * norm of the whole gradient buffer and the factor min(1, max_norm /
 * (norm + 1e-6)); the next gpt2_adamw_step multiplies every gradient by that
 * factor (on the device, no synchronisation), later steps do not unless this
 * is called again.  max_norm > 0.  gpt2_get_grad_norm synchronises and returns
 * the norm (before clipping) of the last gpt2_clip_grad_norm. */
int gpt2_clip_grad_norm(gpt2* m, float max_norm);
int gpt2_get_grad_norm(gpt2* m, float* norm_host);

/* Learning rate at 0-based step: linear warmup to max_lr over `warmup` steps
 * (step s gets max_lr (s+1)/warmup), then a cosine from max_lr down to
 * final_frac * max_lr at step `total`, and that floor afterwards.  Host only. */
float gpt2_lr_schedule(float max_lr, float final_frac, int warmup, int total, int step);

/* One whole step from HOST token arrays (pinned or pageable int32 [B][T]):
 * upload, forward with loss, backward (grads are zeroed first), AdamW at step
 * t, and read the mean loss back into *loss_host (synchronises).  On a
 * created stream the forward/backward part runs as gpt2_graph_step over the
 * model's own token buffers. */
int gpt2_step_host(gpt2* m, const int32_t* tokens_host, const int32_t* targets_host,
                   float lr, float b1, float b2, float eps, float wd, int t, float* loss_host);

/* Inference with a KV cache (the pages' CPU sampler reruns the whole forward
 * for every new token and keeps no cache: "llm.c: GPT-2 training in plain C
 * ...", §6 Reality check; here the keys and values of earlier positions are
 * kept).  The cache is the model's qkv activation buffer; any training
 * forward replaces it, and the inference calls overwrite the training
 * activations.
 *   gpt2_infer_prefill: the forward over tokens_dev [B][T] (logits kept),
 *     taking positions 0..n-1 as the prompt of every sequence (1 <= n <= T;
 *     later positions of tokens_dev only need to hold valid token ids); the
 *     logits of position n-1 become the last logits.
 *   gpt2_infer_step: the forward of one new position pos (== the number of
 *     positions cached, < T) of every sequence from next-token ids
 *     tokens_dev [B] (device int32), reading keys and values 0..pos-1 from the
 *     cache and adding position pos to it; its logits become the last logits.
 *   gpt2_sample: one token per sequence from the last logits into
 *     out_tokens_dev [B] (device int32): temperature 0 takes the largest of
 *     the first V logits (lowest index on ties); a temperature > 0 takes the
 *     first index whose cumulative softmax(logits / temperature) probability
 *     exceeds coins_dev[b] (device float, uniform in [0, 1): the caller draws
 *     them), the sampler of the pages' CPU trainer.
 *   gpt2_get_infer_logits: the last logits as B x Vp host floats
 *     (synchronises; reports a token out of range as GPT2_ERR_TOKEN_RANGE).
 * Asynchronous on the model's stream except gpt2_get_infer_logits. */
int gpt2_infer_prefill(gpt2* m, const int32_t* tokens_dev, int n);
int gpt2_infer_step(gpt2* m, const int32_t* tokens_dev, int pos);
int gpt2_sample(gpt2* m, float temperature, const float* coins_dev, int32_t* out_tokens_dev);
int gpt2_get_infer_logits(gpt2* m, float* host);

/* Host copies (synchronising).  tensor is a GPT2_* id; host holds
 * gpt2_tensor_numel() floats.  Logits: B*T*Vp floats, only after a forward
 * without targets.  Losses: B*T per-position losses of the last forward with
 * targets.  gpt2_get_loss: the mean loss of that forward. */
int gpt2_get_params(gpt2* m, int tensor, float* host);
int gpt2_set_params(gpt2* m, int tensor, const float* host);
int gpt2_get_grads(gpt2* m, int tensor, float* host);
int gpt2_get_logits(gpt2* m, float* host);
int gpt2_get_losses(gpt2* m, float* host);
int gpt2_get_loss(gpt2* m, float* loss_host);

/* Kernel timing for roofline measurement: while enabled, the library records
 * a CUDA event pair on its stream around every GEMM launch (fp32 or tensor
 * core) and sums the algorithmic FLOPs (2*M*N*K) of those launches.
 * gpt2_profile_read synchronises, returns the summed event time, the launch
 * count and the FLOPs since the last read, and resets them.  At most 8192
 * launches are recorded between reads (later ones are not timed). */
int gpt2_profile_gemm(gpt2* m, int enable);
int gpt2_profile_read(gpt2* m, double* ms_total, uint64_t* launches, double* flops_total);

/* Synchronise the stream and report range/timeout flags raised by kernels. */
int gpt2_sync(gpt2* m);
/* Number of kernel launches the library enqueued since creation. */
uint64_t gpt2_launch_count(gpt2* m);
/* Message for the last failure on m ("" if none); m may be NULL for create. */
const char* gpt2_last_error(gpt2* m);
/* Free the handle (host memory only; the device buffer is the caller's). */
void gpt2_destroy(gpt2* m);

#ifdef __cplusplus
}
#endif
#endif /* GPT2_B300_H */
