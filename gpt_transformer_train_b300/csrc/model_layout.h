// The memory planner: every byte the training step touches lives in ONE
// caller-provided device buffer, laid out once at create time.  This is the
// single pre-planned allocation of the llm.c design ("llm.c's Origin and the
// Future of LLM Compilers", [3:47] Pure C: parameters, grads, AdamW m and v
// and activations are planned up front and never allocated again).
#pragma once
#include <cstddef>
#include <cstdint>

#include "../../include/gpt2.h"

struct ParamLayout {
  size_t numel[GPT2_NUM_TENSORS];
  size_t off[GPT2_NUM_TENSORS + 1];  // element offsets, canonical order
  size_t total;
};

inline ParamLayout param_layout(const gpt2_config& c) {
  ParamLayout p{};
  size_t L = c.L, C = c.C;
  size_t n[GPT2_NUM_TENSORS] = {
      (size_t)c.Vp * C, (size_t)c.max_T * C,  // wte, wpe
      L * C, L * C,                           // ln1w, ln1b
      L * 3 * C * C, L * 3 * C,               // qkvw, qkvb
      L * C * C, L * C,                       // attprojw, attprojb
      L * C, L * C,                           // ln2w, ln2b
      L * 4 * C * C, L * 4 * C,               // fcw, fcb
      L * C * 4 * C, L * C,                   // fcprojw, fcprojb
      C, C,                                   // lnfw, lnfb
  };
  size_t o = 0;
  for (int t = 0; t < GPT2_NUM_TENSORS; t++) {
    p.numel[t] = n[t];
    p.off[t] = o;
    o += n[t];
  }
  p.off[GPT2_NUM_TENSORS] = o;
  p.total = o;
  return p;
}

// Byte offsets of every region inside the one buffer (256-byte aligned).
struct BufferLayout {
  size_t params, grads, m, v, pbf;          // fp32 x4, bf16 copy (bf16 mode)
  size_t resid, ln, ln_mean, ln_rstd;       // [(2L+1)][BT][C], stats [(2L+1)][BT]
  size_t qkv, atty, lse, fch, fchg;         // per layer
  size_t proj, logits, losses, loss;        // temporaries / classifier
  size_t lstats;                            // classifier per-tile row statistics (bf16 mode)
  size_t dres, dresc, dfch, dqkv, dsmall;  // activation gradients (dresc, dfch, dqkv: per layer)
  size_t attD, attS, partial, keys, ws, ws_floats, gnorm, flags, tok, tgt;
  size_t dec;                               // one-position inference scratch (see Step::dec_*)
  size_t wfold, fold_s, fold_c;             // ln_fold: folded qkv | fc weights [L][7C][C] bf16, their sums [L][7C]
  size_t decbar;                            // grid-barrier counter of the one-launch decode step
  size_t total;
};

int validate_config(const gpt2_config& c, const char** why);
BufferLayout buffer_layout(const gpt2_config& c);
void init_params_host(const gpt2_config& c, uint64_t seed, float* out);
