"""Write the oracle's expected values for one step of a larger GPT-2 config.

Runs only the CPU oracle (float32, like the pages' CPU trainer).  The step is
that of the batched workload (B sequences of T = 1024 tokens, the mean loss
over all B*T positions), computed one sequence at a time so that the saved
attention matrices of one sequence fit in host memory: the oracle's backward
of sequence b seeds each of its T positions with 1/T, the gradients of all B
sequences accumulate in the oracle's gradient buffers, and the sum is divided
by B at the end -- the gradient of the mean over B*T positions, summed in a
different order than a batched run would (float32 rounding only).

Configs (tokens: Zipf(1.1) over V = 50257 from seed 1234, B*(T+1) drawn and
shifted by one; weights from seed 1234; same as the device side):
  350m  L=24 C=1024 H=16 B=8   -> tests/golden/oracle_350m.npz
  1.6b  L=48 C=1600 H=25 B=8   -> tests/golden/oracle_1p6b.npz
  124m  L=12 C=768  H=12 B=16  -> tests/golden/oracle_124m_logits.npz (forward
        only: logits rows and pos_scale; the rest of the 124M step is in
        oracle_124m.npz)

Stores:
  loss          []          mean loss of the step
  pos_losses    [B*T]       per-position cross-entropy
  logit_pos     [R, 2]      (b, t) of the stored logit rows, one per sequence
  logit_rows    [R, Vp]     the oracle's logits at those positions
  logit_bound   [R, Vp]     sum over channels of |lnf[b,t,c] * wte[v,c]| (the
                            magnitude scale of each logit's dot product)
  pos_scale     [B*T]       per position, that scale at the target logit plus
                            its softmax-weighted mean over the vocabulary (the
                            magnitude scale of the position's loss, lse - z_t)
  grad_idx_<n>, grad_val_<n>, grad_norm_<n>   as in oracle_124m.npz

Usage: python tests/golden/make_oracle_config.py 350m|1.6b|124m
(The 124m run stores the logit rows of the first two sequences only.)
1.6b needs about 35 GB of RAM and a quarter of an hour on an 8-core host.
"""
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402
from synthetic import zipf_tokens  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
CONFIGS = {
    "350m": (O.Config(L=24, C=1024, H=16, V=50257, Vp=50304, maxT=1024), 8, "oracle_350m.npz"),
    "1.6b": (O.Config(L=48, C=1600, H=25, V=50257, Vp=50304, maxT=1024), 8, "oracle_1p6b.npz"),
    "124m": (O.GPT2_124M, 16, "oracle_124m_logits.npz"),
}
T, SEED, SAMPLES = 1024, 1234, 2048


def logit_position(b):
    return (b * 131 + 17) % T


def main():
    name = sys.argv[1]
    cfg, B, fname = CONFIGS[name]
    logits_only = name == "124m"
    tok, tgt = zipf_tokens(B, T, cfg.V, SEED)
    t0 = time.time()
    m = O.GPT2(cfg, SEED, np.float32)
    m.m = m.v = None  # no update is taken: the moments are not needed
    print(f"init {time.time() - t0:.1f}s", flush=True)
    out = {"logit_pos": [], "logit_rows": [], "logit_bound": []}
    losses, scales = [], []
    abs_wte = np.abs(m.params["wte"])
    for b in range(B):
        t0 = time.time()
        loss = m.forward(tok[b:b + 1], tgt[b:b + 1])
        if not logits_only or b < 2:
            t = logit_position(b)
            lnf = m.cache["lnf"][0, t].astype(np.float64)
            out["logit_pos"].append((b, t))
            out["logit_rows"].append(m.cache["logits"][0, t].astype(np.float32))
            out["logit_bound"].append((np.abs(m.params["wte"].astype(np.float64)) @ np.abs(lnf)).astype(np.float32))
        losses.append(m.cache["losses"].reshape(-1).astype(np.float32))
        # per position: sum_c |lnf_c wte_vc| at the target and softmax-weighted over v < V
        S = np.abs(m.cache["lnf"][0]) @ abs_wte.T
        probs = O.softmax_forward(m.cache["logits"][0], cfg.V)
        s_t = np.take_along_axis(S, tgt[b][:, None].astype(np.int64), axis=1)[:, 0]
        scales.append((s_t + (probs * S).sum(axis=1)).astype(np.float32))
        del S, probs
        if not logits_only:
            m.backward()
        m.cache = None
        print(f"sequence {b}: loss {loss:.6f} ({time.time() - t0:.1f}s)", flush=True)
    for k in ("logit_pos", "logit_rows", "logit_bound"):
        out[k] = np.array(out[k])
    out["pos_scale"] = np.concatenate(scales)
    if not logits_only:
        out["pos_losses"] = np.concatenate(losses)
        out["loss"] = np.float64(np.mean(out["pos_losses"].astype(np.float64)))
        rng = np.random.default_rng(4321)
        for n, _ in O.param_shapes(cfg):
            g = m.grads[n].reshape(-1)
            g /= np.float32(B)
            idx = np.sort(rng.choice(g.size, min(SAMPLES, g.size), replace=False)).astype(np.int64)
            out["grad_idx_" + n] = idx
            out["grad_val_" + n] = g[idx].astype(np.float32)
            out["grad_norm_" + n] = np.float64(np.linalg.norm(g.astype(np.float64)))
    path = os.path.join(HERE, fname)
    with open(path + ".tmp", "wb") as f:
        np.savez_compressed(f, **out)
    os.replace(path + ".tmp", path)
    print("wrote", path)


if __name__ == "__main__":
    main()
