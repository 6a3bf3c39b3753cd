"""Write the oracle's expected values for the GPT-2 124M training workload.

Runs only the CPU oracle (float32, like the pages' CPU trainer) on the seeded
synthetic batch: GPT-2 124M (L=12, C=768, H=12, V=50257 -> Vp=50304), B=16,
T=1024, Zipf(1.1) tokens from seed 1234, initial weights from seed 1234,
AdamW lr 6e-4, betas (0.9, 0.95), eps 1e-8, weight decay 0.1 on 2-D tensors,
20 steps on the one fixed batch.

Stores (tests/golden/oracle_124m.npz):
  losses        [20]        mean loss before each update
  pos_losses0   [B*T]       per-position cross-entropy of the first forward
  grad_idx_<n>  [S]         flat indices sampled from tensor n (seed 4321)
  grad_val_<n>  [S]         the oracle's step-0 gradient at those indices
  grad_norm_<n> []          the full tensor's step-0 gradient L2 norm

Usage: python tests/golden/make_oracle_124m.py [--steps 20] [--out PATH]
Takes roughly an hour on an 8-core host and about 35 GB of RAM.
"""
import argparse
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402
from synthetic import zipf_tokens  # noqa: E402

B, T, SEED = 16, 1024, 1234
LR, B1, B2, EPS, WD = 6e-4, 0.9, 0.95, 1e-8, 0.1
SAMPLES = 2048


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--out", default=os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_124m.npz"))
    a = ap.parse_args()
    cfg = O.GPT2_124M
    tok, tgt = zipf_tokens(B, T, cfg.V, SEED)
    t0 = time.time()
    m = O.GPT2(cfg, SEED, np.float32)
    print(f"init {time.time() - t0:.1f}s", flush=True)
    out = {}
    losses = []
    rng = np.random.default_rng(4321)
    for step in range(a.steps):
        t0 = time.time()
        m.zero_grad()
        loss = m.forward(tok, tgt)
        if step == 0:
            out["pos_losses0"] = m.cache["losses"].reshape(-1).astype(np.float32)
        m.backward()
        if step == 0:
            for n, _ in O.param_shapes(cfg):
                g = m.grads[n].reshape(-1)
                idx = np.sort(rng.choice(g.size, min(SAMPLES, g.size), replace=False)).astype(np.int64)
                out["grad_idx_" + n] = idx
                out["grad_val_" + n] = g[idx].astype(np.float32)
                out["grad_norm_" + n] = np.float64(np.linalg.norm(g.astype(np.float64)))
        m.adamw_step(LR, B1, B2, EPS, WD, step + 1)
        losses.append(loss)
        print(f"step {step} loss {loss:.6f} ({time.time() - t0:.1f}s)", flush=True)
        out["losses"] = np.array(losses, dtype=np.float64)
        # write-then-rename, so a reader never sees a half-written file
        with open(a.out + ".tmp", "wb") as f:
            np.savez_compressed(f, **out)
        os.replace(a.out + ".tmp", a.out)


if __name__ == "__main__":
    main()
