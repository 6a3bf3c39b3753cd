"""Element-wise parity bounds shared by the GPU tests.

Every check here is |got - ref| <= bound, element by element, with ref taken
in float64 from exactly the values the kernel saw (its bf16 inputs as
stored).  The bounds follow the arithmetic:

  * bf16 output: one round-to-nearest-even to 8 significant bits, at most
    2^-8 of the value (U8 |ref|); fp32 output: 2^-22 |ref| (a few ulp).
  * fp32 accumulation of a K-long dot product: ACC * sum_k |a_k b_k| with
    ACC = 2^-16.  The worst case of a sequential fp32 sum is K * 2^-24 times
    that sum; the realised error is a random walk far below it, and 2^-16
    stays two orders of magnitude above the realised error for K <= 16384
    while a wrong element (a misplaced tile, a dropped term) misses it by
    orders of magnitude.
  * attention: P and dS enter the tensor-core products as bf16 and a quarter
    of the exponentials come from a polynomial (relative error below 2^-13),
    so each output may move by C_ATT * 2^-8 times the sum of the magnitudes
    of its terms (see attention_bounds) on top of its own output rounding.

The constants are written once here; the design notes list them.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle as O

U8 = 2.0 ** -8        # bf16 unit roundoff (8 significant bits)
U24 = 2.0 ** -22      # fp32 output: a few ulp
ACC = 2.0 ** -16      # fp32 accumulation allowance per unit of sum |a b|
C_ATT_FWD = 2.0       # attention forward: P in bf16 + exponentials
C_ATT_BWD = 4.0       # attention backward: P, dS in bf16, D from the stored output
C_LOGITS = 4.0        # whole-model logits: bf16 weight copy + bf16 activations upstream
TINY = 2.0 ** -126    # fp32 exponentials flush to zero (or clamp) below the smallest normal
SUB = 2.0 ** -133     # bf16 subnormal step: the absolute rounding floor of a bf16 output


def check(got, ref, bound, what=""):
    """Assert |got - ref| <= bound element-wise; report the worst element."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    bound = np.broadcast_to(np.asarray(bound, np.float64), ref.shape)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref)
    bad = ~(err <= bound)  # NaN counts as a failure
    if bad.any():
        ratio = np.where(bad, np.nan_to_num(err / np.maximum(bound, 1e-300), nan=np.inf), 0)
        i = np.unravel_index(np.argmax(ratio), ratio.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of bound; worst at {i}: "
                             f"got {got[i]!r}, ref {ref[i]!r}, bound {bound[i]!r} (ratio {ratio[i]:.3g})")
    worst = float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0
    log = os.environ.get("GPT2_PARITY_LOG")
    if log:  # margin record: the largest |got - ref| / bound of each check
        with open(log, "a") as f:
            f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", ""), "what": what,
                                "n": int(err.size), "max_ratio": worst}) + "\n")
    return worst


def gemm_ref(A, B, akm, bkm, M, N, K):
    Am = A.reshape(M, K) if akm else A.reshape(K, M).T
    Bn = B.reshape(N, K) if bkm else B.reshape(K, N).T
    Am = Am.astype(np.float64)
    Bn = Bn.astype(np.float64)
    return Am @ Bn.T, np.abs(Am) @ np.abs(Bn).T


def gemm_bound(ref, absprod, bf16_out=True):
    return (U8 if bf16_out else U24) * np.abs(ref) + ACC * absprod


def gelu_bound(g_ref, pre):
    """bf16 GELU of a stored pre-activation: output rounding plus the
    exp2/divide approximation (below 2^-21 of the value; 2^-18 |x| allowed)."""
    return U8 * np.abs(g_ref) + 2.0 ** -18 * np.abs(pre)


def gelu_bwd_bound(ref, acc, absprod, pre):
    """bf16 acc * GELU'(pre): output rounding, the accumulation allowance
    scaled by |GELU'|, and 2^-17 |acc| for the approximate GELU'."""
    dg = np.abs(O.gelu_backward(np.asarray(pre, np.float64), np.ones_like(pre, dtype=np.float64)))
    return U8 * np.abs(ref) + ACC * absprod * dg + 2.0 ** -17 * np.abs(acc)


def attention_bounds(qkv, dout, o_kernel, H):
    """Float64 oracle results and element-wise bounds of causal attention.

    qkv [B,T,3C], dout [B,T,C], o_kernel [B,T,C] (the kernel's stored output,
    from which its backward forms D = rowsum(dO * O)).  Returns a dict of
    (ref, bound) for 'out', 'dq', 'dk', 'dv', each [B,T,C].
      out:  U8 |O| + C_ATT_FWD U8 sum_j P_ij |V_j|
      dv:   U8 |dV| + C_ATT_FWD U8 sum_i P_ij |dO_i|
      dq:   U8 |dQ| + C_ATT_BWD U8 s sum_j E_ij |K_j|
      dk:   U8 |dK| + C_ATT_BWD U8 s sum_i E_ij |Q_i|
    with s = 1/sqrt(hd) and E_ij = P_ij (|dP_ij| + |D_i| + sum_d |dO_id O_id|),
    the magnitude of dS_ij = P_ij (dP_ij - D_i) and of its rounding sources.
    Each also gets the underflow floor of fp32 exponentials: a probability
    below 2^-126 comes out as 0 or 2^-126, so every causal term may be off by
    TINY (out: TINY sum_j |V_j|, dv: TINY sum_i |dO_i|, dq/dk: C_ATT_BWD TINY s
    sum (|dP_ij| + |D_i|) |K_j| (|Q_i|)), and the bf16 subnormal step SUB.
    These matter only where the scores span more than 2^126 within a row.
    """
    qkv = np.asarray(qkv, np.float64)
    dout = np.asarray(dout, np.float64)
    B, T, C3 = qkv.shape
    C = C3 // 3
    hd = C // H
    s = 1.0 / math.sqrt(hd)
    ro, att = O.attention_forward(qkv, H)
    rd = O.attention_backward(dout, qkv, att, H)

    def heads(x):
        return x.reshape(B, T, H, hd).transpose(0, 2, 1, 3)

    def merge(x):
        return x.transpose(0, 2, 1, 3).reshape(B, T, C)

    q, k, v = heads(qkv[..., :C]), heads(qkv[..., C:2 * C]), heads(qkv[..., 2 * C:])
    do, ok = heads(dout), heads(np.asarray(o_kernel, np.float64))
    dP = do @ v.transpose(0, 1, 3, 2)
    D = (do * heads(ro)).sum(-1)
    E = att * (np.abs(dP) + np.abs(D)[..., None] + (np.abs(do) * np.abs(ok)).sum(-1)[..., None])
    causal = np.tril(np.ones((T, T)))
    F = causal * (np.abs(dP) + np.abs(D)[..., None])
    out_b = U8 * np.abs(ro) + C_ATT_FWD * U8 * merge(att @ np.abs(v)) + TINY * merge(causal @ np.abs(v)) + SUB
    dv_b = C_ATT_FWD * U8 * merge(att.transpose(0, 1, 3, 2) @ np.abs(do)) + TINY * merge(causal.T @ np.abs(do)) + SUB
    dq_b = C_ATT_BWD * s * merge((U8 * E + TINY * F) @ np.abs(k)) + SUB
    dk_b = C_ATT_BWD * s * merge((U8 * E + TINY * F).transpose(0, 1, 3, 2) @ np.abs(q)) + SUB
    rq, rk, rv = rd[..., :C], rd[..., C:2 * C], rd[..., 2 * C:]
    return {
        "out": (ro, out_b),
        "dq": (rq, U8 * np.abs(rq) + dq_b),
        "dk": (rk, U8 * np.abs(rk) + dk_b),
        "dv": (rv, U8 * np.abs(rv) + dv_b),
    }


def logits_bound(ref, absdot):
    """Whole-model bf16 logits against the fp32/fp64 oracle: output rounding
    plus C_LOGITS * 2^-8 of sum_c |lnf_c wte_vc| (the bf16 weight copy and the
    bf16 activations upstream each move the dot product by at most a few
    2^-8 of that sum)."""
    return U8 * np.abs(ref) + C_LOGITS * U8 * absdot


def loss_bound(ref, pos_scale):
    """Per-position cross-entropy lse - z_target of the bf16 model against the
    oracle: its own output scale plus the logits allowance taken at the
    position's magnitude scale (sum_c |lnf_c wte_vc| at the target plus its
    softmax-weighted mean over the vocabulary, stored with the oracle's
    values)."""
    return U8 * np.abs(ref) + C_LOGITS * U8 * pos_scale
