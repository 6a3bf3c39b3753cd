"""Plain CPU oracle of one GPT-2 training step: forward, hand-derived backward, AdamW.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the test suite, the smoke check in the graft entry
module and bench.py's CPU-baseline leg use it.  It shares no code with the
CUDA library.

What it follows (page titles, then section):
  * "llm.c: GPT-2 training in plain C, with every gradient written by hand"
    (fernfant course page), §2 "How the code works": the layer list of one
    block (layernorm, qkv matmul, attention, attention projection, residual,
    layernorm, fc matmul, GELU, fc projection, residual), the forward saving
    `att` and LayerNorm mean/rstd for the backward, the causal loop t2 <= t,
    and the rule that every forward line `out += a * b` becomes two gradient
    lines (datt += v * dout, dv += att * dout).
  * same page, §3 "Run it, tested": the GPT-2 124M shape (max_seq_len 1024,
    vocab 50257 padded to 50304, 12 layers, 12 heads, 768 channels,
    124,475,904 parameters) and the activation count 73,347,840 at B=4, T=64.
  * "llm.c's Origin and the Future of LLM Compilers" (CUDA MODE talk),
    [3:47] "Pure C": plain float arrays, one pre-planned allocation, a forward
    and a pen-and-paper backward per layer, then the update.
  * The AdamW update and the model step list follow the pages' description of
    gpt2_forward -> gpt2_backward -> gpt2_update.

Readings where the pages are silent (each also listed in the design notes):
  LayerNorm eps 1e-5 with biased variance; GELU in its tanh form; attention
  scale 1/sqrt(hd); qkv columns laid out [Q | K | V] with head h owning
  columns h*hd:(h+1)*hd of each; loss = mean cross-entropy over all B*T
  positions; logits are computed over the padded vocabulary Vp but the
  softmax runs over the first V columns only (pad columns get probability 0
  and gradient 0); weight decay applies to 2-D tensors only; the initial
  weights are N(0, 0.02) (projections into the residual stream scaled by
  1/sqrt(2L)), drawn with a counter-based SplitMix64 stream and Box-Muller.

Every array here is a numpy array of the oracle's dtype (float32 like the
pages' CPU trainer, or float64 for finite-difference pins).  Matmuls go to
numpy's BLAS; there is no blocking, fusion or reordering beyond the
definitions below.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

LN_EPS = 1e-5
GELU_SCALE = math.sqrt(2.0 / math.pi)
GELU_CUBIC = 0.044715

PARAM_NAMES = ("wte", "wpe", "ln1w", "ln1b", "qkvw", "qkvb", "attprojw", "attprojb",
               "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb", "lnfw", "lnfb")
# tensors that receive weight decay (the 2-D matrices)
DECAYED = frozenset({"wte", "wpe", "qkvw", "attprojw", "fcw", "fcprojw"})


@dataclass(frozen=True)
class Config:
    L: int
    C: int
    H: int
    V: int
    Vp: int
    maxT: int

    @property
    def hd(self) -> int:
        return self.C // self.H


GPT2_124M = Config(L=12, C=768, H=12, V=50257, Vp=50304, maxT=1024)


def param_shapes(cfg: Config):
    """Canonical parameter order and shapes, weights stored [out][in]."""
    L, C = cfg.L, cfg.C
    return [
        ("wte", (cfg.Vp, C)), ("wpe", (cfg.maxT, C)),
        ("ln1w", (L, C)), ("ln1b", (L, C)),
        ("qkvw", (L, 3 * C, C)), ("qkvb", (L, 3 * C)),
        ("attprojw", (L, C, C)), ("attprojb", (L, C)),
        ("ln2w", (L, C)), ("ln2b", (L, C)),
        ("fcw", (L, 4 * C, C)), ("fcb", (L, 4 * C)),
        ("fcprojw", (L, C, 4 * C)), ("fcprojb", (L, C)),
        ("lnfw", (C,)), ("lnfb", (C,)),
    ]


def num_parameters(cfg: Config) -> int:
    return sum(int(np.prod(s)) for _, s in param_shapes(cfg))


def num_activations(cfg: Config, B: int, T: int) -> int:
    """Float count of the CPU trainer's forward activation list.

    The list (encoded, ln1, ln1 mean/rstd, qkv, atty, preatt, att, attproj,
    residual2, ln2, ln2 mean/rstd, fch, fch_gelu, fcproj, residual3, lnf,
    lnf mean/rstd, logits, probs, losses) is the one the course page's §2 says
    the forward keeps; its §3 prints the total for GPT-2 124M at B=4, T=64.
    Logits and probs span the padded vocabulary.
    """
    L, C, H, Vp = cfg.L, cfg.C, cfg.H, cfg.Vp
    BT = B * T
    sizes = [
        BT * C,                 # encoded
        L * BT * C,             # ln1
        L * BT, L * BT,         # ln1 mean, rstd
        L * BT * 3 * C,         # qkv
        L * BT * C,             # atty
        L * B * H * T * T,      # preatt
        L * B * H * T * T,      # att
        L * BT * C,             # attproj
        L * BT * C,             # residual2
        L * BT * C,             # ln2
        L * BT, L * BT,         # ln2 mean, rstd
        L * BT * 4 * C,         # fch
        L * BT * 4 * C,         # fch_gelu
        L * BT * C,             # fcproj
        L * BT * C,             # residual3
        BT * C,                 # lnf
        BT, BT,                 # lnf mean, rstd
        BT * Vp,                # logits
        BT * Vp,                # probs
        BT,                     # losses
    ]
    return int(sum(sizes))


# ----------------------------------------------------------------------------
# seeded initialisation: SplitMix64 as a counter-based stream + Box-Muller
# ----------------------------------------------------------------------------
_GAMMA = 0x9E3779B97F4A7C15
_M64 = (1 << 64) - 1


def splitmix64(seed: int, counters: np.ndarray) -> np.ndarray:
    """Output number `counter` of SplitMix64 started at state `seed`.

    SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014; Vigna's public-domain reference): the state
    advances by the golden-ratio increment and each output is the state passed
    through the variant-13 finaliser.  Output j uses state seed + (j+1)*gamma,
    so any element can be drawn on its own.
    """
    with np.errstate(over="ignore"):
        z = np.uint64(seed & _M64) + (counters.astype(np.uint64) + np.uint64(1)) * np.uint64(_GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return z


def standard_normal_at(seed: int, flat_index: np.ndarray) -> np.ndarray:
    """float64 N(0,1) for element `i` from outputs 2i and 2i+1 (Box-Muller).

    u1 = (x>>11 + 1) * 2^-53 lies in (0, 1], u2 = (y>>11) * 2^-53 in [0, 1);
    z = sqrt(-2 ln u1) * cos(2 pi u2).  The logarithm and cosine are the C
    library's (Python's math module), element by element, so a C program that
    calls the same libm gets the same doubles.
    """
    i = flat_index.astype(np.uint64)
    x = splitmix64(seed, np.uint64(2) * i)
    y = splitmix64(seed, np.uint64(2) * i + np.uint64(1))
    u1 = ((x >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (y >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    two_pi = 2.0 * math.pi
    lg = np.fromiter(map(math.log, u1.tolist()), dtype=np.float64, count=u1.size)
    cs = np.fromiter(map(math.cos, (two_pi * u2).tolist()), dtype=np.float64, count=u2.size)
    return np.sqrt(-2.0 * lg) * cs


def init_params(cfg: Config, seed: int, dtype=np.float32) -> dict:
    """GPT-2 initial weights from `seed`, element i of the canonical flat
    vector drawn from generator outputs 2i, 2i+1.

    wte rows < V, wpe, qkvw, fcw: N(0, 0.02); attprojw, fcprojw:
    N(0, 0.02/sqrt(2L)); wte pad rows (>= V): 0; LayerNorm gains 1; all
    biases and LayerNorm shifts 0.  Each value is z*std in float64, rounded
    once to float32.
    """
    std = 0.02
    std_proj = 0.02 / math.sqrt(2.0 * cfg.L)
    params = {}
    off = 0

    def normal_block(first, count, s):
        # elements first .. first+count-1 of the stream, scaled and rounded,
        # drawn a block at a time (each element depends only on its index)
        a = np.empty(count, dtype=np.float32)
        step = 1 << 22
        for b in range(0, count, step):
            e = min(count, b + step)
            z = standard_normal_at(seed, np.arange(first + b, first + e, dtype=np.uint64))
            a[b:e] = (z * s).astype(np.float32)
        return a

    for name, shape in param_shapes(cfg):
        n = int(np.prod(shape))
        if name in ("wte", "wpe", "qkvw", "fcw", "attprojw", "fcprojw"):
            s = std_proj if name in ("attprojw", "fcprojw") else std
            if name == "wte":
                nd = cfg.V * cfg.C
                a = np.zeros(n, dtype=np.float32)
                a[:nd] = normal_block(off, nd, s)
            else:
                a = normal_block(off, n, s)
        elif name in ("ln1w", "ln2w", "lnfw"):
            a = np.ones(n, dtype=np.float32)
        else:
            a = np.zeros(n, dtype=np.float32)
        params[name] = a.reshape(shape).astype(dtype)
        off += n
    return params


def flatten(params: dict, cfg: Config) -> np.ndarray:
    return np.concatenate([params[n].reshape(-1) for n, _ in param_shapes(cfg)])


def unflatten(flat: np.ndarray, cfg: Config) -> dict:
    out, off = {}, 0
    for n, s in param_shapes(cfg):
        k = int(np.prod(s))
        out[n] = flat[off:off + k].reshape(s)
        off += k
    return out


# ----------------------------------------------------------------------------
# layers: forward and backward, one pair per layer (course page §2)
# ----------------------------------------------------------------------------
def encoder_forward(wte, wpe, tokens):
    """out[b,t,:] = wte[tokens[b,t]] + wpe[t]."""
    B, T = tokens.shape
    return wte[tokens] + wpe[:T][None, :, :]


def encoder_backward(dout, tokens, Vp, maxT):
    """dwte[v] = sum of dout rows whose token is v; dwpe[t] = sum over b."""
    B, T, C = dout.shape
    dwte = np.zeros((Vp, C), dtype=dout.dtype)
    np.add.at(dwte, tokens.reshape(-1), dout.reshape(-1, C))
    dwpe = np.zeros((maxT, C), dtype=dout.dtype)
    dwpe[:T] = dout.sum(axis=0)
    return dwte, dwpe


def layernorm_forward(x, w, b, eps=LN_EPS):
    """Per row over the last axis: mean, rstd = 1/sqrt(var + eps) with the
    biased variance, out = (x - mean) * rstd * w + b."""
    mean = x.mean(axis=-1, keepdims=True)
    xc = x - mean
    var = (xc * xc).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + x.dtype.type(eps))
    norm = xc * rstd
    out = norm * w + b
    return out, mean[..., 0], rstd[..., 0]


def layernorm_backward(dout, x, mean, rstd, w):
    """Pen-and-paper LayerNorm backward.

    With norm = (x-mean)*rstd and dnorm = dout*w:
      dx = rstd * (dnorm - mean(dnorm) - norm * mean(dnorm*norm)),
      dw = sum over rows of dout*norm, db = sum over rows of dout.
    """
    C = x.shape[-1]
    norm = (x - mean[..., None]) * rstd[..., None]
    dnorm = dout * w
    dnorm_mean = dnorm.mean(axis=-1, keepdims=True)
    dnorm_norm_mean = (dnorm * norm).mean(axis=-1, keepdims=True)
    dx = (dnorm - dnorm_mean - norm * dnorm_norm_mean) * rstd[..., None]
    rows = dout.reshape(-1, C)
    dw = (rows * norm.reshape(-1, C)).sum(axis=0)
    db = rows.sum(axis=0)
    return dx, dw, db


def matmul_forward(x, w, b=None):
    """out = x @ w^T (+ b), weights stored [out_features][in_features]."""
    out = x @ w.T
    if b is not None:
        out = out + b
    return out


def matmul_backward(dout, x, w, with_bias=True):
    """dx = dout @ w; dw = dout^T @ x; db = sum over rows of dout."""
    OC = w.shape[0]
    IC = w.shape[1]
    d2 = dout.reshape(-1, OC)
    x2 = x.reshape(-1, IC)
    dx = (d2 @ w).reshape(x.shape)
    dw = d2.T @ x2
    db = d2.sum(axis=0) if with_bias else None
    return dx, dw, db


def _split_heads(qkv, H):
    B, T, C3 = qkv.shape
    C = C3 // 3
    hd = C // H
    q = qkv[..., 0 * C:1 * C].reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    k = qkv[..., 1 * C:2 * C].reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    v = qkv[..., 2 * C:3 * C].reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    return q, k, v


def attention_forward(qkv, H):
    """Causal multi-head attention.

    For query t and key t2 <= t: preatt = q.k * 1/sqrt(hd); att = softmax over
    t2 <= t (max-subtracted); out[t] = sum_t2 att[t2] v[t2].  Heads are
    concatenated back to [B, T, C].  Returns (out, att) with att [B,H,T,T],
    zero above the diagonal.
    """
    B, T, C3 = qkv.shape
    C = C3 // 3
    hd = C // H
    q, k, v = _split_heads(qkv, H)
    scale = qkv.dtype.type(1.0 / math.sqrt(hd))
    preatt = (q @ k.transpose(0, 1, 3, 2)) * scale
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)      # True where t2 > t
    preatt[..., mask] = -np.inf
    m = preatt.max(axis=-1, keepdims=True)
    e = np.exp(preatt - m)
    att = e / e.sum(axis=-1, keepdims=True)
    del preatt, e
    out = (att @ v).transpose(0, 2, 1, 3).reshape(B, T, C)
    return out, att


def attention_backward(dout, qkv, att, H):
    """Reverse of attention_forward, line by line.

    out += att*v gives datt = dout.v and dv += att*dout; the softmax gives
    dpreatt = att * (datt - sum_t2 att*datt); preatt = q.k*scale gives
    dq += dpreatt*k*scale and dk += dpreatt*q*scale.
    """
    B, T, C3 = qkv.shape
    C = C3 // 3
    hd = C // H
    q, k, v = _split_heads(qkv, H)
    scale = qkv.dtype.type(1.0 / math.sqrt(hd))
    do = dout.reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    datt = do @ v.transpose(0, 1, 3, 2)
    dv = att.transpose(0, 1, 3, 2) @ do
    dpre = att * (datt - (att * datt).sum(axis=-1, keepdims=True))
    del datt
    dq = (dpre @ k) * scale
    dk = (dpre.transpose(0, 1, 3, 2) @ q) * scale
    dqkv = np.empty_like(qkv)
    dqkv[..., 0 * C:1 * C] = dq.transpose(0, 2, 1, 3).reshape(B, T, C)
    dqkv[..., 1 * C:2 * C] = dk.transpose(0, 2, 1, 3).reshape(B, T, C)
    dqkv[..., 2 * C:3 * C] = dv.transpose(0, 2, 1, 3).reshape(B, T, C)
    return dqkv


def gelu_forward(x):
    """tanh-form GELU: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    t = x.dtype.type
    u = t(GELU_SCALE) * (x + t(GELU_CUBIC) * x * x * x)
    return t(0.5) * x * (t(1.0) + np.tanh(u))


def gelu_backward(x, dout):
    """d/dx of the tanh-form GELU times dout."""
    t = x.dtype.type
    u = t(GELU_SCALE) * (x + t(GELU_CUBIC) * x * x * x)
    th = np.tanh(u)
    du = t(GELU_SCALE) * (t(1.0) + t(3.0 * GELU_CUBIC) * x * x)
    return dout * (t(0.5) * (t(1.0) + th) + t(0.5) * x * (t(1.0) - th * th) * du)


def softmax_forward(logits, V):
    """Max-subtracted softmax over the first V columns; pad columns get 0."""
    z = logits[..., :V]
    m = z.max(axis=-1, keepdims=True)
    probs = np.zeros_like(logits)
    e = probs[..., :V]
    np.subtract(z, m, out=e)
    np.exp(e, out=e)
    e /= e.sum(axis=-1, keepdims=True)
    return probs


def crossentropy_forward(logits, targets, V):
    """losses[b,t] = -log softmax(logits[b,t,:V])[target] (log-sum-exp form)."""
    z = logits[..., :V]
    m = z.max(axis=-1, keepdims=True)
    lse = m[..., 0] + np.log(np.exp(z - m).sum(axis=-1))
    zt = np.take_along_axis(z, targets[..., None].astype(np.int64), axis=-1)[..., 0]
    return lse - zt


def crossentropy_softmax_backward(probs, targets, dloss):
    """dlogits = (probs - onehot(target)) * dloss per position; pads stay 0."""
    d = probs.copy()
    B, T = targets.shape
    bi, ti = np.meshgrid(np.arange(B), np.arange(T), indexing="ij")
    d[bi, ti, targets] -= 1.0
    d *= dloss[..., None]
    return d


# ----------------------------------------------------------------------------
# the model: forward, backward, update
# ----------------------------------------------------------------------------
class GPT2:
    """One model instance: parameters, grads, AdamW moments, saved activations."""

    def __init__(self, cfg: Config, seed: int = 1234, dtype=np.float64, params: dict | None = None):
        self.cfg = cfg
        self.dtype = np.dtype(dtype)
        src = params if params is not None else init_params(cfg, seed, np.float32)
        self.params = {n: np.array(src[n], dtype=self.dtype) for n, _ in param_shapes(cfg)}
        self.grads = {n: np.zeros_like(p) for n, p in self.params.items()}
        self.m = {n: np.zeros_like(p) for n, p in self.params.items()}
        self.v = {n: np.zeros_like(p) for n, p in self.params.items()}
        self.cache = None

    # -- forward ---------------------------------------------------------
    def forward(self, tokens, targets=None):
        """gpt2_forward: encoder, L blocks, final LayerNorm, tied classifier,
        softmax + cross-entropy.  Returns the mean loss (or None)."""
        cfg, p = self.cfg, self.params
        B, T = tokens.shape
        if T > cfg.maxT:
            raise ValueError("T exceeds maxT")
        if tokens.min() < 0 or tokens.max() >= cfg.V:
            raise ValueError("token out of range")
        x = encoder_forward(p["wte"], p["wpe"], tokens)
        layers = []
        residual = x
        for l in range(cfg.L):
            c = {"residual": residual}
            c["ln1"], c["ln1_mean"], c["ln1_rstd"] = layernorm_forward(residual, p["ln1w"][l], p["ln1b"][l])
            c["qkv"] = matmul_forward(c["ln1"], p["qkvw"][l], p["qkvb"][l])
            c["atty"], c["att"] = attention_forward(c["qkv"], cfg.H)
            attproj = matmul_forward(c["atty"], p["attprojw"][l], p["attprojb"][l])
            c["residual2"] = residual + attproj
            c["ln2"], c["ln2_mean"], c["ln2_rstd"] = layernorm_forward(c["residual2"], p["ln2w"][l], p["ln2b"][l])
            c["fch"] = matmul_forward(c["ln2"], p["fcw"][l], p["fcb"][l])
            c["fch_gelu"] = gelu_forward(c["fch"])
            fcproj = matmul_forward(c["fch_gelu"], p["fcprojw"][l], p["fcprojb"][l])
            residual = c["residual2"] + fcproj
            layers.append(c)
        lnf, lnf_mean, lnf_rstd = layernorm_forward(residual, p["lnfw"], p["lnfb"])
        logits = matmul_forward(lnf, p["wte"])
        self.cache = {"tokens": tokens, "targets": targets, "layers": layers, "residualf": residual,
                      "lnf": lnf, "lnf_mean": lnf_mean, "lnf_rstd": lnf_rstd, "logits": logits}
        if targets is None:
            return None
        if targets.min() < 0 or targets.max() >= cfg.V:
            raise ValueError("target out of range")
        self.cache["losses"] = crossentropy_forward(logits, targets, cfg.V)
        return float(self.cache["losses"].mean())

    # -- backward --------------------------------------------------------
    def backward(self):
        """gpt2_backward: the forward read in reverse; grads accumulate (+=)."""
        cfg, p, g, c = self.cfg, self.params, self.grads, self.cache
        if c is None or c.get("targets") is None:
            raise RuntimeError("backward needs a forward with targets")
        tokens, targets = c["tokens"], c["targets"]
        B, T = tokens.shape
        dloss = np.full((B, T), 1.0 / (B * T), dtype=self.dtype)
        probs = softmax_forward(c["logits"], cfg.V)
        dlogits = crossentropy_softmax_backward(probs, targets, dloss)
        del probs
        dlnf, dwte, _ = matmul_backward(dlogits, c["lnf"], p["wte"], with_bias=False)
        g["wte"] += dwte
        del dlogits
        dres, dw, db = layernorm_backward(dlnf, c["residualf"], c["lnf_mean"], c["lnf_rstd"], p["lnfw"])
        g["lnfw"] += dw
        g["lnfb"] += db
        for l in reversed(range(cfg.L)):
            cl = c["layers"][l]
            # residual3 = residual2 + fcproj
            dfch_gelu, dw, db = matmul_backward(dres, cl["fch_gelu"], p["fcprojw"][l])
            g["fcprojw"][l] += dw
            g["fcprojb"][l] += db
            dfch = gelu_backward(cl["fch"], dfch_gelu)
            dln2, dw, db = matmul_backward(dfch, cl["ln2"], p["fcw"][l])
            g["fcw"][l] += dw
            g["fcb"][l] += db
            dx, dw, db = layernorm_backward(dln2, cl["residual2"], cl["ln2_mean"], cl["ln2_rstd"], p["ln2w"][l])
            g["ln2w"][l] += dw
            g["ln2b"][l] += db
            dres = dres + dx                       # grad of residual2
            # residual2 = residual + attproj
            datty, dw, db = matmul_backward(dres, cl["atty"], p["attprojw"][l])
            g["attprojw"][l] += dw
            g["attprojb"][l] += db
            dqkv = attention_backward(datty, cl["qkv"], cl["att"], cfg.H)
            dln1, dw, db = matmul_backward(dqkv, cl["ln1"], p["qkvw"][l])
            g["qkvw"][l] += dw
            g["qkvb"][l] += db
            dx, dw, db = layernorm_backward(dln1, cl["residual"], cl["ln1_mean"], cl["ln1_rstd"], p["ln1w"][l])
            g["ln1w"][l] += dw
            g["ln1b"][l] += db
            dres = dres + dx                       # grad of this block's input
        dwte, dwpe = encoder_backward(dres, tokens, cfg.Vp, cfg.maxT)
        g["wte"] += dwte
        g["wpe"] += dwpe
        self.cache["dresidual0"] = dres

    def zero_grad(self):
        for a in self.grads.values():
            a[...] = 0

    # -- update ----------------------------------------------------------
    def adamw_step(self, lr, b1, b2, eps, wd, t):
        """gpt2_update (AdamW, decoupled decay), t is 1-based:
        m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2;
        mhat = m/(1-b1^t); vhat = v/(1-b2^t);
        p -= lr * (mhat/(sqrt(vhat)+eps) + wd_i p), wd_i = wd on 2-D tensors."""
        for n, _ in param_shapes(self.cfg):
            adamw_update(self.params[n], self.grads[n], self.m[n], self.v[n],
                         lr, b1, b2, eps, wd if n in DECAYED else 0.0, t)

    def grad_norm(self):
        """Global L2 norm of all parameter gradients, sqrt(sum over every
        tensor of sum g^2), accumulated in float64 (the pages' global_norm
        component, "llm.c" tour, detail graph: a cross-tensor gradient norm)."""
        return float(np.sqrt(sum(float(np.sum(np.asarray(g, np.float64) ** 2)) for g in self.grads.values())))

    def clip_grad_norm(self, max_norm):
        """Scale every gradient by min(1, max_norm / (norm + 1e-6)) and return
        the norm before clipping.  The pages name gradient-norm clipping
        without a formula; this is the plainest reading (the 1e-6 guards a
        zero norm)."""
        norm = self.grad_norm()
        coef = max_norm / (norm + 1e-6)
        if coef < 1.0:
            for g in self.grads.values():
                g *= g.dtype.type(coef)
        return norm


def sample_token(logits_row, V, coin, temperature=1.0):
    """The CPU trainer's sampler ("llm.c: GPT-2 training in plain C ...", §2
    How the code works: the file ends with a sampler; §6 Reality check: it
    keeps no KV cache, every new token runs the whole forward again): the
    probabilities are the softmax of the first V logits (divided by the
    temperature), and the token is the first index whose cumulative
    probability exceeds the coin, a uniform number in [0, 1); the last index
    when rounding leaves the total below the coin.  Temperature 0 (our
    addition): the index of the largest logit, the lowest such index on ties.
    Computed in float64."""
    z = np.asarray(logits_row[:V], np.float64)
    if temperature == 0:
        return int(np.argmax(z))
    z = z / temperature
    p = np.exp(z - z.max())
    p /= p.sum()
    cdf = 0.0
    for i in range(V):
        cdf += p[i]
        if coin < cdf:
            return i
    return V - 1


def generate(model, prompt, steps, coins, temperature=1.0):
    """Tokens after `prompt` ([B][n]), the CPU trainer's way: for each new
    token the whole forward runs over the sequence so far and the last
    position's logits are sampled with coins[b][s] (see sample_token).
    Returns (tokens [B][steps], logits [steps][B][Vp] of the sampled positions)."""
    seq = np.array(prompt, np.int32)
    B = seq.shape[0]
    out, logs = [], []
    for s in range(steps):
        model.forward(seq)
        last = model.cache["logits"][:, -1, :]
        nxt = np.array([sample_token(last[b], model.cfg.V, coins[b][s], temperature) for b in range(B)], np.int32)
        out.append(nxt)
        logs.append(np.array(last))
        seq = np.concatenate([seq, nxt[:, None]], axis=1)
    return np.stack(out, 1), np.stack(logs, 0)


def lr_schedule(max_lr, final_frac, warmup, total, step):
    """Learning rate at 0-based `step`: linear warmup to max_lr over `warmup`
    steps (step s gets max_lr (s + 1) / warmup), then cosine decay from max_lr
    to min_lr = final_frac * max_lr at step `total`, min_lr after that.  The
    pages list LR warmup and decay schedulers without formulas (the "llm.c"
    tour, detail graph); this is the plainest reading of "warmup then decay"."""
    if step < warmup:
        return max_lr * (step + 1) / warmup
    min_lr = final_frac * max_lr
    if step >= total:
        return min_lr
    ratio = (step - warmup) / (total - warmup)
    return min_lr + 0.5 * (1.0 + math.cos(math.pi * ratio)) * (max_lr - min_lr)


def adamw_update(p, g, m, v, lr, b1, b2, eps, wd, t):
    """One AdamW update of p, m, v in place (see GPT2.adamw_step)."""
    ty = p.dtype.type
    m[...] = ty(b1) * m + ty(1.0 - b1) * g
    v[...] = ty(b2) * v + ty(1.0 - b2) * g * g
    mhat = m / ty(1.0 - b1 ** t)
    vhat = v / ty(1.0 - b2 ** t)
    p -= ty(lr) * (mhat / (np.sqrt(vhat) + ty(eps)) + ty(wd) * p)
