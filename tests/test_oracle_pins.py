"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test ties one oracle function to something independent: a number printed
on the llm.c pages, a closed form, a brute-force loop on a tiny input, a
library routine (torch, scipy) computing the same textbook operation, or
central finite differences.  A planted-mistake test at the end shows that the
finite-difference pin catches a sign error in a backward formula.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import erf

import oracle as O
from synthetic import zipf_tokens

TINY = O.Config(L=2, C=64, H=4, V=512, Vp=512, maxT=64)


# ---------------------------------------------------------------------------
# numbers printed on the pages
# ---------------------------------------------------------------------------
def test_param_count_124M():
    # "llm.c: GPT-2 training in plain C ...", §3 Run it, tested: num_parameters
    assert O.num_parameters(O.GPT2_124M) == 124_475_904


def test_activation_count_124M_B4_T64():
    # same page, §3: num_activations for B=4, T=64
    assert O.num_activations(O.GPT2_124M, 4, 64) == 73_347_840


def test_checkpoint_sizes_match_param_count():
    # same page, §3 starter pack: 1024-byte header + 4 or 2 bytes per parameter
    n = O.num_parameters(O.GPT2_124M)
    assert 1024 + 4 * n == 497_904_640
    assert 1024 + 2 * n == 248_952_832


def test_tiny_param_count():
    assert O.num_parameters(TINY) == 136_960


# ---------------------------------------------------------------------------
# initialisation
# ---------------------------------------------------------------------------
def test_init_statistics_and_structure():
    cfg = O.Config(L=4, C=128, H=2, V=1000, Vp=1024, maxT=128)
    p = O.init_params(cfg, 7)
    assert np.all(p["wte"][cfg.V:] == 0)
    for n in ("ln1w", "ln2w", "lnfw"):
        assert np.all(p[n] == 1)
    for n in ("ln1b", "ln2b", "lnfb", "qkvb", "attprojb", "fcb", "fcprojb"):
        assert np.all(p[n] == 0)
    for n, std in (("qkvw", 0.02), ("fcw", 0.02), ("wpe", 0.02),
                   ("attprojw", 0.02 / math.sqrt(8)), ("fcprojw", 0.02 / math.sqrt(8))):
        a = p[n].astype(np.float64).ravel()
        se = std / math.sqrt(a.size)
        assert abs(a.mean()) < 5 * se, n
        assert abs(a.std() / std - 1) < 5 / math.sqrt(2 * a.size), n
    w = p["wte"][: cfg.V].astype(np.float64).ravel()
    assert abs(w.std() / 0.02 - 1) < 5 / math.sqrt(2 * w.size)
    # the draw is a function of (seed, flat index) only
    assert np.array_equal(O.init_params(cfg, 7)["fcw"], p["fcw"])
    assert not np.array_equal(O.init_params(cfg, 8)["fcw"], p["fcw"])


def test_splitmix64_known_outputs():
    # SplitMix64 started from state 0: the first outputs of Vigna's reference
    # generator (public-domain splitmix64.c) are these three values.
    out = O.splitmix64(0, np.arange(3, dtype=np.uint64))
    assert [int(x) for x in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_box_muller_is_standard_normal():
    z = O.standard_normal_at(99, np.arange(200_000, dtype=np.uint64))
    assert abs(z.mean()) < 5 / math.sqrt(z.size)
    assert abs(z.var() - 1) < 5 * math.sqrt(2 / z.size)
    # tail mass beyond 2 sigma: 4.55% for N(0,1)
    frac = np.mean(np.abs(z) > 2)
    assert abs(frac - 0.0455) < 0.003


# ---------------------------------------------------------------------------
# layer-level closed forms and library routines
# ---------------------------------------------------------------------------
def test_layernorm_closed_form_and_torch():
    rng = np.random.default_rng(0)
    x = rng.normal(0.3, 2.0, size=(5, 7, 96))
    out, mean, rstd = O.layernorm_forward(x, np.ones(96), np.zeros(96))
    var = x.var(axis=-1)
    assert np.allclose(out.mean(axis=-1), 0, atol=1e-12)
    assert np.allclose(out.var(axis=-1), var / (var + 1e-5), rtol=1e-12)
    w, b = rng.normal(size=96), rng.normal(size=96)
    out, _, _ = O.layernorm_forward(x, w, b)
    ref = F.layer_norm(torch.from_numpy(x), (96,), torch.from_numpy(w), torch.from_numpy(b), eps=1e-5)
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_layernorm_backward_vs_torch_autograd():
    rng = np.random.default_rng(1)
    x, w, b, dy = (rng.normal(size=s) for s in ((3, 4, 40), (40,), (40,), (3, 4, 40)))
    out, mean, rstd = O.layernorm_forward(x, w, b)
    dx, dw, db = O.layernorm_backward(dy, x, mean, rstd, w)
    xt, wt, bt = (torch.tensor(a, requires_grad=True) for a in (x, w, b))
    F.layer_norm(xt, (40,), wt, bt, eps=1e-5).backward(torch.from_numpy(dy))
    for a, t in ((dx, xt), (dw, wt), (db, bt)):
        assert np.allclose(a, t.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_gelu_special_values_and_erf_form():
    x = np.array([0.0, 10.0, -10.0, 30.0])
    g = O.gelu_forward(x)
    assert g[0] == 0.0
    assert abs(g[1] - 10.0) < 1e-12 and abs(g[2]) < 1e-12 and g[3] == 30.0
    # the tanh form approximates x * Phi(x) to within 5e-4 everywhere
    xs = np.linspace(-8, 8, 20001)
    exact = 0.5 * xs * (1 + erf(xs / math.sqrt(2)))
    assert np.max(np.abs(O.gelu_forward(xs) - exact)) < 5e-4
    ref = F.gelu(torch.from_numpy(xs), approximate="tanh").numpy()
    assert np.allclose(O.gelu_forward(xs), ref, rtol=1e-12, atol=1e-14)


def test_gelu_backward_finite_difference():
    xs = np.linspace(-6, 6, 1201)
    h = 1e-6
    fd = (O.gelu_forward(xs + h) - O.gelu_forward(xs - h)) / (2 * h)
    an = O.gelu_backward(xs, np.ones_like(xs))
    assert np.max(np.abs(fd - an)) < 1e-8


def _brute_attention(qkv, H):
    """Explicit loops: for each (b, h, t) a masked score list, a softmax over
    t2 <= t written out, and a weighted sum of value rows."""
    B, T, C3 = qkv.shape
    C = C3 // 3
    hd = C // H
    out = np.zeros((B, T, C))
    for b in range(B):
        for h in range(H):
            for t in range(T):
                q = qkv[b, t, h * hd:(h + 1) * hd]
                scores = []
                for t2 in range(t + 1):
                    k = qkv[b, t2, C + h * hd:C + (h + 1) * hd]
                    scores.append(sum(q[i] * k[i] for i in range(hd)) / math.sqrt(hd))
                mx = max(scores)
                ex = [math.exp(s - mx) for s in scores]
                tot = sum(ex)
                for t2 in range(t + 1):
                    v = qkv[b, t2, 2 * C + h * hd:2 * C + (h + 1) * hd]
                    out[b, t, h * hd:(h + 1) * hd] += (ex[t2] / tot) * v
    return out


@pytest.mark.parametrize("T", [1, 5, 8])
def test_attention_forward_brute_force(T):
    rng = np.random.default_rng(T)
    qkv = rng.normal(size=(2, T, 3 * 12))
    out, att = O.attention_forward(qkv, 3)
    assert np.allclose(out, _brute_attention(qkv, 3), rtol=1e-12, atol=1e-13)
    assert np.allclose(att.sum(-1), 1.0)
    assert np.all(att[..., np.triu_indices(T, 1)[0], np.triu_indices(T, 1)[1]] == 0)


def test_attention_matches_torch_sdpa():
    rng = np.random.default_rng(3)
    B, T, H, hd = 2, 16, 4, 8
    qkv = rng.normal(size=(B, T, 3 * H * hd))
    out, _ = O.attention_forward(qkv, H)
    q, k, v = (torch.from_numpy(qkv[..., i * H * hd:(i + 1) * H * hd]).reshape(B, T, H, hd).transpose(1, 2)
               for i in range(3))
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=True).transpose(1, 2).reshape(B, T, H * hd)
    assert np.allclose(out, ref.numpy(), rtol=1e-11, atol=1e-12)


def test_attention_backward_finite_difference():
    rng = np.random.default_rng(4)
    B, T, H = 1, 6, 2
    qkv = rng.normal(size=(B, T, 3 * 8))
    dout = rng.normal(size=(B, T, 8))
    _, att = O.attention_forward(qkv, H)
    an = O.attention_backward(dout, qkv, att, H)
    h = 1e-6
    fd = np.zeros_like(qkv)
    for idx in np.ndindex(qkv.shape):
        qp = qkv.copy(); qp[idx] += h
        qm = qkv.copy(); qm[idx] -= h
        fd[idx] = (np.sum(O.attention_forward(qp, H)[0] * dout) - np.sum(O.attention_forward(qm, H)[0] * dout)) / (2 * h)
    assert np.allclose(an, fd, rtol=1e-6, atol=1e-9)


def test_cross_entropy_vs_torch_and_pad_masking():
    rng = np.random.default_rng(5)
    B, T, V, Vp = 2, 3, 10, 16
    logits = rng.normal(size=(B, T, Vp))
    logits[..., V:] = 50.0           # pads must not enter the softmax
    tgt = rng.integers(0, V, size=(B, T))
    losses = O.crossentropy_forward(logits, tgt, V)
    ref = F.cross_entropy(torch.from_numpy(logits[..., :V]).reshape(-1, V), torch.from_numpy(tgt).reshape(-1),
                          reduction="none").numpy().reshape(B, T)
    assert np.allclose(losses, ref, rtol=1e-12, atol=1e-12)
    probs = O.softmax_forward(logits, V)
    assert np.allclose(probs.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert np.all(probs[..., V:] == 0)


def test_dlogits_is_softmax_minus_onehot_by_finite_difference():
    rng = np.random.default_rng(6)
    B, T, V, Vp = 2, 2, 7, 8
    logits = rng.normal(size=(B, T, Vp))
    tgt = rng.integers(0, V, size=(B, T))
    dloss = np.full((B, T), 1.0 / (B * T))
    an = O.crossentropy_softmax_backward(O.softmax_forward(logits, V), tgt, dloss)
    h = 1e-6
    fd = np.zeros_like(logits)
    for idx in np.ndindex(logits.shape):
        lp = logits.copy(); lp[idx] += h
        lm = logits.copy(); lm[idx] -= h
        fd[idx] = (O.crossentropy_forward(lp, tgt, V).mean() - O.crossentropy_forward(lm, tgt, V).mean()) / (2 * h)
    assert np.allclose(an, fd, rtol=1e-7, atol=1e-10)
    assert np.all(an[..., V:] == 0)


def test_matmul_backward_vs_torch():
    rng = np.random.default_rng(8)
    x, w, b, dy = (rng.normal(size=s) for s in ((3, 5, 6), (4, 6), (4,), (3, 5, 4)))
    dx, dw, db = O.matmul_backward(dy, x, w)
    xt, wt, bt = (torch.tensor(a, requires_grad=True) for a in (x, w, b))
    F.linear(xt, wt, bt).backward(torch.from_numpy(dy))
    for a, t in ((dx, xt), (dw, wt), (db, bt)):
        assert np.allclose(a, t.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_encoder_backward_is_scatter_add():
    rng = np.random.default_rng(9)
    tok = np.array([[3, 1, 3], [0, 3, 1]])
    dout = rng.normal(size=(2, 3, 4))
    dwte, dwpe = O.encoder_backward(dout, tok, 5, 4)
    assert np.allclose(dwte[3], dout[0, 0] + dout[0, 2] + dout[1, 1])
    assert np.allclose(dwte[1], dout[0, 1] + dout[1, 2])
    assert np.all(dwte[[2, 4]] == 0)
    assert np.allclose(dwpe[:3], dout[0] + dout[1]) and np.all(dwpe[3] == 0)


# ---------------------------------------------------------------------------
# AdamW
# ---------------------------------------------------------------------------
def test_adamw_first_step_closed_form():
    rng = np.random.default_rng(10)
    p0, g = rng.normal(size=100), rng.normal(size=100)
    p, m, v = p0.copy(), np.zeros(100), np.zeros(100)
    lr, eps, wd = 1e-3, 1e-8, 0.1
    O.adamw_update(p, g, m, v, lr, 0.9, 0.95, eps, wd, 1)
    assert np.allclose(p - p0, -lr * g / (np.abs(g) + eps) - lr * wd * p0, rtol=1e-10, atol=1e-15)


def test_adamw_matches_torch_optim_over_steps():
    rng = np.random.default_rng(11)
    p0 = rng.normal(size=64)
    grads = [rng.normal(size=64) for _ in range(6)]
    p, m, v = p0.copy(), np.zeros(64), np.zeros(64)
    pt = torch.tensor(p0, requires_grad=True)
    opt = torch.optim.AdamW([pt], lr=6e-4, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)
    for t, g in enumerate(grads, start=1):
        O.adamw_update(p, g, m, v, 6e-4, 0.9, 0.95, 1e-8, 0.1, t)
        pt.grad = torch.from_numpy(g)
        opt.step()
    assert np.allclose(p, pt.detach().numpy(), rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------------------
# gradient-norm clipping and the learning-rate schedule
# ---------------------------------------------------------------------------
def test_grad_norm_and_clip_match_torch_clip_grad_norm():
    """The oracle's global norm and clipping against torch.nn.utils.clip_grad_norm_
    (an independent implementation of the same definition) on the tiny model's
    real gradients, once clipping and once not."""
    for max_norm in (0.05, 1e6):
        m, tok, tgt = _tiny_model()
        m.forward(tok, tgt)
        m.backward()
        ts = [torch.tensor(m.grads[n].copy()) for n in O.PARAM_NAMES]
        ps = [torch.nn.Parameter(torch.zeros_like(t)) for t in ts]
        for p, t in zip(ps, ts):
            p.grad = t
        tnorm = float(torch.nn.utils.clip_grad_norm_(ps, max_norm))
        norm = m.clip_grad_norm(max_norm)
        assert abs(norm - tnorm) <= 1e-12 * tnorm
        for n, p in zip(O.PARAM_NAMES, ps):
            assert np.allclose(m.grads[n], p.grad.numpy(), rtol=1e-12, atol=0), n
        if max_norm < norm:
            assert abs(m.grad_norm() - max_norm) < 1e-6 * max_norm  # clipped to the threshold


def test_grad_norm_brute_force():
    """Every gradient element squared and summed by a plain Python loop."""
    m, tok, tgt = _tiny_model()
    m.forward(tok, tgt)
    m.backward()
    total = 0.0
    for g in m.grads.values():
        for x in np.asarray(g, np.float64).reshape(-1).tolist():
            total += x * x
    assert abs(m.grad_norm() - math.sqrt(total)) < 1e-12 * math.sqrt(total)


def test_lr_schedule_closed_forms():
    lr, frac, W, N = 6e-4, 0.1, 10, 110
    assert abs(O.lr_schedule(lr, frac, W, N, 0) - lr / W) < 1e-18
    assert abs(O.lr_schedule(lr, frac, W, N, W - 1) - lr) < 1e-18          # warmup ends at max_lr
    assert abs(O.lr_schedule(lr, frac, W, N, W) - lr) < 1e-18              # cosine starts at max_lr
    mid = W + (N - W) // 2
    assert abs(O.lr_schedule(lr, frac, W, N, mid) - (lr + frac * lr) / 2) < 1e-15  # halfway
    assert abs(O.lr_schedule(lr, frac, W, N, N) - frac * lr) < 1e-18       # floor
    assert abs(O.lr_schedule(lr, frac, W, N, N + 50) - frac * lr) < 1e-18
    seq = [O.lr_schedule(lr, frac, W, N, s) for s in range(W, N + 1)]
    assert all(a >= b for a, b in zip(seq, seq[1:]))                       # monotone decay


# ---------------------------------------------------------------------------
# whole model
# ---------------------------------------------------------------------------
def _tiny_model(dtype=np.float64, seed=1234):
    tok, tgt = zipf_tokens(4, 64, TINY.V, seed)
    return O.GPT2(TINY, seed, dtype), tok, tgt


def test_zero_logits_give_loss_ln_V():
    m, tok, tgt = _tiny_model()
    m.params["wte"][...] = 0.0
    loss = m.forward(tok, tgt)
    assert abs(loss - math.log(TINY.V)) < 1e-12
    # padded vocabulary: ln V, not ln Vp
    cfg = O.Config(L=1, C=64, H=4, V=500, Vp=512, maxT=64)
    m2 = O.GPT2(cfg, 3, np.float64)
    m2.params["lnfw"][...] = 0.0
    m2.params["lnfb"][...] = 0.0
    t2, g2 = zipf_tokens(2, 8, cfg.V, 3)
    assert abs(m2.forward(t2, g2) - math.log(500)) < 1e-12


def _torch_forward(params, tok, tgt, cfg):
    """The same GPT-2 built from torch's library layers (float64)."""
    P = {n: torch.tensor(a, requires_grad=True) for n, a in params.items()}
    B, T = tok.shape
    C, H, hd = cfg.C, cfg.H, cfg.hd
    x = P["wte"][torch.from_numpy(tok).long()] + P["wpe"][:T]
    for l in range(cfg.L):
        h = F.layer_norm(x, (C,), P["ln1w"][l], P["ln1b"][l], eps=1e-5)
        qkv = F.linear(h, P["qkvw"][l], P["qkvb"][l])
        q, k, v = (t.reshape(B, T, H, hd).transpose(1, 2) for t in qkv.split(C, dim=-1))
        a = F.scaled_dot_product_attention(q, k, v, is_causal=True).transpose(1, 2).reshape(B, T, C)
        x = x + F.linear(a, P["attprojw"][l], P["attprojb"][l])
        h = F.layer_norm(x, (C,), P["ln2w"][l], P["ln2b"][l], eps=1e-5)
        h = F.gelu(F.linear(h, P["fcw"][l], P["fcb"][l]), approximate="tanh")
        x = x + F.linear(h, P["fcprojw"][l], P["fcprojb"][l])
    x = F.layer_norm(x, (C,), P["lnfw"], P["lnfb"], eps=1e-5)
    logits = x @ P["wte"].T
    loss = F.cross_entropy(logits[..., :cfg.V].reshape(-1, cfg.V), torch.from_numpy(tgt).long().reshape(-1))
    loss.backward()
    return loss.item(), logits.detach().numpy(), {n: t.grad.numpy() for n, t in P.items()}


def test_whole_model_vs_torch_library_layers():
    cfg = O.Config(L=2, C=64, H=4, V=500, Vp=512, maxT=64)
    tok, tgt = zipf_tokens(3, 32, cfg.V, 77)
    m = O.GPT2(cfg, 77, np.float64)
    # non-trivial LN affine and biases so every term is exercised
    rng = np.random.default_rng(77)
    for n in ("ln1w", "ln1b", "ln2w", "ln2b", "lnfw", "lnfb", "qkvb", "attprojb", "fcb", "fcprojb"):
        m.params[n] += rng.normal(scale=0.1, size=m.params[n].shape)
    loss = m.forward(tok, tgt)
    m.backward()
    tl, tlogits, tgrads = _torch_forward(m.params, tok, tgt, cfg)
    assert abs(loss - tl) < 1e-12
    assert np.allclose(m.cache["logits"], tlogits, rtol=1e-10, atol=1e-12)
    for n in m.grads:
        assert np.allclose(m.grads[n], tgrads[n], rtol=1e-8, atol=1e-13), n


def _fd_check(m, tok, tgt, names=None, n_large=64, small=256, seed=0, h=1e-5):
    m.zero_grad()
    m.forward(tok, tgt)
    m.backward()
    rng = np.random.default_rng(seed)
    bad = []
    for name in (names or list(m.params)):
        p = m.params[name].reshape(-1)
        g = m.grads[name].reshape(-1).copy()
        idx = np.arange(p.size) if p.size <= small else rng.choice(p.size, n_large, replace=False)
        for i in idx:
            old = p[i]
            p[i] = old + h
            lp = m.forward(tok, tgt)
            p[i] = old - h
            lm = m.forward(tok, tgt)
            p[i] = old
            fd = (lp - lm) / (2 * h)
            if abs(fd - g[i]) > 1e-6 * abs(g[i]) + 2e-10:
                bad.append((name, int(i), fd, g[i]))
    return bad


def test_finite_differences_every_tensor_tiny():
    """Central differences in float64 on every parameter tensor of the tiny
    config (L=2, C=64, H=4, T=64, B=4, V=512): all elements of tensors with
    at most 256 entries, 64 random elements of the others; rel err <= 1e-6."""
    m, tok, tgt = _tiny_model()
    rng = np.random.default_rng(12)
    for n in ("ln1w", "ln1b", "ln2w", "ln2b", "lnfw", "lnfb", "qkvb", "attprojb", "fcb", "fcprojb"):
        m.params[n] += rng.normal(scale=0.1, size=m.params[n].shape)
    bad = _fd_check(m, tok, tgt)
    assert not bad, bad[:10]


def test_float32_oracle_tracks_float64():
    m64, tok, tgt = _tiny_model(np.float64)
    m32, _, _ = _tiny_model(np.float32)
    l64, l32 = m64.forward(tok, tgt), m32.forward(tok, tgt)
    m64.backward(); m32.backward()
    assert abs(l32 - l64) / l64 < 1e-6
    for n in m64.grads:
        a, b = m64.grads[n], m32.grads[n].astype(np.float64)
        assert np.linalg.norm(a - b) <= 1e-4 * np.linalg.norm(a) + 1e-12, n


# ---------------------------------------------------------------------------
# the pins catch planted mistakes
# ---------------------------------------------------------------------------
def test_planted_sign_error_in_gelu_backward_is_caught(monkeypatch):
    import oracle.gpt2 as G
    real = G.gelu_backward
    monkeypatch.setattr(G, "gelu_backward", lambda x, d: real(x, d) - d * 0.01 * np.sign(x))
    cfg = O.Config(L=1, C=64, H=4, V=128, Vp=128, maxT=16)
    tok, tgt = zipf_tokens(2, 16, cfg.V, 5)
    m = O.GPT2(cfg, 5, np.float64)
    assert _fd_check(m, tok, tgt, names=["fcw", "fcb"], n_large=8, small=0)


def test_planted_mask_error_is_caught(monkeypatch):
    import oracle.gpt2 as G
    real_triu = np.triu
    # off-by-one causal mask (t2 < t instead of t2 <= t): the diagonal goes missing
    monkeypatch.setattr(G.np, "triu", lambda a, k=0: real_triu(a, k=0) if k == 1 else real_triu(a, k))
    rng = np.random.default_rng(13)
    qkv = rng.normal(size=(1, 4, 12))
    with np.errstate(invalid="ignore"):
        out, _ = G.attention_forward(qkv, 1)
    monkeypatch.undo()
    assert not np.allclose(out, _brute_attention(qkv, 1), atol=1e-6)


# ---- sampler and generation (the CPU trainer's sampler, no KV cache) --------
def test_sampler_two_token_closed_form():
    """softmax([a, b]) = [1/(1+e^(b-a)), ...]: coins just below / above the
    first probability pick token 0 / 1; the pads beyond V never count."""
    z = np.array([0.3, -0.9, 50.0], np.float64)  # column 2 is a pad (V = 2)
    p0 = 1.0 / (1.0 + math.exp(-0.9 - 0.3))
    assert O.sample_token(z, 2, p0 - 1e-9) == 0
    assert O.sample_token(z, 2, p0 + 1e-9) == 1
    assert O.sample_token(z, 2, 0.0) == 0
    assert O.sample_token(z, 2, 1.0 - 1e-12) == 1


def test_sampler_stratified_coins_match_probabilities():
    """Coins on a uniform grid of n points land on token i exactly
    round-about n * p_i times (each interval of the CDF gets its share)."""
    rng = np.random.default_rng(7)
    V = 13
    z = rng.normal(0, 2.0, V)
    p = np.exp(z - z.max())
    p /= p.sum()
    n = 20000
    counts = np.bincount([O.sample_token(z, V, (k + 0.5) / n) for k in range(n)], minlength=V)
    assert np.all(np.abs(counts - n * p) <= 1.0 + 1e-9)


def test_sampler_temperature():
    """Temperature 0 is argmax with the lowest index on ties; a tiny positive
    temperature picks the maximum for any coin; temperature 2 equals
    temperature 1 on logits halved."""
    z = np.array([1.0, 3.0, 3.0, -2.0])
    assert O.sample_token(z, 4, 0.7, 0.0) == 1
    z2 = np.array([1.0, 3.5, 3.0, -2.0])
    for coin in (0.0, 0.3, 0.999):
        assert O.sample_token(z2, 4, coin, 1e-3) == 1
        assert O.sample_token(z2, 4, coin, 2.0) == O.sample_token(z2 / 2.0, 4, coin, 1.0)


def test_generate_recomputes_the_prefix_each_step():
    """generate() samples from the last position's logits of a full forward
    over the sequence so far: its first logits equal the prompt's last-position
    logits, and each later one equals the full forward over prompt + the
    tokens generated before it (causality: a longer forward leaves earlier
    positions' logits unchanged)."""
    cfg = O.Config(L=2, C=32, H=2, V=61, Vp=64, maxT=16)
    m = O.GPT2(cfg, 5, np.float64)
    prompt = np.random.default_rng(8).integers(0, 61, size=(2, 5)).astype(np.int32)
    coins = np.random.default_rng(9).random((2, 4))
    toks, logs = O.generate(m, prompt, 4, coins)
    full = np.concatenate([prompt, toks], 1)
    m.forward(full)
    for s in range(4):
        assert np.allclose(logs[s], m.cache["logits"][:, 4 + s, :], rtol=0, atol=1e-12)
        for b in range(2):
            assert toks[b, s] == O.sample_token(logs[s][b], 61, coins[b, s])
