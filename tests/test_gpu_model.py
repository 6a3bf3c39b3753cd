"""Whole-step parity: the library's forward, backward and AdamW through the
model C ABI against the oracle on the same seeded tokens and the same seeded
initial weights (bit-equal, see test_abi_host).

fp32 mode (tiny config: L=2 C=64 H=4 T=64 B=4 V=512): loss rel err <= 1e-5,
logits max abs err <= 1e-3, per-tensor grad rel-L2 <= 1e-3, parameters
after AdamW rel-L2 <= 1e-5 over the whole parameter vector (per tensor, the
key slice of qkvb has an analytically zero gradient, so its post-update
value is set by rounding noise on both sides), 5 steps on one fixed batch.
bf16 mode: loss abs err <= 2e-2, per-tensor grad rel-L2 <= 5e-2, 20-step loss
curve within 2% of the oracle's.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from parity import check, logits_bound, loss_bound
from synthetic import zipf_tokens

pytestmark = pytest.mark.gpu
GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
GOLDEN = os.path.join(GOLDEN_DIR, "oracle_124m.npz")
GOLDEN_LOGITS = os.path.join(GOLDEN_DIR, "oracle_124m_logits.npz")


@pytest.fixture(scope="module")
def g():
    from gpt_transformer_train_b300 import build
    build.build()
    import gpt_transformer_train_b300 as mod
    return mod


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _setup(g, L, C, H, V, Vp, maxT, B, T, prec, seed=1234, dtype=np.float64):
    cfg = g.make_config(L, C, H, V, Vp, maxT, B, T, prec)
    m = g.GPT2(cfg, seed)
    ocfg = O.Config(L, C, H, V, Vp, maxT)
    ref = O.GPT2(ocfg, seed, dtype)
    tok, tgt = zipf_tokens(B, T, V, seed)
    ttok = torch.from_numpy(tok).cuda()
    ttgt = torch.from_numpy(tgt).cuda()
    return cfg, m, ref, tok, tgt, ttok, ttgt


TINY = dict(L=2, C=64, H=4, V=512, Vp=512, maxT=64, B=4, T=64)


def test_fp32_tiny_forward_backward_adamw(g):
    cfg, m, ref, tok, tgt, ttok, ttgt = _setup(g, **TINY, prec=0)
    # logits (forward without targets keeps them)
    m.gpt2_forward(ttok)
    ref.forward(tok)
    assert np.max(np.abs(m.gpt2_get_logits() - ref.cache["logits"])) <= 1e-3
    for step in range(1, 6):
        m.gpt2_zero_grad()
        ref.zero_grad()
        loss = m.gpt2_forward(ttok, ttgt)
        rloss = ref.forward(tok, tgt)
        assert abs(loss - rloss) / rloss <= 1e-5, (step, loss, rloss)
        losses = m.gpt2_get_losses()
        assert np.max(np.abs(losses - ref.cache["losses"])) < 1e-4
        m.gpt2_backward()
        ref.backward()
        if step == 1:
            for n in g.TENSORS:
                e = rel_l2(m.gpt2_get_grads(n), ref.grads[n].reshape(-1))
                assert e <= 1e-3, (n, e)
        m.gpt2_adamw_step(1e-3, 0.9, 0.999, 1e-8, 0.0, step)
        ref.adamw_step(1e-3, 0.9, 0.999, 1e-8, 0.0, step)
        mine = np.concatenate([m.gpt2_get_params(n) for n in g.TENSORS])
        theirs = O.flatten(ref.params, ref.cfg)
        assert rel_l2(mine, theirs) <= 1e-5, step


def test_fp32_tiny_with_clipping_and_schedule(g):
    """Gradient-norm clipping (active: max_norm below the norm) and the
    warmup+cosine learning rate over 6 steps against the oracle."""
    cfg, m, ref, tok, tgt, ttok, ttgt = _setup(g, **TINY, prec=0)
    for step in range(6):
        lr = g.lr_schedule(1e-3, 0.1, 2, 6, step)
        assert abs(lr - O.lr_schedule(1e-3, 0.1, 2, 6, step)) <= 1e-6 * lr
        m.gpt2_zero_grad()
        ref.zero_grad()
        m.gpt2_forward(ttok, ttgt)
        ref.forward(tok, tgt)
        m.gpt2_backward()
        ref.backward()
        rnorm = ref.grad_norm()
        max_norm = 0.5 * rnorm if step % 2 == 0 else 2.0 * rnorm  # clip on even steps only
        m.gpt2_clip_grad_norm(max_norm)
        ref.clip_grad_norm(max_norm)
        assert abs(m.gpt2_get_grad_norm() - rnorm) <= 1e-5 * rnorm, step
        m.gpt2_adamw_step(lr, 0.9, 0.999, 1e-8, 0.01, step + 1)
        ref.adamw_step(lr, 0.9, 0.999, 1e-8, 0.01, step + 1)
        mine = np.concatenate([m.gpt2_get_params(n) for n in g.TENSORS])
        assert rel_l2(mine, O.flatten(ref.params, ref.cfg)) <= 1e-5, step
    # without a new clip call the next update does not scale (factor is one-shot)
    m.gpt2_zero_grad()
    ref.zero_grad()
    m.gpt2_forward(ttok, ttgt)
    ref.forward(tok, tgt)
    m.gpt2_backward()
    ref.backward()
    m.gpt2_adamw_step(1e-4, 0.9, 0.999, 1e-8, 0.01, 7)
    ref.adamw_step(1e-4, 0.9, 0.999, 1e-8, 0.01, 7)
    mine = np.concatenate([m.gpt2_get_params(n) for n in g.TENSORS])
    assert rel_l2(mine, O.flatten(ref.params, ref.cfg)) <= 1e-5


def test_fp32_deterministic(g):
    outs = []
    for _ in range(2):
        cfg, m, ref, tok, tgt, ttok, ttgt = _setup(g, **TINY, prec=0)
        m.gpt2_zero_grad()
        m.gpt2_forward(ttok, ttgt)
        m.gpt2_backward()
        outs.append(np.concatenate([m.gpt2_get_grads(n) for n in g.TENSORS]))
        m.close()
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


SMALL_BF16 = dict(L=2, C=128, H=2, V=1000, Vp=1024, maxT=256, B=4, T=256)


def test_bf16_small_forward_backward_and_curve(g):
    cfg, m, ref, tok, tgt, ttok, ttgt = _setup(g, **SMALL_BF16, prec=1, dtype=np.float32)
    curve, rcurve = [], []
    for step in range(1, 21):
        m.gpt2_zero_grad()
        ref.zero_grad()
        loss = m.gpt2_forward(ttok, ttgt)
        rloss = ref.forward(tok, tgt)
        m.gpt2_backward()
        ref.backward()
        if step == 1:
            assert abs(loss - rloss) <= 2e-2
            for n in g.TENSORS:
                e = rel_l2(m.gpt2_get_grads(n), ref.grads[n].reshape(-1))
                assert e <= 5e-2, (n, e)
        m.gpt2_adamw_step(6e-4, 0.9, 0.95, 1e-8, 0.1, step)
        ref.adamw_step(6e-4, 0.9, 0.95, 1e-8, 0.1, step)
        curve.append(loss)
        rcurve.append(rloss)
    curve, rcurve = np.array(curve), np.array(rcurve)
    assert np.all(np.abs(curve - rcurve) / rcurve <= 0.02), (curve, rcurve)
    assert rcurve[-1] < rcurve[0]


WIDE_BF16 = dict(L=3, C=768, H=12, V=1000, Vp=1024, maxT=128, B=2, T=128)


def test_bf16_wide_step_gradients(g):
    """C = 768 with few tokens: the weight gradients of the attention
    projection and qkv go out as one grouped tensor-core launch (their pair
    tiles together fill more than one wave); every gradient against the oracle."""
    cfg, m, ref, tok, tgt, ttok, ttgt = _setup(g, **WIDE_BF16, prec=1, dtype=np.float32)
    m.gpt2_zero_grad()
    ref.zero_grad()
    loss = m.gpt2_forward(ttok, ttgt)
    rloss = ref.forward(tok, tgt)
    m.gpt2_backward()
    ref.backward()
    assert abs(loss - rloss) <= 2e-2
    for n in g.TENSORS:
        e = rel_l2(m.gpt2_get_grads(n), ref.grads[n].reshape(-1))
        assert e <= 5e-2, (n, e)


@pytest.mark.parametrize("shape", ["small", "wide"])
def test_bf16_logits_against_oracle(g, shape):
    """bf16 mode, forward without targets: every logit (pads included) against
    the float64 oracle's, element by element (tests/parity.py logits_bound:
    output rounding plus 4 * 2^-8 of sum_c |lnf_c wte_vc|)."""
    dims = SMALL_BF16 if shape == "small" else WIDE_BF16
    cfg, m, ref, tok, tgt, ttok, ttgt = _setup(g, **dims, prec=1, dtype=np.float64)
    m.gpt2_forward(ttok)
    ref.forward(tok)
    z = m.gpt2_get_logits()
    zr = ref.cache["logits"]
    absdot = np.abs(ref.cache["lnf"]) @ np.abs(ref.params["wte"]).T
    check(z, zr, logits_bound(zr, absdot), "logits")
    assert np.all(z[..., dims["V"]:] == 0)


def test_nan_loss_reported_and_handle_recovers(g):
    """A NaN planted in one weight (gpt2_set_params) makes the forward's loss
    readback return GPT2_ERR_NAN (-6); with the weight restored the same
    handle computes the oracle's loss again."""
    for prec, dims, tol in ((0, TINY, 1e-5), (1, SMALL_BF16, 2e-2)):
        cfg, m, ref, tok, tgt, ttok, ttgt = _setup(g, **dims, prec=prec)
        w = m.gpt2_get_params("fcw")
        bad = w.copy()
        bad[17] = np.nan
        m.gpt2_set_params("fcw", bad)
        with pytest.raises(g.GPT2Error) as e:
            m.gpt2_forward(ttok, ttgt)
        assert e.value.code == -6
        m.gpt2_set_params("fcw", w)
        loss = m.gpt2_forward(ttok, ttgt)
        rloss = ref.forward(tok, tgt)
        assert abs(loss - rloss) <= tol * (rloss if prec == 0 else 1.0)
        m.close()


def test_bf16_step_host_matches_device_calls(g):
    cfg, m, ref, tok, tgt, ttok, ttgt = _setup(g, **SMALL_BF16, prec=1)
    cfg2, m2, _, _, _, _, _ = _setup(g, **SMALL_BF16, prec=1)
    th = torch.from_numpy(tok).pin_memory()
    gh = torch.from_numpy(tgt).pin_memory()
    for step in (1, 2):
        a = m.gpt2_step_host(th, gh, 6e-4, 0.9, 0.95, 1e-8, 0.1, step)
        m2.gpt2_zero_grad()
        b = m2.gpt2_forward(ttok, ttgt)
        m2.gpt2_backward()
        m2.gpt2_adamw_step(6e-4, 0.9, 0.95, 1e-8, 0.1, step)
        assert a == b
    assert np.array_equal(m.gpt2_get_params("fcw"), m2.gpt2_get_params("fcw"))


def test_graph_step_matches_direct_calls(g):
    """gpt2_graph_step (captured forward + backward writing fresh gradients,
    replayed) gives the same gradients as zero_grad + forward + backward, and a
    replay reads the token arrays' current contents."""
    import torch
    L, C, H, V, Vp, maxT, B, T = SMALL_BF16.values()
    stream = torch.cuda.Stream()
    outs = []
    for use_graph in (False, True):
        cfg = g.make_config(L, C, H, V, Vp, maxT, B, T, 1)
        m = g.GPT2(cfg, 1234, stream=stream)
        tok, tgt = zipf_tokens(B, T, V, 1234)
        tok2, tgt2 = zipf_tokens(B, T, V, 99)
        ttok, ttgt = torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda()
        res = []
        for step, (a, b) in enumerate([(tok, tgt), (tok2, tgt2), (tok, tgt)], start=1):
            with torch.cuda.stream(stream):
                ttok.copy_(torch.from_numpy(a))
                ttgt.copy_(torch.from_numpy(b))
            if use_graph:
                m.gpt2_graph_step(ttok, ttgt)
            else:
                m.gpt2_zero_grad()
                m.gpt2_forward(ttok, ttgt, want_loss=False)
                m.gpt2_backward()
            loss = m.gpt2_get_loss()
            res.append((loss, np.concatenate([m.gpt2_get_grads(n) for n in g.TENSORS])))
            m.gpt2_adamw_step(1e-3, 0.9, 0.95, 1e-8, 0.1, step)
        outs.append(res)
        m.close()
    for (la, ga), (lb, gb) in zip(*outs):
        assert la == lb
        # the graph's backward writes fresh gradients (its first writer of each
        # stores instead of adding to a zeroed buffer): the same numbers, bit for
        # bit, except that an exact zero may carry the other sign (x + 0 vs x)
        assert np.array_equal(ga, gb)
        nz = ga != 0
        assert np.array_equal(ga[nz].view(np.uint32), gb[nz].view(np.uint32))
    assert outs[1][0][0] != outs[1][1][0]  # the second batch really was different


@pytest.mark.parametrize("prec", [0, 1])
def test_activation_recompute_modes(g, prec):
    """recompute 1 (GELU) and 2 (also LayerNorm outputs) against recompute 0 on
    the same weights and batch: the same forward bits; gradients within fp32
    summation-order noise of mode 0 (its weight gradients run batched, the
    recompute modes' layer by layer); modes 1 and 2 identical to the bit (the
    recomputed LayerNorm output is the forward's, bit for bit); a smaller buffer
    for each step up; the bf16 step also against the oracle."""
    L, C, H, V, Vp, maxT, B, T = (TINY if prec == 0 else SMALL_BF16).values()
    res = {}
    for rc in (0, 1, 2):
        cfg = g.make_config(L, C, H, V, Vp, maxT, B, T, prec, recompute=rc)
        res.setdefault("bytes", []).append(g.required_bytes(cfg))
        m = g.GPT2(cfg, 1234)
        tok, tgt = zipf_tokens(B, T, V, 1234)
        ttok, ttgt = torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda()
        losses, grads = [], None
        for step in (1, 2):
            m.gpt2_zero_grad()
            losses.append(m.gpt2_forward(ttok, ttgt))
            m.gpt2_backward()
            if step == 1:
                grads = {n: m.gpt2_get_grads(n) for n in g.TENSORS}
            m.gpt2_adamw_step(1e-3, 0.9, 0.95, 1e-8, 0.1, step)
        res[rc] = (losses, grads)
        m.close()
    b0, b1, b2 = res["bytes"]
    assert b2 < b1 < b0
    assert res[0][0][0] == res[1][0][0] == res[2][0][0]  # step-1 forward: same bits
    for n in g.TENSORS:
        assert np.array_equal(res[1][1][n].view(np.uint32), res[2][1][n].view(np.uint32)), n
        assert rel_l2(res[1][1][n], res[0][1][n]) <= 1e-5, n
    assert abs(res[1][0][1] - res[0][0][1]) <= 1e-4 * abs(res[0][0][1])
    if prec == 1:
        ref = O.GPT2(O.Config(L, C, H, V, Vp, maxT), 1234, np.float32)
        tok, tgt = zipf_tokens(B, T, V, 1234)
        rloss = ref.forward(tok, tgt)
        ref.backward()
        assert abs(res[2][0][0] - rloss) <= 2e-2
        for n in g.TENSORS:
            assert rel_l2(res[2][1][n], ref.grads[n].reshape(-1)) <= 5e-2, n


@pytest.mark.parametrize("dims", ["small", "wide"])
def test_ln_fold_step(g, dims):
    """ln_fold (recompute 2): the LayerNorms before the qkv and fc products
    folded into them.  Two steps against the same model without the fold
    (same weights, batch and recompute mode: loss and every gradient within
    bf16 rounding of each other) and the first step against the oracle."""
    d = SMALL_BF16 if dims == "small" else WIDE_BF16
    L, C, H, V, Vp, maxT, B, T = d.values()
    tok, tgt = zipf_tokens(B, T, V, 1234)
    ttok, ttgt = torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda()
    res = {}
    for fold in (0, 1):
        m = g.GPT2(g.make_config(L, C, H, V, Vp, maxT, B, T, 1, recompute=2, ln_fold=fold), 1234)
        out = []
        for step in (1, 2):
            m.gpt2_zero_grad()
            loss = m.gpt2_forward(ttok, ttgt)
            m.gpt2_backward()
            out.append((loss, {n: m.gpt2_get_grads(n) for n in g.TENSORS}))
            m.gpt2_adamw_step(1e-3, 0.9, 0.95, 1e-8, 0.1, step)
        res[fold] = out
        m.close()
    for step in range(2):
        assert abs(res[1][step][0] - res[0][step][0]) <= 2e-2, step
        for n in g.TENSORS:
            assert rel_l2(res[1][step][1][n], res[0][step][1][n]) <= 5e-2, (step, n)
    ref = O.GPT2(O.Config(L, C, H, V, Vp, maxT), 1234, np.float32)
    rloss = ref.forward(tok, tgt)
    ref.backward()
    assert abs(res[1][0][0] - rloss) <= 2e-2
    for n in g.TENSORS:
        assert rel_l2(res[1][0][1][n], ref.grads[n].reshape(-1)) <= 5e-2, n
    with pytest.raises(g.GPT2Error):  # the fold needs recompute 2
        g.GPT2(g.make_config(L, C, H, V, Vp, maxT, B, T, 1, recompute=0, ln_fold=1), 1234)


def test_error_paths_on_device(g):
    cfg, m, ref, tok, tgt, ttok, ttgt = _setup(g, **TINY, prec=0)
    with pytest.raises(g.GPT2Error) as e:
        m.gpt2_backward()
    assert e.value.code == -3
    bad = ttok.clone()
    bad[1, 5] = 512
    with pytest.raises(g.GPT2Error) as e:
        m.gpt2_forward(bad, ttgt)
    assert e.value.code == -4
    badt = ttgt.clone()
    badt[0, 0] = -1
    with pytest.raises(g.GPT2Error) as e:
        m.gpt2_forward(ttok, badt)
    assert e.value.code == -4
    # the handle stays usable after a flagged batch
    loss = m.gpt2_forward(ttok, ttgt)
    assert math.isfinite(loss)
    with pytest.raises(g.GPT2Error) as e:
        m.gpt2_get_logits()
    assert e.value.code == -3


M124 = dict(L=12, C=768, H=12, V=50257, Vp=50304, maxT=1024, B=16, T=1024)
M350 = dict(L=24, C=1024, H=16, V=50257, Vp=50304, maxT=1024, B=8, T=1024)
M1600 = dict(L=48, C=1600, H=25, V=50257, Vp=50304, maxT=1024, B=8, T=1024)


def _check_logit_rows(g, m, ttok, gold):
    """Forward without targets (logits kept); the stored oracle rows, element
    by element, with the oracle's own sum_c |lnf wte| as the magnitude scale."""
    m.gpt2_forward(ttok)
    z = m.gpt2_get_logits()
    for (b, t), zr, absdot in zip(gold["logit_pos"], gold["logit_rows"], gold["logit_bound"]):
        check(z[b, t], zr, logits_bound(zr.astype(np.float64), absdot.astype(np.float64)), f"logits[{b}, {t}]")


def _check_config_against_golden(g, dims, path):
    """One bf16 step of a large config in the bench's launch configuration
    against the oracle's stored values: logits rows, the mean loss, every
    per-position loss, sampled gradient entries and each gradient's norm."""
    gold = np.load(path)
    cfg = g.make_config(*(dims[k] for k in ("L", "C", "H", "V", "Vp", "maxT", "B", "T")), 1)
    m = g.GPT2(cfg, 1234)
    tok, tgt = zipf_tokens(dims["B"], dims["T"], dims["V"], 1234)
    ttok, ttgt = torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda()
    _check_logit_rows(g, m, ttok, gold)
    m.gpt2_zero_grad()
    loss = m.gpt2_forward(ttok, ttgt)
    assert abs(loss - float(gold["loss"])) <= 2e-2
    check(m.gpt2_get_losses().reshape(-1), gold["pos_losses"], loss_bound(gold["pos_losses"], gold["pos_scale"]),
          "per-position loss")
    m.gpt2_backward()
    for n in g.TENSORS:
        gm = m.gpt2_get_grads(n)
        e = rel_l2(gm[gold["grad_idx_" + n]], gold["grad_val_" + n])
        assert e <= 5e-2, (n, e)
        assert abs(np.linalg.norm(gm.astype(np.float64)) / float(gold["grad_norm_" + n]) - 1) <= 5e-2, n
    m.close()


@pytest.mark.skipif(not os.path.exists(os.path.join(GOLDEN_DIR, "oracle_350m.npz")),
                    reason="stored oracle values for 350M not generated")
def test_bf16_350m_against_stored_oracle(g):
    """GPT-2 350M (L=24, C=1024, H=16), B=8, T=1024: the 16-head layout."""
    _check_config_against_golden(g, M350, os.path.join(GOLDEN_DIR, "oracle_350m.npz"))


@pytest.mark.skipif(not os.path.exists(os.path.join(GOLDEN_DIR, "oracle_1p6b.npz")),
                    reason="stored oracle values for 1.6B not generated")
def test_bf16_1p6b_against_stored_oracle(g):
    """GPT-2 1.6B (L=48, C=1600, H=25: a head count that is not a power of
    two), B=8, T=1024, all state in one 61 GB buffer."""
    _check_config_against_golden(g, M1600, os.path.join(GOLDEN_DIR, "oracle_1p6b.npz"))


@pytest.mark.skipif(not os.path.exists(GOLDEN), reason="stored oracle values for 124M not generated")
def test_bf16_124m_against_stored_oracle(g):
    """GPT-2 124M, B=16, T=1024, bf16 — the benchmarked workload — against
    the oracle's stored fp32 run on the same seeded batch and weights."""
    gold = np.load(GOLDEN)
    cfg = g.make_config(*(M124[k] for k in ("L", "C", "H", "V", "Vp", "maxT", "B", "T")), 1)
    m = g.GPT2(cfg, 1234)
    tok, tgt = zipf_tokens(16, 1024, 50257, 1234)
    ttok, ttgt = torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda()
    rl = gold["losses"]
    gl = np.load(GOLDEN_LOGITS) if os.path.exists(GOLDEN_LOGITS) else None
    if gl is not None:
        _check_logit_rows(g, m, ttok, gl)
    for step in range(1, len(rl) + 1):
        m.gpt2_zero_grad()
        loss = m.gpt2_forward(ttok, ttgt)
        if step == 1:
            assert abs(loss - rl[0]) <= 2e-2
            pl = m.gpt2_get_losses().reshape(-1)
            # every position, not just on average (the magnitude scale of each
            # position's loss comes with the stored logit rows)
            if gl is not None:
                check(pl, gold["pos_losses0"], loss_bound(gold["pos_losses0"], gl["pos_scale"]), "per-position loss")
        m.gpt2_backward()
        if step == 1:
            for n in g.TENSORS:
                gm = m.gpt2_get_grads(n)
                idx = gold["grad_idx_" + n]
                e = rel_l2(gm[idx], gold["grad_val_" + n])
                assert e <= 5e-2, (n, e)
                assert abs(np.linalg.norm(gm.astype(np.float64)) / float(gold["grad_norm_" + n]) - 1) <= 5e-2, n
        m.gpt2_adamw_step(6e-4, 0.9, 0.95, 1e-8, 0.1, step)
        assert abs(loss - rl[step - 1]) / rl[step - 1] <= 0.02, (step, loss, rl[step - 1])
