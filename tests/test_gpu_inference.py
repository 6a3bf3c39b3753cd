"""Inference with a KV cache (gpt2_infer_prefill / gpt2_infer_step /
gpt2_sample) against the oracle's generation, which reruns the whole forward
for every new token as the pages' CPU sampler does ("llm.c: GPT-2 training in
plain C ...", §6 Reality check).  Every decoded position's logits are compared
with the oracle's full forward over the sequence so far; greedy generation
and the sampler's inverse-CDF choice with given coins are compared token by
token.

Tolerances: fp32 mode, logits max abs error <= 1e-3 (the fp32 logits bound);
bf16 mode, per-step logits rel-L2 <= 3e-2 (bf16 weights and activations, the
grad bound's order).  Where a token choice hinges on a float comparison, the
test only asks for the oracle's choice when its margin exceeds the logits
tolerance.
"""
import numpy as np
import pytest
import torch

import oracle as O
from synthetic import zipf_tokens

pytestmark = pytest.mark.gpu

TINY = dict(L=2, C=64, H=4, V=512, Vp=512, maxT=64, B=4, T=64)
SMALL_BF16 = dict(L=2, C=128, H=2, V=1000, Vp=1024, maxT=256, B=4, T=256)
LONG_BF16 = dict(L=1, C=128, H=2, V=1000, Vp=1024, maxT=1024, B=2, T=1024)


@pytest.fixture(scope="module")
def g():
    from gpt_transformer_train_b300 import build
    build.build()
    import gpt_transformer_train_b300 as mod
    return mod


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _model(g, cfgd, prec):
    L, C, H, V, Vp, maxT, B, T = cfgd.values()
    m = g.GPT2(g.make_config(L, C, H, V, Vp, maxT, B, T, prec), 1234)
    ref = O.GPT2(O.Config(L, C, H, V, Vp, maxT), 1234, np.float64)
    return m, ref


def _check_logits(prec, got, want, V):
    if prec == 0:
        assert np.max(np.abs(got - want)) <= 1e-3
    else:
        assert rel_l2(got[:, :V], want[:, :V]) <= 3e-2
    assert np.all(got[:, V:] == got[:, V:])  # finite


@pytest.mark.parametrize("prec,n", [(0, 1), (0, 10), (1, 100), (1, 128), (1, 600)])
def test_kv_cache_decode_matches_full_forward(g, prec, n):
    """n = 600 (bf16): the decode step's attention over 601-606 cached keys,
    several batches of keys per thread with a ragged last one."""
    cfgd = TINY if prec == 0 else (LONG_BF16 if n > 256 else SMALL_BF16)
    m, ref = _model(g, cfgd, prec)
    B, T, V = cfgd["B"], cfgd["T"], cfgd["V"]
    toks, _ = zipf_tokens(B, T, V, 77)
    m.gpt2_infer_prefill(torch.from_numpy(toks).cuda(), n)
    seq = toks[:, :n]
    ref.forward(seq)
    _check_logits(prec, m.gpt2_get_infer_logits(), ref.cache["logits"][:, -1, :], V)
    nxt_all, _ = zipf_tokens(B, 8, V, 78)
    steps = min(6, T - n)
    for s in range(steps):
        nxt = nxt_all[:, s].copy()
        m.gpt2_infer_step(torch.from_numpy(nxt).cuda(), n + s)
        seq = np.concatenate([seq, nxt[:, None]], 1)
        ref.forward(seq)
        _check_logits(prec, m.gpt2_get_infer_logits(), ref.cache["logits"][:, -1, :], V)
    m.close()


def test_kv_cache_last_position(g):
    """Decoding up to position T-1 (the cache's last row)."""
    m, ref = _model(g, TINY, 0)
    B, T, V = 4, 64, 512
    toks, _ = zipf_tokens(B, T, V, 79)
    m.gpt2_infer_prefill(torch.from_numpy(toks).cuda(), T - 2)
    for pos in (T - 2, T - 1):
        m.gpt2_infer_step(torch.from_numpy(toks[:, pos].copy()).cuda(), pos)
    ref.forward(np.concatenate([toks[:, :T - 2], toks[:, T - 2:T]], 1))
    _check_logits(0, m.gpt2_get_infer_logits(), ref.cache["logits"][:, -1, :], V)
    with pytest.raises(g.GPT2Error):
        m.gpt2_infer_step(torch.from_numpy(toks[:, 0].copy()).cuda(), T)  # past the cache
    m.close()


@pytest.mark.parametrize("temperature", [0.0, 1.0, 0.7])
def test_generation_against_oracle(g, temperature):
    """fp32: prefill, then sample / decode alternately; each step's token is
    the oracle generator's (full forward per token) wherever the oracle's own
    choice has a margin above the logits tolerance, else one of the choices
    within it; the sequence then continues with the library's token."""
    m, ref = _model(g, TINY, 0)
    B, T, V = 4, 64, 512
    n, steps = 7, 6
    toks, _ = zipf_tokens(B, T, V, 80)
    coins = np.random.default_rng(81).random((B, steps)).astype(np.float32)
    m.gpt2_infer_prefill(torch.from_numpy(toks).cuda(), n)
    seq = toks[:, :n]
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    for s in range(steps):
        tc = torch.from_numpy(coins[:, s].copy()).cuda()
        m.gpt2_sample(temperature, tc, out)
        got = out.cpu().numpy()
        ref.forward(seq)
        last = ref.cache["logits"][:, -1, :]
        for b in range(B):
            want = O.sample_token(last[b], V, float(coins[b, s]), temperature)
            if got[b] != want:
                # allowed only where a logits perturbation within tolerance could flip the choice
                z = np.array(last[b][:V], np.float64)
                if temperature == 0:
                    assert z.max() - z[got[b]] <= 2e-3, (s, b)
                else:
                    p = np.exp((z - z.max()) / temperature)
                    cdf = np.cumsum(p / p.sum())
                    edge = np.min(np.abs(cdf - float(coins[b, s])))
                    assert edge <= 1e-3, (s, b, edge)
        seq = np.concatenate([seq, got[:, None]], 1)
        m.gpt2_infer_step(out, n + s)
    m.close()


@pytest.mark.parametrize("prec", [0, 1])
def test_sampler_on_library_logits(g, prec):
    """gpt2_sample against the oracle's sampler on the library's own last
    logits (as returned), with coins at the midpoint of a chosen token's CDF
    interval and at 0: exact token agreement."""
    cfgd = TINY if prec == 0 else SMALL_BF16
    m, _ = _model(g, cfgd, prec)
    B, T, V = cfgd["B"], cfgd["T"], cfgd["V"]
    toks, _ = zipf_tokens(B, T, V, 82)
    m.gpt2_infer_prefill(torch.from_numpy(toks).cuda(), 5)
    logits = m.gpt2_get_infer_logits()
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    for temperature in (1.0, 0.5, 2.0):
        for pick in (0, 1):
            coins = np.zeros(B, np.float32)
            for b in range(B):
                z = logits[b, :V].astype(np.float64) / temperature
                p = np.exp(z - z.max())
                p /= p.sum()
                cdf = np.cumsum(p)
                k = int(np.argmax(p)) if pick == 0 else int(np.argsort(p)[-2])
                lo = cdf[k - 1] if k > 0 else 0.0
                coins[b] = np.float32((lo + cdf[k]) / 2)
            m.gpt2_sample(temperature, torch.from_numpy(coins).cuda(), out)
            got = out.cpu().numpy()
            for b in range(B):
                assert got[b] == O.sample_token(logits[b], V, float(coins[b]), temperature), (temperature, b)
    m.gpt2_sample(0.0, None, out)
    assert np.array_equal(out.cpu().numpy(), np.argmax(logits[:, :V], 1))
    m.close()


def test_inference_call_order(g):
    m, _ = _model(g, TINY, 0)
    t1 = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(g.GPT2Error) as e:
        m.gpt2_infer_step(t1, 0)
    assert e.value.code == -3
    toks, _ = zipf_tokens(4, 64, 512, 83)
    m.gpt2_infer_prefill(torch.from_numpy(toks).cuda(), 8)
    with pytest.raises(g.GPT2Error) as e:
        m.gpt2_infer_step(t1, 9)  # must append at position 8
    assert e.value.code == -7
    m.close()
