"""The allocation-free encoder backward against the regular one.

gpt2_op_encoder_backward_noalloc serves callers that cannot allocate device
memory (a host program that owns all of it, or a path that cannot afford
cudaMalloc's synchronisation); its scratch is a library-owned static device
array.  Its results must equal those of gpt2_op_encoder_backward, which takes
caller-provided scratch, exactly (the scatter sums in a fixed order), on two
calls in a row with different shapes and at the array's full size, tokens
outside the table must leave dwte alone, and it must refuse sizes beyond its
array.  This file is collected last so a stop-at-first-failure run has
already run every other test.
"""
import numpy as np
import pytest
import torch

from synthetic import normal_array, zipf_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    import gpt_transformer_train_b300.ops as ops
    return ops


def _both(ops, B, T, C, V, seed):
    tok, _ = zipf_tokens(B, T, V, seed)
    ttok = torch.from_numpy(tok).cuda()
    dres = torch.from_numpy(normal_array((B * T, C), seed + 1)).cuda()
    base_wte = torch.from_numpy(normal_array((V, C), seed + 2)).cuda()
    base_wpe = torch.from_numpy(normal_array((T, C), seed + 3)).cuda()
    ref_wte, ref_wpe = base_wte.clone(), base_wpe.clone()
    ops.gpt2_op_encoder_backward(ref_wte, ref_wpe, dres, ttok, B, T, C)
    na_wte, na_wpe = base_wte.clone(), base_wpe.clone()
    rc = ops.gpt2_op_encoder_backward_noalloc(na_wte, na_wpe, dres, ttok, B, T, C)
    torch.cuda.synchronize()
    assert rc == 0
    return ref_wte, ref_wpe, na_wte, na_wpe


def test_noalloc_encoder_backward_matches_regular_twice(ops):
    # first call: 4 x 1024 positions; second: a smaller ragged batch, so a
    # stale key from the first call would show up as a wrong row
    for (B, T, C, V, seed) in ((4, 1024, 768, 50257, 11), (3, 37, 64, 97, 12)):
        rw, rp, nw, npe = _both(ops, B, T, C, V, seed)
        assert torch.equal(rw, nw)
        assert torch.equal(rp, npe)


@pytest.mark.parametrize("B,T", [(32, 1024), (17, 1000)])
def test_noalloc_full_array_range(ops, B, T):
    """B*T = 32768 fills the whole key array (and needs the sort's largest
    shared-memory size); 17000 is a size just above 16384 that is not a power
    of two, so the padding keys fill the array's tail."""
    rw, rp, nw, npe = _both(ops, B, T, 64, 50257, 13)
    assert torch.equal(rw, nw)
    assert torch.equal(rp, npe)


def test_noalloc_out_of_range_tokens(ops):
    """Tokens -1 and V + 5 add nothing to dwte and raise the token flag.
    dwte is allocated with 65536 rows and only the first V are passed as the
    table, so rows V.. act as a guard band that must stay untouched."""
    B, T, C, V = 2, 100, 64, 500
    tok, _ = zipf_tokens(B, T, V, 21)
    tok[0, 3], tok[1, 50], tok[1, 99] = -1, V + 5, V
    ttok = torch.from_numpy(tok).cuda()
    dres = torch.from_numpy(normal_array((B * T, C), 22)).cuda()
    base = torch.from_numpy(normal_array((65536, C), 23)).cuda()
    dwpe0 = torch.zeros(T, C, device="cuda")
    outs = []
    for fn in (ops.gpt2_op_encoder_backward, ops.gpt2_op_encoder_backward_noalloc):
        w, p, fl = base.clone(), dwpe0.clone(), ops.flags()
        rc = fn(w, p, dres, ttok, B, T, C, V=V, flags_dev=fl)
        torch.cuda.synchronize()
        assert not rc
        assert fl[0].item() & 1
        assert torch.equal(w[V:], base[V:])
        outs.append((w, p))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    # the valid positions' sums against float64; dwpe still takes every position
    good = (tok >= 0) & (tok < V)
    ref = base[:V].double().cpu().numpy().copy()
    d = dres.double().cpu().numpy()
    np.add.at(ref, tok.reshape(-1)[good.reshape(-1)], d[good.reshape(-1)])
    assert np.max(np.abs(outs[0][0][:V].double().cpu().numpy() - ref)) < 1e-4
    assert np.allclose(outs[0][1].double().cpu().numpy(), d.reshape(B, T, C).sum(0), atol=1e-5)


def test_noalloc_rejects_sizes_beyond_its_array(ops):
    dummy = torch.zeros(16, device="cuda")
    tok = torch.zeros(16, dtype=torch.int32, device="cuda")
    # B*T = 32769 > GPT2_NOALLOC_MAX_TOKENS: refused before any launch
    assert ops.gpt2_op_encoder_backward_noalloc(dummy, dummy, dummy, tok, 1, 32769, 4, V=4) == -2
    assert ops.gpt2_op_encoder_backward_noalloc(dummy, dummy, dummy, tok, 1, 4, 6, V=4) == -7
    assert ops.gpt2_op_encoder_backward_noalloc(dummy, dummy, dummy, tok, 1, 4, 4, V=65536) == -7
