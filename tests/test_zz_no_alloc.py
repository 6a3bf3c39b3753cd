"""The allocation-free encoder backward against the regular one.

gpt2_op_encoder_backward_noalloc serves callers that cannot allocate device
memory (a host program that owns all of it, or a path that cannot afford
cudaMalloc's synchronisation); its scratch is a library-owned static device
array.  Its results must equal those of gpt2_op_encoder_backward, which takes
caller-provided scratch, exactly (the scatter sums in a fixed order), on two
calls in a row with different shapes, and it must refuse sizes beyond its
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


def test_noalloc_rejects_sizes_beyond_its_array(ops):
    dummy = torch.zeros(16, device="cuda")
    tok = torch.zeros(16, dtype=torch.int32, device="cuda")
    # B*T = 32769 > GPT2_NOALLOC_MAX_TOKENS: refused before any launch
    assert ops.gpt2_op_encoder_backward_noalloc(dummy, dummy, dummy, tok, 1, 32769, 4) == -2
    assert ops.gpt2_op_encoder_backward_noalloc(dummy, dummy, dummy, tok, 1, 4, 6) == -7
