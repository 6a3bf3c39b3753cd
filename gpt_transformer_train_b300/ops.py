"""Binding of the kernel-level C ABI (include/gpt2_ops.h).

Argument marshalling only; tensors are torch CUDA tensors, scalars are
passed through.  Scratch buffers are allocated by the caller here (torch)
at the sizes the library reports.
"""
from __future__ import annotations

import ctypes

import torch

from . import GPT2Error, PRECISION_BF16, PRECISION_FP32, lib

_P, _i, _ll, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float, ctypes.c_size_t
_sigs = {
    "gpt2_op_encoder_forward": (_i, [_i, _P, _P, _P, _P, _i, _i, _i, _i, _P, _P]),
    "gpt2_op_encoder_backward_scratch_bytes": (_sz, [_i, _i, _i]),
    "gpt2_op_encoder_backward": (_i, [_P, _P, _P, _P, _i, _i, _i, _i, _P, _P, _sz, _P]),
    "gpt2_op_encoder_backward_noalloc": (_i, [_P, _P, _P, _P, _i, _i, _i, _i, _P, _P]),
    "gpt2_op_residual_layernorm_forward": (_i, [_i, _P, _P, _P, _P, _P, _P, _P, _P, _i, _i, _P]),
    "gpt2_op_layernorm_backward_scratch_bytes": (_sz, [_i, _i]),
    "gpt2_op_layernorm_backward": (_i, [_i, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _i, _i, _i, _P, _sz, _P]),
    "gpt2_op_layernorm_backward_rg": (_i, [_i, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _i, _i, _P, _sz, _P]),
    "gpt2_op_matmul_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "gpt2_op_matmul": (_i, [_i, _P, _ll, _i, _P, _ll, _i, _i, _i, _i, _P, _ll, _P, _P, _ll, _i, _i, _P, _P, _sz, _P]),
    "gpt2_op_matmul_rowdot": (_i, [_P, _ll, _P, _ll, _i, _i, _i, _P, _ll, _P, _ll, _P, _i, _i, _P, _P]),
    "gpt2_op_matmul_batched": (_i, [_i, _i, _P, _ll, _ll, _i, _P, _ll, _ll, _i, _i, _i, _i, _P, _ll, _ll, _P, _ll, _ll,
                                    _i, _i, _P, _P]),
    "gpt2_op_attention_forward": (_i, [_i, _P, _P, _P, _i, _i, _i, _i, _i, _P, _P]),
    "gpt2_op_attention_backward_scratch_bytes": (_sz, [_i, _i, _i]),
    "gpt2_op_attention_backward": (_i, [_i, _P, _P, _P, _P, _P, _i, _i, _i, _i, _i, _P, _P, _sz, _P]),
    "gpt2_op_softmax_crossentropy": (_i, [_i, _P, _P, _P, _i, _i, _i, _f, _i, _P, _P]),
    "gpt2_op_logit_stats_tiles": (_i, [_i]),
    "gpt2_op_matmul_logit_stats": (_i, [_P, _ll, _P, _ll, _i, _i, _i, _P, _ll, _P, _i, _P, _P]),
    "gpt2_op_softmax_crossentropy_stats": (_i, [_P, _P, _P, _P, _i, _i, _i, _f, _P, _P]),
    "gpt2_op_adamw": (_i, [_P, _P, _P, _P, _P, _ll, _f, _f, _f, _f, _f, _i, _P, _P]),
    "gpt2_op_grad_norm_scratch_bytes": (_sz, []),
    "gpt2_op_grad_norm": (_i, [_P, _ll, _f, _P, _P, _sz, _P]),
    "gpt2_op_gelu_forward": (_i, [_i, _P, _P, _ll, _P]),
    "gpt2_op_gelu_backward": (_i, [_i, _P, _P, _P, _ll, _P]),
    "gpt2_op_colsum_scratch_bytes": (_sz, [_i, _i]),
    "gpt2_op_colsum": (_i, [_i, _P, _P, _i, _i, _ll, _P, _sz, _P]),
    "gpt2_op_wait_probe": (_i, [_i, _P, _P]),
    "gpt2_op_lnfold_weights": (_i, [_P, _P, _P, _P, _P, _P, _P, _i, _i, _i, _P]),
    "gpt2_op_matmul_lnfold": (_i, [_P, _ll, _P, _P, _P, _ll, _P, _P, _i, _i, _i, _P, _ll, _P, _ll, _P, _P]),
}
for _n, (_r, _a) in _sigs.items():
    _fn = getattr(lib, _n)
    _fn.restype, _fn.argtypes = _r, _a

EPI_STORE, EPI_GELU, EPI_GELU_BWD, EPI_ACC_F32 = 0, 1, 2, 3
PATH_AUTO, PATH_SIMT, PATH_TC = 0, 1, 2


def _p(t):
    return None if t is None else t.data_ptr()


def _dt(t):
    if t.dtype == torch.bfloat16:
        return PRECISION_BF16
    if t.dtype == torch.float32:
        return PRECISION_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _s(stream):
    return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream


def _ck(rc, what):
    if rc:
        raise GPT2Error(rc, what)


def _scratch(nbytes, device):
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def flags(device="cuda"):
    return torch.zeros(4, dtype=torch.int32, device=device)


def gpt2_op_encoder_forward(out, tokens, wte, wpe, B, T, C, V, flags_dev, stream=None):
    _ck(lib.gpt2_op_encoder_forward(_dt(out), _p(out), _p(tokens), _p(wte), _p(wpe), B, T, C, V, _p(flags_dev),
                                    _s(stream)), "encoder_forward")


def gpt2_op_encoder_backward(dwte, dwpe, dres, tokens, B, T, C, V=None, flags_dev=None, stream=None):
    """V defaults to the row count of dwte."""
    n = lib.gpt2_op_encoder_backward_scratch_bytes(B, T, C)
    sc = _scratch(n, dres.device)
    V = dwte.shape[0] if V is None else V
    _ck(lib.gpt2_op_encoder_backward(_p(dwte), _p(dwpe), _p(dres), _p(tokens), B, T, C, V, _p(flags_dev), _p(sc),
                                     sc.numel(), _s(stream)), "encoder_backward")


def gpt2_op_encoder_backward_noalloc(dwte, dwpe, dres, tokens, B, T, C, V=None, flags_dev=None, stream=None):
    """Encoder backward whose scratch is a library-owned static device array
    (no allocation by the library or here); returns the C status code.
    V defaults to the row count of dwte."""
    V = dwte.shape[0] if V is None else V
    return lib.gpt2_op_encoder_backward_noalloc(_p(dwte), _p(dwpe), _p(dres), _p(tokens), B, T, C, V,
                                                _p(flags_dev), _s(stream))


def gpt2_op_residual_layernorm_forward(resid_out, y, mean, rstd, a, b, w, bias, rows, C, stream=None):
    _ck(lib.gpt2_op_residual_layernorm_forward(_dt(y), _p(resid_out), _p(y), _p(mean), _p(rstd), _p(a), _p(b),
                                               _p(w), _p(bias), rows, C, _s(stream)), "residual_layernorm_forward")


def gpt2_op_layernorm_backward(dres, dres_c, dy, x, mean, rstd, w, dw, db, rows, C, accumulate, stream=None,
                               dres_sum=None):
    n = lib.gpt2_op_layernorm_backward_scratch_bytes(rows, C)
    sc = _scratch(n, dy.device)
    _ck(lib.gpt2_op_layernorm_backward(_dt(dy), _p(dres), _p(dres_c), _p(dy), _p(x), _p(mean), _p(rstd), _p(w),
                                       _p(dw), _p(db), _p(dres_sum), rows, C, accumulate, _p(sc), sc.numel(),
                                       _s(stream)), "layernorm_backward")


def gpt2_op_layernorm_backward_rg(dres_out, dres_in, dres_f32, dy, x, mean, rstd, w, dw, db, rows, C, stream=None,
                                  dres_sum=None):
    n = lib.gpt2_op_layernorm_backward_scratch_bytes(rows, C)
    sc = _scratch(n, dy.device)
    _ck(lib.gpt2_op_layernorm_backward_rg(_dt(dy), _p(dres_out), _p(dres_in), _p(dres_f32), _p(dy), _p(x), _p(mean),
                                          _p(rstd), _p(w), _p(dw), _p(db), _p(dres_sum), rows, C, _p(sc), sc.numel(),
                                          _s(stream)), "layernorm_backward_rg")


def gemm_workspace(M, N, K, epilogue=EPI_ACC_F32, device="cuda"):
    """Workspace that lets the fp32-accumulate GEMM split K (None when it would not)."""
    n = lib.gpt2_op_matmul_workspace_bytes(M, N, K, epilogue)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def gpt2_op_matmul(A, lda, a_kmajor, B, ldb, b_kmajor, M, N, K, D, ldd, bias=None, aux=None, ldaux=0,
                   epilogue=EPI_STORE, path=PATH_AUTO, flags_dev=None, workspace=None, stream=None):
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ck(lib.gpt2_op_matmul(_dt(A), _p(A), lda, a_kmajor, _p(B), ldb, b_kmajor, M, N, K, _p(D), ldd, _p(bias),
                           _p(aux), ldaux, epilogue, path, _p(flags_dev), _p(workspace), wsb, _s(stream)), "matmul")


def gpt2_op_matmul_batched(batch, A, lda, sA, a_kmajor, B, ldb, sB, b_kmajor, M, N, K, D, ldd, sD, aux=None, ldaux=0,
                           sAux=0, epilogue=EPI_STORE, path=PATH_AUTO, flags_dev=None, stream=None):
    _ck(lib.gpt2_op_matmul_batched(_dt(A), batch, _p(A), lda, sA, a_kmajor, _p(B), ldb, sB, b_kmajor, M, N, K, _p(D),
                                   ldd, sD, _p(aux), ldaux, sAux, epilogue, path, _p(flags_dev), _s(stream)),
        "matmul_batched")


def gpt2_op_matmul_rowdot(dY, ldy, W, ldw, M, N, K, dX, ldx, O, ldo, D, T, H, flags_dev, stream=None):
    _ck(lib.gpt2_op_matmul_rowdot(_p(dY), ldy, _p(W), ldw, M, N, K, _p(dX), ldx, _p(O), ldo, _p(D), T, H,
                                  _p(flags_dev), _s(stream)), "matmul_rowdot")


def gpt2_op_attention_forward(out, lse, qkv, B, T, C, H, path=PATH_AUTO, flags_dev=None, stream=None):
    _ck(lib.gpt2_op_attention_forward(_dt(qkv), _p(out), _p(lse), _p(qkv), B, T, C, H, path, _p(flags_dev),
                                      _s(stream)), "attention_forward")


def gpt2_op_attention_backward(dqkv, dout, qkv, out, lse, B, T, C, H, path=PATH_AUTO, flags_dev=None, scratch=None,
                               stream=None):
    n = lib.gpt2_op_attention_backward_scratch_bytes(B, T, H)
    sc = _scratch(n, qkv.device) if scratch is None else scratch
    _ck(lib.gpt2_op_attention_backward(_dt(qkv), _p(dqkv), _p(dout), _p(qkv), _p(out), _p(lse), B, T, C, H, path,
                                       _p(flags_dev), _p(sc), sc.numel() * sc.element_size(), _s(stream)),
        "attention_backward")


def gpt2_op_softmax_crossentropy(logits, losses, targets, rows, V, Vp, dloss, write_grad, flags_dev, stream=None):
    _ck(lib.gpt2_op_softmax_crossentropy(_dt(logits), _p(logits), _p(losses), _p(targets), rows, V, Vp, dloss,
                                         write_grad, _p(flags_dev), _s(stream)), "softmax_crossentropy")


def gpt2_op_logit_stats_tiles(N):
    return lib.gpt2_op_logit_stats_tiles(N)


def gpt2_op_matmul_logit_stats(A, lda, B, ldb, M, N, K, D, ldd, stats, stats_cols, flags_dev, stream=None):
    _ck(lib.gpt2_op_matmul_logit_stats(_p(A), lda, _p(B), ldb, M, N, K, _p(D), ldd, _p(stats), stats_cols,
                                       _p(flags_dev), _s(stream)), "matmul_logit_stats")


def gpt2_op_softmax_crossentropy_stats(logits, losses, targets, stats, rows, V, Vp, dloss, flags_dev, stream=None):
    _ck(lib.gpt2_op_softmax_crossentropy_stats(_p(logits), _p(losses), _p(targets), _p(stats), rows, V, Vp, dloss,
                                               _p(flags_dev), _s(stream)), "softmax_crossentropy_stats")


def gpt2_op_adamw(p, g, m, v, p_bf16, lr, b1, b2, eps, wd, t, gscale=None, stream=None):
    _ck(lib.gpt2_op_adamw(_p(p), _p(g), _p(m), _p(v), _p(p_bf16), p.numel(), lr, b1, b2, eps, wd, t, _p(gscale),
                          _s(stream)), "adamw")


def gpt2_op_grad_norm(g, max_norm, out2, stream=None):
    """out2[0] = ||g||, out2[1] = clip factor min(1, max_norm / (norm + 1e-6))."""
    sc = _scratch(lib.gpt2_op_grad_norm_scratch_bytes(), g.device)
    _ck(lib.gpt2_op_grad_norm(_p(g), g.numel(), max_norm, _p(out2), _p(sc), sc.numel(), _s(stream)), "grad_norm")


def gpt2_op_gelu_forward(out, inp, stream=None):
    _ck(lib.gpt2_op_gelu_forward(_dt(inp), _p(out), _p(inp), inp.numel(), _s(stream)), "gelu_forward")


def gpt2_op_gelu_backward(dinp, inp, dout, stream=None):
    _ck(lib.gpt2_op_gelu_backward(_dt(inp), _p(dinp), _p(inp), _p(dout), inp.numel(), _s(stream)), "gelu_backward")


def gpt2_op_colsum(out, X, rows, cols, ldx, stream=None):
    n = lib.gpt2_op_colsum_scratch_bytes(rows, cols)
    sc = _scratch(n, X.device)
    _ck(lib.gpt2_op_colsum(_dt(X), _p(out), _p(X), rows, cols, ldx, _p(sc), sc.numel(), _s(stream)), "colsum")


def gpt2_op_wait_probe(limit_us, flags_dev, stream=None):
    """Run the bounded-wait failure path on purpose; returns the C status code
    (GPT2_ERR_TIMEOUT, -8, is the expected outcome)."""
    return lib.gpt2_op_wait_probe(limit_us, _p(flags_dev), _s(stream))


def gpt2_op_lnfold_weights(Wf, s, c, W, gamma, beta, bias, items, N, K, stream=None):
    _ck(lib.gpt2_op_lnfold_weights(_p(Wf), _p(s), _p(c), _p(W), _p(gamma), _p(beta), _p(bias), items, N, K,
                                   _s(stream)), "lnfold_weights")


def gpt2_op_matmul_lnfold(R, ldr, mean, rstd, Wf, ldw, s, c, M, N, K, D, ldd, aux=None, ldaux=0, flags_dev=None,
                          stream=None):
    _ck(lib.gpt2_op_matmul_lnfold(_p(R), ldr, _p(mean), _p(rstd), _p(Wf), ldw, _p(s), _p(c), M, N, K, _p(D), ldd,
                                  _p(aux), ldaux, _p(flags_dev), _s(stream)), "matmul_lnfold")
