"""Python binding of the GPT-2 B300 training-step library (libgpt2.so).

Argument marshalling only: every step of the forward, backward and AdamW runs
in the library's CUDA kernels.  PyTorch supplies the one device buffer and the
stream.  The functions keep the C names of include/gpt2.h; `GPT2` wraps a
handle for convenience.  If the shared library is missing this module raises
ImportError: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgpt2.so")

GPT2_OK = 0
ERRORS = {-1: "INVALID_CONFIG", -2: "BUFFER_TOO_SMALL", -3: "BAD_ORDER", -4: "TOKEN_RANGE", -5: "CUDA",
          -6: "NAN", -7: "INVALID_ARG", -8: "TIMEOUT"}
PRECISION_FP32, PRECISION_BF16 = 0, 1
TENSORS = ("wte", "wpe", "ln1w", "ln1b", "qkvw", "qkvb", "attprojw", "attprojb",
           "ln2w", "ln2b", "fcw", "fcb", "fcprojw", "fcprojb", "lnfw", "lnfb")

from . import build as _build  # noqa: E402  (the build module has no dependency on this one)

if _build.needs_build():
    try:
        _build.build()
    except Exception as e:  # no silent fallback: the CUDA library is the product
        raise ImportError(f"cannot build {LIB_PATH}: {e}") from e
if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -m gpt_transformer_train_b300.build`")
_lib = ctypes.CDLL(LIB_PATH)


class gpt2_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("L", "C", "H", "max_T", "V", "Vp", "B", "T", "precision", "recompute",
                                            "ln_fold")]


_P = ctypes.c_void_p
_cfgp = ctypes.POINTER(gpt2_config)
_f = ctypes.c_float
_sigs = {
    "gpt2_num_parameters": (ctypes.c_size_t, [_cfgp]),
    "gpt2_tensor_numel": (ctypes.c_size_t, [_cfgp, ctypes.c_int]),
    "gpt2_required_bytes": (ctypes.c_size_t, [_cfgp]),
    "gpt2_init_params_host": (ctypes.c_int, [_cfgp, ctypes.c_uint64, _P]),
    "gpt2_create": (ctypes.c_int, [_cfgp, ctypes.c_uint64, _P, ctypes.c_size_t, _P, ctypes.POINTER(_P)]),
    "gpt2_forward": (ctypes.c_int, [_P, _P, _P, _P]),
    "gpt2_backward": (ctypes.c_int, [_P]),
    "gpt2_zero_grad": (ctypes.c_int, [_P]),
    "gpt2_adamw_step": (ctypes.c_int, [_P, _f, _f, _f, _f, _f, ctypes.c_int]),
    "gpt2_clip_grad_norm": (ctypes.c_int, [_P, _f]),
    "gpt2_graph_step": (ctypes.c_int, [_P, _P, _P]),
    "gpt2_get_grad_norm": (ctypes.c_int, [_P, _P]),
    "gpt2_lr_schedule": (_f, [_f, _f, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "gpt2_step_host": (ctypes.c_int, [_P, _P, _P, _f, _f, _f, _f, _f, ctypes.c_int, _P]),
    "gpt2_infer_prefill": (ctypes.c_int, [_P, _P, ctypes.c_int]),
    "gpt2_infer_step": (ctypes.c_int, [_P, _P, ctypes.c_int]),
    "gpt2_sample": (ctypes.c_int, [_P, _f, _P, _P]),
    "gpt2_get_infer_logits": (ctypes.c_int, [_P, _P]),
    "gpt2_get_params": (ctypes.c_int, [_P, ctypes.c_int, _P]),
    "gpt2_set_params": (ctypes.c_int, [_P, ctypes.c_int, _P]),
    "gpt2_get_grads": (ctypes.c_int, [_P, ctypes.c_int, _P]),
    "gpt2_get_logits": (ctypes.c_int, [_P, _P]),
    "gpt2_get_losses": (ctypes.c_int, [_P, _P]),
    "gpt2_get_loss": (ctypes.c_int, [_P, _P]),
    "gpt2_sync": (ctypes.c_int, [_P]),
    "gpt2_profile_gemm": (ctypes.c_int, [_P, ctypes.c_int]),
    "gpt2_profile_read": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_uint64),
                                         ctypes.POINTER(ctypes.c_double)]),
    "gpt2_launch_count": (ctypes.c_uint64, [_P]),
    "gpt2_last_error": (ctypes.c_char_p, [_P]),
    "gpt2_destroy": (None, [_P]),
}
for _n, (_r, _a) in _sigs.items():
    _fn = getattr(_lib, _n)
    _fn.restype, _fn.argtypes = _r, _a
    globals()[_n] = _fn

lib = _lib


class GPT2Error(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        return a.ctypes.data
    return a.data_ptr()  # torch tensor


def make_config(L, C, H, V, Vp, max_T, B, T, precision=PRECISION_BF16, recompute=0, ln_fold=0):
    return gpt2_config(L, C, H, max_T, V, Vp, B, T, precision, recompute, ln_fold)


def num_parameters(cfg):
    return gpt2_num_parameters(ctypes.byref(cfg))


def lr_schedule(max_lr, final_frac, warmup, total, step):
    return float(gpt2_lr_schedule(max_lr, final_frac, warmup, total, step))


def required_bytes(cfg):
    return gpt2_required_bytes(ctypes.byref(cfg))


def tensor_numel(cfg, t):
    return gpt2_tensor_numel(ctypes.byref(cfg), t)


def init_params_host(cfg, seed):
    out = np.empty(num_parameters(cfg), dtype=np.float32)
    rc = gpt2_init_params_host(ctypes.byref(cfg), seed, out.ctypes.data)
    if rc:
        raise GPT2Error(rc, gpt2_last_error(None).decode())
    return out


class GPT2:
    """A model in one torch-allocated device buffer, driven through the C ABI."""

    def __init__(self, cfg: gpt2_config, seed: int = 1234, stream=None, device="cuda"):
        import torch
        self.cfg = cfg
        nbytes = required_bytes(cfg)
        if nbytes == 0:
            raise GPT2Error(-1, "invalid config")
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.buf.device)
        h = _P()
        rc = gpt2_create(ctypes.byref(cfg), seed, self.buf.data_ptr(), nbytes, _P(self.stream.cuda_stream),
                         ctypes.byref(h))
        if rc:
            raise GPT2Error(rc, gpt2_last_error(None).decode())
        self.h = h

    def _check(self, rc):
        if rc:
            raise GPT2Error(rc, gpt2_last_error(self.h).decode())

    def gpt2_forward(self, tokens, targets=None, want_loss=True):
        loss = np.zeros(1, np.float32)
        self._check(gpt2_forward(self.h, _ptr(tokens), _ptr(targets),
                                 loss.ctypes.data if (targets is not None and want_loss) else None))
        return float(loss[0]) if (targets is not None and want_loss) else None

    def gpt2_backward(self):
        self._check(gpt2_backward(self.h))

    def gpt2_zero_grad(self):
        self._check(gpt2_zero_grad(self.h))

    def gpt2_adamw_step(self, lr, b1, b2, eps, wd, t):
        self._check(gpt2_adamw_step(self.h, lr, b1, b2, eps, wd, t))

    def gpt2_graph_step(self, tokens, targets):
        self._check(gpt2_graph_step(self.h, _ptr(tokens), _ptr(targets)))

    def gpt2_clip_grad_norm(self, max_norm):
        self._check(gpt2_clip_grad_norm(self.h, max_norm))

    def gpt2_get_grad_norm(self):
        out = np.zeros(1, np.float32)
        self._check(gpt2_get_grad_norm(self.h, out.ctypes.data))
        return float(out[0])

    def gpt2_step_host(self, tokens_host, targets_host, lr, b1, b2, eps, wd, t):
        loss = np.zeros(1, np.float32)
        self._check(gpt2_step_host(self.h, _ptr(tokens_host), _ptr(targets_host), lr, b1, b2, eps, wd, t,
                                   loss.ctypes.data))
        return float(loss[0])

    # inference with a KV cache
    def gpt2_infer_prefill(self, tokens, n):
        self._check(gpt2_infer_prefill(self.h, _ptr(tokens), n))

    def gpt2_infer_step(self, next_tokens, pos):
        self._check(gpt2_infer_step(self.h, _ptr(next_tokens), pos))

    def gpt2_sample(self, temperature, coins, out_tokens):
        self._check(gpt2_sample(self.h, temperature, _ptr(coins), _ptr(out_tokens)))

    def gpt2_get_infer_logits(self):
        c = self.cfg
        out = np.empty(c.B * c.Vp, np.float32)
        self._check(gpt2_get_infer_logits(self.h, out.ctypes.data))
        return out.reshape(c.B, c.Vp)

    def numel(self, name):
        return tensor_numel(self.cfg, TENSORS.index(name))

    def gpt2_get_params(self, name):
        out = np.empty(self.numel(name), np.float32)
        self._check(gpt2_get_params(self.h, TENSORS.index(name), out.ctypes.data))
        return out

    def gpt2_set_params(self, name, values):
        v = np.ascontiguousarray(values, dtype=np.float32).reshape(-1)
        assert v.size == self.numel(name)
        self._check(gpt2_set_params(self.h, TENSORS.index(name), v.ctypes.data))

    def gpt2_get_grads(self, name):
        out = np.empty(self.numel(name), np.float32)
        self._check(gpt2_get_grads(self.h, TENSORS.index(name), out.ctypes.data))
        return out

    def gpt2_get_logits(self):
        c = self.cfg
        out = np.empty(c.B * c.T * c.Vp, np.float32)
        self._check(gpt2_get_logits(self.h, out.ctypes.data))
        return out.reshape(c.B, c.T, c.Vp)

    def gpt2_get_losses(self):
        c = self.cfg
        out = np.empty(c.B * c.T, np.float32)
        self._check(gpt2_get_losses(self.h, out.ctypes.data))
        return out.reshape(c.B, c.T)

    def gpt2_get_loss(self):
        out = np.zeros(1, np.float32)
        self._check(gpt2_get_loss(self.h, out.ctypes.data))
        return float(out[0])

    def gpt2_sync(self):
        self._check(gpt2_sync(self.h))

    def gpt2_profile_gemm(self, enable=True):
        self._check(gpt2_profile_gemm(self.h, int(enable)))

    def gpt2_profile_read(self):
        ms, n, fl = ctypes.c_double(), ctypes.c_uint64(), ctypes.c_double()
        self._check(gpt2_profile_read(self.h, ctypes.byref(ms), ctypes.byref(n), ctypes.byref(fl)))
        return ms.value, n.value, fl.value

    def launch_count(self):
        return int(gpt2_launch_count(self.h))

    def close(self):
        if getattr(self, "h", None):
            gpt2_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
