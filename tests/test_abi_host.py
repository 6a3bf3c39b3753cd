"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function its headers declare, validates configs, plans the one buffer,
and draws the same initial parameters as the oracle bit for bit."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def g():
    from gpt_transformer_train_b300 import build
    build.build()
    import gpt_transformer_train_b300 as mod
    return mod


def _declared_functions():
    names = set()
    for h in ("gpt2.h", "gpt2_ops.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(gpt2_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_headers_declare_the_model_api():
    names = _declared_functions()
    for n in ("gpt2_create", "gpt2_forward", "gpt2_backward", "gpt2_zero_grad", "gpt2_adamw_step",
              "gpt2_required_bytes", "gpt2_get_params", "gpt2_last_error", "gpt2_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol(g):
    missing = [n for n in _declared_functions() if not hasattr(g.lib, n)]
    assert not missing, missing


def _cfg(g, L=2, C=64, H=4, V=512, Vp=512, maxT=64, B=4, T=64, prec=0):
    return g.make_config(L, C, H, V, Vp, maxT, B, T, prec)


def test_parameter_counts(g):
    assert g.num_parameters(_cfg(g)) == 136_960
    c124 = g.make_config(12, 768, 12, 50257, 50304, 1024, 16, 1024, 1)
    assert g.num_parameters(c124) == 124_475_904
    assert g.num_parameters(c124) == O.num_parameters(O.GPT2_124M)
    c16 = g.make_config(48, 1600, 25, 50257, 50304, 1024, 8, 1024, 1)
    assert g.num_parameters(c16) == O.num_parameters(O.Config(48, 1600, 25, 50257, 50304, 1024))
    for t, (name, shape) in enumerate(O.param_shapes(O.GPT2_124M)):
        assert g.tensor_numel(c124, t) == int(np.prod(shape)), name


def test_invalid_configs_are_rejected(g):
    bad = [
        _cfg(g, C=63),                       # C % H
        _cfg(g, T=128),                      # T > max_T
        _cfg(g, Vp=500),                     # Vp < V
        _cfg(g, V=70000, Vp=70000),          # V too large
        _cfg(g, prec=1),                     # bf16 needs hd 64, T % 128
        _cfg(g, prec=7),
        _cfg(g, L=0),
        g.make_config(2, 128, 2, 500, 500, 128, 2, 128, 1),   # bf16: Vp % 128
    ]
    for c in bad:
        assert g.required_bytes(c) == 0
        assert g.num_parameters(c) == 0
    assert g.required_bytes(g.make_config(2, 128, 2, 500, 512, 128, 2, 128, 1)) > 0


def test_buffer_plan_fits_and_scales(g):
    c124 = g.make_config(12, 768, 12, 50257, 50304, 1024, 16, 1024, 1)
    n = g.num_parameters(c124)
    total = g.required_bytes(c124)
    # fp32 params/grads/m/v + bf16 copy, plus activations; well under HBM
    assert total > n * 18
    assert total < 20e9
    c16 = g.make_config(48, 1600, 25, 50257, 50304, 1024, 8, 1024, 1)
    assert g.required_bytes(c16) < 100e9


def test_null_and_bad_arguments(g):
    c = _cfg(g)
    h = ctypes.c_void_p()
    assert g.gpt2_create(ctypes.byref(c), 1, None, 0, None, ctypes.byref(h)) == -7
    assert g.gpt2_forward(None, None, None, None) == -7
    assert g.gpt2_backward(None) == -7
    assert g.gpt2_zero_grad(None) == -7
    assert g.gpt2_adamw_step(None, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1) == -7
    bufsize = g.required_bytes(c)
    # too small a buffer is refused before any device work
    fake = ctypes.c_void_p(1 << 20)
    assert g.gpt2_create(ctypes.byref(c), 1, fake, bufsize - 1, None, ctypes.byref(h)) == -2
    assert b"needs" in g.gpt2_last_error(None)


@pytest.mark.parametrize("cfgargs,seed", [
    ((2, 64, 4, 512, 512, 64), 1234),
    ((2, 128, 2, 1000, 1024, 256), 7),
    ((3, 192, 3, 777, 896, 128), 2**40 + 3),
])
def test_host_init_is_bit_equal_to_oracle_init(g, cfgargs, seed):
    L, C, H, V, Vp, maxT = cfgargs
    cfg = g.make_config(L, C, H, V, Vp, maxT, 1, min(64, maxT), 0)
    lib_init = g.init_params_host(cfg, seed)
    ref = O.flatten(O.init_params(O.Config(L, C, H, V, Vp, maxT), seed), O.Config(L, C, H, V, Vp, maxT))
    assert lib_init.dtype == np.float32 and ref.dtype == np.float32
    assert np.array_equal(lib_init.view(np.uint32), ref.view(np.uint32))


def test_lr_schedule_matches_oracle(g):
    """gpt2_lr_schedule (host function of the library) against the oracle's schedule."""
    for step in list(range(0, 30)) + [55, 60, 99, 100, 101, 500]:
        mine = g.lr_schedule(6e-4, 0.1, 10, 100, step)
        ref = O.lr_schedule(6e-4, 0.1, 10, 100, step)
        assert abs(mine - ref) <= 1e-6 * ref, (step, mine, ref)


def test_logit_stats_tile_count(g):
    """Column tiles of the row statistics: 256 wide from N = 512 up (the
    tensor-core kernel's tile there), else 128; the last may be narrower."""
    lib = ctypes.CDLL(g.LIB_PATH)
    f = lib.gpt2_op_logit_stats_tiles
    f.restype, f.argtypes = ctypes.c_int, [ctypes.c_int]
    assert f(50304) == 197  # GPT-2's padded vocabulary: 196 full tiles and one of 128 columns
    assert f(768) == 3 and f(1600) == 7 and f(512) == 2
    assert f(384) == 3 and f(128) == 1 and f(8) == 1
    assert f(0) == 0
