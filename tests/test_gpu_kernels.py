"""Per-kernel parity: each CUDA kernel, called through the kernel-level C ABI,
against the oracle's function for the same layer, on seeded inputs with
ragged sizes (rows not multiples of the tile, odd channel counts).

Tolerances: fp32 kernels against the float64 oracle at 1e-5 relative (sum
order only); bf16 kernels at the bf16 rounding scale, 2^-8 relative per
stored element, with reductions done in fp32.  The tensor-core GEMM and
attention kernels are also held to element-wise bounds (tests/parity.py): a
single wrong element or tile fails them, which a norm would not show.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from parity import (check, gemm_ref, gemm_bound, gelu_bound, gelu_bwd_bound, attention_bounds, U8)
from synthetic import normal_array, zipf_tokens

pytestmark = pytest.mark.gpu

DT = {"fp32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def ops():
    from gpt_transformer_train_b300 import build
    build.build()
    import gpt_transformer_train_b300.ops as ops
    return ops


def dev(a, dt=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda").to(dt)


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


def as_stored(a, dt):
    """The values a kernel actually sees after the input is stored in dt."""
    return host(dev(a, dt))


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


# ---------------------------------------------------------------------------
def test_encoder_forward_fp32_bit_exact(ops):
    B, T, C, V = 3, 37, 64, 500
    tok, _ = zipf_tokens(B, T, V, 1)
    wte, wpe = normal_array((V, C), 2, 0.02), normal_array((T, C), 3, 0.02)
    out = torch.empty(B * T, C, device="cuda")
    fl = ops.flags()
    ops.gpt2_op_encoder_forward(out, dev(tok, torch.int32), dev(wte), dev(wpe), B, T, C, V, fl)
    ref = O.encoder_forward(wte, wpe, tok).reshape(B * T, C)
    assert ref.dtype == np.float32
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert fl.sum().item() == 0


def test_encoder_forward_bf16_gather_exact(ops):
    B, T, C, V = 2, 50, 128, 300
    tok, _ = zipf_tokens(B, T, V, 4)
    wte = dev(normal_array((V, C), 5, 0.02), torch.bfloat16)
    wpe = dev(normal_array((T, C), 6, 0.02), torch.bfloat16)
    out = torch.empty(B * T, C, device="cuda", dtype=torch.bfloat16)
    ops.gpt2_op_encoder_forward(out, dev(tok, torch.int32), wte, wpe, B, T, C, V, ops.flags())
    ref32 = O.encoder_forward(wte.float().cpu().numpy(), wpe.float().cpu().numpy(), tok).reshape(B * T, C)
    ref = torch.from_numpy(ref32).to(torch.bfloat16)          # one rounding of the fp32 sum
    assert torch.equal(out.cpu().view(torch.int16), ref.view(torch.int16))


def test_encoder_forward_flags_bad_tokens(ops):
    B, T, C, V = 1, 8, 64, 16
    tok = np.arange(8, dtype=np.int32).reshape(1, 8)
    tok[0, 3] = 16
    tok[0, 5] = -2
    fl = ops.flags()
    out = torch.empty(8, C, device="cuda")
    ops.gpt2_op_encoder_forward(out, dev(tok, torch.int32), dev(np.ones((V, C), np.float32)),
                                dev(np.ones((T, C), np.float32)), B, T, C, V, fl)
    assert fl[0].item() & 1


@pytest.mark.parametrize("B,T,C", [(2, 7, 64), (4, 64, 192), (1, 300, 768), (3, 700, 64), (16, 1024, 768),
                                   (32, 1000, 64)])
def test_encoder_backward_deterministic_scatter(ops, B, T, C):
    """Scatter-add without atomics: repeated calls give identical bits; values
    match the float64 sums within fp32 rounding; dwpe (a plain sum over the
    batch in increasing b) matches the oracle's float32 sum exactly."""
    V = 97 if B * T < 4096 else 50257
    tok, _ = zipf_tokens(B, T, V, B * T)
    dres = normal_array((B, T, C), 8)
    td, tt = dev(dres), dev(tok, torch.int32)
    outs = []
    for _ in range(2):
        dwte = torch.zeros(V, C, device="cuda")
        dwpe = torch.zeros(T + 3, C, device="cuda")
        ops.gpt2_op_encoder_backward(dwte, dwpe, td, tt, B, T, C)
        outs.append((dwte, dwpe))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    rw, rp = O.encoder_backward(dres.astype(np.float64), tok, V, T + 3)
    dwte, dwpe = host(outs[0][0]), host(outs[0][1])
    # the row sum of n fp32 values is within n * 2^-24 * sum|x| of the exact sum
    bound = np.zeros((V, C))
    np.add.at(bound, tok.reshape(-1), np.abs(dres.reshape(-1, C).astype(np.float64)))
    cnt = np.bincount(tok.reshape(-1), minlength=V)[:, None]
    assert np.all(np.abs(dwte - rw) <= cnt * 2.0 ** -24 * bound + 1e-30)
    assert np.array_equal(host(outs[0][1]).astype(np.float32), O.encoder_backward(dres, tok, V, T + 3)[1])


@pytest.mark.parametrize("B,T", [(2, 100), (17, 1000)])
def test_encoder_backward_out_of_range_tokens(ops, B, T):
    """Both sort forms (radix up to 16384 positions, bitonic above): tokens
    -1, V and V + 5 add nothing to dwte and raise the token flag; dwte has
    65536 rows of which the first V are passed, the rest a guard band."""
    C, V = 64, 500
    tok, _ = zipf_tokens(B, T, V, 31)
    tok[0, 3], tok[1, 50], tok[-1, -1] = -1, V + 5, V
    good = ((tok >= 0) & (tok < V)).reshape(-1)
    dres = normal_array((B * T, C), 32)
    base = normal_array((65536, C), 33)
    w, p, fl = dev(base), torch.zeros(T, C, device="cuda"), ops.flags()
    ops.gpt2_op_encoder_backward(w, p, dev(dres), dev(tok, torch.int32), B, T, C, V=V, flags_dev=fl)
    torch.cuda.synchronize()
    assert fl[0].item() & 1
    assert torch.equal(w[V:], dev(base[V:]))
    ref = base[:V].astype(np.float64)
    np.add.at(ref, tok.reshape(-1)[good], dres.astype(np.float64)[good])
    assert np.max(np.abs(host(w[:V]) - ref)) < 1e-4


@pytest.mark.parametrize("pattern", ["one_token", "blocks_of_32", "blocks_of_33", "ascending"])
def test_encoder_backward_run_patterns(ops, pattern):
    """Token runs that fill whole sorted chunks, end exactly on a chunk
    boundary, straddle one, or are all length 1: the chunked dwte sums against
    float64, bitwise repeatable."""
    B, T, C, V = 4, 256, 128, 600
    n = B * T
    if pattern == "one_token":
        tok = np.full(n, 7, np.int32)
    elif pattern == "blocks_of_32":
        tok = (np.arange(n) // 32).astype(np.int32)[::-1].copy()
    elif pattern == "blocks_of_33":
        tok = ((np.arange(n) * 7919) % n // 33).astype(np.int32)
    else:
        tok = (np.arange(n) % V).astype(np.int32)
    tok = tok.reshape(B, T)
    dres = normal_array((B, T, C), 9)
    td, tt = dev(dres), dev(tok, torch.int32)
    outs = []
    for _ in range(2):
        dwte, dwpe = torch.zeros(V, C, device="cuda"), torch.zeros(T, C, device="cuda")
        ops.gpt2_op_encoder_backward(dwte, dwpe, td, tt, B, T, C)
        outs.append(dwte)
    assert torch.equal(outs[0], outs[1])
    rw, _ = O.encoder_backward(dres.astype(np.float64), tok, V, T)
    bound = np.zeros((V, C))
    np.add.at(bound, tok.reshape(-1), np.abs(dres.reshape(-1, C).astype(np.float64)))
    cnt = np.bincount(tok.reshape(-1), minlength=V)[:, None]
    assert np.all(np.abs(host(outs[0]) - rw) <= cnt * 2.0 ** -24 * bound + 1e-30)


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dt", ["fp32", "bf16"])
@pytest.mark.parametrize("rows,C", [(1, 64), (37, 768), (130, 1600), (5, 2048)])
@pytest.mark.parametrize("fused", [False, True])
def test_residual_layernorm_forward(ops, dt, rows, C, fused):
    a, b = normal_array((rows, C), 10, 1.0), normal_array((rows, C), 11, 0.5)
    w, bias = normal_array((C,), 12, 0.3) + 1, normal_array((C,), 13, 0.1)
    ta, tb, tw, tbias = dev(a, DT[dt]), dev(b, DT[dt]), dev(w, DT[dt]), dev(bias, DT[dt])
    y = torch.empty(rows, C, device="cuda", dtype=DT[dt])
    r = torch.empty_like(y)
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    ops.gpt2_op_residual_layernorm_forward(r if fused else None, y, mean, rstd, ta, tb if fused else None, tw,
                                           tbias, rows, C)
    x = host(ta) + host(tb) if fused else host(ta)
    if fused and dt == "bf16":
        x = as_stored(x, torch.bfloat16)          # the stored residual is rounded first
    ry, rm, rr = O.layernorm_forward(x, host(tw), host(tbias))
    if fused:
        tol = 0 if dt == "fp32" else 0
        assert np.max(np.abs(host(r) - as_stored(x, DT[dt]))) <= tol
    assert np.allclose(host(mean), rm, rtol=1e-5, atol=1e-5)
    assert np.allclose(host(rstd), rr, rtol=1e-5)
    if dt == "fp32":
        assert np.max(np.abs(host(y) - ry)) < 2e-5
    else:
        assert np.max(np.abs(host(y) - ry) / (np.abs(ry) + 1e-2)) < 2 ** -7


@pytest.mark.parametrize("dt", ["fp32", "bf16"])
@pytest.mark.parametrize("rows,C", [(3, 64), (129, 768), (64, 1600), (1000, 1024), (2000, 512), (16384, 768)])
def test_layernorm_backward(ops, dt, rows, C):
    x = normal_array((rows, C), 20, 1.5)
    w = normal_array((C,), 21, 0.2) + 1
    dy = normal_array((rows, C), 22)
    dres0 = normal_array((rows, C), 23)
    tx, tw, tdy = dev(x, DT[dt]), dev(w, DT[dt]), dev(dy, DT[dt])
    xs, ws, dys = host(tx), host(tw), host(tdy)
    _, mean, rstd = O.layernorm_forward(xs, ws, np.zeros(C))
    dres = dev(dres0)
    dres_c = torch.empty(rows, C, device="cuda", dtype=DT[dt])
    dw = torch.zeros(C, device="cuda")
    db = torch.full((C,), 0.5, device="cuda")
    rsum = torch.full((C,), -0.25, device="cuda")
    tmean, trstd = dev(mean.astype(np.float32)), dev(rstd.astype(np.float32))
    ops.gpt2_op_layernorm_backward(dres, dres_c, tdy, tx, tmean, trstd, tw, dw, db, rows, C, 1, dres_sum=rsum)
    rdx, rdw, rdb = O.layernorm_backward(dys, xs, mean, rstd, ws)
    assert rel_l2(host(dres), dres0 + rdx) < 1e-5
    assert rel_l2(host(dw), rdw) < 1e-5
    assert rel_l2(host(db), rdb + 0.5) < 1e-5
    # column sums of the new residual gradient (the next projection's bias gradient)
    assert rel_l2(host(rsum), (dres0 + rdx).sum(0) - 0.25) < 1e-5
    assert np.max(np.abs(host(dres_c) - as_stored(host(dres), DT[dt]))) == 0
    # the same call again from the same state gives identical bits (fixed-order sums)
    dres2, dw2, db2, rsum2 = dev(dres0), torch.zeros(C, device="cuda"), torch.full((C,), 0.5, device="cuda"), \
        torch.full((C,), -0.25, device="cuda")
    ops.gpt2_op_layernorm_backward(dres2, None, tdy, tx, tmean, trstd, tw, dw2, db2, rows, C, 1, dres_sum=rsum2)
    assert torch.equal(dres, dres2) and torch.equal(dw, dw2) and torch.equal(db, db2) and torch.equal(rsum, rsum2)


@pytest.mark.parametrize("dt", ["fp32", "bf16"])
@pytest.mark.parametrize("rows,C", [(3, 64), (129, 768), (64, 1600), (16384, 768)])
@pytest.mark.parametrize("in_place", [False, True])
def test_layernorm_backward_residual_in_dtype(ops, dt, rows, C, in_place):
    """The step's LayerNorm backward: the residual gradient passed along in the
    activation dtype (new = incoming + dx, stored in dtype), an fp32 copy of
    the new value, and the parameter / bias sums, against the oracle; the
    stored value is the fp32 copy rounded once."""
    x = normal_array((rows, C), 120, 1.5)
    w = normal_array((C,), 121, 0.2) + 1
    dy = normal_array((rows, C), 122)
    r0 = normal_array((rows, C), 123)
    tx, tw, tdy, tr0 = dev(x, DT[dt]), dev(w, DT[dt]), dev(dy, DT[dt]), dev(r0, DT[dt])
    xs, ws, dys, r0s = host(tx), host(tw), host(tdy), host(tr0)
    _, mean, rstd = O.layernorm_forward(xs, ws, np.zeros(C))
    tmean, trstd = dev(mean.astype(np.float32)), dev(rstd.astype(np.float32))
    out = tr0 if in_place else torch.empty(rows, C, device="cuda", dtype=DT[dt])
    f32 = torch.empty(rows, C, device="cuda")
    dw, db, rsum = torch.zeros(C, device="cuda"), torch.zeros(C, device="cuda"), torch.zeros(C, device="cuda")
    ops.gpt2_op_layernorm_backward_rg(out, tr0, f32, tdy, tx, tmean, trstd, tw, dw, db, rows, C, dres_sum=rsum)
    rdx, rdw, rdb = O.layernorm_backward(dys, xs, mean, rstd, ws)
    new = r0s + rdx
    assert rel_l2(host(f32), new) < 1e-5
    assert torch.equal(out, f32.to(DT[dt]))
    assert rel_l2(host(dw), rdw) < 1e-5 and rel_l2(host(db), rdb) < 1e-5
    assert rel_l2(host(rsum), new.sum(0)) < 1e-5
    # no incoming gradient: the fp32 copy alone
    f32b = torch.empty(rows, C, device="cuda")
    ops.gpt2_op_layernorm_backward_rg(None, None, f32b, tdy, tx, tmean, trstd, tw, None, None, rows, C)
    assert rel_l2(host(f32b), rdx) < 1e-5


@pytest.mark.parametrize("rows,C", [(77, 768), (16384, 768)])
def test_layernorm_backward_overwrite(ops, rows, C):
    """accumulate=0: the residual gradient is overwritten with dx (the first
    LayerNorm backward of the step), without parameter sums."""
    x, w, dy = normal_array((rows, C), 24, 1.5), normal_array((C,), 25, 0.2) + 1, normal_array((rows, C), 26)
    tx, tw, tdy = dev(x, torch.bfloat16), dev(w, torch.bfloat16), dev(dy, torch.bfloat16)
    xs, ws, dys = host(tx), host(tw), host(tdy)
    _, mean, rstd = O.layernorm_forward(xs, ws, np.zeros(C))
    dres = dev(normal_array((rows, C), 27))  # garbage that must not leak in
    ops.gpt2_op_layernorm_backward(dres, None, tdy, tx, dev(mean.astype(np.float32)), dev(rstd.astype(np.float32)),
                                   tw, None, None, rows, C, 0)
    rdx, _, _ = O.layernorm_backward(dys, xs, mean, rstd, ws)
    assert rel_l2(host(dres), rdx) < 1e-5


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dt", ["fp32", "bf16"])
@pytest.mark.parametrize("akm,bkm", [(1, 1), (1, 0), (0, 0), (0, 1)])
@pytest.mark.parametrize("M,N,K", [(65, 33, 17), (128, 192, 64), (200, 70, 300)])
def test_matmul_simt_layouts(ops, dt, akm, bkm, M, N, K):
    A = normal_array((M * K,), 30)
    B = normal_array((N * K,), 31)
    tA, tB = dev(A, DT[dt]), dev(B, DT[dt])
    D = torch.empty(M, N, device="cuda", dtype=DT[dt])
    ops.gpt2_op_matmul(tA, K if akm else M, akm, tB, K if bkm else N, bkm, M, N, K, D, N, path=ops.PATH_SIMT)
    ref, _ = gemm_ref(host(tA), host(tB), akm, bkm, M, N, K)
    tol = 1e-5 if dt == "fp32" else 2 ** -7
    assert rel_l2(host(D), ref) < tol


@pytest.mark.parametrize("dt", ["fp32", "bf16"])
def test_matmul_simt_epilogues(ops, dt):
    M, N, K = 96, 80, 48
    A, B, bias = normal_array((M, K), 40), normal_array((N, K), 41), normal_array((N,), 42)
    tA, tB, tbias = dev(A, DT[dt]), dev(B, DT[dt]), dev(bias, DT[dt])
    acc = host(tA) @ host(tB).T
    pre = torch.empty(M, N, device="cuda", dtype=DT[dt])
    D = torch.empty(M, N, device="cuda", dtype=DT[dt])
    ops.gpt2_op_matmul(tA, K, 1, tB, K, 1, M, N, K, D, N, bias=tbias, aux=pre, ldaux=N, epilogue=ops.EPI_GELU,
                       path=ops.PATH_SIMT)
    tol = 1e-5 if dt == "fp32" else 2 ** -7
    assert rel_l2(host(pre), acc + host(tbias)) < tol
    assert rel_l2(host(D), O.gelu_forward(acc + host(tbias))) < tol
    D2 = torch.empty_like(D)
    ops.gpt2_op_matmul(tA, K, 1, tB, K, 1, M, N, K, D2, N, aux=pre, ldaux=N, epilogue=ops.EPI_GELU_BWD,
                       path=ops.PATH_SIMT)
    assert rel_l2(host(D2), O.gelu_backward(host(pre), acc)) < tol
    F = dev(np.ones((M, N), np.float32))
    ops.gpt2_op_matmul(tA, K, 1, tB, K, 1, M, N, K, F, N, epilogue=ops.EPI_ACC_F32, path=ops.PATH_SIMT)
    assert rel_l2(host(F), acc + 1) < 1e-5


@pytest.mark.parametrize("dt", ["fp32", "bf16"])
@pytest.mark.parametrize("M,N,K", [(1, 200, 64), (7, 768, 768), (16, 2304, 768), (32, 768, 3072)])
def test_matmul_few_rows(ops, dt, M, N, K):
    """Products with at most 32 rows (the decode step's): path 0 takes the
    few-row kernel; plain, +bias and +bias+GELU (pre-activation in aux)."""
    A, B, bias = normal_array((M, K), 43), normal_array((N, K), 44, 0.05), normal_array((N,), 45)
    tA, tB, tbias = dev(A, DT[dt]), dev(B, DT[dt]), dev(bias, DT[dt])
    acc = host(tA).astype(np.float64) @ host(tB).astype(np.float64).T
    tol = 1e-5 if dt == "fp32" else 2 ** -7
    D = torch.empty(M, N, device="cuda", dtype=DT[dt])
    ops.gpt2_op_matmul(tA, K, 1, tB, K, 1, M, N, K, D, N)
    assert rel_l2(host(D), acc) < tol
    ops.gpt2_op_matmul(tA, K, 1, tB, K, 1, M, N, K, D, N, bias=tbias)
    assert rel_l2(host(D), acc + host(tbias)) < tol
    pre = torch.empty_like(D)
    ops.gpt2_op_matmul(tA, K, 1, tB, K, 1, M, N, K, D, N, bias=tbias, aux=pre, ldaux=N, epilogue=ops.EPI_GELU)
    assert rel_l2(host(pre), acc + host(tbias)) < tol
    assert rel_l2(host(D), O.gelu_forward(host(pre).astype(np.float64))) < tol


# ---- tensor-core (tcgen05/TMA) GEMM --------------------------------------
# Row strides must be multiples of 8 bf16 (16 bytes) for TMA; M, N, K need
# not be tile multiples (K=104, M=136, N=136/264 exercise the ragged edges).
# The last two have enough output tiles for the cluster-pair path (two CTAs
# sharing B tiles by multicast), with an odd number of 128-row tiles.
TC_SHAPES = [(128, 256, 64), (256, 512, 192), (200, 136, 104), (384, 128, 320), (1024, 768, 768), (136, 264, 72),
             (4200, 1280, 320), (8200, 264, 200)]


@pytest.mark.parametrize("akm,bkm", [(1, 1), (1, 0), (0, 0), (0, 1)])
@pytest.mark.parametrize("M,N,K", TC_SHAPES)
def test_matmul_tc_layouts(ops, akm, bkm, M, N, K):
    A = normal_array((M * K,), 130 + M)
    B = normal_array((N * K,), 131 + N)
    tA, tB = dev(A, torch.bfloat16), dev(B, torch.bfloat16)
    D = torch.full((M, N), float("nan"), device="cuda", dtype=torch.bfloat16)
    fl = ops.flags()
    ops.gpt2_op_matmul(tA, K if akm else M, akm, tB, K if bkm else N, bkm, M, N, K, D, N, path=ops.PATH_TC,
                       flags_dev=fl)
    ref, absprod = gemm_ref(host(tA), host(tB), akm, bkm, M, N, K)
    assert fl.sum().item() == 0
    assert rel_l2(host(D), ref) < 2 ** -7
    check(host(D), ref, gemm_bound(ref, absprod), "D")


# (12800, 400, 136): more tiles than CTA pairs, and edge tiles with an odd
# number of live 32- and 64-column chunks, so a CTA's staging-buffer
# alternation carries over from one tile to the next
@pytest.mark.parametrize("M,N,K", [(256, 256, 320), (256, 384, 320), (8200, 640, 136), (12800, 400, 136)])
def test_matmul_tc_epilogues(ops, M, N, K):
    A, B, bias = normal_array((M, K), 140), normal_array((N, K), 141), normal_array((N,), 142)
    tA, tB, tbias = dev(A, torch.bfloat16), dev(B, torch.bfloat16), dev(bias, torch.bfloat16)
    acc, absprod = gemm_ref(host(tA), host(tB), 1, 1, M, N, K)
    hb = host(tbias)
    fl = ops.flags()
    D = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    ops.gpt2_op_matmul(tA, K, 1, tB, K, 1, M, N, K, D, N, bias=tbias, path=ops.PATH_TC, flags_dev=fl)
    assert rel_l2(host(D), acc + hb) < 2 ** -7
    check(host(D), acc + hb, gemm_bound(acc + hb, absprod + np.abs(hb)), "D + bias")
    pre = torch.empty_like(D)
    ops.gpt2_op_matmul(tA, K, 1, tB, K, 1, M, N, K, D, N, bias=tbias, aux=pre, ldaux=N, epilogue=ops.EPI_GELU,
                       path=ops.PATH_TC, flags_dev=fl)
    assert rel_l2(host(pre), acc + hb) < 2 ** -7
    assert rel_l2(host(D), O.gelu_forward(acc + hb)) < 2 ** -7
    check(host(pre), acc + hb, gemm_bound(acc + hb, absprod + np.abs(hb)), "pre-activation")
    g_ref = O.gelu_forward(host(pre))  # GELU of the stored pre-activation
    check(host(D), g_ref, gelu_bound(g_ref, host(pre)), "GELU")
    D2 = torch.empty_like(D)
    ops.gpt2_op_matmul(tA, K, 1, tB, K, 1, M, N, K, D2, N, aux=pre, ldaux=N, epilogue=ops.EPI_GELU_BWD,
                       path=ops.PATH_TC, flags_dev=fl)
    ref2 = O.gelu_backward(host(pre), acc)
    assert rel_l2(host(D2), ref2) < 2 ** -7
    check(host(D2), ref2, gelu_bwd_bound(ref2, acc, absprod, host(pre)), "acc * GELU'")
    F = dev(np.full((M, N), 0.25, np.float32))
    ops.gpt2_op_matmul(tA, K, 1, tB, K, 1, M, N, K, F, N, epilogue=ops.EPI_ACC_F32, path=ops.PATH_TC, flags_dev=fl)
    assert rel_l2(host(F), acc + 0.25) < 2e-5
    check(host(F), acc + 0.25, gemm_bound(acc + 0.25, absprod, bf16_out=False), "F += acc")
    assert fl.sum().item() == 0


def test_matmul_tc_weight_gradient_pattern(ops):
    """dW[N][K] += dY[BT][N]^T . X[BT][K]: both operands MN-major, long K."""
    BT, N, K = 4096, 384, 256
    dY, X = normal_array((BT, N), 150), normal_array((BT, K), 151)
    tdy, tx = dev(dY, torch.bfloat16), dev(X, torch.bfloat16)
    W0 = normal_array((N, K), 152)
    dW = dev(W0)
    fl = ops.flags()
    ops.gpt2_op_matmul(tdy, N, 0, tx, K, 0, N, K, BT, dW, K, epilogue=ops.EPI_ACC_F32, path=ops.PATH_TC,
                       flags_dev=fl)
    acc, absprod = gemm_ref(host(tdy), host(tx), 0, 0, N, K, BT)
    ref = W0 + acc
    assert rel_l2(host(dW), ref) < 2e-5
    check(host(dW), ref, gemm_bound(ref, absprod, bf16_out=False), "dW")
    assert fl.sum().item() == 0


@pytest.mark.parametrize("BT,N,K", [(16384, 768, 768), (8192, 2304, 768), (4096 + 192, 136, 264)])
def test_matmul_tc_split_k_weight_gradient(ops, BT, N, K):
    """Weight-gradient GEMM with a workspace: K = BT is split across CTAs,
    the partials are added in split order (bitwise repeatable), and the
    result matches the float64 product."""
    dY, X = normal_array((BT, N), 153), normal_array((BT, K), 154)
    tdy, tx = dev(dY, torch.bfloat16), dev(X, torch.bfloat16)
    W0 = normal_array((N, K), 155)
    fl = ops.flags()
    ws = ops.gemm_workspace(N, K, BT)
    if BT >= 8192:
        assert ws is not None  # these shapes leave SMs idle without a split
    outs = []
    for _ in range(2):
        dW = dev(W0)
        ops.gpt2_op_matmul(tdy, N, 0, tx, K, 0, N, K, BT, dW, K, epilogue=ops.EPI_ACC_F32, path=ops.PATH_TC,
                           flags_dev=fl, workspace=ws)
        outs.append(dW)
    torch.cuda.synchronize()
    assert fl.sum().item() == 0
    assert torch.equal(outs[0], outs[1])
    acc, absprod = gemm_ref(host(tdy), host(tx), 0, 0, N, K, BT)
    ref = W0.astype(np.float64) + acc
    assert rel_l2(host(outs[0]), ref) < 2e-5
    check(host(outs[0]), ref, gemm_bound(ref, absprod, bf16_out=False), "split-K dW")


@pytest.mark.parametrize("path", ["tc", "simt"])
@pytest.mark.parametrize("batch,BT,N,K,gap", [(3, 1024 + 64, 264, 136, 0), (12, 2048, 256, 512, 16),
                                              (2, 16384, 768, 768, 8)])
def test_matmul_batched_weight_gradient(ops, path, batch, BT, N, K, gap):
    """Batched weight gradients dW_z[N][K] += dY_z^T X_z (both operands
    MN-major) with items `gap` rows apart in their arrays (strided, as a
    model's per-layer tensors are): each item against the float64 product,
    bitwise repeatable."""
    if path == "simt" and BT * N * K * batch > 2e9:
        pytest.skip("SIMT reference path: small cases only")
    sY, sX, sW = (BT + gap) * N, (BT + gap) * K, (N + gap) * K
    dY = normal_array((batch * sY,), 156)
    X = normal_array((batch * sX,), 157)
    W0 = normal_array((batch * sW,), 158)
    tdy, tx = dev(dY, torch.bfloat16), dev(X, torch.bfloat16)
    fl = ops.flags()
    p = ops.PATH_TC if path == "tc" else ops.PATH_SIMT
    outs = []
    for _ in range(2):
        dW = dev(W0)
        ops.gpt2_op_matmul_batched(batch, tdy, N, sY, 0, tx, K, sX, 0, N, K, BT, dW, K, sW,
                                   epilogue=ops.EPI_ACC_F32, path=p, flags_dev=fl)
        outs.append(dW)
    torch.cuda.synchronize()
    assert fl.sum().item() == 0
    assert torch.equal(outs[0], outs[1])
    hy, hx, got = host(tdy), host(tx), host(outs[0])
    for z in range(batch):
        Y = hy[z * sY:z * sY + BT * N].reshape(BT, N).astype(np.float64)
        Xz = hx[z * sX:z * sX + BT * K].reshape(BT, K).astype(np.float64)
        ref = W0[z * sW:z * sW + N * K].reshape(N, K) + Y.T @ Xz
        assert rel_l2(got[z * sW:z * sW + N * K].reshape(N, K), ref) < 2e-5, z
        check(got[z * sW:z * sW + N * K].reshape(N, K), ref,
              gemm_bound(ref, np.abs(Y).T @ np.abs(Xz), bf16_out=False), f"item {z}")
        # the gap rows between items are untouched
        assert np.array_equal(got[z * sW + N * K:(z + 1) * sW], W0[z * sW + N * K:(z + 1) * sW])


@pytest.mark.parametrize("B,T,H,N", [(2, 512, 12, 640), (3, 128, 4, 256), (8, 2048, 5, 256)])
def test_matmul_rowdot_epilogue(ops, B, T, H, N):
    """Attention-projection input gradient whose epilogue also forms the
    attention backward's D[b][h][t] = sum over the head of dX * O (dX as
    stored in bf16), against numpy."""
    M, K = B * T, 64 * H
    dY, W, Oa = normal_array((M, N), 162), normal_array((N, K), 163, 0.05), normal_array((M, K), 164)
    tdy, tw, to = dev(dY, torch.bfloat16), dev(W, torch.bfloat16), dev(Oa, torch.bfloat16)
    dX = torch.full((M, K), float("nan"), device="cuda", dtype=torch.bfloat16)
    D = torch.full((B * H * T,), float("nan"), device="cuda")
    fl = ops.flags()
    ops.gpt2_op_matmul_rowdot(tdy, N, tw, K, M, N, K, dX, K, to, K, D, T, H, fl)
    torch.cuda.synchronize()
    assert fl.sum().item() == 0
    ref, absprod = gemm_ref(host(tdy), host(tw), 1, 0, M, K, N)
    assert rel_l2(host(dX), ref) < 2 ** -7
    check(host(dX), ref, gemm_bound(ref, absprod), "dX")
    x = host(dX).astype(np.float64).reshape(B, T, H, 64)
    o = host(to).astype(np.float64).reshape(B, T, H, 64)
    rD = (x * o).sum(-1).transpose(0, 2, 1)
    assert np.max(np.abs(host(D).reshape(B, H, T) - rD)) < 1e-4 * max(1.0, np.abs(rD).max())
    # D from the stored dX: an fp32 sum of 64 products per head
    check(host(D).reshape(B, H, T), rD, 2.0 ** -20 * np.abs(x * o).sum(-1).transpose(0, 2, 1), "D")


@pytest.mark.parametrize("M,N,K,gelu", [(384, 2304, 768, False), (256 + 136, 3072, 768, True), (200, 136, 64, False)])
def test_matmul_layernorm_folded(ops, M, N, K, gelu):
    """LayerNorm folded into the next product: the weight fold (W gamma in
    bf16, the column sums s and c) and the product on the LayerNorm's input
    with the normalisation in the epilogue, against the oracle's LayerNorm
    followed by the oracle's matmul (and GELU), element by element.  Rows
    with a large common offset check the mean term's cancellation."""
    r = normal_array((M, K), 180, 1.0) + normal_array((M, 1), 181, 3.0)
    gamma, beta = normal_array((K,), 182, 0.2) + 1, normal_array((K,), 183, 0.1)
    W, b = normal_array((N, K), 184, 0.02), normal_array((N,), 185, 0.1)
    tr = dev(r, torch.bfloat16)
    rs_ = host(tr)
    y_ln = torch.empty(M, K, device="cuda", dtype=torch.bfloat16)
    mean, rstd = torch.empty(M, device="cuda"), torch.empty(M, device="cuda")
    ops.gpt2_op_residual_layernorm_forward(None, y_ln, mean, rstd, tr, None, dev(gamma, torch.bfloat16),
                                           dev(beta, torch.bfloat16), M, K)
    Wf = torch.empty(N, K, device="cuda", dtype=torch.bfloat16)
    sv, cv = torch.empty(N, device="cuda"), torch.empty(N, device="cuda")
    ops.gpt2_op_lnfold_weights(Wf, sv, cv, dev(W), dev(gamma), dev(beta), dev(b), 1, N, K)
    # the fold against its definition (bf16 product, sums of the stored values)
    wf = host(Wf)
    assert np.array_equal(wf.astype(np.float32), host(dev(W * gamma[None, :], torch.bfloat16)).astype(np.float32))
    assert np.allclose(host(sv), wf.sum(1), rtol=1e-5, atol=1e-5)
    assert np.allclose(host(cv), b + W.astype(np.float64) @ beta, rtol=1e-5, atol=1e-6)
    D = torch.full((M, N), float("nan"), device="cuda", dtype=torch.bfloat16)
    pre = torch.empty(M, N, device="cuda", dtype=torch.bfloat16) if gelu else None
    fl = ops.flags()
    ops.gpt2_op_matmul_lnfold(tr, K, mean, rstd, Wf, K, sv, cv, M, N, K, D, N, aux=pre, ldaux=N if gelu else 0,
                              flags_dev=fl)
    torch.cuda.synchronize()
    assert fl.sum().item() == 0
    y, _, _ = O.layernorm_forward(rs_, gamma.astype(np.float64), beta.astype(np.float64))
    ref = O.matmul_forward(y, W.astype(np.float64), b.astype(np.float64))
    # output rounding; the bf16 weight fold (2^-8 of sum |xhat gamma W|); fp32
    # accumulation over the raw rows and the mean term (ACC of their magnitudes)
    xhat = (rs_ - rs_.mean(1, keepdims=True)) / np.sqrt(rs_.var(1, keepdims=True) + 1e-5)
    fold_scale = np.abs(xhat) @ np.abs(W * gamma[None, :]).T
    raw = (np.abs(rs_) @ np.abs(wf).T + np.abs(rs_.mean(1, keepdims=True)) * np.abs(wf).sum(1)[None, :]) / \
        np.sqrt(rs_.var(1, keepdims=True) + 1e-5)
    bound = U8 * np.abs(ref) + 2 * U8 * fold_scale + 2 ** -16 * raw
    if not gelu:
        check(host(D), ref, bound, "folded product")
    else:
        check(host(pre), ref, bound, "folded pre-activation")
        g_ref = O.gelu_forward(host(pre))
        check(host(D), g_ref, gelu_bound(g_ref, host(pre)), "GELU of the folded pre-activation")


@pytest.mark.parametrize("epi", ["store", "gelu_bwd"])
def test_matmul_batched_bf16_epilogues(ops, epi):
    """Batched K-major products with bf16 output (and the GELU' epilogue with a
    strided aux), the shape of per-layer input gradients."""
    batch, M, N, K = 3, 1000, 384, 200
    A, B = normal_array((batch, M, K), 159), normal_array((batch, N, K), 160)
    tA, tB = dev(A, torch.bfloat16), dev(B, torch.bfloat16)
    D = torch.full((batch, M, N), float("nan"), device="cuda", dtype=torch.bfloat16)
    fl = ops.flags()
    if epi == "store":
        ops.gpt2_op_matmul_batched(batch, tA, K, M * K, 1, tB, K, N * K, 1, M, N, K, D, N, M * N, path=ops.PATH_TC,
                                   flags_dev=fl)
    else:
        pre = dev(normal_array((batch, M, N), 161), torch.bfloat16)
        ops.gpt2_op_matmul_batched(batch, tA, K, M * K, 1, tB, K, N * K, 1, M, N, K, D, N, M * N, aux=pre, ldaux=N,
                                   sAux=M * N, epilogue=ops.EPI_GELU_BWD, path=ops.PATH_TC, flags_dev=fl)
    assert fl.sum().item() == 0
    hA, hB, got = host(tA), host(tB), host(D)
    for z in range(batch):
        acc, absprod = gemm_ref(hA[z], hB[z], 1, 1, M, N, K)
        ref = acc if epi == "store" else O.gelu_backward(host(pre)[z], acc)
        assert rel_l2(got[z], ref) < 2 ** -7, z
        bound = gemm_bound(ref, absprod) if epi == "store" else gelu_bwd_bound(ref, acc, absprod, host(pre)[z])
        check(got[z], ref, bound, f"item {z}")


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dt", ["fp32", "bf16"])
@pytest.mark.parametrize("B,T,C,H", [(2, 13, 64, 4), (1, 70, 128, 2), (2, 129, 192, 3)])
def test_attention_forward_backward(ops, dt, B, T, C, H):
    qkv = normal_array((B, T, 3 * C), 50)
    dout = normal_array((B, T, C), 51)
    tq, tdo = dev(qkv, DT[dt]), dev(dout, DT[dt])
    qs, dos = host(tq), host(tdo)
    out = torch.empty(B * T, C, device="cuda", dtype=DT[dt])
    lse = torch.empty(B * H * T, device="cuda")
    ops.gpt2_op_attention_forward(out, lse, tq, B, T, C, H, path=ops.PATH_SIMT)
    ro, att = O.attention_forward(qs, H)
    tol = 1e-5 if dt == "fp32" else 2 ** -7
    assert rel_l2(host(out).reshape(B, T, C), ro) < tol
    # LSE: log of the softmax normaliser of the scaled scores
    hd = C // H
    q = qs[..., :C].reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    k = qs[..., C:2 * C].reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    s = q @ k.transpose(0, 1, 3, 2) / math.sqrt(hd)
    s[..., np.triu(np.ones((T, T), bool), 1)] = -np.inf
    mx = s.max(-1)
    rlse = mx + np.log(np.exp(s - mx[..., None]).sum(-1))
    assert np.max(np.abs(host(lse).reshape(B, H, T) - rlse)) < (1e-5 if dt == "fp32" else 1e-3)
    dq = torch.empty(B * T, 3 * C, device="cuda", dtype=DT[dt])
    ops.gpt2_op_attention_backward(dq, tdo, tq, out, lse, B, T, C, H, path=ops.PATH_SIMT)
    # the oracle's backward from the kernel's stored output's inputs
    rd = O.attention_backward(dos, qs, att, H)
    tolb = 1e-4 if dt == "fp32" else 2e-2
    for part in range(3):
        a = host(dq).reshape(B, T, 3 * C)[..., part * C:(part + 1) * C]
        r = rd[..., part * C:(part + 1) * C]
        assert rel_l2(a, r) < tolb, part


def _attention_tc(ops, qkv, dout, B, T, C, H):
    """Run the tensor-core attention forward + backward; returns device tensors."""
    tq, tdo = dev(qkv, torch.bfloat16), dev(dout, torch.bfloat16)
    out = torch.empty(B * T, C, device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(B * H * T, device="cuda")
    dq = torch.empty(B * T, 3 * C, device="cuda", dtype=torch.bfloat16)
    sc = torch.empty(ops.lib.gpt2_op_attention_backward_scratch_bytes(B, T, H), device="cuda", dtype=torch.uint8)
    D = sc[:B * H * T * 4].view(torch.float32)  # D leads the scratch
    fl = ops.flags()
    ops.gpt2_op_attention_forward(out, lse, tq, B, T, C, H, path=ops.PATH_TC, flags_dev=fl)
    ops.gpt2_op_attention_backward(dq, tdo, tq, out, lse, B, T, C, H, path=ops.PATH_TC, flags_dev=fl, scratch=sc)
    torch.cuda.synchronize()
    assert fl.sum().item() == 0
    return tq, tdo, out, lse, dq, D


# LSE of the tensor-core forward: the row sum comes from the tensor core over
# the bf16-rounded probabilities (each within 2^-8 of its value) computed by
# exp2 approximations (relative error below 2^-13), so log of the sum is
# within 2^-8 + 2^-13 of the exact log-sum-exp
LSE_TOL = 2.0 ** -8 + 2.0 ** -13


def _lse_ref(qs, B, T, C, H):
    hd = C // H
    q = qs[..., :C].reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    k = qs[..., C:2 * C].reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    s = q @ k.transpose(0, 1, 3, 2) / math.sqrt(hd)
    s[..., np.triu(np.ones((T, T), bool), 1)] = -np.inf
    mx = s.max(-1)
    return mx + np.log(np.exp(s - mx[..., None]).sum(-1))


@pytest.mark.parametrize("B,T,C,H,sigma", [(1, 128, 64, 1, 1.0), (2, 256, 128, 2, 1.0), (1, 384, 192, 3, 2.0),
                                           (2, 640, 128, 2, 3.0), (1, 1024, 64, 1, 1.0)])
def test_attention_tc_against_oracle(ops, B, T, C, H, sigma):
    """tcgen05 flash attention (head size 64): one and two query tiles per
    CTA (odd tile counts leave a lone tile), several key tiles per row with
    online rescaling, score scales up to sigma^2 * 8."""
    qkv = normal_array((B, T, 3 * C), 70, sigma)
    dout = normal_array((B, T, C), 71)
    tq, tdo, out, lse, dq, D = _attention_tc(ops, qkv, dout, B, T, C, H)
    qs, dos = host(tq), host(tdo)
    ro, att = O.attention_forward(qs, H)
    assert rel_l2(host(out).reshape(B, T, C), ro) < 2 ** -7
    assert np.max(np.abs(host(lse).reshape(B, H, T) - _lse_ref(qs, B, T, C, H))) < LSE_TOL
    # D = rowsum(dO * O) of the kernel's own (stored) output
    o = host(out).reshape(B, T, H, C // H)
    rD = (dos.reshape(B, T, H, C // H) * o).sum(-1).transpose(0, 2, 1)
    assert np.max(np.abs(host(D).reshape(B, H, T) - rD)) < 1e-3 * max(1.0, np.abs(rD).max())
    rd = O.attention_backward(dos, qs, att, H)
    for part in range(3):
        a = host(dq).reshape(B, T, 3 * C)[..., part * C:(part + 1) * C]
        assert rel_l2(a, rd[..., part * C:(part + 1) * C]) < 2e-2, part
    _check_attention_elementwise(qs, dos, host(out).reshape(B, T, C), host(dq).reshape(B, T, 3 * C), H)


@pytest.mark.parametrize("growth", [1.25, 1.8])
def test_attention_tc_growing_scores(ops, growth):
    """Keys scaled by growth^(key tile): the scores of each later key tile run
    further above the earlier ones, so rows keep moving their softmax
    reference after the first tile (growth 1.8: about half the rows of a
    tile, 1.25: a few rows of some warps and none of others), through the path that
    redoes a tile's probabilities and rescales the accumulator.  Element-wise
    against the oracle."""
    B, T, C, H = 2, 1024, 128, 2
    qkv = normal_array((B, T, 3 * C), 78)
    scale = growth ** (np.arange(T) // 128)
    qkv[:, :, C:2 * C] *= scale[None, :, None].astype(np.float32)
    dout = normal_array((B, T, C), 79)
    tq, tdo, out, lse, dq, D = _attention_tc(ops, qkv, dout, B, T, C, H)
    qs, dos = host(tq), host(tdo)
    assert np.max(np.abs(host(lse).reshape(B, H, T) - _lse_ref(qs, B, T, C, H))) < LSE_TOL
    _check_attention_elementwise(qs, dos, host(out).reshape(B, T, C), host(dq).reshape(B, T, 3 * C), H)


def _check_attention_elementwise(qs, dos, o, dqkv, H):
    """O, dQ, dK, dV of the tensor-core kernels element by element against the
    float64 oracle, within the bounds of tests/parity.py."""
    C = qs.shape[-1] // 3
    bd = attention_bounds(qs, dos, o, H)
    check(o, *bd["out"], "O")
    for part, name in enumerate(("dq", "dk", "dv")):
        check(dqkv[..., part * C:(part + 1) * C], *bd[name], name)


def test_attention_tc_deterministic(ops):
    """No atomics anywhere: two backward runs give identical bits."""
    B, T, C, H = 2, 512, 128, 2
    qkv, dout = normal_array((B, T, 3 * C), 72), normal_array((B, T, C), 73)
    r1 = _attention_tc(ops, qkv, dout, B, T, C, H)
    r2 = _attention_tc(ops, qkv, dout, B, T, C, H)
    assert torch.equal(r1[2], r2[2]) and torch.equal(r1[3], r2[3]) and torch.equal(r1[4], r2[4])


def test_attention_tc_full_size_sampled_heads(ops):
    """GPT-2 124M attention shape (B=16, T=1024, C=768, H=12), as the model
    step launches it; the oracle checks sampled (batch, head) pairs."""
    B, T, C, H = 16, 1024, 768, 12
    hd = C // H
    qkv = normal_array((B, T, 3 * C), 74)
    dout = normal_array((B, T, C), 75)
    tq, tdo, out, lse, dq, D = _attention_tc(ops, qkv, dout, B, T, C, H)
    qs, dos = host(tq), host(tdo)
    o_all, dq_all, lse_all = host(out).reshape(B, T, C), host(dq).reshape(B, T, 3 * C), host(lse).reshape(B, H, T)
    for b, h in [(0, 0), (5, 7), (11, 3), (15, 11)]:
        cols = [slice(p * C + h * hd, p * C + (h + 1) * hd) for p in range(3)]
        sq = np.concatenate([qs[b:b + 1, :, c] for c in cols], -1)
        ro, att = O.attention_forward(sq, 1)
        assert rel_l2(o_all[b:b + 1, :, h * hd:(h + 1) * hd], ro) < 2 ** -7, (b, h)
        assert np.max(np.abs(lse_all[b, h] - _lse_ref(sq, 1, T, hd, 1)[0, 0])) < LSE_TOL
        rd = O.attention_backward(dos[b:b + 1, :, h * hd:(h + 1) * hd], sq, att, 1)
        for p in range(3):
            assert rel_l2(dq_all[b:b + 1, :, cols[p]], rd[..., p * hd:(p + 1) * hd]) < 2e-2, (b, h, p)
        _check_attention_elementwise(sq, dos[b:b + 1, :, h * hd:(h + 1) * hd], o_all[b:b + 1, :, h * hd:(h + 1) * hd],
                                     np.concatenate([dq_all[b:b + 1, :, c] for c in cols], -1), 1)


@pytest.mark.parametrize("B,T", [(8, 2048), (4, 4096)])
def test_attention_tc_long_context(ops, B, T):
    """Long sequences at the 124M head layout (C=768, H=12) with the token
    count of the per-kernel sweep (B*T = 16384): many key tiles per query
    row, the online rescaling over up to 32 tiles, and the dS block buffer of
    a 32-tile triangle.  Sampled (batch, head) pairs against the oracle,
    element by element."""
    C, H = 768, 12
    hd = C // H
    qkv = normal_array((B, T, 3 * C), 76)
    dout = normal_array((B, T, C), 77)
    tq, tdo, out, lse, dq, D = _attention_tc(ops, qkv, dout, B, T, C, H)
    qs, dos = host(tq), host(tdo)
    o_all, dq_all, lse_all = host(out).reshape(B, T, C), host(dq).reshape(B, T, 3 * C), host(lse).reshape(B, H, T)
    for b, h in [(0, 0), (B - 1, 7)]:
        cols = [slice(p * C + h * hd, p * C + (h + 1) * hd) for p in range(3)]
        sq = np.concatenate([qs[b:b + 1, :, c] for c in cols], -1)
        assert np.max(np.abs(lse_all[b, h] - _lse_ref(sq, 1, T, hd, 1)[0, 0])) < LSE_TOL
        _check_attention_elementwise(sq, dos[b:b + 1, :, h * hd:(h + 1) * hd], o_all[b:b + 1, :, h * hd:(h + 1) * hd],
                                     np.concatenate([dq_all[b:b + 1, :, c] for c in cols], -1), 1)


def test_attention_tc_path_rejects_unsupported(ops):
    """path=2 (tensor cores only) refuses shapes the kernels do not handle."""
    B, T, C, H = 1, 100, 128, 2  # T not a multiple of 128
    tq = torch.zeros(B * T, 3 * C, device="cuda", dtype=torch.bfloat16)
    out = torch.empty(B * T, C, device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(B * H * T, device="cuda")
    with pytest.raises(Exception):
        ops.gpt2_op_attention_forward(out, lse, tq, B, T, C, H, path=ops.PATH_TC, flags_dev=ops.flags())


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dt", ["fp32", "bf16"])
@pytest.mark.parametrize("rows,V,Vp", [(3, 512, 512), (17, 1000, 1024), (4, 50257, 50304)])
def test_softmax_crossentropy(ops, dt, rows, V, Vp):
    z = normal_array((rows, Vp), 60, 3.0)
    z[:, V:] = 1e4 if dt == "fp32" else 100.0  # pads must not count
    tgt = np.random.default_rng(61).integers(0, V, size=rows).astype(np.int32)
    tz = dev(z, DT[dt])
    zs = host(tz)
    losses = torch.empty(rows, device="cuda")
    fl = ops.flags()
    dloss = 1.0 / rows
    ops.gpt2_op_softmax_crossentropy(tz, losses, dev(tgt, torch.int32), rows, V, Vp, dloss, 1, fl)
    rl = O.crossentropy_forward(zs[None], tgt[None], V)[0]
    assert np.max(np.abs(host(losses) - rl)) < 1e-4
    rd = O.crossentropy_softmax_backward(O.softmax_forward(zs[None], V), tgt[None], np.full((1, rows), dloss))[0]
    got = host(tz)
    assert np.all(got[:, V:] == 0)
    if dt == "fp32":
        assert np.max(np.abs(got - rd)) < 1e-7
    else:
        assert np.max(np.abs(got - rd)) < 2 ** -8 * dloss
    assert fl.sum().item() == 0


@pytest.mark.parametrize("write_grad", [1, 0])
def test_softmax_crossentropy_many_rows(ops, write_grad):
    """GPT-2 vocabulary with more rows than two per SM: the persistent bf16
    kernel's double-buffered row pipeline, a ragged last CTA, one target at
    the last real column; write_grad=0 leaves the logits untouched."""
    rows, V, Vp = 400, 50257, 50304
    z = normal_array((rows, Vp), 63, 3.0)
    z[:, V:] = 100.0
    tgt = np.random.default_rng(64).integers(0, V, size=rows).astype(np.int32)
    tgt[7] = V - 1
    tz = dev(z, torch.bfloat16)
    zs = host(tz)
    losses = torch.empty(rows, device="cuda")
    fl = ops.flags()
    dloss = 1.0 / rows
    ops.gpt2_op_softmax_crossentropy(tz, losses, dev(tgt, torch.int32), rows, V, Vp, dloss, write_grad, fl)
    assert fl.sum().item() == 0
    rl = O.crossentropy_forward(zs[None], tgt[None], V)[0]
    assert np.max(np.abs(host(losses) - rl)) < 1e-4
    got = host(tz)
    if not write_grad:
        assert np.array_equal(got, zs)
        return
    rd = O.crossentropy_softmax_backward(O.softmax_forward(zs[None], V), tgt[None], np.full((1, rows), dloss))[0]
    assert np.all(got[:, V:] == 0)
    assert np.max(np.abs(got - rd)) < 2 ** -8 * dloss


@pytest.mark.parametrize("rows,V,Vp,K", [(300, 50257, 50304, 64), (130, 700, 1024, 128), (257, 700, 768, 64)])
def test_classifier_logit_stats_and_softmax(ops, rows, V, Vp, K):
    """The classifier's fused form: logits by the tensor-core product with each
    row's (max, sum of exp) per column tile taken in its epilogue from the
    stored bf16 values, then softmax/CE from those statistics (one read of each
    row), against numpy on the stored logits.  (130, 700, 1024): a last tile
    with no column below V; (257, 700, 768): a tile cut by V."""
    A, B = normal_array((rows, K), 170), normal_array((Vp, K), 171, 0.3)
    tA, tB = dev(A, torch.bfloat16), dev(B, torch.bfloat16)
    D = torch.empty(rows, Vp, device="cuda", dtype=torch.bfloat16)
    tiles = ops.gpt2_op_logit_stats_tiles(Vp)
    width = 256 if Vp >= 512 else 128
    assert tiles == -(-Vp // width)
    stats = torch.full((rows, tiles, 2), float("nan"), device="cuda")
    fl = ops.flags()
    ops.gpt2_op_matmul_logit_stats(tA, K, tB, K, rows, Vp, K, D, Vp, stats, V, fl)
    torch.cuda.synchronize()
    assert fl.sum().item() == 0
    zs = host(D)
    assert rel_l2(zs, host(tA) @ host(tB).T) < 2 ** -7
    ref, absprod = gemm_ref(host(tA), host(tB), 1, 1, rows, Vp, K)
    check(zs, ref, gemm_bound(ref, absprod), "logits")
    z = zs.astype(np.float64)
    st = host(stats)
    for n in range(tiles):
        c0, c1 = n * width, min((n + 1) * width, V)
        if c1 <= c0:
            assert np.all(st[:, n, 0] == -np.inf) and np.all(st[:, n, 1] == 0)
            continue
        m = z[:, c0:c1].max(axis=1)
        assert np.array_equal(st[:, n, 0], m.astype(np.float32))  # the max of stored values is exact
        sref = np.exp(z[:, c0:c1] - m[:, None]).sum(axis=1)
        assert np.max(np.abs(st[:, n, 1] / sref - 1)) < 1e-5
    tgt = np.random.default_rng(172).integers(0, V, size=rows).astype(np.int32)
    tgt[0] = V - 1
    losses = torch.empty(rows, device="cuda")
    dloss = 1.0 / rows
    ops.gpt2_op_softmax_crossentropy_stats(D, losses, dev(tgt, torch.int32), stats, rows, V, Vp, dloss, fl)
    torch.cuda.synchronize()
    assert fl.sum().item() == 0
    rl = O.crossentropy_forward(zs[None], tgt[None], V)[0]
    assert np.max(np.abs(host(losses) - rl)) < 1e-4
    rd = O.crossentropy_softmax_backward(O.softmax_forward(zs[None], V), tgt[None], np.full((1, rows), dloss))[0]
    got = host(D)
    assert np.all(got[:, V:] == 0)
    assert np.max(np.abs(got - rd)) < 2 ** -8 * dloss


def test_softmax_crossentropy_flags_bad_target_large_vocab(ops):
    z = dev(normal_array((3, 50304), 65), torch.bfloat16)
    fl = ops.flags()
    ops.gpt2_op_softmax_crossentropy(z, torch.empty(3, device="cuda"), dev(np.array([1, 50257, 5], np.int32), torch.int32),
                                     3, 50257, 50304, 0.5, 1, fl)
    assert fl[0].item() & 2


def test_softmax_crossentropy_flags_bad_target(ops):
    z = dev(normal_array((2, 64), 62))
    fl = ops.flags()
    ops.gpt2_op_softmax_crossentropy(z, torch.empty(2, device="cuda"), dev(np.array([1, 64], np.int32), torch.int32),
                                     2, 64, 64, 0.5, 0, fl)
    assert fl[0].item() & 2


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("t", [1, 2, 7])
def test_adamw(ops, t):
    n = 4 * 1001
    p, g = normal_array((n,), 70), normal_array((n,), 71, 1e-2)
    m, v = normal_array((n,), 72, 1e-3), np.abs(normal_array((n,), 73, 1e-4))
    tp, tg, tm, tv = dev(p), dev(g), dev(m), dev(v)
    pb = torch.empty(n, device="cuda", dtype=torch.bfloat16)
    ops.gpt2_op_adamw(tp, tg, tm, tv, pb, 6e-4, 0.9, 0.95, 1e-8, 0.1, t)
    rp, rm, rv = p.astype(np.float64), m.astype(np.float64), v.astype(np.float64)
    O.adamw_update(rp, g.astype(np.float64), rm, rv, 6e-4, 0.9, 0.95, 1e-8, 0.1, t)
    assert rel_l2(host(tm), rm) < 1e-6 and rel_l2(host(tv), rv) < 1e-6
    assert np.max(np.abs(host(tp) - rp)) < 1e-6
    assert torch.equal(pb, tp.to(torch.bfloat16))


@pytest.mark.parametrize("n", [5, 4 * 1001 + 3, 124475904])
def test_grad_norm_and_clip_factor(ops, n):
    """Global norm against a float64 sum; clip factor min(1, max/(norm+1e-6));
    bitwise repeatable (fixed chunks, fixed order).  n = 124475904 is the 124M
    parameter count."""
    g = normal_array((n,), 80, 1e-3) if n < 10**7 else None
    tg = dev(g) if g is not None else torch.randn(n, device="cuda", generator=torch.Generator("cuda").manual_seed(5)) * 1e-3
    ref = float(np.sqrt(np.sum(host(tg) ** 2)))
    for max_norm in (ref / 4, ref * 4):
        out = torch.zeros(2, device="cuda")
        ops.gpt2_op_grad_norm(tg, max_norm, out)
        out2 = torch.zeros(2, device="cuda")
        ops.gpt2_op_grad_norm(tg, max_norm, out2)
        assert torch.equal(out, out2)
        norm, scale = out.tolist()
        assert abs(norm - ref) <= 1e-5 * ref
        assert abs(scale - min(1.0, max_norm / (ref + 1e-6))) <= 2e-6


def test_adamw_with_clip_factor(ops):
    n = 4 * 1001
    p, g = normal_array((n,), 81), normal_array((n,), 82, 1e-2)
    m, v = normal_array((n,), 83, 1e-3), np.abs(normal_array((n,), 84, 1e-4))
    tp, tg, tm, tv = dev(p), dev(g), dev(m), dev(v)
    scale = torch.tensor([0.37], device="cuda")
    ops.gpt2_op_adamw(tp, tg, tm, tv, None, 6e-4, 0.9, 0.95, 1e-8, 0.1, 3, gscale=scale)
    rp, rm, rv = p.astype(np.float64), m.astype(np.float64), v.astype(np.float64)
    O.adamw_update(rp, g.astype(np.float64) * np.float64(np.float32(0.37)), rm, rv, 6e-4, 0.9, 0.95, 1e-8, 0.1, 3)
    assert rel_l2(host(tm), rm) < 1e-6 and rel_l2(host(tv), rv) < 1e-6
    assert np.max(np.abs(host(tp) - rp)) < 1e-6


# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dt", ["fp32", "bf16"])
def test_gelu_standalone(ops, dt):
    # fp32: 1 + tanh(u) cancels for negative x, so the bound is absolute
    # (a few ulp of |x|); bf16: one rounding of the stored output.
    x = normal_array((4096 + 8,), 80, 2.0)
    d = normal_array((4096 + 8,), 81)
    tx, td = dev(x, DT[dt]), dev(d, DT[dt])
    out = torch.empty_like(tx)
    ops.gpt2_op_gelu_forward(out, tx)
    ref = O.gelu_forward(host(tx))
    bound = 2e-6 * np.maximum(1, np.abs(host(tx))) if dt == "fp32" else 2 ** -8 * np.abs(ref) + 1e-6
    assert np.all(np.abs(host(out) - ref) <= bound)
    dinp = torch.empty_like(tx)
    ops.gpt2_op_gelu_backward(dinp, tx, td)
    ref = O.gelu_backward(host(tx), host(td))
    bound = 4e-6 * np.maximum(1, np.abs(host(tx))) * np.abs(host(td)) + 1e-7 if dt == "fp32" \
        else 2 ** -8 * np.abs(ref) + 1e-5 * np.abs(host(td))
    assert np.all(np.abs(host(dinp) - ref) <= bound)


@pytest.mark.parametrize("dt", ["fp32", "bf16"])
@pytest.mark.parametrize("rows,cols,ldx", [(300, 200, 208), (16384, 2304, 2304)])
def test_colsum(ops, dt, rows, cols, ldx):
    X = normal_array((rows, ldx), 90)
    tX = dev(X, DT[dt])
    out = dev(np.ones(cols, np.float32))
    ops.gpt2_op_colsum(out, tX, rows, cols, ldx)
    assert rel_l2(host(out), host(tX)[:, :cols].sum(0) + 1) < 1e-5


# ---------------------------------------------------------------------------
def test_bounded_wait_times_out_and_device_recovers(ops):
    """The tensor-core kernels' failure path, run on purpose: a CTA holding
    tensor memory waits on an mbarrier nothing signals; the wait gives up
    after the 5 ms limit, the CTA frees its tensor memory and sets the timeout
    flag, and the call reports GPT2_ERR_TIMEOUT.  A tensor-core GEMM right
    after it on the same device gives the right result."""
    import time
    fl = ops.flags()
    t0 = time.perf_counter()
    rc = ops.gpt2_op_wait_probe(5000, fl)
    dt = time.perf_counter() - t0
    assert rc == -8
    assert fl[0].item() & 4
    assert 0.004 < dt < 5.0
    M, N, K = 256, 256, 128
    A, B = normal_array((M, K), 190), normal_array((N, K), 191)
    tA, tB = dev(A, torch.bfloat16), dev(B, torch.bfloat16)
    D = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    fl2 = ops.flags()
    ops.gpt2_op_matmul(tA, K, 1, tB, K, 1, M, N, K, D, N, path=ops.PATH_TC, flags_dev=fl2)
    torch.cuda.synchronize()
    assert fl2.sum().item() == 0
    ref, absprod = gemm_ref(host(tA), host(tB), 1, 1, M, N, K)
    check(host(D), ref, gemm_bound(ref, absprod), "D after the timeout")
