"""GPU parity: the CUDA path (called through the C ABI) against the fp64 CPU oracle on the
same seeded inputs.  Small cases span several tiles and ragged tails in M, N and K; the
full-size workloads are checked on sampled rows/columns that the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

import datagen as D
import oracle as O
from parity import assert_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def ops():
    from dora_adapter_linear_gb300.build import build
    build()
    from dora_adapter_linear_gb300 import ops as _ops
    return _ops


def gpu(t):
    return None if t is None else t.to(DEV).contiguous()


def f64(t):
    return None if t is None else to64(t)


def lin_inputs(name, **kw):
    case = D.scaled(D.WORKLOADS[name], **kw)
    t = D.make_linear(case)
    return case, t, {k: gpu(v) for k, v in t.items()}


# ---------------------------------------------------------------------------- infrastructure
def test_bounded_wait_reports_timeout(ops):
    from dora_adapter_linear_gb300 import _lib as L
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    assert L.lora_check_device_error(ws) == 0
    L.lora_debug_wait_timeout(ws, 2000)  # 2 ms limit on a barrier nothing arrives on
    assert L.lora_check_device_error(ws) == 6
    L.lora_clear_device_error(ws)
    assert L.lora_check_device_error(ws) == 0


# ---------------------------------------------------------------------------- LoRA, bf16
SMALL = dict(M=300, d_in=328, d_out=264)


def test_base_gemm_kmajor_strength0(ops):
    case, t, g = lin_inputs("lora_4096_bf16", **SMALL, r=16)
    Y, _ = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], 0.0, save_z=False)
    ref = O.lora_linear_fwd(f64(t["X"]), f64(t["W0"]), f64(t["A"]), f64(t["B"]), 0.0)
    assert_close(Y, ref, "bf16", "X W0^T")


def test_base_gemm_mnmajor_strength0(ops):
    case, t, g = lin_inputs("lora_4096_bf16", **SMALL, r=16)
    dX, dA, dB, _ = ops.lora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], None, g["dY"], 0.0)
    assert_close(dX, f64(t["dY"]) @ f64(t["W0"]), "bf16", "dY W0")
    assert not dA.any() and not dB.any()


@pytest.mark.parametrize("r", [8, 16, 24, 32, 64, 96, 128])
@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("fused_z", ["1", "0"])
def test_lora_fwd_bf16(ops, r, bias, fused_z, monkeypatch):
    """fused_z 1: Z formed inside the GEMM (ranks 8-32, opt-in); 0: the separate down-projection pass."""
    monkeypatch.setenv("LORA_GB300_FUSED_Z", fused_z)
    case, t, g = lin_inputs("lora_4096_bf16", **SMALL, r=r, bias=bias)
    Y, Z = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], case.s, g["bias"])
    X, W0, A, B = (f64(t[k]) for k in ("X", "W0", "A", "B"))
    assert_close(Y, O.lora_linear_fwd(X, W0, A, B, case.s, f64(t["bias"])), "bf16", "Y")
    assert_close(Z, X @ A.T, "bf16", "Z")


@pytest.mark.parametrize("r", [8, 16, 32, 64, 96, 128])
def test_lora_bwd_bf16(ops, r):
    case, t, g = lin_inputs("lora_4096_bf16", **SMALL, r=r)
    _, Z = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], case.s)
    dX, dA, dB, dbias = ops.lora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], Z, g["dY"], case.s, need_dbias=True)
    rX, rA, rB, rb = O.lora_linear_bwd(*(f64(t[k]) for k in ("X", "W0", "A", "B")), case.s, f64(t["dY"]))
    assert_close(dX, rX, "bf16", "dX")
    assert_close(dA, rA, "bf16", "dA")
    assert_close(dB, rB, "bf16", "dB")
    assert_close(dbias, rb[None, :], "bf16", "dbias")


@pytest.mark.parametrize("r", [8, 16, 24, 32])
def test_lora_bwd_one_dy_pass_grid(ops, r):
    """dY side in one pass at a size whose CTA grid has several 64-row blocks per CTA and
    several 512-column groups, with a ragged last row block and a ragged last column chunk."""
    case, t, g = lin_inputs("lora_4096_bf16", M=13000, d_in=136, d_out=1096, r=r)
    _, Z = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], case.s)
    dX, dA, dB, dbias = ops.lora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], Z, g["dY"], case.s, need_dbias=True)
    rX, rA, rB, rb = O.lora_linear_bwd(*(f64(t[k]) for k in ("X", "W0", "A", "B")), case.s, f64(t["dY"]))
    assert_close(dX, rX, "bf16", "dX")
    assert_close(dA, rA, "bf16", "dA")
    assert_close(dB, rB, "bf16", "dB")
    assert_close(dbias, rb[None, :], "bf16", "dbias")


def test_lora_bwd_recomputes_z(ops):
    case, t, g = lin_inputs("lora_4096_bf16", **SMALL, r=16)
    dX, dA, dB, _ = ops.lora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], None, g["dY"], case.s)
    rX, rA, rB, _ = O.lora_linear_bwd(*(f64(t[k]) for k in ("X", "W0", "A", "B")), case.s, f64(t["dY"]))
    assert_close(dA, rA, "bf16", "dA")
    assert_close(dB, rB, "bf16", "dB")


def test_lora_strength0_bit_exact_vs_zero_adapter(ops):
    """Strength 0 takes the base-only path; a zero up-projection takes the fused path: same bits."""
    case, t, g = lin_inputs("lora_4096_bf16", **SMALL, r=16)
    Y0, _ = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], 0.0)
    Yb, _ = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], torch.zeros_like(g["B"]), case.s)
    assert torch.equal(Y0, Yb)


@pytest.mark.parametrize("M", [1, 127, 129])
def test_lora_ragged_m(ops, M):
    case, t, g = lin_inputs("lora_4096_bf16", M=M, d_in=136, d_out=520, r=16, bias=True)
    Y, Z = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], case.s, g["bias"])
    X, W0, A, B = (f64(t[k]) for k in ("X", "W0", "A", "B"))
    assert_close(Y, O.lora_linear_fwd(X, W0, A, B, case.s, f64(t["bias"])), "bf16", "Y")
    dX, dA, dB, _ = ops.lora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], Z, g["dY"], case.s)
    rX, rA, rB, _ = O.lora_linear_bwd(X, W0, A, B, case.s, f64(t["dY"]))
    assert_close(dX, rX, "bf16", "dX")
    assert_close(dA, rA, "bf16", "dA")
    assert_close(dB, rB, "bf16", "dB")


def test_m_zero_is_noop(ops):
    case, t, g = lin_inputs("lora_4096_bf16", M=0, d_in=64, d_out=64, r=8)
    Y, Z = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], case.s)
    assert Y.shape == (0, 64)
    dX, dA, dB, _ = ops.lora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], Z, g["dY"], case.s)
    assert not dA.any() and not dB.any()


# ---------------------------------------------------------------------------- LoRA with input dropout
@pytest.mark.parametrize("M,p,d_in,r", [(300, 0.1, 328, 16), (129, 0.5, 328, 16), (300, 0.1, 336, 16),
                                         (200, 0.5, 336, 32), (130, 0.3, 528, 8), (150, 0.3, 336, 128),
                                         (97, 0.2, 328, 96)])
def test_lora_dropout_fwd_bwd(ops, M, p, d_in, r):
    """d_in 328: Xd is written once and read by the rank-r passes; d_in 336 / 528 (16-byte mask
    rows): those passes read the mask beside X and form Xd in registers."""
    case, t, g = lin_inputs("lora_4096_bf16", M=M, d_in=d_in, d_out=264, r=r, bias=True)
    mask = D.make_dropout_mask(M, case.d_in, p)
    keep = 1.0 / (1.0 - p)
    Y, Z = ops.lora_linear_dropout_fwd(g["X"], gpu(mask), keep, g["W0"], g["A"], g["B"], case.s, g["bias"])
    X, W0, A, B = (f64(t[k]) for k in ("X", "W0", "A", "B"))
    mk = mask.numpy()
    assert_close(Y, O.lora_dropout_fwd(X, mk, keep, W0, A, B, case.s, f64(t["bias"])), "bf16", "Y")
    assert_close(Z, (X * (mk * keep)) @ A.T, "bf16", "Z")
    rX, rA, rB, rb = O.lora_dropout_bwd(X, mk, keep, W0, A, B, case.s, f64(t["dY"]))
    for z in (Z, None):  # saved Z and the recomputed one
        dX, dA, dB, dbias = ops.lora_linear_dropout_bwd(g["X"], gpu(mask), keep, g["W0"], g["A"], g["B"], z,
                                                        g["dY"], case.s, need_dbias=True)
        assert_close(dX, rX, "bf16", "dX")
        assert_close(dA, rA, "bf16", "dA")
        assert_close(dB, rB, "bf16", "dB")
        assert_close(dbias, rb[None, :], "bf16", "dbias")


@pytest.mark.parametrize("r", [16, 32])
def test_lora_dropout_mask_in_passes_matches_written_xd_bits(ops, r, monkeypatch):
    """The mask applied in registers inside the rank-r passes gives the same bits as those passes
    over an explicitly written Xd (the same bf16(x k) values in the same order): Z, Y, dX, dA, dB;
    dX is also checked against the oracle."""
    case, t, g = lin_inputs("lora_4096_bf16", M=333, d_in=400, d_out=264, r=r, bias=True)
    mk = D.make_dropout_mask(333, 400, 0.25)
    mask = gpu(mk)
    args = (g["X"], mask, 1 / 0.75, g["W0"], g["A"], g["B"])
    out = {}
    for xd in ("0", "1"):
        monkeypatch.setenv("LORA_GB300_DROPOUT_XD", xd)
        Y, Z = ops.lora_linear_dropout_fwd(*args, case.s, g["bias"])
        out[xd] = (Y, Z) + tuple(ops.lora_linear_dropout_bwd(*args, None, g["dY"], case.s)[:3])
    for a, b, nm in zip(out["0"], out["1"], ("Y", "Z", "dX", "dA", "dB")):
        assert torch.equal(a, b), nm
    X, W0, A, B = (f64(t[k]) for k in ("X", "W0", "A", "B"))
    rX = O.lora_dropout_bwd(X, mk.numpy(), 1 / 0.75, W0, A, B, case.s, f64(t["dY"]))[0]
    for xd in ("0", "1"):
        assert_close(out[xd][2], rX, "bf16", "dX")


def test_lora_dropout_all_kept_matches_plain_layer(ops):
    """An all-ones mask with unit scale is the plain layer: same values within bf16 rounding."""
    case, t, g = lin_inputs("lora_4096_bf16", **SMALL, r=16)
    ones = torch.ones(SMALL["M"], SMALL["d_in"], dtype=torch.uint8, device=DEV)
    Yd, Zd = ops.lora_linear_dropout_fwd(g["X"], ones, 1.0, g["W0"], g["A"], g["B"], case.s)
    Y, Z = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], case.s)
    assert torch.equal(Yd, Y) and torch.equal(Zd, Z)


def test_lora_dropout_strength0_and_m_zero(ops):
    case, t, g = lin_inputs("lora_4096_bf16", **SMALL, r=16)
    mask = gpu(D.make_dropout_mask(SMALL["M"], SMALL["d_in"], 0.3))
    Y0, _ = ops.lora_linear_dropout_fwd(g["X"], mask, 1 / 0.7, g["W0"], g["A"], g["B"], 0.0, save_z=False)
    Yb, _ = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], 0.0, save_z=False)
    assert torch.equal(Y0, Yb)
    dX, dA, dB, _ = ops.lora_linear_dropout_bwd(g["X"], mask, 1 / 0.7, g["W0"], g["A"], g["B"], None, g["dY"], 0.0)
    assert torch.equal(dX, ops.lora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], None, g["dY"], 0.0)[0])
    assert not dA.any() and not dB.any()
    e = torch.empty(0, SMALL["d_in"], dtype=torch.bfloat16, device=DEV)
    Ye, _ = ops.lora_linear_dropout_fwd(e, mask[:0], 2.0, g["W0"], g["A"], g["B"], case.s)
    assert Ye.shape == (0, SMALL["d_out"])


# ---------------------------------------------------------------------------- LoRA, fp32 (tiny workload)
def test_lora_tiny_f32(ops):
    case, t, g = lin_inputs("lora_tiny_f32")
    Y, Z = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], case.s, g["bias"])
    X, W0, A, B = (f64(t[k]) for k in ("X", "W0", "A", "B"))
    assert_close(Y, O.lora_linear_fwd(X, W0, A, B, case.s, f64(t["bias"])), "f32", "Y")
    dX, dA, dB, dbias = ops.lora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], Z, g["dY"], case.s, need_dbias=True)
    rX, rA, rB, rb = O.lora_linear_bwd(X, W0, A, B, case.s, f64(t["dY"]))
    for got, ref, nm in ((dX, rX, "dX"), (dA, rA, "dA"), (dB, rB, "dB"), (dbias, rb, "dbias")):
        assert_close(got, ref, "f32", nm)


# ---------------------------------------------------------------------------- DoRA
@pytest.mark.parametrize("dtype,r", [("bf16", 32), ("f32", 32), ("bf16", 96), ("bf16", 128), ("f32", 128)])
def test_dora_fwd_bwd(ops, dtype, r):
    case, t, g = lin_inputs("dora_4096x11008_bf16", M=300, d_in=328, d_out=520, r=r, dtype=dtype)
    r0 = ops.dora_rownorm2(g["W0"])
    np.testing.assert_allclose(to64(r0), O.dora_rownorm2(f64(t["W0"])), rtol=1e-5)
    Y, Z, n, V = ops.dora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], r0, case.s, case.eps, g["bias"])
    X, W0, A, B, m, bias, dY = (f64(t[k]) for k in ("X", "W0", "A", "B", "m", "bias", "dY"))
    rY, rn = O.dora_linear_fwd(X, W0, A, B, m, case.s, case.eps, bias)
    assert_close(Y, rY, dtype, "Y")
    np.testing.assert_allclose(to64(n), rn, rtol=1e-4)
    dX, dA, dB, dm, dbias = ops.dora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], g["m"], g["bias"], Y, Z, n, V,
                                                g["dY"], case.s, case.eps, need_dbias=True)
    rX, rA, rB, rm, rb = O.dora_linear_bwd(X, W0, A, B, m, case.s, dY, case.eps)
    for got, ref, nm in ((dX, rX, "dX"), (dA, rA, "dA"), (dB, rB, "dB"), (dm, rm[None], "dm"),
                         (dbias, rb[None], "dbias")):
        assert_close(got, ref, dtype, nm)


def test_dora_init_is_plain_linear(ops):
    case, t, g = lin_inputs("dora_4096x11008_bf16", M=256, d_in=256, d_out=264, r=16)
    g["B"].zero_()
    m = torch.linalg.vector_norm(g["W0"].float(), dim=1).to(torch.bfloat16)
    r0 = ops.dora_rownorm2(g["W0"])
    Y, *_ = ops.dora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], m, r0, case.s, case.eps, g["bias"])
    assert_close(Y, f64(t["X"]) @ f64(t["W0"]).T + f64(t["bias"]), "bf16", "Y")


def test_dora_strength0_is_frozen_base_bits(ops):
    case, t, g = lin_inputs("dora_4096x11008_bf16", M=200, d_in=136, d_out=264, r=16)
    r0 = ops.dora_rownorm2(g["W0"])
    Yd, *_ = ops.dora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], r0, 0.0, case.eps, g["bias"])
    Yl, _ = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], 0.0, g["bias"])
    assert torch.equal(Yd, Yl)


def test_dora_m_zero_and_strength0_backward(ops):
    """No tokens: empty outputs and zero gradients.  Strength 0: the frozen base's backward, dX the
    bits of the plain layer's s = 0 dX, dbias the column sums of dY, no adapter or magnitude
    gradient."""
    case, t, g = lin_inputs("dora_4096x11008_bf16", M=200, d_in=136, d_out=264, r=16)
    r0 = ops.dora_rownorm2(g["W0"])
    e = g["X"][:0]
    Y, Z, n, V = ops.dora_linear_fwd(e, g["W0"], g["A"], g["B"], g["m"], r0, case.s, case.eps, g["bias"])
    assert Y.shape == (0, 264)
    dX, dA, dB, dm, dbias = ops.dora_linear_bwd(e, g["W0"], g["A"], g["B"], g["m"], g["bias"], Y, Z, n, V,
                                                g["dY"][:0], case.s, case.eps, need_dbias=True)
    assert dX.shape == (0, 136)
    assert not dA.any() and not dB.any() and not dm.any() and not dbias.any()
    Y, Z, n, V = ops.dora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], r0, 0.0, case.eps, g["bias"])
    dX, dA, dB, dm, dbias = ops.dora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], g["m"], g["bias"], Y, Z, n, V,
                                                g["dY"], 0.0, case.eps, need_dbias=True)
    assert torch.equal(dX, ops.lora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], None, g["dY"], 0.0)[0])
    assert not dA.any() and not dB.any() and not dm.any()
    assert_close(dbias, f64(t["dY"]).sum(axis=0)[None, :], "bf16", "dbias")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_dora_eps_floor_rows(ops, dtype):
    """eps above some rows' adapted norm: those rows take the floor n = eps and pass no gradient
    through the norm (the clamped branch of the norm and of g), the others stay live."""
    case = D.scaled(D.WORKLOADS["dora_4096x11008_bf16"], M=300, d_in=328, d_out=520, r=32, dtype=dtype)
    t = D.make_linear(case)
    low = [0, 3, 130, 517]
    for k in ("W0", "B"):
        t[k][low] = (t[k][low].float() * 0.05).to(t[k].dtype)
    eps = 0.3
    g = {k: gpu(v) for k, v in t.items()}
    X, W0, A, B, m, bias, dY = (f64(t[k]) for k in ("X", "W0", "A", "B", "m", "bias", "dY"))
    nraw = np.linalg.norm(O.adapted_weight(W0, A, B, case.s), axis=1)
    assert (nraw[low] < eps).all() and (np.delete(nraw, low) > eps).all()
    r0 = ops.dora_rownorm2(g["W0"])
    Y, Z, n, V = ops.dora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], r0, case.s, eps, g["bias"])
    rY, rn = O.dora_linear_fwd(X, W0, A, B, m, case.s, eps, bias)
    assert (to64(n)[low] == np.float32(eps)).all()
    np.testing.assert_allclose(to64(n), rn, rtol=1e-4)
    assert_close(Y, rY, dtype, "Y")
    dX, dA, dB, dm, _ = ops.dora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], g["m"], g["bias"], Y, Z, n, V,
                                            g["dY"], case.s, eps)
    rX, rA, rB, rm, _ = O.dora_linear_bwd(X, W0, A, B, m, case.s, dY, eps)
    for got, ref, nm in ((dX, rX, "dX"), (dA, rA, "dA"), (dB, rB, "dB"), (dm, rm[None], "dm")):
        assert_close(got, ref, dtype, nm)


def test_dora_zero_row_at_default_eps(ops):
    """A row of W0 and B that is exactly zero: its norm is the 1e-12 floor, its output the bias,
    and its up-projection gradient carries the scale m / eps."""
    case = D.scaled(D.WORKLOADS["dora_4096x11008_bf16"], M=260, d_in=200, d_out=264, r=16)
    t = D.make_linear(case)
    t["W0"][7] = 0
    t["B"][7] = 0
    t["m"][7] = 1.5
    g = {k: gpu(v) for k, v in t.items()}
    X, W0, A, B, m, bias, dY = (f64(t[k]) for k in ("X", "W0", "A", "B", "m", "bias", "dY"))
    r0 = ops.dora_rownorm2(g["W0"])
    Y, Z, n, V = ops.dora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], r0, case.s, case.eps, g["bias"])
    assert float(n[7]) == np.float32(case.eps)
    rY, _ = O.dora_linear_fwd(X, W0, A, B, m, case.s, case.eps, bias)
    assert_close(Y, rY, "bf16", "Y")
    dX, dA, dB, dm, _ = ops.dora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], g["m"], g["bias"], Y, Z, n, V,
                                            g["dY"], case.s, case.eps)
    rX, rA, rB, rm, _ = O.dora_linear_bwd(X, W0, A, B, m, case.s, dY, case.eps)
    assert abs(rB[7]).max() > 1e9
    for got, ref, nm in ((dX, rX, "dX"), (dA, rA, "dA"), (dB, rB, "dB"), (dm, rm[None], "dm")):
        assert_close(got, ref, "bf16", nm)


# ---------------------------------------------------------------------------- DoRA (cols)
@pytest.mark.parametrize("r", [32, 16, 128])
def test_dora_cols_fwd_bwd(ops, r):
    case, t, g = lin_inputs("dora_cols_4096x11008_bf16", M=300, d_in=328, d_out=520, r=r)
    c0 = ops.dora_colnorm2(g["W0"])
    np.testing.assert_allclose(to64(c0), O.dora_colnorm2(f64(t["W0"])), rtol=1e-5)
    Y, Z, n, U = ops.dora_cols_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], c0, case.s, case.eps, g["bias"])
    X, W0, A, B, m, bias, dY = (f64(t[k]) for k in ("X", "W0", "A", "B", "m", "bias", "dY"))
    rY, rn = O.dora_cols_fwd(X, W0, A, B, m, case.s, case.eps, bias)
    assert_close(Y, rY, "bf16", "Y")
    np.testing.assert_allclose(to64(n), rn, rtol=1e-4)
    np.testing.assert_allclose(to64(U), (B.T @ W0).T, rtol=1e-4, atol=1e-5)
    dX, dA, dB, dm, dbias = ops.dora_cols_bwd(g["X"], g["W0"], g["A"], g["B"], g["m"], Z, n, U, g["dY"], case.s,
                                              case.eps, need_dbias=True)
    rX, rA, rB, rm, rb = O.dora_cols_bwd(X, W0, A, B, m, case.s, dY, case.eps)
    for got, ref, nm in ((dX, rX, "dX"), (dA, rA, "dA"), (dB, rB, "dB"), (dm, rm[None], "dm"),
                         (dbias, rb[None], "dbias")):
        assert_close(got, ref, "bf16", nm)
    # without dX and without the saved Z: same adapter gradients, bit for bit
    _, dA2, dB2, dm2, _ = ops.dora_cols_bwd(g["X"], g["W0"], g["A"], g["B"], g["m"], None, n, U, g["dY"], case.s,
                                            case.eps, need_dx=False)
    assert torch.equal(dA, dA2) and torch.equal(dB, dB2) and torch.equal(dm, dm2)


def test_dora_cols_eps_floor_columns(ops):
    """Column variant with eps above some columns' adapted norm (floor branch) and the rest live."""
    case = D.scaled(D.WORKLOADS["dora_cols_4096x11008_bf16"], M=300, d_in=328, d_out=520, r=16)
    t = D.make_linear(case)
    low = [0, 5, 200, 327]
    t["W0"][:, low] = (t["W0"][:, low].float() * 0.05).to(torch.bfloat16)
    t["A"][:, low] = (t["A"][:, low].float() * 0.05).to(torch.bfloat16)
    eps = 0.3
    g = {k: gpu(v) for k, v in t.items()}
    X, W0, A, B, m, bias, dY = (f64(t[k]) for k in ("X", "W0", "A", "B", "m", "bias", "dY"))
    nraw = np.linalg.norm(O.adapted_weight(W0, A, B, case.s), axis=0)
    assert (nraw[low] < eps).all() and (np.delete(nraw, low) > eps).all()
    c0 = ops.dora_colnorm2(g["W0"])
    Y, Z, n, U = ops.dora_cols_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], c0, case.s, eps, g["bias"])
    rY, rn = O.dora_cols_fwd(X, W0, A, B, m, case.s, eps, bias)
    assert (to64(n)[low] == np.float32(eps)).all()
    assert_close(Y, rY, "bf16", "Y")
    dX, dA, dB, dm, _ = ops.dora_cols_bwd(g["X"], g["W0"], g["A"], g["B"], g["m"], Z, n, U, g["dY"], case.s, eps)
    rX, rA, rB, rm, _ = O.dora_cols_bwd(X, W0, A, B, m, case.s, dY, eps)
    for got, ref, nm in ((dX, rX, "dX"), (dA, rA, "dA"), (dB, rB, "dB"), (dm, rm[None], "dm")):
        assert_close(got, ref, "bf16", nm)


def test_dora_cols_init_and_strength0(ops):
    case, t, g = lin_inputs("dora_cols_4096x11008_bf16", M=256, d_in=264, d_out=256, r=16)
    c0 = ops.dora_colnorm2(g["W0"])
    Yl, _ = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], 0.0, g["bias"])
    Y0, *_ = ops.dora_cols_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], c0, 0.0, case.eps, g["bias"])
    assert torch.equal(Y0, Yl)   # strength 0: the frozen base, bit for bit
    g["B"].zero_()
    m0 = torch.sqrt(c0).to(torch.bfloat16)
    Yi, *_ = ops.dora_cols_fwd(g["X"], g["W0"], g["A"], g["B"], m0, c0, case.s, case.eps, g["bias"])
    X, W0, bias = f64(t["X"]), f64(t["W0"]), f64(t["bias"])
    assert_close(Yi, X @ W0.T + bias, "bf16", "Y at init")


# ---------------------------------------------------------------------------- SwiGLU MLP
def mlp_inputs(**kw):
    case = D.scaled(D.WORKLOADS["mlp_swiglu_4096x14336_bf16"], **kw)
    t = D.make_mlp(case)
    g = {k: gpu(v) for k, v in t.items()}
    P = {p: {"W": g["W" + p], "A": g["A" + p], "B": g["B" + p], "s": case.scales[p]} for p in "gud"}
    return case, t, g, P


def _mlp_args64(t, s):
    """Oracle arguments; s is one scale for all projections or a dict of per-projection scales."""
    sc = s if isinstance(s, dict) else {p: s for p in "gud"}
    return (f64(t["X"]), f64(t["Wg"]), f64(t["Ag"]), f64(t["Bg"]), sc["g"], f64(t["Wu"]), f64(t["Au"]), f64(t["Bu"]),
            sc["u"], f64(t["Wd"]), f64(t["Ad"]), f64(t["Bd"]), sc["d"])


ACTS = {"swiglu": 0, "geglu": 1}


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
@pytest.mark.parametrize("I", [200, 256])
def test_mlp_fwd_bwd(ops, I, act):
    case, t, g, P = mlp_inputs(M=300, H=136, I=I, r=16, alpha=24.0)
    Y, saved = ops.lora_mlp_swiglu_fwd(g["X"], P["g"], P["u"], P["d"], act=ACTS[act])
    args = _mlp_args64(t, case.s)
    ry, re, ru, rh = O.mlp_swiglu_fwd(*args, act=act)
    assert_close(saved["e"], re, "bf16", "e")
    assert_close(saved["u"], ru, "bf16", "u")
    assert_close(saved["h"], rh, "bf16", "h")
    assert_close(Y, ry, "bf16", "y")
    gr = ops.lora_mlp_swiglu_bwd(g["X"], P["g"], P["u"], P["d"], saved, g["dY"], act=ACTS[act])
    ref = O.mlp_swiglu_bwd(*args, f64(t["dY"]), act=act)
    for k in ("dX", "dAg", "dBg", "dAu", "dBu", "dAd", "dBd"):
        assert_close(gr[k], ref[k], "bf16", k)


# ---------------------------------------------------------------------------- fused-leaf (QKV)
def qkv_inputs(**kw):
    case = D.scaled(D.WORKLOADS["qkv_lora_4096_gqa_bf16"], **kw)
    t = D.make_qkv(case)
    g = {k: gpu(v) for k, v in t.items()}
    L = len(case.n)
    leaves_g = [(g[f"A{l}"], g[f"B{l}"], case.s[l]) for l in range(L)]
    leaves_64 = [(f64(t[f"A{l}"]), f64(t[f"B{l}"]), case.s[l]) for l in range(L)]
    return case, t, g, leaves_g, leaves_64


@pytest.mark.parametrize("n,r,bias", [((256, 72, 72), 16, True), ((256, 72, 72), 8, False),
                                      ((136, 264), 32, False), ((200,), 64, True),
                                      ((256, 72, 72), 32, True), ((128, 64, 64), 64, False),
                                      ((256, 72, 72), 96, True), ((128, 64, 64), 128, False)])
def test_qkv_fwd_bwd(ops, n, r, bias):
    case, t, g, lg_, l64 = qkv_inputs(M=300, d_in=200, n=n, r=r, bias=bias)
    Y, Z = ops.lora_qkv_fwd(g["X"], g["W0"], lg_, g["bias"])
    X, W0, dY, b = f64(t["X"]), f64(t["W0"]), f64(t["dY"]), f64(t["bias"])
    assert_close(Y, O.qkv_lora_fwd(X, W0, l64, b), "bf16", "Y")
    assert_close(Z, np.concatenate([X @ A.T for A, _, _ in l64], axis=1), "bf16", "Z")
    dX, dA, dB, db = ops.lora_qkv_bwd(g["X"], g["W0"], lg_, Z, g["dY"], need_dbias=True)
    rX, rA, rB, rb = O.qkv_lora_bwd(X, W0, l64, dY)
    assert_close(dX, rX, "bf16", "dX")
    assert_close(db[None], rb[None], "bf16", "dbias")
    for i in range(len(n)):
        assert_close(dA[i], rA[i], "bf16", f"dA{i}")
        assert_close(dB[i], rB[i], "bf16", f"dB{i}")
    # without the saved Z the backward recomputes it: same kernels, same bits
    dX2, dA2, dB2, _ = ops.lora_qkv_bwd(g["X"], g["W0"], lg_, None, g["dY"])
    assert torch.equal(dX, dX2)
    assert all(torch.equal(a, b_) for a, b_ in zip(dA + dB, dA2 + dB2))


def test_qkv_zero_strength_leaf_is_frozen_base_bits(ops):
    case, t, g, lg_, _ = qkv_inputs(M=260, d_in=264, n=(256, 64, 64), r=16)
    mixed = [lg_[0], (lg_[1][0], lg_[1][1], 0.0), lg_[2]]
    off = [(A, B, 0.0) for A, B, _ in lg_]
    Y, _ = ops.lora_qkv_fwd(g["X"], g["W0"], mixed)
    Y0, _ = ops.lora_qkv_fwd(g["X"], g["W0"], off)
    assert torch.equal(Y[:, 256:320], Y0[:, 256:320])
    assert not torch.equal(Y[:, :256], Y0[:, :256])
    dX, dA, dB, _ = ops.lora_qkv_bwd(g["X"], g["W0"], mixed, None, g["dY"])
    assert not dA[1].any() and not dB[1].any()
    dX0, dA0, dB0, _ = ops.lora_qkv_bwd(g["X"], g["W0"], off, None, g["dY"])
    assert all(not a.any() for a in dA0 + dB0)
    Bz = torch.zeros(384, 16, dtype=torch.bfloat16, device=DEV)
    ref = ops.lora_linear_bwd(g["X"], g["W0"], lg_[0][0], Bz, None, g["dY"], 0.0)[0]
    assert torch.equal(dX0, ref)    # every strength 0: dX is the frozen base's, bit for bit


def test_qkv_m_zero_is_noop(ops):
    case, t, g, lg_, _ = qkv_inputs(M=8, d_in=64, n=(64, 16, 16), r=8)
    X = g["X"][:0]
    Y, Z = ops.lora_qkv_fwd(X, g["W0"], lg_)
    assert Y.shape == (0, 96) and Z.shape == (0, 24)
    dX, dA, dB, db = ops.lora_qkv_bwd(X, g["W0"], lg_, Z, g["dY"][:0], need_dbias=True)
    assert all(not a.any() for a in dA + dB) and not db.any()


@pytest.mark.parametrize("ranks", [(48, 48, 48), (64, 64, 64), (128, 128, 128), (16, 48, 128), (128, 8, 40)])
def test_mlp_large_rank(ops, ranks):
    """Large and unequal ranks per projection: the gate/up down-projection [Zg | Zu] spans several
    64-column passes, the stacked tail several K-steps with the up half shifted by r_g."""
    rg, ru, rd = ranks
    case, t, g, P = mlp_inputs(M=260, H=136, I=200, r=rg, r_u=ru, r_d=rd, alpha=32.0)
    Y, saved = ops.lora_mlp_swiglu_fwd(g["X"], P["g"], P["u"], P["d"])
    assert saved["Zgu"].shape == (260, rg + ru) and saved["Zd"].shape == (260, rd)
    args = _mlp_args64(t, case.scales)
    ry, re, ru, rh = O.mlp_swiglu_fwd(*args)
    for got, ref, nm in ((saved["e"], re, "e"), (saved["u"], ru, "u"), (saved["h"], rh, "h"), (Y, ry, "y")):
        assert_close(got, ref, "bf16", nm)
    gr = ops.lora_mlp_swiglu_bwd(g["X"], P["g"], P["u"], P["d"], saved, g["dY"])
    ref = O.mlp_swiglu_bwd(*args, f64(t["dY"]))
    for k in ("dX", "dAg", "dBg", "dAu", "dBu", "dAd", "dBd"):
        assert_close(gr[k], ref[k], "bf16", k)


# ---------------------------------------------------------------------------- W8A8
def w8_inputs(**kw):
    case = D.scaled(D.WORKLOADS["w8a8_lora_3072"], **kw)
    t = D.make_w8a8(case)
    Wq, sw = O.quantize_rows(t["W0"].numpy())      # offline weight quantisation (shared bytes)
    Xq, sx = O.quantize_rows(t["X"].float().numpy())
    return case, t, Wq, sw, Xq, sx


def test_w8a8_quantize_bit_exact(ops):
    case, t, *_ = w8_inputs(M=300, d_in=352, d_out=264)
    X = gpu(t["X"])
    X[7].zero_()                                   # an all-zero row
    Xq, sx, Z = ops.w8a8_quantize_rows(X, gpu(t["A"]))
    rq, rs = O.quantize_rows(X.float().cpu().numpy())
    np.testing.assert_array_equal(Xq.cpu().numpy(), rq)
    np.testing.assert_array_equal(sx.cpu().numpy(), rs)
    assert_close(Z, f64(X.cpu()) @ f64(t["A"]).T, "bf16", "Z")


@pytest.mark.parametrize("cols,r", [(1032, 8), (3072, 32), (6400, 24), (6408, 16), (1024, 40)])
def test_w8a8_quantize_with_z_shapes(ops, cols, r):
    """Codes and scales bit-exact and Z within the bf16 bar over column counts with several 64-wide
    stages and a ragged last one, ranks from 8 to 40 (more than one rank-r column chunk per warp
    at 40), a zero row and a row with one dominant entry; both code formats."""
    g = torch.Generator().manual_seed(cols + r)
    M = 200
    X = (torch.randn(M, cols, generator=g) * 0.5).to(torch.bfloat16)
    X[3] = 0
    X[5, 7] = 40.0                                  # one dominant entry in a row
    A = (torch.randn(r, cols, generator=g) / cols ** 0.5).to(torch.bfloat16)
    rq, rs = O.quantize_rows(X.float().numpy())
    Xq, sx, Z = ops.w8a8_quantize_rows(gpu(X), gpu(A))
    np.testing.assert_array_equal(Xq.cpu().numpy(), rq)
    np.testing.assert_array_equal(sx.cpu().numpy(), rs)
    assert_close(Z, f64(X) @ f64(A).T, "bf16", "Z")
    Xc, sx2, Z2 = ops.w8a8_quantize_rows_bf16(gpu(X), gpu(A))
    np.testing.assert_array_equal(Xc.float().cpu().numpy(), rq.astype(np.float32))
    np.testing.assert_array_equal(sx2.cpu().numpy(), rs)
    assert torch.equal(Z, Z2)


def _near_tie_rows(cols=512, rows=48, seed=77):
    """bf16 rows whose quotients x / s sit on or next to half-integers: rows with a power-of-two
    scale (amax = 127 * 2^e) holding exact k + 0.5 multiples of it (ties, rounded to even), and rows
    with an arbitrary scale filled with values whose float32 quotient lies within 2^-14 of a
    half-integer (found by search), all beside their row maximum."""
    rng = np.random.default_rng(seed)
    out = np.zeros((rows, cols), np.float32)
    for i in range(rows):
        if i % 2 == 0:   # exact ties
            e = int(rng.integers(-6, 6))
            amax = np.float32(127.0 * 2.0 ** e)
            k = rng.integers(0, 127, size=cols).astype(np.float32)
            row = (k + np.float32(0.5)) * np.float32(2.0 ** e) * rng.choice([-1, 1], size=cols).astype(np.float32)
        else:            # near ties under an arbitrary scale
            amax = torch.tensor(float(rng.uniform(0.5, 40.0))).to(torch.bfloat16).float().item()
            sc = np.float32(amax) / np.float32(127.0)
            cand = torch.from_numpy(rng.uniform(-amax, amax, size=400000).astype(np.float32))
            cand = cand.to(torch.bfloat16).float().numpy()
            q = cand / sc                                       # float32 quotients (IEEE)
            near = np.abs(np.abs(q) - np.floor(np.abs(q)) - np.float32(0.5)) <= 2.0 ** -14
            pick = cand[near]
            assert pick.size > 0
            row = rng.choice(pick, size=cols)
        row[int(rng.integers(0, cols))] = amax
        out[i] = row
    return torch.from_numpy(out).to(torch.bfloat16)


def test_w8a8_quantize_near_ties_bit_exact(ops):
    """The quantiser's codes where the quotient is a tie or within 2^-14 of one (the values whose
    code depends on the last bits of the correctly rounded quotient) match the oracle's bit for bit."""
    X = _near_tie_rows()
    rq, rs = O.quantize_rows(X.float().numpy())
    Xq, sx, _ = ops.w8a8_quantize_rows(gpu(X))
    np.testing.assert_array_equal(sx.cpu().numpy(), rs)
    np.testing.assert_array_equal(Xq.cpu().numpy(), rq)
    Xc, _, _ = ops.w8a8_quantize_rows_bf16(gpu(X))
    np.testing.assert_array_equal(Xc.float().cpu().numpy(), rq.astype(np.float32))


@pytest.mark.parametrize("bias", [False, True])
def test_w8a8_acc_bit_exact_and_epilogue(ops, bias):
    case, t, Wq, sw, Xq, sx = w8_inputs(M=300, d_in=352, d_out=264, bias=bias)
    Z = (t["X"].double() @ t["A"].double().T).to(torch.bfloat16)
    Y, acc = ops.w8a8_lora_fwd(gpu(torch.from_numpy(Xq)), gpu(torch.from_numpy(sx)), gpu(torch.from_numpy(Wq)),
                               gpu(torch.from_numpy(sw)), gpu(Z), gpu(t["B"]), case.s, gpu(t["bias"]), want_acc=True)
    ry, racc = O.w8a8_lora_fwd(Xq, sx, Wq, sw, f64(Z), f64(t["B"]), case.s, f64(t["bias"]))
    np.testing.assert_array_equal(acc.cpu().numpy().astype(np.int64), racc)
    assert_close(Y, ry, "bf16", "Y")


@pytest.mark.parametrize("path", ["tensor_chunks", "integer_mma"])
def test_w8a8_both_product_paths(ops, path, monkeypatch):
    """The bf16 tensor-core path (codes as bf16, exact 1024-wide K chunks added as int32) and the
    integer MMA path give the same exact int32 product and the same epilogue."""
    if path == "integer_mma":
        monkeypatch.setenv("LORA_GB300_W8A8_IMMA", "1")
    case, t, Wq, sw, Xq, sx = w8_inputs(M=260, d_in=320, d_out=136, bias=True)
    Z = (t["X"].double() @ t["A"].double().T).to(torch.bfloat16)
    Y, acc = ops.w8a8_lora_fwd(gpu(torch.from_numpy(Xq)), gpu(torch.from_numpy(sx)), gpu(torch.from_numpy(Wq)),
                               gpu(torch.from_numpy(sw)), gpu(Z), gpu(t["B"]), case.s, gpu(t["bias"]), want_acc=True)
    ry, racc = O.w8a8_lora_fwd(Xq, sx, Wq, sw, f64(Z), f64(t["B"]), case.s, f64(t["bias"]))
    np.testing.assert_array_equal(acc.cpu().numpy().astype(np.int64), racc)
    assert_close(Y, ry, "bf16", "Y")


@pytest.mark.parametrize("bias,zero_rows", [(False, False), (True, True)])
def test_w8a8_output_with_and_without_int32(ops, bias, zero_rows):
    """The dequantised output matches the oracle, including an all-zero input row and an all-zero
    weight row (scale 0), and has the same bits whether or not the raw int32 product is also
    written."""
    case, t, Wq, sw, Xq, sx = w8_inputs(M=300, d_in=352, d_out=264, bias=bias)
    if zero_rows:
        Xq[5] = 0
        sx[5] = 0.0
        Wq[9] = 0
        sw[9] = 0.0
    Z = (t["X"].double() @ t["A"].double().T).to(torch.bfloat16)
    if zero_rows:
        Z[5] = 0
    args = (gpu(torch.from_numpy(Xq)), gpu(torch.from_numpy(sx)), gpu(torch.from_numpy(Wq)),
            gpu(torch.from_numpy(sw)), gpu(Z), gpu(t["B"]), case.s, gpu(t["bias"]))
    Y, _ = ops.w8a8_lora_fwd(*args)
    ry, racc = O.w8a8_lora_fwd(Xq, sx, Wq, sw, f64(Z), f64(t["B"]), case.s, f64(t["bias"]))
    assert_close(Y, ry, "bf16", "Y")
    Ye, acc = ops.w8a8_lora_fwd(*args, want_acc=True)
    assert torch.equal(Y, Ye)
    np.testing.assert_array_equal(acc.cpu().numpy().astype(np.int64), racc)


@pytest.mark.parametrize("path", ["tensor_chunks", "integer_mma"])
def test_w8a8_deep_k_exact(ops, path, monkeypatch):
    """d_in of 8832 (nine 1024-wide exact chunks, the last one ragged) with all codes at +-127 in
    places, on both product paths: bit-exact int32."""
    if path == "integer_mma":
        monkeypatch.setenv("LORA_GB300_W8A8_IMMA", "1")
    rng = np.random.default_rng(5)
    M, K, N = 200, 8832, 264
    Xq = rng.integers(-127, 128, (M, K)).astype(np.int8)
    Wq = rng.integers(-127, 128, (N, K)).astype(np.int8)
    Xq[3] = 127
    Wq[7] = 127
    Wq[8] = -127
    _, acc = ops.w8a8_lora_fwd(gpu(torch.from_numpy(Xq)), None, gpu(torch.from_numpy(Wq)), None, None, None, 0.0,
                               want_acc=True, want_y=False)
    np.testing.assert_array_equal(acc.cpu().numpy().astype(np.int64), O.int8_accumulate(Xq, Wq))


@pytest.mark.parametrize("bias", [False, True])
def test_w8a8_packed_path(ops, bias):
    """Prepacked operands: the quantiser's bf16 codes, the weight's bf16 codes and dequantised
    copy made once; the packed forward gives the same bits as w8a8_lora_fwd and the exact int32
    product; the backward through the dequantised weight matches the oracle."""
    case, t, Wq, sw, Xq, sx = w8_inputs(M=300, d_in=352, d_out=264, bias=bias)
    X, A = gpu(t["X"]), gpu(t["A"])
    Xc, gsx, gZ = ops.w8a8_quantize_rows_bf16(X, A)
    np.testing.assert_array_equal(Xc.float().cpu().numpy(), Xq.astype(np.float32))    # codes, exactly
    np.testing.assert_array_equal(gsx.cpu().numpy(), sx)
    gWq, gsw = gpu(torch.from_numpy(Wq)), gpu(torch.from_numpy(sw))
    Wb, Wd = ops.w8a8_prepack_weight(gWq, gsw)
    np.testing.assert_array_equal(Wb.float().cpu().numpy(), Wq.astype(np.float32))
    assert_close(Wd, O.w8a8_dequant_weight(Wq, sw), "bf16", "Wd")
    Z = (t["X"].double() @ t["A"].double().T).to(torch.bfloat16)
    ry, racc = O.w8a8_lora_fwd(Xq, sx, Wq, sw, f64(Z), f64(t["B"]), case.s, f64(t["bias"]))
    Yp, accp = ops.w8a8_lora_fwd_packed(Xc, gsx, Wb, gsw, gpu(Z), gpu(t["B"]), case.s, gpu(t["bias"]),
                                        want_acc=True)
    np.testing.assert_array_equal(accp.cpu().numpy().astype(np.int64), racc)
    assert_close(Yp, ry, "bf16", "Y packed")
    Yf, _ = ops.w8a8_lora_fwd_packed(Xc, gsx, Wb, gsw, gpu(Z), gpu(t["B"]), case.s, gpu(t["bias"]))
    Yu, _ = ops.w8a8_lora_fwd(gpu(torch.from_numpy(Xq)), gsx, gWq, gsw, gpu(Z), gpu(t["B"]), case.s, gpu(t["bias"]))
    assert torch.equal(Yf, Yu), "the packed forward runs the same product and epilogue"
    assert torch.equal(Yf, Yp), "the int32 output changes nothing in Y"
    g = torch.Generator().manual_seed(80)
    dY = torch.randn(case.M, case.d_out, generator=g).to(torch.bfloat16)
    dX, dA, dB, db = ops.lora_linear_bwd(X, Wd, A, gpu(t["B"]), gpu(Z), gpu(dY), case.s, need_dbias=True)
    rX, rA, rB, rb = O.w8a8_lora_bwd(f64(t["X"]), Wq, sw, f64(t["A"]), f64(t["B"]), case.s, f64(dY))
    for got, ref, nm in ((dX, rX, "dX"), (dA, rA, "dA"), (dB, rB, "dB"), (db, rb[None], "dbias")):
        assert_close(got, ref, "bf16", nm)


@pytest.mark.parametrize("r", [96, 128])
def test_w8a8_large_rank(ops, r, monkeypatch):
    """Ranks above 64: the quantiser's down-projection in two passes, both epilogues' rank-r
    tail over several K-steps, and the backward through the int8 base."""
    case, t, Wq, sw, Xq, sx = w8_inputs(M=300, d_in=352, d_out=264, r=r, bias=True)
    X = gpu(t["X"])
    gXq, gsx, gZ = ops.w8a8_quantize_rows(X, gpu(t["A"]))
    np.testing.assert_array_equal(gXq.cpu().numpy(), Xq)
    Z = (t["X"].double() @ t["A"].double().T).to(torch.bfloat16)   # the oracle's Z, shared bytes
    assert_close(gZ, f64(Z), "bf16", "Z")
    args = (gpu(torch.from_numpy(Xq)), gpu(torch.from_numpy(sx)), gpu(torch.from_numpy(Wq)),
            gpu(torch.from_numpy(sw)), gpu(Z), gpu(t["B"]), case.s, gpu(t["bias"]))
    ry, racc = O.w8a8_lora_fwd(Xq, sx, Wq, sw, f64(Z), f64(t["B"]), case.s, f64(t["bias"]))
    Y, acc = ops.w8a8_lora_fwd(*args, want_acc=True)                # exact-integer epilogue
    np.testing.assert_array_equal(acc.cpu().numpy().astype(np.int64), racc)
    assert_close(Y, ry, "bf16", "Y (exact epilogue)")
    Yf, _ = ops.w8a8_lora_fwd(*args)                                # folded output-only epilogue
    assert_close(Yf, ry, "bf16", "Y (folded epilogue)")
    g = torch.Generator().manual_seed(79)
    dY = torch.randn(case.M, case.d_out, generator=g).to(torch.bfloat16)
    dX, dA, dB, _ = ops.w8a8_lora_bwd(X, gpu(torch.from_numpy(Wq)), gpu(torch.from_numpy(sw)), gpu(t["A"]),
                                      gpu(t["B"]), gpu(Z), gpu(dY), case.s)
    rX, rA, rB, _ = O.w8a8_lora_bwd(f64(t["X"]), Wq, sw, f64(t["A"]), f64(t["B"]), case.s, f64(dY))
    assert_close(dX, rX, "bf16", "dX")
    assert_close(dA, rA, "bf16", "dA")
    assert_close(dB, rB, "bf16", "dB")


@pytest.mark.parametrize("bias", [False, True])
def test_w8a8_bwd(ops, bias):
    """Backward through the int8 base (straight-through activation quantiser) with the LoRA dgrad."""
    case, t, Wq, sw, Xq, sx = w8_inputs(M=300, d_in=352, d_out=264, bias=bias)
    g = torch.Generator().manual_seed(77)
    dY = torch.randn(case.M, case.d_out, generator=g).to(torch.bfloat16)
    X, A, B = gpu(t["X"]), gpu(t["A"]), gpu(t["B"])
    Z = (t["X"].double() @ t["A"].double().T).to(torch.bfloat16)
    dX, dA, dB, db = ops.w8a8_lora_bwd(X, gpu(torch.from_numpy(Wq)), gpu(torch.from_numpy(sw)), A, B, gpu(Z), gpu(dY),
                                       case.s, need_dbias=True)
    rX, rA, rB, rb = O.w8a8_lora_bwd(f64(t["X"]), Wq, sw, f64(t["A"]), f64(t["B"]), case.s, f64(dY))
    assert_close(dX, rX, "bf16", "dX")
    assert_close(dA, rA, "bf16", "dA")
    assert_close(dB, rB, "bf16", "dB")
    assert_close(db, rb[None], "bf16", "dbias")


def test_w8a8_extreme_codes_exact(ops):
    """All-(+-127) operands: the worst-case |acc| = d_in * 127^2 stays exact in int32."""
    M, K, N = 130, 3072, 136
    Xq = np.full((M, K), 127, np.int8)
    Xq[1::2] = -127
    Wq = np.full((N, K), -127, np.int8)
    Y, acc = ops.w8a8_lora_fwd(gpu(torch.from_numpy(Xq)), None, gpu(torch.from_numpy(Wq)), None, None, None, 0.0,
                               want_acc=True, want_y=False)
    np.testing.assert_array_equal(acc.cpu().numpy().astype(np.int64), O.int8_accumulate(Xq, Wq))
