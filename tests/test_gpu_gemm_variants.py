"""Both tcgen05 GEMM kernels against the oracle: the one-CTA kernel (128 x 256 tiles) and the
CTA-pair kernel (cta_group::2, 256 x 256 tiles over two SMs), selected per call with
LORA_GB300_GEMM_PAIR, in every mode the layer uses (forward, dX with MN-major B, dX with the
DoRA K-scaling warps, SwiGLU forward with stacked B, SwiGLU backward), with ragged M, N, K and
with a capped grid so that every CTA (pair) runs several tiles."""
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


@pytest.fixture(params=["one_cta", "pair"])
def variant(request, monkeypatch):
    monkeypatch.setenv("LORA_GB300_GEMM_PAIR", "1" if request.param == "pair" else "0")
    return request.param


def f64(t):
    return None if t is None else to64(t)


def _ws_ok(ops):
    from dora_adapter_linear_gb300 import _lib as L
    for buf in ops._WS.values():
        assert L.lora_check_device_error(buf) == 0, "a kernel recorded a timed-out wait"


@pytest.mark.parametrize("cap", ["0", "4"])
def test_lora_fwd_bwd(ops, variant, cap, monkeypatch):
    monkeypatch.setenv("LORA_GB300_MAX_CTAS", cap)
    case = D.scaled(D.WORKLOADS["lora_4096_bf16"], M=600, d_in=328, d_out=776, r=16, bias=True)
    t = D.make_linear(case)
    g = {k: v.to(DEV) for k, v in t.items()}
    Y, Z = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], case.s, g["bias"])
    X, W0, A, B = (f64(t[k]) for k in ("X", "W0", "A", "B"))
    assert_close(Y, O.lora_linear_fwd(X, W0, A, B, case.s, f64(t["bias"])), "bf16", "Y")
    dX, dA, dB, _ = ops.lora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], Z, g["dY"], case.s)
    rX, rA, rB, _ = O.lora_linear_bwd(X, W0, A, B, case.s, f64(t["dY"]))
    assert_close(dX, rX, "bf16", "dX")
    assert_close(dA, rA, "bf16", "dA")
    _ws_ok(ops)


@pytest.mark.parametrize("cap", ["0", "4"])
@pytest.mark.parametrize("M", [500, 1024])
def test_lora_even_m_tiles(ops, variant, cap, M, monkeypatch):
    """An even number of M tiles (4 with a ragged last one, and 8), so that the pair kernel's
    256-row tiles are whole or half empty; ragged N and K."""
    monkeypatch.setenv("LORA_GB300_MAX_CTAS", cap)
    case = D.scaled(D.WORKLOADS["lora_4096_bf16"], M=M, d_in=328, d_out=776, r=16, bias=True)
    t = D.make_linear(case)
    g = {k: v.to(DEV) for k, v in t.items()}
    Y, Z = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], case.s, g["bias"])
    X, W0, A, B = (f64(t[k]) for k in ("X", "W0", "A", "B"))
    assert_close(Y, O.lora_linear_fwd(X, W0, A, B, case.s, f64(t["bias"])), "bf16", "Y")
    dX, dA, dB, _ = ops.lora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], Z, g["dY"], case.s)
    rX, rA, rB, _ = O.lora_linear_bwd(X, W0, A, B, case.s, f64(t["dY"]))
    assert_close(dX, rX, "bf16", "dX")
    assert_close(dA, rA, "bf16", "dA")
    assert_close(dB, rB, "bf16", "dB")
    _ws_ok(ops)


def _dora_bwd(ops, g, case):
    r0 = ops.dora_rownorm2(g["W0"])
    Y, Z, n, V = ops.dora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], r0, case.s, case.eps, g["bias"])
    return Y, ops.dora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], g["m"], g["bias"], Y, Z, n, V, g["dY"],
                                  case.s, case.eps, need_dbias=True)


@pytest.mark.parametrize("cap", ["0", "4"])
@pytest.mark.parametrize("M", [500, 1024])
@pytest.mark.parametrize("mode", ["kscale", "slabs"])
def test_dora_kscaled_dx(ops, variant, cap, M, mode, monkeypatch):
    """dP = dY o c for the dX product, either formed inside the dX GEMM (the scaling warps multiply
    each staged dY tile by its 64 scales in shared memory) or written by the column pass one slab of
    rows at a time (slabs of 256 rows here: two to four slabs, the last one ragged) and read back by
    one dX GEMM per slab; ragged M, N and K, several tiles per CTA."""
    monkeypatch.setenv("LORA_GB300_MAX_CTAS", cap)
    if mode == "kscale":
        monkeypatch.setenv("LORA_GB300_DORA_KSCALE", "1")
    else:
        monkeypatch.setenv("LORA_GB300_DORA_SLAB_ROWS", "256")
    case = D.scaled(D.WORKLOADS["dora_4096x11008_bf16"], M=M, d_in=328, d_out=776, r=32)
    t = D.make_linear(case)
    g = {k: v.to(DEV) for k, v in t.items()}
    r0 = ops.dora_rownorm2(g["W0"])
    Y, Z, n, V = ops.dora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], r0, case.s, case.eps, g["bias"])
    X, W0, A, B, m, bias, dY = (f64(t[k]) for k in ("X", "W0", "A", "B", "m", "bias", "dY"))
    assert_close(Y, O.dora_linear_fwd(X, W0, A, B, m, case.s, case.eps, bias)[0], "bf16", "Y")
    dX, dA, dB, dm, _ = ops.dora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], g["m"], g["bias"], Y, Z, n, V, g["dY"],
                                            case.s, case.eps)
    rX, rA, rB, rm, _ = O.dora_linear_bwd(X, W0, A, B, m, case.s, dY, case.eps)
    assert_close(dX, rX, "bf16", "dX")
    assert_close(dA, rA, "bf16", "dA")
    assert_close(dB, rB, "bf16", "dB")
    assert_close(dm, rm[None], "bf16", "dm")
    _ws_ok(ops)


@pytest.mark.parametrize("I", [200, 384])
def test_mlp_swiglu(ops, variant, I, monkeypatch):
    monkeypatch.setenv("LORA_GB300_MAX_CTAS", "4")
    case = D.scaled(D.WORKLOADS["mlp_swiglu_4096x14336_bf16"], M=500, H=200, I=I, r=16, alpha=24.0)
    t = D.make_mlp(case)
    g = {k: v.to(DEV) for k, v in t.items()}
    P = {p: {"W": g["W" + p], "A": g["A" + p], "B": g["B" + p], "s": case.s} for p in "gud"}
    Y, saved = ops.lora_mlp_swiglu_fwd(g["X"], P["g"], P["u"], P["d"])
    args = tuple(x if isinstance(x, float) else f64(x) for x in
                 (t["X"], t["Wg"], t["Ag"], t["Bg"], case.s, t["Wu"], t["Au"], t["Bu"], case.s,
                  t["Wd"], t["Ad"], t["Bd"], case.s))
    ry, re, ru, rh = O.mlp_swiglu_fwd(*args)
    assert_close(saved["h"], rh, "bf16", "h")
    assert_close(Y, ry, "bf16", "y")
    gr = ops.lora_mlp_swiglu_bwd(g["X"], P["g"], P["u"], P["d"], saved, g["dY"])
    ref = O.mlp_swiglu_bwd(*args, f64(t["dY"]))
    for k in ("dX", "dAg", "dBu", "dAd"):
        assert_close(gr[k], ref[k], "bf16", k)
    _ws_ok(ops)


def test_qkv_multistep_tail(ops, variant, monkeypatch):
    """L r = 96: the rank-r tail of both GEMMs spans two K-steps (leaves in two groups)."""
    monkeypatch.setenv("LORA_GB300_MAX_CTAS", "4")
    case = D.scaled(D.WORKLOADS["qkv_lora_4096_gqa_bf16"], M=250, d_in=200, n=(256, 72, 72), r=32)
    t = D.make_qkv(case)
    g = {k: None if v is None else v.to(DEV) for k, v in t.items()}
    lg_ = [(g[f"A{l}"], g[f"B{l}"], case.s[l]) for l in range(3)]
    l64 = [(f64(t[f"A{l}"]), f64(t[f"B{l}"]), case.s[l]) for l in range(3)]
    Y, Z = ops.lora_qkv_fwd(g["X"], g["W0"], lg_)
    X, W0, dY = f64(t["X"]), f64(t["W0"]), f64(t["dY"])
    assert_close(Y, O.qkv_lora_fwd(X, W0, l64), "bf16", "Y")
    dX, dA, dB, _ = ops.lora_qkv_bwd(g["X"], g["W0"], lg_, Z, g["dY"])
    rX, rA, rB, _ = O.qkv_lora_bwd(X, W0, l64, dY)
    assert_close(dX, rX, "bf16", "dX")
    for i in range(3):
        assert_close(dA[i], rA[i], "bf16", f"dA{i}")
        assert_close(dB[i], rB[i], "bf16", f"dB{i}")
    _ws_ok(ops)


@pytest.mark.parametrize("slab_rows", [None, "128", "384"])
def test_dora_slab_copy_matches_kscale_bits(ops, variant, slab_rows, monkeypatch):
    """The slab copy of dY o c (bf16 of the fp32 product, as the scaling warps round it) and the
    in-GEMM scaling give the same dX bits, and with the same slab split of the column pass the same
    dA, dB, dm and dbias bits."""
    monkeypatch.setenv("LORA_GB300_MAX_CTAS", "6")
    if slab_rows:
        monkeypatch.setenv("LORA_GB300_DORA_SLAB_ROWS", slab_rows)
    case = D.scaled(D.WORKLOADS["dora_4096x11008_bf16"], M=900, d_in=264, d_out=536, r=16, bias=True)
    t = D.make_linear(case)
    g = {k: v.to(DEV) for k, v in t.items()}
    _, slab = _dora_bwd(ops, g, case)
    monkeypatch.setenv("LORA_GB300_DORA_KSCALE", "1")
    _, ks = _dora_bwd(ops, g, case)
    for a, b, nm in zip(slab, ks, ("dX", "dA", "dB", "dm", "dbias")):
        assert torch.equal(a, b), nm
    X, W0, A, B, m, bias, dY = (f64(t[k]) for k in ("X", "W0", "A", "B", "m", "bias", "dY"))
    ref = O.dora_linear_bwd(X, W0, A, B, m, case.s, dY, case.eps)
    for got, rr, nm in zip(slab, (ref[0], ref[1], ref[2], ref[3][None], ref[4][None]),
                           ("dX", "dA", "dB", "dm", "dbias")):
        assert_close(got, rr, "bf16", nm)
    _ws_ok(ops)


@pytest.mark.parametrize("cap", ["0", "4"])
@pytest.mark.parametrize("r", [8, 24, 32])
def test_dropout_masked_passes(ops, variant, cap, r, monkeypatch):
    """Input dropout with 16-byte mask rows: the Z pass and the dA pass read the mask beside X and
    form Xd in registers; ragged M, ranks 8-32, a capped grid."""
    monkeypatch.setenv("LORA_GB300_MAX_CTAS", cap)
    case = D.scaled(D.WORKLOADS["lora_4096_bf16"], M=410, d_in=400, d_out=264, r=r, bias=True)
    t = D.make_linear(case)
    g = {k: v.to(DEV) for k, v in t.items()}
    mk = D.make_dropout_mask(410, 400, 0.2)
    keep = 1 / 0.8
    Y, Z = ops.lora_linear_dropout_fwd(g["X"], mk.to(DEV), keep, g["W0"], g["A"], g["B"], case.s, g["bias"])
    X, W0, A, B = (f64(t[k]) for k in ("X", "W0", "A", "B"))
    assert_close(Y, O.lora_dropout_fwd(X, mk.numpy(), keep, W0, A, B, case.s, f64(t["bias"])), "bf16", "Y")
    dX, dA, dB, _ = ops.lora_linear_dropout_bwd(g["X"], mk.to(DEV), keep, g["W0"], g["A"], g["B"], None, g["dY"],
                                                case.s)
    rX, rA, rB, _ = O.lora_dropout_bwd(X, mk.numpy(), keep, W0, A, B, case.s, f64(t["dY"]))
    assert_close(dX, rX, "bf16", "dX")
    assert_close(dA, rA, "bf16", "dA")
    assert_close(dB, rB, "bf16", "dB")
    _ws_ok(ops)
