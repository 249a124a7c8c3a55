"""GPU parity at the workloads' full sizes (sampled outputs the oracle computes one by one),
and small problems run with a capped persistent grid so that every CTA of the tcgen05 GEMM
processes several tiles (ring wrap-around, both accumulator buffers, barrier phases)."""
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


def f64(t):
    return None if t is None else to64(t)


def gpu(t):
    return None if t is None else t.to(DEV).contiguous()


def ws_clear(ops):
    from dora_adapter_linear_gb300 import _lib as L
    for buf in ops._WS.values():
        assert L.lora_check_device_error(buf) == 0, "a kernel recorded a timed-out wait"


# ---------------------------------------------------------------------------- capped grid (persistence)
@pytest.fixture
def two_ctas(monkeypatch):
    monkeypatch.setenv("LORA_GB300_MAX_CTAS", "2")
    yield


def test_persistent_lora(ops, two_ctas):
    case = D.scaled(D.WORKLOADS["lora_4096_bf16"], M=520, d_in=392, d_out=776, r=16, bias=True)
    t = D.make_linear(case)
    g = {k: gpu(v) for k, v in t.items()}
    Y, Z = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], case.s, g["bias"])
    X, W0, A, B = (f64(t[k]) for k in ("X", "W0", "A", "B"))
    assert_close(Y, O.lora_linear_fwd(X, W0, A, B, case.s, f64(t["bias"])), "bf16", "Y")
    dX, dA, dB, _ = ops.lora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], Z, g["dY"], case.s)
    rX, rA, rB, _ = O.lora_linear_bwd(X, W0, A, B, case.s, f64(t["dY"]))
    assert_close(dX, rX, "bf16", "dX")
    assert_close(dA, rA, "bf16", "dA")
    assert_close(dB, rB, "bf16", "dB")
    ws_clear(ops)


def test_persistent_dora(ops, two_ctas):
    case = D.scaled(D.WORKLOADS["dora_4096x11008_bf16"], M=520, d_in=392, d_out=776, r=32)
    t = D.make_linear(case)
    g = {k: gpu(v) for k, v in t.items()}
    r0 = ops.dora_rownorm2(g["W0"])
    Y, Z, n, V = ops.dora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], r0, case.s, case.eps, g["bias"])
    X, W0, A, B, m, bias, dY = (f64(t[k]) for k in ("X", "W0", "A", "B", "m", "bias", "dY"))
    rY, _ = O.dora_linear_fwd(X, W0, A, B, m, case.s, case.eps, bias)
    assert_close(Y, rY, "bf16", "Y")
    dX, dA, dB, dm, _ = ops.dora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], g["m"], g["bias"], Y, Z, n, V, g["dY"],
                                            case.s, case.eps)
    rX, rA, rB, rm, _ = O.dora_linear_bwd(X, W0, A, B, m, case.s, dY, case.eps)
    for got, ref, nm in ((dX, rX, "dX"), (dA, rA, "dA"), (dB, rB, "dB"), (dm, rm[None], "dm")):
        assert_close(got, ref, "bf16", nm)
    ws_clear(ops)


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_persistent_mlp(ops, two_ctas, act):
    case = D.scaled(D.WORKLOADS["mlp_swiglu_4096x14336_bf16"], M=400, H=200, I=520, r=16, alpha=24.0)
    t = D.make_mlp(case)
    g = {k: gpu(v) for k, v in t.items()}
    P = {p: {"W": g["W" + p], "A": g["A" + p], "B": g["B" + p], "s": case.s} for p in "gud"}
    code = {"swiglu": 0, "geglu": 1}[act]
    Y, saved = ops.lora_mlp_swiglu_fwd(g["X"], P["g"], P["u"], P["d"], act=code)
    args = tuple(x if isinstance(x, float) else f64(x) for x in
                 (t["X"], t["Wg"], t["Ag"], t["Bg"], case.s, t["Wu"], t["Au"], t["Bu"], case.s,
                  t["Wd"], t["Ad"], t["Bd"], case.s))
    ry, re, ru, rh = O.mlp_swiglu_fwd(*args, act=act)
    assert_close(Y, ry, "bf16", "y")
    gr = ops.lora_mlp_swiglu_bwd(g["X"], P["g"], P["u"], P["d"], saved, g["dY"], act=code)
    ref = O.mlp_swiglu_bwd(*args, f64(t["dY"]), act=act)
    for k in ("dX", "dAg", "dBg", "dAu", "dBu", "dAd", "dBd"):
        assert_close(gr[k], ref[k], "bf16", k)
    ws_clear(ops)


# ---------------------------------------------------------------------------- full size, sampled
ROWS = [0, 1, 127, 128, 4095, 5000, 8191]


def test_full_lora_4096(ops):
    case = D.WORKLOADS["lora_4096_bf16"]
    t = D.make_linear(case)
    g = {k: gpu(v) for k, v in t.items()}
    Y, Z = ops.lora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], case.s)
    dX, dA, dB, _ = ops.lora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], Z, g["dY"], case.s)
    torch.cuda.synchronize()
    ws_clear(ops)
    X, W0, A, B, dY = (f64(t[k]) for k in ("X", "W0", "A", "B", "dY"))
    assert_close(Y[ROWS], O.lora_fwd_rows(X, W0, A, B, case.s, ROWS), "bf16", "Y rows")
    cols, orows = [0, 63, 64, 2047, 4095], [0, 255, 256, 3000, 4095]
    sX, sA, sB, _ = O.lora_bwd_sampled(X, W0, A, B, case.s, dY, ROWS, cols, orows)
    assert_close(dX[ROWS], sX, "bf16", "dX rows")
    assert_close(dA[:, cols].T, sA.T, "bf16", "dA columns")
    assert_close(dB[orows], sB, "bf16", "dB rows")


def test_full_lora_dropout_4096(ops):
    """The headline layer with input dropout (p = 0.1) at full size, the masked rank-r passes on the
    16-byte mask rows: rows of Y and dX (rows are independent), columns of dA (G does not depend
    on X, so the oracle on those columns of X, the mask, W0 and A gives them) and rows of dB (the
    oracle on those columns of dY and rows of W0 and B)."""
    case = D.WORKLOADS["lora_4096_bf16"]
    t = D.make_linear(case)
    g = {k: gpu(v) for k, v in t.items()}
    mk = D.make_dropout_mask(case.M, case.d_in, 0.1)
    keep = 1.0 / 0.9
    Y, Z = ops.lora_linear_dropout_fwd(g["X"], gpu(mk), keep, g["W0"], g["A"], g["B"], case.s)
    dX, dA, dB, _ = ops.lora_linear_dropout_bwd(g["X"], gpu(mk), keep, g["W0"], g["A"], g["B"], Z, g["dY"], case.s)
    torch.cuda.synchronize()
    ws_clear(ops)
    X, W0, A, B, dY = (f64(t[k]) for k in ("X", "W0", "A", "B", "dY"))
    m = mk.numpy()
    assert_close(Y[ROWS], O.lora_dropout_fwd(X[ROWS], m[ROWS], keep, W0, A, B, case.s), "bf16", "Y rows")
    rX = O.lora_dropout_bwd(X[ROWS], m[ROWS], keep, W0, A, B, case.s, dY[ROWS])[0]
    assert_close(dX[ROWS], rX, "bf16", "dX rows")
    cols, orows = [0, 63, 64, 2047, 4095], [0, 255, 256, 3000, 4095]
    rA = O.lora_dropout_bwd(X[:, cols], m[:, cols], keep, W0[:, cols], A[:, cols], B, case.s, dY)[1]
    assert_close(dA[:, cols].T, rA.T, "bf16", "dA columns")
    rB = O.lora_dropout_bwd(X, m, keep, W0[orows], A, B[orows], case.s, dY[:, orows])[2]
    assert_close(dB[orows], rB, "bf16", "dB rows")


def test_full_dora_4096x11008(ops):
    case = D.WORKLOADS["dora_4096x11008_bf16"]
    t = D.make_linear(case)
    g = {k: gpu(v) for k, v in t.items()}
    r0 = ops.dora_rownorm2(g["W0"])
    Y, Z, n, V = ops.dora_linear_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], r0, case.s, case.eps, g["bias"])
    dX, dA, dB, dm, _ = ops.dora_linear_bwd(g["X"], g["W0"], g["A"], g["B"], g["m"], g["bias"], Y, Z, n, V, g["dY"],
                                            case.s, case.eps)
    torch.cuda.synchronize()
    ws_clear(ops)
    X, W0, A, B, m, bias, dY = (f64(t[k]) for k in ("X", "W0", "A", "B", "m", "bias", "dY"))
    rY, rn = O.dora_fwd_rows(X, W0, A, B, m, case.s, ROWS, case.eps, bias)
    assert_close(Y[ROWS], rY, "bf16", "Y rows")
    np.testing.assert_allclose(to64(n), rn, rtol=1e-4)
    orows = [0, 255, 256, 5000, 11007]
    cols = [0, 1, 63, 64, 2047, 4095]
    sX, sA, sB, sm, _ = O.dora_bwd_sampled(X, W0, A, B, m, case.s, dY, ROWS, cols, orows, case.eps)
    assert_close(dX[ROWS], sX, "bf16", "dX rows")
    assert_close(dA[:, cols].T, sA.T, "bf16", "dA columns")
    assert_close(dB[orows], sB, "bf16", "dB rows")
    assert_close(dm[orows][None], sm[orows][None], "bf16", "dm entries")


def test_full_dora_cols(ops):
    case = D.WORKLOADS["dora_cols_4096x11008_bf16"]
    t = D.make_linear(case)
    g = {k: gpu(v) for k, v in t.items()}
    c0 = ops.dora_colnorm2(g["W0"])
    Y, Z, n, U = ops.dora_cols_fwd(g["X"], g["W0"], g["A"], g["B"], g["m"], c0, case.s, case.eps, g["bias"])
    dX, dA, dB, dm, _ = ops.dora_cols_bwd(g["X"], g["W0"], g["A"], g["B"], g["m"], Z, n, U, g["dY"], case.s,
                                          case.eps)
    torch.cuda.synchronize()
    ws_clear(ops)
    X, W0, A, B, m, bias, dY = (f64(t[k]) for k in ("X", "W0", "A", "B", "m", "bias", "dY"))
    ry, rn = O.dora_cols_fwd_rows(X, W0, A, B, m, case.s, ROWS, case.eps, bias)
    assert_close(Y[ROWS], ry, "bf16", "Y rows")
    np.testing.assert_allclose(to64(n), rn, rtol=1e-4)
    cols = [0, 1, 63, 64, 2047, 4095]
    sX, sA, sm = O.dora_cols_bwd_sampled(X, W0, A, B, m, case.s, dY, ROWS, cols, case.eps)
    assert_close(dX[ROWS], sX, "bf16", "dX rows")
    assert_close(dA[:, cols].T, sA.T, "bf16", "dA columns")
    assert_close(dm[cols][None], sm[None], "bf16", "dm entries")
    orows = [0, 255, 256, 5000, 11007]
    sB = O.dora_cols_bwd_rows_sampled(X, W0, A, B, m, case.s, dY, orows, case.eps)
    assert_close(dB[orows], sB, "bf16", "dB rows")


def test_full_mlp_swiglu(ops):
    case = D.WORKLOADS["mlp_swiglu_4096x14336_bf16"]
    t = D.make_mlp(case)
    g = {k: gpu(v) for k, v in t.items()}
    P = {p: {"W": g["W" + p], "A": g["A" + p], "B": g["B" + p], "s": case.s} for p in "gud"}
    Y, saved = ops.lora_mlp_swiglu_fwd(g["X"], P["g"], P["u"], P["d"])
    gr = ops.lora_mlp_swiglu_bwd(g["X"], P["g"], P["u"], P["d"], saved, g["dY"])
    torch.cuda.synchronize()
    ws_clear(ops)
    rows = [0, 1, 8191, 16383]
    args = tuple(x if isinstance(x, float) else f64(x) for x in
                 (t["X"], t["Wg"], t["Ag"], t["Bg"], case.s, t["Wu"], t["Au"], t["Bu"], case.s,
                  t["Wd"], t["Ad"], t["Bd"], case.s))
    ry, re, ru, rh = O.mlp_fwd_rows(*args, rows)
    assert_close(saved["e"][rows], re, "bf16", "e rows")
    assert_close(saved["u"][rows], ru, "bf16", "u rows")
    assert_close(saved["h"][rows], rh, "bf16", "h rows")
    assert_close(Y[rows], ry, "bf16", "y rows")
    assert_close(gr["dX"][rows], O.mlp_bwd_rows(*args, f64(t["dY"]), rows), "bf16", "dX rows")
    # Adapter gradients at full size: every gradient is linear in dY and each token row adds its
    # own share, so with a dY that is zero outside a spread of sampled rows the oracle needs only
    # those rows, while the kernels run the full-size launch (all row splits and tiles).
    sparse = sorted({int(i) for i in np.linspace(0, case.M - 1, 48)} | {1, 127, 128, 8191})
    dYs = torch.zeros_like(t["dY"])
    dYs[sparse] = t["dY"][sparse]
    gs = ops.lora_mlp_swiglu_bwd(g["X"], P["g"], P["u"], P["d"], saved, gpu(dYs))
    torch.cuda.synchronize()
    ws_clear(ops)
    ref = O.mlp_bwd_sparse_dy(*args, f64(dYs), sparse)
    for k in ("dAg", "dBg", "dAu", "dBu", "dAd", "dBd"):
        assert_close(gs[k], ref[k], "bf16", k)
    assert_close(gs["dX"][sparse], ref["dX"], "bf16", "dX rows (sparse dY)")
    others = [i for i in (2, 5000, 16382) if i not in sparse]
    assert not gs["dX"][others].any(), "dX rows where dY vanishes must be zero"


def test_full_qkv_gqa(ops):
    case = D.WORKLOADS["qkv_lora_4096_gqa_bf16"]
    t = D.make_qkv(case)
    g = {k: gpu(v) for k, v in t.items()}
    leaves = [(g[f"A{l}"], g[f"B{l}"], case.s[l]) for l in range(3)]
    Y, Z = ops.lora_qkv_fwd(g["X"], g["W0"], leaves)
    dX, dA, dB, _ = ops.lora_qkv_bwd(g["X"], g["W0"], leaves, Z, g["dY"])
    torch.cuda.synchronize()
    ws_clear(ops)
    l64 = [(f64(t[f"A{l}"]), f64(t[f"B{l}"]), case.s[l]) for l in range(3)]
    X, W0, dY = f64(t["X"]), f64(t["W0"]), f64(t["dY"])
    rows = [0, 1, 127, 128, 8191, 16383]
    assert_close(Y[rows], O.qkv_fwd_rows(X, W0, l64, rows), "bf16", "Y rows")
    cols = [0, 63, 64, 2047, 4095]
    orows = [[0, 255, 4095], [0, 1023], [1, 1000]]
    sX, sA, sB = O.qkv_bwd_sampled(X, W0, l64, dY, rows, cols, orows)
    assert_close(dX[rows], sX, "bf16", "dX rows")
    for l in range(3):
        assert_close(dA[l][:, cols].T, sA[l].T, "bf16", f"dA{l} cols")
        assert_close(dB[l][orows[l]], sB[l], "bf16", f"dB{l} rows")


def test_full_w8a8_3072(ops):
    case = D.WORKLOADS["w8a8_lora_3072"]
    t = D.make_w8a8(case)
    Wq, sw = O.quantize_rows(t["W0"].numpy())
    X = gpu(t["X"])
    Xq, sx, Z = ops.w8a8_quantize_rows(X, gpu(t["A"]))
    Y, acc = ops.w8a8_lora_fwd(Xq, sx, gpu(torch.from_numpy(Wq)), gpu(torch.from_numpy(sw)), Z, gpu(t["B"]), case.s,
                               want_acc=True)
    torch.cuda.synchronize()
    rows = [0, 1, 777, 16383]
    rq, rs = O.quantize_rows(t["X"][rows].float().numpy())
    np.testing.assert_array_equal(Xq[rows].cpu().numpy(), rq)
    np.testing.assert_array_equal(sx[rows].cpu().numpy(), rs)
    racc = O.int8_accumulate(rq, Wq)
    np.testing.assert_array_equal(acc[rows].cpu().numpy().astype(np.int64), racc)
    Zr = f64(t["X"][rows]) @ f64(t["A"]).T
    assert_close(Z[rows], Zr, "bf16", "Z rows")
    ry, _ = O.w8a8_lora_fwd(rq, rs, Wq, sw, Zr, f64(t["B"]), case.s, acc=racc)
    assert_close(Y[rows], ry, "bf16", "Y rows")
    # backward through the int8 base, sampled rows / columns of the gradients
    g = torch.Generator().manual_seed(78)
    dY = torch.randn(case.M, case.d_out, generator=g).to(torch.bfloat16)
    dX, dA, dB, _ = ops.w8a8_lora_bwd(X, gpu(torch.from_numpy(Wq)), gpu(torch.from_numpy(sw)), gpu(t["A"]),
                                      gpu(t["B"]), Z, gpu(dY), case.s)
    torch.cuda.synchronize()
    cols, orows = [0, 1000, 3071], [0, 1500, 3071]
    sX, sA, sB, _ = O.lora_bwd_sampled(f64(t["X"]), O.w8a8_dequant_weight(Wq, sw), f64(t["A"]), f64(t["B"]), case.s,
                                       f64(dY), rows, cols, orows)
    assert_close(dX[rows], sX, "bf16", "dX rows")
    assert_close(dA[:, cols].T, sA.T, "bf16", "dA columns")
    assert_close(dB[orows], sB, "bf16", "dB rows")
