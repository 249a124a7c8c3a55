"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test checks the oracle against mathematics the pages fix: closed forms,
algebraic identities (fused form == materialised form), special cases that
reduce to a library routine, finite differences, brute force on tiny inputs,
and hand-worked examples under tests/golden/.  The checks are chosen so that a
dropped term, a wrong sign or index, or a transposed operand in the oracle
fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed=0):
    return np.random.default_rng(seed)


def rand_case(M=5, d_in=7, d_out=6, r=3, seed=0):
    g = rng(seed)
    X = g.standard_normal((M, d_in))
    W0 = g.standard_normal((d_out, d_in)) / np.sqrt(d_in)
    A = g.standard_normal((r, d_in)) / np.sqrt(d_in)
    B = g.standard_normal((d_out, r)) * 0.3
    bias = g.standard_normal(d_out) * 0.1
    m = np.sqrt((W0 * W0).sum(1)) * g.uniform(0.9, 1.1, d_out)
    dY = g.standard_normal((M, d_out))
    return X, W0, A, B, bias, m, dY


def rel(a, b):
    return np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(np.asarray(b)), 1e-300)


# ------------------------------------------------------------------ golden worked example
def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            vals[k] = np.array([float(x) for x in v])
    return vals


def test_golden_tiny_lora_dora():
    g = _read_golden("tiny_lora_dora.txt")
    X = g["X"].reshape(1, 2)
    W0 = g["W0"].reshape(2, 2)
    A = g["A"].reshape(1, 2)
    B = g["B"].reshape(2, 1)
    s = float(g["s"][0])
    y = O.lora_linear_fwd(X, W0, A, B, s, g["bias"])
    np.testing.assert_allclose(y[0], g["lora_y"], rtol=0, atol=1e-14)
    yd, n = O.dora_linear_fwd(X, W0, A, B, g["m"], s, 1e-12, g["bias"])
    np.testing.assert_allclose(n, g["dora_n"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(yd[0], g["dora_y"], rtol=0, atol=1e-14)


def test_golden_quantize_rows():
    rows, qs, scales = [], [], []
    with open(os.path.join(GOLD, "quantize_rows.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            x, q, sc = line.split("|")
            rows.append([float(v) for v in x.split()])
            qs.append([int(v) for v in q.split()])
            scales.append(float(sc))
    q, sc = O.quantize_rows(np.array(rows, dtype=np.float32))
    assert q.dtype == np.int8 and sc.dtype == np.float32
    np.testing.assert_array_equal(q, np.array(qs))
    np.testing.assert_array_equal(sc, np.array(scales, dtype=np.float32))


# ------------------------------------------------------------------ LoRA
def test_lora_fused_equals_materialised():
    """y = X W0^T + s (X A^T) B^T + bias is an exact refactoring of X W'^T + bias."""
    X, W0, A, B, bias, _, _ = rand_case(M=33, d_in=40, d_out=24, r=5, seed=1)
    s = 1.7
    fused = X @ W0.T + s * ((X @ A.T) @ B.T) + bias
    assert rel(O.lora_linear_fwd(X, W0, A, B, s, bias), fused) < 1e-13


def test_lora_init_reduces_to_library_linear():
    """B = 0 (standard LoRA init) -> the plain linear layer (torch.nn.functional.linear)."""
    X, W0, A, B, bias, _, _ = rand_case(seed=2)
    y = O.lora_linear_fwd(X, W0, A, np.zeros_like(B), 2.0, bias)
    ref = torch.nn.functional.linear(torch.from_numpy(X), torch.from_numpy(W0), torch.from_numpy(bias)).numpy()
    assert rel(y, ref) < 1e-14


def test_lora_strength_zero_bit_exact():
    X, W0, A, B, bias, _, _ = rand_case(seed=3)
    assert np.array_equal(O.lora_linear_fwd(X, W0, A, B, 0.0), X @ W0.T)


def _fd_grad(f, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + h
        fp = f()
        x[i] = old - h
        fm = f()
        x[i] = old
        g[i] = (fp - fm) / (2 * h)
    return g


def test_lora_grads_finite_difference():
    X, W0, A, B, bias, _, dY = rand_case(M=4, d_in=8, d_out=6, r=2, seed=4)
    s = 1.3
    L = lambda: float((dY * O.lora_linear_fwd(X, W0, A, B, s, bias)).sum())  # noqa: E731
    dX, dA, dB, dbias = O.lora_linear_bwd(X, W0, A, B, s, dY)
    for got, x in ((dX, X), (dA, A), (dB, B), (dbias, bias)):
        assert rel(got, _fd_grad(L, x)) < 1e-8


def test_lora_grads_match_library_autograd():
    X, W0, A, B, bias, _, dY = rand_case(M=9, d_in=12, d_out=10, r=3, seed=5)
    s = 0.7
    t = {k: torch.tensor(v, requires_grad=True) for k, v in dict(X=X, A=A, B=B, bias=bias).items()}
    y = torch.nn.functional.linear(t["X"], torch.tensor(W0) + s * t["B"] @ t["A"], t["bias"])
    y.backward(torch.tensor(dY))
    dX, dA, dB, dbias = O.lora_linear_bwd(X, W0, A, B, s, dY)
    for got, k in ((dX, "X"), (dA, "A"), (dB, "B"), (dbias, "bias")):
        assert rel(got, t[k].grad.numpy()) < 1e-13


# ------------------------------------------------------------------ LoRA with input dropout
def _drop_case(seed, p=0.25, **kw):
    X, W0, A, B, bias, _, dY = rand_case(seed=seed, **kw)
    mask = (rng(seed + 100).uniform(size=X.shape) >= p).astype(np.uint8)
    return X, mask, 1.0 / (1.0 - p), W0, A, B, bias, dY


def test_dropout_all_kept_unit_scale_is_lora():
    X, _, _, W0, A, B, bias, dY = _drop_case(20)
    ones = np.ones(X.shape, np.uint8)
    assert rel(O.lora_dropout_fwd(X, ones, 1.0, W0, A, B, 0.8, bias), O.lora_linear_fwd(X, W0, A, B, 0.8, bias)) < 1e-14
    for got, ref in zip(O.lora_dropout_bwd(X, ones, 1.0, W0, A, B, 0.8, dY), O.lora_linear_bwd(X, W0, A, B, 0.8, dY)):
        assert rel(got, ref) < 1e-14


def test_dropout_all_dropped_leaves_base_branch():
    """The mask acts on the adapter's input only: with every entry dropped the base branch and
    the bias remain, and the adapter factors get no gradient."""
    X, _, scale, W0, A, B, bias, dY = _drop_case(21)
    zeros = np.zeros(X.shape, np.uint8)
    assert np.array_equal(O.lora_dropout_fwd(X, zeros, scale, W0, A, B, 0.8, bias), X @ W0.T + bias[None, :])
    dX, dA, dB, dbias = O.lora_dropout_bwd(X, zeros, scale, W0, A, B, 0.8, dY)
    assert np.array_equal(dX, dY @ W0) and not dA.any() and not dB.any()
    assert np.allclose(dbias, dY.sum(0), rtol=0, atol=1e-14)


def test_dropout_grads_finite_difference():
    X, mask, scale, W0, A, B, bias, dY = _drop_case(22, M=4, d_in=8, d_out=6, r=2)
    s = 1.1
    L = lambda: float((dY * O.lora_dropout_fwd(X, mask, scale, W0, A, B, s, bias)).sum())  # noqa: E731
    for got, x in zip(O.lora_dropout_bwd(X, mask, scale, W0, A, B, s, dY), (X, A, B, bias)):
        assert rel(got, _fd_grad(L, x)) < 1e-8


def test_dropout_grads_match_library_autograd():
    """Library graph: base linear on X plus the adapter chain on X * mask * scale."""
    X, mask, scale, W0, A, B, bias, dY = _drop_case(23, M=9, d_in=12, d_out=10, r=3, p=0.4)
    s = 0.6
    t = {k: torch.tensor(v, requires_grad=True) for k, v in dict(X=X, A=A, B=B, bias=bias).items()}
    xd = t["X"] * (torch.tensor(mask, dtype=torch.float64) * scale)
    y = torch.nn.functional.linear(t["X"], torch.tensor(W0), t["bias"]) + s * torch.nn.functional.linear(
        torch.nn.functional.linear(xd, t["A"]), t["B"])
    y.backward(torch.tensor(dY))
    for got, k in zip(O.lora_dropout_bwd(X, mask, scale, W0, A, B, s, dY), ("X", "A", "B", "bias")):
        assert rel(got, t[k].grad.numpy()) < 1e-13


# ------------------------------------------------------------------ DoRA
def test_dora_closed_form_norm_equals_explicit():
    """||W0 + sBA||^2_row = rowsum(W0^2) + 2s rowsum((W0 A^T) o B) + s^2 rowsum((B (A A^T)) o B)."""
    _, W0, A, B, _, m, _ = rand_case(d_in=50, d_out=30, r=4, seed=6)
    s = 0.9
    q = O.dora_rownorm2(W0) + 2 * s * ((W0 @ A.T) * B).sum(1) + s * s * ((B @ (A @ A.T)) * B).sum(1)
    _, n = O.dora_linear_fwd(np.zeros((1, 50)), W0, A, B, m, s)
    assert rel(np.sqrt(q), n) < 1e-13


def test_dora_rownorm2_explicit_loop():
    W0 = rng(7).standard_normal((5, 9))
    want = [sum(W0[o, k] ** 2 for k in range(9)) for o in range(5)]
    np.testing.assert_allclose(O.dora_rownorm2(W0), want, rtol=1e-15)


def test_dora_at_init_is_plain_linear():
    """B = 0 and m = rownorm(W0) (DoRA init) -> torch.nn.functional.linear(X, W0, bias)."""
    X, W0, A, B, bias, _, _ = rand_case(seed=8)
    m = np.linalg.norm(W0, axis=1)
    y, _ = O.dora_linear_fwd(X, W0, A, np.zeros_like(B), m, 1.5, 1e-12, bias)
    ref = torch.nn.functional.linear(torch.from_numpy(X), torch.from_numpy(W0), torch.from_numpy(bias)).numpy()
    assert rel(y, ref) < 1e-14


def test_dora_is_row_scale_of_lora_output():
    """DoRA rows = diag(m/n) applied to the (base + low-rank) output, bias after."""
    X, W0, A, B, bias, m, _ = rand_case(seed=9)
    s = 0.8
    y, n = O.dora_linear_fwd(X, W0, A, B, m, s, 1e-12, bias)
    p = O.lora_linear_fwd(X, W0, A, B, s)
    assert rel(y, p * (m / n)[None, :] + bias) < 1e-14


def test_dora_direction_scale_invariance():
    """Scaling W0 and B by a > 0 scales W' and its norm alike: y is unchanged."""
    X, W0, A, B, bias, m, _ = rand_case(seed=10)
    y1, _ = O.dora_linear_fwd(X, W0, A, B, m, 1.1, 1e-12, bias)
    y2, _ = O.dora_linear_fwd(X, 3.0 * W0, A, 3.0 * B, m, 1.1, 1e-12, bias)
    assert rel(y2, y1) < 1e-14


def test_dora_strength_zero_is_frozen_base():
    X, W0, A, B, bias, m, dY = rand_case(seed=11)
    y, _ = O.dora_linear_fwd(X, W0, A, B, m, 0.0, 1e-12, bias)
    assert np.array_equal(y, X @ W0.T + bias)
    dX, dA, dB, dm, _ = O.dora_linear_bwd(X, W0, A, B, m, 0.0, dY)
    assert np.array_equal(dX, dY @ W0) and not dA.any() and not dB.any() and not dm.any()


def test_dora_grads_finite_difference():
    X, W0, A, B, bias, m, dY = rand_case(M=4, d_in=8, d_out=6, r=2, seed=12)
    s = 1.2
    L = lambda: float((dY * O.dora_linear_fwd(X, W0, A, B, m, s, 1e-12, bias)[0]).sum())  # noqa: E731
    dX, dA, dB, dm, dbias = O.dora_linear_bwd(X, W0, A, B, m, s, dY)
    for got, x in ((dX, X), (dA, A), (dB, B), (dm, m), (dbias, bias)):
        assert rel(got, _fd_grad(L, x)) < 1e-7


def test_dora_grads_match_library_autograd():
    X, W0, A, B, bias, m, dY = rand_case(M=7, d_in=11, d_out=9, r=3, seed=13)
    s = 0.6
    t = {k: torch.tensor(v, requires_grad=True) for k, v in dict(X=X, A=A, B=B, m=m, bias=bias).items()}
    Wp = torch.tensor(W0) + s * t["B"] @ t["A"]
    n = torch.linalg.vector_norm(Wp, dim=1).clamp_min(1e-12)
    y = torch.nn.functional.linear(t["X"], (t["m"] / n)[:, None] * Wp, t["bias"])
    y.backward(torch.tensor(dY))
    got = O.dora_linear_bwd(X, W0, A, B, m, s, dY)
    for g_, k in zip(got, ("X", "A", "B", "m", "bias")):
        assert rel(g_, t[k].grad.numpy()) < 1e-12


def test_golden_dora_eps_clamped_row():
    """A row whose adapted weight is exactly zero: its norm sits on the eps floor and no
    gradient flows through the norm there (hand-worked values)."""
    g = _read_golden("dora_eps_clamped_row.txt")
    X, W0, A, B = g["X"].reshape(1, 2), g["W0"].reshape(2, 2), g["A"].reshape(1, 2), g["B"].reshape(2, 1)
    s, eps, dY = float(g["s"][0]), float(g["eps"][0]), g["dY"].reshape(1, 2)
    y, n = O.dora_linear_fwd(X, W0, A, B, g["m"], s, eps, g["bias"])
    np.testing.assert_allclose(n, g["n"], rtol=1e-15, atol=0)
    np.testing.assert_allclose(y[0], g["y"], rtol=1e-15, atol=1e-15)
    dX, dA, dB, dm, dbias = O.dora_linear_bwd(X, W0, A, B, g["m"], s, dY, eps)
    for got, k in ((dX[0], "dX"), (dA[0], "dA"), (dB[:, 0], "dB"), (dm, "dm"), (dbias, "dbias")):
        np.testing.assert_allclose(got, g[k], rtol=1e-14, atol=1e-15, err_msg=k)
    sX, sA, sB, sm, _ = O.dora_bwd_sampled(X, W0, A, B, g["m"], s, dY, [0], [0, 1], [0, 1], eps)
    np.testing.assert_allclose(sA, dA, rtol=1e-14)
    np.testing.assert_allclose(sB, dB, rtol=1e-14)
    np.testing.assert_allclose(sm, dm, rtol=1e-14, atol=1e-15)


def _clamped_rows_case(seed, rows=(1, 4), shrink=0.05):
    """rand_case with some rows of W0 and B shrunk so that their adapted norm (~0.05) is below
    an eps of 0.3 while every other row (~1) is above it."""
    X, W0, A, B, bias, m, dY = rand_case(M=4, d_in=8, d_out=6, r=2, seed=seed)
    W0[list(rows)] *= shrink
    B[list(rows)] *= shrink
    return X, W0, A, B, bias, m, dY


def test_dora_eps_clamped_rows_finite_difference():
    """eps above some rows' norms: those rows take the floor (n = eps, no norm gradient) and the
    others stay live; finite differences of the clamped function agree with the oracle's
    gradients in both branches, and the sampled forms agree with the full ones."""
    X, W0, A, B, bias, m, dY = _clamped_rows_case(15)
    s, eps = 1.2, 0.3
    _, n = O.dora_linear_fwd(X, W0, A, B, m, s, eps, bias)
    nraw = np.linalg.norm(O.adapted_weight(W0, A, B, s), axis=1)
    assert (nraw[[1, 4]] < 0.2).all() and (np.delete(nraw, [1, 4]) > 0.5).all()
    assert (n[[1, 4]] == eps).all()
    L = lambda: float((dY * O.dora_linear_fwd(X, W0, A, B, m, s, eps, bias)[0]).sum())  # noqa: E731
    dX, dA, dB, dm, dbias = O.dora_linear_bwd(X, W0, A, B, m, s, dY, eps)
    for got, x in ((dX, X), (dA, A), (dB, B), (dm, m), (dbias, bias)):
        assert rel(got, _fd_grad(L, x)) < 1e-7
    sX, sA, sB, sm, _ = O.dora_bwd_sampled(X, W0, A, B, m, s, dY, [0, 3], list(range(8)), [1, 2, 4], eps)
    assert rel(sA, dA) < 1e-13 and rel(sB, dB[[1, 2, 4]]) < 1e-13 and rel(sm, dm) < 1e-13
    rX, rB, rm = O.dora_bwd_rows_sampled(X, W0, A, B, m, s, dY, [0, 3], [1, 2, 4], eps)
    assert rel(rX, dX[[0, 3]]) < 1e-13 and rel(rB, dB[[1, 2, 4]]) < 1e-13 and rel(rm, dm[[1, 2, 4]]) < 1e-13


def test_dora_eps_zero_row_matches_library_autograd():
    """A zero adapted row at eps = 1e-12, against torch autograd through clamp_min."""
    X, W0, A, B, bias, m, dY = rand_case(M=7, d_in=11, d_out=9, r=3, seed=16)
    W0[2] = 0.0
    B[2] = 0.0
    m[2] = 1.5
    s = 0.6
    t = {k: torch.tensor(v, requires_grad=True) for k, v in dict(X=X, A=A, B=B, m=m, bias=bias).items()}
    Wp = torch.tensor(W0) + s * t["B"] @ t["A"]
    n = torch.linalg.vector_norm(Wp, dim=1).clamp_min(1e-12)
    y = torch.nn.functional.linear(t["X"], (t["m"] / n)[:, None] * Wp, t["bias"])
    y.backward(torch.tensor(dY))
    got = O.dora_linear_bwd(X, W0, A, B, m, s, dY)
    for g_, k in zip(got, ("X", "A", "B", "m", "bias")):
        assert rel(g_, t[k].grad.numpy()) < 1e-12, k
    assert abs(got[2][2]).max() > 1e9      # the floor makes row 2's scale m / eps


# ------------------------------------------------------------------ DoRA (cols)
def cols_case(M=5, d_in=7, d_out=6, r=3, seed=40):
    X, W0, A, B, bias, _, dY = rand_case(M, d_in, d_out, r, seed)
    m = np.sqrt((W0 * W0).sum(0)) * rng(seed + 100).uniform(0.9, 1.1, d_in)
    return X, W0, A, B, bias, m, dY


def test_dora_cols_closed_form_norm_equals_explicit():
    """||W0 + sBA||^2_col = colsum(W0^2) + 2s colsum(A o (B^T W0)) + s^2 colsum(A o ((B^T B) A))."""
    _, W0, A, B, _, m, _ = cols_case(d_in=30, d_out=50, r=4, seed=41)
    s = 0.9
    q = O.dora_colnorm2(W0) + 2 * s * (A * (B.T @ W0)).sum(0) + s * s * (A * ((B.T @ B) @ A)).sum(0)
    _, n = O.dora_cols_fwd(np.zeros((1, 30)), W0, A, B, m, s)
    assert rel(np.sqrt(q), n) < 1e-13


def test_dora_colnorm2_explicit_loop():
    W0 = rng(42).standard_normal((5, 9))
    want = [sum(W0[o, k] ** 2 for o in range(5)) for k in range(9)]
    np.testing.assert_allclose(O.dora_colnorm2(W0), want, rtol=1e-15)


def test_dora_cols_is_transpose_of_rows_variant():
    """The column variant of (W0, A, B) is the row variant of the transposed problem
    (W0^T, B^T as the down factor, A^T as the up factor): feeding identity inputs
    returns each decomposed weight, and the two must be transposes of each other."""
    _, W0, A, B, _, m, _ = cols_case(d_in=8, d_out=11, r=3, seed=43)
    s = 1.3
    Wc, nc = O.dora_cols_fwd(np.eye(8), W0, A, B, m, s)          # = (W' diag(c))^T
    Wr, nr = O.dora_linear_fwd(np.eye(11), W0.T, B.T, A.T, m, s)  # = (diag(c) W'^T)^T
    assert rel(nc, nr) < 1e-14
    assert rel(Wc.T, Wr) < 1e-14


def test_dora_cols_at_init_is_plain_linear():
    X, W0, A, B, bias, _, _ = cols_case(seed=44)
    m = np.linalg.norm(W0, axis=0)
    y, _ = O.dora_cols_fwd(X, W0, A, np.zeros_like(B), m, 1.5, 1e-12, bias)
    ref = torch.nn.functional.linear(torch.from_numpy(X), torch.from_numpy(W0), torch.from_numpy(bias)).numpy()
    assert rel(y, ref) < 1e-14


def test_dora_cols_is_input_scale_of_lora():
    """DoRA cols = the LoRA layer applied to X diag(m / n)."""
    X, W0, A, B, bias, m, _ = cols_case(seed=45)
    s = 0.8
    y, n = O.dora_cols_fwd(X, W0, A, B, m, s, 1e-12, bias)
    assert rel(y, O.lora_linear_fwd(X * (m / n)[None, :], W0, A, B, s, bias)) < 1e-14


def test_dora_cols_direction_scale_invariance_and_strength_zero():
    X, W0, A, B, bias, m, dY = cols_case(seed=46)
    y1, _ = O.dora_cols_fwd(X, W0, A, B, m, 1.1, 1e-12, bias)
    y2, _ = O.dora_cols_fwd(X, 2.5 * W0, A, 2.5 * B, m, 1.1, 1e-12, bias)
    assert rel(y2, y1) < 1e-14
    y0, _ = O.dora_cols_fwd(X, W0, A, B, m, 0.0, 1e-12, bias)
    assert np.array_equal(y0, X @ W0.T + bias)
    dX, dA, dB, dm, _ = O.dora_cols_bwd(X, W0, A, B, m, 0.0, dY)
    assert np.array_equal(dX, dY @ W0) and not dA.any() and not dB.any() and not dm.any()


def test_dora_cols_grads_finite_difference():
    X, W0, A, B, bias, m, dY = cols_case(M=4, d_in=6, d_out=8, r=2, seed=47)
    s = 1.2
    L = lambda: float((dY * O.dora_cols_fwd(X, W0, A, B, m, s, 1e-12, bias)[0]).sum())  # noqa: E731
    dX, dA, dB, dm, db = O.dora_cols_bwd(X, W0, A, B, m, s, dY)
    for got, x in ((dX, X), (dA, A), (dB, B), (dm, m), (db, bias)):
        assert rel(got, _fd_grad(L, x)) < 1e-7


def test_dora_cols_grads_match_library_autograd():
    X, W0, A, B, bias, m, dY = cols_case(M=9, d_in=12, d_out=10, r=3, seed=48)
    s = 0.7
    t = {k: torch.tensor(v, requires_grad=True) for k, v in dict(X=X, A=A, B=B, m=m, bias=bias).items()}
    Wp = torch.tensor(W0) + s * t["B"] @ t["A"]
    n = torch.linalg.vector_norm(Wp, dim=0).clamp_min(1e-12)
    y = torch.nn.functional.linear(t["X"], Wp * (t["m"] / n)[None, :], t["bias"])
    y.backward(torch.tensor(dY))
    got = O.dora_cols_bwd(X, W0, A, B, m, s, dY)
    for g_, k in zip(got, ("X", "A", "B", "m", "bias")):
        assert rel(g_, t[k].grad.numpy()) < 1e-12, k


def test_dora_cols_eps_clamped_columns_finite_difference():
    """Column variant with eps above some columns' norms: floor branch and live branch both
    agree with finite differences, and the sampled forms with the full ones."""
    X, W0, A, B, bias, m, dY = cols_case(M=4, d_in=6, d_out=8, r=2, seed=50)
    W0[:, [1, 4]] *= 0.05
    A[:, [1, 4]] *= 0.05
    s, eps = 1.2, 0.3
    nraw = np.linalg.norm(O.adapted_weight(W0, A, B, s), axis=0)
    assert (nraw[[1, 4]] < 0.2).all() and (np.delete(nraw, [1, 4]) > 0.5).all()
    _, n = O.dora_cols_fwd(X, W0, A, B, m, s, eps, bias)
    assert (n[[1, 4]] == eps).all()
    L = lambda: float((dY * O.dora_cols_fwd(X, W0, A, B, m, s, eps, bias)[0]).sum())  # noqa: E731
    dX, dA, dB, dm, db = O.dora_cols_bwd(X, W0, A, B, m, s, dY, eps)
    for got, x in ((dX, X), (dA, A), (dB, B), (dm, m), (db, bias)):
        assert rel(got, _fd_grad(L, x)) < 1e-7
    sX, sA, sm = O.dora_cols_bwd_sampled(X, W0, A, B, m, s, dY, [0, 3], [1, 2, 4], eps)
    assert rel(sA, dA[:, [1, 2, 4]]) < 1e-13 and rel(sm, dm[[1, 2, 4]]) < 1e-13
    sB = O.dora_cols_bwd_rows_sampled(X, W0, A, B, m, s, dY, [0, 5, 7], eps)
    assert rel(sB, dB[[0, 5, 7]]) < 1e-13


def test_dora_cols_eps_zero_column_matches_library_autograd():
    X, W0, A, B, bias, m, dY = cols_case(M=9, d_in=12, d_out=10, r=3, seed=51)
    W0[:, 3] = 0.0
    A[:, 3] = 0.0
    m[3] = 1.5
    s = 0.7
    t = {k: torch.tensor(v, requires_grad=True) for k, v in dict(X=X, A=A, B=B, m=m, bias=bias).items()}
    Wp = torch.tensor(W0) + s * t["B"] @ t["A"]
    n = torch.linalg.vector_norm(Wp, dim=0).clamp_min(1e-12)
    y = torch.nn.functional.linear(t["X"], Wp * (t["m"] / n)[None, :], t["bias"])
    y.backward(torch.tensor(dY))
    got = O.dora_cols_bwd(X, W0, A, B, m, s, dY)
    for g_, k in zip(got, ("X", "A", "B", "m", "bias")):
        assert rel(g_, t[k].grad.numpy()) < 1e-12, k


def test_dora_cols_sampled_forms_match_full():
    X, W0, A, B, bias, m, dY = cols_case(M=9, d_in=12, d_out=10, r=3, seed=49)
    s = 0.9
    y, n = O.dora_cols_fwd(X, W0, A, B, m, s, 1e-12, bias)
    yr, nr = O.dora_cols_fwd_rows(X, W0, A, B, m, s, [1, 6], 1e-12, bias)
    assert rel(yr, y[[1, 6]]) < 1e-14 and rel(nr, n) == 0
    dX, dA, _, dm, _ = O.dora_cols_bwd(X, W0, A, B, m, s, dY)
    sX, sA, sm = O.dora_cols_bwd_sampled(X, W0, A, B, m, s, dY, [0, 8], [2, 3, 11])
    assert rel(sX, dX[[0, 8]]) < 1e-13 and rel(sA, dA[:, [2, 3, 11]]) < 1e-13 and rel(sm, dm[[2, 3, 11]]) < 1e-13
    _, _, dB, _, _ = O.dora_cols_bwd(X, W0, A, B, m, s, dY)
    assert rel(O.dora_cols_bwd_rows_sampled(X, W0, A, B, m, s, dY, [0, 4, 9]), dB[[0, 4, 9]]) < 1e-13


# ------------------------------------------------------------------ SwiGLU MLP
def mlp_case(M=4, H=6, I=8, r=2, seed=14):
    g = rng(seed)
    d = {"X": g.standard_normal((M, H))}
    for p, (o, i) in (("g", (I, H)), ("u", (I, H)), ("d", (H, I))):
        d["W" + p] = g.standard_normal((o, i)) / np.sqrt(i)
        d["A" + p] = g.standard_normal((r, i)) / np.sqrt(i)
        d["B" + p] = g.standard_normal((o, r)) * 0.3
    d["dY"] = g.standard_normal((M, H))
    return d


def _mlp_args(d, sg=1.1, su=0.9, sd=1.3):
    return (d["X"], d["Wg"], d["Ag"], d["Bg"], sg, d["Wu"], d["Au"], d["Bu"], su, d["Wd"], d["Ad"], d["Bd"], sd)


def test_silu_special_values_and_derivative():
    assert O.silu(np.array(0.0)) == 0.0
    np.testing.assert_allclose(O.silu(np.array([40.0, -40.0])), [40.0, 0.0], atol=1e-15)
    x = np.linspace(-6, 6, 25)
    fd = (O.silu(x + 1e-6) - O.silu(x - 1e-6)) / 2e-6
    np.testing.assert_allclose(O.dsilu(x), fd, rtol=1e-8, atol=1e-10)
    # library cross-check
    np.testing.assert_allclose(O.silu(x), torch.nn.functional.silu(torch.from_numpy(x)).numpy(), rtol=1e-15)


def test_mlp_fused_equals_materialised():
    d = mlp_case(M=9, H=10, I=12, r=3, seed=15)
    args = _mlp_args(d)
    y, e, u, h = O.mlp_swiglu_fwd(*args)
    X = d["X"]
    e2 = X @ d["Wg"].T + 1.1 * (X @ d["Ag"].T) @ d["Bg"].T
    u2 = X @ d["Wu"].T + 0.9 * (X @ d["Au"].T) @ d["Bu"].T
    h2 = e2 / (1 + np.exp(-e2)) * u2
    y2 = h2 @ d["Wd"].T + 1.3 * (h2 @ d["Ad"].T) @ d["Bd"].T
    for a, b in ((e, e2), (u, u2), (h, h2), (y, y2)):
        assert rel(a, b) < 1e-13


def test_mlp_grads_finite_difference():
    d = mlp_case(seed=16)
    args = list(_mlp_args(d))
    L = lambda: float((d["dY"] * O.mlp_swiglu_fwd(*args)[0]).sum())  # noqa: E731
    got = O.mlp_swiglu_bwd(*args, d["dY"])
    for key, idx in (("dX", 0), ("dAg", 2), ("dBg", 3), ("dAu", 6), ("dBu", 7), ("dAd", 10), ("dBd", 11)):
        assert rel(got[key], _fd_grad(L, args[idx])) < 1e-7, key


def test_mlp_grads_match_library_autograd():
    d = mlp_case(M=5, H=7, I=9, r=2, seed=17)
    t = {k: torch.tensor(v, requires_grad=True) for k, v in d.items()}
    s = dict(g=1.1, u=0.9, d=1.3)
    W = {p: t["W" + p].detach() + s[p] * t["B" + p] @ t["A" + p] for p in "gud"}
    e = t["X"] @ W["g"].T
    u = t["X"] @ W["u"].T
    y = (torch.nn.functional.silu(e) * u) @ W["d"].T
    y.backward(t["dY"].detach())
    got = O.mlp_swiglu_bwd(*_mlp_args(d), d["dY"])
    for key in ("dX", "dAg", "dBg", "dAu", "dBu", "dAd", "dBd"):
        assert rel(got[key], t[key[1:]].grad.numpy()) < 1e-12, key


# ------------------------------------------------------------------ GeGLU MLP
def test_gelu_special_values_and_derivative():
    # gelu(0) = 0, gelu(1) = Phi(1), gelu(x) -> x and -> 0 in the tails
    assert O.gelu(np.array(0.0)) == 0.0
    np.testing.assert_allclose(O.gelu(np.array(1.0)), 0.8413447460685429, rtol=1e-15)
    np.testing.assert_allclose(O.gelu(np.array([12.0, -12.0])), [12.0, 0.0], atol=1e-15)
    # Phi(-x) = 1 - Phi(x) gives gelu(x) - gelu(-x) = x
    x = np.linspace(-5, 5, 41)
    np.testing.assert_allclose(O.gelu(x) - O.gelu(-x), x, atol=1e-14)
    # derivative: dgelu(0) = 1/2, finite differences elsewhere
    assert O.dgelu(np.array(0.0)) == 0.5
    fd = (O.gelu(x + 1e-6) - O.gelu(x - 1e-6)) / 2e-6
    np.testing.assert_allclose(O.dgelu(x), fd, rtol=1e-8, atol=1e-10)
    # library cross-check (exact, erf-based variant)
    np.testing.assert_allclose(O.gelu(x), torch.nn.functional.gelu(torch.from_numpy(x)).numpy(), rtol=1e-14,
                               atol=1e-16)


def test_geglu_differs_from_swiglu_and_matches_explicit():
    d = mlp_case(M=6, H=8, I=10, r=2, seed=25)
    args = _mlp_args(d)
    y, e, u, h = O.mlp_swiglu_fwd(*args, act="geglu")
    h2 = np.array([[ev * 0.5 * (1 + math.erf(ev / math.sqrt(2))) for ev in row] for row in e]) * u
    assert rel(h, h2) < 1e-14
    assert rel(y, O.mlp_swiglu_fwd(*args)[0]) > 1e-2


def test_geglu_grads_finite_difference():
    d = mlp_case(seed=26)
    args = list(_mlp_args(d))
    L = lambda: float((d["dY"] * O.mlp_swiglu_fwd(*args, act="geglu")[0]).sum())  # noqa: E731
    got = O.mlp_swiglu_bwd(*args, d["dY"], act="geglu")
    for key, idx in (("dX", 0), ("dAg", 2), ("dBg", 3), ("dAu", 6), ("dBu", 7), ("dAd", 10), ("dBd", 11)):
        assert rel(got[key], _fd_grad(L, args[idx])) < 1e-7, key


def test_geglu_grads_match_library_autograd():
    d = mlp_case(M=5, H=7, I=9, r=2, seed=27)
    t = {k: torch.tensor(v, requires_grad=True) for k, v in d.items()}
    s = dict(g=1.1, u=0.9, d=1.3)
    W = {p: t["W" + p].detach() + s[p] * t["B" + p] @ t["A" + p] for p in "gud"}
    e = t["X"] @ W["g"].T
    u = t["X"] @ W["u"].T
    y = (torch.nn.functional.gelu(e) * u) @ W["d"].T
    y.backward(t["dY"].detach())
    got = O.mlp_swiglu_bwd(*_mlp_args(d), d["dY"], act="geglu")
    for key in ("dX", "dAg", "dBg", "dAu", "dBu", "dAd", "dBd"):
        assert rel(got[key], t[key[1:]].grad.numpy()) < 1e-12, key


# ------------------------------------------------------------------ fused-leaf (QKV)
def qkv_case(M=6, d_in=10, n=(8, 4, 4), r=2, seed=30):
    g = rng(seed)
    X = g.standard_normal((M, d_in))
    W0 = g.standard_normal((sum(n), d_in)) / np.sqrt(d_in)
    leaves = [(g.standard_normal((r, d_in)) / np.sqrt(d_in), g.standard_normal((nl, r)) * 0.3, 0.5 + 0.4 * i)
              for i, nl in enumerate(n)]
    bias = g.standard_normal(sum(n)) * 0.1
    dY = g.standard_normal((M, sum(n)))
    return X, W0, leaves, bias, dY


def test_qkv_fused_equals_per_leaf_low_rank_sum():
    """y[:, leaf l] = X W0[leaf l]^T + s_l (X A_l^T) B_l^T + bias, each leaf's B narrowed to its rows."""
    X, W0, leaves, bias, _ = qkv_case(M=11, d_in=16, n=(16, 8, 8), r=3, seed=31)
    cols, row = [], 0
    for A, B, s in leaves:
        n = B.shape[0]
        cols.append(X @ W0[row:row + n].T + s * ((X @ A.T) @ B.T))
        row += n
    assert rel(O.qkv_lora_fwd(X, W0, leaves, bias), np.concatenate(cols, axis=1) + bias) < 1e-13


def test_qkv_single_leaf_is_lora_linear():
    X, W0, leaves, bias, dY = qkv_case(n=(8,), seed=32)
    A, B, s = leaves[0]
    assert rel(O.qkv_lora_fwd(X, W0, leaves, bias), O.lora_linear_fwd(X, W0, A, B, s, bias)) < 1e-15
    dX, dA, dB, db = O.qkv_lora_bwd(X, W0, leaves, dY)
    rX, rA, rB, rb = O.lora_linear_bwd(X, W0, A, B, s, dY)
    for a, b in ((dX, rX), (dA[0], rA), (dB[0], rB), (db, rb)):
        assert rel(a, b) < 1e-15


def test_qkv_leaf_isolation_and_zero_strength():
    """A leaf's adapter touches only its own columns; strength 0 leaves them the frozen base, bit for bit."""
    X, W0, leaves, _, _ = qkv_case(seed=33)
    y = O.qkv_lora_fwd(X, W0, leaves)
    A1, B1, _ = leaves[1]
    changed = [leaves[0], (A1, B1 * 5.0, leaves[1][2]), leaves[2]]
    y2 = O.qkv_lora_fwd(X, W0, changed)
    assert np.array_equal(y[:, :8], y2[:, :8]) and np.array_equal(y[:, 12:], y2[:, 12:])
    assert not np.allclose(y[:, 8:12], y2[:, 8:12])
    off = [leaves[0], (A1, B1, 0.0), leaves[2]]
    assert np.array_equal(O.qkv_lora_fwd(X, W0, off)[:, 8:12], X @ W0[8:12].T)


def test_qkv_grads_finite_difference():
    X, W0, leaves, bias, dY = qkv_case(M=4, d_in=6, n=(8, 4, 4), r=2, seed=34)
    leaves = [(A.copy(), B.copy(), s) for A, B, s in leaves]
    L = lambda: float((dY * O.qkv_lora_fwd(X, W0, leaves, bias)).sum())  # noqa: E731
    dX, dA, dB, db = O.qkv_lora_bwd(X, W0, leaves, dY)
    assert rel(dX, _fd_grad(L, X)) < 1e-8
    assert rel(db, _fd_grad(L, bias)) < 1e-8
    for i, (A, B, _) in enumerate(leaves):
        assert rel(dA[i], _fd_grad(L, A)) < 1e-8, i
        assert rel(dB[i], _fd_grad(L, B)) < 1e-8, i


def test_qkv_grads_match_library_autograd():
    X, W0, leaves, bias, dY = qkv_case(M=7, d_in=12, n=(16, 8, 8), r=3, seed=35)
    tX = torch.tensor(X, requires_grad=True)
    tl = [(torch.tensor(A, requires_grad=True), torch.tensor(B, requires_grad=True), s) for A, B, s in leaves]
    Wp, row = [], 0
    for A, B, s in tl:
        Wp.append(torch.tensor(W0[row:row + B.shape[0]]) + s * B @ A)
        row += B.shape[0]
    y = torch.nn.functional.linear(tX, torch.cat(Wp), torch.tensor(bias))
    y.backward(torch.tensor(dY))
    dX, dA, dB, _ = O.qkv_lora_bwd(X, W0, leaves, dY)
    assert rel(dX, tX.grad.numpy()) < 1e-13
    for i, (A, B, _) in enumerate(tl):
        assert rel(dA[i], A.grad.numpy()) < 1e-13 and rel(dB[i], B.grad.numpy()) < 1e-13


def test_qkv_sampled_forms_match_full():
    X, W0, leaves, bias, dY = qkv_case(M=9, d_in=12, n=(16, 8, 8), r=3, seed=36)
    assert rel(O.qkv_fwd_rows(X, W0, leaves, [1, 7], bias), O.qkv_lora_fwd(X, W0, leaves, bias)[[1, 7]]) < 1e-14
    fX, fA, fB, _ = O.qkv_lora_bwd(X, W0, leaves, dY)
    orows = [[0, 15], [3], [2, 7]]
    sX, sA, sB = O.qkv_bwd_sampled(X, W0, leaves, dY, [2, 8], [0, 5, 11], orows)
    assert rel(sX, fX[[2, 8]]) < 1e-13
    for i in range(3):
        assert rel(sA[i], fA[i][:, [0, 5, 11]]) < 1e-13
        assert rel(sB[i], fB[i][orows[i]]) < 1e-13


# ------------------------------------------------------------------ W8A8
def test_quantize_rows_properties():
    x = (rng(18).standard_normal((20, 33)) * rng(19).uniform(0.01, 10, (20, 1))).astype(np.float32)
    x[3] = 0
    q, sc = O.quantize_rows(x)
    assert q.dtype == np.int8 and np.abs(q.astype(int)).max() <= 127
    live = sc > 0
    assert not live[3] and (q[3] == 0).all()
    # the row's absmax maps to +-127 and each code is within half a step of x / scale
    assert (np.abs(q[live]).max(1) == 127).all()
    err = np.abs(q[live].astype(np.float64) * sc[live, None] - x[live])
    assert (err <= sc[live, None] * (0.5 + 1e-5)).all()


def test_int8_accumulate_brute_force():
    g = rng(20)
    Xq = g.integers(-127, 128, (3, 5)).astype(np.int8)
    Wq = g.integers(-127, 128, (4, 5)).astype(np.int8)
    acc = O.int8_accumulate(Xq, Wq)
    for i, o in itertools.product(range(3), range(4)):
        assert acc[i, o] == sum(int(Xq[i, k]) * int(Wq[o, k]) for k in range(5))
    # worst case stays inside int32 at the W8A8 workload's depth (in = 3072)
    big = O.int8_accumulate(np.full((1, 3072), 127, np.int8), np.full((1, 3072), -127, np.int8))
    assert big[0, 0] == -3072 * 127 * 127 and abs(big[0, 0]) < 2 ** 31


def test_w8a8_epilogue_brute_force():
    g = rng(21)
    Xq = g.integers(-127, 128, (3, 6)).astype(np.int8)
    Wq = g.integers(-127, 128, (4, 6)).astype(np.int8)
    sx = g.uniform(0.01, 0.1, 3).astype(np.float32)
    sw = g.uniform(0.01, 0.1, 4).astype(np.float32)
    Z = g.standard_normal((3, 2))
    B = g.standard_normal((4, 2))
    bias = g.standard_normal(4)
    y, acc = O.w8a8_lora_fwd(Xq, sx, Wq, sw, Z, B, 0.5, bias)
    for i, o in itertools.product(range(3), range(4)):
        a = sum(int(Xq[i, k]) * int(Wq[o, k]) for k in range(6))
        want = a * float(sx[i]) * float(sw[o]) + 0.5 * sum(Z[i, j] * B[o, j] for j in range(2)) + bias[o]
        assert abs(y[i, o] - want) < 1e-12 * max(1, abs(want))


def test_w8a8_dequant_approximates_float_linear():
    """Dequantised int8 product approximates the float product X W0^T (sanity of scales)."""
    g = rng(22)
    X = g.standard_normal((16, 256)).astype(np.float32)
    W = (g.standard_normal((8, 256)) / 16).astype(np.float32)
    Xq, sx = O.quantize_rows(X)
    Wq, sw = O.quantize_rows(W)
    y, _ = O.w8a8_lora_fwd(Xq, sx, Wq, sw, np.zeros((16, 1)), np.zeros((8, 1)), 0.0)
    assert rel(y, X.astype(np.float64) @ W.T.astype(np.float64)) < 0.02


def test_w8a8_bwd_straight_through_finite_difference():
    """W8A8 backward = gradient of the layer with the activation quantiser as identity
    (straight-through): finite differences of X W_deq^T + s (X A^T) B^T + bias."""
    g = rng(25)
    M, K, N, r = 4, 8, 6, 2
    X = g.standard_normal((M, K))
    Wq = g.integers(-127, 128, (N, K)).astype(np.int8)
    sw = g.uniform(0.001, 0.01, N).astype(np.float32)
    A = g.standard_normal((r, K)) / 3
    B = g.standard_normal((N, r)) * 0.3
    bias = g.standard_normal(N) * 0.1
    dY = g.standard_normal((M, N))
    s = 0.75
    Wd = np.array([[float(sw[o]) * int(Wq[o, k]) for k in range(K)] for o in range(N)])  # written out
    L = lambda: float((dY * (X @ Wd.T + s * (X @ A.T) @ B.T + bias)).sum())  # noqa: E731
    dX, dA, dB, dbias = O.w8a8_lora_bwd(X, Wq, sw, A, B, s, dY)
    for got, x in ((dX, X), (dA, A), (dB, B), (dbias, bias)):
        assert rel(got, _fd_grad(L, x)) < 1e-8


# ------------------------------------------------------------------ sampled forms
def test_sampled_forms_match_full():
    X, W0, A, B, bias, m, dY = rand_case(M=40, d_in=24, d_out=18, r=4, seed=23)
    s = 1.4
    rows, cols, orows = [0, 7, 39], [1, 5, 23], [0, 17]
    dX, dA, dB, db = O.lora_linear_bwd(X, W0, A, B, s, dY)
    sX, sA, sB, sb = O.lora_bwd_sampled(X, W0, A, B, s, dY, rows, cols, orows)
    assert rel(sX, dX[rows]) < 1e-13 and rel(sA, dA[:, cols]) < 1e-13 and rel(sB, dB[orows]) < 1e-13
    assert rel(O.lora_fwd_rows(X, W0, A, B, s, rows, bias), O.lora_linear_fwd(X, W0, A, B, s, bias)[rows]) < 1e-14
    fX, fA, fB, fm, fb = O.dora_linear_bwd(X, W0, A, B, m, s, dY)
    gX, gA, gB, gm, gb = O.dora_bwd_sampled(X, W0, A, B, m, s, dY, rows, cols, orows)
    assert rel(gX, fX[rows]) < 1e-12 and rel(gA, fA[:, cols]) < 1e-12 and rel(gB, fB[orows]) < 1e-12
    assert rel(gm, fm) < 1e-12
    hX, hB, hm = O.dora_bwd_rows_sampled(X, W0, A, B, m, s, dY, rows, orows)
    assert rel(hX, fX[rows]) < 1e-12 and rel(hB, fB[orows]) < 1e-12 and rel(hm, fm[orows]) < 1e-12
    yf, nf = O.dora_linear_fwd(X, W0, A, B, m, s, 1e-12, bias)
    yr, nr = O.dora_fwd_rows(X, W0, A, B, m, s, rows, 1e-12, bias)
    assert rel(yr, yf[rows]) < 1e-14 and rel(nr, nf) == 0
    d = mlp_case(M=10, seed=24)
    args = _mlp_args(d)
    full = O.mlp_swiglu_fwd(*args)
    part = O.mlp_fwd_rows(*args, [2, 9])
    for a, b in zip(part, full):
        assert rel(a, b[[2, 9]]) < 1e-14
    assert rel(O.mlp_bwd_rows(*args, d["dY"], [2, 9]), O.mlp_swiglu_bwd(*args, d["dY"])["dX"][[2, 9]]) < 1e-13
