"""Plain, slow, fp64 CPU oracle of the low-rank-adapted linear layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the C-ABI library and
its Python binding) imports this file; it is used by the tests, by the smoke
check and by the benchmark's CPU-baseline leg.

Every function computes the *materialised* form: it builds the adapted weight
W' = W0 + s*B*A explicitly (an [out, in] matrix) and then does an ordinary
linear layer with it.  The GPU path never builds W'; the two agree because the
fused form is an exact algebraic refactoring of this one ("LoRA/DoRA fast
forward: no weight materialization", What section: the same y is computed
without building an [out, in] tensor).  Gradients are derived here by the
chain rule in weight space (dW' = dY^T X, then through W' = W0 + s B A), a
deliberately different route from the fused backward formulas of the kernels.

Shapes (row-major): X [M, in], W0 [out, in], A [r, in] (down), B [out, r] (up),
bias [out], m [out], dY [M, out].  s = strength * alpha / r.

numpy's matmul (BLAS) and scipy's erf (for GELU) are the only library primitives used; all arrays are
float64 unless a function says otherwise.
"""
from __future__ import annotations

import numpy as np
from scipy.special import erf as _erf

__all__ = [
    "f64", "adapted_weight", "lora_linear_fwd", "lora_linear_bwd", "dora_rownorm2",
    "dora_linear_fwd", "dora_linear_bwd", "dora_colnorm2", "dora_cols_fwd", "dora_cols_bwd",
    "dora_cols_fwd_rows", "dora_cols_bwd_sampled", "dora_cols_bwd_rows_sampled", "silu", "dsilu", "gelu", "dgelu", "mlp_swiglu_fwd", "mlp_swiglu_bwd",
    "quantize_rows", "int8_accumulate", "w8a8_lora_fwd", "w8a8_dequant_weight", "w8a8_lora_bwd",
    "lora_dropout_fwd", "lora_dropout_bwd", "qkv_adapted_weight", "qkv_lora_fwd", "qkv_lora_bwd", "qkv_fwd_rows", "qkv_bwd_sampled",
    "lora_fwd_rows", "lora_bwd_sampled", "dora_fwd_rows", "dora_bwd_sampled", "dora_bwd_rows_sampled",
    "mlp_fwd_rows", "mlp_bwd_rows", "mlp_bwd_sparse_dy",
]


def f64(t):
    """Upcast a CPU tensor / array (any float dtype, incl. bf16) to a float64 ndarray."""
    if t is None:
        return None
    if hasattr(t, "detach"):  # torch tensor
        import torch
        return t.detach().to(torch.float64).cpu().numpy()
    return np.asarray(t, dtype=np.float64)


def adapted_weight(W0, A, B, s):
    """W' = W0 + s * B @ A  -- the materialised low-rank update.

    "How Unsloth's FastLoRA Kernel Differs ...", Fused Forward Pass Architecture
    (the weight update written out as a dense [out, in] matrix, the standard
    form the fused kernels avoid); orientation A [r, in], B [out, r] as the
    lora_down / lora_up pair of "nunchaku-style kernel fusion" (#1680).
    """
    return W0 + s * (B @ A)


# ----------------------------------------------------------------------------- LoRA
def lora_linear_fwd(X, W0, A, B, s, bias=None):
    """y = X W'^T (+ bias), W' = W0 + s B A.

    "LoRA/DoRA fast forward: no weight materialization", What section (the
    low-rank update folded into the data GEMM gives the same y).
    """
    Y = X @ adapted_weight(W0, A, B, s).T
    if bias is not None:
        Y = Y + bias[None, :]
    return Y


def lora_linear_bwd(X, W0, A, B, s, dY):
    """Gradients of y = X W'^T + bias w.r.t. X, A, B and bias (W0 frozen).

    Chain rule through the materialised weight:
      dX = dY W',  dW' = dY^T X,  dA = s B^T dW',  dB = s dW' A^T,  dbias = colsum(dY).
    "How Unsloth's FastLoRA Kernel Differs ...", Custom Backward Pass
    Implementation (dA, dB carry the scaling s).
    """
    Wp = adapted_weight(W0, A, B, s)
    dX = dY @ Wp
    dWp = dY.T @ X
    dA = s * (B.T @ dWp)
    dB = s * (dWp @ A.T)
    dbias = dY.sum(axis=0)
    return dX, dA, dB, dbias


# ----------------------------------------------------------------------------- LoRA with input dropout
def lora_dropout_fwd(X, mask, keep_scale, W0, A, B, s, bias=None):
    """y = X W0^T + s (Xd A^T) B^T (+ bias) with Xd = X o mask * keep_scale.

    The adapter branch sees the dropped-out input and the base branch the plain one, as with a
    dropout layer in front of the down-projection ("How Unsloth's FastLoRA Kernel Differs ...",
    Optimized Dropout and Scaling; "Fused Kernels (experimental)": a call whose mask sits between
    two factors takes the unfused path).  The mask is an input (drawn by the caller).
    """
    Xd = X * (np.asarray(mask, dtype=np.float64) * keep_scale)
    Y = X @ W0.T + s * ((Xd @ A.T) @ B.T)
    if bias is not None:
        Y = Y + bias[None, :]
    return Y


def lora_dropout_bwd(X, mask, keep_scale, W0, A, B, s, dY):
    """Gradients of lora_dropout_fwd w.r.t. X, A, B and bias (W0 frozen).

    With D = diag-free elementwise factor mask * keep_scale: dX = dY W0 + (s (dY B) A) o D,
    dA = s (dY B)^T Xd, dB = s dY^T (Xd A^T), dbias = colsum(dY).
    """
    D = np.asarray(mask, dtype=np.float64) * keep_scale
    Xd = X * D
    G = s * (dY @ B)
    return dY @ W0 + (G @ A) * D, G.T @ Xd, s * (dY.T @ (Xd @ A.T)), dY.sum(axis=0)


# ----------------------------------------------------------------------------- fused-leaf (QKV)
def qkv_adapted_weight(W0, leaves):
    """The fused projection's adapted weight, leaf by leaf.

    W0 [N, in] stacks the leaves' base rows in order; leaf l = (A_l [r, in],
    B_l [n_l, r], s_l) adapts only its own rows: W'[leaf l] = W0[leaf l] + s_l B_l A_l.
    "How Unsloth's FastLoRA Kernel Differs ...", Fused Forward Pass Architecture
    (LoRA_QKV) and "nunchaku-style kernel fusion" (#1680: fused-qkv adapters, each
    lora_up narrowed to its leaf's rows).
    """
    parts, row = [], 0
    for A, B, s in leaves:
        n = B.shape[0]
        parts.append(adapted_weight(W0[row:row + n], A, B, s))
        row += n
    assert row == W0.shape[0], "leaf rows must cover W0"
    return np.concatenate(parts, axis=0)


def qkv_lora_fwd(X, W0, leaves, bias=None):
    """y = X W'^T (+ bias) with the leaf-wise adapted fused weight."""
    Y = X @ qkv_adapted_weight(W0, leaves).T
    if bias is not None:
        Y = Y + bias[None, :]
    return Y


def qkv_lora_bwd(X, W0, leaves, dY):
    """Gradients of qkv_lora_fwd (W0 frozen): dX = dY W', dW' = dY^T X and, per leaf,
    dA_l = s_l B_l^T dW'[leaf l], dB_l = s_l dW'[leaf l] A_l^T; dbias = colsum(dY)."""
    Wp = qkv_adapted_weight(W0, leaves)
    dX = dY @ Wp
    dWp = dY.T @ X
    dA, dB, row = [], [], 0
    for A, B, s in leaves:
        n = B.shape[0]
        dA.append(s * (B.T @ dWp[row:row + n]))
        dB.append(s * (dWp[row:row + n] @ A.T))
        row += n
    return dX, dA, dB, dY.sum(axis=0)


# ----------------------------------------------------------------------------- DoRA
def dora_rownorm2(W0):
    """rowsum(W0^2): the per-layer cached constant of the closed-form DoRA norm.

    "LoRA/DoRA fast forward ...", commit message (a cached rowsum(W0^2) constant)
    and What section (the cached norm constant is a per-layer vector).
    """
    return (W0 * W0).sum(axis=1)


def _dora_norm(Wp, eps):
    """Explicit row norm of the adapted weight, clamped below at eps.

    The pages fix eps = 1e-12 but not its placement; the clamp max(||.||, eps)
    is the reading taken (it matches a normalise-by-norm with a floor).
    """
    nraw = np.sqrt((Wp * Wp).sum(axis=1))
    return np.maximum(nraw, eps), nraw


def dora_linear_fwd(X, W0, A, B, m, s, eps=1e-12, bias=None):
    """DoRA rows: y = X (diag(m / n) W')^T + bias, n = max(||W'_o||_2, eps).

    "LoRA/DoRA fast forward ...", What section: dora-rows is a row scale of the
    (base + low-rank) output; Fidelity section: the bias is added un-scaled
    after the row scale.  Here the norm is taken explicitly, row by row, on the
    materialised W' (the kernels use the closed-form expansion instead).
    Strength 0 short-circuits to the frozen base X W0^T + bias (commit message:
    strength==0 short-circuit; Fidelity: bit-exact vs the frozen base).
    Returns (y, n).
    """
    Wp = adapted_weight(W0, A, B, s)
    n, _ = _dora_norm(Wp, eps)
    if s == 0:
        Y = X @ W0.T
        return (Y if bias is None else Y + bias[None, :]), n
    Wd = (m / n)[:, None] * Wp
    Y = X @ Wd.T
    if bias is not None:
        Y = Y + bias[None, :]
    return Y, n


def dora_linear_bwd(X, W0, A, B, m, s, dY, eps=1e-12):
    """Gradients of DoRA rows w.r.t. X, A, B, m and bias, norm kept in the graph.

    "LoRA/DoRA fast forward ...", Fidelity section: the norm stays in the
    autograd graph (no detach), gradients for A, B and the magnitude.
    Weight-space chain rule: with Wd = diag(c) W', c = m / n,
      dWd = dY^T X,  t_o = <dWd_o, W'_o>,  dm = t / n,
      dW' = diag(c) dWd - diag(t m / (n^2 nraw)) W'   (second term 0 where n was clamped),
      dA = s B^T dW',  dB = s dW' A^T,  dX = dY Wd,  dbias = colsum(dY).
    At strength 0 the layer is the frozen base: dX = dY W0, dA = dB = dm = 0.
    """
    if s == 0:
        z = np.zeros
        return dY @ W0, z(A.shape), z(B.shape), z(m.shape), dY.sum(axis=0)
    Wp = adapted_weight(W0, A, B, s)
    n, nraw = _dora_norm(Wp, eps)
    c = m / n
    Wd = c[:, None] * Wp
    dX = dY @ Wd
    dWd = dY.T @ X
    t = (dWd * Wp).sum(axis=1)
    dm = t / n
    dn = -t * m / (n * n)
    live = nraw > eps
    dnraw = np.where(live, dn, 0.0)
    dWp = c[:, None] * dWd + np.where(live, dnraw / np.where(live, nraw, 1.0), 0.0)[:, None] * Wp
    dA = s * (B.T @ dWp)
    dB = s * (dWp @ A.T)
    dbias = dY.sum(axis=0)
    return dX, dA, dB, dm, dbias


# ----------------------------------------------------------------------------- DoRA (cols)
def dora_colnorm2(W0):
    """colsum(W0^2): the cached constant of the column variant's closed-form norm.

    "LoRA/DoRA fast forward ...", commit message (row/col norm from the closed-form
    norm^2 expansion with a cached constant).
    """
    return (W0 * W0).sum(axis=0)


def dora_cols_fwd(X, W0, A, B, m, s, eps=1e-12, bias=None):
    """DoRA cols: y = X (W' diag(m / n))^T + bias, n[k] = max(||W'[:, k]||_2, eps), m [in].

    "LoRA/DoRA fast forward ...", What section (dora-cols, like dora-rows, needs no
    materialised weight) and Fidelity section (in-graph norm, 1e-12 eps, un-scaled
    bias, strength 0 = frozen base).  The norm is taken explicitly, column by column,
    on the materialised W'.  Returns (y, n).
    """
    Wp = adapted_weight(W0, A, B, s)
    n = np.maximum(np.sqrt((Wp * Wp).sum(axis=0)), eps)
    if s == 0:
        Y = X @ W0.T
        return (Y if bias is None else Y + bias[None, :]), n
    Y = X @ (Wp * (m / n)[None, :]).T
    if bias is not None:
        Y = Y + bias[None, :]
    return Y, n


def dora_cols_bwd(X, W0, A, B, m, s, dY, eps=1e-12):
    """Gradients of DoRA cols w.r.t. X, A, B, m and bias, norm kept in the graph.

    Weight-space chain rule with Wd = W' diag(c), c = m / n:
      dWd = dY^T X,  t_k = <dWd[:, k], W'[:, k]>,  dm = t / n,
      dW' = dWd diag(c) - W' diag(t m / (n^2 nraw))   (second term 0 where n was clamped),
      dA = s B^T dW',  dB = s dW' A^T,  dX = dY Wd,  dbias = colsum(dY).
    Strength 0: the frozen base (dX = dY W0, dA = dB = dm = 0).
    """
    if s == 0:
        z = np.zeros
        return dY @ W0, z(A.shape), z(B.shape), z(m.shape), dY.sum(axis=0)
    Wp = adapted_weight(W0, A, B, s)
    nraw = np.sqrt((Wp * Wp).sum(axis=0))
    n = np.maximum(nraw, eps)
    c = m / n
    Wd = Wp * c[None, :]
    dX = dY @ Wd
    dWd = dY.T @ X
    t = (dWd * Wp).sum(axis=0)
    dm = t / n
    live = nraw > eps
    coef = np.where(live, (-t * m / (n * n)) / np.where(live, nraw, 1.0), 0.0)
    dWp = dWd * c[None, :] + Wp * coef[None, :]
    return dX, s * (B.T @ dWp), s * (dWp @ A.T), dm, dY.sum(axis=0)


# ----------------------------------------------------------------------------- SwiGLU MLP
def silu(x):
    """silu(x) = x * sigmoid(x) = x / (1 + exp(-x))."""
    return x / (1.0 + np.exp(-x))


def dsilu(x):
    """d silu / dx = sigmoid(x) * (1 + x * (1 - sigmoid(x)))."""
    sg = 1.0 / (1.0 + np.exp(-x))
    return sg * (1.0 + x * (1.0 - sg))


def gelu(x):
    """Exact GELU: gelu(x) = x * Phi(x), Phi the standard normal CDF = (1 + erf(x / sqrt 2)) / 2."""
    return x * 0.5 * (1.0 + _erf(x / np.sqrt(2.0)))


def dgelu(x):
    """d gelu / dx = Phi(x) + x * phi(x), phi(x) = exp(-x^2 / 2) / sqrt(2 pi)."""
    return 0.5 * (1.0 + _erf(x / np.sqrt(2.0))) + x * np.exp(-0.5 * x * x) / np.sqrt(2.0 * np.pi)


GATE_ACTS = {"swiglu": (silu, dsilu), "geglu": (gelu, dgelu)}


def mlp_swiglu_fwd(X, Wg, Ag, Bg, sg, Wu, Au, Bu, su, Wd, Ad, Bd, sd, act="swiglu"):
    """LoRA gated MLP forward with each projection's adapter materialised.

    "How Unsloth's FastLoRA Kernel Differs ...", Fused Forward Pass
    Architecture and Activation Function Fusion: e = X Wg'^T, u = X Wu'^T,
    h = act(e) * u, y = h Wd'^T, act = silu (SwiGLU) or gelu (GeGLU).
    Returns (y, e, u, h).
    """
    f, _ = GATE_ACTS[act]
    e = X @ adapted_weight(Wg, Ag, Bg, sg).T
    u = X @ adapted_weight(Wu, Au, Bu, su).T
    h = f(e) * u
    y = h @ adapted_weight(Wd, Ad, Bd, sd).T
    return y, e, u, h


def mlp_swiglu_bwd(X, Wg, Ag, Bg, sg, Wu, Au, Bu, su, Wd, Ad, Bd, sd, dY, act="swiglu"):
    """Backward of the LoRA gated MLP (base weights frozen).

    "How Unsloth's FastLoRA Kernel Differs ...", Custom Backward Pass
    Implementation (down, up and gate adapter gradients, each pre-scaled).
    Returns dict with dX, dAg, dBg, dAu, dBu, dAd, dBd.
    """
    Wgp = adapted_weight(Wg, Ag, Bg, sg)
    Wup = adapted_weight(Wu, Au, Bu, su)
    Wdp = adapted_weight(Wd, Ad, Bd, sd)
    f, df = GATE_ACTS[act]
    e = X @ Wgp.T
    u = X @ Wup.T
    h = f(e) * u
    dh = dY @ Wdp
    dWdp = dY.T @ h
    de = dh * u * df(e)
    du = dh * f(e)
    dX = de @ Wgp + du @ Wup
    dWgp = de.T @ X
    dWup = du.T @ X
    return {
        "dX": dX,
        "dAg": sg * (Bg.T @ dWgp), "dBg": sg * (dWgp @ Ag.T),
        "dAu": su * (Bu.T @ dWup), "dBu": su * (dWup @ Au.T),
        "dAd": sd * (Bd.T @ dWdp), "dBd": sd * (dWdp @ Ad.T),
    }


# ----------------------------------------------------------------------------- W8A8
def quantize_rows(X):
    """Symmetric per-row absmax int8 quantisation, decided in fp32.

    "nunchaku-style kernel fusion" (#1680), commit "Reworks the Triton 8-bit
    matmuls" (axis-wise quantisation feeding the 8-bit matmul, per-row scales).
    The pages do not give the rounding; the reading taken:
      scale = absmax(row) / 127 (fp32, IEEE division),
      q = clamp(round_half_even(x / scale), -127, 127) (fp32 IEEE division),
      an all-zero row gets scale 0 and q = 0.
    Returns (q int8 [rows, cols], scale float32 [rows]).
    """
    x = np.asarray(X, dtype=np.float32)
    absmax = np.abs(x).max(axis=1).astype(np.float32)
    scale = (absmax / np.float32(127.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    ratio = (x / safe[:, None]).astype(np.float32)
    q = np.clip(np.rint(ratio), -127, 127)
    q = np.where(scale[:, None] > 0, q, 0).astype(np.int8)
    return q, scale


def int8_accumulate(Xq, Wq):
    """Exact integer product acc = Xq Wq^T in int64 (the int32 accumulator's value)."""
    return np.asarray(Xq, dtype=np.int64) @ np.asarray(Wq, dtype=np.int64).T


def w8a8_lora_fwd(Xq, sx, Wq, sw, Z, B, s, bias=None, acc=None):
    """y = acc * sx[i] * sw[o] + s * (Z B^T)[i, o] (+ bias), acc = Xq Wq^T exact.

    "nunchaku-style kernel fusion" (#1680), commits "Reworks the Triton 8-bit
    matmuls" (epilogue: per-row dequant scale plus a rank-tiled low-rank update)
    and "The five entry points" (mm_8bit with scale_m, scale_n, lora_xd, lora_up).
    Z is the given low-rank input (lora_xd = X A^T from the unquantised X).
    Returns (y float64, acc int64).
    """
    if acc is None:
        acc = int8_accumulate(Xq, Wq)
    y = acc.astype(np.float64) * f64(sx)[:, None] * f64(sw)[None, :] + s * (f64(Z) @ f64(B).T)
    if bias is not None:
        y = y + f64(bias)[None, :]
    return y, acc


def w8a8_dequant_weight(Wq, sw):
    """W_deq = diag(sw) Wq: the frozen int8 base weight in real units."""
    return f64(sw)[:, None] * np.asarray(Wq, dtype=np.float64)


def w8a8_lora_bwd(X, Wq, sw, A, B, s, dY):
    """Backward of the W8A8 + LoRA layer with W_deq frozen.

    "nunchaku-style kernel fusion" (#1680), commit reworking the 8-bit matmuls: the backward
    runs dX through the 8-bit weight (its B operand rewritten k-major) and folds the LoRA dgrad
    into the same pass; the autograd Function owns the down-projection.  The pages do not say
    how the activation quantiser is differentiated; the reading taken is the straight-through
    one (the quantiser passes gradients unchanged), so the layer's gradients are those of
    y = X W_deq^T + s (X A^T) B^T + bias with X the unquantised input:
      dX = dY W',  dA = s B^T dW',  dB = s dW' A^T,  dbias = colsum(dY),  W' = W_deq + s B A.
    """
    return lora_linear_bwd(f64(X), w8a8_dequant_weight(Wq, sw), f64(A), f64(B), s, f64(dY))


# ----------------------------------------------------------------------------- sampled forms
# For full-size workloads the oracle computes selected outputs one by one with
# the same materialised definitions: rows of y / dX (rows are independent), and
# single columns or rows of the weight-space gradient dW' = dY^T X.

def lora_fwd_rows(X, W0, A, B, s, rows, bias=None):
    """Rows `rows` of y = X W'^T + bias."""
    return lora_linear_fwd(X[rows], W0, A, B, s, bias)


def lora_bwd_sampled(X, W0, A, B, s, dY, rows, in_cols, out_rows):
    """Sampled LoRA gradients: dX[rows], dA[:, in_cols], dB[out_rows], full dbias.

    dA[:, k] = s B^T dW'[:, k] with dW'[:, k] = dY^T X[:, k];
    dB[o, :] = s dW'[o, :] A^T with dW'[o, :] = dY[:, o]^T X.
    """
    Wp = adapted_weight(W0, A, B, s)
    dX = dY[rows] @ Wp
    dWp_cols = dY.T @ X[:, in_cols]            # [out, len(in_cols)]
    dA = s * (B.T @ dWp_cols)
    dWp_rows = dY[:, out_rows].T @ X           # [len(out_rows), in]
    dB = s * (dWp_rows @ A.T)
    return dX, dA, dB, dY.sum(axis=0)


def qkv_fwd_rows(X, W0, leaves, rows, bias=None):
    """Rows `rows` of the fused-leaf output."""
    return qkv_lora_fwd(X[rows], W0, leaves, bias)


def qkv_bwd_sampled(X, W0, leaves, dY, rows, in_cols, out_rows):
    """Sampled fused-leaf gradients: dX[rows], and per leaf l dA_l[:, in_cols] and
    dB_l[out_rows[l]] (rows within the leaf), with the column / row slices of
    dW' = dY^T X formed as in lora_bwd_sampled."""
    dX = dY[rows] @ qkv_adapted_weight(W0, leaves)
    dA, dB, row = [], [], 0
    for (A, B, s), orows in zip(leaves, out_rows):
        n = B.shape[0]
        dYl = dY[:, row:row + n]
        dA.append(s * (B.T @ (dYl.T @ X[:, in_cols])))
        dB.append(s * ((dYl[:, orows].T @ X) @ A.T))
        row += n
    return dX, dA, dB


def dora_cols_fwd_rows(X, W0, A, B, m, s, rows, eps=1e-12, bias=None):
    """Rows `rows` of the DoRA-cols output, plus the full column-norm vector n."""
    return dora_cols_fwd(X[rows], W0, A, B, m, s, eps, bias)


def dora_cols_bwd_sampled(X, W0, A, B, m, s, dY, rows, in_cols, eps=1e-12):
    """Sampled DoRA-cols gradients: dX[rows], dA[:, in_cols], dm[in_cols].

    Column k of the weight-space gradient needs only column k of dWd = dY^T X:
    dWd[:, k] = dY^T X[:, k], t_k = <dWd[:, k], W'[:, k]>, and dW'[:, k] follows
    as in dora_cols_bwd; dA[:, k] = s B^T dW'[:, k].
    """
    Wp = adapted_weight(W0, A, B, s)
    nraw = np.sqrt((Wp * Wp).sum(axis=0))
    n = np.maximum(nraw, eps)
    c = m / n
    dX = dY[rows] @ (Wp * c[None, :])
    Wk = Wp[:, in_cols]
    dWd_k = dY.T @ X[:, in_cols]
    t = (dWd_k * Wk).sum(axis=0)
    nk, rk, mk, ck = n[in_cols], nraw[in_cols], m[in_cols], c[in_cols]
    live = rk > eps
    coef = np.where(live, (-t * mk / (nk * nk)) / np.where(live, rk, 1.0), 0.0)
    dWp_k = dWd_k * ck[None, :] + Wk * coef[None, :]
    return dX, s * (B.T @ dWp_k), t / nk


def dora_cols_bwd_rows_sampled(X, W0, A, B, m, s, dY, out_rows, eps=1e-12):
    """Sampled DoRA-cols up-projection gradient: dB[out_rows].

    Row o of dW' = dWd diag(c) + W' diag(coef) needs coef_k for every input column k, i.e.
    t_k = <dWd[:, k], W'[:, k]> for all k.  It is evaluated as colsum(X * (dY W')) (the same
    number summed in another order), a block of token rows at a time, so that no [out, in]
    gradient is formed; then dB[o] = s dW'[o] A^T as in dora_cols_bwd.
    """
    Wp = adapted_weight(W0, A, B, s)
    nraw = np.sqrt((Wp * Wp).sum(axis=0))
    n = np.maximum(nraw, eps)
    c = m / n
    t = np.zeros(W0.shape[1])
    for i0 in range(0, X.shape[0], 1024):
        t += (X[i0:i0 + 1024] * (dY[i0:i0 + 1024] @ Wp)).sum(axis=0)
    live = nraw > eps
    coef = np.where(live, (-t * m / (n * n)) / np.where(live, nraw, 1.0), 0.0)
    dWd_rows = dY[:, out_rows].T @ X
    dWp_rows = dWd_rows * c[None, :] + Wp[out_rows] * coef[None, :]
    return s * (dWp_rows @ A.T)


def dora_fwd_rows(X, W0, A, B, m, s, rows, eps=1e-12, bias=None):
    """Rows `rows` of the DoRA output, plus the full norm vector n."""
    return dora_linear_fwd(X[rows], W0, A, B, m, s, eps, bias)


def dora_bwd_sampled(X, W0, A, B, m, s, dY, rows, in_cols, out_rows, eps=1e-12):
    """Sampled DoRA gradients: dX[rows], dA[:, in_cols], dB[out_rows], full dm, dbias.

    Needs t_o = <dWd_o, W'_o> for every o, i.e. t = rowsum((dY^T X) * W'), which
    is evaluated as colsum(dY * (X W'^T)) (the same number, summed in another
    order) so that no [out, in] gradient has to be formed.
    """
    Wp = adapted_weight(W0, A, B, s)
    n, nraw = _dora_norm(Wp, eps)
    c = m / n
    t = np.zeros(W0.shape[0])
    for i0 in range(0, X.shape[0], 1024):       # P = X W'^T, [M, out], a block of rows at a time
        P = X[i0:i0 + 1024] @ Wp.T
        t += (dY[i0:i0 + 1024] * P).sum(axis=0)
    dm = t / n
    live = nraw > eps
    coef = np.where(live, (-t * m / (n * n)) / np.where(live, nraw, 1.0), 0.0)
    dX = dY[rows] @ (c[:, None] * Wp)
    dWd_cols = dY.T @ X[:, in_cols]
    dWp_cols = c[:, None] * dWd_cols + coef[:, None] * Wp[:, in_cols]
    dA = s * (B.T @ dWp_cols)
    dWd_rows = dY[:, out_rows].T @ X
    dWp_rows = c[out_rows, None] * dWd_rows + coef[out_rows, None] * Wp[out_rows]
    dB = s * (dWp_rows @ A.T)
    return dX, dA, dB, dm, dY.sum(axis=0)


def dora_bwd_rows_sampled(X, W0, A, B, m, s, dY, rows, out_rows, eps=1e-12):
    """DoRA gradients that need only some output rows: dX[rows], dB[out_rows], dm[out_rows].

    t_o = <dWd_o, W'_o> is evaluated for the sampled o only, as colsum(dY[:, o] * (X W'_o^T)).
    """
    Wp = adapted_weight(W0, A, B, s)
    n, nraw = _dora_norm(Wp, eps)
    c = m / n
    dX = dY[rows] @ (c[:, None] * Wp)
    Wo = Wp[out_rows]
    t = (dY[:, out_rows] * (X @ Wo.T)).sum(axis=0)
    dm = t / n[out_rows]
    live = nraw[out_rows] > eps
    coef = np.where(live, (-t * m[out_rows] / (n[out_rows] ** 2)) / np.where(live, nraw[out_rows], 1.0), 0.0)
    dWd_rows = dY[:, out_rows].T @ X
    dWp_rows = c[out_rows, None] * dWd_rows + coef[:, None] * Wo
    dB = s * (dWp_rows @ A.T)
    return dX, dB, dm


def mlp_fwd_rows(X, Wg, Ag, Bg, sg, Wu, Au, Bu, su, Wd, Ad, Bd, sd, rows, act="swiglu"):
    """Rows `rows` of (y, e, u, h) of the gated MLP."""
    return mlp_swiglu_fwd(X[rows], Wg, Ag, Bg, sg, Wu, Au, Bu, su, Wd, Ad, Bd, sd, act=act)


def mlp_bwd_rows(X, Wg, Ag, Bg, sg, Wu, Au, Bu, su, Wd, Ad, Bd, sd, dY, rows, act="swiglu"):
    """Rows `rows` of dX of the gated MLP (each row of dX depends on its own row only)."""
    return mlp_swiglu_bwd(X[rows], Wg, Ag, Bg, sg, Wu, Au, Bu, su, Wd, Ad, Bd, sd, dY[rows], act=act)["dX"]


def mlp_bwd_sparse_dy(X, Wg, Ag, Bg, sg, Wu, Au, Bu, su, Wd, Ad, Bd, sd, dY, rows, act="swiglu"):
    """All gradients of the gated MLP for an upstream gradient that is zero outside `rows`.

    Every gradient is linear in dY and each token row's contribution depends on that row alone,
    so the rows where dY vanishes add nothing: the adapter gradients are those of the sub-batch
    X[rows], dY[rows], and dX is zero outside `rows`.  Returns the dict of mlp_swiglu_bwd with
    dX restricted to `rows`.
    """
    return mlp_swiglu_bwd(X[rows], Wg, Ag, Bg, sg, Wu, Au, Bu, su, Wd, Ad, Bd, sd, dY[rows], act=act)
