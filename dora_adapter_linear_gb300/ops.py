"""Convenience layer over the C ABI: allocates outputs and workspaces with PyTorch, then calls
the entry point of the same name.  PyTorch is used only for device memory and the stream."""
from __future__ import annotations

import torch

from . import _lib as L

_WS = {}


def workspace(nbytes: int, device) -> torch.Tensor:
    """A cached, zero-initialised scratch buffer of at least nbytes (error word cleared)."""
    key = (str(device), torch.cuda.current_stream(device).cuda_stream)
    buf = _WS.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _WS[key] = buf
    return buf


def _shape_of(X, W0, A):
    return L.shape(X.shape[0], X.shape[1], W0.shape[0], A.shape[0], L.dtype_code(X))


def _check_linear(X, W0, A, B, bias=None, Z=None, dY=None, Y=None):
    """The kernels trust the shapes they are given (tensor maps and strides come from them), so a
    mismatched tensor would be read out of bounds: check every operand against X [M, in],
    W0 [out, in], A [r, in] before anything is launched."""
    if X.dim() != 2 or W0.dim() != 2:
        raise ValueError("X and W0 must be 2-D")
    M, d_in = X.shape
    d_out, r = W0.shape[0], A.shape[0]
    want = {"W0": (W0, (d_out, d_in)), "A": (A, (r, d_in)), "B": (B, (d_out, r)), "bias": (bias, (d_out,)),
            "Z": (Z, (M, r)), "dY": (dY, (M, d_out)), "Y": (Y, (M, d_out))}
    if W0.shape[1] != d_in:
        raise ValueError(f"W0 {tuple(W0.shape)} does not match X {tuple(X.shape)}")
    for name, (t, shape) in [("X", (X, (M, d_in)))] + list(want.items()):
        if t is None:
            continue
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must be {shape}, got {tuple(t.shape)}")
        if t.dtype != X.dtype or t.device != X.device or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {X.dtype} tensor on {X.device}")


def _check_like(name, t, shape, X):
    """t (if given) must have `shape`, X's dtype and device, and a contiguous layout."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != X.dtype or t.device != X.device or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {X.dtype} tensor on {X.device}")


def _check_mlp(X, g, u, d, saved=None, dY=None):
    """Each projection has its own rank: A [r, n_in], B [n_out, r] with r = A.shape[0]."""
    if X.dim() != 2:
        raise ValueError("X must be 2-D")
    M, H = X.shape
    I = g["W"].shape[0]
    for nm, p, n_out, n_in in (("gate", g, I, H), ("up", u, I, H), ("down", d, H, I)):
        r = p["A"].shape[0]
        _check_like(nm + " W", p["W"], (n_out, n_in), X)
        _check_like(nm + " A", p["A"], (r, n_in), X)
        _check_like(nm + " B", p["B"], (n_out, r), X)
    rg, ru, rd = g["A"].shape[0], u["A"].shape[0], d["A"].shape[0]
    if saved is not None:
        for k in ("e", "u", "h"):
            _check_like(k, saved[k], (M, I), X)
        _check_like("Zgu", saved["Zgu"], (M, rg + ru), X)
        _check_like("Zd", saved["Zd"], (M, rd), X)
    _check_like("dY", dY, (M, H), X)


def _mlp_shape(X, g, u, d, act):
    M, H = X.shape
    return L.mlp_shape(M, H, g["W"].shape[0], g["A"].shape[0], u["A"].shape[0], d["A"].shape[0], act=act)


def _check_qkv(X, W0, leaves, bias=None, Z=None, dY=None):
    if X.dim() != 2 or W0.dim() != 2 or not leaves:
        raise ValueError("X and W0 must be 2-D and there must be at least one leaf")
    M, d_in = X.shape
    r = leaves[0][0].shape[0]
    N = sum(B.shape[0] for _, B, _ in leaves)
    _check_like("W0", W0, (N, d_in), X)
    for l, (A, B, _) in enumerate(leaves):
        _check_like(f"A{l}", A, (r, d_in), X)
        _check_like(f"B{l}", B, (B.shape[0], r), X)
    _check_like("bias", bias, (N,), X)
    _check_like("Z", Z, (M, len(leaves) * r), X)
    _check_like("dY", dY, (M, N), X)


def _check_shapes(ref, **named):
    """Each named tensor (None allowed) must have the given shape and dtype, ref's device and a
    contiguous layout; named values are (tensor, shape, dtype) triples.  The kernels read every
    operand with the element size its dtype implies, so a wrong dtype is an out-of-bounds read."""
    for name, (t, shape, dtype) in named.items():
        if t is None:
            continue
        if (tuple(t.shape) != tuple(shape) or t.dtype != dtype or t.device != ref.device
                or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous {tuple(shape)} {dtype} tensor on {ref.device}, "
                             f"got {tuple(t.shape)} {t.dtype} on {t.device}")


def _check_vec(name, t, n, X, dtype):
    """t (if given) must be a contiguous [n] tensor of `dtype` on X's device."""
    if t is not None and (tuple(t.shape) != (n,) or t.dtype != dtype or t.device != X.device
                          or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous [{n}] {dtype} tensor on {X.device}, "
                         f"got {tuple(t.shape)} {t.dtype} on {t.device}")


F32 = torch.float32
BF16 = torch.bfloat16


def lora_linear_fwd(X, W0, A, B, s, bias=None, save_z=True):
    _check_linear(X, W0, A, B, bias)
    sh = _shape_of(X, W0, A)
    Y = torch.empty(X.shape[0], W0.shape[0], dtype=X.dtype, device=X.device)
    Z = torch.empty(X.shape[0], A.shape[0], dtype=X.dtype, device=X.device) if save_z else None
    ws = workspace(L.lora_workspace_bytes(L.OP_LINEAR_FWD, sh), X.device)
    L.lora_linear_fwd(sh, X, W0, A, B, bias, s, Y, Z, ws)
    return Y, Z


def lora_linear_bwd(X, W0, A, B, Z, dY, s, need_dx=True, need_dbias=False):
    _check_linear(X, W0, A, B, Z=Z, dY=dY)
    sh = _shape_of(X, W0, A)
    dX = torch.empty_like(X) if need_dx else None
    dA = torch.empty_like(A)
    dB = torch.empty_like(B)
    dbias = torch.empty(W0.shape[0], dtype=X.dtype, device=X.device) if need_dbias else None
    ws = workspace(L.lora_workspace_bytes(L.OP_LINEAR_BWD, sh), X.device)
    L.lora_linear_bwd(sh, X, W0, A, B, Z, dY, s, dX, dA, dB, dbias, ws)
    return dX, dA, dB, dbias


def _check_mask(mask, X):
    if (mask.dtype != torch.uint8 or tuple(mask.shape) != tuple(X.shape) or not mask.is_contiguous()
            or mask.device != X.device):
        raise ValueError(f"dropout mask must be contiguous uint8 {tuple(X.shape)}, got {mask.dtype} "
                         f"{tuple(mask.shape)}")


def lora_linear_dropout_fwd(X, mask, keep_scale, W0, A, B, s, bias=None, save_z=True):
    """mask: uint8 [M, d_in] (1 = kept), keep_scale = 1 / (1 - p)."""
    _check_linear(X, W0, A, B, bias)
    _check_mask(mask, X)
    sh = _shape_of(X, W0, A)
    Y = torch.empty(X.shape[0], W0.shape[0], dtype=X.dtype, device=X.device)
    Z = torch.empty(X.shape[0], A.shape[0], dtype=X.dtype, device=X.device) if save_z else None
    ws = workspace(L.lora_workspace_bytes(L.OP_DROPOUT_FWD, sh), X.device)
    L.lora_linear_dropout_fwd(sh, X, mask, keep_scale, W0, A, B, bias, s, Y, Z, ws)
    return Y, Z


def lora_linear_dropout_bwd(X, mask, keep_scale, W0, A, B, Z, dY, s, need_dx=True, need_dbias=False):
    _check_linear(X, W0, A, B, Z=Z, dY=dY)
    _check_mask(mask, X)
    sh = _shape_of(X, W0, A)
    dX = torch.empty_like(X) if need_dx else None
    dA = torch.empty_like(A)
    dB = torch.empty_like(B)
    dbias = torch.empty(W0.shape[0], dtype=X.dtype, device=X.device) if need_dbias else None
    ws = workspace(L.lora_workspace_bytes(L.OP_DROPOUT_BWD, sh), X.device)
    L.lora_linear_dropout_bwd(sh, X, mask, keep_scale, W0, A, B, Z, dY, s, dX, dA, dB, dbias, ws)
    return dX, dA, dB, dbias


def dora_rownorm2(W0):
    sh = L.shape(0, W0.shape[1], W0.shape[0], 8, L.dtype_code(W0))
    r0 = torch.empty(W0.shape[0], dtype=torch.float32, device=W0.device)
    L.dora_rownorm2(sh, W0, r0)
    return r0


def dora_linear_fwd(X, W0, A, B, m, r0, s, eps=1e-12, bias=None, save_z=True):
    _check_linear(X, W0, A, B, bias)
    _check_vec("m", m, W0.shape[0], X, X.dtype)
    _check_vec("r0", r0, W0.shape[0], X, F32)
    sh = _shape_of(X, W0, A)
    dev = X.device
    Y = torch.empty(X.shape[0], W0.shape[0], dtype=X.dtype, device=dev)
    Z = torch.empty(X.shape[0], A.shape[0], dtype=X.dtype, device=dev) if save_z else None
    n = torch.empty(W0.shape[0], dtype=torch.float32, device=dev)
    V = torch.empty(W0.shape[0], A.shape[0], dtype=torch.float32, device=dev)
    ws = workspace(L.lora_workspace_bytes(L.OP_DORA_FWD, sh), dev)
    L.dora_linear_fwd(sh, X, W0, A, B, m, bias, r0, s, eps, Y, Z, n, V, ws)
    return Y, Z, n, V


def dora_linear_bwd(X, W0, A, B, m, bias, Y, Z, n, V, dY, s, eps=1e-12, need_dx=True, need_dbias=False):
    _check_linear(X, W0, A, B, bias, Z=Z, dY=dY, Y=Y)
    _check_vec("m", m, W0.shape[0], X, X.dtype)
    _check_vec("n", n, W0.shape[0], X, F32)
    _check_shapes(X, V=(V, (W0.shape[0], A.shape[0]), F32))
    sh = _shape_of(X, W0, A)
    dX = torch.empty_like(X) if need_dx else None
    dA = torch.empty_like(A)
    dB = torch.empty_like(B)
    dm = torch.empty_like(m)
    dbias = torch.empty(W0.shape[0], dtype=X.dtype, device=X.device) if need_dbias else None
    ws = workspace(L.lora_workspace_bytes(L.OP_DORA_BWD, sh), X.device)
    L.dora_linear_bwd(sh, X, W0, A, B, m, bias, Y, Z, n, V, dY, s, eps, dX, dA, dB, dm, dbias, ws)
    return dX, dA, dB, dm, dbias


def dora_colnorm2(W0):
    sh = L.shape(0, W0.shape[1], W0.shape[0], 8, L.dtype_code(W0))
    c0 = torch.empty(W0.shape[1], dtype=torch.float32, device=W0.device)
    L.dora_colnorm2(sh, W0, c0)
    return c0


def dora_cols_fwd(X, W0, A, B, m, c0, s, eps=1e-12, bias=None, save_z=True):
    """m, c0: [d_in].  Returns Y, Z, n [d_in], U [d_in, r] (the last three saved for the backward)."""
    _check_linear(X, W0, A, B, bias)
    _check_vec("m", m, W0.shape[1], X, X.dtype)
    _check_vec("c0", c0, W0.shape[1], X, F32)
    sh = _shape_of(X, W0, A)
    dev = X.device
    Y = torch.empty(X.shape[0], W0.shape[0], dtype=X.dtype, device=dev)
    Z = torch.empty(X.shape[0], A.shape[0], dtype=X.dtype, device=dev) if save_z else None
    n = torch.empty(W0.shape[1], dtype=torch.float32, device=dev)
    U = torch.empty(W0.shape[1], A.shape[0], dtype=torch.float32, device=dev)
    ws = workspace(L.lora_workspace_bytes(L.OP_DORA_COLS_FWD, sh), dev)
    L.dora_cols_fwd(sh, X, W0, A, B, m, bias, c0, s, eps, Y, Z, n, U, ws)
    return Y, Z, n, U


def dora_cols_bwd(X, W0, A, B, m, Z, n, U, dY, s, eps=1e-12, need_dx=True, need_dbias=False):
    _check_linear(X, W0, A, B, Z=Z, dY=dY)
    _check_vec("m", m, W0.shape[1], X, X.dtype)
    _check_vec("n", n, W0.shape[1], X, F32)
    _check_shapes(X, U=(U, (W0.shape[1], A.shape[0]), F32))
    sh = _shape_of(X, W0, A)
    dX = torch.empty_like(X) if need_dx else None
    dA = torch.empty_like(A)
    dB = torch.empty_like(B)
    dm = torch.empty_like(m)
    dbias = torch.empty(W0.shape[0], dtype=X.dtype, device=X.device) if need_dbias else None
    ws = workspace(L.lora_workspace_bytes(L.OP_DORA_COLS_BWD, sh), X.device)
    L.dora_cols_bwd(sh, X, W0, A, B, m, Z, n, U, dY, s, eps, dX, dA, dB, dm, dbias, ws)
    return dX, dA, dB, dm, dbias


def lora_mlp_swiglu_fwd(X, g, u, d, act=0):
    """g, u, d: dicts with W, A, B, s; act 0 SwiGLU, 1 GeGLU.  Returns (Y, saved) where saved
    holds e, u, h, Zgu, Zd."""
    _check_mlp(X, g, u, d)
    M, H = X.shape
    I = g["W"].shape[0]
    sh = _mlp_shape(X, g, u, d, act)
    dev = X.device
    e_ = torch.empty(M, I, dtype=X.dtype, device=dev)
    u_ = torch.empty_like(e_)
    h_ = torch.empty_like(e_)
    Zgu = torch.empty(M, sh.r_g + sh.r_u, dtype=X.dtype, device=dev)
    Zd = torch.empty(M, sh.r_d, dtype=X.dtype, device=dev)
    Y = torch.empty(M, H, dtype=X.dtype, device=dev)
    ws = workspace(L.lora_mlp_workspace_bytes(L.OP_MLP_FWD, sh), dev)
    pg, pu, pd = (L.proj(p["W"], p["A"], p["B"], p["s"]) for p in (g, u, d))
    L.lora_mlp_swiglu_fwd(sh, X, pg, pu, pd, Y, e_, u_, h_, Zgu, Zd, ws)
    return Y, {"e": e_, "u": u_, "h": h_, "Zgu": Zgu, "Zd": Zd}


def lora_mlp_swiglu_bwd(X, g, u, d, saved, dY, need_dx=True, act=0):
    _check_mlp(X, g, u, d, saved, dY)
    sh = _mlp_shape(X, g, u, d, act)
    dX = torch.empty_like(X) if need_dx else None
    grads = {k: torch.empty_like(v) for k, v in
             (("dAg", g["A"]), ("dBg", g["B"]), ("dAu", u["A"]), ("dBu", u["B"]), ("dAd", d["A"]), ("dBd", d["B"]))}
    ws = workspace(L.lora_mlp_workspace_bytes(L.OP_MLP_BWD, sh), X.device)
    pg, pu, pd = (L.proj(p["W"], p["A"], p["B"], p["s"]) for p in (g, u, d))
    L.lora_mlp_swiglu_bwd(sh, X, pg, pu, pd, saved["e"], saved["u"], saved["h"], saved["Zgu"], saved["Zd"], dY, dX,
                          grads["dAg"], grads["dBg"], grads["dAu"], grads["dBu"], grads["dAd"], grads["dBd"], ws)
    grads["dX"] = dX
    return grads


def w8a8_quantize_rows(X, A=None):
    if X.dim() != 2:
        raise ValueError("X must be 2-D")
    rows, cols = X.shape
    _check_shapes(X, X=(X, (rows, cols), BF16), A=(A, (None if A is None else A.shape[0], cols), BF16))
    Xq = torch.empty(rows, cols, dtype=torch.int8, device=X.device)
    sx = torch.empty(rows, dtype=torch.float32, device=X.device)
    Z = torch.empty(rows, A.shape[0], dtype=X.dtype, device=X.device) if A is not None else None
    L.w8a8_quantize_rows(rows, cols, X, Xq, sx, A, 0 if A is None else A.shape[0], Z)
    return Xq, sx, Z


def w8a8_lora_bwd(X, Wq, sw, A, B, Z, dY, s, need_dx=True, need_dbias=False):
    M, d_in = X.shape
    d_out, r = Wq.shape[0], A.shape[0]
    if Wq.dtype != torch.int8:
        raise ValueError("Wq must be int8")
    _check_shapes(X, X=(X, (M, d_in), BF16), Wq=(Wq, (d_out, d_in), torch.int8), sw=(sw, (d_out,), F32),
                  A=(A, (r, d_in), BF16), B=(B, (d_out, r), BF16), Z=(Z, (M, r), BF16), dY=(dY, (M, d_out), BF16))
    dX = torch.empty_like(X) if need_dx else None
    dA = torch.empty_like(A)
    dB = torch.empty_like(B)
    dbias = torch.empty(d_out, dtype=X.dtype, device=X.device) if need_dbias else None
    ws = workspace(L.w8a8_bwd_workspace_bytes(M, d_in, d_out, r), X.device)
    L.w8a8_lora_bwd(M, d_in, d_out, r, X, Wq, sw, A, B, Z, dY, s, dX, dA, dB, dbias, ws)
    return dX, dA, dB, dbias


def w8a8_lora_fwd(Xq, sx, Wq, sw, Z, B, s, bias=None, want_acc=False, want_y=True):
    M, d_in = Xq.shape
    d_out = Wq.shape[0]
    r = 0 if Z is None else Z.shape[1]
    if Xq.dtype != torch.int8 or Wq.dtype != torch.int8:
        raise ValueError("Xq and Wq must be int8")
    _check_shapes(Xq, Xq=(Xq, (M, d_in), torch.int8), sx=(sx, (M,), F32), Wq=(Wq, (d_out, d_in), torch.int8),
                  sw=(sw, (d_out,), F32), Z=(Z, (M, r), BF16), B=(B, (d_out, r), BF16), bias=(bias, (d_out,), BF16))
    Y = torch.empty(M, d_out, dtype=torch.bfloat16, device=Xq.device) if want_y else None
    acc = torch.empty(M, d_out, dtype=torch.int32, device=Xq.device) if want_acc else None
    ws = workspace(L.w8a8_workspace_bytes(M, d_in, d_out), Xq.device)
    L.w8a8_lora_fwd(M, d_in, d_out, r, Xq, sx, Wq, sw, Z, B, s, bias, Y, acc, ws)
    return Y, acc


def lora_qkv_fwd(X, W0, leaves, bias=None, save_z=True):
    """leaves: [(A_l, B_l, s_l)] for the leaves of the fused weight W0 (rows in leaf order)."""
    _check_qkv(X, W0, leaves, bias)
    M, d_in = X.shape
    n = [B.shape[0] for _, B, _ in leaves]
    r = leaves[0][0].shape[0]
    sh = L.qkv_shape(M, d_in, n, r)
    Y = torch.empty(M, sum(n), dtype=X.dtype, device=X.device)
    Z = torch.empty(M, len(leaves) * r, dtype=X.dtype, device=X.device) if save_z else None
    ws = workspace(L.lora_qkv_workspace_bytes(L.OP_QKV_FWD, sh), X.device)
    L.lora_qkv_fwd(sh, X, W0, L.adapters(leaves), bias, Y, Z, ws)
    return Y, Z


def lora_qkv_bwd(X, W0, leaves, Z, dY, need_dx=True, need_dbias=False):
    _check_qkv(X, W0, leaves, Z=Z, dY=dY)
    M, d_in = X.shape
    n = [B.shape[0] for _, B, _ in leaves]
    r = leaves[0][0].shape[0]
    sh = L.qkv_shape(M, d_in, n, r)
    dX = torch.empty_like(X) if need_dx else None
    dA = [torch.empty_like(A) for A, _, _ in leaves]
    dB = [torch.empty_like(B) for _, B, _ in leaves]
    dbias = torch.empty(sum(n), dtype=X.dtype, device=X.device) if need_dbias else None
    ws = workspace(L.lora_qkv_workspace_bytes(L.OP_QKV_BWD, sh), X.device)
    L.lora_qkv_bwd(sh, X, W0, L.adapters(leaves), Z, dY, dX, dA, dB, dbias, ws)
    return dX, dA, dB, dbias


def w8a8_quantize_rows_bf16(X, A=None):
    """Per-token quantisation with the codes returned as bf16 values: (Xcodes, sx, Z)."""
    if X.dim() != 2:
        raise ValueError("X must be 2-D")
    rows, cols = X.shape
    _check_shapes(X, X=(X, (rows, cols), BF16), A=(A, (None if A is None else A.shape[0], cols), BF16))
    Xc = torch.empty(rows, cols, dtype=torch.bfloat16, device=X.device)
    sx = torch.empty(rows, dtype=torch.float32, device=X.device)
    Z = torch.empty(rows, A.shape[0], dtype=X.dtype, device=X.device) if A is not None else None
    L.w8a8_quantize_rows_bf16(rows, cols, X, Xc, sx, A, 0 if A is None else A.shape[0], Z)
    return Xc, sx, Z


def w8a8_prepack_weight(Wq, sw, codes=True, dequant=True):
    """The frozen int8 weight laid out once: Wb the codes as bf16 for the forward, Wd the
    dequantised weight for the backward (each None when not asked for)."""
    if Wq.dtype != torch.int8 or Wq.dim() != 2:
        raise ValueError("Wq must be a 2-D int8 tensor")
    d_out, d_in = Wq.shape
    _check_shapes(Wq, Wq=(Wq, (d_out, d_in), torch.int8), sw=(sw, (d_out,), F32))
    mk = lambda: torch.empty(d_out, d_in, dtype=torch.bfloat16, device=Wq.device)  # noqa: E731
    Wb = mk() if codes else None
    Wd = mk() if dequant else None
    L.w8a8_prepack_weight(d_out, d_in, Wq, sw, Wb, Wd)
    return Wb, Wd


def w8a8_lora_fwd_packed(Xc, sx, Wb, sw, Z, B, s, bias=None, want_acc=False, want_y=True):
    """w8a8_lora_fwd on prepacked operands (Xc from w8a8_quantize_rows_bf16, Wb from
    w8a8_prepack_weight)."""
    M, d_in = Xc.shape
    d_out = Wb.shape[0]
    r = 0 if Z is None else Z.shape[1]
    _check_shapes(Xc, Xc=(Xc, (M, d_in), BF16), sx=(sx, (M,), F32), Wb=(Wb, (d_out, d_in), BF16),
                  sw=(sw, (d_out,), F32), Z=(Z, (M, r), BF16), B=(B, (d_out, r), BF16), bias=(bias, (d_out,), BF16))
    Y = torch.empty(M, d_out, dtype=torch.bfloat16, device=Xc.device) if want_y else None
    acc = torch.empty(M, d_out, dtype=torch.int32, device=Xc.device) if want_acc else None
    ws = workspace(L.w8a8_packed_workspace_bytes(M, d_out), Xc.device)
    L.w8a8_lora_fwd_packed(M, d_in, d_out, r, Xc, sx, Wb, sw, Z, B, s, bias, Y, acc, ws)
    return Y, acc
