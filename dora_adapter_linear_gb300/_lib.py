"""ctypes binding of liblora_gb300.so: argument marshalling only.

Every function here has the name of the C entry point it calls, takes torch tensors (or
None) in the same order, passes their device pointers and the current CUDA stream, and
raises LoraError on a non-OK status.  No arithmetic of the layer happens in Python.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int8, c_int32, c_int64, c_size_t, c_uint32, c_void_p

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblora_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "lora_gb300.h")

LORA_F32, LORA_BF16 = 0, 1
LORA_NOALLOC_SCRATCH_BYTES = 4 << 20   # fixed scratch of lora_linear_fwd_noalloc (header macro)
(OP_LINEAR_FWD, OP_LINEAR_BWD, OP_DORA_FWD, OP_DORA_BWD, OP_MLP_FWD, OP_MLP_BWD, OP_QKV_FWD, OP_QKV_BWD,
 OP_DORA_COLS_FWD, OP_DORA_COLS_BWD, OP_DROPOUT_FWD, OP_DROPOUT_BWD) = range(12)
STATUS = {0: "LORA_OK", 1: "LORA_ERR_INVALID_ARG", 2: "LORA_ERR_UNSUPPORTED", 3: "LORA_ERR_MISALIGNED",
          4: "LORA_ERR_WORKSPACE", 5: "LORA_ERR_CUDA", 6: "LORA_ERR_DEVICE_TIMEOUT"}


class LoraError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({_lib().lora_status_string(status).decode()})")


class LoraShape(ctypes.Structure):
    _fields_ = [("M", c_int64), ("d_in", c_int64), ("d_out", c_int64), ("r", c_int64), ("dtype", c_int32)]


class LoraMlpShape(ctypes.Structure):
    _fields_ = [("M", c_int64), ("H", c_int64), ("I", c_int64), ("r_g", c_int64), ("r_u", c_int64),
                ("r_d", c_int64), ("dtype", c_int32), ("act", c_int32)]


LORA_ACT_SWIGLU, LORA_ACT_GEGLU = 0, 1


class LoraProj(ctypes.Structure):
    _fields_ = [("W", c_void_p), ("A", c_void_p), ("B", c_void_p), ("s", c_float)]


class LoraQkvShape(ctypes.Structure):
    _fields_ = [("M", c_int64), ("d_in", c_int64), ("n", c_int64 * 3), ("L", c_int32), ("r", c_int32),
                ("dtype", c_int32)]


class LoraAdapter(ctypes.Structure):
    _fields_ = [("A", c_void_p), ("B", c_void_p), ("s", c_float)]


P = c_void_p
_SIGS = {
    "lora_status_string": (c_char_p, [c_int]),
    "lora_abi_version": (c_int, []),
    "lora_workspace_bytes": (c_size_t, [c_int, POINTER(LoraShape)]),
    "lora_mlp_workspace_bytes": (c_size_t, [c_int, POINTER(LoraMlpShape)]),
    "lora_clear_device_error": (c_int, [P, P]),
    "lora_check_device_error": (c_int, [P, P]),
    "lora_linear_fwd": (c_int, [POINTER(LoraShape), P, P, P, P, P, c_float, P, P, P, c_size_t, P]),
    "lora_linear_bwd": (c_int, [POINTER(LoraShape), P, P, P, P, P, P, c_float, P, P, P, P, P, c_size_t, P]),
    "lora_linear_dropout_fwd": (c_int, [POINTER(LoraShape), P, P, c_float, P, P, P, P, c_float, P, P, P, c_size_t,
                                        P]),
    "lora_linear_dropout_bwd": (c_int, [POINTER(LoraShape), P, P, c_float, P, P, P, P, P, c_float, P, P, P, P, P,
                                        c_size_t, P]),
    "dora_rownorm2": (c_int, [POINTER(LoraShape), P, P, P]),
    "dora_linear_fwd": (c_int, [POINTER(LoraShape), P, P, P, P, P, P, P, c_float, c_float, P, P, P, P, P,
                                c_size_t, P]),
    "dora_linear_bwd": (c_int, [POINTER(LoraShape), P, P, P, P, P, P, P, P, P, P, P, c_float, c_float,
                                P, P, P, P, P, P, c_size_t, P]),
    "dora_colnorm2": (c_int, [POINTER(LoraShape), P, P, P]),
    "dora_cols_fwd": (c_int, [POINTER(LoraShape), P, P, P, P, P, P, P, c_float, c_float, P, P, P, P, P,
                              c_size_t, P]),
    "dora_cols_bwd": (c_int, [POINTER(LoraShape), P, P, P, P, P, P, P, P, P, c_float, c_float,
                              P, P, P, P, P, P, c_size_t, P]),
    "lora_mlp_swiglu_fwd": (c_int, [POINTER(LoraMlpShape), P, POINTER(LoraProj), POINTER(LoraProj),
                                    POINTER(LoraProj), P, P, P, P, P, P, P, c_size_t, P]),
    "lora_mlp_swiglu_bwd": (c_int, [POINTER(LoraMlpShape), P, POINTER(LoraProj), POINTER(LoraProj),
                                    POINTER(LoraProj), P, P, P, P, P, P, P, P, P, P, P, P, P, P, c_size_t, P]),
    "w8a8_quantize_rows": (c_int, [c_int64, c_int64, P, P, P, P, c_int64, P, P]),
    "w8a8_workspace_bytes": (c_size_t, [c_int64, c_int64, c_int64]),
    "w8a8_lora_fwd": (c_int, [c_int64, c_int64, c_int64, c_int64, P, P, P, P, P, P, c_float, P, P, P, P, c_size_t,
                              P]),
    "w8a8_quantize_rows_bf16": (c_int, [c_int64, c_int64, P, P, P, P, c_int64, P, P]),
    "w8a8_prepack_weight": (c_int, [c_int64, c_int64, P, P, P, P, P]),
    "w8a8_packed_workspace_bytes": (c_size_t, [c_int64, c_int64]),
    "w8a8_lora_fwd_packed": (c_int, [c_int64, c_int64, c_int64, c_int64, P, P, P, P, P, P, c_float, P, P, P, P,
                                     c_size_t, P]),
    "lora_debug_wait_timeout": (c_int, [P, c_uint32, P]),
    "lora_linear_fwd_noalloc": (c_int, [POINTER(LoraShape), P, P, P, P, P, c_float, P, P, P]),
    "w8a8_bwd_workspace_bytes": (c_size_t, [c_int64, c_int64, c_int64, c_int64]),
    "w8a8_lora_bwd": (c_int, [c_int64, c_int64, c_int64, c_int64, P, P, P, P, P, P, P, c_float, P, P, P, P, P,
                              c_size_t, P]),
    "lora_qkv_workspace_bytes": (c_size_t, [c_int, POINTER(LoraQkvShape)]),
    "lora_qkv_fwd": (c_int, [POINTER(LoraQkvShape), P, P, POINTER(LoraAdapter), P, P, P, P, c_size_t, P]),
    "lora_qkv_bwd": (c_int, [POINTER(LoraQkvShape), P, P, POINTER(LoraAdapter), P, P, P, POINTER(c_void_p),
                             POINTER(c_void_p), P, P, c_size_t, P]),
    "lora_launch_count": (ctypes.c_uint64, []),
    "lora_prof_enable": (c_int, [c_int]),
    "lora_prof_gemm": (c_int, [POINTER(ctypes.c_double), POINTER(c_int64), POINTER(ctypes.c_double), c_int]),
    "lora_prof_rank": (c_int, [POINTER(ctypes.c_double), POINTER(c_int64), POINTER(ctypes.c_double), c_int]),
}

_LIB = None


def _lib():
    """Load the library (fails loudly if it has not been built: there is no fallback)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing; build it with dora_adapter_linear_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _LIB = lib
    return _LIB


def ptr(t):
    """Device pointer of a tensor (None -> NULL)."""
    if t is None:
        return None
    return c_void_p(t.data_ptr())


def _stream(stream):
    if stream is not None:
        return c_void_p(stream if isinstance(stream, int) else stream.cuda_stream)
    import torch
    return c_void_p(torch.cuda.current_stream().cuda_stream)


def _ck(status, where):
    if status != 0:
        raise LoraError(status, where)


def dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return LORA_BF16
    if t.dtype == torch.float32:
        return LORA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def shape(M, d_in, d_out, r, dtype) -> LoraShape:
    return LoraShape(M, d_in, d_out, r, dtype)


def mlp_shape(M, H, I, r_g, r_u=None, r_d=None, dtype=LORA_BF16, act=0) -> LoraMlpShape:
    """Ranks of the gate, up and down projections (r_u, r_d default to r_g)."""
    r_u = r_g if r_u is None else r_u
    r_d = r_g if r_d is None else r_d
    return LoraMlpShape(M, H, I, r_g, r_u, r_d, dtype, act)


def proj(W, A, B, s) -> LoraProj:
    return LoraProj(W.data_ptr(), A.data_ptr(), B.data_ptr(), float(s))


def qkv_shape(M, d_in, n, r, dtype=LORA_BF16) -> LoraQkvShape:
    n = list(n)
    return LoraQkvShape(M, d_in, (c_int64 * 3)(*(n + [0] * (3 - len(n)))), len(n), r, dtype)


def adapters(leaves):
    """leaves: sequence of (A, B, s) -> a ctypes array of lora_adapter."""
    arr = (LoraAdapter * max(len(leaves), 1))()
    for i, (A, B, s) in enumerate(leaves):
        arr[i] = LoraAdapter(ptr(A), ptr(B), float(s))
    return arr


def _ptrs(ts):
    return (c_void_p * max(len(ts), 1))(*[ptr(t) for t in ts])


# ------------------------------------------------------------------ entry points
def lora_status_string(status: int) -> str:
    return _lib().lora_status_string(status).decode()


def lora_abi_version() -> int:
    return _lib().lora_abi_version()


def lora_workspace_bytes(op: int, sh: LoraShape) -> int:
    return _lib().lora_workspace_bytes(op, ctypes.byref(sh))


def lora_mlp_workspace_bytes(op: int, sh: LoraMlpShape) -> int:
    return _lib().lora_mlp_workspace_bytes(op, ctypes.byref(sh))


def lora_clear_device_error(ws, stream=None):
    _ck(_lib().lora_clear_device_error(ptr(ws), _stream(stream)), "lora_clear_device_error")


def lora_check_device_error(ws, stream=None) -> int:
    """Returns the status (0 = clear, 6 = a bounded wait ran out); synchronises the stream."""
    return _lib().lora_check_device_error(ptr(ws), _stream(stream))


def lora_debug_wait_timeout(ws, timeout_us: int, stream=None):
    _ck(_lib().lora_debug_wait_timeout(ptr(ws), timeout_us, _stream(stream)), "lora_debug_wait_timeout")


def lora_launch_count() -> int:
    return int(_lib().lora_launch_count())


def lora_prof_enable(on: bool):
    _ck(_lib().lora_prof_enable(1 if on else 0), "lora_prof_enable")


def lora_prof_gemm(reset: bool = True):
    """(device ms, launches, algorithmic flops) of the GEMM launches recorded since the last reset."""
    ms, n, fl = ctypes.c_double(), c_int64(), ctypes.c_double()
    _ck(_lib().lora_prof_gemm(ctypes.byref(ms), ctypes.byref(n), ctypes.byref(fl), 1 if reset else 0),
        "lora_prof_gemm")
    return ms.value, n.value, fl.value


def lora_prof_rank(reset: bool = True):
    """(device ms, launches, algorithmic HBM bytes) of the rank-r passes recorded since the last reset."""
    ms, n, by = ctypes.c_double(), c_int64(), ctypes.c_double()
    _ck(_lib().lora_prof_rank(ctypes.byref(ms), ctypes.byref(n), ctypes.byref(by), 1 if reset else 0),
        "lora_prof_rank")
    return ms.value, n.value, by.value


def lora_linear_fwd(sh, X, W0, A, B, bias, s, Y, Z_save, ws, stream=None):
    _ck(_lib().lora_linear_fwd(ctypes.byref(sh), ptr(X), ptr(W0), ptr(A), ptr(B), ptr(bias), float(s), ptr(Y),
                               ptr(Z_save), ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                               _stream(stream)), "lora_linear_fwd")


def lora_linear_fwd_noalloc(sh, X, W0, A, B, bias, s, Y, Z_save, stream=None):
    """lora_linear_fwd with the library's fixed device scratch instead of a workspace."""
    _ck(_lib().lora_linear_fwd_noalloc(ctypes.byref(sh), ptr(X), ptr(W0), ptr(A), ptr(B), ptr(bias), float(s),
                                       ptr(Y), ptr(Z_save), _stream(stream)), "lora_linear_fwd_noalloc")


def lora_linear_dropout_fwd(sh, X, mask, keep_scale, W0, A, B, bias, s, Y, Z_save, ws, stream=None):
    _ck(_lib().lora_linear_dropout_fwd(ctypes.byref(sh), ptr(X), ptr(mask), float(keep_scale), ptr(W0), ptr(A),
                                       ptr(B), ptr(bias), float(s), ptr(Y), ptr(Z_save), ptr(ws),
                                       0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
        "lora_linear_dropout_fwd")


def lora_linear_dropout_bwd(sh, X, mask, keep_scale, W0, A, B, Z_saved, dY, s, dX, dA, dB, dbias, ws, stream=None):
    _ck(_lib().lora_linear_dropout_bwd(ctypes.byref(sh), ptr(X), ptr(mask), float(keep_scale), ptr(W0), ptr(A),
                                       ptr(B), ptr(Z_saved), ptr(dY), float(s), ptr(dX), ptr(dA), ptr(dB), ptr(dbias),
                                       ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                       _stream(stream)), "lora_linear_dropout_bwd")


def lora_linear_bwd(sh, X, W0, A, B, Z_saved, dY, s, dX, dA, dB, dbias, ws, stream=None):
    _ck(_lib().lora_linear_bwd(ctypes.byref(sh), ptr(X), ptr(W0), ptr(A), ptr(B), ptr(Z_saved), ptr(dY), float(s),
                               ptr(dX), ptr(dA), ptr(dB), ptr(dbias), ptr(ws),
                               0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
        "lora_linear_bwd")


def dora_rownorm2(sh, W0, r0, stream=None):
    _ck(_lib().dora_rownorm2(ctypes.byref(sh), ptr(W0), ptr(r0), _stream(stream)), "dora_rownorm2")


def dora_linear_fwd(sh, X, W0, A, B, m, bias, r0, s, eps, Y, Z_save, n_save, V_save, ws, stream=None):
    _ck(_lib().dora_linear_fwd(ctypes.byref(sh), ptr(X), ptr(W0), ptr(A), ptr(B), ptr(m), ptr(bias), ptr(r0),
                               float(s), float(eps), ptr(Y), ptr(Z_save), ptr(n_save), ptr(V_save), ptr(ws),
                               0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
        "dora_linear_fwd")


def dora_linear_bwd(sh, X, W0, A, B, m, bias, Y, Z_saved, n_saved, V_saved, dY, s, eps, dX, dA, dB, dm, dbias, ws,
                    stream=None):
    _ck(_lib().dora_linear_bwd(ctypes.byref(sh), ptr(X), ptr(W0), ptr(A), ptr(B), ptr(m), ptr(bias), ptr(Y),
                               ptr(Z_saved), ptr(n_saved), ptr(V_saved), ptr(dY), float(s), float(eps), ptr(dX),
                               ptr(dA), ptr(dB), ptr(dm), ptr(dbias), ptr(ws),
                               0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
        "dora_linear_bwd")


def dora_colnorm2(sh, W0, c0, stream=None):
    _ck(_lib().dora_colnorm2(ctypes.byref(sh), ptr(W0), ptr(c0), _stream(stream)), "dora_colnorm2")


def dora_cols_fwd(sh, X, W0, A, B, m, bias, c0, s, eps, Y, Z_save, n_save, U_save, ws, stream=None):
    _ck(_lib().dora_cols_fwd(ctypes.byref(sh), ptr(X), ptr(W0), ptr(A), ptr(B), ptr(m), ptr(bias), ptr(c0),
                             float(s), float(eps), ptr(Y), ptr(Z_save), ptr(n_save), ptr(U_save), ptr(ws),
                             0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)), "dora_cols_fwd")


def dora_cols_bwd(sh, X, W0, A, B, m, Z_saved, n_saved, U_saved, dY, s, eps, dX, dA, dB, dm, dbias, ws,
                  stream=None):
    _ck(_lib().dora_cols_bwd(ctypes.byref(sh), ptr(X), ptr(W0), ptr(A), ptr(B), ptr(m), ptr(Z_saved), ptr(n_saved),
                             ptr(U_saved), ptr(dY), float(s), float(eps), ptr(dX), ptr(dA), ptr(dB), ptr(dm),
                             ptr(dbias), ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                             _stream(stream)), "dora_cols_bwd")


def lora_mlp_swiglu_fwd(sh, X, gate, up, down, Y, e_save, u_save, h_save, Zgu_save, Zd_save, ws, stream=None):
    _ck(_lib().lora_mlp_swiglu_fwd(ctypes.byref(sh), ptr(X), ctypes.byref(gate), ctypes.byref(up),
                                   ctypes.byref(down), ptr(Y), ptr(e_save), ptr(u_save), ptr(h_save), ptr(Zgu_save),
                                   ptr(Zd_save), ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                   _stream(stream)), "lora_mlp_swiglu_fwd")


def lora_mlp_swiglu_bwd(sh, X, gate, up, down, e_saved, u_saved, h_saved, Zgu_saved, Zd_saved, dY, dX, dAg, dBg,
                        dAu, dBu, dAd, dBd, ws, stream=None):
    _ck(_lib().lora_mlp_swiglu_bwd(ctypes.byref(sh), ptr(X), ctypes.byref(gate), ctypes.byref(up),
                                   ctypes.byref(down), ptr(e_saved), ptr(u_saved), ptr(h_saved), ptr(Zgu_saved),
                                   ptr(Zd_saved), ptr(dY), ptr(dX), ptr(dAg), ptr(dBg), ptr(dAu), ptr(dBu), ptr(dAd),
                                   ptr(dBd), ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                   _stream(stream)), "lora_mlp_swiglu_bwd")


def lora_qkv_workspace_bytes(op: int, sh: LoraQkvShape) -> int:
    return _lib().lora_qkv_workspace_bytes(op, ctypes.byref(sh))


def lora_qkv_fwd(sh, X, W0, leaves, bias, Y, Z_save, ws, stream=None):
    """leaves: a ctypes array from adapters()."""
    _ck(_lib().lora_qkv_fwd(ctypes.byref(sh), ptr(X), ptr(W0), leaves, ptr(bias), ptr(Y), ptr(Z_save), ptr(ws),
                            0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)), "lora_qkv_fwd")


def lora_qkv_bwd(sh, X, W0, leaves, Z_saved, dY, dX, dA, dB, dbias, ws, stream=None):
    """dA, dB: sequences of L tensors (or ctypes pointer arrays)."""
    dA = dA if isinstance(dA, ctypes.Array) else _ptrs(dA)
    dB = dB if isinstance(dB, ctypes.Array) else _ptrs(dB)
    _ck(_lib().lora_qkv_bwd(ctypes.byref(sh), ptr(X), ptr(W0), leaves, ptr(Z_saved), ptr(dY), ptr(dX), dA, dB,
                            ptr(dbias), ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                            _stream(stream)), "lora_qkv_bwd")


def w8a8_quantize_rows(rows, cols, X, Xq, sx, A=None, r=0, Z=None, stream=None):
    _ck(_lib().w8a8_quantize_rows(rows, cols, ptr(X), ptr(Xq), ptr(sx), ptr(A), r, ptr(Z), _stream(stream)),
        "w8a8_quantize_rows")


def w8a8_bwd_workspace_bytes(M, d_in, d_out, r) -> int:
    return _lib().w8a8_bwd_workspace_bytes(M, d_in, d_out, r)


def w8a8_lora_bwd(M, d_in, d_out, r, X, Wq, sw, A, B, Z_saved, dY, s, dX, dA, dB, dbias, ws, stream=None):
    _ck(_lib().w8a8_lora_bwd(M, d_in, d_out, r, ptr(X), ptr(Wq), ptr(sw), ptr(A), ptr(B), ptr(Z_saved), ptr(dY),
                             float(s), ptr(dX), ptr(dA), ptr(dB), ptr(dbias), ptr(ws),
                             0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)), "w8a8_lora_bwd")


def w8a8_workspace_bytes(M, d_in, d_out) -> int:
    return _lib().w8a8_workspace_bytes(M, d_in, d_out)


def w8a8_lora_fwd(M, d_in, d_out, r, Xq, sx, Wq, sw, Z, B, s, bias, Y, acc_out, ws, stream=None):
    _ck(_lib().w8a8_lora_fwd(M, d_in, d_out, r, ptr(Xq), ptr(sx), ptr(Wq), ptr(sw), ptr(Z), ptr(B), float(s),
                             ptr(bias), ptr(Y), ptr(acc_out), ptr(ws),
                             0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)), "w8a8_lora_fwd")


def w8a8_quantize_rows_bf16(rows, cols, X, Xcodes, sx, A=None, r=0, Z=None, stream=None):
    _ck(_lib().w8a8_quantize_rows_bf16(rows, cols, ptr(X), ptr(Xcodes), ptr(sx), ptr(A), r, ptr(Z),
                                       _stream(stream)), "w8a8_quantize_rows_bf16")


def w8a8_prepack_weight(d_out, d_in, Wq, sw, Wb, Wd, stream=None):
    _ck(_lib().w8a8_prepack_weight(d_out, d_in, ptr(Wq), ptr(sw), ptr(Wb), ptr(Wd), _stream(stream)),
        "w8a8_prepack_weight")


def w8a8_packed_workspace_bytes(M, d_out) -> int:
    return _lib().w8a8_packed_workspace_bytes(M, d_out)


def w8a8_lora_fwd_packed(M, d_in, d_out, r, Xcodes, sx, Wb, sw, Z, B, s, bias, Y, acc_out, ws, stream=None):
    _ck(_lib().w8a8_lora_fwd_packed(M, d_in, d_out, r, ptr(Xcodes), ptr(sx), ptr(Wb), ptr(sw), ptr(Z),
                                    ptr(B), float(s), ptr(bias), ptr(Y), ptr(acc_out), ptr(ws),
                                    0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
        "w8a8_lora_fwd_packed")
