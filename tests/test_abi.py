"""C-ABI library checks that need no GPU: it builds, loads, exports every symbol the header
declares, and rejects bad arguments before launching anything."""
import ctypes
import re

import pytest

from dora_adapter_linear_gb300 import _lib as L
from dora_adapter_linear_gb300.build import build


@pytest.fixture(scope="module")
def lib():
    build()
    return L._lib()


def header_functions():
    text = open(L.HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = header_functions()
    for must in ("lora_linear_fwd", "lora_linear_bwd", "dora_linear_fwd", "dora_linear_bwd", "dora_rownorm2",
                 "lora_mlp_swiglu_fwd", "lora_mlp_swiglu_bwd", "w8a8_lora_fwd", "w8a8_quantize_rows"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in header_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(header_functions()) == set(L._SIGS), "binding signatures must cover the header exactly"


def test_status_strings(lib):
    assert L.lora_status_string(0) == "ok"
    assert "workspace" in L.lora_status_string(4)
    assert L.lora_status_string(99) == "unknown status"
    assert L.lora_abi_version() == 8


def test_workspace_bytes_rejects_bad_shapes(lib):
    assert L.lora_workspace_bytes(L.OP_LINEAR_FWD, L.shape(64, 256, 256, 8, L.LORA_F32)) > 0
    assert L.lora_workspace_bytes(L.OP_LINEAR_FWD, L.shape(64, 250, 256, 8, L.LORA_F32)) == 0   # in % 8
    for r in range(8, 129, 8):                                                                   # r 8..128
        for op in (L.OP_LINEAR_FWD, L.OP_LINEAR_BWD, L.OP_DORA_FWD, L.OP_DORA_BWD, L.OP_DORA_COLS_BWD):
            assert L.lora_workspace_bytes(op, L.shape(64, 256, 256, r, L.LORA_BF16)) > 0, (op, r)
    assert L.lora_workspace_bytes(L.OP_LINEAR_FWD, L.shape(64, 256, 256, 136, L.LORA_BF16)) == 0  # r > 128
    assert L.lora_workspace_bytes(L.OP_LINEAR_FWD, L.shape(64, 256, 256, 128, L.LORA_F32)) > 0
    assert L.lora_workspace_bytes(L.OP_LINEAR_FWD, L.shape(64, 256, 256, 129, L.LORA_F32)) == 0
    assert L.lora_workspace_bytes(L.OP_LINEAR_FWD, L.shape(64, 256, 256, 12, L.LORA_BF16)) == 0  # r % 8 (bf16)
    assert L.lora_workspace_bytes(L.OP_LINEAR_FWD, L.shape(64, 256, 256, 8, 7)) == 0             # dtype
    assert L.lora_workspace_bytes(99, L.shape(64, 256, 256, 8, L.LORA_F32)) == 0
    assert L.lora_mlp_workspace_bytes(L.OP_MLP_FWD, L.mlp_shape(64, 128, 256, 16)) > 0
    assert L.lora_mlp_workspace_bytes(L.OP_MLP_FWD, L.mlp_shape(64, 128, 256, 40)) > 0           # r 33..64
    assert L.lora_mlp_workspace_bytes(L.OP_MLP_BWD, L.mlp_shape(64, 128, 256, 128, 72, 96)) > 0   # per projection
    small = L.lora_mlp_workspace_bytes(L.OP_MLP_BWD, L.mlp_shape(64, 128, 256, 8, 8, 8))
    assert L.lora_mlp_workspace_bytes(L.OP_MLP_BWD, L.mlp_shape(64, 128, 256, 8, 8, 128)) > small
    for bad_ranks in ((136, 16, 16), (16, 136, 16), (16, 16, 136), (16, 12, 16), (16, 16, 0)):
        assert L.lora_mlp_workspace_bytes(L.OP_MLP_FWD, L.mlp_shape(64, 128, 256, *bad_ranks)) == 0, bad_ranks
    assert L.lora_mlp_workspace_bytes(L.OP_MLP_FWD, L.mlp_shape(64, 128, 256, 16, dtype=L.LORA_F32)) == 0
    assert L.lora_mlp_workspace_bytes(L.OP_MLP_FWD, L.mlp_shape(64, 128, 256, 16, act=L.LORA_ACT_GEGLU)) > 0
    assert L.lora_qkv_workspace_bytes(L.OP_QKV_FWD, L.qkv_shape(64, 128, [64, 32, 32], 128)) > 0
    assert L.lora_qkv_workspace_bytes(L.OP_QKV_FWD, L.qkv_shape(64, 128, [64, 32, 32], 136)) == 0
    assert L.lora_mlp_workspace_bytes(L.OP_MLP_FWD, L.mlp_shape(64, 128, 256, 16, act=2)) == 0         # unknown act


def test_entry_points_validate_before_launch(lib):
    """Null / misaligned pointers and bad scalars return an error code; nothing is launched."""
    sh = L.shape(64, 256, 256, 8, L.LORA_F32)
    fake = ctypes.c_void_p(1 << 20)            # never dereferenced: validation fails first
    odd = ctypes.c_void_p((1 << 20) + 4)
    r = lib.lora_linear_fwd(ctypes.byref(sh), None, fake, fake, fake, None, 1.0, fake, None, fake, 1 << 20, None)
    assert r == 1  # INVALID_ARG (X is NULL)
    r = lib.lora_linear_fwd(ctypes.byref(sh), odd, fake, fake, fake, None, 1.0, fake, None, fake, 1 << 20, None)
    assert r == 3  # MISALIGNED
    r = lib.lora_linear_fwd(ctypes.byref(sh), fake, fake, fake, fake, None, float("nan"), fake, None, fake, 1 << 20,
                            None)
    assert r == 1  # non-finite s
    r = lib.lora_linear_fwd(ctypes.byref(sh), fake, fake, fake, fake, None, 1.0, fake, None, fake, 16, None)
    assert r == 4  # workspace too small
    r = lib.lora_linear_fwd(ctypes.byref(sh), fake, fake, fake, fake, None, 1.0, fake, None, None, 1 << 30, None)
    assert r == 4  # workspace missing
    bad = L.shape(64, 256, 256, 0, L.LORA_F32)
    r = lib.lora_linear_bwd(ctypes.byref(bad), fake, fake, fake, fake, None, fake, 1.0, None, fake, fake, None,
                            fake, 1 << 20, None)
    assert r == 1
    r = lib.dora_linear_fwd(ctypes.byref(sh), fake, fake, fake, fake, None, None, fake, 1.0, 1e-12, fake, None, fake,
                            fake, fake, 1 << 20, None)
    assert r == 1  # m is NULL
    r = lib.w8a8_lora_fwd(64, 100, 64, 16, fake, fake, fake, fake, None, None, 1.0, None, fake, None, fake, 1 << 30,
                          None)
    assert r == 2  # d_in not a multiple of 32
    r = lib.w8a8_lora_fwd(64, 128, 64, 16, fake, fake, fake, fake, fake, None, 1.0, None, fake, None, fake, 1 << 30,
                          None)
    assert r == 1  # Z without B
    r = lib.w8a8_lora_fwd(64, 128, 64, 16, fake, fake, fake, fake, None, None, 1.0, None, fake, None, fake, 16, None)
    assert r == 4  # workspace too small
    assert L.w8a8_workspace_bytes(64, 128, 64) >= 256 + 64 * 128 * 2 + 64 * 128 * 2
    r = lib.w8a8_quantize_rows(4, 12, fake, fake, fake, None, 0, None, None)
    assert r == 2  # cols % 8
    mlp = L.mlp_shape(64, 128, 256, 16)
    pr = L.LoraProj(1 << 20, 1 << 20, 1 << 20, 1.0)
    r = lib.lora_mlp_swiglu_fwd(ctypes.byref(mlp), fake, ctypes.byref(pr), None, ctypes.byref(pr), fake, fake, fake,
                                fake, fake, fake, fake, 1 << 30, None)
    assert r == 1  # up projection missing


def test_dropout_entry_points_validate_before_launch(lib):
    """The input-dropout calls: bf16 only, a mask for M > 0, a finite non-negative keep scale and
    the workspace they ask for (the plain layer's when d_in is a multiple of 16, which lets the
    rank-r passes read the mask beside X; else one that also holds the masked input); nothing is
    launched on any of these errors."""
    sh = L.shape(64, 256, 256, 8, L.LORA_BF16)
    fake = ctypes.c_void_p(1 << 20)
    ws_need = L.lora_workspace_bytes(L.OP_DROPOUT_FWD, sh)
    assert ws_need == L.lora_workspace_bytes(L.OP_LINEAR_FWD, sh)
    assert L.lora_workspace_bytes(L.OP_DROPOUT_BWD, sh) == L.lora_workspace_bytes(L.OP_LINEAR_BWD, sh)
    odd = L.shape(64, 264, 256, 8, L.LORA_BF16)   # 264-byte mask rows: Xd is written
    assert (L.lora_workspace_bytes(L.OP_DROPOUT_FWD, odd)
            >= L.lora_workspace_bytes(L.OP_LINEAR_FWD, odd) + 64 * 264 * 2)
    assert (L.lora_workspace_bytes(L.OP_DROPOUT_BWD, odd)
            >= L.lora_workspace_bytes(L.OP_LINEAR_BWD, odd) + 64 * 264 * 2)
    f32 = L.shape(64, 256, 256, 8, L.LORA_F32)
    r = lib.lora_linear_dropout_fwd(ctypes.byref(f32), fake, fake, 2.0, fake, fake, fake, None, 1.0, fake, None,
                                    fake, 1 << 30, None)
    assert r == 2  # UNSUPPORTED: bf16 only
    r = lib.lora_linear_dropout_fwd(ctypes.byref(sh), fake, None, 2.0, fake, fake, fake, None, 1.0, fake, None,
                                    fake, 1 << 30, None)
    assert r == 1  # mask is NULL
    for bad_scale in (-1.0, float("nan"), float("inf")):
        r = lib.lora_linear_dropout_fwd(ctypes.byref(sh), fake, fake, bad_scale, fake, fake, fake, None, 1.0, fake,
                                        None, fake, 1 << 30, None)
        assert r == 1
    r = lib.lora_linear_dropout_fwd(ctypes.byref(sh), fake, fake, 2.0, fake, fake, fake, None, 1.0, fake, None,
                                    fake, ws_need - 256, None)
    assert r == 4  # workspace too small
    wb = L.lora_workspace_bytes(L.OP_DROPOUT_BWD, sh)
    r = lib.lora_linear_dropout_bwd(ctypes.byref(sh), fake, None, 2.0, fake, fake, fake, None, fake, 1.0, fake, fake,
                                    fake, None, fake, wb, None)
    assert r == 1  # mask is NULL
    r = lib.lora_linear_dropout_bwd(ctypes.byref(sh), fake, fake, 2.0, fake, fake, fake, None, fake, 1.0, fake, fake,
                                    fake, None, fake, wb - 256, None)
    assert r == 4


def test_qkv_validation(lib):
    """Fused-leaf shapes and arguments are validated before anything is launched."""
    ok = L.qkv_shape(64, 256, [256, 64, 64], 16)
    assert L.lora_qkv_workspace_bytes(L.OP_QKV_FWD, ok) > 0
    assert L.lora_qkv_workspace_bytes(L.OP_QKV_BWD, ok) > 0
    assert L.lora_qkv_workspace_bytes(L.OP_QKV_FWD, L.qkv_shape(64, 256, [256, 64, 64], 32)) > 0   # L r = 96
    assert L.lora_qkv_workspace_bytes(L.OP_QKV_BWD, L.qkv_shape(64, 256, [256, 64, 64], 72)) > 0   # r 72..128
    assert L.lora_qkv_workspace_bytes(L.OP_QKV_FWD, L.qkv_shape(64, 256, [256, 64, 64], 136)) == 0  # r > 128
    assert L.lora_qkv_workspace_bytes(L.OP_QKV_FWD, L.qkv_shape(64, 256, [256, 64, 64], 12)) == 0  # r % 8
    assert L.lora_qkv_workspace_bytes(L.OP_QKV_FWD, L.qkv_shape(64, 256, [256, 60], 16)) == 0      # n % 8
    assert L.lora_qkv_workspace_bytes(L.OP_QKV_FWD, L.qkv_shape(64, 256, [256, 0], 16)) == 0       # empty leaf
    assert L.lora_qkv_workspace_bytes(L.OP_QKV_FWD, L.qkv_shape(64, 256, [256], 16, L.LORA_F32)) == 0
    four = L.qkv_shape(64, 256, [64, 64, 64], 8)
    four.L = 4
    assert L.lora_qkv_workspace_bytes(L.OP_QKV_FWD, four) == 0
    fake = ctypes.c_void_p(1 << 20)
    odd = 1 << 20 | 8
    lv = (L.LoraAdapter * 3)(*[L.LoraAdapter(1 << 20, 1 << 20, 1.0) for _ in range(3)])
    r = lib.lora_qkv_fwd(ctypes.byref(ok), fake, fake, None, None, fake, None, fake, 1 << 30, None)
    assert r == 1  # leaves missing
    lv[1] = L.LoraAdapter(1 << 20, odd, 1.0)
    r = lib.lora_qkv_fwd(ctypes.byref(ok), fake, fake, lv, None, fake, None, fake, 1 << 30, None)
    assert r == 3  # misaligned B of leaf 1
    lv[1] = L.LoraAdapter(1 << 20, 1 << 20, float("inf"))
    r = lib.lora_qkv_fwd(ctypes.byref(ok), fake, fake, lv, None, fake, None, fake, 1 << 30, None)
    assert r == 1  # non-finite s
    lv[1] = L.LoraAdapter(1 << 20, 1 << 20, 1.0)
    r = lib.lora_qkv_fwd(ctypes.byref(ok), fake, fake, lv, None, fake, None, fake, 16, None)
    assert r == 4  # workspace too small
    ptrs = (ctypes.c_void_p * 3)(1 << 20, None, 1 << 20)
    r = lib.lora_qkv_bwd(ctypes.byref(ok), fake, fake, lv, None, fake, None, ptrs, ptrs, None, fake, 1 << 30, None)
    assert r == 1  # dA[1] missing
