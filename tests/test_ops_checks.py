"""The Python wrappers check every operand against X [M, in], W0 [out, in] and A [r, in] before
they allocate or launch anything (the kernels take shapes and strides on trust): CPU tensors are
enough to see the checks fire."""
import pytest
import torch

from dora_adapter_linear_gb300 import ops


def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(*shape, dtype=dtype)


def _ok():
    return dict(X=_t(8, 32), W0=_t(16, 32), A=_t(4, 32), B=_t(16, 4))


@pytest.mark.parametrize("name,bad", [
    ("W0", _t(16, 24)),          # in mismatch
    ("A", _t(4, 24)),            # in mismatch
    ("B", _t(16, 8)),            # r mismatch
    ("B", _t(12, 4)),            # out mismatch
    ("B", _t(16, 4, dtype=torch.float32)),   # dtype mismatch
    ("B", _t(4, 16).t()),        # not contiguous
])
def test_linear_forward_rejects_mismatched_operands(name, bad):
    a = _ok()
    a[name] = bad
    with pytest.raises(ValueError):
        ops.lora_linear_fwd(a["X"], a["W0"], a["A"], a["B"], 1.0)


def test_linear_forward_rejects_bias_and_backward_rejects_dy_z():
    a = _ok()
    with pytest.raises(ValueError):
        ops.lora_linear_fwd(a["X"], a["W0"], a["A"], a["B"], 1.0, bias=_t(15))
    with pytest.raises(ValueError):
        ops.lora_linear_bwd(a["X"], a["W0"], a["A"], a["B"], _t(8, 4), _t(8, 15), 1.0)      # dY
    with pytest.raises(ValueError):
        ops.lora_linear_bwd(a["X"], a["W0"], a["A"], a["B"], _t(8, 5), _t(8, 16), 1.0)      # Z


def test_dropout_and_dora_checks():
    a = _ok()
    with pytest.raises(ValueError):
        ops.lora_linear_dropout_fwd(a["X"], torch.ones(8, 32, dtype=torch.int32), 2.0, a["W0"], a["A"], a["B"], 1.0)
    with pytest.raises(ValueError):
        ops.lora_linear_dropout_fwd(a["X"], torch.ones(8, 31, dtype=torch.uint8), 2.0, a["W0"], a["A"], a["B"], 1.0)
    with pytest.raises(ValueError):   # rows variant: m has one entry per output row
        ops.dora_linear_fwd(a["X"], a["W0"], a["A"], a["B"], _t(32), _t(16, dtype=torch.float32), 1.0)
    with pytest.raises(ValueError):   # column variant: m has one entry per input column
        ops.dora_cols_fwd(a["X"], a["W0"], a["A"], a["B"], _t(16), _t(32, dtype=torch.float32), 1.0)


def test_mlp_and_qkv_checks():
    X = _t(8, 32)
    P = {"g": {"W": _t(48, 32), "A": _t(4, 32), "B": _t(48, 4), "s": 1.0},
         "u": {"W": _t(48, 32), "A": _t(4, 32), "B": _t(48, 4), "s": 1.0},
         "d": {"W": _t(32, 48), "A": _t(4, 48), "B": _t(32, 4), "s": 1.0}}
    bad = dict(P, d=dict(P["d"], A=_t(4, 32)))          # down-projection A must span I = 48
    with pytest.raises(ValueError):
        ops.lora_mlp_swiglu_fwd(X, bad["g"], bad["u"], bad["d"])
    bad = dict(P, u=dict(P["u"], B=_t(48, 8)))           # up-projection B rank differs from its A
    with pytest.raises(ValueError):
        ops.lora_mlp_swiglu_fwd(X, bad["g"], bad["u"], bad["d"])
    # each projection has its own rank: the saved Zgu is [M, r_g + r_u], Zd [M, r_d]
    P3 = dict(P, u=dict(P["u"], A=_t(8, 32), B=_t(48, 8)), d=dict(P["d"], A=_t(16, 48), B=_t(32, 16)))
    saved = {"e": _t(8, 48), "u": _t(8, 48), "h": _t(8, 48), "Zgu": _t(8, 4 + 8), "Zd": _t(8, 16)}
    with pytest.raises(ValueError):   # Zgu sized for one shared rank
        ops.lora_mlp_swiglu_bwd(X, P3["g"], P3["u"], P3["d"], dict(saved, Zgu=_t(8, 8)), _t(8, 32))
    with pytest.raises(ValueError):   # Zd of the wrong rank
        ops.lora_mlp_swiglu_bwd(X, P3["g"], P3["u"], P3["d"], dict(saved, Zd=_t(8, 4)), _t(8, 32))
    W0 = _t(96, 32)
    leaves = [(_t(4, 32), _t(64, 4), 1.0), (_t(4, 32), _t(16, 4), 1.0), (_t(4, 32), _t(16, 4), 1.0)]
    with pytest.raises(ValueError):                       # W0 rows must be the leaves' rows
        ops.lora_qkv_fwd(X, _t(80, 32), leaves)
    with pytest.raises(ValueError):                       # one rank for all leaves
        ops.lora_qkv_fwd(X, W0, leaves[:2] + [(_t(8, 32), _t(16, 8), 1.0)])
    with pytest.raises(ValueError):
        ops.lora_qkv_bwd(X, W0, leaves, _t(8, 12), _t(8, 95))


def test_w8a8_checks():
    Xq, Wq = torch.zeros(8, 32, dtype=torch.int8), torch.zeros(16, 32, dtype=torch.int8)
    sx, sw = torch.ones(8), torch.ones(16)
    with pytest.raises(ValueError):          # weight scales: one per output row
        ops.w8a8_lora_fwd(Xq, sx, Wq, torch.ones(15), None, None, 1.0)
    with pytest.raises(ValueError):          # rank-r input and up-projection disagree
        ops.w8a8_lora_fwd(Xq, sx, Wq, sw, _t(8, 4), _t(16, 8), 1.0)
    with pytest.raises(ValueError):
        ops.w8a8_lora_fwd(Xq.float(), sx, Wq, sw, None, None, 1.0)
    with pytest.raises(ValueError):
        ops.w8a8_lora_bwd(_t(8, 32), Wq, sw, _t(4, 32), _t(16, 4), None, _t(8, 12), 1.0)


def test_fp32_side_inputs_must_be_fp32():
    """Vectors and saved factors the kernels read as fp32 (r0, n, c0, V, U, sx, sw) are rejected in
    any other dtype: a bf16 tensor of the right shape holds half the bytes the kernel would read."""
    a = _ok()
    m_rows, m_cols = _t(16), _t(32)
    with pytest.raises(ValueError):   # r0 in bf16
        ops.dora_linear_fwd(a["X"], a["W0"], a["A"], a["B"], m_rows, _t(16), 1.0)
    with pytest.raises(ValueError):   # m in the wrong dtype
        ops.dora_linear_fwd(a["X"], a["W0"], a["A"], a["B"], _t(16, dtype=torch.float32),
                            _t(16, dtype=torch.float32), 1.0)
    Y, Z, dY = _t(8, 16), _t(8, 4), _t(8, 16)
    with pytest.raises(ValueError):   # n in bf16
        ops.dora_linear_bwd(a["X"], a["W0"], a["A"], a["B"], m_rows, None, Y, Z, _t(16),
                            _t(16, 4, dtype=torch.float32), dY, 1.0)
    with pytest.raises(ValueError):   # V in bf16
        ops.dora_linear_bwd(a["X"], a["W0"], a["A"], a["B"], m_rows, None, Y, Z, _t(16, dtype=torch.float32),
                            _t(16, 4), dY, 1.0)
    with pytest.raises(ValueError):   # c0 in bf16
        ops.dora_cols_fwd(a["X"], a["W0"], a["A"], a["B"], m_cols, _t(32), 1.0)
    with pytest.raises(ValueError):   # U in bf16
        ops.dora_cols_bwd(a["X"], a["W0"], a["A"], a["B"], m_cols, Z, _t(32, dtype=torch.float32), _t(32, 4),
                          dY, 1.0)
    Xq, Wq = torch.zeros(8, 32, dtype=torch.int8), torch.zeros(16, 32, dtype=torch.int8)
    with pytest.raises(ValueError):   # sx in bf16
        ops.w8a8_lora_fwd(Xq, _t(8), Wq, torch.ones(16), None, None, 1.0)
    with pytest.raises(ValueError):   # sw in bf16
        ops.w8a8_lora_fwd(Xq, torch.ones(8), Wq, _t(16), None, None, 1.0)
    with pytest.raises(ValueError):   # rank-r input in fp32
        ops.w8a8_lora_fwd(Xq, torch.ones(8), Wq, torch.ones(16), _t(8, 8, dtype=torch.float32), _t(16, 8), 1.0)
    with pytest.raises(ValueError):   # backward: sw in bf16
        ops.w8a8_lora_bwd(_t(8, 32), Wq, _t(16), _t(4, 32), _t(16, 4), None, _t(8, 16), 1.0)
    with pytest.raises(ValueError):   # quantiser input in fp32
        ops.w8a8_quantize_rows(_t(8, 32, dtype=torch.float32))
