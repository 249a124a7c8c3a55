"""lora_linear_fwd_noalloc: the forward for callers that cannot allocate device memory.

It runs the same kernels as lora_linear_fwd with a caller workspace, so its outputs must have
the very same bits, call after call (the shared scratch keeps the previous call's contents);
both are also held to the fp64 oracle.  It must refuse problems larger than its fixed scratch.
This file is collected last so a stop-at-first-failure run has already run every other test;
it also passes on its own in a fresh process.
"""
import pytest
import torch

import datagen as D
import oracle as O
from parity import assert_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def L():
    from dora_adapter_linear_gb300.build import build
    build()
    from dora_adapter_linear_gb300 import _lib
    return _lib


def _inputs(seed):
    case = D.scaled(D.WORKLOADS["lora_4096_bf16"], M=520, d_in=392, d_out=776, r=16, bias=True, seed=seed)
    t = D.make_linear(case)
    return case, {k: v.to(DEV) for k, v in t.items() if v is not None}


def _with_workspace(L, case, g):
    sh = L.shape(case.M, case.d_in, case.d_out, case.r, L.LORA_BF16)
    Y = torch.empty(case.M, case.d_out, dtype=torch.bfloat16, device=DEV)
    Z = torch.empty(case.M, case.r, dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(L.lora_workspace_bytes(L.OP_LINEAR_FWD, sh), dtype=torch.uint8, device=DEV)
    L.lora_linear_fwd(sh, g["X"], g["W0"], g["A"], g["B"], g["bias"], case.s, Y, Z, ws)
    return Y, Z


def _no_alloc(L, case, g):
    sh = L.shape(case.M, case.d_in, case.d_out, case.r, L.LORA_BF16)
    Y = torch.full((case.M, case.d_out), float("nan"), dtype=torch.bfloat16, device=DEV)
    Z = torch.full((case.M, case.r), float("nan"), dtype=torch.bfloat16, device=DEV)
    L.lora_linear_fwd_noalloc(sh, g["X"], g["W0"], g["A"], g["B"], g["bias"], case.s, Y, Z)
    return Y, Z


def test_no_alloc_matches_workspace_entry_point_twice(L):
    for seed in (1301, 1302):   # two calls in a row, different inputs each time
        case, g = _inputs(seed)
        Yn, Zn = _no_alloc(L, case, g)
        Yw, Zw = _with_workspace(L, case, g)
        torch.cuda.synchronize()
        assert torch.equal(Yn, Yw), f"Y differs from the workspace entry point (seed {seed})"
        assert torch.equal(Zn, Zw), f"Z differs from the workspace entry point (seed {seed})"
        X, W0, A, B, bias = (to64(g[k]) for k in ("X", "W0", "A", "B", "bias"))
        assert_close(Yn, O.lora_linear_fwd(X, W0, A, B, case.s, bias), "bf16", f"Y vs oracle (seed {seed})")
        assert_close(Zn, X @ A.T, "bf16", f"Z vs oracle (seed {seed})")


def test_no_alloc_rejects_problems_beyond_its_scratch(L):
    limit = L.LORA_NOALLOC_SCRATCH_BYTES
    M = limit // (2 * 64) + 1024        # M * r * 2 bytes exceeds the fixed scratch at r = 64
    sh = L.shape(M, 64, 64, 64, L.LORA_BF16)
    assert L.lora_workspace_bytes(L.OP_LINEAR_FWD, sh) > limit
    fake = torch.empty(16, dtype=torch.bfloat16, device=DEV)   # never touched: rejected first
    with pytest.raises(L.LoraError) as ei:
        L.lora_linear_fwd_noalloc(sh, fake, fake, fake, fake, None, 1.0, fake, None)
    assert ei.value.status == 4
