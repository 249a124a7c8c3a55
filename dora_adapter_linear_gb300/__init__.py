"""GB300-native (sm_103a) fused low-rank-adapted linear layer.

The compute lives in the C-ABI library ``liblora_gb300.so`` (see ``include/lora_gb300.h``);
``_lib`` is the thin ctypes binding with the ABI's names and ``ops`` allocates outputs and
workspaces with PyTorch before calling it.  There is no CPU or library fallback: if the
library is missing, every call raises.
"""
from . import _lib  # noqa: F401
from . import ops  # noqa: F401
from ._lib import LoraError, lora_abi_version, lora_status_string  # noqa: F401

__all__ = ["_lib", "ops", "LoraError", "lora_abi_version", "lora_status_string"]
