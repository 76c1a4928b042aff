"""GB300-native (sm_103a) token-choice MoE layer: router, top-k, dispatch,
grouped SwiGLU experts (tcgen05 tensor cores for bf16), combine and the Switch
aux loss, forward and backward, behind the C ABI of libmoe (include/moe.h).

Importing the package loads libmoe.so and raises if it is missing: there is
no fallback path.
"""
from . import _lib  # noqa: F401  (loads libmoe.so or raises)
from ._lib import (MoeCfg, MoeError, cfg_from_workload, make_cfg, status_string,  # noqa: F401
                   version, workspace_bytes)
from . import layer  # noqa: F401

__all__ = ["MoeCfg", "MoeError", "cfg_from_workload", "make_cfg", "status_string", "version",
           "workspace_bytes", "layer"]
