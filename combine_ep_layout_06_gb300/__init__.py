"""GB300-native (sm_103a) MoE expert-parallel token layout, dispatch and
combine over W logical ranks held in one GPU's HBM.

The compute path is the CUDA library libep_gb300.so (C ABI in
include/ep_api.h); ``EpDispatchCombineOp`` is a thin ctypes binding over it.
Submodules are imported lazily so that ``combine_ep_layout_06_gb300.inputs``
(the seeded input generator) can be used without loading the library.
"""
__all__ = ["EpDispatchCombineConfig", "EpDispatchCombineOp", "EpError",
           "workspace_size"]


def __getattr__(name):
    if name in ("EpDispatchCombineConfig", "EpDispatchCombineOp",
                "workspace_size"):
        from . import op
        return getattr(op, name)
    if name == "EpError":
        from ._lib import EpError
        return EpError
    raise AttributeError(name)
