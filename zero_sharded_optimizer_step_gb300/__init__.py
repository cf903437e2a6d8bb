"""GB300-native ZeRO sharded optimizer step.

The computation lives in ``libzero.so`` (hand-written CUDA for sm_103a behind
the C ABI declared in ``include/zero.h``); ``binding`` exposes the same entry
points to Python.  PyTorch is used only to own device memory and streams.
"""
from .binding import *  # noqa: F401,F403
from .binding import EXPORTED, LIB_PATH, Ctx, ZeroError  # noqa: F401


def dtype_code(torch_dtype) -> int:
    """The library's element-type code for a torch dtype."""
    import torch
    codes = {torch.float32: ZERO_F32, torch.bfloat16: ZERO_BF16, torch.float16: ZERO_F16}  # noqa: F405
    if torch_dtype not in codes:
        raise ValueError("unsupported dtype %s" % torch_dtype)
    return codes[torch_dtype]


def __getattr__(name):
    # the ZeroAdam facade imports torch; load it on first use
    if name == "ZeroAdam":
        from .optim import ZeroAdam
        return ZeroAdam
    if name == "ShardedZeroAdam":
        from .optim import ShardedZeroAdam
        return ShardedZeroAdam
    if name in ("consolidate_state", "shard_state"):
        from . import optim
        return getattr(optim, name)
    raise AttributeError(name)
