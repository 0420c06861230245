"""GB300-native paged-KV decode attention: bind, append, split-KV decode, merge.

The compute path is libpkv.so (hand-written sm_103a CUDA behind the C ABI of
include/pkv.h); this package only marshals arguments and owns device buffers
through torch.  Importing it loads the library and fails if it is missing.
"""
from . import _abi
from ._abi import *  # noqa: F401,F403  (constants and pkv_* entry points)
from .cascade import CascadeDecoder, choose_prefix_splits
from .engine import BindTracker, DecodeRunner
from .workspace import Workspace

_abi.load()

__all__ = ["Workspace", "DecodeRunner", "BindTracker", "CascadeDecoder", "choose_prefix_splits"] + [
    n for n in dir(_abi) if n.startswith(("pkv_", "PKV_"))]
