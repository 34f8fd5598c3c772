"""GB300-native CONF-KV per-decode-step cache manager.

The decode path (confidence -> budget -> mixed FP16/INT8 decode attention
with attention mass -> EMA -> ranking / bottom-k -> compaction -> INT8
requantisation) runs in the CUDA library libconfkv.so (C ABI declared in
include/confkv.h); this package is its Python binding.
"""
from .binding import (  # noqa: F401
    Cache,
    Config,
    ConfkvError,
    block_offset,
    config_from_workload,
    launch_plan,
    lib,
    make_config,
    status_string,
    workspace_bytes,
)
