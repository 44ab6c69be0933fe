"""GB300-native INT4 per-token-head KV cache with a randomized Hadamard
rotation, and paged attention over it.

The compute lives in libkvint4.so (hand-written CUDA for sm_103a behind the C
ABI in include/kvint4.h); this package only marshals torch tensors to it.
"""

from ._lib import (DEV_BAD_BLOCK, DEV_BAD_SEQ, DEV_BAD_SIGNS, DEV_BAD_SLOT, KvInt4Error, attention,
                   attention_workspace_size, library_path, load, status_string, write)

__all__ = ["write", "attention", "attention_workspace_size", "load", "library_path", "status_string",
           "KvInt4Error", "DEV_BAD_SLOT", "DEV_BAD_BLOCK", "DEV_BAD_SEQ", "DEV_BAD_SIGNS"]
