"""B300-native packed double-binary matmul (DBF / LoRDBA hot path).

The compute path is libdbf.so (CUDA, sm_103a) behind the C ABI in
include/dbf.h; `double_binary_rank_packed_b300.dbf` is its ctypes binding.
Import the binding explicitly: `from double_binary_rank_packed_b300 import dbf`.
"""

__all__ = ["dbf", "build"]
