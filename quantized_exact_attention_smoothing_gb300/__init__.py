"""GB300-native quantized exact attention with K smoothing.

The computation lives in libsattn.so (hand-written sm_103a CUDA kernels behind
the C ABI of include/sattn.h); this package is its Python binding.
"""
from ._binding import (HEAD_DIM, QBLOCK, KV_TILE, STATUS, SattnError, attention, attention_host,
                       check_status, declared_functions, forward, forward_withhold_v_for_test, library_path, load_library,
                       make_shape, prepare, prepare_buffers, prepare_noalloc, query_sizes, sattn_shape,
                       sattn_sizes, NOALLOC_SCRATCH_BYTES)

__all__ = ["HEAD_DIM", "QBLOCK", "KV_TILE", "STATUS", "SattnError", "attention", "attention_host",
           "check_status", "declared_functions", "forward", "forward_withhold_v_for_test", "library_path", "load_library",
           "make_shape", "prepare", "prepare_buffers", "prepare_noalloc", "query_sizes", "sattn_shape",
           "sattn_sizes", "NOALLOC_SCRATCH_BYTES"]
