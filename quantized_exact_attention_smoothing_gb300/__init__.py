"""GB300-native quantized exact attention with K smoothing.

The computation lives in libsattn.so (hand-written sm_103a CUDA kernels behind
the C ABI of include/sattn.h); this package is its Python binding.
"""
from ._binding import (HEAD_DIM, KV_TILE, NOALLOC_SCRATCH_BYTES, QBLOCK, SMALL_MAX_NKV, STATUS, Graph, SattnError,
                       attention, attention_host, attention_small, small_shape_ok, check_status, declared_functions, exp2_for_test, forward, forward_q_bf16,
                       forward_withhold_v_for_test, int8_quantiser_sweep_for_test, library_path, load_library,
                       make_shape, measure_mma_rate, p8_codes_for_test, prepare, prepare_buffers, prepare_kv, prepare_noalloc,
                       prepare_kv_onepass, check_prepare_status, profile_events, query_sizes, sattn_shape, sattn_sizes)

__all__ = ["HEAD_DIM", "KV_TILE", "NOALLOC_SCRATCH_BYTES", "QBLOCK", "SMALL_MAX_NKV", "STATUS", "Graph", "SattnError",
           "attention", "attention_host", "attention_small", "small_shape_ok", "check_status", "declared_functions", "exp2_for_test", "forward", "forward_q_bf16",
           "forward_withhold_v_for_test", "int8_quantiser_sweep_for_test", "library_path", "load_library",
           "make_shape", "measure_mma_rate", "p8_codes_for_test", "prepare", "prepare_buffers", "prepare_kv", "prepare_noalloc",
           "prepare_kv_onepass", "check_prepare_status", "profile_events", "query_sizes", "sattn_shape", "sattn_sizes"]
