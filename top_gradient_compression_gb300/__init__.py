"""GB300 (sm_103a) hot path of SparCML-style sparse gradient reduction.

P data-parallel nodes are emulated side by side in one GPU's memory. Each
node runs Top-k selection with an error-feedback residual, packs the kept
entries into {uint32 index, fp32 value} streams, optionally quantises the
values to 4 bits with stochastic rounding, and the P streams are sum-reduced
into a sparse result that switches to dense fp32 past 25% fill-in.

The compute lives in libsparcml.so (CUDA, C ABI in include/sparcml.h);
``api`` is its thin Python binding.
"""
from .api import (ReduceOut, SparcmlError, densify, dequantize4, get_status, launch_count,
                  pack, quantize4, reduce_out, reduce_workspace_size, segment_k_total,
                  sparse_reduce, sparse_reduce_q4, status_word, topk_ef, topk_ef_segments,
                  topk_ef_segments_workspace_size, topk_ef_workspace_size, total_k,
                  uniform_segments, workspace)

__all__ = ["ReduceOut", "SparcmlError", "densify", "dequantize4", "get_status", "launch_count",
           "pack", "quantize4", "reduce_out", "reduce_workspace_size", "segment_k_total",
           "sparse_reduce", "sparse_reduce_q4", "status_word", "topk_ef", "topk_ef_segments",
           "topk_ef_segments_workspace_size", "topk_ef_workspace_size", "total_k",
           "uniform_segments", "workspace"]
