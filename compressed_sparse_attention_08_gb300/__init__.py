"""GB300-native compressed-sparse-attention (CSA) step: thin Python binding over libdsv4.so.

The functions below carry the C ABI's names (include/dsv4.h) and do argument marshalling
only: every step runs in the library's CUDA kernels. PyTorch supplies device memory and
streams. There is no CPU fallback: if the library is missing the calls raise.
"""
from __future__ import annotations

from ._abi import (  # noqa: F401
    DSV4_OK, DSV4_ERR_INVALID_ARG, DSV4_ERR_LAUNCH, DSV4_ERR_BAD_INDEX, DSV4_ERR_TIMEOUT,
    DSV4_ERR_UNSUPPORTED, DSV4_EWORD_BAD_INDEX, DSV4_EWORD_TIMEOUT, Dsv4Error, library,
    library_path, dsv4_compress, dsv4_compress_step, compress_step_state, dsv4_quantize_rows_fp8,
    dsv4_indexer_topk,
    dsv4_indexer_topk_workspace_size,
    dsv4_index_score, dsv4_index_score_workspace_size,
    dsv4_topk, dsv4_topk_workspace_size, dsv4_topk_noalloc, dsv4_sparse_attn_decode,
    dsv4_sparse_attn_workspace_size, dsv4_csa_decode, dsv4_csa_decode_workspace_size,
    dsv4_read_error_word, dsv4_status_string, dsv4_last_launch_count, dsv4_max_comp,
    dsv4_test_wait_fault, dsv4_copy_async, DSV4_WAIT_FAULT_NONE, DSV4_WAIT_FAULT_SCORER_STAGE,
    DSV4_WAIT_FAULT_ATTN_QUERY, EXPORTED_SYMBOLS,
)
