"""GB300 (sm_103a) MLA prefill attention: cache write, dense, indexer top-k, sparse,
the log-sum-exp merge of partial results, the 656-byte row layout and the
non-absorbed (MHA) path for short prompts.

The compute path is the CUDA library ``libmla.so`` (C ABI in include/mla.h);
``binding`` marshals PyTorch tensors into it. Nothing here falls back to a
CPU or PyTorch implementation.
"""
from .binding import (  # noqa: F401
    MLA_DEVERR_BAD_INDEX,
    MLA_DEVERR_BAD_PAGE,
    MLA_DEVERR_SEQ_MISMATCH,
    MLA_OP_DENSE,
    MLA_OP_DENSE_DS,
    MLA_OP_DENSE_HOST,
    MLA_OP_INDEXER,
    MLA_OP_MHA,
    MLA_OP_SPARSE,
    MlaError,
    Seqs,
    chunk_bounds,
    chunk_seqs,
    chunked_prefill_sparse,
    mla_indexer_topk,
    mla_kv_append,
    mla_merge_attn,
    mla_prefill_dense,
    mla_prefill_dense_ds,
    mla_prefill_dense_host,
    mla_prefill_dense_static,
    mla_prefill_mha,
    mla_prefill_sparse,
    mla_prefill_sparse_ds,
    mla_prefill_sparse_host,
    mla_workspace_size,
)
