"""MiniMax-M3 two-step block-sparse attention on GB300 (sm_103a).

Index scoring -> top-k block selection -> sparse GQA attention, for packed-
document prefill and for a paged decode cache, as CUDA kernels behind the C ABI
of ``libmsa`` (``include/msa.h``).  This package is the thin Python binding:
PyTorch provides device memory and streams only.
"""
from .binding import (  # noqa: F401
    EXPORTS,
    MsaError,
    Workspace,
    library_path,
    load,
    make_config,
    msa_check_bounded_wait,
    msa_index_produce_decode,
    msa_index_produce_prefill,
    msa_pack,
    msa_pack_metadata,
    msa_select_blocks_decode,
    msa_select_blocks_prefill,
    msa_sparse_attend_decode,
    msa_sparse_attend_decode_fp8kv,
    msa_sparse_attend_decode_mxfp8,
    msa_sparse_attend_prefill,
    msa_sparse_attend_prefill_backward,
    msa_unpack,
    sparse_attention,
    workspace_size,
)
from ._build import build  # noqa: F401
