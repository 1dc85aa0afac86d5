"""Deterministic packed assembly on GB300.

Pre-tokenized documents from a weighted mixture of sources become fixed
``[B, T]`` global batches -- tokens, position ids, document ids, loss masks,
a 64-bit fingerprint and a learned-position count per row -- that depend only
on the recipe, the seed and the update index.  The work runs in the CUDA
kernels of ``libnspack.so`` (C ABI in ``include/nspack.h``); this package is
the Python binding.  Importing it fails if the library is not built: there is
no CPU path.
"""
from ._lib import (  # noqa: F401
    NS_ERR_BAD_INPUT,
    NS_ERR_CUDA,
    NS_ERR_DEVICE,
    NS_ERR_EXHAUSTED,
    NS_ERR_HORIZON,
    NS_ERR_INVALID_ARG,
    NS_ERR_OOM,
    NS_OK,
    NS_PACK_DRAIN,
    NS_PACK_HELDOUT,
    NS_PACK_HOST_CORPUS,
    NS_PACK_ORDERED_FREE,
    NS_PACK_SHUFFLE_ROWS,
    NS_PACK_WRAP,
    LIB_PATH,
    SYMBOLS,
    NsPackError,
    ns_pack_batch_fp,
    ns_pack_check,
    ns_pack_fingerprint,
    ns_pack_free,
    ns_pack_info,
    ns_pack_init,
    ns_pack_probe_hash_terms,
    ns_pack_quota_noalloc,
    ns_pack_quota_table,
    ns_pack_step,
    ns_pack_stream_windows,
    ns_pack_strerror,
)
from .packer import Packer, as_u64  # noqa: F401
