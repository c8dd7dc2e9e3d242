"""GB300-native packed-sequence metadata: varlen attention boundaries, the
BSHD -> THD conversion and the trainer-side squeeze, as sm_103a CUDA kernels
behind a C ABI (``include/pseq.h``, ``libpseq.so``).

The compute path is the CUDA library only.  Importing this package does not
load it; the first call does, and raises if ``libpseq.so`` has not been built
(``python -m varlen_attention_metadata_gb300.build``).
"""
from .api import (  # noqa: F401
    PackedSeqParams,
    doc_ids_to_seq_lens,
    first_fit_decreasing,
    pack_ffd,
    pseq_doc_ids_to_lengths,
    split_batch_into_thd_chunks,
    thd_chunks_from_batch,
    thd_mask_from_token_ids,
    thd_padding_mask_from_token_ids,
    _thd_padding_mask,
    check_info,
    pack_squeeze,
    packed_seq_params_from_doc_ids,
    process_input_for_thd,
    pseq_from_doc_ids,
    squeeze_bins,
    thd_from_batch,
    thd_gather,
    thd_meta,
    thd_padding_mask,
    to_flash_attention_kwargs,
)
from ._lib import PseqError, load as load_library  # noqa: F401

__version__ = "0.1.0"
