"""ReplaySSM batched SSM-layer decode for B300 (sm_103a).

The compute lives in the CUDA library ``libreplayssm.so`` (C ABI in
``include/replayssm.h``); this package is its Python binding. Importing it
fails if the library has not been built: run
``python -m recurrent_state_fp32_b300.build``.
"""

from .api import (  # noqa: F401
    LayerDims,
    LayerState,
    ReplaySSMError,
    accept,
    consolidate,
    conventional_accept,
    conventional_gdn_step,
    conventional_gdn_verify,
    conventional_mamba2_step,
    copy_sequences,
    gdn_decode,
    mamba2_decode,
    mamba2_decode_noalloc,
    mamba2_fold_decode,
    mamba2_spec_verify,
    refresh_read_copy,
    spec_verify,
    version,
)
