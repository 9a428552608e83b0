"""GB300 (sm_103a) Gated DeltaNet layer: C-ABI library libgdn + thin binding.

The compute path is the CUDA library ``libgdn.so`` (sources in ``csrc/``, ABI
in ``include/gdn.h``); ``binding`` marshals torch tensors into its calls and
``synth`` draws seeded synthetic inputs shaped like the pages' models.
Importing this package does not load the library; the first call does, and
raises if it has not been built.
"""
from .binding import (BF16, F32, GATES_DIRECT, NO_L2NORM, NO_OUTNORM, OP_CHUNK_PREFILL, OP_CONV_STATE_UPDATE,
                      OP_DECODE_STEP, OP_VARLEN_PREFILL, OP_VERIFY_ROWS, RAW_QKV, Config, GdnError, Params,
                      gdn_chunk_prefill, gdn_commit_rows, gdn_conv_state_update, gdn_decode_step, gdn_varlen_prefill,
                      gdn_verify_rows, gdn_workspace_size, load)

__all__ = ["BF16", "F32", "RAW_QKV", "NO_L2NORM", "GATES_DIRECT", "NO_OUTNORM", "OP_CONV_STATE_UPDATE",
           "OP_DECODE_STEP", "OP_VERIFY_ROWS", "OP_CHUNK_PREFILL", "OP_VARLEN_PREFILL", "Config", "Params",
           "GdnError", "load", "gdn_conv_state_update", "gdn_decode_step", "gdn_verify_rows", "gdn_commit_rows",
           "gdn_chunk_prefill", "gdn_varlen_prefill", "gdn_workspace_size"]
