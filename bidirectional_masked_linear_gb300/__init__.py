"""LION bidirectional masked linear attention on GB300 (sm_103a).

The operator runs in ``liblion.so`` (hand-written CUDA kernels behind the C
ABI of ``include/lion.h``); :mod:`.lion` is its Python binding and
:mod:`.build` compiles it.  :mod:`.synth` draws the seeded synthetic inputs.
"""
from .lion import (  # noqa: F401
    FORM_CHUNK, FORM_FULL, FORM_RNN, MASK_D, MASK_LIT, MASK_S, PHI_DEFAULT, PHI_ELU1,
    PHI_IDENTITY, PHI_SILU_L2, LionError, attn_fwd, load, rnn_step, status_string, sync_status,
    workspace_bytes,
)
