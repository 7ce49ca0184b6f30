"""libkda: Kimi Delta Attention (KDA) on NVIDIA GB300 (sm_103a).

The compute path is the C-ABI shared library ``libkda.so`` (declared in
``include/kda.h``), built from hand-written CUDA in ``csrc/``.  This package is
a thin ctypes binding with the same entry-point names; PyTorch supplies device
memory and streams only.  There is no CPU fallback: every call fails loudly if
the library is missing or no sm_103 GPU is present.
"""
from .kda import (  # noqa: F401
    KDA_ALOG_PER_CHANNEL,
    KDA_ALOG_PER_HEAD,
    KDA_ALOG_PER_HEAD_CHANNEL,
    KDA_BF16,
    KDA_FP32,
    KDAError,
    backward,
    backward_chunked,
    build,
    decode,
    decode_gated,
    decode_indexed,
    gate,
    gate_backward,
    kda_chunk_backward,
    kda_chunk_backward_workspace_size,
    kda_chunk_prefill,
    kda_chunk_prefill_gated,
    kda_chunk_prefill_noalloc,
    kda_chunk_prefill_workspace_size,
    kda_gate_backward,
    kda_gate_backward_workspace_size,
    kda_debug_set_wait_limit,
    kda_gate_fused,
    kda_get_last_device_error,
    kda_recurrent_backward,
    kda_recurrent_backward_workspace_size,
    kda_recurrent_decode,
    kda_recurrent_decode_gated,
    kda_recurrent_decode_indexed,
    kda_short_conv_qkv,
    kda_short_conv_qkv_step,
    kda_status_string,
    kda_version,
    library_path,
    load,
    prefill,
    prefill_gated,
    short_conv,
    short_conv_step,
)
