"""ctypes binding for libkda (include/kda.h): argument marshalling only.

Each ``kda_*`` function takes torch tensors that already live on the GPU,
passes their device pointers and sizes to the C entry point of the same name
on the current torch stream, and raises ``KDAError`` on a non-OK status.
``gate``/``prefill``/``decode`` are conveniences that allocate the outputs
with torch and call the same entry points.  Nothing here computes any part of
KDA; if libkda.so is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

from . import _build

KDA_BF16 = 0
KDA_FP32 = 1
KDA_ALOG_PER_HEAD = 0
KDA_ALOG_PER_CHANNEL = 1
KDA_ALOG_PER_HEAD_CHANNEL = 2

_STATUS_NAMES = {
    0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED_SHAPE",
    3: "KDA_ERR_UNSUPPORTED_DTYPE", 4: "KDA_ERR_MISALIGNED", 5: "KDA_ERR_WORKSPACE_TOO_SMALL",
    6: "KDA_ERR_CUDA", 7: "KDA_ERR_DEVICE_TIMEOUT", 8: "KDA_ERR_NONFINITE",
    9: "KDA_ERR_NOT_IMPLEMENTED", 10: "KDA_ERR_NO_DEVICE", 11: "KDA_ERR_DECAY_RANGE",
}


class KDAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {_STATUS_NAMES.get(self.status, self.status)}")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libkda.so for sm_103a (in-tree)."""
    return _build.build(force=force, verbose=verbose)


def load():
    """Load libkda.so (it must have been built); declares every entry point."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libkda.so is not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        P, I, I64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        lib.kda_version.argtypes = []
        lib.kda_version.restype = I
        lib.kda_status_string.argtypes = [I]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_gate_fused.argtypes = [P, I, P, I, P, I, P, P, P, I64, I, I, P]
        lib.kda_gate_fused.restype = I
        lib.kda_chunk_prefill_workspace_size.argtypes = [I64, I, I, I, I]
        lib.kda_chunk_prefill_workspace_size.restype = ctypes.c_size_t
        lib.kda_chunk_prefill.argtypes = [P, P, P, P, P, P, I, I64, I, I, I, F, P, P, P, I, P,
                                          ctypes.c_size_t, P]
        lib.kda_chunk_prefill.restype = I
        lib.kda_chunk_prefill_gated.argtypes = [P, P, P, P, I, P, I, P, I, P, P, I, I64, I, I, I, F,
                                                P, P, P, I, P, ctypes.c_size_t, P]
        lib.kda_chunk_prefill_gated.restype = I
        lib.kda_chunk_prefill_noalloc.argtypes = [P, P, P, P, P, P, I, I64, I, I, I, F, P, P, P,
                                                  I, P]
        lib.kda_chunk_prefill_noalloc.restype = I
        lib.kda_recurrent_decode.argtypes = [P, P, P, P, P, P, I, I, I, I, F, P, I, P]
        lib.kda_recurrent_decode.restype = I
        lib.kda_recurrent_decode_indexed.argtypes = [P, P, P, P, P, P, I, P, I, I, I, I, I, F, P,
                                                     I, P]
        lib.kda_recurrent_decode_indexed.restype = I
        lib.kda_short_conv_qkv.argtypes = [P, P, P, P, P, P, P, I, I64, I, P, P, P, P, P, P]
        lib.kda_short_conv_qkv.restype = I
        lib.kda_short_conv_qkv_step.argtypes = [P, P, P, P, P, P, P, P, I, I, I, P, P, P, P]
        lib.kda_short_conv_qkv_step.restype = I
        lib.kda_recurrent_backward_workspace_size.argtypes = [I64, I, I, I, I]
        lib.kda_recurrent_backward_workspace_size.restype = ctypes.c_size_t
        lib.kda_recurrent_backward.argtypes = [P, P, P, P, P, P, I, I64, I, I, I, F, P, P, I, P,
                                               P, P, P, P, P, P, P, ctypes.c_size_t, P]
        lib.kda_recurrent_backward.restype = I
        lib.kda_chunk_backward_workspace_size.argtypes = [I64, I, I, I, I]
        lib.kda_chunk_backward_workspace_size.restype = ctypes.c_size_t
        lib.kda_chunk_backward.argtypes = [P, P, P, P, P, P, I, I64, I, I, I, F, P, P, I, P,
                                           P, P, P, P, P, P, P, ctypes.c_size_t, P]
        lib.kda_chunk_backward.restype = I
        lib.kda_chunk_checkpoints_size.argtypes = [I64, I, I, I, I]
        lib.kda_chunk_checkpoints_size.restype = ctypes.c_size_t
        lib.kda_chunk_prefill_checkpointed.argtypes = [P, P, P, P, P, P, I, I64, I, I, I, F, P, P,
                                                       P, I, P, ctypes.c_size_t, P,
                                                       ctypes.c_size_t, P]
        lib.kda_chunk_prefill_checkpointed.restype = I
        lib.kda_chunk_backward_checkpointed_workspace_size.argtypes = [I64, I, I, I, I]
        lib.kda_chunk_backward_checkpointed_workspace_size.restype = ctypes.c_size_t
        lib.kda_chunk_backward_checkpointed.argtypes = [P, P, P, P, P, P, I, I64, I, I, I, F, P,
                                                        ctypes.c_size_t, P, I, P, P, P, P, P, P,
                                                        P, P, ctypes.c_size_t, P]
        lib.kda_chunk_backward_checkpointed.restype = I
        lib.kda_recurrent_decode_gated.argtypes = [P, P, P, P, I, P, I, P, I, P, P, I, P, I, I, I,
                                                   I, I, F, P, I, P]
        lib.kda_recurrent_decode_gated.restype = I
        lib.kda_gate_backward_workspace_size.argtypes = [I64, I, I]
        lib.kda_gate_backward_workspace_size.restype = ctypes.c_size_t
        lib.kda_gate_backward.argtypes = [P, I, P, I, P, I, P, P, P, P, P, P, P, I64, I, I, P,
                                          ctypes.c_size_t, P]
        lib.kda_gate_backward.restype = I
        lib.kda_debug_check_gate_division.argtypes = [P, P]
        lib.kda_debug_check_gate_division.restype = I
        lib.kda_debug_set_wait_limit.argtypes = [I64, I64]
        lib.kda_debug_set_wait_limit.restype = I
        lib.kda_get_last_device_error.argtypes = [P]
        lib.kda_get_last_device_error.restype = I
        _lib = lib
        return lib


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("libkda needs contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream, device=None) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _check(status: int, where: str):
    if status != 0:
        raise KDAError(status, where)


def kda_version() -> int:
    return load().kda_version()


def kda_status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def kda_gate_fused(f, b, A_log, alog_mode, dt_bias, g_out, beta_out, stream=None):
    N, H, K = f.shape
    st = load().kda_gate_fused(_p(f), _dtype_code(f), _p(b), _dtype_code(b) if b is not None else 0,
                               _p(A_log), int(alog_mode), _p(dt_bias), _p(g_out), _p(beta_out),
                               N, H, K, _stream(stream, f.device))
    _check(st, "kda_gate_fused")


def kda_chunk_prefill_workspace_size(N: int, B: int, H: int, K: int = 128, V: int = 128) -> int:
    return int(load().kda_chunk_prefill_workspace_size(N, B, H, K, V))


def kda_chunk_prefill(q, k, v, g, beta, cu_seqlens, scale, initial_state, final_state, o,
                      workspace, stream=None):
    N, H, K = q.shape
    V = v.shape[-1]
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().kda_chunk_prefill(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(cu_seqlens), B, N, H,
                                  K, V, float(scale), _p(initial_state), _p(final_state), _p(o),
                                  _dtype_code(o), _p(workspace), ws_bytes,
                                  _stream(stream, q.device))
    _check(st, "kda_chunk_prefill")


def kda_chunk_prefill_gated(q, k, v, f, b, A_log, alog_mode, dt_bias, cu_seqlens, scale,
                            initial_state, final_state, o, workspace, stream=None):
    """Chunked prefill with the gate computed in the kernel from f, b, A_log, dt_bias."""
    N, H, K = q.shape
    V = v.shape[-1]
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().kda_chunk_prefill_gated(_p(q), _p(k), _p(v), _p(f), _dtype_code(f), _p(b),
                                        _dtype_code(b), _p(A_log), int(alog_mode), _p(dt_bias),
                                        _p(cu_seqlens), B, N, H, K, V, float(scale),
                                        _p(initial_state), _p(final_state), _p(o), _dtype_code(o),
                                        _p(workspace), ws_bytes, _stream(stream, q.device))
    _check(st, "kda_chunk_prefill_gated")


def kda_chunk_prefill_noalloc(q, k, v, g, beta, cu_seqlens, scale, initial_state, final_state, o,
                              stream=None):
    """kda_chunk_prefill with the library's built-in scratch instead of a workspace."""
    N, H, K = q.shape
    V = v.shape[-1]
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    st = load().kda_chunk_prefill_noalloc(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(cu_seqlens), B,
                                          N, H, K, V, float(scale), _p(initial_state),
                                          _p(final_state), _p(o), _dtype_code(o),
                                          _stream(stream, q.device))
    _check(st, "kda_chunk_prefill_noalloc")


def kda_recurrent_decode(q, k, v, g, beta, state, scale, o, stream=None):
    B, H, K = q.shape
    V = v.shape[-1]
    st = load().kda_recurrent_decode(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(state), B, H, K, V,
                                     float(scale), _p(o), _dtype_code(o), _stream(stream, q.device))
    _check(st, "kda_recurrent_decode")


def kda_recurrent_decode_indexed(q, k, v, g, beta, state_pool, state_indices, scale, o,
                                 stream=None):
    B, H, K = q.shape
    V = v.shape[-1]
    st = load().kda_recurrent_decode_indexed(_p(q), _p(k), _p(v), _p(g), _p(beta), _p(state_pool),
                                             _dtype_code(state_pool), _p(state_indices),
                                             state_pool.shape[0], B, H, K, V, float(scale), _p(o),
                                             _dtype_code(o), _stream(stream, q.device))
    _check(st, "kda_recurrent_decode_indexed")


def kda_short_conv_qkv(x_q, x_k, x_v, w_q, w_k, w_v, cu_seqlens, conv_state_in, conv_state_out,
                       q, k, v, stream=None):
    """x_* bf16 [N, C] (or [N, H, 128]); w_* fp32 [C, 4]; states bf16 [B, 3, 3, C]."""
    N = x_q.shape[0]
    C = w_q.shape[0]
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    st = load().kda_short_conv_qkv(_p(x_q), _p(x_k), _p(x_v), _p(w_q), _p(w_k), _p(w_v),
                                   _p(cu_seqlens), B, N, C, _p(conv_state_in),
                                   _p(conv_state_out), _p(q), _p(k), _p(v),
                                   _stream(stream, x_q.device))
    _check(st, "kda_short_conv_qkv")


def kda_short_conv_qkv_step(x_q, x_k, x_v, w_q, w_k, w_v, conv_state_pool, state_indices, q, k,
                            v, stream=None):
    """x_* bf16 [B, C]; conv_state_pool bf16 [num_slots, 3, 3, C]; state_indices int32 [B]
    or None (slot b = sequence b)."""
    B = x_q.shape[0]
    C = w_q.shape[0]
    st = load().kda_short_conv_qkv_step(_p(x_q), _p(x_k), _p(x_v), _p(w_q), _p(w_k), _p(w_v),
                                        _p(conv_state_pool), _p(state_indices),
                                        conv_state_pool.shape[0], B, C, _p(q), _p(k), _p(v),
                                        _stream(stream, x_q.device))
    _check(st, "kda_short_conv_qkv_step")


def kda_recurrent_backward_workspace_size(N, B, H, K=128, V=128) -> int:
    return int(load().kda_recurrent_backward_workspace_size(N, B, H, K, V))


def kda_recurrent_backward(q, k, v, g, beta, cu_seqlens, scale, initial_state, dO, dS_final,
                           dq, dk, dv, dg, dbeta, dS0, workspace, stream=None):
    N, H, K = q.shape
    V = v.shape[-1]
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    st = load().kda_recurrent_backward(
        _p(q), _p(k), _p(v), _p(g), _p(beta), _p(cu_seqlens), B, N, H, K, V, float(scale),
        _p(initial_state), _p(dO), _dtype_code(dO), _p(dS_final), _p(dq), _p(dk), _p(dv), _p(dg),
        _p(dbeta), _p(dS0), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream, q.device))
    _check(st, "kda_recurrent_backward")


def kda_chunk_backward_workspace_size(N, B, H, K=128, V=128) -> int:
    return int(load().kda_chunk_backward_workspace_size(N, B, H, K, V))


def kda_chunk_backward(q, k, v, g, beta, cu_seqlens, scale, initial_state, dO, dS_final,
                       dq, dk, dv, dg, dbeta, dS0, workspace, stream=None):
    N, H, K = q.shape
    V = v.shape[-1]
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    st = load().kda_chunk_backward(
        _p(q), _p(k), _p(v), _p(g), _p(beta), _p(cu_seqlens), B, N, H, K, V, float(scale),
        _p(initial_state), _p(dO), _dtype_code(dO), _p(dS_final), _p(dq), _p(dk), _p(dv), _p(dg),
        _p(dbeta), _p(dS0), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream, q.device))
    _check(st, "kda_chunk_backward")


def kda_chunk_checkpoints_size(N, B, H, K=128, V=128) -> int:
    return int(load().kda_chunk_checkpoints_size(N, B, H, K, V))


def kda_chunk_prefill_checkpointed(q, k, v, g, beta, cu_seqlens, scale, initial_state,
                                   final_state, o, checkpoints, workspace, stream=None):
    N, H, K = q.shape
    V = v.shape[-1]
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().kda_chunk_prefill_checkpointed(
        _p(q), _p(k), _p(v), _p(g), _p(beta), _p(cu_seqlens), B, N, H, K, V, float(scale),
        _p(initial_state), _p(final_state), _p(o), _dtype_code(o), _p(checkpoints),
        checkpoints.numel() * checkpoints.element_size(), _p(workspace), ws_bytes,
        _stream(stream, q.device))
    _check(st, "kda_chunk_prefill_checkpointed")


def kda_chunk_backward_checkpointed_workspace_size(N, B, H, K=128, V=128) -> int:
    return int(load().kda_chunk_backward_checkpointed_workspace_size(N, B, H, K, V))


def kda_chunk_backward_checkpointed(q, k, v, g, beta, cu_seqlens, scale, checkpoints, dO,
                                    dS_final, dq, dk, dv, dg, dbeta, dS0, workspace,
                                    stream=None):
    N, H, K = q.shape
    V = v.shape[-1]
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    st = load().kda_chunk_backward_checkpointed(
        _p(q), _p(k), _p(v), _p(g), _p(beta), _p(cu_seqlens), B, N, H, K, V, float(scale),
        _p(checkpoints), checkpoints.numel() * checkpoints.element_size(), _p(dO),
        _dtype_code(dO), _p(dS_final), _p(dq), _p(dk), _p(dv), _p(dg), _p(dbeta), _p(dS0),
        _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream, q.device))
    _check(st, "kda_chunk_backward_checkpointed")


def kda_recurrent_decode_gated(q, k, v, f, b, A_log, alog_mode, dt_bias, state_pool,
                               state_indices, scale, o, stream=None):
    """state_indices None: slot b for sequence b."""
    B, H, K = q.shape
    V = v.shape[-1]
    st = load().kda_recurrent_decode_gated(
        _p(q), _p(k), _p(v), _p(f), _dtype_code(f), _p(b), _dtype_code(b), _p(A_log),
        int(alog_mode), _p(dt_bias), _p(state_pool), _dtype_code(state_pool), _p(state_indices),
        state_pool.shape[0], B, H, K, V, float(scale), _p(o), _dtype_code(o),
        _stream(stream, q.device))
    _check(st, "kda_recurrent_decode_gated")


def kda_gate_backward_workspace_size(N, H, K) -> int:
    return int(load().kda_gate_backward_workspace_size(N, H, K))


def kda_gate_backward(f, b, A_log, alog_mode, dt_bias, dg, dbeta, df, db, dA_log, ddt_bias,
                      workspace, stream=None):
    N, H, K = f.shape
    st = load().kda_gate_backward(
        _p(f), _dtype_code(f), _p(b), KDA_FP32 if b is None else _dtype_code(b), _p(A_log),
        int(alog_mode), _p(dt_bias), _p(dg), _p(dbeta), _p(df), _p(db), _p(dA_log), _p(ddt_bias),
        N, H, K, _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream, f.device))
    _check(st, "kda_gate_backward")


def kda_debug_check_gate_division(stream=None) -> int:
    """Differing results of the gate's fast division against IEEE division
    over every operand pair of its common path (0: bit-exact)."""
    n = ctypes.c_uint64(0)
    _check(load().kda_debug_check_gate_division(ctypes.byref(n), _stream(stream)),
           "kda_debug_check_gate_division")
    return int(n.value)


def kda_debug_set_wait_limit(copy_polls: int = -1, product_polls: int = -1):
    """Test hook: bound of the chunked prefill's main-loop waits (negative = default)."""
    _check(load().kda_debug_set_wait_limit(int(copy_polls), int(product_polls)),
           "kda_debug_set_wait_limit")


def kda_get_last_device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error word."""
    return int(load().kda_get_last_device_error(_stream(stream)))


# --- conveniences (allocate outputs with torch, then call the entry points) -----

def gate(f, b, A_log, dt_bias, alog_mode=KDA_ALOG_PER_CHANNEL, stream=None
         ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    N, H, K = f.shape
    g = torch.empty(N, H, K, dtype=torch.float32, device=f.device)
    beta = None if b is None else torch.empty(N, H, dtype=torch.float32, device=f.device)
    kda_gate_fused(f, b, A_log, alog_mode, dt_bias, g, beta, stream)
    return g, beta


def prefill(q, k, v, g, beta, cu_seqlens=None, scale=1.0, initial_state=None,
            o_dtype=torch.bfloat16, output_final_state=True, stream=None):
    N, H, K = q.shape
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    o = torch.empty(N, H, v.shape[-1], dtype=o_dtype, device=q.device)
    final = (torch.empty(B, H, K, v.shape[-1], dtype=torch.float32, device=q.device)
             if output_final_state else None)
    ws = torch.empty(max(kda_chunk_prefill_workspace_size(N, B, H, K, v.shape[-1]), 16),
                     dtype=torch.uint8, device=q.device)
    kda_chunk_prefill(q, k, v, g, beta, cu_seqlens, scale, initial_state, final, o, ws, stream)
    return o, final


def prefill_gated(q, k, v, f, b, A_log, dt_bias, alog_mode=KDA_ALOG_PER_CHANNEL, cu_seqlens=None,
                  scale=1.0, initial_state=None, o_dtype=torch.bfloat16, output_final_state=True,
                  stream=None):
    N, H, K = q.shape
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    o = torch.empty(N, H, v.shape[-1], dtype=o_dtype, device=q.device)
    final = (torch.empty(B, H, K, v.shape[-1], dtype=torch.float32, device=q.device)
             if output_final_state else None)
    ws = torch.empty(max(kda_chunk_prefill_workspace_size(N, B, H, K, v.shape[-1]), 16),
                     dtype=torch.uint8, device=q.device)
    kda_chunk_prefill_gated(q, k, v, f, b, A_log, alog_mode, dt_bias, cu_seqlens, scale,
                            initial_state, final, o, ws, stream)
    return o, final


def decode_indexed(q, k, v, g, beta, state_pool, state_indices, scale=1.0, o_dtype=torch.bfloat16,
                   stream=None):
    B, H, K = q.shape
    o = torch.empty(B, H, v.shape[-1], dtype=o_dtype, device=q.device)
    kda_recurrent_decode_indexed(q, k, v, g, beta, state_pool, state_indices, scale, o, stream)
    return o


def short_conv(x_q, x_k, x_v, w_q, w_k, w_v, cu_seqlens=None, conv_state=None,
               output_final_state=True, stream=None):
    """The pre-step on the three streams; returns (q, k, v, final conv state or None)."""
    C = w_q.shape[0]
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    q, k, v = (torch.empty_like(x) for x in (x_q, x_k, x_v))
    final = (torch.empty(B, 3, 3, C, dtype=torch.bfloat16, device=x_q.device)
             if output_final_state else None)
    kda_short_conv_qkv(x_q, x_k, x_v, w_q, w_k, w_v, cu_seqlens, conv_state, final, q, k, v,
                       stream)
    return q, k, v, final


def short_conv_step(x_q, x_k, x_v, w_q, w_k, w_v, conv_state_pool, state_indices=None,
                    stream=None):
    """One token per sequence; the pool is updated in place.  Returns (q, k, v)."""
    q, k, v = (torch.empty_like(x) for x in (x_q, x_k, x_v))
    kda_short_conv_qkv_step(x_q, x_k, x_v, w_q, w_k, w_v, conv_state_pool, state_indices, q, k,
                            v, stream)
    return q, k, v


def backward(q, k, v, g, beta, dO, cu_seqlens=None, scale=1.0, initial_state=None,
             dS_final=None, want_dS0=True, stream=None):
    """Gradients of the recurrence; returns (dq, dk, dv, dg, dbeta, dS0 or None)."""
    N, H, K = q.shape
    V = v.shape[-1]
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    dev = q.device
    dq, dk, dg = (torch.empty(N, H, K, device=dev) for _ in range(3))
    dv = torch.empty(N, H, V, device=dev)
    dbeta = torch.empty(N, H, device=dev)
    dS0 = torch.empty(B, H, K, V, device=dev) if want_dS0 else None
    ws = torch.empty(kda_recurrent_backward_workspace_size(N, B, H, K, V), dtype=torch.uint8,
                     device=dev)
    kda_recurrent_backward(q, k, v, g, beta, cu_seqlens, scale, initial_state, dO, dS_final, dq,
                           dk, dv, dg, dbeta, dS0, ws, stream)
    return dq, dk, dv, dg, dbeta, dS0


def backward_chunked(q, k, v, g, beta, dO, cu_seqlens=None, scale=1.0, initial_state=None,
                     dS_final=None, want_dS0=True, stream=None):
    """Gradients of the recurrence by the chunked tensor-core backward;
    returns (dq, dk, dv, dg, dbeta, dS0 or None)."""
    N, H, K = q.shape
    V = v.shape[-1]
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    dev = q.device
    dq, dk, dg = (torch.empty(N, H, K, device=dev) for _ in range(3))
    dv = torch.empty(N, H, V, device=dev)
    dbeta = torch.empty(N, H, device=dev)
    dS0 = torch.empty(B, H, K, V, device=dev) if want_dS0 else None
    ws = torch.empty(kda_chunk_backward_workspace_size(N, B, H, K, V), dtype=torch.uint8,
                     device=dev)
    kda_chunk_backward(q, k, v, g, beta, cu_seqlens, scale, initial_state, dO, dS_final, dq, dk,
                       dv, dg, dbeta, dS0, ws, stream)
    return dq, dk, dv, dg, dbeta, dS0


def prefill_checkpointed(q, k, v, g, beta, cu_seqlens=None, scale=1.0, initial_state=None,
                         o_dtype=torch.bfloat16, stream=None):
    """The chunked prefill that also keeps the chunk-start states for the backward;
    returns (o, final_state, checkpoints)."""
    N, H, K = q.shape
    V = v.shape[-1]
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    dev = q.device
    o = torch.empty(N, H, V, dtype=o_dtype, device=dev)
    final = torch.empty(B, H, K, V, dtype=torch.float32, device=dev)
    ckpt = torch.empty(kda_chunk_checkpoints_size(N, B, H, K, V), dtype=torch.uint8, device=dev)
    ws = torch.empty(max(kda_chunk_prefill_workspace_size(N, B, H, K, V), 16), dtype=torch.uint8,
                     device=dev)
    kda_chunk_prefill_checkpointed(q, k, v, g, beta, cu_seqlens, scale, initial_state, final, o,
                                   ckpt, ws, stream)
    return o, final, ckpt


def backward_from_checkpoints(q, k, v, g, beta, dO, checkpoints, cu_seqlens=None, scale=1.0,
                              dS_final=None, want_dS0=True, stream=None):
    """Gradients by the chunked backward from the checkpoints of prefill_checkpointed;
    returns (dq, dk, dv, dg, dbeta, dS0 or None)."""
    N, H, K = q.shape
    V = v.shape[-1]
    B = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    dev = q.device
    dq, dk, dg = (torch.empty(N, H, K, device=dev) for _ in range(3))
    dv = torch.empty(N, H, V, device=dev)
    dbeta = torch.empty(N, H, device=dev)
    dS0 = torch.empty(B, H, K, V, device=dev) if want_dS0 else None
    ws = torch.empty(kda_chunk_backward_checkpointed_workspace_size(N, B, H, K, V),
                     dtype=torch.uint8, device=dev)
    kda_chunk_backward_checkpointed(q, k, v, g, beta, cu_seqlens, scale, checkpoints, dO,
                                    dS_final, dq, dk, dv, dg, dbeta, dS0, ws, stream)
    return dq, dk, dv, dg, dbeta, dS0


def decode_gated(q, k, v, f, b, A_log, dt_bias, state_pool, alog_mode=KDA_ALOG_PER_CHANNEL,
                 state_indices=None, scale=1.0, o_dtype=torch.bfloat16, stream=None):
    B, H, K = q.shape
    o = torch.empty(B, H, v.shape[-1], dtype=o_dtype, device=q.device)
    kda_recurrent_decode_gated(q, k, v, f, b, A_log, alog_mode, dt_bias, state_pool,
                               state_indices, scale, o, stream)
    return o


def gate_backward(f, b, A_log, dt_bias, dg, dbeta, alog_mode=KDA_ALOG_PER_CHANNEL,
                  stream=None):
    """Returns (df, db or None, dA_log, ddt_bias)."""
    N, H, K = f.shape
    dev = f.device
    df = torch.empty(N, H, K, device=dev)
    db = None if b is None else torch.empty(N, H, device=dev)
    dA = torch.empty_like(A_log)
    ddt = torch.empty(H, K, device=dev)
    ws = torch.empty(max(kda_gate_backward_workspace_size(N, H, K), 16), dtype=torch.uint8,
                     device=dev)
    kda_gate_backward(f, b, A_log, alog_mode, dt_bias, dg, dbeta, df, db, dA, ddt, ws, stream)
    return df, db, dA, ddt


def decode(q, k, v, g, beta, state, scale=1.0, o_dtype=torch.bfloat16, stream=None):
    B, H, K = q.shape
    o = torch.empty(B, H, v.shape[-1], dtype=o_dtype, device=q.device)
    kda_recurrent_decode(q, k, v, g, beta, state, scale, o, stream)
    return o
