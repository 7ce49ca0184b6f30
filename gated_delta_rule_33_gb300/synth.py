"""Seeded synthetic inputs for KDA, shared by the tests and the benchmark.

This module draws raw inputs only and holds none of the method's arithmetic:
no gate, no decay, no recurrence.  Value distributions follow the Kimi-K3
checkpoint statistics in K3_ARTIFACT_AUDIT.md section 5.1 (A_log median about
-0.15, dt_bias median about -4.6 over a [96, 128] head-channel grid) and the
K3 KDA layer shapes of section 4.1 (96 heads x 128 dims).

Draw order (one CPU ``torch.Generator`` seeded once): sequence lengths (varlen
only), q, k, v, f, b, A_log, dt_bias, initial state.  q and k are N(0, 1)
vectors normalised to unit L2 norm per (token, head) before the cast to the
storage dtype; the parity checks hand the oracle the exact stored values.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import torch

ALOG_PER_HEAD = 0
ALOG_PER_CHANNEL = 1
ALOG_PER_HEAD_CHANNEL = 2


@dataclass
class KDAInputs:
    q: torch.Tensor                 # [N, H, D] (bf16 unless stated)
    k: torch.Tensor                 # [N, H, D]
    v: torch.Tensor                 # [N, H, D]
    f: torch.Tensor                 # [N, H, D] gate pre-activation
    b: torch.Tensor                 # [N, H] fp32 beta logits
    A_log: torch.Tensor             # [D], [H] or [H, D] fp32
    dt_bias: torch.Tensor           # [H, D] fp32
    alog_mode: int
    cu_seqlens: Optional[torch.Tensor]   # int32 [B+1] or None
    initial_state: Optional[torch.Tensor]  # fp32 [B, H, D, D] or None

    @property
    def N(self) -> int:
        return self.q.shape[0]

    @property
    def H(self) -> int:
        return self.q.shape[1]

    @property
    def D(self) -> int:
        return self.q.shape[2]

    @property
    def B(self) -> int:
        return 1 if self.cu_seqlens is None else self.cu_seqlens.numel() - 1


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True)


def varlen_lengths(num_seqs: int, lo: int, hi: int, seed: int = 0) -> List[int]:
    """Lengths drawn uniformly from [lo, hi] (inclusive) with their own generator."""
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (num_seqs,), generator=gen).tolist()


def make_inputs(N: Optional[int] = None, H: int = 96, D: int = 128, *, seed: int = 0,
                lengths: Optional[List[int]] = None, s0_std: float = 0.0,
                dtype: torch.dtype = torch.bfloat16, f_dtype: Optional[torch.dtype] = None,
                alog_mode: int = ALOG_PER_CHANNEL, varlen: bool = False,
                device=None) -> KDAInputs:
    """Draw one KDA problem (on the CPU unless ``device`` is given, in which
    case the same draws come from a generator on that device).

    ``lengths`` (or ``varlen=True`` with N tokens in one sequence) makes a
    packed batch with int32 cu_seqlens.  ``s0_std`` > 0 draws an initial state
    N(0, s0_std) per (sequence, head)."""
    dev = torch.device("cpu") if device is None else torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(seed)
    kw = {"generator": gen, "device": dev}
    if lengths is not None:
        lengths = [int(x) for x in lengths]
        N = sum(lengths)
    if N is None:
        raise ValueError("N or lengths is required")
    f_dtype = dtype if f_dtype is None else f_dtype
    q = _unit_rows(torch.randn(N, H, D, **kw)).to(dtype)
    k = _unit_rows(torch.randn(N, H, D, **kw)).to(dtype)
    v = torch.randn(N, H, D, **kw).to(dtype)
    f = torch.randn(N, H, D, **kw).to(f_dtype)
    b = torch.randn(N, H, **kw)
    if alog_mode == ALOG_PER_HEAD:
        A_log = torch.normal(-0.15, 0.3, (H,), **kw)
    elif alog_mode == ALOG_PER_CHANNEL:
        A_log = torch.normal(-0.15, 0.3, (D,), **kw)
    else:
        A_log = torch.normal(-0.15, 0.3, (H, D), **kw)
    dt_bias = torch.normal(-4.6, 1.2, (H, D), **kw)
    cu = None
    B = 1
    if lengths is not None or varlen:
        lens = lengths if lengths is not None else [N]
        B = len(lens)
        cu = torch.zeros(B + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
        cu = cu.to(dev)
    S0 = None
    if s0_std > 0:
        S0 = torch.normal(0.0, s0_std, (B, H, D, D), **kw)
    return KDAInputs(q, k, v, f, b, A_log.float(), dt_bias.float(), alog_mode, cu, S0)


@dataclass
class DecodeInputs:
    q: torch.Tensor        # [B, H, D] bf16
    k: torch.Tensor
    v: torch.Tensor
    f: torch.Tensor        # [B, H, D] gate pre-activation
    b: torch.Tensor        # [B, H] fp32
    A_log: torch.Tensor
    dt_bias: torch.Tensor
    alog_mode: int
    state: torch.Tensor    # [B, H, D, D] fp32


def make_decode_inputs(B: int, H: int = 96, D: int = 128, *, seed: int = 0,
                       state_std: float = 0.05, dtype: torch.dtype = torch.bfloat16,
                       alog_mode: int = ALOG_PER_CHANNEL,
                       state_device: Optional[torch.device] = None) -> DecodeInputs:
    """One new token per sequence plus a cached state N(0, state_std).

    ``state_device`` draws the (large) state with a generator on that device
    instead of the CPU, seeded from the same seed; the small tensors are
    always drawn on the CPU in the documented order."""
    gen = torch.Generator().manual_seed(seed)
    q = _unit_rows(torch.randn(B, H, D, generator=gen)).to(dtype)
    k = _unit_rows(torch.randn(B, H, D, generator=gen)).to(dtype)
    v = torch.randn(B, H, D, generator=gen).to(dtype)
    f = torch.randn(B, H, D, generator=gen).to(dtype)
    b = torch.randn(B, H, generator=gen)
    if alog_mode == ALOG_PER_HEAD:
        A_log = torch.normal(-0.15, 0.3, (H,), generator=gen)
    elif alog_mode == ALOG_PER_CHANNEL:
        A_log = torch.normal(-0.15, 0.3, (D,), generator=gen)
    else:
        A_log = torch.normal(-0.15, 0.3, (H, D), generator=gen)
    dt_bias = torch.normal(-4.6, 1.2, (H, D), generator=gen)
    if state_device is None or torch.device(state_device).type == "cpu":
        state = torch.normal(0.0, state_std, (B, H, D, D), generator=gen)
    else:
        dgen = torch.Generator(device=state_device).manual_seed(seed + 1)
        state = torch.empty(B, H, D, D, device=state_device)
        state.normal_(0.0, state_std, generator=dgen)
    return DecodeInputs(q, k, v, f, b, A_log.float(), dt_bias.float(), alog_mode, state)


def tiny_config(seed: int = 0) -> KDAInputs:
    """The oracle-scale case: B=1, T=64, H=2, d_k=d_v=16, all fp32, zero state."""
    return make_inputs(64, H=2, D=16, seed=seed, dtype=torch.float32, f_dtype=torch.float32)


@dataclass
class ShortConvInputs:
    x: List[torch.Tensor]            # q, k, v projection outputs, bf16 [N, H*D] each
    w: List[torch.Tensor]            # conv taps, fp32 [H*D, 4] each
    cu_seqlens: Optional[torch.Tensor]
    state: Optional[torch.Tensor]    # bf16 [B, 3, 3, H*D] carried conv state or None


def make_shortconv_inputs(N: Optional[int] = None, H: int = 96, D: int = 128, *, seed: int = 0,
                          lengths: Optional[List[int]] = None, with_state: bool = False,
                          w_std: float = 0.5) -> ShortConvInputs:
    """Inputs of the pre-step: three projection streams x ~ N(0, 1) in bf16,
    taps w ~ N(0, w_std) fp32 per channel (the pages give only their shape,
    [H*D, 1, 4]), optional carried states ~ N(0, 1) in bf16.  Draw order: x_q,
    x_k, x_v, w_q, w_k, w_v, state, from one CPU generator."""
    gen = torch.Generator().manual_seed(seed)
    if lengths is not None:
        lengths = [int(t) for t in lengths]
        N = sum(lengths)
    C = H * D
    x = [torch.randn(N, C, generator=gen).to(torch.bfloat16) for _ in range(3)]
    w = [torch.normal(0.0, w_std, (C, 4), generator=gen) for _ in range(3)]
    cu = None
    B = 1
    if lengths is not None:
        B = len(lengths)
        cu = torch.zeros(B + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    state = None
    if with_state:
        state = torch.randn(B, 3, 3, C, generator=gen).to(torch.bfloat16)
    return ShortConvInputs(x, w, cu, state)
