"""Host-side checks of the libkda C ABI that need no GPU.

The library must load and export every function include/kda.h declares, and
its argument checks (which run before any CUDA call) must reject bad input
with the documented status codes.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def clib():
    import gated_delta_rule_33_gb300 as kda
    kda.build()
    return kda.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("kda_gate_fused", "kda_chunk_prefill", "kda_chunk_prefill_workspace_size",
                     "kda_recurrent_decode", "kda_get_last_device_error", "kda_status_string",
                     "kda_version"):
        assert required in names


def test_library_exports_every_declared_symbol(clib):
    for name in declared_functions():
        assert hasattr(clib, name), f"libkda.so does not export {name}"


def test_version_and_status_strings(clib):
    import gated_delta_rule_33_gb300 as kda
    assert kda.kda_version() == 10200
    assert kda.kda_status_string(0) == "KDA_OK"
    assert kda.kda_status_string(5) == "KDA_ERR_WORKSPACE_TOO_SMALL"
    assert kda.kda_status_string(99) == "KDA_ERR_UNKNOWN"


def test_workspace_size_rules(clib):
    import gated_delta_rule_33_gb300 as kda
    assert kda.kda_chunk_prefill_workspace_size(4096, 1, 96) > 0
    assert kda.kda_chunk_prefill_workspace_size(4096, 1, 96) < 64 * 1024
    assert kda.kda_chunk_prefill_workspace_size(4096, 1, 96, 64, 128) == 0
    assert kda.kda_chunk_prefill_workspace_size(-1, 1, 96) == 0


def test_checkpoint_sizes(clib):
    import gated_delta_rule_33_gb300 as kda
    # split flags (one int32 per sequence and head, padded to 256 bytes), then one fp32
    # 128 x 128 state per chunk start: N / 64 + B slots per head
    assert kda.kda_chunk_checkpoints_size(4096, 1, 96) == 512 + (64 + 1) * 96 * 65536
    assert kda.kda_chunk_checkpoints_size(100, 3, 2) == 256 + (1 + 3) * 2 * 65536
    assert kda.kda_chunk_checkpoints_size(0, 1, 1) == 256 + 65536
    assert kda.kda_chunk_checkpoints_size(64, 1, 1, 64, 128) == 0
    assert kda.kda_chunk_checkpoints_size(-1, 1, 1) == 0
    # the backward from checkpoints: a 512-byte counter and 528 KB per CTA (up to 160)
    per_cta = 528 * 1024
    assert kda.kda_chunk_backward_checkpointed_workspace_size(4096, 1, 96) == 512 + 96 * per_cta
    assert kda.kda_chunk_backward_checkpointed_workspace_size(64, 4, 96) == 512 + 160 * per_cta
    # the self-contained backward holds a counter, the checkpoints and that workspace
    assert kda.kda_chunk_backward_workspace_size(4096, 1, 96) == (
        512 + kda.kda_chunk_checkpoints_size(4096, 1, 96)
        + kda.kda_chunk_backward_checkpointed_workspace_size(4096, 1, 96))


def test_checkpointed_argument_checks(clib):
    P = _fake()
    need = clib.kda_chunk_checkpoints_size(128, 1, 2, 128, 128)

    def fwd(ck=P, ckb=need, K=128, ws=_fake(), wsb=4096):
        return clib.kda_chunk_prefill_checkpointed(P, P, P, P, P, None, 1, 128, 2, K, 128, 1.0,
                                                   None, None, P, 0, ck, ckb, ws, wsb, None)

    assert fwd(K=64) == 2                        # KDA_ERR_UNSUPPORTED_SHAPE
    assert fwd(ckb=need - 1) == 5                # KDA_ERR_WORKSPACE_TOO_SMALL
    assert fwd(ck=None) == 5
    assert fwd(ck=_fake(0x10008)) == 4           # KDA_ERR_MISALIGNED
    assert fwd(wsb=0) == 5
    wneed = clib.kda_chunk_backward_checkpointed_workspace_size(128, 1, 2, 128, 128)

    def bwd(ck=P, ckb=need, dodt=0, ws=_fake(), wsb=wneed, dq=P):
        return clib.kda_chunk_backward_checkpointed(P, P, P, P, P, None, 1, 128, 2, 128, 128,
                                                    1.0, ck, ckb, P, dodt, None, dq, P, P, P, P,
                                                    None, ws, wsb, None)

    assert bwd(dodt=7) == 3                      # KDA_ERR_UNSUPPORTED_DTYPE
    assert bwd(dq=None) == 1                     # KDA_ERR_INVALID_ARG
    assert bwd(ckb=need - 1) == 5
    assert bwd(wsb=wneed - 1) == 5
    assert bwd(ws=_fake(0x10004)) == 4


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def test_prefill_argument_checks(clib):
    P = _fake()
    ws = _fake()
    args = dict(q=P, k=P, v=P, g=P, beta=P, cu=None, B=1, N=64, H=2, K=128, V=128, scale=1.0,
                s0=None, sf=None, o=P, odt=0, ws=ws, wsb=4096, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return clib.kda_chunk_prefill(a["q"], a["k"], a["v"], a["g"], a["beta"], a["cu"], a["B"],
                                      a["N"], a["H"], a["K"], a["V"], a["scale"], a["s0"], a["sf"],
                                      a["o"], a["odt"], a["ws"], a["wsb"], a["stream"])
    assert call(K=64) == 2                       # KDA_ERR_UNSUPPORTED_SHAPE
    assert call(V=256) == 2
    assert call(odt=7) == 3                      # KDA_ERR_UNSUPPORTED_DTYPE
    assert call(N=-1) == 1                       # KDA_ERR_INVALID_ARG
    assert call(B=2) == 1                        # B > 1 needs cu_seqlens
    assert call(q=None) == 1
    assert call(q=_fake(0x10008)) == 4           # KDA_ERR_MISALIGNED
    assert call(wsb=0) == 5                      # KDA_ERR_WORKSPACE_TOO_SMALL
    assert call(ws=None) == 5


def test_decode_and_gate_argument_checks(clib):
    P = _fake()
    assert clib.kda_recurrent_decode(P, P, P, P, P, P, 4, 2, 128, 64, 1.0, P, 0, None) == 2
    assert clib.kda_recurrent_decode(P, P, P, P, P, None, 4, 2, 128, 128, 1.0, P, 0, None) == 1
    assert clib.kda_recurrent_decode(P, P, P, P, P, P, -1, 2, 128, 128, 1.0, P, 0, None) == 1
    assert clib.kda_recurrent_decode(P, _fake(0x10004), P, P, P, P, 4, 2, 128, 128, 1.0, P, 0,
                                     None) == 4
    # a beta output without b (or b without a beta output) is rejected
    assert clib.kda_gate_fused(P, 0, None, 0, P, 1, P, P, P, 16, 2, 128, None) == 1
    assert clib.kda_gate_fused(P, 0, P, 0, P, 5, P, P, P, 16, 2, 128, None) == 1
    assert clib.kda_gate_fused(P, 2, P, 0, P, 1, P, P, P, 16, 2, 128, None) == 3
    # empty work is a no-op that never touches a device
    assert clib.kda_gate_fused(None, 0, None, 0, P, 1, P, None, None, 0, 2, 128, None) == 0
    assert clib.kda_recurrent_decode(None, None, None, None, None, None, 0, 2, 128, 128, 1.0,
                                     None, 0, None) == 0


def test_indexed_decode_and_gated_prefill_argument_checks(clib):
    P = _fake()
    # kda_recurrent_decode_indexed(q,k,v,g,beta,pool,state_dtype,idx,slots,B,H,K,V,scale,o,odt,s)
    assert clib.kda_recurrent_decode_indexed(P, P, P, P, P, P, 0, P, 4, 2, 2, 64, 128, 1.0, P, 0,
                                             None) == 2
    assert clib.kda_recurrent_decode_indexed(P, P, P, P, P, P, 5, P, 4, 2, 2, 128, 128, 1.0, P, 0,
                                             None) == 3
    assert clib.kda_recurrent_decode_indexed(P, P, P, P, P, P, 0, None, 4, 2, 2, 128, 128, 1.0, P,
                                             0, None) == 1
    assert clib.kda_recurrent_decode_indexed(P, P, P, P, P, P, 0, P, -1, 2, 2, 128, 128, 1.0, P,
                                             0, None) == 1
    assert clib.kda_recurrent_decode_indexed(None, None, None, None, None, None, 0, None, 0, 0, 2,
                                             128, 128, 1.0, None, 0, None) == 0
    # kda_chunk_prefill_gated: f must be bf16; alog_mode must be one of the three
    ws = _fake()
    assert clib.kda_chunk_prefill_gated(P, P, P, P, 1, P, 1, P, 1, P, None, 1, 64, 2, 128, 128,
                                        1.0, None, None, P, 0, ws, 4096, None) == 3
    assert clib.kda_chunk_prefill_gated(P, P, P, P, 0, P, 1, P, 7, P, None, 1, 64, 2, 128, 128,
                                        1.0, None, None, P, 0, ws, 4096, None) == 1
    assert clib.kda_chunk_prefill_gated(P, P, P, P, 0, P, 1, None, 1, P, None, 1, 64, 2, 128, 128,
                                        1.0, None, None, P, 0, ws, 4096, None) == 1


def test_short_conv_argument_checks(clib):
    P, Q, R = _fake(0x10000), _fake(0x900000), _fake(0x1900000)
    # kda_short_conv_qkv(xq,xk,xv,wq,wk,wv,cu,B,N,C,st_in,st_out,q,k,v,stream)
    def call(**kw):
        a = dict(x=(P, P, P), w=(P, P, P), cu=None, B=1, N=16, C=256, si=None, so=None,
                 y=(Q, R, _fake(0x2900000)))
        a.update(kw)
        return clib.kda_short_conv_qkv(*a["x"], *a["w"], a["cu"], a["B"], a["N"], a["C"], a["si"],
                                       a["so"], *a["y"], None)
    assert call(C=200) == 2                      # not a multiple of 128
    assert call(C=0) == 2
    assert call(N=-1) == 1
    assert call(B=2) == 1                        # B > 1 needs cu_seqlens
    assert call(x=(None, P, P)) == 1
    assert call(y=(P, R, _fake(0x2900000))) == 1  # output overlaps an input
    assert call(y=(Q, Q, _fake(0x2900000))) == 1  # two outputs overlap
    assert call(si=P, so=P) == 1                 # state in and out overlap
    assert call(x=(_fake(0x10008), P, P)) == 4
    assert call(N=0) == 0                        # nothing to do, no device touched
    # kda_short_conv_qkv_step(xq,xk,xv,wq,wk,wv,pool,idx,num_slots,B,C,q,k,v,stream)
    assert clib.kda_short_conv_qkv_step(P, P, P, P, P, P, P, None, 1, 2, 256, P, P, P, None) == 1
    assert clib.kda_short_conv_qkv_step(P, P, P, P, P, P, P, P, 4, 70000, 256, P, P, P,
                                        None) == 1
    assert clib.kda_short_conv_qkv_step(P, P, P, P, P, P, None, P, 4, 2, 256, P, P, P, None) == 1
    assert clib.kda_short_conv_qkv_step(P, P, P, P, P, P, P, P, 4, 2, 100, P, P, P, None) == 2
    assert clib.kda_short_conv_qkv_step(P, P, P, P, P, P, P, P, 4, 0, 256, P, P, P, None) == 0


def test_backward_argument_checks(clib):
    import gated_delta_rule_33_gb300 as kda
    P, ws = _fake(), _fake()
    need = kda.kda_recurrent_backward_workspace_size(64, 1, 2)
    assert need > 0 and kda.kda_recurrent_backward_workspace_size(64, 1, 2, 64, 128) == 0

    def call(**kw):
        a = dict(q=P, cu=None, B=1, N=64, K=128, dodt=0, ws=ws, wsb=need)
        a.update(kw)
        # (q,k,v,g,beta,cu,B,N,H,K,V,scale,S0,dO,dO_dtype,dSf,dq,dk,dv,dg,dbeta,dS0,ws,wsb,s)
        return clib.kda_recurrent_backward(a["q"], P, P, P, P, a["cu"], a["B"], a["N"], 2, a["K"],
                                           128, 1.0, None, P, a["dodt"], None, P, P, P, P, P,
                                           None, a["ws"], a["wsb"], None)
    assert call(K=64) == 2
    assert call(dodt=9) == 3
    assert call(N=-1) == 1
    assert call(B=3) == 1
    assert call(q=None) == 1
    assert call(q=_fake(0x10004)) == 4
    assert call(wsb=need - 1) == 5
    assert call(ws=None) == 5


def test_gated_decode_argument_checks(clib):
    P = _fake()
    # (q,k,v,f,fdt,b,bdt,A_log,mode,dt,pool,sdt,idx,slots,B,H,K,V,scale,o,odt,s)
    def call(**kw):
        a = dict(fdt=0, bdt=1, mode=1, idx=P, slots=4, B=2, K=128, pool=P)
        a.update(kw)
        return clib.kda_recurrent_decode_gated(P, P, P, P, a["fdt"], P, a["bdt"], P, a["mode"], P,
                                               a["pool"], 0, a["idx"], a["slots"], a["B"], 2,
                                               a["K"], 128, 1.0, P, 0, None)
    assert call(K=64) == 2
    assert call(fdt=4) == 3
    assert call(mode=3) == 1
    assert call(pool=None) == 1
    assert call(idx=None, slots=1) == 1          # dense slots need num_slots >= B
    assert call(B=0) == 0                        # no work, no device touched
def test_gate_backward_argument_checks(clib):
    import gated_delta_rule_33_gb300 as kda
    P, ws = _fake(), _fake()
    need = kda.kda_gate_backward_workspace_size(64, 2, 128)
    assert need == (2 * 64 + 1) * 2 * 128 * 4

    def call(**kw):
        a = dict(f=P, b=P, dbeta=P, db=P, mode=1, K=128, wsb=need, fdt=0)
        a.update(kw)
        # (f,fdt,b,bdt,A_log,mode,dt,dg,dbeta,df,db,dA,ddt,N,H,K,ws,wsb,s)
        return clib.kda_gate_backward(a["f"], a["fdt"], a["b"], 1, P, a["mode"], P, P, a["dbeta"],
                                      P, a["db"], P, P, 64, 2, a["K"], ws, a["wsb"], None)
    assert call(K=12) == 2
    assert call(fdt=3) == 3
    assert call(mode=5) == 1
    assert call(b=None) == 1                     # beta inputs all or none
    assert call(b=None, dbeta=None, db=None) != 1
    assert call(f=_fake(0x10004)) == 4
    assert call(wsb=need - 4) == 5


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "gated_delta_rule_33_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn
                assert "kdaref" not in text, fn
