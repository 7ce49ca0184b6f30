"""GPU parity of the pre-step (kda_short_conv_qkv, kda_short_conv_qkv_step)
against the fp64 oracle in oracle/shortconv.py.

Bound, per element: the kernel computes in fp32 (SFU exp, reciprocal and
rsqrt, each within a few fp32 ulps) and rounds to bf16 once, so
|gpu - ref| <= ulp_bf16(ref) / 2 + 2e-5 |ref| + 1e-6, with ref the exact
fp64 value; and at least 99 % of the outputs must equal ref rounded to bf16.
The carried states are raw inputs, so they must match bit for bit."""
import numpy as np
import pytest
import torch

from oracle import shortconv as sc
from gated_delta_rule_33_gb300 import synth
from parity_utils import DEV

pytestmark = pytest.mark.gpu
D = 128


def check_bf16(gpu, ref, where=""):
    gpu = gpu.float().cpu().double().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    a = np.abs(ref)
    ulp = np.where(a > 0, np.exp2(np.floor(np.log2(np.maximum(a, 1e-300))) - 7), 0.0)
    err = np.abs(gpu - ref)
    bound = 0.5 * ulp + 2e-5 * a + 1e-6
    bad = err > bound
    assert not bad.any(), f"{where}: {bad.sum()} elements off, worst {err[bad].max()} at ref {ref[bad][0]}"
    rn = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    frac = float((gpu == rn).mean()) if gpu.size else 1.0
    assert frac >= 0.99, f"{where}: only {frac:.4f} of outputs equal the rounded exact value"


def oracle_qkv(inp, heads=None):
    """Oracle on all channels or on the channels of a subset of heads."""
    cols = None if heads is None else np.concatenate([np.arange(h * D, (h + 1) * D) for h in heads])
    outs, finals = [], []
    for z in range(3):
        x = inp.x[z].double().numpy()
        w = inp.w[z].double().numpy()
        st = None if inp.state is None else inp.state[:, z].double().numpy()
        if cols is not None:
            x, w = x[:, cols], w[cols]
            st = None if st is None else st[..., cols]
        cu = None if inp.cu_seqlens is None else inp.cu_seqlens.numpy()
        y, fin = sc.short_conv(x, w, cu, st, norm_dim=D if z < 2 else None)
        outs.append(y)
        finals.append(fin)
    return outs, np.stack(finals, axis=1), cols


def run_gpu(lib, inp, final=True):
    xs = [x.to(DEV) for x in inp.x]
    ws = [w.to(DEV) for w in inp.w]
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.to(DEV)
    st = None if inp.state is None else inp.state.to(DEV)
    q, k, v, fin = lib.short_conv(*xs, *ws, cu_seqlens=cu, conv_state=st, output_final_state=final)
    assert lib.kda_get_last_device_error() == 0
    return [q, k, v], fin


@pytest.mark.parametrize("N,H,with_state", [(1, 2, False), (100, 3, False), (300, 4, True),
                                             (129, 1, True)])
def test_single_sequence(lib, N, H, with_state):
    inp = synth.make_shortconv_inputs(N, H=H, seed=N + H, with_state=with_state)
    ys, fin = run_gpu(lib, inp)
    ref, rfin, _ = oracle_qkv(inp)
    for z in range(3):
        check_bf16(ys[z], ref[z], f"stream {z}")
    np.testing.assert_array_equal(fin.float().cpu().numpy(), rfin)


def test_varlen_with_states_and_short_sequences(lib):
    lens = [0, 1, 2, 3, 17, 0, 200, 5, 128, 0]
    inp = synth.make_shortconv_inputs(lengths=lens, H=3, seed=7, with_state=True)
    ys, fin = run_gpu(lib, inp)
    ref, rfin, _ = oracle_qkv(inp)
    for z in range(3):
        check_bf16(ys[z], ref[z], f"stream {z}")
    np.testing.assert_array_equal(fin.float().cpu().numpy(), rfin)


def test_varlen_without_state(lib):
    lens = synth.varlen_lengths(6, 1, 300, seed=3)
    inp = synth.make_shortconv_inputs(lengths=lens, H=2, seed=8)
    ys, fin = run_gpu(lib, inp)
    ref, rfin, _ = oracle_qkv(inp)
    for z in range(3):
        check_bf16(ys[z], ref[z], f"stream {z}")
    np.testing.assert_array_equal(fin.float().cpu().numpy(), rfin)


def test_empty_batch_passes_states_through(lib):
    inp = synth.make_shortconv_inputs(lengths=[0, 0], H=1, seed=9, with_state=True)
    ys, fin = run_gpu(lib, inp)
    np.testing.assert_array_equal(fin.float().cpu().numpy(), inp.state.float().numpy())


def test_k3_size_sampled_heads(lib):
    """T=4096 with all 96 heads on the GPU; the oracle checks 6 heads."""
    inp = synth.make_shortconv_inputs(4096, H=96, seed=0)
    ys, fin = run_gpu(lib, inp)
    heads = [0, 17, 48, 63, 90, 95]
    ref, rfin, cols = oracle_qkv(inp, heads)
    for z in range(3):
        check_bf16(ys[z][:, cols], ref[z], f"stream {z}")
    np.testing.assert_array_equal(fin[..., cols].float().cpu().numpy(), rfin)


def test_prefill_then_steps_equals_one_pass(lib):
    """A prefill of 37 tokens, then 5 one-token steps through a slot pool,
    equals one pass over all 42 tokens."""
    H, T1, steps = 2, 37, 5
    inp = synth.make_shortconv_inputs(T1 + steps, H=H, seed=11)
    ref, rfin, _ = oracle_qkv(inp)
    C = H * D
    head = synth.ShortConvInputs([x[:T1].contiguous() for x in inp.x], inp.w, None, None)
    ys, fin = run_gpu(lib, head)
    pool = torch.zeros(4, 3, 3, C, dtype=torch.bfloat16, device=DEV)
    pool[2] = fin[0]
    idx = torch.tensor([-1, 2], dtype=torch.int32, device=DEV)   # sequence 0 inactive
    ws = [w.to(DEV) for w in inp.w]
    for t in range(T1, T1 + steps):
        xs = [torch.stack([x[t], x[t]]).to(DEV) for x in inp.x]
        out = lib.short_conv_step(*xs, *ws, pool, idx)
        assert lib.kda_get_last_device_error() == 0
        for z in range(3):
            assert float(out[z][0].abs().max()) == 0.0
            check_bf16(out[z][1:2], ref[z][t:t + 1], f"step {t} stream {z}")
    np.testing.assert_array_equal(pool[2].float().cpu().numpy(), rfin[0])
    assert float(pool[[0, 1, 3]].abs().max()) == 0.0


def test_step_out_of_range_slot_reports(lib):
    H = 1
    inp = synth.make_shortconv_inputs(2, H=H, seed=12)
    pool = torch.zeros(2, 3, 3, H * D, dtype=torch.bfloat16, device=DEV)
    idx = torch.tensor([0, 5], dtype=torch.int32, device=DEV)
    xs = [x.to(DEV) for x in inp.x]
    ws = [w.to(DEV) for w in inp.w]
    out = lib.short_conv_step(*xs, *ws, pool, idx)
    assert lib.kda_get_last_device_error() == 1
    for z in range(3):
        assert float(out[z][1].abs().max()) == 0.0
    assert float(pool[1].abs().max()) == 0.0


def test_bad_cu_seqlens_reports(lib):
    inp = synth.make_shortconv_inputs(lengths=[10, 10], H=1, seed=13)
    inp.cu_seqlens[1] = 25          # past cu[2] = 20: not monotone
    xs = [x.to(DEV) for x in inp.x]
    ws = [w.to(DEV) for w in inp.w]
    lib.short_conv(*xs, *ws, cu_seqlens=inp.cu_seqlens.to(DEV))
    assert lib.kda_get_last_device_error() == 1
