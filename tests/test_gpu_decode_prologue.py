"""GPU decode step and fused prologue vs the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.kda_testlib import compare, f64, oracle_prologue_stored, gpu_prefill, oracle_prefill, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_matches_oracle(kda, d, dtype):
    N, H = 37, 3
    inp = synth.custom(N, H, d, dtype, seed=600 + d, lengths=[1] * N, init_std=0.1)
    dv = to_device(inp)
    state = dv["init_state"].clone()
    out = kda.kda_decode_step(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], state)
    ref_out, ref_fin = oracle_prefill(inp)
    compare(out, ref_out, dtype, f"decode out d={d}")
    compare(state, ref_fin, dtype, f"decode state d={d}")


def test_decode_equals_one_token_prefill(kda):
    N, H, d = 20, 4, 128
    dv = to_device(synth.custom(N, H, d, torch.bfloat16, seed=610, lengths=[1] * N,
                                init_std=0.1))
    state = dv["init_state"].clone()
    out_d = kda.kda_decode_step(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], state)
    out_p, fin_p = gpu_prefill(kda, dv)
    compare(out_d, f64(out_p), torch.bfloat16, "decode vs prefill out")
    compare(state, f64(fin_p), torch.bfloat16, "decode vs prefill state")


def test_decode_steps_chain_like_prefill(kda):
    """Eight decode steps on one sequence == prefill of those eight tokens."""
    T, H, d = 8, 2, 128
    inp = synth.custom(T, H, d, torch.bfloat16, seed=611, init_std=0.1)
    dv = to_device(inp)
    state = dv["init_state"].clone()
    outs = []
    for t in range(T):
        sl = slice(t, t + 1)
        outs.append(kda.kda_decode_step(dv["q"][sl], dv["k"][sl], dv["v"][sl],
                                        dv["g"][sl], dv["beta"][sl], state))
    ref_out, ref_fin = oracle_prefill(inp)
    compare(torch.cat(outs), ref_out, torch.bfloat16, "chained decode out")
    compare(state, ref_fin, torch.bfloat16, "chained decode state")


def _prologue_ref(inp):
    return oracle.prologue(f64(inp["q_raw"]), f64(inp["k_raw"]), f64(inp["v_raw"]),
                           f64(inp["conv_w"]), f64(inp["z_g"]), f64(inp["z_beta"]),
                           inp["cu_seqlens"])


@pytest.mark.parametrize("d", [16, 64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("lengths", [[77], [5, 0, 40, 1, 33, 2]])
def test_prologue_matches_oracle(kda, d, dtype, lengths):
    T = sum(lengths)
    inp = synth.custom_raw(T, 5, d, dtype, seed=700 + d + len(lengths), lengths=lengths)
    dv = to_device(inp)
    got = kda.kda_prologue(dv["q_raw"], dv["k_raw"], dv["v_raw"], dv["conv_w"], dv["z_g"],
                           dv["z_beta"], torch.as_tensor(inp["cu_seqlens"], dtype=torch.int32))
    ref = _prologue_ref(inp)
    for name, a, b in zip("qkv", got[:3], ref[:3]):
        compare(a, b, dtype, f"prologue {name}")
    compare(got[3], ref[3], torch.float32, "prologue g")
    compare(got[4], ref[4], torch.float32, "prologue beta")
    gg = got[3]
    assert bool(((gg > -5) & (gg < 0)).all()) or bool(((gg >= -5) & (gg <= 0)).all())


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_prologue_across_tiles_and_head_groups(kda, dtype):
    """Documents crossing the 256-token tiles (the causal window carried from
    the previous tile's tokens, reset at each document), and 17 heads of 128
    channels: a full group of 16 heads per CTA and a group with one head."""
    lengths = [300, 0, 290, 3]
    T = sum(lengths)
    inp = synth.custom_raw(T, 17, 128, dtype, seed=760, lengths=lengths)
    dv = to_device(inp)
    got = kda.kda_prologue(dv["q_raw"], dv["k_raw"], dv["v_raw"], dv["conv_w"], dv["z_g"],
                           dv["z_beta"], torch.as_tensor(inp["cu_seqlens"], dtype=torch.int32))
    ref = _prologue_ref(inp)
    for name, a, b in zip("qkv", got[:3], ref[:3]):
        compare(a, b, dtype, f"prologue {name} across tiles")


def test_prologue_without_gates(kda):
    inp = synth.custom_raw(40, 2, 128, torch.bfloat16, seed=720)
    dv = to_device(inp)
    q, k, v, g, b = kda.kda_prologue(dv["q_raw"], dv["k_raw"], dv["v_raw"], dv["conv_w"])
    assert g is None and b is None
    ref = _prologue_ref(inp)
    compare(k, ref[1], torch.bfloat16, "prologue k without gates")


def test_prologue_then_prefill(kda):
    """The fused input path feeding the prefill, against oracle prologue +
    oracle recurrence (the long-context workload's pipeline, small).  The
    prologue hands q, k, v to the prefill as bf16 tensors (the interface's
    qkv dtype), so the reference recurrence takes the oracle prologue's
    values rounded the same way."""
    lengths = [90, 0, 71]
    T = sum(lengths)
    inp = synth.custom_raw(T, 3, 128, torch.bfloat16, seed=730, lengths=lengths)
    dv = to_device(inp)
    cu = torch.as_tensor(inp["cu_seqlens"], dtype=torch.int32, device="cuda")
    q, k, v, g, b = kda.kda_prologue(dv["q_raw"], dv["k_raw"], dv["v_raw"], dv["conv_w"],
                                     dv["z_g"], dv["z_beta"], cu)
    out, fin = kda.kda_prefill(q, k, v, g, b, None, cu)
    rq, rk, rv, rg, rb = oracle_prologue_stored(_prologue_ref(inp), torch.bfloat16)
    ref_out, ref_fin = oracle.recurrence(rq, rk, rv, rg, rb, None, inp["cu_seqlens"])
    compare(out, ref_out, torch.bfloat16, "prologue+prefill out")
    compare(fin, ref_fin, torch.bfloat16, "prologue+prefill state")
