"""The five KDA workloads at full size, in the launch configuration the
benchmark times, against the fp64 oracle.  Where the oracle would take
minutes (packed and long-context workloads) it runs on a few sampled heads:
heads are independent, so a sampled head is checked element by element over
all of its tokens.  Tolerances: tests/kda_testlib.py."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.kda_testlib import compare, f64, gpu_prefill, oracle_prefill, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]


def test_workload1_tiny_fp32(kda):
    inp = synth.inputs(1)
    out, fin = gpu_prefill(kda, to_device(inp))
    ref_out, ref_fin = oracle_prefill(inp)
    compare(out, ref_out, torch.float32, "w1 out")
    compare(fin, ref_fin, torch.float32, "w1 state")


def test_workload2_single_sequence(kda):
    inp = synth.inputs(2)
    out, fin = gpu_prefill(kda, to_device(inp))
    ref_out, ref_fin = oracle_prefill(inp)
    compare(out, ref_out, torch.bfloat16, "w2 out")
    compare(fin, ref_fin, torch.bfloat16, "w2 state")


def test_workload2_as_benchmarked(kda):
    """The headline call as the benchmark makes it, without offsets (one
    document of whole chunks: the kernel's narrowest instantiation), against
    the oracle, and bit-identical to the call with offsets (the general one)."""
    inp = synth.inputs(2)
    dv = to_device(inp)
    out, fin = kda.kda_prefill(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv.get("init_state"), None)
    ref_out, ref_fin = oracle_prefill(inp)
    compare(out, ref_out, torch.bfloat16, "w2 out (no offsets)")
    compare(fin, ref_fin, torch.bfloat16, "w2 state (no offsets)")
    out_c, fin_c = gpu_prefill(kda, dv)
    torch.cuda.synchronize()
    assert torch.equal(out, out_c) and torch.equal(fin, fin_c)


def test_workload3_packed_documents(kda):
    heads = [0, 41, 95]
    dev = synth.inputs(3, device="cuda")
    out, fin = gpu_prefill(kda, dev)
    ref_out, ref_fin = oracle_prefill(synth.inputs(3, heads=heads))
    compare(out[:, heads], ref_out, torch.bfloat16, "w3 out (sampled heads)")
    compare(fin[:, heads], ref_fin, torch.bfloat16, "w3 state (sampled heads)")


def test_workload4_long_context_with_prologue(kda):
    heads = [0, 77]
    dev = synth.inputs(4, device="cuda")
    T = dev["q_raw"].shape[0]
    q, k, v, g, b = kda.kda_prologue(dev["q_raw"], dev["k_raw"], dev["v_raw"], dev["conv_w"],
                                     dev["z_g"], dev["z_beta"], None)
    del dev
    assert bool(((g >= -5) & (g <= 0)).all())
    out, fin = kda.kda_prefill(q, k, v, g, b, None, None)
    host = synth.inputs(4, heads=heads)
    rq, rk, rv, rg, rb = oracle.prologue(f64(host["q_raw"]), f64(host["k_raw"]),
                                         f64(host["v_raw"]), f64(host["conv_w"]),
                                         f64(host["z_g"]), f64(host["z_beta"]), None)
    compare(q[:, heads], rq, torch.bfloat16, "w4 prologue q")
    compare(k[:, heads], rk, torch.bfloat16, "w4 prologue k")
    compare(v[:, heads], rv, torch.bfloat16, "w4 prologue v")
    compare(g[:, heads], rg, torch.float32, "w4 prologue g")
    compare(b[:, heads], rb, torch.float32, "w4 prologue beta")
    # the prefill against the oracle recurrence on the inputs it was given: the
    # prologue's own outputs (bf16 q, k, v; fp32 g, beta), each checked above.
    # (The fp32 prologue rounds about 3e-5 of its bf16 outputs to the
    # neighbouring value of the exactly rounded fp64 result; with outputs here
    # ~13x smaller than v, one such v flip moves an output by up to ~5% of its
    # RMS, so an oracle fed the fp64 prologue would charge the prefill with the
    # prologue's rounding.)
    ref_out, ref_fin = oracle.recurrence(*(f64(x[:, heads].cpu()) for x in (q, k, v, g, b)))
    compare(out[:, heads], ref_out, torch.bfloat16, "w4 out (sampled heads)")
    compare(fin[:, heads], ref_fin, torch.bfloat16, "w4 state (sampled heads)")
    assert out.shape == (T, 96, 128)


def test_workload4_pipeline_as_benchmarked(kda):
    """The long-context workload through kda_prologue_prefill with the
    benchmark's 16,384-token segments: the segments split at chunk
    boundaries and carry the fp32 state, so the result is bit-identical to
    the prologue and one prefill over the whole document (checked against the
    oracle above)."""
    dev = synth.inputs(4, device="cuda")
    out_p, fin_p = kda.kda_prologue_prefill(dev["q_raw"], dev["k_raw"], dev["v_raw"], dev["conv_w"],
                                            dev["z_g"], dev["z_beta"], None, 16384)
    q, k, v, g, b = kda.kda_prologue(dev["q_raw"], dev["k_raw"], dev["v_raw"], dev["conv_w"],
                                     dev["z_g"], dev["z_beta"], None)
    del dev
    out, fin = kda.kda_prefill(q, k, v, g, b, None, None)
    assert torch.equal(out_p, out)
    assert torch.equal(fin_p, fin[0])


def test_workload5_decode(kda):
    inp = synth.inputs(5)
    dv = to_device(inp)
    state = dv["init_state"]
    out = kda.kda_decode_step(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], state)
    ref_out, ref_fin = oracle_prefill(inp)
    compare(out, ref_out, torch.bfloat16, "w5 out")
    compare(state, ref_fin, torch.bfloat16, "w5 state")
