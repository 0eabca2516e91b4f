"""GPU parity of kda_prologue_prefill (the input path and the recurrence of one
document, segment by segment with the next prologue overlapping the current
prefill) against the fp64 oracle: ShortConv -> Swish -> L2Norm and the gates
("An infra-oriented diagram of Kimi K3", KDA card), then the recurrence.
Segment lengths that split the document unevenly, the conv window crossing
segment boundaries, an initial state, both prefill kernels, T = 0.
Tolerances: tests/kda_testlib.py."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.kda_testlib import compare, f64, oracle_prologue_stored, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]


def check(kda, T, H, d, dtype, seg, seed, with_state):
    raw = synth.custom_raw(T, H, d, dtype, seed=seed)
    dv = to_device(raw)
    s0 = (0.1 * torch.randn(H, d, d, generator=torch.Generator().manual_seed(seed))
          if with_state else None)
    out, fin = kda.kda_prologue_prefill(dv["q_raw"], dv["k_raw"], dv["v_raw"], dv["conv_w"],
                                        dv["z_g"], dv["z_beta"],
                                        None if s0 is None else s0.cuda(), seg)
    # the prologue stores q, k, v in the qkv dtype before the prefill reads them
    rq, rk, rv, rg, rb = oracle_prologue_stored(
        oracle.prologue(f64(raw["q_raw"]), f64(raw["k_raw"]), f64(raw["v_raw"]),
                        f64(raw["conv_w"]), f64(raw["z_g"]), f64(raw["z_beta"]), raw["cu_seqlens"]),
        dtype)
    ref_out, ref_fin = oracle.recurrence(rq, rk, rv, rg, rb,
                                         None if s0 is None else f64(s0)[None], raw["cu_seqlens"])
    compare(out, ref_out, dtype, f"pipeline out T={T} seg={seg}")
    compare(fin, ref_fin[0], dtype, f"pipeline state T={T} seg={seg}")


@pytest.mark.parametrize("T,seg", [(1000, 128), (1000, 300), (700, 4096), (129, 64), (64, 64)])
def test_pipeline_bf16_d128_matches_oracle(kda, T, seg):
    check(kda, T, 3, 128, torch.bfloat16, seg, seed=1100 + T + seg, with_state=True)


def test_pipeline_zero_state(kda):
    check(kda, 800, 2, 128, torch.bfloat16, 192, seed=1150, with_state=False)


@pytest.mark.parametrize("d", [64, 16])
def test_pipeline_fp32_recurrent_path_matches_oracle(kda, d):
    check(kda, 333, 2, d, torch.float32, 128, seed=1170 + d, with_state=True)


def test_pipeline_empty_document_keeps_the_state(kda):
    s0 = torch.randn(2, 128, 128, device="cuda")
    z = torch.empty(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    out, fin = kda.kda_prologue_prefill(z, z, z, torch.zeros(3, 256, 4, device="cuda"),
                                        torch.empty(0, 2, 128, device="cuda"),
                                        torch.empty(0, 2, device="cuda"), s0, 64)
    assert out.numel() == 0
    assert torch.equal(fin, s0)


def test_pipeline_streams_belong_to_the_caller(kda):
    """The prefills run on the caller's stream and the prologues on the
    caller's second stream; the same stream for both runs the segments one
    after another. Either way the results are the same bit for bit, and the
    caller's stream holds the end of the call."""
    raw = to_device(synth.custom_raw(1000, 2, 128, torch.bfloat16, seed=1190))
    args = (raw["q_raw"], raw["k_raw"], raw["v_raw"], raw["conv_w"], raw["z_g"], raw["z_beta"], None, 256)
    main = torch.cuda.Stream(priority=-1)
    side = torch.cuda.Stream(priority=0)
    with torch.cuda.stream(main):
        out_o, fin_o = kda.kda_prologue_prefill(*args, prologue_stream=side)
        done = torch.cuda.Event()
        done.record()
    done.synchronize()                   # the caller's stream alone orders the results
    out_o, fin_o = out_o.clone(), fin_o.clone()
    with torch.cuda.stream(main):
        out_s, fin_s = kda.kda_prologue_prefill(*args, prologue_stream=main)
    torch.cuda.synchronize()
    assert torch.equal(out_o, out_s) and torch.equal(fin_o, fin_s)
