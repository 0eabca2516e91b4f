"""GPU parity of the segmented prefill (one document split into segments that
run as independent documents, joined by the exact scan of their affine state
maps, "From GPT-2 to Kimi K3, from first principles", Chapter 6) against the
fp64 oracle of the whole document: segment counts that divide the chunks
evenly or not, ragged last segments, more segments than chunks, an initial
state, both prefill kernels, and T = 0.  Tolerances: tests/kda_testlib.py."""
import numpy as np
import pytest
import torch

import synth
from tests.kda_testlib import compare, oracle_prefill, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]


def run(kda, inp, nseg):
    dv = to_device(inp)
    s0 = dv.get("init_state")
    return kda.kda_prefill_segmented(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"],
                                     None if s0 is None else s0[0].contiguous(), nseg)


@pytest.mark.parametrize("T,nseg", [(1000, 1), (1000, 2), (1000, 3), (4096, 7), (700, 40),
                                    (129, 2), (64, 3)])
def test_segmented_bf16_d128_matches_oracle(kda, T, nseg):
    inp = synth.custom(T, 3, 128, torch.bfloat16, seed=900 + T + nseg, init_std=0.1)
    out, fin = run(kda, inp, nseg)
    ref_out, ref_fin = oracle_prefill(inp)
    compare(out, ref_out, torch.bfloat16, f"segmented out T={T} nseg={nseg}")
    compare(fin, ref_fin[0], torch.bfloat16, f"segmented state T={T} nseg={nseg}")


@pytest.mark.parametrize("d,dtype", [(64, torch.float32), (16, torch.float32), (128, torch.float32)])
def test_segmented_other_heads_match_oracle(kda, d, dtype):
    T = 777
    inp = synth.custom(T, 2, d, dtype, seed=950 + d, init_std=0.1)
    out, fin = run(kda, inp, 4)
    ref_out, ref_fin = oracle_prefill(inp)
    compare(out, ref_out, dtype, f"segmented out d={d}")
    compare(fin, ref_fin[0], dtype, f"segmented state d={d}")


def test_segmented_and_plain_prefill_from_zero_state(kda):
    T = 2048
    inp = synth.custom(T, 4, 128, torch.bfloat16, seed=970)
    out, fin = run(kda, inp, 5)
    ref_out, ref_fin = oracle_prefill(inp)
    compare(out, ref_out, torch.bfloat16, "segmented out, zero state")
    compare(fin, ref_fin[0], torch.bfloat16, "segmented state, zero state")
    dv = to_device(inp)
    plain_out, plain_fin = kda.kda_prefill(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"])
    compare(plain_out, ref_out, torch.bfloat16, "plain out, zero state")
    compare(plain_fin, ref_fin, torch.bfloat16, "plain state, zero state")


def test_segmented_empty_document_keeps_the_state(kda):
    s0 = torch.randn(2, 128, 128, device="cuda")
    z = torch.empty(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    zg = torch.empty(0, 2, 128, device="cuda")
    zb = torch.empty(0, 2, device="cuda")
    out, fin = kda.kda_prefill_segmented(z, z, z, zg, zb, s0, 4)
    assert out.numel() == 0
    assert torch.equal(fin, s0)
