"""GPU parity at the boundary's size limits, against the fp64 oracle:
the largest document count the prefill accepts (N = 65,535, the grid's y
limit), and decode and output-gate tensors past 2^31 elements (64-bit
offsets).  The oracle runs on sampled documents or units, each checked
element by element; documents and units are independent.  Tolerances:
tests/kda_testlib.py."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.kda_testlib import compare, f64

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]


def test_prefill_at_the_document_limit(kda):
    """65,535 packed documents (mostly 0-3 tokens, some 4-64, a few multi-chunk
    ones), one head, bf16 d=128 on the tensor-core path."""
    N, d = 65535, 128
    lengths = synth.lengths_many(N, long_docs={0: 200, 32767: 1000, N - 2: 64, N - 1: 130})
    T = sum(lengths)
    inp = synth.custom(T, 1, d, dtype=torch.bfloat16, seed=410, lengths=lengths)
    cu = inp["cu_seqlens"]
    dv = {k_: inp[k_].cuda() for k_ in ("q", "k", "v", "g", "beta")}
    out, fin = kda.kda_prefill(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], None,
                               torch.as_tensor(cu, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    rng = np.random.default_rng(411)
    docs = sorted(set(range(60)) | set(range(N - 60, N)) | {32767} |
                  {int(x) for x in rng.integers(0, N, size=120)})
    rows = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in docs])
    sub_cu = synth.cu_seqlens_of([lengths[n] for n in docs])
    pick = lambda t: f64(t)[rows]
    ref_out, ref_fin = oracle.recurrence(pick(inp["q"]), pick(inp["k"]), pick(inp["v"]),
                                         pick(inp["g"]), pick(inp["beta"]), None, sub_cu)
    compare(out.cpu()[rows], ref_out, torch.bfloat16, "N=65535 outputs (sampled documents)")
    got_fin = fin[torch.as_tensor(docs, device="cuda")].cpu()
    nz = [i for i, n in enumerate(docs) if lengths[n] > 0]
    compare(got_fin[nz], ref_fin[nz], torch.bfloat16, "N=65535 states (sampled documents)")
    empty = [i for i, n in enumerate(docs) if lengths[n] == 0]
    assert empty and torch.all(got_fin[empty] == 0)           # zero-length: the zero start state


def test_decode_state_past_2pow31_elements(kda):
    """1,400 sequences x 96 heads x 128 x 128 = 2.2e9 state elements (8.8 GB):
    the last units sit past 2^31 elements and 2^33 bytes."""
    N, H, d = 1400, 96, 128
    assert N * H * d * d > 2 ** 31
    inp = synth.custom(N, H, d, dtype=torch.bfloat16, seed=420)
    state = torch.empty(N, H, d, d, device="cuda")
    state.normal_(0.0, 0.01, generator=torch.Generator(device="cuda").manual_seed(421))
    units = [0, 1, 777 * H + 5, (N - 2) * H + 94, N * H - 2, N * H - 1]
    s0 = synth.state_units(units, d, seed=422)
    flat = state.view(N * H, d, d)
    flat[torch.as_tensor(units, device="cuda")] = torch.from_numpy(s0).cuda()
    dv = {k_: inp[k_].cuda() for k_ in ("q", "k", "v", "g", "beta")}
    out = kda.kda_decode_step(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], state)
    torch.cuda.synchronize()
    for j, u in enumerate(units):
        n, h = divmod(u, H)
        one = lambda t: f64(t)[n:n + 1, h:h + 1]
        ref_out, ref_fin = oracle.recurrence(one(inp["q"]), one(inp["k"]), one(inp["v"]),
                                             one(inp["g"]), one(inp["beta"]),
                                             s0[j].astype(np.float64)[None, None], None)
        compare(out[n:n + 1, h:h + 1].cpu(), ref_out, torch.bfloat16, f"decode unit {u} output")
        compare(flat[u].cpu()[None, None], ref_fin, torch.bfloat16, f"decode unit {u} state")


def test_output_gate_past_2pow31_elements(kda):
    """180,000 tokens x 96 heads x 128 bf16 channels = 2.2e9 elements per
    tensor; sampled rows at both ends and past the 2^31-element mark."""
    T, H, d = 180000, 96, 128
    assert T * H * d > 2 ** 31
    gen = torch.Generator(device="cuda").manual_seed(430)
    o = torch.randn(T, H, d, device="cuda", generator=gen, dtype=torch.bfloat16)
    z = torch.randn(T, H, d, device="cuda", generator=gen, dtype=torch.bfloat16)
    tok = [0, 1, 90000, 174763, 174764, T - 2, T - 1]      # 174,763 x 96 x 128 ~ 2^31
    small = synth.custom(len(tok), H, d, dtype=torch.bfloat16, seed=431, unit_qk=False)
    o[torch.as_tensor(tok, device="cuda")] = small["v"].cuda()
    z[torch.as_tensor(tok, device="cuda")] = small["q"].cuda()
    w = (0.5 + torch.rand(d, generator=torch.Generator().manual_seed(433))).cuda()
    y = kda.kda_output_gate(o, z, w)
    torch.cuda.synchronize()
    ref = oracle.output_gate(f64(small["v"]), f64(small["q"]), f64(w.cpu()))
    compare(y[torch.as_tensor(tok, device="cuda")].cpu(), ref, torch.bfloat16,
            "output gate past 2^31 elements (sampled rows)")
