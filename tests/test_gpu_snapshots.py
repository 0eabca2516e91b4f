"""GPU parity of prefix snapshots (kda_prefill_snapshots): the state of a
document after its tokens before an offset, kept so that a request sharing
that prefix resumes from it ("From GPT-2 to Kimi K3, from first principles",
Chapter 14).  The oracle of a snapshot at offset p is the fp64 recurrence
over the document's tokens [bos, p) alone: its final state.  Checked on the
tensor-core path (bf16, d = 128) and the CUDA-core path (fp32, d = 64), on
packed documents with an empty one, snapshots at document ends, resumption
from a snapshot, and offsets that break the rules.  Tolerances:
tests/kda_testlib.py."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.kda_testlib import compare, f64, gpu_prefill, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]

LENGTHS = [200, 0, 513, 64, 130]


def _offsets(lengths, align=64):
    """Every multiple of `align` inside each document, and each non-empty
    document's end."""
    cu = synth.cu_seqlens_of(lengths)
    offs = []
    for n, L in enumerate(lengths):
        bos = int(cu[n])
        offs += [bos + j for j in range(align, L, align)]
        if L > 0:
            offs.append(bos + L)
    return offs


def _oracle_prefix_state(inp, n, p):
    """The fp64 state of document n after its tokens before offset p."""
    cu = inp["cu_seqlens"]
    bos = int(cu[n])
    sl = slice(bos, p)
    s0 = inp.get("init_state")
    s0 = None if s0 is None else s0[n:n + 1]
    _, fin = oracle.recurrence(f64(inp["q"][sl]), f64(inp["k"][sl]), f64(inp["v"][sl]),
                               f64(inp["g"][sl]), f64(inp["beta"][sl]),
                               None if s0 is None else f64(s0), [0, p - bos])
    return fin[0]


def _doc_of(cu, p):
    return int(np.searchsorted(np.asarray(cu), p, side="left")) - 1


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_snapshots_match_oracle(kda, dtype, d):
    T = sum(LENGTHS)
    inp = synth.custom(T, 2, d, dtype, seed=970, lengths=LENGTHS, init_std=0.05)
    dv = to_device(inp)
    offs = _offsets(LENGTHS)
    cu_t = torch.as_tensor(inp["cu_seqlens"], dtype=torch.int32, device="cuda")
    off_t = torch.as_tensor(offs, dtype=torch.int32, device="cuda")
    ws = torch.empty(kda.kda_prefill_workspace_size(2, d, dtype, T, len(LENGTHS)),
                     dtype=torch.uint8, device="cuda")
    out, fin, snaps = kda.kda_prefill_snapshots(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], off_t,
                                                dv["init_state"], cu_t, workspace=ws)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status(ws) == kda.KDA_DEVICE_OK
    # the snapshots leave the outputs and final states as kda_prefill has them
    ref_out, ref_fin = gpu_prefill(kda, dv)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
    cu = inp["cu_seqlens"]
    for i, p in enumerate(offs):
        n = _doc_of(cu, p)
        # the snapshot at a document's end is its final state
        if p == int(cu[n + 1]):
            assert torch.equal(snaps[i], fin[n]), f"snapshot at the end of document {n}"
        compare(snaps[i].cpu(), _oracle_prefix_state(inp, n, p), dtype,
                f"snapshot {i} (document {n}, offset {p - int(cu[n])})")


def test_resume_from_a_snapshot(kda):
    """The tail [p, T) from the snapshot at p gives the full run's tail outputs
    and final state (against the oracle of the whole document)."""
    T, d, p = 600, 128, 256
    inp = synth.custom(T, 2, d, torch.bfloat16, seed=971, init_std=0.05)
    dv = to_device(inp)
    off_t = torch.as_tensor([p], dtype=torch.int32, device="cuda")
    _, _, snaps = kda.kda_prefill_snapshots(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], off_t,
                                            dv["init_state"])
    tail = {k_: dv[k_][p:].contiguous() for k_ in ("q", "k", "v", "g", "beta")}
    out_t, fin_t = kda.kda_prefill(tail["q"], tail["k"], tail["v"], tail["g"], tail["beta"],
                                   snaps[0:1].contiguous())
    torch.cuda.synchronize()
    ref_out, ref_fin = oracle.recurrence(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["g"]),
                                         f64(inp["beta"]), f64(inp["init_state"]))
    compare(out_t.cpu(), ref_out[p:], torch.bfloat16, "outputs resumed from the snapshot")
    compare(fin_t.cpu(), ref_fin, torch.bfloat16, "final state resumed from the snapshot")


@pytest.mark.parametrize("bad", ["misaligned", "descending", "past_T"])
def test_offsets_that_break_the_rules(kda, bad):
    """Rejected in the status word; outputs and final states unaffected."""
    T, d = sum(LENGTHS), 128
    inp = synth.custom(T, 1, d, torch.bfloat16, seed=972, lengths=LENGTHS)
    dv = to_device(inp)
    offs = {"misaligned": [64, 100], "descending": [128, 64], "past_T": [64, T + 64]}[bad]
    cu_t = torch.as_tensor(inp["cu_seqlens"], dtype=torch.int32, device="cuda")
    ws = torch.empty(kda.kda_prefill_workspace_size(1, d, torch.bfloat16, T, len(LENGTHS)),
                     dtype=torch.uint8, device="cuda")
    out, fin, _ = kda.kda_prefill_snapshots(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"],
                                            torch.as_tensor(offs, dtype=torch.int32, device="cuda"),
                                            None, cu_t, workspace=ws)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status(ws) == kda.KDA_DEVICE_BAD_SNAPSHOT
    ref_out, ref_fin = gpu_prefill(kda, dv)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
