"""GPU prefill vs the fp64 oracle: element by element on small and ragged
shapes that span several 64-token chunks with a ragged tail, packed
documents (including empty and one-token ones), every supported head size
and dtype, and the structural invariants (split runs, aliasing, bad
offsets).  Tolerances: tests/kda_testlib.py."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from tests.kda_testlib import compare, f64, gpu_prefill, oracle_prefill, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]


@pytest.mark.parametrize("T", [1, 2, 15, 16, 17, 63, 64, 65, 200])
def test_lengths_bf16_d128(kda, T):
    inp = synth.custom(T, 3, 128, torch.bfloat16, seed=300 + T, init_std=0.01)
    out, fin = gpu_prefill(kda, to_device(inp))
    ref_out, ref_fin = oracle_prefill(inp)
    compare(out, ref_out, torch.bfloat16, f"out T={T}")
    compare(fin, ref_fin, torch.bfloat16, f"state T={T}")


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_head_sizes_and_dtypes(kda, d, dtype):
    inp = synth.custom(150, 4, d, dtype, seed=400 + d, init_std=0.1)
    out, fin = gpu_prefill(kda, to_device(inp))
    ref_out, ref_fin = oracle_prefill(inp)
    compare(out, ref_out, dtype, f"out d={d}")
    compare(fin, ref_fin, dtype, f"state d={d}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_packed_documents_with_empty_and_single(kda, dtype):
    lengths = [70, 0, 1, 129, 0, 64, 3]
    inp = synth.custom(sum(lengths), 2, 128, dtype, seed=500, lengths=lengths, init_std=0.05)
    out, fin = gpu_prefill(kda, to_device(inp))
    ref_out, ref_fin = oracle_prefill(inp)
    compare(out, ref_out, dtype, "out varlen")
    compare(fin, ref_fin, dtype, "state varlen")
    # an empty document hands its initial state straight back
    assert torch.equal(fin[1].cpu(), inp["init_state"][1])


def test_all_documents_empty(kda):
    H, d = 2, 64
    s0 = torch.randn(3, H, d, d, device="cuda")
    e = torch.empty(0, H, d, device="cuda", dtype=torch.bfloat16)
    ef = torch.empty(0, H, d, device="cuda")
    out, fin = kda.kda_prefill(e, e, e, ef, torch.empty(0, H, device="cuda"), s0,
                               torch.zeros(4, dtype=torch.int32, device="cuda"))
    assert out.numel() == 0 and torch.equal(fin, s0)


@pytest.mark.parametrize("T", [64, 96, 4096, 4100, 37])
def test_kernel_instantiations_agree(kda, T):
    """The tensor-core prefill is compiled three times (every option; no
    snapshots or fp32 outputs; one document of whole chunks) and the launcher
    picks the narrowest that fits the call.  The three give the same bits: a
    call without offsets (the whole-chunk one when T is a multiple of 32), one
    with offsets (the general one) and one with a snapshot at the document's
    end (every option)."""
    inp = synth.custom(T, 4, 128, torch.bfloat16, seed=990 + T, init_std=0.05)
    dv = to_device(inp)
    a_out, a_fin = kda.kda_prefill(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["init_state"], None)
    b_out, b_fin = gpu_prefill(kda, dv)
    cu = torch.as_tensor(inp["cu_seqlens"], dtype=torch.int32, device="cuda")
    off = torch.tensor([T], dtype=torch.int32, device="cuda")
    c_out, c_fin, snaps = kda.kda_prefill_snapshots(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], off,
                                                    dv["init_state"], cu)
    torch.cuda.synchronize()
    assert torch.equal(a_out, b_out) and torch.equal(a_fin, b_fin)
    assert torch.equal(c_out, b_out) and torch.equal(c_fin, b_fin)
    assert torch.equal(snaps[0], c_fin[0])
    ref_out, ref_fin = oracle_prefill(inp)
    compare(a_out, ref_out, torch.bfloat16, f"out T={T}")
    compare(a_fin, ref_fin, torch.bfloat16, f"state T={T}")


def test_split_run_carries_state(kda):
    """prefill(T1) then prefill(T2) from its final state == prefill(T1+T2)."""
    inp = to_device(synth.custom(300, 2, 128, torch.bfloat16, seed=502, init_std=0.05))
    out, fin = gpu_prefill(kda, inp)
    a = {k: (v[:130] if isinstance(v, torch.Tensor) and k != "init_state" else v)
         for k, v in inp.items()}
    a["cu_seqlens"] = np.array([0, 130])
    b = {k: (v[130:] if isinstance(v, torch.Tensor) and k != "init_state" else v)
         for k, v in inp.items()}
    b["cu_seqlens"] = np.array([0, 170])
    out_a, fin_a = gpu_prefill(kda, a)
    b["init_state"] = fin_a
    out_b, fin_b = gpu_prefill(kda, b)
    compare(torch.cat([out_a, out_b]), f64(out), torch.bfloat16, "split out")
    compare(fin_b, f64(fin), torch.bfloat16, "split state")


def test_final_state_may_alias_init_state(kda):
    inp = synth.custom(97, 2, 128, torch.bfloat16, seed=503, init_std=0.05)
    d = to_device(inp)
    ref_out, ref_fin = oracle_prefill(inp)
    state = d["init_state"].clone()
    out, fin = kda.kda_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], state, None,
                               final_state=state)
    compare(state, ref_fin, torch.bfloat16, "aliased state")
    compare(out, ref_out, torch.bfloat16, "aliased out")


def test_bad_offsets_set_the_device_status(kda):
    inp = to_device(synth.custom(40, 2, 64, torch.bfloat16, seed=504))
    ws = torch.zeros(kda.kda_prefill_workspace_size(2, 64, torch.bfloat16, 40, 2),
                     dtype=torch.uint8, device="cuda")
    bad = torch.tensor([0, 30, 20], dtype=torch.int32, device="cuda")   # decreasing
    kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], None, bad,
                    workspace=ws)
    assert kda.kda_get_device_status(ws) == kda.KDA_DEVICE_BAD_OFFSETS
    good = torch.tensor([0, 20, 40], dtype=torch.int32, device="cuda")
    kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], None, good,
                    workspace=ws)
    assert kda.kda_get_device_status(ws) == kda.KDA_DEVICE_OK


def test_bounded_wait_reports_timeout(kda):
    """A device-side wait on a barrier nothing arrives on gives up after its
    limit and records KDA_DEVICE_TIMEOUT; the context stays usable."""
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    st = kda.lib.kda_selftest_wait(2_000_000, ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == kda.KDA_OK
    assert kda.kda_get_device_status(ws) == kda.KDA_DEVICE_TIMEOUT
    inp = to_device(synth.custom(20, 2, 128, torch.bfloat16, seed=505))
    kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], None, None, workspace=ws)
    assert kda.kda_get_device_status(ws) == kda.KDA_DEVICE_OK


@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float32)])
def test_longest_first_dispatch_changes_no_result(kda, d, dtype):
    """Packed documents of mixed lengths: with the default workspace the
    documents get their CTAs longest first (the order a first kernel leaves
    after the status word); with a 256-byte workspace they run in document
    order.  Outputs and states are bit-identical, and the oracle agrees."""
    lengths = [5, 300, 0, 64, 1200, 17, 65, 0, 640, 1, 129, 900]
    N, T, H = len(lengths), sum(lengths), 3
    inp = synth.custom(T, H, d, dtype, seed=450 + d, lengths=lengths, init_std=0.05)
    dv = to_device(inp)
    ws_size = kda.kda_prefill_workspace_size(H, d, dtype, T, N)
    assert ws_size >= 256 + 4 * N
    ws_big = torch.full((ws_size,), 0xAB, dtype=torch.uint8, device="cuda")
    ws_small = torch.empty(256, dtype=torch.uint8, device="cuda")
    out_a, fin_a = gpu_prefill(kda, dv, workspace=ws_big)
    out_b, fin_b = gpu_prefill(kda, dv, workspace=ws_small)
    assert torch.equal(out_a, out_b) and torch.equal(fin_a, fin_b)
    ref_out, ref_fin = oracle_prefill(inp)
    compare(out_a, ref_out, dtype, f"packed out d={d}")
    compare(fin_a, ref_fin, dtype, f"packed state d={d}")
    # the order: a permutation of the documents, chunk counts non-increasing
    # (every count here is below 128 chunks, where the buckets are exact)
    order = ws_big[256:256 + 4 * N].view(torch.int32).cpu().tolist()
    assert sorted(order) == list(range(N))
    chunks = [-(-lengths[n] // 64) for n in order]
    assert chunks == sorted(chunks, reverse=True)


@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float32)])
def test_weak_decay_reaches_every_block(kda, d, dtype):
    """Decay 500 times weaker than the workloads' (g in (-0.01, 0), close to
    DeltaNet): tokens a whole chunk apart still interact, so every block of
    the chunk's (I + L)^-1 and every Gram tile pairing counts in the outputs
    (under the workloads' decay the far blocks weigh about e^-40)."""
    lengths = [320, 75]
    inp = synth.custom(sum(lengths), 3, d, dtype, seed=470 + d, lengths=lengths,
                       init_std=0.05, g_scale=0.002)
    assert float(inp["g"].min()) > -0.0101
    out, fin = gpu_prefill(kda, to_device(inp))
    ref_out, ref_fin = oracle_prefill(inp)
    compare(out, ref_out, dtype, f"weak-decay out d={d}")
    compare(fin, ref_fin, dtype, f"weak-decay state d={d}")


def test_gate_at_its_bound(kda):
    """Every g just above the bounded gate's floor of -5 (Kimi K3's
    lower-bounded decay): the tensor-core prefill's 16-token rescaling
    factors reach their e^80 limit, inside fp32 range, and the results still
    match the oracle."""
    lengths = [200, 64]
    inp = synth.custom(sum(lengths), 3, 128, torch.bfloat16, seed=480, lengths=lengths,
                       init_std=0.05, g_const=-5.0 + 1e-6)
    assert float(inp["g"].min()) >= -5.0
    out, fin = gpu_prefill(kda, to_device(inp))
    ref_out, ref_fin = oracle_prefill(inp)
    compare(out, ref_out, torch.bfloat16, "gate at its bound, out")
    compare(fin, ref_fin, torch.bfloat16, "gate at its bound, state")


@pytest.mark.parametrize("where", ["v", "state"])
def test_fp16_operand_range_is_reported(kda, where):
    """The tensor-core path keeps v and the state in fp16 operands: a value at
    or beyond fp16's largest finite magnitude sets KDA_DEVICE_RANGE in the
    status word (inputs of ordinary size leave it clear)."""
    T, H, d = 96, 2, 128
    inp = to_device(synth.custom(T, H, d, torch.bfloat16, seed=980, init_std=0.05))
    init = inp["init_state"].clone()
    v = inp["v"].clone()
    if where == "v":
        v[40, 1, 7] = 7.0e4                      # one value of v past 65504
    else:
        init[0, 0, 3, 5] = 7.0e4                 # one state entry past 65504
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    kda.kda_prefill(inp["q"], inp["k"], v, inp["g"], inp["beta"], init, workspace=ws)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status(ws) == kda.KDA_DEVICE_RANGE
    kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["init_state"], workspace=ws)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status(ws) == kda.KDA_DEVICE_OK
