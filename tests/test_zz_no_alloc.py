"""kda_prefill_noalloc: the prefill entry point for callers that cannot
allocate device memory (an engine that owns all device memory, a serving
loop that must not allocate after start-up).  It uses scratch that lives in
the library itself instead of a caller workspace.

The tests call it through the C ABI and check its outputs and final states
against the fp64 oracle with the parity tolerance of every other test
(tests/kda_testlib.py), and bit for bit against the ordinary kda_prefill
entry point on the same inputs: both run the same kernels in the same order,
so a difference of any size means the shared scratch leaked between calls.
Calls follow one another on one stream: two different inputs in a row, a
third call without a status word, and a batch above the 16,320 documents
whose dispatch order fits the scratch (those run in document order).  The
file sits on its own so that pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.kda_testlib import compare, f64, gpu_prefill, oracle_prefill, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]


def _noalloc(kda, d, out, fin, status):
    lib = kda.lib
    fn = lib.kda_prefill_noalloc
    P = ctypes.c_void_p
    fn.argtypes = [P, P, P, P, P, P, P, ctypes.c_int32, ctypes.c_int64, kda.kda_dims, P, P, P, P]
    fn.restype = ctypes.c_int
    cu = torch.as_tensor(d["cu_seqlens"], dtype=torch.int32, device="cuda")
    ptr = lambda t: None if t is None else P(t.data_ptr())
    T = d["q"].shape[0]
    return fn(ptr(d["q"]), ptr(d["k"]), ptr(d["v"]), ptr(d["g"]), ptr(d["beta"]),
              ptr(d.get("init_state")), ptr(cu), cu.numel() - 1, T, kda.dims_of(d["q"]),
              ptr(out), ptr(fin), ptr(status), P(torch.cuda.current_stream().cuda_stream))


def _run(kda, d, like_out, like_fin, with_status=True):
    out = torch.full_like(like_out, float("nan"))
    fin = torch.full_like(like_fin, float("nan"))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda") if with_status else None
    st = _noalloc(kda, d, out, fin, status)
    assert st == kda.KDA_OK, kda.kda_last_error()
    torch.cuda.synchronize()
    if with_status:
        assert int(status.item()) == kda.KDA_DEVICE_OK
    return out, fin


def test_noalloc_matches_oracle_and_prefill(kda):
    cases = [synth.custom(150, 3, 128, torch.bfloat16, seed=950, lengths=[70, 80], init_std=0.05),
             synth.custom(97, 3, 128, torch.bfloat16, seed=951, lengths=[0, 33, 64], init_std=0.1)]
    for i, inp in enumerate(cases):
        d = to_device(inp)
        ref_out, ref_fin = gpu_prefill(kda, d)
        torch.cuda.synchronize()
        out, fin = _run(kda, d, ref_out, ref_fin)
        o_out, o_fin = oracle_prefill(inp)
        compare(out.cpu(), o_out, torch.bfloat16, f"no-alloc outputs, call {i}")
        compare(fin.cpu(), o_fin, torch.bfloat16, f"no-alloc final states, call {i}")
        assert torch.equal(out, ref_out), f"call {i}: outputs differ from kda_prefill"
        assert torch.equal(fin, ref_fin), f"call {i}: final states differ from kda_prefill"
    # a third call, with no status word: the same results as the first call's inputs
    d = to_device(cases[0])
    ref_out, ref_fin = gpu_prefill(kda, d)
    torch.cuda.synchronize()
    out, fin = _run(kda, d, ref_out, ref_fin, with_status=False)
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)


def test_noalloc_beyond_the_order_capacity(kda):
    """20,000 packed documents (more than the 16,320 whose dispatch order fits
    the library's scratch): they run in document order.  Sampled documents
    against the oracle; all of them bit for bit against kda_prefill."""
    N, d = 20000, 128
    lengths = synth.lengths_many(N, seed=960, long_docs={0: 150, 10001: 300, N - 1: 97})
    T = sum(lengths)
    inp = synth.custom(T, 1, d, dtype=torch.bfloat16, seed=961, lengths=lengths)
    cu = inp["cu_seqlens"]
    dv = to_device(inp)
    ref_out, ref_fin = gpu_prefill(kda, dv)
    torch.cuda.synchronize()
    out, fin = _run(kda, dv, ref_out, ref_fin)
    assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
    rng = np.random.default_rng(962)
    docs = sorted(set(range(40)) | set(range(N - 40, N)) | {10001} |
                  {int(x) for x in rng.integers(0, N, size=100)})
    rows = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in docs])
    sub_cu = synth.cu_seqlens_of([lengths[n] for n in docs])
    pick = lambda t: f64(t)[rows]
    o_out, o_fin = oracle.recurrence(pick(inp["q"]), pick(inp["k"]), pick(inp["v"]),
                                     pick(inp["g"]), pick(inp["beta"]), None, sub_cu)
    compare(out.cpu()[rows], o_out, torch.bfloat16, "N=20000 no-alloc outputs (sampled documents)")
    got_fin = fin[torch.as_tensor(docs, device="cuda")].cpu()
    nz = [i for i, n in enumerate(docs) if lengths[n] > 0]
    compare(got_fin[nz], o_fin[nz], torch.bfloat16, "N=20000 no-alloc states (sampled documents)")
    empty = [i for i, n in enumerate(docs) if lengths[n] == 0]
    assert empty and torch.all(got_fin[empty] == 0)
