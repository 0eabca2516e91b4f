"""kda_prefill_noalloc: the prefill entry point for callers that cannot
allocate device memory (an engine that owns all device memory, a serving
loop that must not allocate after start-up).  It uses scratch that lives in
the library itself instead of a caller workspace.

The test calls it through the C ABI on two different inputs in a row and
checks each result against the ordinary kda_prefill entry point on the same
inputs, with the bf16 parity tolerance of every other test.  It sits in a
file of its own that pytest collects last."""
import ctypes

import pytest
import torch

import synth
from tests.kda_testlib import compare, gpu_prefill, to_device

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
    st = fn(ptr(d["q"]), ptr(d["k"]), ptr(d["v"]), ptr(d["g"]), ptr(d["beta"]),
            ptr(d.get("init_state")), ptr(cu), cu.numel() - 1, T, kda.dims_of(d["q"]),
            ptr(out), ptr(fin), ptr(status), P(torch.cuda.current_stream().cuda_stream))
    assert st == kda.KDA_OK, kda.kda_last_error()
    return cu


def test_noalloc_matches_prefill_on_two_calls(kda):
    cases = [synth.custom(150, 3, 128, torch.bfloat16, seed=950, lengths=[70, 80], init_std=0.05),
             synth.custom(97, 3, 128, torch.bfloat16, seed=951, lengths=[0, 33, 64], init_std=0.1)]
    for i, inp in enumerate(cases):
        d = to_device(inp)
        ref_out, ref_fin = gpu_prefill(kda, d)
        out = torch.full_like(ref_out, float("nan"))
        fin = torch.full_like(ref_fin, float("nan"))
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        _noalloc(kda, d, out, fin, status)
        torch.cuda.synchronize()
        assert int(status.item()) == kda.KDA_DEVICE_OK
        compare(out, ref_out, torch.bfloat16, f"no-alloc out, call {i}")
        compare(fin, ref_fin, torch.bfloat16, f"no-alloc final state, call {i}")
