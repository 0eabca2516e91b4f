"""GPU parity for the rows beyond the core path, against the fp64 oracle:
decode with the ShortConv cache, multi-token verify with a rollback point,
and the head RMSNorm x output-gate epilogue.  Tolerances: tests/kda_testlib.py."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.kda_testlib import compare, f64, to_device

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a GPU")]


def _run_conv_decode(kda, raw, N, K, H, d, conv_state, state):
    """Step the fused decode K times; raw rows n*K + t are token t of sequence n."""
    dv = to_device(raw)
    outs = []
    for t in range(K):
        rows = torch.arange(N, device="cuda") * K + t
        outs.append(kda.kda_decode_step_conv(
            dv["q_raw"][rows].contiguous(), dv["k_raw"][rows].contiguous(),
            dv["v_raw"][rows].contiguous(), dv["conv_w"], conv_state,
            dv["z_g"][rows].contiguous(), dv["z_beta"][rows].contiguous(), state))
    return torch.stack(outs, 1).reshape(N * K, H, d)


@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float32),
                                     (16, torch.float32)])
def test_decode_with_conv_cache_equals_prologue_plus_prefill(kda, d, dtype):
    """K decode steps from an empty conv cache and zero state == the prologue
    over each whole sequence followed by the recurrence (From GPT-2 to Kimi
    K3, Chapter 5: the conv state is cached during decoding)."""
    N, K, H = 6, 7, 3
    raw = synth.custom_raw(N * K, H, d, dtype, seed=800 + d, lengths=[K] * N)
    conv_state = torch.zeros(N, 3, 3, H, d, dtype=dtype, device="cuda")
    state = torch.zeros(N, H, d, d, device="cuda")
    out = _run_conv_decode(kda, raw, N, K, H, d, conv_state, state)
    rq, rk, rv, rg, rb = oracle.prologue(f64(raw["q_raw"]), f64(raw["k_raw"]), f64(raw["v_raw"]),
                                         f64(raw["conv_w"]), f64(raw["z_g"]), f64(raw["z_beta"]),
                                         raw["cu_seqlens"])
    ref_out, ref_fin = oracle.recurrence(rq, rk, rv, rg, rb, None, raw["cu_seqlens"])
    compare(out, ref_out, dtype, f"conv decode out d={d}")
    compare(state, ref_fin, dtype, f"conv decode state d={d}")
    # the cache now holds each sequence's last three raw inputs, bit for bit
    for i, name in enumerate(("q_raw", "k_raw", "v_raw")):
        last = raw[name].reshape(N, K, H, d)[:, K - 3:]
        assert torch.equal(conv_state[:, :, i].cpu(), last)


def test_decode_with_warm_conv_cache_and_state(kda):
    """A non-empty cache (three earlier raw tokens) and a non-zero state:
    equal to the prologue over history + new tokens, keeping the new rows,
    then the recurrence from that state."""
    N, K, H, d = 4, 5, 2, 128
    dtype = torch.bfloat16
    full = synth.custom_raw(N * (K + 3), H, d, dtype, seed=820, lengths=[K + 3] * N)
    resh = lambda t: t.reshape(N, K + 3, *t.shape[1:])
    new = {n_: resh(full[n_])[:, 3:].reshape(N * K, *full[n_].shape[1:]).contiguous()
           for n_ in ("q_raw", "k_raw", "v_raw", "z_g", "z_beta")}
    new["conv_w"] = full["conv_w"]
    hist = torch.stack([resh(full[n_])[:, :3] for n_ in ("q_raw", "k_raw", "v_raw")], 2)
    conv_state = hist.contiguous().to("cuda")                      # [N, 3, 3, H, d]
    s0 = 0.1 * torch.randn(N, H, d, d, generator=torch.Generator().manual_seed(821))
    state = s0.to("cuda")
    out = _run_conv_decode(kda, new, N, K, H, d, conv_state, state)
    rq, rk, rv, rg, rb = oracle.prologue(f64(full["q_raw"]), f64(full["k_raw"]), f64(full["v_raw"]),
                                         f64(full["conv_w"]), f64(full["z_g"]), f64(full["z_beta"]),
                                         full["cu_seqlens"])
    keep = (np.arange(N * (K + 3)) % (K + 3)) >= 3
    cu = np.arange(N + 1) * K
    ref_out, ref_fin = oracle.recurrence(rq[keep], rk[keep], rv[keep], rg[keep], rb[keep],
                                         f64(s0), cu)
    compare(out, ref_out, dtype, "warm conv decode out")
    compare(state, ref_fin, dtype, "warm conv decode state")


@pytest.mark.parametrize("d,dtype,K,accept", [
    (128, torch.bfloat16, 7, [0, 3, 7, 1, 5]),
    (64, torch.float32, 7, [0, 3, 7, 1, 5]),
    (128, torch.float32, 6, [2, 4, 6, 0, 5]),      # even K: every draft in a pair
    (16, torch.bfloat16, 1, [1, 0, 1, 0, 1]),      # one draft: the odd tail alone
    (64, torch.bfloat16, 2, [1, 2, 0, 2, 1]),
    (128, torch.bfloat16, 1, [1, 0, 1, 0, 1]),     # the odd tail alone, columns split over two CTAs
    (128, torch.bfloat16, 4, [2, 2, 4, 0, 1]),     # the benchmark's draft count
    (32, torch.float32, 3, [3, 0, 2, 1, 3]),       # one CTA per (sequence, head)
])
def test_verify_outputs_and_rollback_state(kda, d, dtype, K, accept):
    """K drafts per sequence from a read-only state: all outputs, and the
    state after the accepted prefix (0, some, or all drafts)."""
    N, H = 5, 3
    inp = synth.custom(N * K, H, d, dtype, seed=840 + d, lengths=[K] * N, init_std=0.1)
    dv = to_device(inp)
    s_in = dv["init_state"].clone()
    out, s_out = kda.kda_decode_verify(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], s_in,
                                       accept, K)
    assert torch.equal(s_in, dv["init_state"])                      # read-only
    f = lambda t: f64(t)
    ref_out, _ = oracle.recurrence(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["g"]),
                                   f(inp["beta"]), f(inp["init_state"]), inp["cu_seqlens"])
    compare(out, ref_out, dtype, f"verify outputs d={d}")
    rows = np.concatenate([np.arange(n * K, n * K + a) for n, a in enumerate(accept)])
    cu = np.concatenate([[0], np.cumsum(accept)])
    sel = lambda t: f(t)[rows]
    _, ref_fin = oracle.recurrence(sel(inp["q"]), sel(inp["k"]), sel(inp["v"]), sel(inp["g"]),
                                   sel(inp["beta"]), f(inp["init_state"]), cu)
    compare(s_out, ref_fin, dtype, f"verify rollback state d={d}")
    for n, a in enumerate(accept):
        if a == 0:
            assert torch.equal(s_out[n], s_in[n])                   # nothing accepted


@pytest.mark.parametrize("d,dtype,weighted", [(128, torch.bfloat16, True),
                                              (128, torch.bfloat16, False),
                                              (64, torch.bfloat16, True),
                                              (32, torch.bfloat16, False),
                                              (64, torch.float32, False),
                                              (128, torch.float32, True),
                                              (16, torch.bfloat16, True)])
def test_output_gate_matches_oracle(kda, d, dtype, weighted):
    T, H = 77, 3
    gen = torch.Generator().manual_seed(860 + d)
    o = torch.randn(T, H, d, generator=gen).to(dtype)
    z = (2 * torch.randn(T, H, d, generator=gen)).to(dtype)
    w = torch.rand(d, generator=gen) + 0.5 if weighted else None
    y = kda.kda_output_gate(o.cuda(), z.cuda(), None if w is None else w.cuda())
    ref = oracle.output_gate(f64(o), f64(z), None if w is None else f64(w))
    compare(y, ref, dtype, f"output gate d={d}")
    # in place
    oc = o.cuda()
    kda.kda_output_gate(oc, z.cuda(), None if w is None else w.cuda(), out=oc)
    compare(oc, ref, dtype, f"output gate in place d={d}")


def test_output_gate_grid_stride_with_ragged_tail(kda):
    """More rows than one pass of the capped grid covers (152 SMs x 32 blocks x
    16 rows = 77,824), with a row count that ends mid-warp: every row written
    once, none past the end."""
    T, H, d = 1013, 97, 128                     # 98,261 rows
    gen = torch.Generator().manual_seed(871)
    o = torch.randn(T, H, d, generator=gen).to(torch.bfloat16)
    z = (2 * torch.randn(T, H, d, generator=gen)).to(torch.bfloat16)
    w = torch.rand(d, generator=gen) + 0.5
    y = torch.full((T + 1, H, d), 7.0, dtype=torch.bfloat16, device="cuda")
    kda.kda_output_gate(o.cuda(), z.cuda(), w.cuda(), out=y[:T])
    ref = oracle.output_gate(f64(o), f64(z), f64(w))
    compare(y[:T], ref, torch.bfloat16, "output gate, grid-stride rows")
    assert torch.all(y[T] == 7.0)               # the row after the end is untouched


def test_binding_rejects_wrong_output_buffers(kda):
    """A caller-supplied output of the wrong shape or dtype is refused before
    any launch (a kernel would otherwise write past its end)."""
    T, H, d, K = 8, 2, 128, 4
    c = lambda *s, dt=torch.float32: torch.zeros(*s, dtype=dt, device="cuda")
    o, z = c(T, H, d, dt=torch.bfloat16), c(T, H, d, dt=torch.bfloat16)
    with pytest.raises(ValueError):
        kda.kda_output_gate(o, z, out=c(T - 1, H, d, dt=torch.bfloat16))
    with pytest.raises(TypeError):
        kda.kda_output_gate(o, z, out=c(T, H, d))
    q = c(2 * K, H, d, dt=torch.bfloat16)
    g, b = c(2 * K, H, d), c(2 * K, H)
    s_in = c(2, H, d, d)
    acc = torch.tensor([1, 2], dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        kda.kda_decode_verify(q, q, q, g, b, s_in, acc, K, out=c(K, H, d, dt=torch.bfloat16))
    with pytest.raises(ValueError):
        kda.kda_decode_verify(q, q, q, g, b, s_in, acc, K, state_out=c(1, H, d, d))
    raw = c(T, H, d, dt=torch.bfloat16)
    w = c(3, H * d, 4)
    zg, zb = c(T, H, d), c(T, H)
    good = lambda: [torch.empty_like(raw) for _ in range(3)] + [c(T, H, d), c(T, H)]
    bad_v = good()
    bad_v[2] = c(T, H, d - 1, dt=torch.bfloat16)
    with pytest.raises(ValueError):
        kda.kda_prologue(raw, raw, raw, w, zg, zb, outs=tuple(bad_v))
    no_g = good()
    no_g[3] = None
    with pytest.raises(ValueError):
        kda.kda_prologue(raw, raw, raw, w, zg, zb, outs=tuple(no_g))
    # gate outputs are not needed without their logits
    q2, k2, v2, g2, b2 = kda.kda_prologue(raw, raw, raw, w, None, None,
                                          outs=tuple(good()[:3]) + (None, None))
    assert g2 is None and b2 is None
