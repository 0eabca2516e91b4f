"""Shared helpers of the GPU parity tests: run the CUDA path through the
binding, run the fp64 oracle on the same inputs, compare.

Tolerances (written here once, used by every parity test):
  * fp32 inputs: max |gpu - oracle| <= 1e-4 (absolute), outputs and states.
  * bf16 inputs, fp32 state ("2e-2 relative to output RMS"):
      - RMS(gpu - oracle) <= 2e-2 * RMS(oracle), for outputs and states;
      - every element of an fp32 result (the final states, the gates):
        |gpu - oracle| <= 2e-2 * RMS(oracle);
      - every element of a bf16 result (the outputs):
        |gpu - oracle| <= 2e-2 * RMS(oracle) + half a bf16 ulp of the oracle
        value, the rounding that storing it in bf16 costs by itself (the
        largest outputs reach ~12x the RMS, where that half ulp is ~0.02 x RMS).
"""
import numpy as np
import torch

import oracle

TOL_F32_ABS = 1e-4
TOL_BF16_REL_RMS = 2e-2


def f64(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu").to(torch.float64).numpy()


def rms(x):
    return float(np.sqrt(np.mean(np.square(x)))) if x.size else 0.0


def half_ulp_bf16(x):
    """Half the spacing of bf16 numbers at |x| (bf16 keeps 8 significant bits)."""
    _, e = np.frexp(np.abs(x))          # |x| = m 2^e with m in [0.5, 1)
    return np.where(x == 0, 0.0, np.ldexp(1.0, e - 9))


LAST = {}   # the last comparison's relative errors, by label (printed with -s)


def compare(got, ref, dtype, what):
    """Assert parity under the tolerance of `dtype`; return (rel_rms, max_rel).

    `got` is the GPU result as it was stored (a bf16 tensor is an output that
    was rounded to bf16 once); `ref` the fp64 oracle value."""
    rounded = isinstance(got, torch.Tensor) and got.dtype == torch.bfloat16
    got, ref = f64(got), f64(ref)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    if not ref.size:
        return 0.0, 0.0
    diff = np.abs(got - ref)
    err = float(diff.max())
    if dtype == torch.float32:
        bound = TOL_F32_ABS
        assert err <= bound, f"{what}: max|err| = {err:.3e} > {bound:.3e}"
        return err, bound
    r = max(rms(ref), 1e-30)
    rel = rms(diff) / r
    LAST[what] = (rel, err / r)
    assert rel <= TOL_BF16_REL_RMS, \
        f"{what}: RMS(err)/RMS(ref) = {rel:.3e} > {TOL_BF16_REL_RMS:.0e}"
    bound = TOL_BF16_REL_RMS * r + (half_ulp_bf16(ref) if rounded else 0.0)
    over = diff > bound
    if over.any():
        i = np.unravel_index(int(np.argmax(diff - bound)), diff.shape)
        raise AssertionError(
            f"{what}: {int(over.sum())} elements above the element bound; worst at {i}: "
            f"|err| = {diff[i]:.3e}, bound {np.broadcast_to(bound, diff.shape)[i]:.3e} "
            f"(2e-2 RMS = {TOL_BF16_REL_RMS * r:.3e}{', + half a bf16 ulp' if rounded else ''})")
    # the share of the 2e-2 RMS budget the worst element uses, beyond its own rounding
    used = float(np.max(diff - (half_ulp_bf16(ref) if rounded else 0.0))) / r
    print(f"[parity] {what}: rel RMS {rel:.2e}, max|err|/RMS {err / r:.2e}, "
          f"max(|err| - rounding)/RMS {used:.2e} (bound 2e-2)")
    return rel, err / r


def as_stored(x, dtype):
    """Round fp64 values to the dtype they are stored in between two operators:
    the prologue's q, k, v are tensors of the workload's qkv dtype, its gates
    fp32, and the prefill consumes exactly those values."""
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(dtype).to(torch.float64).numpy()


def oracle_prologue_stored(prologue_out, dtype):
    """oracle.prologue's (q, k, v, g, beta) as the prefill receives them: q, k, v
    in `dtype`, g and beta in fp32 (None stays None)."""
    q, k, v, g, b = prologue_out
    r = lambda x, dt: None if x is None else as_stored(x, dt)
    return r(q, dtype), r(k, dtype), r(v, dtype), r(g, torch.float32), r(b, torch.float32)


def oracle_prefill(inp, heads=None, threads=0):
    """Oracle outputs for the (optionally sub-selected) heads of `inp`."""
    sel = (lambda t: t) if heads is None else (lambda t: t[:, heads])
    s0 = inp.get("init_state")
    if s0 is not None and heads is not None:
        s0 = s0[:, heads]
    return oracle.recurrence(f64(sel(inp["q"])), f64(sel(inp["k"])), f64(sel(inp["v"])),
                             f64(sel(inp["g"])), f64(sel(inp["beta"])), f64(s0),
                             inp["cu_seqlens"], threads=threads)


def to_device(inp, device="cuda"):
    out = {}
    for key, val in inp.items():
        out[key] = val.to(device) if isinstance(val, torch.Tensor) else val
    return out


def gpu_prefill(kda, dinp, **kw):
    cu = torch.as_tensor(dinp["cu_seqlens"], dtype=torch.int32, device=dinp["q"].device)
    return kda.kda_prefill(dinp["q"], dinp["k"], dinp["v"], dinp["g"], dinp["beta"],
                           dinp.get("init_state"), cu, **kw)
