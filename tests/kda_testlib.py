"""Shared helpers of the GPU parity tests: run the CUDA path through the
binding, run the fp64 oracle on the same inputs, compare.

Tolerances (written here once, used by every parity test):
  * fp32 inputs: max |gpu - oracle| <= 1e-4 (absolute), outputs and states.
  * bf16 inputs, fp32 state: max |gpu - oracle| <= 2e-2 * RMS(oracle),
    separately for the outputs and for the final states.  The reading is
    the stricter one of "2e-2 relative to output RMS": a max-abs error, not
    an RMS error, is held to the bound.
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


def compare(got, ref, dtype, what):
    """Assert parity under the tolerance of `dtype`; return (max_err, bound)."""
    got, ref = f64(got), f64(ref)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    if dtype == torch.float32:
        bound = TOL_F32_ABS
    else:
        bound = TOL_BF16_REL_RMS * rms(ref)
    assert err <= bound, f"{what}: max|err| = {err:.3e} > {bound:.3e} (rms ref {rms(ref):.3e})"
    return err, bound


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
