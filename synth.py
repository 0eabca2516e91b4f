"""Seeded synthetic inputs for the KDA workloads.

This module only draws random numbers with the shapes and distributions of
the five KDA workloads below; it computes nothing of the operator itself.
The CUDA tests, the benchmark and the oracle tests all take their inputs from
here, so both sides of every parity check see the same bytes.

Every large tensor is drawn head by head from its own numpy stream
``default_rng([seed, tensor_id, head])`` (PCG64: identical on x86 and Arm),
so one head of a 262,144-token input can be regenerated alone for the oracle
without drawing the other 95.

Workloads (all H = 96 heads, d_k = d_v = 128 unless stated):
  1 tiny     : N=1, T=64, H=2, d=16, fp32; q,k ~ N(0,1) then scaled to unit
               length per head; v ~ N(0,1); g = -5*sigmoid(N(0,1)) per channel;
               beta = sigmoid(N(0,1)) per head; zero initial state.  seed 0
  2 prefill  : one sequence, T=4096, bf16 q,k,v (q,k unit length), fp32 g and
               beta as above, fp32 zero initial state.                 seed 1
  3 varlen   : 8 packed documents, lengths uniform in [512, 8192], inputs as
               in workload 2, initial state per document ~ 0.01*N(0,1). seed 2
  4 long     : one sequence, T=262,144, RAW bf16 q,k,v ~ N(0,1) for the fused
               prologue, depthwise conv weights ~ 0.5*N(0,1) [3, H*d, 4],
               gate logits z_g, z_beta ~ N(0,1) fp32.                  seed 3
  5 decode   : 256 sequences x one token, fp32 state ~ 0.01*N(0,1)
               [256, H, 128, 128], bf16 q,k,v (q,k unit length), g, beta as
               in workload 2.                                          seed 4

"N(0, s)" in the workload text is read as standard deviation s.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

# stream ids, one per tensor kind
Q, K, V, ZG, ZB, S0, CONV, LENS, UNIT_S0 = 1, 2, 3, 4, 5, 6, 7, 8, 9

GMIN = -5.0


@dataclass
class Workload:
    index: int
    name: str
    H: int
    d: int
    dtype: torch.dtype
    seed: int
    T: int = 0
    n_docs: int = 1
    init_std: float = 0.0          # 0 -> zero initial state
    raw: bool = False              # True -> raw inputs for the fused prologue
    decode: bool = False           # True -> one token per sequence
    lengths: list = field(default_factory=list)


def _workloads():
    w = {
        1: Workload(1, "tiny: N=1 T=64 H=2 d=16 fp32", 2, 16, torch.float32, 0, T=64),
        2: Workload(2, "prefill: N=1 T=4096 H=96 d=128 bf16", 96, 128,
                    torch.bfloat16, 1, T=4096),
        3: Workload(3, "varlen: 8 docs of 512..8192 tokens, H=96 d=128 bf16", 96,
                    128, torch.bfloat16, 2, n_docs=8, init_std=0.01),
        4: Workload(4, "long context: N=1 T=262144 H=96 d=128 bf16, fused prologue",
                    96, 128, torch.bfloat16, 3, T=262144, raw=True),
        5: Workload(5, "decode: 256 sequences x 1 token, H=96 d=128, fp32 state",
                    96, 128, torch.bfloat16, 4, T=256, n_docs=256, init_std=0.01,
                    decode=True),
    }
    rng = np.random.default_rng([w[3].seed, LENS])
    w[3].lengths = [int(x) for x in rng.integers(512, 8193, size=8)]
    w[3].T = sum(w[3].lengths)
    w[1].lengths, w[2].lengths, w[4].lengths = [64], [4096], [262144]
    w[5].lengths = [1] * 256
    return w


WORKLOADS = _workloads()


def cu_seqlens_of(lengths) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return cu


# ---------------------------------------------------------------- drawing

def _stream(seed, tensor_id, head):
    return np.random.default_rng([seed, tensor_id, head])


def _normal(seed, tensor_id, head, shape):
    return _stream(seed, tensor_id, head).standard_normal(shape, dtype=np.float32)


def _unit(x):
    # uniform direction on the sphere: a Gaussian draw scaled to length one
    return x / np.linalg.norm(x.astype(np.float64), axis=-1, keepdims=True)


def _log_decay(z):
    # the workloads state g ~ gmin * sigmoid(N(0,1)); drawn here in fp64
    return GMIN / (1.0 + np.exp(-z.astype(np.float64)))


def _logistic(z):
    return 1.0 / (1.0 + np.exp(-z.astype(np.float64)))


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 4))
    return _POOL


def _heads_tensor(H, heads, draw, dtype, device=None):
    """Tensor [rows..., len(heads), cols]; head slot i holds draw(heads[i]).

    draw(h) returns a numpy array [rows..., cols] for head h.  Heads are drawn
    on a thread pool (numpy releases the GIL while it fills arrays).  With a
    CUDA `device` the result is allocated there and filled head by head, so
    host memory holds only a pool's worth of heads at a time.
    """
    heads = list(range(H)) if heads is None else list(heads)
    first = torch.from_numpy(np.ascontiguousarray(draw(heads[0]))).to(dtype)
    out = torch.empty(tuple(first.shape[:-1]) + (len(heads), first.shape[-1]),
                      dtype=dtype, device=device)
    out.select(-2, 0).copy_(first)
    rest = list(enumerate(heads))[1:]

    def one(ix_h):
        ix, h = ix_h
        a = torch.from_numpy(np.ascontiguousarray(draw(h))).to(dtype)
        if device is None:
            out.select(-2, ix).copy_(a)
            return None
        return ix, a

    if device is None:
        list(_pool().map(one, rest))
    else:
        step = _pool()._max_workers
        for b in range(0, len(rest), step):
            for ix, a in _pool().map(one, rest[b:b + step]):
                out.select(-2, ix).copy_(a)
    return out


def inputs(index: int, heads=None, device=None) -> dict:
    """Inputs of workload `index` as torch CPU tensors.

    heads: optional list of head indices; the result then holds only those
    heads, bit-identical to the same heads of the full draw.
    device: None for CPU tensors, or a CUDA device to fill directly.
    Keys: q,k,v [T,H,d]; g [T,H,d] fp32; beta [T,H] fp32; init_state
    [N,H,d,d] fp32 or None; cu_seqlens int64 numpy [N+1];
    raw workloads give q_raw,k_raw,v_raw, conv_w [3,Hs*d,4], z_g, z_beta.
    """
    w = WORKLOADS[index]
    T, H, d, s = w.T, w.H, w.d, w.seed
    hs = list(range(H)) if heads is None else list(heads)
    res = {"workload": w, "heads": hs, "cu_seqlens": cu_seqlens_of(w.lengths)}
    if w.raw:
        for name, sid in (("q_raw", Q), ("k_raw", K), ("v_raw", V)):
            res[name] = _heads_tensor(H, hs, lambda h, sid=sid:
                                      _normal(s, sid, h, (T, d)), w.dtype, device)
        res["z_g"] = _heads_tensor(H, hs, lambda h: _normal(s, ZG, h, (T, d)),
                                   torch.float32, device)
        res["z_beta"] = _heads_tensor(H, hs, lambda h: _normal(s, ZB, h, (T, 1)),
                                      torch.float32, device)[..., 0]
        conv = torch.stack([
            _heads_tensor(H, hs, lambda h, i=i:
                          (0.5 * _normal(s, CONV * 16 + i, h, (4, d))), torch.float32, device)
            for i in range(3)])                       # [3, 4, Hs, d]
        res["conv_w"] = conv.permute(0, 2, 3, 1).reshape(3, len(hs) * d, 4).contiguous()
        res["init_state"] = None
        return res
    res["q"] = _heads_tensor(H, hs, lambda h: _unit(_normal(s, Q, h, (T, d))),
                             w.dtype, device)
    res["k"] = _heads_tensor(H, hs, lambda h: _unit(_normal(s, K, h, (T, d))),
                             w.dtype, device)
    res["v"] = _heads_tensor(H, hs, lambda h: _normal(s, V, h, (T, d)), w.dtype, device)
    res["g"] = _heads_tensor(H, hs, lambda h: _log_decay(_normal(s, ZG, h, (T, d))),
                             torch.float32, device)
    res["beta"] = _heads_tensor(H, hs, lambda h: _logistic(_normal(s, ZB, h, (T, 1))),
                                torch.float32, device)[..., 0].contiguous()
    N = len(w.lengths)
    if w.init_std > 0:
        st = _heads_tensor(H, hs, lambda h: (w.init_std * _normal(
            s, S0, h, (N, d * d))), torch.float32, device)        # [N, Hs, d*d]
        res["init_state"] = st.reshape(N, len(hs), d, d).contiguous()
    else:
        res["init_state"] = None
    return res


def custom(T, H, d, dtype=torch.float32, seed=100, lengths=None, init_std=0.0,
           unit_qk=True, g_scale=1.0, g_const=None):
    """Small ad-hoc inputs with the workload distributions (edge-case tests);
    g_scale < 1 draws a weaker decay, g = g_scale * gmin * sigmoid(N(0,1));
    g_const fills every g with one value instead (a degenerate case)."""
    lengths = [T] if lengths is None else list(lengths)
    assert sum(lengths) == T
    res = {"cu_seqlens": cu_seqlens_of(lengths)}
    qd = (lambda x: _unit(x)) if unit_qk else (lambda x: x)
    res["q"] = _heads_tensor(H, None, lambda h: qd(_normal(seed, Q, h, (T, d))), dtype)
    res["k"] = _heads_tensor(H, None, lambda h: qd(_normal(seed, K, h, (T, d))), dtype)
    res["v"] = _heads_tensor(H, None, lambda h: _normal(seed, V, h, (T, d)), dtype)
    res["g"] = _heads_tensor(H, None,
                             lambda h: g_scale * _log_decay(_normal(seed, ZG, h, (T, d)))
                             if g_const is None else np.full((T, d), g_const),
                             torch.float32)
    res["beta"] = _heads_tensor(H, None, lambda h: _logistic(_normal(seed, ZB, h, (T, 1))),
                                torch.float32)[..., 0].contiguous()
    N = len(lengths)
    if init_std > 0:
        st = _heads_tensor(H, None, lambda h: init_std * _normal(seed, S0, h, (N, d * d)),
                           torch.float32)
        res["init_state"] = st.reshape(N, H, d, d).contiguous()
    else:
        res["init_state"] = None
    return res


def custom_raw(T, H, d, dtype=torch.bfloat16, seed=200, lengths=None, conv_std=0.5):
    """Raw prologue inputs with the long-context distributions."""
    lengths = [T] if lengths is None else list(lengths)
    assert sum(lengths) == T
    res = {"cu_seqlens": cu_seqlens_of(lengths)}
    for name, sid in (("q_raw", Q), ("k_raw", K), ("v_raw", V)):
        res[name] = _heads_tensor(H, None, lambda h, sid=sid:
                                  _normal(seed, sid, h, (T, d)), dtype)
    res["z_g"] = _heads_tensor(H, None, lambda h: _normal(seed, ZG, h, (T, d)),
                               torch.float32)
    res["z_beta"] = _heads_tensor(H, None, lambda h: _normal(seed, ZB, h, (T, 1)),
                                  torch.float32)[..., 0].contiguous()
    conv = torch.stack([
        _heads_tensor(H, None, lambda h, i=i: conv_std * _normal(seed, CONV * 16 + i, h, (4, d)),
                      torch.float32) for i in range(3)])
    res["conv_w"] = conv.permute(0, 2, 3, 1).reshape(3, H * d, 4).contiguous()
    return res


def state_units(units, d, std=0.01, seed=300) -> np.ndarray:
    """States [len(units), d, d] fp32 ~ std * N(0,1), one stream per unit id
    (sequence * H + head): for tests that fill a large state on the device
    and compare only sampled units, which are then written from here."""
    return np.stack([std * _normal(seed, UNIT_S0, int(u), (d, d)) for u in units])


def lengths_many(n_docs, seed=400, long_docs=()) -> list:
    """Document lengths for the many-documents edge case: mostly 0-3 tokens,
    one in ten 4-64 tokens; `long_docs` maps doc index -> forced length."""
    rng = np.random.default_rng([seed, LENS])
    short = rng.integers(0, 4, size=n_docs)
    mid = rng.integers(4, 65, size=n_docs)
    lengths = np.where(rng.random(n_docs) < 0.1, mid, short)
    for i, n in dict(long_docs).items():
        lengths[i] = n
    return [int(x) for x in lengths]
