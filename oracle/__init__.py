"""fp64 CPU oracle for the KDA operator -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports, links or runs anything here, and nothing here
imports the product: the two share no code.

The arithmetic lives in ``kda_oracle.c`` (plain C, double precision, written
as the definitions on the pages).  This module only builds that file with the
host C compiler, loads it with ctypes and marshals numpy arrays.

Sources, by page title and section:
  * "From GPT-2 to Kimi K3, from first principles", Chapter 5 (KDA recurrence,
    lower-bounded decay) and Chapter 6 (read after the update).
  * "Kimi K3 Architecture Explained", "Step 3: Forgetting, Channel by Channel"
    and "Inside a KDA Layer".
  * "An infra-oriented diagram of Kimi K3", "Kimi Delta Attention: fixed-state
    sequence mixing" (ShortConv width 4, Swish, L2Norm, gates; packed tokens).

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
closed forms, special cases, exact rational arithmetic and library routines;
none is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

GMIN = -5.0        # lower bound of the log-decay (Chapter 5, K3's bounded gate)
RMS_EPS = 1e-6     # reading: the pages give no epsilon for the head RMSNorm
CONV_WIDTH = 4     # ShortConv kernel size (infra diagram, KDA card)
L2_EPS = 1e-6      # reading: the pages give no epsilon for the L2 norm


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``libkda_oracle.so`` next to it."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC",
           "-shared", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.kda_oracle_recurrence.argtypes = [P, P, P, P, P, P, P, i32, i64,
                                                  i32, i32, i32, P, P, i32]
            lib.kda_oracle_short_conv.argtypes = [P, P, P, i32, i64, i32, i32,
                                                  P, i32]
            lib.kda_oracle_swish.argtypes = [P, i64]
            lib.kda_oracle_l2norm.argtypes = [P, i64, i32, f64]
            lib.kda_oracle_decay_gate.argtypes = [P, i64, f64, P]
            lib.kda_oracle_sigmoid.argtypes = [P, i64, P]
            lib.kda_oracle_output_gate.argtypes = [P, P, P, i64, i32, f64, P]
            for fn in (lib.kda_oracle_recurrence, lib.kda_oracle_short_conv,
                       lib.kda_oracle_swish, lib.kda_oracle_l2norm,
                       lib.kda_oracle_decay_gate, lib.kda_oracle_sigmoid,
                       lib.kda_oracle_output_gate):
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _offsets(cu_seqlens, T: int) -> np.ndarray:
    if cu_seqlens is None:
        return np.array([0, T], dtype=np.int64)
    return np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


def recurrence(q, k, v, g, beta, init_state=None, cu_seqlens=None,
               threads: int = 0):
    """Token-by-token KDA recurrence in fp64.

    q, k, g: [T, H, dk]; v: [T, H, dv]; beta: [T, H];
    init_state: [N, H, dk, dv] or None (zeros); cu_seqlens: [N+1] or None.
    Returns (out [T, H, dv], final_state [N, H, dk, dv]).
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    T, H, dk = q.shape
    dv = v.shape[2]
    if k.shape != (T, H, dk) or g.shape != (T, H, dk) or v.shape[:2] != (T, H) \
            or beta.shape != (T, H):
        raise ValueError("inconsistent shapes")
    cu = _offsets(cu_seqlens, T)
    N = cu.shape[0] - 1
    s0 = None
    if init_state is not None:
        s0 = _f64(init_state)
        if s0.shape != (N, H, dk, dv):
            raise ValueError("init_state must be [N, H, dk, dv]")
    out = np.zeros((T, H, dv), dtype=np.float64)
    fin = np.zeros((N, H, dk, dv), dtype=np.float64)
    rc = _load().kda_oracle_recurrence(_ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                       _ptr(beta), _ptr(s0), _ptr(cu), N, T, H,
                                       dk, dv, _ptr(out), _ptr(fin), threads)
    _check(rc, "recurrence")
    return out, fin


def short_conv(x, w, cu_seqlens=None, threads: int = 0):
    """Depthwise causal conv; x: [T, C], w: [C, W] (tap W-1 = current token)."""
    x, w = _f64(x), _f64(w)
    T, C = x.shape
    W = w.shape[1]
    cu = _offsets(cu_seqlens, T)
    y = np.zeros_like(x)
    rc = _load().kda_oracle_short_conv(_ptr(x), _ptr(w), _ptr(cu),
                                       cu.shape[0] - 1, T, C, W, _ptr(y),
                                       threads)
    _check(rc, "short_conv")
    return y


def swish(x):
    y = _f64(x).copy()
    _check(_load().kda_oracle_swish(_ptr(y), y.size), "swish")
    return y


def l2norm(x, eps: float = L2_EPS):
    """Normalise the last axis of x to unit length (sqrt(sum x^2 + eps))."""
    y = _f64(x).copy()
    d = y.shape[-1]
    _check(_load().kda_oracle_l2norm(_ptr(y), y.size // d, d, eps), "l2norm")
    return y


def decay_gate(z, gmin: float = GMIN):
    z = _f64(z)
    g = np.zeros_like(z)
    _check(_load().kda_oracle_decay_gate(_ptr(z), z.size, gmin, _ptr(g)),
           "decay_gate")
    return g


def sigmoid(z):
    z = _f64(z)
    b = np.zeros_like(z)
    _check(_load().kda_oracle_sigmoid(_ptr(z), z.size, _ptr(b)), "sigmoid")
    return b


def prologue(q_raw, k_raw, v_raw, conv_w, z_g=None, z_beta=None,
             cu_seqlens=None, eps: float = L2_EPS, gmin: float = GMIN,
             threads: int = 0):
    """The KDA input path of the infra diagram's KDA card, in fp64.

    q_raw, k_raw, v_raw: [T, H, d]; conv_w: [3, H*d, 4] (q, k, v filters).
    Each of q, k, v: ShortConv -> Swish; q and k then L2Norm per head.
    Gates: g = gmin * sigmoid(z_g) [T, H, d], beta = sigmoid(z_beta) [T, H].
    Returns (q, k, v, g, beta); g / beta are None when their logits are None.
    """
    raws = [_f64(x) for x in (q_raw, k_raw, v_raw)]
    T, H, d = raws[0].shape
    conv_w = _f64(conv_w)
    if conv_w.shape != (3, H * d, CONV_WIDTH):
        raise ValueError("conv_w must be [3, H*d, 4]")
    outs = []
    for i, x in enumerate(raws):
        y = short_conv(x.reshape(T, H * d), conv_w[i], cu_seqlens, threads)
        y = swish(y).reshape(T, H, d)
        if i < 2:
            y = l2norm(y, eps)
        outs.append(y)
    g = None if z_g is None else decay_gate(z_g, gmin)
    beta = None if z_beta is None else sigmoid(z_beta)
    return outs[0], outs[1], outs[2], g, beta


def output_gate(o, z, w=None, eps: float = RMS_EPS):
    """Head RMSNorm times sigmoid(gate): o, z [..., d]; w [d] or None."""
    o, z = _f64(o), _f64(z)
    d = o.shape[-1]
    ww = None if w is None else _f64(w)
    y = np.zeros_like(o)
    _check(_load().kda_oracle_output_gate(_ptr(o), _ptr(z), _ptr(ww), o.size // d, d, eps,
                                          _ptr(y)), "output_gate")
    return y
