"""Python binding of libkda.so (include/kda.h): argument marshalling only.

Every step of the operator runs in the CUDA library; this module checks
tensor shapes, allocates outputs with torch when the caller gives none, and
passes raw device pointers and the current torch stream through ctypes.
Importing it raises if the library has not been built -- there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkda.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with "
                      "`python -m linear_attention_03_gb300.build` (needs nvcc)")

lib = ctypes.CDLL(_LIB_PATH)

KDA_OK, KDA_ERR_INVALID, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT, \
    KDA_ERR_DEVICE = range(6)
KDA_F32, KDA_BF16 = 0, 1
KDA_DEVICE_OK, KDA_DEVICE_BAD_OFFSETS, KDA_DEVICE_TIMEOUT, KDA_DEVICE_RANGE, \
    KDA_DEVICE_BAD_SNAPSHOT = range(5)
KDA_SNAPSHOT_ALIGN = 64
SYMBOLS = ("kda_prefill_workspace_size", "kda_prefill", "kda_decode_step",
           "kda_prologue", "kda_get_device_status", "kda_last_error",
           "kda_kernel_launches", "kda_decode_step_conv", "kda_decode_verify",
           "kda_output_gate", "kda_prefill_noalloc", "kda_selftest_wait",
           "kda_prefill_segmented_workspace_size", "kda_prefill_segmented",
           "kda_prologue_prefill_workspace_size", "kda_prologue_prefill",
           "kda_prefill_snapshots")


class kda_dims(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("qkv_dtype", ctypes.c_int32)]


_P, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
lib.kda_prefill_workspace_size.argtypes = [kda_dims, _i64, _i32]
lib.kda_prefill_workspace_size.restype = _sz
lib.kda_prefill.argtypes = [_P, _P, _P, _P, _P, _P, _P, _i32, _i64, kda_dims, _P, _P, _P,
                            _sz, _P]
lib.kda_prefill_snapshots.argtypes = [_P, _P, _P, _P, _P, _P, _P, _i32, _i64, kda_dims, _P, _P,
                                      _P, _i32, _P, _P, _sz, _P]
lib.kda_prefill_segmented_workspace_size.argtypes = [kda_dims, _i64, _i32]
lib.kda_prefill_segmented_workspace_size.restype = _sz
lib.kda_prefill_segmented.argtypes = [_P, _P, _P, _P, _P, _P, _i64, kda_dims, _i32, _P, _P, _P,
                                      _sz, _P]
lib.kda_prologue_prefill_workspace_size.argtypes = [kda_dims, _i64, _i64]
lib.kda_prologue_prefill_workspace_size.restype = _sz
lib.kda_prologue_prefill.argtypes = [_P, _P, _P, _P, _P, _P, _P, _i64, kda_dims, _i64, _P, _P, _P,
                                     _sz, _P, _P]
lib.kda_decode_step.argtypes = [_P, _P, _P, _P, _P, _P, _P, _i32, kda_dims, _P]
lib.kda_prologue.argtypes = [_P, _P, _P, _P, _P, _P, _P, _i32, _i64, kda_dims, _P, _P, _P,
                             _P, _P, _P]
lib.kda_get_device_status.argtypes = [_P, ctypes.POINTER(ctypes.c_int32), _P]
lib.kda_decode_step_conv.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _i32, kda_dims, _P]
lib.kda_decode_verify.argtypes = [_P, _P, _P, _P, _P, _P, _P, _i32, _i32, kda_dims, _P, _P, _P]
lib.kda_output_gate.argtypes = [_P, _P, _P, _i64, kda_dims, ctypes.c_float, _P, _P]
lib.kda_selftest_wait.argtypes = [_i64, _P, _sz, _P]
lib.kda_selftest_wait.restype = ctypes.c_int
lib.kda_last_error.argtypes = []
lib.kda_last_error.restype = ctypes.c_char_p
lib.kda_kernel_launches.argtypes = []
lib.kda_kernel_launches.restype = ctypes.c_uint64
for _fn in (lib.kda_prefill, lib.kda_prefill_snapshots, lib.kda_prefill_segmented,
            lib.kda_prologue_prefill,
            lib.kda_decode_step, lib.kda_prologue,
            lib.kda_get_device_status,
            lib.kda_decode_step_conv, lib.kda_decode_verify, lib.kda_output_gate):
    _fn.restype = ctypes.c_int


class KDAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where} failed with status {status}: "
                         f"{lib.kda_last_error().decode(errors='replace')}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def _dev(t, name, dtype=None, shape=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _offsets(cu_seqlens, T, device):
    if cu_seqlens is None:
        return None, 1
    if isinstance(cu_seqlens, torch.Tensor) and cu_seqlens.is_cuda:
        cu = _dev(cu_seqlens, "cu_seqlens", torch.int32)
    else:
        cu = torch.as_tensor(cu_seqlens, dtype=torch.int32).to(device)
    return cu, cu.numel() - 1


def dims_of(q: torch.Tensor) -> kda_dims:
    _, H, d = q.shape
    return kda_dims(H, d, d, _dtype_code(q))


def kda_prefill_workspace_size(H: int, d: int, dtype: torch.dtype, T: int, N: int) -> int:
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    return int(lib.kda_prefill_workspace_size(kda_dims(H, d, d, code), T, N))


def kda_prefill(q, k, v, g, beta, init_state=None, cu_seqlens=None, out=None,
                final_state=None, workspace=None, want_final_state=True):
    """Chunked prefill over packed documents; returns (out, final_state).

    workspace: uint8 device tensor, by default kda_prefill_workspace_size
    bytes (the status word, then the documents' longest-first order when
    there are several); 256 bytes also work and run the documents in order.
    """
    out, final_state, _ = _prefill(q, k, v, g, beta, init_state, cu_seqlens, out, final_state,
                                   workspace, want_final_state, None, None)
    return out, final_state


def kda_prefill_snapshots(q, k, v, g, beta, snapshot_offsets, init_state=None, cu_seqlens=None,
                          out=None, final_state=None, snapshots=None, workspace=None):
    """kda_prefill that also returns the states at `snapshot_offsets` (int32
    device tensor of strictly increasing packed-token offsets, each a multiple
    of KDA_SNAPSHOT_ALIGN tokens into its document or its end); returns
    (out, final_state, snapshots [n, H, d, d] fp32)."""
    return _prefill(q, k, v, g, beta, init_state, cu_seqlens, out, final_state, workspace, True,
                    snapshot_offsets, snapshots)


def _prefill(q, k, v, g, beta, init_state, cu_seqlens, out, final_state, workspace,
             want_final_state, snapshot_offsets, snapshots):
    T, H, d = q.shape
    dev = q.device
    _dev(q, "q")
    _dev(k, "k", q.dtype, q.shape)
    _dev(v, "v", q.dtype, q.shape)
    _dev(g, "g", torch.float32, q.shape)
    _dev(beta, "beta", torch.float32, (T, H))
    cu, N = _offsets(cu_seqlens, T, dev)
    _dev(init_state, "init_state", torch.float32, (N, H, d, d))
    if out is None:
        out = torch.empty_like(v)
    _dev(out, "out", q.dtype, q.shape)
    if final_state is None and want_final_state:
        final_state = torch.empty((N, H, d, d), dtype=torch.float32, device=dev)
    _dev(final_state, "final_state", torch.float32, (N, H, d, d))
    dims = dims_of(q)
    ws_bytes = int(lib.kda_prefill_workspace_size(dims, T, N))
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    _dev(workspace, "workspace", torch.uint8)
    if snapshot_offsets is None:
        st = lib.kda_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state),
                             _ptr(cu), N, T, dims, _ptr(out), _ptr(final_state),
                             _ptr(workspace), workspace.numel(), _stream())
        if st != KDA_OK:
            raise KDAError(st, "kda_prefill")
        return out, final_state, None
    _dev(snapshot_offsets, "snapshot_offsets", torch.int32)
    n_snap = snapshot_offsets.numel()
    if snapshots is None:
        snapshots = torch.empty((n_snap, H, d, d), dtype=torch.float32, device=dev)
    _dev(snapshots, "snapshots", torch.float32, (n_snap, H, d, d))
    st = lib.kda_prefill_snapshots(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                   _ptr(init_state), _ptr(cu), N, T, dims, _ptr(out),
                                   _ptr(final_state), _ptr(snapshot_offsets), n_snap,
                                   _ptr(snapshots), _ptr(workspace), workspace.numel(), _stream())
    if st != KDA_OK:
        raise KDAError(st, "kda_prefill_snapshots")
    return out, final_state, snapshots


def kda_prefill_segmented_workspace_size(H: int, d: int, dtype: torch.dtype, T: int,
                                         num_segments: int) -> int:
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    return int(lib.kda_prefill_segmented_workspace_size(kda_dims(H, d, d, code), T, num_segments))


def kda_prefill_segmented(q, k, v, g, beta, init_state=None, num_segments=2, out=None,
                          final_state=None, workspace=None):
    """One document as `num_segments` segments joined by an exact scan of their
    affine state maps; returns (out, final_state [H, d, d])."""
    T, H, d = q.shape
    dev = q.device
    _dev(q, "q")
    _dev(k, "k", q.dtype, q.shape)
    _dev(v, "v", q.dtype, q.shape)
    _dev(g, "g", torch.float32, q.shape)
    _dev(beta, "beta", torch.float32, (T, H))
    _dev(init_state, "init_state", torch.float32, (H, d, d))
    if out is None:
        out = torch.empty_like(v)
    _dev(out, "out", q.dtype, q.shape)
    if final_state is None:
        final_state = torch.empty((H, d, d), dtype=torch.float32, device=dev)
    _dev(final_state, "final_state", torch.float32, (H, d, d))
    dims = dims_of(q)
    ws_bytes = int(lib.kda_prefill_segmented_workspace_size(dims, T, num_segments))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _dev(workspace, "workspace", torch.uint8)
    st = lib.kda_prefill_segmented(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                   _ptr(init_state), T, dims, num_segments, _ptr(out),
                                   _ptr(final_state), _ptr(workspace), workspace.numel(), _stream())
    if st != KDA_OK:
        raise KDAError(st, "kda_prefill_segmented")
    return out, final_state


def kda_prologue_prefill_workspace_size(H: int, d: int, dtype: torch.dtype, T: int,
                                        segment_tokens: int) -> int:
    code = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    return int(lib.kda_prologue_prefill_workspace_size(kda_dims(H, d, d, code), T, segment_tokens))


_side_streams = {}


def _side_stream(dev):
    """This binding's stream for the prologues (one per device, lowest priority)."""
    key = torch.device(dev).index if torch.device(dev).index is not None else torch.cuda.current_device()
    if key not in _side_streams:
        _side_streams[key] = torch.cuda.Stream(device=key, priority=0)
    return _side_streams[key]


def kda_prologue_prefill(q_raw, k_raw, v_raw, conv_w, z_g, z_beta, init_state=None,
                         segment_tokens=16384, out=None, final_state=None, workspace=None,
                         prologue_stream=None):
    """Prologue + prefill of one document from raw projections, segment by
    segment with the next prologue overlapping the current prefill; returns
    (out, final_state [H, d, d]).  The prefills run on the current stream, the
    prologues on `prologue_stream` (a torch.cuda.Stream; by default one that
    this module keeps per device, at the lowest priority: run the call on a
    higher-priority current stream for the best overlap)."""
    T, H, d = q_raw.shape
    dev = q_raw.device
    _dev(q_raw, "q_raw")
    _dev(k_raw, "k_raw", q_raw.dtype, q_raw.shape)
    _dev(v_raw, "v_raw", q_raw.dtype, q_raw.shape)
    _dev(conv_w, "conv_w", torch.float32, (3, H * d, 4))
    _dev(z_g, "z_g", torch.float32, q_raw.shape)
    _dev(z_beta, "z_beta", torch.float32, (T, H))
    _dev(init_state, "init_state", torch.float32, (H, d, d))
    if out is None:
        out = torch.empty_like(v_raw)
    _dev(out, "out", q_raw.dtype, q_raw.shape)
    if final_state is None:
        final_state = torch.empty((H, d, d), dtype=torch.float32, device=dev)
    _dev(final_state, "final_state", torch.float32, (H, d, d))
    dims = dims_of(q_raw)
    ws_bytes = int(lib.kda_prologue_prefill_workspace_size(dims, T, segment_tokens))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    _dev(workspace, "workspace", torch.uint8)
    side = prologue_stream if prologue_stream is not None else _side_stream(dev)
    st = lib.kda_prologue_prefill(_ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(conv_w), _ptr(z_g),
                                  _ptr(z_beta), _ptr(init_state), T, dims, segment_tokens, _ptr(out),
                                  _ptr(final_state), _ptr(workspace), workspace.numel(), _stream(),
                                  ctypes.c_void_p(side.cuda_stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_prologue_prefill")
    return out, final_state


def kda_decode_step(q, k, v, g, beta, state, out=None):
    """One token per sequence; updates `state` in place and returns out."""
    N, H, d = q.shape
    _dev(q, "q")
    _dev(k, "k", q.dtype, q.shape)
    _dev(v, "v", q.dtype, q.shape)
    _dev(g, "g", torch.float32, q.shape)
    _dev(beta, "beta", torch.float32, (N, H))
    _dev(state, "state", torch.float32, (N, H, d, d))
    if out is None:
        out = torch.empty_like(v)
    _dev(out, "out", q.dtype, q.shape)
    st = lib.kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
                             _ptr(out), N, dims_of(q), _stream())
    if st != KDA_OK:
        raise KDAError(st, "kda_decode_step")
    return out


def kda_prologue(q_raw, k_raw, v_raw, conv_w, z_g=None, z_beta=None, cu_seqlens=None,
                 outs=None):
    """Fused ShortConv + Swish + L2Norm(q, k) and the two gates.

    Returns (q, k, v, g, beta); g / beta are None when their logits are None.
    """
    T, H, d = q_raw.shape
    dev = q_raw.device
    _dev(q_raw, "q_raw")
    _dev(k_raw, "k_raw", q_raw.dtype, q_raw.shape)
    _dev(v_raw, "v_raw", q_raw.dtype, q_raw.shape)
    _dev(conv_w, "conv_w", torch.float32, (3, H * d, 4))
    _dev(z_g, "z_g", torch.float32, q_raw.shape)
    _dev(z_beta, "z_beta", torch.float32, (T, H))
    cu, N = _offsets(cu_seqlens, T, dev)
    if outs is None:
        outs = (torch.empty_like(q_raw), torch.empty_like(q_raw), torch.empty_like(q_raw),
                None if z_g is None else torch.empty_like(z_g),
                None if z_beta is None else torch.empty_like(z_beta))
    q, k, v, g, beta = outs
    _dev(q, "q", q_raw.dtype, q_raw.shape)
    _dev(k, "k", q_raw.dtype, q_raw.shape)
    _dev(v, "v", q_raw.dtype, q_raw.shape)
    # the gate outputs are written (and so checked) only when their logits are given
    if z_g is not None:
        if g is None:
            raise ValueError("outs must hold a g buffer when z_g is given")
        _dev(g, "g", torch.float32, q_raw.shape)
    if z_beta is not None:
        if beta is None:
            raise ValueError("outs must hold a beta buffer when z_beta is given")
        _dev(beta, "beta", torch.float32, (T, H))
    st = lib.kda_prologue(_ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(conv_w), _ptr(z_g),
                          _ptr(z_beta), _ptr(cu), N, T, dims_of(q_raw), _ptr(q), _ptr(k),
                          _ptr(v), _ptr(g), _ptr(beta), _stream())
    if st != KDA_OK:
        raise KDAError(st, "kda_prologue")
    return q, k, v, g, beta


def kda_decode_step_conv(q_raw, k_raw, v_raw, conv_w, conv_state, z_g, z_beta, state,
                         out=None):
    """One decode step through the fused prologue with the ShortConv cache.

    conv_state [N, 3, 3, H, d] (raw dtype) and state [N, H, d, d] are updated
    in place; returns out [N, H, d]."""
    N, H, d = q_raw.shape
    _dev(q_raw, "q_raw")
    _dev(k_raw, "k_raw", q_raw.dtype, q_raw.shape)
    _dev(v_raw, "v_raw", q_raw.dtype, q_raw.shape)
    _dev(conv_w, "conv_w", torch.float32, (3, H * d, 4))
    _dev(conv_state, "conv_state", q_raw.dtype, (N, 3, 3, H, d))
    _dev(z_g, "z_g", torch.float32, q_raw.shape)
    _dev(z_beta, "z_beta", torch.float32, (N, H))
    _dev(state, "state", torch.float32, (N, H, d, d))
    if out is None:
        out = torch.empty_like(v_raw)
    _dev(out, "out", q_raw.dtype, q_raw.shape)
    st = lib.kda_decode_step_conv(_ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(conv_w),
                                  _ptr(conv_state), _ptr(z_g), _ptr(z_beta), _ptr(state),
                                  _ptr(out), N, dims_of(q_raw), _stream())
    if st != KDA_OK:
        raise KDAError(st, "kda_decode_step_conv")
    return out


def kda_decode_verify(q, k, v, g, beta, state_in, accept, K, out=None, state_out=None):
    """K draft tokens per sequence from read-only state_in; returns
    (out [N*K, H, d], state_out [N, H, d, d] = state after accept[n] tokens)."""
    NK, H, d = q.shape
    N = NK // K
    if N * K != NK:
        raise ValueError("q must hold N*K rows")
    _dev(q, "q")
    _dev(k, "k", q.dtype, q.shape)
    _dev(v, "v", q.dtype, q.shape)
    _dev(g, "g", torch.float32, q.shape)
    _dev(beta, "beta", torch.float32, (NK, H))
    _dev(state_in, "state_in", torch.float32, (N, H, d, d))
    acc = accept if (isinstance(accept, torch.Tensor) and accept.is_cuda) else \
        torch.as_tensor(accept, dtype=torch.int32).to(q.device)
    _dev(acc, "accept", torch.int32, (N,))
    if out is None:
        out = torch.empty_like(v)
    _dev(out, "out", q.dtype, q.shape)
    if state_out is None:
        state_out = torch.empty_like(state_in)
    _dev(state_out, "state_out", torch.float32, (N, H, d, d))
    st = lib.kda_decode_verify(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_in),
                               _ptr(acc), N, K, dims_of(q), _ptr(out), _ptr(state_out),
                               _stream())
    if st != KDA_OK:
        raise KDAError(st, "kda_decode_verify")
    return out, state_out


def kda_output_gate(o, z, weight=None, eps=1e-6, out=None):
    """Head RMSNorm x sigmoid(gate logits); o, z [T, H, d]; weight [d] or None."""
    T, H, d = o.shape
    _dev(o, "o")
    _dev(z, "z", o.dtype, o.shape)
    _dev(weight, "weight", torch.float32, (d,))
    if out is None:
        out = torch.empty_like(o)
    _dev(out, "out", o.dtype, o.shape)
    st = lib.kda_output_gate(_ptr(o), _ptr(z), _ptr(weight), T, dims_of(o), float(eps),
                             _ptr(out), _stream())
    if st != KDA_OK:
        raise KDAError(st, "kda_output_gate")
    return out


def kda_get_device_status(workspace) -> int:
    """Wait for the current stream and return the workspace status word."""
    word = ctypes.c_int32(0)
    st = lib.kda_get_device_status(_ptr(workspace), ctypes.byref(word), _stream())
    if st not in (KDA_OK, KDA_ERR_DEVICE, KDA_ERR_TIMEOUT):
        raise KDAError(st, "kda_get_device_status")
    return int(word.value)


def kda_last_error() -> str:
    return lib.kda_last_error().decode(errors="replace")


def kda_kernel_launches() -> int:
    """Kernels this library has queued in this process so far."""
    return int(lib.kda_kernel_launches())
