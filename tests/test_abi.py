"""The C-ABI library loads and exports every entry point include/kda.h
declares; argument checks reject bad calls before touching the GPU.
Runs without a GPU: no call here reaches a kernel launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kda():
    from linear_attention_03_gb300 import build
    build.build()
    from linear_attention_03_gb300 import kda as mod
    return mod


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"KDA_API\s+[^;(]*?\b(kda_\w+)\s*\(", text))
    return names


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("kda_prefill", "kda_decode_step", "kda_prologue",
                     "kda_prefill_workspace_size", "kda_last_error",
                     "kda_get_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(kda):
    for name in declared_symbols():
        assert hasattr(kda.lib, name), f"libkda.so does not export {name}"


def test_oracle_is_not_linked_into_the_product(kda):
    so = open(kda._LIB_PATH, "rb").read()
    assert b"kda_oracle" not in so
    src = os.path.join(ROOT, "linear_attention_03_gb300")
    for dirpath, _, files in os.walk(src):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn


def dims(kda, H=96, d=128, dt=1):
    return kda.kda_dims(H, d, d, dt)


FAKE = 0x10000     # 16-byte aligned, never dereferenced: the checks fail first


@pytest.mark.parametrize("bad, code", [
    (dict(d=100), 2), (dict(d=256), 2), (dict(dt=7), 2), (dict(H=0), 1)])
def test_unsupported_dims_rejected(kda, bad, code):
    d = dims(kda, **bad)
    p = ctypes.c_void_p(FAKE)
    st = kda.lib.kda_decode_step(p, p, p, p, p, p, p, 4, d, None)
    assert st == code
    assert kda.kda_last_error()


def test_prefill_argument_checks(kda):
    p = ctypes.c_void_p(FAKE)
    mis = ctypes.c_void_p(FAKE + 4)
    d = dims(kda)
    ws = kda.lib.kda_prefill_workspace_size(d, 64, 1)
    assert ws >= 4
    call = lambda **o: kda.lib.kda_prefill(
        o.get("q", p), p, p, p, p, None, o.get("cu", None), o.get("N", 1), o.get("T", 64), d,
        p, None, o.get("ws", p), o.get("wsb", ws), None)
    assert call(q=None) == kda.KDA_ERR_INVALID
    assert "q" in kda.kda_last_error()
    assert call(q=mis) == kda.KDA_ERR_INVALID
    assert "aligned" in kda.kda_last_error()
    assert call(N=2) == kda.KDA_ERR_INVALID             # N > 1 needs cu_seqlens
    assert call(N=0) == kda.KDA_ERR_INVALID
    assert call(T=-1) == kda.KDA_ERR_INVALID
    assert call(ws=None) == kda.KDA_ERR_INVALID
    assert call(wsb=ws - 1) == kda.KDA_ERR_INVALID


def test_segmented_prefill_argument_checks(kda):
    p = ctypes.c_void_p(FAKE)
    d = dims(kda)
    ws = kda.lib.kda_prefill_segmented_workspace_size(d, 4096, 4)
    assert ws > 4096 * 4 * 128 * 2                       # holds the zero value tile
    assert kda.lib.kda_prefill_segmented_workspace_size(d, 4096, 0) == 0
    call = lambda **o: kda.lib.kda_prefill_segmented(
        o.get("q", p), p, p, p, p, None, o.get("T", 4096), d, o.get("nseg", 4), p, None,
        o.get("ws", p), o.get("wsb", ws), None, None)
    assert call(nseg=0) == kda.KDA_ERR_INVALID and "num_segments" in kda.kda_last_error()
    assert call(q=None) == kda.KDA_ERR_INVALID
    assert call(ws=ctypes.c_void_p(FAKE + 16)) == kda.KDA_ERR_INVALID   # 256-byte alignment
    assert call(wsb=ws - 1) == kda.KDA_ERR_INVALID
    assert call(T=-1) == kda.KDA_ERR_INVALID


def test_prologue_prefill_argument_checks(kda):
    p = ctypes.c_void_p(FAKE)
    d = dims(kda)
    ws = kda.lib.kda_prologue_prefill_workspace_size(d, 4096, 1024)
    assert ws > 2 * 1024 * 4 * 128 * (3 * 2 + 4)          # two segment-sized buffer sets
    assert kda.lib.kda_prologue_prefill_workspace_size(d, 4096, 0) == 0
    call = lambda **o: kda.lib.kda_prologue_prefill(
        p, p, p, p, o.get("zg", p), p, None, o.get("T", 4096), d, o.get("seg", 1024), p, None,
        o.get("ws", p), o.get("wsb", ws), None, None)
    assert call(seg=0) == kda.KDA_ERR_INVALID and "segment_tokens" in kda.kda_last_error()
    assert call(zg=None) == kda.KDA_ERR_INVALID and "z_g" in kda.kda_last_error()
    assert call(ws=ctypes.c_void_p(FAKE + 16)) == kda.KDA_ERR_INVALID
    assert call(wsb=ws - 1) == kda.KDA_ERR_INVALID


def test_prologue_argument_checks(kda):
    p = ctypes.c_void_p(FAKE)
    d = dims(kda)
    st = kda.lib.kda_prologue(p, p, p, None, p, p, None, 1, 64, d, p, p, p, p, p, None)
    assert st == kda.KDA_ERR_INVALID and "conv_w" in kda.kda_last_error()
    st = kda.lib.kda_prologue(p, p, p, p, p, p, None, 1, 64, d, p, p, p, None, p, None)
    assert st == kda.KDA_ERR_INVALID                     # z_g given, g missing


def test_decode_zero_sequences_is_a_no_op(kda):
    assert kda.lib.kda_decode_step(None, None, None, None, None, None, None, 0,
                                   dims(kda), None) == kda.KDA_OK


def test_verify_argument_checks(kda):
    p, q2 = ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + 0x100000)
    mis = ctypes.c_void_p(FAKE + 4)
    call = lambda **o: kda.lib.kda_decode_verify(
        o.get("q", p), p, p, p, p, o.get("sin", p), p, o.get("N", 4), o.get("K", 3),
        o.get("d", dims(kda)), p, o.get("sout", q2), None)
    assert call(K=0) == kda.KDA_ERR_INVALID
    assert call(N=-1) == kda.KDA_ERR_INVALID
    assert call(N=0) == kda.KDA_OK                              # nothing to do
    assert call(N=2 ** 24, K=2) == kda.KDA_ERR_INVALID          # N * K * H past 2^31
    assert call(N=2 ** 24, K=1, d=dims(kda, H=64)) == kda.KDA_ERR_INVALID   # 2 N H past 2^31
    assert call(q=None) == kda.KDA_ERR_INVALID and "q" in kda.kda_last_error()
    assert call(q=mis) == kda.KDA_ERR_INVALID
    assert call(sout=p) == kda.KDA_ERR_INVALID and "alias" in kda.kda_last_error()
    assert call(d=dims(kda, d=48)) == kda.KDA_ERR_UNSUPPORTED


def test_output_gate_argument_checks(kda):
    p, mis = ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + 4)
    call = lambda **o: kda.lib.kda_output_gate(
        o.get("o", p), p, o.get("w", None), o.get("T", 64), dims(kda), o.get("eps", 1e-6),
        o.get("y", p), None)
    assert call(T=-1) == kda.KDA_ERR_INVALID
    assert call(T=0) == kda.KDA_OK
    assert call(eps=-1.0) == kda.KDA_ERR_INVALID
    assert call(eps=float("nan")) == kda.KDA_ERR_INVALID
    assert call(o=None) == kda.KDA_ERR_INVALID and "o" in kda.kda_last_error()
    assert call(y=mis) == kda.KDA_ERR_INVALID
    assert call(w=mis) == kda.KDA_ERR_INVALID


def test_decode_with_conv_cache_argument_checks(kda):
    p = ctypes.c_void_p(FAKE)
    call = lambda **o: kda.lib.kda_decode_step_conv(
        p, p, p, p, o.get("cache", p), p, p, o.get("state", p), p, o.get("N", 8), dims(kda), None)
    assert call(N=-1) == kda.KDA_ERR_INVALID
    assert call(N=0) == kda.KDA_OK
    assert call(cache=None) == kda.KDA_ERR_INVALID and "conv_state" in kda.kda_last_error()
    assert call(state=None) == kda.KDA_ERR_INVALID and "state" in kda.kda_last_error()


def test_prefill_snapshots_argument_checks(kda):
    p = ctypes.c_void_p(FAKE)
    d = dims(kda)
    call = lambda **o: kda.lib.kda_prefill_snapshots(
        p, p, p, p, p, None, None, 1, 256, d, p, None, o.get("offs", p), o.get("n", 2),
        o.get("snaps", p), p, 256, None)
    assert call(n=-1) == kda.KDA_ERR_INVALID and "n_snapshots" in kda.kda_last_error()
    assert call(offs=None) == kda.KDA_ERR_INVALID and "snapshot_offsets" in kda.kda_last_error()
    assert call(snaps=None) == kda.KDA_ERR_INVALID and "snapshots" in kda.kda_last_error()
    assert call(snaps=ctypes.c_void_p(FAKE + 4)) == kda.KDA_ERR_INVALID   # 16-byte alignment
