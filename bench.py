#!/usr/bin/env python
"""KDA benchmark on GB300: prefill tokens/s and decode steps/s (H=96, d=128)
as absolute throughput and as a fraction of the HBM roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kda|reference]

One JSON line on stdout (rank 0).  The headline `value` is prefill tokens/s
on the single-sequence workload (T=4096, H=96, d_k=d_v=128, bf16 q/k/v, fp32
g/beta/state); the same line carries the decode workload (256 sequences x one
token) and the long-context workload (T=262,144 through the fused prologue
and the prefill) as sub-objects, each with its own roofline.

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and a device synchronise on both sides, CUDA events on the launching stream,
max over ranks.  Every workload's inputs exceed the 129 MB L2 (no flush).
With N > 1 (torchrun) every rank runs its own copy of the workload on its GPU
(independent sequences, no collective on the data path): weak scaling.

--impl reference times the fp64 CPU oracle (the only implementation the
pages leave to compare against) on the host cores, on a bounded head sample
of the same workload, and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "KDA prefill tokens/s and decode steps/s (H=96,d=128), % of roofline"
H, D = 96, 128
# algorithmic bytes (each input read once, each output written once)
BYTES_PER_TOKEN = H * D * 2 * 3 + H * D * 4 + H * 4 + H * D * 2   # 147,840
STATE_BYTES = H * D * D * 4                                         # 6,291,456 per document
DECODE_BYTES_PER_SEQ = H * (2 * D * D * 4 + 3 * D * 2 + D * 4 + 4 + D * 2)  # 96 * 132,612
# standalone prologue: raw q,k,v + z_g + z_beta in; q,k,v + g + beta out
PROLOGUE_BYTES_PER_TOKEN = 2 * (H * D * 2 * 3 + H * D * 4 + H * 4)           # 246,528


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# ------------------------------------------------------------------ distributed

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if self.pg is None:
            return x
        dev = "cuda" if torch.cuda.is_available() and self.pg.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (every 50 ms) while GPU work runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="kda_clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval), "-i", str(self.gpu)], stdout=self.out,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        loaded = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------ timing

def time_steps(dist, step, steps, warmup, counter=None):
    """Run `step` warmup + steps times; return (total_ms max over ranks,
    per-step ms list from events around each step on the current stream,
    kernels launched inside the timed region when `counter` is given)."""
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    n0 = counter() if counter else 0
    t0.record()
    for a, b in ev:
        a.record()
        step()
        b.record()
    t1.record()
    n1 = counter() if counter else 0
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    total = dist.max(t0.elapsed_time(t1))
    per = [a.elapsed_time(b) for a, b in ev]
    return (total, per, n1 - n0) if counter else (total, per)


def traffic_for(kernel, units):
    """DRAM bytes per launch from the committed ncu summary, scaled to `units`
    (tokens or sequences) of this launch -- or None when the kernel's source
    changed after the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f)[kernel]
        with open(os.path.join(ROOT, entry["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != entry["sha256"]:
                return None
        return int(entry["dram_bytes"] * units / entry["units"])
    except (OSError, KeyError, ValueError):
        return None


def prologue_traffic(T):
    """DRAM bytes of the two prologue kernels together (conv and gates)."""
    a, b = traffic_for("conv_swish_norm_kernel", T), traffic_for("gates_kernel", T)
    return None if a is None or b is None else a + b


def roofline(bytes_per_launch, launch_ms, peak_gbs, traffic=None):
    achieved = bytes_per_launch / (launch_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak_gbs, "unit": "GB/s",
            "frac": round(achieved / peak_gbs, 4), "traffic": traffic,
            "algorithmic_bytes": int(bytes_per_launch)}


# ------------------------------------------------------------------ workloads

def bench_prefill(kda, synth, dist, args, peaks):
    inp = synth.inputs(2, device="cuda")
    if args.prefill_tokens:
        inp = {k: (v[:args.prefill_tokens].contiguous() if isinstance(v, torch.Tensor) else v)
               for k, v in inp.items()}
    T = inp["q"].shape[0]
    out = torch.empty_like(inp["v"])
    fin = torch.empty(1, H, D, D, dtype=torch.float32, device="cuda")
    ws = torch.empty(kda.kda_prefill_workspace_size(H, D, torch.bfloat16, T, 1),
                     dtype=torch.uint8, device="cuda")

    def step():
        kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], None, None,
                        out=out, final_state=fin, workspace=ws)

    total_ms, per, launches_timed = time_steps(dist, step, args.steps, args.warmup,
                                               counter=kda.kda_kernel_launches)
    bytes_launch = BYTES_PER_TOKEN * T + STATE_BYTES
    res = {"total_ms": total_ms, "tokens": T, "launch_ms": statistics.mean(per),
           "roofline": roofline(bytes_launch, statistics.mean(per), peaks["hbm_gbs"],
                                traffic_for("chunk_kernel", T)),
           "gpu_launches": int(launches_timed)}

    # end to end: pinned host inputs -> device, prefill, outputs -> pinned host
    host = {k: inp[k].cpu().pin_memory() for k in ("q", "k", "v", "g", "beta")}
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_fin = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
    dbuf = {k: torch.empty_like(inp[k]) for k in host}

    def e2e_step():
        for k_, h_ in host.items():
            dbuf[k_].copy_(h_, non_blocking=True)
        kda.kda_prefill(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["g"], dbuf["beta"], None, None,
                        out=out, final_state=fin, workspace=ws)
        h_out.copy_(out, non_blocking=True)
        h_fin.copy_(fin, non_blocking=True)

    e2e_ms, _ = time_steps(dist, e2e_step, args.steps, args.warmup)

    # the same, pipelined: two device buffer sets, and step i+1's host->device
    # copy (its own stream) runs under step i's prefill and read-back; every
    # step still copies its inputs in and its outputs out inside the timed region
    nb = 2
    dbufs = [{k_: torch.empty_like(inp[k_]) for k_ in host} for _ in range(nb)]
    outs = [torch.empty_like(out) for _ in range(nb)]
    fins = [torch.empty_like(fin) for _ in range(nb)]
    wss = [torch.empty_like(ws) for _ in range(nb)]
    h_outs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(nb)]
    h_fins = [torch.empty(fin.shape, dtype=fin.dtype).pin_memory() for _ in range(nb)]
    s_in, s_comp, s_back = (torch.cuda.Stream() for _ in range(3))
    ev_in, ev_comp, ev_back = ([torch.cuda.Event() for _ in range(nb)] for _ in range(3))

    def pipelined(nsteps):
        cur = torch.cuda.current_stream()
        for st_ in (s_in, s_comp, s_back):
            st_.wait_stream(cur)
        for i in range(nsteps):
            b = i % nb
            with torch.cuda.stream(s_in):
                if i >= nb:
                    s_in.wait_event(ev_comp[b])          # step i - nb has consumed buffer set b
                for k_, h_ in host.items():
                    dbufs[b][k_].copy_(h_, non_blocking=True)
                ev_in[b].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev_in[b])
                if i >= nb:
                    s_comp.wait_event(ev_back[b])        # step i - nb's outputs are read back
                kda.kda_prefill(dbufs[b]["q"], dbufs[b]["k"], dbufs[b]["v"], dbufs[b]["g"],
                                dbufs[b]["beta"], None, None, out=outs[b], final_state=fins[b],
                                workspace=wss[b])
                ev_comp[b].record(s_comp)
            with torch.cuda.stream(s_back):
                s_back.wait_event(ev_comp[b])
                h_outs[b].copy_(outs[b], non_blocking=True)
                h_fins[b].copy_(fins[b], non_blocking=True)
                ev_back[b].record(s_back)
        for st_ in (s_in, s_comp, s_back):
            cur.wait_stream(st_)

    pipelined(args.warmup)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    pipelined(args.steps)
    t1.record()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    pipe_ms = dist.max(t0.elapsed_time(t1))
    res["e2e"] = {"value": round(dist.world * T * args.steps / (pipe_ms * 1e-3), 1),
                  "unit": "tokens/s", "pipelined": True,
                  "serial_value": round(dist.world * T * args.steps / (e2e_ms * 1e-3), 1),
                  "h2d_bytes_per_step": int(sum(h.numel() * h.element_size()
                                                for h in host.values())),
                  "d2h_bytes_per_step": int(h_out.numel() * h_out.element_size()
                                            + h_fin.numel() * h_fin.element_size())}
    del inp, host, dbuf, dbufs, outs
    return res


def bench_decode(kda, synth, dist, args, peaks):
    inp = synth.inputs(5, device="cuda")
    if args.decode_seqs:
        inp = {k: (v[:args.decode_seqs].contiguous() if isinstance(v, torch.Tensor) else v)
               for k, v in inp.items()}
    N = inp["q"].shape[0]
    state = inp["init_state"]
    out = torch.empty_like(inp["v"])

    def step():
        kda.kda_decode_step(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], state, out=out)

    total_ms, per = time_steps(dist, step, args.steps, args.warmup)
    steps_s = args.steps / (total_ms * 1e-3)
    return {"workload": "decode: 256 sequences x 1 token, H=96, d=128, fp32 state in place",
            "value": round(steps_s * dist.world, 2), "unit": "steps/s",
            "tokens_per_s": round(steps_s * N * dist.world, 1),
            "ms_per_step": round(total_ms / args.steps, 4),
            "roofline": roofline(DECODE_BYTES_PER_SEQ * N, statistics.mean(per),
                                 peaks["hbm_gbs"], traffic_for("decode_kernel", N))}


def bench_long(kda, dist, args, peaks):
    T = args.long_tokens
    g = torch.Generator(device="cuda").manual_seed(3)
    mk = lambda *s, dt=torch.float32: torch.randn(*s, generator=g, device="cuda",
                                                  dtype=torch.float32).to(dt)
    q_raw, k_raw, v_raw = (mk(T, H, D, dt=torch.bfloat16) for _ in range(3))
    conv_w = 0.5 * mk(3, H * D, 4)
    z_g, z_b = mk(T, H, D), mk(T, H)
    q, k, v = (torch.empty_like(q_raw) for _ in range(3))
    gg, bb = torch.empty_like(z_g), torch.empty_like(z_b)
    out = torch.empty_like(q_raw)
    fin = torch.empty(1, H, D, D, dtype=torch.float32, device="cuda")
    ws = torch.empty(kda.kda_prefill_workspace_size(H, D, torch.bfloat16, T, 1),
                     dtype=torch.uint8, device="cuda")

    def prologue():
        kda.kda_prologue(q_raw, k_raw, v_raw, conv_w, z_g, z_b, None, outs=(q, k, v, gg, bb))

    def prefill():
        kda.kda_prefill(q, k, v, gg, bb, None, None, out=out, final_state=fin, workspace=ws)

    steps = max(1, min(args.steps, args.long_steps))
    for _ in range(min(args.warmup, 3)):
        prologue()
        prefill()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    mk_ev = lambda: torch.cuda.Event(enable_timing=True)
    t0, t1 = mk_ev(), mk_ev()
    evs = [(mk_ev(), mk_ev(), mk_ev()) for _ in range(steps)]
    t0.record()
    for a, b, c in evs:
        a.record()
        prologue()
        b.record()
        prefill()
        c.record()
    t1.record()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    total_ms = dist.max(t0.elapsed_time(t1))
    pro = statistics.mean(a.elapsed_time(b) for a, b, _ in evs)
    pre = statistics.mean(b.elapsed_time(c) for _, b, c in evs)
    bytes_step = BYTES_PER_TOKEN * T + STATE_BYTES + conv_w.numel() * 4
    two = {"ms_per_step": round(total_ms / steps, 3),
           "value": round(dist.world * T * steps / (total_ms * 1e-3), 1),
           "prologue": {"ms": round(pro, 3),
                        "roofline": roofline(PROLOGUE_BYTES_PER_TOKEN * T + conv_w.numel() * 4,
                                             pro, peaks["hbm_gbs"], prologue_traffic(T))},
           "prefill": {"ms": round(pre, 3),
                       "roofline": roofline(BYTES_PER_TOKEN * T + STATE_BYTES, pre,
                                            peaks["hbm_gbs"], traffic_for("chunk_kernel", T))}}
    del q, k, v, gg, bb
    torch.cuda.empty_cache()
    # the library's segment pipeline: the next segment's prologue runs while the
    # current segment's prefill runs, with segment-sized intermediates
    seg = args.segment_tokens
    ws_p = torch.empty(kda.kda_prologue_prefill_workspace_size(H, D, torch.bfloat16, T, seg),
                       dtype=torch.uint8, device="cuda")
    fin1 = torch.empty(H, D, D, dtype=torch.float32, device="cuda")

    # the prefills on a high-priority stream, the prologues on a low-priority one
    hi = torch.cuda.Stream(priority=-1)
    lo = torch.cuda.Stream(priority=0)

    def fused():
        kda.kda_prologue_prefill(q_raw, k_raw, v_raw, conv_w, z_g, z_b, None, seg, out=out,
                                 final_state=fin1, workspace=ws_p, prologue_stream=lo)

    torch.cuda.synchronize()
    with torch.cuda.stream(hi):
        pipe_ms, _ = time_steps(dist, fused, steps, min(args.warmup, 3))
    return {"workload": f"long context: T={T}, H=96, d=128, raw bf16 q/k/v through the "
                        "prologue, then prefill",
            "value": round(dist.world * T * steps / (pipe_ms * 1e-3), 1), "unit": "tokens/s",
            "ms_per_step": round(pipe_ms / steps, 3), "steps": steps,
            "roofline": roofline(bytes_step, pipe_ms / steps, peaks["hbm_gbs"]),
            "note": "bytes credited: raw q/k/v, z_g, z_beta in, out and final state written "
                    f"once (the fused minimum). kda_prologue_prefill, {seg}-token segments: "
                    "the next segment's prologue overlaps the current prefill",
            "two_kernels": two}


# per (sequence, head): state read + written, raw q/k/v, conv cache read +
# written (3 taps x 3 tensors), z_g, z_beta, out
CONV_DECODE_BYTES = 2 * D * D * 4 + 3 * D * 2 + 2 * 9 * D * 2 + D * 4 + 4 + D * 2
# per (sequence, head) for K drafts: state_in read, state_out written, and
# per draft q,k,v (bf16), g, beta, out
def verify_bytes(K):
    return 2 * D * D * 4 + K * (3 * D * 2 + D * 4 + 4 + D * 2)
# per (token, head): o and z read, y written (bf16)
GATE_BYTES = 3 * D * 2


def bench_extras(kda, synth, dist, args, peaks):
    """The rows beyond the core path, each timed on its own."""
    gen = torch.Generator(device="cuda").manual_seed(11)
    rnd = lambda *s, dt=torch.float32, sc=1.0: (sc * torch.randn(*s, generator=gen, device="cuda")).to(dt)
    res = {}
    N = 256
    # decode with the ShortConv cache: 256 sequences x 1 token
    raw = [rnd(N, H, D, dt=torch.bfloat16) for _ in range(3)]
    conv_w = rnd(3, H * D, 4, sc=0.5)
    cache = rnd(N, 3, 3, H, D, dt=torch.bfloat16)
    z_g, z_b = rnd(N, H, D), rnd(N, H)
    state = rnd(N, H, D, D, sc=0.01)
    out = torch.empty_like(raw[0])
    step = lambda: kda.kda_decode_step_conv(raw[0], raw[1], raw[2], conv_w, cache, z_g, z_b, state,
                                            out=out)
    total, per = time_steps(dist, step, args.steps, args.warmup)
    res["decode_conv"] = {"workload": "decode with the ShortConv cache: 256 sequences x 1 token",
                          "value": round(args.steps / (total * 1e-3), 2), "unit": "steps/s",
                          "ms_per_step": round(total / args.steps, 4),
                          "roofline": roofline(CONV_DECODE_BYTES * N * H, statistics.mean(per),
                                               peaks["hbm_gbs"])}
    del cache, raw
    # verify: 256 sequences x 4 drafts from a read-only state, accept 2
    K = 4
    q = torch.nn.functional.normalize(rnd(N * K, H, D), dim=-1).to(torch.bfloat16)
    k = torch.nn.functional.normalize(rnd(N * K, H, D), dim=-1).to(torch.bfloat16)
    v = rnd(N * K, H, D, dt=torch.bfloat16)
    g = -5.0 * torch.sigmoid(rnd(N * K, H, D))
    b = torch.sigmoid(rnd(N * K, H))
    acc = torch.full((N,), 2, dtype=torch.int32, device="cuda")
    s_out = torch.empty_like(state)
    o2 = torch.empty_like(v)
    step = lambda: kda.kda_decode_verify(q, k, v, g, b, state, acc, K, out=o2, state_out=s_out)
    total, per = time_steps(dist, step, args.steps, args.warmup)
    res["verify"] = {"workload": "verify: 256 sequences x 4 drafts, rollback state after 2",
                     "value": round(args.steps / (total * 1e-3), 2), "unit": "verifies/s",
                     "ms_per_step": round(total / args.steps, 4),
                     "roofline": roofline(verify_bytes(K) * N * H, statistics.mean(per),
                                          peaks["hbm_gbs"], traffic_for("verify_pair_kernel", N))}
    del q, k, v, g, b, state, s_out, o2
    # output gate on the T=4096 shape
    T = 4096
    o = rnd(T, H, D, dt=torch.bfloat16)
    z = rnd(T, H, D, dt=torch.bfloat16)
    w = torch.rand(D, device="cuda") + 0.5
    y = torch.empty_like(o)
    step = lambda: kda.kda_output_gate(o, z, w, out=y)
    total, per = time_steps(dist, step, args.steps, args.warmup)
    res["output_gate"] = {"workload": "head RMSNorm x sigmoid(gate), T=4096, H=96, d=128 bf16",
                          "value": round(T * args.steps / (total * 1e-3), 1), "unit": "tokens/s",
                          "ms_per_step": round(total / args.steps, 4),
                          "roofline": roofline(GATE_BYTES * T * H, statistics.mean(per),
                                               peaks["hbm_gbs"],
                                               traffic_for("output_gate_bf16_kernel", T))}
    del o, z, y
    # packed documents (8 of 512..8192 tokens, initial states given): CTAs
    # dispatched longest first (the default workspace) against document order
    # (a workspace with room for the status word only)
    inp = synth.inputs(3, device="cuda")
    cu = torch.as_tensor(inp["cu_seqlens"], dtype=torch.int32, device="cuda")
    T, Nd = inp["q"].shape[0], cu.numel() - 1
    po, pf = torch.empty_like(inp["q"]), torch.empty(Nd, H, D, D, device="cuda")
    ws_full = torch.empty(kda.kda_prefill_workspace_size(H, D, torch.bfloat16, T, Nd),
                          dtype=torch.uint8, device="cuda")
    ws_min = torch.empty(256, dtype=torch.uint8, device="cuda")
    packed = {}
    for name, ws in (("longest_first", ws_full), ("document_order", ws_min)):
        step = lambda ws=ws: kda.kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                             inp["init_state"], cu, out=po, final_state=pf,
                                             workspace=ws)
        total, per = time_steps(dist, step, args.steps, args.warmup)
        packed[name] = (total, per)
    total, per = packed["longest_first"]
    res["packed_documents"] = {
        "workload": f"8 packed documents of 512..8192 tokens (T={T}), H=96, d=128 bf16, initial states",
        "value": round(T * args.steps / (total * 1e-3), 1), "unit": "tokens/s",
        "ms_per_step": round(total / args.steps, 4),
        "document_order_ms_per_step": round(packed["document_order"][0] / args.steps, 4),
        "roofline": roofline(BYTES_PER_TOKEN * T + 2 * Nd * STATE_BYTES, statistics.mean(per),
                             peaks["hbm_gbs"])}
    del inp, po, pf
    # segmented prefill of one long document: with few heads the plain prefill
    # fills only H SMs; the segments give segments x H CTAs at 3x the arithmetic
    for Hs, nseg in ((8, 16), (96, 2)):
        T = 65536
        q = torch.nn.functional.normalize(rnd(T, Hs, D), dim=-1).to(torch.bfloat16)
        k = torch.nn.functional.normalize(rnd(T, Hs, D), dim=-1).to(torch.bfloat16)
        v = rnd(T, Hs, D, dt=torch.bfloat16)
        g = -5.0 * torch.sigmoid(rnd(T, Hs, D))
        b = torch.sigmoid(rnd(T, Hs))
        o3 = torch.empty_like(v)
        fin = torch.empty(Hs, D, D, device="cuda")
        ws = torch.empty(kda.kda_prefill_segmented_workspace_size(Hs, D, torch.bfloat16, T, nseg),
                         dtype=torch.uint8, device="cuda")
        ws1 = torch.empty(kda.kda_prefill_workspace_size(Hs, D, torch.bfloat16, T, 1),
                          dtype=torch.uint8, device="cuda")
        fin1 = torch.empty(1, Hs, D, D, device="cuda")
        seg = lambda: kda.kda_prefill_segmented(q, k, v, g, b, None, nseg, out=o3, final_state=fin,
                                                workspace=ws)
        plain = lambda: kda.kda_prefill(q, k, v, g, b, None, None, out=o3, final_state=fin1,
                                        workspace=ws1)
        steps = max(1, min(args.steps, 5))
        t_seg, _ = time_steps(dist, seg, steps, min(args.warmup, 2))
        t_plain, _ = time_steps(dist, plain, steps, min(args.warmup, 2))
        bytes_step = BYTES_PER_TOKEN // H * Hs * T + Hs * D * D * 4
        res[f"segmented_h{Hs}"] = {
            "workload": f"one document T={T}, H={Hs}, d=128 bf16, {nseg} segments",
            "value": round(T * steps / (t_seg * 1e-3), 1), "unit": "tokens/s",
            "ms_per_step": round(t_seg / steps, 4),
            "plain_prefill_tokens_per_s": round(T * steps / (t_plain * 1e-3), 1),
            "speedup_vs_plain": round(t_plain / t_seg, 3),
            "roofline": roofline(bytes_step, t_seg / steps, peaks["hbm_gbs"])}
        del q, k, v, g, b, o3, ws
    return res


def legs_summary(dec, lng, ext):
    """{value, unit, ms_per_step, frac} per leg (frac: of the measured HBM copy)."""
    def one(r):
        if not r:
            return None
        return {"value": r.get("value"), "unit": r.get("unit"), "ms_per_step": r.get("ms_per_step"),
                "frac": (r.get("roofline") or {}).get("frac")}
    out = {"decode": one(dec), "long_context": one(lng)}
    if lng and lng.get("two_kernels"):
        two = lng["two_kernels"]
        out["long_context"]["prefill_alone_ms"] = two["prefill"]["ms"]
        out["long_context"]["prologue_alone_ms"] = two["prologue"]["ms"]
    ext = ext or {}
    out["packed_documents"] = one(ext.get("packed_documents"))
    out["extras"] = {k: one(v) for k, v in ext.items() if k != "packed_documents" and isinstance(v, dict)
                     and "value" in v}
    return out


def cpu_baseline(synth, heads):
    """fp64 oracle on the host cores over `heads` of the T=4096 workload."""
    import oracle
    from tests.kda_testlib import oracle_prefill
    inp = synth.inputs(2, heads=list(range(heads)))
    T = inp["q"].shape[0]
    t = time.perf_counter()
    oracle_prefill(inp)
    wall = time.perf_counter() - t
    cores = min(heads, os.cpu_count() or 1)
    return {"value": round(T * heads / H / wall, 2), "unit": "tokens/s", "cores": cores,
            "wall_s": round(wall, 4), "kind": "oracle", "sample": f"T=4096 workload, {heads} of 96 heads, all tokens; "
            f"tokens/s scaled to 96 heads ({wall:.2f} s wall)"}


def base_line(args, dist, dtype):
    return {"metric": METRIC, "unit": "tokens/s", "n_gpus": dist.world, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "config": {"workload": "prefill: 1 sequence, T=4096, H=96, d_k=d_v=128, bf16 "
                                   "q/k/v, fp32 g/beta, zero initial state",
                       "T": 4096, "H": H, "d": D, "documents": 1,
                       "l2": "inputs 612 MB > 129 MB L2 (no flush)",
                       "parallelism": f"replicas x{dist.world}" if dist.world > 1 else "1 GPU"}}


def run_reference(args, dist):
    import synth
    if dist.rank != 0:
        return 0
    heads = args.ref_heads
    cb = None
    vals, walls = [], []
    for i in range(args.warmup + args.steps):
        cb = cpu_baseline(synth, heads)
        if i >= args.warmup:
            vals.append(cb["value"])
            walls.append(cb["wall_s"])
    value = statistics.mean(vals)
    line = base_line(args, dist, "f64")
    # a step is the bounded sample (`heads` of the 96 heads, all 4096 tokens):
    # ms_per_step is its measured wall time; value scales it to the 96 heads
    line.update({"impl": "reference", "value": round(value, 2), "n_gpus": dist.world,
                 "ms_per_step": round(statistics.mean(walls) * 1e3, 2),
                 "cpu_baseline": {k: v for k, v in dict(cb, value=round(value, 2)).items()
                                  if k != "wall_s"},
                 "e2e": {"value": round(value, 2), "unit": "tokens/s",
                         "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}})
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kda", choices=["kda", "reference"])
    ap.add_argument("--long-steps", type=int, default=5)
    ap.add_argument("--long-tokens", type=int, default=262144)
    ap.add_argument("--segment-tokens", type=int, default=16384)
    ap.add_argument("--ref-heads", type=int, default=16)
    ap.add_argument("--no-long", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    # smaller cases for profiler captures (the printed line then describes them)
    ap.add_argument("--only", choices=["prefill", "decode", "long", "extras"])
    ap.add_argument("--prefill-tokens", type=int, default=0)
    ap.add_argument("--decode-seqs", type=int, default=0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    dist = Dist()
    if args.impl == "reference":
        return run_reference(args, dist)

    torch.cuda.set_device(dist.local)
    dist.init("nccl")
    import synth
    from linear_attention_03_gb300 import kda

    peaks = load_peaks()
    if args.only:
        run = {"prefill": lambda: bench_prefill(kda, synth, dist, args, peaks),
               "decode": lambda: bench_decode(kda, synth, dist, args, peaks),
               "long": lambda: bench_long(kda, dist, args, peaks),
               "extras": lambda: bench_extras(kda, synth, dist, args, peaks)}[args.only]
        res = run()
        if dist.rank == 0:
            print(json.dumps({"only": args.only, "result": res}), flush=True)
        dist.close()
        return 0
    # the headline's clock record covers the prefill leg only; every other leg
    # carries its own
    def sampled(fn):
        sampler = ClockSampler(dist.local)
        sampler.start()
        res = fn()
        clk_leg = sampler.stop()
        if isinstance(res, dict):
            res["clocks"] = clk_leg
        return res, clk_leg

    pre, clk = sampled(lambda: bench_prefill(kda, synth, dist, args, peaks))
    pre.pop("clocks", None)
    dec = None if args.no_decode else sampled(lambda: bench_decode(kda, synth, dist, args, peaks))[0]
    torch.cuda.empty_cache()
    lng = None if args.no_long else sampled(lambda: bench_long(kda, dist, args, peaks))[0]
    torch.cuda.empty_cache()
    ext = sampled(lambda: bench_extras(kda, synth, dist, args, peaks))[0]
    cb = None
    if dist.rank == 0 and not args.no_cpu_baseline:
        cb = cpu_baseline(synth, H)
        cb.pop("wall_s", None)

    if dist.rank == 0:
        line = base_line(args, dist, "bf16")
        line.update({
            "value": round(dist.world * pre["tokens"] * args.steps / (pre["total_ms"] * 1e-3), 1),
            "ms_per_step": round(pre["total_ms"] / args.steps, 4),
            "roofline": dict(pre["roofline"], peak_source=f"{peaks['source']} HBM copy"),
            "cpu_baseline": cb, "e2e": pre["e2e"], "gpu_launches": pre["gpu_launches"],
            "clocks": clk,
            # the verbose records of the other legs first, their short summaries last,
            # so that a reader of the line's last ~1.5 KB sees every leg's result
            "detail": {"decode": dec, "long_context": lng, "extras": ext},
            "legs": legs_summary(dec, lng, ext)})
        print(json.dumps(line), flush=True)
    dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
