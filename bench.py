"""Benchmark of the Gated DeltaNet layer hot path on GB300.

One JSON line on rank 0. The headline workload is one decode step of a
Qwen3.5-9B-like GDN layer (B=64 rows, T=1, 16 key / 32 value heads, d=128,
fp32 recurrent state): `value` is layer tokens/s with every input resident in
HBM. The other paths of the layer are measured in the same run under
"phases": speculative verify (8 paths x 8 draft tokens from one shared state,
per-token checkpoints, commit of the winner), chunked prefill (one row of
8192 tokens continued in 512-token calls) and packed varlen prefill
(32 rows U{16..2048} padded to chunk buckets, 24 independent layers).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--phases decode,verify,decode_mxfp8,stack,proj,prefill,varlen]

--impl reference times the fp64 CPU oracle (the reference implementation of
this path) on the same decode workload, on the host's cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time
from pathlib import Path

import torch

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

from gated_deltanet_recurrence_delta_gb300 import inputs as I  # noqa: E402

METRIC = "GDN layer tokens/s (prefill, decode, verify) and % of HBM / tensor roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024
TRAFFIC_NOTE = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch; writes still held in L2 when "
                "the launch ends are not counted, so for write-heavy kernels this is a lower bound")
ACTS = ("q", "k", "v", "z", "a", "b")
WN = ("A_log", "dt_bias", "conv_w", "norm_w")


# ----------------------------------------------------------------- helpers

def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "measured")
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# The sources each kernel's code is built from (its own file, the headers it
# includes, and the host dispatch): recorded DRAM counters stay valid while
# these are unchanged, whatever happens to the other kernels' files.
_COMMON_SOURCES = ("gdn_common.cuh", "gdn_launch.h", "gdn_api.cu")
_PREFILL_SOURCES = ("gdn_prefill_tc.cu", "gdn_prefill.cu", "gdn_token.cuh", "gdn_umma.cuh") + _COMMON_SOURCES
KERNEL_SOURCES = {
    "decode_kernel": ("gdn_decode.cu", "gdn_token.cuh") + _COMMON_SOURCES,
    "verify_split_kernel": ("gdn_verify.cu", "gdn_token.cuh") + _COMMON_SOURCES,
    "state_copy_kernel": ("gdn_state_copy.cu",) + _COMMON_SOURCES,
    "decode_kernel_mxfp8": ("gdn_decode.cu", "gdn_token.cuh") + _COMMON_SOURCES,
    "commit_kernel": ("gdn_state_copy.cu",) + _COMMON_SOURCES,
    **{k: ("gdn_proj.cu", "gdn_umma.cuh") + _COMMON_SOURCES
       for k in ("gemm_in_proj_prefill", "gemm_in_proj_decode", "gemm_out_proj_decode")},
    **{k: _PREFILL_SOURCES for k in ("front_kernel", "chunk_state_kernel", "output_kernel", "chunk_kernel",
                                     "state_kernel", "front_kernel_gates", "prefill_call_512", "varlen_layer")},
}


def csrc_hash(kernel: str | None = None) -> str:
    """Hash of the code of `kernel`'s sources (all kernel sources when None):
    comments and whitespace are dropped, so an edit of comments alone keeps the
    counters taken on the same code."""
    h = hashlib.sha256()
    csrc = ROOT / "gated_deltanet_recurrence_delta_gb300" / "csrc"
    files = [csrc / f for f in sorted(KERNEL_SOURCES[kernel])] if kernel else sorted(csrc.glob("*"))
    for p in files:
        t = p.read_text(errors="replace")
        t = re.sub(r"/\*.*?\*/", " ", t, flags=re.S)
        t = re.sub(r"//[^\n]*", " ", t)
        h.update(p.name.encode())
        h.update(" ".join(t.split()).encode())
    return h.hexdigest()[:16]


def dram_traffic(kernel: str, field: str = "bytes_per_launch"):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary (or, with
    field="l2_write_bytes_per_launch", the bytes its SMs wrote into L2), or None
    when absent or taken on other kernel sources."""
    p = ROOT / "profiles" / "dram_traffic.json"
    if not p.exists():
        return None
    d = json.loads(p.read_text())
    e = d.get(kernel)
    if not e or e.get("csrc_hash") != csrc_hash(kernel) or field not in e:
        return None
    return float(e[field])


def scaled(x, k):
    return None if x is None else x * k


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


SPIN_HZ = 2.1e9  # cycles per second assumed when sizing the spin kernel (SM clock up to 2070 MHz)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def timed(world, steps, warmup, step_fn, start_fn=None, end_fn=None):
    """Run warmup steps, then `steps` timed steps bracketed by a barrier and a
    synchronize on both sides; returns ms per step, max over ranks. One event
    pair brackets the whole region: an event recorded between two launches
    may stand between a kernel and its programmatic dependent, so no
    per-launch events are taken. A kernel's average launch duration
    is measured as a region of that kernel alone, launched back to back.

    The device is kept busy by a bounded spin kernel (torch.cuda._sleep)
    queued just before the start event, long enough to cover the host's
    enqueue of all timed steps (measured on the warm-up steps): the start event
    is then reached only once every step is queued behind it, so the events
    time the device work and not the Python launch overhead between launches.
    start_fn / end_fn (optional): called right after the start event and
    before the end event, for steps that also use other streams (those streams
    wait for the start, and the timing stream waits for them at the end)."""
    t0 = time.perf_counter()
    for i in range(warmup):
        step_fn(i, None)
    host_s = (time.perf_counter() - t0) / max(1, warmup)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(int(min(0.5, 2.0 * host_s * (steps + 1) + 2e-3) * SPIN_HZ))
    s.record()
    if start_fn:
        start_fn()  # work on other streams waits for the start event
    for i in range(steps):
        step_fn(warmup + i, None)
    if end_fn:
        end_fn()  # the current stream waits for work on other streams
    e.record()
    torch.cuda.synchronize()
    barrier(world)
    ms = s.elapsed_time(e) / steps
    return max_over_ranks(ms, world)


# ------------------------------------------------------------- workloads

def _host_mapped(t) -> bool:
    """True when the pinned host tensor t is mapped into the device's address
    space at its own address (driver pointer attributes: memory type = host,
    device pointer = the host pointer), so a kernel may read it in place."""
    import ctypes
    try:
        cu = ctypes.CDLL("libcuda.so.1")
    except OSError:
        return False
    cu.cuPointerGetAttribute.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64]
    mt, dp = ctypes.c_uint(0), ctypes.c_uint64(0)
    memory_type, device_pointer, memorytype_host = 2, 3, 1
    if cu.cuPointerGetAttribute(ctypes.byref(mt), memory_type, t.data_ptr()) != 0:
        return False
    if cu.cuPointerGetAttribute(ctypes.byref(dp), device_pointer, t.data_ptr()) != 0:
        return False
    return mt.value == memorytype_host and dp.value == t.data_ptr()


def _dims(gdn, s, B, T, n_slots):
    return gdn.make_dims(B=B, T=T, nk=s.nk, nv=s.nv, dk=s.dk, dv=s.dv, n_slots=n_slots)


def _inp(gdn, d, acts=None, **kw):
    a = acts if acts is not None else d
    return gdn.make_inputs(*(a[n] for n in ACTS), *(d[n] for n in WN), **kw)


def decode_bytes(s, B):
    state = 2 * B * s.nv * s.dk * s.dv * 4
    per_row = (s.C + s.vd + 2 * s.nv + s.vd) * 2 + 2 * 3 * s.C * 2   # x, z, a, b, out; conv tail r+w
    weights = s.C * 4 * 2 + s.nv * 8 + s.dv * 2
    return state + B * per_row + weights


def phase_decode(gdn, world, steps, warmup, peak_hbm, local=0, e2e=True):
    s, B = I.QWEN35_9B, 64
    per_set = B * s.nv * s.dk * s.dv * 4
    n_sets = max(4, math.ceil(3 * L2_BYTES / per_set))
    sets = []
    for i in range(n_sets):
        d = I.decode_batch(seed=1 + 1009 * i, B=B, device="cuda")
        d["out"] = torch.empty((B, 1, s.nv, s.dv), dtype=torch.bfloat16, device="cuda")
        d["dims"] = _dims(gdn, s, B, 1, B)
        d["inp"] = _inp(gdn, d)
        sets.append(d)

    def step(i, _):
        d = sets[i % n_sets]
        gdn.decode_step(d["dims"], d["inp"], d["conv_state"], d["state"], d["out"])

    with ClockSampler(local) as clk:  # around the warm-up and the timed region only
        ms = timed(world, steps, warmup, step)
    kms = ms  # one launch per step and nothing else: the step time is the kernel's average launch duration
    nbytes = decode_bytes(s, B)
    res = {"tokens_per_s": B * world / (ms * 1e-3), "ms_per_step": ms, "tokens_per_step": B,
           "kernel_ms": kms, "launches_per_step": 1,
           "roofline": {"bound": "hbm", "achieved": nbytes / (kms * 1e-3) / 1e9, "peak": peak_hbm,
                        "unit": "GB/s", "frac": nbytes / (kms * 1e-3) / 1e9 / peak_hbm,
                        "traffic": dram_traffic("decode_kernel"), "traffic_note": TRAFFIC_NOTE,
                        "l2_write_bytes": dram_traffic("decode_kernel", "l2_write_bytes_per_launch"),
                        "algorithmic_bytes": nbytes},
           "l2": f"inputs larger than L2: {n_sets} rotating layer buffer sets of {per_set / 2**20:.0f} MiB state",
           "clocks": clk.summary()}
    if e2e:
        # end to end through the C-ABI: the step's activations (q, k, v, z, a,
        # b) sit in one pinned host buffer and go to the device in one copy,
        # into views of one device buffer that the call reads; the output rows
        # come back in one copy
        def pack(tensors, device):
            offs, n = [], 0
            for t in tensors:
                offs.append(n)
                n = (n + t.numel() * t.element_size() + 255) // 256 * 256
            buf = torch.empty(n, dtype=torch.uint8, device=device)
            if device == "cpu":
                buf = buf.pin_memory()
            views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]
            return buf, views

        src = sets[0]
        hbuf, hviews = pack([src[n] for n in ACTS], "cpu")
        for v, n in zip(hviews, ACTS):
            v.copy_(src[n])
        dev_in = []
        for d in sets:
            dbuf, dviews = pack([d[n] for n in ACTS], "cuda")
            dev_in.append((dbuf, _inp(gdn, d, acts=dict(zip(ACTS, dviews)))))
        out_h = torch.empty(src["out"].shape, dtype=src["out"].dtype).pin_memory()
        h2d = sum(src[n].numel() * src[n].element_size() for n in ACTS)
        d2h = out_h.numel() * out_h.element_size()

        # copies on two copy streams, so that step i + 1's inputs travel while
        # step i decodes and step i's outputs travel while step i + 1 decodes;
        # events order each buffer's writes and reads across the streams
        comp = torch.cuda.current_stream()
        h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(n_sets)]    # set k's inputs are on the device
        ev_dec = [torch.cuda.Event() for _ in range(n_sets)]   # set k's decode is done
        ev_out = [torch.cuda.Event() for _ in range(n_sets)]   # set k's outputs are on the host

        def e2e_step(i, _):
            k = i % n_sets
            dd = sets[k]
            dbuf, inp = dev_in[k]
            if i >= n_sets:
                h2d_s.wait_event(ev_dec[k])  # the decode n_sets steps ago has read this input buffer
            with torch.cuda.stream(h2d_s):
                dbuf.copy_(hbuf, non_blocking=True)
            ev_in[k].record(h2d_s)
            comp.wait_event(ev_in[k])
            if i >= n_sets:
                comp.wait_event(ev_out[k])  # the outputs n_sets steps ago have left this buffer
            gdn.decode_step(dd["dims"], inp, dd["conv_state"], dd["state"], dd["out"])
            ev_dec[k].record(comp)
            d2h_s.wait_event(ev_dec[k])
            with torch.cuda.stream(d2h_s):
                out_h.copy_(dd["out"], non_blocking=True)
            ev_out[k].record(d2h_s)

        def e2e_join():  # the timed region ends once the last outputs are on the host
            comp.wait_stream(h2d_s)
            comp.wait_stream(d2h_s)

        def e2e_start():  # and starts before the first inputs leave the host
            h2d_s.wait_stream(comp)
            d2h_s.wait_stream(comp)

        ems = timed(world, steps, warmup, e2e_step, start_fn=e2e_start, end_fn=e2e_join)
        res["e2e_copy_engine"] = {"value": B * world / (ems * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                                  "d2h_bytes_per_step": d2h,
                                  "how": "one cudaMemcpyAsync each way per step on two copy streams, events "
                                         "ordering each buffer's reuse"}
        res["e2e"] = dict(res["e2e_copy_engine"])
        del dev_in

        # the same copies without a copy engine (the contract's e2e when the
        # host buffers are device-mapped): right after step i's decode, one
        # gdn_copy_overlapped call uploads step i+1's activations and reads back
        # step i-1's output rows while step i runs, on the decode's own stream;
        # host sets rotate over more than L2, so every step's bytes cross the
        # link. The last step's rows come back after it, inside the region.
        if _host_mapped(hbuf):
            n_h = math.ceil(L2_BYTES / (h2d + d2h)) + 1
            hs = []
            for _ in range(n_h):
                hb, hv = pack([src[n] for n in ACTS], "cpu")
                for v, n in zip(hv, ACTS):
                    v.copy_(src[n])
                hs.append((hb, torch.empty(src["out"].shape, dtype=src["out"].dtype).pin_memory()))
            staged = [pack([d[n] for n in ACTS], "cuda") for d in sets]
            staged_inp = [_inp(gdn, d, acts=dict(zip(ACTS, views))) for d, (_, views) in zip(sets, staged)]
            assert hs[0][0].numel() == h2d  # the packed activations have no padding between them
            last = [0]

            def st_step(i, _):
                k = i % n_sets
                d = sets[k]
                gdn.decode_step(d["dims"], staged_inp[k], d["conv_state"], d["state"], d["out"])
                gdn.copy_overlapped([(staged[(i + 1) % n_sets][0], hs[(i + 1) % n_h][0], h2d),
                                     (hs[(i - 1) % n_h][1], sets[(i - 1) % n_sets]["out"], d2h)])
                last[0] = i

            def st_end():
                hs[last[0] % n_h][1].copy_(sets[last[0] % n_sets]["out"], non_blocking=True)

            gdn.copy_overlapped([(staged[0][0], hs[0][0], h2d)])  # step 0's activations, before the warm-up
            sms = timed(world, steps, warmup, st_step, end_fn=st_end)
            res["e2e"] = {"value": B * world / (sms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                          "d2h_bytes_per_step": d2h, "host_sets": n_h,
                          "how": "per step one gdn_copy_overlapped kernel on the decode's stream: step i+1's "
                                 "activations up and step i-1's output rows down from / to pinned host memory "
                                 "while step i runs"}
            del hs, staged, staged_inp

        # zero-copy through the same call: the activations and the output rows
        # stay in pinned host memory, which the kernel reads and writes across
        # the host link itself (no copy launches, no events between the
        # decodes); host sets rotate over more than L2, so every step's bytes
        # cross the link
        if _host_mapped(hbuf):
            n_h = math.ceil(L2_BYTES / (h2d + d2h)) + 1
            hz = []
            for _ in range(n_h):
                hb, hv = pack([src[n] for n in ACTS], "cpu")
                for v, n in zip(hv, ACTS):
                    v.copy_(src[n])
                hz.append((hb, _inp(gdn, src, acts=dict(zip(ACTS, hv))),
                           torch.empty(src["out"].shape, dtype=src["out"].dtype).pin_memory()))

            def zc_step(i, _):
                d = sets[i % n_sets]
                _, inp, o = hz[i % n_h]
                gdn.decode_step(d["dims"], inp, d["conv_state"], d["state"], o)

            zms = timed(world, steps, warmup, zc_step)
            res["e2e_zero_copy"] = {"value": B * world / (zms * 1e-3), "unit": "tokens/s",
                                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "host_sets": n_h,
                                    "how": "activations read and output rows written by the decode kernel "
                                           "in pinned host memory (NVLink-C2C), no copy launches"}
            del hz
    del sets
    torch.cuda.empty_cache()
    return res


def decode_mxfp8_bytes(s, B):
    state = 2 * B * s.nv * s.dk * s.dv * 4
    tok = s.C + s.vd  # e4m3 q | k | v and z, one byte each
    per_row = tok + tok // 32 + 2 * s.nv * 2 + s.vd * 2 + 2 * 3 * s.C * 2  # + scales, a, b, out, conv tail r+w
    weights = s.C * 4 * 2 + s.nv * 8 + s.dv * 2
    return state + B * per_row + weights


def phase_decode_mxfp8(gdn, world, steps, warmup, peak_hbm):
    """The headline decode step with the token channels in MXFP8."""
    s, B = I.QWEN35_9B, 64
    per_set = B * s.nv * s.dk * s.dv * 4
    n_sets = max(4, math.ceil(3 * L2_BYTES / per_set))
    sets = []
    for i in range(n_sets):
        d = I.decode_batch(seed=1 + 1009 * i, B=B, device="cuda")
        enc = {n: I.mxfp8(d[n]) for n in ("q", "k", "v", "z")}
        d["enc"] = enc
        d["out"] = torch.empty((B, 1, s.nv, s.dv), dtype=torch.bfloat16, device="cuda")
        d["dims"] = _dims(gdn, s, B, 1, B)
        d["inp"] = gdn.make_inputs_mxfp8(*(enc[n][0] for n in ("q", "k", "v", "z")),
                                         *(enc[n][1] for n in ("q", "k", "v", "z")), d["a"], d["b"],
                                         *(d[n] for n in WN))
        sets.append(d)

    def step(i, _):
        d = sets[i % n_sets]
        gdn.decode_step_mxfp8(d["dims"], d["inp"], d["conv_state"], d["state"], d["out"])

    ms = timed(world, steps, warmup, step)
    nbytes = decode_mxfp8_bytes(s, B)
    res = {"tokens_per_s": B * world / (ms * 1e-3), "ms_per_step": ms, "tokens_per_step": B, "launches_per_step": 1,
           "roofline": {"bound": "hbm", "kernel": "decode_kernel (MXFP8 inputs)",
                        "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": peak_hbm, "unit": "GB/s",
                        "frac": nbytes / (ms * 1e-3) / 1e9 / peak_hbm, "algorithmic_bytes": nbytes,
                        "traffic": dram_traffic("decode_kernel_mxfp8"), "traffic_note": TRAFFIC_NOTE},
           "l2": f"inputs larger than L2: {n_sets} rotating layer buffer sets of {per_set / 2**20:.0f} MiB state"}
    del sets
    torch.cuda.empty_cache()
    return res


def verify_bytes(s, P, K):
    ck = P * K * s.nv * s.dk * s.dv * 4 + P * K * 3 * s.C * 2
    state = s.nv * s.dk * s.dv * 4 + 3 * s.C * 2
    acts = P * K * ((s.C + s.vd + 2 * s.nv + s.vd) * 2)
    commit = 2 * (s.nv * s.dk * s.dv * 4 + 3 * s.C * 2)
    return ck + state + acts + commit


def phase_verify(gdn, world, steps, warmup, peak_hbm):
    s, P, K = I.QWEN35_9B, 8, 8
    n_sets = 2
    sets = []
    for i in range(n_sets):
        d = I.verify_paths(seed=3 + 1009 * i, device="cuda")
        d["out"] = torch.empty((P, K, s.nv, s.dv), dtype=torch.bfloat16, device="cuda")
        d["cks"] = torch.empty((P, K, s.nv, s.dk, s.dv), dtype=torch.float32, device="cuda")
        d["ckc"] = torch.empty((P, K, 3, s.C), dtype=torch.bfloat16, device="cuda")
        d["idx"] = torch.zeros(P, dtype=torch.int32, device="cuda")
        _, src = gdn.commit_source_slot(d["accept_len"].tolist(), K)  # the winner's checkpoint, -1 = none
        d["src"] = torch.tensor([src], dtype=torch.int32, device="cuda")
        d["dst"] = torch.zeros(1, dtype=torch.int32, device="cuda")
        d["dims"] = _dims(gdn, s, P, K, 1)
        d["inp"] = _inp(gdn, d, state_idx=d["idx"])
        d["cdims"] = _dims(gdn, s, 1, 1, 1)
        sets.append(d)

    def verify(i, _):
        d = sets[i % n_sets]
        gdn.verify_with_checkpoints(d["dims"], d["inp"], d["conv_state"], d["state"], d["out"], d["cks"], d["ckc"])

    def step(i, _):
        verify(i, _)
        d = sets[i % n_sets]
        gdn.state_copy(d["cdims"], d["cks"], d["ckc"], d["state"], d["conv_state"], d["src"], d["dst"], 1, P * K, 1)

    ms = timed(world, steps, warmup, step)
    kms = timed(world, steps, warmup, verify)  # the verify kernel alone, back to back
    nbytes = verify_bytes(s, P, K)
    vbytes = nbytes - 2 * (s.nv * s.dk * s.dv * 4 + 3 * s.C * 2)
    res = {"tokens_per_s": P * K * world / (ms * 1e-3), "ms_per_step": ms, "tokens_per_step": P * K,
           "kernel_ms": kms, "launches_per_step": 2, "algorithmic_bytes_per_step": nbytes,
           "step_hbm_frac": nbytes / (ms * 1e-3) / 1e9 / peak_hbm,
           "roofline": {"bound": "hbm", "kernel": "verify_split_kernel", "achieved": vbytes / (kms * 1e-3) / 1e9,
                        "peak": peak_hbm, "unit": "GB/s", "frac": vbytes / (kms * 1e-3) / 1e9 / peak_hbm,
                        "traffic": dram_traffic("verify_split_kernel"), "traffic_note": TRAFFIC_NOTE,
                        "l2_write_bytes": dram_traffic("verify_split_kernel", "l2_write_bytes_per_launch")}}
    del sets
    torch.cuda.empty_cache()
    return res


def phase_stack(gdn, world, steps, warmup, peak_hbm, n_layers=24):
    """A 24-layer stack on per-layer pools, each step one replay of a captured
    CUDA graph: (1) a decode token for 64 rows through every layer; (2) every
    layer's verify of 8 paths x 8 draft tokens from one shared slot, then the
    fused commit of the winner in all layers (one launch)."""
    from gated_deltanet_recurrence_delta_gb300.stack import LayerStack
    s, B = I.QWEN35_9B, 64
    g = torch.Generator(device="cuda").manual_seed(11)
    weights = [I.weights(s, g, device="cuda") for _ in range(n_layers)]
    stack = LayerStack(s, weights, n_slots=B)
    stack.state_pool.normal_(0.0, 0.1, generator=g)
    stack.conv_pool.copy_(torch.randn(stack.conv_pool.shape, generator=g, device="cuda").to(torch.bfloat16))
    dec = stack.capture_decode(B)
    for acts in dec.acts:
        for t in acts.values():
            t.copy_(torch.randn(t.shape, generator=g, device="cuda").to(torch.bfloat16))
    ms = timed(world, steps, warmup, lambda i, _: dec.replay())
    nbytes = n_layers * decode_bytes(s, B)
    res = {"decode": {"tokens_per_s": B * world / (ms * 1e-3), "layer_tokens_per_s": B * n_layers * world / (ms * 1e-3),
                      "ms_per_step": ms, "ms_per_layer": ms / n_layers, "launches_per_step": n_layers,
                      "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / peak_hbm, "algorithmic_bytes_per_step": nbytes,
                      "l2": f"inputs larger than L2: {n_layers} layers x {B * s.nv * s.dk * s.dv * 4 / 2**20:.0f} MiB state"}}
    del dec
    P, K = 8, 8
    ver = stack.capture_verify_commit(P, K, P)
    for acts in ver.acts:
        for t in acts.values():
            t.copy_(torch.randn(t.shape, generator=g, device="cuda").to(torch.bfloat16))
    acc = torch.randint(0, K + 1, (P,), generator=g, device="cuda").to(torch.int32)
    ver.accept_len.copy_(acc)
    ms = timed(world, steps, warmup, lambda i, _: ver.replay())
    nbytes = n_layers * verify_bytes(s, P, K)
    res["verify_commit"] = {"tokens_per_s": P * K * world / (ms * 1e-3), "ms_per_step": ms,
                            "ms_per_layer": ms / n_layers, "launches_per_step": n_layers + 1,
                            "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / peak_hbm, "algorithmic_bytes_per_step": nbytes,
                            "l2": f"inputs larger than L2: {n_layers} layers x 128 MiB of checkpoints"}
    del ver, stack, weights
    torch.cuda.empty_cache()
    return res


def phase_proj(gdn, world, steps, warmup, peak_hbm, peak_tf):
    """The layer's projections (tcgen05 GEMMs) at the Qwen3.5-9B-like layer's
    sizes (hidden 4096): the in-projection, split into the layer's six input
    tensors in its epilogue (12352 output features), and the out-projection
    (4096 x 4096). Decode-sized calls (64 tokens) stream their weights: HBM
    roofline over rotating weight sets larger than L2. Prefill-sized calls
    (8192 tokens): tensor roofline."""
    s, H = I.QWEN35_9B, 4096
    N = 2 * s.kd + 2 * s.vd + 2 * s.nv
    g = torch.Generator(device="cuda").manual_seed(12)
    res = {}
    for M in (64, 8192):
        n_sets = max(2, math.ceil(3 * L2_BYTES / (N * H * 2))) if M == 64 else 1
        w_in = [(torch.randn((N, H), generator=g, device="cuda") * H ** -0.5).to(torch.bfloat16) for _ in range(n_sets)]
        w_out = [(torch.randn((H, s.vd), generator=g, device="cuda") * s.vd ** -0.5).to(torch.bfloat16)
                 for _ in range(max(1, math.ceil(3 * L2_BYTES / (H * s.vd * 2))) if M == 64 else 1)]
        hidden = torch.randn((M, H), generator=g, device="cuda").to(torch.bfloat16)
        o = torch.randn((M, s.vd), generator=g, device="cuda").to(torch.bfloat16)
        outs = {n: torch.empty((M, w), dtype=torch.bfloat16, device="cuda")
                for n, w in (("q", s.kd), ("k", s.kd), ("v", s.vd), ("z", s.vd), ("a", s.nv), ("b", s.nv))}
        y = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
        dm = _dims(gdn, s, 1, 1, 1)

        def step_in(i, _):
            gdn.in_proj(dm, hidden, w_in[i % len(w_in)], outs["q"], outs["k"], outs["v"], outs["z"], outs["a"],
                        outs["b"])

        def step_out(i, _):
            gdn.out_proj(o, w_out[i % len(w_out)], y)

        k = steps if M == 64 else max(3, steps // 20)
        ms_in = timed(world, k, warmup, step_in)
        ms_out = timed(world, k, warmup, step_out)
        for name, ms, nout, kk in (("in_proj", ms_in, N, H), ("out_proj", ms_out, H, s.vd)):
            nbytes = (nout * kk + M * kk + M * nout) * 2
            flops = 2.0 * M * nout * kk
            key = f"{name}_{'decode' if M == 64 else 'prefill'}"
            if M == 64:
                roof = {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": peak_hbm, "unit": "GB/s",
                        "frac": nbytes / (ms * 1e-3) / 1e9 / peak_hbm, "algorithmic_bytes": nbytes}
            else:
                roof = {"bound": "tensor", "achieved": flops / (ms * 1e-3) / 1e12, "peak": peak_tf, "unit": "TFLOP/s",
                        "frac": flops / (ms * 1e-3) / 1e12 / peak_tf, "algorithmic_flops": flops}
            if name == "in_proj" or M == 64:
                roof["traffic"] = dram_traffic(f"gemm_{name}_{'decode' if M == 64 else 'prefill'}")
                roof["traffic_note"] = TRAFFIC_NOTE
            res[key] = {"tokens": M, "features": nout, "k": kk, "ms_per_call": ms, "tokens_per_s": M * world / (ms * 1e-3),
                        "roofline": roof}
        del w_in, w_out, hidden, o, outs, y
        torch.cuda.empty_cache()
    return res


def prefill_flops_per_token(s, C=64):
    d = s.dk
    return s.nv * (10 * C * d + 6 * d * d + (2 / 3) * C * C)


def prefill_bytes_per_token(s):
    return (s.C + s.vd + 2 * s.nv + s.vd) * 2


def phase_prefill(gdn, world, steps, warmup, peak_tf):
    s, T, call = I.QWEN35_9B, 8192, 512
    d = I.prefill_long(seed=2, T=T, device="cuda")
    d["out"] = torch.empty((1, T, s.nv, s.dv), dtype=torch.bfloat16, device="cuda")
    dm = _dims(gdn, s, 1, call, 1)
    ws = gdn.workspace(dm)
    calls = []
    for c in range(T // call):
        sl = slice(c * call, (c + 1) * call)
        a = {n: d[n][:, sl] for n in ACTS}
        calls.append((_inp(gdn, d, acts=a), d["out"][:, sl]))

    def step(i, _):
        for inp, out in calls:
            gdn.prefill_chunked(dm, inp, d["conv_state"], d["state"], out, ws)

    ms = timed(world, steps, warmup, step)
    kms = ms  # the roofline covers the whole call (front, chunk+state and output kernels)
    flops = prefill_flops_per_token(s) * T
    res = {"tokens_per_s": T * world / (ms * 1e-3), "ms_per_step": ms, "tokens_per_step": T,
           "ms_per_512_call": ms / (T // call), "launches_per_step": 3 * (T // call),
           "roofline": {"bound": "tensor", "kernel": "front+chunk_state+output", "achieved": flops / (kms * 1e-3) / 1e12, "peak": peak_tf,
                        "unit": "TFLOP/s", "frac": flops / (kms * 1e-3) / 1e12 / peak_tf,
                        "traffic": scaled(dram_traffic("prefill_call_512"), T // call),
                        "traffic_scope": "16 512-token calls (three kernels each)",
                        "traffic_note": TRAFFIC_NOTE,
                        "algorithmic_flops_per_token": prefill_flops_per_token(s)}}
    del d, calls, ws
    torch.cuda.empty_cache()
    return res


def phase_varlen(gdn, world, steps, warmup, peak_tf, n_layers=24):
    s = I.QWEN35_9B
    layers = []
    for l in range(n_layers):
        d = I.varlen_layer(l, device="cuda")
        d["cu_dev"] = d["cu_seqlens"].to("cuda")
        total = int(d["cu_seqlens"][-1])
        d["out"] = torch.empty((1, total, s.nv, s.dv), dtype=torch.bfloat16, device="cuda")
        d["dims"] = _dims(gdn, s, 32, total, 32)
        d["inp"] = _inp(gdn, d, mask=d["mask"][0], cu_seqlens=d["cu_dev"])
        layers.append(d)
    ws = gdn.workspace(layers[0]["dims"], packed=True)
    real = sum(layers[0]["real"])
    padded = int(layers[0]["cu_seqlens"][-1])

    def step(i, _):
        for d in layers:
            gdn.prefill_chunked(d["dims"], d["inp"], d["conv_state"], d["state"], d["out"], ws)

    ms = timed(world, steps, warmup, step)
    kms = ms  # the roofline covers whole layers (all their kernels)
    flops = prefill_flops_per_token(s) * real * n_layers
    res = {"real_tokens_per_s": real * world / (ms * 1e-3),
           "layer_tokens_per_s": real * n_layers * world / (ms * 1e-3), "ms_per_step": ms,
           "real_tokens": real, "padded_tokens": padded, "layers": n_layers, "launches_per_step": 3 * n_layers,
           "roofline": {"bound": "tensor", "kernel": "front+chunk+state", "achieved": flops / (kms * 1e-3) / 1e12, "peak": peak_tf,
                        "unit": "TFLOP/s", "frac": flops / (kms * 1e-3) / 1e12 / peak_tf,
                        "traffic": scaled(dram_traffic("varlen_layer"), n_layers),
                        "traffic_scope": f"{n_layers} layers (three kernels each)", "traffic_note": TRAFFIC_NOTE}}
    del layers, ws
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------- CPU oracle
#
# The fp64 oracle as it stands (never tuned for this), on the host's cores:
# one baseline per phase, each on the phase's own workload or a bounded
# sample of it (stated in `sample`).

def _oracle():
    from oracle import oracle
    oracle.build()
    return oracle


def _okw(d, s, acts, conv_state, state, threads, **extra):
    return dict(**{n: acts[n] for n in ACTS}, **{n: d[n] for n in WN}, conv_state=conv_state, state=state,
                nk=s.nk, nv=s.nv, dk=s.dk, dv=s.dv, n_threads=threads, **extra)


def oracle_decode_steps(steps, rows=64, d=None):
    """`steps` oracle decode steps over the first `rows` rows of the decode
    workload (64 rows x 1 token x 32 heads); returns (tokens/s, seconds)."""
    oracle = _oracle()
    d = d or I.decode_batch(seed=1)
    s = d["shape"]
    threads = os.cpu_count() or 1
    acts = {n: d[n][:rows] for n in ACTS}
    kw = _okw(d, s, acts, d["conv_state"][:rows], d["state"][:rows], threads)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.layer(**kw)
    el = time.perf_counter() - t0
    return rows * steps / el, el


def cpu_decode(seconds=10.0):
    oracle = _oracle()
    d = I.decode_batch(seed=1)
    oracle_decode_steps(1, d=d)  # load + warm
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        oracle_decode_steps(1, d=d)
        n += 1
    rate = 64 * n / (time.perf_counter() - t0)
    return {"value": rate, "unit": "tokens/s", "cores": os.cpu_count() or 1, "kind": "oracle",
            "sample": f"{n} full decode steps of the workload (64 rows x 32 heads), ~{seconds:.0f} s"}


def cpu_verify(seconds=5.0):
    """Whole verify calls: 8 paths x 8 tokens from the shared state, with the
    per-token state and conv-tail checkpoints."""
    oracle = _oracle()
    d = I.verify_paths(seed=3)
    s = d["shape"]
    threads = os.cpu_count() or 1
    P, K = d["q"].shape[0], d["q"].shape[1]
    kw = _okw(d, s, d, d["conv_state"].expand(P, -1, -1), d["state"].expand(P, -1, -1, -1), threads,
              checkpoints=True)
    oracle.layer(**kw)
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.layer(**kw)
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    rate = P * K * n / (time.perf_counter() - t0)
    return {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} full verify calls (8 paths x 8 tokens, 64 state + conv checkpoints each)"}


def cpu_prefill():
    """The whole 8192-token row, one uninterrupted oracle pass."""
    oracle = _oracle()
    d = I.prefill_long(seed=2)
    s = d["shape"]
    threads = os.cpu_count() or 1
    T = d["q"].shape[1]
    t0 = time.perf_counter()
    oracle.layer(**_okw(d, s, d, d["conv_state"], d["state"], threads))
    el = time.perf_counter() - t0
    return {"value": T / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"the whole workload: one row of {T} tokens, 32 heads, one pass ({el:.1f} s)"}


def cpu_varlen(n_layers=1, stack=24):
    """The first n_layers layers of the varlen stack in full (all 32 rows, one
    oracle call per row, four rows at a time); the rate is real tokens per
    second through the whole stack, from the time per layer."""
    from concurrent.futures import ThreadPoolExecutor
    oracle = _oracle()
    threads = os.cpu_count() or 1
    el, real = 0.0, None
    for layer in range(n_layers):
        d = I.varlen_layer(layer, device="cuda") if torch.cuda.is_available() else I.varlen_layer(layer)
        h = {n: d[n].cpu() for n in ACTS + WN}
        conv0, S0, mask = d["conv_state"].cpu(), d["state"].cpu(), d["mask"].cpu()
        cu, real = d["cu_seqlens"], d["real"]
        s = d["shape"]
        del d

        def row(r):
            a, b_ = int(cu[r]), int(cu[r + 1])
            oracle.layer(**_okw(h, s, {n: h[n][:, a:b_] for n in ACTS}, conv0[r:r + 1], S0[r:r + 1], threads,
                                mask=mask[:, a:b_]))

        order = sorted(range(len(real)), key=lambda r: -real[r])
        t0 = time.perf_counter()
        with ThreadPoolExecutor(max_workers=4) as ex:
            list(ex.map(row, order))
        el += time.perf_counter() - t0
    per_layer = el / n_layers
    return {"value": sum(real) / (per_layer * stack), "unit": "real tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_layers} of the {stack} layers in full (all 32 rows, {sum(real)} real tokens per layer, "
                      f"{per_layer:.1f} s per layer); the layers are alike in cost, so the stack takes {stack} x that"}


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--phases", default="decode,verify,decode_mxfp8,stack,proj,prefill,varlen")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stack-layers", type=int, default=24, help="layers of the captured stack phase")
    ap.add_argument("--oracle-varlen-layers", type=int, default=3,
                    help="varlen layers the oracle baseline runs in full (24 = the whole stack)")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    steps, warmup = args.steps, max(3, args.warmup)

    if args.impl == "reference":
        if rank != 0:
            return
        # the oracle on the headline decode workload: W untimed then exactly K
        # timed steps; a step is every row of the workload unless K full steps
        # would run past ~90 s, then the first `rows` rows (a bounded sample)
        d = I.decode_batch(seed=1)
        _, t1 = oracle_decode_steps(1, d=d)
        rows = 64 if steps * t1 <= 90.0 else max(1, int(64 * 90.0 / (steps * t1)))
        oracle_decode_steps(warmup, rows=rows, d=d)
        rate, el = oracle_decode_steps(steps, rows=rows, d=d)
        threads = os.cpu_count() or 1
        line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": 1,
                "steps": steps, "warmup": warmup, "ms_per_step": el / steps * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": "decode step: B=64 rows, T=1, 16 key / 32 value heads, d=128, fp32 state",
                           "global_batch": 64, "seq_len": 1, "parallelism": "host threads"},
                "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                 "sample": f"{steps} timed steps after {warmup} untimed, each the oracle decode "
                                           f"step of {rows} of the workload's 64 rows x 32 heads"},
                "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    from gated_deltanet_recurrence_delta_gb300 import build as gbuild
    from gated_deltanet_recurrence_delta_gb300 import gdn
    if rank == 0:
        gbuild.build()
    barrier(world)
    gdn.load_library()
    peak_hbm, peak_tf, peak_tf_sus, peak_src = peaks()
    phases = [p for p in args.phases.split(",") if p]
    results = {}
    results["decode"] = phase_decode(gdn, world, steps, warmup, peak_hbm, local=local)
    clocks = results["decode"].pop("clocks")
    # prefill calls and varlen layers take well under a second each, so their
    # tensor roofline is the burst bf16 peak
    if "verify" in phases:
        results["verify"] = phase_verify(gdn, world, steps, warmup, peak_hbm)
    if "decode_mxfp8" in phases:
        results["decode_mxfp8"] = phase_decode_mxfp8(gdn, world, steps, warmup, peak_hbm)
    if "stack" in phases:
        results["stack"] = phase_stack(gdn, world, max(3, steps // 40), warmup, peak_hbm, n_layers=args.stack_layers)
    if "proj" in phases:
        results["proj"] = phase_proj(gdn, world, max(20, steps // 10), warmup, peak_hbm, peak_tf)
    if "prefill" in phases:
        results["prefill"] = phase_prefill(gdn, world, max(3, steps // 400), warmup, peak_tf)
    if "varlen" in phases:
        results["varlen"] = phase_varlen(gdn, world, max(2, steps // 1000), 3, peak_tf)
    gdn.check_status()

    dec = results["decode"]
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_decode(seconds=10.0)
        dec["cpu_baseline"] = cpu
        if "verify" in results:
            results["verify"]["cpu_baseline"] = cpu_verify()
        if "prefill" in results:
            results["prefill"]["cpu_baseline"] = cpu_prefill()
        if "varlen" in results:
            results["varlen"]["cpu_baseline"] = cpu_varlen(n_layers=args.oracle_varlen_layers)
    launches = steps * dec["launches_per_step"]
    line = {
        "metric": METRIC, "value": dec["tokens_per_s"], "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": dec["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "dtype_note": "fp32 state and arithmetic; bf16 activations, conv tail and outputs", "data": "synthetic",
        "config": {"workload": "decode step: B=64 rows, T=1, 16 key / 32 value heads, d=128, fp32 state "
                               "(Qwen3.5-9B-like GDN layer)",
                   "global_batch": 64 * world, "seq_len": 1, "parallelism": f"dp{world} (rows, no collective)",
                   "l2": dec["l2"]},
        "roofline": dict(dec["roofline"], kernel="decode_kernel", peak_source=peak_src),
        "cpu_baseline": cpu,
        "e2e": dec.get("e2e"),
        "gpu_launches": launches,
        "clocks": clocks,
        "phases": results,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
