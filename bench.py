"""Benchmark of the KDA hot path on GB300.

Main line (``value``): chunked prefill tokens/s on a long single sequence,
B=1, H=32, dk=dv=128, T=8192, bf16 q/k/v/g/beta, fp32 state, chunk 64,
checkpoints every 512 tokens (16 pages of 2 MiB written through the pack_heads
layout).  Inputs (336 MB per step) are larger than L2, so no flush is needed.
Extra objects in the same JSON line:
  * ``decode``: 256 consecutive decode steps, B=256, H=32, dk=dv=128, fp32
    state (512 MiB, > L2), fresh bf16 projections per step: state GB/s;
  * ``replay``: speculative verify/replay, B=32, H=16, dk=dv=32, draft 8,
    n_accepted ~ U{0..8}, fp32: amortised GB/s over 64 distinct buffer sets
    (> L2) and the device time of one call.

``--impl reference`` times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

# The fp64 oracle runs single-threaded (einsum plus 64x64 BLAS calls): pin BLAS to one
# thread so the CPU baseline's core count is exact.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from kda_delta_rule_gb300 import dist as D           # noqa: E402
from kda_delta_rule_gb300 import inputs as I         # noqa: E402

H, DK, DV, T, STRIDE, CHUNK = 32, 128, 128, 8192, 512, 64
PREFILL_KERNELS_PER_CALL = 2           # chunk prep + chain, the only launches of a timed step
E2E_SEGMENT = 2048                      # tokens per copy/compute segment of the end-to-end call
DEC_B, DEC_STEPS = 256, 256
REP_B, REP_H, REP_D, REP_DRAFT, REP_SETS = 32, 16, 32, 8, 64
CONV_W = 4                              # ShortConv kernel size of the input-prologue measurements
WORKLOAD = (f"kda_prefill_chunked long single sequence: B=1 H={H} dk=dv={DK} T={T} bf16 "
            f"fp32-state chunk={CHUNK} ckpt_stride={STRIDE} (16 checkpoint pages)")


# DRAM bytes (read + write) of one prefill call measured by ncu on the T=8192 H=32 d=128
# case, keyed by the hash of the kernel source it was taken on: reported as null once
# kda_prefill_tc.cu changes.
PREFILL_TRAFFIC = {"a6a5ee43d015d7b5": 904_326_912}


def prefill_traffic():
    path = os.path.join(ROOT, "kda_delta_rule_gb300", "csrc", "kda_prefill_tc.cu")
    try:
        digest = hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    return PREFILL_TRAFFIC.get(digest)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            m = json.load(fh)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def prefill_bytes(T_, H_, dk, dv, es, n_ck, page_bytes, n_seqs=1):
    tok = T_ * H_ * (3 * dk + 2 * dv + 1) * es            # q,k,g,v,beta in, o out
    state = 2 * n_seqs * H_ * dk * dv * 4                  # S0 read, S_final write
    return tok + state + n_ck * page_bytes


def prefill_flops(T_, H_, dk, dv, C=CHUNK):
    # dense chunk form: 2C^2(3dk + 2dv) + 6 C dk dv per chunk and head
    return (T_ // C) * H_ * (2 * C * C * (3 * dk + 2 * dv) + 6 * C * dk * dv)


# ---------------------------------------------------------------------------
class ClockSampler:
    """SM clocks and clock-event reasons sampled during a region (reads only).

    NVML through ctypes, every 2 ms, on the GPU with the same PCI bus id as the
    CUDA device; nvidia-smi every 200 ms if NVML cannot be loaded.
    """
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, dev: torch.device, interval=0.002):
        self.dev = dev
        self.interval = interval
        self.samples = []          # (sm_mhz, max_mhz, reasons bitmask)
        self.stop = threading.Event()
        self.thread = None
        self.proc = None
        self.lines = []

    def _nvml_handle(self):
        nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if nvml.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(self.dev)
        bus = getattr(props, "pci_bus_id", None)
        if bus is not None:
            busid = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), bus,
                                         getattr(props, "pci_device_id", 0))
            if nvml.nvmlDeviceGetHandleByPciBusId_v2(busid.encode(), ctypes.byref(h)) == 0:
                return nvml, h
        if nvml.nvmlDeviceGetHandleByIndex_v2(self.dev.index or 0, ctypes.byref(h)) != 0:
            raise RuntimeError("no NVML handle")
        return nvml, h

    def _run_nvml(self, nvml, h):
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        get_rs = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop.is_set():
            if nvml.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                    nvml.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 and \
                    get_rs(h, ctypes.byref(rs)) == 0:
                self.samples.append((clk.value, mx.value, rs.value))
            time.sleep(self.interval)

    def __enter__(self):
        try:
            nvml, h = self._nvml_handle()
            self.thread = threading.Thread(target=self._run_nvml, args=(nvml, h), daemon=True)
            self.thread.start()
        except Exception:
            q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap")
            try:
                self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev.index or 0}", f"--query-gpu={q}",
                                              "--format=csv,noheader,nounits", "-lms", "200"],
                                             stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.thread = threading.Thread(target=self._read_smi, daemon=True)
                self.thread.start()
            except Exception:
                self.proc = None
        time.sleep(3 * self.interval)     # first samples before the region starts
        return self

    def _read_smi(self):
        bits = [0x8, 0x40, 0x20, 0x4]
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            try:
                mask = sum(b for b, v in zip(bits, parts[2:6]) if v.lower().startswith("active"))
                self.samples.append((float(parts[0]), float(parts[1]), mask))
            except (ValueError, IndexError):
                continue

    def __exit__(self, *exc):
        time.sleep(2 * self.interval)
        self.stop.set()
        if self.proc is not None:
            self.proc.terminate()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = set()
        for _, _, m in self.samples:
            for bit, name in self.REASONS.items():
                if m & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": max(s[1] for s in self.samples), "reasons": sorted(reasons),
                "samples": len(self.samples)}


# ---------------------------------------------------------------------------
def bench_prefill(K, dev, steps, warmup, rank):
    torch.manual_seed(rank)
    S0, p, cu = I.prefill_inputs([T], H, DK, DV, dtype=torch.bfloat16, seed=100 + rank, device=dev)
    n_ck = K.kda_num_checkpoints(cu, T, STRIDE)
    page_bytes = H * DK * DV * 4
    pool = K.PagePool(page_bytes, n_ck, device=dev)
    ids = torch.tensor(pool.alloc(n_ck), dtype=torch.int32, device=dev)
    pos = torch.empty(n_ck, dtype=torch.int32, device=dev)
    o = torch.empty(T, H, DV, dtype=torch.bfloat16, device=dev)
    S_fin = torch.empty(1, H, DK, DV, dtype=torch.float32, device=dev)
    ws = torch.empty(max(K.kda_prefill_workspace_bytes(cu, T, H, DK, DV, torch.bfloat16), 16),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        K.kda_prefill_chunked(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=cu,
                              ckpt_stride=STRIDE, page_pool=pool, ckpt_page_ids=ids, ckpt_pos=pos,
                              o=o, S_final=S_fin, stream=stream, workspace=ws)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    D.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for a, b in evs:
            a.record(stream)
            step()
            b.record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
    D.barrier()
    total_ms = t0.elapsed_time(t1)
    kern_ms = [a.elapsed_time(b) for a, b in evs]
    bytes_step = prefill_bytes(T, H, DK, DV, 2, n_ck, page_bytes)

    # end to end through the C ABI from pinned host buffers: kda_prefill_chunked_host moves
    # the projections in and the outputs and final state out, segment by segment, with the
    # copies overlapping the kernels; checkpoint pages stay in the device page pool
    host_in = {n: t.to("cpu").pin_memory() for n, t in p.items()}
    host_S0 = S0.to("cpu").pin_memory()
    host_o = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    host_S = torch.empty(S_fin.shape, dtype=S_fin.dtype).pin_memory()
    scratch = torch.empty(K.kda_prefill_host_scratch_bytes(H, DK, DV, torch.bfloat16, STRIDE, E2E_SEGMENT),
                          dtype=torch.uint8, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in host_in.values()) + host_S0.numel() * 4
    d2h = host_o.numel() * 2 + host_S.numel() * 4

    def e2e_step():
        K.kda_prefill_chunked_host(host_S0, host_in["q"], host_in["k"], host_in["v"], host_in["g"],
                                   host_in["beta"], host_o, host_S, scratch, cu_seqlens=cu,
                                   ckpt_stride=STRIDE, page_pool=pool, ckpt_page_ids=ids, ckpt_pos=pos,
                                   segment_tokens=E2E_SEGMENT, stream=stream)

    for _ in range(warmup):
        e2e_step()
    torch.cuda.synchronize(dev)
    D.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    D.barrier()
    e2e_ms = e0.elapsed_time(e1)

    # the host link alone: the same bytes as one end-to-end step, one pinned-memory copy
    # per tensor (cudaMemcpyAsync through torch), host-to-device and device-to-host each
    # timed on its own with CUDA events; the two directions can run at the same time
    dev_in = {n: torch.empty_like(t, device=dev) for n, t in host_in.items()}
    dev_S0 = torch.empty_like(host_S0, device=dev)

    def h2d_copies():
        for n, t in host_in.items():
            dev_in[n].copy_(t, non_blocking=True)
        dev_S0.copy_(host_S0, non_blocking=True)

    def d2h_copies():
        host_o.copy_(o, non_blocking=True)
        host_S.copy_(S_fin, non_blocking=True)

    link = {}
    for name, fn in (("h2d", h2d_copies), ("d2h", d2h_copies)):
        for _ in range(2):
            fn()
        torch.cuda.synchronize(dev)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(steps):
            fn()
        c1.record(stream)
        torch.cuda.synchronize(dev)
        link[name] = c0.elapsed_time(c1) / steps
    return dict(total_ms=total_ms, kern_ms=kern_ms, bytes_step=bytes_step, clocks=clk.summary(),
                n_ck=n_ck, e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, link=link)


def bench_decode(K, dev, warmup=3, runs=3, layout=None):
    """Decode steps on dense (B,H,dk,dv) states, or (layout given) on B slots picked at random
    from a pool of 2B slots stored in that layout (kda_decode_step_slots)."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    n_states = DEC_B if layout is None else 2 * DEC_B
    S = (0.05 * torch.randn(n_states, H, DK, DV, generator=gen, device=dev)).contiguous()
    slots = torch.randperm(n_states, generator=gen, device=dev)[:DEC_B].to(torch.int32)
    projs = [I.decode_step_projections(DEC_B, H, DK, DV, dtype=torch.bfloat16, seed=1000 + t, device=dev)
             for t in range(DEC_STEPS)]
    o = torch.empty(DEC_B, H, DV, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def run():
        for p in projs:
            if layout is None:
                K.kda_decode_step(S, p["q"], p["k"], p["v"], p["g"], p["beta"], o=o, stream=stream)
            else:
                K.kda_decode_step_slots(S, slots, p["q"], p["k"], p["v"], p["g"], p["beta"], o=o, layout=layout,
                                        stream=stream)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(runs):
        run()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms_per_step = a.elapsed_time(b) / (runs * DEC_STEPS)
    bytes_step = 2 * DEC_B * H * DK * DV * 4 + DEC_B * H * (3 * DK + DV + 1) * 2 + DEC_B * H * DV * 2
    del S, projs
    torch.cuda.empty_cache()
    return ms_per_step, bytes_step


def _timed(fn, stream, warmup, runs):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(runs):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / runs


def bench_prologue(K, dev, warmup=3, runs=10):
    """Input prologue: kda_input_prep at the long-prefill size (T=8192, H=32, d=128, bf16,
    ShortConv w=4, SiLU) and the fused decode step at the batched-decode size (B=256)."""
    stream = torch.cuda.current_stream(dev)
    p, cu = I.prologue_inputs([T], H, DK, DV, w=CONV_W, dtype=torch.bfloat16, seed=3, device=dev)
    out = K.kda_input_prep(p["mixed"], p["weight"], p["g_logits"], p["beta_logits"], window_in=p["window"],
                           stream=stream)
    C = H * (2 * DK + DV)
    pre_ms = _timed(lambda: K.kda_input_prep(p["mixed"], p["weight"], p["g_logits"], p["beta_logits"],
                                             window_in=p["window"], out=out, stream=stream), stream, warmup, runs)
    pre_bytes = 2 * (T * C + T * H * DK + T * H) + 2 * (T * H * (3 * DK + DV) + T * H)
    del p, out
    # fused decode: raw rows + conv windows + logits in, state in place
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    S = (0.05 * torch.randn(DEC_B, H, DK, DV, generator=gen, device=dev)).contiguous()
    steps = 16
    raws = [I.prologue_inputs([1] * DEC_B, H, DK, DV, w=CONV_W, dtype=torch.bfloat16, seed=400 + t, device=dev)[0]
            for t in range(steps)]
    win = raws[0]["window"].clone()
    o = torch.empty(DEC_B, H, DV, dtype=torch.bfloat16, device=dev)

    def run():
        for r in raws:
            K.kda_decode_step_fused(S, win, r["mixed"], r["weight"], r["g_logits"], r["beta_logits"], o=o,
                                    stream=stream)
    dec_ms = _timed(run, stream, 2, 3) / steps
    dec_bytes = (2 * DEC_B * H * DK * DV * 4 + DEC_B * C * 2 + 2 * DEC_B * (CONV_W - 1) * C * 2
                 + DEC_B * H * (DK + 1) * 2 + DEC_B * H * DV * 2)
    del S, raws, win
    torch.cuda.empty_cache()
    return pre_ms, pre_bytes, dec_ms, dec_bytes


def bench_scan(K, dev, warmup=2, runs=5, T_long=65536, H_few=4):
    """One long sequence with few heads (T=65536, H=4, d=128, bf16, a checkpoint every 512
    tokens): the serial chain (kda_prefill_chunked) against the sequence-parallel prefill
    (kda_prefill_scan, pieces chosen from the SM count)."""
    S0, p, cu = I.prefill_inputs([T_long], H_few, DK, DV, dtype=torch.bfloat16, seed=9, device=dev)
    n_ck = T_long // STRIDE
    page_bytes = H_few * DK * DV * 4
    pool = K.PagePool(page_bytes, n_ck, device=dev)
    ids = torch.tensor(pool.alloc(n_ck), dtype=torch.int32, device=dev)
    o = torch.empty(T_long, H_few, DV, dtype=torch.bfloat16, device=dev)
    S_fin = torch.empty_like(S0)
    ws = torch.empty(K.kda_prefill_workspace_bytes(cu, T_long, H_few, DK, DV, torch.bfloat16), dtype=torch.uint8,
                     device=dev)
    ws_scan = torch.empty(K.kda_prefill_scan_workspace_bytes(T_long, H_few, DK, DV, torch.bfloat16, STRIDE, 0),
                          dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def serial():
        K.kda_prefill_chunked(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=cu, ckpt_stride=STRIDE,
                              page_pool=pool, ckpt_page_ids=ids, o=o, S_final=S_fin, stream=stream, workspace=ws)

    def scan():
        K.kda_prefill_scan(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], ckpt_stride=STRIDE, o=o, S_final=S_fin,
                           page_pool=pool, ckpt_page_ids=ids, segments=0, workspace=ws_scan, stream=stream)
    ms_serial = _timed(serial, stream, warmup, runs)
    ms_scan = _timed(scan, stream, warmup, runs)
    del S0, p, o, S_fin, ws, ws_scan, pool
    torch.cuda.empty_cache()
    return T_long, H_few, ms_serial, ms_scan


def bench_varlen(K, dev, warmup=1, runs=3):
    """Varlen prefix-cache resume prefill: 64 sequences, lengths log-uniform in [512, 32768]
    rounded to multiples of 64, H=32, dk=dv=128, bf16, S0 ~ N(0, 0.05), a checkpoint page
    every 512 tokens of every sequence."""
    lengths = I.varlen_lengths(64, seed=0)
    S0, p, cu = I.prefill_inputs(lengths, H, DK, DV, dtype=torch.bfloat16, seed=7, device=dev)
    Tv = cu[-1]
    n_ck = K.kda_num_checkpoints(cu, Tv, STRIDE)
    page_bytes = H * DK * DV * 4
    pool = K.PagePool(page_bytes, n_ck, device=dev)
    ids = torch.tensor(pool.alloc(n_ck), dtype=torch.int32, device=dev)
    o = torch.empty(Tv, H, DV, dtype=torch.bfloat16, device=dev)
    S_fin = torch.empty_like(S0)
    ws = torch.empty(max(K.kda_prefill_workspace_bytes(cu, Tv, H, DK, DV, torch.bfloat16), 16),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        K.kda_prefill_chunked(S0, p["q"], p["k"], p["v"], p["g"], p["beta"], cu_seqlens=cu, ckpt_stride=STRIDE,
                              page_pool=pool, ckpt_page_ids=ids, o=o, S_final=S_fin, stream=stream, workspace=ws)
    for _ in range(warmup):
        call()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(runs):
        call()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / runs
    nbytes = prefill_bytes(Tv, H, DK, DV, 2, n_ck, page_bytes, n_seqs=len(lengths))
    del S0, p, o, S_fin, ws, pool
    torch.cuda.empty_cache()
    return ms, Tv, len(lengths), n_ck, nbytes


def bench_replay(K, dev, warmup=3, runs=5):
    sets = []
    n_bytes = 0
    for i in range(REP_SETS):
        S, proj, n_acc = I.replay_inputs(REP_B, REP_H, REP_D, REP_D, REP_DRAFT, dtype=torch.float32,
                                         seed=i, device=dev, state_std=0.1)
        n_acc = n_acc.to(dev)
        S_new = torch.empty_like(S)
        out = torch.empty(REP_B, REP_H, REP_DRAFT, REP_D, device=dev)
        sets.append((S, proj, n_acc, S_new, out))
        acc = int(n_acc.sum())
        n_bytes += 2 * S.numel() * 4 + acc * REP_H * (3 * REP_D + REP_D + 1) * 4 + out.numel() * 4
    stream = torch.cuda.current_stream(dev)

    def call(s):
        S, pr, n_acc, S_new, out = s
        K.kda_verify_replay(S, pr.q, pr.k, pr.v, pr.g, pr.beta, n_acc, S_new=S_new, out=out, stream=stream)

    for _ in range(warmup):
        for s in sets:
            call(s)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(runs):
        for s in sets:
            call(s)
    b.record(stream)
    torch.cuda.synchronize(dev)
    amort_ms = a.elapsed_time(b) / (runs * REP_SETS)
    # the same 64 calls captured once in a CUDA graph: one launch replays them all,
    # so the per-call figure is the kernels' own time on states that miss L2
    graph_ms = None
    try:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            for s in sets:                 # warm the capture stream once
                K.kda_verify_replay(s[0], s[1].q, s[1].k, s[1].v, s[1].g, s[1].beta, s[2], S_new=s[3], out=s[4],
                                    stream=cap)
        cap.synchronize()
        with torch.cuda.graph(g, stream=cap):
            for s in sets:
                K.kda_verify_replay(s[0], s[1].q, s[1].k, s[1].v, s[1].g, s[1].beta, s[2], S_new=s[3], out=s[4],
                                    stream=cap)
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize(dev)
        x, y = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x.record(stream)
        for _ in range(runs):
            g.replay()
        y.record(stream)
        torch.cuda.synchronize(dev)
        graph_ms = x.elapsed_time(y) / (runs * REP_SETS)
    except Exception as e:                 # capture unsupported: report the stream figure only
        print(f"replay graph capture failed: {e}", file=sys.stderr)
    # the same 64 states as the KDA layers of one model: one launch replays them all
    # (each layer its own state and draft projections, the accepted counts shared)
    layers_ms, layers_bytes = None, None
    try:
        n_acc = sets[0][2]
        S_l = torch.stack([s_[0] for s_ in sets])
        pj = {nm: torch.stack([getattr(s_[1], nm) for s_ in sets]) for nm in ("q", "k", "v", "g", "beta")}
        S_lnew = torch.empty_like(S_l)
        out_l = torch.empty(REP_SETS, REP_B, REP_H, REP_DRAFT, REP_D, device=dev)
        acc = int(n_acc.sum())
        layers_bytes = REP_SETS * (2 * sets[0][0].numel() * 4 + acc * REP_H * (3 * REP_D + REP_D + 1) * 4
                                   + sets[0][4].numel() * 4)

        def call_layers():
            K.kda_verify_replay_layers(S_l, pj["q"], pj["k"], pj["v"], pj["g"], pj["beta"], n_acc,
                                       S_new=S_lnew, out=out_l, stream=stream)
        for _ in range(warmup):
            call_layers()
        torch.cuda.synchronize(dev)
        x, y = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x.record(stream)
        for _ in range(runs):
            call_layers()
        y.record(stream)
        torch.cuda.synchronize(dev)
        layers_ms = x.elapsed_time(y) / runs
        del S_l, pj, S_lnew, out_l
    except Exception as e:
        print(f"layered replay failed: {e}", file=sys.stderr)
    single = []
    for s in sets[:16]:
        x, y = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x.record(stream)
        call(s)
        y.record(stream)
        torch.cuda.synchronize(dev)
        single.append(x.elapsed_time(y))
    return amort_ms, n_bytes / REP_SETS, statistics.median(single), graph_ms, (layers_ms, layers_bytes)


# ---------------------------------------------------------------------------
def oracle_sample(heads=2, tokens=T):
    """fp64 oracle on `heads` heads x `tokens` tokens of the workload's input distribution.

    Returns (tokens/s scaled to all H heads, seconds, threads used)."""
    from oracle import kda_oracle as O
    S0, p, cu = I.prefill_inputs([tokens], heads, DK, DV, dtype=torch.bfloat16, seed=100)
    f = I.to_f64_numpy
    args = [f(S0)] + [f(p[n]) for n in ("q", "k", "v", "g", "beta")]
    t0 = time.perf_counter()
    O.prefill_chunked(*args, cu_seqlens=cu, chunk=CHUNK, ckpt_stride=STRIDE)
    dt = time.perf_counter() - t0
    return tokens * heads / H / dt, dt, 1


def run_reference(args, rank, world):
    """The fp64 oracle as it stands, one bounded sample per step: 1 head x 2048 tokens."""
    if rank != 0:
        return
    for _ in range(args.warmup):
        oracle_sample(heads=1, tokens=2048)
    vals, secs = [], []
    for _ in range(args.steps):
        v, dt, threads = oracle_sample(heads=1, tokens=2048)
        vals.append(v)
        secs.append(dt)
    value = len(vals) / sum(1.0 / v for v in vals)
    line = {
        "impl": "reference", "metric": "kda_prefill_tokens_per_s", "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * statistics.mean(secs), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": 1, "seq_len": T, "l2": "host memory"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"per step 1 of {H} heads x 2048 of {T} tokens; tokens/s scaled by "
                                   f"the {H} heads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="skip the decode / replay objects")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    rank, world, local = D.init()
    if args.impl == "reference":
        run_reference(args, rank, world)
        D.finalize()
        return
    args.warmup = max(args.warmup, 3)
    from kda_delta_rule_gb300 import kda as K
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    r = bench_prefill(K, dev, args.steps, args.warmup, rank)
    t_max = D.max_over_ranks(r["total_ms"])
    e2e_max = D.max_over_ranks(r["e2e_ms"])
    tokens_all = T * world * args.steps
    value = tokens_all / (t_max / 1e3)
    hbm, tf, src = peaks()
    kern_avg_ms = sum(r["kern_ms"]) / len(r["kern_ms"])
    achieved = r["bytes_step"] / (kern_avg_ms / 1e3) / 1e9
    flops = prefill_flops(T, H, DK, DV)
    extras = {}
    if not args.no_extras:
        dms, dbytes = bench_decode(K, dev)
        dgbs = dbytes / (dms / 1e3) / 1e9
        extras["decode"] = {"workload": f"B={DEC_B} H={H} dk=dv={DK} fp32 state, bf16 projections, "
                                        f"{DEC_STEPS} consecutive steps",
                            "ms_per_step": dms, "state_GBps": dgbs, "hbm_frac": dgbs / hbm,
                            "bytes_per_step": dbytes, "tokens_per_s": DEC_B / (dms / 1e3)}
        for name, lay in (("kv", K.LAYOUT_KV), ("vk", K.LAYOUT_VK)):
            sms, sbytes = bench_decode(K, dev, layout=lay)
            sgbs = sbytes / (sms / 1e3) / 1e9
            extras["decode"][f"slots_{name}"] = {
                "workload": f"the same steps on {DEC_B} of {2 * DEC_B} slots of a state pool stored "
                            + ("(dk, dv)" if name == "kv" else "transposed, (dv, dk)")
                            + ", kda_decode_step_slots",
                "ms_per_step": sms, "state_GBps": sgbs, "hbm_frac": sgbs / hbm}
        pms, pbytes, fms, fbytes = bench_prologue(K, dev)
        extras["prologue"] = {
            "workload": f"kda_input_prep: T={T} H={H} dk=dv={DK} bf16, ShortConv w={CONV_W}, SiLU, L2Norm, "
                        "gates from logits",
            "ms_per_call": pms, "algorithmic_bytes": pbytes, "achieved_GBps": pbytes / (pms / 1e3) / 1e9,
            "hbm_frac": pbytes / (pms / 1e3) / 1e9 / hbm,
            "decode_fused": {
                "workload": f"kda_decode_step_fused: B={DEC_B} H={H} dk=dv={DK} bf16 raw rows, w={CONV_W}, "
                            "fp32 state in place",
                "ms_per_step": fms, "bytes_per_step": fbytes, "achieved_GBps": fbytes / (fms / 1e3) / 1e9,
                "hbm_frac": fbytes / (fms / 1e3) / 1e9 / hbm}}
        ams, abytes, single_ms, graph_ms, (layers_ms, layers_bytes) = bench_replay(K, dev)
        agbs = abytes / (ams / 1e3) / 1e9
        extras["replay"] = {"workload": f"B={REP_B} H={REP_H} dk=dv={REP_D} draft={REP_DRAFT} fp32, "
                                        f"n_accepted~U{{0..8}}, {REP_SETS} distinct buffer sets",
                            "ms_per_call_amortised": ams, "ms_per_call_single": single_ms,
                            "state_GBps": agbs, "hbm_frac": agbs / hbm, "bytes_per_call": abytes}
        if graph_ms:
            ggbs = abytes / (graph_ms / 1e3) / 1e9
            extras["replay"].update({"ms_per_call_cuda_graph": graph_ms, "state_GBps_cuda_graph": ggbs,
                                     "hbm_frac_cuda_graph": ggbs / hbm})
        if layers_ms:
            lgbs = layers_bytes / (layers_ms / 1e3) / 1e9
            extras["replay"]["layers_batched"] = {
                "workload": f"the {REP_SETS} buffer sets as {REP_SETS} stacked KDA layers of one model, "
                            "one kda_verify_replay_layers launch",
                "ms_per_launch": layers_ms, "ms_per_layer": layers_ms / REP_SETS,
                "bytes_per_launch": layers_bytes, "state_GBps": lgbs, "hbm_frac": lgbs / hbm}
        sT, sH, s_serial, s_scan = bench_scan(K, dev)
        extras["scan"] = {
            "workload": f"one sequence T={sT} H={sH} dk=dv={DK} bf16, ckpt every {STRIDE}: serial chain "
                        "(kda_prefill_chunked) vs sequence-parallel (kda_prefill_scan, pieces from the SM count)",
            "ms_serial": s_serial, "ms_scan": s_scan, "speedup": s_serial / s_scan,
            "tokens_per_s_scan": sT / (s_scan / 1e3)}
        vms, vtok, vseq, vck, vbytes = bench_varlen(K, dev)
        vgbs = vbytes / (vms / 1e3) / 1e9
        extras["varlen"] = {"workload": f"{vseq} sequences, lengths log-uniform in [512, 32768] rounded to 64 "
                                        f"({vtok} tokens), H={H} dk=dv={DK} bf16, S0 ~ N(0,0.05), "
                                        f"ckpt every {STRIDE} ({vck} pages)",
                            "ms_per_call": vms, "tokens_per_s": vtok / (vms / 1e3),
                            "algorithmic_bytes": vbytes, "achieved_GBps": vgbs, "hbm_frac": vgbs / hbm}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, threads = oracle_sample(heads=2)
        cpu = {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"2 of {H} heads, all {T} tokens ({dt:.1f} s of fp64 CPU work), scaled by {H // 2}"}
    if rank == 0:
        line = {
            "metric": "kda_prefill_tokens_per_s", "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": world, "seq_len": T,
                       "parallelism": f"replicas{world}", "l2": "inputs larger than L2 (336 MB/step)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": prefill_traffic(), "peak_source": src,
                         "kernel": "kda_prefill (chunk prep + chain kernels of one call)",
                         "kernel_ms": kern_avg_ms,
                         "algorithmic_bytes": r["bytes_step"],
                         "tc_tflops": flops / (kern_avg_ms / 1e3) / 1e12,
                         "tc_frac": flops / (kern_avg_ms / 1e3) / 1e12 / tf},
            "e2e": {"value": T * world * args.steps / (e2e_max / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                    "ms_per_step": e2e_max / args.steps,
                    # plain pinned copies of the same bytes: the bound the host link sets on e2e
                    "host_link": {"h2d_ms": r["link"]["h2d"], "d2h_ms": r["link"]["d2h"],
                                  "h2d_GBps": r["h2d"] / (r["link"]["h2d"] / 1e3) / 1e9,
                                  "d2h_GBps": r["d2h"] / (r["link"]["d2h"] / 1e3) / 1e9,
                                  "bound_tokens_per_s": T / (max(r["link"]["h2d"], r["link"]["d2h"]) / 1e3)}},
            "gpu_launches": PREFILL_KERNELS_PER_CALL * args.steps,
            "clocks": r["clocks"],
            "cpu_baseline": cpu,
            **extras,
        }
        print(json.dumps(line))
    D.finalize()


if __name__ == "__main__":
    main()
