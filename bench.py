"""Benchmark of the ring AllReduce over N virtual ranks on one GB300.

Headline workload: N=8 virtual ranks, ring order = seeded permutation (seed
3), f32 sum, 64 MiB per rank of normal(0,1) values, 12 channels (mask 0xFFF),
Simple protocol with a 1 MiB FIFO buffer and 4 chunk steps. One step = one
rar_allreduce call (one cooperative launch that runs every rank and channel).

Metric: busBW = (S / t) * 2(N-1)/N in GB/s (1 GB = 1e9 B), S = bytes per rank.
The JSON line also carries the sweep the metric is quoted "vs size per proto"
on: every protocol at 64 MiB, LL at 4 KiB, the one-shot variant, each with its
HBM-roofline fraction.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
With --gpus N > 1 (launched under torchrun) every GPU runs an independent
replica of the workload (the method keeps all ranks on one GPU: replicas
only); value = the sum over GPUs of bytes moved / the slowest GPU's time.
--impl reference times the CPU oracle on the host cores instead.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ring AllReduce busBW"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0

# Per-launch DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of the
# headline kernel from one ncu capture of this workload, and a hash of the
# kernel sources it was captured with: when the sources differ (the kernel
# changed since the capture) the line reports traffic null.
TRAFFIC_BYTES_PER_LAUNCH = 1789786368
TRAFFIC_SOURCES_SHA16 = "c27d2b349b90b797"
TRAFFIC_SOURCES = ("ring_simple.cu", "rar_device.cuh", "rar_geometry.h")


def kernel_sources_sha16():
    import hashlib
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "collective_communication_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def headline_case(args=None):
    """The headline workload, or a variant of it named on the command line
    (used to profile smaller cases of the same kernels)."""
    from collective_communication_gb300 import inputs as gen
    nranks = getattr(args, "nranks", None) or 8
    ring = gen.ring_permutation(nranks, 3)
    kib = getattr(args, "kib", None) or 1024 * (getattr(args, "mib", None) or 64)
    proto = getattr(args, "proto", None) or gen.SIMPLE
    buff = getattr(args, "buff_size", None)
    if buff is None:
        buff = gen.MIB if proto == gen.SIMPLE else 0
    chans = getattr(args, "channels", None) or 12
    dtype = getattr(args, "dtype", None) or gen.F32
    size = f"{kib // 1024}MiB" if kib % 1024 == 0 else f"{kib}KiB"
    name = f"n{nranks}_{dtype}_{size}_ch{chans}_{proto}{buff // 1024 if buff else 'default'}"
    return gen.RingCase(name, nranks, ring, (1 << chans) - 1, proto, kib * gen.KIB // (4 if dtype == gen.F32 else 2),
                        dtype, "normal", 3, buff, 4)


def size_label(nbytes):
    return f"{nbytes >> 20} MiB" if nbytes % (1 << 20) == 0 else f"{nbytes >> 10} KiB"


def busbw(nbytes_per_rank, nranks, seconds):
    return nbytes_per_rank / seconds * 2 * (nranks - 1) / nranks / 1e9


def wire_factor(proto):
    return {"Simple": 1.0, "LL128": 16.0 / 15.0, "LL": 2.0}[proto]


def algorithmic_bytes(case, direct=False):
    """Ideal bytes of one call: every rank reads its input and writes its output
    once (N * 2S), plus each FIFO byte written once and read once, 2(N-1)/N * S
    per rank on the wire (LL doubles it, LL128 adds 1/15). bf16 partial sums
    cross the reduce-scatter half as binary32. Direct all-gather: only the
    reduce-scatter half uses the FIFO; each rank reads back the (N-2) chunks it
    forwards from its own output."""
    n = case.nranks
    s = case.count * (4 if case.dtype == "f32" else 2)
    w = wire_factor(case.proto)
    rs = (n - 1) / n * s * (2 if case.dtype == "bf16" else 1) * w
    ag = (n - 1) / n * s * w
    if direct:
        return n * 2 * s + n * 2 * rs + n * (n - 2) / n * s
    return n * 2 * s + n * 2 * (rs + ag)


def half_algorithmic_bytes(kind, n, block, dtype, proto, direct=False):
    """Ideal bytes of one ReduceScatter ("rs") or AllGather ("ag") call with
    blocks of `block` elements: every rank reads its input and writes its
    output once (n+1 blocks), plus each FIFO byte written once and read once,
    (n-1) blocks per rank on the wire (partial sums as binary32 for
    ReduceScatter; LL doubles, LL128 adds 1/15). Direct AllGather: no FIFO;
    the output blocks are written once (n-1 of them by the previous rank) and
    each rank reads back the (n-2) blocks it forwards."""
    eb = 4 if dtype == "f32" else 2
    m = block * eb
    w = wire_factor(proto)
    if kind == "ag" and direct:
        return n * (2 * n - 1) * m
    hop = block * 4 if kind == "rs" else m
    return n * (n + 1) * m + 2 * n * (n - 1) * hop * w


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while running. `load`
    (seconds -> None), if given, keeps the GPU busy with untimed work for the
    lead-in and lead-out of the sampling, so that the samples next to a short
    timed region are taken under load rather than at idle."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, load=None):
        self.index = index
        self.proc = None
        self.load = load

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        (self.load or time.sleep)(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            (self.load or time.sleep)(0.3)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def rows_like(x, torch):
    """An uninitialised [nranks, count] tensor like x whose rows start on
    256-byte boundaries (the ABI wants 16-byte aligned rank buffers; a ragged
    count would misalign every row after the first in a dense tensor)."""
    n, count = x.shape
    stride = -(-count // 128) * 128
    return torch.empty((n, stride), dtype=x.dtype, device=x.device)[:, :count]


def device_inputs(case, torch):
    g = torch.Generator(device="cuda")
    g.manual_seed(case.seed)
    x = torch.randn((case.nranks, case.count), generator=g, device="cuda", dtype=torch.float32)
    if case.dtype == "bf16":
        x = x.to(torch.bfloat16)
    y = rows_like(x, torch)
    y.copy_(x)
    return y


def time_ring(case, torch, B, steps, warmup, direct=False):
    """Device time per call (CUDA events on the launching stream)."""
    x = device_inputs(case, torch)
    y = rows_like(x, torch)
    send = [x[r] for r in range(case.nranks)]
    recv = [y[r] for r in range(case.nranks)]
    ws = B.Workspace(case.nranks, case.mask, case.proto, case.buff_size)
    stream = torch.cuda.current_stream()
    def call():
        B.allreduce_ex(send, recv, case.ring, case.mask, case.proto, ws, case.buff_size, case.chunk_steps,
                       direct=direct)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    st = B.get_status(ws)
    if st != B.Status.OK:
        raise RuntimeError(f"{case.name}: device status {st.name}")
    ms = [a.elapsed_time(b) for a, b in ev]
    del x, y, ws
    return ms


def time_half(kind, n, block, ring, mask, proto, buff_size, chunk_steps, torch, B, steps, warmup, direct=False,
              dtype="f32"):
    """Device time per ReduceScatter / AllGather call (CUDA events)."""
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    big = torch.randn((n, n * block), generator=g, device="cuda", dtype=torch.float32).to(tdt)
    small = torch.randn((n, block), generator=g, device="cuda", dtype=torch.float32).to(tdt)
    ws = B.Workspace(n, mask, proto, buff_size)
    if kind == "rs":
        send, recv = [big[r] for r in range(n)], [small[r] for r in range(n)]
        call = lambda: B.reduce_scatter(send, recv, ring, mask, proto, ws, buff_size, chunk_steps)  # noqa: E731
    else:
        send, recv = [small[r] for r in range(n)], [big[r] for r in range(n)]
        call = lambda: B.all_gather(send, recv, ring, mask, proto, ws, buff_size, chunk_steps,  # noqa: E731
                                    direct=direct)
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    st = B.get_status(ws)
    if st != B.Status.OK:
        raise RuntimeError(f"{kind}: device status {st.name}")
    ms = [a.elapsed_time(b) for a, b in ev]
    del big, small, ws
    return ms


def sweep(torch, B, steps, warmup, peak):
    from collective_communication_gb300 import inputs as gen
    out = {}
    cases = gen.large_cases()
    cases.append(gen.RingCase("n8_ll_ch12_64MiB", 8, cases[0].ring, 0xFFF, gen.LL, 64 * gen.MIB // 4,
                              gen.F32, "normal", 3, 0, 4))
    runs = [(c, False) for c in cases] + [(c, True) for c in cases if c.proto == gen.SIMPLE]
    for c, direct in runs:
        ms = time_ring(c, torch, B, steps, warmup, direct)
        t = statistics.median(ms) / 1e3
        out[c.name + ("_direct_allgather" if direct else "")] = {
            "busbw_gbs": round(busbw(c.bytes_per_rank, c.nranks, t), 2),
            "us": round(t * 1e6, 1),
            "roofline_frac": round(algorithmic_bytes(c, direct) / t / 1e9 / peak, 3),
            "user_bytes_frac": round(c.nranks * 2 * c.bytes_per_rank / t / 1e9 / peak, 3)}
    # the 64 MiB workload on 1 to 19 contiguous channels (N x C blocks, one per SM;
    # 19 x 8 = 152 uses every SM): how the ring scales with the SMs it runs on
    scaling = {}
    for proto, bs in ((gen.SIMPLE, gen.MIB), (gen.LL128, 0)):
        for nch in (1, 2, 4, 8, 12, 16, 19):
            c = gen.RingCase(f"n8_{proto}_ch{nch}", 8, cases[0].ring, (1 << nch) - 1, proto, 64 * gen.MIB // 4,
                             gen.F32, "normal", 3, bs, 4)
            t = statistics.median(time_ring(c, torch, B, max(3, steps // 2), 2)) / 1e3
            scaling.setdefault(proto, {})[f"ch{nch}"] = {
                "busbw_gbs": round(busbw(c.bytes_per_rank, c.nranks, t), 2), "us": round(t * 1e6, 1),
                "roofline_frac": round(algorithmic_bytes(c) / t / 1e9 / peak, 3)}
    out["channel_scaling_n8_64MiB"] = scaling
    # the halves: N=8, 12 channels, the headline's ring, 8 MiB f32 blocks (the
    # 64 MiB per-rank buffer of the AllReduce); busBW = n*block bytes / t *
    # (N-1)/N, the usual convention for these collectives
    hc = cases[0]
    block = 64 * gen.MIB // 4 // 8
    for kind, proto, bs, direct in (("rs", "Simple", gen.MIB, False), ("ag", "Simple", gen.MIB, False),
                                    ("ag", "Simple", gen.MIB, True), ("rs", "LL128", 0, False),
                                    ("ag", "LL128", 0, False)):
        ms = time_half(kind, 8, block, hc.ring, 0xFFF, proto, bs, 4, torch, B, steps, warmup, direct)
        t = statistics.median(ms) / 1e3
        name = {"rs": "reduce_scatter", "ag": "all_gather"}[kind]
        tag = f"{proto.lower()}{bs // gen.KIB}k" if bs else proto.lower()
        total = 8 * block * 4
        out[f"n8_{name}_{tag}_ch12_64MiB" + ("_direct" if direct else "")] = {
            "busbw_gbs": round(total / t * 7 / 8 / 1e9, 2),
            "us": round(t * 1e6, 1),
            "roofline_frac": round(half_algorithmic_bytes(kind, 8, block, "f32", proto, direct) / t / 1e9 / peak, 3)}
    # 512 KiB per rank, N=4, ring 0-2-3-1: every protocol on 1, 4 and 12
    # channels (Simple with a 1 MiB buffer); device time per call from a CUDA
    # graph of back-to-back calls, and busBW from it
    s512 = {}
    for c in gen.sweep_512k_cases():
        t = graph_latency_ring(c, torch, B) / 1e6
        s512[c.name] = {"us": round(t * 1e6, 2), "busbw_gbs": round(busbw(c.bytes_per_rank, c.nranks, t), 2),
                        "roofline_frac": round(algorithmic_bytes(c) / t / 1e9 / peak, 3)}
    # the same workload on 12 channels with a ring per channel: the six N=4
    # rings through rank 0 listed for channels 0-5 and repeated on 6-11 in
    # the channel-parallel page's 12-channel graph
    six = [[0, 1, 2, 3], [0, 1, 3, 2], [0, 2, 3, 1], [0, 2, 1, 3], [0, 3, 1, 2], [0, 3, 2, 1]]
    for c in gen.sweep_512k_cases():
        if c.mask != 0xFFF:
            continue
        c.ring = six + six
        c.name = c.name.replace("_ch12_", "_ch12_page_rings_")
        t = graph_latency_ring(c, torch, B) / 1e6
        s512[c.name] = {"us": round(t * 1e6, 2), "busbw_gbs": round(busbw(c.bytes_per_rank, c.nranks, t), 2),
                        "roofline_frac": round(algorithmic_bytes(c) / t / 1e9 / peak, 3)}
    out["n4_ring0231_512KiB_f32"] = s512
    # small messages: 4 KiB per rank, N=4, ring 0-2-3-1, one channel. Device
    # latency from a CUDA graph of back-to-back calls (no host enqueue time),
    # and the stream-launch latency as seen between two events.
    for proto in ("LL", "LL128", "Simple"):
        c = gen.small_case()
        c.proto = proto
        c.buff_size = 64 * gen.KIB if proto == "Simple" else 0
        ms = time_ring(c, torch, B, max(steps, 20), warmup)
        out[f"n4_{proto}_ch1_4KiB"] = {"stream_latency_us": round(statistics.median(ms) * 1e3, 2),
                                       "graph_latency_us": graph_latency_ring(c, torch, B)}
    # busBW and roofline fraction vs size per protocol and type: N=8, seeded
    # ring (seed 5), the sparse 8-channel mask 0b101101011011, 1 KiB * 4^k per
    # rank up to 1 GiB with the uneven counts 8 * chunk * k + 13 of that
    # workload; small sizes timed from a CUDA graph (device time only)
    def chunk_elems_of(proto, dtype):
        dt = B.Dtype.F32 if dtype == gen.F32 else B.Dtype.BF16
        return B.describe_geometry(8, 1 << 20, dt, gen.SPARSE_MASK, proto, 0, 4)["chunk_elems"]

    sizes = {}
    for c in gen.sparse_sweep_cases(chunk_elems_of, max_bytes=1 << 30):
        label = c.name.rsplit("_", 1)[1]  # the nominal size per rank
        if c.bytes_per_rank <= 4 * gen.MIB:
            t = graph_latency_ring(c, torch, B) / 1e6
        else:
            t = statistics.median(time_ring(c, torch, B, 3 if c.bytes_per_rank >= 256 * gen.MIB else 5, 2)) / 1e3
        sizes.setdefault(c.dtype, {}).setdefault(c.proto, {})[label] = {
            "count": c.count, "busbw_gbs": round(busbw(c.bytes_per_rank, 8, t), 2), "us": round(t * 1e6, 2),
            "roofline_frac": round(algorithmic_bytes(c) / t / 1e9 / peak, 3)}
    out["size_sweep_n8_sparse_mask_default_buffers"] = sizes
    # one-shot bf16, N=8, 7168 x {1, 512}, and the 4 KiB latency point (2048 bf16 per rank)
    for case in (gen.oneshot_cases()[0], gen.oneshot_cases()[-1],
                 gen.OneShotCase("oneshot_bf16_n8_4KiB", 8, 2048, gen.BF16, "normal", 1)):
        x = device_inputs(gen.RingCase(case.name, case.nranks, [], 0, "", case.count, case.dtype, "normal",
                                       case.seed), torch)
        y = rows_like(x, torch)
        send = [x[r] for r in range(case.nranks)]
        recv = [y[r] for r in range(case.nranks)]
        for _ in range(warmup):
            B.oneshot(send, recv)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(max(steps, 20))]
        s = torch.cuda.current_stream()
        for a, b in ev:
            a.record(s)
            B.oneshot(send, recv)
            b.record(s)
        torch.cuda.synchronize()
        t = statistics.median([a.elapsed_time(b) for a, b in ev]) / 1e3
        nbytes = case.count * 2
        gl = graph_latency(lambda: B.oneshot(send, recv), torch)
        tg = gl * 1e-6 if gl else t
        out[case.name] = {"stream_us": round(t * 1e6, 2), "graph_us": gl,
                          "unique_bytes_frac": round(2 * case.nranks * nbytes / tg / 1e9 / peak, 3)}
        # the staged form (copy into slots, sequence numbers, reduce): unique
        # bytes 4 * N * S (the copy's read and write added to the direct form's)
        ws = B.OneShotWorkspace(case.nranks, case.count, "bf16")
        for _ in range(warmup):
            B.oneshot_staged(send, recv, ws)
        torch.cuda.synchronize()
        for a, b in ev:
            a.record(s)
            B.oneshot_staged(send, recv, ws)
            b.record(s)
        torch.cuda.synchronize()
        if B.get_status(ws) != B.Status.OK:
            raise RuntimeError("staged one-shot: device status")
        t = statistics.median([a.elapsed_time(b) for a, b in ev]) / 1e3
        gl = graph_latency(lambda: B.oneshot_staged(send, recv, ws), torch)
        tg = gl * 1e-6 if gl else t
        out[case.name + "_staged"] = {"stream_us": round(t * 1e6, 2), "graph_us": gl,
                                      "unique_bytes_frac": round(4 * case.nranks * nbytes / tg / 1e9 / peak, 3)}
        del ws
    return out


def graph_latency(call, torch, reps=50):
    """Per-call device time of `reps` back-to-back calls captured in one CUDA
    graph (no host enqueue gaps). None if the capture is refused."""
    try:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(3):
                call()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                call()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        return round(a.elapsed_time(b) * 1e3 / reps, 2)
    except Exception as e:  # capture not possible: report the reason instead of a number
        sys.stderr.write(f"graph capture failed: {e}\n")
        return None


def graph_latency_ring(case, torch, B):
    x = device_inputs(case, torch)
    y = rows_like(x, torch)
    send = [x[r] for r in range(case.nranks)]
    recv = [y[r] for r in range(case.nranks)]
    ws = B.Workspace(case.nranks, case.mask, case.proto, case.buff_size)
    lat = graph_latency(lambda: B.allreduce_ex(send, recv, case.ring, case.mask, case.proto, ws, case.buff_size,
                                               case.chunk_steps), torch)
    if B.get_status(ws) != B.Status.OK:
        raise RuntimeError("graph replay: device status not OK")
    return lat


def e2e_ring(case, torch, B, steps, warmup):
    """The same call measured end to end from pinned host buffers, through the
    public API: every step copies all ranks' inputs host->device, runs the
    AllReduce and copies every rank's output back device->host. Two device
    buffer sets and three streams pipeline consecutive steps, so step k's
    host->device copy overlaps step k-1's device->host copy (the two
    directions of the host link run at once); the AllReduce calls stay ordered
    on one stream and share one workspace."""
    x = device_inputs(case, torch)
    host_in = x.cpu().pin_memory()
    host_out = [torch.empty_like(host_in).pin_memory() for _ in range(2)]
    dx = [rows_like(x, torch) for _ in range(2)]
    dy = [rows_like(x, torch) for _ in range(2)]
    ws = B.Workspace(case.nranks, case.mask, case.proto, case.buff_size)
    s_h2d, s_cmp, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    h2d_done = [ev(), ev()]
    cmp_done = [ev(), ev()]
    d2h_done = [ev(), ev()]
    for e in cmp_done + d2h_done:
        e.record(torch.cuda.current_stream())

    def one(k):
        b = k % 2
        s_h2d.wait_event(cmp_done[b])  # dx[b] no longer read by step k-2
        with torch.cuda.stream(s_h2d):
            dx[b].copy_(host_in, non_blocking=True)
        h2d_done[b].record(s_h2d)
        s_cmp.wait_event(h2d_done[b])
        s_cmp.wait_event(d2h_done[b])  # dy[b] already copied out by step k-2
        B.allreduce([dx[b][r] for r in range(case.nranks)], [dy[b][r] for r in range(case.nranks)], case.ring,
                    case.mask, case.proto, ws, case.buff_size, case.chunk_steps, stream=s_cmp)
        cmp_done[b].record(s_cmp)
        s_d2h.wait_event(cmp_done[b])
        with torch.cuda.stream(s_d2h):
            host_out[b].copy_(dy[b], non_blocking=True)
        d2h_done[b].record(s_d2h)

    for k in range(warmup):
        one(k)
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(cur)
    for s_ in (s_h2d, s_cmp, s_d2h):
        s_.wait_event(start)
    for k in range(warmup, warmup + steps):
        one(k)
    for s_ in (s_h2d, s_cmp, s_d2h):
        cur.wait_stream(s_)
    end.record(cur)
    torch.cuda.synchronize()
    if B.get_status(ws) != B.Status.OK:
        raise RuntimeError("e2e: device status not OK")
    last = (warmup + steps - 1) % 2
    if not torch.equal(host_out[last].view(torch.int32)[0], host_out[last].view(torch.int32)[1]):
        raise RuntimeError("e2e: ranks 0 and 1 returned different results")
    t = start.elapsed_time(end) / 1e3 / steps
    nbytes = case.nranks * case.bytes_per_rank
    return {"value": round(busbw(case.bytes_per_rank, case.nranks, t), 2), "unit": UNIT,
            "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes, "ms_per_step": round(t * 1e3, 3),
            "pipelining": "2 buffer sets; step k host->device overlaps step k-1 device->host"}


def cpu_baseline(case, budget_s=10.0):
    """The CPU oracle's step-by-step simulation of the headline call (full
    size, same inputs recipe), single-threaded, best of the runs that fit in
    about budget_s seconds (at least one, at most 25)."""
    import oracle
    from collective_communication_gb300 import inputs as gen
    x = gen.draw("normal", case.nranks, case.count, case.seed, case.dtype)
    oracle.lib()
    times = []
    t_end = time.time() + budget_s
    while True:
        t0 = time.perf_counter()
        oracle.ring_allreduce_sim(list(x), case.ring, case.mask, oracle.SIMPLE, case.buff_size, case.chunk_steps)
        times.append(time.perf_counter() - t0)
        if time.time() > t_end or len(times) >= 25:
            break
    t = min(times)
    return {"value": round(busbw(case.bytes_per_rank, case.nranks, t), 4), "unit": UNIT, "cores": 1,
            "kind": "oracle",
            "sample": f"the whole headline call (8 ranks x 64 MiB f32) through the oracle's step-by-step "
                      f"simulation, best of {len(times)}, 1 thread; host has {os.cpu_count()} cores",
            "seconds_per_call": round(t, 3)}


def combine_replicas(total_ms, steps, bytes_per_rank, nranks, world, dist=None, device="cpu"):
    """Whole-job figures over `world` independent replicas (one per GPU): the
    time is the slowest replica's (max over ranks); the throughput is the
    bytes of all replicas over that time, as busBW. Returns (ms_per_step,
    value)."""
    if dist is not None and world > 1:
        import torch
        t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / steps
    return ms_per_step, busbw(bytes_per_rank, nranks, ms_per_step / 1e3) * world


def run_gpu(args):
    import torch
    import torch.distributed as dist
    from collective_communication_gb300 import binding as B

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    B.load_library()
    peak, peak_kind = measured_peak()
    case = headline_case(args)

    x = device_inputs(case, torch)
    y = rows_like(x, torch)
    send = [x[r] for r in range(case.nranks)]
    recv = [y[r] for r in range(case.nranks)]
    ws = B.Workspace(case.nranks, case.mask, case.proto, case.buff_size)
    stream = torch.cuda.current_stream()

    def step():
        B.allreduce(send, recv, case.ring, case.mask, case.proto, ws, case.buff_size, case.chunk_steps)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    per = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    def busy(seconds):
        """Untimed calls on the same buffers while nvidia-smi samples around
        the timed region (counted in no figure)."""
        t_end = time.time() + seconds
        while time.time() < t_end:
            for _ in range(8):
                step()
            torch.cuda.synchronize()

    with ClockSampler(local, load=busy) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for a, b in per:
            a.record(stream)
            step()
            b.record(stream)
        end.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
    st = B.get_status(ws)
    if st != B.Status.OK:
        raise RuntimeError(f"device status {st.name}")
    total_ms = start.elapsed_time(end)
    launch_ms = [a.elapsed_time(b) for a, b in per]
    ms_per_step, value = combine_replicas(total_ms, args.steps, case.bytes_per_rank, case.nranks, world,
                                          dist if world > 1 else None, "cuda")
    avg_launch = statistics.mean(launch_ms) / 1e3
    cv = statistics.pstdev(launch_ms) / statistics.mean(launch_ms) if len(launch_ms) > 1 else 0.0
    algo = algorithmic_bytes(case)
    default_case = headline_case(None)
    is_headline = (case.nranks, case.count, case.dtype, case.mask, case.proto, case.buff_size) == (
        default_case.nranks, default_case.count, default_case.dtype, default_case.mask, default_case.proto,
        default_case.buff_size)
    t = "float" if case.dtype == "f32" else "bf16"
    kernel = {"Simple": f"ring_simple_kernel<{t}>",
              "LL": f"ring_line_bulk_kernel<{t}, LL> (ring_line_kernel<{t}, LL> for chunks < 1024)",
              "LL128": f"ring_line_bulk_kernel<{t}, LL128> (ring_line_kernel<{t}, LL128> for chunks < 960)"}[
                  case.proto]
    achieved = algo / avg_launch / 1e9
    traffic = TRAFFIC_BYTES_PER_LAUNCH if is_headline and kernel_sources_sha16() == TRAFFIC_SOURCES_SHA16 else None
    del x, y, ws
    torch.cuda.empty_cache()

    extra = {}
    if rank == 0 and not args.no_sweep:
        extra["sweep"] = sweep(torch, B, max(5, args.steps // 2), args.warmup, peak)
    e2e = e2e_ring(case, torch, B, max(3, args.steps // 4), args.warmup) if rank == 0 and not args.no_e2e else None
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "cv_per_step": round(cv, 4),
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": case.dtype, "data": "synthetic",
        "config": {"workload": f"ring AllReduce, {case.nranks} virtual ranks on one GPU, {case.dtype} sum, "
                               f"{size_label(case.bytes_per_rank)} per rank, ring = seeded permutation (seed 3), "
                               f"{bin(case.mask).count('1')} channels, {case.proto}, "
                               f"{case.buff_size or 'default'} B FIFO, 4 chunk steps",
                   "nranks": case.nranks, "bytes_per_rank": case.bytes_per_rank, "ring_order": case.ring,
                   "channel_mask": hex(case.mask), "proto": case.proto, "buff_size": case.buff_size,
                   "chunk_steps": case.chunk_steps,
                   "l2": f"inputs larger than L2 ({case.nranks} x {size_label(case.bytes_per_rank)} in and out per step)",
                   "clock_sampling": "nvidia-smi every 200 ms; untimed calls keep the GPU busy for 0.3 s on each "
                                     "side of the timed region",
                   "parallelism": f"replicas x{world} (no GPU-to-GPU data path)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 3),
                     # the captured traffic belongs to the headline workload and
                     # the kernel sources it was captured with only
                     "traffic": traffic,
                     "kernel": kernel,
                     "algorithmic_bytes_per_launch": int(algo),
                     "peak_kind": f"{peak_kind} copy peak (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s",
                     "user_bytes_frac": round(case.nranks * 2 * case.bytes_per_rank / avg_launch / 1e9 / peak, 3),
                     # the measured DRAM bytes over the same launch time: what the HBM actually moved
                     "dram_frac": round(traffic / avg_launch / 1e9 / peak, 3) if traffic else None},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
    }
    line.update(extra)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case)
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def run_oneshot_only(args):
    """Time only the one-shot AllReduce: N=8 bf16 ranks, 7168 x T elements each
    (T = --oneshot-tokens), CUDA events around each call, one JSON line.
    --oneshot-staged times the staged form instead of the direct one."""
    import torch
    from collective_communication_gb300 import binding as B
    from collective_communication_gb300 import inputs as gen
    B.load_library()
    peak, _ = measured_peak()
    case = gen.OneShotCase(f"oneshot_bf16_n8_7168x{args.oneshot_tokens}", 8, 7168 * args.oneshot_tokens)
    g = torch.Generator(device="cuda")
    g.manual_seed(case.seed)
    x = torch.randn((8, case.count), generator=g, device="cuda").to(torch.bfloat16)
    y = rows_like(x, torch)
    send = [x[r] for r in range(8)]
    recv = [y[r] for r in range(8)]
    if args.oneshot_staged:
        ws = B.OneShotWorkspace(8, case.count, "bf16")
        call = lambda: B.oneshot_staged(send, recv, ws)  # noqa: E731
    else:
        call = lambda: B.oneshot(send, recv)  # noqa: E731
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:
        a.record(s)
        call()
        b.record(s)
    torch.cuda.synchronize()
    if args.oneshot_staged and B.get_status(ws) != B.Status.OK:
        raise RuntimeError("staged one-shot: device status not OK")
    t = statistics.median([a.elapsed_time(b) for a, b in ev]) / 1e3
    # unique bytes: inputs read and outputs written once (the staged form adds its copy)
    unique = (4 if args.oneshot_staged else 2) * 8 * case.count * 2
    print(json.dumps({"metric": "one-shot AllReduce time", "value": round(t * 1e6, 2), "unit": "us",
                      "higher_is_better": False, "steps": args.steps, "warmup": args.warmup, "dtype": "bf16",
                      "config": {"workload": case.name + ("_staged" if args.oneshot_staged else "")},
                      "unique_bytes_frac": round(unique / t / 1e9 / peak, 3)}))


def run_reference(args):
    """The CPU oracle as the reference arm: each step is one step-by-step
    simulation of the whole headline call, single-threaded."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    case = headline_case()
    from collective_communication_gb300 import inputs as gen
    x = gen.draw("normal", case.nranks, case.count, case.seed, case.dtype)
    oracle.lib()

    def one():
        oracle.ring_allreduce_sim(list(x), case.ring, case.mask, oracle.SIMPLE, case.buff_size, case.chunk_steps)

    for _ in range(args.warmup):
        one()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        one()
        times.append(time.perf_counter() - t0)
    t = sum(times) / len(times)
    v = busbw(case.bytes_per_rank, case.nranks, t)
    sample = (f"the whole headline call (8 ranks x 64 MiB f32) through the oracle's step-by-step simulation, "
              f"1 thread; host has {os.cpu_count()} cores")
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": UNIT,
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t * 1e3, 2), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": "ring AllReduce, 8 virtual ranks, f32 sum, 64 MiB per rank, ring = seeded "
                                   "permutation (seed 3), 12 channels, Simple, 1 MiB FIFO, 4 chunk steps (CPU oracle)"},
            "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    # workload variants (profiling): defaults give the headline workload
    ap.add_argument("--proto", choices=["Simple", "LL", "LL128"])
    ap.add_argument("--buff-size", type=int)
    ap.add_argument("--mib", type=int, help="MiB per rank")
    ap.add_argument("--kib", type=int, help="KiB per rank (instead of --mib)")
    ap.add_argument("--nranks", type=int)
    ap.add_argument("--channels", type=int)
    ap.add_argument("--dtype", choices=["f32", "bf16"], help="element type of a named variant (default f32)")
    ap.add_argument("--oneshot-tokens", type=int, help="time only the one-shot AllReduce of 7168 x T bf16")
    ap.add_argument("--oneshot-staged", action="store_true", help="with --oneshot-tokens: the staged form")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.oneshot_tokens:
        run_oneshot_only(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
