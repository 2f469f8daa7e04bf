"""Benchmark: Q4_0 decode weight GB/s and tokens/s at batch 1 on GB300.

Default workload (no flags): the 8B-shaped decoder stack -- 32 layers of
q/k/v/o/gate/up/down Q4_0 projections (hidden 4096, q 4096, kv 1024, ffn
14336), 3 925 868 544 weight bytes per token, all resident in HBM -- run one
token per step by replaying the decoder's CUDA graph (q4_layer_decode).  The
weights are 30x larger than L2, so every step streams them from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 8b|gemv|70b|70b-stream|sweep]
                  [--batch B] [--impl reference]

--batch B (1..16) runs the stack or the streamed ring on B activation rows per
step (weights read once per step; batch > 1 takes the tensor-core path).
--config sweep times every projection of the resident 8B stack through the
single-product call at B = 1, 2, 4, 8, 16 with each kernel and reports the
fastest kernel per batch size.

One JSON line per run on rank 0.  Under torchrun every rank runs its own
replica (the product has no cross-GPU step): value = all ranks' bytes / the
slowest rank's time.  ``--impl reference`` times the plain CPU oracle on a
bounded sample of the same workload instead (the only baseline that exists).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Q4_0 decode weight GB/s & tokens/s (batch 1), % of HBM / host-link roofline"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = {
    "engine_kernel": ("q4_engine.cu", "q4_device.cuh", "q4_phase.cuh"),
    "tc_engine_kernel": ("q4_tc_engine.cu", "q4_frag.cuh", "q4_device.cuh", "q4_phase.cuh"),
    "oneshot_kernel": ("q4_oneshot.cu", "q4_frag.cuh", "q4_device.cuh"),
    "mma_kernel": ("q4_mma.cu", "q4_frag.cuh", "q4_device.cuh"),
    "bt_engine_kernel": ("q4_bt_engine.cu", "q4_frag.cuh", "q4_device.cuh", "q4_phase.cuh"),
}


def _code_only(text: bytes) -> bytes:
    """Source text without comments and with whitespace runs collapsed, so that
    a documentation-only edit does not mark a profile stale."""
    text = re.sub(rb"/\*.*?\*/", b" ", text, flags=re.S)
    text = re.sub(rb"//[^\n]*", b" ", text)
    return re.sub(rb"\s+", b" ", text).strip()


def kernel_source_hash(kernel: str = "engine_kernel") -> str:
    """Hash of the device code a kernel is built from (the shared header up to
    its host-side declarations), comments and layout excluded."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "weight_streaming_q4_gb300", "csrc", f), "rb") as fh:
            text = fh.read()
        if f == "q4_device.cuh":
            text = text.split(b"// Host-side launchers")[0]
        h.update(_code_only(text))
    return h.hexdigest()[:16]


def ncu_traffic(key: str):
    """DRAM bytes per launch from the committed ncu summary, or None if absent or stale."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        data = json.load(f)
    ent = data.get(key)
    if not ent or ent.get("kernel_sha") != kernel_source_hash(key.split(":")[0]):
        return None
    return ent.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 6:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[2:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(secs: float, device) -> float:
    """The slowest rank's timed-region seconds (every rank gets it)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([secs], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step: int, world: int, per_step_s: float) -> float:
    """Weight GB/s of the whole job: every replica streams its own bytes each step."""
    return bytes_per_step * world / per_step_s / 1e9


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


# ------------------------------------------------------------------ workloads

def stack_cfg(name):
    from weight_streaming_q4_gb300 import synth
    cfg = dict(synth.LLAMA_8B if name in ("8b", "sweep") else synth.LLAMA_70B)
    n_layers = cfg.pop("n_layers")
    return cfg, n_layers


def time_region(torch, stream, fn, steps, warmup, barrier, gpu_index):
    """W untimed steps, then K steps between events on `stream`, barrier + sync on both sides."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index) as clk:
        torch.cuda.synchronize()
        barrier()
        start.record(stream)
        for _ in range(steps):
            fn()
        end.record(stream)
        torch.cuda.synchronize()
    barrier()
    return start.elapsed_time(end) / 1e3, clk.summary()


def run_stack(args, torch, q4, model, synth, stream, barrier, gpu_index):
    cfg, n_layers = stack_cfg(args.config)
    full_layers = n_layers
    if args.layers:
        n_layers = args.layers   # a shorter stack of the same shape (small profiling case)
    B = args.batch
    shape = q4.LayerShape.of(**cfg)
    layer_bytes = q4.q4_layer_offsets(shape)[1]
    wbuf, ptrs = model.resident_layers(shape, n_layers, seed=0)
    ws, offs, ws_bytes = model.workspace(shape, n_layers, B)
    with torch.cuda.stream(stream):
        mode = q4.Q4_DEC_FUSED | (q4.Q4_DEC_BARRIER if args.barrier else 0) | (
            q4.Q4_DEC_CUDA_CORE if args.cuda_core else 0) | (q4.Q4_DEC_BATCH_ENGINE if args.batch_engine else 0)
        dec = q4.q4_decoder_create(shape, ptrs, B, ws, ws_bytes, mode, stream=stream)
        h0 = torch.from_numpy(synth.activations(B, cfg["hidden"], 0).reshape(-1).view("int16").copy())
        h = h0.cuda()
    torch.cuda.synchronize()

    def step():
        q4.q4_layer_decode(dec, h, stream=stream)

    secs, clocks = time_region(torch, stream, step, args.steps, args.warmup, barrier, gpu_index)
    status = q4.q4_decoder_status(dec, stream=stream)
    if status != 0:
        raise RuntimeError(f"decoder kernels reported status {status}")

    # end to end through the public call with host buffers: H2D of the step's
    # input and D2H of its result every step (pinned), host waits for the result
    hin = h0.pin_memory()
    hout = torch.empty_like(hin).pin_memory()
    e2e_steps = max(10, args.steps // 4)
    for _ in range(3):
        h.copy_(hin, non_blocking=True)
        step()
        hout.copy_(h, non_blocking=True)
        stream.synchronize()
    barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            h.copy_(hin, non_blocking=True)
            step()
            hout.copy_(h, non_blocking=True)
            stream.synchronize()
    e2e_secs = time.perf_counter() - t0
    tagged = q4.q4_decoder_tagged(dec)
    q4.q4_decoder_destroy(dec)
    nbytes = layer_bytes * n_layers
    # batch 1 and the batched engine: one persistent launch per token; the
    # per-product path: per layer 4 tensor-core products + 2 glue launches,
    # plus the first layer's input norm
    batched = 2 <= B <= 8 and args.batch_engine
    launches = 1 if B == 1 or batched else 6 * n_layers + 1
    return dict(secs=secs, clocks=clocks, bytes_per_step=nbytes, launches_per_step=launches,
                kernel_launches_per_step=1 if B == 1 or batched else 4 * n_layers,
                e2e_secs=e2e_secs, e2e_steps=e2e_steps, h2d=h0.numel() * 2, d2h=h0.numel() * 2,
                workload=(f"{'8B' if args.config == '8b' else '70B'}-shaped decoder stack, {n_layers} layers, "
                          f"batch {B}, HBM-resident, one CUDA-graph replay per step"),
                kernel=(("engine_kernel" if args.barrier or args.cuda_core else "tc_engine_kernel") if B == 1
                        else "bt_engine_kernel" if batched else "mma_kernel"),
                # the traffic records are for the whole stack: none for fewer layers
                kernel_key=(((f"engine_kernel:{args.config}_stack" if args.barrier or args.cuda_core
                              else f"tc_engine_kernel:{args.config}_stack") if B == 1
                             else f"bt_engine_kernel:{args.config}_stack_b{B}" if batched
                             else f"mma_kernel:{args.config}_stack_b{B}")
                            if n_layers == full_layers else None),
                n_layers=n_layers, cfg=cfg, tagged=tagged)


def run_gemv(args, torch, q4, model, synth, stream, barrier, gpu_index):
    # N = K = 4096: 9.4 MB fits in L2, so each step walks a ring of distinct
    # copies several times larger than L2 (every launch reads from HBM)
    n = k = 4096
    mb = q4.q4_matrix_bytes(n, k)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    copies = max(8, (4 * l2) // mb + 1)
    w = torch.empty(copies * mb, dtype=torch.uint8, device="cuda")
    for c in range(copies):
        synth.device_fill_q4(w.data_ptr() + c * mb, n * k // 32, seed=0, tid=synth.GEMV_TID)
    x = torch.from_numpy(synth.activations(1, k, 0).reshape(-1).view("int16").copy()).cuda()
    y = torch.empty(n, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    # one step = one pass over the ring, captured as a CUDA graph; the
    # products are independent and nothing else runs between them, so they are
    # chained calls (each may start while the one before it finishes)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for c in range(copies):   # first launches outside capture
            q4.q4_gemv(w.data_ptr() + c * mb, x, y, n, k, 1, stream=stream, chain=True)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for c in range(copies):
                q4.q4_gemv(w.data_ptr() + c * mb, x, y, n, k, 1, stream=stream, chain=True)

    def step():
        g.replay()

    with torch.cuda.stream(stream):
        secs, clocks = time_region(torch, stream, step, args.steps, args.warmup, barrier, gpu_index)
    if q4.q4_device_status() != 0:
        raise RuntimeError("q4_gemv kernels reported a failed wait")
    # e2e: x in, y out through pinned host buffers, one product per step
    xin = x.cpu().pin_memory()
    yout = torch.empty(n, dtype=torch.float32).pin_memory()
    e2e_steps = max(50, args.steps)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            x.copy_(xin, non_blocking=True)
            q4.q4_gemv(w.data_ptr() + (i % copies) * mb, x, y, n, k, 1, stream=stream)
            yout.copy_(y, non_blocking=True)
            stream.synchronize()
    e2e_secs = time.perf_counter() - t0
    return dict(secs=secs, clocks=clocks, bytes_per_step=mb * copies, launches_per_step=copies,
                e2e_secs=e2e_secs, e2e_steps=e2e_steps, e2e_bytes_per_step=mb, h2d=2 * k, d2h=4 * n,
                workload=f"single Q4_0 product N=K=4096, batch 1, ring of {copies} weight copies (> L2)",
                kernel="oneshot_kernel", kernel_key="oneshot_kernel:gemv", cfg=dict(n=n, k=k, copies=copies))


def h2d_multi_stream(torch, blocks, nbytes, counts=(1, 2, 4)):
    """Pinned host -> HBM GB/s with n copies of nbytes in flight on n streams."""
    streams = [torch.cuda.Stream() for _ in range(max(counts))]
    dst = [torch.empty(nbytes, dtype=torch.uint8, device="cuda") for _ in range(max(counts))]
    out = {}
    for n in counts:
        best = 0.0
        for _ in range(3):
            torch.cuda.synchronize()
            ev0 = torch.cuda.Event(enable_timing=True)
            ev0.record(streams[0])
            for s in streams[1:n]:
                s.wait_event(ev0)
            for j in range(n):
                with torch.cuda.stream(streams[j]):
                    for r in range(2):
                        dst[j].copy_(blocks[(2 * j + r) % len(blocks)][:nbytes], non_blocking=True)
            for s in streams[1:n]:
                e = torch.cuda.Event()
                e.record(s)
                streams[0].wait_event(e)
            ev1 = torch.cuda.Event(enable_timing=True)
            ev1.record(streams[0])
            torch.cuda.synchronize()
            best = max(best, 2 * n * nbytes / (ev0.elapsed_time(ev1) / 1e3) / 1e9)
        out[str(n)] = round(best, 2)
    del dst
    torch.cuda.empty_cache()
    return out


def numa_report(blocks):
    """NUMA nodes of the host, the GPU's affinity node and where the pinned blocks' pages are."""
    import ctypes, platform
    from collections import Counter
    rep = {}
    try:
        rep["host_nodes"] = len([d for d in os.listdir("/sys/devices/system/node") if d.startswith("node")])
        bus = subprocess.run(["nvidia-smi", "--query-gpu=pci.bus_id", "--format=csv,noheader", "-i",
                              str(int(os.environ.get("LOCAL_RANK", 0)))], capture_output=True, text=True,
                             timeout=30).stdout.strip().lower()
        for cand in (bus, bus[4:]):
            p = f"/sys/bus/pci/devices/{cand}/numa_node"
            if os.path.exists(p):
                rep["gpu_numa_node"] = int(open(p).read().strip())
                break
        nr = {"aarch64": 239, "x86_64": 279}.get(platform.machine())
        if nr is not None:
            libc = ctypes.CDLL(None, use_errno=True)
            ps = os.sysconf("SC_PAGE_SIZE")
            cnt = Counter()
            for b in blocks:
                n = 16
                pages = (ctypes.c_void_p * n)(*[(b.data_ptr() + i * (b.numel() // n)) // ps * ps for i in range(n)])
                status = (ctypes.c_int * n)()
                if libc.syscall(nr, 0, n, pages, None, status, 0) == 0:   # query only: no move
                    cnt.update(int(x) for x in status)
            rep["pinned_page_nodes"] = {str(k): v for k, v in sorted(cnt.items())}
    except Exception as e:   # a report, never a failure
        rep["error"] = str(e)
    return rep


def timeline_summary(tl):
    """Per-layer [copy begin, copy end, compute begin, compute end] (ns) of one
    ring token -> medians and how much of the compute ran under a copy."""
    import numpy as np
    tl = tl.astype(np.int64)
    streamed = tl[:, 0] > 0
    t0 = min(tl[streamed, 0].min() if streamed.any() else tl[:, 2].min(), tl[:, 2].min())
    rel = (tl - t0) / 1e6
    rel[~streamed, :2] = np.nan
    copy = rel[:, 1] - rel[:, 0]
    comp = rel[:, 3] - rel[:, 2]
    wait = np.r_[rel[0, 2], rel[1:, 2] - rel[:-1, 3]]   # compute stream idle before each layer
    spans = [(a, b) for a, b in rel[streamed, :2]]
    covered = 0.0
    for a, b in rel[:, 2:4]:
        covered += sum(max(0.0, min(b, y) - max(a, x)) for x, y in spans)
    end = np.nanmax(rel[:, 3])
    return {"token_ms": round(float(end), 3), "copy_ms_median": round(float(np.nanmedian(copy)), 4),
            "compute_ms_median": round(float(np.median(comp)), 4),
            "compute_wait_ms_median": round(float(np.median(wait[1:])), 4),
            "copy_engine_busy_frac": round(float(np.nansum(copy) / end), 4),
            "compute_under_copy_frac": round(float(covered / comp.sum()), 4),
            "first_layers_ms": [[round(float(v), 3) for v in r] for r in rel[:4]]}


def run_stream(args, torch, q4, model, synth, stream, barrier, gpu_index):
    """70B-shaped stack through the copy/compute ring.  --resident-frac keeps
    that fraction of the layers (a prefix) resident in HBM; --chunked copies
    each streamed layer as four chunks with one event each.  --config
    stream-sweep times resident fractions 0, 1/4, 1/2, 3/4 with merged and
    chunked copies and reports them all."""
    cfg, n_layers = stack_cfg("70b")
    shape = q4.LayerShape.of(**cfg)
    layer_bytes = q4.q4_layer_offsets(shape)[1]
    stride = model.layer_stride(shape)
    # host RAM: all 80 layers distinct if it fits, else a cyclic set (labelled)
    try:
        import psutil
        avail = psutil.virtual_memory().available
    except Exception:
        avail = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    distinct = n_layers if avail > (n_layers + 8) * stride else max(2, int(avail * 0.6 // stride))
    blocks, hptrs = model.host_layers(shape, n_layers, seed=0, distinct=distinct)
    bufs = [torch.empty(stride, dtype=torch.uint8, device="cuda") for _ in range(2)]
    B = args.batch
    ws, offs, ws_bytes = model.workspace(shape, n_layers, B)
    h0 = torch.from_numpy(synth.activations(B, cfg["hidden"], 0).reshape(-1).view("int16").copy())
    h = h0.cuda()
    # pinned host -> HBM copy peak at the ring's transfer size, with 1, 2 and 4
    # copies in flight on separate streams (the link's limit, not one stream's)
    cs = torch.cuda.Stream()
    h2d_streams = h2d_multi_stream(torch, blocks, stride)
    best = max(h2d_streams.values())
    numa = numa_report(blocks)

    # each host block's own copy speed (blocks in slow host memory show up here)
    def block_speed(blk, i):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(cs)
        with torch.cuda.stream(cs):
            bufs[i & 1].copy_(blk, non_blocking=True)
        ev1.record(cs)
        torch.cuda.synchronize()
        return stride / (ev0.elapsed_time(ev1) / 1e3) / 1e9

    block_gbs = [block_speed(blocks[i], i) for i in range(len(blocks))]
    med = statistics.median(block_gbs)
    first_slow = [i for i, g_ in enumerate(block_gbs) if g_ < 0.8 * med]
    # host-memory placement: a block that copies at under half the median speed
    # is allocated again (same bytes, new pinned pages), up to twice, and the
    # faster placement is kept
    replaced = []
    for i in first_slow:
        if block_gbs[i] >= 0.5 * med:
            continue
        for _ in range(2):
            nb = torch.empty(stride, dtype=torch.uint8, pin_memory=True)
            nb.copy_(blocks[i])
            g_new = block_speed(nb, i)
            if g_new > block_gbs[i]:
                blocks[i], block_gbs[i] = nb, g_new
            if block_gbs[i] >= 0.8 * med:
                break
        replaced.append(i)
    hptrs = [blocks[i % len(blocks)].data_ptr() for i in range(n_layers)]
    host_blocks = {"min_gbs": round(min(block_gbs), 2), "median_gbs": round(med, 2), "max_gbs": round(max(block_gbs), 2),
                   "slow_blocks": [i for i, g_ in enumerate(block_gbs) if g_ < 0.8 * med],
                   "slow_at_first_copy": first_slow, "reallocated": replaced}
    sweep = args.config == "stream-sweep"
    fracs = [0.0, 0.25, 0.5, 0.75] if sweep else [args.resident_frac]
    # device copies of every layer a configuration may keep resident (same seeded bytes as the host blocks)
    need = set()
    for frac in fracs:
        for pat in (["prefix", "spread"] if sweep else [args.resident_pattern]):
            need |= set(resident_set(n_layers, int(round(frac * n_layers)), pat))
    dptrs = {}
    dev_blocks = []
    if need:
        for l in sorted(need):
            buf, ptr = model.resident_layers(shape, 1, seed=0, first_layer=l)
            dev_blocks.append(buf)
            dptrs[l] = ptr[0]
    steps = min(args.steps, 20 if not sweep else 6)
    warm = min(args.warmup, 3)
    runs = []
    combos = []
    for frac in fracs:
        R = int(round(frac * n_layers))
        if sweep:
            combos += [(R, "prefix", False, False), (R, "prefix", True, False)] + (
                [(R, "spread", False, False)] if 0 < R < n_layers else [])
        else:
            combos.append((R, args.resident_pattern, args.chunked, args.single_buffer))
    if getattr(args, "with_single", False) and not sweep:
        # the memory-efficient mode on the same pinned blocks: one staging buffer,
        # merged and chunked copies
        combos += [(combos[0][0], combos[0][1], False, True), (combos[0][0], combos[0][1], True, True)]
    for ci, (R, pat, chunked, single) in enumerate(combos):
        if True:
            keep = set(resident_set(n_layers, R, pat))
            host = [0 if i in keep else hptrs[i] for i in range(n_layers)]
            res = [dptrs[i] if i in keep else 0 for i in range(n_layers)]
            flags = (q4.Q4_STREAM_CHUNKED if chunked else 0) | (q4.Q4_STREAM_BARRIER if args.barrier else 0) | (
                q4.Q4_STREAM_CUDA_CORE if args.cuda_core else 0) | (q4.Q4_STREAM_SINGLE_BUFFER if single else 0)
            ring = q4.q4_stream_create_ex(shape, host, res, B, bufs[0], None if single else bufs[1], stride, ws,
                                          ws_bytes, flags)

            def step():
                q4.q4_stream_layers(ring, h, stream=stream)

            secs, clocks = time_region(torch, stream, step, steps, warm, barrier, gpu_index)
            if q4.q4_stream_status(ring, stream=stream) != 0:
                raise RuntimeError("stream ring kernels reported a failed wait")
            t = secs / steps
            runs.append(dict(resident_layers=R, placement=pat, chunked=chunked, single_buffer=single, secs=secs,
                             clocks=clocks,
                             ms_per_token=round(t * 1e3, 3), tokens_per_s=round(B / t, 3),
                             weight_gbs=round(layer_bytes * n_layers / t / 1e9, 2),
                             host_link_gbs=round(layer_bytes * (n_layers - R) / t / 1e9, 2),
                             host_link_frac=round(layer_bytes * (n_layers - R) / t / 1e9 / best, 4)))
            q4.q4_stream_destroy(ring)
    head = runs[0]
    # the first configuration again (rings share the workspace) for the end-to-end run
    R, pat, chunked, single = combos[0]
    keep = set(resident_set(n_layers, R, pat))
    flags = (q4.Q4_STREAM_CHUNKED if chunked else 0) | (q4.Q4_STREAM_BARRIER if args.barrier else 0) | (
        q4.Q4_STREAM_CUDA_CORE if args.cuda_core else 0) | (q4.Q4_STREAM_SINGLE_BUFFER if single else 0)
    last_ring = q4.q4_stream_create_ex(shape, [0 if i in keep else hptrs[i] for i in range(n_layers)],
                                       [dptrs[i] if i in keep else 0 for i in range(n_layers)], B, bufs[0],
                                       None if single else bufs[1], stride, ws, ws_bytes, flags)
    # end to end through the public call: the step's input copied in from pinned
    # host memory and its result read back, every step
    hin = h0.pin_memory()
    hout = torch.empty_like(hin).pin_memory()
    e2e_steps = max(3, min(steps, 6))
    with torch.cuda.stream(stream):
        h.copy_(hin, non_blocking=True)
        q4.q4_stream_layers(last_ring, h, stream=stream)
        stream.synchronize()
    barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            h.copy_(hin, non_blocking=True)
            q4.q4_stream_layers(last_ring, h, stream=stream)
            hout.copy_(h, non_blocking=True)
            stream.synchronize()
    e2e_secs = time.perf_counter() - t0
    tagged = q4.q4_stream_tagged(last_ring)
    q4.q4_stream_destroy(last_ring)
    R = runs[0]["resident_layers"]
    desc = (f"70B-shaped stack, {n_layers} layers, {n_layers - head['resident_layers']} streamed from pinned host "
            f"memory ({distinct} distinct layer blocks) through {'one HBM layer buffer' if head['single_buffer'] else 'two HBM layer buffers'}"
            f"{', ' + str(head['resident_layers']) + ' resident (' + head['placement'] + ')' if head['resident_layers'] else ''}, "
            f"{'chunked' if head['chunked'] else 'merged'} copies, "
            f"{'one staging buffer' if head['single_buffer'] else 'two staging buffers'}, batch {B}")
    # per-layer copy/compute timeline of one token of the headline configuration
    R0, pat0, chunked0, single0 = combos[0]
    timelines = {}
    for single_t in ([single0] + ([not single0] if getattr(args, "with_single", False) else [])):
        flags = (q4.Q4_STREAM_CHUNKED if chunked0 else 0) | (q4.Q4_STREAM_BARRIER if args.barrier else 0) | (
            q4.Q4_STREAM_CUDA_CORE if args.cuda_core else 0) | (q4.Q4_STREAM_SINGLE_BUFFER if single_t else 0) | (
            q4.Q4_STREAM_TIMELINE)
        keep = set(resident_set(n_layers, R0, pat0))
        tl_ring = q4.q4_stream_create_ex(shape, [0 if i in keep else hptrs[i] for i in range(n_layers)],
                                         [dptrs[i] if i in keep else 0 for i in range(n_layers)], B, bufs[0],
                                         None if single_t else bufs[1], stride, ws, ws_bytes, flags)
        with torch.cuda.stream(stream):
            for _ in range(2):
                q4.q4_stream_layers(tl_ring, h, stream=stream)
        tl = q4.q4_stream_timeline(tl_ring, n_layers, stream=stream)
        q4.q4_stream_destroy(tl_ring)
        timelines["single_buffer" if single_t else "double_buffer"] = timeline_summary(tl)
    out = dict(secs=head["secs"], clocks=head["clocks"], bytes_per_step=layer_bytes * n_layers,
               streamed_bytes_per_step=layer_bytes * (n_layers - head["resident_layers"]),
               h2d_streams=h2d_streams, numa=numa, timelines=timelines,
               launches_per_step=n_layers if B == 1 else 6 * n_layers + 1,
               kernel_launches_per_step=n_layers if B == 1 else 4 * n_layers,
               steps_override=steps, warmup_override=warm, h2d_peak_gbs=best,
               e2e_secs=e2e_secs, e2e_steps=e2e_steps, h2d=h0.numel() * 2, d2h=h0.numel() * 2,
               e2e_note=f"measured on the first configuration run ({R} resident layers)",
               workload=desc, kernel=("engine_kernel" if args.barrier or args.cuda_core else "tc_engine_kernel") if B == 1 else "mma_kernel",
               kernel_key=None, cfg=cfg, distinct=distinct, host_blocks=host_blocks, tagged=tagged)
    if sweep or len(runs) > 1:
        out["residency_sweep"] = [{k: v for k, v in r.items() if k not in ("secs", "clocks")} for r in runs]
    return out


def run_kv(args, torch, q4, model, synth, stream, barrier, gpu_index):
    """The 8B stack decoding with per-layer KV caches: each step is one token
    at a fixed position (the position counter is set back before the token),
    attending over `ctx` cached positions in every layer; one CUDA graph per
    bucket (bucket = ctx).  Bytes per step = the weights plus the KV-cache
    rows read (32 layers x 2 x ctx x kv_dim x 2 B)."""
    cfg, n_layers = stack_cfg("8b")
    if args.layers:
        n_layers = args.layers
    shape = q4.LayerShape.of(**cfg)
    layer_bytes = q4.q4_layer_offsets(shape)[1]
    wbuf, ptrs = model.resident_layers(shape, n_layers, seed=0)
    ws, offs, ws_bytes = model.workspace(shape, n_layers, 1)
    kvd, hd = cfg["kv_dim"], cfg["head_dim"]
    n_q, n_kv = cfg["q_dim"] // hd, kvd // hd
    contexts = [int(c) for c in str(args.kv_contexts).split(",")]
    if not contexts or any(c < 128 or c % 128 for c in contexts):
        raise SystemExit("--kv-contexts: multiples of 128")
    h0 = torch.from_numpy(synth.activations(1, cfg["hidden"], 0).reshape(-1).view("int16").copy())
    h = h0.cuda()
    per = {}
    for ctx in contexts:
        cap = ctx
        kc = torch.empty(n_layers, cap * kvd, dtype=torch.int16, device="cuda")
        vc = torch.empty(n_layers, cap * kvd, dtype=torch.int16, device="cuda")
        for l in range(n_layers):
            synth.device_fill_normal_f16(kc[l].data_ptr(), cap * kvd, seed=0, tid=0x40000000 + 2 * l)
            synth.device_fill_normal_f16(vc[l].data_ptr(), cap * kvd, seed=0, tid=0x40000001 + 2 * l)
        pos = torch.zeros(1, dtype=torch.int32, device="cuda")
        pos0 = torch.full((1,), ctx - 1, dtype=torch.int32, device="cuda")
        awb = q4.q4_attn_workspace_bytes(n_q, n_kv, hd, cap)
        aws = torch.empty(awb, dtype=torch.uint8, device="cuda")
        torch.cuda.synchronize()
        dec = q4.q4_decoder_create_kv(shape, ptrs, cap, list(kc), list(vc), pos, aws, awb, ws, ws_bytes,
                                      stream=stream)

        def step():
            pos.copy_(pos0, non_blocking=True)    # the token at position ctx-1 (a device copy, no kernel)
            q4.q4_layer_decode(dec, h, stream=stream)

        with torch.cuda.stream(stream):
            secs, clocks = time_region(torch, stream, step, args.steps, args.warmup, barrier, gpu_index)
        status = q4.q4_decoder_status(dec, stream=stream)
        if status != 0:
            raise RuntimeError(f"KV decoder kernels reported status {status}")
        kv_bytes = n_layers * 2 * ctx * kvd * 2
        t = secs / args.steps
        per[ctx] = dict(secs=secs, clocks=clocks, ms_per_step=round(t * 1e3, 4), tokens_per_s=round(1 / t, 2),
                        kv_bytes_per_step=kv_bytes, dec=dec, keep=(kc, vc, pos, pos0, aws), step=step)
    head = per[contexts[-1]]
    step = head["step"]
    hin = h0.pin_memory()
    hout = torch.empty_like(hin).pin_memory()
    e2e_steps = max(10, args.steps // 4)
    with torch.cuda.stream(stream):
        for _ in range(3):
            h.copy_(hin, non_blocking=True)
            step()
            hout.copy_(h, non_blocking=True)
            stream.synchronize()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            h.copy_(hin, non_blocking=True)
            step()
            hout.copy_(h, non_blocking=True)
            stream.synchronize()
    e2e_secs = time.perf_counter() - t0
    for r in per.values():
        q4.q4_decoder_destroy(r.pop("dec"))
    ctx = contexts[-1]
    wbytes = layer_bytes * n_layers
    return dict(secs=head["secs"], clocks=head["clocks"], bytes_per_step=wbytes + head["kv_bytes_per_step"],
                launches_per_step=2 * n_layers + 2, kernel_launches_per_step=n_layers + 1,
                e2e_secs=e2e_secs, e2e_steps=e2e_steps, h2d=h0.numel() * 2, d2h=h0.numel() * 2,
                workload=(f"8B-shaped decoder stack with per-layer binary16 KV caches, {n_layers} layers, batch 1, "
                          f"one token at position {ctx - 1} (context {ctx}, bucket {ctx}), HBM-resident, "
                          f"one CUDA-graph replay per step"),
                kernel="tc_engine_kernel", kernel_key=None, n_layers=n_layers, cfg=cfg, tagged=True,
                kv_contexts={str(c): {k: v for k, v in r.items() if k in ("ms_per_step", "tokens_per_s",
                                                                          "kv_bytes_per_step")}
                             for c, r in per.items()},
                weight_bytes_per_step=wbytes)


def run_attn(args, torch, q4, model, synth, stream, barrier, gpu_index):
    """Decode attention over the KV caches of all 32 layers of the 8B shape
    (32 query heads, 8 value heads, head_dim 128), one CUDA graph per context
    bucket (512, 1024, 2048, 4096), every position in use; the caches of one
    step (32 layers x 2 x ctx x 1024 x 2 B) exceed L2 from the 1024 bucket up."""
    import numpy as np
    n_q, n_kv, hd, L = 32, 8, 128, 32
    kv = n_kv * hd
    buckets = [512, 1024, 2048, 4096]
    cap = max(buckets)
    kc = torch.empty(L, cap * kv, dtype=torch.int16, device="cuda")
    vc = torch.empty(L, cap * kv, dtype=torch.int16, device="cuda")
    for l in range(L):
        synth.device_fill_normal_f16(kc[l].data_ptr(), cap * kv, seed=0, tid=0x40000000 + 2 * l)
        synth.device_fill_normal_f16(vc[l].data_ptr(), cap * kv, seed=0, tid=0x40000001 + 2 * l)
    q_host = torch.from_numpy((np.random.default_rng(0).normal(size=n_q * hd) * 0.25).astype(np.float32))
    q = q_host.cuda()
    out = torch.empty(L, n_q * hd, dtype=torch.int16, device="cuda")
    ctx = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsb = q4.q4_attn_workspace_bytes(n_q, n_kv, hd, cap)
    ws = torch.zeros(L, (wsb + 255) // 256 * 256, dtype=torch.uint8, device="cuda")
    steps = max(10, min(args.steps, 200))
    per = {}
    for b in buckets:
        ctx.fill_(b)

        def enqueue():
            for l in range(L):
                q4.q4_attn_decode(q, kc[l], vc[l], ctx, b, n_q, n_kv, hd, out[l], ws[l], wsb, stream=stream)

        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            enqueue()
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                enqueue()
        with torch.cuda.stream(stream):
            secs, clocks = time_region(torch, stream, g.replay, steps, 3, barrier, gpu_index)
        t = secs / steps
        nbytes = L * 2 * b * kv * 2
        per[b] = dict(secs=secs, clocks=clocks, ms_per_step=round(t * 1e3, 4), kv_gbs=round(nbytes / t / 1e9, 2),
                      bytes_per_step=nbytes)
        last_graph = g
    head = per[cap]
    # end to end through the public call: q in from pinned memory, the outputs back, every step
    qin = q_host.pin_memory()
    oout = torch.empty(L, n_q * hd, dtype=torch.int16).pin_memory()
    e2e_steps = max(10, steps // 4)
    with torch.cuda.stream(stream):
        q.copy_(qin, non_blocking=True)
        last_graph.replay()
        stream.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            q.copy_(qin, non_blocking=True)
            last_graph.replay()
            oout.copy_(out, non_blocking=True)
            stream.synchronize()
    e2e_secs = time.perf_counter() - t0
    return dict(secs=head["secs"], clocks=head["clocks"], bytes_per_step=head["bytes_per_step"],
                launches_per_step=2 * L, kernel_launches_per_step=L, steps_override=steps, warmup_override=3,
                e2e_secs=e2e_secs, e2e_steps=e2e_steps, h2d=q_host.numel() * 4, d2h=out.numel() * 2,
                workload=(f"decode attention, 8B heads (32 q, 8 kv, head_dim 128), {L} layers' binary16 KV caches, "
                          f"context {cap} (bucket {cap}), one CUDA graph per bucket"),
                kernel="attn_mma_kernel", kernel_key=None, cfg=dict(n_q=n_q, n_kv=n_kv, hd=hd),
                attn_buckets={str(b): {k: v for k, v in r.items() if k not in ("secs", "clocks")}
                              for b, r in per.items()})


def resident_set(n_layers, n_res, pattern):
    """Which layers stay resident: the first n_res ("prefix") or n_res spread evenly over the stack
    ("spread", so the copies of the streamed layers are spaced out between resident ones)."""
    if n_res <= 0:
        return []
    if pattern == "prefix":
        return list(range(n_res))
    return sorted({min(n_layers - 1, (i * n_layers) // n_res) for i in range(n_res)})


def run_sweep(args, torch, q4, model, synth, stream, barrier, gpu_index):
    """Every projection of the resident 8B stack through q4_gemv_ex, per batch
    size and kernel, one CUDA graph per (batch, kernel) holding all 224 products."""
    cfg, n_layers = stack_cfg("8b")
    shape = q4.LayerShape.of(**cfg)
    offs, layer_bytes = q4.q4_layer_offsets(shape)
    wbuf, ptrs = model.resident_layers(shape, n_layers, seed=0)
    dims = synth.layer_dims(cfg["hidden"], cfg["q_dim"], cfg["kv_dim"], cfg["ffn"])
    kmax = max(k for _, k in dims)
    nmax = max(n for n, _ in dims)
    x = torch.from_numpy(synth.activations(16, kmax, 0).reshape(-1).view("int16").copy()).cuda()
    y = torch.empty(16 * nmax, dtype=torch.float32, device="cuda")
    # the one-shot products are chained calls: independent, nothing in between
    kernels = {"oneshot": q4.Q4_KERNEL_ONESHOT | q4.Q4_GEMV_CHAIN, "tc_engine": q4.Q4_KERNEL_TC,
               "engine": q4.Q4_KERNEL_STREAM, "mma": q4.Q4_KERNEL_MMA, "simple": q4.Q4_KERNEL_SIMPLE}
    nbytes = layer_bytes * n_layers
    steps = max(5, min(args.steps, 50))
    results = {}
    for B in (1, 2, 4, 8, 16):
        for name, kern in kernels.items():
            if name in ("oneshot", "tc_engine", "engine") and B != 1:   # batch-1 kernels
                continue

            def enqueue():
                for p in ptrs:
                    for j, (n, k) in enumerate(dims):
                        q4.q4_gemv_ex(p + offs[j], x, y, n, k, B, kern, stream=stream)

            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                enqueue()
                stream.synchronize()
                with torch.cuda.graph(g, stream=stream):
                    enqueue()
            with torch.cuda.stream(stream):
                secs, clocks = time_region(torch, stream, g.replay, steps, 3, barrier, gpu_index)
            if q4.q4_device_status() != 0:
                raise RuntimeError(f"{name} kernel reported a failed wait at batch {B}")
            t = secs / steps
            results.setdefault(B, {})[name] = dict(ms_per_step=round(t * 1e3, 4),
                                                   weight_gbs=round(nbytes / t / 1e9, 2),
                                                   tokens_per_s=round(B / t, 1), clocks_mhz=clocks["sm_mhz"])
            del g
    best = {B: max(r, key=lambda k: r[k]["weight_gbs"]) for B, r in results.items()}
    # headline of this config: batch 1 with its fastest kernel
    b1 = results[1][best[1]]
    return dict(secs=b1["ms_per_step"] * steps / 1e3, clocks=clocks, bytes_per_step=nbytes,
                launches_per_step=7 * n_layers, kernel_launches_per_step=7 * n_layers,
                steps_override=steps, warmup_override=3, e2e_secs=None,
                workload=(f"8B-shaped projections ({n_layers} layers x 7, {nbytes} B), one single-product call each, "
                          f"batch sweep 1-16"),
                kernel=f"{best[1]} (q4_gemv_ex)", kernel_key=None, cfg=cfg,
                sweep={str(B): dict(results[B], fastest=best[B]) for B in results})


# ------------------------------------------------------------------ CPU oracle

def cpu_oracle_rate(cfg_name: str, budget_s: float, torch=None, q4=None, model=None):
    """The CPU oracle's weight GB/s on a bounded sample: whole projections of
    layer 0, 1, ... (row-parallel over all host cores) until budget_s passes."""
    import numpy as np

    import oracle as ora
    from weight_streaming_q4_gb300 import synth
    cores = os.cpu_count() or 1
    if cfg_name == "gemv":
        dims = [(4096, 4096, synth.GEMV_TID)]
        layers = [0]
    else:
        cfg, n_layers = stack_cfg(cfg_name)
        dims = None
        layers = list(range(n_layers))
    done_bytes, t_total, done_layers = 0, 0.0, 0
    for layer in layers:
        if dims is None:
            mats = [(n, k, synth.tensor_id(layer, p)) for p, (n, k) in
                    enumerate(synth.layer_dims(cfg["hidden"], cfg["q_dim"], cfg["kv_dim"], cfg["ffn"]))]
        else:
            mats = dims
        for (n, k, tid) in mats:
            # bounded row sample of this projection, rows spread over the matrix
            rows = n if n * k <= (1 << 26) else max(64, (1 << 26) // k)
            sel = np.linspace(0, n - 1, rows).astype(np.int64)
            w = synth.q4_rows(sel, k, 0, tid).reshape(-1)
            x = synth.activations(1, k, 0)
            t0 = time.perf_counter()
            ora.gemv(w, x, rows, k, threads=cores)
            t_total += time.perf_counter() - t0
            done_bytes += rows * k // 32 * 18
            if t_total >= budget_s:
                break
        done_layers += 1
        if t_total >= budget_s:
            break
    gbs = done_bytes / t_total / 1e9
    return gbs, cores, done_bytes, t_total


def cpu_attn_rate(budget_s: float):
    """The oracle's decode attention (fp64) on 8B heads, context 4096, one
    layer's cache after another until budget_s passes (one host thread)."""
    import numpy as np

    import oracle as ora
    n_q, n_kv, hd, ctx = 32, 8, 128, 4096
    rng = np.random.default_rng(0)
    q = rng.normal(size=n_q * hd) * 0.25
    done, t_total = 0, 0.0
    while t_total < budget_s:
        kc = rng.normal(size=(ctx, n_kv * hd)).astype(np.float16).view(np.uint16)
        vc = rng.normal(size=(ctx, n_kv * hd)).astype(np.float16).view(np.uint16)
        t0 = time.perf_counter()
        ora.attn_decode(q, kc, vc, ctx, n_q, n_kv, hd)
        t_total += time.perf_counter() - t0
        done += 2 * ctx * n_kv * hd * 2
    return done / t_total / 1e9, 1, done, t_total


# ------------------------------------------------------------------ main

def extra_result(r, steps, peak):
    """Short summary of another workload's run, added to the default line."""
    per_step = r["secs"] / steps
    kl = r.get("kernel_launches_per_step", r["launches_per_step"])
    achieved = r["bytes_per_step"] / per_step / 1e9
    d = {"workload": r["workload"], "ms_per_token": round(per_step * 1e3, 4), "tokens_per_s": round(1 / per_step, 2),
         "gbs": round(achieved, 2), "hbm_frac_of_measured": round(achieved / peak, 4),
         "launches_per_token": r["launches_per_step"], "engine_launches_per_token": kl, "steps": steps,
         "clocks_sm_mhz": (r["clocks"] or {}).get("sm_mhz")}
    if "streamed_bytes_per_step" in r:
        sb = r["streamed_bytes_per_step"]
        d["host_link"] = {"achieved_gbs": round(sb / per_step / 1e9, 2),
                          "pinned_h2d_peak_gbs": round(r["h2d_peak_gbs"], 2),
                          "frac": round(sb / per_step / 1e9 / r["h2d_peak_gbs"], 4) if sb else None,
                          "streamed_bytes_per_token": sb, "distinct_host_layers": r["distinct"],
                          "peak_by_concurrent_streams": r["h2d_streams"], "numa": r["numa"]}
        d["timelines"] = r["timelines"]
        d["hbm_frac_of_measured"] = None
        d["gbs_note"] = "weight bytes per token over the token time, most of them copied over the host link"
    if "residency_sweep" in r:
        d["modes"] = r["residency_sweep"]
    if "kv_contexts" in r:
        d["kv_contexts"] = r["kv_contexts"]
        d["weight_bytes_per_token"] = r["weight_bytes_per_step"]
        d["gbs_note"] = "weight bytes and KV-cache bytes read per token over the token time"
    return d


def run_extras(args, torch, q4, model, synth, stream, barrier, gpu_index, peak):
    import copy
    extras = {}
    for name, runner, overrides in (("70b", run_stack, {}), ("70b_stream", run_stream, {"resident_frac": 0.0, "with_single": True}),
                                    ("8b_kv", run_kv, {})):
        a = copy.copy(args)
        a.config = {"70b": "70b", "70b_stream": "70b-stream", "8b_kv": "8b-kv"}[name]
        a.steps, a.warmup, a.layers = min(args.steps, 50), min(args.warmup, 5), 0
        for k, v in overrides.items():
            setattr(a, k, v)
        try:
            r = runner(a, torch, q4, model, synth, stream, barrier, gpu_index)
            extras[name] = extra_result(r, r.get("steps_override", a.steps), peak)
        except Exception as e:   # an extra never hides the headline number
            extras[name] = {"failed": f"{type(e).__name__}: {e}"}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return extras


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="8b",
                    choices=["8b", "gemv", "70b", "70b-stream", "stream-sweep", "sweep", "attn", "8b-kv"])
    ap.add_argument("--kv-contexts", default="1024,4096",
                    help="8b-kv: contexts timed (multiples of 128); the last one is the line's value")
    ap.add_argument("--resident-frac", type=float, default=0.0,
                    help="70b-stream: fraction of the layers (a prefix) kept resident in HBM")
    ap.add_argument("--chunked", action="store_true", help="70b-stream: copy each layer as four chunks")
    ap.add_argument("--single-buffer", action="store_true",
                    help="70b-stream: one staging buffer (memory-efficient mode)")
    ap.add_argument("--with-single", action="store_true",
                    help="70b-stream: also time the single-buffer mode (merged and chunked) on the same blocks")
    ap.add_argument("--resident-pattern", default="prefix", choices=["prefix", "spread"],
                    help="70b-stream: which layers stay resident")
    ap.add_argument("--batch", type=int, default=1, help="activation rows per step (1..16)")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--layers", type=int, default=0, help="run only this many layers of the stack (profiling)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline (profiling runs)")
    ap.add_argument("--no-extras", action="store_true",
                    help="8b at N=1: skip the 70b, 70b-stream and 8b-kv results added to the line")
    ap.add_argument("--cuda-core", action="store_true",
                    help="batch-1 stacks and rings: the CUDA-core engine instead of the tensor-core one (comparison)")
    ap.add_argument("--barrier", action="store_true",
                    help="batch-1 stacks: flag barrier after every phase instead of tagged words (comparison)")
    ap.add_argument("--batch-engine", action="store_true",
                    help="batch 2..8 stacks: the persistent batched engine instead of one product launch per "
                         "projection (comparison)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank, world, local_rank = dist_env()

    if args.impl == "reference":
        return main_reference(args, rank, world)

    import torch
    import weight_streaming_q4_gb300 as q4
    from weight_streaming_q4_gb300 import build as qbuild, model, synth
    qbuild.build()
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        barrier = lambda: dist.barrier()
    else:
        barrier = lambda: None
    stream = torch.cuda.Stream()
    if not 1 <= args.batch <= 16 or (args.batch != 1 and args.config not in ("8b", "70b", "70b-stream",
                                                                               "stream-sweep")):
        raise SystemExit("--batch: 1..16, for the 8b, 70b and stream configs")
    runner = {"8b": run_stack, "70b": run_stack, "gemv": run_gemv, "70b-stream": run_stream,
              "stream-sweep": run_stream, "sweep": run_sweep, "attn": run_attn, "8b-kv": run_kv}[args.config]
    r = runner(args, torch, q4, model, synth, stream, barrier, local_rank)
    steps = r.get("steps_override", args.steps)
    warmup = r.get("warmup_override", args.warmup)
    secs = r["secs"]
    if world > 1:
        secs = max_over_ranks(secs, "cuda")
    per_step = secs / steps
    gbs = whole_job_gbs(r["bytes_per_step"], world, per_step)
    peak, peak_kind = peaks()
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    # the dominant kernel's launches carry all the weight bytes; with one launch
    # per step (batch 1 resident) its duration is the step's, otherwise the
    # step time (glue launches included) divided among its launches bounds it
    kl = r.get("kernel_launches_per_step", r["launches_per_step"])
    per_launch_s = per_step / kl
    bytes_per_launch = r["bytes_per_step"] / kl
    out = {
        "metric": METRIC,
        "value": round(gbs, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": round(per_step * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "q4_0 weights x f16 activations, f32 accumulate",
        "data": "synthetic (seeded Philox: uniform 4-bit codes, |N(0,0.02)| binary16 scales, N(0,1) binary16 x)",
        "config": {"workload": r["workload"], "batch": args.batch, "parallelism": f"replicas x{world}",
                   "l2": "weights per step exceed L2 (no flush needed)"},
    }
    if "tagged" in r:
        out["config"]["phase_sync"] = "tagged words" if r["tagged"] else "flag barrier per phase"
    if args.config in ("8b", "70b"):
        out["tokens_per_s"] = round(world * args.batch / per_step, 2)
        out["config"]["n_layers"] = r["n_layers"]
        out["config"]["weight_bytes_per_token"] = r["bytes_per_step"]
    if args.config in ("70b-stream", "stream-sweep"):
        out["tokens_per_s"] = round(world * args.batch / per_step, 3)
        sb = r["streamed_bytes_per_step"]
        out["host_link"] = {"achieved_gbs": round(sb / per_step / 1e9, 2),
                            "pinned_h2d_peak_gbs": round(r["h2d_peak_gbs"], 2),
                            "frac": round(sb / per_step / 1e9 / r["h2d_peak_gbs"], 4) if sb else None,
                            "streamed_bytes_per_token": sb,
                            "peak_by_concurrent_streams": r["h2d_streams"], "numa": r["numa"]}
        out["timelines"] = r["timelines"]
        out["config"]["distinct_host_layers"] = r["distinct"]
        out["host_link"]["host_blocks"] = r["host_blocks"]
        if "residency_sweep" in r:
            out["residency_sweep"] = r["residency_sweep"]
    achieved = bytes_per_launch / per_launch_s / 1e9
    out["roofline"] = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                       "frac": round(achieved / peak, 4), "peak_source": f"hbm_gbs {peak_kind}",
                       "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                       "traffic": ncu_traffic(r["kernel_key"]) if r["kernel_key"] else None,
                       "kernel": r.get("kernel", "engine_kernel"), "bytes_per_launch": int(bytes_per_launch)}
    if kl != 1 or r["launches_per_step"] != 1:
        out["roofline"]["timing"] = "step time / launches of the kernel per step (glue launches included)"
    if "sweep" in r:
        out["sweep"] = r["sweep"]
    if "kv_contexts" in r:
        out["tokens_per_s"] = round(world / per_step, 2)
        out["kv_contexts"] = r["kv_contexts"]
        out["config"]["n_layers"] = r["n_layers"]
        out["config"]["weight_bytes_per_token"] = r["weight_bytes_per_step"]
        out["metric_note"] = "value counts the weight bytes and the KV-cache bytes read per token"
        out["roofline"]["timing"] = ("step time / engine launches per step (one per layer and the first "
                                     "q|k|v; attention and position launches included)")
    if "attn_buckets" in r:
        out["attn_buckets"] = r["attn_buckets"]
        out["metric_note"] = "value = GB/s of KV-cache bytes read (keys and values), not weight bytes"
    if r.get("e2e_secs"):
        e2e_bytes = r.get("e2e_bytes_per_step", r["bytes_per_step"])
        out["e2e"] = {"value": round(e2e_bytes / (r["e2e_secs"] / r["e2e_steps"]) / 1e9, 2), "unit": "GB/s",
                      "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                      "ms_per_step": round(r["e2e_secs"] / r["e2e_steps"] * 1e3, 4)}
        if r.get("e2e_note"):
            out["e2e"]["note"] = r["e2e_note"]
    out["gpu_launches"] = r["launches_per_step"] * steps
    out["clocks"] = r["clocks"]
    if args.config == "8b" and args.batch == 1 and world == 1 and not args.no_extras and not args.layers:
        out["extra"] = run_extras(args, torch, q4, model, synth, stream, barrier, local_rank, peak)
    # the CPU oracle on a bounded sample of the same workload (rank 0 only)
    if args.no_cpu:
        out["cpu_baseline"] = None
        print(json.dumps(out), flush=True)
        return
    try:
        if args.config == "attn":
            gbs_cpu, cores, nbytes, t = cpu_attn_rate(args.cpu_budget)
        else:
            gbs_cpu, cores, nbytes, t = cpu_oracle_rate("gemv" if args.config == "gemv" else
                                                        ("8b" if args.config in ("8b", "sweep", "8b-kv") else "70b"),
                                                        args.cpu_budget)
        what = ("KV-cache bytes of whole 8B-head attention calls at context 4096" if args.config == "attn" else
                "weight bytes of row-sampled projections of the same workload")
        out["cpu_baseline"] = {"value": round(gbs_cpu, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                               "sample": f"{nbytes} {what} in {t:.1f} s, fp64, {cores} threads"}
    except Exception as e:  # the baseline is context; never hide the GPU number
        out["cpu_baseline"] = {"value": None, "unit": "GB/s", "cores": 0, "kind": "oracle", "sample": f"failed: {e}"}
    print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def reference_config(args, world):
    """The native arm's config for the same flags (the reference arm times the oracle on it)."""
    if args.config == "gemv":
        return {"workload": "single Q4_0 product N=K=4096, batch 1", "batch": 1,
                "parallelism": f"replicas x{world}"}
    name = "8b" if args.config in ("8b", "sweep", "8b-kv") else "70b"
    cfg, n_layers = stack_cfg(name)
    if args.layers:
        n_layers = args.layers
    from weight_streaming_q4_gb300 import synth
    layer_bytes = sum(n * k // 32 * 18 for n, k in synth.layer_dims(cfg["hidden"], cfg["q_dim"], cfg["kv_dim"],
                                                                       cfg["ffn"]))
    return {"workload": (f"{'8B' if name == '8b' else '70B'}-shaped decoder stack, {n_layers} layers, "
                         f"batch {args.batch}, HBM-resident, one CUDA-graph replay per step"),
            "batch": args.batch, "parallelism": f"replicas x{world}",
            "l2": "weights per step exceed L2 (no flush needed)", "n_layers": n_layers,
            "weight_bytes_per_token": layer_bytes * n_layers}


def main_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg_name = "gemv" if args.config == "gemv" else ("8b" if args.config == "8b" else "70b")
    # each step: a bounded sample of the workload (row-sampled projections) on all host cores
    per_step_budget = max(0.02, min(0.15, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_oracle_rate(cfg_name, per_step_budget)
    tot_bytes, tot_t = 0, 0.0
    cores = os.cpu_count() or 1
    for _ in range(args.steps):
        gbs, cores, nbytes, t = cpu_oracle_rate(cfg_name, per_step_budget)
        tot_bytes += nbytes
        tot_t += t
    value = tot_bytes / tot_t / 1e9
    out = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "q4_0 weights x f16 activations, f64 accumulate",
        "data": "synthetic (seeded Philox, same recipe as the native arm)", "impl": "reference",
        "config": reference_config(args, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": (f"{tot_bytes} weight bytes of row-sampled projections of the same workload "
                                    f"over {args.steps} steps ({per_step_budget:.2f} s of oracle time each), "
                                    f"fp64, {cores} threads")},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
