"""CSA2 layer benchmark on GB300.

One step = the whole hot path over one batch: csa2_write_cache -> csa2_index_topk ->
csa2_attend, on seeded synthetic inputs already resident in HBM.  The headline workload is
the T=4096 prefill from an empty cache (prefill_4k); the 1M-context decode (decode_1m,
B=8) is measured in the same run and reported under "decode".  A decode step (T = 1) is
timed both as the three calls launched one by one and as one replay of a CUDA graph that holds
them, with the positions read from device memory (the way a serving loop runs decode); the
graph replay is the decode objects' ms_per_step.  L2 is flushed (a 256 MiB write) before every
timed step; each step is timed with CUDA events on the launch stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs its own replica of the workload (independent sequences,
no data-path collective): value = all ranks' tokens / max step time over ranks.
--impl reference times the fp64 CPU oracle on the host cores on a bounded sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time
from pathlib import Path

import numpy as np
import torch

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "CSA2 decode tok/s & prefill tok/s on 1 GB300; % of HBM / tensor-core roofline"
H, D, DI, HI = 64, 512, 128, 32


# ------------------------------------------------------------------ distributed plumbing
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, ws


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist

    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def seed_for_rank(base: int, rank: int) -> int:
    """Each rank draws its own independent sequences (weak scaling)."""
    return base + 1000 * rank


# ------------------------------------------------------------------ work models
def attention_rows(p0: int, T: int, ratio: int = 2) -> np.ndarray:
    t = p0 + np.arange(T, dtype=np.int64)
    return np.minimum(128, t + 1) + np.minimum(512, (t + 1) // ratio)


def attention_flops(B: int, p0: int, T: int, ratio: int = 2) -> float:
    """QG^T and AG: 2 * 2 * 64 * n_t * 512 flops per query."""
    return float(B * 4 * H * D * attention_rows(p0, T, ratio).sum())


def indexer_pairs(B: int, p0: int, T: int, ratio: int = 2) -> int:
    t = p0 + np.arange(T, dtype=np.int64)
    return int(B * ((t + 1) // ratio).sum())


def hsi_bytes(B: int, p0: int, ratio: int = 2) -> dict:
    """Algorithmic HBM bytes of the hierarchical indexer at decode (T=1): the owner layer reads
    every visible key (68 B) and writes the top-512 and the 2048-block pool; a later layer reads
    its pool and the keys of at most 2048 blocks of 8 and writes its top-512."""
    E = (p0 + 1) // ratio
    q = HI * DI * 2 + HI * 2
    n_re = min(E, 8 * 2048)
    return dict(owner=B * (E * 68 + q + 512 * 4 + 2048 * 4), reindex=B * (2048 * 4 + n_re * 68 + q + 512 * 4))


def decode_bytes(B: int, p0: int, ratio: int = 2) -> dict:
    """Algorithmic HBM bytes of one decode step (T=1): indexer keys over all visible entries,
    the 512 selected Z rows, 128 window rows, Q, Q^I, w^I, the output, the step's writes."""
    E = (p0 + 1) // ratio
    k = min(512, E)
    idx_keys = B * E * 68
    rows = B * (k * 272 + min(128, p0 + 1) * 512)
    small = B * (H * D * 2 + HI * DI * 2 + HI * 2 + H * D * 2 + 3 * D * 2 + D + 512 * 4)
    return dict(indexer=idx_keys, step=idx_keys + rows + small)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampled every 50 ms from before the timed region; summary() keeps the samples
    whose timestamps fall inside the window marked by mark_start() / mark_end()."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str | None = None):
        self.proc = None
        self.gpu = gpu_index
        # the raw samples: a file the caller names (--clocks-csv), else one in the temp directory
        self.path = Path(path) if path else Path(tempfile.gettempdir()) / f"csa2_clocks_gpu{gpu_index}.csv"

    def __enter__(self):
        try:
            self.path.parent.mkdir(parents=True, exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.5)  # nvidia-smi start-up
        except Exception:
            self.proc = None
        self.t0 = self.t1 = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            self.proc.wait(timeout=5)
            self.f.close()

    def summary(self) -> dict:
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        import datetime as _dt

        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.path.read_text().splitlines():
            p = [x.strip() for x in line.split(",")]
            if len(p) < 10:
                continue
            try:
                ts = _dt.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(p[2]), float(p[3]), p[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 and self.t1 and self.t0 - 0.05 <= r[0] <= self.t1 + 0.05]
        note = "samples within the timed region"
        if not inside:  # region shorter than the sampling period: nearest samples around it
            inside = sorted(rows, key=lambda r: abs(r[0] - (self.t0 or 0)))[:3]
            note = "timed region shorter than the 50 ms sampling period: nearest samples"
        reasons = set()
        for r in inside:
            for nm, v in zip(names, r[3]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        mx = inside[0][2] if inside else None
        return {"sm_mhz": statistics.median(r[1] for r in inside) if inside else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(inside), "note": note}


# ------------------------------------------------------------------ our implementation
class Step:
    """Resident buffers and the three C-ABI calls of one workload step."""

    def __init__(self, csa2, inputs, wl, seed, dev):
        self.csa2, self.wl = csa2, wl
        x = {}
        x.update(inputs.layer_params(seed, dev))
        x.update(inputs.step_inputs(wl.B, wl.T, seed, dev))
        x.update(inputs.cache_state(wl.B, wl.T, wl.p0, wl.cap, seed, dev, wl.ratio))
        self.x = x
        self.h = csa2.csa2_create(ratio=wl.ratio)
        self.p0 = [wl.p0] * wl.B
        self.idx = torch.empty(wl.B, wl.T, 512, dtype=torch.int32, device=dev)
        self.out = torch.empty(wl.B, wl.T, H, D, dtype=torch.bfloat16, device=dev)
        self.ws_i = csa2.workspace(self.h, csa2.OP_INDEX_TOPK, wl.B, wl.T, wl.cap, dev)
        self.ws_a = csa2.workspace(self.h, csa2.OP_ATTEND, wl.B, wl.T, 0, dev)

    def write(self, s):
        x = self.x
        self.csa2.csa2_write_cache(self.h, x["kc"], x["gc"], x["wa"], x["gamma_c"], x["w_ik"], x["gamma_ik"],
                                   x["gamma_w"], self.p0, x["z_codes"], x["z_scales"], x["ki_codes"], x["ki_scales"],
                                   x["window"], x["pair_kc"], x["pair_gc"], stream=s)

    def index(self, s):
        x = self.x
        self.csa2.csa2_index_topk(self.h, x["qi"], x["wI"], x["ki_codes"], x["ki_scales"], self.p0, self.idx,
                                  ws=self.ws_i, stream=s)

    def attend(self, s):
        x = self.x
        self.csa2.csa2_attend(self.h, x["q"], x["sinks"], x["z_codes"], x["z_scales"], x["window"], self.idx, self.p0,
                              self.out, ws=self.ws_a, stream=s)


def time_workload(step: Step, steps: int, warmup: int, ws: int, flush: torch.Tensor, clocks=None):
    s = torch.cuda.current_stream()
    names = ("write", "index", "attend")
    for _ in range(warmup):
        step.write(s); step.index(s); step.attend(s)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    barrier(ws)
    torch.cuda.synchronize()
    ctx = clocks if clocks is not None else _Null()
    launches0 = step.csa2.csa2_kernel_launches()
    with ctx:
        if clocks is not None:
            clocks.mark_start()
        for i in range(steps):
            flush.zero_()  # evict L2 before each step (not timed)
            e = ev[i]
            e[0].record(s)
            step.write(s)
            e[1].record(s)
            step.index(s)
            e[2].record(s)
            step.attend(s)
            e[3].record(s)
        torch.cuda.synchronize()
        if clocks is not None:
            clocks.mark_end()
    launches = step.csa2.csa2_kernel_launches() - launches0  # the library's own kernels, timed steps only
    barrier(ws)
    per = {n: [ev[i][k].elapsed_time(ev[i][k + 1]) for i in range(steps)] for k, n in enumerate(names)}
    total = [sum(per[n][i] for n in names) for i in range(steps)]
    return statistics.mean(total), {n: statistics.mean(v) for n, v in per.items()}, launches


def time_decode_graph(csa2, step: Step, steps: int, warmup: int, ws: int, flush: torch.Tensor):
    """The decode step as a serving loop runs it: the three calls captured once in a CUDA graph,
    with the positions read from device memory (csa2_set_device_positions), one replay per step
    (L2 flushed before each).  The replays' indices and outputs are compared bit for bit with
    those of the eager calls timed just before (same inputs, same positions)."""
    wl, dev = step.wl, step.idx.device
    s = torch.cuda.current_stream()
    ref_idx, ref_out = step.idx.clone(), step.out.clone()
    hg = csa2.csa2_create(ratio=wl.ratio)
    p0_dev = torch.tensor(step.p0, dtype=torch.int64, device=dev)
    csa2.csa2_set_device_positions(hg, p0_dev, wl.p0)
    h_eager, step.h = step.h, hg
    try:
        step.write(s); step.index(s); step.attend(s)  # uncaptured: loads the kernels
        torch.cuda.synchronize()
        g, cs = torch.cuda.CUDAGraph(), torch.cuda.Stream()
        cs.wait_stream(s)
        n0 = csa2.csa2_kernel_launches()
        with torch.cuda.stream(cs):
            with torch.cuda.graph(g, stream=cs):
                c = torch.cuda.current_stream()
                step.write(c); step.index(c); step.attend(c)
        per_replay = csa2.csa2_kernel_launches() - n0  # the library's kernels in the graph
        s.wait_stream(cs)
        torch.cuda.synchronize()
        step.idx.zero_(); step.out.zero_()
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        barrier(ws)
        torch.cuda.synchronize()
        for i in range(steps):
            flush.zero_()
            ev[i][0].record(s)
            g.replay()
            ev[i][1].record(s)
        torch.cuda.synchronize()
        barrier(ws)
        identical = bool(torch.equal(step.idx, ref_idx) and torch.equal(step.out, ref_out))
        checked = csa2.csa2_check(hg) == 0
        del g
    finally:
        step.h = h_eager
        hg.close()
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    return {"ms_per_step": ms, "identical_to_eager": identical and checked, "gpu_launches": per_replay * steps}


def time_hsi(csa2, step: Step, steps: int, warmup: int, ws: int, flush: torch.Tensor):
    """Owner layer (csa2_index_pool) and a later layer (csa2_reindex_topk over that pool), one
    after the other on the step's resident queries and keys; per-call device times."""
    wl, x, dev = step.wl, step.x, step.idx.device
    pool = torch.empty(wl.B, wl.T, csa2.HSI_BLOCKS, dtype=torch.int32, device=dev)
    idx2 = torch.empty_like(step.idx)
    ws_p = csa2.workspace(step.h, csa2.OP_INDEX_POOL, wl.B, wl.T, wl.cap, dev)
    ws_r = csa2.workspace(step.h, csa2.OP_REINDEX_TOPK, wl.B, wl.T, wl.cap, dev)
    s = torch.cuda.current_stream()

    def owner():
        csa2.csa2_index_pool(step.h, x["qi"], x["wI"], x["ki_codes"], x["ki_scales"], step.p0, step.idx, pool,
                             ws=ws_p, stream=s)

    def later():
        csa2.csa2_reindex_topk(step.h, x["qi"], x["wI"], x["ki_codes"], x["ki_scales"], step.p0, pool, idx2,
                               ws=ws_r, stream=s)

    for _ in range(warmup):
        owner(); later()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    barrier(ws)
    torch.cuda.synchronize()
    launches0 = csa2.csa2_kernel_launches()
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(s)
        owner()
        ev[i][1].record(s)
        later()
        ev[i][2].record(s)
    torch.cuda.synchronize()
    launches = csa2.csa2_kernel_launches() - launches0
    barrier(ws)
    own = statistics.mean(ev[i][0].elapsed_time(ev[i][1]) for i in range(steps))
    re = statistics.mean(ev[i][1].elapsed_time(ev[i][2]) for i in range(steps))
    return own, re, launches


def time_out_proj(csa2, inputs, M, steps, warmup, ws, flush, bf16, src, rank):
    """The grouped output projection W_OA on M attention-output rows (prefill_4k: M = 4096)."""
    x = inputs.out_proj_inputs(M, seed_for_rank(1, rank), "cuda")
    h = csa2.csa2_create()
    out = torch.empty(M, 8, 1024, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        csa2.csa2_out_group_proj(h, x["o"], x["w_oa"], out, stream=s)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(ws)
    launches0 = csa2.csa2_kernel_launches()
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(s)
        csa2.csa2_out_group_proj(h, x["o"], x["w_oa"], out, stream=s)
        ev[i][1].record(s)
    torch.cuda.synchronize()
    launches = csa2.csa2_kernel_launches() - launches0
    barrier(ws)
    ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in ev), ws)
    flops = 2.0 * M * 8 * 1024 * 4096
    tf = flops / (ms / 1e3) / 1e12
    return {"rows": M, "ms": ms, "gpu_launches": launches,
            "roofline": {"kernel": "outproj_kernel", "bound": "tensor", "achieved": tf, "peak": bf16,
                         "unit": "TFLOP/s", "frac": tf / bf16, "flops_per_launch": flops,
                         "peak_source": f"{src} bf16 burst",
                         "traffic": profiled_traffic("outproj_kernel_prefill_4k.md", OUTPROJ_SOURCES) if M == 4096
                         else None}}


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def time_e2e(step: Step, steps: int, warmup: int):
    """Same metric through the public API with HOST buffers.  Every step copies its inputs
    from pinned host memory, runs the three calls and reads its output back; as in a serving
    pipeline the copies overlap the neighbouring steps' compute: two device buffer sets, one
    stream each for host-to-device copies, compute and device-to-host copies."""
    x, wl = step.x, step.wl
    keys = ("kc", "gc", "wa", "q", "qi", "wI")
    host = {k: x[k].cpu().pin_memory() for k in keys}
    out_h = [torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory() for _ in range(2)]
    bufs = [dict(x), dict(x)]  # parameters and caches shared; per-step inputs double-buffered
    for k in keys:
        bufs[1][k] = torch.empty_like(x[k])
    outs = [step.out, torch.empty_like(step.out)]
    h2d = sum(host[k].numel() * host[k].element_size() for k in keys)
    d2h = out_h[0].numel() * out_h[0].element_size()
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    e_in, e_run, e_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    csa2 = step.csa2

    def one(i):
        b = i & 1
        xb = bufs[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(e_run[b])  # the compute two steps back is done with these inputs
            for k in keys:
                xb[k].copy_(host[k], non_blocking=True)
            e_in[b].record(s_in)
        s_run.wait_event(e_in[b])
        if i >= 2:
            s_run.wait_event(e_out[b])  # the output of two steps back has been read
        csa2.csa2_write_cache(step.h, xb["kc"], xb["gc"], xb["wa"], xb["gamma_c"], xb["w_ik"], xb["gamma_ik"],
                              xb["gamma_w"], step.p0, xb["z_codes"], xb["z_scales"], xb["ki_codes"], xb["ki_scales"],
                              xb["window"], xb["pair_kc"], xb["pair_gc"], stream=s_run)
        csa2.csa2_index_topk(step.h, xb["qi"], xb["wI"], xb["ki_codes"], xb["ki_scales"], step.p0, step.idx,
                             ws=step.ws_i, stream=s_run)
        csa2.csa2_attend(step.h, xb["q"], xb["sinks"], xb["z_codes"], xb["z_scales"], xb["window"], step.idx, step.p0,
                         outs[b], ws=step.ws_a, stream=s_run)
        e_run[b].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(e_run[b])
            out_h[b].copy_(outs[b], non_blocking=True)
            e_out[b].record(s_out)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(warmup, warmup + steps):
        one(i)
    s_in.wait_stream(s_out)
    z.record(s_in)
    torch.cuda.synchronize()
    ms = a.elapsed_time(z) / steps
    return {"value": wl.B * wl.T / (ms / 1e3), "unit": "tok/s", "ms_per_step": ms, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "overlap": "copies of neighbouring steps overlap compute (2 buffer sets, 3 streams)"}


def profiled_traffic(profile: str, sources) -> int | None:
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from the ncu summary
    under profiles/, or None when the kernel sources changed since that capture."""
    p = ROOT / "profiles" / profile
    if not p.exists():
        return None
    txt = p.read_text()
    sha = re.search(r"source_sha256_16: ([0-9a-f]{16})", txt)
    byt = re.search(r"traffic_bytes_per_launch: (\d+)", txt)
    if not sha or not byt:
        return None
    now = hashlib.sha256(b"".join((ROOT / s).read_bytes() for s in sources)).hexdigest()[:16]
    return int(byt.group(1)) if now == sha.group(1) else None


CSRC = "compressed_sparse_attention_03_gb300/csrc/"
# sources a profiled kernel is built from (a change to any of them makes its ncu traffic stale)
_HDRS = [CSRC + "csa2_common.cuh", CSRC + "csa2_fp16.cuh", CSRC + "csa2_sm100.cuh", CSRC + "csa2_internal.h"]
ATTEND_SOURCES = [CSRC + "csa2_attend.cu"] + _HDRS
INDEX_SOURCES = [CSRC + "csa2_index_tc.cu", CSRC + "csa2_indexer.cu"] + _HDRS
OUTPROJ_SOURCES = [CSRC + "csa2_outproj.cu"] + _HDRS


def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


def decode_object(dw, dms, dper, dlaunches, ws, hbm, src, profile=None, graph=None):
    """Throughput and HBM rooflines of a decode workload (T = 1): the whole step and the index call.
    With `graph` (time_decode_graph), the step's time is the graph replay's; the eager calls'
    total and per-call times stay under eager_ms_per_step and kernels_ms."""
    by = decode_bytes(dw.B, dw.p0, dw.ratio)
    idx_ms = dper["index"]
    eager_ms = dms
    if graph is not None:
        dms = graph["ms_per_step"]
    return {
        "workload": dw.name, "B": dw.B, "p0": dw.p0, "ratio": dw.ratio, "value": ws * dw.B / (dms / 1e3),
        "unit": "tok/s", "ms_per_step": dms, "eager_ms_per_step": eager_ms, "kernels_ms": dper,
        "step_launch": ("one CUDA-graph replay of the three calls, positions read from device memory"
                        if graph is not None else "the three calls launched one by one"),
        "graph": graph,
        "roofline_step": {"bound": "hbm", "achieved": by["step"] / (dms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                          "frac": by["step"] / (dms / 1e3) / 1e9 / hbm, "bytes": by["step"],
                          "peak_source": f"{src} copy bandwidth"},
        "roofline_index": {"bound": "hbm", "achieved": by["indexer"] / (idx_ms / 1e3) / 1e9, "peak": hbm,
                           "unit": "GB/s", "frac": by["indexer"] / (idx_ms / 1e3) / 1e9 / hbm,
                           "bytes": by["indexer"], "peak_source": f"{src} copy bandwidth",
                           "traffic": profiled_traffic(profile, INDEX_SOURCES) if profile else None},
        "gpu_launches": dlaunches,
    }


def measure_tensor_rates(csa2, iters=8192):
    """The tensor-core rate of each MMA kind the kernels use, measured here (csa2_tc_rate)."""
    h = csa2.csa2_create()
    r = {k: csa2.csa2_tc_rate(h, i, iters) for i, k in enumerate(("f16", "e5m2", "mxf4"))}
    h.close()
    r.update({"unit": "TFLOP/s", "source": f"csa2_tc_rate: best of 3 launches, {iters} MMAs M=128 N=256 per SM, "
                                           "operands in shared memory (burst)"})
    return r


def prefill_rooflines(wl, per, bf16, src, ws=1, e5m2=None):
    """Tensor rooflines of a prefill workload: attention (fp16 operands, against the bf16 peak),
    the indexer score GEMM (E5M2 operands on kind::f8f6f4 MMAs: against the measured E5M2 rate
    when given) and the two together (against the bf16 peak)."""
    af = attention_flops(wl.B, wl.p0, wl.T, wl.ratio)
    xf = 8192.0 * indexer_pairs(wl.B, wl.p0, wl.T, wl.ratio)
    a_ach = af / (per["attend"] / 1e3) / 1e12
    x_ach = xf / (per["index"] / 1e3) / 1e12
    both = (af + xf) / ((per["attend"] + per["index"]) / 1e3) / 1e12
    peak_src = f"{src} bf16 burst"
    xpeak = e5m2 if e5m2 else 2.0 * bf16
    xsrc = ("measured kind::f8f6f4 E5M2 MMA rate (csa2_tc_rate, burst)" if e5m2
            else f"{src} bf16 burst x 2 (the nominal E5M2 / bf16 ratio)")
    return {
        "roofline_attend": {"bound": "tensor", "achieved": a_ach, "peak": bf16, "unit": "TFLOP/s", "frac": a_ach / bf16,
                            "flops_per_launch": af, "peak_source": peak_src},
        "roofline_index": {"bound": "tensor", "achieved": x_ach, "peak": xpeak, "unit": "TFLOP/s", "frac": x_ach / xpeak,
                           "flops_per_call": xf, "peak_source": xsrc,
                           "note": "whole csa2_index_topk call: score GEMM + fp32 score rows + top-512 select"},
        "roofline_attend_plus_index": {"bound": "tensor", "achieved": both, "peak": bf16, "unit": "TFLOP/s",
                                       "frac": both / bf16, "flops": af + xf, "peak_source": peak_src},
    }


def run_ours(args, rank, ws):
    import compressed_sparse_attention_03_gb300 as csa2
    from compressed_sparse_attention_03_gb300 import inputs

    dev = "cuda"
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    hbm, bf16, src = peaks()
    rates = measure_tensor_rates(csa2)
    wl = inputs.WORKLOADS[args.workload]
    step = Step(csa2, inputs, wl, seed_for_rank(wl.seed, rank), dev)
    clocks = ClockSampler(torch.cuda.current_device(), args.clocks_csv)
    ms, per, launches = time_workload(step, args.steps, args.warmup, ws, flush, clocks)
    ms_max = max_over_ranks(ms, ws)
    per = {k: max_over_ranks(v, ws) for k, v in per.items()}
    att_ms = per["attend"]
    flops = attention_flops(wl.B, wl.p0, wl.T, wl.ratio)
    achieved = flops / (att_ms / 1e3) / 1e12
    e2e = time_e2e(step, max(2, args.steps // 2), 1)
    e2e["value"] *= ws
    line = {
        "metric": METRIC, "value": ws * wl.B * wl.T / (ms_max / 1e3), "unit": "tok/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "p0": wl.p0, "seed": wl.seed,
                   "l2": "flushed before each timed step (256 MiB write)", "parallelism": f"replicas x{ws}"},
        "kernels_ms": per,
        "roofline": {"kernel": "attend_kernel", "bound": "tensor", "achieved": achieved, "peak": bf16,
                     "unit": "TFLOP/s", "frac": achieved / bf16, "peak_source": f"{src} bf16 burst",
                     "flops_per_launch": flops,
                     "traffic": profiled_traffic("attend_tc_kernel_prefill_4k.md", ATTEND_SOURCES),
                     "traffic_source": "profiles/attend_tc_kernel_prefill_4k.md (null once the kernel changed)"},
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks.summary(),
        "tensor_rates": rates,
    }
    line.update({k: v for k, v in prefill_rooflines(wl, per, bf16, src, e5m2=rates["e5m2"]).items()
                 if k != "roofline_attend"})
    del step
    torch.cuda.empty_cache()
    # the other workloads, one object each: decode at 8K (B=1), 128K (B=64) and 1M (B=8) context,
    # a ratio-1 (decoder owner) layer, and the 32K-token chunk on a 256K-token prefix
    others = [("decode_8k", args.decode8k_workload, None), ("decode_128k", args.decode128k_workload, None),
              ("decode", args.decode_workload, "index_decode_decode_1m.md"),
              ("decode_ratio1", args.ratio1_workload, None), ("chunk_32k", args.chunk_workload, None)]
    for key, name, prof in others:
        if args.no_decode or not name:
            continue
        dw = inputs.WORKLOADS[name]
        dstep = Step(csa2, inputs, dw, seed_for_rank(dw.seed, rank), dev)
        steps = args.steps if dw.T == 1 else max(3, args.steps // 4)
        dms, dper, dlaunches = time_workload(dstep, steps, args.warmup, ws, flush)
        dms = max_over_ranks(dms, ws)
        dper = {k: max_over_ranks(v, ws) for k, v in dper.items()}
        if dw.T == 1:
            graph = time_decode_graph(csa2, dstep, steps, args.warmup, ws, flush)
            graph["ms_per_step"] = max_over_ranks(graph["ms_per_step"], ws)
            line[key] = decode_object(dw, dms, dper, dlaunches, ws, hbm, src, prof, graph)
        else:
            line[key] = {"workload": dw.name, "B": dw.B, "T": dw.T, "p0": dw.p0, "ratio": dw.ratio, "steps": steps,
                         "value": ws * dw.B * dw.T / (dms / 1e3), "unit": "tok/s", "ms_per_step": dms,
                         "kernels_ms": dper, "gpu_launches": dlaunches,
                         **prefill_rooflines(dw, dper, bf16, src, e5m2=rates["e5m2"])}
        del dstep
        torch.cuda.empty_cache()
    if not args.no_decode and args.hsi_workload:
        hw = inputs.WORKLOADS[args.hsi_workload]
        hstep = Step(csa2, inputs, hw, seed_for_rank(hw.seed, rank), dev)
        own_ms, re_ms, hl = time_hsi(csa2, hstep, args.steps, args.warmup, ws, flush)
        own_ms, re_ms = max_over_ranks(own_ms, ws), max_over_ranks(re_ms, ws)
        hb = hsi_bytes(hw.B, hw.p0, hw.ratio)
        line["hsi"] = {
            "workload": hw.name, "B": hw.B, "p0": hw.p0, "ratio": hw.ratio,
            "owner_ms": own_ms, "reindex_ms": re_ms,
            "roofline_owner": {"bound": "hbm", "achieved": hb["owner"] / (own_ms / 1e3) / 1e9, "peak": hbm,
                               "unit": "GB/s", "frac": hb["owner"] / (own_ms / 1e3) / 1e9 / hbm, "bytes": hb["owner"]},
            "roofline_reindex": {"bound": "hbm", "achieved": hb["reindex"] / (re_ms / 1e3) / 1e9, "peak": hbm,
                                 "unit": "GB/s", "frac": hb["reindex"] / (re_ms / 1e3) / 1e9 / hbm,
                                 "bytes": hb["reindex"]},
            "gpu_launches": hl,
        }
        del hstep
    if not args.no_decode and args.out_proj_rows:
        line["out_proj"] = time_out_proj(csa2, inputs, args.out_proj_rows, args.steps, args.warmup, ws, flush, bf16,
                                         src, rank)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_seconds)
    return line


# ------------------------------------------------------------------ the oracle (CPU baseline / reference arm)
def oracle_rows(wl, cores: int) -> np.ndarray:
    """The fixed, seeded query rows both oracle timings sample: 16 per host thread, spread over
    the step (all rows when the step has fewer)."""
    n = min(wl.T, 16 * max(1, cores))
    return np.sort(np.random.default_rng(0).choice(wl.T, size=n, replace=False))


class OracleStep:
    """One sampled oracle step: the writer over every token of one sequence, then indexer, top-512
    and attention for the fixed row sample; the step time is extrapolated per row and sequence."""

    def __init__(self, wl):
        from compressed_sparse_attention_03_gb300 import inputs

        x = {}
        x.update(inputs.layer_params(wl.seed, "cpu"))
        x.update(inputs.step_inputs(wl.B, wl.T, wl.seed, "cpu"))
        x.update(inputs.cache_state(wl.B, wl.T, wl.p0, wl.cap, wl.seed, "cpu", wl.ratio))
        self.wl, self.x = wl, x
        self.cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
        self.rows = oracle_rows(wl, self.cores)

    def run(self):
        """Returns (writer seconds, row seconds) of one sampled step."""
        import oracle

        wl, x, r = self.wl, self.x, self.rows
        f = lambda t: t.float().numpy()
        t0 = time.perf_counter()
        w = oracle.write_seq(f(x["kc"][0]), f(x["gc"][0]), f(x["wa"][0]), f(x["gamma_c"]), f(x["w_ik"]),
                             f(x["gamma_ik"]), f(x["gamma_w"]), wl.p0, wl.cap, z_codes=x["z_codes"][0].numpy().copy(),
                             z_scales=x["z_scales"][0].numpy().copy(), ki_codes=x["ki_codes"][0].numpy().copy(),
                             ki_scales=x["ki_scales"][0].numpy().copy(), pair_k=f(x["pair_kc"][0]),
                             pair_g=f(x["pair_gc"][0]), window_prefix=x["window"][0, :127].numpy(), ratio=wl.ratio)
        t1 = time.perf_counter()
        pos = wl.p0 + r
        sc = oracle.index_scores(pos, f(x["qi"][0][r]), f(x["wI"][0][r]), w["ki_codes"], w["ki_scales"], wl.cap,
                                 ratio=wl.ratio)
        oidx, _, _ = oracle.topk(sc, (pos + 1) // wl.ratio)
        oracle.attend(pos, f(x["q"][0][r]), f(x["sinks"]), w["z_codes"], w["z_scales"], wl.cap, w["window"],
                      wl.p0 - 127, oidx)
        return t1 - t0, time.perf_counter() - t1

    def step_seconds(self, t_write, t_rows):
        """Extrapolated time of the whole step: the writer timed on one sequence, the rows per row."""
        return t_write * self.wl.B + t_rows / len(self.rows) * self.wl.T * self.wl.B

    def describe(self, t_write, t_rows, n_steps):
        wl = self.wl
        return (f"writer over all {wl.T} tokens of 1 sequence + indexer/top-512/attention for the same fixed "
                f"{len(self.rows)} query rows (seeded, 16 per thread), {n_steps} timed pass(es); per pass "
                f"{t_write:.3f} s + {t_rows:.3f} s; step time extrapolated x{wl.T * wl.B / len(self.rows):.1f} "
                f"over rows and sequences")


def cpu_baseline(wl, budget_s: float = 15.0) -> dict:
    """The fp64 oracle, as it stands, on the host cores: the sampled step of OracleStep, repeated
    until about budget_s seconds were spent; tokens/s from the mean extrapolated step time."""
    o = OracleStep(wl)
    o.run()  # untimed: first touch of the inputs and the oracle library
    runs, spent = [], 0.0
    while spent < budget_s or not runs:
        tw, tr = o.run()
        runs.append((tw, tr))
        spent += tw + tr
    tw = statistics.mean(a for a, _ in runs)
    tr = statistics.mean(b for _, b in runs)
    t_step = o.step_seconds(tw, tr)
    return {"value": wl.B * wl.T / t_step, "unit": "tok/s", "cores": o.cores, "kind": "oracle",
            "sample": o.describe(tw, tr, len(runs)), "seconds": spent, "extrapolated_step_s": t_step}


def run_reference(args, rank, ws):
    from compressed_sparse_attention_03_gb300 import inputs

    wl = inputs.WORKLOADS[args.workload]
    o = OracleStep(wl)
    runs = []
    for i in range(args.warmup + args.steps):
        tw, tr = o.run()
        if i >= args.warmup:
            runs.append((tw, tr))
    tw = statistics.mean(a for a, _ in runs)
    tr = statistics.mean(b for _, b in runs)
    t_step = o.step_seconds(tw, tr)
    v = wl.B * wl.T / t_step
    measured = sum(a + b for a, b in runs)
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "p0": wl.p0, "seed": wl.seed,
                       "parallelism": "host cores (OpenMP)"},
            "measured_seconds": measured,
            "note": "each step runs a fixed sample of the step's query rows; ms_per_step is that sample "
                    "extrapolated to the whole step (see cpu_baseline.sample)",
            "cpu_baseline": {"value": v, "unit": "tok/s", "cores": o.cores, "kind": "oracle",
                             "sample": o.describe(tw, tr, len(runs))},
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill_4k")
    ap.add_argument("--decode-workload", default="decode_1m")
    ap.add_argument("--decode8k-workload", default="decode_8k", help="empty: skip")
    ap.add_argument("--decode128k-workload", default="decode_128k", help="empty: skip")
    ap.add_argument("--chunk-workload", default="chunk_32k", help="empty: skip")
    ap.add_argument("--ratio1-workload", default="decode_512k_r1", help="empty: skip the ratio-1 decode object")
    ap.add_argument("--out-proj-rows", type=int, default=4096, help="0: skip the output-projection object")
    ap.add_argument("--hsi-workload", default="decode_1m", help="empty: skip the hierarchical-indexer object")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--clocks-csv", default=None, help="where to keep the raw nvidia-smi samples (default: temp dir)")
    args = ap.parse_args()
    if args.impl == "reference":
        # the oracle runs on rank 0's host cores only; the other ranks exit without work
        rank, ws = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
        if rank == 0:
            print(json.dumps(run_reference(args, rank, ws)), flush=True)
        return
    rank, ws = dist_setup()
    line = run_ours(args, rank, ws)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
