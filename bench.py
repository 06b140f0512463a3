#!/usr/bin/env python3
"""Benchmark: paged KV insert (RoPE + MXFP8) + dequant-gather round trip on GB300.

One step = kv_insert of 16384 bf16 tokens into a V4.1 (528 B record) paged cache
of 512 pages x 64 slots, then kv_gather of the same 16384 slot ids (the -1 ones
come back as zeros) into bf16 [16384, 512].  Metric: tokens per second.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0:
  value      exactly K steps per timed region, as replays of captured CUDA graphs of at
             most 60 steps; consecutive regions fill at least 0.3 s (CUDA events around
             each region on the launching stream, a barrier and a device synchronise on
             both sides of the whole timed span); value = K steps over the median region
             (max over ranks), `timing` gives the spread; six input sets (~300 MB
             together, more than the 126 MB L2) rotate across steps and regions so no
             step finds its inputs in L2;
  early_metadata  the same graph with the early_metadata launch option (beside value);
  roofline   the dominant kernel's algorithmic bytes over its mean launch time, timed as
             back-to-back launches of that kernel alone in a graph over the same sets,
             against the measured HBM copy bandwidth; DRAM traffic from the recorded ncu
             capture while the kernel sources are unchanged; torch's elementwise kernel
             moving the same bytes, for scale;
  kernels    both kernels back to back, with event nodes around them, and alone after an
             L2 flush;
  e2e        the same step through the public API from pinned host memory, uploads,
             kernels and downloads pipelined on three streams (serial and copies-only
             figures beside it);
  sweep      kernel-only times of the other workloads (N = 1);
  cpu_baseline  the CPU oracle on one core and on every core (N = 1);
  clocks     nvidia-smi samples during the timed region.

`--impl reference` times the CPU oracle (test infrastructure) on the same workload on
every host core, each run held to a few minutes.  `--profile WORKLOAD` runs one
workload's kernels a few times for profiler captures.  Under torchrun with N > 1 every
rank runs its own replica (no collective on the data path; weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import shutil
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "KV insert+gather tokens/s and HBM GB/s (% of GB300 peak) at 1 GPU"
WORKLOAD = "roundtrip_v41_16384"
FALLBACK_HBM_GBS = 6800.0
ROTATE = 6            # input sets rotated through the steps
GRAPH_STEPS = 60      # steps per captured graph at most (a multiple of ROTATE)
REGION_SECONDS = 0.3  # the timed regions together last at least this long
MAX_REGIONS = 20000


# the arithmetic type the path computes in: bf16 inputs are widened exactly to fp32, the
# rotation and the scale decision run on fp32 values, e4m3 codes are cast from fp32; the
# storage types of every stage are listed beside it
DTYPE = "fp32"
DTYPES = {"arithmetic": "fp32", "kv_in": "bf16", "cos_sin": "fp32",
          "record": "e4m3 codes + ue8m0 scales (528 B)", "gather_out": "bf16"}


def workload_config(case) -> dict:
    """The workload of a bench line: the same dict for both arms (the GPU kernels and the
    CPU oracle run the same step over the same inputs)."""
    return {"workload": WORKLOAD, "record": case.record, "tokens": int(case.num_tokens),
            "block_size": case.block_size, "num_pages": case.num_pages,
            "gathered": int(case.indices.size),
            "l2": f"GPU arm: inputs larger than L2 ({ROTATE} input sets rotated through the "
                  "steps, ~300 MB together)"}


# ----------------------------------------------------------------------------- setup

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=48000)
    ap.add_argument("--warmup", type=int, default=60)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the larger-workload kernel sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU time budget of the oracle baseline sample")
    ap.add_argument("--profile", default=None, metavar="WORKLOAD",
                    help="run only this workload's kernel(s) a few times (for profiler "
                         "captures) and print their CUDA-event times; WORKLOAD is one of "
                         "workloads.PROFILE_WORKLOADS, or fp8_<insert workload> for the same "
                         "insert into an fp8 cache")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--insert-stream-min", type=int, default=None, metavar="TOKENS",
                    help="token count from which inserts use the streaming kernel "
                         "(default: the library's)")
    return ap.parse_args(argv)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def reduce_max(value: float, dist=None) -> float:
    """Max of a host scalar over all ranks (a timing reduction, not a data-path
    collective).  With no process group it returns the value unchanged."""
    if dist is None:
        return value
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist=None):
    if dist is not None:
        dist.barrier()


def measured_peaks() -> tuple[float, str]:
    p = ROOT / "MEASURED_PEAKS.json"
    try:
        v = float(json.loads(p.read_text())["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs: STREAM-style copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 measurement)"


def code_only(text: str) -> str:
    """C++ source without its comments, whitespace runs collapsed to one space: what the
    compiler sees, so that a comment edit leaves a capture's record valid."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":                                   # string or character literal
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code (every .cu / .cuh / .h of the extension, comments
    and whitespace removed)."""
    h = hashlib.sha256()
    csrc = ROOT / "gather_kv_rope_gb300" / "csrc"
    for f in sorted(list(csrc.glob("*.cu")) + list(csrc.glob("*.cuh")) + list(csrc.glob("*.h"))):
        h.update(f.name.encode())
        h.update(code_only(f.read_text(encoding="utf-8")).encode())
    return h.hexdigest()[:16]


def ncu_record(kernel: str, workload: str):
    """The line of profiles/ncu_traffic.txt recorded from an ncu capture of `kernel` on
    `workload` (DRAM bytes per launch, and the serialised launch time where recorded), or
    None when absent or taken on a different kernel source."""
    f = ROOT / "profiles" / "ncu_traffic.txt"
    if not f.exists():
        return None
    src = kernel_source_hash()
    for line in f.read_text().splitlines():
        kv = dict(p.split("=", 1) for p in line.split() if "=" in p)
        if kv.get("kernel") == kernel and kv.get("workload") == workload \
                and kv.get("source_hash") == src:
            return kv
    return None


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch recorded from an ncu capture, or None."""
    kv = ncu_record(kernel, workload)
    return None if kv is None else int(kv["dram_bytes_per_launch"])


def ncu_dram_rate(kernel: str, workload: str, peak: float):
    """DRAM bytes over the serialised, cold launch time of a full-size ncu capture, as
    GB/s and as a fraction of the measured peak; None when not recorded."""
    kv = ncu_record(kernel, workload)
    if kv is None or "ncu_us" not in kv:
        return None
    b, us = int(kv["dram_bytes_per_launch"]), float(kv["ncu_us"])
    return {"dram_bytes": b, "us": us, "gbs": b / (us * 1e-6) / 1e9,
            "frac_of_peak": b / (us * 1e-6) / 1e9 / peak,
            "what": "ncu DRAM read + write bytes of one launch over its duration, serialised "
                    "with cold caches (profiles/ncu_traffic.txt)"}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ["timestamp", "clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.active", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.samples: list[tuple[float, list[str]]] = []
        self.proc = None
        self.error = None

    def start(self):
        exe = shutil.which("nvidia-smi")
        if exe is None:
            self.error = "nvidia-smi not found"
            return self
        try:
            self.proc = subprocess.Popen(
                [exe, f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", self.gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError as e:
            self.error = str(e)
            return self
        first = threading.Event()

        def reader():
            for line in self.proc.stdout:
                self.samples.append((time.time(), [x.strip() for x in line.split(",")]))
                first.set()
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        first.wait(timeout=5.0)
        return self

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        if self.error:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": self.error}
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        note = f"{len(inside)} samples at 20 ms during the timed region"
        if not inside:     # region shorter than the sampling interval: nearest samples
            inside = [s for t, s in self.samples if t0 - 0.25 <= t <= t1 + 0.25]
            note = f"timed region shorter than the sampling interval; {len(inside)} samples within 0.25 s"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "no samples"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[1]) for s in inside if num(s[1]) is not None]
        smax = [num(s[2]) for s in inside if num(s[2]) is not None]
        pw = [num(s[3]) for s in inside if num(s[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in inside for n, v in zip(names, s[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(inside), "note": note}


# ----------------------------------------------------------------------------- bytes

def insert_bytes(slots: np.ndarray, record: int) -> int:
    """Algorithmic bytes of one insert: 16 B (slot + position) per token, plus the
    1024 B bf16 row read and the record written for every valid slot.  The cos/sin
    rows are not counted (a bandwidth-optimal kernel reads each row once)."""
    return 16 * slots.size + int((slots >= 0).sum()) * (1024 + record)


def compressed_insert_bytes(slots: np.ndarray, positions: np.ndarray, ratio: int,
                            record: int) -> int:
    """Algorithmic bytes of one compressed-KV insert: 16 B (slot + position) per token,
    plus the bf16 row read and the record written for every token that is written
    (valid slot and (position + 1) % ratio == 0)."""
    written = int(((slots >= 0) & ((positions + 1) % ratio == 0)).sum())
    return 16 * slots.size + written * (1024 + record)


def csc_bytes(slots: np.ndarray, positions: np.ndarray, ratio: int = 1) -> int:
    """The cos/sin rows an insert reads, reported beside (not inside) the algorithmic
    bytes: 256 B per distinct row among the tokens it writes (the row of position pos,
    or of the group start pos + 1 - ratio in the compressed insert)."""
    w = (slots >= 0) & ((positions + 1) % ratio == 0)
    return 256 * int(np.unique(positions[w] + 1 - ratio).size)


def qside_bytes(slots: np.ndarray, record: int, num_heads: int, num_heads_padded: int,
                q_out_bytes: int = 1024) -> int:
    """Algorithmic bytes of one fused attention write: the KV insert's bytes plus, per
    token, the query heads read (num_heads x 1024 B) and written (num_heads_padded x
    q_out_bytes: 1024 B bf16 or 512 B e4m3, padded heads included)."""
    T = int(np.asarray(slots).size)
    return insert_bytes(slots, record) + T * (1024 * num_heads + q_out_bytes * num_heads_padded)


def logits_bytes(indices: np.ndarray, record: int, num_heads: int) -> int:
    """Algorithmic bytes of one sparse-logits launch: per query its heads read (num_heads
    x 1024 B) and its logits written (num_heads x topk x 4 B); per entry its index (4 B)
    and, when valid, its record (or cache row) read."""
    idx = np.asarray(indices)
    Q, K = idx.shape
    return Q * num_heads * (1024 + 4 * K) + 4 * idx.size + int((idx >= 0).sum()) * record


def logits_flops(indices: np.ndarray, num_heads: int) -> int:
    """Tensor-core FLOPs of one sparse-logits launch: 2 x 512 per (query, head, entry)."""
    return 2 * 512 * num_heads * int(np.asarray(indices).size)


def gather_bytes(indices: np.ndarray, record: int) -> int:
    """Algorithmic bytes of one gather: 4 B index + 1024 B bf16 row written per
    index, plus the record read for every valid index."""
    return indices.size * (4 + 1024) + int((indices >= 0).sum()) * record


# ----------------------------------------------------------------------------- GPU arm

def _timing_event(torch, external: bool):
    if external:
        return torch.cuda.Event(enable_timing=True, external=True)
    return torch.cuda.Event(enable_timing=True)


def _supports_external_events(torch) -> bool:
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        return True
    except TypeError:
        return False


def device_sets(case, device, n_sets: int, record: int | None = None, clone_kv: bool = True):
    """n_sets copies of the case's inputs on the device, each with its own cache (of
    the case's record, or of `record`) and gather output (kv shared when not clone_kv)."""
    import torch
    import gather_kv_rope_gb300 as gkr
    record = case.record if record is None else record
    kv = torch.from_numpy(case.kv.view(np.int16)).view(torch.bfloat16).to(device)
    slots = torch.from_numpy(case.slots).to(device)
    pos = torch.from_numpy(case.positions).to(device)
    csc = torch.from_numpy(case.csc).to(device)
    idx = torch.from_numpy(case.indices).to(device) if case.indices is not None else None
    sets = []
    for _ in range(n_sets):
        sets.append(dict(
            kv=kv.clone() if clone_kv else kv, slots=slots.clone(), pos=pos.clone(), csc=csc,
            idx=None if idx is None else idx.clone(),
            cache=gkr.alloc_cache(case.num_pages, case.block_size, record, device, fill=0),
            out=None if idx is None else torch.empty(case.indices.shape + (512,),
                                                     dtype=torch.bfloat16, device=device)))
    return sets


def compressed_sets(case, device, alg_bytes: int):
    """Input sets for a compressed insert, which reads only its group-boundary tokens' rows:
    set k reads kv through the window [k, k + T) of one buffer of T + n rows (k < R, so each
    set's boundary tokens read other rows) and owns its slots, positions and cache; n sets
    together touch more than 320 MB (or n = R)."""
    import torch
    R = case.meta["compress_ratio"]
    n_sets = int(min(R, max(1, -(-320_000_000 // alg_bytes))))
    T = case.num_tokens
    kv_big = torch.from_numpy(np.concatenate([case.kv, case.kv[:n_sets]]).view(np.int16)) \
        .view(torch.bfloat16).to(device)
    sets = device_sets(case, device, n_sets, clone_kv=False)
    for k, st in enumerate(sets):
        st["kv"] = kv_big[k:k + T]
    return sets


def step(gkr, case, s, ev=None):
    """One pass of the hot path on one input set; optional events around each kernel."""
    if ev is not None:
        ev[0].record()
    gkr.kv_insert(s["kv"], s["cache"], s["slots"], s["pos"], s["csc"], case.block_size,
                  case.record)
    if ev is not None:
        ev[1].record()
    if s["idx"] is not None:
        gkr.kv_gather(s["cache"], s["idx"], s["out"])
        if ev is not None:
            ev[2].record()


def capture_steps(torch, device, body, n: int):
    """body(0) once on a side stream (lazy set-up stays out of the capture), then
    body(0) .. body(n-1) captured into one CUDA graph, replayed once untimed."""
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        body(0)
    torch.cuda.current_stream(device).wait_stream(side)
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for k in range(n):
            body(k)
    g.replay()
    torch.cuda.synchronize(device)
    return g


def stream_same_bytes(torch, device, nbytes: int, peak: float, replays: int = 5) -> dict:
    """torch's elementwise kernel (fp32 negation, nbytes/2 read and nbytes/2 written)
    launched back to back in a CUDA graph over rotating buffer pairs that together exceed
    L2: what a plain streaming kernel reaches at that transfer size, launch and ramp-up
    included."""
    n = nbytes // 8
    pairs = [(torch.ones(n, dtype=torch.float32, device=device),
              torch.empty(n, dtype=torch.float32, device=device))
             for _ in range(int(max(1, -(-320_000_000 // (8 * n)))))]
    per_graph = max(12, len(pairs))
    g = capture_steps(torch, device, lambda k: torch.neg(pairs[k % len(pairs)][0],
                                                         out=pairs[k % len(pairs)][1]), per_graph)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(replays):
        g.replay()
    b.record()
    torch.cuda.synchronize(device)
    ms = a.elapsed_time(b) / (per_graph * replays)
    del g, pairs
    torch.cuda.empty_cache()
    return {"bytes": 8 * n, "us": ms * 1e3, "gbs": 8 * n / (ms * 1e-3) / 1e9,
            "frac_of_peak": 8 * n / (ms * 1e-3) / 1e9 / peak,
            "kernel": "torch elementwise (fp32 negation)",
            "l2": "rotating buffer pairs touching more than 320 MB"}


def roundtrip_graph(torch, gkr, case, sets, device, events=None, n: int = GRAPH_STEPS,
                    offset: int = 0):
    """The timed launch configuration: n steps over the rotating input sets in one CUDA
    graph, step k on set (offset + k) % len(sets) (with event nodes around every kernel
    when `events` is given)."""
    return capture_steps(torch, device, lambda k: step(
        gkr, case, sets[(offset + k) % len(sets)], None if events is None else events[k]), n)


class TimedRegion:
    """Exactly K steps of the hot path, as replays of captured graphs of at most
    GRAPH_STEPS steps (whole graphs, then one graph of the remainder).  Global step j runs
    on input set j % ROTATE, and consecutive regions continue the rotation, so no step
    finds its inputs in L2 however K divides.  Graphs are captured once per (first set,
    length)."""

    def __init__(self, torch, gkr, case, sets, device, K: int):
        self.torch, self.gkr, self.case, self.sets, self.device = torch, gkr, case, sets, device
        self.K = K
        self.G = min(K, GRAPH_STEPS)
        self.graphs = {}
        self.next_step = 0

    def _graph(self, offset: int, n: int):
        key = (offset % len(self.sets), n)
        if key not in self.graphs:
            self.graphs[key] = roundtrip_graph(self.torch, self.gkr, self.case, self.sets,
                                               self.device, n=n, offset=key[0])
        return self.graphs[key]

    def prepare(self, regions: int) -> None:
        """Capture every graph that `regions` consecutive regions replay."""
        j = self.next_step
        for _ in range(regions):
            for n in self.pieces():
                self._graph(j, n)
                j += n

    def pieces(self):
        q, rem = divmod(self.K, self.G)
        return [self.G] * q + ([rem] if rem else [])

    def run(self) -> None:
        """Enqueue one region (K steps); no host synchronisation."""
        for n in self.pieces():
            self._graph(self.next_step, n).replay()
            self.next_step += n


def time_roundtrip(args, device, dist):
    import torch
    import gather_kv_rope_gb300 as gkr
    import workloads as W

    case = W.roundtrip_v41_16384()
    sets = device_sets(case, device, ROTATE)
    T = case.num_tokens
    for k in range(args.warmup):
        step(gkr, case, sets[k % ROTATE])
    torch.cuda.synchronize(device)

    G = GRAPH_STEPS
    K = max(1, args.steps)                          # exactly the requested steps
    region = TimedRegion(torch, gkr, case, sets, device, K)
    # one region, untimed, sizes the number of regions timed: enough to fill
    # REGION_SECONDS (and at least 3), so the clock sampler sees the timed work
    region.prepare(ROTATE)
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    region.run()
    b.record()
    torch.cuda.synchronize(device)
    one = max(a.elapsed_time(b), 1e-3)
    repeats = int(min(MAX_REGIONS, max(3, -(-REGION_SECONDS * 1e3 // one))))
    repeats = int(reduce_max(float(repeats), dist))  # every rank times the same regions
    region.prepare(repeats)
    graph = roundtrip_graph(torch, gkr, case, sets, device)     # G steps (supplementary timings)
    external = _supports_external_events(torch)
    kev = None
    if external:                                    # same steps with event nodes per kernel
        kev = [[_timing_event(torch, True) for _ in range(3)] for _ in range(G)]
        graph_ev = roundtrip_graph(torch, gkr, case, sets, device, kev)

    sampler = ClockSampler(_gpu_id(torch, device)).start()
    stream = torch.cuda.current_stream(device)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(repeats)]
    barrier(dist)
    torch.cuda.synchronize(device)
    h0 = time.time()
    for e0, e1 in evs:                              # back to back: no host sync between regions
        e0.record(stream)
        region.run()
        e1.record(stream)
    torch.cuda.synchronize(device)
    h1 = time.time()
    barrier(dist)
    sampler.stop()
    region_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    total_ms_max = reduce_max(statistics.median(region_ms), dist)
    spread = {"regions": repeats, "steps_per_region": K,
              "median_ms": statistics.median(region_ms), "min_ms": min(region_ms),
              "max_ms": max(region_ms),
              "p10_ms": float(np.percentile(region_ms, 10)),
              "p90_ms": float(np.percentile(region_ms, 90)),
              "timed_region_s": h1 - h0,
              "what": f"{repeats} consecutive timed regions of exactly {K} steps each (graph "
                      f"replays: {len(region.pieces())} per region), CUDA events around each "
                      "region; value uses the median region (max over ranks)"}

    # the same step with early metadata reads (the early_metadata launch option): the slot lists,
    # positions and indices are inputs that no kernel of the step writes
    with gkr.launch_policy(early_metadata=True):
        graph_em = roundtrip_graph(torch, gkr, case, sets, device)
        n_em = 100
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        a.record(stream)
        for _ in range(n_em):
            graph_em.replay()
        b.record(stream)
        torch.cuda.synchronize(device)
        em_ms = reduce_max(a.elapsed_time(b) / (n_em * G), dist)
        del graph_em

    # per-kernel durations: the event graph (each kernel bracketed by event nodes, so
    # no launch overlap between kernels) replayed right after the timed region, or an
    # eager pass with the stream held back by a sleep so launches queue up first
    if kev is not None:
        ins, gat = [], []
        for _ in range(5):
            graph_ev.replay()
            torch.cuda.synchronize(device)
            ins += [kev[k][0].elapsed_time(kev[k][1]) for k in range(G)]
            gat += [kev[k][1].elapsed_time(kev[k][2]) for k in range(G)]
        how = (f"CUDA events captured around every kernel in a graph of the same {G} steps, "
               "5 replays after the timed region")
    else:
        ins, gat = eager_kernel_times(torch, gkr, case, sets, G, device)
        how = "CUDA events around eager launches queued behind a device sleep"
    clocks = sampler.summary(h0, h1)
    # per-kernel launch duration as the roofline uses it: the same kernel launched G
    # times back to back over the rotating input sets in a graph of its own, CUDA
    # events around 5 replays (no event nodes between the launches)
    b2b, flushed = {}, {}
    flush = torch.ones(64 << 20, dtype=torch.int32, device=device)      # 256 MiB, 2x the L2
    for name, fn in (("insert", lambda s: gkr.kv_insert(s["kv"], s["cache"], s["slots"],
                                                          s["pos"], s["csc"], case.block_size,
                                                          case.record)),
                     ("gather", lambda s: gkr.kv_gather(s["cache"], s["idx"], s["out"]))):
        g = capture_steps(torch, device, lambda k: fn(sets[k % ROTATE]), G)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(5):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize(device)
        b2b[name] = a.elapsed_time(b) / (5 * G)
        # the same kernel launched alone after an L2 flush, CUDA events around it only:
        # median over 25 launches, each after a max-reduction over 256 MiB (L2 then holds
        # clean lines of that buffer, so the kernel pays no write-backs of the flush)
        ev = []
        for k in range(25):
            flush.max()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn(sets[k % ROTATE])
            e1.record(stream)
            ev.append((e0, e1))
        torch.cuda.synchronize(device)
        flushed[name] = statistics.median(x.elapsed_time(y) for x, y in ev)
    return dict(case=case, K=K, total_ms=total_ms_max, spread=spread, em_ms=em_ms, ins_ms=b2b["insert"],
                gat_ms=b2b["gather"], ins_iso_ms=float(np.mean(ins)),
                gat_iso_ms=float(np.mean(gat)), ins_flushed_ms=flushed["insert"],
                gat_flushed_ms=flushed["gather"],
                kernel_timing=(f"CUDA events around 5 replays of a graph of {G} back-to-back "
                               "launches of the kernel alone over the same rotating input sets"),
                iso_timing=how, clocks=clocks, T=T)


def eager_kernel_times(torch, gkr, case, sets, n, device):
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    torch.cuda.synchronize(device)
    torch.cuda._sleep(int(2e8))          # hold the stream while the launches queue up
    for k in range(n):
        step(gkr, case, sets[k % ROTATE], evs[k])
    torch.cuda.synchronize(device)
    return ([e[0].elapsed_time(e[1]) for e in evs], [e[1].elapsed_time(e[2]) for e in evs])


def _gpu_id(torch, device) -> str:
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        return str(device.index or 0)


def time_e2e(args, device, case, dist=None):
    """Same metric through the public API from pinned host buffers: every step
    copies kv / slots / positions / indices to the device, inserts, gathers and
    copies the gathered rows back, all inside the timed region.

    Steps are pipelined the way a serving loop runs them: host->device copies on
    one stream, kv_insert + kv_gather on another, device->host copies on a third,
    with NB buffer sets so that step i+1's upload and step i-1's download overlap
    step i's kernels.  Events order the three streams per buffer set (a set is
    re-uploaded only after the kernels that read it finished, and its output is
    overwritten only after its download finished).  The same steps issued one
    after another on a single stream are timed too and reported as "serial"."""
    import torch
    import gather_kv_rope_gb300 as gkr
    NB = 3
    # one pinned staging buffer per buffer set holds the step's inputs back to back
    # (kv | slot_mapping | positions | indices), so each step uploads with one copy
    parts = [("kv", case.kv.view(np.uint8), torch.bfloat16, (case.num_tokens, 512)),
             ("slots", case.slots.view(np.uint8), torch.int64, (case.num_tokens,)),
             ("pos", case.positions.view(np.uint8), torch.int64, (case.num_tokens,)),
             ("idx", case.indices.view(np.uint8), torch.int32, case.indices.shape)]
    offs, total = {}, 0
    for name, raw, _, _ in parts:
        offs[name] = total
        total += -(-raw.size // 16) * 16                # keep every part 16-byte aligned
    staged = np.zeros(total, np.uint8)
    for name, raw, _, _ in parts:
        staged[offs[name]:offs[name] + raw.size] = raw.reshape(-1)
    pin = [torch.from_numpy(staged).pin_memory() for _ in range(NB)]
    dbuf = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(NB)]

    def views(buf):
        return {name: buf[offs[name]:offs[name] + raw.size].view(dt).view(shape)
                for name, raw, dt, shape in parts}
    d = [views(b) for b in dbuf]
    out_shape = case.indices.shape + (512,)
    out_h = [torch.empty(out_shape, dtype=torch.bfloat16).pin_memory() for _ in range(NB)]
    out = [torch.empty(out_shape, dtype=torch.bfloat16, device=device) for _ in range(NB)]
    csc = torch.from_numpy(case.csc).to(device)
    cache = gkr.alloc_cache(case.num_pages, case.block_size, case.record, device, fill=0)
    h2d = sum(raw.size for _, raw, _, _ in parts)
    d2h = out_h[0].numel() * out_h[0].element_size()
    s_up, s_run, s_down = (torch.cuda.Stream(device) for _ in range(3))
    ev = lambda: torch.cuda.Event()
    loaded, computed, drained = ([ev() for _ in range(NB)] for _ in range(3))
    started = [False] * NB

    def kernels(b, stream):
        with torch.cuda.stream(stream):
            gkr.kv_insert(d[b]["kv"], cache, d[b]["slots"], d[b]["pos"], csc,
                          case.block_size, case.record)
            gkr.kv_gather(cache, d[b]["idx"], out[b])

    def piped(i):
        b = i % NB
        if started[b]:
            s_up.wait_event(computed[b])           # inputs of set b no longer read
        with torch.cuda.stream(s_up):
            dbuf[b].copy_(pin[b], non_blocking=True)
        loaded[b].record(s_up)
        s_run.wait_event(loaded[b])
        if started[b]:
            s_run.wait_event(drained[b])           # out[b] downloaded by the last user
        kernels(b, s_run)
        computed[b].record(s_run)
        s_down.wait_event(computed[b])
        with torch.cuda.stream(s_down):
            out_h[b].copy_(out[b], non_blocking=True)
        drained[b].record(s_down)
        started[b] = True

    def copies_only(i):                            # the step's two transfers, no kernels
        b = i % NB
        with torch.cuda.stream(s_up):
            dbuf[b].copy_(pin[b], non_blocking=True)
        with torch.cuda.stream(s_down):
            out_h[b].copy_(out[b], non_blocking=True)

    def serial(i):
        b = i % NB
        cur = torch.cuda.current_stream(device)
        dbuf[b].copy_(pin[b], non_blocking=True)
        kernels(b, cur)
        out_h[b].copy_(out[b], non_blocking=True)

    def timed(step, n):
        cur = torch.cuda.current_stream(device)
        for i in range(5):
            step(i)
        torch.cuda.synchronize(device)
        barrier(dist)                      # every rank's copies share the host link
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for s in (s_up, s_run, s_down):
            s.wait_stream(cur)
        for i in range(n):
            step(i)
        for s in (s_up, s_run, s_down):
            cur.wait_stream(s)
        e1.record(cur)
        torch.cuda.synchronize(device)
        return reduce_max(e0.elapsed_time(e1) / n, dist)

    world = 1 if dist is None else dist.get_world_size()
    ms_serial = timed(serial, args.e2e_steps)
    ms_copies = timed(copies_only, args.e2e_steps)
    ms = timed(piped, args.e2e_steps)
    # every step inserts and gathers the same inputs: each downloaded buffer must hold
    # the same rows as the device-side result (a race between the streams shows here)
    ref = out[0].cpu()
    if not all(torch.equal(h.view(torch.int16), ref.view(torch.int16)) for h in out_h):
        raise RuntimeError("pipelined end-to-end steps returned different results")
    return {"value": world * case.num_tokens / (ms * 1e-3), "unit": "tokens/s",
            "ms_per_step": ms, "steps": args.e2e_steps, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "serial": {"value": world * case.num_tokens / (ms_serial * 1e-3),
                       "ms_per_step": ms_serial},
            "copies_only": {"ms_per_step": ms_copies,
                            "host_link_gbs": (h2d + d2h) / (ms_copies * 1e-3) / 1e9,
                            "what": "the step's upload and download alone, concurrent on "
                                    "their two streams: the host-link bound of the step"},
            "path": "one pinned host -> device copy of the step's inputs, kv_insert, kv_gather, "
                    f"device -> pinned host copy of the rows; three streams, {NB} buffer sets"}


def sweep(device, peak):
    """Kernel-only timings of the larger workloads: launches captured back to back in a
    CUDA graph, the graph replayed after warm-up, time per launch = CUDA-event time /
    launches; no host-side launch overhead is inside the measurement.  Each launch
    touches more than L2, or the launches rotate over input sets that together do."""
    import torch
    import gather_kv_rope_gb300 as gkr
    import workloads as W
    res = {}

    def graph_ms(body, per_graph, replays):
        g = capture_steps(torch, device, body, per_graph)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(replays):
            g.replay()
        b.record()
        torch.cuda.synchronize(device)
        return a.elapsed_time(b) / (per_graph * replays)

    def timed(fn, sets, replays=5):
        """ms per launch of fn, launched back to back over `sets` (at least 12 launches,
        every set at least once) in a CUDA graph."""
        for k in range(3):
            fn(sets[k % len(sets)])
        torch.cuda.synchronize(device)
        return graph_ms(lambda k: fn(sets[k % len(sets)]), max(12, len(sets)), replays)

    # the smallest configuration: 1024 tokens, launch- and latency-bound
    case = W.insert_v41_1024()
    b = insert_bytes(case.slots, 528)
    sets = device_sets(case, device, int(max(1, -(-320_000_000 // b))))
    ms = timed(lambda s: gkr.kv_insert(s["kv"], s["cache"], s["slots"], s["pos"], s["csc"],
                                       case.block_size, 528), sets)
    res["insert_v41_1024"] = {"kernel": "insert", "launch": gkr.insert_kernel_for(1024),
                              "us": ms * 1e3, "tokens_per_s": 1024 / (ms * 1e-3), "alg_bytes": b,
                              "alg_gbs": b / (ms * 1e-3) / 1e9,
                              "frac_of_peak": b / (ms * 1e-3) / 1e9 / peak,
                              "csc_bytes": csc_bytes(case.slots, case.positions),
                              "l2": f"{len(sets)} rotating input sets"}
    del sets
    torch.cuda.empty_cache()

    res["floor"] = launch_floors(torch, gkr, W, device, timed)

    for name, n_sets in (("insert_v4_65536", 3), ("insert_v41_262144", 1)):
        case = getattr(W, name)()
        sets = device_sets(case, device, n_sets)
        ms = timed(lambda s: gkr.kv_insert(s["kv"], s["cache"], s["slots"], s["pos"], s["csc"],
                                           case.block_size, case.record), sets)
        b = insert_bytes(case.slots, case.record)
        res[name] = {"kernel": "insert", "us": ms * 1e3, "tokens_per_s": case.num_tokens / (ms * 1e-3),
                     "alg_bytes": b, "alg_gbs": b / (ms * 1e-3) / 1e9,
                     "frac_of_peak": b / (ms * 1e-3) / 1e9 / peak,
                     "csc_bytes": csc_bytes(case.slots, case.positions),
                     "ncu": ncu_dram_rate(gkr.insert_kernel_for(case.num_tokens), name, peak)}
        res[f"stream_same_bytes_as_{name}"] = stream_same_bytes(torch, device, b, peak)
        del sets
        torch.cuda.empty_cache()

    # the token counts the pages time on GB300 (16384 .. 65536; 262144 is above): V4.1
    # inserts with random slots and positions, rotating over sets that exceed L2 together
    for T in (16384, 32768, 65536):
        case = W.random_insert(f"insert_v41_{T}", T, 528, 64, 2 * T // 64, 8192, 0.05, seed=1)
        b = insert_bytes(case.slots, 528)
        sets = device_sets(case, device, int(max(1, -(-320_000_000 // b))))
        ms = timed(lambda s: gkr.kv_insert(s["kv"], s["cache"], s["slots"], s["pos"], s["csc"],
                                           64, 528), sets)
        res[f"insert_v41_{T}"] = {"kernel": "insert", "launch": gkr.insert_kernel_for(T),
                                  "us": ms * 1e3, "tokens_per_s": T / (ms * 1e-3), "alg_bytes": b,
                                  "alg_gbs": b / (ms * 1e-3) / 1e9,
                                  "frac_of_peak": b / (ms * 1e-3) / 1e9 / peak,
                                  "csc_bytes": csc_bytes(case.slots, case.positions),
                                  "l2": f"{len(sets)} rotating input sets",
                                  "ncu": ncu_dram_rate(gkr.insert_kernel_for(T),
                                                       f"roundtrip_v41_{T}", peak)}
        if T == 65536:   # the round trip's gather at this size: the slots just written
            for st in sets:
                st["idx"] = st["slots"].to(torch.int32)
                st["out"] = torch.empty(T, 512, dtype=torch.bfloat16, device=device)
            ms = timed(lambda s: gkr.kv_gather(s["cache"], s["idx"], s["out"]), sets)
            b = gather_bytes(case.slots.astype(np.int32), 528)
            res[f"gather_v41_{T}"] = {"kernel": "gather", "us": ms * 1e3,
                                      "indices_per_s": T / (ms * 1e-3), "alg_bytes": b,
                                      "alg_gbs": b / (ms * 1e-3) / 1e9,
                                      "frac_of_peak": b / (ms * 1e-3) / 1e9 / peak,
                                      "l2": f"{len(sets)} rotating input sets",
                                      "ncu": ncu_dram_rate("gather_kernel",
                                                           f"roundtrip_v41_{T}", peak)}
        del sets
        torch.cuda.empty_cache()

    for name in ("compressed_v41_r4_262144", "compressed_v41_r128_262144"):
        case = W.WORKLOADS[name]()
        R = case.meta["compress_ratio"]
        b = compressed_insert_bytes(case.slots, case.positions, R, case.record)
        # a launch touches only the rows of the group-boundary tokens (less than L2): the
        # sets read kv through windows of one buffer shifted by k rows (k < R, so each set
        # reads other rows), with their own slots, positions and cache, until the sets
        # together touch more than 320 MB
        sets = compressed_sets(case, device, b)
        n_sets = len(sets)
        ms = timed(lambda s: gkr.rope_quant_insert(s["kv"], s["cache"], s["slots"], s["pos"],
                                                   s["csc"], case.block_size, R, True,
                                                   case.record), sets)
        res[name] = {"kernel": "insert_sparse_staged", "compress_ratio": R, "sanitize_nans": True,
                     "l2": f"{n_sets} rotating input sets touching {n_sets * b / 1e6:.0f} MB",
                     "us": ms * 1e3, "tokens_per_s": case.num_tokens / (ms * 1e-3),
                     "alg_bytes": b, "alg_gbs": b / (ms * 1e-3) / 1e9,
                     "frac_of_peak": b / (ms * 1e-3) / 1e9 / peak,
                     "csc_bytes": csc_bytes(case.slots, case.positions, R)}
        del sets
        torch.cuda.empty_cache()

    # the plain KV-only caches: the 262144-token insert into bf16 rows and fp8 rows (at a
    # general scale, and at 1.0, a power of two, which takes the single-product quotient)
    case = W.insert_v41_262144()
    scale = torch.tensor([0.01], dtype=torch.float32, device=device)
    scale_one = torch.tensor([1.0], dtype=torch.float32, device=device)
    for record, fmt, sc in ((1024, "bf16", None), (512, "fp8", scale),
                            (512, "fp8_scale1", scale_one)):
        sets = device_sets(case, device, 1, record=record)
        ms = timed(lambda s: gkr.kv_insert(s["kv"], s["cache"], s["slots"], s["pos"], s["csc"],
                                           case.block_size, record, fp8_scale=sc), sets)
        b = insert_bytes(case.slots, record)
        res[f"insert_{fmt}_262144"] = {
            "kernel": "insert", "record": record, "us": ms * 1e3,
            "fp8_scale": None if sc is None else float(sc.item()),
            "tokens_per_s": case.num_tokens / (ms * 1e-3), "alg_bytes": b,
            "alg_gbs": b / (ms * 1e-3) / 1e9, "frac_of_peak": b / (ms * 1e-3) / 1e9 / peak,
            "csc_bytes": csc_bytes(case.slots, case.positions)}
        del sets
        torch.cuda.empty_cache()

    # the fused attention write (query heads normed and rotated, padded heads zeroed, the
    # KV rows inserted into the V4.1 cache): a decode batch (256 tokens x 128 heads) and a
    # prefill chunk (8192 tokens x 16 heads padded to 64), random slots and positions
    for name, T, H, Hp in (("qnorm_rope_kv_insert_decode_256x128", 256, 128, 128),
                           ("qnorm_rope_kv_insert_prefill_8192x16p64", 8192, 16, 64)):
        case = W.random_insert(name, T, 528, 64, 2 * T // 64 + 2, 8192, 0.05, seed=3)
        b = qside_bytes(case.slots, 528, H, Hp)
        sets = device_sets(case, device, int(max(1, -(-320_000_000 // b))))
        g = torch.Generator(device="cpu").manual_seed(0)
        for st in sets:
            st["q"] = torch.randn(T, H, 512, generator=g).to(torch.bfloat16).to(device)
            st["q_out"] = torch.empty(T, Hp, 512, dtype=torch.bfloat16, device=device)
        ms = timed(lambda st: gkr.qnorm_rope_kv_insert(
            st["q"], st["kv"], st["cache"], st["slots"], st["pos"], st["csc"], Hp, 1e-6, 64,
            True, q_out=st["q_out"]), sets)
        res[name] = {"kernel": "qnorm_rope_kv_insert", "tokens": T, "heads": H,
                     "heads_padded": Hp, "us": ms * 1e3, "tokens_per_s": T / (ms * 1e-3),
                     "alg_bytes": b, "alg_gbs": b / (ms * 1e-3) / 1e9,
                     "frac_of_peak": b / (ms * 1e-3) / 1e9 / peak,
                     "l2": f"{len(sets)} rotating input sets",
                     "ncu": ncu_dram_rate("qnorm_rope_kv_insert_kernel",
                                          "qnorm_prefill_8192x16p64", peak)
                     if name.endswith("prefill_8192x16p64") else None}
        del sets
        torch.cuda.empty_cache()

    # the same two shapes with the e4m3 query output (one fp32 query scale)
    for name, T, H, Hp in (("qnorm_rope_kv_insert_fp8q_decode_256x128", 256, 128, 128),
                           ("qnorm_rope_kv_insert_fp8q_prefill_8192x16p64", 8192, 16, 64)):
        case = W.random_insert(name, T, 528, 64, 2 * T // 64 + 2, 8192, 0.05, seed=3)
        b = qside_bytes(case.slots, 528, H, Hp, q_out_bytes=512)
        sets = device_sets(case, device, int(max(1, -(-320_000_000 // b))))
        g = torch.Generator(device="cpu").manual_seed(0)
        qs = torch.tensor([0.05], dtype=torch.float32, device=device)
        for st in sets:
            st["q"] = torch.randn(T, H, 512, generator=g).to(torch.bfloat16).to(device)
            st["q_out"] = torch.empty(T, Hp, 512, dtype=torch.float8_e4m3fn, device=device)
        ms = timed(lambda st: gkr.qnorm_rope_kv_insert(
            st["q"], st["kv"], st["cache"], st["slots"], st["pos"], st["csc"], Hp, 1e-6, 64,
            True, q_out=st["q_out"], q_scale=qs), sets)
        res[name] = {"kernel": "qnorm_rope_kv_insert (e4m3 q_out)", "tokens": T, "heads": H,
                     "heads_padded": Hp, "q_scale": 0.05, "us": ms * 1e3,
                     "tokens_per_s": T / (ms * 1e-3), "alg_bytes": b,
                     "alg_gbs": b / (ms * 1e-3) / 1e9,
                     "frac_of_peak": b / (ms * 1e-3) / 1e9 / peak,
                     "l2": f"{len(sets)} rotating input sets"}
        del sets
        torch.cuda.empty_cache()

    case = W.gather_v41_sparse()
    kv = torch.from_numpy(case.kv.view(np.int16)).view(torch.bfloat16).to(device)
    idx = torch.from_numpy(case.indices).to(device)
    outs = [torch.empty(case.indices.shape + (512,), dtype=torch.bfloat16, device=device)
            for _ in range(2)]
    res.update(sparse_logits_entries(torch, gkr, W, case, kv, idx, device, peak, timed))
    for record, name in ((528, "gather_v41_sparse"), (584, "gather_v4_sparse"),
                         (512, "gather_fp8_sparse"), (1024, "gather_bf16_sparse")):
        sc = scale if record == 512 else None
        cache = gkr.alloc_cache(case.num_pages, 64, record, device, fill=0)
        gkr.kv_insert(kv, cache, torch.from_numpy(case.slots).to(device),
                      torch.from_numpy(case.positions).to(device),
                      torch.from_numpy(case.csc).to(device), 64, record, fp8_scale=sc)
        ms = timed(lambda o: gkr.kv_gather(cache, idx, o, fp8_scale=sc), outs)
        b = gather_bytes(case.indices, record)
        res[name] = {"kernel": "gather", "record": record, "us": ms * 1e3,
                     "indices_per_s": case.indices.size / (ms * 1e-3), "alg_bytes": b,
                     "alg_gbs": b / (ms * 1e-3) / 1e9,
                     "frac_of_peak": b / (ms * 1e-3) / 1e9 / peak,
                     "ncu": ncu_dram_rate("gather_kernel", "gather_v41_sparse", peak)
                     if record == 528 else None}
        del cache
        torch.cuda.empty_cache()
    return res


def sparse_logits_entries(torch, gkr, W, case, kv, idx, device, peak, timed) -> dict:
    """The dequant-gather fused into its consumer: logits of 128 decode queries x 128 heads
    over their 2048 top-k records of the 1M-token V4.1 cache, against the same result
    computed unfused (kv_gather to bf16 rows, then torch's bf16 batched matmul)."""
    res = {}
    cache = gkr.alloc_cache(case.num_pages, 64, 528, device, fill=0)
    gkr.kv_insert(kv, cache, torch.from_numpy(case.slots).to(device),
                  torch.from_numpy(case.positions).to(device),
                  torch.from_numpy(case.csc).to(device), 64, 528)
    Q, K = case.indices.shape
    H = 128
    q = torch.from_numpy(W.decode_queries(Q, H).view(np.int16)).view(torch.bfloat16).to(device)
    outs = [torch.empty(Q, H, K, dtype=torch.float32, device=device) for _ in range(2)]
    ms = timed(lambda o: gkr.sparse_logits(q, cache, idx, 512 ** -0.5, out=o), outs)
    b, f = logits_bytes(case.indices, 528, H), logits_flops(case.indices, H)
    res["sparse_logits_v41_128x2048_h128"] = {
        "kernel": "sparse_logits_kernel", "queries": Q, "topk": K, "heads": H, "us": ms * 1e3,
        "entries_per_s": Q * K / (ms * 1e-3), "alg_bytes": b, "alg_gbs": b / (ms * 1e-3) / 1e9,
        "frac_of_peak": b / (ms * 1e-3) / 1e9 / peak, "tflops": f / (ms * 1e-3) / 1e12,
        "bound": "hbm", "ncu": ncu_dram_rate("sparse_logits_kernel", "sparse_logits", peak)}
    rows = torch.empty(Q, K, 512, dtype=torch.bfloat16, device=device)
    outs_bf16 = [torch.empty(Q, H, K, dtype=torch.bfloat16, device=device) for _ in range(2)]

    def unfused(o):
        gkr.kv_gather(cache, idx, rows)
        torch.bmm(q, rows.transpose(1, 2), out=o)
    ms_u = timed(unfused, outs_bf16)
    res["sparse_logits_unfused_gather_then_bmm"] = {
        "us": ms_u * 1e3, "what": "kv_gather into bf16 [128, 2048, 512], then torch.bmm of the "
                                  "same queries (bf16 logits: half the fused path's fp32 "
                                  "output bytes): the unfused path",
        "fused_speedup": ms_u / ms}
    del cache, rows, outs, outs_bf16
    torch.cuda.empty_cache()
    return res


def launch_floors(torch, gkr, W, device, timed) -> dict:
    """What a launch costs before its row traffic, timed like every kernel here (back to
    back in a CUDA graph, programmatic dependent launch on): a 1-token insert and a
    1-index gather, with the token skipped / the index -1 (the launch, the wait for the
    previous kernel and one dependent load of the slot or index) and valid (plus the
    dependent row loads and the stores); and the 16384-token insert of the benchmark step
    with every slot -1 (the whole grid's slot and position round trip, no row traffic)."""
    case = W.roundtrip_v41_16384()
    out = {}
    for label, slot in (("skipped", -1), ("valid", int(case.slots[case.slots >= 0][0]))):
        one = W.InsertCase("one", 528, 64, case.num_pages, case.kv[:1].copy(),
                           np.array([slot], np.int64), case.positions[:1].copy(), case.csc)
        one.indices = one.slots.astype(np.int32)
        sets = device_sets(one, device, 1)
        ms = timed(lambda s: gkr.kv_insert(s["kv"], s["cache"], s["slots"], s["pos"],
                                           s["csc"], 64, 528), sets)
        out[f"insert_1_token_{label}_us"] = ms * 1e3
        ms = timed(lambda s: gkr.kv_gather(s["cache"], s["idx"], s["out"]), sets)
        out[f"gather_1_index_{label}_us"] = ms * 1e3
        del sets
    skip = W.InsertCase("skip", 528, 64, case.num_pages, case.kv, np.full_like(case.slots, -1),
                        case.positions, case.csc)
    sets = device_sets(skip, device, ROTATE)
    ms = timed(lambda s: gkr.kv_insert(s["kv"], s["cache"], s["slots"], s["pos"], s["csc"],
                                       64, 528), sets)
    out["insert_16384_tokens_all_skipped_us"] = ms * 1e3
    del sets
    torch.cuda.empty_cache()
    out["what"] = ("launch floors, back to back in a CUDA graph with programmatic dependent "
                   "launch: 1-token inserts / 1-index gathers (skipped or valid) and the "
                   "benchmark step's 16384-token insert with every slot -1")
    return out


# ----------------------------------------------------------------------------- CPU oracle

def oracle_steps(case, tokens: int, steps: int):
    """Run `steps` oracle steps (insert + gather of `tokens` tokens of the workload).
    Returns seconds per step."""
    import oracle
    ps = oracle.page_stride(case.record, case.block_size)
    cache = np.zeros(case.num_pages * ps, np.uint8)
    kv, slots, pos = case.kv[:tokens], case.slots[:tokens], case.positions[:tokens]
    idx = case.indices[:tokens]
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.insert(kv, cache, case.record, case.block_size, case.num_pages, ps, slots, pos,
                      case.csc)
        oracle.gather(cache, case.record, case.block_size, case.num_pages, ps, idx)
    return (time.perf_counter() - t0) / steps


def _oracle_chunk(job):
    """Worker of the all-cores oracle timing: insert + gather of one disjoint token range
    (its own copy of the cache), `steps` times.  Returns the seconds it took."""
    kv, slots, pos, idx, csc, record, bs, pages, steps = job
    import oracle
    ps = oracle.page_stride(record, bs)
    cache = np.zeros(pages * ps, np.uint8)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.insert(kv, cache, record, bs, pages, ps, slots, pos, csc)
        oracle.gather(cache, record, bs, pages, ps, idx)
    return time.perf_counter() - t0


def _cpu_model() -> str:
    try:
        text = Path("/proc/cpuinfo").read_text()
    except OSError:
        return "unknown"
    for key in ("model name", "CPU part"):
        for line in text.splitlines():
            if line.startswith(key):
                return f"{key}: {line.split(':', 1)[1].strip()}"
    return "unknown"


def cpu_baseline(case, seconds: float) -> dict:
    """The oracle on the host: single-threaded (the line's value), and the same code run
    on every core over disjoint token ranges (slots are unique, so the ranges write
    disjoint records and each range gathers its own slots), in a spawn-started pool."""
    import multiprocessing as mp
    per = oracle_steps(case, 1024, 1)                 # calibrate on 1024 tokens
    tok_s = 1024 / per
    tokens = int(min(case.num_tokens, max(1024, tok_s * seconds / 3)))
    steps = max(1, int(seconds / (tokens / tok_s)))
    sec = oracle_steps(case, tokens, steps)
    ncpu = os.cpu_count() or 1
    out = {"value": tokens / sec, "unit": "tokens/s", "cores": 1, "kind": "oracle",
           "sample": f"{steps} x insert+gather of the first {tokens} of the 16384 tokens "
                     f"(single-threaded C oracle, {ncpu} host cores present)",
           "cpu_model": _cpu_model()}
    if ncpu > 1:
        T = case.num_tokens
        bounds = np.linspace(0, T, ncpu + 1).astype(int)
        psteps = max(1, int(steps * ncpu * tokens / T))   # about the same total work
        jobs = [(case.kv[a:b], case.slots[a:b], case.positions[a:b], case.indices[a:b],
                 case.csc, case.record, case.block_size, case.num_pages, psteps)
                for a, b in zip(bounds[:-1], bounds[1:])]
        with mp.get_context("spawn").Pool(ncpu) as pool:
            pool.map(_oracle_chunk, [j[:8] + (1,) for j in jobs])      # warm the workers
            times = pool.map(_oracle_chunk, jobs)
        out["all_cores"] = {"value": T * psteps / max(times), "unit": "tokens/s",
                            "cores": ncpu,
                            "sample": f"{psteps} x insert+gather of all {T} tokens, split "
                                      f"into {ncpu} disjoint ranges, one process per core"}
    return out


_REF = {}


def _ref_init(case_arrays):
    """Worker start-up for the reference arm: keep the inputs and a private cache."""
    import oracle
    kv, slots, pos, idx, csc, record, bs, pages = case_arrays
    ps = oracle.page_stride(record, bs)
    _REF.update(kv=kv, slots=slots, pos=pos, idx=idx, csc=csc, record=record, bs=bs,
                pages=pages, ps=ps, cache=np.zeros(pages * ps, np.uint8))


def _ref_range(bounds):
    """One step's share of a worker: insert + gather of the token range [a, b)."""
    import oracle
    a, b = bounds
    r = _REF
    oracle.insert(r["kv"][a:b], r["cache"], r["record"], r["bs"], r["pages"], r["ps"],
                  r["slots"][a:b], r["pos"][a:b], r["csc"])
    oracle.gather(r["cache"], r["record"], r["bs"], r["pages"], r["ps"], r["idx"][a:b])
    return b - a


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on every host core.  Each step is
    the benchmark step's insert + gather of its 16384 tokens, split into one disjoint
    token range per core (slots are unique, so the ranges write disjoint records and
    each gathers its own), run by a spawn-started pool whose workers hold the inputs;
    the step time is wall-clock, dispatch included.  The whole --steps/--warmup run is
    held to about 150 s: when a full step does not fit, every step takes the first
    tokens of the workload, and when even a pool dispatch does not fit, one process
    runs a bounded sample.  The single-core rate is reported beside it."""
    import multiprocessing as mp
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import workloads as W
    case = W.roundtrip_v41_16384()
    T = case.num_tokens
    ncpu = os.cpu_count() or 1
    per = oracle_steps(case, 512, 1)
    single = {"value": 512 / per, "cores": 1, "sample": "insert+gather of 512 tokens"}
    budget = 150.0 / max(1, args.steps + args.warmup)     # seconds per step, about 150 s total
    arrays = (case.kv, case.slots, case.positions, case.indices, case.csc, case.record,
              case.block_size, case.num_pages)

    def ranges(n):
        edges = np.linspace(0, n, ncpu + 1).astype(int)
        return [(int(a), int(b)) for a, b in zip(edges[:-1], edges[1:])]

    with mp.get_context("spawn").Pool(ncpu, initializer=_ref_init, initargs=(arrays,)) as pool:
        pool.map(_ref_range, ranges(T))                     # warm the workers
        t0 = time.perf_counter()
        pool.map(_ref_range, ranges(T))
        full = time.perf_counter() - t0
        t0 = time.perf_counter()
        pool.map(_ref_range, ranges(0))
        dispatch = time.perf_counter() - t0
        if budget >= full:
            tokens = T
        elif budget > 3 * dispatch:                          # a sample of every step
            tokens = int(max(ncpu, T * (budget - dispatch) / max(full - dispatch, 1e-9)))
        else:
            tokens = 0                                       # too many steps for a pool
        if tokens:
            for _ in range(args.warmup):
                pool.map(_ref_range, ranges(tokens))
            t0 = time.perf_counter()
            for _ in range(args.steps):
                pool.map(_ref_range, ranges(tokens))
            sec = (time.perf_counter() - t0) / max(1, args.steps)
    if tokens:
        cores, how = ncpu, (f"insert+gather of {'all' if tokens == T else 'the first'} {tokens} "
                            f"of the {T} tokens per step, one disjoint token range per core "
                            f"({ncpu} processes)")
    else:                                                    # one process, bounded sample
        tokens = int(np.clip(512 / per * budget, 16, T))
        if args.warmup:
            oracle_steps(case, tokens, args.warmup)
        sec = oracle_steps(case, tokens, args.steps)
        cores, how = 1, (f"insert+gather of the first {tokens} of the {T} tokens per step "
                         "(one process: too many steps for a pool dispatch per step)")
    value = tokens / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": DTYPE, "dtypes": DTYPES, "data": "synthetic",
            "config": workload_config(case),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": how, "cpu_model": _cpu_model(), "single_core": single},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- profiling

def run_profile(args):
    """Run one workload's kernel(s): 2 warm-up launches then --launches timed ones.
    Inserts go to a fresh zeroed cache per launch set; the sparse gathers read a cache
    filled once by the insert (that fill is one extra insert launch before them)."""
    import torch
    import gather_kv_rope_gb300 as gkr
    import workloads as W
    dev = torch.device("cuda:0")
    gkr.build()
    if args.insert_stream_min is not None:
        gkr.set_insert_stream_min(args.insert_stream_min)
    name = args.profile
    if name in ("sparse_logits", "sparse_logits_262144"):
        return _profile_sparse_logits(args, torch, gkr, W, dev, name)
    if name == "qnorm_prefill_8192x16p64":
        return _profile_qside(args, torch, gkr, W, dev, name)
    fp8 = name.startswith("fp8_")                     # the same case into an fp8 cache
    case = W.PROFILE_WORKLOADS[name[4:] if fp8 else name]()
    record = 512 if fp8 else case.record
    s = device_sets(case, dev, 1, record=record)[0]
    res = {"workload": name}
    scale = torch.tensor([0.01], dtype=torch.float32, device=dev) if fp8 else None
    R = case.meta.get("compress_ratio")
    if R:                                             # compressed insert, with sanitising
        ins = lambda: gkr.rope_quant_insert(s["kv"], s["cache"], s["slots"], s["pos"], s["csc"],
                                            case.block_size, R, True, record)
    else:
        ins = lambda: gkr.kv_insert(s["kv"], s["cache"], s["slots"], s["pos"], s["csc"],
                                    case.block_size, record, fp8_scale=scale)
    if args.profile.startswith("gather"):
        ins()                                       # fill the cache once
        fns = {"gather": lambda: gkr.kv_gather(s["cache"], s["idx"], s["out"])}
    elif s["idx"] is not None:
        fns = {"insert": ins, "gather": lambda: gkr.kv_gather(s["cache"], s["idx"], s["out"])}
    else:
        fns = {"insert": ins}
    for name, fn in fns.items():
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(args.launches):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            ts.append((a, b))
        torch.cuda.synchronize()
        res[name + "_us"] = [round(a.elapsed_time(b) * 1e3, 2) for a, b in ts]
    print(json.dumps(res), flush=True)
    return 0


def _time_launches(torch, fn, n):
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    return [round(a.elapsed_time(b) * 1e3, 2) for a, b in ts]


def _profile_qside(args, torch, gkr, W, dev, name):
    """The fused attention write at the prefill shape of the sweep (8192 tokens, 16 heads
    padded to 64, V4.1 cache)."""
    T, H, Hp = 8192, 16, 64
    case = W.random_insert(name, T, 528, 64, 2 * T // 64 + 2, 8192, 0.05, seed=3)
    s = device_sets(case, dev, 1)[0]
    q = torch.randn(T, H, 512, generator=torch.Generator().manual_seed(0)).to(torch.bfloat16).to(dev)
    q_out = torch.empty(T, Hp, 512, dtype=torch.bfloat16, device=dev)
    fn = lambda: gkr.qnorm_rope_kv_insert(q, s["kv"], s["cache"], s["slots"], s["pos"], s["csc"],
                                          Hp, 1e-6, 64, True, q_out=q_out)
    print(json.dumps({"workload": name, "qnorm_rope_kv_insert_us": _time_launches(torch, fn,
                                                                                 args.launches)}),
          flush=True)
    return 0


def _profile_sparse_logits(args, torch, gkr, W, dev, name):
    """The sparse logits (128 heads) over the sparse-decode cache: the full workload
    (1M-token cache, 128 queries x 2048) or its 262144-token profiling size (32 queries)."""
    case = W.gather_v41_sparse() if name == "sparse_logits" else W.gather_v41_sparse_262144()
    kv = torch.from_numpy(case.kv.view(np.int16)).view(torch.bfloat16).to(dev)
    cache = gkr.alloc_cache(case.num_pages, 64, 528, dev, fill=0)
    gkr.kv_insert(kv, cache, torch.from_numpy(case.slots).to(dev),
                  torch.from_numpy(case.positions).to(dev), torch.from_numpy(case.csc).to(dev),
                  64, 528)
    del kv
    Q = case.indices.shape[0]
    q = torch.from_numpy(W.decode_queries(Q, 128).view(np.int16)).view(torch.bfloat16).to(dev)
    idx = torch.from_numpy(case.indices).to(dev)
    out = torch.empty(Q, 128, case.indices.shape[1], dtype=torch.float32, device=dev)
    fn = lambda: gkr.sparse_logits(q, cache, idx, 512 ** -0.5, out=out)
    print(json.dumps({"workload": name, "sparse_logits_us": _time_launches(torch, fn,
                                                                          args.launches)}),
          flush=True)
    return 0


# ----------------------------------------------------------------------------- main

def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile(args)

    import torch
    import gather_kv_rope_gb300 as gkr
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU path)")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = init_dist(world, "nccl")
    gkr.build()
    gkr.lib()
    if args.insert_stream_min is not None:
        gkr.set_insert_stream_min(args.insert_stream_min)

    peak, peak_src = measured_peaks()
    r = time_roundtrip(args, device, dist)
    case, K, T = r["case"], r["K"], r["T"]
    ms_step = r["total_ms"] / K
    value = world * K * T / (r["total_ms"] * 1e-3)

    ib, gb = insert_bytes(case.slots, 528), gather_bytes(case.indices, 528)
    kern = {"insert": {"us": r["ins_ms"] * 1e3, "alg_bytes": ib,
                       "gbs": ib / (r["ins_ms"] * 1e-3) / 1e9,
                       "frac_of_peak": ib / (r["ins_ms"] * 1e-3) / 1e9 / peak,
                       "traffic": ncu_traffic(gkr.insert_kernel_for(T), WORKLOAD),
                       "csc_bytes": csc_bytes(case.slots, case.positions),
                       "isolated_us": r["ins_iso_ms"] * 1e3,
                       "after_l2_flush_us": r["ins_flushed_ms"] * 1e3},
            "gather": {"us": r["gat_ms"] * 1e3, "alg_bytes": gb,
                       "gbs": gb / (r["gat_ms"] * 1e-3) / 1e9,
                       "frac_of_peak": gb / (r["gat_ms"] * 1e-3) / 1e9 / peak,
                       "traffic": ncu_traffic("gather_kernel", WORKLOAD),
                       "isolated_us": r["gat_iso_ms"] * 1e3,
                       "after_l2_flush_us": r["gat_flushed_ms"] * 1e3},
            "isolated_timing": r["iso_timing"],
            "after_l2_flush_timing": ("median of 25 launches, each alone after a max-reduction "
                                      "over a 256 MiB buffer, CUDA events around the kernel")}
    dom = "insert" if r["ins_ms"] >= r["gat_ms"] else "gather"
    ach = kern[dom]["gbs"]
    kname = {"insert": gkr.insert_kernel_for(T),
             "gather": "gather_kernel"}[dom]
    same = stream_same_bytes(torch, device, kern[dom]["alg_bytes"], peak)
    roofline = {"bound": "hbm", "kernel": kname, "achieved": ach, "peak": peak, "unit": "GB/s",
                "frac": ach / peak, "peak_source": peak_src,
                "traffic": ncu_traffic(kname, WORKLOAD),
                "alg_bytes_per_launch": kern[dom]["alg_bytes"],
                "timing": r["kernel_timing"],
                "stream_same_bytes": {"gbs": same["gbs"], "us": same["us"],
                                      "frac_of_peak": same["frac_of_peak"],
                                      "kernel_vs_stream": ach / same["gbs"],
                                      "what": "torch's elementwise kernel moving the same bytes "
                                              "per launch, back to back over rotating buffers"}}

    out = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
           "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": DTYPE, "dtypes": DTYPES,
           "data": "synthetic", "config": workload_config(case),
           "timing": r["spread"],
           "early_metadata": {"value": world * T / (r["em_ms"] * 1e-3), "unit": "tokens/s",
                              "ms_per_step": r["em_ms"],
                              "what": "the same step with the early_metadata launch option: the "
                                      "kernels read slot_mapping, positions and indices "
                                      "before waiting for the kernel ahead of them (off by "
                                      "default; valid here, no kernel of the step writes "
                                      "them)"},
           "roofline": roofline, "kernels": kern, "gpu_launches": 2 * K * world,
           "gpu_launches_per_rank": 2 * K,
           "gpu_launches_note": "launches of this library's kernels per timed region of K "
                                "steps (one insert and one gather per step); "
                                f"{r['spread']['regions']} such regions were timed",
           "clocks": r["clocks"]}
    out["e2e"] = time_e2e(args, device, case, dist)            # every rank, max over ranks
    if rank == 0:
        if not args.no_sweep and world == 1:
            out["sweep"] = sweep(device, peak)
        if not args.no_cpu_baseline and world == 1:
            out["cpu_baseline"] = cpu_baseline(case, args.cpu_seconds)
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
