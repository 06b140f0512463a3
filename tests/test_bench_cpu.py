"""Host logic of bench.py on the CPU: byte accounting, the max-over-ranks timing
reduction with two gloo ranks, and the reference (oracle) arm's JSON line."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import numpy as np
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def test_algorithmic_bytes():
    import bench
    slots = np.array([-1, 0, 5, -1, 7], np.int64)
    assert bench.insert_bytes(slots, 528) == 5 * 16 + 3 * (1024 + 528)
    assert bench.insert_bytes(slots, 584) == 5 * 16 + 3 * (1024 + 584)
    pos = np.array([3, 3, 6, 5, 11], np.int64)
    # ratio 4: tokens 1 (pos 3) and 4 (pos 11) are written; token 2 (pos 6) ends no group
    assert bench.compressed_insert_bytes(slots, pos, 4, 528) == 5 * 16 + 2 * (1024 + 528)
    assert bench.compressed_insert_bytes(slots, pos, 1, 584) == bench.insert_bytes(slots, 584)
    idx = np.array([[-1, 2], [3, -1]], np.int32)
    assert bench.gather_bytes(idx, 528) == 4 * 1028 + 2 * 528
    # the fused attention write: the insert's bytes plus every token's heads read and
    # padded heads written (skipped slots still carry their query heads)
    assert bench.qside_bytes(slots, 528, 3, 8) == bench.insert_bytes(slots, 528) + 5 * 11 * 1024
    assert bench.qside_bytes(slots, 584, 0, 0) == bench.insert_bytes(slots, 584)
    # an e4m3 query output writes 512 B per padded head
    assert bench.qside_bytes(slots, 528, 3, 8, q_out_bytes=512) == \
        bench.insert_bytes(slots, 528) + 5 * (3 * 1024 + 8 * 512)
    # cos/sin rows: one per distinct row among the written tokens (tokens 1 and 2 share
    # position 3's row; the skipped token's position 5 is not read)
    pos = np.array([3, 3, 3, 5, 11], np.int64)
    assert bench.csc_bytes(slots, pos) == 2 * 256
    # ratio 4: tokens 1, 2 (pos 3) and 4 (pos 11) read the rows of group starts 0 and 8
    assert bench.csc_bytes(slots, pos, 4) == 2 * 256
    assert bench.csc_bytes(slots, np.array([3, 2, 6, 5, 10], np.int64), 4) == 0


def test_compressed_input_sets_read_shifted_windows():
    """The sweep's compressed-insert sets: set k reads kv rows k .. k + T - 1 of one buffer
    (so each set's boundary tokens read other rows) and owns its slots, positions and
    cache; the number of sets is capped at the ratio."""
    import torch
    import bench
    import workloads as W
    case = W.compressed_insert("sets", 2, 32, 4, 528, block_size=32, seed=1)
    T = case.num_tokens
    sets = bench.compressed_sets(case, "cpu", 1000)           # 320 MB / 1000 B > R: R sets
    assert len(sets) == 4
    kv0 = torch.from_numpy(case.kv.view(np.int16))
    for k, s in enumerate(sets):
        assert s["kv"].shape == (T, 512)
        assert s["kv"].data_ptr() - sets[0]["kv"].data_ptr() == k * 1024
        assert torch.equal(s["kv"][: T - k].view(torch.int16), kv0[k:])
        assert torch.equal(s["kv"][T - k:].view(torch.int16), kv0[:k])
    for key in ("slots", "pos", "cache"):
        assert len({s[key].data_ptr() for s in sets}) == 4
    assert len(bench.compressed_sets(case, "cpu", 400_000_000)) == 1


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, str(ROOT))
    import bench
    dist = bench.init_dist(world, "gloo")
    bench.barrier(dist)
    got = bench.reduce_max(10.0 + 5.0 * rank, dist)
    q.put((rank, got))
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = dict(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 15.0, 1: 15.0}


def test_reduce_max_single_process_is_identity():
    import bench
    assert bench.reduce_max(3.5, None) == 3.5


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True,
                       cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["config"]["workload"] == "roundtrip_v41_16384"
    import bench
    import workloads as W
    # the same workload dict as the GPU arm's line
    assert d["config"] == bench.workload_config(W.roundtrip_v41_16384())
    assert d["steps"] == 2 and d["warmup"] == 1 and d["dtype"] == bench.DTYPE


def test_timed_region_runs_exactly_k_steps_and_continues_the_rotation(monkeypatch):
    """The timed region is K steps (whole graphs of at most GRAPH_STEPS, then the
    remainder), and region after region the input sets keep rotating: global step j runs
    on set j % ROTATE whatever K is."""
    import bench
    seen = []

    class FakeGraph:
        def __init__(self, n, offset):
            self.n, self.offset = n, offset

        def replay(self):
            seen.extend((self.offset + k) % bench.ROTATE for k in range(self.n))

    captured = []

    def fake_graph(torch, gkr, case, sets, device, events=None, n=bench.GRAPH_STEPS, offset=0):
        captured.append((offset, n))
        return FakeGraph(n, offset)

    monkeypatch.setattr(bench, "roundtrip_graph", fake_graph)
    for K in (1, 20, 60, 61, 125):
        seen.clear()
        captured.clear()
        r = bench.TimedRegion(None, None, None, list(range(bench.ROTATE)), None, K)
        assert sum(r.pieces()) == K and max(r.pieces()) <= bench.GRAPH_STEPS
        r.prepare(4)
        n_captured = len(captured)
        for _ in range(4):
            r.run()
        assert len(captured) == n_captured          # every graph was captured up front
        assert seen == [j % bench.ROTATE for j in range(4 * K)]


def test_code_only_drops_comments_and_whitespace_only():
    """The kernel-source hash ignores comments and layout, not code (string and character
    literals that look like comments stay)."""
    import bench
    a = 'int a = 1; // one\n/* two\n lines */ const char* s = "//x/*"; char c = \'/\';\n'
    b = 'int a = 1;\n\n   const char* s = "//x/*";   char c = \'/\';'
    assert bench.code_only(a) == bench.code_only(b) == \
        'int a = 1; const char* s = "//x/*"; char c = \'/\';'
    assert bench.code_only("int a = 1;") != bench.code_only("int a = 2;")
