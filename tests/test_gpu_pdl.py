"""The launches carry the programmatic-dependent-launch attribute: captured into a CUDA
graph, an insert followed by a gather are joined by a programmatic edge while PDL is on
(gkr_set_pdl), and by a full dependency while it is off.  (The pages checked the same
property by intercepting the launch call and reading its attributes: page "PR #56441
[Perf][DSpark] KV-only context insertion across V4.1 cache formats", section "评论区精华"
item 1.)"""
from __future__ import annotations

import ctypes

import pytest
import torch

import workloads as W
from helpers import device_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
PROGRAMMATIC = 1       # cudaGraphDependencyTypeProgrammatic


class EdgeData(ctypes.Structure):
    _fields_ = [("from_port", ctypes.c_ubyte), ("to_port", ctypes.c_ubyte),
                ("type", ctypes.c_ubyte), ("reserved", ctypes.c_ubyte * 5)]


def _cudart():
    for name in ("libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so.13",
                 "/usr/local/cuda/lib64/libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    pytest.skip("no CUDA runtime library to query graph edges with")


def _edge_types(graph: torch.cuda.CUDAGraph) -> list[int]:
    rt = _cudart()
    rt.cudaGraphGetEdges.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.POINTER(ctypes.c_size_t)]
    h = ctypes.c_void_p(graph.raw_cuda_graph())
    n = ctypes.c_size_t(0)
    assert rt.cudaGraphGetEdges(h, None, None, None, ctypes.byref(n)) == 0
    frm, to = (ctypes.c_void_p * n.value)(), (ctypes.c_void_p * n.value)()
    data = (EdgeData * n.value)()
    assert rt.cudaGraphGetEdges(h, frm, to, data, ctypes.byref(n)) == 0
    return [int(e.type) for e in data]


def _captured_step(gkr):
    case = W.random_insert("pdl", 512, 528, 64, 16, 512, 0.05, seed=3)
    kv, slots, pos, csc = device_inputs(case, DEV)
    cache = gkr.alloc_cache(case.num_pages, 64, 528, DEV, fill=0)
    idx = slots.to(torch.int32)
    out = torch.empty(idx.numel(), 512, dtype=torch.bfloat16, device=DEV)

    def step():
        gkr.kv_insert(kv, cache, slots, pos, csc, 64, 528)
        gkr.kv_gather(cache, idx, out)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    try:
        g = torch.cuda.CUDAGraph(keep_graph=True)     # keeps the cudaGraph_t to inspect
    except TypeError:
        pytest.skip("this torch cannot keep a captured graph")
    with torch.cuda.graph(g):
        step()
    return g


@pytest.mark.parametrize("how", ["per_call", "process_default"])
@pytest.mark.parametrize("pdl", [True, False])
def test_insert_to_gather_edge_follows_the_pdl_setting(gkr, pdl, how):
    """The pdl launch option of the calls (launch_policy), or the process-wide default
    (gkr_set_pdl) when the calls leave it unset."""
    if how == "per_call":
        with gkr.launch_policy(pdl=pdl):
            g = _captured_step(gkr)
    else:
        before = gkr.get_pdl()
        gkr.set_pdl(pdl)
        try:
            g = _captured_step(gkr)
        finally:
            gkr.set_pdl(before)
    types = _edge_types(g)
    assert len(types) == 1, types                    # insert -> gather, nothing else
    assert types[0] == (PROGRAMMATIC if pdl else 0), types
    if hasattr(g, "instantiate"):
        g.instantiate()
    g.replay()
    torch.cuda.synchronize()
