"""The bench's algorithmic byte model and its table of captured DRAM traffic, checked on the CPU.

The byte model (per touched virtual expert its weight rows, per distinct activation row its
bytes, per pair its intermediate and output bytes) is recomputed here independently by walking
the oracle's routed blocks, as the kernels do. Each traffic entry must carry the algorithmic
bytes of the launch it was captured on (the workload's first layer), and its DRAM bytes must not
exceed them (no re-reads) by more than a few sectors."""

from types import SimpleNamespace

import numpy as np
import pytest

import bench
import oracle
from synth import WORKLOADS, make_layer


def _routing(name):
    wl = WORKLOADS[name]
    li = make_layer(wl, 0, layer=0)
    vt = oracle.virtual_topk(li.topk_ids, li.lora_ids, wl.E, wl.L).reshape(-1)
    s, e, n = oracle.align_block_size(vt, wl.V, wl.BM)
    return wl, li, vt, s, e, n


def _walked_bytes(wl, st, s, e, n):
    """Bytes the stage's shrink and expand must move, from the routed blocks: each touched
    virtual expert's weights once, each distinct activation row once, each pair's
    intermediate row written then read, each pair's output row read and written."""
    S, r, K, R, N = st.stage.S, st.stage.r, st.stage.K, st.stage.R, st.stage.N
    experts, xrows, pairs = set(), set(), 0
    for t in range(n // wl.BM):
        v = int(e[t])
        if v < 0:
            continue
        ids = s[t * wl.BM:(t + 1) * wl.BM]
        ids = ids[ids < wl.numel]
        if ids.size == 0:
            continue
        experts.add(v)
        xrows.update((ids // st.x_row_div).tolist())
        pairs += int(ids.size)
    shrink = len(experts) * R * K * 2 + len(xrows) * K * 2 + pairs * R * 4
    expand = len(experts) * N * r * 2 + pairs * R * 4 + pairs * N * 2 * 2
    return shrink, expand


def _model_bytes(wl, li, vt, si):
    valid = vt >= 0
    pairs = int(valid.sum())
    touched = int(np.unique(vt[valid]).size)
    token_rows = int(np.unique(np.nonzero(valid)[0] // wl.topk).size)
    layer = SimpleNamespace(stages=[{"st": st} for st in li.stages], ranks=None)
    return bench.LayerState.stage_bytes(layer, si, pairs, touched, token_rows, None)


@pytest.mark.parametrize("name", ["tiny", "decode", "wide"])
def test_byte_model_matches_walked_blocks(name):
    wl, li, vt, s, e, n = _routing(name)
    for si, st in enumerate(li.stages):
        assert _model_bytes(wl, li, vt, si) == _walked_bytes(wl, st, s, e, n)


@pytest.mark.parametrize("key", sorted(bench.TRAFFIC))
def test_traffic_entries_belong_to_their_launch(key):
    name, kernel = key
    traffic, launch_bytes, src, digest = bench.TRAFFIC[key]
    assert len(digest) == 16 and int(digest, 16) >= 0
    assert len(bench.kernel_source_digest(src)) == 16  # the file exists
    wl, li, vt, s, e, n = _routing(name)
    kind, stage_name = kernel.split("_", 1)
    si = [st.stage.name for st in li.stages].index(stage_name)
    shrink, expand = _walked_bytes(wl, li.stages[si], s, e, n)
    assert launch_bytes == (shrink if kind == "shrink" else expand)
    # no re-reads: at most the algorithmic bytes plus a little (partial sectors); output rows
    # written into L2 may reach DRAM only after the launch, so the capture can be lower
    assert 0.85 * launch_bytes <= traffic <= 1.02 * launch_bytes


class _FakeGraph:
    def __init__(self, fn, log):
        self.fn, self.log = fn, log

    def replay(self):
        self.fn()


def test_timed_steps_are_exact_and_every_graph_is_warmed(monkeypatch):
    """The timed region runs exactly K layer steps, no layer as a graph of its own when K is
    not a multiple of the rotation, and every graph it replays was replayed before."""
    log = []
    graphs = []

    def fake_capture(torch, fn):
        g = _FakeGraph(fn, log)
        graphs.append(g)
        return g

    class L:
        def __init__(self, i):
            self.i = i

        def forward(self, mol):
            log.append(self.i)

    monkeypatch.setattr(bench, "capture", fake_capture)
    torch = SimpleNamespace(cuda=SimpleNamespace(synchronize=lambda: None))
    layers = [L(i) for i in range(8)]
    cap = 8 * bench.GRAPH_ROTATIONS
    for steps in (20, 16, 5, 1, cap, 2 * cap + 13):
        graphs.clear()
        run, warm = bench.layer_steps_timer(torch, None, layers, steps)
        replayed = set()
        for g in graphs:
            orig = g.replay
            g.replay = (lambda o=orig, g=g: (replayed.add(id(g)), o()))
        log.clear()
        warm(5)
        assert len(log) >= 5
        assert replayed == {id(g) for g in graphs}     # every graph warmed
        log.clear()
        run()
        assert len(log) == steps
        assert log == [i % 8 for i in range(steps)]   # step i on layer i % 8
        assert len(graphs) == (steps >= cap) + (steps % cap != 0)
