"""A whole MoL LoRA layer (routing + gate_up stage + down stage) captured in a CUDA graph.

Replays must reproduce the eager result bit for bit (the path is deterministic)
and match the oracle.
"""

import numpy as np
import pytest

import oracle
from synth import WORKLOADS, make_layer
from tests.gpu_util import bf16_host, check_out, mol_lib, to_dev_i32, torch_cuda, valid_pairs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [1, 2])
def test_layer_graph_replay_matches_eager(mode):
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    wl = WORKLOADS["decode"]
    li = make_layer(wl, seed=3)
    topk = to_dev_i32(li.topk_ids, dev)
    lora = to_dev_i32(li.lora_ids, dev)
    routing = mol.alloc_routing(wl.numel, wl.V, wl.BM, dev)
    ws = mol.alloc_workspace(wl.numel, wl.V, wl.BM, dev)
    stages = []
    for st in li.stages:
        stages.append(dict(st=st, x=st.x.to_device(dev), A=st.A.to_device(dev), B=st.B.to_device(dev),
                           out0=st.out0.to_device(dev),
                           out=torch.empty((wl.numel, st.stage.N), dtype=torch.bfloat16, device=dev),
                           inter=torch.zeros((wl.numel, st.stage.R), dtype=torch.float32, device=dev)))

    def layer():
        for si, d in enumerate(stages):
            d["out"].copy_(d["out0"])
            mol.mol_lora_forward(d["x"], d["st"].x_row_div, topk, lora, wl.E, wl.L, d["A"], d["B"],
                                 d["st"].stage.S, wl.scale, d["out"], routing, d["inter"],
                                 compute_routing=(mode if si == 0 else 0), workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [bf16_host(d["out"]) for d in stages]
    eager_sorted = routing.sorted_token_ids.cpu().numpy()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer()
    for d in stages:
        d["out"].zero_()
    routing.sorted_token_ids.fill_(-9)
    for _ in range(20):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(routing.sorted_token_ids.cpu().numpy(), eager_sorted)
    for d, e in zip(stages, eager):
        assert np.array_equal(bf16_host(d["out"]), e)

    vt = oracle.virtual_topk(li.topk_ids, li.lora_ids, wl.E, wl.L).reshape(-1)
    s, ex, n = oracle.align_block_size(vt, wl.V, wl.BM)
    assert np.array_equal(eager_sorted, s)
    pairs = valid_pairs(s, ex, n, wl.BM, wl.numel)
    for d, e in zip(stages, eager):
        st = d["st"]
        ref = oracle.lora_forward_stage(st.x, st.x_row_div, li.topk_ids, li.lora_ids, wl.E, wl.L,
                                        st.A, st.B, st.stage.S, st.stage.r, st.stage.Ns, wl.scale,
                                        None, st.out0.host_all(), wl.BM)
        check_out(e, ref["out"], pairs)
