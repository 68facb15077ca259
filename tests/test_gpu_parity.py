"""GPU parity of the MoL LoRA path against the CPU oracle on the workload shapes.

Routing outputs (virtual ids, sorted_token_ids, expert_ids,
num_tokens_post_padded) must be bit-exact. fp32 intermediates must satisfy
|gpu - ref| <= 1e-3 (|ref| + rms(row)); bf16 outputs |gpu - ref| <= 1e-2 (1 + |ref|).
Every workload is compared everywhere: every routing output, and the
intermediates and outputs of every pair that gets a delta (the large ones once,
seed 0; the small ones for seeds 0-4).
"""

import numpy as np
import pytest

import oracle
from synth import WORKLOADS, make_layer
from tests.gpu_util import (bf16_host, check_inter, check_out, mol_lib, to_dev_i32, torch_cuda,
                            valid_pairs)

pytestmark = pytest.mark.gpu


def run_layer_gpu(wl, li, dev, mode=1):
    """All stages of one layer through mol_lora_forward (routing computed by the first stage,
    with compute_routing = mode)."""
    import torch

    mol = mol_lib()
    topk = to_dev_i32(li.topk_ids, dev)
    lora = to_dev_i32(li.lora_ids, dev)
    routing = mol.alloc_routing(wl.numel, wl.V, wl.BM, dev)
    ws = mol.alloc_workspace(wl.numel, wl.V, wl.BM, dev)
    res = []
    for si, st in enumerate(li.stages):
        x = st.x.to_device(dev)
        A = st.A.to_device(dev)
        B = st.B.to_device(dev)
        out = st.out0.to_device(dev)
        inter = torch.full((wl.numel, st.stage.R), float("nan"), dtype=torch.float32, device=dev)
        mol.mol_lora_forward(x, st.x_row_div, topk, lora, wl.E, wl.L, A, B, st.stage.S, wl.scale,
                             out, routing, inter, compute_routing=(mode if si == 0 else 0),
                             workspace=ws)
        torch.cuda.synchronize()
        res.append((inter.cpu().numpy(), bf16_host(out)))
        del x, A, B, out, inter
    rt = dict(vtopk=routing.vtopk_ids.cpu().numpy(), sorted_ids=routing.sorted_token_ids.cpu().numpy(),
              expert_ids=routing.expert_ids.cpu().numpy(),
              ntpp=int(routing.num_tokens_post_padded.item()))
    return rt, res


def check_routing(wl, li, rt):
    vt = oracle.virtual_topk(li.topk_ids, li.lora_ids, wl.E, wl.L).reshape(-1)
    s, e, n = oracle.align_block_size(vt, wl.V, wl.BM)
    assert np.array_equal(rt["vtopk"].reshape(-1), vt)
    assert rt["ntpp"] == n
    assert np.array_equal(rt["sorted_ids"], s)
    assert np.array_equal(rt["expert_ids"], e)
    return s, e, n


@pytest.mark.parametrize("name", ["tiny", "decode", "wide", "wide1k"])
@pytest.mark.parametrize("seed", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("mode", [1, 2])
def test_full_parity_small(name, seed, mode):
    """mode 2: the ids are declared ready early; at these sizes the shrink computes its own
    items' routing from them (the align still writes the routing the other kernels read)."""
    torch = torch_cuda()
    dev = torch.device("cuda:0")
    wl = WORKLOADS[name]
    li = make_layer(wl, seed)
    rt, res = run_layer_gpu(wl, li, dev, mode)
    s, e, n = check_routing(wl, li, rt)
    pairs = valid_pairs(s, e, n, wl.BM, wl.numel)
    others = np.setdiff1d(np.arange(wl.numel), pairs)
    for st, (g_inter, g_out) in zip(li.stages, res):
        out0 = st.out0.host_all()
        ref_inter = oracle.lora_shrink(st.x, st.x_row_div, st.A, s, e, n, wl.BM, wl.numel,
                                       np.full((wl.numel, st.stage.R), np.nan, np.float32))
        ref_out = oracle.lora_expand(ref_inter, st.B, st.stage.S, st.stage.r, st.stage.Ns,
                                     wl.scale, None, s, e, n, wl.BM, wl.numel, out0)
        check_inter(g_inter, ref_inter, pairs)
        check_out(g_out, ref_out, pairs)
        assert np.all(np.isnan(g_inter[others]))             # rows without a delta: not written
        assert np.array_equal(g_out[others], out0[others])   # and bit-unchanged


@pytest.mark.slow
@pytest.mark.parametrize("name", ["prefill", "ep", "dense"])
def test_full_parity_large(name):
    """Full-size workloads: routing bit-exact, and both stages' intermediates and outputs
    compared with the oracle on every routed block (every pair that gets a delta)."""
    torch = torch_cuda()
    dev = torch.device("cuda:0")
    wl = WORKLOADS[name]
    li = make_layer(wl, seed=0)
    rt, res = run_layer_gpu(wl, li, dev)
    s, e, n = check_routing(wl, li, rt)
    pairs = valid_pairs(s, e, n, wl.BM, wl.numel)
    assert pairs.size == np.count_nonzero(rt["vtopk"] >= 0)  # every valid pair is in a real block
    others = np.setdiff1d(np.arange(wl.numel), pairs)
    for st, (g_inter, g_out) in zip(li.stages, res):
        out0 = st.out0.host_all()
        ref_inter = oracle.lora_shrink(st.x, st.x_row_div, st.A, s, e, n, wl.BM, wl.numel,
                                       np.full((wl.numel, st.stage.R), np.nan, np.float32))
        check_inter(g_inter, ref_inter, pairs)
        assert np.all(np.isnan(g_inter[others]))             # rows without a delta: not written
        ref_out = oracle.lora_expand(ref_inter, st.B, st.stage.S, st.stage.r, st.stage.Ns,
                                     wl.scale, None, s, e, n, wl.BM, wl.numel, out0)
        check_out(g_out, ref_out, pairs)
        assert np.array_equal(g_out[others], out0[others])   # and bit-unchanged
