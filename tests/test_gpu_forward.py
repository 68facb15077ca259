"""mol_lora_forward against the oracle, call after call on the same buffers.

Shapes cover one and several k chunks per shrink job (whole-K jobs and
chunked ones), every supported rank, slices, token or pair activation rows,
crowded buckets (several row groups per routed block) and spare capacity.
"""

import numpy as np
import pytest

import oracle
from tests.gpu_util import (bf16_host, check_inter, check_out, mol_lib, to_dev_bf16, to_dev_i32,
                            torch_cuda, valid_pairs)

pytestmark = pytest.mark.gpu


def bits(a):
    return oracle.f64_to_bf16(np.asarray(a, np.float64))


CASES = [
    # T, k, E, L, BM, K, S, r, Ns, token_rows, weights, extra_blocks
    (23, 8, 16, 4, 16, 2048, 2, 32, 96, True, False, 0),
    (20, 4, 6, 2, 32, 768, 1, 16, 200, False, True, 3),
    (30, 6, 5, 3, 64, 520, 3, 64, 72, True, False, 1),
    (9, 8, 4, 2, 16, 4104, 1, 128, 136, True, True, 0),
    (200, 8, 8, 2, 128, 256, 2, 32, 48, False, False, 2),   # crowded buckets: several row groups
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("use_ws", [True, False])
@pytest.mark.parametrize("mode", [1, 2])
def test_forward_paths(case, use_ws, mode):
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    T, k, E, L, BM, K, S, r, Ns, token_rows, use_w, extra = case
    rng = np.random.default_rng(sum(case[:9]))
    numel, V, R, N = T * k, E * L, S * r, S * Ns
    topk = np.stack([rng.permutation(E)[:k] if k <= E else rng.integers(0, E, k) for _ in range(T)]).astype(np.int32)
    topk[rng.random((T, k)) < 0.1] = -1
    lora = rng.integers(-1, L, size=T).astype(np.int32)
    rows_x = T if token_rows else numel
    xdiv = k if token_rows else 1
    x = bits(rng.standard_normal((rows_x, K)))
    A = bits(rng.standard_normal((V, R, K)) * 0.05)
    B = bits(rng.standard_normal((V, N, r)) * 0.05)
    w = rng.random(numel).astype(np.float32) if use_w else None

    cap = mol.align_capacity(numel, V, BM) + extra * BM
    i32 = dict(dtype=torch.int32, device=dev)
    routing = mol.Routing(torch.empty(numel, **i32), torch.empty(cap, **i32),
                          torch.empty(cap // BM, **i32), torch.empty(1, **i32), BM, numel, V)
    ws = mol.alloc_workspace(numel, V, BM, dev) if use_ws else None
    xd, Ad, Bd = to_dev_bf16(x, dev), to_dev_bf16(A, dev), to_dev_bf16(B, dev)
    wd = None if w is None else torch.from_numpy(w).to(dev)

    vt = oracle.virtual_topk(topk, lora, E, L).reshape(-1)
    s, e, n = oracle.align_block_size(vt, V, BM, cap)
    pairs = valid_pairs(s, e, n, BM, numel)
    others = np.setdiff1d(np.arange(numel), pairs)
    for call in range(3):  # same workspace, fresh outputs each call
        out0 = bits(rng.standard_normal((numel, N)))
        out = to_dev_bf16(out0, dev)
        inter = torch.full((numel, R), float("nan"), dtype=torch.float32, device=dev)
        mol.mol_lora_forward(xd, xdiv, to_dev_i32(topk, dev), to_dev_i32(lora, dev), E, L, Ad, Bd, S,
                             0.5, out, routing, inter, compute_routing=mode, topk_weights=wd,
                             workspace=ws)
        torch.cuda.synchronize()
        assert np.array_equal(routing.sorted_token_ids.cpu().numpy(), s)
        assert np.array_equal(routing.expert_ids.cpu().numpy(), e)
        ref_inter = oracle.lora_shrink(x, xdiv, A, s, e, n, BM, numel,
                                       np.full((numel, R), np.nan, np.float32))
        ref_out = oracle.lora_expand(ref_inter, B, S, r, Ns, 0.5, w, s, e, n, BM, numel, out0)
        g_inter, g_out = inter.cpu().numpy(), bf16_host(out)
        check_inter(g_inter, ref_inter, pairs)
        check_out(g_out, ref_out, pairs)
        assert np.all(np.isnan(g_inter[others]))
        assert np.array_equal(g_out[others], out0[others])


@pytest.mark.parametrize("token_rows", [True, False])
def test_empty_batch(token_rows):
    """No tokens: inputs built from empty arrays (whose strides may be 0) are accepted; the
    stage computing the routing launches only the align, which writes an empty routing
    (num_tokens_post_padded = 0); the stage reusing it launches nothing; no fault."""
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    T, k, E, L, BM, K, S, r, Ns = 0, 8, 16, 4, 16, 256, 2, 32, 96
    V, R, N = E * L, S * r, S * Ns
    x = to_dev_bf16(bits(np.zeros((0, K + 8))), dev)[:, :K]
    topk = to_dev_i32(np.zeros((0, k), np.int32), dev)
    lora = to_dev_i32(np.zeros(0, np.int32), dev)
    A = to_dev_bf16(bits(np.ones((V, R, K)) * 0.01), dev)
    B = to_dev_bf16(bits(np.ones((V, N, r)) * 0.01), dev)
    out = to_dev_bf16(bits(np.zeros((0, N))), dev)
    inter = torch.zeros((0, R), dtype=torch.float32, device=dev)
    routing = mol.alloc_routing(0, V, BM, dev)
    routing.num_tokens_post_padded.fill_(-7)
    xdiv = k if token_rows else 1
    before = mol.mol_launch_count()
    mol.mol_lora_forward(x, xdiv, topk, lora, E, L, A, B, S, 0.5, out, routing, inter,
                         compute_routing=True, workspace=mol.alloc_workspace(0, V, BM, dev))
    torch.cuda.synchronize()
    assert mol.mol_launch_count() == before + 1
    assert int(routing.num_tokens_post_padded.cpu().item()) == 0
    mol.mol_lora_forward(x, xdiv, None, None, E, L, A, B, S, 0.5, out, routing, inter,
                         compute_routing=False, num_tokens=0, topk=k)
    torch.cuda.synchronize()
    assert mol.mol_launch_count() == before + 1
    assert mol.mol_take_fault_flags() == 0
