"""The tensor-core (tcgen05) shrink against the oracle.

It runs when every routed block is full enough for a real contraction: at
least 32 pairs per virtual expert on average, R a multiple of 64, K a
multiple of 64 and BLOCK_M 64 or 128 (one adapter for every token, as in the
`dense` workload). Shapes here take that path with several k stages, several
128-row tiles of R, partial blocks, sentinels and both BLOCK_M values.
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
    # T, k, E, BM, K, S, r, Ns, token_rows, sentinel fraction
    (256, 2, 4, 64, 256, 2, 64, 96, True, 0.0),
    (300, 4, 8, 64, 512, 1, 128, 64, False, 0.1),
    (512, 2, 4, 128, 192, 2, 128, 72, True, 0.05),
    (200, 8, 16, 64, 1024, 2, 64, 40, True, 0.0),
    (130, 2, 2, 128, 128, 1, 128, 32, False, 0.2),
    (256, 2, 4, 64, 64, 2, 64, 32, True, 0.0),      # one k stage
    (300, 4, 8, 64, 512, 1, 64, 64, False, 0.1),    # R = 64: half a tile
    (256, 3, 4, 64, 256, 3, 64, 48, True, 0.0),     # R = 192: one and a half tiles
    (256, 2, 4, 64, 8192, 1, 64, 32, True, 0.0),    # long K: 128 stages per item
]


@pytest.mark.parametrize("case", CASES)
def test_tc_shrink_matches_oracle(case):
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    T, k, E, BM, K, S, r, Ns, token_rows, sent = case
    rng = np.random.default_rng(sum(case[:8]))
    L, V, R, N, numel = 1, E, S * r, S * Ns, T * k
    assert numel >= 32 * min(numel, V) and R % 64 == 0 and K % 64 == 0
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    topk[rng.random((T, k)) < sent] = -1
    lora = np.zeros(T, np.int32)
    xdiv = k if token_rows else 1
    x = bits(rng.standard_normal((T if token_rows else numel, K)))
    A = bits(rng.standard_normal((V, R, K)) * 0.05)
    B = bits(rng.standard_normal((V, N, r)) * 0.05)
    out0 = bits(rng.standard_normal((numel, N)))
    vt = oracle.virtual_topk(topk, lora, E, L).reshape(-1)
    s, e, n = oracle.align_block_size(vt, V, BM)
    ref_inter = oracle.lora_shrink(x, xdiv, A, s, e, n, BM, numel, np.full((numel, R), np.nan, np.float32))
    ref_out = oracle.lora_expand(ref_inter, B, S, r, Ns, 0.5, None, s, e, n, BM, numel, out0)
    pairs = valid_pairs(s, e, n, BM, numel)
    others = np.setdiff1d(np.arange(numel), pairs)

    routing = mol.alloc_routing(numel, V, BM, dev)
    ws = mol.alloc_workspace(numel, V, BM, dev)
    xd, Ad, Bd = to_dev_bf16(x, dev), to_dev_bf16(A, dev), to_dev_bf16(B, dev)
    for call in range(2):
        out = to_dev_bf16(out0, dev)
        inter = torch.full((numel, R), float("nan"), dtype=torch.float32, device=dev)
        mol.mol_lora_forward(xd, xdiv, to_dev_i32(topk, dev), to_dev_i32(lora, dev), E, L, Ad, Bd, S,
                             0.5, out, routing, inter, workspace=ws)
        torch.cuda.synchronize()
        g_inter, g_out = inter.cpu().numpy(), bf16_host(out)
        check_inter(g_inter, ref_inter, pairs)
        check_out(g_out, ref_out, pairs)
        assert np.all(np.isnan(g_inter[others]))
        assert np.array_equal(g_out[others], out0[others])


def test_tc_shrink_small_integers_exact():
    """Integer-valued bf16 inputs with exact fp32 sums: the tensor-core result is bit-exact."""
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    T, k, E, BM, K, R = 256, 2, 4, 64, 256, 128
    rng = np.random.default_rng(5)
    numel, V = T * k, E
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    x = bits(rng.integers(-3, 4, (T, K)))
    A = bits(rng.integers(-3, 4, (V, R, K)))
    vt = oracle.virtual_topk(topk, np.zeros(T, np.int32), E, 1).reshape(-1)
    s, e, n = oracle.align_block_size(vt, V, BM)
    ref = oracle.lora_shrink(x, k, A, s, e, n, BM, numel, np.full((numel, R), np.nan, np.float32))
    routing = mol.alloc_routing(numel, V, BM, dev)
    mol.mol_align_block_size(to_dev_i32(vt, dev), V, BM, routing=routing)
    inter = torch.full((numel, R), float("nan"), dtype=torch.float32, device=dev)
    mol.mol_lora_shrink(to_dev_bf16(x, dev), k, to_dev_bf16(A, dev), 1, routing, inter)
    torch.cuda.synchronize()
    assert np.array_equal(inter.cpu().numpy(), ref)
