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


# ------------------------------------------------------------------ tcgen05 expand
#
# The expand of full routed blocks of rank 64 runs on tcgen05 when the slice
# width is a multiple of 128 and no adapter arrays are passed. Shapes: one to
# three slices, one m-tile up to a ragged group of nine (two items per routed
# block and slice), both BLOCK_M values, padded output rows, routed weights,
# sentinel pairs, and one hot expert.

EXPAND_CASES = [
    # T, k, E, BM, S, Ns, token-row weights, sentinel fraction, out_pad, hot expert
    (256, 2, 4, 64, 1, 128, False, 0.0, 0, False),
    (300, 4, 8, 64, 2, 256, True, 0.1, 8, False),
    (512, 2, 4, 128, 1, 1152, False, 0.05, 0, False),
    (200, 8, 16, 64, 3, 384, True, 0.0, 16, False),
    (130, 2, 2, 128, 2, 128, False, 0.2, 0, True),
    (700, 4, 8, 64, 1, 2048, False, 0.1, 0, True),
]


def _expand_case(case, seed):
    T, k, E, BM, S, Ns, use_w, sent, out_pad, hot = case
    rng = np.random.default_rng(seed)
    r, V, numel, N = 64, E, T * k, S * Ns
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    if hot:
        topk[:, 0] = 0
    topk[rng.random((T, k)) < sent] = -1
    vt = oracle.virtual_topk(topk, np.zeros(T, np.int32), E, 1).reshape(-1)
    assert numel >= 32 * min(numel, V)
    inter = (rng.standard_normal((numel, S * r)) * 2.0).astype(np.float32)
    B = bits(rng.standard_normal((V, N, r)) * 0.05)
    out0 = bits(rng.standard_normal((numel, N + out_pad)))
    w = rng.random(numel).astype(np.float32) if use_w else None
    return dict(T=T, k=k, E=E, BM=BM, S=S, Ns=Ns, r=r, V=V, numel=numel, N=N, topk=topk, vt=vt,
                inter=inter, B=B, out0=out0, w=w, out_pad=out_pad)


@pytest.mark.parametrize("case", EXPAND_CASES)
def test_tc_expand_matches_oracle(case):
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    c = _expand_case(case, sum(case[:6]))
    V, BM, numel, N, S = c["V"], c["BM"], c["numel"], c["N"], c["S"]
    s, e, n = oracle.align_block_size(c["vt"], V, BM)
    pairs = valid_pairs(s, e, n, BM, numel)
    others = np.setdiff1d(np.arange(numel), pairs)
    ref = oracle.lora_expand(c["inter"], c["B"], S, 64, c["Ns"], 0.5, c["w"], s, e, n, BM, numel,
                             c["out0"][:, :N])
    routing = mol.alloc_routing(numel, V, BM, dev)
    mol.mol_align_block_size(to_dev_i32(c["vt"], dev), V, BM, routing=routing)
    out = to_dev_bf16(c["out0"], dev)
    wd = None if c["w"] is None else torch.from_numpy(c["w"]).to(dev)
    for call in range(2):  # the second call adds the delta again: compare the first
        if call:
            out = to_dev_bf16(c["out0"], dev)
        mol.mol_lora_expand(torch.from_numpy(c["inter"]).to(dev), to_dev_bf16(c["B"], dev), S, 0.5,
                            routing, out[:, :N], topk_weights=wd)
        torch.cuda.synchronize()
        assert mol.mol_take_fault_flags() == 0
        g = bf16_host(out)
        check_out(g[:, :N], ref, pairs)
        assert np.array_equal(g[others], c["out0"][others])          # rows without a delta
        assert np.array_equal(g[:, N:], c["out0"][:, N:])            # padding columns


@pytest.mark.parametrize("BM", [64, 128])
def test_tc_expand_small_integers_exact(BM):
    """Integer intermediates and weights: every sum is exact, so the bf16 output equals the
    oracle's bit for bit (the intermediate's tail is zero)."""
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    T, k, E, S, Ns = 512, 2, 4, 2, 256
    rng = np.random.default_rng(9 + BM)
    numel, V, N = T * k, E, S * Ns
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    vt = oracle.virtual_topk(topk, np.zeros(T, np.int32), E, 1).reshape(-1)
    inter = rng.integers(-3, 4, (numel, S * 64)).astype(np.float32)
    B = bits(rng.integers(-2, 3, (V, N, 64)))
    out0 = bits(rng.integers(-64, 65, (numel, N)))
    s, e, n = oracle.align_block_size(vt, V, BM)
    ref = oracle.lora_expand(inter, B, S, 64, Ns, 0.5, None, s, e, n, BM, numel, out0)
    routing = mol.alloc_routing(numel, V, BM, dev)
    mol.mol_align_block_size(to_dev_i32(vt, dev), V, BM, routing=routing)
    out = to_dev_bf16(out0, dev)
    mol.mol_lora_expand(torch.from_numpy(inter).to(dev), to_dev_bf16(B, dev), S, 0.5, routing, out)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host(out), ref)


def test_tc_expand_forward_dense_shape():
    """A whole stage through mol_lora_forward on a dense-like shape (tcgen05 shrink and
    tcgen05 expand): routing bit-exact, intermediate and output against the oracle."""
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    T, k, E, BM, K, S, Ns = 512, 4, 8, 64, 512, 2, 384
    rng = np.random.default_rng(21)
    numel, V, R, N = T * k, E, S * 64, S * Ns
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    topk[rng.random((T, k)) < 0.05] = -1
    lora = np.zeros(T, np.int32)
    x = bits(rng.standard_normal((T, K)))
    A = bits(rng.standard_normal((V, R, K)) * 0.05)
    B = bits(rng.standard_normal((V, N, 64)) * 0.05)
    out0 = bits(rng.standard_normal((numel, N)))
    ref = oracle.lora_forward_stage(x, k, topk, lora, E, 1, A, B, S, 64, Ns, 0.5, None, out0, BM)
    routing = mol.alloc_routing(numel, V, BM, dev)
    inter = torch.full((numel, R), float("nan"), dtype=torch.float32, device=dev)
    out = to_dev_bf16(out0, dev)
    mol.mol_lora_forward(to_dev_bf16(x, dev), k, to_dev_i32(topk, dev), to_dev_i32(lora, dev), E, 1,
                         to_dev_bf16(A, dev), to_dev_bf16(B, dev), S, 0.5, out, routing, inter,
                         workspace=mol.alloc_workspace(numel, V, BM, dev))
    torch.cuda.synchronize()
    assert mol.mol_take_fault_flags() == 0
    s, e, n = ref["sorted_ids"], ref["expert_ids"], ref["ntpp"]
    assert np.array_equal(routing.sorted_token_ids.cpu().numpy(), s)
    pairs = valid_pairs(s, e, n, BM, numel)
    check_inter(inter.cpu().numpy(), ref["inter"], pairs)
    check_out(bf16_host(out), ref["out"], pairs)
