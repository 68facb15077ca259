"""Per-adapter rank and scaling, and per-token adapter ids, on the GPU against the oracle."""

import numpy as np
import pytest

import oracle
from tests.gpu_util import (bf16_host, check_inter, check_out, mol_lib, to_dev_bf16, to_dev_i32,
                            torch_cuda, valid_pairs)

pytestmark = pytest.mark.gpu


def bits(a):
    return oracle.f64_to_bf16(np.asarray(a, np.float64))


# ------------------------------------------------------------------ token ids

def _token_case(seed, nreq, max_len, L, with_ranks, tail):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, max_len + 1, nreq)
    seg = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    num_tokens = int(seg[-1]) + tail
    wi = rng.integers(-2, L + 2, nreq).astype(np.int32)
    ranks = rng.choice([0, 8, 16, 64], L).astype(np.int32) if with_ranks else None
    return wi, seg, num_tokens, ranks


@pytest.mark.parametrize("seed,nreq,max_len,L,with_ranks,tail", [
    (0, 1, 5, 1, False, 0), (1, 7, 9, 3, True, 2), (2, 64, 40, 8, True, 0),
    (3, 300, 400, 16, False, 5), (4, 1000, 1, 63, True, 3), (5, 0, 1, 4, False, 6),
    (6, 4096, 64, 8, True, 1),
])
def test_token_lora_ids(seed, nreq, max_len, L, with_ranks, tail):
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    wi, seg, num_tokens, ranks = _token_case(seed, nreq, max_len, L, with_ranks, tail)
    ref = oracle.token_lora_ids(wi, seg, num_tokens, L, ranks)
    out = torch.full((num_tokens,), -7, dtype=torch.int32, device=dev)
    mol.mol_token_lora_ids(to_dev_i32(wi, dev), to_dev_i32(seg, dev), num_tokens, L,
                           None if ranks is None else to_dev_i32(ranks, dev), out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref)


def test_token_lora_ids_golden_guard():
    import json
    import os
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))
    g = g["token_lora_ids_guard"]
    args = (to_dev_i32(np.array(g["weight_indices"]), dev), to_dev_i32(np.array(g["seg_indptr"]), dev),
            g["num_tokens"], g["max_loras"])
    assert mol.mol_token_lora_ids(*args).cpu().tolist() == g["expected_no_ranks"]
    ranks = to_dev_i32(np.array(g["lora_ranks"]), dev)
    assert mol.mol_token_lora_ids(*args, lora_ranks=ranks).cpu().tolist() == g["expected_with_ranks"]


# ------------------------------------------------------------------ ranks and scalings

CASES = [
    # T, k, E, L, BM, K, S, r, Ns, token_rows, ranks per adapter
    (23, 8, 16, 4, 16, 2048, 2, 32, 96, True, [32, 8, 0, 24]),
    (20, 4, 6, 3, 32, 768, 1, 16, 200, False, [16, 0, 8]),
    (30, 6, 5, 3, 64, 520, 2, 64, 72, True, [40, 64, 16]),
    (9, 8, 4, 2, 16, 4104, 1, 128, 136, True, [128, 56]),
    (200, 8, 8, 2, 128, 256, 2, 32, 48, False, [16, 32]),
    # ranks that are not multiples of 8: weight chunks straddle the rank
    (40, 8, 8, 4, 16, 1032, 2, 32, 104, True, [5, 32, 19, 1]),
    (24, 4, 6, 3, 32, 776, 1, 16, 64, False, [3, 13, 16]),
    (16, 8, 8, 2, 64, 1544, 2, 64, 40, True, [33, 61]),
    # more than four expand items per resident block: blocks loop over items (rank 16:
    # 512-column items; rank 64: 256-column items), adapters of rank 0 skipped in the loop
    (600, 8, 64, 4, 16, 256, 2, 16, 2048, True, [16, 0, 8, 12]),
    (400, 8, 32, 4, 16, 128, 1, 64, 4096, False, [64, 0, 40, 17]),
    (1200, 8, 128, 4, 16, 128, 1, 8, 3072, True, [8, 0, 5, 3]),  # rank 8, 768-column items
]


def _setup(case, seed):
    T, k, E, L, BM, K, S, r, Ns, token_rows, ranks = case
    rng = np.random.default_rng(seed)
    V, R, N, numel = E * L, S * r, S * Ns, T * k
    topk = np.stack([rng.permutation(E)[:k] if k <= E else rng.integers(0, E, k) for _ in range(T)]).astype(np.int32)
    topk[rng.random((T, k)) < 0.1] = -1
    lora = rng.integers(-1, L, size=T).astype(np.int32)
    xdiv = k if token_rows else 1
    x = bits(rng.standard_normal((T if token_rows else numel, K)))
    A = bits(rng.standard_normal((V, R, K)) * 0.05)
    B = bits(rng.standard_normal((V, N, r)) * 0.05)
    scalings = rng.uniform(0.25, 2.0, L).astype(np.float32)
    out0 = bits(rng.standard_normal((numel, N)))
    return dict(T=T, k=k, E=E, L=L, BM=BM, K=K, S=S, r=r, Ns=Ns, V=V, R=R, numel=numel, topk=topk,
                lora=lora, xdiv=xdiv, x=x, A=A, B=B, ranks=np.array(ranks, np.int32),
                scalings=scalings, out0=out0)


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("path", ["forward", "steps"])
def test_ranks_and_scalings(case, path):
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    c = _setup(case, sum(case[:9]))
    E, L, V, BM, numel, S, r, Ns = c["E"], c["L"], c["V"], c["BM"], c["numel"], c["S"], c["r"], c["Ns"]
    vt = oracle.virtual_topk(c["topk"], c["lora"], E, L).reshape(-1)
    s, e, n = oracle.align_block_size(vt, V, BM)
    ref_inter = oracle.lora_shrink(c["x"], c["xdiv"], c["A"], s, e, n, BM, numel,
                                   np.full((numel, c["R"]), np.nan, np.float32), S, E, c["ranks"])
    ref_out = oracle.lora_expand(ref_inter, c["B"], S, r, Ns, 0.5, None, s, e, n, BM, numel, c["out0"],
                                 num_experts=E, lora_ranks=c["ranks"], lora_scalings=c["scalings"])
    pairs = valid_pairs(s, e, n, BM, numel)
    live = np.array([i for i in pairs if c["ranks"][vt[i] // E] > 0], np.int64)
    untouched = np.setdiff1d(np.arange(numel), live)

    routing = mol.alloc_routing(numel, V, BM, dev)
    xd, Ad, Bd = to_dev_bf16(c["x"], dev), to_dev_bf16(c["A"], dev), to_dev_bf16(c["B"], dev)
    ranks_d, scal_d = to_dev_i32(c["ranks"], dev), torch.from_numpy(c["scalings"]).to(dev)
    for call in range(2):
        out = to_dev_bf16(c["out0"], dev)
        inter = torch.full((numel, c["R"]), float("nan"), dtype=torch.float32, device=dev)
        if path == "forward":
            mol.mol_lora_forward(xd, c["xdiv"], to_dev_i32(c["topk"], dev), to_dev_i32(c["lora"], dev),
                                 E, L, Ad, Bd, S, 0.5, out, routing, inter, compute_routing=True,
                                 workspace=mol.alloc_workspace(numel, V, BM, dev),
                                 lora_ranks=ranks_d, lora_scalings=scal_d)
        else:
            mol.mol_virtual_topk(to_dev_i32(c["topk"], dev), to_dev_i32(c["lora"], dev), E, L,
                                 routing.vtopk_ids)
            mol.mol_align_block_size(routing.vtopk_ids, V, BM, routing=routing,
                                     workspace=mol.alloc_workspace(numel, V, BM, dev))
            mol.mol_lora_shrink(xd, c["xdiv"], Ad, S, routing, inter, lora_ranks=ranks_d, num_experts=E)
            mol.mol_lora_expand(inter, Bd, S, 0.5, routing, out, lora_ranks=ranks_d,
                                lora_scalings=scal_d, num_experts=E)
        torch.cuda.synchronize()
        g_inter, g_out = inter.cpu().numpy(), bf16_host(out)
        check_inter(g_inter, ref_inter, live)
        check_out(g_out, ref_out, live)
        assert np.all(np.isnan(g_inter[untouched]))
        assert np.array_equal(g_out[untouched], c["out0"][untouched])
        # columns past each adapter's rank are exact zeros
        for i in live[:64]:
            rl = c["ranks"][vt[i] // E]
            for sl in range(S):
                assert np.all(g_inter[i, sl * r + rl:(sl + 1) * r] == 0)


@pytest.mark.parametrize("case", CASES)
def test_padding_past_rank_is_ignored(case):
    """NaN in lora_a rows and lora_b columns past each adapter's rank, and (for the expand alone)
    in the intermediate columns past it, leaves every result as the oracle's, which reads none
    of them."""
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    c = _setup(case, 11 + sum(case[:9]))
    E, L, V, BM, numel, S, r, Ns = c["E"], c["L"], c["V"], c["BM"], c["numel"], c["S"], c["r"], c["Ns"]
    A, B = c["A"].copy(), c["B"].copy()
    for v in range(V):
        rl = int(c["ranks"][v // E])
        for sl in range(S):
            A[v, sl * r + rl:(sl + 1) * r, :] = 0x7FC0
        B[v, :, rl:] = 0x7FC0
    vt = oracle.virtual_topk(c["topk"], c["lora"], E, L).reshape(-1)
    s, e, n = oracle.align_block_size(vt, V, BM)
    ref_inter = oracle.lora_shrink(c["x"], c["xdiv"], A, s, e, n, BM, numel,
                                   np.full((numel, c["R"]), np.nan, np.float32), S, E, c["ranks"])
    ref_out = oracle.lora_expand(ref_inter, B, S, r, Ns, 0.5, None, s, e, n, BM, numel, c["out0"],
                                 num_experts=E, lora_ranks=c["ranks"], lora_scalings=c["scalings"])
    pairs = valid_pairs(s, e, n, BM, numel)
    live = np.array([i for i in pairs if c["ranks"][vt[i] // E] > 0], np.int64)
    assert live.size > 0

    routing = mol.alloc_routing(numel, V, BM, dev)
    xd, Ad, Bd = to_dev_bf16(c["x"], dev), to_dev_bf16(A, dev), to_dev_bf16(B, dev)
    ranks_d, scal_d = to_dev_i32(c["ranks"], dev), torch.from_numpy(c["scalings"]).to(dev)
    out = to_dev_bf16(c["out0"], dev)
    inter = torch.full((numel, c["R"]), float("nan"), dtype=torch.float32, device=dev)
    mol.mol_lora_forward(xd, c["xdiv"], to_dev_i32(c["topk"], dev), to_dev_i32(c["lora"], dev),
                         E, L, Ad, Bd, S, 0.5, out, routing, inter, compute_routing=True,
                         workspace=mol.alloc_workspace(numel, V, BM, dev),
                         lora_ranks=ranks_d, lora_scalings=scal_d)
    torch.cuda.synchronize()
    check_inter(inter.cpu().numpy(), ref_inter, live)
    check_out(bf16_host(out), ref_out, live)

    # the expand alone, on an intermediate whose columns past each rank hold NaN
    poisoned = ref_inter.copy()
    for i in live:
        rl = int(c["ranks"][vt[i] // E])
        for sl in range(S):
            poisoned[i, sl * r + rl:(sl + 1) * r] = np.nan
    ref_out2 = oracle.lora_expand(poisoned, B, S, r, Ns, 0.5, None, s, e, n, BM, numel, c["out0"],
                                  num_experts=E, lora_ranks=c["ranks"], lora_scalings=c["scalings"])
    assert np.array_equal(ref_out2, ref_out)
    out2 = to_dev_bf16(c["out0"], dev)
    mol.mol_lora_expand(torch.from_numpy(poisoned).to(dev), Bd, S, 0.5, routing, out2,
                        lora_ranks=ranks_d, lora_scalings=scal_d, num_experts=E)
    torch.cuda.synchronize()
    g_out2 = bf16_host(out2)
    check_out(g_out2, ref_out, live)
    untouched = np.setdiff1d(np.arange(numel), live)
    assert np.array_equal(g_out2[untouched], c["out0"][untouched])


def test_full_ranks_unit_scalings_bit_identical():
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    c = _setup(CASES[0], 3)
    E, L, V, BM, numel, S = c["E"], c["L"], c["V"], c["BM"], c["numel"], c["S"]
    xd, Ad, Bd = to_dev_bf16(c["x"], dev), to_dev_bf16(c["A"], dev), to_dev_bf16(c["B"], dev)
    res = []
    for adapters in (False, True):
        routing = mol.alloc_routing(numel, V, BM, dev)
        out = to_dev_bf16(c["out0"], dev)
        inter = torch.full((numel, c["R"]), float("nan"), dtype=torch.float32, device=dev)
        kw = {}
        if adapters:
            kw = dict(lora_ranks=torch.full((L,), c["r"], dtype=torch.int32, device=dev),
                      lora_scalings=torch.ones(L, dtype=torch.float32, device=dev))
        mol.mol_lora_forward(xd, c["xdiv"], to_dev_i32(c["topk"], dev), to_dev_i32(c["lora"], dev),
                             E, L, Ad, Bd, S, 0.5, out, routing, inter, **kw)
        torch.cuda.synchronize()
        res.append((inter.cpu().numpy(), bf16_host(out)))
    assert np.array_equal(res[0][0], res[1][0], equal_nan=True)
    assert np.array_equal(res[0][1], res[1][1])
