"""The persistent fused stage against the two-launch path and the oracle.

Given a workspace of mol_forward_workspace_bytes, mol_lora_forward runs a stage
with few rows per virtual expert as one persistent launch: shrink items, then
expand items that wait (bounded) on their routed block's count of finished
shrink jobs. Without that workspace the same call runs a shrink launch and an
expand launch. Both use the same arithmetic in the same order, so their
results must be bit-identical; both must match the oracle; and the counts left
in the workspace must let the next calls (the same stage again, and a second
stage reusing the routing) run correctly.
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
    # T, k, E, L, BM, K, S, r, Ns, hot, weights
    (23, 8, 64, 4, 16, 2048, 2, 32, 768, 0.0, False),    # the decode gate_up widths
    (23, 8, 64, 4, 16, 768, 1, 32, 2048, 0.0, True),     # decode down widths
    (30, 4, 48, 2, 32, 2056, 2, 16, 200, 0.9, False),    # a hot block of > 16 rows: two row tiles
    (30, 6, 64, 3, 16, 264, 3, 8, 1024, 0.2, True),      # rank 8, three slices
    (12, 8, 32, 2, 64, 1032, 1, 64, 296, 0.5, False),    # rank 64, 64-slot blocks, column tail
]


def _small_layer(numel, V, BM, K, S, r, Ns, sms=148):
    """The rule under which mol_lora_forward takes the one-block-per-routed-block stage instead."""
    cap = oracle.align_capacity(numel, V, BM)
    return cap // BM <= sms and 2 * (S * r * K + S * Ns * r) <= 2 * 52 * 1024


def _case(case):
    T, k, E, L, BM, K, S, r, Ns, hot, use_w = case
    rng = np.random.default_rng(sum(case[:9]) + 17)
    numel, V = T * k, E * L
    assert numel < 4 * min(numel, V)  # few rows per virtual expert: the persistent stage's regime
    assert not _small_layer(numel, V, BM, K, S, r, Ns)
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    lora = rng.integers(-1, L, size=T).astype(np.int32)
    hot_t = rng.random(T) < hot
    for t in np.nonzero(hot_t)[0]:
        if 0 not in topk[t]:
            topk[t, 0] = 0
    lora[hot_t] = 0
    topk[rng.random((T, k)) < 0.05] = -1
    return dict(T=T, k=k, E=E, L=L, BM=BM, K=K, S=S, r=r, Ns=Ns, numel=numel, V=V, topk=topk,
                lora=lora, x=bits(rng.standard_normal((T, K))),
                A=bits(rng.standard_normal((V, S * r, K)) * 0.05),
                B=bits(rng.standard_normal((V, S * Ns, r)) * 0.05),
                out0=bits(rng.standard_normal((numel, S * Ns))),
                w=rng.random(numel).astype(np.float32) if use_w else None,
                x2=bits(rng.standard_normal((numel, 264))),
                A2=bits(rng.standard_normal((V, r, 264)) * 0.05),
                B2=bits(rng.standard_normal((V, 136, r)) * 0.05),
                o2=bits(rng.standard_normal((numel, 136))))


def _layer(mol, torch, c, dev, ws):
    """Gate_up-like stage computing the routing, then a down-like stage reusing it."""
    numel, V, BM, R = c["numel"], c["V"], c["BM"], c["S"] * c["r"]
    routing = mol.alloc_routing(numel, V, BM, dev)
    inter = torch.full((numel, R), float("nan"), dtype=torch.float32, device=dev)
    out = to_dev_bf16(c["out0"], dev)
    w = None if c["w"] is None else torch.from_numpy(c["w"]).to(dev)
    mol.mol_lora_forward(to_dev_bf16(c["x"], dev), c["k"], to_dev_i32(c["topk"], dev),
                         to_dev_i32(c["lora"], dev), c["E"], c["L"], to_dev_bf16(c["A"], dev),
                         to_dev_bf16(c["B"], dev), c["S"], 0.5, out, routing, inter,
                         compute_routing=True, topk_weights=w, workspace=ws)
    inter2 = torch.full((numel, c["r"]), float("nan"), dtype=torch.float32, device=dev)
    out2 = to_dev_bf16(c["o2"], dev)
    mol.mol_lora_forward(to_dev_bf16(c["x2"], dev), 1, None, None, c["E"], c["L"],
                         to_dev_bf16(c["A2"], dev), to_dev_bf16(c["B2"], dev), 1, 2.0, out2,
                         routing, inter2, compute_routing=False, workspace=ws,
                         num_tokens=c["T"], topk=c["k"])
    torch.cuda.synchronize()
    return (inter.cpu().numpy(), bf16_host(out), inter2.cpu().numpy(), bf16_host(out2),
            routing.sorted_token_ids.cpu().numpy())


@pytest.mark.parametrize("case", CASES)
def test_persistent_stage_bit_identical_to_two_launches_and_matches_oracle(case):
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    c = _case(case)
    numel, V, BM = c["numel"], c["V"], c["BM"]
    ws_full = mol.alloc_workspace(numel, V, BM, dev)               # persistent stage
    ws_align = mol.alloc_workspace(numel, V, BM, dev, stage=False)  # shrink + expand launches
    assert ws_full is not None and (ws_align is None or ws_full.numel() > ws_align.numel())
    mol.mol_take_fault_flags()
    two = _layer(mol, torch, c, dev, ws_align)
    runs = [_layer(mol, torch, c, dev, ws_full) for _ in range(3)]  # the counts reset every call
    assert mol.mol_take_fault_flags() == 0
    for got in runs:
        for g, t in zip(got, two):
            assert np.array_equal(g, t, equal_nan=True)
    # and the oracle
    vt = oracle.virtual_topk(c["topk"], c["lora"], c["E"], c["L"]).reshape(-1)
    s, e, n = oracle.align_block_size(vt, V, BM)
    assert np.array_equal(two[4], s)
    pairs = valid_pairs(s, e, n, BM, numel)
    others = np.setdiff1d(np.arange(numel), pairs)
    R = c["S"] * c["r"]
    ri = oracle.lora_shrink(c["x"], c["k"], c["A"], s, e, n, BM, numel,
                            np.full((numel, R), np.nan, np.float32))
    ro = oracle.lora_expand(ri, c["B"], c["S"], c["r"], c["Ns"], 0.5, c["w"], s, e, n, BM, numel,
                            c["out0"])
    check_inter(two[0], ri, pairs)
    check_out(two[1], ro, pairs)
    assert np.all(np.isnan(two[0][others]))
    assert np.array_equal(two[1][others], c["out0"][others])
    ri2 = oracle.lora_shrink(c["x2"], 1, c["A2"], s, e, n, BM, numel,
                             np.full((numel, c["r"]), np.nan, np.float32))
    ro2 = oracle.lora_expand(ri2, c["B2"], 1, c["r"], 136, 2.0, None, s, e, n, BM, numel, c["o2"])
    check_inter(two[2], ri2, pairs)
    check_out(two[3], ro2, pairs)
    assert np.array_equal(two[3][others], c["o2"][others])


def test_persistent_stage_counts_left_at_zero():
    """After a layer, both count arrays in the workspace are zero again."""
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    c = _case(CASES[0])
    numel, V, BM = c["numel"], c["V"], c["BM"]
    ws = mol.alloc_workspace(numel, V, BM, dev)
    align_part = mol.workspace_bytes(numel, V, BM)
    nblk = mol.align_capacity(numel, V, BM) // BM
    ws[align_part:].fill_(0x7F)  # garbage: the align of the first stage zeroes the counts
    _layer(mol, torch, c, dev, ws)
    assert mol.mol_take_fault_flags() == 0
    counts = ws[align_part:align_part + 8 * nblk].view(torch.int32)
    assert int(counts.abs().sum().item()) == 0


def test_launches_per_layer():
    """The library's launch count: a decode-like layer is 3 launches with the persistent stage
    (align, gate_up stage, down stage) and 5 without it (align, then a shrink and an expand per
    stage)."""
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    c = _case(CASES[0])
    numel, V, BM = c["numel"], c["V"], c["BM"]
    for stage, want in ((True, 3), (False, 5)):
        ws = mol.alloc_workspace(numel, V, BM, dev, stage=stage)
        n0 = mol.mol_launch_count()
        _layer(mol, torch, c, dev, ws)
        assert mol.mol_launch_count() - n0 == want
