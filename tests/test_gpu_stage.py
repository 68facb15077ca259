"""The fused stage (shrink then expand per routed block in one launch) against the oracle.

mol_lora_forward takes the fused stage for small layers: every routed block
on an SM of its own (capacity / block_m at most the SM count), a virtual
expert's weights within two 52 KB stages (2 (R K + N r) bytes), rank 8, 16, 32
or 64, R <= 128, no per-adapter arrays, and not the tensor-core shrink's
regime. These cases are built to land there (`in_fused_regime` restates the
rule) and to reach its corners: a hot virtual expert whose routed block holds
more than 16 rows (the stage repeated per 16-row tile), k-chunked shrink jobs
(wide K with many rows), output widths that end inside a 256-column tile,
padded row strides, routed weights, one to three slices, and a second stage
that reuses the routing (its weights are read before the kernel's dependency
wait).
"""

import numpy as np
import pytest

import oracle
from tests.gpu_util import (bf16_host, check_inter, check_out, mol_lib, to_dev_bf16, to_dev_i32,
                            torch_cuda, valid_pairs)

pytestmark = pytest.mark.gpu


def in_fused_regime(numel, V, BM, K, S, r, Ns, sms=148):
    cap = oracle.align_capacity(numel, V, BM)
    R, N = S * r, S * Ns
    tc = (R % 64 == 0 and K % 64 == 0 and BM in (64, 128) and numel >= 32 * min(numel, V))
    return (r in (8, 16, 32, 64) and R <= 128 and not tc and cap // BM <= sms
            and 2 * (R * K + N * r) <= 2 * 52 * 1024)


def bits(a):
    return oracle.f64_to_bf16(np.asarray(a, np.float64))


CASES = [
    # T, k, E, L, BM, K, S, r, Ns, hot, x_pad, out_pad, weights
    (16, 2, 8, 2, 16, 256, 1, 16, 128, 0.0, 0, 0, False),       # the tiny workload's widths
    (10, 4, 8, 2, 16, 2048, 1, 8, 64, 0.9, 8, 8, True),         # rank 8, hot block: k-chunked jobs
    (40, 2, 4, 2, 64, 128, 2, 16, 40, 0.8, 16, 0, True),        # hot expert: > 16 rows, row tiles
    (12, 4, 6, 2, 16, 64, 1, 64, 296, 0.2, 8, 8, True),         # rank 64, column tail 40
    (30, 3, 5, 2, 32, 96, 3, 32, 24, 0.8, 0, 24, False),        # three slices, rank 32, hot
    (60, 2, 3, 1, 128, 64, 2, 16, 8, 0.9, 0, 0, False),         # one hot block of 128 slots
]

@pytest.mark.parametrize("case", CASES)
def test_fused_stage_matches_oracle(case):
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    T, k, E, L, BM, K, S, r, Ns, hot, x_pad, out_pad, use_w = case
    rng = np.random.default_rng(sum(case[:9]))
    numel, V, R, N = T * k, E * L, S * r, S * Ns
    assert in_fused_regime(numel, V, BM, K, S, r, Ns)
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    lora = rng.integers(-1, L, size=T).astype(np.int32)
    hot_t = rng.random(T) < hot  # a hot virtual expert: expert 0 with adapter 0
    for t in np.nonzero(hot_t)[0]:
        if 0 not in topk[t]:
            topk[t, 0] = 0
    lora[hot_t] = 0
    topk[rng.random((T, k)) < 0.1] = -1
    x_full = bits(rng.standard_normal((T, K + x_pad)))
    A = bits(rng.standard_normal((V, R, K)) * 0.05)
    B = bits(rng.standard_normal((V, N, r)) * 0.05)
    out_full = bits(rng.standard_normal((numel, N + out_pad)))
    w = rng.random(numel).astype(np.float32) if use_w else None

    vt = oracle.virtual_topk(topk, lora, E, L).reshape(-1)
    s, e, n = oracle.align_block_size(vt, V, BM)
    if BM > 16:  # one routed block holds several 16-row tiles
        assert np.bincount(vt[vt >= 0], minlength=V).max() > 16
    pairs = valid_pairs(s, e, n, BM, numel)
    others = np.setdiff1d(np.arange(numel), pairs)

    routing = mol.alloc_routing(numel, V, BM, dev)
    ws = mol.alloc_workspace(numel, V, BM, dev)
    inter = torch.full((numel, R), float("nan"), dtype=torch.float32, device=dev)
    out_d = to_dev_bf16(out_full, dev)
    mol.mol_lora_forward(to_dev_bf16(x_full, dev)[:, :K], k, to_dev_i32(topk, dev),
                         to_dev_i32(lora, dev), E, L, to_dev_bf16(A, dev), to_dev_bf16(B, dev), S,
                         0.5, out_d[:, :N], routing, inter, compute_routing=True, workspace=ws,
                         topk_weights=None if w is None else torch.from_numpy(w).to(dev))
    torch.cuda.synchronize()
    assert mol.mol_take_fault_flags() == 0
    assert np.array_equal(routing.sorted_token_ids.cpu().numpy(), s)

    ref_inter = oracle.lora_shrink(x_full[:, :K], k, A, s, e, n, BM, numel,
                                   np.full((numel, R), np.nan, np.float32))
    ref_out = oracle.lora_expand(ref_inter, B, S, r, Ns, 0.5, w, s, e, n, BM, numel,
                                 out_full[:, :N])
    g_inter, g_out = inter.cpu().numpy(), bf16_host(out_d)
    check_inter(g_inter, ref_inter, pairs)
    check_out(g_out[:, :N], ref_out, pairs)
    assert np.all(np.isnan(g_inter[others]))
    assert np.array_equal(g_out[others], out_full[others])
    assert np.array_equal(g_out[:, N:], out_full[:, N:])  # padding columns never written

    # a second stage on the same routing (pair-row activations), read early
    K2, r2, Ns2 = 256 + 8 * (case[0] % 5), r, 136
    assert in_fused_regime(numel, V, BM, K2, 1, r2, Ns2)
    x2 = bits(rng.standard_normal((numel, K2)))
    A2 = bits(rng.standard_normal((V, r2, K2)) * 0.05)
    B2 = bits(rng.standard_normal((V, Ns2, r2)) * 0.05)
    o2 = bits(rng.standard_normal((numel, Ns2)))
    inter2 = torch.full((numel, r2), float("nan"), dtype=torch.float32, device=dev)
    out2 = to_dev_bf16(o2, dev)
    mol.mol_lora_forward(to_dev_bf16(x2, dev), 1, None, None, E, L, to_dev_bf16(A2, dev),
                         to_dev_bf16(B2, dev), 1, 2.0, out2, routing, inter2,
                         compute_routing=False, num_tokens=T, topk=k)
    torch.cuda.synchronize()
    assert mol.mol_take_fault_flags() == 0
    ri2 = oracle.lora_shrink(x2, 1, A2, s, e, n, BM, numel, np.full((numel, r2), np.nan, np.float32))
    ro2 = oracle.lora_expand(ri2, B2, 1, r2, Ns2, 2.0, None, s, e, n, BM, numel, o2)
    g2 = bf16_host(out2)
    check_inter(inter2.cpu().numpy(), ri2, pairs)
    check_out(g2, ro2, pairs)
    assert np.array_equal(g2[others], o2[others])


@pytest.mark.parametrize("r", [8, 16, 32, 64])
def test_fused_stage_small_integers_bit_exact(r):
    """Integer-valued inputs make every fp32 sum exact: the fused stage must match bit for bit."""
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(900 + r)
    T, k, E, L, BM, K, S, Ns = 30, 4, 24, 2, 16, 128, 2, 40
    numel, V, R, N = T * k, E * L, S * r, S * Ns
    assert in_fused_regime(numel, V, BM, K, S, r, Ns)
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    lora = rng.integers(-1, L, size=T).astype(np.int32)
    x = bits(rng.integers(-3, 4, size=(T, K)))
    A = bits(rng.integers(-3, 4, size=(V, R, K)))
    B = bits(rng.integers(-2, 3, size=(V, N, r)))
    out0 = bits(rng.integers(-8, 9, size=(numel, N)))
    routing = mol.alloc_routing(numel, V, BM, dev)
    inter = torch.full((numel, R), float("nan"), dtype=torch.float32, device=dev)
    out = to_dev_bf16(out0, dev)
    mol.mol_lora_forward(to_dev_bf16(x, dev), k, to_dev_i32(topk, dev), to_dev_i32(lora, dev), E, L,
                         to_dev_bf16(A, dev), to_dev_bf16(B, dev), S, 1.0, out, routing, inter)
    torch.cuda.synchronize()
    vt = oracle.virtual_topk(topk, lora, E, L).reshape(-1)
    s, e, n = oracle.align_block_size(vt, V, BM)
    ref_inter = oracle.lora_shrink(x, k, A, s, e, n, BM, numel, np.full((numel, R), np.nan, np.float32))
    ref_out = oracle.lora_expand(ref_inter, B, S, r, Ns, 1.0, None, s, e, n, BM, numel, out0)
    g = inter.cpu().numpy()
    assert np.array_equal(np.isnan(g), np.isnan(ref_inter))
    assert np.array_equal(g[~np.isnan(g)], ref_inter[~np.isnan(ref_inter)])
    assert np.array_equal(bf16_host(out), ref_out)
