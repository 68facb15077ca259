"""GPU parity of each C-ABI step on its own, and the edge cases of the method.

Each entry point is called with inputs both sides see (routing built by the
oracle where a step consumes one) and compared with the oracle: bit-exact for
remap and align, stated tolerances for the contractions, bit-exact again when
small-integer inputs make every sum exact.
"""

import numpy as np
import pytest

import oracle
from tests.gpu_util import (bf16_host, check_inter, check_out, mol_lib, to_dev_bf16, to_dev_i32,
                            torch_cuda, valid_pairs)

pytestmark = pytest.mark.gpu


def _dev():
    torch = torch_cuda()
    return torch, torch.device("cuda:0")


def bits(a):
    return oracle.f64_to_bf16(np.asarray(a, np.float64))


# ---------------------------------------------------------------- remap ----

@pytest.mark.parametrize("T,k,E,L", [(1, 1, 1, 1), (23, 8, 128, 8), (333, 6, 60, 7), (8192, 8, 256, 16)])
def test_virtual_topk(T, k, E, L):
    torch, dev = _dev()
    mol = mol_lib()
    rng = np.random.default_rng(T + k)
    topk = rng.integers(-3, E + 2, size=(T, k)).astype(np.int32)
    lora = rng.integers(-2, L + 2, size=T).astype(np.int32)
    got = mol.mol_virtual_topk(to_dev_i32(topk, dev), to_dev_i32(lora, dev), E, L)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), oracle.virtual_topk(topk, lora, E, L))


# ---------------------------------------------------------------- align ----

ALIGN_CASES = [
    # numel, V, BM, kind
    (0, 16, 16, "random"),
    (1, 1, 16, "random"),
    (37, 5, 32, "random"),
    (184, 1024, 16, "random"),
    (4096, 8191, 128, "random"),
    (4097, 100, 16, "random"),
    (32768, 8064, 64, "random"),
    (65536, 4096, 64, "random"),
    (70001, 8191, 64, "random"),
    (200000, 33, 16, "random"),
    (131072, 8191, 16, "random"),      # the largest one-cluster align
    (131073, 8191, 16, "random"),      # the smallest tiles-scan-scatter align
    (20000, 1, 16, "random"),          # fewer buckets than cluster blocks
    (12289, 3, 128, "random"),
    (5000, 64, 32, "all_invalid"),
    (3000, 64, 64, "single_bucket"),
    (9000, 8191, 16, "top_bucket"),
]


@pytest.mark.parametrize("numel,V,BM,kind", ALIGN_CASES)
@pytest.mark.parametrize("extra_blocks", [0, 3])
def test_align_block_size(numel, V, BM, kind, extra_blocks):
    torch, dev = _dev()
    mol = mol_lib()
    rng = np.random.default_rng(numel + V)
    if kind == "random":
        vid = rng.integers(-2, V + 2, size=numel).astype(np.int32)
    elif kind == "all_invalid":
        vid = rng.choice(np.array([-1, -7, V, V + 5], np.int32), size=numel)
    elif kind == "single_bucket":
        vid = np.full(numel, V // 2, np.int32)
    else:
        vid = np.where(rng.random(numel) < 0.5, V - 1, -1).astype(np.int32)
    cap = oracle.align_capacity(numel, V, BM) + extra_blocks * BM
    s_ref, e_ref, n_ref = oracle.align_block_size(vid, V, BM, cap)
    i32 = dict(dtype=torch.int32, device=dev)
    routing = mol.Routing(to_dev_i32(vid, dev), torch.full((cap,), -77, **i32),
                          torch.full((cap // BM,), -77, **i32), torch.full((1,), -77, **i32),
                          BM, numel, V)
    mol.mol_align_block_size(routing.vtopk_ids, V, BM, routing=routing)
    torch.cuda.synchronize()
    assert int(routing.num_tokens_post_padded.item()) == n_ref
    assert np.array_equal(routing.sorted_token_ids.cpu().numpy(), s_ref)
    assert np.array_equal(routing.expert_ids.cpu().numpy(), e_ref)


def test_align_is_reproducible():
    torch, dev = _dev()
    mol = mol_lib()
    vid = np.random.default_rng(9).integers(-1, 4096, size=65536).astype(np.int32)
    outs = []
    for _ in range(3):
        r = mol.mol_align_block_size(to_dev_i32(vid, dev), 4096, 64)
        torch.cuda.synchronize()
        outs.append((r.sorted_token_ids.cpu().numpy(), r.expert_ids.cpu().numpy()))
    for o in outs[1:]:
        assert np.array_equal(o[0], outs[0][0]) and np.array_equal(o[1], outs[0][1])


# ------------------------------------------------------- shrink / expand ----

def _routing_from_oracle(mol, vid, V, BM, dev):
    s, e, n = oracle.align_block_size(vid, V, BM)
    import torch

    r = mol.Routing(to_dev_i32(vid, dev), to_dev_i32(s, dev), to_dev_i32(e, dev),
                    torch.tensor([n], dtype=torch.int32, device=dev), BM, len(vid), V)
    return r, s, e, n


SHAPES = [
    # T, k, E, L, BM, K, S, r, Ns, token_rows, x_pad, out_pad, weights, sparse
    (16, 2, 8, 2, 16, 256, 1, 16, 128, True, 0, 0, False, 0.1),
    (23, 8, 16, 4, 16, 200, 2, 32, 40, True, 8, 16, False, 0.0),
    (50, 4, 3, 2, 64, 264, 1, 64, 136, False, 0, 8, True, 0.2),
    (300, 8, 4, 1, 128, 96, 3, 16, 1000, True, 16, 0, False, 0.3),
    (64, 8, 2, 2, 32, 512, 1, 128, 72, False, 8, 8, True, 0.0),
    (97, 3, 5, 3, 16, 8, 2, 16, 8, False, 0, 0, False, 0.5),
    (12, 4, 3, 2, 16, 7168, 1, 16, 64, True, 0, 0, False, 0.0),    # one weight-tile buffer
    (40, 8, 6, 2, 32, 4096, 2, 32, 96, True, 0, 0, False, 0.1),    # two buffers
    (6, 2, 2, 1, 16, 65536, 1, 16, 16, True, 8, 0, False, 0.0),    # largest K of the contract
    (20, 2, 2, 1, 32, 64, 8, 128, 16, False, 0, 8, False, 0.0),    # largest R = 8 x 128
    (30, 4, 5, 2, 16, 320, 1, 8, 200, True, 8, 8, True, 0.1),      # rank 8, one slice (R = 8)
    (25, 2, 3, 2, 32, 128, 2, 8, 48, False, 0, 0, False, 0.2),     # rank 8, two slices
    # four to 32 pairs per virtual expert: 16-row shrink items, 512-column expand items
    # with a ragged last item
    (120, 8, 16, 4, 32, 256, 2, 16, 1288, True, 0, 8, True, 0.1),
    (100, 6, 12, 3, 16, 136, 1, 8, 1096, False, 8, 0, False, 0.2),
    (90, 8, 12, 2, 16, 200, 2, 16, 768, True, 0, 8, True, 0.1),    # 768-column items
]


@pytest.mark.parametrize("shape", SHAPES)
def test_shrink_and_expand_entries(shape):
    torch, dev = _dev()
    mol = mol_lib()
    T, k, E, L, BM, K, S, r, Ns, token_rows, x_pad, out_pad, use_w, sparse = shape
    rng = np.random.default_rng(sum(shape[:9]))
    numel, V, R, N = T * k, E * L, S * r, S * Ns
    topk = rng.integers(0, E, size=(T, k)).astype(np.int32)
    topk[rng.random((T, k)) < sparse] = -1
    lora = rng.integers(-1, L, size=T).astype(np.int32)
    vid = oracle.virtual_topk(topk, lora, E, L).reshape(-1)
    routing, s, e, n = _routing_from_oracle(mol, vid, V, BM, dev)
    rows_x = T if token_rows else numel
    xdiv = k if token_rows else 1
    x_full = bits(rng.standard_normal((rows_x, K + x_pad)))
    A = bits(rng.standard_normal((V, R, K)) * 0.05)
    B = bits(rng.standard_normal((V, N, r)) * 0.05)
    out_full = bits(rng.standard_normal((numel, N + out_pad)))
    w = rng.random(numel).astype(np.float32) if use_w else None

    x_d = to_dev_bf16(x_full, dev)[:, :K]
    inter = torch.full((numel, R), float("nan"), dtype=torch.float32, device=dev)
    mol.mol_lora_shrink(x_d, xdiv, to_dev_bf16(A, dev), S, routing, inter)
    ref_inter = oracle.lora_shrink(x_full[:, :K], xdiv, A, s, e, n, BM, numel,
                                   np.full((numel, R), np.nan, np.float32))
    torch.cuda.synchronize()
    g_inter = inter.cpu().numpy()
    pairs = valid_pairs(s, e, n, BM, numel)
    check_inter(g_inter, ref_inter, pairs)
    others = np.setdiff1d(np.arange(numel), pairs)
    assert np.all(np.isnan(g_inter[others]))

    # expand alone, on the oracle's intermediates (NaN on rows without a delta)
    out_d = to_dev_bf16(out_full, dev)
    mol.mol_lora_expand(torch.from_numpy(ref_inter).to(dev), to_dev_bf16(B, dev), S, 0.5, routing,
                        out_d[:, :N], topk_weights=None if w is None else torch.from_numpy(w).to(dev))
    torch.cuda.synchronize()
    ref_out = oracle.lora_expand(ref_inter, B, S, r, Ns, 0.5, w, s, e, n, BM, numel, out_full[:, :N])
    g_out = bf16_host(out_d)
    check_out(g_out[:, :N], ref_out, pairs)
    assert np.array_equal(g_out[others], out_full[others])          # untouched rows
    assert np.array_equal(g_out[:, N:], out_full[:, N:])            # padding columns untouched


@pytest.mark.parametrize("r", [8, 16, 32, 64, 128])
@pytest.mark.parametrize("BM", [16, 128])
def test_small_integers_bit_exact(r, BM):
    """Integer-valued inputs make every fp32 sum exact: the GPU must match bit for bit."""
    torch, dev = _dev()
    mol = mol_lib()
    rng = np.random.default_rng(r + BM)
    T, k, E, L, K, S, Ns = 40, 4, 6, 2, 128, 2, 24
    numel, V, R, N = T * k, E * L, S * r, S * Ns
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    topk[:, 0] = 1                                   # a crowded bucket: several row tiles
    lora = rng.integers(-1, L, size=T).astype(np.int32)
    vid = oracle.virtual_topk(topk, lora, E, L).reshape(-1)
    routing, s, e, n = _routing_from_oracle(mol, vid, V, BM, dev)
    x = bits(rng.integers(-3, 4, size=(T, K)))
    A = bits(rng.integers(-3, 4, size=(V, R, K)))
    B = bits(rng.integers(-2, 3, size=(V, N, r)))
    out0 = bits(rng.integers(-8, 9, size=(numel, N)))
    inter = torch.full((numel, R), float("nan"), dtype=torch.float32, device=dev)
    mol.mol_lora_shrink(to_dev_bf16(x, dev), k, to_dev_bf16(A, dev), S, routing, inter)
    out = to_dev_bf16(out0, dev)
    mol.mol_lora_expand(inter, to_dev_bf16(B, dev), S, 1.0, routing, out)
    torch.cuda.synchronize()
    ref_inter = oracle.lora_shrink(x, k, A, s, e, n, BM, numel, np.full((numel, R), np.nan, np.float32))
    ref_out = oracle.lora_expand(ref_inter, B, S, r, Ns, 1.0, None, s, e, n, BM, numel, out0)
    g = inter.cpu().numpy()
    assert np.array_equal(np.isnan(g), np.isnan(ref_inter))
    assert np.array_equal(g[~np.isnan(g)], ref_inter[~np.isnan(ref_inter)])
    assert np.array_equal(bf16_host(out), ref_out)


@pytest.mark.parametrize("E,BM,r,few_rows", [
    (64, 64, 32, True),    # 64 virtual experts, 128 pairs: one staged row tile at a time
    (64, 128, 64, True),
    (4, 64, 32, False),    # 4 virtual experts: the next row tile is prefetched
    (4, 128, 16, False),
    (4, 64, 8, False),
])
def test_expand_hot_expert_many_row_tiles(E, BM, r, few_rows):
    """One expert takes most pairs, so its routed blocks hold up to block_m rows (several
    16-row tiles), whether or not the call counts as many rows per virtual expert."""
    torch, dev = _dev()
    mol = mol_lib()
    rng = np.random.default_rng(E + BM + r)
    T, k, L, K, S, Ns = 64, 2, 1, 64, 2, 264
    numel, V, R, N = T * k, E * L, S * r, S * Ns
    assert (numel < 32 * min(numel, V)) == few_rows
    topk = np.where(rng.random((T, k)) < 0.85, 0, rng.integers(1, E, (T, k))).astype(np.int32)
    topk[:, 1] = np.where(topk[:, 0] == topk[:, 1], (topk[:, 1] + 1) % E, topk[:, 1])
    lora = np.zeros(T, np.int32)
    vid = oracle.virtual_topk(topk, lora, E, L).reshape(-1)
    routing, s, e, n = _routing_from_oracle(mol, vid, V, BM, dev)
    assert np.bincount(vid, minlength=V).max() > 32
    inter = rng.standard_normal((numel, R)).astype(np.float32)
    B = bits(rng.standard_normal((V, N, r)) * 0.05)
    out0 = bits(rng.standard_normal((numel, N)))
    w = rng.random(numel).astype(np.float32)
    out_d = to_dev_bf16(out0, dev)
    mol.mol_lora_expand(torch.from_numpy(inter).to(dev), to_dev_bf16(B, dev), S, 0.5, routing, out_d,
                        topk_weights=torch.from_numpy(w).to(dev))
    torch.cuda.synchronize()
    ref = oracle.lora_expand(inter, B, S, r, Ns, 0.5, w, s, e, n, BM, numel, out0)
    pairs = valid_pairs(s, e, n, BM, numel)
    g_out = bf16_host(out_d)
    check_out(g_out, ref, pairs)
    others = np.setdiff1d(np.arange(numel), pairs)
    assert np.array_equal(g_out[others], out0[others])


def test_expand_ignores_poisoned_rows():
    """NaN intermediates on rows outside every block never reach the output."""
    torch, dev = _dev()
    mol = mol_lib()
    rng = np.random.default_rng(4)
    T, k, E, L, BM, r, Ns = 30, 4, 5, 2, 16, 32, 64
    numel, V = T * k, E * L
    topk = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    lora = rng.integers(-1, L, size=T).astype(np.int32)
    vid = oracle.virtual_topk(topk, lora, E, L).reshape(-1)
    routing, s, e, n = _routing_from_oracle(mol, vid, V, BM, dev)
    pairs = valid_pairs(s, e, n, BM, numel)
    inter = rng.standard_normal((numel, r)).astype(np.float32)
    mask = np.ones(numel, bool)
    mask[pairs] = False
    inter[mask] = np.nan
    B = bits(rng.standard_normal((V, Ns, r)) * 0.1)
    out0 = bits(rng.standard_normal((numel, Ns)))
    out = to_dev_bf16(out0, dev)
    mol.mol_lora_expand(torch.from_numpy(inter).to(dev), to_dev_bf16(B, dev), 1, 2.0, routing, out)
    torch.cuda.synchronize()
    g = bf16_host(out)
    assert np.array_equal(g[mask], out0[mask])
    assert np.all(np.isfinite(oracle.bf16_to_f64(g[pairs])))
    ref = oracle.lora_expand(inter, B, 1, r, Ns, 2.0, None, s, e, n, BM, numel, out0)
    check_out(g, ref, pairs)


def test_empty_and_all_sentinel_forward():
    torch, dev = _dev()
    mol = mol_lib()
    E, L, BM, K, r, Ns = 8, 2, 16, 64, 16, 32
    V = E * L
    A = torch.zeros((V, r, K), dtype=torch.bfloat16, device=dev)
    B = torch.zeros((V, Ns, r), dtype=torch.bfloat16, device=dev)
    # zero tokens
    routing = mol.alloc_routing(0, V, BM, dev)
    x = torch.zeros((1, K), dtype=torch.bfloat16, device=dev)
    out = torch.zeros((1, Ns), dtype=torch.bfloat16, device=dev)
    inter = torch.zeros((1, r), dtype=torch.float32, device=dev)
    mol.mol_lora_forward(x, 1, torch.zeros((0, 4), dtype=torch.int32, device=dev),
                         torch.zeros(0, dtype=torch.int32, device=dev), E, L, A, B, 1, 1.0, out,
                         routing, inter)
    torch.cuda.synchronize()
    assert int(routing.num_tokens_post_padded.item()) == 0
    # every pair a sentinel or without adapter
    T, k = 20, 4
    topk = torch.full((T, k), -1, dtype=torch.int32, device=dev)
    topk[::2] = 3
    lora = torch.full((T,), -1, dtype=torch.int32, device=dev)
    lora[1::2] = 1
    routing = mol.alloc_routing(T * k, V, BM, dev)
    x = torch.randn((T, K), device=dev).to(torch.bfloat16)
    out = torch.randn((T * k, Ns), device=dev).to(torch.bfloat16)
    out0 = out.clone()
    inter = torch.full((T * k, r), float("nan"), dtype=torch.float32, device=dev)
    mol.mol_lora_forward(x, k, topk, lora, E, L, A, B, 1, 1.0, out, routing, inter)
    torch.cuda.synchronize()
    assert int(routing.num_tokens_post_padded.item()) == 80
    assert torch.all(routing.expert_ids == -1)
    assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
    assert torch.all(torch.isnan(inter))


def test_invalid_arguments_launch_nothing():
    torch, dev = _dev()
    mol = mol_lib()
    lib = mol.library()
    i32 = dict(dtype=torch.int32, device=dev)
    vid = torch.zeros(64, **i32)
    s = torch.full((4096,), -5, **i32)
    e = torch.full((256,), -5, **i32)
    n = torch.full((1,), -5, **i32)
    P = lambda t: None if t is None else t.data_ptr()
    st = lambda: torch.cuda.current_stream().cuda_stream
    assert lib.mol_align_block_size(P(vid), 64, 16, 48, P(s), 4096, P(e), P(n), None, 0, st()) == mol.MOL_ERR_UNSUPPORTED
    assert lib.mol_align_block_size(P(vid), 64, 16, 16, P(s), 16, P(e), P(n), None, 0, st()) == mol.MOL_ERR_CAPACITY
    assert lib.mol_align_block_size(P(vid), 64, 8192, 16, P(s), 4096, P(e), P(n), None, 0, st()) == mol.MOL_ERR_UNSUPPORTED
    assert lib.mol_align_block_size(P(vid), -1, 16, 16, P(s), 4096, P(e), P(n), None, 0, st()) == mol.MOL_ERR_INVALID_ARG
    assert lib.mol_align_block_size(None, 64, 16, 16, P(s), 4096, P(e), P(n), None, 0, st()) == mol.MOL_ERR_INVALID_ARG
    big = 200000  # past the one-cluster align: a workspace is needed
    assert lib.mol_workspace_bytes(big, 100, 16) > 0
    assert lib.mol_align_block_size(P(vid), big, 100, 16, P(s), 1 << 20, P(e), P(n), None, 0, st()) in (mol.MOL_ERR_CAPACITY,)
    x = torch.zeros((8, 64), dtype=torch.bfloat16, device=dev)
    A = torch.zeros((16, 16, 64), dtype=torch.bfloat16, device=dev)
    inter = torch.zeros((64, 16), dtype=torch.float32, device=dev)
    # K not a multiple of 8, rank/slices not giving R % 8 == 0, misaligned pointer
    assert lib.mol_lora_shrink(P(x), 64, 8, 60, P(A), 1, 16, P(s), P(e), P(n), 4096, 16, 64, 16, P(inter), 0, None, st()) == mol.MOL_ERR_UNSUPPORTED
    assert lib.mol_lora_shrink(P(x), 64, 8, 64, P(A), 1, 12, P(s), P(e), P(n), 4096, 16, 64, 16, P(inter), 0, None, st()) == mol.MOL_ERR_UNSUPPORTED
    assert lib.mol_lora_shrink(P(x) + 2, 64, 8, 64, P(A), 1, 16, P(s), P(e), P(n), 4096, 16, 64, 16, P(inter), 0, None, st()) == mol.MOL_ERR_UNSUPPORTED
    assert lib.mol_lora_expand(P(inter), P(A), 1, 24, 16, 1.0, None, P(s), P(e), P(n), 4096, 16, 64, 16, P(x), 64, 0, None, None, st()) == mol.MOL_ERR_UNSUPPORTED
    assert lib.mol_lora_expand(P(inter), P(A), 1, 16, 12, 1.0, None, P(s), P(e), P(n), 4096, 16, 64, 16, P(x), 64, 0, None, None, st()) == mol.MOL_ERR_UNSUPPORTED
    assert lib.mol_lora_expand(P(inter), P(A), 2, 16, 64, 1.0, None, P(s), P(e), P(n), 4096, 16, 64, 16, P(x), 64, 0, None, None, st()) == mol.MOL_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(s == -5) and torch.all(e == -5) and torch.all(n == -5)
    assert torch.all(inter == 0)
    with pytest.raises(mol.MolError):
        mol.mol_align_block_size(vid, 8191, 48)


def test_no_wait_ran_out():
    """After a forward on every path, no kernel recorded a bounded wait running out."""
    torch = torch_cuda()
    mol = mol_lib()
    mol.mol_take_fault_flags()  # clear whatever earlier tests left
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(11)
    for (T, k, E, BM, K, R, N) in [(23, 8, 16, 16, 2048, 64, 256), (256, 2, 4, 64, 256, 128, 64)]:
        numel, V = T * k, E
        topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        lora = np.zeros(T, np.int32)
        x = to_dev_bf16(oracle.f64_to_bf16(rng.standard_normal((T, K))), dev)
        A = to_dev_bf16(oracle.f64_to_bf16(rng.standard_normal((V, R, K)) * 0.05), dev)
        B = to_dev_bf16(oracle.f64_to_bf16(rng.standard_normal((V, 2 * N, R // 2)) * 0.05), dev)
        out = torch.zeros((numel, 2 * N), dtype=torch.bfloat16, device=dev)
        routing = mol.alloc_routing(numel, V, BM, dev)
        inter = torch.empty((numel, R), dtype=torch.float32, device=dev)
        mol.mol_lora_forward(x, k, to_dev_i32(topk, dev), to_dev_i32(lora, dev), E, 1, A, B, 2, 1.0,
                             out, routing, inter)
    assert mol.mol_take_fault_flags() == 0
