"""A bounded wait that runs out: the kernel records a fault bit, leaves, and the device stays usable.

mol_debug_wait_test makes the shrink's producer warps leave before they issue
any copy, so every consumer's wait on a stage finds nothing arriving and gives
up after the (shortened) wall-clock limit. No copy is in flight, nothing traps
and nothing hangs: the call returns, mol_take_fault_flags reports bit 0, no
intermediate row was written, and a normal forward right after it on the same
device matches the oracle with no bit set.
"""

import numpy as np
import pytest

import oracle
from tests.gpu_util import (bf16_host, check_inter, check_out, mol_lib, to_dev_bf16, to_dev_i32,
                            torch_cuda, valid_pairs)

pytestmark = pytest.mark.gpu


def bits(a):
    return oracle.f64_to_bf16(np.asarray(a, np.float64))


def _inputs(rng):
    T, k, E, L, BM, K, S, r, Ns = 23, 8, 16, 4, 16, 1024, 2, 32, 96
    numel, V = T * k, E * L
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    lora = rng.integers(-1, L, size=T).astype(np.int32)
    x = bits(rng.standard_normal((T, K)))
    A = bits(rng.standard_normal((V, S * r, K)) * 0.05)
    B = bits(rng.standard_normal((V, S * Ns, r)) * 0.05)
    out0 = bits(rng.standard_normal((numel, S * Ns)))
    return dict(T=T, k=k, E=E, L=L, BM=BM, K=K, S=S, r=r, Ns=Ns, numel=numel, V=V, topk=topk,
                lora=lora, x=x, A=A, B=B, out0=out0)


def test_wait_runs_out_sets_flag_then_device_recovers():
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    c = _inputs(np.random.default_rng(5))
    numel, V, BM, R = c["numel"], c["V"], c["BM"], c["S"] * c["r"]
    mol.mol_take_fault_flags()  # clear whatever earlier tests left

    vid = oracle.virtual_topk(c["topk"], c["lora"], c["E"], c["L"]).reshape(-1)
    s, e, n = oracle.align_block_size(vid, V, BM)
    routing = mol.Routing(to_dev_i32(vid, dev), to_dev_i32(s, dev), to_dev_i32(e, dev),
                          torch.tensor([n], dtype=torch.int32, device=dev), BM, numel, V)
    x_d, A_d = to_dev_bf16(c["x"], dev), to_dev_bf16(c["A"], dev)
    inter = torch.full((numel, R), float("nan"), dtype=torch.float32, device=dev)
    try:
        mol.mol_debug_wait_test(True, 2_000_000)  # waits give up after 2 ms
        mol.mol_lora_shrink(x_d, c["k"], A_d, c["S"], routing, inter)
        flags = mol.mol_take_fault_flags()
    finally:
        mol.mol_debug_wait_test(False, 0)
    assert flags == 1
    assert torch.all(torch.isnan(inter)), "no job ran, so no intermediate row was written"

    # same process, same device: a normal forward is exact against the oracle, no bit set
    out_d = to_dev_bf16(c["out0"], dev)
    inter2 = torch.full((numel, R), float("nan"), dtype=torch.float32, device=dev)
    routing2 = mol.alloc_routing(numel, V, BM, dev)
    mol.mol_lora_forward(x_d, c["k"], to_dev_i32(c["topk"], dev), to_dev_i32(c["lora"], dev),
                         c["E"], c["L"], A_d, to_dev_bf16(c["B"], dev), c["S"], 0.5, out_d,
                         routing2, inter2)
    torch.cuda.synchronize()
    assert mol.mol_take_fault_flags() == 0
    ref_inter = oracle.lora_shrink(c["x"], c["k"], c["A"], s, e, n, BM, numel,
                                   np.full((numel, R), np.nan, np.float32))
    ref_out = oracle.lora_expand(ref_inter, c["B"], c["S"], c["r"], c["Ns"], 0.5, None, s, e, n,
                                 BM, numel, c["out0"])
    pairs = valid_pairs(s, e, n, BM, numel)
    check_inter(inter2.cpu().numpy(), ref_inter, pairs)
    check_out(bf16_host(out_d), ref_out, pairs)


def test_wait_limit_restored_by_default():
    """Setting the limit to 0 restores the one-second default: a normal shrink records nothing."""
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    c = _inputs(np.random.default_rng(6))
    numel, V, BM, R = c["numel"], c["V"], c["BM"], c["S"] * c["r"]
    mol.mol_debug_wait_test(False, 0)
    vid = oracle.virtual_topk(c["topk"], c["lora"], c["E"], c["L"]).reshape(-1)
    s, e, n = oracle.align_block_size(vid, V, BM)
    routing = mol.Routing(to_dev_i32(vid, dev), to_dev_i32(s, dev), to_dev_i32(e, dev),
                          torch.tensor([n], dtype=torch.int32, device=dev), BM, numel, V)
    inter = torch.full((numel, R), float("nan"), dtype=torch.float32, device=dev)
    mol.mol_lora_shrink(to_dev_bf16(c["x"], dev), c["k"], to_dev_bf16(c["A"], dev), c["S"], routing,
                        inter)
    assert mol.mol_take_fault_flags() == 0
    ref = oracle.lora_shrink(c["x"], c["k"], c["A"], s, e, n, BM, numel,
                             np.full((numel, R), np.nan, np.float32))
    check_inter(inter.cpu().numpy(), ref, valid_pairs(s, e, n, BM, numel))


def test_tc_expand_wait_runs_out_sets_flag_then_device_recovers():
    """The tensor-core expand (full routed blocks of rank 64): with its weight producer issuing
    nothing, the MMA, epilogue, copier and converter waits all run out; the call returns, bit 0
    is reported, no output row changed, and a normal expand right after matches the oracle."""
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(7)
    T, k, E, BM, S, Ns, r = 256, 2, 4, 64, 2, 256, 64
    numel, V, N = T * k, E, S * Ns
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    vid = oracle.virtual_topk(topk, np.zeros(T, np.int32), E, 1).reshape(-1)
    s, e, n = oracle.align_block_size(vid, V, BM)
    inter = (rng.standard_normal((numel, S * r))).astype(np.float32)
    B = bits(rng.standard_normal((V, N, r)) * 0.05)
    out0 = bits(rng.standard_normal((numel, N)))
    routing = mol.Routing(to_dev_i32(vid, dev), to_dev_i32(s, dev), to_dev_i32(e, dev),
                          torch.tensor([n], dtype=torch.int32, device=dev), BM, numel, V)
    inter_d, B_d = torch.from_numpy(inter).to(dev), to_dev_bf16(B, dev)
    mol.mol_take_fault_flags()
    out = to_dev_bf16(out0, dev)
    try:
        mol.mol_debug_wait_test(True, 2_000_000)  # waits give up after 2 ms
        mol.mol_lora_expand(inter_d, B_d, S, 0.5, routing, out)
        flags = mol.mol_take_fault_flags()
    finally:
        mol.mol_debug_wait_test(False, 0)
    assert flags == 1
    assert np.array_equal(bf16_host(out), out0), "no product ran, so no output row changed"

    out = to_dev_bf16(out0, dev)
    mol.mol_lora_expand(inter_d, B_d, S, 0.5, routing, out)
    torch.cuda.synchronize()
    assert mol.mol_take_fault_flags() == 0
    ref = oracle.lora_expand(inter, B, S, r, Ns, 0.5, None, s, e, n, BM, numel, out0)
    check_out(bf16_host(out), ref, valid_pairs(s, e, n, BM, numel))
