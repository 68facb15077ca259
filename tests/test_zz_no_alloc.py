"""The no-allocation align entry point against the regular one.

mol_align_block_size_noalloc serves callers that cannot allocate device
memory when they route a batch (a runtime that owns nearly all of HBM and
hands an operator only its inputs and outputs, or a loop that cannot afford
an allocation's implicit synchronisation). It uses a 1 MiB scratch array
compiled into the library instead of a caller workspace (up to 131072 pairs the
align needs no scratch at all; the cases here are mostly larger, with few
enough buckets that the scratch holds them). Its results must be
bit-identical to mol_align_block_size's and to the oracle's, call after call,
even though the scratch keeps whatever the previous call left in it.

This file is collected last so that a failure here comes after every other test.
"""

import ctypes

import numpy as np
import pytest

import oracle
from tests.gpu_util import mol_lib, to_dev_i32, torch_cuda

pytestmark = pytest.mark.gpu


def _routing(torch, mol, numel, V, BM, dev, fill):
    cap = mol.align_capacity(numel, V, BM)
    i32 = dict(dtype=torch.int32, device=dev)
    return (torch.full((cap,), fill, **i32), torch.full((cap // BM,), fill, **i32),
            torch.full((1,), fill, **i32), cap)


def _noalloc(lib, torch, vid, numel, V, BM, out):
    s, e, n, cap = out
    return lib.mol_align_block_size_noalloc(
        ctypes.c_void_p(vid.data_ptr()), numel, V, BM, ctypes.c_void_p(s.data_ptr()), cap,
        ctypes.c_void_p(e.data_ptr()), ctypes.c_void_p(n.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _regular(lib, torch, mol, vid, numel, V, BM, out):
    s, e, n, cap = out
    ws = mol.alloc_workspace(numel, V, BM, vid.device)
    return lib.mol_align_block_size(
        ctypes.c_void_p(vid.data_ptr()), numel, V, BM, ctypes.c_void_p(s.data_ptr()), cap,
        ctypes.c_void_p(e.data_ptr()), ctypes.c_void_p(n.data_ptr()),
        None if ws is None else ctypes.c_void_p(ws.data_ptr()), 0 if ws is None else ws.numel(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("numel,V,BM", [(200000, 100, 16), (240000, 127, 64), (150000, 255, 32),
                                        (65536, 4096, 64), (184, 1024, 16)])
def test_noalloc_matches_regular_two_calls_in_a_row(numel, V, BM):
    torch = torch_cuda()
    mol = mol_lib()
    lib = mol.library()
    dev = torch.device("cuda:0")
    for call in range(2):
        rng = np.random.default_rng(1000 * call + numel)
        vid = to_dev_i32(rng.integers(-2, V + 2, size=numel).astype(np.int32), dev)
        got = _routing(torch, mol, numel, V, BM, dev, -55)
        want = _routing(torch, mol, numel, V, BM, dev, -66)
        assert _noalloc(lib, torch, vid, numel, V, BM, got) == mol.MOL_OK
        assert _regular(lib, torch, mol, vid, numel, V, BM, want) == mol.MOL_OK
        torch.cuda.synchronize()
        for g, w in zip(got[:3], want[:3]):
            assert torch.equal(g, w), f"call {call}: outputs differ"
        # and against the oracle directly (the sorted ids, block experts and padded count)
        s, e, n = oracle.align_block_size(vid.cpu().numpy(), V, BM, capacity=got[3])
        assert int(got[2].item()) == n
        assert np.array_equal(got[0].cpu().numpy(), s)
        assert np.array_equal(got[1].cpu().numpy(), e)


def _largest_accepted(mol, V, BM):
    """Largest numel whose align workspace fits the 1 MiB scratch (workspace grows with numel)."""
    lo, hi = 0, mol.MOL_MAX_NUMEL
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if mol.workspace_bytes(mid, V, BM) <= (1 << 20):
            lo = mid
        else:
            hi = mid - 1
    return lo


def test_noalloc_accepts_the_largest_size_that_fits_and_rejects_the_next():
    torch = torch_cuda()
    mol = mol_lib()
    lib = mol.library()
    dev = torch.device("cuda:0")
    assert _largest_accepted(mol, 8191, 16) == 131072  # the size the header states for 8192 buckets
    V, BM = 100, 16  # few buckets: the largest accepted size runs on the scratch array
    top = _largest_accepted(mol, V, BM)
    assert top > 131072 and 0 < mol.workspace_bytes(top, V, BM) <= (1 << 20)
    rng = np.random.default_rng(77)
    for _ in range(2):  # two calls in a row on the shared scratch
        vid = to_dev_i32(rng.integers(-1, V + 1, size=top).astype(np.int32), dev)
        out = _routing(torch, mol, top, V, BM, dev, -11)
        assert _noalloc(lib, torch, vid, top, V, BM, out) == mol.MOL_OK
        torch.cuda.synchronize()
        s, e, n = oracle.align_block_size(vid.cpu().numpy(), V, BM, capacity=out[3])
        assert int(out[2].item()) == n
        assert np.array_equal(out[0].cpu().numpy(), s)
        assert np.array_equal(out[1].cpu().numpy(), e)
    over = top + 1
    assert mol.workspace_bytes(over, V, BM) > (1 << 20)
    vid = torch.zeros(over, dtype=torch.int32, device=dev)
    out = _routing(torch, mol, over, V, BM, dev, -12)
    assert _noalloc(lib, torch, vid, over, V, BM, out) == mol.MOL_ERR_CAPACITY
    torch.cuda.synchronize()
    assert torch.all(out[0] == -12) and torch.all(out[2] == -12)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    torch = torch_cuda()
    mol = mol_lib()
    lib = mol.library()
    dev = torch.device("cuda:0")
    numel, V, BM = 200000, 8191, 16
    assert mol.workspace_bytes(numel, V, BM) > (1 << 20)
    vid = torch.zeros(numel, dtype=torch.int32, device=dev)
    out = _routing(torch, mol, numel, V, BM, dev, -77)
    assert _noalloc(lib, torch, vid, numel, V, BM, out) == mol.MOL_ERR_CAPACITY
    torch.cuda.synchronize()
    assert torch.all(out[0] == -77) and torch.all(out[2] == -77)
