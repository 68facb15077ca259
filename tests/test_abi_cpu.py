"""CPU checks of the C-ABI library: it builds, loads, exports every declared symbol,
and its host-side arithmetic and argument validation behave as declared.

No call here reaches a kernel: validation rejects the arguments first, or the
entry point is pure host arithmetic.
"""

import ctypes
import os
import re
import shutil

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mol.h")

needs_nvcc = pytest.mark.skipif(not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def mol():
    from moe_lora_virtual_gb300.build import build_all

    build_all()
    import moe_lora_virtual_gb300 as m

    m.library()
    return m


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mol_\w+)\s*\(", src)))


@needs_nvcc
def test_exports_every_declared_symbol(mol):
    lib = mol.library()
    names = declared_functions()
    assert len(names) == 17
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(mol.EXPORTS)


@needs_nvcc
def test_checked_build_exports_the_same_symbols(mol):
    """libmol_checked.so is the same library with device-side index checks compiled in."""
    lib = mol.library()
    with mol.use_library(mol.CHECKED_LIB_PATH) as chk:
        for n in declared_functions():
            assert hasattr(chk, n), n
        assert mol.mol_checked_build() is True
        assert chk.mol_version() == lib.mol_version()
    assert mol.mol_checked_build() is False
    assert mol.library() is lib


def test_check_sites_match_header(mol):
    src = open(HEADER).read()
    sites = {int(v): k for k, v in re.findall(r"#define MOL_CHECK_(\w+) (\d+)", src)}
    assert sites == mol.CHECK_SITES


def test_check_record_decoding(mol):
    r = mol.decode_check_record((2 << 48) | 12345, 7)
    assert (r.count, r.site, r.value, r.site_name) == (7, 2, 12345, "ROUTE_PAIR")
    r = mol.decode_check_record((3 << 48) | ((-5) & 0xFFFFFFFFFFFF), 1)
    assert (r.site, r.value, r.site_name) == (3, -5, "ROUTE_NTPP")
    assert mol.decode_check_record(0, 0).site_name == "none"


@needs_nvcc
def test_status_strings_and_version(mol):
    lib = mol.library()
    assert lib.mol_version() == 100
    for code in (0, -1, -2, -3, -4, 7):
        assert isinstance(lib.mol_status_string(code), bytes)
    assert lib.mol_last_cuda_error() == 0
    assert lib.mol_launch_count() >= 0


@needs_nvcc
@pytest.mark.parametrize("numel,V,BM", [(0, 1, 16), (1, 1, 16), (184, 1024, 16), (32768, 8064, 64),
                                        (65536, 4096, 64), (10, 3, 4), (7, 100, 128)])
def test_capacity_matches_oracle(mol, numel, V, BM):
    assert mol.align_capacity(numel, V, BM) == oracle.align_capacity(numel, V, BM)


@needs_nvcc
def test_workspace_sizes(mol):
    assert mol.workspace_bytes(184, 1024, 16) == 0          # one block does the whole align
    assert mol.workspace_bytes(4096, 8191, 16) == 0
    assert mol.workspace_bytes(65536, 4096, 64) == 0        # one cluster does the whole align
    assert mol.workspace_bytes(131072, 8191, 16) == 0
    w = mol.workspace_bytes(131073, 4096, 64)               # tiles, scan and scatter launches
    assert w >= 4 * (33 * 4097 + 4097 + 131073) and w % 256 == 0
    assert mol.workspace_bytes(1 << 22, 8191, 16) <= 4 * (128 * 8192 + 8192 + (1 << 22)) + 256
    assert mol.workspace_bytes(-1, 16, 16) == 0
    assert mol.workspace_bytes(16, 8192, 16) == 0           # rejected sizes report 0


@needs_nvcc
def test_validation_rejects_before_any_launch(mol):
    lib = mol.library()
    P = ctypes.c_void_p
    # align: bad block_m, bucket cap, negative sizes, capacity, missing workspace
    assert lib.mol_align_block_size(P(16), 64, 16, 48, P(16), 4096, P(16), P(16), None, 0, None) == -3
    assert lib.mol_align_block_size(P(16), 64, 8192, 16, P(16), 4096, P(16), P(16), None, 0, None) == -3
    assert lib.mol_align_block_size(P(16), -5, 16, 16, P(16), 4096, P(16), P(16), None, 0, None) == -1
    assert lib.mol_align_block_size(P(16), 64, 16, 16, P(16), 64, P(16), P(16), None, 0, None) == -2
    assert lib.mol_align_block_size(P(16), 200000, 16, 16, P(16), 1 << 20, P(16), P(16), None, 0, None) == -2
    assert lib.mol_align_block_size(P(16), (1 << 22) + 1, 16, 16, P(16), 1 << 30, P(16), P(16), None, 0, None) == -3
    # shrink / expand contracts
    assert lib.mol_lora_shrink(P(16), 64, 1, 60, P(16), 1, 16, P(16), P(16), P(16), 64, 16, 8, 4, P(16), 0, None, None) == -3
    assert lib.mol_lora_shrink(P(16), 64, 1, 64, P(16), 1, 12, P(16), P(16), P(16), 64, 16, 8, 4, P(16), 0, None, None) == -3
    # rank 8 is inside the contract: the shape checks pass and the missing pointer is reported
    assert lib.mol_lora_shrink(None, 64, 1, 64, P(16), 1, 8, P(16), P(16), P(16), 64, 16, 8, 4, P(16), 0, None, None) == -1
    assert lib.mol_lora_expand(None, P(16), 1, 8, 16, 1.0, None, P(16), P(16), P(16), 64, 16, 8, 4, P(16), 16, 0, None, None, None) == -1
    assert lib.mol_lora_expand(None, P(16), 1, 12, 16, 1.0, None, P(16), P(16), P(16), 64, 16, 8, 4, P(16), 16, 0, None, None, None) == -3
    assert lib.mol_debug_wait_test(2, 0) == -1
    assert lib.mol_lora_shrink(P(18), 64, 1, 64, P(16), 1, 16, P(16), P(16), P(16), 64, 16, 8, 4, P(16), 0, None, None) == -3
    assert lib.mol_lora_shrink(P(16), 64, 0, 64, P(16), 1, 16, P(16), P(16), P(16), 64, 16, 8, 4, P(16), 0, None, None) == -1
    assert lib.mol_lora_shrink(P(16), 64, 1, 64, P(16), 1, 16, P(16), P(16), P(16), 65, 16, 8, 4, P(16), 0, None, None) == -1
    assert lib.mol_lora_expand(P(16), P(16), 1, 24, 16, 1.0, None, P(16), P(16), P(16), 64, 16, 8, 4, P(16), 16, 0, None, None, None) == -3
    assert lib.mol_lora_expand(P(16), P(16), 1, 16, 12, 1.0, None, P(16), P(16), P(16), 64, 16, 8, 4, P(16), 16, 0, None, None, None) == -3
    assert lib.mol_lora_expand(P(16), P(16), 2, 16, 64, 1.0, None, P(16), P(16), P(16), 64, 16, 8, 4, P(16), 64, 0, None, None, None) == -1
    assert lib.mol_lora_expand(P(16), P(16), 1, 16, 64, 1.0, None, P(16), P(16), P(16), 64, 16, 8, 4, P(24), 64, 0, None, None, None) == -3
    # per-adapter ranks / scalings: num_experts missing or not dividing V, too many adapters
    assert lib.mol_lora_shrink(P(16), 64, 1, 64, P(16), 1, 16, P(16), P(16), P(16), 64, 16, 8, 4, P(16), 0, P(16), None) == -1
    assert lib.mol_lora_shrink(P(16), 64, 1, 64, P(16), 1, 16, P(16), P(16), P(16), 64, 16, 8, 6, P(16), 4, P(16), None) == -1
    assert lib.mol_lora_shrink(P(16), 64, 1, 64, P(16), 1, 16, P(16), P(16), P(16), 64, 16, 8, 4100, P(16), 2, P(16), None) == -3
    assert lib.mol_lora_expand(P(16), P(16), 1, 16, 16, 1.0, None, P(16), P(16), P(16), 64, 16, 8, 4, P(16), 16, 3, None, P(16), None) == -1
    # per-token adapter ids
    assert lib.mol_token_lora_ids(P(16), P(16), -1, 8, 4, None, P(16), None) == -1
    assert lib.mol_token_lora_ids(P(16), P(16), 2, 8, 0, None, P(16), None) == -1
    assert lib.mol_token_lora_ids(P(16), P(16), 2, (1 << 22) + 1, 4, None, P(16), None) == -3
    assert lib.mol_token_lora_ids(None, P(16), 2, 8, 4, None, P(16), None) == -1
    assert lib.mol_token_lora_ids(P(16), P(16), 2, 8, 4, None, None, None) == -1
    assert lib.mol_token_lora_ids(None, None, 0, 0, 4, None, None, None) == 0
    # remap
    assert lib.mol_virtual_topk(P(16), P(16), -1, 8, 4, 4, P(16), None) == -1
    assert lib.mol_virtual_topk(P(16), P(16), 1 << 20, 8, 4, 4, P(16), None) == -3
    # forward: V + 1 over the bucket cap
    assert lib.mol_lora_forward(P(16), 64, 1, 64, P(16), P(16), 4, 2, 4096, 2, P(16), P(16), 1, 16, 16,
                                1.0, None, P(16), 16, 16, 1, P(16), P(16), 4096, P(16), P(16), P(16),
                                None, None, None, 0, None) == -3
    # forward: compute_routing outside {0, 1, 2}
    for mode in (-1, 3):
        assert lib.mol_lora_forward(P(16), 64, 1, 64, P(16), P(16), 4, 2, 8, 2, P(16), P(16), 1, 16,
                                    16, 1.0, None, P(16), 16, 16, mode, P(16), P(16), 4096, P(16),
                                    P(16), P(16), None, None, None, 0, None) == -1


def test_binding_fails_loudly_without_library(tmp_path):
    import moe_lora_virtual_gb300 as m

    saved = m._lib
    try:
        m._lib = None
        with pytest.raises(RuntimeError, match="not built"):
            m.library(str(tmp_path / "missing.so"))
    finally:
        m._lib = saved


def test_row_stride_of_binding_tensors(mol):
    """The binding's row stride: a 2-D tensor with unit column stride gives its row stride; a
    tensor with no elements (an empty batch, whose strides may be 0) is accepted; others are
    rejected before any call."""
    import torch

    x = torch.zeros(6, 40)[:, :32]
    assert mol._row_stride(x, "x") == 40
    empty = torch.from_numpy(np.zeros((0, 40), np.float32))[:, :32]  # strides (0, 0)
    assert mol._row_stride(empty, "x") == 32
    with pytest.raises(ValueError):
        mol._row_stride(torch.zeros(6, 40)[:, ::2], "x")
    with pytest.raises(ValueError):
        mol._row_stride(torch.zeros(6), "x")
