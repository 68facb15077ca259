"""Helpers for the GPU parity tests: upload inputs, run the library, compare with the oracle."""

from __future__ import annotations

import numpy as np
import pytest

import oracle

# |gpu - ref| <= 1e-3 * (|ref| + max(rms(ref row), rms(ref, every checked row))) on fp32
# intermediates: 1e-3 relative to the scale of the intermediate, not of an element or row that
# cancellation (or an adapter rank of one or two columns) has made small
INTER_RTOL = 1e-3
OUT_RTOL = 1e-2     # |gpu - ref| <= 1e-2 * (1 + |ref|) on bf16 outputs


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def mol_lib():
    from moe_lora_virtual_gb300.build import build_library

    build_library()
    import moe_lora_virtual_gb300 as mol

    mol.library()
    return mol


def to_dev_bf16(a: np.ndarray, dev):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def to_dev_i32(a: np.ndarray, dev):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def bf16_host(t) -> np.ndarray:
    import torch

    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def check_inter(gpu: np.ndarray, ref: np.ndarray, rows) -> None:
    rows = np.asarray(rows, dtype=np.int64)
    if rows.size == 0:
        return
    g = gpu[rows].astype(np.float64)
    r = ref[rows].astype(np.float64)
    assert np.all(np.isfinite(g)), "non-finite intermediate on a valid row"
    rms = np.sqrt(np.mean(r * r, axis=1, keepdims=True))
    rms_all = np.sqrt(np.mean(r * r))
    err = np.abs(g - r)
    bound = INTER_RTOL * (np.abs(r) + np.maximum(rms, rms_all))
    bad = err > bound
    assert not bad.any(), f"inter mismatch at {np.argwhere(bad)[:5].tolist()}, max err {err.max():.3e}"


def check_out(gpu_bits: np.ndarray, ref_bits: np.ndarray, rows) -> None:
    rows = np.asarray(rows, dtype=np.int64)
    if rows.size == 0:
        return
    g = oracle.bf16_to_f64(gpu_bits[rows])
    r = oracle.bf16_to_f64(ref_bits[rows])
    assert np.all(np.isfinite(g))
    err = np.abs(g - r)
    bad = err > OUT_RTOL * (1 + np.abs(r))
    assert not bad.any(), f"out mismatch at {np.argwhere(bad)[:5].tolist()}, max err {err.max():.3e}"


def valid_pairs(sorted_ids, expert_ids, ntpp, block_m, numel, blocks=None) -> np.ndarray:
    """Flat pair ids that the consuming stages process (optionally only in `blocks`)."""
    out = []
    rng = range(ntpp // block_m) if blocks is None else blocks
    for t in rng:
        if expert_ids[t] < 0:
            continue
        ids = sorted_ids[t * block_m:(t + 1) * block_m]
        out.append(ids[(ids >= 0) & (ids < numel)])
    return np.concatenate(out) if out else np.zeros(0, np.int64)
