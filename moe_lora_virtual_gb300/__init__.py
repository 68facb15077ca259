"""Python binding of the MoL ("virtual experts") LoRA library for GB300.

Argument marshalling only: every step runs in the CUDA kernels of
``libmol.so`` through its C ABI (``include/mol.h``). PyTorch supplies device
memory and the current stream. The functions keep the C names; each raises
``MolError`` on a non-zero status. There is no CPU fallback: if the library
is missing, the first call raises.
"""

from __future__ import annotations

import contextlib
import ctypes
import os
from typing import NamedTuple, Optional

import torch

from .build import CHECKED_LIB_PATH, LIB_PATH

MOL_OK = 0
MOL_ERR_INVALID_ARG = -1
MOL_ERR_CAPACITY = -2
MOL_ERR_UNSUPPORTED = -3
MOL_ERR_CUDA = -4
MOL_MAX_BUCKETS = 8192
MOL_MAX_NUMEL = 1 << 22

EXPORTS = (
    "mol_version", "mol_status_string", "mol_last_cuda_error", "mol_align_capacity",
    "mol_workspace_bytes", "mol_virtual_topk", "mol_align_block_size", "mol_lora_shrink",
    "mol_lora_expand", "mol_lora_forward", "mol_align_block_size_noalloc", "mol_token_lora_ids",
    "mol_take_fault_flags", "mol_debug_wait_test", "mol_launch_count", "mol_checked_build",
    "mol_take_check_record",
)

# Check sites of the checked build (include/mol.h, MOL_CHECK_*).
CHECK_SITES = {
    1: "ROUTE_EXPERT", 2: "ROUTE_PAIR", 3: "ROUTE_NTPP", 4: "ALIGN_SLOT", 5: "ALIGN_BLOCK",
    6: "ALIGN_TOTAL", 7: "ALIGN_WORKSPACE", 8: "ROW", 9: "COLUMN", 10: "SMEM", 11: "TMA_COORD",
    12: "WEIGHT_ROW",
}

_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F32 = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGS = {
    "mol_version": (_I32, []),
    "mol_status_string": (ctypes.c_char_p, [_I32]),
    "mol_last_cuda_error": (_I32, []),
    "mol_launch_count": (_I64, []),
    "mol_align_capacity": (_I64, [_I64, _I32, _I32]),
    "mol_workspace_bytes": (_SZ, [_I64, _I32, _I32]),
    "mol_virtual_topk": (_I32, [_P, _P, _I64, _I32, _I32, _I32, _P, _P]),
    "mol_align_block_size": (_I32, [_P, _I64, _I32, _I32, _P, _I64, _P, _P, _P, _SZ, _P]),
    "mol_align_block_size_noalloc": (_I32, [_P, _I64, _I32, _I32, _P, _I64, _P, _P, _P]),
    "mol_lora_shrink": (_I32, [_P, _I64, _I32, _I32, _P, _I32, _I32, _P, _P, _P, _I64, _I32, _I64,
                               _I32, _P, _I32, _P, _P]),
    "mol_lora_expand": (_I32, [_P, _P, _I32, _I32, _I32, _F32, _P, _P, _P, _P, _I64, _I32, _I64,
                               _I32, _P, _I64, _I32, _P, _P, _P]),
    "mol_lora_forward": (_I32, [_P, _I64, _I32, _I32, _P, _P, _I64, _I32, _I32, _I32, _P, _P, _I32,
                                _I32, _I32, _F32, _P, _P, _I64, _I32, _I32, _P, _P, _I64, _P, _P,
                                _P, _P, _P, _P, _SZ, _P]),
    "mol_token_lora_ids": (_I32, [_P, _P, _I32, _I64, _I32, _P, _P, _P]),
    "mol_take_fault_flags": (_I32, [ctypes.POINTER(ctypes.c_uint32)]),
    "mol_debug_wait_test": (_I32, [ctypes.c_uint32, ctypes.c_uint64]),
    "mol_checked_build": (_I32, []),
    "mol_take_check_record": (_I32, [ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]),
}


class MolError(RuntimeError):
    def __init__(self, fn: str, status: int):
        lib = library()
        msg = lib.mol_status_string(status).decode()
        cuda = lib.mol_last_cuda_error() if status == MOL_ERR_CUDA else 0
        super().__init__(f"{fn}: status {status} ({msg})" + (f", cudaError {cuda}" if cuda else ""))
        self.status = status
        self.cuda_error = cuda


_loaded = {}


def _load(p: str) -> ctypes.CDLL:
    if p not in _loaded:
        if not os.path.exists(p):
            raise RuntimeError(f"MoL CUDA library not built ({p} missing): run "
                               "moe_lora_virtual_gb300.build.build_library() first")
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _loaded[p] = lib
    return _loaded[p]


def library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libmol.so once and declare every export's signature."""
    global _lib
    if _lib is None:
        _lib = _load(path or LIB_PATH)
    return _lib


@contextlib.contextmanager
def use_library(path: str):
    """Route every call of this module through the library at `path` (for instance the
    checked build, CHECKED_LIB_PATH) inside the block; the previous one is restored after.
    Both libraries keep their own device state; do not mix their routing buffers' users
    across a stream without a synchronisation."""
    global _lib
    prev = _lib
    _lib = _load(path)
    try:
        yield _lib
    finally:
        _lib = prev


def _check(fn: str, status: int) -> None:
    if status != MOL_OK:
        raise MolError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: torch.Tensor, dtype: torch.dtype, name: str) -> None:
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA tensor")


def _row_stride(t: torch.Tensor, name: str) -> int:
    if t.dim() != 2:
        raise ValueError(f"{name}: expected a 2-D tensor with unit column stride")
    if t.numel() == 0:  # no elements: its strides mean nothing (an empty array's may be 0)
        return max(int(t.shape[1]), 1)
    if t.stride(1) != 1:
        raise ValueError(f"{name}: expected a 2-D tensor with unit column stride")
    return t.stride(0)


def align_capacity(numel: int, num_vexperts: int, block_m: int) -> int:
    return int(library().mol_align_capacity(numel, num_vexperts, block_m))


def workspace_bytes(numel: int, num_vexperts: int, block_m: int) -> int:
    return int(library().mol_workspace_bytes(numel, num_vexperts, block_m))


class Routing(NamedTuple):
    vtopk_ids: torch.Tensor            # int32 [numel]
    sorted_token_ids: torch.Tensor     # int32 [capacity]
    expert_ids: torch.Tensor           # int32 [capacity // block_m]
    num_tokens_post_padded: torch.Tensor  # int32 [1]
    block_m: int
    numel: int
    num_vexperts: int

    @property
    def capacity(self) -> int:
        return self.sorted_token_ids.numel()


def alloc_routing(numel: int, num_vexperts: int, block_m: int, device) -> Routing:
    cap = align_capacity(numel, num_vexperts, block_m)
    i32 = dict(dtype=torch.int32, device=device)
    return Routing(torch.empty(numel, **i32), torch.empty(cap, **i32),
                   torch.empty(cap // block_m, **i32), torch.empty(1, **i32),
                   block_m, numel, num_vexperts)


def alloc_workspace(numel: int, num_vexperts: int, block_m: int, device) -> Optional[torch.Tensor]:
    n = workspace_bytes(numel, num_vexperts, block_m)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def mol_virtual_topk(topk_ids: torch.Tensor, lora_ids: torch.Tensor, num_experts: int,
                     max_loras: int, vtopk_ids: Optional[torch.Tensor] = None, stream=None):
    _need(topk_ids, torch.int32, "topk_ids")
    _need(lora_ids, torch.int32, "lora_ids")
    T, k = topk_ids.shape
    if vtopk_ids is None:
        vtopk_ids = torch.empty_like(topk_ids)
    _check("mol_virtual_topk", library().mol_virtual_topk(
        _ptr(topk_ids.contiguous()), _ptr(lora_ids.contiguous()), T, k, num_experts, max_loras,
        _ptr(vtopk_ids), _stream(stream)))
    return vtopk_ids


def mol_align_block_size(vtopk_ids: torch.Tensor, num_vexperts: int, block_m: int,
                         routing: Optional[Routing] = None,
                         workspace: Optional[torch.Tensor] = None, stream=None) -> Routing:
    _need(vtopk_ids, torch.int32, "vtopk_ids")
    v = vtopk_ids.reshape(-1)
    numel = v.numel()
    if routing is None:
        routing = alloc_routing(numel, num_vexperts, block_m, v.device)
        routing = routing._replace(vtopk_ids=v)
    if workspace is None:
        workspace = alloc_workspace(numel, num_vexperts, block_m, v.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("mol_align_block_size", library().mol_align_block_size(
        _ptr(v), numel, num_vexperts, block_m, _ptr(routing.sorted_token_ids), routing.capacity,
        _ptr(routing.expert_ids), _ptr(routing.num_tokens_post_padded), _ptr(workspace), wsb,
        _stream(stream)))
    return routing


def mol_align_block_size_noalloc(vtopk_ids: torch.Tensor, num_vexperts: int, block_m: int,
                                 routing: Optional[Routing] = None, stream=None) -> Routing:
    """mol_align_block_size with the library's own 1 MiB scratch instead of a workspace.

    For callers that cannot allocate device memory at routing time; calls that
    overlap on the GPU share the scratch and must be serialised by the caller.
    """
    _need(vtopk_ids, torch.int32, "vtopk_ids")
    v = vtopk_ids.reshape(-1)
    numel = v.numel()
    if routing is None:
        routing = alloc_routing(numel, num_vexperts, block_m, v.device)._replace(vtopk_ids=v)
    _check("mol_align_block_size_noalloc", library().mol_align_block_size_noalloc(
        _ptr(v), numel, num_vexperts, block_m, _ptr(routing.sorted_token_ids), routing.capacity,
        _ptr(routing.expert_ids), _ptr(routing.num_tokens_post_padded), _stream(stream)))
    return routing


def _adapter_arrays(lora_ranks, lora_scalings):
    if lora_ranks is not None:
        _need(lora_ranks, torch.int32, "lora_ranks")
    if lora_scalings is not None:
        _need(lora_scalings, torch.float32, "lora_scalings")


def mol_lora_shrink(x: torch.Tensor, x_row_div: int, lora_a: torch.Tensor, num_slices: int,
                    routing: Routing, inter: Optional[torch.Tensor] = None, stream=None,
                    lora_ranks: Optional[torch.Tensor] = None, num_experts: int = 0):
    _need(x, torch.bfloat16, "x")
    _adapter_arrays(lora_ranks, None)
    _need(lora_a, torch.bfloat16, "lora_a")
    V, R, K = lora_a.shape
    if inter is None:
        inter = torch.empty(routing.numel, R, dtype=torch.float32, device=x.device)
    _need(inter, torch.float32, "inter")
    _check("mol_lora_shrink", library().mol_lora_shrink(
        _ptr(x), _row_stride(x, "x"), x_row_div, K, _ptr(lora_a), num_slices, R // num_slices,
        _ptr(routing.sorted_token_ids), _ptr(routing.expert_ids),
        _ptr(routing.num_tokens_post_padded), routing.capacity, routing.block_m, routing.numel,
        routing.num_vexperts, _ptr(inter), num_experts, _ptr(lora_ranks), _stream(stream)))
    return inter


def mol_lora_expand(inter: torch.Tensor, lora_b: torch.Tensor, num_slices: int, scale: float,
                    routing: Routing, out: torch.Tensor,
                    topk_weights: Optional[torch.Tensor] = None, stream=None,
                    lora_ranks: Optional[torch.Tensor] = None,
                    lora_scalings: Optional[torch.Tensor] = None, num_experts: int = 0):
    _need(inter, torch.float32, "inter")
    _adapter_arrays(lora_ranks, lora_scalings)
    _need(lora_b, torch.bfloat16, "lora_b")
    _need(out, torch.bfloat16, "out")
    if topk_weights is not None:
        _need(topk_weights, torch.float32, "topk_weights")
    V, N, r = lora_b.shape
    _check("mol_lora_expand", library().mol_lora_expand(
        _ptr(inter), _ptr(lora_b), num_slices, r, N // num_slices, float(scale), _ptr(topk_weights),
        _ptr(routing.sorted_token_ids), _ptr(routing.expert_ids),
        _ptr(routing.num_tokens_post_padded), routing.capacity, routing.block_m, routing.numel,
        routing.num_vexperts, _ptr(out), _row_stride(out, "out"), num_experts, _ptr(lora_ranks),
        _ptr(lora_scalings), _stream(stream)))
    return out


def mol_lora_forward(x: torch.Tensor, x_row_div: int, topk_ids: Optional[torch.Tensor],
                     lora_ids: Optional[torch.Tensor], num_experts: int, max_loras: int,
                     lora_a: torch.Tensor, lora_b: torch.Tensor, num_slices: int, scale: float,
                     out: torch.Tensor, routing: Routing, inter: torch.Tensor,
                     compute_routing: int = True, topk_weights: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, num_tokens: Optional[int] = None,
                     topk: Optional[int] = None, stream=None,
                     lora_ranks: Optional[torch.Tensor] = None,
                     lora_scalings: Optional[torch.Tensor] = None) -> None:
    """One MoL LoRA stage; with compute_routing the routing buffers are (re)computed.

    compute_routing: False/0 reuses the routing; True/1 computes it; 2 computes it and
    declares that topk_ids and lora_ids were complete before the kernel preceding the call
    began, so the stage may start reading them (and the weights they select) early."""
    _need(x, torch.bfloat16, "x")
    _adapter_arrays(lora_ranks, lora_scalings)
    if topk_ids is not None:
        _need(topk_ids, torch.int32, "topk_ids")
        num_tokens, topk = topk_ids.shape
    if lora_ids is not None:
        _need(lora_ids, torch.int32, "lora_ids")
    V, R, K = lora_a.shape
    _, N, r = lora_b.shape
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("mol_lora_forward", library().mol_lora_forward(
        _ptr(x), _row_stride(x, "x"), x_row_div, K, _ptr(topk_ids), _ptr(lora_ids), num_tokens,
        topk, num_experts, max_loras, _ptr(lora_a), _ptr(lora_b), num_slices, r,
        N // num_slices, float(scale), _ptr(topk_weights), _ptr(out), _row_stride(out, "out"),
        routing.block_m, int(compute_routing), _ptr(routing.vtopk_ids),
        _ptr(routing.sorted_token_ids), routing.capacity, _ptr(routing.expert_ids),
        _ptr(routing.num_tokens_post_padded), _ptr(inter), _ptr(lora_ranks), _ptr(lora_scalings),
        _ptr(workspace), wsb, _stream(stream)))


def mol_token_lora_ids(weight_indices: torch.Tensor, seg_indptr: torch.Tensor, num_tokens: int,
                       max_loras: int, lora_ranks: Optional[torch.Tensor] = None,
                       lora_ids: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Per-token adapter ids from per-request slots (-1 = no adapter)."""
    _need(weight_indices, torch.int32, "weight_indices")
    _need(seg_indptr, torch.int32, "seg_indptr")
    _adapter_arrays(lora_ranks, None)
    num_reqs = weight_indices.numel()
    if seg_indptr.numel() != num_reqs + 1:
        raise ValueError("seg_indptr: expected num_reqs + 1 entries")
    if lora_ids is None:
        lora_ids = torch.empty(num_tokens, dtype=torch.int32, device=weight_indices.device)
    _need(lora_ids, torch.int32, "lora_ids")
    _check("mol_token_lora_ids", library().mol_token_lora_ids(
        _ptr(weight_indices), _ptr(seg_indptr), num_reqs, num_tokens, max_loras, _ptr(lora_ranks),
        _ptr(lora_ids), _stream(stream)))
    return lora_ids


def mol_take_fault_flags() -> int:
    """Bits recorded by kernels whose bounded waits ran out since the last call (0 = none);
    synchronizes the device and clears them."""
    v = ctypes.c_uint32(0)
    _check("mol_take_fault_flags", library().mol_take_fault_flags(ctypes.byref(v)))
    return int(v.value)


def mol_debug_wait_test(stall_producer: bool, wait_limit_ns: int = 0) -> None:
    """Test hook of the bounded waits: with stall_producer the shrink's producer warps issue
    nothing, so its consumers' waits run out (after wait_limit_ns; 0 = one second) and record
    a fault bit. Synchronizes the device."""
    _check("mol_debug_wait_test", library().mol_debug_wait_test(int(bool(stall_producer)),
                                                                int(wait_limit_ns)))


def mol_launch_count() -> int:
    """Kernels the library has enqueued in this process so far."""
    return int(library().mol_launch_count())


def mol_checked_build() -> bool:
    """True when the loaded library is the checked build."""
    return bool(library().mol_checked_build())


class CheckRecord(NamedTuple):
    count: int   # failed checks since the last read (0 in the release build)
    site: int    # MOL_CHECK_* of the first one recorded, 0 if none
    value: int   # the index or value it recorded

    @property
    def site_name(self) -> str:
        return CHECK_SITES.get(self.site, "none" if self.site == 0 else f"site {self.site}")


def mol_take_check_record() -> CheckRecord:
    """Reads and clears the checked build's record of failed device-side checks;
    synchronizes the device."""
    first, count = ctypes.c_uint64(0), ctypes.c_uint64(0)
    _check("mol_take_check_record",
           library().mol_take_check_record(ctypes.byref(first), ctypes.byref(count)))
    return decode_check_record(int(first.value), int(count.value))


def decode_check_record(first: int, count: int) -> CheckRecord:
    """(site << 48) | (value & 0xFFFFFFFFFFFF), with the value sign-extended from 48 bits."""
    value = first & 0xFFFFFFFFFFFF
    if value >= 1 << 47:
        value -= 1 << 48
    return CheckRecord(count, first >> 48, value)
