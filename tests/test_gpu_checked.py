"""The checked build (libmol_checked.so): device-side index checks on every kernel.

Every kernel of the path checks its computed indices against their buffers
before it uses them (align slots and block entries against capacity, rows
against numel, columns against the row, shared-memory extents, tensor-copy
coordinates, weight rows against the adapter tensor) and records a failure
instead of touching memory. These tests run the checked build

- on the workloads and on shapes that reach every kernel variant (single-block,
  cluster and multi-tile align; item shrink with and without adapter ranks;
  tcgen05 shrink; register, staged, two-tile and tcgen05 expands; the fused
  stage) and
  on adversarial routings of the align, and assert that no check failed and
  that the results still match the oracle;
- on routing data passed in by the caller with entries that every build skips
  (an expert id past V, slots outside [0, numel], a post-padded count past
  capacity), and assert that the checked build records exactly those while the
  results match the oracle on the same routing.
"""

import numpy as np
import pytest

import oracle
from synth import WORKLOADS, make_layer
from tests.gpu_util import (bf16_host, check_inter, check_out, mol_lib, to_dev_bf16, to_dev_i32,
                            torch_cuda, valid_pairs)
from tests.test_gpu_parity import check_routing, run_layer_gpu

pytestmark = pytest.mark.gpu


def bits(a):
    return oracle.f64_to_bf16(np.asarray(a, np.float64))


@pytest.fixture(scope="module")
def checked():
    torch_cuda()
    mol = mol_lib()
    from moe_lora_virtual_gb300.build import build_library

    path = build_library(checked=True)
    with mol.use_library(path):
        assert mol.mol_checked_build()
        mol.mol_take_check_record()  # start from a clear record
        yield mol
    assert not mol.mol_checked_build()


def assert_clean(mol):
    rec = mol.mol_take_check_record()
    assert rec.count == 0, f"{rec.count} failed checks, first {rec.site_name} value {rec.value}"
    assert mol.mol_take_fault_flags() == 0


@pytest.mark.parametrize("name", ["tiny", "decode", "wide", "wide1k"])
def test_workload_layers_pass_every_check(checked, name):
    torch = torch_cuda()
    dev = torch.device("cuda:0")
    wl = WORKLOADS[name]
    li = make_layer(wl, 0)
    rt, res = run_layer_gpu(wl, li, dev)
    assert_clean(checked)
    s, e, n = check_routing(wl, li, rt)
    pairs = valid_pairs(s, e, n, wl.BM, wl.numel)
    for st, (g_inter, g_out) in zip(li.stages, res):
        ref_inter = oracle.lora_shrink(st.x, st.x_row_div, st.A, s, e, n, wl.BM, wl.numel,
                                       np.full((wl.numel, st.stage.R), np.nan, np.float32))
        ref_out = oracle.lora_expand(ref_inter, st.B, st.stage.S, st.stage.r, st.stage.Ns,
                                     wl.scale, None, s, e, n, wl.BM, wl.numel, st.out0.host_all())
        check_inter(g_inter, ref_inter, pairs)
        check_out(g_out, ref_out, pairs)


# T, k, E, L, BM, K, S, r, Ns, token_rows, sentinel fraction, adapter arrays; the comment names
# the kernels the shape reaches through mol_lora_forward
FORWARD_SHAPES = [
    (16, 2, 8, 2, 16, 256, 1, 16, 128, True, 0.1, False),     # fused stage (a small layer)
    (23, 8, 16, 4, 16, 2048, 2, 32, 768, True, 0.0, False),   # item shrink, staged expand
    (64, 8, 2, 2, 32, 512, 1, 128, 72, False, 0.0, False),    # register expand (rank 128)
    (300, 8, 4, 1, 128, 96, 3, 16, 2000, True, 0.3, False),   # two staged row tiles
    (256, 2, 4, 1, 64, 256, 2, 64, 96, True, 0.0, False),     # tcgen05 shrink, R = 128
    (300, 4, 8, 1, 64, 512, 1, 64, 64, False, 0.1, False),    # tcgen05 shrink, 64-row box
    (40, 8, 6, 2, 32, 4096, 2, 32, 96, True, 0.1, True),      # item shrink with ranks, k chunks
    (30, 4, 5, 2, 16, 320, 1, 8, 200, True, 0.1, True),       # rank 8 with ranks and scalings
    (700, 8, 64, 2, 16, 128, 1, 16, 64, True, 0.1, False),    # cluster align (5600 pairs)
    (256, 2, 4, 1, 64, 256, 2, 64, 384, True, 0.05, False),   # tcgen05 shrink and expand
    # 16-row shrink items, 768-column expand items in a looping grid, one-pass cluster align
    (1200, 8, 128, 4, 16, 256, 2, 16, 1536, True, 0.3, False),
    (1200, 8, 128, 4, 16, 256, 2, 16, 1536, True, 0.3, True),  # the same with adapter arrays
]


def _forward_case(mol, case, dev, routing_override=None, mode=1):
    """Random inputs of one shape; returns (gpu inter, gpu out, oracle inter, oracle out, pairs)."""
    import torch

    T, k, E, L, BM, K, S, r, Ns, token_rows, sent, adapt = case
    rng = np.random.default_rng(sum(case[:9]))
    numel, V, R, N = T * k, E * L, S * r, S * Ns
    topk = rng.integers(0, E, size=(T, k)).astype(np.int32)
    topk[rng.random((T, k)) < sent] = -1
    lora = (np.zeros(T, np.int32) if L == 1 else rng.integers(-1, L, size=T).astype(np.int32))
    xdiv = k if token_rows else 1
    x = bits(rng.standard_normal((T if token_rows else numel, K)))
    A = bits(rng.standard_normal((V, R, K)) * 0.05)
    B = bits(rng.standard_normal((V, N, r)) * 0.05)
    out0 = bits(rng.standard_normal((numel, N)))
    ranks = rng.integers(1, r + 1, size=L).astype(np.int32) if adapt else None  # every row live
    scal = rng.uniform(0.5, 2.0, size=L).astype(np.float32) if adapt else None
    vt = oracle.virtual_topk(topk, lora, E, L).reshape(-1)
    s, e, n = oracle.align_block_size(vt, V, BM)
    if routing_override is not None:
        s, e, n = routing_override(s.copy(), e.copy(), n)
    # the oracle on the routing as the kernels read it: blocks with an expert id past V and
    # blocks past the end of the buffers are skipped
    e_or, n_or = np.where(e < V, e, -1), min(n, len(s))
    kw = dict(num_experts=E, lora_ranks=ranks) if adapt else {}
    ref_inter = oracle.lora_shrink(x, xdiv, A, s, e_or, n_or, BM, numel,
                                   np.full((numel, R), np.nan, np.float32), S, **kw)
    ref_out = oracle.lora_expand(ref_inter, B, S, r, Ns, 0.5, None, s, e_or, n_or, BM, numel, out0,
                                 lora_scalings=scal, **kw)
    pairs = valid_pairs(s, e_or, n_or, BM, numel)

    xd, Ad, Bd = to_dev_bf16(x, dev), to_dev_bf16(A, dev), to_dev_bf16(B, dev)
    out = to_dev_bf16(out0, dev)
    inter = torch.full((numel, R), float("nan"), dtype=torch.float32, device=dev)
    rk_d = None if ranks is None else to_dev_i32(ranks, dev)
    sc_d = None if scal is None else torch.from_numpy(scal).to(dev)
    if routing_override is None:
        routing = mol.alloc_routing(numel, V, BM, dev)
        ws = mol.alloc_workspace(numel, V, BM, dev)
        mol.mol_lora_forward(xd, xdiv, to_dev_i32(topk, dev), to_dev_i32(lora, dev), E, L, Ad, Bd,
                             S, 0.5, out, routing, inter, workspace=ws, lora_ranks=rk_d,
                             lora_scalings=sc_d, compute_routing=mode)
    else:
        # the caller's routing: the stage runs on it as given (no align)
        routing = mol.Routing(to_dev_i32(vt, dev), to_dev_i32(s, dev), to_dev_i32(e, dev),
                              torch.tensor([n], dtype=torch.int32, device=dev), BM, numel, V)
        mol.mol_lora_forward(xd, xdiv, None, None, E, L, Ad, Bd, S, 0.5, out, routing, inter,
                             compute_routing=False, num_tokens=T, topk=k, lora_ranks=rk_d,
                             lora_scalings=sc_d)
    torch.cuda.synchronize()
    return inter.cpu().numpy(), bf16_host(out), ref_inter, ref_out, pairs, (s, e, n)


@pytest.mark.parametrize("case", FORWARD_SHAPES)
@pytest.mark.parametrize("mode", [1, 2])
def test_forward_shapes_pass_every_check(checked, case, mode):
    torch = torch_cuda()
    g_inter, g_out, ref_inter, ref_out, pairs, _ = _forward_case(checked, case, torch.device("cuda:0"),
                                                                  mode=mode)
    assert_clean(checked)
    check_inter(g_inter, ref_inter, pairs)
    check_out(g_out, ref_out, pairs)


def _align_keys(kind, numel, V, rng):
    if kind == "random":
        return rng.integers(-1, V, size=numel).astype(np.int32)
    if kind == "one_bucket":
        return np.full(numel, V - 1, np.int32)
    if kind == "all_sentinel":
        return np.full(numel, -1, np.int32)
    if kind == "past_v":  # ids >= V go to the sentinel bucket
        return rng.integers(V - 2, V + 50, size=numel).astype(np.int32)
    if kind == "one_per_bucket":  # the capacity bound is reached
        return np.resize(np.arange(V, dtype=np.int32), numel)
    raise ValueError(kind)


# numel, V, BM, kind: single block (<= 4096), one cluster (<= 131072), tiles + scan + scatter
ALIGN_CASES = [
    (4096, 257, 16, "one_per_bucket"),
    (3000, 64, 128, "one_bucket"),
    (4097, 8191, 16, "random"),
    (131072, 8191, 16, "one_per_bucket"),
    (131072, 16, 64, "one_bucket"),
    (100000, 1024, 32, "past_v"),
    (50000, 300, 16, "all_sentinel"),
    (200000, 8191, 16, "one_per_bucket"),
    (300000, 64, 128, "random"),
]


@pytest.mark.parametrize("numel,V,BM,kind", ALIGN_CASES)
def test_align_passes_every_check_on_adversarial_routing(checked, numel, V, BM, kind):
    torch = torch_cuda()
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(numel + V + BM)
    vid = _align_keys(kind, numel, V, rng)
    r = checked.mol_align_block_size(to_dev_i32(vid, dev), V, BM)
    torch.cuda.synchronize()
    assert_clean(checked)
    s, e, n = oracle.align_block_size(vid, V, BM)
    assert int(r.num_tokens_post_padded.item()) == n
    assert np.array_equal(r.sorted_token_ids.cpu().numpy(), s)
    assert np.array_equal(r.expert_ids.cpu().numpy(), e)


# ------------------------------------------------- caller routing, recorded ----

def _first_real_block(s, e, n, BM, numel):
    for t in range(n // BM):
        ids = s[t * BM:(t + 1) * BM]
        if e[t] >= 0 and np.count_nonzero((ids >= 0) & (ids < numel)) >= 2:
            return t
    raise AssertionError("no block with two pairs")


CORRUPTIONS = ["expert_past_v", "negative_slot", "slot_past_numel", "ntpp_past_capacity"]


@pytest.mark.parametrize("case", [FORWARD_SHAPES[1], FORWARD_SHAPES[2], FORWARD_SHAPES[4],
                                  FORWARD_SHAPES[0], FORWARD_SHAPES[3], FORWARD_SHAPES[9]])
@pytest.mark.parametrize("corruption", CORRUPTIONS)
def test_bad_caller_routing_is_recorded_and_skipped(checked, case, corruption):
    """Entries that every build skips are recorded by the checked build, site and value;
    the results equal the oracle's on the same routing (which skips them too)."""
    torch = torch_cuda()
    T, k, E, L, BM = case[:5]
    numel, V = T * k, E * L
    where = {}

    def corrupt(s, e, n):
        t = _first_real_block(s, e, n, BM, numel)
        if corruption == "expert_past_v":
            e[t] = V + 3
            where.update(site="ROUTE_EXPERT", value=t)
        elif corruption == "negative_slot":
            q = t * BM + int(np.flatnonzero(s[t * BM:(t + 1) * BM] < numel)[0])
            s[q] = -7
            where.update(site="ROUTE_PAIR", value=q)
        elif corruption == "slot_past_numel":
            q = t * BM + int(np.flatnonzero(s[t * BM:(t + 1) * BM] < numel)[-1])
            s[q] = numel + 5
            where.update(site="ROUTE_PAIR", value=q)
        else:  # blocks between the real count and capacity carry -1 and are skipped
            n = len(s) + BM
            where.update(site="ROUTE_NTPP", value=n)
        return s, e, n

    g_inter, g_out, ref_inter, ref_out, pairs, _ = _forward_case(checked, case, torch.device("cuda:0"),
                                                                  routing_override=corrupt)
    rec = checked.mol_take_check_record()
    assert checked.mol_take_fault_flags() == 0
    assert rec.count >= 1
    assert (rec.site_name, rec.value) == (where["site"], where["value"])
    check_inter(g_inter, ref_inter, pairs)
    check_out(g_out, ref_out, pairs)


def test_release_build_records_nothing():
    """The release library compiles the checks out: the same bad routing leaves no record."""
    torch = torch_cuda()
    mol = mol_lib()
    from moe_lora_virtual_gb300.build import LIB_PATH

    def corrupt(s, e, n):
        e[_first_real_block(s, e, n, 16, 23 * 8)] = 16 * 4 + 3
        return s, e, n

    with mol.use_library(LIB_PATH):
        assert not mol.mol_checked_build()
        g_inter, g_out, ref_inter, ref_out, pairs, _ = _forward_case(
            mol, FORWARD_SHAPES[1], torch.device("cuda:0"), routing_override=corrupt)
        rec = mol.mol_take_check_record()
        assert mol.mol_take_fault_flags() == 0
    assert (rec.count, rec.site) == (0, 0)
    check_inter(g_inter, ref_inter, pairs)
    check_out(g_out, ref_out, pairs)
