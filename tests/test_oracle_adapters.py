"""Pins of the oracle's adapter handling: per-adapter rank and scaling, and the
per-request -> per-token adapter ids (the step before the remap)."""

import json
import os

import numpy as np
import pytest

from oracle import (align_block_size, bf16_to_f64, brute_force_stage, f64_to_bf16, lora_expand,
                    lora_forward_stage, lora_shrink, token_lora_ids, virtual_topk)
from synth import WORKLOADS, make_layer

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def bits(a):
    return f64_to_bf16(np.asarray(a, np.float64))


# ------------------------------------------------------------ per-token adapter ids

def test_worked_token_ids():
    g = GOLDEN["token_lora_ids_guard"]
    got = token_lora_ids(g["weight_indices"], g["seg_indptr"], g["num_tokens"], g["max_loras"])
    assert got.tolist() == g["expected_no_ranks"]
    got = token_lora_ids(g["weight_indices"], g["seg_indptr"], g["num_tokens"], g["max_loras"],
                         g["lora_ranks"])
    assert got.tolist() == g["expected_with_ranks"]


def _per_token(wi, seg, num_tokens, max_loras, ranks):
    """Token by token: the first request whose segment holds the token, then the guard."""
    out = []
    for t in range(num_tokens):
        val = -1
        for q in range(len(wi)):
            if seg[q] <= t < seg[q + 1]:
                w = wi[q]
                ok = 0 <= w < max_loras and (ranks is None or ranks[w] > 0)
                val = w if ok else -1
                break
        out.append(val)
    return out


@pytest.mark.parametrize("seed", range(6))
def test_token_ids_against_per_token_scan(seed):
    rng = np.random.default_rng(seed)
    nreq = int(rng.integers(0, 12))
    lens = rng.integers(0, 7, nreq)
    seg = np.concatenate([[0], np.cumsum(lens)]).astype(int).tolist()
    num_tokens = seg[-1] + int(rng.integers(0, 3))
    L = int(rng.integers(1, 6))
    wi = rng.integers(-2, L + 2, nreq).tolist()
    ranks = rng.choice([0, 8, 16], L).tolist() if seed % 2 else None
    got = token_lora_ids(wi, seg, num_tokens, L, ranks)
    assert got.tolist() == _per_token(wi, seg, num_tokens, L, ranks)


def test_token_ids_negative_index_never_reads_ranks():
    # -1 must not wrap to the last slot: the last slot has a positive rank here
    got = token_lora_ids([-1, 1], [0, 2, 3], 3, 2, [0, 16])
    assert got.tolist() == [-1, -1, 1]


def test_token_ids_empty():
    assert token_lora_ids([], [0], 0, 4).tolist() == []
    assert token_lora_ids([], [0], 3, 4).tolist() == [-1, -1, -1]


# ------------------------------------------------------------ per-adapter rank and scaling

def test_worked_rank_limited():
    g = GOLDEN["rank_limited_adapter"]
    sorted_ids, expert_ids, ntpp = np.array([0], np.int32), np.array([0], np.int32), 1
    x, A, B = bits(g["x"]), bits(g["lora_a"])[None], bits(g["lora_b"])[None]
    inter0 = np.full((1, 2), np.nan, np.float32)
    inter = lora_shrink(x, 1, A, sorted_ids, expert_ids, ntpp, 1, 1, inter0, 1, 1, [g["rank"]])
    assert inter[0].tolist() == g["inter"]
    out = lora_expand(inter, B, 1, 2, 1, g["scale"], None, sorted_ids, expert_ids, ntpp, 1, 1,
                      bits([g["out0"]]), num_experts=1, lora_ranks=[g["rank"]],
                      lora_scalings=[g["scaling"]])
    assert out[0].tolist() == g["out_bits"]
    inter = lora_shrink(x, 1, A, sorted_ids, expert_ids, ntpp, 1, 1, inter0, 1, 1, [0])
    assert np.all(np.isnan(inter))
    out = lora_expand(inter0, B, 1, 2, 1, g["scale"], None, sorted_ids, expert_ids, ntpp, 1, 1,
                      bits([g["out0"]]), num_experts=1, lora_ranks=[0])
    assert out[0].tolist() == g["rank0_out_bits"]


def _stage(name, seed):
    wl = WORKLOADS[name]
    li = make_layer(wl, seed)
    st = li.stages[0]
    vt = virtual_topk(li.topk_ids, li.lora_ids, wl.E, wl.L).reshape(-1)
    s, e, n = align_block_size(vt, wl.V, wl.BM)
    return wl, li, st, (vt, s, e, n)


def _run(wl, li, st, routing, ranks=None, scalings=None, A=None, B=None, scale=None):
    A = st.A.host_all() if A is None else A
    B = st.B.host_all() if B is None else B
    return lora_forward_stage(st.x.host_all(), st.x_row_div, li.topk_ids, li.lora_ids, wl.E, wl.L,
                              A, B, st.stage.S, st.stage.r, st.stage.Ns,
                              wl.scale if scale is None else scale, None, st.out0.host_all(),
                              wl.BM, routing=routing, lora_ranks=ranks, lora_scalings=scalings)


@pytest.mark.parametrize("seed", [0, 1])
def test_full_ranks_and_unit_scalings_change_nothing(seed):
    wl, li, st, routing = _stage("tiny", seed)
    plain = _run(wl, li, st, routing)
    full = _run(wl, li, st, routing, ranks=[st.stage.r] * wl.L, scalings=[1.0] * wl.L)
    assert np.array_equal(plain["inter"], full["inter"], equal_nan=True)
    assert np.array_equal(plain["out"], full["out"])


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_rank_equals_zero_padded_weights(seed):
    """An adapter of rank r_l gives the same result as full rank with its weights zeroed past r_l."""
    wl, li, st, routing = _stage("tiny", seed)
    rng = np.random.default_rng(100 + seed)
    r, S = st.stage.r, st.stage.S
    ranks = rng.integers(1, r + 1, wl.L).tolist()
    A, B = st.A.host_all().copy(), st.B.host_all().copy()
    for v in range(wl.V):
        rl = ranks[v // wl.E]
        for s in range(S):
            A[v, s * r + rl:(s + 1) * r, :] = 0
        B[v, :, rl:] = 0
    ranked = _run(wl, li, st, routing, ranks=ranks)
    padded = _run(wl, li, st, routing, A=A, B=B)
    assert np.array_equal(ranked["inter"], padded["inter"], equal_nan=True)  # -0 == +0
    assert np.array_equal(ranked["out"], padded["out"])


@pytest.mark.parametrize("seed", [0, 1])
def test_weights_past_rank_take_no_part(seed):
    """Weight rows of lora_a and columns of lora_b past an adapter's rank are padding: NaN
    there changes nothing (the sums run over j < r_l only)."""
    wl, li, st, routing = _stage("tiny", seed)
    rng = np.random.default_rng(200 + seed)
    r, S = st.stage.r, st.stage.S
    ranks = [0, int(rng.integers(1, r))]
    A, B = st.A.host_all().copy(), st.B.host_all().copy()
    nan_bits = np.uint16(0x7FC0)
    for v in range(wl.V):
        rl = ranks[v // wl.E]
        for s in range(S):
            A[v, s * r + rl:(s + 1) * r, :] = nan_bits
        B[v, :, rl:] = nan_bits
    clean = _run(wl, li, st, routing, ranks=ranks)
    poisoned = _run(wl, li, st, routing, ranks=ranks, A=A, B=B)
    assert np.array_equal(clean["inter"], poisoned["inter"], equal_nan=True)
    assert np.array_equal(clean["out"], poisoned["out"])
    vt = routing[0]
    live = vt >= wl.E  # adapter 1, rank >= 1
    assert live.any() and not np.any(np.isnan(poisoned["inter"][live]))


def test_rank_zero_writes_nothing():
    wl, li, st, routing = _stage("tiny", 0)
    res = _run(wl, li, st, routing, ranks=[0, st.stage.r])
    vt = routing[0]
    adapter0 = (vt >= 0) & (vt < wl.E)              # virtual experts of adapter 0
    assert np.all(np.isnan(res["inter"][adapter0]))
    assert np.array_equal(res["out"][adapter0], st.out0.host_all()[adapter0])
    other = (vt >= wl.E)
    assert other.any() and not np.any(np.isnan(res["inter"][other]))


def test_scaling_multiplies_the_delta():
    wl, li, st, routing = _stage("tiny", 1)
    both = _run(wl, li, st, routing, scalings=[3.0, 3.0])
    tripled = _run(wl, li, st, routing, scale=3.0 * wl.scale)
    assert np.array_equal(both["out"], tripled["out"])
    one = _run(wl, li, st, routing, scalings=[1.0, 3.0])
    vt = routing[0]
    a0, a1 = (vt >= 0) & (vt < wl.E), vt >= wl.E
    plain = _run(wl, li, st, routing)
    assert np.array_equal(one["out"][a0], plain["out"][a0])
    assert np.array_equal(one["out"][a1], tripled["out"][a1])


@pytest.mark.parametrize("seed", [0, 1])
def test_brute_force_with_ranks_and_scalings(seed):
    wl, li, st, routing = _stage("tiny", seed)
    rng = np.random.default_rng(7 + seed)
    ranks = [int(rng.integers(0, st.stage.r + 1)), int(rng.integers(1, st.stage.r + 1))]
    scalings = rng.uniform(0.25, 2.0, wl.L).astype(np.float32).tolist()
    res = _run(wl, li, st, routing, ranks=ranks, scalings=scalings)
    inters, out_bf = brute_force_stage(li.topk_ids, li.lora_ids, wl.E, wl.L, st.x.host_all(),
                                       st.x_row_div, st.A.host_all(), st.B.host_all(), st.stage.S,
                                       st.stage.r, st.stage.Ns, wl.scale, None, st.out0.host_all(),
                                       lora_ranks=ranks, lora_scalings=scalings)
    for pair, h in inters.items():
        assert np.array_equal(res["inter"][pair], np.array(h, np.float32))
    assert np.array_equal(res["out"], out_bf)
