"""Pins of the oracle's LoRA shrink / expand (steps a3, a4) and their composition."""

import json
import os

import numpy as np
import pytest

from oracle import (align_block_size, bf16_to_f64, brute_force_stage, f64_to_bf16,
                    lora_expand, lora_forward_stage, lora_shrink, virtual_topk)
from synth import WORKLOADS, make_layer

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def bits(a):
    return f64_to_bf16(np.asarray(a, np.float64))


def one_block_routing(c, BM):
    sorted_ids = np.full(BM, c, np.int32)
    sorted_ids[:c] = np.arange(c)
    return sorted_ids, np.array([0], np.int32), BM


def test_worked_one_pair():
    g = GOLDEN["shrink_expand_one_pair"]
    s, e, n = one_block_routing(1, 1)
    x = bits(g["x"])
    A = bits(g["lora_a"])[None]
    B = bits(g["lora_b"])[None]
    inter = lora_shrink(x, 1, A, s, e, n, 1, 1, np.full((1, 2), np.nan, np.float32))
    assert inter[0].tolist() == g["inter"]
    out = lora_expand(inter, B, 1, 2, 2, g["scale"], None, s, e, n, 1, 1, bits([g["out0"]]))
    assert out[0].tolist() == g["out_bits"]


def test_worked_two_slices():
    g = GOLDEN["two_slices"]
    s, e, n = one_block_routing(1, 1)
    inter = np.array([g["inter"]], np.float32)
    B = bits(g["lora_b"])[None]
    out = lora_expand(inter, B, 2, 1, 1, g["scale"], None, s, e, n, 1, 1, bits([g["out0"]]))
    assert out[0].tolist() == g["out_bits"]


def _tiny_stage(seed):
    wl = WORKLOADS["tiny"]
    li = make_layer(wl, seed)
    st = li.stages[0]
    return wl, li, st


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_brute_force_tiny(seed):
    wl, li, st = _tiny_stage(seed)
    x, A, B, out0 = st.x.host_all(), st.A.host_all(), st.B.host_all(), st.out0.host_all()
    res = lora_forward_stage(x, st.x_row_div, li.topk_ids, li.lora_ids, wl.E, wl.L, A, B,
                             st.stage.S, st.stage.r, st.stage.Ns, wl.scale, None, out0, wl.BM)
    inters, out_bf = brute_force_stage(li.topk_ids, li.lora_ids, wl.E, wl.L, x, st.x_row_div,
                                       A, B, st.stage.S, st.stage.r, st.stage.Ns, wl.scale, None, out0)
    assert len(inters) > 0
    for pair, h in inters.items():
        np.testing.assert_allclose(res["inter"][pair], np.array(h, np.float32), rtol=1e-6, atol=1e-6)
    assert np.array_equal(res["out"], out_bf)
    # pairs without a delta are the remaining rows: NaN intermediates, untouched output
    no_delta = sorted(set(range(wl.numel)) - set(inters))
    assert np.all(np.isnan(res["inter"][no_delta]))
    assert np.array_equal(res["out"][no_delta], out0[no_delta])


def test_brute_force_two_slices_with_weights():
    rng = np.random.default_rng(5)
    E, L, T, k, K, r, Ns, S = 3, 2, 5, 2, 24, 4, 6, 2
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    topk[1, 0] = -1
    lora = np.array([0, 1, -1, 1, 0], np.int32)
    x = bits(rng.standard_normal((T, K)))
    A = bits(rng.standard_normal((E * L, S * r, K)) * 0.1)
    B = bits(rng.standard_normal((E * L, S * Ns, r)) * 0.1)
    out0 = bits(rng.standard_normal((T * k, S * Ns)))
    w = rng.random(T * k).astype(np.float32)
    res = lora_forward_stage(x, k, topk, lora, E, L, A, B, S, r, Ns, 0.75, w, out0, 4)
    _, out_bf = brute_force_stage(topk, lora, E, L, x, k, A, B, S, r, Ns, 0.75, w, out0)
    assert np.array_equal(res["out"], out_bf)


def _int_bits(rng, shape, lo, hi):
    return bits(rng.integers(lo, hi + 1, size=shape).astype(np.float64))


def test_small_integers_exact():
    """Integer-valued bf16 inputs: every sum is an exact integer; compare with Python ints."""
    rng = np.random.default_rng(7)
    V, R, K, N, c, BM = 3, 8, 64, 16, 5, 8
    x = _int_bits(rng, (c, K), -4, 4)
    A = _int_bits(rng, (V, R, K), -4, 4)
    B = _int_bits(rng, (V, N, R), -2, 2)
    out0 = _int_bits(rng, (c, N), -8, 8)
    sorted_ids = np.array([0, 1, 2, 5, 5, 5, 5, 5, 3, 4, 5, 5, 5, 5, 5, 5], np.int32)
    expert_ids = np.array([2, 0], np.int32)
    inter = lora_shrink(x, 1, A, sorted_ids, expert_ids, 16, BM, c, np.zeros((c, R), np.float32))
    out = lora_expand(inter, B, 1, R, N, 1.0, None, sorted_ids, expert_ids, 16, BM, c, out0)
    xi, Ai, Bi, oi = (bf16_to_f64(a).astype(np.int64) for a in (x, A, B, out0))
    for i in range(c):
        v = 2 if i < 3 else 0
        h = [sum(int(xi[i, q]) * int(Ai[v, j, q]) for q in range(K)) for j in range(R)]
        assert inter[i].tolist() == h
        for n in range(N):
            want = int(oi[i, n]) + sum(h[j] * int(Bi[v, n, j]) for j in range(R))
            assert out[i, n] == int(f64_to_bf16(float(want)))


def test_one_hot_x_selects_weight_column():
    rng = np.random.default_rng(3)
    V, R, K = 4, 16, 40
    A = bits(rng.standard_normal((V, R, K)))
    x = np.zeros((K, K), np.uint16)
    x[np.arange(K), np.arange(K)] = 0x3F80                       # identity rows
    sorted_ids = np.arange(K, dtype=np.int32)
    inter = lora_shrink(x, 1, A, sorted_ids, np.full(K // 8, 3, np.int32), K, 8, K,
                        np.zeros((K, R), np.float32))
    assert np.array_equal(inter, bf16_to_f64(A[3]).T.astype(np.float32))


def test_zero_weights_and_scale_leave_output():
    wl, li, st = _tiny_stage(0)
    x, A, B, out0 = st.x.host_all(), st.A.host_all(), st.B.host_all(), st.out0.host_all()
    args = (st.x_row_div, li.topk_ids, li.lora_ids, wl.E, wl.L)
    geo = (st.stage.S, st.stage.r, st.stage.Ns)
    res = lora_forward_stage(x, *args, np.zeros_like(A), B, *geo, wl.scale, None, out0, wl.BM)
    valid = ~np.isnan(res["inter"][:, 0])
    assert np.all(res["inter"][valid] == 0)
    assert np.array_equal(res["out"], out0)
    for A_, B_, sc in [(A, B, 0.0), (A, np.zeros_like(B), wl.scale)]:
        res = lora_forward_stage(x, *args, A_, B_, *geo, sc, None, out0, wl.BM)
        assert np.array_equal(res["out"], out0)


def test_slices_read_their_own_columns():
    rng = np.random.default_rng(11)
    S, r, Ns, c = 2, 4, 8, 3
    inter = rng.standard_normal((c, S * r)).astype(np.float32)
    B = bits(rng.standard_normal((1, S * Ns, r)))
    out0 = bits(rng.standard_normal((c, S * Ns)))
    s_ids, e_ids, n = one_block_routing(c, 4)
    full = lora_expand(inter, B, S, r, Ns, 1.0, None, s_ids, e_ids, n, 4, c, out0)
    inter2 = inter.copy()
    inter2[:, r:] = 0.0                                          # kill slice 1's inputs
    half = lora_expand(inter2, B, S, r, Ns, 1.0, None, s_ids, e_ids, n, 4, c, out0)
    assert np.array_equal(half[:, :Ns], full[:, :Ns])
    assert np.array_equal(half[:, Ns:], out0[:, Ns:])


def test_topk_weight_zero_and_linearity():
    rng = np.random.default_rng(12)
    c, r, N = 4, 8, 8
    inter = rng.integers(-3, 4, size=(c, r)).astype(np.float32)
    B = _int_bits(rng, (1, N, r), -2, 2)
    out0 = np.zeros((c, N), np.uint16)
    s_ids, e_ids, n = one_block_routing(c, 4)
    w1 = np.ones(c, np.float32)
    w = np.array([0.0, 1.0, 2.0, 0.5], np.float32)
    o1, p1 = lora_expand(inter, B, 1, r, N, 1.0, w1, s_ids, e_ids, n, 4, c, out0, return_f64=True)
    o2, p2 = lora_expand(inter, B, 1, r, N, 1.0, w, s_ids, e_ids, n, 4, c, out0, return_f64=True)
    assert np.array_equal(o2[0], out0[0])
    np.testing.assert_array_equal(p2, p1 * w[:, None].astype(np.float64))


def test_transposed_weights_would_be_caught():
    # lora_a rows run over K; a transposed read (R x K vs K x R) changes the result
    rng = np.random.default_rng(13)
    R, K = 16, 16
    A = bits(rng.standard_normal((1, R, K)))
    x = bits(rng.standard_normal((1, K)))
    s_ids, e_ids, n = one_block_routing(1, 1)
    inter = lora_shrink(x, 1, A, s_ids, e_ids, n, 1, 1, np.zeros((1, R), np.float32))
    want = bf16_to_f64(A[0]) @ bf16_to_f64(x[0])
    wrong = bf16_to_f64(A[0]).T @ bf16_to_f64(x[0])
    np.testing.assert_allclose(inter[0], want, rtol=1e-6)
    assert not np.allclose(want, wrong)
