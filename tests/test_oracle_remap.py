"""Pins of the oracle's virtual top-k remap (step a1)."""

import json
import os

import numpy as np

from oracle import virtual_topk

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def test_worked_example():
    g = GOLDEN["remap_then_align"]
    got = virtual_topk(np.array(g["topk_ids"]), np.array(g["lora_ids"]), g["num_experts"], g["max_loras"])
    assert got.tolist() == g["vtopk_ids"]


def test_negative_sentinels_preserved():
    # sglang PR 24171, "Implementation breakdown" item 2: negative sentinels are kept
    rng = np.random.default_rng(1)
    topk = -rng.integers(1, 50, size=(40, 4)).astype(np.int32)
    for lora in (-1, 0, 3, 7):
        got = virtual_topk(topk, np.full(40, lora, np.int32), 16, 8)
        assert np.array_equal(got, topk)


def test_positive_topk_remapped_correctly():
    rng = np.random.default_rng(2)
    E, L = 32, 5
    topk = rng.integers(0, E, size=(64, 6)).astype(np.int32)
    lora = rng.integers(0, L, size=64).astype(np.int32)
    got = virtual_topk(topk, lora, E, L)
    assert np.all(got >= 0) and np.all(got < E * L)
    # decomposition: the virtual id names (expert, adapter) back
    assert np.array_equal(got % E, topk)
    assert np.array_equal(got // E, np.broadcast_to(lora[:, None], topk.shape))


def test_brute_force_enumeration():
    """Virtual expert ids enumerate (adapter, expert) pairs adapter-major, one per pair."""
    for E, L in [(1, 1), (3, 2), (5, 4), (8, 3)]:
        table = {}
        counter = 0
        for l in range(L):
            for e in range(E):
                table[(e, l)] = counter
                counter += 1
        bases = np.arange(-3, E + 3)
        loras = np.arange(-3, L + 3)
        topk = np.repeat(bases[None, :], len(loras), axis=0).astype(np.int32)
        got = virtual_topk(topk, loras.astype(np.int32), E, L)
        for a, l in enumerate(loras):
            for b, e in enumerate(bases):
                if e < 0:
                    want = e
                elif (int(e), int(l)) in table:
                    want = table[(int(e), int(l))]
                else:
                    want = -1
                assert got[a, b] == want, (E, L, e, l)
        valid = got[got >= 0]
        assert len(np.unique(valid)) == len(valid) == E * L   # one id per (expert, adapter)


def test_no_adapter_never_maps_to_adapter_zero():
    # fork PR #24 "-1 = no adapter": a base-only token must not pick up adapter 0's delta
    topk = np.arange(8, dtype=np.int32).reshape(2, 4)
    got = virtual_topk(topk, np.array([-1, -1], np.int32), 8, 4)
    assert np.all(got == -1)
