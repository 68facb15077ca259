"""Pins of the oracle's align_block_size with a sentinel bucket (step a2)."""

import json
import os

import numpy as np
import pytest

from oracle import align_block_size, align_capacity, virtual_topk
from synth import WORKLOADS, make_routing

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def brute_align(vid, V, BM):
    """Scan-per-bucket construction with plain loops (no sort)."""
    numel = len(vid)
    cap = 0
    seq = []
    exp = []
    for b in range(V + 1):
        members = [i for i in range(numel) if (vid[i] if 0 <= vid[i] < V else V) == b]
        if not members:
            continue
        while len(members) % BM:
            members.append(numel)
        seq.extend(members)
        exp.extend([b if b < V else -1] * (len(members) // BM))
    ntpp = len(seq)
    return seq, exp, ntpp


def check_invariants(vid, V, BM, sorted_ids, expert_ids, ntpp):
    vid = np.asarray(vid, np.int64)
    numel = len(vid)
    cap = len(sorted_ids)
    assert cap % BM == 0 and len(expert_ids) == cap // BM
    assert ntpp % BM == 0 and 0 <= ntpp <= cap
    bucket = np.where((vid >= 0) & (vid < V), vid, V)
    body = sorted_ids[:ntpp]
    real = body[body < numel]
    # every pair appears exactly once, and only pads follow ntpp
    assert np.array_equal(np.sort(real), np.arange(numel))
    assert np.all(sorted_ids[ntpp:] == numel)
    assert np.all(expert_ids[ntpp // BM:] == -1)
    blocks = body.reshape(-1, BM)
    prev = -1
    for t, row in enumerate(blocks):
        ids = row[row < numel]
        e = expert_ids[t]
        if ids.size:
            bs = np.unique(bucket[ids])
            assert bs.size == 1                       # one bucket per block
            b = bs[0]
            assert e == (b if b < V else -1)          # sentinel blocks carry -1
            assert np.all(np.diff(ids) > 0)           # ascending (stable)
            pads = row >= numel
            assert not np.any(pads[:-1] & ~pads[1:])  # pads only at the end of a block
        if e >= 0:
            assert e >= prev                          # real blocks in bucket order
            prev = e
        # a block's valid pairs never come from a different bucket than its id
        if e >= 0:
            assert np.all(bucket[ids] == e)
    # the real buckets' counts equal the histogram
    counts = np.bincount(bucket, minlength=V + 1)
    for b in np.nonzero(counts[:V])[0]:
        tb = np.nonzero(expert_ids == b)[0]
        assert len(tb) == -(-counts[b] // BM)
        members = blocks[tb].reshape(-1)
        assert np.sum(members < numel) == counts[b]


@pytest.mark.parametrize("key", ["align_sentinel_bucket", "remap_then_align"])
def test_worked_examples(key):
    g = GOLDEN[key]
    BM = g["block_m"]
    if "num_vexperts" in g:
        V, vid = g["num_vexperts"], np.array(g["vtopk_ids"])
    else:
        V = g["num_experts"] * g["max_loras"]
        vid = virtual_topk(np.array(g["topk_ids"]), np.array(g["lora_ids"]), g["num_experts"], g["max_loras"])
    assert align_capacity(vid.size, V, BM) == g["capacity"]
    s, e, n = align_block_size(vid, V, BM)
    assert s.tolist() == g["sorted_token_ids"]
    assert e.tolist() == g["expert_ids"]
    assert n == g["num_tokens_post_padded"]


@pytest.mark.parametrize("seed", range(40))
def test_brute_force_small(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(1, 12))
    BM = int(rng.choice([1, 2, 3, 4, 8, 16]))
    numel = int(rng.integers(0, 60))
    vid = rng.integers(-3, V + 3, size=numel)
    s, e, n = align_block_size(vid, V, BM)
    seq, exp, ntpp = brute_align(vid.tolist(), V, BM)
    assert n == ntpp
    assert s[:n].tolist() == seq
    assert e[: n // BM].tolist() == exp
    check_invariants(vid, V, BM, s, e, n)


@pytest.mark.parametrize("name", ["tiny", "decode", "wide", "wide1k", "prefill", "ep", "dense"])
def test_invariants_on_workloads(name):
    wl = WORKLOADS[name]
    topk, lora = make_routing(wl, seed=0)
    vid = virtual_topk(topk, lora, wl.E, wl.L).reshape(-1)
    s, e, n = align_block_size(vid, wl.V, wl.BM)
    assert len(s) == align_capacity(wl.numel, wl.V, wl.BM)
    check_invariants(vid, wl.V, wl.BM, s, e, n)


def test_empty():
    s, e, n = align_block_size(np.zeros(0, np.int32), 16, 16)
    assert n == 0 and s.size == 0 and e.size == 0


def test_all_invalid():
    vid = np.array([-1, -5, 99, -1, 16, -1, -1], np.int32)
    s, e, n = align_block_size(vid, 16, 4)
    assert n == 8                                   # ceil_BM(numel), all in the sentinel bucket
    assert np.all(e == -1)
    assert s[:7].tolist() == list(range(7)) and s[7] == 7


def test_single_bucket():
    vid = np.full(37, 5, np.int32)
    s, e, n = align_block_size(vid, 8, 16)
    assert n == 48
    assert e[:3].tolist() == [5, 5, 5] and np.all(e[3:] == -1)
    assert s[:37].tolist() == list(range(37)) and np.all(s[37:] == 37)


def test_max_buckets():
    # 8191 virtual experts + the sentinel bucket = 8192 buckets (sglang PR 24262, "Risks" item 2)
    V = 8191
    vid = np.array([V - 1, -1, 0, V - 1], np.int32)
    s, e, n = align_block_size(vid, V, 16)
    assert n == 48
    assert e[:3].tolist() == [0, V - 1, -1]
    assert s[:3].tolist() == [2, 4, 4] and s[16:18].tolist() == [0, 3] and s[32] == 1


def test_capacity_is_attained():
    # one pair per bucket: every bucket pads BM-1 slots and ntpp reaches the bound
    for BM in (2, 16, 64):
        V = 40
        vid = np.arange(30, dtype=np.int32)
        s, e, n = align_block_size(vid, V, BM)
        assert n == len(s) == align_capacity(30, V, BM) == 30 * BM
