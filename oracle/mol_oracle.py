"""CPU oracle for the MoL ("virtual experts") LoRA hot path -- test infrastructure.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline /
reference arm may import this module. The product path (the CUDA library and
its Python binding) never imports, calls or links it, and it shares no code
with that path.

It is written to be read against the pages, not to be fast: numpy in float64,
one library primitive per step (a stable argsort, a matmul), loops over
blocks in the order the method walks them.

Sources (the three pages this subject is drawn from):

* [PR24] fork PR #24 "feat(mol): SGLANG_OPT_MOL_LORA_STAGE_CFG -- MoL LoRA
  stage N-tile tuning" (MindLab-Research/sglang): the "...and grid blowup /
  Root cause" commit, the code-review commit that follows it, the PR body
  sections "Background (measured attribution)", "Root cause" and "Fix", and
  the two LoRA-pool commits "feat(lora): base takes no pool slot" and
  "fix(lora): complete the '-1 = no adapter' sentinel guards".
* [PR24262] prhub summary of sglang PR 24262 (CUDA-JIT align_block_size):
  "Implementation breakdown", "Key source snippet", "Risks".
* [PR24171] prhub summary of sglang PR 24171 (EP correctness of MoE LoRA):
  "Implementation breakdown" item 2, "Key source snippets"
  (_fused_virtual_topk_ids_kernel, _align_block_size_torch), "Risks" item 2.

Readings where the pages are silent or ambiguous (each is restated at the
function that takes it):

* no-adapter tokens (lora id -1, or >= max_loras) remap to -1, like a
  sentinel, so they land in the sentinel bucket and get no delta;
* the sentinel bucket is the last bucket, is padded like the others and is
  counted in num_tokens_post_padded; its blocks carry expert id -1;
* inside a bucket, flat pair indices are in ascending order (stable);
* padding slots of sorted_token_ids hold ``numel``; expert_ids past the last
  block hold -1; the buffer capacity is the tight worst case
  ``ceil_BM(numel + min(numel, V+1) * (BM-1))``;
* lora_a is [V, S*r, K] and lora_b is [V, S*Ns, r], rows contiguous in the
  contracted dim; slice s of lora_b contracts with inter columns
  [s*r, (s+1)*r);
* the shrink writes fp32 intermediates; the expand accumulates, scales, adds
  into the bf16 output and rounds once to nearest-even;
* per-adapter ranks: the weights of an adapter of rank r_l < r are zero-padded,
  so intermediate columns [r_l, r) of each slice are 0 and the expand uses
  only the first r_l; rank 0 returns early (no row written); an optional
  per-adapter scaling multiplies the scalar scale;
* per-token adapter ids come from per-request slot indices; a negative slot,
  one past max_loras, or an adapter of rank 0 gives -1 (no delta).
"""

from __future__ import annotations

import numpy as np

MAX_BUCKETS = 8192  # [PR24262] "Implementation breakdown" item 2: up to 8192 experts


# ---------------------------------------------------------------------------
# bf16 <-> float64, from the IEEE-754 binary16-brain layout
# (1 sign bit, 8 exponent bits with bias 127, 7 fraction bits)
# ---------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns: they are the top half of a binary32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(v) -> np.ndarray:
    """Round float64 values to bf16 bit patterns, once, to nearest, ties to even.

    The quantum of a bf16 number in binade [2^E, 2^(E+1)) is 2^(E-7) (8
    significant bits); below the smallest normal 2^-126 it is the subnormal
    step 2^-133. The value divided by its quantum is rounded half-to-even
    (np.rint) and scaled back, which is exact in float64. Results past the
    largest finite bf16 become infinity, as round-to-nearest requires.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    with np.errstate(invalid="ignore", over="ignore"):
        _, ex = np.frexp(a)                       # a = m * 2^ex, 0.5 <= m < 1
        e = ex.astype(np.int64) - 1               # a in [2^e, 2^(e+1))
        qexp = np.maximum(e - 7, -133)
        n = np.ldexp(a, -qexp)                    # a / quantum, exact
        r = np.ldexp(np.rint(n), qexp)            # round half to even, rescale
        r = np.where(np.isinf(a), np.inf, r)
        r = np.copysign(r, v)
        f = r.astype(np.float32)                  # exact unless it overflowed to inf
    bits = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    return np.where(np.isnan(v), np.uint16(0x7FC0), bits).astype(np.uint16)


# ---------------------------------------------------------------------------
# a1: virtual top-k remap
# ---------------------------------------------------------------------------

def virtual_topk(topk_ids, lora_ids, num_experts: int, max_loras: int) -> np.ndarray:
    """Map each (routed expert, token adapter) pair to a virtual expert id.

    [PR24171] "Key source snippets", _fused_virtual_topk_ids_kernel: the
    virtual id is ``base + lora * num_experts`` and a negative ``base`` (an EP
    sentinel, [PR24171] "Motivation" item 2) is kept verbatim. [PR24] "Root
    cause" commit: the virtual expert space has ``max_loras x n_routed``
    experts, so the id is lora-major.

    Reading: a token with no adapter (lora id -1, [PR24] "fix(lora): -1 = no
    adapter" commit: consumers must write no delta) or an out-of-range
    adapter/expert gets -1, so it lands in the sentinel bucket.
    """
    base = np.asarray(topk_ids, dtype=np.int64)
    lora = np.asarray(lora_ids, dtype=np.int64).reshape(-1, *([1] * (base.ndim - 1)))
    lora = np.broadcast_to(lora, base.shape)
    shifted = base + lora * num_experts
    no_delta = (lora < 0) | (lora >= max_loras) | (base >= num_experts)
    out = np.where(base < 0, base, np.where(no_delta, -1, shifted))
    return out.astype(np.int32)


# ---------------------------------------------------------------------------
# a2: align_block_size with a sentinel bucket
# ---------------------------------------------------------------------------

def ceil_to(n: int, m: int) -> int:
    return -(-n // m) * m


def align_capacity(numel: int, num_vexperts: int, block_m: int) -> int:
    """Length of sorted_token_ids: the worst case over all routings.

    [PR24] code-review commit: sorted_token_ids is the "worst-case untrimmed
    routing buffer". Reading: each of at most min(numel, V+1) non-empty buckets
    adds at most BM-1 padding slots.
    """
    nb = min(numel, num_vexperts + 1)
    return ceil_to(numel + nb * (block_m - 1), block_m)


def align_block_size(vtopk_ids, num_vexperts: int, block_m: int, capacity: int | None = None):
    """Group flat (token, slot) pairs by virtual expert in BLOCK_M-padded buckets.

    [PR24171] "Key source snippets", _align_block_size_torch: ids outside
    [0, V) go to a sentinel bucket numbered V (bucket_count = V + 1), the flat
    ids are argsorted by bucket, and the sentinel bucket's blocks keep expert
    id -1 so that consuming kernels skip them ([PR24171] "Risks" item 2).
    [PR24262] "Implementation breakdown" item 1: histogram, prefix sum,
    expert_ids assignment, token scatter. [PR24] "Root cause" commit: every
    touched bucket is padded to a whole BLOCK_M block.

    Returns (sorted_token_ids int32 [capacity], expert_ids int32
    [capacity // BM], num_tokens_post_padded int).
    """
    vid = np.asarray(vtopk_ids, dtype=np.int64).reshape(-1)
    numel = vid.size
    V, BM = int(num_vexperts), int(block_m)
    assert V + 1 <= MAX_BUCKETS
    if capacity is None:
        capacity = align_capacity(numel, V, BM)

    bucket = np.where((vid >= 0) & (vid < V), vid, V)                 # sentinel bucket = V
    counts = np.bincount(bucket, minlength=V + 1)                     # histogram
    padded = -(-counts // BM) * BM                                    # each bucket to a multiple of BM
    offsets = np.concatenate([[0], np.cumsum(padded)[:-1]])           # exclusive prefix sum
    ntpp = int(padded.sum())
    assert ntpp <= capacity

    order = np.argsort(bucket, kind="stable")                         # ascending flat index in a bucket
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    sorted_ids = np.full(capacity, numel, dtype=np.int64)             # pad value: numel
    expert_ids = np.full(capacity // BM, -1, dtype=np.int64)          # pad / sentinel blocks: -1
    for b in range(V + 1):
        c = counts[b]
        if c == 0:
            continue
        o = offsets[b]
        sorted_ids[o: o + c] = order[starts[b]: starts[b] + c]
        if b < V:
            expert_ids[o // BM: (o + padded[b]) // BM] = b
    return sorted_ids.astype(np.int32), expert_ids.astype(np.int32), ntpp


# ---------------------------------------------------------------------------
# a3 / a4: per-block LoRA shrink and expand
# ---------------------------------------------------------------------------

def _rows(t, idx) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t[idx]
    return np.stack([t[int(i)] for i in idx]) if len(idx) else np.zeros((0,) + tuple(t.row_shape), np.uint16)


def _blocks(sorted_ids, expert_ids, ntpp: int, block_m: int, numel: int):
    """Yield (virtual expert, valid flat pair ids) per block the consumers process.

    A block is processed when it lies below num_tokens_post_padded and its
    expert id is not -1; a row is a pair when its id is in [0, numel).
    """
    for t in range(ntpp // block_m):
        v = int(expert_ids[t])
        if v < 0:
            continue
        ids = np.asarray(sorted_ids[t * block_m:(t + 1) * block_m], dtype=np.int64)
        ids = ids[(ids >= 0) & (ids < numel)]
        if ids.size:
            yield v, ids


def _rank_of(v: int, num_experts, lora_ranks, full_rank: int) -> int:
    """Rank of the adapter of virtual expert v, clamped to [0, full_rank].

    [PR24] "fix(lora): complete the '-1 = no adapter' sentinel guards":
    kernels index lora_ranks by adapter slot and return early on rank 0.
    The adapter of virtual expert v is v // num_experts ([PR24171] remap:
    v = base + lora * E).
    """
    if lora_ranks is None:
        return full_rank
    rl = int(lora_ranks[v // int(num_experts)])
    return min(max(rl, 0), full_rank)


def lora_shrink(x, x_row_div: int, lora_a, sorted_ids, expert_ids, ntpp: int,
                block_m: int, numel: int, inter, num_slices: int = 1, num_experts=None,
                lora_ranks=None):
    """inter[i, j] = sum_k x[i // x_row_div, k] * lora_a[v, j, k] for pairs i of virtual expert v.

    [PR24] "Root cause" commit: the shrink stage is a fused-MoE GEMM over the
    virtual experts with N = S*r (2r = 64 for gate_up) and K = the input
    width; [PR24] code-review commit: its weight is laid out [E, N, K]
    (taken as the correction of the PR body's [E, K, N]).
    Accumulated in float64, rounded once to fp32. Rows of pairs that are in no
    processed block are left as they were.
    With ``lora_ranks`` (per adapter, with ``num_experts``): an adapter of rank
    0 writes nothing; of rank r_l < r writes 0 to columns [r_l, r) of every
    slice (its weight rows there are zero padding and are not read).
    """
    inter = np.array(inter, dtype=np.float32, copy=True)
    R = np.asarray(inter).shape[1]
    r = R // int(num_slices)
    for v, ids in _blocks(sorted_ids, expert_ids, ntpp, block_m, numel):
        rl = _rank_of(v, num_experts, lora_ranks, r)
        if rl == 0:
            continue
        X = bf16_to_f64(_rows(x, ids // x_row_div))        # [c, K]
        Av = bf16_to_f64(lora_a[v])                         # [R, K]
        res = np.zeros((ids.size, R), np.float64)
        for s in range(int(num_slices)):
            res[:, s * r:s * r + rl] = X @ Av[s * r:s * r + rl].T
        inter[ids] = res.astype(np.float32)
    return inter


def lora_expand(inter, lora_b, num_slices: int, rank: int, slice_n: int, scale: float,
                topk_weights, sorted_ids, expert_ids, ntpp: int, block_m: int, numel: int,
                out, return_f64: bool = False, num_experts=None, lora_ranks=None,
                lora_scalings=None):
    """out[i, s*Ns+n] = bf16(out + scale * w_i * sum_j inter[i, s*r+j] * lora_b[v, s*Ns+n, j]).

    [PR24] PR body "Background (measured attribution)": the expand is an
    M x N output with a narrow K = rank contraction, added into the MoE
    output; "Fix": its weight view is [E, N, K]. Slice s of a stacked
    adapter reads inter columns [s*r, (s+1)*r). Accumulation, scaling and the
    add into the old output are in float64, then one round to nearest-even
    bf16. ``topk_weights`` (optional, per pair) multiplies the delta. Rows of
    pairs in no processed block are bit-unchanged ([PR24] "-1 = no adapter":
    no delta is written).
    With ``lora_ranks``: the sum runs over j < r_l only, and rank 0 returns
    early (rows bit-unchanged, [PR24] "complete the '-1 = no adapter'
    sentinel guards": same meaning as the rank == 0 branch). With
    ``lora_scalings``: the delta is further multiplied by the adapter's scaling.
    """
    out = np.array(out, dtype=np.uint16, copy=True)
    S, r, Ns = int(num_slices), int(rank), int(slice_n)
    pre = np.full(out.shape, np.nan) if return_f64 else None
    I_all = np.asarray(inter)
    for v, ids in _blocks(sorted_ids, expert_ids, ntpp, block_m, numel):
        rl = _rank_of(v, num_experts, lora_ranks, r)
        if rl == 0:
            continue
        sc = float(scale)
        if lora_scalings is not None:
            sc *= float(np.float32(lora_scalings[v // int(num_experts)]))
        Bv = bf16_to_f64(lora_b[v])                          # [S*Ns, r]
        w = 1.0 if topk_weights is None else np.asarray(topk_weights, np.float64)[ids][:, None]
        for s in range(S):
            I = I_all[ids, s * r:s * r + rl].astype(np.float64)    # [c, r_l]
            acc = I @ Bv[s * Ns:(s + 1) * Ns, :rl].T               # [c, Ns]
            cols = slice(s * Ns, (s + 1) * Ns)
            new = bf16_to_f64(out[ids, cols]) + sc * w * acc
            if pre is not None:
                pre[ids, cols] = new
            out[ids, cols] = f64_to_bf16(new)
    return (out, pre) if return_f64 else out


def lora_forward_stage(x, x_row_div, topk_ids, lora_ids, num_experts, max_loras,
                       lora_a, lora_b, num_slices, rank, slice_n, scale, topk_weights,
                       out, block_m, inter_fill=np.nan, routing=None, lora_ranks=None,
                       lora_scalings=None):
    """One stage end to end: remap -> align -> shrink -> expand (a1..a4).

    ``routing`` = (vtopk, sorted_ids, expert_ids, ntpp) reuses a routing (the
    down stage reuses the gate_up routing, [PR24] "Background": one
    moe_align_block_size per layer feeds all MoL stages).
    """
    topk = np.asarray(topk_ids)
    numel = topk.size
    V = num_experts * max_loras
    if routing is None:
        vtopk = virtual_topk(topk, lora_ids, num_experts, max_loras)
        sorted_ids, expert_ids, ntpp = align_block_size(vtopk, V, block_m)
    else:
        vtopk, sorted_ids, expert_ids, ntpp = routing
    R = num_slices * rank
    inter0 = np.full((numel, R), inter_fill, dtype=np.float32)
    inter = lora_shrink(x, x_row_div, lora_a, sorted_ids, expert_ids, ntpp, block_m, numel, inter0,
                        num_slices, num_experts, lora_ranks)
    new_out = lora_expand(inter, lora_b, num_slices, rank, slice_n, scale, topk_weights,
                          sorted_ids, expert_ids, ntpp, block_m, numel, out,
                          num_experts=num_experts, lora_ranks=lora_ranks,
                          lora_scalings=lora_scalings)
    return dict(vtopk=vtopk, sorted_ids=sorted_ids, expert_ids=expert_ids, ntpp=ntpp,
                inter=inter, out=new_out)


# ---------------------------------------------------------------------------
# c5: per-pair brute force, no routing and no sorting (small inputs only)
# ---------------------------------------------------------------------------

def brute_force_stage(topk_ids, lora_ids, num_experts, max_loras, x, x_row_div,
                      lora_a, lora_b, num_slices, rank, slice_n, scale, topk_weights, out,
                      lora_ranks=None, lora_scalings=None):
    """Delta of every (token, slot) pair computed straight from (expert e, adapter l).

    Weights of (e, l) are read from the lora-major stacks viewed as
    [max_loras][num_experts] ([PR24] "Root cause": max_loras x n_routed
    virtual experts). Pure-Python loops; the intermediate is rounded to fp32
    as the method defines. Returns (inter dict {pair: fp32 list}, out uint16).
    """
    topk = np.asarray(topk_ids)
    T, k = topk.shape
    out = np.array(out, dtype=np.uint16, copy=True)
    S, r, Ns = num_slices, rank, slice_n
    inters = {}
    for t in range(T):
        l = int(lora_ids[t])
        for kk in range(k):
            e = int(topk[t, kk])
            pair = t * k + kk
            if e < 0 or e >= num_experts or l < 0 or l >= max_loras:
                continue
            rl = r if lora_ranks is None else min(max(int(lora_ranks[l]), 0), r)
            if rl == 0:  # rank 0: early return, nothing written
                continue
            sc = scale if lora_scalings is None else scale * float(np.float32(lora_scalings[l]))
            slot = l * num_experts + e
            xa = [float(v) for v in bf16_to_f64(x[pair // x_row_div])]
            Aw = bf16_to_f64(lora_a[slot])
            Bw = bf16_to_f64(lora_b[slot])
            h = []
            for j in range(S * r):
                if j % r >= rl:  # beyond the adapter's rank: zero padding
                    h.append(0.0)
                    continue
                row = Aw[j]
                h.append(float(np.float32(sum(xa[q] * float(row[q]) for q in range(len(xa))))))
            inters[pair] = h
            w = 1.0 if topk_weights is None else float(topk_weights[pair])
            for s in range(S):
                for n in range(Ns):
                    col = s * Ns + n
                    acc = sum(h[s * r + j] * float(Bw[col, j]) for j in range(rl))
                    old = float(bf16_to_f64(out[pair, col]))
                    out[pair, col] = f64_to_bf16(old + sc * w * acc)
    return inters, out


# ---------------------------------------------------------------------------
# per-request adapter slots -> per-token adapter ids (the step before a1)
# ---------------------------------------------------------------------------

def token_lora_ids(weight_indices, seg_indptr, num_tokens: int, max_loras: int,
                   lora_ranks=None) -> np.ndarray:
    """lora_ids[t] = the adapter slot of the request that token t belongs to, or -1.

    [PR24] "feat(lora): base takes no pool slot": a request without an
    adapter has weight index -1 ("no adapter"); "fix(lora): complete the
    '-1 = no adapter' sentinel guards": every consumer checks for a negative
    index BEFORE it indexes lora_ranks, with the meaning of the existing
    rank == 0 branch (no delta), and the CPU path of _compute_moe_lora_info
    filters negative indices before its scatter. Request q owns tokens
    [seg_indptr[q], seg_indptr[q+1]). Reading: a slot outside [0, max_loras),
    or of rank 0 when lora_ranks is given, gives -1; tokens outside every
    request's segment get -1.
    """
    wi = np.asarray(weight_indices, dtype=np.int64)
    seg = np.asarray(seg_indptr, dtype=np.int64)
    out = np.full(int(num_tokens), -1, dtype=np.int32)
    for q in range(wi.size):
        w = int(wi[q])
        if w < 0 or w >= max_loras:
            continue
        if lora_ranks is not None and int(lora_ranks[w]) <= 0:
            continue
        lo, hi = max(int(seg[q]), 0), min(int(seg[q + 1]), int(num_tokens))
        if hi > lo:
            out[lo:hi] = w
    return out

