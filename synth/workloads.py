"""Workload shapes and seeded input generators for the MoL LoRA hot path.

Every array here is an *input*: per-token routing (top-k routed expert ids
with -1 sentinels, one adapter id per token with -1 = no adapter), bf16
activations, the two LoRA weight stacks per stage and the bf16 MoE output
that the LoRA delta is added into. bf16 arrays are carried as numpy uint16
bit patterns.

Large float tensors are drawn as *windows* of one seeded normal pool: row q of
the tensor is the contiguous run ``pool[off_q : off_q + row_len]`` of an
extended pool. When the whole tensor fits in the pool the offsets are
``q * row_len`` (the windows tile the pool: a plain i.i.d. array). Above 2**24
elements the offsets are distinct random multiples of 64, so every row has the
stated N(0, sigma) marginal, distinct rows hold distinct data, and an 8 GB
weight stack costs one 2**24-value draw instead of 4G draws.

Workloads follow the pages' MoL decode attribution (fork PR #24, "Background
(measured attribution)": bs=23 decode, rank-32 adapters, down-delta expand to
N=6144) and the EP sentinel case of sglang PR 24171 ("Motivation": -1 topk ids
after expert-parallel dispatch).
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np

POOL_MAX = 1 << 24


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16) with torch's round-to-nearest-even cast."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@dataclass(frozen=True)
class Stage:
    """One LoRA stage of a MoE layer: shrink K -> S*r, expand S*r -> S*Ns."""

    name: str
    K: int            # shrink contraction dim (hidden for gate_up, moe_intermediate for down)
    S: int            # slices stacked in one adapter (2 = [gate; up], 1 = down)
    r: int            # LoRA rank per slice
    Ns: int           # output width per slice
    token_rows: bool  # x rows are token rows (pair i reads row i // topk), else pair rows

    @property
    def R(self) -> int:
        return self.S * self.r

    @property
    def N(self) -> int:
        return self.S * self.Ns


@dataclass(frozen=True)
class Workload:
    name: str
    T: int                      # tokens
    E: int                      # routed experts
    topk: int
    L: int                      # max_loras (adapter slots)
    BM: int                     # BLOCK_M of the align step
    stages: Sequence[Stage]
    scale: float = 2.0          # alpha / r
    expert_dist: str = "uniform"   # "uniform" | "zipf"
    zipf_s: float = 1.1
    sentinel: str = "none"      # "none" | "frac" (sentinel_frac of flat ids) | "half"
    sentinel_frac: float = 0.0
    lora_dist: str = "uniform"  # "uniform" over {-1..L-1} | "zero" (every token adapter 0)
    note: str = ""

    @property
    def V(self) -> int:
        return self.E * self.L

    @property
    def numel(self) -> int:
        return self.T * self.topk


def _gate_up(K, r, inter):
    return Stage("gate_up", K=K, S=2, r=r, Ns=inter, token_rows=True)


def _down(K, r, hidden):
    return Stage("down", K=K, S=1, r=r, Ns=hidden, token_rows=False)


WORKLOADS = {
    "tiny": Workload(
        "tiny", T=16, E=8, topk=2, L=2, BM=16,
        stages=(Stage("single", K=256, S=1, r=16, Ns=128, token_rows=True),),
        sentinel="frac", sentinel_frac=0.10,
        note="16 tokens, 8 experts, top-2, 2 adapters -> 16 virtual experts"),
    "decode": Workload(
        "decode", T=23, E=128, topk=8, L=8, BM=16,
        stages=(_gate_up(2048, 32, 768), _down(768, 32, 2048)),
        note="bs=23 decode, 128 experts x 8 adapters -> 1024 virtual experts"),
    "wide": Workload(
        "wide", T=23, E=128, topk=8, L=8, BM=16,
        stages=(_down(2560, 32, 6144),),
        expert_dist="zipf",
        note="down-delta decode with N=6144 output, Zipf(1.1) expert popularity"),
    "wide1k": Workload(
        "wide1k", T=138, E=128, topk=8, L=8, BM=16,
        stages=(_down(2560, 32, 6144),),
        expert_dist="zipf",
        note="wide with 138 tokens (23 requests x 6 verify tokens) -> ~1.1k real pairs"),
    "prefill": Workload(
        "prefill", T=4096, E=128, topk=8, L=63, BM=64,
        stages=(_gate_up(4096, 64, 1536), _down(1536, 64, 4096)),
        note="4096-token prefill, 8064 virtual experts (+1 sentinel bucket)"),
    "ep": Workload(
        "ep", T=8192, E=256, topk=8, L=16, BM=64,
        stages=(_gate_up(2048, 16, 768), _down(768, 16, 2048)),
        sentinel="half",
        note="expert-parallel prefill: half of the flat topk ids are -1 (non-local experts)"),
    "dense": Workload(
        "dense", T=4096, E=128, topk=8, L=1, BM=64,
        stages=(_gate_up(4096, 64, 1536), _down(1536, 64, 4096)),
        lora_dist="zero",
        note="one adapter for every token: ~256 rows per virtual expert"),
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng([int(k) & 0xFFFFFFFF for k in key])


_TAGS = {"topk": 1, "sent": 2, "lora": 3, "x": 10, "A": 11, "B": 12, "out": 13, "w": 14}


def make_routing(wl: Workload, seed: int, layer: int = 0):
    """topk_ids int32 [T, topk] (distinct experts per token, -1 sentinels) and lora_ids int32 [T].

    k distinct experts per token are drawn without replacement with the
    Gumbel-top-k construction over log-popularity (uniform or Zipf rank^-s).
    """
    T, E, k = wl.T, wl.E, wl.topk
    rng = _rng(seed, layer, _TAGS["topk"])
    if wl.expert_dist == "zipf":
        logp = -wl.zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
    else:
        logp = np.zeros(E)
    g = rng.gumbel(size=(T, E))
    topk_ids = np.argsort(-(logp[None, :] + g), axis=1, kind="stable")[:, :k].astype(np.int32)

    numel = T * k
    flat = topk_ids.reshape(-1)
    srng = _rng(seed, layer, _TAGS["sent"])
    if wl.sentinel == "frac":
        n_s = int(round(wl.sentinel_frac * numel))
        flat[srng.permutation(numel)[:n_s]] = -1
    elif wl.sentinel == "half":
        flat[srng.permutation(numel)[: numel // 2]] = -1
    topk_ids = flat.reshape(T, k)

    lrng = _rng(seed, layer, _TAGS["lora"])
    if wl.lora_dist == "zero":
        lora_ids = np.zeros(T, dtype=np.int32)
    else:
        lora_ids = lrng.integers(-1, wl.L, size=T).astype(np.int32)
    return np.ascontiguousarray(topk_ids), lora_ids


class WindowedWeights:
    """A bf16 tensor [rows, *row_shape] drawn as windows of one N(0, sigma) pool."""

    def __init__(self, rows: int, row_shape: Sequence[int], sigma: float,
                 pool_key: Sequence[int], off_key: Sequence[int]):
        self.rows = int(rows)
        self.row_shape = tuple(int(s) for s in row_shape)
        self.row_len = int(np.prod(self.row_shape))
        total = self.rows * self.row_len
        P = min(total, POOL_MAX)
        P = max(P, self.row_len)
        pool = _rng(*pool_key).standard_normal(P, dtype=np.float32) * np.float32(sigma)
        pool16 = bf16_bits_from_f32(pool)
        if total <= P:
            self.offsets = np.arange(self.rows, dtype=np.int64) * self.row_len
        else:
            n_slots = P // 64
            orng = _rng(*off_key)
            if self.rows <= n_slots:
                slots = orng.choice(n_slots, size=self.rows, replace=False)
            else:
                slots = orng.integers(0, n_slots, size=self.rows)
            self.offsets = slots.astype(np.int64) * 64
        # extended pool: a window never wraps
        self.pool = np.concatenate([pool16, pool16[: self.row_len]])

    @property
    def shape(self):
        return (self.rows,) + self.row_shape

    def host(self, q: int) -> np.ndarray:
        o = int(self.offsets[q])
        return self.pool[o: o + self.row_len].reshape(self.row_shape)

    def __getitem__(self, q):
        return self.host(int(q))

    def __len__(self):
        return self.rows

    def host_all(self) -> np.ndarray:
        win = np.lib.stride_tricks.sliding_window_view(self.pool, self.row_len)
        return np.ascontiguousarray(win[self.offsets]).reshape(self.shape)

    def to_device(self, device):
        """torch.bfloat16 tensor of the full shape, built on `device` (plumbing only)."""
        import torch

        pool = torch.from_numpy(self.pool.view(np.int16)).to(device)
        out = torch.empty((self.rows, self.row_len), dtype=torch.int16, device=device)
        win = pool.unfold(0, self.row_len, 1)
        offs = torch.from_numpy(self.offsets).to(device)
        chunk = max(1, (1 << 27) // max(1, self.row_len))
        for q0 in range(0, self.rows, chunk):
            q1 = min(self.rows, q0 + chunk)
            out[q0:q1] = win.index_select(0, offs[q0:q1])
        del pool
        return out.view(torch.bfloat16).reshape(self.shape)


@dataclass
class StageInputs:
    stage: Stage
    x: WindowedWeights       # [rows_x, K]
    A: WindowedWeights       # [V, R, K]   (lora_a, K-contiguous rows)
    B: WindowedWeights       # [V, N, r]   (lora_b, r-contiguous rows)
    out0: WindowedWeights    # [numel, N]  initial MoE output (per pair)
    x_row_div: int           # pair i reads x row i // x_row_div


@dataclass
class LayerInputs:
    wl: Workload
    seed: int
    layer: int
    topk_ids: np.ndarray
    lora_ids: np.ndarray
    stages: list = field(default_factory=list)


def make_layer(wl: Workload, seed: int, layer: int = 0,
               x_sigma: float = 1.0, w_sigma: float = 0.02, out_sigma: float = 1.0) -> LayerInputs:
    """Routing plus per-stage x, lora_a, lora_b and initial output for one MoE layer.

    Pools are keyed by (seed, stage, tensor); window offsets also by layer, so
    layers of one run hold distinct weights drawn from shared pools.
    """
    topk_ids, lora_ids = make_routing(wl, seed, layer)
    li = LayerInputs(wl, seed, layer, topk_ids, lora_ids)
    for si, st in enumerate(wl.stages):
        rows_x = wl.T if st.token_rows else wl.numel
        base = (seed, si)
        x = WindowedWeights(rows_x, (st.K,), x_sigma,
                            base + (_TAGS["x"],), base + (_TAGS["x"], layer, 7))
        A = WindowedWeights(wl.V, (st.R, st.K), w_sigma,
                            base + (_TAGS["A"],), base + (_TAGS["A"], layer, 7))
        B = WindowedWeights(wl.V, (st.N, st.r), w_sigma,
                            base + (_TAGS["B"],), base + (_TAGS["B"], layer, 7))
        out0 = WindowedWeights(wl.numel, (st.N,), out_sigma,
                               base + (_TAGS["out"],), base + (_TAGS["out"], layer, 7))
        if layer:
            # distinct activations/outputs per layer: re-key the pools of the small tensors
            x = WindowedWeights(rows_x, (st.K,), x_sigma,
                                base + (_TAGS["x"], layer), base + (_TAGS["x"], layer, 7))
            out0 = WindowedWeights(wl.numel, (st.N,), out_sigma,
                                   base + (_TAGS["out"], layer), base + (_TAGS["out"], layer, 7))
        li.stages.append(StageInputs(st, x, A, B, out0, wl.topk if st.token_rows else 1))
    return li


def topk_weights(numel: int, seed: int) -> np.ndarray:
    """Per-pair routed weights in [0, 1) (fp32), for the optional weighted delta."""
    return _rng(seed, _TAGS["w"]).random(numel, dtype=np.float32)
