"""Large seeded random stages against the oracle: thousands of pairs and up to 4096 virtual
experts, ranks 8-64 with and without per-adapter arrays, one or two slices, BLOCK_M 16-128,
so that the paths of large calls run (the cluster and multi-tile aligns, 16-row shrink items,
512- and 768-column expand items, blocks that loop over items, the two-tile expand, the
tensor-core shrink and expand). Routing bit-exact; intermediates and outputs of every pair
that gets a delta within the parity bars; every other row untouched."""
import numpy as np
import pytest

import oracle
from tests.gpu_util import (bf16_host, check_inter, check_out, mol_lib, to_dev_bf16, to_dev_i32,
                            torch_cuda, valid_pairs)

pytestmark = pytest.mark.gpu
LIM = 48_000_000


def bits(a):
    return oracle.f64_to_bf16(np.asarray(a, np.float64))


def _draw(seed):
    rng = np.random.default_rng(90000 + seed)
    BM = int(rng.choice([16, 32, 64, 128]))
    r = int(rng.choice([8, 16, 32, 64]))
    S = int(rng.integers(1, 3))
    E = int(rng.choice([16, 64, 128, 256]))
    L = int(rng.choice([1, 2, 4, 8, 16]))
    k = int(rng.choice([2, 4, 8]))
    T = int(rng.integers(300, 4000))
    K = int(rng.choice([128, 256, 768, 2048]))
    Ns = int(rng.choice([128, 256, 768, 1536, 2048]))
    V, R = E * L, S * r
    while V * R * K > LIM and K > 64:
        K //= 2
    while V * S * Ns * r > LIM and Ns > 64:
        Ns //= 2
    return dict(BM=BM, r=r, S=S, E=E, L=L, k=k, T=T, K=K, Ns=Ns, V=V, R=R,
                sparse=float(rng.choice([0.0, 0.5])), adapters=bool(rng.integers(0, 2)),
                token_rows=bool(rng.integers(0, 2)), rng=rng)


@pytest.mark.parametrize("seed", range(24))
def test_large_random_stage(seed):
    torch = torch_cuda()
    mol = mol_lib()
    dev = torch.device("cuda:0")
    c = _draw(seed)
    rng = c["rng"]
    E, L, V, BM, S, r, Ns, K, R, T, k = (c[n] for n in ("E", "L", "V", "BM", "S", "r", "Ns", "K", "R", "T", "k"))
    numel, N = T * k, S * Ns
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    topk[rng.random((T, k)) < c["sparse"]] = -1
    lora = rng.integers(-1, L, size=T).astype(np.int32)
    xdiv = k if c["token_rows"] else 1
    x = bits(rng.standard_normal((T if c["token_rows"] else numel, K)))
    A = bits(rng.standard_normal((V, R, K)) * 0.05)
    B = bits(rng.standard_normal((V, N, r)) * 0.05)
    out0 = bits(rng.standard_normal((numel, N)))
    ranks = scal = None
    if c["adapters"]:
        ranks = rng.integers(0, r + 1, L).astype(np.int32)
        ranks[rng.random(L) < 0.3] = r
        scal = rng.uniform(0.25, 2.0, L).astype(np.float32)
    ref = oracle.lora_forward_stage(x, xdiv, topk, lora, E, L, A, B, S, r, Ns, 0.5, None, out0, BM,
                                    lora_ranks=ranks, lora_scalings=scal)
    routing = mol.alloc_routing(numel, V, BM, dev)
    ws = mol.alloc_workspace(numel, V, BM, dev)
    out = to_dev_bf16(out0, dev)
    inter = torch.full((numel, R), float("nan"), dtype=torch.float32, device=dev)
    kw = {}
    if ranks is not None:
        kw = dict(lora_ranks=to_dev_i32(ranks, dev), lora_scalings=torch.from_numpy(scal).to(dev))
    mol.mol_lora_forward(to_dev_bf16(x, dev), xdiv, to_dev_i32(topk, dev), to_dev_i32(lora, dev), E, L,
                         to_dev_bf16(A, dev), to_dev_bf16(B, dev), S, 0.5, out, routing, inter,
                         compute_routing=1 + seed % 2, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert mol.mol_take_fault_flags() == 0
    ntpp = int(routing.num_tokens_post_padded.cpu().item())
    assert ntpp == ref["ntpp"]
    assert np.array_equal(routing.sorted_token_ids.cpu().numpy()[:ntpp], ref["sorted_ids"][:ntpp])
    assert np.array_equal(routing.expert_ids.cpu().numpy()[:ntpp // BM], ref["expert_ids"][:ntpp // BM])
    vt = ref["vtopk"].reshape(-1)
    live = np.nonzero(vt >= 0)[0]
    if ranks is not None:
        live = live[ranks[vt[live] // E] > 0]
    g_inter, g_out = inter.cpu().numpy(), bf16_host(out)
    check_inter(g_inter, ref["inter"], live)
    check_out(g_out, ref["out"], live)
    rest = np.setdiff1d(np.arange(numel), live)
    assert np.all(np.isnan(g_inter[rest]))
    assert np.array_equal(g_out[rest], out0[rest])
