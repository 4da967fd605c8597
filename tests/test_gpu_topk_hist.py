"""GPU tests of the per-row histogram the bf16 indexer sweep hands to the
cluster top-K (each row's valid scores counted by the top 12 bits of their
keys, at the start of the indexer's workspace; the top-K reads it instead of
sampling the row and clears it).  The selection must be exact whatever the
workspace held before -- zeros, garbage, the counts a Full or a Reindex call
left -- and the counts must be zero after every call."""
import math

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import check_topk

pytestmark = pytest.mark.gpu

HIST_BINS = 4096   # counts per row


@pytest.fixture(scope="module")
def c2():
    import sparse_attention_fp4_csa2_gb300.build as b
    b.build()
    import sparse_attention_fp4_csa2_gb300 as c
    c.set_topk_kernel(c.TOPK_AUTO)
    yield c


def _case(seed, B, cap, n_vis):
    q_idx = synth.normal((B, 32, 128), seed, 3, std=1 / math.sqrt(128))
    w = synth.uniform((B, 32), seed, 4)
    k = synth.indexer_keys(seed, B, cap)
    return q_idx, w, k, torch.tensor(n_vis, dtype=torch.int32)


def _select(c2, p, q_idx, w, k, nv, cap, ws, pool=None):
    B = q_idx.shape[0]
    topk = torch.full((B, p.index_topk), -7, dtype=torch.int32, device="cuda")
    c2.indexer_score_topk(q_idx.cuda(), w.cuda(), k.cuda(), nv.cuda(), cap, p, topk, ws,
                          pool_blocks=None if pool is None else pool.cuda())
    torch.cuda.synchronize()
    assert c2.get_device_status() == 0
    return topk.cpu().numpy()


def _counts_zero(ws, B):
    return bool((ws[:B * HIST_BINS * 4] == 0).all())


def _check_full(orc, sel, q_idx, w, k, n_vis, K):
    for i in range(len(n_vis)):
        s = orc.index_scores(q_idx[i], w[i], k[i, :n_vis[i]])
        check_topk(sel[i], orc.topk(s, K), s, n_valid=n_vis[i])


def test_hist_any_prior_workspace(c2, orc):
    """Garbage (all ones, then random bytes) and a reused workspace give the
    same exact selection, and leave the counts zero."""
    B, cap, K = 4, 65536, 512
    n_vis = [65536, 65000, 40000, 4100]
    q_idx, w, k, nv = _case(71, B, cap, n_vis)
    p = c2.Params.make(index_topk=K)
    ws = c2.workspace(c2.OP_INDEXER, B, cap, p)
    first = _select(c2, p, q_idx, w, k, nv, cap, ws)
    _check_full(orc, first, q_idx, w, k, n_vis, K)
    assert _counts_zero(ws, B)
    again = _select(c2, p, q_idx, w, k, nv, cap, ws)
    assert np.array_equal(first, again)
    ws.fill_(0xFF)
    assert np.array_equal(first, _select(c2, p, q_idx, w, k, nv, cap, ws))
    assert _counts_zero(ws, B)
    g = torch.Generator().manual_seed(5)
    ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, generator=g).cuda())
    assert np.array_equal(first, _select(c2, p, q_idx, w, k, nv, cap, ws))
    assert _counts_zero(ws, B)


def test_hist_full_reindex_full_one_workspace(c2, orc):
    """A Reindex call between two Full calls on one workspace (the counts sit
    in the same place for both)."""
    B, cap, K = 3, 50000, 512
    n_vis = [50000, 30001, 9000]
    q_idx, w, k, nv = _case(72, B, cap, n_vis)
    p = c2.Params.make(index_topk=K, candidate_topk_blocks=1024)
    ws = c2.workspace(c2.OP_INDEXER, B, cap, p)
    first = _select(c2, p, q_idx, w, k, nv, cap, ws)
    _check_full(orc, first, q_idx, w, k, n_vis, K)
    g = torch.Generator().manual_seed(72)
    pool = torch.full((B, 1024), -1, dtype=torch.int32)
    for b in range(B):
        nb = (n_vis[b] + 7) // 8
        m = min(1024, nb)
        pool[b, :m] = torch.randperm(nb, generator=g)[:m].sort().values.to(torch.int32)
    re = _select(c2, p, q_idx, w, k, nv, cap, ws, pool=pool)
    for i in range(B):
        pos = orc.pool_positions(pool[i].numpy(), n_vis[i])
        s_full = np.full(cap, -np.inf)
        s_full[pos] = orc.index_scores(q_idx[i], w[i], k[i][pos])
        check_topk(re[i], orc.reindex_topk(q_idx[i], w[i], k[i], pool[i].numpy(), n_vis[i], K), s_full)
    assert _counts_zero(ws, B)
    assert np.array_equal(first, _select(c2, p, q_idx, w, k, nv, cap, ws))


@pytest.mark.parametrize("n_top,n_tie", [(100, 5000), (0, 3000), (511, 2000), (100, 1500), (0, 1024)])
def test_hist_tied_threshold_bin(c2, orc, n_top, n_tie):
    """Ties at the k-th score: a threshold bin that holds more keys than the
    leader's list (the top-K samples the row instead) or fewer (it selects
    from the counted bin); ties toward the lower index either way."""
    B, cap, K = 2, 32768, 512
    g = torch.Generator().manual_seed(n_top + n_tie)
    q_idx = torch.zeros(B, 32, 128, dtype=torch.bfloat16)
    q_idx[:, :, 0] = 1.0
    w = torch.ones(B, 32) / 32
    k = torch.zeros(B, cap, 128, dtype=torch.bfloat16)
    for b in range(B):
        x = torch.rand(cap, generator=g) * 0.5             # the body: scores below 0.5
        perm = torch.randperm(cap, generator=g)
        x[perm[:n_tie]] = 2.0                               # a crowded bin holding the k-th score
        x[perm[n_tie:n_tie + n_top]] = 3.0 + torch.rand(n_top, generator=g)
        k[b, :, 0] = x.to(torch.bfloat16)
    nv = torch.tensor([cap, cap - 333], dtype=torch.int32)
    p = c2.Params.make(index_topk=K)
    ws = c2.workspace(c2.OP_INDEXER, B, cap, p)
    sel = _select(c2, p, q_idx, w, k, nv, cap, ws)
    for i in range(B):
        s = orc.index_scores(q_idx[i], w[i], k[i, :int(nv[i])])
        assert np.array_equal(sel[i], orc.topk(s, K))
    assert _counts_zero(ws, B)


def test_hist_random_shapes_one_workspace(c2, orc):
    """Seeded random batches, lengths, visible counts and k on one workspace
    sized for the largest (a call's layout follows its own batch, so a call
    may start from another call's scores): every selection exact, the
    call's counts zero after it."""
    g = np.random.default_rng(2024)
    Bmax, capmax = 6, 40000
    pmax = c2.Params.make(index_topk=2048, candidate_topk_blocks=2048)
    ws = c2.workspace(c2.OP_INDEXER, Bmax, capmax, pmax)
    for trial in range(8):
        B = int(g.integers(1, Bmax + 1))
        cap = int(g.integers(1, capmax // 4) * 4)
        K = int(g.choice([16, 100, 512, 2048]))
        n_vis = [int(g.integers(0, cap + 1)) for _ in range(B)]
        n_vis[0] = cap
        q_idx, w, k, nv = _case(300 + trial, B, cap, n_vis)
        p = c2.Params.make(index_topk=K)
        sel = _select(c2, p, q_idx, w, k, nv, cap, ws)
        for i in range(B):
            s = orc.index_scores(q_idx[i], w[i], k[i, :n_vis[i]])
            check_topk(sel[i], orc.topk(s, K), s, n_valid=n_vis[i])
        assert _counts_zero(ws, B)
