"""GPU parity of the one-CTA-per-row top-K against the cluster top-K (both
exact: the same scores must give the same selection, bit for bit) and
against the oracle, through the indexer, the HSI pool and the Reindex
selection.  Cases cover the candidate path (ragged rows, several ring
stages, rows shorter than k, k = 16 / 512 / 2048, the longest row it takes)
and the whole-row fallback (a threshold bin holding more keys than the
candidate list: all-equal and four-valued scores)."""
import math

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import check_topk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def c2():
    import sparse_attention_fp4_csa2_gb300.build as b
    b.build()
    import sparse_attention_fp4_csa2_gb300 as c
    yield c
    c.set_topk_kernel(c.TOPK_AUTO)


def _both(c2, run):
    """run() under the cluster kernel, then under the row kernel."""
    out = []
    for kern in (c2.TOPK_CLUSTER, c2.TOPK_ROW):
        c2.set_topk_kernel(kern)
        try:
            out.append(run())
        finally:
            c2.set_topk_kernel(c2.TOPK_AUTO)
        assert c2.get_device_status() == 0
    return out


def _index_case(seed, B, cap, n_vis):
    q_idx = synth.normal((B, 32, 128), seed, 3, std=1 / math.sqrt(128))
    w = synth.uniform((B, 32), seed, 4)
    k = synth.indexer_keys(seed, B, cap)
    return q_idx, w, k, torch.tensor(n_vis, dtype=torch.int32)


def _topk(c2, q_idx, w, k, nv, cap, K, pool=None, cand=None):
    kw = {"index_topk": K}
    if cand:
        kw["candidate_topk_blocks"] = cand
    p = c2.Params.make(**kw)
    ws = c2.workspace(c2.OP_INDEXER, q_idx.shape[0], cap, p)
    topk = torch.full((q_idx.shape[0], K), -7, dtype=torch.int32, device="cuda")
    c2.indexer_score_topk(q_idx.cuda(), w.cuda(), k.cuda(), nv.cuda(), cap, p, topk, ws,
                          pool_blocks=None if pool is None else pool.cuda())
    torch.cuda.synchronize()
    return topk.cpu().numpy()


@pytest.mark.parametrize("B,cap,n_vis,K", [
    (3, 4096, [4096, 4000, 9], 512),          # one stage; a row shorter than k
    (3, 3000, [3000, 1000, 77], 16),          # small k
    (2, 70000, [70000, 65537], 512),          # 18 ring stages, ragged tail
    (2, 131072, [131072, 100003], 2048),      # the longest row, the pool's k
    (17, 8192, [8192 - 13 * i for i in range(17)], 512),   # many rows
])
def test_row_topk_matches_cluster_and_oracle(c2, orc, B, cap, n_vis, K):
    q_idx, w, k, nv = _index_case(100 + B + K, B, cap, n_vis)
    a, b = _both(c2, lambda: _topk(c2, q_idx, w, k, nv, cap, K))
    assert np.array_equal(a, b)
    for i in range(B):
        s = orc.index_scores(q_idx[i], w[i], k[i, :n_vis[i]])
        check_topk(b[i], orc.topk(s, K), s, n_valid=n_vis[i])


@pytest.mark.parametrize("cap,values", [(20000, 1), (100000, 4)])
def test_row_topk_whole_row_fallback(c2, orc, cap, values):
    """All-equal scores (every key in one bin: the candidate list overflows)
    and four-valued scores over a long row: the exact whole-row path, ties
    toward the lower index."""
    B, K = 2, 512
    q_idx = torch.zeros(B, 32, 128, dtype=torch.bfloat16)
    q_idx[:, :, 0] = 1.0
    w = torch.ones(B, 32)
    g = torch.Generator().manual_seed(cap + values)
    k = torch.zeros(B, cap, 128, dtype=torch.bfloat16)
    if values > 1:
        k[:, :, 0] = torch.randint(0, values, (B, cap), generator=g).to(torch.bfloat16)
    nv = torch.tensor([cap, cap - 1001], dtype=torch.int32)
    a, b = _both(c2, lambda: _topk(c2, q_idx, w, k, nv, cap, K))
    assert np.array_equal(a, b)
    for i in range(B):
        s = orc.index_scores(q_idx[i], w[i], k[i, :int(nv[i])])
        assert np.array_equal(b[i], orc.topk(s, K))


def _random_pool(seed, B, n_vis, n_pool, slots):
    g = torch.Generator().manual_seed(seed)
    pool = torch.full((B, slots), -1, dtype=torch.int32)
    for b in range(B):
        nb = (n_vis[b] + 7) // 8
        m = min(n_pool, nb)
        pool[b, :m] = torch.randperm(nb, generator=g)[:m].sort().values.to(torch.int32)
    return pool


def test_row_topk_reindex_pool_mapping(c2, orc):
    """Reindex rows: the selection over the pool's positions, mapped back
    through the pool."""
    B, cap = 3, 30000
    n_vis = [30000, 9000, 1001]
    q_idx, w, k, nv = _index_case(41, B, cap, n_vis)
    pool = _random_pool(41, B, n_vis, 1000, 1024)
    a, b = _both(c2, lambda: _topk(c2, q_idx, w, k, nv, cap, 512, pool=pool, cand=1024))
    assert np.array_equal(a, b)
    for i in range(B):
        pos = orc.pool_positions(pool[i].numpy(), n_vis[i])
        s_full = np.full(cap, -np.inf)
        s_full[pos] = orc.index_scores(q_idx[i], w[i], k[i][pos])
        check_topk(b[i], orc.reindex_topk(q_idx[i], w[i], k[i], pool[i].numpy(), n_vis[i], 512), s_full)


def test_row_topk_hsi_pool(c2, orc):
    """The HSI pool's top-2048 blocks (the newest block forced in)."""
    B, cap = 2, 40000
    q_idx, w, k, nv = _index_case(51, B, cap, [40000, 12345])
    p = c2.Params.make(candidate_topk_blocks=2048)
    nblk = (cap + 7) // 8

    def run():
        ws = c2.workspace(c2.OP_DECODE, B, cap, p)
        bs = torch.empty(B, nblk, dtype=torch.float32, device="cuda")
        topk = torch.empty(B, 512, dtype=torch.int32, device="cuda")
        c2.indexer_score_topk(q_idx.cuda(), w.cuda(), k.cuda(), nv.cuda(), cap, p, topk, ws, block_scores=bs)
        pool = torch.empty(B, 2048, dtype=torch.int32, device="cuda")
        c2.hier_pool_select(bs, nv.cuda(), cap, p, pool, ws)
        torch.cuda.synchronize()
        return pool.cpu().numpy()

    a, b = _both(c2, run)
    assert np.array_equal(a, b)
    for i in range(B):
        n = int(nv[i])
        s = orc.index_scores(q_idx[i], w[i], k[i, :n])
        ob = orc.block_scores(s, n, 8)
        ob[(n - 1) // 8] = np.inf
        check_topk(b[i], orc.hsi_pool(s, n, 8, 2048), ob)
        assert (n - 1) // 8 in set(b[i].tolist())
