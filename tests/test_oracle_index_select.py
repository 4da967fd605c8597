"""Pins for the oracle's indexer score, top-K and hierarchical pool.

Indexer score s_n = sum_h w_h ReLU(q_h . k_n) over 32 heads x 128 dims
("DeepSeek-V4.1-Flash - Architecture" section 2 main attention settings).
Top-K selection: the 512 highest, ties toward the lower index (a reading),
checked against a brute-force sort.  HSI (en.mycoding.id section 2.3.4,
Architecture notes section 3): block max over 8 positions with -inf padding of
the last block, the latest block forced in, top-2048 blocks, expanded to
positions and truncated to the visible width."""
import math

import numpy as np
import torch


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)


def test_index_scores_match_einsum(orc):
    rng = np.random.default_rng(0)
    q = _bf16(rng.standard_normal((32, 128)) / math.sqrt(128))
    w = rng.uniform(0, 1, 32).astype(np.float32)
    k = _bf16(rng.standard_normal((300, 128)))
    s = orc.index_scores(q, w, k)
    dots = np.einsum("hd,nd->nh", q.double().numpy(), k.double().numpy())
    ref = (np.maximum(dots, 0.0) * w.astype(np.float64)).sum(1)
    assert np.allclose(s, ref, rtol=1e-12, atol=1e-12)


def test_index_scores_closed_form_onehot(orc):
    rng = np.random.default_rng(1)
    q = _bf16(rng.standard_normal((32, 128)))
    w = rng.uniform(-1, 1, 32).astype(np.float32)
    k = torch.zeros(128, 128, dtype=torch.bfloat16)
    k[torch.arange(128), torch.arange(128)] = 1.0
    s = orc.index_scores(q, w, k)
    qd = q.double().numpy()
    for d in range(128):
        exp = sum(float(w[h]) * max(0.0, qd[h, d]) for h in range(32))
        assert abs(s[d] - exp) < 1e-12


def test_index_scores_relu_kills_negative_heads(orc):
    q = torch.zeros(32, 128, dtype=torch.bfloat16)
    q[:, 0] = -1.0
    k = torch.zeros(4, 128, dtype=torch.bfloat16)
    k[:, 0] = torch.tensor([1.0, 2.0, -1.0, 0.0])
    w = np.ones(32, np.float32)
    s = orc.index_scores(q, w, k)
    assert list(s) == [0.0, 0.0, 32.0, 0.0]


def _topk_brute(s, k, valid=None):
    cand = [i for i in range(len(s)) if valid is None or valid[i]]
    cand.sort(key=lambda i: (-s[i], i))
    sel = sorted(cand[:k])
    return sel + [-1] * (k - len(sel))


def test_topk_bruteforce_with_ties(orc):
    rng = np.random.default_rng(2)
    for trial in range(30):
        n = int(rng.integers(1, 200))
        k = int(rng.integers(1, 80))
        s = rng.integers(-5, 5, n).astype(np.float64)     # many ties
        valid = rng.integers(0, 2, n).astype(np.uint8) if trial % 3 == 0 else None
        got = list(orc.topk(s, k, valid))
        assert got == _topk_brute(list(s), k, valid)


def test_topk_k_at_least_n_returns_all(orc):
    s = np.random.default_rng(3).standard_normal(37)
    got = orc.topk(s, 64)
    assert list(got[:37]) == list(range(37)) and np.all(got[37:] == -1)


def _blocks_brute(s, n_vis, bs, reduce_sum=False):
    out = []
    for b in range((n_vis + bs - 1) // bs):
        vals = [s[p] if p < n_vis else -math.inf for p in range(b * bs, b * bs + bs)]
        out.append(sum(v for v in vals if v != -math.inf) if reduce_sum else max(vals))
    return out


def test_block_scores_match_bruteforce(orc):
    rng = np.random.default_rng(4)
    for n_vis in [1, 7, 8, 9, 64, 101]:
        s = rng.standard_normal(n_vis)
        assert list(orc.block_scores(s, n_vis, 8)) == _blocks_brute(list(s), n_vis, 8)
        assert np.allclose(orc.block_scores(s, n_vis, 8, reduce_sum=True), _blocks_brute(list(s), n_vis, 8, True))


def test_hsi_pool_forces_latest_block(orc):
    n_vis = 8 * 50 + 3
    s = np.linspace(10, 0, n_vis)          # latest block has the lowest scores
    pool = orc.hsi_pool(s, n_vis, 8, 5)
    assert (n_vis - 1) // 8 in set(pool.tolist())
    assert list(pool) == [0, 1, 2, 3, (n_vis - 1) // 8]


def test_hsi_pool_bruteforce(orc):
    rng = np.random.default_rng(5)
    for n_vis in [17, 200, 333]:
        s = rng.integers(0, 6, n_vis).astype(np.float64)
        bsc = _blocks_brute(list(s), n_vis, 8)
        bsc[(n_vis - 1) // 8] = math.inf
        exp = _topk_brute(bsc, 7)
        assert list(orc.hsi_pool(s, n_vis, 8, 7)) == exp


def test_pool_positions_truncate_to_width(orc):
    pos = orc.pool_positions(np.array([0, 2, -1]), 20, 8)
    assert list(pos) == list(range(8)) + list(range(16, 20))


def test_pool_covering_all_blocks_equals_flat_indexer(orc):
    """A hierarchical pool that covers every block leaves the flat indexer's
    top-K unchanged."""
    rng = np.random.default_rng(6)
    n_vis = 8 * 40 + 5
    q = _bf16(rng.standard_normal((32, 128)) / math.sqrt(128))
    w = rng.uniform(0, 1, 32).astype(np.float32)
    q2 = _bf16(rng.standard_normal((32, 128)) / math.sqrt(128))
    k = _bf16(rng.standard_normal((n_vis, 128)))
    s = orc.index_scores(q, w, k)
    pool = orc.hsi_pool(s, n_vis, 8, 2048)
    assert np.array_equal(orc.pool_positions(pool, n_vis), np.arange(n_vis))
    flat = orc.topk(orc.index_scores(q2, w, k), 32)
    assert np.array_equal(orc.reindex_topk(q2, w, k, pool, n_vis, 32), flat)


def test_planted_blocks_recalled(orc):
    import synth
    n_vis = 8 * 512
    q = synth.normal((1, 32, 128), 7, 3, std=1 / math.sqrt(128))
    w = synth.uniform((1, 32), 7, 4)
    k = synth.indexer_keys(7, 1, n_vis)
    ids = synth.plant_blocks(k, q, w, n_vis, 16, 7)
    s = orc.index_scores(q[0], w[0], k[0])
    pool = orc.hsi_pool(s, n_vis, 8, 64)
    assert set(ids[0].tolist()) <= set(pool.tolist())
