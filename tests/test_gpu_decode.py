"""GPU parity of the indexer sweep + top-K, the HSI pool, the Reindex sweep,
the sparse readout and the Full / Reindex / Reuse modes against the oracle
(small sizes that still span several tiles and a ragged tail)."""
import math

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import check_attn, check_lse, check_topk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def c2():
    import sparse_attention_fp4_csa2_gb300.build as b
    b.build()
    import sparse_attention_fp4_csa2_gb300 as c
    return c


def _params(c2, **kw):
    return c2.Params.make(**kw)


def _index_case(seed, B, cap, n_vis):
    q_idx = synth.normal((B, 32, 128), seed, 3, std=1 / math.sqrt(128))
    w = synth.uniform((B, 32), seed, 4)
    k = synth.indexer_keys(seed, B, cap)
    return q_idx, w, k, torch.tensor(n_vis, dtype=torch.int32)


@pytest.mark.parametrize("B,cap,n_vis,K", [(1, 4096, [4096], 512), (3, 3000, [3000, 1000, 77], 512),
                                           (2, 700, [700, 333], 1024), (1, 128, [5], 16)])
def test_full_indexer_topk_and_block_scores(c2, orc, B, cap, n_vis, K):
    q_idx, w, k, nv = _index_case(10 + B, B, cap, n_vis)
    p = _params(c2, index_topk=K)
    n_max = cap
    ws = c2.workspace(c2.OP_INDEXER, B, n_max, p)
    topk = torch.full((B, K), -7, dtype=torch.int32, device="cuda")
    nblk = (n_max + 7) // 8
    bs = torch.empty(B, nblk, dtype=torch.float32, device="cuda")
    c2.indexer_score_topk(q_idx.cuda(), w.cuda(), k.cuda(), nv.cuda(), n_max, p, topk, ws, block_scores=bs)
    assert c2.get_device_status() == 0
    topk, bs = topk.cpu().numpy(), bs.cpu().numpy()
    for b in range(B):
        s = orc.index_scores(q_idx[b], w[b], k[b, :n_vis[b]])
        check_topk(topk[b], orc.topk(s, K), s, n_valid=n_vis[b])
        ob = orc.block_scores(s, n_vis[b], 8)
        nb = len(ob)
        assert np.allclose(bs[b, :nb], ob, rtol=1e-4, atol=1e-4)
        assert np.all(np.isneginf(bs[b, nb:]))


def test_all_equal_scores_ties_to_lower_index(c2):
    """Zero keys give every position the same score: the top-K must be the K
    lowest positions (ties toward the lower index)."""
    B, cap, K = 2, 5000, 512
    q_idx = torch.ones(B, 32, 128, dtype=torch.bfloat16)
    w = torch.ones(B, 32)
    k = torch.zeros(B, cap, 128, dtype=torch.bfloat16)
    nv = torch.tensor([5000, 4000], dtype=torch.int32)
    p = _params(c2, index_topk=K)
    ws = c2.workspace(c2.OP_INDEXER, B, cap, p)
    topk = torch.empty(B, K, dtype=torch.int32, device="cuda")
    c2.indexer_score_topk(q_idx.cuda(), w.cuda(), k.cuda(), nv.cuda(), cap, p, topk, ws)
    assert np.array_equal(topk.cpu().numpy(), np.tile(np.arange(K), (B, 1)))


def test_hsi_pool_select(c2, orc):
    B, cap = 2, 40000
    q_idx, w, k, nv = _index_case(21, B, cap, [40000, 12345])
    ids = synth.plant_blocks(k, q_idx, w, 12345, 16, 21)
    p = _params(c2, candidate_topk_blocks=512)
    ws = c2.workspace(c2.OP_DECODE, B, cap, p)
    nblk = (cap + 7) // 8
    bs = torch.empty(B, nblk, dtype=torch.float32, device="cuda")
    topk = torch.empty(B, 512, dtype=torch.int32, device="cuda")
    c2.indexer_score_topk(q_idx.cuda(), w.cuda(), k.cuda(), nv.cuda(), cap, p, topk, ws, block_scores=bs)
    pool = torch.empty(B, 512, dtype=torch.int32, device="cuda")
    c2.hier_pool_select(bs, nv.cuda(), cap, p, pool, ws)
    assert c2.get_device_status() == 0
    pool = pool.cpu().numpy()
    for b in range(B):
        n = int(nv[b])
        s = orc.index_scores(q_idx[b], w[b], k[b, :n])
        ob = orc.block_scores(s, n, 8)
        ob[(n - 1) // 8] = np.inf
        check_topk(pool[b], orc.hsi_pool(s, n, 8, 512), ob)
        assert (n - 1) // 8 in set(pool[b].tolist())
    assert set(ids[1].tolist()) <= set(pool[1].tolist())


def test_block_sum_reduction_and_pool(c2, orc):
    """block_reduce = 1 (blocks scored by the sum of their 8 positions, the
    other reading of "sums scores over blocks of 8"): the sweep's block scores
    and the HSI pool built from them follow the oracle's sum reduction."""
    B, cap = 2, 9000
    n_vis = [9000, 4321]
    q_idx, w, k, nv = _index_case(23, B, cap, n_vis)
    p = _params(c2, candidate_topk_blocks=256, block_reduce=1)
    ws = c2.workspace(c2.OP_DECODE, B, cap, p)
    nblk = (cap + 7) // 8
    bs = torch.empty(B, nblk, dtype=torch.float32, device="cuda")
    topk = torch.empty(B, 512, dtype=torch.int32, device="cuda")
    c2.indexer_score_topk(q_idx.cuda(), w.cuda(), k.cuda(), nv.cuda(), cap, p, topk, ws, block_scores=bs)
    pool = torch.empty(B, 256, dtype=torch.int32, device="cuda")
    c2.hier_pool_select(bs, nv.cuda(), cap, p, pool, ws)
    assert c2.get_device_status() == 0
    bs, pool = bs.cpu().numpy(), pool.cpu().numpy()
    for b in range(B):
        n = n_vis[b]
        s = orc.index_scores(q_idx[b], w[b], k[b, :n])
        ob = orc.block_scores(s, n, 8, reduce_sum=True)
        nb = len(ob)
        assert not np.allclose(ob, orc.block_scores(s, n, 8))          # the two readings differ here
        assert np.allclose(bs[b, :nb], ob, rtol=1e-4, atol=1e-4 * np.abs(ob).max())
        assert np.all(np.isneginf(bs[b, nb:]))
        ob[(n - 1) // 8] = np.inf                                      # the latest block is forced
        check_topk(pool[b], orc.hsi_pool(s, n, 8, 256, reduce_sum=True), ob)
        assert (n - 1) // 8 in set(pool[b].tolist())


@pytest.mark.parametrize("n_blocks", [4096, 8192])
def test_hsi_pool_select_past_2048_blocks(c2, orc, n_blocks):
    """Pools larger than the pages' 2,048 blocks go through the multi-pass
    radix selection; it must give the oracle's pool (ties toward the lower
    block), including a sequence with fewer blocks than asked for."""
    B, cap = 3, 100_000
    n_vis = [100_000, 70_001, 20_000]
    g = np.random.default_rng(n_blocks)
    nblk = (cap + 7) // 8
    bs = np.full((B, nblk), -np.inf, dtype=np.float32)
    scores = []
    for b in range(B):
        s = g.standard_normal(n_vis[b]).astype(np.float32)
        s[1000:1080] = 2.5                                             # tied blocks straddling the cut
        scores.append(s.astype(np.float64))
        ob = orc.block_scores(scores[b], n_vis[b], 8)
        bs[b, :len(ob)] = ob
    p = _params(c2, candidate_topk_blocks=n_blocks)
    ws = c2.workspace(c2.OP_POOL, B, cap, p)
    pool = torch.full((B, n_blocks), -5, dtype=torch.int32, device="cuda")
    c2.hier_pool_select(torch.from_numpy(bs).cuda(), torch.tensor(n_vis, dtype=torch.int32, device="cuda"), cap,
                        p, pool, ws)
    assert c2.get_device_status() == 0
    pool = pool.cpu().numpy()
    for b in range(B):
        n = n_vis[b]
        ob = orc.block_scores(scores[b], n, 8)
        ob[(n - 1) // 8] = np.inf
        # exact block scores and ties broken toward the lower block: one right answer
        assert check_topk(pool[b], orc.hsi_pool(scores[b], n, 8, n_blocks), ob) == 0
        assert (n - 1) // 8 in set(pool[b].tolist())


def test_hsi_pool_small_context_takes_all(c2):
    B, cap = 1, 100
    bs = torch.randn(B, 13, device="cuda")
    bs[0, 13 - 1] = -1e9
    nv = torch.tensor([100], dtype=torch.int32, device="cuda")
    p = _params(c2)
    ws = c2.workspace(c2.OP_POOL, B, cap, p)
    pool = torch.empty(B, 2048, dtype=torch.int32, device="cuda")
    c2.hier_pool_select(bs, nv, cap, p, pool, ws)
    got = pool.cpu().numpy()[0]
    assert list(got[:13]) == list(range(13)) and np.all(got[13:] == -1)


def _random_pool(seed, B, n_vis, nb, n_pool_blocks):
    g = torch.Generator().manual_seed(seed)
    out = torch.full((B, n_pool_blocks), -1, dtype=torch.int32)
    for b in range(B):
        nblk = (n_vis[b] + 7) // 8
        take = min(nb, nblk)
        out[b, :take] = torch.randperm(nblk, generator=g)[:take].sort().values.to(torch.int32)
    return out


def test_reindex_over_pool(c2, orc):
    B, cap = 3, 30000
    n_vis = [30000, 9000, 1001]
    q_idx, w, k, nv = _index_case(31, B, cap, n_vis)
    p = _params(c2, candidate_topk_blocks=1024)
    pool = _random_pool(31, B, n_vis, 1000, 1024)
    ws = c2.workspace(c2.OP_INDEXER, B, cap, p)
    topk = torch.empty(B, 512, dtype=torch.int32, device="cuda")
    c2.indexer_score_topk(q_idx.cuda(), w.cuda(), k.cuda(), nv.cuda(), cap, p, topk, ws, pool_blocks=pool.cuda())
    assert c2.get_device_status() == 0
    topk = topk.cpu().numpy()
    for b in range(B):
        pos = orc.pool_positions(pool[b].numpy(), n_vis[b])
        s_pool = orc.index_scores(q_idx[b], w[b], k[b][pos])
        s_full = np.full(cap, -np.inf)
        s_full[pos] = s_pool
        check_topk(topk[b], orc.reindex_topk(q_idx[b], w[b], k[b], pool[b].numpy(), n_vis[b], 512), s_full)
        assert set(topk[b][topk[b] >= 0].tolist()) <= set(pos.tolist())


def _attn_inputs(seed, B, cap, K, W, swa_len, n_valid_idx):
    lat = synth.context_latent(seed, B, cap)
    li = synth.layer_inputs(seed, B, window=max(W, 1))
    idx = synth.random_positions(seed, B, cap, K)
    for b in range(B):
        if n_valid_idx[b] < K:
            idx[b, n_valid_idx[b]:] = -1
    return lat, li, idx, torch.tensor(swa_len, dtype=torch.int32)


def _kv_cache(c2, lat):
    B, cap = lat.shape[0], lat.shape[1]
    kv = torch.empty(B, cap, 288, dtype=torch.uint8, device="cuda")
    pos = torch.arange(cap, dtype=torch.int64, device="cuda").repeat(B)
    slot = torch.arange(B * cap, dtype=torch.int64, device="cuda")
    c2.kv_quant_write(lat.cuda().reshape(B * cap, 512), None, 1, pos, slot, kv.view(B * cap, 288))
    return kv


@pytest.mark.parametrize("B,K,W,swa_len,n_valid", [
    (2, 512, 128, [128, 77], [512, 300]),      # full top-K + SWA, ragged SWA / top-K
    (1, 100, 0, [0], [100]),                   # top-K only, K not a multiple of 128
    (1, 512, 128, [128], [0]),                 # SWA only
    (1, 256, 200, [200], [256]),               # two SWA chunks
    (2, 1024, 128, [128, 5], [1024, 700]),     # 9 chunks: merged by the separate combine kernel
])
@pytest.mark.parametrize("ak", [1, 2])            # keys split over a cluster, one CTA per token
def test_sparse_attn_reuse(c2, orc, B, K, W, swa_len, n_valid, ak):
    cap = 3000
    lat, li, idx, sl = _attn_inputs(41 + K, B, cap, K, W, swa_len, n_valid)
    p = _params(c2, index_topk=K, sliding_window=W, attn_kernel=ak)
    ws = c2.workspace(c2.OP_ATTN, B, cap, p)
    kv = _kv_cache(c2, lat)
    out = torch.empty(B, 64, 512, dtype=torch.float32, device="cuda")
    lse = torch.empty(B, 64, dtype=torch.float32, device="cuda")
    swa = li.swa[:, :W].contiguous() if W else torch.zeros(B, 1, 512, dtype=torch.uint8)
    sc = li.swa_scale[:, :W].contiguous() if W else torch.zeros(B, 1)
    c2.sparse_attn(p, li.q.cuda(), kv, idx.cuda(), swa.cuda(), sc.cuda(), sl.cuda(), out, ws, lse=lse)
    assert c2.get_device_status() == 0
    kvh = orc.kv_entries(lat.reshape(-1, 512), None, 1, np.tile(np.arange(cap), B)).reshape(B, cap, 288)
    for b in range(B):
        o, l = orc.sparse_attn(li.q[b], kvh[b], idx[b].numpy(), swa[b], sc[b], int(sl[b]))
        check_attn(out[b].cpu().numpy(), o)
        check_lse(lse[b].cpu().numpy(), l)


@pytest.mark.parametrize("K,W,ak", [(512, 128, 0), (384, 96, 0), (512, 128, 2)])
def test_sparse_attn_mixed_layout(c2, orc, K, W, ak):
    """Enough tokens that the split layout's chunks outnumber the SMs: the
    kernel takes 128 top-K entries + 32 SWA rows per chunk.  Ragged SWA
    lengths (0 .. W) and top-K fills, every token checked."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_split = -(-K // 128) + -(-W // 128)
    B = sms // n_split + 1
    cap = 1024
    rng = np.random.default_rng(K + W)
    swa_len = [int(x) for x in rng.integers(0, W + 1, B)]
    swa_len[0], swa_len[1] = W, 0
    n_valid = [int(x) for x in rng.integers(0, K + 1, B)]
    n_valid[0], n_valid[2] = K, 0
    lat, li, idx, sl = _attn_inputs(97 + K, B, cap, K, W, swa_len, n_valid)
    p = _params(c2, index_topk=K, sliding_window=W, attn_kernel=ak)
    ws = c2.workspace(c2.OP_ATTN, B, cap, p)
    kv = _kv_cache(c2, lat)
    out = torch.empty(B, 64, 512, dtype=torch.float32, device="cuda")
    lse = torch.empty(B, 64, dtype=torch.float32, device="cuda")
    swa = li.swa[:, :W].contiguous()
    sc = li.swa_scale[:, :W].contiguous()
    c2.sparse_attn(p, li.q.cuda(), kv, idx.cuda(), swa.cuda(), sc.cuda(), sl.cuda(), out, ws, lse=lse)
    assert c2.get_device_status() == 0
    kvh = orc.kv_entries(lat.reshape(-1, 512), None, 1, np.tile(np.arange(cap), B)).reshape(B, cap, 288)
    for b in range(B):
        o, l = orc.sparse_attn(li.q[b], kvh[b], idx[b].numpy(), swa[b], sc[b], int(sl[b]))
        if swa_len[b] == 0 and n_valid[b] == 0:
            assert torch.all(out[b] == 0) and torch.all(torch.isneginf(lse[b]))
            continue
        check_attn(out[b].cpu().numpy(), o)
        check_lse(lse[b].cpu().numpy(), l)


def test_sparse_attn_more_tokens_than_sms(c2, orc):
    """More tokens than SMs: one chunk per token, keys in blocks of 64 through
    two tiles, CTAs walking several tokens (item boundaries inside a CTA).
    Ragged top-K fills and SWA lengths, tokens with no key at all, every token
    checked."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, cap, K, W = sms + 8, 1024, 512, 128
    rng = np.random.default_rng(7)
    swa_len = [int(x) for x in rng.integers(0, W + 1, B)]
    n_valid = [int(x) for x in rng.integers(0, K + 1, B)]
    swa_len[0], n_valid[0] = W, K
    swa_len[1], n_valid[1] = 0, 0
    swa_len[sms], n_valid[sms] = 3, 70          # the second item of CTA 0
    lat, li, idx, sl = _attn_inputs(131, B, cap, K, W, swa_len, n_valid)
    p = _params(c2, index_topk=K, sliding_window=W)
    ws = c2.workspace(c2.OP_ATTN, B, cap, p)
    kv = _kv_cache(c2, lat)
    out = torch.empty(B, 64, 512, dtype=torch.float32, device="cuda")
    lse = torch.empty(B, 64, dtype=torch.float32, device="cuda")
    swa = li.swa[:, :W].contiguous()
    sc = li.swa_scale[:, :W].contiguous()
    c2.sparse_attn(p, li.q.cuda(), kv, idx.cuda(), swa.cuda(), sc.cuda(), sl.cuda(), out, ws, lse=lse)
    assert c2.get_device_status() == 0
    kvh = orc.kv_entries(lat.reshape(-1, 512), None, 1, np.tile(np.arange(cap), B)).reshape(B, cap, 288)
    for b in range(B):
        o, l = orc.sparse_attn(li.q[b], kvh[b], idx[b].numpy(), swa[b], sc[b], int(sl[b]))
        if swa_len[b] == 0 and n_valid[b] == 0:
            assert torch.all(out[b] == 0) and torch.all(torch.isneginf(lse[b]))
            continue
        check_attn(out[b].cpu().numpy(), o)
        check_lse(lse[b].cpu().numpy(), l)


@pytest.mark.parametrize("ak", [1, 2])
def test_sparse_attn_no_keys(c2, ak):
    B, cap, K = 1, 64, 128
    p = _params(c2, index_topk=K, sliding_window=128, attn_kernel=ak)
    ws = c2.workspace(c2.OP_ATTN, B, cap, p)
    kv = torch.zeros(B, cap, 288, dtype=torch.uint8, device="cuda")
    idx = torch.full((B, K), -1, dtype=torch.int32, device="cuda")
    swa = torch.zeros(B, 128, 512, dtype=torch.uint8, device="cuda")
    sc = torch.ones(B, 128, device="cuda")
    sl = torch.zeros(B, dtype=torch.int32, device="cuda")
    q = torch.randn(B, 64, 512, device="cuda").to(torch.bfloat16)
    out = torch.full((B, 64, 512), 7.0, device="cuda")
    lse = torch.zeros(B, 64, device="cuda")
    c2.sparse_attn(p, q, kv, idx, swa, sc, sl, out, ws, lse=lse)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_full_decode_chain_c0(c2, orc):
    """Config 0: 1 sequence, N = 4096, Full layer with HSI, then Reuse with the
    same query and SWA reproduces the Full output exactly."""
    cfg = synth.CONFIGS["decode_1x4k"]
    B, N = cfg.batch, cfg.n_ctx
    lat = synth.context_latent(0, B, N)
    k = synth.indexer_keys(0, B, N)
    li = synth.layer_inputs(0, B)
    kv = _kv_cache(c2, lat)
    p = _params(c2)
    ws = c2.workspace(c2.OP_DECODE, B, N, p)
    nv = torch.full((B,), N, dtype=torch.int32, device="cuda")
    topk = torch.empty(B, 512, dtype=torch.int32, device="cuda")
    pool = torch.empty(B, 2048, dtype=torch.int32, device="cuda")
    out = torch.empty(B, 64, 512, device="cuda")
    lse = torch.empty(B, 64, device="cuda")
    args = dict(q_idx=li.q_idx.cuda(), w=li.w.cuda(), k_idx=k.cuda(), pool_blocks=pool, lse=lse)
    c2.sparse_decode("full", p, li.q.cuda(), kv, nv, N, li.swa.cuda(), li.swa_scale.cuda(), li.swa_len.cuda(),
                     topk, out, ws, **args)
    assert c2.get_device_status() == 0
    s = orc.index_scores(li.q_idx[0], li.w[0], k[0])
    o_idx = orc.topk(s, 512)
    check_topk(topk[0].cpu().numpy(), o_idx, s)
    check_topk(pool[0].cpu().numpy(), orc.hsi_pool(s, N, 8, 2048),
               np.where(np.arange(N // 8) == (N - 1) // 8, np.inf, orc.block_scores(s, N, 8)))
    kvh = orc.kv_entries(lat[0], None, 1, np.arange(N))
    # the readout is checked on the GPU's own selection (it may differ from the
    # oracle's only inside the tie band, which check_topk bounds above)
    o, l = orc.sparse_attn(li.q[0], kvh, topk[0].cpu().numpy(), li.swa[0], li.swa_scale[0], 128)
    check_attn(out[0].cpu().numpy(), o)
    check_lse(lse[0].cpu().numpy(), l)
    out_r = torch.empty_like(out)
    c2.sparse_decode("reuse", p, li.q.cuda(), kv, nv, N, li.swa.cuda(), li.swa_scale.cuda(), li.swa_len.cuda(),
                     topk, out_r, ws)
    assert torch.equal(out, out_r)
    # Reindex over a pool covering every block reproduces the Full top-K
    p2 = _params(c2, candidate_topk_blocks=512)
    allb = torch.arange(512, dtype=torch.int32, device="cuda").unsqueeze(0)
    topk_r = torch.empty_like(topk)
    ws2 = c2.workspace(c2.OP_DECODE, B, N, p2)
    c2.sparse_decode("reindex", p2, li.q.cuda(), kv, nv, N, li.swa.cuda(), li.swa_scale.cuda(),
                     li.swa_len.cuda(), topk_r, out_r, ws2, q_idx=li.q_idx.cuda(), w=li.w.cuda(), k_idx=k.cuda(),
                     pool_blocks=allb)
    assert torch.equal(topk, topk_r)
    assert torch.equal(out, out_r)


def test_topk_many_ties_across_cluster(c2, orc):
    """Scores drawn from four values over a long row: the selection must take
    the lowest indices of the tied value, across the CTAs of the cluster."""
    B, cap, K = 2, 200_000, 512
    q_idx = torch.zeros(B, 32, 128, dtype=torch.bfloat16)
    q_idx[:, :, 0] = 1.0
    w = synth.uniform((B, 32), 5, 4)
    g = torch.Generator().manual_seed(9)
    k = torch.zeros(B, cap, 128, dtype=torch.bfloat16)
    k[:, :, 0] = torch.randint(0, 4, (B, cap), generator=g).to(torch.bfloat16)
    k[0, :, 0] = torch.where(torch.arange(cap) % 1000 == 0, 3.0, 1.0).to(torch.bfloat16)   # 200 threes
    nv = torch.tensor([cap, 150_001], dtype=torch.int32)
    p = _params(c2, index_topk=K)
    ws = c2.workspace(c2.OP_INDEXER, B, cap, p)
    topk = torch.empty(B, K, dtype=torch.int32, device="cuda")
    c2.indexer_score_topk(q_idx.cuda(), w.cuda(), k.cuda(), nv.cuda(), cap, p, topk, ws)
    assert c2.get_device_status() == 0
    topk = topk.cpu().numpy()
    for b in range(B):
        s = orc.index_scores(q_idx[b], w[b], k[b, :int(nv[b])])
        assert np.array_equal(topk[b], orc.topk(s, K))


def test_topk_long_row_1m(c2, orc):
    """One 1M-position row (the longest context): the cluster spans 16 CTAs."""
    B, cap, K = 1, 1 << 20, 512
    q_idx, w, k, nv = _index_case(77, B, cap, [cap - 3])
    p = _params(c2, index_topk=K)
    ws = c2.workspace(c2.OP_INDEXER, B, cap, p)
    topk = torch.empty(B, K, dtype=torch.int32, device="cuda")
    c2.indexer_score_topk(q_idx.cuda(), w.cuda(), k.cuda(), nv.cuda(), cap, p, topk, ws)
    assert c2.get_device_status() == 0
    s = orc.index_scores(q_idx[0], w[0], k[0, :cap - 3])
    check_topk(topk[0].cpu().numpy(), orc.topk(s, K), s, n_valid=cap - 3)
