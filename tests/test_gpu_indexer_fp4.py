"""GPU parity of the MXFP4 indexer ("DeepSeek-v4.1 Flash: Pushing the Limits of
KV Cache Compression", section 2.4.4: FP4 indexer Q and K; section 3.1: 68 B per
128-d entry): the indexer-K write is bit-exact against the oracle's MXFP4
codec, and the Full / Reindex sweeps + top-K match the oracle's scores of the
dequantised operands (fp64) within the top-K rule of the bf16 indexer."""
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
    return c


def _fp4_cache(c2, k):
    """k bf16 [B, cap, 128] -> the MXFP4 cache of B * cap rows, row b * cap + n."""
    B, cap = k.shape[0], k.shape[1]
    cache = c2.indexer_k_fp4_cache(B * cap)
    c2.indexer_k_quant(k.reshape(-1, 128).cuda(), torch.arange(B * cap, device="cuda"), cache)
    return cache


def _oracle_scores(orc, q_idx, w, k):
    codes, scales = orc.mxfp4_quantise(k)
    return orc.index_scores_mxfp4(q_idx, w, codes, scales)


def _hard_keys(n, seed):
    """Rows whose blocks span a wide range of scales, with zero blocks, bf16
    subnormals, the bf16 extremes, exact E2M1 midpoints (ties) and signed
    zeros."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, 128, generator=g, dtype=torch.float64)
    x *= torch.exp2(torch.randint(-40, 40, (n, 4), generator=g).double()).repeat_interleave(32, 1)
    x[0] = 0.0
    x[1, :32] = 0.0
    x[1, 32:64] = -0.0
    x[2, :32] = 1e-39                                      # bf16 subnormal block
    x[2, 32:64] = -2.0 ** -126
    x[3, :32] = 3.3e38
    x[3, 32:64] = -3.3e38
    mids = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 6.5, -0.25, -5.0, 0.1], dtype=torch.float64)
    x[4, :12] = mids
    x[4, 12] = 6.0                                         # block max 7 -> scale 2^0: 7, 6.5 saturate to 6
    x[4, 32:44] = mids * 2.0 ** 20
    x[4, 44] = 6.0 * 2.0 ** 20
    x[5, 64:96] = -1e-3
    return x.to(torch.bfloat16)


def test_indexer_k_quant_bit_exact(c2, orc):
    n, rows = 1000, 1024
    k = torch.cat([_hard_keys(200, 1), synth.indexer_keys(2, 1, 800)[0]])
    slot = torch.randperm(rows, generator=torch.Generator().manual_seed(3))[:n]
    cache = c2.indexer_k_fp4_cache(rows)
    c2.indexer_k_quant(k.cuda(), slot.cuda(), cache)
    assert c2.get_device_status() == 0
    codes, scales = (t.cpu().numpy() for t in c2.indexer_k_fp4_planes(cache))
    oc, os_ = orc.mxfp4_quantise(k)
    s = slot.numpy()
    assert np.array_equal(codes[s], oc)
    assert np.array_equal(scales[s], os_)
    untouched = np.setdiff1d(np.arange(rows), s)
    assert not codes[untouched].any() and not scales[untouched].any()


def test_indexer_k_quant_skips_bad_slots(c2, orc):
    k = synth.indexer_keys(4, 1, 8)[0]
    slot = torch.tensor([0, 1, -1, 3, 8, 5, 6, 7])
    cache = c2.indexer_k_fp4_cache(8)
    c2.indexer_k_quant(k.cuda(), slot.cuda(), cache)
    assert c2.get_device_status() == 0x2
    codes, scales = (t.cpu().numpy() for t in c2.indexer_k_fp4_planes(cache))
    oc, os_ = orc.mxfp4_quantise(k)
    for i, r in enumerate(slot.tolist()):
        if 0 <= r < 8:
            assert np.array_equal(codes[r], oc[i]) and np.array_equal(scales[r], os_[i])
    assert not codes[[2, 4]].any() and not scales[[2, 4]].any()


def _index_case(seed, B, cap, n_vis, wide=False):
    q_idx = synth.normal((B, 32, 128), seed, 3, std=1 / math.sqrt(128))
    w = synth.uniform((B, 32), seed, 4)
    k = synth.indexer_keys(seed, B, cap)
    if wide:
        # rows (keys and query heads) scaled over 2^-30 .. 2^30 and their
        # blocks spread over a further 2^-10 .. 1: the sweep's 8-bit operands
        # hold code x 2^(E - Emax) exactly for blocks within 2^15 of their
        # row's largest, so these scores are still the exact ones
        g = torch.Generator().manual_seed(seed)

        def spread(shape):
            e = torch.randint(-30, 31, shape[:-1] + (1,), generator=g) + torch.randint(-10, 1, shape, generator=g)
            return torch.exp2(e.float()).repeat_interleave(32, -1)
        k = (k.float() * spread((B, cap, 4))).to(torch.bfloat16)
        q_idx = (q_idx.float() * spread((B, 32, 4))).to(torch.bfloat16)
    return q_idx, w, k, torch.tensor(n_vis, dtype=torch.int32)


@pytest.mark.parametrize("B,cap,n_vis,K,wide", [(1, 4096, [4096], 512, False), (3, 3000, [3000, 1000, 77], 512, False),
                                                (2, 700, [700, 333], 1024, False), (1, 128, [5], 16, False),
                                                (2, 2052, [2052, 1500], 512, True)])
def test_fp4_full_indexer_topk_and_block_scores(c2, orc, B, cap, n_vis, K, wide):
    q_idx, w, k, nv = _index_case(40 + B, B, cap, n_vis, wide)
    p = c2.Params.make(index_topk=K, indexer_fp4=1)
    ws = c2.workspace(c2.OP_INDEXER, B, cap, p)
    cache = _fp4_cache(c2, k)
    topk = torch.full((B, K), -7, dtype=torch.int32, device="cuda")
    nblk = (cap + 7) // 8
    bs = torch.empty(B, nblk, dtype=torch.float32, device="cuda")
    c2.indexer_score_topk(q_idx.cuda(), w.cuda(), cache, nv.cuda(), cap, p, topk, ws, block_scores=bs)
    assert c2.get_device_status() == 0
    topk, bs = topk.cpu().numpy(), bs.cpu().numpy()
    for b in range(B):
        s = _oracle_scores(orc, q_idx[b], w[b], k[b, :n_vis[b]])
        check_topk(topk[b], orc.topk(s, K), s, n_valid=n_vis[b])
        ob = orc.block_scores(s, n_vis[b], 8)
        nb = len(ob)
        assert np.allclose(bs[b, :nb], ob, rtol=1e-4, atol=1e-4 * np.abs(ob).max())
        assert np.all(np.isneginf(bs[b, nb:]))


def test_fp4_block_sum_reduction_and_pool(c2, orc):
    """block_reduce = 1 with the MXFP4 sweep: block scores are sums of the 8
    positions' MXFP4 scores, and the HSI pool follows the oracle's sum
    reduction."""
    B, cap = 2, 5000
    n_vis = [5000, 2345]
    q_idx, w, k, nv = _index_case(61, B, cap, n_vis)
    p = c2.Params.make(candidate_topk_blocks=256, block_reduce=1, indexer_fp4=1)
    ws = c2.workspace(c2.OP_DECODE, B, cap, p)
    nblk = (cap + 7) // 8
    bs = torch.empty(B, nblk, dtype=torch.float32, device="cuda")
    topk = torch.empty(B, 512, dtype=torch.int32, device="cuda")
    c2.indexer_score_topk(q_idx.cuda(), w.cuda(), _fp4_cache(c2, k), nv.cuda(), cap, p, topk, ws, block_scores=bs)
    pool = torch.empty(B, 256, dtype=torch.int32, device="cuda")
    c2.hier_pool_select(bs, nv.cuda(), cap, p, pool, ws)
    assert c2.get_device_status() == 0
    bs, pool = bs.cpu().numpy(), pool.cpu().numpy()
    for b in range(B):
        n = n_vis[b]
        s = _oracle_scores(orc, q_idx[b], w[b], k[b, :n])
        ob = orc.block_scores(s, n, 8, reduce_sum=True)
        nb = len(ob)
        assert np.allclose(bs[b, :nb], ob, rtol=1e-4, atol=1e-4 * np.abs(ob).max())
        assert np.all(np.isneginf(bs[b, nb:]))
        ob[(n - 1) // 8] = np.inf
        check_topk(pool[b], orc.hsi_pool(s, n, 8, 256, reduce_sum=True), ob)
        assert (n - 1) // 8 in set(pool[b].tolist())


def test_fp4_ranking_follows_the_quantised_keys(c2, orc):
    """The FP4 path scores the quantised operands: keys whose dim-0 values
    2.75, 2.90625, 3.1875 all round to E2M1 3 (and 3.625 to 4) tie in MXFP4,
    so the top-2 is {3, 0} (ties toward the lower position) where bf16 scores
    give {3, 2}."""
    B, cap, K = 1, 1024, 2
    q_idx = torch.zeros(B, 32, 128, dtype=torch.bfloat16)
    q_idx[:, :, 0] = 1.0
    q_idx[:, :, 1] = 6.0                                   # block max 6: scale 2^0, exact
    w = torch.ones(B, 32)
    k = torch.zeros(B, cap, 128, dtype=torch.bfloat16)
    k[0, :, 1] = 4.0                                       # block max 4: scale 2^0
    k[0, :4, 0] = torch.tensor([2.75, 2.90625, 3.1875, 3.625]).to(torch.bfloat16)
    nv = torch.tensor([cap], dtype=torch.int32)
    p = c2.Params.make(index_topk=K, indexer_fp4=1)
    ws = c2.workspace(c2.OP_INDEXER, B, cap, p)
    topk = torch.empty(B, K, dtype=torch.int32, device="cuda")
    c2.indexer_score_topk(q_idx.cuda(), w.cuda(), _fp4_cache(c2, k), nv.cuda(), cap, p, topk, ws)
    assert c2.get_device_status() == 0
    s = _oracle_scores(orc, q_idx[0], w[0], k[0])
    assert list(orc.topk(s, K)) == [0, 3]
    assert list(orc.topk(orc.index_scores(q_idx[0], w[0], k[0]), K)) == [2, 3]
    assert topk[0].cpu().tolist() == [0, 3]


def _random_pool(seed, B, n_vis, nb, n_pool_blocks):
    g = torch.Generator().manual_seed(seed)
    out = torch.full((B, n_pool_blocks), -1, dtype=torch.int32)
    for b in range(B):
        nblk = (n_vis[b] + 7) // 8
        take = min(nb, nblk)
        out[b, :take] = torch.randperm(nblk, generator=g)[:take].sort().values.to(torch.int32)
    return out


@pytest.mark.parametrize("B,cap,n_vis", [(3, 30000, [30000, 9000, 1001]), (2, 1004, [1004, 1004])])
def test_fp4_reindex_over_pool(c2, orc, B, cap, n_vis):
    """Reindex over a pool; cap = 1004 puts the last sequence's last block
    past the end of the cache (its scale copy is cut to the rows that exist)."""
    q_idx, w, k, nv = _index_case(51, B, cap, n_vis)
    p = c2.Params.make(candidate_topk_blocks=1024, indexer_fp4=1)
    pool = _random_pool(51, B, n_vis, 1000, 1024)
    ws = c2.workspace(c2.OP_INDEXER, B, cap, p)
    topk = torch.empty(B, 512, dtype=torch.int32, device="cuda")
    c2.indexer_score_topk(q_idx.cuda(), w.cuda(), _fp4_cache(c2, k), nv.cuda(), cap, p, topk, ws,
                          pool_blocks=pool.cuda())
    assert c2.get_device_status() == 0
    topk = topk.cpu().numpy()
    for b in range(B):
        pos = orc.pool_positions(pool[b].numpy(), n_vis[b])
        s_pool = _oracle_scores(orc, q_idx[b], w[b], k[b][pos])
        sel = orc.topk(s_pool, 512)
        o_idx = np.where(sel >= 0, pos[np.clip(sel, 0, None)], -1)
        s_full = np.full(cap, -np.inf)
        s_full[pos] = s_pool
        check_topk(topk[b], o_idx, s_full)
        assert set(topk[b][topk[b] >= 0].tolist()) <= set(pos.tolist())


def test_fp4_decode_chain(c2, orc):
    """A Full decode layer with the MXFP4 indexer: its top-K follows the
    MXFP4 oracle, and a Reindex over a pool of every block reproduces it."""
    cfg = synth.CONFIGS["decode_1x4k"]
    B, N = cfg.batch, cfg.n_ctx
    lat = synth.context_latent(0, B, N)
    k = synth.indexer_keys(0, B, N)
    li = synth.layer_inputs(0, B)
    kv = torch.empty(B, N, 288, dtype=torch.uint8, device="cuda")
    c2.kv_quant_write(lat.cuda().reshape(B * N, 512), None, 1, torch.arange(N, device="cuda").repeat(B),
                      torch.arange(B * N, device="cuda"), kv.view(B * N, 288))
    p = c2.Params.make(indexer_fp4=1)
    ws = c2.workspace(c2.OP_DECODE, B, N, p)
    nv = torch.full((B,), N, dtype=torch.int32, device="cuda")
    topk = torch.empty(B, 512, dtype=torch.int32, device="cuda")
    pool = torch.empty(B, 2048, dtype=torch.int32, device="cuda")
    out = torch.empty(B, 64, 512, device="cuda")
    cache = _fp4_cache(c2, k)
    c2.sparse_decode("full", p, li.q.cuda(), kv, nv, N, li.swa.cuda(), li.swa_scale.cuda(), li.swa_len.cuda(),
                     topk, out, ws, q_idx=li.q_idx.cuda(), w=li.w.cuda(), k_idx=cache, pool_blocks=pool)
    assert c2.get_device_status() == 0
    s = _oracle_scores(orc, li.q_idx[0], li.w[0], k[0])
    check_topk(topk[0].cpu().numpy(), orc.topk(s, 512), s)
    p2 = c2.Params.make(candidate_topk_blocks=512, indexer_fp4=1)
    allb = torch.arange(512, dtype=torch.int32, device="cuda").unsqueeze(0)
    topk_r = torch.empty_like(topk)
    out_r = torch.empty_like(out)
    ws2 = c2.workspace(c2.OP_DECODE, B, N, p2)
    c2.sparse_decode("reindex", p2, li.q.cuda(), kv, nv, N, li.swa.cuda(), li.swa_scale.cuda(),
                     li.swa_len.cuda(), topk_r, out_r, ws2, q_idx=li.q_idx.cuda(), w=li.w.cuda(), k_idx=cache,
                     pool_blocks=allb)
    assert torch.equal(topk, topk_r)
    assert torch.equal(out, out_r)
