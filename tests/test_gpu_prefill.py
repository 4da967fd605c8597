"""GPU parity of csa2_prefill_chunk (chunked prefill at m = 2) against the
oracle, on sampled chunk tokens of a scaled-down workload (4,096-token context
+ 1,024-token chunk, 2 sequences) and on the first chunk of a sequence (short
windows, fewer visible entries than index_topk).  Every token's selection is
also checked for validity; sampled tokens are recomputed by the oracle from
the same inputs: index scores over the visible entries, top-K, readout with
the token's own causal SWA window."""
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


def _prefill_case(c2, seed, B, ctx_tokens, T, m=2, W=128, K=512):
    E = (ctx_tokens + T) // m                     # entries after the chunk is written
    lat = synth.context_latent(seed, B, E, m=m)   # [B, E, 2, 512]
    z = synth.compression_logits(seed, B, E, m=m)
    kv = torch.empty(B, E, 288, dtype=torch.uint8, device="cuda")
    pos = (torch.arange(E, dtype=torch.int64) * m + m - 1).repeat(B).cuda()
    slot = torch.arange(B * E, dtype=torch.int64, device="cuda")
    c2.kv_quant_write(lat.cuda().reshape(B * E, m, 512), z.cuda().reshape(B * E, m, 512), m, pos, slot,
                      kv.view(B * E, 288))
    k_idx = synth.indexer_keys(seed, B, E)
    q = synth.normal((B, T, 64, 512), seed, 2)
    q_idx = synth.normal((B, T, 32, 128), seed, 3, std=1 / math.sqrt(128))
    w = synth.uniform((B, T, 32), seed, 4)
    first_pos = ctx_tokens
    swa_first = max(first_pos - W + 1, 0)
    rows = first_pos + T - swa_first
    swa, swa_scale = synth.fp8_rows(synth.normal((B, rows, 512), seed, 5, dtype=torch.float32))
    p = c2.Params.make(index_topk=K, sliding_window=W)
    ws = c2.workspace(c2.OP_PREFILL, B, E, p)
    topk = torch.full((B, T, K), -7, dtype=torch.int32, device="cuda")
    out = torch.empty(B, T, 64, 512, device="cuda")
    lse = torch.empty(B, T, 64, device="cuda")
    c2.prefill_chunk(p, q.cuda(), q_idx.cuda(), w.cuda(), kv, k_idx.cuda(), first_pos, m, swa.cuda(),
                     swa_scale.cuda(), swa_first, topk, out, ws, lse=lse)
    assert c2.get_device_status() == 0
    return dict(lat=lat, z=z, k_idx=k_idx, q=q, q_idx=q_idx, w=w, swa=swa, swa_scale=swa_scale,
                swa_first=swa_first, first_pos=first_pos, topk=topk.cpu().numpy(), out=out.cpu().numpy(),
                lse=lse.cpu().numpy(), E=E, m=m, W=W, K=K)


def _check_tokens(orc, d, samples):
    m, W, K = d["m"], d["W"], d["K"]
    kvh = {}
    for b, i in samples:
        pos = d["first_pos"] + i
        nvis = (pos + 1) // m
        s = orc.index_scores(d["q_idx"][b, i], d["w"][b, i], d["k_idx"][b, :nvis])
        check_topk(d["topk"][b, i], orc.topk(s, K), s, n_valid=nvis)
        # every sampled token's readout is checked on the GPU's own selection
        # (it may differ from the oracle's only inside the tie band above)
        if b not in kvh:
            kvh[b] = orc.kv_entries(d["lat"][b], d["z"][b], m, np.arange(d["E"]) * m + m - 1)
        start = max(pos - W + 1, 0)
        r0, r1 = start - d["swa_first"], pos - d["swa_first"] + 1
        o, l = orc.sparse_attn(d["q"][b, i], kvh[b], d["topk"][b, i], d["swa"][b, r0:r1], d["swa_scale"][b, r0:r1],
                               r1 - r0)
        check_attn(d["out"][b, i], o)
        check_lse(d["lse"][b, i], l)


def _check_all_valid(d):
    m = d["m"]
    T = d["topk"].shape[1]
    for b in range(d["topk"].shape[0]):
        for i in range(T):
            nvis = (d["first_pos"] + i + 1) // m
            g = d["topk"][b, i]
            v = g[g >= 0]
            assert len(v) == min(d["K"], nvis) and np.all(g[len(v):] == -1)
            assert np.all(np.diff(v) > 0) and (len(v) == 0 or v[-1] < nvis)


def test_prefill_chunk_sampled_tokens(c2, orc):
    d = _prefill_case(c2, 401, 2, 4096, 1024)
    _check_all_valid(d)
    rng = np.random.default_rng(4)
    samples = [(b, i) for b in range(2) for i in (0, 1, 2, 511, 512, 1023)]
    samples += [(int(rng.integers(0, 2)), int(rng.integers(0, 1024))) for _ in range(6)]
    _check_tokens(orc, d, samples)


def test_prefill_first_chunk_of_sequence(c2, orc):
    """Positions from 0: short SWA windows and fewer visible entries than K."""
    d = _prefill_case(c2, 402, 1, 0, 1024 + 256)
    _check_all_valid(d)
    _check_tokens(orc, d, [(0, i) for i in (0, 1, 2, 7, 126, 127, 128, 1023, 1024, 1279)])


def test_prefill_full_context_block(c2, orc):
    """A 131,072-token context and one 1,024-token block: the per-block launch
    configuration of the 2 x 131,072 + 16,384 workload (1,024 top-K rows of
    ~65.5K entries -- one CTA per row, several rounds per slice)."""
    d = _prefill_case(c2, 403, 1, 131072, 1024)
    _check_all_valid(d)
    _check_tokens(orc, d, [(0, i) for i in (0, 1, 333, 512, 1022, 1023)])
