"""Pins for the oracle's sparse-attention readout and the Full/Reindex/Reuse
modes.

Readout (en.mycoding.id sections 3.3.1-3.3.2; Architecture notes section 2):
one softmax over the selected main-KV entries and the SWA window, key = value =
the latent, so the output is a convex combination of the selected vectors.
Checks: dense softmax attention from torch when every position is selected
and there is no SWA; weights non-negative and summing to one; outputs inside
the per-channel hull; identical keys reproduce the key; order does not matter;
Reuse with the same query and SWA reproduces Full; Reindex with a pool that
covers everything reproduces Full; the schedule's refresh counts."""
import json
import math
import os

import numpy as np
import torch

import synth

HERE = os.path.dirname(os.path.abspath(__file__))
FACTS = json.load(open(os.path.join(HERE, "golden", "pages_facts.json")))


def _setup(seed=0, n=64, swa_len=16):
    li = synth.layer_inputs(seed, 1, window=max(swa_len, 1))
    lat = synth.context_latent(seed, 1, n)[0]
    kv = None
    return li, lat


def _kv(orc, lat):
    return orc.kv_entries(lat, None, 1, np.arange(lat.shape[0]))


def test_dense_case_equals_sdpa(orc):
    li, lat = _setup(0, 96)
    kv = _kv(orc, lat)
    idx = np.arange(96)
    out, lse = orc.sparse_attn(li.q[0], kv, idx, li.swa[0], li.swa_scale[0], 0)
    keys = torch.from_numpy(np.stack([orc.fp4_dequant(e) for e in kv]))       # [96, 512]
    q = li.q[0].double()
    ref = torch.nn.functional.scaled_dot_product_attention(q[None], keys[None], keys[None])[0]
    assert np.allclose(out, ref.numpy(), rtol=1e-10, atol=1e-12)
    ref_lse = torch.logsumexp(q @ keys.T / math.sqrt(512), dim=-1)
    assert np.allclose(lse, ref_lse.numpy(), rtol=1e-12)


def test_swa_only_equals_sdpa(orc):
    li, lat = _setup(1, 8, 32)
    idx = -np.ones(4, np.int64)
    out, _ = orc.sparse_attn(li.q[0], _kv(orc, lat), idx, li.swa[0], li.swa_scale[0], 32)
    keys = li.swa[0].view(torch.float8_e4m3fn).double() * li.swa_scale[0].double()[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(li.q[0].double()[None], keys[None], keys[None])[0]
    assert np.allclose(out, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_weights_simplex_and_convex_hull(orc):
    li, lat = _setup(2, 200, 24)
    kv = _kv(orc, lat)
    idx = np.array(sorted(np.random.default_rng(2).choice(200, 40, replace=False)) + [-1] * 8)
    out, _, wts = orc.sparse_attn(li.q[0], kv, idx, li.swa[0], li.swa_scale[0], 24, want_weights=True)
    assert np.all(wts >= 0)
    assert np.allclose(wts.sum(1), 1.0, atol=1e-12)
    assert np.all(wts[:, 40:48] == 0)
    sel = [orc.fp4_dequant(kv[i]) for i in idx if i >= 0]
    sel += list(li.swa[0][:24].view(torch.float8_e4m3fn).double().numpy() * li.swa_scale[0][:24].double().numpy()[:, None])
    sel = np.stack(sel)
    lo, hi = sel.min(0), sel.max(0)
    assert np.all(out >= lo - 1e-12) and np.all(out <= hi + 1e-12)


def test_identical_keys_reproduce_key(orc):
    li, lat = _setup(3, 4)
    kv = _kv(orc, lat)
    idx = np.zeros(9, np.int64)          # the same entry nine times
    out, _ = orc.sparse_attn(li.q[0], kv, idx, li.swa[0], li.swa_scale[0], 0)
    assert np.allclose(out, np.tile(orc.fp4_dequant(kv[0]), (64, 1)), rtol=1e-14)


def test_order_invariance(orc):
    li, lat = _setup(4, 120, 20)
    kv = _kv(orc, lat)
    rng = np.random.default_rng(4)
    idx = rng.choice(120, 30, replace=False)
    out1, lse1 = orc.sparse_attn(li.q[0], kv, idx, li.swa[0], li.swa_scale[0], 20)
    perm = rng.permutation(20)
    out2, lse2 = orc.sparse_attn(li.q[0], kv, idx[::-1].copy(), li.swa[0][perm], li.swa_scale[0][perm], 20)
    assert np.allclose(out1, out2, rtol=1e-12, atol=1e-14) and np.allclose(lse1, lse2, rtol=1e-13)


def _full_layer(orc, li, lat, kidx, n_vis, k=64):
    kv = _kv(orc, lat)
    s = orc.index_scores(li.q_idx[0], li.w[0], kidx[0][:n_vis])
    idx = orc.topk(s, k)
    out, lse = orc.sparse_attn(li.q[0], kv, idx, li.swa[0], li.swa_scale[0], int(li.swa_len[0]))
    return idx, out, lse, s


def test_reuse_with_same_query_equals_full(orc):
    n = 300
    li = synth.layer_inputs(5, 1, window=32)
    lat = synth.context_latent(5, 1, n)[0]
    kidx = synth.indexer_keys(5, 1, n)
    idx, out, lse, _ = _full_layer(orc, li, lat, kidx, n)
    # Reuse: no indexing, the latest indices, the same query and SWA
    out_r, lse_r = orc.sparse_attn(li.q[0], _kv(orc, lat), idx, li.swa[0], li.swa_scale[0], 32)
    assert np.array_equal(out, out_r) and np.array_equal(lse, lse_r)


def test_reindex_with_full_pool_equals_full(orc):
    n = 8 * 30 + 1
    li = synth.layer_inputs(6, 1, window=16)
    lat = synth.context_latent(6, 1, n)[0]
    kidx = synth.indexer_keys(6, 1, n)
    idx, out, _, s = _full_layer(orc, li, lat, kidx, n)
    pool = orc.hsi_pool(s, n, 8, 2048)
    idx_r = orc.reindex_topk(li.q_idx[0], li.w[0], kidx[0], pool, n, 64)
    assert np.array_equal(idx, idx_r)


def test_schedule_refresh_counts():
    """content x4 (Full layers), address x8 (Full + Reindex), query x40 (every
    layer) over the 40-layer model, from the encoder and decoder schedules."""
    L = FACTS["model_layers"]
    enc = ["swa"] * L["encoder_swa_only_layers"] + L["encoder_group"] * L["encoder_groups"]
    dec = synth.decoder_layer_modes(L["decoder_groups"], len(L["decoder_first_group"]))
    assert dec[:4] == L["decoder_first_group"] and dec[4:8] == L["decoder_later_group"]
    assert len(enc) == L["encoder_layers"] and len(dec) == L["decoder_layers"]
    layers = enc + dec
    rc = FACTS["refresh_timescales"]
    assert sum(m == "full" for m in layers) == rc["content"]
    assert sum(m in ("full", "reindex") for m in layers) == rc["address"]
    assert len(layers) == rc["query"]
    assert [20 + i for i, m in enumerate(dec) if m == "reindex"] == L["decoder_reindex_layers"]
    assert dec.index("full") + 20 == L["decoder_full_layer"]
