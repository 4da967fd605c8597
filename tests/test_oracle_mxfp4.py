"""Pins for the oracle's MXFP4 indexer codec (E2M1 elements, one UE8M0 power-
of-two scale per 32; "DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache
Compression" section 2.4.4: FP4 indexer Q and K; section 3.1: a 128-d MXFP4
indexer-K entry is 68 B).  Checked against the OCP Microscaling definitions
(the scaled block maximum lies in [4, 8) -- the E2M1 top binade -- and the
elements round to the nearest E2M1 value, ties to even, saturating at 6), a
brute-force nearest search, exact round trips and the bf16 indexer path."""
import json
import math
import os

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
FACTS = json.load(open(os.path.join(HERE, "golden", "pages_facts.json")))


def e2m1_from_bits(c):
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    v = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
    return -v if s else v


def _codes(c):
    """[n, 64] bytes -> [n, 128] codes (element 2j in the low nibble of byte j)."""
    out = np.empty((c.shape[0], 128), np.uint8)
    out[:, 0::2] = c & 15
    out[:, 1::2] = c >> 4
    return out


def _nearest(t):
    """Nearest E2M1 code of a scaled value: ties to the even code, saturate."""
    best, bd = None, None
    for c in range(8):
        d = abs(abs(t) - e2m1_from_bits(c))
        if best is None or d < bd or (d == bd and c % 2 == 0):
            best, bd = c, d
    return best | (8 if np.signbit(t) else 0)


def test_entry_is_68_bytes(orc):
    codes, scales = orc.mxfp4_quantise(np.ones((1, 128), np.float32))
    assert codes.nbytes + scales.nbytes == 68
    f = FACTS["main_attention_settings"]
    assert f["indexer_head_dim"] // 2 + f["indexer_head_dim"] // 32 == 68


def test_scale_puts_block_max_in_top_binade(orc):
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((200, 128)) * np.exp(rng.uniform(-20, 20, (200, 1)))).astype(np.float32)
    _, scales = orc.mxfp4_quantise(x)
    for r in range(200):
        for b in range(4):
            amax = np.abs(x[r, 32 * b:32 * b + 32]).astype(np.float64).max()
            e = int(scales[r, b]) - 127
            assert 4.0 * 2.0 ** e <= amax < 8.0 * 2.0 ** e


def test_elements_are_nearest_e2m1(orc):
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((40, 128)) * 3).astype(np.float32)
    x[0, :32] = np.array([4.5, 5.0, 5.5, 7.9, -7.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5] + [0.1] * 21, np.float32)
    codes, scales = orc.mxfp4_quantise(x)
    cd = _codes(codes)
    for r in range(40):
        for d in range(128):
            t = float(x[r, d]) / 2.0 ** (int(scales[r, d // 32]) - 127)
            assert cd[r, d] == _nearest(t), (r, d, t)


def test_representable_blocks_round_trip(orc):
    """code x 2^E with a block maximum of 4 or 6 (times 2^E) returns the same
    codes and exponent, for every exponent a float32 block can carry."""
    rng = np.random.default_rng(2)
    for e in list(range(-126, 126, 7)) + [-126, 125]:
        c = rng.integers(0, 16, size=128).astype(np.uint8)
        for b in range(4):
            c[32 * b] = (c[32 * b] & 8) | (6 + (b & 1))      # |code value| 4 or 6 leads each block
        x = np.array([e2m1_from_bits(int(v)) * 2.0 ** e for v in c], np.float64)
        xf = x.astype(np.float32)
        assert np.array_equal(xf.astype(np.float64), x)
        codes, scales = orc.mxfp4_quantise(xf[None])
        got = _codes(codes)[0]
        # +0 / -0 are different codes with the same value
        assert np.array_equal(got & 7, c & 7) and np.array_equal(got[(c & 7) != 0] >> 3, c[(c & 7) != 0] >> 3)
        assert np.all(scales == e + 127)
        assert np.array_equal(orc.mxfp4_dequant(codes, scales)[0], x)


def test_zero_block_and_signs(orc):
    x = np.zeros((1, 128), np.float32)
    x[0, 40] = -3.0
    codes, scales = orc.mxfp4_quantise(x)
    assert scales[0, 0] == 0 and np.all(codes[0, :16] == 0)    # all-zero block: E = -127
    neg, _ = orc.mxfp4_quantise(-x)
    assert np.array_equal(_codes(neg)[0, 32:64] & 7, _codes(codes)[0, 32:64] & 7)
    assert orc.mxfp4_dequant(codes, scales)[0, 40] == -3.0


def test_bf16_rows_match_float_rows(orc):
    x = torch.randn(16, 128).to(torch.bfloat16)
    a = orc.mxfp4_quantise(x)
    b = orc.mxfp4_quantise(x.float().numpy())
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_index_scores_on_representable_operands_equal_bf16_path(orc):
    """When q and k are already MXFP4 values, quantising changes nothing and
    the score is the bf16 indexer's score of the same values."""
    rng = np.random.default_rng(3)

    def representable(n, e):
        c = rng.integers(0, 16, size=(n, 128))
        c[:, ::32] = 7                                        # block max 6 x 2^e
        return np.vectorize(lambda v: e2m1_from_bits(int(v)))(c) * 2.0 ** e

    q = torch.from_numpy(representable(32, -4).astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(representable(50, -1).astype(np.float32)).to(torch.bfloat16)
    w = rng.uniform(0, 1, 32).astype(np.float32)
    kc, ks = orc.mxfp4_quantise(k)
    assert np.allclose(orc.index_scores_mxfp4(q, w, kc, ks), orc.index_scores(q, w, k), rtol=0, atol=0)


def test_index_scores_mxfp4_matches_einsum_of_dequantised(orc):
    rng = np.random.default_rng(4)
    q = torch.from_numpy((rng.standard_normal((32, 128)) / math.sqrt(128)).astype(np.float32)).to(torch.bfloat16)
    k = torch.from_numpy(rng.standard_normal((300, 128)).astype(np.float32)).to(torch.bfloat16)
    w = rng.uniform(0, 1, 32).astype(np.float32)
    kc, ks = orc.mxfp4_quantise(k)
    qd = orc.mxfp4_dequant(*orc.mxfp4_quantise(q))
    kd = orc.mxfp4_dequant(kc, ks)
    ref = (np.maximum(np.einsum("hd,nd->nh", qd, kd), 0.0) * w.astype(np.float64)).sum(1)
    assert np.allclose(orc.index_scores_mxfp4(q, w, kc, ks), ref, rtol=1e-12, atol=1e-12)
