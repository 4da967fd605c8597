"""Pins for the oracle's FP4 main-KV codec (E2M1 codes + one E4M3 scale per 16
channels, no global scale; "DeepSeek-V4.1-Flash - Architecture" section 4,
en.mycoding.id section 2.4.4).  Each check compares the oracle with something
other than itself: the bit-level format definitions, torch's float8 cast, a
brute-force nearest-value search, exact round trips and the 890 B/token claim."""
import json
import os

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
FACTS = json.load(open(os.path.join(HERE, "golden", "pages_facts.json")))


def e2m1_from_bits(c):
    """E2M1 from its bit fields: sign, 2-bit exponent (bias 1), 1-bit mantissa."""
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    v = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
    return -v if s else v


def test_e2m1_decode_matches_bit_definition(orc):
    for c in range(16):
        assert orc.e2m1_decode(c) == e2m1_from_bits(c)
    assert max(abs(orc.e2m1_decode(c)) for c in range(16)) == 6.0


def test_e4m3_decode_matches_torch_float8(orc):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([orc.e4m3_decode(b) for b in range(256)])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(np.where(both_nan, 0, ref), np.where(both_nan, 0, got))
    assert np.nanmax(got) == 448.0


def _e4m3_grid():
    vals = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    return np.sort(vals)


def test_e4m3_encode_matches_torch_cast_in_range(orc):
    grid = _e4m3_grid()
    mids = (grid[1:] + grid[:-1]) / 2
    rng = np.random.default_rng(1)
    xs = np.concatenate([grid, mids, rng.uniform(0, 460, 4000), np.exp(rng.uniform(-16, 6, 4000))])
    xs = xs[xs < 464].astype(np.float32)
    xs = np.concatenate([xs, -xs])
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(x)) for x in xs], dtype=np.uint8)
    # torch keeps the sign of an underflow to zero as well
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates(orc):
    for x in [448.0, 464.0, 500.0, 1e6, float("inf")]:
        assert orc.e4m3_encode(x) == 0x7E
        assert orc.e4m3_encode(-x) == 0xFE


def _e2m1_bruteforce(x):
    """Nearest E2M1 value by exhaustive search; ties to the even code; saturate."""
    best, best_d = None, None
    for c in range(8):
        v = e2m1_from_bits(c)
        d = abs(abs(x) - v)
        if best is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return best | (8 if np.signbit(x) else 0)


def test_e2m1_encode_matches_bruteforce(orc):
    grid = np.array([e2m1_from_bits(c) for c in range(8)])
    mids = (grid[1:] + grid[:-1]) / 2
    rng = np.random.default_rng(2)
    xs = np.concatenate([grid, mids, rng.uniform(0, 7, 3000), [0.0, 1e-30, 6.0, 6.5, 100.0]])
    xs = np.concatenate([xs, -xs]).astype(np.float32)
    for x in xs:
        assert orc.e2m1_encode(float(x)) == _e2m1_bruteforce(float(x)), x


def test_fp4_roundtrip_exact_groups(orc):
    """Every group of representable values code*scale whose amax is 6*scale
    quantises back to the same codes and scale, for every positive finite
    non-zero E4M3 scale."""
    rng = np.random.default_rng(3)
    for s in range(1, 127):
        sd = orc.e4m3_decode(s)
        codes = rng.integers(0, 16, size=512).astype(np.uint8)
        codes[::16] = 7 | (codes[::16] & 8)        # amax of each group = 6 * sd
        x = np.array([orc.e2m1_decode(c) * sd for c in codes], dtype=np.float32)
        assert np.array_equal(x.astype(np.float64), np.array([orc.e2m1_decode(c) * sd for c in codes]))
        ent = orc.fp4_quantise(x)
        assert np.all(ent[256:] == s)
        got_codes = np.empty(512, np.uint8)
        got_codes[0::2] = ent[:256] & 15
        got_codes[1::2] = ent[:256] >> 4
        # +0 and -0 are different codes with the same value; the input -0.0 keeps its sign
        assert np.array_equal(got_codes, codes)
        assert np.array_equal(orc.fp4_dequant(ent), x.astype(np.float64))


def test_fp4_quantisation_error_bound(orc):
    """|x - dq(x)| <= half the local E2M1 gap times the scale, unless saturated;
    and the scale is E4M3(amax/6)."""
    rng = np.random.default_rng(4)
    for trial in range(50):
        x = (rng.standard_normal(512) * rng.uniform(0.01, 50)).astype(np.float32)
        ent = orc.fp4_quantise(x)
        dq = orc.fp4_dequant(ent)
        for g in range(32):
            sd = orc.e4m3_decode(ent[256 + g])
            grp = x[16 * g:16 * g + 16].astype(np.float64)
            assert ent[256 + g] == orc.e4m3_encode(np.float32(np.abs(grp).max() / np.float32(6.0)))
            err = np.abs(grp - dq[16 * g:16 * g + 16])
            t = np.abs(grp) / sd
            gap = np.where(t < 2, 0.5, np.where(t < 4, 1.0, 2.0))
            sat = t > 6
            assert np.all((err <= gap / 2 * sd * (1 + 1e-6)) | sat)


def test_zero_and_tiny_groups(orc):
    x = np.zeros(512, np.float32)
    x[16:32] = 1e-6     # amax/6 underflows to a zero scale
    ent = orc.fp4_quantise(x)
    assert np.all(ent == 0)
    assert np.all(orc.fp4_dequant(ent) == 0)


def test_entry_bytes_and_890_accounting(orc):
    """The entry sizes reproduce the pages' 890 B/token global-KV claim:
    main entry 512*4 bits + 512/16 one-byte scales = 288 B; an MXFP4 indexer-K
    entry of 128 dims with a one-byte scale per 32 = 68 B; three encoder source
    layers at m=2 plus one decoder source layer at m=1."""
    f = FACTS["main_attention_settings"]
    main = f["query_head_dim"] // 2 + f["query_head_dim"] // FACTS["fp4_main_kv"]["channels_per_scale"]
    assert main == orc.ENTRY_BYTES == 288
    idx = f["indexer_head_dim"] // 2 + f["indexer_head_dim"] // 32
    L = FACTS["model_layers"]
    total = L["encoder_groups"] * (main + idx) / L["encoder_m"] + 1 * (main + idx) / L["decoder_m"]
    assert total == FACTS["global_kv_bytes_per_token"]["value"]
    # the latent splits 448 + 64 and the V4-Flash entry is 584 B
    ls = FACTS["latent_split"]
    assert ls["nope_channels"] + ls["rope_channels"] == f["query_head_dim"] == orc.D
    v4 = FACTS["v4_flash_main_kv_entry"]
    assert v4["nope_fp8_bytes"] + v4["rope_bf16_bytes"] + v4["scale_bytes"] == v4["total"]
    assert v4["nope_fp8_bytes"] == ls["nope_channels"] and v4["rope_bf16_bytes"] == 2 * ls["rope_channels"]


def test_format_max_magnitude(orc):
    """Without a global scale the format reaches 6 * 448 = 2688 (the pages'
    point that the range is far above the cache's magnitudes)."""
    x = np.zeros(512, np.float32)
    x[0] = 2688.0
    ent = orc.fp4_quantise(x)
    assert orc.fp4_dequant(ent)[0] == 2688.0
    x[0] = 1e5
    assert orc.fp4_dequant(orc.fp4_quantise(x))[0] == 2688.0
