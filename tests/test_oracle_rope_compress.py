"""Pins for the oracle's RoPE-on-the-tail and m=2 compressor.

The pages fix that RoPE rotates only the tail channels of the 512-d latent
(448 NoPE + 64 RoPE) and that it is an orthogonal, position-dependent rotation
that preserves the norm (en.mycoding.id sections 2.4.4 and 3.3.2.5); the pairing
and the base are conventions (parity unpinned), so the checks here are the
invariants, plus an independent complex-number formulation of the same
convention.  The compressor is gated pooling with channel-wise softmax weights
over the m positions (section 2.3.1), which reduces to the mean for equal
logits and to one position for a dominant logit."""
import numpy as np
import torch


def test_rope_position_zero_is_identity(orc):
    x = np.random.default_rng(0).standard_normal(512).astype(np.float32)
    assert np.array_equal(orc.rope_tail(x, 0), x)


def test_rope_touches_only_the_tail(orc):
    x = np.random.default_rng(1).standard_normal(512).astype(np.float32)
    y = orc.rope_tail(x, 12345)
    assert np.array_equal(y[:448], x[:448])
    assert not np.array_equal(y[448:], x[448:])


def test_rope_preserves_pair_norms(orc):
    rng = np.random.default_rng(2)
    for pos in [1, 7, 4095, 65535, 1048575]:
        x = rng.standard_normal(512).astype(np.float32)
        y = orc.rope_tail(x, pos).astype(np.float64)
        xp = x[448:].astype(np.float64).reshape(32, 2)
        yp = y[448:].reshape(32, 2)
        assert np.allclose(np.linalg.norm(xp, axis=1), np.linalg.norm(yp, axis=1), rtol=1e-6, atol=1e-7)


def test_rope_matches_complex_rotation(orc):
    """Same convention written as a complex multiply x * exp(i * pos * theta_i)."""
    rng = np.random.default_rng(3)
    for pos in [3, 1000, 262143]:
        x = rng.standard_normal(512).astype(np.float32)
        y = orc.rope_tail(x, pos).astype(np.float64)
        inv = (10000.0 ** (-(2.0 * np.arange(32)) / 64.0)).astype(np.float32).astype(np.float64)
        z = (x[448::2].astype(np.float64) + 1j * x[449::2].astype(np.float64)) * np.exp(1j * pos * inv)
        assert np.allclose(y[448::2], z.real, atol=2e-6)
        assert np.allclose(y[449::2], z.imag, atol=2e-6)


def test_rope_composes(orc):
    x = np.random.default_rng(4).standard_normal(512).astype(np.float32)
    y = orc.rope_tail(orc.rope_tail(x, 300), 700)
    assert np.allclose(y, orc.rope_tail(x, 1000), atol=1e-5)


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)


def test_compress_equal_logits_gives_mean(orc):
    rng = np.random.default_rng(5)
    x = _bf16(rng.standard_normal((2, 512)))
    z = _bf16(np.tile(rng.standard_normal(512), (2, 1)))
    e = orc.compress(x, z, 2)
    xf = x.double().numpy()
    assert np.array_equal(e, ((xf[0] + xf[1]) / 2).astype(np.float32))


def test_compress_dominant_logit_selects_position(orc):
    rng = np.random.default_rng(6)
    x = _bf16(rng.standard_normal((2, 512)))
    z = torch.zeros(2, 512, dtype=torch.bfloat16)
    z[0] = 80.0
    e = orc.compress(x, z, 2)
    assert np.array_equal(e, x[0].float().numpy())


def test_compress_matches_torch_softmax(orc):
    rng = np.random.default_rng(7)
    x = _bf16(rng.standard_normal((2, 512)))
    z = _bf16(rng.standard_normal((2, 512)) * 3)
    w = torch.softmax(z.double(), dim=0)
    ref = (w * x.double()).sum(0).numpy()
    e = orc.compress(x, z, 2).astype(np.float64)
    assert np.all(np.abs(e - ref) <= np.abs(ref) * 2.0 ** -23 + 1e-30)


def test_compress_m1_is_identity(orc):
    x = _bf16(np.random.default_rng(8).standard_normal((1, 512)))
    assert np.array_equal(orc.compress(x, None, 1), x[0].float().numpy())


def test_kv_entry_is_quantise_after_rope(orc):
    rng = np.random.default_rng(9)
    lat = _bf16(rng.standard_normal((3, 512)))
    pos = np.array([0, 17, 4095], np.int64)
    ent = orc.kv_entries(lat, None, 1, pos)
    for i in range(3):
        ref = orc.fp4_quantise(orc.rope_tail(lat[i].float().numpy(), int(pos[i])))
        assert np.array_equal(ent[i], ref)
