"""GPU parity of csa2_kv_quant_write against the oracle: codes and scales
bit-exact (RoPE on the tail, then E2M1 + one E4M3 scale per 16 channels;
"DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression" 2.4.4)."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def c2():
    import sparse_attention_fp4_csa2_gb300.build as b
    b.build()
    import sparse_attention_fp4_csa2_gb300 as c
    return c


def _write(c2, latent, z, m, pos, rows=None):
    n = pos.numel()
    rows = rows or n
    kv = torch.zeros(rows, 288, dtype=torch.uint8, device="cuda")
    slot = torch.arange(n, dtype=torch.int64, device="cuda")
    c2.kv_quant_write(latent.cuda().contiguous(), None if z is None else z.cuda().contiguous(), m, pos.cuda(),
                      slot, kv)
    assert c2.get_device_status() == 0
    return kv.cpu().numpy()


def test_random_entries_c0(c2, orc):
    lat = synth.context_latent(0, 1, 4096)[0]
    pos = torch.arange(4096, dtype=torch.int64)
    got = _write(c2, lat, None, 1, pos)
    exp = orc.kv_entries(lat, None, 1, pos.numpy())
    assert np.array_equal(got, exp)


def test_far_positions_and_scaled_latents(c2, orc):
    lat = (synth.context_latent(11, 1, 2048)[0].float() * torch.logspace(-4, 3, 2048)[:, None]).to(torch.bfloat16)
    pos = torch.randint(0, 1 << 20, (2048,), generator=torch.Generator().manual_seed(5), dtype=torch.int64)
    got = _write(c2, lat, None, 1, pos)
    exp = orc.kv_entries(lat, None, 1, pos.numpy())
    assert np.array_equal(got, exp)


def test_all_bf16_values_as_channels(c2, orc):
    """Every finite bf16 pattern appears as a channel value, in groups whose
    amax spans the whole E4M3 scale range (subnormal, normal, saturated)."""
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    vals = bits.view(torch.bfloat16)
    vals = vals[torch.isfinite(vals.float())]
    n = (vals.numel() + 511) // 512 * 512
    pad = torch.zeros(n - vals.numel(), dtype=torch.bfloat16)
    lat = torch.cat([vals, pad]).reshape(-1, 512)
    lat = lat[torch.randperm(lat.shape[0], generator=torch.Generator().manual_seed(1))]
    pos = torch.zeros(lat.shape[0], dtype=torch.int64)     # position 0: RoPE is the identity
    got = _write(c2, lat, None, 1, pos)
    exp = orc.kv_entries(lat, None, 1, pos.numpy())
    assert np.array_equal(got, exp)


def test_e2m1_midpoints_every_scale(c2, orc):
    """Groups with amax = 6 * s for every positive finite E4M3 scale s and the
    other channels on the E2M1 rounding midpoints (ties to even)."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.1, 0.3, 5.9, 6.0, 2.0, 0.0, 4.4, 1.0])
    rows = []
    for s in range(1, 127):
        sd = orc.e4m3_decode(s)
        g = np.concatenate([[6.0], mids]) * sd
        sign = np.where(np.arange(16) % 3 == 1, -1.0, 1.0)
        rows.append(np.tile(g * sign, 32))
    lat = torch.tensor(np.stack(rows), dtype=torch.float32).to(torch.bfloat16)
    pos = torch.zeros(lat.shape[0], dtype=torch.int64)
    got = _write(c2, lat, None, 1, pos)
    exp = orc.kv_entries(lat, None, 1, pos.numpy())
    assert np.array_equal(got, exp)


def test_compressor_m2(c2, orc):
    lat = synth.context_latent(40, 1, 1024, m=2)[0]       # [1024, 2, 512]
    z = synth.compression_logits(40, 1, 1024)[0]
    pos = torch.arange(1024, dtype=torch.int64) * 2 + 1
    got = _write(c2, lat, z, 2, pos)
    exp = orc.kv_entries(lat, z, 2, pos.numpy())
    assert np.array_equal(got, exp)


def test_slots_scatter_and_bad_slot(c2, orc):
    lat = synth.context_latent(3, 1, 16)[0].cuda()
    pos = torch.arange(16, dtype=torch.int64, device="cuda")
    slot = torch.arange(16, dtype=torch.int64, device="cuda").flip(0) * 2
    slot[3] = 1000                                          # outside the cache
    kv = torch.zeros(32, 288, dtype=torch.uint8, device="cuda")
    c2.kv_quant_write(lat, None, 1, pos, slot, kv)
    assert c2.get_device_status() & 0x2
    assert c2.get_device_status() == 0                      # cleared by the read
    exp = orc.kv_entries(lat.cpu(), None, 1, np.arange(16))
    got = kv.cpu().numpy()
    for i in range(16):
        if i == 3:
            continue
        assert np.array_equal(got[int(slot[i])], exp[i])
    assert not got[1::2].any()


def test_empty_is_noop(c2):
    kv = torch.zeros(4, 288, dtype=torch.uint8, device="cuda")
    e = torch.empty(0, dtype=torch.int64, device="cuda")
    c2.kv_quant_write(torch.empty(0, 512, dtype=torch.bfloat16, device="cuda"), None, 1, e, e, kv)
    assert c2.last_launch_count() == 0


@pytest.mark.parametrize("m", [1, 2])
def test_kv_write_with_indexer_projection(c2, orc, m):
    """csa2_kv_quant_write_ik: the main-KV entry equals the plain writer's and
    the oracle's bit for bit; the indexer key W_ik e is the oracle's fp64
    projection rounded to bf16 (within one bf16 step, equal almost
    everywhere: the GPU sums in fp32); its MXFP4 form equals the oracle's
    codec of the oracle's key wherever the two bf16 keys agree."""
    n, rows = 300, 512
    g = torch.Generator().manual_seed(70 + m)
    lat = torch.randn((n, m, 512) if m == 2 else (n, 512), generator=g).to(torch.bfloat16)
    z = torch.randn(n, 2, 512, generator=g).to(torch.bfloat16) if m == 2 else None
    w_ik = (torch.randn(128, 512, generator=g) / 512 ** 0.5).to(torch.bfloat16)
    pos = torch.randint(0, 1 << 20, (n,), generator=g, dtype=torch.int64)
    slot = torch.randperm(rows, generator=g)[:n].to(torch.int64)
    slot[7] = rows + 3                                        # skipped, flags an index error
    kv_plain = torch.zeros(rows, 288, dtype=torch.uint8, device="cuda")
    kv = torch.zeros_like(kv_plain)
    kv4 = torch.zeros_like(kv_plain)
    k_bf = torch.zeros(rows, 128, dtype=torch.bfloat16, device="cuda")
    k_f4 = c2.indexer_k_fp4_cache(rows)
    zz = z.cuda() if z is not None else None
    c2.kv_quant_write(lat.cuda(), zz, m, pos.cuda(), slot.cuda(), kv_plain)
    assert c2.get_device_status() == 0x2
    c2.kv_quant_write_ik(lat.cuda(), zz, m, pos.cuda(), slot.cuda(), kv, w_ik.cuda(), k_bf)
    assert c2.get_device_status() == 0x2
    c2.kv_quant_write_ik(lat.cuda(), zz, m, pos.cuda(), slot.cuda(), kv4, w_ik.cuda(), k_f4, indexer_fp4=True)
    assert c2.get_device_status() == 0x2
    ok = np.arange(n) != 7
    okt = torch.from_numpy(ok)
    s = slot.numpy()[ok]
    assert torch.equal(kv, kv_plain) and torch.equal(kv4, kv_plain)
    want = orc.kv_entries(lat[okt], z[okt] if z is not None else None, m, pos.numpy()[ok])
    assert np.array_equal(kv.cpu().numpy()[s], want)
    k_or = orc.indexer_k_project(lat[okt], z[okt] if z is not None else None, m, pos.numpy()[ok], w_ik)
    got = k_bf.cpu()[s]
    a, b = got.float().numpy().astype(np.float64), k_or.float().numpy().astype(np.float64)
    # the oracle's own pre-quantisation entries e, for the fp32 sum's error
    # bound: both sides round to bf16 once (half a step each), and the GPU's
    # fp32 sum of 512 products (16-term chains, then a 5-level tree) is
    # within 32 u sum |w e| of the exact one
    lat_ok, z_ok = lat[okt], (z[okt] if z is not None else None)
    e = np.stack([orc.rope_tail(orc.compress(lat_ok[i].reshape(m, 512),
                                             z_ok[i] if z_ok is not None else None, m), int(p))
                  for i, p in enumerate(pos.numpy()[ok])]).astype(np.float64)
    bound = np.abs(e) @ np.abs(w_ik.double().numpy()).T * 32 * 2.0 ** -24
    step = lambda x: np.exp2(np.floor(np.log2(np.maximum(np.abs(x), 1e-30))) - 7)
    assert np.all(np.abs(a - b) <= 0.5 * step(a) + 0.5 * step(b) + bound)
    same_row = (got.view(torch.int16) == k_or.view(torch.int16)).all(dim=1).numpy()
    assert same_row.mean() > 0.8
    oc, os_ = orc.mxfp4_quantise(k_or)
    codes, scales = (t.cpu().numpy() for t in c2.indexer_k_fp4_planes(k_f4))
    assert np.array_equal(codes[s][same_row], oc[same_row]) and np.array_equal(scales[s][same_row], os_[same_row])
    untouched = np.setdiff1d(np.arange(rows), s)
    assert not k_bf.cpu()[untouched].float().abs().sum() and not codes[untouched].any()
