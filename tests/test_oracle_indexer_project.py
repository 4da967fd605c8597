"""Pins for the oracle's indexer-K projection (the Full layer obtains its
indexer K by projecting the main-KV entry: "DeepSeek-v4.1 Flash: Pushing the
Limits of KV Cache Compression", section 2.3.1).  Checked against closed forms
at position 0 (where RoPE is the identity), an fp64 matrix product, exact
linearity, the position independence of the non-RoPE channels, the rotation's
pair norm, and the m = 2 mean for equal logits."""
import numpy as np
import torch

D, DI = 512, 128


def _bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def _sel(cols):
    """W [128, 512] with row o selecting channel cols[o]."""
    w = torch.zeros(DI, D)
    w[torch.arange(DI), torch.as_tensor(cols)] = 1.0
    return w.to(torch.bfloat16)


def test_selection_at_position_zero_returns_the_channels(orc):
    g = torch.Generator().manual_seed(0)
    lat = torch.randn(20, D, generator=g).to(torch.bfloat16)
    cols = torch.randint(0, D, (DI,), generator=g)
    k = orc.indexer_k_project(lat, None, 1, np.zeros(20, np.int64), _sel(cols))
    assert torch.equal(k, lat[:, cols])


def test_dense_projection_equals_fp64_matmul(orc):
    g = torch.Generator().manual_seed(1)
    lat = torch.randn(50, D, generator=g).to(torch.bfloat16)
    w = (torch.randn(DI, D, generator=g) / D ** 0.5).to(torch.bfloat16)
    k = orc.indexer_k_project(lat, None, 1, np.zeros(50, np.int64), w).float().numpy()
    ref = lat.double().numpy() @ w.double().numpy().T          # exact products, fp64 sums
    ulp = np.exp2(np.floor(np.log2(np.abs(ref))) - 7)
    assert np.all(np.abs(k - ref) <= 0.5 * ulp * (1 + 1e-9))   # rounded once, to nearest
    assert np.mean(k == _bf16(ref).float().numpy()) > 0.99


def test_linear_in_the_entry(orc):
    g = torch.Generator().manual_seed(2)
    lat = torch.randn(10, D, generator=g).to(torch.bfloat16)
    w = (torch.randn(DI, D, generator=g) / D ** 0.5).to(torch.bfloat16)
    pos = np.arange(10, dtype=np.int64) * 977
    k1 = orc.indexer_k_project(lat, None, 1, pos, w)
    k2 = orc.indexer_k_project((lat.float() * 2).to(torch.bfloat16), None, 1, pos, w)
    assert torch.equal(k2.float(), k1.float() * 2)


def test_non_rope_channels_do_not_depend_on_position_and_pairs_keep_their_norm(orc):
    g = torch.Generator().manual_seed(3)
    lat = torch.randn(8, D, generator=g).to(torch.bfloat16)
    cols = torch.randint(0, 448, (DI,), generator=g)
    for pos in (1, 12345, 4000000):
        k = orc.indexer_k_project(lat, None, 1, np.full(8, pos, np.int64), _sel(cols))
        assert torch.equal(k, lat[:, cols])
    # rows selecting the RoPE pair (448 + 2i, 449 + 2i): the pair's norm is kept
    cols = torch.tensor([448 + (o % 64) for o in range(DI)])
    k = orc.indexer_k_project(lat, None, 1, np.full(8, 31337, np.int64), _sel(cols)).double()
    x = lat.double()
    for i in range(32):
        n_in = x[:, 448 + 2 * i] ** 2 + x[:, 449 + 2 * i] ** 2
        n_out = k[:, 2 * i] ** 2 + k[:, 2 * i + 1] ** 2
        assert torch.allclose(n_out, n_in, rtol=2e-2, atol=1e-6)


def test_m2_equal_logits_give_the_pair_mean(orc):
    g = torch.Generator().manual_seed(4)
    lat = torch.randn(6, 2, D, generator=g).to(torch.bfloat16)
    z = torch.zeros(6, 2, D, dtype=torch.bfloat16)
    cols = torch.randint(0, 448, (DI,), generator=g)
    k = orc.indexer_k_project(lat, z, 2, np.arange(6, dtype=np.int64) * 2 + 1, _sel(cols))
    mean = ((lat[:, 0].double() + lat[:, 1].double()) / 2).float()   # the pooled fp32 entry
    assert torch.equal(k, mean[:, cols].to(torch.bfloat16))
