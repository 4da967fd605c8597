"""Seeded synthetic inputs for the CSA2 decode / prefill workloads.

This module is shared by the tests, the benchmark and the oracle checks, and
holds none of the method's arithmetic: it only draws random tensors with the
shapes and distributions of the workloads the DeepSeek-V4.1-Flash pages
describe (64 query heads x 512, 32 indexer heads x 128, top-512, SWA-128,
HSI pool 2048 x 8; "DeepSeek-V4.1-Flash - Architecture", section 2 "Main
attention settings" and section 3 "Hierarchical Sparse Indexer").

Every tensor is drawn from a torch generator seeded from (seed, stream id), on
the device it is requested on.  A CPU draw and a CUDA draw with the same seed
give different numbers; a test that compares the GPU path with the oracle
draws once and hands the very same tensor (or its host copy) to both sides.

The sliding-window (SWA) entries are inputs of the hot path, stored as FP8
E4M3 with one fp32 scale per token: they are produced here with torch's own
float8 cast (a library routine), scale = amax / 448.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

# Fixed head geometry of the path ("Main attention settings").
D = 512            # latent / query head dim (key = value = latent)
ROPE_DIM = 64      # RoPE'd tail channels of the latent
H = 64             # query heads
HI = 32            # indexer heads
DI = 128           # indexer head dim
TOPK = 512         # index_topk
WINDOW = 128       # sliding_window
BLOCK = 8          # candidate_block_size
POOL_BLOCKS = 2048 # candidate_topk_blocks

# Stream ids: each tensor kind draws from its own generator stream.
_S_LATENT, _S_KIDX, _S_Q, _S_QIDX, _S_W, _S_SWA, _S_Z, _S_PLANT, _S_IDX, _S_POS = range(10)


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + stream * 7_919 + 12_345) % (2**63 - 1))
    return g


def normal(shape, seed, stream, device="cpu", dtype=torch.bfloat16, std=1.0):
    g = _gen(seed, stream, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def uniform(shape, seed, stream, device="cpu", lo=0.0, hi=1.0):
    g = _gen(seed, stream, device)
    x = torch.rand(*shape, generator=g, device=device, dtype=torch.float32)
    return x.mul_(hi - lo).add_(lo)


def fp8_rows(x: torch.Tensor):
    """Per-row E4M3 codes (uint8 view) and fp32 scale = amax/448 via torch's cast."""
    xf = x.float()
    amax = xf.abs().amax(dim=-1, keepdim=True).clamp_min(1e-30)
    scale = amax / 448.0
    codes = (xf / scale).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), scale.squeeze(-1).contiguous()


@dataclass
class LayerInputs:
    """Per-layer fresh operands of one decode step (query side + own SWA window)."""
    q: torch.Tensor          # bf16 [B, 64, 512]
    q_idx: torch.Tensor      # bf16 [B, 32, 128]  (~N(0,1)/sqrt(128))
    w: torch.Tensor          # fp32 [B, 32]       (~U(0,1))
    swa: torch.Tensor        # uint8 (E4M3 bits) [B, 128, 512]
    swa_scale: torch.Tensor  # fp32 [B, 128]
    swa_len: torch.Tensor    # int32 [B]


def layer_inputs(seed: int, batch: int, device="cpu", window: int = WINDOW) -> LayerInputs:
    q = normal((batch, H, D), seed, _S_Q, device)
    q_idx = normal((batch, HI, DI), seed, _S_QIDX, device, std=1.0 / math.sqrt(DI))
    w = uniform((batch, HI), seed, _S_W, device)
    swa_f = normal((batch, window, D), seed, _S_SWA, device, dtype=torch.float32)
    swa, swa_scale = fp8_rows(swa_f)
    swa_len = torch.full((batch,), window, dtype=torch.int32, device=device)
    return LayerInputs(q, q_idx, w, swa, swa_scale, swa_len)


def context_latent(seed: int, batch: int, n: int, device="cpu", m: int = 1) -> torch.Tensor:
    """Main-KV source latents ~N(0,1) bf16: [B, n, 512] (m=1) or [B, n, 2, 512] (m=2)."""
    shape = (batch, n, D) if m == 1 else (batch, n, m, D)
    return normal(shape, seed, _S_LATENT, device)


def compression_logits(seed: int, batch: int, n: int, device="cpu", m: int = 2) -> torch.Tensor:
    """Compressor logits Z ~N(0,1) bf16 [B, n, m, 512]."""
    return normal((batch, n, m, D), seed, _S_Z, device)


def indexer_keys(seed: int, batch: int, n: int, device="cpu") -> torch.Tensor:
    """Indexer K ~N(0,1) bf16 [B, n, 128]."""
    return normal((batch, n, DI), seed, _S_KIDX, device)


def random_positions(seed: int, batch: int, n_vis: int, k: int, device="cpu") -> torch.Tensor:
    """k distinct positions per sequence in [0, n_vis), ascending, int32 [B, k] (-1 pad)."""
    g = _gen(seed, _S_IDX, "cpu")
    out = torch.full((batch, k), -1, dtype=torch.int32)
    kk = min(k, n_vis)
    for b in range(batch):
        sel = torch.randperm(n_vis, generator=g)[:kk].sort().values
        out[b, :kk] = sel.to(torch.int32)
    return out.to(device)


def plant_blocks(k_idx: torch.Tensor, q_idx: torch.Tensor, w: torch.Tensor, n_vis: int,
                 n_blocks: int, seed: int, gain: float = 4.0, noise: float = 0.1):
    """Overwrite n_blocks random complete blocks of 8 keys per sequence with keys
    aligned to the direction sum_h w_h q_h (gain * unit * sqrt(128) + N(0, noise^2)).
    Returns the planted block ids, int64 [B, n_blocks] sorted."""
    B = k_idx.shape[0]
    g = _gen(seed, _S_PLANT, "cpu")
    n_full = n_vis // BLOCK
    ids = torch.stack([torch.randperm(n_full, generator=g)[:n_blocks].sort().values for _ in range(B)])
    dirv = (w.float().unsqueeze(-1) * q_idx.float()).sum(dim=1)            # [B, 128]
    dirv = dirv / dirv.norm(dim=-1, keepdim=True)
    for b in range(B):
        noise_t = normal((n_blocks, BLOCK, DI), seed * 7 + b, _S_PLANT, k_idx.device,
                         dtype=torch.float32, std=noise)
        keys = gain * math.sqrt(DI) * dirv[b].to(k_idx.device) + noise_t  # [n_blocks, 8, 128]
        rows = (ids[b].to(k_idx.device).unsqueeze(-1) * BLOCK
                + torch.arange(BLOCK, device=k_idx.device)).reshape(-1)
        k_idx[b, rows] = keys.reshape(-1, DI).to(k_idx.dtype)
    return ids


@dataclass
class Config:
    """One workload of the decode / prefill path (shapes of the pages' workloads)."""
    name: str
    batch: int
    n_ctx: int
    schedule: list = field(default_factory=list)   # list of "full" / "reindex" / "reuse" / "swa"
    hsi: bool = False
    planted_blocks: int = 0
    m: int = 1
    chunk: int = 0          # prefill: new tokens appended per sequence (m=2: chunk/2 entries)
    layer_seeds: list = field(default_factory=list)


def decoder_layer_modes(groups: int = 5, per_group: int = 4, first: str = "full", later: str = "reindex"):
    """The decoder's CSA2 schedule: groups of `per_group` layers; group 1 opens
    with a Full layer, the later groups with a Reindex layer, the rest Reuse
    ("DeepSeek-V4.1-Flash - Architecture", section 2 "Layer schedule")."""
    modes = []
    for gi in range(groups):
        modes.append(first if gi == 0 else later)
        modes.extend(["reuse"] * (per_group - 1))
    return modes


def encoder_layer_modes(swa_layers: int = 2, groups: int = 3, per_group: int = 6):
    """The encoder's schedule: SWA-only layers, then groups of one Full layer
    (its own m = 2 cache copy) and Reuse layers ("DeepSeek-V4.1-Flash -
    Architecture", section 2; "DeepSeek-v4.1 Flash: Pushing the Limits of KV
    Cache Compression", section 2.3.3)."""
    modes = ["swa"] * swa_layers
    for _ in range(groups):
        modes.append("full")
        modes.extend(["reuse"] * (per_group - 1))
    return modes


CONFIGS = {
    # tiny single-layer Full decode, seed 0
    "decode_1x4k": Config("decode_1x4k", 1, 4096, ["full"], layer_seeds=[0]),
    # decoder group decode: Full + 3 Reuse, seeds 1..4
    "group_decode_32x64k": Config("group_decode_32x64k", 32, 65536, ["full", "reuse", "reuse", "reuse"],
                 layer_seeds=[1, 2, 3, 4]),
    # hierarchical indexer: Full (HSI) + 4 Reindex, planted blocks
    "hsi_reindex_16x256k": Config("hsi_reindex_16x256k", 16, 262144, ["full", "reindex", "reindex", "reindex", "reindex"],
                 hsi=True, planted_blocks=16, layer_seeds=[2000 + i for i in range(5)]),
    # long-context full 20-layer decoder step
    "decoder20_4x1m": Config("decoder20_4x1m", 4, 1048576, decoder_layer_modes(), hsi=True,
                 layer_seeds=[3000 + i for i in range(20)]),
    # the encoder's 20 layers at decode: 2 SWA-only, 3 x [Full + 5 Reuse] over
    # three m=2 cache copies; a 65,536-token context (32,768 entries per copy)
    # and a step whose token completes an entry pair
    "encoder_decode_32x64k": Config("encoder_decode_32x64k", 32, 65536, encoder_layer_modes(), m=2,
                 layer_seeds=[5000 + i for i in range(20)]),
    # chunked prefill at m=2: 131072-token context + 16384-token chunk
    "prefill_m2_2x128k": Config("prefill_m2_2x128k+16k", 2, 131072, ["full"], m=2, chunk=16384,
                 layer_seeds=[4000]),
}
