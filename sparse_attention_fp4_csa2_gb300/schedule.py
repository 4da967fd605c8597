"""CSA2 layer schedule (host logic).

"DeepSeek-V4.1-Flash - Architecture", section 2 "Layer schedule": the decoder
has five groups of four layers; the first group opens with a Full layer, the
other four with a Reindex layer, and every other layer is Reuse (decoder
layers 20 Full, 24/28/32/36 Reindex -- "DeepSeek-v4.1 Flash: Pushing the
Limits of KV Cache Compression", section 3.3.3).  The encoder has two SWA-only
layers, then three groups of one Full and five Reuse layers at m = 2.

Modes ("CSA2 modes" table): Full writes new main KV / indexer K and a new
top-K; Reindex reuses the cache with a new top-K; Reuse reuses the latest
top-K.  A Reuse layer therefore needs an earlier index layer in its stack.
"""
from __future__ import annotations

from enum import Enum


class Mode(str, Enum):
    FULL = "full"
    REINDEX = "reindex"
    REUSE = "reuse"
    SWA = "swa"


def decoder_modes(groups: int = 5, per_group: int = 4) -> list:
    out = []
    for g in range(groups):
        out.append(Mode.FULL if g == 0 else Mode.REINDEX)
        out.extend([Mode.REUSE] * (per_group - 1))
    return out


def encoder_modes(swa_layers: int = 2, groups: int = 3, per_group: int = 6) -> list:
    out = [Mode.SWA] * swa_layers
    for _ in range(groups):
        out.append(Mode.FULL)
        out.extend([Mode.REUSE] * (per_group - 1))
    return out


def validate(modes) -> None:
    """A Reindex or Reuse layer needs an earlier Full layer in the stack."""
    seen_full = False
    for i, m in enumerate(modes):
        m = Mode(m)
        if m == Mode.FULL:
            seen_full = True
        elif m in (Mode.REINDEX, Mode.REUSE) and not seen_full:
            raise ValueError(f"layer {i}: {m.value} before any Full layer")


def cache_copies(modes) -> int:
    """Main-KV / indexer-K copies a stack keeps: one per Full layer (Reindex
    and Reuse layers read the latest one)."""
    return sum(Mode(m) == Mode.FULL for m in modes)


def global_kv_bytes_per_token(entry_bytes: int, indexer_entry_bytes: int, encoder=None, decoder=None,
                              m_encoder: int = 2, m_decoder: int = 1) -> float:
    """Global cache growth per token ("DeepSeek-v4.1 Flash: Pushing the Limits
    of KV Cache Compression", section 3.1): every cache copy adds one main-KV
    entry and one indexer-K entry per m tokens.  The encoder keeps a copy per
    Full layer at m = 2, the decoder its own at m = 1."""
    enc = encoder_modes() if encoder is None else encoder
    dec = decoder_modes() if decoder is None else decoder
    per_entry = entry_bytes + indexer_entry_bytes
    return cache_copies(enc) * per_entry / m_encoder + cache_copies(dec) * per_entry / m_decoder
