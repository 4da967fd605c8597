"""The benchmark's roofline accounting (host logic, no GPU): algorithmic bytes
per step of each decode workload, built from the per-unit figures (an FP4
entry 288 B, an indexer-K row 256 B bf16 / 68 B MXFP4, the readout's 412,160
B per token and layer, 16,384 pool positions per Reindex layer)."""
import synth

import bench


def test_group_decode_step_bytes():
    cfg = synth.CONFIGS["group_decode_32x64k"]
    B, N = cfg.batch, cfg.n_ctx
    per_seq = (1024 + 288 + 16) + 4 * 412160 + (256 * N + 32 * 128 * 2 + 32 * 4 + 512 * 4)
    assert bench.ATTN_BYTES == 412160
    assert bench.algorithmic_bytes(cfg, 0) == B * per_seq == 590001664   # 590.0 MB per step
    # the MXFP4 indexer reads 68 B per position and writes the new key's entry
    fp4 = B * (per_seq - 256 * N + 68 * N + 256 + 68)
    assert bench.algorithmic_bytes(cfg, 0, fp4=True) == fp4
    # a projected key: W_ik read once and the key written instead
    assert bench.algorithmic_bytes(cfg, 0, fp4=True, project=True) == fp4 - B * (256 + 68) + 128 * 512 * 2 + B * 68


def test_reindex_and_decoder_step_bytes():
    cfg = synth.CONFIGS["hsi_reindex_16x256k"]
    B, N = cfg.batch, cfg.n_ctx
    full = (1024 + 288 + 16) + (256 * N + 8320 + 2048)
    reindex = 16384 * 256 + 18560
    assert bench.algorithmic_bytes(cfg, 1) == B * (full + 4 * reindex + 5 * 412160)
    dec = synth.CONFIGS["decoder20_4x1m"]
    assert sum(m == "reindex" for m in dec.schedule) == 4 and len(dec.schedule) == 20
    assert bench.algorithmic_bytes(dec, 1) == dec.batch * (
        (1024 + 288 + 16) + (256 * dec.n_ctx + 8320 + 2048) + 4 * reindex + 20 * 412160)


def test_encoder_step_bytes():
    cfg = synth.CONFIGS["encoder_decode_32x64k"]
    B, E = cfg.batch, cfg.n_ctx // 2
    write_m2 = 2 * 1024 + 2 * 1024 + 288 + 16                 # the pair, its logits, the entry
    sweep = 256 * E + 8320 + 2048
    swa_only = 412160 - 512 * 288 - 512 * 4                    # no selected entries
    assert bench.kv_write_bytes(2) == write_m2
    assert bench.algorithmic_bytes(cfg, 0) == B * (3 * (write_m2 + sweep) + 18 * 412160 + 2 * swa_only)
