"""CPU-side checks of the C ABI: the library builds for sm_103a, loads, exports
every function include/csa2.h declares, and rejects bad arguments on the host
without launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def c2():
    import sparse_attention_fp4_csa2_gb300.build as b
    b.build()
    import sparse_attention_fp4_csa2_gb300 as c
    return c


def declared_functions():
    src = open(os.path.join(ROOT, "include", "csa2.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(c2):
    names = declared_functions()
    assert len(names) >= 10
    L = c2.lib()
    for n in names:
        assert hasattr(L, n), n


def test_defaults_and_sizes(c2):
    p = c2.default_params()
    assert (p.index_topk, p.sliding_window, p.candidate_block_size, p.candidate_topk_blocks, p.block_reduce,
            p.hsi, p.attn_kernel, p.indexer_fp4) == (512, 128, 8, 2048, 0, 1, 0, 0)
    assert c2.entry_bytes() == 288
    assert c2.indexer_entry_bytes(False) == 256 and c2.indexer_entry_bytes(True) == 68 == c2.FP4_ENTRY_BYTES
    assert c2.lib().csa2_status_string(3) == b"workspace too small"


def test_topk_kernel_choice(c2):
    """csa2_set_topk_kernel takes 0 (automatic), 1 (a cluster per row) or 2
    (a CTA per row) and rejects anything else; the choice is host state."""
    L = c2.lib()
    for v in (1, 2, 0):
        assert L.csa2_set_topk_kernel(v) == 0
    for v in (-1, 3, 100):
        assert L.csa2_set_topk_kernel(v) == c2.lib().csa2_set_topk_kernel(v) != 0
    with pytest.raises(c2.Csa2Error):
        c2.set_topk_kernel(7)
    c2.set_topk_kernel(c2.TOPK_AUTO)


def test_workspace_sizes(c2):
    p = c2.Params.make()
    for op in range(4):
        assert c2.workspace_bytes(op, 32, 65536, p) > 0
    # decode workspace covers every stage
    d = c2.workspace_bytes(c2.OP_DECODE, 4, 1 << 20, p)
    assert d >= c2.workspace_bytes(c2.OP_INDEXER, 4, 1 << 20, p)
    assert d >= c2.workspace_bytes(c2.OP_ATTN, 4, 1 << 20, p)
    bad = c2.Params.make(candidate_block_size=16)
    assert c2.workspace_bytes(c2.OP_DECODE, 4, 1000, bad) == 0
    assert c2.workspace_bytes(c2.OP_ATTN, 4, 1000, c2.Params.make(attn_kernel=3)) == 0
    assert c2.workspace_bytes(c2.OP_ATTN, 4, 1000, c2.Params.make(attn_kernel=2)) > 0
    assert c2.workspace_bytes(c2.OP_DECODE, 0, 1000, p) == 0
    # the MXFP4 indexer adds its E5M2 query rows (128 B) and folded weights (4 B)
    f4 = c2.Params.make(indexer_fp4=1)
    assert c2.workspace_bytes(c2.OP_INDEXER, 4, 4096, f4) >= c2.workspace_bytes(c2.OP_INDEXER, 4, 4096, p) + 4 * 32 * (128 + 4)
    assert c2.workspace_bytes(c2.OP_INDEXER, 4, 4096, c2.Params.make(indexer_fp4=2)) == 0


def test_host_validation_rejects_without_launch(c2):
    L = c2.lib()
    P = ctypes.c_void_p
    p = c2.Params.make()
    fake = P(0x1000)          # never dereferenced: validation fails first
    odd = P(0x1001)
    # null pointers
    assert L.csa2_kv_quant_write(None, None, 1, 4, fake, fake, fake, 4, 10000.0, None) == 1
    # misaligned latent
    assert L.csa2_kv_quant_write(odd, None, 1, 4, fake, fake, fake, 4, 10000.0, None) == 1
    # m = 2 without logits
    assert L.csa2_kv_quant_write(fake, None, 2, 4, fake, fake, fake, 4, 10000.0, None) == 1
    # empty write is OK and launches nothing
    assert L.csa2_kv_quant_write(None, None, 1, 0, None, None, None, 0, 10000.0, None) == 0
    assert c2.last_launch_count() == 0
    # unsupported block width
    bad = c2.Params.make(candidate_block_size=4)
    assert L.csa2_indexer_score_topk(fake, fake, fake, 1, 100, fake, 100, None, ctypes.byref(bad), fake, None,
                                     P(0x1000), 1 << 30, None) == 2
    # workspace too small
    assert L.csa2_indexer_score_topk(fake, fake, fake, 1, 100, fake, 100, None, ctypes.byref(p), fake, None,
                                     P(0x1000), 16, None) == 3
    # n_max above the cache capacity
    assert L.csa2_indexer_score_topk(fake, fake, fake, 1, 100, fake, 200, None, ctypes.byref(p), fake, None,
                                     P(0x1000), 1 << 30, None) == 1
    # the projecting KV write needs W_ik and a key cache; MXFP4 rows a multiple of 4
    assert L.csa2_kv_quant_write_ik(fake, None, 1, 4, fake, fake, fake, 4, 10000.0, None, fake, 8, 0, None) == 1
    assert L.csa2_kv_quant_write_ik(fake, None, 1, 4, fake, fake, fake, 4, 10000.0, fake, None, 8, 0, None) == 1
    assert L.csa2_kv_quant_write_ik(fake, None, 1, 4, fake, fake, fake, 4, 10000.0, odd, fake, 8, 0, None) == 1
    assert L.csa2_kv_quant_write_ik(fake, None, 1, 4, fake, fake, fake, 4, 10000.0, fake, fake, 6, 1, None) == 1
    assert L.csa2_kv_quant_write_ik(None, None, 1, 0, None, None, None, 0, 10000.0, None, None, 0, 0, None) == 0
    assert c2.last_launch_count() == 0
    # MXFP4 indexer-K write: rows must be a multiple of 4, pointers aligned; n = 0 is a no-op
    assert L.csa2_indexer_k_quant(fake, 4, fake, fake, 6, None) == 1
    assert L.csa2_indexer_k_quant(odd, 4, fake, fake, 8, None) == 1
    assert L.csa2_indexer_k_quant(fake, 4, fake, odd, 8, None) == 1
    assert L.csa2_indexer_k_quant(None, 4, fake, fake, 8, None) == 1
    assert L.csa2_indexer_k_quant(None, 0, None, None, 0, None) == 0
    assert c2.last_launch_count() == 0
    # MXFP4 cache capacity must be a multiple of 4; the prefill has no MXFP4 indexer
    f4 = c2.Params.make(indexer_fp4=1)
    assert L.csa2_indexer_score_topk(fake, fake, fake, 1, 102, fake, 100, None, ctypes.byref(f4), fake, None,
                                     P(0x1000), 1 << 30, None) == 1
    assert L.csa2_prefill_chunk(ctypes.byref(f4), 1, 64, 0, 1, fake, fake, fake, fake, fake, 128, fake, fake, 0, 0,
                                fake, fake, None, P(0x1000), 1 << 30, None) == 2
    # REINDEX needs a pool
    assert L.csa2_sparse_decode(1, ctypes.byref(p), 1, fake, fake, fake, fake, fake, 100, fake, 100, fake, fake,
                                fake, fake, None, fake, None, P(0x1000), 1 << 30, None) == 1
    # bad mode
    assert L.csa2_sparse_decode(7, ctypes.byref(p), 1, fake, fake, fake, fake, fake, 100, fake, 100, fake, fake,
                                fake, fake, fake, fake, None, P(0x1000), 1 << 30, None) == 1


def test_encoder_decode_workload_schedule():
    """The encoder decode workload follows the pages' schedule: two SWA-only
    layers, then three groups of Full + five Reuse, each Full layer with its
    own cache copy, at m = 2 ("DeepSeek-V4.1-Flash - Architecture", section 2)."""
    import sys
    sys.path.insert(0, ROOT)
    import synth
    from sparse_attention_fp4_csa2_gb300 import schedule as s
    cfg = synth.CONFIGS["encoder_decode_32x64k"]
    assert cfg.m == 2 and cfg.n_ctx % 2 == 0 and len(cfg.schedule) == 20 and len(cfg.layer_seeds) == 20
    assert cfg.schedule[:2] == ["swa", "swa"]
    assert cfg.schedule[2:] == (["full"] + ["reuse"] * 5) * 3
    assert cfg.schedule == [m.value for m in s.encoder_modes()]


def test_schedule_host_logic():
    from sparse_attention_fp4_csa2_gb300 import schedule as s
    dec = s.decoder_modes()
    assert [m.value for m in dec[:8]] == ["full", "reuse", "reuse", "reuse", "reindex", "reuse", "reuse", "reuse"]
    assert len(dec) == 20 and sum(m == s.Mode.REINDEX for m in dec) == 4
    enc = s.encoder_modes()
    assert len(enc) == 20 and sum(m == s.Mode.FULL for m in enc) == 3
    s.validate(dec)
    with pytest.raises(ValueError):
        s.validate(["reuse", "full"])


def test_global_cache_bytes_per_token_from_library_sizes(c2):
    """The pages' 890 B/token ("DeepSeek-v4.1 Flash: Pushing the Limits of KV
    Cache Compression", section 3.1): three encoder copies at m = 2 and one
    decoder copy at m = 1, each adding a main-KV and an MXFP4 indexer-K entry,
    from this library's own entry sizes and schedules."""
    import json
    from sparse_attention_fp4_csa2_gb300 import schedule as s
    facts = json.load(open(os.path.join(ROOT, "tests", "golden", "pages_facts.json")))
    lay = facts["model_layers"]
    enc, dec = s.encoder_modes(), s.decoder_modes()
    assert len(enc) == lay["encoder_layers"] and len(dec) == lay["decoder_layers"]
    assert s.cache_copies(enc) == lay["encoder_groups"] and s.cache_copies(dec) == 1
    got = s.global_kv_bytes_per_token(c2.entry_bytes(), c2.indexer_entry_bytes(True), enc, dec,
                                      m_encoder=lay["encoder_m"], m_decoder=lay["decoder_m"])
    assert got == facts["global_kv_bytes_per_token"]["value"]
    # with the bf16 indexer entry the same schedule grows 1,360 B per token
    assert s.global_kv_bytes_per_token(c2.entry_bytes(), c2.indexer_entry_bytes(False), enc, dec) == 1360
