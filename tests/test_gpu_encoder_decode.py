"""GPU parity of the encoder's decode group at m = 2 ("DeepSeek-V4.1-Flash -
Architecture", section 2 "Layer schedule": two SWA-only layers, then groups of
one Full and five Reuse layers; "DeepSeek-v4.1 Flash: Pushing the Limits of
KV Cache Compression", sections 2.3.1 and 2.3.3): a decode step whose token
completes an entry pair writes that entry (channel-wise softmax pooling of the
pair, RoPE at position 2j + 1, FP4), the Full layer scores every complete
entry, selects its top-512 and attends with its SWA rows, the Reuse layers
attend with the same selection, and a SWA-only layer attends to its window
alone."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import check_attn, check_lse, check_topk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def c2():
    import sparse_attention_fp4_csa2_gb300.build as b
    b.build()
    import sparse_attention_fp4_csa2_gb300 as c
    return c


@pytest.mark.parametrize("fp4", [False, True])
def test_encoder_group_step_m2(c2, orc, fp4):
    B, E = 2, 3000                     # 6,000 context tokens: 3,000 entries per sequence
    lat = synth.context_latent(61, B, E, m=2)
    z = synth.compression_logits(62, B, E, m=2)
    k = synth.indexer_keys(63, B, E)
    li = [synth.layer_inputs(6400 + i, B) for i in range(3)]   # SWA-only, Full, Reuse
    kv = torch.zeros(B, E, 288, dtype=torch.uint8, device="cuda")
    pos = torch.arange(E, dtype=torch.int64).repeat(B) * 2 + 1
    slot = torch.arange(B * E, dtype=torch.int64)
    old = torch.arange(E) < E - 1
    keep = old.repeat(B)
    # the context before the step: entries 0 .. E-2
    c2.kv_quant_write(lat.reshape(B * E, 2, 512)[keep].cuda(), z.reshape(B * E, 2, 512)[keep].cuda(), 2,
                      pos[keep].cuda(), slot[keep].cuda(), kv.view(B * E, 288))
    p = c2.Params.make(hsi=0, indexer_fp4=int(fp4))
    if fp4:
        k_cache = c2.indexer_k_fp4_cache(B * E)
        c2.indexer_k_quant(k.reshape(B * E, 128)[keep].cuda(), slot[keep].cuda(), k_cache)
    else:
        k_cache = k.clone().cuda()
    # the step: its token completes pair E-1; the Full layer writes that entry
    new = torch.arange(B, dtype=torch.int64) * E + (E - 1)
    c2.kv_quant_write(lat[:, E - 1].contiguous().cuda(), z[:, E - 1].contiguous().cuda(), 2,
                      torch.full((B,), 2 * (E - 1) + 1, dtype=torch.int64).cuda(), new.cuda(), kv.view(B * E, 288))
    if fp4:
        c2.indexer_k_quant(k[:, E - 1].contiguous().cuda(), new.cuda(), k_cache)
    assert c2.get_device_status() == 0
    # the new entry is the oracle's pooled, RoPE'd, FP4-quantised pair
    for b in range(B):
        want = orc.kv_entries(lat[b, E - 1:E], z[b, E - 1:E], 2, np.array([2 * (E - 1) + 1]))
        assert np.array_equal(kv[b, E - 1].cpu().numpy(), want[0])

    ws = c2.workspace(c2.OP_DECODE, B, E, p)
    nv = torch.full((B,), E, dtype=torch.int32, device="cuda")
    topk = torch.empty(B, 512, dtype=torch.int32, device="cuda")
    none = torch.full((B, 512), -1, dtype=torch.int32, device="cuda")
    outs = [torch.empty(B, 64, 512, device="cuda") for _ in range(3)]
    lses = [torch.empty(B, 64, device="cuda") for _ in range(3)]

    def run(mode, i, idx, **kw):
        c2.sparse_decode(mode, p, li[i].q.cuda(), kv, nv, E, li[i].swa.cuda(), li[i].swa_scale.cuda(),
                         li[i].swa_len.cuda(), idx, outs[i], ws, lse=lses[i], **kw)

    run("reuse", 0, none)                                      # SWA-only layer
    run("full", 1, topk, q_idx=li[1].q_idx.cuda(), w=li[1].w.cuda(), k_idx=k_cache)
    run("reuse", 2, topk)
    assert c2.get_device_status() == 0

    topk_h = topk.cpu().numpy()
    no_rows = np.zeros((0, 288), np.uint8)
    for b in range(B):
        o, l = orc.sparse_attn(li[0].q[b], no_rows, np.arange(0), li[0].swa[b], li[0].swa_scale[b], 128)
        check_attn(outs[0][b].cpu().numpy(), o)
        check_lse(lses[0][b].cpu().numpy(), l)
        if fp4:
            codes, scales = orc.mxfp4_quantise(k[b])
            s = orc.index_scores_mxfp4(li[1].q_idx[b], li[1].w[b], codes, scales)
        else:
            s = orc.index_scores(li[1].q_idx[b], li[1].w[b], k[b])
        check_topk(topk_h[b], orc.topk(s, 512), s, n_valid=E)
        # the readouts are checked on the GPU's own selection (it may differ
        # from the oracle's only inside the tie band bounded above)
        sel = topk_h[b][topk_h[b] >= 0]
        rows = orc.kv_entries(lat[b][sel], z[b][sel], 2, sel * 2 + 1)
        for i in (1, 2):
            o, l = orc.sparse_attn(li[i].q[b], rows, np.arange(len(sel)), li[i].swa[b], li[i].swa_scale[b], 128)
            check_attn(outs[i][b].cpu().numpy(), o)
            check_lse(lses[i][b].cpu().numpy(), l)

