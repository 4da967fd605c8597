"""Python binding of the CSA2 sparse FP4 decode library (libcsa2.so).

Thin ctypes marshalling over the C ABI declared in ``include/csa2.h``: every
function here has the C call's name without the ``csa2_`` prefix, takes torch
CUDA tensors, passes their device pointers and the current CUDA stream, and
raises ``Csa2Error`` on a non-OK status.  All computation happens in the CUDA
kernels of the library; there is no CPU path.  If the library has not been
built (``python -m sparse_attention_fp4_csa2_gb300.build``, or
``__graft_entry__.build()``), importing the kernels raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .schedule import decoder_modes, Mode  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libcsa2.so")

D, ROPE_DIM, H, HI, DI, ENTRY_BYTES, BLOCK = 512, 64, 64, 32, 128, 288, 8

OP_INDEXER, OP_POOL, OP_ATTN, OP_DECODE = 0, 1, 2, 3
MODE = {"full": 0, "reindex": 1, "reuse": 2}
DEV_ERR = {0x1: "n_vis out of range", 0x2: "index out of range", 0x4: "bounded wait timed out",
           0x8: "pool block out of range"}


class Csa2Error(RuntimeError):
    pass


class Params(ctypes.Structure):
    """csa2_params: index_topk, sliding_window, candidate_block_size,
    candidate_topk_blocks, block_reduce (0 max, 1 sum), hsi, attn_kernel (0
    automatic, 1 keys split over a cluster, 2 one CTA per token), indexer_fp4 (0 bf16 indexer K
    cache, 1 MXFP4 planes written by ``indexer_k_quant``)."""
    _fields_ = [("index_topk", ctypes.c_int32), ("sliding_window", ctypes.c_int32),
                ("candidate_block_size", ctypes.c_int32), ("candidate_topk_blocks", ctypes.c_int32),
                ("block_reduce", ctypes.c_int32), ("hsi", ctypes.c_int32), ("attn_kernel", ctypes.c_int32),
                ("indexer_fp4", ctypes.c_int32)]

    @classmethod
    def make(cls, index_topk=512, sliding_window=128, candidate_block_size=8, candidate_topk_blocks=2048,
             block_reduce=0, hsi=1, attn_kernel=0, indexer_fp4=0):
        return cls(index_topk, sliding_window, candidate_block_size, candidate_topk_blocks, block_reduce, hsi,
                   attn_kernel, indexer_fp4)


_lib = None


def lib():
    """Load libcsa2.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise Csa2Error(f"CSA2 CUDA library not built: {LIB_PATH} is missing "
                            "(run sparse_attention_fp4_csa2_gb300.build.build())")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        PP = ctypes.POINTER(Params)
        L.csa2_default_params.argtypes, L.csa2_default_params.restype = [], Params
        L.csa2_entry_bytes.argtypes, L.csa2_entry_bytes.restype = [], i32
        L.csa2_indexer_entry_bytes.argtypes, L.csa2_indexer_entry_bytes.restype = [i32], i32
        L.csa2_last_launch_count.argtypes, L.csa2_last_launch_count.restype = [], i32
        L.csa2_status_string.argtypes, L.csa2_status_string.restype = [ctypes.c_int], ctypes.c_char_p
        L.csa2_workspace_bytes.argtypes, L.csa2_workspace_bytes.restype = [ctypes.c_int, i32, i64, PP], sz
        L.csa2_get_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
        L.csa2_get_device_status.restype = ctypes.c_int
        L.csa2_kv_quant_write.argtypes = [P, P, i32, i64, P, P, P, i64, f32, P]
        L.csa2_indexer_k_quant.argtypes = [P, i64, P, P, i64, P]
        L.csa2_kv_quant_write_ik.argtypes = [P, P, i32, i64, P, P, P, i64, f32, P, P, i64, i32, P]
        L.csa2_indexer_score_topk.argtypes = [P, P, P, i32, i64, P, i64, P, PP, P, P, P, sz, P]
        L.csa2_hier_pool_select.argtypes = [P, P, i32, i64, PP, P, P, sz, P]
        L.csa2_sparse_attn.argtypes = [PP, i32, P, P, i64, P, P, P, P, P, P, P, sz, P]
        L.csa2_sparse_decode.argtypes = [ctypes.c_int, PP, i32, P, P, P, P, P, i64, P, i64, P, P, P, P, P, P, P, P,
                                         sz, P]
        L.csa2_prefill_chunk.argtypes = [PP, i32, i32, i64, i32, P, P, P, P, P, i64, P, P, i64, i64, P, P, P, P, sz, P]
        L.csa2_prefill_chunk.restype = ctypes.c_int
        L.csa2_set_profile_events.argtypes, L.csa2_set_profile_events.restype = [ctypes.c_int, P, P], ctypes.c_int
        L.csa2_set_topk_kernel.argtypes, L.csa2_set_topk_kernel.restype = [ctypes.c_int32], ctypes.c_int
        for f in ("csa2_kv_quant_write", "csa2_kv_quant_write_ik", "csa2_indexer_k_quant", "csa2_indexer_score_topk", "csa2_hier_pool_select",
                  "csa2_sparse_attn", "csa2_sparse_decode"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int, what: str):
    if status != 0:
        raise Csa2Error(f"{what}: {lib().csa2_status_string(status).decode()} (status {status})")


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise Csa2Error(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise Csa2Error(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise Csa2Error(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def default_params() -> Params:
    return lib().csa2_default_params()


def entry_bytes() -> int:
    return lib().csa2_entry_bytes()


def indexer_entry_bytes(fp4: bool = False) -> int:
    return lib().csa2_indexer_entry_bytes(int(bool(fp4)))


def last_launch_count() -> int:
    """Kernels enqueued by the last successful call made on this thread."""
    return lib().csa2_last_launch_count()


def workspace_bytes(op: int, batch: int, n_max: int, params: Params) -> int:
    return int(lib().csa2_workspace_bytes(op, batch, n_max, ctypes.byref(params)))


def workspace(op: int, batch: int, n_max: int, params: Params, device=None) -> torch.Tensor:
    """A caller-owned scratch buffer of the size the operation needs, zeroed
    (the indexer keeps per-row counts in it between its kernels and leaves
    them zero: a zeroed buffer lets the first call use them too)."""
    n = workspace_bytes(op, batch, n_max, params)
    if n == 0:
        raise Csa2Error("invalid workspace request")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error bits."""
    bits = ctypes.c_uint32(0)
    st = lib().csa2_get_device_status(_stream(stream), ctypes.byref(bits))
    if st not in (0, 5):
        _check(st, "csa2_get_device_status")
    return int(bits.value)


def kv_quant_write(latent, z, m, entry_pos, slot, kv, rope_theta=10000.0, stream=None):
    """latent/z bf16 [n, m, 512] (z None at m=1); entry_pos, slot int64 [n]; kv uint8 [rows, 288]."""
    n = entry_pos.numel()
    _check(lib().csa2_kv_quant_write(_ptr(latent, torch.bfloat16, "latent"), _ptr(z, torch.bfloat16, "z"), m, n,
                                     _ptr(entry_pos, torch.int64, "entry_pos"), _ptr(slot, torch.int64, "slot"),
                                     _ptr(kv, torch.uint8, "kv"), kv.numel() // ENTRY_BYTES, float(rope_theta),
                                     _stream(stream)), "csa2_kv_quant_write")


def kv_quant_write_ik(latent, z, m, entry_pos, slot, kv, w_ik, k_idx, indexer_fp4=False, rope_theta=10000.0,
                     stream=None):
    """kv_quant_write plus each entry's indexer key W_ik e: w_ik bf16 [128, 512];
    k_idx bf16 [rows, 128] or, with indexer_fp4, an MXFP4 cache of
    ``indexer_k_fp4_cache``."""
    n = entry_pos.numel()
    if indexer_fp4:
        k_ptr, k_rows = _ptr(k_idx, torch.uint8, "k_idx"), k_idx.numel() // FP4_ENTRY_BYTES
    else:
        k_ptr, k_rows = _ptr(k_idx, torch.bfloat16, "k_idx"), k_idx.numel() // 128
    _check(lib().csa2_kv_quant_write_ik(_ptr(latent, torch.bfloat16, "latent"), _ptr(z, torch.bfloat16, "z"), m, n,
                                        _ptr(entry_pos, torch.int64, "entry_pos"), _ptr(slot, torch.int64, "slot"),
                                        _ptr(kv, torch.uint8, "kv"), kv.numel() // ENTRY_BYTES, float(rope_theta),
                                        _ptr(w_ik, torch.bfloat16, "w_ik"), k_ptr, k_rows, int(bool(indexer_fp4)),
                                        _stream(stream)), "csa2_kv_quant_write_ik")


FP4_ENTRY_BYTES = 68


def indexer_k_fp4_cache(rows: int, device=None) -> torch.Tensor:
    """An MXFP4 indexer-K cache of `rows` entries (rows a multiple of 4): the
    codes plane [rows][64] followed by the scales plane [rows][4]."""
    if rows % 4:
        raise Csa2Error("MXFP4 indexer cache rows must be a multiple of 4")
    return torch.zeros(rows * FP4_ENTRY_BYTES, dtype=torch.uint8, device=device or "cuda")


def indexer_k_fp4_planes(k_fp4: torch.Tensor):
    """Views (codes [rows, 64], scales [rows, 4]) of an MXFP4 indexer-K cache."""
    rows = k_fp4.numel() // FP4_ENTRY_BYTES
    return k_fp4[:rows * 64].view(rows, 64), k_fp4[rows * 64:rows * FP4_ENTRY_BYTES].view(rows, 4)


def indexer_k_quant(k, slot, k_fp4, stream=None):
    """k bf16 [n, 128]; slot int64 [n]; k_fp4 uint8 cache of ``indexer_k_fp4_cache``."""
    n = slot.numel()
    _check(lib().csa2_indexer_k_quant(_ptr(k, torch.bfloat16, "k"), n, _ptr(slot, torch.int64, "slot"),
                                      _ptr(k_fp4, torch.uint8, "k_fp4"), k_fp4.numel() // FP4_ENTRY_BYTES,
                                      _stream(stream)), "csa2_indexer_k_quant")


def _k_idx(k_idx, params, batch, cap):
    """Pointer to the indexer K cache: bf16 [B, cap, 128], or with
    params.indexer_fp4 the uint8 MXFP4 cache of exactly B * cap rows (its
    scale plane starts after B * cap rows of codes)."""
    if k_idx is None:
        return None
    if params.indexer_fp4:
        if k_idx.numel() != batch * cap * FP4_ENTRY_BYTES:
            raise Csa2Error(f"k_idx: an MXFP4 cache of {batch} x {cap} rows has {batch * cap * FP4_ENTRY_BYTES} "
                            f"bytes, got {k_idx.numel()}")
        return _ptr(k_idx, torch.uint8, "k_idx")
    if k_idx.numel() != batch * cap * 128:
        raise Csa2Error(f"k_idx: expected bf16 [{batch}, {cap}, 128]")
    return _ptr(k_idx, torch.bfloat16, "k_idx")


def indexer_score_topk(q_idx, w, k_idx, n_vis, n_max, params, topk_idx, ws, pool_blocks=None, block_scores=None,
                       stream=None):
    """q_idx bf16 [B,32,128]; w fp32 [B,32]; k_idx bf16 [B,cap,128] (with params.indexer_fp4 the
    uint8 MXFP4 cache of B*cap rows); n_vis int32 [B]; topk_idx int32 [B,K] (out);
    block_scores fp32 [B, ceil(n_max/8)] (out, Full) or None."""
    B = q_idx.shape[0]
    cap = k_idx.numel() // (B * FP4_ENTRY_BYTES) if params.indexer_fp4 else k_idx.shape[1]
    _check(lib().csa2_indexer_score_topk(
        _ptr(q_idx, torch.bfloat16, "q_idx"), _ptr(w, torch.float32, "w"), _k_idx(k_idx, params, B, cap),
        B, cap, _ptr(n_vis, torch.int32, "n_vis"), int(n_max), _ptr(pool_blocks, torch.int32, "pool_blocks"),
        ctypes.byref(params), _ptr(topk_idx, torch.int32, "topk_idx"),
        _ptr(block_scores, torch.float32, "block_scores"), _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
        _stream(stream)), "csa2_indexer_score_topk")


def hier_pool_select(block_scores, n_vis, n_max, params, pool_blocks, ws, stream=None):
    """block_scores fp32 [B, ceil(n_max/8)]; pool_blocks int32 [B, candidate_topk_blocks] (out)."""
    B = block_scores.shape[0]
    _check(lib().csa2_hier_pool_select(
        _ptr(block_scores, torch.float32, "block_scores"), _ptr(n_vis, torch.int32, "n_vis"), B, int(n_max),
        ctypes.byref(params), _ptr(pool_blocks, torch.int32, "pool_blocks"), _ptr(ws, None, "ws"),
        ws.numel() * ws.element_size(), _stream(stream)), "csa2_hier_pool_select")


def sparse_attn(params, q, kv, topk_idx, swa, swa_scale, swa_len, out, ws, lse=None, stream=None):
    """q bf16 [B,64,512]; kv uint8 [B,cap,288]; topk_idx int32 [B,K]; swa uint8 [B,W,512];
    swa_scale fp32 [B,W]; swa_len int32 [B]; out fp32 [B,64,512]; lse fp32 [B,64] or None."""
    B, cap = kv.shape[0], kv.shape[1]
    _check(lib().csa2_sparse_attn(
        ctypes.byref(params), B, _ptr(q, torch.bfloat16, "q"), _ptr(kv, torch.uint8, "kv"), cap,
        _ptr(topk_idx, torch.int32, "topk_idx"), _ptr(swa, torch.uint8, "swa"),
        _ptr(swa_scale, torch.float32, "swa_scale"), _ptr(swa_len, torch.int32, "swa_len"),
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"), _ptr(ws, None, "ws"),
        ws.numel() * ws.element_size(), _stream(stream)), "csa2_sparse_attn")


def sparse_decode(mode, params, q, kv, n_vis, n_max, swa, swa_scale, swa_len, topk_idx, out, ws, q_idx=None,
                  w=None, k_idx=None, pool_blocks=None, lse=None, stream=None):
    """One CSA2 layer of a decode step; mode is 'full', 'reindex' or 'reuse'."""
    B, cap = kv.shape[0], kv.shape[1]
    _check(lib().csa2_sparse_decode(
        MODE[mode] if isinstance(mode, str) else int(mode), ctypes.byref(params), B,
        _ptr(q, torch.bfloat16, "q"), _ptr(q_idx, torch.bfloat16, "q_idx"), _ptr(w, torch.float32, "w"),
        _ptr(kv, torch.uint8, "kv"), _k_idx(k_idx, params, B, cap), cap,
        _ptr(n_vis, torch.int32, "n_vis"), int(n_max), _ptr(swa, torch.uint8, "swa"),
        _ptr(swa_scale, torch.float32, "swa_scale"), _ptr(swa_len, torch.int32, "swa_len"),
        _ptr(topk_idx, torch.int32, "topk_idx"), _ptr(pool_blocks, torch.int32, "pool_blocks"),
        _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"), _ptr(ws, None, "ws"),
        ws.numel() * ws.element_size(), _stream(stream)), "csa2_sparse_decode")


KERNEL_INDEXER_SWEEP, KERNEL_SPARSE_ATTN, KERNEL_PREFILL_INDEXER, KERNEL_TOPK = 0, 1, 2, 3


def set_profile_events(kernel: int, start=None, stop=None):
    """Record torch.cuda.Event `start` / `stop` around every launch of the
    chosen kernel by later calls on this thread (None, None switches it off)."""
    sp = ctypes.c_void_p(start.cuda_event) if start is not None else None
    ep = ctypes.c_void_p(stop.cuda_event) if stop is not None else None
    _check(lib().csa2_set_profile_events(kernel, sp, ep), "csa2_set_profile_events")


TOPK_AUTO, TOPK_CLUSTER, TOPK_ROW = 0, 1, 2


def set_topk_kernel(which: int):
    """Kernel of the top-K selections made by later calls in this process:
    TOPK_AUTO, TOPK_CLUSTER (one thread-block cluster per row) or TOPK_ROW
    (one CTA per row, rows of at most 131,072 scores)."""
    _check(lib().csa2_set_topk_kernel(which), "csa2_set_topk_kernel")


OP_PREFILL = 4


def prefill_chunk(params, q, q_idx, w, kv, k_idx, first_pos, m, swa, swa_scale, swa_first_pos, topk_idx, out,
                  ws, lse=None, stream=None):
    """Every token of a prefill chunk: indexer over its visible entries, top-K,
    readout with its causal SWA window.  q bf16 [B,T,64,512]; q_idx bf16
    [B,T,32,128]; w fp32 [B,T,32]; kv uint8 [B,cap,288]; k_idx bf16 [B,cap,128];
    swa uint8 [B,rows,512] + swa_scale fp32 [B,rows] (row r = position
    swa_first_pos + r); topk_idx int32 [B,T,K]; out fp32 [B,T,64,512]."""
    B, T = q.shape[0], q.shape[1]
    cap = kv.shape[1]
    _check(lib().csa2_prefill_chunk(
        ctypes.byref(params), B, T, int(first_pos), int(m), _ptr(q, torch.bfloat16, "q"),
        _ptr(q_idx, torch.bfloat16, "q_idx"), _ptr(w, torch.float32, "w"), _ptr(kv, torch.uint8, "kv"),
        _ptr(k_idx, torch.bfloat16, "k_idx"), cap, _ptr(swa, torch.uint8, "swa"),
        _ptr(swa_scale, torch.float32, "swa_scale"), swa.shape[1], int(swa_first_pos),
        _ptr(topk_idx, torch.int32, "topk_idx"), _ptr(out, torch.float32, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _stream(stream)), "csa2_prefill_chunk")
