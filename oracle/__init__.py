"""The CSA2 ORACLE -- test infrastructure, not part of the product.

A plain fp64 CPU implementation (``csa2_oracle.c``) of the decode-time CSA2
path, loaded through ctypes.  Only the tests, ``__graft_entry__.smoke()`` and
the benchmark's ``cpu_baseline`` / ``--impl reference`` legs may import it.
It shares no code with the CUDA library and never calls it.

Every function states the passage it follows in the C source.  Functions
marked "parity unpinned" there (RoPE constants, m=2 pooling form) restate a
convention the pages leave open; everything else is pinned by the tests in
``tests/test_oracle_*.py`` against values fixed by the pages, library
routines, closed forms and brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa2_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libcsa2_oracle.so")

D, ROPE_DIM, H, HI, DI, GROUP, ENTRY_BYTES = 512, 64, 64, 32, 128, 16, 288


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if available, else serial)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-std=gnu11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:-1] + ["-fopenmp", "-lm"], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, f32, f64, u8, i32 = ctypes.c_int64, ctypes.c_float, ctypes.c_double, ctypes.c_uint8, ctypes.c_int
        L.csa2o_e4m3_decode.argtypes, L.csa2o_e4m3_decode.restype = [u8], f64
        L.csa2o_e4m3_encode.argtypes, L.csa2o_e4m3_encode.restype = [f32], u8
        L.csa2o_e2m1_decode.argtypes, L.csa2o_e2m1_decode.restype = [u8], f64
        L.csa2o_e2m1_encode.argtypes, L.csa2o_e2m1_encode.restype = [f32], u8
        L.csa2o_rope_tail.argtypes, L.csa2o_rope_tail.restype = [P, i64, f64, P], None
        L.csa2o_compress.argtypes, L.csa2o_compress.restype = [P, P, i32, P], None
        L.csa2o_fp4_quantise.argtypes, L.csa2o_fp4_quantise.restype = [P, P], None
        L.csa2o_fp4_dequant.argtypes, L.csa2o_fp4_dequant.restype = [P, P], None
        L.csa2o_kv_entry.argtypes, L.csa2o_kv_entry.restype = [P, P, i32, i64, f64, P], None
        L.csa2o_kv_entries.argtypes, L.csa2o_kv_entries.restype = [P, P, i32, i64, P, f64, P], None
        L.csa2o_indexer_k_project.argtypes = [P, P, i32, i64, P, f64, P, P]
        L.csa2o_indexer_k_project.restype = None
        L.csa2o_index_scores.argtypes, L.csa2o_index_scores.restype = [P, P, P, i64, P], None
        L.csa2o_mxfp4_quantise.argtypes, L.csa2o_mxfp4_quantise.restype = [P, P, P], None
        L.csa2o_mxfp4_quantise_rows.argtypes, L.csa2o_mxfp4_quantise_rows.restype = [P, i64, P, P], None
        L.csa2o_mxfp4_dequant.argtypes, L.csa2o_mxfp4_dequant.restype = [P, P, P], None
        L.csa2o_index_scores_mxfp4.argtypes, L.csa2o_index_scores_mxfp4.restype = [P, P, P, P, i64, P], None
        L.csa2o_topk.argtypes, L.csa2o_topk.restype = [P, P, i64, i64, P], i64
        L.csa2o_block_scores.argtypes, L.csa2o_block_scores.restype = [P, i64, i32, i32, P], None
        L.csa2o_hsi_pool.argtypes, L.csa2o_hsi_pool.restype = [P, i64, i32, i64, i32, P], i64
        L.csa2o_sparse_attn.argtypes, L.csa2o_sparse_attn.restype = [P, P, P, i64, P, P, i64, P, P, P], None
        L.csa2o_num_threads.argtypes, L.csa2o_num_threads.restype = [], i32
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    """bf16 data as its uint16 bit patterns (accepts a torch bf16 tensor or uint16 array)."""
    if hasattr(a, "view") and hasattr(a, "dtype") and "bfloat16" in str(a.dtype):
        import torch
        return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    return np.ascontiguousarray(np.asarray(a, dtype=np.uint16))


def _np(a, dtype):
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


def num_threads() -> int:
    return lib().csa2o_num_threads()


# ------------------------------------------------------------------ codecs
def e4m3_decode(b: int) -> float:
    return lib().csa2o_e4m3_decode(int(b))


def e4m3_encode(x: float) -> int:
    return lib().csa2o_e4m3_encode(float(x))


def e2m1_decode(c: int) -> float:
    return lib().csa2o_e2m1_decode(int(c))


def e2m1_encode(x: float) -> int:
    return lib().csa2o_e2m1_encode(float(x))


# ------------------------------------------------------------ KV entries
def rope_tail(x, pos: int, base: float = 10000.0) -> np.ndarray:
    x = _np(x, np.float32)
    y = np.empty(D, np.float32)
    lib().csa2o_rope_tail(_p(x), int(pos), float(base), _p(y))
    return y


def compress(x, z, m: int) -> np.ndarray:
    """x, z: bf16 [m, 512] -> fp32 [512] pooled entry (z ignored at m=1)."""
    xx = _u16(x)
    zz = _u16(z) if z is not None else None
    e = np.empty(D, np.float32)
    lib().csa2o_compress(_p(xx), _p(zz), int(m), _p(e))
    return e


def fp4_quantise(x) -> np.ndarray:
    x = _np(x, np.float32)
    out = np.empty(ENTRY_BYTES, np.uint8)
    lib().csa2o_fp4_quantise(_p(x), _p(out))
    return out


def fp4_dequant(entry) -> np.ndarray:
    e = _np(entry, np.uint8)
    out = np.empty(D, np.float64)
    lib().csa2o_fp4_dequant(_p(e), _p(out))
    return out


def kv_entries(latent, z, m: int, pos, base: float = 10000.0) -> np.ndarray:
    """latent (and z): bf16 [n, m, 512] (or [n, 512] at m=1); pos int64 [n] -> uint8 [n, 288]."""
    lat = _u16(latent).reshape(-1, m * D)
    n = lat.shape[0]
    zz = _u16(z).reshape(n, m * D) if z is not None else None
    pp = _np(pos, np.int64).reshape(n)
    out = np.empty((n, ENTRY_BYTES), np.uint8)
    lib().csa2o_kv_entries(_p(lat), _p(zz), int(m), int(n), _p(pp), float(base), _p(out))
    return out


def indexer_k_project(latent, z, m: int, pos, w, base: float = 10000.0):
    """The Full layer's indexer keys: latent (and z) bf16 [n, m, 512] (or
    [n, 512] at m=1), pos int64 [n], w bf16 [128, 512] -> bf16 [n, 128]
    (a torch tensor)."""
    import torch
    lat = _u16(latent).reshape(-1, m * D)
    n = lat.shape[0]
    zz = _u16(z).reshape(n, m * D) if z is not None else None
    pp = _np(pos, np.int64).reshape(n)
    ww = _u16(w).reshape(DI * D)
    out = np.empty((n, DI), np.uint16)
    lib().csa2o_indexer_k_project(_p(lat), _p(zz), int(m), int(n), _p(pp), float(base), _p(ww), _p(out))
    return torch.from_numpy(out.view(np.int16)).view(torch.bfloat16)


# ---------------------------------------------------------------- indexer
def index_scores(q_idx, w, k_rows) -> np.ndarray:
    """q_idx bf16 [32,128], w fp32 [32], k_rows bf16 [n,128] -> fp64 [n]."""
    q = _u16(q_idx).reshape(HI * DI)
    ww = _np(w, np.float32).reshape(HI)
    kk = _u16(k_rows).reshape(-1, DI)
    s = np.empty(kk.shape[0], np.float64)
    lib().csa2o_index_scores(_p(q), _p(ww), _p(kk), int(kk.shape[0]), _p(s))
    return s


# ------------------------------------------------------------------ MXFP4
def mxfp4_quantise(x):
    """Rows [n, 128] (bf16 tensor or float array) -> (codes uint8 [n, 64],
    scales uint8 [n, 4]) by the OCP MX rule (see csa2o_mxfp4_quantise)."""
    if hasattr(x, "dtype") and "bfloat16" in str(x.dtype):
        xx = _u16(x).reshape(-1, DI)
        n = xx.shape[0]
        codes = np.empty((n, DI // 2), np.uint8)
        scales = np.empty((n, DI // 32), np.uint8)
        lib().csa2o_mxfp4_quantise_rows(_p(xx), int(n), _p(codes), _p(scales))
        return codes, scales
    xf = _np(x, np.float32).reshape(-1, DI)
    n = xf.shape[0]
    codes = np.empty((n, DI // 2), np.uint8)
    scales = np.empty((n, DI // 32), np.uint8)
    for r in range(n):
        row = np.ascontiguousarray(xf[r])
        lib().csa2o_mxfp4_quantise(_p(row), _p(codes[r]), _p(scales[r]))
    return codes, scales


def mxfp4_dequant(codes, scales) -> np.ndarray:
    """codes [n, 64], scales [n, 4] -> fp64 [n, 128]."""
    cc = _np(codes, np.uint8).reshape(-1, DI // 2)
    ss = _np(scales, np.uint8).reshape(-1, DI // 32)
    out = np.empty((cc.shape[0], DI), np.float64)
    for r in range(cc.shape[0]):
        lib().csa2o_mxfp4_dequant(_p(np.ascontiguousarray(cc[r])), _p(np.ascontiguousarray(ss[r])), _p(out[r]))
    return out


def index_scores_mxfp4(q_idx, w, k_codes, k_scales) -> np.ndarray:
    """q_idx bf16 [32,128] (quantised to MXFP4 inside), w fp32 [32], MXFP4 keys
    (codes [n,64], scales [n,4]) -> fp64 [n]."""
    q = _u16(q_idx).reshape(HI * DI)
    ww = _np(w, np.float32).reshape(HI)
    cc = _np(k_codes, np.uint8).reshape(-1, DI // 2)
    ss = _np(k_scales, np.uint8).reshape(-1, DI // 32)
    s = np.empty(cc.shape[0], np.float64)
    lib().csa2o_index_scores_mxfp4(_p(q), _p(ww), _p(cc), _p(ss), int(cc.shape[0]), _p(s))
    return s


def topk(scores, k: int, valid=None) -> np.ndarray:
    """Top-k by (score desc, index asc); ascending indices, -1 padded (int64 [k])."""
    s = _np(scores, np.float64)
    v = None if valid is None else _np(valid, np.uint8)
    out = np.empty(k, np.int64)
    lib().csa2o_topk(_p(s), _p(v), int(s.shape[0]), int(k), _p(out))
    return out


def block_scores(scores, n_vis: int, block: int = 8, reduce_sum: bool = False) -> np.ndarray:
    s = _np(scores, np.float64)
    nb = (n_vis + block - 1) // block
    out = np.empty(nb, np.float64)
    lib().csa2o_block_scores(_p(s), int(n_vis), int(block), int(reduce_sum), _p(out))
    return out


def hsi_pool(scores, n_vis: int, block: int = 8, n_blocks: int = 2048, reduce_sum: bool = False) -> np.ndarray:
    s = _np(scores, np.float64)
    out = np.empty(n_blocks, np.int64)
    lib().csa2o_hsi_pool(_p(s), int(n_vis), int(block), int(n_blocks), int(reduce_sum), _p(out))
    return out


def pool_positions(blocks, n_vis: int, block: int = 8) -> np.ndarray:
    """Expand selected block ids to their positions, truncated to [0, n_vis)."""
    b = _np(blocks, np.int64)
    b = b[b >= 0]
    pos = (b[:, None] * block + np.arange(block)[None, :]).reshape(-1)
    return pos[pos < n_vis]


def reindex_topk(q_idx, w, k_all, pool_blocks, n_vis: int, k: int = 512, block: int = 8) -> np.ndarray:
    """Reindex layer: score only the pool's positions, top-k within the pool,
    returned as ascending positions (-1 padded)."""
    pos = pool_positions(pool_blocks, n_vis, block)
    kk = _u16(k_all).reshape(-1, DI)[pos]
    s = index_scores(q_idx, w, kk)
    sel = topk(s, k)
    return np.where(sel >= 0, pos[np.clip(sel, 0, None)], -1)


# -------------------------------------------------------------- attention
def sparse_attn(q, kv_rows, idx, swa, swa_scale, swa_len: int, want_weights: bool = False):
    """q bf16 [64,512]; kv_rows uint8 [rows,288] (idx indexes rows); idx int [k];
    swa uint8 E4M3 [>=swa_len,512]; swa_scale fp32 [>=swa_len].
    Returns (out fp64 [64,512], lse fp64 [64][, weights fp64 [64, k+swa_len]])."""
    qq = _u16(q).reshape(H * D)
    kv = _np(kv_rows, np.uint8).reshape(-1, ENTRY_BYTES)
    ii = _np(idx, np.int64).reshape(-1)
    sw = _np(swa, np.uint8).reshape(-1, D) if swa_len > 0 else np.zeros((1, D), np.uint8)
    ss = _np(swa_scale, np.float32).reshape(-1) if swa_len > 0 else np.zeros(1, np.float32)
    out = np.empty((H, D), np.float64)
    lse = np.empty(H, np.float64)
    wts = np.empty((H, ii.shape[0] + swa_len), np.float64) if want_weights else None
    lib().csa2o_sparse_attn(_p(qq), _p(kv), _p(ii), int(ii.shape[0]), _p(sw), _p(ss), int(swa_len),
                            _p(out), _p(lse), _p(wts))
    return (out, lse, wts) if want_weights else (out, lse)
