"""ctypes front end of the fp64 CPU oracle (``mla_oracle.c``).

TEST INFRASTRUCTURE: only the test suite, ``__graft_entry__.smoke()`` and the
bench's ``cpu_baseline`` / reference leg may import this module. The CUDA
library never calls it and it never calls the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_SO = os.path.join(_HERE, "libmla_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, fp64, OpenMP; no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        i32, i64, vp, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
        L.ora_e4m3.restype = dbl
        L.ora_e4m3.argtypes = [ctypes.c_uint8]
        L.ora_bf16.restype = dbl
        L.ora_bf16.argtypes = [ctypes.c_uint16]
        L.ora_bf16_to_f64.argtypes = [vp, i64, vp]
        seq = [i32, vp, vp, vp, i32, i32]
        L.ora_mla_dense.restype = ctypes.c_int
        L.ora_mla_dense.argtypes = seq + [vp, vp, i64, i32, vp, vp, dbl, vp, vp]
        L.ora_mla_sparse.restype = ctypes.c_int
        L.ora_mla_sparse.argtypes = seq + [vp, vp, i64, i32, vp, vp, dbl, vp, i32, vp, vp]
        L.ora_mla_dense_fmt.restype = ctypes.c_int
        L.ora_mla_dense_fmt.argtypes = [ctypes.c_int] + seq + [vp, vp, i64, i32, vp, vp, dbl, vp, vp]
        L.ora_mla_sparse_fmt.restype = ctypes.c_int
        L.ora_mla_sparse_fmt.argtypes = [ctypes.c_int] + seq + [vp, vp, i64, i32, vp, vp, dbl, vp, i32, vp, vp]
        L.ora_mla_mha.restype = ctypes.c_int
        L.ora_mla_mha.argtypes = seq + [vp, vp, i64, i32, vp, vp, vp, dbl, vp, vp]
        L.ora_indexer_topk.restype = ctypes.c_int
        L.ora_indexer_topk.argtypes = seq + [vp, vp, i64, vp, i64, vp, vp, i32, vp, vp, i64]
        L.ora_e4m3_nearest.restype = ctypes.c_uint8
        L.ora_e4m3_nearest.argtypes = [ctypes.c_float]
        L.ora_quantize_row.restype = None
        L.ora_quantize_row.argtypes = [vp, i64, vp, vp]
        L.ora_kv_append.restype = ctypes.c_int
        L.ora_kv_append.argtypes = seq + [vp, vp, vp, vp, vp, vp]
        L.ora_merge.restype = None
        L.ora_merge.argtypes = [i32, vp, vp, i64, i64, vp, vp]
        _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def e4m3_value(code: int) -> float:
    return lib().ora_e4m3(code)


def bf16_value(bits: int) -> float:
    return lib().ora_bf16(bits)


def bf16_to_f64(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib().ora_bf16_to_f64(_p(b), b.size, _p(out))
    return out


def _seq_args(seqs):
    cu = _c(seqs.cu_seqlens_q, np.int32)
    pl = _c(seqs.prefix_lens, np.int32)
    bt = _c(seqs.block_table, np.int32)
    return (cu, pl, bt), [seqs.batch, _p(cu), _p(pl), _p(bt), bt.shape[1], seqs.num_blocks]


def mla_dense(seqs, q, tokens, kv, kv_scale, sm_scale):
    """fp64 dense causal MLA for the selected tokens.
    q: bf16 bits [n, H, 576] (uint16) or fp64 values; returns (out [n,H,512], lse [n,H])."""
    q = np.asarray(q)
    qd = bf16_to_f64(q) if q.dtype == np.uint16 else _c(q, np.float64)
    n, H = qd.shape[0], qd.shape[1]
    tok = _c(tokens, np.int64)
    if tok.shape != (n,) or qd.shape[2] != 576:
        raise ValueError("q must be [len(tokens), H, 576]")
    kvc, kvs = _c(kv, np.uint8), _c(kv_scale, np.float32)
    keep, sa = _seq_args(seqs)
    out = np.zeros((n, H, 512), dtype=np.float64)
    lse = np.zeros((n, H), dtype=np.float64)
    rc = lib().ora_mla_dense(*sa, _p(qd), _p(tok), n, H, _p(kvc), _p(kvs), float(sm_scale), _p(out), _p(lse))
    if rc != 0:
        raise ValueError(f"oracle dense: {-rc} rows failed (token out of range or unmapped page)")
    return out, lse


def mla_sparse(seqs, q, tokens, kv, kv_scale, sm_scale, idx):
    """fp64 sparse MLA for the selected tokens over idx [n, topk] (-1 = padding)."""
    q = np.asarray(q)
    qd = bf16_to_f64(q) if q.dtype == np.uint16 else _c(q, np.float64)
    n, H = qd.shape[0], qd.shape[1]
    ix = _c(idx, np.int32)
    tok = _c(tokens, np.int64)
    if tok.shape != (n,) or ix.shape[0] != n or qd.shape[2] != 576:
        raise ValueError("q must be [len(tokens), H, 576] and idx [len(tokens), topk]")
    kvc, kvs = _c(kv, np.uint8), _c(kv_scale, np.float32)
    keep, sa = _seq_args(seqs)
    out = np.zeros((n, H, 512), dtype=np.float64)
    lse = np.zeros((n, H), dtype=np.float64)
    rc = lib().ora_mla_sparse(*sa, _p(qd), _p(tok), n, H, _p(kvc), _p(kvs), float(sm_scale),
                              _p(ix), ix.shape[1], _p(out), _p(lse))
    if rc != 0:
        raise ValueError(f"oracle sparse: {-rc} rows failed")
    return out, lse



FMT_656 = 1


def mla_dense_ds(seqs, q, tokens, kv_ds, sm_scale):
    """fp64 dense causal MLA over a cache of 656-byte rows [num_blocks, 256, 656]
    (512 e4m3 latent codes, four fp32 scales, 64 bf16 RoPE values per token).
    q: bf16 bits [n, H, 576] (uint16) or fp64; returns (out [n,H,512], lse [n,H])."""
    q = np.asarray(q)
    qd = bf16_to_f64(q) if q.dtype == np.uint16 else _c(q, np.float64)
    n, H = qd.shape[0], qd.shape[1]
    tok = _c(tokens, np.int64)
    if tok.shape != (n,) or qd.shape[2] != 576:
        raise ValueError("q must be [len(tokens), H, 576]")
    kvc = _c(kv_ds, np.uint8)
    if kvc.shape[-1] != 656:
        raise ValueError("kv_ds must hold 656-byte rows")
    keep, sa = _seq_args(seqs)
    out = np.zeros((n, H, 512), dtype=np.float64)
    lse = np.zeros((n, H), dtype=np.float64)
    dummy = np.ones(1, dtype=np.float32)
    rc = lib().ora_mla_dense_fmt(FMT_656, *sa, _p(qd), _p(tok), n, H, _p(kvc), _p(dummy), float(sm_scale), _p(out),
                                 _p(lse))
    if rc != 0:
        raise ValueError(f"oracle dense: {-rc} rows failed (token out of range or unmapped page)")
    return out, lse


def mla_sparse_ds(seqs, q, tokens, kv_ds, sm_scale, idx):
    """fp64 sparse MLA over idx [n, topk] (-1 = padding) on 656-byte rows."""
    q = np.asarray(q)
    qd = bf16_to_f64(q) if q.dtype == np.uint16 else _c(q, np.float64)
    n, H = qd.shape[0], qd.shape[1]
    ix = _c(idx, np.int32)
    tok = _c(tokens, np.int64)
    if tok.shape != (n,) or ix.shape[0] != n or qd.shape[2] != 576:
        raise ValueError("q must be [len(tokens), H, 576] and idx [len(tokens), topk]")
    kvc = _c(kv_ds, np.uint8)
    if kvc.shape[-1] != 656:
        raise ValueError("kv_ds must hold 656-byte rows")
    keep, sa = _seq_args(seqs)
    out = np.zeros((n, H, 512), dtype=np.float64)
    lse = np.zeros((n, H), dtype=np.float64)
    dummy = np.ones(1, dtype=np.float32)
    rc = lib().ora_mla_sparse_fmt(FMT_656, *sa, _p(qd), _p(tok), n, H, _p(kvc), _p(dummy), float(sm_scale), _p(ix),
                                  ix.shape[1], _p(out), _p(lse))
    if rc != 0:
        raise ValueError(f"oracle sparse: {-rc} rows failed")
    return out, lse

def mla_mha(seqs, q, tokens, kv, kv_scale, w_ukv, sm_scale):
    """fp64 non-absorbed (MHA) dense causal prefill for the selected tokens:
    per head, keys [W_UK_h c_s ; r_s] (192 dims) and values W_UV_h c_s (128
    dims) from the 580-byte cache rows. q: bf16 bits [n, H, 192] (uint16) or
    fp64; w_ukv: bf16 bits or fp64 [H, 256, 512] (rows 0..127 of head h W_UK_h,
    rows 128..255 W_UV_h). Returns (out [n, H, 128], lse [n, H])."""
    q = np.asarray(q)
    qd = bf16_to_f64(q) if q.dtype == np.uint16 else _c(q, np.float64)
    w = np.asarray(w_ukv)
    wd = bf16_to_f64(w) if w.dtype == np.uint16 else _c(w, np.float64)
    n, H = qd.shape[0], qd.shape[1]
    tok = _c(tokens, np.int64)
    if tok.shape != (n,) or qd.shape[2] != 192:
        raise ValueError("q must be [len(tokens), H, 192]")
    if wd.shape != (H, 256, 512):
        raise ValueError("w_ukv must be [H, 256, 512]")
    kvc, kvs = _c(kv, np.uint8), _c(kv_scale, np.float32)
    keep, sa = _seq_args(seqs)
    out = np.zeros((n, H, 128), dtype=np.float64)
    lse = np.zeros((n, H), dtype=np.float64)
    rc = lib().ora_mla_mha(*sa, _p(qd), _p(tok), n, H, _p(kvc), _p(kvs), _p(wd), float(sm_scale), _p(out), _p(lse))
    if rc != 0:
        raise ValueError(f"oracle mha: {-rc} rows failed (token out of range or unmapped page)")
    return out, lse


def indexer_topk(seqs, qi, w, w_stride, tokens, ki, ki_scale, topk, want_scores=False, ctx_cap=0):
    """Exact top-k selection per selected token; returns idx [n, topk] ascending,
    -1 padded (and the fp64 scores [n, ctx_cap] when want_scores)."""
    qc = _c(qi, np.uint8)
    n = qc.shape[0]
    wc = _c(w, np.float32)
    tok = _c(tokens, np.int64)
    if tok.shape != (n,) or qc.shape[1:] != (64, 128):
        raise ValueError("qi must be [len(tokens), 64, 128]")
    if (w_stride == 0 and wc.size < 64) or (w_stride > 0 and wc.size < (n - 1) * w_stride + 64):
        raise ValueError("w too small for its stride")
    kc, ksc = _c(ki, np.uint8), _c(ki_scale, np.float32)
    keep, sa = _seq_args(seqs)
    idx = np.empty((n, topk), dtype=np.int32)
    sc = np.full((n, ctx_cap), np.nan) if want_scores else None
    rc = lib().ora_indexer_topk(*sa, _p(qc), _p(wc), int(w_stride), _p(tok), n, _p(kc), _p(ksc), int(topk),
                                _p(idx), _p(sc) if want_scores else None, int(ctx_cap))
    if rc != 0:
        raise ValueError(f"oracle indexer: {-rc} rows failed")
    return (idx, sc) if want_scores else idx


def e4m3_nearest(v) -> np.ndarray:
    """Nearest e4m3 codes (ties to even, clamped at 448) of float32 values."""
    x = np.ascontiguousarray(v, dtype=np.float32)
    f = lib().ora_e4m3_nearest
    return np.array([f(float(a)) for a in x.ravel()], dtype=np.uint8).reshape(x.shape)


def quantize_row(x_bf16):
    """Per-row absmax/448 quantisation of bf16 bits [n] -> (codes u8 [n], scale f32)."""
    x = _c(x_bf16, np.uint16)
    codes = np.empty(x.shape, dtype=np.uint8)
    sc = ctypes.c_float()
    lib().ora_quantize_row(_p(x), x.size, _p(codes), ctypes.byref(sc))
    return codes, np.float32(sc.value)


def kv_append(seqs, latent, kidx, kv, kv_scale, ki=None, ki_scale=None):
    """Write the new tokens' quantised rows into copies of the caches.
    latent: bf16 bits [Tq, 576]; kidx: bf16 bits [Tq, 128] or None.
    Returns (kv, kv_scale, ki, ki_scale) (the last two None without kidx)."""
    lat = _c(latent, np.uint16)
    if lat.ndim != 2 or lat.shape[1] != 576 or lat.shape[0] != int(seqs.cu_seqlens_q[-1]):
        raise ValueError("latent must be [Tq, 576]")
    kvc, kvs = np.array(kv, dtype=np.uint8, order="C"), np.array(kv_scale, dtype=np.float32, order="C")
    kic = kis = kx = None
    if kidx is not None:
        kx = _c(kidx, np.uint16)
        if kx.shape != (lat.shape[0], 128):
            raise ValueError("kidx must be [Tq, 128]")
        kic, kis = np.array(ki, dtype=np.uint8, order="C"), np.array(ki_scale, dtype=np.float32, order="C")
    keep, sa = _seq_args(seqs)
    rc = lib().ora_kv_append(*sa, _p(lat), _p(kx) if kx is not None else None, _p(kvc), _p(kvs),
                             _p(kic) if kic is not None else None, _p(kis) if kis is not None else None)
    if rc != 0:
        raise ValueError(f"oracle kv append: {-rc} tokens have no valid page")
    return kvc, kvs, kic, kis


def merge(outs, lses):
    """Merge partial results over disjoint key sets: outs [n, rows, dv] (fp64, or
    bf16 bits as uint16), lses [n, rows] (natural log, -inf = empty part).
    Returns (out [rows, dv], lse [rows]) in fp64."""
    o = np.asarray(outs)
    od = bf16_to_f64(o) if o.dtype == np.uint16 else _c(o, np.float64)
    ls = _c(lses, np.float64)
    n, rows, dv = od.shape
    if ls.shape != (n, rows):
        raise ValueError("lses must be [n_parts, rows]")
    out = np.empty((rows, dv), dtype=np.float64)
    lse = np.empty(rows, dtype=np.float64)
    lib().ora_merge(n, _p(od), _p(ls), rows, dv, _p(out), _p(lse))
    return out, lse
