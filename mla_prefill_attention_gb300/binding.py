"""Thin Python binding of ``libmla.so`` (the C ABI declared in include/mla.h).

Argument marshalling only: every step of the computation runs in the CUDA
library. PyTorch supplies device memory and the current stream. If the
library is missing or fails to load, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla.so")

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA, MLA_ERR_WORKSPACE = range(5)
MLA_DEVERR_BAD_PAGE, MLA_DEVERR_BAD_INDEX, MLA_DEVERR_TIMEOUT, MLA_DEVERR_INTERNAL = 1, 2, 4, 8
MLA_DEVERR_SEQ_MISMATCH = 16
MLA_OP_DENSE, MLA_OP_INDEXER, MLA_OP_SPARSE, MLA_OP_DENSE_HOST, MLA_OP_MHA, MLA_OP_DENSE_DS = 0, 1, 2, 3, 4, 5

EXPORTS = ("mla_workspace_size", "mla_prefill_dense", "mla_indexer_topk", "mla_prefill_sparse", "mla_last_error",
           "mla_prefill_dense_static", "mla_kv_append", "mla_merge_attn", "mla_prefill_dense_host",
           "mla_prefill_sparse_host", "mla_prefill_dense_ds", "mla_prefill_sparse_ds", "mla_prefill_mha")
DENSE_STATIC_MAX_WORK_ITEMS = 65536
DENSE_HOST_MAX_CHUNKS = 64


class MlaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"status {status}: {msg}")
        self.status = status


class mla_seqs_t(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("cu_seqlens_q", ctypes.c_void_p),
        ("cu_seqlens_q_host", ctypes.c_void_p),
        ("prefix_lens", ctypes.c_void_p),
        ("prefix_lens_host", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
    ]


class mla_sparse_inputs_t(ctypes.Structure):
    _fields_ = [("q_bf16", ctypes.c_void_p), ("qi_e4m3", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("kv_e4m3", ctypes.c_void_p), ("kv_scale", ctypes.c_void_p), ("ki_e4m3", ctypes.c_void_p),
                ("ki_scale", ctypes.c_void_p)]


class mla_sparse_outputs_t(ctypes.Structure):
    _fields_ = [("out_bf16", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("idx", ctypes.c_void_p)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libmla.so (raises if it is absent: build it with build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise FileNotFoundError(f"{path} not built; run mla_prefill_attention_gb300.build.build()")
    L = ctypes.CDLL(path)
    vp, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    L.mla_workspace_size.restype = sz
    L.mla_workspace_size.argtypes = [ctypes.c_int, ctypes.POINTER(mla_seqs_t), i32, i32]
    L.mla_prefill_dense.restype = ctypes.c_int
    L.mla_prefill_dense.argtypes = [ctypes.POINTER(mla_seqs_t), vp, i32, vp, vp, f32, vp, vp, vp, sz, vp, vp]
    L.mla_indexer_topk.restype = ctypes.c_int
    L.mla_indexer_topk.argtypes = [ctypes.POINTER(mla_seqs_t), vp, vp, i64, vp, vp, i32, vp, vp, sz, vp, vp]
    L.mla_prefill_sparse.restype = ctypes.c_int
    L.mla_prefill_sparse.argtypes = [ctypes.POINTER(mla_seqs_t), vp, i32, vp, vp, f32, vp, i32, vp, vp, vp, sz,
                                     vp, vp]
    L.mla_prefill_dense_static.restype = ctypes.c_int
    L.mla_prefill_dense_static.argtypes = [ctypes.POINTER(mla_seqs_t), vp, i32, vp, vp, f32, vp, vp, vp, vp]
    L.mla_prefill_dense_host.restype = ctypes.c_int
    L.mla_prefill_dense_host.argtypes = [ctypes.POINTER(mla_seqs_t), vp, i32, vp, vp, f32, vp, vp, vp, vp, vp, vp, vp,
                                         i32, vp, sz, vp, vp]
    L.mla_prefill_sparse_host.restype = ctypes.c_int
    L.mla_prefill_sparse_host.argtypes = [ctypes.POINTER(mla_seqs_t), i32, f32, i64, i32,
                                          ctypes.POINTER(mla_sparse_inputs_t), ctypes.POINTER(mla_sparse_inputs_t),
                                          ctypes.POINTER(mla_sparse_outputs_t), ctypes.POINTER(mla_sparse_outputs_t),
                                          i32, vp, sz, vp, vp]
    L.mla_prefill_dense_ds.restype = ctypes.c_int
    L.mla_prefill_dense_ds.argtypes = [ctypes.POINTER(mla_seqs_t), vp, i32, vp, f32, vp, vp, vp, sz, vp, vp]
    L.mla_prefill_sparse_ds.restype = ctypes.c_int
    L.mla_prefill_sparse_ds.argtypes = [ctypes.POINTER(mla_seqs_t), vp, i32, vp, f32, vp, i32, vp, vp, vp, vp]
    L.mla_prefill_mha.restype = ctypes.c_int
    L.mla_prefill_mha.argtypes = [ctypes.POINTER(mla_seqs_t), vp, i32, vp, vp, vp, f32, vp, vp, vp, sz, vp, vp]
    L.mla_kv_append.restype = ctypes.c_int
    L.mla_kv_append.argtypes = [ctypes.POINTER(mla_seqs_t), vp, vp, vp, vp, vp, vp, vp, vp]
    L.mla_merge_attn.restype = ctypes.c_int
    L.mla_merge_attn.argtypes = [i32, vp, vp, i64, vp, vp, vp]
    L.mla_last_error.restype = ctypes.c_char_p
    L.mla_last_error.argtypes = []
    _lib = L
    return L


def _check(status: int):
    if status != MLA_OK:
        raise MlaError(status, load().mla_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


class Seqs:
    """Ragged batch over a paged cache: device tensors plus pinned host mirrors."""

    def __init__(self, cu_seqlens_q, prefix_lens, block_table, num_blocks: int, device="cuda"):
        self.cu_host = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
        self.prefix_host = np.ascontiguousarray(prefix_lens, dtype=np.int32)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        self.cu = torch.from_numpy(self.cu_host).to(device)
        self.prefix = torch.from_numpy(self.prefix_host).to(device)
        self.block_table = torch.from_numpy(bt).to(device)
        self.num_blocks = int(num_blocks)
        self.batch = int(self.prefix_host.shape[0])
        self.total_q = int(self.cu_host[-1])
        self.max_blocks = int(bt.shape[1])

    @classmethod
    def from_paged(cls, ps, device="cuda"):
        return cls(ps.cu_seqlens_q, ps.prefix_lens, ps.block_table, ps.num_blocks, device)

    def c(self) -> mla_seqs_t:
        return mla_seqs_t(self.batch, self.cu.data_ptr(), self.cu_host.ctypes.data, self.prefix.data_ptr(),
                          self.prefix_host.ctypes.data, self.block_table.data_ptr(), self.max_blocks,
                          self.num_blocks)


def mla_workspace_size(op: int, seqs: Seqs, num_heads: int = 64, topk: int = 2048) -> int:
    c = seqs.c()
    return int(load().mla_workspace_size(op, ctypes.byref(c), num_heads, topk))


def _workspace(op, seqs, num_heads, topk, workspace):
    n = mla_workspace_size(op, seqs, num_heads, topk)
    if workspace is None and n > 0:
        workspace = torch.empty(n, dtype=torch.uint8, device=seqs.cu.device)
    return workspace, (0 if workspace is None else workspace.numel() * workspace.element_size())


def mla_prefill_dense(seqs: Seqs, q: torch.Tensor, kv: torch.Tensor, kv_scale: torch.Tensor, sm_scale: float,
                      out=None, lse=None, want_lse: bool = True, workspace=None, dev_err=None):
    """Dense causal MLA prefill. q bf16 [Tq,H,576]; kv uint8 [nb,256,576]; kv_scale f32 [nb,256].
    Returns (out bf16 [Tq,H,512], lse f32 [Tq,H] or None)."""
    H = q.shape[1]
    if out is None:
        out = torch.empty((q.shape[0], H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((q.shape[0], H), dtype=torch.float32, device=q.device)
    ws, wsb = _workspace(MLA_OP_DENSE, seqs, H, 0, workspace)
    c = seqs.c()
    _check(load().mla_prefill_dense(ctypes.byref(c), _ptr(q), H, _ptr(kv), _ptr(kv_scale), float(sm_scale),
                                    _ptr(out), _ptr(lse), _ptr(ws), wsb, _ptr(dev_err), _stream()))
    return out, lse


def mla_prefill_mha(seqs: Seqs, q: torch.Tensor, w_ukv: torch.Tensor, kv: torch.Tensor, kv_scale: torch.Tensor,
                    sm_scale: float, out=None, lse=None, want_lse: bool = True, workspace=None, dev_err=None):
    """Non-absorbed (MHA) dense causal prefill. q bf16 [Tq,H,192] (128 no-RoPE dims,
    then 64 RoPE dims); w_ukv bf16 [H,256,512] (rows 0..127 of head h W_UK_h, rows
    128..255 W_UV_h); kv uint8 [nb,256,576]; kv_scale f32 [nb,256].
    Returns (out bf16 [Tq,H,128], lse f32 [Tq,H] or None)."""
    H = q.shape[1]
    if out is None:
        out = torch.empty((q.shape[0], H, 128), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((q.shape[0], H), dtype=torch.float32, device=q.device)
    ws, wsb = _workspace(MLA_OP_MHA, seqs, H, 0, workspace)
    c = seqs.c()
    _check(load().mla_prefill_mha(ctypes.byref(c), _ptr(q), H, _ptr(w_ukv), _ptr(kv), _ptr(kv_scale),
                                  float(sm_scale), _ptr(out), _ptr(lse), _ptr(ws), wsb, _ptr(dev_err), _stream()))
    return out, lse


def mla_prefill_dense_static(seqs: Seqs, q: torch.Tensor, kv: torch.Tensor, kv_scale: torch.Tensor,
                             sm_scale: float, out=None, lse=None, want_lse: bool = True, dev_err=None):
    """Dense prefill that allocates nothing inside the library: same result as
    mla_prefill_dense, for callers that may not allocate device memory (its
    scratch is a fixed array inside libmla.so; calls on different streams that
    overlap on the GPU race on it). Returns (out, lse)."""
    H = q.shape[1]
    if out is None:
        out = torch.empty((q.shape[0], H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((q.shape[0], H), dtype=torch.float32, device=q.device)
    c = seqs.c()
    _check(load().mla_prefill_dense_static(ctypes.byref(c), _ptr(q), H, _ptr(kv), _ptr(kv_scale), float(sm_scale),
                                           _ptr(out), _ptr(lse), _ptr(dev_err), _stream()))
    return out, lse


def mla_prefill_dense_host(seqs: Seqs, q_host: torch.Tensor, kv_host: torch.Tensor, kv_scale_host: torch.Tensor,
                           sm_scale: float, q: torch.Tensor, kv: torch.Tensor, kv_scale: torch.Tensor,
                           out_host: torch.Tensor, out: torch.Tensor, lse_host=None, lse=None, n_chunks: int = 8,
                           workspace=None, dev_err=None):
    """Dense prefill from host tensors to host tensors (pinned for overlap): the
    cache and, piece by piece, the query rows are copied into the device buffers
    q / kv / kv_scale, each piece's attention runs as its rows arrive and its
    out (and lse) rows are copied back into out_host (lse_host) as it finishes.
    Same results as mla_prefill_dense. Ordered on the current stream."""
    H = q.shape[1]
    ws, wsb = _workspace(MLA_OP_DENSE_HOST, seqs, H, 0, workspace)
    c = seqs.c()
    _check(load().mla_prefill_dense_host(ctypes.byref(c), _ptr(q_host), H, _ptr(kv_host), _ptr(kv_scale_host),
                                         float(sm_scale), _ptr(out_host), _ptr(lse_host), _ptr(q), _ptr(kv),
                                         _ptr(kv_scale), _ptr(out), _ptr(lse), int(n_chunks), _ptr(ws), wsb,
                                         _ptr(dev_err), _stream()))
    return out_host, lse_host


SPARSE_INPUTS = ("q", "qi", "w", "kv", "ks", "ki", "kis")   # field order of mla_sparse_inputs_t


def _inputs(t: dict) -> mla_sparse_inputs_t:
    return mla_sparse_inputs_t(*[None if t.get(k) is None else t[k].data_ptr() for k in SPARSE_INPUTS])


def _outputs(t: dict) -> mla_sparse_outputs_t:
    return mla_sparse_outputs_t(*[None if t.get(k) is None else t[k].data_ptr() for k in ("out", "lse", "idx")])


def mla_prefill_sparse_host(seqs: Seqs, host_in: dict, dev_in: dict, host_out: dict, dev_out: dict, sm_scale: float,
                            w_token_stride: int = 0, topk: int = 2048, n_chunks: int = 8, workspace=None,
                            dev_err=None):
    """The sparse step (indexer top-k, then sparse attention) from host tensors
    to host tensors (pinned for overlap). host_in / dev_in: dicts with keys q,
    qi, w, kv, ks, ki, kis (the tensors of mla_indexer_topk and
    mla_prefill_sparse, once in host and once in device memory); host_out /
    dev_out: out, idx and optionally lse. Same results as the two device calls.
    Ordered on the current stream."""
    H = dev_in["q"].shape[1]
    ws, wsb = _workspace(MLA_OP_INDEXER, seqs, H, topk, workspace)
    c = seqs.c()
    hi, di, ho, do = _inputs(host_in), _inputs(dev_in), _outputs(host_out), _outputs(dev_out)
    _check(load().mla_prefill_sparse_host(ctypes.byref(c), H, float(sm_scale), int(w_token_stride), int(topk),
                                          ctypes.byref(hi), ctypes.byref(di), ctypes.byref(ho), ctypes.byref(do),
                                          int(n_chunks), _ptr(ws), wsb, _ptr(dev_err), _stream()))
    return host_out


def mla_indexer_topk(seqs: Seqs, qi: torch.Tensor, w: torch.Tensor, w_token_stride: int, ki: torch.Tensor,
                     ki_scale: torch.Tensor, topk: int = 2048, idx_out=None, workspace=None, dev_err=None):
    """Indexer scores + exact top-k. qi uint8 [Tq,64,128]; w f32; ki uint8 [nb,256,128].
    Returns idx int32 [Tq, topk] (distinct positions in a fixed order, -1 padded)."""
    if idx_out is None:
        idx_out = torch.empty((qi.shape[0], topk), dtype=torch.int32, device=qi.device)
    ws, wsb = _workspace(MLA_OP_INDEXER, seqs, 64, topk, workspace)
    c = seqs.c()
    _check(load().mla_indexer_topk(ctypes.byref(c), _ptr(qi), _ptr(w), int(w_token_stride), _ptr(ki),
                                   _ptr(ki_scale), int(topk), _ptr(idx_out), _ptr(ws), wsb, _ptr(dev_err),
                                   _stream()))
    return idx_out


def mla_prefill_sparse(seqs: Seqs, q: torch.Tensor, kv: torch.Tensor, kv_scale: torch.Tensor, sm_scale: float,
                       idx: torch.Tensor, out=None, lse=None, want_lse: bool = True, workspace=None, dev_err=None):
    """Sparse MLA over idx [Tq, topk] (-1 skipped). Returns (out, lse)."""
    H = q.shape[1]
    if out is None:
        out = torch.empty((q.shape[0], H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((q.shape[0], H), dtype=torch.float32, device=q.device)
    ws, wsb = _workspace(MLA_OP_SPARSE, seqs, H, idx.shape[1], workspace)
    c = seqs.c()
    _check(load().mla_prefill_sparse(ctypes.byref(c), _ptr(q), H, _ptr(kv), _ptr(kv_scale), float(sm_scale),
                                     _ptr(idx), int(idx.shape[1]), _ptr(out), _ptr(lse), _ptr(ws), wsb,
                                     _ptr(dev_err), _stream()))
    return out, lse


def mla_prefill_dense_ds(seqs: Seqs, q: torch.Tensor, kv_ds: torch.Tensor, sm_scale: float, out=None, lse=None,
                         want_lse: bool = True, workspace=None, dev_err=None):
    """Dense causal MLA prefill on a cache of 656-byte rows kv_ds uint8 [nb,256,656]
    (512 e4m3 codes, four fp32 group scales, 64 bf16 RoPE values). Returns (out, lse)."""
    H = q.shape[1]
    if out is None:
        out = torch.empty((q.shape[0], H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((q.shape[0], H), dtype=torch.float32, device=q.device)
    ws, wsb = _workspace(MLA_OP_DENSE_DS, seqs, H, 0, workspace)
    c = seqs.c()
    _check(load().mla_prefill_dense_ds(ctypes.byref(c), _ptr(q), H, _ptr(kv_ds), float(sm_scale), _ptr(out),
                                       _ptr(lse), _ptr(ws), wsb, _ptr(dev_err), _stream()))
    return out, lse


def mla_prefill_sparse_ds(seqs: Seqs, q: torch.Tensor, kv_ds: torch.Tensor, sm_scale: float, idx: torch.Tensor,
                          out=None, lse=None, want_lse: bool = True, dev_err=None):
    """Sparse MLA over idx [Tq, topk] (-1 skipped) on a cache of 656-byte rows. Returns (out, lse)."""
    H = q.shape[1]
    if out is None:
        out = torch.empty((q.shape[0], H, 512), dtype=torch.bfloat16, device=q.device)
    if lse is None and want_lse:
        lse = torch.empty((q.shape[0], H), dtype=torch.float32, device=q.device)
    c = seqs.c()
    _check(load().mla_prefill_sparse_ds(ctypes.byref(c), _ptr(q), H, _ptr(kv_ds), float(sm_scale), _ptr(idx),
                                        int(idx.shape[1]), _ptr(out), _ptr(lse), _ptr(dev_err), _stream()))
    return out, lse


def mla_kv_append(seqs: Seqs, latent: torch.Tensor, kv: torch.Tensor, kv_scale: torch.Tensor, kidx=None, ki=None,
                  ki_scale=None, dev_err=None):
    """Quantise the new tokens' rows into the paged caches (in place).
    latent bf16 [Tq,576] -> kv uint8 [nb,256,576] + kv_scale f32 [nb,256];
    kidx bf16 [Tq,128] (optional) -> ki uint8 [nb,256,128] + ki_scale f32 [nb,256]."""
    c = seqs.c()
    _check(load().mla_kv_append(ctypes.byref(c), _ptr(latent), _ptr(kidx), _ptr(kv), _ptr(kv_scale), _ptr(ki),
                                _ptr(ki_scale), _ptr(dev_err), _stream()))


MLA_MERGE_MAX_PARTS = 8


def mla_merge_attn(outs, lses, out=None, lse=None, want_lse: bool = True):
    """Log-sum-exp merge of partial results over disjoint key sets.
    outs: list of bf16 [..., 512] tensors, lses: list of f32 tensors of the
    matching leading shape. Returns (out, lse) (out may be passed as outs[0])."""
    n = len(outs)
    if n != len(lses):
        raise ValueError("outs and lses differ in length")
    rows = outs[0].numel() // 512
    if out is None:
        out = torch.empty_like(outs[0])
    if lse is None and want_lse:
        lse = torch.empty_like(lses[0])
    po = (ctypes.c_void_p * n)(*[t.data_ptr() for t in outs])
    pl = (ctypes.c_void_p * n)(*[t.data_ptr() for t in lses])
    _check(load().mla_merge_attn(n, po, pl, rows, _ptr(out), _ptr(lse), _stream()))
    return out, lse


def chunk_bounds(total: int, chunk: int):
    """[start, end) of each prefill chunk: full chunks of `chunk` tokens, the last ragged."""
    return [(s, min(s + chunk, total)) for s in range(0, total, chunk)]


def chunk_seqs(block_table, num_blocks: int, total: int, chunk: int, device="cuda"):
    """One Seqs per prefill chunk of a prompt of `total` tokens: chunk c holds
    the new tokens [c*chunk, min((c+1)*chunk, total)) after a cached prefix of
    c*chunk tokens, over the prompt's block-table row."""
    return [Seqs([0, e - s], [s], block_table, num_blocks, device=device) for s, e in chunk_bounds(total, chunk)]


def chunked_prefill_sparse(block_table, num_blocks: int, total: int, chunk: int, q_chunk_fn, kv, kv_scale, qi_chunk_fn,
                           w, w_token_stride: int, ki, ki_scale, sm_scale: float, topk: int = 2048,
                           on_chunk=None, dev_err=None, out=None, lse=None, idx=None, workspace=None,
                           seqs_list=None, before_chunk=None, after_indexer=None):
    """Chunked prefill of one prompt of `total` tokens (GLM-5.3-Flash page,
    section on snapshots: prompts are read in fixed-size chunks). Chunk c covers
    new tokens [c*chunk, min((c+1)*chunk, total)) after a cached prefix of
    c*chunk tokens; each runs the indexer + top-k and then sparse MLA over the
    selected rows. q_chunk_fn(start, end) / qi_chunk_fn(start, end) return the
    chunk's device query tensors. on_chunk(c, start, end, out, lse, idx) sees
    every chunk's result (the caller keeps what it needs); without it the
    results are returned as a list.

    out, lse, idx: optional device buffers of at least `chunk` rows, reused by
    every chunk (then on_chunk must take what it keeps before returning);
    workspace: an optional buffer of mla_workspace_size(MLA_OP_INDEXER, ...)
    bytes for the largest chunk; seqs_list: the chunks' Seqs (chunk_seqs),
    built here if absent. before_chunk(c) / after_indexer(c) are called before
    chunk c's first call and between its two calls (e.g. to record events)."""
    results = []
    seqs_list = seqs_list or chunk_seqs(block_table, num_blocks, total, chunk, device=kv.device)
    for c, (s, e) in enumerate(chunk_bounds(total, chunk)):
        n = e - s
        seqs = seqs_list[c]
        if before_chunk is not None:
            before_chunk(c)
        ix = mla_indexer_topk(seqs, qi_chunk_fn(s, e), w, w_token_stride, ki, ki_scale, topk,
                              idx_out=None if idx is None else idx[:n], workspace=workspace, dev_err=dev_err)
        if after_indexer is not None:
            after_indexer(c)
        o, l = mla_prefill_sparse(seqs, q_chunk_fn(s, e), kv, kv_scale, sm_scale, ix,
                                  out=None if out is None else out[:n], lse=None if lse is None else lse[:n],
                                  dev_err=dev_err)
        if on_chunk is not None:
            on_chunk(c, s, e, o, l, ix)
        else:
            results.append((o, l, ix))
    return results
