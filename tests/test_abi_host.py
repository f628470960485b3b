"""The C ABI library without a GPU: it builds, exports every declared entry
point, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

from mla_prefill_attention_gb300 import binding as B
from mla_prefill_attention_gb300 import build as mlabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mlabuild.build()
    return B.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "mla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    syms = declared_symbols()
    assert set(syms) == set(B.EXPORTS)
    for s in syms:
        assert hasattr(lib, s), s


class HostSeqs:
    """mla_seqs_t over host arrays only (device pointers are fake but never touched)."""

    def __init__(self, q_lens, prefix, max_blocks=None, num_blocks=None):
        self.cu = np.zeros(len(q_lens) + 1, np.int32)
        self.cu[1:] = np.cumsum(q_lens)
        self.pre = np.asarray(prefix, np.int32)
        need = max(-(-(p + t) // 256) for p, t in zip(prefix, q_lens))
        self.mb = max_blocks if max_blocks is not None else max(1, need)
        self.nb = num_blocks if num_blocks is not None else self.mb * len(q_lens)
        fake = 0x10000
        self.c = B.mla_seqs_t(len(q_lens), fake, self.cu.ctypes.data, fake, self.pre.ctypes.data, fake, self.mb,
                              self.nb)


FAKE = ctypes.c_void_p(0x100000)        # 16-byte aligned, never dereferenced on these paths
FAKE_MIS = ctypes.c_void_p(0x100004)


def dense(lib, s, H=64, q=FAKE, out=FAKE, ws=None, wsb=0, scale=0.07):
    return lib.mla_prefill_dense(ctypes.byref(s.c), q, H, FAKE, FAKE, scale, out, None, ws, wsb, None, None)


def test_rejects_bad_arguments(lib):
    s = HostSeqs([100], [0])
    assert lib.mla_prefill_dense(None, FAKE, 64, FAKE, FAKE, 0.1, FAKE, None, None, 0, None, None) == B.MLA_ERR_INVALID_ARG
    assert b"seqs" in lib.mla_last_error()
    assert dense(lib, s, H=48) == B.MLA_ERR_UNSUPPORTED
    assert dense(lib, s, q=FAKE_MIS) == B.MLA_ERR_INVALID_ARG
    assert dense(lib, s, q=None) == B.MLA_ERR_INVALID_ARG
    assert dense(lib, s, scale=float("nan")) == B.MLA_ERR_INVALID_ARG
    assert dense(lib, s) == B.MLA_ERR_WORKSPACE                 # no workspace given
    assert dense(lib, s, ws=FAKE, wsb=16) == B.MLA_ERR_WORKSPACE
    short = HostSeqs([600], [0], max_blocks=2)                  # needs 3 pages
    assert dense(lib, short) == B.MLA_ERR_INVALID_ARG
    assert b"pages" in lib.mla_last_error()
    bad_cu = HostSeqs([10, 5], [0, 0])
    bad_cu.cu[2] = 3                                            # decreasing
    assert dense(lib, bad_cu) == B.MLA_ERR_INVALID_ARG
    neg = HostSeqs([10], [0])
    neg.pre[0] = -1
    assert dense(lib, neg) == B.MLA_ERR_INVALID_ARG
    for k in (0, 2049):
        assert lib.mla_prefill_sparse(ctypes.byref(s.c), FAKE, 64, FAKE, FAKE, 0.1, FAKE, k, FAKE, None, None, 0,
                                      None, None) == B.MLA_ERR_UNSUPPORTED
        assert lib.mla_indexer_topk(ctypes.byref(s.c), FAKE, FAKE, 0, FAKE, FAKE, k, FAKE, None, 0, None,
                                    None) == B.MLA_ERR_UNSUPPORTED
    assert lib.mla_indexer_topk(ctypes.byref(s.c), FAKE, FAKE, -1, FAKE, FAKE, 2048, FAKE, None, 0, None,
                                None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_indexer_topk(ctypes.byref(s.c), FAKE, FAKE, 6, FAKE, FAKE, 2048, FAKE, None, 0, None,
                                None) == B.MLA_ERR_INVALID_ARG          # token stride not a multiple of 4
    w4 = ctypes.c_void_p(0x100004)                              # w needs 16-byte alignment (float4 loads)
    assert lib.mla_indexer_topk(ctypes.byref(s.c), FAKE, w4, 0, FAKE, FAKE, 2048, FAKE, None, 0, None,
                                None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_indexer_topk(ctypes.byref(s.c), FAKE, FAKE, 0, FAKE, FAKE, 2048, FAKE, None, 0, None,
                                None) == B.MLA_ERR_WORKSPACE
    odd = ctypes.c_void_p(0x100002)                             # idx needs 4-byte alignment
    assert lib.mla_prefill_sparse(ctypes.byref(s.c), FAKE, 64, FAKE, FAKE, 0.1, odd, 2048, FAKE, None, None,
                                  0, None, None) == B.MLA_ERR_INVALID_ARG


def dense_host(lib, s, H=64, qh=FAKE, kvh=FAKE, ksh=FAKE, oh=FAKE, lh=None, lse=None, chunks=4, ws=None, wsb=0):
    return lib.mla_prefill_dense_host(ctypes.byref(s.c), qh, H, kvh, ksh, 0.07, oh, lh, FAKE, FAKE, FAKE, FAKE, lse,
                                      chunks, ws, wsb, None, None)


def test_dense_host_rejects_bad_arguments(lib):
    s = HostSeqs([100], [0])
    for kw in ({"qh": None}, {"kvh": None}, {"ksh": None}, {"oh": None}, {"lh": FAKE}):
        assert dense_host(lib, s, **kw) == B.MLA_ERR_INVALID_ARG, kw
    for c in (0, B.DENSE_HOST_MAX_CHUNKS + 1):
        assert dense_host(lib, s, chunks=c) == B.MLA_ERR_INVALID_ARG
        assert b"n_chunks" in lib.mla_last_error()
    assert dense_host(lib, s, H=48) == B.MLA_ERR_UNSUPPORTED
    assert dense_host(lib, s) == B.MLA_ERR_WORKSPACE
    assert dense_host(lib, s, ws=FAKE, wsb=16) == B.MLA_ERR_WORKSPACE
    assert dense_host(lib, HostSeqs([0, 0], [5, 0])) == B.MLA_OK          # nothing to do, nothing touched
    # room for every piece's work list: the plain list plus at most one half-pair per
    # (piece, sequence) share
    for q_lens, H in (([100], 64), ([700, 33, 300], 16), ([5000], 128)):
        hs = HostSeqs(q_lens, [0] * len(q_lens))
        tiles = sum(-(-t * H // 64) for t in q_lens)
        ws = lib.mla_workspace_size(B.MLA_OP_DENSE_HOST, ctypes.byref(hs.c), H, 0)
        assert ws % 256 == 0 and ws >= (tiles // 2 + len(q_lens) + B.DENSE_HOST_MAX_CHUNKS) * 16


def sparse_host(lib, s, hi=None, di=None, ho=None, do=None, topk=2048, chunks=4, ws=None, wsb=0, H=64):
    full_in = B.mla_sparse_inputs_t(*([0x100000] * 7))
    full_out = B.mla_sparse_outputs_t(0x100000, None, 0x100000)
    hi, di = hi or full_in, di or full_in
    ho, do = ho or full_out, do or full_out
    return lib.mla_prefill_sparse_host(ctypes.byref(s.c), H, 0.07, 0, topk, ctypes.byref(hi), ctypes.byref(di),
                                       ctypes.byref(ho), ctypes.byref(do), chunks, ws, wsb, None, None)


def test_sparse_host_rejects_bad_arguments(lib):
    s = HostSeqs([100], [0])
    assert lib.mla_prefill_sparse_host(ctypes.byref(s.c), 64, 0.07, 0, 2048, None, None, None, None, 4, None, 0,
                                       None, None) == B.MLA_ERR_INVALID_ARG
    for i in range(7):                                      # each host input left out in turn
        fields = [0x100000] * 7
        fields[i] = None
        assert sparse_host(lib, s, hi=B.mla_sparse_inputs_t(*fields)) == B.MLA_ERR_INVALID_ARG, i
    for i in range(7):                                      # and each device input
        fields = [0x100000] * 7
        fields[i] = None
        assert sparse_host(lib, s, di=B.mla_sparse_inputs_t(*fields)) == B.MLA_ERR_INVALID_ARG, i
    assert sparse_host(lib, s, ho=B.mla_sparse_outputs_t(None, None, 0x100000)) == B.MLA_ERR_INVALID_ARG
    assert sparse_host(lib, s, ho=B.mla_sparse_outputs_t(0x100000, 0x100000, 0x100000)) == B.MLA_ERR_INVALID_ARG
    assert b"lse" in lib.mla_last_error()                   # lse on one side only
    for c in (0, B.DENSE_HOST_MAX_CHUNKS + 1):
        assert sparse_host(lib, s, chunks=c) == B.MLA_ERR_INVALID_ARG
    assert sparse_host(lib, s, topk=0) == B.MLA_ERR_UNSUPPORTED
    assert sparse_host(lib, s, H=48) == B.MLA_ERR_UNSUPPORTED
    assert sparse_host(lib, s) == B.MLA_ERR_WORKSPACE
    assert sparse_host(lib, HostSeqs([0, 0], [5, 0])) == B.MLA_OK


def test_empty_batch_is_a_noop(lib):
    s = HostSeqs([0, 0], [5, 0])
    assert dense(lib, s) == B.MLA_OK
    assert lib.mla_prefill_sparse(ctypes.byref(s.c), FAKE, 64, FAKE, FAKE, 0.1, FAKE, 2048, FAKE, None, None, 0,
                                  None, None) == B.MLA_OK
    assert lib.mla_indexer_topk(ctypes.byref(s.c), FAKE, FAKE, 0, FAKE, FAKE, 2048, FAKE, None, 0, None,
                                None) == B.MLA_OK


def test_workspace_sizes(lib):
    s = HostSeqs([4096], [12288])
    dense_ws = lib.mla_workspace_size(B.MLA_OP_DENSE, ctypes.byref(s.c), 64, 0)
    tiles = 4096 * 64 // 64
    assert dense_ws == -(-((tiles + 1) // 2 * 16) // 256) * 256
    # the indexer keeps its scores on chip: only its work list (one 16-byte item
    # per group of three tokens) and a 4-byte flag per item need device memory,
    # whatever the context length
    idx_ws = lib.mla_workspace_size(B.MLA_OP_INDEXER, ctypes.byref(s.c), 64, 2048)
    items = -(-4096 // 3)
    assert idx_ws == -(-(items * 16) // 256) * 256 + -(-(items * 4) // 256) * 256
    long_ctx = HostSeqs([4096], [196608])
    assert lib.mla_workspace_size(B.MLA_OP_INDEXER, ctypes.byref(long_ctx.c), 64, 2048) == idx_ws
    assert lib.mla_workspace_size(B.MLA_OP_SPARSE, ctypes.byref(s.c), 64, 2048) == 0
    assert lib.mla_workspace_size(B.MLA_OP_DENSE, None, 64, 0) == 0
    assert lib.mla_workspace_size(B.MLA_OP_DENSE, ctypes.byref(s.c), 40, 0) == 0


def test_kv_append_rejects_bad_arguments(lib):
    s = HostSeqs([100], [300])

    def app(lat=FAKE, kidx=None, kv=FAKE, kvs=FAKE, ki=None, kis=None, seqs=s):
        return lib.mla_kv_append(ctypes.byref(seqs.c) if seqs is not None else None, lat, kidx, kv, kvs, ki, kis,
                                 None, None)

    assert app(seqs=None) == B.MLA_ERR_INVALID_ARG
    assert app(lat=None) == B.MLA_ERR_INVALID_ARG
    assert app(lat=FAKE_MIS) == B.MLA_ERR_INVALID_ARG
    assert app(kv=FAKE_MIS) == B.MLA_ERR_INVALID_ARG
    assert app(kvs=ctypes.c_void_p(0x100002)) == B.MLA_ERR_INVALID_ARG
    assert app(kidx=FAKE) == B.MLA_ERR_INVALID_ARG             # key given without its cache
    assert b"ki" in lib.mla_last_error()
    assert app(kidx=FAKE_MIS, ki=FAKE, kis=FAKE) == B.MLA_ERR_INVALID_ARG
    short = HostSeqs([300], [0], max_blocks=1)                   # needs 2 pages
    assert app(seqs=short) == B.MLA_ERR_INVALID_ARG
    assert app(seqs=HostSeqs([0, 0], [7, 0])) == B.MLA_OK      # nothing to write: no launch


def test_merge_rejects_bad_arguments(lib):
    def arr(*ps):
        return (ctypes.c_void_p * len(ps))(*ps)

    two = arr(0x100000, 0x200000)
    lses = arr(0x300000, 0x400000)
    ok = lib.mla_merge_attn(2, two, lses, 0, FAKE, None, None)
    assert ok == B.MLA_OK                                       # no rows: nothing to launch
    assert lib.mla_merge_attn(0, two, lses, 10, FAKE, None, None) == B.MLA_ERR_UNSUPPORTED
    assert lib.mla_merge_attn(9, arr(*[0x100000] * 9), arr(*[0x300000] * 9), 10, FAKE, None,
                              None) == B.MLA_ERR_UNSUPPORTED
    assert lib.mla_merge_attn(2, None, lses, 10, FAKE, None, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_merge_attn(2, two, lses, 10, None, None, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_merge_attn(2, two, lses, -1, FAKE, None, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_merge_attn(2, arr(0x100000, 0x200008), lses, 10, FAKE, None, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_merge_attn(2, two, arr(0x300000, 0x400002), 10, FAKE, None, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_merge_attn(2, arr(0x100000, 0), lses, 10, FAKE, None, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_merge_attn(2, two, lses, 10, FAKE_MIS, None, None) == B.MLA_ERR_INVALID_ARG
    assert lib.mla_merge_attn(2, two, lses, 10, FAKE, ctypes.c_void_p(0x500002), None) == B.MLA_ERR_INVALID_ARG


def test_mha_rejects_bad_arguments_and_sizes_its_workspace(lib):
    s = HostSeqs([300, 77], [0, 40])

    def mha(seqs=s, H=64, q=FAKE, w=FAKE, out=FAKE, ws=None, wsb=0, scale=0.07):
        return lib.mla_prefill_mha(ctypes.byref(seqs.c) if seqs is not None else None, q, H, w, FAKE, FAKE, scale,
                                   out, None, ws, wsb, None, None)

    assert mha(seqs=None) == B.MLA_ERR_INVALID_ARG
    assert mha(H=48) == B.MLA_ERR_UNSUPPORTED
    assert mha(q=FAKE_MIS) == B.MLA_ERR_INVALID_ARG
    assert mha(w=None) == B.MLA_ERR_INVALID_ARG
    assert mha(w=FAKE_MIS) == B.MLA_ERR_INVALID_ARG
    assert mha(scale=float("inf")) == B.MLA_ERR_INVALID_ARG
    assert mha() == B.MLA_ERR_WORKSPACE
    # work lists (two 16-byte items per 128 new tokens, one per 128 context rows),
    # then k and v (256 bytes per row and head) and the RoPE dims (128 bytes per row)
    H = 64
    rows = 384 + 128                      # contexts 300 and 117, each padded to 128
    at = (3 + 1) * 2 * 16
    up = (3 + 1) * 16
    rnd = lambda x: -(-x // 256) * 256
    want = rnd(at) + rnd(up) + 2 * rnd(H * rows * 256) + rnd(rows * 128)
    assert lib.mla_workspace_size(B.MLA_OP_MHA, ctypes.byref(s.c), H, 0) == want
    assert mha(ws=FAKE, wsb=want - 1) == B.MLA_ERR_WORKSPACE
    assert mha(ws=ctypes.c_void_p(0x100010), wsb=want) == B.MLA_ERR_WORKSPACE      # not 256-byte aligned
    assert mha(seqs=HostSeqs([0, 0], [5, 0])) == B.MLA_OK                         # no new tokens: no launch


def test_dense_ds_workspace_holds_the_converted_rows(lib):
    """Dense calls on 656-byte rows convert every context row once: the workspace
    holds the work list, the per-sequence bases and lengths, 1,152 bytes of f16
    per row (contexts padded to 80-key tiles) and 960 bytes of metadata per tile."""
    s = HostSeqs([100, 0, 37], [500, 9, 0])
    H = 64
    rnd = lambda x: -(-x // 256) * 256
    tiles = [(100 * H + 63) // 64, (37 * H + 63) // 64]
    items = sum((t + 1) // 2 for t in tiles)
    rows = 640 + 80                        # contexts 600 and 37 padded to 80; the empty sequence adds none
    want = rnd(items * 16) + rnd(2 * 3 * 4) + rnd(rows * 1152) + rnd(rows // 80 * 960)
    assert lib.mla_workspace_size(B.MLA_OP_DENSE_DS, ctypes.byref(s.c), H, 0) == want

    def dds(ws=None, wsb=0):
        return lib.mla_prefill_dense_ds(ctypes.byref(s.c), FAKE, H, FAKE, 0.07, FAKE, None, ws, wsb, None, None)

    assert dds() == B.MLA_ERR_WORKSPACE
    assert dds(FAKE, want - 1) == B.MLA_ERR_WORKSPACE
    assert dds(ctypes.c_void_p(0x100010), want) == B.MLA_ERR_WORKSPACE        # not 256-byte aligned
