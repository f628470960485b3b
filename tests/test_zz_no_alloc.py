"""mla_prefill_dense_static: the dense call for callers that cannot allocate.

Some callers of this library are handed only their inputs and outputs and may
not allocate device memory: a plugin inside a framework that owns the whole
device pool, or a path that must avoid the device-wide synchronisation of
cudaMalloc. For them the library offers one dense entry point whose scratch
(the tile work list) is a fixed device array inside libmla.so.

These tests call it through the C ABI twice in a row, with two different
batches, and compare each result with the regular workspace entry point. Both
run the same attention kernel on the same tile pairs, so the results must be
bit-identical. The file sorts last so that a failure here stops a
first-failure run only after every other test has run.
"""
import ctypes

import numpy as np
import pytest

from tests.parity import Problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_prefill_attention_gb300 import build
    build.build()


def _static_call(seqs, d, sm_scale, H, out=None, lse=None, expect_err=0):
    """One call of the allocation-free entry point straight through ctypes."""
    import torch
    from mla_prefill_attention_gb300 import binding as B
    T = d["q"].shape[0]
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda") if out is None else out
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda") if lse is None else lse
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    c = seqs.c()
    st = B.load().mla_prefill_dense_static(ctypes.byref(c), ctypes.c_void_p(d["q"].data_ptr()), H,
                                           ctypes.c_void_p(d["kv"].data_ptr()), ctypes.c_void_p(d["ks"].data_ptr()),
                                           float(sm_scale), ctypes.c_void_p(out.data_ptr()),
                                           ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(err.data_ptr()),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == B.MLA_OK, B.load().mla_last_error()
    torch.cuda.synchronize()
    assert int(err.item()) == expect_err
    return out, lse


def test_static_matches_workspace_entry_point_twice():
    import torch
    from mla_prefill_attention_gb300 import mla_prefill_dense
    # a larger ragged batch first, then a smaller one: the second call must not
    # see anything the first left in the shared array
    cases = [Problem([300, 17, 129], [0, 700, 255], 64, seed=901, sm_scale=0.08),
             Problem([45], [1000], 16, seed=902, sm_scale=0.11)]
    for pb in cases:
        d = pb.device()
        H = pb.heads
        out_s, lse_s = _static_call(d["seqs"], d, pb.sm_scale, H)
        out_r, lse_r = mla_prefill_dense(d["seqs"], d["q"], d["kv"], d["ks"], pb.sm_scale)
        torch.cuda.synchronize()
        assert torch.equal(out_s.view(torch.int16), out_r.view(torch.int16)) and torch.equal(lse_s, lse_r)


@pytest.mark.parametrize("q_lens,prefix,H", [
    ([3] * 1500, [7] * 1500, 16),        # more sequences than the work-list kernel's 1,024 threads
    ([70, 1, 33], [0, 300, 129], 128),   # two tiles per token
])
def test_static_long_batches_and_128_heads(q_lens, prefix, H):
    import torch
    from mla_prefill_attention_gb300 import mla_prefill_dense
    pb = Problem(q_lens, prefix, H, seed=903 + H, sm_scale=0.09)
    d = pb.device()
    out_s, lse_s = _static_call(d["seqs"], d, pb.sm_scale, H)
    out_r, lse_r = mla_prefill_dense(d["seqs"], d["q"], d["kv"], d["ks"], pb.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(out_s.view(torch.int16), out_r.view(torch.int16)) and torch.equal(lse_s, lse_r)


def test_static_device_counts_fewer_tokens_than_host():
    """The device cu_seqlens counts 50 new tokens, its host mirror 100: the
    work list gets empty filler items, which the attention kernel skips; the
    mismatch is reported, the 50 tokens both count come out as a 50-token call
    gives them, and nothing outside the output buffer (guard rows on both
    sides) or in the other 50 rows is written."""
    import torch
    from mla_prefill_attention_gb300 import MLA_DEVERR_SEQ_MISMATCH, Seqs, mla_prefill_dense
    pb = Problem([100], [40], 64, seed=904, sm_scale=0.09)
    d = pb.device()
    seqs = d["seqs"]
    seqs.cu = torch.tensor([0, 50], dtype=torch.int32, device="cuda")
    sentinel = torch.tensor(12345, dtype=torch.int16)
    full = torch.full((102, 64, 512), int(sentinel), dtype=torch.int16, device="cuda")
    lse_full = torch.full((102, 64), 7.0, dtype=torch.float32, device="cuda")
    out, lse = full[1:101].view(torch.bfloat16), lse_full[1:101]
    _static_call(seqs, d, pb.sm_scale, 64, out=out, lse=lse, expect_err=MLA_DEVERR_SEQ_MISMATCH)
    assert bool((full[0] == sentinel).all()) and bool((full[101] == sentinel).all())
    assert bool((full[51:101] == sentinel).all()) and bool((lse_full[51:] == 7.0).all())
    assert bool((lse_full[0] == 7.0).all())
    ref = Seqs([0, 50], [40], pb.ps.block_table, pb.ps.num_blocks)
    out_r, lse_r = mla_prefill_dense(ref, d["q"][:50], d["kv"], d["ks"], pb.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(out[:50].view(torch.int16), out_r.view(torch.int16)) and torch.equal(lse[:50], lse_r)


def test_static_rejects_batches_beyond_its_array():
    from mla_prefill_attention_gb300 import Seqs
    from mla_prefill_attention_gb300 import binding as B
    # 65,537 tokens x 128 heads = 131,074 tiles of 64 rows = 65,537 pairs > 65,536
    seqs = Seqs([0, 65537], [0], np.zeros((1, 257), np.int32), 257)
    fake = ctypes.c_void_p(0x100000)
    c = seqs.c()
    st = B.load().mla_prefill_dense_static(ctypes.byref(c), fake, 128, fake, fake, 0.1, fake, None, None, None)
    assert st == B.MLA_ERR_UNSUPPORTED
    assert b"MLA_DENSE_STATIC_MAX_WORK_ITEMS" in B.load().mla_last_error()
