"""mla_prefill_dense_static: the dense call for callers that cannot allocate.

Some callers of this library are handed only their inputs and outputs and may
not allocate device memory: a plugin inside a framework that owns the whole
device pool, or a path that must avoid the device-wide synchronisation of
cudaMalloc. For them the library offers one dense entry point whose scratch
(the tile work list) is a fixed device array inside libmla.so.

These tests call it through the C ABI twice in a row, with two different
batches, and compare each result with the regular workspace entry point
within the parity tolerance. The file sorts last so that a failure here
stops a first-failure run only after every other test has run.
"""
import ctypes

import numpy as np
import pytest

from tests.parity import Problem, bf16_to_np, check_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_prefill_attention_gb300 import build
    build.build()


def _static_call(seqs, d, sm_scale, H):
    """One call of the allocation-free entry point straight through ctypes."""
    import torch
    from mla_prefill_attention_gb300 import binding as B
    T = d["q"].shape[0]
    out = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    c = seqs.c()
    st = B.load().mla_prefill_dense_static(ctypes.byref(c), ctypes.c_void_p(d["q"].data_ptr()), H,
                                           ctypes.c_void_p(d["kv"].data_ptr()), ctypes.c_void_p(d["ks"].data_ptr()),
                                           float(sm_scale), ctypes.c_void_p(out.data_ptr()),
                                           ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(err.data_ptr()),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == B.MLA_OK, B.load().mla_last_error()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
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
        check_attention(bf16_to_np(out_s), bf16_to_np(out_r), lse_s.cpu().numpy(),
                        lse_r.cpu().numpy().astype(np.float64), "static vs workspace")


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
