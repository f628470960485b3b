"""Dense and sparse MLA on the 656-byte cache rows (512 e4m3 latent codes, one
fp32 scale per 128 dims, 64 bf16 RoPE values; GLM-5.3-Optimierungen Teil 2,
footnote 1), element by element against the fp64 oracle, plus every row of
the sparse64k workload against an fp32 reference in plain PyTorch.

The rows' group scales make the key values inexact in any 16-bit tensor-core
operand, and the kernel rounds each once to f16; the log-sum-exp check adds
the bound that rounding implies per row (ds_lse_bound) to the usual 1e-3."""
import math

import numpy as np
import pytest

from oracle import oracle as O
from mla_prefill_attention_gb300 import inputs as I
from tests.parity import (UNIFORM_ROWS, bf16_to_np, check_attention, check_attention_torch,
                          ds_lse_bound, sample_rows, sparse_reference_ds_torch)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_prefill_attention_gb300 import build
    build.build()


class DsProblem:
    def __init__(self, q_lens, prefix_lens, heads, seed, sm_scale=1.0 / math.sqrt(192.0), indexer=False):
        self.ps = I.make_seqs(q_lens, prefix_lens, seed, True)
        self.heads, self.sm_scale, self.seed = heads, sm_scale, seed
        self.q = I.gen_q_bf16(seed, self.ps.total_q, heads)
        self.kv = I.gen_latent_cache_ds(seed, self.ps)
        if indexer:
            self.qi, self.w, self.ki, self.kis = I.gen_indexer_inputs(seed, self.ps)

    def device(self):
        import torch
        from mla_prefill_attention_gb300 import Seqs
        d = {"seqs": Seqs.from_paged(self.ps), "kv": torch.from_numpy(self.kv).cuda(),
             "q": torch.from_numpy(self.q.view(np.int16)).view(torch.bfloat16).cuda()}
        if hasattr(self, "qi"):
            for k in ("qi", "w", "ki", "kis"):
                d[k] = torch.from_numpy(getattr(self, k)).cuda()
        return d


def run_dense(pb, d):
    import torch
    from mla_prefill_attention_gb300 import mla_prefill_dense_ds
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = mla_prefill_dense_ds(d["seqs"], d["q"], d["kv"], pb.sm_scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out, lse


def run_sparse(pb, d, idx):
    import torch
    from mla_prefill_attention_gb300 import mla_prefill_sparse_ds
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = mla_prefill_sparse_ds(d["seqs"], d["q"], d["kv"], pb.sm_scale, idx, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out, lse


@pytest.mark.parametrize("q_lens,prefix,H", [
    ([1], [0], 16),                       # one row group, one key
    ([77], [300], 16),                    # prefix not page aligned, ragged tail tile
    ([130, 1, 65], [0, 255, 700], 32),    # ragged batch, a one-token sequence
    ([40], [0], 128),                     # two tiles per token
    ([90], [513], 64),
    ([0, 50], [10, 0], 64),               # an empty sequence in the batch
])
def test_dense_ds_small_full(q_lens, prefix, H):
    pb = DsProblem(q_lens, prefix, H, seed=600 + H + len(q_lens), sm_scale=0.09)
    d = pb.device()
    out, lse = run_dense(pb, d)
    toks = np.arange(pb.ps.total_q)
    ora, ora_lse = O.mla_dense_ds(pb.ps, pb.q, toks, pb.kv, pb.sm_scale)
    check_attention(bf16_to_np(out), ora, lse.cpu().numpy(), ora_lse, f"ds {q_lens}/{prefix}/H{H}",
                    lse_extra=ds_lse_bound(pb.ps, d["q"], d["kv"], pb.sm_scale, toks))


def test_dense_ds_wide_group_scales():
    """The four group scales of every row spread over 2^6 (x 2^-3, 2^-1, 2^1,
    2^3) and the RoPE values scaled by 8, so the loaders' group ratios run from
    1/64 to 1 and the RoPE values far from the latent ones. (A spread of 2^12
    within a row takes this f16 path's largest error to ~2.1e-2 of the row RMS,
    past the bound; cache writes that take each group's scale from its own
    absmax keep a row's scales within small factors.)"""
    pb = DsProblem([70], [200], 64, seed=611, sm_scale=0.07)
    kv = pb.kv.reshape(-1, 656).copy()
    sc = kv[:, 512:528].copy().view("<f4")
    sc *= np.exp2(np.array([-3.0, -1.0, 1.0, 3.0], np.float32))[None, :]
    kv[:, 512:528] = sc.view(np.uint8)
    rope = kv[:, 528:].copy().view("<u2")
    rope_v = O.bf16_to_f64(rope) * 8.0
    kv[:, 528:] = I.bf16_bits(rope_v).astype("<u2").view(np.uint8)
    pb.kv = kv.reshape(pb.kv.shape)
    d = pb.device()
    out, lse = run_dense(pb, d)
    toks = np.arange(pb.ps.total_q)
    ora, ora_lse = O.mla_dense_ds(pb.ps, pb.q, toks, pb.kv, pb.sm_scale)
    check_attention(bf16_to_np(out), ora, lse.cpu().numpy(), ora_lse, "ds wide scales",
                    lse_extra=ds_lse_bound(pb.ps, d["q"], d["kv"], pb.sm_scale, toks))


@pytest.mark.parametrize("H", [16, 64, 128])
def test_sparse_ds_small_vs_oracle(H):
    from mla_prefill_attention_gb300 import mla_indexer_topk
    import torch
    pb = DsProblem([50, 30], [700, 100], H, seed=620 + H, sm_scale=0.08, indexer=True)
    d = pb.device()
    idx = mla_indexer_topk(d["seqs"], d["qi"], d["w"], 0, d["ki"], d["kis"], 256)
    torch.cuda.synchronize()
    out, lse = run_sparse(pb, d, idx)
    toks = np.arange(pb.ps.total_q)
    ora, ora_lse = O.mla_sparse_ds(pb.ps, pb.q, toks, pb.kv, pb.sm_scale, idx.cpu().numpy())
    check_attention(bf16_to_np(out), ora, lse.cpu().numpy(), ora_lse, f"sparse ds H{H}",
                    lse_extra=ds_lse_bound(pb.ps, d["q"], d["kv"], pb.sm_scale, toks, idx))


def test_prefix12k_ds_sampled():
    w = I.WORKLOADS["prefix12k"]
    pb = DsProblem(w.q_lens, w.prefix_lens, w.heads, w.seed, w.sm_scale)
    d = pb.device()
    out, lse = run_dense(pb, d)
    toks = sample_rows(pb.ps.cu_seqlens_q, seed=5, n_uniform=max(1, UNIFORM_ROWS // 4))
    ora, ora_lse = O.mla_dense_ds(pb.ps, pb.q[toks], toks, pb.kv, pb.sm_scale)
    check_attention(bf16_to_np(out[toks]), ora, lse[toks].cpu().numpy(), ora_lse, "prefix12k ds",
                    lse_extra=ds_lse_bound(pb.ps, d["q"], d["kv"], pb.sm_scale, toks))


def test_sparse64k_ds_sampled_and_every_row():
    """The sparse64k workload on 656-byte rows: sampled rows against the fp64
    oracle and every row against an fp32 reference (plain PyTorch)."""
    import torch
    from mla_prefill_attention_gb300 import mla_indexer_topk
    w = I.WORKLOADS["sparse64k"]
    pb = DsProblem(w.q_lens, w.prefix_lens, w.heads, w.seed, w.sm_scale, indexer=True)
    d = pb.device()
    idx = mla_indexer_topk(d["seqs"], d["qi"], d["w"], 0, d["ki"], d["kis"], w.topk)
    torch.cuda.synchronize()
    out, lse = run_sparse(pb, d, idx)
    toks = sample_rows(pb.ps.cu_seqlens_q, seed=6, n_uniform=max(1, UNIFORM_ROWS // 4))
    ora, ora_lse = O.mla_sparse_ds(pb.ps, pb.q[toks], toks, pb.kv, pb.sm_scale, idx[toks].cpu().numpy())
    check_attention(bf16_to_np(out[toks]), ora, lse[toks].cpu().numpy(), ora_lse, "sparse64k ds",
                    lse_extra=ds_lse_bound(pb.ps, d["q"], d["kv"], pb.sm_scale, toks, idx))
    ref, ref_lse = sparse_reference_ds_torch(pb.ps, d["q"], d["kv"], pb.sm_scale, idx)
    check_attention_torch(out, ref, None, None, "sparse64k ds, every row")


def test_dense_ds_page_shuffle_and_repeat_are_bit_identical():
    """The converted rows are laid out by position, so where the pages sit in the
    cache cannot change a bit of the result; nor can a second call."""
    import torch
    a = DsProblem([150, 300], [20, 0], 32, seed=631)
    ps_b = I.make_seqs([150, 300], [20, 0], 631, shuffle=True, extra_blocks=9)
    assert not np.array_equal(a.ps.block_table, ps_b.block_table)
    kv_b = I.gen_latent_cache_ds(631, ps_b)
    from mla_prefill_attention_gb300 import Seqs
    da = a.device()
    db = dict(da, seqs=Seqs.from_paged(ps_b), kv=torch.from_numpy(kv_b).cuda())
    oa, la = run_dense(a, da)
    ob, lb = run_dense(a, db)
    oa2, la2 = run_dense(a, da)
    assert torch.equal(oa, ob) and torch.equal(la, lb)
    assert torch.equal(oa, oa2) and torch.equal(la, la2)


def test_dense_ds_bad_page_sets_device_flag():
    """A block-table entry outside [0, num_blocks) is reported by the conversion
    (its rows become zero keys) and the kernels do not fault."""
    import torch
    from mla_prefill_attention_gb300 import MLA_DEVERR_BAD_PAGE, Seqs, mla_prefill_dense_ds
    pb = DsProblem([40], [300], 16, seed=632)
    bt = pb.ps.block_table.copy()
    bt[0, 0] = pb.ps.num_blocks + 5
    d = pb.device()
    seqs = Seqs(pb.ps.cu_seqlens_q, pb.ps.prefix_lens, bt, pb.ps.num_blocks)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = mla_prefill_dense_ds(seqs, d["q"], d["kv"], pb.sm_scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & MLA_DEVERR_BAD_PAGE
    assert bool(torch.isfinite(out.float()).all())
