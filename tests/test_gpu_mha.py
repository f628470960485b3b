"""The non-absorbed (MHA) path for short prompts ("GLM-5.3-Optimierungen, Teil
2", section Ausprobieren): per head, keys [W_UK c ; r] (192 dims) and values
W_UV c (128 dims) up-projected from the e4m3 cache, then causal attention,
element by element against the fp64 oracle, plus every row of the mha_short
workload against an fp32 reference in plain PyTorch.

The kernels keep the up-projected keys and values in f16; the log-sum-exp
check adds the bound that rounding each key to f16 implies per row (u = 2^-11
of sm_scale * max_s sum_d |q_d||k_s[d]|) to the usual 1e-3."""
import math

import numpy as np
import pytest

from oracle import oracle as O
from mla_prefill_attention_gb300 import inputs as I
from tests.parity import bf16_to_np, check_attention, check_attention_torch, mha_reference_torch, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_prefill_attention_gb300 import build
    build.build()


class MhaProblem:
    def __init__(self, q_lens, prefix_lens, heads, seed, sm_scale=1.0 / math.sqrt(192.0), shuffle=True,
                 extra_blocks=0):
        self.ps = I.make_seqs(q_lens, prefix_lens, seed, shuffle, extra_blocks)
        self.heads, self.sm_scale, self.seed = heads, sm_scale, seed
        self.q = I.gen_q_mha(seed, self.ps.total_q, heads)
        self.w = I.gen_w_ukv(seed, heads)
        self.kv, self.ks = I.gen_latent_cache(seed, self.ps)

    def device(self):
        import torch
        from mla_prefill_attention_gb300 import Seqs
        bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
        return {"seqs": Seqs.from_paged(self.ps), "q": bf(self.q), "w": bf(self.w),
                "kv": torch.from_numpy(self.kv).cuda(), "ks": torch.from_numpy(self.ks).cuda()}


def run_mha(pb, d, err=None):
    import torch
    from mla_prefill_attention_gb300 import mla_prefill_mha
    own = err is None
    if own:
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = mla_prefill_mha(d["seqs"], d["q"], d["w"], d["kv"], d["ks"], pb.sm_scale, dev_err=err)
    torch.cuda.synchronize()
    if own:
        assert int(err.item()) == 0
    return out, lse


def check_vs_oracle(pb, d, out, lse, toks, what):
    import torch
    ora, ora_lse = O.mla_mha(pb.ps, pb.q[toks], toks, pb.kv, pb.ks, pb.w, pb.sm_scale)
    _, _, bnd = mha_reference_torch(pb.ps, d["q"], d["w"], d["kv"], d["ks"], pb.sm_scale, toks=toks)
    t = torch.from_numpy(toks).cuda()
    check_attention(bf16_to_np(out[t]), ora, lse[t].cpu().numpy(), ora_lse, what, lse_extra=bnd.cpu().numpy())


@pytest.mark.parametrize("q_lens,prefix,H", [
    ([37, 200], [0, 64], 16),          # ragged tails, a prefix, two sequences in one 128-row up-projection tile each
    ([130], [0], 64),                  # one full 128-token tile and a 2-token tail
    ([5, 1, 260], [300, 0, 10], 128),  # 128 heads, a single-token sequence, prefixes past a page
    ([0, 70], [9, 0], 32),             # a sequence without new tokens
])
def test_mha_small_full(q_lens, prefix, H):
    pb = MhaProblem(q_lens, prefix, H, seed=31 + H)
    d = pb.device()
    out, lse = run_mha(pb, d)
    check_vs_oracle(pb, d, out, lse, np.arange(pb.ps.total_q), f"mha {q_lens} {prefix} H={H}")


def test_mha_short_sampled_and_every_row():
    """The batch of eight short prompts (77-2,048 tokens, 64 heads): sampled
    rows against the fp64 oracle, then every row against the fp32 reference."""
    w = I.WORKLOADS["mha_short"]
    pb = MhaProblem(w.q_lens, w.prefix_lens, w.heads, w.seed, w.sm_scale, w.shuffle)
    d = pb.device()
    out, lse = run_mha(pb, d)
    toks = sample_rows(pb.ps.cu_seqlens_q, seed=5, n_uniform=96, edge=16, chunks=8)
    check_vs_oracle(pb, d, out, lse, toks, "mha_short sampled")
    ref, ref_lse, bnd = mha_reference_torch(pb.ps, d["q"], d["w"], d["kv"], d["ks"], pb.sm_scale)
    check_attention_torch(out, ref, lse, ref_lse, "mha_short, every row", lse_extra=bnd)


def test_mha_page_shuffle_and_repeat_are_bit_identical():
    import torch
    a = MhaProblem([150, 300], [20, 0], 32, seed=41, shuffle=True, extra_blocks=9)
    b = MhaProblem([150, 300], [20, 0], 32, seed=41, shuffle=False)
    assert not np.array_equal(a.ps.block_table, b.ps.block_table)
    da, db = a.device(), b.device()
    oa, la = run_mha(a, da)
    ob, lb = run_mha(b, db)
    oa2, la2 = run_mha(a, da)
    assert torch.equal(oa, ob) and torch.equal(la, lb)
    assert torch.equal(oa, oa2) and torch.equal(la, la2)


def test_mha_bad_page_sets_device_flag():
    import torch
    from mla_prefill_attention_gb300 import MLA_DEVERR_BAD_PAGE, Seqs
    pb = MhaProblem([40], [200], 16, seed=43)
    d = pb.device()
    bt = pb.ps.block_table.copy()
    bt[0, 0] = pb.ps.num_blocks + 5                  # outside the cache
    d["seqs"] = Seqs(pb.ps.cu_seqlens_q, pb.ps.prefix_lens, bt, pb.ps.num_blocks)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_mha(pb, d, err=err)
    assert int(err.item()) & MLA_DEVERR_BAD_PAGE
    assert bool(torch.isfinite(out.float()).all())


def test_mha_long_prompt_with_prefix_sampled_and_every_row():
    """The path takes any length: 4,200 new tokens after a 1,000-token prefix
    (contexts past the top-k, tiles of up to 81 key tiles), 64 heads; sampled
    rows against the fp64 oracle, every row against the fp32 reference."""
    pb = MhaProblem([4200], [1000], 64, seed=45)
    d = pb.device()
    out, lse = run_mha(pb, d)
    toks = sample_rows(pb.ps.cu_seqlens_q, seed=6, n_uniform=48, edge=8, chunks=8)
    check_vs_oracle(pb, d, out, lse, toks, "mha 4200 after 1000 sampled")
    ref, ref_lse, bnd = mha_reference_torch(pb.ps, d["q"], d["w"], d["kv"], d["ks"], pb.sm_scale)
    check_attention_torch(out, ref, lse, ref_lse, "mha 4200 after 1000, every row", lse_extra=bnd)
