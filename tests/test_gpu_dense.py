"""Dense MLA prefill on the GPU, element by element against the fp64 oracle."""
import numpy as np
import pytest

from oracle import oracle as O
from mla_prefill_attention_gb300 import inputs as I
from tests.parity import UNIFORM_ROWS, Problem, bf16_to_np, check_attention, rel_errors, sample_rows, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_prefill_attention_gb300 import build
    build.build()


def run_dense(pb, d=None):
    import torch
    from mla_prefill_attention_gb300 import mla_prefill_dense
    d = d or pb.device()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = mla_prefill_dense(d["seqs"], d["q"], d["kv"], d["ks"], pb.sm_scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out, lse


def check_rows(pb, out, lse, toks, what):
    ora, ora_lse = O.mla_dense(pb.ps, pb.q[toks], toks, pb.kv, pb.ks, pb.sm_scale)
    return check_attention(bf16_to_np(out[toks]), ora, lse[toks].cpu().numpy(), ora_lse, what)


def test_tiny512_full():
    w = I.WORKLOADS["tiny512"]
    pb = Problem(w.q_lens, w.prefix_lens, w.heads, w.seed, w.shuffle, w.sm_scale)
    out, lse = run_dense(pb)
    check_rows(pb, out, lse, np.arange(pb.ps.total_q), "tiny512")


@pytest.mark.parametrize("q_lens,prefix,H", [
    ([1], [0], 16),                       # a single row group, one key
    ([3], [0], 64),                       # fewer rows than one tile
    ([77], [300], 16),                    # prefix not page aligned, ragged tail tile
    ([130, 1, 65], [0, 255, 700], 32),    # ragged batch, one-token sequence
    ([40], [0], 128),                     # two tiles per token
    ([90], [513], 64),
    ([0, 50], [10, 0], 64),               # an empty sequence in the batch
])
def test_small_full(q_lens, prefix, H):
    pb = Problem(q_lens, prefix, H, seed=100 + H + len(q_lens), shuffle=True, sm_scale=0.09)
    out, lse = run_dense(pb)
    check_rows(pb, out, lse, np.arange(pb.ps.total_q), f"{q_lens}/{prefix}/H{H}")


def test_unwritten_cache_slots_are_ignored():
    """Slots of a sequence's last page past its last token, and whole pages no
    sequence owns, hold NaN codes (0x7F) and huge scales: nothing may leak into
    the output (a NaN multiplied by a zero weight stays NaN)."""
    import torch
    pb = Problem([37, 5], [150, 700], 64, seed=77, shuffle=True, sm_scale=0.09, extra_blocks=2)
    used = np.zeros(pb.kv.shape[:2], dtype=bool)
    for bq in range(pb.ps.batch):
        sp = np.arange(pb.ps.seq_len(bq))
        used[pb.ps.block_table[bq, sp // 256], sp % 256] = True
    pb.kv[~used] = 0x7F
    pb.ks[~used] = 1e30
    out, lse = run_dense(pb)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    check_rows(pb, out, lse, np.arange(pb.ps.total_q), "NaN-filled unwritten slots")


def dense_via_sparse_slices(pb, d, out_dense, lse_dense, what, block=4096):
    """Every row of a dense call against an independent path over the same
    keys: for each token, sparse attention over each 2,048-position slice of
    its visible keys (positions as index lists), the slices' partial results
    merged by their log-sum-exp. Runs on the GPU over all rows, so a fault
    confined to some CTAs of the dense grid (a wrong work item, tile or stage)
    shows even where the sampled oracle rows miss it. Each side rounds to bf16
    on its own (the slices, their merge and the dense output), so the bounds
    are four times the oracle bounds; a wrong tile errs by the whole row."""
    import torch
    from mla_prefill_attention_gb300 import Seqs, mla_merge_attn, mla_prefill_sparse
    ps, K = pb.ps, 2048
    worst = (0.0, 0.0, 0.0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for b in range(ps.batch):
        c0, n, P = int(ps.cu_seqlens_q[b]), ps.seq_len(b) - int(ps.prefix_lens[b]), int(ps.prefix_lens[b])
        for t0 in range(0, n, block):
            nb = min(block, n - t0)
            seqs = Seqs([0, nb], [P + t0], ps.block_table[b:b + 1], ps.num_blocks)
            q = d["q"][c0 + t0:c0 + t0 + nb]
            pos = torch.arange(P + t0, P + t0 + nb, device="cuda", dtype=torch.int32)[:, None]
            outs, lses = [], []
            for j in range((P + t0 + nb - 1) // K + 1):
                idx = torch.arange(j * K, (j + 1) * K, device="cuda", dtype=torch.int32)[None, :].expand(nb, K)
                idx = torch.where(idx <= pos, idx, torch.full_like(idx, -1)).contiguous()
                o, l = mla_prefill_sparse(seqs, q, d["kv"], d["ks"], pb.sm_scale, idx, dev_err=err)
                outs.append(o)
                lses.append(l)
            while len(outs) > 1:      # groups of up to 8 parts: at most two merge levels here
                g = [(outs[i:i + 8], lses[i:i + 8]) for i in range(0, len(outs), 8)]
                outs, lses = map(list, zip(*[mla_merge_attn(o, l) if len(o) > 1 else (o[0], l[0]) for o, l in g]))
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            ref_o = out_dense[c0 + t0:c0 + t0 + nb].float()
            rms = ref_o.pow(2).mean(dim=-1, keepdim=True).sqrt()
            rel = (outs[0].float() - ref_o).abs() / torch.where(rms > 0, rms, torch.ones_like(rms))
            mx, mean = float(rel.max()), float(rel.mean())
            dl = float((lses[0] - lse_dense[c0 + t0:c0 + t0 + nb]).abs().max())
            worst = (max(worst[0], mx), max(worst[1], mean), max(worst[2], dl))
    assert worst[0] <= 4 * 2e-2 and worst[1] <= 4 * 2e-3 and worst[2] <= 4e-3, f"{what}: slices vs dense {worst}"
    return worst


def test_prefix12k_sampled():
    w = I.WORKLOADS["prefix12k"]
    pb = Problem(w.q_lens, w.prefix_lens, w.heads, w.seed, w.shuffle, w.sm_scale)
    d = pb.device()
    out, lse = run_dense(pb, d)
    toks = sample_rows(pb.ps.cu_seqlens_q, seed=1, extra_boundaries=range(0, 4096, 256))
    check_rows(pb, out, lse, toks, "prefix12k")
    dense_via_sparse_slices(pb, d, out, lse, "prefix12k")


@pytest.mark.parametrize("name", ["dense32k", "ragged4"])
def test_32k_sampled(name):
    """Sampled rows against the oracle: per sequence the first and last 64, the
    16 chunk boundaries +-2 and uniform draws (1,024 for the single 32k prompt,
    256 per prompt of the ragged batch); then every row against the sparse
    slice path."""
    w = I.WORKLOADS[name]
    pb = Problem(w.q_lens, w.prefix_lens, w.heads, w.seed, w.shuffle, w.sm_scale)
    d = pb.device()
    out, lse = run_dense(pb, d)
    n_uni = None if len(w.q_lens) == 1 else max(1, UNIFORM_ROWS // 4)
    toks = sample_rows(pb.ps.cu_seqlens_q, seed=2, n_uniform=n_uni)
    check_rows(pb, out, lse, toks, name)
    dense_via_sparse_slices(pb, d, out, lse, name)


def test_page_shuffle_is_bit_identical():
    import torch
    pb = Problem([300], [200], 64, seed=5, shuffle=False)
    out_a, lse_a = run_dense(pb)
    perm = np.random.default_rng(9).permutation(pb.ps.num_blocks).astype(np.int32)
    kv2, ks2 = np.empty_like(pb.kv), np.empty_like(pb.ks)
    kv2[perm], ks2[perm] = pb.kv, pb.ks
    pb.kv, pb.ks = kv2, ks2
    pb.ps = I.PagedSeqs(pb.ps.cu_seqlens_q, pb.ps.prefix_lens, perm[pb.ps.block_table], pb.ps.num_blocks)
    out_b, lse_b = run_dense(pb)
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)


def test_ragged_batch_equals_each_alone_bitwise():
    import torch
    pb = Problem([70, 33, 129], [10, 600, 0], 16, seed=6)
    out, lse = run_dense(pb)
    cu = pb.ps.cu_seqlens_q
    for b in range(3):
        one = Problem.__new__(Problem)
        one.ps = I.PagedSeqs(np.array([0, cu[b + 1] - cu[b]], np.int32), pb.ps.prefix_lens[b:b + 1],
                             pb.ps.block_table[b:b + 1], pb.ps.num_blocks)
        one.q, one.kv, one.ks, one.sm_scale, one.heads = pb.q[cu[b]:cu[b + 1]], pb.kv, pb.ks, pb.sm_scale, 16
        o1, l1 = run_dense(one)
        assert torch.equal(o1, out[cu[b]:cu[b + 1]]) and torch.equal(l1, lse[cu[b]:cu[b + 1]])


def test_deterministic():
    import torch
    pb = Problem([257], [31], 64, seed=7)
    d = pb.device()
    a = run_dense(pb, d)
    b = run_dense(pb, d)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_bad_page_sets_device_flag():
    """A block-table entry outside [0, num_blocks) is skipped and reported
    through dev_err; the kernel does not fault."""
    import torch
    from mla_prefill_attention_gb300 import MLA_DEVERR_BAD_PAGE, Seqs, mla_prefill_dense
    pb = Problem([64], [256], 16, seed=8)
    bt = pb.ps.block_table.copy()
    bt[0, 0] = pb.ps.num_blocks + 5
    d = pb.device()
    seqs = Seqs(pb.ps.cu_seqlens_q, pb.ps.prefix_lens, bt, pb.ps.num_blocks)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = mla_prefill_dense(seqs, d["q"], d["kv"], d["ks"], pb.sm_scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & MLA_DEVERR_BAD_PAGE
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("q_lens,prefix,H,chunks", [
    ([700, 33, 300], [100, 0, 2000], 64, 5),   # pieces cross sequence boundaries
    ([257], [40], 16, 3),                      # four tokens per tile: pieces move to tile boundaries
    ([129, 64], [0, 300], 128, 64),            # two tiles per token, the most pieces
    ([0, 50], [10, 0], 64, 8),                 # an empty sequence
    ([3], [0], 32, 8),                         # fewer tiles than pieces: some pieces empty
])
def test_dense_from_host_matches_device_call(q_lens, prefix, H, chunks):
    """The host-to-host call (copies overlapped with attention, piece by piece)
    returns exactly what the device call returns, and both match the oracle."""
    import torch
    from mla_prefill_attention_gb300 import mla_prefill_dense_host
    pb = Problem(q_lens, prefix, H, seed=400 + H + chunks, shuffle=True, sm_scale=0.09)
    d = pb.device()
    out_d, lse_d = run_dense(pb, d)
    T = pb.ps.total_q
    qh = torch.from_numpy(pb.q.view(np.int16)).view(torch.bfloat16).pin_memory()
    kvh, ksh = torch.from_numpy(pb.kv).pin_memory(), torch.from_numpy(pb.ks).pin_memory()
    oh = torch.full((T, H, 512), float("nan"), dtype=torch.bfloat16).pin_memory()
    lh = torch.full((T, H), float("nan"), dtype=torch.float32).pin_memory()
    q2, kv2, ks2 = torch.zeros_like(d["q"]), torch.zeros_like(d["kv"]), torch.zeros_like(d["ks"])
    o2, l2 = torch.zeros_like(out_d), torch.zeros_like(lse_d)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla_prefill_dense_host(d["seqs"], qh, kvh, ksh, pb.sm_scale, q2, kv2, ks2, oh, o2, lse_host=lh, lse=l2,
                           n_chunks=chunks, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(oh.view(torch.int16), out_d.cpu().view(torch.int16))
    assert torch.equal(lh, lse_d.cpu())
    toks = np.arange(T)
    ora, ora_lse = O.mla_dense(pb.ps, pb.q, toks, pb.kv, pb.ks, pb.sm_scale)
    check_attention(bf16_to_np(oh), ora, lh.numpy(), ora_lse, f"from host {q_lens}/H{H}/{chunks}")


def test_device_counts_fewer_tokens_than_host():
    """The device cu_seqlens counts 50 new tokens, its host mirror 100. The host
    pairs row tile i with tile 99-i, and every such pair holds a tile the device
    does not back, so every work item is skipped whole and reported
    (MLA_DEVERR_SEQ_MISMATCH): nothing in or around the output buffer (guard
    rows on both sides) is written."""
    import torch
    from mla_prefill_attention_gb300 import MLA_DEVERR_SEQ_MISMATCH, mla_prefill_dense
    pb = Problem([100], [40], 64, seed=78, sm_scale=0.09)
    d = pb.device()
    seqs = d["seqs"]
    seqs.cu = torch.tensor([0, 50], dtype=torch.int32, device="cuda")
    full = torch.full((102, 64, 512), 12345, dtype=torch.int16, device="cuda")
    lse_full = torch.full((102, 64), 7.0, dtype=torch.float32, device="cuda")
    out, lse = full[1:101].view(torch.bfloat16), lse_full[1:101]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla_prefill_dense(seqs, d["q"], d["kv"], d["ks"], pb.sm_scale, out=out, lse=lse, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == MLA_DEVERR_SEQ_MISMATCH
    assert bool((full == 12345).all()) and bool((lse_full == 7.0).all())
