"""Dense MLA prefill on the GPU, element by element against the fp64 oracle."""
import numpy as np
import pytest

from oracle import oracle as O
from mla_prefill_attention_gb300 import inputs as I
from tests.parity import Problem, bf16_to_np, check_attention, sample_tokens

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


def test_prefix12k_sampled():
    w = I.WORKLOADS["prefix12k"]
    pb = Problem(w.q_lens, w.prefix_lens, w.heads, w.seed, w.shuffle, w.sm_scale)
    out, lse = run_dense(pb)
    toks = sample_tokens(pb.ps.total_q, 24, seed=1, boundaries=range(0, 4096, 256))
    check_rows(pb, out, lse, toks, "prefix12k")


@pytest.mark.parametrize("name", ["dense32k", "ragged4"])
def test_32k_sampled(name):
    w = I.WORKLOADS[name]
    pb = Problem(w.q_lens, w.prefix_lens, w.heads, w.seed, w.shuffle, w.sm_scale)
    out, lse = run_dense(pb)
    cu = pb.ps.cu_seqlens_q
    bounds = list(cu) + [int(cu[-1]) * k // 16 for k in range(16)]
    toks = sample_tokens(pb.ps.total_q, 16, seed=2, edge=4, boundaries=bounds)
    check_rows(pb, out, lse, toks, name)


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
