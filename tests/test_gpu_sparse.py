"""Indexer top-k (bit-exact) and sparse MLA (within tolerance) on the GPU
against the fp64 oracle, plus the chunked long-prompt driver."""
import numpy as np
import pytest

from oracle import oracle as O
from mla_prefill_attention_gb300 import inputs as I
from tests.parity import (TOL_MAX, TOL_MEAN, UNIFORM_ROWS, Problem, bf16_to_np, check_attention, check_attention_torch,
                          check_topk_torch, rel_errors, sample_rows, sample_tokens, sparse_reference_torch)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_prefill_attention_gb300 import build
    build.build()


def run_indexer(pb, d, topk):
    import torch
    from mla_prefill_attention_gb300 import mla_indexer_topk
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = mla_indexer_topk(d["seqs"], d["qi"], d["w"], 0, d["ki"], d["kis"], topk, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return idx


def run_sparse(pb, d, idx):
    import torch
    from mla_prefill_attention_gb300 import mla_prefill_sparse
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = mla_prefill_sparse(d["seqs"], d["q"], d["kv"], d["ks"], pb.sm_scale, idx, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out, lse


def check_idx(pb, idx, toks, topk):
    ref = O.indexer_topk(pb.ps, pb.qi[toks], pb.w, 0, toks, pb.ki, pb.kis, topk)
    got = np.sort(idx[toks].cpu().numpy(), axis=1)
    ref = np.sort(ref, axis=1)
    bad = np.nonzero(np.any(got != ref, axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ, first token {toks[bad[0]]}"


@pytest.mark.parametrize("q_lens,prefix,topk", [
    ([40], [0], 16),                       # short rows keep everything, long rows select
    ([300, 7, 129], [0, 2000, 513], 64),   # ragged batch with prefixes
    ([64], [3000], 2048),                  # all rows longer than topk
    ([20], [2030], 2048),                  # rows cross t+1 = topk
    ([7], [20000], 16),                    # a small k over a long context
    ([2, 1], [5000, 2047], 2048),          # a group of one token; a sequence with one short row
])
def test_indexer_small_exact(q_lens, prefix, topk):
    pb = Problem(q_lens, prefix, 16, seed=200 + topk, with_indexer=True)
    d = pb.device()
    idx = run_indexer(pb, d, topk)
    check_idx(pb, idx, np.arange(pb.ps.total_q), topk)
    # distinct positions, -1 padding only at the end; a second call gives the same rows
    a = idx.cpu().numpy()
    for r in a:
        v = r[r >= 0]
        assert len(np.unique(v)) == len(v) and np.all(r[len(v):] == -1)
    assert np.array_equal(a, run_indexer(pb, d, topk).cpu().numpy())


def test_indexer_per_token_weights():
    """One weight row per token (token stride 64) instead of a shared row."""
    import torch
    pb = Problem([40, 24], [600, 200], 16, seed=33, with_indexer=True)
    rng = np.random.default_rng(33)
    wt = (2.0 ** -rng.integers(0, 5, (pb.ps.total_q, 64))).astype(np.float32)   # exact like the shared row
    d = pb.device()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    from mla_prefill_attention_gb300 import mla_indexer_topk
    idx = mla_indexer_topk(d["seqs"], d["qi"], torch.from_numpy(wt).cuda(), 64, d["ki"], d["kis"], 300, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    toks = np.arange(pb.ps.total_q)
    ref = O.indexer_topk(pb.ps, pb.qi, wt, 64, toks, pb.ki, pb.kis, 300)
    got = np.sort(idx.cpu().numpy(), axis=1)
    assert np.array_equal(np.sort(ref, axis=1), got)


def test_indexer_signed_scores_and_zero_ties():
    """Per-token weights of both signs make over a quarter of the scores
    negative; 40% of the key rows are zero, so every row holds a block of zero
    scores, and with k near half the row the cut falls inside that block for
    most rows: the lower positions must go first."""
    import torch
    pb = Problem([64, 40], [2000, 1900], 16, seed=34, with_indexer=True)
    rng = np.random.default_rng(34)
    T = pb.ps.total_q
    wt = (rng.choice([-1.0, 1.0], (T, 64)) * 2.0 ** -rng.integers(0, 5, (T, 64))).astype(np.float32)
    ki = pb.ki.reshape(-1, 128).copy()
    ki[rng.random(ki.shape[0]) < 0.4] = 0                        # e4m3 code 0 is +0
    pb.ki = ki.reshape(pb.ki.shape)
    d = pb.device()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    from mla_prefill_attention_gb300 import mla_indexer_topk
    idx = mla_indexer_topk(d["seqs"], d["qi"], torch.from_numpy(wt).cuda(), 64, d["ki"], d["kis"], 1000, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    toks = np.arange(T)
    ref, sc = O.indexer_topk(pb.ps, pb.qi, wt, 64, toks, pb.ki, pb.kis, 1000, want_scores=True, ctx_cap=2100)
    # the case is what it claims: for most rows the 1000th largest score is a zero
    kth = np.array([np.sort(sc[t, :int(pb.ps.prefix_lens[0 if t < 64 else 1]) + (t if t < 64 else t - 64) + 1])[::-1][999]
                    for t in toks])
    assert np.mean(kth == 0.0) > 0.5 and np.any(sc[~np.isnan(sc)] < 0)
    got = idx.cpu().numpy()
    assert np.array_equal(np.sort(ref, axis=1), np.sort(got, axis=1))
    assert all(len(np.unique(r)) == len(r) for r in got)


def test_indexer_clustered_winners():
    """The largest scores all sit in the first 1,500 positions (their key scales
    are 2^10 times the others, exact): after the first compaction the running
    threshold lies above every later score, so the rest of the stream adds
    nothing. The premise is checked on the oracle: every selected position is
    below 1,500."""
    pb = Problem([16], [30000], 16, seed=35, with_indexer=True)
    bt = pb.ps.block_table[0]
    kis = pb.kis.copy()
    for s in range(1500):
        kis[bt[s // 256], s % 256] *= 1024.0
    pb.kis = kis
    d = pb.device()
    k = 1000
    idx = run_indexer(pb, d, k)
    toks = np.arange(16)
    ref = O.indexer_topk(pb.ps, pb.qi, pb.w, 0, toks, pb.ki, pb.kis, k)
    assert np.all(ref < 1500)
    got = idx.cpu().numpy()
    assert np.array_equal(np.sort(ref, axis=1), np.sort(got, axis=1))
    assert all(len(np.unique(r)) == len(r) for r in got)


def test_indexer_rising_scores():
    """Key scales double every 512 positions (exact powers of two), so nearly
    every key scores above the running threshold when it arrives: the buffer
    refills and is compacted every few thousand keys, the worst case for the
    streaming selection. The premise is checked on the oracle: most selected
    positions lie in the last 2k."""
    pb = Problem([4], [30000], 16, seed=36, with_indexer=True)
    n, k = 30004, 1000
    bt = pb.ps.block_table[0]
    kis = pb.kis.copy()
    for s in range(n):
        kis[bt[s // 256], s % 256] = 2.0 ** (s // 512)
    pb.kis = kis
    d = pb.device()
    idx = run_indexer(pb, d, k)
    toks = np.arange(4)
    ref = O.indexer_topk(pb.ps, pb.qi, pb.w, 0, toks, pb.ki, pb.kis, k)
    assert np.mean(ref >= 30000 - 2 * k) > 0.9
    got = idx.cpu().numpy()
    assert np.array_equal(np.sort(ref, axis=1), np.sort(got, axis=1))
    assert all(len(np.unique(r)) == len(r) for r in got)


def test_indexer_all_scores_equal():
    """Every key row is the same, so every score of a token is equal: each
    compaction must fall back to the exact k-th key and keep the lowest
    positions, and the result is positions 0..k-1."""
    pb = Problem([6], [20000], 16, seed=37, with_indexer=True)
    pb.ki[:] = pb.ki.reshape(-1, 128)[0]
    d = pb.device()
    k = 2048
    idx = run_indexer(pb, d, k)
    got = idx.cpu().numpy()
    assert np.array_equal(got, np.tile(np.arange(k, dtype=np.int32), (6, 1)))
    check_idx(pb, idx, np.arange(6), k)


def sample_tile_ids(n_keys):
    """The key tiles (of 128) the indexer's fast path scores first for a group
    whose keys are 0 .. n_keys-1: one every n_tiles // S tiles, S from 8 to 32
    (none when every key fits a token's 5,120-entry buffer)."""
    n_tiles = -(-n_keys // 128)
    if n_tiles * 128 <= 5120:
        return []
    S = min(32, max(8, n_tiles // 32))
    g = n_tiles // S
    return [i * g + g // 2 for i in range(S)]


def test_indexer_fallback_when_the_sample_misleads():
    """The keys of the sampled tiles score 2^10 times higher than the rest
    (their key scales, exact powers of two), so the threshold the sample gives
    lies above every other key and fewer than k keys reach the buffer: the
    group must be redone on the exact streaming path and still match the
    oracle."""
    pb = Problem([1], [30000], 16, seed=38, with_indexer=True)
    n, k = 30001, 1000
    bt = pb.ps.block_table[0]
    kis = pb.kis.copy()
    for tile in sample_tile_ids(n):
        for s in range(tile * 128, min(n, tile * 128 + 128)):
            kis[bt[s // 256], s % 256] *= 1024.0
    pb.kis = kis
    d = pb.device()
    idx = run_indexer(pb, d, k)
    check_idx(pb, idx, np.arange(1), k)
    assert len(np.unique(idx.cpu().numpy()[0])) == k


def test_indexer_fallback_when_a_warp_overflows():
    """The keys in the first 32 slots of every 128-key tile (one TMEM lane
    quadrant, so one epilogue warp) score 2^10 times higher than the rest, so
    far more than a warp's quarter of the candidate buffer clears the sampled
    threshold in that one warp: the group must be redone on the exact path."""
    pb = Problem([2], [30000], 16, seed=39, with_indexer=True)
    n, k = 30002, 1500
    bt = pb.ps.block_table[0]
    kis = pb.kis.copy()
    for s in range(n):
        if s % 128 < 32:
            kis[bt[s // 256], s % 256] *= 1024.0
    pb.kis = kis
    d = pb.device()
    idx = run_indexer(pb, d, k)
    ref = O.indexer_topk(pb.ps, pb.qi, pb.w, 0, np.arange(2), pb.ki, pb.kis, k)
    assert np.all(ref % 128 < 32)
    got = idx.cpu().numpy()
    assert np.array_equal(np.sort(ref, axis=1), np.sort(got, axis=1))
    assert all(len(np.unique(r)) == len(r) for r in got)


def test_indexer_ties_go_to_lower_position():
    """Keys repeat three rows, so whole groups of scores tie at the cut."""
    import torch
    pb = Problem([16], [900], 16, seed=31, with_indexer=True)
    rng = np.random.default_rng(31)
    base = I.e4m3_bits(rng.integers(-3, 4, (3, 128)).astype(np.float64))
    pb.ki = base[rng.integers(0, 3, pb.ps.num_blocks * 256)].reshape(pb.ps.num_blocks, 256, 128)
    d = pb.device()
    idx = run_indexer(pb, d, 100)
    check_idx(pb, idx, np.arange(16), 100)


@pytest.mark.parametrize("H", [16, 64, 128])
def test_sparse_small_vs_oracle(H):
    pb = Problem([50, 30], [700, 100], H, seed=300 + H, with_indexer=True, sm_scale=0.08)
    d = pb.device()
    idx = run_indexer(pb, d, 256)
    out, lse = run_sparse(pb, d, idx)
    toks = np.arange(pb.ps.total_q)
    ora, ora_lse = O.mla_sparse(pb.ps, pb.q, toks, pb.kv, pb.ks, pb.sm_scale, idx.cpu().numpy())
    check_attention(bf16_to_np(out), ora, lse.cpu().numpy(), ora_lse, f"sparse H{H}")


def test_sparse_with_all_keys_matches_dense():
    import torch
    from mla_prefill_attention_gb300 import mla_prefill_dense
    pb = Problem([100], [500], 64, seed=41, with_indexer=True)
    d = pb.device()
    idx = run_indexer(pb, d, 1024)                     # every row keeps all of its <= 600 keys
    out_s, lse_s = run_sparse(pb, d, idx)
    out_d, lse_d = mla_prefill_dense(d["seqs"], d["q"], d["kv"], d["ks"], pb.sm_scale)
    torch.cuda.synchronize()
    # both against the dense oracle: with every key selected the sparse path is the dense one
    toks = np.arange(pb.ps.total_q)
    ora, ora_lse = O.mla_dense(pb.ps, pb.q, toks, pb.kv, pb.ks, pb.sm_scale)
    check_attention(bf16_to_np(out_s), ora, lse_s.cpu().numpy(), ora_lse, "sparse(all) vs dense oracle")
    check_attention(bf16_to_np(out_d), ora, lse_d.cpu().numpy(), ora_lse, "dense vs dense oracle")
    # and against each other: two bf16 results, each rounded on its own, may sit up to
    # two half-ulps apart, so the bound is twice the oracle bound
    mx, mean, _ = rel_errors(bf16_to_np(out_s), bf16_to_np(out_d))
    assert mx <= 2 * TOL_MAX and mean <= 2 * TOL_MEAN, f"sparse(all) vs dense: max {mx:.3e} mean {mean:.3e}"


def test_sparse_padding_and_bad_index():
    import torch
    from mla_prefill_attention_gb300 import MLA_DEVERR_BAD_INDEX, mla_prefill_sparse
    pb = Problem([4], [300], 64, seed=42)
    d = pb.device()
    idx = np.full((4, 64), -1, np.int32)
    idx[0, :3] = [0, 10, 300]
    idx[1, :2] = [5, 301]
    idx[3, 0] = 302                                   # beyond token 3's position 303? no: valid
    idx[3, 1] = 400                                   # beyond its position: flagged, skipped
    ti = torch.from_numpy(idx).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = mla_prefill_sparse(d["seqs"], d["q"], d["kv"], d["ks"], pb.sm_scale, ti, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & MLA_DEVERR_BAD_INDEX
    idx_ok = idx.copy()
    idx_ok[3, 1] = -1
    ora, ora_lse = O.mla_sparse(pb.ps, pb.q, np.arange(4), pb.kv, pb.ks, pb.sm_scale, idx_ok)
    keep = [0, 1, 3]
    check_attention(bf16_to_np(out[keep]), ora[keep], lse[keep].cpu().numpy(), ora_lse[keep], "padding")
    assert torch.all(out[2] == 0) and torch.isinf(lse[2]).all()          # no valid index at all


def test_sparse64k_sampled():
    """8,192 query tokens after 57,344 cached ones. Sampled rows against the
    fp64 oracle (first and last 64, the 16 chunk boundaries +-2, 1,024 uniform):
    index sets bit-exact and attention within the bounds. Then every row: the
    selection against exact fp32 scores and the attention against an fp32
    reference over the selected rows, both in plain PyTorch on the GPU."""
    w = I.WORKLOADS["sparse64k"]
    pb = Problem(w.q_lens, w.prefix_lens, w.heads, w.seed, w.shuffle, w.sm_scale, with_indexer=True)
    d = pb.device()
    idx = run_indexer(pb, d, w.topk)
    toks = sample_rows(pb.ps.cu_seqlens_q, seed=3)
    check_idx(pb, idx, toks, w.topk)
    out, lse = run_sparse(pb, d, idx)
    ora, ora_lse = O.mla_sparse(pb.ps, pb.q[toks], toks, pb.kv, pb.ks, pb.sm_scale, idx[toks].cpu().numpy())
    check_attention(bf16_to_np(out[toks]), ora, lse[toks].cpu().numpy(), ora_lse, "sparse64k")
    check_topk_torch(pb.ps, d["qi"], d["w"], 0, d["ki"], d["kis"], w.topk, idx)
    ref, ref_lse = sparse_reference_torch(pb.ps, d["q"], d["kv"], d["ks"], pb.sm_scale, idx)
    check_attention_torch(out, ref, lse, ref_lse, "sparse64k, every row")


def test_chunked200k_driver():
    """The 200,000-token prompt through the library's chunk driver
    (chunked_prefill_sparse: 33 chunks of 6,144 tokens, each attending to every
    earlier token through the indexer, top-k and sparse attention). Every
    chunk: all rows' selections against exact fp32 scores (plain PyTorch on the
    GPU), and sampled rows (first and last 4, 16 uniform) against the fp64
    oracle, index sets bit-exact and attention within the bounds. The last
    chunk also runs the dense path, 64+ rows against its own oracle."""
    import torch
    from mla_prefill_attention_gb300 import Seqs, chunk_bounds, chunked_prefill_sparse, mla_prefill_dense
    w = I.WORKLOADS["chunked200k"]
    N = w.q_lens[0]
    ps = w.seqs()
    kv, ks = I.gen_latent_cache(w.seed, ps)
    ki, kis = I.gen_indexer_keys(w.seed, ps)
    wh = I.gen_indexer_w(w.seed)
    dkv, dks = torch.from_numpy(kv).cuda(), torch.from_numpy(ks).cuda()
    dki, dkis, dw = torch.from_numpy(ki).cuda(), torch.from_numpy(kis).cuda(), torch.from_numpy(wh).cuda()
    bounds = chunk_bounds(N, w.chunk)
    assert len(bounds) == 33 and bounds[-1] == (196608, 200000)
    n_uni = max(4, UNIFORM_ROWS // 64)
    picks = [sample_tokens(e - s, n_uni, seed=c, edge=4) for c, (s, e) in enumerate(bounds)]
    got = {}
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev_q = {}

    def q_fn(s, e):
        q = torch.from_numpy(I.gen_q_bf16(w.seed, N, w.heads, token_rows=np.arange(s, e)).view(np.int16))
        dev_q["q"] = q.view(torch.bfloat16).cuda()
        return dev_q["q"]

    def qi_fn(s, e):
        dev_q["qi"] = torch.from_numpy(I.gen_indexer_q(w.seed, N, token_rows=np.arange(s, e))).cuda()
        return dev_q["qi"]

    def on_chunk(c, s, e, out, lse, idx):
        sub = I.PagedSeqs(np.array([0, e - s], np.int32), np.array([s], np.int32), ps.block_table, ps.num_blocks)
        check_topk_torch(sub, dev_q["qi"], dw, 0, dki, dkis, w.topk, idx)
        t = torch.from_numpy(picks[c]).cuda()
        got[c] = (bf16_to_np(out[t]), lse[t].cpu().numpy(), idx[t].cpu().numpy())
        if c == len(bounds) - 1:
            seqs = Seqs.from_paged(sub)
            outd, lsed = mla_prefill_dense(seqs, dev_q["q"], dkv, dks, w.sm_scale, dev_err=err)
            td = sample_tokens(e - s, 48, seed=99, edge=8)
            got["dense"] = (td, bf16_to_np(outd[torch.from_numpy(td).cuda()]),
                            lsed[torch.from_numpy(td).cuda()].cpu().numpy())

    chunked_prefill_sparse(ps.block_table, ps.num_blocks, N, w.chunk, q_fn, dkv, dks, qi_fn, dw, 0, dki, dkis,
                           w.sm_scale, topk=w.topk, on_chunk=on_chunk, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for c, (s, e) in enumerate(bounds):
        toks = picks[c]
        sub = I.PagedSeqs(np.array([0, e - s], np.int32), np.array([s], np.int32), ps.block_table, ps.num_blocks)
        qi = I.gen_indexer_q(w.seed, N, token_rows=toks + s)
        ref = O.indexer_topk(sub, qi, wh, 0, toks, ki, kis, w.topk)
        out, lse, idx = got[c]
        assert np.array_equal(np.sort(idx, 1), np.sort(ref, 1)), f"chunk {c}"
        q = I.gen_q_bf16(w.seed, N, w.heads, token_rows=toks + s)
        ora, ora_lse = O.mla_sparse(sub, q, toks, kv, ks, w.sm_scale, ref)
        check_attention(out, ora, lse, ora_lse, f"chunk {c}")
    s, e = bounds[-1]
    td, outd, lsed = got["dense"]
    assert len(td) >= 64
    sub = I.PagedSeqs(np.array([0, e - s], np.int32), np.array([s], np.int32), ps.block_table, ps.num_blocks)
    q = I.gen_q_bf16(w.seed, N, w.heads, token_rows=td + s)
    ora_d, ora_dl = O.mla_dense(sub, q, td, kv, ks, w.sm_scale)
    check_attention(outd, ora_d, lsed, ora_dl, "last chunk dense")


@pytest.mark.parametrize("q_lens,prefix,H,chunks,per_token_w", [
    ([50, 30], [700, 100], 64, 5, False),     # pieces cross a sequence boundary
    ([64, 40], [3000, 200], 128, 3, True),    # one weight row per token, 128 heads
    ([7], [300], 16, 64, False),              # more pieces than 3-token groups: some pieces empty
])
def test_sparse_from_host_matches_device_calls(q_lens, prefix, H, chunks, per_token_w):
    """The host-to-host sparse step (copies overlapped with the indexer, top-k
    and sparse attention of other pieces) returns exactly what the two device
    calls return, and both match the oracle."""
    import torch
    from mla_prefill_attention_gb300 import mla_indexer_topk, mla_prefill_sparse, mla_prefill_sparse_host
    pb = Problem(q_lens, prefix, H, seed=500 + H + chunks, with_indexer=True, sm_scale=0.08)
    T, topk = pb.ps.total_q, 256
    w = pb.w
    if per_token_w:
        rng = np.random.default_rng(7)
        w = (2.0 ** -rng.integers(0, 5, (T, 64))).astype(np.float32)
    stride = 64 if per_token_w else 0
    d = pb.device()
    dw = torch.from_numpy(w).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx_d = mla_indexer_topk(d["seqs"], d["qi"], dw, stride, d["ki"], d["kis"], topk, dev_err=err)
    out_d, lse_d = mla_prefill_sparse(d["seqs"], d["q"], d["kv"], d["ks"], pb.sm_scale, idx_d, dev_err=err)
    torch.cuda.synchronize()
    host_in = {"q": torch.from_numpy(pb.q.view(np.int16)).view(torch.bfloat16), "qi": torch.from_numpy(pb.qi),
               "w": torch.from_numpy(w), "kv": torch.from_numpy(pb.kv), "ks": torch.from_numpy(pb.ks),
               "ki": torch.from_numpy(pb.ki), "kis": torch.from_numpy(pb.kis)}
    host_in = {k: v.pin_memory() for k, v in host_in.items()}
    dev_in = {k: torch.zeros_like(v, device="cuda") for k, v in host_in.items()}
    host_out = {"out": torch.empty((T, H, 512), dtype=torch.bfloat16).pin_memory(),
                "lse": torch.empty((T, H), dtype=torch.float32).pin_memory(),
                "idx": torch.empty((T, topk), dtype=torch.int32).pin_memory()}
    dev_out = {k: torch.zeros_like(v, device="cuda") for k, v in host_out.items()}
    mla_prefill_sparse_host(d["seqs"], host_in, dev_in, host_out, dev_out, pb.sm_scale, w_token_stride=stride,
                            topk=topk, n_chunks=chunks, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(host_out["idx"], idx_d.cpu())
    assert torch.equal(host_out["out"].view(torch.int16), out_d.cpu().view(torch.int16))
    assert torch.equal(host_out["lse"], lse_d.cpu())
    toks = np.arange(T)
    ref = O.indexer_topk(pb.ps, pb.qi, w, stride, toks, pb.ki, pb.kis, topk)
    assert np.array_equal(np.sort(ref, axis=1), np.sort(host_out["idx"].numpy(), axis=1))
    ora, ora_lse = O.mla_sparse(pb.ps, pb.q, toks, pb.kv, pb.ks, pb.sm_scale, host_out["idx"].numpy())
    check_attention(bf16_to_np(host_out["out"]), ora, host_out["lse"].numpy(), ora_lse, f"sparse from host {q_lens}")
