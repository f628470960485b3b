"""Pins of the CPU oracle to things other than itself.

Each test checks the oracle against a closed form, an invariant of softmax
attention, a second formulation (the explicit per-head MLA; exact integer
arithmetic; mpmath exponentials without the max shift) or a library routine.
A dropped term, a wrong sign or index, or a transposed operand in the oracle
fails at least one of them. No GPU is needed.
"""
import math
import os

import numpy as np
import pytest

mpmath = pytest.importorskip("mpmath")

from mla_prefill_attention_gb300 import inputs as I
from mla_prefill_attention_gb300 import flops as F
from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kv_value(kv, ks, bt, b, s, d):
    """sigma_s * dec(code) for position s of sequence b, via torch's e4m3 decoder."""
    import torch
    page = bt[b, s // 256]
    code = int(kv[page, s % 256, d])
    v = torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).double().item()
    return float(ks[page, s % 256]) * v


def _tiny_problem(q_lens, prefix_lens, heads, seed, shuffle=True):
    seqs = I.make_seqs(q_lens, prefix_lens, seed, shuffle)
    q = I.gen_q_bf16(seed, seqs.total_q, heads)
    kv, ks = I.gen_latent_cache(seed, seqs)
    return seqs, q, kv, ks


# --------------------------------------------------------------------------
# closed form (hand-derived two/three-key example)
# --------------------------------------------------------------------------

def test_closed_form_three_keys():
    """P=1 cached token, two new tokens, 1 head, sm_scale 1/2; keys carry
    distinct per-token scales and a RoPE-dim component. Values derived by hand:
      token 0 (position 1): logits (1.5, 1.0); V0=(1,0), V1=(0,2)
      token 1 (position 2): logits (-1.0, 1.0, 0.5); V2=(0.5,0.5)."""
    seqs = I.PagedSeqs(np.array([0, 2], np.int32), np.array([1], np.int32),
                       np.array([[0]], np.int32), 1)
    kv = np.zeros((1, 256, 576), np.uint8)
    ks = np.ones((1, 256), np.float32)
    one, two = 0x38, 0x40                      # e4m3 codes of 1.0 and 2.0
    kv[0, 0, 0], kv[0, 0, 575], ks[0, 0] = one, two, 1.0
    kv[0, 1, 1], kv[0, 1, 575], ks[0, 1] = one, one, 2.0
    kv[0, 2, 0], kv[0, 2, 1], ks[0, 2] = one, one, 0.5
    q = np.zeros((2, 1, 576), np.uint16)
    q[0, 0, 0], q[0, 0, 575] = 0x3F80, 0x3F80   # 1.0, 1.0
    q[1, 0, 1], q[1, 0, 575] = 0x4000, 0xBF80   # 2.0, -1.0
    out, lse = O.mla_dense(seqs, q, [0, 1], kv, ks, 0.5)
    w = 1.0 / (1.0 + math.exp(-0.5))
    assert out[0, 0, 0] == pytest.approx(w, rel=1e-14)
    assert out[0, 0, 1] == pytest.approx(2.0 * (1.0 - w), rel=1e-14)
    assert lse[0, 0] == pytest.approx(1.5 + math.log1p(math.exp(-0.5)), rel=1e-14)
    z = math.exp(-1.0) + math.exp(1.0) + math.exp(0.5)
    assert out[1, 0, 0] == pytest.approx((math.exp(-1.0) + 0.5 * math.exp(0.5)) / z, rel=1e-14)
    assert out[1, 0, 1] == pytest.approx((2.0 * math.exp(1.0) + 0.5 * math.exp(0.5)) / z, rel=1e-14)
    assert lse[1, 0] == pytest.approx(math.log(z), rel=1e-14)
    assert np.all(out[:, :, 2:] == 0.0)


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------

def test_row0_equals_v0_exactly():
    """With no prefix the first token sees only itself: out = V_0 exactly and
    lse = its own logit."""
    seqs, q, kv, ks = _tiny_problem([40], [0], 4, seed=11)
    out, lse = O.mla_dense(seqs, q[[0]], [0], kv, ks, 1.0 / math.sqrt(192))
    page = seqs.block_table[0, 0]
    v0 = np.array([_kv_value(kv, ks, seqs.block_table, 0, 0, d) for d in range(512)])
    for h in range(4):
        assert np.array_equal(out[0, h], v0)
        qh = O.bf16_to_f64(q[0, h])
        k0 = np.array([_kv_value(kv, ks, seqs.block_table, 0, 0, d) for d in range(576)])
        assert lse[0, h] == pytest.approx(math.fsum(qh * k0) / math.sqrt(192), rel=1e-12)
    assert page >= 0


def test_weights_sum_to_one():
    """Every key's value dims equal one constant c (its RoPE dims vary): any
    convex combination returns c, so out == c iff the weights sum to 1."""
    seqs, q, kv, ks = _tiny_problem([37], [300], 2, seed=12)
    kv[:, :, :512] = 0x38                        # 1.0
    ks[:] = 0.75
    out, _ = O.mla_dense(seqs, q, np.arange(37), kv, ks, 0.3)
    assert np.max(np.abs(out - 0.75)) < 1e-12


def test_page_shuffle_invariance():
    """Moving the pages (and the block table with them) changes nothing."""
    seqs, q, kv, ks = _tiny_problem([70], [600], 3, seed=13, shuffle=False)
    sel = np.arange(0, 70, 7)
    out_a, lse_a = O.mla_dense(seqs, q[sel], sel, kv, ks, 0.07)
    perm = np.random.default_rng(5).permutation(seqs.num_blocks).astype(np.int32)
    kv2 = np.empty_like(kv)
    ks2 = np.empty_like(ks)
    kv2[perm] = kv
    ks2[perm] = ks
    bt2 = perm[seqs.block_table]
    seqs2 = I.PagedSeqs(seqs.cu_seqlens_q, seqs.prefix_lens, bt2, seqs.num_blocks)
    out_b, lse_b = O.mla_dense(seqs2, q[sel], sel, kv2, ks2, 0.07)
    assert np.array_equal(out_a, out_b) and np.array_equal(lse_a, lse_b)


def test_prefix_equals_one_shot():
    """New token i after a cached prefix P equals token P+i of a prefill of the
    whole prompt from scratch over the same cache."""
    seqs_full, q_full, kv, ks = _tiny_problem([330], [0], 2, seed=14)
    seqs_pre = I.PagedSeqs(np.array([0, 30], np.int32), np.array([300], np.int32),
                           seqs_full.block_table, seqs_full.num_blocks)
    q_new = q_full[300:]
    out_a, lse_a = O.mla_dense(seqs_full, q_full[[300, 317, 329]], [300, 317, 329], kv, ks, 0.1)
    out_b, lse_b = O.mla_dense(seqs_pre, q_new[[0, 17, 29]], [0, 17, 29], kv, ks, 0.1)
    assert np.array_equal(out_a, out_b) and np.array_equal(lse_a, lse_b)


def test_ragged_batch_equals_each_sequence_alone():
    seqs, q, kv, ks = _tiny_problem([20, 45, 9], [250, 0, 513], 2, seed=15)
    toks = [0, 19, 20, 64, 65, 73]
    out, lse = O.mla_dense(seqs, q[toks], toks, kv, ks, 0.05)
    for b in range(3):
        lo, hi = int(seqs.cu_seqlens_q[b]), int(seqs.cu_seqlens_q[b + 1])
        one = I.PagedSeqs(np.array([0, hi - lo], np.int32), seqs.prefix_lens[b:b + 1],
                          seqs.block_table[b:b + 1], seqs.num_blocks)
        for j, t in enumerate(toks):
            if lo <= t < hi:
                o1, l1 = O.mla_dense(one, q[[t]], [t - lo], kv, ks, 0.05)
                assert np.array_equal(o1[0], out[j]) and np.array_equal(l1[0], lse[j])


# --------------------------------------------------------------------------
# second formulations
# --------------------------------------------------------------------------

def test_bruteforce_mpmath_no_max_shift():
    """Direct softmax in 40-digit arithmetic without subtracting the max,
    dot products by exact summation (fsum of exact products)."""
    seqs, q, kv, ks = _tiny_problem([6, 4], [258, 1], 2, seed=16)
    sm = 1.0 / math.sqrt(192)
    toks = [0, 5, 6, 9]
    out, lse = O.mla_dense(seqs, q[toks], toks, kv, ks, sm)
    mpmath.mp.dps = 40
    for j, t in enumerate(toks):
        b = 0 if t < seqs.cu_seqlens_q[1] else 1
        p = int(seqs.prefix_lens[b]) + t - int(seqs.cu_seqlens_q[b])
        keys = np.array([[_kv_value(kv, ks, seqs.block_table, b, s, d) for d in range(576)]
                         for s in range(p + 1)])
        for h in range(2):
            qh = O.bf16_to_f64(q[t, h])
            logits = [mpmath.mpf(math.fsum(qh * keys[s])) * mpmath.mpf(sm) for s in range(p + 1)]
            e = [mpmath.exp(x) for x in logits]
            z = mpmath.fsum(e)
            for d in (0, 1, 255, 511):
                ref = mpmath.fsum(e[s] * keys[s, d] for s in range(p + 1)) / z
                assert out[j, h, d] == pytest.approx(float(ref), rel=1e-11, abs=1e-14)
            assert lse[j, h] == pytest.approx(float(mpmath.log(z)), rel=1e-12)


def test_absorbed_equals_explicit_per_head_form():
    """Weight absorption: with per-head up-projections W_UK, W_UV (128 x 512),
    explicit heads k_h = [W_UK c ; r] (192 dims), v_h = W_UV c, q_h = [q_nope ;
    q_rope], scale 1/sqrt(192), equal W_UV applied to the latent output of the
    absorbed query [W_UK^T q_nope ; q_rope] over K = [c ; r], V = c."""
    rng = np.random.default_rng(7)
    H, T, P = 3, 5, 260
    seqs = I.make_seqs([T], [P], 17, True)
    _, _, kv, ks = _tiny_problem([T], [P], 1, seed=17)
    n = P + T
    lat = np.array([[_kv_value(kv, ks, seqs.block_table, 0, s, d) for d in range(576)] for s in range(n)])
    c, r = lat[:, :512], lat[:, 512:]
    W_UK = rng.standard_normal((H, 128, 512)) / 16.0
    W_UV = rng.standard_normal((H, 128, 512)) / 16.0
    q_nope = rng.standard_normal((T, H, 128))
    q_rope = rng.standard_normal((T, H, 64))
    scale = 1.0 / math.sqrt(192.0)
    q_abs = np.concatenate([np.einsum("hkd,thk->thd", W_UK, q_nope), q_rope], axis=2)
    lat_out, _ = O.mla_dense(seqs, q_abs, np.arange(T), kv, ks, scale)
    o_abs = np.einsum("hkd,thd->thk", W_UV, lat_out)
    for t in range(T):
        p = P + t
        for h in range(H):
            k = np.concatenate([c[: p + 1] @ W_UK[h].T, r[: p + 1]], axis=1)     # [p+1, 192]
            v = c[: p + 1] @ W_UV[h].T                                         # [p+1, 128]
            qh = np.concatenate([q_nope[t, h], q_rope[t, h]])
            lg = k @ qh * scale
            w = np.exp(lg - lg.max())
            o = (w[:, None] * v).sum(0) / w.sum()
            np.testing.assert_allclose(o_abs[t, h], o, rtol=1e-10, atol=1e-12)


def test_sparse_with_all_keys_equals_dense():
    seqs, q, kv, ks = _tiny_problem([12], [400], 2, seed=18)
    toks = np.arange(12)
    topk = 512
    idx = np.full((12, topk), -1, np.int32)
    rng = np.random.default_rng(3)
    for t in toks:
        p = 400 + t
        idx[t, : p + 1] = rng.permutation(p + 1)          # order and padding do not matter
    out_d, lse_d = O.mla_dense(seqs, q, toks, kv, ks, 0.07)
    out_s, lse_s = O.mla_sparse(seqs, q, toks, kv, ks, 0.07, idx)
    np.testing.assert_allclose(out_s, out_d, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse_s, lse_d, rtol=1e-13)


def test_sparse_subset_matches_restricted_softmax():
    """Sparse over a subset equals dense attention over a cache in which only
    that subset is visible (other keys' logits pushed to -inf by construction)."""
    seqs, q, kv, ks = _tiny_problem([3], [50], 1, seed=19)
    idx = np.full((3, 8), -1, np.int32)
    idx[:, :4] = [[0, 7, 31, 50], [1, 2, 3, 51], [52, 10, 20, 30]]
    out_s, lse_s = O.mla_sparse(seqs, q, np.arange(3), kv, ks, 0.09, idx)
    for t in range(3):
        keys = np.array([[_kv_value(kv, ks, seqs.block_table, 0, s, d) for d in range(576)]
                         for s in idx[t, :4]])
        lg = keys @ O.bf16_to_f64(q[t, 0]) * 0.09
        w = np.exp(lg - lg.max())
        np.testing.assert_allclose(out_s[t, 0], (w[:, None] * keys[:, :512]).sum(0) / w.sum(), rtol=1e-12)
        assert lse_s[t, 0] == pytest.approx(lg.max() + math.log(w.sum()), rel=1e-13)


def _indexer_bruteforce_int(qi, w_j, ki, kscale_pow, bt, prefix, tokens, topk):
    """Exact integer scores: q,k are small integers, w_h = 2^-j_h, key scale 2^e_s.
    score * 2^16 is an integer; rank by (score desc, s asc)."""
    import torch
    qv = torch.from_numpy(qi).view(torch.float8_e4m3fn).double().numpy().astype(np.int64)
    kvals = torch.from_numpy(ki).view(torch.float8_e4m3fn).double().numpy().astype(np.int64)
    res = []
    for j, t in enumerate(tokens):
        p = prefix + t
        best = []
        for s in range(p + 1):
            pg, sl = bt[0, s // 256], s % 256
            dots = qv[j] @ kvals[pg, sl]                              # [64] exact ints
            acc = 0
            for h in range(64):
                if dots[h] > 0:
                    acc += int(dots[h]) << (8 - int(w_j[h]))              # w = 2^-j, j <= 8
            acc = acc << (8 + int(kscale_pow[pg, sl]))                    # key scale 2^e, e >= -8
            best.append((-acc, s))
        best.sort()
        sel = sorted(s for _, s in best[:topk])
        res.append(sel + [-1] * (topk - len(sel)))
    return np.array(res, np.int32)


def test_indexer_matches_integer_bruteforce_with_ties():
    """Small integer q/k (many tied scores), power-of-two head weights and key
    scales: the oracle's fp64 selection equals an exact int64 ranking."""
    seqs = I.make_seqs([24], [280], 21, True)
    T = 24
    rng = np.random.default_rng(21)
    qi = I.e4m3_bits(rng.integers(-2, 3, (T, 64, 128)).astype(np.float64))
    ki = np.zeros((seqs.num_blocks, 256, 128), np.uint8)
    ki[:] = I.e4m3_bits(rng.integers(-2, 3, ki.shape).astype(np.float64))
    w_j = rng.integers(0, 5, 64)
    w = np.ldexp(1.0, -w_j).astype(np.float32)
    e = rng.integers(-2, 3, (seqs.num_blocks, 256))
    kscale = np.ldexp(1.0, e).astype(np.float32)
    topk = 64
    toks = np.arange(T)
    got = O.indexer_topk(seqs, qi, w, 0, toks, ki, kscale, topk)
    ref = _indexer_bruteforce_int(qi, w_j, ki, e, seqs.block_table, 280, toks, topk)
    assert np.array_equal(got, ref)


def test_indexer_tie_break_lower_position():
    """Keys repeat one of three rows, so scores tie in large groups; the cut
    inside a tied group keeps the lowest positions."""
    seqs = I.make_seqs([4], [700], 24, True)
    rng = np.random.default_rng(24)
    qi = I.e4m3_bits(rng.integers(-3, 4, (4, 64, 128)).astype(np.float64))
    base = I.e4m3_bits(rng.integers(-3, 4, (3, 128)).astype(np.float64))
    which = rng.integers(0, 3, seqs.num_blocks * 256)
    ki = base[which].reshape(seqs.num_blocks, 256, 128)
    ks = np.ones((seqs.num_blocks, 256), np.float32)
    w = np.ones(64, np.float32)
    topk = 100
    got = O.indexer_topk(seqs, qi, w, 0, np.arange(4), ki, ks, topk)
    ref = _indexer_bruteforce_int(qi, np.zeros(64, np.int64), ki, np.zeros((seqs.num_blocks, 256), np.int64),
                                  seqs.block_table, 700, np.arange(4), topk)
    assert np.array_equal(got, ref)
    # the cut falls inside a tied group for at least one token
    bt = seqs.block_table
    pos_row = [which[bt[0, s // 256] * 256 + s % 256] for s in range(704)]
    assert any(len(set(pos_row[s] for s in got[t])) < 3 for t in range(4))


def test_indexer_short_context_keeps_all():
    seqs = I.make_seqs([10], [0], 22, False)
    qi, w, ki, ks = I.gen_indexer_inputs(22, seqs)
    idx = O.indexer_topk(seqs, qi, w, 0, np.arange(10), ki, ks, 16)
    for t in range(10):
        assert list(idx[t, : t + 1]) == list(range(t + 1))
        assert np.all(idx[t, t + 1:] == -1)


def test_indexer_per_token_weights_stride():
    """w with a token stride equals w broadcast when every token row is the same."""
    seqs = I.make_seqs([5], [300], 23, True)
    qi, w, ki, ks = I.gen_indexer_inputs(23, seqs)
    w_tok = np.tile(w, (5, 1))
    a = O.indexer_topk(seqs, qi, w, 0, np.arange(5), ki, ks, 32)
    b = O.indexer_topk(seqs, qi, w_tok, 64, np.arange(5), ki, ks, 32)
    assert np.array_equal(a, b)


# --------------------------------------------------------------------------
# the pages' printed accounting
# --------------------------------------------------------------------------

def _golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = v
    return vals


def test_flop_and_byte_accounting_matches_footnote():
    g = _golden("footnote1_sparse_mla.txt")
    assert F.FLOPS_PER_PAIR_HEAD == int(g["flops_per_row_head"])
    topk, rb, ib = int(g["topk"]), int(g["row_bytes"]), int(g["index_bytes"])
    assert round(topk * (rb + ib) / 1e6, 2) == float(g["rows_mb"])
    for H in (8, 64):
        fl = topk * H * F.FLOPS_PER_PAIR_HEAD
        by = F.sparse_bytes_per_query(topk, H, rb, ib)
        assert round(fl / 1e6, 1 if H == 8 else 0) == float(g[f"heads_{H}_mflop"])
        assert round(by / 1e6, 2) == float(g[f"heads_{H}_mb"])
        assert round(fl / by) == int(g[f"heads_{H}_flop_per_byte"])


def test_pair_counts():
    assert F.causal_pairs(512, 0) == 131328
    assert F.causal_pairs(4096, 12288) == 58722304
    assert F.causal_pairs(32768, 0) == 536887296
    assert F.dense_pairs([9216, 16384, 24576, 32768], [0] * 4) == 1015587328
    assert F.causal_pairs(8192, 57344) == 503320576
    # sparse pair count equals the brute-force count of min(topk, p+1)
    for t, p, k in [(100, 0, 16), (50, 10, 40), (3000, 1000, 2048), (10, 5000, 2048)]:
        assert F.sparse_pairs([t], [p], k) == sum(min(k, p + i + 1) for i in range(t))
