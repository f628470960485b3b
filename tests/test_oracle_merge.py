"""Pins of the oracle's merge of partial attention results: closed forms, and
the identity it exists for (attention over each part of a split key set,
merged, equals attention over the whole set), checked against the oracle's
dense attention, which has its own pins. No GPU is needed."""
import math

import numpy as np
import pytest

from mla_prefill_attention_gb300 import inputs as I
from oracle import oracle as O


def test_single_part_is_returned_unchanged():
    rng = np.random.default_rng(0)
    o = rng.standard_normal((1, 5, 512))
    lse = rng.standard_normal((1, 5)) * 30
    out, l = O.merge(o, lse)
    np.testing.assert_array_equal(out, o[0])
    np.testing.assert_allclose(l, lse[0], rtol=0, atol=1e-12)


def test_equal_weights_average_and_add_ln_n():
    rng = np.random.default_rng(1)
    o = rng.standard_normal((3, 4, 512))
    lse = np.tile(rng.standard_normal(4), (3, 1))
    out, l = O.merge(o, lse)
    np.testing.assert_allclose(out, o.mean(axis=0), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(l, lse[0] + math.log(3), rtol=0, atol=1e-12)


def test_two_parts_closed_form_and_shift_invariance():
    """Two parts with lse a and b: weights 1/(1+e^(b-a)) and 1/(1+e^(a-b)),
    lse = a + ln(1 + e^(b-a)); adding c to both lse moves lse by c only."""
    o = np.stack([np.full((1, 512), 2.0), np.full((1, 512), -1.0)])
    a, b = 0.3, -1.2
    out, l = O.merge(o, np.array([[a], [b]]))
    wa = 1.0 / (1.0 + math.exp(b - a))
    np.testing.assert_allclose(out[0], 2.0 * wa - 1.0 * (1 - wa), rtol=1e-14)
    assert abs(l[0] - (a + math.log1p(math.exp(b - a)))) < 1e-14
    out2, l2 = O.merge(o, np.array([[a + 700.0], [b + 700.0]]))
    np.testing.assert_allclose(out2, out, rtol=1e-13)
    assert abs(l2[0] - l[0] - 700.0) < 1e-10


def test_empty_parts():
    rng = np.random.default_rng(2)
    o = rng.standard_normal((2, 3, 512))
    lse = np.array([[0.5, -np.inf, -np.inf], [-np.inf, 1.5, -np.inf]])
    out, l = O.merge(o, lse)
    np.testing.assert_array_equal(out[0], o[0, 0])
    np.testing.assert_array_equal(out[1], o[1, 1])
    assert np.all(out[2] == 0) and l[2] == -np.inf
    assert l[0] == 0.5 and l[1] == 1.5


def _partials(seqs, q, kv, ks, toks, sets, sm):
    """Oracle sparse attention of each token over each of its key subsets."""
    outs, lses = [], []
    width = max(1, max(len(s) for per in sets for s in per))
    for part in range(len(sets[0])):
        idx = np.full((len(toks), width), -1, np.int32)
        for j, per in enumerate(sets):
            idx[j, :len(per[part])] = per[part]
        o, l = O.mla_sparse(seqs, q[toks], toks, kv, ks, sm, idx)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


@pytest.mark.parametrize("split", ["round_robin_4", "random_3"])
def test_merged_partials_equal_attention_over_the_union(split):
    """DCP stores every n-th token on one GPU (GLM-5.3 Teil 2, DCP section); the
    merge of the shards' partial results must be attention over all keys."""
    seqs = I.make_seqs([40, 25], [100, 0], 7, True)
    q = I.gen_q_bf16(7, seqs.total_q, 4)
    kv, ks = I.gen_latent_cache(7, seqs)
    sm = 1.0 / math.sqrt(192.0)
    toks = np.arange(seqs.total_q)
    rng = np.random.default_rng(11)
    sets = []
    for t in toks:
        b = 0 if t < 40 else 1
        p = int(seqs.prefix_lens[b]) + int(t - seqs.cu_seqlens_q[b])
        keys = np.arange(p + 1)
        if split == "round_robin_4":
            sets.append([keys[keys % 4 == r] for r in range(4)])
        else:
            lab = rng.integers(0, 3, p + 1)
            sets.append([keys[lab == r] for r in range(3)])
    outs, lses = _partials(seqs, q, kv, ks, toks, sets, sm)
    H = q.shape[1]
    out, lse = O.merge(outs.reshape(outs.shape[0], -1, 512), lses.reshape(lses.shape[0], -1))
    ref, ref_lse = O.mla_dense(seqs, q, toks, kv, ks, sm)
    np.testing.assert_allclose(out.reshape(len(toks), H, 512), ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(len(toks), H), ref_lse, rtol=0, atol=1e-12)
