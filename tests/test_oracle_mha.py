"""Pins of the oracle's non-absorbed (MHA) form ("GLM-5.3-Optimierungen, Teil 2",
section Ausprobieren: without sparse_mla_force_mqa, prefill batches whose
prompts fit within the top-k of 2,048 tokens take the dense MHA path).

Each pin is independent of the MHA function's code:
* the absorption identity: per head, attention with keys [W_UK c ; r] and
  values W_UV c equals W_UV applied to the absorbed attention whose query is
  [W_UK^T q_nope ; q_rope] (the absorbed oracle is pinned on its own, in
  test_oracle_pins.py), with the same log-sum-exp;
* a one-key context: the output is W_UV c_0 and the lse the single logit,
  written out here with numpy from the e4m3 bit fields;
* heads are independent: permuting the heads of q and of the weights permutes
  the outputs exactly."""
import math

import numpy as np
import pytest

from mla_prefill_attention_gb300 import inputs as I
from oracle import oracle as O

pytestmark = pytest.mark.filterwarnings("ignore")


@pytest.fixture(scope="module", autouse=True)
def _built():
    I.build_generator()
    O.build()


def _e4m3_value(codes):
    """Values of e4m3 codes from the OCP bit fields (written out here, apart from
    the oracle's table)."""
    c = np.asarray(codes, dtype=np.int64)
    s = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1 + m / 8.0) * 2.0 ** (e - 7.0))
    return s * mag


def _bf16(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("q_lens,prefix,H,shuffle", [([5, 9], [3, 0], 4, True), ([1, 17], [40, 260], 2, True)])
def test_mha_equals_the_absorbed_form(q_lens, prefix, H, shuffle):
    ps = I.make_seqs(q_lens, prefix, 21, shuffle=shuffle)
    kv, ks = I.gen_latent_cache(21, ps)
    q = _bf16(I.gen_q_mha(21, ps.total_q, H))
    W = _bf16(I.gen_w_ukv(21, H))
    toks = np.arange(ps.total_q)
    sm = 1.0 / math.sqrt(192.0)
    out, lse = O.mla_mha(ps, q, toks, kv, ks, W, sm)
    qa = np.zeros((ps.total_q, H, 576))
    qa[:, :, :512] = np.einsum("thi,hid->thd", q[:, :, :128], W[:, :128, :])
    qa[:, :, 512:] = q[:, :, 128:]
    out_a, lse_a = O.mla_dense(ps, qa, toks, kv, ks, sm)
    want = np.einsum("hid,thd->thi", W[:, 128:, :], out_a)
    scale = np.abs(want).max()
    assert np.max(np.abs(out - want)) <= 1e-11 * scale
    assert np.max(np.abs(lse - lse_a)) <= 1e-11


def test_mha_one_key_context_closed_form():
    """The first token of a sequence without a prefix sees only itself."""
    H = 3
    ps = I.make_seqs([1, 4], [0, 0], 22, shuffle=True)
    kv, ks = I.gen_latent_cache(22, ps)
    qb = I.gen_q_mha(22, ps.total_q, H)
    q = _bf16(qb)
    W = _bf16(I.gen_w_ukv(22, H))
    sm = 0.11
    for t, b in ((0, 0), (1, 1)):
        out, lse = O.mla_mha(ps, qb[t:t + 1], np.array([t]), kv, ks, I.gen_w_ukv(22, H), sm)
        pg = ps.block_table[b, 0]
        k = float(ks[pg, 0]) * _e4m3_value(kv[pg, 0])
        for h in range(H):
            v = W[h, 128:] @ k[:512]
            kn = W[h, :128] @ k[:512]
            logit = sm * (q[t, h, :128] @ kn + q[t, h, 128:] @ k[512:])
            assert np.allclose(out[0, h], v, rtol=1e-13, atol=1e-13 * np.abs(v).max())
            assert abs(lse[0, h] - logit) <= 1e-12 * max(1.0, abs(logit))


def test_mha_heads_are_independent():
    H = 4
    ps = I.make_seqs([6, 3], [2, 5], 23, shuffle=True)
    kv, ks = I.gen_latent_cache(23, ps)
    q = I.gen_q_mha(23, ps.total_q, H)
    W = I.gen_w_ukv(23, H)
    toks = np.arange(ps.total_q)
    out, lse = O.mla_mha(ps, q, toks, kv, ks, W, 0.09)
    perm = np.array([2, 0, 3, 1])
    out_p, lse_p = O.mla_mha(ps, q[:, perm], toks, kv, ks, W[perm], 0.09)
    assert np.array_equal(out_p, out[:, perm]) and np.array_equal(lse_p, lse[:, perm])
    # a subset of the tokens gives the same rows
    sub = np.array([8, 1, 4])
    out_s, lse_s = O.mla_mha(ps, q[sub], sub, kv, ks, W, 0.09)
    assert np.array_equal(out_s, out[sub]) and np.array_equal(lse_s, lse[sub])
