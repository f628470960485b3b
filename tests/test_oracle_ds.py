"""Pins of the oracle's 656-byte row format ("GLM-5.3-Optimierungen, Teil 2",
footnote 1: 656 FP8 KV bytes per token in the fp8_ds_mla format), read as 512
e4m3 latent codes, one fp32 scale per 128 latent dims and 64 bf16 RoPE values.
Each pin is independent of the oracle's code: an equivalence with the
580-byte format where both hold the same numbers, a scaling invariance that
fixes which scale serves which dims, and an exact round trip through the
generator's packer."""
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


def _ds_row(codes512, scales4, rope_bits64):
    row = np.zeros(656, dtype=np.uint8)
    row[:512] = codes512
    row[512:528] = np.asarray(scales4, dtype="<f4").view(np.uint8)
    row[528:] = np.asarray(rope_bits64, dtype="<u2").view(np.uint8)
    return row


def _cases(seed, n_tok):
    rng = np.random.default_rng(seed)
    ps = I.make_seqs([n_tok], [3], seed, shuffle=True)
    n_keys = ps.seq_len(0)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    lat = rng.choice(finite, (n_keys, 512))
    rope_codes = rng.choice(finite, (n_keys, 64))
    sig_exp = rng.integers(-6, 3, n_keys)
    return ps, lat, rope_codes, sig_exp


def test_equal_scales_match_the_580_byte_rows_exactly():
    """With the four scales of a row equal to one power of two sigma and the RoPE
    values equal to sigma * dec(code) (bf16-exact), a 656-byte row holds the
    same 576 numbers as the 580-byte row (codes, sigma): dense and sparse
    attention agree bit for bit."""
    ps, lat, rope_codes, sig_exp = _cases(11, 9)
    n_keys = ps.seq_len(0)
    sig = np.exp2(sig_exp.astype(np.float64))
    rope_vals = sig[:, None] * _e4m3_value(rope_codes)
    rope_bits = I.bf16_bits(rope_vals)
    assert np.array_equal(rope_bits.astype(np.uint32) << 16,
                          rope_vals.astype(np.float32).view(np.uint32))          # bf16-exact
    codes580 = np.zeros((ps.num_blocks, 256, 576), np.uint8)
    scale580 = np.ones((ps.num_blocks, 256), np.float32)
    ds = np.tile(_ds_row(np.zeros(512, np.uint8), [1, 1, 1, 1], np.zeros(64, np.uint16)), (ps.num_blocks, 256, 1))
    for s in range(n_keys):
        pg, sl = ps.block_table[0, s // 256], s % 256
        codes580[pg, sl, :512] = lat[s]
        codes580[pg, sl, 512:] = rope_codes[s]
        scale580[pg, sl] = sig[s]
        ds[pg, sl] = _ds_row(lat[s], [sig[s]] * 4, rope_bits[s])
    q = I.gen_q_bf16(11, ps.total_q, 4)
    toks = np.arange(ps.total_q)
    a_out, a_lse = O.mla_dense(ps, q, toks, codes580, scale580, 0.07)
    b_out, b_lse = O.mla_dense_ds(ps, q, toks, ds, 0.07)
    assert np.array_equal(a_out, b_out) and np.array_equal(a_lse, b_lse)
    idx = np.full((ps.total_q, 8), -1, np.int32)
    for t in range(ps.total_q):
        idx[t, : min(8, 4 + t)] = np.arange(min(8, 4 + t))[::-1]
    a_out, a_lse = O.mla_sparse(ps, q, toks, codes580, scale580, 0.07, idx)
    b_out, b_lse = O.mla_sparse_ds(ps, q, toks, ds, 0.07, idx)
    assert np.array_equal(a_out, b_out) and np.array_equal(a_lse, b_lse)


@pytest.mark.parametrize("g", [0, 1, 2, 3])
def test_a_group_scale_serves_its_128_dims(g):
    """Doubling scale g of every key while halving query dims 128g..128g+127
    leaves every logit unchanged (power-of-two factors are exact), so the lse
    stays and exactly output dims 128g..128g+127 double."""
    ps = I.make_seqs([6], [20], 12, shuffle=True)
    ds = I.gen_latent_cache_ds(12, ps)
    q = I.bf16_bits(np.random.default_rng(12).standard_normal((ps.total_q, 2, 576)))
    qd = O.bf16_to_f64(q)
    toks = np.arange(ps.total_q)
    out0, lse0 = O.mla_dense_ds(ps, qd, toks, ds, 0.09)
    ds2 = ds.copy()
    sc = ds2[..., 512:528].copy().view("<f4")
    sc[..., g] *= 2.0
    ds2[..., 512:528] = sc.view(np.uint8)
    q2 = qd.copy()
    q2[..., 128 * g:128 * (g + 1)] *= 0.5
    out1, lse1 = O.mla_dense_ds(ps, q2, toks, ds2, 0.09)
    assert np.array_equal(lse0, lse1)
    want = out0.copy()
    want[..., 128 * g:128 * (g + 1)] *= 2.0
    assert np.array_equal(out1, want)


def test_packer_round_trip_is_exact():
    """Rows whose values are exactly (group absmax/448) * e4m3 values and
    bf16-exact RoPE values pack and decode to themselves: with one key the
    output is the key's first 512 values, and a query that is a unit vector
    on RoPE dim i gives lse = sm_scale * K[512 + i]."""
    rng = np.random.default_rng(13)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F and (c & 0x7F) != 0x7E], dtype=np.uint8)
    x = np.zeros((1, 576))
    for g in range(4):
        codes = rng.choice(finite, 128)
        codes[0] = 0x7E                                  # 448: the group's absmax
        x[0, 128 * g:128 * (g + 1)] = 2.0 ** (g - 2) * _e4m3_value(codes)
    x[0, 512:] = O.bf16_to_f64(I.bf16_bits(rng.standard_normal(64)))
    row = I.pack_ds_rows(x)
    ps = I.make_seqs([1], [0], 13, shuffle=False)
    cache = np.tile(row[0], (ps.num_blocks, 256, 1))
    qv = np.zeros((1, 65, 576))
    for i in range(64):
        qv[0, i, 512 + i] = 1.0
    qv[0, 64, 0] = 1.0
    out, lse = O.mla_dense_ds(ps, qv, np.arange(1), cache, 0.5)
    assert np.array_equal(out[0, 0], x[0, :512])
    assert np.array_equal(lse[0, :64], 0.5 * x[0, 512:])
