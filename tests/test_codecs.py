"""Storage codecs: the oracle's decoders and the generator's encoders against
the format definitions and against PyTorch's own float8/bfloat16 routines."""
import os

import numpy as np
import pytest
import torch

from mla_prefill_attention_gb300 import inputs as I
from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_special_values():
    for line in open(os.path.join(GOLDEN, "e4m3_special_values.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        code, val = line.split()
        got = O.e4m3_value(int(code, 16))
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == float(val)
            assert np.signbit(got) == val.startswith("-")


def test_e4m3_table_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([O.e4m3_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_monotone_and_roundtrip():
    pos = np.array([O.e4m3_value(c) for c in range(0x7F)])
    assert np.all(np.diff(pos) > 0)                 # codes 0x00..0x7E strictly increasing
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = np.array([O.e4m3_value(int(c)) for c in codes])
    assert np.array_equal(I.e4m3_bits(vals), codes)


def test_e4m3_encoder_rne_and_saturation():
    cases = {1.0625: 0x38, 1.1875: 0x3A, 2.0 ** -10: 0x00, 3 * 2.0 ** -11: 0x01,
             15 * 2.0 ** -10: 0x08, 500.0: 0x7E, 1e9: 0x7E, -1e9: 0xFE, 464.0: 0x7E}
    for x, c in cases.items():
        assert int(I.e4m3_bits(np.array([x]))[0]) == c, x


def test_e4m3_encoder_matches_torch_rounding():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(5000) * 0.01])
    x = x[np.abs(x) < 448]
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # x is float32-exact, so torch's single rounding float32 -> e4m3 is the reference
    got = I.e4m3_bits(x.astype(np.float32).astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_decode_and_encode_match_torch():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, 50000, dtype=np.uint64).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = O.bf16_to_f64(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    x = (rng.standard_normal(50000) * 10.0).astype(np.float32)
    ref_b = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(I.bf16_bits(x.astype(np.float64)), ref_b)


def test_bf16_ties_to_even():
    cases = {1.0 + 2.0 ** -8: 0x3F80, 1.0 + 3 * 2.0 ** -8: 0x3F82, 1.0 + 2.0 ** -7: 0x3F81}
    for x, c in cases.items():
        assert int(I.bf16_bits(np.array([x]))[0]) == c


def test_generator_rows_are_independent_streams():
    a = I.gen_q_bf16(5, 10, 4)
    b = I.gen_q_bf16(5, 10, 4, token_rows=[7, 2])
    assert np.array_equal(a[[7, 2]], b)
    seqs = I.make_seqs([10], [20], 5, True)
    kv, ks = I.gen_latent_cache(5, seqs)
    c, s = I.latent_rows(5, 0, [3, 29])
    bt = seqs.block_table
    assert np.array_equal(kv[bt[0, 0], 3], c[0]) and ks[bt[0, 0], 29] == s[1]
    # per-token scale is absmax/448 of the drawn row, so the largest code is +-448
    vals = np.array([O.e4m3_value(int(x)) for x in c[0]])
    assert np.max(np.abs(vals)) == 448.0


def test_parity_rounding_allowance():
    """The attention check measures error beyond the bf16 rounding of the output:
    the exact result rounded to bf16 scores zero there (while its raw error is
    not zero), and a planted error of 3e-2 of a row's RMS still fails."""
    torch = pytest.importorskip("torch")
    from tests.parity import TOL_MAX, bf16_half_spacing, rel_errors
    rng = np.random.default_rng(5)
    ora = rng.standard_normal((200, 512)) * np.exp2(rng.uniform(-6, 6, (200, 1)))
    ora[:, 7] *= 6.0                                         # entries far above their row's RMS
    rounded = torch.from_numpy(ora).to(torch.bfloat16).double().numpy()
    assert np.all(np.abs(rounded - ora) <= bf16_half_spacing(ora))
    raw_mx, _, _ = rel_errors(rounded, ora)
    mx, mean, _ = rel_errors(rounded, ora, beyond_rounding=True)
    assert raw_mx > 0.01 and mx == 0.0 and mean == 0.0
    bad = rounded.copy()
    rms = np.sqrt(np.mean(ora[3] ** 2))
    bad[3, 100] += 3e-2 * rms
    mx, _, _ = rel_errors(bad, ora, beyond_rounding=True)
    assert mx > TOL_MAX
