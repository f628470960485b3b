"""Pins of the oracle's cache write (per-token absmax/448 e4m3 quantisation and
paged placement) to things other than itself: torch's e4m3 conversion (a
library routine), a brute-force nearest-value search over torch's decoder,
rows whose codes and scale are known in closed form, and the error bound of
round-to-nearest. No GPU is needed."""
import numpy as np
import pytest
import torch

from mla_prefill_attention_gb300 import inputs as I
from oracle import oracle as O


def _torch_codes(v32):
    """torch's float32 -> e4m3fn conversion after clamping to +-448 (torch maps
    magnitudes past the largest finite value to NaN instead of saturating)."""
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_values():
    """Values of all 256 codes by torch's decoder (NaN at 0x7f and 0xff)."""
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def _samples(seed=0):
    vals = _torch_values()
    fin = np.sort(np.unique(np.abs(vals[np.isfinite(vals)])))
    mids = ((fin[1:] + fin[:-1]) / 2).astype(np.float32)         # exact ties (5 significant bits)
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    rng = np.random.default_rng(seed)
    rand = np.exp2(rng.uniform(-14, 10, 20000)).astype(np.float32)
    big = np.array([448, 460, 463.99, 464, 464.01, 470, 479, 480, 1e6, 3e38], np.float32)
    tiny = np.array([0.0, 2.0 ** -10, 2.0 ** -11, 1e-30, 2.0 ** -9 * 1.5, 2.0 ** -9 * 7.5], np.float32)
    pos = np.concatenate([mids, up, dn, rand, big, tiny, fin.astype(np.float32)])
    return np.concatenate([pos, -pos])


def test_nearest_matches_torch_conversion():
    v = _samples()
    np.testing.assert_array_equal(O.e4m3_nearest(v), _torch_codes(v))


def test_nearest_by_bruteforce_over_torch_decoder():
    vals = _torch_values()
    finite = np.where(np.isfinite(vals))[0]
    v = _samples(1)[::7]
    got = O.e4m3_nearest(v)
    for x, c in zip(v.astype(np.float64), got):
        a = min(abs(x), 448.0)
        d = np.abs(np.abs(vals[finite]) - a)
        best = finite[d == d.min()]
        best = best[best < 128]                                    # magnitude codes
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert (int(c) & 0x7F) == int(want), (x, int(c), best)
        assert (int(c) >> 7) == int(np.signbit(x))


def test_roundtrip_of_every_finite_code():
    vals = _torch_values()
    codes = np.array([c for c in range(256) if np.isfinite(vals[c])], np.uint8)
    np.testing.assert_array_equal(O.e4m3_nearest(vals[codes].astype(np.float32)), codes)


def test_row_of_scaled_codes_gives_back_codes_and_power_of_two_scale():
    """x = dec(c) * 2^k with one element at 448 * 2^k: the scale is exactly
    2^k and every code comes back (no rounding is involved anywhere)."""
    vals = _torch_values()
    rng = np.random.default_rng(3)
    finite = np.array([c for c in range(256) if np.isfinite(vals[c])])
    for k in (-20, -7, 0, 5, 19):
        c = rng.choice(finite, 576).astype(np.uint8)
        c[rng.integers(576)] = 0xFE if k % 2 else 0x7E
        x = I.bf16_bits(vals[c] * 2.0 ** k)
        codes, scale = O.quantize_row(x)
        assert scale == np.float32(2.0 ** k)
        np.testing.assert_array_equal(codes, c)


def test_zero_row_has_scale_one():
    x = np.zeros(576, np.uint16)
    x[::3] = 0x8000                                                 # -0 keeps its sign
    codes, scale = O.quantize_row(x)
    assert scale == 1.0
    assert set(codes[::3]) == {0x80} and set(np.delete(codes, np.s_[::3])) == {0}


def test_tiny_row_scale_is_floored_at_smallest_normal():
    """amax / 448 below 2^-126 (a row of bf16 subnormals): the scale stops at
    2^-126, whose reciprocal 2^126 is exact, so codes are nearest(x * 2^126)."""
    x = np.zeros(576, np.uint16)
    x[:8] = [1, 2, 3, 0x8005, 0x7F, 0x40, 0x8001, 0x11]           # bf16 subnormals k * 2^-133
    codes, scale = O.quantize_row(x)
    assert scale == np.float32(2.0 ** -126)
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(codes, _torch_codes((xf * 2.0 ** 126).astype(np.float32)))


def test_row_error_bound_and_peak_code():
    """Round to nearest: |dec(code) * scale - x| is at most half a step of the
    e4m3 grid at x / scale (relative 2^-4 in the normal range, 2^-10 absolute
    below 2^-6), plus the binary32 rounding of the reciprocal and the product;
    the largest magnitude lands on +-448; the scale is amax / 448 within
    binary32 rounding."""
    rows = I.gen_new_rows_bf16(5, 64, 576)
    for x in rows:
        xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
        codes, scale = O.quantize_row(x)
        amax = np.abs(xf).max()
        assert abs(float(scale) - amax / 448.0) <= amax / 448.0 * 2.0 ** -24
        dec = _torch_values()[codes] * float(scale)
        q = np.abs(xf) / float(scale)
        step = np.where(q >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(q, 2.0 ** -6))) - 3), 2.0 ** -9)
        err = np.abs(dec - xf)
        assert np.all(err <= (0.5 * step + q * 2.0 ** -22) * float(scale))
        i = int(np.argmax(np.abs(xf)))
        assert codes[i] & 0x7F == 0x7E


def test_append_places_rows_by_block_table_and_touches_nothing_else():
    seqs = I.make_seqs([10, 0, 300], [250, 7, 500], seed=4, shuffle=True, extra_blocks=2)
    T = seqs.total_q
    lat = I.gen_new_rows_bf16(4, T, 576)
    kid = I.gen_new_rows_bf16(4, T, 128, I.T_NEWKIDX)
    nb = seqs.num_blocks
    kv0 = np.full((nb, 256, 576), 0x55, np.uint8)
    ks0 = np.full((nb, 256), -7.0, np.float32)
    ki0 = np.full((nb, 256, 128), 0x33, np.uint8)
    kis0 = np.full((nb, 256), -3.0, np.float32)
    kv, ks, ki, kis = O.kv_append(seqs, lat, kid, kv0, ks0, ki0, kis0)
    written = np.zeros((nb, 256), bool)
    t = 0
    for b in range(seqs.batch):
        n = int(seqs.cu_seqlens_q[b + 1] - seqs.cu_seqlens_q[b])
        for i in range(n):
            p = int(seqs.prefix_lens[b]) + i
            page, slot = seqs.block_table[b, p // 256], p % 256
            c, sc = O.quantize_row(lat[t])
            np.testing.assert_array_equal(kv[page, slot], c)
            assert ks[page, slot] == sc
            c, sc = O.quantize_row(kid[t])
            np.testing.assert_array_equal(ki[page, slot], c)
            assert kis[page, slot] == sc
            written[page, slot] = True
            t += 1
    assert t == T and written.sum() == T
    assert np.all(kv[~written] == 0x55) and np.all(ks[~written] == -7.0)
    assert np.all(ki[~written] == 0x33) and np.all(kis[~written] == -3.0)
    kv2, ks2, ki2, kis2 = O.kv_append(seqs, lat, None, kv0, ks0)
    assert ki2 is None and np.array_equal(kv2, kv) and np.array_equal(ks2, ks)


def test_append_rejects_unmapped_page():
    seqs = I.make_seqs([4], [0], seed=0, shuffle=False)
    seqs.block_table[0, 0] = seqs.num_blocks
    lat = I.gen_new_rows_bf16(0, 4, 576)
    with pytest.raises(ValueError):
        O.kv_append(seqs, lat, None, np.zeros((seqs.num_blocks, 256, 576), np.uint8),
                    np.ones((seqs.num_blocks, 256), np.float32))
