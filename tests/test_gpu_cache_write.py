"""Cache write of the new tokens on the GPU against the oracle: codes and scales
bit for bit, rows placed through the block table, nothing else touched."""
import numpy as np
import pytest

from oracle import oracle as O
from mla_prefill_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_prefill_attention_gb300 import build
    build.build()


def _special_rows(lat, d):
    """Overwrite a few rows with the quantiser's edge cases (when there are enough)."""
    vals = np.array([O.e4m3_value(c) for c in range(128)])
    mids = (vals[1:127] + vals[:126]) / 2
    rng = np.random.default_rng(d)
    rows = []
    rows.append(np.zeros(d))                                            # scale 1
    rows.append(-np.zeros(d))                                           # -0 everywhere
    r = rng.choice(mids, d) * rng.choice([-1.0, 1.0], d) * 2.0 ** -3    # exact ties at scale 2^-3
    r[5] = 448 * 2.0 ** -3
    rows.append(r)
    rows.append(np.full(d, -3.25))                                      # every code at -448
    r = rng.standard_normal(d) * 1e37                                   # near the bf16 maximum
    r[0] = 3.3895313892515355e38
    rows.append(r)
    rows.append(rng.standard_normal(d) * 1e-39)                         # bf16 subnormals: subnormal scale
    r = np.zeros(d)
    r[d - 1] = 2.0 ** -133                                              # the smallest bf16 alone
    rows.append(r)
    n = min(len(rows), lat.shape[0])
    lat[:n] = I.bf16_bits(np.stack(rows[:n]))
    return lat


def _case(q_lens, prefix, seed, extra_blocks=1):
    seqs = I.make_seqs(q_lens, prefix, seed, True, extra_blocks)
    T = seqs.total_q
    lat = _special_rows(I.gen_new_rows_bf16(seed, T, 576), 576)
    kid = _special_rows(I.gen_new_rows_bf16(seed, T, 128, I.T_NEWKIDX), 128)[::-1].copy()
    nb = seqs.num_blocks
    rng = np.random.default_rng(seed)
    kv0 = rng.integers(0, 256, (nb, 256, 576), dtype=np.uint8)
    ks0 = rng.standard_normal((nb, 256)).astype(np.float32)
    ki0 = rng.integers(0, 256, (nb, 256, 128), dtype=np.uint8)
    kis0 = rng.standard_normal((nb, 256)).astype(np.float32)
    return seqs, lat, kid, (kv0, ks0, ki0, kis0)


def _run_gpu(seqs, lat, kid, caches, dev_err_expected=0):
    import torch
    from mla_prefill_attention_gb300 import Seqs, mla_kv_append
    kv0, ks0, ki0, kis0 = caches
    dev = "cuda"
    kv, ks = torch.from_numpy(kv0).to(dev), torch.from_numpy(ks0).to(dev)
    ki, kis = torch.from_numpy(ki0).to(dev), torch.from_numpy(kis0).to(dev)
    latd = torch.from_numpy(lat.view(np.int16)).to(dev).view(torch.bfloat16)
    kidd = None if kid is None else torch.from_numpy(kid.view(np.int16)).to(dev).view(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    mla_kv_append(Seqs.from_paged(seqs), latd, kv, ks, kidd, ki if kid is not None else None,
                  kis if kid is not None else None, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == dev_err_expected
    return kv.cpu().numpy(), ks.cpu().numpy(), ki.cpu().numpy(), kis.cpu().numpy()


def _same(a, b, what):
    a, b = np.asarray(a), np.asarray(b)
    if a.dtype == np.float32:
        a, b = a.view(np.uint32), b.view(np.uint32)
    bad = np.argwhere(a != b)
    assert bad.size == 0, f"{what}: {len(bad)} mismatches, first at {bad[:3].tolist()}"


@pytest.mark.parametrize("q_lens,prefix,with_key", [
    ([1], [0], True),
    ([10, 0, 300], [250, 7, 500], True),      # ragged, an empty sequence, page crossings
    ([513], [255], False),                    # latent only
    ([7, 9, 33], [0, 1000, 31], True),
])
def test_append_bitexact(q_lens, prefix, with_key):
    seqs, lat, kid, caches = _case(q_lens, prefix, seed=sum(q_lens) + len(prefix))
    kid = kid if with_key else None
    g = _run_gpu(seqs, lat, kid, caches)
    o = O.kv_append(seqs, lat, kid, caches[0], caches[1], caches[2] if with_key else None,
                    caches[3] if with_key else None)
    _same(g[0], o[0], "latent codes")
    _same(g[1], o[1], "latent scales")
    if with_key:
        _same(g[2], o[2], "key codes")
        _same(g[3], o[3], "key scales")
    else:
        _same(g[2], caches[2], "key cache untouched")
        _same(g[3], caches[3], "key scales untouched")


def test_unmapped_page_writes_nothing_for_that_token():
    from mla_prefill_attention_gb300 import MLA_DEVERR_BAD_PAGE
    seqs, lat, kid, caches = _case([20, 300], [0, 200], seed=9)
    seqs.block_table[1, 1] = seqs.num_blocks + 3          # positions 256..511 of sequence 1
    g = _run_gpu(seqs, lat, kid, caches, dev_err_expected=MLA_DEVERR_BAD_PAGE)
    ok = I.make_seqs([20, 300], [0, 200], 9, True, 1)
    # the oracle without the bad page: sequence 1 keeps only positions 200..255
    keep = np.r_[np.arange(20), 20 + np.arange(56)]
    sub = I.PagedSeqs(np.array([0, 20, 76], np.int32), ok.prefix_lens.copy(), ok.block_table.copy(), ok.num_blocks)
    o = O.kv_append(sub, lat[keep], kid[keep], *caches)
    for i, what in enumerate(("latent codes", "latent scales", "key codes", "key scales")):
        _same(g[i], o[i], what)


def test_append_then_attend_matches_oracle():
    """Write-then-attend: the new tokens' rows go into a cache that already
    holds a generated prefix, then dense attention reads them back."""
    import torch
    from mla_prefill_attention_gb300 import Seqs, mla_prefill_dense
    from tests.parity import bf16_to_np, check_attention
    seqs = I.make_seqs([200, 70], [300, 0], 21, True)
    kvp, ksp = I.gen_latent_cache(21, seqs)          # prefix rows (new positions get overwritten)
    T = seqs.total_q
    lat = I.gen_new_rows_bf16(21, T, 576)
    g = _run_gpu(seqs, lat, None, (kvp, ksp, np.zeros((1, 256, 128), np.uint8), np.zeros((1, 256), np.float32)))
    okv, oks, _, _ = O.kv_append(seqs, lat, None, kvp, ksp)
    _same(g[0], okv, "latent codes")
    _same(g[1], oks, "latent scales")
    q = I.gen_q_bf16(21, T, 16)
    d = Seqs.from_paged(seqs)
    out, lse = mla_prefill_dense(d, torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16),
                                 torch.from_numpy(g[0]).cuda(), torch.from_numpy(g[1]).cuda(), 0.08)
    torch.cuda.synchronize()
    toks = np.arange(T)
    ora, ora_lse = O.mla_dense(seqs, q, toks, okv, oks, 0.08)
    check_attention(bf16_to_np(out), ora, lse.cpu().numpy(), ora_lse, "append+dense")


@pytest.mark.slow
def test_append_full_size_32k():
    """The size the bench times: 32,768 new tokens of one sequence, shuffled pages."""
    seqs, lat, kid, caches = _case([32768], [0], seed=2)
    g = _run_gpu(seqs, lat, kid, caches)
    o = O.kv_append(seqs, lat, kid, *caches)
    for i, what in enumerate(("latent codes", "latent scales", "key codes", "key scales")):
        _same(g[i], o[i], what)
