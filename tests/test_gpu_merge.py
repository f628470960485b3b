"""Log-sum-exp merge of partial attention results on the GPU: against the
oracle's merge on the same inputs, and composed with the sparse kernel over a
DCP-style round-robin split of the keys, against the oracle's dense attention."""
import math

import numpy as np
import pytest

from oracle import oracle as O
from mla_prefill_attention_gb300 import inputs as I
from tests.parity import TOL_LSE_ABS, TOL_MAX, TOL_MEAN, bf16_to_np, check_attention, rel_errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_prefill_attention_gb300 import build
    build.build()


def _parts(n, rows, seed):
    rng = np.random.default_rng(seed)
    o = I.bf16_bits(rng.standard_normal((n, rows, 512)) * np.exp2(rng.uniform(-3, 3, (n, rows, 1))))
    lse = rng.uniform(-5.0, 30.0, (n, rows)).astype(np.float32)
    lse[:, rows // 3] = -np.inf                                  # a row with no keys in any part
    if n > 1:
        lse[0, ::5] = -np.inf                                    # part 0 empty on some rows
        lse[1:, 1::7] = -np.inf                                  # only part 0 on others
        lse[1, 2::11] = lse[0, 2::11] + 60.0                     # one part dominates
    return o, lse


def _gpu_merge(o, lse, in_place=False):
    import torch
    from mla_prefill_attention_gb300 import mla_merge_attn
    outs = [torch.from_numpy(p.view(np.int16)).cuda().view(torch.bfloat16) for p in o]
    lses = [torch.from_numpy(l).cuda() for l in lse]
    out, l = mla_merge_attn(outs, lses, out=outs[0] if in_place else None)
    torch.cuda.synchronize()
    return bf16_to_np(out), l.cpu().numpy()


@pytest.mark.parametrize("n,rows,in_place", [(1, 37, False), (2, 1000, False), (3, 513, True), (8, 64, False)])
def test_merge_matches_oracle(n, rows, in_place):
    o, lse = _parts(n, rows, seed=n * 100 + rows)
    got, got_lse = _gpu_merge(o, lse, in_place)
    ref, ref_lse = O.merge(o, lse.astype(np.float64))
    empty = np.isneginf(ref_lse)
    assert np.all(got[empty] == 0) and np.all(np.isneginf(got_lse[empty]))
    assert np.all(np.isfinite(got_lse[~empty]))
    # fp32 arithmetic and one bf16 rounding: within 2^-8 of each value
    rms = np.sqrt(np.mean(ref[~empty] ** 2, axis=1, keepdims=True))
    err = np.abs(got[~empty] - ref[~empty])
    assert np.all(err <= np.abs(ref[~empty]) * 2.0 ** -8 + rms * 1e-5)
    assert np.max(np.abs(got_lse[~empty] - ref_lse[~empty])) <= 1e-5 * max(1.0, np.abs(ref_lse[~empty]).max())


def _check_composed(parts, part_refs, out, lse, ref, ref_lse, what):
    """A merge of GPU partial results, checked stage by stage: every part
    against the oracle on its own keys (the attention tolerance), the merge
    against the oracle's merge of the same bf16 parts (fp32 arithmetic plus one
    bf16 rounding), and the result against the oracle on all keys. The last
    carries two bf16 roundings (the parts', then the merge's) and the parts'
    kernel errors through a convex combination, so its bound is twice the
    single-call tolerance, as for any comparison of two rounded GPU results."""
    import torch
    for i, ((o, l), (ro, rl)) in enumerate(zip(parts, part_refs)):
        gl = l.cpu().numpy().astype(np.float64)
        empty = np.isneginf(rl)                                  # a part with no keys for that row
        assert np.array_equal(np.isneginf(gl), empty), f"{what}: part {i} empty rows differ"
        check_attention(bf16_to_np(o), ro, np.where(empty, 0.0, gl), np.where(empty, 0.0, rl), f"{what}: part {i}")
    po = np.stack([o.float().cpu().numpy().astype(np.float64).reshape(-1, 512) for o, _ in parts])
    pl = np.stack([l.cpu().numpy().astype(np.float64).reshape(-1) for _, l in parts])
    mo, ml = O.merge(po, pl)
    g = bf16_to_np(out).reshape(-1, 512)
    keep = ~np.isneginf(ml)
    rms = np.sqrt(np.mean(mo[keep] ** 2, axis=1, keepdims=True))
    assert np.all(np.abs(g[keep] - mo[keep]) <= np.abs(mo[keep]) * 2.0 ** -8 + rms * 1e-5), f"{what}: merge stage"
    mx, mean, _ = rel_errors(bf16_to_np(out), ref)
    assert mx <= 2 * TOL_MAX and mean <= 2 * TOL_MEAN, f"{what}: end to end max {mx:.3e} mean {mean:.3e}"
    dl = float(np.max(np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse)))
    assert dl <= 2 * TOL_LSE_ABS, f"{what}: lse {dl:.3e}"
    assert torch.isfinite(out.float()).all()


def _sparse(seqs_d, q, kv, ks, idx, sm):
    import torch
    from mla_prefill_attention_gb300 import mla_prefill_sparse
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = mla_prefill_sparse(seqs_d, q, kv, ks, sm, torch.from_numpy(idx).cuda(), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out, lse


def test_round_robin_shards_merge_to_dense():
    """DCP keeps every n-th token on one GPU (GLM-5.3 Teil 2, DCP section):
    attention over each of four round-robin shards (the sparse kernel with the
    shard's positions as its index list), merged, is attention over all keys."""
    import torch
    from mla_prefill_attention_gb300 import Seqs, mla_merge_attn
    seqs = I.make_seqs([300, 5], [900, 0], 31, True)
    H = 64
    q = I.gen_q_bf16(31, seqs.total_q, H)
    kv, ks = I.gen_latent_cache(31, seqs)
    sm = 1.0 / math.sqrt(192.0)
    T = seqs.total_q
    pos = np.array([int(seqs.prefix_lens[0]) + t if t < 300 else t - 300 for t in range(T)])
    d = Seqs.from_paged(seqs)
    qd = torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16)
    kvd, ksd = torch.from_numpy(kv).cuda(), torch.from_numpy(ks).cuda()
    toks = np.arange(T)
    parts, refs = [], []
    for r in range(4):
        idx = np.full((T, 320), -1, np.int32)
        for t in range(T):
            sel = np.arange(r, pos[t] + 1, 4)
            idx[t, :len(sel)] = sel
        parts.append(_sparse(d, qd, kvd, ksd, idx, sm))
        refs.append(O.mla_sparse(seqs, q, toks, kv, ks, sm, idx))
    out, lse = mla_merge_attn([o for o, _ in parts], [l for _, l in parts])
    torch.cuda.synchronize()
    ref, ref_lse = O.mla_dense(seqs, q, toks, kv, ks, sm)
    _check_composed(parts, refs, out, lse, ref, ref_lse, "round-robin shards merged")


def test_split_index_lists_merge_to_sparse():
    """Each token's selected set cut in two (first half, second half of its
    list), each half attended by the sparse kernel, merged: attention over the
    whole set."""
    import torch
    from mla_prefill_attention_gb300 import Seqs, mla_merge_attn
    seqs = I.make_seqs([64], [3000], 41, True)
    H = 64
    q = I.gen_q_bf16(41, seqs.total_q, H)
    kv, ks = I.gen_latent_cache(41, seqs)
    sm = 1.0 / math.sqrt(192.0)
    rng = np.random.default_rng(41)
    T = seqs.total_q
    idx = np.full((T, 2048), -1, np.int32)
    for t in range(T):
        p = 3000 + t
        idx[t] = np.sort(rng.choice(p + 1, 2048, replace=False))
    d = Seqs.from_paged(seqs)
    qd = torch.from_numpy(q.view(np.int16)).cuda().view(torch.bfloat16)
    kvd, ksd = torch.from_numpy(kv).cuda(), torch.from_numpy(ks).cuda()
    toks = np.arange(T)
    halves = [np.ascontiguousarray(idx[:, :1024]), np.ascontiguousarray(idx[:, 1024:])]
    parts = [_sparse(d, qd, kvd, ksd, h, sm) for h in halves]
    refs = [O.mla_sparse(seqs, q, toks, kv, ks, sm, h) for h in halves]
    out, lse = mla_merge_attn([o for o, _ in parts], [l for _, l in parts])
    torch.cuda.synchronize()
    ref, ref_lse = O.mla_sparse(seqs, q, toks, kv, ks, sm, idx)
    _check_composed(parts, refs, out, lse, ref, ref_lse, "split lists merged")
