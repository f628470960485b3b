"""Shared helpers of the GPU parity tests: problem construction from the
seeded generators, upload, sampling of rows, and the tolerance check."""
from __future__ import annotations

import math
import os

import numpy as np

from mla_prefill_attention_gb300 import inputs as I

# attention tolerance, relative to the rms of each oracle output row
TOL_MAX = 2e-2
TOL_MEAN = 2e-3
TOL_LSE_ABS = 1e-3
# How far the raw error may sit above the floor that rounding the exact result
# to bf16 already gives on the same rows, as a fraction of the bounds above.
FLOOR_MARGIN = 0.5

# Uniform rows per sequence or chunk in the sampled checks of the large
# workloads (first and last 64 rows and every chunk boundary +-2 come on top).
UNIFORM_ROWS = int(os.environ.get("MLA_TEST_UNIFORM_ROWS", "1024"))
EDGE_ROWS = 64


def rel_errors(gpu: np.ndarray, ora: np.ndarray, beyond_rounding: bool = False):
    """Errors relative to the RMS of each output row (one (token, head) vector
    of 512 values): returns (max, mean) of |gpu - ora| / rms_row, and the global
    rms. Rows whose oracle output is exactly zero are compared absolutely.

    Reading of "relative to the output RMS": per output row. Against a single
    RMS over the whole output the max bound cannot be met by any bf16 result
    once a row's entries exceed ~5x the global RMS (rounding a value to bf16
    moves it by up to 2^-8 of itself); early causal rows, which average only a
    few cache rows, reach 12x on the tiny workload.

    beyond_rounding: the error of each element is first reduced by half the
    bf16 spacing at the oracle's value, the most that rounding the exact
    result to bf16 can move it, so an exact result delivered in bf16 scores
    zero and what remains is the computation's own error."""
    o = ora.astype(np.float64).reshape(-1, ora.shape[-1])
    g = gpu.astype(np.float64).reshape(-1, ora.shape[-1])
    rms_row = np.sqrt(np.mean(o ** 2, axis=1, keepdims=True))
    rms_row[rms_row == 0] = 1.0
    d = np.abs(g - o)
    if beyond_rounding:
        d = np.maximum(d - bf16_half_spacing(o), 0.0)
    r = d / rms_row
    return float(r.max()), float(r.mean()), math.sqrt(float(np.mean(o ** 2)))


def bf16_half_spacing(x):
    """Half the distance between neighbouring bf16 values at |x| (8 significant
    bits: 2^(e-8) for |x| in [2^e, 2^(e+1))), the most rounding x to bf16 can
    move it; 0 at 0."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def round_bf16(x):
    """x rounded to the nearest bf16 value (8 significant bits, ties to even),
    as float64; the bf16 exponent range is not modelled (attention outputs lie
    far inside it)."""
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.rint(m * 256.0), e - 8)


def attention_errors(gpu_out, ora_out):
    """(own max, own mean, raw max, raw mean, floor max, floor mean, rms): the
    error beyond the bf16 rounding of the output, the raw error, and the raw
    error of the oracle's own result rounded to bf16 (the floor no bf16 output
    can go below), all relative to each row's RMS."""
    mx, mean, rms = rel_errors(gpu_out, ora_out, beyond_rounding=True)
    raw_mx, raw_mean, _ = rel_errors(gpu_out, ora_out)
    fl_mx, fl_mean, _ = rel_errors(round_bf16(ora_out), ora_out)
    return mx, mean, raw_mx, raw_mean, fl_mx, fl_mean, rms


def check_attention(gpu_out, ora_out, gpu_lse=None, ora_lse=None, what="", lse_extra=None):
    """Two bounds, both relative to each output row's RMS:
    * the error beyond the bf16 rounding of the exact result (rel_errors with
      beyond_rounding) is at most TOL_MAX (max) and TOL_MEAN (mean);
    * the raw error is at most the floor that rounding the oracle's exact
      result to bf16 gives on the same rows, plus FLOOR_MARGIN of those bounds.
    LSE within TOL_LSE_ABS absolute, plus lse_extra per row where a format's own
    rounding of the keys adds a known amount (see ds_lse_bound)."""
    assert np.all(np.isfinite(gpu_out)), f"{what}: non-finite output"
    mx, mean, raw_mx, raw_mean, fl_mx, fl_mean, rms = attention_errors(gpu_out, ora_out)
    msg = (f"{what}: beyond bf16 rounding max {mx:.3e} mean {mean:.3e}; raw max {raw_mx:.3e} mean {raw_mean:.3e}; "
           f"bf16 floor max {fl_mx:.3e} mean {fl_mean:.3e} (rms {rms:.3e})")
    print(msg)
    assert mx <= TOL_MAX and mean <= TOL_MEAN, msg
    assert raw_mx <= fl_mx + FLOOR_MARGIN * TOL_MAX and raw_mean <= fl_mean + FLOOR_MARGIN * TOL_MEAN, msg
    if gpu_lse is not None:
        err = np.abs(gpu_lse.astype(np.float64) - ora_lse)
        tol = TOL_LSE_ABS + (0.0 if lse_extra is None else np.asarray(lse_extra, dtype=np.float64))
        assert np.all(err <= tol), f"{what}: lse max abs err {float(err.max()):.3e} (allowed {float(np.max(tol)):.3e})"
    return mx, mean


# f16 keeps 11 significant bits: rounding to nearest moves a value by at most 2^-11 of it
F16_UNIT_ROUNDOFF = 2.0 ** -11


def ds_lse_bound(ps, q, kv_ds, sm_scale, toks, idx=None):
    """Per (token, head) row of the selected tokens: how far the logits can move
    when a 656-byte row's keys are rounded once to f16 (their per-group scales
    make them inexact in any 16-bit operand), u * sm_scale * max_s sum_d
    |q_d| |K_s[d]| over the row's keys s (u = 2^-11), which bounds the move of the
    log-sum-exp. q: torch bf16 [Tq, H, 576] on the GPU, kv_ds: torch uint8 cache;
    idx: the sparse index lists (default: the causal dense keys)."""
    import torch
    kvf = kv_ds.view(-1, 656)
    cu = [int(x) for x in ps.cu_seqlens_q]
    out = np.zeros((len(toks), q.shape[1]))
    for n, t in enumerate(toks):
        b = max(i for i in range(ps.batch) if cu[i] <= t)
        p = int(ps.prefix_lens[b]) + int(t) - cu[b]
        pos = (torch.arange(p + 1, device=q.device) if idx is None else idx[int(t)].long())
        pos = pos[pos >= 0]
        K = decode_ds_rows_torch(kvf[_cache_rows(ps, b, pos)]).abs().double()
        mag = q[int(t)].double().abs() @ K.t()                  # [H, keys]
        out[n] = (F16_UNIT_ROUNDOFF * sm_scale * mag.max(dim=1).values).cpu().numpy()
    return out


def bf16_to_np(t):
    """torch bf16 tensor -> float64 numpy."""
    return t.float().cpu().numpy().astype(np.float64)


class Problem:
    """One dense/sparse workload on host (seeded) and, on demand, device."""

    def __init__(self, q_lens, prefix_lens, heads, seed, shuffle=True, sm_scale=1.0 / math.sqrt(192.0),
                 with_indexer=False, extra_blocks=0):
        self.ps = I.make_seqs(q_lens, prefix_lens, seed, shuffle, extra_blocks)
        self.seed, self.heads, self.sm_scale = seed, heads, sm_scale
        self.q = I.gen_q_bf16(seed, self.ps.total_q, heads)
        self.kv, self.ks = I.gen_latent_cache(seed, self.ps)
        if with_indexer:
            self.qi, self.w, self.ki, self.kis = I.gen_indexer_inputs(seed, self.ps)

    def device(self):
        import torch
        from mla_prefill_attention_gb300 import Seqs
        d = {"seqs": Seqs.from_paged(self.ps)}
        d["q"] = torch.from_numpy(self.q.view(np.int16)).view(torch.bfloat16).cuda()
        d["kv"] = torch.from_numpy(self.kv).cuda()
        d["ks"] = torch.from_numpy(self.ks).cuda()
        if hasattr(self, "qi"):
            d["qi"] = torch.from_numpy(self.qi).cuda()
            d["w"] = torch.from_numpy(self.w).cuda()
            d["ki"] = torch.from_numpy(self.ki).cuda()
            d["kis"] = torch.from_numpy(self.kis).cuda()
        return d


def sample_tokens(total: int, n_uniform: int, seed: int, edge: int = 8, boundaries=(), reach: int = 1):
    """First/last `edge` tokens, tokens within +-reach of each boundary, n_uniform random."""
    rng = np.random.default_rng(seed)
    s = set(range(min(edge, total))) | set(range(max(0, total - edge), total))
    for b in boundaries:
        for d in range(-reach, reach + 1):
            if 0 <= b + d < total:
                s.add(b + d)
    s |= set(rng.integers(0, total, n_uniform).tolist()) if total > 0 else set()
    return np.array(sorted(s), dtype=np.int64)


def sample_rows(cu_seqlens, seed: int, n_uniform: int = None, edge: int = EDGE_ROWS, chunks: int = 16,
                extra_boundaries=()):
    """The stratified sample of the large workloads' checks, per sequence: its
    first and last `edge` tokens, the tokens within +-2 of each boundary of its
    `chunks` equal chunks (and of extra_boundaries, global indices), and
    n_uniform (UNIFORM_ROWS by default) uniform draws. Returns sorted global
    token indices."""
    n_uniform = UNIFORM_ROWS if n_uniform is None else n_uniform
    cu = [int(x) for x in cu_seqlens]
    out = set()
    for b in range(len(cu) - 1):
        c0, n = cu[b], cu[b + 1] - cu[b]
        if n == 0:
            continue
        bounds = [n * k // chunks for k in range(1, chunks)]
        bounds += [x - c0 for x in extra_boundaries if c0 <= x < c0 + n]
        local = sample_tokens(n, n_uniform, seed + 7919 * b, edge=edge, boundaries=bounds, reach=2)
        out |= set((local + c0).tolist())
    return np.array(sorted(out), dtype=np.int64)


# ---------------------------------------------------------------------------
# full-size checks on the GPU in plain PyTorch (an independent calculation,
# used where the fp64 oracle cannot cover every row in reasonable time)
# ---------------------------------------------------------------------------
def check_attention_torch(gpu_out, ref_out, gpu_lse=None, ref_lse=None, what="", lse_extra=None):
    """check_attention on the GPU against an fp32 reference (torch tensors
    [..., 512]); the reference's own error (~1e-6 of a row) is far below the
    bounds. Returns (own max, own mean, raw max, raw mean)."""
    import torch
    g, r = gpu_out.float().reshape(-1, gpu_out.shape[-1]), ref_out.float().reshape(-1, ref_out.shape[-1])
    assert bool(torch.isfinite(g).all()), f"{what}: non-finite output"
    rms = r.pow(2).mean(dim=1, keepdim=True).sqrt()
    rms = torch.where(rms > 0, rms, torch.ones_like(rms))
    _, e = torch.frexp(r)
    hs = torch.where(r != 0, torch.ldexp(torch.ones_like(r), (e - 9).float()), torch.zeros_like(r))
    d = (g - r).abs()
    own = (d - hs).clamp_min(0) / rms
    raw = d / rms
    fl = (r.to(torch.bfloat16).float() - r).abs() / rms
    vals = [float(x) for x in (own.max(), own.mean(), raw.max(), raw.mean(), fl.max(), fl.mean())]
    msg = (f"{what}: beyond bf16 rounding max {vals[0]:.3e} mean {vals[1]:.3e}; raw max {vals[2]:.3e} "
           f"mean {vals[3]:.3e}; bf16 floor max {vals[4]:.3e} mean {vals[5]:.3e}")
    assert vals[0] <= TOL_MAX and vals[1] <= TOL_MEAN, msg
    assert vals[2] <= vals[4] + FLOOR_MARGIN * TOL_MAX and vals[3] <= vals[5] + FLOOR_MARGIN * TOL_MEAN, msg
    print(msg)
    if gpu_lse is not None:
        dl = (gpu_lse.double() - ref_lse.double()).abs()
        tol = TOL_LSE_ABS + (0.0 if lse_extra is None else lse_extra.double())
        assert bool((dl <= tol).all()), f"{what}: lse max abs err {float(dl.max()):.3e}"
    return vals[:4]


def _cache_rows(ps, b, positions):
    """Physical cache rows of positions (int64 tensor) of sequence b."""
    import torch
    bt = torch.as_tensor(ps.block_table[b], device=positions.device, dtype=torch.int64)
    return bt[positions // 256] * 256 + positions % 256


def sparse_reference_torch(ps, q, kv, ks, sm_scale, idx, block=64):
    """Sparse MLA in plain PyTorch fp32 (TF32 off) for every new token:
    gathered rows K_s = ks_s * dec(kv_s), V_s = K_s[:512], softmax over the
    token's index list (-1 skipped). Returns (out f32 [Tq,H,512], lse [Tq,H])."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        T, H = q.shape[0], q.shape[1]
        out = torch.empty((T, H, 512), dtype=torch.float32, device=q.device)
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
        kvf = kv.view(-1, 576)
        ksf = ks.view(-1)
        cu = [int(x) for x in ps.cu_seqlens_q]
        for b in range(ps.batch):
            for t0 in range(cu[b], cu[b + 1], block):
                t1 = min(t0 + block, cu[b + 1])
                ix = idx[t0:t1].long()
                ok = ix >= 0
                rows = _cache_rows(ps, b, ix.clamp_min(0))
                K = kvf[rows].view(torch.float8_e4m3fn).float() * ksf[rows][..., None]   # [n, k, 576]
                lg = torch.einsum("thd,tsd->ths", q[t0:t1].float(), K) * sm_scale
                lg = lg.masked_fill(~ok[:, None, :], float("-inf"))
                l = torch.logsumexp(lg, dim=-1)
                p = torch.exp(lg - torch.where(torch.isfinite(l), l, torch.zeros_like(l))[..., None])
                out[t0:t1] = torch.einsum("ths,tsd->thd", p, K[..., :512])
                lse[t0:t1] = l
        return out, lse
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def check_topk_torch(ps, qi, w, w_stride, ki, kis, topk, idx, block=16, tokens=None):
    """Every row of an indexer top-k result against scores computed in plain
    PyTorch fp32 on the GPU. With integer e4m3 inputs and power-of-two weights
    and key scales every product and partial sum is an exact fp32 value, so
    these scores equal the fp64 definition under any summation order. The
    expected set of a row is every position scoring above the k-th largest
    score plus the lowest positions scoring equal to it (ties go to the lower
    position); rows of p+1 <= topk keep 0..p. Also checks the row layout:
    distinct positions, -1 padding only at the end. tokens: (t0, t1) global range
    to check (default all)."""
    import torch
    f8 = torch.float8_e4m3fn
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        kif, kisf = ki.view(-1, 128), kis.view(-1)
        cu = [int(x) for x in ps.cu_seqlens_q]
        lo, hi = tokens if tokens is not None else (0, cu[-1])
        for b in range(ps.batch):
            P = int(ps.prefix_lens[b])
            c0, c1 = max(cu[b], lo), min(cu[b + 1], hi)
            if c1 <= c0:
                continue
            ctx = P + (c1 - cu[b])
            rows = _cache_rows(ps, b, torch.arange(ctx, device=qi.device))
            K = kif[rows].view(f8).float()            # [ctx, 128]
            sig = kisf[rows]
            for t0 in range(c0, c1, block):
                t1 = min(t0 + block, c1)
                n = t1 - t0
                pos = P + (t0 - cu[b]) + torch.arange(n, device=qi.device)
                m = int(pos[-1]) + 1
                Q = qi[t0:t1].view(f8).float()         # [n, 64, 128]
                if w_stride == 0:
                    W = w.view(-1)[:64][None, :].expand(n, 64)
                else:
                    W = w.view(-1)[(torch.arange(t0, t1, device=qi.device)[:, None] * w_stride +
                                   torch.arange(64, device=qi.device)[None, :])]
                D = torch.matmul(Q.reshape(n * 64, 128), K[:m].t()).view(n, 64, m)
                sc = (D.clamp_min(0) * W[:, :, None]).sum(dim=1) * sig[None, :m]
                valid = torch.arange(m, device=qi.device)[None, :] <= pos[:, None]
                exp = torch.zeros((n, m), dtype=torch.bool, device=qi.device)
                short = pos + 1 <= topk
                exp[short] = valid[short]
                long_rows = ~short
                if bool(long_rows.any()):
                    s = torch.where(valid, sc, torch.full_like(sc, float("-inf")))[long_rows]
                    kth = torch.topk(s, topk, dim=1).values[:, -1:]
                    v = valid[long_rows]
                    gt, eq = (s > kth) & v, (s == kth) & v
                    need = topk - gt.sum(dim=1, keepdim=True)
                    exp[long_rows] = gt | (eq & (eq.cumsum(dim=1) <= need))
                g = idx[t0:t1].long()
                okg = g >= 0
                assert bool((g >= -1).all()), f"tokens {t0}..{t1}: index below -1"
                cnt = okg.sum(dim=1)
                assert bool((cnt == torch.clamp(pos + 1, max=topk)).all()), f"tokens {t0}..{t1}: wrong counts"
                assert bool((okg[:, :-1] | ~okg[:, 1:]).all()), f"tokens {t0}..{t1}: -1 before a position"
                gs = torch.sort(torch.where(okg, g, torch.full_like(g, 1 << 40)), dim=1).values
                assert bool((gs[:, 1:] != gs[:, :-1])[okg[:, 1:]].all()), f"tokens {t0}..{t1}: repeated position"
                # padding and any out-of-range entry land in a spare last column
                got = torch.zeros((n, m + 1), dtype=torch.bool, device=qi.device)
                got.scatter_(1, torch.where(okg & (g < m), g, torch.full_like(g, m)), torch.ones_like(okg))
                bad = (got[:, :m] != exp).any(dim=1) | (got[:, m] & (okg & (g >= m)).any(dim=1))
                assert not bool(bad.any()), f"token {t0 + int(bad.nonzero()[0])}: selection differs"
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def decode_ds_rows_torch(rows):
    """656-byte rows (uint8 [..., 656], torch) -> fp32 keys [..., 576]: 512 e4m3
    codes times the scale of their 128-dim group, then 64 bf16 RoPE values."""
    import torch
    codes = rows[..., :512].contiguous().view(torch.float8_e4m3fn).float()
    scales = rows[..., 512:528].contiguous().view(torch.float32)
    rope = rows[..., 528:656].contiguous().view(torch.bfloat16).float()
    lat = (codes.unflatten(-1, (4, 128)) * scales[..., None]).flatten(-2)
    return torch.cat([lat, rope], dim=-1)


def sparse_reference_ds_torch(ps, q, kv_ds, sm_scale, idx, block=64):
    """sparse_reference_torch over a cache of 656-byte rows."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        T, H = q.shape[0], q.shape[1]
        out = torch.empty((T, H, 512), dtype=torch.float32, device=q.device)
        lse = torch.empty((T, H), dtype=torch.float32, device=q.device)
        kvf = kv_ds.view(-1, 656)
        cu = [int(x) for x in ps.cu_seqlens_q]
        for b in range(ps.batch):
            for t0 in range(cu[b], cu[b + 1], block):
                t1 = min(t0 + block, cu[b + 1])
                ix = idx[t0:t1].long()
                ok = ix >= 0
                K = decode_ds_rows_torch(kvf[_cache_rows(ps, b, ix.clamp_min(0))])
                lg = torch.einsum("thd,tsd->ths", q[t0:t1].float(), K) * sm_scale
                lg = lg.masked_fill(~ok[:, None, :], float("-inf"))
                l = torch.logsumexp(lg, dim=-1)
                p = torch.exp(lg - torch.where(torch.isfinite(l), l, torch.zeros_like(l))[..., None])
                out[t0:t1] = torch.einsum("ths,tsd->thd", p, K[..., :512])
                lse[t0:t1] = l
        return out, lse
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


# ---------------------------------------------------------------------------
# the non-absorbed (MHA) path
# ---------------------------------------------------------------------------
def mha_reference_torch(ps, q, w, kv, ks, sm_scale, toks=None, q_block=256):
    """The non-absorbed path in plain PyTorch, fp32 (TF32 off), on the GPU, for
    every new token (or the global tokens `toks`): c_s = ks_s * dec(kv_s),
    k = [W_UK c ; r], v = W_UV c per head, causal softmax. Also returns the
    per-row bound on the move of the log-sum-exp when the kernel rounds each
    key to f16: u * sm_scale * max_s sum_d |q_d| |k_s[d]| (u = 2^-11).
    q: bf16 [Tq, H, 192]; w: bf16 [H, 256, 512]. Returns (out [n, H, 128], lse
    [n, H], lse_bound [n, H]) in token order."""
    import torch
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        H = q.shape[1]
        wf = w.float()
        kvf, ksf = kv.view(-1, 576), ks.view(-1)
        cu = [int(x) for x in ps.cu_seqlens_q]
        want = torch.arange(cu[-1], device=q.device) if toks is None else torch.as_tensor(toks, device=q.device)
        out = torch.zeros((want.numel(), H, 128), dtype=torch.float32, device=q.device)
        lse = torch.zeros((want.numel(), H), dtype=torch.float32, device=q.device)
        bnd = torch.zeros((want.numel(), H), dtype=torch.float64, device=q.device)
        for b in range(ps.batch):
            sel = ((want >= cu[b]) & (want < cu[b + 1])).nonzero().flatten()
            if sel.numel() == 0:
                continue
            P = int(ps.prefix_lens[b])
            tq = want[sel]
            ctx = P + int(tq.max()) - cu[b] + 1
            rows = _cache_rows(ps, b, torch.arange(ctx, device=q.device))
            C = kvf[rows].view(torch.float8_e4m3fn).float() * ksf[rows][:, None]          # [ctx, 576]
            Kn = torch.einsum("sd,hid->hsi", C[:, :512], wf[:, :128, :])                  # [H, ctx, 128]
            V = torch.einsum("sd,hid->hsi", C[:, :512], wf[:, 128:, :])
            K = torch.cat([Kn, C[None, :, 512:].expand(H, ctx, 64)], dim=2)              # [H, ctx, 192]
            for j0 in range(0, sel.numel(), q_block):
                js = sel[j0:j0 + q_block]
                t = want[js]
                pos = P + (t - cu[b])
                qb = q[t].float().permute(1, 0, 2)                                      # [H, n, 192]
                lg = torch.einsum("hnd,hsd->hns", qb, K) * sm_scale
                mask = torch.arange(ctx, device=q.device)[None, :] > pos[:, None]       # [n, ctx]
                lg = lg.masked_fill(mask[None], float("-inf"))
                l = torch.logsumexp(lg, dim=-1)                                         # [H, n]
                p = torch.exp(lg - l[..., None])
                out[js] = torch.einsum("hns,hsi->nhi", p, V)
                lse[js] = l.t()
                mag = torch.einsum("hnd,hsd->hns", qb.abs().double(), K.abs().double())
                mag = mag.masked_fill(mask[None], 0.0)
                bnd[js] = (F16_UNIT_ROUNDOFF * sm_scale * mag.amax(dim=-1)).t()
        return out, lse, bnd
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
