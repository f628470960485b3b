"""Shared helpers of the GPU parity tests: problem construction from the
seeded generators, upload, sampling of rows, and the tolerance check."""
from __future__ import annotations

import math

import numpy as np

from mla_prefill_attention_gb300 import inputs as I

# attention tolerance, relative to the rms of the oracle output over the checked rows
TOL_MAX = 2e-2
TOL_MEAN = 2e-3
TOL_LSE_ABS = 1e-3


def rel_errors(gpu: np.ndarray, ora: np.ndarray, beyond_rounding: bool = False):
    """Errors relative to the RMS of each output row (one (token, head) vector
    of 512 values): returns (max, mean) of |gpu - ora| / rms_row, and the global
    rms. Rows whose oracle output is exactly zero are compared absolutely.

    Reading of "relative to the output RMS": per output row. Against a single
    RMS over the whole output the max bound cannot be met by any bf16 result
    once a row's entries exceed ~5x the global RMS (rounding a value to bf16
    moves it by up to 2^-8 of itself); early causal rows, which average only a
    few cache rows, reach 12x on the tiny workload.

    beyond_rounding: the error of each element is first reduced by the most
    that rounding to bf16 can move it (half the bf16 spacing at the oracle's or
    the GPU's value, whichever is larger), so an exact result delivered in bf16
    scores zero and what remains is the computation's own error."""
    o = ora.astype(np.float64).reshape(-1, ora.shape[-1])
    g = gpu.astype(np.float64).reshape(-1, ora.shape[-1])
    rms_row = np.sqrt(np.mean(o ** 2, axis=1, keepdims=True))
    rms_row[rms_row == 0] = 1.0
    d = np.abs(g - o)
    if beyond_rounding:
        d = np.maximum(d - np.maximum(bf16_half_spacing(o), bf16_half_spacing(g)), 0.0)
    r = d / rms_row
    return float(r.max()), float(r.mean()), math.sqrt(float(np.mean(o ** 2)))


def bf16_half_spacing(x):
    """Half the distance between neighbouring bf16 values at |x| (8 significant
    bits: 2^(e-8) for |x| in [2^e, 2^(e+1))), the most rounding x to bf16 can
    move it; 0 at 0."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(e - 8), 0.0)


def check_attention(gpu_out, ora_out, gpu_lse=None, ora_lse=None, what=""):
    """Output within the bounds beyond the bf16 rounding of the output (see
    rel_errors); the raw errors, rounding included, are in the message."""
    mx, mean, rms = rel_errors(gpu_out, ora_out, beyond_rounding=True)
    raw_mx, raw_mean, _ = rel_errors(gpu_out, ora_out)
    assert np.all(np.isfinite(gpu_out)), f"{what}: non-finite output"
    assert mx <= TOL_MAX and mean <= TOL_MEAN, (f"{what}: beyond bf16 rounding max {mx:.3e} mean {mean:.3e}; "
                                                f"raw max {raw_mx:.3e} mean {raw_mean:.3e} (rms {rms:.3e})")
    if gpu_lse is not None:
        dl = float(np.max(np.abs(gpu_lse.astype(np.float64) - ora_lse)))
        assert dl <= TOL_LSE_ABS, f"{what}: lse max abs err {dl:.3e}"
    return mx, mean


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


def sample_tokens(total: int, n_uniform: int, seed: int, edge: int = 8, boundaries=()):
    """First/last `edge` tokens, tokens at +-1 of each boundary, n_uniform random."""
    rng = np.random.default_rng(seed)
    s = set(range(min(edge, total))) | set(range(max(0, total - edge), total))
    for b in boundaries:
        for d in (-1, 0, 1):
            if 0 <= b + d < total:
                s.add(b + d)
    s |= set(rng.integers(0, total, n_uniform).tolist()) if total > 0 else set()
    return np.array(sorted(s), dtype=np.int64)
