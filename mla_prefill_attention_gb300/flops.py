"""Algorithmic work and traffic of the hot path (host arithmetic for the bench).

Per (query, key, head) pair the absorbed MLA does a 576-dim dot product for
QK and a 512-dim multiply-add for PV: 2*576 + 2*512 = 2,176 FLOPs, the figure
of "GLM-5.3-Optimierungen, Teil 2", footnote 1 ("QK over 576 dims, PV over
512"). Masked-out pairs are not counted. The indexer costs 2*128 FLOPs per
(query, key, indexer head) pair (64 heads x 128 dims).
"""
from __future__ import annotations

D_QK, D_V, D_IDX, H_IDX = 576, 512, 128, 64

FLOPS_PER_PAIR_HEAD = 2 * D_QK + 2 * D_V          # 2,176


def causal_pairs(q_len: int, prefix: int) -> int:
    """Visible (query, key) pairs of one sequence: sum over i < q_len of prefix + i + 1."""
    return q_len * prefix + q_len * (q_len + 1) // 2


def dense_pairs(q_lens, prefix_lens) -> int:
    return sum(causal_pairs(int(t), int(p)) for t, p in zip(q_lens, prefix_lens))


def dense_flops(q_lens, prefix_lens, heads: int) -> int:
    return dense_pairs(q_lens, prefix_lens) * heads * FLOPS_PER_PAIR_HEAD


def sparse_pairs(q_lens, prefix_lens, topk: int) -> int:
    """(query, selected key) pairs: min(topk, position + 1) keys per query."""
    n = 0
    for t, p in zip(q_lens, prefix_lens):
        t, p = int(t), int(p)
        # positions p .. p+t-1 see p+1 .. p+t keys; capped at topk
        lo, hi = p + 1, p + t                     # key counts of first / last query
        if hi <= topk:
            n += (lo + hi) * t // 2
        elif lo >= topk:
            n += t * topk
        else:
            k_small = topk - lo                   # queries with count < topk: counts lo..topk-1
            n += (lo + topk - 1) * k_small // 2 + (t - k_small) * topk
    return n


def sparse_flops(q_lens, prefix_lens, heads: int, topk: int) -> int:
    return sparse_pairs(q_lens, prefix_lens, topk) * heads * FLOPS_PER_PAIR_HEAD


def indexer_flops(q_lens, prefix_lens) -> int:
    return dense_pairs(q_lens, prefix_lens) * H_IDX * D_IDX * 2


def sparse_bytes_per_query(topk: int, heads: int, row_bytes: int, index_bytes: int = 4) -> int:
    """Bytes one query moves in sparse MLA: topk gathered rows (plus their
    index) and, per head, its bf16 query (576) and output (512) rows."""
    return topk * (row_bytes + index_bytes) + heads * 2 * (D_QK + D_V)


def dense_min_bytes(total_q: int, heads: int, cache_tokens: int) -> int:
    """Compulsory HBM bytes of one dense call: bf16 Q and O, the e4m3 cache
    rows with their fp32 scales, fp32 LSE."""
    return total_q * heads * (2 * D_QK + 2 * D_V + 4) + cache_tokens * (D_QK + 4)


def sparse_gathered_bytes(q_lens, prefix_lens, topk: int, heads: int = 64, row_bytes: int = D_QK + 4) -> int:
    """Bytes sparse MLA moves when every selected row is read from HBM (no
    reuse across queries): per (query, selected key) pair the 580-byte row and
    its 4-byte index, and per query its bf16 query and output rows (the
    arithmetic intensity of "GLM-5.3-Optimierungen, Teil 2", footnote 1, in
    this library's 580-byte row format: ~214 FLOP/B at 64 heads)."""
    tq = sum(int(t) for t in q_lens)
    return sparse_pairs(q_lens, prefix_lens, topk) * (row_bytes + 4) + tq * heads * 2 * (D_QK + D_V)
