"""Seeded synthetic inputs for MLA prefill attention.

This module is the one place both sides of every check draw their inputs
from: the CUDA path (tests, bench) and the CPU oracle (tests, cpu baseline).
It holds no attention arithmetic. It only makes numbers and packs them into
the storage formats the library consumes:

* a counter-based random stream (SplitMix64, Steele/Lea/Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014): draw ``j`` of the
  stream keyed ``(seed, tensor, row)`` is the ``j``-th output of a SplitMix64
  generator whose state starts at that key, so any row of any tensor can be
  regenerated on its own;
* Box-Muller normals from pairs of those uniforms;
* an IEEE round-to-nearest-even bf16 encoder and an OCP e4m3fn
  (bias 7, max 448, no infinities) round-to-nearest-even saturating encoder;
* the per-token absmax/448 quantisation of a latent row (the KV storage format:
  576 e4m3 codes plus one fp32 scale per token, 256-token pages);
* the workload recipes (shapes, distributions, page shuffles) of the five
  workloads the library is measured on.

Readings of the source pages that this module fixes:

* The FP8 KV cache of the pages ("FP8 (weights and KV cache)", More throughput
  from fewer GPUs, section System architecture) is stored as e4m3 codes with a
  per-token fp32 scale equal to absmax/448 over the 576 latent+RoPE dims; an
  all-zero row gets scale 1.
* The 256-token KV granularity (same page, section KV hand-off and caching) is
  the page size of the paged cache.
* Indexer keys are 128 FP8 values plus a 4-byte scale per token (GLM-5.3
  Optimierungen Teil 2, footnote 3); the generator draws small integers so
  that every indexer score is exact in fp32, and sets the key scale to 1.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

PAGE = 256          # tokens per KV page
D_QK = 576          # latent (512) + RoPE (64) dims per query/key row
D_V = 512           # latent dims read as the value
D_IDX = 128         # indexer head dim
H_IDX = 64          # indexer heads

# tensor ids of the counter-based streams
T_Q, T_KV, T_QIDX, T_KIDX, T_WIDX, T_PERM, T_MISC, T_NEWKV, T_NEWKIDX, T_GAIN = 1, 2, 3, 4, 5, 6, 7, 8, 9, 10
T_QMHA, T_WUKV = 11, 12
D_HEAD_QK = 192     # non-absorbed form: 128 no-RoPE + 64 RoPE dims per head
D_HEAD_V = 128

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "inputs_gen.c")
_SO = os.path.join(_HERE, "libmla_inputs.so")
_lib = None


def build_generator(force: bool = False) -> str:
    """Compile the bulk generator (plain C, OpenMP) next to this file."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _gen():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_generator())
        u64, i64, i32, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        lib.gen_stream_key.restype = u64
        lib.gen_stream_key.argtypes = [u64, u64, u64]
        for name in ("gen_uniform", "gen_normal_f64", "gen_normal_bf16"):
            getattr(lib, name).argtypes = [u64, u64, vp, i64, i64, vp]
        lib.gen_latent_e4m3.argtypes = [u64, u64, vp, i64, i64, vp, vp]
        lib.gen_int_e4m3.argtypes = [u64, u64, vp, i64, i64, i32, i32, vp]
        lib.gen_encode_bf16.argtypes = [vp, i64, vp]
        lib.gen_encode_e4m3.argtypes = [vp, i64, vp]
        _lib = lib
    return _lib


def _rows(rows) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int64).astype(np.uint64).reshape(-1))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def uniform_rows(seed: int, tensor: int, rows, n: int) -> np.ndarray:
    """float64 uniforms in [0,1), shape (len(rows), n): draw j of each row stream."""
    r = _rows(rows)
    out = np.empty((r.shape[0], n), dtype=np.float64)
    _gen().gen_uniform(seed, tensor, _p(r), r.shape[0], n, _p(out))
    return out


def normal_rows(seed: int, tensor: int, rows, n: int) -> np.ndarray:
    """float64 N(0,1) draws, shape (len(rows), n), by Box-Muller on draw pairs."""
    r = _rows(rows)
    out = np.empty((r.shape[0], n), dtype=np.float64)
    _gen().gen_normal_f64(seed, tensor, _p(r), r.shape[0], n, _p(out))
    return out


def int_rows(seed: int, tensor: int, rows, n: int, lo: int, hi: int) -> np.ndarray:
    """int64 draws uniform on {lo..hi}, shape (len(rows), n)."""
    u = uniform_rows(seed, tensor, rows, n)
    return lo + np.floor(u * (hi - lo + 1)).astype(np.int64)


# ----------------------------------------------------------------------------
# storage encoders (round to nearest, ties to even)
# ----------------------------------------------------------------------------

def bf16_bits(x) -> np.ndarray:
    """Round float64 values to bfloat16 (RNE, single rounding); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _gen().gen_encode_bf16(_p(x), x.size, _p(out))
    return out


def e4m3_bits(y) -> np.ndarray:
    """Encode float64 values as OCP e4m3fn codes, RNE, saturating at +-448."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    out = np.empty(y.shape, dtype=np.uint8)
    _gen().gen_encode_e4m3(_p(y), y.size, _p(out))
    return out


def quantize_latent_rows(x: np.ndarray):
    """Per-token absmax/448 e4m3 quantisation of rows [n, d] -> (codes u8, scale f32)."""
    x = np.asarray(x, dtype=np.float64)
    amax = np.max(np.abs(x), axis=1)
    scale = np.where(amax > 0, amax / 448.0, 1.0).astype(np.float32)
    codes = e4m3_bits(x / scale.astype(np.float64)[:, None])
    return codes, scale


# ----------------------------------------------------------------------------
# workload containers
# ----------------------------------------------------------------------------

@dataclass
class PagedSeqs:
    """Ragged batch of sequences over a paged cache (host arrays)."""
    cu_seqlens_q: np.ndarray      # int32 [B+1]: new query tokens per sequence
    prefix_lens: np.ndarray       # int32 [B]: cached tokens before the new ones
    block_table: np.ndarray       # int32 [B, max_blocks]: page id per 256-token block
    num_blocks: int

    @property
    def batch(self) -> int:
        return int(self.prefix_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.cu_seqlens_q[-1])

    def seq_len(self, b: int) -> int:
        """Tokens visible at the end of sequence b (prefix + new)."""
        return int(self.prefix_lens[b] + self.cu_seqlens_q[b + 1] - self.cu_seqlens_q[b])


def make_seqs(q_lens, prefix_lens, seed: int, shuffle: bool, extra_blocks: int = 0) -> PagedSeqs:
    """Lay out B sequences over 256-token pages; shuffle=True draws a random
    permutation of the physical pages (tensor T_PERM), else pages are in order."""
    q_lens = [int(x) for x in q_lens]
    prefix_lens = [int(x) for x in prefix_lens]
    B = len(q_lens)
    nblk = [-(-(p + t) // PAGE) for p, t in zip(prefix_lens, q_lens)]
    total = sum(nblk) + extra_blocks
    if shuffle:
        perm = np.argsort(uniform_rows(seed, T_PERM, [0], total)[0], kind="stable").astype(np.int32)
    else:
        perm = np.arange(total, dtype=np.int32)
    maxb = max(1, max(nblk))
    bt = np.full((B, maxb), -1, dtype=np.int32)
    o = 0
    for b in range(B):
        bt[b, : nblk[b]] = perm[o: o + nblk[b]]
        o += nblk[b]
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    return PagedSeqs(cu, np.asarray(prefix_lens, dtype=np.int32), bt, total)


def gen_q_bf16(seed: int, total_q: int, heads: int, token_rows=None, dim: int = D_QK, tensor: int = T_Q) -> np.ndarray:
    """bf16 bits [n, heads, dim] of N(0,1) queries; row stream = token*heads + head.
    token_rows selects global query tokens (default: all total_q)."""
    toks = np.arange(total_q, dtype=np.int64) if token_rows is None else np.asarray(token_rows, np.int64)
    rows = _rows((toks[:, None] * heads + np.arange(heads, dtype=np.int64)[None, :]).reshape(-1))
    out = np.empty((toks.shape[0], heads, dim), dtype=np.uint16)
    _gen().gen_normal_bf16(seed, tensor, _p(rows), rows.shape[0], dim, _p(out))
    return out


def gen_q_mha(seed: int, total_q: int, heads: int, token_rows=None) -> np.ndarray:
    """bf16 bits [n, heads, 192] of N(0,1) per-head queries of the non-absorbed
    form (128 no-RoPE dims, then 64 RoPE dims)."""
    return gen_q_bf16(seed, total_q, heads, token_rows, dim=D_HEAD_QK, tensor=T_QMHA)


def gen_w_ukv(seed: int, heads: int) -> np.ndarray:
    """bf16 bits [heads, 256, 512] of the key/value up-projection (random-init:
    no trained weights): N(0,1) * 2^-4 rounded to bf16, so a no-RoPE key or a
    value dim of an N(0,1) latent row has a standard deviation near sqrt(512)/16.
    Rows 0..127 of head h are W_UK_h, rows 128..255 W_UV_h; row stream h*256 + i."""
    rows = np.arange(heads * 256, dtype=np.int64)
    x = normal_rows(seed, T_WUKV, rows, D_V) * 2.0 ** -4
    return bf16_bits(x).reshape(heads, 256, D_V)


def latent_rows(seed: int, b: int, positions, tensor: int = T_KV):
    """(codes u8 [n, 576], scale f32 [n]) of tokens at `positions` of sequence b."""
    s = np.asarray(positions, dtype=np.int64)
    rows = _rows((np.int64(b) << 32) | s)
    codes = np.empty((rows.shape[0], D_QK), dtype=np.uint8)
    scales = np.empty(rows.shape[0], dtype=np.float32)
    _gen().gen_latent_e4m3(seed, tensor, _p(rows), rows.shape[0], D_QK, _p(codes), _p(scales))
    return codes, scales


def gen_latent_cache(seed: int, seqs: PagedSeqs, tensor: int = T_KV):
    """Paged e4m3 latent cache [num_blocks, 256, 576] + fp32 scales [num_blocks, 256].
    Token s of sequence b draws from row stream (b << 32) | s; unused slots stay 0
    with scale 1."""
    nb = seqs.num_blocks
    codes = np.zeros((nb, PAGE, D_QK), dtype=np.uint8)
    scales = np.ones((nb, PAGE), dtype=np.float32)
    for b in range(seqs.batch):
        s = np.arange(seqs.seq_len(b), dtype=np.int64)
        c, sc = latent_rows(seed, b, s, tensor)
        pg = seqs.block_table[b, s // PAGE]
        codes[pg, s % PAGE] = c
        scales[pg, s % PAGE] = sc
    return codes, scales


# ----------------------------------------------------------------------------
# the 656-byte row format
# ----------------------------------------------------------------------------
# Reading of "GLM-5.3-Optimierungen, Teil 2", footnote 1 ("656 FP8-KV im
# fp8_ds_mla-Format"): 656 bytes per token hold the 512 latent dims as e4m3 codes
# with one fp32 scale per 128 dims (absmax/448, 1 for an all-zero group) and the
# 64 RoPE dims as bf16: bytes 0..511 codes, 512..527 the four scales
# (little-endian), 528..655 the RoPE values (little-endian).
DS_ROW = 656
DS_GROUPS = 4


def pack_ds_rows(x: np.ndarray) -> np.ndarray:
    """Latent rows [n, 576] (float64) -> 656-byte rows [n, 656] (uint8)."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[0]
    lat = x[:, :D_V].reshape(n, DS_GROUPS, D_V // DS_GROUPS)
    amax = np.max(np.abs(lat), axis=2)
    scale = np.where(amax > 0, amax / 448.0, 1.0).astype(np.float32)
    codes = e4m3_bits(lat / scale.astype(np.float64)[:, :, None]).reshape(n, D_V)
    rope = bf16_bits(x[:, D_V:])
    out = np.empty((n, DS_ROW), dtype=np.uint8)
    out[:, :D_V] = codes
    out[:, D_V:D_V + 16] = np.ascontiguousarray(scale.astype("<f4")).view(np.uint8).reshape(n, 16)
    out[:, D_V + 16:] = np.ascontiguousarray(rope.astype("<u2")).view(np.uint8).reshape(n, 128)
    return out


def ds_rows(seed: int, b: int, positions, tensor: int = T_KV) -> np.ndarray:
    """656-byte rows of tokens at `positions` of sequence b (the same N(0,1) draws
    as latent_rows)."""
    s = np.asarray(positions, dtype=np.int64)
    return pack_ds_rows(normal_rows(seed, tensor, (np.int64(b) << 32) | s, D_QK))


def gen_latent_cache_ds(seed: int, seqs: PagedSeqs, tensor: int = T_KV) -> np.ndarray:
    """Paged cache of 656-byte rows [num_blocks, 256, 656]; unused slots hold zero
    codes, scales 1 and zero RoPE values."""
    nb = seqs.num_blocks
    empty = pack_ds_rows(np.zeros((1, D_QK)))[0]
    cache = np.tile(empty, (nb, PAGE, 1))
    for b in range(seqs.batch):
        s = np.arange(seqs.seq_len(b), dtype=np.int64)
        pg = seqs.block_table[b, s // PAGE]
        for c0 in range(0, s.shape[0], 65536):
            sl = s[c0:c0 + 65536]
            cache[pg[c0:c0 + 65536], sl % PAGE] = ds_rows(seed, b, sl, tensor)
    return cache


def _int_e4m3(seed, tensor, rows, n, lo, hi):
    r = _rows(rows)
    out = np.empty((r.shape[0], n), dtype=np.uint8)
    _gen().gen_int_e4m3(seed, tensor, _p(r), r.shape[0], n, lo, hi, _p(out))
    return out


def gen_indexer_q(seed: int, total_q: int, token_rows=None) -> np.ndarray:
    """Indexer queries, e4m3 codes [n, 64, 128] of integers uniform in [-4, 4]."""
    toks = np.arange(total_q, dtype=np.int64) if token_rows is None else np.asarray(token_rows, np.int64)
    rows = (toks[:, None] * H_IDX + np.arange(H_IDX, dtype=np.int64)[None, :]).reshape(-1)
    return _int_e4m3(seed, T_QIDX, rows, D_IDX, -4, 4).reshape(toks.shape[0], H_IDX, D_IDX)


def gen_indexer_w(seed: int) -> np.ndarray:
    """Per-head indexer weights w_h = 2^-j, j uniform in {0..4}, f32 [64]."""
    j = int_rows(seed, T_WIDX, [0], H_IDX, 0, 4)[0]
    return np.ldexp(1.0, -j).astype(np.float32)


def gen_indexer_keys(seed: int, seqs: PagedSeqs):
    """Paged indexer keys: e4m3 codes [nb, 256, 128] of integers in [-4, 4], scale 1."""
    nb = seqs.num_blocks
    k = np.zeros((nb, PAGE, D_IDX), dtype=np.uint8)
    ks = np.ones((nb, PAGE), dtype=np.float32)
    for b in range(seqs.batch):
        s = np.arange(seqs.seq_len(b), dtype=np.int64)
        pg = seqs.block_table[b, s // PAGE]
        k[pg, s % PAGE] = _int_e4m3(seed, T_KIDX, (np.int64(b) << 32) | s, D_IDX, -4, 4)
    return k, ks


def gen_indexer_inputs(seed: int, seqs: PagedSeqs, token_rows=None):
    """(q_idx u8 [n,64,128], w f32 [64] (token stride 0), k_idx u8 [nb,256,128], k_scale f32 [nb,256])."""
    q = gen_indexer_q(seed, seqs.total_q, token_rows)
    k, ks = gen_indexer_keys(seed, seqs)
    return q, gen_indexer_w(seed), k, ks


def gen_new_rows_bf16(seed: int, total_q: int, dim: int, tensor: int = T_NEWKV) -> np.ndarray:
    """bf16 bits [total_q, dim] of the new tokens' unquantised cache rows (the
    latent row with dim 576 under T_NEWKV, the indexer key with dim 128 under
    T_NEWKIDX): N(0,1) draws times a per-token gain 2^g, g uniform in [-4, 4),
    so that the per-token scales spread over eight octaves. Row stream = token."""
    toks = np.arange(total_q, dtype=np.int64)
    gain = np.exp2(uniform_rows(seed, T_GAIN * 16 + tensor, toks, 1)[:, 0] * 8.0 - 4.0)
    return bf16_bits(normal_rows(seed, tensor, toks, dim) * gain[:, None])


# ----------------------------------------------------------------------------
# the measured workloads
# ----------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    seed: int
    heads: int
    q_lens: list
    prefix_lens: list
    shuffle: bool
    sparse: bool = False
    topk: int = 2048
    chunk: int = 0            # >0: chunked prefill of a single prompt in chunks of this many tokens
    sm_scale: float = 1.0 / math.sqrt(192.0)
    notes: str = ""
    meta: dict = field(default_factory=dict)

    def seqs(self, extra_blocks: int = 0) -> PagedSeqs:
        return make_seqs(self.q_lens, self.prefix_lens, self.seed, self.shuffle, extra_blocks)


K1 = 1024
WORKLOADS = {
    # tiny dense prefill, identity block table
    "tiny512": Workload("tiny512", 0, 16, [512], [0], False,
                        notes="1 sequence of 512 new tokens, no prefix, 16 heads, identity pages"),
    # prefix-cache hit: 12,288 cached tokens in shuffled pages + 4,096 new tokens
    "prefix12k": Workload("prefix12k", 1, 64, [4096], [12288], True,
                          notes="64 heads, 12,288-token cached prefix in shuffled pages, 4,096 new tokens"),
    # dense causal prefill at 32k (the headline workload)
    "dense32k": Workload("dense32k", 2, 64, [32768], [0], True,
                         notes="64 heads, 32,768 new tokens, batch 1, 16-chunk pairing"),
    # ragged batch 9k/16k/24k/32k (k = 1024)
    "ragged4": Workload("ragged4", 2, 64, [9 * K1, 16 * K1, 24 * K1, 32 * K1], [0, 0, 0, 0], True,
                        notes="4 ragged prompts of 9,216/16,384/24,576/32,768 tokens"),
    # sparse top-2048 at 64k context: 8,192 new tokens after a 57,344-token prefix
    "sparse64k": Workload("sparse64k", 3, 64, [8192], [57344], True, sparse=True,
                          notes="indexer 64x128 + top-2048 + sparse MLA, 8,192 queries at the end of 65,536"),
    # a batch of short prompts (each within the top-k of 2,048), the non-absorbed (MHA) path's workload
    "mha_short": Workload("mha_short", 5, 64, [2048, 1536, 1024, 1024, 768, 512, 300, 77], [0] * 8, True,
                          notes="8 prompts of 77-2,048 tokens (7,289 in all), 64 heads, non-absorbed MHA path"),
    # chunked prefill of a 200,000-token prompt in 6,144-token chunks
    "chunked200k": Workload("chunked200k", 4, 64, [200000], [0], True, sparse=True, chunk=6144,
                            notes="200,000-token prompt in 6,144-token chunks (32 full + 3,392)"),
}
