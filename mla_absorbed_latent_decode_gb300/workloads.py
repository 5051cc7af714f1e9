"""Seeded synthetic inputs for absorbed-MLA decode (shared by tests, smoke and bench).

This module only draws and lays out inputs: weights, queries, cache rows,
context lengths, paged block tables and the FP8 tensor scale.  It holds none of
the method's arithmetic (no RoPE, no projection, no attention); both the CUDA
path and the CPU oracle consume what it returns.

Values are drawn with ``numpy.random.default_rng(seed)`` (PCG64) as float64,
cast to float32 and rounded to bfloat16 (nearest even).  bf16 tensors are
returned as their uint16 bit patterns.

The five named workloads follow the decode configurations the pages motivate:
a DeepSeek-V2-Lite layer ("DeepSeek-V2-Lite 真实权重执行审计" §1.2: 16 heads,
qk no-RoPE/RoPE 128/64, value 128, KV LoRA rank 512, hidden 2048) and
DeepSeek-V3 shapes ("G5 MLA KV 访存建模设计规格" 用例说明: kv_lora_rank 512,
qk_rope 64, 128 heads, history 4096, FP8 cache).  No public dataset is
involved; real weights are not available, so weights are N(0, 0.02^2).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

PAGE_SIZE = 64
D_C = 512
D_ROPE = 64
D_NOPE = 128
D_V = 128
ROPE_BASE = 10000.0
WEIGHT_STD = 0.02
CACHE_BF16 = 1
CACHE_FP8 = 2
CACHE_FP8_BLOCK = 3          # 656-byte rows: 512 e4m3 latent codes, 4 fp32 block scales, 64 bf16 RoPE values
ROW_BYTES = {1: 1152, 2: 576, 3: 656}


def to_bf16_bits(x) -> np.ndarray:
    """float64/float32 -> float32 -> bfloat16 bit patterns, round to nearest even."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class Workload:
    """One decode problem.  Arrays are host numpy arrays.

    rows      [sum(ctx_len), d_c + d_rope] bf16 bits: cache rows in (sequence, position) order,
              latent first, then the unrotated RoPE key.
    row_seq   [N] int32 sequence of each row; row_pos [N] int32 absolute position of each row.
    q         [B, n_h, d_nope + d_rope] bf16 bits (no-RoPE part first).
    w_uk      [n_h, d_nope, d_c] bf16 bits; w_uv [n_h, d_v, d_c] bf16 bits.
    ctx_len   [B] int32; block_table [B, max_pages] int32 (-1 past the sequence's pages).
    """
    name: str
    n_h: int
    B: int
    ctx_len: np.ndarray
    block_table: np.ndarray
    num_pages: int
    w_uk: np.ndarray
    w_uv: np.ndarray
    q: np.ndarray
    rows: np.ndarray
    row_seq: np.ndarray
    row_pos: np.ndarray
    cache_dtype: int = CACHE_BF16
    fp8_scale: float = 0.0
    seed: int = 0
    d_c: int = D_C
    d_rope: int = D_ROPE
    d_nope: int = D_NOPE
    d_v: int = D_V
    page_size: int = PAGE_SIZE
    rope_base: float = ROPE_BASE
    extra: dict = field(default_factory=dict)

    @property
    def total_tokens(self) -> int:
        return int(np.sum(self.ctx_len.astype(np.int64)))

    @property
    def max_ctx(self) -> int:
        return int(np.max(self.ctx_len)) if self.B else 0

    def last_row_index(self) -> np.ndarray:
        """Index into ``rows`` of each sequence's last row (the decode token's own row)."""
        return np.cumsum(self.ctx_len.astype(np.int64)) - 1


def _normal_bf16(rng, shape, std=1.0, chunk=1 << 24):
    """Draw N(0, std^2) in float64 in one stream order, return bf16 bits (chunked to bound memory)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        out[a:b] = to_bf16_bits(rng.standard_normal(b - a) * std)
    return out.reshape(shape)


def _paged_layout(rng, ctx_len, page_size, spare_pages, shuffle=True):
    """Block table over a pool whose pages are handed out in a seeded shuffled order."""
    n_pages = [(int(s) + page_size - 1) // page_size for s in ctx_len]
    total = int(sum(n_pages)) + int(spare_pages)
    order = rng.permutation(total).astype(np.int32)     # drawn either way: the stream stays aligned
    if not shuffle:
        order = np.arange(total, dtype=np.int32)
    max_pages = max(1, max(n_pages) if n_pages else 1)
    bt = np.full((len(ctx_len), max_pages), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(n_pages):
        bt[b, :n] = order[off:off + n]
        off += n
    return bt, total


def _rows_index(ctx_len):
    seq = np.repeat(np.arange(len(ctx_len), dtype=np.int32), ctx_len)
    starts = np.cumsum(np.concatenate([[0], ctx_len[:-1]])).astype(np.int64)
    pos = (np.arange(int(np.sum(ctx_len)), dtype=np.int64) - np.repeat(starts, ctx_len)).astype(np.int32)
    return seq, pos


def fp8_tensor_scale(rows_bits, d_c) -> float:
    """One fp32 tensor scale ``amax / 448`` for an FP8 (e4m3) cache.

    ``amax`` must bound every value the cache will store.  The latent columns
    are stored as given; a RoPE key pair (a, b) is stored rotated, and no
    rotation makes either coordinate exceed ``sqrt(a^2 + b^2)``.  So amax is the
    larger of ``max |latent|`` and the largest pair norm of the RoPE key.
    """
    r = bf16_bits_to_f32(rows_bits).astype(np.float64)
    lat = float(np.max(np.abs(r[:, :d_c]))) if r.size else 0.0
    kr = r[:, d_c:]
    pair = float(np.sqrt(np.max(kr[:, 0::2] ** 2 + kr[:, 1::2] ** 2))) if r.size else 0.0
    amax = max(lat, pair, 1e-30)
    return float(np.float32(amax / 448.0))


def make_decode(name, seed, n_h, ctx_len, *, cache_dtype=CACHE_BF16, shuffle=True,
                spare_pages=8, row_std=1.0, q_std=1.0) -> Workload:
    """Batched decode workload in the fixed draw order: context lengths (by the
    caller), page permutation, W_UK, W_UV, cache rows, queries."""
    rng = np.random.default_rng(seed)
    return _finish_decode(rng, name, seed, n_h, np.asarray(ctx_len, np.int32), cache_dtype,
                          shuffle, spare_pages, row_std, q_std)


def _finish_decode(rng, name, seed, n_h, ctx_len, cache_dtype, shuffle, spare_pages, row_std, q_std):
    bt, num_pages = _paged_layout(rng, ctx_len, PAGE_SIZE, spare_pages, shuffle)
    w_uk = _normal_bf16(rng, (n_h, D_NOPE, D_C), WEIGHT_STD)
    w_uv = _normal_bf16(rng, (n_h, D_V, D_C), WEIGHT_STD)
    total = int(np.sum(ctx_len.astype(np.int64)))
    rows = _normal_bf16(rng, (total, D_C + D_ROPE), row_std)
    q = _normal_bf16(rng, (len(ctx_len), n_h, D_NOPE + D_ROPE), q_std)
    seq, pos = _rows_index(ctx_len)
    wl = Workload(name=name, n_h=n_h, B=len(ctx_len), ctx_len=ctx_len, block_table=bt,
                  num_pages=num_pages, w_uk=w_uk, w_uv=w_uv, q=q, rows=rows,
                  row_seq=seq, row_pos=pos, cache_dtype=cache_dtype, seed=seed)
    if cache_dtype == CACHE_FP8:
        wl.fp8_scale = fp8_tensor_scale(rows, D_C)
    return wl


# ---------------------------------------------------------------------------
# the five named workloads
# ---------------------------------------------------------------------------

def make_prefill(name, seed, n_h, ctx_len, q_len=None, *, q_std=1.0, cache_dtype=CACHE_BF16) -> Workload:
    """Prefill inputs: a decode workload's cache rows, weights and paged layout (same draws as
    ``make_decode``), plus query rows for the last ``q_len[b]`` positions of every sequence
    (every position when ``q_len`` is None), packed [total_q][n_h][d_nope + d_rope] in
    sequence order and drawn from a second stream of the same seed."""
    wl = make_decode(name, seed, n_h, ctx_len, cache_dtype=cache_dtype)
    ql = wl.ctx_len.copy() if q_len is None else np.asarray(q_len, np.int32)
    rng = np.random.default_rng([seed, 1])
    q = _normal_bf16(rng, (int(np.sum(ql.astype(np.int64))), n_h, D_NOPE + D_ROPE), q_std)
    starts = np.concatenate([[0], np.cumsum(ql.astype(np.int64))[:-1]]).astype(np.int32)
    wl.extra["prefill"] = {"q": q, "q_len": ql, "q_start": starts}
    return wl


def v3_prefill(seed=5, B=2, s_ctx=4096, n_h=128) -> Workload:
    """DeepSeek-V3 shapes, B=2 whole prompts of 4096 tokens (query length = context length)."""
    wl = make_prefill("v3_prefill_b2_s4096", seed, n_h, np.full(B, s_ctx, np.int32))
    return wl


def v2lite_single_step_inputs(seed=0, tokens=26, hidden=2048, n_h=16):
    """V2-Lite layer inputs for a 25-token prefill plus one decode token.

    Draw order: W_DKV [576, hidden], W_Q [n_h * 192, hidden], W_UK, W_UV
    (all N(0, 0.02^2)), then x [tokens, hidden] ~ N(0, 1).  The projections
    ``W_DKV x`` and ``W_Q x`` are the caller's (the layer before the cache).
    """
    rng = np.random.default_rng(seed)
    w_dkv = _normal_bf16(rng, (D_C + D_ROPE, hidden), WEIGHT_STD)
    w_q = _normal_bf16(rng, (n_h * (D_NOPE + D_ROPE), hidden), WEIGHT_STD)
    w_uk = _normal_bf16(rng, (n_h, D_NOPE, D_C), WEIGHT_STD)
    w_uv = _normal_bf16(rng, (n_h, D_V, D_C), WEIGHT_STD)
    x = _normal_bf16(rng, (tokens, hidden), 1.0)
    return dict(w_dkv=w_dkv, w_q=w_q, w_uk=w_uk, w_uv=w_uv, x=x, n_h=n_h, tokens=tokens)


def v2lite_single_step(projected_rows_bits, projected_q_bits, w_uk, w_uv, n_h=16, seed=0) -> Workload:
    """Wrap caller-projected rows ``[T, 576]`` and the last token's query ``[n_h, 192]``
    (bf16 bits) as a B=1 decode workload with one 64-token page."""
    T = projected_rows_bits.shape[0]
    ctx = np.array([T], np.int32)
    rng = np.random.default_rng(seed + 1000)
    bt, num_pages = _paged_layout(rng, ctx, PAGE_SIZE, 2, True)
    seq, pos = _rows_index(ctx)
    return Workload(name="v2lite_b1_s26", n_h=n_h, B=1, ctx_len=ctx, block_table=bt,
                    num_pages=num_pages, w_uk=w_uk, w_uv=w_uv,
                    q=projected_q_bits.reshape(1, n_h, -1), rows=projected_rows_bits,
                    row_seq=seq, row_pos=pos, seed=seed)


def v2lite_batched(seed=1, B=32, max_len=4096, n_h=16) -> Workload:
    """V2-Lite shapes, B=32, per-sequence length uniform on the integers [1, 4096], shuffled pages."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(1, max_len + 1, size=B).astype(np.int32)
    return _finish_decode(rng, "v2lite_b32_ragged", seed, n_h, ctx, CACHE_BF16, True, 8, 1.0, 1.0)


def v3_decode(seed=2, B=64, s_ctx=4096, n_h=128) -> Workload:
    """DeepSeek-V3 shapes, B=64, every sequence 4096 tokens, bf16 cache."""
    rng = np.random.default_rng(seed)
    ctx = np.full(B, s_ctx, np.int32)
    return _finish_decode(rng, "v3_b64_s4096_bf16", seed, n_h, ctx, CACHE_BF16, True, 8, 1.0, 1.0)


def v3_fp8_decode(seed=3, B=128, s_ctx=4096, n_h=128) -> Workload:
    """DeepSeek-V3 shapes, B=128, 4096 tokens each, all 576 columns cached as FP8 e4m3."""
    rng = np.random.default_rng(seed)
    ctx = np.full(B, s_ctx, np.int32)
    return _finish_decode(rng, "v3_b128_s4096_fp8", seed, n_h, ctx, CACHE_FP8, True, 8, 1.0, 1.0)


def v3_fp8_block_decode(seed=3, B=128, s_ctx=4096, n_h=128) -> Workload:
    """The FP8 configuration's shapes and draws (B=128, 4096 tokens each) with the per-block
    format: each row 512 e4m3 latent codes, 4 fp32 block scales and the bf16 RoPE key."""
    rng = np.random.default_rng(seed)
    ctx = np.full(B, s_ctx, np.int32)
    return _finish_decode(rng, "v3_b128_s4096_fp8blk", seed, n_h, ctx, CACHE_FP8_BLOCK, True, 8, 1.0, 1.0)


def v3_long_decode(seed=4, B=8, short=32768, long=65536, n_h=128) -> Workload:
    """DeepSeek-V3 shapes, B=8: the first half of the sequences 32768 tokens, the rest 65536."""
    rng = np.random.default_rng(seed)
    ctx = np.array([short] * (B // 2) + [long] * (B - B // 2), np.int32)
    return _finish_decode(rng, "v3_b8_long", seed, n_h, ctx, CACHE_BF16, True, 8, 1.0, 1.0)


NAMED = {
    "v2lite_b32_ragged": v2lite_batched,
    "v3_b64_s4096_bf16": v3_decode,
    "v3_b128_s4096_fp8": v3_fp8_decode,
    "v3_b8_long": v3_long_decode,
}

# further workloads (not among the five configurations)
EXTRA = {
    "v3_b128_s4096_fp8blk": v3_fp8_block_decode,
}
