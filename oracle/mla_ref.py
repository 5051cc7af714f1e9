"""fp64 reference for MLA decode: naive (expanded) path and absorbed path.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path.

Notation follows the pages: ``d_c`` is the KV latent width (kv_lora_rank, 512),
``d_rope`` the decoupled RoPE key width (64), ``n_h`` heads, ``d_nope`` the
no-RoPE query/key width per head (128), ``d_v`` the value width per head (128).
A cached row is ``[c_kv (d_c) | k_r (d_rope)]``; a query head is
``[q_nope (d_nope) | q_pe (d_rope)]``.  All arithmetic is float64 unless a
function says otherwise.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def rope_inv_freq(d_rope: int, base: float) -> np.ndarray:
    """Per-pair inverse frequency ``base ** -(2i / d_rope)``, i = 0 .. d_rope/2 - 1.

    "80 行 PyTorch 从零写 DeepSeek 的 MLA", 附录 A (``build_rope``): the
    exponent steps over even indices 0, 2, 4, ... divided by the rotary width.
    """
    two_i = np.arange(0, d_rope, 2, dtype=np.float64)
    return 1.0 / (float(base) ** (two_i / d_rope))


def rope_angles(pos, d_rope: int, base: float) -> np.ndarray:
    """Angle ``theta[..., i] = pos * inv_freq[i]`` in float64 (shape pos.shape + (d_rope/2,))."""
    pos = np.asarray(pos, dtype=np.float64)
    return pos[..., None] * rope_inv_freq(d_rope, base)


def rope(x: np.ndarray, pos, base: float) -> np.ndarray:
    """Rotate interleaved pairs ``(x[2i], x[2i+1])`` by ``theta_i = pos * inv_freq_i``.

    "80 行 PyTorch 从零写 DeepSeek 的 MLA", 附录 A (``rotate_half`` /
    ``apply_rope``): ``rotate_half`` maps a pair (a, b) to (-b, a) and
    ``apply_rope`` returns ``x * cos + rotate_half(x) * sin`` with each angle
    repeated over its pair, i.e.

        out[2i]   = x[2i]   cos(theta_i) - x[2i+1] sin(theta_i)
        out[2i+1] = x[2i+1] cos(theta_i) + x[2i]   sin(theta_i)

    ``x`` has shape ``[..., d_rope]``; ``pos`` broadcasts against ``x.shape[:-1]``.
    """
    x = np.asarray(x, dtype=np.float64)
    theta = rope_angles(pos, x.shape[-1], base)
    cos, sin = np.cos(theta), np.sin(theta)
    even, odd = x[..., 0::2], x[..., 1::2]
    out = np.empty(np.broadcast_shapes(x.shape, theta.shape[:-1] + (x.shape[-1],)))
    out[..., 0::2] = even * cos - odd * sin
    out[..., 1::2] = odd * cos + even * sin
    return out


# ---------------------------------------------------------------------------
# softmax attention
# ---------------------------------------------------------------------------

def softmax(s: np.ndarray, axis: int = -1) -> np.ndarray:
    """Softmax with the maximum subtracted first (float64).

    The pages use ``F.scaled_dot_product_attention`` ("80 行 PyTorch 从零写
    DeepSeek 的 MLA", §2); this is the textbook definition it computes.
    """
    s = np.asarray(s, dtype=np.float64)
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def default_scale(d_nope: int, d_rope: int) -> float:
    """Softmax scale ``1 / sqrt(d_nope + d_rope)``: the query/key head width is
    ``d_nope + d_rope`` ("80 行 PyTorch 从零写 DeepSeek 的 MLA", §2: q and k are
    the concatenation of the content and rope parts, scored by SDPA's default
    scale)."""
    return 1.0 / np.sqrt(float(d_nope + d_rope))


# ---------------------------------------------------------------------------
# decode of one query token of one sequence
# ---------------------------------------------------------------------------

def naive_decode(q, c_kv, k_r_rot, w_uk, w_uv, pos_q, scale, base):
    """Standard-mode MLA decode: expand every cached latent into per-head K and V.

    "DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §2.1 and
    "80 行 PyTorch 从零写 DeepSeek 的 MLA" §2 (``k_c = Wuk(c_kv)``,
    ``v = Wuv(c_kv)``, ``k = cat(k_c, k_r)``, ``q = cat(q_c, q_r)``, SDPA):

        k_{h,t} = [ W_UK[h] c_t ; k_r,t ]          (k_r,t already rotated at t)
        v_{h,t} = W_UV[h] c_t
        q_h     = [ q_nope,h ; RoPE(q_pe,h, pos_q) ]
        o_h     = sum_t softmax_t(scale * q_h . k_{h,t}) v_{h,t}

    Shapes: q [n_h, d_nope + d_rope], c_kv [T, d_c], k_r_rot [T, d_rope],
    w_uk [n_h, d_nope, d_c], w_uv [n_h, d_v, d_c].  Returns [n_h, d_v].
    """
    q = np.asarray(q, np.float64)
    c_kv = np.asarray(c_kv, np.float64)
    k_r_rot = np.asarray(k_r_rot, np.float64)
    n_h, d_nope, _ = w_uk.shape
    d_v = w_uv.shape[1]
    q_nope = q[:, :d_nope]
    q_pe = rope(q[:, d_nope:], pos_q, base)
    out = np.empty((n_h, d_v))
    for h in range(n_h):
        k_c = c_kv @ np.asarray(w_uk[h], np.float64).T          # [T, d_nope]
        v = c_kv @ np.asarray(w_uv[h], np.float64).T            # [T, d_v]
        k = np.concatenate([k_c, k_r_rot], axis=1)               # [T, d_nope + d_rope]
        q_h = np.concatenate([q_nope[h], q_pe[h]])
        p = softmax(scale * (k @ q_h))
        out[h] = p @ v
    return out


def absorb_query(q, w_uk, pos_q, base):
    """The absorbed query of every head: ``[W_UK[h]^T q_nope,h ; RoPE(q_pe,h, pos_q)]``.

    "DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §2.2:
    ``q^T (W^K c) = (W^K^T q)^T c``, so the no-RoPE query moves into latent
    space; the RoPE part cannot be absorbed (§2.4) and is rotated at the query
    position.  Returns [n_h, d_c + d_rope].
    """
    q = np.asarray(q, np.float64)
    d_nope = w_uk.shape[1]
    q_lat = np.einsum("hn,hnc->hc", q[:, :d_nope], np.asarray(w_uk, np.float64))
    q_pe = rope(q[:, d_nope:], pos_q, base)
    return np.concatenate([q_lat, q_pe], axis=1)


def absorbed_latent(q_abs, c_kv, k_r_rot, scale):
    """Softmax-weighted latent sum for absorbed queries: ``o_lat = sum_t p_t c_t``.

    "DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §2.2-§2.4 and
    "80 行 PyTorch 从零写 DeepSeek 的 MLA" §5 (content score ``Q_abs . c_kv``
    plus rope score ``q_r . k_r``, then the latent context ``[B, H, 1, d_c]``).

    q_abs [n_h, d_c + d_rope]; returns (o_lat [n_h, d_c], lse [n_h]) where
    ``lse`` is the natural log of the softmax normaliser of the scaled scores.
    """
    c_kv = np.asarray(c_kv, np.float64)
    k_r_rot = np.asarray(k_r_rot, np.float64)
    d_c = c_kv.shape[1]
    s = scale * (q_abs[:, :d_c] @ c_kv.T + q_abs[:, d_c:] @ k_r_rot.T)   # [n_h, T]
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    z = np.sum(e, axis=1, keepdims=True)
    o_lat = (e / z) @ c_kv
    return o_lat, (m + np.log(z))[:, 0]


def up_project(o_lat, w_uv):
    """Per-head value up-projection ``o_h = W_UV[h] o_lat,h`` after the latent sum.

    "DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §2.3:
    ``sum_t p_t (W^V c_t) = W^V (sum_t p_t c_t)``.  Returns [n_h, d_v].
    """
    return np.einsum("hvc,hc->hv", np.asarray(w_uv, np.float64), o_lat)


def absorbed_decode(q, c_kv, k_r_rot, w_uk, w_uv, pos_q, scale, base):
    """Absorb-mode MLA decode of one token (the path the GPU implements).

    "DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §2.2-§2.4;
    "80 行 PyTorch 从零写 DeepSeek 的 MLA" §5.  Same inputs and output as
    :func:`naive_decode`; in exact arithmetic the two are the same function.
    """
    q_abs = absorb_query(q, w_uk, pos_q, base)
    o_lat, _ = absorbed_latent(q_abs, c_kv, k_r_rot, scale)
    return up_project(o_lat, w_uv)


def split_latent(q_abs, c_kv, k_r_rot, scale, bounds):
    """The absorbed latent sum computed over token chunks, then merged by log-sum-exp.

    Not on the pages: chunking the context and merging the chunks' partial
    softmax sums by their log-sum-exp is the standard identity
    ``softmax over the union = sum_j exp(lse_j - lse) * softmax over chunk j``.
    ``bounds`` lists chunk edges ``[0, b1, ..., T]``.  Returns (o_lat, lse).
    """
    parts = [absorbed_latent(q_abs, c_kv[a:b], k_r_rot[a:b], scale)
             for a, b in zip(bounds[:-1], bounds[1:])]
    lses = np.stack([p[1] for p in parts])               # [J, n_h]
    lse = np.max(lses, axis=0) + np.log(np.sum(np.exp(lses - np.max(lses, axis=0)), axis=0))
    w = np.exp(lses - lse)                               # [J, n_h]
    o_lat = sum(w[j][:, None] * parts[j][0] for j in range(len(parts)))
    return o_lat, lse


# ---------------------------------------------------------------------------
# one-shot causal forward (the incremental-decode pin)
# ---------------------------------------------------------------------------

def project_inputs(x, w_dkv, w_q, n_h, d_c):
    """Input projections of one layer: ``kv_row = W_DKV x`` and ``q = W_Q x``.

    "DeepSeek-V2-Lite 真实权重执行审计" §3.1: ``kv_a_proj_with_mqa`` emits
    ``[B, T, 512 + 64]`` (latent then RoPE key); V2-Lite has a direct
    ``q_proj`` to ``n_h x (128 + 64)``.  Returns (c_kv [L, d_c],
    k_r [L, d_rope] unrotated, q [L, n_h, d_q]).
    """
    x = np.asarray(x, np.float64)
    kv = x @ np.asarray(w_dkv, np.float64).T
    q = (x @ np.asarray(w_q, np.float64).T).reshape(x.shape[0], n_h, -1)
    return kv[:, :d_c], kv[:, d_c:], q


def rms_norm(x, w, eps):
    """RMSNorm of each row (Zhang & Sennrich, "Root Mean Square Layer Normalization", 2019):
    ``y = x / sqrt(mean(x^2) + eps) * w``, float64.

    The pages name the norm of the KV latent ("DeepSeek MLA 吸收式缓存：真实权重执行与
    FlashMLA 架构边界" §3.3: ``kv_a_layernorm.weight`` is the reference's ``kv_norm.weight``;
    §3.1: the layer's input RMSNorm) without restating it; this is the published definition.
    x [..., n], w [n].
    """
    x = np.asarray(x, np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + float(eps)) * np.asarray(w, np.float64)


def low_rank_query(x, w_dq, w_uq, w_qr, n_h):
    """The low-rank query path: ``qz = W_DQ x``, ``q_c = W_UQ qz`` (content, n_h x d_nope),
    ``q_r = W_QR qz`` (rope, n_h x d_rope), joined per head as ``[q_c ; q_r]``.

    "80 行 PyTorch 从零写 DeepSeek 的 MLA" §2: the query also goes through a low-rank
    factorisation (``Wdq``, then ``Wuq`` and ``Wqr``).  x [L, d_model]; returns
    [L, n_h, d_nope + d_rope].
    """
    qz = np.asarray(x, np.float64) @ np.asarray(w_dq, np.float64).T
    q_c = (qz @ np.asarray(w_uq, np.float64).T).reshape(qz.shape[0], n_h, -1)
    q_r = (qz @ np.asarray(w_qr, np.float64).T).reshape(qz.shape[0], n_h, -1)
    return np.concatenate([q_c, q_r], axis=2)


def causal_forward_naive(x, w_dkv, w_q, w_uk, w_uv, scale, base):
    """One-shot causal forward over all L tokens with expanded K/V.

    "80 行 PyTorch 从零写 DeepSeek 的 MLA" §2: with no cache the whole
    sequence is projected, K_C/V are rebuilt from ``c_kv``, the rope key is
    rotated at positions ``0..L-1``, the queries at the same positions, and SDPA
    runs with ``is_causal=True``.  Here the full ``[n_h, L, L]`` score matrix is
    formed and masked.  Returns [L, n_h, d_v].
    """
    n_h, d_nope, d_c = w_uk.shape
    c_kv, k_r, q = project_inputs(x, w_dkv, w_q, n_h, d_c)
    L = c_kv.shape[0]
    pos = np.arange(L)
    k_r_rot = rope(k_r, pos, base)                       # [L, d_rope]
    q_pe = rope(q[:, :, d_nope:], pos[:, None], base)    # [L, n_h, d_rope]
    out = np.empty((L, n_h, w_uv.shape[1]))
    mask = np.tril(np.ones((L, L), dtype=bool))
    for h in range(n_h):
        k = np.concatenate([c_kv @ np.asarray(w_uk[h], np.float64).T, k_r_rot], axis=1)
        v = c_kv @ np.asarray(w_uv[h], np.float64).T
        qh = np.concatenate([q[:, h, :d_nope], q_pe[:, h]], axis=1)   # [L, d_q]
        s = scale * (qh @ k.T)
        s = np.where(mask, s, -np.inf)
        out[:, h] = softmax(s, axis=1) @ v
    return out


# ---------------------------------------------------------------------------
# prefill of a chunk of queries over the cached rows
# ---------------------------------------------------------------------------

def prefill_naive(q, c_kv, k_r_rot, w_uk, w_uv, pos0, scale, base):
    """Causal prefill of ``n_q`` query tokens in standard (MHA) mode over a sequence's rows.

    "G5 MLA KV 访存建模设计规格", 名词定义 and 用例 2: prefill handles every prompt
    token in one pass (query length = prompt length) and is compute-bound;
    "DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §6.1: dense prefill
    runs in MHA mode, i.e. with the latent expanded per head (§2.1):

        k_{h,t} = [ W_UK[h] c_t ; k_r,t ],   v_{h,t} = W_UV[h] c_t
        q_{h,i} = [ q_nope,h,i ; RoPE(q_pe,h,i, pos0 + i) ]
        o_{h,i} = sum_{t <= pos0 + i} softmax_t(scale * q_{h,i} . k_{h,t}) v_{h,t}

    Query i sits at position ``pos0 + i`` and sees the rows ``0 .. pos0 + i`` (a
    chunk after a cached prefix of ``pos0`` rows; ``pos0 = 0`` is a whole prompt).
    The full masked score matrix is formed per head.  Shapes: q [n_q, n_h, d_q],
    c_kv [T, d_c], k_r_rot [T, d_rope] (rotated at their positions) with
    T >= pos0 + n_q.  Returns [n_q, n_h, d_v].
    """
    q = np.asarray(q, np.float64)
    n_q = q.shape[0]
    T = pos0 + n_q
    c_kv = np.asarray(c_kv, np.float64)[:T]
    k_r_rot = np.asarray(k_r_rot, np.float64)[:T]
    n_h, d_nope, _ = w_uk.shape
    qpos = pos0 + np.arange(n_q)
    q_pe = rope(q[:, :, d_nope:], qpos[:, None], base)          # [n_q, n_h, d_rope]
    visible = np.arange(T)[None, :] <= qpos[:, None]             # [n_q, T]
    out = np.empty((n_q, n_h, w_uv.shape[1]))
    for h in range(n_h):
        k = np.concatenate([c_kv @ np.asarray(w_uk[h], np.float64).T, k_r_rot], axis=1)   # [T, d_q]
        v = c_kv @ np.asarray(w_uv[h], np.float64).T                                     # [T, d_v]
        qh = np.concatenate([q[:, h, :d_nope], q_pe[:, h]], axis=1)                      # [n_q, d_q]
        s = np.where(visible, scale * (qh @ k.T), -np.inf)
        out[:, h] = softmax(s, axis=1) @ v
    return out


# ---------------------------------------------------------------------------
# the paged latent cache (stored values of a row)
# ---------------------------------------------------------------------------

def page_slot(block_table, seq, pos, page_size):
    """Where the row of token ``pos`` of sequence ``seq`` lives: ``(page, slot)``.

    The pages require a paged latent-only cache for production
    ("DeepSeek-V2-Lite 真实权重执行审计" §3.3) without fixing its layout; the
    layout read here is a block table of page ids per sequence, token ``pos``
    in page ``block_table[seq][pos // page_size]`` at slot ``pos % page_size``.
    """
    return int(block_table[seq][pos // page_size]), int(pos % page_size)


def rope_row_fp32(k_r, pos, base):
    """RoPE of a cached key computed the way the stored code is decided: in fp32.

    The rotation is "80 行 PyTorch 从零写 DeepSeek 的 MLA" 附录 A (see
    :func:`rope`).  The value written to a bf16 or e4m3 cache is a rounding
    decision; it is taken in the precision the kernel takes it in: the angle
    in float64, cos/sin rounded to float32, then each product and each sum
    rounded to float32 separately (no fused multiply-add).
    """
    k_r = np.asarray(k_r, np.float32)
    theta = rope_angles(pos, k_r.shape[-1], base)
    cos, sin = np.cos(theta).astype(np.float32), np.sin(theta).astype(np.float32)
    even, odd = k_r[..., 0::2], k_r[..., 1::2]
    out = np.empty(k_r.shape, np.float32)
    out[..., 0::2] = (even * cos) - (odd * sin)
    out[..., 1::2] = (odd * cos) + (even * sin)
    return out


def bf16_round(x):
    """Round float32 values to bfloat16, nearest-even; returns the bf16 bit patterns (uint16)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(np.asarray(x, np.float32))
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return np.where(nan, np.uint16(0x7FC0), r)


def bf16_to_f64(bits):
    """Exact value of bf16 bit patterns."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def stored_row_bf16(row_bf16_bits, pos, d_c, base):
    """The 576 bf16 codes a bf16 cache holds for one appended row.

    The latent part is stored as given; the RoPE key is rotated at the row's
    absolute position before it is cached ("DeepSeek MLA 吸收式缓存：真实权重执行与
    FlashMLA 架构边界" §2.4: the rope key is position dependent and is cached;
    "80 行 PyTorch 从零写 DeepSeek 的 MLA" §2: keys are rotated at
    ``arange(Lt)``) and rounded to bf16.
    """
    row = bf16_to_f64(row_bf16_bits).astype(np.float32)
    out = np.array(row_bf16_bits, dtype=np.uint16, copy=True)
    out[..., d_c:] = bf16_round(rope_row_fp32(row[..., d_c:], pos, base))
    return out


def stored_row_e4m3(row_bf16_bits, pos, d_c, base, scale):
    """The 576 e4m3 codes an FP8 cache holds for one appended row.

    All cached columns are stored as FP8 E4M3 with one fp32 tensor scale
    ("G5 MLA KV 访存建模设计规格" 用例说明, use case 1: DeepSeek-V3 decode with an
    FP8 latent cache, 1 byte per element): each value (latent as given, RoPE key
    rotated as in :func:`stored_row_bf16`) is divided by the scale in float32
    and encoded round-to-nearest-even, saturating at +-448.
    """
    from .e4m3 import encode
    row = bf16_to_f64(row_bf16_bits).astype(np.float32)
    vals = row.copy()
    vals[..., d_c:] = rope_row_fp32(row[..., d_c:], pos, base)
    return encode(vals / np.float32(scale))


FP8_BLOCK = 128          # latent values per scale in the per-block FP8 format


def stored_row_fp8_block(row_bf16_bits, pos, d_c, base):
    """The 656 bytes a per-block-scaled FP8 cache holds for one appended row.

    "G5 MLA KV 访存建模设计规格" 附录 A (FlashMLA row): the deployed FP8 cache
    holds 656 bytes per token with per-block scales, against 576 for the pure
    latent; the page does not break the 656 down.  Reading taken (it sums to
    656 exactly): ``[512 e4m3 latent codes | 4 fp32 scales, one per 128 latent
    values | 64 bf16 RoPE-key values]``.  A block's scale is its largest
    magnitude divided by 448 (the largest e4m3 magnitude) in float32, 0 for an
    all-zero block; each latent value is divided by its block's scale in float32
    and encoded e4m3 nearest-even, saturating; the RoPE key is rotated and
    rounded to bf16 exactly as in :func:`stored_row_bf16` (not quantised).
    Input [..., 576] bf16 bits; returns uint8 [..., 656].
    """
    from .e4m3 import encode
    bits = np.asarray(row_bf16_bits, np.uint16)
    lead = bits.shape[:-1]
    x = bf16_to_f64(bits).astype(np.float32).reshape(-1, bits.shape[-1])
    n, nb = x.shape[0], d_c // FP8_BLOCK
    lat = x[:, :d_c].reshape(n, nb, FP8_BLOCK)
    scale = (np.max(np.abs(lat), axis=2) / np.float32(448.0)).astype(np.float32)          # [n, nb]
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    codes = np.where(scale[:, :, None] > 0, encode(lat / safe[:, :, None]), np.uint8(0)).astype(np.uint8)
    rope = bf16_round(rope_row_fp32(x[:, d_c:], np.asarray(pos).reshape(-1) if np.ndim(pos) else pos, base))
    out = np.concatenate([codes.reshape(n, d_c), scale.astype("<f4").view(np.uint8).reshape(n, 4 * nb),
                          rope.astype("<u2").view(np.uint8).reshape(n, -1)], axis=1)
    return out.reshape(lead + (out.shape[-1],))


def fp8_block_values(stored, d_c):
    """float64 values of per-block FP8 rows (see :func:`stored_row_fp8_block`): each latent
    code's value times its block's scale, then the bf16 RoPE key.  Returns [..., d_c + d_rope]."""
    from .e4m3 import decode
    st = np.asarray(stored, np.uint8)
    lead = st.shape[:-1]
    st = st.reshape(-1, st.shape[-1])
    nb = d_c // FP8_BLOCK
    scale = np.ascontiguousarray(st[:, d_c:d_c + 4 * nb]).view("<f4").astype(np.float64)       # [n, nb]
    lat = decode(st[:, :d_c]).reshape(-1, nb, FP8_BLOCK) * scale[:, :, None]
    rope = bf16_to_f64(np.ascontiguousarray(st[:, d_c + 4 * nb:]).view("<u2"))
    out = np.concatenate([lat.reshape(-1, d_c), rope], axis=1)
    return out.reshape(lead + (out.shape[-1],))


# ---------------------------------------------------------------------------
# byte accounting
# ---------------------------------------------------------------------------

def absorb_cache_bytes(tokens, d_c, d_rope, elem_bytes):
    """Latent cache bytes ``tokens * (d_c + d_rope) * e``.

    "G5 MLA KV 访存建模设计规格" 算法与公式, eq. gmkv-cache (per token and
    layer), times the number of tokens.
    """
    return int(tokens) * (int(d_c) + int(d_rope)) * int(elem_bytes)


def naive_cache_bytes(tokens, n_h, d_nope, d_rope, d_v, elem_bytes):
    """Expanded K/V cache bytes: keys ``n_h x (d_nope + d_rope)`` and values ``n_h x d_v`` per token.

    "DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界" §2.1 (key 16 x
    (128 + 64), value 16 x 128 elements per token and layer).
    """
    return int(tokens) * int(n_h) * (int(d_nope) + int(d_rope) + int(d_v)) * int(elem_bytes)


def decode_kv_read_bytes(batch, s_ctx, d_c, d_rope, elem_bytes):
    """Decode-step HBM latent read ``B * s_ctx * (d_c + d_rope) * e`` (no head count).

    "G5 MLA KV 访存建模设计规格" 算法与公式, eq. gmkv-read.  ``s_ctx`` may be a
    sequence of per-sequence lengths, in which case their sum replaces
    ``B * s_ctx``.
    """
    if np.ndim(s_ctx) == 0:
        total = int(batch) * int(s_ctx)
    else:
        total = int(np.sum(np.asarray(s_ctx, dtype=np.int64)))
    return total * (int(d_c) + int(d_rope)) * int(elem_bytes)


def mha_ratio(d_c, d_rope, n_h, d_h):
    """Latent cache over an equal-size MHA cache: ``(d_c + d_rope) / (2 n_h d_h)``.

    "G5 MLA KV 访存建模设计规格" 算法与公式, eq. gmkv-ratio.
    """
    return (d_c + d_rope) / (2.0 * n_h * d_h)


# ---------------------------------------------------------------------------
# batched decode over a paged cache (what the GPU's mla_decode computes)
# ---------------------------------------------------------------------------

def gather_sequence(cache_values, block_table, seq, length, page_size):
    """Rows ``0..length-1`` of sequence ``seq`` from a paged cache of values ``[P, page, width]``.

    Row t is read from :func:`page_slot` ``(block_table, seq, t)``; whole pages are
    gathered in block-table order and the tail past ``length`` dropped.
    """
    n_pages = (length + page_size - 1) // page_size
    pages = [cache_values[int(block_table[seq][i])] for i in range(n_pages)]
    rows = np.concatenate(pages, axis=0)[:length] if pages else np.zeros((0, cache_values.shape[-1]))
    return rows


def decode_batch(q, cache_values, block_table, ctx_len, w_uk, w_uv, d_c, page_size,
                 scale, base, seqs=None, path="absorbed"):
    """Decode of one token per sequence over a paged cache of dequantised values.

    For sequence b the context is its first ``ctx_len[b]`` cached rows and the
    query sits at position ``ctx_len[b] - 1`` ("80 行 PyTorch 从零写 DeepSeek 的
    MLA" §2: the query positions are ``arange(Lt - L, Lt)``, here L = 1 and the
    decode token's own row has been appended first).  ``cache_values`` holds the
    stored rows as float64 (k_r already rotated).  Returns [len(seqs), n_h, d_v].
    """
    fn = absorbed_decode if path == "absorbed" else naive_decode
    seqs = range(q.shape[0]) if seqs is None else seqs
    out = []
    for b in seqs:
        L = int(ctx_len[b])
        rows = gather_sequence(cache_values, block_table, b, L, page_size)
        out.append(fn(q[b], rows[:, :d_c], rows[:, d_c:], w_uk, w_uv, L - 1, scale, base))
    return np.stack(out)
