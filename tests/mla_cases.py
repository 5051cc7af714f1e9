"""Helpers for the GPU parity tests: run a workload through the C ABI and through
the fp64 oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np

from mla_absorbed_latent_decode_gb300 import workloads as W
from oracle import e4m3, mla_ref

BF16_TOL = 1e-2      # max |gpu - ref| <= tol * max |ref| over the whole output, bf16 cache
FP8_TOL = 5e-2       # same, FP8 cache, against the oracle on its own dequantised cache


def tolerance(wl) -> float:
    return BF16_TOL if wl.cache_dtype == W.CACHE_BF16 else FP8_TOL


def oracle_stored(wl) -> np.ndarray:
    """The codes the oracle's cache holds for every workload row, in row order (chunked)."""
    fp8 = wl.cache_dtype == W.CACHE_FP8
    if wl.cache_dtype == W.CACHE_FP8_BLOCK:
        out = np.empty((wl.rows.shape[0], W.ROW_BYTES[W.CACHE_FP8_BLOCK]), np.uint8)
    else:
        out = np.empty(wl.rows.shape, np.uint8 if fp8 else np.uint16)
    step = 1 << 15
    for a in range(0, wl.rows.shape[0], step):
        r, p = wl.rows[a:a + step], wl.row_pos[a:a + step]
        if wl.cache_dtype == W.CACHE_FP8_BLOCK:
            out[a:a + step] = mla_ref.stored_row_fp8_block(r, p, wl.d_c, wl.rope_base)
        elif fp8:
            out[a:a + step] = mla_ref.stored_row_e4m3(r, p, wl.d_c, wl.rope_base, np.float32(wl.fp8_scale))
        else:
            out[a:a + step] = mla_ref.stored_row_bf16(r, p, wl.d_c, wl.rope_base)
    return out


def oracle_values(wl, stored) -> np.ndarray:
    """float64 values of stored codes (e4m3 codes times the tensor or block scale)."""
    if wl.cache_dtype == W.CACHE_FP8_BLOCK:
        return mla_ref.fp8_block_values(stored, wl.d_c)
    if wl.cache_dtype == W.CACHE_FP8:
        return e4m3.decode(stored) * float(np.float32(wl.fp8_scale))
    return mla_ref.bf16_to_f64(stored)


def oracle_decode(wl, values, seqs=None, path="absorbed") -> np.ndarray:
    """Oracle decode output [len(seqs), n_h, d_v] from the oracle's own cache values.

    The rows of a sequence are contiguous in row order, so the per-sequence
    context is sliced directly; the paged indirection is covered by
    ``oracle_decode_paged`` on small cases."""
    seqs = range(wl.B) if seqs is None else seqs
    starts = np.concatenate([[0], np.cumsum(wl.ctx_len.astype(np.int64))])
    q = mla_ref.bf16_to_f64(wl.q)
    w_uk = mla_ref.bf16_to_f64(wl.w_uk)
    w_uv = mla_ref.bf16_to_f64(wl.w_uv)
    scale = mla_ref.default_scale(wl.d_nope, wl.d_rope)
    fn = mla_ref.absorbed_decode if path == "absorbed" else mla_ref.naive_decode
    out = []
    for b in seqs:
        rows = values[starts[b]:starts[b + 1]]
        L = int(wl.ctx_len[b])
        out.append(fn(q[b], rows[:, :wl.d_c], rows[:, wl.d_c:], w_uk, w_uv, L - 1, scale, wl.rope_base))
    return np.stack(out)


def oracle_decode_paged(wl, values) -> np.ndarray:
    """Oracle decode through its own paged cache (values scattered by the block table)."""
    cache = np.full((wl.num_pages, wl.page_size, wl.d_c + wl.d_rope), np.nan)
    for i in range(values.shape[0]):
        page, slot = mla_ref.page_slot(wl.block_table, int(wl.row_seq[i]), int(wl.row_pos[i]), wl.page_size)
        cache[page, slot] = values[i]
    return mla_ref.decode_batch(mla_ref.bf16_to_f64(wl.q), cache, wl.block_table, wl.ctx_len,
                                mla_ref.bf16_to_f64(wl.w_uk), mla_ref.bf16_to_f64(wl.w_uv), wl.d_c,
                                wl.page_size, mla_ref.default_scale(wl.d_nope, wl.d_rope), wl.rope_base)


def gpu_rows(wl, cache_bytes: np.ndarray) -> np.ndarray:
    """Read every workload row back out of a GPU cache image (codes, row order)."""
    fp8 = wl.cache_dtype != W.CACHE_BF16
    flat = cache_bytes.reshape(wl.num_pages * wl.page_size, -1)
    pages = wl.block_table[wl.row_seq, wl.row_pos // wl.page_size].astype(np.int64)
    slots = pages * wl.page_size + wl.row_pos % wl.page_size
    rows = flat[slots]
    return rows if fp8 else rows.view(np.uint16)


def compare(out_gpu: np.ndarray, ref: np.ndarray, tol: float):
    """max |gpu - ref| / max |ref| over the whole output; asserts finiteness."""
    assert np.all(np.isfinite(out_gpu)), "non-finite GPU output"
    err = float(np.max(np.abs(out_gpu - ref)))
    scale = float(np.max(np.abs(ref)))
    return err / scale, err, scale


def bf16_out_to_f64(t) -> np.ndarray:
    return mla_ref.bf16_to_f64(t.view(__import__("torch").int16).cpu().numpy().view(np.uint16))


# ---------------------------------------------------------------------------
# inputs that force the online softmax's lazy rescale
# ---------------------------------------------------------------------------

LOG2E = 1.4426950408889634
RESCALE_STEP = 8.0        # the kernels rescale O when a row's running maximum grows by more than this (log2 units)


def controlled_rows(q_lat, q_pe_rot, k_r, targets, scale, seed):
    """Latent rows whose scores against the given queries are prescribed.

    q_lat [P, d_c] and q_pe_rot [P, d_rope] are the absorbed queries (latent part; RoPE part
    rotated at the query's position) of P (query, head) pairs; k_r [T, d_rope] the RoPE keys of
    the T rows as cached (rotated at their positions); targets [T, P] the wanted scores
    ``scale * (q_lat . c_t + q_pe . k_r,t)`` in log2 units.  Returns the latent rows c [T, d_c]:
    the minimum-norm solution in the span of the q_lat rows plus a random component
    orthogonal to that span (which leaves every score unchanged).  P <= d_c."""
    sc = scale * LOG2E
    want = targets / sc - k_r @ q_pe_rot.T                     # [T, P]: latent part of each raw score
    gram = q_lat @ q_lat.T
    u = (q_lat.T @ np.linalg.solve(gram, want.T)).T           # [T, d_c]
    r = np.random.default_rng(seed).standard_normal(u.shape)
    r -= (q_lat.T @ np.linalg.solve(gram, q_lat @ r.T)).T
    return u + r


def rescale_targets(n_rows, n_pairs, tile, visible, seed, plateau=16.0, jump=9.0, groups=6):
    """Scores [n_rows, n_pairs] (log2 units) that force every (query, head) pair to rescale once.

    Pair p sees rows 0 .. visible[p] - 1.  Its rows in key tiles 0 .. g(p) - 1 score within
    0.25 of ``plateau``; one row of tile g(p) scores ``plateau + jump`` (jump > the rescale
    step, so the running maximum must grow there, at a tile j = g(p) > 0); every later row scores
    about ``plateau - 12``.  g(p) cycles through 1 .. groups (both parities), capped by the
    pair's last visible tile.  The plateau's 64 g(p) rows keep a weight of about
    64 g(p) 2^-jump against the single high row, so a wrong rescale factor shows in the output.
    Returns (targets, g, row of the jump)."""
    rng = np.random.default_rng(seed)
    d = plateau - 12.0 + rng.uniform(-0.5, 0.5, (n_rows, n_pairs))
    tile_of = np.arange(n_rows)[:, None] // tile
    last_tile = (np.asarray(visible) - 1) // tile
    g = np.minimum(1 + np.arange(n_pairs) % groups, last_tile)
    early = tile_of < g[None, :]
    d[early] = plateau + rng.uniform(-0.25, 0.25, int(early.sum()))
    hit = np.minimum(g * tile + (np.arange(n_pairs) * 7) % tile, np.asarray(visible) - 1)
    d[hit, np.arange(n_pairs)] = plateau + jump
    return d, g, hit


def force_decode_rescale(wl, seed=3, jump=None):
    """Rewrite the latent part of every sequence's rows (of at least 3 pages) so that each head
    rescales at a tile of its own (:func:`rescale_targets` with 64-token tiles, the decode
    kernel's tile; n_h <= d_c / 4 keeps the rows of moderate size).  An e4m3 cache moves scores by up to ~0.3 (log2 units), so its jump is 10
    instead of 9.  Returns {sequence: g per head} for the sequences rewritten."""
    if jump is None:
        jump = 9.0 if wl.cache_dtype == W.CACHE_BF16 else 10.0
    q = mla_ref.bf16_to_f64(wl.q)
    w_uk = mla_ref.bf16_to_f64(wl.w_uk)
    scale = mla_ref.default_scale(wl.d_nope, wl.d_rope)
    starts = np.concatenate([[0], np.cumsum(wl.ctx_len.astype(np.int64))])
    forced = {}
    for b in range(wl.B):
        L = int(wl.ctx_len[b])
        if L < 2 * wl.page_size + 1:
            continue
        qa = mla_ref.absorb_query(q[b], w_uk, L - 1, wl.rope_base)             # [n_h, 576]
        rows = mla_ref.bf16_to_f64(wl.rows[starts[b]:starts[b + 1]])
        k_r = mla_ref.rope(rows[:, wl.d_c:], np.arange(L), wl.rope_base)
        d, g, _ = rescale_targets(L, wl.n_h, wl.page_size, np.full(wl.n_h, L), seed + b, jump=jump)
        c = controlled_rows(qa[:, :wl.d_c], qa[:, wl.d_c:], k_r, d, scale, seed + 1000 + b)
        rows[:, :wl.d_c] = c
        wl.rows[starts[b]:starts[b + 1]] = mla_ref.bf16_round(rows.astype(np.float32))
        forced[b] = g
    if wl.cache_dtype == W.CACHE_FP8:                  # the tensor scale bounds the rewritten rows too
        wl.fp8_scale = W.fp8_tensor_scale(wl.rows, wl.d_c)
    return forced


PREFILL_KEY_TILE = 128    # keys per tile of the prefill attention kernel


def force_prefill_rescale(wl, seed=5):
    """Same for a prefill workload: every (query, head) pair of every sequence whose chunk sees at
    least three key tiles rescales at a key tile of its own (128-key tiles).  The chunk's
    q_len * n_h pairs must not exceed d_c / 4.  Returns {sequence: g per pair}."""
    p = wl.extra["prefill"]
    q = mla_ref.bf16_to_f64(p["q"])
    w_uk = mla_ref.bf16_to_f64(wl.w_uk)
    scale = mla_ref.default_scale(wl.d_nope, wl.d_rope)
    starts = np.concatenate([[0], np.cumsum(wl.ctx_len.astype(np.int64))])
    forced = {}
    for b in range(wl.B):
        L, n, a = int(wl.ctx_len[b]), int(p["q_len"][b]), int(p["q_start"][b])
        pos0 = L - n
        if n == 0 or pos0 + 1 < 2 * PREFILL_KEY_TILE + 1:
            continue
        # few pairs against d_c unknowns keep the system well conditioned (rows of moderate size)
        assert n * wl.n_h <= wl.d_c // 4, "too many (query, head) pairs to prescribe every score"
        qa = np.concatenate([mla_ref.absorb_query(q[a + i], w_uk, pos0 + i, wl.rope_base) for i in range(n)])
        visible = np.repeat(pos0 + 1 + np.arange(n), wl.n_h)
        rows = mla_ref.bf16_to_f64(wl.rows[starts[b]:starts[b + 1]])
        k_r = mla_ref.rope(rows[:, wl.d_c:], np.arange(L), wl.rope_base)
        d, g, _ = rescale_targets(L, n * wl.n_h, PREFILL_KEY_TILE, visible, seed + b)
        rows[:, :wl.d_c] = controlled_rows(qa[:, :wl.d_c], qa[:, wl.d_c:], k_r, d, scale, seed + 1000 + b)
        wl.rows[starts[b]:starts[b + 1]] = mla_ref.bf16_round(rows.astype(np.float32))
        forced[b] = g
    return forced


def decode_scores_log2(wl, values, b):
    """The oracle's scores of sequence b in log2 units [n_h, L] (fp64, from its cached values)."""
    starts = np.concatenate([[0], np.cumsum(wl.ctx_len.astype(np.int64))])
    L = int(wl.ctx_len[b])
    rows = values[starts[b]:starts[b + 1]]
    qa = mla_ref.absorb_query(mla_ref.bf16_to_f64(wl.q[b]), mla_ref.bf16_to_f64(wl.w_uk), L - 1, wl.rope_base)
    return mla_ref.default_scale(wl.d_nope, wl.d_rope) * LOG2E * (qa @ rows.T)
