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
