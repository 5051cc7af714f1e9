"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each.

Each mutation replaces one oracle function with a subtly wrong variant; the
test passes when at least one ``pin_*`` of ``tests/oracle_pins.py`` fails
against the mutated oracle.
"""
import numpy as np
import pytest

from oracle import mla_ref
from tests import oracle_pins

_orig = {name: getattr(mla_ref, name) for name in dir(mla_ref) if not name.startswith("_")}


def _rope_with(sign=1.0, freq_step=2, halves=False):
    def rope(x, pos, base):
        x = np.asarray(x, np.float64)
        d = x.shape[-1]
        inv = 1.0 / (float(base) ** (np.arange(0, d // 2) * freq_step / d))
        theta = np.asarray(pos, np.float64)[..., None] * inv
        c, s = np.cos(theta), sign * np.sin(theta)
        if halves:
            a, b = x[..., : d // 2], x[..., d // 2:]
        else:
            a, b = x[..., 0::2], x[..., 1::2]
        shape = np.broadcast_shapes(x.shape, theta.shape[:-1] + (d,))
        out = np.empty(shape)
        if halves:
            out[..., : d // 2] = a * c - b * s
            out[..., d // 2:] = b * c + a * s
        else:
            out[..., 0::2] = a * c - b * s
            out[..., 1::2] = b * c + a * s
        return out
    return rope


def _absorbed_latent_no_rope(q_abs, c_kv, k_r_rot, scale):
    d_c = c_kv.shape[1]
    s = scale * (q_abs[:, :d_c] @ np.asarray(c_kv, np.float64).T)
    p = _orig["softmax"](s, axis=1)
    m = np.max(s, axis=1)
    return p @ c_kv, m + np.log(np.sum(np.exp(s - m[:, None]), axis=1))


def _absorb_query_shifted(q, w_uk, pos_q, base):
    return _orig["absorb_query"](q, w_uk, pos_q + 1, base)


def _naive_without_rope_key(q, c_kv, k_r_rot, w_uk, w_uv, pos_q, scale, base):
    return _orig["naive_decode"](q, c_kv, np.zeros_like(np.asarray(k_r_rot, np.float64)),
                                 w_uk, w_uv, pos_q, scale, base)


def _softmax_unnormalised(s, axis=-1):
    s = np.asarray(s, np.float64)
    return np.exp(s - np.max(s, axis=axis, keepdims=True))


def _causal_unmasked(x, w_dkv, w_q, w_uk, w_uv, scale, base):
    n_h, d_nope, d_c = w_uk.shape
    c_kv, k_r, q = _orig["project_inputs"](x, w_dkv, w_q, n_h, d_c)
    L = c_kv.shape[0]
    pos = np.arange(L)
    k_r_rot = mla_ref.rope(k_r, pos, base)
    q_pe = mla_ref.rope(q[:, :, d_nope:], pos[:, None], base)
    out = np.empty((L, n_h, w_uv.shape[1]))
    for h in range(n_h):
        k = np.concatenate([c_kv @ w_uk[h].T, k_r_rot], axis=1)
        v = c_kv @ w_uv[h].T
        qh = np.concatenate([q[:, h, :d_nope], q_pe[:, h]], axis=1)
        out[:, h] = _orig["softmax"](scale * (qh @ k.T), axis=1) @ v
    return out


def _split_linear_merge(q_abs, c_kv, k_r_rot, scale, bounds):
    parts = [_orig["absorbed_latent"](q_abs, c_kv[a:b], k_r_rot[a:b], scale)
             for a, b in zip(bounds[:-1], bounds[1:])]
    w = np.stack([np.exp(p[1]) for p in parts])
    w = w / w.sum(0)
    lens = np.array([b - a for a, b in zip(bounds[:-1], bounds[1:])], float)
    w = (w.T * lens / lens.mean()).T            # wrong: weights chunks by length too
    return sum(w[j][:, None] * parts[j][0] for j in range(len(parts))), np.log(np.exp(np.stack([p[1] for p in parts])).sum(0))


def _prefill_with(strict_mask=False, chunk_position=False):
    def prefill(q, c_kv, k_r_rot, w_uk, w_uv, pos0, scale, base):
        q = np.asarray(q, np.float64)
        n_q, T = q.shape[0], pos0 + q.shape[0]
        n_h, d_nope, _ = w_uk.shape
        qpos = pos0 + np.arange(n_q)
        q_pe = mla_ref.rope(q[:, :, d_nope:], (np.full(n_q, pos0) if chunk_position else qpos)[:, None], base)
        visible = (np.arange(T)[None, :] < qpos[:, None]) if strict_mask else (np.arange(T)[None, :] <= qpos[:, None])
        visible[:, 0] = True                     # keep every row defined
        out = np.empty((n_q, n_h, w_uv.shape[1]))
        for h in range(n_h):
            k = np.concatenate([c_kv[:T] @ w_uk[h].T, k_r_rot[:T]], axis=1)
            qh = np.concatenate([q[:, h, :d_nope], q_pe[:, h]], axis=1)
            s = np.where(visible, scale * (qh @ k.T), -np.inf)
            out[:, h] = _orig["softmax"](s, axis=1) @ (c_kv[:T] @ w_uv[h].T)
        return out
    return prefill


def _fp8_block_with(per_row=False, sat=448.0, quantise_rope=False):
    from oracle import e4m3

    def stored(row_bf16_bits, pos, d_c, base):
        bits = np.asarray(row_bf16_bits, np.uint16).reshape(-1, 576)
        x = mla_ref.bf16_to_f64(bits).astype(np.float32)
        n = x.shape[0]
        lat = x[:, :d_c].reshape(n, 4, 128)
        amax = np.max(np.abs(lat), axis=2)
        if per_row:
            amax = np.repeat(np.max(amax, axis=1, keepdims=True), 4, axis=1)
        scale = (amax / np.float32(sat)).astype(np.float32)
        safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
        codes = np.where(scale[:, :, None] > 0, e4m3.encode(lat / safe[:, :, None]), 0).astype(np.uint8)
        rr = mla_ref.rope_row_fp32(x[:, d_c:], np.asarray(pos).reshape(-1) if np.ndim(pos) else pos, base)
        if quantise_rope:
            rr = e4m3.decode(e4m3.encode(rr)).astype(np.float32)
        rope = mla_ref.bf16_round(rr)
        return np.concatenate([codes.reshape(n, d_c), scale.astype("<f4").view(np.uint8).reshape(n, 16),
                               rope.astype("<u2").view(np.uint8).reshape(n, -1)], axis=1)
    return stored


def _gather_pages_sorted(cache_values, block_table, seq, length, page_size):
    n_pages = (length + page_size - 1) // page_size
    ids = sorted(int(block_table[seq][i]) for i in range(n_pages))
    pages = [cache_values[i] for i in ids]
    return np.concatenate(pages, axis=0)[:length] if pages else np.zeros((0, cache_values.shape[-1]))


def _decode_batch_query_at_len(q, cache_values, block_table, ctx_len, w_uk, w_uv, d_c, page_size, scale, base,
                               seqs=None, path="absorbed"):
    fn = _orig["absorbed_decode"] if path == "absorbed" else _orig["naive_decode"]
    out = []
    for b in (range(q.shape[0]) if seqs is None else seqs):
        L = int(ctx_len[b])
        rows = _orig["gather_sequence"](cache_values, block_table, b, L, page_size)
        out.append(fn(q[b], rows[:, :d_c], rows[:, d_c:], w_uk, w_uv, L, scale, base))
    return np.stack(out)


MUTATIONS = {
    "rope_rotates_backwards": ("rope", _rope_with(sign=-1.0)),
    "rope_frequency_step_1": ("rope", _rope_with(freq_step=1)),
    "rope_pairs_by_halves": ("rope", _rope_with(halves=True)),
    "scale_without_rope_width": ("default_scale", lambda d_nope, d_rope: 1.0 / np.sqrt(float(d_nope))),
    "absorbed_drops_rope_score": ("absorbed_latent", _absorbed_latent_no_rope),
    "query_position_off_by_one": ("absorb_query", _absorb_query_shifted),
    "naive_drops_rope_key": ("naive_decode", _naive_without_rope_key),
    "softmax_unnormalised": ("softmax", _softmax_unnormalised),
    "causal_mask_missing": ("causal_forward_naive", _causal_unmasked),
    "fp8_block_one_scale_per_row": ("stored_row_fp8_block", _fp8_block_with(per_row=True)),
    "fp8_block_saturation_127": ("stored_row_fp8_block", _fp8_block_with(sat=127.0)),
    "fp8_block_rope_quantised": ("stored_row_fp8_block", _fp8_block_with(quantise_rope=True)),
    "rms_norm_without_root": ("rms_norm", lambda x, w, eps: np.asarray(x, float) / (np.mean(np.asarray(x, float) ** 2, axis=-1, keepdims=True) + eps) * w),
    "rms_norm_eps_outside_root": ("rms_norm", lambda x, w, eps: np.asarray(x, float) / (np.sqrt(np.mean(np.asarray(x, float) ** 2, axis=-1, keepdims=True)) + eps) * w),
    "low_rank_query_swaps_content_and_rope": ("low_rank_query", lambda x, w_dq, w_uq, w_qr, n_h: _orig["low_rank_query"](x, w_dq, w_qr, w_uq, n_h) if w_uq.shape == w_qr.shape else np.concatenate([(np.asarray(x) @ np.asarray(w_dq).T @ np.asarray(w_qr).T).reshape(len(x), n_h, -1), (np.asarray(x) @ np.asarray(w_dq).T @ np.asarray(w_uq).T).reshape(len(x), n_h, -1)], axis=2)),
    "prefill_mask_excludes_diagonal": ("prefill_naive", _prefill_with(strict_mask=True)),
    "prefill_queries_rotated_at_chunk_start": ("prefill_naive", _prefill_with(chunk_position=True)),
    "cache_bytes_without_rope": ("absorb_cache_bytes", lambda t, d_c, d_r, e: int(t) * int(d_c) * int(e)),
    "naive_bytes_without_values": ("naive_cache_bytes", lambda t, n, dn, dr, dv, e: int(t) * int(n) * (int(dn) + int(dr)) * int(e)),
    "read_bytes_times_heads": ("decode_kv_read_bytes", lambda B, s, d_c, d_r, e: _orig["decode_kv_read_bytes"](B, s, d_c, d_r, e) * 2),
    "split_merge_weighted_by_length": ("split_latent", _split_linear_merge),
    "up_projection_skipped": ("up_project", lambda o_lat, w_uv: o_lat[:, : w_uv.shape[1]]),
    "page_slot_divides_the_wrong_way": ("page_slot", lambda bt, seq, pos, ps: (int(bt[seq][pos % ps]), int(pos // ps))),
    "page_slot_off_by_one_page": ("page_slot", lambda bt, seq, pos, ps: (int(bt[seq][(pos + 1) // ps]), int(pos % ps))),
    "gather_pages_in_id_order": ("gather_sequence", _gather_pages_sorted),
    "decode_batch_query_at_len": ("decode_batch", _decode_batch_query_at_len),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_some_pin_catches(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(mla_ref, attr, fn)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mla_ref)
        except Exception as e:     # an assertion or a shape error both mean "caught"
            caught.append(pin.__name__)
    assert caught, f"mutation {name} passed every pin"
