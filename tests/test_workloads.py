"""The seeded input generators: determinism, shapes, page layout, FP8 scale bound (CPU)."""
import numpy as np

from mla_absorbed_latent_decode_gb300 import workloads as W
from oracle import mla_ref


def test_deterministic_and_chunk_invariant():
    a = W.make_decode("t", 5, 16, [3, 70, 129])
    b = W.make_decode("t", 5, 16, [3, 70, 129])
    for k in ("rows", "q", "w_uk", "w_uv", "block_table"):
        assert np.array_equal(getattr(a, k), getattr(b, k))
    # drawing in chunks gives the same stream as one draw
    r1 = W._normal_bf16(np.random.default_rng(9), (1000, 7), chunk=333)
    r2 = W._normal_bf16(np.random.default_rng(9), (1000, 7), chunk=1 << 30)
    assert np.array_equal(r1, r2)


def test_bf16_rounding_matches_oracle_independently():
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    assert np.array_equal(W.to_bf16_bits(x), mla_ref.bf16_round(x))


def test_paged_layout_is_a_permutation():
    wl = W.v2lite_batched()
    assert wl.B == 32 and wl.n_h == 16
    assert wl.ctx_len.min() >= 1 and wl.ctx_len.max() <= 4096
    used = []
    for b in range(wl.B):
        n = (int(wl.ctx_len[b]) + 63) // 64
        used.extend(wl.block_table[b, :n].tolist())
        assert np.all(wl.block_table[b, n:] == -1)
    assert len(used) == len(set(used)) and max(used) < wl.num_pages
    assert used != sorted(used)                                   # shuffled
    assert wl.rows.shape == (wl.total_tokens, 576)
    assert np.array_equal(wl.row_seq[wl.last_row_index()], np.arange(wl.B))
    assert np.array_equal(wl.row_pos[wl.last_row_index()], wl.ctx_len - 1)


def test_fp8_scale_bounds_every_rotated_value():
    wl = W.make_decode("f", 3, 128, [100, 64], cache_dtype=W.CACHE_FP8)
    rows = mla_ref.bf16_to_f64(wl.rows)
    amax = 0.0
    for i in range(rows.shape[0]):
        for pos in (int(wl.row_pos[i]), 12345, 65535):
            amax = max(amax, np.max(np.abs(mla_ref.rope(rows[i, 512:], pos, 10000.0))))
    amax = max(amax, np.max(np.abs(rows[:, :512])))
    assert amax <= wl.fp8_scale * 448.0 * (1 + 1e-6)
    assert wl.fp8_scale * 448.0 <= amax * 1.05


def test_named_shapes_small_draws():
    wl = W.make_decode("v3", 2, 128, [4096, 1])
    assert wl.q.shape == (2, 128, 192) and wl.w_uk.shape == (128, 128, 512)
    assert wl.w_uv.shape == (128, 128, 512)
    w = mla_ref.bf16_to_f64(wl.w_uk)
    assert 0.015 < w.std() < 0.025


def test_prefill_inputs_follow_the_decode_draws():
    """make_prefill keeps make_decode's rows, weights and pages (same seed, same stream) and adds
    the chunk's queries from a second stream: packed in sequence order, deterministic."""
    a = W.make_prefill("p", 9, 16, [130, 5, 64], [30, 5, 1])
    d = W.make_decode("p", 9, 16, [130, 5, 64])
    assert np.array_equal(a.rows, d.rows) and np.array_equal(a.block_table, d.block_table)
    assert np.array_equal(a.w_uk, d.w_uk) and np.array_equal(a.q, d.q)
    p = a.extra["prefill"]
    assert p["q"].shape == (36, 16, 192)
    assert list(p["q_start"]) == [0, 30, 35] and list(p["q_len"]) == [30, 5, 1]
    b = W.make_prefill("p", 9, 16, [130, 5, 64], [30, 5, 1])
    assert np.array_equal(p["q"], b.extra["prefill"]["q"])
    whole = W.make_prefill("p", 9, 16, [130, 5, 64])
    assert list(whole.extra["prefill"]["q_len"]) == [130, 5, 64]


def test_cache_row_bytes():
    assert W.ROW_BYTES == {W.CACHE_BF16: 1152, W.CACHE_FP8: 576, W.CACHE_FP8_BLOCK: 656}
