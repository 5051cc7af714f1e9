"""The decode with heads on the MMAs' N dimension (MLA_OPT_SMALL_HEADS; bf16 cache, n_h <= 32):
one CTA per work unit, S^T = C . Q^T with 64-token M = 64 accumulators, O^T += C^T . P^T over four
128-row latent quarters.  Compared element by element with the fp64 oracle on ragged lengths
(partial last pages, 1-token sequences), forced split counts (the partials and their log-sum-exps
the merge reads), inputs that force the online softmax's rescale, bad lengths and page ids, the
bounded waits, and the full V2-Lite batch; and against the 128-row layout of the same inputs."""
import time

import numpy as np
import pytest

from mla_absorbed_latent_decode_gb300 import binding as B
from mla_absorbed_latent_decode_gb300 import workloads as W
from mla_absorbed_latent_decode_gb300.runner import DecodeSession
from tests.mla_cases import (BF16_TOL, bf16_out_to_f64, compare, force_decode_rescale, oracle_decode,
                             oracle_decode_paged, oracle_stored, oracle_values)

pytestmark = pytest.mark.gpu

RAGGED = [1, 2, 63, 64, 65, 130, 257, 1000]


def _run(wl, splits=0, small_heads=True):
    s = DecodeSession(wl, splits=splits, small_heads=small_heads)
    s.append_rows()
    out = bf16_out_to_f64(s.decode())
    return s, out, s.status()


@pytest.mark.parametrize("n_h", [16, 24, 32, 5])
def test_small_heads_match_oracle_ragged(n_h):
    wl = W.make_decode("sh_ragged", 210 + n_h, n_h, RAGGED)
    s, out, flags = _run(wl)
    assert flags == 0
    ref = oracle_decode_paged(wl, oracle_values(wl, oracle_stored(wl)))
    rel, err, scale = compare(out, ref, BF16_TOL)
    assert rel <= BF16_TOL, (rel, err, scale)
    s.close()


def test_small_heads_split_counts():
    """Forced splits write fp32 partials and log-sum-exps for the merge; the split only changes
    fp32 rounding."""
    wl = W.make_decode("sh_split", 251, 16, [3000, 1500, 64, 1])
    ref = oracle_decode(wl, oracle_values(wl, oracle_stored(wl)))
    outs = []
    for k in (1, 2, 7, 64):
        s, out, flags = _run(wl, splits=k)
        assert flags == 0
        rel, err, scale = compare(out, ref, BF16_TOL)
        assert rel <= BF16_TOL, (k, rel, err, scale)
        outs.append(out)
        s.close()
    for o in outs:
        assert np.max(np.abs(o - outs[0])) <= 4 * 2.0 ** -8 * np.max(np.abs(outs[0]))


@pytest.mark.parametrize("n_h,splits", [(16, 0), (16, 3), (32, 0), (32, 64)])
def test_small_heads_forced_rescale(n_h, splits):
    """Every head of every sequence of at least 3 pages rescales at a tile of its own, so the
    per-head running maximum grows inside a unit and O^T's columns are re-based there."""
    wl = W.make_decode("sh_rescale", 290 + n_h, n_h, [1000, 700, 300, 129, 65, 1])
    assert sorted(force_decode_rescale(wl)) == [0, 1, 2, 3]
    s, out, flags = _run(wl, splits=splits)
    assert flags == 0
    ref = oracle_decode_paged(wl, oracle_values(wl, oracle_stored(wl)))
    rel, err, scale = compare(out, ref, BF16_TOL)
    assert rel <= BF16_TOL, (rel, err, scale)
    s.close()


def test_small_heads_agree_with_the_128_row_layout():
    wl = W.make_decode("sh_ab", 261, 16, [4096, 700, 129, 64, 3])
    a, out_a, fa = _run(wl, small_heads=True)
    b, out_b, fb = _run(wl, small_heads=False)
    assert fa == 0 and fb == 0
    assert np.max(np.abs(out_a - out_b)) <= 4 * 2.0 ** -8 * np.max(np.abs(out_b))
    a.close()
    b.close()


def test_small_heads_bad_lengths_and_pages_zero_only_their_sequence():
    wl = W.make_decode("sh_bad", 271, 16, [100, 200, 300, 64])
    s, good, flags = _run(wl)
    assert flags == 0
    ctx = s.ctx_len.clone()
    ctx[1] = 0
    ctx[2] = wl.max_ctx + 1
    s.mla.decode(s.q, ctx, wl.max_ctx, s.block_table, s.cache, wl.num_pages, s.workspace, s.out)
    out = bf16_out_to_f64(s.out)
    assert s.status() == B.MLA_CHECK_CTX_LEN
    assert np.all(out[1] == 0) and np.all(out[2] == 0)
    assert np.array_equal(out[0], good[0]) and np.array_equal(out[3], good[3])
    bt = s.block_table.clone()
    bt[3, 0] = -7
    s.mla.decode(s.q, s.ctx_len, wl.max_ctx, bt, s.cache, wl.num_pages, s.workspace, s.out)
    out = bf16_out_to_f64(s.out)
    assert s.status() == B.MLA_CHECK_PAGE_ID
    assert np.all(out[3] == 0) and np.array_equal(out[:3], good[:3])
    s.close()


def test_small_heads_wait_that_never_completes_times_out():
    wl = W.make_decode("sh_stall", 241, 16, [65, 300])
    s = DecodeSession(wl, splits=1, small_heads=True)
    s.append_rows()
    assert s.status() == 0
    s.mla.set_option(B.MLA_OPT_TEST_STALL, 2)              # the first unit never loads its tile 1
    t0 = time.monotonic()
    s.decode()
    flags = s.status()
    waited = time.monotonic() - t0
    assert flags & B.MLA_CHECK_TIMEOUT, flags
    assert 0.2 < waited < 60.0, waited
    s.mla.set_option(B.MLA_OPT_TEST_STALL, 0)
    ref = oracle_decode_paged(wl, oracle_values(wl, oracle_stored(wl)))
    for _ in range(2):
        out = bf16_out_to_f64(s.decode())
        assert s.status() == 0
        rel, err, scale = compare(out, ref, BF16_TOL)
        assert rel <= BF16_TOL, (rel, err, scale)
    s.close()


def test_small_heads_v2lite_batch():
    """The V2-Lite ragged batch (32 sequences of 1-4096 tokens, 16 heads) at full size."""
    wl = W.NAMED["v2lite_b32_ragged"]()
    s = DecodeSession(wl, small_heads=True)
    s.prefill()
    s.append_step(*s.step_inputs())
    out = bf16_out_to_f64(s.decode())
    assert s.status() == 0
    ref = oracle_decode(wl, oracle_values(wl, oracle_stored(wl)))
    rel, err, scale = compare(out, ref, BF16_TOL)
    assert rel <= BF16_TOL, (rel, err, scale)
    s.close()
