"""mla_decode on the GPU against the fp64 oracle on the same seeded inputs, at sizes
that span several pages and a ragged tail, plus the bookkeeping and the
invariances the method implies (split count, page order, repeatability)."""
import numpy as np
import pytest
import torch

from mla_absorbed_latent_decode_gb300 import binding as B
from mla_absorbed_latent_decode_gb300 import workloads as W
from mla_absorbed_latent_decode_gb300.runner import DecodeSession
from tests.mla_cases import (BF16_TOL, FP8_TOL, bf16_out_to_f64, compare, force_decode_rescale, oracle_decode,
                             oracle_decode_paged, oracle_stored, oracle_values, tolerance)

pytestmark = pytest.mark.gpu

RAGGED = [1, 2, 63, 64, 65, 130, 257, 1000]


def _run(wl, splits=0, max_position=None):
    s = DecodeSession(wl, splits=splits, max_position=max_position)
    s.append_rows()
    out = s.decode()
    flags = s.status()
    return s, bf16_out_to_f64(out), flags


@pytest.mark.parametrize("n_h", [16, 128, 40])
@pytest.mark.parametrize("dtype", [W.CACHE_BF16, W.CACHE_FP8])
def test_decode_matches_oracle_ragged(n_h, dtype):
    wl = W.make_decode("ragged", 21 + n_h, n_h, RAGGED, cache_dtype=dtype)
    s, out, flags = _run(wl)
    assert flags == 0
    ref = oracle_decode_paged(wl, oracle_values(wl, oracle_stored(wl)))
    rel, err, scale = compare(out, ref, BF16_TOL if dtype == W.CACHE_BF16 else FP8_TOL)
    assert rel <= (BF16_TOL if dtype == W.CACHE_BF16 else FP8_TOL), (rel, err, scale)
    s.close()


def test_naive_and_absorbed_oracles_agree_on_the_gpu_case():
    wl = W.make_decode("naive", 31, 16, [5, 70])
    vals = oracle_values(wl, oracle_stored(wl))
    a = oracle_decode(wl, vals)
    n = oracle_decode(wl, vals, path="naive")
    assert np.max(np.abs(a - n)) < 1e-10
    s, out, _ = _run(wl)
    assert compare(out, n, BF16_TOL)[0] <= BF16_TOL
    s.close()


def _workspace_layout(batch, n_h, max_units):
    al = lambda x: (x + 255) & ~255
    off = {}
    o = 0
    for name, size in (("counters", 256), ("units", 16 * max_units), ("seqs", 8 * batch),
                       ("q_abs", 2 * batch * n_h * 576), ("o_lat", 2 * batch * n_h * 512)):
        off[name] = o
        o = al(o + size)
    return off


def plan_reference(ctx_len, max_ctx, num_pairs, forced=0):
    """The planner's rule restated: per-sequence page counts (a sequence is valid when
    1 <= ctx_len <= max_ctx; page ids are checked later, by the decode kernel), a per-pair
    page target, balanced splits."""
    pages = [(L + 63) // 64 if 1 <= L <= max_ctx else 0 for L in ctx_len]
    pairs = max(1, num_pairs)
    budget = max(pairs, sum(1 for n in pages if n > 0))
    target = max(1, -(-sum(pages) // pairs))
    while sum(-(-n // target) for n in pages if n > 0) > budget:
        target += 1
    units, seqs = [], []
    for b, np_b in enumerate(pages):
        ns = 0 if np_b == 0 else (min(forced, np_b) if forced else -(-np_b // target))
        seqs.append((len(units), ns))
        first = len(units)
        for j in range(ns):
            units.append((b, j * np_b // ns, (j + 1) * np_b // ns, first + j if ns > 1 else -1))
    return units, seqs


@pytest.mark.parametrize("small_heads", [False, True])
@pytest.mark.parametrize("forced", [0, 3])
def test_plan_is_bit_exact(forced, small_heads):
    """The work list against the rule restated.  A wave is one unit per SM pair, or per SM when
    the decode runs one CTA per unit (MLA_OPT_SMALL_HEADS); a bf16 handle of at most 32 heads
    sizes its workspace for the SM wave either way."""
    ctx = [1, 4096, 65, 700, 3000, 64, 129, 2048] * 4
    wl = W.make_decode("plan", 41, 16, ctx)
    s = DecodeSession(wl, splits=forced, small_heads=small_heads)
    s.append_rows()
    s.decode()
    assert s.status() == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    wave = sms if small_heads else sms // 2
    max_units = wl.B * max(1, forced) + sms
    off = _workspace_layout(wl.B, wl.n_h, max_units)
    ws = s.workspace.cpu().numpy()
    n_units = int(ws[off["counters"]:off["counters"] + 4].view(np.int32)[0])
    units = ws[off["units"]:off["units"] + 16 * n_units].view(np.int32).reshape(-1, 4)
    seqs = ws[off["seqs"]:off["seqs"] + 8 * wl.B].view(np.int32).reshape(-1, 2)
    ref_units, ref_seqs = plan_reference(wl.ctx_len.tolist(), wl.max_ctx, wave, forced)
    assert n_units == len(ref_units)
    assert [tuple(u) for u in units.tolist()] == ref_units
    assert [tuple(x) for x in seqs.tolist()] == ref_seqs
    s.close()


@pytest.mark.parametrize("batch,splits", [(256, 0), (257, 0), (300, 3)])
def test_large_batches_match_oracle(batch, splits):
    """Batches of more sequences than SM pairs, short ragged contexts: the planner's page-count
    arrays span several of its passes over the batch, and forced splits (three per sequence of
    three pages or more) number hundreds of partial slots."""
    lens = np.random.default_rng(batch).integers(1, 200, size=batch).tolist()
    wl = W.make_decode("bigbatch", 400 + batch, 16, lens)
    s, out, flags = _run(wl, splits=splits)
    assert flags == 0
    ref = oracle_decode_paged(wl, oracle_values(wl, oracle_stored(wl)))
    rel, err, scale = compare(out, ref, BF16_TOL)
    assert rel <= BF16_TOL, (rel, err, scale)
    s.close()


@pytest.mark.parametrize("n_h,batch", [(16, 13), (32, 20)])
def test_small_head_up_projection_tiles(n_h, batch):
    """With few heads the up-projection takes tiles of 8 sequences (its MMA still multiplies 16
    rows and drops the next tile's); the last tile is partial.  Forced splits route every
    sequence of more than one page through the merge, and a bad page zeroes one sequence of a
    later tile."""
    lens = np.random.default_rng(batch).integers(1, 700, size=batch).tolist()
    wl = W.make_decode("uptiles", 500 + n_h + batch, n_h, lens)
    s, out, flags = _run(wl, splits=3)
    assert flags == 0
    ref = oracle_decode_paged(wl, oracle_values(wl, oracle_stored(wl)))
    rel, err, scale = compare(out, ref, BF16_TOL)
    assert rel <= BF16_TOL, (rel, err, scale)
    bt = s.block_table.clone()
    victim = batch - 2
    bt[victim, 0] = wl.num_pages + 3
    s.mla.decode(s.q, s.ctx_len, wl.max_ctx, bt, s.cache, wl.num_pages, s.workspace, s.out)
    out2 = bf16_out_to_f64(s.out)
    assert s.status() == B.MLA_CHECK_PAGE_ID
    assert np.all(out2[victim] == 0)
    keep = [i for i in range(batch) if i != victim]
    assert np.array_equal(out2[keep], out[keep])
    s.close()


def test_split_count_does_not_change_the_result():
    wl = W.make_decode("split", 51, 128, [3000, 1500, 64, 1])
    outs = []
    for k in (1, 2, 7, 64):
        s, out, flags = _run(wl, splits=k)
        assert flags == 0
        outs.append(out)
        s.close()
    ref = oracle_decode(wl, oracle_values(wl, oracle_stored(wl)))
    for o in outs:
        assert compare(o, ref, BF16_TOL)[0] <= BF16_TOL
        # the split changes only fp32 rounding: a couple of bf16 ulps at most
        assert np.max(np.abs(o - outs[0])) <= 4 * 2.0 ** -8 * np.max(np.abs(outs[0]))


def test_page_order_and_repeat_are_bit_identical():
    ctx = [500, 64, 1234]
    a = W.make_decode("order", 61, 128, ctx, shuffle=True)
    b = W.make_decode("order", 61, 128, ctx, shuffle=False)
    assert not np.array_equal(a.block_table, b.block_table)
    sa, oa, _ = _run(a)
    sb, ob, _ = _run(b)
    assert np.array_equal(oa, ob)
    again = bf16_out_to_f64(sa.decode())
    assert np.array_equal(again, oa)
    sa.close()
    sb.close()


def test_bad_lengths_and_pages_zero_only_their_sequence():
    wl = W.make_decode("badlen", 71, 16, [100, 200, 300, 64])
    s = DecodeSession(wl)
    s.append_rows()
    good = bf16_out_to_f64(s.decode())
    assert s.status() == 0
    ctx = s.ctx_len.clone()
    ctx[1] = 0                                                      # empty context: invalid
    ctx[2] = wl.max_ctx + 1                                         # longer than max_ctx
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


def test_bad_page_in_a_tile_without_splits_zeroes_only_its_sequence():
    """With one unit per sequence the up-projection loads the latent rows before it reads the
    bad-page flags; a bad sequence's rows must still come out as zeros."""
    wl = W.make_decode("badpage1", 77, 16, [100, 200, 300, 64])
    s = DecodeSession(wl, splits=1)
    s.append_rows()
    good = bf16_out_to_f64(s.decode())
    assert s.status() == 0
    ref = oracle_decode_paged(wl, oracle_values(wl, oracle_stored(wl)))
    rel, err, scale = compare(good, ref, BF16_TOL)
    assert rel <= BF16_TOL, (rel, err, scale)
    bt = s.block_table.clone()
    bt[1, 2] = wl.num_pages + 5
    s.mla.decode(s.q, s.ctx_len, wl.max_ctx, bt, s.cache, wl.num_pages, s.workspace, s.out)
    out = bf16_out_to_f64(s.out)
    assert s.status() == B.MLA_CHECK_PAGE_ID
    assert np.all(out[1] == 0)
    assert np.array_equal(out[0], good[0]) and np.array_equal(out[2:], good[2:])
    s.close()


def test_decode_host_argument_errors():
    wl = W.make_decode("args", 81, 16, [10, 20])
    s = DecodeSession(wl)
    with pytest.raises(B.MlaError) as e:
        s.mla.decode(s.q, s.ctx_len, wl.max_ctx, s.block_table, s.cache, wl.num_pages, s.workspace[:16], s.out)
    assert e.value.status == B.MLA_ERR_WORKSPACE
    with pytest.raises(B.MlaError) as e:
        s.mla.decode(s.q, s.ctx_len, 10 ** 6, s.block_table, s.cache, wl.num_pages, s.workspace, s.out)
    assert e.value.status == B.MLA_ERR_INVALID_ARG
    s.close()


RESCALE_LENS = [1000, 700, 300, 129, 65, 1]


@pytest.mark.parametrize("n_h,splits,dtype", [
    (16, 0, W.CACHE_BF16), (16, 3, W.CACHE_BF16), (40, 0, W.CACHE_BF16),
    (128, 0, W.CACHE_BF16), (128, 1, W.CACHE_BF16), (128, 3, W.CACHE_BF16), (128, 64, W.CACHE_BF16),
    (128, 0, W.CACHE_FP8), (24, 2, W.CACHE_FP8_BLOCK),
])
def test_forced_rescale_matches_oracle(n_h, splits, dtype):
    """Every head of every sequence of at least 3 pages has a score plateau, then a row more than
    the rescale step above it in a tile j >= 1 of its own (both tile parities), so the running
    maximum grows inside a unit and O, the row sums and the two tile groups' maxima are re-based
    there (tests/test_rescale_inputs.py checks the construction on the oracle's scores); the
    plateau keeps 13-60 % of the final weight, so a wrong rescale factor shows.  Forced splits
    move the unit boundaries (64: one page per unit, the rescale then happens in the merge)."""
    wl = W.make_decode("rescale", 90 + n_h, n_h, RESCALE_LENS, cache_dtype=dtype)
    forced = force_decode_rescale(wl)
    assert sorted(forced) == [0, 1, 2, 3]
    s, out, flags = _run(wl, splits=splits)
    assert flags == 0
    ref = oracle_decode_paged(wl, oracle_values(wl, oracle_stored(wl)))
    rel, err, scale = compare(out, ref, tolerance(wl))
    assert rel <= tolerance(wl), (rel, err, scale)
    s.close()
