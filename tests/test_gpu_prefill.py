"""Causal prefill in MHA mode (mla_prefill) against the oracle's prefill on the same seeded
inputs: whole prompts and chunks after a cached prefix, ragged lengths that span several
128-query blocks and 128-key tiles with ragged tails, 16 and 128 heads; the last query of a
whole prompt against the absorbed decode of that token; device checks."""
import numpy as np
import pytest
import torch

from mla_absorbed_latent_decode_gb300 import binding as B
from mla_absorbed_latent_decode_gb300 import workloads as W
from mla_absorbed_latent_decode_gb300.runner import DecodeSession, bf16_tensor
from oracle import mla_ref
from tests.mla_cases import (BF16_TOL, FP8_TOL, bf16_out_to_f64, compare, force_prefill_rescale, oracle_stored,
                             oracle_values)

pytestmark = pytest.mark.gpu


def _prefill(s, wl, ctx_len=None, q_len=None, q_start=None, max_q=None):
    p = wl.extra["prefill"]
    dev = s.device
    q = bf16_tensor(p["q"], dev)
    ql = torch.from_numpy((p["q_len"] if q_len is None else q_len).astype(np.int32)).to(dev)
    qs = torch.from_numpy((p["q_start"] if q_start is None else q_start).astype(np.int32)).to(dev)
    ctx = s.ctx_len if ctx_len is None else torch.from_numpy(ctx_len.astype(np.int32)).to(dev)
    ws = torch.empty(s.mla.prefill_workspace_size(wl.B, wl.max_ctx), dtype=torch.uint8, device=dev)
    out = torch.full((q.shape[0], wl.n_h, wl.d_v), float("nan"), dtype=torch.bfloat16, device=dev)
    s.mla.prefill(q, qs, ql, int(max_q or max(1, int(p["q_len"].max()))), ctx, wl.max_ctx, s.block_table, s.cache,
                  wl.num_pages, ws, out)
    return out


def _oracle(wl, seqs=None):
    p = wl.extra["prefill"]
    vals = oracle_values(wl, oracle_stored(wl))
    starts = np.concatenate([[0], np.cumsum(wl.ctx_len.astype(np.int64))])
    w_uk, w_uv = mla_ref.bf16_to_f64(wl.w_uk), mla_ref.bf16_to_f64(wl.w_uv)
    q = mla_ref.bf16_to_f64(p["q"])
    scale = mla_ref.default_scale(wl.d_nope, wl.d_rope)
    ref = {}
    for b in (range(wl.B) if seqs is None else seqs):
        rows = vals[starts[b]:starts[b + 1]]
        L, n = int(wl.ctx_len[b]), int(p["q_len"][b])
        a = int(p["q_start"][b])
        ref[b] = mla_ref.prefill_naive(q[a:a + n], rows[:, :wl.d_c], rows[:, wl.d_c:], w_uk, w_uv, L - n, scale,
                                       wl.rope_base)
    return ref


CASES = {
    "odd_heads_empty_and_single_token_chunks": (5, [1, 200, 77, 130], [1, 0, 77, 129]),
    "single_query_chunks_long_prefix": (16, [700, 4100], [1, 3]),
    "whole_prompts_16h": (16, [1, 64, 127, 128, 129, 300, 515], None),
    "chunks_after_prefix_16h": (16, [200, 300, 64, 700, 5], [37, 300, 1, 129, 5]),
    "whole_prompts_128h": (128, [130, 257], None),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_prefill_matches_the_oracle(case):
    n_h, ctx, ql = CASES[case]
    wl = W.make_prefill("prefill_" + case, 71, n_h, ctx, ql)
    s = DecodeSession(wl)
    s.append_rows()
    out = bf16_out_to_f64(_prefill(s, wl))
    assert s.status() == 0
    p = wl.extra["prefill"]
    for b, ref in _oracle(wl).items():
        a, n = int(p["q_start"][b]), int(p["q_len"][b])
        if n == 0:                                    # an empty chunk: nothing to compare
            continue
        err = compare(out[a:a + n], ref, BF16_TOL)
        assert err[0] <= BF16_TOL, (b, err)
    s.close()


FP8_CASES = {
    "chunks_and_whole_prompts_16h": (16, [1, 200, 515, 130], [1, 77, 515, 129]),
    "whole_prompts_128h": (128, [130, 257], None),
}


@pytest.mark.parametrize("cache", [W.CACHE_FP8, W.CACHE_FP8_BLOCK])
@pytest.mark.parametrize("case", sorted(FP8_CASES))
def test_prefill_over_an_fp8_cache_matches_the_oracle(case, cache):
    """An FP8 cache (one tensor scale, or the per-block format) against the oracle on its own
    dequantised cache: the expansion decodes the codes exactly (times the tensor or block scale)."""
    n_h, ctx, ql = FP8_CASES[case]
    wl = W.make_prefill("prefill8_" + case, 73, n_h, ctx, ql, cache_dtype=cache)
    s = DecodeSession(wl)
    s.append_rows()
    out = bf16_out_to_f64(_prefill(s, wl))
    assert s.status() == 0
    p = wl.extra["prefill"]
    for b, ref in _oracle(wl).items():
        a, n = int(p["q_start"][b]), int(p["q_len"][b])
        err = compare(out[a:a + n], ref, FP8_TOL)
        assert err[0] <= FP8_TOL, (b, err)
    s.close()


def test_last_prefill_row_is_the_decode_of_that_token():
    """A whole prompt's last query is the decode step at ctx_len: the prefill (MHA mode) and the
    absorbed decode are two implementations of the same function."""
    wl = W.make_prefill("prefill_vs_decode", 72, 128, [700, 64, 1000])
    s = DecodeSession(wl)
    s.append_rows()
    out = bf16_out_to_f64(_prefill(s, wl))
    p = wl.extra["prefill"]
    last = p["q_start"] + p["q_len"] - 1
    q_dec = bf16_tensor(np.ascontiguousarray(p["q"][last]), s.device)
    dec = bf16_out_to_f64(s.decode(q=q_dec))
    assert s.status() == 0
    # each side within BF16_TOL of the same function
    assert compare(out[last], dec, BF16_TOL)[0] <= 2 * BF16_TOL
    s.close()


def test_prefill_device_checks():
    wl = W.make_prefill("prefill_bad", 73, 16, [150, 90, 260], [150, 40, 200])
    s = DecodeSession(wl)
    s.append_rows()
    p = wl.extra["prefill"]
    good = bf16_out_to_f64(_prefill(s, wl))
    assert s.status() == 0
    rows = lambda b: slice(int(p["q_start"][b]), int(p["q_start"][b] + p["q_len"][b]))
    # q_len above ctx_len: that sequence's rows are zero, the others unchanged
    ctx = wl.ctx_len.copy()
    ctx[1] = 30
    out = bf16_out_to_f64(_prefill(s, wl, ctx_len=ctx))
    assert s.status() == B.MLA_CHECK_CTX_LEN
    assert np.all(out[rows(1)] == 0)
    assert np.array_equal(out[rows(0)], good[rows(0)]) and np.array_equal(out[rows(2)], good[rows(2)])
    s.close()
    # a page id out of range in the pages a sequence's queries see
    s = DecodeSession(wl)
    s.append_rows()
    bt = wl.block_table.copy()
    bt[2, 1] = wl.num_pages + 5
    s.block_table = torch.from_numpy(bt).to(s.device)
    out = bf16_out_to_f64(_prefill(s, wl))
    assert s.status() == B.MLA_CHECK_PAGE_ID
    assert np.all(out[rows(2)] == 0)
    assert np.array_equal(out[rows(0)], good[rows(0)]) and np.array_equal(out[rows(1)], good[rows(1)])
    s.close()


def test_prefill_argument_errors():
    wl = W.make_prefill("prefill_args", 74, 16, [10])
    s = DecodeSession(wl)
    dev = s.device
    i = torch.zeros(1, dtype=torch.int32, device=dev)
    q = torch.zeros((10, 16, 192), dtype=torch.bfloat16, device=dev)
    out = torch.zeros((10, 16, 128), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(s.mla.prefill_workspace_size(1, 10), dtype=torch.uint8, device=dev)
    with pytest.raises(B.MlaError) as e:
        s.mla.prefill(q, i, i, 11, s.ctx_len, 10, s.block_table, s.cache, wl.num_pages, ws, out)
    assert e.value.status == B.MLA_ERR_INVALID_ARG and "max_q" in e.value.message
    with pytest.raises(B.MlaError) as e:
        s.mla.prefill(q, i, i, 10, s.ctx_len, 10, s.block_table, s.cache, wl.num_pages, ws[:-1], out)
    assert e.value.status == B.MLA_ERR_WORKSPACE
    s.close()


@pytest.mark.parametrize("n_h,ctx,ql", [(16, [700, 1100, 64], [8, 4, 64]), (5, [900, 300], [25, 12])])
def test_prefill_forced_rescale_matches_the_oracle(n_h, ctx, ql):
    """Every (query, head) pair of the long chunks has a score plateau and then, in a key tile
    j >= 1 of its own, a key more than the rescale step above it, so the prefill's running row
    maximum grows and O is re-based there (tests/test_rescale_inputs.py checks the construction)."""
    wl = W.make_prefill("prefill_rescale", 95 + n_h, n_h, ctx, ql)
    forced = force_prefill_rescale(wl)
    assert forced
    s = DecodeSession(wl)
    s.append_rows()
    out = bf16_out_to_f64(_prefill(s, wl))
    assert s.status() == 0
    p = wl.extra["prefill"]
    for b, ref in _oracle(wl).items():
        a, n = int(p["q_start"][b]), int(p["q_len"][b])
        err = compare(out[a:a + n], ref, BF16_TOL)
        assert err[0] <= BF16_TOL, (b, err)
    s.close()
