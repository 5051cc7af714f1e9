"""The inputs that force the online softmax's lazy rescale do what they claim (CPU only).

For every (query, head) pair they rewrite, the oracle's own scores (fp64, from its cached
values) must stay on a plateau before the pair's tile g >= 1 and jump by more than the
kernels' rescale step inside tile g, so a kernel that follows its lazy-rescale rule must
rescale there; and the construction must touch both tile parities."""
import numpy as np
import pytest

from mla_absorbed_latent_decode_gb300 import workloads as W
from oracle import mla_ref
from tests.mla_cases import (LOG2E, PREFILL_KEY_TILE, RESCALE_STEP, decode_scores_log2, force_decode_rescale,
                             force_prefill_rescale, oracle_stored, oracle_values)


@pytest.mark.parametrize("n_h,dtype", [(16, W.CACHE_BF16), (128, W.CACHE_BF16), (40, W.CACHE_FP8)])
def test_decode_inputs_force_a_rescale_per_head(n_h, dtype):
    wl = W.make_decode("rescale_in", 90 + n_h, n_h, [1000, 300, 129, 65, 1], cache_dtype=dtype)
    forced = force_decode_rescale(wl)
    assert sorted(forced) == [0, 1, 2]                    # every sequence of at least 3 pages
    vals = oracle_values(wl, oracle_stored(wl))
    margin = 0.5
    parities = set()
    for b, g in forced.items():
        x = decode_scores_log2(wl, vals, b)
        assert np.all(g >= 1)
        for h in range(n_h):
            before = x[h, :64 * g[h]].max()
            at = x[h, 64 * g[h]:64 * (g[h] + 1)].max()
            assert at - before > RESCALE_STEP + margin, (b, h, before, at)
            assert x[h].max() == at                       # the jump is the row's maximum
            parities.add(int(g[h]) % 2)
    assert parities == {0, 1}
    assert np.max(np.abs(vals)) < 128.0                   # rows stay of moderate size (a well-posed problem)


@pytest.mark.parametrize("n_h,ctx,ql", [(16, [700, 1100, 64], [8, 4, 64]), (5, [900, 300], [25, 12])])
def test_prefill_inputs_force_a_rescale_per_pair(n_h, ctx, ql):
    wl = W.make_prefill("rescale_pf", 95 + n_h, n_h, ctx, ql)
    forced = force_prefill_rescale(wl)
    assert sorted(forced) == [0, 1]
    vals = oracle_values(wl, oracle_stored(wl))
    assert np.max(np.abs(vals)) < 128.0
    p = wl.extra["prefill"]
    starts = np.concatenate([[0], np.cumsum(wl.ctx_len.astype(np.int64))])
    scale = mla_ref.default_scale(wl.d_nope, wl.d_rope) * LOG2E
    for b, g in forced.items():
        L, n, a = int(wl.ctx_len[b]), int(p["q_len"][b]), int(p["q_start"][b])
        rows = vals[starts[b]:starts[b + 1]]
        for i in range(n):
            qa = mla_ref.absorb_query(mla_ref.bf16_to_f64(p["q"][a + i]), mla_ref.bf16_to_f64(wl.w_uk),
                                      L - n + i, wl.rope_base)
            x = scale * (qa @ rows[:L - n + i + 1].T)
            for h in range(wl.n_h):
                gg = g[i * wl.n_h + h]
                assert gg >= 1
                t0 = PREFILL_KEY_TILE * gg
                assert x[h, t0:t0 + PREFILL_KEY_TILE].max() - x[h, :t0].max() > RESCALE_STEP + 0.5
