"""The FP8 tensor-core decode's own rounding, emulated in fp64 on the oracle's values, against the
oracle: the budget that the GPU's FP8-MMA parity tests then hold.

The pages fix the FP8 cache (e4m3 codes with one tensor scale) but not how an FP8 contraction
rounds its other operands.  The reading taken: each CTA half's 256 latent query values of a head
share one scale s = max|q| / 448 and become e4m3(q / s); that half's 32 RoPE query values stay
bf16, divided by s, so both parts accumulate into one fp32 score that is multiplied by s
afterwards; P (at most 2^8 after the lazy rescale) is rounded to e4m3 without a scale for P . C,
while the running sum uses the unrounded P.  The emulation below follows those steps in fp64 (a
plain online softmax over 64-token tiles, the same lazy rescale threshold) and must land within
the FP8 tolerance of the exact absorbed decode, with margin, on N(0,1) inputs and on inputs that
force the rescale.  Two controls: with neither FP8 rounding the emulation reproduces the oracle to
the bf16 rounding of the stored query (so its own online softmax adds nothing), and the FP8
roundings are visible above that.  (On N(0,1) inputs the error is mostly P's rounding, the
softmax being flat; where the rescale is forced it is mostly the query's.)"""
import numpy as np
import pytest

from mla_absorbed_latent_decode_gb300 import workloads as W
from oracle import e4m3, mla_ref
from tests.mla_cases import BF16_TOL, FP8_TOL, LOG2E, force_decode_rescale, oracle_decode, oracle_stored, oracle_values

RESCALE_STEP = 8.0      # log2 units the running maximum must be exceeded by before O is re-based


def _bf16(x):
    return mla_ref.bf16_to_f64(mla_ref.bf16_round(np.asarray(x, np.float32)))


def _e4m3(x):
    return e4m3.decode(e4m3.encode(x))


def emulate(wl, values, round_q=True, round_p=True):
    """Decode every sequence with the FP8-MMA arithmetic reading; returns [B, n_h, d_v].  With
    round_q / round_p False the query's latent part (bf16) / P stays unrounded."""
    starts = np.concatenate([[0], np.cumsum(wl.ctx_len.astype(np.int64))])
    q = mla_ref.bf16_to_f64(wl.q)
    w_uk = mla_ref.bf16_to_f64(wl.w_uk)
    w_uv = mla_ref.bf16_to_f64(wl.w_uv)
    scale = mla_ref.default_scale(wl.d_nope, wl.d_rope) * LOG2E
    half_c, half_r = wl.d_c // 2, wl.d_rope // 2
    out = []
    for b in range(wl.B):
        n = int(wl.ctx_len[b])
        rows = values[starts[b]:starts[b + 1]]
        qa = _bf16(mla_ref.absorb_query(q[b], w_uk, n - 1, wl.rope_base))     # the absorbed query, bf16
        x = np.zeros((wl.n_h, n))
        for r in range(2):                                                   # the two CTA halves
            lat = qa[:, half_c * r:half_c * (r + 1)]
            rope = qa[:, wl.d_c + half_r * r:wl.d_c + half_r * (r + 1)]
            amax = np.max(np.abs(lat), axis=1, keepdims=True)
            s = np.where(amax > 0, amax / 448.0, 1.0) if round_q else np.ones_like(amax)
            part = ((_e4m3(lat / s) if round_q else lat) @ rows[:, half_c * r:half_c * (r + 1)].T
                    + (_bf16(rope / s) if round_q else rope) @ rows[:, wl.d_c + half_r * r:wl.d_c + half_r * (r + 1)].T)
            x += s * part * scale
        m = np.full(wl.n_h, -np.inf)
        l = np.zeros(wl.n_h)
        o = np.zeros((wl.n_h, wl.d_c))
        for t0 in range(0, n, 64):
            xt = x[:, t0:t0 + 64]
            mt = xt.max(axis=1)
            m_new = np.where(mt > m + RESCALE_STEP, mt, m)
            alpha = np.where(np.isfinite(m), np.exp2(m - m_new), 0.0)
            o *= alpha[:, None]
            l *= alpha
            m = m_new
            p = np.exp2(xt - m[:, None])
            l += p.sum(axis=1)
            o += (_e4m3(p) if round_p else p) @ rows[t0:t0 + 64, :wl.d_c]
        out.append(mla_ref.up_project(o / l[:, None], w_uv))
    return np.stack(out)


@pytest.mark.parametrize("n_h", [16, 128])
@pytest.mark.parametrize("forced", [False, True])
def test_fp8_mma_reading_is_within_the_fp8_tolerance(n_h, forced):
    wl = W.make_decode("fp8read", 9 + n_h, n_h, [1000, 300, 129, 65], cache_dtype=W.CACHE_FP8)
    if forced:
        assert sorted(force_decode_rescale(wl)) == [0, 1, 2]
    vals = oracle_values(wl, oracle_stored(wl))
    ref = oracle_decode(wl, vals)
    scale = np.max(np.abs(ref))
    err = np.max(np.abs(emulate(wl, vals) - ref)) / scale
    assert err <= 0.7 * FP8_TOL, err
    err_none = np.max(np.abs(emulate(wl, vals, round_q=False, round_p=False) - ref)) / scale
    assert err_none <= BF16_TOL / 4, err_none
    assert err >= 2 * err_none, (err, err_none)
