"""The five decode configurations at full size on the GPU against the fp64 oracle.

Every output of every configuration is compared (the oracle's absorbed path is
a few BLAS calls per sequence).  Tolerance: max |gpu - ref| <= tau * max |ref|
over the whole output, tau = 1e-2 for a bf16 cache and 5e-2 for an FP8 cache
(the oracle then runs on its own dequantised e4m3 cache).  The launch
configuration is the one bench.py times (planner-chosen splits)."""
import numpy as np
import pytest

from mla_absorbed_latent_decode_gb300 import workloads as W
from mla_absorbed_latent_decode_gb300.runner import DecodeSession
from oracle import mla_ref
from tests.mla_cases import (bf16_out_to_f64, compare, gpu_rows, oracle_decode, oracle_stored,
                             oracle_values, tolerance)

pytestmark = pytest.mark.gpu


def _check(wl, check_codes=True, fp8_mma=None):
    s = DecodeSession(wl, fp8_mma=fp8_mma)
    s.prefill()
    rows, seq, pos = s.step_inputs()
    s.append_step(rows, seq, pos)                       # the decode token's own row, as in a step
    out = bf16_out_to_f64(s.decode())
    assert s.status() == 0
    stored = oracle_stored(wl)
    if check_codes:
        got = gpu_rows(wl, s.cache.cpu().numpy())
        assert np.array_equal(got[:, :512], stored[:, :512])
    ref = oracle_decode(wl, oracle_values(wl, stored))
    rel, err, scale = compare(out, ref, tolerance(wl))
    s.close()
    return rel, err, scale


def test_v2lite_single_step_26_tokens():
    """DeepSeek-V2-Lite layer shapes: a 25-token prefill, then one decode token (s_ctx = 26).
    The caller-side projections W_DKV x and W_Q x are done here in float64 and rounded to bf16."""
    inp = W.v2lite_single_step_inputs(seed=0)
    x = mla_ref.bf16_to_f64(inp["x"])
    c, kr, q = mla_ref.project_inputs(x, mla_ref.bf16_to_f64(inp["w_dkv"]), mla_ref.bf16_to_f64(inp["w_q"]),
                                      16, 512)
    rows = mla_ref.bf16_round(np.concatenate([c, kr], axis=1).astype(np.float32))
    qb = mla_ref.bf16_round(q[-1].astype(np.float32))
    wl = W.v2lite_single_step(rows, qb, inp["w_uk"], inp["w_uv"])
    rel, err, scale = _check(wl)
    assert rel <= tolerance(wl), (rel, err, scale)
    # the GPU step also agrees with the one-shot fp64 forward of the same layer (bf16 inputs aside)
    full = mla_ref.causal_forward_naive(x, mla_ref.bf16_to_f64(inp["w_dkv"]), mla_ref.bf16_to_f64(inp["w_q"]),
                                        mla_ref.bf16_to_f64(inp["w_uk"]), mla_ref.bf16_to_f64(inp["w_uv"]),
                                        mla_ref.default_scale(128, 64), 10000.0)
    s = DecodeSession(wl)
    s.append_rows()
    out = bf16_out_to_f64(s.decode())[0]
    s.close()
    assert np.max(np.abs(out - full[-1])) <= 2e-2 * np.max(np.abs(full[-1]))


@pytest.mark.parametrize("name", ["v2lite_b32_ragged", "v3_b64_s4096_bf16", "v3_b128_s4096_fp8", "v3_b8_long"])
def test_named_config(name):
    wl = W.NAMED[name]()
    rel, err, scale = _check(wl)
    assert rel <= tolerance(wl), (name, rel, err, scale)


def test_fp8_config_with_bf16_conversion():
    """The V3 B=128 x 4096 per-tensor FP8 configuration on the other FP8 path (MLA_OPT_FP8_MMA = 0:
    codes converted to bf16 in shared memory, bf16 contractions); the default, FP8 MMAs, is
    test_named_config's."""
    wl = W.NAMED["v3_b128_s4096_fp8"]()
    rel, err, scale = _check(wl, fp8_mma=False)
    assert rel <= tolerance(wl), (rel, err, scale)
