"""The decode with FP8 tensor-core contractions (MLA_OPT_FP8_MMA, per-tensor e4m3 cache).

QK^T reads the cached e4m3 codes as stored against the absorbed query quantised to e4m3 (one scale
per head and half of the latent columns; the RoPE part stays bf16); P . C reads P in e4m3 against
a token-contiguous copy of the tile's codes.  Compared element by element with the fp64 oracle on
its own dequantised cache at the FP8 tolerance (5e-2 of max |ref|), on ragged lengths (partial last
pages, 1-token sequences), forced split counts and inputs that force the online softmax's rescale."""
import numpy as np
import pytest

from mla_absorbed_latent_decode_gb300 import binding as B
from mla_absorbed_latent_decode_gb300 import workloads as W
from mla_absorbed_latent_decode_gb300.runner import DecodeSession
from tests.mla_cases import (FP8_TOL, bf16_out_to_f64, compare, force_decode_rescale, oracle_decode,
                             oracle_decode_paged, oracle_stored, oracle_values)

pytestmark = pytest.mark.gpu

RAGGED = [1, 2, 63, 64, 65, 130, 257, 1000]


def _run(wl, splits=0, fp8_mma=True):
    s = DecodeSession(wl, splits=splits, fp8_mma=fp8_mma)
    s.append_rows()
    out = bf16_out_to_f64(s.decode())
    return s, out, s.status()


@pytest.mark.parametrize("n_h", [16, 40, 128])
def test_fp8_mma_matches_oracle_ragged(n_h):
    wl = W.make_decode("fp8mma", 61 + n_h, n_h, RAGGED, cache_dtype=W.CACHE_FP8)
    s, out, flags = _run(wl)
    assert flags == 0
    ref = oracle_decode_paged(wl, oracle_values(wl, oracle_stored(wl)))
    rel, err, scale = compare(out, ref, FP8_TOL)
    assert rel <= FP8_TOL, (rel, err, scale)
    s.close()


@pytest.mark.parametrize("splits", [1, 3, 64])
def test_fp8_mma_split_counts(splits):
    wl = W.make_decode("fp8mmasplit", 91, 128, [4096, 700, 129, 64], cache_dtype=W.CACHE_FP8)
    s, out, flags = _run(wl, splits=splits)
    assert flags == 0
    ref = oracle_decode(wl, oracle_values(wl, oracle_stored(wl)))
    rel, err, scale = compare(out, ref, FP8_TOL)
    assert rel <= FP8_TOL, (splits, rel, err, scale)
    s.close()


@pytest.mark.parametrize("n_h", [16, 128])
def test_fp8_mma_forced_rescale(n_h):
    wl = W.make_decode("fp8mmar", 71 + n_h, n_h, [1000, 700, 300, 129, 65, 1], cache_dtype=W.CACHE_FP8)
    forced = force_decode_rescale(wl)
    assert sorted(forced) == [0, 1, 2, 3]
    s, out, flags = _run(wl)
    assert flags == 0
    ref = oracle_decode(wl, oracle_values(wl, oracle_stored(wl)))
    rel, err, scale = compare(out, ref, FP8_TOL)
    assert rel <= FP8_TOL, (rel, err, scale)
    s.close()


@pytest.mark.parametrize("n_h", [16, 128])
def test_conversion_path_matches_oracle_ragged(n_h):
    """The other FP8 path (MLA_OPT_FP8_MMA = 0: codes converted to bf16 in shared memory)."""
    wl = W.make_decode("fp8conv", 63 + n_h, n_h, RAGGED, cache_dtype=W.CACHE_FP8)
    s, out, flags = _run(wl, fp8_mma=False)
    assert flags == 0
    ref = oracle_decode_paged(wl, oracle_values(wl, oracle_stored(wl)))
    rel, err, scale = compare(out, ref, FP8_TOL)
    assert rel <= FP8_TOL, (rel, err, scale)
    s.close()


def test_fp8_mma_and_conversion_paths_agree():
    """The two FP8 paths differ only by the e4m3 rounding of the query and of P."""
    wl = W.make_decode("fp8mmaab", 97, 128, [3000, 64, 257], cache_dtype=W.CACHE_FP8)
    s8, out8, f8 = _run(wl, fp8_mma=True)
    s16, out16, f16 = _run(wl, fp8_mma=False)
    assert f8 == 0 and f16 == 0
    rel, err, scale = compare(out8, out16, FP8_TOL)
    assert rel <= FP8_TOL, (rel, err, scale)
    assert not np.array_equal(out8, out16)       # the option does change the arithmetic
    s8.close()
    s16.close()


def test_fp8_mma_option_values():
    wl = W.make_decode("fp8mmaopt", 5, 16, [10], cache_dtype=W.CACHE_FP8)
    s = DecodeSession(wl)
    with pytest.raises(B.MlaError, match="MLA_OPT_FP8_MMA"):
        s.mla.set_option(B.MLA_OPT_FP8_MMA, 2)
    s.mla.set_option(B.MLA_OPT_FP8_MMA, 1)
    s.mla.set_option(B.MLA_OPT_FP8_MMA, 0)
    s.close()
