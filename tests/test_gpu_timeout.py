"""The bounded in-kernel waits.  With MLA_OPT_TEST_STALL on, one copy of the next decode or prefill
call is withheld -- the query-absorb kernel's query copy (1), one cache tile of the first work unit (2), or
one partial-score copy between the two CTAs of that unit (3), one weight box of the prefill's
expansion kernel (4) or one key box of its attention kernel (5) -- so the thread waiting for it has
nothing that will ever complete its barrier: the wait gives up after about a second, the kernel
drains its own copies in flight (for the score exchange: every copy the peer sent it), the step
still finishes, the host reads MLA_CHECK_TIMEOUT from the device check word, and the context stays
usable -- the next step, with the option off, matches the oracle."""
import time

import pytest

from mla_absorbed_latent_decode_gb300 import binding as B
from mla_absorbed_latent_decode_gb300 import workloads as W
from mla_absorbed_latent_decode_gb300.runner import DecodeSession
from tests.mla_cases import BF16_TOL, FP8_TOL, bf16_out_to_f64, compare, oracle_decode_paged, oracle_stored, oracle_values

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cache", [W.CACHE_BF16, W.CACHE_FP8])
@pytest.mark.parametrize("stall", [1, 2, 3])
def test_a_wait_that_never_completes_times_out_and_the_context_survives(stall, cache):
    """(with an FP8 cache: the default FP8-MMA path, whose transposing and RoPE-converting warps
    wait on the withheld tile too)"""
    wl = W.make_decode("stall", 41, 16, [65, 300], cache_dtype=cache)
    # one unit per sequence, so the first unit has the tile 1 that stalls 2 and 3 withhold
    s = DecodeSession(wl, splits=1)
    s.append_rows()
    assert s.status() == 0
    with pytest.raises(B.MlaError, match="MLA_OPT_TEST_STALL"):
        s.mla.set_option(B.MLA_OPT_TEST_STALL, 6)
    s.mla.set_option(B.MLA_OPT_TEST_STALL, stall)
    t0 = time.monotonic()
    s.decode()
    flags = s.status()
    waited = time.monotonic() - t0
    assert flags & B.MLA_CHECK_TIMEOUT, flags
    assert 0.2 < waited < 60.0, waited             # a few bounded waits of ~2e9 clocks each
    s.mla.set_option(B.MLA_OPT_TEST_STALL, 0)
    ref = oracle_decode_paged(wl, oracle_values(wl, oracle_stored(wl)))
    for _ in range(2):
        out = s.decode()
        assert s.status() == 0
        tol = BF16_TOL if cache == W.CACHE_BF16 else FP8_TOL
        rel, err, scale = compare(bf16_out_to_f64(out), ref, tol)
        assert rel <= tol, (rel, err, scale)
    s.close()


@pytest.mark.parametrize("stall", [4, 5])
def test_prefill_wait_that_never_completes_times_out_and_the_context_survives(stall):
    from tests.test_gpu_prefill import _oracle, _prefill
    wl = W.make_prefill("stall_prefill", 43, 16, [300, 129], [40, 129])
    s = DecodeSession(wl)
    s.append_rows()
    assert s.status() == 0
    s.mla.set_option(B.MLA_OPT_TEST_STALL, stall)
    t0 = time.monotonic()
    _prefill(s, wl)
    flags = s.status()
    waited = time.monotonic() - t0
    assert flags & B.MLA_CHECK_TIMEOUT, flags
    assert 0.2 < waited < 60.0, waited
    s.mla.set_option(B.MLA_OPT_TEST_STALL, 0)
    p = wl.extra["prefill"]
    for _ in range(2):
        out = bf16_out_to_f64(_prefill(s, wl))
        assert s.status() == 0
        for b, ref in _oracle(wl).items():
            a, n = int(p["q_start"][b]), int(p["q_len"][b])
            rel, err, scale = compare(out[a:a + n], ref, BF16_TOL)
            assert rel <= BF16_TOL, (b, rel, err, scale)
    s.close()
