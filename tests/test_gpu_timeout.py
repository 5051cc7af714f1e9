"""The bounded in-kernel waits.  With MLA_OPT_TEST_STALL on, the query-absorb kernel withholds its
query copy, so the thread waiting for it has nothing that will ever complete its barrier: the
wait gives up after about a second, the step still finishes, the host reads MLA_CHECK_TIMEOUT
from the device check word, and the context stays usable -- the next step, with the option off,
matches the oracle."""
import time

import pytest

from mla_absorbed_latent_decode_gb300 import binding as B
from mla_absorbed_latent_decode_gb300 import workloads as W
from mla_absorbed_latent_decode_gb300.runner import DecodeSession
from tests.mla_cases import BF16_TOL, bf16_out_to_f64, compare, oracle_decode_paged, oracle_stored, oracle_values

pytestmark = pytest.mark.gpu


def test_a_wait_that_never_completes_times_out_and_the_context_survives():
    wl = W.make_decode("stall", 41, 16, [65, 300])
    s = DecodeSession(wl)
    s.append_rows()
    assert s.status() == 0
    with pytest.raises(B.MlaError, match="MLA_OPT_TEST_STALL"):
        s.mla.set_option(B.MLA_OPT_TEST_STALL, 2)
    s.mla.set_option(B.MLA_OPT_TEST_STALL, 1)
    t0 = time.monotonic()
    s.decode()
    flags = s.status()
    waited = time.monotonic() - t0
    assert flags & B.MLA_CHECK_TIMEOUT, flags
    assert 0.2 < waited < 60.0, waited             # one or two bounded waits of ~2e9 clocks each
    s.mla.set_option(B.MLA_OPT_TEST_STALL, 0)
    out = s.decode()
    assert s.status() == 0
    ref = oracle_decode_paged(wl, oracle_values(wl, oracle_stored(wl)))
    rel, err, scale = compare(bf16_out_to_f64(out), ref, BF16_TOL)
    assert rel <= BF16_TOL, (rel, err, scale)
    s.close()
