"""mla_decode_fixed_scratch (the decode step with the library's own fixed scratch array)
against mla_decode with a caller workspace, on the same inputs, two calls in a row.

Collected last on purpose: the fixed array is shared by every call on the device, so this
file also shows that whatever earlier tests left in it does not matter."""
import numpy as np
import pytest
import torch

from mla_absorbed_latent_decode_gb300 import binding as B
from mla_absorbed_latent_decode_gb300 import workloads as W
from mla_absorbed_latent_decode_gb300.runner import DecodeSession, bf16_tensor
from tests.mla_cases import BF16_TOL, FP8_TOL, bf16_out_to_f64, compare

pytestmark = pytest.mark.gpu

RAGGED = [1, 2, 63, 64, 65, 130, 257, 1000]


def _second_query(wl, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((wl.B, wl.n_h, 192)).astype(np.float32)
    return W.to_bf16_bits(q)


@pytest.mark.parametrize("n_h,lengths,dtype", [
    (16, RAGGED, W.CACHE_BF16),
    (128, RAGGED, W.CACHE_BF16),
    (128, [4096] * 4 + [3001] * 4, W.CACHE_BF16),
    (40, RAGGED, W.CACHE_FP8),
    (24, RAGGED, W.CACHE_FP8_BLOCK),
])
def test_fixed_scratch_matches_workspace_decode(n_h, lengths, dtype):
    wl = W.make_decode("fixed", 77 + n_h, n_h, lengths, cache_dtype=dtype)
    s = DecodeSession(wl)
    s.append_rows()
    tol = BF16_TOL if dtype != W.CACHE_FP8 else FP8_TOL
    queries = [s.q, bf16_tensor(_second_query(wl, 1234 + n_h), s.device)]
    for q in queries:                                     # two calls in a row, different inputs
        ref = bf16_out_to_f64(s.decode(q=q).clone())
        out = torch.full_like(s.out, float("nan"))
        s.mla.decode_fixed_scratch(q, s.ctx_len, wl.max_ctx, s.block_table, s.cache, wl.num_pages, out,
                                   s.stream)
        got = bf16_out_to_f64(out)
        assert np.all(np.isfinite(got))
        rel, err, scale = compare(got, ref, tol)
        assert rel <= tol, (rel, err, scale)
    assert s.status() == 0
    s.close()


def test_fixed_scratch_rejects_a_batch_beyond_its_size():
    wl = W.make_decode("fixed_big", 5, 128, [4096] * 26)   # split partials for 26 + 76 units: > 32 MiB
    s = DecodeSession(wl)
    need = s.mla.decode_workspace_size(wl.B, wl.max_ctx)
    assert need > B.MLA_FIXED_SCRATCH_BYTES
    out = torch.zeros_like(s.out)
    with pytest.raises(B.MlaError) as ei:
        s.mla.decode_fixed_scratch(s.q, s.ctx_len, wl.max_ctx, s.block_table, s.cache, wl.num_pages, out,
                                   s.stream)
    assert "MLA_ERR_WORKSPACE" in str(ei.value) and "fixed" in str(ei.value)
    torch.cuda.synchronize()
    assert not torch.any(out.view(torch.int16) != 0)      # nothing was enqueued
    s.close()
