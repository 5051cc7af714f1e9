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
from tests.mla_cases import (BF16_TOL, FP8_TOL, bf16_out_to_f64, compare, oracle_decode_paged, oracle_stored,
                             oracle_values)

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


def test_fixed_scratch_matches_the_oracle():
    """The scratch-array path against the fp64 oracle itself (not only against mla_decode)."""
    wl = W.make_decode("fixed_oracle", 301, 128, RAGGED + [4096])
    s = DecodeSession(wl)
    s.append_rows()
    out = torch.full_like(s.out, float("nan"))
    for _ in range(2):
        s.mla.decode_fixed_scratch(s.q, s.ctx_len, wl.max_ctx, s.block_table, s.cache, wl.num_pages, out, s.stream)
        assert s.status() == 0
        got = bf16_out_to_f64(out)
        ref = oracle_decode_paged(wl, oracle_values(wl, oracle_stored(wl)))
        rel, err, scale = compare(got, ref, BF16_TOL)
        assert rel <= BF16_TOL, (rel, err, scale)
    s.close()


def test_fixed_scratch_limit_is_the_workspace_size():
    """The largest batch the array takes is the one whose mla_decode_workspace_size fits in it: at
    128 heads and max_ctx 4096 that batch is accepted and one more sequence is rejected (short
    contexts, so only the sizing differs from a full step)."""
    max_ctx = 4096
    wl = W.make_decode("fixed_edge", 302, 128, [10] * 40)
    s = DecodeSession(wl, max_position=max_ctx)
    sizes = {b: s.mla.decode_workspace_size(b, max_ctx) for b in range(1, 41)}
    fit = max(b for b, n in sizes.items() if n <= B.MLA_FIXED_SCRATCH_BYTES)
    assert fit < 40 and sizes[fit + 1] > B.MLA_FIXED_SCRATCH_BYTES
    bt = torch.full((wl.B, (max_ctx + 63) // 64), -1, dtype=torch.int32, device=s.device)
    bt[:, :1] = s.block_table[:, :1]
    s.append_rows()
    for batch, ok in ((fit, True), (fit + 1, False)):
        out = torch.zeros((batch, wl.n_h, wl.d_v), dtype=torch.bfloat16, device=s.device)
        args = (s.q[:batch], s.ctx_len[:batch], max_ctx, bt[:batch], s.cache, wl.num_pages, out, s.stream)
        if ok:
            s.mla.decode_fixed_scratch(*args)
            assert s.status() == 0
            ref = bf16_out_to_f64(s.decode()[:batch].clone())
            got = bf16_out_to_f64(out)
            assert compare(got, ref, BF16_TOL)[0] <= BF16_TOL
        else:
            with pytest.raises(B.MlaError) as ei:
                s.mla.decode_fixed_scratch(*args)
            assert ei.value.status == B.MLA_ERR_WORKSPACE
    s.close()
