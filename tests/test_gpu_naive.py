"""Standard-mode (naive) decode over the expanded per-head cache: mla_expand_kv and
mla_decode_naive against the oracle's naive path (expanded K = [W_UK c ; k_r], V = W_UV c,
plain softmax attention), against the absorbed GPU decode (the same function), and the
expanded values themselves against float64 products."""
import numpy as np
import pytest
import torch

from mla_absorbed_latent_decode_gb300 import binding as B
from mla_absorbed_latent_decode_gb300 import workloads as W
from mla_absorbed_latent_decode_gb300.runner import DecodeSession
from oracle import mla_ref
from tests.mla_cases import BF16_TOL, bf16_out_to_f64, compare, oracle_decode, oracle_stored, oracle_values

pytestmark = pytest.mark.gpu

RAGGED = [1, 2, 63, 64, 65, 130, 257, 1000]


def _expanded(s, wl):
    kvx = torch.empty((wl.num_pages, wl.page_size, wl.n_h, 320), dtype=torch.bfloat16, device="cuda")
    s.mla.expand_kv(s.cache, wl.num_pages, kvx)
    return kvx


def _naive(s, wl, kvx, ctx_len=None):
    ctx = s.ctx_len if ctx_len is None else ctx_len
    ws = torch.empty(s.mla.decode_naive_workspace_size(wl.B, wl.max_ctx), dtype=torch.uint8, device="cuda")
    out = torch.empty((wl.B, wl.n_h, 128), dtype=torch.bfloat16, device="cuda")
    s.mla.decode_naive(s.q, ctx, wl.max_ctx, s.block_table, kvx, wl.num_pages, ws, out)
    return bf16_out_to_f64(out)


@pytest.mark.parametrize("n_h", [16, 128])
def test_naive_decode_matches_the_oracle_and_the_absorbed_decode(n_h):
    wl = W.make_decode("naive_gpu", 91 + n_h, n_h, RAGGED)
    s = DecodeSession(wl)
    s.append_rows()
    kvx = _expanded(s, wl)
    naive = _naive(s, wl, kvx)
    assert s.status() == 0
    absorbed = bf16_out_to_f64(s.decode())
    vals = oracle_values(wl, oracle_stored(wl))
    ref = oracle_decode(wl, vals, path="naive")
    assert compare(naive, ref, BF16_TOL)[0] <= BF16_TOL
    # two independently rounded paths, each within BF16_TOL of the same function
    assert compare(naive, absorbed, BF16_TOL)[0] <= 2 * BF16_TOL
    s.close()


def test_expanded_values_are_the_products():
    wl = W.make_decode("expand", 93, 16, [130, 5])
    s = DecodeSession(wl)
    s.append_rows()
    kvx = _expanded(s, wl).cpu().view(torch.int16).numpy().view(np.uint16)
    cache = s.cache.cpu().view(torch.int16).numpy().view(np.uint16)
    w_uk, w_uv = mla_ref.bf16_to_f64(wl.w_uk), mla_ref.bf16_to_f64(wl.w_uv)
    for b, t in ((0, 0), (0, 129), (1, 4)):
        page, slot = int(wl.block_table[b, t // 64]), t % 64
        row = cache[page, slot]
        c = mla_ref.bf16_to_f64(row[:512])
        for h in (0, 7, 15):
            got = mla_ref.bf16_to_f64(kvx[page, slot, h])
            # bf16 rounding (2^-8 relative) after a 512-term fp32 sum (first-order bound 512 * 2^-24 * sum |terms|)
            for w, sl in ((w_uk[h], slice(0, 128)), (w_uv[h], slice(192, 320))):
                want = w @ c
                assert np.all(np.abs(got[sl] - want) <= 2.0 ** -8 * np.abs(want) + 2.0 ** -15 * (np.abs(w) @ np.abs(c)))
            assert np.array_equal(kvx[page, slot, h, 128:192], row[512:])        # the cached RoPE key, as is
    s.close()


def test_naive_decode_device_checks_and_fp8_refusal():
    wl = W.make_decode("naive_bad", 95, 16, [100, 200, 70])
    s = DecodeSession(wl)
    s.append_rows()
    kvx = _expanded(s, wl)
    good = _naive(s, wl, kvx)
    ctx = s.ctx_len.clone()
    ctx[1] = 0
    out = _naive(s, wl, kvx, ctx)
    assert s.status() == B.MLA_CHECK_CTX_LEN
    assert np.all(out[1] == 0) and np.array_equal(out[0], good[0]) and np.array_equal(out[2], good[2])
    s.close()
    f8 = DecodeSession(W.make_decode("naive_fp8", 96, 16, [10], cache_dtype=W.CACHE_FP8))
    with pytest.raises(B.MlaError) as e:
        f8.mla.expand_kv(f8.cache, f8.wl.num_pages, torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == B.MLA_ERR_UNSUPPORTED
    f8.close()
