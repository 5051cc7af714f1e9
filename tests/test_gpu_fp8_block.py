"""The per-block FP8 cache (656-byte rows: 512 e4m3 latent codes, 4 fp32 block scales, 64
bf16 RoPE values) on the GPU against the oracle: the bytes mla_kv_append writes (codes and
scales bit-exact, RoPE key within one bf16 code at a rounding tie of the fp32 table), and the
decode against the oracle's decode on its own dequantised per-block cache -- ragged lengths,
16 and 128 heads, the V3 B=128 shape at full size; device checks; calls that do not take the
format refuse it."""
import numpy as np
import pytest
import torch

from mla_absorbed_latent_decode_gb300 import binding as B
from mla_absorbed_latent_decode_gb300 import workloads as W
from mla_absorbed_latent_decode_gb300.runner import SENTINEL, DecodeSession
from tests.mla_cases import (BF16_TOL, FP8_TOL, bf16_out_to_f64, compare, gpu_rows, oracle_decode, oracle_stored,
                             oracle_values)

pytestmark = pytest.mark.gpu

RAGGED = [1, 2, 63, 64, 65, 130, 257, 1000, 4097]


def _rope_distance(a, b):
    ua = np.ascontiguousarray(a).view("<u2").astype(np.int64)
    ub = np.ascontiguousarray(b).view("<u2").astype(np.int64)
    same = (ua & 0x8000) == (ub & 0x8000)
    return np.where(same, np.abs((ua & 0x7FFF) - (ub & 0x7FFF)), (ua & 0x7FFF) + (ub & 0x7FFF))


def test_append_writes_the_oracle_bytes():
    wl = W.make_decode("blk_append", 41, 16, RAGGED, cache_dtype=W.CACHE_FP8_BLOCK)
    wl.rows[3, 128:256] = 0                      # an all-zero block
    wl.rows[7, :128] = W.to_bf16_bits(np.full(128, 3.0e4))
    s = DecodeSession(wl, max_position=8192)
    s.append_rows()
    assert s.status() == 0
    cache = s.cache.cpu().numpy()
    got, exp = gpu_rows(wl, cache), oracle_stored(wl)
    assert got.shape[1] == 656
    assert np.array_equal(got[:, :528], exp[:, :528])          # latent codes and block scales
    d = _rope_distance(got[:, 528:], exp[:, 528:])
    assert d.max() <= 1 and np.mean(d == 0) >= 0.999
    written = np.zeros((wl.num_pages, 64), bool)
    written[wl.block_table[wl.row_seq, wl.row_pos // 64], wl.row_pos % 64] = True
    assert np.all(cache[~written] == SENTINEL)
    s.close()


@pytest.mark.parametrize("n_h", [16, 128])
def test_decode_matches_the_oracle(n_h):
    wl = W.make_decode("blk_decode", 42 + n_h, n_h, RAGGED, cache_dtype=W.CACHE_FP8_BLOCK)
    s = DecodeSession(wl)
    s.append_rows()
    out = bf16_out_to_f64(s.decode())
    assert s.status() == 0
    stored = gpu_rows(wl, s.cache.cpu().numpy())               # the codes the GPU decodes
    ref = oracle_decode(wl, oracle_values(wl, stored))
    rel = compare(out, ref, FP8_TOL)[0]
    # the kernel's only roundings past the cache are bf16 ones (converted values, P): the bf16 bar
    assert rel <= BF16_TOL, rel
    s.close()


def test_v3_b128_full_size_sampled():
    """The V3 FP8 shape (B=128, 4096 tokens each) in the per-block format, in bench.py's launch
    configuration; the oracle decodes every 16th sequence."""
    wl = W.EXTRA["v3_b128_s4096_fp8blk"]()
    s = DecodeSession(wl)
    s.prefill()
    rows, seq, pos = s.step_inputs()
    s.append_step(rows, seq, pos)
    out = bf16_out_to_f64(s.decode())
    assert s.status() == 0
    seqs = list(range(0, wl.B, 16))
    ref = oracle_decode(wl, oracle_values(wl, oracle_stored(wl)), seqs=seqs)
    rel = compare(out[seqs], ref, FP8_TOL)[0]
    assert rel <= FP8_TOL, rel
    s.close()


def test_bad_page_zeroes_that_sequence():
    wl = W.make_decode("blk_bad", 45, 16, [300, 200, 90], cache_dtype=W.CACHE_FP8_BLOCK)
    s = DecodeSession(wl)
    s.append_rows()
    good = bf16_out_to_f64(s.decode()).copy()
    bt = wl.block_table.copy()
    bt[1, 2] = wl.num_pages + 3
    s.block_table = torch.from_numpy(bt).to(s.device)
    out = bf16_out_to_f64(s.decode())
    assert s.status() == B.MLA_CHECK_PAGE_ID
    assert np.all(out[1] == 0) and np.array_equal(out[0], good[0]) and np.array_equal(out[2], good[2])
    s.close()


def test_calls_without_the_format_refuse_it():
    wl = W.make_decode("blk_refuse", 46, 16, [10], cache_dtype=W.CACHE_FP8_BLOCK)
    s = DecodeSession(wl)
    dev = s.device
    with pytest.raises(B.MlaError) as e:
        s.mla.expand_kv(s.cache, wl.num_pages, torch.empty(16, dtype=torch.uint8, device=dev))
    assert e.value.status == B.MLA_ERR_UNSUPPORTED
    s.close()
