"""mla_kv_append on the GPU against the oracle's stored rows: slot addressing and
latent codes bit-exact, RoPE-key codes equal (within one code at a rounding tie
of the fp32 table), untouched slots untouched, bad indices flagged not written."""
import numpy as np
import pytest
import torch

from mla_absorbed_latent_decode_gb300 import binding as B
from mla_absorbed_latent_decode_gb300 import workloads as W
from mla_absorbed_latent_decode_gb300.runner import SENTINEL, DecodeSession, bf16_tensor
from tests.mla_cases import gpu_rows, oracle_stored

pytestmark = pytest.mark.gpu

LENGTHS = [1, 63, 64, 65, 200, 4097]


def _code_distance(a, b, fp8):
    """|a - b| in units of the code's magnitude ordering (same sign assumed for near values)."""
    if fp8:
        ma, mb = (a & 0x7F).astype(np.int64), (b & 0x7F).astype(np.int64)
        same = (a & 0x80) == (b & 0x80)
    else:
        ma, mb = (a & 0x7FFF).astype(np.int64), (b & 0x7FFF).astype(np.int64)
        same = (a & 0x8000) == (b & 0x8000)
    d = np.abs(ma - mb)
    return np.where(same, d, ma + mb)


@pytest.mark.parametrize("dtype", [W.CACHE_BF16, W.CACHE_FP8])
def test_append_matches_oracle(dtype):
    wl = W.make_decode("append", 11, 16, LENGTHS, cache_dtype=dtype)
    s = DecodeSession(wl, max_position=8192)
    s.append_rows()
    assert s.status() == 0
    cache = s.cache.cpu().numpy()
    got = gpu_rows(wl, cache)
    exp = oracle_stored(wl)
    assert np.array_equal(got[:, :512], exp[:, :512])               # latent: exact copy / exact encode
    d = _code_distance(got[:, 512:], exp[:, 512:], dtype == W.CACHE_FP8)
    assert d.max() <= 1
    assert np.mean(d == 0) >= 0.999
    # every slot not named by a row still holds the fill pattern
    written = np.zeros((wl.num_pages, 64), bool)
    pages = wl.block_table[wl.row_seq, wl.row_pos // 64]
    written[pages, wl.row_pos % 64] = True
    assert np.all(cache[~written] == SENTINEL)
    s.close()


def test_append_positions_rotate_only_the_key():
    """Position 0 stores the row unchanged (RoPE at 0 is the identity)."""
    wl = W.make_decode("pos0", 12, 16, [1, 1, 1])
    s = DecodeSession(wl)
    s.append_rows()
    got = gpu_rows(wl, s.cache.cpu().numpy())
    assert np.array_equal(got, wl.rows)
    s.close()


def test_append_bad_indices_are_flagged_and_skipped():
    wl = W.make_decode("bad", 13, 16, [70, 10])
    s = DecodeSession(wl, max_position=128)
    dev = s.device
    rows = bf16_tensor(wl.rows[:4], dev)
    bt = s.block_table.clone()
    bt[1, 0] = wl.num_pages + 5                                      # bad page id for sequence 1
    cases = [
        ([5, 0], [0, 0], B.MLA_CHECK_APPEND_INDEX),                 # seq out of range
        ([0, 0], [128, 1], B.MLA_CHECK_APPEND_INDEX),               # pos >= max_position
        ([0, 0], [-1, 2], B.MLA_CHECK_APPEND_INDEX),                # negative pos
        ([1, 0], [3, 4], B.MLA_CHECK_PAGE_ID),                      # page id out of range
    ]
    for seq, pos, flag in cases:
        before = s.cache.clone()
        sq = torch.tensor(seq, dtype=torch.int32, device=dev)
        ps = torch.tensor(pos, dtype=torch.int32, device=dev)
        s.mla.kv_append(rows[:2], sq, ps, bt, s.cache, wl.num_pages)
        assert s.status() & flag
        changed = (s.cache != before).reshape(wl.num_pages * 64, -1).any(1).nonzero().flatten().tolist()
        # only the good row (second) may have been written
        good_page = int(bt[seq[1], pos[1] // 64])
        assert set(changed) <= {good_page * 64 + pos[1] % 64}
    assert s.status() == 0                                          # the word is cleared by reading it
    s.close()


def test_append_host_argument_errors():
    wl = W.make_decode("args", 14, 16, [5])
    s = DecodeSession(wl)
    rows, seq, pos = s.step_inputs()
    with pytest.raises(B.MlaError) as e:
        s.mla.kv_append(rows, seq, pos, s.block_table, s.cache, 0)
    assert e.value.status == B.MLA_ERR_INVALID_ARG
    s.mla.kv_append(rows[:0], seq[:0], pos[:0], s.block_table, s.cache, wl.num_pages)   # n = 0 is a no-op
    s.close()
