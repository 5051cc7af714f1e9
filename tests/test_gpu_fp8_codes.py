"""Every finite e4m3 code through the FP8 decode path, exactly.

A one-token context makes the softmax weight exactly 1, so the normalised latent
sum is the stored row itself (the code times the tensor scale, here 1); a 0/1
W_UV that routes latent column (h * 128 + v) % 512 to output value v of head h
then prints that row back, bit for bit, through kv_append's encoder, the decode
kernel's in-shared-memory e4m3 -> bf16 conversion, and the up-projection.  The
values are fixed by the e4m3 format itself (OCP: bias 7, no infinities, 0x7F and
0xFF are NaN), not by any code of the library."""
import numpy as np
import pytest

from mla_absorbed_latent_decode_gb300 import workloads as W
from mla_absorbed_latent_decode_gb300.runner import DecodeSession
from tests.mla_cases import bf16_out_to_f64

pytestmark = pytest.mark.gpu


def e4m3_value(code: int) -> float:
    """The value of an e4m3 code from the format's definition (NaN codes excluded by the caller)."""
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 0:
        return sign * m * 2.0 ** -9                      # subnormal: m / 8 * 2^(1 - 7)
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def _workload():
    n_h = 16
    codes = [c for c in range(256) if c not in (0x7F, 0xFF)]
    vals = np.array([e4m3_value(c) for c in codes], dtype=np.float64)
    latent = vals[np.arange(W.D_C) % len(vals)]
    row = np.concatenate([latent, np.zeros(W.D_ROPE)])
    rows = W.to_bf16_bits(row)[None, :]
    assert np.array_equal(W.bf16_bits_to_f32(rows[0, :W.D_C]).astype(np.float64), latent)   # exact in bf16
    w_uv = np.zeros((n_h, W.D_V, W.D_C))
    for h in range(n_h):
        for v in range(W.D_V):
            w_uv[h, v, (h * W.D_V + v) % W.D_C] = 1.0
    wl = W.Workload(
        name="fp8_codes", n_h=n_h, B=1, ctx_len=np.array([1], dtype=np.int32),
        block_table=np.array([[1]], dtype=np.int32), num_pages=2,
        w_uk=W.to_bf16_bits(np.zeros((n_h, W.D_NOPE, W.D_C))), w_uv=W.to_bf16_bits(w_uv),
        q=W.to_bf16_bits(np.zeros((1, n_h, W.D_NOPE + W.D_ROPE))), rows=rows,
        row_seq=np.array([0], dtype=np.int32), row_pos=np.array([0], dtype=np.int32),
        cache_dtype=W.CACHE_FP8, fp8_scale=1.0, seed=0)
    return wl, latent


def test_every_finite_e4m3_code_decodes_exactly():
    wl, latent = _workload()
    s = DecodeSession(wl)
    s.append_rows()
    out = bf16_out_to_f64(s.decode())
    assert s.status() == 0
    got = out[0, :4].reshape(-1)                          # heads 0..3 cover latent columns 0..511
    want = latent[np.arange(4 * W.D_V) % W.D_C]
    assert np.array_equal(got, want), np.flatnonzero(got != want)[:8]
    s.close()
