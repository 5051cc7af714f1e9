"""The oracle's e4m3 / bf16 codecs and stored-row values against independent definitions (CPU)."""
import numpy as np
import pytest
import torch

from oracle import e4m3, mla_ref
from tests.conftest import load_golden


def test_e4m3_codebook_matches_ocp_table():
    g = load_golden("e4m3_ocp.json")
    book = e4m3.codebook()
    for row in g["codes"]:
        v = book[row["code"]]
        if row["value"] == "nan":
            assert np.isnan(v)
        else:
            assert v == row["value"] and np.signbit(v) == np.signbit(row["value"])
    finite = book[~np.isnan(book)]
    assert len(finite) == 254 and np.max(finite) == 448.0 and np.min(finite) == -448.0


def test_e4m3_round_trip_every_code():
    codes = np.arange(256, dtype=np.uint8)
    vals = e4m3.decode(codes)
    ok = ~np.isnan(vals)
    assert np.array_equal(e4m3.encode(vals[ok]), codes[ok])


def test_e4m3_encode_is_nearest_even_by_brute_force():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 3, rng.standard_normal(2000) * 200,
                        rng.standard_normal(2000) * 0.01])
    book = e4m3.codebook()
    finite_codes = np.array([c for c in range(256) if not np.isnan(book[c])])
    vals = book[finite_codes]
    for xi, ci in zip(x, e4m3.encode(x)):
        xs = np.clip(xi, -448.0, 448.0)
        d = np.abs(vals - xs)
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:                                   # a tie: keep the even mantissa
            best = [b for b in best if finite_codes[b] % 2 == 0 and (xs != 0 or np.signbit(vals[b]) == np.signbit(xs))]
        assert ci in finite_codes[best] or book[ci] == vals[best[0]], (xi, ci)


def test_e4m3_matches_torch_in_range_and_saturates():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(50000) * 50).astype(np.float32)
    x = x[np.abs(x) < 448]
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3.encode(x), t)
    assert e4m3.encode(np.array([500.0, -1e6, 448.0, 463.9]))[0] == 0x7E
    assert list(e4m3.encode(np.array([500.0, -1e6, 448.0, 463.9]))) == [0x7E, 0xFE, 0x7E, 0x7E]
    assert e4m3.encode(np.array([np.nan]))[0] == 0x7F


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(100000), rng.standard_normal(1000) * 1e30]).astype(np.float32)
    ours = mla_ref.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(mla_ref.bf16_to_f64(ours), torch.from_numpy(x).to(torch.bfloat16).double().numpy())


def test_stored_row_bf16():
    rng = np.random.default_rng(3)
    rows = mla_ref.bf16_round(rng.standard_normal((50, 576)).astype(np.float32))
    pos = rng.integers(0, 70000, 50)
    st = np.stack([mla_ref.stored_row_bf16(rows[i], pos[i], 512, 10000.0) for i in range(50)])
    assert np.array_equal(st[:, :512], rows[:, :512])               # latent copied bit for bit
    exact = np.stack([mla_ref.rope(mla_ref.bf16_to_f64(rows[i, 512:]), pos[i], 10000.0) for i in range(50)])
    got = mla_ref.bf16_to_f64(st[:, 512:])
    ulp = np.maximum(np.abs(exact), 1e-30) * 2.0 ** -8              # one bf16 ulp bound
    assert np.all(np.abs(got - exact) <= ulp)
    # position 0 leaves the key unrotated
    assert np.array_equal(mla_ref.stored_row_bf16(rows[0], 0, 512, 10000.0), rows[0])


def test_stored_row_e4m3():
    rng = np.random.default_rng(4)
    rows = mla_ref.bf16_round(rng.standard_normal((40, 576)).astype(np.float32))
    scale = np.float32(6.0 / 448.0)
    st = np.stack([mla_ref.stored_row_e4m3(rows[i], 100 + i, 512, 10000.0, scale) for i in range(40)])
    vals = mla_ref.bf16_to_f64(rows)
    vals[:, 512:] = np.stack([mla_ref.rope(vals[i, 512:], 100 + i, 10000.0) for i in range(40)])
    back = e4m3.decode(st) * float(scale)
    # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 for normals, absolute 2^-10 * scale below
    err = np.abs(back - np.clip(vals, -448 * float(scale), 448 * float(scale)))
    assert np.all(err <= np.maximum(np.abs(vals) * 2.0 ** -4, 2.0 ** -10 * float(scale)) + 1e-12)
