"""The device-side projections around the decode: mla_project (W_Q, W_O) and the fused
down-projection + cache write mla_kv_project_append, against float64 products, against the
two-call path they fuse (bit for bit), and as the whole V2-Lite layer step on the GPU
against the oracle's one-shot causal forward."""
import numpy as np
import pytest
import torch

from mla_absorbed_latent_decode_gb300 import binding as B
from mla_absorbed_latent_decode_gb300 import workloads as W
from mla_absorbed_latent_decode_gb300.runner import SENTINEL, DecodeSession, bf16_tensor
from oracle import mla_ref
from tests.mla_cases import BF16_TOL, bf16_out_to_f64, compare

pytestmark = pytest.mark.gpu


def _bits(rng, shape, std):
    return W.to_bf16_bits(rng.standard_normal(shape) * std)


def _handle(n_h=16, cache_dtype=W.CACHE_BF16, fp8_scale=0.0, max_position=4096):
    rng = np.random.default_rng(5)
    cfg = B.make_config(n_h, cache_dtype=cache_dtype, max_position=max_position, rope_base=10000.0,
                        fp8_scale=fp8_scale)
    w_uk = bf16_tensor(_bits(rng, (n_h, 128, 512), 0.02), "cuda")
    w_uv = bf16_tensor(_bits(rng, (n_h, 128, 512), 0.02), "cuda")
    return B.Mla(cfg, w_uk, w_uv)


@pytest.mark.parametrize("m,k,n_out", [(1, 256, 16), (26, 2048, 3072), (33, 2048, 576), (70, 512, 48),
                                       (1, 2048, 2048)])
def test_project_matches_float64(m, k, n_out):
    rng = np.random.default_rng(m * 7 + k + n_out)
    xb, wb = _bits(rng, (m, k), 1.0), _bits(rng, (n_out, k), 0.02)
    mla = _handle()
    y = torch.empty((m, n_out), dtype=torch.bfloat16, device="cuda")
    mla.project(bf16_tensor(xb, "cuda"), bf16_tensor(wb, "cuda"), y)
    got = bf16_out_to_f64(y)
    x, w = mla_ref.bf16_to_f64(xb), mla_ref.bf16_to_f64(wb)
    ref = x @ w.T
    # bf16 rounding of the fp32 sum (half an ulp, 2^-9 relative) plus the fp32 accumulation error
    bound = 2.0 ** -8 * np.abs(ref) + 2.0 ** -18 * (np.abs(x) @ np.abs(w).T)
    assert np.all(np.abs(got - ref) <= bound), np.max(np.abs(got - ref) - bound)
    mla.close()


@pytest.mark.parametrize("cache", [W.CACHE_BF16, W.CACHE_FP8, W.CACHE_FP8_BLOCK])
def test_kv_project_append_writes_the_bytes_of_project_then_append(cache):
    rng = np.random.default_rng(11 + cache)
    n, hidden, num_pages, bt_stride = 70, 2048, 12, 4
    xb, wb = _bits(rng, (n, hidden), 1.0), _bits(rng, (576, hidden), 0.02)
    fp8 = cache == W.CACHE_FP8
    mla = _handle(cache_dtype=cache, fp8_scale=0.01 if fp8 else 0.0)
    bt = torch.from_numpy(rng.permutation(num_pages)[:3 * bt_stride].astype(np.int32).reshape(3, bt_stride)).cuda()
    slots = rng.choice(3 * bt_stride * 64, size=n, replace=False)
    seq_np, pos_np = (slots // (bt_stride * 64)).astype(np.int32), (slots % (bt_stride * 64)).astype(np.int32)
    seq_np[5] = 3                                                   # outside the block table: skipped, flagged
    seq, pos = torch.from_numpy(seq_np).cuda(), torch.from_numpy(pos_np).cuda()
    row_bytes = W.ROW_BYTES[cache]
    fused = torch.full((num_pages, 64, row_bytes), SENTINEL, dtype=torch.uint8, device="cuda")
    split = fused.clone()
    x, w = bf16_tensor(xb, "cuda"), bf16_tensor(wb, "cuda")
    mla.kv_project_append(x, w, seq, pos, bt, fused, num_pages)
    assert mla.get_status() == B.MLA_CHECK_APPEND_INDEX
    rows = torch.empty((n, 576), dtype=torch.bfloat16, device="cuda")
    mla.project(x, w, rows)
    mla.kv_append(rows, seq, pos, bt, split, num_pages)
    assert mla.get_status() == B.MLA_CHECK_APPEND_INDEX
    assert torch.equal(fused, split)
    assert int((fused != SENTINEL).any(dim=2).sum()) == n - 1       # every valid row written, once
    mla.close()


def test_kv_project_append_argument_errors():
    mla = _handle()
    x = torch.zeros((4, 300), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((576, 300), dtype=torch.bfloat16, device="cuda")
    i = torch.zeros(4, dtype=torch.int32, device="cuda")
    bt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    cache = torch.zeros((1, 64, 1152), dtype=torch.uint8, device="cuda")
    with pytest.raises(B.MlaError) as e:
        mla.kv_project_append(x, w, i, i, bt, cache, 1)
    assert e.value.status == B.MLA_ERR_INVALID_ARG and "hidden" in e.value.message
    with pytest.raises(B.MlaError) as e:
        mla.project(x[:, :256], torch.zeros((20, 256), dtype=torch.bfloat16, device="cuda"),
                    torch.zeros((4, 20), dtype=torch.bfloat16, device="cuda"))
    assert e.value.status == B.MLA_ERR_INVALID_ARG
    mla.close()


def test_v2lite_layer_step_entirely_on_the_gpu():
    """x -> (W_Q, W_DKV) -> cache -> absorbed decode -> out, for the 26-token V2-Lite layer,
    against the one-shot fp64 causal forward of the same layer (row 25) and against the
    path whose projections are done by the caller in float64."""
    inp = W.v2lite_single_step_inputs(seed=0)
    n_h, T = inp["n_h"], inp["tokens"]
    xf = mla_ref.bf16_to_f64(inp["x"])
    c, kr, q = mla_ref.project_inputs(xf, mla_ref.bf16_to_f64(inp["w_dkv"]), mla_ref.bf16_to_f64(inp["w_q"]), n_h, 512)
    rows = mla_ref.bf16_round(np.concatenate([c, kr], axis=1).astype(np.float32))
    wl = W.v2lite_single_step(rows, mla_ref.bf16_round(q[-1].astype(np.float32)), inp["w_uk"], inp["w_uv"])
    host = DecodeSession(wl)
    host.append_rows()
    out_host = bf16_out_to_f64(host.decode())[0]
    host.close()

    s = DecodeSession(wl)
    x = bf16_tensor(inp["x"], "cuda")
    qall = torch.empty((T, n_h * 192), dtype=torch.bfloat16, device="cuda")
    s.mla.project(x, bf16_tensor(inp["w_q"], "cuda"), qall)
    seq = torch.zeros(T, dtype=torch.int32, device="cuda")
    pos = torch.arange(T, dtype=torch.int32, device="cuda")
    s.mla.kv_project_append(x, bf16_tensor(inp["w_dkv"], "cuda"), seq, pos, s.block_table, s.cache, wl.num_pages)
    out = bf16_out_to_f64(s.decode(q=qall[-1:].reshape(1, n_h, 192).contiguous()))[0]
    assert s.status() == 0
    s.close()
    full = mla_ref.causal_forward_naive(xf, mla_ref.bf16_to_f64(inp["w_dkv"]), mla_ref.bf16_to_f64(inp["w_q"]),
                                        mla_ref.bf16_to_f64(inp["w_uk"]), mla_ref.bf16_to_f64(inp["w_uv"]),
                                        mla_ref.default_scale(128, 64), 10000.0)
    assert np.max(np.abs(out - full[-1])) <= 2e-2 * np.max(np.abs(full[-1]))
    assert compare(out, out_host, BF16_TOL)[0] <= BF16_TOL


@pytest.mark.parametrize("m,n,ld,in_place", [(70, 512, 576, True), (33, 1536, 1536, False), (1, 8, 8, False)])
def test_rmsnorm_matches_float64(m, n, ld, in_place):
    rng = np.random.default_rng(m + n)
    xb = _bits(rng, (m, ld), 1.7)
    wb = W.to_bf16_bits(1.0 + 0.1 * rng.standard_normal(n))
    mla = _handle()
    x = bf16_tensor(xb, "cuda")
    y = x if in_place else torch.empty((m, ld), dtype=torch.bfloat16, device="cuda")
    mla.rmsnorm(x, n, bf16_tensor(wb, "cuda"), 1e-6, y)
    got = bf16_out_to_f64(y)
    ref = mla_ref.rms_norm(mla_ref.bf16_to_f64(xb)[:, :n], mla_ref.bf16_to_f64(wb), 1e-6)
    # bf16 rounding of the fp32 result plus the fp32 sum of squares
    assert np.all(np.abs(got[:, :n] - ref) <= 2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * np.max(np.abs(ref)))
    if in_place:                                   # the RoPE part of the rows is left alone
        assert np.array_equal(got[:, n:], mla_ref.bf16_to_f64(xb)[:, n:])
    with pytest.raises(B.MlaError):
        mla.rmsnorm(x, 12, bf16_tensor(wb, "cuda"), 1e-6, y)
    mla.close()


def test_layer_step_with_low_rank_query_and_kv_norm():
    """x -> W_DQ -> [W_UQ ; W_QR] (the low-rank query of "80 行 PyTorch 从零写 DeepSeek 的 MLA"
    section 2), x -> W_DKV -> kv_norm (RMSNorm of the latent) -> cache -> absorbed decode, all on
    the GPU, against the oracle's float64 forward of the same layer (multi-stage bf16 rounding:
    2e-2 of the output's largest magnitude)."""
    rng = np.random.default_rng(77)
    T, hidden, d_cq, n_h = 40, 1024, 512, 16
    eps = 1e-6
    xb = _bits(rng, (T, hidden), 1.0)
    w_dq, w_uq, w_qr = _bits(rng, (d_cq, hidden), 0.02), _bits(rng, (n_h * 128, d_cq), 0.05), _bits(rng, (n_h * 64, d_cq), 0.05)
    w_dkv = _bits(rng, (576, hidden), 0.02)
    w_kvn = W.to_bf16_bits(1.0 + 0.1 * rng.standard_normal(512))
    w_uk, w_uv = _bits(rng, (n_h, 128, 512), 0.02), _bits(rng, (n_h, 128, 512), 0.02)
    # the query weights joined per head as [content rows ; rope rows], so one projection gives q
    w_uqr = np.concatenate([w_uq.reshape(n_h, 128, d_cq), w_qr.reshape(n_h, 64, d_cq)], axis=1).reshape(n_h * 192, d_cq)
    wl = W.v2lite_single_step(np.zeros((T, 576), np.uint16), np.zeros((n_h, 192), np.uint16), w_uk, w_uv, n_h=n_h)
    s = DecodeSession(wl)
    x = bf16_tensor(xb, "cuda")
    qz = torch.empty((T, d_cq), dtype=torch.bfloat16, device="cuda")
    s.mla.project(x, bf16_tensor(w_dq, "cuda"), qz)
    q_all = torch.empty((T, n_h * 192), dtype=torch.bfloat16, device="cuda")
    s.mla.project(qz, bf16_tensor(w_uqr, "cuda"), q_all)
    rows = torch.empty((T, 576), dtype=torch.bfloat16, device="cuda")
    s.mla.project(x, bf16_tensor(w_dkv, "cuda"), rows)
    s.mla.rmsnorm(rows, 512, bf16_tensor(w_kvn, "cuda"), eps, rows)          # kv_norm, in place
    s.append_step(rows, torch.zeros(T, dtype=torch.int32, device="cuda"), torch.arange(T, dtype=torch.int32, device="cuda"))
    out = bf16_out_to_f64(s.decode(q=q_all[-1:].reshape(1, n_h, 192).contiguous()))[0]
    assert s.status() == 0
    s.close()
    xf = mla_ref.bf16_to_f64(xb)
    kv = xf @ mla_ref.bf16_to_f64(w_dkv).T
    c = mla_ref.rms_norm(kv[:, :512], mla_ref.bf16_to_f64(w_kvn), eps)
    kr = mla_ref.rope(kv[:, 512:], np.arange(T), 10000.0)
    q = mla_ref.low_rank_query(xf, mla_ref.bf16_to_f64(w_dq), mla_ref.bf16_to_f64(w_uq), mla_ref.bf16_to_f64(w_qr), n_h)
    ref = mla_ref.absorbed_decode(q[-1], c, kr, mla_ref.bf16_to_f64(w_uk), mla_ref.bf16_to_f64(w_uv), T - 1,
                                  mla_ref.default_scale(128, 64), 10000.0)
    assert np.max(np.abs(out - ref)) <= 2e-2 * np.max(np.abs(ref))
