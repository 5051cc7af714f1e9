"""Pins of the fp64 oracle: checks against what the pages and the mathematics fix.

Each ``pin_*`` function takes the oracle module and raises AssertionError when
the oracle disagrees with a fixed value, a closed form, an invariant or an
identity.  ``test_oracle_pins.py`` runs them as tests; ``test_oracle_mutations.py``
plants plausible mistakes in the oracle and checks that some pin fails.
"""
import numpy as np

from tests.conftest import load_golden

BASE = 10000.0


def _rand(seed, *shape, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def _tiny_problem(seed, n_h=3, d_nope=4, d_rope=4, d_c=6, d_v=5, T=7):
    q = _rand(seed, n_h, d_nope + d_rope)
    c = _rand(seed + 1, T, d_c)
    kr = _rand(seed + 2, T, d_rope)
    w_uk = _rand(seed + 3, n_h, d_nope, d_c, std=0.5)
    w_uv = _rand(seed + 4, n_h, d_v, d_c, std=0.5)
    return q, c, kr, w_uk, w_uv


# --------------------------------------------------------------------------- RoPE

def pin_rope_closed_forms(ref):
    # position 0 is the identity
    x = _rand(0, 5, 64)
    assert np.array_equal(ref.rope(x, 0, BASE), x)
    # a unit vector on pair 0 at position p lands on (cos p, sin p): inv_freq_0 = 1
    e0 = np.zeros(64); e0[0] = 1.0
    r = ref.rope(e0, 3, BASE)
    assert abs(r[0] - np.cos(3.0)) < 1e-15 and abs(r[1] - np.sin(3.0)) < 1e-15
    assert np.all(r[2:] == 0.0)
    # pair i rotates at base^(-2i/d): for d = 4, pair 1 turns at 0.01 rad per position
    e1 = np.array([0.0, 0.0, 1.0, 0.0])
    r = ref.rope(e1, 7, BASE)
    assert abs(r[2] - np.cos(0.07)) < 1e-15 and abs(r[3] - np.sin(0.07)) < 1e-15
    # equivalent complex form: pair (a, b) -> (a + i b) * exp(i theta)
    pos = 1234
    theta = pos * BASE ** (-np.arange(0, 64, 2) / 64.0)
    z = (x[:, 0::2] + 1j * x[:, 1::2]) * np.exp(1j * theta)
    r = ref.rope(x, pos, BASE)
    assert np.max(np.abs(r[:, 0::2] - z.real)) < 1e-12 and np.max(np.abs(r[:, 1::2] - z.imag)) < 1e-12


def pin_rope_relative_position(ref):
    q, k = _rand(1, 64), _rand(2, 64)
    for m, n, d in [(5, 3, 100), (4000, 17, 60000), (0, 65535, 1)]:
        a = ref.rope(q, m, BASE) @ ref.rope(k, n, BASE)
        b = ref.rope(q, m + d, BASE) @ ref.rope(k, n + d, BASE)
        assert abs(a - b) < 1e-9 * (1 + abs(a))
    # pair norms are preserved
    r = ref.rope(q, 777, BASE)
    assert np.allclose(r[0::2] ** 2 + r[1::2] ** 2, q[0::2] ** 2 + q[1::2] ** 2, rtol=1e-13)


# --------------------------------------------------------------------------- attention

def pin_scale_worked_example(ref):
    """Two tokens, one head, identity W_UK, zero RoPE parts: the weight of token 0 is
    sigmoid(a * scale) with scale = 1/sqrt(d_nope + d_rope) = 1/2; a = 2 ln 3 gives 3/4."""
    a = 2.0 * np.log(3.0)
    q = np.array([[a, 0.0, 0.0, 0.0]])                   # [q_nope (2) | q_pe (2)]
    c = np.array([[1.0, 0.0], [0.0, 1.0]])
    kr = np.zeros((2, 2))
    w_uk = np.eye(2)[None]                               # [1, d_nope=2, d_c=2]
    w_uv = np.array([[[1.0, 0.0]]])                      # [1, d_v=1, d_c=2]
    scale = ref.default_scale(2, 2)
    assert scale == 0.5
    for fn in (ref.naive_decode, ref.absorbed_decode):
        o = fn(q, c, kr, w_uk, w_uv, 1, scale, BASE)
        assert abs(o[0, 0] - 0.75) < 1e-15, o
    # the RoPE score counts too: put the same logit on the rope branch instead
    q2 = np.array([[0.0, 0.0, a, 0.0]])
    kr2 = ref.rope(np.array([[1.0, 0.0], [0.0, 0.0]]), np.array([0, 1]), BASE)
    # query rotated at position 1, key 0 at position 0: score = a cos(1) * scale
    for fn in (ref.naive_decode, ref.absorbed_decode):
        o = fn(q2, c, kr2, w_uk, w_uv, 1, scale, BASE)
        p0 = 1.0 / (1.0 + np.exp(-a * np.cos(1.0) * scale))
        assert abs(o[0, 0] - p0) < 1e-14, (o, p0)


def pin_naive_equals_absorbed(ref):
    """Exact-arithmetic identity of the two paths ("DeepSeek MLA 吸收式缓存" §2.2-2.3, §5.3)."""
    printed = load_golden("printed_discrepancies.json")
    for seed in (0, 10, 20):
        q, c, kr, w_uk, w_uv = _tiny_problem(seed)
        kr_rot = ref.rope(kr, np.arange(kr.shape[0]), BASE)
        scale = ref.default_scale(4, 4)
        a = ref.naive_decode(q, c, kr_rot, w_uk, w_uv, 6, scale, BASE)
        b = ref.absorbed_decode(q, c, kr_rot, w_uk, w_uv, 6, scale, BASE)
        assert np.max(np.abs(a - b)) <= 1e-12
    # V2-Lite head shapes, 37 tokens, weights N(0, 0.02^2) as in the configurations
    rng = np.random.default_rng(5)
    n_h, T = 16, 37
    q = rng.standard_normal((n_h, 192))
    c = rng.standard_normal((T, 512))
    kr = ref.rope(rng.standard_normal((T, 64)), np.arange(T), BASE)
    w_uk = rng.standard_normal((n_h, 128, 512)) * 0.02
    w_uv = rng.standard_normal((n_h, 128, 512)) * 0.02
    scale = ref.default_scale(128, 64)
    a = ref.naive_decode(q, c, kr, w_uk, w_uv, T - 1, scale, BASE)
    b = ref.absorbed_decode(q, c, kr, w_uk, w_uv, T - 1, scale, BASE)
    d = np.max(np.abs(a - b))
    assert d <= 1e-10 and d < printed["naive_vs_absorb_fp32_max_abs"]


def pin_rope_on_content_breaks_absorption(ref):
    """The counter-example of "80 行 PyTorch 从零写 DeepSeek 的 MLA" §4: rotate the
    content key by position and the absorbed score (against the unrotated latent)
    no longer matches."""
    rng = np.random.default_rng(7)
    n_h, T = 4, 50
    q_nope = rng.standard_normal((n_h, 128))
    c = rng.standard_normal((T, 512))
    w_uk = rng.standard_normal((n_h, 128, 512)) * 0.05
    q_abs = ref.absorb_query(np.concatenate([q_nope, np.zeros((n_h, 64))], 1), w_uk, 0, BASE)
    absorbed = q_abs[:, :512] @ c.T
    expanded = np.stack([(c @ w_uk[h].T) @ q_nope[h] for h in range(n_h)])
    assert np.max(np.abs(absorbed - expanded)) < 1e-10
    rotated = np.stack([ref.rope(c @ w_uk[h].T, np.arange(T), BASE) @ q_nope[h]
                        for h in range(n_h)])
    printed = load_golden("printed_discrepancies.json")
    assert np.max(np.abs(absorbed - rotated)) > printed["rope_on_content_divergence"] / 10


def pin_closed_forms(ref):
    q, c, kr, w_uk, w_uv = _tiny_problem(3)
    kr_rot = ref.rope(kr, np.arange(kr.shape[0]), BASE)
    s = ref.default_scale(4, 4)
    # one cached token: the output is W_UV[h] c_0 for every head
    o = ref.absorbed_decode(q, c[:1], kr_rot[:1], w_uk, w_uv, 0, s, BASE)
    assert np.max(np.abs(o - np.einsum("hvc,c->hv", w_uv, c[0]))) < 1e-14
    # zero query: uniform weights, the latent sum is the mean row
    o_lat, lse = ref.absorbed_latent(np.zeros((3, 10)), c, kr_rot, s)
    assert np.max(np.abs(o_lat - c.mean(0))) < 1e-14
    assert np.max(np.abs(lse - np.log(c.shape[0]))) < 1e-14
    # identical cached rows: the latent sum is that row whatever the query
    crep = np.repeat(c[:1], 9, 0)
    krep = np.repeat(kr_rot[:1], 9, 0)
    o_lat, _ = ref.absorbed_latent(ref.absorb_query(q, w_uk, 8, BASE), crep, krep, s)
    assert np.max(np.abs(o_lat - c[0])) < 1e-14


def pin_split_lse_identity(ref):
    q, c, kr, w_uk, _ = _tiny_problem(4, T=40)
    kr_rot = ref.rope(kr, np.arange(40), BASE)
    q_abs = ref.absorb_query(q, w_uk, 39, BASE)
    s = ref.default_scale(4, 4)
    full, lse = ref.absorbed_latent(q_abs, c, kr_rot, s)
    for bounds in ([0, 40], [0, 1, 40], [0, 13, 27, 40], list(range(0, 41, 5))):
        o, l = ref.split_latent(q_abs, c, kr_rot, s, bounds)
        assert np.max(np.abs(o - full)) < 1e-13 and np.max(np.abs(l - lse)) < 1e-13


def pin_one_shot_equals_incremental(ref):
    """"80 行 PyTorch 从零写 DeepSeek 的 MLA" §2 cache-equivalence test at V2-Lite
    shapes: prefill 25 tokens, decode the 26th, against one causal pass over 26."""
    printed = load_golden("printed_discrepancies.json")
    rng = np.random.default_rng(11)
    hidden, n_h, L = 256, 16, 26
    x = rng.standard_normal((L, hidden))
    w_dkv = rng.standard_normal((576, hidden)) * 0.02
    w_q = rng.standard_normal((n_h * 192, hidden)) * 0.02
    w_uk = rng.standard_normal((n_h, 128, 512)) * 0.02
    w_uv = rng.standard_normal((n_h, 128, 512)) * 0.02
    s = ref.default_scale(128, 64)
    full = ref.causal_forward_naive(x, w_dkv, w_q, w_uk, w_uv, s, BASE)
    prefill = ref.causal_forward_naive(x[:L - 1], w_dkv, w_q, w_uk, w_uv, s, BASE)
    assert np.max(np.abs(full[:L - 1] - prefill)) <= 1e-13
    c, kr, q = ref.project_inputs(x, w_dkv, w_q, n_h, 512)
    kr_rot = ref.rope(kr, np.arange(L), BASE)
    dec = ref.absorbed_decode(q[L - 1], c, kr_rot, w_uk, w_uv, L - 1, s, BASE)
    d = np.max(np.abs(dec - full[L - 1]))
    assert d <= 1e-12 and d < printed["cache_equivalence_decoded_max_diff_fp32"]
    nv = ref.naive_decode(q[L - 1], c, kr_rot, w_uk, w_uv, L - 1, s, BASE)
    assert np.max(np.abs(nv - full[L - 1])) <= 1e-12


def pin_prefill_rows_are_decodes(ref):
    """A causal prefill chunk is the per-position decode of each of its queries: row i of a
    chunk after a prefix of pos0 rows is the decode (naive and absorbed) of query i over the
    rows 0 .. pos0 + i; a whole prompt (pos0 = 0) is the one-shot causal forward; and a prompt
    prefilled in two chunks gives the rows of the single pass."""
    n_h, T, pos0 = 3, 11, 6
    rng = np.random.default_rng(21)
    q = rng.standard_normal((T, n_h, 8))
    _, c, kr, w_uk, w_uv = _tiny_problem(22, T=T)
    kr_rot = ref.rope(kr, np.arange(T), BASE)
    s = ref.default_scale(4, 4)
    chunk = ref.prefill_naive(q[pos0:], c, kr_rot, w_uk, w_uv, pos0, s, BASE)
    assert chunk.shape == (T - pos0, n_h, 5)
    for i in range(T - pos0):
        p = pos0 + i
        nv = ref.naive_decode(q[p], c[:p + 1], kr_rot[:p + 1], w_uk, w_uv, p, s, BASE)
        ab = ref.absorbed_decode(q[p], c[:p + 1], kr_rot[:p + 1], w_uk, w_uv, p, s, BASE)
        assert np.max(np.abs(chunk[i] - nv)) <= 1e-13 and np.max(np.abs(chunk[i] - ab)) <= 1e-12
    whole = ref.prefill_naive(q, c, kr_rot, w_uk, w_uv, 0, s, BASE)
    assert np.max(np.abs(whole[pos0:] - chunk)) <= 1e-13
    head = ref.prefill_naive(q[:pos0], c, kr_rot, w_uk, w_uv, 0, s, BASE)
    assert np.max(np.abs(whole[:pos0] - head)) <= 1e-13
    # from hidden states: the one-shot causal forward of the projected prompt
    L, hidden = 9, 32
    x = rng.standard_normal((L, hidden))
    w_dkv = rng.standard_normal((10, hidden)) * 0.3
    w_q = rng.standard_normal((n_h * 8, hidden)) * 0.3
    cx, krx, qx = ref.project_inputs(x, w_dkv, w_q, n_h, 6)
    pre = ref.prefill_naive(qx, cx, ref.rope(krx, np.arange(L), BASE), w_uk, w_uv, 0, s, BASE)
    one = ref.causal_forward_naive(x, w_dkv, w_q, w_uk, w_uv, s, BASE)
    assert np.max(np.abs(pre - one)) <= 1e-12


# --------------------------------------------------------------------------- bytes

def pin_cache_bytes(ref):
    g = load_golden("cache_bytes_v2lite.json")
    sh = g["shape"]
    T = g["active_tokens"]
    a = ref.absorb_cache_bytes(T, sh["d_c"], sh["d_rope"], sh["elem_bytes"])
    n = ref.naive_cache_bytes(T, sh["n_h"], sh["d_nope"], sh["d_rope"], sh["d_v"], sh["elem_bytes"])
    assert a == g["absorb_total_active"]
    assert ref.absorb_cache_bytes(T, sh["d_c"], 0, 2) == g["absorb_latent_active"]
    assert ref.absorb_cache_bytes(T, 0, sh["d_rope"], 2) == g["absorb_rope_active"]
    assert n == g["naive_total_active"]
    assert ref.naive_cache_bytes(T, sh["n_h"], sh["d_nope"], sh["d_rope"], 0, 2) == g["naive_key_active"]
    assert ref.naive_cache_bytes(T, sh["n_h"], 0, 0, sh["d_v"], 2) == g["naive_value_active"]
    assert abs(n / a - g["ratio_naive_over_absorb"]) < 1e-12
    assert abs(100.0 * (1 - a / n) - g["reduction_percent"]) < 1e-12
    S = g["allocated_slots"]
    assert ref.absorb_cache_bytes(S, sh["d_c"], sh["d_rope"], 2) == g["absorb_total_allocated"]
    assert ref.naive_cache_bytes(S, sh["n_h"], sh["d_nope"], sh["d_rope"], sh["d_v"], 2) == g["naive_total_allocated"]
    assert ref.absorb_cache_bytes(1, sh["d_c"], sh["d_rope"], 2) == g["per_token_latent_bytes"]
    assert ref.naive_cache_bytes(1, sh["n_h"], sh["d_nope"], sh["d_rope"], sh["d_v"], 2) == g["per_token_eager_bytes"]


def pin_mha_ratio_and_read_bytes(ref):
    g = load_golden("mha_ratio.json")
    v = g["v2_style"]
    r = ref.mha_ratio(v["d_c"], v["d_r"], v["n_h"], v["d_h"])
    assert ref.absorb_cache_bytes(1, v["d_c"], v["d_r"], 2) == g["mla_bytes_per_token"]
    assert abs(1.0 / r - g["printed_ratio"]) < 0.05
    assert round(1.0 / r) == g["g5_ratio_approx_inverse"]
    for row in g["allocation_log"]:
        mla = ref.decode_kv_read_bytes(1, row["L"], v["d_c"], v["d_r"], 2)
        assert abs(mla / 2 ** 20 - row["mla_mb"]) < 0.005
    six = g["sixty_layers_32k"]
    tot = six["layers"] * ref.decode_kv_read_bytes(1, six["L"], v["d_c"], v["d_r"], 2)
    assert abs(tot / 2 ** 30 - six["mla_gb"]) < 0.005
    u = load_golden("g5_acceptance.json")["use_case_1"]
    b = ref.decode_kv_read_bytes(1, u["s_ctx"], u["d_c"], u["d_rope"], u["elem_bytes"])
    assert b == u["bytes_per_sequence"]
    # linear in B, monotone in s_ctx, and a list of lengths sums like B * s_ctx
    assert ref.decode_kv_read_bytes(64, 4096, 512, 64, 2) == 64 * b * 2
    prev = -1
    for s in (1, 2, 64, 65, 4096, 65536):
        cur = ref.decode_kv_read_bytes(8, s, 512, 64, 2)
        assert cur > prev
        prev = cur
    assert ref.decode_kv_read_bytes(3, [5, 6, 7], 512, 64, 1) == 18 * 576


def pin_fp8_block_format(ref):
    """The per-block FP8 row: 656 bytes per token, the pages' figure against 576 for the pure
    latent; in every non-zero block the largest magnitude lands exactly on the largest e4m3
    code and every value within e4m3's half-step of its block; a block's scale belongs to that
    block alone (a power-of-two change of one block's values moves only its scale); the RoPE
    key is the bf16 cache's, not quantised; an all-zero block is zeros."""
    g = load_golden("fp8_block_format.json")
    rng = np.random.default_rng(31)
    n = 6
    x = rng.standard_normal((n, 576)) * np.array([1.0, 30.0, 1e-3, 7.0] * 128 + [1.0] * 64)[None, :]
    x[3, 128:256] = 0.0                                              # an all-zero block
    bits = ref.bf16_round(x.astype(np.float32))
    pos = np.arange(n) * 37
    st = ref.stored_row_fp8_block(bits, pos, 512, BASE)
    assert st.shape == (n, g["bytes_per_token"]) and 512 + 64 == g["pure_latent_bytes_per_token"]
    codes = st[:, :512].reshape(n, 4, 128)
    vals = ref.fp8_block_values(st, 512)
    xv = ref.bf16_to_f64(bits)
    for r in range(n):
        for k in range(4):
            blk = xv[r, 128 * k:128 * (k + 1)]
            if not np.any(blk):
                assert not np.any(codes[r, k]) and not np.any(vals[r, 128 * k:128 * (k + 1)])
                continue
            mag = codes[r, k] & 0x7F
            assert mag.max() == 0x7E and mag[np.argmax(np.abs(blk))] == 0x7E
            sc = np.max(np.abs(blk)) / 448.0
            err = np.abs(vals[r, 128 * k:128 * (k + 1)] - blk)
            assert np.all(err <= 2.0 ** -4 * np.abs(blk) * (1 + 2.0 ** -20) + sc * 2.0 ** -10)
    # one block scaled by 4: only that block's scale moves (times 4); every code stays
    y = xv.copy()
    y[:, 256:384] *= 4.0
    st4 = ref.stored_row_fp8_block(ref.bf16_round(y.astype(np.float32)), pos, 512, BASE)
    assert np.array_equal(st4[:, :512], st[:, :512])
    s1 = np.ascontiguousarray(st[:, 512:528]).view("<f4")
    s4 = np.ascontiguousarray(st4[:, 512:528]).view("<f4")
    assert np.array_equal(s4[:, [0, 1, 3]], s1[:, [0, 1, 3]]) and np.array_equal(s4[:, 2], 4 * s1[:, 2])
    # the RoPE key: the bf16 cache's codes
    bf = ref.stored_row_bf16(bits, pos, 512, BASE)
    assert np.array_equal(np.ascontiguousarray(st[:, 528:]).view("<u2"), bf[:, 512:])
    assert np.array_equal(vals[:, 512:], ref.bf16_to_f64(bf[:, 512:]))


def pin_rms_norm(ref):
    """RMSNorm against closed forms: a constant row c gives sign(c) w (eps = 0); the output
    does not change when a row is scaled by a > 0 (eps = 0); with unit weights every row's
    mean square is 1 (eps = 0), and eps enters under the root (a row of 3s with eps = 7 gives
    3 / 4 = 0.75)."""
    rng = np.random.default_rng(41)
    n = 48
    w = rng.standard_normal(n)
    for c in (2.5, -0.25):
        assert np.max(np.abs(ref.rms_norm(np.full((1, n), c), w, 0.0) - np.sign(c) * w)) <= 1e-15
    x = rng.standard_normal((4, n))
    assert np.max(np.abs(ref.rms_norm(3.7 * x, w, 0.0) - ref.rms_norm(x, w, 0.0))) <= 1e-14
    y = ref.rms_norm(x, np.ones(n), 0.0)
    assert np.max(np.abs(np.mean(y * y, axis=1) - 1.0)) <= 1e-14
    assert abs(ref.rms_norm(np.full((1, n), 3.0), np.ones(n), 7.0)[0, 0] - 0.75) <= 1e-15


def pin_low_rank_query(ref):
    """The low-rank query path is the composition of its three maps: with W_DQ the identity it
    is [W_UQ x ; W_QR x] per head, and it is linear in x."""
    rng = np.random.default_rng(42)
    n_h, d, dn, dr = 3, 8, 4, 2
    x = rng.standard_normal((5, d))
    w_uq, w_qr = rng.standard_normal((n_h * dn, d)), rng.standard_normal((n_h * dr, d))
    q = ref.low_rank_query(x, np.eye(d), w_uq, w_qr, n_h)
    assert q.shape == (5, n_h, dn + dr)
    for h in range(n_h):
        assert np.max(np.abs(q[:, h, :dn] - x @ w_uq[h * dn:(h + 1) * dn].T)) <= 1e-13
        assert np.max(np.abs(q[:, h, dn:] - x @ w_qr[h * dr:(h + 1) * dr].T)) <= 1e-13
    w_dq, w_uq2, w_qr2 = rng.standard_normal((6, d)), rng.standard_normal((n_h * dn, 6)), rng.standard_normal((n_h * dr, 6))
    a = ref.low_rank_query(2.0 * x, w_dq, w_uq2, w_qr2, n_h)
    b = ref.low_rank_query(x, w_dq, w_uq2, w_qr2, n_h)
    assert np.max(np.abs(a - 2.0 * b)) <= 1e-12
    qz = x @ w_dq.T                                  # and the composition, head by head
    assert np.max(np.abs(b[:, 1, :dn] - qz @ w_uq2[dn:2 * dn].T)) <= 1e-13


# --------------------------------------------------------------------------- paged cache

def pin_paged_cache(ref):
    """The paged indirection (a reading of "DeepSeek-V2-Lite 真实权重执行审计" §3.3, which asks
    for a paged latent-only cache without fixing its layout): token ``pos`` of a sequence
    lives in the page its block-table row names at ``pos // page``, slot ``pos % page``.

    Fixed by hand on a 3-sequence table with 4-token pages (slots and pages written out,
    not computed); gathering follows block-table order, not page-id order; and the batched
    decode over a shuffled paged cache equals the contiguous decode of each sequence's
    rows with the query at position ``len - 1``."""
    bt = np.array([[5, 2, -1], [0, 7, 3], [4, -1, -1]], np.int32)
    expect = {(0, 0): (5, 0), (0, 3): (5, 3), (0, 5): (2, 1), (1, 3): (0, 3), (1, 4): (7, 0),
              (1, 9): (3, 1), (1, 11): (3, 3), (2, 2): (4, 2)}
    for (seq, pos), ps in expect.items():
        assert ref.page_slot(bt, seq, pos, 4) == ps, (seq, pos, ref.page_slot(bt, seq, pos, 4))
    # value of a cached row = 1000 page + slot: sequence 1's first 10 rows, written out
    cache = np.full((8, 4, 2), np.nan)
    for page in range(8):
        for slot in range(4):
            cache[page, slot] = (1000.0 * page + slot, -1.0)
    got = ref.gather_sequence(cache, bt, 1, 10, 4)[:, 0]
    assert got.tolist() == [0, 1, 2, 3, 7000, 7001, 7002, 7003, 3000, 3001], got
    assert ref.gather_sequence(cache, bt, 0, 6, 4)[:, 0].tolist() == [5000, 5001, 5002, 5003, 2000, 2001]
    assert ref.gather_sequence(cache, bt, 2, 1, 4)[:, 0].tolist() == [4000]
    # decode over a shuffled pool (NaN everywhere no row was written) = contiguous decode
    rng = np.random.default_rng(31)
    n_h, d_c, d_r, lens, page = 3, 6, 4, [5, 9, 1], 4
    q = rng.standard_normal((3, n_h, 4 + d_r))
    w_uk = rng.standard_normal((n_h, 4, d_c)) * 0.5
    w_uv = rng.standard_normal((n_h, 5, d_c)) * 0.5
    rows = [rng.standard_normal((L, d_c + d_r)) for L in lens]
    order = rng.permutation(9)                       # 2 + 3 + 1 pages used out of 9
    table = np.full((3, 3), -1, np.int32)
    pool = np.full((9, page, d_c + d_r), np.nan)
    nxt = 0
    for b, L in enumerate(lens):
        for i in range(-(-L // page)):               # whole pages copied block by block
            table[b, i] = order[nxt]
            blk = rows[b][i * page:(i + 1) * page]
            pool[order[nxt], :len(blk)] = blk
            nxt += 1
    s = ref.default_scale(4, d_r)
    out = ref.decode_batch(q, pool, table, np.array(lens), w_uk, w_uv, d_c, page, s, BASE)
    for b, L in enumerate(lens):
        want = ref.absorbed_decode(q[b], rows[b][:, :d_c], rows[b][:, d_c:], w_uk, w_uv, L - 1, s, BASE)
        assert np.all(np.isfinite(out[b])) and np.max(np.abs(out[b] - want)) <= 1e-13
    nv = ref.decode_batch(q, pool, table, np.array(lens), w_uk, w_uv, d_c, page, s, BASE, path="naive")
    assert np.max(np.abs(nv - out)) <= 1e-12


ALL_PINS = [
    pin_rope_closed_forms, pin_rope_relative_position, pin_scale_worked_example,
    pin_naive_equals_absorbed, pin_rope_on_content_breaks_absorption, pin_closed_forms,
    pin_split_lse_identity, pin_one_shot_equals_incremental, pin_prefill_rows_are_decodes, pin_cache_bytes,
    pin_mha_ratio_and_read_bytes, pin_fp8_block_format, pin_rms_norm, pin_low_rank_query,
    pin_paged_cache,
]
