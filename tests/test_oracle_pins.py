"""Pins for the CPU oracle: worked examples, closed forms, invariants and an
independent fp64 brute force.  These run without a GPU and never touch the CUDA
library; they establish that the oracle computes what the pages define before
it is trusted as the reference for the kernels."""
import json
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------- RMSNorm
def test_rmsnorm_worked_example(orc):
    g = _golden("rmsnorm_worked_example.json")
    y = orc.rms_norm(np.array([g["x"]], np.float32), np.array(g["gains"], np.float32), eps=g["eps"])[0]
    tol = 0.5 * 10 ** -g["printed_decimals"] + 1e-7
    np.testing.assert_allclose(y, g["normalized_printed"], atol=tol, rtol=0)
    # closed form: x / sqrt(7.5)
    exact = np.array(g["x"]) / math.sqrt(g["mean_sq"])
    np.testing.assert_allclose(y, exact, rtol=3e-7, atol=0)


@pytest.mark.parametrize("n", [4, 896, 1024, 1001])
def test_rmsnorm_unit_rms_and_gains(orc, n):
    r = _rng(n)
    x = r.standard_normal((5, n)).astype(np.float32) * 3.0
    y = orc.rms_norm(x, None, eps=0.0)
    rms = np.sqrt(np.mean(y.astype(np.float64) ** 2, axis=1))
    np.testing.assert_allclose(rms, 1.0, rtol=2e-6)
    # eps shrinks the rms to sqrt(ms / (ms + eps))
    eps = 0.5
    y2 = orc.rms_norm(x, None, eps=eps)
    ms = np.mean(x.astype(np.float64) ** 2, axis=1)
    np.testing.assert_allclose(np.sqrt(np.mean(y2.astype(np.float64) ** 2, axis=1)),
                               np.sqrt(ms / (ms + eps)), rtol=2e-6)
    # gains multiply element-wise after normalisation
    w = r.uniform(0.5, 1.5, n).astype(np.float32)
    yw = orc.rms_norm(x, w, eps=0.0)
    np.testing.assert_allclose(yw, y * w, rtol=2e-7, atol=0)


def test_rmsnorm_no_mean_subtraction_and_alias(orc):
    x = np.full((1, 8), -2.5, np.float32)
    y = orc.rms_norm(x, None, eps=0.0)
    np.testing.assert_array_equal(y, -np.ones_like(x))  # LayerNorm would give 0
    r = _rng(1)
    x = r.standard_normal((3, 64)).astype(np.float32)
    ref = orc.rms_norm(x, None, eps=1e-6)
    orc.rms_norm(x, None, eps=1e-6, out=x)  # y aliases x
    np.testing.assert_array_equal(x, ref)


def test_rmsnorm_scale_invariant(orc):
    r = _rng(2)
    x = r.standard_normal((4, 128)).astype(np.float32)
    np.testing.assert_array_equal(orc.rms_norm(x, None, eps=0.0), orc.rms_norm(x * 8.0, None, eps=0.0))


# --------------------------------------------------------------------------- RoPE
def test_rope_freq_table_properties(orc):
    g = _golden("rope_worked_example.json")
    f = orc.rope_freqs(g["hd"], g["base"], 1.0)
    np.testing.assert_array_equal(f, np.array(g["freqs_by_formula"], np.float32))
    for hd, theta, fs in [(64, 1e6, 1.0), (128, 1e6, 1.0), (128, 1e4, 0.25)]:
        f = orc.rope_freqs(hd, theta, fs).astype(np.float64)
        assert f[0] == np.float32(fs)                       # subspace 0 spins at freq_scale
        assert np.all(np.diff(f) < 0)                        # strictly slower
        ratios = f[1:] / f[:-1]                              # geometric with ratio theta^(-2/hd)
        np.testing.assert_allclose(ratios, theta ** (-2.0 / hd), rtol=2e-7)
        # the middle subspace (2i/hd = 1/2) turns at freq_scale / sqrt(theta)
        np.testing.assert_allclose(f[hd // 4], fs / math.sqrt(theta), rtol=6e-8)


def test_rope_pos0_identity_and_norms(orc):
    r = _rng(3)
    x = r.standard_normal((3, 4, 64)).astype(np.float32)
    y = orc.rope(x.copy(), [0, 0, 0], 4, 64, 1e6)
    np.testing.assert_array_equal(y, x)  # cos 0 = 1, sin 0 = 0: bit-exact
    pos = [5, 1000, 40960]
    for style in (0, 1):
        y = orc.rope(x.copy(), pos, 4, 64, 1e6, style=style)
        if style == 0:
            a, b = x[..., :32], x[..., 32:]
            ya, yb = y[..., :32], y[..., 32:]
        else:
            a, b = x[..., 0::2], x[..., 1::2]
            ya, yb = y[..., 0::2], y[..., 1::2]
        n0 = np.hypot(a.astype(np.float64), b.astype(np.float64))
        n1 = np.hypot(ya.astype(np.float64), yb.astype(np.float64))
        np.testing.assert_allclose(n1, n0, rtol=3e-7, atol=1e-7)


def test_rope_worked_example(orc):
    g = _golden("rope_worked_example.json")
    # NonInterleaved pairs for hd=4 are (0,2) and (1,3); put (1,0) in both
    x = np.array([[1.0, 1.0, 0.0, 0.0]], np.float32)
    y = orc.rope(x, [g["pos"]], 1, g["hd"], g["base"])[0]
    a0 = g["pair0_angle_rad"]
    a1 = g["pos"] * 0.01
    np.testing.assert_allclose(y, [math.cos(a0), math.cos(a1), math.sin(a0), math.sin(a1)],
                               rtol=0, atol=2e-7)


def test_rope_rotation_direction(orc):
    # hd = 2, freq_0 = freq_scale = pi/2, pos = 1: (1, 0) turns counter-clockwise to (0, 1)
    y = orc.rope(np.array([1.0, 0.0], np.float32), [1], 1, 2, 1e4, freq_scale=math.pi / 2)
    np.testing.assert_allclose(y, [0.0, 1.0], atol=1e-7)
    y = orc.rope(np.array([0.0, 1.0], np.float32), [1], 1, 2, 1e4, freq_scale=math.pi / 2)
    np.testing.assert_allclose(y, [-1.0, 0.0], atol=1e-7)


def test_rope_relative_position(orc):
    # q.k after RoPE depends only on m - n (11 · Attention..., §2.3)
    r = _rng(4)
    hd = 64
    q = r.standard_normal(hd).astype(np.float32)
    k = r.standard_normal(hd).astype(np.float32)
    dots = []
    for m, n in [(7, 3), (107, 103), (1007, 1003), (4, 0)]:
        qa = orc.rope(q.copy(), [m], 1, hd, 1e4)
        ka = orc.rope(k.copy(), [n], 1, hd, 1e4)
        dots.append(float(np.dot(qa.astype(np.float64), ka.astype(np.float64))))
    np.testing.assert_allclose(dots, dots[0], rtol=2e-4, atol=2e-4)
    qa = orc.rope(q.copy(), [9], 1, hd, 1e4)
    ka = orc.rope(k.copy(), [3], 1, hd, 1e4)
    assert abs(float(np.dot(qa, ka)) - dots[0]) > 1e-2  # a different offset does change it


def test_rope_styles_are_a_permutation(orc):
    r = _rng(5)
    hd, nh = 8, 3
    x = r.standard_normal((2, nh, hd)).astype(np.float32)
    perm = np.empty(hd, dtype=np.int64)  # NonInterleaved slot (i, i+half) -> Interleaved (2i, 2i+1)
    half = hd // 2
    for i in range(half):
        perm[2 * i] = i
        perm[2 * i + 1] = i + half
    y_non = orc.rope(x.copy(), [3, 11], nh, hd, 1e4, style=0)
    y_int = orc.rope(np.ascontiguousarray(x[..., perm]), [3, 11], nh, hd, 1e4, style=1)
    np.testing.assert_array_equal(y_int, y_non[..., perm])


# --------------------------------------------------------------------------- KV store
def test_kv_append_placement_and_errors(orc):
    r = _rng(6)
    cap, W = 10, 16
    k_reg = r.standard_normal((cap, W)).astype(np.float32)
    v_reg = r.standard_normal((cap, W)).astype(np.float32)
    k0, v0 = k_reg.copy(), v_reg.copy()
    k = r.standard_normal((3, W)).astype(np.float32)
    v = r.standard_normal((3, W)).astype(np.float32)
    orc.kv_append(k_reg, v_reg, k, v, [4, 9, 0])
    for t, p in enumerate([4, 9, 0]):
        np.testing.assert_array_equal(k_reg[p], k[t])
        np.testing.assert_array_equal(v_reg[p], v[t])
    untouched = [i for i in range(cap) if i not in (4, 9, 0)]
    np.testing.assert_array_equal(k_reg[untouched], k0[untouched])
    np.testing.assert_array_equal(v_reg[untouched], v0[untouched])
    # pos >= cap is an error, never a clamp; rows before it were written, rows after not
    k1, v1 = k_reg.copy(), v_reg.copy()
    st = orc.kv_append(k_reg, v_reg, k, v, [2, cap, 3], check=False)
    assert st == orc.ERR_POS
    np.testing.assert_array_equal(k_reg[2], k[0])
    np.testing.assert_array_equal(k_reg[3], k1[3])
    np.testing.assert_array_equal(v_reg[3], v1[3])
    assert orc.kv_append(k_reg, v_reg, k[:1], v[:1], [-1], check=False) == orc.ERR_POS


# --------------------------------------------------------------------------- attention
def _example_regions():
    g = _golden("attention_worked_examples.json")
    k = np.array(g["k_rows"], np.float32)
    v = np.array(g["v_rows"], np.float32)
    return g, k, v


def test_attention_worked_example_blend(orc):
    g, k, v = _example_regions()
    b = g["blend"]
    q = np.array([b["q"]], np.float32)
    out = orc.gqa_attn(q, k, v, [b["pos"]], 1, 1, 4, 4, scale=g["scale"])
    np.testing.assert_array_equal(out[0], np.array(b["out_printed"], np.float32))
    # with a masked third slot in the window (a second token at pos 2 makes nkv = 3)
    q2 = np.array([b["q"], [0, 0, 0, 0]], np.float32)
    out = orc.gqa_attn(q2, k, v, [b["pos"], 2], 1, 1, 4, 4, scale=g["scale"])
    np.testing.assert_array_equal(out[0], np.array(b["out_printed"], np.float32))


def test_attention_worked_example_tilt(orc):
    g, k, v = _example_regions()
    t = g["tilt"]
    out = orc.gqa_attn(np.array([t["q"]], np.float32), k, v, [t["pos"]], 1, 1, 4, 4, scale=g["scale"])
    w0 = 1.0 / (1.0 + math.exp(-0.5))
    w1 = 1.0 - w0
    exp = w0 * v[0].astype(np.float64) + w1 * v[1].astype(np.float64)
    np.testing.assert_allclose(out[0], exp, rtol=0, atol=1e-6)
    assert abs(w0 - t["weights_printed"][0]) > 0.1  # the printed weights are not the closed form


def test_attention_worked_example_decode_step(orc):
    g, k, v = _example_regions()
    d = g["decode_step"]
    # the three tokens of the page's decode example, as a 3-token prefill
    q = np.array([[1, 1, 0, 0], g["blend"]["q"], d["q"]], np.float32)
    out = orc.gqa_attn(q, k, v, [0, 1, 2], 1, 1, 4, 4, scale=g["scale"])
    np.testing.assert_array_equal(out[0], v[0])              # token 0 sees only row 0
    np.testing.assert_array_equal(out[1], np.array(g["blend"]["out_printed"], np.float32))
    e = math.exp(0.5)
    w = np.array([1.0, e, e]) / (1.0 + 2.0 * e)
    np.testing.assert_allclose(w, [0.23270, 0.38365, 0.38365], atol=5e-6)
    exp = w @ v.astype(np.float64)
    np.testing.assert_allclose(out[2], exp, rtol=0, atol=2e-6)
    assert abs(out[2][1] - 2.0) <= 2e-6
    # the same token as a decode step (nt = 1 at pos 2) gives the same row
    out_dec = orc.gqa_attn(q[2:3], k, v, [2], 1, 1, 4, 4, scale=g["scale"])
    np.testing.assert_array_equal(out_dec[0], out[2])


def test_single_cached_key_returns_its_value(orc):
    r = _rng(7)
    nh, nk, hd = 6, 2, 32
    q = r.standard_normal((1, nh, hd)).astype(np.float32)
    k = r.standard_normal((5, nk * hd)).astype(np.float32)
    v = r.standard_normal((5, nk * hd)).astype(np.float32)
    out = orc.gqa_attn(q, k, v, [0], nh, nk, hd, hd)
    for h in range(nh):
        hk = h // (nh // nk)
        np.testing.assert_array_equal(out[0, h * hd:(h + 1) * hd], v[0, hk * hd:(hk + 1) * hd])


def test_softmax_weights_sum_to_one(orc):
    r = _rng(8)
    nh, nk, hd, L = 4, 2, 64, 300
    q = r.standard_normal((1, nh, hd)).astype(np.float32) * 2
    k = r.standard_normal((L, nk * hd)).astype(np.float32)
    v = np.ones((L, nk * hd), np.float32)
    out = orc.gqa_attn(q, k, v, [L - 1], nh, nk, hd, hd)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=3e-6)


TINY_CASES = [
    # (nh, nk, hd, hdkv, cap, positions)
    (1, 1, 4, 4, 6, [0, 1, 2, 3, 4, 5]),          # MHA, full causal prefill
    (14, 2, 64, 64, 20, [19]),                    # Qwen2.5-0.5B geometry, one decode step
    (16, 8, 128, 128, 9, [3, 8, 0, 5]),           # Qwen3-0.6B geometry, scattered positions
    (6, 3, 16, 16, 7, [2, 2, 6]),                 # repeated positions
    (4, 2, 128, 64, 12, [11, 4]),                 # hd > hd_kv: dot over the first hd_kv
    (4, 4, 8, 8, 5, [7, 1]),                      # pos beyond the region: window clamps at cap
    (8, 1, 32, 32, 33, list(range(20, 33))),      # multi-query (one kv head)
]


@pytest.mark.parametrize("case", TINY_CASES)
def test_attention_matches_bruteforce(orc, case):
    nh, nk, hd, hdkv, cap, pos = case
    r = _rng(hash(str(case)) & 0xFFFF)
    nt = len(pos)
    q = r.standard_normal((nt, nh, hd)).astype(np.float32)
    k = r.standard_normal((cap, nk * hdkv)).astype(np.float32)
    v = r.standard_normal((cap, nk * hdkv)).astype(np.float32)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(hd)))
    out = orc.gqa_attn(q, k, v, pos, nh, nk, hd, hdkv, scale=scale)
    ref = orc.attn_bruteforce_f64(q, k, v, pos, nh, nk, hd, hdkv, scale)
    err = np.abs(out - ref)
    assert np.all(err <= 1e-5 + 1e-4 * np.abs(ref)), float(err.max())


def test_bruteforce_is_not_vacuous(orc):
    # a wrong kv-head mapping, a wrong window or a dropped scale would all move the
    # result by far more than the tolerance used above
    r = _rng(9)
    nh, nk, hd, cap = 4, 2, 16, 8
    q = r.standard_normal((2, nh, hd)).astype(np.float32)
    k = r.standard_normal((cap, nk * hd)).astype(np.float32)
    v = r.standard_normal((cap, nk * hd)).astype(np.float32)
    scale = 0.25
    ref = orc.attn_bruteforce_f64(q, k, v, [5, 7], nh, nk, hd, hd, scale)
    swapped = orc.attn_bruteforce_f64(q, k[:, ::-1].copy(), v[:, ::-1].copy(), [5, 7], nh, nk, hd, hd, scale)
    assert np.abs(ref - swapped).max() > 1e-2
    shorter = orc.attn_bruteforce_f64(q, k, v, [4, 7], nh, nk, hd, hd, scale)
    assert np.abs(ref[0] - shorter[0]).max() > 1e-2
    unscaled = orc.attn_bruteforce_f64(q, k, v, [5, 7], nh, nk, hd, hd, 1.0)
    assert np.abs(ref - unscaled).max() > 1e-2


def test_gqa_equals_mha_with_repeated_kv(orc):
    r = _rng(10)
    nh, nk, hd, cap = 14, 2, 64, 40
    g = nh // nk
    pos = [39, 17, 3]
    q = r.standard_normal((3, nh, hd)).astype(np.float32)
    k = r.standard_normal((cap, nk * hd)).astype(np.float32)
    v = r.standard_normal((cap, nk * hd)).astype(np.float32)
    rep = lambda a: np.repeat(a.reshape(cap, nk, hd), g, axis=1).reshape(cap, nh * hd)
    out_gqa = orc.gqa_attn(q, k, v, pos, nh, nk, hd, hd)
    out_mha = orc.gqa_attn(q, rep(k), rep(v), pos, nh, nh, hd, hd)
    np.testing.assert_array_equal(out_gqa, out_mha)


def test_prefill_equals_successive_decode_steps(orc):
    r = _rng(11)
    nh, nk, hd, nt = 8, 2, 32, 24
    q = r.standard_normal((nt, nh, hd)).astype(np.float32)
    k = r.standard_normal((nt + 4, nk * hd)).astype(np.float32)
    v = r.standard_normal((nt + 4, nk * hd)).astype(np.float32)
    pre = orc.gqa_attn(q, k, v, list(range(nt)), nh, nk, hd, hd)
    for t in range(nt):
        dec = orc.gqa_attn(q[t:t + 1], k, v, [t], nh, nk, hd, hd)
        np.testing.assert_array_equal(dec[0], pre[t])


def test_bit_identical_at_any_thread_count(orc):
    r = _rng(12)
    nh, nk, hd, nt = 16, 8, 128, 9
    q = r.standard_normal((nt, nh, hd)).astype(np.float32)
    k = r.standard_normal((64, nk * hd)).astype(np.float32)
    v = r.standard_normal((64, nk * hd)).astype(np.float32)
    pos = [63, 10, 0, 31, 32, 5, 60, 62, 1]
    ref = orc.gqa_attn(q, k, v, pos, nh, nk, hd, hd, n_threads=1)
    for n in (2, 3, 7, 16):
        np.testing.assert_array_equal(orc.gqa_attn(q, k, v, pos, nh, nk, hd, hd, n_threads=n), ref)


def test_masked_rows_contribute_nothing(orc):
    r = _rng(13)
    nh, nk, hd, cap = 2, 1, 8, 10
    q = r.standard_normal((2, nh, hd)).astype(np.float32)
    k = r.standard_normal((cap, nk * hd)).astype(np.float32)
    v = r.standard_normal((cap, nk * hd)).astype(np.float32)
    ref = orc.gqa_attn(q, k, v, [2, 5], nh, nk, hd, hd)
    k2, v2 = k.copy(), v.copy()
    k2[3:6] *= 1e3    # inside nkv = 6 but beyond token 0's window: weight exactly 0
    v2[3:6] = 1e30
    k2[6:] = np.nan   # beyond nkv: never read
    v2[6:] = np.nan
    out = orc.gqa_attn(q, k2, v2, [2, 5], nh, nk, hd, hd)
    np.testing.assert_array_equal(out[0], ref[0])


def test_geometry_errors(orc):
    q = np.zeros((1, 4, 8), np.float32)
    kv = np.zeros((4, 16), np.float32)
    with pytest.raises(orc.OracleError) as e:
        orc.gqa_attn(q, kv, kv, [0], 4, 1, 8, 16)   # hd < hd_kv is refused
    assert e.value.status == orc.ERR_GEOMETRY
    with pytest.raises(orc.OracleError) as e:
        orc.gqa_attn(np.zeros((1, 5, 8), np.float32), kv, kv, [0], 5, 2, 8, 8)
    assert e.value.status == orc.ERR_GEOMETRY


# --------------------------------------------------------------------------- SiLU, layer step
def test_silu_mul(orc):
    x = np.array([0.0, 1.0, -1.0, 20.0, -20.0, 3.5], np.float32)
    up = np.array([1.0, 2.0, 1.0, 1.0, 1.0, -1.0], np.float32)
    y = orc.silu_mul(x, up)
    exp = [v / (1.0 + math.exp(-v)) * u for v, u in zip(x.tolist(), up.tolist())]
    np.testing.assert_allclose(y, exp, rtol=3e-7, atol=1e-12)
    assert y[0] == 0.0


def test_silu_mul_closed_forms(orc):
    """Pins that do not restate the formula: sigma(ln 3) = 3/4 exactly, the reflection
    silu(-x) = silu(x) - x, the gate's minimum at x* = -1 - W(1/e) where silu(x*) = x* + 1
    (sigma(x*) = 1 + 1/x*), and up scaling the product linearly."""
    ln3 = math.log(3.0)
    x = np.array([ln3, -ln3], np.float32)
    y = orc.silu_mul(x, np.ones(2, np.float32))
    np.testing.assert_allclose(y, [float(x[0]) * 0.75, float(x[1]) * 0.25], rtol=2e-7)
    xs = np.linspace(-12.0, 12.0, 97).astype(np.float32)
    ones = np.ones_like(xs)
    yp, ym = orc.silu_mul(xs, ones), orc.silu_mul(-xs, ones)
    np.testing.assert_allclose(ym, yp - xs, atol=3e-6)
    # x* solves 1 + x(1 - sigma(x)) = 0, i.e. x* = -1 - W(1/e) with W(1/e) = 0.2784645427610738
    x_star = -1.2784645427610738
    y_star = orc.silu_mul(np.array([x_star, x_star - 0.01, x_star + 0.01], np.float32), np.ones(3, np.float32))
    assert abs(float(y_star[0]) - (x_star + 1.0)) < 1e-6
    assert y_star[1] > y_star[0] and y_star[2] > y_star[0]
    up = np.array([2.0, -3.0, 0.5], np.float32)
    g = np.array([0.7, -0.3, 5.0], np.float32)
    np.testing.assert_allclose(orc.silu_mul(g, up), orc.silu_mul(g, np.ones(3, np.float32)) * up, rtol=2e-7)


def test_layer_step_is_the_composition(orc):
    r = _rng(14)
    nh, nk, hd, hdkv, n_embd, cap = 4, 2, 16, 16, 24, 12
    nt = 3
    pos = [7, 8, 9]
    h = r.standard_normal((nt, n_embd)).astype(np.float32)
    gain = r.uniform(0.5, 1.5, n_embd).astype(np.float32)
    q = r.standard_normal((nt, nh * hd)).astype(np.float32)
    k = r.standard_normal((nt, nk * hdkv)).astype(np.float32)
    v = r.standard_normal((nt, nk * hdkv)).astype(np.float32)
    K = r.standard_normal((cap, nk * hdkv)).astype(np.float32)
    V = r.standard_normal((cap, nk * hdkv)).astype(np.float32)
    qs, ks, Ks, Vs = q.copy(), k.copy(), K.copy(), V.copy()
    xn, out = orc.layer_attn_step(h, gain, qs, ks, v, pos, Ks, Vs, n_head=nh, n_kv_head=nk, hd=hd,
                                  hd_kv=hdkv, eps=1e-6, theta=1e6)
    np.testing.assert_array_equal(xn, orc.rms_norm(h, gain, eps=1e-6))
    q2 = orc.rope(q.copy(), pos, nh, hd, 1e6)
    k2 = orc.rope(k.copy(), pos, nk, hdkv, 1e6)
    np.testing.assert_array_equal(qs, q2)
    np.testing.assert_array_equal(ks, k2)
    K2, V2 = K.copy(), V.copy()
    orc.kv_append(K2, V2, k2, v, pos)
    np.testing.assert_array_equal(Ks, K2)
    np.testing.assert_array_equal(Vs, V2)
    ref = orc.attn_bruteforce_f64(q2, K2, V2, pos, nh, nk, hd, hdkv, 1.0 / math.sqrt(hd))
    assert np.all(np.abs(out - ref) <= 1e-5 + 1e-4 * np.abs(ref))


# --------------------------------------------------------------------------- f16 cache
# "11 . Attention, vec ops, and the KV cache", §2.5: the GPU backends may keep the K/V regions
# in f16; the store converts and the attention read converts back.  The conversion is IEEE
# binary16, round to nearest even (the pages name no rounding); numpy's float16 cast is an
# independent implementation of the same definition.
def test_f16_conversion_closed_forms(orc):
    vals = {1.0: 0x3C00, -2.0: 0xC000, 65504.0: 0x7BFF, 2.0 ** -24: 0x0001, 2.0 ** -14: 0x0400,
            0.5: 0x3800, 1.0 + 2.0 ** -10: 0x3C01, 1.0 + 2.0 ** -11: 0x3C00,  # tie -> even
            1.0 + 3 * 2.0 ** -11: 0x3C02,  # tie -> even (up)
            65520.0: 0x7C00, 2.0 ** -25: 0x0000, 3 * 2.0 ** -25: 0x0002, float("inf"): 0x7C00}
    x = np.array(list(vals), np.float32)
    got = orc.f32_to_f16(x)
    assert [int(g) for g in got] == list(vals.values())
    exact = [1.0, -2.0, 65504.0, 2.0 ** -24, 2.0 ** -14, 0.5, 1.0 + 2.0 ** -10]
    np.testing.assert_array_equal(orc.f16_to_f32(orc.f32_to_f16(np.array(exact, np.float32))),
                                  np.array(exact, np.float32))
    assert np.isnan(orc.f16_to_f32(np.array([0x7E00], np.uint16)))[0]
    assert np.isnan(orc.f16_to_f32(orc.f32_to_f16(np.array([np.nan], np.float32))))[0]


def test_f16_conversion_matches_the_format_everywhere(orc):
    r = _rng(40)
    mag = np.exp2(r.uniform(-30, 17, 200000)).astype(np.float32)
    x = np.concatenate([mag, -mag, r.standard_normal(50000).astype(np.float32),
                        np.array([0.0, -0.0, 65519.996, 65520.0, 1e30, -1e30, 6.0e-8, 5.9e-8],
                                 np.float32)])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(orc.f32_to_f16(x), ref)
    # every bit pattern reads back as numpy reads it
    allh = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.f16_to_f32(allh)
    ref = allh.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_kv_append_f16_placement_and_errors(orc):
    r = _rng(41)
    cap, W = 9, 16
    k_reg = orc.f32_to_f16(r.standard_normal((cap, W)).astype(np.float32))
    v_reg = orc.f32_to_f16(r.standard_normal((cap, W)).astype(np.float32))
    k0, v0 = k_reg.copy(), v_reg.copy()
    k = (r.standard_normal((3, W)) * 100).astype(np.float32)
    v = r.standard_normal((3, W)).astype(np.float32)
    orc.kv_append_f16(k_reg, v_reg, k, v, [5, 8, 0])
    for t, p in enumerate([5, 8, 0]):
        np.testing.assert_array_equal(k_reg[p], k[t].astype(np.float16).view(np.uint16))
        np.testing.assert_array_equal(v_reg[p], v[t].astype(np.float16).view(np.uint16))
    untouched = [i for i in range(cap) if i not in (5, 8, 0)]
    np.testing.assert_array_equal(k_reg[untouched], k0[untouched])
    np.testing.assert_array_equal(v_reg[untouched], v0[untouched])
    k1 = k_reg.copy()
    assert orc.kv_append_f16(k_reg, v_reg, k, v, [1, cap, 2], check=False) == orc.ERR_POS
    np.testing.assert_array_equal(k_reg[2], k1[2])
    assert orc.kv_append_f16(k_reg, v_reg, k[:1], v[:1], [-1], check=False) == orc.ERR_POS


def test_f16_layer_step_equals_f32_step_on_representable_values(orc):
    # At pos 0 RoPE is the identity, so with k, v and the cached rows already binary16 values the
    # f16 store loses nothing: the f16 step must equal the fp32 step bit for bit.
    r = _rng(42)
    nh, nk, hd, hdkv, n_embd, cap = 4, 2, 16, 16, 24, 6
    f16 = lambda a: a.astype(np.float16).astype(np.float32)
    h = r.standard_normal((1, n_embd)).astype(np.float32)
    gain = r.uniform(0.5, 1.5, n_embd).astype(np.float32)
    q = r.standard_normal((1, nh * hd)).astype(np.float32)
    k = f16(r.standard_normal((1, nk * hdkv)))
    v = f16(r.standard_normal((1, nk * hdkv)))
    K = f16(r.standard_normal((cap, nk * hdkv)))
    V = f16(r.standard_normal((cap, nk * hdkv)))
    pos = [0]
    K16, V16 = orc.f32_to_f16(K), orc.f32_to_f16(V)
    xa, oa = orc.layer_attn_step(h, gain, q.copy(), k.copy(), v, pos, K.copy(), V.copy(), n_head=nh,
                                 n_kv_head=nk, hd=hd, hd_kv=hdkv)
    xb, ob = orc.layer_attn_step_f16(h, gain, q.copy(), k.copy(), v, pos, K16, V16, n_head=nh,
                                     n_kv_head=nk, hd=hd, hd_kv=hdkv)
    np.testing.assert_array_equal(xa, xb)
    np.testing.assert_array_equal(oa, ob)
    np.testing.assert_array_equal(K16[0], orc.f32_to_f16(k[0]))


def test_f16_layer_step_reads_what_it_stored(orc):
    # Anywhere else the f16 step is the fp32 attention over the regions it leaves behind: the
    # brute-force fp64 attention over the stored (rounded) values agrees within fp32 tolerance,
    # and the rounding moves the output by no more than binary16 precision allows.
    r = _rng(43)
    nh, nk, hd, hdkv, n_embd, cap = 6, 2, 32, 32, 40, 20
    nt, pos = 3, [11, 12, 13]
    h = r.standard_normal((nt, n_embd)).astype(np.float32)
    gain = np.ones(n_embd, np.float32)
    q = r.standard_normal((nt, nh * hd)).astype(np.float32)
    k = r.standard_normal((nt, nk * hdkv)).astype(np.float32)
    v = r.standard_normal((nt, nk * hdkv)).astype(np.float32)
    K = r.standard_normal((cap, nk * hdkv)).astype(np.float32)
    V = r.standard_normal((cap, nk * hdkv)).astype(np.float32)
    K16, V16 = orc.f32_to_f16(K), orc.f32_to_f16(V)
    qs = q.copy()
    _, out = orc.layer_attn_step_f16(h, gain, qs, k.copy(), v, pos, K16, V16, n_head=nh, n_kv_head=nk,
                                     hd=hd, hd_kv=hdkv)
    ref = orc.attn_bruteforce_f64(qs, orc.f16_to_f32(K16), orc.f16_to_f32(V16), pos, nh, nk, hd, hdkv,
                                  1.0 / math.sqrt(hd))
    assert np.all(np.abs(out - ref) <= 1e-5 + 1e-4 * np.abs(ref))
    _, out32 = orc.layer_attn_step(h, gain, q.copy(), k.copy(), v, pos, K.copy(), V.copy(), n_head=nh,
                                   n_kv_head=nk, hd=hd, hd_kv=hdkv)
    d = np.abs(out - out32)
    assert d.max() < 2e-2 and d.max() > 0  # binary16 keeps ~3 decimal digits, and it is not a no-op


# --------------------------------------------------------------------------- paged regions
# "IV.2: Zero-copy KV cache": the paged cache keeps a sequence as scattered fixed-size blocks;
# "13 . The decode loop and graph reuse", §2.2: the attention reads the cells a window names.
# Reading through a block table must give exactly what the same rows give contiguously, in
# whatever order the blocks sit in the pool.
def _paged_case(r, n_seq, max_blocks, block_rows, W, shuffle):
    n_blocks = n_seq * max_blocks
    regions = r.standard_normal((n_seq, max_blocks * block_rows, W)).astype(np.float32)
    perm = r.permutation(n_blocks) if shuffle else np.arange(n_blocks)
    pool = np.empty((n_blocks * block_rows, W), np.float32)
    table = np.empty((n_seq, max_blocks), np.int32)
    for s in range(n_seq):
        for b in range(max_blocks):
            phys = int(perm[s * max_blocks + b])
            table[s, b] = phys
            pool[phys * block_rows:(phys + 1) * block_rows] = regions[s, b * block_rows:(b + 1) * block_rows]
    return regions, pool, table


@pytest.mark.parametrize("shuffle", [False, True])
def test_paged_attention_equals_contiguous(orc, shuffle):
    r = _rng(60 + shuffle)
    nh, nk, hd, hdkv, block_rows, max_blocks, n_seq = 6, 2, 16, 16, 4, 5, 3
    W = nk * hdkv
    K, Kp, table = _paged_case(r, n_seq, max_blocks, block_rows, W, shuffle)
    V, Vp, _ = _paged_case(np.random.default_rng(99), n_seq, max_blocks, block_rows, W, False)
    # V follows the same table as K
    Vp = np.empty_like(Kp)
    for s in range(n_seq):
        for b in range(max_blocks):
            Vp[table[s, b] * block_rows:(table[s, b] + 1) * block_rows] = V[s, b * block_rows:(b + 1) * block_rows]
    q = r.standard_normal((n_seq, nh, hd)).astype(np.float32)
    pos = np.array([0, 9, 19], np.int32)  # one row, a partial block, the whole table
    got = orc.gqa_attn_paged(q, Kp, Vp, table, block_rows, pos, nh, nk, hd, hdkv, scale=0.25)
    for s in range(n_seq):
        ref = orc.gqa_attn(q[s:s + 1], K[s], V[s], [pos[s]], nh, nk, hd, hdkv, scale=0.25)
        np.testing.assert_array_equal(got[s:s + 1], ref)
    # a window past the table is clamped to it, like a region's cap
    far = orc.gqa_attn_paged(q, Kp, Vp, table, block_rows, [50, 50, 50], nh, nk, hd, hdkv, scale=0.25)
    np.testing.assert_array_equal(far[2:], got[2:])


def test_paged_append_places_rows_and_reports_missing_blocks(orc):
    r = _rng(62)
    block_rows, max_blocks, n_seq, W = 4, 3, 2, 8
    _, Kp, table = _paged_case(r, n_seq, max_blocks, block_rows, W, True)
    Vp = Kp.copy()
    K0 = Kp.copy()
    k = r.standard_normal((n_seq, W)).astype(np.float32)
    v = r.standard_normal((n_seq, W)).astype(np.float32)
    pos = [5, 11]
    orc.kv_append_paged(Kp, Vp, table, block_rows, k, v, pos)
    for s, p in enumerate(pos):
        row = table[s, p // block_rows] * block_rows + p % block_rows
        np.testing.assert_array_equal(Kp[row], k[s])
        np.testing.assert_array_equal(Vp[row], v[s])
    changed = np.flatnonzero(np.any(Kp != K0, axis=1))
    assert sorted(changed) == sorted(table[s, p // block_rows] * block_rows + p % block_rows
                                     for s, p in enumerate(pos))
    missing = table.copy()
    missing[0, 1] = -1
    assert orc.kv_append_paged(Kp, Vp, missing, block_rows, k, v, [5, 0], check=False) == orc.ERR_POS
    assert orc.kv_append_paged(Kp, Vp, table, block_rows, k, v, [12, 0], check=False) == orc.ERR_POS
    with pytest.raises(orc.OracleError):
        orc.gqa_attn_paged(r.standard_normal((2, 2, 8)).astype(np.float32), Kp, Vp, missing, block_rows, [6, 0],
                           2, 1, 8, 8)


# --------------------------------------------------------------------------- Q8_0 cache
# "11 . Attention, vec ops, and the KV cache", §2.5: Q8_0 block rows, 32 values to a block of one
# f16 scale and 32 int8 quants (34 bytes), 3.76x smaller than f32; the store quantizes and the
# read dequantizes.  Quantizer: d = max|x|/127, q = round(x/d), halves away from zero.
def _q8_parts(q, W):
    quants = q[:, :W].view(np.int8)
    scales = q[:, W:W + W // 16].copy().view(np.uint16)
    return quants, scales


def test_q8_row_layout_and_size(orc):
    assert orc.q8_row_bytes(1024) == 1088          # 32 blocks of 34 bytes: the pages' 3.76x
    assert 4 * 1024 / orc.q8_row_bytes(1024) == pytest.approx(3.7647, abs=1e-4)
    assert orc.q8_row_bytes(128) == 144             # 136 bytes, padded to a multiple of 16
    assert orc.q8_row_bytes(64) == 80
    x = _rng(70).standard_normal((3, 128)).astype(np.float32)
    q = orc.q8_quantize(x)
    assert q.shape == (3, 144) and not q[:, 136:].any()  # the padding is zero


def test_q8_exact_when_the_block_is_on_the_grid(orc):
    # values k * 2^-5 with max |k| = 127: d = 2^-5 exactly, so q = k and the read-back is exact
    r = _rng(71)
    k = r.integers(-127, 128, size=(4, 64))
    k[:, 0] = 127
    k[:, 32] = -127
    x = (k * 2.0 ** -5).astype(np.float32)
    q = orc.q8_quantize(x)
    quants, scales = _q8_parts(q, 64)
    np.testing.assert_array_equal(quants, k)
    assert np.all(scales == 0x2800)                  # binary16 of 2^-5
    np.testing.assert_array_equal(orc.q8_dequant(q, 64), x)


def test_q8_rounding_ties_zero_blocks_and_symmetry(orc):
    x = np.zeros((2, 32), np.float32)
    x[0, :4] = [127.0, 2.5, -2.5, 0.5]               # d = 1: halves round away from zero
    q = orc.q8_quantize(x)
    quants, scales = _q8_parts(q, 32)
    assert list(quants[0, :4]) == [127, 3, -3, 1]
    assert scales[0, 0] == 0x3C00 and scales[1, 0] == 0 and not quants[1].any()  # an all-zero block
    np.testing.assert_array_equal(orc.q8_dequant(q, 32)[1], np.zeros(32, np.float32))
    y = _rng(72).standard_normal((5, 96)).astype(np.float32)
    qa, qb = orc.q8_quantize(y), orc.q8_quantize(-y)
    np.testing.assert_array_equal(_q8_parts(qa, 96)[0], -_q8_parts(qb, 96)[0].astype(np.int16))
    np.testing.assert_array_equal(_q8_parts(qa, 96)[1], _q8_parts(qb, 96)[1])


def test_q8_error_bound(orc):
    # |x - x'| <= d/2 from the rounding, plus |q| * |f16(d) - d| from the scale, where binary16
    # rounds d to within half an ulp: 2^-11 * d for normal scales, 2^-25 for subnormal ones
    r = _rng(73)
    x = (r.standard_normal((200, 256)) * np.exp2(r.uniform(-10, 10, (200, 1)))).astype(np.float32)
    back = orc.q8_dequant(orc.q8_quantize(x), 256)
    d = np.abs(x).reshape(200, 8, 32).max(axis=2) / 127.0
    bound = np.repeat((0.5 * d + 127 * np.maximum(2.0 ** -11 * d, 2.0 ** -25)) * (1 + 1e-5), 32, axis=1)
    assert np.all(np.abs(back - x) <= bound)
    assert np.abs(back - x).max() > 0                # and it is not a copy


def test_kv_append_q8_placement_and_errors(orc):
    r = _rng(74)
    cap, W = 7, 64
    rb = orc.q8_row_bytes(W)
    K0 = r.integers(0, 256, size=(cap, rb)).astype(np.uint8)
    Kr, Vr = K0.copy(), K0.copy()
    k = r.standard_normal((2, W)).astype(np.float32)
    v = r.standard_normal((2, W)).astype(np.float32)
    orc.kv_append_q8(Kr, Vr, W, k, v, [6, 1])
    np.testing.assert_array_equal(Kr[[6, 1]], orc.q8_quantize(k))
    np.testing.assert_array_equal(Vr[[6, 1]], orc.q8_quantize(v))
    keep = [0, 2, 3, 4, 5]
    np.testing.assert_array_equal(Kr[keep], K0[keep])
    assert orc.kv_append_q8(Kr, Vr, W, k, v, [cap, 0], check=False) == orc.ERR_POS
    assert orc.kv_append_q8(Kr, Vr, W, k[:1], v[:1], [-1], check=False) == orc.ERR_POS


# --------------------------------------------------------------------------- fused QKV op
# "13 . The decode loop and graph reuse", §2.3: the fused QKV op merges the three projections,
# their biases, the two RoPEs and the two KV stores.  Pins: the projections against numpy's
# float64 matmul (an independent implementation), selection weights that reduce the op to the
# already-pinned RMSNorm, RoPE and store, and the store's placement.
def _qkv_case(r, nt=2, nh=4, nk=2, hd=16, hdkv=16, n_embd=48):
    n_out = nh * hd + 2 * nk * hdkv
    h = r.standard_normal((nt, n_embd)).astype(np.float32)
    gain = r.uniform(0.5, 1.5, n_embd).astype(np.float32)
    w = (r.standard_normal((n_out, n_embd)) / np.sqrt(n_embd)).astype(np.float32)
    b = r.standard_normal(n_out).astype(np.float32)
    return h, gain, w, b, (nh, nk, hd, hdkv)


def test_fused_qkv_projection_matches_float64_matmul(orc):
    r = _rng(80)
    h, gain, w, b, (nh, nk, hd, hdkv) = _qkv_case(r)
    cap, W = 10, nk * hdkv
    K, V = np.zeros((cap, W), np.float32), np.zeros((cap, W), np.float32)
    xn, q, k, v = orc.fused_qkv(h, gain, w, b, [0, 0], K, V, n_head=nh, n_kv_head=nk, hd=hd, hd_kv=hdkv)
    np.testing.assert_array_equal(xn, orc.rms_norm(h, gain, eps=1e-6))
    y = (xn.astype(np.float64) @ w.astype(np.float64).T).astype(np.float32) + b  # pos 0: RoPE is the identity
    nq = nh * hd
    np.testing.assert_allclose(q, y[:, :nq], rtol=0, atol=4e-7 * np.abs(y).max())
    np.testing.assert_allclose(k, y[:, nq:nq + W], rtol=0, atol=4e-7 * np.abs(y).max())
    np.testing.assert_allclose(v, y[:, nq + W:], rtol=0, atol=4e-7 * np.abs(y).max())


def test_fused_qkv_with_selection_weights_is_rmsnorm_rope_store(orc):
    r = _rng(81)
    h, gain, _, b, (nh, nk, hd, hdkv) = _qkv_case(r, n_embd=64)
    n_embd = h.shape[1]
    nq, W = nh * hd, nk * hdkv
    n_out = nq + 2 * W
    sel = r.integers(0, n_embd, size=n_out)
    w = np.zeros((n_out, n_embd), np.float32)
    w[np.arange(n_out), sel] = 1.0                    # output j picks xn[sel[j]] exactly
    cap, pos = 12, [3, 7]
    K, V = r.standard_normal((cap, W)).astype(np.float32), r.standard_normal((cap, W)).astype(np.float32)
    K0, V0 = K.copy(), V.copy()
    xn, q, k, v = orc.fused_qkv(h, gain, w, b, pos, K, V, n_head=nh, n_kv_head=nk, hd=hd, hd_kv=hdkv)
    y = xn[:, sel] + b
    np.testing.assert_array_equal(q, orc.rope(y[:, :nq].copy(), pos, nh, hd, 1e6))
    np.testing.assert_array_equal(k, orc.rope(y[:, nq:nq + W].copy(), pos, nk, hdkv, 1e6))
    np.testing.assert_array_equal(v, y[:, nq + W:])
    orc.kv_append(K0, V0, k, v, pos)
    np.testing.assert_array_equal(K, K0)
    np.testing.assert_array_equal(V, V0)
    # without a bias the outputs are the selected values themselves
    _, q2, _, _ = orc.fused_qkv(h, gain, w, None, [0, 0], K, V, n_head=nh, n_kv_head=nk, hd=hd, hd_kv=hdkv)
    np.testing.assert_array_equal(q2, xn[:, sel[:nq]])
