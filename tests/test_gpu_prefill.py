"""GPU parity of the tensor-core causal prefill (QK^T on tcgen05 with binary16 hi/lo halves of
power-of-two-scaled rows, PV with TF32 hi/lo halves, fp32 softmax) against the CPU oracle.  Two
bounds: the tensor-core tolerance (max-abs 2e-3), and -- because the hi/lo operand split makes
the products fp32-accurate -- the fp32 tolerance |d| <= 1e-5 + 1e-4 |ref| used for the
CUDA-core kernels.  Window and error handling are exact."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

TC_ATOL = 2e-3


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gqa_attention_kv_rope_gb300 as pkg
    from gqa_attention_kv_rope_gb300 import build

    build.build()
    pkg.binding.lib()
    return pkg


def rnd(shape, seed):
    return torch.randn(*shape, generator=torch.Generator().manual_seed(seed))


def run_prefill(m, q, K, V, pos, nh, nk, hd, hdkv):
    nt = len(pos)
    out = torch.full((nt, nh * hdkv), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = float(np.float32(1.0) / np.sqrt(np.float32(hd)))
    ws = m.kv.prefill_workspace(nt, nh, nk, hdkv, K.shape[0])
    m.minf_gqa_attn_prefill(out, q.contiguous().cuda(), K.cuda(), V.cuda(),
                            torch.as_tensor(np.asarray(pos, np.int32)).cuda(), nh, nk, hd, hdkv, scale, ws, err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(err.item()), scale


def close32(got, ref, what):
    """CUDA-core outputs (RMSNorm, rotations, stored K rows): |d| <= 1e-5 + 1e-4 |ref| element by element."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    d = np.abs(got - ref)
    bad = d > 1e-5 + 1e-4 * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} elements off, max abs {d.max():.3g}"


def check(got, ref, what):
    d = np.abs(got.astype(np.float64) - ref)
    assert np.isfinite(got).all(), what
    print(f"[prefill error] {what}: max abs {d.max():.3g}, max rel-bound {np.max(d / (1e-5 + 1e-4 * np.abs(ref))):.3g}")
    assert d.max() <= TC_ATOL, f"{what}: max abs {d.max():.3g}"
    assert np.all(d <= 1e-5 + 1e-4 * np.abs(ref)), f"{what}: outside the fp32 tolerance"


@pytest.mark.parametrize("geom", [
    (14, 2, 64, 64, 512, 1024),     # causal prefill, Qwen2.5-0.5B shape (one layer)
    (16, 8, 128, 128, 511, 1023),   # the decode loop's 511-token prefill, Qwen3-0.6B shape
    (4, 2, 64, 64, 77, 80),         # ragged tile, window close to the region end
    (8, 8, 128, 128, 1, 16),        # a single token
    (6, 2, 128, 64, 130, 200),      # hd > hd_kv: q head stride hd, dot over the first hd_kv
])
def test_prefill_causal(m, orc, geom):
    nh, nk, hd, hdkv, nt, cap = geom
    K = rnd((cap, nk * hdkv), nt)
    V = rnd((cap, nk * hdkv), nt + 1)
    q = rnd((nt, nh, hd), nt + 2)
    pos = np.arange(nt, dtype=np.int32)
    got, err, scale = run_prefill(m, q, K, V, pos, nh, nk, hd, hdkv)
    ref = orc.attn_bruteforce_f64(q.numpy(), K.numpy(), V.numpy(), pos, nh, nk, hd, hdkv, scale)
    assert err == 0
    check(got, ref, f"prefill {geom}")
    fp32 = orc.gqa_attn(q.numpy(), K.numpy(), V.numpy(), pos, nh, nk, hd, hdkv, scale=scale, n_threads=8)
    check(got, fp32, f"prefill vs fp32 oracle {geom}")


def test_prefill_continues_an_existing_cache(m, orc):
    """Delta prefill: 64 new tokens at positions 200..263 over 200 cached rows."""
    nh, nk, hd, cap = 16, 8, 128, 300
    K = rnd((cap, nk * hd), 5)
    V = rnd((cap, nk * hd), 6)
    q = rnd((64, nh, hd), 7)
    pos = np.arange(200, 264, dtype=np.int32)
    got, err, scale = run_prefill(m, q, K, V, pos, nh, nk, hd, hd)
    assert err == 0
    check(got, orc.gqa_attn(q.numpy(), K.numpy(), V.numpy(), pos, nh, nk, hd, hd, scale=scale, n_threads=8),
          "delta prefill")


def test_prefill_repeated_calls_reuse_the_workspace(m, orc):
    """Long windows split over several key chunks; back-to-back calls share one workspace."""
    nh, nk, hd, cap = 16, 8, 128, 2048
    K = rnd((cap, nk * hd), 11)
    V = rnd((cap, nk * hd), 12)
    for i, nt in enumerate((700, 1500)):
        q = rnd((nt, nh, hd), 13 + i)
        pos = np.arange(cap - nt, cap, dtype=np.int32)  # continue a long cache: windows up to 2048
        got, err, scale = run_prefill(m, q, K, V, pos, nh, nk, hd, hd)
        assert err == 0
        check(got, orc.gqa_attn(q.numpy(), K.numpy(), V.numpy(), pos, nh, nk, hd, hd, scale=scale, n_threads=8),
              f"long-window prefill {nt}")


def test_prefill_long_windows_hd64(m, orc):
    """hd_kv 64 (two K, V^T and P buffers) with windows of 1449..2048 keys: 12 to 16 key chunks
    per query tile, all folded by the last chunk to arrive."""
    nh, nk, hd, cap, nt = 8, 2, 64, 2048, 600
    K = rnd((cap, nk * hd), 21)
    V = rnd((cap, nk * hd), 22)
    q = rnd((nt, nh, hd), 23)
    pos = np.arange(cap - nt, cap, dtype=np.int32)
    got, err, scale = run_prefill(m, q, K, V, pos, nh, nk, hd, hd)
    assert err == 0
    check(got, orc.gqa_attn(q.numpy(), K.numpy(), V.numpy(), pos, nh, nk, hd, hd, scale=scale, n_threads=8),
          "long-window prefill hd_kv 64")


def test_prefill_scattered_positions_and_bad_ones(m, orc):
    nh, nk, hd, cap = 8, 2, 64, 150
    K = rnd((cap, nk * hd), 8)
    V = rnd((cap, nk * hd), 9)
    pos = np.array([5, 149, 0, 77, 160, 33, -1, 120], np.int32)  # 160 >= cap clamps, -1 is empty
    q = rnd((len(pos), nh, hd), 10)
    got, err, scale = run_prefill(m, q, K, V, pos, nh, nk, hd, hd)
    assert err & m.ERRBIT_ATTN_POS and not err & m.ERRBIT_TIMEOUT
    ok = pos >= 0
    ref = orc.gqa_attn(q.numpy()[ok], K.numpy(), V.numpy(), pos[ok], nh, nk, hd, hd, scale=scale)
    check(got[ok], ref, "scattered positions")
    assert np.all(got[~ok] == 0.0)


def test_prefill_layer_step_matches_oracle(m, orc):
    """Causal prefill through the layer step (RMSNorm, RoPE + store, tensor-core attention)."""
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN25_05B
    nt, cap = 512, 1024
    x = wl.layer_inputs(g, "prefill", 3, nt)
    d = {k: v.cuda() for k, v in x.items()}
    K = torch.zeros(cap, g.row_width, device="cuda")
    V = torch.zeros(cap, g.row_width, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    xn = torch.empty_like(d["h"])
    out = torch.empty(nt, g.out_width, device="cuda")
    pos = torch.arange(nt, dtype=torch.int32, device="cuda")
    ws = m.kv.prefill_workspace(nt, g.n_head, g.n_kv_head, g.hd_kv, cap)
    m.minf_layer_attn_step(xn, d["h"], d["gain"], g.eps, d["q"], d["k"], d["v"], pos, K, V, g.n_head, g.n_kv_head,
                           g.hd, g.hd_kv, g.theta, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    q, k = x["q"].numpy().copy(), x["k"].numpy().copy()
    Ko = np.zeros((cap, g.row_width), np.float32)
    Vo = np.zeros((cap, g.row_width), np.float32)
    xn_ref, out_ref = orc.layer_attn_step(x["h"].numpy(), x["gain"].numpy(), q, k, x["v"].numpy(), np.arange(nt),
                                          Ko, Vo, n_head=g.n_head, n_kv_head=g.n_kv_head, hd=g.hd, hd_kv=g.hd_kv,
                                          eps=g.eps, theta=g.theta, n_threads=8)
    assert err.item() == 0
    check(out.cpu().numpy(), out_ref, "layer step out")
    assert np.array_equal(V.cpu().numpy(), Vo)
    close32(xn.cpu().numpy(), xn_ref, "xn")
    close32(d["q"].cpu().numpy(), q, "q rotated")
    close32(d["k"].cpu().numpy(), k, "k rotated")
    close32(K.cpu().numpy(), Ko, "K region")
