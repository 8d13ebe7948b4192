"""GPU parity of the fused QKV decode op ("13 . The decode loop and graph reuse", §2.3: the
three projections, their biases, the two RoPEs and the two KV stores as one op; here with the
RMSNorm in front), for the two model shapes and a wide one.  Synthetic weights ~ N(0, 1/n_embd) and biases ~ N(0, 1): outputs within
1e-5 + 1e-4|ref| of the oracle (double-accumulated projections); V rows stored as computed
(compared with the oracle at the same tolerance); the attention after the op against the
oracle's attention over the regions the GPU left."""
from types import SimpleNamespace

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-5, 1e-4


@pytest.fixture(scope="module")
def m():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gqa_attention_kv_rope_gb300 as pkg
    from gqa_attention_kv_rope_gb300 import build

    build.build()
    pkg.binding.lib()
    return pkg


def close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    d = np.abs(got - ref)
    bad = d > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off, max abs {d.max():.3g}"


def rnd(shape, seed, scale=1.0):
    return (torch.randn(*shape, generator=torch.Generator().manual_seed(seed)) * scale).numpy()


def dev(x):
    return None if x is None else torch.as_tensor(np.ascontiguousarray(x)).cuda()


def err_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _case(g, nt, seed, bias=True):
    n_out = g.q_width + 2 * g.row_width
    h = rnd((nt, g.n_embd), seed)
    gain = np.random.default_rng(seed).uniform(0.5, 1.5, g.n_embd).astype(np.float32)
    w = rnd((n_out, g.n_embd), seed + 1, scale=1.0 / np.sqrt(g.n_embd))
    b = rnd((n_out,), seed + 2) if bias else None
    return h, gain, w, b


# A wide geometry (n_embd 4096: four 128-bit loads a lane per weight row) beside the two model
# shapes.
WIDE = SimpleNamespace(n_embd=4096, n_head=32, n_kv_head=8, hd=128, hd_kv=128, eps=1e-6, theta=1e6,
                       q_width=32 * 128, row_width=8 * 128)


def geometry(which):
    from gqa_attention_kv_rope_gb300 import workloads as wl

    return {"qwen25": wl.QWEN25_05B, "qwen3": wl.QWEN3_06B, "wide": WIDE}[which]


@pytest.mark.parametrize("which,nt,bias,style", [("qwen25", 1, True, 0), ("qwen3", 1, False, 0),
                                                 ("qwen3", 7, True, 0), ("qwen25", 16, True, 1),
                                                 ("qwen3", 3, True, 1), ("wide", 1, True, 0),
                                                 ("wide", 5, False, 1), ("wide", 13, True, 0)])
def test_fused_qkv(m, orc, which, nt, bias, style):
    g = geometry(which)
    cap = 900
    h, gain, w, b = _case(g, nt, 10 + nt, bias)
    pos = np.sort(np.random.default_rng(nt).choice(cap, nt, replace=False)).astype(np.int32)
    K0, V0 = rnd((cap, g.row_width), 20), rnd((cap, g.row_width), 21)
    Kd, Vd = dev(K0), dev(V0)
    xn = torch.empty(nt, g.n_embd, device="cuda")
    q = torch.empty(nt, g.q_width, device="cuda")
    k = torch.empty(nt, g.row_width, device="cuda")
    v = torch.empty(nt, g.row_width, device="cuda")
    err = err_word()
    m.minf_fused_qkv(xn, dev(h), dev(gain), g.eps, dev(w), dev(b), dev(pos), q, k, v, Kd, Vd, g.n_head, g.n_kv_head,
                     g.hd, g.hd_kv, g.theta, 1.0, style, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    Ko, Vo = K0.copy(), V0.copy()
    xn_r, q_r, k_r, v_r = orc.fused_qkv(h, gain, w, b, pos, Ko, Vo, n_head=g.n_head, n_kv_head=g.n_kv_head, hd=g.hd,
                                        hd_kv=g.hd_kv, eps=g.eps, theta=g.theta, style=style)
    close(xn.cpu().numpy(), xn_r, what="xn")
    close(q.cpu().numpy(), q_r, what="q")
    kg, vg = k.cpu().numpy(), v.cpu().numpy()
    close(kg, k_r, what="k")
    close(vg, v_r, what="v")
    Kn, Vn = Kd.cpu().numpy(), Vd.cpu().numpy()
    assert np.array_equal(Kn[pos], kg) and np.array_equal(Vn[pos], vg)  # stored exactly what it returned
    keep = np.setdiff1d(np.arange(cap), pos)
    assert np.array_equal(Kn[keep], K0[keep]) and np.array_equal(Vn[keep], V0[keep])


def test_fused_qkv_too_wide(m):
    """16 tokens of 4096 values are 256 KB of normalized inputs: more shared memory than a CTA
    has, refused on the host before any launch."""
    g, nt = WIDE, 16
    h, gain, w, b = _case(g, nt, 50)
    bufs = [torch.empty(nt, n, device="cuda") for n in (g.n_embd, g.q_width, g.row_width, g.row_width)]
    Kd = dev(rnd((8, g.row_width), 51))
    err = err_word()
    with pytest.raises(m.binding.MinfError) as e:
        m.minf_fused_qkv(bufs[0], dev(h), dev(gain), g.eps, dev(w), dev(b), dev(np.arange(nt, dtype=np.int32) % 8),
                         *bufs[1:], Kd, Kd.clone(), g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, err)
    assert e.value.status == 3
    torch.cuda.synchronize()
    assert err.item() == 0


def test_fused_qkv_position_errors(m):
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN3_06B
    cap = 64
    h, gain, w, b = _case(g, 2, 30)
    K0 = rnd((cap, g.row_width), 31)
    Kd, Vd = dev(K0), dev(K0)
    bufs = [torch.empty(2, n, device="cuda") for n in (g.n_embd, g.q_width, g.row_width, g.row_width)]
    err = err_word()
    m.minf_fused_qkv(bufs[0], dev(h), dev(gain), g.eps, dev(w), dev(b), dev(np.array([-1, cap], np.int32)), *bufs[1:],
                     Kd, Vd, g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, err)
    torch.cuda.synchronize()
    assert err.item() == 0x1 | 0x2  # not rotated (pos < 0), not stored (both)
    assert np.array_equal(Kd.cpu().numpy(), K0) and np.array_equal(Vd.cpu().numpy(), K0)


def test_fused_qkv_one_token_edges(m, orc):
    """One token (the one-token instantiation): without a gain (a gain of ones in the oracle),
    and at a position past the region (rotated, written, not stored) and before it (not
    rotated, not stored)."""
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g, cap = wl.QWEN25_05B, 64
    h, gain, w, b = _case(g, 1, 60)
    K0 = rnd((cap, g.row_width), 61)
    for p, want in ((5, 0), (cap, m.ERRBIT_STORE_POS), (-1, m.ERRBIT_STORE_POS | m.ERRBIT_ROPE_POS)):
        Kd, Vd = dev(K0), dev(K0)
        xn = torch.empty(1, g.n_embd, device="cuda")
        q = torch.empty(1, g.q_width, device="cuda")
        k = torch.empty(1, g.row_width, device="cuda")
        v = torch.empty(1, g.row_width, device="cuda")
        err = err_word()
        m.minf_fused_qkv(xn, dev(h), None, g.eps, dev(w), dev(b), dev(np.array([p], np.int32)), q, k, v, Kd, Vd,
                         g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, err)
        torch.cuda.synchronize()
        assert err.item() == want, (p, err.item())
        # the oracle stores every token, so it gets a region that holds row p (and row 0 for p < 0)
        Ko = np.zeros((max(p, 0) + 1, g.row_width), np.float32)
        Vo = Ko.copy()
        xn_r, q_r, k_r, v_r = orc.fused_qkv(h, np.ones(g.n_embd, np.float32), w, b, np.array([max(p, 0)], np.int32),
                                            Ko, Vo, n_head=g.n_head, n_kv_head=g.n_kv_head, hd=g.hd, hd_kv=g.hd_kv,
                                            eps=g.eps, theta=g.theta, style=0)
        close(xn.cpu().numpy(), xn_r, what="xn")
        close(v.cpu().numpy(), v_r, what="v")
        if p >= 0:  # rotated at p
            close(q.cpu().numpy(), q_r, what="q")
            close(k.cpu().numpy(), k_r, what="k")
        if 0 <= p < cap:
            assert np.array_equal(Kd.cpu().numpy()[p], k.cpu().numpy()[0])
        else:
            assert np.array_equal(Kd.cpu().numpy(), K0) and np.array_equal(Vd.cpu().numpy(), K0)


@pytest.mark.parametrize("which", ["qwen25", "qwen3"])
def test_layer_step_qkv_decode(m, orc, which):
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN25_05B if which == "qwen25" else wl.QWEN3_06B
    cap, p = 1200, 777
    h, gain, w, b = _case(g, 1, 40, bias=which == "qwen25")
    K0, V0 = rnd((cap, g.row_width), 41), rnd((cap, g.row_width), 42)
    Kd, Vd = dev(K0), dev(V0)
    xn = torch.empty(1, g.n_embd, device="cuda")
    q = torch.empty(1, g.q_width, device="cuda")
    k = torch.empty(1, g.row_width, device="cuda")
    v = torch.empty(1, g.row_width, device="cuda")
    out, err = torch.empty(1, g.out_width, device="cuda"), err_word()
    ws = m.kv.decode_workspace(1, g.n_head, g.n_kv_head, g.hd_kv, cap)
    m.minf_layer_attn_step_qkv(xn, dev(h), dev(gain), g.eps, dev(w), dev(b), dev(np.array([p], np.int32)), q, k, v,
                               Kd, Vd, g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    Ko, Vo = K0.copy(), V0.copy()
    _, q_r, _, _ = orc.fused_qkv(h, gain, w, b, [p], Ko, Vo, n_head=g.n_head, n_kv_head=g.n_kv_head, hd=g.hd,
                                 hd_kv=g.hd_kv, eps=g.eps, theta=g.theta)
    close(q.cpu().numpy(), q_r, what="q")
    scale = float(np.float32(1.0) / np.sqrt(np.float32(g.hd)))
    ref = orc.gqa_attn(q.cpu().numpy().reshape(1, g.n_head, g.hd), Kd.cpu().numpy(), Vd.cpu().numpy(), [p],
                       g.n_head, g.n_kv_head, g.hd, g.hd_kv, scale=scale)
    close(out.cpu().numpy(), ref, what="out")
