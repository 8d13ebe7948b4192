"""GPU parity of the single-launch prefill layer step (RMSNorm, RoPE on q and k, the K/V store and
the tensor-core causal attention in one cooperative launch with a grid barrier) against the CPU
oracle, on the cases that launch adds: positions that are scattered or out of range, the
interleaved pair style, hd > hd_kv (q and k rotate with different angular speeds), and calls of
different grid sizes one after another on one workspace, whose grid-barrier counts (in its first
256 bytes, the control block) every call leaves at zero.  Outputs of the tensor cores pass the
max-abs 2e-3 bound and the fp32 bound element by element; RMSNorm, rotations and stored K rows
pass the fp32 bound element by element; stored V rows are bit-exact."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ATOL = 2e-3  # the tensor-core tolerance of the prefill tests; the fp32 bound is checked as well


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


def close(got, ref, what):
    """Tensor-core outputs: max-abs 2e-3, and the fp32 bound element by element."""
    d = np.abs(got.astype(np.float64) - ref)
    assert np.isfinite(got).all(), what
    assert d.max() <= ATOL, f"{what}: max abs {d.max():.3g}"
    assert np.all(d <= 1e-5 + 1e-4 * np.abs(ref)), f"{what}: outside the fp32 tolerance"


def close32(got, ref, what):
    """CUDA-core outputs (RMSNorm, rotations, stored K rows): |d| <= 1e-5 + 1e-4 |ref| element by element."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    d = np.abs(got - ref)
    bad = d > 1e-5 + 1e-4 * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} elements off, max abs {d.max():.3g}"


def counts_zero(ws):
    """The workspace's control block (its first 256 bytes) after a call: the grid barrier's
    arrival and departure counts and the decode counters at zero, the layout tag a prefill
    layout's ('MI' in the high half, kind 2 in the low bits) and nothing else set."""
    ctl = ws[:256].cpu().numpy().view(np.int32)
    tag = int(ctl[4]) & 0xFFFFFFFF
    return not ctl[:4].any() and not ctl[5:].any() and (tag >> 16) == 0x4D49 and (tag & 3) == 2


def run_step(m, x, pos, cap, geo, ws, theta=1e6, style=0):
    """One layer step on the GPU; returns (xn, out, q, k, K, V, err) on the host."""
    nh, nk, hd, hdkv, n_embd = geo
    nt = len(pos)
    d = {k: v.clone().cuda() for k, v in x.items()}
    K = torch.zeros(cap, nk * hdkv, device="cuda")
    V = torch.zeros(cap, nk * hdkv, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    xn = torch.empty(nt, n_embd, device="cuda")
    out = torch.full((nt, nh * hdkv), float("nan"), device="cuda")
    p = torch.as_tensor(np.asarray(pos, np.int32)).cuda()
    m.minf_layer_attn_step(xn, d["h"], d["gain"], 1e-6, d["q"], d["k"], d["v"], p, K, V, nh, nk, hd, hdkv, theta,
                           1.0, style, out, ws, err)
    torch.cuda.synchronize()
    return (xn.cpu().numpy(), out.cpu().numpy(), d["q"].cpu().numpy(), d["k"].cpu().numpy(), K.cpu().numpy(),
            V.cpu().numpy(), int(err.item()))


def inputs(nt, geo, seed):
    nh, nk, hd, hdkv, n_embd = geo
    return {"h": rnd((nt, n_embd), seed), "gain": rnd((n_embd,), seed + 1).abs() + 0.5,
            "q": rnd((nt, nh * hd), seed + 2), "k": rnd((nt, nk * hdkv), seed + 3),
            "v": rnd((nt, nk * hdkv), seed + 4)}


def oracle_step(orc, x, pos, cap, geo, theta=1e6, style=0):
    nh, nk, hd, hdkv, n_embd = geo
    q, k = x["q"].numpy().copy(), x["k"].numpy().copy()
    Ko = np.zeros((cap, nk * hdkv), np.float32)
    Vo = np.zeros((cap, nk * hdkv), np.float32)
    xn, out = orc.layer_attn_step(x["h"].numpy(), x["gain"].numpy(), q, k, x["v"].numpy(), np.asarray(pos, np.int32),
                                  Ko, Vo, n_head=nh, n_kv_head=nk, hd=hd, hd_kv=hdkv, eps=1e-6, theta=theta,
                                  style=style, n_threads=8)
    return xn, out, q, k, Ko, Vo


@pytest.mark.parametrize("geo,nt,cap,style", [
    ((14, 2, 64, 64, 896), 300, 512, 1),     # interleaved pairs, a ragged last query tile
    ((8, 2, 128, 64, 512), 200, 256, 0),     # hd > hd_kv: q and k with their own angular speeds
    ((16, 8, 128, 128, 1024), 129, 300, 0),  # one token past a query tile
])
def test_step_matches_oracle(m, orc, geo, nt, cap, style):
    x = inputs(nt, geo, 40 + nt)
    pos = np.arange(nt, dtype=np.int32)
    ws = m.kv.prefill_workspace(nt, geo[0], geo[1], geo[3], cap)
    xn, out, q, k, K, V, err = run_step(m, x, pos, cap, geo, ws, style=style)
    xr, outr, qr, kr, Kr, Vr = oracle_step(orc, x, pos, cap, geo, style=style)
    assert err == 0
    close(out, outr, f"out {geo}")
    close32(xn, xr, "xn")
    for got, ref, what in ((q, qr, "q"), (k, kr, "k"), (K, Kr, "K region")):
        close32(got, ref, what)
    assert np.array_equal(V, Vr)
    assert counts_zero(ws), "the barrier counts are left at zero"


def test_step_scattered_and_bad_positions(m, orc):
    """Positions in any order over an existing window, one < 0 (skipped, zero output) and one
    >= cap (rotated, not stored, attends over the whole region)."""
    geo = (14, 2, 64, 64, 896)
    nh, nk, hd, hdkv, n_embd = geo
    cap = 400
    rng = np.random.default_rng(7)
    good = rng.permutation(np.arange(20, 320))[:240].astype(np.int32)
    pos = np.concatenate([good[:100], [-3], good[100:], [cap + 5]]).astype(np.int32)
    nt = len(pos)
    x = inputs(nt, geo, 90)
    ws = m.kv.prefill_workspace(nt, nh, nk, hdkv, cap)
    xn, out, q, k, K, V, err = run_step(m, x, pos, cap, geo, ws)
    assert err & m.ERRBIT_ROPE_POS and err & m.ERRBIT_STORE_POS and err & m.ERRBIT_ATTN_POS
    assert not err & m.ERRBIT_TIMEOUT
    ok = (pos >= 0) & (pos < cap)
    xv = {kk: vv[torch.as_tensor(ok)] for kk, vv in x.items() if kk != "gain"}
    xv["gain"] = x["gain"]
    xr, outr, qr, kr, Kr, Vr = oracle_step(orc, xv, pos[ok], cap, geo)
    close(out[ok], outr, "scattered positions")
    assert np.array_equal(V, Vr)
    close32(K, Kr, "K region")
    close32(q[ok], qr, "q")
    close32(k[ok], kr, "k")
    neg = pos < 0
    assert np.all(out[neg] == 0.0)
    assert np.array_equal(q[neg], x["q"].numpy()[neg]) and np.array_equal(k[neg], x["k"].numpy()[neg])
    # the token past the region: its own rotation, and the attention over all cap rows
    big = pos >= cap
    qb = x["q"].numpy()[big].copy()
    orc.rope(qb, pos[big], nh, hd, 1e6)
    close32(q[big], qb, "q of the token past the region")
    ref_big = orc.gqa_attn(qb, Kr, Vr, pos[big], nh, nk, hd, hdkv, scale=float(np.float32(1) / np.sqrt(np.float32(hd))))
    close(out[big], ref_big, "token past the region")
    close32(xn, orc.rms_norm(x["h"].numpy(), x["gain"].numpy(), eps=1e-6), "xn")
    assert counts_zero(ws)


def test_step_grid_sizes_share_a_workspace(m, orc):
    """Steps whose grids differ (a few items, then a full grid) on one workspace, twice over."""
    geo = (14, 2, 64, 64, 896)
    cap = 1024
    ws = m.kv.prefill_workspace(900, geo[0], geo[1], geo[3], cap)
    for rep in range(2):
        for nt in (3, 900, 130):
            x = inputs(nt, geo, 200 + nt + rep)
            pos = np.arange(nt, dtype=np.int32)
            _, out, _, _, K, V, err = run_step(m, x, pos, cap, geo, ws)
            _, outr, _, _, Kr, Vr = oracle_step(orc, x, pos, cap, geo)
            assert err == 0
            close(out, outr, f"nt {nt}")
            assert np.array_equal(V, Vr)
            assert counts_zero(ws)
