"""GPU parity of the Q8_0 K/V cache ("11 . Attention, vec ops, and the KV cache", §2.5: the store
quantizes each row into blocks of 32 values with one f16 scale and int8 quants, the attention
read dequantizes).

The store is compared byte for byte with the oracle's quantizer (the GPU performs the same IEEE
fp32 operations: max, d = max/127, 1/d, x * (1/d), rounding halves away from zero, binary16 of
d).  A K row the GPU rotates itself is compared with the oracle's quantization of the GPU's
rotated k.  Attention outputs are held to the fp32 tolerance against the oracle's fp32 attention
over the dequantized regions (dequantization is exact in fp32)."""
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
    return torch.as_tensor(np.ascontiguousarray(x)).cuda()


def err_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def test_row_bytes(m, orc):
    for W in (32, 64, 128, 256, 896, 1024):
        assert m.minf_q8_row_bytes(W) == orc.q8_row_bytes(W) == m.kv.q8_row_bytes(W)
    assert m.minf_q8_row_bytes(100) == 0


@pytest.mark.parametrize("W", [128, 1024])
def test_kv_append_q8_bytes(m, orc, W):
    cap, nt = 200, 37
    R0 = np.random.default_rng(1).integers(0, 256, size=(cap, orc.q8_row_bytes(W))).astype(np.uint8)
    k = rnd((nt, W), 2, scale=3.0)
    v = rnd((nt, W), 3, scale=1e-6)          # tiny scales: binary16 subnormal d
    k[0, :32] = 0.0                           # an all-zero block
    k[1, :4] = [127.0, 2.5, -2.5, 0.5]        # a block whose d is exactly 1: ties away from zero
    k[1, 4:32] = 0.0
    pos = np.random.default_rng(4).permutation(cap)[:nt].astype(np.int32)
    Kd, Vd, err = dev(R0), dev(R0), err_word()
    m.minf_kv_append_q8(Kd, Vd, dev(k), dev(v), dev(pos), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    Ko, Vo = R0.copy(), R0.copy()
    orc.kv_append_q8(Ko, Vo, W, k, v, pos)
    assert np.array_equal(Kd.cpu().numpy(), Ko)
    assert np.array_equal(Vd.cpu().numpy(), Vo)


def _decode_q8(m, orc, nh, nk, hd, hdkv, caps, pos, seed):
    W = nk * hdkv
    n_seq = len(caps)
    offs = np.concatenate([[0], np.cumsum(caps)[:-1]]).astype(np.int64)
    rows = int(np.sum(caps))
    Kq = orc.q8_quantize(rnd((rows, W), seed))
    Vq = orc.q8_quantize(rnd((rows, W), seed + 1))
    q = rnd((n_seq, nh, hd), seed + 2)
    pos = np.asarray(pos, np.int32)
    out = torch.empty(n_seq, nh * hdkv, device="cuda")
    max_cap = int(max(caps))
    ws = m.kv.decode_workspace(n_seq, nh, nk, hdkv, max_cap)
    err = err_word()
    scale = float(np.float32(1.0) / np.sqrt(np.float32(hd)))
    m.minf_gqa_attn_decode_q8(out, dev(q), dev(Kq), dev(Vq), dev(offs), dev(np.asarray(caps, np.int32)), max_cap,
                              dev(pos), nh, nk, hd, hdkv, scale, ws, err)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    Kf, Vf = orc.q8_dequant(Kq, W), orc.q8_dequant(Vq, W)
    for s in range(n_seq):
        o, c = int(offs[s]), int(caps[s])
        ref = orc.gqa_attn(q[s:s + 1], Kf[o:o + c], Vf[o:o + c], [pos[s]], nh, nk, hd, hdkv, scale=scale)
        close(got[s:s + 1], ref, what=f"q8 decode seq {s} (pos {pos[s]})")
    return err


@pytest.mark.parametrize("L", [1, 127, 128, 129, 1000, 4097])
def test_decode_q8_qwen3(m, orc, L):
    err = _decode_q8(m, orc, 16, 8, 128, 128, [4200], [L - 1], seed=10 + L)
    assert err.item() == 0


@pytest.mark.parametrize("L", [1, 255, 256, 257, 639])
def test_decode_q8_qwen25(m, orc, L):
    err = _decode_q8(m, orc, 14, 2, 64, 64, [639], [L - 1], seed=30 + L)
    assert err.item() == 0


def test_decode_q8_batched_and_batch_mode(m, orc):
    r = np.random.default_rng(50)
    small = [int(x) for x in r.integers(1, 900, size=9)]
    assert _decode_q8(m, orc, 16, 8, 128, 128, [ln + 3 for ln in small], [ln - 1 for ln in small], 51).item() == 0
    many = [int(x) for x in r.integers(1, 2000, size=24)]  # 192 (sequence, kv head) pairs: batch mode
    assert _decode_q8(m, orc, 16, 8, 128, 128, [ln + 3 for ln in many], [ln - 1 for ln in many], 52).item() == 0


def _inputs(g, n, seed):
    h = rnd((n, g.n_embd), seed)
    gain = np.random.default_rng(seed).uniform(0.5, 1.5, g.n_embd).astype(np.float32)
    return h, gain, rnd((n, g.q_width), seed + 1), rnd((n, g.row_width), seed + 2), rnd((n, g.row_width), seed + 3)


def _check(orc, g, pos, h, gain, q, k, v, xn, qg, kg, out, Kn, Vn, K0, V0):
    """The GPU step's outputs and regions against the oracle (one sequence's region)."""
    n = len(pos)
    W = g.row_width
    close(xn, orc.rms_norm(h, gain, eps=g.eps), what="xn")
    q_ref = orc.rope(q.copy(), pos, g.n_head, g.hd, g.theta)
    close(qg, q_ref.reshape(n, -1), what="q rotated")
    close(kg, orc.rope(k.copy(), pos, g.n_kv_head, g.hd_kv, g.theta).reshape(n, -1), what="k rotated")
    Ko, Vo = K0.copy(), V0.copy()
    orc.kv_append_q8(Ko, Vo, W, kg, v, pos)  # K rows: the GPU's rotated k, quantized by the oracle
    assert np.array_equal(Kn, Ko), "K region"
    assert np.array_equal(Vn, Vo), "V region"
    scale = float(np.float32(1.0) / np.sqrt(np.float32(g.hd)))
    ref = orc.gqa_attn(q_ref.reshape(n, g.n_head, g.hd), orc.q8_dequant(Kn, W), orc.q8_dequant(Vn, W), pos,
                       g.n_head, g.n_kv_head, g.hd, g.hd_kv, scale=scale)
    close(out, ref, what="out")


@pytest.mark.parametrize("which", ["qwen25", "qwen3"])
def test_layer_step_q8_decode_loop(m, orc, which):
    # four consecutive single-token steps on one region: each reads what the earlier appended
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN25_05B if which == "qwen25" else wl.QWEN3_06B
    cap, p0 = 1000, 600
    R0 = orc.q8_quantize(rnd((cap, g.row_width), 60))
    Kd, Vd = dev(R0), dev(orc.q8_quantize(rnd((cap, g.row_width), 61)))
    K0, V0 = Kd.cpu().numpy(), Vd.cpu().numpy()
    ws = m.kv.decode_workspace(1, g.n_head, g.n_kv_head, g.hd_kv, cap)
    for step in range(4):
        h, gain, q, k, v = _inputs(g, 1, 62 + 10 * step)
        qd, kd = dev(q), dev(k)
        xn, out, err = torch.empty(1, g.n_embd, device="cuda"), torch.empty(1, g.out_width, device="cuda"), err_word()
        m.minf_layer_attn_step_q8(xn, dev(h), dev(gain), g.eps, qd, kd, dev(v), dev(np.array([p0 + step], np.int32)),
                                  Kd, Vd, g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, out, ws, err)
        torch.cuda.synchronize()
        assert err.item() == 0
        Kn, Vn = Kd.cpu().numpy(), Vd.cpu().numpy()
        _check(orc, g, [p0 + step], h, gain, q, k, v, xn.cpu().numpy(), qd.cpu().numpy(), kd.cpu().numpy(),
               out.cpu().numpy(), Kn, Vn, K0, V0)
        K0, V0 = Kn, Vn


def test_layer_step_batched_q8(m, orc):
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN3_06B
    lengths = wl.batched_lengths(seed=5, n_seq=20, lo=1, hi=3000)
    caps = [ln + 9 for ln in lengths]
    arena = m.kv.KvArena(1, g.row_width, caps, dtype=torch.uint8)
    K0 = orc.q8_quantize(rnd((arena.rows, g.row_width), 70))
    V0 = orc.q8_quantize(rnd((arena.rows, g.row_width), 71))
    arena.k[0].copy_(dev(K0))
    arena.v[0].copy_(dev(V0))
    n = len(lengths)
    h, gain, q, k, v = _inputs(g, n, 72)
    qd, kd = dev(q), dev(k)
    xn, out, err = torch.empty(n, g.n_embd, device="cuda"), torch.empty(n, g.out_width, device="cuda"), err_word()
    ws = m.kv.decode_workspace(n, g.n_head, g.n_kv_head, g.hd_kv, arena.max_cap)
    k_ar, v_ar = arena.view(0)
    m.minf_layer_attn_step_batched_q8(xn, dev(h), dev(gain), g.eps, qd, kd, dev(v), dev(np.asarray(lengths, np.int32)),
                                      k_ar, v_ar, arena.row_off, arena.cap, arena.max_cap, g.n_head, g.n_kv_head,
                                      g.hd, g.hd_kv, g.theta, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    Kn, Vn, xg, qg, kg, og = (t.cpu().numpy() for t in (arena.k[0], arena.v[0], xn, qd, kd, out))
    for s in range(n):
        o, c = arena.offsets_host[s], arena.caps_host[s]
        _check(orc, g, [lengths[s]], h[s:s + 1], gain, q[s:s + 1], k[s:s + 1], v[s:s + 1], xg[s:s + 1],
               qg[s:s + 1], kg[s:s + 1], og[s:s + 1], Kn[o:o + c], Vn[o:o + c], K0[o:o + c], V0[o:o + c])


@pytest.mark.parametrize("geom", [(14, 2, 64, 64, 512, 1024), (16, 8, 128, 128, 300, 700)])
def test_prefill_q8(m, orc, geom):
    nh, nk, hd, hdkv, nt, cap = geom
    W = nk * hdkv
    Kq = orc.q8_quantize(rnd((cap, W), 80))
    Vq = orc.q8_quantize(rnd((cap, W), 81))
    q = rnd((nt, nh, hd), 82)
    pos = np.arange(nt, dtype=np.int32) + 11
    out, err = torch.full((nt, nh * hdkv), float("nan"), device="cuda"), err_word()
    scale = float(np.float32(1.0) / np.sqrt(np.float32(hd)))
    ws = m.kv.prefill_workspace(nt, nh, nk, hdkv, cap)
    m.minf_gqa_attn_prefill_q8(out, dev(q), dev(Kq), dev(Vq), dev(pos), nh, nk, hd, hdkv, scale, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = orc.gqa_attn(q, orc.q8_dequant(Kq, W), orc.q8_dequant(Vq, W), pos, nh, nk, hd, hdkv, scale=scale,
                       n_threads=8)
    close(out.cpu().numpy(), ref, what="prefill q8")


def test_layer_step_q8_prefill_path(m, orc):
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN25_05B
    nt, cap = 200, 712
    R0 = np.zeros((cap, orc.q8_row_bytes(g.row_width)), np.uint8)
    h, gain, q, k, v = _inputs(g, nt, 90)
    pos = list(range(nt))
    Kd, Vd = dev(R0), dev(R0)
    qd, kd = dev(q), dev(k)
    xn, out, err = torch.empty(nt, g.n_embd, device="cuda"), torch.empty(nt, g.out_width, device="cuda"), err_word()
    ws = m.kv.prefill_workspace(nt, g.n_head, g.n_kv_head, g.hd_kv, cap)
    m.minf_layer_attn_step_q8(xn, dev(h), dev(gain), g.eps, qd, kd, dev(v), dev(np.asarray(pos, np.int32)), Kd, Vd,
                              g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    _check(orc, g, pos, h, gain, q, k, v, xn.cpu().numpy(), qd.cpu().numpy(), kd.cpu().numpy(), out.cpu().numpy(),
           Kd.cpu().numpy(), Vd.cpu().numpy(), R0, R0)


def test_paged_q8_step_and_decode(m, orc):
    # the batched step through a table over a Q8_0 pool, then the plain paged decode on the result
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN3_06B
    n, block_rows, max_blocks = 5, 64, 10
    pool_blocks = n * max_blocks + 4
    W = g.row_width
    P0 = orc.q8_quantize(rnd((pool_blocks * block_rows, W), 100))
    table = np.random.default_rng(101).permutation(pool_blocks)[:n * max_blocks].reshape(n, max_blocks)
    table = table.astype(np.int32)
    pos = np.array([0, 64, 300, 500, 638], np.int32)
    Kd, Vd, td = dev(P0), dev(P0), dev(table)
    h, gain, q, k, v = _inputs(g, n, 102)
    qd, kd = dev(q), dev(k)
    xn, out, err = torch.empty(n, g.n_embd, device="cuda"), torch.empty(n, g.out_width, device="cuda"), err_word()
    ws = m.kv.decode_workspace(n, g.n_head, g.n_kv_head, g.hd_kv, max_blocks * block_rows)
    m.minf_layer_attn_step_paged_q8(xn, dev(h), dev(gain), g.eps, qd, kd, dev(v), dev(pos), Kd, Vd, td, block_rows,
                                    g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    kg = kd.cpu().numpy()
    Ko, Vo = P0.copy(), P0.copy()
    for s in range(n):
        row = table[s, pos[s] // block_rows] * block_rows + pos[s] % block_rows
        Ko[row], Vo[row] = orc.q8_quantize(kg[s:s + 1])[0], orc.q8_quantize(v[s:s + 1])[0]
    assert np.array_equal(Kd.cpu().numpy(), Ko) and np.array_equal(Vd.cpu().numpy(), Vo)
    q_ref = orc.rope(q.copy(), pos, g.n_head, g.hd, g.theta).reshape(n, g.n_head, g.hd)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(g.hd)))
    ref = orc.gqa_attn_paged(q_ref, orc.q8_dequant(Ko, W), orc.q8_dequant(Vo, W), table, block_rows, pos, g.n_head,
                             g.n_kv_head, g.hd, g.hd_kv, scale=scale)
    close(out.cpu().numpy(), ref, what="paged q8 step")
    out2, err2 = torch.empty_like(out), err_word()
    m.minf_gqa_attn_decode_paged_q8(out2, dev(q_ref), Kd, Vd, td, block_rows, dev(pos), g.n_head, g.n_kv_head, g.hd,
                                    g.hd_kv, scale, ws, err2)
    torch.cuda.synchronize()
    assert err2.item() == 0
    close(out2.cpu().numpy(), ref, what="paged q8 decode")
    # the standalone paged store
    k2, v2 = rnd((n, W), 103), rnd((n, W), 104)
    pos2 = pos + 1
    m.minf_kv_append_paged_q8(Kd, Vd, td, block_rows, dev(k2), dev(v2), dev(pos2), err2)
    torch.cuda.synchronize()
    assert err2.item() == 0
    for s in range(n):
        row = table[s, pos2[s] // block_rows] * block_rows + pos2[s] % block_rows
        Ko[row], Vo[row] = orc.q8_quantize(k2[s:s + 1])[0], orc.q8_quantize(v2[s:s + 1])[0]
    assert np.array_equal(Kd.cpu().numpy(), Ko) and np.array_equal(Vd.cpu().numpy(), Vo)
