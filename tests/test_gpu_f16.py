"""GPU parity of the f16 K/V cache ("11 . Attention, vec ops, and the KV cache", §2.5: the GPU
backends may keep the regions in f16; the store converts, the attention read converts back).

The store is compared bit for bit with the oracle's binary16 conversion (round to nearest
even).  The attention kernels read the regions exactly, so their outputs are held to the same
fp32 tolerance as with fp32 regions, against the oracle's fp32 attention over the values the
regions hold.  The one value that may differ is a K row the GPU rotates itself (sincosf
against the oracle's double-precision sine before rounding): it is checked to be the GPU's
own rotated k converted by the oracle, and within one binary16 step of the oracle's row."""
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


def close(got, ref, atol=ATOL, rtol=RTOL, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    d = np.abs(got - ref)
    bad = d > atol + rtol * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off, max abs {d.max():.3g}"


def rnd(shape, seed, scale=1.0):
    return (torch.randn(*shape, generator=torch.Generator().manual_seed(seed)) * scale).numpy()


def half_dev(bits):
    """uint16 bit patterns -> a CUDA float16 tensor holding them."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.float16)).cuda()


def half_bits(t):
    return t.cpu().numpy().view(np.uint16)


def f32_dev(x):
    return torch.as_tensor(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def i32_dev(x):
    return torch.as_tensor(np.asarray(x, np.int32)).cuda()


def err_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# --------------------------------------------------------------------------- the store
def test_kv_append_f16_bit_exact(m, orc):
    cap, W, nt = 300, 1024, 40
    K0 = orc.f32_to_f16(rnd((cap, W), 1))
    V0 = orc.f32_to_f16(rnd((cap, W), 2))
    k = rnd((nt, W), 3, scale=300.0)  # spans binary16's range, rounding and overflow to inf
    v = rnd((nt, W), 4, scale=1e-3)   # and its subnormals
    k[0, :4] = [65519.0, 65520.0, -7e4, 2.0 ** -25 * 3]
    pos = np.random.default_rng(5).permutation(cap)[:nt].astype(np.int32)
    Kd, Vd, err = half_dev(K0), half_dev(V0), err_word()
    m.minf_kv_append_f16(Kd, Vd, f32_dev(k), f32_dev(v), i32_dev(pos), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    Ko, Vo = K0.copy(), V0.copy()
    orc.kv_append_f16(Ko, Vo, k, v, pos)
    assert np.array_equal(half_bits(Kd), Ko)  # the whole region, untouched rows included
    assert np.array_equal(half_bits(Vd), Vo)


def test_kv_append_f16_out_of_range_is_reported_not_written(m, orc):
    cap, W = 16, 128
    K0 = orc.f32_to_f16(rnd((cap, W), 6))
    Kd, Vd, err = half_dev(K0), half_dev(K0), err_word()
    m.minf_kv_append_f16(Kd, Vd, f32_dev(rnd((2, W), 7)), f32_dev(rnd((2, W), 8)), i32_dev([cap, -1]), err)
    torch.cuda.synchronize()
    assert err.item() & 0x1
    assert np.array_equal(half_bits(Kd), K0) and np.array_equal(half_bits(Vd), K0)


def test_rope_kv_append_f16(m, orc):
    nh, nk, hd, hdkv, cap, nt = 16, 8, 128, 128, 700, 33
    W = nk * hdkv
    q, k, v = rnd((nt, nh * hd), 10), rnd((nt, W), 11), rnd((nt, W), 12)
    pos = np.sort(np.random.default_rng(13).choice(cap, nt, replace=False)).astype(np.int32)
    K0 = orc.f32_to_f16(rnd((cap, W), 14))
    V0 = orc.f32_to_f16(rnd((cap, W), 15))
    qd, kd, Kd, Vd, err = f32_dev(q), f32_dev(k), half_dev(K0), half_dev(V0), err_word()
    m.minf_rope_kv_append_f16(qd, kd, f32_dev(v), i32_dev(pos), nh, nk, hd, hdkv, 1e6, 1.0, 0, Kd, Vd, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    q_ref = orc.rope(q.copy(), pos, nh, hd, 1e6)
    k_ref = orc.rope(k.copy(), pos, nk, hdkv, 1e6)
    close(qd.cpu().numpy().reshape(nt, -1), q_ref.reshape(nt, -1), what="q")
    k_gpu = kd.cpu().numpy().reshape(nt, -1)
    close(k_gpu, k_ref.reshape(nt, -1), what="k")
    Kn, Vn = half_bits(Kd), half_bits(Vd)
    Vo = V0.copy()
    Vo[pos] = orc.f32_to_f16(v)
    assert np.array_equal(Vn, Vo)                                   # V rows: the oracle's conversion
    assert np.array_equal(Kn[pos], orc.f32_to_f16(k_gpu))            # K rows: the GPU's rotated k, converted
    d = np.abs(Kn[pos].astype(np.int32) - orc.f32_to_f16(k_ref.reshape(nt, -1)).astype(np.int32))
    assert d.max() <= 1                                              # within one binary16 step of the oracle
    keep = np.setdiff1d(np.arange(cap), pos)
    assert np.array_equal(Kn[keep], K0[keep])


# --------------------------------------------------------------------------- decode attention
def _decode_f16(m, orc, nh, nk, hd, hdkv, caps, pos, seed):
    W = nk * hdkv
    n_seq = len(caps)
    offs = np.concatenate([[0], np.cumsum(caps)[:-1]]).astype(np.int64)
    rows = int(np.sum(caps))
    K16 = orc.f32_to_f16(rnd((rows, W), seed))
    V16 = orc.f32_to_f16(rnd((rows, W), seed + 1))
    q = rnd((n_seq, nh, hd), seed + 2)
    pos = np.asarray(pos, np.int32)
    out = torch.empty(n_seq, nh * hdkv, device="cuda")
    max_cap = int(max(caps))
    ws = m.kv.decode_workspace(n_seq, nh, nk, hdkv, max_cap)
    err = err_word()
    scale = float(np.float32(1.0) / np.sqrt(np.float32(hd)))
    m.minf_gqa_attn_decode_f16(out, f32_dev(q), half_dev(K16), half_dev(V16),
                               torch.as_tensor(offs).cuda(), i32_dev(caps), max_cap, i32_dev(pos), nh, nk, hd,
                               hdkv, scale, ws, err)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    Kf, Vf = orc.f16_to_f32(K16), orc.f16_to_f32(V16)
    for s in range(n_seq):
        o, c = int(offs[s]), int(caps[s])
        if pos[s] < 0:
            assert not np.any(got[s]), f"seq {s}: empty window gave a non-zero output"
            continue
        ref = orc.gqa_attn(q[s:s + 1], Kf[o:o + c], Vf[o:o + c], [pos[s]], nh, nk, hd, hdkv, scale=scale)
        close(got[s:s + 1], ref, what=f"decode f16 seq {s} (pos {pos[s]})")
    return err


@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 127, 128, 129, 300, 1000, 4097])
def test_decode_f16_qwen3_geometry(m, orc, L):
    err = _decode_f16(m, orc, 16, 8, 128, 128, [4200], [L - 1], seed=20 + L)
    assert err.item() == 0


@pytest.mark.parametrize("L", [1, 255, 256, 257, 639])
def test_decode_f16_qwen25_geometry(m, orc, L):
    err = _decode_f16(m, orc, 14, 2, 64, 64, [639], [L - 1], seed=40 + L)
    assert err.item() == 0


def test_decode_f16_batched_ragged(m, orc):
    r = np.random.default_rng(50)
    lengths = [int(x) for x in r.integers(1, 900, size=11)] + [1, 2, 899]
    err = _decode_f16(m, orc, 16, 8, 128, 128, [ln + 5 for ln in lengths], [ln - 1 for ln in lengths], seed=51)
    assert err.item() == 0


def test_decode_f16_batch_longest_first(m, orc):
    # pairs fill the SMs: units drawn from the counter, sequences longest first; one empty window
    r = np.random.default_rng(52)
    lengths = [int(x) for x in r.integers(1, 1500, size=22)] + [5000, 2049, 1]
    pos = [ln - 1 for ln in lengths]
    pos[3] = -1
    err = _decode_f16(m, orc, 16, 8, 128, 128, [ln + 2 for ln in lengths], pos, seed=53)
    assert err.item() == 0x4


# --------------------------------------------------------------------------- layer step
def _step_inputs(g, seed, nt=1):
    h = rnd((nt, g.n_embd), seed)
    gain = np.random.default_rng(seed).uniform(0.5, 1.5, g.n_embd).astype(np.float32)
    q = rnd((nt, g.q_width), seed + 1)
    k = rnd((nt, g.row_width), seed + 2)
    v = rnd((nt, g.row_width), seed + 3)
    return h, gain, q, k, v


def _check_step(orc, g, got_out, got_xn, got_q, got_k, Kn, Vn, K0, V0, h, gain, q, k, v, pos):
    """The GPU step against the oracle's f16 step; the attention against the oracle over the
    GPU's own regions (their appended K rows are the GPU's rotation, rounded)."""
    nt = len(pos)
    Ko, Vo = K0.copy(), V0.copy()
    qo, ko = q.copy(), k.copy()
    xn_ref, _ = orc.layer_attn_step_f16(h, gain, qo, ko, v, pos, Ko, Vo, n_head=g.n_head, n_kv_head=g.n_kv_head,
                                        hd=g.hd, hd_kv=g.hd_kv, eps=g.eps, theta=g.theta)
    close(got_xn, xn_ref, what="xn")
    close(got_q.reshape(nt, -1), qo.reshape(nt, -1), what="q rotated")
    close(got_k.reshape(nt, -1), ko.reshape(nt, -1), what="k rotated")
    assert np.array_equal(Vn, Vo), "V region"
    rows = np.asarray(pos)
    assert np.array_equal(Kn[rows], orc.f32_to_f16(got_k.reshape(nt, -1))), "K rows: the GPU's rotated k"
    keep = np.setdiff1d(np.arange(K0.shape[0]), rows)
    assert np.array_equal(Kn[keep], K0[keep]), "K region outside the appended rows"
    scale = float(np.float32(1.0) / np.sqrt(np.float32(g.hd)))
    ref = orc.gqa_attn(qo.reshape(nt, g.n_head, g.hd), orc.f16_to_f32(Kn), orc.f16_to_f32(Vn), pos, g.n_head,
                       g.n_kv_head, g.hd, g.hd_kv, scale=scale)
    close(got_out, ref, what="out")


@pytest.mark.parametrize("which", ["qwen25", "qwen3"])
def test_layer_step_f16_single_decode(m, orc, which):
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN25_05B if which == "qwen25" else wl.QWEN3_06B
    cap, p = 1000, 700
    K0 = orc.f32_to_f16(rnd((cap, g.row_width), 60))
    V0 = orc.f32_to_f16(rnd((cap, g.row_width), 61))
    h, gain, q, k, v = _step_inputs(g, 62)
    Kd, Vd = half_dev(K0), half_dev(V0)
    qd, kd, xn = f32_dev(q), f32_dev(k), torch.empty(1, g.n_embd, device="cuda")
    out, err = torch.empty(1, g.out_width, device="cuda"), err_word()
    ws = m.kv.decode_workspace(1, g.n_head, g.n_kv_head, g.hd_kv, cap)
    m.minf_layer_attn_step_f16(xn, f32_dev(h), f32_dev(gain), g.eps, qd, kd, f32_dev(v), i32_dev([p]), Kd, Vd,
                               g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    _check_step(orc, g, out.cpu().numpy(), xn.cpu().numpy(), qd.cpu().numpy(), kd.cpu().numpy(), half_bits(Kd),
                half_bits(Vd), K0, V0, h, gain, q, k, v, [p])


def test_layer_step_f16_graph_replayed_decode_loop(m, orc):
    # one captured step replayed at positions 300..309: each step reads the rows the earlier
    # steps appended (the tile holding the new row is patched in shared memory)
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN3_06B
    cap, p0, n = 512, 300, 10
    K0 = orc.f32_to_f16(rnd((cap, g.row_width), 70))
    V0 = orc.f32_to_f16(rnd((cap, g.row_width), 71))
    Kd, Vd = half_dev(K0), half_dev(V0)
    ins = [_step_inputs(g, 72 + 5 * i) for i in range(n)]
    hb, gb, qb, kb, vb = (torch.empty(1, w, device="cuda") for w in (g.n_embd, g.n_embd, g.q_width, g.row_width,
                                                                      g.row_width))
    gb = torch.empty(g.n_embd, device="cuda")
    xn, out, err = torch.empty(1, g.n_embd, device="cuda"), torch.empty(1, g.out_width, device="cuda"), err_word()
    pos = i32_dev([p0])
    ws = m.kv.decode_workspace(1, g.n_head, g.n_kv_head, g.hd_kv, cap)
    stream = torch.cuda.Stream()

    def step():
        m.minf_layer_attn_step_f16(xn, hb, gb, g.eps, qb, kb, vb, pos, Kd, Vd, g.n_head, g.n_kv_head, g.hd, g.hd_kv,
                                   g.theta, 1.0, 0, out, ws, err, stream=stream)

    with torch.cuda.stream(stream):
        for t, x in zip((hb, gb, qb, kb, vb), ins[0]):
            t.copy_(torch.as_tensor(x).reshape(t.shape))
        step()  # warm-up outside the capture, then undo its append
    torch.cuda.synchronize()
    Kd.copy_(half_dev(K0))
    Vd.copy_(half_dev(V0))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    Ko, Vo = K0.copy(), V0.copy()
    for i in range(n):
        h, gain, q, k, v = ins[i]
        for t, x in zip((hb, gb, qb, kb, vb), (h, gain, q, k, v)):
            t.copy_(torch.as_tensor(x).reshape(t.shape))
        pos.fill_(p0 + i)
        graph.replay()
        torch.cuda.synchronize()
        assert err.item() == 0
        Kn, Vn = half_bits(Kd), half_bits(Vd)
        _check_step(orc, g, out.cpu().numpy(), xn.cpu().numpy(), qb.cpu().numpy(), kb.cpu().numpy(), Kn, Vn, Ko,
                    Vo, h, gain, q, k, v, [p0 + i])
        Ko, Vo = Kn, Vn


def test_layer_step_batched_f16(m, orc):
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN3_06B
    lengths = wl.batched_lengths(seed=4, n_seq=20, lo=1, hi=3000)
    caps = [ln + 1 + 8 for ln in lengths]
    arena = m.kv.KvArena(1, g.row_width, caps, dtype=torch.float16)
    K0 = orc.f32_to_f16(rnd((arena.rows, g.row_width), 80))
    V0 = orc.f32_to_f16(rnd((arena.rows, g.row_width), 81))
    arena.k[0].copy_(half_dev(K0))
    arena.v[0].copy_(half_dev(V0))
    n = len(lengths)
    h, gain, q, k, v = _step_inputs(g, 82, nt=n)
    gain = gain[:g.n_embd]
    qd, kd = f32_dev(q), f32_dev(k)
    xn, out, err = torch.empty(n, g.n_embd, device="cuda"), torch.empty(n, g.out_width, device="cuda"), err_word()
    ws = m.kv.decode_workspace(n, g.n_head, g.n_kv_head, g.hd_kv, arena.max_cap)
    k_ar, v_ar = arena.view(0)
    m.minf_layer_attn_step_batched_f16(xn, f32_dev(h), f32_dev(gain), g.eps, qd, kd, f32_dev(v),
                                       i32_dev(lengths), k_ar, v_ar, arena.row_off, arena.cap, arena.max_cap,
                                       g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    got, Kn, Vn = out.cpu().numpy(), half_bits(arena.k[0]), half_bits(arena.v[0])
    qg, kg = qd.cpu().numpy(), kd.cpu().numpy()
    for s in range(n):
        o, c = arena.offsets_host[s], arena.caps_host[s]
        _check_step(orc, g, got[s:s + 1], xn.cpu().numpy()[s:s + 1], qg[s:s + 1], kg[s:s + 1], Kn[o:o + c],
                    Vn[o:o + c], K0[o:o + c], V0[o:o + c], h[s:s + 1], gain, q[s:s + 1], k[s:s + 1], v[s:s + 1],
                    [lengths[s]])


# --------------------------------------------------------------------------- prefill
@pytest.mark.parametrize("geom", [(14, 2, 64, 64, 512, 1024), (16, 8, 128, 128, 300, 700)])
def test_prefill_f16(m, orc, geom):
    nh, nk, hd, hdkv, nt, cap = geom
    W = nk * hdkv
    K16 = orc.f32_to_f16(rnd((cap, W), 90))
    V16 = orc.f32_to_f16(rnd((cap, W), 91))
    q = rnd((nt, nh, hd), 92)
    pos = np.arange(nt, dtype=np.int32) + 17  # a continuation over 17 cached rows
    out, err = torch.full((nt, nh * hdkv), float("nan"), device="cuda"), err_word()
    scale = float(np.float32(1.0) / np.sqrt(np.float32(hd)))
    ws = m.kv.prefill_workspace(nt, nh, nk, hdkv, cap)
    m.minf_gqa_attn_prefill_f16(out, f32_dev(q), half_dev(K16), half_dev(V16), i32_dev(pos), nh, nk, hd, hdkv,
                                scale, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = orc.gqa_attn(q, orc.f16_to_f32(K16), orc.f16_to_f32(V16), pos, nh, nk, hd, hdkv, scale=scale, n_threads=8)
    close(out.cpu().numpy(), ref, what="prefill f16")


def test_layer_step_f16_prefill_path(m, orc):
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN25_05B
    nt, cap = 200, 712
    K0 = orc.f32_to_f16(np.zeros((cap, g.row_width), np.float32))
    h, gain, q, k, v = _step_inputs(g, 95, nt=nt)
    gain = gain[:g.n_embd]
    pos = list(range(nt))
    Kd, Vd = half_dev(K0), half_dev(K0)
    qd, kd = f32_dev(q), f32_dev(k)
    xn, out, err = torch.empty(nt, g.n_embd, device="cuda"), torch.empty(nt, g.out_width, device="cuda"), err_word()
    ws = m.kv.prefill_workspace(nt, g.n_head, g.n_kv_head, g.hd_kv, cap)
    m.minf_layer_attn_step_f16(xn, f32_dev(h), f32_dev(gain), g.eps, qd, kd, f32_dev(v), i32_dev(pos), Kd, Vd,
                               g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    _check_step(orc, g, out.cpu().numpy(), xn.cpu().numpy(), qd.cpu().numpy(), kd.cpu().numpy(), half_bits(Kd),
                half_bits(Vd), K0, K0, h, gain, q, k, v, pos)
