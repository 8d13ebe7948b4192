"""GPU parity: every kernel, called through the C ABI, against the CPU oracle on the
same seeded inputs.  Tolerances: the KV store is bit-exact; fp32 CUDA-core outputs
pass when |gpu - oracle| <= 1e-5 + 1e-4 * |oracle| element by element."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-5, 1e-4
TC_ATOL = 2e-3  # tensor-core (TF32) prefill outputs: max-abs bound


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
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g) * scale


def dev(x, dtype=None):
    t = torch.as_tensor(x)
    if dtype is not None:
        t = t.to(dtype)
    return t.contiguous().cuda()


def err_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# --------------------------------------------------------------------------- RMSNorm
# rows of 128..2048 values in whole 128-value chunks take the register-resident kernel (one
# read of x); the others (2176, 1001, 4) the two-pass one
@pytest.mark.parametrize("rows,n", [(1, 896), (512, 896), (1, 1024), (4096, 1024), (5, 128), (9, 2048),
                                    (3, 640), (2, 2176), (3, 1001), (7, 4),
                                    # many rows: more blocks than one wave of the GPU
                                    (9001, 1024), (3001, 2048)])
def test_rms_norm(m, orc, rows, n):
    x = rnd((rows, n), 1 + n)
    w = torch.rand(n, generator=torch.Generator().manual_seed(2)) + 0.5
    y = torch.empty(rows, n, device="cuda")
    m.minf_rms_norm(y, dev(x), dev(w), 1e-6)
    torch.cuda.synchronize()
    close(y.cpu(), orc.rms_norm(x.numpy(), w.numpy(), eps=1e-6), what="rms_norm")
    xd = dev(x)  # in place
    m.minf_rms_norm(xd, xd, None, 1e-6)
    close(xd.cpu(), orc.rms_norm(x.numpy(), None, eps=1e-6), what="rms_norm alias")


# --------------------------------------------------------------------------- RoPE
@pytest.mark.parametrize("nt,nh,hd,style,pmax", [(1, 14, 64, 0, 127), (512, 14, 64, 0, 511),
                                                 (16, 16, 128, 0, 40960), (5, 8, 128, 1, 40960),
                                                 (3, 2, 256, 0, 100000), (4, 3, 2, 1, 9)])
def test_rope(m, orc, nt, nh, hd, style, pmax):
    x = rnd((nt, nh, hd), nt * hd)
    pos = np.linspace(0, pmax, nt).astype(np.int32)
    xd = dev(x)
    err = err_word()
    m.minf_rope(xd, dev(pos), nh, hd, 1e6, 1.0, style, err)
    torch.cuda.synchronize()
    ref = orc.rope(x.numpy().copy(), pos, nh, hd, 1e6, 1.0, style)
    close(xd.cpu(), ref, what="rope")
    assert err.item() == 0
    # pos 0 is the identity, bit for bit
    xd = dev(x)
    m.minf_rope(xd, dev(np.zeros(nt, np.int32)), nh, hd, 1e6, 1.0, style, err)
    assert torch.equal(xd.cpu(), x)


def test_rope_negative_position_flagged(m):
    x = rnd((2, 2, 8), 3)
    xd = dev(x)
    err = err_word()
    m.minf_rope(xd, dev(np.array([-1, 0], np.int32)), 2, 8, 1e4, 1.0, 0, err)
    torch.cuda.synchronize()
    assert err.item() & m.ERRBIT_ROPE_POS
    assert torch.equal(xd.cpu(), x)


# --------------------------------------------------------------------------- KV store
def test_kv_append_bit_exact(m, orc):
    cap, W, guard = 64, 128, 8
    K = rnd((cap + guard, W), 10)
    V = rnd((cap + guard, W), 11)
    k = rnd((5, W), 12)
    v = rnd((5, W), 13)
    pos = np.array([0, 63, 17, 18, 40], np.int32)
    Kd, Vd = dev(K), dev(V)
    err = err_word()
    m.minf_kv_append(Kd[:cap], Vd[:cap], dev(k), dev(v), dev(pos), err)
    torch.cuda.synchronize()
    Ko, Vo = K.numpy().copy(), V.numpy().copy()
    orc.kv_append(Ko[:cap], Vo[:cap], k.numpy(), v.numpy(), pos)
    assert np.array_equal(Kd.cpu().numpy(), Ko) and np.array_equal(Vd.cpu().numpy(), Vo)
    assert err.item() == 0


def test_kv_append_out_of_range_is_reported_not_written(m):
    cap, W, guard = 16, 64, 8
    K = rnd((cap + guard, W), 20)
    V = rnd((cap + guard, W), 21)
    k = rnd((3, W), 22)
    v = rnd((3, W), 23)
    Kd, Vd = dev(K), dev(V)
    err = err_word()
    m.minf_kv_append(Kd[:cap], Vd[:cap], dev(k), dev(v), dev(np.array([2, cap, -3], np.int32)), err)
    torch.cuda.synchronize()
    assert err.item() & m.ERRBIT_STORE_POS
    Kn, Vn = Kd.cpu(), Vd.cpu()
    assert torch.equal(Kn[2], k[0]) and torch.equal(Vn[2], v[0])      # the valid row is written
    rest = [i for i in range(cap + guard) if i != 2]
    assert torch.equal(Kn[rest], K[rest]) and torch.equal(Vn[rest], V[rest])  # nothing else moved


def test_rope_kv_append_fused(m, orc):
    nh, nk, hd, hdkv, cap = 16, 8, 128, 128, 1023
    nt = 7
    pos = np.array([0, 1, 100, 511, 574, 1000, 1022], np.int32)
    q = rnd((nt, nh * hd), 30)
    k = rnd((nt, nk * hdkv), 31)
    v = rnd((nt, nk * hdkv), 32)
    K = rnd((cap, nk * hdkv), 33)
    V = rnd((cap, nk * hdkv), 34)
    qd, kd, vd, Kd, Vd = dev(q), dev(k), dev(v), dev(K), dev(V)
    err = err_word()
    m.minf_rope_kv_append(qd, kd, vd, dev(pos), nh, nk, hd, hdkv, 1e6, 1.0, 0, Kd, Vd, err)
    # the same k through the standalone RoPE kernel
    k_alone = dev(k)
    m.minf_rope(k_alone, dev(pos), nk, hdkv, 1e6, 1.0, 0, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    close(qd.cpu(), orc.rope(q.numpy().copy(), pos, nh, hd, 1e6), what="q")
    close(kd.cpu(), orc.rope(k.numpy().copy(), pos, nk, hdkv, 1e6), what="k")
    assert torch.equal(kd.cpu(), k_alone.cpu())
    Kn, Vn = Kd.cpu(), Vd.cpu()
    Vo = V.numpy().copy()
    Vo[pos] = v.numpy()
    assert np.array_equal(Vn.numpy(), Vo)                       # V rows: bit-exact copy
    assert torch.equal(Kn[pos], k_alone.cpu())                  # K rows: the GPU's own RoPE output
    keep = np.setdiff1d(np.arange(cap), pos)
    assert torch.equal(Kn[keep], K[keep])


# --------------------------------------------------------------------------- decode attention
def _decode_case(m, orc, nh, nk, hd, hdkv, caps, lengths, seed, arena=True):
    W = nk * hdkv
    n_seq = len(caps)
    offs = np.concatenate([[0], np.cumsum(caps)[:-1]]).astype(np.int64)
    rows = int(np.sum(caps))
    K = rnd((rows, W), seed)
    V = rnd((rows, W), seed + 1)
    q = rnd((n_seq, nh, hd), seed + 2)
    pos = np.array(lengths, np.int32)
    out = torch.empty(n_seq, nh * hdkv, device="cuda")
    max_cap = int(max(caps))
    ws = m.kv.decode_workspace(n_seq, nh, nk, hdkv, max_cap)
    err = err_word()
    scale = float(np.float32(1.0) / np.sqrt(np.float32(hd)))
    m.minf_gqa_attn_decode(out, dev(q), dev(K), dev(V), dev(offs), dev(np.array(caps, np.int32)),
                           max_cap, dev(pos), nh, nk, hd, hdkv, scale, ws, err)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for s in range(n_seq):
        o, c = int(offs[s]), int(caps[s])
        if pos[s] < 0:  # empty window: defined as a zero output
            assert not np.any(got[s]), f"decode seq {s}: empty window gave a non-zero output"
            continue
        ref = orc.gqa_attn(q[s:s + 1].numpy(), K[o:o + c].numpy(), V[o:o + c].numpy(), [pos[s]], nh, nk,
                           hd, hdkv, scale=scale)
        close(got[s:s + 1], ref, what=f"decode seq {s} (L={pos[s] + 1})")
    return err, ws


@pytest.mark.parametrize("L", [1, 2, 31, 32, 33, 100, 128, 257, 575, 1023])
def test_decode_qwen3_geometry(m, orc, L):
    err, _ = _decode_case(m, orc, 16, 8, 128, 128, [1023], [L - 1], seed=L)
    assert err.item() == 0


@pytest.mark.parametrize("geom,caps,seed", [((14, 2, 64, 64), [639], 300),            # 7 heads a unit: ticket merge
                                             ((16, 8, 128, 128), [1023, 700], 310),    # 2 heads a unit: polling merge
                                             ((16, 2, 64, 64), [900, 300, 640], 320)])  # 8 heads a unit
def test_decode_workspace_left_clean(m, orc, geom, caps, seed):
    """Three calls with multi-split windows on one workspace, each against the oracle: after
    every call the workspace is zero except the layout tag (partials consumed, counters and
    merge tickets back at zero), so graph replays need no clearing."""
    nh, nk, hd, hdkv = geom
    W = nk * hdkv
    offs = np.concatenate([[0], np.cumsum(caps)[:-1]]).astype(np.int64)
    rows = int(np.sum(caps))
    ws = m.kv.decode_workspace(len(caps), nh, nk, hdkv, max(caps))
    scale = float(np.float32(1.0) / np.sqrt(np.float32(hd)))
    for call in range(3):
        K = rnd((rows, W), seed + 10 * call)
        V = rnd((rows, W), seed + 10 * call + 1)
        q = rnd((len(caps), nh, hd), seed + 10 * call + 2)
        pos = np.array([c - 1 - 37 * call for c in caps], np.int32)  # long windows: several splits
        out = torch.empty(len(caps), nh * hdkv, device="cuda")
        err = err_word()
        m.minf_gqa_attn_decode(out, dev(q), dev(K), dev(V), dev(offs), dev(np.array(caps, np.int32)), max(caps),
                               dev(pos), nh, nk, hd, hdkv, scale, ws, err)
        torch.cuda.synchronize()
        assert err.item() == 0
        got = out.cpu().numpy()
        for s_, (o, c) in enumerate(zip(offs, caps)):
            ref = orc.gqa_attn(q[s_:s_ + 1].numpy(), K[o:o + c].numpy(), V[o:o + c].numpy(), [pos[s_]], nh, nk, hd,
                               hdkv, scale=scale)
            close(got[s_:s_ + 1], ref, what=f"call {call} seq {s_}")
        words = ws.cpu().numpy().view(np.int32).copy()
        assert (words[4] >> 16) & 0xFFFF == 0x4D49  # the decode layout's tag
        words[4] = 0
        assert not words.any(), f"call {call}: {int(np.count_nonzero(words))} workspace words left non-zero"


@pytest.mark.parametrize("L", [1, 9, 128, 639])
def test_decode_qwen25_geometry(m, orc, L):
    err, _ = _decode_case(m, orc, 14, 2, 64, 64, [639], [L - 1], seed=100 + L)
    assert err.item() == 0


@pytest.mark.parametrize("geom", [(8, 8, 64, 64), (4, 1, 128, 128), (32, 4, 128, 128), (16, 2, 64, 64),
                                  (12, 4, 128, 64), (6, 2, 256, 128)])
def test_decode_other_geometries(m, orc, geom):
    nh, nk, hd, hdkv = geom
    err, _ = _decode_case(m, orc, nh, nk, hd, hdkv, [300, 77], [299, 40], seed=sum(geom))
    assert err.item() == 0


def test_decode_batched_ragged(m, orc):
    r = np.random.default_rng(5)
    lengths = [int(x) for x in r.integers(1, 700, size=12)] + [1, 2, 699]
    caps = [ln + 5 for ln in lengths]
    err, _ = _decode_case(m, orc, 16, 8, 128, 128, caps, [ln - 1 for ln in lengths], seed=7)
    assert err.item() == 0


def test_decode_batch_longest_first_with_long_windows(m, orc):
    # Enough (sequence, kv head) pairs to fill the SMs: the batch is visited longest first and
    # units are drawn from the workspace counter; windows past 4096 rows are also split.  The
    # second call reuses the workspace, so the counter and tickets must have been reset.
    r = np.random.default_rng(11)
    for call in range(2):
        lengths = [int(x) for x in r.integers(1, 1500, size=21)] + [9001, 4097, 4096, 1, 2, 1025]
        caps = [ln + 3 for ln in lengths]
        caps[-3] = 1  # window clamped to a one-row region (pos >= cap flags the attention bit)
        pos = [ln - 1 for ln in lengths]
        pos[-3] = 5
        err, _ = _decode_case(m, orc, 16, 8, 128, 128, caps, pos, seed=90 + call)
        assert err.item() == 0x4


def test_decode_batch_empty_window_is_zero_and_flagged(m, orc):
    r = np.random.default_rng(12)
    lengths = [int(x) for x in r.integers(1, 400, size=40)]
    pos = [ln - 1 for ln in lengths]
    pos[7] = -1
    err, _ = _decode_case(m, orc, 14, 2, 64, 64, [ln + 2 for ln in lengths], pos, seed=13)
    assert err.item() == 0x4


def test_decode_batch_beyond_sort_limit(m, orc):
    # more sequences than the longest-first ordering handles: visited in index order
    r = np.random.default_rng(14)
    lengths = [int(x) for x in r.integers(1, 200, size=300)]
    err, _ = _decode_case(m, orc, 16, 8, 128, 128, [ln + 1 for ln in lengths], [ln - 1 for ln in lengths],
                          seed=15)
    assert err.item() == 0


def test_decode_window_clamps_and_flags(m, orc):
    # pos >= cap: the window is the whole region (as nkv = min(max pos + 1, n_ctx)) and the bit is set
    err, _ = _decode_case(m, orc, 16, 8, 128, 128, [64], [64], seed=3)
    assert err.item() & 0x4


def test_decode_repeat_calls_reuse_workspace(m, orc):
    # the workspace is left clean, so back-to-back calls need no clearing
    for i in range(3):
        err, ws = _decode_case(m, orc, 16, 8, 128, 128, [4096], [4095 - 7 * i], seed=50 + i)
        assert err.item() == 0


# --------------------------------------------------------------------------- layer step
def test_layer_step_single_decode_config(m, orc):
    """Single decode step, one layer, Qwen2.5-0.5B shape: 127 cached rows (seed 0), token at 127."""
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN25_05B
    cap, p = 639, wl.SINGLE_STEP_CACHED_ROWS
    kc, vc = wl.cache_rows(g, "single-step", 0, p)
    inp = wl.layer_inputs(g, "single-step", 0, 1)
    K = torch.zeros(cap, g.row_width)
    V = torch.zeros(cap, g.row_width)
    K[:p], V[:p] = kc, vc
    d = {k: dev(v) for k, v in inp.items()}
    Kd, Vd = dev(K), dev(V)
    xn = torch.empty_like(d["h"])
    out = torch.empty(1, g.out_width, device="cuda")
    ws = m.kv.decode_workspace(1, g.n_head, g.n_kv_head, g.hd_kv, cap)
    err = err_word()
    m.minf_layer_attn_step(xn, d["h"], d["gain"], g.eps, d["q"], d["k"], d["v"], dev(np.array([p], np.int32)),
                           Kd, Vd, g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    q, k = inp["q"].numpy().copy(), inp["k"].numpy().copy()
    Ko, Vo = K.numpy().copy(), V.numpy().copy()
    xn_ref, out_ref = orc.layer_attn_step(inp["h"].numpy(), inp["gain"].numpy(), q, k, inp["v"].numpy(), [p],
                                          Ko, Vo, n_head=g.n_head, n_kv_head=g.n_kv_head, hd=g.hd,
                                          hd_kv=g.hd_kv, eps=g.eps, theta=g.theta)
    assert err.item() == 0
    close(xn.cpu(), xn_ref, what="xn")
    close(d["q"].cpu(), q, what="q rotated")
    close(d["k"].cpu(), k, what="k rotated")
    close(out.cpu(), out_ref, what="out")
    assert np.array_equal(Vd.cpu().numpy(), Vo)
    close(Kd.cpu(), Ko, what="K region")


def test_layer_step_prefill_then_graph_replayed_decode(m, orc):
    """Decode loop in miniature (Qwen3-0.6B geometry): a prefill through the layer step, then
    decode steps replayed from one captured CUDA graph with only the position changing."""
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN3_06B
    n_prompt, cap, steps = 40, 64, 6
    inp = wl.layer_inputs(g, "loop-test", 0, n_prompt + steps)
    Kd = torch.zeros(cap, g.row_width, device="cuda")
    Vd = torch.zeros(cap, g.row_width, device="cuda")
    err = err_word()
    ws = m.kv.prefill_workspace(n_prompt, g.n_head, g.n_kv_head, g.hd_kv, cap)
    d = {k: dev(v[:n_prompt]) for k, v in inp.items() if k != "gain"}
    gain = dev(inp["gain"])
    xn = torch.empty_like(d["h"])
    out = torch.empty(n_prompt, g.out_width, device="cuda")
    m.minf_layer_attn_step(xn, d["h"], gain, g.eps, d["q"], d["k"], d["v"], dev(np.arange(n_prompt, dtype=np.int32)),
                           Kd, Vd, g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    Ko = np.zeros((cap, g.row_width), np.float32)
    Vo = np.zeros((cap, g.row_width), np.float32)
    q0, k0 = inp["q"][:n_prompt].numpy().copy(), inp["k"][:n_prompt].numpy().copy()
    _, out_ref = orc.layer_attn_step(inp["h"][:n_prompt].numpy(), inp["gain"].numpy(), q0, k0,
                                     inp["v"][:n_prompt].numpy(), np.arange(n_prompt), Ko, Vo,
                                     n_head=g.n_head, n_kv_head=g.n_kv_head, hd=g.hd, hd_kv=g.hd_kv,
                                     eps=g.eps, theta=g.theta, n_threads=8)
    close(out.cpu(), out_ref, atol=TC_ATOL, rtol=0.0, what="prefill out (tensor cores, TF32)")
    # decode: static buffers, one capture, replays with a new position each time
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    hq = torch.empty(1, g.n_embd, device="cuda")
    qq = torch.empty(1, g.q_width, device="cuda")
    kk = torch.empty(1, g.row_width, device="cuda")
    vv = torch.empty(1, g.row_width, device="cuda")
    xo = torch.empty(1, g.n_embd, device="cuda")
    oo = torch.empty(1, g.out_width, device="cuda")
    wsd = m.kv.decode_workspace(1, g.n_head, g.n_kv_head, g.hd_kv, cap)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        pos.fill_(n_prompt)  # warm-up call outside the capture
    stream.synchronize()
    Kw, Vw = Kd.clone(), Vd.clone()
    with torch.cuda.graph(graph, stream=stream):
        m.minf_layer_attn_step(xo, hq, gain, g.eps, qq, kk, vv, pos, Kw, Vw, g.n_head, g.n_kv_head, g.hd,
                               g.hd_kv, g.theta, 1.0, 0, oo, wsd, err)
    torch.cuda.synchronize()
    Kw.copy_(Kd)
    Vw.copy_(Vd)
    for i in range(steps):
        t = n_prompt + i
        hq.copy_(dev(inp["h"][t:t + 1]))
        qq.copy_(dev(inp["q"][t:t + 1]))
        kk.copy_(dev(inp["k"][t:t + 1]))
        vv.copy_(dev(inp["v"][t:t + 1]))
        pos.fill_(t)
        graph.replay()
        torch.cuda.synchronize()
        q1, k1 = inp["q"][t:t + 1].numpy().copy(), inp["k"][t:t + 1].numpy().copy()
        _, ref = orc.layer_attn_step(inp["h"][t:t + 1].numpy(), inp["gain"].numpy(), q1, k1,
                                     inp["v"][t:t + 1].numpy(), [t], Ko, Vo, n_head=g.n_head,
                                     n_kv_head=g.n_kv_head, hd=g.hd, hd_kv=g.hd_kv, eps=g.eps, theta=g.theta)
        close(oo.cpu(), ref, what=f"replay at pos {t}")
        assert np.array_equal(Vw.cpu().numpy(), Vo)
    assert err.item() == 0


@pytest.mark.parametrize("n_seq,hi", [(9, 600), (24, 5000)])
def test_layer_step_batched(m, orc, n_seq, hi):
    # 24 sequences x 8 kv heads fill the SMs: the fused kernel then draws units longest first
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN3_06B
    lengths = wl.batched_lengths(seed=3, n_seq=n_seq, lo=1, hi=hi)
    caps = [ln + 1 + 8 for ln in lengths]
    arena = m.kv.KvArena(1, g.row_width, caps)
    Kh = rnd((arena.rows, g.row_width), 70)
    Vh = rnd((arena.rows, g.row_width), 71)
    arena.k[0].copy_(Kh)
    arena.v[0].copy_(Vh)
    n = len(lengths)
    inp = wl.layer_inputs(g, "batched-test", 0, n)
    d = {k: dev(v) for k, v in inp.items()}
    pos = dev(np.array(lengths, np.int32))
    xn = torch.empty_like(d["h"])
    out = torch.empty(n, g.out_width, device="cuda")
    ws = m.kv.decode_workspace(n, g.n_head, g.n_kv_head, g.hd_kv, arena.max_cap)
    err = err_word()
    k_ar, v_ar = arena.view(0)
    m.minf_layer_attn_step_batched(xn, d["h"], d["gain"], g.eps, d["q"], d["k"], d["v"], pos, k_ar, v_ar,
                                   arena.row_off, arena.cap, arena.max_cap, g.n_head, g.n_kv_head, g.hd,
                                   g.hd_kv, g.theta, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    close(xn.cpu(), orc.rms_norm(inp["h"].numpy(), inp["gain"].numpy(), eps=g.eps), what="xn")
    got = out.cpu().numpy()
    for s in range(n):
        o, c = arena.offsets_host[s], arena.caps_host[s]
        Ko, Vo = Kh[o:o + c].numpy().copy(), Vh[o:o + c].numpy().copy()
        q, k = inp["q"][s:s + 1].numpy().copy(), inp["k"][s:s + 1].numpy().copy()
        _, ref = orc.layer_attn_step(inp["h"][s:s + 1].numpy(), inp["gain"].numpy(), q, k, inp["v"][s:s + 1].numpy(),
                                     [lengths[s]], Ko, Vo, n_head=g.n_head, n_kv_head=g.n_kv_head, hd=g.hd,
                                     hd_kv=g.hd_kv, eps=g.eps, theta=g.theta)
        close(got[s:s + 1], ref, what=f"batched seq {s}")
        assert np.array_equal(arena.v[0, o:o + c].cpu().numpy(), Vo)


# --------------------------------------------------------------------------- SiLU * up
@pytest.mark.parametrize("n", [4, 1000, 1 << 20, 1023, (1 << 23) + 40])  # the last: several grid strides
def test_silu_mul(m, orc, n):
    gate = rnd((n,), n, 4.0)
    up = rnd((n,), n + 1)
    y = torch.empty(n, device="cuda")
    m.minf_silu_mul(y, dev(gate), dev(up))
    torch.cuda.synchronize()
    close(y.cpu(), orc.silu_mul(gate.numpy(), up.numpy()), what="silu_mul")


# --------------------------------------------------------------------------- host errors
def test_host_errors_raise(m):
    q = torch.zeros(1, 4, 64, device="cuda")
    K = torch.zeros(8, 128, device="cuda")
    out = torch.zeros(1, 4 * 128, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.MinfError) as e:
        m.minf_gqa_attn_decode(out, q, K, K, None, None, 8, dev(np.array([0], np.int32)), 4, 1, 64, 128,
                               0.1, ws, err_word())
    assert e.value.status == m.MINF_ERR_GEOMETRY


# --------------------------------------------------------------------------- fused decode step
def _step_inputs(g, nt, seed):
    return {"h": rnd((nt, g.n_embd), seed), "gain": torch.rand(g.n_embd, generator=torch.Generator().manual_seed(seed + 1)) + 0.5,
            "q": rnd((nt, g.q_width), seed + 2), "k": rnd((nt, g.row_width), seed + 3),
            "v": rnd((nt, g.row_width), seed + 4)}


def test_fused_step_multilayer_graph_with_shared_workspace(m, orc):
    """Four layers captured in one graph (each layer one launch, programmatically dependent
    on the previous one, all sharing one workspace), replayed at two positions."""
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN3_06B
    n_layer, cap = 4, 300
    regions = m.kv.KvRegions(n_layer, g.row_width, cap)
    Kh = [rnd((cap, g.row_width), 200 + i) for i in range(n_layer)]
    Vh = [rnd((cap, g.row_width), 300 + i) for i in range(n_layer)]
    for i in range(n_layer):
        regions.k[i].copy_(Kh[i])
        regions.v[i].copy_(Vh[i])
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    err = err_word()
    ws = m.kv.decode_workspace(1, g.n_head, g.n_kv_head, g.hd_kv, cap)
    bufs = [{k: torch.empty_like(dev(v)) for k, v in _step_inputs(g, 1, 0).items()} for _ in range(n_layer)]
    for b in bufs:
        b["xn"] = torch.empty(1, g.n_embd, device="cuda")
        b["out"] = torch.empty(1, g.out_width, device="cuda")

    def step():
        for i, b in enumerate(bufs):
            K, V = regions.view(i)
            m.minf_layer_attn_step(b["xn"], b["h"], b["gain"], g.eps, b["q"], b["k"], b["v"], pos, K, V, g.n_head,
                                   g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, b["out"], ws, err)

    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    torch.cuda.synchronize()
    Ko = [k.numpy().copy() for k in Kh]
    Vo = [v.numpy().copy() for v in Vh]
    for p in (257, 258):
        inputs = [_step_inputs(g, 1, 1000 * p + i) for i in range(n_layer)]
        for b, x in zip(bufs, inputs):
            for key in ("h", "gain", "q", "k", "v"):
                b[key].copy_(dev(x[key]))
        pos.fill_(p)
        graph.replay()
        torch.cuda.synchronize()
        for i, (b, x) in enumerate(zip(bufs, inputs)):
            q, k = x["q"].numpy().copy(), x["k"].numpy().copy()
            xn_ref, ref = orc.layer_attn_step(x["h"].numpy(), x["gain"].numpy(), q, k, x["v"].numpy(), [p], Ko[i],
                                              Vo[i], n_head=g.n_head, n_kv_head=g.n_kv_head, hd=g.hd, hd_kv=g.hd_kv,
                                              eps=g.eps, theta=g.theta)
            close(b["out"].cpu(), ref, what=f"layer {i} out at pos {p}")
            close(b["xn"].cpu(), xn_ref, what=f"layer {i} xn")
            close(b["q"].cpu(), q, what=f"layer {i} q rotated")
            close(b["k"].cpu(), k, what=f"layer {i} k rotated")
            assert np.array_equal(regions.v[i].cpu().numpy(), Vo[i])
            close(regions.k[i].cpu(), Ko[i], what=f"layer {i} K region")
    assert err.item() == 0


@pytest.mark.parametrize("style", [0, 1])
def test_fused_step_matches_unfused_semantics(m, orc, style):
    """The fused one-launch step and the oracle agree for both RoPE styles, including
    the K row it appends, which must equal the standalone RoPE kernel's output bit for bit."""
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN25_05B
    cap, p = 200, 150
    K = rnd((cap, g.row_width), 61)
    V = rnd((cap, g.row_width), 62)
    x = _step_inputs(g, 1, 63)
    d = {k: dev(v) for k, v in x.items()}
    Kd, Vd = dev(K), dev(V)
    err = err_word()
    xn = torch.empty_like(d["h"])
    out = torch.empty(1, g.out_width, device="cuda")
    ws = m.kv.decode_workspace(1, g.n_head, g.n_kv_head, g.hd_kv, cap)
    k_alone = dev(x["k"])
    m.minf_rope(k_alone, dev(np.array([p], np.int32)), g.n_kv_head, g.hd_kv, g.theta, 1.0, style, err)
    m.minf_layer_attn_step(xn, d["h"], d["gain"], g.eps, d["q"], d["k"], d["v"], dev(np.array([p], np.int32)),
                           Kd, Vd, g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, style, out, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    q, k = x["q"].numpy().copy(), x["k"].numpy().copy()
    Ko, Vo = K.numpy().copy(), V.numpy().copy()
    _, ref = orc.layer_attn_step(x["h"].numpy(), x["gain"].numpy(), q, k, x["v"].numpy(), [p], Ko, Vo,
                                 n_head=g.n_head, n_kv_head=g.n_kv_head, hd=g.hd, hd_kv=g.hd_kv, eps=g.eps,
                                 theta=g.theta, style=style)
    close(out.cpu(), ref, what="out")
    close(d["q"].cpu(), q, what="q")
    assert torch.equal(d["k"].cpu(), k_alone.cpu())
    assert torch.equal(Kd[p].cpu(), k_alone[0].cpu())
    assert np.array_equal(Vd.cpu().numpy(), Vo)


def test_fused_step_position_beyond_region(m, orc):
    """pos >= cap: nothing is stored, both bits are set, the window is the whole region and
    q and k are still rotated -- the same as the three-launch path."""
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN3_06B
    cap, p = 96, 96
    K = rnd((cap + 4, g.row_width), 81)
    V = rnd((cap + 4, g.row_width), 82)
    x = _step_inputs(g, 1, 83)
    d = {k: dev(v) for k, v in x.items()}
    Kd, Vd = dev(K), dev(V)
    err = err_word()
    out = torch.empty(1, g.out_width, device="cuda")
    ws = m.kv.decode_workspace(1, g.n_head, g.n_kv_head, g.hd_kv, cap)
    m.minf_layer_attn_step(torch.empty_like(d["h"]), d["h"], d["gain"], g.eps, d["q"], d["k"], d["v"],
                           dev(np.array([p], np.int32)), Kd[:cap], Vd[:cap], g.n_head, g.n_kv_head, g.hd, g.hd_kv,
                           g.theta, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    assert err.item() & m.ERRBIT_STORE_POS and err.item() & m.ERRBIT_ATTN_POS
    assert torch.equal(Kd.cpu(), K) and torch.equal(Vd.cpu(), V)   # nothing written, guard rows intact
    q_ref = orc.rope(x["q"].numpy().copy(), [p], g.n_head, g.hd, g.theta)
    k_ref = orc.rope(x["k"].numpy().copy(), [p], g.n_kv_head, g.hd_kv, g.theta)
    close(d["q"].cpu(), q_ref, what="q")
    close(d["k"].cpu(), k_ref, what="k")
    ref = orc.gqa_attn(q_ref, K[:cap].numpy(), V[:cap].numpy(), [p], g.n_head, g.n_kv_head, g.hd, g.hd_kv)
    close(out.cpu(), ref, what="out (window clamped to the region)")


def test_layer_step_unfused_geometry(m, orc):
    """hd > hd_kv takes the three-launch path; same results as the oracle."""
    nh, nk, hd, hdkv, n_embd, cap, p = 4, 2, 128, 64, 256, 50, 33
    K = rnd((cap, nk * hdkv), 91)
    V = rnd((cap, nk * hdkv), 92)
    h = rnd((1, n_embd), 93)
    gain = torch.rand(n_embd, generator=torch.Generator().manual_seed(94)) + 0.5
    q = rnd((1, nh * hd), 95)
    k = rnd((1, nk * hdkv), 96)
    v = rnd((1, nk * hdkv), 97)
    d = {n: dev(t) for n, t in dict(h=h, gain=gain, q=q, k=k, v=v).items()}
    Kd, Vd = dev(K), dev(V)
    err = err_word()
    xn = torch.empty(1, n_embd, device="cuda")
    out = torch.empty(1, nh * hdkv, device="cuda")
    ws = m.kv.decode_workspace(1, nh, nk, hdkv, cap)
    m.minf_layer_attn_step(xn, d["h"], d["gain"], 1e-6, d["q"], d["k"], d["v"], dev(np.array([p], np.int32)), Kd, Vd,
                           nh, nk, hd, hdkv, 1e4, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    qo, ko = q.numpy().copy(), k.numpy().copy()
    Ko, Vo = K.numpy().copy(), V.numpy().copy()
    xn_ref, ref = orc.layer_attn_step(h.numpy(), gain.numpy(), qo, ko, v.numpy(), [p], Ko, Vo, n_head=nh,
                                      n_kv_head=nk, hd=hd, hd_kv=hdkv, eps=1e-6, theta=1e4)
    assert err.item() == 0
    close(out.cpu(), ref, what="out")
    close(xn.cpu(), xn_ref, what="xn")
    assert np.array_equal(Vd.cpu().numpy(), Vo)
