"""GPU tests of two call contracts of the layer step, through the C ABI, against the CPU oracle.

Ordering.  minf_layer_attn_step reads nothing -- the position included -- before the launch
ahead of it on the stream has finished, so a decode loop that writes the position with a kernel
right before each call (an eager pos.fill_(t), no graph, the loop "13 . The decode loop and
graph reuse" describes in §2.3) gets the oracle's results.  The _chained form (early start) is
for a launch before it that writes neither the position nor cached rows; its results are the
same bits.

Workspace.  The workspace's control block (its first 256 bytes) records the layout of the last
call that used it.  A prefill step may follow decode steps on one workspace; a decode after a
prefill, a decode of another shape, or a workspace never zero-filled is refused on the device
(MINF_ERRBIT_WORKSPACE, the attention output left unwritten) until it is zero-filled again.
Every refusal here is made on the host, by the workspace's bytes: nothing faults or waits out a
budget.  Tolerances: |d| <= 1e-5 + 1e-4 |ref| element by element (fp32 CUDA-core outputs),
stored V rows bit-exact."""
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


def close(got, ref, what, atol=ATOL, rtol=RTOL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    d = np.abs(got - ref)
    bad = d > atol + rtol * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} elements off, max abs {d.max():.3g}"


def rnd(shape, seed):
    return torch.randn(*shape, generator=torch.Generator().manual_seed(seed))


def qwen3():
    from gqa_attention_kv_rope_gb300 import workloads as wl

    return wl.QWEN3_06B


# --------------------------------------------------------------------------- ordering
def test_eager_position_kernel_before_the_default_step(m, orc):
    """pos written by a fill kernel immediately before each decode step, eagerly, on one stream:
    every step matches the oracle (which appends its own rows as it goes)."""
    g = qwen3()
    cap, n0, steps = 400, 150, 8
    K0, V0 = rnd((cap, g.row_width), 1), rnd((cap, g.row_width), 2)
    K0[n0:] = 0
    V0[n0:] = 0
    Kd, Vd = K0.cuda(), V0.cuda()
    Ko, Vo = K0.numpy().copy(), V0.numpy().copy()
    gain = (torch.rand(g.n_embd, generator=torch.Generator().manual_seed(3)) + 0.5)
    gain_d = gain.cuda()
    ws = m.kv.decode_workspace(1, g.n_head, g.n_kv_head, g.hd_kv, cap)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    xn = torch.empty(1, g.n_embd, device="cuda")
    out = torch.empty(1, g.out_width, device="cuda")
    for i in range(steps):
        t = n0 + i
        h, q, k, v = (rnd((1, w), 100 * t + j) for j, w in enumerate((g.n_embd, g.q_width, g.row_width,
                                                                       g.row_width)))
        hd_, qd, kd, vd = h.cuda(), q.cuda(), k.cuda(), v.cuda()
        torch.cuda.synchronize()
        pos.fill_(t)  # a kernel, the launch just before the step
        m.minf_layer_attn_step(xn, hd_, gain_d, g.eps, qd, kd, vd, pos, Kd, Vd, g.n_head, g.n_kv_head, g.hd,
                               g.hd_kv, g.theta, 1.0, 0, out, ws, err)
        torch.cuda.synchronize()
        qo, ko = q.numpy().copy(), k.numpy().copy()
        xn_ref, ref = orc.layer_attn_step(h.numpy(), gain.numpy(), qo, ko, v.numpy(), [t], Ko, Vo,
                                          n_head=g.n_head, n_kv_head=g.n_kv_head, hd=g.hd, hd_kv=g.hd_kv,
                                          eps=g.eps, theta=g.theta)
        assert err.item() == 0, t
        close(out.cpu(), ref, f"out at pos {t}")
        close(xn.cpu(), xn_ref, f"xn at pos {t}")
        close(qd.cpu(), qo, f"q at pos {t}")
        assert np.array_equal(Vd[t].cpu().numpy(), Vo[t])
        close(Kd[t].cpu(), Ko[t], f"appended K row at pos {t}")


@pytest.mark.parametrize("kind", ["f32", "f16", "q8"])
def test_chained_form_gives_the_same_bits(m, kind):
    """Four layers on one workspace, eagerly: the default step and the early-start form give
    bit-identical outputs, rotated q and k, and regions."""
    g = qwen3()
    cap, p, n_layer = 600, 517, 4
    if kind == "f32":
        mk = lambda s: rnd((cap, g.row_width), s).cuda()
        fns = (m.minf_layer_attn_step, m.minf_layer_attn_step_chained)
    elif kind == "f16":
        mk = lambda s: rnd((cap, g.row_width), s).half().cuda()
        fns = (m.minf_layer_attn_step_f16, m.minf_layer_attn_step_chained_f16)
    else:
        rb = m.minf_q8_row_bytes(g.row_width)

        def mk(s):
            t = torch.randint(0, 256, (cap, rb), dtype=torch.uint8, generator=torch.Generator().manual_seed(s))
            t[:, g.row_width:g.row_width + g.row_width // 16].view(torch.float16).fill_(1.0 / 64)
            t[:, g.row_width + g.row_width // 16:] = 0
            return t.cuda()
        fns = (m.minf_layer_attn_step_q8, m.minf_layer_attn_step_chained_q8)
    regions = [(mk(10 + 2 * i), mk(11 + 2 * i)) for i in range(n_layer)]
    ins = [{n: rnd((1, w), 50 + 5 * i + j).cuda() for j, (n, w) in
            enumerate((("h", g.n_embd), ("q", g.q_width), ("k", g.row_width), ("v", g.row_width)))}
           for i in range(n_layer)]
    gain = torch.ones(g.n_embd, device="cuda")
    pos = torch.tensor([p], dtype=torch.int32, device="cuda")
    res = []
    for fn in fns:
        regs = [(K.clone(), V.clone()) for K, V in regions]
        xs = [{n: t.clone() for n, t in d.items()} for d in ins]
        outs = [torch.empty(1, g.out_width, device="cuda") for _ in range(n_layer)]
        xns = [torch.empty(1, g.n_embd, device="cuda") for _ in range(n_layer)]
        ws = m.kv.decode_workspace(1, g.n_head, g.n_kv_head, g.hd_kv, cap)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        for i in range(n_layer):
            fn(xns[i], xs[i]["h"], gain, g.eps, xs[i]["q"], xs[i]["k"], xs[i]["v"], pos, regs[i][0], regs[i][1],
               g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, outs[i], ws, err)
        torch.cuda.synchronize()
        assert err.item() == 0
        res.append((outs, xns, xs, regs))
    (o0, x0, s0, r0), (o1, x1, s1, r1) = res
    for i in range(n_layer):
        assert torch.equal(o0[i], o1[i]) and torch.equal(x0[i], x1[i])
        assert torch.equal(s0[i]["q"], s1[i]["q"]) and torch.equal(s0[i]["k"], s1[i]["k"])
        assert torch.equal(r0[i][0], r1[i][0]) and torch.equal(r0[i][1], r1[i][1])


# --------------------------------------------------------------------------- workspace
def _ctl(ws):
    return ws[:256].cpu().numpy().view(np.int32)


def _decode_step(m, g, ws, cap, p, seed, nan_out=True):
    """One default decode step on fresh regions; returns (out, err, K, V, inputs) on the host."""
    K = rnd((cap, g.row_width), seed).cuda()
    V = rnd((cap, g.row_width), seed + 1).cuda()
    x = {n: rnd((1, w), seed + 2 + j) for j, (n, w) in
         enumerate((("h", g.n_embd), ("q", g.q_width), ("k", g.row_width), ("v", g.row_width)))}
    d = {n: t.cuda() for n, t in x.items()}
    gain = torch.ones(g.n_embd, device="cuda")
    out = torch.full((1, g.out_width), float("nan") if nan_out else 0.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.minf_layer_attn_step(torch.empty(1, g.n_embd, device="cuda"), d["h"], gain, g.eps, d["q"], d["k"], d["v"],
                           torch.tensor([p], dtype=torch.int32, device="cuda"), K, V, g.n_head, g.n_kv_head, g.hd,
                           g.hd_kv, g.theta, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(err.item()), K.cpu().numpy(), V.cpu().numpy(), x


def _decode_ref(orc, g, x, K, V, p):
    q = x["q"].numpy().copy()
    orc.rope(q.reshape(1, g.n_head, g.hd), [p], g.n_head, g.hd, g.theta)
    return orc.gqa_attn(q.reshape(1, g.n_head, g.hd), K, V, [p], g.n_head, g.n_kv_head, g.hd, g.hd_kv)


def _prefill_step(m, g, ws, cap, nt, seed):
    x = {n: rnd((nt, w), seed + j) for j, (n, w) in
         enumerate((("h", g.n_embd), ("q", g.q_width), ("k", g.row_width), ("v", g.row_width)))}
    d = {n: t.cuda() for n, t in x.items()}
    K = torch.zeros(cap, g.row_width, device="cuda")
    V = torch.zeros(cap, g.row_width, device="cuda")
    gain = torch.ones(g.n_embd, device="cuda")
    out = torch.full((nt, g.out_width), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.minf_layer_attn_step(torch.empty(nt, g.n_embd, device="cuda"), d["h"], gain, g.eps, d["q"], d["k"], d["v"],
                           torch.arange(nt, dtype=torch.int32, device="cuda"), K, V, g.n_head, g.n_kv_head, g.hd,
                           g.hd_kv, g.theta, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(err.item()), x


def _prefill_ref(orc, g, x, cap, nt):
    q, k = x["q"].numpy().copy(), x["k"].numpy().copy()
    Ko = np.zeros((cap, g.row_width), np.float32)
    Vo = np.zeros((cap, g.row_width), np.float32)
    _, out = orc.layer_attn_step(x["h"].numpy(), np.ones(g.n_embd, np.float32), q, k, x["v"].numpy(),
                                 np.arange(nt), Ko, Vo, n_head=g.n_head, n_kv_head=g.n_kv_head, hd=g.hd,
                                 hd_kv=g.hd_kv, eps=g.eps, theta=g.theta, n_threads=8)
    return out


def test_workspace_decode_then_prefill_then_decode(m, orc):
    g = qwen3()
    cap, nt = 1024, 300
    size = max(m.minf_attn_decode_workspace_bytes(1, g.n_head, g.n_kv_head, g.hd_kv, cap),
               m.minf_attn_prefill_workspace_bytes(nt, g.n_head, g.n_kv_head, g.hd_kv, cap))
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    # decode twice (same layout): both right
    for rep in range(2):
        out, err, K, V, x = _decode_step(m, g, ws, cap, 700, 10 + rep)
        assert err == 0
        close(out, _decode_ref(orc, g, x, K, V, 700), f"decode {rep}")
    assert not _ctl(ws)[:4].any()
    # a prefill step may follow decode on the same workspace
    out, err, x = _prefill_step(m, g, ws, cap, nt, 30)
    assert err == 0
    close(out, _prefill_ref(orc, g, x, cap, nt), "prefill step after decode", atol=2e-3, rtol=0.0)
    close(out, _prefill_ref(orc, g, x, cap, nt), "prefill step after decode (fp32 bound)")
    # decode after the prefill: refused, its output left as it was
    out, err, _, _, _ = _decode_step(m, g, ws, cap, 700, 40)
    assert err & m.ERRBIT_WORKSPACE and not err & m.ERRBIT_TIMEOUT
    assert np.isnan(out).all()
    # zero-filled again: accepted
    ws.zero_()
    out, err, K, V, x = _decode_step(m, g, ws, cap, 700, 50)
    assert err == 0
    close(out, _decode_ref(orc, g, x, K, V, 700), "decode after zero-fill")


def test_workspace_decode_of_another_shape_is_refused(m, orc):
    g = qwen3()
    small, large = 300, 3000  # 5 and 19 splits per kv head: two layouts
    size = max(m.minf_attn_decode_workspace_bytes(1, g.n_head, g.n_kv_head, g.hd_kv, c) for c in (small, large))
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    out, err, K, V, x = _decode_step(m, g, ws, large, 2500, 60)
    assert err == 0
    close(out, _decode_ref(orc, g, x, K, V, 2500), "large")
    out, err, _, _, _ = _decode_step(m, g, ws, small, 250, 61)
    assert err & m.ERRBIT_WORKSPACE and np.isnan(out).all()
    ws.zero_()
    out, err, K, V, x = _decode_step(m, g, ws, small, 250, 62)
    assert err == 0
    close(out, _decode_ref(orc, g, x, K, V, 250), "small after zero-fill")


def test_workspace_never_zero_filled_is_refused(m):
    """A workspace of 0xFF bytes (never zero-filled): the decode step and the single-launch
    prefill step both refuse it -- no barrier is entered, no wait runs out."""
    g = qwen3()
    cap, nt = 1024, 300
    size = max(m.minf_attn_decode_workspace_bytes(1, g.n_head, g.n_kv_head, g.hd_kv, cap),
               m.minf_attn_prefill_workspace_bytes(nt, g.n_head, g.n_kv_head, g.hd_kv, cap))
    ws = torch.full((size,), 255, dtype=torch.uint8, device="cuda")
    out, err, _, _, _ = _decode_step(m, g, ws, cap, 700, 70)
    assert err & m.ERRBIT_WORKSPACE and not err & m.ERRBIT_TIMEOUT and np.isnan(out).all()
    ws.fill_(255)
    out, err, _ = _prefill_step(m, g, ws, cap, nt, 80)
    assert err & m.ERRBIT_WORKSPACE and not err & m.ERRBIT_TIMEOUT and np.isnan(out).all()


def test_workspace_two_launch_prefill_after_decode_is_refused(m, orc):
    """The prefill attention alone (key chunks merged through tickets) after a decode call on
    the same workspace: refused; after a zero-fill: the oracle's result."""
    g = qwen3()
    cap, nt = 1024, 200
    size = max(m.minf_attn_decode_workspace_bytes(1, g.n_head, g.n_kv_head, g.hd_kv, cap),
               m.minf_attn_prefill_workspace_bytes(nt, g.n_head, g.n_kv_head, g.hd_kv, cap))
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    _, err, _, _, _ = _decode_step(m, g, ws, cap, 700, 90)
    assert err == 0
    K = rnd((cap, g.row_width), 91)
    V = rnd((cap, g.row_width), 92)
    q = rnd((nt, g.n_head, g.hd), 93)
    pos = np.arange(800, 800 + nt, dtype=np.int32)  # windows of 801..1000 keys: several key chunks
    scale = float(np.float32(1.0) / np.sqrt(np.float32(g.hd)))

    def run():
        out = torch.full((nt, g.out_width), float("nan"), device="cuda")
        e = torch.zeros(1, dtype=torch.int32, device="cuda")
        m.minf_gqa_attn_prefill(out, q.cuda(), K.cuda(), V.cuda(), torch.as_tensor(pos).cuda(), g.n_head,
                                g.n_kv_head, g.hd, g.hd_kv, scale, ws, e)
        torch.cuda.synchronize()
        return out.cpu().numpy(), int(e.item())

    out, err = run()
    assert err & m.ERRBIT_WORKSPACE and not err & m.ERRBIT_TIMEOUT
    ws.zero_()
    out, err = run()
    assert err == 0
    ref = orc.gqa_attn(q.numpy(), K.numpy(), V.numpy(), pos, g.n_head, g.n_kv_head, g.hd, g.hd_kv, scale=scale,
                       n_threads=8)
    close(out, ref, "prefill attention", atol=2e-3, rtol=0.0)
    close(out, ref, "prefill attention (fp32 bound)")
