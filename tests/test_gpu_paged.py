"""GPU parity of paged K/V regions ("IV.2: Zero-copy KV cache": the paged cache keeps a
sequence as scattered fixed-size blocks of a pool; "13 . The decode loop and graph reuse",
§2.2: the window the attention reads is an explicit input).

Pools are filled at random and each sequence's blocks are scattered over them; the kernels
are compared with the oracle's paged attention (which gathers the rows the table names) at
the fp32 tolerance, and the store bit for bit."""
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
    d = np.abs(got - ref)
    bad = d > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off, max abs {d.max():.3g}"


def rnd(shape, seed):
    return torch.randn(*shape, generator=torch.Generator().manual_seed(seed)).numpy()


def dev(x, dtype=None):
    t = torch.as_tensor(np.ascontiguousarray(x))
    return (t.to(dtype) if dtype is not None else t).cuda()


def err_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def scattered_table(n_seq, max_blocks, pool_blocks, seed):
    """Each sequence's blocks: distinct pool blocks in a random order."""
    perm = np.random.default_rng(seed).permutation(pool_blocks)[:n_seq * max_blocks]
    return perm.reshape(n_seq, max_blocks).astype(np.int32)


def _decode(m, orc, nh, nk, hd, hdkv, block_rows, max_blocks, pos, seed, f16=False):
    n_seq = len(pos)
    W = nk * hdkv
    pool_blocks = n_seq * max_blocks + 3  # spare blocks nobody owns
    Kp = rnd((pool_blocks * block_rows, W), seed)
    Vp = rnd((pool_blocks * block_rows, W), seed + 1)
    if f16:
        Kp, Vp = Kp.astype(np.float16).astype(np.float32), Vp.astype(np.float16).astype(np.float32)
    table = scattered_table(n_seq, max_blocks, pool_blocks, seed + 2)
    q = rnd((n_seq, nh, hd), seed + 3)
    pos = np.asarray(pos, np.int32)
    out = torch.empty(n_seq, nh * hdkv, device="cuda")
    ws = m.kv.decode_workspace(n_seq, nh, nk, hdkv, max_blocks * block_rows)
    err = err_word()
    scale = float(np.float32(1.0) / np.sqrt(np.float32(hd)))
    fn = m.minf_gqa_attn_decode_paged_f16 if f16 else m.minf_gqa_attn_decode_paged
    dt = torch.float16 if f16 else torch.float32
    fn(out, dev(q), dev(Kp, dt), dev(Vp, dt), dev(table), block_rows, dev(pos), nh, nk, hd, hdkv, scale, ws, err)
    torch.cuda.synchronize()
    ref = orc.gqa_attn_paged(q, Kp, Vp, table, block_rows, pos, nh, nk, hd, hdkv, scale=scale)
    close(out.cpu().numpy(), ref, what=f"paged decode (block_rows {block_rows})")
    return err


@pytest.mark.parametrize("block_rows", [16, 32, 64, 256, 1024])
def test_decode_paged_qwen3(m, orc, block_rows):
    max_blocks = max(2, 4096 // block_rows)
    cap = max_blocks * block_rows
    pos = [0, 17, block_rows - 1, block_rows, cap // 2 + 3, cap - 1, cap + 50]  # the last is clamped and flagged
    err = _decode(m, orc, 16, 8, 128, 128, block_rows, max_blocks, pos, seed=block_rows)
    assert err.item() == 0x4


@pytest.mark.parametrize("block_rows", [16, 128, 512])
def test_decode_paged_qwen25_f16(m, orc, block_rows):
    max_blocks = max(2, 2048 // block_rows)
    pos = [5, 300, max_blocks * block_rows - 1]
    err = _decode(m, orc, 14, 2, 64, 64, block_rows, max_blocks, pos, seed=200 + block_rows, f16=True)
    assert err.item() == 0


def test_decode_paged_batch_mode(m, orc):
    # enough (sequence, kv head) pairs to fill the SMs: units from the counter, longest first
    r = np.random.default_rng(7)
    pos = [int(x) for x in r.integers(0, 3000, size=26)]
    err = _decode(m, orc, 16, 8, 128, 128, 64, 48, pos, seed=300)
    assert err.item() == 0


def test_decode_paged_missing_block_is_reported(m, orc):
    nh, nk, hd, hdkv, block_rows, max_blocks = 16, 8, 128, 128, 64, 4
    W = nk * hdkv
    Kp = dev(rnd((8 * block_rows, W), 400))
    table = np.array([[0, 1, -1, 2], [3, 4, 5, 6]], np.int32)
    out, err = torch.empty(2, nh * hdkv, device="cuda"), err_word()
    ws = m.kv.decode_workspace(2, nh, nk, hdkv, max_blocks * block_rows)
    m.minf_gqa_attn_decode_paged(out, dev(rnd((2, nh, hd), 401)), Kp, Kp, dev(table), block_rows,
                                 dev(np.array([200, 100], np.int32)), nh, nk, hd, hdkv, 0.088, ws, err)
    torch.cuda.synchronize()
    assert err.item() & 0x10
    # a window that stops before the missing block needs nothing from it
    err2 = err_word()
    m.minf_gqa_attn_decode_paged(out, dev(rnd((2, nh, hd), 401)), Kp, Kp, dev(table), block_rows,
                                 dev(np.array([100, 100], np.int32)), nh, nk, hd, hdkv, 0.088, ws, err2)
    torch.cuda.synchronize()
    assert err2.item() == 0


@pytest.mark.parametrize("f16", [False, True])
def test_kv_append_paged(m, orc, f16):
    n_seq, max_blocks, block_rows, W = 5, 4, 32, 1024
    pool_blocks = 24
    P0 = rnd((pool_blocks * block_rows, W), 500)
    table = scattered_table(n_seq, max_blocks, pool_blocks, 501)
    k, v = rnd((n_seq, W), 502), rnd((n_seq, W), 503)
    pos = np.array([0, 31, 32, 127, 60], np.int32)
    dt = torch.float16 if f16 else torch.float32
    Kd, Vd, err = dev(P0, dt), dev(P0, dt), err_word()
    fn = m.minf_kv_append_paged_f16 if f16 else m.minf_kv_append_paged
    fn(Kd, Vd, dev(table), block_rows, dev(k), dev(v), dev(pos), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    if f16:
        Ko = orc.f32_to_f16(P0)
        Vo = Ko.copy()
        for s, p in enumerate(pos):
            row = table[s, p // block_rows] * block_rows + p % block_rows
            Ko[row], Vo[row] = orc.f32_to_f16(k[s]), orc.f32_to_f16(v[s])
        got_k, got_v = Kd.cpu().numpy().view(np.uint16), Vd.cpu().numpy().view(np.uint16)
    else:
        Ko, Vo = P0.copy(), P0.copy()
        orc.kv_append_paged(Ko, Vo, table, block_rows, k, v, pos)
        got_k, got_v = Kd.cpu().numpy(), Vd.cpu().numpy()
    assert np.array_equal(got_k, Ko) and np.array_equal(got_v, Vo)
    bad = table.copy()
    bad[1, 0] = -1
    err2 = err_word()
    fn(Kd, Vd, dev(bad), block_rows, dev(k), dev(v), dev(np.array([0, 5, 0, 0, 0], np.int32)), err2)
    torch.cuda.synchronize()
    assert err2.item() & 0x10


def _step_inputs(g, n, seed):
    h = rnd((n, g.n_embd), seed)
    gain = np.random.default_rng(seed).uniform(0.5, 1.5, g.n_embd).astype(np.float32)
    return h, gain, rnd((n, g.q_width), seed + 1), rnd((n, g.row_width), seed + 2), rnd((n, g.row_width), seed + 3)


@pytest.mark.parametrize("geom", ["qwen3", "unfused"])
def test_layer_step_paged_decode_loop(m, orc, geom):
    # four steps of a batch through one table: each step appends through the table and the next
    # reads the rows the earlier steps stored
    import dataclasses

    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN3_06B
    if geom == "unfused":  # hd != hd_kv: RMSNorm/RoPE/store launch, then the decode kernel
        g = dataclasses.replace(g, n_head=12, n_kv_head=4, hd=128, hd_kv=64)
    n, block_rows, max_blocks = 6, 64, 8
    pool_blocks = n * max_blocks + 2
    Kp0 = rnd((pool_blocks * block_rows, g.row_width), 600)
    Vp0 = rnd((pool_blocks * block_rows, g.row_width), 601)
    table = scattered_table(n, max_blocks, pool_blocks, 602)
    pos0 = np.array([0, 63, 64, 200, 400, 505], np.int32)
    Kd, Vd, td = dev(Kp0), dev(Vp0), dev(table)
    Ko, Vo = Kp0.copy(), Vp0.copy()
    ws = m.kv.decode_workspace(n, g.n_head, g.n_kv_head, g.hd_kv, max_blocks * block_rows)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(g.hd)))
    for step in range(4):
        h, gain, q, k, v = _step_inputs(g, n, 610 + 10 * step)
        pos = pos0 + step
        qd, kd = dev(q), dev(k)
        xn, out, err = torch.empty(n, g.n_embd, device="cuda"), torch.empty(n, g.out_width, device="cuda"), err_word()
        m.minf_layer_attn_step_paged(xn, dev(h), dev(gain), g.eps, qd, kd, dev(v), dev(pos), Kd, Vd, td, block_rows,
                                     g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, out, ws, err)
        torch.cuda.synchronize()
        assert err.item() == 0
        q_ref = orc.rope(q.copy(), pos, g.n_head, g.hd, g.theta)
        k_ref = orc.rope(k.copy(), pos, g.n_kv_head, g.hd_kv, g.theta)
        close(xn.cpu().numpy(), orc.rms_norm(h, gain, eps=g.eps), what="xn")
        close(qd.cpu().numpy(), q_ref.reshape(n, -1), what="q rotated")
        k_gpu = kd.cpu().numpy()
        close(k_gpu, k_ref.reshape(n, -1), what="k rotated")
        # the store: V as given, K as the GPU rotated it, through the table
        orc.kv_append_paged(Ko, Vo, table, block_rows, k_gpu, v, pos)
        assert np.array_equal(Vd.cpu().numpy(), Vo)
        assert np.array_equal(Kd.cpu().numpy(), Ko)
        ref = orc.gqa_attn_paged(q_ref.reshape(n, g.n_head, g.hd), Ko, Vo, table, block_rows, pos, g.n_head,
                                 g.n_kv_head, g.hd, g.hd_kv, scale=scale)
        close(out.cpu().numpy(), ref, what=f"out step {step}")


def test_layer_step_paged_f16_batch_mode(m, orc):
    from gqa_attention_kv_rope_gb300 import workloads as wl

    g = wl.QWEN3_06B
    n, block_rows, max_blocks = 24, 128, 24
    pool_blocks = n * max_blocks
    P = rnd((pool_blocks * block_rows, g.row_width), 700).astype(np.float16)
    table = scattered_table(n, max_blocks, pool_blocks, 701)
    pos = np.random.default_rng(702).integers(0, max_blocks * block_rows, size=n).astype(np.int32)
    Kd, Vd = dev(P), dev(P)
    h, gain, q, k, v = _step_inputs(g, n, 703)
    qd, kd = dev(q), dev(k)
    xn, out, err = torch.empty(n, g.n_embd, device="cuda"), torch.empty(n, g.out_width, device="cuda"), err_word()
    ws = m.kv.decode_workspace(n, g.n_head, g.n_kv_head, g.hd_kv, max_blocks * block_rows)
    m.minf_layer_attn_step_paged_f16(xn, dev(h), dev(gain), g.eps, qd, kd, dev(v), dev(pos), Kd, Vd, dev(table),
                                     block_rows, g.n_head, g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, out, ws, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    k_gpu = kd.cpu().numpy()
    Kn = Kd.cpu().numpy().view(np.uint16)
    Vn = Vd.cpu().numpy().view(np.uint16)
    P16 = P.view(np.uint16)
    Ko, Vo = P16.copy(), P16.copy()
    for s in range(n):
        row = table[s, pos[s] // block_rows] * block_rows + pos[s] % block_rows
        Ko[row], Vo[row] = orc.f32_to_f16(k_gpu[s]), orc.f32_to_f16(v[s])
    assert np.array_equal(Kn, Ko) and np.array_equal(Vn, Vo)
    q_ref = orc.rope(q.copy(), pos, g.n_head, g.hd, g.theta)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(g.hd)))
    ref = orc.gqa_attn_paged(q_ref.reshape(n, g.n_head, g.hd), orc.f16_to_f32(Kn), orc.f16_to_f32(Vn), table,
                             block_rows, pos, g.n_head, g.n_kv_head, g.hd, g.hd_kv, scale=scale)
    close(out.cpu().numpy(), ref, what="paged f16 batch")


def test_paged_rejects_bad_block_rows(m):
    from gqa_attention_kv_rope_gb300 import binding

    g_out = torch.empty(1, 1024, device="cuda")
    P = torch.zeros(96 * 2, 1024, device="cuda")
    ws = m.kv.decode_workspace(1, 16, 8, 128, 192)
    for br in (8, 48, 96):
        with pytest.raises(binding.MinfError) as e:
            m.minf_gqa_attn_decode_paged(g_out, torch.zeros(1, 16, 128, device="cuda"), P, P,
                                         torch.zeros(1, 2, dtype=torch.int32, device="cuda"), br,
                                         torch.zeros(1, dtype=torch.int32, device="cuda"), 16, 8, 128, 128, 0.1, ws,
                                         err_word())
        assert e.value.status == binding.MINF_ERR_UNSUPPORTED
