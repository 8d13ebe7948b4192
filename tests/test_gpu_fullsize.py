"""Parity at the benchmark's full sizes, in the launch configuration bench.py times.

Long-context decode (Qwen3-0.6B shape, 28 layers, fp32 regions of 40961 rows, 9.4 GB): the
bench's captured 28-layer graph is replayed at every cache length of the sweep (1024, 4096,
16384, 40960 cached rows, token at pos = n); layers 0 and 27 are checked against the oracle
whole -- the RMSNorm row, q rotated at pos, the appended K row (rotated k) and V row (v, bit
for bit), rows other than pos untouched, and the attention output over [0, n].

Batched decode (64 sequences, lengths U{1..8192} from seed 0, 28 layers, one arena per
layer, ~60 GB): the bench's 28 batched layer steps run once; layers 0 and 27 are checked for
all 64 sequences, one sequence at a time on the host.

Decode loop (Qwen3-0.6B shape, 28 layers): the bench's 511-token prefill into 1023-row regions,
then its captured decode step replayed at pos 511..574; layers 0 and 27 checked at the prefill
and at every step.

Causal prefill (Qwen2.5-0.5B shape, 24 layers, 512 tokens): the bench's captured graph replayed
once; layers 0 and 23 checked whole.

Tolerance: |d| <= 1e-5 + 1e-4 |ref| per element (fp32 arithmetic against the oracle's
double-accumulated reference); tensor-core prefill outputs also within max-abs 2e-3."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-5, 1e-4
CHECK_LAYERS = (0, 27)


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
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} off, max abs {d.max():.3g}"


def test_long_context_sweep_full_size(m, orc):
    import bench
    from gqa_attention_kv_rope_gb300 import workloads as wl

    dev = torch.device("cuda")
    S = bench.setup_long_context(m, torch, wl, wl.LONG_CONTEXT_SWEEP[-1], dev)
    g = S["g"]
    inputs0 = S["inputs"].clone()  # the step rotates q and k in place
    regions0 = {layer: [t.clone() for t in S["regions"].view(layer)] for layer in CHECK_LAYERS}
    stream = torch.cuda.Stream()
    graph = bench.capture(torch, stream, lambda: bench.decode_step(m, S))
    scale = float(np.float32(1.0) / np.sqrt(np.float32(g.hd)))
    try:
        for n in wl.LONG_CONTEXT_SWEEP:
            S["inputs"].copy_(inputs0)
            S["pos"].fill_(n)
            S["err"].zero_()
            with torch.cuda.stream(stream):
                graph.replay()
            torch.cuda.synchronize()
            assert int(S["err"].item()) == 0, n
            for layer in CHECK_LAYERS:
                h0, q0, k0, v0 = (t.cpu().numpy() for t in bench.views({**S, "inputs": inputs0}, layer)[:4])
                _, q, k, _, xn, out = (t.cpu().numpy() for t in bench.views(S, layer))
                K, V = (t[: n + 1].cpu().numpy() for t in S["regions"].view(layer))
                gain = S["gains"][layer].cpu().numpy()
                close(xn, orc.rms_norm(h0, gain, g.eps), what=f"xn n={n} layer={layer}")
                q_ref = orc.rope(q0.copy().reshape(1, g.n_head, g.hd), [n], g.n_head, g.hd, g.theta)
                close(q, q_ref.reshape(1, -1), what=f"q n={n} layer={layer}")
                k_ref = orc.rope(k0.copy().reshape(1, g.n_kv_head, g.hd_kv), [n], g.n_kv_head, g.hd_kv, g.theta)
                close(k, k_ref.reshape(1, -1), what=f"k n={n} layer={layer}")
                assert np.array_equal(K[n], k[0]), "appended K row = the step's rotated k"
                assert np.array_equal(V[n], v0[0]), "appended V row = v, bit for bit"
                ref = orc.gqa_attn(q.reshape(1, g.n_head, g.hd), K, V, [n], g.n_head, g.n_kv_head, g.hd, g.hd_kv,
                                   scale=scale, n_threads=8)
                close(out, ref, what=f"out n={n} layer={layer}")
        # rows the sweep never appended to are as they were
        appended = list(wl.LONG_CONTEXT_SWEEP)
        for layer in CHECK_LAYERS:
            K, V = S["regions"].view(layer)
            K0, V0 = regions0[layer]
            keep = torch.ones(K.shape[0], dtype=torch.bool, device=K.device)
            keep[appended] = False
            assert torch.equal(K[keep], K0[keep]) and torch.equal(V[keep], V0[keep])
    finally:
        del graph, S, regions0
        torch.cuda.empty_cache()


def test_batched_full_size(m, orc):
    from gqa_attention_kv_rope_gb300 import workloads as wl

    dev = torch.device("cuda")
    g = wl.QWEN3_06B
    lengths = wl.batched_lengths(seed=0)
    caps = [ln + 1 + wl.KV_HEADROOM_ROWS for ln in lengths]
    arena = m.kv.KvArena(g.n_layer, g.row_width, caps, device=dev)
    gen = torch.Generator(device=dev)
    for layer in range(g.n_layer):
        gen.manual_seed(wl.sub_seed("batched", layer, "K"))
        arena.k[layer].normal_(generator=gen)
        gen.manual_seed(wl.sub_seed("batched", layer, "V"))
        arena.v[layer].normal_(generator=gen)
    n = len(lengths)
    pos = torch.tensor(lengths, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = m.kv.decode_workspace(n, g.n_head, g.n_kv_head, g.hd_kv, arena.max_cap, device=dev)
    L = []
    for layer in range(g.n_layer):
        d = {k: v.to(dev) for k, v in wl.layer_inputs(g, "batched", layer, n).items()}
        d["xn"] = torch.empty_like(d["h"])
        d["out"] = torch.empty(n, g.out_width, device=dev)
        L.append(d)
    orig = {layer: {k: L[layer][k].cpu().numpy().copy() for k in ("h", "gain", "q", "k", "v")} for layer in CHECK_LAYERS}

    def step():
        for layer in range(g.n_layer):
            d = L[layer]
            K, V = arena.view(layer)
            m.binding.minf_layer_attn_step_batched(d["xn"], d["h"], d["gain"], g.eps, d["q"], d["k"], d["v"], pos, K,
                                                   V, arena.row_off, arena.cap, arena.max_cap, g.n_head,
                                                   g.n_kv_head, g.hd, g.hd_kv, g.theta, 1.0, 0, d["out"], ws, err)

    try:
        step()  # the launches the bench's graph holds, in the same configuration
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        scale = float(np.float32(1.0) / np.sqrt(np.float32(g.hd)))
        row_off = arena.row_off.cpu().numpy()
        for layer in CHECK_LAYERS:
            o = orig[layer]
            d = L[layer]
            close(d["xn"].cpu().numpy(), orc.rms_norm(o["h"], o["gain"], g.eps), what=f"xn layer={layer}")
            q_ref = orc.rope(o["q"].copy().reshape(n, g.n_head, g.hd), lengths, g.n_head, g.hd, g.theta)
            q = d["q"].cpu().numpy()
            close(q, q_ref.reshape(n, -1), what=f"q layer={layer}")
            k = d["k"].cpu().numpy()
            out = d["out"].cpu().numpy()
            K, V = arena.view(layer)
            for s, ln in enumerate(lengths):
                r0 = int(row_off[s])
                Ks = K[r0:r0 + ln + 1].cpu().numpy()
                Vs = V[r0:r0 + ln + 1].cpu().numpy()
                assert np.array_equal(Ks[ln], k[s]) and np.array_equal(Vs[ln], o["v"][s]), (layer, s)
                ref = orc.gqa_attn(q[s].reshape(1, g.n_head, g.hd), Ks, Vs, [ln], g.n_head, g.n_kv_head, g.hd,
                                   g.hd_kv, scale=scale, n_threads=8)
                close(out[s:s + 1], ref, what=f"out layer={layer} seq={s} len={ln}")
    finally:
        del arena, L
        torch.cuda.empty_cache()


def test_decode_loop_full_size(m, orc):
    """Decode loop (Qwen3-0.6B shape, 28 layers): the bench's 511-token prefill into 1023-row
    regions, then its captured decode step replayed at pos 511..574 with the step's seeded
    inputs.  Layers 0 and 27 are checked at the prefill and at every step of the loop."""
    import bench
    from gqa_attention_kv_rope_gb300 import workloads as wl

    dev = torch.device("cuda")
    D = bench.setup_decode_loop(m, torch, wl, dev)
    g, n0, steps = D["g"], D["n0"], D["steps"]
    scale = float(np.float32(1.0) / np.sqrt(np.float32(g.hd)))
    inp = {layer: {k: v.cpu().numpy() for k, v in D["inputs"][layer].items()} for layer in CHECK_LAYERS}
    stream = torch.cuda.Stream()
    try:
        with torch.cuda.stream(stream):
            D["prefill"]()
        torch.cuda.synchronize()
        assert int(D["err"].item()) == 0
        pos_p = np.arange(n0, dtype=np.int32)
        for layer in CHECK_LAYERS:
            x, b = inp[layer], D["prefill_bufs"][layer]
            K, V = (t[:n0].cpu().numpy() for t in D["regions"].view(layer))
            q = b["q"].cpu().numpy()
            k = b["k"].cpu().numpy()
            close(b["xn"].cpu().numpy(), orc.rms_norm(x["h"][:n0], x["gain"], g.eps), what=f"prefill xn {layer}")
            close(q, orc.rope(x["q"][:n0].copy().reshape(n0, g.n_head, g.hd), pos_p, g.n_head, g.hd,
                              g.theta).reshape(n0, -1), what=f"prefill q {layer}")
            close(k, orc.rope(x["k"][:n0].copy().reshape(n0, g.n_kv_head, g.hd_kv), pos_p, g.n_kv_head, g.hd_kv,
                              g.theta).reshape(n0, -1), what=f"prefill k {layer}")
            assert np.array_equal(K, k) and np.array_equal(V, x["v"][:n0]), layer
            ref = orc.gqa_attn(q.reshape(n0, g.n_head, g.hd), K, V, pos_p, g.n_head, g.n_kv_head, g.hd, g.hd_kv,
                               scale=scale, n_threads=8)
            got = b["out"].cpu().numpy()
            assert np.abs(got - ref).max() <= 2e-3, f"prefill out {layer}: tensor-core bound"
            close(got, ref, what=f"prefill out {layer}")
        D["load"](n0)
        torch.cuda.synchronize()
        graph = bench.capture(torch, stream, D["step"])  # its warm-up ran the step at pos 511 once
        pos_host = torch.empty(1, dtype=torch.int32).pin_memory()
        for i in range(steps):
            t = n0 + i
            pos_host.fill_(t)
            with torch.cuda.stream(stream):
                D["load"](t)
                D["pos"].copy_(pos_host, non_blocking=True)
                graph.replay()
            torch.cuda.synchronize()
            assert int(D["err"].item()) == 0, t
            for layer in CHECK_LAYERS:
                x, b = inp[layer], D["bufs"][layer]
                K, V = (r[: t + 1].cpu().numpy() for r in D["regions"].view(layer))
                q, k = b["q"].cpu().numpy(), b["k"].cpu().numpy()
                close(b["xn"].cpu().numpy(), orc.rms_norm(x["h"][t:t + 1], x["gain"], g.eps), what=f"xn {t} {layer}")
                close(q, orc.rope(x["q"][t:t + 1].copy().reshape(1, g.n_head, g.hd), [t], g.n_head, g.hd,
                                  g.theta).reshape(1, -1), what=f"q {t} {layer}")
                close(k, orc.rope(x["k"][t:t + 1].copy().reshape(1, g.n_kv_head, g.hd_kv), [t], g.n_kv_head,
                                  g.hd_kv, g.theta).reshape(1, -1), what=f"k {t} {layer}")
                assert np.array_equal(K[t], k[0]) and np.array_equal(V[t], x["v"][t]), (t, layer)
                ref = orc.gqa_attn(q.reshape(1, g.n_head, g.hd), K, V, [t], g.n_head, g.n_kv_head, g.hd, g.hd_kv,
                                   scale=scale, n_threads=8)
                close(b["out"].cpu().numpy(), ref, what=f"out {t} {layer}")
        del graph
    finally:
        D.clear()
        torch.cuda.empty_cache()


def test_prefill_full_size(m, orc):
    """Causal prefill (Qwen2.5-0.5B shape, 24 layers, 512 tokens at 0..511): the bench's
    captured graph replayed once on its seeded inputs; layers 0 and 23 checked whole -- xn, q
    and k rotated, the stored K/V rows, and the tensor-core attention output (max-abs 2e-3 and
    the fp32 bound element by element)."""
    import bench
    from gqa_attention_kv_rope_gb300 import workloads as wl

    dev = torch.device("cuda")
    P = bench.setup_prefill(m, torch, wl, dev)
    g, nt = P["g"], P["nt"]
    layers = (0, g.n_layer - 1)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(g.hd)))
    stream = torch.cuda.Stream()
    try:
        graph = bench.capture(torch, stream, P["step"])  # the warm-up rotated q and k in place
        P["reset"]()
        P["regions"].k.zero_()
        P["regions"].v.zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        assert int(P["err"].item()) == 0
        pos = np.arange(nt, dtype=np.int32)
        for layer in layers:
            x = wl.layer_inputs(g, "prefill", layer, nt)
            d = P["layers"][layer]
            K, V = (t[:nt].cpu().numpy() for t in P["regions"].view(layer))
            q, k = d["q"].cpu().numpy(), d["k"].cpu().numpy()
            close(d["xn"].cpu().numpy(), orc.rms_norm(x["h"].numpy(), x["gain"].numpy(), g.eps), what=f"xn {layer}")
            close(q, orc.rope(x["q"].numpy().copy().reshape(nt, g.n_head, g.hd), pos, g.n_head, g.hd,
                              g.theta).reshape(nt, -1), what=f"q {layer}")
            close(k, orc.rope(x["k"].numpy().copy().reshape(nt, g.n_kv_head, g.hd_kv), pos, g.n_kv_head, g.hd_kv,
                              g.theta).reshape(nt, -1), what=f"k {layer}")
            assert np.array_equal(K, k) and np.array_equal(V, x["v"].numpy()), layer
            rest = P["regions"].k[layer][nt:]
            assert not rest.any().item(), "rows past the prompt untouched"
            ref = orc.gqa_attn(q.reshape(nt, g.n_head, g.hd), K, V, pos, g.n_head, g.n_kv_head, g.hd, g.hd_kv,
                               scale=scale, n_threads=8)
            got = d["out"].cpu().numpy()
            assert np.abs(got - ref).max() <= 2e-3, f"out {layer}: tensor-core bound"
            close(got, ref, what=f"out {layer}")
        del graph
    finally:
        P.clear()
        torch.cuda.empty_cache()
