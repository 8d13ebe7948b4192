"""The allocation-free decode entry point (for callers that cannot allocate device memory):
called through the C ABI, its output must match minf_gqa_attn_decode's, which uses a
caller-allocated workspace, on two calls in a row that share the library's fixed scratch, and
both must match the CPU oracle (|d| <= 1e-5 + 1e-4 |ref| element by element), so that a
mistake the two entry points share cannot pass.  This file is collected last so that a failure
here does not hide the other GPU tests."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1e-5, 1e-4


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_attention_kv_rope_gb300 import binding, build

    build.build()
    return binding.lib()


def _rnd(shape, seed):
    return torch.randn(*shape, generator=torch.Generator().manual_seed(seed)).cuda()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def test_static_workspace_matches_the_allocating_entry_point(lib, orc):
    from gqa_attention_kv_rope_gb300 import binding, kv

    nh, nk, hd = 16, 8, 128
    caps = [700, 1500, 90, 4000]
    n = len(caps)
    rows = sum(caps)
    offs = torch.tensor(np.concatenate([[0], np.cumsum(caps)[:-1]]), dtype=torch.int64).cuda()
    cap_t = torch.tensor(caps, dtype=torch.int32).cuda()
    K = _rnd((rows, nk * hd), 1)
    V = _rnd((rows, nk * hd), 2)
    q = _rnd((n, nh, hd), 3)
    scale = float(np.float32(1.0) / np.sqrt(np.float32(hd)))
    max_cap = max(caps)
    ws = kv.decode_workspace(n, nh, nk, hd, max_cap)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, lengths in enumerate(([699, 1000, 89, 3999], [350, 1499, 10, 2048])):
        pos = torch.tensor(lengths, dtype=torch.int32).cuda()
        ref = torch.empty(n, nh * hd, device="cuda")
        got = torch.full((n, nh * hd), float("nan"), device="cuda")
        err_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
        err_got = torch.zeros(1, dtype=torch.int32, device="cuda")
        st = lib.minf_gqa_attn_decode(_ptr(ref), _ptr(q), _ptr(K), _ptr(V), _ptr(offs), _ptr(cap_t), max_cap,
                                      rows, _ptr(pos), n, nh, nk, hd, hd, scale, _ptr(ws), ws.numel(),
                                      _ptr(err_ref), stream)
        assert st == binding.MINF_OK
        st = lib.minf_gqa_attn_decode_static_ws(_ptr(got), _ptr(q), _ptr(K), _ptr(V), _ptr(offs), _ptr(cap_t),
                                                max_cap, rows, _ptr(pos), n, nh, nk, hd, hd, scale,
                                                _ptr(err_got), stream)
        assert st == binding.MINF_OK, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert err_got.item() == 0 and err_ref.item() == 0
        r, g = ref.cpu().numpy(), got.cpu().numpy()
        assert np.all(np.abs(g - r) <= ATOL + RTOL * np.abs(r)), f"call {call}: max abs {np.abs(g - r).max()}"
        # and the oracle, one sequence at a time over its own rows of the arena
        Kh, Vh, qh = K.cpu().numpy(), V.cpu().numpy(), q.cpu().numpy()
        o = offs.cpu().numpy()
        for s_, (c, ln) in enumerate(zip(caps, lengths)):
            Ks, Vs = Kh[o[s_]:o[s_] + c], Vh[o[s_]:o[s_] + c]
            want = orc.gqa_attn(qh[s_:s_ + 1], Ks, Vs, [ln], nh, nk, hd, hd, scale=scale, n_threads=8)
            d = np.abs(g[s_:s_ + 1].astype(np.float64) - want)
            assert np.all(d <= ATOL + RTOL * np.abs(want)), f"call {call}, sequence {s_}: max abs {d.max()}"


def test_static_workspace_rejects_oversized_calls(lib):
    from gqa_attention_kv_rope_gb300 import binding

    # 4096 sequences need far more than the fixed scratch: refused before any launch
    n, nh, nk, hd, max_cap = 4096, 16, 8, 128, 8192
    assert lib.minf_attn_decode_workspace_bytes(n, nh, nk, hd, max_cap) > (8 << 20)
    dummy = torch.zeros(16, device="cuda")
    pos = torch.zeros(n, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = lib.minf_gqa_attn_decode_static_ws(_ptr(dummy), _ptr(dummy), _ptr(dummy), _ptr(dummy), None, None,
                                            max_cap, 0, _ptr(pos), n, nh, nk, hd, hd, 0.1, _ptr(err),
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == binding.MINF_ERR_WORKSPACE
