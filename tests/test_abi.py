"""CPU-side checks of the C ABI: the library builds and loads, exports every symbol
the header declares, validates arguments before touching the GPU, and its RoPE
angular-speed table is bit-identical to the oracle's independently computed one."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from gqa_attention_kv_rope_gb300 import binding, build

    build.build()
    return binding.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "minf.h")).read()
    return sorted(set(re.findall(r"MINF_API\s+[\w\s\*]*?\b(minf_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("minf_rms_norm", "minf_rope", "minf_kv_append", "minf_gqa_attn_decode",
              "minf_gqa_attn_prefill", "minf_layer_attn_step"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from gqa_attention_kv_rope_gb300 import binding

    handle = ctypes.CDLL(binding.lib_path())
    for name in _declared():
        assert hasattr(handle, name), name


def test_binding_covers_every_declared_symbol():
    from gqa_attention_kv_rope_gb300 import binding

    assert sorted(binding._SIGS) == _declared()


def test_rope_table_bit_equal_to_oracle(lib, orc):
    from gqa_attention_kv_rope_gb300 import binding

    for hd, theta, fs in [(64, 1e6, 1.0), (128, 1e6, 1.0), (128, 1e4, 1.0), (4, 1e4, 1.0),
                          (256, 5e5, 0.125), (2, 10.0, 3.0)]:
        a = np.array(binding.minf_rope_freqs(hd, theta, fs), dtype=np.float32)
        b = orc.rope_freqs(hd, theta, fs)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), (hd, theta, fs)


def test_status_strings(lib):
    assert lib.minf_status_string(0) == b"ok"
    assert b"geometry" in lib.minf_status_string(2)
    assert lib.minf_version() >= 100


def test_host_validation_needs_no_gpu(lib):
    from gqa_attention_kv_rope_gb300 import binding as b

    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: validation rejects before any launch
    # hd < hd_kv is refused
    assert lib.minf_gqa_attn_decode(fake, fake, fake, fake, None, None, 16, 0, fake, 1, 4, 2, 64, 128,
                                    0.1, fake, 1 << 20, fake, None) == b.MINF_ERR_GEOMETRY
    # n_head not a multiple of n_kv_head
    assert lib.minf_gqa_attn_decode(fake, fake, fake, fake, None, None, 16, 0, fake, 1, 5, 2, 64, 64,
                                    0.1, fake, 1 << 20, fake, None) == b.MINF_ERR_GEOMETRY
    # an hd_kv the kernels do not implement
    assert lib.minf_gqa_attn_decode(fake, fake, fake, fake, None, None, 16, 0, fake, 1, 4, 2, 96, 96,
                                    0.1, fake, 1 << 20, fake, None) == b.MINF_ERR_UNSUPPORTED
    # null pointers, odd head dim, bad style
    assert lib.minf_rope(None, fake, 1, 1, 64, 1e4, 1.0, 0, fake, None) == b.MINF_ERR_ARG
    assert lib.minf_rope(fake, fake, 1, 1, 63, 1e4, 1.0, 0, fake, None) == b.MINF_ERR_ARG
    assert lib.minf_rope(fake, fake, 1, 1, 64, 1e4, 1.0, 2, fake, None) == b.MINF_ERR_ARG
    assert lib.minf_kv_append(fake, fake, 0, 128, fake, fake, fake, 1, fake, None) == b.MINF_ERR_ARG
    assert lib.minf_kv_append(fake, fake, 8, 126, fake, fake, fake, 1, fake, None) == b.MINF_ERR_ARG
    # misaligned float pointer
    assert lib.minf_kv_append(P(0x1004), fake, 8, 128, fake, fake, fake, 1, fake, None) == b.MINF_ERR_ARG
    # a workspace smaller than required
    need = lib.minf_attn_decode_workspace_bytes(1, 16, 8, 128, 4096)
    assert need > 0
    assert lib.minf_gqa_attn_decode(fake, fake, fake, fake, None, None, 4096, 0, fake, 1, 16, 8, 128,
                                    128, 0.1, fake, need - 256, fake, None) == b.MINF_ERR_WORKSPACE
    assert lib.minf_silu_mul(None, fake, fake, 4, None) == b.MINF_ERR_ARG


def test_workspace_sizes(lib):
    assert lib.minf_attn_decode_workspace_bytes(0, 16, 8, 128, 4096) == 0
    a = lib.minf_attn_decode_workspace_bytes(1, 16, 8, 128, 1023)
    b = lib.minf_attn_decode_workspace_bytes(1, 16, 8, 128, 40961)
    assert 0 < a <= b
    assert lib.minf_attn_decode_workspace_bytes(64, 16, 8, 128, 8705) > b // 64


def test_prefill_workspace_sizes(lib):
    """Every nt > 0 needs at least the single-launch step's 256 bytes of grid-barrier counts;
    more tokens or a longer region never need less."""
    from gqa_attention_kv_rope_gb300 import binding as b

    assert lib.minf_attn_prefill_workspace_bytes(0, 14, 2, 64, 1024) == 0
    sizes = [lib.minf_attn_prefill_workspace_bytes(nt, 14, 2, 64, 1024) for nt in (1, 2, 128, 129, 512, 900)]
    assert sizes[0] >= 256 and sizes == sorted(sizes)
    assert lib.minf_attn_prefill_workspace_bytes(512, 14, 2, 64, 4096) >= sizes[4]
    # the layer step refuses a short workspace before it launches anything
    P = ctypes.c_void_p
    fake = P(0x1000)
    need = lib.minf_attn_prefill_workspace_bytes(512, 14, 2, 64, 1024)
    assert lib.minf_layer_attn_step(fake, fake, fake, 1e-6, 896, fake, fake, fake, fake, 512, fake, fake, 1024, 14, 2,
                                    64, 64, 1e6, 1.0, 0, fake, fake, need - 1, fake, None) == b.MINF_ERR_WORKSPACE
    assert lib.minf_layer_attn_step(fake, fake, fake, 1e-6, 896, fake, fake, fake, fake, 512, fake, fake, 1024, 14, 2,
                                    64, 64, 1e6, 1.0, 0, fake, None, 0, fake, None) == b.MINF_ERR_WORKSPACE
