"""Seeded synthetic inputs and the workload shapes.

This module holds shapes and random draws only -- none of the attention stage's
arithmetic -- so that both the CUDA path's tests/benchmark and the CPU oracle
can be fed the same inputs without sharing any computation.

Shapes follow the model geometries the pages use ("11 . Attention, vec ops, and
the KV cache" §2.2/§2.4 for Qwen2.5-0.5B; "IV.2: Zero-copy KV cache" for
Qwen3-0.6B and its 512-row append headroom).  Distributions: hidden states,
q/k/v rows and cached K/V ~ N(0, 1); RMSNorm gains ~ U(0.5, 1.5).
"""
from __future__ import annotations

import dataclasses
import zlib

import torch

# Rows reserved beyond a prefill for in-place appends ("IV.2: Zero-copy KV
# cache", the cache appends in place: prompt + 512 rows of headroom).
KV_HEADROOM_ROWS = 512


@dataclasses.dataclass(frozen=True)
class Geometry:
    name: str
    n_embd: int
    n_head: int
    n_kv_head: int
    hd: int
    hd_kv: int
    n_layer: int
    theta: float = 1e6
    eps: float = 1e-6
    freq_scale: float = 1.0

    @property
    def row_width(self) -> int:  # K/V row width (n_kv_embd)
        return self.n_kv_head * self.hd_kv

    @property
    def q_width(self) -> int:
        return self.n_head * self.hd

    @property
    def out_width(self) -> int:
        return self.n_head * self.hd_kv


QWEN25_05B = Geometry("qwen2.5-0.5b", n_embd=896, n_head=14, n_kv_head=2, hd=64, hd_kv=64, n_layer=24)
QWEN3_06B = Geometry("qwen3-0.6b", n_embd=1024, n_head=16, n_kv_head=8, hd=128, hd_kv=128, n_layer=28)

# Workloads (sizes as named by the benchmark configurations).
SINGLE_STEP_CACHED_ROWS = 127          # one decode step, token at pos 127
PREFILL_TOKENS = 512                   # causal prefill, positions 0..511
DECODE_LOOP_PROMPT = 511               # decode loop: 511-token prefill ...
DECODE_LOOP_STEPS = 64                 # ... then 64 decode steps at pos 511..574
BATCHED_SEQS = 64                      # batched decode: 64 sequences
BATCHED_MAX_LEN = 8192                 # cached lengths ~ U{1..8192}
LONG_CONTEXT_SWEEP = (1024, 4096, 16384, 40960)  # cached rows; token at pos = n
LONG_CONTEXT_CAP = 40961


def sub_seed(*keys) -> int:
    """A deterministic 31-bit seed for a (workload, layer, tensor, ...) key."""
    return zlib.crc32("/".join(str(k) for k in keys).encode()) & 0x7FFFFFFF


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int, device="cpu") -> torch.Tensor:
    return torch.randn(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32)


def uniform(shape, lo: float, hi: float, seed: int, device="cpu") -> torch.Tensor:
    u = torch.rand(*shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    return u * (hi - lo) + lo


def layer_inputs(geom: Geometry, workload: str, layer: int, nt: int, device="cpu") -> dict:
    """Per-layer step inputs: h [nt, n_embd], gain [n_embd], q [nt, nh*hd],
    k [nt, nk*hd_kv], v [nt, nk*hd_kv]; each tensor from its own sub-seed."""
    return {
        "h": normal((nt, geom.n_embd), sub_seed(workload, layer, "h"), device),
        "gain": uniform((geom.n_embd,), 0.5, 1.5, sub_seed(workload, layer, "gain"), device),
        "q": normal((nt, geom.q_width), sub_seed(workload, layer, "q"), device),
        "k": normal((nt, geom.row_width), sub_seed(workload, layer, "k"), device),
        "v": normal((nt, geom.row_width), sub_seed(workload, layer, "v"), device),
    }


def cache_rows(geom: Geometry, workload: str, layer: int, rows: int, device="cpu"):
    """Pre-existing cached K and V rows [rows, W] ~ N(0, 1)."""
    k = normal((rows, geom.row_width), sub_seed(workload, layer, "K"), device)
    v = normal((rows, geom.row_width), sub_seed(workload, layer, "V"), device)
    return k, v


def batched_lengths(seed: int = 0, n_seq: int = BATCHED_SEQS, lo: int = 1,
                    hi: int = BATCHED_MAX_LEN) -> list[int]:
    """Cached lengths ~ U{lo..hi}, seeded."""
    g = _gen(sub_seed("batched-lengths", seed), "cpu")
    return [int(x) for x in torch.randint(lo, hi + 1, (n_seq,), generator=g)]
