"""The device KV-region manager.

Each layer owns two persistent fp32 regions, K and V, of [cap, W] rows, where
row p holds the K (or V) vector of the token at position p ("11 . Attention, vec
ops, and the KV cache", §2.2 and §3.2.3).  They are allocated once, with
headroom beyond the prompt ("IV.2: Zero-copy KV cache": prompt + 512 rows), and
never move: an append writes one row in place, and attention reads the region
through a view, never a copy.  Because nothing is ever reallocated, a captured
decode step stays valid for every position ("13 . The decode loop and graph
reuse", §2.3/§2.5: the regions survive and positions are data).

Growing past `cap` is an error reported by the kernels, never a silent move; a
caller that needs more rows builds a new manager (and re-captures its graphs).

Regions may also be kept in f16 (dtype=torch.float16: IEEE binary16, §2.5 of the
same page: the GPU backends may keep the K/V regions in f16, halving the bytes an
attention read moves) or in Q8_0 blocks (dtype=torch.uint8: each row is W int8 quants,
W/32 binary16 scales and padding to 16 bytes, q8_row_bytes(W) bytes); the library's
`_f16` and `_q8` entry points read and write them.
"""
from __future__ import annotations

import torch

from . import binding

_KINDS = (torch.float32, torch.float16, torch.uint8)


def q8_row_bytes(row_width: int) -> int:
    """Bytes of a Q8_0 row of row_width values (quants, scales, padding to 16 bytes)."""
    if row_width <= 0 or row_width % 32:
        raise ValueError("Q8_0 rows hold whole 32-value blocks")
    return row_width + ((row_width // 32) * 2 + 15) // 16 * 16


def _row_cols(row_width: int, dtype) -> int:
    return q8_row_bytes(row_width) if dtype == torch.uint8 else row_width


class KvRegions:
    """Per-layer regions for one sequence: k[layer], v[layer] are [cap, W] views."""

    def __init__(self, n_layer: int, row_width: int, cap: int, device="cuda", dtype=torch.float32):
        if n_layer <= 0 or row_width <= 0 or cap <= 0:
            raise ValueError("n_layer, row_width and cap must be positive")
        if dtype not in _KINDS:
            raise ValueError("regions are float32, float16 or uint8 (Q8_0 rows)")
        self.n_layer, self.row_width, self.cap, self.dtype = n_layer, row_width, cap, dtype
        cols = _row_cols(row_width, dtype)
        self.k = torch.empty((n_layer, cap, cols), dtype=dtype, device=device)
        self.v = torch.empty((n_layer, cap, cols), dtype=dtype, device=device)

    def view(self, layer: int):
        """(K region, V region) of a layer: views into the persistent storage."""
        return self.k[layer], self.v[layer]

    @property
    def nbytes(self) -> int:
        return 2 * self.k.numel() * self.k.element_size()


class KvArena:
    """Batched regions: per layer one arena [sum(cap_s), W]; sequence s owns rows
    [row_off[s], row_off[s] + cap[s]).  The descriptors live on the device so a
    captured batched step reads them at replay time."""

    def __init__(self, n_layer: int, row_width: int, caps: list[int], device="cuda", dtype=torch.float32):
        if not caps or min(caps) <= 0:
            raise ValueError("every sequence needs a positive capacity")
        if dtype not in _KINDS:
            raise ValueError("arenas are float32, float16 or uint8 (Q8_0 rows)")
        self.n_layer, self.row_width, self.dtype = n_layer, row_width, dtype
        self.caps_host = list(int(c) for c in caps)
        offs, acc = [], 0
        for c in self.caps_host:
            offs.append(acc)
            acc += c
        self.offsets_host = offs
        self.rows = acc
        self.max_cap = max(self.caps_host)
        cols = _row_cols(row_width, dtype)
        self.k = torch.empty((n_layer, acc, cols), dtype=dtype, device=device)
        self.v = torch.empty((n_layer, acc, cols), dtype=dtype, device=device)
        self.row_off = torch.tensor(offs, dtype=torch.int64, device=device)
        self.cap = torch.tensor(self.caps_host, dtype=torch.int32, device=device)

    def view(self, layer: int):
        return self.k[layer], self.v[layer]

    def seq_view(self, layer: int, s: int):
        o, c = self.offsets_host[s], self.caps_host[s]
        return self.k[layer, o:o + c], self.v[layer, o:o + c]


def decode_workspace(n_seq: int, n_head: int, n_kv_head: int, hd_kv: int, max_cap: int,
                     device="cuda") -> torch.Tensor:
    """Zero-filled workspace for the split-KV decode path (the library leaves it zeroed)."""
    n = binding.minf_attn_decode_workspace_bytes(n_seq, n_head, n_kv_head, hd_kv, max_cap)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def prefill_workspace(nt: int, n_head: int, n_kv_head: int, hd_kv: int, cap: int,
                      device="cuda") -> torch.Tensor:
    n = binding.minf_attn_prefill_workspace_bytes(nt, n_head, n_kv_head, hd_kv, cap)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)
