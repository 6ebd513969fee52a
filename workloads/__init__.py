"""Seeded synthetic inputs for the Muon step: layouts and gradients.

This module builds what both sides of a parity check consume -- parameter
tables, partition tables, flat storage buffers and gradients -- and nothing
else.  It holds none of the method's arithmetic (no momentum, no
normalisation, no Newton-Schulz, no norms, no clipping); the CUDA library and
the CPU oracle each implement those on their own.

Table formats (little-endian, packed exactly like the C structs of the
library header):

* parameter row  ``{int64 offset; int32 rows, cols, num_heads, use_muon}``
  ``offset`` is the flat element index of element (0, 0); a parameter covers
  ``rows*cols`` consecutive flat indices in row-major order.
* partition row  ``{int64 flat_begin, flat_end, storage_offset}``
  flat index ``i`` of partition ``p`` lives at storage element
  ``storage_offset + (i - flat_begin)`` of every flat buffer (accum,
  momentum, master, gradient).

Layout reading (the pages give no byte layout): each parameter group is its
own flat segment, parameters packed back to back in group order, the segment
padded at its end to a multiple of ``alignment * nparts`` and cut into
``nparts`` equal partitions, one per emulated data-parallel rank.  This is how
a ZeRO-style flat buffer of one group is split ("Support Muon in
BF16_Optimizer with FP32 gradient accumulation": PR description -- flat,
rank-partitioned buffers with alignment padding).
"""
from __future__ import annotations

from dataclasses import dataclass, field
import math

import numpy as np

PARAM_DTYPE = np.dtype([("offset", "<i8"), ("rows", "<i4"), ("cols", "<i4"),
                        ("num_heads", "<i4"), ("use_muon", "<i4")])
PART_DTYPE = np.dtype([("flat_begin", "<i8"), ("flat_end", "<i8"),
                       ("storage_offset", "<i8")])

assert PARAM_DTYPE.itemsize == 24 and PART_DTYPE.itemsize == 24


@dataclass
class ParamSpec:
    name: str
    rows: int
    cols: int
    num_heads: int = 0
    use_muon: bool = True

    @property
    def numel(self) -> int:
        return self.rows * self.cols


@dataclass
class Layout:
    specs: list            # ParamSpec, table order
    params: np.ndarray     # PARAM_DTYPE
    parts: np.ndarray      # PART_DTYPE, sorted by flat_begin
    flat_size: int
    storage_size: int
    alignment: int
    nparts: int            # partitions per segment (emulated ranks)
    meta: dict = field(default_factory=dict)

    @property
    def n_muon_elements(self) -> int:
        return int(sum(s.numel for s in self.specs if s.use_muon))

    @property
    def n_param_elements(self) -> int:
        return int(sum(s.numel for s in self.specs))


def _round_up(x: int, m: int) -> int:
    return ((x + m - 1) // m) * m


def build_layout(groups, alignment: int, nparts: int, storage: str = "identity",
                 seed: int = 0) -> Layout:
    """Pack parameter groups into segments and cut each into ``nparts``.

    storage: "identity"   -- storage index == flat index;
             "rank_major" -- all partitions of rank 0 (in segment order),
                             then rank 1, ... (the storage of a real rank's
                             flat buffers laid side by side);
             "shuffled"   -- partitions in a seeded random order with
                             random gaps of 1..7 elements between them, so
                             storage offsets have arbitrary alignment.
    """
    specs, rows = [], []
    parts = []           # (flat_begin, flat_end, rank)
    cursor = 0
    for group in groups:
        seg_begin = cursor
        for s in group:
            specs.append(s)
            rows.append((cursor, s.rows, s.cols, s.num_heads, int(bool(s.use_muon))))
            cursor += s.numel
        seg_len = _round_up(max(cursor - seg_begin, 1), alignment * nparts)
        plen = seg_len // nparts
        for r in range(nparts):
            parts.append((seg_begin + r * plen, seg_begin + (r + 1) * plen, r))
        cursor = seg_begin + seg_len
    flat_size = cursor

    order = list(range(len(parts)))
    if storage == "identity":
        offsets = [p[0] for p in parts]
        storage_size = flat_size
    else:
        if storage == "rank_major":
            order.sort(key=lambda k: (parts[k][2], parts[k][0]))
            gaps = [0] * len(parts)
        elif storage == "shuffled":
            rng = np.random.default_rng(seed)
            order = list(rng.permutation(len(parts)))
            gaps = list(rng.integers(1, 8, size=len(parts)))
        else:
            raise ValueError(storage)
        offsets = [0] * len(parts)
        pos = 0
        for j, k in enumerate(order):
            pos += int(gaps[j])
            offsets[k] = pos
            pos += parts[k][1] - parts[k][0]
        storage_size = pos + 3

    ptab = np.zeros(len(rows), dtype=PARAM_DTYPE)
    for i, r in enumerate(rows):
        ptab[i] = r
    qtab = np.zeros(len(parts), dtype=PART_DTYPE)
    for i, (b, e, _) in enumerate(parts):
        qtab[i] = (b, e, offsets[i])
    return Layout(specs, ptab, qtab, flat_size, storage_size, alignment, nparts)


# ---------------------------------------------------------------- configs

def tiny_layout(nparts: int = 2, storage: str = "identity", seed: int = 0) -> Layout:
    """Two fp32 Muon matrices 17x13 and 9x17 plus an 8x5 auxiliary group,
    16-element alignment, 2 partitions per segment ("Support Muon in
    BF16_Optimizer with FP32 gradient accumulation": validation table, the
    eager engine E2E row)."""
    groups = [[ParamSpec("w17x13", 17, 13)],
              [ParamSpec("w9x17", 9, 17)],
              [ParamSpec("aux8x5", 8, 5, use_muon=False)]]
    return build_layout(groups, 16, nparts, storage, seed)


GPT2_DIM = 768
GPT2_FF = 3072


def gpt2_small_specs(layers: int = 12):
    d, f = GPT2_DIM, GPT2_FF
    out = []
    for l in range(layers):
        out += [ParamSpec(f"h{l}.q", d, d, 12), ParamSpec(f"h{l}.k", d, d, 12),
                ParamSpec(f"h{l}.v", d, d), ParamSpec(f"h{l}.o", d, d),
                ParamSpec(f"h{l}.up", f, d), ParamSpec(f"h{l}.down", d, f)]
    return out


def gpt2_small_layout(layers: int = 12, nparts: int = 8, storage: str = "identity",
                      seed: int = 0) -> Layout:
    return build_layout([gpt2_small_specs(layers)], 128, nparts, storage, seed)


def llama3_8b_specs(layers: int = 32):
    d, kv, f = 4096, 1024, 14336
    out = []
    for l in range(layers):
        out += [ParamSpec(f"l{l}.q", d, d), ParamSpec(f"l{l}.k", kv, d),
                ParamSpec(f"l{l}.v", kv, d), ParamSpec(f"l{l}.o", d, d),
                ParamSpec(f"l{l}.gate", f, d), ParamSpec(f"l{l}.up", f, d),
                ParamSpec(f"l{l}.down", d, f)]
    return out


def llama3_8b_layout(layers: int = 32, nparts: int = 64) -> Layout:
    return build_layout([llama3_8b_specs(layers)], 128, nparts)


def ragged_specs(count: int = 8192, seed: int = 1003):
    rng = np.random.default_rng([seed, 0xA11])
    rows = rng.choice([32, 64, 128, 256], size=count)
    cols = rng.choice([128, 256, 512, 1024], size=count)
    tall = rng.random(count) < 0.5
    out = []
    for i in range(count):
        r, c = int(rows[i]), int(cols[i])
        if tall[i]:
            r, c = c, r
        out.append(ParamSpec(f"r{i}", r, c))
    return out


def ragged_layout(count: int = 8192, nparts: int = 1, seed: int = 1003) -> Layout:
    return build_layout([ragged_specs(count, seed)], 128, nparts)


SWEEP_SHAPES = [(1024, 1024), (2048, 2048), (4096, 4096), (8192, 8192),
                (16384, 16384), (4096, 16384), (16384, 4096)]

CONFIG_SEED = {"tiny": 1000, "gpt2": 1001, "llama": 1002, "ragged": 1003, "sweep": 1004}


# ---------------------------------------------------------------- packing

def pack(layout: Layout, mats, dtype=np.float32, fill=0.0) -> np.ndarray:
    """Place per-parameter arrays (table order) into one storage buffer."""
    buf = np.full(layout.storage_size, fill, dtype=dtype)
    for spec, prow, mat in zip(layout.specs, layout.params, mats):
        src = np.asarray(mat, dtype=dtype).reshape(-1)
        pb, pe = int(prow["offset"]), int(prow["offset"]) + spec.numel
        for q in layout.parts:
            lo, hi = max(pb, int(q["flat_begin"])), min(pe, int(q["flat_end"]))
            if lo < hi:
                s = int(q["storage_offset"]) + lo - int(q["flat_begin"])
                buf[s:s + hi - lo] = src[lo - pb:hi - pb]
    return buf


def unpack(layout: Layout, buf: np.ndarray):
    """Inverse of :func:`pack`: one (rows, cols) array per parameter."""
    out = []
    for spec, prow in zip(layout.specs, layout.params):
        pb, pe = int(prow["offset"]), int(prow["offset"]) + spec.numel
        dst = np.empty(spec.numel, dtype=buf.dtype)
        for q in layout.parts:
            lo, hi = max(pb, int(q["flat_begin"])), min(pe, int(q["flat_end"]))
            if lo < hi:
                s = int(q["storage_offset"]) + lo - int(q["flat_begin"])
                dst[lo - pb:hi - pb] = buf[s:s + hi - lo]
        out.append(dst.reshape(spec.rows, spec.cols))
    return out


def padding_mask(layout: Layout) -> np.ndarray:
    """True at storage elements no parameter covers (padding and gaps)."""
    covered = pack(layout, [np.ones(s.numel, np.int8) for s in layout.specs],
                   dtype=np.int8, fill=0)
    return covered == 0


# ---------------------------------------------------------------- values

def to_bf16_values(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even) with torch's
    conversion and return them as float32.  Input generation only."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array holding bf16 values -> uint16 bit patterns."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def rng_for(seed: int, *keys: int) -> np.random.Generator:
    return np.random.default_rng([int(seed)] + [int(k) for k in keys])


def gaussian_grads(layout: Layout, seed: int, micro_batch: int, sigmas=None, bf16=True):
    """Per-parameter N(0, sigma_i) gradients for one micro-batch."""
    mats = []
    for i, s in enumerate(layout.specs):
        g = rng_for(seed, i, micro_batch).standard_normal((s.rows, s.cols), dtype=np.float32)
        if sigmas is not None:
            g *= np.float32(sigmas[i])
        mats.append(to_bf16_values(g) if bf16 else g)
    return mats


def loguniform_sigmas(layout: Layout, seed: int, lo: float, hi: float) -> np.ndarray:
    r = rng_for(seed, 0x5161).random(len(layout.specs))
    return np.exp(np.log(lo) + r * (np.log(hi) - np.log(lo))).astype(np.float32)


def bf16_storage_grad(layout: Layout, mats, padding_value: float = 0.0) -> np.ndarray:
    """Storage-ordered uint16 bf16 bit patterns for one micro-batch."""
    return to_bf16_bits(pack(layout, mats, np.float32, fill=padding_value))


def llama_grad_into(layout: Layout, seed: int, micro_batch: int, out, params=None):
    """Fills a device bfloat16 storage tensor (identity storage) with one
    micro-batch of Llama-shaped gradients, generated on the device with
    torch's seeded generator: even-indexed parameters are low-rank plus
    noise (U V^T with U, V N(0,1) of rank 8, plus 1e-3 N(0,1)), odd-indexed
    ones N(0,1).  `params` restricts generation to those parameter indices
    (the rest of `out` is left alone).  Input generation only."""
    import torch
    dev = out.device
    for i, (spec, prow) in enumerate(zip(layout.specs, layout.params)):
        if params is not None and i not in params:
            continue
        g = torch.Generator(device=dev).manual_seed(int(seed) * 1_000_003 + i * 7919 + micro_batch)
        r, c = spec.rows, spec.cols
        if i % 2 == 0:
            U = torch.randn((r, 8), generator=g, device=dev)
            V = torch.randn((8, c), generator=g, device=dev)
            m = U @ V
            m.add_(torch.randn((r, c), generator=g, device=dev), alpha=1e-3)
        else:
            m = torch.randn((r, c), generator=g, device=dev)
        off = int(prow["offset"])
        out[off:off + r * c].copy_(m.reshape(-1).to(torch.bfloat16))
        del m


NAN_SENTINEL_BITS = np.uint32(0x7FC0DEAD)   # a quiet NaN with a payload


def storage_with_sentinels(layout: Layout, mats) -> np.ndarray:
    """float32 storage buffer, padding/gaps hold a NaN with a fixed payload."""
    buf = pack(layout, mats, np.float32, fill=0.0)
    mask = padding_mask(layout)
    buf.view(np.uint32)[mask] = NAN_SENTINEL_BITS
    return buf
