"""Seeded synthetic workloads for the paged quantized KV decode step.

This module only draws random inputs and lays out block tables and slot
mappings; it holds none of the method's arithmetic (no quantization, no
attention).  It serves both the CUDA path and the CPU checker in the tests and
in the benchmark, so that both sides see the very same inputs.

The five workloads follow the shapes the pages describe: 7B-class 32-layer
models with 32 Q heads and 8 (GQA) or 32 (MHA) KV heads, head_dim 128,
block_size 16/32, 2K-32K contexts and 64-256 concurrent sequences
("KV Cache优化实战：大模型推理显存占用与加速方案详解", 0539edu.com/news/5800990,
§1.2, §2.1, §3; xpshop.cn article-312 §二/§三: max_num_seqs 256, block_size 16).
Values are N(0,1) fp16 with the outlier / drift structure listed per workload.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# Cache formats (numbering of the public C enum).
FP16 = 0
INT8_PER_TOKEN = 1
INT8_PER_CHANNEL = 2
INT8_PER_GROUP = 3
FP8_E4M3_PER_TOKEN = 4
INT4_PER_GROUP = 5
FP8_E5M2 = 6


@dataclasses.dataclass
class Workload:
    """One decode step's shapes and layout (shared by every layer)."""

    name: str
    layers: int
    S: int
    Hq: int
    Hkv: int
    D: int
    bs: int
    num_blocks: int
    context_lens: np.ndarray          # int32 [S], length AFTER this step's append
    block_table: np.ndarray           # int32 [S, max_blocks]
    layer_formats: list               # [(fmt, group)] per layer
    outlier_channels: np.ndarray      # int [n, 2] (kv_head, d) pairs scaled by outlier_gain
    outlier_gain: float
    drift_sigma: float                # per-token random-walk sigma of a per-channel mean
    seed: int
    shared_prefix_tokens: int = 0

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def slots_for(self, s: int, t0: int, t1: int) -> np.ndarray:
        """Slots (physical_block * bs + offset) of tokens [t0, t1) of sequence s."""
        t = np.arange(t0, t1, dtype=np.int64)
        return self.block_table[s, t // self.bs].astype(np.int64) * self.bs + t % self.bs

    def fill_slots(self) -> np.ndarray:
        """Slots of every cached token before this step (positions 0..L-2),
        sequence-major.  Shared prefix tokens appear once (in sequence 0);
        later sequences map the same blocks and skip them."""
        out = []
        for s in range(self.S):
            t0 = self.shared_prefix_tokens if s > 0 else 0
            out.append(self.slots_for(s, min(t0, int(self.context_lens[s]) - 1),
                                      int(self.context_lens[s]) - 1))
        return np.concatenate(out) if out else np.zeros(0, np.int64)

    def fill_token_index(self) -> np.ndarray:
        """(sequence, position) of each fill slot, same order as fill_slots()."""
        rows = []
        for s in range(self.S):
            t0 = self.shared_prefix_tokens if s > 0 else 0
            t = np.arange(min(t0, int(self.context_lens[s]) - 1), int(self.context_lens[s]) - 1)
            rows.append(np.stack([np.full_like(t, s), t], 1))
        return np.concatenate(rows) if rows else np.zeros((0, 2), np.int64)

    def step_slots(self) -> np.ndarray:
        """Slot of this step's new token for each sequence (position L-1)."""
        return np.array([self.slots_for(s, int(L) - 1, int(L))[0]
                         for s, L in enumerate(self.context_lens)], np.int64)


def _table_from_lens(rng, lens, bs, num_blocks, prefix_blocks=0):
    """Random, non-overlapping physical blocks for every logical block; the
    first ``prefix_blocks`` logical blocks of every sequence map to the same
    physical blocks (prefix sharing)."""
    nblk = [(int(L) + bs - 1) // bs for L in lens]
    need = prefix_blocks + sum(n - prefix_blocks for n in nblk)
    assert need <= num_blocks, (need, num_blocks)
    perm = rng.permutation(num_blocks).astype(np.int32)
    maxb = max(nblk) if nblk else 1
    table = np.zeros((len(lens), maxb), np.int32)
    shared = perm[:prefix_blocks]
    nxt = prefix_blocks
    for s, n in enumerate(nblk):
        table[s, :prefix_blocks] = shared
        k = n - prefix_blocks
        table[s, prefix_blocks:n] = perm[nxt:nxt + k]
        nxt += k
    return table


def _outliers(rng, Hkv, D, count):
    flat = rng.choice(Hkv * D, size=count, replace=False)
    return np.stack([flat // D, flat % D], 1).astype(np.int64)


def workload(name: str, *, S: int | None = None, L: int | None = None,
             layers: int | None = None, bs: int | None = None,
             seed: int | None = None) -> Workload:
    """The named workload; S / L / layers / bs shrink or vary it for tests."""
    if name == "tiny":
        # 1 layer, 4 sequences with context 17/33/64/100, 4 Q heads over 1 KV
        # head, head_dim 64, block 16, a 64-block pool in random physical order,
        # INT8 per-group 64, N(0,1) with 2 channels x20.
        sd = 0 if seed is None else seed
        rng = np.random.default_rng(sd)
        lens = np.array([17, 33, 64, 100], np.int32)
        if S is not None:
            lens = lens[:S]
        bsz = bs or 16
        nb = 64
        table = _table_from_lens(rng, lens, bsz, nb)
        return Workload("tiny", layers or 1, len(lens), 4, 1, 64, bsz, nb, lens, table,
                        [(INT8_PER_GROUP, 64)], _outliers(rng, 1, 64, 2), 20.0, 0.0, sd)
    if name in ("gqa_64x2048", "gqa_64x2048_int4", "gqa_64x2048_e5m2"):
        # 32 layers, 64 x 2048, 32 Q / 8 KV heads, head_dim 128, block 16,
        # INT8 per-group 128 (variants: _int4 INT4 per-group 128, _e5m2
        # unscaled FP8 e5m2), pool = 90% of the needed blocks + 10% headroom,
        # N(0,1) with 1% of the Hkv*D channels x10.
        sd = 1 if seed is None else seed
        rng = np.random.default_rng(sd)
        Sx, Lx, bsz = S or 64, L or 2048, bs or 16
        lens = np.full(Sx, Lx, np.int32)
        need = Sx * ((Lx + bsz - 1) // bsz)
        nb = math.ceil(need / 0.9)
        table = _table_from_lens(rng, lens, bsz, nb)
        fmt = {"int4": (INT4_PER_GROUP, 128), "e5m2": (FP8_E5M2, 0)}.get(
            name.rsplit("_", 1)[1], (INT8_PER_GROUP, 128))
        return Workload(name, layers or 32, Sx, 32, 8, 128, bsz, nb, lens, table,
                        [fmt] * (layers or 32),
                        _outliers(rng, 8, 128, max(1, round(0.01 * 8 * 128))), 10.0, 0.0, sd)
    if name.startswith("mha_100"):
        # 32 layers, 100 sequences with lengths uniform in [256, 2048], MHA 32/32,
        # head_dim 128, block 16.  The format is chosen by the suffix:
        # mha_100_fp16, mha_100_fp8, mha_100_int8ch, mha_100_int8g64.
        sd = 2 if seed is None else seed
        rng = np.random.default_rng(sd)
        Sx, bsz = S or 100, bs or 16
        hi = L or 2048
        lens = rng.integers(min(256, hi), hi + 1, size=Sx).astype(np.int32)
        fmt = {"fp16": (FP16, 0), "fp8": (FP8_E4M3_PER_TOKEN, 0),
               "int8ch": (INT8_PER_CHANNEL, 0), "int8g64": (INT8_PER_GROUP, 64)}[
                   name.split("_", 2)[2] if name.count("_") >= 2 else "int8g64"]
        need = int(sum((int(x) + bsz - 1) // bsz for x in lens))
        nb = math.ceil(need / 0.9)
        table = _table_from_lens(rng, lens, bsz, nb)
        return Workload(name, layers or 32, Sx, 32, 32, 128, bsz, nb, lens, table,
                        [fmt] * (layers or 32), np.zeros((0, 2), np.int64), 1.0, 0.0, sd)
    if name == "long_8x32k":
        # 32 layers, 8 x 32768, 32 Q / 8 KV heads, head_dim 128, block 16 or 32,
        # INT8 per-group 128; K/V = N(0,1) + a per-channel random-walk mean
        # (sigma 0.01 per token).
        sd = 3 if seed is None else seed
        rng = np.random.default_rng(sd)
        Sx, Lx, bsz = S or 8, L or 32768, bs or 16
        lens = np.full(Sx, Lx, np.int32)
        need = Sx * ((Lx + bsz - 1) // bsz)
        table = _table_from_lens(rng, lens, bsz, need)
        return Workload("long_8x32k", layers or 32, Sx, 32, 8, 128, bsz, need, lens, table,
                        [(INT8_PER_GROUP, 128)] * (layers or 32),
                        np.zeros((0, 2), np.int64), 1.0, 0.01, sd)
    if name == "mixed_256":
        # 32 layers, 256 sequences; each is a 512-token shared system prefix plus
        # a log-normal suffix (median 1024, sigma 1.0) clipped to [64, 8192];
        # the prefix maps to the same 32 physical blocks in every table; layers
        # 0-27 INT8 per-group 128, layers 28-31 FP16; 32 Q / 8 KV, head_dim 128,
        # block 16.
        sd = 4 if seed is None else seed
        rng = np.random.default_rng(sd)
        Sx, bsz = S or 256, bs or 16
        nl = layers or 32
        prefix = 512
        suffix = np.clip(np.round(rng.lognormal(math.log(1024), 1.0, size=Sx)), 64, L or 8192)
        lens = (prefix + suffix).astype(np.int32)
        pblk = prefix // bsz
        need = pblk + int(sum((int(x) + bsz - 1) // bsz - pblk for x in lens))
        nb = math.ceil(need / 0.9)
        table = _table_from_lens(rng, lens, bsz, nb, prefix_blocks=pblk)
        # The last 4 layers stay FP16; a shortened test stack keeps its last
        # half (at least one layer, when it has two or more) in FP16.
        n16 = 4 if nl >= 8 else (nl // 2 if nl > 1 else 0)
        fmts = [(INT8_PER_GROUP, 128) if i < nl - n16 else (FP16, 0) for i in range(nl)]
        return Workload("mixed_256", nl, Sx, 32, 8, 128, bsz, nb, lens, table, fmts,
                        np.zeros((0, 2), np.int64), 1.0, 0.0, sd, shared_prefix_tokens=prefix)
    if name == "shared4k_256":
        # A prefix-heavy batch: 256 sequences that share a 4096-token prefix
        # (256 physical blocks) and each add a suffix uniform in [64, 512];
        # 32 Q / 8 KV heads, head_dim 128, block 16, INT8 per-group 128.
        sd = 5 if seed is None else seed
        rng = np.random.default_rng(sd)
        Sx, bsz = S or 256, bs or 16
        nl = layers or 32
        prefix = 4096
        suffix = rng.integers(64, (L or 512) + 1, size=Sx)
        lens = (prefix + suffix).astype(np.int32)
        pblk = prefix // bsz
        need = pblk + int(sum((int(x) + bsz - 1) // bsz - pblk for x in lens))
        nb = math.ceil(need / 0.9)
        table = _table_from_lens(rng, lens, bsz, nb, prefix_blocks=pblk)
        return Workload("shared4k_256", nl, Sx, 32, 8, 128, bsz, nb, lens, table,
                        [(INT8_PER_GROUP, 128)] * nl, np.zeros((0, 2), np.int64), 1.0, 0.0, sd,
                        shared_prefix_tokens=prefix)
    raise KeyError(name)


def layer_rng(w: Workload, layer: int, stream: str) -> np.random.Generator:
    """Independent generator per (workload seed, layer, stream name)."""
    tag = sum((i + 1) * ord(c) for i, c in enumerate(stream))
    return np.random.default_rng([w.seed, layer, tag])


def kv_tokens(w: Workload, layer: int, seq_pos: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """fp16 K and V [n, Hkv, D] for the (sequence, position) rows of seq_pos.

    Each (layer, sequence) has its own stream, so any subset of tokens can be
    regenerated on its own: the rows of one sequence are drawn for positions
    0..max needed and then indexed, which keeps the drift random walk and the
    values identical however the tokens are grouped."""
    n = seq_pos.shape[0]
    k = np.empty((n, w.Hkv, w.D), np.float16)
    v = np.empty((n, w.Hkv, w.D), np.float16)
    if n == 0:
        return k, v

    def one(s):  # sequences fill disjoint rows; numpy draws outside the GIL
        rows = np.nonzero(seq_pos[:, 0] == s)[0]
        pos = seq_pos[rows, 1]
        upto = int(pos.max()) + 1
        kk, vv = _seq_kv(w, layer, int(s), upto)
        k[rows] = kk[pos]
        v[rows] = vv[pos]

    seqs = np.unique(seq_pos[:, 0])
    if len(seqs) > 1 and n > 4096:
        import concurrent.futures
        import os

        with concurrent.futures.ThreadPoolExecutor(min(len(seqs), os.cpu_count() or 1)) as ex:
            list(ex.map(one, seqs))
    else:
        for s in seqs:
            one(s)
    return k, v


def _seq_kv(w: Workload, layer: int, s: int, upto: int):
    # One generator per (layer, sequence, stream): row t of every stream is the
    # same whatever ``upto`` is, so token t's values never depend on how many
    # tokens were asked for.  Shared prefix tokens come from sequence 0.
    def gen(tag):
        return np.random.default_rng([w.seed, layer, tag, s])

    shape = (upto, w.Hkv, w.D)
    k = gen(7919).standard_normal(shape, dtype=np.float32)
    v = gen(7927).standard_normal(shape, dtype=np.float32)
    if w.drift_sigma > 0:
        k += np.cumsum(w.drift_sigma * gen(7933).standard_normal(shape, dtype=np.float32), axis=0)
        v += np.cumsum(w.drift_sigma * gen(7937).standard_normal(shape, dtype=np.float32), axis=0)
    for h, d in w.outlier_channels:
        k[:, h, d] *= w.outlier_gain
        v[:, h, d] *= w.outlier_gain
    if s > 0 and w.shared_prefix_tokens > 0:
        p = min(w.shared_prefix_tokens, upto)
        k0, v0 = _seq_kv(w, layer, 0, p)
        k[:p] = k0
        v[:p] = v0
    return k.astype(np.float16), v.astype(np.float16)


def queries(w: Workload, layer: int) -> np.ndarray:
    """fp16 Q [S, Hq, D] of this step for one layer."""
    rng = np.random.default_rng([w.seed, layer, 104729])
    q = rng.standard_normal((w.S, w.Hq, w.D), dtype=np.float32)
    for h, d in w.outlier_channels:
        q[:, h * w.G:(h + 1) * w.G, d] *= w.outlier_gain
    return q.astype(np.float16)


def step_kv(w: Workload, layer: int) -> tuple[np.ndarray, np.ndarray]:
    """fp16 K/V [S, Hkv, D] of this step's new token (position L-1) per sequence."""
    idx = np.stack([np.arange(w.S), w.context_lens.astype(np.int64) - 1], 1)
    return kv_tokens(w, layer, idx)


# ---------------------------------------------------------------- on-device draws
# The benchmark fills 32 layers of multi-GB pools; drawing those values on the
# host would take minutes, so it draws them with torch's device generator
# (same distributions and structure as above, different random streams).
def _device_gen(device, *key):
    import torch

    g = torch.Generator(device=device)
    h = 0
    for k in key:
        h = (h * 1000003 + int(k)) & 0x7FFFFFFFFFFFFFFF
    g.manual_seed(h)
    return g


def device_kv(w: Workload, layer: int, seq: int, t0: int, t1: int, device):
    """fp16 K, V [t1-t0, Hkv, D] for positions t0..t1-1 of one sequence,
    drawn on the device (positions are independent unless the workload has
    drift, in which case t0 must be 0)."""
    import torch

    n = max(t1 - t0, 0)
    k = torch.randn((n, w.Hkv, w.D), generator=_device_gen(device, w.seed, layer, seq, t0, 1),
                    device=device, dtype=torch.float32)
    v = torch.randn((n, w.Hkv, w.D), generator=_device_gen(device, w.seed, layer, seq, t0, 2),
                    device=device, dtype=torch.float32)
    if w.drift_sigma > 0 and n:
        assert t0 == 0
        gk = _device_gen(device, w.seed, layer, seq, t0, 3)
        gv = _device_gen(device, w.seed, layer, seq, t0, 4)
        k += torch.cumsum(w.drift_sigma * torch.randn(k.shape, generator=gk, device=device), 0)
        v += torch.cumsum(w.drift_sigma * torch.randn(v.shape, generator=gv, device=device), 0)
    for h, d in w.outlier_channels:
        k[:, h, d] *= w.outlier_gain
        v[:, h, d] *= w.outlier_gain
    return k.half(), v.half()


def device_queries(w: Workload, layer: int, device):
    import torch

    q = torch.randn((w.S, w.Hq, w.D), generator=_device_gen(device, w.seed, layer, 104729),
                    device=device, dtype=torch.float32)
    for h, d in w.outlier_channels:
        q[:, h * w.G:(h + 1) * w.G, d] *= w.outlier_gain
    return q.half()
