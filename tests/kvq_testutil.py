"""Shared helpers for the GPU parity tests: build one layer of a workload on
both sides (the CUDA pool through the C ABI, the CPU oracle's slot store) from
the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_quantized_kv_kvq_gb300 as kvq
from paged_quantized_kv_kvq_gb300 import synth

TOL = 1e-3  # max abs error of attention outputs vs the float64 oracle
# Prefill outputs whose softmax weights reach P.V with fp32-level precision
# (an fp16 high plus an fp16 low part) stay well inside this on the prefill
# precision case; fp16 weights alone miss it by several times (the CPU check
# of the case shows both).
PREC_TOL = 2e-4


def layer_tokens(w: synth.Workload, layer: int, seqs=None):
    """fp16 K/V and slots of every cached token plus this step's token, for the
    given sequences (all by default).  Shared prefix tokens are included once."""
    idx = w.fill_token_index()
    slots = w.fill_slots()
    if seqs is not None:
        keep = np.isin(idx[:, 0], seqs)
        if w.shared_prefix_tokens and 0 not in seqs:
            # the shared prefix is stored once, under sequence 0
            keep |= (idx[:, 0] == 0) & (idx[:, 1] < w.shared_prefix_tokens)
        idx, slots = idx[keep], slots[keep]
    k, v = synth.kv_tokens(w, layer, idx)
    ks, vs = synth.step_kv(w, layer)
    st = w.step_slots()
    sel = np.arange(w.S) if seqs is None else np.asarray(seqs)
    return (np.concatenate([k, ks[sel]]), np.concatenate([v, vs[sel]]),
            np.concatenate([slots, st[sel]]))


def gpu_pool(w, fmt, group, dev, k, v, slots, chunk=1 << 16, calib=None):
    pool = kvq.KVPool(w.num_blocks, w.bs, w.Hkv, w.D, fmt, group, device=dev)
    if fmt == kvq.KVQ_INT8_PER_CHANNEL:
        ck, cv = calib
        kvq.kvq_calibrate_channel_scales(pool.handle, torch.from_numpy(ck).to(dev),
                                         torch.from_numpy(cv).to(dev))
    for a in range(0, len(slots), chunk):
        b = min(len(slots), a + chunk)
        pool.append(torch.from_numpy(k[a:b]).to(dev), torch.from_numpy(v[a:b]).to(dev),
                    torch.from_numpy(slots[a:b]).to(dev))
    return pool


def compact(w, seqs):
    """Block table of the given sequences relabelled onto 0..n-1 (the oracle's
    result does not depend on where blocks live), and the slot map old->new."""
    table = w.block_table[seqs]
    used = np.unique(np.concatenate([table[i, :(int(w.context_lens[s]) + w.bs - 1) // w.bs]
                                     for i, s in enumerate(seqs)]))
    remap = np.full(w.num_blocks, -1, np.int64)
    remap[used] = np.arange(len(used))
    new_table = np.where(table >= 0, remap[np.clip(table, 0, None)], 0).astype(np.int32)
    return new_table, remap, len(used)


def oracle_layer(w, fmt, group, k, v, slots, seqs, calib=None):
    """Oracle cache holding only the blocks of `seqs`, relabelled compactly."""
    table, remap, nb = compact(w, seqs)
    blk = slots // w.bs
    keep = remap[blk] >= 0
    new_slots = remap[blk[keep]] * w.bs + slots[keep] % w.bs
    c = oracle.OracleCache(fmt, max(nb, 1), w.bs, w.Hkv, w.D, group)
    if fmt == oracle.INT8_PER_CHANNEL:
        c.calibrate(*calib)
    if keep.all():
        c.append(k, v, new_slots)
    else:
        c.append(k[keep], v[keep], new_slots)
    return c, table, remap


def oracle_slots(remap, slots, bs):
    """Oracle-side slot of each (kept) device slot."""
    return remap[slots // bs] * bs + slots % bs


def run_gpu_decode(pool, w, q, dev, split_blocks=0, lens=None, table=None, max_ctx=None):
    lens = w.context_lens if lens is None else lens
    table = w.block_table if table is None else table
    out = pool.decode(torch.from_numpy(q).to(dev), torch.from_numpy(table).to(dev),
                      torch.from_numpy(np.asarray(lens, np.int32)).to(dev),
                      int(max(lens.max(), 1)) if max_ctx is None else max_ctx,
                      split_blocks=split_blocks)
    torch.cuda.synchronize()
    return out.cpu().numpy()
