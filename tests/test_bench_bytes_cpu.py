"""The bench's algorithmic byte model against an independent count: the bytes
the decode actually has to fetch, from the library's own page layout
(kvq_pool_layout_query) -- whole pages of K/V codes with their group scales,
per-token scales, Q, the block-table entries and the lengths.  For contexts
that fill whole blocks the two must agree exactly.  CPU only."""
import importlib.util
import os

import numpy as np
import pytest

import paged_quantized_kv_kvq_gb300 as kvq
from paged_quantized_kv_kvq_gb300 import synth

_spec = importlib.util.spec_from_file_location(
    "bench", os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)


def _fetched(w, fmt, group):
    """Bytes one decode call fetches: its pages, their side scales, Q, tables."""
    lay = kvq.kvq_pool_layout_query(1, w.bs, w.Hkv, w.D, fmt, group)
    L = w.context_lens.astype(np.int64)
    blocks = (L + w.bs - 1) // w.bs
    pages = int(blocks.sum()) * w.Hkv
    side = 0
    if fmt in (kvq.KVQ_INT8_PER_TOKEN, kvq.KVQ_FP8_E4M3_PER_TOKEN):
        side = int(L.sum()) * 2 * 4                     # [block][K|V][token] fp32
    elif fmt == kvq.KVQ_INT8_PER_CHANNEL:
        side = 2 * w.Hkv * w.D * 4                      # [K|V][head][channel] fp32
    q = w.S * w.Hq * w.D * 2
    tables = int(blocks.sum()) * 4 + w.S * 4
    return pages * lay["page_bytes"] + side + q + tables


@pytest.mark.parametrize("fmt,group", [(kvq.KVQ_INT8_PER_GROUP, 128), (kvq.KVQ_INT8_PER_GROUP, 32),
                                       (kvq.KVQ_INT8_PER_TOKEN, 0), (kvq.KVQ_INT8_PER_CHANNEL, 0),
                                       (kvq.KVQ_FP8_E4M3_PER_TOKEN, 0), (kvq.KVQ_FP16, 0),
                                       (kvq.KVQ_INT4_PER_GROUP, 128), (kvq.KVQ_FP8_E5M2, 0)])
@pytest.mark.parametrize("bs", [8, 16, 32, 64])
def test_decode_bytes_equal_the_pages_fetched(fmt, group, bs):
    if bs == 8 and fmt == kvq.KVQ_INT4_PER_GROUP:
        pytest.skip("INT4 takes 16-token blocks or larger")
    w = synth.workload("gqa_64x2048", bs=bs)             # 2048 tokens: whole blocks
    assert bench.layer_bytes(w, fmt, group)["decode"] == _fetched(w, fmt, group)


def test_headline_bytes_per_call():
    # 64 x 2048, 8 kv heads, head_dim 128, INT8 per-group 128: the figure the
    # roofline divides by
    w = synth.workload("gqa_64x2048")
    assert bench.layer_bytes(w, kvq.KVQ_INT8_PER_GROUP, 128)["decode"] == 277_381_376


def test_step_sums_its_layers_formats():
    w = synth.workload("mixed_256")
    step = bench.step_bytes(w)
    int8 = bench.layer_bytes(w, kvq.KVQ_INT8_PER_GROUP, 128)
    fp16 = bench.layer_bytes(w, kvq.KVQ_FP16, 0)
    for k in ("decode", "append", "codes", "scales"):
        assert step[k] == 28 * int8[k] + 4 * fp16[k]


def test_shared_prefix_counted_once_in_unique_bytes():
    w = synth.workload("shared4k_256")
    b = bench.layer_bytes(w, kvq.KVQ_INT8_PER_GROUP, 128)
    per_token = w.Hkv * w.D * 2 + w.Hkv * 2 * 4          # codes + group scales, K and V
    assert b["decode"] - b["unique_decode"] == (w.S - 1) * w.shared_prefix_tokens * per_token


def test_append_bytes():
    # per new token: fp16 K and V in, codes and scales out, the slot
    w = synth.workload("gqa_64x2048")
    b = bench.layer_bytes(w, kvq.KVQ_INT8_PER_GROUP, 128)
    per = w.Hkv * w.D * 2 * 2 + w.Hkv * w.D * 2 + w.Hkv * 2 * 4 + 8
    assert b["append"] == w.S * per
