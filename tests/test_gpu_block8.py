"""GPU parity of pools with 8-token blocks ("KV Cache优化实战", §3.2: block
size 8 for short contexts at high concurrency).  A page then holds half of a
16-token tile and the decode pairs consecutive pages of a sequence into one
tile, so these cases cover: codes and scales of every slot bit-exact through
the read-back (the 8-token V order is its own), decode outputs within 1e-3
of the float64 oracle for every format but INT4, ragged tails (a short last
page with no partner), units cut at odd pages by fixed splits, the step form,
the full 64 x 2048 batch, and the refusals (INT4, prefill, cascade)."""
import numpy as np
import pytest
import torch

import oracle
import paged_quantized_kv_kvq_gb300 as kvq
from paged_quantized_kv_kvq_gb300 import synth
from kvq_testutil import TOL, gpu_pool, layer_tokens, oracle_layer, oracle_slots, run_gpu_decode

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

FORMATS = [(kvq.KVQ_INT8_PER_GROUP, 128), (kvq.KVQ_INT8_PER_GROUP, 64), (kvq.KVQ_INT8_PER_GROUP, 32),
           (kvq.KVQ_INT8_PER_GROUP, 16), (kvq.KVQ_INT8_PER_TOKEN, 0), (kvq.KVQ_INT8_PER_CHANNEL, 0),
           (kvq.KVQ_FP8_E4M3_PER_TOKEN, 0), (kvq.KVQ_FP16, 0), (kvq.KVQ_FP8_E5M2, 0)]


def _t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def _codes_match(pool, ref, slots, ref_slots):
    codes, scales = pool.read_slots(_t(slots))
    torch.cuda.synchronize()
    c = codes.cpu().numpy()
    if pool.dtype == kvq.KVQ_FP16:
        np.testing.assert_array_equal(c.astype(np.float32), ref.codes[ref_slots])
    else:
        np.testing.assert_array_equal(c.view(np.uint8), ref.codes[ref_slots].view(np.uint8))
    if scales is not None:
        np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32),
                                      ref.scales[ref_slots].view(np.uint32))


def _case(name, fmt, group, **kw):
    w = synth.workload(name, layers=1, bs=8, **kw)
    w.layer_formats = [(fmt, group)]
    k, v, slots = layer_tokens(w, 0)
    calib = (k, v) if fmt == kvq.KVQ_INT8_PER_CHANNEL else None
    pool = gpu_pool(w, fmt, group, DEV, k, v, slots, calib=calib)
    ref, table, remap = oracle_layer(w, fmt, group, k, v, slots, list(range(w.S)), calib=calib)
    uniq = np.unique(slots)
    _codes_match(pool, ref, uniq, oracle_slots(remap, uniq, w.bs))
    return w, pool, ref, table


@pytest.mark.parametrize("fmt,group", FORMATS)
@pytest.mark.parametrize("D", [64, 128])
def test_block8_append_bitexact(fmt, group, D):
    if group > D:
        pytest.skip("group larger than head_dim")
    rng = np.random.default_rng(100 + D + fmt + group)
    nb, bs, hkv, T = 20, 8, 3, 90
    x = rng.standard_normal((2, T, hkv, D)).astype(np.float32)
    x[:, :, :, rng.integers(0, D, 3)] *= 20.0
    x[:, 4] = 0.0
    k, v = x.astype(np.float16)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[[2, 30]] = -1
    pool = kvq.KVPool(nb, bs, hkv, D, fmt, group, device=DEV, fill_byte=0x5A)
    ref = oracle.OracleCache(fmt, nb, bs, hkv, D, group, sentinel_code=0x5A)
    if fmt == kvq.KVQ_INT8_PER_CHANNEL:
        kvq.kvq_calibrate_channel_scales(pool.handle, _t(k[:60]), _t(v[:60]))
        ref.calibrate(k[:60], v[:60])
    pool.append(_t(k), _t(v), _t(slots))
    ref.append(k, v, slots)
    assert pool.error() == kvq.KVQ_OK
    written = np.sort(slots[slots >= 0])
    _codes_match(pool, ref, written, written)
    # untouched slots keep the fill: no write strayed into a neighbour's bytes
    untouched = np.setdiff1d(np.arange(nb * bs), written)
    codes, _ = pool.read_slots(_t(untouched))
    sentinel = 0x5A ^ 0x80 if fmt in (kvq.KVQ_INT8_PER_TOKEN, kvq.KVQ_INT8_PER_CHANNEL,
                                      kvq.KVQ_INT8_PER_GROUP) else 0x5A
    assert np.all(codes.cpu().numpy().view(np.uint8) == sentinel)
    pool.close()


@pytest.mark.parametrize("fmt,group", FORMATS)
def test_block8_decode_parity(fmt, group):
    # 301 tokens: 37 full pages and a 5-token last page without a partner
    w, pool, ref, table = _case("gqa_64x2048", fmt, group, S=3, L=301)
    q = synth.queries(w, 0)
    got = run_gpu_decode(pool, w, q, DEV)
    np.testing.assert_allclose(got, ref.decode(q, table, w.context_lens), rtol=0, atol=TOL)
    assert pool.error() == kvq.KVQ_OK
    pool.close()


@pytest.mark.parametrize("name,kw", [("mha_100_int8g64", dict(S=6, L=300)),
                                     ("mha_100_fp16", dict(S=6, L=300)),
                                     ("long_8x32k", dict(S=1, L=3001))])
def test_block8_workloads(name, kw):
    w0 = synth.workload(name, layers=1)
    fmt, group = w0.layer_formats[0]
    w, pool, ref, table = _case(name, fmt, group, **kw)
    q = synth.queries(w, 0)
    got = run_gpu_decode(pool, w, q, DEV)
    np.testing.assert_allclose(got, ref.decode(q, table, w.context_lens), rtol=0, atol=TOL,
                               err_msg=name)
    assert pool.error() == kvq.KVQ_OK
    pool.close()


def test_block8_split_invariance_and_short_sequences():
    # contexts of 1..9 tokens and a long one; fixed splits of 1, 2, 3, 5, 7
    # pages start units' pieces at odd pages, so tiles pair pages across the
    # piece boundary differently
    w = synth.workload("gqa_64x2048", S=6, L=200, layers=1, bs=8)
    w.context_lens = np.array([1, 7, 8, 9, 200, 17], np.int32)
    fmt, group = kvq.KVQ_INT8_PER_GROUP, 128
    w.layer_formats = [(fmt, group)]
    k, v, slots = layer_tokens(w, 0)
    pool = gpu_pool(w, fmt, group, DEV, k, v, slots)
    ref, table, _ = oracle_layer(w, fmt, group, k, v, slots, list(range(w.S)))
    q = synth.queries(w, 0)
    got = run_gpu_decode(pool, w, q, DEV)
    np.testing.assert_allclose(got, ref.decode(q, table, w.context_lens), rtol=0, atol=TOL)
    for sb in (1, 2, 3, 5, 7):
        np.testing.assert_allclose(run_gpu_decode(pool, w, q, DEV, split_blocks=sb), got,
                                   rtol=2e-5, atol=2e-5, err_msg="split %d" % sb)
    assert pool.error() == kvq.KVQ_OK
    pool.close()


@pytest.mark.parametrize("fmt,group", [(kvq.KVQ_INT8_PER_GROUP, 128), (kvq.KVQ_FP16, 0),
                                       (kvq.KVQ_FP8_E4M3_PER_TOKEN, 0)])
def test_block8_decode_step(fmt, group):
    w = synth.workload("gqa_64x2048", S=4, L=77, layers=1, bs=8)
    w.layer_formats = [(fmt, group)]
    k, v, slots = layer_tokens(w, 0)
    S = w.S
    pool = gpu_pool(w, fmt, group, DEV, k[:-S], v[:-S], slots[:-S])
    ref, table, remap = oracle_layer(w, fmt, group, k, v, slots, list(range(S)))
    q = synth.queries(w, 0)
    out = pool.decode_step(_t(k[-S:]), _t(v[-S:]), _t(q), _t(w.block_table), _t(w.context_lens),
                           int(w.context_lens.max()))
    torch.cuda.synchronize()
    assert pool.error() == kvq.KVQ_OK
    _codes_match(pool, ref, slots[-S:], oracle_slots(remap, slots[-S:], w.bs))
    np.testing.assert_allclose(out.cpu().numpy(), ref.decode(q, table, w.context_lens), rtol=0,
                               atol=TOL)
    pool.close()


def test_block8_refusals():
    with pytest.raises(kvq.KVQError) as ei:
        kvq.KVPool(16, 8, 2, 128, kvq.KVQ_INT4_PER_GROUP, 128, device=DEV)
    assert ei.value.status == kvq.KVQ_ERR_UNSUPPORTED
    w = synth.workload("gqa_64x2048", S=2, L=40, layers=1, bs=8)
    pool = kvq.KVPool(w.num_blocks, 8, w.Hkv, w.D, kvq.KVQ_INT8_PER_GROUP, 128, device=DEV)
    q = _t(synth.queries(w, 0))
    table, lens = _t(w.block_table), _t(w.context_lens)
    out = torch.empty((w.S, w.Hq, w.D), dtype=torch.float32, device=DEV)
    with pytest.raises(kvq.KVQError) as ei:
        qs = _t(np.array([0, 1, 2], np.int32))
        kvq.kvq_prefill(pool.handle, q, qs, 1, table, lens, 40, w.D ** -0.5, out)
    assert ei.value.status == kvq.KVQ_ERR_UNSUPPORTED
    ws = torch.empty(kvq.kvq_cascade_workspace_bytes(pool.handle, w.S, w.Hq, 40), dtype=torch.uint8,
                     device=DEV)
    with pytest.raises(kvq.KVQError) as ei:
        kvq.kvq_cascade_decode(pool.handle, q, table, lens, 40, 2, w.D ** -0.5, out, ws)
    assert ei.value.status == kvq.KVQ_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert pool.error() == kvq.KVQ_OK
    pool.close()
