"""GPU parity of the shared-prefix cascade decode: the blocks every sequence
shares are attended once for all sequences (prefix kernel) and folded into the
paged decode of the remaining blocks.  Outputs within 1e-3 of the float64
oracle (which attends every sequence's blocks through its own table row) and
equal to kvq_paged_decode up to fp32 rounding order."""
import numpy as np
import pytest
import torch

import paged_quantized_kv_kvq_gb300 as kvq
from paged_quantized_kv_kvq_gb300 import synth
from kvq_testutil import TOL, gpu_pool, layer_tokens, oracle_layer

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
# the cascade sums the prefix and the rest separately: fp32 reassociation only
REORDER = 3e-5

FORMATS = [(kvq.KVQ_INT8_PER_GROUP, 128), (kvq.KVQ_INT8_PER_GROUP, 32), (kvq.KVQ_INT8_PER_TOKEN, 0),
           (kvq.KVQ_INT8_PER_CHANNEL, 0), (kvq.KVQ_FP8_E4M3_PER_TOKEN, 0), (kvq.KVQ_FP16, 0),
           (kvq.KVQ_INT4_PER_GROUP, 128), (kvq.KVQ_INT4_PER_GROUP, 32), (kvq.KVQ_FP8_E5M2, 0)]


def _t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def _case(fmt, group, S=6, L=200):
    w = synth.workload("mixed_256", S=S, L=L, layers=1)
    w.layer_formats = [(fmt, group)]
    k, v, slots = layer_tokens(w, 0)
    calib = (k, v) if fmt == kvq.KVQ_INT8_PER_CHANNEL else None
    pool = gpu_pool(w, fmt, group, DEV, k, v, slots, calib=calib)
    ref, table, _ = oracle_layer(w, fmt, group, k, v, slots, list(range(w.S)), calib=calib)
    return w, pool, ref, table, (k, v, slots, calib)


def _run(pool, w, q, lens, P, max_ctx=None):
    mc = int(max(lens.max(), 1)) if max_ctx is None else max_ctx
    out = pool.cascade_decode(_t(q), _t(w.block_table), _t(lens), mc, P)
    plain = pool.decode(_t(q), _t(w.block_table), _t(lens), mc)
    torch.cuda.synchronize()
    return out.cpu().numpy(), plain.cpu().numpy()


@pytest.mark.parametrize("fmt,group", FORMATS)
def test_cascade_parity(fmt, group):
    w, pool, ref, table, _ = _case(fmt, group)
    P = w.shared_prefix_tokens // w.bs
    q = synth.queries(w, 0)
    got, plain = _run(pool, w, q, w.context_lens, P)
    assert pool.error() == kvq.KVQ_OK
    np.testing.assert_allclose(got, ref.decode(q, table, w.context_lens), rtol=0, atol=TOL)
    np.testing.assert_allclose(got, plain, rtol=REORDER, atol=REORDER)
    pool.close()


@pytest.mark.parametrize("fmt,group", [(kvq.KVQ_INT8_PER_GROUP, 128), (kvq.KVQ_FP16, 0)])
def test_cascade_short_sequences_and_partial_prefix(fmt, group):
    """Sequences that end inside the prefix (or are empty), a prefix shorter
    than the shared one, and prefix_blocks = 0 (plain decode, same bits)."""
    w, pool, ref, table, _ = _case(fmt, group, S=7)
    P = w.shared_prefix_tokens // w.bs
    q = synth.queries(w, 0)
    lens = w.context_lens.copy()
    lens[1], lens[2], lens[3], lens[4], lens[5] = 100, P * w.bs, P * w.bs + 1, 16, 0
    got, plain = _run(pool, w, q, lens, P)
    assert pool.error() == kvq.KVQ_OK
    np.testing.assert_allclose(got, ref.decode(q, table, lens), rtol=0, atol=TOL)
    np.testing.assert_allclose(got, plain, rtol=REORDER, atol=REORDER)
    assert not got[5].any()
    for p_part in (1, 5, P - 1):
        got, _ = _run(pool, w, q, w.context_lens, p_part)
        np.testing.assert_allclose(got, ref.decode(q, table, w.context_lens), rtol=0, atol=TOL)
    got, plain = _run(pool, w, q, w.context_lens, 0)
    np.testing.assert_array_equal(got, plain)
    assert pool.error() == kvq.KVQ_OK
    pool.close()


def test_cascade_many_row_tiles():
    """64 sequences x 4 heads per kv head: 16 row tiles per kv head, a prefix
    of 32 blocks split over the 4 warps of each tile."""
    w, pool, ref, table, _ = _case(kvq.KVQ_INT8_PER_GROUP, 128, S=64, L=96)
    P = w.shared_prefix_tokens // w.bs
    q = synth.queries(w, 0)
    got, plain = _run(pool, w, q, w.context_lens, P)
    sel = [0, 13, 31, 47, 63]
    np.testing.assert_allclose(got[sel], ref.decode(q, table, w.context_lens)[sel], rtol=0, atol=TOL)
    np.testing.assert_allclose(got, plain, rtol=REORDER, atol=REORDER)
    pool.close()


def test_cascade_step_equals_append_then_cascade():
    w = synth.workload("mixed_256", S=5, L=150, layers=1)
    fmt, group = w.layer_formats[0]
    k, v, slots = layer_tokens(w, 0)
    S = w.S
    P = w.shared_prefix_tokens // w.bs
    q = _t(synth.queries(w, 0))
    table, lens = _t(w.block_table), _t(w.context_lens)
    mc = int(w.context_lens.max())
    pool_a = gpu_pool(w, fmt, group, DEV, k[:-S], v[:-S], slots[:-S])
    pool_b = gpu_pool(w, fmt, group, DEV, k, v, slots)
    ws_n = kvq.kvq_cascade_workspace_bytes(pool_a.handle, S, w.Hq, mc)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=DEV)
    out_a = torch.empty((S, w.Hq, w.D), dtype=torch.float32, device=DEV)
    kvq.kvq_cascade_decode_step(pool_a.handle, _t(k[-S:]), _t(v[-S:]), q, table, lens, mc, P,
                                w.D ** -0.5, out_a, ws)
    out_b = pool_b.cascade_decode(q, table, lens, mc, P)
    torch.cuda.synchronize()
    assert pool_a.error() == kvq.KVQ_OK
    np.testing.assert_array_equal(out_a.cpu().numpy(), out_b.cpu().numpy())
    ref, rtable, _ = oracle_layer(w, fmt, group, k, v, slots, list(range(S)))
    np.testing.assert_allclose(out_a.cpu().numpy(), ref.decode(synth.queries(w, 0), rtable,
                                                               w.context_lens), rtol=0, atol=TOL)
    pool_a.close()
    pool_b.close()


def test_cascade_host_validation():
    w = synth.workload("mixed_256", S=3, L=100, layers=1)
    pool = kvq.KVPool(w.num_blocks, w.bs, w.Hkv, w.D, kvq.KVQ_INT8_PER_GROUP, 128, device=DEV)
    q = torch.zeros((3, 32, 128), dtype=torch.float16, device=DEV)
    table, lens = _t(w.block_table), _t(w.context_lens)
    out = torch.empty((3, 32, 128), dtype=torch.float32, device=DEV)
    mc = int(w.context_lens.max())
    need = kvq.kvq_cascade_workspace_bytes(pool.handle, 3, 32, mc)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_cascade_decode(pool.handle, q, table, lens, mc, w.max_blocks + 1, 0.1, out, ws)
    assert e.value.status == kvq.KVQ_ERR_INVALID_ARG
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_cascade_decode(pool.handle, q, table, lens, mc, 4, 0.1, out, ws[:256])
    assert e.value.status == kvq.KVQ_ERR_WORKSPACE
    pool.close()
