"""GPU parity of prefill / chunked prefill over the paged quantized cache: each
sequence's new query tokens attend causally to its cache (the chunk's own K/V
already appended).  The float64 oracle is the decode definition applied per
query token with the causal length: query token i of sequence s is a decode
over positions 0 .. L_s - n_s + i through the same block-table row."""
import numpy as np
import pytest
import torch

import paged_quantized_kv_kvq_gb300 as kvq
from paged_quantized_kv_kvq_gb300 import synth
from kvq_testutil import PREC_TOL, TOL, gpu_pool, layer_tokens, oracle_layer

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

FORMATS = [(kvq.KVQ_INT8_PER_GROUP, 128), (kvq.KVQ_INT8_PER_GROUP, 32), (kvq.KVQ_INT8_PER_TOKEN, 0),
           (kvq.KVQ_INT8_PER_CHANNEL, 0), (kvq.KVQ_FP8_E4M3_PER_TOKEN, 0), (kvq.KVQ_FP16, 0),
           (kvq.KVQ_INT4_PER_GROUP, 128), (kvq.KVQ_INT4_PER_GROUP, 32), (kvq.KVQ_FP8_E5M2, 0)]


def _t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def _queries(Tq, Hq, D, seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((Tq, Hq, D)).astype(np.float16)


def _expand(table, lens, nq):
    """Per query token: its sequence's table row and causal length."""
    rows, L = [], []
    for s, (Ls, n) in enumerate(zip(lens, nq)):
        for i in range(n):
            rows.append(table[s])
            L.append(max(0, int(Ls) - int(n) + i + 1))
    return np.array(rows, np.int32), np.array(L, np.int32)


def _prefill(api, pool, q, qs, mq, table, lens, mc, sm, out):
    """One prefill call: "one_pass" = kvq_prefill, "two_pass" = kvq_prefill_ex
    with its workspace (the staged fp16 key steps)."""
    if api == "one_pass":
        kvq.kvq_prefill(pool.handle, q, qs, mq, table, lens, mc, sm, out)
        return
    S = qs.numel() - 1
    nb = kvq.kvq_prefill_workspace_bytes(pool.handle, S, mc)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=DEV) if nb else None
    kvq.kvq_prefill_ex(pool.handle, q, qs, mq, table, lens, mc, sm, out, ws)


APIS = ["one_pass", "two_pass"]


def _case(fmt, group, name="gqa_64x2048", S=3, L=300, nq=(50, 17, 64), lens=None, seed=0,
          heads=None, api="one_pass", **kw):
    w = synth.workload(name, S=S, L=L, layers=1, **kw)
    w.layer_formats = [(fmt, group)]
    if heads is not None:
        w.Hq, w.Hkv = heads
        w.outlier_channels = w.outlier_channels[w.outlier_channels[:, 0] < w.Hkv]
    k, v, slots = layer_tokens(w, 0)
    calib = (k, v) if fmt == kvq.KVQ_INT8_PER_CHANNEL else None
    pool = gpu_pool(w, fmt, group, DEV, k, v, slots, calib=calib)
    ref, table, _ = oracle_layer(w, fmt, group, k, v, slots, list(range(w.S)), calib=calib)
    lens = w.context_lens.copy() if lens is None else np.asarray(lens, np.int32)
    nq = np.asarray(nq, np.int32)
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    q = _queries(int(qs[-1]), w.Hq, w.D, seed)
    out = torch.empty((int(qs[-1]), w.Hq, w.D), dtype=torch.float32, device=DEV)
    _prefill(api, pool, _t(q), _t(qs), int(nq.max()), _t(w.block_table), _t(lens),
             int(max(lens.max(), 1)), w.D ** -0.5, out)
    torch.cuda.synchronize()
    t_exp, l_exp = _expand(table, lens, nq)
    exp = ref.decode(q, t_exp, l_exp)
    return pool, out.cpu().numpy(), exp, l_exp


@pytest.mark.parametrize("api", APIS)
@pytest.mark.parametrize("fmt,group", FORMATS)
def test_prefill_parity(fmt, group, api):
    pool, got, exp, _ = _case(fmt, group, api=api)
    assert pool.error() == kvq.KVQ_OK
    np.testing.assert_allclose(got, exp, rtol=0, atol=TOL)
    pool.close()


@pytest.mark.parametrize("api", APIS)
@pytest.mark.parametrize("fmt,group", [(kvq.KVQ_INT8_PER_GROUP, 128), (kvq.KVQ_FP16, 0),
                                       (kvq.KVQ_INT8_PER_CHANNEL, 0), (kvq.KVQ_INT4_PER_GROUP, 32)])
def test_prefill_weights_keep_fp32_precision(fmt, group, api):
    """The softmax weights enter P.V as an fp16 high part plus an fp16 low
    part (the two-pass kernel stores the low part negated and negates the
    operand back in the MMA).  Both parts must arrive with the right sign:
    with the high part alone, or the low part subtracted, the weights carry
    an fp16 rounding error and the outputs miss the float64 oracle by
    several times PREC_TOL (shown on the CPU for this very case)."""
    pool, got, exp, _ = _case(fmt, group, S=2, L=600, nq=(600, 200), api=api)
    err = float(np.abs(got - exp).max())
    print("max abs error vs oracle: %.3g" % err)
    assert err <= PREC_TOL
    pool.close()


@pytest.mark.parametrize("api", APIS)
def test_prefill_whole_prompt_and_long_context(api):
    """A fresh prompt (chunk = whole context) and a chunk deep into a long
    context, MHA with head_dim 128, and GQA 4:1 with D 64 (tiny)."""
    pool, got, exp, _ = _case(kvq.KVQ_INT8_PER_GROUP, 128, S=2, L=1300, nq=(1300, 300), api=api)
    np.testing.assert_allclose(got, exp, rtol=0, atol=TOL)
    assert pool.error() == kvq.KVQ_OK
    pool.close()
    pool, got, exp, _ = _case(kvq.KVQ_INT8_PER_GROUP, 64, name="mha_100_int8g64", S=2, L=400,
                              nq=(33, 1), api=api)
    np.testing.assert_allclose(got, exp, rtol=0, atol=TOL)
    pool.close()
    pool, got, exp, _ = _case(kvq.KVQ_INT8_PER_GROUP, 64, name="tiny", S=4, L=None, nq=(17, 5, 64, 3),
                              api=api)
    np.testing.assert_allclose(got, exp, rtol=0, atol=TOL)
    pool.close()


def test_prefill_one_token_chunks_equal_decode():
    """A chunk of one token per sequence is exactly the decode problem."""
    w = synth.workload("gqa_64x2048", S=4, L=200, layers=1)
    fmt, group = w.layer_formats[0]
    k, v, slots = layer_tokens(w, 0)
    pool = gpu_pool(w, fmt, group, DEV, k, v, slots)
    q = synth.queries(w, 0)
    qs = np.arange(w.S + 1, dtype=np.int32)
    out = torch.empty((w.S, w.Hq, w.D), dtype=torch.float32, device=DEV)
    kvq.kvq_prefill(pool.handle, _t(q), _t(qs), 1, _t(w.block_table), _t(w.context_lens), 200,
                    w.D ** -0.5, out)
    dec = pool.decode(_t(q), _t(w.block_table), _t(w.context_lens), 200)
    torch.cuda.synchronize()
    np.testing.assert_allclose(out.cpu().numpy(), dec.cpu().numpy(), rtol=2e-5, atol=2e-5)
    pool.close()


@pytest.mark.parametrize("api", APIS)
def test_prefill_edges(api):
    """Ragged tiles, a grid wider than the chunks, an empty chunk, and a
    context shorter than its chunk (flagged; the rows left without a position
    get zeros)."""
    pool, got, exp, l_exp = _case(kvq.KVQ_FP16, 0, nq=(5, 0, 1), api=api)
    np.testing.assert_allclose(got, exp, rtol=0, atol=TOL)
    assert pool.error() == kvq.KVQ_OK
    pool.close()
    pool, got, exp, l_exp = _case(kvq.KVQ_INT8_PER_GROUP, 128, nq=(20, 3, 7), lens=(10, 300, 300),
                                  api=api)
    assert pool.error() == kvq.KVQ_ERR_OUT_OF_RANGE
    assert not got[:10].any()          # positions before the start of the context
    np.testing.assert_allclose(got[10:], exp[10:], rtol=0, atol=TOL)
    pool.close()


@pytest.mark.parametrize("fmt,group,kw,nq", [
    (kvq.KVQ_INT8_PER_GROUP, 128, dict(S=2, L=700, bs=32), (700, 129)),
    (kvq.KVQ_INT8_PER_TOKEN, 0, dict(S=2, L=700, bs=64), (333, 700)),
    (kvq.KVQ_FP8_E4M3_PER_TOKEN, 0, dict(S=2, L=515, bs=32), (64, 515)),
    (kvq.KVQ_INT4_PER_GROUP, 128, dict(S=2, L=640, bs=64), (640, 65)),
])
@pytest.mark.parametrize("api", APIS)
def test_prefill_block_sizes(fmt, group, kw, nq, api):
    """Blocks of 32 and 64 tokens: a 64-token key step spans two pages or one;
    ragged ends of the context and of the chunk."""
    pool, got, exp, _ = _case(fmt, group, nq=nq, api=api, **kw)
    assert pool.error() == kvq.KVQ_OK
    np.testing.assert_allclose(got, exp, rtol=0, atol=TOL)
    pool.close()


@pytest.mark.parametrize("heads,nq", [((32, 32), (300, 1, 129)), ((32, 4), (100, 37, 16)),
                                      ((32, 1), (40, 3, 1)), ((24, 2), (77, 50, 9))])
@pytest.mark.parametrize("api", APIS)
def test_prefill_head_groups(heads, nq, api):
    """MHA (one Q head per kv head: 128 query tokens per tile), GQA 8:1, MQA
    (32 heads: 4 query tokens per tile) and GQA 12:1 (tiles that split a
    token's heads), with the per-token format whose scale spans all heads."""
    pool, got, exp, _ = _case(kvq.KVQ_INT8_PER_TOKEN, 0, S=3, L=300, nq=nq, heads=heads, api=api)
    assert pool.error() == kvq.KVQ_OK
    np.testing.assert_allclose(got, exp, rtol=0, atol=TOL)
    pool.close()


def test_prefill_ex_workspace_rules():
    """kvq_prefill_ex refuses a missing or short workspace for the formats it
    stages, and needs none (runs kvq_prefill) for per-group formats with
    several groups per head."""
    w = synth.workload("gqa_64x2048", S=2, L=100, layers=1)
    for fmt, group in [(kvq.KVQ_INT8_PER_GROUP, 128), (kvq.KVQ_INT8_PER_GROUP, 32)]:
        pool = kvq.KVPool(w.num_blocks, w.bs, w.Hkv, w.D, fmt, group, device=DEV)
        nb = kvq.kvq_prefill_workspace_bytes(pool.handle, w.S, 100)
        q = torch.zeros((10, w.Hq, w.D), dtype=torch.float16, device=DEV)
        qs = _t(np.array([0, 5, 10], np.int32))
        out = torch.empty((10, w.Hq, w.D), dtype=torch.float32, device=DEV)
        args = (pool.handle, q, qs, 5, _t(w.block_table), _t(w.context_lens), 100, 0.1, out)
        if group == 128:
            assert nb == w.S * 2 * w.Hkv * 33792     # two 64-token steps per sequence
            with pytest.raises(kvq.KVQError) as e:
                kvq.kvq_prefill_ex(*args, None)
            assert e.value.status == kvq.KVQ_ERR_WORKSPACE
            with pytest.raises(kvq.KVQError) as e:
                kvq.kvq_prefill_ex(*args, torch.empty(nb - 256, dtype=torch.uint8, device=DEV))
            assert e.value.status == kvq.KVQ_ERR_WORKSPACE
        else:
            assert nb == 0
            kvq.kvq_prefill_ex(*args, None)
        torch.cuda.synchronize()
        pool.close()
