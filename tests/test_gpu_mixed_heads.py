"""Per-head mixed precision (xpshop.cn article-312 §六: the attention heads
that quantization hurts stay FP16, the others are quantized): two pools per
layer over a contiguous split of the kv heads, filled and read through head
slices of the full rows (kvq_append_strided / kvq_paged_decode_strided).
Outputs within 1e-3 of the float64 oracle built from the same split."""
import numpy as np
import pytest
import torch

import oracle
import paged_quantized_kv_kvq_gb300 as kvq
from paged_quantized_kv_kvq_gb300 import synth
from kvq_testutil import TOL, gpu_pool, layer_tokens

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.mark.parametrize("split,qfmt,group", [(2, kvq.KVQ_INT8_PER_GROUP, 128),
                                              (3, kvq.KVQ_FP8_E4M3_PER_TOKEN, 0),
                                              (1, kvq.KVQ_INT4_PER_GROUP, 32)])
def test_fp16_heads_beside_quantized_heads(split, qfmt, group):
    w = synth.workload("gqa_64x2048", S=4, L=300, layers=1)
    k, v, slots = layer_tokens(w, 0)
    q = synth.queries(w, 0)
    G, D = w.G, w.D
    kd, vd = torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV)
    sl = torch.from_numpy(slots).to(DEV)
    qd = torch.from_numpy(q).to(DEV)
    table, lens = torch.from_numpy(w.block_table).to(DEV), torch.from_numpy(w.context_lens).to(DEV)
    mc = int(w.context_lens.max())
    parts = [(kvq.KVQ_FP16, 0, 0, split), (qfmt, group, split, w.Hkv)]
    out = torch.full((w.S, w.Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    exp = np.zeros((w.S, w.Hq, D))
    for fmt, g, h0, h1 in parts:
        pool = kvq.KVPool(w.num_blocks, w.bs, h1 - h0, D, fmt, g, device=DEV)
        kvq.kvq_append_strided(pool.handle, kd[:, h0:h1], vd[:, h0:h1], sl)
        nws = kvq.kvq_decode_workspace_bytes(pool.handle, w.S, (h1 - h0) * G, mc)
        ws = torch.empty(max(nws, 256), dtype=torch.uint8, device=DEV)
        kvq.kvq_paged_decode_strided(pool.handle, qd[:, h0 * G:h1 * G], table, lens, mc,
                                     D ** -0.5, out[:, h0 * G:h1 * G], ws)
        torch.cuda.synchronize()
        assert pool.error() == kvq.KVQ_OK
        ref = oracle.OracleCache(fmt, w.num_blocks, w.bs, h1 - h0, D, g)
        ref.append(k[:, h0:h1], v[:, h0:h1], slots)
        exp[:, h0 * G:h1 * G] = ref.decode(q[:, h0 * G:h1 * G], w.block_table, w.context_lens)
        pool.close()
    np.testing.assert_allclose(out.cpu().numpy(), exp, rtol=0, atol=TOL)


def test_strided_equals_dense_and_refuses_bad_strides():
    w = synth.workload("gqa_64x2048", S=3, L=200, layers=1)
    fmt, g = w.layer_formats[0]
    k, v, slots = layer_tokens(w, 0)
    pool = gpu_pool(w, fmt, g, DEV, k, v, slots)
    q = torch.from_numpy(synth.queries(w, 0)).to(DEV)
    table, lens = torch.from_numpy(w.block_table).to(DEV), torch.from_numpy(w.context_lens).to(DEV)
    dense = pool.decode(q, table, lens, 200)
    # the same call through the strided entry point with padded rows
    qpad = torch.zeros((w.S, w.Hq + 8, w.D), dtype=torch.float16, device=DEV)
    qpad[:, :w.Hq] = q
    opad = torch.zeros((w.S, w.Hq + 3, w.D), dtype=torch.float32, device=DEV)
    nws = kvq.kvq_decode_workspace_bytes(pool.handle, w.S, w.Hq, 200)
    ws = torch.empty(max(nws, 256), dtype=torch.uint8, device=DEV)
    kvq.kvq_paged_decode_strided(pool.handle, qpad[:, :w.Hq], table, lens, 200, w.D ** -0.5,
                                 opad[:, :w.Hq], ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(opad[:, :w.Hq].cpu().numpy(), dense.cpu().numpy())
    assert not opad[:, w.Hq:].any()               # nothing written past the slice
    kd = torch.from_numpy(k[:4]).to(DEV)
    short = torch.as_strided(kd, (4, w.Hkv, w.D), (8, w.D, 1))  # rows overlap
    with pytest.raises(kvq.KVQError) as e:        # a row stride shorter than the row
        kvq.kvq_append_strided(pool.handle, short, short, torch.from_numpy(slots[:4]).to(DEV))
    assert e.value.status == kvq.KVQ_ERR_INVALID_ARG
    pool.close()
