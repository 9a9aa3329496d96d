"""Failure detection without a GPU fault: a pipeline wait that nothing will
complete (a page copy announced to its barrier but never issued) gives up
after its bound, the pool's error word reports a timeout, and the context
keeps working -- the next decode matches the oracle."""
import time

import numpy as np
import pytest
import torch

import paged_quantized_kv_kvq_gb300 as kvq
from paged_quantized_kv_kvq_gb300 import synth
from kvq_testutil import TOL, gpu_pool, layer_tokens, oracle_layer, run_gpu_decode

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def test_bounded_wait_times_out_and_context_survives():
    w = synth.workload("gqa_64x2048", S=4, L=600, layers=1)
    fmt, g = w.layer_formats[0]
    k, v, slots = layer_tokens(w, 0)
    pool = gpu_pool(w, fmt, g, DEV, k, v, slots)
    ref, table, _ = oracle_layer(w, fmt, g, k, v, slots, list(range(w.S)))
    q = synth.queries(w, 0)
    mc = int(w.context_lens.max())
    ws = torch.empty(max(kvq.kvq_decode_workspace_bytes(pool.handle, w.S, w.Hq, mc), 256),
                     dtype=torch.uint8, device=DEV)
    out = torch.empty((w.S, w.Hq, w.D), dtype=torch.float32, device=DEV)
    assert pool.error() == kvq.KVQ_OK
    t0 = time.perf_counter()
    kvq.kvq_selftest_decode_timeout(pool.handle, _t(q), _t(w.block_table), _t(w.context_lens), mc,
                                    out, ws, wait_tries=20)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 30.0        # bounded: 20 tries of <= ~1 ms each
    assert pool.error() == kvq.KVQ_ERR_TIMEOUT
    assert pool.error() == kvq.KVQ_OK             # read and cleared
    got = run_gpu_decode(pool, w, q, DEV)         # the context is still healthy
    np.testing.assert_allclose(got, ref.decode(q, table, w.context_lens), rtol=0, atol=TOL)
    assert pool.error() == kvq.KVQ_OK
    with pytest.raises(kvq.KVQError):
        kvq.kvq_selftest_decode_timeout(pool.handle, _t(q), _t(w.block_table), _t(w.context_lens),
                                        mc, out, ws, wait_tries=0)
    pool.close()
