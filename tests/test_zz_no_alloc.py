"""kvq_paged_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (a serving loop with all memory reserved up front, a
capped allocator, host code where cudaMalloc is not allowed).  Its split-K
scratch is a fixed array inside the library instead of a caller workspace.

The test calls it through the C ABI twice in a row and checks each result
against kvq_paged_decode with a caller-allocated workspace, within the
parity tolerance used for decode; it also checks that a call needing more
scratch than the fixed maximum is refused before anything is launched.  It
sits in a file of its own, collected last, and works in a fresh process (the
first call on the device looks up the array's address) as well as after the
other tests (the array then holds an earlier call's partials)."""
import numpy as np
import pytest
import torch

import paged_quantized_kv_kvq_gb300 as kvq
from paged_quantized_kv_kvq_gb300 import synth
from kvq_testutil import TOL, gpu_pool, layer_tokens

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def test_noalloc_decode_matches_workspace_decode():
    w = synth.workload("gqa_64x2048", S=8, L=1000, layers=1)
    fmt, g = w.layer_formats[0]
    k, v, slots = layer_tokens(w, 0)
    pool = gpu_pool(w, fmt, g, DEV, k, v, slots)
    q = torch.from_numpy(synth.queries(w, 0)).to(DEV)
    table = torch.from_numpy(w.block_table).to(DEV)
    lens = torch.from_numpy(w.context_lens).to(DEV)
    max_ctx = int(w.context_lens.max())
    sm = w.D ** -0.5
    need = kvq.kvq_decode_workspace_bytes(pool.handle, w.S, w.Hq, max_ctx)
    assert 0 < need <= kvq.KVQ_NOALLOC_SCRATCH_BYTES   # the call really uses split scratch

    ref = pool.decode(q, table, lens, max_ctx, sm)      # caller-provided workspace
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        kvq.kvq_paged_decode_noalloc(pool.handle, q, table, lens, max_ctx, sm, out)
        torch.cuda.synchronize()
        diff = (out - ref).abs().max().item()
        assert np.isfinite(diff) and diff <= TOL, diff
    assert pool.error() == kvq.KVQ_OK

    # forcing one block per split for 32 sequences needs more than the fixed scratch
    S2 = 32
    q2 = torch.zeros((S2, w.Hq, w.D), dtype=torch.float16, device=DEV)
    t2 = torch.zeros((S2, w.max_blocks), dtype=torch.int32, device=DEV)
    l2 = torch.zeros(S2, dtype=torch.int32, device=DEV)
    o2 = torch.zeros((S2, w.Hq, w.D), dtype=torch.float32, device=DEV)
    assert kvq.kvq_decode_workspace_bytes(pool.handle, S2, w.Hq, max_ctx, 1) > kvq.KVQ_NOALLOC_SCRATCH_BYTES
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_paged_decode_noalloc(pool.handle, q2, t2, l2, max_ctx, sm, o2, split_blocks=1)
    assert e.value.status == kvq.KVQ_ERR_WORKSPACE
    pool.close()
