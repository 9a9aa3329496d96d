"""The prefill precision case, on the CPU: the tolerance PREC_TOL separates
softmax weights of fp32-level precision from fp16 weights.

The GPU prefill kernels hand the weights p * s_V to the tensor core as an fp16
high part plus an fp16 low part.  The GPU test of that case only shows that
the low part arrived with the right sign if dropping it, or flipping its sign,
would fail the same bound.  This test computes, in float64 over the oracle's
dequantized cache, the outputs of sampled query rows of the same case three
ways: exact weights, weights rounded to fp32, and weights rounded to fp16
(relative spacing 2^-11, the rounding a lone high part carries)."""
import numpy as np
import pytest

import paged_quantized_kv_kvq_gb300 as kvq
from paged_quantized_kv_kvq_gb300 import synth
from kvq_testutil import PREC_TOL, layer_tokens, oracle_layer

FORMATS = [(kvq.KVQ_INT8_PER_GROUP, 128), (kvq.KVQ_FP16, 0), (kvq.KVQ_INT8_PER_CHANNEL, 0),
           (kvq.KVQ_INT4_PER_GROUP, 32)]


def _outputs(fmt, group, S=2, L=600, nq=(600, 200), seed=0, every=23):
    """The same workload, cache and queries as the GPU precision test."""
    w = synth.workload("gqa_64x2048", S=S, L=L, layers=1)
    w.layer_formats = [(fmt, group)]
    k, v, slots = layer_tokens(w, 0)
    calib = (k, v) if fmt == kvq.KVQ_INT8_PER_CHANNEL else None
    ref, table, _ = oracle_layer(w, fmt, group, k, v, slots, list(range(w.S)), calib=calib)
    K, V = ref.dequantized(0), ref.dequantized(1)
    nq = np.asarray(nq)
    q_all = np.random.default_rng(seed).standard_normal((int(nq.sum()), w.Hq, w.D)).astype(np.float16)
    G = w.Hq // w.Hkv
    err32 = err16 = 0.0
    base = 0
    for s in range(S):
        Ls, n = int(w.context_lens[s]), int(nq[s])
        idx = (table[s][:, None] * w.bs + np.arange(w.bs)[None]).ravel()[:Ls]
        Ks, Vs = K[idx], V[idx]
        for i in range(0, n, every):
            Lc = Ls - n + i + 1  # causal length of query token i of the chunk
            q = q_all[base + i].astype(np.float64)
            for h in range(w.Hq):
                sc = Ks[:Lc, h // G] @ q[h] * w.D ** -0.5
                p = np.exp(sc - sc.max())
                o = p @ Vs[:Lc, h // G] / p.sum()
                p32 = p.astype(np.float32).astype(np.float64)
                p16 = (p * 2.0 ** 13).astype(np.float16).astype(np.float64) / 2.0 ** 13
                err32 = max(err32, float(np.abs(p32 @ Vs[:Lc, h // G] / p.sum() - o).max()))
                err16 = max(err16, float(np.abs(p16 @ Vs[:Lc, h // G] / p.sum() - o).max()))
        base += n
    return err32, err16


@pytest.mark.parametrize("fmt,group", FORMATS)
def test_precision_tolerance_separates_fp16_weights(fmt, group):
    err32, err16 = _outputs(fmt, group)
    assert err32 < PREC_TOL / 100, err32
    assert err16 > 2 * PREC_TOL, err16
