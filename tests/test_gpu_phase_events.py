"""kvq_set_phase_events, the per-kernel timing aid: events recorded after the
library's kernel launches split a call into its kernels (decode kernel, then
split merge; append, decode, merge for the step; staging, then attention for
the two-pass prefill) without changing any result bit, and recording stops
after the events handed over."""
import numpy as np
import pytest
import torch

import paged_quantized_kv_kvq_gb300 as kvq
from paged_quantized_kv_kvq_gb300 import synth
from kvq_testutil import gpu_pool, layer_tokens

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def _events(n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def _case():
    w = synth.workload("gqa_64x2048", S=6, L=700, layers=1)  # 44 blocks per unit: cut units
    fmt, group = w.layer_formats[0]
    k, v, slots = layer_tokens(w, 0)
    S = w.S
    return w, fmt, group, k, v, slots, S


def test_phase_events_split_the_decode_call():
    w, fmt, group, k, v, slots, S = _case()
    pool = gpu_pool(w, fmt, group, DEV, k, v, slots)
    q, table, lens = _t(synth.queries(w, 0)), _t(w.block_table), _t(w.context_lens)
    L = int(w.context_lens.max())
    plain = pool.decode(q, table, lens, L, split_blocks=5)
    torch.cuda.synchronize()
    ev = _events(4)
    kvq.kvq_set_phase_events(ev[1:3])            # decode kernel, merge kernel
    ev[0].record()
    timed = pool.decode(q, table, lens, L, split_blocks=5)
    ev[3].record()
    torch.cuda.synchronize()
    assert pool.error() == kvq.KVQ_OK
    assert torch.equal(plain, timed)
    t_dec, t_merge, t_all = ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2]), ev[0].elapsed_time(ev[3])
    assert t_dec > 0 and t_merge >= 0
    assert t_dec + t_merge <= t_all + 1e-3
    # both events used: the next call records nothing, so they keep their times
    pool.decode(q, table, lens, L, split_blocks=5)
    torch.cuda.synchronize()
    assert ev[0].elapsed_time(ev[2]) == pytest.approx(t_dec + t_merge, abs=2e-3)
    pool.close()


def test_phase_events_split_the_decode_step():
    w, fmt, group, k, v, slots, S = _case()
    q, table, lens = _t(synth.queries(w, 0)), _t(w.block_table), _t(w.context_lens)
    L = int(w.context_lens.max())
    outs = []
    for with_events in (False, True):
        pool = gpu_pool(w, fmt, group, DEV, k[:-S], v[:-S], slots[:-S])
        ev = _events(4)
        if with_events:
            kvq.kvq_set_phase_events(ev[1:])      # append, decode, merge
        ev[0].record()
        outs.append(pool.decode_step(_t(k[-S:]), _t(v[-S:]), q, table, lens, L))
        torch.cuda.synchronize()
        assert pool.error() == kvq.KVQ_OK
        if with_events:
            times = [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]
            assert all(t >= 0 for t in times) and times[1] > 0
        pool.close()
    assert torch.equal(outs[0], outs[1])


def test_phase_events_split_the_two_pass_prefill():
    w = synth.workload("gqa_64x2048", S=2, L=300, layers=1)
    fmt, group = w.layer_formats[0]
    k, v, slots = layer_tokens(w, 0)
    pool = gpu_pool(w, fmt, group, DEV, k, v, slots)
    n = 40                                        # each sequence's last 40 tokens are the chunk
    rng = np.random.default_rng(3)
    q = _t(rng.standard_normal((w.S * n, w.Hq, w.D)).astype(np.float16))
    q_start = _t(np.arange(w.S + 1, dtype=np.int32) * n)
    table, lens = _t(w.block_table), _t(w.context_lens)
    L = int(w.context_lens.max())
    nb = kvq.kvq_prefill_workspace_bytes(pool.handle, w.S, L)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=DEV)
    outs = [torch.empty((w.S * n, w.Hq, w.D), dtype=torch.float32, device=DEV) for _ in range(2)]
    args = (pool.handle, q, q_start, n, table, lens, L, w.D ** -0.5)
    kvq.kvq_prefill_ex(*args, outs[0], ws)
    torch.cuda.synchronize()
    ev = _events(3)
    kvq.kvq_set_phase_events(ev[1:])              # staging kernel, attention kernel
    ev[0].record()
    kvq.kvq_prefill_ex(*args, outs[1], ws)
    torch.cuda.synchronize()
    plain, timed = outs
    assert pool.error() == kvq.KVQ_OK
    assert torch.equal(plain, timed)
    assert ev[0].elapsed_time(ev[1]) > 0 and ev[1].elapsed_time(ev[2]) > 0
    pool.close()


def test_phase_events_cleared():
    ev = _events(2)
    kvq.kvq_set_phase_events(ev)
    kvq.kvq_set_phase_events([])                  # nothing recorded from here on
    w, fmt, group, k, v, slots, S = _case()
    pool = gpu_pool(w, fmt, group, DEV, k, v, slots)
    torch.cuda.synchronize()
    stamp = ev[0].elapsed_time(ev[1])             # the events' own first records
    pool.decode(_t(synth.queries(w, 0)), _t(w.block_table), _t(w.context_lens),
                int(w.context_lens.max()))
    torch.cuda.synchronize()
    assert ev[0].elapsed_time(ev[1]) == stamp
    pool.close()


def test_phase_events_split_the_cascade_and_carry_over():
    """The cascade's three kernels (shared-prefix rows, decode, merge) each
    take an event; events beyond one call's launches go to the next call's
    (the count runs across calls): five events over a cascade call (three
    launches) and a plain decode call (two)."""
    w = synth.workload("mixed_256", S=4, L=100, layers=1)
    fmt, group = w.layer_formats[0]
    k, v, slots = layer_tokens(w, 0)
    pool = gpu_pool(w, fmt, group, DEV, k, v, slots)
    q, table, lens = _t(synth.queries(w, 0)), _t(w.block_table), _t(w.context_lens)
    L = int(w.context_lens.max())
    P = w.shared_prefix_tokens // w.bs
    plain = pool.cascade_decode(q, table, lens, L, P)
    torch.cuda.synchronize()
    ev = _events(6)
    kvq.kvq_set_phase_events(ev[1:])
    ev[0].record()
    timed = pool.cascade_decode(q, table, lens, L, P)   # rows, decode, merge: ev[1..3]
    dec = pool.decode(q, table, lens, L)                # decode, merge: ev[4..5]
    torch.cuda.synchronize()
    assert pool.error() == kvq.KVQ_OK
    assert torch.equal(plain, timed)
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(5)]
    assert all(t >= 0 for t in times) and times[1] > 0 and times[3] > 0
    np.testing.assert_allclose(dec.cpu().numpy(), timed.cpu().numpy(), rtol=0, atol=3e-5)
    pool.close()
