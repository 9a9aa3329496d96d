"""The seeded input recipes hold the shapes and structure of the workloads they
stand for (the 7B-class decode configurations of "KV Cache优化实战", §1.2,
§2.1, §3, and xpshop.cn article-312 §三), and the host generator gives every
token the same values whatever subset is asked for -- the property the
full-size parity tests rely on when the oracle regenerates only sampled
sequences.  CPU only."""
import math

import numpy as np
import pytest

from paged_quantized_kv_kvq_gb300 import synth


def _check_table(w, prefix_blocks=0):
    nblk = (w.context_lens.astype(np.int64) + w.bs - 1) // w.bs
    used = []
    for s in range(w.S):
        row = w.block_table[s, :nblk[s]]
        assert np.all((row >= 0) & (row < w.num_blocks))
        used.append(row[prefix_blocks:])
        if prefix_blocks:
            np.testing.assert_array_equal(row[:prefix_blocks], w.block_table[0, :prefix_blocks])
    used = np.concatenate(used + [w.block_table[0, :prefix_blocks]])
    assert len(np.unique(used)) == len(used), "two logical blocks share a physical block"
    return nblk


def test_tiny():
    w = synth.workload("tiny")
    assert (w.S, w.Hq, w.Hkv, w.D, w.bs, w.num_blocks) == (4, 4, 1, 64, 16, 64)
    np.testing.assert_array_equal(w.context_lens, [17, 33, 64, 100])
    assert w.layer_formats == [(synth.INT8_PER_GROUP, 64)]
    assert len(w.outlier_channels) == 2 and w.outlier_gain == 20.0
    nblk = _check_table(w)
    assert nblk.sum() == 16


@pytest.mark.parametrize("name,fmt", [("gqa_64x2048", (synth.INT8_PER_GROUP, 128)),
                                      ("gqa_64x2048_int4", (synth.INT4_PER_GROUP, 128)),
                                      ("gqa_64x2048_e5m2", (synth.FP8_E5M2, 0))])
def test_gqa_64x2048(name, fmt):
    w = synth.workload(name)
    assert (w.layers, w.S, w.Hq, w.Hkv, w.D, w.bs) == (32, 64, 32, 8, 128, 16)
    assert np.all(w.context_lens == 2048)
    assert all(f == fmt for f in w.layer_formats)
    need = 64 * 2048 // 16
    assert w.num_blocks == math.ceil(need / 0.9)        # 90% of the pool is used
    assert len(w.outlier_channels) == round(0.01 * 8 * 128) and w.outlier_gain == 10.0
    _check_table(w)


@pytest.mark.parametrize("name,fmt", [("mha_100_fp16", (synth.FP16, 0)),
                                      ("mha_100_fp8", (synth.FP8_E4M3_PER_TOKEN, 0)),
                                      ("mha_100_int8ch", (synth.INT8_PER_CHANNEL, 0)),
                                      ("mha_100_int8g64", (synth.INT8_PER_GROUP, 64))])
def test_mha_100(name, fmt):
    w = synth.workload(name)
    assert (w.layers, w.S, w.Hq, w.Hkv, w.D, w.bs) == (32, 100, 32, 32, 128, 16)
    assert w.context_lens.min() >= 256 and w.context_lens.max() <= 2048
    assert len(np.unique(w.context_lens)) > 50                # a length mix, not one length
    assert all(f == fmt for f in w.layer_formats)
    _check_table(w)


@pytest.mark.parametrize("bs", [16, 32])
def test_long_8x32k(bs):
    w = synth.workload("long_8x32k", bs=bs)
    assert (w.layers, w.S, w.Hq, w.Hkv, w.D, w.bs) == (32, 8, 32, 8, 128, bs)
    assert np.all(w.context_lens == 32768) and w.drift_sigma == 0.01
    _check_table(w)


def test_long_drift_is_a_random_walk():
    # the per-channel mean walks: far-apart tokens drift apart more than near ones
    w = synth.workload("long_8x32k", S=1, L=4096, layers=1)
    idx = np.stack([np.zeros(4096, np.int64), np.arange(4096)], 1)
    k, _ = synth.kv_tokens(w, 0, idx)
    m = k.astype(np.float64).reshape(64, 64, w.Hkv, w.D).mean(axis=1)  # 64-token window means
    near = np.abs(m[1:] - m[:-1]).mean()
    far = np.abs(m[63] - m[0]).mean()
    assert far > 3 * near


def test_mixed_256():
    w = synth.workload("mixed_256")
    assert (w.layers, w.S, w.Hq, w.Hkv, w.D, w.bs) == (32, 256, 32, 8, 128, 16)
    assert w.shared_prefix_tokens == 512
    suffix = w.context_lens - 512
    assert suffix.min() >= 64 and suffix.max() <= 8192
    assert 600 < np.median(suffix) < 1700                    # log-normal, median 1024
    assert w.layer_formats[:28] == [(synth.INT8_PER_GROUP, 128)] * 28
    assert w.layer_formats[28:] == [(synth.FP16, 0)] * 4
    _check_table(w, prefix_blocks=512 // 16)


def test_shared4k_256():
    w = synth.workload("shared4k_256")
    assert w.S == 256 and w.shared_prefix_tokens == 4096
    _check_table(w, prefix_blocks=4096 // 16)


@pytest.mark.parametrize("name,kw", [("gqa_64x2048", dict(S=4, L=300)),
                                     ("long_8x32k", dict(S=2, L=700)),
                                     ("mixed_256", dict(S=5, L=200))])
def test_tokens_do_not_depend_on_the_subset(name, kw):
    w = synth.workload(name, layers=1, **kw)
    idx = w.fill_token_index()
    k_all, v_all = synth.kv_tokens(w, 0, idx)
    rng = np.random.default_rng(0)
    pick = np.sort(rng.choice(len(idx), size=min(50, len(idx)), replace=False))
    k_sub, v_sub = synth.kv_tokens(w, 0, idx[pick])
    np.testing.assert_array_equal(k_sub, k_all[pick])
    np.testing.assert_array_equal(v_sub, v_all[pick])
    # a later sequence's shared-prefix tokens are sequence 0's
    if w.shared_prefix_tokens:
        p = np.stack([np.full(4, 3), np.arange(4)], 1)
        q0 = np.stack([np.zeros(4, np.int64), np.arange(4)], 1)
        np.testing.assert_array_equal(synth.kv_tokens(w, 0, p)[0], synth.kv_tokens(w, 0, q0)[0])


def test_slots_cover_every_cached_token_once():
    w = synth.workload("mixed_256", S=6, L=300, layers=1)
    fill, step = w.fill_slots(), w.step_slots()
    assert len(np.unique(fill)) == len(fill)
    assert not np.isin(step, fill).any()
    # every position 0 .. L-2 of every sequence maps to a filled slot (the
    # prefix once, under sequence 0), position L-1 to the step slot
    for s in range(w.S):
        L = int(w.context_lens[s])
        np.testing.assert_array_equal(np.isin(w.slots_for(s, 0, L - 1), fill), True)
        assert w.slots_for(s, L - 1, L)[0] == step[s]
