"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle on
the same seeded inputs.  Codes, scales and slot placement must match bit for
bit; attention outputs within 1e-3 (max abs) of the float64 oracle on the same
dequantized cache.  Sizes here span several blocks and ragged tails; the
full-size workloads are checked on sampled sequences in test_gpu_fullsize."""
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
           (kvq.KVQ_FP8_E4M3_PER_TOKEN, 0), (kvq.KVQ_FP16, 0), (kvq.KVQ_INT4_PER_GROUP, 128),
           (kvq.KVQ_INT4_PER_GROUP, 32), (kvq.KVQ_INT4_PER_GROUP, 16), (kvq.KVQ_FP8_E5M2, 0)]


def _calib(fmt, k, v):
    return (k, v) if fmt == kvq.KVQ_INT8_PER_CHANNEL else None


def _compare_codes(pool, ref, slots_np, ref_slots=None):
    """Bit-exact codes and scales of device slots vs the oracle's store."""
    ref_slots = slots_np if ref_slots is None else ref_slots
    codes, scales = pool.read_slots(torch.from_numpy(slots_np).to(DEV))
    torch.cuda.synchronize()
    c = codes.cpu().numpy()
    if pool.dtype == kvq.KVQ_FP16:
        np.testing.assert_array_equal(c.astype(np.float32), ref.codes[ref_slots])
    else:
        np.testing.assert_array_equal(c.view(np.uint8), ref.codes[ref_slots].view(np.uint8))
    if scales is not None:
        np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32),
                                      ref.scales[ref_slots].view(np.uint32))


def _layer_case(w, layer, fmt, group, seqs=None):
    seqs = list(range(w.S)) if seqs is None else seqs
    k, v, slots = layer_tokens(w, layer)
    calib = _calib(fmt, k, v)
    pool = gpu_pool(w, fmt, group, DEV, k, v, slots, calib=calib)
    ref, table, remap = oracle_layer(w, fmt, group, k, v, slots, seqs, calib=calib)
    # every appended slot holds exactly the oracle's codes and scales
    last = {int(x): i for i, x in enumerate(slots)}
    uniq = np.array(sorted(last), np.int64)
    _compare_codes(pool, ref, uniq, oracle_slots(remap, uniq, w.bs))
    return pool, ref, table, (k, v, slots)


@pytest.mark.parametrize("fmt,group", FORMATS)
@pytest.mark.parametrize("D", [64, 128])
def test_append_bitexact_and_sentinels(fmt, group, D):
    if group > D:
        pytest.skip("group larger than head_dim")
    rng = np.random.default_rng(D + fmt + group)
    nb, bs, hkv = 12, 16, 3
    T = 70
    x = rng.standard_normal((2, T, hkv, D)).astype(np.float32)
    x[:, :, :, rng.integers(0, D, 3)] *= 20.0          # outlier channels
    x[:, 5] = 0.0                                       # an all-zero token
    x[:, 7, 1, :] = 0.0                                 # an all-zero head
    x[:, 9] *= 1e-4                                     # tiny values
    k, v = x.astype(np.float16)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[[3, 11, 40]] = -1                             # padding tokens
    # INT4 pools get a fill whose every nibble is the same (9 = code +1)
    fill = 0x99 if fmt == kvq.KVQ_INT4_PER_GROUP else 0x5A
    pool = kvq.KVPool(nb, bs, hkv, D, fmt, group, device=DEV, fill_byte=fill)
    ref = oracle.OracleCache(fmt, nb, bs, hkv, D, group,
                             sentinel_code=1 if fmt == kvq.KVQ_INT4_PER_GROUP else fill)
    if fmt == kvq.KVQ_INT8_PER_CHANNEL:
        kvq.kvq_calibrate_channel_scales(pool.handle, torch.from_numpy(k[:50]).to(DEV),
                                         torch.from_numpy(v[:50]).to(DEV))
        ref.calibrate(k[:50], v[:50])
    pool.append(torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV),
                torch.from_numpy(slots).to(DEV))
    ref.append(k, v, slots)
    assert pool.error() == kvq.KVQ_OK
    written = np.sort(slots[slots >= 0])
    _compare_codes(pool, ref, written)
    # untouched slots still hold the sentinel bytes
    untouched = np.setdiff1d(np.arange(nb * bs), written)
    codes, scales = pool.read_slots(torch.from_numpy(untouched).to(DEV))
    # the read-back returns signed codes; the pool stores INT8 biased by 128
    # and INT4 nibbles biased by 8
    sentinel = {kvq.KVQ_INT8_PER_TOKEN: 0x5A ^ 0x80, kvq.KVQ_INT8_PER_CHANNEL: 0x5A ^ 0x80,
                kvq.KVQ_INT8_PER_GROUP: 0x5A ^ 0x80, kvq.KVQ_INT4_PER_GROUP: 9 - 8}.get(fmt, 0x5A)
    assert np.all(codes.cpu().numpy().view(np.uint8) == sentinel)
    if scales is not None:
        assert np.all(scales.cpu().numpy().view(np.uint32) == fill * 0x01010101)
    pool.close()


@pytest.mark.parametrize("fmt,group", FORMATS)
def test_decode_small_parity(fmt, group):
    w = synth.workload("gqa_64x2048", S=3, L=301, layers=1)
    w.layer_formats = [(fmt, group)]
    pool, ref, table, _ = _layer_case(w, 0, fmt, group)
    q = synth.queries(w, 0)
    got = run_gpu_decode(pool, w, q, DEV)
    exp = ref.decode(q, table, w.context_lens)
    np.testing.assert_allclose(got, exp, rtol=0, atol=TOL)
    assert pool.error() == kvq.KVQ_OK
    pool.close()


def test_per_channel_decode_attends_saturated_codes():
    """Per-channel scales calibrated on the first 32 cached tokens only: tokens
    beyond that range append as +-127, and the decode must attend those
    clipped codes exactly as the oracle's store holds them."""
    w = synth.workload("mha_100_int8ch", S=5, L=300, layers=1)
    fmt, group = kvq.KVQ_INT8_PER_CHANNEL, 0
    k, v, slots = layer_tokens(w, 0)
    calib = (k[:32], v[:32])
    pool = gpu_pool(w, fmt, group, DEV, k, v, slots, calib=calib)
    ref, table, remap = oracle_layer(w, fmt, group, k, v, slots, list(range(w.S)), calib=calib)
    last = {int(x): i for i, x in enumerate(slots)}
    uniq = np.array(sorted(last), np.int64)
    _compare_codes(pool, ref, uniq, oracle_slots(remap, uniq, w.bs))
    codes = ref.codes[oracle_slots(remap, uniq, w.bs)].view(np.int8)
    assert np.mean(np.abs(codes.astype(np.int32)) == 127) > 0.005   # many clipped codes
    q = synth.queries(w, 0)
    got = run_gpu_decode(pool, w, q, DEV)
    np.testing.assert_allclose(got, ref.decode(q, table, w.context_lens), rtol=0, atol=TOL)
    assert pool.error() == kvq.KVQ_OK
    pool.close()


def test_tiny_workload_full():
    w = synth.workload("tiny")
    fmt, g = w.layer_formats[0]
    pool, ref, table, (k, v, slots) = _layer_case(w, 0, fmt, g)
    q = synth.queries(w, 0)
    got = run_gpu_decode(pool, w, q, DEV)
    exp = ref.decode(q, table, w.context_lens)
    np.testing.assert_allclose(got, exp, rtol=0, atol=TOL)
    for sb in (1, 2, 3, 7):
        np.testing.assert_allclose(run_gpu_decode(pool, w, q, DEV, split_blocks=sb), got,
                                   rtol=2e-5, atol=2e-5)
    pool.close()


@pytest.mark.parametrize("name,kw", [
    ("mha_100_fp16", dict(S=5, L=300)), ("mha_100_fp8", dict(S=5, L=300)),
    ("mha_100_int8ch", dict(S=5, L=300)), ("mha_100_int8g64", dict(S=5, L=300)),
    ("long_8x32k", dict(S=1, L=3001, bs=16)), ("long_8x32k", dict(S=1, L=3001, bs=32)),
    ("long_8x32k", dict(S=1, L=3001, bs=64)),
    ("mixed_256", dict(S=5, L=200, layers=2)), ("gqa_64x2048_int4", dict(S=3, L=500)),
    ("gqa_64x2048_e5m2", dict(S=3, L=500)),
])
def test_workload_reduced_parity(name, kw):
    w = synth.workload(name, **kw)
    for layer, (fmt, group) in enumerate(w.layer_formats):
        pool, ref, table, _ = _layer_case(w, layer, fmt, group)
        q = synth.queries(w, layer)
        got = run_gpu_decode(pool, w, q, DEV)
        exp = ref.decode(q, table, w.context_lens)
        np.testing.assert_allclose(got, exp, rtol=0, atol=TOL, err_msg="%s layer %d" % (name, layer))
        assert pool.error() == kvq.KVQ_OK
        pool.close()


@pytest.mark.parametrize("bs", [16, 32])
def test_split_k_invariance(bs):
    w = synth.workload("long_8x32k", S=2, L=2500, bs=bs, layers=1)
    pool, ref, table, _ = _layer_case(w, 0, *w.layer_formats[0])
    q = synth.queries(w, 0)
    base = run_gpu_decode(pool, w, q, DEV, split_blocks=10 ** 6)   # one split
    np.testing.assert_allclose(base, ref.decode(q, table, w.context_lens), rtol=0, atol=TOL)
    # Only the fp32 summation order changes with the split: one block per
    # piece merges up to ~160 partials, ~160 * 2^-24 relative, hence 2e-5.
    for sb in (1, 2, 7, 0):
        np.testing.assert_allclose(run_gpu_decode(pool, w, q, DEV, split_blocks=sb), base,
                                   rtol=2e-5, atol=2e-5, err_msg="split_blocks=%d" % sb)
    pool.close()


@pytest.mark.parametrize("bs", [16, 32])
def test_split_merge_chunks(bs):
    """Warp ranges of 1024 tokens or more make the merge load 16 pieces per
    round trip: 21 pieces per unit (a whole chunk and a partial one) and 12
    (one partial chunk), and one-page pieces (1500 or 750 per unit, many
    chunks of 8), each against the oracle.  The bound is tighter than the
    path's 1e-3: with ranges of at most 2048 tokens the tensor cores' fp32
    accumulation of P.V stays within ~4e-5 here (a single 24000-token range
    drifts to ~5e-4; the error grows with the tokens one accumulator sums)."""
    w = synth.workload("long_8x32k", S=1, L=24000, bs=bs, layers=1)
    pool, ref, table, _ = _layer_case(w, 0, *w.layer_formats[0])
    q = synth.queries(w, 0)
    exp = ref.decode(q, table, w.context_lens)
    for sb in (1152 // bs, 2048 // bs, 1):
        np.testing.assert_allclose(run_gpu_decode(pool, w, q, DEV, split_blocks=sb), exp,
                                   rtol=0, atol=1e-4, err_msg="split_blocks=%d" % sb)
    pool.close()


def test_gqa_ratios_and_head_tiles():
    # MQA (32 Q heads over 1 KV head: four head tiles) and GQA 12:1 (a ragged tile)
    for hq, hkv in ((32, 1), (24, 2), (4, 4)):
        w = synth.workload("gqa_64x2048", S=2, L=130, layers=1)
        w.Hq, w.Hkv = hq, hkv
        w.outlier_channels = w.outlier_channels[w.outlier_channels[:, 0] < hkv]
        fmt, g = kvq.KVQ_INT8_PER_GROUP, 128
        pool, ref, table, _ = _layer_case(w, 0, fmt, g)
        q = synth.queries(w, 0)
        np.testing.assert_allclose(run_gpu_decode(pool, w, q, DEV), ref.decode(q, table, w.context_lens),
                                   rtol=0, atol=TOL, err_msg="Hq=%d Hkv=%d" % (hq, hkv))
        pool.close()


def test_prefix_shared_equals_copied_on_gpu():
    w = synth.workload("mixed_256", S=4, L=100, layers=1)
    w.num_blocks += 3 * (w.shared_prefix_tokens // w.bs)   # room for private prefix copies
    fmt, g = w.layer_formats[0]
    pool, ref, table, (k, v, slots) = _layer_case(w, 0, fmt, g)
    q = synth.queries(w, 0)
    shared = run_gpu_decode(pool, w, q, DEV)
    # copy the 32 shared blocks into fresh blocks for sequences 1..3 and point their tables there
    pblk = w.shared_prefix_tokens // w.bs
    used = set(np.unique(w.block_table).tolist())
    free = [b for b in range(w.num_blocks) if b not in used]
    table2 = w.block_table.copy()
    kk, vv, ss = [k], [v], [slots]
    pre_idx = np.stack([np.zeros(w.shared_prefix_tokens, np.int64), np.arange(w.shared_prefix_tokens)], 1)
    kp, vp = synth.kv_tokens(w, 0, pre_idx)
    for s in range(1, w.S):
        new = np.array(free[:pblk]); free = free[pblk:]
        table2[s, :pblk] = new
        t = np.arange(w.shared_prefix_tokens)
        kk.append(kp); vv.append(vp); ss.append(new[t // w.bs].astype(np.int64) * w.bs + t % w.bs)
    pool.append(torch.from_numpy(np.concatenate(kk[1:])).to(DEV), torch.from_numpy(np.concatenate(vv[1:])).to(DEV),
                torch.from_numpy(np.concatenate(ss[1:])).to(DEV))
    copied = run_gpu_decode(pool, w, q, DEV, table=table2)
    np.testing.assert_array_equal(shared, copied)
    pool.close()


def test_edge_cases_zero_length_and_single_token():
    w = synth.workload("gqa_64x2048", S=4, L=40, layers=1)
    fmt, g = w.layer_formats[0]
    pool, ref, table, _ = _layer_case(w, 0, fmt, g)
    q = synth.queries(w, 0)
    lens = np.array([0, 1, 17, 40], np.int32)
    got = run_gpu_decode(pool, w, q, DEV, lens=lens, max_ctx=40)
    exp = ref.decode(q, table, lens)
    assert not got[0].any()
    np.testing.assert_allclose(got, exp, rtol=0, atol=TOL)
    # L == 1: the output is the dequantized first value, for every head
    np.testing.assert_allclose(got[1], exp[1], rtol=0, atol=1e-5)
    # no sequences / no tokens: no-ops
    kvq.kvq_append(pool.handle, torch.zeros((0, w.Hkv, w.D), dtype=torch.float16, device=DEV),
                   torch.zeros((0, w.Hkv, w.D), dtype=torch.float16, device=DEV),
                   torch.zeros(0, dtype=torch.int64, device=DEV))
    assert pool.error() == kvq.KVQ_OK
    pool.close()


def test_device_range_errors_do_not_fault():
    w = synth.workload("gqa_64x2048", S=3, L=64, layers=1)
    fmt, g = w.layer_formats[0]
    pool, ref, table, _ = _layer_case(w, 0, fmt, g)
    q = synth.queries(w, 0)
    good = run_gpu_decode(pool, w, q, DEV)
    # a slot past the pool end: flagged, skipped, and the valid token still lands
    kk = torch.zeros((2, w.Hkv, w.D), dtype=torch.float16, device=DEV)
    pool.append(kk, kk, torch.tensor([w.num_blocks * w.bs + 3, -1], dtype=torch.int64, device=DEV))
    assert pool.error() == kvq.KVQ_ERR_OUT_OF_RANGE
    assert pool.error() == kvq.KVQ_OK  # cleared by the read
    # a block id outside the pool in sequence 1: flagged; other sequences unaffected
    bad = w.block_table.copy()
    bad[1, 1] = w.num_blocks + 7
    got = run_gpu_decode(pool, w, q, DEV, table=bad)
    assert pool.error() == kvq.KVQ_ERR_OUT_OF_RANGE
    np.testing.assert_array_equal(got[0], good[0])
    np.testing.assert_array_equal(got[2], good[2])
    bad[1, 1] = -5
    run_gpu_decode(pool, w, q, DEV, table=bad)
    assert pool.error() == kvq.KVQ_ERR_OUT_OF_RANGE
    # a context longer than the promised maximum: flagged and clamped
    run_gpu_decode(pool, w, q, DEV, max_ctx=32)
    assert pool.error() == kvq.KVQ_ERR_OUT_OF_RANGE
    # the GPU is still healthy
    np.testing.assert_array_equal(run_gpu_decode(pool, w, q, DEV), good)
    assert pool.error() == kvq.KVQ_OK
    pool.close()


def test_block_size_past_the_shared_memory_stages_is_refused():
    # head_dim 128, FP16 blocks of 64 tokens: two 32 KB stages for each of 4
    # warps exceed the shared memory of a CTA, so the decode refuses before
    # launching anything; INT8 blocks of 64 fit
    big = kvq.KVPool(8, 64, 2, 128, kvq.KVQ_FP16, 0, device=DEV)
    assert kvq.kvq_decode_workspace_bytes(big.handle, 1, 2, 64) == 0
    q = torch.zeros((1, 2, 128), dtype=torch.float16, device=DEV)
    t = torch.zeros((1, 8), dtype=torch.int32, device=DEV)
    ln = torch.ones(1, dtype=torch.int32, device=DEV)
    with pytest.raises(kvq.KVQError) as ei:
        big.decode(q, t, ln, 64)
    assert ei.value.status == kvq.KVQ_ERR_UNSUPPORTED
    big.close()
    ok = kvq.KVPool(8, 64, 2, 128, kvq.KVQ_INT8_PER_GROUP, 128, device=DEV)
    assert kvq.kvq_decode_workspace_bytes(ok.handle, 1, 2, 64) > 0
    ok.close()


def test_host_validation():
    w = synth.workload("gqa_64x2048", S=2, L=64, layers=1)
    pool = kvq.KVPool(w.num_blocks, w.bs, w.Hkv, w.D, kvq.KVQ_INT8_PER_GROUP, 128, device=DEV)
    q = torch.zeros((2, 32, 128), dtype=torch.float16, device=DEV)
    table = torch.from_numpy(w.block_table).to(DEV)
    lens = torch.from_numpy(w.context_lens).to(DEV)
    out = torch.empty((2, 32, 128), dtype=torch.float32, device=DEV)
    with pytest.raises(kvq.KVQError) as e:   # context longer than the table can hold
        kvq.kvq_paged_decode(pool.handle, q, table, lens, w.max_blocks * w.bs + 1, 0.1, out)
    assert e.value.status == kvq.KVQ_ERR_INVALID_ARG
    with pytest.raises(kvq.KVQError) as e:   # Hq not a multiple of Hkv
        kvq.kvq_paged_decode(pool.handle, q[:, :30].contiguous(), table, lens, 64, 0.1, out)
    assert e.value.status == kvq.KVQ_ERR_INVALID_ARG
    need = kvq.kvq_decode_workspace_bytes(pool.handle, 2, 32, 64, split_blocks=1)
    assert need > 0
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_paged_decode(pool.handle, q, table, lens, 64, 0.1, out, None, split_blocks=1)
    assert e.value.status == kvq.KVQ_ERR_WORKSPACE
    with pytest.raises(ValueError):
        kvq.kvq_append(pool.handle, q[:, :8].float(), q[:, :8].float(),
                       torch.zeros(2, dtype=torch.int64, device=DEV))
    pool.close()


@pytest.mark.parametrize("fmt,group", [(kvq.KVQ_INT8_PER_GROUP, 128), (kvq.KVQ_INT8_PER_TOKEN, 0),
                                       (kvq.KVQ_FP16, 0), (kvq.KVQ_INT4_PER_GROUP, 32),
                                       (kvq.KVQ_FP8_E4M3_PER_TOKEN, 0)])
def test_copy_blocks_copy_on_write(fmt, group):
    w = synth.workload("gqa_64x2048", S=3, L=200, layers=1)
    w.layer_formats = [(fmt, group)]
    pool, ref, table, (k, v, slots) = _layer_case(w, 0, fmt, group)
    used = set(np.unique(w.block_table[w.block_table >= 0]).tolist())
    free = np.array([b for b in range(w.num_blocks) if b not in used][:5], np.int32)
    src = w.block_table[1, :5].astype(np.int32)
    q = synth.queries(w, 0)
    before = run_gpu_decode(pool, w, q, DEV)
    kvq.kvq_copy_blocks(pool.handle, torch.from_numpy(src).to(DEV), torch.from_numpy(free).to(DEV))
    assert pool.error() == kvq.KVQ_OK
    # the copies hold exactly the source blocks' codes and scales
    s_slots = (src[:, None].astype(np.int64) * w.bs + np.arange(w.bs)).ravel()
    d_slots = (free[:, None].astype(np.int64) * w.bs + np.arange(w.bs)).ravel()
    cs, ss = pool.read_slots(torch.from_numpy(s_slots).to(DEV))
    cd, sd = pool.read_slots(torch.from_numpy(d_slots).to(DEV))
    np.testing.assert_array_equal(cd.cpu().numpy(), cs.cpu().numpy())
    if ss is not None:
        np.testing.assert_array_equal(sd.cpu().numpy().view(np.uint32), ss.cpu().numpy().view(np.uint32))
    # a table that reads the copies decodes to the same bits
    t2 = w.block_table.copy()
    t2[1, :5] = free
    np.testing.assert_array_equal(run_gpu_decode(pool, w, q, DEV, table=t2), before)
    # out-of-pool ids are flagged and skipped
    bad = torch.tensor([w.num_blocks + 3], dtype=torch.int32, device=DEV)
    kvq.kvq_copy_blocks(pool.handle, bad, torch.tensor([int(free[0])], dtype=torch.int32, device=DEV))
    assert pool.error() == kvq.KVQ_ERR_OUT_OF_RANGE
    pool.close()
