"""GPU parity of kvq_decode_step (append of each sequence's new token at
position L-1, slot taken from the block table, then decode as a programmatic
dependent launch): codes of the new tokens bit-exact against the oracle's
append, outputs within 1e-3 of the float64 oracle, and identical to the two
separate calls kvq_append + kvq_paged_decode."""
import numpy as np
import pytest
import torch

import oracle
import paged_quantized_kv_kvq_gb300 as kvq
from paged_quantized_kv_kvq_gb300 import synth
from kvq_testutil import TOL, gpu_pool, layer_tokens, oracle_layer, oracle_slots

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def _step_case(name, fmt, group, **kw):
    w = synth.workload(name, layers=1, **kw)
    w.layer_formats = [(fmt, group)]
    k, v, slots = layer_tokens(w, 0)
    S = w.S
    calib = (k, v) if fmt == kvq.KVQ_INT8_PER_CHANNEL else None
    # the cache before the step: every token but the last S (this step's)
    pool = gpu_pool(w, fmt, group, DEV, k[:-S], v[:-S], slots[:-S], calib=calib)
    ref, table, remap = oracle_layer(w, fmt, group, k, v, slots, list(range(S)), calib=calib)
    q = synth.queries(w, 0)
    out = pool.decode_step(_t(k[-S:]), _t(v[-S:]), _t(q), _t(w.block_table), _t(w.context_lens),
                           int(w.context_lens.max()))
    torch.cuda.synchronize()
    assert pool.error() == kvq.KVQ_OK
    got = out.cpu().numpy()
    # the new tokens landed where the block table says, with the oracle's codes
    step = slots[-S:]
    codes, scales = pool.read_slots(_t(step))
    rs = oracle_slots(remap, step, w.bs)
    c = codes.cpu().numpy()
    if fmt == kvq.KVQ_FP16:
        np.testing.assert_array_equal(c.astype(np.float32), ref.codes[rs])
    else:
        np.testing.assert_array_equal(c.view(np.uint8), ref.codes[rs].view(np.uint8))
    if scales is not None:
        np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32),
                                      ref.scales[rs].view(np.uint32))
    exp = ref.decode(q, table, w.context_lens)
    np.testing.assert_allclose(got, exp, rtol=0, atol=TOL)
    return w, pool, (k, v, slots), q, got


@pytest.mark.parametrize("fmt,group", [(kvq.KVQ_INT8_PER_GROUP, 128), (kvq.KVQ_INT8_PER_GROUP, 32),
                                       (kvq.KVQ_INT8_PER_TOKEN, 0), (kvq.KVQ_INT8_PER_CHANNEL, 0),
                                       (kvq.KVQ_FP8_E4M3_PER_TOKEN, 0), (kvq.KVQ_FP16, 0),
                                       (kvq.KVQ_INT4_PER_GROUP, 128), (kvq.KVQ_FP8_E5M2, 0)])
def test_decode_step_parity(fmt, group):
    w, pool, (k, v, slots), q, got = _step_case("gqa_64x2048", fmt, group, S=5, L=333)
    # the same step as two separate calls on a second pool gives the same bits
    calib = (k, v) if fmt == kvq.KVQ_INT8_PER_CHANNEL else None
    pool2 = gpu_pool(w, fmt, group, DEV, k, v, slots, calib=calib)
    sep = pool2.decode(_t(q), _t(w.block_table), _t(w.context_lens), int(w.context_lens.max()))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(sep.cpu().numpy(), got)
    pool.close()
    pool2.close()


@pytest.mark.parametrize("name,kw", [("long_8x32k", dict(S=2, L=2000, bs=32)),
                                     ("mha_100_int8g64", dict(S=7, L=150)),
                                     ("tiny", dict())])
def test_decode_step_workloads(name, kw):
    w0 = synth.workload(name, layers=1, **kw)
    fmt, group = w0.layer_formats[0]
    _, pool, _, _, _ = _step_case(name, fmt, group, **kw)
    pool.close()


@pytest.mark.parametrize("hq,hkv", [(32, 1), (24, 2), (8, 1), (4, 4)])
def test_decode_step_head_tiles(hq, hkv):
    # MQA with four head tiles of 8, GQA 12:1 (a ragged tile), 8:1 (one full
    # tile) and MHA, with the per-token format whose scale spans every kv head
    # of the token: the oracle's codes and the separate calls' bits.
    w = synth.workload("gqa_64x2048", S=3, L=130, layers=1)
    w.Hq, w.Hkv = hq, hkv
    w.outlier_channels = w.outlier_channels[w.outlier_channels[:, 0] < hkv]
    fmt, group = kvq.KVQ_INT8_PER_TOKEN, 0
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
    codes, scales = pool.read_slots(_t(slots[-S:]))
    rs = oracle_slots(remap, slots[-S:], w.bs)
    np.testing.assert_array_equal(codes.cpu().numpy().view(np.uint8), ref.codes[rs].view(np.uint8))
    np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32), ref.scales[rs].view(np.uint32))
    got = out.cpu().numpy()
    np.testing.assert_allclose(got, ref.decode(q, table, w.context_lens), rtol=0, atol=TOL)
    pool2 = gpu_pool(w, fmt, group, DEV, k, v, slots)
    sep = pool2.decode(_t(q), _t(w.block_table), _t(w.context_lens), int(w.context_lens.max()))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(sep.cpu().numpy(), got)
    pool.close()
    pool2.close()


def test_decode_step_edges():
    """L == 0 stores nothing and outputs zeros; L > max_context_len stores
    nothing and is flagged; an unmapped block at L-1 is flagged, not written."""
    w = synth.workload("gqa_64x2048", S=3, L=48, layers=1)
    fmt, g = w.layer_formats[0]
    k, v, slots = layer_tokens(w, 0)
    pool = kvq.KVPool(w.num_blocks, w.bs, w.Hkv, w.D, fmt, g, device=DEV, fill_byte=0x5A)
    kn = _t(k[-3:])
    vn = _t(v[-3:])
    q = _t(synth.queries(w, 0))
    table = _t(w.block_table)
    everything = _t(np.arange(w.num_blocks * w.bs, dtype=np.int64))
    before = pool.read_slots(everything)[0].cpu().numpy()
    lens = _t(np.array([0, 0, 0], np.int32))
    out = pool.decode_step(kn, vn, q, table, lens, 48)
    torch.cuda.synchronize()
    assert pool.error() == kvq.KVQ_OK
    assert not out.cpu().numpy().any()
    np.testing.assert_array_equal(pool.read_slots(everything)[0].cpu().numpy(), before)
    # a length past the promised maximum: flagged, nothing stored
    pool.decode_step(kn, vn, q, table, _t(np.array([0, 40, 0], np.int32)), 32)
    assert pool.error() == kvq.KVQ_ERR_OUT_OF_RANGE
    np.testing.assert_array_equal(pool.read_slots(everything)[0].cpu().numpy(), before)
    # position L-1 in an unmapped block: flagged, nothing stored
    bad = w.block_table.copy()
    bad[2, 0] = -1
    pool.decode_step(kn, vn, q, _t(bad), _t(np.array([0, 0, 5], np.int32)), 48)
    assert pool.error() == kvq.KVQ_ERR_OUT_OF_RANGE
    np.testing.assert_array_equal(pool.read_slots(everything)[0].cpu().numpy(), before)
    # host-side checks
    with pytest.raises(ValueError):
        pool.decode_step(kn[:2], vn[:2], q, table, lens, 48)
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_decode_step(pool.handle, kn, vn, q, table, lens, w.max_blocks * w.bs + 1, 0.1,
                            torch.empty((3, 32, 128), dtype=torch.float32, device=DEV))
    assert e.value.status == kvq.KVQ_ERR_INVALID_ARG
    pool.close()


@pytest.fixture(scope="module")
def late_writer(tmp_path_factory):
    """ctypes handle of tests/late_writer.cu, compiled for this GPU."""
    import ctypes
    import os
    import shutil
    import subprocess

    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "late_writer.cu")
    so = str(tmp_path_factory.mktemp("late_writer") / "late_writer.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
                    "-Xcompiler", "-fPIC", "-o", so, src], check=True)
    lib = ctypes.CDLL(so)
    lib.late_write.restype = ctypes.c_int
    lib.late_write.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                               ctypes.c_ulonglong, ctypes.c_void_p]
    return lib


def test_decode_step_after_late_length_writer(late_writer):
    """The kernel just before the step lets its dependents launch early and
    writes this step's context lengths ~0.2 ms later.  The step must use the
    written lengths: its append waits for that kernel, and the decode launches
    only once the append has passed that wait."""
    w = synth.workload("gqa_64x2048", S=5, L=333, layers=1)
    fmt, group = w.layer_formats[0]
    k, v, slots = layer_tokens(w, 0)
    S = w.S
    pool = gpu_pool(w, fmt, group, DEV, k[:-S], v[:-S], slots[:-S])
    ref, table, remap = oracle_layer(w, fmt, group, k, v, slots, list(range(S)))
    q = synth.queries(w, 0)
    lens = _t(np.ones(S, np.int32))            # stale lengths, overwritten late
    truth = _t(w.context_lens)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        lens.fill_(1)
        torch.cuda.synchronize()
        assert late_writer.late_write(lens.data_ptr(), truth.data_ptr(), S, 200000,
                                      stream.cuda_stream) == 0
        out = pool.decode_step(_t(k[-S:]), _t(v[-S:]), _t(q), _t(w.block_table), lens,
                               int(w.context_lens.max()))
        torch.cuda.synchronize()
        assert pool.error() == kvq.KVQ_OK
        np.testing.assert_allclose(out.cpu().numpy(), ref.decode(q, table, w.context_lens),
                                   rtol=0, atol=TOL)
    codes, _ = pool.read_slots(_t(slots[-S:]))
    rs = oracle_slots(remap, slots[-S:], w.bs)
    np.testing.assert_array_equal(codes.cpu().numpy().view(np.uint8), ref.codes[rs].view(np.uint8))
    pool.close()
