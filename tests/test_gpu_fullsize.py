"""Full-size parity: each decode workload at its full size, one layer (every
layer of a step runs the same launches), through the call the bench times --
kvq_decode_step (append of each sequence's new token, then the decode as a
dependent launch), or kvq_cascade_decode_step for the long shared prefix --
so the persistent grid, the split of the context over warps and the merge
are the ones of the measured runs.  The oracle computes sampled sequences
one by one: their cached tokens are the seeded host draws the oracle also
gets; every other cached token is a device normal draw (it only has to be
there, at its slot, for the launch to be the full one).  Outputs of the
sampled sequences within 1e-3 of the float64 oracle; their new tokens' codes
and scales bit-exact."""
import numpy as np
import pytest
import torch

import paged_quantized_kv_kvq_gb300 as kvq
from paged_quantized_kv_kvq_gb300 import synth
from kvq_testutil import TOL, oracle_layer, oracle_slots

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
CHUNK = 1 << 16


def _t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(DEV)


def _full_pool(w, layer, fmt, group, k, v, slots, calib, with_step=False):
    """Pool with every cached token of the workload (and this step's, with
    with_step): device draws first, then the sampled sequences' host tokens
    over their own slots."""
    pool = kvq.KVPool(w.num_blocks, w.bs, w.Hkv, w.D, fmt, group, device=DEV)
    if fmt == kvq.KVQ_INT8_PER_CHANNEL:
        kvq.kvq_calibrate_channel_scales(pool.handle, _t(calib[0]), _t(calib[1]))
    fs = w.fill_slots()
    fill = _t(np.concatenate([fs, w.step_slots()]) if with_step else fs)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(1000 + layer)
    for a in range(0, fill.numel(), CHUNK):
        b = min(fill.numel(), a + CHUNK)
        kd = torch.randn((b - a, w.Hkv, w.D), generator=gen, device=DEV).half()
        vd = torch.randn((b - a, w.Hkv, w.D), generator=gen, device=DEV).half()
        pool.append(kd, vd, fill[a:b])
    for a in range(0, len(slots), CHUNK):
        b = min(len(slots), a + CHUNK)
        pool.append(_t(k[a:b]), _t(v[a:b]), _t(slots[a:b]))
    return pool


def _sample_tokens(w, layer, seqs):
    """Host K/V and slots of the sampled sequences' cached tokens (shared
    prefix included once) followed by their new tokens at position L-1."""
    idx = w.fill_token_index()
    keep = np.isin(idx[:, 0], seqs)
    if w.shared_prefix_tokens and 0 not in seqs:
        keep |= (idx[:, 0] == 0) & (idx[:, 1] < w.shared_prefix_tokens)
    step_idx = np.stack([np.asarray(seqs, np.int64), w.context_lens[seqs].astype(np.int64) - 1], 1)
    k, v = synth.kv_tokens(w, layer, np.concatenate([idx[keep], step_idx]))
    slots = np.concatenate([w.fill_slots()[keep], w.step_slots()[seqs]])
    return k, v, slots


def _check(name, layer, seqs, fmt=None, group=None, cascade=False, calib_rows=None, **kw):
    """calib_rows: per-channel scales from the first calib_rows sampled tokens
    only (the rest may saturate at +-127), instead of from all of them."""
    w = synth.workload(name, layers=layer + 1, **kw)
    if fmt is None:
        fmt, group = w.layer_formats[layer]
    n = len(seqs)
    k, v, slots = _sample_tokens(w, layer, seqs)
    calib = None
    if fmt == kvq.KVQ_INT8_PER_CHANNEL:
        calib = (k, v) if calib_rows is None else (k[:calib_rows], v[:calib_rows])
    pool = _full_pool(w, layer, fmt, group, k[:-n], v[:-n], slots[:-n], calib)
    # this step's new tokens: device draws, the sampled sequences' from the host
    gen = torch.Generator(device=DEV)
    gen.manual_seed(2000 + layer)
    ks = torch.randn((w.S, w.Hkv, w.D), generator=gen, device=DEV).half()
    vs = torch.randn((w.S, w.Hkv, w.D), generator=gen, device=DEV).half()
    ks[list(seqs)] = _t(k[-n:])
    vs[list(seqs)] = _t(v[-n:])
    q = synth.queries(w, layer)
    table, lens = _t(w.block_table), _t(w.context_lens)
    mc = int(w.context_lens.max())
    out = torch.empty((w.S, w.Hq, w.D), dtype=torch.float32, device=DEV)
    if cascade:
        P = w.shared_prefix_tokens // w.bs
        ws = torch.empty(kvq.kvq_cascade_workspace_bytes(pool.handle, w.S, w.Hq, mc),
                         dtype=torch.uint8, device=DEV)
        kvq.kvq_cascade_decode_step(pool.handle, ks, vs, _t(q), table, lens, mc, P,
                                    w.D ** -0.5, out, ws)
    else:
        pool.decode_step(ks, vs, _t(q), table, lens, mc, out=out)
    torch.cuda.synchronize()
    assert pool.error() == kvq.KVQ_OK
    ref, rtable, remap = oracle_layer(w, fmt, group, k, v, slots, list(seqs), calib=calib)
    # the sampled sequences' new tokens: codes and scales as the oracle's append
    codes, scales = pool.read_slots(_t(slots[-n:]))
    rs = oracle_slots(remap, slots[-n:], w.bs)
    c = codes.cpu().numpy()
    if fmt == kvq.KVQ_FP16:
        np.testing.assert_array_equal(c.astype(np.float32), ref.codes[rs])
    else:
        np.testing.assert_array_equal(c.view(np.uint8), ref.codes[rs].view(np.uint8))
    if scales is not None:
        np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32),
                                      ref.scales[rs].view(np.uint32))
    exp = ref.decode(np.ascontiguousarray(q[list(seqs)]), rtable, w.context_lens[list(seqs)])
    got = out.cpu().numpy()[list(seqs)]
    np.testing.assert_allclose(got, exp, rtol=0, atol=TOL, err_msg="%s layer %d" % (name, layer))
    pool.close()


def test_gqa_64x2048_all_sequences_full():
    # the headline step: every one of the 64 sequences against the oracle, so
    # every unit the grid's warp ranges cut goes through the split merge
    _check("gqa_64x2048", 0, list(range(64)))


@pytest.mark.parametrize("name", ["gqa_64x2048_int4", "gqa_64x2048_e5m2"])
def test_gqa_64x2048_full(name):
    # first, middle and last sequence: the last ends the persistent grid's range
    _check(name, 0, [0, 31, 63])


def test_gqa_64x2048_block8_full():
    # the same batch in 8-token blocks: every tile pairs two pages
    _check("gqa_64x2048", 0, [0, 31, 63], bs=8)


@pytest.mark.parametrize("name", ["mha_100_fp16", "mha_100_fp8", "mha_100_int8ch",
                                  "mha_100_int8g64"])
def test_mha_100_full(name):
    _check(name, 0, [0, 57, 99])


def test_mha_100_int8ch_saturated_full():
    # per-channel scales from the first 64 sampled tokens only: the decode
    # attends codes clipped at +-127 (the append saturates them) at full size
    _check("mha_100_int8ch", 0, [0, 57, 99], calib_rows=64)


@pytest.mark.parametrize("bs", [16, 32])
def test_long_8x32k_full(bs):
    # the last sequence (its 32K-token drift walk is the slow host draw)
    _check("long_8x32k", 0, [7], bs=bs)


@pytest.mark.parametrize("layer", [0, 31])
def test_mixed_256_full(layer):
    # layer 0 INT8 per-group 128, layer 31 FP16; the 512-token prefix is shared
    _check("mixed_256", layer, [0, 128, 255])


def test_shared4k_256_cascade_full():
    _check("shared4k_256", 0, [0, 255], cascade=True)


def test_prefill_8x2048_full():
    """Prompt prefill at the size the bench times: 8 prompts of 2048 tokens of
    the 64x2048 layout (INT8 per-group 128), each whole prompt one chunk, all
    in one kvq_prefill_ex call; sampled query rows of the first and last prompt
    (the first rows, the sub-tile and page edges, the middle and the end),
    each against the oracle's decode over its causal length."""
    w = synth.workload("gqa_64x2048", S=8, layers=1)
    fmt, group = w.layer_formats[0]
    seqs = [0, 7]
    k, v, slots = _sample_tokens(w, 0, seqs)
    pool = _full_pool(w, 0, fmt, group, k, v, slots, None, with_step=True)
    lens = w.context_lens.astype(np.int64)
    qs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(qs[-1])
    gen = torch.Generator(device=DEV)
    gen.manual_seed(3000)
    q = torch.randn((T, w.Hq, w.D), generator=gen, device=DEV).half()
    rng = np.random.default_rng(11)
    qh = {s: rng.standard_normal((int(lens[s]), w.Hq, w.D)).astype(np.float16) for s in seqs}
    for s in seqs:
        q[int(qs[s]):int(qs[s + 1])] = _t(qh[s])
    out = torch.empty((T, w.Hq, w.D), dtype=torch.float32, device=DEV)
    mc = int(lens.max())
    # through kvq_prefill_ex, as the bench times it (key steps staged once)
    ws = torch.empty(kvq.kvq_prefill_workspace_bytes(pool.handle, w.S, mc), dtype=torch.uint8,
                     device=DEV)
    kvq.kvq_prefill_ex(pool.handle, q, _t(qs), mc, _t(w.block_table), _t(w.context_lens), mc,
                       w.D ** -0.5, out, ws)
    torch.cuda.synchronize()
    assert pool.error() == kvq.KVQ_OK
    ref, rtable, _ = oracle_layer(w, fmt, group, k, v, slots, seqs)
    got = out.cpu().numpy()
    for i, s in enumerate(seqs):
        n = int(lens[s])
        rows = np.array([0, 1, 15, 16, 17, 31, 32, 1000, n - 17, n - 2, n - 1])
        exp = ref.decode(np.ascontiguousarray(qh[s][rows]), np.repeat(rtable[i:i + 1], len(rows), 0),
                         (rows + 1).astype(np.int32))
        np.testing.assert_allclose(got[int(qs[s]) + rows], exp, rtol=0, atol=TOL,
                                   err_msg="prompt %d" % s)
    pool.close()
