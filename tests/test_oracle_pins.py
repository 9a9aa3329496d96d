"""Pins for the CPU oracle (no GPU): closed forms, definitions and invariants.

Each test checks the oracle against something other than itself: hand-derived
values from the quantizer's definition, the OCP e4m3 table, a library fp8
cast, dense brute-force attention through scipy's softmax, or an exact
invariance the method must have.  Sources: "KV Cache优化实战：大模型推理显存占用与
加速方案详解" (0539edu.com/news/5800990) §1.1, §1.2, §2.1-§2.3, §3.3.
"""
import json
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from paged_quantized_kv_kvq_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
pytestmark = pytest.mark.usefixtures("oracle_mod")


# ---------------------------------------------------------------- quantizers
def _golden_int8():
    rows = []
    for line in open(os.path.join(GOLDEN, "int8_absmax_cases.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        x, s, c = (p.strip() for p in line.split("|"))
        rows.append((np.array(x.split(), np.float32), np.float32(s),
                     np.array(c.split(), np.int8)))
    return rows


@pytest.mark.parametrize("case", range(len(_golden_int8())))
def test_int8_closed_form(case):
    x, s_exp, c_exp = _golden_int8()[case]
    c, s = oracle.quant_int8_group(x)
    assert s == s_exp
    np.testing.assert_array_equal(c, c_exp)


def test_int8_error_bound_and_range():
    # |x - c*s| <= s/2 for every element of every dynamic-scale group, the
    # absmax element maps to +-127, all codes lie in [-127, 127].
    rng = np.random.default_rng(11)
    for n in (16, 64, 128, 1024):
        for _ in range(50):
            x = (rng.standard_normal(n) * rng.choice([1e-3, 1, 30])).astype(np.float16)
            c, s = oracle.quant_int8_group(x)
            xs = x.astype(np.float64)
            err = np.abs(xs - c.astype(np.float64) * np.float64(s))
            # s/2 from rounding to an integer, plus the fp32 rounding of the
            # quotient x/s (|x/s| <= 127, one half-ulp of 2^-24 relative)
            assert np.all(err <= np.float64(s) * (0.5 + 128 * 2.0 ** -24))
            assert np.abs(c).max() == 127
            assert c[np.argmax(np.abs(xs))] == np.sign(xs[np.argmax(np.abs(xs))]) * 127
            assert s == np.float32(np.float32(np.abs(x).max()) / np.float32(127))


def _golden_int4():
    rows = []
    for line in open(os.path.join(GOLDEN, "int4_absmax_cases.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        x, s, c = (p.strip() for p in line.split("|"))
        rows.append((np.array(x.split(), np.float32), np.float32(s),
                     np.array(c.split(), np.int8)))
    return rows


@pytest.mark.parametrize("case", range(len(_golden_int4())))
def test_int4_closed_form(case):
    x, s_exp, c_exp = _golden_int4()[case]
    c, s = oracle.quant_int4_group(x)
    assert s == s_exp
    np.testing.assert_array_equal(c, c_exp)


def test_int4_error_bound_and_range():
    # |x - c*s| <= s/2, the absmax element maps to +-7, all codes in [-7, 7]
    rng = np.random.default_rng(12)
    for n in (16, 32, 64, 128):
        for _ in range(50):
            x = (rng.standard_normal(n) * rng.choice([1e-3, 1, 30])).astype(np.float16)
            c, s = oracle.quant_int4_group(x)
            xs = x.astype(np.float64)
            err = np.abs(xs - c.astype(np.float64) * np.float64(s))
            assert np.all(err <= np.float64(s) * (0.5 + 8 * 2.0 ** -24))
            assert np.abs(c).max() == 7
            assert c[np.argmax(np.abs(xs))] == np.sign(xs[np.argmax(np.abs(xs))]) * 7
            assert s == np.float32(np.float32(np.abs(x).max()) / np.float32(7))


def test_int8_static_saturates_and_rounds():
    x = np.array([1.0, -1.0, 300.0, -300.0, 2.5, 0.0, 5.0], np.float32)
    s = np.array([1.0, 1.0, 1.0, 1.0, 1.0, 1.0, 0.0], np.float32)
    np.testing.assert_array_equal(oracle.quant_int8_static(x, s), [1, -1, 127, -127, 2, 0, 0])


def test_calibration_closed_form():
    # channel c has absmax 127 * (c + 1) -> scale exactly c + 1
    T, C = 5, 6
    x = np.zeros((T, C), np.float32)
    for c in range(C):
        x[c % T, c] = (-1) ** c * 127.0 * (c + 1)
    np.testing.assert_array_equal(oracle.calibrate_channels(x), np.arange(1, C + 1, dtype=np.float32))


def _golden_e4m3():
    rows = []
    for line in open(os.path.join(GOLDEN, "e4m3_cases.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        v, code = line.split()[:2]
        rows.append((float(v), int(code, 16)))
    return rows


@pytest.mark.parametrize("value,code", _golden_e4m3())
def test_e4m3_golden(value, code):
    assert oracle.e4m3_encode(value) == code


def test_e4m3_exhaustive_roundtrip_and_even_ties():
    finite = [c for c in range(256) if (c & 0x7F) != 0x7F]
    vals = {c: oracle.e4m3_decode(c) for c in finite}
    for c in finite:
        assert oracle.e4m3_encode(vals[c]) == c
    assert np.isnan(oracle.e4m3_decode(0x7F)) and np.isnan(oracle.e4m3_decode(0xFF))
    # every midpoint between neighbouring non-negative codes goes to the even code
    for c in range(0, 0x7E):
        mid = (vals[c] + vals[c + 1]) / 2
        assert np.float32(mid) == mid
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == even
        assert oracle.e4m3_encode(-mid) == even | 0x80


def test_e4m3_matches_torch_cast():
    # library cross-check: torch's CPU float8_e4m3fn cast on in-range values
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(4000) * 50, rng.standard_normal(2000) * 1e-2,
                        rng.uniform(-448, 448, 2000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(v) for v in x], np.uint8)
    np.testing.assert_array_equal(ours, ref)


def _golden_e5m2():
    rows = []
    for line in open(os.path.join(GOLDEN, "e5m2_cases.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        x, c = (p.strip() for p in line.split("|"))
        rows.append((float(x), int(c, 16)))
    return rows


@pytest.mark.parametrize("value,code", _golden_e5m2())
def test_e5m2_golden(value, code):
    assert oracle.e5m2_encode(value) == code


def test_e5m2_exhaustive_roundtrip_and_even_ties():
    finite = [c for c in range(256) if ((c >> 2) & 0x1F) != 0x1F]
    vals = {c: oracle.e5m2_decode(c) for c in finite}
    for c in finite:
        assert oracle.e5m2_encode(vals[c]) == c
    assert np.isinf(oracle.e5m2_decode(0x7C)) and np.isnan(oracle.e5m2_decode(0x7D))
    for c in range(0, 0x7B):
        mid = (vals[c] + vals[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e5m2_encode(mid) == even
        assert oracle.e5m2_encode(-mid) == even | 0x80
    # an e5m2 code is the top byte of the fp16 with the same value
    for c in finite:
        assert np.array([c << 8], np.uint16).view(np.float16)[0] == np.float16(vals[c])


def test_e5m2_matches_torch_cast():
    # library cross-check: torch's CPU float8_e5m2 cast on in-range values
    rng = np.random.default_rng(6)
    x = np.concatenate([rng.standard_normal(4000) * 50, rng.standard_normal(2000) * 1e-3,
                        rng.uniform(-57344, 57344, 2000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    ours = np.array([oracle.e5m2_encode(v) for v in x], np.uint8)
    np.testing.assert_array_equal(ours, ref)


def test_e4m3_group_scale():
    c, s = oracle.quant_e4m3_group(np.array([448, 1, -224, 0.5], np.float32))
    assert s == 1.0
    np.testing.assert_array_equal(c, [0x7E, 0x38, 0xF6, 0x30])
    c, s = oracle.quant_e4m3_group(np.array([896, 2, 34], np.float32))
    assert s == 2.0
    np.testing.assert_array_equal(c, [0x7E, 0x38, 0x58])
    c, s = oracle.quant_e4m3_group(np.zeros(4, np.float32))
    assert s == 0.0 and not c.any()


# ---------------------------------------------------------------- size formula
def test_kv_size_formula_examples():
    spec = json.load(open(os.path.join(GOLDEN, "kv_size_examples.json")))
    for case in spec["cases"]:
        a = case["args"]
        assert oracle.kv_cache_bytes(a["batch"], a["seq_len"], a["layers"], a["kv_heads"],
                                     a["head_dim"], a["precision_bytes"]) == case["bytes"]


@pytest.mark.parametrize("dims", [(1, 1, 1, 1, 8, 1), (2, 3, 4, 2, 16, 2), (3, 17, 2, 8, 64, 1)])
def test_kv_size_formula_brute_force(dims):
    b, L, layers, hkv, d, nbytes = dims
    dt = {1: np.int8, 2: np.float16}[nbytes]
    store = np.zeros((2, b, L, layers, hkv, d), dt)  # one element per cached value
    assert oracle.kv_cache_bytes(b, L, layers, hkv, d, nbytes) == store.nbytes


# ---------------------------------------------------------------- append
FORMATS = [(oracle.INT8_PER_GROUP, 16), (oracle.INT8_PER_GROUP, 32), (oracle.INT8_PER_TOKEN, 0),
           (oracle.INT8_PER_CHANNEL, 0), (oracle.FP8_E4M3_PER_TOKEN, 0), (oracle.FP16, 0),
           (oracle.INT4_PER_GROUP, 16), (oracle.INT4_PER_GROUP, 32), (oracle.FP8_E5M2, 0)]


def _cache(fmt, g, nb=8, bs=4, hkv=2, d=32, **kw):
    return oracle.OracleCache(fmt, nb, bs, hkv, d, g, **kw)


@pytest.mark.parametrize("fmt,g", FORMATS)
def test_append_places_slots_and_keeps_sentinels(fmt, g):
    rng = np.random.default_rng(3)
    c = _cache(fmt, g, sentinel_code=77, sentinel_scale=-5.0)
    k = rng.standard_normal((5, 2, 32)).astype(np.float16)
    v = rng.standard_normal((5, 2, 32)).astype(np.float16)
    if fmt == oracle.INT8_PER_CHANNEL:
        c.calibrate(k, v)
    slots = np.array([9, 0, -1, 31, 17], np.int64)
    c.append(k, v, slots)
    written = {9: 0, 0: 1, 31: 3, 17: 4}
    for slot in range(c.num_slots):
        if slot not in written:
            assert np.all(c.codes[slot] == c.codes.dtype.type(77))
            if c.scales.ndim > 1:
                assert np.all(c.scales[slot] == -5.0)
            continue
        t = written[slot]
        for kv, x in ((0, k), (1, v)):
            if fmt == oracle.FP16:
                np.testing.assert_array_equal(c.codes[slot, kv], x[t].astype(np.float32))
            elif fmt in oracle.GROUP_FORMATS:
                quant = (oracle.quant_int8_group if fmt == oracle.INT8_PER_GROUP
                         else oracle.quant_int4_group)
                for h in range(2):
                    for gi in range(32 // g):
                        cc, s = quant(x[t, h, gi * g:(gi + 1) * g])
                        np.testing.assert_array_equal(c.codes[slot, kv, h, gi * g:(gi + 1) * g], cc)
                        assert c.scales[slot, kv, h, gi] == s
            elif fmt == oracle.INT8_PER_TOKEN:
                cc, s = oracle.quant_int8_group(x[t])
                np.testing.assert_array_equal(c.codes[slot, kv].ravel(), cc)
                assert c.scales[slot, kv] == s
            elif fmt == oracle.FP8_E4M3_PER_TOKEN:
                cc, s = oracle.quant_e4m3_group(x[t])
                np.testing.assert_array_equal(c.codes[slot, kv].ravel(), cc)
                assert c.scales[slot, kv] == s
            elif fmt == oracle.FP8_E5M2:
                cc = [oracle.e5m2_encode(val) for val in x[t].ravel()]
                np.testing.assert_array_equal(c.codes[slot, kv].ravel(), cc)
            else:
                cc = oracle.quant_int8_static(x[t], c.chan_scales[kv])
                np.testing.assert_array_equal(c.codes[slot, kv].ravel(), cc)


def test_append_later_token_wins():
    c = _cache(oracle.INT8_PER_TOKEN, 0)
    k = np.stack([np.full((2, 32), 1.0), np.full((2, 32), -2.0)]).astype(np.float16)
    c.append(k, k, np.array([5, 5]))
    assert c.scales[5, 0] == np.float32(2.0) / np.float32(127)
    assert np.all(c.codes[5, 0] == -127)


def test_per_token_scale_spans_all_heads():
    c = _cache(oracle.INT8_PER_TOKEN, 0)
    k = np.zeros((1, 2, 32), np.float16)
    k[0, 0, 0] = 127.0
    k[0, 1, 5] = 1.0
    c.append(k, k, np.array([3]))
    assert c.scales[3, 0] == 1.0 and c.codes[3, 0, 1, 5] == 1


# ---------------------------------------------------------------- decode
def _filled(fmt, g, S=3, Hq=4, Hkv=2, D=32, bs=4, lens=(5, 1, 11), seed=0, nb=None):
    rng = np.random.default_rng(seed)
    lens = np.array(lens, np.int32)
    nblk = [(L + bs - 1) // bs for L in lens]
    nb = nb or sum(nblk) + 3
    perm = rng.permutation(nb)
    table = np.zeros((S, max(nblk)), np.int32)
    i = 0
    for s in range(S):
        table[s, :nblk[s]] = perm[i:i + nblk[s]]
        i += nblk[s]
    c = oracle.OracleCache(fmt, nb, bs, Hkv, D, g)
    toks = [(s, t) for s in range(S) for t in range(lens[s])]
    k = (rng.standard_normal((len(toks), Hkv, D)) * 2).astype(np.float16)
    v = (rng.standard_normal((len(toks), Hkv, D)) * 2).astype(np.float16)
    if fmt == oracle.INT8_PER_CHANNEL:
        c.calibrate(k, v)
    slots = np.array([table[s, t // bs] * bs + t % bs for s, t in toks], np.int64)
    c.append(k, v, slots)
    q = rng.standard_normal((S, Hq, D)).astype(np.float16)
    return c, q, table, lens


def _dense(c, q, table, lens, sm_scale):
    """Unpaged brute force: gather the dequantized cache into contiguous arrays,
    then softmax(q k^T * scale) v with scipy's softmax."""
    S, Hq, D = q.shape
    G = Hq // c.Hkv
    kd, vd = c.dequantized(0), c.dequantized(1)
    out = np.zeros((S, Hq, D))
    for s in range(S):
        L = int(lens[s])
        if L == 0:
            continue
        slots = np.array([table[s, t // c.bs] * c.bs + t % c.bs for t in range(L)])
        K, V = kd[slots], vd[slots]                       # [L, Hkv, D]
        for hq in range(Hq):
            z = K[:, hq // G] @ q[s, hq].astype(np.float64) * sm_scale
            out[s, hq] = scipy.special.softmax(z) @ V[:, hq // G]
    return out


@pytest.mark.parametrize("fmt,g", FORMATS)
def test_decode_matches_dense_bruteforce(fmt, g):
    c, q, table, lens = _filled(fmt, g)
    for sm in (1 / np.sqrt(32), 0.7):
        got = c.decode(q, table, lens, sm)
        np.testing.assert_allclose(got, _dense(c, q, table, lens, sm), rtol=1e-12, atol=1e-12)


def test_decode_single_token_returns_value():
    c, q, table, lens = _filled(oracle.INT8_PER_GROUP, 16, lens=(1, 1, 1))
    out = c.decode(q, table, lens)
    vd = c.dequantized(1)
    for s in range(3):
        for hq in range(4):
            np.testing.assert_array_equal(out[s, hq], vd[table[s, 0] * 4, hq // 2])


def test_decode_identical_keys_gives_mean_value():
    c = oracle.OracleCache(oracle.INT8_PER_GROUP, 4, 4, 1, 16, 16)
    rng = np.random.default_rng(1)
    k = np.tile(rng.standard_normal((1, 1, 16)), (7, 1, 1)).astype(np.float16)
    v = rng.standard_normal((7, 1, 16)).astype(np.float16)
    table = np.array([[2, 0]], np.int32)
    slots = np.array([table[0, t // 4] * 4 + t % 4 for t in range(7)])
    c.append(k, v, slots)
    out = c.decode(rng.standard_normal((1, 2, 16)).astype(np.float16), table, np.array([7]))
    mean = c.dequantized(1)[slots, 0].mean(0)
    np.testing.assert_allclose(out[0, 0], mean, rtol=0, atol=1e-12)
    np.testing.assert_allclose(out[0, 1], mean, rtol=0, atol=1e-12)


def test_decode_zero_length_is_zero():
    c, q, table, lens = _filled(oracle.INT8_PER_TOKEN, 0, lens=(3, 0, 2))
    assert not c.decode(q, table, lens)[1].any()


def test_decode_invariant_under_block_permutation():
    c, q, table, lens = _filled(oracle.INT8_PER_GROUP, 16, seed=4)
    ref = c.decode(q, table, lens)
    nb = c.num_slots // c.bs
    perm = np.random.default_rng(9).permutation(nb)
    c2 = oracle.OracleCache(c.fmt, nb, c.bs, c.Hkv, c.D, c.g)
    for b in range(nb):   # physical block b moves to perm[b]
        c2.codes[perm[b] * c.bs:(perm[b] + 1) * c.bs] = c.codes[b * c.bs:(b + 1) * c.bs]
        c2.scales[perm[b] * c.bs:(perm[b] + 1) * c.bs] = c.scales[b * c.bs:(b + 1) * c.bs]
    np.testing.assert_array_equal(c2.decode(q, perm[table].astype(np.int32), lens), ref)


def test_decode_prefix_shared_equals_copied():
    rng = np.random.default_rng(2)
    bs, D, nb = 4, 16, 16
    pre = 8   # two shared blocks
    lens = np.array([11, 14], np.int32)
    shared = oracle.OracleCache(oracle.INT8_PER_GROUP, nb, bs, 1, D, 16)
    copied = oracle.OracleCache(oracle.INT8_PER_GROUP, nb, bs, 1, D, 16)
    t_sh = np.array([[0, 1, 2, 3], [0, 1, 4, 5]], np.int32)
    t_cp = np.array([[0, 1, 2, 3], [6, 7, 4, 5]], np.int32)
    kp, vp = (rng.standard_normal((2, pre, 1, D)).astype(np.float16))
    for cache, table in ((shared, t_sh), (copied, t_cp)):
        for s in range(2):
            if cache is shared and s == 1:
                start = pre
            else:
                start = 0
            toks = range(start, lens[s])
            r = np.random.default_rng(100 + s)
            ks = r.standard_normal((lens[s], 1, D)).astype(np.float16)
            vs = r.standard_normal((lens[s], 1, D)).astype(np.float16)
            ks[:pre], vs[:pre] = kp, vp
            slots = np.array([table[s, t // bs] * bs + t % bs for t in toks])
            cache.append(ks[start:], vs[start:], slots)
    q = rng.standard_normal((2, 2, D)).astype(np.float16)
    np.testing.assert_array_equal(shared.decode(q, t_sh, lens), copied.decode(q, t_cp, lens))


def test_decode_gqa_equals_mha_with_replicated_heads():
    rng = np.random.default_rng(8)
    bs, D, Hq = 4, 16, 4
    lens = np.array([9], np.int32)
    table = np.array([[1, 0, 2]], np.int32)
    slots = np.array([table[0, t // bs] * bs + t % bs for t in range(9)])
    k = rng.standard_normal((9, 1, D)).astype(np.float16)
    v = rng.standard_normal((9, 1, D)).astype(np.float16)
    q = rng.standard_normal((1, Hq, D)).astype(np.float16)
    gqa = oracle.OracleCache(oracle.INT8_PER_GROUP, 3, bs, 1, D, 16)
    gqa.append(k, v, slots)
    mha = oracle.OracleCache(oracle.INT8_PER_GROUP, 3, bs, Hq, D, 16)
    mha.append(np.repeat(k, Hq, 1), np.repeat(v, Hq, 1), slots)
    np.testing.assert_array_equal(gqa.decode(q, table, lens), mha.decode(q, table, lens))


def test_fp16_layer_equals_plain_attention():
    c, q, table, lens = _filled(oracle.FP16, 0, seed=6)
    rng = np.random.default_rng(6)
    got = c.decode(q, table, lens)
    # plain attention on the raw fp16 values, torch CPU float64
    for s in range(3):
        L = lens[s]
        slots = [table[s, t // 4] * 4 + t % 4 for t in range(L)]
        K = torch.from_numpy(c.codes[slots, 0].astype(np.float64))
        V = torch.from_numpy(c.codes[slots, 1].astype(np.float64))
        for hq in range(4):
            qq = torch.from_numpy(q[s, hq].astype(np.float64))
            ref = torch.softmax(K[:, hq // 2] @ qq / np.sqrt(32), 0) @ V[:, hq // 2]
            np.testing.assert_allclose(got[s, hq], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_copy_blocks_then_remap_gives_identical_decode():
    # copy-on-write: after copying blocks, a table that reads the copies gives
    # the same output bit for bit, and the copies hold the source's codes
    c, q, table, lens = _filled(oracle.INT8_PER_GROUP, 16, seed=9, nb=40)
    used = set(np.unique(table).tolist())
    free = [b for b in range(c.num_slots // c.bs) if b not in used][:3]
    src = table[2, :3].copy()
    before = c.decode(q, table, lens)
    c.copy_blocks(src, free)
    for s, d in zip(src, free):
        np.testing.assert_array_equal(c.codes[d * c.bs:(d + 1) * c.bs], c.codes[s * c.bs:(s + 1) * c.bs])
        np.testing.assert_array_equal(c.scales[d * c.bs:(d + 1) * c.bs], c.scales[s * c.bs:(s + 1) * c.bs])
    t2 = table.copy()
    t2[2, :3] = free
    np.testing.assert_array_equal(c.decode(q, t2, lens), before)


def test_half_to_float_is_exact_on_every_code(oracle_mod):
    """The oracle's binary16 widening against numpy's on all 65536 codes:
    every finite value and infinity bit for bit, NaNs as NaN with the sign."""
    h = np.arange(1 << 16, dtype=np.uint16).view(np.float16)
    got = oracle_mod.half_to_float(h)
    ref = h.astype(np.float32)
    fin = ~np.isnan(ref)
    np.testing.assert_array_equal(got[fin].view(np.uint32), ref[fin].view(np.uint32))
    assert np.isnan(got[~fin]).all()
    np.testing.assert_array_equal(np.signbit(got[~fin]), np.signbit(ref[~fin]))
    # the extremes by hand: the smallest subnormal, the largest finite value
    assert oracle_mod.half_to_float(np.array([0x0001], np.uint16).view(np.float16))[0] == 2.0 ** -24
    assert oracle_mod.half_to_float(np.array([0x7BFF], np.uint16).view(np.float16))[0] == 65504.0
