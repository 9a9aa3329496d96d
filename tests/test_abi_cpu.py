"""Host-only checks of the C ABI (no GPU): the library builds and loads, it
exports every function include/kvq.h declares, and its byte accounting follows
the KV-size formula of "KV Cache优化实战" §1.2
(2 x tokens x layers x kv_heads x head_dim x bytes)."""
import ctypes

import pytest

import oracle
import paged_quantized_kv_kvq_gb300 as kvq
from paged_quantized_kv_kvq_gb300 import build as kbuild


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return kvq.lib()


def test_exports_every_declared_symbol(L):
    names = kvq.header_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(L, n), n
        assert isinstance(getattr(L, n), ctypes._CFuncPtr)


def test_phase_event_argument_checks(L):
    """kvq_set_phase_events only stores handles (no CUDA call): its range and
    NULL checks run without a GPU, and n = 0 clears whatever was set."""
    arr = (ctypes.c_void_p * 9)()
    assert L.kvq_set_phase_events(None, 0) == kvq.KVQ_OK
    assert L.kvq_set_phase_events(None, 1) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_set_phase_events(arr, -1) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_set_phase_events(arr, 9) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_set_phase_events(arr, 8) == kvq.KVQ_OK
    assert L.kvq_set_phase_events(None, 0) == kvq.KVQ_OK
    class Ev:  # stands in for a torch.cuda.Event whose CUDA event exists
        cuda_event = 1

    with pytest.raises(kvq.KVQError):
        kvq.kvq_set_phase_events([Ev()] * 9)
    kvq.kvq_set_phase_events([])


def test_status_strings(L):
    for st in range(7):
        assert kvq.kvq_status_string(st)
    assert kvq.kvq_status_string(99) == "unknown status"


# bytes per element, in halves (INT4 stores two codes per byte)
HALF_BYTES = {kvq.KVQ_FP16: 4, kvq.KVQ_INT8_PER_TOKEN: 2, kvq.KVQ_INT8_PER_CHANNEL: 2,
              kvq.KVQ_INT8_PER_GROUP: 2, kvq.KVQ_FP8_E4M3_PER_TOKEN: 2, kvq.KVQ_INT4_PER_GROUP: 1,
              kvq.KVQ_FP8_E5M2: 2}


@pytest.mark.parametrize("dtype,group", [(kvq.KVQ_FP16, 0), (kvq.KVQ_INT8_PER_TOKEN, 0),
                                         (kvq.KVQ_INT8_PER_CHANNEL, 0), (kvq.KVQ_INT8_PER_GROUP, 128),
                                         (kvq.KVQ_INT8_PER_GROUP, 64), (kvq.KVQ_FP8_E4M3_PER_TOKEN, 0),
                                         (kvq.KVQ_INT4_PER_GROUP, 128), (kvq.KVQ_INT4_PER_GROUP, 32),
                                         (kvq.KVQ_FP8_E5M2, 0)])
@pytest.mark.parametrize("nb,bs,hkv,d", [(9103, 16, 8, 128), (64, 16, 1, 64), (100, 32, 32, 128),
                                         (300, 8, 8, 128), (17, 8, 2, 64)])
def test_code_bytes_follow_formula(L, dtype, group, nb, bs, hkv, d):
    if dtype in kvq.GROUP_FORMATS and d % group:
        group = d
    if bs == 8 and dtype == kvq.KVQ_INT4_PER_GROUP:
        pytest.skip("INT4 takes block sizes that are multiples of 16")
    lay = kvq.kvq_pool_layout_query(nb, bs, hkv, d, dtype, group)
    tokens = nb * bs  # whole blocks
    # the size formula with the element size in half bytes, halved
    assert lay["code_bytes"] == oracle.kv_cache_bytes(1, tokens, 1, hkv, d, HALF_BYTES[dtype]) // 2
    exp_scales = {kvq.KVQ_FP16: 0, kvq.KVQ_INT8_PER_TOKEN: tokens * 2 * 4,
                  kvq.KVQ_FP8_E4M3_PER_TOKEN: tokens * 2 * 4,
                  kvq.KVQ_INT8_PER_CHANNEL: 2 * hkv * d * 4,
                  kvq.KVQ_INT8_PER_GROUP: tokens * 2 * hkv * (d // max(group, 1)) * 4,
                  kvq.KVQ_INT4_PER_GROUP: tokens * 2 * hkv * (d // max(group, 1)) * 4,
                  kvq.KVQ_FP8_E5M2: 0}[dtype]
    assert lay["scale_bytes"] == exp_scales
    assert lay["total_bytes"] == kvq.kvq_pool_bytes(nb, bs, hkv, d, dtype, group)
    assert lay["total_bytes"] >= lay["code_bytes"] + lay["scale_bytes"]
    assert lay["header_bytes"] < 1024
    assert lay["total_bytes"] % 256 == 0


def test_layer_stack_matches_formula(L):
    # 32 layers, 64 sequences x 2048 tokens, 8 KV heads, head_dim 128, INT8:
    # the code bytes of 32 per-layer pools sized exactly for the tokens equal
    # the formula with layers = 32.
    per_layer = kvq.kvq_pool_layout_query(64 * 2048 // 16, 16, 8, 128, kvq.KVQ_INT8_PER_GROUP, 128)
    assert 32 * per_layer["code_bytes"] == oracle.kv_cache_bytes(64, 2048, 32, 8, 128, 1)


@pytest.mark.parametrize("args,status", [
    ((0, 16, 8, 128, kvq.KVQ_INT8_PER_GROUP, 128), kvq.KVQ_ERR_INVALID_ARG),
    ((8, 16, 8, 100, kvq.KVQ_INT8_PER_GROUP, 128), kvq.KVQ_ERR_INVALID_ARG),
    ((8, 16, 8, 128, kvq.KVQ_INT8_PER_GROUP, 48), kvq.KVQ_ERR_INVALID_ARG),
    ((8, 16, 8, 128, kvq.KVQ_INT8_PER_GROUP, 8), kvq.KVQ_ERR_UNSUPPORTED),
    ((8, 24, 8, 128, kvq.KVQ_INT8_PER_GROUP, 128), kvq.KVQ_ERR_UNSUPPORTED),
    ((8, 48, 8, 128, kvq.KVQ_INT8_PER_GROUP, 128), kvq.KVQ_ERR_UNSUPPORTED),
    ((8, 96, 8, 128, kvq.KVQ_INT8_PER_GROUP, 128), kvq.KVQ_ERR_UNSUPPORTED),
    ((8, 128, 8, 64, kvq.KVQ_FP16, 0), kvq.KVQ_ERR_UNSUPPORTED),
    ((8, 4, 8, 128, kvq.KVQ_INT8_PER_GROUP, 128), kvq.KVQ_ERR_UNSUPPORTED),
    ((8, 8, 8, 128, kvq.KVQ_INT4_PER_GROUP, 128), kvq.KVQ_ERR_UNSUPPORTED),
    ((8, 16, 8, 256, kvq.KVQ_FP16, 0), kvq.KVQ_ERR_UNSUPPORTED),
    ((8, 16, 8, 128, 9, 0), kvq.KVQ_ERR_INVALID_ARG),
])
def test_layout_refusals(L, args, status):
    with pytest.raises(kvq.KVQError) as ei:
        kvq.kvq_pool_layout_query(*args)
    assert ei.value.status == status
    assert kvq.kvq_pool_bytes(*args) == 0


def test_null_handles_are_refused(L):
    assert L.kvq_free_pool(None) == kvq.KVQ_OK
    assert L.kvq_append(None, None, None, None, 1, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_get_error(None, None) == kvq.KVQ_ERR_INVALID_ARG
    assert L.kvq_decode_workspace_bytes(None, 1, 1, 1) == 0
    out = ctypes.c_void_p()
    assert L.kvq_alloc_pool(0, 16, 1, 64, 3, 64, None, 0, ctypes.byref(out)) == kvq.KVQ_ERR_INVALID_ARG
