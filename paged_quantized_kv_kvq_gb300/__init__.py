"""Python binding of the paged quantized KV-cache library (libkvq.so, sm_103a).

Thin argument marshalling over the C ABI declared in ``include/kvq.h``: every
function below has the C function's name, checks dtypes/devices of the torch
tensors it is given, and passes raw device pointers, sizes and the current
CUDA stream.  All computation happens in the CUDA kernels of libkvq.so; there
is no CPU fallback, and importing a function whose library is missing raises.

Method: decode-step attention over a block-paged KV cache stored as INT8/FP8
codes with per-token, per-channel or per-group fp32 scales, or FP16
("KV Cache优化实战：大模型推理显存占用与加速方案详解", 0539edu.com/news/5800990,
§1.1, §2.1-§2.3, §3.3, §4.3).
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "kvq.h")

# kvq_dtype
KVQ_FP16 = 0
KVQ_INT8_PER_TOKEN = 1
KVQ_INT8_PER_CHANNEL = 2
KVQ_INT8_PER_GROUP = 3
KVQ_FP8_E4M3_PER_TOKEN = 4
KVQ_INT4_PER_GROUP = 5
KVQ_FP8_E5M2 = 6
GROUP_FORMATS = (KVQ_INT8_PER_GROUP, KVQ_INT4_PER_GROUP)

# kvq_status
KVQ_OK = 0
KVQ_ERR_INVALID_ARG = 1
KVQ_ERR_UNSUPPORTED = 2
KVQ_ERR_CUDA = 3
KVQ_ERR_OUT_OF_RANGE = 4
KVQ_ERR_WORKSPACE = 5
KVQ_ERR_TIMEOUT = 6

_lock = threading.Lock()
_lib = None


class KVQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, kvq_status_string(status), status))


class _Layout(ctypes.Structure):
    _fields_ = [("total_bytes", ctypes.c_size_t), ("code_bytes", ctypes.c_size_t),
                ("scale_bytes", ctypes.c_size_t), ("header_bytes", ctypes.c_size_t),
                ("page_bytes", ctypes.c_size_t)]


def header_functions() -> list[str]:
    """Names of the functions include/kvq.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", text)))


def lib() -> ctypes.CDLL:
    """The loaded libkvq.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libkvq.so is not built (run __graft_entry__.build() or "
                                   "python -m paged_quantized_kv_kvq_gb300.build)")
            L = ctypes.CDLL(LIB_PATH)
            _declare(L)
            _lib = L
        return _lib


def _declare(L):
    P, i32, i64, sz, f32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                            ctypes.c_float)
    sigs = {
        "kvq_pool_layout_query": (i32, [i64, i32, i32, i32, i32, i32, ctypes.POINTER(_Layout)]),
        "kvq_pool_bytes": (sz, [i64, i32, i32, i32, i32, i32]),
        "kvq_alloc_pool": (i32, [i64, i32, i32, i32, i32, i32, P, sz, ctypes.POINTER(P)]),
        "kvq_free_pool": (i32, [P]),
        "kvq_set_channel_scales": (i32, [P, P, P, P]),
        "kvq_calibrate_channel_scales": (i32, [P, P, P, i64, P]),
        "kvq_append": (i32, [P, P, P, P, i64, P]),
        "kvq_copy_blocks": (i32, [P, P, P, i32, P]),
        "kvq_append_strided": (i32, [P, P, P, i64, P, i64, P]),
        "kvq_paged_decode_strided": (i32, [P, P, i64, i32, i32, P, i32, P, i32, f32, P, i64, P, sz,
                                           P]),
        "kvq_decode_workspace_bytes": (sz, [P, i32, i32, i32]),
        "kvq_decode_workspace_bytes_ex": (sz, [P, i32, i32, i32, i32]),
        "kvq_paged_decode": (i32, [P, P, i32, i32, P, i32, P, i32, f32, P, P, sz, P]),
        "kvq_paged_decode_ex": (i32, [P, P, i32, i32, P, i32, P, i32, f32, P, P, sz, i32, P]),
        "kvq_paged_decode_noalloc": (i32, [P, P, i32, i32, P, i32, P, i32, f32, P, i32, P]),
        "kvq_decode_step": (i32, [P, P, P, P, i32, i32, P, i32, P, i32, f32, P, P, sz, P]),
        "kvq_cascade_workspace_bytes": (sz, [P, i32, i32, i32]),
        "kvq_prefill": (i32, [P, P, i32, i32, P, i32, P, i32, P, i32, f32, P, P]),
        "kvq_prefill_workspace_bytes": (sz, [P, i32, i32]),
        "kvq_prefill_ex": (i32, [P, P, i32, i32, P, i32, P, i32, P, i32, f32, P, P, sz, P]),
        "kvq_selftest_decode_timeout": (i32, [P, P, i32, i32, P, i32, P, i32, P, P, sz, i32, P]),
        "kvq_cascade_decode": (i32, [P, P, i32, i32, P, i32, P, i32, i32, f32, P, P, sz, P]),
        "kvq_cascade_decode_step": (i32, [P, P, P, P, i32, i32, P, i32, P, i32, i32, f32, P, P, sz,
                                          P]),
        "kvq_read_slots": (i32, [P, P, i64, P, P, P]),
        "kvq_get_error": (i32, [P, P]),
        "kvq_status_string": (ctypes.c_char_p, [i32]),
        "kvq_set_phase_events": (i32, [P, i32]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args


def _check(st: int, where: str) -> None:
    if st != KVQ_OK:
        raise KVQError(st, where)


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


# ------------------------------------------------------------------ C ABI
def kvq_status_string(status: int) -> str:
    return lib().kvq_status_string(int(status)).decode()


def kvq_pool_layout_query(num_blocks, block_size, kv_heads, head_dim, dtype, group=0) -> dict:
    lay = _Layout()
    _check(lib().kvq_pool_layout_query(num_blocks, block_size, kv_heads, head_dim, dtype, group,
                                       ctypes.byref(lay)), "kvq_pool_layout_query")
    return {f: int(getattr(lay, f)) for f, _ in _Layout._fields_}


def kvq_pool_bytes(num_blocks, block_size, kv_heads, head_dim, dtype, group=0) -> int:
    return int(lib().kvq_pool_bytes(num_blocks, block_size, kv_heads, head_dim, dtype, group))


def kvq_alloc_pool(num_blocks, block_size, kv_heads, head_dim, dtype, group=0, device_buf=None):
    """Returns an opaque handle (ctypes.c_void_p).  device_buf: optional torch
    uint8 CUDA tensor of at least kvq_pool_bytes(..) bytes, owned by the caller."""
    h = ctypes.c_void_p()
    ptr = _ptr(device_buf, name="device_buf") if device_buf is not None else None
    nbytes = device_buf.numel() * device_buf.element_size() if device_buf is not None else 0
    _check(lib().kvq_alloc_pool(num_blocks, block_size, kv_heads, head_dim, dtype, group, ptr,
                                nbytes, ctypes.byref(h)), "kvq_alloc_pool")
    return h


def kvq_free_pool(pool) -> None:
    _check(lib().kvq_free_pool(pool), "kvq_free_pool")


def kvq_set_channel_scales(pool, k_scale, v_scale, stream=None) -> None:
    import torch

    _check(lib().kvq_set_channel_scales(pool, _ptr(k_scale, torch.float32, "k_scale"),
                                        _ptr(v_scale, torch.float32, "v_scale"), _stream(stream)),
           "kvq_set_channel_scales")


def kvq_calibrate_channel_scales(pool, k, v, stream=None) -> None:
    import torch

    _check(lib().kvq_calibrate_channel_scales(pool, _ptr(k, torch.float16, "k"),
                                              _ptr(v, torch.float16, "v"), k.shape[0],
                                              _stream(stream)), "kvq_calibrate_channel_scales")


def kvq_append(pool, k, v, slot_mapping, stream=None) -> None:
    import torch

    if k.shape != v.shape or k.shape[0] != slot_mapping.numel():
        raise ValueError("k, v must be [T, kv_heads, head_dim] and slot_mapping [T]")
    _check(lib().kvq_append(pool, _ptr(k, torch.float16, "k"), _ptr(v, torch.float16, "v"),
                            _ptr(slot_mapping, torch.int64, "slot_mapping"), k.shape[0],
                            _stream(stream)), "kvq_append")


def _rows_view(t, dtype, name):
    """Pointer and row stride (elements) of a [rows, heads, head_dim] view whose
    heads and channels are contiguous (a head slice of wider rows)."""
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError("%s must be [rows, heads, head_dim] with contiguous heads" % name)
    return ctypes.c_void_p(t.data_ptr()), int(t.stride(0))


def kvq_append_strided(pool, k, v, slot_mapping, stream=None) -> None:
    """kvq_append for head slices of wider token rows (per-head mixed precision)."""
    import torch

    kp, ks = _rows_view(k, torch.float16, "k")
    vp, vs = _rows_view(v, torch.float16, "v")
    if ks != vs or k.shape != v.shape or k.shape[0] != slot_mapping.numel():
        raise ValueError("k and v must be equal-shaped views with the same row stride")
    _check(lib().kvq_append_strided(pool, kp, vp, ks, _ptr(slot_mapping, torch.int64, "slot_mapping"),
                                    k.shape[0], _stream(stream)), "kvq_append_strided")


def kvq_paged_decode_strided(pool, q, block_table, context_lens, max_context_len, sm_scale, out,
                             workspace=None, stream=None) -> None:
    """kvq_paged_decode for head slices of wider q / out rows (per-head mixed precision)."""
    import torch

    qp, qs = _rows_view(q, torch.float16, "q")
    op, os_ = _rows_view(out, torch.float32, "out")
    S, Hq, _ = q.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().kvq_paged_decode_strided(
        pool, qp, qs, S, Hq, _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
        _ptr(context_lens, torch.int32, "context_lens"), int(max_context_len), float(sm_scale),
        op, os_, _ptr(workspace, None, "workspace") if workspace is not None else None, ws_bytes,
        _stream(stream)), "kvq_paged_decode_strided")


def kvq_copy_blocks(pool, src_blocks, dst_blocks, stream=None) -> None:
    """Block dst_blocks[i] becomes a copy of block src_blocks[i] (copy-on-write)."""
    import torch

    if src_blocks.numel() != dst_blocks.numel():
        raise ValueError("src_blocks and dst_blocks must have the same length")
    _check(lib().kvq_copy_blocks(pool, _ptr(src_blocks, torch.int32, "src_blocks"),
                                 _ptr(dst_blocks, torch.int32, "dst_blocks"), src_blocks.numel(),
                                 _stream(stream)), "kvq_copy_blocks")


def kvq_decode_workspace_bytes(pool, num_seqs, num_q_heads, max_context_len, split_blocks=0) -> int:
    return int(lib().kvq_decode_workspace_bytes_ex(pool, num_seqs, num_q_heads, max_context_len,
                                                   split_blocks))


def kvq_paged_decode(pool, q, block_table, context_lens, max_context_len, sm_scale, out,
                     workspace=None, split_blocks=0, stream=None) -> None:
    import torch

    S, Hq, _ = q.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().kvq_paged_decode_ex(
        pool, _ptr(q, torch.float16, "q"), S, Hq, _ptr(block_table, torch.int32, "block_table"),
        block_table.shape[1], _ptr(context_lens, torch.int32, "context_lens"), int(max_context_len),
        float(sm_scale), _ptr(out, torch.float32, "out"),
        _ptr(workspace, None, "workspace") if workspace is not None else None, ws_bytes,
        int(split_blocks), _stream(stream)), "kvq_paged_decode")


def kvq_decode_step(pool, k_new, v_new, q, block_table, context_lens, max_context_len, sm_scale,
                    out, workspace=None, stream=None) -> None:
    """Append each sequence's new token at position context_lens[s]-1, then
    decode (kvq_decode_step in include/kvq.h)."""
    import torch

    S, Hq, _ = q.shape
    if k_new.shape != v_new.shape or k_new.shape[0] != S:
        raise ValueError("k_new, v_new must be [num_seqs, kv_heads, head_dim]")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().kvq_decode_step(
        pool, _ptr(k_new, torch.float16, "k_new"), _ptr(v_new, torch.float16, "v_new"),
        _ptr(q, torch.float16, "q"), S, Hq, _ptr(block_table, torch.int32, "block_table"),
        block_table.shape[1], _ptr(context_lens, torch.int32, "context_lens"), int(max_context_len),
        float(sm_scale), _ptr(out, torch.float32, "out"),
        _ptr(workspace, None, "workspace") if workspace is not None else None, ws_bytes,
        _stream(stream)), "kvq_decode_step")


def kvq_cascade_workspace_bytes(pool, num_seqs, num_q_heads, max_context_len) -> int:
    return int(lib().kvq_cascade_workspace_bytes(pool, num_seqs, num_q_heads, max_context_len))


def kvq_cascade_decode(pool, q, block_table, context_lens, max_context_len, prefix_blocks,
                       sm_scale, out, workspace, stream=None) -> None:
    """Decode whose first prefix_blocks blocks (shared by every sequence) are
    attended once for all sequences (kvq_cascade_decode in include/kvq.h)."""
    import torch

    S, Hq, _ = q.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().kvq_cascade_decode(
        pool, _ptr(q, torch.float16, "q"), S, Hq, _ptr(block_table, torch.int32, "block_table"),
        block_table.shape[1], _ptr(context_lens, torch.int32, "context_lens"), int(max_context_len),
        int(prefix_blocks), float(sm_scale), _ptr(out, torch.float32, "out"),
        _ptr(workspace, None, "workspace") if workspace is not None else None, ws_bytes,
        _stream(stream)), "kvq_cascade_decode")


def kvq_cascade_decode_step(pool, k_new, v_new, q, block_table, context_lens, max_context_len,
                            prefix_blocks, sm_scale, out, workspace, stream=None) -> None:
    """kvq_decode_step with the shared-prefix cascade decode."""
    import torch

    S, Hq, _ = q.shape
    if k_new.shape != v_new.shape or k_new.shape[0] != S:
        raise ValueError("k_new, v_new must be [num_seqs, kv_heads, head_dim]")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().kvq_cascade_decode_step(
        pool, _ptr(k_new, torch.float16, "k_new"), _ptr(v_new, torch.float16, "v_new"),
        _ptr(q, torch.float16, "q"), S, Hq, _ptr(block_table, torch.int32, "block_table"),
        block_table.shape[1], _ptr(context_lens, torch.int32, "context_lens"), int(max_context_len),
        int(prefix_blocks), float(sm_scale), _ptr(out, torch.float32, "out"),
        _ptr(workspace, None, "workspace") if workspace is not None else None, ws_bytes,
        _stream(stream)), "kvq_cascade_decode_step")


def kvq_prefill(pool, q, q_start, max_q_len, block_table, context_lens, max_context_len, sm_scale,
                out, stream=None) -> None:
    """Causal attention of each sequence's new query tokens over its cache
    (kvq_prefill in include/kvq.h).  q: [Tq, Hq, D] fp16, q_start: [S+1] int32."""
    import torch

    Tq, Hq, _ = q.shape
    S = q_start.numel() - 1
    _check(lib().kvq_prefill(
        pool, _ptr(q, torch.float16, "q"), S, Hq, _ptr(q_start, torch.int32, "q_start"),
        int(max_q_len), _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
        _ptr(context_lens, torch.int32, "context_lens"), int(max_context_len), float(sm_scale),
        _ptr(out, torch.float32, "out"), _stream(stream)), "kvq_prefill")


def kvq_prefill_workspace_bytes(pool, num_seqs, max_context_len) -> int:
    return int(lib().kvq_prefill_workspace_bytes(pool, int(num_seqs), int(max_context_len)))


def kvq_prefill_ex(pool, q, q_start, max_q_len, block_table, context_lens, max_context_len,
                   sm_scale, out, workspace, stream=None) -> None:
    """kvq_prefill in two passes through a caller workspace (kvq_prefill_ex in
    include/kvq.h); workspace: uint8 device tensor of at least
    kvq_prefill_workspace_bytes(...) bytes, or None when that is 0."""
    import torch

    Tq, Hq, _ = q.shape
    S = q_start.numel() - 1
    ws = None if workspace is None else _ptr(workspace, torch.uint8, "workspace")
    nbytes = 0 if workspace is None else workspace.numel()
    _check(lib().kvq_prefill_ex(
        pool, _ptr(q, torch.float16, "q"), S, Hq, _ptr(q_start, torch.int32, "q_start"),
        int(max_q_len), _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
        _ptr(context_lens, torch.int32, "context_lens"), int(max_context_len), float(sm_scale),
        _ptr(out, torch.float32, "out"), ws, nbytes, _stream(stream)), "kvq_prefill_ex")


def kvq_selftest_decode_timeout(pool, q, block_table, context_lens, max_context_len, out,
                                workspace, wait_tries=20, stream=None) -> None:
    """Decode with one page copy withheld so that a bounded wait runs out
    (kvq_selftest_decode_timeout in include/kvq.h)."""
    import torch

    S, Hq, _ = q.shape
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().kvq_selftest_decode_timeout(
        pool, _ptr(q, torch.float16, "q"), S, Hq, _ptr(block_table, torch.int32, "block_table"),
        block_table.shape[1], _ptr(context_lens, torch.int32, "context_lens"), int(max_context_len),
        _ptr(out, torch.float32, "out"),
        _ptr(workspace, None, "workspace") if workspace is not None else None, ws_bytes,
        int(wait_tries), _stream(stream)), "kvq_selftest_decode_timeout")


KVQ_NOALLOC_SCRATCH_BYTES = 16 << 20


def kvq_paged_decode_noalloc(pool, q, block_table, context_lens, max_context_len, sm_scale, out,
                             split_blocks=0, stream=None) -> None:
    """kvq_paged_decode without a workspace argument, for callers that cannot
    allocate device memory: the split scratch is a fixed 16 MiB array inside
    the library (see kvq_paged_decode_noalloc in include/kvq.h)."""
    import torch

    S, Hq, _ = q.shape
    _check(lib().kvq_paged_decode_noalloc(
        pool, _ptr(q, torch.float16, "q"), S, Hq, _ptr(block_table, torch.int32, "block_table"),
        block_table.shape[1], _ptr(context_lens, torch.int32, "context_lens"), int(max_context_len),
        float(sm_scale), _ptr(out, torch.float32, "out"), int(split_blocks), _stream(stream)),
        "kvq_paged_decode_noalloc")


def kvq_read_slots(pool, slots, codes_out, scales_out=None, stream=None) -> None:
    import torch

    _check(lib().kvq_read_slots(pool, _ptr(slots, torch.int64, "slots"), slots.numel(),
                                _ptr(codes_out, None, "codes_out"),
                                _ptr(scales_out, torch.float32, "scales_out")
                                if scales_out is not None else None, _stream(stream)),
           "kvq_read_slots")


def kvq_get_error(pool, stream=None) -> int:
    """Synchronises the stream; returns (and clears) the pool's device error status."""
    return int(lib().kvq_get_error(pool, _stream(stream)))


def kvq_set_phase_events(events) -> None:
    """Measurement aid: the calling thread's next len(events) kernel launches
    by the library each record one of these torch.cuda.Event objects on their
    stream right after the launch (an empty list clears them; see kvq.h)."""
    handles = []
    for ev in events:
        if not ev.cuda_event:  # torch creates the CUDA event at its first record
            ev.record()
        handles.append(ev.cuda_event)
    arr = (ctypes.c_void_p * len(handles))(*handles) if handles else None
    _check(lib().kvq_set_phase_events(arr, len(handles)), "kvq_set_phase_events")


# ------------------------------------------------------------------ convenience
class KVPool:
    """One layer's pool in caller-owned (torch) device memory."""

    def __init__(self, num_blocks, block_size, kv_heads, head_dim, dtype, group=0, device="cuda",
                 fill_byte: int | None = None):
        import torch

        self.num_blocks, self.block_size, self.kv_heads, self.head_dim = (
            num_blocks, block_size, kv_heads, head_dim)
        self.dtype, self.group = dtype, (group if dtype in GROUP_FORMATS else 0)
        nbytes = kvq_pool_bytes(num_blocks, block_size, kv_heads, head_dim, dtype, self.group)
        if nbytes == 0:
            kvq_pool_layout_query(num_blocks, block_size, kv_heads, head_dim, dtype, self.group)
            raise KVQError(KVQ_ERR_INVALID_ARG, "KVPool")
        self.buffer = torch.empty(nbytes, dtype=torch.uint8, device=device)
        if fill_byte is not None:
            self.buffer.fill_(fill_byte)
        self.handle = kvq_alloc_pool(num_blocks, block_size, kv_heads, head_dim, dtype, self.group,
                                     self.buffer)

    def close(self):
        if getattr(self, "handle", None) is not None:
            kvq_free_pool(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def append(self, k, v, slot_mapping, stream=None):
        kvq_append(self.handle, k, v, slot_mapping, stream)

    def decode(self, q, block_table, context_lens, max_context_len, sm_scale=None, out=None,
               split_blocks=0, stream=None):
        import torch

        S, Hq, D = q.shape
        if sm_scale is None:
            sm_scale = D ** -0.5
        if out is None:
            out = torch.empty((S, Hq, D), dtype=torch.float32, device=q.device)
        nws = kvq_decode_workspace_bytes(self.handle, S, Hq, max_context_len, split_blocks)
        ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=q.device) if nws else None
        kvq_paged_decode(self.handle, q, block_table, context_lens, max_context_len, sm_scale, out,
                         ws, split_blocks, stream)
        return out

    def decode_step(self, k_new, v_new, q, block_table, context_lens, max_context_len,
                    sm_scale=None, out=None, stream=None):
        import torch

        S, Hq, D = q.shape
        if sm_scale is None:
            sm_scale = D ** -0.5
        if out is None:
            out = torch.empty((S, Hq, D), dtype=torch.float32, device=q.device)
        nws = kvq_decode_workspace_bytes(self.handle, S, Hq, max_context_len)
        ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=q.device) if nws else None
        kvq_decode_step(self.handle, k_new, v_new, q, block_table, context_lens, max_context_len,
                        sm_scale, out, ws, stream)
        return out

    def cascade_decode(self, q, block_table, context_lens, max_context_len, prefix_blocks,
                       sm_scale=None, out=None, stream=None):
        import torch

        S, Hq, D = q.shape
        if sm_scale is None:
            sm_scale = D ** -0.5
        if out is None:
            out = torch.empty((S, Hq, D), dtype=torch.float32, device=q.device)
        nws = kvq_cascade_workspace_bytes(self.handle, S, Hq, max_context_len)
        ws = torch.empty(max(nws, 256), dtype=torch.uint8, device=q.device)
        kvq_cascade_decode(self.handle, q, block_table, context_lens, max_context_len,
                           prefix_blocks, sm_scale, out, ws, stream)
        return out

    def read_slots(self, slots, stream=None):
        import torch

        n = slots.numel()
        cdt = torch.float16 if self.dtype == KVQ_FP16 else (
            torch.uint8 if self.dtype in (KVQ_FP8_E4M3_PER_TOKEN, KVQ_FP8_E5M2) else torch.int8)
        codes = torch.empty((n, 2, self.kv_heads, self.head_dim), dtype=cdt, device=slots.device)
        scales = None
        if self.dtype in GROUP_FORMATS:
            scales = torch.empty((n, 2, self.kv_heads, self.head_dim // self.group),
                                 dtype=torch.float32, device=slots.device)
        elif self.dtype in (KVQ_INT8_PER_TOKEN, KVQ_FP8_E4M3_PER_TOKEN):
            scales = torch.empty((n, 2), dtype=torch.float32, device=slots.device)
        kvq_read_slots(self.handle, slots, codes, scales, stream)
        return codes, scales

    def error(self, stream=None) -> int:
        return kvq_get_error(self.handle, stream)
