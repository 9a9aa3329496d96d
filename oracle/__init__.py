"""CPU oracle for the paged quantized KV decode step -- TEST INFRASTRUCTURE.

This package is a plain, slow restatement of the method, written to check the
CUDA library against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg and ``--impl reference`` arm of ``bench.py`` may import it.  The product package never
imports it and shares no code with it; the only thing both sides share is the
seeded input generator module, which holds none of the method's arithmetic.

The arithmetic lives in ``kvq_oracle.c`` (C11, fp32 quantizer, float64
attention); this module compiles it with gcc and marshals numpy arrays.

Sources: "KV Cache优化实战：大模型推理显存占用与加速方案详解"
(0539edu.com/news/5800990) §1.1, §1.2, §2.1-§2.3, §3.3; xpshop.cn article-402
§三 and article-312 §三 (paged INT8/FP8 KV case studies).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, the OCP e4m3 table, dense brute-force attention, invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# Cache formats (same numbering as the library's public enum).
FP16 = 0
INT8_PER_TOKEN = 1
INT8_PER_CHANNEL = 2
INT8_PER_GROUP = 3
FP8_E4M3_PER_TOKEN = 4
INT4_PER_GROUP = 5
FP8_E5M2 = 6
GROUP_FORMATS = (INT8_PER_GROUP, INT4_PER_GROUP)

FORMAT_NAMES = {
    FP16: "fp16",
    INT8_PER_TOKEN: "int8_token",
    INT8_PER_CHANNEL: "int8_channel",
    INT8_PER_GROUP: "int8_group",
    FP8_E4M3_PER_TOKEN: "fp8_e4m3_token",
    INT4_PER_GROUP: "int4_group",
    FP8_E5M2: "fp8_e5m2",
}


def compile_source(src: str, so: str) -> str:
    """Compile one oracle C source into a shared library (gcc, -O2, no FP
    contraction, OpenMP when available)."""
    base = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", src, "-o", so + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(so + ".tmp", so)
    return so


def build(force: bool = False) -> str:
    """Compile kvq_oracle.c into liboracle.so.  Returns the library's path."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    return compile_source(_SRC, _SO)


class use_library:
    """Context manager: route every oracle call through another build of the
    oracle (the mutation tests load deliberately broken copies this way)."""

    def __init__(self, so_path: str):
        self.so_path = so_path

    def __enter__(self):
        global _lib
        with _lock:
            self._saved = _lib
            L = ctypes.CDLL(self.so_path)
            _declare(L)
            _lib = L
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self._saved
        return False


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _declare(_lib)
        return _lib


def _declare(L: ctypes.CDLL) -> None:
    P = ctypes.c_void_p
    i32, i64, u64, f32, f64 = (ctypes.c_int, ctypes.c_int64, ctypes.c_uint64,
                               ctypes.c_float, ctypes.c_double)
    L.oracle_num_threads.restype = i32
    L.oracle_num_threads.argtypes = []
    L.oracle_half_to_float.restype = None
    L.oracle_half_to_float.argtypes = [P, P, i64]
    L.oracle_set_num_threads.restype = None
    L.oracle_set_num_threads.argtypes = [i32]
    L.oracle_kv_cache_bytes.restype = u64
    L.oracle_kv_cache_bytes.argtypes = [u64] * 6
    L.oracle_e4m3_decode.restype = f64
    L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    L.oracle_e4m3_encode.argtypes = [f32]
    L.oracle_e5m2_decode.restype = f64
    L.oracle_e5m2_decode.argtypes = [ctypes.c_uint8]
    L.oracle_e5m2_encode.restype = ctypes.c_uint8
    L.oracle_e5m2_encode.argtypes = [f32]
    L.oracle_quant_int8_group.restype = None
    L.oracle_quant_int8_group.argtypes = [P, i32, P, P]
    L.oracle_quant_int4_group.restype = None
    L.oracle_quant_int4_group.argtypes = [P, i32, P, P]
    L.oracle_quant_int8_static.restype = None
    L.oracle_quant_int8_static.argtypes = [P, P, i32, P]
    L.oracle_quant_e4m3_group.restype = None
    L.oracle_quant_e4m3_group.argtypes = [P, i32, P, P]
    L.oracle_calibrate_channels.restype = None
    L.oracle_calibrate_channels.argtypes = [P, i64, i32, P]
    L.oracle_append.restype = None
    L.oracle_append.argtypes = [i32, i64, i32, i32, i32, P, P, P, P, P, P]
    L.oracle_decode.restype = None
    L.oracle_decode.argtypes = [i32, i32, i32, i32, i32, i32, i32, P, P, i32, P, f64,
                                P, P, P, P]


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def half_to_float(x) -> np.ndarray:
    """float16 array widened exactly to float32 by the oracle's own routine."""
    h = np.ascontiguousarray(np.asarray(x, dtype=np.float16))
    out = np.empty(h.shape, np.float32)
    lib().oracle_half_to_float(_ptr(h), _ptr(out), h.size)
    return out


def _f32(x) -> np.ndarray:
    """fp16 (or fp32) input widened exactly to a contiguous float32 array."""
    x = np.asarray(x)
    if x.dtype == np.float16:
        return half_to_float(x)
    return np.ascontiguousarray(x, dtype=np.float32)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))


def kv_cache_bytes(batch, seq_len, layers, kv_heads, head_dim, precision_bytes) -> int:
    """KV size formula of KV Cache优化实战 §1.2."""
    return int(lib().oracle_kv_cache_bytes(batch, seq_len, layers, kv_heads, head_dim,
                                           precision_bytes))


def e4m3_decode(code: int) -> float:
    return float(lib().oracle_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(x: float) -> int:
    return int(lib().oracle_e4m3_encode(float(np.float32(x))))


def e5m2_decode(code: int) -> float:
    return float(lib().oracle_e5m2_decode(int(code) & 0xFF))


def e5m2_encode(x: float) -> int:
    return int(lib().oracle_e5m2_encode(float(np.float32(x))))


def quant_int8_group(x) -> tuple[np.ndarray, np.float32]:
    x = _f32(x).ravel()
    codes = np.zeros(x.size, np.int8)
    s = np.zeros(1, np.float32)
    lib().oracle_quant_int8_group(_ptr(x), x.size, _ptr(codes), _ptr(s))
    return codes, s[0]


def quant_int4_group(x) -> tuple[np.ndarray, np.float32]:
    x = _f32(x).ravel()
    codes = np.zeros(x.size, np.int8)
    s = np.zeros(1, np.float32)
    lib().oracle_quant_int4_group(_ptr(x), x.size, _ptr(codes), _ptr(s))
    return codes, s[0]


def quant_int8_static(x, scales) -> np.ndarray:
    x = _f32(x).ravel()
    sc = _f32(scales).ravel()
    assert sc.size == x.size
    codes = np.zeros(x.size, np.int8)
    lib().oracle_quant_int8_static(_ptr(x), _ptr(sc), x.size, _ptr(codes))
    return codes


def quant_e4m3_group(x) -> tuple[np.ndarray, np.float32]:
    x = _f32(x).ravel()
    codes = np.zeros(x.size, np.uint8)
    s = np.zeros(1, np.float32)
    lib().oracle_quant_e4m3_group(_ptr(x), x.size, _ptr(codes), _ptr(s))
    return codes, s[0]


def calibrate_channels(x) -> np.ndarray:
    """Per-channel scale absmax/127 over the calibration tokens; x is [T][C]."""
    x = _f32(x)
    T = x.shape[0]
    x2 = x.reshape(T, -1)
    C = x2.shape[1]
    s = np.zeros(C, np.float32)
    lib().oracle_calibrate_channels(_ptr(np.ascontiguousarray(x2)), T, C, _ptr(s))
    return s.reshape(x.shape[1:])


class OracleCache:
    """The oracle's slot-indexed cache for one layer.

    codes  : [num_slots, 2, Hkv, D]  int8 / uint8 (e4m3) / float32 (fp16 values)
    scales : per-group [num_slots, 2, Hkv, D/g]; per-token [num_slots, 2]
    chan_scales (per-channel only): [2, Hkv, D]
    Untouched slots keep the sentinel they were created with.
    """

    def __init__(self, fmt: int, num_blocks: int, block_size: int, kv_heads: int,
                 head_dim: int, group: int = 0, sentinel_code: int = 0,
                 sentinel_scale: float = 0.0):
        self.fmt, self.bs, self.Hkv, self.D = fmt, block_size, kv_heads, head_dim
        self.g = group if fmt in GROUP_FORMATS else 0
        if fmt in GROUP_FORMATS and (group <= 0 or head_dim % group):
            raise ValueError("the group size must divide head_dim")
        self.num_slots = num_blocks * block_size
        shape = (self.num_slots, 2, kv_heads, head_dim)
        if fmt == FP16:
            self.codes = np.full(shape, np.float32(sentinel_code), np.float32)
        elif fmt in (FP8_E4M3_PER_TOKEN, FP8_E5M2):
            self.codes = np.full(shape, sentinel_code & 0xFF, np.uint8)
        else:
            self.codes = np.full(shape, sentinel_code, np.int8)
        if fmt in GROUP_FORMATS:
            self.scales = np.full((self.num_slots, 2, kv_heads, head_dim // group),
                                  sentinel_scale, np.float32)
        elif fmt in (INT8_PER_TOKEN, FP8_E4M3_PER_TOKEN):
            self.scales = np.full((self.num_slots, 2), sentinel_scale, np.float32)
        else:
            self.scales = np.zeros((1,), np.float32)
        self.chan_scales = np.zeros((2, kv_heads, head_dim), np.float32)

    def set_channel_scales(self, k_scale, v_scale) -> None:
        self.chan_scales[0] = _f32(k_scale).reshape(self.Hkv, self.D)
        self.chan_scales[1] = _f32(v_scale).reshape(self.Hkv, self.D)

    def calibrate(self, k, v) -> None:
        """Per-channel calibration over the given tokens ([T, Hkv, D] each)."""
        self.set_channel_scales(calibrate_channels(k), calibrate_channels(v))

    def append(self, k, v, slots) -> None:
        k = _f32(k)
        v = _f32(v)
        slots = np.ascontiguousarray(slots, dtype=np.int64)
        T = slots.size
        assert k.shape == (T, self.Hkv, self.D) and v.shape == k.shape
        assert int(slots.max(initial=-1)) < self.num_slots
        # Tokens are appended in order, so a repeated slot ends up holding its
        # last token: keep only that one (the C loop takes distinct slots).
        live = np.nonzero(slots >= 0)[0]
        _, last = np.unique(slots[live][::-1], return_index=True)
        keep = np.sort(live[live.size - 1 - last])
        if keep.size != T:
            k, v, slots = (np.ascontiguousarray(k[keep]), np.ascontiguousarray(v[keep]),
                           np.ascontiguousarray(slots[keep]))
            T = slots.size
        lib().oracle_append(self.fmt, T, self.Hkv, self.D, self.g or 1, _ptr(k), _ptr(v),
                            _ptr(slots), _ptr(self.chan_scales), _ptr(self.codes),
                            _ptr(self.scales))

    def copy_blocks(self, src, dst) -> None:
        """Copy-on-write ("KV Cache优化实战：大模型推理显存占用与加速方案详解" §4.4): block
        dst[i] takes the codes and scales of every slot of block src[i]."""
        for s, d in zip(np.asarray(src).ravel(), np.asarray(dst).ravel()):
            a, b = int(s) * self.bs, int(d) * self.bs
            self.codes[b:b + self.bs] = self.codes[a:a + self.bs]
            if self.scales.ndim > 1:
                self.scales[b:b + self.bs] = self.scales[a:a + self.bs]

    def decode(self, q, block_table, context_lens, sm_scale: float | None = None) -> np.ndarray:
        """Float64 attention output [S, Hq, D] over the dequantized cache."""
        q = _f32(q)
        S, Hq, D = q.shape
        assert D == self.D and Hq % self.Hkv == 0
        table = np.ascontiguousarray(block_table, dtype=np.int32)
        lens = np.ascontiguousarray(context_lens, dtype=np.int32)
        assert table.shape[0] == S and lens.shape == (S,)
        if sm_scale is None:
            sm_scale = 1.0 / np.sqrt(D)
        out = np.zeros((S, Hq, D), np.float64)
        lib().oracle_decode(self.fmt, S, Hq, self.Hkv, D, self.g or 1, self.bs, _ptr(q),
                            _ptr(table), table.shape[1], _ptr(lens), float(sm_scale),
                            _ptr(self.codes), _ptr(self.scales), _ptr(self.chan_scales),
                            _ptr(out))
        return out

    def dequantized(self, kv: int) -> np.ndarray:
        """Float64 dequantized cache [num_slots, Hkv, D] for K (kv=0) or V (kv=1),
        computed with numpy from the stored codes and scales (used by the dense
        brute-force pin, which must not reuse the C decode loop)."""
        c = self.codes[:, kv]
        if self.fmt == FP16:
            return c.astype(np.float64)
        if self.fmt == FP8_E4M3_PER_TOKEN:
            table = np.array([e4m3_decode(i) for i in range(256)], np.float64)
            vals = table[c]
        elif self.fmt == FP8_E5M2:
            table = np.array([e5m2_decode(i) for i in range(256)], np.float64)
            return table[c]
        else:
            vals = c.astype(np.float64)
        if self.fmt in GROUP_FORMATS:
            s = np.repeat(self.scales[:, kv].astype(np.float64), self.g, axis=2)
            return vals * s
        if self.fmt in (INT8_PER_TOKEN, FP8_E4M3_PER_TOKEN):
            return vals * self.scales[:, kv].astype(np.float64)[:, None, None]
        if self.fmt == INT8_PER_CHANNEL:
            return vals * self.chan_scales[kv].astype(np.float64)[None]
        raise ValueError(self.fmt)
