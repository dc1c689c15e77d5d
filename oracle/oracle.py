"""ctypes wrapper over the fp64 OSCAR oracle (test infrastructure only).

Every function takes and returns numpy arrays.  bf16 tensors travel as their
uint16 bit patterns, fp16 scale/zero pairs as uint16 bit patterns, so no value
is rounded on the way in or out.  The arithmetic lives in ``oscar_oracle.cpp``;
this module only marshals arguments.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oscar_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboscar_oracle.so")

__all__ = [
    "OracleDims", "build_oracle", "load", "bf16_to_f64", "f16_to_f64", "f64_to_f16",
    "rotate", "clip", "group_params", "quantize", "codes_given_params", "append", "append_prequant",
    "attend_mixed", "dequant_row", "decode", "bf16_decode", "extend",
]


def build_oracle(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with gcc (strict IEEE fp64: no fast-math, no FMA contraction)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
               src, "-o", out + ".tmp"]
        subprocess.run(cmd, check=True)
        os.replace(out + ".tmp", out)
    return out


class OracleDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_q_heads", "num_kv_heads", "head_dim", "page_size", "group_size", "num_pages",
        "max_pages_per_seq")]


_P = ctypes.c_void_p
_LIBS: dict = {}


def load(path: str | None = None):
    """Load (building if needed) the oracle library; ``path`` selects another build."""
    if path is None:
        path = build_oracle()
    if path in _LIBS:
        return _LIBS[path]
    lib = ctypes.CDLL(path)
    sigs = {
        "orc_bf16_to_f64": (ctypes.c_double, [ctypes.c_uint16]),
        "orc_f16_to_f64": (ctypes.c_double, [ctypes.c_uint16]),
        "orc_f64_to_f16": (ctypes.c_uint16, [ctypes.c_double]),
        "orc_rotate": (None, [ctypes.c_int32, _P, _P, _P]),
        "orc_clip": (None, [ctypes.c_int32, _P, _P]),
        "orc_group_params": (None, [ctypes.c_int32, _P, _P, _P]),
        "orc_quantize": (ctypes.c_int32, [ctypes.c_double, ctypes.c_uint16, ctypes.c_uint16, _P]),
        "orc_offset_key": (None, [ctypes.c_int32, _P, _P, _P]),
        "orc_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
        "orc_append_prequant": (ctypes.c_int32, [_P, ctypes.c_int64, _P, _P, _P, _P, _P, _P, _P, _P]),
        "orc_codes_given_params": (None, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P]),
        "orc_append": (ctypes.c_int32, [_P, ctypes.c_int64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
        "orc_append_mixed": (ctypes.c_int32, [_P, ctypes.c_int64, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P]),
        "orc_attend_mixed": (None, [ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P, _P,
                                    ctypes.c_double, _P, _P]),
        "orc_dequant_row": (None, [_P, _P, _P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                   ctypes.c_int32, _P]),
        "orc_decode": (ctypes.c_int32, [_P, ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                        ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                        ctypes.c_int32, _P, _P]),
        "orc_bf16_decode": (ctypes.c_int32, [_P, ctypes.c_int32, _P, _P, _P, _P, ctypes.c_double,
                                             ctypes.c_int32, _P, _P]),
        "orc_extend": (ctypes.c_int32, [_P, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                        _P, _P, ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                        ctypes.c_int32, _P, _P]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIBS[path] = lib
    return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dims(d) -> OracleDims:
    if isinstance(d, OracleDims):
        return d
    return OracleDims(*[int(d[n]) for n, _ in OracleDims._fields_])


# --- number formats ---------------------------------------------------------

def bf16_to_f64(bits, lib=None) -> np.ndarray:
    lib = lib or load()
    b = np.asarray(bits, dtype=np.uint16)
    return np.array([lib.orc_bf16_to_f64(int(x)) for x in b.ravel()], dtype=np.float64).reshape(b.shape)


def f16_to_f64(bits, lib=None) -> np.ndarray:
    lib = lib or load()
    b = np.asarray(bits, dtype=np.uint16)
    return np.array([lib.orc_f16_to_f64(int(x)) for x in b.ravel()], dtype=np.float64).reshape(b.shape)


def f64_to_f16(vals, lib=None) -> np.ndarray:
    lib = lib or load()
    v = np.asarray(vals, dtype=np.float64)
    return np.array([lib.orc_f64_to_f16(float(x)) for x in v.ravel()], dtype=np.uint16).reshape(v.shape)


# --- append steps -------------------------------------------------------------

def rotate(x_bf16_bits: np.ndarray, R: np.ndarray, lib=None) -> np.ndarray:
    """x_rot = x . R for one vector (x as bf16 bits [D], R fp32 [D][D])."""
    lib = lib or load()
    x = _c(x_bf16_bits, np.uint16)
    Rm = _c(R, np.float32)
    D = x.shape[0]
    out = np.empty(D, np.float64)
    lib.orc_rotate(D, _ptr(x), _ptr(Rm), _ptr(out))
    return out


def offset_key(k_bf16_bits: np.ndarray, c: np.ndarray, lib=None) -> np.ndarray:
    """fp32(k - c) of one key (bf16 bits [D]) and its offset (fp32 [D]), as fp64."""
    lib = lib or load()
    k = _c(k_bf16_bits, np.uint16)
    cc = _c(c, np.float32)
    out = np.empty(k.shape[0], np.float64)
    lib.orc_offset_key(k.shape[0], _ptr(k), _ptr(cc), _ptr(out))
    return out


def f32_to_bf16(vals, lib=None) -> np.ndarray:
    lib = lib or load()
    v = np.asarray(vals, dtype=np.float32)
    return np.array([lib.orc_f32_to_bf16(float(x)) for x in v.ravel()], dtype=np.uint16).reshape(v.shape)


def _offset(offset_k):
    return None if offset_k is None else _c(offset_k, np.float32)


def clip(x: np.ndarray, c: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    y = _c(x, np.float64).copy()
    cc = _c(c, np.float32)
    lib.orc_clip(y.shape[0], _ptr(y), _ptr(cc))
    return y


def group_params(xg: np.ndarray, lib=None) -> tuple[int, int]:
    """(scale bits, zero bits) of one group."""
    lib = lib or load()
    x = _c(xg, np.float64)
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    lib.orc_group_params(x.shape[0], _ptr(x), _ptr(s), _ptr(z))
    return int(s[0]), int(z[0])


def quantize(x: float, s_bits: int, z_bits: int, lib=None) -> tuple[int, float]:
    """(code, u) of one value given the stored fp16 scale and zero."""
    lib = lib or load()
    u = ctypes.c_double(0.0)
    c = lib.orc_quantize(float(x), int(s_bits), int(z_bits), ctypes.byref(u))
    return int(c), float(u.value)


def codes_given_params(x: np.ndarray, sz_bits: np.ndarray, group_size: int, lib=None):
    """Codes and u of rows x [n][D] given stored (scale, zero) bits [n][D/G][2]."""
    lib = lib or load()
    xx = _c(x, np.float64)
    n, D = xx.shape
    s = _c(sz_bits, np.uint16).reshape(n, D // group_size, 2)
    codes = np.empty((n, D), np.int32)
    u = np.empty((n, D), np.float64)
    lib.orc_codes_given_params(n, D, group_size, _ptr(xx), _ptr(s), _ptr(codes), _ptr(u))
    return codes, u


def append_prequant(dims, k_bits, v_bits, R_k, R_v, clip_k, clip_v, offset_k=None, lib=None) -> np.ndarray:
    """Rotated+clipped fp64 values [T][Hkv][2][D] of every (token, head, K|V);
    ``offset_k`` (fp32 [Hkv][D] or None) is subtracted from every key first."""
    lib = lib or load()
    d = _dims(dims)
    k = _c(k_bits, np.uint16)
    v = _c(v_bits, np.uint16)
    T = k.shape[0]
    out = np.empty((T, d.num_kv_heads, 2, d.head_dim), np.float64)
    args = [_c(a, np.float32) for a in (R_k, R_v, clip_k, clip_v)]
    off = _offset(offset_k)
    lib.orc_append_prequant(ctypes.byref(d), T, _ptr(k), _ptr(v), *[_ptr(a) for a in args], _ptr(off), _ptr(out))
    return out


def append(dims, k_bits, v_bits, R_k, R_v, clip_k, clip_v, slot_mapping, int2_pages, scale_zero_pages,
           offset_k=None, lib=None) -> int:
    """Append into the given host pools in place (uint8 codes, uint16 fp16-bits scale/zero)."""
    lib = lib or load()
    d = _dims(dims)
    k = _c(k_bits, np.uint16)
    v = _c(v_bits, np.uint16)
    slots = _c(slot_mapping, np.int64)
    assert int2_pages.dtype == np.uint8 and int2_pages.flags.c_contiguous
    assert scale_zero_pages.dtype == np.uint16 and scale_zero_pages.flags.c_contiguous
    args = [_c(a, np.float32) for a in (R_k, R_v, clip_k, clip_v)]
    off = _offset(offset_k)
    return lib.orc_append(ctypes.byref(d), k.shape[0], _ptr(k), _ptr(v), *[_ptr(a) for a in args], _ptr(off),
                          _ptr(slots), _ptr(int2_pages), _ptr(scale_zero_pages))


def append_mixed(dims, k_bits, v_bits, R_k, R_v, clip_k, clip_v, slot_mapping, seq_ids, positions, seq_lens,
                 sink_len, window_len, int2_pages, scale_zero_pages, sink_bits, window_bits, offset_k=None,
                 lib=None) -> int:
    """Append into the host INT2 pools and the BF16 sink/window (uint16 bf16 bits,
    [B][2][Hkv][S|W][D]) in place."""
    lib = lib or load()
    d = _dims(dims)
    k = _c(k_bits, np.uint16)
    v = _c(v_bits, np.uint16)
    slots = _c(slot_mapping, np.int64)
    sid, pos, lens = (_c(a, np.int32) for a in (seq_ids, positions, seq_lens))
    for a, t in ((int2_pages, np.uint8), (scale_zero_pages, np.uint16), (sink_bits, np.uint16),
                 (window_bits, np.uint16)):
        assert a.dtype == t and a.flags.c_contiguous
    args = [_c(a, np.float32) for a in (R_k, R_v, clip_k, clip_v)]
    off = _offset(offset_k)
    return lib.orc_append_mixed(ctypes.byref(d), k.shape[0], _ptr(k), _ptr(v), *[_ptr(a) for a in args],
                                _ptr(off), _ptr(slots), _ptr(sid), _ptr(pos), _ptr(lens), lens.shape[0], int(sink_len),
                                int(window_len), _ptr(int2_pages), _ptr(scale_zero_pages), _ptr(sink_bits),
                                _ptr(window_bits))


# --- decode -------------------------------------------------------------------

def attend_mixed(q, q_rot, keys, vals, is_rot, sm_scale, R_v, lib=None) -> np.ndarray:
    lib = lib or load()
    qv = _c(q, np.float64)
    qr = _c(q_rot, np.float64)
    K = _c(keys, np.float64)
    V = _c(vals, np.float64)
    rot = _c(is_rot, np.int32)
    R = _c(R_v, np.float32)
    D = qv.shape[0]
    out = np.empty(D, np.float64)
    lib.orc_attend_mixed(D, K.shape[0], _ptr(qv), _ptr(qr), _ptr(K), _ptr(V), _ptr(rot), float(sm_scale),
                         _ptr(R), _ptr(out))
    return out


def dequant_row(dims, int2_pages, scale_zero_pages, page, h, kv, off, lib=None) -> np.ndarray:
    lib = lib or load()
    d = _dims(dims)
    out = np.empty(d.head_dim, np.float64)
    lib.orc_dequant_row(ctypes.byref(d), _ptr(int2_pages), _ptr(scale_zero_pages), int(page), int(h), int(kv),
                        int(off), _ptr(out))
    return out


def decode(dims, batch, q_bits, R_k, R_v, int2_pages, scale_zero_pages, sink_bits, window_bits, page_table,
           seq_lens, sink_len, window_len, sm_scale, pairs=None, lib=None) -> np.ndarray:
    """fp64 output [n_pairs][D] (all (b, hq) pairs in order when ``pairs`` is None)."""
    lib = lib or load()
    d = _dims(dims)
    if pairs is None:
        pairs = [(b, h) for b in range(batch) for h in range(d.num_q_heads)]
    pr = _c(np.asarray(pairs, dtype=np.int32).reshape(-1, 2), np.int32)
    q = _c(q_bits, np.uint16)
    Rk = _c(R_k, np.float32)
    Rv = _c(R_v, np.float32)
    codes = _c(int2_pages, np.uint8)
    sz = _c(scale_zero_pages, np.uint16)
    sink = None if sink_bits is None else _c(sink_bits, np.uint16)
    win = None if window_bits is None else _c(window_bits, np.uint16)
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    out = np.empty((pr.shape[0], d.head_dim), np.float64)
    rc = lib.orc_decode(ctypes.byref(d), int(batch), _ptr(q), _ptr(Rk), _ptr(Rv), _ptr(codes), _ptr(sz),
                        _ptr(sink), _ptr(win), _ptr(pt), _ptr(sl), int(sink_len), int(window_len),
                        float(sm_scale), pr.shape[0], _ptr(pr), _ptr(out))
    if rc != 0:
        raise ValueError("oracle decode: page id or length outside the pool / page table")
    return out


def extend(dims, batch, q_bits, row_seq, row_pos, R_k, R_v, int2_pages, scale_zero_pages, sink_bits, window_bits,
           page_table, seq_lens, sink_len, window_len, sm_scale, pairs=None, lib=None) -> np.ndarray:
    """Extend attention, fp64 output [n_pairs][D] for (query row, query head) pairs
    (all pairs in order when ``pairs`` is None); q_bits is [num_rows][Hq][D]."""
    lib = lib or load()
    d = _dims(dims)
    q = _c(q_bits, np.uint16)
    num_rows = q.shape[0]
    if pairs is None:
        pairs = [(r, h) for r in range(num_rows) for h in range(d.num_q_heads)]
    pr = _c(np.asarray(pairs, dtype=np.int32).reshape(-1, 2), np.int32)
    rs = _c(row_seq, np.int32)
    rp = _c(row_pos, np.int32)
    Rk = _c(R_k, np.float32)
    Rv = _c(R_v, np.float32)
    codes = _c(int2_pages, np.uint8)
    sz = _c(scale_zero_pages, np.uint16)
    sink = None if sink_bits is None else _c(sink_bits, np.uint16)
    win = None if window_bits is None else _c(window_bits, np.uint16)
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    out = np.empty((pr.shape[0], d.head_dim), np.float64)
    rc = lib.orc_extend(ctypes.byref(d), int(batch), int(num_rows), _ptr(q), _ptr(rs), _ptr(rp), _ptr(Rk), _ptr(Rv),
                        _ptr(codes), _ptr(sz), _ptr(sink), _ptr(win), _ptr(pt), _ptr(sl), int(sink_len),
                        int(window_len), float(sm_scale), pr.shape[0], _ptr(pr), _ptr(out))
    if rc != 0:
        raise ValueError("oracle extend: sequence, position, page id or length out of range")
    return out


def bf16_decode(dims, batch, q_bits, bf16_pages_bits, page_table, seq_lens, sm_scale, pairs=None,
                lib=None) -> np.ndarray:
    lib = lib or load()
    d = _dims(dims)
    if pairs is None:
        pairs = [(b, h) for b in range(batch) for h in range(d.num_q_heads)]
    pr = _c(np.asarray(pairs, dtype=np.int32).reshape(-1, 2), np.int32)
    q = _c(q_bits, np.uint16)
    pages = _c(bf16_pages_bits, np.uint16)
    pt = _c(page_table, np.int32)
    sl = _c(seq_lens, np.int32)
    out = np.empty((pr.shape[0], d.head_dim), np.float64)
    rc = lib.orc_bf16_decode(ctypes.byref(d), int(batch), _ptr(q), _ptr(pages), _ptr(pt), _ptr(sl),
                             float(sm_scale), pr.shape[0], _ptr(pr), _ptr(out))
    if rc != 0:
        raise ValueError("oracle bf16 decode: page id or length outside the pool / page table")
    return out
