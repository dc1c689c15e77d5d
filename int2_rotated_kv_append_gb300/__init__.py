"""OSCAR INT2 rotated KV append + mixed-precision paged decode for GB300.

Thin ctypes binding over ``liboscar.so`` (the C ABI declared in
``include/oscar.h``).  The functions carry the C names and only marshal
torch tensors to pointers; every step of the path runs in the CUDA kernels.
The library must have been built (``int2_rotated_kv_append_gb300.build``):
it is loaded on first use, and any call without it raises ImportError --
there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liboscar.so")

OSCAR_OK = 0
OSCAR_ERR_INVALID_ARG = 1
OSCAR_ERR_UNSUPPORTED = 2
OSCAR_ERR_WORKSPACE = 3
OSCAR_ERR_CUDA = 4

OSCAR_DEVERR_SLOT = 0x1
OSCAR_DEVERR_PAGE_ID = 0x2
OSCAR_DEVERR_SEQ_LEN = 0x4
OSCAR_DEVERR_TIMEOUT = 0x8
OSCAR_DEVERR_POSITION = 0x10


class OscarError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)}")
        self.status = status


class oscar_dims_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_q_heads", "num_kv_heads", "head_dim", "page_size", "group_size", "num_pages",
        "max_pages_per_seq")]


class oscar_calib_out_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("R", "clip", "eigenvalues", "cov", "sweeps")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"OSCAR CUDA library not built ({LIB_PATH} missing); run "
                          "int2_rotated_kv_append_gb300.build.build() -- there is no CPU fallback")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    D = ctypes.POINTER(oscar_dims_t)
    sigs = {
        "oscar_append": (I32, [D, I64, P, P, P, P, P, P, P, P, P, P, P, P]),
        "oscar_append_mixed": (I32, [D, I64, P, P, P, P, P, P, P, P, P, P, P, P, I32, I32, I32, P, P, P, P, P]),
        "oscar_decode_workspace_bytes": (SZ, [D, I32, I32, I32, I32, I32]),
        "oscar_decode_plan": (I32, [D, I32, I32, I32, I32, I32, ctypes.POINTER(I32), ctypes.POINTER(I32),
                                    ctypes.POINTER(I32)]),
        "oscar_decode": (I32, [D, I32, I32, I32, P, P, P, P, P, P, P, P, P, I32, I32, F32, P, P, SZ, P]),
        "oscar_append_decode": (I32, [D, I32, I32, I32, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, I32, I32, F32,
                                      P, P, SZ, P]),
        "oscar_decode_noalloc": (I32, [D, I32, I32, I32, P, P, P, P, P, P, P, P, P, I32, I32, F32, P, P]),
        "oscar_extend_workspace_bytes": (SZ, [D, I32, I32, I32, I32, I32]),
        "oscar_extend": (I32, [D, I32, I32, I32, I32, P, P, P, P, P, P, P, P, P, P, P, I32, I32, F32, P, P, SZ, P]),
        "oscar_extend_varlen_workspace_bytes": (SZ, [D, I32, I32, I32, I32, I32]),
        "oscar_extend_varlen": (I32, [D, I32, I32, I32, I32, I32, P, P, P, P, P, P, P, P, P, P, I32, I32, F32, P, P, SZ,
                                      P]),
        "oscar_bf16_append": (I32, [D, I64, P, P, P, P, P]),
        "oscar_bf16_decode_workspace_bytes": (SZ, [D, I32, I32, I32]),
        "oscar_bf16_decode": (I32, [D, I32, I32, I32, P, P, P, P, F32, P, P, SZ, P]),
        "oscar_calibrate_workspace_bytes": (SZ, [D, I64]),
        "oscar_calibrate": (I32, [D, I64, P, P, I32, ctypes.c_double, ctypes.POINTER(oscar_calib_out_t),
                                  ctypes.POINTER(oscar_calib_out_t), P, SZ, P]),
        "oscar_status_string": (ctypes.c_char_p, [I32]),
        "oscar_device_errors": (I32, [ctypes.POINTER(ctypes.c_uint32), I32]),
        "oscar_test_stall_page_waits": (I32, [I64]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


class _LazyLib:
    """Loads liboscar.so on first attribute access (raises ImportError if absent)."""

    _handle = None

    def __getattr__(self, name):
        if _LazyLib._handle is None:
            _LazyLib._handle = _load()
        return getattr(_LazyLib._handle, name)


lib = _LazyLib()


def load_library():
    """Load the CUDA library now; returns the ctypes handle."""
    lib.oscar_status_string  # noqa: B018 -- forces the load
    return _LazyLib._handle


def status_string(status: int) -> str:
    return lib.oscar_status_string(int(status)).decode()


def make_dims(num_q_heads, num_kv_heads, head_dim, page_size, group_size, num_pages, max_pages_per_seq):
    return oscar_dims_t(int(num_q_heads), int(num_kv_heads), int(head_dim), int(page_size), int(group_size),
                        int(num_pages), int(max_pages_per_seq))


def _dims(d) -> oscar_dims_t:
    if isinstance(d, oscar_dims_t):
        return d
    return make_dims(**d)


def _ptr(t) -> ctypes.c_void_p | None:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("OSCAR tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


def _check(status: int, where: str):
    if status != OSCAR_OK:
        raise OscarError(status, where)


def oscar_append(dims, k, v, R_k, R_v, clip_k, clip_v, page_table, slot_mapping, int2_pages, scale_zero_pages,
                 stream=None, offset_k=None):
    """Rotate, clip, INT2-quantise and store k/v (bf16 [T][Hkv][D]) at slot_mapping;
    ``offset_k`` (fp32 [Hkv][D] or None) is subtracted from every key first."""
    _check(lib.oscar_append(ctypes.byref(_dims(dims)), int(k.shape[0]), _ptr(k), _ptr(v), _ptr(R_k), _ptr(R_v),
                            _ptr(clip_k), _ptr(clip_v), _ptr(offset_k), _ptr(page_table), _ptr(slot_mapping),
                            _ptr(int2_pages), _ptr(scale_zero_pages), _stream(stream)), "oscar_append")


def oscar_append_mixed(dims, k, v, R_k, R_v, clip_k, clip_v, page_table, slot_mapping, seq_ids, positions,
                       seq_lens, sink_len, window_len, int2_pages, scale_zero_pages, bf16_sink, bf16_window,
                       stream=None, offset_k=None):
    """oscar_append plus the tokens' bf16 rows in the sink (position < sink_len) and
    the window ring (positions of the window after this append); with ``offset_k``
    the K rows are the offset keys."""
    _check(lib.oscar_append_mixed(ctypes.byref(_dims(dims)), int(k.shape[0]), _ptr(k), _ptr(v), _ptr(R_k),
                                  _ptr(R_v), _ptr(clip_k), _ptr(clip_v), _ptr(offset_k), _ptr(page_table),
                                  _ptr(slot_mapping),
                                  _ptr(seq_ids), _ptr(positions), _ptr(seq_lens), int(seq_lens.shape[0]),
                                  int(sink_len), int(window_len), _ptr(int2_pages), _ptr(scale_zero_pages),
                                  _ptr(bf16_sink), _ptr(bf16_window), _stream(stream)), "oscar_append_mixed")


def oscar_decode_workspace_bytes(dims, batch, max_seq_len, pages_per_split, sink_len, window_len) -> int:
    return int(lib.oscar_decode_workspace_bytes(ctypes.byref(_dims(dims)), int(batch), int(max_seq_len),
                                                int(pages_per_split), int(sink_len), int(window_len)))


def oscar_decode_plan(dims, batch, max_seq_len, pages_per_split, sink_len, window_len) -> dict:
    """The decode's schedule for these sizes: {"fused": 0|1, "splits": INT2 splits per
    (sequence, KV head), "pages_per_split": pages per INT2 split}."""
    f, s, pps = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib.oscar_decode_plan(ctypes.byref(_dims(dims)), int(batch), int(max_seq_len), int(pages_per_split),
                                 int(sink_len), int(window_len), ctypes.byref(f), ctypes.byref(s), ctypes.byref(pps)),
           "oscar_decode_plan")
    return {"fused": f.value, "splits": s.value, "pages_per_split": pps.value}


def oscar_decode(dims, batch, max_seq_len, pages_per_split, q, R_k, R_v, int2_pages, scale_zero_pages, bf16_sink,
                 bf16_window, page_table, seq_lens, sink_len, window_len, sm_scale, out, workspace, stream=None):
    """One mixed-precision decode step; writes fp32 out [B][Hq][D]."""
    _check(lib.oscar_decode(ctypes.byref(_dims(dims)), int(batch), int(max_seq_len), int(pages_per_split), _ptr(q),
                            _ptr(R_k), _ptr(R_v), _ptr(int2_pages), _ptr(scale_zero_pages), _ptr(bf16_sink),
                            _ptr(bf16_window), _ptr(page_table), _ptr(seq_lens), int(sink_len), int(window_len),
                            float(sm_scale), _ptr(out), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream)), "oscar_decode")


def oscar_append_decode(dims, batch, max_seq_len, pages_per_split, q, k, v, R_k, R_v, clip_k, clip_v, slot_mapping,
                        int2_pages, scale_zero_pages, bf16_sink, bf16_window, page_table, seq_lens, sink_len,
                        window_len, sm_scale, out, workspace, stream=None, offset_k=None):
    """One decode step: appends each sequence's current token k, v [B][Hkv][D] (position
    seq_lens[b] - 1, slot slot_mapping[b]), then decodes q; writes fp32 out [B][Hq][D]."""
    _check(lib.oscar_append_decode(ctypes.byref(_dims(dims)), int(batch), int(max_seq_len), int(pages_per_split),
                                   _ptr(q), _ptr(k), _ptr(v), _ptr(R_k), _ptr(R_v), _ptr(clip_k), _ptr(clip_v),
                                   _ptr(offset_k), _ptr(slot_mapping), _ptr(int2_pages), _ptr(scale_zero_pages),
                                   _ptr(bf16_sink), _ptr(bf16_window), _ptr(page_table), _ptr(seq_lens),
                                   int(sink_len), int(window_len), float(sm_scale), _ptr(out), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
           "oscar_append_decode")


def oscar_extend_workspace_bytes(dims, num_rows, max_seq_len, pages_per_split, sink_len, window_len) -> int:
    return int(lib.oscar_extend_workspace_bytes(ctypes.byref(_dims(dims)), int(num_rows), int(max_seq_len),
                                                int(pages_per_split), int(sink_len), int(window_len)))


def oscar_extend(dims, batch, max_seq_len, pages_per_split, q, row_seq, row_pos, R_k, R_v, int2_pages,
                 scale_zero_pages, bf16_sink, bf16_window, page_table, seq_lens, sink_len, window_len, sm_scale, out,
                 workspace, stream=None):
    """Causal attention of query rows q [rows][Hq][D] (row r: sequence row_seq[r],
    position row_pos[r]) over the cache; writes fp32 out [rows][Hq][D]."""
    _check(lib.oscar_extend(ctypes.byref(_dims(dims)), int(batch), int(q.shape[0]), int(max_seq_len),
                            int(pages_per_split), _ptr(q), _ptr(row_seq), _ptr(row_pos), _ptr(R_k), _ptr(R_v),
                            _ptr(int2_pages), _ptr(scale_zero_pages), _ptr(bf16_sink), _ptr(bf16_window),
                            _ptr(page_table), _ptr(seq_lens), int(sink_len), int(window_len), float(sm_scale),
                            _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                            _stream(stream)), "oscar_extend")


def oscar_extend_varlen_workspace_bytes(dims, num_rows, max_seq_len, pages_per_split, sink_len, window_len) -> int:
    return int(lib.oscar_extend_varlen_workspace_bytes(ctypes.byref(_dims(dims)), int(num_rows), int(max_seq_len),
                                                       int(pages_per_split), int(sink_len), int(window_len)))


def oscar_extend_varlen(dims, batch, max_seq_len, max_rows_per_seq, pages_per_split, q, q_start, R_k, R_v, int2_pages,
                        scale_zero_pages, bf16_sink, bf16_window, page_table, seq_lens, sink_len, window_len, sm_scale,
                        out, workspace, stream=None):
    """Causal attention of the rows q [rows][Hq][D]: rows q_start[b] .. q_start[b+1]-1 are
    the last positions of sequence b; writes fp32 out [rows][Hq][D]."""
    _check(lib.oscar_extend_varlen(ctypes.byref(_dims(dims)), int(batch), int(q.shape[0]), int(max_seq_len),
                                   int(max_rows_per_seq), int(pages_per_split), _ptr(q), _ptr(q_start), _ptr(R_k),
                                   _ptr(R_v), _ptr(int2_pages), _ptr(scale_zero_pages), _ptr(bf16_sink),
                                   _ptr(bf16_window), _ptr(page_table), _ptr(seq_lens), int(sink_len),
                                   int(window_len), float(sm_scale), _ptr(out), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
           "oscar_extend_varlen")


OSCAR_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def oscar_decode_noalloc(dims, batch, max_seq_len, pages_per_split, q, R_k, R_v, int2_pages, scale_zero_pages,
                         bf16_sink, bf16_window, page_table, seq_lens, sink_len, window_len, sm_scale, out,
                         stream=None):
    """oscar_decode with the library's static device scratch instead of a caller
    workspace (for callers that cannot allocate device memory; calls must not
    overlap on the GPU)."""
    _check(lib.oscar_decode_noalloc(ctypes.byref(_dims(dims)), int(batch), int(max_seq_len), int(pages_per_split),
                                    _ptr(q), _ptr(R_k), _ptr(R_v), _ptr(int2_pages), _ptr(scale_zero_pages),
                                    _ptr(bf16_sink), _ptr(bf16_window), _ptr(page_table), _ptr(seq_lens),
                                    int(sink_len), int(window_len), float(sm_scale), _ptr(out), _stream(stream)),
           "oscar_decode_noalloc")


def oscar_bf16_append(dims, k, v, slot_mapping, bf16_pages, stream=None):
    _check(lib.oscar_bf16_append(ctypes.byref(_dims(dims)), int(k.shape[0]), _ptr(k), _ptr(v), _ptr(slot_mapping),
                                 _ptr(bf16_pages), _stream(stream)), "oscar_bf16_append")


def oscar_bf16_decode_workspace_bytes(dims, batch, max_seq_len, pages_per_split) -> int:
    return int(lib.oscar_bf16_decode_workspace_bytes(ctypes.byref(_dims(dims)), int(batch), int(max_seq_len),
                                                     int(pages_per_split)))


def oscar_bf16_decode(dims, batch, max_seq_len, pages_per_split, q, bf16_pages, page_table, seq_lens, sm_scale, out,
                      workspace, stream=None):
    _check(lib.oscar_bf16_decode(ctypes.byref(_dims(dims)), int(batch), int(max_seq_len), int(pages_per_split),
                                 _ptr(q), _ptr(bf16_pages), _ptr(page_table), _ptr(seq_lens), float(sm_scale),
                                 _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream)), "oscar_bf16_decode")


def oscar_calibrate_workspace_bytes(dims, num_samples) -> int:
    return int(lib.oscar_calibrate_workspace_bytes(ctypes.byref(_dims(dims)), int(num_samples)))


def _calib_out(o):
    if o is None:
        return None
    return ctypes.byref(oscar_calib_out_t(*(_ptr(o.get(n)) for n in ("R", "clip", "eigenvalues", "cov", "sweeps"))))


def oscar_calibrate(dims, num_samples, k, v, centered, clip_quantile, out_k, out_v, workspace, stream=None):
    """Covariance, spectral rotation and quantile clipping thresholds per KV head from
    bf16 samples [N][Hkv][D]; ``out_k`` / ``out_v``: dicts of output tensors (keys R,
    clip and optionally eigenvalues, cov, sweeps) or None with ``k`` / ``v`` None."""
    _check(lib.oscar_calibrate(ctypes.byref(_dims(dims)), int(num_samples), _ptr(k), _ptr(v), int(centered),
                               float(clip_quantile), _calib_out(out_k), _calib_out(out_v), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream)), "oscar_calibrate")


def oscar_test_stall_page_waits(cycles: int) -> None:
    """Test hook: INT2 split warps of later decodes give up their first page wait
    after ``cycles`` clock cycles (0 = normal operation)."""
    _check(lib.oscar_test_stall_page_waits(int(cycles)), "oscar_test_stall_page_waits")


def oscar_device_errors(reset: bool = False) -> int:
    flags = ctypes.c_uint32(0)
    _check(lib.oscar_device_errors(ctypes.byref(flags), int(bool(reset))), "oscar_device_errors")
    return int(flags.value)
