"""The C-ABI library loads, exports every declared entry point, and rejects bad
arguments on the host (no GPU needed: nothing is launched)."""

import ctypes
import os
import re

import pytest

import int2_rotated_kv_append_gb300 as ok
from int2_rotated_kv_append_gb300 import build

HEADER = os.path.join(build.INCLUDE, "oscar.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ok.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(oscar_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("oscar_append", "oscar_decode", "oscar_decode_workspace_bytes", "oscar_bf16_decode"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def _dims(**kw):
    d = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16, group_size=64, num_pages=100,
             max_pages_per_seq=20)
    d.update(kw)
    return ok.make_dims(**d)


P = ctypes.c_void_p(16)  # never dereferenced: validation fails before any launch


def _append(lib, dims, T=4, ptr=P, offset=None):
    return lib.oscar_append(ctypes.byref(dims) if dims is not None else None, T, ptr, ptr, ptr, ptr, ptr, ptr,
                            offset, None, ptr, ptr, ptr, None)


def test_append_validation(lib):
    assert _append(lib, None) == ok.OSCAR_ERR_INVALID_ARG
    assert _append(lib, _dims(head_dim=96, group_size=32)) == ok.OSCAR_ERR_UNSUPPORTED
    assert _append(lib, _dims(num_q_heads=30)) == ok.OSCAR_ERR_INVALID_ARG
    assert _append(lib, _dims(group_size=48)) == ok.OSCAR_ERR_INVALID_ARG
    assert _append(lib, _dims(group_size=16)) == ok.OSCAR_ERR_UNSUPPORTED
    assert _append(lib, _dims(page_size=32)) == ok.OSCAR_ERR_UNSUPPORTED
    assert _append(lib, _dims(num_q_heads=128)) == ok.OSCAR_ERR_UNSUPPORTED  # GQA 16
    assert _append(lib, _dims(num_pages=0)) == ok.OSCAR_ERR_INVALID_ARG
    assert _append(lib, _dims(), T=-1) == ok.OSCAR_ERR_INVALID_ARG
    assert _append(lib, _dims(), T=0) == ok.OSCAR_OK  # no-op
    assert _append(lib, _dims(), ptr=None) == ok.OSCAR_ERR_INVALID_ARG
    assert _append(lib, _dims(), ptr=ctypes.c_void_p(18)) == ok.OSCAR_ERR_INVALID_ARG  # misaligned
    assert _append(lib, _dims(), offset=ctypes.c_void_p(24)) == ok.OSCAR_ERR_INVALID_ARG  # misaligned key offset


def test_append_rejects_each_misaligned_buffer(lib):
    # k, v, R_k, R_v and both pools: each one 2 bytes off a 16-byte boundary is refused.
    bad = ctypes.c_void_p(18)
    for i in (0, 1, 2, 3, 7, 8):
        a = [P] * 9
        a[i] = bad
        rc = lib.oscar_append(ctypes.byref(_dims()), 4, a[0], a[1], a[2], a[3], a[4], a[5], None, None, a[6], a[7],
                              a[8], None)
        assert rc == ok.OSCAR_ERR_INVALID_ARG, i
    d = _dims(); bd = ok.OSCAR_ERR_INVALID_ARG
    assert lib.oscar_bf16_append(ctypes.byref(d), 4, bad, P, P, P, None) == bd
    assert lib.oscar_bf16_append(ctypes.byref(d), 4, P, P, P, bad, None) == bd


def _append_mixed(lib, dims, T=4, ptr=P, batch=2, S=4, W=8, sink=P, win=P, ids=P, offset=None):
    return lib.oscar_append_mixed(ctypes.byref(dims), T, ptr, ptr, ptr, ptr, ptr, ptr, offset, None, ptr, ids, ids,
                                  ids, batch, S, W, ptr, ptr, sink, win, None)


def test_append_mixed_validation(lib):
    assert _append_mixed(lib, _dims(), batch=-1) == ok.OSCAR_ERR_INVALID_ARG
    assert _append_mixed(lib, _dims(), S=-1) == ok.OSCAR_ERR_INVALID_ARG
    assert _append_mixed(lib, _dims(), W=-2) == ok.OSCAR_ERR_INVALID_ARG
    assert _append_mixed(lib, _dims(), batch=0) == ok.OSCAR_ERR_INVALID_ARG  # tokens but no sequences
    assert _append_mixed(lib, _dims(), ids=None) == ok.OSCAR_ERR_INVALID_ARG
    assert _append_mixed(lib, _dims(), sink=None) == ok.OSCAR_ERR_INVALID_ARG
    assert _append_mixed(lib, _dims(), win=None) == ok.OSCAR_ERR_INVALID_ARG
    assert _append_mixed(lib, _dims(), S=0, sink=None, W=0, win=None, T=0) == ok.OSCAR_OK  # no-op
    assert _append_mixed(lib, _dims(head_dim=96, group_size=32)) == ok.OSCAR_ERR_UNSUPPORTED
    assert _append_mixed(lib, _dims(), ptr=None) == ok.OSCAR_ERR_INVALID_ARG
    assert _append_mixed(lib, _dims(), sink=ctypes.c_void_p(20)) == ok.OSCAR_ERR_INVALID_ARG  # misaligned
    assert _append_mixed(lib, _dims(), win=ctypes.c_void_p(24)) == ok.OSCAR_ERR_INVALID_ARG
    assert _append_mixed(lib, _dims(), offset=ctypes.c_void_p(40)) == ok.OSCAR_ERR_INVALID_ARG


def test_extend_validation(lib):
    d = _dims()
    def ext(batch=2, rows=3, rs=P, rp=P, ws_bytes=1 << 30):
        return lib.oscar_extend(ctypes.byref(d), batch, rows, 100, 8, P, rs, rp, P, P, P, P, P, P, P, P, 4, 8, 0.0, P,
                                ctypes.c_void_p(256), ws_bytes, None)
    assert ext(rows=0) == ok.OSCAR_OK  # nothing to attend
    assert ext(rs=None) == ok.OSCAR_ERR_INVALID_ARG
    assert ext(rp=None) == ok.OSCAR_ERR_INVALID_ARG
    assert ext(batch=0) == ok.OSCAR_ERR_INVALID_ARG  # rows but no sequences
    assert ext(rows=-1) == ok.OSCAR_ERR_INVALID_ARG
    need = lib.oscar_extend_workspace_bytes(ctypes.byref(d), 3, 100, 8, 4, 8)
    assert need > 0 and lib.oscar_decode_workspace_bytes(ctypes.byref(d), 3, 100, 8, 4, 8) > 0
    assert ext(ws_bytes=need - 1) == ok.OSCAR_ERR_WORKSPACE


def test_extend_varlen_validation(lib):
    d = _dims()
    def ext(batch=2, rows=3, mr=2, qs=P, ws_bytes=1 << 30):
        return lib.oscar_extend_varlen(ctypes.byref(d), batch, rows, 100, mr, 8, P, qs, P, P, P, P, P, P, P, P, 4, 8,
                                       0.0, P, ctypes.c_void_p(256), ws_bytes, None)
    assert ext(rows=0) == ok.OSCAR_OK
    assert ext(qs=None) == ok.OSCAR_ERR_INVALID_ARG
    assert ext(batch=0) == ok.OSCAR_ERR_INVALID_ARG
    assert ext(mr=0) == ok.OSCAR_ERR_INVALID_ARG
    assert ext(rows=-1) == ok.OSCAR_ERR_INVALID_ARG
    need = lib.oscar_extend_varlen_workspace_bytes(ctypes.byref(d), 3, 100, 8, 4, 8)
    assert need > lib.oscar_extend_workspace_bytes(ctypes.byref(d), 3, 100, 8, 4, 8) > 0
    assert ext(ws_bytes=need - 1) == ok.OSCAR_ERR_WORKSPACE


def _decode(lib, dims, batch=2, msl=100, pps=8, S=4, W=8, ws_bytes=1 << 30, ws=ctypes.c_void_p(256), sink=P):
    return lib.oscar_decode(ctypes.byref(dims), batch, msl, pps, P, P, P, P, P, sink, P, P, P, S, W, 0.0, P, ws,
                            ws_bytes, None)


def test_decode_validation(lib):
    d = _dims()
    assert _decode(lib, d, batch=-1) == ok.OSCAR_ERR_INVALID_ARG
    assert _decode(lib, d, batch=0) == ok.OSCAR_OK
    assert _decode(lib, d, msl=20 * 16 + 1) == ok.OSCAR_ERR_INVALID_ARG  # beyond the page table
    assert _decode(lib, d, S=-1) == ok.OSCAR_ERR_INVALID_ARG
    assert _decode(lib, d, W=-2) == ok.OSCAR_ERR_INVALID_ARG
    assert _decode(lib, d, pps=-1) == ok.OSCAR_ERR_INVALID_ARG
    assert _decode(lib, d, sink=None) == ok.OSCAR_ERR_INVALID_ARG  # S > 0 needs a sink buffer
    assert _decode(lib, d, ws=ctypes.c_void_p(260)) == ok.OSCAR_ERR_INVALID_ARG  # misaligned workspace
    need = lib.oscar_decode_workspace_bytes(ctypes.byref(d), 2, 100, 8, 4, 8)
    assert need > 0
    assert _decode(lib, d, ws_bytes=need - 1) == ok.OSCAR_ERR_WORKSPACE


def test_workspace_sizes(lib):
    d = _dims(max_pages_per_seq=2048)
    a = lib.oscar_decode_workspace_bytes(ctypes.byref(d), 1, 32768, 64, 64, 128)
    b = lib.oscar_decode_workspace_bytes(ctypes.byref(d), 1, 32768, 16, 64, 128)
    assert 0 < a < b and a % 256 == 0
    assert lib.oscar_decode_workspace_bytes(ctypes.byref(d), 1, 2048 * 16 + 1, 64, 64, 128) == 0
    assert lib.oscar_bf16_decode_workspace_bytes(ctypes.byref(d), 1, 32768, 64) > 0


def test_status_strings(lib):
    for s in range(5):
        assert ok.status_string(s).startswith("OSCAR")


def test_calibrate_validation(lib):
    d = _dims()
    out = ok.oscar_calib_out_t(P, P, None, None, None)
    bad_R = ok.oscar_calib_out_t(ctypes.c_void_p(24), P, None, None, None)
    no_clip = ok.oscar_calib_out_t(P, None, None, None, None)
    need = lib.oscar_calibrate_workspace_bytes(ctypes.byref(d), 1000)
    assert need > 0
    assert lib.oscar_calibrate_workspace_bytes(ctypes.byref(d), 0) == 0
    assert lib.oscar_calibrate_workspace_bytes(ctypes.byref(d), 2000) > need

    def cal(N=1000, k=P, v=P, centered=1, q=0.99, ok_=ctypes.byref(out), ov=ctypes.byref(out),
            ws=ctypes.c_void_p(256), ws_bytes=1 << 40, dims=d):
        return lib.oscar_calibrate(ctypes.byref(dims), N, k, v, centered, q, ok_, ov, ws, ws_bytes, None)

    E = ok.OSCAR_ERR_INVALID_ARG
    assert cal(N=0) == E
    assert cal(N=-5) == E
    assert cal(N=1 << 31) == E
    assert cal(N=(1 << 31) - 255) == E          # the largest accepted is 2^31 - 256
    assert cal(k=None) == E                       # k missing but out_k given
    assert cal(ov=None) == E                      # v given but out_v missing
    assert cal(k=None, v=None, ok_=None, ov=None) == E  # nothing to calibrate
    assert cal(q=0.0) == E
    assert cal(q=1.5) == E
    assert cal(q=float("nan")) == E
    assert cal(centered=2) == E
    assert cal(ok_=ctypes.byref(bad_R)) == E      # misaligned R
    assert cal(ov=ctypes.byref(no_clip)) == E
    assert cal(k=ctypes.c_void_p(40)) == E        # misaligned samples
    assert cal(ws=None) == E
    assert cal(ws=ctypes.c_void_p(264)) == E      # misaligned workspace
    assert cal(dims=_dims(head_dim=96, group_size=32)) == ok.OSCAR_ERR_UNSUPPORTED
    assert cal(ws_bytes=need - 1) == ok.OSCAR_ERR_WORKSPACE


def test_decode_plan_respects_grid_limits(lib):
    # the split index is a grid dimension (<= 65535): a plan with more splits is refused
    d = _dims(max_pages_per_seq=70000)
    assert lib.oscar_decode_workspace_bytes(ctypes.byref(d), 1, 70000 * 16, 1, 64, 128) == 0
    assert lib.oscar_decode_workspace_bytes(ctypes.byref(d), 1, 70000 * 16, 2, 64, 128) > 0
    assert _decode(lib, d, batch=1, msl=70000 * 16, pps=1, S=64, W=128) == ok.OSCAR_ERR_INVALID_ARG


def test_decode_plan_fused_form_rules(lib):
    # Host logic only (no kernel runs): the automatic split size takes the fused
    # single-wave form only with at least 8 split CTAs per (sequence, KV head) of at
    # most 960 pages (512 at GQA 8); a split size given by the caller is kept.
    def plan(Hq, B, L, W, pps=0):
        dims = ok.make_dims(Hq, 8, 128, 16, 64, B * (L // 16 + 1), L // 16 + 1)
        return ok.oscar_decode_plan(dims, B, L, pps, 64, W)
    p1 = plan(32, 1, 32768, 128)
    assert p1["fused"] == 1 and p1["splits"] >= 8 and p1["pages_per_split"] <= 960
    assert plan(32, 3, 32768, 128)["fused"] == 0      # about 5 splits per unit
    assert plan(32, 2, 131072, 128)["fused"] == 0     # about 1023 pages per split
    assert plan(64, 2, 131072, 256)["fused"] == 0     # GQA 8: more than 512 pages per split
    assert plan(64, 1, 131072, 256)["fused"] == 1     # GQA 8: about 455 pages per split
    assert plan(64, 4, 131072, 256, pps=2800)["fused"] == 1
