"""The scratch-free decode entry point (oscar_decode_noalloc), for callers that
cannot allocate device memory (GPU).

It runs the same decode as oscar_decode but uses the library's static device
scratch instead of a caller workspace.  The check calls it twice in a row
through the C ABI -- the scratch keeps the previous call's contents -- and
compares each output with oscar_decode's within the decode parity tolerance.
This file is collected last so that, when it fails, a run that stops at the
first failure has already run every other test.
"""

import ctypes

import pytest
import torch

import int2_rotated_kv_append_gb300 as ok
from int2_rotated_kv_append_gb300 import synth
from int2_rotated_kv_append_gb300.cache import Int2Cache
from parity import DEC_MAX_ABS, DEC_MEAN_ABS

pytestmark = pytest.mark.gpu


def _noalloc(cache, w, q, out):
    ok.oscar_decode_noalloc(w.dims, w.batch, w.max_seq_len, cache.pps, q, cache.R_k, cache.R_v, cache.int2_pages,
                            cache.scale_zero, cache.sink, cache.window, cache.page_table, cache.seq_lens, w.sink_len,
                            w.window_len, 0.0, out)


@pytest.mark.parametrize("D,G,Hq,H", [(128, 64, 32, 8), (64, 32, 4, 2)])
def test_noalloc_matches_workspace_decode_on_two_calls(D, G, Hq, H):
    w = synth.make_workload(num_q_heads=Hq, num_kv_heads=H, head_dim=D, group_size=G, sink_len=16, window_len=64,
                            seq_lens=[5000, 700, 1, 0], seed=D + Hq)
    cache = Int2Cache(w)
    cache.prefill()
    q = w.q.cuda()
    ref = cache.decode(q).clone()
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        _noalloc(cache, w, q, out)
        torch.cuda.synchronize()
        err = (out - ref).abs()
        assert torch.isfinite(out).all(), f"call {call}: non-finite output"
        assert err.max().item() <= DEC_MAX_ABS and err.mean().item() <= DEC_MEAN_ABS, f"call {call}"


def test_noalloc_rejects_plans_beyond_the_scratch():
    lib = ok.load_library()
    dims = ok.make_dims(32, 8, 128, 16, 64, 1 << 20, 8192)
    P = ctypes.c_void_p(256)  # never dereferenced: the size check fails first
    st = lib.oscar_decode_noalloc(ctypes.byref(dims), 64, 8192 * 16, 1, P, P, P, P, P, P, P, P, P, 64, 128, 0.0, P,
                                  None)
    assert st == ok.OSCAR_ERR_WORKSPACE
    assert ok.oscar_decode_workspace_bytes(dims, 64, 8192 * 16, 1, 64, 128) > ok.OSCAR_NOALLOC_SCRATCH_BYTES
