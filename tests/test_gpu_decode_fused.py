"""GPU parity of the single-wave fused decode (small batches): INT2 split CTAs
that rotate the query and un-rotate their own output, one BF16 sink/window CTA
per (sequence, KV head), a log-sum-exp merge.  The oracle recomputes every
output from the GPU's own codes and scale/zero (max-abs <= 2e-3, mean-abs
<= 2e-4); each case first checks that the library schedules the fused form."""

import numpy as np
import pytest
import torch

import int2_rotated_kv_append_gb300 as ok
from int2_rotated_kv_append_gb300 import synth
from int2_rotated_kv_append_gb300.cache import Int2Cache
from parity import compare_decode, oracle_decode_on_gpu_cache

pytestmark = pytest.mark.gpu


def _plan(w, pps, max_seq_len=None):
    msl = w.max_seq_len if max_seq_len is None else max_seq_len
    return ok.oscar_decode_plan(w.dims, w.batch, msl, pps, w.sink_len, w.window_len)


def _built(w, pps=0):
    cache = Int2Cache(w, pages_per_split=pps)
    cache.prefill()
    return cache


def test_plan_fused_for_small_batches_only():
    def plan(Hq, B, L, W, pps=0):
        dims = ok.make_dims(Hq, 8, 128, 16, 64, B * (L // 16 + 1), L // 16 + 1)
        return ok.oscar_decode_plan(dims, B, L, pps, 64, W)
    assert plan(32, 1, 32768, 128)["fused"] == 1           # batch 1, 32K
    assert plan(32, 2, 32768, 128)["fused"] == 1           # batch 2, 32K: 8 splits of 255 pages
    assert plan(32, 3, 32768, 128)["fused"] == 0           # batch 3: 5 splits per unit, the general grid
    assert plan(32, 64, 16384, 128)["fused"] == 0          # 512 (sequence, KV head) units: more than one wave
    assert plan(64, 4, 131072, 256)["fused"] == 0          # batch 4, 131K, GQA 8: 3 splits per unit
    assert plan(64, 1, 131072, 256)["fused"] == 1          # batch 1, 131K, GQA 8: 18 splits of 455 pages
    assert plan(64, 4, 131072, 256, pps=2800)["fused"] == 1  # the same with the split size given
    assert plan(32, 1, 32768, 128, pps=1)["fused"] == 0    # 2036 splits of one page: more than one wave


@pytest.mark.parametrize("pps", [0, 8, 40, 400])
def test_fused_split_counts(pps):
    w = synth.make_workload(num_q_heads=8, num_kv_heads=2, head_dim=128, group_size=64, sink_len=16, window_len=64,
                            seq_lens=[5000], seed=31)
    plan = _plan(w, pps)
    assert plan["fused"] == 1, plan
    cache = _built(w, pps)
    out = cache.decode(w.q.cuda())
    compare_decode(out, oracle_decode_on_gpu_cache(w, cache))


@pytest.mark.parametrize("Hq,H,G", [(8, 8, 64), (16, 8, 128), (12, 4, 64), (24, 4, 64), (64, 8, 64), (64, 8, 128),
                                    (7, 1, 64)])
def test_fused_gqa_shapes_and_edge_lengths(Hq, H, G):
    S, W = 5, 19
    # as many sequences as keep 8 split CTAs per (sequence, KV head) unit (the
    # automatic fused plan): the edge lengths with 4 KV heads or fewer
    lens = [3000, S + W + 1, 0, 1, S - 1, 16 * 9 + 3]
    w = synth.make_workload(num_q_heads=Hq, num_kv_heads=H, head_dim=128, group_size=G, sink_len=S, window_len=W,
                            seq_lens=lens[:max(1, 152 // (9 * H))], seed=Hq + H + G, spare_pages=3)
    assert _plan(w, 0)["fused"] == 1
    cache = _built(w)
    out = cache.decode(w.q.cuda())
    compare_decode(out, oracle_decode_on_gpu_cache(w, cache))


@pytest.mark.parametrize("S,W", [(0, 0), (64, 0), (0, 256)])
def test_fused_without_sink_or_window(S, W):
    w = synth.make_workload(num_q_heads=32, num_kv_heads=8, head_dim=128, group_size=64, sink_len=S, window_len=W,
                            seq_lens=[4100, 333], seed=S + W + 1)
    assert _plan(w, 0)["fused"] == 1
    cache = _built(w)
    out = cache.decode(w.q.cuda())
    compare_decode(out, oracle_decode_on_gpu_cache(w, cache))


def test_fused_lengths_below_the_bound():
    # splits are planned over max_seq_len = 2000; the decoded lengths are shorter (the
    # sink/window buffers hold what they hold: GPU and oracle read the same rows)
    w = synth.make_workload(num_q_heads=32, num_kv_heads=8, head_dim=128, group_size=64, sink_len=64, window_len=128,
                            seq_lens=[2000, 900], seed=33)
    cache = _built(w)
    assert _plan(w, 0, 2000)["fused"] == 1
    lens = torch.tensor([1500, 611], dtype=torch.int32)
    out = cache.decode(w.q.cuda(), seq_lens=lens.cuda(), max_seq_len=2000)
    compare_decode(out, oracle_decode_on_gpu_cache(w, cache, seq_lens=lens))


def test_fused_bad_page_id_is_flagged_and_finite():
    w = synth.make_workload(num_q_heads=8, num_kv_heads=2, head_dim=128, group_size=64, sink_len=8, window_len=16,
                            seq_lens=[900], seed=34)
    assert _plan(w, 0)["fused"] == 1
    cache = _built(w)
    ok.oscar_device_errors(reset=True)
    pt = cache.page_table.clone()
    pt[0, 20] = w.num_pages + 7
    cache.page_table = pt
    out = cache.decode(w.q.cuda())
    assert ok.oscar_device_errors(reset=True) & ok.OSCAR_DEVERR_PAGE_ID
    assert torch.isfinite(out).all()


def test_fused_repeat_calls_bit_identical():
    w = synth.make_config(1, device="cuda")
    cache = _built(w)
    a = cache.decode(w.q).clone()
    b = cache.decode(w.q).clone()
    assert torch.equal(a, b)
