"""GPU parity of oscar_decode: the oracle recomputes every checked output from
the GPU's own codes and scale/zero (max-abs <= 2e-3, mean-abs <= 2e-4)."""

import numpy as np
import pytest
import torch

import int2_rotated_kv_append_gb300 as ok
from int2_rotated_kv_append_gb300 import synth
from int2_rotated_kv_append_gb300.cache import Int2Cache
from parity import compare_decode, oracle_decode_on_gpu_cache

pytestmark = pytest.mark.gpu


def _built(w, pps=None):
    cache = Int2Cache(w, pages_per_split=pps)
    cache.prefill()
    return cache


def test_decode_tiny_config():
    w = synth.make_config(0)
    cache = _built(w)
    out = cache.decode(w.q.cuda())
    compare_decode(out, oracle_decode_on_gpu_cache(w, cache))


def test_decode_batch1_32k_config_all_heads():
    w = synth.make_config(1, device="cuda")
    cache = _built(w)
    out = cache.decode(w.q)
    compare_decode(out, oracle_decode_on_gpu_cache(w, cache))


def test_decode_batch64_config_sampled():
    w = synth.make_config(2, device="cuda")
    cache = _built(w)
    out = cache.decode(w.q)
    lens = w.seq_lens.numpy()
    # 16 sequences (the shortest, the longest and 14 drawn) x 3 query heads of different KV heads
    rest = [int(b) for b in np.random.default_rng(2).permutation(len(lens)) if b not in (np.argmin(lens), np.argmax(lens))]
    bs = [int(np.argmin(lens)), int(np.argmax(lens))] + rest[:14]
    pairs = [(b, (5 * b + 11 * j) % 32) for b in bs for j in range(3)]
    compare_decode(out, oracle_decode_on_gpu_cache(w, cache, pairs=pairs), pairs=pairs)


def test_decode_131k_gqa8_config_sampled():
    w = synth.make_config(3, device="cuda")
    cache = _built(w)
    out = cache.decode(w.q)
    # every (sequence, KV head) once, a different query head of the GQA group each time, plus the group ends
    pairs = [(b, 8 * h + (3 * b + h) % 8) for b in range(4) for h in range(8)] + [(0, 0), (1, 7), (2, 56), (3, 63)]
    compare_decode(out, oracle_decode_on_gpu_cache(w, cache, pairs=pairs), pairs=pairs)


@pytest.mark.parametrize("Hq,H,B", [(6, 1, 311), (4, 2, 157), (8, 8, 40)])
def test_decode_large_batch_merge(Hq, H, B):
    # At least two (sequence, KV head) units per SM: the merge takes the GQA groups
    # of several sequences per CTA (16 query heads; 12 for GQA 6), the last CTA ragged.
    g = np.random.default_rng(B + Hq)
    lens = g.integers(1, 200, B).tolist()
    w = synth.make_workload(num_q_heads=Hq, num_kv_heads=H, head_dim=128, group_size=64, sink_len=8, window_len=16,
                            seq_lens=lens, seed=B, device="cuda")
    cache = _built(w)
    out = cache.decode(w.q)
    compare_decode(out, oracle_decode_on_gpu_cache(w, cache))


@pytest.mark.parametrize("D,G,Hq,H", [(64, 32, 1, 1), (64, 64, 4, 2), (128, 64, 8, 2), (128, 32, 6, 3),
                                      (128, 128, 8, 1), (128, 64, 2, 2)])
def test_decode_edge_lengths(D, G, Hq, H):
    # Lengths around every boundary: empty, single token, inside the sink, at the
    # sink/window edge, bulk starting mid-page, window ends mid-page, multi-split.
    S, W = 5, 19
    lens = [0, 1, S - 1, S, S + 1, S + W, S + W + 1, S + W + 16, 16 * 9 + 3, 700]
    w = synth.make_workload(num_q_heads=Hq, num_kv_heads=H, head_dim=D, group_size=G, sink_len=S, window_len=W,
                            seq_lens=lens, seed=D + Hq, spare_pages=5)
    for pps in (0, 1, 3):
        cache = _built(w, pps=pps)
        out = cache.decode(w.q.cuda())
        compare_decode(out, oracle_decode_on_gpu_cache(w, cache))


@pytest.mark.parametrize("S,W", [(0, 0), (0, 32), (16, 0), (64, 256)])
def test_decode_sink_window_extremes(S, W):
    w = synth.make_workload(num_q_heads=8, num_kv_heads=2, head_dim=128, group_size=64, sink_len=S, window_len=W,
                            seq_lens=[300, 1000, 77], seed=S + W)
    cache = _built(w)
    out = cache.decode(w.q.cuda())
    compare_decode(out, oracle_decode_on_gpu_cache(w, cache))


def test_decode_split_size_invariance():
    w = synth.make_workload(num_q_heads=8, num_kv_heads=2, head_dim=128, group_size=64, sink_len=16, window_len=32,
                            seq_lens=[3000, 1234], seed=11)
    outs = []
    for pps in (1, 2, 7, 64, 0):
        cache = _built(w, pps=pps)
        out = cache.decode(w.q.cuda())
        compare_decode(out, oracle_decode_on_gpu_cache(w, cache))
        outs.append(out.cpu())
    # fp16 hi+lo operands (about 22 bits) and tensor-core fp32 accumulation: split
    # sizes agree to ~1e-5; the bound is 20x below the 2e-3 parity tolerance.
    for o in outs[1:]:
        assert torch.max(torch.abs(o - outs[0])).item() <= 1e-4


def test_plan_fills_whole_waves_at_the_split_cap():
    # batch 16 at 8K: one wave at the 128-page cap would be 512 split CTAs and 256
    # sink/window CTAs, a few more than one wave; the plan takes smaller splits that
    # fill two waves instead
    dims = ok.make_dims(32, 8, 128, 16, 64, 16 * 513, 513)
    plan = ok.oscar_decode_plan(dims, 16, 8192, 0, 64, 128)
    assert plan["fused"] == 0 and plan["pages_per_split"] < 128, plan
    # batch 64 with 16K sequences keeps splits near the cap
    dims = ok.make_dims(32, 8, 128, 16, 64, 64 * 1025, 1025)
    assert ok.oscar_decode_plan(dims, 64, 16384, 0, 64, 128)["pages_per_split"] >= 120


@pytest.mark.parametrize("Hq,H,pps", [(8, 2, 4), (16, 2, 0), (4, 4, 1)])
def test_decode_batch_permutation_bit_identical(Hq, H, pps):
    # Variable lengths give the INT2 splits of a decode different page counts and the
    # CTAs of a sequence different places in the grid; a permuted batch must give every
    # sequence bit-identical outputs, and both match the oracle.  Empty splits (short
    # sequences) and sequences inside the sink included.
    g = np.random.default_rng(Hq + pps)
    lens = [3, 9, 40] + g.integers(41, 1500, 37).tolist()
    w = synth.make_workload(num_q_heads=Hq, num_kv_heads=H, head_dim=128, group_size=64, sink_len=16, window_len=32,
                            seq_lens=lens, seed=Hq * 3 + pps, device="cuda")
    cache = _built(w, pps=pps)
    out = cache.decode(w.q)
    compare_decode(out, oracle_decode_on_gpu_cache(w, cache))
    perm = torch.as_tensor(g.permutation(len(lens)), device="cuda")
    out_p = torch.empty_like(out)
    ok.oscar_decode(cache.dims, w.batch, w.max_seq_len, cache.pps, w.q[perm].contiguous(), cache.R_k, cache.R_v,
                    cache.int2_pages, cache.scale_zero, cache.sink[perm].contiguous(), cache.window[perm].contiguous(),
                    cache.page_table[perm].contiguous(), cache.seq_lens[perm].contiguous(), w.sink_len, w.window_len,
                    0.0, out_p, cache.workspace(w.max_seq_len))
    assert torch.equal(out_p, out[perm])


def test_decode_page_shuffle_bit_identical():
    w = synth.make_workload(num_q_heads=4, num_kv_heads=1, head_dim=128, group_size=64, sink_len=8, window_len=16,
                            seq_lens=[900], seed=12, spare_pages=10)
    cache = _built(w)
    out1 = cache.decode(w.q.cuda()).clone()
    perm = torch.randperm(w.num_pages, generator=torch.Generator().manual_seed(1))
    codes = cache.int2_pages.view(w.num_pages, -1)
    sz = cache.scale_zero.view(w.num_pages, -1)
    new_codes, new_sz = torch.empty_like(codes), torch.empty_like(sz)
    new_codes[perm.cuda()] = codes
    new_sz[perm.cuda()] = sz
    cache.int2_pages.copy_(new_codes.view(-1))
    cache.scale_zero.copy_(new_sz.view(-1))
    cache.page_table = perm.to(torch.int32)[w.page_table.long().clamp(min=0)].cuda()
    out2 = cache.decode(w.q.cuda())
    assert torch.equal(out1, out2)


def test_decode_bad_page_id_is_flagged_and_finite():
    w = synth.make_workload(num_q_heads=4, num_kv_heads=1, head_dim=64, group_size=32, sink_len=4, window_len=8,
                            seq_lens=[200], seed=13)
    cache = _built(w)
    ok.oscar_device_errors(reset=True)
    pt = cache.page_table.clone()
    pt[0, 3] = w.num_pages + 100
    cache.page_table = pt
    out = cache.decode(w.q.cuda())
    flags = ok.oscar_device_errors(reset=True)
    assert flags & ok.OSCAR_DEVERR_PAGE_ID
    assert torch.isfinite(out).all()


def test_decode_seq_len_over_bound_is_flagged():
    w = synth.make_workload(num_q_heads=2, num_kv_heads=1, head_dim=64, group_size=32, sink_len=4, window_len=8,
                            seq_lens=[100], seed=14)
    cache = _built(w)
    ok.oscar_device_errors(reset=True)
    cache.decode(w.q.cuda(), seq_lens=torch.tensor([150], dtype=torch.int32, device="cuda"), max_seq_len=100)
    assert ok.oscar_device_errors(reset=True) & ok.OSCAR_DEVERR_SEQ_LEN


def test_decode_unattended_bf16_rows_never_read():
    # Sink rows at or past min(S, L) and window slots whose position is below S
    # (or does not exist yet) hold NaN bits: they must not reach the output.
    S, W = 24, 40
    lens = [3, 30, 50, 64, 200]
    w = synth.make_workload(num_q_heads=8, num_kv_heads=2, head_dim=128, group_size=64, sink_len=S, window_len=W,
                            seq_lens=lens, seed=21)
    cache = _built(w)
    nan = torch.tensor(0x7FC0, dtype=torch.int16).view(torch.bfloat16)
    sink, win = cache.sink.clone(), cache.window.clone()
    for b, L in enumerate(lens):
        for p in range(S):
            if p >= min(S, L):
                sink[b, :, :, p, :] = nan
        for r in range(W):
            back = (L - 1 - r) % W
            pos = L - 1 - back
            if L == 0 or pos < S:
                win[b, :, :, r, :] = nan
    cache.sink, cache.window = sink, win
    out = cache.decode(w.q.cuda())
    assert torch.isfinite(out).all()
    compare_decode(out, oracle_decode_on_gpu_cache(w, cache))


def test_decode_after_append_mixed_equals_generator_buffers():
    # sink/window written by oscar_append_mixed give the same decode, bit for bit,
    # as the generator's sink/window of the same tokens
    import int2_rotated_kv_append_gb300 as ok
    S, W = 16, 48
    w = synth.make_workload(num_q_heads=8, num_kv_heads=2, head_dim=128, group_size=64, sink_len=S, window_len=W,
                            seq_lens=[10, 60, 600], seed=23)
    cache = _built(w)
    out_ref = cache.decode(w.q.cuda()).clone()
    sink = torch.zeros_like(cache.sink)
    win = torch.zeros_like(cache.window)
    ok.oscar_append_mixed(w.dims, w.k.cuda(), w.v.cuda(), cache.R_k, cache.R_v, cache.clip_k, cache.clip_v, None,
                          w.slot_mapping.cuda(), w.tok_seq.cuda(), w.tok_pos.cuda(), w.seq_lens.cuda(), S, W,
                          cache.int2_pages, cache.scale_zero, sink, win)
    cache.sink, cache.window = sink, win
    out = cache.decode(w.q.cuda())
    assert torch.equal(out, out_ref)
