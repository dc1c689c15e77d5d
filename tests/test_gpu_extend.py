"""GPU parity of oscar_extend (chunked prefill / extend attention): the oracle
recomputes every output from the GPU's own codes and scale/zero (decode
tolerances: max-abs <= 2e-3, mean-abs <= 2e-4)."""

import numpy as np
import pytest
import torch

import int2_rotated_kv_append_gb300 as ok
from int2_rotated_kv_append_gb300 import synth
from int2_rotated_kv_append_gb300.cache import Int2Cache
from parity import compare_decode, oracle_extend_on_gpu_cache

pytestmark = pytest.mark.gpu


def _rows(lens, S, W, chunk, seed):
    """For each sequence: the last `chunk` positions (the new tokens), plus one row in
    the sink, one in the INT2 bulk and one at the first window position when they exist."""
    g = np.random.default_rng(seed)
    seqs, pos = [], []
    for b, L in enumerate(lens):
        ps = set(range(max(0, L - chunk), L))
        if L > 0:
            ps.add(int(min(S, L) // 2))
        if L > S + W + 2:
            ps.add(int(g.integers(S, L - W)))
            if W > 0:
                ps.add(L - W)
        for p in sorted(ps):
            seqs.append(b)
            pos.append(p)
    return np.array(seqs, np.int32), np.array(pos, np.int32)


@pytest.mark.parametrize("D,G,Hq,H,lens,S,W,chunk", [
    (128, 64, 8, 2, [70, 300, 45, 1200], 8, 24, 5),      # tensor-core INT2 kernel, GQA 4
    (128, 128, 8, 1, [33, 517], 16, 32, 17),             # GQA 8, chunk longer than a page
    (64, 32, 4, 2, [90, 400], 4, 16, 9),                 # CUDA-core split body
    (128, 64, 2, 2, [260, 20], 0, 0, 6),                 # no sink, no window: all INT2
])
def test_extend_matches_oracle(D, G, Hq, H, lens, S, W, chunk):
    w = synth.make_workload(num_q_heads=Hq, num_kv_heads=H, head_dim=D, group_size=G, sink_len=S, window_len=W,
                            seq_lens=lens, seed=D + G + len(lens) + chunk)
    cache = Int2Cache(w)
    cache.prefill()
    rs, rp = _rows(lens, S, W, chunk, seed=chunk)
    g = torch.Generator().manual_seed(7)
    q = torch.randn((len(rs), Hq, D), generator=g).to(torch.bfloat16).cuda()
    out = cache.extend(q, torch.as_tensor(rs).cuda(), torch.as_tensor(rp).cuda())
    torch.cuda.synchronize()
    compare_decode(out, oracle_extend_on_gpu_cache(w, cache, q, rs, rp))


def test_extend_last_rows_equal_decode():
    # one row per sequence at position L - 1 with the decode's queries.  With one-page
    # splits the decode takes the general form, the extend's plan and kernels: the same
    # outputs bit for bit.  With the automatic split the decode runs the single-wave
    # form (another summation order): equal within the split-size invariance bound.
    w = synth.make_workload(num_q_heads=8, num_kv_heads=2, head_dim=128, group_size=64, sink_len=8, window_len=24,
                            seq_lens=[70, 300, 45, 1200], seed=5)
    rs = torch.arange(w.batch, dtype=torch.int32).cuda()
    rp = (w.seq_lens - 1).to(torch.int32).cuda()
    cache = Int2Cache(w, pages_per_split=1)
    cache.prefill()
    assert ok.oscar_decode_plan(w.dims, w.batch, w.max_seq_len, 1, w.sink_len, w.window_len)["fused"] == 0
    dec = cache.decode(w.q.cuda())
    ext = cache.extend(w.q.cuda(), rs, rp)
    torch.cuda.synchronize()
    assert torch.equal(dec, ext)
    auto = Int2Cache(w, pages_per_split=0)
    auto.int2_pages, auto.scale_zero, auto.sink, auto.window = cache.int2_pages, cache.scale_zero, cache.sink, cache.window
    assert ok.oscar_decode_plan(w.dims, w.batch, w.max_seq_len, 0, w.sink_len, w.window_len)["fused"] == 1
    dec_fused = auto.decode(w.q.cuda())
    torch.cuda.synchronize()
    assert torch.max(torch.abs(dec_fused - ext)).item() <= 1e-4


def test_extend_bad_rows_attend_nothing_and_are_flagged():
    w = synth.make_workload(num_q_heads=4, num_kv_heads=1, head_dim=128, group_size=64, sink_len=4, window_len=8,
                            seq_lens=[40, 60], seed=6)
    cache = Int2Cache(w)
    cache.prefill()
    ok.oscar_device_errors(reset=True)
    rs = torch.tensor([0, 2, 1, -1, 1], dtype=torch.int32).cuda()
    rp = torch.tensor([39, 0, 60, 3, 10], dtype=torch.int32).cuda()
    q = torch.randn((5, 4, 128)).to(torch.bfloat16).cuda()
    out = cache.extend(q, rs, rp)
    torch.cuda.synchronize()
    flags = ok.oscar_device_errors(reset=True)
    assert flags & ok.OSCAR_DEVERR_POSITION
    assert torch.all(out[1:4] == 0)
    assert torch.any(out[0] != 0) and torch.all(torch.isfinite(out[4]))


def test_chunked_prefill_flow_append_mixed_then_extend():
    # The serving flow: the cached prefix, then a chunk of new tokens, both appended
    # with oscar_append_mixed (INT2 + sink/window rows); the chunk's query rows then
    # attend causally.  The ring after the two appends equals the one-shot buffers.
    S, W, chunk = 16, 48, 12
    lens = [300, 700, 40]
    w = synth.make_workload(num_q_heads=8, num_kv_heads=2, head_dim=128, group_size=64, sink_len=S, window_len=W,
                            seq_lens=lens, seed=31)
    cache = Int2Cache(w)
    sink = torch.zeros_like(w.sink_window()[0]).cuda()
    win = torch.zeros_like(w.sink_window()[1]).cuda()
    pos = w.tok_pos.numpy()
    seq = w.tok_seq.numpy()
    final = np.array(lens)
    new = pos >= final[seq] - chunk
    for part, seq_lens in ((~new, final - chunk), (new, final)):
        idx = torch.as_tensor(np.nonzero(part)[0])
        ok.oscar_append_mixed(w.dims, w.k[idx].cuda(), w.v[idx].cuda(), cache.R_k, cache.R_v, cache.clip_k,
                              cache.clip_v, None, w.slot_mapping[idx].cuda(), w.tok_seq[idx].cuda(),
                              w.tok_pos[idx].cuda(), torch.as_tensor(seq_lens, dtype=torch.int32).cuda(), S, W,
                              cache.int2_pages, cache.scale_zero, sink, win)
    torch.cuda.synchronize()
    ref_sink, ref_win = w.sink_window()
    assert torch.equal(sink.cpu(), ref_sink) and torch.equal(win.cpu(), ref_win)
    cache.sink, cache.window = sink, win
    rs = np.repeat(np.arange(len(lens), dtype=np.int32), chunk)
    rp = np.concatenate([np.arange(L - chunk, L, dtype=np.int32) for L in lens])
    g = torch.Generator().manual_seed(8)
    q = torch.randn((len(rs), 8, 128), generator=g).to(torch.bfloat16).cuda()
    out = cache.extend(q, torch.as_tensor(rs).cuda(), torch.as_tensor(rp).cuda())
    torch.cuda.synchronize()
    compare_decode(out, oracle_extend_on_gpu_cache(w, cache, q, rs, rp))


@pytest.mark.parametrize("D,G,Hq,H,lens,S,W,chunks", [
    (128, 64, 8, 2, [300, 700, 40, 1200], 16, 48, [5, 17, 0, 40]),   # tiles of 16 rows (GQA 4), ragged, empty
    (128, 128, 16, 2, [500, 90], 8, 24, [9, 1]),                    # tiles of 8 rows (GQA 8)
    (128, 64, 4, 2, [260, 33], 0, 0, [3, 33]),                       # no sink, no window; a whole sequence as rows
    (64, 32, 4, 2, [90, 400], 4, 16, [9, 2]),                        # other shapes: one decode row per query row
])
def test_extend_varlen_matches_oracle(D, G, Hq, H, lens, S, W, chunks):
    w = synth.make_workload(num_q_heads=Hq, num_kv_heads=H, head_dim=D, group_size=G, sink_len=S, window_len=W,
                            seq_lens=lens, seed=sum(chunks) + D + Hq)
    cache = Int2Cache(w)
    cache.prefill()
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    rs = np.repeat(np.arange(len(lens), dtype=np.int32), chunks)
    rp = np.concatenate([np.arange(L - n, L, dtype=np.int32) for L, n in zip(lens, chunks)])
    g = torch.Generator().manual_seed(9)
    q = torch.randn((len(rs), Hq, D), generator=g).to(torch.bfloat16).cuda()
    out = cache.extend_varlen(q, torch.as_tensor(q_start).cuda(), max(chunks))
    torch.cuda.synchronize()
    assert ok.oscar_device_errors(reset=True) == 0
    compare_decode(out, oracle_extend_on_gpu_cache(w, cache, q, rs, rp))


def test_extend_varlen_rows_beyond_the_tokens_are_flagged():
    w = synth.make_workload(num_q_heads=8, num_kv_heads=2, head_dim=128, group_size=64, sink_len=4, window_len=8,
                            seq_lens=[5, 60], seed=12)
    cache = Int2Cache(w)
    cache.prefill()
    ok.oscar_device_errors(reset=True)
    q = torch.randn((9, 8, 128)).to(torch.bfloat16).cuda()
    q_start = torch.tensor([0, 7, 9], dtype=torch.int32).cuda()  # 7 rows for a 5-token sequence
    out = cache.extend_varlen(q, q_start, 7)
    torch.cuda.synchronize()
    assert ok.oscar_device_errors(reset=True) & ok.OSCAR_DEVERR_POSITION
    assert torch.all(out[:2] == 0)            # positions -2 and -1: nothing attended
    assert torch.all(torch.isfinite(out))


def test_extend_varlen_full_workload_sampled():
    # the extend workload the benchmark times: 32 sequences x 8192 cached tokens, the
    # last 16 of each as query rows (tiles of 16 rows), sampled (row, query head) pairs
    B, L, chunk = 32, 8192, 16
    w = synth.make_workload(num_q_heads=32, num_kv_heads=8, head_dim=128, group_size=64, sink_len=64,
                            window_len=128, seq_lens=[L] * B, seed=11, device="cuda")
    cache = Int2Cache(w)
    cache.prefill()
    q_start = torch.arange(0, B * chunk + 1, chunk, dtype=torch.int32, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(3)
    q = torch.randn((B * chunk, 32, 128), generator=g, device="cuda").to(torch.bfloat16)
    ok.oscar_device_errors(reset=True)
    out = cache.extend_varlen(q, q_start, chunk)
    torch.cuda.synchronize()
    assert ok.oscar_device_errors(reset=True) == 0
    rs = np.repeat(np.arange(B, dtype=np.int32), chunk)
    rp = np.tile(np.arange(L - chunk, L, dtype=np.int32), B)
    rng = np.random.default_rng(5)
    rows = sorted(set([0, chunk - 1, B * chunk - 1] + rng.choice(B * chunk, 21, replace=False).tolist()))
    pairs = [(r, int(h)) for r in rows for h in rng.choice(32, 2, replace=False)]
    compare_decode(out, oracle_extend_on_gpu_cache(w, cache, q, rs, rp, pairs=pairs), pairs=pairs)


@pytest.mark.parametrize("G,Hq,H", [(64, 8, 2), (128, 16, 2)])
def test_extend_tiles_exact_maxima_paths(G, Hq, H):
    # The tcgen05 tile kernel keeps a column's running maximum while logits stay within
    # 2^12 of it and V scales within 15.  Values x 64 (no clipping) put every chunk on the
    # exact-maximum path; one key x 16 in the middle of each sequence raises the running
    # maxima far past the margin, so the output accumulator is rescaled mid-split.
    # Scaling the values by 64 scales every output, and its fp32 rounding, by 64: both
    # sides are divided by 64 before the decode bounds are applied.
    lens, chunks = [1500, 700], [16, 9]
    w = synth.make_workload(num_q_heads=Hq, num_kv_heads=H, head_dim=128, group_size=G, sink_len=16, window_len=32,
                            seq_lens=lens, seed=41 + G, clip_frac=None)
    w.v = (w.v.float() * 64).to(torch.bfloat16)
    pos, seq = w.tok_pos.numpy(), w.tok_seq.numpy()
    spike = np.nonzero(((seq == 0) & (pos == 900)) | ((seq == 1) & (pos == 400)))[0]
    k = w.k.float()
    k[torch.as_tensor(spike)] *= 16
    w.k = k.to(torch.bfloat16)
    cache = Int2Cache(w)
    cache.prefill()
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    rs = np.repeat(np.arange(len(lens), dtype=np.int32), chunks)
    rp = np.concatenate([np.arange(L - n, L, dtype=np.int32) for L, n in zip(lens, chunks)])
    g = torch.Generator().manual_seed(10)
    q = torch.randn((len(rs), Hq, 128), generator=g).to(torch.bfloat16).cuda()
    ok.oscar_device_errors(reset=True)
    out = cache.extend_varlen(q, torch.as_tensor(q_start).cuda(), max(chunks))
    torch.cuda.synchronize()
    assert ok.oscar_device_errors(reset=True) == 0
    compare_decode(out / 64, oracle_extend_on_gpu_cache(w, cache, q, rs, rp) / 64)


def test_extend_tiles_page_wait_timeout_is_reported_and_recovers():
    # the test hook stalls the tile kernel's first page wait: the INT2 part is dropped
    # (no sink or window here, so the output is zero), flagged, and the next call matches
    lens, chunk = [900, 400], 16
    w = synth.make_workload(num_q_heads=8, num_kv_heads=2, head_dim=128, group_size=64, sink_len=0, window_len=0,
                            seq_lens=lens, seed=43)
    cache = Int2Cache(w)
    cache.prefill()
    q_start = torch.tensor([0, chunk, 2 * chunk], dtype=torch.int32).cuda()
    q = torch.randn((2 * chunk, 8, 128), generator=torch.Generator().manual_seed(11)).to(torch.bfloat16).cuda()
    before = cache.extend_varlen(q, q_start, chunk).clone()
    assert torch.count_nonzero(before) > 0 and ok.oscar_device_errors(reset=True) == 0
    ok.oscar_test_stall_page_waits(1_000_000)
    try:
        stalled = cache.extend_varlen(q, q_start, chunk).clone()
        torch.cuda.synchronize()
    finally:
        ok.oscar_test_stall_page_waits(0)
    assert ok.oscar_device_errors(reset=True) & ok.OSCAR_DEVERR_TIMEOUT
    assert torch.count_nonzero(stalled) == 0 and torch.isfinite(stalled).all()
    after = cache.extend_varlen(q, q_start, chunk).clone()
    assert ok.oscar_device_errors(reset=True) == 0
    assert torch.equal(after, before)
