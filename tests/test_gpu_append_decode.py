"""GPU parity of oscar_append_decode (one decode step: append each sequence's current
token, then decode).  The cache of every sequence but its last token is built first;
then two copies take the step, one as oscar_append_mixed + oscar_decode and one as
oscar_append_decode.  The BF16 rows must be equal, the codes of the appended tokens
must match the oracle's append (boundary band exempt), and the outputs must be equal
to the two-call step and match the oracle's decode of the resulting cache."""

import numpy as np
import pytest
import torch

import int2_rotated_kv_append_gb300 as ok
from int2_rotated_kv_append_gb300 import synth
from int2_rotated_kv_append_gb300.cache import Int2Cache
from parity import check_append, compare_decode, oracle_decode_on_gpu_cache, pools_to_host

pytestmark = pytest.mark.gpu


def _step_pair(w, pps=0):
    """Cache of all tokens but the last of each sequence, in two copies; the current
    tokens (one per sequence, in sequence order)."""
    d = torch.device("cuda")
    cache = Int2Cache(w, pages_per_split=pps)
    B, H, D = w.batch, w.num_kv_heads, w.head_dim
    cache.sink = torch.zeros((B, 2, H, max(w.sink_len, 1), D), dtype=torch.bfloat16, device=d)
    cache.window = torch.zeros((B, 2, H, max(w.window_len, 1), D), dtype=torch.bfloat16, device=d)
    lens = w.seq_lens.numpy()
    pos, seq = w.tok_pos.numpy(), w.tok_seq.numpy()
    cur = np.array([np.nonzero((seq == b) & (pos == lens[b] - 1))[0][0] for b in range(B)])
    past = np.setdiff1d(np.arange(len(pos)), cur)
    ip = torch.as_tensor(past)
    if len(past):
        ok.oscar_append_mixed(w.dims, w.k[ip].to(d), w.v[ip].to(d), cache.R_k, cache.R_v, cache.clip_k, cache.clip_v,
                              None, w.slot_mapping[ip].to(d), w.tok_seq[ip].to(d), w.tok_pos[ip].to(d),
                              torch.as_tensor(np.maximum(lens - 1, 0), dtype=torch.int32).to(d), w.sink_len,
                              w.window_len, cache.int2_pages, cache.scale_zero, cache.sink, cache.window,
                              offset_k=cache.offset_k)
    other = Int2Cache(w, pages_per_split=pps)
    other.int2_pages, other.scale_zero = cache.int2_pages.clone(), cache.scale_zero.clone()
    other.sink, other.window = cache.sink.clone(), cache.window.clone()
    return cache, other, cur, past


def _run_two_calls(w, cache, cur):
    d = torch.device("cuda")
    ic = torch.as_tensor(cur)
    ok.oscar_append_mixed(w.dims, w.k[ic].to(d), w.v[ic].to(d), cache.R_k, cache.R_v, cache.clip_k, cache.clip_v,
                          None, w.slot_mapping[ic].to(d), torch.arange(w.batch, dtype=torch.int32, device=d),
                          w.tok_pos[ic].to(d), cache.seq_lens, w.sink_len, w.window_len, cache.int2_pages,
                          cache.scale_zero, cache.sink, cache.window, offset_k=cache.offset_k)
    return cache.decode(w.q.cuda())


def _run_fused(w, cache, cur):
    d = torch.device("cuda")
    ic = torch.as_tensor(cur)
    out = torch.empty((w.batch, w.num_q_heads, w.head_dim), dtype=torch.float32, device=d)
    ws = cache.workspace(w.max_seq_len)
    ok.oscar_append_decode(w.dims, w.batch, w.max_seq_len, cache.pps, w.q.cuda(), w.k[ic].to(d).contiguous(),
                           w.v[ic].to(d).contiguous(), cache.R_k, cache.R_v, cache.clip_k, cache.clip_v,
                           w.slot_mapping[ic].to(d).contiguous(), cache.int2_pages, cache.scale_zero, cache.sink,
                           cache.window, cache.page_table, cache.seq_lens, w.sink_len, w.window_len, 0.0, out, ws,
                           offset_k=cache.offset_k)
    return out


@pytest.mark.parametrize("name,Hq,H,G,lens,S,W,key_offset,fused", [
    ("batch1_gqa4", 32, 8, 64, [3000], 64, 128, False, 1),       # single-wave form: the append in the BF16 CTAs
    ("batch2_gqa4_g128", 8, 2, 128, [900, 1700], 16, 48, False, 1),
    ("batch1_gqa8", 16, 2, 64, [2500], 32, 64, False, 1),        # the 8-warp single-wave form
    ("batch1_key_offset", 8, 2, 64, [1200], 16, 32, True, 1),
    ("current_in_sink", 8, 2, 64, [5, 700], 16, 32, False, 1),    # a current token inside the sink
    ("no_window", 8, 2, 64, [600, 300], 16, 0, False, 1),         # W = 0: the two calls one after the other
    # general split form: the append in the dense CTA that holds the current row
    ("batch64", 32, 8, 64, [300 + 37 * i for i in range(64)], 16, 64, False, 0),
    # 5 dense CTAs per unit (4 sink + 32 window pages): the current rows spread over all of them
    ("batch48_many_dense_ctas", 32, 8, 64, [700 + 29 * i for i in range(48)], 64, 512, False, 0),
    ("batch40_gqa8_g128", 32, 4, 128, [900 + 53 * i for i in range(40)], 32, 96, True, 0),
    ("batch48_some_in_sink", 16, 4, 64, [3 + 40 * i for i in range(48)], 64, 32, False, 0),
    ("batch64_no_window", 32, 8, 64, [300 + 37 * i for i in range(64)], 16, 0, False, 0),  # sequential
])
def test_append_decode_equals_append_then_decode(name, Hq, H, G, lens, S, W, key_offset, fused):
    w = synth.make_workload(num_q_heads=Hq, num_kv_heads=H, head_dim=128, group_size=G, sink_len=S, window_len=W,
                            seq_lens=lens, seed=len(lens) * 7 + Hq + G + S + W, key_offset=key_offset)
    assert ok.oscar_decode_plan(w.dims, w.batch, w.max_seq_len, 0, S, W)["fused"] == fused
    if name == "batch48_many_dense_ctas":  # the current rows fall in every dense CTA (8 pages each)
        nsp = S // 16
        ctas = {((L - 1) // 16 if L - 1 < S else nsp + ((L - 1) % W) // 16) // 8 for L in lens}
        assert ctas == set(range((nsp + W // 16 + 7) // 8))
    a, b, cur, past = _step_pair(w)
    ok.oscar_device_errors(reset=True)
    out_a = _run_two_calls(w, a, cur)
    out_b = _run_fused(w, b, cur)
    torch.cuda.synchronize()
    assert ok.oscar_device_errors(reset=True) == 0
    # the BF16 rows are the same bf16 conversions of the same inputs
    assert torch.equal(a.sink, b.sink) and torch.equal(a.window, b.window)
    # the appended tokens' codes and scale/zero against the oracle's append
    ic = torch.as_tensor(cur)
    codes, sz = pools_to_host(b)
    check_append(w, codes, sz, w.k[ic], w.v[ic], w.slot_mapping[ic].numpy(), written_slots=w.slot_mapping.numpy())
    # the decode of this step does not read the appended token's codes (it is in the
    # window or the sink): equal outputs whenever the BF16 rows are equal
    if W > 0:
        assert torch.equal(out_a, out_b)
    compare_decode(out_b, oracle_decode_on_gpu_cache(w, b))


def test_append_decode_slot_out_of_range_is_flagged():
    w = synth.make_workload(num_q_heads=8, num_kv_heads=2, head_dim=128, group_size=64, sink_len=8, window_len=16,
                            seq_lens=[400], seed=77)
    assert ok.oscar_decode_plan(w.dims, w.batch, w.max_seq_len, 0, 8, 16)["fused"] == 1
    a, b, cur, past = _step_pair(w)
    d = torch.device("cuda")
    ic = torch.as_tensor(cur)
    slots = torch.full((1,), w.num_pages * w.page_size, dtype=torch.int64, device=d)  # one past the pool
    out = torch.empty((1, 8, 128), dtype=torch.float32, device=d)
    before = b.int2_pages.clone()
    ok.oscar_device_errors(reset=True)
    ok.oscar_append_decode(w.dims, 1, w.max_seq_len, b.pps, w.q.cuda(), w.k[ic].to(d).contiguous(),
                           w.v[ic].to(d).contiguous(), b.R_k, b.R_v, b.clip_k, b.clip_v, slots, b.int2_pages,
                           b.scale_zero, b.sink, b.window, b.page_table, b.seq_lens, 8, 16, 0.0, out,
                           b.workspace(w.max_seq_len))
    torch.cuda.synchronize()
    assert ok.oscar_device_errors(reset=True) & ok.OSCAR_DEVERR_SLOT
    assert torch.equal(b.int2_pages, before)  # no code written
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("lens,W", [([900 + 37 * i for i in range(40)], 64), ([700], 128)])
def test_append_decode_negative_slots_skip_the_token(lens, W):
    # A negative slot skips the token entirely (no codes, no BF16 row), as in
    # oscar_append_mixed: the general form (40 sequences) and the single-wave form.
    w = synth.make_workload(num_q_heads=32, num_kv_heads=8, head_dim=128, group_size=64, sink_len=16, window_len=W,
                            seq_lens=lens, seed=len(lens) + W)
    a, b, cur, past = _step_pair(w)
    d = torch.device("cuda")
    ic = torch.as_tensor(cur)
    slots = w.slot_mapping[ic].clone()
    slots[::3] = -1
    slots = slots.to(d)
    ok.oscar_device_errors(reset=True)
    ok.oscar_append_mixed(w.dims, w.k[ic].to(d), w.v[ic].to(d), a.R_k, a.R_v, a.clip_k, a.clip_v, None, slots,
                          torch.arange(w.batch, dtype=torch.int32, device=d), w.tok_pos[ic].to(d), a.seq_lens,
                          w.sink_len, w.window_len, a.int2_pages, a.scale_zero, a.sink, a.window, offset_k=a.offset_k)
    out_a = a.decode(w.q.cuda())
    out_b = torch.empty_like(out_a)
    ok.oscar_append_decode(w.dims, w.batch, w.max_seq_len, b.pps, w.q.cuda(), w.k[ic].to(d).contiguous(),
                           w.v[ic].to(d).contiguous(), b.R_k, b.R_v, b.clip_k, b.clip_v, slots, b.int2_pages,
                           b.scale_zero, b.sink, b.window, b.page_table, b.seq_lens, w.sink_len, w.window_len, 0.0,
                           out_b, b.workspace(w.max_seq_len), offset_k=b.offset_k)
    torch.cuda.synchronize()
    assert ok.oscar_device_errors(reset=True) == 0
    assert torch.equal(a.sink, b.sink) and torch.equal(a.window, b.window)
    assert torch.equal(a.int2_pages, b.int2_pages) and torch.equal(a.scale_zero, b.scale_zero)
    assert torch.equal(out_a, out_b)


def test_append_decode_general_form_slot_out_of_range_is_flagged():
    lens = [600 + 31 * i for i in range(40)]
    w = synth.make_workload(num_q_heads=32, num_kv_heads=8, head_dim=128, group_size=64, sink_len=16, window_len=64,
                            seq_lens=lens, seed=91)
    assert ok.oscar_decode_plan(w.dims, w.batch, w.max_seq_len, 0, 16, 64)["fused"] == 0
    a, b, cur, past = _step_pair(w)
    d = torch.device("cuda")
    ic = torch.as_tensor(cur)
    slots = w.slot_mapping[ic].clone()
    slots[7] = w.num_pages * w.page_size  # one past the pool
    before = b.int2_pages.clone()
    out = torch.empty((w.batch, 32, 128), dtype=torch.float32, device=d)
    ok.oscar_device_errors(reset=True)
    ok.oscar_append_decode(w.dims, w.batch, w.max_seq_len, b.pps, w.q.cuda(), w.k[ic].to(d).contiguous(),
                           w.v[ic].to(d).contiguous(), b.R_k, b.R_v, b.clip_k, b.clip_v, slots.to(d), b.int2_pages,
                           b.scale_zero, b.sink, b.window, b.page_table, b.seq_lens, 16, 64, 0.0, out,
                           b.workspace(w.max_seq_len))
    torch.cuda.synchronize()
    assert ok.oscar_device_errors(reset=True) & ok.OSCAR_DEVERR_SLOT
    assert torch.isfinite(out).all()
    # only pages holding the other tokens' slots change: the flagged token writes no code
    changed = (b.int2_pages != before).view(w.num_pages, -1).any(dim=1).nonzero().flatten().cpu().numpy()
    written = {int(s) // w.page_size for j, s in enumerate(slots.numpy()) if j != 7}
    assert set(changed.tolist()) <= written


@pytest.mark.parametrize("lens,Hq,H", [([700 + 37 * i for i in range(39)] + [0], 32, 8), ([0, 900], 8, 2)])
def test_append_decode_lengths_out_of_range_follow_append_mixed(lens, Hq, H):
    # Lengths are taken as oscar_append_mixed takes positions: a sequence of length 0
    # gets no sink/window row (flagged) but its codes at the slot (here in the page
    # that sequence owns and no decode reads), and with max_seq_len below the longest
    # sequence that one is appended at its length - 1 while the decode flags the length.
    # The general form (40 sequences) and the single-wave form, each against the two calls.
    w = synth.make_workload(num_q_heads=Hq, num_kv_heads=H, head_dim=128, group_size=64, sink_len=16, window_len=48,
                            seq_lens=lens, seed=len(lens) + 5)
    d = torch.device("cuda")
    B = w.batch
    lens_np = w.seq_lens.numpy()
    pos, seq = w.tok_pos.numpy(), w.tok_seq.numpy()
    zb = int(np.argmin(lens_np))
    cur_idx = {b: int(np.nonzero((seq == b) & (pos == lens_np[b] - 1))[0][0]) for b in range(B) if lens_np[b] > 0}
    past = np.setdiff1d(np.arange(len(pos)), list(cur_idx.values()))
    k_cur = torch.stack([w.k[cur_idx.get(b, 0)] for b in range(B)]).to(d).contiguous()
    v_cur = torch.stack([w.v[cur_idx.get(b, 0)] for b in range(B)]).to(d).contiguous()
    slots = torch.tensor([int(w.slot_mapping[cur_idx[b]]) if b in cur_idx else int(w.page_table[zb, 0]) * w.page_size
                          for b in range(B)], dtype=torch.int64, device=d)
    positions = torch.tensor([int(lens_np[b]) - 1 for b in range(B)], dtype=torch.int32, device=d)
    msl = int(lens_np.max()) - 5
    caches = []
    for _ in range(2):
        c = Int2Cache(w)
        c.sink = torch.zeros((B, 2, H, 16, 128), dtype=torch.bfloat16, device=d)
        c.window = torch.zeros((B, 2, H, 48, 128), dtype=torch.bfloat16, device=d)
        ip = torch.as_tensor(past)
        ok.oscar_append_mixed(w.dims, w.k[ip].to(d), w.v[ip].to(d), c.R_k, c.R_v, c.clip_k, c.clip_v, None,
                              w.slot_mapping[ip].to(d), w.tok_seq[ip].to(d), w.tok_pos[ip].to(d),
                              torch.as_tensor(np.maximum(lens_np - 1, 0), dtype=torch.int32).to(d), 16, 48,
                              c.int2_pages, c.scale_zero, c.sink, c.window)
        caches.append(c)
    a, b = caches
    assert ok.oscar_decode_plan(w.dims, B, msl, 0, 16, 48)["fused"] == (1 if B == 2 else 0)
    torch.cuda.synchronize()
    ok.oscar_device_errors(reset=True)
    ok.oscar_append_mixed(w.dims, k_cur, v_cur, a.R_k, a.R_v, a.clip_k, a.clip_v, None, slots,
                          torch.arange(B, dtype=torch.int32, device=d), positions, a.seq_lens, 16, 48, a.int2_pages,
                          a.scale_zero, a.sink, a.window)
    out_a = a.decode(w.q.cuda(), max_seq_len=msl)
    torch.cuda.synchronize()
    flags_a = ok.oscar_device_errors(reset=True)
    out_b = torch.empty_like(out_a)
    ok.oscar_append_decode(w.dims, B, msl, b.pps, w.q.cuda(), k_cur, v_cur, b.R_k, b.R_v, b.clip_k, b.clip_v, slots,
                           b.int2_pages, b.scale_zero, b.sink, b.window, b.page_table, b.seq_lens, 16, 48, 0.0, out_b,
                           b.workspace(msl))
    torch.cuda.synchronize()
    flags_b = ok.oscar_device_errors(reset=True)
    assert flags_a & ok.OSCAR_DEVERR_POSITION and flags_a & ok.OSCAR_DEVERR_SEQ_LEN
    assert flags_b == flags_a
    assert torch.equal(a.sink, b.sink) and torch.equal(a.window, b.window)
    assert torch.equal(a.int2_pages, b.int2_pages) and torch.equal(a.scale_zero, b.scale_zero)
    assert torch.equal(out_a, out_b)


@pytest.mark.parametrize("lens0,fused", [([3000], 1), ([500 + 41 * i for i in range(40)], 0)])
def test_append_decode_loop_of_steps(lens0, fused):
    # 40 consecutive decode steps per sequence with a 32-row window: tokens pass
    # through the window ring and leave it for the INT2 bulk, which each step reads
    # from codes written by earlier steps.  Every step equals the two calls; at the
    # end every code matches the oracle's append, the sink and window hold the
    # expected bf16 rows, and the last step's output matches the oracle's decode.
    N, S, W = 40, 16, 32
    lens = [L + N for L in lens0]
    w = synth.make_workload(num_q_heads=32, num_kv_heads=8, head_dim=128, group_size=64, sink_len=S, window_len=W,
                            seq_lens=lens, seed=len(lens0) + 123)
    d = torch.device("cuda")
    B = w.batch
    L0 = np.array(lens0)
    pos, seq = w.tok_pos.numpy(), w.tok_seq.numpy()
    past = np.nonzero(pos < L0[seq])[0]
    caches = []
    for _ in range(2):
        c = Int2Cache(w)
        c.sink = torch.zeros((B, 2, 8, S, 128), dtype=torch.bfloat16, device=d)
        c.window = torch.zeros((B, 2, 8, W, 128), dtype=torch.bfloat16, device=d)
        ip = torch.as_tensor(past)
        ok.oscar_append_mixed(w.dims, w.k[ip].to(d), w.v[ip].to(d), c.R_k, c.R_v, c.clip_k, c.clip_v, None,
                              w.slot_mapping[ip].to(d), w.tok_seq[ip].to(d), w.tok_pos[ip].to(d),
                              torch.as_tensor(L0, dtype=torch.int32).to(d), S, W, c.int2_pages, c.scale_zero,
                              c.sink, c.window)
        caches.append(c)
    a, b = caches
    msl = w.max_seq_len
    assert ok.oscar_decode_plan(w.dims, B, msl, 0, S, W)["fused"] == fused
    q = w.q.cuda()
    ok.oscar_device_errors(reset=True)
    for n in range(N):
        cur = torch.as_tensor([int(np.nonzero((seq == bb) & (pos == L0[bb] + n))[0][0]) for bb in range(B)])
        sl = torch.as_tensor(L0 + n + 1, dtype=torch.int32).to(d)
        k_cur, v_cur, s_cur = w.k[cur].to(d).contiguous(), w.v[cur].to(d).contiguous(), w.slot_mapping[cur].to(d)
        ok.oscar_append_mixed(w.dims, k_cur, v_cur, a.R_k, a.R_v, a.clip_k, a.clip_v, None, s_cur,
                              torch.arange(B, dtype=torch.int32, device=d), w.tok_pos[cur].to(d), sl, S, W,
                              a.int2_pages, a.scale_zero, a.sink, a.window)
        out_a = a.decode(q, seq_lens=sl)
        out_b = torch.empty_like(out_a)
        ok.oscar_append_decode(w.dims, B, msl, b.pps, q, k_cur, v_cur, b.R_k, b.R_v, b.clip_k, b.clip_v, s_cur,
                               b.int2_pages, b.scale_zero, b.sink, b.window, b.page_table, sl, S, W, 0.0, out_b,
                               b.workspace(msl))
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_b), f"step {n}"
    assert ok.oscar_device_errors(reset=True) == 0
    assert torch.equal(a.sink, b.sink) and torch.equal(a.window, b.window)
    # the codes of every token appended by the steps and of 3000 earlier tokens
    # against the oracle's append (every slot was written)
    codes, sz = pools_to_host(b)
    loop_tok = np.nonzero(pos >= L0[seq])[0]
    sample = np.concatenate([loop_tok, np.random.default_rng(5).choice(past, min(3000, len(past)), replace=False)])
    check_append(w, codes, sz, w.k, w.v, w.slot_mapping.numpy(), sample=sample,
                 written_slots=w.slot_mapping.numpy())
    # sink rows: positions 0 .. S-1; window slot r: the latest position p = r (mod W)
    kb, vb = w.k.view(torch.int16).numpy(), w.v.view(torch.int16).numpy()
    sink_h, win_h = b.sink.view(torch.int16).cpu().numpy(), b.window.view(torch.int16).cpu().numpy()
    for bb in range(B):
        L = lens[bb]
        idx = {int(p): i for i, p in zip(np.nonzero(seq == bb)[0], pos[seq == bb])}
        for p in range(S):
            assert np.array_equal(sink_h[bb, 0, :, p], kb[idx[p]]) and np.array_equal(sink_h[bb, 1, :, p], vb[idx[p]])
        for r in range(W):
            p = L - 1 - ((L - 1 - r) % W)
            assert np.array_equal(win_h[bb, 0, :, r], kb[idx[p]]) and np.array_equal(win_h[bb, 1, :, r], vb[idx[p]])
    # the last step's output against the oracle's decode of the final cache
    pairs = None if B == 1 else [(bb, (7 * bb + 3) % 32) for bb in range(0, B, 2)]
    compare_decode(out_b, oracle_decode_on_gpu_cache(w, b, pairs=pairs), pairs=pairs)
