"""GPU parity of oscar_append against the oracle (bit-exact codes and layout)."""

import numpy as np
import pytest
import torch

from int2_rotated_kv_append_gb300 import synth
from int2_rotated_kv_append_gb300.cache import Int2Cache
from parity import check_append, pools_to_host

pytestmark = pytest.mark.gpu


def _append_all(w, cache):
    cache.append(w.k.cuda(), w.v.cuda(), w.slot_mapping.cuda())
    torch.cuda.synchronize()
    return pools_to_host(cache)


def test_append_tiny_config():
    w = synth.make_config(0)
    cache = Int2Cache(w)
    codes, sz = _append_all(w, cache)
    stats = check_append(w, codes, sz, w.k, w.v, w.slot_mapping.numpy())
    assert stats["elements"] == 512 * 2 * 64


@pytest.mark.parametrize("D,G", [(64, 32), (64, 64), (128, 32), (128, 64), (128, 128)])
@pytest.mark.parametrize("H", [1, 3])
def test_append_sweep_random_slots(D, G, H):
    # 70 tokens (3 tiles, ragged) into random distinct slots of a 12-page pool; some slots skipped.
    w = synth.make_workload(num_q_heads=H, num_kv_heads=H, head_dim=D, group_size=G, sink_len=0, window_len=0,
                            seq_lens=[70], seed=D + G + H, spare_pages=7)
    g = torch.Generator().manual_seed(D * 7 + G + H)
    slots = torch.randperm(w.num_pages * 16, generator=g)[:70].to(torch.int64)
    slots[5] = -1
    slots[40] = -7
    cache = Int2Cache(w)
    cache.append(w.k.cuda(), w.v.cuda(), slots.cuda())
    torch.cuda.synchronize()
    codes, sz = pools_to_host(cache)
    check_append(w, codes, sz, w.k, w.v, slots.numpy())


def test_append_unclipped_identity_rotation():
    # R = I and infinite clip: the codes quantise the raw bf16 values.
    w = synth.make_workload(num_q_heads=2, num_kv_heads=2, head_dim=128, group_size=64, sink_len=0, window_len=0,
                            seq_lens=[45], seed=3, clip_frac=None)
    w.R_k = torch.eye(128).expand(2, 128, 128).contiguous()
    w.R_v = w.R_k.clone()
    cache = Int2Cache(w)
    codes, sz = _append_all(w, cache)
    check_append(w, codes, sz, w.k, w.v, w.slot_mapping.numpy(), exact=True)


def test_append_zero_clip_degenerate():
    w = synth.make_workload(num_q_heads=1, num_kv_heads=1, head_dim=64, group_size=32, sink_len=0, window_len=0,
                            seq_lens=[20], seed=4)
    w.clip_k = torch.zeros_like(w.clip_k)
    w.clip_v = torch.zeros_like(w.clip_v)
    cache = Int2Cache(w)
    codes, sz = _append_all(w, cache)
    check_append(w, codes, sz, w.k, w.v, w.slot_mapping.numpy())
    rows = codes.reshape(w.num_pages, 1, 2, 16, 16)
    pt = w.page_table.numpy()[0]
    assert np.all(rows[pt[0], :, :, :16] == 0) and np.all(rows[pt[1], :, :, :4] == 0)


def test_append_prefill_config_sampled():
    # Prefill append of 16384 tokens x 8 heads x D=128 at full size; the oracle checks a sample.
    w = synth.make_config(4, device="cuda")
    cache = Int2Cache(w)
    codes, sz = _append_all(w, cache)
    g = np.random.default_rng(0)
    sample = np.sort(g.choice(w.num_tokens, 1024, replace=False))
    sample = np.concatenate([sample, [0, w.num_tokens - 1]])
    check_append(w, codes, sz, w.k, w.v, w.slot_mapping.numpy(), sample=sample)


@pytest.mark.parametrize("G", [32, 64, 128])
@pytest.mark.parametrize("H", [1, 3])
def test_append_tensor_core_rotation_sweep(G, H):
    # > 512 tokens at D = 128: the tensor-core rotation (64-token tiles; 1000 = 15 tiles + a
    # ragged 40) into random distinct slots, some skipped.
    T = 1000
    w = synth.make_workload(num_q_heads=H, num_kv_heads=H, head_dim=128, group_size=G, sink_len=0, window_len=0,
                            seq_lens=[T], seed=G + 11 * H, spare_pages=9)
    g = torch.Generator().manual_seed(G * 5 + H)
    slots = torch.randperm(w.num_pages * 16, generator=g)[:T].to(torch.int64)
    slots[0] = -1
    slots[999] = -1
    slots[517] = -3
    cache = Int2Cache(w)
    cache.append(w.k.cuda(), w.v.cuda(), slots.cuda())
    torch.cuda.synchronize()
    codes, sz = pools_to_host(cache)
    check_append(w, codes, sz, w.k, w.v, slots.numpy())


def test_append_tensor_core_many_tiles_per_cta():
    # 8 KV heads, 4685 tokens = 36 full 128-token tiles + a ragged 77: the CTAs of a
    # (head, K|V) take 4-5 tiles each, so the x ring wraps and both accumulators are used.
    w = synth.make_workload(num_q_heads=8, num_kv_heads=8, head_dim=128, group_size=64, sink_len=0, window_len=0,
                            seq_lens=[4685], seed=21, device="cuda")
    cache = Int2Cache(w)
    codes, sz = _append_all(w, cache)
    check_append(w, codes, sz, w.k, w.v, w.slot_mapping.numpy())


def test_append_tensor_core_groups_outside_the_code_range():
    # R = I, no clip, x ~ 1e-6: scale and zero fall in the fp16 subnormal range, where the
    # rounding of the zero is comparable to the scale, so (y - zero) / scale leaves
    # [-0.5, 3.5) in some groups and the kernel's clamped quotient path runs there.
    w = synth.make_workload(num_q_heads=2, num_kv_heads=2, head_dim=128, group_size=64, sink_len=0, window_len=0,
                            seq_lens=[600], seed=8, clip_frac=None)
    w.R_k = torch.eye(128).expand(2, 128, 128).contiguous()
    w.R_v = w.R_k.clone()
    g = torch.Generator().manual_seed(9)
    w.k = (1e-6 * (1 + 0.2 * torch.rand(w.k.shape, generator=g))).to(torch.bfloat16)
    w.v = (-3e-6 * (1 + 0.1 * torch.rand(w.v.shape, generator=g))).to(torch.bfloat16)
    # the case is present: groups whose extreme values map outside [-0.5, 3.5)
    y = torch.cat([w.k, w.v]).float().numpy().reshape(-1, 64)
    mn, mx = y.min(1), y.max(1)
    sc = ((mx - mn) / np.float32(3)).astype(np.float16).astype(np.float32)
    z = mn.astype(np.float16).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.where(sc != 0, np.float32(1) / sc, np.float32(0)).astype(np.float32)
    out = ((mn - z) * inv < -0.5) | ((mx - z) * inv >= 3.5)
    assert out.sum() > 0
    cache = Int2Cache(w)
    codes, sz = _append_all(w, cache)
    check_append(w, codes, sz, w.k, w.v, w.slot_mapping.numpy(), exact=True)


def test_append_tensor_core_identity_rotation_exact():
    # R = I splits into (1, 0, 0) exactly, so the tensor-core path quantises the raw bf16 values.
    w = synth.make_workload(num_q_heads=2, num_kv_heads=2, head_dim=128, group_size=64, sink_len=0, window_len=0,
                            seq_lens=[600], seed=5, clip_frac=None)
    w.R_k = torch.eye(128).expand(2, 128, 128).contiguous()
    w.R_v = w.R_k.clone()
    cache = Int2Cache(w)
    codes, sz = _append_all(w, cache)
    check_append(w, codes, sz, w.k, w.v, w.slot_mapping.numpy(), exact=True)


def test_append_decode_batch_random_slots():
    # Decode append: 256 single tokens at random slots of a pool, every token checked.
    w = synth.make_workload(num_q_heads=32, num_kv_heads=8, head_dim=128, group_size=64, sink_len=64,
                            window_len=128, seq_lens=[4096], seed=4, device="cuda")
    k, v, slots = synth.decode_append_batch(w, 256)
    cache = Int2Cache(w)
    cache.append(k, v, slots.cuda())
    torch.cuda.synchronize()
    codes, sz = pools_to_host(cache)
    check_append(w, codes, sz, k, v, slots.numpy())


def test_append_slot_past_pool_is_flagged():
    import int2_rotated_kv_append_gb300 as ok
    ok.oscar_device_errors(reset=True)
    w = synth.make_workload(num_q_heads=1, num_kv_heads=1, head_dim=64, group_size=32, sink_len=0, window_len=0,
                            seq_lens=[8], seed=6)
    slots = w.slot_mapping.clone()
    slots[3] = w.num_pages * 16 + 5
    cache = Int2Cache(w)
    cache.append(w.k.cuda(), w.v.cuda(), slots.cuda())
    flags = ok.oscar_device_errors(reset=True)
    assert flags & ok.OSCAR_DEVERR_SLOT
    codes, sz = pools_to_host(cache)
    keep = np.array([i for i in range(8) if i != 3])
    check_append(w, codes, sz, w.k, w.v, slots.numpy(), sample=keep)


# --- oscar_append_mixed: INT2 append plus the BF16 sink/window rows ------------

def _mixed_run(w, S, W, ids=None, fill=0xFFFF):
    """GPU append_mixed of every token of w (one call) into sentinel-filled buffers;
    returns the INT2 pools, sink and window (host), and the plain append's pools."""
    import int2_rotated_kv_append_gb300 as ok
    B, H, D = w.batch, w.num_kv_heads, w.head_dim
    fill16 = fill - 0x10000 if fill >= 0x8000 else fill
    sink = torch.full((B, 2, H, max(S, 1), D), fill16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    win = torch.full((B, 2, H, max(W, 1), D), fill16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    cache = Int2Cache(w)
    ids = w.tok_seq if ids is None else ids
    ok.oscar_append_mixed(w.dims, w.k.cuda(), w.v.cuda(), cache.R_k, cache.R_v, cache.clip_k, cache.clip_v, None,
                          w.slot_mapping.cuda(), ids.cuda(), w.tok_pos.cuda(), w.seq_lens.cuda(), S, W,
                          cache.int2_pages, cache.scale_zero, sink, win)
    torch.cuda.synchronize()
    plain = Int2Cache(w)
    plain.append(w.k.cuda(), w.v.cuda(), w.slot_mapping.cuda())
    torch.cuda.synchronize()
    return pools_to_host(cache), pools_to_host(plain), synth.bits16(sink), synth.bits16(win)


def _oracle_mixed(w, S, W, fill=0xFFFF):
    from oracle import oracle as O
    B, H, D, G = w.batch, w.num_kv_heads, w.head_dim, w.group_size
    pool = np.zeros(w.num_pages * H * 2 * 16 * D // 4, np.uint8)
    sz = np.zeros(w.num_pages * H * 2 * 16 * (D // G) * 2, np.uint16)
    sink = np.full((B, 2, H, max(S, 1), D), fill, np.uint16)
    win = np.full((B, 2, H, max(W, 1), D), fill, np.uint16)
    O.append_mixed(w.dims, synth.bits16(w.k), synth.bits16(w.v), w.R_k.cpu().numpy(), w.R_v.cpu().numpy(),
                   w.clip_k.cpu().numpy(), w.clip_v.cpu().numpy(), w.slot_mapping.numpy(), w.tok_seq.numpy(),
                   w.tok_pos.numpy(), w.seq_lens.numpy(), S, W, pool, sz, sink, win)
    return sink, win


@pytest.mark.parametrize("lens,S,W", [([5, 40, 70, 300], 8, 24), ([700, 300], 64, 128), ([3, 17], 0, 16),
                                      ([33], 16, 0)])
def test_append_mixed_matches_oracle(lens, S, W):
    # few tokens (the small kernel) and > 512 tokens (the tiled kernel); sink or window absent
    w = synth.make_workload(num_q_heads=4, num_kv_heads=2, head_dim=128, group_size=64, sink_len=S, window_len=W,
                            seq_lens=lens, seed=sum(lens) + S + W)
    (codes, sz), (codes_p, sz_p), sink, win = _mixed_run(w, S, W)
    assert np.array_equal(codes, codes_p) and np.array_equal(sz, sz_p)  # INT2 part = plain append
    o_sink, o_win = _oracle_mixed(w, S, W)
    if S > 0:
        assert np.array_equal(sink, o_sink)
    if W > 0:
        assert np.array_equal(win, o_win)


def test_append_mixed_bad_sequence_id_is_flagged():
    import int2_rotated_kv_append_gb300 as ok
    w = synth.make_workload(num_q_heads=2, num_kv_heads=1, head_dim=64, group_size=32, sink_len=4, window_len=8,
                            seq_lens=[12], seed=5)
    ids = w.tok_seq.clone()
    ids[2] = 7  # no such sequence: its BF16 rows are skipped (position 2 of the sink stays untouched)
    ok.oscar_device_errors(reset=True)
    _, _, sink, win = _mixed_run(w, 4, 8, ids=ids)
    assert ok.oscar_device_errors(reset=True) & ok.OSCAR_DEVERR_POSITION
    assert np.all(sink[0, :, :, 2] == 0xFFFF)
    assert not np.all(sink[0, :, :, 1] == 0xFFFF)
