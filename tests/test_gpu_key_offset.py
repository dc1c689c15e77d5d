"""GPU parity of the key offset removal (the OptR abstract on the OSCAR paper
page: an attention-equivalent key reparameterisation that removes per-channel
key offsets without changing softmax).  Appends given a per-(KV head, channel)
offset c rotate fp32(k - c), leave V alone and store bf16(k - c) as the BF16 key
rows.  Each append kernel (few tokens, tiled FFMA at head_dim 64, tcgen05 at
head_dim 128) is checked against the oracle under the append contract; the BF16
rows bit for bit; the decode of an offset cache against the oracle's decode of
the same buffers."""

import math

import numpy as np
import pytest
import torch

import int2_rotated_kv_append_gb300 as ok
from int2_rotated_kv_append_gb300 import synth
from int2_rotated_kv_append_gb300.cache import Int2Cache
from oracle import oracle as O
from parity import check_append, compare_decode, oracle_decode_on_gpu_cache, pools_to_host

pytestmark = pytest.mark.gpu


def _workload(D, G, lens, S=0, W=0, H=2, Hq=8, seed=0):
    return synth.make_workload(num_q_heads=Hq, num_kv_heads=H, head_dim=D, group_size=G, sink_len=S, window_len=W,
                               seq_lens=lens, seed=seed, key_offset=True)


@pytest.mark.parametrize("D,G,lens", [(128, 64, [300]),          # few-token kernel
                                      (128, 64, [1500, 700]),     # tcgen05 kernel, ragged last tile
                                      (128, 32, [900]),
                                      (128, 128, [777]),
                                      (64, 32, [1200]),           # tiled FFMA kernel
                                      (64, 64, [40])])
def test_append_with_key_offset(D, G, lens):
    w = _workload(D, G, lens, seed=D + G + sum(lens))
    assert w.offset_k is not None and float(w.offset_k.abs().max()) > 1.0  # keys with real channel offsets
    cache = Int2Cache(w)
    cache.append(w.k.cuda(), w.v.cuda(), w.slot_mapping.cuda())
    torch.cuda.synchronize()
    codes, sz = pools_to_host(cache)
    n = w.num_tokens
    sample = None if n <= 600 else np.random.default_rng(n).choice(n, 600, replace=False)
    check_append(w, codes, sz, w.k, w.v, w.slot_mapping.numpy(), sample=sample)


def test_zero_offset_is_no_offset():
    w = _workload(128, 64, [1100, 90], seed=5)
    a, b = Int2Cache(w), Int2Cache(w)
    a.append(w.k.cuda(), w.v.cuda(), w.slot_mapping.cuda())
    b.offset_k = torch.zeros_like(b.offset_k)
    b.append(w.k.cuda(), w.v.cuda(), w.slot_mapping.cuda())
    c = Int2Cache(w)
    c.offset_k = None
    c.append(w.k.cuda(), w.v.cuda(), w.slot_mapping.cuda())
    torch.cuda.synchronize()
    assert torch.equal(b.int2_pages, c.int2_pages) and torch.equal(b.scale_zero.view(torch.int16),
                                                                   c.scale_zero.view(torch.int16))
    assert not torch.equal(a.int2_pages, c.int2_pages)
    # values are never offset: the V rows of every page are the same with and without
    H, D, P = w.num_kv_heads, w.head_dim, w.page_size
    va = a.int2_pages.view(w.num_pages, H, 2, P, D // 4)[:, :, 1]
    vc = c.int2_pages.view(w.num_pages, H, 2, P, D // 4)[:, :, 1]
    assert torch.equal(va, vc)


def _oracle_mixed(w, S, W):
    B, H, D, G = w.batch, w.num_kv_heads, w.head_dim, w.group_size
    pool = np.zeros(w.num_pages * H * 2 * 16 * D // 4, np.uint8)
    sz = np.zeros(w.num_pages * H * 2 * 16 * (D // G) * 2, np.uint16)
    sink = np.zeros((B, 2, H, max(S, 1), D), np.uint16)
    win = np.zeros((B, 2, H, max(W, 1), D), np.uint16)
    O.append_mixed(w.dims, synth.bits16(w.k), synth.bits16(w.v), w.R_k.cpu().numpy(), w.R_v.cpu().numpy(),
                   w.clip_k.cpu().numpy(), w.clip_v.cpu().numpy(), w.slot_mapping.numpy(), w.tok_seq.numpy(),
                   w.tok_pos.numpy(), w.seq_lens.numpy(), S, W, pool, sz, sink, win,
                   offset_k=w.offset_k.cpu().numpy())
    return sink, win


@pytest.mark.parametrize("D,G,lens,S,W", [(128, 64, [5, 40, 70, 300], 8, 24),   # few-token kernel
                                          (128, 64, [700, 300], 64, 128),        # tcgen05 kernel
                                          (64, 32, [900, 20], 16, 32)])          # tiled FFMA kernel
def test_append_mixed_offset_rows_bit_exact(D, G, lens, S, W):
    w = _workload(D, G, lens, S=S, W=W, seed=sum(lens) + S)
    cache = Int2Cache(w)
    cache.prefill()               # oscar_append_mixed with the offset
    torch.cuda.synchronize()
    o_sink, o_win = _oracle_mixed(w, S, W)
    assert np.array_equal(synth.bits16(cache.sink), o_sink)
    assert np.array_equal(synth.bits16(cache.window), o_win)
    codes, sz = pools_to_host(cache)
    n = w.num_tokens
    sample = None if n <= 600 else np.random.default_rng(n).choice(n, 600, replace=False)
    check_append(w, codes, sz, w.k, w.v, w.slot_mapping.numpy(), sample=sample)


@pytest.mark.parametrize("lens", [[5000], [3000, 1400, 17]])
def test_decode_of_offset_cache(lens):
    # fused (batch 1) and general split paths read an offset cache exactly like any other
    w = _workload(128, 64, lens, S=16, W=64, H=8, Hq=32, seed=len(lens) + 70)
    cache = Int2Cache(w)
    cache.prefill()
    out = cache.decode(w.q.cuda())
    pairs = [(b, h) for b in range(w.batch) for h in range(0, w.num_q_heads, 3)]
    compare_decode(out, oracle_decode_on_gpu_cache(w, cache, pairs=pairs), pairs=pairs)


def _exact_attention(w, pairs):
    """fp64 softmax attention over the ORIGINAL bf16 keys and values."""
    k = w.k.float().cpu().numpy().astype(np.float64)
    v = w.v.float().cpu().numpy().astype(np.float64)
    q = w.q.float().cpu().numpy().astype(np.float64)
    start = np.concatenate([[0], np.cumsum(w.seq_lens.numpy())[:-1]])
    gqa = w.num_q_heads // w.num_kv_heads
    out = []
    for b, hq in pairs:
        rows = slice(start[b], start[b] + int(w.seq_lens[b]))
        logits = k[rows, hq // gqa] @ q[b, hq] / math.sqrt(w.head_dim)
        p = np.exp(logits - logits.max())
        out.append((p[:, None] * v[rows, hq // gqa]).sum(0) / p.sum())
    return np.stack(out)


def test_offset_lowers_attention_error():
    # keys with large per-channel means: removing them shrinks the INT2 groups' range,
    # so the decode lands closer to exact attention over the original keys
    # (the same seed draws the same keys, values, queries and rotations; the plain
    # workload's clipping thresholds are those of the keys themselves)
    w_off = _workload(128, 64, [4000], S=0, W=0, H=8, Hq=32, seed=91)
    w_plain = synth.make_workload(num_q_heads=32, num_kv_heads=8, head_dim=128, group_size=64, sink_len=0,
                                  window_len=0, seq_lens=[4000], seed=91)
    assert torch.equal(w_off.k, w_plain.k) and torch.equal(w_off.q, w_plain.q)
    pairs = [(0, h) for h in range(32)]
    exact = _exact_attention(w_off, pairs)
    err = {}
    for name, w in (("offset", w_off), ("plain", w_plain)):
        cache = Int2Cache(w)
        cache.append(w.k.cuda(), w.v.cuda(), w.slot_mapping.cuda())
        cache.sink = torch.zeros((1, 2, 8, 1, 128), dtype=torch.bfloat16, device="cuda")
        cache.window = torch.zeros_like(cache.sink)
        out = cache.decode(w.q.cuda()).cpu().numpy().astype(np.float64)
        err[name] = float(np.sqrt(np.mean((out[0] - exact) ** 2)))
    assert err["offset"] < err["plain"], err
