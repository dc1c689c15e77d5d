"""Checks of the seeded input generator (CPU)."""

import numpy as np
import torch

from int2_rotated_kv_append_gb300 import synth


def test_haar_rotation_orthogonal_fp64():
    g = torch.Generator().manual_seed(0)
    Q = synth.haar_orthogonal(4, 128, g)
    eye = torch.eye(128, dtype=torch.float64)
    for i in range(4):
        assert torch.max(torch.abs(Q[i].T @ Q[i] - eye)).item() < 1e-12


def test_fp32_rotation_near_orthogonal():
    w = synth.make_config(0)
    R = w.R_k[0].double()
    assert torch.max(torch.abs(R.T @ R - torch.eye(64, dtype=torch.float64))).item() < 1e-6


def test_tiny_config_shapes_and_slots():
    w = synth.make_config(0)
    assert (w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.group_size) == (1, 1, 1, 64, 32)
    assert (w.sink_len, w.window_len, w.page_size) == (4, 32, 16)
    assert w.k.shape == (512, 1, 64) and w.k.dtype == torch.bfloat16
    # every token has a distinct slot inside the pool, matching the page table
    slots = w.slot_mapping.numpy()
    assert len(set(slots.tolist())) == 512 and slots.max() < w.num_pages * 16
    pt = w.page_table.numpy()
    for t in range(512):
        p = int(w.tok_pos[t])
        assert slots[t] == pt[0, p // 16] * 16 + p % 16
    # clip = 0.9 x max |x R| per channel
    xr = w.k[:, 0].double() @ w.R_k[0].double()
    assert torch.allclose(w.clip_k[0].double(), 0.9 * xr.abs().amax(0), rtol=1e-6)


def test_sink_window_buffers():
    w = synth.make_workload(num_q_heads=2, num_kv_heads=1, head_dim=64, group_size=32, sink_len=3, window_len=5,
                            seq_lens=[20, 2, 7], seed=5)
    sink, win = w.sink_window()
    starts = np.cumsum([0] + w.seq_lens.tolist())
    for b, L in enumerate(w.seq_lens.tolist()):
        for p in range(L):
            t = starts[b] + p
            if p < 3:
                assert torch.equal(sink[b, 0, :, p], w.k[t]) and torch.equal(sink[b, 1, :, p], w.v[t])
            elif p >= max(3, L - 5):
                assert torch.equal(win[b, 0, :, p % 5], w.k[t]) and torch.equal(win[b, 1, :, p % 5], w.v[t])


def test_config2_lengths_and_seeding():
    lens = synth.config_seq_lens(2)
    assert len(lens) == 64 and min(lens) >= 1024 and max(lens) <= 16384
    assert synth.config_seq_lens(2) == lens
    a = synth.make_workload(num_q_heads=4, num_kv_heads=2, head_dim=64, group_size=32, sink_len=4,
                            window_len=8, seq_lens=[40, 50], seed=9)
    b = synth.make_workload(num_q_heads=4, num_kv_heads=2, head_dim=64, group_size=32, sink_len=4,
                            window_len=8, seq_lens=[40, 50], seed=9)
    assert torch.equal(a.k, b.k) and torch.equal(a.page_table, b.page_table) and torch.equal(a.R_v, b.R_v)
