"""GPU parity of the BF16 paged decode (the speedup reference) against the oracle."""

import numpy as np
import pytest
import torch

from int2_rotated_kv_append_gb300 import synth
from int2_rotated_kv_append_gb300.cache import Bf16Cache
from int2_rotated_kv_append_gb300.synth import bits16
from oracle import oracle as O
from parity import compare_decode

pytestmark = pytest.mark.gpu


def _oracle(w, cache, pairs=None):
    pages = bits16(cache.pages)
    return O.bf16_decode(w.dims, w.batch, bits16(w.q), pages, w.page_table.numpy(), w.seq_lens.numpy(), 0.0,
                         pairs=pairs)


@pytest.mark.parametrize("D,Hq,H,lens", [(64, 1, 1, [512]), (128, 8, 2, [0, 1, 15, 16, 17, 900]),
                                         (128, 16, 2, [2000, 33])])
def test_bf16_decode_small(D, Hq, H, lens):
    w = synth.make_workload(num_q_heads=Hq, num_kv_heads=H, head_dim=D, group_size=64 if D == 128 else 32,
                            sink_len=0, window_len=0, seq_lens=lens, seed=D + Hq)
    cache = Bf16Cache(w)
    cache.prefill()
    out = cache.decode(w.q.cuda())
    compare_decode(out, _oracle(w, cache))


def test_bf16_decode_batch1_32k_config():
    w = synth.make_config(1, device="cuda")
    cache = Bf16Cache(w)
    cache.prefill()
    out = cache.decode(w.q)
    pairs = [(0, h) for h in range(32)]
    compare_decode(out, _oracle(w, cache, pairs), pairs=pairs)


@pytest.mark.parametrize("Hq,H,lens", [(64, 8, [6000, 2500]), (16, 4, [7000, 4001, 15, 0])])
def test_bf16_decode_small_batch_ragged(Hq, H, lens):
    # GQA 8 and 4, a sequence shorter than one split, an empty one.
    w = synth.make_workload(num_q_heads=Hq, num_kv_heads=H, head_dim=128, group_size=64, sink_len=0, window_len=0,
                            seq_lens=lens, seed=Hq + len(lens))
    cache = Bf16Cache(w)
    cache.prefill()
    out = cache.decode(w.q.cuda())
    compare_decode(out, _oracle(w, cache))
