"""The bounded device waits run out without faulting, hanging or losing the
context.  The library's test hook makes every INT2 split warp wait for its first
page on an mbarrier phase that nothing completes (its copies all land as usual);
the wait gives up after about half a millisecond.  The decode must report
OSCAR_DEVERR_TIMEOUT, drop the splits' work (with no BF16 sink/window the output
is then exactly zero) and leave the next call bit-identical to one made before."""

import pytest
import torch

import int2_rotated_kv_append_gb300 as ok
from int2_rotated_kv_append_gb300 import synth
from int2_rotated_kv_append_gb300.cache import Int2Cache

pytestmark = pytest.mark.gpu

STALL_CYCLES = 1_000_000


@pytest.mark.parametrize("lens", [[3000],                 # batch 1: single-wave fused form
                                  [900] * 48 + [2000] * 16])  # 512 units: general split form
def test_page_wait_timeout_is_reported_and_recovers(lens):
    w = synth.make_workload(num_q_heads=32, num_kv_heads=8, head_dim=128, group_size=64, sink_len=0, window_len=0,
                            seq_lens=lens, seed=len(lens) + 7)
    plan = ok.oscar_decode_plan(w.dims, w.batch, w.max_seq_len, 0, 0, 0)
    assert plan["fused"] == (1 if len(lens) == 1 else 0)
    cache = Int2Cache(w)
    cache.prefill()
    q = w.q.cuda()
    before = cache.decode(q).clone()
    assert torch.count_nonzero(before) > 0
    assert ok.oscar_device_errors(reset=True) == 0
    ok.oscar_test_stall_page_waits(STALL_CYCLES)
    try:
        stalled = cache.decode(q).clone()
        torch.cuda.synchronize()
    finally:
        ok.oscar_test_stall_page_waits(0)
    assert ok.oscar_device_errors(reset=True) & ok.OSCAR_DEVERR_TIMEOUT
    assert torch.count_nonzero(stalled) == 0 and torch.isfinite(stalled).all()
    after = cache.decode(q).clone()
    assert ok.oscar_device_errors(reset=True) == 0
    assert torch.equal(after, before)


def test_stall_hook_rejects_negative():
    with pytest.raises(ok.OscarError):
        ok.oscar_test_stall_page_waits(-1)
