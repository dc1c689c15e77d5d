"""Comparison of GPU results with the CPU oracle (tolerances and exemption rules).

Append (bit-exact contract): every code equals the oracle's code computed from
the oracle's fp64 pre-rounding value and the GPU's stored fp16 scale/zero,
except elements whose value u = (x - zero)/scale lies within 1e-5 (in code
units) of a rounding boundary k + 1/2; those are counted and must stay at most
1e-4 of all elements.  Scales match the oracle's to 1e-3 relative; zeros to
1e-3 of max(|zero|, scale).  Bytes of rows that were not written keep the
fill pattern.
Decode: the oracle recomputes the output from the GPU's own codes and
scale/zero; max-abs <= 2e-3 and mean-abs <= 2e-4 in fp32.
"""

from __future__ import annotations

import json
import os

import numpy as np
import torch

from int2_rotated_kv_append_gb300.synth import Workload, bits16
from oracle import oracle as O

BAND = 1e-5
MAX_EXEMPT_FRAC = 1e-4
SZ_RTOL = 1e-3
DEC_MAX_ABS = 2e-3
DEC_MEAN_ABS = 2e-4


def unpack_codes(byte_rows: np.ndarray, D: int) -> np.ndarray:
    """[..., D/4] bytes -> [..., D] codes (channel j in byte j//4, bits 2*(j%4))."""
    b = byte_rows.astype(np.uint8)
    parts = [(b >> (2 * i)) & 3 for i in range(4)]
    return np.stack(parts, axis=-1).reshape(*b.shape[:-1], D).astype(np.int32)


def pools_to_host(cache):
    codes = cache.int2_pages.cpu().numpy()
    sz = cache.scale_zero.view(torch.int16).cpu().numpy().view(np.uint16)
    return codes, sz


def _log(kind: str, stats: dict):
    path = os.environ.get("OSCAR_PARITY_LOG")
    if path:
        test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
        with open(path, "a") as f:
            f.write(json.dumps({"test": test, "kind": kind, **stats}) + "\n")


def check_append(w: Workload, codes_gpu: np.ndarray, sz_gpu: np.ndarray, k: torch.Tensor, v: torch.Tensor,
                 slots: np.ndarray, sample: np.ndarray | None = None, fill: int = 0xA5,
                 written_slots: np.ndarray | None = None, exact: bool = False) -> dict:
    """Check the GPU pools after appending k/v at ``slots``; ``sample`` restricts the
    oracle to some tokens.  ``written_slots``: every slot any append wrote (for the
    untouched-row check; defaults to ``slots``).  ``exact``: every code must match
    with no exemption (inputs whose exact ties both sides round to even, e.g.
    unrotated bf16 data, where the near-boundary share is large by construction)."""
    H, D, P, G = w.num_kv_heads, w.head_dim, w.page_size, w.group_size
    NP = w.num_pages
    rows = codes_gpu.reshape(NP, H, 2, P, D // 4)
    szr = sz_gpu.reshape(NP, H, 2, P, D // G, 2)
    idx = np.arange(len(slots)) if sample is None else np.asarray(sample)
    idx = idx[slots[idx] >= 0]
    idx = idx[slots[idx] < NP * P]
    ks, vs = bits16(k[torch.as_tensor(idx, device=k.device)]), bits16(v[torch.as_tensor(idx, device=v.device)])
    Rk, Rv = w.R_k.cpu().numpy(), w.R_v.cpu().numpy()
    ck, cv = w.clip_k.cpu().numpy(), w.clip_v.cpu().numpy()
    offset_k = None if w.offset_k is None else w.offset_k.cpu().numpy()
    pre = O.append_prequant(w.dims, ks, vs, Rk, Rv, ck, cv, offset_k=offset_k)   # [n][H][2][D]
    page, off = slots[idx] // P, slots[idx] % P
    g_codes = unpack_codes(rows[page, :, :, off], D)                  # [n][H][2][D]
    g_sz = szr[page, :, :, off]                                       # [n][H][2][D/G][2]
    exp_codes, u = O.codes_given_params(pre.reshape(-1, D), g_sz.reshape(-1, D // G * 2), G)
    exp_codes = exp_codes.reshape(g_codes.shape)
    u = u.reshape(g_codes.shape)
    dist = np.min(np.abs(u[..., None] - (np.arange(3) + 0.5)), axis=-1)
    near = np.nan_to_num(dist, nan=1.0) < BAND
    mismatch = g_codes != exp_codes
    bad = mismatch & ~near
    assert not bad.any(), f"{int(bad.sum())} codes differ away from a rounding boundary"
    n_el = g_codes.size
    if exact:
        assert not mismatch.any(), f"{int(mismatch.sum())} codes differ"
    else:
        assert near.sum() <= MAX_EXEMPT_FRAC * n_el + 0.5, f"{int(near.sum())} near-boundary elements of {n_el}"
    # Scale/zero against the oracle's own append of the same tokens.
    o_codes = np.full(codes_gpu.shape, fill, np.uint8)
    o_sz = np.full(sz_gpu.shape, fill * 0x101, np.uint16)
    rc = O.append(w.dims, ks, vs, Rk, Rv, ck, cv, slots[idx], o_codes, o_sz, offset_k=offset_k)
    assert rc == 0
    o_szr = o_sz.reshape(NP, H, 2, P, D // G, 2)[page, :, :, off].view(np.float16).astype(np.float64)
    gs = g_sz.view(np.float16).astype(np.float64)
    ds = np.abs(gs[..., 0] - o_szr[..., 0])
    dz = np.abs(gs[..., 1] - o_szr[..., 1])
    assert np.all(ds <= SZ_RTOL * np.abs(o_szr[..., 0])), "scale mismatch"
    assert np.all(dz <= SZ_RTOL * np.maximum(np.abs(o_szr[..., 1]), o_szr[..., 0])), "zero mismatch"
    # Rows of slots nobody wrote keep the fill pattern.
    written = slots if written_slots is None else written_slots
    mask = np.zeros(NP * P, bool)
    ws = written[(written >= 0) & (written < NP * P)]
    mask[ws] = True
    untouched = np.nonzero(~mask)[0]
    if untouched.size:
        pu, ou = untouched // P, untouched % P
        assert np.all(rows[pu, :, :, ou] == fill), "bytes of an unwritten row changed"
        assert np.all(szr[pu, :, :, ou] == fill * 0x101), "scale/zero of an unwritten row changed"
    stats = dict(elements=n_el, near_boundary=int(near.sum()), mismatches=int(mismatch.sum()),
                 max_scale_rel=float(np.max(ds / np.maximum(np.abs(o_szr[..., 0]), 1e-30), initial=0.0)),
                 scale_diffs=int(np.count_nonzero(ds)), zero_diffs=int(np.count_nonzero(dz)))
    _log("append", stats)
    return stats


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:
        return max(1, min(32, os.cpu_count() or 1))


def oracle_decode_on_gpu_cache(w: Workload, cache, pairs=None, q=None, seq_lens=None, sm_scale=0.0) -> np.ndarray:
    """The oracle's decode of the GPU's cache; a list of (sequence, query head)
    pairs is spread over host threads (the oracle call releases the GIL)."""
    codes, sz = pools_to_host(cache)
    sink = bits16(cache.sink) if cache.sink is not None else None
    win = bits16(cache.window) if cache.window is not None else None
    qb = bits16(w.q if q is None else q)
    sl = (w.seq_lens if seq_lens is None else seq_lens).cpu().numpy()
    Rk, Rv, pt = w.R_k.cpu().numpy(), w.R_v.cpu().numpy(), w.page_table.numpy()

    def run(pr):
        return O.decode(w.dims, w.batch, qb, Rk, Rv, codes, sz, sink, win, pt, sl, w.sink_len, w.window_len,
                        sm_scale, pairs=pr)
    if pairs is None or len(pairs) < 2:
        return run(pairs)
    import concurrent.futures
    chunks = [list(c) for c in np.array_split(np.arange(len(pairs)), min(_threads(), len(pairs))) if len(c)]
    with concurrent.futures.ThreadPoolExecutor(len(chunks)) as ex:
        parts = list(ex.map(lambda ix: run([pairs[i] for i in ix]), chunks))
    return np.concatenate(parts, axis=0)


def oracle_extend_on_gpu_cache(w: Workload, cache, q: torch.Tensor, row_seq: np.ndarray, row_pos: np.ndarray,
                               pairs=None, sm_scale=0.0) -> np.ndarray:
    codes, sz = pools_to_host(cache)
    sink = bits16(cache.sink) if cache.sink is not None else None
    win = bits16(cache.window) if cache.window is not None else None
    return O.extend(w.dims, w.batch, bits16(q), row_seq, row_pos, w.R_k.cpu().numpy(), w.R_v.cpu().numpy(), codes,
                    sz, sink, win, w.page_table.numpy(), cache.seq_lens.cpu().numpy(), w.sink_len, w.window_len,
                    sm_scale, pairs=pairs)


def compare_decode(gpu_out: torch.Tensor, ref: np.ndarray, pairs=None) -> dict:
    g = gpu_out.detach().cpu().numpy().astype(np.float64)
    if pairs is not None:
        g = np.stack([g[b, h] for b, h in pairs])
    else:
        g = g.reshape(ref.shape)
    err = np.abs(g - ref)
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    stats = dict(max_abs=float(err.max(initial=0.0)), mean_abs=float(err.mean()) if err.size else 0.0,
                 ref_max=float(np.abs(ref).max(initial=0.0)), n=int(err.size))
    _log("decode", stats)
    assert stats["max_abs"] <= DEC_MAX_ABS, stats
    assert stats["mean_abs"] <= DEC_MEAN_ABS, stats
    return stats
