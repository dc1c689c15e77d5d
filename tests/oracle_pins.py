"""Pins of the CPU oracle: checks against closed forms, brute force, library
routines and hand-derived values -- never against the oracle itself.

Each ``pin_*`` function takes a loaded oracle library and raises
AssertionError on a mismatch.  ``test_oracle_pins.py`` runs them against the
real oracle; ``test_oracle_mutants.py`` runs them against copies of the oracle
with a planted mistake and requires that some pin fails for each mistake.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --- independent helpers (plain reading of the documented formats) ----------

def bf16_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_vals(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f16_val(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def unpack_row(pool: np.ndarray, dims: dict, page: int, h: int, kv: int, off: int) -> np.ndarray:
    """Codes of one stored row: pool uint8 [num_pages][Hkv][2][P][D/4]; element j
    in byte j // 4 at bits 2*(j % 4)."""
    D = dims["head_dim"]
    view = pool.reshape(dims["num_pages"], dims["num_kv_heads"], 2, dims["page_size"], D // 4)
    row = view[page, h, kv, off]
    return np.array([(int(row[j // 4]) >> (2 * (j % 4))) & 3 for j in range(D)], dtype=np.int64)


def sz_of_row(sz: np.ndarray, dims: dict, page: int, h: int, kv: int, off: int) -> tuple[np.ndarray, np.ndarray]:
    D, G = dims["head_dim"], dims["group_size"]
    view = sz.reshape(dims["num_pages"], dims["num_kv_heads"], 2, dims["page_size"], D // G, 2)
    r = view[page, h, kv, off]
    return f16_val(r[:, 0]), f16_val(r[:, 1])


def nearest_code(x: float, s: float, z: float) -> int:
    """Brute force: the code c in {0,1,2,3} minimising |x - (c*s + z)|, ties to
    the even code; a zero scale gives 0."""
    if s == 0.0:
        return 0
    best, best_err = None, None
    for c in range(4):
        err = abs(x - (c * s + z))
        if best is None or err < best_err - 1e-300 or (err == best_err and c % 2 == 0 and best % 2 == 1):
            best, best_err = c, err
    return best


def fwht(x: np.ndarray) -> np.ndarray:
    """Fast Walsh-Hadamard transform (Sylvester order), unnormalised."""
    y = x.astype(np.float64).copy()
    n = y.shape[0]
    hlen = 1
    while hlen < n:
        for i in range(0, n, 2 * hlen):
            a = y[i:i + hlen].copy()
            b = y[i + hlen:i + 2 * hlen].copy()
            y[i:i + hlen] = a + b
            y[i + hlen:i + 2 * hlen] = a - b
        hlen *= 2
    return y


def sylvester(n: int) -> np.ndarray:
    h = np.array([[1.0]])
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def exact_orthogonal(D: int, seed: int) -> np.ndarray:
    """An orthogonal matrix whose fp32 entries are exact: signed permutation of
    block-diagonal normalised 16x16 Hadamard blocks (entries +-1/4)."""
    rng = np.random.default_rng(seed)
    Hb = sylvester(16) / 4.0
    M = np.zeros((D, D))
    for b in range(D // 16):
        M[16 * b:16 * b + 16, 16 * b:16 * b + 16] = Hb
    perm = rng.permutation(D)
    signs = rng.choice([-1.0, 1.0], size=D)
    return (M[perm] * signs[None, :]).astype(np.float32)


def dense_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Textbook softmax(q K^T * scale) V in fp64."""
    logits = (K @ q) * scale
    w = np.exp(logits - logits.max())
    return (w[:, None] * V).sum(0) / w.sum()


def _dims(Hq, H, D, P, G, num_pages, max_pages):
    return dict(num_q_heads=Hq, num_kv_heads=H, head_dim=D, page_size=P, group_size=G, num_pages=num_pages,
                max_pages_per_seq=max_pages)


# --- number formats -----------------------------------------------------------

def pin_f16_rounding(lib):
    """fp64 -> fp16 (RNE) agrees with numpy's float32 -> float16 conversion."""
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
        np.array([0.0, -0.0, 1.0, 65504.0, 65519.0, 65520.0, 70000.0, -65520.0, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -14, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -10,
                  2049.0, 2051.0, -2049.0, 1e-9, 6.1e-5, 5.96e-8]),
    ]).astype(np.float32)
    got = O.f64_to_f16(vals.astype(np.float64), lib=lib)
    with np.errstate(over="ignore"):
        want = vals.astype(np.float16).view(np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"fp16 rounding differs at {vals[bad[:5]]}: {got[bad[:5]]} vs {want[bad[:5]]}"


def pin_f16_decode(lib):
    """fp16 bits -> value agrees with numpy for every finite pattern."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = O.f16_to_f64(bits, lib=lib)
    fin = np.isfinite(want)
    assert np.array_equal(got[fin], want[fin])
    assert np.all(np.isinf(got[np.isinf(want)])) and np.all(np.isnan(got[np.isnan(want)]))


def pin_bf16_decode(lib):
    rng = np.random.default_rng(12)
    bits = bf16_bits(rng.standard_normal(1000) * 100)
    got = O.bf16_to_f64(bits, lib=lib)
    want = torch.as_tensor(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(got, want)


# --- rotation / clip ----------------------------------------------------------

def pin_rotate_identity_and_permutation(lib):
    """R = I leaves x unchanged; a signed permutation permutes it exactly."""
    rng = np.random.default_rng(13)
    D = 64
    xb = bf16_bits(rng.standard_normal(D) * 5)
    x = bf16_vals(xb)
    assert np.array_equal(O.rotate(xb, np.eye(D, dtype=np.float32), lib=lib), x)
    perm = rng.permutation(D)
    signs = rng.choice([-1.0, 1.0], D)
    R = np.zeros((D, D), np.float32)
    R[perm, np.arange(D)] = signs       # x_rot[j] = signs[j] * x[perm[j]]
    assert np.array_equal(O.rotate(xb, R, lib=lib), signs * x[perm])


def pin_rotate_hadamard_fwht(lib):
    """R = H/sqrt(D) (normalised Sylvester Hadamard) equals an FWHT / sqrt(D)."""
    rng = np.random.default_rng(14)
    for D in (16, 64):
        xb = bf16_bits(rng.standard_normal(D))
        R = (sylvester(D) / math.sqrt(D)).astype(np.float32)
        got = O.rotate(xb, R, lib=lib)
        want = fwht(bf16_vals(xb)) * np.float64(np.float32(1 / math.sqrt(D)))
        assert np.allclose(got, want, rtol=0, atol=1e-12)


def pin_rotate_random_matmul(lib):
    """A random fp32 R agrees with a library fp64 matrix product."""
    rng = np.random.default_rng(15)
    D = 128
    xb = bf16_bits(rng.standard_normal(D) * 3)
    R = rng.standard_normal((D, D)).astype(np.float32)
    want = bf16_vals(xb) @ R.astype(np.float64)
    assert np.allclose(O.rotate(xb, R, lib=lib), want, rtol=1e-12, atol=1e-12)


def pin_clip(lib):
    x = np.array([-5.0, -1.0, 0.0, 0.5, 3.0, 7.0])
    c = np.array([1.0, 2.0, 0.0, np.inf, 3.0, 6.5], dtype=np.float32)
    assert np.array_equal(O.clip(x, c, lib=lib), np.array([-1.0, -1.0, 0.0, 0.5, 3.0, 6.5]))


# --- quantiser ------------------------------------------------------------------

def pin_group_params_library(lib):
    """scale/zero bits equal numpy's fp16 of fp32((max-min)/3) and fp32(min)."""
    rng = np.random.default_rng(16)
    for _ in range(300):
        xg = rng.standard_normal(64) * 10 ** rng.uniform(-3, 2)
        s, z = O.group_params(xg, lib=lib)
        ws = np.float16(np.float32((xg.max() - xg.min()) / 3.0)).view(np.uint16)
        wz = np.float16(np.float32(xg.min())).view(np.uint16)
        assert (s, z) == (int(ws), int(wz))


def pin_golden_groups(lib):
    """Hand-derived groups (tests/golden/int2_groups.json)."""
    with open(os.path.join(GOLDEN, "int2_groups.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        xg = np.array(case["x"], dtype=np.float64)
        s, z = O.group_params(xg, lib=lib)
        assert f16_val(s) == case["scale"] and f16_val(z) == case["zero"], case["name"]
        codes = [O.quantize(x, s, z, lib=lib)[0] for x in xg]
        assert codes == case["codes"], case["name"]


def pin_quantize_brute_force(lib):
    """The code is the nearest of the 4 levels (ties to even), in {0..3}."""
    rng = np.random.default_rng(17)
    for _ in range(3000):
        s = float(f16_val(np.float16(abs(rng.standard_normal()) * 2).view(np.uint16)))
        z = float(f16_val(np.float16(rng.standard_normal() * 3).view(np.uint16)))
        x = z + rng.uniform(-1.0, 4.0) * s
        sb = int(np.float16(s).view(np.uint16))
        zb = int(np.float16(z).view(np.uint16))
        c, u = O.quantize(x, sb, zb, lib=lib)
        assert c == nearest_code(x, s, z), (x, s, z, c)
        assert 0 <= c <= 3
    # exact ties go to the even code
    for k, want in ((0.5, 0), (1.5, 2), (2.5, 2)):
        c, _ = O.quantize(k, int(np.float16(1.0).view(np.uint16)), 0, lib=lib)
        assert c == want
    # zero scale
    assert O.quantize(3.0, 0, int(np.float16(3.0).view(np.uint16)), lib=lib)[0] == 0


# --- full append through the pool -------------------------------------------------

def _append_case(lib, D=64, G=32, H=2, P=16, T=40, R_kind="identity", clip_inf=True, seed=18, scale=1.0):
    rng = np.random.default_rng(seed)
    num_pages = 6
    dims = _dims(H, H, D, P, G, num_pages, 4)
    kb = bf16_bits(rng.standard_normal((T, H, D)) * scale)
    vb = bf16_bits(rng.standard_normal((T, H, D)) * scale)
    if R_kind == "identity":
        Rk = np.broadcast_to(np.eye(D, dtype=np.float32), (H, D, D)).copy()
        Rv = Rk.copy()
    else:
        Rk = np.stack([exact_orthogonal(D, seed + h) for h in range(H)])
        Rv = np.stack([exact_orthogonal(D, seed + 100 + h) for h in range(H)])
    if clip_inf:
        ck = np.full((H, D), np.inf, np.float32)
        cv = ck.copy()
    else:
        ck = (rng.uniform(0.3, 1.5, (H, D))).astype(np.float32)
        cv = (rng.uniform(0.3, 1.5, (H, D))).astype(np.float32)
    slots = rng.permutation(num_pages * P)[:T].astype(np.int64)
    slots[3] = -1
    pool = np.full(num_pages * H * 2 * P * (D // 4), 0xA5, np.uint8)
    sz = np.full(num_pages * H * 2 * P * (D // G) * 2, 0xA5A5, np.uint16)
    rc = O.append(dims, kb, vb, Rk, Rv, ck, cv, slots, pool, sz, lib=lib)
    return dims, kb, vb, Rk, Rv, ck, cv, slots, pool, sz, rc


def pin_append_identity_error_bound(lib):
    """R = I, infinite clip: every dequantised value is within scale/2 of the
    input (plus fp16 rounding slack of scale and zero at the ends, reading R4),
    codes are in {0..3}, and each code is the brute-force nearest level."""
    dims, kb, vb, Rk, Rv, ck, cv, slots, pool, sz, rc = _append_case(lib)
    assert rc == 0
    D, G, P = dims["head_dim"], dims["group_size"], dims["page_size"]
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        page, off = divmod(int(slot), P)
        for h in range(dims["num_kv_heads"]):
            for kv, src in ((0, kb), (1, vb)):
                x = bf16_vals(src[t, h])
                codes = unpack_row(pool, dims, page, h, kv, off)
                s, z = sz_of_row(sz, dims, page, h, kv, off)
                for g in range(D // G):
                    xs = x[g * G:(g + 1) * G]
                    s_exact = (xs.max() - xs.min()) / 3.0
                    slack = abs(z[g]) * 2.0 ** -11 + 3 * abs(s[g]) * 2.0 ** -11
                    deq = codes[g * G:(g + 1) * G] * s[g] + z[g]
                    assert np.all(np.abs(xs - deq) <= s_exact / 2 + slack + 1e-12)
                    for i in range(G):
                        assert codes[g * G + i] == nearest_code(xs[i], s[g], z[g])


def pin_append_layout_and_sentinel(lib):
    """Rows land at page slot // P, offset slot % P; rows of untouched slots and
    the token with slot < 0 leave the 0xA5 sentinel in place; an out-of-pool
    slot is reported."""
    dims, kb, vb, Rk, Rv, ck, cv, slots, pool, sz, rc = _append_case(lib, R_kind="exact", clip_inf=False)
    assert rc == 0
    P, D, G, H = dims["page_size"], dims["head_dim"], dims["group_size"], dims["num_kv_heads"]
    written = {int(s) for s in slots if s >= 0}
    view = pool.reshape(dims["num_pages"], H, 2, P, D // 4)
    szv = sz.reshape(dims["num_pages"], H, 2, P, D // G, 2)
    for slot in range(dims["num_pages"] * P):
        page, off = divmod(slot, P)
        if slot not in written:
            assert np.all(view[page, :, :, off] == 0xA5)
            assert np.all(szv[page, :, :, off] == 0xA5A5)
    # Values: x.R with the exact orthogonal R, then clip, then quantise.
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        page, off = divmod(int(slot), P)
        for h in range(H):
            for kv, src, R, c in ((0, kb, Rk, ck), (1, vb, Rv, cv)):
                y = bf16_vals(src[t, h]) @ R[h].astype(np.float64)
                y = np.minimum(np.maximum(y, -c[h].astype(np.float64)), c[h].astype(np.float64))
                codes = unpack_row(pool, dims, page, h, kv, off)
                s, z = sz_of_row(sz, dims, page, h, kv, off)
                for g in range(D // G):
                    ys = y[g * G:(g + 1) * G]
                    assert s[g] == np.float64(np.float16(np.float32((ys.max() - ys.min()) / 3.0)))
                    assert z[g] == np.float64(np.float16(np.float32(ys.min())))
                    for i in range(G):
                        assert codes[g * G + i] == nearest_code(ys[i], s[g], z[g])
    # out-of-pool slot
    bad = slots.copy()
    bad[0] = dims["num_pages"] * P
    rc = O.append(dims, kb, vb, Rk, Rv, ck, cv, bad, pool.copy(), sz.copy(), lib=lib)
    assert rc == -1


def pin_append_zero_clip_degenerate(lib):
    """clip = 0 collapses every group: scale 0, zero 0, codes 0."""
    rng = np.random.default_rng(19)
    D, G, H, P = 64, 32, 1, 16
    dims = _dims(1, H, D, P, G, 2, 2)
    kb = bf16_bits(rng.standard_normal((5, H, D)))
    R = np.eye(D, dtype=np.float32)[None]
    c0 = np.zeros((H, D), np.float32)
    pool = np.full(2 * H * 2 * P * D // 4, 0xFF, np.uint8)
    sz = np.full(2 * H * 2 * P * (D // G) * 2, 0xFFFF, np.uint16)
    O.append(dims, kb, kb, R, R, c0, c0, np.arange(5, dtype=np.int64), pool, sz, lib=lib)
    for t in range(5):
        for kv in range(2):
            assert np.all(unpack_row(pool, dims, 0, 0, kv, t) == 0)
            s, z = sz_of_row(sz, dims, 0, 0, kv, t)
            assert np.all(s == 0) and np.all(z == 0)


def pin_prequant_matches_append(lib):
    """The rotated+clipped values reported for exemption checks are the ones the
    codes were made from (brute-force nearest level against stored s,z)."""
    dims, kb, vb, Rk, Rv, ck, cv, slots, pool, sz, rc = _append_case(lib, R_kind="exact", clip_inf=False, T=12)
    pre = O.append_prequant(dims, kb, vb, Rk, Rv, ck, cv, lib=lib)
    P, D, G = dims["page_size"], dims["head_dim"], dims["group_size"]
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        page, off = divmod(int(slot), P)
        for h in range(dims["num_kv_heads"]):
            for kv, src, R, c in ((0, kb, Rk, ck), (1, vb, Rv, cv)):
                y = bf16_vals(src[t, h]) @ R[h].astype(np.float64)
                y = np.clip(y, -c[h].astype(np.float64), c[h].astype(np.float64))
                assert np.allclose(pre[t, h, kv], y, rtol=0, atol=1e-12)


# --- attention core ---------------------------------------------------------------

def pin_attend_rotation_equivalence(lib):
    """Attention with (q.R, K.R, V.R) then . R^T equals attention with (q, K, V)
    on unquantised data (exactly orthogonal R)."""
    rng = np.random.default_rng(20)
    D, n = 64, 37
    R = exact_orthogonal(D, 5)
    Rd = R.astype(np.float64)
    q = rng.standard_normal(D)
    K = rng.standard_normal((n, D)) * 3
    V = rng.standard_normal((n, D))
    plain = O.attend_mixed(q, q, K, V, np.zeros(n, np.int32), 0.125, R, lib=lib)
    rot = O.attend_mixed(q, q @ Rd, K @ Rd, V @ Rd, np.ones(n, np.int32), 0.125, R, lib=lib)
    assert np.allclose(plain, rot, rtol=0, atol=1e-12)
    # mixing spaces token by token changes nothing either
    mix = (np.arange(n) % 3 == 0).astype(np.int32)
    Km = np.where(mix[:, None] == 1, K @ Rd, K)
    Vm = np.where(mix[:, None] == 1, V @ Rd, V)
    mixed = O.attend_mixed(q, q @ Rd, Km, Vm, mix, 0.125, R, lib=lib)
    assert np.allclose(plain, mixed, rtol=0, atol=1e-12)
    # and equals the textbook routine
    assert np.allclose(plain, dense_attention(q, K, V, 0.125), rtol=0, atol=1e-12)


# --- full decode --------------------------------------------------------------------

def _decode_case(lib, *, L, S, W, D=64, G=32, Hq=2, H=1, P=16, seed=21, zero_q=False, exact_R=True,
                 shuffle=True, num_pages=None):
    rng = np.random.default_rng(seed)
    max_pages = max(1, -(-L // P))
    num_pages = num_pages or max_pages + 3
    dims = _dims(Hq, H, D, P, G, num_pages, max_pages)
    kb = bf16_bits(rng.standard_normal((L, H, D)) * 2)
    vb = bf16_bits(rng.standard_normal((L, H, D)))
    if exact_R:
        Rk = np.stack([exact_orthogonal(D, seed + h) for h in range(H)])
        Rv = np.stack([exact_orthogonal(D, seed + 50 + h) for h in range(H)])
    else:
        Rk = np.stack([np.linalg.qr(rng.standard_normal((D, D)))[0] for _ in range(H)]).astype(np.float32)
        Rv = np.stack([np.linalg.qr(rng.standard_normal((D, D)))[0] for _ in range(H)]).astype(np.float32)
    ck = np.full((H, D), np.inf, np.float32)
    pages = rng.permutation(num_pages)[:max_pages] if shuffle else np.arange(max_pages)
    page_table = pages.astype(np.int32)[None]
    slots = np.array([page_table[0, p // P] * P + p % P for p in range(L)], np.int64)
    pool = np.zeros(num_pages * H * 2 * P * D // 4, np.uint8)
    sz = np.zeros(num_pages * H * 2 * P * (D // G) * 2, np.uint16)
    assert O.append(dims, kb, vb, Rk, Rv, ck, ck, slots, pool, sz, lib=lib) == 0
    Sb, Wb = max(S, 1), max(W, 1)
    sink = np.zeros((1, 2, H, Sb, D), np.uint16)
    win = np.zeros((1, 2, H, Wb, D), np.uint16)
    for p in range(min(S, L)):
        sink[0, 0, :, p] = kb[p]
        sink[0, 1, :, p] = vb[p]
    for p in range(max(S, L - W), L):
        win[0, 0, :, p % Wb] = kb[p]
        win[0, 1, :, p % Wb] = vb[p]
    qb = np.zeros((1, Hq, D), np.uint16) if zero_q else bf16_bits(rng.standard_normal((1, Hq, D)))
    out = O.decode(dims, 1, qb, Rk, Rv, pool, sz, sink, win, page_table, np.array([L], np.int32), S, W, 0.0,
                   lib=lib)
    return dict(dims=dims, kb=kb, vb=vb, Rk=Rk, Rv=Rv, pool=pool, sz=sz, sink=sink, win=win, qb=qb,
                page_table=page_table, L=L, S=S, W=W, out=out)


def _bulk_dequant(c, p, kv):
    d = c["dims"]
    P = d["page_size"]
    page = int(c["page_table"][0, p // P])
    out = []
    for h in range(d["num_kv_heads"]):
        codes = unpack_row(c["pool"], d, page, h, kv, p % P)
        s, z = sz_of_row(c["sz"], d, page, h, kv, p % P)
        G = d["group_size"]
        out.append(np.array([codes[j] * s[j // G] + z[j // G] for j in range(d["head_dim"])]))
    return np.stack(out)


def pin_decode_all_bf16(lib):
    """sink + window cover every token: the output is textbook dense softmax
    attention over the bf16 K/V (no INT2 read)."""
    # (30, 4, 32): the window holds fewer than W tokens, so the ring slot p % W
    # matters (a full window is only a permutation, which softmax ignores).
    for L, S, W in ((40, 8, 32), (20, 32, 8), (1, 4, 4), (33, 0, 40), (30, 4, 32)):
        c = _decode_case(lib, L=L, S=S, W=W)
        d = c["dims"]
        gqa = d["num_q_heads"] // d["num_kv_heads"]
        for hq in range(d["num_q_heads"]):
            h = hq // gqa
            want = dense_attention(bf16_vals(c["qb"][0, hq]), bf16_vals(c["kb"][:, h]), bf16_vals(c["vb"][:, h]),
                                   1 / math.sqrt(d["head_dim"]))
            assert np.allclose(c["out"][hq], want, rtol=0, atol=1e-12), (L, S, W)


def pin_decode_zero_query_mean(lib):
    """q = 0: every logit is 0, so the output is the plain mean over the L tokens
    of v (bf16 v for sink/window, dequantised v . R_v^T for the bulk)."""
    for L, S, W in ((100, 4, 32), (77, 0, 5), (64, 16, 0)):
        c = _decode_case(lib, L=L, S=S, W=W, zero_q=True, exact_R=False, seed=22)
        d = c["dims"]
        gqa = d["num_q_heads"] // d["num_kv_heads"]
        for hq in range(d["num_q_heads"]):
            h = hq // gqa
            acc = np.zeros(d["head_dim"])
            for p in range(L):
                if p < S or p >= max(S, L - W):
                    acc += bf16_vals(c["vb"][p, h])
                else:
                    acc += _bulk_dequant(c, p, 1)[h] @ c["Rv"][h].astype(np.float64).T
            assert np.allclose(c["out"][hq], acc / L, rtol=0, atol=1e-11), (L, S, W)


def pin_decode_single_token(lib):
    """L = 1: the output is v_0 (from the sink when S >= 1, from the window otherwise)."""
    for S, W in ((1, 8), (0, 8), (4, 0)):
        c = _decode_case(lib, L=1, S=S, W=W)
        for hq in range(c["dims"]["num_q_heads"]):
            h = hq // (c["dims"]["num_q_heads"] // c["dims"]["num_kv_heads"])
            assert np.allclose(c["out"][hq], bf16_vals(c["vb"][0, h]), rtol=0, atol=1e-14)
    # L = 1 with no sink and no window: the only token is INT2
    c = _decode_case(lib, L=1, S=0, W=0, exact_R=False)
    want = _bulk_dequant(c, 0, 1)[0] @ c["Rv"][0].astype(np.float64).T
    assert np.allclose(c["out"][0], want, rtol=0, atol=1e-12)


def pin_decode_brute_force_small(lib):
    """Brute force with plain Python loops on a 6-token case (sink 1, window 2,
    3 INT2 tokens across a page boundary, page size 2, D=8, G=4, GQA 2)."""
    rng = np.random.default_rng(23)
    D, G, P, Hq, H, L, S, W = 8, 4, 2, 2, 1, 6, 1, 2
    num_pages = 5
    dims = _dims(Hq, H, D, P, G, num_pages, 3)
    kb = bf16_bits(rng.standard_normal((L, H, D)) * 2)
    vb = bf16_bits(rng.standard_normal((L, H, D)))
    Rk = np.linalg.qr(rng.standard_normal((D, D)))[0].astype(np.float32)[None]
    Rv = np.linalg.qr(rng.standard_normal((D, D)))[0].astype(np.float32)[None]
    ck = np.full((H, D), 1.2, np.float32)
    pt = np.array([[4, 0, 2]], np.int32)
    slots = np.array([pt[0, p // P] * P + p % P for p in range(L)], np.int64)
    pool = np.zeros(num_pages * H * 2 * P * D // 4, np.uint8)
    sz = np.zeros(num_pages * H * 2 * P * (D // G) * 2, np.uint16)
    assert O.append(dims, kb, vb, Rk, Rv, ck, ck, slots, pool, sz, lib=lib) == 0
    sink = np.zeros((1, 2, H, S, D), np.uint16)
    win = np.zeros((1, 2, H, W, D), np.uint16)
    sink[0, 0, 0, 0], sink[0, 1, 0, 0] = kb[0, 0], vb[0, 0]
    for p in (4, 5):
        win[0, 0, 0, p % W], win[0, 1, 0, p % W] = kb[p, 0], vb[p, 0]
    qb = bf16_bits(rng.standard_normal((1, Hq, D)))
    out = O.decode(dims, 1, qb, Rk, Rv, pool, sz, sink, win, pt, np.array([L], np.int32), S, W, 0.3, lib=lib)
    for hq in range(Hq):
        q = [float(x) for x in bf16_vals(qb[0, hq])]
        qr = [sum(q[i] * float(Rk[0, i, j]) for i in range(D)) for j in range(D)]
        logits, values, rotated = [], [], []
        for p in range(L):
            if p < S or p >= L - W:
                kk = [float(x) for x in bf16_vals(kb[p, 0])]
                vv = [float(x) for x in bf16_vals(vb[p, 0])]
                logits.append(0.3 * sum(q[j] * kk[j] for j in range(D)))
                rotated.append(False)
            else:
                page, off = int(pt[0, p // P]), p % P
                kc, vc = unpack_row(pool, dims, page, 0, 0, off), unpack_row(pool, dims, page, 0, 1, off)
                ks, kz = sz_of_row(sz, dims, page, 0, 0, off)
                vs, vz = sz_of_row(sz, dims, page, 0, 1, off)
                kk = [kc[j] * ks[j // G] + kz[j // G] for j in range(D)]
                vv = [vc[j] * vs[j // G] + vz[j // G] for j in range(D)]
                logits.append(0.3 * sum(qr[j] * kk[j] for j in range(D)))
                rotated.append(True)
            values.append(vv)
        m = max(logits)
        w = [math.exp(x - m) for x in logits]
        tot = sum(w)
        o = [0.0] * D
        for p in range(L):
            if rotated[p]:
                for c in range(D):
                    o[c] += w[p] / tot * sum(values[p][j] * float(Rv[0, c, j]) for j in range(D))
            else:
                for c in range(D):
                    o[c] += w[p] / tot * values[p][c]
        assert np.allclose(out[hq], o, rtol=0, atol=1e-12)


def pin_decode_page_shuffle_invariance(lib):
    """Moving every page to another physical page (and updating the table)
    leaves the output bit-identical."""
    c = _decode_case(lib, L=150, S=4, W=20, seed=24)
    d = c["dims"]
    rng = np.random.default_rng(25)
    perm = rng.permutation(d["num_pages"])  # new physical id of old page i is perm[i]
    per_page_codes = c["pool"].reshape(d["num_pages"], -1)
    per_page_sz = c["sz"].reshape(d["num_pages"], -1)
    pool2 = np.empty_like(per_page_codes)
    sz2 = np.empty_like(per_page_sz)
    pool2[perm] = per_page_codes
    sz2[perm] = per_page_sz
    pt2 = perm[c["page_table"]].astype(np.int32)
    out2 = O.decode(d, 1, c["qb"], c["Rk"], c["Rv"], pool2.ravel(), sz2.ravel(), c["sink"], c["win"], pt2,
                    np.array([c["L"]], np.int32), c["S"], c["W"], 0.0, lib=lib)
    assert np.array_equal(out2, c["out"])


def pin_decode_gqa_mapping(lib):
    """Query head hq reads KV head hq // (Hq/Hkv): with two KV heads whose caches
    differ, each query head's output equals a one-head decode of its KV head."""
    rng = np.random.default_rng(26)
    D, G, P, L, S, W = 64, 32, 16, 70, 4, 16
    Hq, H = 4, 2
    num_pages = 6
    dims = _dims(Hq, H, D, P, G, num_pages, 5)
    kb = bf16_bits(rng.standard_normal((L, H, D)))
    vb = bf16_bits(rng.standard_normal((L, H, D)))
    Rk = np.stack([exact_orthogonal(D, 1), exact_orthogonal(D, 2)])
    Rv = np.stack([exact_orthogonal(D, 3), exact_orthogonal(D, 4)])
    ck = np.full((H, D), np.inf, np.float32)
    pt = np.array([[5, 3, 1, 0, 2]], np.int32)
    slots = np.array([pt[0, p // P] * P + p % P for p in range(L)], np.int64)
    pool = np.zeros(num_pages * H * 2 * P * D // 4, np.uint8)
    sz = np.zeros(num_pages * H * 2 * P * (D // G) * 2, np.uint16)
    O.append(dims, kb, vb, Rk, Rv, ck, ck, slots, pool, sz, lib=lib)
    sink = np.zeros((1, 2, H, S, D), np.uint16)
    win = np.zeros((1, 2, H, W, D), np.uint16)
    for p in range(S):
        sink[0, 0, :, p], sink[0, 1, :, p] = kb[p], vb[p]
    for p in range(L - W, L):
        win[0, 0, :, p % W], win[0, 1, :, p % W] = kb[p], vb[p]
    qb = bf16_bits(rng.standard_normal((1, Hq, D)))
    out = O.decode(dims, 1, qb, Rk, Rv, pool, sz, sink, win, pt, np.array([L], np.int32), S, W, 0.0, lib=lib)
    for h in range(H):
        d1 = _dims(2, 1, D, P, G, num_pages, 5)
        pool1 = pool.reshape(num_pages, H, -1)[:, h].copy().ravel()
        sz1 = sz.reshape(num_pages, H, -1)[:, h].copy().ravel()
        o1 = O.decode(d1, 1, qb[:, 2 * h:2 * h + 2], Rk[h:h + 1], Rv[h:h + 1], pool1, sz1,
                      sink[:, :, h:h + 1].copy(), win[:, :, h:h + 1].copy(), pt, np.array([L], np.int32), S, W,
                      0.0, lib=lib)
        assert np.array_equal(out[2 * h:2 * h + 2], o1)


def pin_decode_closed_form_golden(lib):
    """Two bf16 tokens with logits 0 and a: weights 1/(1+e^a), e^a/(1+e^a)
    (tests/golden/decode_two_tokens.json)."""
    with open(os.path.join(GOLDEN, "decode_two_tokens.json")) as f:
        g = json.load(f)
    D, P = 4, 4
    dims = _dims(1, 1, D, P, 4, 1, 1)
    sink = bf16_bits(np.array(g["sink_kv"], np.float32)).reshape(1, 2, 1, 1, D)
    win = bf16_bits(np.array(g["window_kv"], np.float32)).reshape(1, 2, 1, 1, D)
    qb = bf16_bits(np.array(g["q"], np.float32)).reshape(1, 1, D)
    R = np.eye(D, dtype=np.float32)[None]
    out = O.decode(dims, 1, qb, R, R, np.zeros(P, np.uint8), np.zeros(2 * P * 2, np.uint16), sink, win,
                   np.zeros((1, 1), np.int32), np.array([2], np.int32), 1, 1, g["sm_scale"], lib=lib)
    a = g["logit_gap"]
    w1 = math.exp(a) / (1 + math.exp(a))
    want = (1 - w1) * np.array(g["sink_kv"][1]) + w1 * np.array(g["window_kv"][1])
    assert np.allclose(out[0], want, rtol=0, atol=1e-12)
    assert np.allclose(out[0], g["expected_out"], rtol=0, atol=1e-9)


def pin_bf16_decode_dense(lib):
    """The BF16 paged decode equals textbook dense attention over the gathered pages."""
    rng = np.random.default_rng(27)
    D, P, H, Hq, L = 64, 16, 2, 4, 83
    num_pages = 9
    dims = _dims(Hq, H, D, P, 64, num_pages, 6)
    pages = bf16_bits(rng.standard_normal((num_pages, H, 2, P, D)))
    pt = rng.permutation(num_pages)[:6].astype(np.int32)[None]
    qb = bf16_bits(rng.standard_normal((1, Hq, D)))
    out = O.bf16_decode(dims, 1, qb, pages, pt, np.array([L], np.int32), 0.0, lib=lib)
    for hq in range(Hq):
        h = hq // 2
        K = np.stack([bf16_vals(pages[pt[0, p // P], h, 0, p % P]) for p in range(L)])
        V = np.stack([bf16_vals(pages[pt[0, p // P], h, 1, p % P]) for p in range(L)])
        assert np.allclose(out[hq], dense_attention(bf16_vals(qb[0, hq]), K, V, 1 / 8), rtol=0, atol=1e-12)


def _mixed_inputs(seed=31, lens=(5, 40, 70), S=4, W=16, D=64, G=32, H=2, P=16):
    """Tokens of several sequences in position order, random slots of one pool."""
    rng = np.random.default_rng(seed)
    T = sum(lens)
    num_pages = (T + P - 1) // P + 3
    dims = _dims(H, H, D, P, G, num_pages, (max(lens) + P - 1) // P)
    kb = bf16_bits(rng.standard_normal((T, H, D)))
    vb = bf16_bits(rng.standard_normal((T, H, D)))
    Rk = np.stack([exact_orthogonal(D, seed + h) for h in range(H)])
    Rv = np.stack([exact_orthogonal(D, seed + 50 + h) for h in range(H)])
    ck = np.full((H, D), np.inf, np.float32)
    cv = ck.copy()
    slots = rng.permutation(num_pages * P)[:T].astype(np.int64)
    seq = np.concatenate([np.full(L, b, np.int32) for b, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens])
    return dict(dims=dims, kb=kb, vb=vb, Rk=Rk, Rv=Rv, ck=ck, cv=cv, slots=slots, seq=seq, pos=pos,
                lens=np.array(lens, np.int32), S=S, W=W, D=D, G=G, H=H, P=P, num_pages=num_pages)


def _mixed_buffers(c):
    B, H, D, P, G = len(c["lens"]), c["H"], c["D"], c["P"], c["G"]
    pool = np.full(c["num_pages"] * H * 2 * P * (D // 4), 0xA5, np.uint8)
    sz = np.full(c["num_pages"] * H * 2 * P * (D // G) * 2, 0xA5A5, np.uint16)
    sink = np.full((B, 2, H, max(c["S"], 1), D), 0xFFFF, np.uint16)
    win = np.full((B, 2, H, max(c["W"], 1), D), 0xFFFF, np.uint16)
    return pool, sz, sink, win


def _mixed_call(lib, c, idx, lens_now, bufs):
    pool, sz, sink, win = bufs
    return O.append_mixed(c["dims"], c["kb"][idx], c["vb"][idx], c["Rk"], c["Rv"], c["ck"], c["cv"],
                          c["slots"][idx], c["seq"][idx], c["pos"][idx], lens_now, c["S"], c["W"],
                          pool, sz, sink, win, lib=lib)


def _attended_rows(L, S, W):
    """(buffer, row, position) of every row the decode reads for length L."""
    rows = [("sink", p, p) for p in range(min(S, L))]
    rows += [("win", p % W, p) for p in range(max(S, L - W), L)] if W > 0 else []
    return rows


def pin_append_mixed_streaming_equals_batch(lib):
    """One append of every token (final lengths) leaves the same INT2 pool and the
    same attended sink/window rows as appending the tokens one at a time in
    position order (each with its length at that time): the batch rule that skips
    window rows a later token of the same append overwrites is the streaming ring."""
    c = _mixed_inputs()
    batch = _mixed_buffers(c)
    assert _mixed_call(lib, c, np.arange(len(c["seq"])), c["lens"], batch) == 0
    stream = _mixed_buffers(c)
    order = sorted(range(len(c["seq"])), key=lambda t: (c["pos"][t], c["seq"][t]))
    now = np.zeros_like(c["lens"])
    for t in order:
        now[c["seq"][t]] = c["pos"][t] + 1
        assert _mixed_call(lib, c, np.array([t]), now.copy(), stream) == 0
    assert np.array_equal(batch[0], stream[0]) and np.array_equal(batch[1], stream[1])
    for b, L in enumerate(c["lens"]):
        for buf, row, _ in _attended_rows(int(L), c["S"], c["W"]):
            i = 2 if buf == "sink" else 3
            assert np.array_equal(batch[i][b, :, :, row], stream[i][b, :, :, row]), (b, buf, row)


def pin_append_mixed_bf16_rows_and_int2(lib):
    """The attended sink/window rows hold the token's original bf16 K and V (read
    straight from the inputs by position), rows the decode never reads are not
    written, and the INT2 pool equals that of the plain append."""
    c = _mixed_inputs(seed=33, lens=(3, 20, 37), S=8, W=12)
    bufs = _mixed_buffers(c)
    assert _mixed_call(lib, c, np.arange(len(c["seq"])), c["lens"], bufs) == 0
    pool, sz, sink, win = bufs
    ref_pool, ref_sz, _, _ = _mixed_buffers(c)
    O.append(c["dims"], c["kb"], c["vb"], c["Rk"], c["Rv"], c["ck"], c["cv"], c["slots"], ref_pool, ref_sz, lib=lib)
    assert np.array_equal(pool, ref_pool) and np.array_equal(sz, ref_sz)
    start = np.concatenate([[0], np.cumsum(c["lens"])[:-1]])
    for b, L in enumerate(c["lens"]):
        seen_sink, seen_win = set(), set()
        for buf, row, p in _attended_rows(int(L), c["S"], c["W"]):
            t = start[b] + p
            got = (sink if buf == "sink" else win)[b, :, :, row]
            assert np.array_equal(got[0], c["kb"][t]) and np.array_equal(got[1], c["vb"][t]), (b, buf, p)
            (seen_sink if buf == "sink" else seen_win).add(row)
        for r in range(c["S"]):
            if r not in seen_sink:
                assert np.all(sink[b, :, :, r] == 0xFFFF)
        for r in range(c["W"]):
            if r not in seen_win:
                assert np.all(win[b, :, :, r] == 0xFFFF)


# --- key offset removal (OptR abstract on the OSCAR paper page) ------------------

def _golden_offset():
    with open(os.path.join(GOLDEN, "key_offset.json")) as f:
        return json.load(f)


def pin_key_offset_golden_differences(lib):
    """fp32(k - c) and its bf16 rounding for hand-derived keys and offsets
    (tests/golden/key_offset.json): both round to nearest even."""
    for case in _golden_offset()["differences"]:
        k = np.array([case["k_bits"]], np.uint16)
        c = np.array([float.fromhex(case["c"])], np.float32)
        got = float(O.offset_key(k, c, lib=lib)[0])
        assert got == float.fromhex(case["diff"]), case["name"]
        assert int(O.f32_to_bf16(np.float32(got), lib=lib)) == case["bf16_bits"], case["name"]


def pin_key_offset_golden_append(lib):
    """One token appended with a key offset (R = I, infinite clip, sink of one
    row): the INT2 codes, scale and zero are those of k - c, V is untouched, the
    BF16 sink rows hold bf16(k - c) and v (tests/golden/key_offset.json)."""
    g = _golden_offset()["append"]
    dims = g["dims"]
    D, P, G = dims["head_dim"], dims["page_size"], dims["group_size"]
    kb = bf16_bits(np.array(g["k"]).reshape(1, 1, D))
    vb = bf16_bits(np.array(g["v"]).reshape(1, 1, D))
    R = np.eye(D, dtype=np.float32)[None]
    ck = np.full((1, D), np.inf, np.float32)
    off = np.array(g["offset_k"], np.float32).reshape(1, D)
    pre = O.append_prequant(dims, kb, vb, R, R, ck, ck, offset_k=off, lib=lib)
    assert np.array_equal(pre[0, 0, 0], g["k_shifted"]) and np.array_equal(pre[0, 0, 1], g["v"])
    pool = np.full(P * 2 * (D // 4), 0xA5, np.uint8)
    sz = np.full(P * 2 * (D // G) * 2, 0xA5A5, np.uint16)
    sink = np.full((1, 2, 1, 1, D), 0xFFFF, np.uint16)
    win = np.full((1, 2, 1, 1, D), 0xFFFF, np.uint16)
    one = np.array([1], np.int32)
    zero = np.array([0], np.int32)
    rc = O.append_mixed(dims, kb, vb, R, R, ck, ck, np.array([g["slot"]], np.int64), zero, zero, one, 1, 0, pool,
                        sz, sink, win, offset_k=off, lib=lib)
    assert rc == 0
    szv = sz.reshape(2, P, D // G, 2)
    assert pool[0] == g["k_code_byte"] and pool[P] == g["v_code_byte"]
    assert tuple(szv[0, 0, 0]) == (g["k_scale_bits"], g["k_zero_bits"])
    assert tuple(szv[1, 0, 0]) == (g["v_scale_bits"], g["v_zero_bits"])
    assert list(sink[0, 0, 0, 0]) == g["k_row_bf16_bits"] and list(sink[0, 1, 0, 0]) == g["v_row_bf16_bits"]
    assert np.all(pool[1:P] == 0xA5) and np.all(pool[P + 1:] == 0xA5)


def _offset_case(seed):
    """Keys and per-(head, channel) offsets on a 1/16 grid, so that k - c has at
    most 7 significant bits and is exact in bf16; finite clips."""
    rng = np.random.default_rng(seed)
    c = _mixed_inputs(seed=seed, lens=(6, 30, 45), S=4, W=12)
    H, D = c["H"], c["D"]
    k = rng.integers(-64, 65, size=c["kb"].shape) / 16.0
    off = (rng.integers(-32, 33, size=(H, D)) / 16.0).astype(np.float32)
    c["kb"] = bf16_bits(k)
    c["shifted"] = bf16_bits(k - off[None].astype(np.float64))
    assert np.array_equal(bf16_vals(c["shifted"]), k - off[None])
    c["ck"] = rng.uniform(1.0, 3.0, (H, D)).astype(np.float32)
    c["cv"] = rng.uniform(1.0, 3.0, (H, D)).astype(np.float32)
    return c, off


def _mixed_with(lib, c, keys, offset):
    bufs = _mixed_buffers(c)
    n = len(c["seq"])
    rc = O.append_mixed(c["dims"], keys, c["vb"], c["Rk"], c["Rv"], c["ck"], c["cv"], c["slots"], c["seq"],
                        c["pos"], c["lens"], c["S"], c["W"], *bufs, offset_k=offset, lib=lib)
    assert rc == 0 and n == keys.shape[0]
    return bufs


def pin_key_offset_equals_shifted_input(lib):
    """With k - c exact in bf16, appending k with the offset c leaves the same
    INT2 pool, scale/zero and BF16 sink/window as appending k - c with no offset
    (values untouched, each KV head with its own offset); a zero offset is no
    offset."""
    c, off = _offset_case(61)
    with_off = _mixed_with(lib, c, c["kb"], off)
    shifted = _mixed_with(lib, c, c["shifted"], None)
    for a, b in zip(with_off, shifted):
        assert np.array_equal(a, b)
    zero = _mixed_with(lib, c, c["kb"], np.zeros_like(off))
    none = _mixed_with(lib, c, c["kb"], None)
    for a, b in zip(zero, none):
        assert np.array_equal(a, b)
    assert not np.array_equal(with_off[0], none[0])     # the offset did change the INT2 keys


def pin_key_offset_softmax_invariance(lib):
    """Every key in the BF16 sink/window (S + W >= L) and k - c exact in bf16:
    the decode of the cache appended with an offset equals textbook attention
    over the ORIGINAL keys, since q . c is the same for every key of a query."""
    c, off = _offset_case(62)
    d = c["dims"]
    H, D, P = c["H"], c["D"], c["P"]
    c["W"] = 64                                          # S + W >= every length
    pool, sz, sink, win = _mixed_with(lib, c, c["kb"], off)
    rng = np.random.default_rng(63)
    B = len(c["lens"])
    qb = bf16_bits(rng.standard_normal((B, d["num_q_heads"], D)))
    pt = np.zeros((B, d["max_pages_per_seq"]), np.int32)   # no INT2 page is read
    out = O.decode(d, B, qb, c["Rk"], c["Rv"], pool, sz, sink, win, pt, c["lens"], c["S"], c["W"], 0.0, lib=lib)
    out = out.reshape(B, d["num_q_heads"], D)
    start = np.concatenate([[0], np.cumsum(c["lens"])[:-1]])
    gqa = d["num_q_heads"] // H
    for b, L in enumerate(c["lens"]):
        rows = slice(start[b], start[b] + L)
        for hq in range(d["num_q_heads"]):
            h = hq // gqa
            want = dense_attention(bf16_vals(qb[b, hq]), bf16_vals(c["kb"][rows, h]), bf16_vals(c["vb"][rows, h]),
                                   1 / math.sqrt(D))
            assert np.allclose(out[b, hq], want, rtol=0, atol=1e-11), (b, hq)


def _extend_rows(lib, c, rows_pos, seed=41, row_seq=None):
    """Extend output [rows][Hq][D] over the single-sequence cache of case ``c`` for query rows
    at the given positions (fresh queries)."""
    d = c["dims"]
    rng = np.random.default_rng(seed)
    nr = len(rows_pos)
    qb = bf16_bits(rng.standard_normal((nr, d["num_q_heads"], d["head_dim"])))
    rs = np.zeros(nr, np.int32) if row_seq is None else np.asarray(row_seq, np.int32)
    out = O.extend(d, 1, qb, rs, np.asarray(rows_pos, np.int32), c["Rk"], c["Rv"], c["pool"], c["sz"], c["sink"],
                   c["win"], c["page_table"], np.array([c["L"]], np.int32), c["S"], c["W"], 0.0, lib=lib)
    return qb, out.reshape(nr, d["num_q_heads"], d["head_dim"])


def pin_extend_last_row_is_decode(lib):
    """A query row at the last position L - 1 is the decode query: identical output."""
    for L, S, W in ((70, 4, 16), (33, 0, 0), (50, 8, 64)):
        c = _decode_case(lib, L=L, S=S, W=W, exact_R=False, seed=43)
        d = c["dims"]
        out = O.extend(d, 1, c["qb"], np.zeros(1, np.int32), np.array([L - 1], np.int32), c["Rk"], c["Rv"],
                       c["pool"], c["sz"], c["sink"], c["win"], c["page_table"], np.array([L], np.int32), S, W,
                       0.0, lib=lib)
        assert np.array_equal(out, c["out"]), (L, S, W)


def pin_extend_all_bf16_is_causal_dense(lib):
    """sink + window hold the whole cache: the row at position p is textbook dense
    softmax attention over the bf16 K/V of positions 0..p."""
    for L, S, W in ((40, 8, 32), (30, 0, 40), (25, 25, 0)):
        c = _decode_case(lib, L=L, S=S, W=W, seed=44)
        d = c["dims"]
        gqa = d["num_q_heads"] // d["num_kv_heads"]
        rows = [0, 3, L // 2, L - 2, L - 1]
        qb, out = _extend_rows(lib, c, rows, seed=45)
        for i, p in enumerate(rows):
            for hq in range(d["num_q_heads"]):
                h = hq // gqa
                want = dense_attention(bf16_vals(qb[i, hq]), bf16_vals(c["kb"][: p + 1, h]),
                                       bf16_vals(c["vb"][: p + 1, h]), 1 / math.sqrt(d["head_dim"]))
                assert np.allclose(out[i, hq], want, rtol=0, atol=1e-12), (L, S, W, p)


def pin_extend_causal_brute_force(lib):
    """Mixed cache (sink, INT2 bulk, window ring of the final length L): each row at
    position p, by a plain loop over positions 0..p with the split of length L."""
    L, S, W = 60, 4, 16
    c = _decode_case(lib, L=L, S=S, W=W, exact_R=False, seed=46)
    d = c["dims"]
    D, gqa = d["head_dim"], d["num_q_heads"] // d["num_kv_heads"]
    rows = [0, 2, 3, 5, 20, 43, 44, 50, 59]
    qb, out = _extend_rows(lib, c, rows, seed=47)
    scale = 1 / math.sqrt(D)
    for i, p in enumerate(rows):
        for hq in range(d["num_q_heads"]):
            h = hq // gqa
            q = bf16_vals(qb[i, hq])
            qr = q @ c["Rk"][h].astype(np.float64)
            logits, vals, rot = [], [], []
            for t in range(p + 1):
                if t < S or t >= max(S, L - W):
                    logits.append(scale * float(q @ bf16_vals(c["kb"][t, h])))
                    vals.append(bf16_vals(c["vb"][t, h]))
                    rot.append(False)
                else:
                    logits.append(scale * float(qr @ _bulk_dequant(c, t, 0)[h]))
                    vals.append(_bulk_dequant(c, t, 1)[h])
                    rot.append(True)
            w = np.exp(np.array(logits) - max(logits))
            plain = sum(w[k] * vals[k] for k in range(p + 1) if not rot[k])
            rotd = sum(w[k] * vals[k] for k in range(p + 1) if rot[k])
            want = (plain + (rotd @ c["Rv"][h].astype(np.float64).T if any(rot) else 0)) / w.sum()
            assert np.allclose(out[i, hq], want, rtol=0, atol=1e-11), (p, hq)


def pin_extend_rejects_out_of_range_rows(lib):
    """A row at a position >= L or of a sequence outside the batch is refused."""
    c = _decode_case(lib, L=20, S=2, W=4, seed=48)
    for pos, seq in ((20, 0), (-1, 0), (3, 1), (3, -1)):
        try:
            _extend_rows(lib, c, [pos], row_seq=[seq])
        except ValueError:
            continue
        raise AssertionError(f"row at position {pos} of sequence {seq} was accepted")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
