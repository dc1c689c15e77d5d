"""GPU calibration (oscar_calibrate) against the fp64 calibration oracle.

What is unique is compared directly: the covariance, the eigenvalues, the
eigenvectors whose eigenvalue stands apart (a posteriori bound from the
residual against the oracle's covariance) and the clipping thresholds of those
columns.  Where eigenvalues (nearly) coincide the eigenbasis is open, so the
GPU result is checked for validity instead: R orthogonal, R^T C R diagonal with
the GPU eigenvalues on it (against the oracle's C), descending order, the sign
rule, and every threshold equal to the k-th smallest |x . r_j| of its own
column (fp64) within the rounding of the tensor-core rotation.
"""

import numpy as np
import pytest
import torch

from int2_rotated_kv_append_gb300.cache import calibrate
from int2_rotated_kv_append_gb300.synth import bits16, calibration_samples
from oracle import calibration as CAL

pytestmark = pytest.mark.gpu

COV_RTOL = 2e-5      # chunk sums, centring and fp32 storage: |dC_ij| <= (COV_RTOL + acc) sqrt(M_ii M_jj)
RESID_RTOL = 1e-4    # backward error of the fp32 Jacobi relative to lambda_max
ORTHO_TOL = 2e-5     # |R^T R - I| (fp32 rotations accumulated)
ROT_RTOL = 3e-5      # |y_gpu - y| <= ROT_RTOL sum_i |x_i r_ij| (three bf16 terms, fp32 sums)


def _accumulation_rtol(N: int, H: int) -> float:
    """Bound of the fp32 tensor-core accumulation of one chunk's sums: the chunk's
    ceil(tiles / chunks) tiles of 128 samples take 8 accumulating MMAs each, and
    every accumulation may be off by one unit in the last place (2^-23) of the
    running sum.  Chunks: one CTA per SM over the 2 H matrices, at most one per tile."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = -(-N // 128)
    chunks = max(1, min(tiles, sms // (2 * H)))
    return 8 * -(-tiles // chunks) * 2.0 ** -23


def _check_side(x_bits, res, centered, q, expect_unique_min=0):
    """Compare one side's GPU outputs with the oracle; returns the number of columns
    whose eigenvector was compared directly."""
    xv = CAL.bf16_bits_to_f64(x_bits)
    N, H, D = xv.shape
    cov_rtol = COV_RTOL + _accumulation_rtol(N, H)
    C = CAL.covariance(x_bits, centered)
    M = CAL.covariance(x_bits, False)
    R_o, lam_o = CAL.rotation(C)
    R = res["R"].double().cpu().numpy()
    lam = res["eigenvalues"].double().cpu().numpy()
    clip = res["clip"].double().cpu().numpy()
    cov = res["cov"].double().cpu().numpy()
    sweeps = res["sweeps"].cpu().numpy()
    k = CAL.quantile_index(q, N)
    unique = 0
    for h in range(H):
        # covariance, element by element
        scale = np.sqrt(np.outer(np.diag(M[h]), np.diag(M[h])))
        dC = np.abs(cov[h] - C[h])
        assert np.all(dC <= cov_rtol * scale + 1e-30), (h, float(np.max(dC / (scale + 1e-30))), cov_rtol)
        dC2 = np.linalg.norm(cov[h] - C[h], 2)
        lmax = max(abs(lam_o[h, 0]), abs(lam_o[h, -1]), 1e-30)
        # eigenvalues (Weyl) and order
        assert np.all(np.abs(lam[h] - lam_o[h]) <= dC2 + RESID_RTOL * lmax), h
        assert np.all(np.diff(lam[h]) <= 0), "eigenvalues not descending"
        assert 1 <= sweeps[h] < 40, sweeps[h]
        # R: orthogonal, an eigenbasis of the oracle's C, sign rule
        assert np.max(np.abs(R[h].T @ R[h] - np.eye(D))) <= ORTHO_TOL
        Rn = R[h] / np.linalg.norm(R[h], axis=0)  # unit columns (the angle bound is for unit vectors)
        E = C[h] @ Rn - Rn * lam[h]
        rho = np.linalg.norm(E, axis=0)
        assert np.all(rho <= RESID_RTOL * lmax + 2 * dC2), (h, float(np.max(rho) / lmax))
        for j in range(D):
            i = int(np.argmax(np.abs(R[h][:, j])))
            assert R[h][i, j] > 0, "sign rule"
        # thresholds: the k-th smallest |x . r_j| of the GPU's own columns
        y = np.abs(xv[:, h, :] @ R[h])
        bound = np.abs(xv[:, h, :]) @ np.abs(R[h])
        kth = np.sort(y, axis=0)[k - 1]
        assert np.all(np.abs(clip[h] - kth) <= ROT_RTOL * bound.max(axis=0) + 1e-30), h
        # columns whose eigenvalue stands apart: compare with the oracle's eigenvector
        xnorm = np.linalg.norm(xv[:, h, :], axis=1).max()
        clip_o = CAL.clip_thresholds(x_bits[:, h:h + 1, :], R_o[h][None], q)[0]
        for j in range(D):
            others = np.delete(lam_o[h], j)
            gap = np.min(np.abs(others - lam[h, j])) if D > 1 else np.inf
            # residual plus the fp64 rounding of its own evaluation
            theta = (rho[j] + 1e-13 * lmax) / gap if gap > 0 else np.inf
            col = np.sort(np.abs(R_o[h][:, j]))
            if theta > 0.05 or col[-1] - col[-2] <= 4 * theta:
                continue
            # the angle to the oracle's eigenvector is at most asin(rho_j / gap_j)
            diff = np.linalg.norm(Rn[:, j] - R_o[h][:, j])
            assert diff <= 2.5 * theta + 1e-7, (h, j, diff, theta)
            assert abs(clip[h, j] - clip_o[j]) <= xnorm * diff + ROT_RTOL * bound[:, j].max() + 1e-30, (h, j)
            unique += 1
    assert unique >= expect_unique_min, unique
    return unique


def _run(kind, N, H, D, centered, q, seed, sides=("k", "v")):
    x = {s: calibration_samples(N, H, D, seed + i, kind, device="cuda") for i, s in enumerate(sides)}
    res = calibrate(x.get("k"), x.get("v"), centered=centered, clip_quantile=q, with_cov=True)
    torch.cuda.synchronize()
    return x, res


@pytest.mark.parametrize("D,H,N,centered,q", [
    (64, 2, 3000, True, 0.99),
    (64, 1, 1000, False, 1.0),
    (128, 2, 4000, True, 0.999),
    (128, 3, 2049, True, 0.5),
    (128, 1, 300, False, 0.9),
])
def test_calibrate_matches_oracle(D, H, N, centered, q):
    x, res = _run("spectrum", N, H, D, centered, q, seed=100 + D + N)
    for s in ("k", "v"):
        _check_side(bits16(x[s]), res[s], centered, q, expect_unique_min=H * D // 4)


@pytest.mark.parametrize("side", ["k", "v"])
def test_calibrate_one_side(side):
    x, res = _run("spectrum", 1500, 2, 128, True, 0.95, seed=7, sides=(side,))
    assert list(res) == [side]
    _check_side(bits16(x[side]), res[side], True, 0.95, expect_unique_min=2 * 128 // 4)


def test_calibrate_workload_distributions():
    # K like the decode workloads (outlier channels: a near-degenerate cluster) and
    # isotropic V: validity and the unique parts only
    N, H, D = 16384, 8, 128
    k = calibration_samples(N, H, D, 4, "qwen", device="cuda")
    v = calibration_samples(N, H, D, 5, "normal", device="cuda")
    for centered in (True, False):
        res = calibrate(k, v, centered=centered, clip_quantile=0.999, with_cov=True)
        torch.cuda.synchronize()
        _check_side(bits16(k), res["k"], centered, 0.999)
        _check_side(bits16(v), res["v"], centered, 0.999)


def test_calibrate_quantile_extremes():
    N, H, D = 777, 1, 64
    x = calibration_samples(N, H, D, 9, "spectrum", device="cuda")
    for q in (1.0, 1.0 / N, 0.5, 0.25 + 1e-12):
        res = calibrate(x, None, centered=True, clip_quantile=q, with_cov=True)
        torch.cuda.synchronize()
        _check_side(bits16(x), res["k"], True, q)


def test_calibrate_degenerate_inputs():
    H, D = 2, 64
    # all samples zero: C = 0, R = I, eigenvalues 0, thresholds 0
    z = torch.zeros(300, H, D, dtype=torch.bfloat16, device="cuda")
    res = calibrate(z, None, centered=True, clip_quantile=0.9, with_cov=True)["k"]
    torch.cuda.synchronize()
    assert torch.equal(res["R"].cpu(), torch.eye(D).expand(H, D, D))
    assert torch.count_nonzero(res["eigenvalues"]).item() == 0
    assert torch.count_nonzero(res["clip"]).item() == 0
    assert torch.count_nonzero(res["cov"]).item() == 0
    # one constant sample repeated: centred covariance 0, second moment rank one
    c = torch.arange(D, dtype=torch.float32, device="cuda").div(8).sub(3).to(torch.bfloat16)
    x = c.view(1, 1, D).expand(500, H, D).contiguous()
    res = calibrate(x, None, centered=True, clip_quantile=1.0, with_cov=True)["k"]
    torch.cuda.synchronize()
    assert torch.count_nonzero(res["cov"]).item() == 0
    assert torch.equal(res["R"].cpu(), torch.eye(D).expand(H, D, D))
    res = calibrate(x, None, centered=False, clip_quantile=1.0, with_cov=True)["k"]
    torch.cuda.synchronize()
    _check_side(bits16(x), res, False, 1.0)
    cf = c.double().cpu().numpy()
    lam = res["eigenvalues"].double().cpu().numpy()
    assert abs(lam[0, 0] - cf @ cf) <= 1e-5 * (cf @ cf)
    r0 = res["R"][0, :, 0].double().cpu().numpy()
    np.testing.assert_allclose(r0, cf / np.linalg.norm(cf), atol=1e-5)  # largest entry positive


def test_calibrate_deterministic():
    x = calibration_samples(5000, 4, 128, 3, "spectrum", device="cuda")
    a = calibrate(x, x, centered=True, clip_quantile=0.99, with_cov=True)
    b = calibrate(x, x, centered=True, clip_quantile=0.99, with_cov=True)
    torch.cuda.synchronize()
    for s in ("k", "v"):
        for name in ("R", "clip", "eigenvalues", "cov", "sweeps"):
            assert torch.equal(a[s][name], b[s][name]), (s, name)
    for name in ("R", "clip", "eigenvalues", "cov"):
        assert torch.equal(a["k"][name], a["v"][name]), name


def test_calibrate_many_samples_d64():
    # more than 2^16 samples per head (ragged), eight heads, keys and values
    N, H, D = 70001, 8, 64
    k = calibration_samples(N, H, D, 21, "spectrum", device="cuda")
    v = calibration_samples(N, H, D, 22, "qwen", device="cuda")
    res = calibrate(k, v, centered=True, clip_quantile=0.9999, with_cov=True)
    torch.cuda.synchronize()
    _check_side(bits16(k), res["k"], True, 0.9999, expect_unique_min=H * D // 4)
    _check_side(bits16(v), res["v"], True, 0.9999)


def test_calibrate_stale_workspace():
    # the workspace is never cleared: a call after one of another size gives the same result
    x = calibration_samples(3000, 2, 128, 31, "spectrum", device="cuda")
    y = calibration_samples(9000, 2, 128, 32, "spectrum", device="cuda")
    import int2_rotated_kv_append_gb300 as ok
    dims = ok.make_dims(2, 2, 128, 16, 128, 1, 1)
    ws = torch.full((ok.oscar_calibrate_workspace_bytes(dims, 9000),), 0x7F, dtype=torch.uint8, device="cuda")
    a = calibrate(x, None, centered=True, clip_quantile=0.99)
    calibrate(y, None, centered=True, clip_quantile=0.99, workspace=ws)
    b = calibrate(x, None, centered=True, clip_quantile=0.99, workspace=ws)
    torch.cuda.synchronize()
    for name in ("R", "clip", "eigenvalues", "sweeps"):
        assert torch.equal(a["k"][name], b["k"][name]), name
