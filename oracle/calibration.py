"""OSCAR offline calibration, CPU oracle -- TEST INFRASTRUCTURE ONLY.

Plain fp64 numpy restatement of the offline step that produces the fixed
rotation R and the clipping thresholds the append consumes.  Only the
test-suite, the smoke check and the benchmark's CPU-baseline leg may import
it; it shares no code with the CUDA library.

Sources, cited by title and section:
  [Summary]   "OSCAR: Cut LLM Inference Costs 8x with 2-bit KV Cache
              Quantization", section "How OSCAR Works": an offline analysis of
              the covariance structure of the KV cache designs the rotations;
              fixed clipping thresholds follow.
  [Card]      project card "FutureMLS-Lab/OSCAR", section "How it works":
              activations captured on a small calibration set give covariance
              structures of keys and values, from which per-layer orthogonal
              rotations and clipping thresholds are derived.
  [Abstract]  "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV
              Cache Quantization", abstract: covariance estimated offline,
              fixed rotations and clipping thresholds derived from it.

The pages name the ingredients (covariance, spectral rotation, clipping
thresholds) but print no formula, so every step below is the plainest
reading of those words:
  (C1) the covariance of one KV head is the sample covariance of its N
       calibration vectors, C = (1/N) sum_t (x_t - mu)(x_t - mu)^T with
       mu = (1/N) sum_t x_t; with ``centered`` false it is the second moment
       (1/N) sum_t x_t x_t^T.  The "attention-aware" weighting is not defined
       on the pages and is not modelled.
  (C2) "spectral rotation": R's columns are orthonormal eigenvectors of C in
       descending eigenvalue order, so x.R has the principal components of x
       as its channels.  An eigenvector is fixed up to sign: each column is
       signed so that its entry of largest magnitude (the lowest row index on
       a tie) is positive.  Equal eigenvalues leave the basis of their
       eigenspace open.
  (C3) clipping threshold of channel j: the k-th smallest of |x_t . R[:, j]|
       over the N samples, k = ceil(q N) evaluated in double precision and
       kept within [1, N], for a quantile level q in (0, 1] (q = 1 gives the
       largest magnitude seen).
Inputs are bf16 bit patterns [N][H][D] (the layout the append takes);
everything is computed in fp64.

Parity status: each function is pinned by tests against closed forms, exact
rational brute force, planted spectra and order-statistic brute force; the
pages print no calibration example, so end-to-end values on real activations
are parity unpinned.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = ["bf16_bits_to_f64", "covariance", "rotation", "quantile_index", "clip_thresholds", "calibrate"]


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values (a bf16 is the top half of an fp32)."""
    b = np.ascontiguousarray(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def covariance(x_bits: np.ndarray, centered: bool = True) -> np.ndarray:
    """(C1): per-head covariance (or second moment) [H][D][D] of samples [N][H][D]."""
    x = bf16_bits_to_f64(x_bits)
    N, H, D = x.shape
    C = np.zeros((H, D, D))
    for h in range(H):
        xh = x[:, h, :]
        if centered:
            mu = xh.sum(axis=0) / N
            xh = xh - mu
        C[h] = (xh.T @ xh) / N
    return C


def rotation(C: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(C2): per head, R (columns = eigenvectors, descending eigenvalues, sign rule)
    and the eigenvalues in the same order.  C: [H][D][D] symmetric."""
    H, D, _ = C.shape
    R = np.zeros((H, D, D))
    lam = np.zeros((H, D))
    for h in range(H):
        w, V = np.linalg.eigh(C[h])     # ascending eigenvalues, orthonormal columns
        order = np.argsort(-w, kind="stable")
        w, V = w[order], V[:, order]
        for j in range(D):
            col = V[:, j]
            i_big = int(np.argmax(np.abs(col)))  # first index of the largest magnitude
            if col[i_big] < 0:
                V[:, j] = -col
        R[h] = V
        lam[h] = w
    return R, lam


def quantile_index(q: float, N: int) -> int:
    """(C3): 1-based rank of the threshold among N sorted magnitudes."""
    k = int(math.ceil(float(q) * float(N)))
    return min(max(k, 1), N)


def clip_thresholds(x_bits: np.ndarray, R: np.ndarray, q: float) -> np.ndarray:
    """(C3): per head and rotated channel, the k-th smallest |x . R[:, j]|.  R: [H][D][D]."""
    x = bf16_bits_to_f64(x_bits)
    N, H, D = x.shape
    k = quantile_index(q, N)
    clip = np.zeros((H, D))
    for h in range(H):
        y = np.abs(x[:, h, :] @ np.asarray(R[h], dtype=np.float64))  # [N][D]
        clip[h] = np.sort(y, axis=0)[k - 1]
    return clip


def calibrate(x_bits: np.ndarray, centered: bool = True, q: float = 1.0):
    """(C1)-(C3) in order: returns (C, R, eigenvalues, clip)."""
    C = covariance(x_bits, centered)
    R, lam = rotation(C)
    clip = clip_thresholds(x_bits, R, q)
    return C, R, lam, clip
