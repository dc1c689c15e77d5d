// OSCAR offline calibration on the GPU: per KV head, the covariance of the
// calibration vectors, its eigenvectors as the rotation R (descending
// eigenvalues, each column signed so that its largest entry is positive) and
// per rotated channel a clipping threshold at a quantile of |x . R|.
//
// Sources: "OSCAR: Cut LLM Inference Costs 8x with 2-bit KV Cache Quantization",
// section "How OSCAR Works" (an offline analysis of the KV covariance designs
// the rotations; fixed clipping thresholds); project card "FutureMLS-Lab/OSCAR",
// section "How it works" (covariance structures of keys and values from a small
// calibration set give per-layer orthogonal rotations and clipping thresholds);
// "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
// Quantization", abstract.
//
// Kernels, in stream order:
//   calib_moments_kernel  sum_t x_t x_t^T and sum_t x_t per chunk of samples on the
//                         tensor cores (the sample tile is the MN-major operand on
//                         both sides; a constant column of ones yields the sums);
//   calib_eig_kernel      chunk partials summed and centred, cyclic Jacobi in shared
//                         memory (several CTAs per matrix, each with its rows of V);
//   calib_finalize_kernel re-orthogonalisation, eigenvalue order, column signs;
//   calib_rotate_kernel   |x . R| for every sample on the tensor cores (R split into
//                         three bf16 terms), stored per channel;
//   calib_select_kernel   one CTA per (matrix, channel): radix selection of the
//                         k-th smallest magnitude.
#include <cuda.h>

#include <cmath>

#include "common.cuh"
#include "ptx.cuh"
#include "umma.cuh"

namespace {

using namespace oscar;

constexpr int kTok = 128;                   // samples per tile
constexpr uint32_t kBlockBytes = kTok * 128;  // 64 channels x 128 samples, bf16

struct CalibIO {
  float* R[2];
  float* clip[2];
  float* eig[2];
  float* cov[2];
  int32_t* sweeps[2];
};

// Entry kv (0: keys, 1: values) of a pair of output pointers, chosen without
// indexing the kernel parameter at run time (which would copy it to local memory).
template <typename T>
__device__ __forceinline__ T* pick(T* const (&a)[2], int kv) {
  return kv ? a[1] : a[0];
}

// ---- second moments --------------------------------------------------------------------
//
// For one (KV head, K|V) and every per-th tile of 128 samples: D[m][n] += sum_t
// X[t][m] X[t][n] with M = 128 rows (channels) and N = D + 16 columns, K = samples.
// A stage holds the D/64 TMA boxes of the tile and one constant block whose
// channel-0 entry is 1 for every sample: as column D of B it makes D[m][D] the sum
// of channel m (and, for D = 64, the same block fills rows 64..127 of A).
constexpr int kMoStages = 4;
constexpr int kMoThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2..5 read TMEM
constexpr int kMoBars = 2 * kMoStages + 1;

template <int D>
__host__ __device__ constexpr size_t mo_stage_bytes() {
  return static_cast<size_t>(D / 64 + 1) * kBlockBytes;
}
template <int D>
constexpr size_t mo_smem() {
  return 1024 + kMoStages * mo_stage_bytes<D>() + kMoBars * 8 + 16;
}

template <int D>
__global__ void __launch_bounds__(kMoThreads, 1) calib_moments_kernel(
    const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v, int64_t num_samples,
    int H, int kv_base, float* __restrict__ part_m, float* __restrict__ part_s) {
  constexpr int XB = D / 64;
  constexpr uint32_t kStage = static_cast<uint32_t>(mo_stage_bytes<D>());
  constexpr int N = D + 16;
  constexpr uint32_t kTmemCols = 256;
  extern __shared__ uint8_t msm_raw[];
  uint8_t* msm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(msm_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t x_s = smem_u32(msm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(msm + kMoStages * kStage);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kMoBars);
  uint32_t* flags = tmem_slot + 1;  // [0] tiles requested, [1] tiles consumed, [2] chains committed
  auto x_full = [&](int st) { return smem_u32(&bars[st]); };
  auto x_empty = [&](int st) { return smem_u32(&bars[kMoStages + st]); };
  const uint32_t acc_full = smem_u32(&bars[2 * kMoStages]);
  const int h = blockIdx.y, kv = kv_base + blockIdx.z, mat = kv * H + h;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t ntiles = (num_samples + kTok - 1) / kTok;
  const int per = gridDim.x, j0 = blockIdx.x;
  const int n_my = static_cast<int>((ntiles - j0 + per - 1) / per);  // tiles j0, j0 + per, ...
  const CUtensorMap* map = kv ? &map_v : &map_k;

  // constant block of every stage: zero, then 1.0 at channel 0 of each sample row
  for (int st = 0; st < kMoStages; ++st) {
    uint4* blk = reinterpret_cast<uint4*>(msm + st * kStage + XB * kBlockBytes);
    for (int i = tid; i < static_cast<int>(kBlockBytes / 16); i += kMoThreads) blk[i] = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  for (int st = 0; st < kMoStages; ++st)
    for (int r = tid; r < kTok; r += kMoThreads) {
      uint16_t* row = reinterpret_cast<uint16_t*>(msm + st * kStage + XB * kBlockBytes + r * 128 + ((r & 7) << 4));
      row[0] = 0x3F80u;  // bf16 1.0
    }
  if (tid == 0) {
    for (int i = 0; i < kMoStages; ++i) {
      mbar_init(x_full(i), 1);
      mbar_init(x_empty(i), 1);
    }
    mbar_init(acc_full, 1);
    flags[0] = flags[1] = flags[2] = 0;
    umma::prefetch_map(map);
    mbar_init_fence();
  }
  if (warp == 1) umma::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // constant blocks visible to the tensor cores
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int i = 0;
      for (; i < n_my; ++i) {
        const int st = i % kMoStages;
        if (i >= kMoStages && !mbar_wait_bounded(x_empty(st), ((i / kMoStages) - 1) & 1)) break;
        const int t0 = static_cast<int>((j0 + static_cast<int64_t>(i) * per) * kTok);
        mbar_arrive_expect_tx(x_full(st), XB * kBlockBytes);
#pragma unroll
        for (int b = 0; b < XB; ++b) umma::tma_load_3d(x_s + st * kStage + b * kBlockBytes, map, 64 * b, h, t0, x_full(st));
        flags[0] = i + 1;
      }
      if (i < n_my) record_error(OSCAR_DEVERR_TIMEOUT);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = umma::idesc_bf16_f32_mn(128, N);
      int i = 0;
      for (; i < n_my; ++i) {
        const int st = i % kMoStages;
        if (!mbar_wait_bounded(x_full(st), (i / kMoStages) & 1)) break;
        flags[1] = i + 1;
        umma::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kTok / 16; ++kk) {
          const uint64_t dsc = umma::desc_mn_sw128(x_s + st * kStage + kk * 2048, kBlockBytes);
          umma::mma_bf16(tmem, dsc, dsc, idesc, (i | kk) != 0);
        }
        umma::commit(x_empty(st));
        flags[2] = i + 1;
      }
      if (i < n_my) record_error(OSCAR_DEVERR_TIMEOUT);
      umma::commit(acc_full);  // after every chain issued so far
    }
  } else {
    // TMEM lanes 32 (warp % 4) .. + 31: row m = channel m of the accumulator
    const int m = 32 * (warp & 3) + lane;
    if (32 * (warp & 3) < D) {
      const bool ok = mbar_wait_bounded(acc_full, 0);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) record_error(OSCAR_DEVERR_TIMEOUT);
      } else if (n_my > 0) {
        umma::fence_after_sync();
        const size_t base = static_cast<size_t>(mat) * per + j0;
        float* pm = part_m + base * D * D;
#pragma unroll 1
        for (int c = 0; c < (N + 31) / 32; ++c) {
          uint32_t vb[32];
          umma::tmem_ld32(tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + 32 * c, vb);
          umma::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int n = 32 * c + i;
            if (n < D) pm[static_cast<size_t>(n) * D + m] = __uint_as_float(vb[i]);  // row n, column m
            if (n == D) part_s[base * D + m] = __uint_as_float(vb[i]);
          }
        }
      } else {
        // no tile: zero partials
        const size_t base = static_cast<size_t>(mat) * per + j0;
        for (int n = 0; n < D; ++n) part_m[(base * D + n) * D + m] = 0.f;
        part_s[base * D + m] = 0.f;
      }
    }
  }

  // ---- teardown: nothing of this CTA may still be in flight ----
  __syncthreads();
  if (tid == 0) {
    for (uint32_t i = flags[1]; i < flags[0]; ++i) mbar_wait_bounded(x_full(i % kMoStages), (i / kMoStages) & 1);
    mbar_wait_bounded(acc_full, 0);
    if (flags[2] > 0) {
      const uint32_t i = flags[2] - 1;
      mbar_wait_bounded(x_empty(i % kMoStages), (i / kMoStages) & 1);
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- eigendecomposition ------------------------------------------------------------------
//
// Cyclic Jacobi in fp32 over (KV head, K|V) matrices.  kSlices CTAs serve one
// matrix: each sums the chunk partials in fp32 in a fixed order, symmetrises and (if
// asked) centres them in fp64, and runs the same sweeps on A (so all of them hold the
// same A, bit for bit), while accumulating only its own D / kSlices rows of
// V = J_1 J_2 ...; the rotations need no exchange between the CTAs.
//   * A is kept as its upper triangle (element (i, j) at min/max), in shared memory;
//   * a sweep is D - 1 rounds of the round-robin pairing (position D - 1 fixed, the
//     others turning), each round rotating D / 2 disjoint pairs at once;
//   * a pair is rotated when |a_pq| > kJacobiTol sqrt(|a_pp a_qq|); the sweeps stop
//     after one without rotations (or at kMaxSweeps);
//   * each 2 x 2 block of A between two pairs is updated once by J1^T A J2; a pair's
//     own block takes the stable form a_pp - t a_pq, a_qq + t a_pq, 0.
// The V rows and the eigenvalues go to the workspace; calib_finalize_kernel
// re-orthogonalises V, orders and signs the columns.
constexpr int kEigThreads = 512;
constexpr int kFinThreads = 512;
constexpr int kSlices = 8;
constexpr float kJacobiTol = 0x1p-21f;
constexpr int kMaxSweeps = 40;

template <int D>
constexpr size_t eig_smem() {
  return static_cast<size_t>(D * (D + 1) + (D / kSlices) * (D + 1)) * 4 + (D / 2) * 16 + (D / 2) * 8 + D * 8 + 16;
}

// Index of element (i, j) of the symmetric matrix in its upper-triangle storage.
template <int LD>
__device__ __forceinline__ int sym_at(int i, int j) {
  return i < j ? i * LD + j : j * LD + i;
}

template <int D>
__global__ void __launch_bounds__(kEigThreads, 1) calib_eig_kernel(const float* __restrict__ part_m,
                                                                    const float* __restrict__ part_s, int per,
                                                                    int64_t num_samples, int centered, int H,
                                                                    int kv_base, CalibIO io, float* __restrict__ v_ws,
                                                                    float* __restrict__ lam_ws) {
  constexpr int NP = D / 2, LD = D + 1, RS = D / kSlices;
  extern __shared__ __align__(16) uint8_t esm_raw[];
  float* A = reinterpret_cast<float*>(esm_raw);         // [D][LD], upper triangle
  float* V = A + D * LD;                                // [RS][LD]: rows s RS .. s RS + RS - 1
  float4* rot = reinterpret_cast<float4*>(V + RS * LD);  // (c, s, t, active) per pair
  int2* pr = reinterpret_cast<int2*>(rot + NP);          // (p, q) per pair
  double* mu = reinterpret_cast<double*>(pr + NP);       // [D]
  int* cnt = reinterpret_cast<int*>(mu + D);             // [2]
  const int h = blockIdx.x, kv = kv_base + blockIdx.y, mat = kv * H + h, slice = blockIdx.z;
  const int tid = threadIdx.x;
  const float* pm = part_m + static_cast<size_t>(mat) * per * D * D;
  const float* ps = part_s + static_cast<size_t>(mat) * per * D;
  const double n = static_cast<double>(num_samples);

  // sums over the chunks (fixed order), then A = M / N - mu mu^T, symmetrised
  if (tid < D) {
    float s = 0.f;
    for (int c = 0; c < per; ++c) s += ps[static_cast<size_t>(c) * D + tid];
    mu[tid] = centered ? static_cast<double>(s) / n : 0.0;
  }
  for (int e = tid; e < D * D; e += kEigThreads) {
    float s = 0.f;
    for (int c = 0; c < per; ++c) s += pm[static_cast<size_t>(c) * D * D + e];
    A[(e / D) * LD + (e % D)] = s;
  }
  for (int e = tid; e < RS * D; e += kEigThreads) {
    const int i = e / D, j = e % D;
    V[i * LD + j] = (slice * RS + i == j) ? 1.f : 0.f;
  }
  __syncthreads();
  float* cov = (pick(io.cov, kv) && slice == 0) ? pick(io.cov, kv) + static_cast<size_t>(h) * D * D : nullptr;
  float cij[(D * D + kEigThreads - 1) / kEigThreads];
#pragma unroll
  for (int u = 0; u < (D * D + kEigThreads - 1) / kEigThreads; ++u) {
    const int e = tid + u * kEigThreads;
    if (e < D * D) {
      const int i = e / D, j = e % D;
      const double m = 0.5 * (static_cast<double>(A[i * LD + j]) + static_cast<double>(A[j * LD + i]));
      const float c = static_cast<float>(m / n - mu[i] * mu[j]);
      cij[u] = c;
      if (cov) cov[e] = c;
    }
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < (D * D + kEigThreads - 1) / kEigThreads; ++u) {
    const int e = tid + u * kEigThreads;
    if (e < D * D) A[(e / D) * LD + (e % D)] = cij[u];
  }

  // cnt[s & 1] counts the rotations of sweep s; cnt[(s + 1) & 1] is cleared during
  // sweep s (after its first barrier, when every thread has read it for sweep s - 1)
  if (tid == 0) cnt[0] = cnt[1] = 0;
  __syncthreads();
  int sweep = 0;
  for (; sweep < kMaxSweeps; ++sweep) {
    for (int r = 0; r < D - 1; ++r) {
      if (tid < NP) {
        int p, q;
        if (tid == 0) {
          p = r;
          q = D - 1;
        } else {
          p = (r + tid) % (D - 1);
          q = (r - tid + (D - 1)) % (D - 1);
        }
        const float app = A[p * LD + p], aqq = A[q * LD + q], apq = A[sym_at<LD>(p, q)];
        float c = 1.f, s = 0.f, t = 0.f, act = 0.f;
        if (apq != 0.f && fabsf(apq) > kJacobiTol * sqrtf(fabsf(app) * fabsf(aqq))) {
          // tan of the rotation angle (the root of t^2 + 2 theta t - 1 of magnitude <= 1)
          const float theta = (aqq - app) / (2.f * apq);
          const float at = fabsf(theta);
          t = at > 1e18f ? 0.5f / theta : copysignf(1.f / (at + sqrtf(theta * theta + 1.f)), theta);
          c = 1.f / sqrtf(t * t + 1.f);
          s = t * c;
          act = 1.f;
          atomicAdd(&cnt[sweep & 1], 1);
        }
        rot[tid] = make_float4(c, s, t, act);
        pr[tid] = make_int2(p, q);
      }
      __syncthreads();
      if (r == 0 && tid == 0) cnt[(sweep + 1) & 1] = 0;
      // blocks (k1, k1 + o mod NP) for o = 0 .. NP/2 - 1, and (k1, k1 + NP/2) for k1 < NP/2:
      // every unordered pair of pairs once
      constexpr int kBlocks = NP * (NP / 2) + NP / 2;
      for (int b = tid; b < kBlocks; b += kEigThreads) {
        int k1, k2;
        if (b < NP * (NP / 2)) {
          k1 = b / (NP / 2);
          k2 = (k1 + b % (NP / 2)) % NP;
        } else {
          k1 = b - NP * (NP / 2);
          k2 = k1 + NP / 2;
        }
        const float4 r1 = rot[k1], r2 = rot[k2];
        if (r1.w == 0.f && r2.w == 0.f) continue;
        const int2 P1 = pr[k1], P2 = pr[k2];
        if (k1 == k2) {
          const int o = sym_at<LD>(P1.x, P1.y);
          const float apq = A[o];
          A[P1.x * LD + P1.x] -= r1.z * apq;
          A[P1.y * LD + P1.y] += r1.z * apq;
          A[o] = 0.f;
          continue;
        }
        const int o11 = sym_at<LD>(P1.x, P2.x), o12 = sym_at<LD>(P1.x, P2.y);
        const int o21 = sym_at<LD>(P1.y, P2.x), o22 = sym_at<LD>(P1.y, P2.y);
        const float a11 = A[o11], a12 = A[o12], a21 = A[o21], a22 = A[o22];
        const float r11 = r1.x * a11 - r1.y * a21, r21 = r1.y * a11 + r1.x * a21;
        const float r12 = r1.x * a12 - r1.y * a22, r22 = r1.y * a12 + r1.x * a22;
        A[o11] = r2.x * r11 - r2.y * r12;
        A[o12] = r2.y * r11 + r2.x * r12;
        A[o21] = r2.x * r21 - r2.y * r22;
        A[o22] = r2.y * r21 + r2.x * r22;
      }
      // V <- V J on this CTA's rows: columns p, q
      for (int e = tid; e < RS * NP; e += kEigThreads) {
        const int k = e / RS, i = e % RS;
        const float4 rr = rot[k];
        if (rr.w == 0.f) continue;
        const int2 P = pr[k];
        const float vp = V[i * LD + P.x], vq = V[i * LD + P.y];
        V[i * LD + P.x] = rr.x * vp - rr.y * vq;
        V[i * LD + P.y] = rr.y * vp + rr.x * vq;
      }
      __syncthreads();
    }
    if (cnt[sweep & 1] == 0) break;
  }

  float* vw = v_ws + static_cast<size_t>(mat) * D * D;
  for (int e = tid; e < RS * D; e += kEigThreads) vw[static_cast<size_t>(slice * RS + e / D) * D + e % D] = V[(e / D) * LD + e % D];
  if (slice == 0) {
    if (tid < D) lam_ws[static_cast<size_t>(mat) * D + tid] = A[tid * LD + tid];
    if (pick(io.sweeps, kv) && tid == 0) pick(io.sweeps, kv)[h] = sweep < kMaxSweeps ? sweep + 1 : kMaxSweeps;
  }
}

// One CTA per matrix: one Newton-Schulz step V <- V (3 I - V^T V) / 2 (the columns
// lose orthogonality by rounding over the sweeps' rotations; the step brings them
// back within fp32 rounding), then the eigenvalues in descending order (ties by
// index) and each column signed so that its entry of largest magnitude (lowest row
// on a tie) is positive.
template <int D>
constexpr size_t fin_smem() {
  return static_cast<size_t>(2 * D * (D + 1)) * 4 + D * 4 * 4;
}

template <int D>
__global__ void __launch_bounds__(kFinThreads, 1) calib_finalize_kernel(const float* __restrict__ v_ws,
                                                                         const float* __restrict__ lam_ws, int H,
                                                                         int kv_base, CalibIO io) {
  constexpr int LD = D + 1;
  extern __shared__ __align__(16) uint8_t fsm_raw[];
  float* V = reinterpret_cast<float*>(fsm_raw);  // [D][LD]
  float* W = V + D * LD;                          // [D][LD]
  float* lam = W + D * LD;                        // [D]
  float* sgn = lam + D;                           // [D]
  int* rank = reinterpret_cast<int*>(sgn + D);    // [D]
  int* inv = rank + D;                            // [D]
  const int h = blockIdx.x, kv = kv_base + blockIdx.y, mat = kv * H + h;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float* vw = v_ws + static_cast<size_t>(mat) * D * D;
  for (int e = tid; e < D * D; e += kFinThreads) V[(e / D) * LD + e % D] = vw[e];
  if (tid < D) {
    lam[tid] = lam_ws[static_cast<size_t>(mat) * D + tid];
    inv[tid] = tid;
  }
  __syncthreads();
  {
    constexpr int TI = D / 32, TJ = D / 16;  // per thread: rows ti + 32 a, columns tj + 16 b
    const int ti = tid >> 4, tj = tid & 15;
    float acc[TI][TJ];
#pragma unroll
    for (int a = 0; a < TI; ++a)
#pragma unroll
      for (int b = 0; b < TJ; ++b) acc[a][b] = 0.f;
    for (int r = 0; r < D; ++r) {  // V^T V
      float va[TI], vb[TJ];
#pragma unroll
      for (int a = 0; a < TI; ++a) va[a] = V[r * LD + ti + 32 * a];
#pragma unroll
      for (int b = 0; b < TJ; ++b) vb[b] = V[r * LD + tj + 16 * b];
#pragma unroll
      for (int a = 0; a < TI; ++a)
#pragma unroll
        for (int b = 0; b < TJ; ++b) acc[a][b] = fmaf(va[a], vb[b], acc[a][b]);
    }
#pragma unroll
    for (int a = 0; a < TI; ++a)
#pragma unroll
      for (int b = 0; b < TJ; ++b) {
        const int i = ti + 32 * a, j = tj + 16 * b;
        W[i * LD + j] = (i == j ? 1.5f : 0.f) - 0.5f * acc[a][b];
      }
    __syncthreads();
#pragma unroll
    for (int a = 0; a < TI; ++a)
#pragma unroll
      for (int b = 0; b < TJ; ++b) acc[a][b] = 0.f;
    for (int r = 0; r < D; ++r) {  // V (3 I - V^T V) / 2, rows ti + 32 a of V
      float va[TI], wb[TJ];
#pragma unroll
      for (int a = 0; a < TI; ++a) va[a] = V[(ti + 32 * a) * LD + r];
#pragma unroll
      for (int b = 0; b < TJ; ++b) wb[b] = W[r * LD + tj + 16 * b];
#pragma unroll
      for (int a = 0; a < TI; ++a)
#pragma unroll
        for (int b = 0; b < TJ; ++b) acc[a][b] = fmaf(va[a], wb[b], acc[a][b]);
    }
    __syncthreads();
#pragma unroll
    for (int a = 0; a < TI; ++a)
#pragma unroll
      for (int b = 0; b < TJ; ++b) V[(ti + 32 * a) * LD + tj + 16 * b] = acc[a][b];
  }
  if (tid < D) {
    const float l = lam[tid];
    int rk = 0;
    for (int i = 0; i < D; ++i) {
      const float li = lam[i];
      rk += (li > l) || (li == l && i < tid);
    }
    rank[tid] = rk;
  }
  __syncthreads();
  for (int j = warp; j < D; j += kFinThreads / 32) {
    float best = -1.f;
    int bi = 0;
    for (int i = lane; i < D; i += 32) {
      const float a = fabsf(V[i * LD + j]);
      if (a > best) {
        best = a;
        bi = i;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ob > best || (ob == best && oi < bi)) {
        best = ob;
        bi = oi;
      }
    }
    if (lane == 0) sgn[j] = V[bi * LD + j] < 0.f ? -1.f : 1.f;
  }
  if (tid < D) inv[rank[tid]] = tid;
  __syncthreads();
  float* R = pick(io.R, kv) + static_cast<size_t>(h) * D * D;
  for (int e = tid; e < D * D; e += kFinThreads) {
    const int i = e / D, col = e % D, j = inv[col];
    R[e] = sgn[j] * V[i * LD + j];
  }
  if (pick(io.eig, kv) && tid < D) pick(io.eig, kv)[static_cast<size_t>(h) * D + rank[tid]] = lam[tid];
}

// ---- |x . R| per sample and channel --------------------------------------------------------
//
// The prefill append's tensor-core rotation without its quantiser: R (fp32) split into
// three bf16 terms stored once as R^T (K-major, swizzled), x tiles by TMA into a
// 3-stage ring, one UMMA chain of M = 128 samples, N = D, K = 3 D per tile, groups of
// four epilogue warps taking tiles in turn; a thread owns one sample and stores the
// bits of |y_j| at Y[mat][j][t] (a warp's 32 samples are 128 contiguous bytes).
constexpr int kRoStages = 3;
constexpr int kRoGroups = 4;
constexpr int kRoThreads = 64 + 128 * kRoGroups;
constexpr int kRoBars = 2 * kRoStages + 2 * kRoGroups;

template <int D>
constexpr size_t ro_smem() {
  return 1024 + 3 * static_cast<size_t>(D) * D * 2 + kRoStages * static_cast<size_t>(D / 64) * kBlockBytes +
         kRoBars * 8 + 16;
}

__device__ __forceinline__ uint32_t bf16_pair(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) | (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

template <int D>
__global__ void __launch_bounds__(kRoThreads, 1) calib_rotate_kernel(
    const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v, int64_t num_samples,
    int64_t n_pad, int H, int kv_base, CalibIO io, uint32_t* __restrict__ Y) {
  constexpr int XB = D / 64;
  constexpr uint32_t kXBytes = XB * kBlockBytes;
  constexpr uint32_t kRPart = D * D * 2;
  constexpr uint32_t kTmemCols = D * kRoGroups;
  static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM allocation must be a power of two");
  extern __shared__ uint8_t rsm_raw[];
  uint8_t* rsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rsm_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t r_s = smem_u32(rsm);
  const uint32_t x_s = r_s + 3 * kRPart;
  uint64_t* bars = reinterpret_cast<uint64_t*>(rsm + 3 * kRPart + kRoStages * kXBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kRoBars);
  uint32_t* flags = tmem_slot + 1;
  auto x_full = [&](int st) { return smem_u32(&bars[st]); };
  auto x_empty = [&](int st) { return smem_u32(&bars[kRoStages + st]); };
  auto acc_full = [&](int g) { return smem_u32(&bars[2 * kRoStages + g]); };
  auto acc_empty = [&](int g) { return smem_u32(&bars[2 * kRoStages + kRoGroups + g]); };
  const int h = blockIdx.y, kv = kv_base + blockIdx.z, mat = kv * H + h;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t ntiles = (num_samples + kTok - 1) / kTok;
  const int per = gridDim.x, j0 = blockIdx.x;
  const int n_my = static_cast<int>((ntiles - j0 + per - 1) / per);
  const float* R = pick(io.R, kv) + static_cast<size_t>(h) * D * D;
  const CUtensorMap* map = kv ? &map_v : &map_k;

  if (tid == 0) {
    for (int i = 0; i < kRoStages; ++i) {
      mbar_init(x_full(i), 1);
      mbar_init(x_empty(i), 1);
    }
    for (int g = 0; g < kRoGroups; ++g) {
      mbar_init(acc_full(g), 1);
      mbar_init(acc_empty(g), 4);
    }
    flags[0] = flags[1] = flags[2] = 0;
    umma::prefetch_map(map);
    mbar_init_fence();
  }
  if (warp == 1) umma::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  // R^T terms: item (k pair kp, output n) takes R[2kp][n] and R[2kp + 1][n]
  for (int it = tid; it < (D / 2) * D; it += kRoThreads) {
    const int kp = it % (D / 2), n = it / (D / 2);
    const float e0 = __ldg(R + static_cast<size_t>(2 * kp) * D + n), e1 = __ldg(R + static_cast<size_t>(2 * kp + 1) * D + n);
    const __nv_bfloat16 h0 = __float2bfloat16_rn(e0), h1 = __float2bfloat16_rn(e1);
    const float d0 = e0 - __bfloat162float(h0), d1 = e1 - __bfloat162float(h1);
    const __nv_bfloat16 m0 = __float2bfloat16_rn(d0), m1 = __float2bfloat16_rn(d1);
    const __nv_bfloat16 l0 = __float2bfloat16_rn(d0 - __bfloat162float(m0));
    const __nv_bfloat16 l1 = __float2bfloat16_rn(d1 - __bfloat162float(m1));
    const uint32_t off = r_s + umma::sw128_offset(n, 2 * kp, D);
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(off), "r"(bf16_pair(h0, h1)) : "memory");
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(off + kRPart), "r"(bf16_pair(m0, m1)) : "memory");
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(off + 2 * kRPart), "r"(bf16_pair(l0, l1)) : "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int i = 0;
      for (; i < n_my; ++i) {
        const int st = i % kRoStages;
        if (i >= kRoStages && !mbar_wait_bounded(x_empty(st), ((i / kRoStages) - 1) & 1)) break;
        const int t0 = static_cast<int>((j0 + static_cast<int64_t>(i) * per) * kTok);
        mbar_arrive_expect_tx(x_full(st), kXBytes);
#pragma unroll
        for (int b = 0; b < XB; ++b) umma::tma_load_3d(x_s + st * kXBytes + b * kBlockBytes, map, 64 * b, h, t0, x_full(st));
        flags[0] = i + 1;
      }
      if (i < n_my) record_error(OSCAR_DEVERR_TIMEOUT);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = umma::idesc_bf16_f32(128, D);
      int i = 0;
      for (; i < n_my; ++i) {
        const int st = i % kRoStages, b = i % kRoGroups;
        if (!mbar_wait_bounded(x_full(st), (i / kRoStages) & 1)) break;
        flags[1] = i + 1;
        if (i >= kRoGroups && !mbar_wait_bounded(acc_empty(b), ((i / kRoGroups) - 1) & 1)) break;
        umma::fence_after_sync();
        const uint32_t d = tmem + b * D;
#pragma unroll 1
        for (int part = 0; part < 3; ++part)
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t koff_x = (ks >> 2) * kBlockBytes + (ks & 3) * 32;
            const uint32_t koff_r = (ks >> 2) * (D * 128) + (ks & 3) * 32;
            umma::mma_bf16(d, umma::desc_k_sw128(x_s + st * kXBytes + koff_x),
                           umma::desc_k_sw128(r_s + part * kRPart + koff_r), idesc, (part | ks) != 0);
          }
        umma::commit(x_empty(st));
        umma::commit(acc_full(b));
        flags[2] = i + 1;
      }
      if (i < n_my) record_error(OSCAR_DEVERR_TIMEOUT);
    }
  } else {
    const int e = (warp - 2) >> 2, q = warp & 3;
    const int row = 32 * q + lane;
    uint32_t* Ym = Y + static_cast<size_t>(mat) * D * n_pad;
    for (int i = e; i < n_my; i += kRoGroups) {
      const int64_t t = (j0 + static_cast<int64_t>(i) * per) * kTok + row;
      const bool ok = mbar_wait_bounded(acc_full(e), (i / kRoGroups) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) record_error(OSCAR_DEVERR_TIMEOUT);
        break;
      }
      umma::fence_after_sync();
      const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) + e * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t vb[32];
        umma::tmem_ld32(ta + 32 * c, vb);
        umma::tmem_ld_wait();
        if (t < num_samples) {
#pragma unroll
          for (int j = 0; j < 32; ++j) Ym[static_cast<size_t>(32 * c + j) * n_pad + t] = vb[j] & 0x7FFFFFFFu;
        }
      }
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(e));
    }
  }

  __syncthreads();
  if (tid == 0) {
    for (uint32_t i = flags[1]; i < flags[0]; ++i) mbar_wait_bounded(x_full(i % kRoStages), (i / kRoStages) & 1);
    if (flags[2] > 0) {
      const uint32_t i = flags[2] - 1;
      mbar_wait_bounded(acc_full(i % kRoGroups), (i / kRoGroups) & 1);
      mbar_wait_bounded(x_empty(i % kRoStages), (i / kRoStages) & 1);
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- k-th smallest magnitude per channel ------------------------------------------------------
//
// Magnitudes are non-negative fp32 bit patterns, whose unsigned order is their
// numeric order.  Three histogram passes over the column fix bits 31..21, 20..10 and
// 9..0 of the k-th smallest value: each pass counts the values that share the bits
// fixed so far, the bin where the running count reaches the rank is the next digit,
// and the rank drops by the count below that bin.
constexpr int kSelThreads = 256;
constexpr int kSelBins = 2048;

__global__ void __launch_bounds__(kSelThreads) calib_select_kernel(const uint32_t* __restrict__ Y, int64_t num_samples,
                                                                   int64_t n_pad, int64_t k, int D, int H, int kv_base,
                                                                   CalibIO io) {
  __shared__ uint32_t hist[kSelBins];
  __shared__ uint32_t warp_tot[kSelThreads / 32];
  __shared__ uint32_t sel[2];
  const int j = blockIdx.x, h = blockIdx.y, kv = kv_base + blockIdx.z, mat = kv * H + h;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint4* col = reinterpret_cast<const uint4*>(Y + (static_cast<size_t>(mat) * D + j) * n_pad);
  const int64_t n4 = n_pad / 4;
  uint32_t prefix = 0;
  uint32_t rank = static_cast<uint32_t>(k);  // 1-based within the values sharing the prefix
  const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int sh = shifts[pass], nb = 1 << widths[pass];
    const int hi = sh + widths[pass];  // bits >= hi must equal the prefix
    for (int b = tid; b < nb; b += kSelThreads) hist[b] = 0;
    __syncthreads();
    for (int64_t i = tid; i < n4; i += kSelThreads) {
      const uint4 w = __ldg(col + i);
      const uint32_t vals[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (4 * i + u >= num_samples) break;
        const uint32_t x = vals[u];
        if (hi >= 32 || (x >> hi) == prefix) atomicAdd(&hist[(x >> sh) & (nb - 1)], 1u);
      }
    }
    __syncthreads();
    // the bin where the inclusive running count first reaches rank
    const int per_t = nb / kSelThreads;  // 8 or 4 bins per thread
    uint32_t local = 0;
    for (int b = 0; b < per_t; ++b) local += hist[tid * per_t + b];
    uint32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    uint32_t before = incl - local;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    if (before < rank && rank <= before + local) {
      uint32_t run = before;
      for (int b = 0; b < per_t; ++b) {
        const uint32_t cb = hist[tid * per_t + b];
        if (run + cb >= rank) {
          sel[0] = static_cast<uint32_t>(tid * per_t + b);
          sel[1] = run;
          break;
        }
        run += cb;
      }
    }
    __syncthreads();
    prefix = (prefix << widths[pass]) | sel[0];
    rank -= sel[1];
    __syncthreads();
  }
  if (tid == 0) pick(io.clip, kv)[static_cast<size_t>(h) * D + j] = __uint_as_float(prefix);
}

// ---- host ---------------------------------------------------------------------------------------

bool sample_map(CUtensorMap* m, const void* x, int64_t N, int H, int D) {
  umma::EncodeTiledFn fn = umma::encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(N)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
  const cuuint32_t box[3] = {64, 1, kTok};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Chunks of samples per matrix for the moments (the partials' count): one CTA per
// SM over all 2 H matrices, at most one chunk per tile.
int64_t moment_chunks(int H, int64_t N) {
  const int64_t ntiles = (N + kTok - 1) / kTok;
  int64_t per = num_sms() / (2 * H);
  if (per < 1) per = 1;
  if (per > ntiles) per = ntiles;
  return per;
}

struct WsLayout {
  size_t part_m, part_s, y, v, lam, total;
  int64_t per, n_pad;
};

WsLayout ws_layout(int H, int D, int64_t N) {
  WsLayout w{};
  w.per = moment_chunks(H, N);
  w.n_pad = (N + 3) / 4 * 4;
  const size_t mats = 2 * static_cast<size_t>(H);
  w.part_m = 0;
  w.part_s = align_up(w.part_m + mats * w.per * D * D * 4, 256);
  w.y = align_up(w.part_s + mats * w.per * D * 4, 256);
  w.v = align_up(w.y + mats * D * static_cast<size_t>(w.n_pad) * 4, 256);
  w.lam = align_up(w.v + mats * D * D * 4, 256);
  w.total = align_up(w.lam + mats * D * 4, 256);
  return w;
}

template <int D>
cudaError_t run_calibration(int H, int64_t N, const void* k, const void* v, int centered, int64_t rank,
                            const CalibIO& io, uint8_t* ws, const WsLayout& w, cudaStream_t stream) {
  CUtensorMap mk, mv;
  const void* first = k ? k : v;
  if (!sample_map(&mk, k ? k : first, N, H, D) || !sample_map(&mv, v ? v : first, N, H, D)) return cudaErrorInvalidValue;
  const int kv_base = k ? 0 : 1;
  const int nkv = (k && v) ? 2 : 1;
  float* part_m = reinterpret_cast<float*>(ws + w.part_m);
  float* part_s = reinterpret_cast<float*>(ws + w.part_s);
  uint32_t* Y = reinterpret_cast<uint32_t*>(ws + w.y);

  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(calib_moments_kernel<D>), mo_smem<D>());
  if (e != cudaSuccess) return e;
  calib_moments_kernel<D><<<dim3(static_cast<unsigned>(w.per), H, nkv), kMoThreads, mo_smem<D>(), stream>>>(
      mk, mv, N, H, kv_base, part_m, part_s);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  float* v_ws = reinterpret_cast<float*>(ws + w.v);
  float* lam_ws = reinterpret_cast<float*>(ws + w.lam);
  e = set_smem_limit_once(reinterpret_cast<const void*>(calib_eig_kernel<D>), eig_smem<D>());
  if (e != cudaSuccess) return e;
  calib_eig_kernel<D><<<dim3(H, nkv, kSlices), kEigThreads, eig_smem<D>(), stream>>>(
      part_m, part_s, static_cast<int>(w.per), N, centered, H, kv_base, io, v_ws, lam_ws);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  e = set_smem_limit_once(reinterpret_cast<const void*>(calib_finalize_kernel<D>), fin_smem<D>());
  if (e != cudaSuccess) return e;
  calib_finalize_kernel<D><<<dim3(H, nkv), kFinThreads, fin_smem<D>(), stream>>>(v_ws, lam_ws, H, kv_base, io);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  const int64_t ntiles = (N + kTok - 1) / kTok;
  int64_t per_r = num_sms() / (nkv * H);
  if (per_r < 1) per_r = 1;
  if (per_r > ntiles) per_r = ntiles;
  e = set_smem_limit_once(reinterpret_cast<const void*>(calib_rotate_kernel<D>), ro_smem<D>());
  if (e != cudaSuccess) return e;
  calib_rotate_kernel<D><<<dim3(static_cast<unsigned>(per_r), H, nkv), kRoThreads, ro_smem<D>(), stream>>>(
      mk, mv, N, w.n_pad, H, kv_base, io, Y);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  calib_select_kernel<<<dim3(D, H, nkv), kSelThreads, 0, stream>>>(Y, N, w.n_pad, rank, D, H, kv_base, io);
  return cudaGetLastError();
}

bool bad_out(const oscar_calib_out_t* o) {
  return o->R == nullptr || o->clip == nullptr || misaligned16(o->R);
}

}  // namespace

extern "C" size_t oscar_calibrate_workspace_bytes(const oscar_dims_t* dims, int64_t num_samples) {
  if (check_dims(dims) != OSCAR_OK || num_samples <= 0) return 0;
  return ws_layout(dims->num_kv_heads, dims->head_dim, num_samples).total;
}

extern "C" oscar_status_t oscar_calibrate(const oscar_dims_t* dims, int64_t num_samples, const void* k, const void* v,
                                          int32_t centered, double clip_quantile, const oscar_calib_out_t* out_k,
                                          const oscar_calib_out_t* out_v, void* workspace, size_t workspace_bytes,
                                          void* stream) {
  const oscar_status_t st = check_dims(dims);
  if (st != OSCAR_OK) return st;
  if (num_samples <= 0 || num_samples > (static_cast<int64_t>(1) << 31) - 2 * kTok) return OSCAR_ERR_INVALID_ARG;
  if ((k == nullptr) != (out_k == nullptr) || (v == nullptr) != (out_v == nullptr)) return OSCAR_ERR_INVALID_ARG;
  if (k == nullptr && v == nullptr) return OSCAR_ERR_INVALID_ARG;
  if ((out_k && bad_out(out_k)) || (out_v && bad_out(out_v))) return OSCAR_ERR_INVALID_ARG;
  if ((k && misaligned16(k)) || (v && misaligned16(v))) return OSCAR_ERR_INVALID_ARG;
  if (centered != 0 && centered != 1) return OSCAR_ERR_INVALID_ARG;
  if (!(clip_quantile > 0.0 && clip_quantile <= 1.0)) return OSCAR_ERR_INVALID_ARG;
  if (workspace == nullptr || misaligned16(workspace)) return OSCAR_ERR_INVALID_ARG;
  const int H = dims->num_kv_heads, D = dims->head_dim;
  const WsLayout w = ws_layout(H, D, num_samples);
  if (workspace_bytes < w.total) return OSCAR_ERR_WORKSPACE;
  if (umma::encode_tiled() == nullptr) return OSCAR_ERR_CUDA;
  // rank of the threshold: ceil(q N) in double precision, within [1, N]
  int64_t rank = static_cast<int64_t>(std::ceil(clip_quantile * static_cast<double>(num_samples)));
  if (rank < 1) rank = 1;
  if (rank > num_samples) rank = num_samples;
  CalibIO io{};
  const oscar_calib_out_t* outs[2] = {out_k, out_v};
  for (int i = 0; i < 2; ++i)
    if (outs[i]) {
      io.R[i] = outs[i]->R;
      io.clip[i] = outs[i]->clip;
      io.eig[i] = outs[i]->eigenvalues;
      io.cov[i] = outs[i]->cov;
      io.sweeps[i] = outs[i]->sweeps;
    }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const cudaError_t e = D == 128 ? run_calibration<128>(H, num_samples, k, v, centered, rank, io, ws, w, as_stream(stream))
                                 : run_calibration<64>(H, num_samples, k, v, centered, rank, io, ws, w, as_stream(stream));
  return e == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

oscar_status_t oscar_internal_calib_errors(uint32_t* flags, int reset) {
  return read_unit_errors(flags, reset) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}
