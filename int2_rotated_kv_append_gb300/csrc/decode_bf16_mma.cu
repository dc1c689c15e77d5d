// Tensor-core split kernel of the all-BF16 paged decode, the speedup reference
// the OSCAR pages compare against ("OSCAR: Offline Spectral Covariance-Aware
// Rotation for 2-bit KV Cache Quantization", summary "Practical Summary":
// faster decoding than BF16).
//
// Shape covered: head_dim 128, GQA 1..8.  One CTA of 4 warps owns one split of
// one (sequence, KV head); each warp takes every 4th page of the split.
// Per warp and page (16 tokens, K and V rows of 256 bytes):
//   * the 32 rows arrive by 32 bulk async copies (one per lane) into a padded
//     shared-memory stage (272-byte rows, so ldmatrix is bank-conflict free),
//     a ring of kStages pages per warp guarded by mbarriers with bounded waits;
//   * QK:  S^T[token][query] = K[token][ch] . Q[ch][query], A from ldmatrix,
//     B = q * scale * log2(e) split into bf16 hi + lo (16 significant bits);
//   * online softmax per query with warp shuffles;
//   * PV:  O^T[ch][query] += V^T[ch][token] . P[token][query], A from
//     ldmatrix.trans, B = p split into bf16 hi + lo;
// then a log-sum-exp merge of the warps through shared memory.
#include <mutex>

#include "decode_common.cuh"

namespace oscar_dec {
namespace {

constexpr int kD = 128;
constexpr int kWarps = 4;
constexpr int kStages = 2;  // 2 pages per warp: three 4-warp CTAs fit in shared memory
constexpr int kRowBytes = kD * 2;            // one token row of K or V
constexpr int kRowPitch = kRowBytes + 16;    // padded row in shared memory
constexpr int kStageBytes = 32 * kRowPitch;  // 16 K rows then 16 V rows
constexpr int kMaxPps = 256;
constexpr size_t kSmem = static_cast<size_t>(kWarps) * kStages * kStageBytes + kWarps * kStages * 8 + kMaxPps * 4;

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) | (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

// bf16 hi + lo of x (lo = bf16(x - hi)).
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

template <int NT>
__global__ void __launch_bounds__(kWarps * 32) bf16_mma_split_kernel(Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int gqa = p.gqa;
  const int L = clamp_len(p, b);
  const int r0 = s * p.pps * kPageSize, r1 = min(r0 + p.pps * kPageSize, L);
  const size_t bh0 = static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * gqa;
  grid_dep_launch_dependents();
  if (r1 <= r0) {
    for (int i = tid; i < gqa * kD; i += kWarps * 32)
      p.part_o[((bh0 + i / kD) * p.ns + s) * kD + i % kD] = 0.f;
    if (tid < gqa) {
      p.part_ml[((bh0 + tid) * p.ns + s) * 2 + 0] = -INFINITY;
      p.part_ml[((bh0 + tid) * p.ns + s) * 2 + 1] = 0.f;
    }
    return;
  }
  const int pg0 = r0 / kPageSize;
  const int npg = (r1 - 1) / kPageSize + 1 - pg0;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * kStages * kStageBytes);
  int* pid_s = reinterpret_cast<int*>(bars + kWarps * kStages);
  for (int i = tid; i < npg; i += kWarps * 32) {
    int pid = __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pg0 + i);
    if (pid < 0 || pid >= p.num_pages) {
      record_error(OSCAR_DEVERR_PAGE_ID);
      pid = -1;
    }
    pid_s[i] = pid;
  }
  if (lane == 0)
    for (int i = 0; i < kStages; ++i) mbar_init(smem_u32(&bars[warp * kStages + i]), 1);
  mbar_init_fence();
  __syncthreads();

  const int n_my = npg > warp ? (npg - warp + kWarps - 1) / kWarps : 0;
  uint8_t* my_stages = smem + warp * kStages * kStageBytes;
  uint64_t* my_bars = bars + warp * kStages;
  auto issue = [&](int i) {  // whole warp: lane r copies row r of the (page, head): K rows 0..15, V rows 16..31
    const int pid = pid_s[warp + i * kWarps];
    const uint32_t bar = smem_u32(&my_bars[i % kStages]);
    if (pid < 0) {
      if (lane == 0) mbar_arrive(bar);
      return;
    }
    if (lane == 0) mbar_arrive_expect_tx(bar, 32 * kRowBytes);
    __syncwarp();
    uint8_t* st = my_stages + (i % kStages) * kStageBytes;
    const size_t row0 = (static_cast<size_t>(pid) * p.H + h) * 2 * kPageSize;  // K row 0 of (page, head)
    // K token r -> stage row r; V token v -> stage row 16 + 2*(v % 8) + v / 8, so each
    // transposed ldmatrix below reads 8 consecutive rows (distinct bank groups).
    const int v = lane - 16;
    const int srow = lane < 16 ? lane : 16 + 2 * (v & 7) + (v >> 3);
    bulk_g2s(smem_u32(st + srow * kRowPitch), p.pages + (row0 + lane) * kD, kRowBytes, bar);
  };
  for (int i = 0; i < n_my && i < kStages; ++i) issue(i);

  // q * scale * log2(e) as bf16 hi/lo B fragments: k-step ks, rows 2t, 2t+1 -> channels
  // 16 ks + 2t, +1; rows 2t+8, 2t+9 -> 16 ks + 2t + 8, +9; column g -> query g/2, part g%2.
  const __nv_bfloat16* qb = p.q + bh0 * kD;
  uint32_t bq[NT][8][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int qi = 4 * nt + (g >> 1);
    const bool use = qi < gqa;
    const bool lo_part = (g & 1) != 0;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      __nv_bfloat16 v[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int ch = 16 * ks + 2 * t + (c & 1) + 8 * (c >> 1);
        const float x = use ? __bfloat162float(qb[qi * kD + ch]) * p.scale_log2 : 0.f;
        __nv_bfloat16 hi, lo;
        split_bf16(x, hi, lo);
        v[c] = lo_part ? lo : hi;
      }
      bq[nt][ks][0] = pack_bf16x2(v[0], v[1]);
      bq[nt][ks][1] = pack_bf16x2(v[2], v[3]);
    }
  }

  float m_run[NT], l_run[NT], O[NT][8][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt] = -INFINITY;
    l_run[nt] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) O[nt][i][c] = 0.f;
  }
  // ldmatrix row addresses.  K (non-transposed): matrix lm = lane/8 covers tokens
  // 8*(lm&1) .. +7 and channels 8*(lm>>1) .. +7 of a k-step.  V (transposed): the
  // k index of PV is a token order chosen so that the two tokens of a B register
  // (k = 2t', 2t'+1) are tokens t', t'+8 and (k = 2t'+8, 2t'+9) are t'+4, t'+12,
  // which is how the softmax fragments already pair them; with the V row
  // placement of `issue`, row lr of matrix lm is stage row 16 + lr + 8*(lm>>1).
  const int lr = lane & 7, lm = lane >> 3;
  const int k_row = lr + 8 * (lm & 1);
  const int k_col = 8 * (lm >> 1);
  const int v_row = lr + 8 * (lm >> 1);
  const int v_col = 8 * (lm & 1);
  const int src1 = 4 * t + (g >> 1), src2 = src1 + 16;
  bool aborted = false;
  int i = 0;
  for (; i < n_my; ++i) {
    const uint32_t bar = smem_u32(&my_bars[i % kStages]);
    const bool ok = mbar_wait_bounded(bar, (i / kStages) & 1);
    if (__any_sync(0xffffffffu, !ok)) {
      aborted = true;
      break;
    }
    const uint8_t* st = my_stages + (i % kStages) * kStageBytes;
    const int jpage = warp + i * kWarps;
    const bool page_ok = pid_s[jpage] >= 0;
    const int pos0 = (pg0 + jpage) * kPageSize + g;
    const bool v0 = page_ok && pos0 >= r0 && pos0 < r1;
    const bool v1 = page_ok && pos0 + 8 >= r0 && pos0 + 8 < r1;
    const uint32_t kbase = smem_u32(st) + k_row * kRowPitch + k_col * 2;
    const uint32_t vbase = smem_u32(st) + (16 + v_row) * kRowPitch + v_col * 2;

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[nt][c] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4(kbase + ks * 32, a0, a1, a2, a3);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16(acc[nt], a0, a1, a2, a3, bq[nt][ks][0], bq[nt][ks][1]);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float sc0 = v0 ? acc[nt][0] + acc[nt][1] : -INFINITY;
      const float sc1 = v1 ? acc[nt][2] + acc[nt][3] : -INFINITY;
      float mx = fmaxf(sc0, sc1);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(m_run[nt], mx);
      if (__any_sync(0xffffffffu, m_new > m_run[nt])) {
        const float alpha = m_run[nt] == -INFINITY ? 0.f : fast_exp2(m_run[nt] - m_new);
        l_run[nt] *= alpha;
#pragma unroll
        for (int mi = 0; mi < 8; ++mi)
#pragma unroll
          for (int c = 0; c < 4; ++c) O[nt][mi][c] *= alpha;
        m_run[nt] = m_new;
      }
      const float p0 = v0 ? fast_exp2(sc0 - m_new) : 0.f;
      const float p1 = v1 ? fast_exp2(sc1 - m_new) : 0.f;
      l_run[nt] += p0 + p1;
      __nv_bfloat16 h0, e0, h1, e1;
      split_bf16(p0, h0, e0);
      split_bf16(p1, h1, e1);
      const uint32_t xhi = pack_bf16x2(h0, h1), xlo = pack_bf16x2(e0, e1);
      const uint32_t h_1 = __shfl_sync(0xffffffffu, xhi, src1), l_1 = __shfl_sync(0xffffffffu, xlo, src1);
      const uint32_t h_2 = __shfl_sync(0xffffffffu, xhi, src2), l_2 = __shfl_sync(0xffffffffu, xlo, src2);
      const uint32_t bp0 = (g & 1) ? l_1 : h_1, bp1 = (g & 1) ? l_2 : h_2;
#pragma unroll
      for (int mi = 0; mi < 8; ++mi) {
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4_trans(vbase + mi * 32, a0, a1, a2, a3);
        mma_bf16(O[nt][mi], a0, a1, a2, a3, bp0, bp1);
      }
    }
    __syncwarp();
    if (i + kStages < n_my) issue(i + kStages);
  }
  if (aborted) {
    if (lane == 0) record_error(OSCAR_DEVERR_TIMEOUT);
    const int issued = min(n_my, i + kStages);
    for (int k = i; k < issued; ++k) mbar_wait_bounded(smem_u32(&my_bars[k % kStages]), (k / kStages) & 1);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_run[nt] = -INFINITY;
      l_run[nt] = 0.f;
#pragma unroll
      for (int mi = 0; mi < 8; ++mi)
#pragma unroll
        for (int c = 0; c < 4; ++c) O[nt][mi][c] = 0.f;
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], off);
  __syncthreads();
  float* mw = reinterpret_cast<float*>(smem);
  float* lw = mw + kWarps * kMaxGqa;
  float* ow = lw + kWarps * kMaxGqa;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int qi = 4 * nt + t;
    if (qi < gqa) {
      if (g == 0) {
        mw[warp * kMaxGqa + qi] = m_run[nt];
        lw[warp * kMaxGqa + qi] = l_run[nt];
      }
      // m-tile mi: channels 16 mi + g (rows g) and 16 mi + g + 8 (rows g + 8)
#pragma unroll
      for (int mi = 0; mi < 8; ++mi) {
        ow[(warp * kMaxGqa + qi) * kD + 16 * mi + g] = O[nt][mi][0] + O[nt][mi][1];
        ow[(warp * kMaxGqa + qi) * kD + 16 * mi + g + 8] = O[nt][mi][2] + O[nt][mi][3];
      }
    }
  }
  __syncthreads();
  for (int idx = tid; idx < gqa * kD; idx += kWarps * 32) {
    const int qi = idx / kD, ch = idx % kD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mw[w * kMaxGqa + qi]);
    float o = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mwq = mw[w * kMaxGqa + qi];
        if (mwq != -INFINITY) o += fast_exp2(mwq - M) * ow[(w * kMaxGqa + qi) * kD + ch];
      }
    }
    p.part_o[((bh0 + qi) * p.ns + s) * kD + ch] = o;
  }
  if (tid < gqa) {
    float M = -INFINITY, l = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mw[w * kMaxGqa + tid]);
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mwq = mw[w * kMaxGqa + tid];
        if (mwq != -INFINITY) l += fast_exp2(mwq - M) * lw[w * kMaxGqa + tid];
      }
    }
    p.part_ml[((bh0 + tid) * p.ns + s) * 2 + 0] = M;
    p.part_ml[((bh0 + tid) * p.ns + s) * 2 + 1] = l;
  }
}

template <int NT>
cudaError_t launch_impl(const Params& p, cudaStream_t stream) {
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(bf16_mma_split_kernel<NT>), kSmem);
  if (e != cudaSuccess) return e;
  bf16_mma_split_kernel<NT><<<dim3(p.ns, p.H, p.B), kWarps * 32, kSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int bf16_mma_ctas_per_sm(int gqa) {
  static std::mutex mu;
  static int cache[64][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 2;
  const int two = gqa > 4 ? 1 : 0;
  std::lock_guard<std::mutex> lock(mu);
  int& c = cache[dev][two];
  if (c == 0) {
    const void* k = two ? reinterpret_cast<const void*>(bf16_mma_split_kernel<2>)
                        : reinterpret_cast<const void*>(bf16_mma_split_kernel<1>);
    int n = 0;
    if (set_smem_limit_once(k, kSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kWarps * 32, kSmem) != cudaSuccess || n <= 0)
      n = 2;
    c = n;
  }
  return c;
}

bool bf16_mma_supported(const Params& p) { return p.D == kD && p.gqa >= 1 && p.gqa <= 8 && p.pps <= kMaxPps; }

cudaError_t bf16_mma_split(const Params& p, cudaStream_t stream) {
  return p.gqa > 4 ? launch_impl<2>(p, stream) : launch_impl<1>(p, stream);
}

}  // namespace oscar_dec

oscar_status_t oscar_internal_decode_bf16_errors(uint32_t* flags, int reset) {
  return oscar::read_unit_errors(flags, reset) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}
