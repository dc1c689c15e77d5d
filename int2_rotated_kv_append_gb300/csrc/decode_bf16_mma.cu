// Tensor-core split kernel of the all-BF16 paged decode, the speedup reference
// the OSCAR pages compare against ("OSCAR: Offline Spectral Covariance-Aware
// Rotation for 2-bit KV Cache Quantization", summary "Practical Summary":
// faster decoding than BF16).
//
// Shape covered: head_dim 128, GQA 1..8.  One CTA of 4 warps owns one split of
// one (sequence, KV head); each warp takes every 4th page of the split.
// Per warp and page (16 tokens, K and V rows of 256 bytes):
//   * the 8 KB of the page arrive by 16-byte asynchronous copies, 16 per lane (each
//     instruction moves two whole rows, coalesced), into a padded shared-memory
//     stage (272-byte rows, so ldmatrix is bank-conflict free); every lane's copies
//     complete an arrival on the stage's mbarrier, a ring of kStages pages per warp
//     with bounded waits;
//   * QK:  S^T[token][query] = K[token][ch] . Q[ch][query], A from ldmatrix,
//     B = q * scale * log2(e) split into bf16 hi + lo (16 significant bits);
//   * online softmax per query with warp shuffles;
//   * PV:  O^T[ch][query] += V^T[ch][token] . P[token][query], A from
//     ldmatrix.trans, B = p split into bf16 hi + lo;
// then a log-sum-exp merge of the warps through shared memory.
#include <mutex>

#include "bf16_page.cuh"

namespace oscar_dec {
namespace {

using bf16pg::kD;
using bf16pg::kRowBytes;
using bf16pg::kRowPitch;
using bf16pg::kStageBytes;
constexpr int kWarps = 4;
constexpr int kStages = 2;  // 2 pages per warp: three 4-warp CTAs fit in shared memory
constexpr int kMaxPps = 256;
constexpr size_t kSmem = static_cast<size_t>(kWarps) * kStages * kStageBytes + kWarps * kStages * 8 + kMaxPps * 4;

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
  if (r1 <= r0) {  // nothing of the sequence in this split: an empty partial (the merge skips it)
    if (tid < gqa) {
      p.part_ml[((bh0 + tid) * p.ml_ns + s) * 2 + 0] = -INFINITY;
      p.part_ml[((bh0 + tid) * p.ml_ns + s) * 2 + 1] = 0.f;
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
    for (int i = 0; i < kStages; ++i) mbar_init(smem_u32(&bars[warp * kStages + i]), 32);  // one arrival per lane
  mbar_init_fence();
  __syncthreads();

  const int n_my = npg > warp ? (npg - warp + kWarps - 1) / kWarps : 0;
  uint8_t* my_stages = smem + warp * kStages * kStageBytes;
  uint64_t* my_bars = bars + warp * kStages;
  // Whole warp: copy k moves rows 2k, 2k + 1 of the (page, head) block (K rows 0..15,
  // V rows 16..31): lane l takes 16-byte chunk l % 16 of row 2k + l / 16.  A page with
  // an invalid id is zeroed instead (its tokens are masked; zero V rows keep p * v finite).
  const int c16 = lane & 15, rsel = lane >> 4;
  auto issue = [&](int i) {
    const int pid = pid_s[warp + i * kWarps];
    const uint32_t st = smem_u32(my_stages + (i % kStages) * kStageBytes);
    if (pid >= 0) {
      const __nv_bfloat16* src = p.pages + (static_cast<size_t>(pid) * p.H + h) * 2 * kPageSize * kD + c16 * 8;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int r = 2 * k + rsel;
        cp_async16(st + bf16pg::stage_row(r) * kRowPitch + c16 * 16, src + r * kD);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int r = 2 * k + rsel;
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(st + bf16pg::stage_row(r) * kRowPitch + c16 * 16),
                     "r"(0u) : "memory");
      }
    }
    cp_async_arrive(smem_u32(&my_bars[i % kStages]));
  };
  for (int i = 0; i < n_my && i < kStages; ++i) issue(i);

  uint32_t bq[NT][8][2];
  bf16pg::build_bq<NT>(p.q + bh0 * kD, p.scale_log2, gqa, g, t, bq);
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
  const bf16pg::LaneOffsets lo = bf16pg::lane_offsets(lane);
  bool aborted = false;
  int i = 0;
  for (; i < n_my; ++i) {
    const uint32_t bar = smem_u32(&my_bars[i % kStages]);
    const bool ok = mbar_wait_bounded(bar, (i / kStages) & 1);
    if (__any_sync(0xffffffffu, !ok)) {
      aborted = true;
      break;
    }
    const int jpage = warp + i * kWarps;
    const bool page_ok = pid_s[jpage] >= 0;
    const int pos0 = (pg0 + jpage) * kPageSize + g;
    const bool v0 = page_ok && pos0 >= r0 && pos0 < r1;
    const bool v1 = page_ok && pos0 + 8 >= r0 && pos0 + 8 < r1;
    bf16pg::page<NT>(smem_u32(my_stages + (i % kStages) * kStageBytes), lo, g, v0, v1, bq, m_run, l_run, O);
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
  bf16pg::store_warp<NT>(O, m_run, l_run, mw, lw, ow, warp, g, t, gqa);
  __syncthreads();
  merge_warps_store<kWarps, kD, kWarps * 32>(p, mw, lw, ow, s, bh0, tid);
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

bool bf16_mma_supported(const Params& p) {
  return p.mma != 0 && p.D == kD && p.gqa >= 1 && p.gqa <= 8 && p.pps <= kMaxPps;
}

cudaError_t bf16_mma_split(const Params& p, cudaStream_t stream) {
  return p.gqa > 4 ? launch_impl<2>(p, stream) : launch_impl<1>(p, stream);
}

}  // namespace oscar_dec

oscar_status_t oscar_internal_decode_bf16_errors(uint32_t* flags, int reset) {
  return oscar::read_unit_errors(flags, reset) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}
