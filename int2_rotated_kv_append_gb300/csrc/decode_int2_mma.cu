// Tensor-core split kernel of the OSCAR decode for the INT2 bulk
// ("OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
// Quantization", abstract: INT2 attention kernel over a paged KV cache;
// project card "How it works": fused mixed-precision attention).
//
// Shape covered: head_dim 128, group 64 or 128, GQA 1..8.  One CTA of 4 warps
// owns one split (a run of pages) of one (sequence, KV head); BF16 sink/window
// splits of the same grid run the CUDA-core body of decode_common.cuh.
//
// Per warp and page (16 tokens x 128 channels, K and V):
//   * the page's 1024 code bytes and 128/256 scale-zero bytes arrive by two
//     bulk async copies (cp.async.bulk + mbarrier) into a per-warp ring of
//     kStages pages, so many pages per SM are in flight;
//   * QK:  S^T[token][query] = C_k[token][ch] . Qs[ch][query] on mma.sync
//     m16n8k16 (fp16 in, fp32 accumulate), one accumulator per group.  A is
//     built from the packed codes with one AND per register: the 2-bit code at
//     bit position k of an fp16 half is the subnormal c * 2^(k-24), exact.  B
//     holds q.R_k (already in log2 units) times 2^(E_q - k) for that channel,
//     split into fp16 hi + lo (about 22 significant bits), so the product
//     c * q * 2^(E_q - 24) is exact for every channel;
//   * logits: sum_g scale_g * 2^(24 - E_q) * acc_g + zero_g * sum_{ch in g} q;
//     online softmax per query with warp shuffles;
//   * PV:  O^T[ch][query] += C_v^T[ch][token] . P'[token][query] on the same
//     MMA; A pairs two tokens of one channel (one byte-permute + one AND), B is
//     P' = p * scale_g (p <= 1, so P' <= scale <= 65504 never overflows fp16)
//     split into fp16 hi + lo; lo is subnormal for small weights, an absolute
//     error of at most 2^-25 per weight.  The zero term sum p * zero_g and the
//     per-channel power of two are applied once at the end;
//   * pages entirely inside the split's range take a path without per-token
//     masking.
// The warps of a CTA are merged through shared memory by log-sum-exp and the
// CTA writes one (max, sum, output) partial per query head.
#include <mutex>

#include "append_token.cuh"
#include "int2_page.cuh"

namespace oscar_dec {
namespace {

constexpr int kWarps = 4;
constexpr int kStages = 6;               // pages in flight per warp
constexpr int kFirstIssue = 2;           // pages per warp requested before the query fragments
constexpr int kMaxPps = 256;             // page ids of one split staged in shared memory
constexpr int kDenseStage = bf16pg::kStageBytes;  // one BF16 sink/window page per warp

constexpr int kDensePagesPerCta = 8;  // 16-row sink/window pages per dense CTA (2 per warp)

template <int NG>
struct Geo {
  static constexpr int kSzBytes = PageGeo<NG>::kSzBytes;
  static constexpr int kStageBytes = PageGeo<NG>::kStageBytes;
  // page stages (or one BF16 stage per warp) | mbarriers | page ids
  static constexpr size_t kStageArea = static_cast<size_t>(kWarps) * kStages * kStageBytes > kWarps * kDenseStage
                                           ? static_cast<size_t>(kWarps) * kStages * kStageBytes
                                           : static_cast<size_t>(kWarps) * kDenseStage;
  // | QK operand block (kQfragBytes) | its mbarrier
  static constexpr size_t kPagedSmem = kStageArea + kWarps * kStages * 8 + kMaxPps * 4 + kQfragBytes + 16;
  static constexpr size_t kSmem = kPagedSmem > split_body_smem(kD) ? kPagedSmem : split_body_smem(kD);
};

// ---- the kernel --------------------------------------------------------------

template <int NT, int NG>
__global__ void __launch_bounds__(kWarps * 32, NT == 1 ? 5 : 3) int2_mma_split_kernel(Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  // Dispatch order: KV head fastest, then sequence, split index slowest, so the
  // last CTAs to start are the high splits that only long sequences have.
  const int s = blockIdx.z + p.split_base, h = blockIdx.x, b = blockIdx.y;
  if (s >= p.n_paged) {  // BF16 sink/window pages (and, in oscar_append_decode, the current token's append)
    if (p.app_k != nullptr && s - p.n_paged == current_token_dense_cta(p, b, kDensePagesPerCta))
      fused_append_token<kWarps>(p, b, h, smem);
    dense_part<NT, kWarps>(p, (s - p.n_paged) * kDensePagesPerCta, kDensePagesPerCta, s, h, b, smem);
    return;
  }
  constexpr int kStageBytes = Geo<NG>::kStageBytes;
  constexpr int kSzBytes = Geo<NG>::kSzBytes;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int gqa = p.gqa;
  // Page ids of the whole split are loaded together with the sequence length (they
  // do not depend on it); only the pages in range are validated and used.
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Geo<NG>::kStageArea);
  int* pid_all = reinterpret_cast<int*>(bars + kWarps * kStages);
  uint32_t* qbuf = reinterpret_cast<uint32_t*>(pid_all + kMaxPps);  // [32 lanes][kQfragWords]
  uint64_t* qbar = reinterpret_cast<uint64_t*>(qbuf + 32 * kQfragWords);
  const int sp0 = s * p.pps;
  const int spn = max(0, min(p.pps, p.max_pages - sp0));
  const RowView rv = row_view(p, b);
  for (int k = tid; k < spn; k += kWarps * 32)
    pid_all[k] = __ldg(p.page_table + static_cast<size_t>(rv.seq) * p.max_pages + sp0 + k);
  const int L = rv.L;
  const int win_begin = max(p.S, L - p.W);
  const int lo_pos = s * p.pps * kPageSize;
  const int r0 = max(lo_pos, p.S), r1 = min(lo_pos + p.pps * kPageSize, min(win_begin, rv.A));
  const size_t bh0 = static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * gqa;

  if (r1 <= r0) {  // nothing of the bulk falls in this split: an empty partial (the merge skips it)
    grid_dep_launch_dependents();
    if (tid < gqa) {
      p.part_ml[((bh0 + tid) * p.ml_ns + s) * 2 + 0] = -INFINITY;
      p.part_ml[((bh0 + tid) * p.ml_ns + s) * 2 + 1] = 0.f;
    }
    grid_dep_wait();  // keeps completion ordered after the q-rotation kernel
    return;
  }
  const int pg0 = r0 / kPageSize;
  const int npg = (r1 - 1) / kPageSize + 1 - pg0;

  uint8_t* stages = smem;
  const int* pid_s = pid_all + (pg0 - sp0);  // page ids from the split's first page in range
  if (lane == 0)
    for (int i = 0; i < kStages; ++i) mbar_init(smem_u32(&bars[warp * kStages + i]), 1);
  if (tid == 0) mbar_init(smem_u32(qbar), 1);
  mbar_init_fence();
  __syncthreads();

  const int n_my = npg > warp ? (npg - warp + kWarps - 1) / kWarps : 0;
  uint8_t* my_stages = stages + warp * kStages * kStageBytes;
  uint64_t* my_bars = bars + warp * kStages;
  const uint32_t stage_base = smem_u32(my_stages);
  // Pages are read once: for GQA 8 they are marked evict-first in L2, so that the
  // stream of pages does not push out what is read again soon (the split partials
  // the merge reads, R_k and R_v, page tables).  Measured: 3% faster at 131K tokens
  // with 64-page splits (GQA 8), 1% slower at batch 64 (GQA 4), where it is off.
  const uint64_t stream_policy = l2_evict_first_policy();
  // Whole warp: bring local pages [i0, i1) of this warp (at most 16) into their
  // stages.  Lane 2j handles page i0 + j's codes, lane 2j + 1 its scale/zero, so the
  // whole batch is requested by one bulk-copy instruction: the issue of a bulk
  // copy takes a few hundred cycles, and copies requested by one lane one after
  // another would hold the warp that long for each of them.
  auto issue = [&](int i0, int i1) {
    const int i = i0 + (lane >> 1), part = lane & 1;
    const bool active = i < i1;
    const int pid = active ? pid_s[warp + i * kWarps] : 0;
    const bool bad = pid < 0 || pid >= p.num_pages;
    const uint32_t bar = smem_u32(&my_bars[i % kStages]);
    if (active && part == 0) {
      if (bad) {
        record_error(OSCAR_DEVERR_PAGE_ID);
        mbar_arrive(bar);
      } else {
        mbar_arrive_expect_tx(bar, kStageBytes);
      }
    }
    __syncwarp();
    if (active && !bad) {
      const size_t ph = static_cast<size_t>(pid) * p.H + h;
      const uint8_t* src = part ? reinterpret_cast<const uint8_t*>(p.sz) + ph * kSzBytes : p.codes + ph * kCodeBytes;
      const uint32_t dst = stage_base + (i % kStages) * kStageBytes + (part ? kCodeBytes : 0);
      if (NT == 2) bulk_g2s_hint(dst, src, part ? kSzBytes : kCodeBytes, bar, stream_policy);
      else bulk_g2s(dst, src, part ? kSzBytes : kCodeBytes, bar);
    }
  };
  grid_dep_launch_dependents();
  uint32_t bq[NT][8][2];
  float F[NT], qs[NT][NG];
  bool aborted = false;
  // Pages are read only after the preceding kernels have completed (an append may
  // have written them): the preceding kernel is the q-rotation, which completes
  // after the kernel before it.
  grid_dep_wait();

  // ---- query side: this lane's QK B-fragments and per-query factors ----
  // (built by the q-rotation kernel, kQfragWords words per lane).  Per n-tile nt
  // the lane's C columns belong to query 4*nt + t and its B column to query
  // 4*nt + (g >> 1), part g & 1.
  // The block of the (sequence, KV head) arrives by one bulk copy: all the split
  // CTAs of a head read it at the same time, and whole-line requests load the L2
  // far less than per-lane 16-byte loads.  The remaining pages are requested once
  // it has landed.
  // The first kFirstIssue pages of each warp are requested before the operand
  // block, the rest once it has landed: a request made behind every page of the
  // grid would wait for most of the page traffic.
  issue(0, min(n_my, kFirstIssue));
  if (tid == 0) {
    mbar_arrive_expect_tx(smem_u32(qbar), kQfragBytes);
    bulk_g2s(smem_u32(qbuf), p.qfrag + (static_cast<size_t>(b) * p.H + h) * (32 * kQfragWords), kQfragBytes,
             smem_u32(qbar));
  }
  const bool q_ok = __any_sync(0xffffffffu, !mbar_wait_bounded(smem_u32(qbar), 0)) == 0;
  aborted = !q_ok;
  issue(min(n_my, kFirstIssue), min(n_my, kStages));
  const uint4* qw4 = reinterpret_cast<const uint4*>(qbuf + lane * kQfragWords);
  // GQA 8 (two n-tiles): the page body reads the QK B-fragments from the operand
  // block in shared memory, which keeps the kernel at 168 registers, 3 CTAs per SM
  // instead of 2 (131K decode 194.5 -> 190.9 us; with one page per iteration
  // instead of two it was 200.5 us)
  constexpr bool kBqs = NT == 2;
  const uint32_t bqs = smem_u32(qbuf + lane * kQfragWords);
  {
    uint4 v[4 * NT], f[3];
    if (!kBqs) {
#pragma unroll
      for (int k = 0; k < 4 * NT; ++k) v[k] = qw4[k];
    }
#pragma unroll
    for (int k = 0; k < 3; ++k) f[k] = qw4[8 + k];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        bq[nt][2 * k][0] = kBqs ? 0u : v[4 * nt + k].x;
        bq[nt][2 * k][1] = kBqs ? 0u : v[4 * nt + k].y;
        bq[nt][2 * k + 1][0] = kBqs ? 0u : v[4 * nt + k].z;
        bq[nt][2 * k + 1][1] = kBqs ? 0u : v[4 * nt + k].w;
      }
    const uint32_t fw[12] = {f[0].x, f[0].y, f[0].z, f[0].w, f[1].x, f[1].y,
                             f[1].z, f[1].w, f[2].x, f[2].y, f[2].z, f[2].w};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      F[nt] = __uint_as_float(fw[5 * nt]);
      // group sums from the four 32-column block sums
      const float c0 = __uint_as_float(fw[5 * nt + 1]), c1 = __uint_as_float(fw[5 * nt + 2]);
      const float c2 = __uint_as_float(fw[5 * nt + 3]), c3 = __uint_as_float(fw[5 * nt + 4]);
      if (NG == 2) {
        qs[nt][0] = c0 + c1;
        qs[nt][NG - 1] = c2 + c3;
      } else {
        qs[nt][0] = (c0 + c1) + (c2 + c3);
      }
    }
  }
  // ---- main loop over this warp's pages ----
  float m_run[NT], O[NT][8][4];
  float2 l2[NT], z2[NT][NG];  // per token slot (g, g + 8) of the page body
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt] = -INFINITY;
    l2[nt] = make_float2(0.f, 0.f);
#pragma unroll
    for (int gg = 0; gg < NG; ++gg) z2[nt][gg] = make_float2(0.f, 0.f);
#pragma unroll
    for (int mi = 0; mi < 8; ++mi)
#pragma unroll
      for (int c = 0; c < 4; ++c) O[nt][mi][c] = 0.f;
  }
  const uint32_t vsel = (2 * (g & 1)) | ((2 * (g & 1) + 1) << 4) | ((4 + 2 * (g & 1)) << 8) | ((5 + 2 * (g & 1)) << 12);
  int i = 0;
  // Stage of local page k: k % kStages (kStages even: a pair never wraps).  Under the
  // stall test the first page is awaited on the operand barrier's second phase, which
  // nothing completes (its first phase has completed: q_ok).
  auto wait_page = [&](int k) {
    if (p.stall_cycles > 0 && k == 0) return mbar_wait_bounded(smem_u32(qbar), 1, p.stall_cycles);
    return mbar_wait_bounded(smem_u32(&my_bars[k % kStages]), (k / kStages) & 1);
  };
  auto page_full = [&](int k) {
    const int jpage = warp + k * kWarps;
    const int pos_base = (pg0 + jpage) * kPageSize;
    const int pid = pid_s[jpage];
    return pid >= 0 && pid < p.num_pages && pos_base >= r0 && pos_base + kPageSize <= r1;
  };
  auto token_ok = [&](int k, int tok) {
    const int jpage = warp + k * kWarps;
    const int pid = pid_s[jpage];
    const int pos = (pg0 + jpage) * kPageSize + tok;
    return pid >= 0 && pid < p.num_pages && pos >= r0 && pos < r1;
  };
  for (; !aborted && i + 1 < n_my; i += 2) {
    if (__any_sync(0xffffffffu, !wait_page(i) || !wait_page(i + 1))) {
      aborted = true;
      break;
    }
    const uint32_t st2[2] = {stage_base + (i % kStages) * kStageBytes, stage_base + ((i + 1) % kStages) * kStageBytes};
    if (page_full(i) && page_full(i + 1)) {
      bool t2[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) t2[nt][0] = t2[nt][1] = true;
      int2_pages<NT, NG, 2, true, kBqs>(st2, g, t, t2, t2, vsel, bq, F, qs, m_run, l2, z2, O, bqs);
    } else {
      const bool b00 = token_ok(i, g), b01 = token_ok(i + 1, g), b10 = token_ok(i, g + 8), b11 = token_ok(i + 1, g + 8);
      bool a0[NT][2], a1[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        a0[nt][0] = b00;
        a0[nt][1] = b01;
        a1[nt][0] = b10;
        a1[nt][1] = b11;
      }
      int2_pages<NT, NG, 2, false, kBqs>(st2, g, t, a0, a1, vsel, bq, F, qs, m_run, l2, z2, O, bqs);
    }
    __syncwarp();
    issue(min(n_my, i + kStages), min(n_my, i + 2 + kStages));
  }
  if (!aborted && i < n_my) {  // odd last page
    if (__any_sync(0xffffffffu, !wait_page(i))) {
      aborted = true;
    } else {
      const uint32_t st1[1] = {stage_base + (i % kStages) * kStageBytes};
      const bool b0 = token_ok(i, g), b1 = token_ok(i, g + 8);
      bool a0[NT][1], a1[NT][1];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        a0[nt][0] = b0;
        a1[nt][0] = b1;
      }
      int2_pages<NT, NG, 1, false, kBqs>(st1, g, t, a0, a1, vsel, bq, F, qs, m_run, l2, z2, O, bqs);
      ++i;
    }
  }
  if (aborted) {
    if (lane == 0) record_error(OSCAR_DEVERR_TIMEOUT);
    // Let the copies already issued land (bounded) before the shared memory is reused:
    // the operand block if its wait gave up, and the pages requested so far.
    if (!q_ok && lane == 0) mbar_wait_bounded(smem_u32(qbar), 0);
    const int issued = min(n_my, i + kStages);
    for (int k = i; k < issued; ++k) mbar_wait_bounded(smem_u32(&my_bars[k % kStages]), (k / kStages) & 1);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_run[nt] = -INFINITY;
      l2[nt] = make_float2(0.f, 0.f);
#pragma unroll
      for (int gg = 0; gg < NG; ++gg) z2[nt][gg] = make_float2(0.f, 0.f);
#pragma unroll
      for (int mi = 0; mi < 8; ++mi)
#pragma unroll
        for (int c = 0; c < 4; ++c) O[nt][mi][c] = 0.f;
    }
  }

  // ---- warp totals, then a log-sum-exp merge of the 4 warps ----
  float l_run[NT], zacc[NT][NG];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    l_run[nt] = l2[nt].x + l2[nt].y;
#pragma unroll
    for (int gg = 0; gg < NG; ++gg) zacc[nt][gg] = z2[nt][gg].x + z2[nt][gg].y;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], off);
#pragma unroll
      for (int gg = 0; gg < NG; ++gg) zacc[nt][gg] += __shfl_xor_sync(0xffffffffu, zacc[nt][gg], off);
    }
  }
  __syncthreads();  // every stage consumed: the stage area becomes the merge buffer
  float* mw = reinterpret_cast<float*>(smem);  // [kWarps][kMaxGqa]
  float* lw = mw + kWarps * kMaxGqa;           // [kWarps][kMaxGqa]
  float* ow = lw + kWarps * kMaxGqa;           // [kWarps][kMaxGqa][kD]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int qi = 4 * nt + t;
    if (qi < gqa) {
      if (g == 0) {
        mw[warp * kMaxGqa + qi] = m_run[nt];
        lw[warp * kMaxGqa + qi] = l_run[nt];
      }
#pragma unroll
      for (int mi = 0; mi < 8; ++mi) {
        const int gg = mi * NG / 8;
        const int word = (mi < 4 ? 0 : 4) + (g >> 1);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int e = 2 * (mi & 3) + r;
          const int ch = 16 * word + 8 * (g & 1) + e;
          ow[(warp * kMaxGqa + qi) * kD + ch] =
              (O[nt][mi][2 * r] + O[nt][mi][2 * r + 1]) * pow2i(24 - kpos(e)) + zacc[nt][gg];
        }
      }
    }
  }
  __syncthreads();
  merge_warps_store<kWarps, kD, kWarps * 32>(p, mw, lw, ow, s, bh0, tid);
}

template <int NT, int NG>
cudaError_t launch_impl(const Params& p, cudaStream_t stream) {
  constexpr size_t smem = Geo<NG>::kSmem;
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(int2_mma_split_kernel<NT, NG>), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(int2_mma_split_kernel<NT, NG>, dim3(p.H, p.B, p.ns - p.split_base), dim3(kWarps * 32), smem,
                    stream, p);
}

}  // namespace

int int2_mma_ctas_per_sm(int gqa, int G) {
  static std::mutex mu;
  static int cache[64][2][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 2;
  const int two = gqa > 4 ? 1 : 0, g64 = G == 64 ? 1 : 0;
  std::lock_guard<std::mutex> lock(mu);
  int& c = cache[dev][two][g64];
  if (c == 0) {
    const void* k = two ? (g64 ? reinterpret_cast<const void*>(int2_mma_split_kernel<2, 2>)
                               : reinterpret_cast<const void*>(int2_mma_split_kernel<2, 1>))
                        : (g64 ? reinterpret_cast<const void*>(int2_mma_split_kernel<1, 2>)
                               : reinterpret_cast<const void*>(int2_mma_split_kernel<1, 1>));
    const size_t smem = g64 ? Geo<2>::kSmem : Geo<1>::kSmem;
    int n = 0;
    if (set_smem_limit_once(k, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kWarps * 32, smem) != cudaSuccess || n <= 0)
      n = 2;
    c = n;
  }
  return c;
}

bool int2_mma_supported(const Params& p) {
  return p.mma != 0 && p.D == kD && (p.G == 64 || p.G == 128) && p.gqa >= 1 && p.gqa <= 8 && p.pps <= kMaxPps;
}

cudaError_t int2_mma_split(const Params& p, cudaStream_t stream) {
  const bool two = p.gqa > 4;
  if (p.G == 64) return two ? launch_impl<2, 2>(p, stream) : launch_impl<1, 2>(p, stream);
  return two ? launch_impl<2, 1>(p, stream) : launch_impl<1, 1>(p, stream);
}

}  // namespace oscar_dec

oscar_status_t oscar_internal_decode_mma_errors(uint32_t* flags, int reset) {
  return oscar::read_unit_errors(flags, reset) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}
