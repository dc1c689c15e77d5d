// Single-wave fused decode of the OSCAR mixed-precision attention for small
// batches ("OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
// Quantization", project card "How it works": rotate the query once so stored
// keys stay rotated, a BF16 sink and recent window beside the INT2 bulk, one
// un-rotation of the output; abstract: INT2 attention over a paged KV cache).
//
// Used when every (sequence, KV head) unit can be given its own CTAs in one wave
// of one CTA per SM: unit u gets n_s INT2 split CTAs and, when the sink or
// window is non-empty, one BF16 CTA.  Two kernels per call:
//   fused  an INT2 split CTA (NW warps) first rotates the unit's queries itself,
//          q_rot = q . R_k[h] from R_k staged in shared memory, and builds each
//          lane's tensor-core QK operands; this prologue reads only q and R_k and
//          runs before the dependency wait, so it overlaps the preceding kernel.
//          After the wait it stages its page ids, streams its pages through
//          per-warp rings of bulk async copies (the page body of int2_page.cuh),
//          merges its warps by log-sum-exp, un-rotates the merged output by
//          R_v[h]^T (staged while the pages streamed) and writes one
//          (max, sum, output) partial per query head in the original space.  The
//          BF16 CTA attends the sink and window rows and writes its partial;
//   merge  one warp per (sequence, query head): log-sum-exp of the unit's
//          partials and the normalisation (no rotation left to undo).
// Logits are in log2 units (scale * log2 e folded into the query operands).
#include <mutex>

#include "append_token.cuh"
#include "int2_page.cuh"

namespace oscar_dec {
namespace {

// page ids of one split staged in shared memory (the 8-warp form has room for more)
template <int NW>
constexpr int fused_max_pps() { return NW >= 16 ? 2048 : 4096; }
constexpr int kOwPitch = kD + 4;    // padded row of a warp's output in the merge area

constexpr size_t cmax(size_t a, size_t b) { return a > b ? a : b; }

// Pages in flight per warp: enough that the ring (about 164 KB) holds every page
// of a typical split at once.
template <int NG, int NW>
constexpr int fused_stages() { return (164 * 1024) / (NW * PageGeo<NG>::kStageBytes); }

template <int NT, int NG, int NW>
struct FusedGeo {
  static constexpr int kStages = fused_stages<NG, NW>();
  static constexpr int kStageBytes = PageGeo<NG>::kStageBytes;
  static constexpr int kSzBytes = PageGeo<NG>::kSzBytes;
  // Area 0, reused in turn: (a) the page ring; (b) the warps' states after the loop;
  // (c) for the BF16 CTA, one 16-row stage per warp and its barriers.
  static constexpr size_t kRing = static_cast<size_t>(NW) * kStages * kStageBytes;
  static constexpr size_t kWarpState = static_cast<size_t>(NW) * kMaxGqa * (2 + kOwPitch) * 4 + 4 * NT * kD * 4;
  static constexpr size_t kDense = static_cast<size_t>(NW) * bf16pg::kStageBytes + NW * 8;
  static constexpr size_t kArea0 = cmax(kRing, cmax(kWarpState, kDense));
  // The q-rotation's QK operand block of the unit (kQfragBytes), in use while the ring fills.
  static constexpr size_t kOffFrag = (kArea0 + 127) / 128 * 128;
  static constexpr size_t kOffMisc = kOffFrag + kQfragBytes;
  static constexpr size_t kOffPid = kOffMisc + 64 * 4;              // page ids [fused_max_pps]
  static constexpr size_t kOffBars = kOffPid + fused_max_pps<NW>() * 4;  // NW * kStages ring barriers
  static constexpr size_t kSmem = kOffBars + (NW * kStages + 1) * 8;  // + the operand block's barrier
};

// INT2 split CTA s < n_paged of unit (b, h), or the unit's BF16 CTA (s == n_paged).
// The 16-warp form is held to 96 registers (the bound of a 20-warp CTA), so that the
// small q-rotation and merge CTAs of neighbouring calls fit on an SM beside it.
template <int NT, int NG, int NW>
__global__ void __launch_bounds__(NT == 1 ? 640 : NW * 32, 1) int2_fused_kernel(Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  using Geo = FusedGeo<NT, NG, NW>;
  constexpr int T = NW * 32;
  constexpr int kStages = Geo::kStages;
  constexpr int kStageBytes = Geo::kStageBytes;
  constexpr int kSzBytes = Geo::kSzBytes;
  constexpr int kQ = 4 * NT;  // query heads the CTA is compiled for (gqa <= kQ)
  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (s >= p.n_paged) {  // the unit's BF16 sink / window rows (and, fused, the current token's append)
    if (p.app_k != nullptr) fused_append_token<NW>(p, b, h, smem);
    dense_part<NT, NW>(p, 0, p.n_dense_pages, s, h, b, smem);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int gqa = p.gqa;
  const uint32_t* frag = reinterpret_cast<const uint32_t*>(smem + Geo::kOffFrag);
  float* misc = reinterpret_cast<float*>(smem + Geo::kOffMisc);
  float* Ms = misc + 24;  // [8] CTA maximum per query
  float* Ls = misc + 32;  // [8] CTA sum per query
  int* pids = reinterpret_cast<int*>(smem + Geo::kOffPid);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Geo::kOffBars);
  const uint32_t fbar = smem_u32(&bars[NW * kStages]);
  const size_t bh0 = static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * gqa;

  if (tid == 0) {
    for (int i = 0; i <= NW * kStages; ++i) mbar_init(smem_u32(&bars[i]), 1);
    mbar_init_fence();
  }
  __syncthreads();
  grid_dep_launch_dependents();
  {
    // Before the dependency wait (the preceding kernels may still run): the split's
    // pages as the current length and page table give them are prefetched into L2.
    // This reads the length and the page table early but only as a hint: every value
    // used below is read again after the wait, and a prefetched line is still updated
    // by any later write, so a page an earlier kernel changes is read correctly.
    int L = __ldg(p.seq_lens + b);
    L = L < 0 ? 0 : (L > p.max_seq_len ? p.max_seq_len : L);
    const int wb = max(p.S, L - p.W);
    const int lo = (p.bulk_lo + s * p.pps) * kPageSize;
    const int q0 = max(lo, p.S), q1 = min(lo + p.pps * kPageSize, wb);
    const int pf0 = q0 / kPageSize, npf = q1 > q0 ? (q1 - 1) / kPageSize + 1 - pf0 : 0;
    // (line by line through the load/store path: bulk prefetches would queue in the
    // bulk-copy unit ahead of the split's own copies)
    constexpr int kLines = (kCodeBytes + kSzBytes) / 128;  // 10 (group 64) or 9 (group 128)
    for (int k = tid; k < npf * kLines; k += T) {
      const int pg = k / kLines, ln = k % kLines;
      const int pid = __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pf0 + pg);
      if (pid >= 0 && pid < p.num_pages) {
        const size_t ph = static_cast<size_t>(pid) * p.H + h;
        prefetch_l2_line(ln < kCodeBytes / 128 ? p.codes + ph * kCodeBytes + ln * 128
                                               : reinterpret_cast<const uint8_t*>(p.sz) + ph * kSzBytes +
                                                     (ln - kCodeBytes / 128) * 128);
      }
    }
  }
  // ---- the q-rotation's operands, lengths, page ids and pages may come from the
  // preceding kernels (the q-rotation, and an append before it) ----
  grid_dep_wait();
  if (tid == 0) {  // the unit's operand block (5.6 KB) by one bulk copy
    mbar_arrive_expect_tx(fbar, kQfragBytes);
    bulk_g2s(smem_u32(frag), p.qfrag + (static_cast<size_t>(b) * p.H + h) * (32 * kQfragWords), kQfragBytes, fbar);
  }
  const RowView rv = row_view(p, b);
  const int win_begin = max(p.S, rv.L - p.W);
  const int lo_pos = (p.bulk_lo + s * p.pps) * kPageSize;
  const int r0 = max(lo_pos, p.S), r1 = min(lo_pos + p.pps * kPageSize, min(win_begin, rv.A));
  const int pg0 = r0 / kPageSize;
  const int npg = r1 > r0 ? (r1 - 1) / kPageSize + 1 - pg0 : 0;
  for (int k = tid; k < npg; k += T)
    pids[k] = __ldg(p.page_table + static_cast<size_t>(rv.seq) * p.max_pages + pg0 + k);
  __syncthreads();
  if (npg == 0) {  // nothing of the bulk in this split: an empty partial (the merge skips it)
    if (tid < gqa) {
      p.part_ml[((bh0 + tid) * p.ml_ns + s) * 2 + 0] = -INFINITY;
      p.part_ml[((bh0 + tid) * p.ml_ns + s) * 2 + 1] = 0.f;
    }
    if (tid == 0) mbar_wait_bounded(fbar, 0);  // the operand copy lands before the CTA exits
    return;
  }

  const int n_my = npg > warp ? (npg - warp + NW - 1) / NW : 0;
  uint64_t* my_bars = bars + warp * kStages;
  const uint64_t stream_policy = l2_evict_first_policy();
  const uint32_t stage_base = smem_u32(smem) + warp * kStages * kStageBytes;
  // Whole warp: local pages [i0, i1) of this warp (at most 16) into their stages;
  // lane 2j requests page i0 + j's codes, lane 2j + 1 its scale/zero, so a batch
  // of copies is one instruction.
  auto issue = [&](int i0, int i1) {
    const int i = i0 + (lane >> 1), part_sel = lane & 1;
    const bool active = i < i1;
    const int pid = active ? pids[warp + i * NW] : 0;
    const bool bad = pid < 0 || pid >= p.num_pages;
    const uint32_t bar = smem_u32(&my_bars[i % kStages]);
    if (active && part_sel == 0) {
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
      const uint8_t* src = part_sel ? reinterpret_cast<const uint8_t*>(p.sz) + ph * kSzBytes
                                    : p.codes + ph * kCodeBytes;
      bulk_g2s_hint(stage_base + (i % kStages) * kStageBytes + (part_sel ? kCodeBytes : 0), src,
                    part_sel ? kSzBytes : kCodeBytes, bar, stream_policy);
    }
  };
  for (int i0 = 0; i0 < min(n_my, kStages); i0 += 16) issue(i0, min(min(n_my, kStages), i0 + 16));

  // ---- this lane's QK B-fragments and per-query factors from the operand block
  // (kQfragWords words per lane, written by the q-rotation: per n-tile nt the lane's
  // C columns belong to query 4*nt + t and its B column to query 4*nt + (g >> 1),
  // part g & 1) ----
  const bool frag_ok = __any_sync(0xffffffffu, !mbar_wait_bounded(fbar, 0)) == 0;
  uint32_t bq[NT][8][2];
  float F[NT], qs[NT][NG];
  {
    const uint4* qw4 = reinterpret_cast<const uint4*>(frag + lane * kQfragWords);
    uint4 v[4 * NT], f[3];
#pragma unroll
    for (int k = 0; k < 4 * NT; ++k) v[k] = qw4[k];
#pragma unroll
    for (int k = 0; k < 3; ++k) f[k] = qw4[8 + k];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        bq[nt][2 * k][0] = v[4 * nt + k].x;
        bq[nt][2 * k][1] = v[4 * nt + k].y;
        bq[nt][2 * k + 1][0] = v[4 * nt + k].z;
        bq[nt][2 * k + 1][1] = v[4 * nt + k].w;
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
  // Under the stall test the first page is awaited on the operand barrier's second
  // phase, which nothing completes (its first phase has completed: frag_ok).
  auto wait_page = [&](int k) {
    if (p.stall_cycles > 0 && k == 0) return mbar_wait_bounded(fbar, 1, p.stall_cycles);
    return mbar_wait_bounded(smem_u32(&my_bars[k % kStages]), (k / kStages) & 1);
  };
  auto page_full = [&](int k) {
    const int jpage = warp + k * NW;
    const int pos_base = (pg0 + jpage) * kPageSize;
    const int pid = pids[jpage];
    return pid >= 0 && pid < p.num_pages && pos_base >= r0 && pos_base + kPageSize <= r1;
  };
  auto token_ok = [&](int k, int tok) {
    const int jpage = warp + k * NW;
    const int pid = pids[jpage];
    const int pos = (pg0 + jpage) * kPageSize + tok;
    return pid >= 0 && pid < p.num_pages && pos >= r0 && pos < r1;
  };
  bool aborted = !frag_ok;
  int i = 0;
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
      int2_pages<NT, NG, 2, true>(st2, g, t, t2, t2, vsel, bq, F, qs, m_run, l2, z2, O);
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
      int2_pages<NT, NG, 2, false>(st2, g, t, a0, a1, vsel, bq, F, qs, m_run, l2, z2, O);
    }
    if (i + kStages < n_my) {  // refill the two stages just consumed
      __syncwarp();
      issue(i + kStages, min(n_my, i + 2 + kStages));
    }
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
      int2_pages<NT, NG, 1, false>(st1, g, t, a0, a1, vsel, bq, F, qs, m_run, l2, z2, O);
      ++i;
    }
  }
  if (aborted) {
    if (lane == 0) record_error(OSCAR_DEVERR_TIMEOUT);
    // let the copies already requested land (bounded) before the shared memory is reused:
    // the operand block if its wait gave up, and the pages
    if (!frag_ok && lane == 0) mbar_wait_bounded(fbar, 0);
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

  // ---- warp totals, then a log-sum-exp merge of the NW warps ----
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
  __syncthreads();  // every stage consumed: the ring becomes the warps' state area
  float* mw = reinterpret_cast<float*>(smem);  // [NW][8]
  float* lw = mw + NW * kMaxGqa;               // [NW][8]
  float* ow = lw + NW * kMaxGqa;               // [NW][8][kOwPitch], rotated space
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int qi = 4 * nt + t;
    if (qi < gqa) {
      if (g == 0) {
        mw[warp * kMaxGqa + qi] = m_run[nt];
        lw[warp * kMaxGqa + qi] = l_run[nt];
      }
      float* orow = ow + (warp * kMaxGqa + qi) * kOwPitch;
#pragma unroll
      for (int mi = 0; mi < 8; ++mi) {
        const int gg = mi * NG / 8;
        const int ch = 16 * ((mi < 4 ? 0 : 4) + (g >> 1)) + 8 * (g & 1) + 2 * (mi & 3);
        const float2 v = make_float2((O[nt][mi][0] + O[nt][mi][1]) * pow2i(24 - kpos(2 * (mi & 3))) + zacc[nt][gg],
                                     (O[nt][mi][2] + O[nt][mi][3]) * pow2i(24 - kpos(2 * (mi & 3) + 1)) + zacc[nt][gg]);
        *reinterpret_cast<float2*>(orow + ch) = v;
      }
    }
  }
  // this warp's rows of R_v for the un-rotation (lane l: columns 4l .. 4l+3), loaded
  // while the other warps finish
  constexpr int kUnrotWarps = NW >= 16 ? 16 : NW;  // warps that take rows of R_v
  constexpr int kRowsPerWarp = kD / kUnrotWarps;    // 8 or 16
  float4 rvr[kRowsPerWarp];
  if (warp < kUnrotWarps) {
    const float4* Rv4 = reinterpret_cast<const float4*>(p.R_v + static_cast<size_t>(h) * kD * kD);
#pragma unroll
    for (int u = 0; u < kRowsPerWarp; ++u) rvr[u] = __ldg(Rv4 + (warp * kRowsPerWarp + u) * (kD / 4) + lane);
  }
  __syncthreads();
  if (warp < gqa) {  // CTA maximum and sum of query `warp`, lane w for warp w's state; mw becomes the weights
    const float mwq = lane < NW ? mw[lane * kMaxGqa + warp] : -INFINITY;
    float M = mwq;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float wt = (M == -INFINITY || mwq == -INFINITY) ? 0.f : fast_exp2(mwq - M);
    float l = lane < NW ? wt * lw[lane * kMaxGqa + warp] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    if (lane < NW) mw[lane * kMaxGqa + warp] = wt;
    if (lane == 0) {
      Ms[warp] = M;
      Ls[warp] = l;
    }
  }
  const bool ok = __syncthreads_and(!aborted);
  // the CTA's output in rotated space (unnormalised), behind the warps' states
  float* orot = ow + NW * kMaxGqa * kOwPitch;  // [kQ][D]
  for (int idx = tid; idx < kQ * (kD / 4); idx += T) {
    const int qi = idx / (kD / 4), c4 = idx % (kD / 4);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (qi < gqa) {
#pragma unroll 4
      for (int w = 0; w < NW; ++w) {
        const float wt = mw[w * kMaxGqa + qi];
        const float4 v = reinterpret_cast<const float4*>(ow + (w * kMaxGqa + qi) * kOwPitch)[c4];
        if (wt != 0.f) {
          o.x = fmaf(wt, v.x, o.x); o.y = fmaf(wt, v.y, o.y); o.z = fmaf(wt, v.z, o.z); o.w = fmaf(wt, v.w, o.w);
        }
      }
    }
    reinterpret_cast<float4*>(orot)[idx] = o;
  }
  __syncthreads();
  // ---- un-rotation, out[c] = sum_j o_rot[j] R_v[h][c][j]: warp w < kUnrotWarps holds
  // rows c0 .. c0 + kRowsPerWarp - 1 of R_v (read from L2 above), forms every (row,
  // query) partial dot product of its lane's columns, then a reduce-scatter across the
  // lanes leaves one total per lane ----
  if (warp < kUnrotWarps) {
    constexpr int kVals = kRowsPerWarp * kQ;       // 32 or 128 partial sums per lane
    const int c0 = warp * kRowsPerWarp;
    float4 oq[kQ];
#pragma unroll
    for (int qi = 0; qi < kQ; ++qi) oq[qi] = reinterpret_cast<const float4*>(orot + qi * kD)[lane];
#pragma unroll
    for (int half = 0; half < kVals / 32; ++half) {
      // values v = 0..31 of this pass: row u = (32 half + v) / kQ, query (32 half + v) % kQ
      float val[32];
#pragma unroll
      for (int v = 0; v < 32; ++v) {
        const int idx = 32 * half + v, u = idx / kQ, qi = idx % kQ;
        val[v] = fmaf(rvr[u].x, oq[qi].x, fmaf(rvr[u].y, oq[qi].y, fmaf(rvr[u].z, oq[qi].z, rvr[u].w * oq[qi].w)));
      }
      // reduce-scatter: after the round with offset o, a lane keeps the half of its
      // values selected by its bit o; at the end lane l holds the total of value l
#pragma unroll
      for (int off = 16, n = 16; off > 0; off >>= 1, n >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int v = 0; v < n; ++v) {
          const float send = upper ? val[v] : val[v + n];
          const float keep = upper ? val[v + n] : val[v];
          val[v] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      // lane l holds value index l (the bits of l chose the halves in order)
      const int idx = 32 * half + lane, u = idx / kQ, qi = idx % kQ;
      if (qi < gqa) p.part_o[((bh0 + qi) * p.ns + s) * kD + c0 + u] = ok ? val[0] : 0.f;
    }
  }
  if (tid < gqa) {
    p.part_ml[((bh0 + tid) * p.ml_ns + s) * 2 + 0] = ok ? Ms[tid] : -INFINITY;
    p.part_ml[((bh0 + tid) * p.ml_ns + s) * 2 + 1] = ok ? Ls[tid] : 0.f;
  }
  if (!ok && tid == 0) record_error(OSCAR_DEVERR_TIMEOUT);
}

// The merge of one (sequence, query head) row per CTA of kLseWarps warps: warp w
// takes splits w, w + kLseWarps, ... (their loads issued together), keeps an online
// log-sum-exp state, and the warps' states are combined through shared memory:
//   out = sum_s w_s o_s / sum_s w_s l_s,  w_s = 2^(m_s - max m),
// every partial already in the original space.  Splits that attended nothing
// (m = -inf) are skipped and their outputs are not read.
constexpr int kLseWarps = 4;
constexpr int kLseChunk = 8;  // splits per warp whose loads are in flight together

__global__ void __launch_bounds__(kLseWarps * 32) fused_merge_kernel(Params p) {
  __shared__ float sm_m[kLseWarps], sm_l[kLseWarps];
  __shared__ float4 sm_o[kLseWarps][kD / 4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row = blockIdx.x;  // b * Hq + hq
  const int ns = p.ns;
  grid_dep_launch_dependents();
  grid_dep_wait();  // the partials come from the preceding kernel
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml + row * p.ml_ns * 2);
  const float4* po = reinterpret_cast<const float4*>(p.part_o + row * ns * kD) + lane;
  float M = -INFINITY, l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = warp; s0 < ns; s0 += kLseWarps * kLseChunk) {
    float2 v[kLseChunk];
    float4 o[kLseChunk];
#pragma unroll
    for (int u = 0; u < kLseChunk; ++u) {
      const int sp = s0 + u * kLseWarps;
      v[u] = sp < ns ? ml[sp] : make_float2(-INFINITY, 0.f);
      o[u] = sp < ns ? po[static_cast<size_t>(sp) * (kD / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float Mc = M;
#pragma unroll
    for (int u = 0; u < kLseChunk; ++u) Mc = fmaxf(Mc, v[u].x);
    if (Mc == -INFINITY) continue;
    const float f = M == -INFINITY ? 0.f : fast_exp2(M - Mc);
    l *= f;
    acc.x *= f; acc.y *= f; acc.z *= f; acc.w *= f;
    M = Mc;
#pragma unroll
    for (int u = 0; u < kLseChunk; ++u) {
      if (v[u].x == -INFINITY) continue;
      const float w = fast_exp2(v[u].x - M);
      l = fmaf(w, v[u].y, l);
      acc.x = fmaf(w, o[u].x, acc.x); acc.y = fmaf(w, o[u].y, acc.y);
      acc.z = fmaf(w, o[u].z, acc.z); acc.w = fmaf(w, o[u].w, acc.w);
    }
  }
  if (lane == 0) {
    sm_m[warp] = M;
    sm_l[warp] = l;
  }
  sm_o[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    float Mt = -INFINITY;
#pragma unroll
    for (int w = 0; w < kLseWarps; ++w) Mt = fmaxf(Mt, sm_m[w]);
    float lt = 0.f;
    float4 ot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kLseWarps; ++w) {
      if (sm_m[w] == -INFINITY) continue;
      const float f = fast_exp2(sm_m[w] - Mt);
      const float4 x = sm_o[w][lane];
      lt = fmaf(f, sm_l[w], lt);
      ot.x = fmaf(f, x.x, ot.x); ot.y = fmaf(f, x.y, ot.y); ot.z = fmaf(f, x.z, ot.z); ot.w = fmaf(f, x.w, ot.w);
    }
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    reinterpret_cast<float4*>(p.out + row * kD)[lane] = make_float4(ot.x * inv, ot.y * inv, ot.z * inv, ot.w * inv);
  }
}

template <int NT, int NG, int NW>
const void* fused_kernel_ptr() {
  return reinterpret_cast<const void*>(int2_fused_kernel<NT, NG, NW>);
}

template <int NT, int NG, int NW>
cudaError_t launch_fused_impl(const Params& p, cudaStream_t stream) {
  constexpr size_t smem = FusedGeo<NT, NG, NW>::kSmem;
  cudaError_t e = set_smem_limit_once(fused_kernel_ptr<NT, NG, NW>(), smem);
  if (e != cudaSuccess) return e;
  // the query rotation and its QK operand blocks, once per (sequence, KV head)
  const int chunks = (p.B + p.qrot_spc - 1) / p.qrot_spc;
  e = launch_pdl(qrot_kernel<kD>, dim3(chunks * p.H, kD / 32), dim3(kQrotThreads), 0, stream, p);
  if (e != cudaSuccess) return e;
  e = launch_pdl(int2_fused_kernel<NT, NG, NW>, dim3(p.ns, p.H, p.B), dim3(NW * 32), smem, stream, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(fused_merge_kernel, dim3(p.B * p.Hq), dim3(kLseWarps * 32), 0, stream, p);
}

// Warps per CTA: 16 for up to 4 query heads per KV head, 8 for more (the 8-query page
// body holds about 220 registers).
constexpr int kFusedWarpsNarrow = 16;
constexpr int kFusedWarpsWide = 8;

}  // namespace

bool int2_fused_shape(int D, int G, int gqa) {
  return D == kD && (G == 64 || G == 128) && gqa >= 1 && gqa <= kMaxGqa;
}

int int2_fused_max_pps(int gqa) {
  return gqa > 4 ? fused_max_pps<kFusedWarpsWide>() : fused_max_pps<kFusedWarpsNarrow>();
}



int int2_fused_ctas_per_sm(int gqa, int G) {
  static std::mutex mu;
  static int cache[64][2][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  const int two = gqa > 4 ? 1 : 0, g64 = G == 64 ? 1 : 0;
  std::lock_guard<std::mutex> lock(mu);
  int& c = cache[dev][two][g64];
  if (c == 0) {
    const void* k = two ? (g64 ? fused_kernel_ptr<2, 2, kFusedWarpsWide>() : fused_kernel_ptr<2, 1, kFusedWarpsWide>())
                        : (g64 ? fused_kernel_ptr<1, 2, kFusedWarpsNarrow>()
                               : fused_kernel_ptr<1, 1, kFusedWarpsNarrow>());
    const size_t smem = two ? (g64 ? FusedGeo<2, 2, kFusedWarpsWide>::kSmem : FusedGeo<2, 1, kFusedWarpsWide>::kSmem)
                            : (g64 ? FusedGeo<1, 2, kFusedWarpsNarrow>::kSmem
                                   : FusedGeo<1, 1, kFusedWarpsNarrow>::kSmem);
    const int threads = (two ? kFusedWarpsWide : kFusedWarpsNarrow) * 32;
    int n = 0;
    if (set_smem_limit_once(k, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, threads, smem) != cudaSuccess || n <= 0)
      n = 1;
    c = n;
  }
  return c;
}

cudaError_t int2_fused_decode(const Params& p, cudaStream_t stream) {
  const bool two = p.gqa > 4;
  if (p.G == 64)
    return two ? launch_fused_impl<2, 2, kFusedWarpsWide>(p, stream) : launch_fused_impl<1, 2, kFusedWarpsNarrow>(p, stream);
  return two ? launch_fused_impl<2, 1, kFusedWarpsWide>(p, stream) : launch_fused_impl<1, 1, kFusedWarpsNarrow>(p, stream);
}

}  // namespace oscar_dec

oscar_status_t oscar_internal_decode_fused_errors(uint32_t* flags, int reset) {
  return oscar::read_unit_errors(flags, reset) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}
