// Tensor-core page bodies of the OSCAR decode shared by its split kernels
// ("OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
// Quantization", abstract: INT2 attention kernel over a paged KV cache; project
// card "How it works": a BF16 sink and recent window beside the INT2 bulk).
//
// int2_pages: NP staged 16-token INT2 pages of one KV head for all GQA query
// heads of one warp (QK and PV on mma.sync with the codes as exact fp16
// subnormals, online softmax); dense_part: the BF16 sink/window rows of one
// (sequence, KV head) on the BF16 page body of bf16_page.cuh.  The operand
// layouts are described in decode_int2_mma.cu.
#pragma once

#include "bf16_page.cuh"

namespace oscar_dec {
namespace {

constexpr int kD = 128;
constexpr int kCodeBytes = 2 * 16 * 32;  // K then V codes of one (page, KV head)

// Bytes of one staged INT2 page (codes, then K and V fp16 (scale, zero) of 16 tokens).
template <int NG>
struct PageGeo {
  static constexpr int kSzBytes = 2 * 16 * NG * 2 * 2;
  static constexpr int kStageBytes = kCodeBytes + kSzBytes;
};

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Bit position, inside its fp16 half, of channel e (0..15) of a packed word
// after the extraction below: e%8 <= 4 sit at 2*(e%8) of the raw word's half,
// e%8 >= 5 at 2*(e%8) - 10 after a right shift by 10.
__host__ __device__ constexpr int kpos(int e) { return (e & 7) <= 4 ? 2 * (e & 7) : 2 * (e & 7) - 10; }

// fp16x2 register holding channels e and e+8 of packed word w (e in 0..7) as the
// subnormals c_e * 2^(kpos(e) - 24) (low half) and c_{e+8} * 2^(kpos(e) - 24).
template <int E>
__device__ __forceinline__ uint32_t extract_pair(uint32_t w, uint32_t w_shr10) {
  constexpr int k = kpos(E);
  constexpr uint32_t mask = (3u << k) | (3u << (16 + k));
  return ((E & 7) <= 4 ? w : w_shr10) & mask;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Shared-memory load at a 32-bit shared address (the stage was filled by a bulk
// copy whose mbarrier phase the caller has already observed).
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float2 lds_h2f(uint32_t addr) {
  const uint32_t v = lds32(addr);
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

// NP (1 or 2) 16-token pages of one warp: QK on tensor cores, online softmax
// (one running maximum update for all NP pages), PV on tensor cores.  With two
// pages the two QK chains and the two PV chains are independent, which hides
// tensor-core and shared-memory latency.  st[k] is page k's stage in shared
// memory.  FULL: every token of the pages is in range (no per-token masking);
// otherwise v0[k] / v1[k] say whether this thread's tokens g and g + 8 of page k
// are.
// A lane's softmax values come in pairs (token g, token g + 8) and are computed as
// packed fp32 pairs.  The PV B operand P' = p * scale of a lane's column (query
// g/2, fp16 part g%2) and tokens 2t, 2t+1 / 2t+8, 2t+9 is the transpose of the
// (token, hi|lo) values the lane holds for query t: one movmatrix per 8 tokens.
// The running sums l_run and the zero terms zacc are kept per token slot of the
// pair and added by the caller at the end.
// BQS: the QK B-fragments are read from shared memory at bqs (this lane's operand
// words: n-tile nt, k-step ks at word nt * 16 + ks * 2) instead of the registers bq,
// which frees 16 registers per n-tile.
template <int NT, int NG, int NP, bool FULL, bool BQS = false>
__device__ __forceinline__ void int2_pages(const uint32_t (&st)[NP], int g, int t, const bool (&v0)[NT][NP],
                                           const bool (&v1)[NT][NP], uint32_t vsel, const uint32_t (&bq)[NT][8][2],
                                           const float (&F)[NT], const float (&qs)[NT][NG], float (&m_run)[NT],
                                           float2 (&l_run)[NT], float2 (&zacc)[NT][NG], float (&O)[NT][8][4],
                                           uint32_t bqs = 0) {
  // K words t and t + 4 of tokens g and g + 8; V words g/2 and 4 + g/2 of tokens
  // 2t, 2t + 1 (xa) and 2t + 8, 2t + 9 (xb); (scale, zero) pairs of K and V for
  // tokens (g, g + 8) per group
  uint32_t kw[NP][4], xa[NP][2], xb[NP][2];
  float2 sk[NP][NG], zk[NP][NG], sv[NP][NG], zv[NP][NG];
#pragma unroll
  for (int pg = 0; pg < NP; ++pg) {
    const uint32_t kp = st[pg] + g * 32 + 4 * t;
    kw[pg][0] = lds32(kp);
    kw[pg][1] = lds32(kp + 16);
    kw[pg][2] = lds32(kp + 256);
    kw[pg][3] = lds32(kp + 272);
    const uint32_t vp = st[pg] + 512 + t * 64 + 4 * (g >> 1);
    xa[pg][0] = __byte_perm(lds32(vp), lds32(vp + 32), vsel);
    xa[pg][1] = __byte_perm(lds32(vp + 16), lds32(vp + 48), vsel);
    xb[pg][0] = __byte_perm(lds32(vp + 256), lds32(vp + 288), vsel);
    xb[pg][1] = __byte_perm(lds32(vp + 272), lds32(vp + 304), vsel);
    const uint32_t sp = st[pg] + kCodeBytes + g * NG * 4;
#pragma unroll
    for (int gg = 0; gg < NG; ++gg) {
      const float2 kg = lds_h2f(sp + 4 * gg), kh = lds_h2f(sp + 32 * NG + 4 * gg);
      const float2 vg = lds_h2f(sp + 64 * NG + 4 * gg), vh = lds_h2f(sp + 96 * NG + 4 * gg);
      sk[pg][gg] = make_float2(kg.x, kh.x);
      zk[pg][gg] = make_float2(kg.y, kh.y);
      sv[pg][gg] = make_float2(vg.x, vh.x);
      zv[pg][gg] = make_float2(vg.y, vh.y);
    }
  }

  float acc[NP][NT][NG][4];
#pragma unroll
  for (int pg = 0; pg < NP; ++pg)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int gg = 0; gg < NG; ++gg)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[pg][nt][gg][c] = 0.f;
#pragma unroll
  for (int pg = 0; pg < NP; ++pg) {
    const uint32_t kw0 = kw[pg][0], kw1 = kw[pg][1], kw2 = kw[pg][2], kw3 = kw[pg][3];
    const uint32_t kw0s = kw0 >> 10, kw1s = kw1 >> 10, kw2s = kw2 >> 10, kw3s = kw3 >> 10;
#define OSCAR_QK_STEP(KS)                                                                         \
  {                                                                                               \
    constexpr int gg = (KS) * NG / 8;                                                             \
    constexpr int j = 2 * ((KS) & 3);                                                             \
    const uint32_t wa = (KS) < 4 ? kw0 : kw1, was = (KS) < 4 ? kw0s : kw1s;                       \
    const uint32_t wb = (KS) < 4 ? kw2 : kw3, wbs = (KS) < 4 ? kw2s : kw3s;                       \
    const uint32_t a0 = extract_pair<j>(wa, was), a1 = extract_pair<j>(wb, wbs);                  \
    const uint32_t a2 = extract_pair<j + 1>(wa, was), a3 = extract_pair<j + 1>(wb, wbs);          \
    _Pragma("unroll") for (int nt = 0; nt < NT; ++nt) {                                           \
      uint32_t b0 = bq[nt][KS][0], b1 = bq[nt][KS][1];                                            \
      if (BQS) {                                                                                  \
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"                                           \
                     : "=r"(b0), "=r"(b1) : "r"(bqs + (nt * 16 + (KS) * 2) * 4));                 \
      }                                                                                           \
      mma16816(acc[pg][nt][gg], a0, a1, a2, a3, b0, b1);                                          \
    }                                                                                             \
  }
    OSCAR_QK_STEP(0) OSCAR_QK_STEP(1) OSCAR_QK_STEP(2) OSCAR_QK_STEP(3)
    OSCAR_QK_STEP(4) OSCAR_QK_STEP(5) OSCAR_QK_STEP(6) OSCAR_QK_STEP(7)
#undef OSCAR_QK_STEP
  }

#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    // logits of tokens (g, g + 8): F * sum_g scale_g * acc_g + sum_g zero_g * qsum_g
    float2 sc[NP];
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      float2 A[NG];
#pragma unroll
      for (int gg = 0; gg < NG; ++gg)
        A[gg] = make_float2(acc[pg][nt][gg][0] + acc[pg][nt][gg][1], acc[pg][nt][gg][2] + acc[pg][nt][gg][3]);
      float2 X = f2mul(sk[pg][0], A[0]);
      float2 Z = f2mul(zk[pg][0], make_float2(qs[nt][0], qs[nt][0]));
      if (NG == 2) {
        X = f2fma(sk[pg][NG - 1], A[NG - 1], X);
        Z = f2fma(zk[pg][NG - 1], make_float2(qs[nt][NG - 1], qs[nt][NG - 1]), Z);
      }
      float2 a = f2fma(make_float2(F[nt], F[nt]), X, Z);
      if (!FULL) {
        a.x = v0[nt][pg] ? a.x : -INFINITY;
        a.y = v1[nt][pg] ? a.y : -INFINITY;
      }
      sc[pg] = a;
    }
    float mx = NP == 2 ? fmaxf(fmax3(sc[0].x, sc[0].y, sc[NP - 1].x), sc[NP - 1].y) : fmaxf(sc[0].x, sc[0].y);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float m_new = fmaxf(m_run[nt], mx);
    if (__any_sync(0xffffffffu, m_new > m_run[nt])) {
      const float alpha = m_run[nt] == -INFINITY ? 0.f : fast_exp2(m_run[nt] - m_new);
      const float2 al = make_float2(alpha, alpha);
      l_run[nt] = f2mul(l_run[nt], al);
#pragma unroll
      for (int gg = 0; gg < NG; ++gg) zacc[nt][gg] = f2mul(zacc[nt][gg], al);
#pragma unroll
      for (int mi = 0; mi < 8; ++mi)
#pragma unroll
        for (int c = 0; c < 4; ++c) O[nt][mi][c] *= alpha;
      m_run[nt] = m_new;
    }
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      float2 pr = f2sub(sc[pg], make_float2(m_new, m_new));
      pr.x = fast_exp2(pr.x);
      pr.y = fast_exp2(pr.y);
      if (!FULL) {
        pr.x = v0[nt][pg] ? pr.x : 0.f;
        pr.y = v1[nt][pg] ? pr.y : 0.f;
      }
      l_run[nt] = f2add(l_run[nt], pr);
      uint32_t bp[NG][2];
#pragma unroll
      for (int gg = 0; gg < NG; ++gg) {
        float2 q = f2mul(pr, sv[pg][gg]);
        if (FULL) {
          zacc[nt][gg] = f2fma(pr, zv[pg][gg], zacc[nt][gg]);
        } else {  // masked tokens may hold any bits: never multiply them in
          float2 z = f2mul(pr, zv[pg][gg]);
          q.x = v0[nt][pg] ? q.x : 0.f;
          q.y = v1[nt][pg] ? q.y : 0.f;
          z.x = v0[nt][pg] ? z.x : 0.f;
          z.y = v1[nt][pg] ? z.y : 0.f;
          zacc[nt][gg] = f2add(zacc[nt][gg], z);
        }
        // fp16 hi + lo of each weight, (hi, lo) of a token in one register
        const float2 hf = __half22float2(__floats2half2_rn(q.x, q.y));
        const float2 d = f2sub(q, hf);
        bp[gg][0] = movmatrix_trans(h2_bits(__floats2half2_rn(hf.x, d.x)));
        bp[gg][1] = movmatrix_trans(h2_bits(__floats2half2_rn(hf.y, d.y)));
      }
      // PV: m-tile mi covers channels 16*word + 8*(g&1) + 2*(mi&3) + {0 (row g), 1 (row g+8)},
      // word = g/2 for mi < 4 and 4 + g/2 for mi >= 4.
      const uint32_t xas[2] = {xa[pg][0] >> 10, xa[pg][1] >> 10}, xbs[2] = {xb[pg][0] >> 10, xb[pg][1] >> 10};
#define OSCAR_PV_TILE(MI)                                                                          \
  {                                                                                                \
    constexpr int hw = (MI) >> 2;                                                                  \
    constexpr int gg = (MI) * NG / 8;                                                              \
    constexpr int e = 2 * ((MI) & 3);                                                              \
    mma16816(O[nt][MI], extract_pair<e>(xa[pg][hw], xas[hw]), extract_pair<e + 1>(xa[pg][hw], xas[hw]), \
             extract_pair<e>(xb[pg][hw], xbs[hw]), extract_pair<e + 1>(xb[pg][hw], xbs[hw]), bp[gg][0], \
             bp[gg][1]);                                                                           \
  }
      OSCAR_PV_TILE(0) OSCAR_PV_TILE(1) OSCAR_PV_TILE(2) OSCAR_PV_TILE(3)
      OSCAR_PV_TILE(4) OSCAR_PV_TILE(5) OSCAR_PV_TILE(6) OSCAR_PV_TILE(7)
#undef OSCAR_PV_TILE
    }
  }
}

// ---- BF16 sink / window part ---------------------------------------------------

// Dense pages [first, first + count) of (b, h): the BF16 sink and recent-window rows on tensor cores,
// unrotated (the query is q itself).  The rows of (b, K|V, h) form 16-row pages:
// sink pages cover positions [16k, 16k + 16), window pages ring slots
// [16k', 16k' + 16); page k < ceil(S/16) is a sink page.  A sink row is attended
// when its position is below min(S, L); window slot r holds position
// L - 1 - ((L - 1 - r) mod W), attended when that position is at least S (the
// sink wins on overlap).  Rows that are not attended are not read: the warp
// zeroes them in shared memory so that p = 0 never meets stale bits.
// NW warps take the pages in turn (warp w: first + w, first + w + NW, ...), one
// 16-row stage of bf16pg::kStageBytes each at the start of `smem`, NW mbarriers
// after the stages; the CTA's (max, sum, output) partial goes to split s.
template <int NT, int NW>
__device__ __forceinline__ void dense_part(const Params& p, int first, int count, int s, int h, int b,
                                          uint8_t* smem) {
  constexpr int kDenseStage = bf16pg::kStageBytes;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int gqa = p.gqa;
  const size_t bh0 = static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * gqa;
  grid_dep_launch_dependents();
  grid_dep_wait();  // the sink/window rows may come from the preceding kernel (an append)
  const RowView rv = row_view(p, b);
  const int L = rv.L, A = rv.A, bs = rv.seq;
  const int nsp = (p.S + kPageSize - 1) / kPageSize, nwp = (p.W + kPageSize - 1) / kPageSize;
  const int cnt = max(0, min(count, nsp + nwp - first));
  const int sink_end = min(min(p.S, L), A);  // attended sink positions
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NW * kDenseStage);
  if (lane == 0) mbar_init(smem_u32(&bars[warp]), 1);
  mbar_init_fence();
  __syncthreads();

  const int n_my = cnt > warp ? (cnt - warp + NW - 1) / NW : 0;
  const uint32_t st = smem_u32(smem + warp * kDenseStage);
  const uint32_t bar = smem_u32(&bars[warp]);
  const int kv = lane >> 4, r = lane & 15;  // lane r: K row r (r < 16) or V row r - 16
  const uint32_t dst = st + bf16pg::stage_row(lane) * bf16pg::kRowPitch;
  // Whole warp: bring dense page `i` of this warp into the stage; returns the
  // mask of attended rows (bit r for token r).
  auto issue = [&](int i) -> uint32_t {
    const int k = first + warp + i * NW;
    const __nv_bfloat16* src = nullptr;
    if (k < nsp) {
      const int pos = k * kPageSize + r;
      if (pos < sink_end)
        src = p.sink + (((static_cast<size_t>(bs) * 2 + kv) * p.H + h) * p.S + pos) * kD;
    } else {
      const int slot = (k - nsp) * kPageSize + r;
      if (slot < p.W && L > 0) {
        int back = (L - 1 - slot) % p.W;
        if (back < 0) back += p.W;
        const int wpos = L - 1 - back;  // the position the ring slot holds
        if (wpos >= p.S && wpos < A)
          src = p.win + (((static_cast<size_t>(bs) * 2 + kv) * p.H + h) * p.W + slot) * kD;
      }
    }
    const uint32_t mask = __ballot_sync(0xffffffffu, src != nullptr);
    if (src == nullptr) {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int c = 0; c < bf16pg::kRowBytes / 16; ++c)
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst + 16 * c), "r"(z.x), "r"(z.y), "r"(z.z),
                     "r"(z.w)
                     : "memory");
    }
    // this lane's generic writes (zeros, earlier reads) before its next bulk copy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      const uint32_t bytes = static_cast<uint32_t>(__popc(mask)) * bf16pg::kRowBytes;
      if (bytes) mbar_arrive_expect_tx(bar, bytes);
      else mbar_arrive(bar);
    }
    __syncwarp();
    if (src != nullptr) bulk_g2s(dst, src, bf16pg::kRowBytes, bar);
    return mask & 0xffffu;  // K rows (lanes 0..15) and V rows share the mask
  };
  uint32_t mask = n_my > 0 ? issue(0) : 0u;

  uint32_t bq[NT][8][2];
  bf16pg::build_bq<NT>(p.q + bh0 * kD, p.scale_log2, gqa, g, t, bq);
  float m_run[NT], l_run[NT], O[NT][8][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt] = -INFINITY;
    l_run[nt] = 0.f;
#pragma unroll
    for (int mi = 0; mi < 8; ++mi)
#pragma unroll
      for (int c = 0; c < 4; ++c) O[nt][mi][c] = 0.f;
  }
  const bf16pg::LaneOffsets lo = bf16pg::lane_offsets(lane);
  bool aborted = false;
  int i = 0;
  for (; i < n_my; ++i) {
    if (__any_sync(0xffffffffu, !mbar_wait_bounded(bar, i & 1))) {
      aborted = true;
      break;
    }
    __syncwarp();  // zeroed rows of other lanes are visible
    bf16pg::page<NT>(st, lo, g, (mask >> g) & 1u, (mask >> (g + 8)) & 1u, bq, m_run, l_run, O);
    __syncwarp();
    if (i + 1 < n_my) mask = issue(i + 1);
  }
  if (aborted) {
    if (lane == 0) record_error(OSCAR_DEVERR_TIMEOUT);
    // the one copy in flight (page i) may still land: wait for it (bounded) before
    // the stage area is reused
    mbar_wait_bounded(bar, i & 1);
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
  float* lw = mw + NW * kMaxGqa;
  float* ow = lw + NW * kMaxGqa;
  bf16pg::store_warp<NT>(O, m_run, l_run, mw, lw, ow, warp, g, t, gqa);
  __syncthreads();
  merge_warps_store<NW, kD, NW * 32>(p, mw, lw, ow, s, bh0, tid);
}

}  // namespace
}  // namespace oscar_dec
