// BF16 tensor-core page body shared by the all-BF16 paged reference decode and
// the BF16 sink/window part of the OSCAR decode ("OSCAR: Offline Spectral
// Covariance-Aware Rotation for 2-bit KV Cache Quantization", project card
// "How it works": sink and recent window kept in BF16).
//
// A page is 16 tokens of one KV head at head_dim 128: 16 K rows then 16 V rows
// of 256 bytes, staged in shared memory with a 272-byte pitch (ldmatrix reads
// are then bank-conflict free).  V token v sits in stage row 16 + 2*(v%8) + v/8
// so that one transposed ldmatrix reads 8 consecutive rows.
//   QK:  S^T[token][query] = K[token][ch] . Q[ch][query], A from ldmatrix,
//        B = q * scale * log2(e) split into bf16 hi + lo (16 significant bits);
//   online softmax per query with warp shuffles;
//   PV:  O^T[ch][query] += V^T[ch][token] . P[token][query], A from
//        ldmatrix.trans, B = p split into bf16 hi + lo.
// Per n-tile nt a lane's C columns belong to query 4*nt + t (hi and lo parts in
// columns 2t, 2t+1), its B column to query 4*nt + g/2, part g%2.
#pragma once

#include "decode_common.cuh"

namespace oscar_dec {
namespace {
namespace bf16pg {

constexpr int kD = 128;
constexpr int kRowBytes = kD * 2;            // one token row of K or V
constexpr int kRowPitch = kRowBytes + 16;    // padded row in shared memory
constexpr int kStageBytes = 32 * kRowPitch;  // 16 K rows then 16 V rows

// Stage row of K token r (r < 16) or V token r - 16 (r >= 16).
__device__ __forceinline__ int stage_row(int r) { return r < 16 ? r : 16 + 2 * ((r - 16) & 7) + ((r - 16) >> 3); }

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

// QK B fragments from the bf16 queries of one KV head (qb: query 0 of the
// head's GQA group): k-step ks, rows 2t, 2t+1 -> channels 16 ks + 2t, +1; rows
// 2t+8, 2t+9 -> 16 ks + 2t + 8, +9; column g -> query g/2, part g%2.
template <int NT>
__device__ __forceinline__ void build_bq(const __nv_bfloat16* qb, float scale_log2, int gqa, int g, int t,
                                         uint32_t (&bq)[NT][8][2]) {
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
        const float x = use ? __bfloat162float(qb[qi * kD + ch]) * scale_log2 : 0.f;
        __nv_bfloat16 hi, lo;
        split_bf16(x, hi, lo);
        v[c] = lo_part ? lo : hi;
      }
      bq[nt][ks][0] = pack_bf16x2(v[0], v[1]);
      bq[nt][ks][1] = pack_bf16x2(v[2], v[3]);
    }
  }
}

// Per-lane ldmatrix offsets inside a stage.  K (non-transposed): matrix lm =
// lane/8 covers tokens 8*(lm&1) .. +7 and channels 8*(lm>>1) .. +7 of a k-step.
// V (transposed): the k index of PV is a token order chosen so that the two
// tokens of a B register (k = 2t', 2t'+1) are tokens t', t'+8 and (k = 2t'+8,
// 2t'+9) are t'+4, t'+12, which is how the softmax fragments already pair them;
// with the V row placement of stage_row, row lr of matrix lm is stage row
// 16 + lr + 8*(lm>>1).
struct LaneOffsets {
  uint32_t k_off, v_off;
  int src1, src2;
};

__device__ __forceinline__ LaneOffsets lane_offsets(int lane) {
  const int g = lane >> 2, t = lane & 3, lr = lane & 7, lm = lane >> 3;
  LaneOffsets o;
  o.k_off = (lr + 8 * (lm & 1)) * kRowPitch + 8 * (lm >> 1) * 2;
  o.v_off = (16 + lr + 8 * (lm >> 1)) * kRowPitch + 8 * (lm & 1) * 2;
  o.src1 = 4 * t + (g >> 1);
  o.src2 = o.src1 + 16;
  return o;
}

// One staged page: QK, online softmax (v0 / v1: this lane's tokens g and g + 8
// are attended), PV.  Masked tokens get p = 0; their V rows must hold finite
// values (the callers copy or zero every row).
template <int NT>
__device__ __forceinline__ void page(uint32_t st, const LaneOffsets& lo, int g, bool v0, bool v1,
                                     const uint32_t (&bq)[NT][8][2], float (&m_run)[NT], float (&l_run)[NT],
                                     float (&O)[NT][8][4]) {
  const uint32_t kbase = st + lo.k_off, vbase = st + lo.v_off;
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
    const uint32_t h_1 = __shfl_sync(0xffffffffu, xhi, lo.src1), l_1 = __shfl_sync(0xffffffffu, xlo, lo.src1);
    const uint32_t h_2 = __shfl_sync(0xffffffffu, xhi, lo.src2), l_2 = __shfl_sync(0xffffffffu, xlo, lo.src2);
    const uint32_t bp0 = (g & 1) ? l_1 : h_1, bp1 = (g & 1) ? l_2 : h_2;
#pragma unroll
    for (int mi = 0; mi < 8; ++mi) {
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4_trans(vbase + mi * 32, a0, a1, a2, a3);
      mma_bf16(O[nt][mi], a0, a1, a2, a3, bp0, bp1);
    }
  }
}

// Writes a warp's state to the CTA's merge area: m and l per query and the
// unnormalised output (m-tile mi holds channels 16 mi + g and 16 mi + g + 8).
template <int NT>
__device__ __forceinline__ void store_warp(const float (&O)[NT][8][4], const float (&m_run)[NT],
                                           const float (&l_run)[NT], float* mw, float* lw, float* ow, int warp,
                                           int g, int t, int gqa) {
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
        ow[(warp * kMaxGqa + qi) * kD + 16 * mi + g] = O[nt][mi][0] + O[nt][mi][1];
        ow[(warp * kMaxGqa + qi) * kD + 16 * mi + g + 8] = O[nt][mi][2] + O[nt][mi][3];
      }
    }
  }
}

}  // namespace bf16pg

// Log-sum-exp merge of the NW warps' states in shared memory (mw, lw:
// [NW][kMaxGqa]; ow: [NW][kMaxGqa][D]) into the CTA's split partial s.  Called
// by every thread of the CTA (NTHREADS); mw is overwritten with the warps'
// weights 2^(m_w - M).
template <int NW, int D, int NTHREADS>
__device__ __forceinline__ void merge_warps_store(const Params& p, float* mw, const float* lw, const float* ow,
                                                  int s, size_t bh0, int tid) {
  const int gqa = p.gqa;
  if (tid < gqa) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mw[w * kMaxGqa + tid]);
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mwq = mw[w * kMaxGqa + tid];
      const float wt = (M == -INFINITY || mwq == -INFINITY) ? 0.f : fast_exp2(mwq - M);
      l = fmaf(wt, lw[w * kMaxGqa + tid], l);
      mw[w * kMaxGqa + tid] = wt;
    }
    p.part_ml[((bh0 + tid) * p.ml_ns + s) * 2 + 0] = M;
    p.part_ml[((bh0 + tid) * p.ml_ns + s) * 2 + 1] = l;
  }
  __syncthreads();
  for (int idx = tid; idx < gqa * (D / 4); idx += NTHREADS) {
    const int qi = idx / (D / 4), c4 = idx % (D / 4);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float wt = mw[w * kMaxGqa + qi];
      if (wt != 0.f) {
        const float4 v = reinterpret_cast<const float4*>(ow + (w * kMaxGqa + qi) * D)[c4];
        o.x = fmaf(wt, v.x, o.x); o.y = fmaf(wt, v.y, o.y); o.z = fmaf(wt, v.z, o.z); o.w = fmaf(wt, v.w, o.w);
      }
    }
    reinterpret_cast<float4*>(p.part_o + ((bh0 + qi) * p.ns + s) * D)[c4] = o;
  }
}

}  // namespace
}  // namespace oscar_dec
