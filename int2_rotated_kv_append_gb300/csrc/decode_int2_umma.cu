// Extend (chunked prefill) in tiles on the fifth-generation tensor cores: the
// INT2 bulk of the query rows of one sequence, 64 query columns per CTA
// ("OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
// Quantization", abstract: INT2 attention kernel over a paged KV cache; project
// card "How it works": fused mixed-precision attention over the quantised cache).
//
// Shape covered: head_dim 128, group 64 or 128, GQA 4 or 8.  One CTA of 16 warps per
// (INT2 split, KV head, sequence x tile of rows); a tile holds 64 query columns (16
// rows of GQA 4 or 8 rows of GQA 8).  The split's pages go through in chunks of 8
// (128 tokens), staged by bulk async copies in a ring of two chunks:
//   * expansion: the chunk's K and V codes become fp16 operands in shared memory,
//     once per CTA.  The 2-bit code at bit position k of an fp16 half is the exact
//     subnormal c * 2^(k-24), taken with one AND per pair of codes; a 32-bit word
//     holds channels (j, j + 8) of a 16-channel word, so the K (and M) index runs
//     through the channels in that order (both operands use it);
//   * QK: S^T[token][column] = C_k[token][.] . Q[column][.] on tcgen05 with M = 128
//     tokens and N = 128 (the 64 columns' fp16 high parts, then their low parts),
//     one TMEM accumulator per group.  Q holds q.R_k * sm_scale * log2(e) *
//     2^(E - k) per channel (E one exponent for the tile, from the largest |q|), so
//     every code x query product is exact;
//   * softmax, one thread per (token, 16 columns): logits scale_g * 2^(24 - E) *
//     acc_g + zero_g * sum_{ch in g} q (log2 units); weights 2^(s - m) against the
//     running maxima, which are taken anew (a warp butterfly, then shared memory)
//     only when a logit exceeds them by more than 8; P'_g = p * scale_g split into
//     fp16 high and low parts, written as the B operand of the PV product;
//   * PV: O_g^T[channel][column] += C_v^T . P'_g on tcgen05 with M = 128 channels,
//     N = 128 (high, low parts), one TMEM accumulator per group (the rows of the
//     other group's channels are not read); O is rescaled in TMEM when a maximum
//     moves;
//   * the sums of p and of p * zero_g per column are kept per thread and reduced
//     once; the CTA writes one (max, sum, output) partial per column, the output in
//     rotated space, exactly as the decode's splits do.
// Pipelining: the K side of chunk c + 1 (page wait, K codes expanded, V codes set
// aside so the page's stage is refilled at once) follows the logits of c; after one
// barrier a thread of warp 13 issues QK(c + 1) while the warps finish c; after a
// second barrier threads of warps 14 and 15 issue the PV products of c, one per
// group, and warp 12 requests pages two chunks ahead.  Single threads issuing many
// MMAs fall behind the other warps, so the issue is spread and the MMAs kept large.
#include <math.h>

#include <mutex>

#include "int2_page.cuh"
#include "umma.cuh"

namespace oscar_dec {
namespace {

constexpr int kUtThreads = 512;               // 16 warps
constexpr int kUtQkIssuer = 13 * 32;          // the thread that issues the QK products (warp 13)
constexpr int kUtPvIssuer = 14 * 32;          // group g's PV products: thread kUtPvIssuer + 32 g (warps 14, 15)
constexpr int kUtFetchWarp = 12;              // its lanes request the pages
constexpr int kUtTok = 128;                   // tokens per chunk
constexpr int kUtPages = kUtTok / kPageSize;  // pages per chunk
constexpr int kUtRing = 2 * kUtPages;         // staged pages: two chunks
constexpr int kUtCols = 64;                   // query columns per tile
constexpr int kUtMaxPps = 256;                // page ids of one split staged in shared memory
constexpr uint32_t kUtBlock = 128 * 128;      // one operand block: 128 rows of 128 bytes (16 KB)
constexpr float kLazy = 12.f;                 // a running maximum is kept while logits stay below it + kLazy
constexpr float kLazyScale = 15.f;            // ... and V scales at most this: 2^kLazy * 15 < 65504 (fp16)

// Shared-memory layout (offsets from a 1024-byte aligned base).
template <int NG>
struct UtGeo {
  static constexpr uint32_t kStage = PageGeo<NG>::kStageBytes;
  static constexpr uint32_t kAK = 0;                                   // K codes, K-major, 2 K blocks
  static constexpr uint32_t kAV = kAK + 2 * kUtBlock;                  // V codes, MN-major
  static constexpr uint32_t kVb1 = kUtBlock;                          // channels 64..127
  static constexpr uint32_t kBq = kAV + 2 * kUtBlock;                  // query operand, K-major, 2 K blocks
  static constexpr uint32_t kBp = kBq + 2 * kUtBlock;                  // P' per group, MN-major (high, low)
  static constexpr uint32_t kRing = kBp + NG * 2 * kUtBlock;           // staged pages
  static constexpr uint32_t kTok = kRing + kUtRing * kStage;           // per token (scale, zero): K x 2, V x 2
  static constexpr uint32_t kVraw = kTok + kUtTok * 4 * NG * 4;        // V codes of two chunks (32 B per token)
  static constexpr uint32_t kCol = kVraw + 2 * kUtTok * 32;            // per-column values
  // m_run, m_use, alpha, attend bound | qs[NG] | reductions [3][4] | sums [1 + NG]
  static constexpr int kColFloats = 64 * (4 + NG + 12 + 1 + NG);
  static constexpr uint32_t kBars = kCol + kColFloats * 4;
  static constexpr int kNumBars = kUtRing + 2 + NG;  // page ring | QK done | never completed | PV done per group
  static constexpr uint32_t kPid = kBars + kNumBars * 8;
  static constexpr uint32_t kMisc = kPid + kUtMaxPps * 4;  // TMEM address, largest |q|, rescale flags, abort flag
  static constexpr size_t kSmem = 1024 + kMisc + 32;  // misc: TMEM address, max |q|, 4 rescale flags, abort
  static constexpr uint32_t kTmemCols = NG == 2 ? 512 : 256;  // NG QK accumulators, then NG O accumulators (128 each)
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Channels j and j + 8 of a 16-channel code word as two fp16 subnormals, at bit
// position code_kpos(j) (the word shifted right by 10 serves pairs 5..7).
__device__ __forceinline__ uint32_t code_pair(uint32_t w, uint32_t wsh, int j) {
  return j <= 4 ? (w & (0x00030003u << (2 * j))) : (wsh & (0x00030003u << (2 * j - 10)));
}

// Two 16-channel code words (words i0, i0 + 1 of channels 64 b .. 64 b + 63) of one
// token into row t of a 128-row operand block with the 128-byte swizzle: pair j of
// word i is the 32-bit slot j % 4 of 16-byte chunk 2 i + j / 4.
__device__ __forceinline__ void expand_row(uint32_t blk, int t, int i0, const uint32_t (&wd)[2]) {
#pragma unroll
  for (int ii = 0; ii < 2; ++ii) {
    const int i = i0 + ii;
    const uint32_t w = wd[ii], wsh = w >> 10;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int q = 2 * i + hf;
      st_shared_v4(blk + t * 128 + ((q ^ (t & 7)) << 4), code_pair(w, wsh, 4 * hf), code_pair(w, wsh, 4 * hf + 1),
                   code_pair(w, wsh, 4 * hf + 2), code_pair(w, wsh, 4 * hf + 3));
    }
  }
}

// Column reduction (max or sum) of the 32 x 16 values of a warp (lane = row, all
// lanes with the same 16 columns): afterwards lanes l and l + 16 hold the reduction of
// column l % 16.  Lanes l and l ^ 16 are combined first, then a transposing butterfly
// over the 16 lanes halves the values held per lane at each step.
template <bool MAX>
__device__ __forceinline__ float warp_cols16(float (&v)[16], int lane) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float o = __shfl_xor_sync(0xffffffffu, v[j], 16);
    v[j] = MAX ? fmaxf(v[j], o) : v[j] + o;
  }
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = up ? v[i] : v[i + o];
      const float keep = up ? v[i + o] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

template <int NG>
__global__ void __launch_bounds__(kUtThreads, 1) int2_umma_tile_kernel(Params p) {
  using Geo = UtGeo<NG>;
  extern __shared__ uint8_t ut_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ut_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  float* m_run = reinterpret_cast<float*>(sm + Geo::kCol);  // running maximum per column
  float* m_use = m_run + 64;                                // maximum used for the weights (0 when -inf)
  float* alpha = m_use + 64;                                // rescale of the previous chunks
  int* r1c = reinterpret_cast<int*>(alpha + 64);            // attended bound per column (exclusive)
  float* qs = reinterpret_cast<float*>(r1c + 64);           // [NG][64]: sum over the group of q * scale
  float* red = qs + NG * 64;                                // [3][4][64]: per-warp partial reductions
  float* fin = red + 3 * 4 * 64;                            // [1 + NG][64]: sum of p, sums of p * zero_g
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Geo::kBars);
  int* pid_all = reinterpret_cast<int*>(sm + Geo::kPid);
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + Geo::kMisc);
  const uint32_t bar_s = smem_u32(&bars[kUtRing]), bar_never = smem_u32(&bars[kUtRing + 1]);
  auto bar_o = [&](int g) { return smem_u32(&bars[kUtRing + 2 + g]); };
  auto full = [&](int k) { return smem_u32(&bars[k % kUtRing]); };

  const int s = blockIdx.x, h = blockIdx.y;
  const int b = blockIdx.z / p.tiles, tile = blockIdx.z % p.tiles;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gqa = p.gqa;  // 4 or 8
  const int rpt = kUtCols / gqa;
  grid_dep_launch_dependents();
  // the rotated queries come from the q-rotation, the pages from appends before it
  grid_dep_wait();
  const int q0 = __ldg(p.q_start + b), q1 = __ldg(p.q_start + b + 1);
  const int r_begin = q0 + tile * rpt;
  if (r_begin >= q1) return;  // no rows in this tile
  const int n_rows = min(rpt, q1 - r_begin);
  const int L = clamp_len(p, b);
  const int win_begin = max(p.S, L - p.W);
  const int lo_pos = s * p.pps * kPageSize, hi_pos = lo_pos + p.pps * kPageSize;
  const int r0 = max(lo_pos, p.S);
  // positions [0, A) of a row, clipped to this split's part of the bulk
  auto attend_end = [&](int row) {
    const int pos = __ldg(p.row_pos + row);
    const int A = (pos >= 0 && pos < L) ? pos + 1 : 0;
    return min(hi_pos, min(win_begin, A));
  };
  auto col_valid = [&](int c) { return c / gqa < n_rows; };
  auto col_bh = [&](int c) { return static_cast<size_t>(r_begin + c / gqa) * p.Hq + h * gqa + c % gqa; };
  // the tile's range: its last row has the largest position
  const int r1_tile = attend_end(r_begin + n_rows - 1);
  if (tid < n_rows) {  // a row outside its sequence attends nothing and is flagged
    const int pos = __ldg(p.row_pos + r_begin + tid);
    if (pos < 0 || pos >= L) record_error(OSCAR_DEVERR_POSITION);
  }
  if (r1_tile <= r0) {  // nothing of the bulk: empty partials for every column of the tile
    if (tid < kUtCols && col_valid(tid)) {
      const size_t bh = col_bh(tid);
      p.part_ml[(bh * p.ml_ns + s) * 2 + 0] = -INFINITY;
      p.part_ml[(bh * p.ml_ns + s) * 2 + 1] = 0.f;
    }
    return;
  }
  const int pg0 = r0 / kPageSize;
  const int npg = (r1_tile - 1) / kPageSize + 1 - pg0;  // <= pps <= kUtMaxPps
  const int nchunks = (npg + kUtPages - 1) / kUtPages;
  for (int k = tid; k < npg; k += kUtThreads)
    pid_all[k] = __ldg(p.page_table + static_cast<size_t>(b) * p.max_pages + pg0 + k);
  if (tid < kUtCols) {
    r1c[tid] = col_valid(tid) ? attend_end(r_begin + tid / gqa) : 0;
    m_run[tid] = -INFINITY;
  }
  if (tid == 0) {
    for (int i = 0; i < Geo::kNumBars; ++i) mbar_init(smem_u32(&bars[i]), 1);
    misc[1] = 0u;
    misc[6] = 0u;  // abort flag
    mbar_init_fence();
  }
  if (warp == 0) umma::tmem_alloc(smem_u32(&misc[0]), Geo::kTmemCols);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = misc[0];

  auto pid_ok = [&](int k) {
    const int pid = pid_all[k];
    return pid >= 0 && pid < p.num_pages;
  };
  // one thread: page k of the range into stage k % kUtRing
  auto issue = [&](int k) {
    const int pid = pid_all[k];
    const uint32_t bar = full(k);
    if (pid < 0 || pid >= p.num_pages) {
      record_error(OSCAR_DEVERR_PAGE_ID);
      mbar_arrive(bar);
      return;
    }
    const size_t ph = static_cast<size_t>(pid) * p.H + h;
    const uint32_t dst = sb + Geo::kRing + (k % kUtRing) * Geo::kStage;
    mbar_arrive_expect_tx(bar, Geo::kStage);
    bulk_g2s(dst, p.codes + ph * kCodeBytes, kCodeBytes, bar);
    bulk_g2s(dst + kCodeBytes, reinterpret_cast<const uint8_t*>(p.sz) + ph * PageGeo<NG>::kSzBytes,
             PageGeo<NG>::kSzBytes, bar);
  };
  // pages requested so far and MMA chains committed (the same in every thread)
  int issued = min(npg, kUtRing), qk_issued = 0, pv_issued = 0;
  if (warp == kUtFetchWarp && lane < issued) issue(lane);

  // ---- query operand: per (column, quarter of the channels) sum and largest |q| ----
  const float sl = p.scale_log2;
  {
    const int c = tid >> 3, qq = tid & 7;
    float sum = 0.f, mx = 0.f;
    if (col_valid(c)) {
      const float4* src = reinterpret_cast<const float4*>(p.q_rot + col_bh(c) * kD + 16 * qq);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 v = __ldg(src + i);
        sum += (v.x + v.y) + (v.z + v.w);
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
      }
    }
    red[qq * 64 + c] = sum;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) atomicMax(reinterpret_cast<int*>(&misc[1]), __float_as_int(mx));
  }
  __syncthreads();
  if (tid < kUtCols) {
    const float* r8 = red + tid;  // 8 blocks of 16 channels, 64 apart
    const float s0 = (r8[0] + r8[64]) + (r8[128] + r8[192]), s1 = (r8[256] + r8[320]) + (r8[384] + r8[448]);
    if constexpr (NG == 2) {
      qs[tid] = s0 * sl;
      qs[64 + tid] = s1 * sl;
    } else {
      qs[tid] = (s0 + s1) * sl;
    }
  }
  // E: every |q * scale| * 2^(E - kpos) < 2^15, so the fp16 high part cannot overflow
  int E = 15;
  {
    const float bound = __int_as_float(static_cast<int>(misc[1])) * fabsf(sl) * (1.f + 1.f / 1024.f);
    int e = 0;
    if (bound > 0.f) frexpf(bound, &e);
    E = min(max(15 - e, -100), 100);
  }
  const float F = pow2i(24 - E);
  // rows 0..63: the columns' fp16 high parts; rows 64..127: the low parts
  for (int idx = tid; idx < kUtCols * 64; idx += kUtThreads) {
    const int c = idx >> 6, pi = idx & 63, w = pi >> 3, j = pi & 7;
    uint32_t hi = 0u, lo = 0u;
    if (col_valid(c)) {
      const float* src = p.q_rot + col_bh(c) * kD + 16 * w + j;
      const float sc = sl * pow2i(E - code_kpos(j));
      const float x0 = __ldg(src) * sc, x1 = __ldg(src + 8) * sc;
      const __half2 hh = __floats2half2_rn(x0, x1);
      const float2 hf = __half22float2(hh);
      const __half2 ll = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
      hi = *reinterpret_cast<const uint32_t*>(&hh);
      lo = *reinterpret_cast<const uint32_t*>(&ll);
    }
    const int kk = 16 * w + 2 * j;
    st_shared_b32(sb + Geo::kBq + umma::sw128_offset(c, kk, 128), hi);
    st_shared_b32(sb + Geo::kBq + umma::sw128_offset(64 + c, kk, 128), lo);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // query operand visible to the tensor cores
  __syncthreads();

  const int q4 = warp & 3, hq = warp >> 2;  // TMEM lanes 32 q4 .. + 31; columns 16 hq .. + 15
  const int tr = 32 * q4 + lane;            // token row of the softmax; channel row of O
  const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * q4) << 16);
  // O row tr holds channel ch_tr (codes at bit position code_kpos(ch_tr)), in the
  // accumulator of its group
  const int ch_tr = 16 * (tr >> 4) + ((tr & 15) >> 1) + 8 * (tr & 1);
  const uint32_t o_col = NG * 128 + (NG == 2 ? (ch_tr >> 6) * 128 : 0);
  int r1_min = hi_pos;  // below it no column needs a causal mask
  for (int c = 0; c < kUtCols; ++c)
    if (col_valid(c)) r1_min = min(r1_min, r1c[c]);
  // per-thread column sums (pairs of columns): of p, and of p * zero_g
  float2 l2[8], z2[NG][8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    l2[j] = make_float2(0.f, 0.f);
#pragma unroll
    for (int g = 0; g < NG; ++g) z2[g][j] = make_float2(0.f, 0.f);
  }
  // expansion: thread (row xr, code words 2 xq, 2 xq + 1) of a chunk
  const int xr = tid & 127, xq = tid >> 7;
  uint32_t* tokK = reinterpret_cast<uint32_t*>(sm + Geo::kTok);  // [2][128][NG]: K (scale, zero) by chunk parity
  uint32_t* tokV = tokK + 2 * kUtTok * NG;                       // [2][128][NG]: V (scale, zero) by chunk parity
  uint8_t* vraw = sm + Geo::kVraw;                               // [2][128][32 B]: V codes by chunk parity
  volatile int* need_rs = reinterpret_cast<volatile int*>(&misc[2]);  // [4]: a column quarter's O needs rescaling
  auto stage_of = [&](int k) { return sm + Geo::kRing + (k % kUtRing) * Geo::kStage; };
  // The K side of chunk c: wait for the row's page, expand its K codes into the K
  // operand, keep the token's K and V (scale, zero).  False if the wait gave up.
  auto k_side = [&](int c) {
    const int k = c * kUtPages + (xr >> 4);
    bool ok = true;
    if (k < npg) {
      // under oscar_test_stall_page_waits the first chunk waits on a barrier nothing completes
      ok = (p.stall_cycles > 0 && c == 0) ? mbar_wait_bounded(bar_never, 0, p.stall_cycles)
                                          : mbar_wait_bounded(full(k), (k / kUtRing) & 1);
    }
    const bool have = ok && k < npg && pid_ok(k);
    const uint8_t* st = stage_of(k);
    uint32_t wd[2] = {0u, 0u};
    uint2 vw = make_uint2(0u, 0u);
    if (have) {
      const uint2 v = *reinterpret_cast<const uint2*>(st + (xr & 15) * 32 + 8 * xq);
      wd[0] = v.x, wd[1] = v.y;
      vw = *reinterpret_cast<const uint2*>(st + 512 + (xr & 15) * 32 + 8 * xq);
    }
    // the V codes wait in the side buffer, so the page's stage can be refilled at once
    *reinterpret_cast<uint2*>(vraw + ((c & 1) * kUtTok + xr) * 32 + 8 * xq) = vw;
    expand_row(sb + Geo::kAK + (xq >> 1) * kUtBlock, xr, 2 * (xq & 1), wd);
    if (xq < 2) {
      uint32_t* dst = (xq == 0 ? tokK : tokV) + ((c & 1) * kUtTok + xr) * NG;
#pragma unroll
      for (int g = 0; g < NG; ++g)
        dst[g] = have ? *reinterpret_cast<const uint32_t*>(st + kCodeBytes + ((xq * 16 + (xr & 15)) * NG + g) * 4)
                      : 0u;
    }
    return ok;
  };
  // The V codes of chunk c (from the side buffer) into the V operand.
  auto v_side = [&](int c) {
    const uint2 v = *reinterpret_cast<const uint2*>(vraw + ((c & 1) * kUtTok + xr) * 32 + 8 * xq);
    const uint32_t wd[2] = {v.x, v.y};
    expand_row(sb + Geo::kAV + ((xq >> 1) ? Geo::kVb1 : 0u), xr, 2 * (xq & 1), wd);
  };
  // the issuing thread: QK of the chunk whose K operand is in place
  auto issue_qk = [&]() {
    umma::fence_after_sync();
    constexpr uint32_t idesc = umma::idesc_f16_f32(128, 128, false);
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int ks = 0; ks < 8 / NG; ++ks) {
        const int kk = g * (8 / NG) + ks;  // 16-channel step
        const uint32_t koff = (kk >> 2) * kUtBlock + (kk & 3) * 32;
        umma::mma_bf16(tmem + g * 128, umma::desc_k_sw128(sb + Geo::kAK + koff),
                       umma::desc_k_sw128(sb + Geo::kBq + koff), idesc, ks != 0);
      }
    umma::commit(bar_s);
  };
  // group g's issuing thread: PV of chunk c into O_g (accumulating from the first chunk
  // on; the rows of the other group's channels are not used)
  auto issue_pv = [&](int c, int g) {
    umma::fence_after_sync();
    constexpr uint32_t idesc = umma::idesc_f16_f32(128, 128, true);
    const uint32_t b0 = sb + Geo::kBp + g * 2 * kUtBlock;
#pragma unroll
    for (int ks = 0; ks < kUtTok / 16; ++ks)
      umma::mma_bf16(tmem + NG * 128 + g * 128, umma::desc_mn_sw128(sb + Geo::kAV + ks * 2048, kUtBlock),
                     umma::desc_mn_sw128(b0 + ks * 2048, kUtBlock), idesc, (c | ks) != 0);
    umma::commit(bar_o(g));
  };

  // Pipeline per chunk c: logits of c | K side of c + 1 (page wait, K codes expanded,
  // V codes set aside) | one barrier, then QK(c + 1) issued and the pages of c + 3
  // requested | (only when a maximum moves) exact column maxima | weights of c |
  // (PV(c - 1) done) P' of c, O rescaled, V codes of c expanded | one barrier, then
  // PV(c).  The tensor cores run PV(c - 1) and QK(c + 1) while the warps work on c.
  bool aborted = false;
  int k_ok_chunks = 0;  // chunks whose pages every thread has awaited
  volatile int* abort_flag = reinterpret_cast<volatile int*>(&misc[6]);
  // the pages of chunk c + 2, one page per lane of the fetch warp (their stages held chunk c)
  auto refill = [&](int c) {
    const int want = min(npg, (c + 3) * kUtPages);
    if (warp == kUtFetchWarp && issued + lane < want) issue(issued + lane);
    issued = max(issued, want);
  };
  {
    const bool ok = k_side(0);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (__syncthreads_or(!ok)) {
      aborted = true;
    } else {
      k_ok_chunks = 1;
      if (tid == kUtQkIssuer) issue_qk();
      qk_issued = 1;
      refill(0);
    }
  }
  int ci = 0;
  if (!aborted) {
    for (; ci < nchunks; ++ci) {
      // ---- logits of chunk ci: thread (token tr, columns 16 hq ..) ----
      const bool ok1 = mbar_wait_bounded(bar_s, ci & 1);
      umma::fence_after_sync();
      const int tk = ci * kUtPages + (tr >> 4);
      const int pos = (pg0 + tk) * kPageSize + (tr & 15);
      const bool tok_ok = tk < npg && pid_ok(tk) && pos >= r0 && pos < r1_tile;
      float sv[16];
      {
        const __half2* tk2 = reinterpret_cast<const __half2*>(tokK) + ((ci & 1) * kUtTok + tr) * NG;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          uint32_t hi[16], lo[16];
          umma::tmem_ld16(t_lane + g * 128 + 16 * hq, hi);
          umma::tmem_ld16(t_lane + g * 128 + 64 + 16 * hq, lo);
          umma::tmem_ld_wait();
          const float f = F * __low2float(tk2[g]);
          const float2 ag = make_float2(f, f);
#pragma unroll
          for (int jj = 0; jj < 16; jj += 2) {
            const float2 a = f2add(make_float2(__uint_as_float(hi[jj]), __uint_as_float(hi[jj + 1])),
                                   make_float2(__uint_as_float(lo[jj]), __uint_as_float(lo[jj + 1])));
            const float2 v = g == 0 ? f2mul(ag, a) : f2fma(ag, a, make_float2(sv[jj], sv[jj + 1]));
            sv[jj] = v.x;
            sv[jj + 1] = v.y;
          }
        }
        const float4* qs4 = reinterpret_cast<const float4*>(qs);
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const float z = __high2float(tk2[g]);
          const float2 zg = make_float2(z, z);
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            const float4 qv = qs4[g * 16 + 4 * hq + j4];
            const float2 a = f2fma(zg, make_float2(qv.x, qv.y), make_float2(sv[4 * j4], sv[4 * j4 + 1]));
            const float2 c2 = f2fma(zg, make_float2(qv.z, qv.w), make_float2(sv[4 * j4 + 2], sv[4 * j4 + 3]));
            sv[4 * j4] = a.x, sv[4 * j4 + 1] = a.y, sv[4 * j4 + 2] = c2.x, sv[4 * j4 + 3] = c2.y;
          }
        }
      }
      if (!tok_ok) {
#pragma unroll
        for (int j = 0; j < 16; ++j) sv[j] = -INFINITY;
      } else if (pos >= r1_min) {  // causal bounds inside the chunk
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (pos >= r1c[16 * hq + j]) sv[j] = -INFINITY;
      }
      // ---- the K side of chunk ci + 1 (QK(ci) has finished reading the K operand) ----
      bool ok2 = true;
      if (ci + 1 < nchunks) ok2 = k_side(ci + 1);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      // Lazy maxima: the chunk keeps the running maxima unless one of its logits exceeds
      // them by more than kLazy (weights up to 2^kLazy) or a V scale exceeds kLazyScale
      // (P' = p * scale would leave the fp16 range); then the maxima are taken exactly
      // and O is rescaled.  The partials carry the maxima used, so either way they are
      // exact.
      const __half2* tv2 = reinterpret_cast<const __half2*>(tokV) + ((ci & 1) * kUtTok + tr) * NG;
      bool over = false;
      {
        const float4* mr4 = reinterpret_cast<const float4*>(m_run + 16 * hq);
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          const float4 mr = mr4[j4];
          over |= (sv[4 * j4] > mr.x + kLazy) | (sv[4 * j4 + 1] > mr.y + kLazy) |
                  (sv[4 * j4 + 2] > mr.z + kLazy) | (sv[4 * j4 + 3] > mr.w + kLazy);
        }
#pragma unroll
        for (int g = 0; g < NG; ++g) over |= tok_ok && !(__low2float(tv2[g]) <= kLazyScale);
      }
      if (!ok1 || !ok2) *abort_flag = 1;
      const bool slow = __syncthreads_or(over) != 0;
      if (*abort_flag != 0) {
        aborted = true;
        break;
      }
      if (ci + 1 < nchunks) {
        k_ok_chunks = ci + 2;
        if (tid == kUtQkIssuer) issue_qk();
        ++qk_issued;
        refill(ci + 1);
      }
      if (slow) {
        {
          float v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = sv[j];
          const float m = warp_cols16<true>(v, lane);
          if (lane < 16) red[q4 * 64 + 16 * hq + lane] = m;
        }
        __syncthreads();
        if (tid < kUtCols) {  // warps 0 and 1: columns 0..31 and 32..63
          const float mo = m_run[tid];
          const float mn = fmaxf(mo, fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid])));
          const float a = mn == -INFINITY ? 1.f : fast_exp2(mo - mn);
          alpha[tid] = a;
          m_run[tid] = mn;
          m_use[tid] = mn == -INFINITY ? 0.f : mn;
          const uint32_t bal = __ballot_sync(0xffffffffu, a != 1.f);
          if (lane == 0) {
            need_rs[2 * warp] = (bal & 0xffffu) != 0u;
            need_rs[2 * warp + 1] = (bal >> 16) != 0u;
          }
        }
        __syncthreads();
      }
      // ---- weights of chunk ci (kept in sv) and the column sums ----
      {
        const float4* mu4 = reinterpret_cast<const float4*>(m_use + 16 * hq);
#pragma unroll
        for (int j4 = 0; j4 < 4; ++j4) {
          const float4 mu = mu4[j4];
          const float2 d01 = f2sub(make_float2(sv[4 * j4], sv[4 * j4 + 1]), make_float2(mu.x, mu.y));
          const float2 d23 = f2sub(make_float2(sv[4 * j4 + 2], sv[4 * j4 + 3]), make_float2(mu.z, mu.w));
          sv[4 * j4] = fast_exp2(d01.x), sv[4 * j4 + 1] = fast_exp2(d01.y);
          sv[4 * j4 + 2] = fast_exp2(d23.x), sv[4 * j4 + 3] = fast_exp2(d23.y);
        }
        if (slow) {  // earlier chunks' sums rescaled to the new maxima
          const float4* al4 = reinterpret_cast<const float4*>(alpha + 16 * hq);
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            const float4 a = al4[j4];
            const float2 a01 = make_float2(a.x, a.y), a23 = make_float2(a.z, a.w);
            l2[2 * j4] = f2mul(l2[2 * j4], a01);
            l2[2 * j4 + 1] = f2mul(l2[2 * j4 + 1], a23);
#pragma unroll
            for (int g = 0; g < NG; ++g) {
              z2[g][2 * j4] = f2mul(z2[g][2 * j4], a01);
              z2[g][2 * j4 + 1] = f2mul(z2[g][2 * j4 + 1], a23);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) l2[j] = f2add(l2[j], make_float2(sv[2 * j], sv[2 * j + 1]));
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const float z = __high2float(tv2[g]);
          const float2 vz2 = make_float2(z, z);
#pragma unroll
          for (int j = 0; j < 8; ++j) z2[g][j] = f2fma(make_float2(sv[2 * j], sv[2 * j + 1]), vz2, z2[g][j]);
        }
      }
      // ---- once PV(ci - 1) has finished: P' of chunk ci, O rescaled, V codes of chunk ci ----
      bool ok3 = true;
      if (ci > 0)
#pragma unroll
        for (int g = 0; g < NG; ++g) ok3 = mbar_wait_bounded(bar_o(g), (ci - 1) & 1) && ok3;
      umma::fence_after_sync();
      {  // P'_g = p * scale_g, fp16 high and low parts: row tr of the MN-major B blocks
        const uint32_t row_off = (tr >> 3) * 1024 + (tr & 7) * 128;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const float vs = __low2float(tv2[g]);
          const float2 vs2 = make_float2(vs, vs);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 x = f2mul(make_float2(sv[8 * q + 2 * e], sv[8 * q + 2 * e + 1]), vs2);
              const __half2 hh = __floats2half2_rn(x.x, x.y);
              const float2 d = f2sub(x, __half22float2(hh));
              const __half2 ll = __floats2half2_rn(d.x, d.y);
              hw[e] = *reinterpret_cast<const uint32_t*>(&hh);
              lw[e] = *reinterpret_cast<const uint32_t*>(&ll);
            }
            const uint32_t off = row_off + (((2 * hq + q) ^ (tr & 7)) << 4);
            const uint32_t blk = sb + Geo::kBp + g * 2 * kUtBlock;
            st_shared_v4(blk + off, hw[0], hw[1], hw[2], hw[3]);
            st_shared_v4(blk + kUtBlock + off, lw[0], lw[1], lw[2], lw[3]);
          }
        }
      }
      if (slow && ci > 0 && need_rs[hq] != 0) {  // O rows of channel tr, these 16 columns, high and low parts
        const float4* al4 = reinterpret_cast<const float4*>(alpha + 16 * hq);
#pragma unroll
        for (int part = 0; part < 2; ++part) {  // high and low parts
          uint32_t o[16];
          umma::tmem_ld16(t_lane + o_col + 64 * part + 16 * hq, o);
          umma::tmem_ld_wait();
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            const float4 a = al4[j4];
            const float2 x = f2mul(make_float2(__uint_as_float(o[4 * j4]), __uint_as_float(o[4 * j4 + 1])),
                                   make_float2(a.x, a.y));
            const float2 y = f2mul(make_float2(__uint_as_float(o[4 * j4 + 2]), __uint_as_float(o[4 * j4 + 3])),
                                   make_float2(a.z, a.w));
            o[4 * j4] = __float_as_uint(x.x), o[4 * j4 + 1] = __float_as_uint(x.y);
            o[4 * j4 + 2] = __float_as_uint(y.x), o[4 * j4 + 3] = __float_as_uint(y.y);
          }
          umma::tmem_st16(t_lane + o_col + 64 * part + 16 * hq, o);
        }
        umma::tmem_st_wait();
      }
      v_side(ci);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // P', V codes visible to the tensor cores
      umma::fence_before_sync();
      if (__syncthreads_or(!ok3)) {
        aborted = true;
        break;
      }
#pragma unroll
      for (int g = 0; g < NG; ++g)
        if (tid == kUtPvIssuer + 32 * g) issue_pv(ci, g);
      ++pv_issued;
    }
  }
  if (!aborted) {
    bool okf = true;
#pragma unroll
    for (int g = 0; g < NG; ++g) okf = mbar_wait_bounded(bar_o(g), (nchunks - 1) & 1) && okf;
    if (__syncthreads_or(!okf)) aborted = true;
  }

  if (!aborted) {
    umma::fence_after_sync();
    // column sums of p and of p * zero_g over the 128 token rows
    {
      float v[16];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[2 * j] = l2[j].x, v[2 * j + 1] = l2[j].y;
      float r = warp_cols16<false>(v, lane);
      if (lane < 16) red[q4 * 64 + 16 * hq + lane] = r;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[2 * j] = z2[g][j].x, v[2 * j + 1] = z2[g][j].y;
        r = warp_cols16<false>(v, lane);
        if (lane < 16) red[(1 + g) * 256 + q4 * 64 + 16 * hq + lane] = r;
      }
    }
    __syncthreads();
    if (tid < kUtCols) {
#pragma unroll
      for (int x = 0; x < 1 + NG; ++x)
        fin[x * 64 + tid] = (red[x * 256 + tid] + red[x * 256 + 64 + tid]) +
                            (red[x * 256 + 128 + tid] + red[x * 256 + 192 + tid]);
    }
    __syncthreads();
    // O row tr holds channel ch (codes at bit position code_kpos(ch)): times 2^(24 - kpos) plus
    // the zero term of its group
    const int ch = ch_tr;
    const float unscale = pow2i(24 - code_kpos(ch & 15));
    const float* zsum = fin + 64 * (1 + (NG == 2 ? ch >> 6 : 0));
    {
      uint32_t oh[16], ol[16];
      umma::tmem_ld16(t_lane + o_col + 16 * hq, oh);
      umma::tmem_ld16(t_lane + o_col + 64 + 16 * hq, ol);
      umma::tmem_ld_wait();
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int c = 16 * hq + jj;
        if (col_valid(c))
          p.part_o[(col_bh(c) * p.ns + s) * kD + ch] =
              (__uint_as_float(oh[jj]) + __uint_as_float(ol[jj])) * unscale + zsum[c];
      }
    }
    if (tid < kUtCols && col_valid(tid)) {
      const size_t bh = col_bh(tid);
      p.part_ml[(bh * p.ml_ns + s) * 2 + 0] = m_run[tid];
      p.part_ml[(bh * p.ml_ns + s) * 2 + 1] = fin[tid];
    }
  } else {
    if (tid == 0) record_error(OSCAR_DEVERR_TIMEOUT);
    for (int idx = tid; idx < kUtCols * kD; idx += kUtThreads) {
      const int c = idx / kD;
      if (col_valid(c)) p.part_o[(col_bh(c) * p.ns + s) * kD + idx % kD] = 0.f;
    }
    if (tid < kUtCols && col_valid(tid)) {
      const size_t bh = col_bh(tid);
      p.part_ml[(bh * p.ml_ns + s) * 2 + 0] = -INFINITY;
      p.part_ml[(bh * p.ml_ns + s) * 2 + 1] = 0.f;
    }
  }

  // ---- teardown: nothing of this CTA may still be in flight ----
  umma::fence_before_sync();
  __syncthreads();
  if (tid == 0) {
    // pages requested but not awaited by every thread (after a timeout)
    for (int k = k_ok_chunks * kUtPages; k < issued; ++k) mbar_wait_bounded(full(k), (k / kUtRing) & 1);
    if (qk_issued > 0) mbar_wait_bounded(bar_s, (qk_issued - 1) & 1);
    if (pv_issued > 0)
      for (int g = 0; g < NG; ++g) mbar_wait_bounded(bar_o(g), (pv_issued - 1) & 1);
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, Geo::kTmemCols);
  }
}

template <int NG>
cudaError_t launch_umma_tile(const Params& p, cudaStream_t stream) {
  constexpr size_t smem = UtGeo<NG>::kSmem;
  static_assert(smem <= 232448, "shared memory per CTA");
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(int2_umma_tile_kernel<NG>), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(int2_umma_tile_kernel<NG>, dim3(p.n_paged, p.H, p.num_seqs * p.tiles), dim3(kUtThreads), smem,
                    stream, p);
}

// ---- the extend tiles' BF16 sink/window part on tcgen05 ----
//
// One CTA of 16 warps per (sequence x tile of rows, KV head, dense split); a dense split
// is 8 pages of 16 rows of the sink buffer, then of the window ring (the decode's
// enumeration), 128 tokens: one chunk, so no running maximum is needed.  The K and V
// rows (bf16) are the A operands as they are (K-major for QK, the same bytes MN-major
// for PV), the unrotated bf16 queries the QK B operand (exact products, fp32 sums);
// the weights p <= 1 are split into bf16 high and low parts (16 significant bits) as
// the PV B operand, written over the K operand once QK has read it.  The partial of
// each column is unrotated, in the decode's format.
constexpr int kDtThreads = 512;
constexpr uint32_t kDtAK = 0, kDtAV = 2 * kUtBlock, kDtBq = 4 * kUtBlock;      // Bq: 2 K blocks of 64 rows
constexpr uint32_t kDtCol = kDtBq + kUtBlock;                                     // per-token / per-column values
constexpr size_t kDtSmem = 1024 + kDtCol + (128 + 64 + 4 * 64 + 4 * 64 + 2 * 64) * 4 + 4 * 8 + 16;

__global__ void __launch_bounds__(kDtThreads, 2) bf16_dense_tile_kernel(Params p) {
  extern __shared__ uint8_t dt_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dt_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  int* tokpos = reinterpret_cast<int*>(sm + kDtCol);  // [128]: position of the token, -1 when not in the cache
  int* colA = tokpos + 128;                            // [64]: attended positions [0, A) of the column
  float* red = reinterpret_cast<float*>(colA + 64);    // [4][64]: per-warp column maxima
  float* red2 = red + 4 * 64;                          // [4][64]: per-warp column sums
  float* mcol = red2 + 4 * 64;                         // [64]: column maximum (log2 units)
  float* mused = mcol + 64;                            // [64]: the maximum the weights use
  uint64_t* bars = reinterpret_cast<uint64_t*>(mused + 64);
  uint32_t* misc = reinterpret_cast<uint32_t*>(bars + 4);  // TMEM address
  const uint32_t bar_s = smem_u32(&bars[0]), bar_o = smem_u32(&bars[1]);
  const int h = blockIdx.y, ds = blockIdx.z;
  const int b = blockIdx.x / p.tiles, tile = blockIdx.x % p.tiles;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gqa = p.gqa, rpt = kUtCols / gqa;
  const int sidx = p.n_paged + ds;  // this split's partial index
  grid_dep_launch_dependents();
  // the rows' positions come from the row kernel, the sink/window rows from appends before
  grid_dep_wait();
  const int q0 = __ldg(p.q_start + b), q1 = __ldg(p.q_start + b + 1);
  const int r_begin = q0 + tile * rpt;
  if (r_begin >= q1) return;  // no rows in this tile
  const int n_rows = min(rpt, q1 - r_begin);
  const int L = clamp_len(p, b);
  auto col_valid = [&](int c) { return c / gqa < n_rows; };
  auto col_bh = [&](int c) { return static_cast<size_t>(r_begin + c / gqa) * p.Hq + h * gqa + c % gqa; };
  const int nsp = (p.S + kPageSize - 1) / kPageSize, nwp = (p.W + kPageSize - 1) / kPageSize;
  const int first = ds * kDenseMmaPages;
  if (first >= nsp + nwp) {  // no pages in this split: empty partials
    if (tid < kUtCols && col_valid(tid)) {
      const size_t bh = col_bh(tid);
      p.part_ml[(bh * p.ml_ns + sidx) * 2 + 0] = -INFINITY;
      p.part_ml[(bh * p.ml_ns + sidx) * 2 + 1] = 0.f;
    }
    return;
  }
  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init_fence();
  }
  if (warp == 0) umma::tmem_alloc(smem_u32(misc), 128);  // S^T (64 columns), then O (64)
  if (tid < kUtCols) {
    int A = 0;
    if (col_valid(tid)) {
      const int pos = __ldg(p.row_pos + r_begin + tid / gqa);
      A = (pos >= 0 && pos < L) ? pos + 1 : 0;  // a row outside its sequence attends nothing
    }
    colA[tid] = A;
  }
  // token t of the split: K row half (part 0, 1) or V row half (part 2, 3), 128 bytes
  {
    const int t = tid & 127, part = tid >> 7, kv = part >> 1, half = part & 1;
    const int k = first + (t >> 4), r = t & 15;
    const __nv_bfloat16* src = nullptr;
    int pos = -1;
    if (k < nsp) {
      const int sp = k * kPageSize + r;
      if (sp < min(p.S, L)) {
        pos = sp;
        src = p.sink + (((static_cast<size_t>(b) * 2 + kv) * p.H + h) * p.S + sp) * kD;
      }
    } else if (k < nsp + nwp) {
      const int slot = (k - nsp) * kPageSize + r;
      if (slot < p.W && L > 0) {
        int back = (L - 1 - slot) % p.W;
        if (back < 0) back += p.W;
        const int wpos = L - 1 - back;  // the position the ring slot holds
        if (wpos >= p.S) {
          pos = wpos;
          src = p.win + (((static_cast<size_t>(b) * 2 + kv) * p.H + h) * p.W + slot) * kD;
        }
      }
    }
    if (part == 0) tokpos[t] = pos;
    const uint32_t blk = sb + (kv ? kDtAV : kDtAK) + half * kUtBlock;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (src != nullptr) v = __ldg(reinterpret_cast<const uint4*>(src + 64 * half) + q);
      st_shared_v4(blk + t * 128 + ((q ^ (t & 7)) << 4), v.x, v.y, v.z, v.w);
    }
  }
  {  // the queries (unrotated bf16): column c, 16 channels e
    const int c = tid >> 3, e = tid & 7;
    uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
    if (col_valid(c)) {
      const uint4* src = reinterpret_cast<const uint4*>(p.q + col_bh(c) * kD + 16 * e);
      v0 = __ldg(src);
      v1 = __ldg(src + 1);
    }
    const uint32_t blk = sb + kDtBq + (e >> 2) * (64 * 128);
    const int q = 2 * (e & 3);
    st_shared_v4(blk + c * 128 + ((q ^ (c & 7)) << 4), v0.x, v0.y, v0.z, v0.w);
    st_shared_v4(blk + c * 128 + (((q + 1) ^ (c & 7)) << 4), v1.x, v1.y, v1.z, v1.w);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *misc;
  if (tid == 0) {  // QK: S^T[token][column], M = 128, N = 64
    constexpr uint32_t idesc = umma::idesc_bf16_f32(128, 64);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      umma::mma_bf16(tmem, umma::desc_k_sw128(sb + kDtAK + (ks >> 2) * kUtBlock + (ks & 3) * 32),
                     umma::desc_k_sw128(sb + kDtBq + (ks >> 2) * (64 * 128) + (ks & 3) * 32), idesc, ks != 0);
    umma::commit(bar_s);
  }
  const int q4 = warp & 3, hq = warp >> 2, tr = 32 * q4 + lane;
  const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * q4) << 16);
  const bool ok1 = mbar_wait_bounded(bar_s, 0);
  umma::fence_after_sync();
  float sv[16];
  {
    uint32_t a[16];
    umma::tmem_ld16(t_lane + 16 * hq, a);
    umma::tmem_ld_wait();
    const int pos = tokpos[tr];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      sv[j] = (pos >= 0 && pos < colA[16 * hq + j]) ? __uint_as_float(a[j]) * p.scale_log2 : -INFINITY;
  }
  {
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = sv[j];
    const float m = warp_cols16<true>(v, lane);
    if (lane < 16) red[q4 * 64 + 16 * hq + lane] = m;
  }
  const bool ok_a = __syncthreads_and(ok1);
  if (tid < kUtCols) {
    const float m = fmaxf(fmaxf(red[tid], red[64 + tid]), fmaxf(red[128 + tid], red[192 + tid]));
    mcol[tid] = m;
    mused[tid] = m == -INFINITY ? 0.f : m;
  }
  __syncthreads();
  {  // weights, their column sums, and p as bf16 high and low parts over the K operand
    const float4* mu4 = reinterpret_cast<const float4*>(mused + 16 * hq);
#pragma unroll
    for (int j4 = 0; j4 < 4; ++j4) {
      const float4 mu = mu4[j4];
      sv[4 * j4] = fast_exp2(sv[4 * j4] - mu.x);
      sv[4 * j4 + 1] = fast_exp2(sv[4 * j4 + 1] - mu.y);
      sv[4 * j4 + 2] = fast_exp2(sv[4 * j4 + 2] - mu.z);
      sv[4 * j4 + 3] = fast_exp2(sv[4 * j4 + 3] - mu.w);
    }
    const uint32_t row_off = (tr >> 3) * 1024 + (tr & 7) * 128;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x0 = sv[8 * q + 2 * e], x1 = sv[8 * q + 2 * e + 1];
        const __nv_bfloat162 hh = __floats2bfloat162_rn(x0, x1);
        const float2 hf = __bfloat1622float2(hh);
        const __nv_bfloat162 ll = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
        hw[e] = *reinterpret_cast<const uint32_t*>(&hh);
        lw[e] = *reinterpret_cast<const uint32_t*>(&ll);
      }
      const uint32_t off = row_off + (((2 * hq + q) ^ (tr & 7)) << 4);
      st_shared_v4(sb + kDtAK + off, hw[0], hw[1], hw[2], hw[3]);
      st_shared_v4(sb + kDtAK + kUtBlock + off, lw[0], lw[1], lw[2], lw[3]);
    }
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = sv[j];
    const float l = warp_cols16<false>(v, lane);
    if (lane < 16) red2[q4 * 64 + 16 * hq + lane] = l;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  umma::fence_before_sync();
  __syncthreads();
  if (tid == 0 && ok_a) {  // PV: O^T[channel][column], M = 128, N = 64, high then low parts
    umma::fence_after_sync();
    constexpr uint32_t idesc = umma::idesc_bf16_f32_mn(128, 64);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
      for (int part = 0; part < 2; ++part)
        umma::mma_bf16(tmem + 64, umma::desc_mn_sw128(sb + kDtAV + ks * 2048, kUtBlock),
                       umma::desc_mn_sw128(sb + kDtAK + part * kUtBlock + ks * 2048, kUtBlock), idesc,
                       (ks | part) != 0);
    umma::commit(bar_o);
  }
  const bool ok2 = ok_a && mbar_wait_bounded(bar_o, 0);
  const bool ok_b = __syncthreads_and(ok2);
  umma::fence_after_sync();
  if (ok_b) {
    uint32_t o[16];
    umma::tmem_ld16(t_lane + 64 + 16 * hq, o);
    umma::tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int c = 16 * hq + j;
      if (col_valid(c) && mcol[c] != -INFINITY)
        p.part_o[(col_bh(c) * p.ns + sidx) * kD + tr] = __uint_as_float(o[j]);
    }
  }
  if (tid < kUtCols && col_valid(tid)) {
    const size_t bh = col_bh(tid);
    const float l = (red2[tid] + red2[64 + tid]) + (red2[128 + tid] + red2[192 + tid]);
    p.part_ml[(bh * p.ml_ns + sidx) * 2 + 0] = ok_b ? mcol[tid] : -INFINITY;
    p.part_ml[(bh * p.ml_ns + sidx) * 2 + 1] = ok_b ? l : 0.f;
  }
  if (!ok_b && tid == 0) record_error(OSCAR_DEVERR_TIMEOUT);
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, 128);
  }
}

// ---- the extend tiles' merge: the partials of a tile's 64 columns, un-rotated once ----
//
// One CTA of 16 warps per (sequence x tile of rows, KV head):
//   phase A  warp w, columns 4w .. 4w + 3, lane = split: the largest split maximum M,
//            the weights 2^(m_s - M) (0 for splits that attended nothing) and the
//            denominator sum_s 2^(m_s - M) l_s;
//   phase B  thread (warp w, lane): columns 4w + r, channels lane + 32 k: the weighted
//            sums of the rotated (INT2 splits) and plain (BF16 sink/window splits)
//            partial outputs, every split's loads issued together; the rotated sums go
//            to shared memory;
//   phase C  the same thread: out[c][i] = (plain[c][i] + sum_j rot[c][j] R_v[i][j]) / den[c]
//            (the single un-rotation by R_v^T), R_v staged in shared memory in rows of
//            129 floats so that the 32 lanes' rows fall in 32 different banks.
constexpr int kEmThreads = 512;
constexpr int kEmRow = kD + 1;
constexpr int kEmMaxNs = 64;  // splits per row the tile merge takes (weights staged in shared memory)
constexpr size_t kEmSmem = (static_cast<size_t>(kD) * kEmRow + 64 * kD + 64 + 64 * kEmMaxNs) * 4;

__global__ void __launch_bounds__(kEmThreads, 2) extend_merge_kernel(Params p) {
  extern __shared__ __align__(16) float em[];
  float* Rs = em;                  // [128][129]
  float* rot = Rs + kD * kEmRow;   // [64][128]: rotated sums
  float* den_s = rot + 64 * kD;    // [64]
  float* wts = den_s + 64;         // [64][kEmMaxNs]: split weights 2^(m_s - M)
  const int h = blockIdx.y;
  const int b = blockIdx.x / p.tiles, tile = blockIdx.x % p.tiles;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {  // R_v[h] is an input of the call, not an output of the kernels before: read before the wait
    const float4* R4 = reinterpret_cast<const float4*>(p.R_v + static_cast<size_t>(h) * kD * kD);
    for (int idx = tid; idx < kD * kD / 4; idx += kEmThreads) {
      const float4 v = __ldg(R4 + idx);
      float* dst = Rs + (idx >> 5) * kEmRow + (idx & 31) * 4;
      dst[0] = v.x, dst[1] = v.y, dst[2] = v.z, dst[3] = v.w;
    }
  }
  grid_dep_launch_dependents();
  grid_dep_wait();  // the partials come from the split kernels before
  const int gqa = p.gqa, rpt = kUtCols / gqa;
  const int q0 = __ldg(p.q_start + b), q1 = __ldg(p.q_start + b + 1);
  const int r_begin = q0 + tile * rpt;
  if (r_begin >= q1) return;  // no rows in this tile
  const int n_rows = min(rpt, q1 - r_begin);
  auto col_valid = [&](int c) { return c / gqa < n_rows; };
  auto col_bh = [&](int c) { return static_cast<size_t>(r_begin + c / gqa) * p.Hq + h * gqa + c % gqa; };
  const int ns = p.ns, np = p.n_paged;  // ns <= kEmMaxNs (checked at launch)
  // phase A: lane = split (and split + 32), the warp's 4 columns at once
  {
    float2 v[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int c = 4 * warp + r;
      const float2* ml = reinterpret_cast<const float2*>(p.part_ml + col_bh(col_valid(c) ? c : 0) * p.ml_ns * 2);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int sp = lane + 32 * u;
        v[r][u] = (col_valid(c) && sp < ns) ? ml[sp] : make_float2(-INFINITY, 0.f);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int c = 4 * warp + r;
      float M = fmaxf(v[r][0].x, v[r][1].x);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      float den = 0.f;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        // splits that attended nothing get weight 0 (and their outputs are not used)
        const float w = (v[r][u].x == -INFINITY) ? 0.f : fast_exp2(v[r][u].x - M);
        den = fmaf(w, v[r][u].y, den);
        const int sp = lane + 32 * u;
        if (sp < kEmMaxNs) wts[c * kEmMaxNs + sp] = w;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
      if (lane == 0) den_s[c] = den;
    }
  }
  __syncwarp();  // phase B reads the weights of the warp's own columns
  // phase B: every split's partial of the 4 columns requested together
  float acc[4][4];  // [column r][channel k]: the plain sums, then the outputs
  {
    float ar[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int k = 0; k < 4; ++k) ar[r][k] = acc[r][k] = 0.f;
    // the warp's 4 columns are 4 consecutive query heads of one row (GQA 4 or 8): their
    // partials are ns * 128 floats apart
    const float* po = p.part_o + col_bh(col_valid(4 * warp) ? 4 * warp : 0) * ns * kD + lane;
    for (int sp = 0; sp < ns; ++sp) {
      float o[4][4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int k = 0; k < 4; ++k) o[r][k] = po[(static_cast<size_t>(r) * ns + sp) * kD + 32 * k];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float w = wts[(4 * warp + r) * kEmMaxNs + sp];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float t = w != 0.f ? w * o[r][k] : 0.f;  // a skipped split's output is never used
          if (sp < np)
            ar[r][k] += t;
          else
            acc[r][k] += t;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int k = 0; k < 4; ++k) rot[(4 * warp + r) * kD + lane + 32 * k] = ar[r][k];
  }
  __syncthreads();
  // phase C
  const float* Rrow = Rs + lane * kEmRow;  // rows lane + 32 k are Rrow + 32 k * kEmRow
#pragma unroll 2
  for (int j = 0; j < kD; j += 4) {
    float4 o[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) o[r] = *reinterpret_cast<const float4*>(rot + (4 * warp + r) * kD + j);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      float rv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) rv[k] = Rrow[32 * k * kEmRow + j + jj];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float ov = jj == 0 ? o[r].x : jj == 1 ? o[r].y : jj == 2 ? o[r].z : o[r].w;
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[r][k] = fmaf(ov, rv[k], acc[r][k]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int c = 4 * warp + r;
    if (!col_valid(c)) continue;
    const float den = den_s[c];
    float* out = p.out + col_bh(c) * kD + lane;
#pragma unroll
    for (int k = 0; k < 4; ++k) out[32 * k] = den > 0.f ? acc[r][k] / den : 0.f;
  }
}

}  // namespace

bool int2_umma_tile_supported(const Params& p) {
  return p.D == kD && (p.G == 64 || p.G == 128) && (p.gqa == 4 || p.gqa == 8) && p.pps <= kUtMaxPps &&
         p.q_rot != nullptr;
}

cudaError_t int2_umma_tile_split(const Params& p, cudaStream_t stream) {
  return p.G == 64 ? launch_umma_tile<2>(p, stream) : launch_umma_tile<1>(p, stream);
}

bool extend_tile_merge_supported(const Params& p) { return p.ns <= kEmMaxNs; }

cudaError_t bf16_dense_tile(const Params& p, cudaStream_t stream) {
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(bf16_dense_tile_kernel), kDtSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(bf16_dense_tile_kernel, dim3(p.num_seqs * p.tiles, p.H, p.n_dense), dim3(kDtThreads), kDtSmem,
                    stream, p);
}

cudaError_t extend_tile_merge(const Params& p, cudaStream_t stream) {
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(extend_merge_kernel), kEmSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(extend_merge_kernel, dim3(p.num_seqs * p.tiles, p.H), dim3(kEmThreads), kEmSmem, stream, p);
}

}  // namespace oscar_dec

oscar_status_t oscar_internal_decode_umma_errors(uint32_t* flags, int reset) {
  return oscar::read_unit_errors(flags, reset) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}
