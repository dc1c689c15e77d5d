// KV append: rotate by the fixed per-head R, clip per channel, quantise per
// group to asymmetric INT2 with fp16 scale/zero, pack 4 codes per byte and
// scatter the rows into the paged pool ("OSCAR: Offline Spectral
// Covariance-Aware Rotation for 2-bit KV Cache Quantization": summary
// "Practical Summary" -- fixed rotations and clipping thresholds, 2-bit KV
// cache; abstract -- paged KV cache).
//
// With a key offset c (fp32 [Hkv][D]; the OptR abstract on the same paper page:
// an attention-equivalent key reparameterisation that removes per-channel key
// offsets without changing softmax), every key is rotated as k - c, and the BF16
// sink/window key rows hold bf16(k - c); values are never offset.
//
// One CTA owns a tile of 32 tokens of one (KV head, K|V) pair, so R (fp32,
// 64 KB at D = 128) is staged once in shared memory and reused by all tokens of
// the tile.  Each warp rotates 4 tokens; lane l owns channels [l*D/32,
// (l+1)*D/32), so a group of G channels is G*32/D consecutive lanes and the
// group min/max is a warp-shuffle reduction.
#include "common.cuh"
#include "ptx.cuh"
#include "umma.cuh"

namespace {

using namespace oscar;

constexpr int kTokTile = 32;
constexpr int kThreads = 256;  // 8 warps x 4 tokens each
constexpr int64_t kSmallTokenLimit = 512;  // at most this many tokens use the few-token kernel

// Where the original bf16 rows of each appended token go besides the INT2 pool
// (oscar_append_mixed; OSCAR project card "How it works": a BF16 sink of the
// first tokens and a BF16 recent window).  Inactive (sink == win == nullptr) for
// oscar_append.
struct MixedDst {
  const int32_t* seq_ids;    // [T]; null: token t is the current token of sequence t (position seq_lens[t] - 1)
  const int32_t* positions;  // [T] (null with seq_ids)
  const int32_t* seq_lens;   // [B] lengths after this append
  int B, S, W;
  __nv_bfloat16* sink;       // [B][2][Hkv][S][D]
  __nv_bfloat16* win;        // [B][2][Hkv][W][D], ring slot p mod W
  __host__ __device__ bool active() const { return sink != nullptr || win != nullptr; }
};

// Element offset of token t's row (head h, K|V kv) in the sink (returned with
// *which = 0) or the window ring (*which = 1), or -1: position p < S goes to the
// sink, p >= max(S, L - W) to ring slot p mod W (L = the sequence's length after
// this append), other positions are INT2 only.  Tokens with a negative slot are
// skipped like the INT2 write; a sequence id or position out of range is skipped
// and flagged.
__device__ __forceinline__ int64_t mixed_row(const MixedDst& md, int64_t t, int64_t slot, int H, int D, int h,
                                             int kv, int* which) {
  *which = 0;
  if (slot < 0) return -1;
  const int b = md.seq_ids != nullptr ? __ldg(md.seq_ids + t) : static_cast<int>(t);
  if (b < 0 || b >= md.B) {
    record_error(OSCAR_DEVERR_POSITION);
    return -1;
  }
  const int L = __ldg(md.seq_lens + b);
  const int p = md.seq_ids != nullptr ? __ldg(md.positions + t) : L - 1;
  if (p < 0 || p >= L) {
    record_error(OSCAR_DEVERR_POSITION);
    return -1;
  }
  if (p < md.S) return ((((static_cast<int64_t>(b) * 2 + kv) * H + h) * md.S) + p) * D;
  if (md.W > 0 && p >= max(md.S, L - md.W)) {
    *which = 1;
    return ((((static_cast<int64_t>(b) * 2 + kv) * H + h) * md.W) + p % md.W) * D;
  }
  return -1;
}

// Clip, group min/max, fp16 scale/zero, codes, pack and store of one rotated
// vector held by a warp (lane l owns channels [l*CPL, (l+1)*CPL)).  Called by
// all 32 lanes of the warp with a warp-uniform slot.
template <int D>
__device__ __forceinline__ void quantize_store(const float (&acc)[D / 32], const float (&cl)[D / 32], int64_t slot,
                                               int H, int G, int num_pages, int h, int kv, int lane,
                                               uint8_t* __restrict__ codes, __half* __restrict__ sz) {
  constexpr int CPL = D / 32;
  if (slot < 0) return;
  if (slot >= static_cast<int64_t>(num_pages) * kPageSize) {
    if (lane == 0) record_error(OSCAR_DEVERR_SLOT);
    return;
  }
  const int lanes_per_group = G / CPL;
  float y[CPL];
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    y[c] = fminf(fmaxf(acc[c], -cl[c]), cl[c]);
    mn = fminf(mn, y[c]);
    mx = fmaxf(mx, y[c]);
  }
  for (int off = 1; off < lanes_per_group; off <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  const __half sh = __float2half_rn((mx - mn) / 3.0f);
  const __half zh = __float2half_rn(mn);
  const float s = __half2float(sh), z = __half2float(zh);
  uint32_t packed = 0;
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    uint32_t code = 0;
    if (s != 0.f) {
      const float u = (y[c] - z) / s;
      code = static_cast<uint32_t>(fminf(fmaxf(rintf(u), 0.f), 3.f));
    }
    packed |= code << (2 * c);
  }
  const int64_t page = slot / kPageSize;
  const int off = static_cast<int>(slot % kPageSize);
  const size_t row = ((static_cast<size_t>(page) * H + h) * 2 + kv) * kPageSize + off;
  uint8_t* row_codes = codes + row * (D / 4);
  if constexpr (CPL == 4) {
    row_codes[lane] = static_cast<uint8_t>(packed);
  } else {
    const uint32_t hi = __shfl_down_sync(0xffffffffu, packed, 1);
    if ((lane & 1) == 0) row_codes[lane / 2] = static_cast<uint8_t>(packed | (hi << 4));
  }
  if (lane % lanes_per_group == 0) {
    const int g = lane / lanes_per_group;
    reinterpret_cast<__half2*>(sz + row * (D / G) * 2)[g] = __halves2half2(sh, zh);
  }
}

// Stages the bf16 rows of tokens [t0, t0 + ntok) of head h into xs (fp32 [ntok][D]),
// subtracting the key offset off (nullptr: none) in fp32, and writes each token's
// BF16 row (the offset key rounded to bf16) to its sink/window row when it has one.
template <int D>
__device__ __forceinline__ void stage_rows(const __nv_bfloat16* __restrict__ x, const float* __restrict__ off,
                                           int64_t t0, int ntok, int64_t num_tokens, int H, int h,
                                           const MixedDst& md, const int64_t* dst_row, const int* dst_buf,
                                           float* xs) {
  for (int i = threadIdx.x; i < ntok * D / 2; i += blockDim.x) {
    const int tt = i / (D / 2), c2 = i % (D / 2);
    const int64_t t = t0 + tt;
    float2 val = make_float2(0.f, 0.f);
    if (t < num_tokens) {
      __nv_bfloat162 raw = reinterpret_cast<const __nv_bfloat162*>(x + (static_cast<size_t>(t) * H + h) * D)[c2];
      val = __bfloat1622float2(raw);
      if (off != nullptr) {
        const float2 c = __ldg(reinterpret_cast<const float2*>(off) + c2);
        val = make_float2(__fsub_rn(val.x, c.x), __fsub_rn(val.y, c.y));
        raw = __floats2bfloat162_rn(val.x, val.y);
      }
      if (md.active() && dst_row[tt] >= 0)
        reinterpret_cast<__nv_bfloat162*>((dst_buf[tt] ? md.win : md.sink) + dst_row[tt])[c2] = raw;
    }
    xs[tt * D + 2 * c2] = val.x;
    xs[tt * D + 2 * c2 + 1] = val.y;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) append_kernel(
    int64_t num_tokens, int H, int G, int num_pages, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const float* __restrict__ R_k, const float* __restrict__ R_v,
    const float* __restrict__ clip_k, const float* __restrict__ clip_v, const float* __restrict__ offset_k,
    const int64_t* __restrict__ slots, uint8_t* __restrict__ codes, __half* __restrict__ sz, MixedDst md) {
  grid_dep_launch_dependents();  // a following q-rotation (reads neither output) may start
  constexpr int CPL = D / 32;  // channels per lane
  extern __shared__ __align__(16) float smem[];
  __shared__ int64_t dst_row[kTokTile];
  __shared__ int dst_buf[kTokTile];
  float* Rs = smem;           // [D][D]
  float* xs = smem + D * D;   // [kTokTile][D]
  const int h = blockIdx.y, kv = blockIdx.z;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTokTile;
  const float* R = (kv ? R_v : R_k) + static_cast<size_t>(h) * D * D;
  const float* clip = (kv ? clip_v : clip_k) + static_cast<size_t>(h) * D;
  const __nv_bfloat16* x = kv ? v : k;

  for (int i = threadIdx.x; i < D * D / 4; i += kThreads)
    reinterpret_cast<float4*>(Rs)[i] = __ldg(reinterpret_cast<const float4*>(R) + i);
  if (md.active() && threadIdx.x < kTokTile) {
    const int64_t t = t0 + threadIdx.x;
    int which = 0;
    dst_row[threadIdx.x] = t < num_tokens ? mixed_row(md, t, __ldg(slots + t), H, D, h, kv, &which) : -1;
    dst_buf[threadIdx.x] = which;
  }
  if (md.active()) __syncthreads();
  const float* off = (kv == 0 && offset_k != nullptr) ? offset_k + static_cast<size_t>(h) * D : nullptr;
  stage_rows<D>(x, off, t0, kTokTile, num_tokens, H, h, md, dst_row, dst_buf, xs);
  __syncthreads();

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  float acc[4][CPL];
#pragma unroll
  for (int m = 0; m < 4; ++m)
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[m][c] = 0.f;

  // y_j = sum_i x_i R[i][j], accumulated in i order.
#pragma unroll 4
  for (int i = 0; i < D; ++i) {
    float r[CPL];
    if constexpr (CPL == 4) {
      const float4 rv = *reinterpret_cast<const float4*>(Rs + i * D + 4 * lane);
      r[0] = rv.x; r[1] = rv.y; r[2] = rv.z; r[3] = rv.w;
    } else {
      const float2 rv = *reinterpret_cast<const float2*>(Rs + i * D + 2 * lane);
      r[0] = rv.x; r[1] = rv.y;
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float xv = xs[(warp + 8 * m) * D + i];
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[m][c] = fmaf(xv, r[c], acc[m][c]);
    }
  }

  float cl[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) cl[c] = __ldg(clip + CPL * lane + c);
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int64_t t = t0 + warp + 8 * m;
    if (t >= num_tokens) break;  // warp-uniform
    quantize_store<D>(acc[m], cl, __ldg(slots + t), H, G, num_pages, h, kv, lane, codes, sz);
  }
}

// Few-token variant (decode-time append): the D rows of R are split over the 8
// warps (D/8 rows each, read from L2 without staging all of R), each warp keeps
// partial sums for up to kSmallTok tokens, and the partials are added in a
// fixed warp order through shared memory before the same quantise/store step.
constexpr int kSmallTok = 8;

// Two bf16 values as one 32-bit word (lo in the low half).
__device__ __forceinline__ uint32_t bf16_pair(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) | (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

// ---- prefill append on tcgen05 (head_dim 128) ---------------------------------------
//
// One CTA per SM serves a share of the 128-token tiles of one (KV head, K|V):
//   * y = x . R for a tile is one UMMA chain of M = 128 tokens, N = 128 outputs and
//     K = 3 x 128: R (fp32) is split into three bf16 terms hi + mid + lo (about 24
//     significant bits), stored once as R^T in shared memory, and the same x tile
//     multiplies each term, accumulating in fp32 in TMEM;
//   * warp 0 streams x tiles by TMA (3-D map: channel, head, token; 128-byte swizzle)
//     into a 3-stage ring; warp 1 owns the TMEM allocation and issues the MMAs;
//   * kUmGroups groups of 4 epilogue warps take tiles in turn (one TMEM accumulator
//     each); a thread owns one token row: a first pass over its 128 outputs clips
//     and takes the group min/max, a second pass forms the codes and packs them.
// Codes: u = (y - zero) / scale is formed as (y - zero) * (1 / scale), whose
// rounding to an integer equals that of the correctly rounded quotient unless u
// lies within 2^-18 of a half-integer; a 32-channel chunk with such an element is
// recomputed with the quotient itself.
constexpr int kUmTok = 128;
constexpr int kUmStages = 3;
constexpr int kUmGroups = 4;
constexpr int kUmThreads = 64 + 128 * kUmGroups;
constexpr uint32_t kUmXBytes = kUmTok * 128 * 2;  // one x tile (two K blocks of 16 KB)
constexpr uint32_t kUmRPart = 128 * 128 * 2;      // one bf16 term of R^T
constexpr uint32_t kUmTmemCols = 128 * kUmGroups; // one 128-column fp32 accumulator per group
static_assert(kUmTmemCols == 512 || kUmTmemCols == 256, "TMEM allocation must be a power of two");
// barriers: x_full, x_empty per stage; acc_full, acc_empty per group
constexpr int kUmBars = 2 * kUmStages + 2 * kUmGroups;
// R^T terms | x stages | clip | c . R | partial c . R (4 x 128) | mbarriers | TMEM address,
// counters; +1 KB to align to 1024
constexpr size_t kUmSmem = 1024 + 3 * kUmRPart + kUmStages * kUmXBytes + 6 * 128 * 4 + kUmBars * 8 + 16;

// Two bf16 keys (one 32-bit word) minus their offsets in fp32, rounded back to bf16.
__device__ __forceinline__ uint32_t offset_pair(uint32_t w, float c0, float c1) {
  const float a = __uint_as_float(w << 16), b = __uint_as_float(w & 0xffff0000u);
  return bf16_pair(__float2bfloat16_rn(__fsub_rn(a, c0)), __float2bfloat16_rn(__fsub_rn(b, c1)));
}

// Exact code of one value (the quotient path of the append's rule).
__device__ __forceinline__ uint32_t exact_code(float y, float z, float s) {
  return s != 0.f ? static_cast<uint32_t>(fminf(fmaxf(rintf((y - z) / s), 0.f), 3.f)) : 0u;
}

template <int G>
__global__ void __launch_bounds__(kUmThreads, 1) append_umma_kernel(
    const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v, int64_t num_tokens, int H,
    int num_pages, const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
    const float* __restrict__ R_k, const float* __restrict__ R_v, const float* __restrict__ clip_k,
    const float* __restrict__ clip_v, const float* __restrict__ offset_k, const int64_t* __restrict__ slots,
    uint8_t* __restrict__ codes, __half* __restrict__ sz, MixedDst md) {
  grid_dep_launch_dependents();  // a following q-rotation (reads neither output) may start
  constexpr int D = 128, NGRP = D / G;
  extern __shared__ uint8_t usm_raw[];
  uint8_t* usm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(usm_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t r_s = smem_u32(usm);       // 3 terms of R^T, K-major, swizzled
  const uint32_t x_s = r_s + 3 * kUmRPart;  // x stages
  float* clip_s = reinterpret_cast<float*>(usm + 3 * kUmRPart + kUmStages * kUmXBytes);
  float* cr_s = clip_s + 128;    // c . R of the key offset (K with an offset only)
  float* cr_part = cr_s + 128;   // its four partial sums over 32 rows of R each
  uint64_t* bars = reinterpret_cast<uint64_t*>(cr_part + 4 * 128);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kUmBars);
  uint32_t* flags = tmem_slot + 1;  // [0]: x tiles requested, [1]: x tiles consumed, [2]: MMA chains committed
  auto x_full = [&](int st) { return smem_u32(&bars[st]); };
  auto x_empty = [&](int st) { return smem_u32(&bars[kUmStages + st]); };
  auto acc_full = [&](int g) { return smem_u32(&bars[2 * kUmStages + g]); };
  auto acc_empty = [&](int g) { return smem_u32(&bars[2 * kUmStages + kUmGroups + g]); };
  const int h = blockIdx.y, kv = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t ntiles = (num_tokens + kUmTok - 1) / kUmTok;
  const int per = gridDim.x, j0 = blockIdx.x;
  const int n_my = static_cast<int>((ntiles - j0 + per - 1) / per);  // tiles j0, j0 + per, ...
  const float* R = (kv ? R_v : R_k) + static_cast<size_t>(h) * D * D;
  const CUtensorMap* map = kv ? &map_v : &map_k;
  // With a key offset c the K accumulator x . R is reduced by c . R (= (x - c) . R).
  const float* key_off = (kv == 0 && offset_k != nullptr) ? offset_k + static_cast<size_t>(h) * D : nullptr;

  if (tid == 0) {
    for (int i = 0; i < kUmStages; ++i) {
      mbar_init(x_full(i), 1);
      mbar_init(x_empty(i), 1);
    }
    for (int g = 0; g < kUmGroups; ++g) {
      mbar_init(acc_full(g), 1);
      mbar_init(acc_empty(g), 4);
    }
    flags[0] = flags[1] = flags[2] = 0;
    umma::prefetch_map(map);
    mbar_init_fence();
  }
  if (warp == 1) umma::tmem_alloc(smem_u32(tmem_slot), kUmTmemCols);
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  // The first x tiles are requested before R^T is built (they do not depend on it).
  const int first_issue = n_my < kUmStages ? n_my : kUmStages;
  if (tid == 0) {
    for (int i = 0; i < first_issue; ++i) {
      const int t0 = static_cast<int>((j0 + static_cast<int64_t>(i) * per) * kUmTok);
      mbar_arrive_expect_tx(x_full(i), kUmXBytes);
      umma::tma_load_3d(x_s + i * kUmXBytes, map, 0, h, t0, x_full(i));
      umma::tma_load_3d(x_s + i * kUmXBytes + kUmXBytes / 2, map, 64, h, t0, x_full(i));
    }
    flags[0] = first_issue;
  }
  // R^T terms: thread item (k pair kp, 4 outputs n4) reads R[2kp][4n4 ..] and
  // R[2kp + 1][4n4 ..]; a warp's 32 consecutive kp store 32 distinct banks.
  for (int it0 = 0; it0 < 64 * 32; it0 += kUmThreads * 2) {
    float4 a0[2], a1[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int it = it0 + u * kUmThreads + tid;
      if (it < 64 * 32) {
        const int kp = it & 63, n4 = it >> 6;
        a0[u] = __ldg(reinterpret_cast<const float4*>(R + static_cast<size_t>(2 * kp) * D) + n4);
        a1[u] = __ldg(reinterpret_cast<const float4*>(R + static_cast<size_t>(2 * kp + 1) * D) + n4);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int it = it0 + u * kUmThreads + tid;
      if (it < 64 * 32) {
        const int kp = it & 63, n4 = it >> 6;
        const float e0[4] = {a0[u].x, a0[u].y, a0[u].z, a0[u].w}, e1[4] = {a1[u].x, a1[u].y, a1[u].z, a1[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat16 h0 = __float2bfloat16_rn(e0[i]), h1 = __float2bfloat16_rn(e1[i]);
          const float d0 = e0[i] - __bfloat162float(h0), d1 = e1[i] - __bfloat162float(h1);
          const __nv_bfloat16 m0 = __float2bfloat16_rn(d0), m1 = __float2bfloat16_rn(d1);
          const __nv_bfloat16 l0 = __float2bfloat16_rn(d0 - __bfloat162float(m0));
          const __nv_bfloat16 l1 = __float2bfloat16_rn(d1 - __bfloat162float(m1));
          const uint32_t off = r_s + umma::sw128_offset(4 * n4 + i, 2 * kp, 128);
          asm volatile("st.shared.b32 [%0], %1;" ::"r"(off), "r"(bf16_pair(h0, h1)) : "memory");
          asm volatile("st.shared.b32 [%0], %1;" ::"r"(off + kUmRPart), "r"(bf16_pair(m0, m1)) : "memory");
          asm volatile("st.shared.b32 [%0], %1;" ::"r"(off + 2 * kUmRPart), "r"(bf16_pair(l0, l1)) : "memory");
        }
      }
    }
  }
  if (tid < D) clip_s[tid] = __ldg((kv ? clip_v : clip_k) + static_cast<size_t>(h) * D + tid);
  if (key_off != nullptr && tid < 4 * D) {  // partial (c . R)_j over rows 32 qq .. 32 qq + 31
    const int j = tid & (D - 1), qq = tid / D;
    float a = 0.f;
#pragma unroll 8
    for (int i = 32 * qq; i < 32 * qq + 32; ++i) a = fmaf(__ldg(key_off + i), __ldg(R + static_cast<size_t>(i) * D + j), a);
    cr_part[tid] = a;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // R^T visible to the tensor cores
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  if (key_off != nullptr) {  // CTA-uniform
    if (tid < D) cr_s[tid] = (cr_part[tid] + cr_part[D + tid]) + (cr_part[2 * D + tid] + cr_part[3 * D + tid]);
    __syncthreads();
  }

  if (warp == 0) {
    // ---- TMA producer ----
    if (lane == 0) {
      int i = first_issue;
      for (; i < n_my; ++i) {
        const int st = i % kUmStages;
        if (!mbar_wait_bounded(x_empty(st), ((i / kUmStages) - 1) & 1)) break;
        const int t0 = static_cast<int>((j0 + static_cast<int64_t>(i) * per) * kUmTok);
        mbar_arrive_expect_tx(x_full(st), kUmXBytes);
        umma::tma_load_3d(x_s + st * kUmXBytes, map, 0, h, t0, x_full(st));
        umma::tma_load_3d(x_s + st * kUmXBytes + kUmXBytes / 2, map, 64, h, t0, x_full(st));
        flags[0] = i + 1;
      }
      if (i < n_my) record_error(OSCAR_DEVERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // ---- MMA issuer: tile i accumulates in TMEM columns 128 (i % kUmGroups) ----
    if (lane == 0) {
      constexpr uint32_t idesc = umma::idesc_bf16_f32(128, 128);
      int i = 0;
      for (; i < n_my; ++i) {
        const int st = i % kUmStages, b = i % kUmGroups;
        if (!mbar_wait_bounded(x_full(st), (i / kUmStages) & 1)) break;
        flags[1] = i + 1;
        if (i >= kUmGroups && !mbar_wait_bounded(acc_empty(b), ((i / kUmGroups) - 1) & 1)) break;
        umma::fence_after_sync();
        const uint32_t d = tmem + b * 128;
#pragma unroll 1
        for (int part = 0; part < 3; ++part)
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t koff = (ks >> 2) * (kUmXBytes / 2) + (ks & 3) * 32;
            umma::mma_bf16(d, umma::desc_k_sw128(x_s + st * kUmXBytes + koff),
                           umma::desc_k_sw128(r_s + part * kUmRPart + koff), idesc, (part | ks) != 0);
          }
        umma::commit(x_empty(st));  // the x stage may be refilled
        umma::commit(acc_full(b));  // the accumulator is ready
        flags[2] = i + 1;
      }
      if (i < n_my) record_error(OSCAR_DEVERR_TIMEOUT);
    }
  } else {
    // ---- epilogue: group e takes local tiles e, e + kUmGroups, ...; thread = token row ----
    const int e = (warp - 2) >> 2, q = warp & 3;  // TMEM lanes 32q .. 32q + 31
    const int row = 32 * q + lane;
    const float4* clip4 = reinterpret_cast<const float4*>(clip_s);
    for (int i = e; i < n_my; i += kUmGroups) {
      const int64_t t = (j0 + static_cast<int64_t>(i) * per) * kUmTok + row;
      const int64_t slot = t < num_tokens ? __ldg(slots + t) : -1;  // in flight during the wait
      const bool ok = mbar_wait_bounded(acc_full(e), (i / kUmGroups) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) record_error(OSCAR_DEVERR_TIMEOUT);
        break;
      }
      umma::fence_after_sync();
      const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) + e * 128;
      // pass 1: clip (written back to TMEM), group min / max (four independent chains per chunk)
      float mn[NGRP], mx[NGRP];
#pragma unroll
      for (int gi = 0; gi < NGRP; ++gi) {
        mn[gi] = INFINITY;
        mx[gi] = -INFINITY;
      }
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t vb[32];
        umma::tmem_ld32(ta + 32 * c, vb);
        umma::tmem_ld_wait();
        if (key_off != nullptr) {
          const float4* cr4 = reinterpret_cast<const float4*>(cr_s) + 8 * c;
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const float4 o = cr4[i4];
            const float ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
            for (int r = 0; r < 4; ++r) vb[4 * i4 + r] = __float_as_uint(__uint_as_float(vb[4 * i4 + r]) - ov[r]);
          }
        }
        float lo[4] = {INFINITY, INFINITY, INFINITY, INFINITY}, hi[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const float4 cl = clip4[8 * c + i4];
          const float cv[4] = {cl.x, cl.y, cl.z, cl.w};
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float y = fminf(fmaxf(__uint_as_float(vb[4 * i4 + r]), -cv[r]), cv[r]);
            vb[4 * i4 + r] = __float_as_uint(y);
            lo[r] = fminf(lo[r], y);
            hi[r] = fmaxf(hi[r], y);
          }
        }
        umma::tmem_st32(ta + 32 * c, vb);
        const float cmn = fminf(fminf(lo[0], lo[1]), fminf(lo[2], lo[3]));
        const float cmx = fmaxf(fmaxf(hi[0], hi[1]), fmaxf(hi[2], hi[3]));
#pragma unroll
        for (int gi = 0; gi < NGRP; ++gi) {
          const bool hit = gi == 32 * c / G;
          mn[gi] = hit ? fminf(mn[gi], cmn) : mn[gi];
          mx[gi] = hit ? fmaxf(mx[gi], cmx) : mx[gi];
        }
      }
      umma::tmem_st_wait();
      float zg[NGRP], sg[NGRP], ig[NGRP];
      bool fastg[NGRP];
      uint32_t szw[NGRP];
#pragma unroll
      for (int gi = 0; gi < NGRP; ++gi) {
        const __half sh = __float2half_rn((mx[gi] - mn[gi]) / 3.0f);
        const __half zh = __float2half_rn(mn[gi]);
        szw[gi] = static_cast<uint32_t>(__half_as_ushort(sh)) | (static_cast<uint32_t>(__half_as_ushort(zh)) << 16);
        sg[gi] = __half2float(sh);
        zg[gi] = __half2float(zh);
        ig[gi] = sg[gi] != 0.f ? 1.0f / sg[gi] : 0.f;  // scale 0: every code is 0
        // u = (y - zero) * (1 / scale) is monotone in y: when it spans [-0.5, 3.5) at the
        // group's extremes, rint(u) is a code 0..3 without clamping.
        fastg[gi] = (mn[gi] - zg[gi]) * ig[gi] >= -0.5f && (mx[gi] - zg[gi]) * ig[gi] < 3.5f;
      }
      const bool store = slot >= 0 && slot < static_cast<int64_t>(num_pages) * kPageSize;
      const size_t rrow = store ? ((static_cast<size_t>(slot / kPageSize) * H + h) * 2 + kv) * kPageSize +
                                      static_cast<size_t>(slot % kPageSize)
                                : 0;
      uint2* crow = reinterpret_cast<uint2*>(codes + rrow * (D / 4));
      // pass 2: codes, two packed words (8 bytes of the row) per 32-channel chunk.
      // m = u + 1.5 * 2^23 rounds u to an integer (ties to even) whose value is the low
      // bits of m, so bits(m) = bits(1.5 * 2^23) + code; the 16 codes of a word are
      // summed as bits(m_j) * 4^j and the constant part is taken off once.
      constexpr float kRound = 12582912.0f;
      constexpr uint32_t kWordBias = 0x4B400000u * 0x55555555u;  // bits(kRound) * sum_j 4^j (mod 2^32)
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float z = zg[0], inv = ig[0], s = sg[0];
        bool fast = fastg[0];
#pragma unroll
        for (int gi = 1; gi < NGRP; ++gi) {
          const bool hit = gi == 32 * c / G;
          z = hit ? zg[gi] : z;
          inv = hit ? ig[gi] : inv;
          s = hit ? sg[gi] : s;
          fast = hit ? fastg[gi] : fast;
        }
        uint32_t vb[32];
        umma::tmem_ld32(ta + 32 * c, vb);
        umma::tmem_ld_wait();
        const uint64_t z2 = umma::f2_pack(z, z), inv2 = umma::f2_pack(inv, inv), kr2 = umma::f2_pack(kRound, kRound);
        uint32_t w[2] = {0u - kWordBias, 0u - kWordBias};
        float emax = 0.f;
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const uint64_t y2 = umma::f2_pack(__uint_as_float(vb[j]), __uint_as_float(vb[j + 1]));
          const uint64_t u2 = umma::f2_mul(umma::f2_sub(y2, z2), inv2);
          const uint64_t m2 = umma::f2_add(u2, kr2);
          const uint64_t r2 = umma::f2_sub(u2, umma::f2_sub(m2, kr2));  // u - rint(u), exact
          float m0, m1, e0, e1;
          umma::f2_unpack(m2, m0, m1);
          umma::f2_unpack(r2, e0, e1);
          emax = fmaxf(emax, fmaxf(fabsf(e0), fabsf(e1)));
          w[j >> 4] += __float_as_uint(m0) * (1u << (2 * (j & 15)));
          w[j >> 4] += __float_as_uint(m1) * (1u << (2 * ((j + 1) & 15)));
        }
        if (__any_sync(0xffffffffu, !fast || emax > 0.5f - 0x1p-18f)) {
          // out-of-range values or one near a rounding boundary in the warp's chunk: the
          // quotient itself, clamped (the clipped values are in TMEM)
          w[0] = w[1] = 0u;
#pragma unroll 1
          for (int j = 0; j < 32; ++j) {
            uint32_t one;
            asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(one) : "r"(ta + 32 * c + j) : "memory");
            umma::tmem_ld_wait();
            const uint32_t code = exact_code(__uint_as_float(one), z, s);
            if (j < 16) w[0] |= code << (2 * j);
            else w[1] |= code << (2 * (j - 16));
          }
        }
        if (store) crow[c] = make_uint2(w[0], w[1]);
      }
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(e));  // the accumulator may be overwritten

      if (t >= num_tokens) continue;
      if (md.active()) {  // oscar_append_mixed: the token's bf16 row (sink or window)
        int which = 0;
        const int64_t dst = mixed_row(md, t, slot, H, D, h, kv, &which);
        if (dst >= 0) {
          const uint4* src = reinterpret_cast<const uint4*>((kv ? v : k) + (static_cast<size_t>(t) * H + h) * D);
          uint4* out = reinterpret_cast<uint4*>((which ? md.win : md.sink) + dst);
          if (key_off != nullptr) {  // the offset key, rounded to bf16
            const float4* c4 = reinterpret_cast<const float4*>(key_off);
#pragma unroll 4
            for (int c = 0; c < D / 8; ++c) {
              const uint4 w = __ldg(src + c);
              const float4 ca = __ldg(c4 + 2 * c), cb = __ldg(c4 + 2 * c + 1);
              out[c] = make_uint4(offset_pair(w.x, ca.x, ca.y), offset_pair(w.y, ca.z, ca.w),
                                  offset_pair(w.z, cb.x, cb.y), offset_pair(w.w, cb.z, cb.w));
            }
          } else {
#pragma unroll 4
            for (int c = 0; c < D / 8; ++c) out[c] = __ldg(src + c);
          }
        }
      }
      if (slot >= static_cast<int64_t>(num_pages) * kPageSize) {
        record_error(OSCAR_DEVERR_SLOT);
        continue;
      }
      if (!store) continue;
      void* zdst = sz + rrow * NGRP * 2;
      if constexpr (NGRP == 4) *static_cast<uint4*>(zdst) = make_uint4(szw[0], szw[1], szw[2], szw[3]);
      if constexpr (NGRP == 2) *static_cast<uint2*>(zdst) = make_uint2(szw[0], szw[1]);
      if constexpr (NGRP == 1) *static_cast<uint32_t*>(zdst) = szw[0];
    }
  }

  // ---- teardown: nothing of this CTA may still be in flight ----
  __syncthreads();
  if (tid == 0) {
    // x tiles requested but never consumed (only after a timeout)
    for (uint32_t i = flags[1]; i < flags[0]; ++i) mbar_wait_bounded(x_full(i % kUmStages), (i / kUmStages) & 1);
    // the last committed MMA chain (both of its completion barriers)
    if (flags[2] > 0) {
      const uint32_t i = flags[2] - 1;
      mbar_wait_bounded(acc_full(i % kUmGroups), (i / kUmGroups) & 1);
      mbar_wait_bounded(x_empty(i % kUmStages), (i / kUmStages) & 1);
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kUmTmemCols);
  }
}

using umma::encode_tiled;
using umma::EncodeTiledFn;

// Map of x [T][H][128] bf16 as (channel, head, token) with a 64 x 1 x 128 box:
// one K block (64 channels) of 128 tokens of one head, 128-byte swizzled.
bool x_tensor_map(CUtensorMap* m, const void* x, int64_t T, int H) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
  const cuuint64_t strides[2] = {256, static_cast<cuuint64_t>(H) * 256};
  const cuuint32_t box[3] = {64, 1, kUmTok};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int G>
cudaError_t launch_append_umma(int64_t T, const oscar_dims_t* d, const void* k, const void* v, const float* R_k,
                               const float* R_v, const float* clip_k, const float* clip_v, const float* offset_k,
                               const int64_t* slots, uint8_t* codes, void* sz, const MixedDst& md,
                               cudaStream_t stream) {
  CUtensorMap mk, mv;
  if (!x_tensor_map(&mk, k, T, d->num_kv_heads) || !x_tensor_map(&mv, v, T, d->num_kv_heads))
    return cudaErrorInvalidValue;
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(append_umma_kernel<G>), kUmSmem);
  if (e != cudaSuccess) return e;
  // One CTA per SM: the (KV head, K|V) pairs share the SMs evenly, each CTA takes
  // every per-th tile of its pair.
  const int64_t ntiles = (T + kUmTok - 1) / kUmTok;
  const int hkv = 2 * d->num_kv_heads;
  int64_t per = num_sms() / hkv;
  if (per < 1) per = 1;
  if (per > ntiles) per = ntiles;
  const dim3 grid(static_cast<unsigned>(per), d->num_kv_heads, 2);
  append_umma_kernel<G><<<grid, kUmThreads, kUmSmem, stream>>>(
      mk, mv, T, d->num_kv_heads, d->num_pages, static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), R_k, R_v, clip_k, clip_v, offset_k, slots, codes,
      static_cast<__half*>(sz), md);
  return cudaGetLastError();
}

template <int D>
__global__ void __launch_bounds__(kThreads) append_small_kernel(
    int64_t num_tokens, int H, int G, int num_pages, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const float* __restrict__ R_k, const float* __restrict__ R_v,
    const float* __restrict__ clip_k, const float* __restrict__ clip_v, const float* __restrict__ offset_k,
    const int64_t* __restrict__ slots, uint8_t* __restrict__ codes, __half* __restrict__ sz, MixedDst md) {
  grid_dep_launch_dependents();  // a following q-rotation (reads neither output) may start
  constexpr int CPL = D / 32;
  constexpr int kWarpsA = kThreads / 32;
  __shared__ int64_t dst_row[kSmallTok];
  __shared__ int dst_buf[kSmallTok];
  constexpr int kRows = D / kWarpsA;
  __shared__ __align__(16) float xs[kSmallTok * D];
  __shared__ __align__(16) float part[kWarpsA * kSmallTok * D];
  const int h = blockIdx.y, kv = blockIdx.z;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kSmallTok;
  const float* R = (kv ? R_v : R_k) + static_cast<size_t>(h) * D * D;
  const float* clip = (kv ? clip_v : clip_k) + static_cast<size_t>(h) * D;
  const __nv_bfloat16* x = kv ? v : k;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Every load is issued before any is used: this warp's kRows rows of R (one
  // round trip instead of one per few rows), the clip thresholds and the slot of
  // the token it finishes.
  float rv[kRows][CPL];
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int i = warp * kRows + r;
    if constexpr (CPL == 4) {
      const float4 q4 = __ldg(reinterpret_cast<const float4*>(R + static_cast<size_t>(i) * D) + lane);
      rv[r][0] = q4.x; rv[r][1] = q4.y; rv[r][2] = q4.z; rv[r][3] = q4.w;
    } else {
      const float2 q2 = __ldg(reinterpret_cast<const float2*>(R + static_cast<size_t>(i) * D) + lane);
      rv[r][0] = q2.x; rv[r][1] = q2.y;
    }
  }
  float cl[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) cl[c] = __ldg(clip + CPL * lane + c);
  const int64_t t_mine = t0 + warp;  // the token this warp finishes (if any)
  const int64_t slot_mine = warp < kSmallTok && t_mine < num_tokens ? __ldg(slots + t_mine) : -1;
  if (md.active() && threadIdx.x < kSmallTok) {
    const int64_t t = t0 + threadIdx.x;
    int which = 0;
    dst_row[threadIdx.x] = t < num_tokens ? mixed_row(md, t, __ldg(slots + t), H, D, h, kv, &which) : -1;
    dst_buf[threadIdx.x] = which;
  }
  if (md.active()) __syncthreads();
  const float* off = (kv == 0 && offset_k != nullptr) ? offset_k + static_cast<size_t>(h) * D : nullptr;
  // Launched as a programmatic dependent: R, the thresholds and the slots above were
  // read while the kernel before may still run; the token rows are read, and every
  // output written, only after it has completed.
  grid_dep_wait();
  stage_rows<D>(x, off, t0, kSmallTok, num_tokens, H, h, md, dst_row, dst_buf, xs);
  __syncthreads();
  float acc[kSmallTok][CPL];
#pragma unroll
  for (int m = 0; m < kSmallTok; ++m)
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[m][c] = 0.f;
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int i = warp * kRows + r;
#pragma unroll
    for (int m = 0; m < kSmallTok; ++m) {
      const float xv = xs[m * D + i];
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[m][c] = fmaf(xv, rv[r][c], acc[m][c]);
    }
  }
#pragma unroll
  for (int m = 0; m < kSmallTok; ++m)
#pragma unroll
    for (int c = 0; c < CPL; ++c) part[(warp * kSmallTok + m) * D + CPL * lane + c] = acc[m][c];
  __syncthreads();
  // warp m finishes token m
  const int m = warp;
  const int64_t t = t0 + m;
  if (m >= kSmallTok || t >= num_tokens) return;
  float tot[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < kWarpsA; ++w) a += part[(w * kSmallTok + m) * D + CPL * lane + c];
    tot[c] = a;
  }
  quantize_store<D>(tot, cl, slot_mine, H, G, num_pages, h, kv, lane, codes, sz);
}

// Plain copy of bf16 rows into the BF16 paged pool, 16 bytes per thread.
__global__ void bf16_append_kernel(int64_t num_tokens, int H, int D, int num_pages,
                                   const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                                   const int64_t* __restrict__ slots, __nv_bfloat16* __restrict__ pages) {
  grid_dep_launch_dependents();  // a following q-rotation (reads neither output) may start
  const int chunks = D / 8;  // 16-byte chunks per row
  const int64_t total = num_tokens * H * 2 * chunks;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % chunks);
    const int kv = static_cast<int>((i / chunks) % 2);
    const int h = static_cast<int>((i / (2 * chunks)) % H);
    const int64_t t = i / (2 * chunks * H);
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;
    if (slot >= static_cast<int64_t>(num_pages) * kPageSize) {
      record_error(OSCAR_DEVERR_SLOT);
      continue;
    }
    const __nv_bfloat16* src = (kv ? v : k) + (static_cast<size_t>(t) * H + h) * D;
    const int64_t page = slot / kPageSize;
    const int off = static_cast<int>(slot % kPageSize);
    __nv_bfloat16* dst = pages + (((static_cast<size_t>(page) * H + h) * 2 + kv) * kPageSize + off) * D;
    reinterpret_cast<uint4*>(dst)[c] = __ldg(reinterpret_cast<const uint4*>(src) + c);
  }
}

template <int D>
cudaError_t launch_append(int64_t T, const oscar_dims_t* d, const void* k, const void* v, const float* R_k,
                          const float* R_v, const float* clip_k, const float* clip_v, const float* offset_k,
                          const int64_t* slots, uint8_t* codes, void* sz, const MixedDst& md,
                          cudaStream_t stream) {
  // Few tokens per (head, K|V): spread R's rows over warps instead of staging all of R.
  if (T <= kSmallTokenLimit) {
    // programmatic stream serialisation: the kernel may start while the one before ends
    // (it waits for it before reading the token rows or writing anything)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((T + kSmallTok - 1) / kSmallTok), d->num_kv_heads, 2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, append_small_kernel<D>, T, d->num_kv_heads, d->group_size, d->num_pages,
                              static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), R_k, R_v,
                              clip_k, clip_v, offset_k, slots, codes, static_cast<__half*>(sz), md);
  }
  if (D == 128 && T < 0x7fffffffLL - kUmTok) {  // the rotation on tcgen05 tensor cores
    switch (d->group_size) {
      case 32: return launch_append_umma<32>(T, d, k, v, R_k, R_v, clip_k, clip_v, offset_k, slots, codes, sz, md,
                                               stream);
      case 64: return launch_append_umma<64>(T, d, k, v, R_k, R_v, clip_k, clip_v, offset_k, slots, codes, sz, md,
                                               stream);
      default: return launch_append_umma<128>(T, d, k, v, R_k, R_v, clip_k, clip_v, offset_k, slots, codes, sz, md,
                                               stream);
    }
  }
  const size_t smem = (static_cast<size_t>(D) * D + kTokTile * D) * sizeof(float);
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(append_kernel<D>), smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((T + kTokTile - 1) / kTokTile), d->num_kv_heads, 2);
  append_kernel<D><<<grid, kThreads, smem, stream>>>(
      T, d->num_kv_heads, d->group_size, d->num_pages, static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), R_k, R_v, clip_k, clip_v, offset_k, slots, codes,
      static_cast<__half*>(sz), md);
  return cudaGetLastError();
}

}  // namespace

namespace {

oscar_status_t run_append(const oscar_dims_t* dims, int64_t num_tokens, const void* k, const void* v,
                          const float* R_k, const float* R_v, const float* clip_k, const float* clip_v,
                          const float* offset_k, const int64_t* slot_mapping, uint8_t* int2_pages,
                          void* scale_zero_pages, const MixedDst& md, void* stream) {
  oscar_status_t st = check_dims(dims);
  if (st != OSCAR_OK) return st;
  if (num_tokens < 0) return OSCAR_ERR_INVALID_ARG;
  if (num_tokens == 0) return OSCAR_OK;
  if (!k || !v || !R_k || !R_v || !clip_k || !clip_v || !slot_mapping || !int2_pages || !scale_zero_pages)
    return OSCAR_ERR_INVALID_ARG;
  if (misaligned16(k) || misaligned16(v) || misaligned16(R_k) || misaligned16(R_v) || misaligned16(int2_pages) ||
      misaligned16(scale_zero_pages) || misaligned16(md.sink) || misaligned16(md.win) || misaligned16(offset_k))
    return OSCAR_ERR_INVALID_ARG;
  if ((num_tokens + kTokTile - 1) / kTokTile > 0x7fffffffLL) return OSCAR_ERR_UNSUPPORTED;
  cudaError_t e = dims->head_dim == 128
                      ? launch_append<128>(num_tokens, dims, k, v, R_k, R_v, clip_k, clip_v, offset_k,
                                           slot_mapping, int2_pages, scale_zero_pages, md, as_stream(stream))
                      : launch_append<64>(num_tokens, dims, k, v, R_k, R_v, clip_k, clip_v, offset_k,
                                          slot_mapping, int2_pages, scale_zero_pages, md, as_stream(stream));
  return e == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

}  // namespace

extern "C" oscar_status_t oscar_append(const oscar_dims_t* dims, int64_t num_tokens, const void* k, const void* v,
                                       const float* R_k, const float* R_v, const float* clip_k,
                                       const float* clip_v, const float* offset_k, const int32_t* page_table,
                                       const int64_t* slot_mapping, uint8_t* int2_pages, void* scale_zero_pages,
                                       void* stream) {
  (void)page_table;
  return run_append(dims, num_tokens, k, v, R_k, R_v, clip_k, clip_v, offset_k, slot_mapping, int2_pages,
                    scale_zero_pages, MixedDst{}, stream);
}

extern "C" oscar_status_t oscar_append_mixed(const oscar_dims_t* dims, int64_t num_tokens, const void* k,
                                             const void* v, const float* R_k, const float* R_v,
                                             const float* clip_k, const float* clip_v, const float* offset_k,
                                             const int32_t* page_table,
                                             const int64_t* slot_mapping, const int32_t* seq_ids,
                                             const int32_t* positions, const int32_t* seq_lens, int32_t batch,
                                             int32_t sink_len, int32_t window_len, uint8_t* int2_pages,
                                             void* scale_zero_pages, void* bf16_sink, void* bf16_window,
                                             void* stream) {
  (void)page_table;
  if (batch < 0 || sink_len < 0 || window_len < 0) return OSCAR_ERR_INVALID_ARG;
  if (num_tokens > 0 && (batch == 0 || !seq_ids || !positions || !seq_lens)) return OSCAR_ERR_INVALID_ARG;
  if ((sink_len > 0 && !bf16_sink) || (window_len > 0 && !bf16_window)) return OSCAR_ERR_INVALID_ARG;
  MixedDst md{};
  md.seq_ids = seq_ids;
  md.positions = positions;
  md.seq_lens = seq_lens;
  md.B = batch;
  md.S = sink_len;
  md.W = window_len;
  md.sink = sink_len > 0 ? static_cast<__nv_bfloat16*>(bf16_sink) : nullptr;
  md.win = window_len > 0 ? static_cast<__nv_bfloat16*>(bf16_window) : nullptr;
  return run_append(dims, num_tokens, k, v, R_k, R_v, clip_k, clip_v, offset_k, slot_mapping, int2_pages,
                    scale_zero_pages, md, stream);
}

// The current token of every sequence (token b at position seq_lens[b] - 1 of sequence
// b): oscar_append_mixed with those ids and positions (oscar_append_decode's sequential
// form).
oscar_status_t oscar_internal_append_current(const oscar_dims_t* dims, int32_t batch, const void* k, const void* v,
                                             const float* R_k, const float* R_v, const float* clip_k,
                                             const float* clip_v, const float* offset_k,
                                             const int64_t* slot_mapping, const int32_t* seq_lens,
                                             int32_t sink_len, int32_t window_len, uint8_t* int2_pages,
                                             void* scale_zero_pages, void* bf16_sink, void* bf16_window,
                                             void* stream) {
  if (batch < 0 || sink_len < 0 || window_len < 0) return OSCAR_ERR_INVALID_ARG;
  if (batch > 0 && !seq_lens) return OSCAR_ERR_INVALID_ARG;
  if ((sink_len > 0 && !bf16_sink) || (window_len > 0 && !bf16_window)) return OSCAR_ERR_INVALID_ARG;
  MixedDst md{};
  md.seq_lens = seq_lens;
  md.B = batch;
  md.S = sink_len;
  md.W = window_len;
  md.sink = sink_len > 0 ? static_cast<__nv_bfloat16*>(bf16_sink) : nullptr;
  md.win = window_len > 0 ? static_cast<__nv_bfloat16*>(bf16_window) : nullptr;
  return run_append(dims, batch, k, v, R_k, R_v, clip_k, clip_v, offset_k, slot_mapping, int2_pages,
                    scale_zero_pages, md, stream);
}

extern "C" oscar_status_t oscar_bf16_append(const oscar_dims_t* dims, int64_t num_tokens, const void* k,
                                            const void* v, const int64_t* slot_mapping, void* bf16_pages,
                                            void* stream) {
  oscar_status_t st = check_dims(dims);
  if (st != OSCAR_OK) return st;
  if (num_tokens < 0) return OSCAR_ERR_INVALID_ARG;
  if (num_tokens == 0) return OSCAR_OK;
  if (!k || !v || !slot_mapping || !bf16_pages) return OSCAR_ERR_INVALID_ARG;
  if (misaligned16(k) || misaligned16(v) || misaligned16(bf16_pages)) return OSCAR_ERR_INVALID_ARG;
  const int64_t total = num_tokens * dims->num_kv_heads * 2 * (dims->head_dim / 8);
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 16;
  if (blocks > cap) blocks = cap;
  bf16_append_kernel<<<static_cast<unsigned>(blocks), threads, 0, as_stream(stream)>>>(
      num_tokens, dims->num_kv_heads, dims->head_dim, dims->num_pages, static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), slot_mapping, static_cast<__nv_bfloat16*>(bf16_pages));
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

oscar_status_t oscar_internal_append_errors(uint32_t* flags, int reset) {
  return read_unit_errors(flags, reset) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}
