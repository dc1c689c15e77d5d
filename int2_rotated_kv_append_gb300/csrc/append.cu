// KV append: rotate by the fixed per-head R, clip per channel, quantise per
// group to asymmetric INT2 with fp16 scale/zero, pack 4 codes per byte and
// scatter the rows into the paged pool ("OSCAR: Offline Spectral
// Covariance-Aware Rotation for 2-bit KV Cache Quantization": summary
// "Practical Summary" -- fixed rotations and clipping thresholds, 2-bit KV
// cache; abstract -- paged KV cache).
//
// One CTA owns a tile of 32 tokens of one (KV head, K|V) pair, so R (fp32,
// 64 KB at D = 128) is staged once in shared memory and reused by all tokens of
// the tile.  Each warp rotates 4 tokens; lane l owns channels [l*D/32,
// (l+1)*D/32), so a group of G channels is G*32/D consecutive lanes and the
// group min/max is a warp-shuffle reduction.
#include "common.cuh"
#include "ptx.cuh"

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
  const int32_t* seq_ids;    // [T]
  const int32_t* positions;  // [T]
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
  const int b = __ldg(md.seq_ids + t), p = __ldg(md.positions + t);
  if (b < 0 || b >= md.B || p < 0) {
    record_error(OSCAR_DEVERR_POSITION);
    return -1;
  }
  const int L = __ldg(md.seq_lens + b);
  if (p >= L) {
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

template <int D>
__global__ void __launch_bounds__(kThreads) append_kernel(
    int64_t num_tokens, int H, int G, int num_pages, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const float* __restrict__ R_k, const float* __restrict__ R_v,
    const float* __restrict__ clip_k, const float* __restrict__ clip_v, const int64_t* __restrict__ slots,
    uint8_t* __restrict__ codes, __half* __restrict__ sz, MixedDst md) {
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
  for (int i = threadIdx.x; i < kTokTile * D / 2; i += kThreads) {
    const int tt = i / (D / 2), c2 = i % (D / 2);
    const int64_t t = t0 + tt;
    float2 val = make_float2(0.f, 0.f);
    if (t < num_tokens) {
      const __nv_bfloat162 raw = reinterpret_cast<const __nv_bfloat162*>(x + (static_cast<size_t>(t) * H + h) * D)[c2];
      val = __bfloat1622float2(raw);
      if (md.active() && dst_row[tt] >= 0)
        reinterpret_cast<__nv_bfloat162*>((dst_buf[tt] ? md.win : md.sink) + dst_row[tt])[c2] = raw;
    }
    xs[tt * D + 2 * c2] = val.x;
    xs[tt * D + 2 * c2 + 1] = val.y;
  }
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

// ---- prefill append with the rotation on tensor cores (head_dim 128) -----------
//
// y = x . R for tiles of kTcTok tokens of one (KV head, K|V) on mma.sync m16n8k16
// (bf16 in, fp32 accumulate).  x is bf16 and exact as an operand; R (fp32) is split
// into three bf16 terms hi + mid + lo (about 24 significant bits), each multiplied
// in and accumulated in fp32, so y carries fp32-level rounding like the FFMA
// rotation.  Each CTA serves one (head, K|V) and loops over every gridDim.x-th
// token tile: R^T's three parts stay in shared memory (split once per CTA), the
// next tile's x is loaded into registers while the current one is multiplied, and
// the clip / group min-max / fp16 scale-zero / codes / pack step runs on the
// accumulators in registers (a quad of lanes holds a token row).  Shared rows are
// 256 bytes with their 16-byte chunks XOR-swizzled by row, so ldmatrix reads are
// conflict free.  Each of the 4 warps computes 16 tokens x 128 outputs.
constexpr int kTcTok = 64;
constexpr int kTcThreads = 128;
constexpr int kTcLoads = kTcTok * 16 / kTcThreads;     // 16-byte chunks of x per thread per tile
constexpr size_t kTcSmem = (3 * 128 + kTcTok) * 256;  // R^T parts, x tile: two CTAs fit an SM

__device__ __forceinline__ uint32_t swz(int row, int chunk) { return row * 256 + ((chunk ^ (row & 7)) << 4); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t bf16_pair(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) | (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

// x rows of token tile `tile` (zeros past the end), chunk u*kTcThreads + tid.
__device__ __forceinline__ void tc_load_x(const __nv_bfloat16* __restrict__ x, int64_t num_tokens, int H, int h,
                                          int64_t tile, int tid, uint4 (&raw)[kTcLoads]) {
#pragma unroll
  for (int u = 0; u < kTcLoads; ++u) {
    const int it = u * kTcThreads + tid, tt = it >> 4, c = it & 15;
    const int64_t t = tile * kTcTok + tt;
    raw[u] = t < num_tokens ? __ldg(reinterpret_cast<const uint4*>(x + (static_cast<size_t>(t) * H + h) * 128) + c)
                            : make_uint4(0u, 0u, 0u, 0u);
  }
}

template <int G>
__global__ void __launch_bounds__(kTcThreads, 2) append_tc_kernel(
    int64_t num_tokens, int H, int num_pages, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const float* __restrict__ R_k, const float* __restrict__ R_v,
    const float* __restrict__ clip_k, const float* __restrict__ clip_v, const int64_t* __restrict__ slots,
    uint8_t* __restrict__ codes, __half* __restrict__ sz, MixedDst md) {
  grid_dep_launch_dependents();  // a following q-rotation (reads neither output) may start
  constexpr int D = 128, NPG = G / 8, NGRP = D / G;  // n-tiles per group, groups per row
  extern __shared__ __align__(128) uint8_t tsm[];
  __shared__ int64_t dst_row[kTcTok];
  __shared__ int dst_buf[kTcTok];
  const int h = blockIdx.y, kv = blockIdx.z;
  const float* R = (kv ? R_v : R_k) + static_cast<size_t>(h) * D * D;
  const __nv_bfloat16* x = kv ? v : k;
  const uint32_t rt = smem_u32(tsm);       // R^T part p: rows n at rt + p * 128 * 256
  const uint32_t xt = rt + 3 * 128 * 256;  // x tile: token rows
  const float* clip = (kv ? clip_v : clip_k) + static_cast<size_t>(h) * D;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t ntiles = (num_tokens + kTcTok - 1) / kTcTok;

  uint4 raw[kTcLoads];
  tc_load_x(x, num_tokens, H, h, blockIdx.x, tid, raw);  // the first tile's x is in flight during the split
  // R^T in three bf16 parts.  Thread: k pair kp = tid % 64 (rows 2kp, 2kp + 1 of R),
  // 4 consecutive n per item; a warp's stores fall on 32 distinct banks.
  {
    const int kp = tid & 63;
#pragma unroll 1
    for (int b = 0; b < 2; ++b) {
      float4 r0[8], r1[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int n4 = 2 * (8 * b + u) + (tid >> 6);
        r0[u] = __ldg(reinterpret_cast<const float4*>(R + static_cast<size_t>(2 * kp) * D) + n4);
        r1[u] = __ldg(reinterpret_cast<const float4*>(R + static_cast<size_t>(2 * kp + 1) * D) + n4);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int n4 = 2 * (8 * b + u) + (tid >> 6);
        const float a0[4] = {r0[u].x, r0[u].y, r0[u].z, r0[u].w}, a1[4] = {r1[u].x, r1[u].y, r1[u].z, r1[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat16 h0 = __float2bfloat16_rn(a0[i]), h1 = __float2bfloat16_rn(a1[i]);
          const float e0 = a0[i] - __bfloat162float(h0), e1 = a1[i] - __bfloat162float(h1);
          const __nv_bfloat16 m0 = __float2bfloat16_rn(e0), m1 = __float2bfloat16_rn(e1);
          const __nv_bfloat16 l0 = __float2bfloat16_rn(e0 - __bfloat162float(m0));
          const __nv_bfloat16 l1 = __float2bfloat16_rn(e1 - __bfloat162float(m1));
          const uint32_t off = rt + swz(4 * n4 + i, kp >> 2) + (kp & 3) * 4;
          asm volatile("st.shared.b32 [%0], %1;" ::"r"(off), "r"(bf16_pair(h0, h1)) : "memory");
          asm volatile("st.shared.b32 [%0], %1;" ::"r"(off + 128 * 256), "r"(bf16_pair(m0, m1)) : "memory");
          asm volatile("st.shared.b32 [%0], %1;" ::"r"(off + 2 * 128 * 256), "r"(bf16_pair(l0, l1)) : "memory");
        }
      }
    }
  }

  const int a_row = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1), a_hi = lane >> 4;
  const int b_row = (lane & 7) + 8 * (lane >> 4), b_hi = (lane >> 3) & 1;
  const int g = lane >> 2, tq = lane & 3;
#pragma unroll 1
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t t0 = tile * kTcTok;
    __syncthreads();  // the previous tile's x reads are done (first pass: R^T is stored)
    if (md.active()) {
      if (tid < kTcTok) {
        const int64_t t = t0 + tid;
        int which = 0;
        dst_row[tid] = t < num_tokens ? mixed_row(md, t, __ldg(slots + t), H, D, h, kv, &which) : -1;
        dst_buf[tid] = which;
      }
      __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < kTcLoads; ++u) {
      const int it = u * kTcThreads + tid, tt = it >> 4, c = it & 15;
      if (md.active() && t0 + tt < num_tokens && dst_row[tt] >= 0)  // oscar_append_mixed: the bf16 row
        reinterpret_cast<uint4*>((dst_buf[tt] ? md.win : md.sink) + dst_row[tt])[c] = raw[u];
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(xt + swz(tt, c)), "r"(raw[u].x), "r"(raw[u].y),
                   "r"(raw[u].z), "r"(raw[u].w)
                   : "memory");
    }
    __syncthreads();
    tc_load_x(x, num_tokens, H, h, tile + gridDim.x, tid, raw);  // next tile (zeros past the end)

    // y[16 tokens of this warp][128] = x . (R_hi + R_mid + R_lo)
    float acc[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[n][c] = 0.f;
#pragma unroll 1
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(xt + swz(a_row, 2 * ks + a_hi), a0, a1, a2, a3);
#pragma unroll
      for (int part = 0; part < 3; ++part) {
#pragma unroll
        for (int np = 0; np < 8; ++np) {  // n-tiles 2np, 2np + 1
          uint32_t b0, b1, b2, b3;
          ldsm_x4(rt + part * 128 * 256 + swz(16 * np + b_row, 2 * ks + b_hi), b0, b1, b2, b3);
          mma_bf16_16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
          mma_bf16_16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }

    // Quantise from the accumulators.  Quad g of the warp holds tokens 16w + g (elements
    // 0, 1) and 16w + g + 8 (elements 2, 3); lane tq holds channels 8n + 2tq, 8n + 2tq + 1.
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int64_t t = t0 + 16 * warp + g + 8 * hf;
      int64_t slot = t < num_tokens ? __ldg(slots + t) : -1;
      if (slot >= static_cast<int64_t>(num_pages) * kPageSize) {
        if (tq == 0) record_error(OSCAR_DEVERR_SLOT);
        slot = -1;
      }
      uint32_t szw[NGRP];  // (scale, zero) of each group as stored: scale in the low half
      uint32_t nib[16];
#pragma unroll
      for (int j = 0; j < NGRP; ++j) {
        float mn = INFINITY, mx = -INFINITY;
#pragma unroll
        for (int n = j * NPG; n < (j + 1) * NPG; ++n)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float cl = __ldg(clip + 8 * n + 2 * tq + e);
            const float y = fminf(fmaxf(acc[n][2 * hf + e], -cl), cl);
            acc[n][2 * hf + e] = y;
            mn = fminf(mn, y);
            mx = fmaxf(mx, y);
          }
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const __half sh = __float2half_rn((mx - mn) / 3.0f);
        const __half zh = __float2half_rn(mn);
        szw[j] = static_cast<uint32_t>(__half_as_ushort(sh)) | (static_cast<uint32_t>(__half_as_ushort(zh)) << 16);
        const float s = __half2float(sh), z = __half2float(zh);
#pragma unroll
        for (int n = j * NPG; n < (j + 1) * NPG; ++n) {
          uint32_t c2 = 0;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            uint32_t code = 0;
            if (s != 0.f) {
              const float uq = (acc[n][2 * hf + e] - z) / s;
              code = static_cast<uint32_t>(fminf(fmaxf(rintf(uq), 0.f), 3.f));
            }
            c2 |= code << (2 * e);
          }
          nib[n] = c2;
        }
      }
      // Channel 8n + 2tq + e is byte 2n + tq / 2, bits 4 (tq & 1) + 2e: the quad's four
      // nibbles of n-tile n form 16 bits; n-tiles 2w, 2w + 1 form the row's word w.
      uint32_t word[8];
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        uint32_t vw = (nib[2 * w] | (nib[2 * w + 1] << 16)) << (4 * tq);
        vw |= __shfl_xor_sync(0xffffffffu, vw, 1);
        vw |= __shfl_xor_sync(0xffffffffu, vw, 2);
        word[w] = vw;
      }
      if (slot >= 0) {
        const int64_t page = slot / kPageSize;
        const int off = static_cast<int>(slot % kPageSize);
        const size_t row = ((static_cast<size_t>(page) * H + h) * 2 + kv) * kPageSize + off;
        uint32_t lo = word[0], hi = word[1];
#pragma unroll
        for (int q = 1; q < 4; ++q)
          if (tq == q) {
            lo = word[2 * q];
            hi = word[2 * q + 1];
          }
        reinterpret_cast<uint2*>(codes + row * (D / 4))[tq] = make_uint2(lo, hi);
        if (tq == 0) {  // the row's NGRP pairs in one store
          void* dst = sz + row * NGRP * 2;
          if constexpr (NGRP == 4) *static_cast<uint4*>(dst) = make_uint4(szw[0], szw[1], szw[2], szw[3]);
          if constexpr (NGRP == 2) *static_cast<uint2*>(dst) = make_uint2(szw[0], szw[1]);
          if constexpr (NGRP == 1) *static_cast<uint32_t*>(dst) = szw[0];
        }
      }
    }
  }
}

template <int G>
cudaError_t launch_append_tc(int64_t T, const oscar_dims_t* d, const void* k, const void* v, const float* R_k,
                             const float* R_v, const float* clip_k, const float* clip_v, const int64_t* slots,
                             uint8_t* codes, void* sz, const MixedDst& md, cudaStream_t stream) {
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(append_tc_kernel<G>), kTcSmem);
  if (e != cudaSuccess) return e;
  // Two CTAs per SM over all (head, K|V); each loops over its share of the token tiles.
  const int64_t ntiles = (T + kTcTok - 1) / kTcTok;
  const int hkv = 2 * d->num_kv_heads;
  int64_t per = (2 * static_cast<int64_t>(num_sms()) + hkv - 1) / hkv;
  if (per > ntiles) per = ntiles;
  const dim3 grid(static_cast<unsigned>(per), d->num_kv_heads, 2);
  append_tc_kernel<G><<<grid, kTcThreads, kTcSmem, stream>>>(
      T, d->num_kv_heads, d->num_pages, static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v),
      R_k, R_v, clip_k, clip_v, slots, codes, static_cast<__half*>(sz), md);
  return cudaGetLastError();
}

template <int D>
__global__ void __launch_bounds__(kThreads) append_small_kernel(
    int64_t num_tokens, int H, int G, int num_pages, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const float* __restrict__ R_k, const float* __restrict__ R_v,
    const float* __restrict__ clip_k, const float* __restrict__ clip_v, const int64_t* __restrict__ slots,
    uint8_t* __restrict__ codes, __half* __restrict__ sz, MixedDst md) {
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
  for (int i = threadIdx.x; i < kSmallTok * D / 2; i += kThreads) {
    const int tt = i / (D / 2), c2 = i % (D / 2);
    const int64_t t = t0 + tt;
    float2 val = make_float2(0.f, 0.f);
    if (t < num_tokens) {
      const __nv_bfloat162 raw = reinterpret_cast<const __nv_bfloat162*>(x + (static_cast<size_t>(t) * H + h) * D)[c2];
      val = __bfloat1622float2(raw);
      if (md.active() && dst_row[tt] >= 0)
        reinterpret_cast<__nv_bfloat162*>((dst_buf[tt] ? md.win : md.sink) + dst_row[tt])[c2] = raw;
    }
    xs[tt * D + 2 * c2] = val.x;
    xs[tt * D + 2 * c2 + 1] = val.y;
  }
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
                          const float* R_v, const float* clip_k, const float* clip_v, const int64_t* slots,
                          uint8_t* codes, void* sz, const MixedDst& md, cudaStream_t stream) {
  // Few tokens per (head, K|V): spread R's rows over warps instead of staging all of R.
  if (T <= kSmallTokenLimit) {
    const dim3 grid(static_cast<unsigned>((T + kSmallTok - 1) / kSmallTok), d->num_kv_heads, 2);
    append_small_kernel<D><<<grid, kThreads, 0, stream>>>(
        T, d->num_kv_heads, d->group_size, d->num_pages, static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(v), R_k, R_v, clip_k, clip_v, slots, codes, static_cast<__half*>(sz), md);
    return cudaGetLastError();
  }
  if constexpr (D == 128) {  // the rotation on tensor cores
    switch (d->group_size) {
      case 32: return launch_append_tc<32>(T, d, k, v, R_k, R_v, clip_k, clip_v, slots, codes, sz, md, stream);
      case 64: return launch_append_tc<64>(T, d, k, v, R_k, R_v, clip_k, clip_v, slots, codes, sz, md, stream);
      default: return launch_append_tc<128>(T, d, k, v, R_k, R_v, clip_k, clip_v, slots, codes, sz, md, stream);
    }
  }
  const size_t smem = (static_cast<size_t>(D) * D + kTokTile * D) * sizeof(float);
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(append_kernel<D>), smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((T + kTokTile - 1) / kTokTile), d->num_kv_heads, 2);
  append_kernel<D><<<grid, kThreads, smem, stream>>>(
      T, d->num_kv_heads, d->group_size, d->num_pages, static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), R_k, R_v, clip_k, clip_v, slots, codes, static_cast<__half*>(sz), md);
  return cudaGetLastError();
}

}  // namespace

namespace {

oscar_status_t run_append(const oscar_dims_t* dims, int64_t num_tokens, const void* k, const void* v,
                          const float* R_k, const float* R_v, const float* clip_k, const float* clip_v,
                          const int64_t* slot_mapping, uint8_t* int2_pages, void* scale_zero_pages,
                          const MixedDst& md, void* stream) {
  oscar_status_t st = check_dims(dims);
  if (st != OSCAR_OK) return st;
  if (num_tokens < 0) return OSCAR_ERR_INVALID_ARG;
  if (num_tokens == 0) return OSCAR_OK;
  if (!k || !v || !R_k || !R_v || !clip_k || !clip_v || !slot_mapping || !int2_pages || !scale_zero_pages)
    return OSCAR_ERR_INVALID_ARG;
  if (misaligned16(k) || misaligned16(v) || misaligned16(R_k) || misaligned16(R_v) || misaligned16(int2_pages) ||
      misaligned16(scale_zero_pages) || misaligned16(md.sink) || misaligned16(md.win))
    return OSCAR_ERR_INVALID_ARG;
  if ((num_tokens + kTokTile - 1) / kTokTile > 0x7fffffffLL) return OSCAR_ERR_UNSUPPORTED;
  cudaError_t e = dims->head_dim == 128
                      ? launch_append<128>(num_tokens, dims, k, v, R_k, R_v, clip_k, clip_v, slot_mapping,
                                           int2_pages, scale_zero_pages, md, as_stream(stream))
                      : launch_append<64>(num_tokens, dims, k, v, R_k, R_v, clip_k, clip_v, slot_mapping,
                                          int2_pages, scale_zero_pages, md, as_stream(stream));
  return e == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

}  // namespace

extern "C" oscar_status_t oscar_append(const oscar_dims_t* dims, int64_t num_tokens, const void* k, const void* v,
                                       const float* R_k, const float* R_v, const float* clip_k,
                                       const float* clip_v, const int32_t* page_table,
                                       const int64_t* slot_mapping, uint8_t* int2_pages, void* scale_zero_pages,
                                       void* stream) {
  (void)page_table;
  return run_append(dims, num_tokens, k, v, R_k, R_v, clip_k, clip_v, slot_mapping, int2_pages, scale_zero_pages,
                    MixedDst{}, stream);
}

extern "C" oscar_status_t oscar_append_mixed(const oscar_dims_t* dims, int64_t num_tokens, const void* k,
                                             const void* v, const float* R_k, const float* R_v,
                                             const float* clip_k, const float* clip_v, const int32_t* page_table,
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
  return run_append(dims, num_tokens, k, v, R_k, R_v, clip_k, clip_v, slot_mapping, int2_pages, scale_zero_pages,
                    md, stream);
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
