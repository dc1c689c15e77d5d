// The current token's append inside a decode (oscar_append_decode): used by the
// single-wave fused decode and by the general split kernel, in the CTA that
// attends the sink/window rows holding that token.
#pragma once

#include "int2_page.cuh"

namespace oscar_dec {
namespace {

// oscar_append_decode's fused form, in the CTA that attends the sink/window rows
// holding the current token of sequence b (position L - 1, L = seq_lens[b]), for KV
// head h.  The token is appended as oscar_append_mixed appends it: K (minus the key
// offset, in fp32) and V rotated by R_k[h] and R_v[h] (y_j = sum_i x_i R[i][j], in
// the few-token append kernel's order of operations), clipped, quantised
// per group of G channels (fp16 scale (max - min) / 3 and zero min, codes
// rint((y - zero) / scale) clamped to 0..3, 0 when the scale is 0) and written to the
// pool row of slot_mapping[b]; the BF16 rows (the offset key rounded to bf16, and V)
// go to the sink row or the window slot of position L - 1.  No INT2 split reads that
// position (with a window it lies in the sink or the window), and the BF16 rows are
// written before this CTA's own sink/window copies read them.
template <int NW>
__device__ __forceinline__ void fused_append_token(const Params& p, int b, int h, uint8_t* smem) {
  constexpr int T = NW * 32;  // 128 .. 512 threads
  // x . R summed as the few-token append kernel sums it, so that the codes equal
  // those of oscar_append_mixed on the same token bit for bit: 8 slices of 16 rows,
  // each an fma chain in row order from 0 (lane l: channels 4l .. 4l + 3), the
  // slices then added in order.  Warp w takes the (K|V, slice) tasks w, w + NW, ...
  constexpr int kSlices = 8, kSliceRows = kD / kSlices, kChunk = 8;
  float* xs = reinterpret_cast<float*>(smem);  // [2][kD]: the token's K (offset) and V
  float* part = xs + 2 * kD;                   // [2][kSlices][kD]: per-slice partial sums
  float* cmn = part + 2 * kSlices * kD;        // [2][4]: min of each 32-channel chunk
  float* cmx = cmn + 8;                        // [2][4]: max
  float* ys = cmx + 8;                         // [2][kD]: the clipped rotated values
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  grid_dep_wait();  // the previous step's reads of the window row this token replaces are over
  const int64_t slot = __ldg(p.app_slots + b);  // a negative slot: the token is skipped entirely
  if (slot < 0) return;
  const int L = __ldg(p.seq_lens + b);
  const int pos = L - 1;
  // as oscar_append_mixed at position L - 1: a sequence of length < 1 has no row for
  // the token (flagged; its codes are still written at the slot)
  if (pos < 0 && tid == 0) record_error(OSCAR_DEVERR_POSITION);
  for (int i = tid; i < kD; i += T) {  // (K|V, channel pair)
    const int kv = i >> 6, c2 = i & 63;
    const __nv_bfloat16* x = (kv ? p.app_v : p.app_k) + (static_cast<size_t>(b) * p.H + h) * kD;
    __nv_bfloat162 raw = reinterpret_cast<const __nv_bfloat162*>(x)[c2];
    float2 val = __bfloat1622float2(raw);
    if (kv == 0 && p.app_offset_k != nullptr) {
      const float2 c = __ldg(reinterpret_cast<const float2*>(p.app_offset_k + static_cast<size_t>(h) * kD) + c2);
      val = make_float2(__fsub_rn(val.x, c.x), __fsub_rn(val.y, c.y));
      raw = __floats2bfloat162_rn(val.x, val.y);
    }
    xs[kv * kD + 2 * c2] = val.x;
    xs[kv * kD + 2 * c2 + 1] = val.y;
    __nv_bfloat16* dst = nullptr;
    if (pos < 0)
      dst = nullptr;
    else if (pos < p.S)
      dst = p.app_sink + (((static_cast<size_t>(b) * 2 + kv) * p.H + h) * p.S + pos) * kD;
    else if (p.W > 0 && pos >= max(p.S, L - p.W))
      dst = p.app_win + (((static_cast<size_t>(b) * 2 + kv) * p.H + h) * p.W + pos % p.W) * kD;
    if (dst != nullptr) reinterpret_cast<__nv_bfloat162*>(dst)[c2] = raw;
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");  // the rows, for this CTA's bulk copies
  __syncthreads();
#pragma unroll 1
  for (int task = warp; task < 2 * kSlices; task += NW) {
    const int kv = task / kSlices, sl = task % kSlices;
    const float* R = (kv ? p.R_v : p.R_k) + static_cast<size_t>(h) * kD * kD +
                     static_cast<size_t>(sl * kSliceRows) * kD + 4 * lane;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int r0 = 0; r0 < kSliceRows; r0 += kChunk) {  // the rows' loads in two rounds (registers)
      float4 rr[kChunk];
#pragma unroll
      for (int r = 0; r < kChunk; ++r) rr[r] = __ldg(reinterpret_cast<const float4*>(R + (r0 + r) * kD));
#pragma unroll
      for (int r = 0; r < kChunk; ++r) {
        const float xv = xs[kv * kD + sl * kSliceRows + r0 + r];
        acc.x = fmaf(xv, rr[r].x, acc.x);
        acc.y = fmaf(xv, rr[r].y, acc.y);
        acc.z = fmaf(xv, rr[r].z, acc.z);
        acc.w = fmaf(xv, rr[r].w, acc.w);
      }
    }
    *reinterpret_cast<float4*>(part + (kv * kSlices + sl) * kD + 4 * lane) = acc;
  }
  __syncthreads();
  // items (K|V, channel) 0 .. 255 in blocks of T threads; a warp holds 32 consecutive channels
#pragma unroll 1
  for (int it = tid; it < 2 * kD; it += T) {
    const int kv = it >> 7, j = it & (kD - 1);
    float y = 0.f;
#pragma unroll
    for (int sl = 0; sl < kSlices; ++sl) y += part[(kv * kSlices + sl) * kD + j];
    const float cl = __ldg((kv ? p.app_clip_v : p.app_clip_k) + static_cast<size_t>(h) * kD + j);
    y = fminf(fmaxf(y, -cl), cl);
    ys[it] = y;
    float mn = y, mx = y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (lane == 0) {
      cmn[kv * 4 + (j >> 5)] = mn;
      cmx[kv * 4 + (j >> 5)] = mx;
    }
  }
  __syncthreads();
#pragma unroll 1
  for (int it = tid; it < 2 * kD; it += T) {
    const int kv = it >> 7, j = it & (kD - 1);
    const float y = ys[it];
    const int G = p.G, ng = kD / G, g = j / G;
    float mn = INFINITY, mx = -INFINITY;
    for (int c = g * G / 32; c < (g + 1) * G / 32; ++c) {
      mn = fminf(mn, cmn[kv * 4 + c]);
      mx = fmaxf(mx, cmx[kv * 4 + c]);
    }
    const __half sh = __float2half_rn((mx - mn) / 3.0f), zh = __float2half_rn(mn);
    const float sc = __half2float(sh), z = __half2float(zh);
    uint32_t code = 0;
    if (sc != 0.f) code = static_cast<uint32_t>(fminf(fmaxf(rintf((y - z) / sc), 0.f), 3.f));
    uint32_t wv = code << (2 * (j & 15));  // 16 channels per 32-bit word, channel j at bits 2 (j % 16)
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) wv |= __shfl_xor_sync(0xffffffffu, wv, o);
    if (slot < static_cast<int64_t>(p.num_pages) * kPageSize) {
      const size_t row =
          ((static_cast<size_t>(slot / kPageSize) * p.H + h) * 2 + kv) * kPageSize + static_cast<size_t>(slot % kPageSize);
      if ((j & 15) == 0) reinterpret_cast<uint32_t*>(p.app_codes + row * (kD / 4))[j >> 4] = wv;
      if (j % G == 0) reinterpret_cast<__half2*>(p.app_sz + row * ng * 2)[g] = __halves2half2(sh, zh);
    } else if (it == 0) {
      record_error(OSCAR_DEVERR_SLOT);
    }
  }
  __syncthreads();  // the shared memory holds the sink/window stages next
}

// The index of the dense CTA (of `per` 16-row sink/window pages each, in the order
// dense_part takes them: sink pages, then window pages) whose pages hold position
// L - 1 of sequence b (L = seq_lens[b] as given, as oscar_append_mixed takes it);
// CTA 0 when L < 1 (the token has no row: that CTA writes its codes and flags it);
// -1 when the position is past the sink and there is no window.  Waits for the
// preceding kernel first (the lengths are read after it, as everywhere).
__device__ __forceinline__ int current_token_dense_cta(const Params& p, int b, int per) {
  grid_dep_launch_dependents();
  grid_dep_wait();
  const int L = __ldg(p.seq_lens + b);
  if (L < 1) return 0;
  const int pos = L - 1;
  if (pos < p.S) return (pos / kPageSize) / per;
  if (p.W < 1) return -1;
  return ((p.S + kPageSize - 1) / kPageSize + (pos % p.W) / kPageSize) / per;
}

}  // namespace
}  // namespace oscar_dec
