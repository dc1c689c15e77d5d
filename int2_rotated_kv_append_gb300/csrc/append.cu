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
