// Shared pieces of the split-KV decode kernels: the split plan, kernel
// parameters, programmatic-dependent-launch helpers, and the CUDA-core split
// body and merge kernel (used for the BF16 sink/window splits, the BF16 paged
// reference and the shapes the tensor-core kernels do not cover).
#pragma once

#include <math.h>

#include "common.cuh"
#include "ptx.cuh"

namespace oscar_dec {

using namespace oscar;

constexpr int kThreads = 128;
constexpr int kTile = 32;        // positions per softmax tile (one per lane)
constexpr int kBf16Chunk = 32;   // sink/window positions per split (one softmax tile)
constexpr size_t kMergeStageMax = 96 * 1024;    // partials staged in the merge's shared memory up to this size
constexpr size_t kMergeSmemLimit = 200 * 1024;  // dynamic shared-memory limit set for the merge kernel

enum Mode { kMixed = 0, kBf16Paged = 1 };

struct Plan {
  int pps = 0;         // pages per INT2 (or BF16-paged) split
  int n_paged = 0;     // splits over the paged pool
  int n_dense = 0;     // splits over the BF16 sink/window buffers
  int ns = 0;          // n_paged + n_dense
  size_t off_qrot = 0, off_po = 0, off_pml = 0, total = 0;
};

struct Params {
  int B, Hq, H, D, G, gqa, num_pages, max_pages, max_seq_len;
  int S, W, pps, n_paged, n_dense, ns;
  float scale_log2;
  int merge_stage;  // 1: the merge kernel stages the split partials in shared memory
  const __nv_bfloat16* q;
  const float* R_k;
  const float* R_v;
  const uint8_t* codes;       // INT2 pool (mixed mode)
  const __half* sz;           // scale/zero pool (mixed mode)
  const __nv_bfloat16* sink;  // [B][2][H][S][D]
  const __nv_bfloat16* win;   // [B][2][H][W][D]
  const __nv_bfloat16* pages; // BF16 pool (BF16 mode)
  const int32_t* page_table;
  const int32_t* seq_lens;
  float* out;
  float* q_rot;
  float* part_o;
  float* part_ml;
};

// Tensor-core split kernels for the shapes they cover (decode_int2_mma.cu,
// decode_bf16_mma.cu).
bool int2_mma_supported(const Params& p);
cudaError_t int2_mma_split(const Params& p, cudaStream_t stream);
bool bf16_mma_supported(const Params& p);
cudaError_t bf16_mma_split(const Params& p, cudaStream_t stream);

// Launches `kernel` with programmatic stream serialisation: it may overlap the
// tail of the preceding kernel in the stream and must call grid_dep_wait()
// before reading that kernel's output.
template <typename... Args>
cudaError_t launch_pdl(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// grid_dep_wait() blocks until the preceding kernel has completed and its
// writes are visible (a no-op without a programmatic dependency);
// grid_dep_launch_dependents() lets the following kernel start launching.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

namespace {  // internal linkage in every unit that includes this header

bool make_plan(const oscar_dims_t* d, int B, int max_seq_len, int pps_req, int S, int W, Mode mode, Plan* p) {
  if (B < 0 || max_seq_len < 0 || pps_req < 0 || S < 0 || W < 0) return false;
  if (max_seq_len > d->max_pages_per_seq * kPageSize) return false;
  const int max_pages = (max_seq_len + kPageSize - 1) / kPageSize;
  int pps = pps_req;
  if (pps == 0) {
    const long long units = static_cast<long long>(B) * d->num_kv_heads;
    long long want = (static_cast<long long>(max_pages) * units + 2LL * num_sms() - 1) / (2LL * num_sms());
    if (want < 8) want = 8;
    if (want > 64) want = 64;
    pps = static_cast<int>(want);
  }
  p->pps = pps;
  p->n_paged = max_pages == 0 ? 0 : (max_pages + pps - 1) / pps;
  const int dense = mode == kMixed ? (S + W < max_seq_len ? S + W : max_seq_len) : 0;
  p->n_dense = (dense + kBf16Chunk - 1) / kBf16Chunk;
  p->ns = p->n_paged + p->n_dense;
  if (p->ns == 0) p->ns = 1;
  const size_t bh = static_cast<size_t>(B) * d->num_q_heads;
  size_t off = 0;
  p->off_qrot = off;
  if (mode == kMixed) off += align_up(bh * d->head_dim * sizeof(float), 256);
  p->off_po = off;
  off += align_up(bh * p->ns * d->head_dim * sizeof(float), 256);
  p->off_pml = off;
  off += align_up(bh * p->ns * 2 * sizeof(float), 256);
  p->total = off;
  return true;
}

__device__ __forceinline__ int clamp_len(const Params& p, int b) {
  int L = p.seq_lens[b];
  if (L < 0 || L > p.max_seq_len) {
    record_error(OSCAR_DEVERR_SEQ_LEN);
    L = L < 0 ? 0 : p.max_seq_len;
  }
  return L;
}

// q_rot[b][hq] = q[b][hq] . R_k[h] for the GQA query heads hq of one (b, h):
// R_k[h] arrives in shared memory by one bulk copy and thread j computes column
// j for every query head.  Dynamic shared memory: qrot_smem(D) bytes.
constexpr size_t qrot_smem(int D) { return static_cast<size_t>(D) * D * 4 + static_cast<size_t>(kMaxGqa) * D * 4 + 16; }

constexpr int kQrotThreads = 512;  // 4 groups of 128 threads, each summing a quarter of the rows

template <int D>
__global__ void __launch_bounds__(kQrotThreads) qrot_kernel(Params p) {
  extern __shared__ __align__(128) float qsm[];
  float* Rs = qsm;                 // [D][D]
  float* qs = Rs + D * D;          // [gqa][D]
  uint64_t* bar = reinterpret_cast<uint64_t*>(qs + kMaxGqa * D);
  grid_dep_launch_dependents();
  const int b = blockIdx.x / p.H, h = blockIdx.x % p.H;
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(smem_u32(bar), 1);
    mbar_init_fence();
    mbar_arrive_expect_tx(smem_u32(bar), D * D * 4);
    bulk_g2s(smem_u32(Rs), p.R_k + static_cast<size_t>(h) * D * D, D * D * 4, smem_u32(bar));
  }
  const size_t q0 = (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(h) * p.gqa) * D;
  for (int i = tid; i < p.gqa * D; i += kQrotThreads) qs[i] = __bfloat162float(p.q[q0 + i]);
  __syncthreads();
  if (!mbar_wait_bounded(smem_u32(bar), 0)) {
    if (tid == 0) record_error(OSCAR_DEVERR_TIMEOUT);
    mbar_wait_bounded(smem_u32(bar), 0);  // give a late copy one more bounded chance to land
  }
  // Thread (quarter qt, column j) sums rows [qt*D/4, (qt+1)*D/4); the quarters are
  // then added in order through shared memory (the R_k area is no longer needed).
  const int j = tid % D, qt = tid / D;
  constexpr int kGroups = kQrotThreads / D;
  float acc[kMaxGqa];
#pragma unroll
  for (int qi = 0; qi < kMaxGqa; ++qi) acc[qi] = 0.f;
  if (qt < kGroups) {
    const int i0 = qt * (D / kGroups);
#pragma unroll 4
    for (int i = i0; i < i0 + D / kGroups; ++i) {
      const float r = Rs[i * D + j];
#pragma unroll
      for (int qi = 0; qi < kMaxGqa; ++qi)
        if (qi < p.gqa) acc[qi] = fmaf(qs[qi * D + i], r, acc[qi]);
    }
  }
  __syncthreads();
  float* part = Rs;  // [kGroups][kMaxGqa][D]
  if (qt < kGroups) {
#pragma unroll
    for (int qi = 0; qi < kMaxGqa; ++qi)
      if (qi < p.gqa) part[(qt * kMaxGqa + qi) * D + j] = acc[qi];
  }
  __syncthreads();
  for (int idx = tid; idx < p.gqa * D; idx += kQrotThreads) {
    const int qi = idx / D, jj = idx % D;
    float tot = 0.f;
#pragma unroll
    for (int g = 0; g < kGroups; ++g) tot += part[(g * kMaxGqa + qi) * D + jj];
    p.q_rot[q0 + idx] = tot;
  }
}

// Shared memory (bytes) of split_body for head dimension D.
constexpr size_t split_body_smem(int D) {
  return sizeof(float) * (static_cast<size_t>(kMaxGqa) * D + 2 * kTile * (D + 1) + kMaxGqa * kTile + 3 * kMaxGqa) +
         sizeof(int) * 2 * kTile;
}

// CUDA-core split: one CTA of kThreads threads attends positions of split s of
// (sequence b, KV head h) for all its GQA query heads.  `smem` provides
// split_body_smem(D) bytes (16-byte aligned).
template <int D, Mode MODE>
__device__ __forceinline__ void split_body(const Params& p, int s, int h, int b, float* smem) {
  constexpr int DP = D + 1;  // padded row: conflict-free column reads
  float* qv = smem;
  float* kt = qv + kMaxGqa * D;
  float* vt = kt + kTile * DP;
  float* pr = vt + kTile * DP;
  float* alpha_s = pr + kMaxGqa * kTile;
  float* m_s = alpha_s + kMaxGqa;
  float* l_s = m_s + kMaxGqa;
  int* page_s = reinterpret_cast<int*>(l_s + kMaxGqa);
  int* pos_s = page_s + kTile;

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int gqa = p.gqa;
  grid_dep_launch_dependents();
  grid_dep_wait();  // q_rot comes from the preceding kernel
  const int L = clamp_len(p, b);

  // Position range of this split.
  const bool paged = s < p.n_paged;
  int begin = 0, count = 0;         // paged: absolute positions [begin, begin+count)
  int sink_end = 0, win_begin = 0;  // dense: enumerated sink then window
  if (MODE == kMixed) {
    sink_end = min(p.S, L);
    win_begin = max(p.S, L - p.W);
  }
  if (paged) {
    const int lo = s * p.pps * kPageSize, hi = lo + p.pps * kPageSize;
    const int r0 = MODE == kMixed ? max(lo, p.S) : lo;
    const int r1 = MODE == kMixed ? min(hi, win_begin) : min(hi, L);
    begin = r0;
    count = max(0, r1 - r0);
  } else {
    const int n_dense = sink_end + max(0, L - win_begin);
    begin = (s - p.n_paged) * kBf16Chunk;
    count = max(0, min(kBf16Chunk, n_dense - begin));
  }

  const bool rotated = MODE == kMixed && paged;
  for (int i = tid; i < gqa * D; i += kThreads) {
    const size_t qi = (static_cast<size_t>(b) * p.Hq + h * gqa) * D + i;
    qv[i] = (rotated ? p.q_rot[qi] : __bfloat162float(p.q[qi])) * p.scale_log2;
  }
  if (tid < kMaxGqa) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
  }
  float o_acc[kMaxGqa];
#pragma unroll
  for (int k = 0; k < kMaxGqa; ++k) o_acc[k] = 0.f;
  __syncthreads();

  for (int t0 = 0; t0 < count; t0 += kTile) {
    // Resolve the position and (for paged data) the physical page of each lane's token.
    if (tid < kTile) {
      const int e = t0 + tid;
      int page = -1, pos = -1;
      if (e < count) {
        if (paged) {
          pos = begin + e;
          page = p.page_table[static_cast<size_t>(b) * p.max_pages + pos / kPageSize];
          if (page < 0 || page >= p.num_pages) {
            record_error(OSCAR_DEVERR_PAGE_ID);
            page = -1;
            pos = -1;
          }
        } else {
          const int idx = begin + e;
          pos = idx < sink_end ? idx : win_begin + (idx - sink_end);
        }
      }
      page_s[tid] = page;
      pos_s[tid] = pos;
    }
    __syncthreads();
    // Load (and dequantise) K and V of the tile into shared memory, 16 channels per
    // item: all global loads of the thread are issued first, then converted.
    constexpr int kItems = 2 * kTile * (D / 16);
    constexpr int kPer = (kItems + kThreads - 1) / kThreads;
    uint4 raw[kPer][2];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int w = tid + k * kThreads;
      raw[k][0] = make_uint4(0u, 0u, 0u, 0u);
      raw[k][1] = make_uint4(0u, 0u, 0u, 0u);
      if (w >= kItems) continue;
      const int kvsel = w / (kTile * (D / 16));
      const int rem = w % (kTile * (D / 16));
      const int tt = rem / (D / 16), word = rem % (D / 16);
      const int pos = pos_s[tt];
      if (pos < 0) continue;
      if (MODE == kMixed && paged) {
        const size_t row = ((static_cast<size_t>(page_s[tt]) * p.H + h) * 2 + kvsel) * kPageSize + pos % kPageSize;
        const int g = word * 16 / p.G;
        raw[k][0].x = __ldg(reinterpret_cast<const uint32_t*>(p.codes + row * (D / 4)) + word);
        raw[k][0].y = __ldg(reinterpret_cast<const unsigned int*>(p.sz + row * (D / p.G) * 2) + g);
      } else {
        const __nv_bfloat16* src;
        if (MODE == kBf16Paged) {
          src = p.pages + (((static_cast<size_t>(page_s[tt]) * p.H + h) * 2 + kvsel) * kPageSize + pos % kPageSize) * D;
        } else if (pos < sink_end) {
          src = p.sink + (((static_cast<size_t>(b) * 2 + kvsel) * p.H + h) * p.S + pos) * D;
        } else {
          src = p.win + (((static_cast<size_t>(b) * 2 + kvsel) * p.H + h) * p.W + pos % p.W) * D;
        }
        const uint4* s4 = reinterpret_cast<const uint4*>(src + word * 16);
        raw[k][0] = __ldg(s4);
        raw[k][1] = __ldg(s4 + 1);
      }
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int w = tid + k * kThreads;
      if (w >= kItems) continue;
      const int kvsel = w / (kTile * (D / 16));
      const int rem = w % (kTile * (D / 16));
      const int tt = rem / (D / 16), word = rem % (D / 16);
      float vals[16];
      if (MODE == kMixed && paged) {
        const uint32_t bits = raw[k][0].x;
        const uint32_t szb = raw[k][0].y;
        const float sc = __half2float(__ushort_as_half(static_cast<unsigned short>(szb & 0xffffu)));
        const float ze = __half2float(__ushort_as_half(static_cast<unsigned short>(szb >> 16)));
        const bool ok = pos_s[tt] >= 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) vals[i] = ok ? fmaf(static_cast<float>((bits >> (2 * i)) & 3u), sc, ze) : 0.f;
      } else {
        const uint32_t wds[8] = {raw[k][0].x, raw[k][0].y, raw[k][0].z, raw[k][0].w,
                                 raw[k][1].x, raw[k][1].y, raw[k][1].z, raw[k][1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          vals[2 * i] = bf16_bits_to_float(wds[i] & 0xffffu);
          vals[2 * i + 1] = bf16_bits_to_float(wds[i] >> 16);
        }
      }
      float* dst = (kvsel ? vt : kt) + tt * DP + word * 16;
#pragma unroll
      for (int i = 0; i < 16; ++i) dst[i] = vals[i];
    }
    __syncthreads();
    // Logits (log2 units) of every (query, token) pair of the tile.
    for (int pi = tid; pi < gqa * kTile; pi += kThreads) {
      const int qi = pi / kTile, tt = pi % kTile;
      float dot = 0.f;
#pragma unroll 8
      for (int i = 0; i < D; ++i) dot = fmaf(qv[qi * D + i], kt[tt * DP + i], dot);
      pr[pi] = pos_s[tt] >= 0 ? dot : -INFINITY;
    }
    __syncthreads();
    // Online softmax: one warp per query head, one lane per token.
    for (int qi = warp; qi < gqa; qi += kThreads / 32) {
      const float sc = pr[qi * kTile + lane];
      float mx = sc;
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_old = m_s[qi];
      const float m_new = fmaxf(m_old, mx);
      float pv = 0.f, alpha = 1.f;
      if (m_new != -INFINITY) {
        pv = exp2f(sc - m_new);
        alpha = exp2f(m_old - m_new);
      }
      float sum = pv;
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      pr[qi * kTile + lane] = pv;
      __syncwarp();
      if (lane == 0) {
        l_s[qi] = l_s[qi] * alpha + sum;
        m_s[qi] = m_new;
        alpha_s[qi] = alpha;
      }
    }
    __syncthreads();
    // o[q][d] = o[q][d] * alpha[q] + sum_t p[q][t] v[t][d]
#pragma unroll
    for (int k = 0; k < kMaxGqa; ++k) {
      const int pi = tid + k * kThreads;
      if (pi < gqa * D) {
        const int qi = pi / D, dd = pi % D;
        float acc = o_acc[k] * alpha_s[qi];
#pragma unroll 8
        for (int tt = 0; tt < kTile; ++tt) acc = fmaf(pr[qi * kTile + tt], vt[tt * DP + dd], acc);
        o_acc[k] = acc;
      }
    }
    __syncthreads();
  }

  // Partial results of this split.
#pragma unroll
  for (int k = 0; k < kMaxGqa; ++k) {
    const int pi = tid + k * kThreads;
    if (pi < gqa * D) {
      const int qi = pi / D, dd = pi % D;
      const size_t bh = static_cast<size_t>(b) * p.Hq + h * gqa + qi;
      p.part_o[(bh * p.ns + s) * D + dd] = o_acc[k];
    }
  }
  if (tid < gqa) {
    const size_t bh = static_cast<size_t>(b) * p.Hq + h * gqa + tid;
    p.part_ml[(bh * p.ns + s) * 2 + 0] = m_s[tid];
    p.part_ml[(bh * p.ns + s) * 2 + 1] = l_s[tid];
  }
}

template <int D, Mode MODE>
__global__ void __launch_bounds__(kThreads) split_kernel(Params p) {
  extern __shared__ __align__(16) float dyn_smem[];
  split_body<D, MODE>(p, blockIdx.x, blockIdx.y, blockIdx.z, dyn_smem);
}

// Log-sum-exp merge of the splits of one (b, hq), un-rotation of the INT2 part
// by R_v^T and normalisation.  R_v[h] (mixed mode) is staged by a bulk copy
// before the wait for the split kernel, the partials by a second bulk copy
// after it (when they fit, merge_stage).  Dynamic shared memory:
// merge_smem(D, ns, mixed, stage) bytes.
constexpr size_t merge_smem(int D, int ns, bool mixed, bool stage) {
  return (mixed ? static_cast<size_t>(D) * D * 4 : 0) + (stage ? static_cast<size_t>(ns) * D * 4 : 0) +
         static_cast<size_t>(ns + 2) * 4 + 32;
}

template <int D, Mode MODE>
__global__ void __launch_bounds__(kThreads) merge_kernel(Params p) {
  __shared__ float o_rot[D];
  __shared__ float o_plain[D];
  __shared__ float red[kThreads / 32];
  extern __shared__ __align__(128) float msm[];
  constexpr bool kRot = MODE == kMixed;
  const int ns = p.ns;
  float* Rs = msm;                                      // [D][D] (mixed)
  float* po_s = Rs + (kRot ? D * D : 0);                // [ns][D] (staged)
  float* wts = po_s + (p.merge_stage ? ns * D : 0);     // [ns]
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uintptr_t>(wts + ns + 2 + 1) & ~uintptr_t(7));
  const int bh = blockIdx.x;
  const int h = (bh % p.Hq) / p.gqa;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  if (tid == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    mbar_init_fence();
    if (kRot) {
      mbar_arrive_expect_tx(smem_u32(&bars[0]), D * D * 4);
      bulk_g2s(smem_u32(Rs), p.R_v + static_cast<size_t>(h) * D * D, D * D * 4, smem_u32(&bars[0]));
    }
  }
  __syncthreads();
  grid_dep_wait();  // the split partials come from the preceding kernel
  const float* ml = p.part_ml + static_cast<size_t>(bh) * ns * 2;
  const float* po = p.part_o + static_cast<size_t>(bh) * ns * D;
  if (tid == 0 && p.merge_stage) {
    mbar_arrive_expect_tx(smem_u32(&bars[1]), ns * D * 4);
    bulk_g2s(smem_u32(po_s), po, ns * D * 4, smem_u32(&bars[1]));
  }
  // M = max_s m_s, weights w_s = 2^(m_s - M), denominator sum_s w_s l_s.
  float M = -INFINITY;
  for (int s = tid; s < ns; s += kThreads) M = fmaxf(M, ml[2 * s]);
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) M = fmaxf(M, red[w]);
  __syncthreads();
  float den = 0.f;
  for (int s = tid; s < ns; s += kThreads) {
    const float m = ml[2 * s];
    const float w = (m == -INFINITY || M == -INFINITY) ? 0.f : fast_exp2(m - M);
    wts[s] = w;
    den = fmaf(w, ml[2 * s + 1], den);
  }
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  if (lane == 0) red[warp] = den;
  __syncthreads();
  den = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) den += red[w];
  bool ok = true;
  if (p.merge_stage) ok = mbar_wait_bounded(smem_u32(&bars[1]), 0);
  if (!ok && tid == 0) record_error(OSCAR_DEVERR_TIMEOUT);
  const float* src = p.merge_stage ? po_s : po;
  if (tid < D) {
    float a_rot = 0.f, a_plain = 0.f;
    const int n_rot = kRot ? p.n_paged : 0;
#pragma unroll 4
    for (int s = 0; s < n_rot; ++s) a_rot = fmaf(wts[s], src[static_cast<size_t>(s) * D + tid], a_rot);
#pragma unroll 4
    for (int s = n_rot; s < ns; ++s) a_plain = fmaf(wts[s], src[static_cast<size_t>(s) * D + tid], a_plain);
    o_rot[tid] = a_rot;
    o_plain[tid] = a_plain;
  }
  __syncthreads();
  const float inv = (ok && den > 0.f) ? 1.f / den : 0.f;
  float* out = p.out + static_cast<size_t>(bh) * D;
  if (!kRot) {
    if (tid < D) out[tid] = o_plain[tid] * inv;
    return;
  }
  if (!mbar_wait_bounded(smem_u32(&bars[0]), 0)) {
    if (tid == 0) record_error(OSCAR_DEVERR_TIMEOUT);
    if (tid < D) out[tid] = 0.f;
    return;
  }
  // out[c] = (o_plain[c] + sum_j o_rot[j] R_v[h][c][j]) * inv, thread c.  Thread c
  // visits j in the order (c + k) mod D, so at every step the 32 lanes of a warp
  // read 32 different banks of R_v's row-major rows and of o_rot.
  if (tid < D) {
    const int c = tid;
    float part = 0.f;
#pragma unroll 8
    for (int k = 0; k < D; ++k) {
      const int j = (c + k) & (D - 1);
      part = fmaf(o_rot[j], Rs[c * D + j], part);
    }
    out[c] = (o_plain[c] + part) * inv;
  }
}

}  // namespace
}  // namespace oscar_dec
