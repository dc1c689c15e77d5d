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
// Per (sequence, KV head): the QK B-fragments of the tensor-core INT2 kernel for
// each of the 32 lanes (2 n-tiles x 8 k-steps x 2 words) and the lane's per-query
// factors (2 n-tiles x (score factor + 4 column-block sums)), 44 words per lane.
constexpr int kQfragWords = 44;
constexpr int kQfragBytes = 32 * kQfragWords * 4;
constexpr size_t kMergeSmemLimit = 160 * 1024;  // dynamic shared-memory limit set for the merge kernel

enum Mode { kMixed = 0, kBf16Paged = 1 };

constexpr int kDenseMmaPages = 8;  // 16-row sink/window pages per dense split of the tensor-core kernel
constexpr int kMmaMaxPps = 256;    // largest split the tensor-core kernels stage page ids for
constexpr int kMinFusedSplits = 8; // fewest INT2 split CTAs per unit for the automatic fused plan
constexpr int kFusedMaxPps = 960;      // most pages per split CTA for that plan (16 warps, GQA <= 4)
constexpr int kFusedMaxPpsGqa8 = 512;  // the same for GQA 8 (8 warps)

struct Plan {
  int pps = 0;         // pages per INT2 (or BF16-paged) split
  int n_paged = 0;     // splits over the paged pool
  int n_dense = 0;     // splits over the BF16 sink/window buffers
  int ns = 0;          // n_paged + n_dense
  int ml_ns = 0;       // row stride (splits) of the (m, l) partials: ns rounded up to even (16-byte rows)
  int mma = 0;         // 1: the tensor-core split kernel runs (dense splits of kDenseMmaPages pages)
  int fused = 0;       // 1: the single-wave fused decode (decode_fused.cu) runs
  int bulk_lo = 0;     // fused: first page of INT2 split 0 (splits cover the bulk pages only)
  size_t off_qrot = 0, off_qfrag = 0, off_po = 0, off_pml = 0, total = 0;
};

struct Params {
  int B, Hq, H, D, G, gqa, num_pages, max_pages, max_seq_len;
  int S, W, pps, n_paged, n_dense, ns, ml_ns;
  float scale_log2;
  int merge_qpc;    // query heads per merge CTA (divides gqa, or merge_spc * gqa)
  int merge_spc;    // sequences per merge CTA: 1, or > 1 for the large-batch form (merge_qpc = spc * gqa)
  int qrot_spc;     // sequences per q-rotation CTA (qrot_spc * gqa <= kQrotMaxQ)
  int merge_stage;  // merge kernel: kStageRv (R_v staged before the wait) | kStagePartials
  int mma;          // 1: tensor-core split kernel (INT2 mode: head_dim 128, group 64 or 128)
  // Fused single-wave decode (decode_fused.cu): n_paged INT2 split CTAs per unit starting
  // at page bulk_lo, then n_dense (0 or 1) BF16 CTAs covering n_dense_pages 16-row pages.
  int fused, bulk_lo, n_dense_pages;
  // > 0 only under oscar_test_stall_page_waits: each INT2 split warp waits for its
  // first page on a barrier phase that never completes and gives up after this many
  // cycles, taking the kernels' timeout path.
  long long stall_cycles;
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
  // Extend rows (null for a decode): query row b belongs to sequence row_seq[b]
  // (< num_seqs) and attends positions 0 .. row_pos[b] of it.
  const int32_t* row_seq;
  const int32_t* row_pos;
  int num_seqs;
  int split_base;             // first split index of the launch (the grid's x covers splits split_base ..)
  // Extend in tiles (int2_umma_tile_split): the rows of sequence b are q_start[b] .. q_start[b + 1) - 1,
  // in tiles of 64 / gqa rows, `tiles` per sequence.
  const int32_t* q_start;
  int tiles;
  float* out;
  // oscar_append_decode's fused form: the current token of sequence b (position
  // seq_lens[b] - 1) is appended by the unit's BF16 CTA (null app_k: no append)
  const __nv_bfloat16* app_k;  // [B][H][D]
  const __nv_bfloat16* app_v;
  const float* app_clip_k;     // [H][D]
  const float* app_clip_v;
  const float* app_offset_k;   // [H][D] or null
  const int64_t* app_slots;    // [B]
  uint8_t* app_codes;          // the INT2 pool (the same as codes)
  __half* app_sz;              // the scale/zero pool (the same as sz)
  __nv_bfloat16* app_sink;     // the sink and window buffers (the same as sink, win)
  __nv_bfloat16* app_win;
  float* q_rot;
  uint32_t* qfrag;  // kQfragBytes per (sequence, KV head); null when not needed
  float* part_o;
  float* part_ml;
};

// Tensor-core split kernels for the shapes they cover (decode_int2_mma.cu,
// decode_bf16_mma.cu).
bool int2_mma_supported(const Params& p);
int int2_mma_ctas_per_sm(int gqa, int G);  // resident CTAs per SM of the INT2 kernel
int bf16_mma_ctas_per_sm(int gqa);         // resident CTAs per SM of the BF16 kernel
cudaError_t int2_mma_split(const Params& p, cudaStream_t stream);
// Extend in tiles of query rows on tcgen05 (decode_int2_umma.cu): the INT2 splits only.
bool int2_umma_tile_supported(const Params& p);
cudaError_t int2_umma_tile_split(const Params& p, cudaStream_t stream);
// The merge of those tiles' rows: one CTA per (sequence x tile, KV head), R_v staged once;
// for up to 64 splits per row.
bool extend_tile_merge_supported(const Params& p);
// The BF16 sink/window splits of those tiles on tcgen05: one CTA per (sequence x tile,
// KV head, dense split of kDenseMmaPages pages).
cudaError_t bf16_dense_tile(const Params& p, cudaStream_t stream);
cudaError_t extend_tile_merge(const Params& p, cudaStream_t stream);
bool bf16_mma_supported(const Params& p);
cudaError_t bf16_mma_split(const Params& p, cudaStream_t stream);
// Fused single-wave decode (decode_fused.cu).
bool int2_fused_shape(int D, int G, int gqa);
int int2_fused_max_pps(int gqa);
int int2_fused_ctas_per_sm(int gqa, int G);
cudaError_t int2_fused_decode(const Params& p, cudaStream_t stream);

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


namespace {  // internal linkage in every unit that includes this header

// Number of sink/window splits: the tensor-core kernel takes kDenseMmaPages
// 16-row pages per split (sink and window buffers paged separately), the
// CUDA-core body kBf16Chunk positions.
int dense_splits(int S, int W, int max_seq_len, bool mma) {
  if (mma) {
    const int pages = (S + kPageSize - 1) / kPageSize + (W + kPageSize - 1) / kPageSize;
    return (pages + kDenseMmaPages - 1) / kDenseMmaPages;
  }
  const int dense = S + W < max_seq_len ? S + W : max_seq_len;
  return (dense + kBf16Chunk - 1) / kBf16Chunk;
}

// Split plan.  With pages_per_split == 0 the split size is chosen so that the
// paged splits of the whole batch fill about one wave of resident CTAs
// (ctas_per_sm x SMs, the sink/window splits counted; 5/3 x SMs for the BF16
// reference), 4..128 pages per split; at the 128-page cap, whole waves.
// The tensor-core split kernels cover head_dim 128 (INT2: group 64 or 128) and
// splits of at most kMmaMaxPps pages.
// Fused single-wave plan of a decode (no extend rows): unit (sequence, KV head) u
// gets n_s INT2 split CTAs over its bulk pages [S/16, ceil(max(S, max_seq_len - W)/16))
// and one BF16 CTA when S + W > 0; used when every unit's CTAs fit one wave of the
// fused kernel (about one CTA per SM), a split's page ids fit its table and, with
// the split size chosen here, a unit gets at least kMinFusedSplits split CTAs of at
// most kFusedMaxPps (GQA 8: kFusedMaxPpsGqa8) pages.
bool make_fused_plan(const oscar_dims_t* d, int B, int max_seq_len, int pps_req, int S, int W, Plan* p) {
  const int gqa = d->num_q_heads / d->num_kv_heads;
  if (B <= 0 || !int2_fused_shape(d->head_dim, d->group_size, gqa)) return false;
  const long long units = static_cast<long long>(B) * d->num_kv_heads;
  const long long slots = static_cast<long long>(int2_fused_ctas_per_sm(gqa, d->group_size)) * num_sms();
  const int n_d = S + W > 0 ? 1 : 0;
  const int bulk_lo = S / kPageSize;
  const int bulk_hi = ((S > max_seq_len - W ? S : max_seq_len - W) + kPageSize - 1) / kPageSize;
  const int nb = bulk_hi > bulk_lo ? bulk_hi - bulk_lo : 0;
  int pps = pps_req;
  if (pps == 0) {
    long long n_s = slots / units - n_d;
    // With fewer than kMinFusedSplits split CTAs per unit the general split grid
    // (several CTAs per SM) is faster.  Measured at 32K tokens, GQA 4, fused against
    // general: batch 2 (8 splits) 22.1 / 24.0 us, batch 3 (5) 32.9 / 31.0 us, batch 4
    // (3) 48.0 / 38.0 us, batch 8 (1) 142.9 / 68.1 us; batch 1 at 131K (18 splits,
    // 455 pages each) 54.5 / 63.6 us at GQA 8 and 35.2 / 36.8 us at GQA 4.
    if (n_s < kMinFusedSplits) return false;
    pps = static_cast<int>((nb + n_s - 1) / n_s);
    if (pps < 1) pps = 1;
    // ... and with more than about 60 pages per warp of a split CTA (16 warps at GQA
    // <= 4, 8 at GQA 8): fused against general, batch 2 at 131K 71.3 / 63.4 us (GQA 4,
    // 1023 pages per split) and 117.7 / 98.0 us (GQA 8, 1022), batch 1 at 262K, GQA 8
    // (910) 105.4 / 96.8 us; the fused form led with batch 1 at 262K, GQA 4 (910
    // pages: 63.8 / 64.9 us) and batch 2 at 64K, GQA 8 (510 pages: 58.1 / 63.4 us)
    if (pps > (gqa > 4 ? kFusedMaxPpsGqa8 : kFusedMaxPps)) return false;
  }
  const int n_s = nb > 0 ? (nb + pps - 1) / pps : 1;
  if (pps > int2_fused_max_pps(gqa) || units * (n_s + n_d) > slots) return false;
  p->fused = 1;
  p->mma = 1;
  p->bulk_lo = bulk_lo;
  p->pps = pps;
  p->n_paged = n_s;
  p->n_dense = n_d;
  p->ns = n_s + n_d;
  p->ml_ns = (p->ns + 1) & ~1;
  const size_t bh = static_cast<size_t>(B) * d->num_q_heads;
  p->off_qrot = 0;
  p->off_qfrag = 0;  // the q-rotation's QK operand blocks, kQfragBytes per (sequence, KV head)
  p->off_po = align_up(static_cast<size_t>(B) * d->num_kv_heads * kQfragBytes, 256);
  p->off_pml = p->off_po + align_up(bh * p->ns * d->head_dim * sizeof(float), 256);
  p->total = p->off_pml + align_up(bh * p->ml_ns * 2 * sizeof(float), 256);
  return true;
}

bool make_plan(const oscar_dims_t* d, int B, int max_seq_len, int pps_req, int S, int W, Mode mode, int ctas_per_sm,
               Plan* p, bool allow_fused = false) {
  if (B < 0 || max_seq_len < 0 || pps_req < 0 || S < 0 || W < 0) return false;
  if (max_seq_len > d->max_pages_per_seq * kPageSize) return false;
  *p = Plan{};
  if (allow_fused && mode == kMixed && make_fused_plan(d, B, max_seq_len, pps_req, S, W, p)) return true;
  const int max_pages = (max_seq_len + kPageSize - 1) / kPageSize;
  const bool shape_mma = d->head_dim == 128 && (mode == kBf16Paged || d->group_size == 64 || d->group_size == 128);
  p->n_dense = mode == kMixed ? dense_splits(S, W, max_seq_len, shape_mma) : 0;
  int pps = pps_req;
  if (pps == 0) {
    const long long units = static_cast<long long>(B) * d->num_kv_heads;
    long long slots = static_cast<long long>(ctas_per_sm > 0 ? ctas_per_sm : 2) * num_sms() - units * p->n_dense;
    // The BF16 reference at small batches: about 5/3 CTAs per SM rather than the 3
    // that fit (B=1, 32K tokens: 31 splits instead of 57, 28.6 against 30.0 us for
    // the call; fewer partials to merge, each CTA streaming longer)
    if (mode == kBf16Paged) slots = static_cast<long long>(num_sms()) * 5 / 3;
    const long long total = mode == kBf16Paged ? slots : slots + units * p->n_dense;  // CTA slots of a wave
    const long long dense = units * p->n_dense;
    if (slots < units) slots = units;
    const long long splits = (slots + units - 1) / units;
    long long want = (max_pages + splits - 1) / splits;
    if (want < 4) want = 4;
    const bool capped = want >= 128;
    if (capped) want = 128;
    // At the 128-page cap and more than one wave: fill k whole waves instead of
    // spilling a few CTAs into one more (32K tokens, batch 8: 68.3 -> 65.9 us; 8K
    // tokens, batch 16: 56.5 -> 47.9 us; 131K, batch 2, GQA 8: 98.1 -> 93.9 us).
    // Below the cap one wave that a few sink/window CTAs overflow measured best.
    const long long n_at = (max_pages + want - 1) / want;
    if (capped && units * n_at + dense > total) {
      const long long k = (units * n_at + dense + total - 1) / total;
      const long long sk = (k * total - dense) / units;
      if (sk > n_at) {
        want = (max_pages + sk - 1) / sk;
        if (want < 4) want = 4;
      }
    }
    pps = static_cast<int>(want);
  }
  p->mma = shape_mma && pps <= kMmaMaxPps ? 1 : 0;
  if (mode == kMixed && !p->mma) p->n_dense = dense_splits(S, W, max_seq_len, false);
  p->pps = pps;
  p->n_paged = max_pages == 0 ? 0 : (max_pages + pps - 1) / pps;
  p->ns = p->n_paged + p->n_dense;
  if (p->ns == 0) p->ns = 1;
  if (p->ns > 65535 || B > 65535) return false;  // split index and sequence are grid y/z dimensions
  const size_t bh = static_cast<size_t>(B) * d->num_q_heads;
  size_t off = 0;
  p->off_qrot = off;
  if (mode == kMixed) off += align_up(bh * d->head_dim * sizeof(float), 256);
  p->off_qfrag = off;
  if (mode == kMixed) off += align_up(static_cast<size_t>(B) * d->num_kv_heads * kQfragBytes, 256);
  p->off_po = off;
  off += align_up(bh * p->ns * d->head_dim * sizeof(float), 256);
  p->off_pml = off;
  p->ml_ns = (p->ns + 1) & ~1;
  off += align_up(bh * p->ml_ns * 2 * sizeof(float), 256);
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

// The cache a query row reads: sequence `seq` of length L (which fixes the
// sink / window / bulk split), positions [0, A) attended.  A decode row b is
// sequence b with A = L; an extend row attends 0 .. row_pos[b] of sequence
// row_seq[b].  A row naming a sequence or position out of range is flagged and
// attends nothing.
struct RowView {
  int seq, L, A;
};
__device__ __forceinline__ RowView row_view(const Params& p, int b) {
  if (p.row_seq == nullptr) {
    const int L = clamp_len(p, b);
    return {b, L, L};
  }
  const int seq = __ldg(p.row_seq + b);
  if (seq < 0 || seq >= p.num_seqs) {
    record_error(OSCAR_DEVERR_POSITION);
    return {0, 0, 0};
  }
  const int L = clamp_len(p, seq);
  const int pos = __ldg(p.row_pos + b);
  if (pos < 0 || pos >= L) {
    record_error(OSCAR_DEVERR_POSITION);
    return {seq, L, 0};
  }
  return {seq, L, pos + 1};
}

// q_rot[b][hq] = q[b][hq] . R_k[h] for the GQA query heads hq of one (b, h):
// R_k[h] arrives in shared memory by one bulk copy and thread j computes column
// j for every query head.  Dynamic shared memory: qrot_smem(D) bytes.
constexpr int kQrotThreads = 128;  // 4 warps, each summing a quarter of the rows of R

// Bit position, inside its fp16 half, at which the tensor-core INT2 kernel
// extracts channel e (0..15) of a packed 16-channel word (see decode_int2_mma.cu).
__host__ __device__ constexpr int code_kpos(int e) { return (e & 7) <= 4 ? 2 * (e & 7) : 2 * (e & 7) - 10; }

// Exponent E of a query's tensor-core QK operands: E = 15 - ceil(log2(||q_rot|| *
// |scale_log2| * (1 + 2^-10))), so that every operand q_rot[ch] * scale_log2 *
// 2^(E - kpos) is below 2^15 in magnitude (|q_rot[ch]| <= ||q_rot||).
__device__ __forceinline__ int qk_exponent(float norm, float scale_log2) {
  const float bound = norm * fabsf(scale_log2) * (1.f + 1.f / 1024.f);
  int e = 0;
  if (bound > 0.f) frexpf(bound, &e);
  return min(max(15 - e, -100), 100);
}

// One 32-bit B-operand word of the INT2 kernel's QK product: channels ch_lo and
// ch_lo + 8 of a query (rotated values v_lo, v_hi), scaled by scale_log2 *
// 2^(E - kpos(channel)), as the fp16 high part or (lo_part) the fp16 remainder.
__device__ __forceinline__ uint32_t qk_word(float v_lo, float v_hi, float scale_log2, int E, int ch_lo,
                                            bool lo_part) {
  const float x0 = v_lo * scale_log2 * pow2i(E - code_kpos(ch_lo & 15));
  const float x1 = v_hi * scale_log2 * pow2i(E - code_kpos((ch_lo + 8) & 15));
  __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
  if (lo_part) {
    h0 = __float2half_rn(x0 - __half2float(h0));
    h1 = __float2half_rn(x1 - __half2float(h1));
  }
  return static_cast<uint32_t>(__half_as_ushort(h0)) | (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
}

// q_rot[b][hq] = q[b][hq] . R_k[h] for the GQA query heads of qrot_spc
// consecutive sequences b of one KV head h, one CTA per block of 32 output
// columns (grid (ceil(B / spc) * Hkv, D/32)): the CTA reads its block of R_k
// once for all of them.  Warp w sums rows [w*D/4, (w+1)*D/4) of the block's
// columns, read straight from global memory (D/4 independent coalesced loads per
// lane); the warps' sums are added in order through shared memory.
// For the tensor-core INT2 kernel (D = 128, qfrag non-null) the CTA also writes
// the per-lane QK B-fragments of its two 16-channel words for each (b, h) and,
// per query of every n-tile,
//   * F = 2^(24 - E) (the exact power of two the codes' subnormal scale undoes),
//   * the block sum of q_rot * scale * log2(e) (the kernel adds the blocks of a
//     group).
// E = 15 - ceil(log2(||q|| * scale * log2(e) * (1 + 2^-10))): since R is
// orthogonal every |q_rot[ch]| <= ||q||, so every B value fits fp16.
constexpr int kQrotMaxQ = 32;  // query heads per q-rotation CTA (qrot_spc * gqa)

template <int D>
__global__ void __launch_bounds__(kQrotThreads) qrot_kernel(Params p) {
  constexpr int kRows = D / 4;
  __shared__ __align__(16) float qs[kQrotMaxQ * D];
  __shared__ float part[4][kQrotMaxQ][32];
  __shared__ float qrb[kQrotMaxQ][32];
  __shared__ int E_s[kQrotMaxQ];
  grid_dep_launch_dependents();
  const int spc = p.qrot_spc;
  const int h = blockIdx.x % p.H, b0 = (blockIdx.x / p.H) * spc, cb = blockIdx.y;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int gqa = p.gqa;
  const int nb = min(spc, p.B - b0);  // sequences of this CTA
  const int nq = nb * gqa;            // query j * gqa + qi: head h * gqa + qi of sequence b0 + j
  const float* R = p.R_k + static_cast<size_t>(h) * D * D + static_cast<size_t>(warp) * kRows * D + 32 * cb + lane;
  float r[kRows];
#pragma unroll
  for (int rr = 0; rr < kRows; ++rr) r[rr] = __ldg(R + static_cast<size_t>(rr) * D);
  {  // q of the CTA's queries: 16-byte loads, all issued before any is used
    constexpr int kQv = kQrotMaxQ * D / 8 / kQrotThreads;
    uint4 qv[kQv];
#pragma unroll
    for (int u = 0; u < kQv; ++u) {
      const int i = u * kQrotThreads + tid;  // 8-element chunk
      if (i < nq * D / 8) {
        const int j = (8 * i) / (gqa * D), rem = (8 * i) % (gqa * D);
        qv[u] = __ldg(reinterpret_cast<const uint4*>(
            p.q + (static_cast<size_t>(b0 + j) * p.Hq + static_cast<size_t>(h) * gqa) * D + rem));
      }
    }
#pragma unroll
    for (int u = 0; u < kQv; ++u) {
      const int i = u * kQrotThreads + tid;
      if (i < nq * D / 8) {
        const uint32_t wv[4] = {qv[u].x, qv[u].y, qv[u].z, qv[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          qs[8 * i + 2 * e] = __uint_as_float(wv[e] << 16);
          qs[8 * i + 2 * e + 1] = __uint_as_float(wv[e] & 0xffff0000u);
        }
      }
    }
  }
  __syncthreads();
  if (D == 128 && p.qfrag != nullptr) {
    // fp16 exponents of the QK operands from ||q|| (one warp per query): since R
    // is orthogonal every |q_rot[ch]| <= ||q||
    for (int qq = warp; qq < nq; qq += kQrotThreads / 32) {
      float ss = 0.f;
      for (int i = lane; i < D; i += 32) ss = fmaf(qs[qq * D + i], qs[qq * D + i], ss);
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      if (lane == 0) E_s[qq] = qk_exponent(sqrtf(ss), p.scale_log2);
    }
  }
  for (int q0 = 0; q0 < nq; q0 += 4) {  // four independent chains; q read 4 rows at a time
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r4 = 0; r4 < kRows; r4 += 4)
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (q0 + k < nq) {
          const float4 qv = *reinterpret_cast<const float4*>(&qs[(q0 + k) * D + warp * kRows + r4]);
          acc[k] = fmaf(qv.w, r[r4 + 3], fmaf(qv.z, r[r4 + 2], fmaf(qv.y, r[r4 + 1], fmaf(qv.x, r[r4], acc[k]))));
        }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (q0 + k < nq) part[warp][q0 + k][lane] = acc[k];
  }
  __syncthreads();
  for (int idx = tid; idx < nq * 32; idx += kQrotThreads) {
    const int qq = idx / 32, c = idx % 32;
    const float tot = ((part[0][qq][c] + part[1][qq][c]) + part[2][qq][c]) + part[3][qq][c];
    const int j = qq / gqa, qi = qq % gqa;
    if (p.q_rot != nullptr)  // the fp32 rotated queries are kept only for the CUDA-core split body
      p.q_rot[((static_cast<size_t>(b0 + j) * p.Hq + static_cast<size_t>(h) * gqa + qi)) * D + 32 * cb + c] = tot;
    qrb[qq][c] = tot;
  }
  if (p.qfrag == nullptr) {
    grid_dep_wait();  // completion stays ordered after the preceding kernel
    return;
  }
  if constexpr (D == 128) {
  __syncthreads();  // qrb (all columns of the block) complete
  // fragment words of this block's two 16-channel words w = 2*cb, 2*cb + 1, for
  // each sequence: lanes with t = w % 4 (8 values of g), k-steps 4*(w/4) .. +3,
  // c2 in {0,1}, nt in {0,1}
  for (int idx = tid; idx < nb * 256; idx += kQrotThreads) {
    const int j = idx >> 8, it = idx & 255;
    uint32_t* dst = p.qfrag + (static_cast<size_t>(b0 + j) * p.H + h) * (32 * kQfragWords);
    const int w = 2 * cb + (it >> 7);
    const int gg8 = (it >> 4) & 7, kk = (it >> 2) & 3, c2 = (it >> 1) & 1, nt = it & 1;
    const int t = w & 3, L = 4 * gg8 + t, ks = 4 * (w >> 2) + kk;
    const int qb = 4 * nt + (gg8 >> 1);
    const int jw = 2 * kk + c2;
    const int ch_lo = 16 * w + jw, ch_hi = ch_lo + 8;
    uint32_t word = 0;
    if (qb < gqa)
      word = qk_word(qrb[j * gqa + qb][ch_lo - 32 * cb], qrb[j * gqa + qb][ch_hi - 32 * cb], p.scale_log2,
                     E_s[j * gqa + qb], ch_lo, gg8 & 1);
    dst[L * kQfragWords + nt * 16 + ks * 2 + c2] = word;
  }
  // factors: block sums of query 4*nt + t for the 32 lanes (and F from block 0)
  for (int idx = tid; idx < nb * 64; idx += kQrotThreads) {
    const int j = idx >> 6, L = (idx & 63) / 2, nt = idx & 1;
    uint32_t* dst = p.qfrag + (static_cast<size_t>(b0 + j) * p.H + h) * (32 * kQfragWords);
    const int qi = 4 * nt + (L & 3);
    float sum = 0.f, F = 0.f;
    if (qi < gqa) {
      for (int c = 0; c < 32; ++c) sum += qrb[j * gqa + qi][c];
      sum *= p.scale_log2;
      F = pow2i(24 - E_s[j * gqa + qi]);
    }
    dst[L * kQfragWords + 32 + 5 * nt + 1 + cb] = __float_as_uint(sum);
    if (cb == 0) {
      dst[L * kQfragWords + 32 + 5 * nt] = __float_as_uint(F);
      dst[L * kQfragWords + 42] = 0u;
      dst[L * kQfragWords + 43] = 0u;
    }
  }
  }  // D == 128
  // This kernel may start while the preceding kernel (for example the append of
  // the current token) still runs: it reads only q and R_k.  It completes only
  // after that kernel, so the split kernel, which waits for this one, sees the
  // preceding kernel's writes.
  grid_dep_wait();
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
  const RowView rv = row_view(p, b);
  const int L = rv.L, A = rv.A, bs = rv.seq;

  // Position range of this split (positions below A only).
  int sink_att = 0;
  const bool paged = s < p.n_paged;
  int begin = 0, count = 0;         // paged: absolute positions [begin, begin+count)
  int sink_end = 0, win_begin = 0;  // dense: enumerated sink then window
  if (MODE == kMixed) {
    sink_end = min(p.S, L);
    win_begin = max(p.S, L - p.W);
    sink_att = min(sink_end, A);
  }
  if (paged) {
    const int lo = s * p.pps * kPageSize, hi = lo + p.pps * kPageSize;
    const int r0 = MODE == kMixed ? max(lo, p.S) : lo;
    const int r1 = MODE == kMixed ? min(hi, min(win_begin, A)) : min(hi, A);
    begin = r0;
    count = max(0, r1 - r0);
  } else {
    const int n_dense = sink_att + max(0, A - win_begin);
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
          page = p.page_table[static_cast<size_t>(bs) * p.max_pages + pos / kPageSize];
          if (page < 0 || page >= p.num_pages) {
            record_error(OSCAR_DEVERR_PAGE_ID);
            page = -1;
            pos = -1;
          }
        } else {
          const int idx = begin + e;
          pos = idx < sink_att ? idx : win_begin + (idx - sink_att);
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
          src = p.sink + (((static_cast<size_t>(bs) * 2 + kvsel) * p.H + h) * p.S + pos) * D;
        } else {
          src = p.win + (((static_cast<size_t>(bs) * 2 + kvsel) * p.H + h) * p.W + pos % p.W) * D;
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
    p.part_ml[(bh * p.ml_ns + s) * 2 + 0] = m_s[tid];
    p.part_ml[(bh * p.ml_ns + s) * 2 + 1] = l_s[tid];
  }
}

template <int D, Mode MODE>
__global__ void __launch_bounds__(kThreads) split_kernel(Params p) {
  extern __shared__ __align__(16) float dyn_smem[];
  split_body<D, MODE>(p, blockIdx.x + p.split_base, blockIdx.y, blockIdx.z, dyn_smem);
}

// Log-sum-exp merge of the split partials and, in INT2 mode, the single
// un-rotation by R_v^T (OSCAR project card "How it works": rotate the query once,
// un-rotate the output once):
//   out[c] = (sum_plain w_s o_s[c] + sum_j (sum_rot w_s o_s[j]) R_v[h][c][j]) / sum_s w_s l_s,
//   w_s = 2^(m_s - max_s m_s),
// where the rotated partials are the INT2 splits (s < n_paged) and the plain ones
// the BF16 sink/window splits; splits that attended nothing (m = -inf) have
// weight 0 and their outputs are not read.  One CTA covers merge_qpc query heads
// of one (sequence, KV head): grid B * Hkv * (gqa / merge_qpc); or, for large
// batches, the gqa query heads of one KV head in merge_spc consecutive sequences
// (grid ceil(B / spc) * Hkv), so that R_v is read once for all of them.
//   phase A  one warp per query: maximum, denominator, weights;
//   phase B  thread (query, 4-channel quad, split group) sums a strided subset of
//            the splits, then the split groups are added in order;
//   phase C  thread (channel c, column part) dots the rotated sum with its part of
//            row c of R_v, then the parts are added in order.
// A small grid, launched while the splits still run, stages R_v in shared memory
// before it waits for them (kStageRv) and the partials with one bulk copy after
// (kStagePartials); a large grid reads both from L2.
constexpr int kMergeThreadsLarge = 256;  // threads per merge CTA, large grids
constexpr int kMergeThreadsBatch = 512;  // threads per merge CTA, several sequences per CTA
constexpr int kMergeQBatch = 16;         // query heads per CTA of that form
constexpr int kMergeThreadsSmall = 256;  // threads per merge CTA, grids of at most one CTA per SM (one query head each)
constexpr int kStageRv = 1, kStagePartials = 2;

// Dynamic shared memory of the merge kernel: [R_v D x D] [partials qpc x ns x D,
// (m, l) qpc x ml_ns x 2] weights [qpc][ns], denominators [16] and group maxima/sums [48], phase B/C scratch
// (max(8, qpc) x kMergeThreads floats), rotated and plain sums [qpc][D], two mbarriers.
constexpr size_t merge_smem(int D, int ns, int qpc, int stage, int threads) {
  return ((stage & kStageRv) ? static_cast<size_t>(D) * D * 4 : 0) +
         ((stage & kStagePartials) ? static_cast<size_t>(qpc) * ns * D * 4 + static_cast<size_t>(qpc) * ((ns + 1) & ~1) * 8
                                   : 0) +
         (static_cast<size_t>((qpc * ns + 3) & ~3) + 64) * 4 + static_cast<size_t>(qpc > 8 ? qpc : 8) * threads * 4 +
         2 * static_cast<size_t>(qpc) * D * 4 + 16;
}

// kQMax: most query heads per CTA the kernel is compiled for (1 for the
// small-grid form: less code, whose first run is not delayed by instruction fetch).
template <int D, Mode MODE, int kMergeThreads, int kQMax>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(Params p) {
  extern __shared__ __align__(128) float msm[];
  constexpr bool kRot = MODE == kMixed;
  constexpr int kQuads = D / 4;
  const int qpc = p.merge_qpc, spc = p.merge_spc;
  int h, b0;
  size_t row0 = 0;
  if (spc > 1) {  // query heads qi of sequences b0 + qi / gqa, KV head h
    h = blockIdx.x % p.H;
    b0 = (blockIdx.x / p.H) * spc;
  } else {
    const int qch = p.gqa / qpc;
    const int unit = blockIdx.x / qch, qc = blockIdx.x % qch;
    b0 = unit / p.H;
    h = unit % p.H;
    row0 = static_cast<size_t>(b0) * p.Hq + static_cast<size_t>(h) * p.gqa + static_cast<size_t>(qc) * qpc;
  }
  // (sequence, query head) row of query qi, and how many queries of the CTA exist
  auto row_of = [&](int qi) -> size_t {
    return spc > 1 ? static_cast<size_t>(b0 + qi / p.gqa) * p.Hq + static_cast<size_t>(h) * p.gqa + qi % p.gqa
                   : row0 + qi;
  };
  const int q_valid = spc > 1 ? min(qpc, (p.B - b0) * p.gqa) : qpc;
  const int ns = p.ns, np = kRot ? p.n_paged : 0;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool st_rv = kRot && (p.merge_stage & kStageRv) != 0;
  const bool st_po = (p.merge_stage & kStagePartials) != 0;
  float* Rs = msm;                                                          // [D][D] (st_rv)
  float* po_s = Rs + (st_rv ? D * D : 0);                                   // [qpc][ns][D] (st_po)
  float* ml_s = po_s + (st_po ? static_cast<size_t>(qpc) * ns * D : 0);     // [qpc][ml_ns][2] (st_po)
  float* wts = ml_s + (st_po ? static_cast<size_t>(qpc) * p.ml_ns * 2 : 0);  // [qpc][ns]
  float* den_s = wts + ((qpc * ns + 3) & ~3);                               // [16] (+ group maxima, sums)
  float4* red = reinterpret_cast<float4*>(den_s + 64);                      // [2][kMergeThreads]; phase C parts
  float* o_rot = reinterpret_cast<float*>(red) + (qpc > 8 ? qpc : 8) * kMergeThreads;  // [qpc][D]
  float* o_plain = o_rot + qpc * D;                                         // [qpc][D]
  uint64_t* bars = reinterpret_cast<uint64_t*>(o_plain + qpc * D);         // [2]
  if (tid == 0 && (st_rv || st_po)) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    mbar_init_fence();
    if (st_rv) {
      mbar_arrive_expect_tx(smem_u32(&bars[0]), D * D * 4);
      bulk_g2s(smem_u32(Rs), p.R_v + static_cast<size_t>(h) * D * D, D * D * 4, smem_u32(&bars[0]));
    }
  }
  __syncthreads();
  grid_dep_wait();  // the split partials come from the preceding kernel
  bool ok = true;
  if (st_po) {  // the partials and their (m, l) in one phase of bars[1]
    if (tid == 0) {
      const uint32_t bytes = static_cast<uint32_t>(qpc) * ns * D * 4;
      const uint32_t ml_bytes = static_cast<uint32_t>(qpc) * p.ml_ns * 8;
      mbar_arrive_expect_tx(smem_u32(&bars[1]), bytes + ml_bytes);
      bulk_g2s(smem_u32(po_s), p.part_o + row0 * ns * D, bytes, smem_u32(&bars[1]));
      bulk_g2s(smem_u32(ml_s), p.part_ml + row0 * p.ml_ns * 2, ml_bytes, smem_u32(&bars[1]));
    }
    ok = mbar_wait_bounded(smem_u32(&bars[1]), 0);
  }

  if constexpr (kQMax == 1) {
    // One query head per CTA: phases A and B in one pass.  Thread (quad cq, group
    // grp) runs an online log-sum-exp over its splits grp, grp + sg, ... (rotated
    // and plain sums kept apart); the groups are then combined in order.
    constexpr int items = kQuads;
    constexpr int sg = kMergeThreads / items;
    static_assert(sg <= 24, "group maxima and sums are staged for at most 24 groups");
    float* gm = den_s + 16;  // [sg] group maxima
    float* gl = den_s + 40;  // [sg] group denominators
    const int cq = tid % items, grp = tid / items;
    const float2* ml = reinterpret_cast<const float2*>(st_po ? ml_s : p.part_ml + row0 * p.ml_ns * 2);
    const float4* po = reinterpret_cast<const float4*>(st_po ? po_s : p.part_o + row0 * ns * D) + cq;
    float m = -INFINITY, l = 0.f;
    float4 ar = make_float4(0.f, 0.f, 0.f, 0.f), ap = ar;
    for (int sp = grp; sp < ns; sp += sg) {
      const float2 v = ml[sp];
      if (v.x == -INFINITY) continue;  // the split attended nothing: its output is not read
      if (v.x > m) {
        const float f = m == -INFINITY ? 0.f : fast_exp2(m - v.x);
        l *= f;
        ar.x *= f; ar.y *= f; ar.z *= f; ar.w *= f;
        ap.x *= f; ap.y *= f; ap.z *= f; ap.w *= f;
        m = v.x;
      }
      const float wgt = fast_exp2(v.x - m);
      const float4 o = po[static_cast<size_t>(sp) * kQuads];
      l = fmaf(wgt, v.y, l);
      float4& acc = sp < np ? ar : ap;
      acc.x = fmaf(wgt, o.x, acc.x); acc.y = fmaf(wgt, o.y, acc.y);
      acc.z = fmaf(wgt, o.z, acc.z); acc.w = fmaf(wgt, o.w, acc.w);
    }
    red[grp * items + cq] = ar;
    red[kMergeThreads + grp * items + cq] = ap;
    if (cq == 0) {
      gm[grp] = m;
      gl[grp] = l;
    }
    ok = __syncthreads_and(ok);
    if (tid < items) {
      float M = -INFINITY;
#pragma unroll
      for (int g = 0; g < sg; ++g) M = fmaxf(M, gm[g]);
      float4 sr = make_float4(0.f, 0.f, 0.f, 0.f), sp4 = sr;
      float den = 0.f;
#pragma unroll
      for (int g = 0; g < sg; ++g) {
        const float f = gm[g] == -INFINITY ? 0.f : fast_exp2(gm[g] - M);
        const float4 x = red[g * items + tid], y = red[kMergeThreads + g * items + tid];
        sr.x = fmaf(f, x.x, sr.x); sr.y = fmaf(f, x.y, sr.y); sr.z = fmaf(f, x.z, sr.z); sr.w = fmaf(f, x.w, sr.w);
        sp4.x = fmaf(f, y.x, sp4.x); sp4.y = fmaf(f, y.y, sp4.y); sp4.z = fmaf(f, y.z, sp4.z); sp4.w = fmaf(f, y.w, sp4.w);
        den = fmaf(f, gl[g], den);
      }
      reinterpret_cast<float4*>(o_rot)[tid] = sr;
      reinterpret_cast<float4*>(o_plain)[tid] = sp4;
      if (tid == 0) den_s[0] = den;
    }
  } else {
    // phase A: one pass over (m, l) with a running maximum per lane, combined
    // across the warp by log-sum-exp; then the weights from the staged maxima
    for (int qi = warp; qi < qpc; qi += kMergeThreads / 32) {
      float* wq = wts + qi * ns;
      if (qi >= q_valid) {  // past the last sequence: no partials, weight 0
        for (int s = lane; s < ns; s += 32) wq[s] = 0.f;
        if (lane == 0) den_s[qi] = 0.f;
        continue;
      }
      const float2* ml = reinterpret_cast<const float2*>(st_po ? ml_s + static_cast<size_t>(qi) * p.ml_ns * 2
                                                               : p.part_ml + row_of(qi) * p.ml_ns * 2);
      float M = -INFINITY, den = 0.f;
      for (int s0 = lane; s0 < ns; s0 += 4 * 32) {
        float2 v[4];
  #pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = s0 + 32 * k < ns ? ml[s0 + 32 * k] : make_float2(-INFINITY, 0.f);
  #pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (s0 + 32 * k < ns) wq[s0 + 32 * k] = v[k].x;
          if (v[k].x != -INFINITY) {
            if (v[k].x > M) {
              den = M == -INFINITY ? 0.f : den * fast_exp2(M - v[k].x);
              M = v[k].x;
            }
            den = fmaf(fast_exp2(v[k].x - M), v[k].y, den);
          }
        }
      }
      float Mw = M;
  #pragma unroll
      for (int off = 16; off > 0; off >>= 1) Mw = fmaxf(Mw, __shfl_xor_sync(0xffffffffu, Mw, off));
      den = M == -INFINITY ? 0.f : den * fast_exp2(M - Mw);
  #pragma unroll
      for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
      for (int s = lane; s < ns; s += 32) {
        const float m = wq[s];
        wq[s] = (m == -INFINITY || Mw == -INFINITY) ? 0.f : fast_exp2(m - Mw);
      }
      if (lane == 0) den_s[qi] = den;
    }
    ok = __syncthreads_and(ok);

    // phase B
    const int items = qpc * kQuads;
    const int sg = kMergeThreads / items;
    if (tid < items * sg) {
      const int item = tid % items, grp = tid / items;
      const int qi = item / kQuads, cq = item % kQuads;
      const float4* po = reinterpret_cast<const float4*>(st_po ? po_s + static_cast<size_t>(qi) * ns * D
                                                               : p.part_o + row_of(qi) * ns * D) + cq;
      const float* wq = wts + qi * ns;
      float4 ar = make_float4(0.f, 0.f, 0.f, 0.f), ap = ar;
      constexpr int kU = kQMax >= 16 ? 8 : 4;  // partials in flight per thread
      for (int s0 = grp; s0 < ns; s0 += kU * sg) {
        float w[kU];
        float4 v[kU];
  #pragma unroll
        for (int k = 0; k < kU; ++k) {
          const int s = s0 + k * sg;
          w[k] = s < ns ? wq[s] : 0.f;
          v[k] = w[k] != 0.f ? po[static_cast<size_t>(s) * kQuads] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
  #pragma unroll
        for (int k = 0; k < kU; ++k) {
          const float wr = s0 + k * sg < np ? w[k] : 0.f, wp = w[k] - wr;
          ar.x = fmaf(wr, v[k].x, ar.x); ar.y = fmaf(wr, v[k].y, ar.y);
          ar.z = fmaf(wr, v[k].z, ar.z); ar.w = fmaf(wr, v[k].w, ar.w);
          ap.x = fmaf(wp, v[k].x, ap.x); ap.y = fmaf(wp, v[k].y, ap.y);
          ap.z = fmaf(wp, v[k].z, ap.z); ap.w = fmaf(wp, v[k].w, ap.w);
        }
      }
      red[grp * items + item] = ar;
      red[kMergeThreads + grp * items + item] = ap;
    }
    __syncthreads();
    if (tid < items) {
      float4 ar = red[tid], ap = red[kMergeThreads + tid];
      for (int grp = 1; grp < sg; ++grp) {
        const float4 x = red[grp * items + tid], y = red[kMergeThreads + grp * items + tid];
        ar.x += x.x; ar.y += x.y; ar.z += x.z; ar.w += x.w;
        ap.x += y.x; ap.y += y.y; ap.z += y.z; ap.w += y.w;
      }
      reinterpret_cast<float4*>(o_rot)[tid] = ar;  // item = qi * kQuads + cq
      reinterpret_cast<float4*>(o_plain)[tid] = ap;
    }
  }
  if (st_rv) ok = mbar_wait_bounded(smem_u32(&bars[0]), 0) && ok;
  ok = __syncthreads_and(ok);

  // phase C: thread (c, jp) visits the 4-column chunks of its part starting at
  // chunk c mod (kJ/4), so 8 consecutive lanes read distinct shared-memory banks.
  float* part = reinterpret_cast<float*>(red);  // [kParts][qpc][D]
  constexpr int kParts = kMergeThreads / D;     // column parts per channel
  constexpr int kJ = D / kParts;                // columns per part
  constexpr int kChunks = kJ / 4;
  if (kRot) {
    const int c = tid % D, jp = tid / D;
    const float4* Rrow = reinterpret_cast<const float4*>((st_rv ? Rs + static_cast<size_t>(c) * D
                                                                 : p.R_v + (static_cast<size_t>(h) * D + c) * D) +
                                                         jp * kJ);
    const float4* orow = reinterpret_cast<const float4*>(o_rot + jp * kJ);
    float acc[kQMax], acc2[kQMax];  // two chains per query (even and odd chunks)
#pragma unroll
    for (int qi = 0; qi < kQMax; ++qi) acc[qi] = acc2[qi] = 0.f;
#pragma unroll
    for (int k0 = 0; k0 < kChunks; k0 += 8) {
      float4 r[8];
      int ch[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        ch[k] = (k0 + k + c) & (kChunks - 1);
        r[k] = k0 + k < kChunks ? (st_rv ? Rrow[ch[k]] : __ldg(Rrow + ch[k])) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int qi = 0; qi < kQMax; ++qi) {
        if (qi < qpc) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (k0 + k < kChunks) {
              const float4 o = orow[qi * kQuads + ch[k]];
              float& a = (k & 1) ? acc2[qi] : acc[qi];
              a = fmaf(o.x, r[k].x, fmaf(o.y, r[k].y, fmaf(o.z, r[k].z, fmaf(o.w, r[k].w, a))));
            }
          }
        }
      }
    }
#pragma unroll
    for (int qi = 0; qi < kQMax; ++qi)
      if (qi < qpc) part[(jp * qpc + qi) * D + c] = acc[qi] + acc2[qi];
    __syncthreads();
  }
  if (!ok && tid == 0) record_error(OSCAR_DEVERR_TIMEOUT);
  for (int idx = tid; idx < qpc * D; idx += kMergeThreads) {
    const int qi = idx / D, cc = idx % D;
    float u = o_plain[idx];
    if (kRot) {
#pragma unroll
      for (int jp = 0; jp < kParts; ++jp) u += part[(jp * qpc + qi) * D + cc];
    }
    const float den = den_s[qi];
    if (qi < q_valid) p.out[row_of(qi) * D + cc] = (ok && den > 0.f) ? u / den : 0.f;
  }
}

}  // namespace
}  // namespace oscar_dec
