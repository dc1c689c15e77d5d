// Split-KV paged decode attention: the mixed-precision OSCAR decode (BF16 sink
// + BF16 recent window + INT2 bulk; "OSCAR: Offline Spectral Covariance-Aware
// Rotation for 2-bit KV Cache Quantization", project card "How it works" and
// abstract) and the all-BF16 paged decode used as its speedup reference.
//
// Three kernels per call, on one stream:
//   qrot   q_rot = q . R_k[h] once per query head (so INT2 keys stay rotated);
//   split  one CTA per (split, KV head, sequence): a range of positions is
//          attended with an online softmax for all GQA query heads of the KV
//          head at once; the CTA writes (max, sum, unnormalised output);
//   merge  one CTA per (sequence, query head): log-sum-exp merge of the splits,
//          one un-rotation of the INT2 part by R_v^T, normalisation.
// Logits are kept in log2 units (scale * log2 e folded into the query side).
#include <atomic>
#include <mutex>

#include "decode_common.cuh"

namespace {

using namespace oscar;
using namespace oscar_dec;

template <int D, Mode MODE>
cudaError_t merge(const Params& p, cudaStream_t stream) {
  if (p.merge_spc > 1) {  // large batch: several sequences per CTA, R_v staged once per CTA
    const int grid = (p.B + p.merge_spc - 1) / p.merge_spc * p.H;
    const size_t smem = merge_smem(D, p.ns, p.merge_qpc, p.merge_stage, kMergeThreadsBatch);
    auto k = merge_kernel<D, MODE, kMergeThreadsBatch, kMergeQBatch>;
    cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(k), kMergeSmemLimit);
    if (e != cudaSuccess) return e;
    // launched as a programmatic dependent: its CTAs take the SMs the last split
    // CTAs leave and stage R_v before their dependency wait
    return launch_pdl(k, dim3(grid), dim3(kMergeThreadsBatch), smem, stream, p);
  }
  const int grid = p.B * p.H * (p.gqa / p.merge_qpc);
  // A grid of at most one CTA per SM (one query head per CTA) is launched early
  // (programmatic dependent launch) so that it is resident, with R_v staged, when
  // the splits finish, and runs a form compiled for one query head; a larger grid
  // would take SM slots from the last split CTAs and waits for them.
  if (grid <= num_sms() && p.merge_qpc == 1) {
    const size_t smem = merge_smem(D, p.ns, p.merge_qpc, p.merge_stage, kMergeThreadsSmall);
    auto k = merge_kernel<D, MODE, kMergeThreadsSmall, 1>;
    cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(k), kMergeSmemLimit);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, dim3(grid), dim3(kMergeThreadsSmall), smem, stream, p);
  }
  const size_t smem = merge_smem(D, p.ns, p.merge_qpc, p.merge_stage, kMergeThreadsLarge);
  auto k = merge_kernel<D, MODE, kMergeThreadsLarge, kMaxGqa>;
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(k), kMergeSmemLimit);
  if (e != cudaSuccess) return e;
  k<<<grid, kMergeThreadsLarge, smem, stream>>>(p);
  return cudaGetLastError();
}

// Query heads per merge CTA and what the merge stages in shared memory (see
// merge_kernel): with at least two (sequence, KV head) units per SM (INT2 mode),
// the GQA groups of several sequences per CTA with R_v staged once; with at least
// one, a KV head's GQA group per CTA; otherwise one query head per CTA (more
// CTAs), with R_v and, when they fit, the partials staged.
void merge_config(const oscar_dims_t* d, int B, int ns, Mode mode, int* qpc, int* stage, int* spc) {
  const int gqa = d->num_q_heads / d->num_kv_heads;
  const long long units = static_cast<long long>(B) * d->num_kv_heads;
  *spc = 1;
  if (mode == kMixed && units >= 2LL * num_sms() &&
      merge_smem(d->head_dim, ns, kMergeQBatch, kStageRv, kMergeThreadsBatch) <= kMergeSmemLimit) {
    *spc = kMergeQBatch / gqa;
    *qpc = *spc * gqa;
    *stage = kStageRv;
    return;
  }
  *qpc = units >= num_sms() && merge_smem(d->head_dim, ns, gqa, 0, kMergeThreadsLarge) <= kMergeSmemLimit ? gqa : 1;
  *stage = 0;
  if (units * (gqa / *qpc) <= num_sms()) {
    const int t = kMergeThreadsSmall;
    if (mode == kMixed && merge_smem(d->head_dim, ns, *qpc, kStageRv, t) <= kMergeSmemLimit) *stage |= kStageRv;
    if (merge_smem(d->head_dim, ns, *qpc, *stage | kStagePartials, t) <= kMergeSmemLimit) *stage |= kStagePartials;
  }
}

template <int D, Mode MODE>
cudaError_t launch(const Params& p, cudaStream_t stream) {
  if (MODE == kMixed) {
    const int chunks = (p.B + p.qrot_spc - 1) / p.qrot_spc;
    cudaError_t e = launch_pdl(qrot_kernel<D>, dim3(chunks * p.H, D / 32), dim3(kQrotThreads), 0, stream, p);
    if (e != cudaSuccess) return e;
  }
  const bool mma = MODE == kMixed ? int2_mma_supported(p) : bf16_mma_supported(p);
  cudaError_t e;
  if (mma) {
    e = MODE == kMixed ? int2_mma_split(p, stream) : bf16_mma_split(p, stream);
  } else {
    constexpr size_t smem = split_body_smem(D);
    e = set_smem_limit_once(reinterpret_cast<const void*>(split_kernel<D, MODE>), smem);
    if (e == cudaSuccess) {
      if (MODE == kMixed) {
        e = launch_pdl(split_kernel<D, MODE>, dim3(p.ns, p.H, p.B), dim3(kThreads), smem, stream, p);
      } else {
        split_kernel<D, MODE><<<dim3(p.ns, p.H, p.B), kThreads, smem, stream>>>(p);
        e = cudaGetLastError();
      }
    }
  }
  if (e != cudaSuccess) return e;
  return merge<D, MODE>(p, stream);
}

oscar_status_t run(Params p, Mode mode, void* stream) {
  cudaError_t e;
  if (p.D == 128) e = mode == kMixed ? launch<128, kMixed>(p, as_stream(stream)) : launch<128, kBf16Paged>(p, as_stream(stream));
  else e = mode == kMixed ? launch<64, kMixed>(p, as_stream(stream)) : launch<64, kBf16Paged>(p, as_stream(stream));
  return e == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

// Resident CTAs per SM of the split kernel a shape will use (for split sizing).
int split_ctas_per_sm(const oscar_dims_t* d, Mode mode) {
  const int gqa = d->num_q_heads / d->num_kv_heads;
  if (d->head_dim == 128) {
    if (mode == kBf16Paged) return bf16_mma_ctas_per_sm(gqa);
    if (d->group_size == 64 || d->group_size == 128) return int2_mma_ctas_per_sm(gqa, d->group_size);
  }
  return 4;
}

// Cycles after which an INT2 split warp's first page wait gives up, for the timeout
// test (0: no stall).
std::atomic<long long> g_stall_cycles{0};

Params base_params(const oscar_dims_t* d, int B, int max_seq_len, const Plan& plan, Mode mode, float sm_scale,
                   void* ws) {
  Params p{};
  p.B = B;
  p.Hq = d->num_q_heads;
  p.H = d->num_kv_heads;
  p.D = d->head_dim;
  p.G = d->group_size;
  p.gqa = d->num_q_heads / d->num_kv_heads;
  p.num_pages = d->num_pages;
  p.max_pages = d->max_pages_per_seq;
  p.max_seq_len = max_seq_len;
  p.pps = plan.pps;
  p.n_paged = plan.n_paged;
  p.n_dense = plan.n_dense;
  p.ns = plan.ns;
  p.ml_ns = plan.ml_ns;
  merge_config(d, B, plan.ns, mode, &p.merge_qpc, &p.merge_stage, &p.merge_spc);
  // q-rotation: about four CTAs per SM; a CTA takes up to kQrotMaxQ query heads
  // (several sequences of one KV head) so that R_k is read once for all of them.
  {
    const long long ctas = static_cast<long long>(B) * d->num_kv_heads * (d->head_dim / 32);
    long long spc = (ctas + 4LL * num_sms() - 1) / (4LL * num_sms());
    const int cap = kQrotMaxQ / p.gqa;
    if (spc > cap) spc = cap;
    if (spc < 1) spc = 1;
    p.qrot_spc = static_cast<int>(spc);
  }
  p.mma = plan.mma;
  p.fused = plan.fused;
  p.bulk_lo = plan.bulk_lo;
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf(static_cast<float>(d->head_dim));
  p.scale_log2 = scale * 1.4426950408889634f;
  char* w = static_cast<char*>(ws);
  p.q_rot = reinterpret_cast<float*>(w + plan.off_qrot);
  p.qfrag = reinterpret_cast<uint32_t*>(w + plan.off_qfrag);
  p.part_o = reinterpret_cast<float*>(w + plan.off_po);
  p.part_ml = reinterpret_cast<float*>(w + plan.off_pml);
  p.stall_cycles = g_stall_cycles.load(std::memory_order_relaxed);
  return p;
}

}  // namespace

extern "C" size_t oscar_decode_workspace_bytes(const oscar_dims_t* dims, int32_t batch, int32_t max_seq_len,
                                               int32_t pages_per_split, int32_t sink_len, int32_t window_len) {
  if (check_dims(dims) != OSCAR_OK) return 0;
  Plan plan;
  if (!make_plan(dims, batch, max_seq_len, pages_per_split, sink_len, window_len, kMixed,
                 split_ctas_per_sm(dims, kMixed), &plan, /*allow_fused=*/true))
    return 0;
  return plan.total;
}

extern "C" oscar_status_t oscar_decode_plan(const oscar_dims_t* dims, int32_t batch, int32_t max_seq_len,
                                            int32_t pages_per_split, int32_t sink_len, int32_t window_len,
                                            int32_t* fused, int32_t* splits, int32_t* pages_per_split_used) {
  const oscar_status_t st = check_dims(dims);
  if (st != OSCAR_OK) return st;
  Plan plan;
  if (!make_plan(dims, batch, max_seq_len, pages_per_split, sink_len, window_len, kMixed,
                 split_ctas_per_sm(dims, kMixed), &plan, /*allow_fused=*/true))
    return OSCAR_ERR_INVALID_ARG;
  if (fused) *fused = plan.fused;
  if (splits) *splits = plan.n_paged;
  if (pages_per_split_used) *pages_per_split_used = plan.pps;
  return OSCAR_OK;
}

namespace {
// Workspace of the row-wise attention of the extend entry points (never the fused plan).
size_t extend_plan_bytes(const oscar_dims_t* dims, int32_t rows, int32_t max_seq_len, int32_t pages_per_split,
                         int32_t sink_len, int32_t window_len) {
  if (check_dims(dims) != OSCAR_OK) return 0;
  Plan plan;
  if (!make_plan(dims, rows, max_seq_len, pages_per_split, sink_len, window_len, kMixed,
                 split_ctas_per_sm(dims, kMixed), &plan))
    return 0;
  return plan.total;
}
}  // namespace

namespace {

// oscar_append_decode's append: the current token of every sequence.
struct CurrentAppend {
  const void* k;
  const void* v;
  const float* clip_k;
  const float* clip_v;
  const float* offset_k;
  const int64_t* slot_mapping;
  uint8_t* int2_pages;
  void* scale_zero_pages;
  void* bf16_sink;
  void* bf16_window;
};

// The mixed-precision attention of `rows` query rows: a decode (row_seq null,
// row b is sequence b and attends its whole cache) or an extend (row b attends
// positions 0 .. row_pos[b] of sequence row_seq[b] < num_seqs).
oscar_status_t mixed_attention(const oscar_dims_t* dims, int32_t rows, int32_t num_seqs, const int32_t* row_seq,
                               const int32_t* row_pos, int32_t max_seq_len, int32_t pages_per_split, const void* q,
                               const float* R_k, const float* R_v, const uint8_t* int2_pages,
                               const void* scale_zero_pages, const void* bf16_sink, const void* bf16_window,
                               const int32_t* page_table, const int32_t* seq_lens, int32_t sink_len,
                               int32_t window_len, float sm_scale, float* out, void* workspace,
                               size_t workspace_bytes, void* stream, const CurrentAppend* app = nullptr) {
  oscar_status_t st = check_dims(dims);
  if (st != OSCAR_OK) return st;
  if (rows < 0 || num_seqs < 0 || max_seq_len < 0 || pages_per_split < 0 || sink_len < 0 || window_len < 0)
    return OSCAR_ERR_INVALID_ARG;
  if (rows == 0) return OSCAR_OK;
  if (!q || !R_k || !R_v || !int2_pages || !scale_zero_pages || !page_table || !seq_lens || !out || !workspace)
    return OSCAR_ERR_INVALID_ARG;
  if ((sink_len > 0 && !bf16_sink) || (window_len > 0 && !bf16_window)) return OSCAR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return OSCAR_ERR_INVALID_ARG;
  if (misaligned16(q) || misaligned16(R_k) || misaligned16(R_v) || misaligned16(int2_pages) ||
      misaligned16(scale_zero_pages) || misaligned16(bf16_sink) || misaligned16(bf16_window))
    return OSCAR_ERR_INVALID_ARG;
  Plan plan;
  if (!make_plan(dims, rows, max_seq_len, pages_per_split, sink_len, window_len, kMixed,
                 split_ctas_per_sm(dims, kMixed), &plan, /*allow_fused=*/row_seq == nullptr))
    return OSCAR_ERR_INVALID_ARG;
  if (workspace_bytes < plan.total) return OSCAR_ERR_WORKSPACE;
  if (merge_smem(dims->head_dim, plan.ns, 1, 0, kMergeThreadsSmall) > kMergeSmemLimit) return OSCAR_ERR_UNSUPPORTED;
  if (static_cast<long long>(rows) * dims->num_q_heads > 0x7fffffffLL || plan.ns > 0x7fffffff) return OSCAR_ERR_UNSUPPORTED;
  Params p = base_params(dims, rows, max_seq_len, plan, kMixed, sm_scale, workspace);
  p.S = sink_len;
  p.W = window_len;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.R_k = R_k;
  p.R_v = R_v;
  p.codes = int2_pages;
  p.sz = static_cast<const __half*>(scale_zero_pages);
  p.sink = static_cast<const __nv_bfloat16*>(bf16_sink);
  p.win = static_cast<const __nv_bfloat16*>(bf16_window);
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.row_seq = row_seq;
  p.row_pos = row_pos;
  p.num_seqs = num_seqs;
  p.out = out;
  // The current token goes into the sink or the window when W >= 1, and no INT2 split
  // reads its position: the CTA that attends its sink/window rows appends it (the
  // fused single-wave kernel's BF16 CTA, or the tensor-core split kernel's dense CTA).
  // Otherwise (no window, or the CUDA-core split body) the append runs first.
  if (app != nullptr && !(window_len >= 1 && (p.fused || int2_mma_supported(p)))) {
    // sequential form: the append, then the decode (one stream)
    const oscar_status_t sa = oscar_internal_append_current(
        dims, rows, app->k, app->v, R_k, R_v, app->clip_k, app->clip_v, app->offset_k, app->slot_mapping, seq_lens,
        sink_len, window_len, app->int2_pages, app->scale_zero_pages, app->bf16_sink, app->bf16_window, stream);
    if (sa != OSCAR_OK) return sa;
    app = nullptr;
  }
  if (app != nullptr) {  // fused form
    p.app_k = static_cast<const __nv_bfloat16*>(app->k);
    p.app_v = static_cast<const __nv_bfloat16*>(app->v);
    p.app_clip_k = app->clip_k;
    p.app_clip_v = app->clip_v;
    p.app_offset_k = app->offset_k;
    p.app_slots = app->slot_mapping;
    p.app_codes = app->int2_pages;
    p.app_sz = static_cast<__half*>(app->scale_zero_pages);
    p.app_sink = static_cast<__nv_bfloat16*>(app->bf16_sink);
    p.app_win = static_cast<__nv_bfloat16*>(app->bf16_window);
  }
  if (p.fused) {
    p.q_rot = nullptr;
    p.n_dense_pages = (sink_len + kPageSize - 1) / kPageSize + (window_len + kPageSize - 1) / kPageSize;
    return int2_fused_decode(p, as_stream(stream)) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
  }
  if (!int2_mma_supported(p)) p.qfrag = nullptr;
  return run(p, kMixed, stream);
}

}  // namespace

extern "C" oscar_status_t oscar_decode(const oscar_dims_t* dims, int32_t batch, int32_t max_seq_len,
                                       int32_t pages_per_split, const void* q, const float* R_k, const float* R_v,
                                       const uint8_t* int2_pages, const void* scale_zero_pages,
                                       const void* bf16_sink, const void* bf16_window, const int32_t* page_table,
                                       const int32_t* seq_lens, int32_t sink_len, int32_t window_len,
                                       float sm_scale, float* out, void* workspace, size_t workspace_bytes,
                                       void* stream) {
  return mixed_attention(dims, batch, batch, nullptr, nullptr, max_seq_len, pages_per_split, q, R_k, R_v,
                         int2_pages, scale_zero_pages, bf16_sink, bf16_window, page_table, seq_lens, sink_len,
                         window_len, sm_scale, out, workspace, workspace_bytes, stream);
}

extern "C" oscar_status_t oscar_append_decode(const oscar_dims_t* dims, int32_t batch, int32_t max_seq_len,
                                              int32_t pages_per_split, const void* q, const void* k, const void* v,
                                              const float* R_k, const float* R_v, const float* clip_k,
                                              const float* clip_v, const float* offset_k,
                                              const int64_t* slot_mapping, uint8_t* int2_pages,
                                              void* scale_zero_pages, void* bf16_sink, void* bf16_window,
                                              const int32_t* page_table, const int32_t* seq_lens, int32_t sink_len,
                                              int32_t window_len, float sm_scale, float* out, void* workspace,
                                              size_t workspace_bytes, void* stream) {
  if (batch < 0) return OSCAR_ERR_INVALID_ARG;
  if (batch == 0) return check_dims(dims);
  if (!k || !v || !clip_k || !clip_v || !slot_mapping) return OSCAR_ERR_INVALID_ARG;
  if (misaligned16(k) || misaligned16(v) || misaligned16(clip_k) || misaligned16(clip_v) ||
      misaligned16(offset_k))
    return OSCAR_ERR_INVALID_ARG;
  const CurrentAppend app{k, v, clip_k, clip_v, offset_k, slot_mapping, int2_pages, scale_zero_pages, bf16_sink,
                          bf16_window};
  return mixed_attention(dims, batch, batch, nullptr, nullptr, max_seq_len, pages_per_split, q, R_k, R_v,
                         int2_pages, scale_zero_pages, bf16_sink, bf16_window, page_table, seq_lens, sink_len,
                         window_len, sm_scale, out, workspace, workspace_bytes, stream, &app);
}

namespace oscar_extend_rows {

using namespace oscar;
using namespace oscar_dec;

// Rows of sequence b: q_start[b] .. q_start[b + 1) - 1, the last n_b = q_start[b + 1]
// - q_start[b] positions of the sequence (the tokens just appended), in order.
__global__ void extend_rows_kernel(const int32_t* q_start, const int32_t* seq_lens, int rows, int max_seq_len,
                                   int32_t* row_seq, int32_t* row_pos) {
  grid_dep_launch_dependents();
  const int b = blockIdx.x;
  const int q0 = q_start[b], q1 = q_start[b + 1];
  int L = seq_lens[b];
  if (L < 0 || L > max_seq_len) L = L < 0 ? 0 : max_seq_len;  // the attention kernels flag it
  for (int j = threadIdx.x; q0 + j < q1; j += blockDim.x) {
    const int r = q0 + j;
    if (r < 0 || r >= rows) {
      record_error(OSCAR_DEVERR_POSITION);
      continue;
    }
    row_seq[r] = b;
    row_pos[r] = L - (q1 - q0) + j;  // negative when the rows outnumber the tokens: flagged later
  }
}

// Extend in tiles: the rows' (sequence, position), the BF16 sink/window splits and the
// INT2 splits in tiles of rows (the q-rotation between them), the merge per tile.
template <int D>
cudaError_t launch_extend_tiles(Params p, int batch, cudaStream_t stream) {
  extend_rows_kernel<<<batch, 128, 0, stream>>>(p.q_start, p.seq_lens, p.B, p.max_seq_len,
                                                const_cast<int32_t*>(p.row_seq), const_cast<int32_t*>(p.row_pos));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.n_dense > 0) {  // the sink/window rows once per tile of rows, on tcgen05
    e = bf16_dense_tile(p, stream);
    if (e != cudaSuccess) return e;
  }
  const int chunks = (p.B + p.qrot_spc - 1) / p.qrot_spc;
  // the tcgen05 tile kernel reads the fp32 rotated queries only: no mma.sync operand blocks
  Params pq = p;
  pq.qfrag = nullptr;
  e = launch_pdl(qrot_kernel<D>, dim3(chunks * p.H, D / 32), dim3(kQrotThreads), 0, stream, pq);
  if (e != cudaSuccess) return e;
  if (p.n_paged > 0) {
    e = int2_umma_tile_split(p, stream);
    if (e != cudaSuccess) return e;
  }
  return extend_tile_merge_supported(p) ? extend_tile_merge(p, stream) : ::merge<D, kMixed>(p, stream);
}

}  // namespace oscar_extend_rows

extern "C" size_t oscar_extend_varlen_workspace_bytes(const oscar_dims_t* dims, int32_t num_rows,
                                                      int32_t max_seq_len, int32_t pages_per_split,
                                                      int32_t sink_len, int32_t window_len) {
  const size_t base = extend_plan_bytes(dims, num_rows, max_seq_len, pages_per_split, sink_len, window_len);
  if (base == 0) return 0;
  return base + 2 * align_up(static_cast<size_t>(num_rows) * 4, 256);
}

extern "C" oscar_status_t oscar_extend_varlen(const oscar_dims_t* dims, int32_t batch, int32_t num_rows,
                                              int32_t max_seq_len, int32_t max_rows_per_seq, int32_t pages_per_split,
                                              const void* q, const int32_t* q_start, const float* R_k,
                                              const float* R_v, const uint8_t* int2_pages,
                                              const void* scale_zero_pages, const void* bf16_sink,
                                              const void* bf16_window, const int32_t* page_table,
                                              const int32_t* seq_lens, int32_t sink_len, int32_t window_len,
                                              float sm_scale, float* out, void* workspace, size_t workspace_bytes,
                                              void* stream) {
  oscar_status_t st = check_dims(dims);
  if (st != OSCAR_OK) return st;
  if (batch < 0 || num_rows < 0 || max_seq_len < 0 || max_rows_per_seq < 0 || pages_per_split < 0 || sink_len < 0 ||
      window_len < 0)
    return OSCAR_ERR_INVALID_ARG;
  if (num_rows == 0) return OSCAR_OK;
  if (batch == 0 || max_rows_per_seq == 0 || !q_start || !q || !R_k || !R_v || !int2_pages || !scale_zero_pages ||
      !page_table || !seq_lens || !out || !workspace)
    return OSCAR_ERR_INVALID_ARG;
  if ((sink_len > 0 && !bf16_sink) || (window_len > 0 && !bf16_window)) return OSCAR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return OSCAR_ERR_INVALID_ARG;
  if (misaligned16(q) || misaligned16(R_k) || misaligned16(R_v) || misaligned16(int2_pages) ||
      misaligned16(scale_zero_pages) || misaligned16(bf16_sink) || misaligned16(bf16_window))
    return OSCAR_ERR_INVALID_ARG;
  Plan plan;
  if (!make_plan(dims, num_rows, max_seq_len, pages_per_split, sink_len, window_len, kMixed,
                 split_ctas_per_sm(dims, kMixed), &plan))
    return OSCAR_ERR_INVALID_ARG;
  const size_t need = plan.total + 2 * align_up(static_cast<size_t>(num_rows) * 4, 256);
  if (workspace_bytes < need) return OSCAR_ERR_WORKSPACE;
  if (merge_smem(dims->head_dim, plan.ns, 1, 0, kMergeThreadsSmall) > kMergeSmemLimit) return OSCAR_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_rows) * dims->num_q_heads > 0x7fffffffLL) return OSCAR_ERR_UNSUPPORTED;
  Params p = base_params(dims, num_rows, max_seq_len, plan, kMixed, sm_scale, workspace);
  p.S = sink_len;
  p.W = window_len;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.R_k = R_k;
  p.R_v = R_v;
  p.codes = int2_pages;
  p.sz = static_cast<const __half*>(scale_zero_pages);
  p.sink = static_cast<const __nv_bfloat16*>(bf16_sink);
  p.win = static_cast<const __nv_bfloat16*>(bf16_window);
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.out = out;
  p.num_seqs = batch;
  p.q_start = q_start;
  char* w = static_cast<char*>(workspace);
  p.row_seq = reinterpret_cast<const int32_t*>(w + plan.total);
  p.row_pos = reinterpret_cast<const int32_t*>(w + plan.total + align_up(static_cast<size_t>(num_rows) * 4, 256));
  if (!int2_mma_supported(p)) p.qfrag = nullptr;
  // tiles: the sink/window splits run the tensor-core split kernel, the INT2 bulk the tcgen05 tile kernel
  const bool tiles = p.qfrag != nullptr && int2_umma_tile_supported(p);
  if (tiles) {
    const int rpt = 64 / p.gqa;
    const long long t = (static_cast<long long>(max_rows_per_seq) + rpt - 1) / rpt;
    if (t * batch > 65535) return OSCAR_ERR_UNSUPPORTED;
    p.tiles = static_cast<int>(t);
    const cudaError_t e = oscar_extend_rows::launch_extend_tiles<128>(p, batch, as_stream(stream));
    return e == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
  }
  // other shapes: one decode row per query row
  oscar_extend_rows::extend_rows_kernel<<<batch, 128, 0, as_stream(stream)>>>(q_start, seq_lens, num_rows, max_seq_len,
                                                           const_cast<int32_t*>(p.row_seq),
                                                           const_cast<int32_t*>(p.row_pos));
  if (cudaGetLastError() != cudaSuccess) return OSCAR_ERR_CUDA;
  return run(p, kMixed, stream);
}

extern "C" size_t oscar_extend_workspace_bytes(const oscar_dims_t* dims, int32_t num_rows, int32_t max_seq_len,
                                               int32_t pages_per_split, int32_t sink_len, int32_t window_len) {
  return extend_plan_bytes(dims, num_rows, max_seq_len, pages_per_split, sink_len, window_len);
}

extern "C" oscar_status_t oscar_extend(const oscar_dims_t* dims, int32_t batch, int32_t num_rows,
                                       int32_t max_seq_len, int32_t pages_per_split, const void* q,
                                       const int32_t* row_seq, const int32_t* row_pos, const float* R_k,
                                       const float* R_v, const uint8_t* int2_pages, const void* scale_zero_pages,
                                       const void* bf16_sink, const void* bf16_window, const int32_t* page_table,
                                       const int32_t* seq_lens, int32_t sink_len, int32_t window_len,
                                       float sm_scale, float* out, void* workspace, size_t workspace_bytes,
                                       void* stream) {
  if (batch < 0 || num_rows < 0) return OSCAR_ERR_INVALID_ARG;
  if (num_rows > 0 && (batch == 0 || !row_seq || !row_pos)) return OSCAR_ERR_INVALID_ARG;
  return mixed_attention(dims, num_rows, batch, row_seq, row_pos, max_seq_len, pages_per_split, q, R_k, R_v,
                         int2_pages, scale_zero_pages, bf16_sink, bf16_window, page_table, seq_lens, sink_len,
                         window_len, sm_scale, out, workspace, workspace_bytes, stream);
}

extern "C" size_t oscar_bf16_decode_workspace_bytes(const oscar_dims_t* dims, int32_t batch, int32_t max_seq_len,
                                                    int32_t pages_per_split) {
  if (check_dims(dims) != OSCAR_OK) return 0;
  Plan plan;
  if (!make_plan(dims, batch, max_seq_len, pages_per_split, 0, 0, kBf16Paged, split_ctas_per_sm(dims, kBf16Paged), &plan)) return 0;
  return plan.total;
}

extern "C" oscar_status_t oscar_bf16_decode(const oscar_dims_t* dims, int32_t batch, int32_t max_seq_len,
                                            int32_t pages_per_split, const void* q, const void* bf16_pages,
                                            const int32_t* page_table, const int32_t* seq_lens, float sm_scale,
                                            float* out, void* workspace, size_t workspace_bytes, void* stream) {
  oscar_status_t st = check_dims(dims);
  if (st != OSCAR_OK) return st;
  if (batch < 0 || max_seq_len < 0 || pages_per_split < 0) return OSCAR_ERR_INVALID_ARG;
  if (batch == 0) return OSCAR_OK;
  if (!q || !bf16_pages || !page_table || !seq_lens || !out || !workspace) return OSCAR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return OSCAR_ERR_INVALID_ARG;
  if (misaligned16(bf16_pages)) return OSCAR_ERR_INVALID_ARG;
  Plan plan;
  if (!make_plan(dims, batch, max_seq_len, pages_per_split, 0, 0, kBf16Paged, split_ctas_per_sm(dims, kBf16Paged), &plan)) return OSCAR_ERR_INVALID_ARG;
  if (workspace_bytes < plan.total) return OSCAR_ERR_WORKSPACE;
  if (merge_smem(dims->head_dim, plan.ns, 1, 0, kMergeThreadsSmall) > kMergeSmemLimit) return OSCAR_ERR_UNSUPPORTED;
  Params p = base_params(dims, batch, max_seq_len, plan, kBf16Paged, sm_scale, workspace);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.pages = static_cast<const __nv_bfloat16*>(bf16_pages);
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.out = out;
  p.qfrag = nullptr;
  return run(p, kBf16Paged, stream);
}

// ---- decode without a caller workspace ----------------------------------------
// Scratch of oscar_decode_noalloc: one file-scope device array, present on every
// device that loads this library until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[OSCAR_NOALLOC_SCRATCH_BYTES];

// Identity of the calling thread's current CUDA context: cuCtxGetId of
// cuCtxGetCurrent, reached through the runtime's driver entry points (no link
// against the driver library).  Unlike a context handle, the id is never reused
// within a process, so a context destroyed (cudaDeviceReset) and created again
// gets a new one.  False when the driver offers neither call or no context is
// current.
static bool current_context_id(unsigned long long* id) {
  using GetCurrentFn = int (*)(void**);
  using GetIdFn = int (*)(void*, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(f);
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  void* ctx = nullptr;
  if (get_current(&ctx) != 0 || ctx == nullptr) return false;
  return get_id(ctx, id) == 0;
}

// Device address of g_noalloc_scratch in the current context.  The host-side
// name is only a stand-in, so the address is looked up with cudaGetSymbolAddress
// (with the device current) and cached per device together with the id of the
// context it belongs to.  A call from another context of that device (the
// primary context reset and created again, which may load the library's module
// at a new address) looks it up again instead of using a stale address.
static oscar_status_t noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* cached[64] = {};
  static unsigned long long cached_ctx[64] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return OSCAR_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long ctx = 0;
  const bool have_ctx = current_context_id(&ctx);
  if (cached[dev] == nullptr || !have_ctx || ctx != cached_ctx[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return OSCAR_ERR_CUDA;
    // the lookup makes the device's primary context current if none was
    if (!current_context_id(&ctx)) ctx = 0;
    cached[dev] = ptr;
    cached_ctx[dev] = ctx;
  }
  *out = cached[dev];
  return OSCAR_OK;
}

extern "C" oscar_status_t oscar_decode_noalloc(const oscar_dims_t* dims, int32_t batch, int32_t max_seq_len,
                                               int32_t pages_per_split, const void* q, const float* R_k,
                                               const float* R_v, const uint8_t* int2_pages,
                                               const void* scale_zero_pages, const void* bf16_sink,
                                               const void* bf16_window, const int32_t* page_table,
                                               const int32_t* seq_lens, int32_t sink_len, int32_t window_len,
                                               float sm_scale, float* out, void* stream) {
  // Size check first, so an oversized request fails before any CUDA call.
  if (check_dims(dims) == OSCAR_OK && batch > 0 && max_seq_len >= 0 && pages_per_split >= 0 && sink_len >= 0 &&
      window_len >= 0) {
    Plan plan;
    if (make_plan(dims, batch, max_seq_len, pages_per_split, sink_len, window_len, kMixed,
                  split_ctas_per_sm(dims, kMixed), &plan, /*allow_fused=*/true) &&
        plan.total > OSCAR_NOALLOC_SCRATCH_BYTES)
      return OSCAR_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  if (batch > 0) {
    const oscar_status_t st = noalloc_scratch(&ws);
    if (st != OSCAR_OK) return st;
  }
  // The workspace of oscar_decode needs no initialisation: every byte it reads
  // was written earlier in the same call.
  return oscar_decode(dims, batch, max_seq_len, pages_per_split, q, R_k, R_v, int2_pages, scale_zero_pages,
                      bf16_sink, bf16_window, page_table, seq_lens, sink_len, window_len, sm_scale, out, ws,
                      OSCAR_NOALLOC_SCRATCH_BYTES, stream);
}

oscar_status_t oscar_internal_decode_errors(uint32_t* flags, int reset) {
  return read_unit_errors(flags, reset) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

extern "C" oscar_status_t oscar_test_stall_page_waits(int64_t cycles) {
  if (cycles < 0) return OSCAR_ERR_INVALID_ARG;
  g_stall_cycles.store(cycles, std::memory_order_relaxed);
  return OSCAR_OK;
}
