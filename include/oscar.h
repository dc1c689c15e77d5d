/*
 * oscar.h -- C ABI of the OSCAR INT2 rotated KV-cache library (GB300, sm_103a).
 *
 * The method ("OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV
 * Cache Quantization"; described by the summary "OSCAR: Cut LLM Inference Costs
 * 8x with 2-bit KV Cache Quantization", the project card "FutureMLS-Lab/OSCAR"
 * and the paper's abstract):
 *   - new K/V head vectors are multiplied by a fixed orthogonal rotation R and
 *     clipped to fixed per-channel thresholds, both found offline
 *     (summary "Practical Summary"; project card "How it works");
 *   - the bulk of the KV cache is stored in 2 bits, inside a paged KV cache
 *     (abstract: "custom INT2 attention kernel ... compatible with paged
 *     KV-cache serving");
 *   - a small sink of initial tokens and a recent window stay in BF16 and are
 *     attended together with the INT2 bulk (project card "How it works").
 * The pages print no formulas; the readings below are stated at each call.
 *
 * Conventions shared by every call
 *   - Pointers named as device buffers must point to device memory (or
 *     managed memory) of the current CUDA device.  The caller owns every
 *     buffer; the library keeps no pointer after a call returns and allocates
 *     no device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls are asynchronous and stream-ordered; they never
 *     synchronise the device.
 *   - Errors: arguments are checked on the host before anything is launched;
 *     a failed check returns OSCAR_ERR_INVALID_ARG / _UNSUPPORTED / _WORKSPACE
 *     and launches nothing.  A launch failure returns OSCAR_ERR_CUDA.  Kernels
 *     never trap: a bad page id, slot or sequence length met on the device is
 *     skipped and recorded in a device error word (oscar_device_errors).
 *   - Outputs never alias inputs.
 *   - q, k, v, R_k, R_v, the page pools and the BF16 sink/window buffers are moved with
 *     bulk async copies or 16-byte loads and stores and must be 16-byte aligned (any
 *     cudaMalloc or torch allocation is); a misaligned pointer is rejected with
 *     OSCAR_ERR_INVALID_ARG.
 *   - Supported shapes: head_dim 64 or 128; page_size 16; group_size 32, 64
 *     or 128 dividing head_dim; num_q_heads / num_kv_heads (GQA) 1..8.
 */
#ifndef OSCAR_H_
#define OSCAR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  OSCAR_OK = 0,
  OSCAR_ERR_INVALID_ARG = 1, /* null pointer, negative or inconsistent size      */
  OSCAR_ERR_UNSUPPORTED = 2, /* valid but not implemented (head_dim 96, ...)     */
  OSCAR_ERR_WORKSPACE = 3,   /* workspace smaller than the *_workspace_bytes call */
  OSCAR_ERR_CUDA = 4         /* a CUDA call or launch failed                     */
} oscar_status_t;

/* Device error bits recorded by kernels (read with oscar_device_errors). */
#define OSCAR_DEVERR_SLOT 0x1u      /* append: slot >= num_pages * page_size (token skipped)  */
#define OSCAR_DEVERR_PAGE_ID 0x2u   /* decode: page id outside [0, num_pages) (page skipped)  */
#define OSCAR_DEVERR_SEQ_LEN 0x4u   /* decode: seq_len < 0 or > max_seq_len (clamped)         */
#define OSCAR_DEVERR_TIMEOUT 0x8u   /* a bounded wait on an async copy ran out (work skipped) */
#define OSCAR_DEVERR_POSITION 0x10u /* append_mixed: sequence id or position out of range (BF16 row skipped) */

/* Cache geometry. */
typedef struct {
  int32_t num_q_heads;       /* Hq, a multiple of num_kv_heads                          */
  int32_t num_kv_heads;      /* Hkv                                                     */
  int32_t head_dim;          /* D                                                       */
  int32_t page_size;         /* P: tokens per page                                      */
  int32_t group_size;        /* G: channels sharing one fp16 (scale, zero) pair         */
  int32_t num_pages;         /* pages in the pool                                       */
  int32_t max_pages_per_seq; /* row stride of page_table                                */
} oscar_dims_t;

/*
 * oscar_append -- rotate, clip, quantise to INT2 and store new K/V vectors.
 *
 * Defined by: summary "Practical Summary" (fixed rotations and clipping
 * thresholds, 2-bit KV cache) and abstract (paged KV cache).  For every token
 * t with slot_mapping[t] >= 0, every KV head h, and separately for K (R_k,
 * clip_k) and V (R_v, clip_v):
 *   y = x . R[h]                      row vector times fp32 [D][D] row-major R
 *   y_j = min(max(y_j, -clip[h][j]), +clip[h][j])      (+inf = no clipping)
 *   per group g of G consecutive channels: mn, mx = min, max of the group;
 *     scale = fp16(fp32((mx - mn) / 3)), zero = fp16(fp32(mn));
 *     code_j = clamp(rint((y_j - zero) / scale), 0, 3), ties to even, computed
 *     from the stored fp16 scale and zero (code 0 when scale == 0);
 *   the codes and pairs are written to page slot / P at offset slot % P.
 * Arguments
 *   k, v          device bf16 [num_tokens][Hkv][D]
 *   R_k, R_v      device fp32 [Hkv][D][D]
 *   clip_k/_v     device fp32 [Hkv][D]
 *   offset_k      device fp32 [Hkv][D], finite, 16-byte aligned, or NULL (no
 *                 offset).  Key offset removal (the OptR abstract on the OSCAR
 *                 paper page: an attention-equivalent key reparameterisation
 *                 that removes per-channel key offsets without changing the
 *                 softmax distribution): every key is taken as
 *                 x = fp32(k - offset_k[h]) (round to nearest even) before the
 *                 rotation; values are never offset.  Softmax is unchanged since
 *                 q . offset_k[h] is the same for every key of a query, so the
 *                 decode needs no change; the caller keeps the offset fixed for
 *                 the life of the cache.
 *   page_table    unused (may be NULL): placement is by slot_mapping only
 *   slot_mapping  device int64 [num_tokens]; page * P + offset; < 0 skips the token
 *   int2_pages    device uint8 [num_pages][Hkv][2 = K,V][P][D/4]; channel j of a
 *                 row is byte j/4, bits 2*(j%4)..2*(j%4)+1
 *   scale_zero_pages device fp16 [num_pages][Hkv][2][P][D/G][2 = scale, zero]
 * Only the rows of the given slots are written.  A slot past the pool is
 * skipped and flagged OSCAR_DEVERR_SLOT.  num_tokens == 0 is a no-op.
 * Arithmetic: y is accumulated in fp32.  Calls of more than 512 tokens at D = 128
 * multiply on tensor cores with R split into three
 * bf16 terms (about 24 significant bits), so y may differ from a sequential fp32
 * sum by rounding, and a value within rounding of a code boundary may take the
 * neighbouring code.  With an offset that path forms (x . R) - (offset . R), equal
 * to (k - offset) . R up to rounding.
 */
oscar_status_t oscar_append(const oscar_dims_t* dims, int64_t num_tokens, const void* k, const void* v,
                            const float* R_k, const float* R_v, const float* clip_k, const float* clip_v,
                            const float* offset_k, const int32_t* page_table, const int64_t* slot_mapping, uint8_t* int2_pages,
                            void* scale_zero_pages, void* stream);

/*
 * oscar_append_mixed -- oscar_append plus the BF16 rows of the sink and the
 * recent window (project card "How it works": a BF16 sink of the first tokens
 * and a BF16 window of the most recent ones), in the same pass over K/V.
 * Every token with slot_mapping >= 0 is appended to the INT2 pool exactly as by
 * oscar_append.  Its original (unrotated) bf16 K and V rows are also written
 * (with offset_k, the K row is bf16(fp32(k - offset_k[h])), round to nearest even),
 * for sequence b = seq_ids[t] at position p = positions[t], with
 * L = seq_lens[b] the sequence's length after this append:
 *   p < sink_len                      -> bf16_sink[b][K|V][h][p][:]
 *   p >= max(sink_len, L - window_len) -> bf16_window[b][K|V][h][p % window_len][:]
 * Other positions are stored in INT2 only: the decode reads them from there, and
 * a later token of the same call would take their ring slot.  The result is the
 * same as appending the tokens one at a time in position order.
 * Arguments (beyond oscar_append's)
 *   seq_ids, positions  device int32 [num_tokens]
 *   seq_lens            device int32 [batch], lengths after this append
 *   bf16_sink           device bf16 [batch][2][Hkv][sink_len][D] (may be NULL if sink_len == 0)
 *   bf16_window         device bf16 [batch][2][Hkv][window_len][D] (may be NULL if window_len == 0)
 * Errors: OSCAR_ERR_INVALID_ARG for null or negative arguments.  A sequence id
 * outside [0, batch) or a position outside [0, L) skips that token's BF16 rows
 * and sets OSCAR_DEVERR_POSITION.  Rows the call does not write are untouched.
 */
oscar_status_t oscar_append_mixed(const oscar_dims_t* dims, int64_t num_tokens, const void* k, const void* v,
                                  const float* R_k, const float* R_v, const float* clip_k, const float* clip_v,
                                  const float* offset_k, const int32_t* page_table, const int64_t* slot_mapping, const int32_t* seq_ids,
                                  const int32_t* positions, const int32_t* seq_lens, int32_t batch,
                                  int32_t sink_len, int32_t window_len, uint8_t* int2_pages, void* scale_zero_pages,
                                  void* bf16_sink, void* bf16_window, void* stream);

/*
 * Workspace (device bytes) oscar_decode needs for `batch` sequences of at most
 * max_seq_len tokens, splits of pages_per_split pages (0 = automatic) and the
 * given BF16 sink/window lengths.  Returns 0 when the arguments are invalid.
 */
size_t oscar_decode_workspace_bytes(const oscar_dims_t* dims, int32_t batch, int32_t max_seq_len,
                                    int32_t pages_per_split, int32_t sink_len, int32_t window_len);

/*
 * oscar_decode_plan -- how oscar_decode (and oscar_decode_noalloc) runs a decode
 * of these sizes; the arguments are those of oscar_decode_workspace_bytes.  No
 * page defines this call: it reports the library's own schedule.
 *   *fused            1: the single-wave form (head_dim 128, group 64 or 128, when
 *                     every (sequence, KV head) gets its own CTAs in one wave of
 *                     one CTA per SM): INT2 split CTAs that rotate the query
 *                     themselves and un-rotate their own output, one BF16
 *                     sink/window CTA per (sequence, KV head), then a log-sum-exp
 *                     merge -- two kernels;
 *                     0: the general form -- q-rotation, split and merge kernels
 *   *splits           INT2 splits per (sequence, KV head)
 *   *pages_per_split_used  pages per INT2 split
 * Any output pointer may be NULL.  Invalid sizes return OSCAR_ERR_INVALID_ARG.
 */
oscar_status_t oscar_decode_plan(const oscar_dims_t* dims, int32_t batch, int32_t max_seq_len,
                                 int32_t pages_per_split, int32_t sink_len, int32_t window_len, int32_t* fused,
                                 int32_t* splits, int32_t* pages_per_split_used);

/*
 * oscar_decode -- one decode step of mixed-precision paged GQA attention.
 *
 * Defined by: project card "How it works" (a BF16 sink of initial tokens and a
 * BF16 recent window, the bulk in INT2, fused mixed-precision attention) and
 * abstract (INT2 attention kernel over a paged KV cache).  For each sequence b
 * and query head hq (KV head h = hq / (Hq/Hkv)), with L = seq_lens[b]:
 *   sink   positions [0, min(S, L))          bf16_sink[b][K|V][h][p]
 *   window positions [max(S, L-W), L)        bf16_window[b][K|V][h][p % W]
 *   bulk   positions [S, L-W)                INT2 pool, page page_table[b][p/P],
 *                                            offset p % P
 *   logits: sm_scale * q.k for sink/window tokens (original space);
 *           sm_scale * (q.R_k[h]).(c*scale + zero) for bulk tokens (rotated
 *           space, so stored keys are never un-rotated);
 *   out = ( sum_bf16 w_p v_p + (sum_bulk w_p (c*scale+zero)_v) . R_v[h]^T ) / sum_p w_p
 *   with w_p = exp(logit_p - max logit).  A sequence with L == 0 gets zeros.
 * The bulk is cut into splits of pages_per_split pages (flash-decoding); each
 * split keeps (max, sum, partial output) and a merge combines them by
 * log-sum-exp before the single un-rotation.
 * Arguments
 *   max_seq_len   host bound on every seq_lens[b] (<= max_pages_per_seq * P);
 *                 larger device values are clamped and flagged
 *   pages_per_split  0 = chosen from the grid size; else >= 1 (at most 65535 splits
 *                    per sequence, and batch <= 65535: grid dimensions)
 *   q             device bf16 [batch][Hq][D]
 *   R_k, R_v      device fp32 [Hkv][D][D] (the rotations used at append time)
 *   int2_pages, scale_zero_pages   the pools written by oscar_append
 *   bf16_sink     device bf16 [batch][2][Hkv][S][D] (NULL allowed when S == 0)
 *   bf16_window   device bf16 [batch][2][Hkv][W][D] ring (NULL allowed when W == 0)
 *   page_table    device int32 [batch][max_pages_per_seq]
 *   seq_lens      device int32 [batch], tokens in the cache including the current one
 *   sm_scale      softmax scale; <= 0 selects 1/sqrt(D)
 *   out           device fp32 [batch][Hq][D]
 *   workspace     device scratch of at least oscar_decode_workspace_bytes(...)
 *                 bytes, 256-byte aligned; its contents need no initialisation
 */
oscar_status_t oscar_decode(const oscar_dims_t* dims, int32_t batch, int32_t max_seq_len, int32_t pages_per_split,
                            const void* q, const float* R_k, const float* R_v, const uint8_t* int2_pages,
                            const void* scale_zero_pages, const void* bf16_sink, const void* bf16_window,
                            const int32_t* page_table, const int32_t* seq_lens, int32_t sink_len,
                            int32_t window_len, float sm_scale, float* out, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * oscar_append_decode -- one decode step in one call: the current token of every
 * sequence is appended (exactly oscar_append_mixed with token b at position
 * seq_lens[b] - 1 of sequence b: INT2 codes and scale/zero into the pool at
 * slot_mapping[b], the BF16 row into the sink or the window ring), then the queries
 * are decoded (exactly oscar_decode, the appended token included).  The result equals
 * those two calls, bit for bit for up to 512 sequences (the append forms x.R with
 * the FP32 operations of oscar_append_mixed's few-token kernel; for more tokens that
 * call forms x.R on tensor cores, so a code can differ where x.R lies within
 * rounding error of a code boundary).  When window_len >= 1 and the decode runs on its tensor-core
 * kernels (head_dim 128, group 64 or 128, GQA 1..8; the appended position is then in
 * the sink or the window, never read from the INT2 pool by this decode),
 * the append runs inside the decode, in the CTA that attends the sink/window rows
 * holding that position, beside the INT2 splits instead of before them; otherwise
 * the two run one after the other.  Lengths are taken as given, as oscar_append_mixed
 * takes positions: a sequence with seq_lens[b] < 1 has no sink/window row for its
 * token (flagged OSCAR_DEVERR_POSITION; its codes are still written at the slot, and
 * in the fused form that write is not ordered before this decode's reads of the same
 * page), and one longer than max_seq_len is appended at position seq_lens[b] - 1
 * while the decode flags the length.  A negative slot skips the token entirely.
 * (OSCAR project card "How it works": the new K/V are rotated, clipped and quantised
 * as they are appended, and the decode attends a BF16 recent window.)
 * Arguments: those of oscar_decode, plus
 *   k, v          bf16 [batch][Hkv][D]: the current token of each sequence (16-byte aligned)
 *   clip_k, clip_v, offset_k, slot_mapping   as oscar_append_mixed (slot_mapping [batch])
 *   int2_pages, scale_zero_pages, bf16_sink, bf16_window   written (the append) and read
 * Workspace: oscar_decode_workspace_bytes.  Errors: those of both calls; nothing is
 * launched on an argument error.
 */
oscar_status_t oscar_append_decode(const oscar_dims_t* dims, int32_t batch, int32_t max_seq_len,
                                   int32_t pages_per_split, const void* q, const void* k, const void* v,
                                   const float* R_k, const float* R_v, const float* clip_k, const float* clip_v,
                                   const float* offset_k, const int64_t* slot_mapping, uint8_t* int2_pages,
                                   void* scale_zero_pages, void* bf16_sink, void* bf16_window,
                                   const int32_t* page_table, const int32_t* seq_lens, int32_t sink_len,
                                   int32_t window_len, float sm_scale, float* out, void* workspace,
                                   size_t workspace_bytes, void* stream);

/*
 * oscar_extend -- mixed-precision paged attention of many query tokens per
 * sequence (chunked prefill / extend) over the same INT2 + BF16 cache.
 *
 * The decode of oscar_decode generalised to query rows at earlier positions
 * (a reading: the pages describe the fused mixed-precision attention kernels
 * of the serving stack, project card "How it works", abstract "fused kernel
 * pipelines", without fixing the multi-token case).  Query row r belongs to
 * sequence b = row_seq[r] and sits at position p = row_pos[r]; it attends, causally,
 * the positions [0, p] of sequence b's cache of length L = seq_lens[b] (the new
 * tokens are appended first, e.g. by oscar_append_mixed).  Which positions are
 * BF16 (sink, window) and which INT2 is the split of length L, exactly as in
 * oscar_decode; a row at p = L - 1 is a decode query and gives the same output.
 * Arguments (beyond oscar_decode's, whose pools, buffers and tables they share)
 *   batch         number of sequences (rows of page_table, seq_lens, sink, window)
 *   num_rows      number of query rows
 *   max_seq_len   host bound on seq_lens (as oscar_decode)
 *   q             device bf16 [num_rows][Hq][D]
 *   row_seq       device int32 [num_rows], in [0, batch)
 *   row_pos       device int32 [num_rows], in [0, seq_lens[row_seq[r]])
 *   out           device fp32 [num_rows][Hq][D]
 *   workspace     at least oscar_extend_workspace_bytes(dims, num_rows, ...) bytes
 * A row with a sequence or position out of range attends nothing (zeros) and
 * sets OSCAR_DEVERR_POSITION.  Every row reads its pages itself (rows of one
 * sequence share them through L2).
 */
size_t oscar_extend_workspace_bytes(const oscar_dims_t* dims, int32_t num_rows, int32_t max_seq_len,
                                    int32_t pages_per_split, int32_t sink_len, int32_t window_len);
oscar_status_t oscar_extend(const oscar_dims_t* dims, int32_t batch, int32_t num_rows, int32_t max_seq_len,
                            int32_t pages_per_split, const void* q, const int32_t* row_seq, const int32_t* row_pos,
                            const float* R_k, const float* R_v, const uint8_t* int2_pages,
                            const void* scale_zero_pages, const void* bf16_sink, const void* bf16_window,
                            const int32_t* page_table, const int32_t* seq_lens, int32_t sink_len,
                            int32_t window_len, float sm_scale, float* out, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * oscar_extend_varlen -- oscar_extend for the common layout of chunked prefill: the
 * query rows of sequence b are rows q_start[b] .. q_start[b+1]-1 and sit at the
 * last n_b = q_start[b+1] - q_start[b] positions of that sequence (the tokens just
 * appended), in order.  Same result as oscar_extend with those rows.  For head_dim
 * 128, group 64 or 128 and GQA 4 or 8, the INT2 part runs in tiles of 64 / GQA rows
 * of one sequence on tcgen05: every page is fetched and its codes turned into
 * tensor-core operands once per tile instead of once per row.
 * Arguments (beyond oscar_extend's)
 *   num_rows          q_start[batch]; q and out have num_rows rows
 *   max_rows_per_seq  host bound on every n_b (sizes the grid)
 *   q_start           device int32 [batch + 1], non-decreasing, q_start[0] = 0,
 *                     q_start[batch] = num_rows; n_b <= seq_lens[b]
 *   workspace         at least oscar_extend_varlen_workspace_bytes(...) bytes
 * A row beyond a sequence's tokens (n_b > seq_lens[b]) attends nothing and sets
 * OSCAR_DEVERR_POSITION.
 */
size_t oscar_extend_varlen_workspace_bytes(const oscar_dims_t* dims, int32_t num_rows, int32_t max_seq_len,
                                           int32_t pages_per_split, int32_t sink_len, int32_t window_len);
oscar_status_t oscar_extend_varlen(const oscar_dims_t* dims, int32_t batch, int32_t num_rows, int32_t max_seq_len,
                                   int32_t max_rows_per_seq, int32_t pages_per_split, const void* q,
                                   const int32_t* q_start, const float* R_k, const float* R_v,
                                   const uint8_t* int2_pages, const void* scale_zero_pages, const void* bf16_sink,
                                   const void* bf16_window, const int32_t* page_table, const int32_t* seq_lens,
                                   int32_t sink_len, int32_t window_len, float sm_scale, float* out, void* workspace,
                                   size_t workspace_bytes, void* stream);

/*
 * oscar_decode_noalloc -- oscar_decode without a caller workspace.
 *
 * The OSCAR pages have no counterpart for this call; it is a convenience of this
 * library.  It exists for callers that cannot call cudaMalloc, for example a
 * serving engine whose device memory is owned entirely by its own pool (an
 * allocation behind the pool's back breaks its accounting), or a plugin
 * interface that hands the kernel only its input and output buffers.
 * Arguments and results are those of oscar_decode; the workspace is a static
 * device array of OSCAR_NOALLOC_SCRATCH_BYTES inside the library, which every GPU
 * that loads the library holds until the process exits.
 *   - The first call on a device looks up that array's device address (a host
 *     call made once per device, with that device current); make this first call
 *     before any stream capture.  The address is remembered together with the
 *     context it belongs to: after the device's context is destroyed and created
 *     again (cudaDeviceReset), the next call looks it up anew, so that first call
 *     too must come before any stream capture.
 *   - A call whose plan (see oscar_decode_workspace_bytes) needs more than
 *     OSCAR_NOALLOC_SCRATCH_BYTES returns OSCAR_ERR_WORKSPACE and launches nothing.
 *   - Every call shares the one array and it keeps the last call's contents.
 *     Nothing in it needs to start at zero, but calls that overlap on the GPU
 *     (several streams, or several host threads) race on it: serialise them.
 *   - No memory is allocated, by this call or by anything it calls.
 */
#define OSCAR_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
oscar_status_t oscar_decode_noalloc(const oscar_dims_t* dims, int32_t batch, int32_t max_seq_len,
                                    int32_t pages_per_split, const void* q, const float* R_k, const float* R_v,
                                    const uint8_t* int2_pages, const void* scale_zero_pages, const void* bf16_sink,
                                    const void* bf16_window, const int32_t* page_table, const int32_t* seq_lens,
                                    int32_t sink_len, int32_t window_len, float sm_scale, float* out, void* stream);

/*
 * oscar_bf16_append -- store K/V vectors unchanged into a BF16 paged pool (the
 * speedup reference's cache; the pages compare OSCAR against BF16 decoding,
 * summary "Practical Summary").
 *   k, v          device bf16 [num_tokens][Hkv][D], 16-byte aligned
 *   slot_mapping  device int64 [num_tokens]; < 0 skips; past the pool is flagged
 *   bf16_pages    device bf16 [num_pages][Hkv][2][P][D], 16-byte aligned
 * Misaligned k, v or bf16_pages return OSCAR_ERR_INVALID_ARG.
 */
oscar_status_t oscar_bf16_append(const oscar_dims_t* dims, int64_t num_tokens, const void* k, const void* v,
                                 const int64_t* slot_mapping, void* bf16_pages, void* stream);

size_t oscar_bf16_decode_workspace_bytes(const oscar_dims_t* dims, int32_t batch, int32_t max_seq_len,
                                         int32_t pages_per_split);

/*
 * oscar_bf16_decode -- paged GQA decode attention over an all-BF16 cache (the
 * speedup reference).  Every position [0, L) is read from
 * bf16_pages[page_table[b][p/P]][h][K|V][p % P]; out = softmax(sm_scale q.k) v
 * in fp32.  Split-KV with a log-sum-exp merge, as oscar_decode.
 */
oscar_status_t oscar_bf16_decode(const oscar_dims_t* dims, int32_t batch, int32_t max_seq_len,
                                 int32_t pages_per_split, const void* q, const void* bf16_pages,
                                 const int32_t* page_table, const int32_t* seq_lens, float sm_scale, float* out,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * oscar_calibrate -- the offline calibration that produces R and the clipping
 * thresholds consumed by oscar_append, computed on the GPU from calibration
 * samples of the keys and/or values (summary "How OSCAR Works": an offline
 * analysis of the KV covariance designs the rotations, fixed clipping thresholds
 * follow; project card "How it works": covariance structures of keys and values
 * from a small calibration set give the orthogonal rotations and thresholds;
 * abstract).  The pages give no formulas; the readings, per KV head h:
 *   C_h    = (1/N) sum_t (x_t - mu)(x_t - mu)^T, mu = (1/N) sum_t x_t
 *            (centered = 1), or the second moment (1/N) sum_t x_t x_t^T
 *            (centered = 0); the "attention-aware" weighting is not defined on the
 *            pages and is not applied;
 *   R_h    = orthonormal eigenvectors of C_h as columns, eigenvalues descending
 *            (ties by index), each column signed so that its entry of largest
 *            magnitude (lowest row on a tie) is positive; x_rot = x . R_h;
 *   clip_h[j] = the k-th smallest |x_t . R_h[:, j]| over the N samples, with
 *            k = ceil(q N) evaluated in double and kept within [1, N].
 * Arithmetic: the sums of x x^T and x are taken on the tensor cores from the bf16
 * samples with fp32 accumulation (products exact; each chunk of samples is one
 * accumulation chain of 8 MMAs per 128 samples, so its relative error grows with the
 * chunk's length, about N / (16 x number of SMs / (2 Hkv)) units of 2^-23); the chunk
 * partials are added in fp32 in a fixed order, then symmetrised and centred in fp64;
 * the eigenvectors come from cyclic Jacobi in fp32 (a pair is left alone once
 * |a_pq| <= 2^-21 sqrt(|a_pp a_qq|); at most 40 sweeps) followed by one Newton-Schulz
 * step that restores orthogonality to fp32 rounding; |x . R| is formed on the tensor cores
 * with R split into three bf16 terms (about 24 bits) and fp32 accumulation, and the
 * k-th smallest of those fp32 values is selected exactly.  The centred covariance
 * loses relative accuracy in proportion to |mu|^2 / variance (fp32 sums).  Where
 * eigenvalues coincide (or nearly, relative to fp32 rounding) the basis of their
 * eigenspace is not unique and the columns there may differ from another solver's.
 * Arguments
 *   num_samples   N, 1 .. 2^31 - 256
 *   k, v          device bf16 [N][Hkv][D] (the layout oscar_append takes), 16-byte
 *                 aligned; either may be NULL (then its out_* must be NULL too)
 *   centered      1: covariance about the sample mean; 0: second moment
 *   clip_quantile q in (0, 1]; 1 gives the largest magnitude seen
 *   out_k, out_v  outputs for the keys / values (fields below; device buffers):
 *                   R            fp32 [Hkv][D][D] row-major, 16-byte aligned
 *                   clip         fp32 [Hkv][D]
 *                   eigenvalues  fp32 [Hkv][D], descending (may be NULL)
 *                   cov          fp32 [Hkv][D][D], C_h as used (may be NULL)
 *                   sweeps       int32 [Hkv], Jacobi sweeps taken (may be NULL)
 *   workspace     at least oscar_calibrate_workspace_bytes(dims, N) bytes, 16-byte
 *                 aligned; holds per-chunk partial sums and |x . R| for every sample
 *                 (about 4 N Hkv D bytes per side)
 * Only head_dim, num_kv_heads and the general shape checks of dims matter here.
 * Invalid arguments (null R or clip, q outside (0, 1], centered not 0/1, N out of
 * range, k and out_k not both given or both NULL, nothing to calibrate, misaligned
 * pointers) return OSCAR_ERR_INVALID_ARG; a short workspace OSCAR_ERR_WORKSPACE.
 */
typedef struct {
  float* R;
  float* clip;
  float* eigenvalues;
  float* cov;
  int32_t* sweeps;
} oscar_calib_out_t;

size_t oscar_calibrate_workspace_bytes(const oscar_dims_t* dims, int64_t num_samples);
oscar_status_t oscar_calibrate(const oscar_dims_t* dims, int64_t num_samples, const void* k, const void* v,
                               int32_t centered, double clip_quantile, const oscar_calib_out_t* out_k,
                               const oscar_calib_out_t* out_v, void* workspace, size_t workspace_bytes,
                               void* stream);

/* Human-readable name of a status code (static string). */
const char* oscar_status_string(oscar_status_t status);

/*
 * Reads the device error word (OSCAR_DEVERR_* bits) of the current device,
 * OR-ed over all kernels since the last reset; clears it when reset != 0.
 * Synchronises the device.  Returns OSCAR_ERR_CUDA if the read fails.
 */
oscar_status_t oscar_device_errors(uint32_t* flags, int32_t reset);

/*
 * Test hook for the bounded waits (not for production use).  With cycles > 0,
 * every oscar_decode / oscar_decode_noalloc / oscar_extend / oscar_extend_varlen
 * call launched afterwards makes each warp of its INT2 split kernel (single-wave
 * fused form, general form, or the extend's tcgen05 tile kernel) wait for its
 * first page on an mbarrier phase that nothing completes; the wait gives up after
 * `cycles` SM clock cycles.  The kernels then take their timeout path: OSCAR_DEVERR_TIMEOUT
 * is recorded, the copies already issued are awaited, and the split's work is
 * dropped (its partial attends nothing).  cycles == 0 restores normal operation.
 * The setting is process-wide and read at launch time (a captured CUDA graph keeps
 * the value it was captured with).  Returns OSCAR_ERR_INVALID_ARG for cycles < 0.
 */
oscar_status_t oscar_test_stall_page_waits(int64_t cycles);

#ifdef __cplusplus
}
#endif

#endif /* OSCAR_H_ */
