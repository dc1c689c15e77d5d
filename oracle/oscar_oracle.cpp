// OSCAR CPU oracle -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, single-threaded fp64 restatement of what the OSCAR hot path
// computes.  Only the test-suite, the smoke check and the benchmark's CPU
// baseline leg may load this library; the product path never does.  It shares
// no code, header, table or helper with the CUDA library.
//
// Sources (three web pages on OSCAR), cited by title and section:
//   [Summary]   "OSCAR: Cut LLM Inference Costs 8x with 2-bit KV Cache
//               Quantization", sections "Practical Summary" and "How OSCAR Works":
//               fixed rotations and clipping thresholds, 2-bit KV cache.
//   [Card]      project card "FutureMLS-Lab/OSCAR", section "How it works":
//               per-layer orthogonal rotations and clipping thresholds from
//               offline calibration; a BF16 "sink" of initial tokens and a BF16
//               recent window, INT2 bulk.
//   [Abstract]  "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV
//               Cache Quantization", abstract: fixed rotations and clipping
//               thresholds, INT2 attention kernel compatible with paged KV-cache
//               serving.
//   [OptR]      the OptR abstract on that same paper page (a follow-up on
//               output-aware rotations): an attention-equivalent key
//               reparameterisation that removes large per-channel key offsets
//               without changing the softmax distribution, paged format kept.
// The pages give no formulas; the arithmetic below is the plainest reading of
// the words (rotate, clip, per-group asymmetric INT2 with fp16 scale/zero,
// paged storage, softmax attention).  Each such reading carries a tag (R#) and
// is stated in full where it is used.
//
// Parity status: every function here is pinned by tests against closed forms,
// brute force or library routines; the end-to-end numerical values of OSCAR on
// real models are not printed on the pages (parity unpinned for those).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

extern "C" {

// Dimensions of the paged cache, declared here independently of the library.
typedef struct {
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t group_size;
  int32_t num_pages;
  int32_t max_pages_per_seq;
} orc_dims_t;

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------

// bf16 bit pattern -> exact double (bf16 is the top half of an fp32).
double orc_bf16_to_f64(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// IEEE binary16 bit pattern -> exact double.
double orc_f16_to_f64(uint16_t h) {
  const int sign = h >> 15;
  const int e = (h >> 10) & 0x1f;
  const int m = h & 0x3ff;
  double v;
  if (e == 0) {
    v = std::ldexp(static_cast<double>(m), -24);          // subnormal
  } else if (e == 31) {
    v = m ? std::nan("") : HUGE_VAL;
  } else {
    v = std::ldexp(static_cast<double>(m | 0x400), e - 25);  // 1.m * 2^(e-15)
  }
  return sign ? -v : v;
}

// double -> binary16, round to nearest, ties to even.  binary16 keeps 11
// significant bits and its smallest exponent is -14, so the value is rounded
// to a multiple of 2^(max(floor(log2|v|), -14) - 10).
uint16_t orc_f64_to_f16(double v) {
  if (std::isnan(v)) return 0x7e00;
  const uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  const double a = std::fabs(v);
  if (a == 0.0) return sign;
  if (std::isinf(a)) return sign | 0x7c00;
  int e;
  std::frexp(a, &e);                 // a = f * 2^e, f in [0.5, 1)
  int E = e - 1;                     // floor(log2 a)
  if (E < -14) E = -14;
  const double quantum = std::ldexp(1.0, E - 10);
  const double r = std::nearbyint(a / quantum) * quantum;  // default mode: ties to even
  if (r > 65504.0) return sign | 0x7c00;
  if (r < std::ldexp(1.0, -14)) {
    return sign | static_cast<uint16_t>(r / std::ldexp(1.0, -24));
  }
  std::frexp(r, &e);
  E = e - 1;
  const int mant = static_cast<int>(r / std::ldexp(1.0, E - 10)) - 1024;
  return sign | static_cast<uint16_t>(((E + 15) << 10) | mant);
}

// ---------------------------------------------------------------------------
// Append: rotate, clip, quantise, pack, place   ([Summary] Practical Summary,
// [Card] How it works, [Abstract]: fixed rotation R and fixed per-channel clip; INT2)
// ---------------------------------------------------------------------------

// Step A2 (rotation, reading R7): row vector convention, x_rot = x . R, with
// x_rot[j] = sum_i x[i] * R[i][j].  R is row-major fp32 [D][D]; x is given in fp64.
static void rotate_f64(int32_t D, const double* x, const float* R, double* x_rot) {
  for (int j = 0; j < D; ++j) {
    double acc = 0.0;
    for (int i = 0; i < D; ++i) acc += x[i] * static_cast<double>(R[static_cast<size_t>(i) * D + j]);
    x_rot[j] = acc;
  }
}

// Step A2 for a bf16 vector.
void orc_rotate(int32_t D, const uint16_t* x_bf16, const float* R, double* x_rot) {
  std::vector<double> x(D);
  for (int i = 0; i < D; ++i) x[i] = orc_bf16_to_f64(x_bf16[i]);
  rotate_f64(D, x.data(), R, x_rot);
}

// Key offset removal ([OptR]: an attention-equivalent reparameterisation of the
// keys; the subtraction and its precision are reading R26): every key k is replaced by k' = k - c with a fixed per-(KV head,
// channel) fp32 offset c, the difference taken in fp32 (round to nearest even).
// Softmax is unchanged, since q . c is the same for all keys of a query.  Values
// are not offset.  out[i] = fp32(bf16(k_i) - c_i) as an exact double.
void orc_offset_key(int32_t D, const uint16_t* k_bf16, const float* c, double* out) {
  for (int i = 0; i < D; ++i) {
    // the fp64 difference of a bf16 and an fp32 value is exact when their exponents
    // differ by at most 28; otherwise the smaller operand is below a sixteenth of an
    // fp32 ulp of the larger and both roundings give the larger operand's fp32 value
    out[i] = static_cast<double>(static_cast<float>(orc_bf16_to_f64(k_bf16[i]) - static_cast<double>(c[i])));
  }
}

// fp32 -> bf16 bit pattern, round to nearest even (finite inputs).
uint16_t orc_f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  const uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return static_cast<uint16_t>(u >> 16);
}

// The vector that is rotated for token row x of KV head h (K when kv == 0): the key
// minus its offset when an offset is given (reading R26), else the bf16 values.
static void pre_rotation(int32_t D, const uint16_t* x, int kv, const float* offset_k, int h, double* out) {
  if (kv == 0 && offset_k != nullptr) {
    orc_offset_key(D, x, offset_k + static_cast<size_t>(h) * D, out);
  } else {
    for (int i = 0; i < D; ++i) out[i] = orc_bf16_to_f64(x[i]);
  }
}

// Step A3 (clip, reading R6): symmetric per-channel clamp to [-clip_j, +clip_j]
// in rotated space; +inf leaves the channel unchanged.
void orc_clip(int32_t D, double* x, const float* clip) {
  for (int j = 0; j < D; ++j) {
    const double c = static_cast<double>(clip[j]);
    if (x[j] > c) x[j] = c;
    if (x[j] < -c) x[j] = -c;
  }
}

// Step A4 (group parameters, readings R2/R3): asymmetric min/max INT2 over the
// n values of one group.  scale = (max - min) / 3, zero = min; both are stored
// as fp16, rounded through fp32 (the width the values are computed in).
void orc_group_params(int32_t n, const double* xg, uint16_t* s_bits, uint16_t* z_bits) {
  double mn = xg[0], mx = xg[0];
  for (int i = 1; i < n; ++i) {
    if (xg[i] < mn) mn = xg[i];
    if (xg[i] > mx) mx = xg[i];
  }
  const float s32 = static_cast<float>((mx - mn) / 3.0);
  const float z32 = static_cast<float>(mn);
  *s_bits = orc_f64_to_f16(static_cast<double>(s32));
  *z_bits = orc_f64_to_f16(static_cast<double>(z32));
}

// Step A5 (code of one value, readings R3/R5/R5b): the code is computed from
// the STORED fp16 scale and zero, u = (x - z) / s, c = clamp(rint(u), 0, 3),
// ties to even; a zero scale gives code 0.  *u_out receives u (NaN when s==0).
int32_t orc_quantize(double x, uint16_t s_bits, uint16_t z_bits, double* u_out) {
  const double s = orc_f16_to_f64(s_bits);
  const double z = orc_f16_to_f64(z_bits);
  if (s == 0.0) {
    if (u_out) *u_out = std::nan("");
    return 0;
  }
  const double u = (x - z) / s;
  if (u_out) *u_out = u;
  double c = std::nearbyint(u);
  if (c < 0.0) c = 0.0;
  if (c > 3.0) c = 3.0;
  return static_cast<int32_t>(c);
}

// Step A5 over whole rows: codes of n rows of D pre-quantisation values x
// ([n][D] fp64) given stored (scale, zero) bits sz ([n][D/G][2]), with u as in
// orc_quantize.  codes: int32 [n][D]; u: fp64 [n][D].
void orc_codes_given_params(int64_t n, int32_t D, int32_t G, const double* x, const uint16_t* sz,
                            int32_t* codes, double* u) {
  for (int64_t r = 0; r < n; ++r) {
    for (int j = 0; j < D; ++j) {
      const size_t e = static_cast<size_t>(r) * D + j;
      const size_t g = (static_cast<size_t>(r) * (D / G) + j / G) * 2;
      codes[e] = orc_quantize(x[e], sz[g], sz[g + 1], &u[e]);
    }
  }
}

// Byte offset of the packed code row of (page, kv head, K|V, offset): the INT2
// pool is uint8 [num_pages][Hkv][2][P][D/4] (reading R17).
static size_t code_row(const orc_dims_t* d, int64_t page, int h, int kv, int off) {
  return (((static_cast<size_t>(page) * d->num_kv_heads + h) * 2 + kv) * d->page_size + off) *
         static_cast<size_t>(d->head_dim / 4);
}

// Element offset (in fp16 units) of the (scale, zero) pairs of that row: the
// pool is fp16 [num_pages][Hkv][2][P][D/G][2] (reading R17).
static size_t sz_row(const orc_dims_t* d, int64_t page, int h, int kv, int off) {
  return (((static_cast<size_t>(page) * d->num_kv_heads + h) * 2 + kv) * d->page_size + off) *
         static_cast<size_t>(d->head_dim / d->group_size) * 2;
}

// Rotated and clipped values of every (token, head, K|V) vector, fp64
// [T][Hkv][2][D]; tokens whose slot is negative are still computed.
int32_t orc_append_prequant(const orc_dims_t* d, int64_t T, const uint16_t* k, const uint16_t* v,
                            const float* R_k, const float* R_v, const float* clip_k,
                            const float* clip_v, const float* offset_k, double* out) {
  const int H = d->num_kv_heads, D = d->head_dim;
  std::vector<double> x0(D);
  for (int64_t t = 0; t < T; ++t) {
    for (int h = 0; h < H; ++h) {
      for (int kv = 0; kv < 2; ++kv) {
        const uint16_t* x = (kv ? v : k) + (static_cast<size_t>(t) * H + h) * D;
        const float* R = (kv ? R_v : R_k) + static_cast<size_t>(h) * D * D;
        const float* clip = (kv ? clip_v : clip_k) + static_cast<size_t>(h) * D;
        double* y = out + ((static_cast<size_t>(t) * H + h) * 2 + kv) * D;
        pre_rotation(D, x, kv, offset_k, h, x0.data());
        rotate_f64(D, x0.data(), R, y);
        orc_clip(D, y, clip);
      }
    }
  }
  return 0;
}

// Full append (steps A1..A6): for every token t with slot_mapping[t] >= 0,
// every KV head h and each of K and V, rotate, clip, quantise per group and
// write the packed codes and (scale, zero) into page slot / P at offset
// slot % P.  Packing (reading R16): element j of a vector lives in byte j/4 of
// its row, bits 2*(j%4) .. 2*(j%4)+1.  Returns 0, or -1 for a slot outside the
// pool (nothing is written for that token).
int32_t orc_append(const orc_dims_t* d, int64_t T, const uint16_t* k, const uint16_t* v,
                   const float* R_k, const float* R_v, const float* clip_k, const float* clip_v,
                   const float* offset_k, const int64_t* slot_mapping, uint8_t* int2_pages,
                   uint16_t* scale_zero_pages) {
  const int H = d->num_kv_heads, D = d->head_dim, P = d->page_size, G = d->group_size;
  std::vector<double> y(D), x0(D);
  int32_t status = 0;
  for (int64_t t = 0; t < T; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int64_t page = slot / P;
    const int off = static_cast<int>(slot % P);
    if (page >= d->num_pages) {
      status = -1;
      continue;
    }
    for (int h = 0; h < H; ++h) {
      for (int kv = 0; kv < 2; ++kv) {
        const uint16_t* x = (kv ? v : k) + (static_cast<size_t>(t) * H + h) * D;
        const float* R = (kv ? R_v : R_k) + static_cast<size_t>(h) * D * D;
        const float* clip = (kv ? clip_v : clip_k) + static_cast<size_t>(h) * D;
        pre_rotation(D, x, kv, offset_k, h, x0.data());
        rotate_f64(D, x0.data(), R, y.data());
        orc_clip(D, y.data(), clip);
        uint8_t* row = int2_pages + code_row(d, page, h, kv, off);
        uint16_t* sz = scale_zero_pages + sz_row(d, page, h, kv, off);
        std::memset(row, 0, static_cast<size_t>(D / 4));
        for (int g = 0; g < D / G; ++g) {
          uint16_t s_bits, z_bits;
          orc_group_params(G, y.data() + g * G, &s_bits, &z_bits);
          sz[2 * g + 0] = s_bits;
          sz[2 * g + 1] = z_bits;
          for (int i = 0; i < G; ++i) {
            const int j = g * G + i;
            const int32_t c = orc_quantize(y[j], s_bits, z_bits, nullptr);
            row[j / 4] = static_cast<uint8_t>(row[j / 4] | (c << (2 * (j % 4))));
          }
        }
      }
    }
  }
  return status;
}

// Append with the BF16 parts ([Card] "How it works": a BF16 sink of the first
// tokens and a BF16 window of the most recent ones next to the INT2 bulk).  Every
// token t with slot_mapping[t] >= 0 is appended to the INT2 pool exactly as
// orc_append does ("dual write", reading R13).  Its original bf16 K and V rows are
// also stored, unrotated (reading R12; with a key offset the K row is the offset
// key, reading R26), for sequence b = seq_ids[t] at position
// p = positions[t], with L = seq_lens[b] the sequence length after this append
// (reading R18):
//   p < S                  -> sink[b][K|V][h][p][:]
//   p >= max(S, L - W)     -> window[b][K|V][h][p mod W][:]  (reading R11)
// Tokens in neither range are INT2 only: the decode never reads them from the
// BF16 buffers, and a later token of the same append takes their ring slot.
// sink: bf16 bits [B][2][Hkv][S][D]; window: bf16 bits [B][2][Hkv][W][D].
// Returns orc_append's status, or -2 if a token's sequence id or position is out
// of range (its BF16 rows are not written).
int32_t orc_append_mixed(const orc_dims_t* d, int64_t T, const uint16_t* k, const uint16_t* v,
                         const float* R_k, const float* R_v, const float* clip_k, const float* clip_v,
                         const float* offset_k, const int64_t* slot_mapping, const int32_t* seq_ids,
                         const int32_t* positions, const int32_t* seq_lens, int32_t B, int32_t S, int32_t W,
                         uint8_t* int2_pages, uint16_t* scale_zero_pages, uint16_t* sink, uint16_t* window) {
  int32_t status = orc_append(d, T, k, v, R_k, R_v, clip_k, clip_v, offset_k, slot_mapping, int2_pages,
                              scale_zero_pages);
  const int H = d->num_kv_heads, D = d->head_dim;
  std::vector<double> x0(D);
  for (int64_t t = 0; t < T; ++t) {
    if (slot_mapping[t] < 0) continue;
    const int32_t b = seq_ids[t], p = positions[t];
    if (b < 0 || b >= B || p < 0 || p >= seq_lens[b]) {
      status = -2;
      continue;
    }
    const int32_t L = seq_lens[b];
    const int32_t win_begin = (L - W > S) ? L - W : S;
    for (int kv = 0; kv < 2; ++kv) {
      for (int h = 0; h < H; ++h) {
        const uint16_t* x = (kv ? v : k) + (static_cast<size_t>(t) * H + h) * D;
        uint16_t* dst = nullptr;
        if (p < S) {
          dst = sink + (((static_cast<size_t>(b) * 2 + kv) * H + h) * S + p) * D;
        } else if (W > 0 && p >= win_begin) {
          dst = window + (((static_cast<size_t>(b) * 2 + kv) * H + h) * W + p % W) * D;
        }
        if (dst == nullptr) continue;
        if (kv == 0 && offset_k != nullptr) {  // the stored key is the offset key, rounded to bf16
          orc_offset_key(D, x, offset_k + static_cast<size_t>(h) * D, x0.data());
          for (int i = 0; i < D; ++i) dst[i] = orc_f32_to_bf16(static_cast<float>(x0[i]));
        } else {
          std::memcpy(dst, x, static_cast<size_t>(D) * sizeof(uint16_t));
        }
      }
    }
  }
  return status;
}

// ---------------------------------------------------------------------------
// Decode: mixed-precision attention over BF16 sink + BF16 window + INT2 bulk
// ([Card] "How it works": sink of initial tokens and recent window in BF16, the
// bulk in INT2; [Abstract]: paged KV cache)
// ---------------------------------------------------------------------------

// Softmax attention of one query over n tokens, some scored in original space
// (is_rot[i] == 0: logit = sm_scale * q . key_i) and some in rotated space
// (is_rot[i] == 1: logit = sm_scale * q_rot . key_i).  The output is
//   ( sum_{unrotated} w_i v_i  +  (sum_{rotated} w_i v_i) . R_v^T ) / sum_i w_i
// with w_i = exp(logit_i - max logit).  Keys/values are fp64 [n][D].
// An empty token set (n == 0) attends to nothing; its output is zero.
void orc_attend_mixed(int32_t D, int32_t n, const double* q, const double* q_rot,
                      const double* keys, const double* vals, const int32_t* is_rot,
                      double sm_scale, const float* R_v, double* out) {
  if (n == 0) {
    for (int c = 0; c < D; ++c) out[c] = 0.0;
    return;
  }
  std::vector<double> logit(n);
  double m = -HUGE_VAL;
  for (int i = 0; i < n; ++i) {
    const double* qq = is_rot[i] ? q_rot : q;
    double dot = 0.0;
    for (int j = 0; j < D; ++j) dot += qq[j] * keys[static_cast<size_t>(i) * D + j];
    logit[i] = sm_scale * dot;
    if (logit[i] > m) m = logit[i];
  }
  std::vector<double> acc_plain(D, 0.0), acc_rot(D, 0.0);
  double denom = 0.0;
  for (int i = 0; i < n; ++i) {
    const double w = std::exp(logit[i] - m);
    denom += w;
    std::vector<double>& acc = is_rot[i] ? acc_rot : acc_plain;
    for (int j = 0; j < D; ++j) acc[j] += w * vals[static_cast<size_t>(i) * D + j];
  }
  bool any_rot = false;
  for (int i = 0; i < n; ++i) any_rot = any_rot || is_rot[i];
  for (int c = 0; c < D; ++c) {
    // (acc_rot . R^T)[c] = sum_j acc_rot[j] * R[c][j]; R_v is only read when
    // some token was rotated.
    double unrot = 0.0;
    if (any_rot) {
      for (int j = 0; j < D; ++j) unrot += acc_rot[j] * static_cast<double>(R_v[static_cast<size_t>(c) * D + j]);
    }
    out[c] = (acc_plain[c] + unrot) / denom;
  }
}

// Dequantised rotated vector of one stored INT2 row: x~_j = c_j * s_g + z_g.
void orc_dequant_row(const orc_dims_t* d, const uint8_t* int2_pages, const uint16_t* scale_zero_pages,
                     int64_t page, int32_t h, int32_t kv, int32_t off, double* x) {
  const int D = d->head_dim, G = d->group_size;
  const uint8_t* row = int2_pages + code_row(d, page, h, kv, off);
  const uint16_t* sz = scale_zero_pages + sz_row(d, page, h, kv, off);
  for (int j = 0; j < D; ++j) {
    const int c = (row[j / 4] >> (2 * (j % 4))) & 3;
    const double s = orc_f16_to_f64(sz[2 * (j / G) + 0]);
    const double z = orc_f16_to_f64(sz[2 * (j / G) + 1]);
    x[j] = c * s + z;
  }
}

// Attention of one query (bf16 bits q_row, head hq) of sequence b over the
// cache of length L, restricted to positions p < A (A <= L).  The cache split
// is the one of length L (readings R11-R13):
//   sink   p in [0, min(S, L))                 from bf16_sink[b][K|V][h][p]
//   window p in [max(S, L - W), L)              from bf16_window[b][K|V][h][p % W]
//   bulk   p in [S, L - W)                      from the INT2 pool at page
//          page_table[b][p / P], offset p % P, scored with q_rot = q . R_k[h]
// softmax with scale sm_scale, bulk output un-rotated by R_v[h]^T.  Returns 0,
// or -1 when a page id is outside the pool.
static int32_t attend_query(const orc_dims_t* d, const uint16_t* q_row, int hq, int b, int L, int A,
                            const float* R_k, const float* R_v, const uint8_t* int2_pages,
                            const uint16_t* scale_zero_pages, const uint16_t* bf16_sink,
                            const uint16_t* bf16_window, const int32_t* page_table, int S, int W,
                            double sm_scale, double* out) {
  const int Hq = d->num_q_heads, H = d->num_kv_heads, D = d->head_dim, P = d->page_size;
  const int gqa = Hq / H;
  const int h = hq / gqa;
  std::vector<double> qv(D), qr(D);
  for (int j = 0; j < D; ++j) qv[j] = orc_bf16_to_f64(q_row[j]);
  // q_rot = q . R_k[h]
  const float* Rk = R_k + static_cast<size_t>(h) * D * D;
  for (int j = 0; j < D; ++j) {
    double acc = 0.0;
    for (int i = 0; i < D; ++i) acc += qv[i] * static_cast<double>(Rk[static_cast<size_t>(i) * D + j]);
    qr[j] = acc;
  }
  std::vector<double> keys(static_cast<size_t>(A) * D), vals(static_cast<size_t>(A) * D);
  std::vector<int32_t> is_rot(A, 0);
  int n = 0;
  const int sink_end = L < S ? L : S;
  const int win_begin = (L - W > S) ? L - W : S;
  for (int p = 0; p < A; ++p) {
    double* kk = keys.data() + static_cast<size_t>(n) * D;
    double* vv = vals.data() + static_cast<size_t>(n) * D;
    if (p < sink_end) {
      const size_t kb = ((static_cast<size_t>(b) * 2 + 0) * H + h) * S + p;
      const size_t vb = ((static_cast<size_t>(b) * 2 + 1) * H + h) * S + p;
      for (int j = 0; j < D; ++j) {
        kk[j] = orc_bf16_to_f64(bf16_sink[kb * D + j]);
        vv[j] = orc_bf16_to_f64(bf16_sink[vb * D + j]);
      }
      is_rot[n] = 0;
    } else if (p >= win_begin) {
      const size_t kb = ((static_cast<size_t>(b) * 2 + 0) * H + h) * W + (p % W);
      const size_t vb = ((static_cast<size_t>(b) * 2 + 1) * H + h) * W + (p % W);
      for (int j = 0; j < D; ++j) {
        kk[j] = orc_bf16_to_f64(bf16_window[kb * D + j]);
        vv[j] = orc_bf16_to_f64(bf16_window[vb * D + j]);
      }
      is_rot[n] = 0;
    } else {
      const int64_t page = page_table[static_cast<size_t>(b) * d->max_pages_per_seq + p / P];
      if (page < 0 || page >= d->num_pages) return -1;
      orc_dequant_row(d, int2_pages, scale_zero_pages, page, h, 0, p % P, kk);
      orc_dequant_row(d, int2_pages, scale_zero_pages, page, h, 1, p % P, vv);
      is_rot[n] = 1;
    }
    ++n;
  }
  orc_attend_mixed(D, n, qv.data(), qr.data(), keys.data(), vals.data(), is_rot.data(), sm_scale,
                   R_v + static_cast<size_t>(h) * D * D, out);
  return 0;
}

// Decode for a list of (batch index, query head) pairs.  For pair (b, hq):
// kv head h = hq / (Hq / Hkv) (reading R10); L = seq_lens[b] (reading R18); the
// query attends every position [0, L) of the cache (attend_query).  sm_scale
// <= 0 means 1/sqrt(D) (reading R9).  out: fp64 [n_pairs][D].
// Returns 0, or -1 when a page id is outside the pool or L exceeds the table.
int32_t orc_decode(const orc_dims_t* d, int32_t batch, const uint16_t* q, const float* R_k,
                   const float* R_v, const uint8_t* int2_pages, const uint16_t* scale_zero_pages,
                   const uint16_t* bf16_sink, const uint16_t* bf16_window, const int32_t* page_table,
                   const int32_t* seq_lens, int32_t sink_len, int32_t window_len, double sm_scale,
                   int32_t n_pairs, const int32_t* pairs, double* out) {
  const int Hq = d->num_q_heads, D = d->head_dim, P = d->page_size;
  if (sm_scale <= 0.0) sm_scale = 1.0 / std::sqrt(static_cast<double>(D));
  for (int pi = 0; pi < n_pairs; ++pi) {
    const int b = pairs[2 * pi], hq = pairs[2 * pi + 1];
    const int L = seq_lens[b];
    if (L > d->max_pages_per_seq * P || b >= batch) return -1;
    if (attend_query(d, q + (static_cast<size_t>(b) * Hq + hq) * D, hq, b, L, L, R_k, R_v, int2_pages,
                     scale_zero_pages, bf16_sink, bf16_window, page_table, sink_len, window_len, sm_scale,
                     out + static_cast<size_t>(pi) * D) != 0)
      return -1;
  }
  return 0;
}

// Extend (chunked prefill) attention for a list of (query row, query head)
// pairs: query row r belongs to sequence b = row_seq[r] at position
// row_pos[r] and attends, causally, the positions [0, row_pos[r]] of that
// sequence's cache of length L = seq_lens[b] (the new tokens are already in the
// cache; the sink/window/bulk split is the one of length L; reading R24).  A
// row at position L - 1 is exactly a decode query.  out: fp64 [n_pairs][D].
// Returns 0, or -1 for a sequence or position out of range or a bad page id.
int32_t orc_extend(const orc_dims_t* d, int32_t batch, int32_t num_rows, const uint16_t* q,
                   const int32_t* row_seq, const int32_t* row_pos, const float* R_k, const float* R_v,
                   const uint8_t* int2_pages, const uint16_t* scale_zero_pages, const uint16_t* bf16_sink,
                   const uint16_t* bf16_window, const int32_t* page_table, const int32_t* seq_lens,
                   int32_t sink_len, int32_t window_len, double sm_scale, int32_t n_pairs, const int32_t* pairs,
                   double* out) {
  const int Hq = d->num_q_heads, D = d->head_dim, P = d->page_size;
  if (sm_scale <= 0.0) sm_scale = 1.0 / std::sqrt(static_cast<double>(D));
  for (int pi = 0; pi < n_pairs; ++pi) {
    const int r = pairs[2 * pi], hq = pairs[2 * pi + 1];
    if (r < 0 || r >= num_rows) return -1;
    const int b = row_seq[r];
    if (b < 0 || b >= batch) return -1;
    const int L = seq_lens[b];
    if (L > d->max_pages_per_seq * P) return -1;
    const int pos = row_pos[r];
    if (pos < 0 || pos >= L) return -1;
    if (attend_query(d, q + (static_cast<size_t>(r) * Hq + hq) * D, hq, b, L, pos + 1, R_k, R_v, int2_pages,
                     scale_zero_pages, bf16_sink, bf16_window, page_table, sink_len, window_len, sm_scale,
                     out + static_cast<size_t>(pi) * D) != 0)
      return -1;
  }
  return 0;
}

// BF16 paged decode (the speedup reference): every token p in [0, L) is read
// from the bf16 pool [num_pages][Hkv][2][P][D] at page_table[b][p / P], offset
// p % P, in original space; plain softmax attention.  out: fp64 [n_pairs][D].
int32_t orc_bf16_decode(const orc_dims_t* d, int32_t batch, const uint16_t* q, const uint16_t* bf16_pages,
                        const int32_t* page_table, const int32_t* seq_lens, double sm_scale,
                        int32_t n_pairs, const int32_t* pairs, double* out) {
  const int Hq = d->num_q_heads, H = d->num_kv_heads, D = d->head_dim, P = d->page_size;
  const int gqa = Hq / H;
  if (sm_scale <= 0.0) sm_scale = 1.0 / std::sqrt(static_cast<double>(D));
  for (int pi = 0; pi < n_pairs; ++pi) {
    const int b = pairs[2 * pi], hq = pairs[2 * pi + 1];
    const int h = hq / gqa;
    const int L = seq_lens[b];
    if (L > d->max_pages_per_seq * P || b >= batch) return -1;
    std::vector<double> qv(D);
    for (int j = 0; j < D; ++j) qv[j] = orc_bf16_to_f64(q[(static_cast<size_t>(b) * Hq + hq) * D + j]);
    std::vector<double> keys(static_cast<size_t>(L) * D), vals(static_cast<size_t>(L) * D);
    std::vector<int32_t> is_rot(L, 0);
    for (int p = 0; p < L; ++p) {
      const int64_t page = page_table[static_cast<size_t>(b) * d->max_pages_per_seq + p / P];
      if (page < 0 || page >= d->num_pages) return -1;
      const size_t kb = (((static_cast<size_t>(page) * H + h) * 2 + 0) * P + p % P) * D;
      const size_t vb = (((static_cast<size_t>(page) * H + h) * 2 + 1) * P + p % P) * D;
      for (int j = 0; j < D; ++j) {
        keys[static_cast<size_t>(p) * D + j] = orc_bf16_to_f64(bf16_pages[kb + j]);
        vals[static_cast<size_t>(p) * D + j] = orc_bf16_to_f64(bf16_pages[vb + j]);
      }
    }
    // No rotated tokens, so R_v is never read.
    orc_attend_mixed(D, L, qv.data(), qv.data(), keys.data(), vals.data(), is_rot.data(), sm_scale,
                     nullptr, out + static_cast<size_t>(pi) * D);
  }
  return 0;
}

}  // extern "C"
