// Shared host/device helpers of the OSCAR CUDA library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <set>
#include <utility>

#include "oscar.h"

namespace oscar {

// Each translation unit keeps its own device error word (the library is built
// without relocatable device code); oscar_device_errors ORs them together.
static __device__ unsigned int g_dev_err = 0;

__device__ __forceinline__ void record_error(unsigned int bits) { atomicOr(&g_dev_err, bits); }

// Host side: read this unit's error word, optionally clearing it.
static inline cudaError_t read_unit_errors(uint32_t* out, int reset) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_dev_err, sizeof(v));
  if (e != cudaSuccess) return e;
  *out |= v;
  if (reset) {
    v = 0;
    e = cudaMemcpyToSymbol(g_dev_err, &v, sizeof(v));
  }
  return e;
}

constexpr int kPageSize = 16;
constexpr int kMaxGqa = 8;

// Common shape checks; returns OSCAR_OK or the status to report.
static inline oscar_status_t check_dims(const oscar_dims_t* d) {
  if (d == nullptr) return OSCAR_ERR_INVALID_ARG;
  if (d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0 || d->page_size <= 0 ||
      d->group_size <= 0 || d->num_pages <= 0 || d->max_pages_per_seq <= 0)
    return OSCAR_ERR_INVALID_ARG;
  if (d->num_q_heads % d->num_kv_heads != 0) return OSCAR_ERR_INVALID_ARG;
  if (d->head_dim % d->group_size != 0) return OSCAR_ERR_INVALID_ARG;
  if (d->head_dim != 64 && d->head_dim != 128) return OSCAR_ERR_UNSUPPORTED;
  if (d->page_size != kPageSize) return OSCAR_ERR_UNSUPPORTED;
  if (d->group_size != 32 && d->group_size != 64 && d->group_size != 128) return OSCAR_ERR_UNSUPPORTED;
  if (d->num_q_heads / d->num_kv_heads > kMaxGqa) return OSCAR_ERR_UNSUPPORTED;
  return OSCAR_OK;
}

static inline bool misaligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

static inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Number of SMs of the current device (cached per process for device 0..63).
static inline int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

// Sets a kernel's dynamic shared-memory limit once per (kernel, device), so
// later launches (including ones recorded into a CUDA graph) only launch.
static inline cudaError_t set_smem_limit_once(const void* func, size_t bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({func, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) done.insert({func, dev});
  return e;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

}  // namespace oscar

// oscar_append_mixed of the current token of every sequence (append.cu).
oscar_status_t oscar_internal_append_current(const oscar_dims_t* dims, int32_t batch, const void* k, const void* v,
                                             const float* R_k, const float* R_v, const float* clip_k,
                                             const float* clip_v, const float* offset_k,
                                             const int64_t* slot_mapping, const int32_t* seq_lens,
                                             int32_t sink_len, int32_t window_len, uint8_t* int2_pages,
                                             void* scale_zero_pages, void* bf16_sink, void* bf16_window,
                                             void* stream);

// Per-unit error readers (each defined in its own .cu file).
oscar_status_t oscar_internal_append_errors(uint32_t* flags, int reset);
oscar_status_t oscar_internal_decode_errors(uint32_t* flags, int reset);
oscar_status_t oscar_internal_decode_mma_errors(uint32_t* flags, int reset);
oscar_status_t oscar_internal_decode_fused_errors(uint32_t* flags, int reset);
oscar_status_t oscar_internal_decode_bf16_errors(uint32_t* flags, int reset);
oscar_status_t oscar_internal_decode_umma_errors(uint32_t* flags, int reset);
oscar_status_t oscar_internal_calib_errors(uint32_t* flags, int reset);
