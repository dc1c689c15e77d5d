// Library-wide C ABI entries: status names and the device error word.
#include "common.cuh"

extern "C" const char* oscar_status_string(oscar_status_t status) {
  switch (status) {
    case OSCAR_OK: return "OSCAR_OK";
    case OSCAR_ERR_INVALID_ARG: return "OSCAR_ERR_INVALID_ARG: null pointer or invalid size";
    case OSCAR_ERR_UNSUPPORTED: return "OSCAR_ERR_UNSUPPORTED: shape not implemented";
    case OSCAR_ERR_WORKSPACE: return "OSCAR_ERR_WORKSPACE: workspace too small";
    case OSCAR_ERR_CUDA: return "OSCAR_ERR_CUDA: CUDA call or launch failed";
  }
  return "OSCAR: unknown status";
}

extern "C" oscar_status_t oscar_device_errors(uint32_t* flags, int32_t reset) {
  if (flags == nullptr) return OSCAR_ERR_INVALID_ARG;
  *flags = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return OSCAR_ERR_CUDA;
  oscar_status_t st = oscar_internal_append_errors(flags, reset);
  if (st == OSCAR_OK) st = oscar_internal_decode_errors(flags, reset);
  if (st == OSCAR_OK) st = oscar_internal_decode_mma_errors(flags, reset);
  if (st == OSCAR_OK) st = oscar_internal_decode_fused_errors(flags, reset);
  if (st == OSCAR_OK) st = oscar_internal_decode_bf16_errors(flags, reset);
  if (st == OSCAR_OK) st = oscar_internal_decode_umma_errors(flags, reset);
  if (st == OSCAR_OK) st = oscar_internal_calib_errors(flags, reset);
  return st;
}
