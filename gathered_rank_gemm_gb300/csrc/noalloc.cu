// lora_apply_noalloc: grouping + shrink + expand for one layer without any
// device allocation.  For callers that cannot call cudaMalloc at all - code
// running where the CUDA allocator is off limits (a custom memory manager
// that owns the whole device, a plugin host that hands out no memory, a
// region of a program that must not allocate), so they cannot provide the
// workspace the other entry points ask for.  Their workspace lives here
// instead, in one file-scope device array.
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "gathered_rank_gemm.h"
#include "launch.h"

namespace {

// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kScratchBytes = LORA_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device.  In host code
// the array's name only stands in for the symbol; its device address has to
// be looked up once per device, with that device current.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LORA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return LORA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return LORA_OK;
}

}  // namespace

#pragma GCC visibility push(default)
extern "C" int lora_apply_noalloc(const int32_t* token_lora_mapping, const int32_t* num_tokens,
                                  int64_t max_num_tokens, int64_t max_loras, const uint16_t* x,
                                  int64_t x_row_stride, int64_t hidden,
                                  const uint16_t* const* lora_a, const uint16_t* const* lora_b,
                                  const int64_t* slice_width, int num_slices, int rank,
                                  float scale, const float* lora_scales, float* u, uint16_t* y,
                                  int64_t y_row_stride,
                                  int32_t* sorted_token_ids, int32_t* num_tokens_per_lora,
                                  int32_t* lora_token_start_loc, uint32_t* status, void* stream) {
  const size_t need = lora_workspace_size(max_num_tokens, max_loras);
  if (need == 0) return LORA_ERR_SHAPE;
  if (need > kScratchBytes) return LORA_ERR_WORKSPACE;  // beyond the static scratch
  void* ws = nullptr;
  const int rc0 = scratch_address(&ws);
  if (rc0 != LORA_OK) return rc0;
  // every argument is checked before anything is enqueued
  const int rc1 = grg::check_layer_args(
      token_lora_mapping, num_tokens, max_num_tokens, max_loras, x, x_row_stride, hidden, lora_a,
      lora_b, slice_width, num_slices, rank, u, y, y_row_stride, sorted_token_ids,
      num_tokens_per_lora, lora_token_start_loc, ws, kScratchBytes);
  if (rc1 != LORA_OK) return rc1;
  if (status != nullptr && (reinterpret_cast<uintptr_t>(status) & 3u) != 0) return LORA_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the status word is OR-ed by the grouping kernel: start this call from zero
  if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), s) != cudaSuccess) return LORA_ERR_CUDA;
  int rc = lora_prepare_metadata(token_lora_mapping, num_tokens, max_num_tokens, max_loras,
                                 sorted_token_ids, num_tokens_per_lora, lora_token_start_loc, ws,
                                 kScratchBytes, stream);
  if (rc != LORA_OK) return rc;
  rc = lora_shrink(x, x_row_stride, hidden, lora_a, num_slices, rank, scale, lora_scales, u,
                   sorted_token_ids,
                   lora_token_start_loc, max_num_tokens, max_loras, ws, kScratchBytes, stream);
  if (rc != LORA_OK) return rc;
  rc = lora_expand(u, lora_b, slice_width, num_slices, rank, y, y_row_stride, sorted_token_ids,
                   lora_token_start_loc, max_num_tokens, max_loras, ws, kScratchBytes, stream);
  if (rc != LORA_OK) return rc;
  if (status != nullptr &&
      cudaMemcpyAsync(status, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return LORA_ERR_CUDA;
  return LORA_OK;
}
#pragma GCC visibility pop
