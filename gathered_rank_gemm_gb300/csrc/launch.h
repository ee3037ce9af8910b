// Host-side launch helpers shared by the kernel launchers (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace grg {

// Raises a kernel's dynamic shared-memory limit once per (device, kernel).
int ensure_smem_attr(const void* func, size_t smem_bytes);

// Test hook: while on, every shrink / expand / fused kernel launched arms the
// first barrier it waits on with one arrival too many, issues no copy and
// gives up its waits after 1 ms.  set_wait_fault returns the previous setting.
int set_wait_fault(int on);
int wait_fault();

// Streaming multiprocessors of the current device (cached).
int device_sm_count();

// Resident CTAs per SM for a kernel (cached per device, kernel, block, smem).
int occupancy_blocks(const void* func, int threads, size_t smem_bytes);
// Resident CTAs per SM from the kernel's registers, shared memory and threads
// alone (for kernels the occupancy calculator under-reports).
int resident_blocks(const void* func, int threads, size_t smem_bytes);

// Launches func(params) with programmatic dependent launch allowed and, when
// cluster > 0, a 1-D thread-block cluster of that size.  Returns 0 or a
// LORA_ERR_* code.
int launch_raw(const void* func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
               int cluster, void* params);

template <typename P>
int launch_pdl(const void* func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
               int cluster, P* params) {
  return launch_raw(func, grid, block, smem, stream, cluster, static_cast<void*>(params));
}

// 2-D tensor map over a row-major bf16 matrix [rows][cols] for TMA tile loads
// of box_rows x 64 columns with the 128-byte swizzle (out of range -> zeros).
int make_weight_tmap(CUtensorMap* map, const void* base, long long cols, long long rows,
                     int box_rows);
// The same over a matrix whose rows are row_stride_bytes apart (a multiple of 16).
int make_tmap_2d(CUtensorMap* map, const void* base, long long cols, long long rows,
                 long long row_stride_bytes, int box_rows);

int launch_metadata(const int32_t* mapping, const int32_t* num_tokens, int max_num_tokens,
                    int num_loras, int32_t* sorted_ids, int32_t* counts, int32_t* starts,
                    void* workspace, cudaStream_t stream);

struct ShrinkArgs {
  const void* x;
  long long x_row_stride;
  int hidden;
  const void* lora_a[3];
  int num_slices;
  int rank;
  float scale;
  const float* lora_scales = nullptr;  // per-adapter factors on scale (device, [num_loras])
  float* u;
  const int32_t* sorted_ids;
  const int32_t* starts;
  int max_num_tokens;
  int num_loras;
  const void* workspace;
  // split-K mode: each CTA's partial tile goes to partials[tile][split][16][S*R]
  // (no cluster reduction, u is not written); null for the normal mode
  float* partials = nullptr;
  // paged weights: per slice a device table of max_loras addresses of A_s[l]
  // ([rank][hidden] bf16); all null for stacked weights (lora_a)
  const uint64_t* a_tables[3] = {nullptr, nullptr, nullptr};
  bool f16 = false;  // fp16 x and A (else bf16)
  // the expand of the same call follows at once (the one-call paths): keep
  // the shrink's CTAs small, so that the expand's start beside them, and (in
  // the cluster pair) prefetch the first stages into L2 before the wait
  bool expand_follows = false;
};
int launch_shrink(const ShrinkArgs& a, cudaStream_t stream);
// CTAs sharing one tile's hidden dimension for this shape on the current
// device: the cluster size of the normal mode (at most 8), or the split of
// split-K mode (at most split_k_max(rank): no cluster, so no portable limit).
int shrink_split(const ShrinkArgs& a, bool split_k);
// Largest split-K split for a rank (bounds the expand's staging of partial
// tiles and the workspace's partial-tile area).
constexpr int split_k_max(int rank) { return rank <= 16 ? 16 : 8; }

struct ExpandArgs {
  const float* u;
  const void* lora_b[3];
  int slice_width[3];
  int num_slices;
  int rank;
  void* y;
  long long y_row_stride;
  const int32_t* sorted_ids;
  const int32_t* starts;
  int max_num_tokens;
  int num_loras;
  const void* workspace;
  // split-K mode: sum the shrink's partial tiles (split of them), scale, and
  // write u instead of reading it; null for the normal mode
  const float* partials = nullptr;
  int split = 0;
  float scale = 1.0f;
  const float* lora_scales = nullptr;
  // paged weights: per slice a device table of max_loras addresses of B_s[l]
  // ([rank][slice_width] bf16); all null for stacked weights (lora_b)
  const uint64_t* b_tables[3] = {nullptr, nullptr, nullptr};
  bool f16 = false;  // fp16 y and B (else bf16)
  // y may be read before the dependency wait: only when the expand directly
  // follows this library's shrink on the stream (the one-call path)
  bool y_early = false;
};
int launch_expand(const ExpandArgs& a, cudaStream_t stream);
// The tcgen05 expand (rank 128, stacked weights, more than 1024 tokens): 1
// when launched, 0 when the arguments are not its case, < 0 on error.
int launch_expand_tc(const ExpandArgs& a, cudaStream_t stream);
int expand_tc_applies(const ExpandArgs& a);

// Fused shrink -> expand: 1 when launched, 0 when the shape does not fit the
// fused kernel (run launch_shrink + launch_expand instead), < 0 on error.
int launch_fused(const ShrinkArgs& s, const ExpandArgs& e, cudaStream_t stream);
// 1 when lora_shrink_expand would run the fused kernel for this shape on the
// current device.
int fused_fits(int max_num_tokens, int num_loras, int hidden, const int* widths, int num_slices,
               int rank);

// Every argument check of lora_prepare_metadata, lora_shrink and lora_expand
// for one layer (bf16, stacked weights), without launching anything: LORA_OK
// or the LORA_ERR_* code the first failing call would return.
int check_layer_args(const int32_t* token_lora_mapping, const int32_t* num_tokens,
                     int64_t max_num_tokens, int64_t max_loras, const uint16_t* x,
                     int64_t x_row_stride, int64_t hidden, const uint16_t* const* lora_a,
                     const uint16_t* const* lora_b, const int64_t* slice_width, int num_slices,
                     int rank, float* u, uint16_t* y, int64_t y_row_stride,
                     const int32_t* sorted_token_ids, const int32_t* num_tokens_per_lora,
                     const int32_t* lora_token_start_loc, const void* workspace,
                     size_t workspace_bytes);

}  // namespace grg
