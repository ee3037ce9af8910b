// The C ABI: argument validation and dispatch to the kernel launchers.
// Declarations and the full contract live in include/gathered_rank_gemm.h.
#include <cstdint>

#include "gathered_rank_gemm.h"
#include "gathered_rank_gemm_testing.h"
#include "common.cuh"
#include "launch.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool sizes_ok(int64_t max_num_tokens, int64_t max_loras) {
  return max_num_tokens >= 1 && max_num_tokens <= LORA_MAX_NUM_TOKENS && max_loras >= 1 &&
         max_loras <= LORA_MAX_LORAS;
}

bool rank_ok(int rank) {
  return rank == 8 || rank == 16 || rank == 32 || rank == 64 || rank == 128;
}

constexpr int64_t kMaxHidden = 1 << 20;
constexpr int64_t kMaxWidth = 1 << 20;

// Argument checks of lora_shrink; fills the launcher's arguments.
// Weights come either stacked (lora_a) or paged (a_tables: per slice a device
// table of max_loras addresses); exactly one of the two is given.
int shrink_args(const uint16_t* x, int64_t x_row_stride, int64_t hidden,
                const uint16_t* const* lora_a, const uint64_t* const* a_tables, int num_slices,
                int rank, float scale, const float* lora_scales, float* u,
                const int32_t* sorted_token_ids, const int32_t* lora_token_start_loc,
                int64_t max_num_tokens, int64_t max_loras, const void* workspace,
                size_t workspace_bytes, grg::ShrinkArgs* out, bool need_u = true) {
  const bool paged = a_tables != nullptr;
  if (!x || (!lora_a && !paged) || (need_u && !u) || !sorted_token_ids ||
      !lora_token_start_loc || !workspace)
    return LORA_ERR_NULL;
  if (num_slices < 1 || num_slices > LORA_MAX_SLICES) return LORA_ERR_SHAPE;
  for (int s = 0; s < num_slices; ++s)
    if (paged ? !a_tables[s] : !lora_a[s]) return LORA_ERR_NULL;
  if (!sizes_ok(max_num_tokens, max_loras) || !rank_ok(rank) || hidden < 8 ||
      hidden > kMaxHidden || (hidden % 8) != 0 || x_row_stride < hidden)
    return LORA_ERR_SHAPE;
  if (!aligned16(x) || (x_row_stride % 8) != 0 || (need_u && !aligned16(u)) ||
      !aligned16(workspace))
    return LORA_ERR_ALIGN;
  for (int s = 0; s < num_slices; ++s)
    if (paged ? (reinterpret_cast<uintptr_t>(a_tables[s]) % 8) != 0 : !aligned16(lora_a[s]))
      return LORA_ERR_ALIGN;
  if (workspace_bytes < grg::workspace_bytes_needed(max_num_tokens, max_loras))
    return LORA_ERR_WORKSPACE;
  grg::ShrinkArgs& a = *out;
  a.x = x;
  a.x_row_stride = x_row_stride;
  a.hidden = static_cast<int>(hidden);
  for (int s = 0; s < 3; ++s) {
    a.lora_a[s] = paged ? nullptr : (s < num_slices ? lora_a[s] : lora_a[0]);
    a.a_tables[s] = paged ? (s < num_slices ? a_tables[s] : a_tables[0]) : nullptr;
  }
  a.num_slices = num_slices;
  a.rank = rank;
  a.scale = scale;
  a.lora_scales = lora_scales;
  a.u = u;
  a.sorted_ids = sorted_token_ids;
  a.starts = lora_token_start_loc;
  a.max_num_tokens = static_cast<int>(max_num_tokens);
  a.num_loras = static_cast<int>(max_loras);
  a.workspace = workspace;
  return LORA_OK;
}

// Argument checks of lora_expand; fills the launcher's arguments.
int expand_args(const float* u, const uint16_t* const* lora_b, const uint64_t* const* b_tables,
                const int64_t* slice_width, int num_slices, int rank, uint16_t* y,
                int64_t y_row_stride, const int32_t* sorted_token_ids,
                const int32_t* lora_token_start_loc, int64_t max_num_tokens, int64_t max_loras,
                const void* workspace, size_t workspace_bytes, grg::ExpandArgs* out) {
  const bool paged = b_tables != nullptr;
  if (!u || (!lora_b && !paged) || !slice_width || !y || !sorted_token_ids ||
      !lora_token_start_loc || !workspace)
    return LORA_ERR_NULL;
  if (num_slices < 1 || num_slices > LORA_MAX_SLICES) return LORA_ERR_SHAPE;
  int64_t total = 0;
  for (int s = 0; s < num_slices; ++s) {
    if (paged ? !b_tables[s] : !lora_b[s]) return LORA_ERR_NULL;
    if (slice_width[s] < 8 || slice_width[s] > kMaxWidth || (slice_width[s] % 8) != 0)
      return LORA_ERR_SHAPE;
    total += slice_width[s];
  }
  if (!sizes_ok(max_num_tokens, max_loras) || !rank_ok(rank) || y_row_stride < total)
    return LORA_ERR_SHAPE;
  if (!aligned16(u) || !aligned16(y) || (y_row_stride % 8) != 0 || !aligned16(workspace))
    return LORA_ERR_ALIGN;
  for (int s = 0; s < num_slices; ++s)
    if (paged ? (reinterpret_cast<uintptr_t>(b_tables[s]) % 8) != 0 : !aligned16(lora_b[s]))
      return LORA_ERR_ALIGN;
  if (workspace_bytes < grg::workspace_bytes_needed(max_num_tokens, max_loras))
    return LORA_ERR_WORKSPACE;
  grg::ExpandArgs& a = *out;
  a.u = u;
  for (int s = 0; s < 3; ++s) {
    a.lora_b[s] = paged ? nullptr : (s < num_slices ? lora_b[s] : lora_b[0]);
    a.b_tables[s] = paged ? (s < num_slices ? b_tables[s] : b_tables[0]) : nullptr;
    a.slice_width[s] = s < num_slices ? static_cast<int>(slice_width[s]) : 0;
  }
  a.num_slices = num_slices;
  a.rank = rank;
  a.y = y;
  a.y_row_stride = y_row_stride;
  a.sorted_ids = sorted_token_ids;
  a.starts = lora_token_start_loc;
  a.max_num_tokens = static_cast<int>(max_num_tokens);
  a.num_loras = static_cast<int>(max_loras);
  a.workspace = workspace;
  return LORA_OK;
}

}  // namespace

#pragma GCC visibility push(default)
extern "C" {

size_t lora_workspace_size(int64_t max_num_tokens, int64_t max_loras) {
  if (!sizes_ok(max_num_tokens, max_loras)) return 0;
  return grg::workspace_bytes_needed(max_num_tokens, max_loras);
}

namespace {
// Split-K one-call path: batches of up to 1024 tokens (16-token tiles) and
// ranks up to 32.  Its partial tiles follow the metadata part of the
// workspace: [16-token tile][split <= split_k_max(rank)][16][S*R] fp32.
constexpr int64_t kSplitMaxTokens = 1024;
constexpr int kSplitMaxRank = 32;
bool split_shape(int64_t max_num_tokens, int rank) {
  return max_num_tokens <= kSplitMaxTokens && rank <= kSplitMaxRank;
}
// The partial tiles, behind the metadata part of the workspace.
size_t split_scratch_bytes(int64_t max_num_tokens, int64_t max_loras, int num_slices, int rank) {
  return static_cast<size_t>(grg::tile_list_capacity(max_num_tokens, max_loras, 0)) *
         grg::split_k_max(rank) * 16 * num_slices * rank * 4;
}
float* split_partials(const void* workspace, int64_t max_num_tokens, int64_t max_loras) {
  return reinterpret_cast<float*>(static_cast<char*>(const_cast<void*>(workspace)) +
                                  grg::workspace_bytes_needed(max_num_tokens, max_loras));
}
}  // namespace

size_t lora_shrink_expand_workspace_size(int64_t max_num_tokens, int64_t max_loras,
                                         int64_t hidden, const int64_t* slice_width,
                                         int num_slices, int rank) {
  const size_t base = lora_workspace_size(max_num_tokens, max_loras);
  if (base == 0 || !slice_width || num_slices < 1 || num_slices > LORA_MAX_SLICES ||
      !rank_ok(rank) || hidden < 8 || hidden > kMaxHidden || (hidden % 8) != 0)
    return 0;
  for (int s = 0; s < num_slices; ++s)
    if (slice_width[s] < 8 || slice_width[s] > kMaxWidth || (slice_width[s] % 8) != 0) return 0;
  if (!split_shape(max_num_tokens, rank)) return base;
  return base + split_scratch_bytes(max_num_tokens, max_loras, num_slices, rank);
}

namespace {
// CTAs per tile of the split-K shrink for a shape (the shrink's cluster rule).
int split_of(int64_t max_num_tokens, int64_t max_loras, int64_t hidden, int num_slices,
             int rank) {
  grg::ShrinkArgs a;
  a.hidden = static_cast<int>(hidden);
  a.num_slices = num_slices;
  a.rank = rank;
  a.max_num_tokens = static_cast<int>(max_num_tokens);
  a.num_loras = static_cast<int>(max_loras);
  return grg::shrink_split(a, true);
}
}  // namespace

namespace {
int shrink_partials(const uint16_t* x, int64_t x_row_stride, int64_t hidden,
                    const uint16_t* const* lora_a, int num_slices, int rank,
                    const int32_t* sorted_token_ids, const int32_t* lora_token_start_loc,
                    int64_t max_num_tokens, int64_t max_loras, void* workspace,
                    size_t workspace_bytes, void* stream, bool f16) {
  grg::ShrinkArgs sa;
  const int rc = shrink_args(x, x_row_stride, hidden, lora_a, nullptr, num_slices, rank, 1.0f,
                             nullptr, nullptr, sorted_token_ids, lora_token_start_loc,
                             max_num_tokens, max_loras, workspace, workspace_bytes, &sa, false);
  if (rc != LORA_OK) return rc;
  if (!split_shape(max_num_tokens, rank)) return LORA_ERR_SHAPE;
  const size_t base = grg::workspace_bytes_needed(max_num_tokens, max_loras);
  if (workspace_bytes < base + split_scratch_bytes(max_num_tokens, max_loras, num_slices, rank))
    return LORA_ERR_WORKSPACE;
  sa.partials = split_partials(workspace, max_num_tokens, max_loras);
  sa.f16 = f16;
  return grg::launch_shrink(sa, static_cast<cudaStream_t>(stream));
}
}  // namespace

int lora_shrink_partials(const uint16_t* x, int64_t x_row_stride, int64_t hidden,
                         const uint16_t* const* lora_a, int num_slices, int rank,
                         const int32_t* sorted_token_ids, const int32_t* lora_token_start_loc,
                         int64_t max_num_tokens, int64_t max_loras, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return shrink_partials(x, x_row_stride, hidden, lora_a, num_slices, rank, sorted_token_ids,
                         lora_token_start_loc, max_num_tokens, max_loras, workspace,
                         workspace_bytes, stream, false);
}

int lora_shrink_partials_f16(const uint16_t* x, int64_t x_row_stride, int64_t hidden,
                             const uint16_t* const* lora_a, int num_slices, int rank,
                             const int32_t* sorted_token_ids, const int32_t* lora_token_start_loc,
                             int64_t max_num_tokens, int64_t max_loras, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return shrink_partials(x, x_row_stride, hidden, lora_a, num_slices, rank, sorted_token_ids,
                         lora_token_start_loc, max_num_tokens, max_loras, workspace,
                         workspace_bytes, stream, true);
}

namespace {
int expand_partials(int64_t hidden, const uint16_t* const* lora_b, const int64_t* slice_width,
                    int num_slices, int rank, float scale, const float* lora_scales, float* u,
                    uint16_t* y,
                    int64_t y_row_stride, const int32_t* sorted_token_ids,
                    const int32_t* lora_token_start_loc, int64_t max_num_tokens,
                    int64_t max_loras, const void* workspace, size_t workspace_bytes,
                    void* stream, bool y_early, bool f16) {
  grg::ExpandArgs ea;
  const int rc = expand_args(u, lora_b, nullptr, slice_width, num_slices, rank, y, y_row_stride,
                             sorted_token_ids, lora_token_start_loc, max_num_tokens, max_loras,
                             workspace, workspace_bytes, &ea);
  if (rc != LORA_OK) return rc;
  if (hidden < 8 || hidden > kMaxHidden || (hidden % 8) != 0 ||
      !split_shape(max_num_tokens, rank))
    return LORA_ERR_SHAPE;
  const size_t base = grg::workspace_bytes_needed(max_num_tokens, max_loras);
  if (workspace_bytes < base + split_scratch_bytes(max_num_tokens, max_loras, num_slices, rank))
    return LORA_ERR_WORKSPACE;
  ea.partials = split_partials(workspace, max_num_tokens, max_loras);
  ea.split = split_of(max_num_tokens, max_loras, hidden, num_slices, rank);
  ea.scale = scale;
  ea.lora_scales = lora_scales;
  ea.y_early = y_early;
  ea.f16 = f16;
  return grg::launch_expand(ea, static_cast<cudaStream_t>(stream));
}
}  // namespace

int lora_expand_partials(int64_t hidden, const uint16_t* const* lora_b,
                         const int64_t* slice_width, int num_slices, int rank, float scale,
                         const float* lora_scales, float* u, uint16_t* y, int64_t y_row_stride,
                         const int32_t* sorted_token_ids, const int32_t* lora_token_start_loc,
                         int64_t max_num_tokens, int64_t max_loras, const void* workspace,
                         size_t workspace_bytes, void* stream) {
  // the caller may run anything between the halves: y only after the wait
  return expand_partials(hidden, lora_b, slice_width, num_slices, rank, scale, lora_scales, u, y,
                         y_row_stride, sorted_token_ids, lora_token_start_loc, max_num_tokens,
                         max_loras, workspace, workspace_bytes, stream, false, false);
}

int lora_expand_partials_f16(int64_t hidden, const uint16_t* const* lora_b,
                             const int64_t* slice_width, int num_slices, int rank, float scale,
                             const float* lora_scales, float* u, uint16_t* y,
                             int64_t y_row_stride, const int32_t* sorted_token_ids,
                             const int32_t* lora_token_start_loc, int64_t max_num_tokens,
                             int64_t max_loras, const void* workspace, size_t workspace_bytes,
                             void* stream) {
  return expand_partials(hidden, lora_b, slice_width, num_slices, rank, scale, lora_scales, u, y,
                         y_row_stride, sorted_token_ids, lora_token_start_loc, max_num_tokens,
                         max_loras, workspace, workspace_bytes, stream, false, true);
}

}  // extern "C"

namespace {
// Argument checks of lora_prepare_metadata.
int metadata_args(const int32_t* token_lora_mapping, const int32_t* num_tokens,
                  int64_t max_num_tokens, int64_t max_loras, const int32_t* sorted_token_ids,
                  const int32_t* num_tokens_per_lora, const int32_t* lora_token_start_loc,
                  const void* workspace, size_t workspace_bytes) {
  if (!token_lora_mapping || !num_tokens || !sorted_token_ids || !num_tokens_per_lora ||
      !lora_token_start_loc || !workspace)
    return LORA_ERR_NULL;
  if (!sizes_ok(max_num_tokens, max_loras)) return LORA_ERR_SHAPE;
  if (!aligned16(workspace) || (reinterpret_cast<uintptr_t>(token_lora_mapping) & 3u) ||
      (reinterpret_cast<uintptr_t>(num_tokens) & 3u) ||
      (reinterpret_cast<uintptr_t>(sorted_token_ids) & 3u) ||
      (reinterpret_cast<uintptr_t>(num_tokens_per_lora) & 3u) ||
      (reinterpret_cast<uintptr_t>(lora_token_start_loc) & 3u))
    return LORA_ERR_ALIGN;
  if (workspace_bytes < grg::workspace_bytes_needed(max_num_tokens, max_loras))
    return LORA_ERR_WORKSPACE;
  return LORA_OK;
}
}  // namespace

namespace grg {
// Every argument check of lora_prepare_metadata, lora_shrink and lora_expand
// for one layer, without launching anything.
__attribute__((visibility("hidden"))) int check_layer_args(
    const int32_t* token_lora_mapping, const int32_t* num_tokens,
                     int64_t max_num_tokens, int64_t max_loras, const uint16_t* x,
                     int64_t x_row_stride, int64_t hidden, const uint16_t* const* lora_a,
                     const uint16_t* const* lora_b, const int64_t* slice_width, int num_slices,
                     int rank, float* u, uint16_t* y, int64_t y_row_stride,
                     const int32_t* sorted_token_ids, const int32_t* num_tokens_per_lora,
                     const int32_t* lora_token_start_loc, const void* workspace,
                     size_t workspace_bytes) {
  int rc = metadata_args(token_lora_mapping, num_tokens, max_num_tokens, max_loras,
                         sorted_token_ids, num_tokens_per_lora, lora_token_start_loc, workspace,
                         workspace_bytes);
  if (rc != LORA_OK) return rc;
  ShrinkArgs sa;
  rc = shrink_args(x, x_row_stride, hidden, lora_a, nullptr, num_slices, rank, 1.0f, nullptr, u,
                   sorted_token_ids, lora_token_start_loc, max_num_tokens, max_loras, workspace,
                   workspace_bytes, &sa);
  if (rc != LORA_OK) return rc;
  ExpandArgs ea;
  return expand_args(u, lora_b, nullptr, slice_width, num_slices, rank, y, y_row_stride,
                     sorted_token_ids, lora_token_start_loc, max_num_tokens, max_loras,
                     workspace, workspace_bytes, &ea);
}
}  // namespace grg

extern "C" {

int lora_prepare_metadata(const int32_t* token_lora_mapping, const int32_t* num_tokens,
                          int64_t max_num_tokens, int64_t max_loras, int32_t* sorted_token_ids,
                          int32_t* num_tokens_per_lora, int32_t* lora_token_start_loc,
                          void* workspace, size_t workspace_bytes, void* stream) {
  const int rc = metadata_args(token_lora_mapping, num_tokens, max_num_tokens, max_loras,
                               sorted_token_ids, num_tokens_per_lora, lora_token_start_loc,
                               workspace, workspace_bytes);
  if (rc != LORA_OK) return rc;
  return grg::launch_metadata(token_lora_mapping, num_tokens, static_cast<int>(max_num_tokens),
                              static_cast<int>(max_loras), sorted_token_ids, num_tokens_per_lora,
                              lora_token_start_loc, workspace, static_cast<cudaStream_t>(stream));
}

int lora_shrink(const uint16_t* x, int64_t x_row_stride, int64_t hidden,
                const uint16_t* const* lora_a, int num_slices, int rank, float scale,
                const float* lora_scales, float* u,
                const int32_t* sorted_token_ids, const int32_t* lora_token_start_loc,
                int64_t max_num_tokens, int64_t max_loras, const void* workspace,
                size_t workspace_bytes, void* stream) {
  grg::ShrinkArgs a;
  const int rc = shrink_args(x, x_row_stride, hidden, lora_a, nullptr, num_slices, rank, scale,
                             lora_scales, u, sorted_token_ids, lora_token_start_loc,
                             max_num_tokens, max_loras, workspace, workspace_bytes, &a);
  if (rc != LORA_OK) return rc;
  return grg::launch_shrink(a, static_cast<cudaStream_t>(stream));
}

int lora_expand(const float* u, const uint16_t* const* lora_b, const int64_t* slice_width,
                int num_slices, int rank, uint16_t* y, int64_t y_row_stride,
                const int32_t* sorted_token_ids, const int32_t* lora_token_start_loc,
                int64_t max_num_tokens, int64_t max_loras, const void* workspace,
                size_t workspace_bytes, void* stream) {
  grg::ExpandArgs a;
  const int rc = expand_args(u, lora_b, nullptr, slice_width, num_slices, rank, y, y_row_stride,
                             sorted_token_ids, lora_token_start_loc, max_num_tokens, max_loras,
                             workspace, workspace_bytes, &a);
  if (rc != LORA_OK) return rc;
  return grg::launch_expand(a, static_cast<cudaStream_t>(stream));
}

int lora_shrink_paged(const uint16_t* x, int64_t x_row_stride, int64_t hidden,
                      const uint64_t* const* lora_a_tables, int num_slices, int rank,
                      float scale, const float* lora_scales, float* u,
                      const int32_t* sorted_token_ids, const int32_t* lora_token_start_loc,
                      int64_t max_num_tokens, int64_t max_loras, const void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!lora_a_tables) return LORA_ERR_NULL;
  grg::ShrinkArgs a;
  const int rc = shrink_args(x, x_row_stride, hidden, nullptr, lora_a_tables, num_slices, rank,
                             scale, lora_scales, u, sorted_token_ids, lora_token_start_loc,
                             max_num_tokens, max_loras, workspace, workspace_bytes, &a);
  if (rc != LORA_OK) return rc;
  return grg::launch_shrink(a, static_cast<cudaStream_t>(stream));
}

int lora_expand_paged(const float* u, const uint64_t* const* lora_b_tables,
                      const int64_t* slice_width, int num_slices, int rank, uint16_t* y,
                      int64_t y_row_stride, const int32_t* sorted_token_ids,
                      const int32_t* lora_token_start_loc, int64_t max_num_tokens,
                      int64_t max_loras, const void* workspace, size_t workspace_bytes,
                      void* stream) {
  if (!lora_b_tables) return LORA_ERR_NULL;
  grg::ExpandArgs a;
  const int rc = expand_args(u, nullptr, lora_b_tables, slice_width, num_slices, rank, y,
                             y_row_stride, sorted_token_ids, lora_token_start_loc,
                             max_num_tokens, max_loras, workspace, workspace_bytes, &a);
  if (rc != LORA_OK) return rc;
  return grg::launch_expand(a, static_cast<cudaStream_t>(stream));
}

namespace {
// The split-K one-call path applies: a decode-sized shape, a workspace with
// room for the partial tiles, and a split of at least 2.
bool split_path_ok(const grg::ShrinkArgs& sa, size_t workspace_bytes) {
  const int64_t T = sa.max_num_tokens, L = sa.num_loras;
  return split_shape(T, sa.rank) &&
         workspace_bytes >= grg::workspace_bytes_needed(T, L) +
                                split_scratch_bytes(T, L, sa.num_slices, sa.rank) &&
         grg::shrink_split(sa, true) >= 2;
}

// One layer in one call, for validated arguments (stacked or paged weights):
// the fused kernel when the batch fits it, else the split-K pair when the
// workspace has room for the partial tiles, else the two kernels.
int shrink_expand(grg::ShrinkArgs& sa, grg::ExpandArgs& ea, int64_t hidden,
                  const void* workspace, size_t workspace_bytes, cudaStream_t s) {
  int rc = grg::launch_fused(sa, ea, s);
  if (rc < 0) return rc;
  if (rc == 1) return LORA_OK;
  // the expand directly follows the shrink, which never writes y
  ea.y_early = true;
  sa.expand_follows = true;
  // split-K: with the larger workspace, the shrink's CTAs write partial tiles
  // and the expand sums them in rank order (no cluster-wide steps)
  const int64_t T = sa.max_num_tokens, L = sa.num_loras;
  if (split_path_ok(sa, workspace_bytes)) {
    sa.partials = split_partials(workspace, T, L);
    rc = grg::launch_shrink(sa, s);
    if (rc != LORA_OK) return rc;
    ea.partials = sa.partials;
    ea.split = split_of(T, L, hidden, sa.num_slices, sa.rank);
    ea.scale = sa.scale;
    ea.lora_scales = sa.lora_scales;
    return grg::launch_expand(ea, s);
  }
  rc = grg::launch_shrink(sa, s);
  if (rc != LORA_OK) return rc;
  return grg::launch_expand(ea, s);
}
}  // namespace

int lora_shrink_expand(const uint16_t* x, int64_t x_row_stride, int64_t hidden,
                       const uint16_t* const* lora_a, const uint16_t* const* lora_b,
                       const int64_t* slice_width, int num_slices, int rank, float scale,
                       const float* lora_scales, float* u, uint16_t* y, int64_t y_row_stride,
                       const int32_t* sorted_token_ids, const int32_t* lora_token_start_loc,
                       int64_t max_num_tokens, int64_t max_loras, const void* workspace,
                       size_t workspace_bytes, void* stream) {
  grg::ShrinkArgs sa;
  grg::ExpandArgs ea;
  int rc = shrink_args(x, x_row_stride, hidden, lora_a, nullptr, num_slices, rank, scale,
                       lora_scales, u, sorted_token_ids, lora_token_start_loc, max_num_tokens,
                       max_loras, workspace, workspace_bytes, &sa);
  if (rc != LORA_OK) return rc;
  rc = expand_args(u, lora_b, nullptr, slice_width, num_slices, rank, y, y_row_stride,
                   sorted_token_ids, lora_token_start_loc, max_num_tokens, max_loras, workspace,
                   workspace_bytes, &ea);
  if (rc != LORA_OK) return rc;
  return shrink_expand(sa, ea, hidden, workspace, workspace_bytes,
                       static_cast<cudaStream_t>(stream));
}

int lora_shrink_expand_paged(const uint16_t* x, int64_t x_row_stride, int64_t hidden,
                             const uint64_t* const* lora_a_tables,
                             const uint64_t* const* lora_b_tables, const int64_t* slice_width,
                             int num_slices, int rank, float scale, const float* lora_scales,
                             float* u, uint16_t* y, int64_t y_row_stride,
                             const int32_t* sorted_token_ids, const int32_t* lora_token_start_loc,
                             int64_t max_num_tokens, int64_t max_loras, const void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (!lora_a_tables || !lora_b_tables) return LORA_ERR_NULL;
  grg::ShrinkArgs sa;
  grg::ExpandArgs ea;
  int rc = shrink_args(x, x_row_stride, hidden, nullptr, lora_a_tables, num_slices, rank, scale,
                       lora_scales, u, sorted_token_ids, lora_token_start_loc, max_num_tokens,
                       max_loras, workspace, workspace_bytes, &sa);
  if (rc != LORA_OK) return rc;
  rc = expand_args(u, nullptr, lora_b_tables, slice_width, num_slices, rank, y, y_row_stride,
                   sorted_token_ids, lora_token_start_loc, max_num_tokens, max_loras, workspace,
                   workspace_bytes, &ea);
  if (rc != LORA_OK) return rc;
  return shrink_expand(sa, ea, hidden, workspace, workspace_bytes,
                       static_cast<cudaStream_t>(stream));
}

int lora_shrink_f16(const uint16_t* x, int64_t x_row_stride, int64_t hidden,
                    const uint16_t* const* lora_a, int num_slices, int rank, float scale,
                    const float* lora_scales, float* u, const int32_t* sorted_token_ids,
                    const int32_t* lora_token_start_loc, int64_t max_num_tokens,
                    int64_t max_loras, const void* workspace, size_t workspace_bytes,
                    void* stream) {
  grg::ShrinkArgs a;
  const int rc = shrink_args(x, x_row_stride, hidden, lora_a, nullptr, num_slices, rank, scale,
                             lora_scales, u, sorted_token_ids, lora_token_start_loc,
                             max_num_tokens, max_loras, workspace, workspace_bytes, &a);
  if (rc != LORA_OK) return rc;
  a.f16 = true;
  return grg::launch_shrink(a, static_cast<cudaStream_t>(stream));
}

int lora_expand_f16(const float* u, const uint16_t* const* lora_b, const int64_t* slice_width,
                    int num_slices, int rank, uint16_t* y, int64_t y_row_stride,
                    const int32_t* sorted_token_ids, const int32_t* lora_token_start_loc,
                    int64_t max_num_tokens, int64_t max_loras, const void* workspace,
                    size_t workspace_bytes, void* stream) {
  grg::ExpandArgs a;
  const int rc = expand_args(u, lora_b, nullptr, slice_width, num_slices, rank, y, y_row_stride,
                             sorted_token_ids, lora_token_start_loc, max_num_tokens, max_loras,
                             workspace, workspace_bytes, &a);
  if (rc != LORA_OK) return rc;
  a.f16 = true;
  return grg::launch_expand(a, static_cast<cudaStream_t>(stream));
}

int lora_shrink_expand_f16(const uint16_t* x, int64_t x_row_stride, int64_t hidden,
                           const uint16_t* const* lora_a, const uint16_t* const* lora_b,
                           const int64_t* slice_width, int num_slices, int rank, float scale,
                           const float* lora_scales, float* u, uint16_t* y, int64_t y_row_stride,
                           const int32_t* sorted_token_ids, const int32_t* lora_token_start_loc,
                           int64_t max_num_tokens, int64_t max_loras, const void* workspace,
                           size_t workspace_bytes, void* stream) {
  grg::ShrinkArgs sa;
  grg::ExpandArgs ea;
  int rc = shrink_args(x, x_row_stride, hidden, lora_a, nullptr, num_slices, rank, scale,
                       lora_scales, u, sorted_token_ids, lora_token_start_loc, max_num_tokens,
                       max_loras, workspace, workspace_bytes, &sa);
  if (rc != LORA_OK) return rc;
  rc = expand_args(u, lora_b, nullptr, slice_width, num_slices, rank, y, y_row_stride,
                   sorted_token_ids, lora_token_start_loc, max_num_tokens, max_loras, workspace,
                   workspace_bytes, &ea);
  if (rc != LORA_OK) return rc;
  sa.f16 = true;
  ea.f16 = true;
  return shrink_expand(sa, ea, hidden, workspace, workspace_bytes,
                       static_cast<cudaStream_t>(stream));
}

int lora_shrink_expand_kernels(int64_t max_num_tokens, int64_t max_loras, int64_t hidden,
                               const int64_t* slice_width, int num_slices, int rank) {
  if (!slice_width) return LORA_ERR_NULL;
  if (num_slices < 1 || num_slices > LORA_MAX_SLICES || !sizes_ok(max_num_tokens, max_loras) ||
      !rank_ok(rank) || hidden < 8 || hidden > kMaxHidden || (hidden % 8) != 0)
    return LORA_ERR_SHAPE;
  int w[3] = {0, 0, 0};
  for (int s = 0; s < num_slices; ++s) {
    if (slice_width[s] < 8 || slice_width[s] > kMaxWidth || (slice_width[s] % 8) != 0)
      return LORA_ERR_SHAPE;
    w[s] = static_cast<int>(slice_width[s]);
  }
  return grg::fused_fits(static_cast<int>(max_num_tokens), static_cast<int>(max_loras),
                         static_cast<int>(hidden), w, num_slices, rank)
             ? 1
             : 2;
}

int lora_shrink_expand_path(int64_t max_num_tokens, int64_t max_loras, int64_t hidden,
                            const int64_t* slice_width, int num_slices, int rank,
                            size_t workspace_bytes, int fp16, int paged) {
  if (!slice_width) return LORA_ERR_NULL;
  if (num_slices < 1 || num_slices > LORA_MAX_SLICES || !sizes_ok(max_num_tokens, max_loras) ||
      !rank_ok(rank) || hidden < 8 || hidden > kMaxHidden || (hidden % 8) != 0)
    return LORA_ERR_SHAPE;
  if ((fp16 && paged) ||
      workspace_bytes < grg::workspace_bytes_needed(max_num_tokens, max_loras))
    return LORA_ERR_SHAPE;
  int w[3] = {0, 0, 0};
  for (int s = 0; s < num_slices; ++s) {
    if (slice_width[s] < 8 || slice_width[s] > kMaxWidth || (slice_width[s] % 8) != 0)
      return LORA_ERR_SHAPE;
    w[s] = static_cast<int>(slice_width[s]);
  }
  const int T = static_cast<int>(max_num_tokens), L = static_cast<int>(max_loras);
  const int H = static_cast<int>(hidden);
  if (!paged && grg::fused_fits(T, L, H, w, num_slices, rank)) return LORA_PATH_FUSED;
  grg::ShrinkArgs sa;
  sa.hidden = H;
  sa.num_slices = num_slices;
  sa.rank = rank;
  sa.max_num_tokens = T;
  sa.num_loras = L;
  if (split_path_ok(sa, workspace_bytes)) return LORA_PATH_SPLIT_PAIR;
  return LORA_PATH_PAIR;
}

int lora_read_status(void* workspace, uint32_t* status, void* stream) {
  if (!workspace || !status) return LORA_ERR_NULL;
  if (!aligned16(workspace)) return LORA_ERR_ALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t host = 0;
  if (cudaMemcpyAsync(&host, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return LORA_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return LORA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LORA_ERR_CUDA;
  *status = host;
  return LORA_OK;
}

int lora_testing_inject_timeout(int on) { return grg::set_wait_fault(on); }

const char* lora_error_string(int code) {
  switch (code) {
    case LORA_OK: return "ok";
    case LORA_ERR_NULL: return "a required pointer is NULL";
    case LORA_ERR_ALIGN: return "a pointer or row stride is not 16-byte aligned";
    case LORA_ERR_SHAPE: return "a size is outside the supported set";
    case LORA_ERR_WORKSPACE: return "workspace too small (see lora_workspace_size)";
    case LORA_ERR_LAUNCH: return "CUDA kernel launch failed";
    case LORA_ERR_CUDA: return "a CUDA runtime call failed";
    default: return "unknown error code";
  }
}

}  // extern "C"
#pragma GCC visibility pop
