// Shared device helpers and the workspace layout for the LoRA kernels (sm_103a).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace grg {

// ---------------------------------------------------------------- workspace
// [0]   uint32 status word (LORA_STATUS_* bits, OR-ed by the metadata kernel)
// [4]   int32  n after clamping
// [16]  int32  num_tiles[kNumTileSizes]: records in each work list
// [64]  work lists, one per tile height rows = 16 << i.  Record j of list i is
//       rows + 4 int32: {lora, count, pos, 0, token[0 .. rows-1]}: `count`
//       (1..rows) tokens of adapter `lora`, taken from sorted_token_ids[pos..]
//       and copied inline so that a CTA gets its whole tile with one load.
constexpr int kNumTileSizes = 4;
constexpr int kWsHeaderBytes = 64;
constexpr int kRecordHeaderInts = 4;

__host__ __device__ constexpr int tile_rows_of(int i) { return 16 << i; }
__host__ __device__ inline int tile_index_of(int rows) {
  return rows == 16 ? 0 : rows == 32 ? 1 : rows == 64 ? 2 : 3;
}
__host__ __device__ constexpr int record_ints(int rows) { return rows + kRecordHeaderInts; }
__host__ __device__ inline int64_t tile_list_capacity(int64_t max_num_tokens, int64_t max_loras,
                                                      int i) {
  const int64_t rows = tile_rows_of(i);
  return (max_num_tokens + rows - 1) / rows + max_loras;
}
__host__ __device__ inline int64_t tile_list_offset(int64_t max_num_tokens, int64_t max_loras,
                                                    int i) {
  int64_t off = kWsHeaderBytes;
  for (int j = 0; j < i; ++j)
    off += 4LL * record_ints(tile_rows_of(j)) * tile_list_capacity(max_num_tokens, max_loras, j);
  return off;
}
inline size_t workspace_bytes_needed(int64_t max_num_tokens, int64_t max_loras) {
  int64_t end = tile_list_offset(max_num_tokens, max_loras, kNumTileSizes);
  return static_cast<size_t>((end + 255) / 256 * 256);
}

struct WsView {
  uint32_t* status;
  int32_t* n;
  int32_t* num_tiles;
  int32_t* lists[kNumTileSizes];
};
inline WsView ws_view(void* ws, int64_t max_num_tokens, int64_t max_loras) {
  char* b = static_cast<char*>(ws);
  WsView v;
  v.status = reinterpret_cast<uint32_t*>(b);
  v.n = reinterpret_cast<int32_t*>(b + 4);
  v.num_tiles = reinterpret_cast<int32_t*>(b + 16);
  for (int i = 0; i < kNumTileSizes; ++i)
    v.lists[i] = reinterpret_cast<int32_t*>(b + tile_list_offset(max_num_tokens, max_loras, i));
  return v;
}

// Copies tile record `item` of a list (rows + 4 ints, 16-byte aligned) into
// shared memory with 16-byte loads; the caller synchronises afterwards.
template <int ROWS>
__device__ __forceinline__ void load_record(const int32_t* list, int item, int32_t* srec) {
  const int4* src = reinterpret_cast<const int4*>(list + static_cast<long long>(item) * record_ints(ROWS));
  for (int i = threadIdx.x; i < record_ints(ROWS) / 4; i += blockDim.x)
    reinterpret_cast<int4*>(srec)[i] = src[i];
}

// Decoded tile: adapter, token count and the token of row r (-1 past count).
// Fields are range-checked, so a workspace that was never prepared cannot
// send an access out of bounds.
struct TileView {
  int lora;
  int count;
  __device__ __forceinline__ static TileView of(const int32_t* srec, int rows, int num_loras) {
    TileView t;
    const int l = srec[0], c = srec[1];
    const bool ok = l >= 0 && l < num_loras && c > 0 && c <= rows;
    t.lora = ok ? l : 0;
    t.count = ok ? c : 0;
    return t;
  }
};
__device__ __forceinline__ int record_token(const int32_t* srec, int r, int count,
                                            int max_num_tokens) {
  const int t = r < count ? srec[kRecordHeaderInts + r] : -1;
  return (t >= 0 && t < max_num_tokens) ? t : -1;
}

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared copy; when !pred nothing is read and zeros are written.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, bool pred) {
  const int bytes = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D += A * B, m16n8k16, bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Thread-block cluster helpers.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n"
      "barrier.cluster.wait.acquire.aligned;\n" ::
          : "memory");
}
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Programmatic dependent launch: wait for the preceding grid's memory, and let
// the next grid on the stream start its launch early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// bf16 pair <-> float pair.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w);
  return __bfloat1622float2(v);
}

// Split two floats into bf16 high parts and bf16 residuals: v ~= hi + lo with
// about 16 significant bits kept.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}

}  // namespace grg
