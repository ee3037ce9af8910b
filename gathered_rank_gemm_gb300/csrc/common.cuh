// Shared device helpers and the workspace layout for the LoRA kernels (sm_103a).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
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

// Same, asynchronously (cp.async, part of the caller's next commit group).
template <int ROWS>
__device__ __forceinline__ void load_record_async(const int32_t* list, int item, int32_t* srec) {
  const int32_t* src = list + static_cast<long long>(item) * record_ints(ROWS);
  const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(srec));
  for (int i = threadIdx.x; i < record_ints(ROWS) / 4; i += blockDim.x)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;\n" ::"r"(dst + 16 * i), "l"(src + 4 * i)
                 : "memory");
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
// An L2 policy that marks the lines a load brings in as the first to evict
// (for data this kernel reads once and nothing after it reads again).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
// Waits until at most n of this thread's most recent cp.async groups are pending.
__device__ __forceinline__ void cp_async_wait_dyn(int n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    case 7: cp_async_wait<7>(); break;
    default: cp_async_wait<8>(); break;
  }
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

// D += A * B, m16n8k16, fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Barrier among the first `threads` threads of the block (named barrier `id`).
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
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

// ---------------------------------------------------------------- TMA bulk copies + mbarriers
// Spin limit for every mbarrier wait: a wait that has not completed after this
// many nanoseconds of %globaltimer gives up and reports LORA_STATUS_TIMEOUT.
constexpr unsigned long long kWaitLimitNs = 200ull * 1000ull * 1000ull;
constexpr uint32_t kStatusTimeout = 0x4u;
constexpr uint32_t kStatusBadWeight = 0x8u;  // a paged weight address was not 16-byte aligned

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
// Makes barrier initialisation visible to the async proxy (and the cluster).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_count(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(count)
               : "memory");
}
// Arrives on the mbarrier once all of this thread's earlier cp.async copies
// have landed (the arrival is part of the barrier's expected count).
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}
// Bounded waiting by a CTA that gives up as a whole.  The first of its waits
// that runs out sets a flag in the CTA's shared memory; every later wait then
// returns false at once, the kernel issues no further copy and stores no
// output, and before it exits it waits (bounded again, mbar_drain) for the
// bulk copies it had already issued, so that none is still writing its shared
// memory when it leaves.  Every block-wide or named barrier is still reached
// by every thread: giving up changes no control flow around them.
struct CtaAbort {
  volatile int* flag;           // in shared memory, 0 until a wait runs out
  unsigned long long limit_ns;  // kWaitLimitNs, or 1 ms under the test hook
  __device__ __forceinline__ bool raised() const { return *flag != 0; }
  // Waits for the phase with the given parity; false if the time limit
  // passed (which raises the flag) or the flag was already up.
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
    if (*flag != 0) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
      if (*flag != 0) return false;
      if (global_ns() - t0 > limit_ns) {
        *flag = 1;
        return false;
      }
    }
    return true;
  }
};
// After giving up: waits, with the limit, for a copy issued on the barrier's
// phase of the given parity to land.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity,
                                           unsigned long long limit_ns) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit_ns) return;
}
// The test hook's wait limit.
constexpr unsigned long long kTestWaitLimitNs = 1000ull * 1000ull;
// global -> shared bulk copy (16-byte aligned, size a multiple of 16) that
// completes `bytes` transactions on the mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// 2-D tiled TMA load of box (x, y) of a tensor map into shared memory,
// completing the box's bytes on the mbarrier.  x must be a multiple of 8
// bf16 elements (16 bytes); out-of-range elements are filled with zeros.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// tma_load_2d with an L2 cache policy (createpolicy) for the loaded lines.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int x,
                                                 int y, uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
      : "memory");
}
// Prefetch of box (x, y) of a tensor map into L2 (no shared memory, no
// barrier); the same alignment rule for x as tma_load_2d.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];\n" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Offset inside a 1024-byte-aligned [rows][128 B] box written by TMA with the
// 128-byte swizzle: 16-byte chunk ch of row r lands at chunk ch ^ (r % 8).
__device__ __forceinline__ uint32_t swz128(int row, int ch) {
  return static_cast<uint32_t>(row * 128 + ((ch ^ (row & 7)) << 4));
}

// shared -> global bulk copy, tracked by the thread's bulk async-groups.
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
// The thread's bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}
// The thread's bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// Bulk prefetch of [src, src + bytes) into L2 (16-byte aligned, multiple of 16).
// L2 is the coherence point of the GPU, so prefetching data that an earlier
// kernel may still be writing is harmless: later reads through L2 see the
// final values.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
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

// fp16 pair <-> float pair, and the fp16 high / residual split.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack_f16x2(uint32_t w) {
  __half2 v = *reinterpret_cast<__half2*>(&w);
  return __half22float2(v);
}
__device__ __forceinline__ void split_f16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  __half2 h = __floats2half2_rn(a, b);
  float2 hf = __half22float2(h);
  __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}

// The 16-bit element type as a template switch: F16 = fp16, else bf16.  The
// weights and activations move as raw 16-bit words; only the MMA and the
// fp32 conversions of y and u depend on the type.
template <bool F16>
__device__ __forceinline__ void mma_t(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                      uint32_t b1) {
  if constexpr (F16) mma_f16(d, a, b0, b1); else mma_bf16(d, a, b0, b1);
}
template <bool F16>
__device__ __forceinline__ uint32_t pack_t(float lo, float hi) {
  if constexpr (F16) return pack_f16x2(lo, hi); else return pack_bf16x2(lo, hi);
}
template <bool F16>
__device__ __forceinline__ float2 unpack_t(uint32_t w) {
  if constexpr (F16) return unpack_f16x2(w); else return unpack_bf16x2(w);
}
template <bool F16>
__device__ __forceinline__ void split_t(float a, float b, uint32_t& hi, uint32_t& lo) {
  if constexpr (F16) split_f16x2(a, b, hi, lo); else split_bf16x2(a, b, hi, lo);
}

// ---------------------------------------------------------------- tcgen05
// tcgen05 shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version of the tcgen05 instructions
  d |= 2ull << 61;  // swizzle: 128 bytes
  return d;
}
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace grg
