// Host-side launch helpers: per-device caches and the cudaLaunchKernelEx call.
#include "launch.h"

#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>
#include <unordered_map>
#include <utility>

namespace grg {

namespace {
std::atomic<int> g_wait_fault{0};
std::mutex g_mu;
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};

struct Key {
  int dev;
  const void* fn;
  long long a;
  long long b;
  bool operator==(const Key& o) const { return dev == o.dev && fn == o.fn && a == o.a && b == o.b; }
};
struct KeyHash {
  size_t operator()(const Key& k) const {
    size_t h = std::hash<const void*>()(k.fn);
    h ^= std::hash<long long>()(k.a * 1000003LL + k.b) + 0x9e3779b97f4a7c15ULL + (h << 6) + (h >> 2);
    return h ^ static_cast<size_t>(k.dev);
  }
};
std::unordered_map<Key, int, KeyHash> g_smem_set;   // largest smem limit set
std::unordered_map<Key, int, KeyHash> g_occupancy;  // blocks per SM

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}
}  // namespace

int set_wait_fault(int on) { return g_wait_fault.exchange(on ? 1 : 0); }
int wait_fault() { return g_wait_fault.load(); }

int device_sm_count() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return -1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

int ensure_smem_attr(const void* func, size_t smem_bytes) {
  const int dev = current_device();
  if (dev < 0) return -1;
  std::lock_guard<std::mutex> lk(g_mu);
  Key k{dev, func, 0, 0};
  auto it = g_smem_set.find(k);
  if (it != g_smem_set.end() && it->second >= static_cast<long long>(smem_bytes)) return 0;
  if (smem_bytes > 48 * 1024) {
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_bytes)) != cudaSuccess)
      return -1;
  }
  g_smem_set[k] = static_cast<int>(smem_bytes);
  return 0;
}

int occupancy_blocks(const void* func, int threads, size_t smem_bytes) {
  const int dev = current_device();
  if (dev < 0) return 1;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_occupancy.find(Key{dev, func, threads, static_cast<long long>(smem_bytes)});
    if (it != g_occupancy.end()) return it->second;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, smem_bytes) != cudaSuccess)
    n = 1;
  std::lock_guard<std::mutex> lk(g_mu);
  g_occupancy[Key{dev, func, threads, static_cast<long long>(smem_bytes)}] = n;
  return n;
}

int resident_blocks(const void* func, int threads, size_t smem_bytes) {
  const int dev = current_device();
  if (dev < 0) return 1;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, func) != cudaSuccess || fa.numRegs <= 0) return 1;
  int regs_sm = 0, smem_sm = 0, reserved = 0, threads_sm = 0, blocks_sm = 0;
  if (cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&blocks_sm, cudaDevAttrMaxBlocksPerMultiprocessor, dev) != cudaSuccess)
    return 1;
  // registers are allocated per warp in units of 256
  const long long warp_regs = (static_cast<long long>(fa.numRegs) * 32 + 255) / 256 * 256;
  const long long warps = (threads + 31) / 32;
  const long long by_regs = regs_sm / (warp_regs * warps);
  const long long by_smem =
      smem_sm / (static_cast<long long>(smem_bytes) + fa.sharedSizeBytes + reserved);
  const long long by_threads = threads_sm / threads;
  long long n = by_regs;
  if (by_smem < n) n = by_smem;
  if (by_threads < n) n = by_threads;
  if (blocks_sm < n) n = blocks_sm;
  return n < 1 ? 1 : static_cast<int>(n);
}

int launch_raw(const void* func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
               int cluster, void* params) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cluster > 0) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = static_cast<unsigned>(cluster);
    attrs[na].val.clusterDim.y = 1;
    attrs[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  void* args[1] = {params};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, func, args);
  if (e != cudaSuccess) return -5;
  return 0;
}

int make_weight_tmap(CUtensorMap* map, const void* base, long long cols, long long rows,
                     int box_rows) {
  return make_tmap_2d(map, base, cols, rows, cols * 2, box_rows);
}

int make_tmap_2d(CUtensorMap* map, const void* base, long long cols, long long rows,
                 long long row_stride_bytes, int box_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!encode) return -6;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_stride_bytes)};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -6;
}

}  // namespace grg
