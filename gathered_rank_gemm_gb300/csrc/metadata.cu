// Device metadata: stable grouping of the batch's tokens by LoRA id.
//
// "[V1] LoRA - Add triton kernels for V1" (vLLM PR 13096), "Why do we need a
// new set of kernels": V1 batches are not sorted by LoRA id, so the kernels
// need, on the device, which tokens belong to which adapter.  "[Kernel] LoRA -
// Enable CUDAGraphs for V1" (vLLM PR 14626): the map is a static buffer of
// max_num_tokens entries and the pad rows past n hold garbage.
//
// A cluster of C CTAs of 16 warps (C = 1 up to 1024 tokens, up to 8 beyond:
// a size known at capture time) runs a stable counting sort over bins 0..L
// (bin L = no adapter):
//   1. warp w of CTA c takes the contiguous token range [g*seg, (g+1)*seg),
//      g = 16 c + w, and counts its tokens per bin (lanes with the same bin
//      are grouped with __match_any_sync, the group leader adds the size);
//   2. per bin, an exclusive scan over the CTA's 16 warp counts gives each
//      warp's offset inside the CTA's share of the bin; the CTAs' totals are
//      exchanged through distributed shared memory, giving every CTA the bin
//      totals and its own offset (the sum over lower-ranked CTAs); one block
//      scan over the bin totals (and, per tile height, the tiles per adapter)
//      gives lora_token_start_loc and the first tile of every adapter;
//   3. each warp walks its range again in order; a token's slot is
//      start[bin] + CTA offset + warp offset + (earlier lanes of its group).
// Ranges are in token order (CTA, then warp, then lane), so equal ids keep
// ascending token order (stable).  The grid depends only on max_num_tokens,
// so the launch is graph-safe.  The kernel also writes, for each tile height
// in {16, 32, 64, 128}, the list of tile records (adapter, count and the
// tile's token ids inline) that the shrink and expand kernels walk with a
// fixed grid.
#include "common.cuh"
#include "launch.h"

namespace grg {

constexpr int kMetaThreads = 512;
constexpr int kMetaWarps = kMetaThreads / 32;
constexpr int kMetaChunk = 16;  // 32-token steps per warp whose bins stay in registers
constexpr int kScanArrays = 1 + kNumTileSizes;  // bin starts + tile offsets per tile height

// Exclusive scans of kScanArrays arrays at once: in[a][0..count) ->
// out[a][0..count], out[a][count] = total of array a.  `in` and `out` are
// strided by in_stride / out_stride ints per array and must not overlap.
// Called by every thread of the block.
__device__ void block_exclusive_scan_multi(const int32_t* in, int in_stride, int32_t* out,
                                           int out_stride, int count, int32_t* warp_sums) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nwarps = nthreads >> 5;
  const int per = (count + nthreads - 1) / nthreads;
  const int begin = min(tid * per, count), end = min(begin + per, count);
  int local[kScanArrays], incl[kScanArrays];
#pragma unroll
  for (int a = 0; a < kScanArrays; ++a) {
    local[a] = 0;
    for (int i = begin; i < end; ++i) local[a] += in[a * in_stride + i];
    incl[a] = local[a];
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int a = 0; a < kScanArrays; ++a) {
      const int y = __shfl_up_sync(0xffffffffu, incl[a], o);
      if (lane >= o) incl[a] += y;
    }
  }
  if (lane == 31)
#pragma unroll
    for (int a = 0; a < kScanArrays; ++a) warp_sums[a * 32 + warp] = incl[a];
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int a = 0; a < kScanArrays; ++a) {
      const int w = lane < nwarps ? warp_sums[a * 32 + lane] : 0;
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
      }
      if (lane < nwarps) warp_sums[a * 32 + lane] = wi - w;
    }
  }
  __syncthreads();
#pragma unroll
  for (int a = 0; a < kScanArrays; ++a) {
    int run = warp_sums[a * 32 + warp] + incl[a] - local[a];
    for (int i = begin; i < end; ++i) {
      out[a * out_stride + i] = run;
      run += in[a * in_stride + i];
    }
    if (tid == nthreads - 1) out[a * out_stride + count] = run;
  }
  __syncthreads();
}

struct MetaParams {
  const int32_t* mapping;
  const int32_t* num_tokens;
  int max_num_tokens;
  int num_loras;
  int32_t* sorted_ids;
  int32_t* counts;
  int32_t* starts;
  WsView ws;
};

__global__ void __launch_bounds__(kMetaThreads, 1) lora_metadata_kernel(MetaParams p) {
  extern __shared__ int32_t sm[];
  __shared__ int32_t warp_sums[32 * kScanArrays];
  __shared__ int s_n;
  __shared__ uint32_t s_status;

  const int L = p.num_loras;
  const int nbins = L + 1;
  int32_t* hist = sm;                          // [kMetaWarps][nbins], then warp offsets
  int32_t* total = hist + kMetaWarps * nbins;  // [nbins]
  int32_t* start = total + nbins;              // [nbins + 1]
  int32_t* cnts = start + nbins + 1;           // [kScanArrays][nbins]: totals, tiles per height
  int32_t* offs = cnts + kScanArrays * nbins;   // [kScanArrays][nbins + 1]: starts, tile offsets
  int32_t* ctot = offs + kScanArrays * (nbins + 1);  // [nbins]: this CTA's tokens per bin
  int32_t* coff = ctot + nbins;                      // [nbins]: lower-ranked CTAs' tokens per bin

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t cl_size;
  asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(cl_size));
  const int C = static_cast<int>(cl_size);
  const int crank = static_cast<int>(cluster_ctarank());
  const int gwarp = crank * kMetaWarps + warp;
  const int cthreads = C * kMetaThreads;  // threads of the whole cluster
  const int ctid = crank * kMetaThreads + tid;
  // Dependents are released only at the very end, after a fence: kernels of
  // this library read the work list before their own dependency wait.
  pdl_wait();

  if (tid == 0) {
    int n = *p.num_tokens;
    uint32_t st = 0;
    if (n < 0) { n = 0; st |= 2u; }
    if (n > p.max_num_tokens) { n = p.max_num_tokens; st |= 2u; }
    s_n = n;
    s_status = st;
  }
  for (int i = tid; i < kMetaWarps * nbins; i += kMetaThreads) hist[i] = 0;
  __syncthreads();
  const int n = s_n;

  const int seg = ((n + C * kMetaWarps - 1) / (C * kMetaWarps) + 31) & ~31;
  const int lo = min(gwarp * seg, n), hi = min(lo + seg, n);
  int32_t* my_hist = hist + warp * nbins;

  // Bins of this lane's tokens for one chunk of kMetaChunk 32-token steps:
  // all loads are issued before any is used (one memory round trip).
  int bins[kMetaChunk];
  bool bad = false;
  auto load_chunk = [&](int base0) {
    int ids[kMetaChunk];
#pragma unroll
    for (int j = 0; j < kMetaChunk; ++j) {
      const int t = base0 + 32 * j + lane;
      ids[j] = t < hi ? p.mapping[t] : -1;
    }
#pragma unroll
    for (int j = 0; j < kMetaChunk; ++j) {
      const int t = base0 + 32 * j + lane;
      int bin = nbins;  // never a real bin: marks idle lanes
      if (t < hi) {
        const int id = ids[j];
        if (id >= 0 && id < L) {
          bin = id;
        } else {
          bin = L;
          bad |= (id != -1);
        }
      }
      bins[j] = bin;
    }
  };
  const int chunk_tokens = 32 * kMetaChunk;
  const bool one_chunk = hi - lo <= chunk_tokens;

  // pass 1: per-warp histogram (lanes of a bin grouped with __match_any_sync)
  for (int base0 = lo; base0 < hi; base0 += chunk_tokens) {
    load_chunk(base0);
#pragma unroll
    for (int j = 0; j < kMetaChunk; ++j) {
      if (base0 + 32 * j >= hi) break;
      const int bin = bins[j];
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (bin < nbins && lane == __ffs(peers) - 1) my_hist[bin] += __popc(peers);
      __syncwarp();
    }
  }
  if (bad) atomicOr(&s_status, 1u);
  __syncthreads();

  // pass 2: warp offsets inside the CTA's share of each bin, the CTA's bin
  // counts; the cluster's counts give the bin totals and this CTA's offsets;
  // then one scan gives the bin starts and, per tile height, each adapter's
  // first tile
  for (int b = tid; b < nbins; b += kMetaThreads) {
    int run = 0;
    for (int w = 0; w < kMetaWarps; ++w) {
      const int c = hist[w * nbins + b];
      hist[w * nbins + b] = run;
      run += c;
    }
    ctot[b] = run;
  }
  if (C > 1) {
    cluster_sync_all();  // every CTA's counts are in its shared memory
    const uint32_t ctot_addr = smem_u32(ctot);
    for (int b = tid; b < nbins; b += kMetaThreads) {
      int below = 0, all = 0;
      for (int c = 0; c < C; ++c) {
        int v;
        asm volatile("ld.shared::cluster.s32 %0, [%1];\n"
                     : "=r"(v)
                     : "r"(mapa_shared(ctot_addr + 4u * b, static_cast<uint32_t>(c)))
                     : "memory");
        if (c < crank) below += v;
        all += v;
      }
      coff[b] = below;
      total[b] = all;
    }
  } else {
    __syncthreads();
    for (int b = tid; b < nbins; b += kMetaThreads) {
      coff[b] = 0;
      total[b] = ctot[b];
    }
  }
  __syncthreads();
  for (int b = tid; b < nbins; b += kMetaThreads) {
    const int run = total[b];
    cnts[b] = run;
#pragma unroll
    for (int k = 0; k < kNumTileSizes; ++k) {
      const int rows = tile_rows_of(k);
      cnts[(1 + k) * nbins + b] = b < L ? (run + rows - 1) / rows : 0;
    }
  }
  __syncthreads();
  block_exclusive_scan_multi(cnts, nbins, offs, nbins + 1, nbins, warp_sums);
  for (int b = tid; b <= nbins; b += kMetaThreads) start[b] = offs[b];
  __syncthreads();
  const int32_t* toff = offs + (nbins + 1);  // [k][L + 1]: tile offsets, stride nbins + 1

  // pass 3: stable scatter into sorted_token_ids and into the tile records
  for (int base0 = lo; base0 < hi; base0 += chunk_tokens) {
    if (!one_chunk) load_chunk(base0);  // a single chunk still holds its bins
#pragma unroll
    for (int j = 0; j < kMetaChunk; ++j) {
      if (base0 + 32 * j >= hi) break;
      const int t = base0 + 32 * j + lane;
      const int bin = bins[j];
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (bin < nbins) {
        const int rel = coff[bin] + my_hist[bin] + __popc(peers & ((1u << lane) - 1u));
        p.sorted_ids[start[bin] + rel] = t;
        if (bin < L) {
#pragma unroll
          for (int k = 0; k < kNumTileSizes; ++k) {
            const int tile = toff[k * (nbins + 1) + bin] + (rel >> (4 + k));
            p.ws.lists[k][static_cast<long long>(tile) * record_ints(tile_rows_of(k)) +
                          kRecordHeaderInts + (rel & (tile_rows_of(k) - 1))] = t;
          }
        }
      }
      __syncwarp();
      if (bin < nbins && lane == __ffs(peers) - 1) my_hist[bin] += __popc(peers);
      __syncwarp();
    }
  }
  for (int t = n + ctid; t < p.max_num_tokens; t += cthreads) p.sorted_ids[t] = -1;
  if (crank == 0) {
    for (int b = tid; b < nbins; b += kMetaThreads) p.counts[b] = total[b];
    for (int b = tid; b <= nbins; b += kMetaThreads) p.starts[b] = start[b];
  }

  // record headers
#pragma unroll
  for (int k = 0; k < kNumTileSizes; ++k) {
    const int rows = tile_rows_of(k);
    const int32_t* off = toff + k * (nbins + 1);
    const int count = off[L];
    int32_t* list = p.ws.lists[k];
    for (int i = ctid; i < count; i += cthreads) {
      // largest l with off[l] <= i (adapters with no tile share the next offset)
      int a = 0, b = L - 1;
      while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (off[mid] <= i) a = mid; else b = mid - 1;
      }
      const int j = i - off[a];
      int4 h = make_int4(a, min(rows, total[a] - j * rows), start[a] + j * rows, 0);
      *reinterpret_cast<int4*>(list + static_cast<long long>(i) * record_ints(rows)) = h;
    }
    if (ctid == 0) p.ws.num_tiles[k] = count;
  }
  if (tid == 0) {
    if (crank == 0) *p.ws.n = n;
    if (s_status) atomicOr(p.ws.status, s_status);
  }
  __threadfence();
  // no CTA exits while another may still read its counts
  if (C > 1)
    cluster_sync_all();
  else
    __syncthreads();
  pdl_launch_dependents();
}

// Short batches (max_num_tokens <= 1024, at most 128 adapters): one CTA,
// one token per thread, and fewer dependent steps than the cluster kernel.
// n and every thread's mapping entry load in one round trip (the entries
// past n are loaded but never used); per-warp bin counts
// (__match_any_sync); per bin, one warp scans the warps' counts into the
// warps' offsets and the bin total; one warp scans the bins for the bin starts
// and, per tile height, each adapter's first tile; then every thread writes
// its token's slots.  Same outputs, bit for bit, as the cluster kernel.
constexpr int kSmallMaxTokens = 1024;
constexpr int kSmallMaxLoras = 128;
constexpr int kSmallBins = kSmallMaxLoras + 1;

__global__ void __launch_bounds__(kSmallMaxTokens, 1) lora_metadata_small_kernel(MetaParams p) {
  __shared__ int32_t cnt[32][kSmallBins];  // per warp and bin: count, then offset in the bin
  __shared__ int32_t total[kSmallBins];
  __shared__ int32_t start[kSmallBins + 1];
  __shared__ int32_t toff[kNumTileSizes][kSmallBins + 1];  // first tile of each adapter

  const int L = p.num_loras, nbins = L + 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = static_cast<int>(blockDim.x) >> 5;
  pdl_wait();

  const int t = tid;
  int n = *p.num_tokens;
  const int id = t < p.max_num_tokens ? p.mapping[t] : -1;
  for (int i = tid; i < 32 * kSmallBins; i += blockDim.x) (&cnt[0][0])[i] = 0;
  uint32_t st = 0;
  if (n < 0) {
    n = 0;
    st = 2u;
  }
  if (n > p.max_num_tokens) {
    n = p.max_num_tokens;
    st = 2u;
  }
  // bin of this thread's token (nbins: no token)
  int bin = nbins;
  bool bad = false;
  if (t < n) {
    if (id >= 0 && id < L) {
      bin = id;
    } else {
      bin = L;
      bad = id != -1;
    }
  }
  if (__syncthreads_or(bad)) st |= 1u;  // (and the counts are zeroed)
  const unsigned peers = __match_any_sync(0xffffffffu, bin);
  if (bin < nbins && lane == __ffs(peers) - 1) cnt[warp][bin] = __popc(peers);
  __syncthreads();

  // per bin: the warps' offsets inside the bin (warp scan over the warps) and the total
  for (int b = warp; b < nbins; b += nwarps) {
    const int c = lane < nwarps ? cnt[lane][b] : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane < nwarps) cnt[lane][b] = incl - c;
    if (lane == 31) total[b] = incl;
  }
  __syncthreads();

  // one warp: bin starts and, per tile height, each adapter's first tile
  if (warp == 0) {
    int run[1 + kNumTileSizes] = {0, 0, 0, 0, 0};
    for (int b0 = 0; b0 < nbins; b0 += 32) {
      const int b = b0 + lane;
      int v[1 + kNumTileSizes];
      const int tot = b < nbins ? total[b] : 0;
      v[0] = tot;
#pragma unroll
      for (int k = 0; k < kNumTileSizes; ++k)
        v[1 + k] = b < L ? (tot + tile_rows_of(k) - 1) / tile_rows_of(k) : 0;
#pragma unroll
      for (int a = 0; a < 1 + kNumTileSizes; ++a) {
        int incl = v[a];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int excl = run[a] + incl - v[a];
        if (b <= nbins) {
          if (a == 0) start[b] = excl;
          else toff[a - 1][b] = excl;
        }
        run[a] += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    // the entries past the last bin (b == nbins when nbins is a multiple of 32)
    if (lane == 0 && nbins % 32 == 0) {
      start[nbins] = run[0];
#pragma unroll
      for (int k = 0; k < kNumTileSizes; ++k) toff[k][nbins] = run[1 + k];
    }
  }
  __syncthreads();

  // this thread's token: sorted_token_ids and its entry in every tile list
  if (bin < nbins) {
    const int rel = cnt[warp][bin] + __popc(peers & ((1u << lane) - 1u));
    p.sorted_ids[start[bin] + rel] = t;
    if (bin < L) {
#pragma unroll
      for (int k = 0; k < kNumTileSizes; ++k) {
        const int tile = toff[k][bin] + (rel >> (4 + k));
        p.ws.lists[k][static_cast<long long>(tile) * record_ints(tile_rows_of(k)) +
                      kRecordHeaderInts + (rel & (tile_rows_of(k) - 1))] = t;
      }
    }
  } else if (t >= n && t < p.max_num_tokens) {
    p.sorted_ids[t] = -1;
  }
  for (int b = tid; b < nbins; b += blockDim.x) p.counts[b] = total[b];
  for (int b = tid; b <= nbins; b += blockDim.x) p.starts[b] = start[b];
  // record headers (largest adapter l with toff[l] <= i: adapters without a
  // tile share the next offset)
#pragma unroll
  for (int k = 0; k < kNumTileSizes; ++k) {
    const int rows = tile_rows_of(k);
    const int count = toff[k][L];
    int32_t* list = p.ws.lists[k];
    for (int i = tid; i < count; i += blockDim.x) {
      int a = 0, b = L - 1;
      while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (toff[k][mid] <= i) a = mid; else b = mid - 1;
      }
      const int j = i - toff[k][a];
      *reinterpret_cast<int4*>(list + static_cast<long long>(i) * record_ints(rows)) =
          make_int4(a, min(rows, total[a] - j * rows), start[a] + j * rows, 0);
    }
    if (tid == 0) p.ws.num_tiles[k] = count;
  }
  if (tid == 0) {
    *p.ws.n = n;
    if (st) atomicOr(p.ws.status, st);
  }
  __threadfence();
  __syncthreads();
  pdl_launch_dependents();
}

static size_t meta_smem_bytes(int num_loras) {
  const size_t nb = static_cast<size_t>(num_loras) + 1;
  return sizeof(int32_t) * (kMetaWarps * nb + nb + (nb + 1) + kScanArrays * nb +
                            kScanArrays * (nb + 1) + 2 * nb);
}

int launch_metadata(const int32_t* mapping, const int32_t* num_tokens, int max_num_tokens,
                    int num_loras, int32_t* sorted_ids, int32_t* counts, int32_t* starts,
                    void* workspace, cudaStream_t stream) {
  MetaParams p;
  p.mapping = mapping;
  p.num_tokens = num_tokens;
  p.max_num_tokens = max_num_tokens;
  p.num_loras = num_loras;
  p.sorted_ids = sorted_ids;
  p.counts = counts;
  p.starts = starts;
  p.ws = ws_view(workspace, max_num_tokens, num_loras);
  if (max_num_tokens <= kSmallMaxTokens && num_loras <= kSmallMaxLoras) {
    const int threads = (max_num_tokens + 31) / 32 * 32;
    return launch_pdl(reinterpret_cast<const void*>(lora_metadata_small_kernel), dim3(1),
                      dim3(static_cast<unsigned>(threads)), 0, stream, 0, &p);
  }
  const size_t smem = meta_smem_bytes(num_loras);
  if (ensure_smem_attr(reinterpret_cast<const void*>(lora_metadata_kernel), smem) != 0)
    return -6;
  // one CTA per 1024 tokens of the buffer, a power of two up to 8: one cluster
  int cluster = 1;
  while (cluster < 8 && static_cast<long long>(cluster) * 1024 < max_num_tokens) cluster *= 2;
  return launch_pdl(reinterpret_cast<const void*>(lora_metadata_kernel), dim3(cluster),
                    dim3(kMetaThreads), smem, stream, cluster, &p);
}

}  // namespace grg
