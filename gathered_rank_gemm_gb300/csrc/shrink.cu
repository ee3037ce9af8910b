// Shrink: u[s][t][r] = scale * sum_h x[t][h] * A_s[m[t]][r][h] over the
// tokens of an unsorted batch ("[V1] LoRA - Add triton kernels for V1",
// "Why do we need a new set of kernels" and "Kernel Code Change" point 2: the
// input tokens are loaded through the token -> LoRA grouping, the rest is the
// SGMV-style matmul).
//
// Work decomposition (fixed grid, graph-safe): the metadata kernel wrote a
// list of tiles, each up to BM tokens of one LoRA.  A thread-block cluster of
// C CTAs owns one tile at a time and splits the hidden dimension H into C
// contiguous ranges; clusters walk the list with a stride of the cluster
// count, so the grid depends only on the device.
//
// Data movement, per 64-column k-block, into a ring of NST stages:
//  - the adapter's R x 64 block of every slice with one TMA tile load each
//    (tensor map, 128-byte swizzle), completing on the stage's mbarrier;
//  - the BM gathered x rows with 16-byte cp.async (zero-filled past the
//    tile's tokens and past H), one commit group per stage.
// The adapter blocks of the first tile are requested before
// griddepcontrol.wait (weights are never written by the preceding kernel) and
// the first x rows are prefetched into L2 there.
//
// Compute: tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate); warps
// split the S*R columns and/or the k-steps.  The C partial tiles are summed in
// rank order through distributed shared memory (no atomics, no global
// scratch), scaled once and stored to u.
#include "common.cuh"
#include "launch.h"

namespace grg {

constexpr int kShrinkThreads = 128;
constexpr int kBK = 64;  // bf16 columns per k-block: one 128-byte (swizzled) row chunk

struct ShrinkParams {
  CUtensorMap tmap[3];  // A_s viewed as [L * R][hidden], boxes of R x 64
  const __nv_bfloat16* x;
  long long x_stride;
  int hidden;
  int kblocks;      // ceil(hidden / kBK)
  int kb_per_rank;  // k-blocks owned by each CTA of a cluster
  int num_slices;
  int rank;
  int rank_shift;  // log2(rank)
  int sr;          // num_slices * rank: stacked A rows
  float scale;
  float* u;
  int max_num_tokens;
  const int32_t* records;  // tile records of height BM
  const int32_t* num_tiles;
  uint32_t* status;
  int tile_capacity;  // records the list can hold
  int num_loras;
  int warps_n;     // warps splitting the S*R columns (1, 2 or 4)
  int ntw;         // n8 column tiles per warp
  int stage_bytes;
  int rec_offset;  // byte offsets from the 1024-aligned base
  int bar_offset;
};

template <int BM, int NTW, int NST>
__global__ void __launch_bounds__(kShrinkThreads, BM == 32 ? 3 : 4)
    lora_shrink_kernel(const __grid_constant__ ShrinkParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // TMA's 128-byte swizzle is laid out on 1024-byte boundaries
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (sbase - raw);
  int32_t* rec = reinterpret_cast<int32_t*>(smem + p.rec_offset);
  const uint32_t bars = sbase + p.bar_offset;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int SR = p.sr;
  const int NT = SR >> 3;
  const int WK = 4 / p.warps_n;
  const int wn = warp % p.warps_n, wk = warp / p.warps_n;
  const int nt0 = wn * p.ntw;
  const int nt_cnt = min(p.ntw, NT - nt0);

  uint32_t cl_size;
  asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(cl_size));
  const int C = static_cast<int>(cl_size);
  const int crank = static_cast<int>(cluster_ctarank());
  const int cluster_id = blockIdx.x / C;
  const int nclusters = gridDim.x / C;
  const int kb0 = crank * p.kb_per_rank;
  const int kb1 = min(kb0 + p.kb_per_rank, p.kblocks);
  const int nkb = max(kb1 - kb0, 0);

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(bars + 8 * s, 1);
    fence_mbar_init();
    for (int s = 0; s < p.num_slices; ++s) prefetch_tmap(&p.tmap[s]);
  }
  __syncthreads();

  // the work list is metadata output: safe to read before the dependency wait
  const int ntiles = min(max(*p.num_tiles, 0), p.tile_capacity);
  uint32_t phase = 0;  // bit s: parity of the next phase of stage s
  bool waited = false, timed_out = false;

  // this thread's x chunks: rows (tid >> 3) + 16 j, chunk tid & 7
  constexpr int XJ = BM / 16;
  const int xch = tid & 7;

  for (int item = cluster_id; item < ntiles; item += nclusters) {
    load_record<BM>(p.records, item, rec);
    __syncthreads();
    const TileView tv = TileView::of(rec, BM, p.num_loras);
    const int lora = tv.lora, cnt = tv.count;
    const __nv_bfloat16* xrow[XJ];
#pragma unroll
    for (int j = 0; j < XJ; ++j) {
      const int t = record_token(rec, (tid >> 3) + 16 * j, cnt, p.max_num_tokens);
      xrow[j] = t >= 0 ? p.x + static_cast<long long>(t) * p.x_stride + xch * 8 : nullptr;
    }

    // A blocks of all slices for k-block kb -> stage st (thread 0)
    auto fill_a = [&](int st, int kb) {
      const uint32_t bar = bars + 8 * st;
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(SR * 128));
      const uint32_t sa = sbase + st * p.stage_bytes + BM * 128;
      for (int s = 0; s < p.num_slices; ++s)
        tma_load_2d(sa + s * p.rank * 128, &p.tmap[s], kb * kBK, lora * p.rank, bar);
    };
    // gathered x rows for k-block kb -> stage st (every thread, one group)
    auto fill_x = [&](int st, int kb) {
      const uint32_t sx = sbase + st * p.stage_bytes;
      const int kcol = kb * kBK + xch * 8;
#pragma unroll
      for (int j = 0; j < XJ; ++j) {
        const int row = (tid >> 3) + 16 * j;
        const bool ok = xrow[j] != nullptr && kcol < p.hidden;
        cp_async_16(sx + swz128(row, xch), ok ? xrow[j] + kb * kBK : p.x, ok);
      }
      cp_async_commit();
    };

    const int npro = min(nkb, NST);
    if (tid == 0)
      for (int s = 0; s < npro; ++s) fill_a(s, kb0 + s);
    if (!waited) {
      if (npro > 0) {
        // warm L2 (and the TLB) with this CTA's first x rows while the
        // previous kernel finishes; the copies below then hit L2
        const int kcol = kb0 * kBK;
        const int bytes = min(npro * kBK, p.hidden - kcol) * 2;
        for (int r = tid; r < cnt; r += kShrinkThreads) {
          const int t = record_token(rec, r, cnt, p.max_num_tokens);
          if (t >= 0) prefetch_l2(p.x + static_cast<long long>(t) * p.x_stride + kcol, bytes);
        }
      }
      pdl_wait();
      pdl_launch_dependents();
      waited = true;
    }
    for (int s = 0; s < npro; ++s) fill_x(s, kb0 + s);
    int issued = npro;

    float acc[BM / 16][NTW][4];
#pragma unroll
    for (int mi = 0; mi < BM / 16; ++mi)
#pragma unroll
      for (int j = 0; j < NTW; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mi][j][e] = 0.f;

    for (int i = 0; i < nkb; ++i) {
      const int st = i % NST;
      cp_async_wait_dyn(issued - 1 - i);
      __syncthreads();  // everyone's x chunks of this stage are in
      if (!mbar_wait(bars + 8 * st, (phase >> st) & 1u)) timed_out = true;
      phase ^= 1u << st;
      const uint32_t sx = sbase + st * p.stage_bytes;
      const uint32_t sw = sx + BM * 128;
#pragma unroll
      for (int ks = 0; ks < kBK / 16; ++ks) {
        if ((ks & (WK - 1)) != wk) continue;
        uint32_t af[BM / 16][4];
#pragma unroll
        for (int mi = 0; mi < BM / 16; ++mi)
          ldsm_x4(af[mi], sx + swz128(mi * 16 + (lane & 15), ks * 2 + (lane >> 4)));
#pragma unroll
        for (int j = 0; j < NTW; j += 2) {
          if (j < nt_cnt) {
            const int n0 = (nt0 + j) * 8;
            uint32_t bf[4];
            if (j + 1 < nt_cnt) {
              ldsm_x4(bf, sw + swz128(n0 + (lane & 7) + ((lane >> 4) << 3),
                                      ks * 2 + ((lane >> 3) & 1)));
            } else {
              uint32_t b2[2];
              ldsm_x2(b2, sw + swz128(n0 + (lane & 7), ks * 2 + ((lane >> 3) & 1)));
              bf[0] = b2[0];
              bf[1] = b2[1];
              bf[2] = 0u;
              bf[3] = 0u;
            }
#pragma unroll
            for (int mi = 0; mi < BM / 16; ++mi) {
              mma_bf16(acc[mi][j], af[mi], bf[0], bf[1]);
              if (j + 1 < NTW && j + 1 < nt_cnt) mma_bf16(acc[mi][j + 1], af[mi], bf[2], bf[3]);
            }
          }
        }
      }
      if (i + NST < nkb) {
        __syncthreads();  // every warp is done with this stage
        if (tid == 0) fill_a(st, kb0 + i + NST);
        fill_x(st, kb0 + i + NST);
        ++issued;
      }
    }
    __syncthreads();  // the ring is free: it becomes the reduction buffer

    // partial tile -> red[wk][row][col], then the k-split warps are summed into red[0]
    float* red = reinterpret_cast<float*>(smem);
    {
      const int g = lane >> 2, q = lane & 3;
#pragma unroll
      for (int mi = 0; mi < BM / 16; ++mi)
#pragma unroll
        for (int j = 0; j < NTW; ++j) {
          if (j < nt_cnt) {
            const int col = (nt0 + j) * 8 + 2 * q;
            const int r0 = mi * 16 + g;
            *reinterpret_cast<float2*>(red + (wk * BM + r0) * SR + col) =
                make_float2(acc[mi][j][0], acc[mi][j][1]);
            *reinterpret_cast<float2*>(red + (wk * BM + r0 + 8) * SR + col) =
                make_float2(acc[mi][j][2], acc[mi][j][3]);
          }
        }
    }
    const int e4 = (BM * SR) >> 2;
    if (WK > 1) {
      __syncthreads();
      for (int idx = tid; idx < e4; idx += kShrinkThreads) {
        float4 v = reinterpret_cast<float4*>(red)[idx];
        for (int w = 1; w < WK; ++w) {
          const float4 o = reinterpret_cast<float4*>(red + w * BM * SR)[idx];
          v.x += o.x;
          v.y += o.y;
          v.z += o.z;
          v.w += o.w;
        }
        reinterpret_cast<float4*>(red)[idx] = v;
      }
    }
    cluster_sync_all();

    // cluster reduction in rank order, scale, store the valid rows
    for (int idx = crank * kShrinkThreads + tid; idx < e4; idx += C * kShrinkThreads) {
      const int e = idx << 2;
      const int row = e / SR;
      const int col = e - row * SR;
      const int t = record_token(rec, row, cnt, p.max_num_tokens);
      if (t < 0) continue;
      const uint32_t local = sbase + static_cast<uint32_t>(e * 4);
      float4 part[8];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        if (c < C) part[c] = ld_dsmem_f4(mapa_shared(local, static_cast<uint32_t>(c)));
      float4 sum = part[0];
#pragma unroll
      for (int c = 1; c < 8; ++c) {
        if (c < C) {
          sum.x += part[c].x;
          sum.y += part[c].y;
          sum.z += part[c].z;
          sum.w += part[c].w;
        }
      }
      const int s = col >> p.rank_shift;
      const int r = col - (s << p.rank_shift);
      float* dst = p.u + (static_cast<long long>(s) * p.max_num_tokens + t) * p.rank + r;
      *reinterpret_cast<float4*>(dst) =
          make_float4(sum.x * p.scale, sum.y * p.scale, sum.z * p.scale, sum.w * p.scale);
    }
    fence_proxy_async();  // generic use of the ring before the next item's TMA writes
    cluster_sync_all();
  }
  if (timed_out) atomicOr(p.status, kStatusTimeout);
}

template <int BM, int NTW, int NST>
static int run_shrink(const ShrinkParams& prm, int cluster, size_t smem, cudaStream_t stream,
                      long long max_tiles) {
  const void* fn = reinterpret_cast<const void*>(lora_shrink_kernel<BM, NTW, NST>);
  if (ensure_smem_attr(fn, smem) != 0) return -6;
  const int sms = device_sm_count();
  if (sms <= 0) return -6;
  int per_sm = occupancy_blocks(fn, kShrinkThreads, smem);
  if (per_sm < 1) per_sm = 1;
  long long grid = static_cast<long long>(sms) * per_sm / cluster * cluster;
  const long long useful = max_tiles * cluster;
  if (grid > useful) grid = useful;
  if (grid < cluster) grid = cluster;
  ShrinkParams p = prm;
  return launch_pdl(fn, dim3(static_cast<unsigned>(grid)), dim3(kShrinkThreads), smem, stream,
                    cluster, &p);
}

int launch_shrink(const ShrinkArgs& a, cudaStream_t stream) {
  const int SR = a.num_slices * a.rank;
  const int NT = SR / 8;
  const int warps_n = NT <= 8 ? 1 : (NT <= 16 ? 2 : 4);
  const int ntw = (NT + warps_n - 1) / warps_n;
  const int WK = 4 / warps_n;
  const int BM = (SR >= 192 || a.max_num_tokens <= 1024) ? 16 : 32;
  const int kblocks = (a.hidden + kBK - 1) / kBK;
  const long long max_tiles = tile_list_capacity(a.max_num_tokens, a.num_loras, tile_index_of(BM));
  const int sms = device_sm_count();
  // split the hidden dimension over a cluster until ~3 CTAs per SM have work
  int cluster = 1;
  while (cluster < 8 && static_cast<long long>(cluster) * max_tiles < 3LL * sms &&
         kblocks >= 8 * cluster)
    cluster *= 2;
  const int kb_per = (kblocks + cluster - 1) / cluster;
  // a deep ring keeps up to 8 k-blocks in flight per CTA (all of a short range)
  const int stage = (BM + SR) * 128;  // a multiple of 1024: BM and S*R are multiples of 8
  const int nst = (8 * stage <= 64 * 1024 && ntw <= 8) ? 8 : (4 * stage <= 96 * 1024 ? 4 : 2);

  ShrinkParams p;
  for (int s = 0; s < 3; ++s) {
    if (s < a.num_slices) {
      if (make_weight_tmap(&p.tmap[s], a.lora_a[s], a.hidden,
                           static_cast<long long>(a.num_loras) * a.rank, a.rank) != 0)
        return -6;
    } else {
      p.tmap[s] = p.tmap[0];
    }
  }
  p.x = static_cast<const __nv_bfloat16*>(a.x);
  p.x_stride = a.x_row_stride;
  p.hidden = a.hidden;
  p.kblocks = kblocks;
  p.kb_per_rank = kb_per;
  p.num_slices = a.num_slices;
  p.rank = a.rank;
  p.rank_shift = __builtin_ctz(static_cast<unsigned>(a.rank));
  p.sr = SR;
  p.scale = a.scale;
  p.u = a.u;
  p.max_num_tokens = a.max_num_tokens;
  WsView ws = ws_view(const_cast<void*>(a.workspace), a.max_num_tokens, a.num_loras);
  p.records = ws.lists[tile_index_of(BM)];
  p.num_tiles = ws.num_tiles + tile_index_of(BM);
  p.status = ws.status;
  p.tile_capacity = static_cast<int>(max_tiles);
  p.num_loras = a.num_loras;
  p.warps_n = warps_n;
  p.ntw = ntw;
  p.stage_bytes = stage;
  const int ring = nst * stage;
  const int red = WK * BM * SR * 4;
  const int body = ((ring > red ? ring : red) + 127) / 128 * 128;
  p.rec_offset = body;
  p.bar_offset = body + record_ints(BM) * 4;
  const size_t smem = 1024 + static_cast<size_t>(p.bar_offset) + 8 * 8;

  if (BM == 16) {
    if (ntw > 8) {
      if (nst == 4) return run_shrink<16, 12, 4>(p, cluster, smem, stream, max_tiles);
      return run_shrink<16, 12, 2>(p, cluster, smem, stream, max_tiles);
    }
    if (nst == 8) return run_shrink<16, 8, 8>(p, cluster, smem, stream, max_tiles);
    if (nst == 4) return run_shrink<16, 8, 4>(p, cluster, smem, stream, max_tiles);
    return run_shrink<16, 8, 2>(p, cluster, smem, stream, max_tiles);
  }
  if (nst == 8) return run_shrink<32, 8, 8>(p, cluster, smem, stream, max_tiles);
  if (nst == 4) return run_shrink<32, 8, 4>(p, cluster, smem, stream, max_tiles);
  return run_shrink<32, 8, 2>(p, cluster, smem, stream, max_tiles);
}

}  // namespace grg
