// Shrink: u[s][t][r] = scale * sum_h x[t][h] * A_s[m[t]][r][h] over the
// tokens of an unsorted batch ("[V1] LoRA - Add triton kernels for V1",
// "Why do we need a new set of kernels" and "Kernel Code Change" point 2: the
// input tokens are loaded through the token -> LoRA grouping, the rest is the
// SGMV-style matmul).
//
// Work decomposition (fixed grid, graph-safe): the metadata kernel wrote a
// list of tiles, each up to BM tokens of one LoRA.  A thread-block cluster of
// C CTAs owns one tile at a time and splits the hidden dimension H into C
// contiguous ranges; every CTA streams its range of the gathered x rows and of
// the adapter's A rows (all slices stacked, S*R rows) through a 4-stage
// cp.async ring into XOR-swizzled shared memory and multiplies them on the
// tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate).  The C partial
// tiles are then summed in a fixed order through distributed shared memory
// (no atomics, no global scratch), scaled once and stored to u.  Clusters loop
// over the tile list with a stride of the cluster count, so the grid depends
// only on the device, never on the batch.
#include "common.cuh"
#include "launch.h"

namespace grg {

constexpr int kShrinkThreads = 128;
constexpr int kBK = 64;  // bf16 columns per k-block: one 128-byte row chunk

struct ShrinkParams {
  const __nv_bfloat16* x;
  long long x_stride;
  int hidden;
  int kblocks;      // ceil(hidden / kBK)
  int kb_per_rank;  // k-blocks owned by each CTA of a cluster
  const __nv_bfloat16* a0;
  const __nv_bfloat16* a1;
  const __nv_bfloat16* a2;
  int rank;
  int rank_shift;  // log2(rank)
  int sr;          // num_slices * rank: stacked A rows
  float scale;
  float* u;
  int max_num_tokens;
  const int32_t* records;    // tile records of height BM
  const int32_t* num_tiles;
  int tile_capacity;         // records the list can hold
  int num_loras;
  int warps_n;     // warps splitting the S*R columns (1, 2 or 4)
  int ntw;         // n8 column tiles per warp
  int rec_offset;  // byte offset of the tile record in shared memory
};

// Byte offset of 16-byte chunk ch (0..7) of a 128-byte row, XOR-swizzled so
// that eight consecutive rows read at the same chunk hit distinct banks.
__device__ __forceinline__ uint32_t swz128(int row, int ch) {
  return static_cast<uint32_t>(row * 128 + ((ch ^ (row & 7)) << 4));
}

template <int BM, int NTW, int NST>
__global__ void __launch_bounds__(kShrinkThreads, 4) lora_shrink_kernel(const ShrinkParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  int32_t* rec = reinterpret_cast<int32_t*>(smem + p.rec_offset);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int SR = p.sr;
  const int NT = SR >> 3;
  const int WK = 4 / p.warps_n;
  const int wn = warp % p.warps_n, wk = warp / p.warps_n;
  const int nt0 = wn * p.ntw;
  const int nt_cnt = min(p.ntw, NT - nt0);
  const int stage_bytes = (BM + SR) * 128;
  const uint32_t smem_base = smem_u32(smem);

  uint32_t cl_size;
  asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(cl_size));
  const int C = static_cast<int>(cl_size);
  const int crank = static_cast<int>(cluster_ctarank());
  const int cluster_id = blockIdx.x / C;
  const int nclusters = gridDim.x / C;
  const int kb0 = crank * p.kb_per_rank;
  const int kb1 = min(kb0 + p.kb_per_rank, p.kblocks);
  const int nkb = max(kb1 - kb0, 0);

  pdl_wait();
  pdl_launch_dependents();
  // the first record is fetched together with the count (it may be unused)
  if (cluster_id < p.tile_capacity) load_record<BM>(p.records, cluster_id, rec);
  const int ntiles = min(max(*p.num_tiles, 0), p.tile_capacity);

  for (int item = cluster_id; item < ntiles; item += nclusters) {
    if (item != cluster_id) load_record<BM>(p.records, item, rec);
    __syncthreads();
    const TileView tv = TileView::of(rec, BM, p.num_loras);
    const int lora = tv.lora, cnt = tv.count;

    auto load_stage = [&](int st, int kb) {
      const uint32_t sx = smem_base + st * stage_bytes;
      const uint32_t sw = sx + BM * 128;
      const int col = kb * kBK;
      for (int c = tid; c < BM * 8; c += kShrinkThreads) {
        const int row = c >> 3, ch = c & 7;
        const int t = record_token(rec, row, cnt, p.max_num_tokens);
        const int kcol = col + ch * 8;
        const bool ok = (t >= 0) && (kcol < p.hidden);
        const __nv_bfloat16* src = ok ? p.x + static_cast<long long>(t) * p.x_stride + kcol : p.x;
        cp_async_16(sx + swz128(row, ch), src, ok);
      }
      for (int c = tid; c < SR * 8; c += kShrinkThreads) {
        const int row = c >> 3, ch = c & 7;
        const int s = row >> p.rank_shift;
        const int r = row - (s << p.rank_shift);
        const int kcol = col + ch * 8;
        const bool ok = kcol < p.hidden && cnt > 0;
        const __nv_bfloat16* a = s == 0 ? p.a0 : (s == 1 ? p.a1 : p.a2);
        const __nv_bfloat16* src =
            ok ? a + (static_cast<long long>(lora) * p.rank + r) * p.hidden + kcol : p.a0;
        cp_async_16(sw + swz128(row, ch), src, ok);
      }
    };

    float acc[BM / 16][NTW][4];
#pragma unroll
    for (int mi = 0; mi < BM / 16; ++mi)
#pragma unroll
      for (int j = 0; j < NTW; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mi][j][e] = 0.f;

    // keep NST - 1 k-blocks in flight (all of them when the range is short)
#pragma unroll
    for (int s = 0; s < NST - 1; ++s) {
      if (s < nkb) load_stage(s, kb0 + s);
      cp_async_commit();
    }

    for (int i = 0; i < nkb; ++i) {
      cp_async_wait<NST - 2>();
      __syncthreads();
      const int nxt = i + NST - 1;
      if (nxt < nkb) load_stage(nxt % NST, kb0 + nxt);
      cp_async_commit();

      const uint32_t sx = smem_base + (i % NST) * stage_bytes;
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
    }
    cp_async_wait<0>();
    __syncthreads();

    // partial tile -> red[wk][row][col] (aliases the stage ring)
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
    cluster_sync_all();

    // cluster reduction in a fixed order, scale, store the valid rows
    const int e4 = (BM * SR) >> 2;
    for (int idx = crank * kShrinkThreads + tid; idx < e4; idx += C * kShrinkThreads) {
      const int e = idx << 2;
      const int row = e / SR;
      const int col = e - row * SR;
      const int t = record_token(rec, row, cnt, p.max_num_tokens);
      if (t < 0) continue;
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c = 0; c < C; ++c) {
        for (int w = 0; w < WK; ++w) {
          const uint32_t local =
              smem_base + static_cast<uint32_t>(((w * BM + row) * SR + col) * 4);
          const float4 v = ld_dsmem_f4(mapa_shared(local, static_cast<uint32_t>(c)));
          sum.x += v.x;
          sum.y += v.y;
          sum.z += v.z;
          sum.w += v.w;
        }
      }
      const int s = col >> p.rank_shift;
      const int r = col - (s << p.rank_shift);
      float* dst = p.u + (static_cast<long long>(s) * p.max_num_tokens + t) * p.rank + r;
      *reinterpret_cast<float4*>(dst) =
          make_float4(sum.x * p.scale, sum.y * p.scale, sum.z * p.scale, sum.w * p.scale);
    }
    cluster_sync_all();
  }
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
  int cluster = 1;
  while (cluster < 8 && static_cast<long long>(cluster) * 2 * max_tiles <= 2LL * sms) cluster *= 2;
  while (cluster > 1 && cluster > kblocks) cluster /= 2;
  const int kb_per = (kblocks + cluster - 1) / cluster;
  // deep ring when a CTA's whole k-range fits: every load is in flight at once
  const size_t stage = static_cast<size_t>(BM + SR) * 128;
  const int nst = (kb_per <= 8 && 8 * stage <= 96 * 1024 && ntw <= 8) ? 8 : 4;

  ShrinkParams p;
  p.x = static_cast<const __nv_bfloat16*>(a.x);
  p.x_stride = a.x_row_stride;
  p.hidden = a.hidden;
  p.kblocks = kblocks;
  p.kb_per_rank = kb_per;
  p.a0 = static_cast<const __nv_bfloat16*>(a.lora_a[0]);
  p.a1 = static_cast<const __nv_bfloat16*>(a.num_slices > 1 ? a.lora_a[1] : a.lora_a[0]);
  p.a2 = static_cast<const __nv_bfloat16*>(a.num_slices > 2 ? a.lora_a[2] : a.lora_a[0]);
  p.rank = a.rank;
  p.rank_shift = __builtin_ctz(static_cast<unsigned>(a.rank));
  p.sr = SR;
  p.scale = a.scale;
  p.u = a.u;
  p.max_num_tokens = a.max_num_tokens;
  WsView ws = ws_view(const_cast<void*>(a.workspace), a.max_num_tokens, a.num_loras);
  p.records = ws.lists[tile_index_of(BM)];
  p.num_tiles = ws.num_tiles + tile_index_of(BM);
  p.tile_capacity = static_cast<int>(max_tiles);
  p.num_loras = a.num_loras;
  p.warps_n = warps_n;
  p.ntw = ntw;
  const size_t ring = static_cast<size_t>(nst) * stage;
  const size_t red = static_cast<size_t>(WK) * BM * SR * 4;
  const size_t body = ring > red ? ring : red;
  p.rec_offset = static_cast<int>(body);
  const size_t smem = body + record_ints(BM) * sizeof(int32_t);

  if (BM == 16) {
    if (ntw > 8) return run_shrink<16, 12, 4>(p, cluster, smem, stream, max_tiles);
    if (nst == 8) return run_shrink<16, 8, 8>(p, cluster, smem, stream, max_tiles);
    return run_shrink<16, 8, 4>(p, cluster, smem, stream, max_tiles);
  }
  if (nst == 8) return run_shrink<32, 8, 8>(p, cluster, smem, stream, max_tiles);
  return run_shrink<32, 8, 4>(p, cluster, smem, stream, max_tiles);
}

}  // namespace grg
