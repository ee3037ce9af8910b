// One-kernel layer for decode-sized batches: split-K shrink, then the expand,
// in a single launch ("[V1] LoRA - Add triton kernels for V1": the shrink and
// the expand load the batch's tokens through the token -> LoRA grouping; the
// launch grid depends only on the static sizes, so it can be graph-captured).
//
// CTA (tile T, split j) of a grid of tile_capacity x split CTAs:
//  1. shrink: multiplies the 16 gathered x rows of tile T by A over its
//     contiguous share of the hidden dimension (every k-block of the share in
//     shared memory at once: x rows by cp.async, A blocks by TMA) with
//     mma.sync (bf16 or fp16 in, fp32 accumulate), sums its warps and stores
//     the fp32 partial tile into the workspace;
//  2. hand-off: publishes the partial with a release (fence, then an atomic
//     add on tile T's arrival counter) and waits, with an acquire load, until
//     every CTA of tile T has published;
//  3. expand: sums tile T's split partial tiles in CTA order (the operations
//     of the two-kernel split-K path, so the results are bit for bit those of
//     lora_shrink_partials + lora_expand_partials), scales, stores u (CTA 0),
//     and adds u * B into its 256-column blocks j, j + split, ... of tile T's
//     y rows; B blocks (TMA) and y segments (cp.async) were requested right
//     after the dependency wait, so they land while the shrink runs.
// The waits in 2 end because every CTA of the grid is resident at once (the
// host launches this kernel only when the grid fits the device at its
// occupancy; CTAs from the kernel ahead on the stream finish on their own,
// and no dependent kernel can start before all of this grid's CTAs have run
// its trigger) and, like every wait here, they give up after a time limit and
// report LORA_STATUS_TIMEOUT.
//
// Arrival counters: each CTA adds 16 / split (split is a power of two up to
// 16), so a finished tile adds 16 and every counter is a multiple of 16 when a
// launch starts; a CTA's target is its own fetched value rounded down to a
// multiple of 16, plus 16.  lora_prepare_metadata zeroes the counters; nothing
// has to reset them between launches.
//
// Before griddepcontrol.wait a CTA reads its tile record and prefetches its
// x rows, A, B blocks and y rows into L2; everything else comes after it.
#include <cstring>

#include "common.cuh"
#include "launch.h"

namespace grg {

constexpr int kSFThreads = 128;
constexpr int kSFBM = 16;         // tokens per tile
constexpr int kSFEN = 256;        // output columns per expand item (64 per warp)
constexpr int kSFYPitch = 528;    // staged y row bytes (512 + 16)
constexpr int kSFMaxStages = 3;
constexpr int kSFMaxSplit = 16;

struct SplitFusedParams {
  CUtensorMap amap[3];  // A_s viewed as [L * R][hidden], boxes of R x 64
  CUtensorMap bmap[3];  // B_s viewed as [L * R][N_s], boxes of R x 64
  const __nv_bfloat16* x;
  long long x_stride;
  int hidden;
  int kblocks;
  int kb_per;  // k-blocks per split CTA
  int split;
  int num_slices;
  int sr;  // num_slices * rank
  float scale;
  const float* lora_scales;  // per-adapter factors on scale, or null
  float* u;
  int max_num_tokens;
  __nv_bfloat16* y;
  long long y_stride;
  int width[3];
  int col_off[3];
  int cb_start[4];  // cumulative 256-column blocks per slice
  int items_per;    // expand items per CTA
  int nstages;      // expand ring stages (1..3)
  int warps_n;      // shrink: warps splitting the S*R columns (1 or 2)
  int ntw;          // shrink: n8 column tiles per warp
  const int32_t* records;  // tile records of height 16
  const int32_t* num_tiles;
  uint32_t* status;
  int tile_capacity;
  int num_loras;
  float* partials;          // [tile][split][16][sr] fp32
  unsigned int* arrivals;   // [tile_capacity]
  // shared-memory plan (byte offsets from the 1024-aligned base)
  int off_xa;   // per k-block: x rows [16][128 B], then A rows [sr][128 B]
  int off_u;    // u tile [16][u_pitch]
  int u_pitch;
  int off_st;   // expand stages: B boxes [4][R][128 B], then y [16][kSFYPitch]
  int stage_bytes;
  int off_rec;
  int off_bar;  // barA, barB[kSFMaxStages]
};

__device__ __forceinline__ float4 ld_cg_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

template <int RANK, int NTW, bool F16>
__global__ void __launch_bounds__(kSFThreads)
    lora_split_fused_kernel(const __grid_constant__ SplitFusedParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (sbase - raw);
  int32_t* rec = reinterpret_cast<int32_t*>(smem + p.off_rec);
  const uint32_t bar_a = sbase + p.off_bar;
  const uint32_t bar_b = bar_a + 8;
  __shared__ unsigned int s_flag;  // bit 0: a wait timed out; bit 1: the hand-off failed

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int SR = p.sr;
  const int tile = blockIdx.x / p.split;
  const int j = blockIdx.x - tile * p.split;
  const int ntiles = min(max(*p.num_tiles, 0), p.tile_capacity);
  if (tile >= ntiles) {
    // no work, but the grid must not complete before the kernel ahead of it
    pdl_wait();
    pdl_launch_dependents();
    return;
  }

  if (tid == 0) {
    s_flag = 0;
    for (int i = 0; i < 1 + kSFMaxStages; ++i) mbar_init(bar_a + 8 * i, 1);
    fence_mbar_init();
    for (int s = 0; s < p.num_slices; ++s) {
      prefetch_tmap(&p.amap[s]);
      prefetch_tmap(&p.bmap[s]);
    }
  }
  load_record<kSFBM>(p.records, tile, rec);  // lora_prepare_metadata's output
  __syncthreads();
  const TileView tv = TileView::of(rec, kSFBM, p.num_loras);
  const int lora = tv.lora, cnt = tv.count;
  const int kb0 = j * p.kb_per;
  const int nkb = max(min(kb0 + p.kb_per, p.kblocks) - kb0, 0);

  // expand item k of this CTA: column block j + k * split of the tile
  struct Item {
    int s, c0, width, off;
    bool ok;
  };
  auto item_of = [&](int k) {
    Item it;
    const int cb = j + k * p.split;
    it.ok = k < p.items_per && cb < p.cb_start[p.num_slices];
    const int s = cb >= p.cb_start[1] ? (cb >= p.cb_start[2] ? 2 : 1) : 0;
    it.s = s;
    it.c0 = (cb - p.cb_start[s]) * kSFEN;
    it.width = p.width[s];
    it.off = p.col_off[s];
    return it;
  };
  int nitems = 0;
  while (nitems < p.items_per && item_of(nitems).ok) ++nitems;
  const int NS = p.nstages;

  // ---- before the dependency wait: L2 prefetches only (L2 is the coherence
  // point, so the copies after the wait still read the final values)
  if (tid == 0) {
    for (int i = 0; i < nkb; ++i)
      for (int s = 0; s < p.num_slices; ++s)
        tma_prefetch_2d(&p.amap[s], (kb0 + i) * 64, lora * RANK);
    for (int k = 0; k < min(nitems, NS); ++k) {
      const Item it = item_of(k);
      const int boxes = min(4, (it.width - it.c0 + 63) / 64);
      for (int b = 0; b < boxes; ++b)
        tma_prefetch_2d(&p.bmap[it.s], it.c0 + 64 * b, lora * RANK);
    }
  }
  for (int r = tid; r < cnt; r += kSFThreads) {
    const int t = record_token(rec, r, cnt, p.max_num_tokens);
    if (t < 0) continue;
    if (nkb > 0)
      prefetch_l2(p.x + static_cast<long long>(t) * p.x_stride + kb0 * 64,
                  min(nkb * 64, p.hidden - kb0 * 64) * 2);
    for (int k = 0; k < min(nitems, NS); ++k) {
      const Item it = item_of(k);
      prefetch_l2(p.y + static_cast<long long>(t) * p.y_stride + it.off + it.c0,
                  min(kSFEN, it.width - it.c0) * 2);
    }
  }
  pdl_wait();
  pdl_launch_dependents();

  // ---- copies: A blocks (TMA), x rows (group 0), then per stage the B block
  // (TMA) and the y segments (one cp.async group per item)
  auto issue_item = [&](int k) {
    const Item it = item_of(k);
    const uint32_t st = sbase + p.off_st + (k % NS) * p.stage_bytes;
    if (tid == 0) {
      const uint32_t bar = bar_b + 8 * (k % NS);
      const int boxes = min(4, (it.width - it.c0 + 63) / 64);
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(boxes * RANK * 128));
      for (int b = 0; b < boxes; ++b)
        tma_load_2d(st + b * RANK * 128, &p.bmap[it.s], it.c0 + 64 * b, lora * RANK, bar);
    }
    const int ych = tid & 31;
    const int col = it.c0 + ych * 8;
#pragma unroll
    for (int i = 0; i < kSFBM / 4; ++i) {
      const int row = (tid >> 5) + 4 * i;
      const int t = record_token(rec, row, cnt, p.max_num_tokens);
      const bool ok = t >= 0 && col < it.width;
      cp_async_16(st + 4 * RANK * 128 + row * kSFYPitch + ych * 16,
                  ok ? p.y + static_cast<long long>(t) * p.y_stride + it.off + col : p.y, ok);
    }
    cp_async_commit();
  };
  if (tid == 0 && nkb > 0) {
    mbar_arrive_expect_tx(bar_a, static_cast<uint32_t>(nkb * SR * 128));
    for (int i = 0; i < nkb; ++i)
      for (int s = 0; s < p.num_slices; ++s)
        tma_load_2d(sbase + p.off_xa + i * (kSFBM + SR) * 128 + kSFBM * 128 + s * RANK * 128,
                    &p.amap[s], (kb0 + i) * 64, lora * RANK, bar_a);
  }
  for (int c = tid; c < nkb * kSFBM * 8; c += kSFThreads) {
    const int i = c >> 7, row = (c >> 3) & 15, ch = c & 7;
    const int t = record_token(rec, row, cnt, p.max_num_tokens);
    const int kcol = (kb0 + i) * 64 + ch * 8;
    const bool ok = t >= 0 && kcol < p.hidden;
    cp_async_16(sbase + p.off_xa + i * (kSFBM + SR) * 128 + swz128(row, ch),
                ok ? p.x + static_cast<long long>(t) * p.x_stride + kcol : p.x, ok);
  }
  cp_async_commit();
  const int npro = min(nitems, NS);
  for (int k = 0; k < npro; ++k) issue_item(k);

  bool timed_out = false;
  // ---- 1. shrink over this CTA's k-range
  {
    const int NT = SR >> 3;
    const int WK = 4 / p.warps_n;
    const int wn = warp % p.warps_n, wk = warp / p.warps_n;
    const int nt0 = wn * p.ntw;
    const int nt_cnt = min(p.ntw, NT - nt0);
    float acc[NTW][4];
#pragma unroll
    for (int jj = 0; jj < NTW; ++jj)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[jj][e] = 0.f;
    cp_async_wait_dyn(npro);  // the x rows (the items' groups may stay in flight)
    __syncthreads();
    if (nkb > 0 && !mbar_wait(bar_a, 0)) timed_out = true;
    for (int i = 0; i < nkb; ++i) {
      const uint32_t sx = sbase + p.off_xa + i * (kSFBM + SR) * 128;
      const uint32_t sw = sx + kSFBM * 128;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        if ((ks & (WK - 1)) != wk) continue;
        uint32_t af[4];
        ldsm_x4(af, sx + swz128(lane & 15, ks * 2 + (lane >> 4)));
#pragma unroll
        for (int jj = 0; jj < NTW; jj += 2) {
          if (jj < nt_cnt) {
            const int n0 = (nt0 + jj) * 8;
            uint32_t bf[4];
            if (jj + 1 < nt_cnt) {
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
            mma_t<F16>(acc[jj], af, bf[0], bf[1]);
            if (jj + 1 < NTW && jj + 1 < nt_cnt) mma_t<F16>(acc[jj + 1], af, bf[2], bf[3]);
          }
        }
      }
    }
    __syncthreads();  // every warp is done with the x / A blocks
    // partial tile of each k-split warp -> red[wk][row][col] (aliases x / A)
    float* red = reinterpret_cast<float*>(smem + p.off_xa);
#pragma unroll
    for (int jj = 0; jj < NTW; ++jj) {
      if (jj < nt_cnt) {
        const int col = (nt0 + jj) * 8 + 2 * q;
        *reinterpret_cast<float2*>(red + (wk * kSFBM + g) * SR + col) =
            make_float2(acc[jj][0], acc[jj][1]);
        *reinterpret_cast<float2*>(red + (wk * kSFBM + g + 8) * SR + col) =
            make_float2(acc[jj][2], acc[jj][3]);
      }
    }
    __syncthreads();
    // the CTA's partial tile (its warps summed in order) -> the workspace
    const int e4 = (kSFBM * SR) >> 2;
    float4* dst = reinterpret_cast<float4*>(p.partials) +
                  (static_cast<long long>(tile) * p.split + j) * e4;
    for (int idx = tid; idx < e4; idx += kSFThreads) {
      float4 v = reinterpret_cast<float4*>(red)[idx];
      for (int w = 1; w < WK; ++w) {
        const float4 o = reinterpret_cast<float4*>(red + w * kSFBM * SR)[idx];
        v.x += o.x;
        v.y += o.y;
        v.z += o.z;
        v.w += o.w;
      }
      dst[idx] = v;
    }
  }

  // ---- 2. hand-off: publish (release), then wait for the tile's split CTAs
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned int mine = static_cast<unsigned int>(kSFMaxSplit / p.split);
    const unsigned int got = atomicAdd(p.arrivals + tile, mine);
    const unsigned int target = (got & ~15u) + 16u;
    bool ok = true;
    if (static_cast<int>(ld_acquire_u32(p.arrivals + tile) - target) < 0) {
      const unsigned long long t0 = global_ns();
      while (static_cast<int>(ld_acquire_u32(p.arrivals + tile) - target) < 0) {
        if (global_ns() - t0 > kWaitLimitNs) {
          ok = false;
          break;
        }
      }
    }
    if (!ok) s_flag |= 2u;
  }
  __syncthreads();
  const bool handoff_ok = (s_flag & 2u) == 0;
  if (!handoff_ok) timed_out = true;

  // ---- 3. u = c(lora) * (sum of the split's partial tiles in CTA order)
  {
    const int e4 = (kSFBM * SR) >> 2;
    const int q4 = SR >> 2;
    const float* P = p.partials + static_cast<long long>(tile) * p.split * kSFBM * SR;
    const float c = p.lora_scales != nullptr ? p.scale * p.lora_scales[lora] : p.scale;
    for (int idx = tid; idx < e4; idx += kSFThreads) {
      const int row = idx / q4, c4 = idx - row * q4;
      float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
      if (row < cnt && handoff_ok) {
        float4 part[kSFMaxSplit];
#pragma unroll
        for (int cc = 0; cc < kSFMaxSplit; ++cc)
          if (cc < p.split) part[cc] = ld_cg_f4(P + (cc * kSFBM + row) * SR + c4 * 4);
        sum = part[0];
#pragma unroll
        for (int cc = 1; cc < kSFMaxSplit; ++cc) {
          if (cc < p.split) {
            sum.x += part[cc].x;
            sum.y += part[cc].y;
            sum.z += part[cc].z;
            sum.w += part[cc].w;
          }
        }
        sum = make_float4(sum.x * c, sum.y * c, sum.z * c, sum.w * c);
      }
      *reinterpret_cast<float4*>(smem + p.off_u + row * p.u_pitch + c4 * 16) = sum;
      const int t = record_token(rec, row, cnt, p.max_num_tokens);
      if (j == 0 && t >= 0 && handoff_ok) {
        const int col = c4 * 4;
        const int s = col / RANK, r = col - s * RANK;
        *reinterpret_cast<float4*>(p.u + (static_cast<long long>(s) * p.max_num_tokens + t) *
                                             RANK + r) = sum;
      }
    }
    __syncthreads();
  }

  // ---- 4. expand: y += u * B over this CTA's column blocks of the tile
  for (int k = 0; k < nitems; ++k) {
    // item k's cp.async group; later items' groups may stay in flight
    cp_async_wait_dyn(min(k + NS, nitems) - k - 1);
    __syncthreads();
    if (!mbar_wait(bar_b + 8 * (k % NS), (k / NS) & 1)) timed_out = true;
    const Item it = item_of(k);
    unsigned char* stp = smem + p.off_st + (k % NS) * p.stage_bytes;
    const uint32_t st = sbase + p.off_st + (k % NS) * p.stage_bytes;
    unsigned char* ystage = stp + 4 * RANK * 128;
    if (handoff_ok && cnt > 0) {
      float accx[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) accx[nt][e] = 0.f;
      const float* u0 =
          reinterpret_cast<const float*>(smem + p.off_u + g * p.u_pitch) + it.s * RANK;
      const float* u1 =
          reinterpret_cast<const float*>(smem + p.off_u + (g + 8) * p.u_pitch) + it.s * RANK;
      const uint32_t bw = st + warp * RANK * 128;  // B box of this warp's 64 columns
      if constexpr (RANK == 8) {
        // k = 0..7 carry the high parts, k = 8..15 the residuals; B rows repeat
        const float2 v0 = *reinterpret_cast<const float2*>(u0 + 2 * q);
        const float2 v1 = *reinterpret_cast<const float2*>(u1 + 2 * q);
        uint32_t a[4];
        split_t<F16>(v0.x, v0.y, a[0], a[2]);
        split_t<F16>(v1.x, v1.y, a[1], a[3]);
#pragma unroll
        for (int nt = 0; nt < 8; nt += 4) {
          uint32_t bfr[4];
          ldsm_x4_trans(bfr, bw + swz128(lane & 7, nt + (lane >> 3)));
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) mma_t<F16>(accx[nt + jj], a, bfr[jj], bfr[jj]);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < RANK / 16; ++kk) {
          const int kc = kk * 16 + 2 * q;
          const float2 v00 = *reinterpret_cast<const float2*>(u0 + kc);
          const float2 v10 = *reinterpret_cast<const float2*>(u1 + kc);
          const float2 v01 = *reinterpret_cast<const float2*>(u0 + kc + 8);
          const float2 v11 = *reinterpret_cast<const float2*>(u1 + kc + 8);
          uint32_t ah[4], al[4];
          split_t<F16>(v00.x, v00.y, ah[0], al[0]);
          split_t<F16>(v10.x, v10.y, ah[1], al[1]);
          split_t<F16>(v01.x, v01.y, ah[2], al[2]);
          split_t<F16>(v11.x, v11.y, ah[3], al[3]);
#pragma unroll
          for (int nt = 0; nt < 8; nt += 2) {
            uint32_t bfr[4];
            const int mat = lane >> 3;
            ldsm_x4_trans(bfr, bw + swz128(kk * 16 + ((mat & 1) << 3) + (lane & 7),
                                           nt + (mat >> 1)));
            mma_t<F16>(accx[nt], ah, bfr[0], bfr[1]);
            mma_t<F16>(accx[nt], al, bfr[0], bfr[1]);
            mma_t<F16>(accx[nt + 1], ah, bfr[2], bfr[3]);
            mma_t<F16>(accx[nt + 1], al, bfr[2], bfr[3]);
          }
        }
      }
      // staged y + acc -> 16-bit, written back into the stage
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int cbyte = (warp * 64 + nt * 8 + 2 * q) * 2;
        uint32_t* y0 = reinterpret_cast<uint32_t*>(ystage + g * kSFYPitch + cbyte);
        uint32_t* y1 = reinterpret_cast<uint32_t*>(ystage + (g + 8) * kSFYPitch + cbyte);
        const float2 f0 = unpack_t<F16>(*y0);
        const float2 f1 = unpack_t<F16>(*y1);
        *y0 = pack_t<F16>(f0.x + accx[nt][0], f0.y + accx[nt][1]);
        *y1 = pack_t<F16>(f1.x + accx[nt][2], f1.y + accx[nt][3]);
      }
    }
    __syncthreads();  // the updated stage is complete
    if (handoff_ok) {
      const int ych = tid & 31;
      const int col = it.c0 + ych * 8;
#pragma unroll
      for (int i = 0; i < kSFBM / 4; ++i) {
        const int row = (tid >> 5) + 4 * i;
        const int t = record_token(rec, row, cnt, p.max_num_tokens);
        if (t >= 0 && col < it.width)
          *reinterpret_cast<int4*>(p.y + static_cast<long long>(t) * p.y_stride + it.off + col) =
              *reinterpret_cast<const int4*>(ystage + row * kSFYPitch + ych * 16);
      }
    }
    __syncthreads();  // stage k % NS is free again
    if (k + NS < nitems) {
      fence_proxy_async();  // generic reads of the stage before the TMA refill
      issue_item(k + NS);
    }
  }
  if (timed_out) atomicOr(p.status, kStatusTimeout);
}

namespace {
struct SplitFusedPlan {
  int ok;
  int split, kb_per, items_per, nstages, warps_n, ntw;
  int off_xa, off_u, u_pitch, off_st, stage_bytes, off_rec, off_bar;
  size_t smem;
};

SplitFusedPlan split_fused_plan(int hidden, int num_slices, int rank, int cb_total, int split,
                                int nstages) {
  SplitFusedPlan f = {};
  const int SR = num_slices * rank;
  const int NT = SR / 8;
  f.warps_n = NT <= 8 ? 1 : 2;
  f.ntw = (NT + f.warps_n - 1) / f.warps_n;
  if (f.ntw > 8 || split < 2 || split > kSFMaxSplit || (kSFMaxSplit % split) != 0) return f;
  const int kblocks = (hidden + 63) / 64;
  f.split = split;
  f.kb_per = (kblocks + split - 1) / split;
  f.items_per = (cb_total + split - 1) / split;
  f.nstages = f.items_per < nstages ? f.items_per : nstages;
  const int xa = f.kb_per * (kSFBM + SR) * 128;
  const int red = 4 * kSFBM * SR * 4;
  int off = 0;
  f.off_xa = off;
  off += (xa > red ? xa : red);
  off = (off + 1023) / 1024 * 1024;
  f.off_st = off;
  f.stage_bytes = (4 * rank * 128 + kSFBM * kSFYPitch + 1023) / 1024 * 1024;
  off += f.nstages * f.stage_bytes;
  f.u_pitch = SR * 4 + 16;
  f.off_u = off;
  off += kSFBM * f.u_pitch;
  f.off_rec = off;
  off += record_ints(kSFBM) * 4;
  off = (off + 15) / 16 * 16;
  f.off_bar = off;
  off += 8 * (1 + kSFMaxStages);
  f.smem = 1024 + static_cast<size_t>(off);
  f.ok = f.smem <= 200 * 1024 && f.items_per >= 1;
  return f;
}

template <int RANK, int NTW, bool F16>
const void* split_fused_fn() {
  return reinterpret_cast<const void*>(lora_split_fused_kernel<RANK, NTW, F16>);
}

const void* split_fused_kernel_for(int rank, bool f16) {
  switch (rank) {
    case 8: return f16 ? split_fused_fn<8, 4, true>() : split_fused_fn<8, 4, false>();
    case 16: return f16 ? split_fused_fn<16, 8, true>() : split_fused_fn<16, 8, false>();
    case 32: return f16 ? split_fused_fn<32, 8, true>() : split_fused_fn<32, 8, false>();
    default: return nullptr;
  }
}

// The plan with the most expand stages (3, 2, then 1) whose whole grid is
// resident at once on the current device; ok = 0 when none is.
SplitFusedPlan split_fused_choose(int max_num_tokens, int num_loras, int hidden,
                                  const int* widths, int num_slices, int rank, int split,
                                  bool f16, const void** fn_out, long long* grid_out) {
  SplitFusedPlan none = {};
  const void* fn = split_fused_kernel_for(rank, f16);
  if (fn == nullptr || max_num_tokens > 1024) return none;
  int cb_total = 0;
  for (int s = 0; s < num_slices; ++s) cb_total += (widths[s] + kSFEN - 1) / kSFEN;
  const long long grid = tile_list_capacity(max_num_tokens, num_loras, 0) * split;
  const int sms = device_sm_count();
  if (sms <= 0) return none;
  for (int ns = kSFMaxStages; ns >= 1; --ns) {
    const SplitFusedPlan f = split_fused_plan(hidden, num_slices, rank, cb_total, split, ns);
    if (!f.ok) return none;
    if (ensure_smem_attr(fn, f.smem) != 0) return none;
    const int per_sm = occupancy_blocks(fn, kSFThreads, f.smem);
    if (per_sm >= 1 && grid <= static_cast<long long>(sms) * per_sm) {
      *fn_out = fn;
      *grid_out = grid;
      return f;
    }
    if (f.nstages < ns) break;  // fewer items than stages: fewer stages change nothing
  }
  return none;
}
}  // namespace

int split_fused_fits(int max_num_tokens, int num_loras, int hidden, const int* widths,
                     int num_slices, int rank, int split, bool f16) {
  const void* fn = nullptr;
  long long grid = 0;
  return split_fused_choose(max_num_tokens, num_loras, hidden, widths, num_slices, rank, split,
                            f16, &fn, &grid)
      .ok;
}

int launch_split_fused(const ShrinkArgs& sa, const ExpandArgs& ea, int split, float* partials,
                       unsigned int* arrivals, cudaStream_t stream) {
  if (sa.a_tables[0] != nullptr || ea.b_tables[0] != nullptr) return 0;  // paged: not here
  const int rank = sa.rank;
  int cb_start[4] = {0, 0, 0, 0};
  for (int s = 0; s < 3; ++s)
    cb_start[s + 1] = cb_start[s] + (s < ea.num_slices ? (ea.slice_width[s] + kSFEN - 1) / kSFEN : 0);
  // every CTA of the grid must be resident at once (the hand-off waits on
  // other CTAs of the same tile)
  const void* fn = nullptr;
  long long grid = 0;
  const SplitFusedPlan f =
      split_fused_choose(sa.max_num_tokens, sa.num_loras, sa.hidden, ea.slice_width,
                         sa.num_slices, rank, split, sa.f16, &fn, &grid);
  if (!f.ok) return 0;

  SplitFusedParams p;
  memset(&p, 0, sizeof(p));
  for (int s = 0; s < 3; ++s) {
    if (s < sa.num_slices) {
      if (make_weight_tmap(&p.amap[s], sa.lora_a[s], sa.hidden,
                           static_cast<long long>(sa.num_loras) * rank, rank) != 0 ||
          make_weight_tmap(&p.bmap[s], ea.lora_b[s], ea.slice_width[s],
                           static_cast<long long>(sa.num_loras) * rank, rank) != 0)
        return -6;
      p.width[s] = ea.slice_width[s];
    } else {
      p.amap[s] = p.amap[0];
      p.bmap[s] = p.bmap[0];
    }
  }
  for (int s = 0, acc = 0; s < 3; ++s) {
    p.col_off[s] = acc;
    acc += p.width[s];
  }
  for (int s = 0; s < 4; ++s) p.cb_start[s] = cb_start[s];
  p.x = static_cast<const __nv_bfloat16*>(sa.x);
  p.x_stride = sa.x_row_stride;
  p.hidden = sa.hidden;
  p.kblocks = (sa.hidden + 63) / 64;
  p.kb_per = f.kb_per;
  p.split = f.split;
  p.num_slices = sa.num_slices;
  p.sr = sa.num_slices * rank;
  p.scale = sa.scale;
  p.lora_scales = sa.lora_scales;
  p.u = sa.u;
  p.max_num_tokens = sa.max_num_tokens;
  p.y = static_cast<__nv_bfloat16*>(ea.y);
  p.y_stride = ea.y_row_stride;
  p.items_per = f.items_per;
  p.nstages = f.nstages;
  p.warps_n = f.warps_n;
  p.ntw = f.ntw;
  WsView ws = ws_view(const_cast<void*>(sa.workspace), sa.max_num_tokens, sa.num_loras);
  p.records = ws.lists[0];
  p.num_tiles = ws.num_tiles;
  p.status = ws.status;
  p.tile_capacity = static_cast<int>(grid / f.split);
  p.num_loras = sa.num_loras;
  p.partials = partials;
  p.arrivals = arrivals;
  p.off_xa = f.off_xa;
  p.off_u = f.off_u;
  p.u_pitch = f.u_pitch;
  p.off_st = f.off_st;
  p.stage_bytes = f.stage_bytes;
  p.off_rec = f.off_rec;
  p.off_bar = f.off_bar;
  const int rc = launch_pdl(fn, dim3(static_cast<unsigned>(grid)), dim3(kSFThreads), f.smem,
                            stream, 0, &p);
  return rc == 0 ? 1 : rc;
}

}  // namespace grg
