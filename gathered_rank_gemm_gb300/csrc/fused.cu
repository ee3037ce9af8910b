// Fused shrink -> expand for one layer (u = scale * x A^T, then y += u B),
// for batches small enough that one cluster can hold a tile's whole problem
// on chip (decode-sized batches).  The computation is the one of lora_shrink
// followed by lora_expand ("[V1] LoRA - Add triton kernels for V1": gather
// each token's rows through the token -> LoRA grouping, shrink, expand); u is
// still written to global memory, but the expand reads it from shared memory,
// so a layer costs one launch and one pass over the activations.
//
// A cluster of C CTAs owns one tile of up to 16 tokens of one LoRA:
//  - CTA c multiplies the tile's x rows by A over its 1/C of the hidden
//    dimension (all its 64-column k-blocks resident in shared memory at once:
//    A blocks by TMA, x rows by cp.async) with mma.sync (bf16, fp32 acc.);
//  - the C partial tiles are summed in rank order through distributed shared
//    memory by every CTA, so each CTA holds the full fp32 u tile; the CTAs
//    store disjoint parts of it to u;
//  - CTA c then owns 1/C of the output columns (64-column units of the
//    slices): B blocks by TMA and the gathered y segments by cp.async were
//    requested together with x, so the whole read traffic of the layer is in
//    flight at once; u enters the tensor cores as bf16 high + residual terms,
//    y is added in fp32, rounded once and stored with 16-byte stores.
// Before griddepcontrol.wait a CTA only reads its tile record and prefetches
// its weight blocks (A, B) and x / y rows into L2; every copy into shared
// memory comes after the wait.
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "launch.h"

namespace grg {

constexpr int kFusedThreads = 128;
constexpr int kFBM = 16;          // tokens per tile
constexpr int kFusedMaxKb = 16;   // k-blocks per CTA held at once
constexpr int kFusedMaxUnits = 48;

struct FusedParams {
  CUtensorMap amap[3];  // A_s [L*R][H], boxes of R x 64
  CUtensorMap bmap[3];  // B_s [L*R][N_s], boxes of R x 64
  const __nv_bfloat16* x;
  long long x_stride;
  int hidden;
  int kblocks;
  int kb_per_rank;
  int num_slices;
  int rank;
  int rank_shift;
  int sr;
  float scale;
  const float* lora_scales;  // per-adapter factors on scale, or null
  float* u;
  int max_num_tokens;
  __nv_bfloat16* y;
  long long y_stride;
  int width[3];
  int col_off[3];
  int unit_start[4];  // cumulative 64-column units per slice
  int units_per_rank;
  const int32_t* records;  // tile records of height 16
  const int32_t* num_tiles;
  uint32_t* status;
  int tile_capacity;
  int num_loras;
  int warps_n;
  int ntw;
  int off_a, off_x, off_b, off_y, off_u, off_red, off_rec, off_bar;
  // the bounded waits' limit; under the test hook (wait_fault) no copy is
  // issued and the first A barrier is armed with one arrival too many
  unsigned long long wait_limit_ns;
  int wait_fault;
};

template <int NTW, bool F16>
__global__ void __launch_bounds__(kFusedThreads, 1)
    lora_fused_kernel(const __grid_constant__ FusedParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (sbase - raw);
  int32_t* rec = reinterpret_cast<int32_t*>(smem + p.off_rec);
  float* red = reinterpret_cast<float*>(smem + p.off_red);
  float* utile = reinterpret_cast<float*>(smem + p.off_u);
  const uint32_t bar_a = sbase + p.off_bar;                // one per k-block
  const uint32_t bar_b = bar_a + 8 * kFusedMaxKb;          // B blocks

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int SR = p.sr, R = p.rank;
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
  const int nkb = max(min(kb0 + p.kb_per_rank, p.kblocks) - kb0, 0);
  const int units_total = p.unit_start[p.num_slices];
  const int un0 = crank * p.units_per_rank;
  const int nun = max(min(un0 + p.units_per_rank, units_total) - un0, 0);

  // giving up (CtaAbort): the flag after the barriers; the CTA keeps walking
  // its items in step with its cluster (the cluster barriers) but issues no
  // copy and stores nothing more, nor under the test hook
  const CtaAbort cta_abort{reinterpret_cast<int*>(smem + p.off_bar + 8 * (kFusedMaxKb + 1)),
                           p.wait_limit_ns};
  auto stopped = [&]() { return cta_abort.raised() || p.wait_fault != 0; };
  if (tid == 0) {
    *cta_abort.flag = 0;
    for (int i = 0; i < kFusedMaxKb + 1; ++i)
      mbar_init(bar_a + 8 * i, 1 + (p.wait_fault && i == 0 ? 1 : 0));
    fence_mbar_init();
    for (int s = 0; s < p.num_slices; ++s) {
      prefetch_tmap(&p.amap[s]);
      prefetch_tmap(&p.bmap[s]);
    }
  }
  __syncthreads();

  // unit -> slice and first column inside the slice
  auto unit_slice = [&](int unit) {
    return unit >= p.unit_start[1] ? (unit >= p.unit_start[2] ? 2 : 1) : 0;
  };

  const int ntiles = min(max(*p.num_tiles, 0), p.tile_capacity);
  bool waited = false;
  uint32_t phase = 0;
  int issued_phase = -1;  // thread 0: the barrier phase of its last TMA loads

  for (int item = cluster_id; item < ntiles; item += nclusters) {
    load_record<kFBM>(p.records, item, rec);
    __syncthreads();
    const TileView tv = TileView::of(rec, kFBM, p.num_loras);
    const int lora = tv.lora, cnt = tv.count;

    if (!waited) {
      // The kernel ahead on the stream may still be writing any input:
      // before the wait only L2 prefetches (L2 is the coherence point, so the
      // copies after the wait read the final values) of this CTA's weight
      // blocks and x / y rows
      if (tid == 0 && !p.wait_fault) {  // (the test hook issues nothing)
        for (int i = 0; i < nkb; ++i)
          for (int s = 0; s < p.num_slices; ++s)
            tma_prefetch_2d(&p.amap[s], (kb0 + i) * 64, lora * R);
        for (int j = 0; j < nun; ++j) {
          const int unit = un0 + j;
          const int s = unit_slice(unit);
          tma_prefetch_2d(&p.bmap[s], (unit - p.unit_start[s]) * 64, lora * R);
        }
      }
      for (int r = tid; r < cnt && !p.wait_fault; r += kFusedThreads) {
        const int t = record_token(rec, r, cnt, p.max_num_tokens);
        if (t < 0) continue;
        if (nkb > 0)
          prefetch_l2(p.x + static_cast<long long>(t) * p.x_stride + kb0 * 64,
                      min(nkb * 64, p.hidden - kb0 * 64) * 2);
        for (int s = 0; s < p.num_slices; ++s) {
          const int a = max(un0, p.unit_start[s]), b = min(un0 + nun, p.unit_start[s + 1]);
          if (a >= b) continue;
          const int c0 = (a - p.unit_start[s]) * 64;
          const int c1 = min((b - p.unit_start[s]) * 64, p.width[s]);
          prefetch_l2(p.y + static_cast<long long>(t) * p.y_stride + p.col_off[s] + c0,
                      (c1 - c0) * 2);
        }
      }
      pdl_wait();
      pdl_launch_dependents();
      waited = true;
    }
    // weights (A blocks of this CTA's k-range, B blocks of its units) by TMA
    // (none once the CTA has given up: every wait of earlier items is over,
    // so one value for all)
    const bool copy = !stopped();
    if (tid == 0 && copy) {
      issued_phase = static_cast<int>(phase);
      for (int i = 0; i < nkb; ++i) {
        mbar_arrive_expect_tx(bar_a + 8 * i, static_cast<uint32_t>(SR * 128));
        for (int s = 0; s < p.num_slices; ++s)
          tma_load_2d(sbase + p.off_a + i * SR * 128 + s * R * 128, &p.amap[s], (kb0 + i) * 64,
                      lora * R, bar_a + 8 * i);
      }
      if (nun > 0) {
        mbar_arrive_expect_tx(bar_b, static_cast<uint32_t>(nun * R * 128));
        for (int j = 0; j < nun; ++j) {
          const int unit = un0 + j;
          const int s = unit_slice(unit);
          tma_load_2d(sbase + p.off_b + j * R * 128, &p.bmap[s], (unit - p.unit_start[s]) * 64,
                      lora * R, bar_b);
        }
      }
    }
    // activations: x rows of the k-range (group 1), y segments of the units (group 2)
    for (int c = tid; copy && c < nkb * kFBM * 8; c += kFusedThreads) {
      const int i = c >> 7, row = (c >> 3) & 15, ch = c & 7;
      const int t = record_token(rec, row, cnt, p.max_num_tokens);
      const int kcol = (kb0 + i) * 64 + ch * 8;
      const bool ok = t >= 0 && kcol < p.hidden;
      cp_async_16(sbase + p.off_x + i * 2048 + swz128(row, ch),
                  ok ? p.x + static_cast<long long>(t) * p.x_stride + kcol : p.x, ok);
    }
    cp_async_commit();
    for (int c = tid; copy && c < nun * kFBM * 8; c += kFusedThreads) {
      const int j = c >> 7, row = (c >> 3) & 15, ch = c & 7;
      const int unit = un0 + j;
      const int s = unit_slice(unit);
      const int col = (unit - p.unit_start[s]) * 64 + ch * 8;
      const int t = record_token(rec, row, cnt, p.max_num_tokens);
      const bool ok = t >= 0 && col < p.width[s];
      cp_async_16(sbase + p.off_y + j * 2048 + swz128(row, ch),
                  ok ? p.y + static_cast<long long>(t) * p.y_stride + p.col_off[s] + col : p.y,
                  ok);
    }
    cp_async_commit();

    // ---- shrink over this CTA's k-range
    float acc[NTW][4];
#pragma unroll
    for (int j = 0; j < NTW; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
    cp_async_wait<1>();
    __syncthreads();  // x rows are in
    for (int i = 0; i < nkb; ++i) {
      cta_abort.wait(bar_a + 8 * i, phase);  // (after giving up: garbage in, nothing out)
      const uint32_t sx = sbase + p.off_x + i * 2048;
      const uint32_t sw = sbase + p.off_a + i * SR * 128;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        if ((ks & (WK - 1)) != wk) continue;
        uint32_t af[4];
        ldsm_x4(af, sx + swz128(lane & 15, ks * 2 + (lane >> 4)));
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
            mma_t<F16>(acc[j], af, bf[0], bf[1]);
            if (j + 1 < NTW && j + 1 < nt_cnt) mma_t<F16>(acc[j + 1], af, bf[2], bf[3]);
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < NTW; ++j) {
      if (j < nt_cnt) {
        const int col = (nt0 + j) * 8 + 2 * q;
        *reinterpret_cast<float2*>(red + (wk * kFBM + g) * SR + col) =
            make_float2(acc[j][0], acc[j][1]);
        *reinterpret_cast<float2*>(red + (wk * kFBM + g + 8) * SR + col) =
            make_float2(acc[j][2], acc[j][3]);
      }
    }
    const int e4 = (kFBM * SR) >> 2;
    __syncthreads();
    if (WK > 1) {
      for (int idx = tid; idx < e4; idx += kFusedThreads) {
        float4 v = reinterpret_cast<float4*>(red)[idx];
        for (int w = 1; w < WK; ++w) {
          const float4 o = reinterpret_cast<float4*>(red + w * kFBM * SR)[idx];
          v.x += o.x;
          v.y += o.y;
          v.z += o.z;
          v.w += o.w;
        }
        reinterpret_cast<float4*>(red)[idx] = v;
      }
    }
    cluster_sync_all();
    const bool store_u = !stopped();  // (the A waits are over: one value for all)

    // ---- every CTA sums the C partial tiles in rank order -> full u tile
    for (int idx = tid; idx < e4; idx += kFusedThreads) {
      const uint32_t local = sbase + p.off_red + static_cast<uint32_t>(idx * 16);
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
      const float sc = p.lora_scales != nullptr ? p.scale * p.lora_scales[lora] : p.scale;
      sum = make_float4(sum.x * sc, sum.y * sc, sum.z * sc, sum.w * sc);
      reinterpret_cast<float4*>(utile)[idx] = sum;
      const int e = idx << 2;
      const int row = e / SR;
      const int col = e - row * SR;
      const int t = record_token(rec, row, cnt, p.max_num_tokens);
      if (t >= 0 && (idx % C) == crank && store_u) {
        const int s = col >> p.rank_shift;
        const int r = col - (s << p.rank_shift);
        *reinterpret_cast<float4*>(p.u + (static_cast<long long>(s) * p.max_num_tokens + t) * R + r) =
            sum;
      }
    }
    cp_async_wait<0>();
    __syncthreads();  // u tile complete, y segments are in
    if (nun > 0) cta_abort.wait(bar_b, phase);

    // ---- expand over this CTA's units (warps take units round-robin)
    for (int j = warp; j < nun; j += 4) {
      const int s = unit_slice(un0 + j);
      const float* u0 = utile + g * SR + s * R;
      const float* u1 = utile + (g + 8) * SR + s * R;
      const uint32_t bw = sbase + p.off_b + j * R * 128;
      float eacc[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) eacc[nt][e] = 0.f;
      if (R == 8) {
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
          for (int jj = 0; jj < 4; ++jj) mma_t<F16>(eacc[nt + jj], a, bfr[jj], bfr[jj]);
        }
      } else {
        for (int kk = 0; kk < R / 16; ++kk) {
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
            ldsm_x4_trans(bfr, bw + swz128(kk * 16 + ((mat & 1) << 3) + (lane & 7), nt + (mat >> 1)));
            mma_t<F16>(eacc[nt], ah, bfr[0], bfr[1]);
            mma_t<F16>(eacc[nt], al, bfr[0], bfr[1]);
            mma_t<F16>(eacc[nt + 1], ah, bfr[2], bfr[3]);
            mma_t<F16>(eacc[nt + 1], al, bfr[2], bfr[3]);
          }
        }
      }
      // staged y (swizzled 128-byte rows) + acc -> bf16, in place
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        uint32_t* y0 = reinterpret_cast<uint32_t*>(smem + p.off_y + j * 2048 + swz128(g, nt) + 4 * q);
        uint32_t* y1 =
            reinterpret_cast<uint32_t*>(smem + p.off_y + j * 2048 + swz128(g + 8, nt) + 4 * q);
        const float2 f0 = unpack_t<F16>(*y0);
        const float2 f1 = unpack_t<F16>(*y1);
        *y0 = pack_t<F16>(f0.x + eacc[nt][0], f0.y + eacc[nt][1]);
        *y1 = pack_t<F16>(f1.x + eacc[nt][2], f1.y + eacc[nt][3]);
      }
    }
    __syncthreads();
    // 16-byte stores of the valid rows and columns (none once the CTA has
    // given up; every wait of this item is over, so one value for all)
    const bool store_y = !stopped();
    for (int c = tid; store_y && c < nun * kFBM * 8; c += kFusedThreads) {
      const int j = c >> 7, row = (c >> 3) & 15, ch = c & 7;
      const int unit = un0 + j;
      const int s = unit_slice(unit);
      const int col = (unit - p.unit_start[s]) * 64 + ch * 8;
      const int t = record_token(rec, row, cnt, p.max_num_tokens);
      if (t >= 0 && col < p.width[s])
        *reinterpret_cast<int4*>(p.y + static_cast<long long>(t) * p.y_stride + p.col_off[s] + col) =
            *reinterpret_cast<const int4*>(smem + p.off_y + j * 2048 + swz128(row, ch));
    }
    phase ^= 1u;
    fence_proxy_async();  // generic smem use before the next item's TMA writes
    cluster_sync_all();   // remote reads of red[] are done before it is reused or freed
  }
  if (!waited) {
    // a cluster without a tile still waits: the grid must not complete (and
    // so release the next kernel's wait) before the kernel ahead of it has
    pdl_wait();
    pdl_launch_dependents();
  }
  // after giving up, thread 0's last TMA loads land before the CTA leaves
  // (waiting on one that landed returns at once; each item's cp.async groups
  // were waited for inside the item)
  if (tid == 0 && cta_abort.raised()) {
    if (issued_phase >= 0) {
      for (int i = 0; i < nkb; ++i) mbar_drain(bar_a + 8 * i, issued_phase, p.wait_limit_ns);
      if (nun > 0) mbar_drain(bar_b, issued_phase, p.wait_limit_ns);
    }
    atomicOr(p.status, kStatusTimeout);
  }
}

struct FusedPlan {
  int ok;  // the shape fits the fused kernel
  int cluster, kb_per, warps_n, ntw, wk, kblocks;
  int unit_start[4];
  int units_per_rank;
  int off_a, off_x, off_b, off_y, off_u, off_red, off_rec, off_bar;
  size_t smem;
  long long max_tiles;
};

// Cluster size, per-CTA ranges and the shared-memory plan of the fused kernel
// for a shape; ok = 0 when it does not fit on chip.
static FusedPlan fused_plan(int max_num_tokens, int num_loras, int hidden, const int* widths,
                            int num_slices, int rank, int sms) {
  FusedPlan f = {};
  const int SR = num_slices * rank;
  const int NT = SR / 8;
  f.warps_n = NT <= 8 ? 1 : (NT <= 16 ? 2 : 4);
  f.ntw = (NT + f.warps_n - 1) / f.warps_n;
  f.wk = 4 / f.warps_n;
  if (f.ntw > 8 || sms <= 0) return f;
  f.kblocks = (hidden + 63) / 64;
  f.max_tiles = tile_list_capacity(max_num_tokens, num_loras, 0);
  f.cluster = 1;
  while (f.cluster < 8 && static_cast<long long>(f.cluster) * f.max_tiles < 3LL * sms &&
         f.kblocks >= 4 * f.cluster)
    f.cluster *= 2;
  f.kb_per = (f.kblocks + f.cluster - 1) / f.cluster;
  f.unit_start[0] = 0;
  for (int s = 0; s < 3; ++s)
    f.unit_start[s + 1] = f.unit_start[s] + (s < num_slices ? (widths[s] + 63) / 64 : 0);
  f.units_per_rank = (f.unit_start[3] + f.cluster - 1) / f.cluster;
  if (f.kb_per > kFusedMaxKb || f.units_per_rank > kFusedMaxUnits) return f;
  int off = 0;
  f.off_a = off;   off += f.kb_per * SR * 128;
  f.off_x = off;   off += f.kb_per * kFBM * 128;
  f.off_b = off;   off += f.units_per_rank * rank * 128;
  f.off_y = off;   off += f.units_per_rank * kFBM * 128;
  f.off_u = off;   off += kFBM * SR * 4;
  f.off_red = off; off += f.wk * kFBM * SR * 4;
  f.off_rec = off; off += record_ints(kFBM) * 4;
  off = (off + 15) / 16 * 16;
  f.off_bar = off; off += 8 * (kFusedMaxKb + 1) + 16;  // the barriers, then the abort flag
  f.smem = 1024 + static_cast<size_t>(off);
  f.ok = f.smem <= 200 * 1024;
  return f;
}

// Clusters of the fused kernel the device holds at once.
static int fused_active_clusters_query(const void* fn, int cluster, size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster));
  cfg.blockDim = dim3(kFusedThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = static_cast<unsigned>(cluster);
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// Same, cached per (device, kernel, cluster size, shared memory).
static int fused_active_clusters(const void* fn, int cluster, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, int, size_t>, int> cache;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const auto key = std::make_tuple(dev, fn, cluster, smem);
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  const int n = fused_active_clusters_query(fn, cluster, smem);
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = n;
  return n;
}

static const void* fused_fn(int ntw, bool f16) {
  if (f16)
    return ntw <= 4 ? reinterpret_cast<const void*>(lora_fused_kernel<4, true>)
                    : reinterpret_cast<const void*>(lora_fused_kernel<8, true>);
  return ntw <= 4 ? reinterpret_cast<const void*>(lora_fused_kernel<4, false>)
                  : reinterpret_cast<const void*>(lora_fused_kernel<8, false>);
}

// The fused kernel pays off only when every tile's cluster runs in one wave:
// a cluster holds one tile's whole problem, so a second wave doubles the time.
static bool fused_one_wave(const FusedPlan& f) {
  if (!f.ok) return false;
  const void* fn = fused_fn(f.ntw, false);
  if (ensure_smem_attr(fn, f.smem) != 0) return false;
  return static_cast<long long>(fused_active_clusters(fn, f.cluster, f.smem)) >= f.max_tiles;
}

int fused_fits(int max_num_tokens, int num_loras, int hidden, const int* widths, int num_slices,
               int rank) {
  return fused_one_wave(fused_plan(max_num_tokens, num_loras, hidden, widths, num_slices, rank,
                                   device_sm_count()));
}

// Returns 1 when the fused kernel was launched, 0 when the shape does not fit
// it (the caller then runs the separate kernels), or a negative error code.
int launch_fused(const ShrinkArgs& sa, const ExpandArgs& ea, cudaStream_t stream) {
  if (sa.a_tables[0] != nullptr || ea.b_tables[0] != nullptr) return 0;  // paged: tensor maps only
  const int S = sa.num_slices, R = sa.rank, SR = S * R;
  const int sms = device_sm_count();
  if (sms <= 0) return -6;
  const FusedPlan f = fused_plan(sa.max_num_tokens, sa.num_loras, sa.hidden, ea.slice_width, S, R,
                                 sms);
  if (!fused_one_wave(f)) return 0;
  const int cluster = f.cluster, kb_per = f.kb_per, kblocks = f.kblocks;
  const long long max_tiles = f.max_tiles;
  const size_t smem = f.smem;
  (void)SR;

  FusedParams p;
  for (int s = 0; s < 3; ++s) {
    if (s < S) {
      if (make_weight_tmap(&p.amap[s], sa.lora_a[s], sa.hidden,
                           static_cast<long long>(sa.num_loras) * R, R) != 0 ||
          make_weight_tmap(&p.bmap[s], ea.lora_b[s], ea.slice_width[s],
                           static_cast<long long>(sa.num_loras) * R, R) != 0)
        return -6;
    } else {
      p.amap[s] = p.amap[0];
      p.bmap[s] = p.bmap[0];
    }
  }
  p.x = static_cast<const __nv_bfloat16*>(sa.x);
  p.x_stride = sa.x_row_stride;
  p.hidden = sa.hidden;
  p.kblocks = kblocks;
  p.kb_per_rank = kb_per;
  p.num_slices = S;
  p.rank = R;
  p.rank_shift = __builtin_ctz(static_cast<unsigned>(R));
  p.sr = SR;
  p.scale = sa.scale;
  p.lora_scales = sa.lora_scales;
  p.u = sa.u;
  p.max_num_tokens = sa.max_num_tokens;
  p.y = static_cast<__nv_bfloat16*>(ea.y);
  p.y_stride = ea.y_row_stride;
  int acc_off = 0;
  for (int s = 0; s < 3; ++s) {
    p.width[s] = s < S ? ea.slice_width[s] : 0;
    p.col_off[s] = acc_off;
    acc_off += p.width[s];
  }
  for (int s = 0; s < 4; ++s) p.unit_start[s] = f.unit_start[s];
  p.units_per_rank = f.units_per_rank;
  WsView ws = ws_view(const_cast<void*>(sa.workspace), sa.max_num_tokens, sa.num_loras);
  p.records = ws.lists[0];
  p.num_tiles = ws.num_tiles;
  p.status = ws.status;
  p.tile_capacity = static_cast<int>(max_tiles);
  p.num_loras = sa.num_loras;
  p.warps_n = f.warps_n;
  p.ntw = f.ntw;
  p.off_a = f.off_a;
  p.off_x = f.off_x;
  p.off_b = f.off_b;
  p.off_y = f.off_y;
  p.off_u = f.off_u;
  p.off_red = f.off_red;
  p.off_rec = f.off_rec;
  p.off_bar = f.off_bar;
  p.wait_fault = wait_fault() ? 1 : 0;
  p.wait_limit_ns = p.wait_fault ? kTestWaitLimitNs : kWaitLimitNs;

  const void* fn = fused_fn(f.ntw, sa.f16);
  if (ensure_smem_attr(fn, smem) != 0) return -6;
  int per_sm = occupancy_blocks(fn, kFusedThreads, smem);
  if (per_sm < 1) per_sm = 1;
  long long grid = static_cast<long long>(sms) * per_sm / cluster * cluster;
  if (grid > max_tiles * cluster) grid = max_tiles * cluster;
  if (grid < cluster) grid = cluster;
  const int rc = launch_pdl(fn, dim3(static_cast<unsigned>(grid)), dim3(kFusedThreads), smem,
                            stream, cluster, &p);
  return rc == 0 ? 1 : rc;
}

}  // namespace grg
