// Expand: y[t][off_s + j] = bf16(y[t][off_s + j] + sum_r u[s][t][r] * B_s[m[t]][r][j])
// over the tokens of an unsorted batch ("[V1] LoRA - Add triton kernels for
// V1": the expand kernel loads its tokens through the same token -> LoRA
// grouping as the shrink and adds the rank -> width product into the output).
//
// Work decomposition (fixed grid, graph-safe): an item is one tile of up to BM
// tokens of one LoRA (a record of the metadata kernel's list) times one block
// of 256 output columns of one slice.  CTAs walk the items with a stride of
// the grid.
//
// Data movement, per item, into a shared-memory stage:
//  - the adapter block B_s[lora][0:R][block] as four R x 64 TMA tile loads
//    (tensor map, 128-byte swizzle), completing on the stage's mbarrier;
//  - the gathered 256-column segments of y and the gathered rows of u with
//    16-byte cp.async (rows padded so the epilogue hits distinct banks).
// Ranks up to 32 use two stages, so the next item's copies fly while the
// current one is computed (one in partial mode, whose CTAs have one or two
// items).  Before griddepcontrol.wait only the first tile
// records are copied and the first B block and y rows are prefetched into
// L2; B, u and y are copied after it - except directly after this library's
// shrink in the one-call paths, where B and y load before the wait.
//
// Compute: four warps, 64 columns each; per 16-token m-tile a warp runs
// mma.sync m16n8k16 (bf16 operands, fp32 accumulate) of the u rows against B.
// u enters the tensor cores as two bf16 terms (high part + residual), so about
// 16 significant bits of the fp32 u reach the product.  The sum is added to
// the staged y in fp32, rounded once to bf16, written back into the stage and
// stored with coalesced 16-byte stores.
#include <cstring>

#include "common.cuh"
#include "launch.h"

namespace grg {

constexpr int kExpandThreads = 128;
constexpr int kEN = 256;     // output columns per item (64 per warp)
constexpr int kYPitch = 528; // staged y row bytes (512 + 16)

struct ExpandParams {
  CUtensorMap tmap[3];  // B_s viewed as [L * R][N_s], boxes of R x 64
  const float* u;        // u to read, or (partial mode) u to write
  const float* partials; // partial mode: the shrink's [tile][split][BM][S*R] partial tiles
  int split;
  int sr;
  float scale;
  const float* lora_scales;  // partial mode: per-adapter factors on scale, or null
  int y_early;  // y may be read before the dependency wait (the one-call path)
  // paged weights: per slice a device table of max_loras addresses of B_s[l]
  // ([R][N_s] bf16), loaded by cp.async; null for stacked weights (tensor maps)
  const uint64_t* b_tab[3];
  int paged;
  int f16;  // fp16 y and B (u is split into fp16 terms), else bf16
  int max_num_tokens;
  int w0, w1, w2;        // slice widths
  int off0, off1, off2;  // slice column offsets in y
  int cb0, cb1;          // column blocks of slices 0 and 1
  int cb_total;          // column blocks over all slices
  __nv_bfloat16* y;
  long long y_stride;
  const int32_t* records;  // tile records of height BM
  const int32_t* num_tiles;
  uint32_t* status;
  int tile_capacity;
  int num_loras;
  // the bounded waits' limit; under the test hook (wait_fault) no copy is
  // issued and the first record barrier is armed with one arrival too many
  unsigned long long wait_limit_ns;
  int wait_fault;
};


template <int BM, int RANK, int NS, bool PARTIAL>
struct ExpandLayout {
  static constexpr int kUPitch = RANK * 4 + 16;  // staged u row bytes
  static constexpr int kB = 0;                   // 4 boxes of [RANK][128 B], 1024-aligned
  static constexpr int kY = 4 * RANK * 128;
  static constexpr int kU = kY + BM * kYPitch;
  static constexpr int kP = kU + BM * kUPitch;   // partial mode: [split][BM][RANK] fp32
  static constexpr int kPBytes = PARTIAL ? split_k_max(RANK) * BM * RANK * 4 : 0;
  static constexpr int kStage = (kP + kPBytes + 1023) / 1024 * 1024;
  static constexpr int kRecSlots = NS + 1;
  static constexpr int kRecBytes = record_ints(BM) * 4;
  static constexpr int kRec = NS * kStage;
  static constexpr int kBar = kRec + kRecSlots * kRecBytes;  // NS stage + kRecSlots record barriers
  // then the CtaAbort flag and thread 0's last record / B block issued
  static constexpr int kFlag = kBar + 8 * (NS + kRecSlots);
  static constexpr int kSmem = 1024 + kFlag + 16;
};

// Stage count per rank (more stages cost occupancy: two stages at three
// CTAs per SM beat three or four stages at two).
template <int RANK>
constexpr int expand_stages() {
  return RANK <= 32 ? 2 : 1;
}

template <int BM, int RANK, int NS, bool PARTIAL, bool PAGED, bool F16>
__global__ void __launch_bounds__(kExpandThreads, RANK >= 64 ? 2 : 4)
    lora_expand_kernel(const __grid_constant__ ExpandParams p) {
  using Lay = ExpandLayout<BM, RANK, NS, PARTIAL>;
  constexpr int MT = BM / 16;
  constexpr int RS = Lay::kRecSlots;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // TMA's 128-byte swizzle is laid out on 1024-byte boundaries
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (sbase - raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  const uint32_t stage_bar = sbase + Lay::kBar;
  const uint32_t rec_bar = stage_bar + 8 * NS;

  // the work list is metadata output: safe to read before the dependency wait
  const int ntiles = min(max(*p.num_tiles, 0), p.tile_capacity);
  const int nitems = ntiles * p.cb_total;
  // items in tile-major order with a stride of the grid: at any moment the
  // CTAs cover every column block of a band of tiles, so whole y rows are
  // read and written together (DRAM page locality)
  const int G = gridDim.x;
  const int nloc = static_cast<int>(blockIdx.x) < nitems
                       ? (nitems - 1 - static_cast<int>(blockIdx.x)) / G + 1
                       : 0;
  if (nloc <= 0) {
    // this CTA writes nothing, but still waits: the grid must not complete
    // (and so release the next kernel's wait) before the kernel ahead of it has
    pdl_wait();
    pdl_launch_dependents();
    return;
  }

  // giving up (CtaAbort): no copy and no store once a wait has run out, nor
  // under the test hook
  volatile int* const flags = reinterpret_cast<int*>(smem + Lay::kFlag);
  const CtaAbort cta_abort{flags, p.wait_limit_ns};
  auto stopped = [&]() { return cta_abort.raised() || p.wait_fault != 0; };
  if (tid == 0) {
    flags[0] = 0;
    flags[1] = -1;  // the last item whose record went out
    flags[2] = -1;  // the last item whose B block went out
    for (int s = 0; s < NS + RS; ++s)
      mbar_init(stage_bar + 8 * s, 1 + (p.wait_fault && s == NS ? 1 : 0));
    fence_mbar_init();
    if constexpr (!PAGED)
      for (int s = 0; s < 3; ++s) prefetch_tmap(&p.tmap[s]);
  }
  __syncthreads();

  auto rec_of = [&](int k) {
    return reinterpret_cast<int32_t*>(smem + Lay::kRec + (k % RS) * Lay::kRecBytes);
  };
  struct Item {
    int s, width, off, c0, tile;
  };
  auto item_of = [&](int k) {
    const int item = static_cast<int>(blockIdx.x) + k * G;
    const int tl = item / p.cb_total;
    int cb = item - tl * p.cb_total;
    Item it;
    it.tile = tl;
    it.s = 0;
    if (cb >= p.cb0) {
      cb -= p.cb0;
      it.s = 1;
      if (cb >= p.cb1) {
        cb -= p.cb1;
        it.s = 2;
      }
    }
    it.width = it.s == 0 ? p.w0 : (it.s == 1 ? p.w1 : p.w2);
    it.off = it.s == 0 ? p.off0 : (it.s == 1 ? p.off1 : p.off2);
    it.c0 = cb * kEN;
    return it;
  };
  // tile record of item k -> its slot (thread 0, bulk copy on the slot's barrier)
  auto issue_rec = [&](int k) {
    if (stopped()) return;
    flags[1] = k;
    const uint32_t bar = rec_bar + 8 * (k % RS);
    mbar_arrive_expect_tx(bar, Lay::kRecBytes);
    bulk_g2s(smem_u32(rec_of(k)),
             p.records + static_cast<long long>(item_of(k).tile) * record_ints(BM), Lay::kRecBytes,
             bar);
  };
  auto wait_rec = [&](int k) { cta_abort.wait(rec_bar + 8 * (k % RS), (k / RS) & 1); };
  // B block of item k -> stage (thread 0): boxes starting past the slice are skipped
  auto issue_b = [&](int k) {
    if (stopped()) return;
    flags[2] = k;
    const Item it = item_of(k);
    const TileView tv = TileView::of(rec_of(k), BM, p.num_loras);
    const uint32_t st = sbase + (k % NS) * Lay::kStage;
    const uint32_t bar = stage_bar + 8 * (k % NS);
    if constexpr (PAGED) {  // the rows come with the item's cp.async group (issue_y)
      mbar_arrive(bar);
      return;
    }
    const int boxes = min(4, (it.width - it.c0 + 63) / 64);
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(boxes * RANK * 128));
    for (int b = 0; b < boxes; ++b)
      tma_load_2d(st + Lay::kB + b * RANK * 128, &p.tmap[it.s], it.c0 + 64 * b, tv.lora * RANK,
                  bar);
  };
  // gathered y segments of item k -> stage (every thread; part of the next group)
  auto issue_y = [&](int k) {
    const Item it = item_of(k);
    const int32_t* rec = rec_of(k);
    const TileView tv = TileView::of(rec, BM, p.num_loras);
    const uint32_t st = sbase + (k % NS) * Lay::kStage;
    const int ych = tid & 31;
    const int col = it.c0 + ych * 8;
    if (stopped()) return;  // (the group is closed by issue_u all the same)
#pragma unroll
    for (int i = 0; i < BM / 4; ++i) {
      const int row = (tid >> 5) + 4 * i;
      const int t = record_token(rec, row, tv.count, p.max_num_tokens);
      const bool ok = t >= 0 && col < it.width;
      cp_async_16(st + Lay::kY + row * kYPitch + ych * 16,
                  ok ? p.y + static_cast<long long>(t) * p.y_stride + it.off + col : p.y, ok);
    }
    if constexpr (PAGED) {
      // paged weights: B_s[lora] rows of the item's 256 columns, into the
      // layout of the four TMA boxes (a null or misaligned table entry reads
      // as an all-zero adapter and sets LORA_STATUS_BAD_WEIGHT)
      const uint64_t a = p.b_tab[it.s][tv.lora];
      const __nv_bfloat16* base =
          (a & 15u) == 0 ? reinterpret_cast<const __nv_bfloat16*>(a) : nullptr;
      if (a != 0 && base == nullptr && tid == 0) atomicOr(p.status, kStatusBadWeight);
      for (int c = tid; c < 4 * RANK * 8; c += kExpandThreads) {
        const int box = c / (RANK * 8), rem = c - box * RANK * 8;
        const int r = rem >> 3, ch = rem & 7;
        const int bcol = it.c0 + box * 64 + ch * 8;
        const bool ok = base != nullptr && bcol < it.width;
        cp_async_16(st + Lay::kB + box * RANK * 128 + swz128(r, ch),
                    ok ? base + static_cast<long long>(r) * it.width + bcol : p.y, ok);
      }
    }
  };
  // rows of u (or of the split's partial tiles) of item k -> stage, closing the group
  auto issue_u = [&](int k) {
    const Item it = item_of(k);
    const int32_t* rec = rec_of(k);
    const TileView tv = TileView::of(rec, BM, p.num_loras);
    const uint32_t st = sbase + (k % NS) * Lay::kStage;
    constexpr int UCH = RANK / 4;  // 16-byte chunks per u row
    if (stopped()) {
      cp_async_commit();  // an empty group: the count of groups stays the same
      return;
    }
    if constexpr (PARTIAL) {
      // the split's partial rows of this slice (the valid rows only)
      const float* base = p.partials + static_cast<long long>(it.tile) * p.split * BM * p.sr +
                          it.s * RANK;
      for (int c = tid; c < p.split * BM * UCH; c += kExpandThreads) {
        const int ch = c % UCH;
        const int row = (c / UCH) % BM;
        const int part = c / (UCH * BM);
        if (row < tv.count)
          cp_async_16(st + Lay::kP + ((part * BM + row) * RANK + ch * 4) * 4,
                      base + (static_cast<long long>(part) * BM + row) * p.sr + ch * 4, true);
      }
    } else {
      for (int c = tid; c < BM * UCH; c += kExpandThreads) {
        const int row = c / UCH, ch = c - row * UCH;
        const int t = record_token(rec, row, tv.count, p.max_num_tokens);
        const bool ok = t >= 0;
        cp_async_16(st + Lay::kU + row * Lay::kUPitch + ch * 16,
                    ok ? p.u + (static_cast<long long>(it.s) * p.max_num_tokens + t) * RANK + ch * 4
                       : p.u,
                    ok);
      }
    }
    cp_async_commit();
  };
  auto issue_uy = [&](int k) {
    issue_y(k);
    issue_u(k);
  };

  // prologue: the records of the first items (lora_prepare_metadata's output,
  // visible before it released its dependents) before the dependency wait
  const int npro = min(nloc, NS);
  if (tid == 0) {
    for (int k = 0; k < min(nloc, RS); ++k) issue_rec(k);
  }
  if (p.y_early) {
    // Directly after this library's shrink of the same call: that kernel
    // writes neither B nor y and released this launch only after its own
    // dependency wait, so every kernel before it has completed.  The first
    // items' B blocks and y segments load before the wait, u / partials after
    for (int k = 0; k < npro; ++k) {
      wait_rec(k);
      if (tid == 0) issue_b(k);
      issue_y(k);
    }
    pdl_wait();
    pdl_launch_dependents();
    for (int k = 0; k < npro; ++k) issue_u(k);
  } else {
    // The kernel ahead on the stream may still be writing any input: before
    // the wait only L2 prefetches (L2 is the coherence point, so the copies
    // after the wait read the final values) of item 0's B block and y rows
    wait_rec(0);
    if (!stopped()) {  // (no prefetch from a record that did not arrive)
      const Item it = item_of(0);
      const int32_t* rec = rec_of(0);
      const TileView tv = TileView::of(rec, BM, p.num_loras);
      if constexpr (!PAGED) {
        if (tid == 0) {
          const int boxes = min(4, (it.width - it.c0 + 63) / 64);
          for (int b = 0; b < boxes; ++b)
            tma_prefetch_2d(&p.tmap[it.s], it.c0 + 64 * b, tv.lora * RANK);
        }
      }
      const int bytes = min(kEN, it.width - it.c0) * 2;
      for (int r = tid; r < tv.count; r += kExpandThreads) {
        const int t = record_token(rec, r, tv.count, p.max_num_tokens);
        if (t >= 0)
          prefetch_l2(p.y + static_cast<long long>(t) * p.y_stride + it.off + it.c0, bytes);
      }
    }
    pdl_wait();
    pdl_launch_dependents();
    if (tid == 0) issue_b(0);
    issue_uy(0);
    for (int k = 1; k < npro; ++k) {
      wait_rec(k);
      if (tid == 0) issue_b(k);
      issue_uy(k);
    }
  }

  for (int k = 0; k < nloc; ++k) {
    // item k's copies: its cp.async group (later groups may stay pending) and its B block
    cp_async_wait_dyn(min(NS, nloc - k) - 1);
    __syncthreads();
    cta_abort.wait(stage_bar + 8 * (k % NS), (k / NS) & 1);  // (after giving up: garbage in)

    const Item it = item_of(k);
    const int32_t* rec = rec_of(k);
    const TileView tv = TileView::of(rec, BM, p.num_loras);
    unsigned char* stp = smem + (k % NS) * Lay::kStage;
    const uint32_t st = sbase + (k % NS) * Lay::kStage;

    if constexpr (PARTIAL) {
      // u = scale * (sum of the split's partial tiles in rank order), the same
      // operations in the same order as the shrink's cluster reduction; the
      // slice's first column block also stores its rows of u
      constexpr int UCH = RANK / 4;
      const float* P = reinterpret_cast<const float*>(stp + Lay::kP);
      for (int e = tid; e < BM * UCH; e += kExpandThreads) {
        const int row = e / UCH, ch = e - row * UCH;
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row < tv.count) {
          sum = *reinterpret_cast<const float4*>(P + row * RANK + ch * 4);
          for (int c = 1; c < p.split; ++c) {
            const float4 v = *reinterpret_cast<const float4*>(P + (c * BM + row) * RANK + ch * 4);
            sum.x += v.x;
            sum.y += v.y;
            sum.z += v.z;
            sum.w += v.w;
          }
          const float c = p.lora_scales != nullptr ? p.scale * p.lora_scales[tv.lora] : p.scale;
          sum = make_float4(sum.x * c, sum.y * c, sum.z * c, sum.w * c);
        }
        *reinterpret_cast<float4*>(stp + Lay::kU + row * Lay::kUPitch + ch * 16) = sum;
        const int t = record_token(rec, row, tv.count, p.max_num_tokens);
        if (it.c0 == 0 && t >= 0 && !stopped())
          *reinterpret_cast<float4*>(const_cast<float*>(p.u) +
                                     (static_cast<long long>(it.s) * p.max_num_tokens + t) * RANK +
                                     ch * 4) = sum;
      }
      __syncthreads();
    }

#pragma unroll
    for (int mi = 0; mi < MT; ++mi) {
      if (mi * 16 >= tv.count) break;
      float acc[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
      const float* u0 =
          reinterpret_cast<const float*>(stp + Lay::kU + (mi * 16 + g) * Lay::kUPitch);
      const float* u1 =
          reinterpret_cast<const float*>(stp + Lay::kU + (mi * 16 + g + 8) * Lay::kUPitch);
      // B box of this warp's 64 columns
      const uint32_t bw = st + Lay::kB + warp * RANK * 128;

      if constexpr (RANK == 8) {
        // k = 0..7 carry the high parts, k = 8..15 the residuals; B rows repeat.
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
          for (int j = 0; j < 4; ++j) mma_t<F16>(acc[nt + j], a, bfr[j], bfr[j]);
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
            mma_t<F16>(acc[nt], ah, bfr[0], bfr[1]);
            mma_t<F16>(acc[nt], al, bfr[0], bfr[1]);
            mma_t<F16>(acc[nt + 1], ah, bfr[2], bfr[3]);
            mma_t<F16>(acc[nt + 1], al, bfr[2], bfr[3]);
          }
        }
      }

      // staged y + acc -> bf16, written back into the stage
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int cbyte = (warp * 64 + nt * 8 + 2 * q) * 2;
        uint32_t* y0 =
            reinterpret_cast<uint32_t*>(stp + Lay::kY + (mi * 16 + g) * kYPitch + cbyte);
        uint32_t* y1 =
            reinterpret_cast<uint32_t*>(stp + Lay::kY + (mi * 16 + g + 8) * kYPitch + cbyte);
        const float2 f0 = unpack_t<F16>(*y0);
        const float2 f1 = unpack_t<F16>(*y1);
        *y0 = pack_t<F16>(f0.x + acc[nt][0], f0.y + acc[nt][1]);
        *y1 = pack_t<F16>(f1.x + acc[nt][2], f1.y + acc[nt][3]);
      }
    }
    __syncthreads();  // the updated stage is complete

    // One stage (ranks of 64 and more): the stage's B block is free now (the
    // MMAs are done), its y rows only once they are stored, so the next
    // item's B block goes out before the stores (mlp_gate_up expand 72.9 ->
    // 72.3 us; prefetching its y rows into L2 here as well cost 9 us)
    constexpr bool kEarlyB = NS == 1 && !PARTIAL && !PAGED;
    if constexpr (kEarlyB) {
      if (k + 1 < nloc) {
        wait_rec(k + 1);
        if (tid == 0) issue_b(k + 1);
      }
    }

    // coalesced 16-byte stores of the valid rows and columns (none once the
    // CTA has given up; every wait of this item is over, so one value for all)
    if (!stopped()) {
      const int ych = tid & 31;
      const int col = it.c0 + ych * 8;
#pragma unroll
      for (int i = 0; i < BM / 4; ++i) {
        const int row = (tid >> 5) + 4 * i;
        const int t = record_token(rec, row, tv.count, p.max_num_tokens);
        if (t >= 0 && col < it.width)
          *reinterpret_cast<int4*>(p.y + static_cast<long long>(t) * p.y_stride + it.off + col) =
              *reinterpret_cast<const int4*>(stp + Lay::kY + row * kYPitch + ych * 16);
      }
    }
    __syncthreads();  // stage k % NS and record slot k % RS are free again

    // refill: item k + NS into the stage just freed, record k + RS into its slot
    if (k + NS < nloc) {
      if constexpr (!kEarlyB) {
        wait_rec(k + NS);
        if (tid == 0) issue_b(k + NS);
      }
      issue_uy(k + NS);
    }
    if (tid == 0 && k + RS < nloc) issue_rec(k + RS);
  }
  // Leave with no copy in flight: the cp.async groups, and after giving up
  // thread 0's last bulk copies (a slot is refilled only once its previous
  // contents were consumed, so only the last NS B blocks and RS records can be
  // pending; waiting on one that landed returns at once).  The flag is final
  // here: the last item's waits came before its block-wide barriers.
  cp_async_wait<0>();
  if (tid == 0 && cta_abort.raised()) {
    for (int k = max(0, flags[2] - NS + 1); k <= flags[2]; ++k)
      mbar_drain(stage_bar + 8 * (k % NS), (k / NS) & 1, p.wait_limit_ns);
    for (int k = max(0, flags[1] - RS + 1); k <= flags[1]; ++k)
      mbar_drain(rec_bar + 8 * (k % RS), (k / RS) & 1, p.wait_limit_ns);
    atomicOr(p.status, kStatusTimeout);
  }
}

template <int BM, int RANK, bool PARTIAL>
static int run_expand(const ExpandParams& prm, cudaStream_t stream, long long max_items) {
  // partial mode (the split-K pair of decode-sized batches): a CTA has one or
  // two items, so a second stage is rarely used and only keeps CTAs from
  // starting beside the shrink's (decode expand 6.26 -> 5.0 us with one)
  constexpr int NS = PARTIAL ? 1 : expand_stages<RANK>();
  // fp16 inputs come with stacked weights only
  if (prm.paged && prm.f16) return -3;
  const void* fn =
      prm.paged
          ? reinterpret_cast<const void*>(lora_expand_kernel<BM, RANK, NS, PARTIAL, true, false>)
      : prm.f16
          ? reinterpret_cast<const void*>(lora_expand_kernel<BM, RANK, NS, PARTIAL, false, true>)
          : reinterpret_cast<const void*>(lora_expand_kernel<BM, RANK, NS, PARTIAL, false, false>);
  const size_t smem = ExpandLayout<BM, RANK, NS, PARTIAL>::kSmem;
  if (ensure_smem_attr(fn, smem) != 0) return -6;
  const int sms = device_sm_count();
  if (sms <= 0) return -6;
  int per_sm = occupancy_blocks(fn, kExpandThreads, smem);
  if (per_sm < 1) per_sm = 1;
  long long grid = static_cast<long long>(sms) * per_sm;
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  ExpandParams p = prm;
  return launch_pdl(fn, dim3(static_cast<unsigned>(grid)), dim3(kExpandThreads), smem, stream, 0,
                    &p);
}

template <int BM>
static int launch_expand_bm(const ExpandArgs& a, cudaStream_t stream) {
  ExpandParams p;
  memset(&p, 0, sizeof(p));
  p.paged = a.b_tables[0] != nullptr;
  p.f16 = a.f16 ? 1 : 0;
  for (int s = 0; s < 3; ++s) p.b_tab[s] = s < a.num_slices ? a.b_tables[s] : a.b_tables[0];
  p.u = a.u;
  p.partials = a.partials;
  p.split = a.split;
  p.sr = a.num_slices * a.rank;
  p.scale = a.scale;
  p.lora_scales = a.lora_scales;
  p.y_early = a.y_early ? 1 : 0;
  p.max_num_tokens = a.max_num_tokens;
  int w[3] = {0, 0, 0}, off[3] = {0, 0, 0}, cbs[3] = {0, 0, 0};
  int acc_off = 0, cb_total = 0;
  for (int s = 0; s < 3; ++s) {
    if (s < a.num_slices) {
      w[s] = a.slice_width[s];
      off[s] = acc_off;
      acc_off += w[s];
      cbs[s] = (w[s] + kEN - 1) / kEN;
      cb_total += cbs[s];
      if (!p.paged && make_weight_tmap(&p.tmap[s], a.lora_b[s], w[s],
                                       static_cast<long long>(a.num_loras) * a.rank, a.rank) != 0)
        return -6;
    } else {
      p.tmap[s] = p.tmap[0];
    }
  }
  p.w0 = w[0];
  p.w1 = w[1];
  p.w2 = w[2];
  p.off0 = off[0];
  p.off1 = off[1];
  p.off2 = off[2];
  p.cb0 = cbs[0];
  p.cb1 = cbs[1];
  p.cb_total = cb_total;
  p.y = static_cast<__nv_bfloat16*>(a.y);
  p.y_stride = a.y_row_stride;
  WsView ws = ws_view(const_cast<void*>(a.workspace), a.max_num_tokens, a.num_loras);
  p.records = ws.lists[tile_index_of(BM)];
  p.num_tiles = ws.num_tiles + tile_index_of(BM);
  p.status = ws.status;
  p.tile_capacity =
      static_cast<int>(tile_list_capacity(a.max_num_tokens, a.num_loras, tile_index_of(BM)));
  p.num_loras = a.num_loras;
  p.wait_fault = wait_fault() ? 1 : 0;
  p.wait_limit_ns = p.wait_fault ? kTestWaitLimitNs : kWaitLimitNs;
  const long long max_items = static_cast<long long>(p.tile_capacity) * cb_total;
  if (a.partials != nullptr) {
    // partial mode: 16-token tiles and ranks up to 32 only
    if constexpr (BM == 16) {
      if (a.split < 1 || a.split > split_k_max(a.rank)) return -3;
      switch (a.rank) {
        case 8: return run_expand<BM, 8, true>(p, stream, max_items);
        case 16: return run_expand<BM, 16, true>(p, stream, max_items);
        case 32: return run_expand<BM, 32, true>(p, stream, max_items);
        default: return -3;
      }
    }
    return -3;
  }
  switch (a.rank) {
    case 8: return run_expand<BM, 8, false>(p, stream, max_items);
    case 16: return run_expand<BM, 16, false>(p, stream, max_items);
    case 32: return run_expand<BM, 32, false>(p, stream, max_items);
    case 64: return run_expand<BM, 64, false>(p, stream, max_items);
    case 128: return run_expand<BM, 128, false>(p, stream, max_items);
    default: return -3;
  }
}

int launch_expand(const ExpandArgs& a, cudaStream_t stream) {
  // rank 128 on large batches: the tcgen05 kernel (128-token tiles)
  const int tc = launch_expand_tc(a, stream);
  if (tc < 0) return tc;
  if (tc == 1) return 0;
  // small batches: 16-token tiles give more, shorter items (latency); large
  // batches: 32-token tiles amortise each item's B block over more rows
  if (a.max_num_tokens <= 1024) return launch_expand_bm<16>(a, stream);
  if (a.partials != nullptr) return -3;
  return launch_expand_bm<32>(a, stream);
}

}  // namespace grg
