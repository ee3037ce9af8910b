// Expand on the 5th-generation tensor cores (tcgen05, accumulators in TMEM)
// for rank 128 on large batches:
//   y[t][off_s + j] = 16-bit( y[t][off_s + j] + sum_r u[s][t][r] * B_s[m[t]][r][j] )
// over the tokens of an unsorted batch ("[V1] LoRA - Add triton kernels for
// V1": the expand loads its tokens through the token -> LoRA grouping and adds
// the rank -> width product into the layer's output; "[Tracking] Multi-LoRA
// Serving", Overview: one launch covers every adapter's segment).
//
// Work: items (128-token tile of one adapter, 128-column block of one slice)
// in tile-major order; each CTA (one per SM, persistent) takes a contiguous
// run of items, so the u tile it holds changes rarely.  Per item one MMA chain
// D[128 x 128] = u_hi * B + u_lo * B (M = 128, N = 128, K = rank, bf16 or
// fp16 operands, fp32 accumulate; u enters as a 16-bit high part plus the
// 16-bit residual, as in the mma.sync expand).
//
// Warp roles (576 threads):
//  - warp 0, producer: per item, into a ring of stages, the B block (two TMA
//    boxes of rank x 64, 128-byte swizzle: the MN-major operand layout);
//  - warp 1, MMA: allocates 256 TMEM columns (two 128-column accumulators),
//    and per item one thread issues the tcgen05.mma chain into the free
//    accumulator and commits it to that accumulator's "full" mbarrier;
//  - warps 2-17, epilogue: four per TMEM lane quarter (a warp may only
//    read its quarter's 32 lanes), each taking 32 of the item's 128 columns;
//    thread = token row.  Each thread loads its own y segment of an item
//    (cp.async, rows padded to 272 bytes so the row-per-thread accesses hit
//    distinct banks) as many items ahead as there are stages; when the
//    (tile, slice) changes the threads load the new u rows, split them into
//    the 16-bit high / residual terms of the swizzled K-major A operand and
//    release the MMA warp; per item they read the accumulator (tcgen05.ld
//    32x32b), add their y segment, round once, free the accumulator and the
//    stage's B block, and store their warp's 32 segments with 16-byte stores
//    (a trace showed four epilogue warps per SM, one per quarter, were the
//    bottleneck: about 2.4 us per item each).
// Before griddepcontrol.wait a CTA only initialises barriers and TMEM and
// reads the tile count (lora_prepare_metadata's output); every copy comes
// after the wait.  Every mbarrier wait is bounded (LORA_STATUS_TIMEOUT).
#include <cstring>

#include "common.cuh"
#include "launch.h"

namespace grg {

constexpr int kTcGroups = 2;                     // epilogue groups (items alternate)
constexpr int kTcCPW = 2;                        // warps per TMEM lane quarter in a group
constexpr int kTcGroupWarps = 4 * kTcCPW;        // each takes 128 / kTcCPW columns
constexpr int kTcEpiWarps = kTcGroups * kTcGroupWarps;
constexpr int kTcThreads = 64 + 32 * kTcEpiWarps;
constexpr int kTcBM = 128;       // tokens per tile (the MMA's M)
constexpr int kTcBN = 128;       // output columns per item (the MMA's N)
constexpr int kTcYPitch = 272;   // staged y row bytes (256 + 16)

struct ExpandTcParams {
  CUtensorMap tmap[3];  // B_s viewed as [L * R][N_s], boxes of R x 64
  const float* u;
  __nv_bfloat16* y;
  long long y_stride;
  int max_num_tokens;
  int w[3];       // slice widths
  int off[3];     // slice column offsets in y
  int cb[4];      // cumulative 128-column blocks per slice
  const int32_t* records;  // tile records of height 128
  const int32_t* num_tiles;
  uint32_t* status;
  int tile_capacity;
  int num_loras;
  int nsb;          // B ring stages (2 * R * 128 bytes each)
  int nsy;          // y stages per epilogue group ([128][kTcYPitch] each)
  int off_u;        // u hi then u lo, R / 64 atoms of [128][128 B] each
  int off_b;
  int off_y;        // [group][nsy] y stages
  int off_tok;      // [group][nsy][kTcCPW][128] token of each row
  int off_bar;      // the barriers, then three ints: the abort flag, the last
                    // item whose B block went out, the last item committed
  // the bounded waits' limit; under the test hook (wait_fault) no copy is
  // issued and the first B barrier is armed with one arrival too many
  unsigned long long wait_limit_ns;
  int wait_fault;
};

template <int RANK, bool F16>
__global__ void __launch_bounds__(kTcThreads, 1)
    lora_expand_tc_kernel(const __grid_constant__ ExpandTcParams p) {
  constexpr int KATOMS = RANK / 64;                  // 64-element K atoms of u
  constexpr uint32_t kUAtomBytes = kTcBM * 128;      // one atom: [128 rows][128 B]
  constexpr uint32_t kUBytes = KATOMS * kUAtomBytes; // u hi (then u lo)
  constexpr uint32_t kBBytes = 2 * RANK * 128;       // two B boxes of [R][128 B]
  constexpr uint32_t kYBytes = kTcBM * kTcYPitch;    // one y stage
  constexpr uint32_t kAccCols = kTcBN;
  // instruction descriptor: D fp32, A / B bf16 (1) or fp16 (0), A K-major,
  // B MN-major, N = 128, M = 128
  constexpr uint32_t kFmt = F16 ? 0u : 1u;
  constexpr uint32_t kIdesc = (1u << 4) | (kFmt << 7) | (kFmt << 10) | (1u << 16) |
                              (static_cast<uint32_t>(kTcBN >> 3) << 17) |
                              (static_cast<uint32_t>(kTcBM >> 4) << 24);

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (sbase - raw);
  const int NSB = p.nsb, NSY = p.nsy;
  const uint32_t full_b = sbase + p.off_bar;         // [NSB]: B block landed (TMA)
  const uint32_t empty_b = full_b + 8 * NSB;         // [NSB]: B block consumed (the MMAs' commit)
  const uint32_t acc_full = empty_b + 8 * NSB;       // [2]: accumulator computed
  const uint32_t acc_empty = acc_full + 16;          // [2]: accumulator read (a group's warps)
  const uint32_t u_ready = acc_empty + 16;           // u tile written (1 arrival)
  __shared__ uint32_t s_taddr;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ntiles = min(max(*p.num_tiles, 0), p.tile_capacity);
  const int cbt = p.cb[3];
  const long long nitems = static_cast<long long>(ntiles) * cbt;
  const long long per = (nitems + gridDim.x - 1) / gridDim.x;
  const long long it0 = static_cast<long long>(blockIdx.x) * per;
  const long long it1 = min(it0 + per, nitems);
  if (it0 >= it1) {
    // no work, but the grid must not complete before the kernel ahead of it
    pdl_wait();
    pdl_launch_dependents();
    return;
  }
  const int nloc = static_cast<int>(it1 - it0);

  // giving up (CtaAbort): no copy, no MMA and no store once a wait has run
  // out, nor under the test hook
  volatile int* const flags = reinterpret_cast<int*>(smem + p.off_bar + 8 * (2 * NSB + 5));
  const CtaAbort cta_abort{flags, p.wait_limit_ns};
  auto stopped = [&]() { return cta_abort.raised() || p.wait_fault != 0; };
  if (tid == 0) {
    flags[0] = 0;
    flags[1] = -1;
    flags[2] = -1;
    for (int i = 0; i < NSB; ++i) {
      // the producer's expect_tx (+ one that never comes: the test hook)
      mbar_init(full_b + 8 * i, 1 + (p.wait_fault && i == 0 ? 1 : 0));
      mbar_init(empty_b + 8 * i, 1);                // the commit of the item's MMAs
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(acc_full + 8 * i, 1);               // the MMA warp's commit
      mbar_init(acc_empty + 8 * i, kTcGroupWarps);  // the warps of the owning group
    }
    mbar_init(u_ready, 1);
    fence_mbar_init();
    for (int s = 0; s < 3; ++s) prefetch_tmap(&p.tmap[s]);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     smem_u32(&s_taddr)),
                 "r"(2 * kAccCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = s_taddr;

  pdl_wait();
  pdl_launch_dependents();

  // The CTA's items in order: (tile, column block), walked one step at a time
  // (no division per item).
  struct Item {
    int tile, cb, s, c0, width, off, group;
    __device__ void set(const ExpandTcParams& q) {
      s = cb >= q.cb[1] ? (cb >= q.cb[2] ? 2 : 1) : 0;
      c0 = (cb - q.cb[s]) * kTcBN;
      width = q.w[s];
      off = q.off[s];
      group = tile * 3 + s;  // u changes with (tile, slice)
    }
    __device__ void next(const ExpandTcParams& q, int cbt_) {
      if (++cb == cbt_) {
        cb = 0;
        ++tile;
      }
      set(q);
    }
  };
  Item first;
  first.tile = static_cast<int>(it0 / cbt);
  first.cb = static_cast<int>(it0 - static_cast<long long>(first.tile) * cbt);
  first.set(p);
  // a tile's adapter and token count, range-checked (lora_prepare_metadata's output)
  auto tile_head = [&](int tile) {
    const int2 h = __ldcg(reinterpret_cast<const int2*>(
        p.records + static_cast<long long>(tile) * record_ints(kTcBM)));
    TileView tv;
    const bool ok = h.x >= 0 && h.x < p.num_loras && h.y > 0 && h.y <= kTcBM;
    tv.lora = ok ? h.x : 0;
    tv.count = ok ? h.y : 0;
    return tv;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    // the B block of each item (two TMA boxes) into the B ring
    int tile = -1, lora = 0;
    Item it = first;
    // L2 prefetch of the B blocks kPf items beyond the ring, so the TMA loads
    // of the ring are served from L2
    constexpr int kPf = 2;
    Item pf = first;
    int pf_tile = -1, pf_lora = 0, pf_k = 0;
    for (int k = 0; k < nloc; ++k, it.next(p, cbt)) {
      const int si = k % NSB;
      if (it.tile != tile) {
        tile = it.tile;
        lora = tile_head(tile).lora;
      }
      for (; pf_k < min(k + NSB + kPf, nloc); ++pf_k, pf.next(p, cbt)) {
        if (pf_k < NSB) continue;  // the ring's first loads go out right away
        if (pf.tile != pf_tile) {
          pf_tile = pf.tile;
          pf_lora = tile_head(pf_tile).lora;
        }
        if (lane == 0 && !stopped()) {
          const int boxes = min(2, (pf.width - pf.c0 + 63) / 64);
          for (int bx = 0; bx < boxes; ++bx)
            tma_prefetch_2d(&p.tmap[pf.s], pf.c0 + 64 * bx, pf_lora * RANK);
        }
      }
      if (k >= NSB) cta_abort.wait(empty_b + 8 * si, ((k / NSB) - 1) & 1);
      if (lane == 0 && !stopped()) {
        flags[1] = k;
        const uint32_t st = sbase + p.off_b + si * kBBytes;
        const int boxes = min(2, (it.width - it.c0 + 63) / 64);
        const uint32_t bar = full_b + 8 * si;
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(boxes * RANK * 128));
        for (int bx = 0; bx < boxes; ++bx)
          tma_load_2d(st + bx * RANK * 128, &p.tmap[it.s], it.c0 + 64 * bx, lora * RANK, bar);
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    // item k into accumulator k & 1 (owned by epilogue group k & 1)
    int group = -1, ngroups = 0;
    Item it = first;
    for (int k = 0; k < nloc; ++k, it.next(p, cbt)) {
      const int si = k % NSB, b = k & 1;
      if (it.group != group) {  // wait for the new u tile
        cta_abort.wait(u_ready, ngroups & 1);
        group = it.group;
        ++ngroups;
      }
      cta_abort.wait(full_b + 8 * si, (k / NSB) & 1);
      if (k >= 2) cta_abort.wait(acc_empty + 8 * b, ((k >> 1) - 1) & 1);
      tc_fence_after();
      if (lane == 0 && !stopped()) {
        const uint32_t d = taddr + b * kAccCols;
        const uint32_t sbm = sbase + p.off_b + si * kBBytes;
        const uint32_t su = sbase + p.off_u;
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // u high part, then the residual
#pragma unroll
          for (int kk = 0; kk < RANK / 16; ++kk) {
            const uint64_t a = umma_desc_sw128(
                su + half * kUBytes + (kk >> 2) * kUAtomBytes + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = umma_desc_sw128(sbm + kk * 16 * 128, RANK * 128, 1024);
            umma_f16(d, a, bd, kIdesc, (half | kk) != 0 ? 1u : 0u);
          }
        }
        umma_commit(acc_full + 8 * b);
        // the B stage is free once the MMAs that read it complete, before
        // the epilogue has read the accumulator
        umma_commit(empty_b + 8 * si);
        flags[2] = k;
      }
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    // Two groups take the items in turn (group g: items g, g + 2, ...), each
    // with its own accumulator and y stages, so two items are in flight.  In a
    // group, warp (quarter, part) owns the 32 token rows of TMEM lane quarter
    // `quarter` (a warp may only read its quarter's lanes) and columns
    // part * CW .. + CW.  Each thread loads its own y segment of its group's
    // items (cp.async, rows padded to 272 bytes so row-per-thread accesses
    // hit distinct banks) NSY items ahead.
    constexpr int CW = kTcBN / kTcCPW;     // columns per warp
    constexpr int CCH = CW / 8;            // 16-byte chunks per row segment
    const int ew = warp - 2;
    const int grp = ew / kTcGroupWarps;    // 0 or 1
    const int quarter = warp & 3;          // TMEM lanes 32 * quarter .. + 31
    const int part = (ew % kTcGroupWarps) >> 2;
    const int row = 32 * quarter + lane;
    const int gtid = (ew % kTcGroupWarps) * 32 + lane;  // 0 .. 255 in the group
    int* tok = reinterpret_cast<int*>(smem + p.off_tok);
    auto tok_at = [&](int j, int r) -> int& {
      return tok[((grp * NSY + j) * kTcCPW + part) * kTcBM + r];
    };
    auto ystage = [&](int j) { return p.off_y + (grp * NSY + j) * kYBytes; };
    // the items come in tile order, so a row's token changes only with the
    // tile: it is loaded (header and row entry at once) only then
    int cur_tile = -1, cur_tok = -1;
    Item ahead = first;  // the next item of this group whose y is requested
    if (grp == 1) ahead.next(p, cbt);
    int ahead_k = grp;
    auto issue_y = [&]() {
      const Item it = ahead;
      const int j = (ahead_k >> 1) % NSY;
      ahead.next(p, cbt);
      ahead.next(p, cbt);
      ahead_k += 2;
      if (it.tile != cur_tile) {
        cur_tile = it.tile;
        const int32_t* rec = p.records + static_cast<long long>(it.tile) * record_ints(kTcBM);
        const TileView tv = tile_head(it.tile);
        const int v = __ldcg(rec + kRecordHeaderInts + row);
        cur_tok = (row < tv.count && v >= 0 && v < p.max_num_tokens) ? v : -1;
      }
      const int t = stopped() ? -1 : cur_tok;  // no copy once the CTA has given up
      tok_at(j, row) = t;
      if (t >= 0) {
        const uint32_t dst = sbase + ystage(j) + row * kTcYPitch + part * CW * 2;
        const int c0 = it.c0 + part * CW;
        const __nv_bfloat16* src = p.y + static_cast<long long>(t) * p.y_stride + it.off + c0;
#pragma unroll
        for (int ch = 0; ch < CCH; ++ch) {
          const bool ok = c0 + ch * 8 < it.width;
          cp_async_16(dst + ch * 16, ok ? src + ch * 8 : p.y, ok);
        }
      }
      cp_async_commit();
    };
    const int mine = (nloc - grp + 1) / 2;  // items of this group
    for (int i = 0; i < min(NSY, mine); ++i) issue_y();
      Item prev = first;                      // item k - 1 (for the u hand-over)
    Item it = first;
    if (grp == 1) {
      prev = first;
      it.next(p, cbt);
    }
    for (int i = 0, k = grp; i < mine; ++i, k += 2) {
      const int j = i % NSY, b = k & 1;
      unsigned char* ys = smem + ystage(j);
      const int t = tok_at(j, row);
      const bool new_u = (k == 0) || it.group != prev.group;
      if (new_u) {
        // the first item of a (tile, slice): once every MMA on the old u tile
        // has completed (item k - 1's accumulator is full: the other group's
        // item), split the new u rows into the swizzled K-major high / residual
        // operands (each part its chunks)
        if (k > 0) cta_abort.wait(acc_full + 8 * ((k - 1) & 1), ((k - 1) >> 1) & 1);
        const float* urow =
            p.u + (static_cast<long long>(it.s) * p.max_num_tokens + (t >= 0 ? t : 0)) * RANK;
        unsigned char* uh = smem + p.off_u;
        constexpr int UCH = RANK / 8 / kTcCPW;  // u chunks (8 elements) per part
#pragma unroll
        for (int cc = 0; cc < UCH; ++cc) {
          const int c = part * UCH + cc;
          float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
          if (t >= 0) {  // u was written by the kernel ahead: read it from L2
            v0 = __ldcg(reinterpret_cast<const float4*>(urow + 8 * c));
            v1 = __ldcg(reinterpret_cast<const float4*>(urow + 8 * c + 4));
          }
          uint4 hi, lo;
          split_t<F16>(v0.x, v0.y, hi.x, lo.x);
          split_t<F16>(v0.z, v0.w, hi.y, lo.y);
          split_t<F16>(v1.x, v1.y, hi.z, lo.z);
          split_t<F16>(v1.z, v1.w, hi.w, lo.w);
          const uint32_t o = (c >> 3) * kUAtomBytes + swz128(row, c & 7);
          *reinterpret_cast<uint4*>(uh + o) = hi;
          *reinterpret_cast<uint4*>(uh + kUBytes + o) = lo;
        }
        fence_proxy_async();  // generic writes before the tensor core reads them
        named_barrier_sync(1 + grp, 32 * kTcGroupWarps);
        if (gtid == 0) mbar_arrive(u_ready);
      }
      // a warp whose 32 rows hold no token only frees the accumulator and B block
      const bool active = __any_sync(0xffffffffu, t >= 0);
      cp_async_wait_dyn(min(NSY, mine - i) - 1);  // my y segment of item k has landed
      cta_abort.wait(acc_full + 8 * b, (k >> 1) & 1);
      tc_fence_after();
      if (!active) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(acc_empty + 8 * b);
        }
        if (i + NSY < mine) issue_y();
        prev = it;
        prev.next(p, cbt);
        it.next(p, cbt);
        it.next(p, cbt);
        continue;
      }
      // accumulator row segment + staged y -> 16-bit, written back into the stage
      unsigned char* yseg = ys + row * kTcYPitch + part * CW * 2;
      const uint32_t tseg = taddr + (static_cast<uint32_t>(32 * quarter) << 16) + b * kAccCols +
                            part * CW;
#pragma unroll
      for (int c32 = 0; c32 < CW / 32; ++c32) {
        float acc[32];
        tmem_ld32(tseg + c32 * 32, acc);
        if (t >= 0) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 yv = *reinterpret_cast<const uint4*>(yseg + (c32 * 4 + q) * 16);
            const float2 f0 = unpack_t<F16>(yv.x), f1 = unpack_t<F16>(yv.y);
            const float2 f2 = unpack_t<F16>(yv.z), f3 = unpack_t<F16>(yv.w);
            const float* a = acc + 8 * q;
            yv.x = pack_t<F16>(f0.x + a[0], f0.y + a[1]);
            yv.y = pack_t<F16>(f1.x + a[2], f1.y + a[3]);
            yv.z = pack_t<F16>(f2.x + a[4], f2.y + a[5]);
            yv.w = pack_t<F16>(f3.x + a[6], f3.y + a[7]);
            *reinterpret_cast<uint4*>(yseg + (c32 * 4 + q) * 16) = yv;
          }
        }
      }
      tc_fence_before();
      __syncwarp();  // the warp's 32 row segments are updated
      if (lane == 0) {
        mbar_arrive(acc_empty + 8 * b);
      }
      // this warp's 32 row segments: 32 / CCH rows per instruction, 16 B per lane
      {
        constexpr int RPI = 32 / CCH;  // rows per instruction
        const int ch = lane % CCH;
        const int col = it.c0 + part * CW + ch * 8;
#pragma unroll
        for (int r0 = 0; r0 < 32; r0 += RPI) {
          const int r = 32 * quarter + r0 + lane / CCH;
          const int tr = tok_at(j, r);
          if (tr >= 0 && col < it.width && !stopped())
            *reinterpret_cast<int4*>(p.y + static_cast<long long>(tr) * p.y_stride + it.off +
                                     col) =
                *reinterpret_cast<const int4*>(ys + r * kTcYPitch + part * CW * 2 + ch * 16);
        }
      }
      __syncwarp();  // the warp's segments of this stage are stored
      if (i + NSY < mine) issue_y();
      prev = it;
      prev.next(p, cbt);  // item k + 1 (the other group's), whose successor is k + 2
      it.next(p, cbt);
      it.next(p, cbt);
    }
    cp_async_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // After giving up (the flag is final here: every wait came before the
  // barrier above), the producer's last TMA loads land and the last MMAs
  // complete (their commit) before the CTA frees its TMEM and leaves; waiting
  // on a copy that landed returns at once.
  const bool gave_up = cta_abort.raised();
  if (gave_up && warp == 0 && lane == 0)
    for (int k = max(0, flags[1] - NSB + 1); k <= flags[1]; ++k)
      mbar_drain(full_b + 8 * (k % NSB), (k / NSB) & 1, p.wait_limit_ns);
  if (warp == 1) {
    if (gave_up) {
      if (lane == 0 && flags[2] >= 0)
        mbar_drain(acc_full + 8 * (flags[2] & 1), (flags[2] >> 1) & 1, p.wait_limit_ns);
      __syncwarp();
    }
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr),
                 "r"(2 * kAccCols)
                 : "memory");
  }
  if (tid == 0 && gave_up) atomicOr(p.status, kStatusTimeout);
}

namespace {
template <int RANK, bool F16>
int run_expand_tc(ExpandTcParams& p, cudaStream_t stream) {
  // rank 64: 3 B stages and 2 y stages per group (216 KB); rank 128: 2 B
  // stages and 1 y stage per group (199 KB) - the u tile takes 64 KB
  p.nsb = RANK == 64 ? 3 : 2;
  p.nsy = RANK == 64 ? 2 : 1;
  p.off_u = 0;
  p.off_b = 2 * (RANK / 64) * kTcBM * 128;
  p.off_y = p.off_b + p.nsb * 2 * RANK * 128;
  p.off_tok = p.off_y + kTcGroups * p.nsy * kTcBM * kTcYPitch;
  p.off_bar = p.off_tok + kTcGroups * p.nsy * kTcCPW * kTcBM * 4;
  const size_t smem = 1024 + static_cast<size_t>(p.off_bar) + 8 * (2 * p.nsb + 5) + 16;
  const void* fn = reinterpret_cast<const void*>(lora_expand_tc_kernel<RANK, F16>);
  if (ensure_smem_attr(fn, smem) != 0) return -6;
  const int sms = device_sm_count();
  if (sms <= 0) return -6;
  long long grid = sms;
  const long long max_items = static_cast<long long>(p.tile_capacity) * p.cb[3];
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  const int rc = launch_pdl(fn, dim3(static_cast<unsigned>(grid)), dim3(kTcThreads), smem, stream,
                            0, &p);
  return rc == 0 ? 1 : rc;
}
}  // namespace

// Rank 128 on large batches.  Measured on GB300 against the mma.sync expand:
// 5000 tokens of 128 adapters, width 4096: 51 us either way; rank 64 (2048
// tokens, Zipf over 32 adapters, two slices of 11008) ran at 101 us against
// 73 us, the thread-per-row epilogue of full 128-row tiles being the limit,
// so rank 64 stays on the mma.sync kernel.
int expand_tc_applies(const ExpandArgs& a) {
  return a.rank == 128 && a.b_tables[0] == nullptr && a.partials == nullptr &&
         a.max_num_tokens > 1024;
}

int launch_expand_tc(const ExpandArgs& a, cudaStream_t stream) {
  if (!expand_tc_applies(a)) return 0;
  ExpandTcParams p;
  memset(&p, 0, sizeof(p));
  int acc = 0, cbs = 0;
  p.cb[0] = 0;
  for (int s = 0; s < 3; ++s) {
    if (s < a.num_slices) {
      p.w[s] = a.slice_width[s];
      p.off[s] = acc;
      acc += p.w[s];
      cbs += (p.w[s] + kTcBN - 1) / kTcBN;
      if (make_weight_tmap(&p.tmap[s], a.lora_b[s], p.w[s],
                           static_cast<long long>(a.num_loras) * a.rank, a.rank) != 0)
        return -6;
    } else {
      p.tmap[s] = p.tmap[0];
    }
    p.cb[s + 1] = cbs;
  }
  p.u = a.u;
  p.y = static_cast<__nv_bfloat16*>(a.y);
  p.y_stride = a.y_row_stride;
  p.max_num_tokens = a.max_num_tokens;
  WsView ws = ws_view(const_cast<void*>(a.workspace), a.max_num_tokens, a.num_loras);
  p.records = ws.lists[tile_index_of(kTcBM)];
  p.num_tiles = ws.num_tiles + tile_index_of(kTcBM);
  p.status = ws.status;
  p.tile_capacity =
      static_cast<int>(tile_list_capacity(a.max_num_tokens, a.num_loras, tile_index_of(kTcBM)));
  p.num_loras = a.num_loras;
  p.wait_fault = wait_fault() ? 1 : 0;
  p.wait_limit_ns = p.wait_fault ? kTestWaitLimitNs : kWaitLimitNs;
  return a.f16 ? run_expand_tc<128, true>(p, stream) : run_expand_tc<128, false>(p, stream);
}

}  // namespace grg
