// Expand on the 5th-generation tensor cores (tcgen05, accumulators in TMEM)
// for ranks 64 and 128 on large batches:
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
// Warp roles (192 threads):
//  - warp 0, producer: per item, into a ring of stages, the tile record, the
//    B block (two TMA boxes of rank x 64, 128-byte swizzle: the MN-major
//    operand layout) and the gathered y rows (cp.async into rows padded to
//    272 bytes, so the epilogue's row-per-thread accesses hit distinct banks);
//  - warp 1, MMA: allocates 256 TMEM columns (two 128-column accumulators),
//    and per item one thread issues the tcgen05.mma chain into the free
//    accumulator and commits it to that accumulator's "full" mbarrier;
//  - warps 2-5, epilogue: thread = token row (TMEM lane); when the (tile,
//    slice) changes they load the new u rows, split them into the 16-bit
//    high / residual terms of the swizzled K-major A operand and release the
//    MMA warp; per item they read the accumulator (tcgen05.ld 32x32b), add
//    the staged y, round once, write the row back to the stage, free the
//    accumulator and store their 32 rows with 16-byte stores.
// Before griddepcontrol.wait a CTA only initialises barriers and TMEM and
// reads the tile count (lora_prepare_metadata's output); every copy comes
// after the wait.  Every mbarrier wait is bounded (LORA_STATUS_TIMEOUT).
#include <cstring>

#include "common.cuh"
#include "launch.h"

namespace grg {

constexpr int kTcThreads = 192;
constexpr int kTcBM = 128;       // tokens per tile (the MMA's M)
constexpr int kTcBN = 128;       // output columns per item (the MMA's N)
constexpr int kTcYPitch = 272;   // staged y row bytes (256 + 16)
constexpr int kTcRecBytes = record_ints(kTcBM) * 4;

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
  int nstages;
  int stage_bytes;  // B region (2 * R * 128) + y region (128 * kTcYPitch) + record
  int off_u;        // u hi then u lo, R / 64 atoms of [128][128 B] each
  int off_st;
  int off_bar;
};

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

template <int RANK, bool F16>
__global__ void __launch_bounds__(kTcThreads, 1)
    lora_expand_tc_kernel(const __grid_constant__ ExpandTcParams p) {
  constexpr int KATOMS = RANK / 64;                  // 64-element K atoms of u
  constexpr uint32_t kUAtomBytes = kTcBM * 128;      // one atom: [128 rows][128 B]
  constexpr uint32_t kUBytes = KATOMS * kUAtomBytes; // u hi (then u lo)
  constexpr uint32_t kBBytes = 2 * RANK * 128;       // two B boxes of [R][128 B]
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
  const int NS = p.nstages;
  const uint32_t full_b = sbase + p.off_bar;         // [NS]: B block landed (TMA)
  const uint32_t full_y = full_b + 8 * NS;           // [NS]: record + y rows landed
  const uint32_t empty = full_y + 8 * NS;            // [NS]: stage free (4 epilogue warps)
  const uint32_t acc_full = empty + 8 * NS;          // [2]: accumulator computed
  const uint32_t acc_empty = acc_full + 16;          // [2]: accumulator read (4 warps)
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

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full_b + 8 * i, 1);   // the producer's expect_tx
      mbar_init(full_y + 8 * i, 32);  // one cp.async arrival per producer lane
      mbar_init(empty + 8 * i, 4);    // one per epilogue warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(acc_full + 8 * i, 1);   // the MMA warp's commit
      mbar_init(acc_empty + 8 * i, 4);  // one per epilogue warp
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

  // item k of this CTA -> tile, slice, first column inside the slice
  struct Item {
    int tile, s, c0, width, off, group;
  };
  auto item_of = [&](int k) {
    const long long item = it0 + k;
    Item it;
    it.tile = static_cast<int>(item / cbt);
    int cb = static_cast<int>(item - static_cast<long long>(it.tile) * cbt);
    it.s = cb >= p.cb[1] ? (cb >= p.cb[2] ? 2 : 1) : 0;
    it.c0 = (cb - p.cb[it.s]) * kTcBN;
    it.width = p.w[it.s];
    it.off = p.off[it.s];
    it.group = it.tile * 3 + it.s;  // u changes with (tile, slice)
    return it;
  };
  bool timed_out = false;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    for (int k = 0; k < nloc; ++k) {
      const int si = k % NS;
      if (k >= NS && !mbar_wait(empty + 8 * si, ((k / NS) - 1) & 1)) timed_out = true;
      const Item it = item_of(k);
      const uint32_t st = sbase + p.off_st + si * p.stage_bytes;
      unsigned char* stp = smem + p.off_st + si * p.stage_bytes;
      int32_t* rec = reinterpret_cast<int32_t*>(stp + kBBytes + kTcBM * kTcYPitch);
      // the tile record (its token ids) travels with the stage
      const int4* src =
          reinterpret_cast<const int4*>(p.records + static_cast<long long>(it.tile) * record_ints(kTcBM));
      for (int i = lane; i < kTcRecBytes / 16; i += 32) reinterpret_cast<int4*>(rec)[i] = __ldcg(src + i);
      __syncwarp();
      const TileView tv = TileView::of(rec, kTcBM, p.num_loras);
      if (lane == 0) {
        const int boxes = min(2, (it.width - it.c0 + 63) / 64);
        const uint32_t bar = full_b + 8 * si;
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(boxes * RANK * 128));
        for (int b = 0; b < boxes; ++b)
          tma_load_2d(st + b * RANK * 128, &p.tmap[it.s], it.c0 + 64 * b, tv.lora * RANK, bar);
      }
      // y rows of the tile's tokens: two rows per instruction, 16 lanes x 16 B each
      const uint32_t sy = st + kBBytes;
      const int ch = lane & 15;
      const int col = it.c0 + ch * 8;
      for (int r = lane >> 4; r < tv.count; r += 2) {
        const int t = record_token(rec, r, tv.count, p.max_num_tokens);
        const bool ok = t >= 0 && col < it.width;
        cp_async_16(sy + r * kTcYPitch + ch * 16,
                    ok ? p.y + static_cast<long long>(t) * p.y_stride + it.off + col : p.y, ok);
      }
      cp_async_mbar_arrive(full_y + 8 * si);
    }
    cp_async_wait<0>();  // leave with no copy of this warp in flight
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    int group = -1, ngroups = 0;
    for (int k = 0; k < nloc; ++k) {
      const int si = k % NS, b = k & 1;
      const Item it = item_of(k);
      if (it.group != group) {  // wait for the epilogue warps' new u tile
        if (!mbar_wait(u_ready, ngroups & 1)) timed_out = true;
        group = it.group;
        ++ngroups;
      }
      if (!mbar_wait(full_b + 8 * si, (k / NS) & 1)) timed_out = true;
      if (k >= 2 && !mbar_wait(acc_empty + 8 * b, ((k >> 1) - 1) & 1)) timed_out = true;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t d = taddr + b * kAccCols;
        const uint32_t sbm = sbase + p.off_st + si * p.stage_bytes;
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
      }
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;          // TMEM lanes 32 * quarter .. + 31
    const int row = 32 * quarter + lane;   // this thread's token row in the tile
    const int etid = tid - 64;             // 0..127
    int group = -1;
    for (int k = 0; k < nloc; ++k) {
      const int si = k % NS, b = k & 1;
      const Item it = item_of(k);
      unsigned char* stp = smem + p.off_st + si * p.stage_bytes;
      const int32_t* rec = reinterpret_cast<const int32_t*>(stp + kBBytes + kTcBM * kTcYPitch);
      if (!mbar_wait(full_y + 8 * si, (k / NS) & 1)) timed_out = true;
      const TileView tv = TileView::of(rec, kTcBM, p.num_loras);
      const int t = record_token(rec, row, tv.count, p.max_num_tokens);
      if (it.group != group) {
        // a new (tile, slice): every MMA on the old u tile has completed (the
        // previous item's accumulator was read); split the new u rows into the
        // swizzled K-major high / residual operands
        group = it.group;
        const float* urow =
            p.u + (static_cast<long long>(it.s) * p.max_num_tokens + (t >= 0 ? t : 0)) * RANK;
        unsigned char* uh = smem + p.off_u;
#pragma unroll 4
        for (int c = 0; c < RANK / 8; ++c) {  // 8 elements = one 16-byte chunk
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
        named_barrier_sync(1, 128);
        if (etid == 0) mbar_arrive(u_ready);
      }
      if (!mbar_wait(acc_full + 8 * b, (k >> 1) & 1)) timed_out = true;
      tc_fence_after();
      // accumulator row + staged y -> 16-bit, written back into the stage
      unsigned char* yrow = stp + kBBytes + row * kTcYPitch;
      const uint32_t trow = taddr + (static_cast<uint32_t>(32 * quarter) << 16) + b * kAccCols;
#pragma unroll
      for (int c32 = 0; c32 < kTcBN / 32; ++c32) {
        float acc[32];
        tmem_ld32(trow + c32 * 32, acc);
        if (t >= 0) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 yv = *reinterpret_cast<const uint4*>(yrow + (c32 * 4 + q) * 16);
            const float2 f0 = unpack_t<F16>(yv.x), f1 = unpack_t<F16>(yv.y);
            const float2 f2 = unpack_t<F16>(yv.z), f3 = unpack_t<F16>(yv.w);
            const float* a = acc + 8 * q;
            yv.x = pack_t<F16>(f0.x + a[0], f0.y + a[1]);
            yv.y = pack_t<F16>(f1.x + a[2], f1.y + a[3]);
            yv.z = pack_t<F16>(f2.x + a[4], f2.y + a[5]);
            yv.w = pack_t<F16>(f3.x + a[6], f3.y + a[7]);
            *reinterpret_cast<uint4*>(yrow + (c32 * 4 + q) * 16) = yv;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + 8 * b);
      // this warp's 32 rows: two rows per instruction, 16 lanes x 16 B each
      const int ch = lane & 15;
      const int col = it.c0 + ch * 8;
      for (int r = 32 * quarter + (lane >> 4); r < 32 * quarter + 32; r += 2) {
        const int tr = record_token(rec, r, tv.count, p.max_num_tokens);
        if (tr >= 0 && col < it.width)
          *reinterpret_cast<int4*>(p.y + static_cast<long long>(tr) * p.y_stride + it.off + col) =
              *reinterpret_cast<const int4*>(stp + kBBytes + r * kTcYPitch + ch * 16);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + 8 * si);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr),
                 "r"(2 * kAccCols)
                 : "memory");
  if (timed_out) atomicOr(p.status, kStatusTimeout);
}

namespace {
template <int RANK>
constexpr int tc_stages() {
  return RANK == 64 ? 3 : 2;
}
template <int RANK, bool F16>
int run_expand_tc(ExpandTcParams& p, cudaStream_t stream) {
  constexpr int NS = tc_stages<RANK>();
  const int stage = 2 * RANK * 128 + kTcBM * kTcYPitch + kTcRecBytes;
  p.nstages = NS;
  p.stage_bytes = (stage + 1023) / 1024 * 1024;
  p.off_u = 0;
  p.off_st = 2 * (RANK / 64) * kTcBM * 128;
  p.off_bar = p.off_st + NS * p.stage_bytes;
  const size_t smem = 1024 + static_cast<size_t>(p.off_bar) + 8 * (3 * NS + 5);
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

int expand_tc_applies(const ExpandArgs& a) {
  return (a.rank == 64 || a.rank == 128) && a.b_tables[0] == nullptr && a.partials == nullptr &&
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
  if (a.rank == 64) return a.f16 ? run_expand_tc<64, true>(p, stream) : run_expand_tc<64, false>(p, stream);
  return a.f16 ? run_expand_tc<128, true>(p, stream) : run_expand_tc<128, false>(p, stream);
}

}  // namespace grg
