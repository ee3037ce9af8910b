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
// Warp-specialised pipeline over 64-column k-blocks and a ring of NST stages:
//  - a producer warp fills a stage with the adapter's R x 64 block of every
//    slice (one TMA tile load each: tensor map, 128-byte swizzle) and the BM
//    gathered x rows (16-byte cp.async, zero-filled past the tile's tokens and
//    past H; a run tile's rows as one TMA box); TMA bytes and
//    the lanes' cp.async arrivals complete the stage's "full" mbarrier;
//  - four consumer warps wait on "full", run the tensor-core MMAs (mma.sync
//    m16n8k16, bf16 in, fp32 accumulate) and release the stage on its "empty"
//    mbarrier; no block-wide barrier inside the k-loop.  With S*R = 128 the
//    MMAs run on tcgen05 instead: one thread issues a k-block's four
//    tcgen05.mma (M = the 128 stacked adapter rows, N = the tile's tokens,
//    K = 16; both operands K-major, straight from the ring) into a TMEM
//    accumulator and commits them to the stage's "empty" barrier, and the
//    four warps read the accumulator (transposed) once per tile.
// Before griddepcontrol.wait a CTA reads only its first tile record
// (lora_prepare_metadata's output) and, in the cluster pair of the one call,
// prefetches that tile's first adapter blocks and x rows into L2; every copy
// into shared memory comes after it.  The C partial tiles are summed in rank
// order through distributed shared memory (no atomics, no global scratch),
// scaled once and stored to u.
#include <cstring>

#include "common.cuh"
#include "launch.h"

namespace grg {

constexpr int kConsumerWarps = 4;
constexpr int kShrinkThreads = 32 * (kConsumerWarps + 1);  // + one producer warp
constexpr int kBK = 64;  // bf16 columns per k-block: one 128-byte (swizzled) row chunk

struct ShrinkParams {
  CUtensorMap tmap[3];  // A_s viewed as [L * R][hidden], boxes of R x 64
  CUtensorMap xmap;     // x viewed as [max_num_tokens][hidden], boxes of BM x 64
  const __nv_bfloat16* x;
  long long x_stride;
  int hidden;
  int kblocks;      // ceil(hidden / kBK)
  int num_slices;
  int rank;
  int rank_shift;  // log2(rank)
  int sr;          // num_slices * rank: stacked A rows
  float scale;
  const float* lora_scales;  // per-adapter factors on scale, or null
  float* u;
  int max_num_tokens;
  const int32_t* records;  // tile records of height BM
  const int32_t* num_tiles;
  uint32_t* status;
  int tile_capacity;  // records the list can hold
  int num_loras;
  int warps_n;     // consumer warps splitting the S*R columns (1, 2 or 4)
  int ntw;         // n8 column tiles per consumer warp
  int stage_bytes;
  int rec_offset;  // byte offsets from the 1024-aligned base
  int bar_offset;  // full[NST] then empty[NST]
  float* partials;  // split-K mode: [tile][split][BM][S*R] partial tiles; null otherwise
  int split;        // split-K mode: CTAs per tile (consecutive blocks, no cluster)
  // paged weights: per slice a device table of max_loras addresses of
  // A_s[l] ([R][hidden] bf16); null for stacked weights (tensor maps)
  const uint64_t* a_tab[3];
  int paged;
  int f16;  // fp16 x and A (else bf16)
  // the bounded waits' limit; under the test hook (wait_fault) no copy is
  // issued and the first stage's barrier is armed with one arrival too many
  unsigned long long wait_limit_ns;
  int wait_fault;
  int prefetch;  // L2 prefetches before the dependency wait (the cluster one call)
  int tc;        // S*R = 128: tcgen05 MMAs into TMEM instead of mma.sync
  // k-groups in the one call: the expand is released only when this grid ends
  // (no explicit trigger), not once the last stage is issued
  int release_at_exit;
};

template <int BM, int NTW, int NST, int KS, bool TC, bool PAGED, bool F16>
__global__ void __launch_bounds__(kShrinkThreads, ((BM == 32 && NTW > 4) || NTW > 8) ? 3 : 4)
    lora_shrink_kernel(const __grid_constant__ ShrinkParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // TMA's 128-byte swizzle is laid out on 1024-byte boundaries
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (sbase - raw);
  int32_t* rec = reinterpret_cast<int32_t*>(smem + p.rec_offset);
  const uint32_t full_bar = sbase + p.bar_offset;
  const uint32_t empty_bar = full_bar + 8 * NST;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool producer = warp == kConsumerWarps;
  const int SR = p.sr;
  const int NT = SR >> 3;
  // k-split consumer warps (mma.sync); the tensor-core path accumulates in TMEM
  const int WK = TC ? 1 : kConsumerWarps / p.warps_n;
  const int wn = warp % p.warps_n, wk = warp / p.warps_n;
  const int nt0 = wn * p.ntw;
  const int nt_cnt = min(p.ntw, NT - nt0);
  // at most four n8 column tiles per warp means one column warp group (more
  // than four tiles are split over two or four column groups only from nine
  // tiles up), so WK = 4 and warp wk takes k-step wk of every k-block
  constexpr bool kOneStep = !TC && NTW <= 4;

  // x is read once: a run tile's TMA box of x loads under an L2 evict-first
  // policy, leaving the L2 to the adapter blocks every tile of a LoRA re-reads
  const uint64_t x_pol = l2_evict_first_policy();

  uint32_t cl_size;
  asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(cl_size));
  const bool split_k = p.partials != nullptr;
  const int C = split_k ? p.split : static_cast<int>(cl_size);
  const int crank = split_k ? static_cast<int>(blockIdx.x % p.split)
                            : static_cast<int>(cluster_ctarank());
  const int cluster_id = blockIdx.x / C;
  const int nclusters = gridDim.x / C;
  // A stage holds a k-group: KS consecutive k-blocks (the last group may be
  // shorter), filled under one expect_tx and released once, so the per-stage
  // costs (barrier round trip, issue) are paid once per KS k-blocks.
  // Cluster mode: the CTAs of a tile take its k-groups round-robin (group i
  // of this CTA is crank + i * C), so at any moment they read neighbouring
  // pieces of the same rows (prefill shrink 4 % faster than contiguous
  // halves).  Split-K mode: contiguous ranges of k-groups (decode 1 % faster).
  const int ngroups = (p.kblocks + KS - 1) / KS;
  const int kbp = (ngroups + C - 1) / C;
  const int kb0 = split_k ? crank * kbp : crank;
  const int kstep = split_k ? 1 : C;
  const int nkb = split_k ? max(min(kb0 + kbp, ngroups) - kb0, 0)
                          : (crank < ngroups ? (ngroups - crank + C - 1) / C : 0);
  auto kb_of = [&](int i) { return kb0 + i * kstep; };            // the CTA's i-th k-group
  auto nsub_of = [&](int grp) {  // its k-blocks (a stage of one k-block is always full)
    return KS == 1 ? 1 : min(KS, p.kblocks - grp * KS);
  };
  // stage layout: KS x boxes of [BM][128 B], then KS adapter blocks of [S*R][128 B]
  constexpr int kXSub = BM * 128;
  const int a_off = KS * kXSub, a_sub = SR * 128;

  // giving up (CtaAbort): the flag after the barriers; then (tensor-core
  // path) two more barriers and the TMEM address
  const CtaAbort cta_abort{reinterpret_cast<int*>(smem + p.bar_offset + 2 * 8 * 8), p.wait_limit_ns};
  const uint32_t acc_bar = full_bar + 2 * 8 * 8 + 16, fin_bar = acc_bar + 8;
  uint32_t* const taddr_slot = reinterpret_cast<uint32_t*>(smem + p.bar_offset + 2 * 8 * 8 + 32);
  if (tid == 0) {
    *cta_abort.flag = 0;
    for (int s = 0; s < NST; ++s) {
      // expect_tx + one per thread (+ one that never comes: the test hook)
      mbar_init(full_bar + 8 * s, 1 + kShrinkThreads + (p.wait_fault && s == 0 ? 1 : 0));
      // one arrival per consumer warp, or the commit of the stage's MMAs
      mbar_init(empty_bar + 8 * s, TC ? 1 : kConsumerWarps);
    }
    if constexpr (TC) {
      mbar_init(acc_bar, 1);  // an item's MMAs have completed
      mbar_init(fin_bar, 1);  // every MMA of the CTA has completed (before TMEM is freed)
    }
    fence_mbar_init();
    if constexpr (!PAGED)
      for (int s = 0; s < p.num_slices; ++s) prefetch_tmap(&p.tmap[s]);
  }
  __syncthreads();
  // tensor-core path: 32 TMEM columns hold the tile's partial product,
  // transposed (lane r: row r of the S*R = 128 stacked adapter rows, column
  // t: token t)
  uint32_t taddr = 0;
  if constexpr (TC) {
    if (warp == 0) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                       smem_u32(taddr_slot)),
                   "r"(32)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    taddr = *taddr_slot;
  }
  int n_acc = 0;  // tensor-core path: items whose MMAs were committed to acc_bar

  // the work list is metadata output: safe to read before the dependency wait
  const int ntiles = min(max(*p.num_tiles, 0), p.tile_capacity);
  bool waited = false;
  int kb_global = 0;  // k-groups (stages) processed by this CTA so far (stage phases)
  int issued_g = -1;  // producer lane 0: the last stage whose TMA part went out
  // no copy and no store once the CTA has given up, nor under the test hook
  auto stopped = [&]() { return cta_abort.raised() || p.wait_fault != 0; };

  for (int item = cluster_id; item < ntiles; item += nclusters) {
    load_record<BM>(p.records, item, rec);
    __syncthreads();
    const TileView tv = TileView::of(rec, BM, p.num_loras);
    const int lora = tv.lora, cnt = tv.count;
    const int npro = min(nkb, NST);
    // A full tile whose tokens are consecutive (a request's run of prompt
    // tokens, the usual case in prefill: the grouping keeps each adapter's
    // tokens in ascending order, so first + BM - 1 == last means a run) has
    // its x rows at one place: one TMA box per k-block moves them, in the
    // same swizzled layout the per-row copies give.
    const int t_first = rec[kRecordHeaderInts];
    const bool xbox = cnt == BM && t_first >= 0 &&
                      rec[kRecordHeaderInts + BM - 1] - t_first == BM - 1 &&
                      t_first <= p.max_num_tokens - BM;

    // x chunk (sub-block, row, 16-byte chunk) c of k-group grp -> stage st
    auto x_chunk = [&](int st, int grp, int c) {
      const int j = c / (BM * 8), rc = c - j * (BM * 8);
      const int row = rc >> 3, ch = rc & 7;
      const int t = record_token(rec, row, cnt, p.max_num_tokens);
      const int kcol = (grp * KS + j) * kBK + ch * 8;
      const bool ok = t >= 0 && kcol < p.hidden;
      cp_async_16(sbase + st * p.stage_bytes + j * kXSub + swz128(row, ch),
                  ok ? p.x + static_cast<long long>(t) * p.x_stride + kcol : p.x, ok);
    };
    // the TMA part of k-group grp -> stage st (one thread): the adapter blocks
    // (stacked weights) and the x boxes (a run tile); with neither, a plain
    // arrival stands in for the transaction count
    auto issue_a = [&](int st, int grp) {
      if (stopped()) return;
      issued_g = kb_global + (grp - kb0) / kstep;
      const int nsub = nsub_of(grp);
      const uint32_t bar = full_bar + 8 * st;
      const uint32_t bytes = static_cast<uint32_t>(nsub) *
                             ((PAGED ? 0u : static_cast<uint32_t>(SR * 128)) +
                              (xbox ? static_cast<uint32_t>(kXSub) : 0u));
      if (bytes == 0) {
        mbar_arrive(bar);
        return;
      }
      mbar_arrive_expect_tx(bar, bytes);
      const uint32_t sx = sbase + st * p.stage_bytes;
      for (int j = 0; j < nsub; ++j) {
        const int kcol = (grp * KS + j) * kBK;
        if constexpr (!PAGED)
          for (int s = 0; s < p.num_slices; ++s)
            tma_load_2d(sx + a_off + j * a_sub + s * p.rank * 128, &p.tmap[s], kcol, lora * p.rank,
                        bar);
        if (xbox) tma_load_2d_hint(sx + j * kXSub, &p.xmap, kcol, t_first, bar, x_pol);
      }
    };
    auto wait_empty = [&](int g) {  // stage of global k-block g may be refilled
      const int st = g % NST, use = g / NST;
      if (use > 0) cta_abort.wait(empty_bar + 8 * st, (use - 1) & 1);
    };

    if (!waited) {
      // Before the dependency wait nothing is copied into shared memory: the
      // kernel ahead on the stream may still be writing any input (weights
      // included).  Only L2 prefetches go out - L2 is the GPU's coherence
      // point, so a line prefetched early still reads the final values - of
      // the first stages' adapter blocks and of this CTA's first x columns
      // (cluster mode: the span of the first npro rounds, its rows shared out
      // between the cluster's CTAs); the copies after the wait then hit L2.
      // Only in the cluster pair of the one call: elsewhere the wait returns
      // before the prefetches land (0.5-0.9 us after them on decode) and the
      // copies queue behind them (decode's first stage landed 2.0 instead of
      // 1.6 us after the wait; one call 9.95 -> 9.06 us without them)
      if (producer && npro > 0 && p.prefetch && !p.wait_fault) {  // (the test hook issues nothing)
        if constexpr (!PAGED) {
          if (lane == 0)
            for (int i = 0; i < npro; ++i)
              for (int j = 0; j < nsub_of(kb_of(i)); ++j)
                for (int s = 0; s < p.num_slices; ++s)
                  tma_prefetch_2d(&p.tmap[s], (kb_of(i) * KS + j) * kBK, lora * p.rank);
        }
        if (xbox) {
          if (lane == 0)
            for (int i = 0; i < npro; ++i)
              for (int j = 0; j < nsub_of(kb_of(i)); ++j)
                tma_prefetch_2d(&p.xmap, (kb_of(i) * KS + j) * kBK, t_first);
        } else {
          const int kcol = kb_of(0) * KS * kBK;
          const int r0 = split_k ? lane : crank + C * lane, rstep = split_k ? 32 : 32 * C;
          const int bytes = min(npro * kstep * KS * kBK, p.hidden - (split_k ? kcol : 0)) * 2;
          for (int r = r0; r < cnt; r += rstep) {
            const int t = record_token(rec, r, cnt, p.max_num_tokens);
            if (t >= 0)
              prefetch_l2(p.x + static_cast<long long>(t) * p.x_stride + (split_k ? kcol : 0),
                          bytes);
          }
        }
      }
      pdl_wait();
      // k-group stages release the next kernel only once this CTA's last
      // stage is issued (below), or in the one call only at the grid's end:
      // its CTAs, started early, would load their own inputs while this
      // kernel streams (prefill one call 56.3 -> 48 us with four-k-block
      // stages); single k-block stages release it here
      if constexpr (KS == 1) pdl_launch_dependents();
      waited = true;
    }

    // paged weights: this adapter's A_s (a null or misaligned table entry
    // reads as an all-zero adapter and sets LORA_STATUS_BAD_WEIGHT)
    const __nv_bfloat16* abase[3] = {nullptr, nullptr, nullptr};
    if constexpr (PAGED) {
      for (int s = 0; s < p.num_slices; ++s) {
        const uint64_t a = p.a_tab[s][lora];
        if ((a & 15u) == 0) abase[s] = reinterpret_cast<const __nv_bfloat16*>(a);
        else if (tid == 0) atomicOr(p.status, kStatusBadWeight);
      }
    }
    // paged weights: the adapter rows of k-group grp -> stage st by cp.async,
    // into the layout the TMA boxes would give (chunks first, first + step, ...)
    auto a_chunks = [&](int st, int grp, int first, int step) {
      for (int j = 0; j < nsub_of(grp); ++j) {
        const uint32_t sa = sbase + st * p.stage_bytes + a_off + j * a_sub;
        for (int c = first; c < SR * 8; c += step) {
          const int row = c >> 3, ch = c & 7;
          const int s = row >> p.rank_shift, r = row - (s << p.rank_shift);
          const int kcol = (grp * KS + j) * kBK + ch * 8;
          const __nv_bfloat16* base = abase[s];
          const bool ok = base != nullptr && kcol < p.hidden;
          cp_async_16(sa + swz128(row, ch),
                      ok ? base + static_cast<long long>(r) * p.hidden + kcol : p.x, ok);
        }
      }
    };

    // first stages: the producer's lane 0 issues the TMA part, then every
    // thread issues its share of the x rows (per-row tiles) and arrives on the
    // stage's barrier once its copies have landed
    if (producer && lane == 0) {
      for (int i = 0; i < npro; ++i) {
        wait_empty(kb_global + i);
        issue_a((kb_global + i) % NST, kb_of(i));
      }
    }
    const bool copy = !stopped();  // no copy once the CTA has given up
    if constexpr (PAGED) {
      // every stage is free here (the previous tile ended with a block-wide
      // barrier); each thread's adapter chunks complete with its x chunks
      if (copy)
        for (int i = 0; i < npro; ++i)
          a_chunks((kb_global + i) % NST, kb_of(i), tid, kShrinkThreads);
    }
    for (int i = 0; i < npro && copy; ++i) {
      const int st = (kb_global + i) % NST;
      if (!xbox)
        for (int c = tid; c < nsub_of(kb_of(i)) * BM * 8; c += kShrinkThreads)
          x_chunk(st, kb_of(i), c);
      cp_async_mbar_arrive(full_bar + 8 * st);
    }

    if (producer) {
      // refills: the producer warp alone; lane 0 also arrives for the 128
      // consumer threads so that every phase counts 1 + kShrinkThreads arrivals.
      // Each lane's rows (lane >> 3) + 4 j and chunk lane & 7 are fixed per tile.
      constexpr int XJ = BM / 4;
      const int xch = lane & 7;
      const __nv_bfloat16* xrow[XJ];
#pragma unroll
      for (int j = 0; j < XJ; ++j) {
        const int t = record_token(rec, (lane >> 3) + 4 * j, cnt, p.max_num_tokens);
        xrow[j] = t >= 0 ? p.x + static_cast<long long>(t) * p.x_stride + xch * 8 : nullptr;
      }
      for (int i = npro; i < nkb; ++i) {
        const int g = kb_global + i;
        const int st = g % NST;
        wait_empty(g);  // every lane: the consumers released the stage
        __syncwarp();
        const bool go = !stopped();  // no further copy once the CTA has given up
        if (lane == 0 && go) {
          issue_a(st, kb_of(i));
          mbar_arrive_count(full_bar + 8 * st, kShrinkThreads - 32);
        }
        if constexpr (PAGED)
          if (go) a_chunks(st, kb_of(i), lane, 32);
        if (!xbox && go) {
          const uint32_t sx = sbase + st * p.stage_bytes;
          const int grp = kb_of(i), nsub = nsub_of(grp);
#pragma unroll
          for (int jj = 0; jj < KS; ++jj) {
            if (jj < nsub) {
              const int kb = grp * KS + jj;
              const bool kin = kb * kBK + xch * 8 < p.hidden;
#pragma unroll
              for (int j = 0; j < XJ; ++j) {
                const bool ok = xrow[j] != nullptr && kin;
                cp_async_16(sx + jj * kXSub + swz128((lane >> 3) + 4 * j, xch),
                            ok ? xrow[j] + kb * kBK : p.x, ok);
              }
            }
          }
        }
        if (go) cp_async_mbar_arrive(full_bar + 8 * st);
      }
      if constexpr (KS > 1)
        if (lane == 0 && item + nclusters >= ntiles && !p.release_at_exit)
          pdl_launch_dependents();  // last issue done
    } else if constexpr (TC) {
      // Tensor cores (S*R = 128): per stage one thread issues the k-block's
      // four tcgen05.mma (M = 128 adapter rows, N = BM tokens, K = 16; both
      // operands K-major in the ring's 128-byte-swizzled layout) into the
      // TMEM accumulator and commits them to the stage's "empty" barrier
      constexpr uint32_t kFmt = F16 ? 0u : 1u;
      constexpr uint32_t kIdesc = (1u << 4) | (kFmt << 7) | (kFmt << 10) |
                                  (static_cast<uint32_t>(BM >> 3) << 17) | (8u << 24);
      if (warp == 0) {
        for (int i = 0; i < nkb; ++i) {
          const int g = kb_global + i;
          const int st = g % NST;
          cta_abort.wait(full_bar + 8 * st, (g / NST) & 1);
          tc_fence_after();
          if (lane == 0 && !stopped()) {
            // gathered rows arrive by cp.async (generic proxy); the tensor
            // cores read through the async proxy
            fence_proxy_async();
            const uint32_t stg = sbase + st * p.stage_bytes;
            const int nsub = nsub_of(kb_of(i));
            for (int jj = 0; jj < KS; ++jj) {
              if (jj >= nsub) break;
              const uint32_t sx = stg + jj * kXSub, sw = stg + a_off + jj * a_sub;
#pragma unroll
              for (int ks = 0; ks < kBK / 16; ++ks)
                umma_f16(taddr, umma_desc_sw128(sw + ks * 32, 16, 1024),
                         umma_desc_sw128(sx + ks * 32, 16, 1024), kIdesc,
                         (i | jj | ks) != 0 ? 1u : 0u);
            }
            umma_commit(empty_bar + 8 * st);  // the stage is free once these complete
          }
          __syncwarp();
        }
        if (lane == 0 && nkb > 0 && !stopped()) umma_commit(acc_bar);
        __syncwarp();
      }
      // every consumer warp: lane r = 32 warp + lane of the accumulator holds
      // row r of S*R for the tile's tokens (columns) -> red[token][r]
      const bool have = nkb > 0 && cta_abort.wait(acc_bar, n_acc & 1);
      if (nkb > 0) ++n_acc;
      tc_fence_after();
      named_barrier_sync(1, 32 * kConsumerWarps);  // every MMA on the ring has completed
      float d[32];
      tmem_ld32(taddr + (static_cast<uint32_t>(32 * warp) << 16), d);
      tc_fence_before();
      float* red = reinterpret_cast<float*>(smem);
      const int r = 32 * warp + lane;
#pragma unroll
      for (int t = 0; t < BM; ++t) red[t * SR + r] = have ? d[t] : 0.f;
    } else {
      float acc[BM / 16][NTW][4];
#pragma unroll
      for (int mi = 0; mi < BM / 16; ++mi)
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[mi][j][e] = 0.f;

      for (int i = 0; i < nkb; ++i) {
        const int g = kb_global + i;
        const int st = g % NST;
        cta_abort.wait(full_bar + 8 * st, (g / NST) & 1);  // (after giving up: garbage in, nothing out)
        const uint32_t stg = sbase + st * p.stage_bytes;
        const int nsub = nsub_of(kb_of(i));
#pragma unroll
        for (int jj = 0; jj < KS; ++jj) {
          if (jj >= nsub) break;
          const uint32_t sx = stg + jj * kXSub;       // x rows of k-block jj of the group
          const uint32_t sw = stg + a_off + jj * a_sub;  // its adapter rows
#pragma unroll
          for (int kk = 0; kk < (kOneStep ? 1 : kBK / 16); ++kk) {
            const int ks = kOneStep ? wk : kk;
            if (!kOneStep && (ks & (WK - 1)) != wk) continue;
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
                  mma_t<F16>(acc[mi][j], af[mi], bf[0], bf[1]);
                  if (j + 1 < NTW && j + 1 < nt_cnt)
                    mma_t<F16>(acc[mi][j + 1], af[mi], bf[2], bf[3]);
                }
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar + 8 * st);
      }
      named_barrier_sync(1, 32 * kConsumerWarps);  // every consumer warp is done with the ring
      // partial tile -> red[wk][row][col] (aliases the ring)
      float* red = reinterpret_cast<float*>(smem);
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
    kb_global += nkb;
    __syncthreads();  // all partials are in red[] (the producer has issued everything)
    const bool store = !stopped();  // (every wait of this item is over: one value for all)

    // sum the k-split warps into red[0]
    float* red = reinterpret_cast<float*>(smem);
    const int e4 = (BM * SR) >> 2;
    if (split_k) {
      // split-K mode: this CTA's partial tile (its warps summed in the same
      // order) goes to the workspace; the expand sums the split in rank order
      float4* dst = reinterpret_cast<float4*>(p.partials) +
                    (static_cast<long long>(item) * C + crank) * e4;
      for (int idx = tid; idx < e4 && store; idx += kShrinkThreads) {
        float4 v = reinterpret_cast<float4*>(red)[idx];
        for (int w = 1; w < WK; ++w) {
          const float4 o = reinterpret_cast<float4*>(red + w * BM * SR)[idx];
          v.x += o.x;
          v.y += o.y;
          v.z += o.z;
          v.w += o.w;
        }
        dst[idx] = v;
      }
      fence_proxy_async();  // generic use of the ring before the next item's TMA writes
      __syncthreads();
      continue;
    }
    if (WK > 1) {
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
    for (int idx = crank * kShrinkThreads + tid; idx < e4 && store; idx += C * kShrinkThreads) {
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
      const float c = p.lora_scales != nullptr ? p.scale * p.lora_scales[lora] : p.scale;
      *reinterpret_cast<float4*>(dst) = make_float4(sum.x * c, sum.y * c, sum.z * c, sum.w * c);
    }
    fence_proxy_async();  // generic use of the ring before the next item's TMA writes
    cluster_sync_all();
  }
  if (!waited) {
    // a CTA without a tile still waits: the grid must not complete (and so
    // release the next kernel's wait) before the kernel ahead of it has
    pdl_wait();
    pdl_launch_dependents();
  }
  // Leave with no copy in flight: each thread's cp.async, and after giving
  // up the producer's last TMA loads (a stage is refilled only once its
  // previous load was consumed, so only the last NST can be pending; waiting
  // on one that landed returns at once).  The flag is final here: the last
  // wait of the last item came before that item's block-wide barrier.
  cp_async_wait<0>();
  if (cta_abort.raised()) {
    if (producer && lane == 0)
      for (int g = max(0, issued_g - NST + 1); g <= issued_g; ++g)
        mbar_drain(full_bar + 8 * (g % NST), (g / NST) & 1, p.wait_limit_ns);
    if (tid == 0) atomicOr(p.status, kStatusTimeout);
  }
  if constexpr (TC) {
    // the MMA thread's last commit covers every MMA it issued (also after
    // giving up): TMEM is freed only once they have all completed
    if (tid == 0) {
      umma_commit(fin_bar);
      mbar_drain(fin_bar, 0, p.wait_limit_ns);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(32)
                   : "memory");
  }
}

template <int BM, int NTW, int NST, int KS>
static int run_shrink(const ShrinkParams& prm, int cluster, size_t smem, cudaStream_t stream,
                      long long max_tiles) {
  // fp16 inputs come with stacked weights only
  if (prm.paged && prm.f16) return -3;
  const void* fn = nullptr;
  if (prm.tc) {
    // S*R = 128 (8 column tiles per warp): the tensor-core path
    // (stacked weights only)
    if constexpr (NTW == 8) {
      if (prm.paged) return -6;
      fn = prm.f16 ? reinterpret_cast<const void*>(lora_shrink_kernel<BM, NTW, NST, KS, true, false, true>)
                   : reinterpret_cast<const void*>(
                         lora_shrink_kernel<BM, NTW, NST, KS, true, false, false>);
    } else {
      return -6;
    }
  } else {
    fn = prm.paged ? reinterpret_cast<const void*>(lora_shrink_kernel<BM, NTW, NST, KS, false, true, false>)
         : prm.f16 ? reinterpret_cast<const void*>(lora_shrink_kernel<BM, NTW, NST, KS, false, false, true>)
                   : reinterpret_cast<const void*>(
                         lora_shrink_kernel<BM, NTW, NST, KS, false, false, false>);
  }
  if (ensure_smem_attr(fn, smem) != 0) return -6;
  const int sms = device_sm_count();
  if (sms <= 0) return -6;
  // the occupancy calculator reports one CTA per SM for the tcgen05
  // instantiations (three fit by registers and shared memory, and run: the
  // down_proj_graph shrink takes 73.7 us with three, 139.7 us with one)
  int per_sm = prm.tc ? resident_blocks(fn, kShrinkThreads, smem)
                      : occupancy_blocks(fn, kShrinkThreads, smem);
  if (per_sm < 1) per_sm = 1;
  long long grid = static_cast<long long>(sms) * per_sm / cluster * cluster;
  const long long useful = max_tiles * cluster;
  if (grid > useful) grid = useful;
  if (grid < cluster) grid = cluster;
  ShrinkParams p = prm;
  // split-K mode: a tile's CTAs are consecutive blocks, no cluster launch
  return launch_pdl(fn, dim3(static_cast<unsigned>(grid)), dim3(kShrinkThreads), smem, stream,
                    p.partials != nullptr ? 0 : cluster, &p);
}

static int shrink_tile_rows(const ShrinkArgs& a) {
  return (a.num_slices * a.rank >= 192 || a.max_num_tokens <= 1024) ? 16 : 32;
}

int shrink_split(const ShrinkArgs& a, bool split_k) {
  const int SR = a.num_slices * a.rank;
  const int BM = shrink_tile_rows(a);
  const int kblocks = (a.hidden + kBK - 1) / kBK;
  const long long max_tiles = tile_list_capacity(a.max_num_tokens, a.num_loras, tile_index_of(BM));
  const int sms = device_sm_count();
  // split the hidden dimension over a cluster until ~3 CTAs per SM have work
  // (the rank-order reduction reads BM x S*R floats from every cluster CTA:
  // wide tiles keep the cluster small).  Split-K mode has no cluster: on a
  // decode batch (256 tokens, hidden 4096, three 4096-wide slices of rank 8)
  // a split of 16 ran a layer 9 % faster than 8.
  const int max_cluster =
      split_k ? (SR <= 64 ? split_k_max(a.rank) : 8) : (SR <= 64 ? 8 : (SR <= 128 ? 4 : 2));
  int cluster = 1;
  while (cluster < max_cluster && static_cast<long long>(cluster) * max_tiles < 3LL * sms &&
         kblocks >= 8 * cluster)
    cluster *= 2;
  return cluster;
}

int launch_shrink(const ShrinkArgs& a, cudaStream_t stream) {
  const int SR = a.num_slices * a.rank;
  const int NT = SR / 8;
  const int warps_n = NT <= 8 ? 1 : (NT <= 16 ? 2 : 4);
  const int ntw = (NT + warps_n - 1) / warps_n;
  const int WK = kConsumerWarps / warps_n;
  const int BM = shrink_tile_rows(a);
  const int kblocks = (a.hidden + kBK - 1) / kBK;
  const long long max_tiles = tile_list_capacity(a.max_num_tokens, a.num_loras, tile_index_of(BM));
  const int cluster = shrink_split(a, a.partials != nullptr);
  if (a.partials != nullptr && BM != 16) return -3;
  // k-blocks per stage: narrow adapters on 32-token tiles (prefill: S*R <=
  // 32, 6 KB per k-block) spend more on the per-stage round trip and issue
  // than on the bytes (a per-CTA trace: ~1100 cycles per stage, at any ring
  // depth), so a stage takes four k-blocks there (prefill shrink 21.3 ->
  // 18.3 us).  In the one call the expand's CTAs, which would start beside the
  // shrink's under programmatic launch, find no room next to the 50 KB CTAs
  // this needs (some started only as others finished: prefill one call 48.9
  // -> 54.1 us), so there the expand is released only when the shrink's grid
  // ends (one call 47.9 -> 46.9 us against one-k-block stages)
  const int ks = (a.partials == nullptr && BM == 32 && SR <= 32 && kblocks >= 32) ? 4 : 1;
  const int kb_per = ((kblocks + ks - 1) / ks + cluster - 1) / cluster;  // stages per CTA
  // Ring depth: a short k-range (up to 8 blocks) keeps all of it in flight;
  // long ranges prefer occupancy (smaller rings, more CTAs per SM, and room
  // for the next kernel's CTAs to start under programmatic launch).  Up to 4
  // blocks, 4 stages hold the whole range and leave the room to the expand
  // CTAs that start under this kernel (decode layer 8.72 -> 8.49 us)
  const int stage = ks * (BM + SR) * 128;  // a multiple of 1024: BM and S*R are multiples of 8
  int nst;
  if (ks == 4)
    nst = 2;  // two stages of up to 32 KB keep four CTAs per SM
  else if (kb_per <= 4 && ntw <= 8)
    nst = 4;
  else if (kb_per <= 8)
    nst = (8 * stage <= 64 * 1024 && ntw <= 8) ? 8 : (4 * stage <= 96 * 1024 ? 4 : 2);
  else if (SR == 128)
    // three stages keep three CTAs per SM: on down_proj_graph (11008 wide)
    // every tile's cluster is resident at once (shrink 96.4 -> 88.5 us, two
    // stages had too few bytes in flight, four left too few clusters for the
    // tiles); on mlp_gate_up the smaller CTAs let the expand's start beside
    // them (one call 103.6 -> 91.8 us)
    nst = 3;
  else
    nst = 4 * stage > 96 * 1024 ? 2 : 4;

  ShrinkParams p;
  memset(&p, 0, sizeof(p));
  p.paged = a.a_tables[0] != nullptr;
  p.f16 = a.f16 ? 1 : 0;
  p.prefetch = (a.expand_follows && a.partials == nullptr) ? 1 : 0;
  // the tensor-core path for S*R = 128 with stacked weights; paged weights
  // (adapter rows gathered by cp.async) keep the mma.sync consumers, which
  // were faster there (down_proj_graph paged shrink 160.6 vs 281.9 us)
  p.tc = (SR == 128 && a.partials == nullptr && !p.paged) ? 1 : 0;
  p.wait_fault = wait_fault() ? 1 : 0;
  p.release_at_exit = (ks > 1 && a.expand_follows) ? 1 : 0;
  p.wait_limit_ns = p.wait_fault ? kTestWaitLimitNs : kWaitLimitNs;
  for (int s = 0; s < 3; ++s) {
    p.a_tab[s] = s < a.num_slices ? a.a_tables[s] : a.a_tables[0];
    if (p.paged) continue;
    if (s < a.num_slices) {
      if (make_weight_tmap(&p.tmap[s], a.lora_a[s], a.hidden,
                           static_cast<long long>(a.num_loras) * a.rank, a.rank) != 0)
        return -6;
    } else {
      p.tmap[s] = p.tmap[0];
    }
  }
  // x as a [max_num_tokens][hidden] matrix of row stride x_row_stride, in
  // boxes of BM rows x 64 columns (run tiles)
  if (make_tmap_2d(&p.xmap, a.x, a.hidden, a.max_num_tokens, a.x_row_stride * 2, BM) != 0)
    return -6;
  p.x = static_cast<const __nv_bfloat16*>(a.x);
  p.x_stride = a.x_row_stride;
  p.hidden = a.hidden;
  p.kblocks = kblocks;
  p.num_slices = a.num_slices;
  p.rank = a.rank;
  p.rank_shift = __builtin_ctz(static_cast<unsigned>(a.rank));
  p.sr = SR;
  p.scale = a.scale;
  p.lora_scales = a.lora_scales;
  p.u = a.u;
  p.max_num_tokens = a.max_num_tokens;
  WsView ws = ws_view(const_cast<void*>(a.workspace), a.max_num_tokens, a.num_loras);
  p.records = ws.lists[tile_index_of(BM)];
  p.num_tiles = ws.num_tiles + tile_index_of(BM);
  p.status = ws.status;
  p.tile_capacity = static_cast<int>(max_tiles);
  p.num_loras = a.num_loras;
  p.partials = a.partials;
  p.split = cluster;
  p.warps_n = warps_n;
  p.ntw = ntw;
  p.stage_bytes = stage;
  const int ring = nst * stage;
  const int red = WK * BM * SR * 4;
  const int body = ((ring > red ? ring : red) + 127) / 128 * 128;
  p.rec_offset = body;
  p.bar_offset = body + record_ints(BM) * 4;
  // + the flag (16 bytes), the tensor-core path's two barriers and TMEM address (32)
  const size_t smem = 1024 + static_cast<size_t>(p.bar_offset) + 2 * 8 * 8 + 48;

  // Every (tile height, column tiles per warp, ring depth, k-blocks per stage)
  // the rules above can produce has its own instantiation; the shared-memory
  // plan was sized for exactly that ring, so any other combination is refused,
  // never rounded.
  using Run = int (*)(const ShrinkParams&, int, size_t, cudaStream_t, long long);
  Run run = nullptr;
  const int ntw_t = ntw <= 4 ? 4 : (ntw <= 8 ? 8 : 12);
  if (ntw_t <= 4 && WK != kConsumerWarps) return -6;  // those kernels take one k-step per warp
  if (BM == 16 && ntw_t == 4 && ks == 1 && nst == 8) run = run_shrink<16, 4, 8, 1>;
  if (BM == 16 && ntw_t == 4 && ks == 1 && nst == 4) run = run_shrink<16, 4, 4, 1>;
  if (BM == 16 && ntw_t == 8 && ks == 1 && nst == 8) run = run_shrink<16, 8, 8, 1>;
  if (BM == 16 && ntw_t == 8 && ks == 1 && nst == 4) run = run_shrink<16, 8, 4, 1>;
  if (BM == 16 && ntw_t == 8 && ks == 1 && nst == 2) run = run_shrink<16, 8, 2, 1>;
  if (BM == 16 && ntw_t == 8 && ks == 1 && nst == 3) run = run_shrink<16, 8, 3, 1>;
  if (BM == 16 && ntw_t == 12 && ks == 1 && nst == 4) run = run_shrink<16, 12, 4, 1>;
  if (BM == 16 && ntw_t == 12 && ks == 1 && nst == 2) run = run_shrink<16, 12, 2, 1>;
  if (BM == 32 && ntw_t == 4 && ks == 1 && nst == 8) run = run_shrink<32, 4, 8, 1>;
  if (BM == 32 && ntw_t == 4 && ks == 1 && nst == 4) run = run_shrink<32, 4, 4, 1>;
  if (BM == 32 && ntw_t == 8 && ks == 1 && nst == 8) run = run_shrink<32, 8, 8, 1>;
  if (BM == 32 && ntw_t == 8 && ks == 1 && nst == 4) run = run_shrink<32, 8, 4, 1>;
  if (BM == 32 && ntw_t == 8 && ks == 1 && nst == 2) run = run_shrink<32, 8, 2, 1>;
  if (BM == 32 && ntw_t == 8 && ks == 1 && nst == 3) run = run_shrink<32, 8, 3, 1>;
  if (BM == 32 && ntw_t == 4 && ks == 4 && nst == 2) run = run_shrink<32, 4, 2, 4>;
  // one or two column tiles (S*R <= 16) on 32-token tiles: the accumulators
  // of two tiles only (prefill lora_shrink 16.7 -> 16.5 us)
  if (BM == 32 && ntw <= 2 && ks == 4 && nst == 2) run = run_shrink<32, 2, 2, 4>;
  if (BM == 32 && ntw <= 2 && ks == 1 && nst == 4) run = run_shrink<32, 2, 4, 1>;
  if (run == nullptr) return -6;
  return run(p, cluster, smem, stream, max_tiles);
}

}  // namespace grg
