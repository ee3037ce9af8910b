// Expand: y[t][off_s + j] = bf16(y[t][off_s + j] + sum_r u[s][t][r] * B_s[m[t]][r][j])
// over the tokens of an unsorted batch ("[V1] LoRA - Add triton kernels for
// V1": the expand kernel loads its tokens through the same token -> LoRA
// grouping as the shrink and adds the rank -> width product into the output).
//
// Work decomposition (fixed grid, graph-safe): an item is one tile of up to BM
// tokens of one LoRA (from the metadata kernel's list) times one block of 256
// output columns of one slice.  A CTA of four warps copies the adapter's
// B_s[lora][0:R][block] into XOR-swizzled shared memory with cp.async, while
// every warp issues the loads of its 64 columns of the gathered y rows into
// registers; then each warp runs tensor-core MMAs (m16n8k16, fp32 accumulate)
// of the 16-token x R slice of u against B, and adds the product into y with
// one bf16 rounding per element.  u is fed to the tensor cores as two bf16
// terms (high part + residual), so about 16 significant bits of the fp32 u
// reach the product.  CTAs loop over the items with a stride of the grid.
#include "common.cuh"
#include "launch.h"

namespace grg {

constexpr int kExpandThreads = 128;
constexpr int kEN = 256;  // output columns per item (64 per warp)

struct ExpandParams {
  const float* u;
  int max_num_tokens;
  const __nv_bfloat16* b0;
  const __nv_bfloat16* b1;
  const __nv_bfloat16* b2;
  int w0, w1, w2;       // slice widths
  int off0, off1, off2; // slice column offsets in y
  int cb0, cb1;         // column blocks of slices 0 and 1
  int cb_total;         // column blocks over all slices
  __nv_bfloat16* y;
  long long y_stride;
  const int32_t* records;  // tile records of height BM
  const int32_t* num_tiles;
  int tile_capacity;
  int num_loras;
};

// Byte offset of 16-byte chunk ch (0..31) of row k of a [R][256] bf16 tile.
__device__ __forceinline__ uint32_t swz512(int k, int ch) {
  return static_cast<uint32_t>(k * 512 + (((ch & ~7) | ((ch ^ k) & 7)) << 4));
}

template <int RANK>
struct UFrag {
  // k-steps of 16 ranks (rank 8 packs high and low parts into one k-step)
  static constexpr int KK = RANK == 8 ? 1 : RANK / 16;
  float2 v[KK][4];  // rows g / g+8 x columns 2q / 2q+8 of each k-step
};

template <int RANK>
__device__ __forceinline__ void load_u(UFrag<RANK>& f, const float* u0, const float* u1, bool ok0,
                                       bool ok1, int q) {
  const float2 z = make_float2(0.f, 0.f);
#pragma unroll
  for (int kk = 0; kk < UFrag<RANK>::KK; ++kk) {
    const int kc = kk * 16 + 2 * q;
    f.v[kk][0] = ok0 ? *reinterpret_cast<const float2*>(u0 + kc) : z;
    f.v[kk][1] = ok1 ? *reinterpret_cast<const float2*>(u1 + kc) : z;
    if (RANK != 8) {
      f.v[kk][2] = ok0 ? *reinterpret_cast<const float2*>(u0 + kc + 8) : z;
      f.v[kk][3] = ok1 ? *reinterpret_cast<const float2*>(u1 + kc + 8) : z;
    }
  }
}

template <int BM, int RANK>
__global__ void __launch_bounds__(kExpandThreads, RANK >= 128 ? 2 : 4) lora_expand_kernel(const ExpandParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  int32_t* rec = reinterpret_cast<int32_t*>(smem + RANK * 512);
  const uint32_t sb = smem_u32(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q = lane & 3;
  // u fragments are prefetched with y when they are small enough to sit in registers
  constexpr bool kPrefetchU = RANK <= 32;
  constexpr int MT = BM / 16;

  pdl_wait();
  pdl_launch_dependents();
  {
    const int first = blockIdx.x / max(p.cb_total, 1);
    if (first < p.tile_capacity) load_record<BM>(p.records, first, rec);
  }
  // clamped so that a workspace that was never prepared stays in bounds
  const int ntiles = min(max(*p.num_tiles, 0), p.tile_capacity);
  const int nitems = ntiles * p.cb_total;
  int loaded = blockIdx.x / max(p.cb_total, 1);

  for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
    const int tile = item / p.cb_total;
    int cb = item - tile * p.cb_total;
    int s = 0;
    if (cb >= p.cb0) {
      cb -= p.cb0;
      s = 1;
      if (cb >= p.cb1) {
        cb -= p.cb1;
        s = 2;
      }
    }
    const int width = s == 0 ? p.w0 : (s == 1 ? p.w1 : p.w2);
    const int off = s == 0 ? p.off0 : (s == 1 ? p.off1 : p.off2);
    const __nv_bfloat16* bsl = s == 0 ? p.b0 : (s == 1 ? p.b1 : p.b2);
    if (tile != loaded) {
      load_record<BM>(p.records, tile, rec);
      loaded = tile;
    }
    __syncthreads();  // record visible
    const TileView tv = TileView::of(rec, BM, p.num_loras);
    const int lora = tv.lora, cnt = tv.count;
    const int c0 = cb * kEN;

    // B_s[lora][0:RANK][c0:c0+256] -> shared memory
    const __nv_bfloat16* bl = bsl + static_cast<long long>(lora) * RANK * width;
    for (int c = tid; c < RANK * 32; c += kExpandThreads) {
      const int k = c >> 5, ch = c & 31;
      const int col = c0 + ch * 8;
      const bool ok = col < width && cnt > 0;
      cp_async_16(sb + swz512(k, ch), ok ? bl + static_cast<long long>(k) * width + col : bsl, ok);
    }
    cp_async_commit();

    // this warp's 64 columns of the gathered y rows (and u) -> registers
    const int colw = c0 + warp * 64;
    int tk[MT][2];
    uint32_t yv[MT][8][2];
    UFrag<RANK> uf[kPrefetchU ? MT : 1];
#pragma unroll
    for (int mi = 0; mi < MT; ++mi) {
      tk[mi][0] = record_token(rec, mi * 16 + g, cnt, p.max_num_tokens);
      tk[mi][1] = record_token(rec, mi * 16 + g + 8, cnt, p.max_num_tokens);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int col = colw + nt * 8 + 2 * q;
        const bool cok = col < width;
#pragma unroll
        for (int h = 0; h < 2; ++h)
          yv[mi][nt][h] = (cok && tk[mi][h] >= 0)
                              ? *reinterpret_cast<const uint32_t*>(
                                    p.y + static_cast<long long>(tk[mi][h]) * p.y_stride + off + col)
                              : 0u;
      }
      if constexpr (kPrefetchU) {
        const float* u0 = p.u + (static_cast<long long>(s) * p.max_num_tokens + max(tk[mi][0], 0)) * RANK;
        const float* u1 = p.u + (static_cast<long long>(s) * p.max_num_tokens + max(tk[mi][1], 0)) * RANK;
        load_u<RANK>(uf[mi], u0, u1, tk[mi][0] >= 0, tk[mi][1] >= 0, q);
      }
    }
    cp_async_wait<0>();
    __syncthreads();  // B tile visible

#pragma unroll
    for (int mi = 0; mi < MT; ++mi) {
      const int t0 = tk[mi][0], t1 = tk[mi][1];
      if (__all_sync(0xffffffffu, t0 < 0 && t1 < 0)) continue;
      float acc[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
      UFrag<RANK> ul;
      if constexpr (kPrefetchU) {
        ul = uf[mi];
      } else {
        const float* u0 = p.u + (static_cast<long long>(s) * p.max_num_tokens + max(t0, 0)) * RANK;
        const float* u1 = p.u + (static_cast<long long>(s) * p.max_num_tokens + max(t1, 0)) * RANK;
        load_u<RANK>(ul, u0, u1, t0 >= 0, t1 >= 0, q);
      }

      if constexpr (RANK == 8) {
        // k = 0..7 carry the high parts, k = 8..15 the residuals; B rows repeat.
        uint32_t a[4];
        split_bf16x2(ul.v[0][0].x, ul.v[0][0].y, a[0], a[2]);
        split_bf16x2(ul.v[0][1].x, ul.v[0][1].y, a[1], a[3]);
#pragma unroll
        for (int nt = 0; nt < 8; nt += 4) {
          uint32_t bfr[4];
          ldsm_x4_trans(bfr, sb + swz512(lane & 7, warp * 8 + nt + (lane >> 3)));
#pragma unroll
          for (int j = 0; j < 4; ++j) mma_bf16(acc[nt + j], a, bfr[j], bfr[j]);
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < RANK / 16; ++kk) {
          uint32_t ah[4], al[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split_bf16x2(ul.v[kk][e].x, ul.v[kk][e].y, ah[e], al[e]);
#pragma unroll
          for (int nt = 0; nt < 8; nt += 2) {
            uint32_t bfr[4];
            const int mat = lane >> 3;
            ldsm_x4_trans(bfr, sb + swz512(kk * 16 + ((mat & 1) << 3) + (lane & 7),
                                           warp * 8 + nt + (mat >> 1)));
            mma_bf16(acc[nt], ah, bfr[0], bfr[1]);
            mma_bf16(acc[nt], al, bfr[0], bfr[1]);
            mma_bf16(acc[nt + 1], ah, bfr[2], bfr[3]);
            mma_bf16(acc[nt + 1], al, bfr[2], bfr[3]);
          }
        }
      }

#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int col = colw + nt * 8 + 2 * q;
        if (col < width) {
          if (t0 >= 0) {
            const float2 yf = unpack_bf16x2(yv[mi][nt][0]);
            *reinterpret_cast<uint32_t*>(p.y + static_cast<long long>(t0) * p.y_stride + off + col) =
                pack_bf16x2(yf.x + acc[nt][0], yf.y + acc[nt][1]);
          }
          if (t1 >= 0) {
            const float2 yf = unpack_bf16x2(yv[mi][nt][1]);
            *reinterpret_cast<uint32_t*>(p.y + static_cast<long long>(t1) * p.y_stride + off + col) =
                pack_bf16x2(yf.x + acc[nt][2], yf.y + acc[nt][3]);
          }
        }
      }
    }
    __syncthreads();  // before the next item overwrites the record and the B tile
  }
}

template <int BM, int RANK>
static int run_expand(const ExpandParams& prm, cudaStream_t stream, long long max_items) {
  const void* fn = reinterpret_cast<const void*>(lora_expand_kernel<BM, RANK>);
  const size_t smem = static_cast<size_t>(RANK) * 512 + record_ints(BM) * sizeof(int32_t);
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

int launch_expand(const ExpandArgs& a, cudaStream_t stream) {
  constexpr int BM = 32;
  ExpandParams p;
  p.u = a.u;
  p.max_num_tokens = a.max_num_tokens;
  const __nv_bfloat16* b[3];
  int w[3] = {0, 0, 0}, off[3] = {0, 0, 0}, cbs[3] = {0, 0, 0};
  int acc_off = 0, cb_total = 0;
  for (int s = 0; s < 3; ++s) {
    const int ss = s < a.num_slices ? s : 0;
    b[s] = static_cast<const __nv_bfloat16*>(a.lora_b[ss]);
    if (s < a.num_slices) {
      w[s] = a.slice_width[s];
      off[s] = acc_off;
      acc_off += w[s];
      cbs[s] = (w[s] + kEN - 1) / kEN;
      cb_total += cbs[s];
    }
  }
  p.b0 = b[0]; p.b1 = b[1]; p.b2 = b[2];
  p.w0 = w[0]; p.w1 = w[1]; p.w2 = w[2];
  p.off0 = off[0]; p.off1 = off[1]; p.off2 = off[2];
  p.cb0 = cbs[0]; p.cb1 = cbs[1];
  p.cb_total = cb_total;
  p.y = static_cast<__nv_bfloat16*>(a.y);
  p.y_stride = a.y_row_stride;
  WsView ws = ws_view(const_cast<void*>(a.workspace), a.max_num_tokens, a.num_loras);
  p.records = ws.lists[tile_index_of(BM)];
  p.num_tiles = ws.num_tiles + tile_index_of(BM);
  p.tile_capacity =
      static_cast<int>(tile_list_capacity(a.max_num_tokens, a.num_loras, tile_index_of(BM)));
  p.num_loras = a.num_loras;
  const long long max_items =
      tile_list_capacity(a.max_num_tokens, a.num_loras, tile_index_of(BM)) * cb_total;
  switch (a.rank) {
    case 8: return run_expand<BM, 8>(p, stream, max_items);
    case 16: return run_expand<BM, 16>(p, stream, max_items);
    case 32: return run_expand<BM, 32>(p, stream, max_items);
    case 64: return run_expand<BM, 64>(p, stream, max_items);
    case 128: return run_expand<BM, 128>(p, stream, max_items);
    default: return -3;
  }
}

}  // namespace grg
