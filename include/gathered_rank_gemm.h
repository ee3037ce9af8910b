/*
 * gathered_rank_gemm — multi-LoRA shrink / expand over an unsorted,
 * mixed-adapter token batch, for NVIDIA GB300 (sm_103a).
 *
 * The operation (one LoRA-wrapped linear layer):
 *
 *   "[V1] LoRA - Add triton kernels for V1" (vLLM PR 13096), section "Why do
 *   we need a new set of kernels": the batch is NOT sorted by LoRA id; the
 *   kernels are given the token -> LoRA map and use it to load each token's
 *   rows, then run the low-rank (SGMV-style) matmuls.  Point 1 of "Kernel Code
 *   Change": the launch grid must not depend on the batch, so the calls can be
 *   captured once in a CUDA graph.
 *   "[Kernel] LoRA - Enable CUDAGraphs for V1" (vLLM PR 14626): buffers are
 *   static, sized by max_num_tokens, and the pad rows past the valid tokens are
 *   not zeroed, so they must never be read into an output.
 *
 * With m = token_lora_mapping (-1 = no adapter), n valid tokens, L adapter
 * slots, rank R and S in {1,2,3} output slices of widths N_s at column
 * offsets off_s = N_0 + ... + N_{s-1}:
 *
 *   lora_prepare_metadata: stable grouping of t in [0, n) by m[t]
 *   lora_shrink:  u[s][t][r] = scale * sum_h x[t][h] * A_s[m[t]][r][h]   (fp32 out)
 *   lora_expand:  y[t][off_s + j] = bf16( y[t][off_s + j]
 *                                       + sum_r u[s][t][r] * B_s[m[t]][r][j] )
 *
 * for t < n with 0 <= m[t] < L.  Rows of tokens with m[t] = -1 and rows t >= n
 * are never read from x and never read from or written to u and y.
 *
 * Conventions for every call:
 *  - Every array argument is a DEVICE pointer owned by the caller, except the
 *    small per-slice arrays (lora_a, lora_b, slice_width), which are HOST
 *    arrays of num_slices entries read during the call (their device pointers
 *    are copied into the kernel parameters).  The library never allocates,
 *    frees or synchronises (lora_read_status excepted).
 *  - bf16 data is passed as uint16_t bit patterns (IEEE bfloat16).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) on the current device, so every call can be captured into a CUDA
 *    graph.  The number of valid tokens n lives in device memory, so one
 *    captured graph serves every n <= max_num_tokens.
 *  - Kernels are launched with programmatic dependent launch enabled, so a
 *    kernel may start while the one ahead of it on the stream is finishing.
 *    Before its dependency wait (which returns once every earlier kernel on
 *    the stream has completed and its writes are visible) a kernel of this
 *    library only
 *      - reads the tile records in the workspace, which only
 *        lora_prepare_metadata writes and which it makes visible before it
 *        lets the next kernel start (so nothing else may write the workspace
 *        while calls that use it are in flight), and
 *      - prefetches weights and activation rows into L2, which is the GPU's
 *        coherence point: a prefetch never yields stale data.
 *    Every copy into shared memory and every other read comes after the
 *    wait, with one exception inside lora_shrink_expand (and its fp16 and
 *    paged forms): its second kernel loads B and its y rows before the wait,
 *    because the kernel ahead of it is the same call's shrink, which writes
 *    neither and lets the second kernel start only after its own wait.  So
 *    any kernel may come right before any call, including one that rewrites
 *    the weights, x or y.  A kernel whose CTAs have no work still waits
 *    before it exits, so stream order holds through it.
 *  - Return value: LORA_OK when the work was enqueued, a negative LORA_ERR_*
 *    code when an argument was rejected (nothing is launched) or the launch
 *    failed.  Problems that only the data reveals (a LoRA id outside [-1, L),
 *    n outside [0, max_num_tokens]) cannot be reported synchronously: they set
 *    bits in the status word inside the workspace (lora_read_status), and the
 *    offending tokens are treated as having no adapter / n is clamped.
 */
#ifndef GATHERED_RANK_GEMM_H
#define GATHERED_RANK_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LORA_OK 0
#define LORA_ERR_NULL (-1)       /* a required pointer is NULL */
#define LORA_ERR_ALIGN (-2)      /* a pointer or row stride breaks the 16-byte rule */
#define LORA_ERR_SHAPE (-3)      /* a size is outside the supported set */
#define LORA_ERR_WORKSPACE (-4)  /* workspace too small */
#define LORA_ERR_LAUNCH (-5)     /* the CUDA launch failed (cudaGetLastError) */
#define LORA_ERR_CUDA (-6)       /* another CUDA runtime call failed */

#define LORA_STATUS_BAD_LORA_ID 0x1u     /* some m[t], t < n, was outside [-1, L) */
#define LORA_STATUS_BAD_NUM_TOKENS 0x2u  /* n was outside [0, max_num_tokens]; clamped */
#define LORA_STATUS_TIMEOUT 0x4u         /* a kernel's bounded wait for its own copies gave up;
                                            the outputs of that call are unspecified */
#define LORA_STATUS_BAD_WEIGHT 0x8u      /* a paged weight address was not 16-byte aligned */

#define LORA_MAX_SLICES 3
#define LORA_MAX_LORAS 1024
#define LORA_MAX_NUM_TOKENS (1 << 22)

/*
 * Bytes of device workspace that lora_prepare_metadata fills and lora_shrink /
 * lora_expand read: a status word, the clamped n and, for tile heights of
 * 16, 32, 64 and 128 tokens, the list of tile records (adapter, count and the
 * tile's token ids) that the fixed-grid kernels walk.  About 4 * 4 bytes per
 * token plus 1 KB per adapter (277 KB at 8192 tokens and 128 LoRAs).  Returns
 * 0 for sizes outside the supported range.  Besides the grouping kernel, the
 * shrink and expand kernels may OR LORA_STATUS_TIMEOUT into its status word.
 */
size_t lora_workspace_size(int64_t max_num_tokens, int64_t max_loras);

/*
 * Stable grouping of the batch's tokens by LoRA id ("[V1] LoRA - Add triton
 * kernels for V1", "Why do we need a new set of kernels": V1 keeps the batch
 * unsorted, so the grouping is computed on the device from the token -> LoRA
 * map; "[Kernel] LoRA - Enable CUDAGraphs for V1": the map is a static
 * max_num_tokens buffer).  A histogram / prefix-sum / stable scatter, run by
 * one CTA when max_num_tokens <= 1024 and max_loras <= 128 (one token per
 * thread), else by one thread-block cluster (one CTA per 1024 tokens of
 * max_num_tokens, up to 8); the grid depends only on max_num_tokens and
 * max_loras, not on the data.
 *
 *   token_lora_mapping   int32[max_num_tokens]; entries t >= n may be loaded
 *                        (the one-CTA kernel loads every entry at once with
 *                        n) but never affect any output
 *   num_tokens           device int32: n
 *   sorted_token_ids     int32[max_num_tokens] out: tokens of LoRA 0 in
 *                        ascending order, then LoRA 1, ..., then the tokens
 *                        without an adapter; entries n.. are -1
 *   num_tokens_per_lora  int32[max_loras + 1] out: entry L counts tokens
 *                        without an adapter
 *   lora_token_start_loc int32[max_loras + 2] out: exclusive prefix sum of the
 *                        counts; entry L+1 equals n
 *   workspace            lora_workspace_size(max_num_tokens, max_loras) bytes,
 *                        16-byte aligned; its status word is OR-ed (never
 *                        cleared here) and the rest is overwritten
 * Sizes: 1 <= max_num_tokens <= LORA_MAX_NUM_TOKENS, 1 <= max_loras <= LORA_MAX_LORAS.
 */
int lora_prepare_metadata(const int32_t *token_lora_mapping, const int32_t *num_tokens,
                          int64_t max_num_tokens, int64_t max_loras,
                          int32_t *sorted_token_ids, int32_t *num_tokens_per_lora,
                          int32_t *lora_token_start_loc, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * Shrink ("[V1] LoRA - Add triton kernels for V1": gather each token's input
 * row through the token -> LoRA information and multiply by its adapter's A):
 *   u[s][t][r] = c(m[t]) * sum_h x[t][h] * A_s[m[t]][r][h]  (bf16 in, fp32 out)
 *   c(l) = scale, or scale * lora_scales[l] (in fp32) when lora_scales is given
 *
 *   x                bf16[max_num_tokens][x_row_stride], hidden columns used
 *   lora_a           HOST array of num_slices device pointers, each
 *                    bf16[max_loras][rank][hidden] row-major
 *   lora_scales      NULL, or device fp32[max_loras]: a per-adapter factor on
 *                    scale (the pages are silent on per-LoRA scales)
 *   u                fp32[num_slices][max_num_tokens][rank] out; only rows of
 *                    adapter tokens t < n are written
 *   sorted_token_ids, lora_token_start_loc, workspace: from lora_prepare_metadata
 *                    with the same max_num_tokens / max_loras
 * Sizes: hidden a multiple of 8, rank in {8, 16, 32, 64, 128}, 1 <= num_slices
 * <= 3; x, every A_s and u 16-byte aligned, x_row_stride a multiple of 8 and
 * >= hidden.  Accumulation is fp32 (tensor cores, bf16 operands).
 */
int lora_shrink(const uint16_t *x, int64_t x_row_stride, int64_t hidden,
                const uint16_t *const *lora_a, int num_slices, int rank, float scale,
                const float *lora_scales, float *u, const int32_t *sorted_token_ids,
                const int32_t *lora_token_start_loc,
                int64_t max_num_tokens, int64_t max_loras, const void *workspace,
                size_t workspace_bytes, void *stream);

/*
 * Expand ("[V1] LoRA - Add triton kernels for V1": same token loading, rank ->
 * width matmul added into the layer's output):
 *   y[t][off_s + j] = bf16( float(y[t][off_s + j]) + sum_r u[s][t][r] * B_s[m[t]][r][j] )
 * one round-to-nearest-even per element; y is updated in place.
 *
 *   u                fp32[num_slices][max_num_tokens][rank] (from lora_shrink)
 *   lora_b           HOST array of num_slices device pointers, each
 *                    bf16[max_loras][rank][slice_width[s]] row-major
 *   slice_width      HOST array of num_slices widths, each a multiple of 8
 *   y                bf16[max_num_tokens][y_row_stride] in/out; slice s covers
 *                    columns off_s .. off_s + slice_width[s] - 1
 *   sorted_token_ids, lora_token_start_loc, workspace: from lora_prepare_metadata
 * Sizes: y_row_stride a multiple of 8 and >= the sum of the widths; rank in
 * {8, 16, 32, 64, 128}; u, y and every B_s 16-byte aligned.  The rank
 * contraction runs on tensor cores with u split into two bf16 terms
 * (high + low part), so u keeps about 16 significant bits.
 */
int lora_expand(const float *u, const uint16_t *const *lora_b, const int64_t *slice_width,
                int num_slices, int rank, uint16_t *y, int64_t y_row_stride,
                const int32_t *sorted_token_ids, const int32_t *lora_token_start_loc,
                int64_t max_num_tokens, int64_t max_loras, const void *workspace,
                size_t workspace_bytes, void *stream);

/*
 * Shrink then expand for one layer in one call: the same arguments, results
 * and rules as lora_shrink followed by lora_expand (u is written too).  When
 * the batch is small enough for a thread-block cluster to hold a tile's whole
 * problem on chip (decode-sized batches: up to 16 k-blocks of 64 columns and
 * 48 output units of 64 columns per CTA) and every tile's cluster fits in one
 * wave, one fused kernel does both steps and the expand reads u from shared
 * memory.  Otherwise, with a workspace of at least
 * lora_shrink_expand_workspace_size bytes and a batch of up to 1024 tokens
 * with rank <= 32, the split-K path runs: the shrink's CTAs (up to 16 per
 * tile, no cluster) write partial tiles of u into the workspace and the
 * expand adds them up in CTA order (u and y then match the two separate calls
 * up to the order of the fp32 partial sums).  Else the kernels of
 * lora_shrink and lora_expand run unchanged.  Either way the work stays on
 * the GPU; lora_shrink_expand_path tells which path a shape takes.  The
 * split-K path keeps its partial tiles in the workspace: order calls that
 * share a workspace on one stream.
 */
int lora_shrink_expand(const uint16_t *x, int64_t x_row_stride, int64_t hidden,
                       const uint16_t *const *lora_a, const uint16_t *const *lora_b,
                       const int64_t *slice_width, int num_slices, int rank, float scale,
                       const float *lora_scales, float *u, uint16_t *y, int64_t y_row_stride,
                       const int32_t *sorted_token_ids, const int32_t *lora_token_start_loc,
                       int64_t max_num_tokens, int64_t max_loras, const void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * Workspace bytes that let lora_shrink_expand take its split-K path for this
 * shape: lora_workspace_size plus P * 16 * num_slices * rank * 4 bytes of
 * partial tiles per 16-token tile of the batch (P = 16 for rank <= 16, 8 for
 * rank 32: the largest split) when max_num_tokens <= 1024 and rank <= 32
 * (else just lora_workspace_size); 0 for sizes the calls reject.
 * A smaller workspace (at least lora_workspace_size) is still valid for
 * every call.
 */
size_t lora_shrink_expand_workspace_size(int64_t max_num_tokens, int64_t max_loras,
                                         int64_t hidden, const int64_t *slice_width,
                                         int num_slices, int rank);

/*
 * fp16 variants (the pages fix no input precision; models served in fp16
 * need them): the same arguments, results and rules as lora_shrink,
 * lora_expand, lora_shrink_expand, lora_shrink_partials and
 * lora_expand_partials (stacked weights), with x, A_s, B_s and y holding IEEE
 * fp16 words instead of bf16.  Accumulation stays fp32; u enters the
 * expand's tensor cores as an fp16 high part plus an fp16 residual, so |u|
 * must stay below the fp16 range (65504); y is rounded once to fp16 (round
 * to nearest even).  Paged weights and lora_apply_noalloc are bf16 only.
 */
int lora_shrink_f16(const uint16_t *x, int64_t x_row_stride, int64_t hidden,
                    const uint16_t *const *lora_a, int num_slices, int rank, float scale,
                    const float *lora_scales, float *u, const int32_t *sorted_token_ids,
                    const int32_t *lora_token_start_loc, int64_t max_num_tokens,
                    int64_t max_loras, const void *workspace, size_t workspace_bytes,
                    void *stream);
int lora_expand_f16(const float *u, const uint16_t *const *lora_b, const int64_t *slice_width,
                    int num_slices, int rank, uint16_t *y, int64_t y_row_stride,
                    const int32_t *sorted_token_ids, const int32_t *lora_token_start_loc,
                    int64_t max_num_tokens, int64_t max_loras, const void *workspace,
                    size_t workspace_bytes, void *stream);
int lora_shrink_expand_f16(const uint16_t *x, int64_t x_row_stride, int64_t hidden,
                           const uint16_t *const *lora_a, const uint16_t *const *lora_b,
                           const int64_t *slice_width, int num_slices, int rank, float scale,
                           const float *lora_scales, float *u, uint16_t *y, int64_t y_row_stride,
                           const int32_t *sorted_token_ids, const int32_t *lora_token_start_loc,
                           int64_t max_num_tokens, int64_t max_loras, const void *workspace,
                           size_t workspace_bytes, void *stream);
int lora_shrink_partials_f16(const uint16_t *x, int64_t x_row_stride, int64_t hidden,
                             const uint16_t *const *lora_a, int num_slices, int rank,
                             const int32_t *sorted_token_ids, const int32_t *lora_token_start_loc,
                             int64_t max_num_tokens, int64_t max_loras, void *workspace,
                             size_t workspace_bytes, void *stream);
int lora_expand_partials_f16(int64_t hidden, const uint16_t *const *lora_b,
                             const int64_t *slice_width, int num_slices, int rank, float scale,
                             const float *lora_scales, float *u, uint16_t *y,
                             int64_t y_row_stride, const int32_t *sorted_token_ids,
                             const int32_t *lora_token_start_loc, int64_t max_num_tokens,
                             int64_t max_loras, const void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * Paged adapter weights (the S-LoRA idea of the pages' "[Tracking] Multi-LoRA
 * Serving" overview: adapters live in separately allocated pages rather than
 * one stacked tensor).  Same arguments, results and rules as lora_shrink,
 * lora_expand and lora_shrink_expand, except that each slice's weights come
 * as a table instead of a stacked tensor:
 *   lora_a_tables   HOST array of num_slices device pointers, each to
 *                   uint64[max_loras]: the device address of adapter l's
 *                   A_s[l], bf16[rank][hidden] row-major
 *   lora_b_tables   the same for B_s[l], bf16[rank][slice_width[s]]
 * Table pointers must be 8-byte aligned.  An entry must be 16-byte aligned
 * or 0; 0 reads as an all-zero adapter (its tokens get u = 0, y unchanged),
 * and a misaligned entry reads the same way and sets LORA_STATUS_BAD_WEIGHT.
 * The tables and the weights they point to are read after the kernels'
 * dependency wait, like stacked weights.  The weights move by 16-byte cp.async
 * instead of TMA tensor maps; the one-call entry point never takes the
 * fused kernel.
 */
int lora_shrink_paged(const uint16_t *x, int64_t x_row_stride, int64_t hidden,
                      const uint64_t *const *lora_a_tables, int num_slices, int rank,
                      float scale, const float *lora_scales, float *u,
                      const int32_t *sorted_token_ids, const int32_t *lora_token_start_loc,
                      int64_t max_num_tokens, int64_t max_loras, const void *workspace,
                      size_t workspace_bytes, void *stream);
int lora_expand_paged(const float *u, const uint64_t *const *lora_b_tables,
                      const int64_t *slice_width, int num_slices, int rank, uint16_t *y,
                      int64_t y_row_stride, const int32_t *sorted_token_ids,
                      const int32_t *lora_token_start_loc, int64_t max_num_tokens,
                      int64_t max_loras, const void *workspace, size_t workspace_bytes,
                      void *stream);
int lora_shrink_expand_paged(const uint16_t *x, int64_t x_row_stride, int64_t hidden,
                             const uint64_t *const *lora_a_tables,
                             const uint64_t *const *lora_b_tables, const int64_t *slice_width,
                             int num_slices, int rank, float scale, const float *lora_scales,
                             float *u, uint16_t *y, int64_t y_row_stride,
                             const int32_t *sorted_token_ids, const int32_t *lora_token_start_loc,
                             int64_t max_num_tokens, int64_t max_loras, const void *workspace,
                             size_t workspace_bytes, void *stream);

/*
 * The two halves of lora_shrink_expand's split-K path, for callers that want
 * to place other work between them (and for timing each kernel).  Same
 * arguments and rules as lora_shrink / lora_expand, with these differences:
 *   - the shape must have max_num_tokens <= 1024 and rank <= 32, and the
 *     workspace must hold lora_shrink_expand_workspace_size bytes
 *     (LORA_ERR_SHAPE / LORA_ERR_WORKSPACE otherwise);
 *   - lora_shrink_partials splits each 16-token tile's hidden dimension over
 *     up to P CTAs (as for the workspace size above; no cluster) and writes
 *     each CTA's fp32 partial tile (its warps summed) into the workspace
 *     behind the metadata: [tile][split][16][num_slices * rank].  It does not
 *     scale and does not write u.
 *   - lora_expand_partials takes `hidden` (it fixes the split), `scale` and
 *     `lora_scales`, sums each tile's partials in CTA order, multiplies by
 *     c(lora) as lora_shrink does, writes the result to u (rows of tokens
 *     with an adapter) and adds u * B into y.
 * Run back to back on one stream they give the u and y of lora_shrink
 * followed by lora_expand up to the order of the fp32 partial sums (bit for
 * bit when the split equals lora_shrink's cluster size).  The partials of one
 * call pair live in
 * the workspace: a second pair on the same workspace must be ordered after
 * the first expand (same stream, or an event).
 */
int lora_shrink_partials(const uint16_t *x, int64_t x_row_stride, int64_t hidden,
                         const uint16_t *const *lora_a, int num_slices, int rank,
                         const int32_t *sorted_token_ids, const int32_t *lora_token_start_loc,
                         int64_t max_num_tokens, int64_t max_loras, void *workspace,
                         size_t workspace_bytes, void *stream);
int lora_expand_partials(int64_t hidden, const uint16_t *const *lora_b,
                         const int64_t *slice_width, int num_slices, int rank, float scale,
                         const float *lora_scales, float *u, uint16_t *y, int64_t y_row_stride,
                         const int32_t *sorted_token_ids, const int32_t *lora_token_start_loc,
                         int64_t max_num_tokens, int64_t max_loras, const void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * Whether one lora_shrink_expand call for this shape on the current device
 * runs the fused kernel: 1 (it does) or 2 (it does not: the split-K or the
 * two-kernel path, see lora_shrink_expand_path); a negative LORA_ERR_* code
 * for sizes the calls reject.  Host-only, no GPU work.
 */
int lora_shrink_expand_kernels(int64_t max_num_tokens, int64_t max_loras, int64_t hidden,
                               const int64_t *slice_width, int num_slices, int rank);

/*
 * Which kernels one lora_shrink_expand call (fp16 != 0: lora_shrink_expand_f16;
 * paged != 0: lora_shrink_expand_paged) runs for this shape, workspace size
 * and the current device; host-only, no GPU work:
 *   LORA_PATH_FUSED        one kernel holding a tile's whole problem on chip
 *                          (tiny batches; never with paged weights)
 *   LORA_PATH_SPLIT_PAIR   the split-K shrink, then the partial-sum expand
 *                          (needs lora_shrink_expand_workspace_size bytes)
 *   LORA_PATH_PAIR         the kernels of lora_shrink, then of lora_expand
 * A negative LORA_ERR_* code for sizes the calls reject.
 */
#define LORA_PATH_FUSED 1
#define LORA_PATH_SPLIT_PAIR 3
#define LORA_PATH_PAIR 4
int lora_shrink_expand_path(int64_t max_num_tokens, int64_t max_loras, int64_t hidden,
                            const int64_t *slice_width, int num_slices, int rank,
                            size_t workspace_bytes, int fp16, int paged);

/*
 * Copies the workspace's status word (LORA_STATUS_* bits OR-ed by every
 * lora_prepare_metadata since the last read) to *status, then clears it.
 * Synchronises `stream`.  Not capturable in a CUDA graph.
 */
int lora_read_status(void *workspace, uint32_t *status, void *stream);

/*
 * One layer - grouping, shrink and expand - without allocating anything.
 * The pages describe no counterpart to this call: it exists for callers that
 * cannot call cudaMalloc (a memory manager that owns the whole device, a
 * plugin host that hands out no device memory, code that must not allocate)
 * and so cannot provide the workspace the three calls above take.
 *
 * Arguments are those of lora_prepare_metadata, lora_shrink and lora_expand
 * (same meaning, layout and rules), minus the workspace; the caller still
 * passes every input and output, u and the three metadata arrays included.
 * `status` (optional, device pointer) receives this call's LORA_STATUS_* bits.
 *
 * The workspace is a file-scope device array of LORA_NOALLOC_SCRATCH_BYTES
 * (384 KB) in the library, which every GPU that loads the library holds
 * until the process exits.  It fits 8192 tokens with 128 adapters; sizes
 * whose workspace (lora_workspace_size) exceeds it are rejected with
 * LORA_ERR_WORKSPACE before anything is enqueued.  The first call on a
 * device looks up the array's device address (once per device, with that
 * device current): make that first call before any stream capture.  Every
 * call uses the same array and leaves its contents behind; the call clears
 * the status word it needs zeroed itself.  Calls that overlap on the GPU
 * (other streams, other threads) race on the array: serialise them.  Every
 * argument is checked before anything is enqueued.
 */
#define LORA_NOALLOC_SCRATCH_BYTES (384 * 1024)
int lora_apply_noalloc(const int32_t *token_lora_mapping, const int32_t *num_tokens,
                       int64_t max_num_tokens, int64_t max_loras, const uint16_t *x,
                       int64_t x_row_stride, int64_t hidden, const uint16_t *const *lora_a,
                       const uint16_t *const *lora_b, const int64_t *slice_width,
                       int num_slices, int rank, float scale, const float *lora_scales,
                       float *u, uint16_t *y, int64_t y_row_stride, int32_t *sorted_token_ids,
                       int32_t *num_tokens_per_lora, int32_t *lora_token_start_loc,
                       uint32_t *status, void *stream);

/* Static text for a LORA_OK / LORA_ERR_* code. */
const char *lora_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* GATHERED_RANK_GEMM_H */
