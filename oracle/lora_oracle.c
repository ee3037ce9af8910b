/*
 * fp64 CPU oracle for multi-LoRA shrink/expand over an unsorted mixed-adapter
 * batch.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU
 * baseline leg of the benchmark call it; the product path never does.  It
 * shares no code, header, table or constant with the CUDA library.
 *
 * What it computes (one LoRA-wrapped linear layer):
 *
 *   "[V1] LoRA - Add triton kernels for V1" (vLLM PR 13096), section "Why do
 *   we need a new set of kernels": V1 does not sort requests by LoRA id; the
 *   kernels are told which input token maps to which LoRA id and load the
 *   right tokens themselves; the rest is the SGMV low-rank matmul.
 *   "[Tracking] Multi-LoRA Serving" (MLC-LLM), Overview: SGMV gathers each
 *   segment's adapter weights and applies the low-rank product per request.
 *   "[Kernel] LoRA - Enable CUDAGraphs for V1" (vLLM PR 14626): buffers are
 *   static, sized by max_num_tokens, and the CUDA-graph pad region past the
 *   valid tokens is not zeroed, so it must never reach an output.
 *
 * With m = token_lora_mapping (-1 = no adapter), L adapters, rank R,
 * S output slices of widths N_s at offsets off_s:
 *
 *   metadata:  stable grouping of t in [0, n) by m[t] (bin L = no adapter)
 *   shrink:    u[s][t][r] = scale * sum_h x[t][h] * A_s[m[t]][r][h]
 *              (times lora_scales[m[t]] when a per-adapter factor is given)
 *   expand:    y[t][off_s + j] += sum_r u[s][t][r] * B_s[m[t]][r][j]
 *
 * for t < n with 0 <= m[t] < L only.  Inputs (x, A, B, y) are 16-bit words:
 * bf16 by default, IEEE binary16 (fp16) when the f16 flag is set; the pages
 * fix no input precision, and both types are decoded exactly to double.
 * Everything is plain loops in the
 * order the definition states, accumulated in double.  Tokens are
 * independent, so the token loop may run on several host threads (OpenMP)
 * without changing any result.
 */
#include <stdint.h>
#include <stdlib.h>
#include <math.h>
#include <string.h>

/* status bits reported by the metadata oracle */
#define ORACLE_STATUS_BAD_LORA_ID 1u   /* an id outside [-1, L) among t < n */
#define ORACLE_STATUS_BAD_NUM_TOKENS 2u /* n outside [0, max_num_tokens] */
#define ORACLE_STATUS_NO_MEMORY 0x80000000u /* host allocation failed */

static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits; exponent 0 holds zeros and subnormals (fraction * 2^-24), exponent
 * 31 infinities (fraction 0) and NaNs. */
static double f16_bits_to_double(uint16_t bits)
{
    const int sign = (bits >> 15) & 1, exp = (bits >> 10) & 31, frac = bits & 1023;
    double v;
    if (exp == 0)
        v = ldexp((double)frac, -24);
    else if (exp == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + (double)frac, exp - 25);
    return sign ? -v : v;
}

/* A 16-bit input word as a double: fp16 when f16 is set, else bf16. */
static double bits_to_double(uint16_t bits, int f16)
{
    return f16 ? f16_bits_to_double(bits) : bf16_bits_to_double(bits);
}

/* Bin of one token: its LoRA id, or L when it has no (valid) adapter. */
static int64_t bin_of(int32_t id, int64_t num_loras, uint32_t *status)
{
    if (id >= 0 && (int64_t)id < num_loras) return id;
    if (id != -1) *status |= ORACLE_STATUS_BAD_LORA_ID;
    return num_loras;
}

/*
 * Stable counting sort of the token indices 0..n-1 by their bin.
 *   num_tokens_per_lora   [L+1]  count of each bin (bin L = no adapter)
 *   lora_token_start_loc  [L+2]  exclusive prefix sum, last entry = n
 *   sorted_token_ids      [T_max] bin 0's tokens ascending, then bin 1's, ...
 *                                 entries n..T_max-1 are -1
 * Mapping entries at t >= n are never read.  Returns the status bits.
 */
uint32_t oracle_prepare_metadata(const int32_t *token_lora_mapping, int64_t num_tokens,
                                 int64_t max_num_tokens, int64_t num_loras,
                                 int32_t *sorted_token_ids, int32_t *num_tokens_per_lora,
                                 int32_t *lora_token_start_loc)
{
    uint32_t status = 0;
    int64_t n = num_tokens;
    if (n < 0) { n = 0; status |= ORACLE_STATUS_BAD_NUM_TOKENS; }
    if (n > max_num_tokens) { n = max_num_tokens; status |= ORACLE_STATUS_BAD_NUM_TOKENS; }

    /* histogram */
    for (int64_t b = 0; b <= num_loras; ++b) num_tokens_per_lora[b] = 0;
    for (int64_t t = 0; t < n; ++t)
        num_tokens_per_lora[bin_of(token_lora_mapping[t], num_loras, &status)] += 1;

    /* exclusive prefix sum */
    lora_token_start_loc[0] = 0;
    for (int64_t b = 0; b <= num_loras; ++b)
        lora_token_start_loc[b + 1] = lora_token_start_loc[b] + num_tokens_per_lora[b];

    /* stable scatter: walk the tokens in order; each goes to its bin's next free slot */
    int64_t *cursor = (int64_t *)malloc((size_t)(num_loras + 1) * sizeof *cursor);
    if (!cursor) return status | ORACLE_STATUS_NO_MEMORY;
    for (int64_t b = 0; b <= num_loras; ++b) cursor[b] = lora_token_start_loc[b];
    for (int64_t t = 0; t < n; ++t) {
        uint32_t seen = 0;
        int64_t b = bin_of(token_lora_mapping[t], num_loras, &seen);
        sorted_token_ids[cursor[b]++] = (int32_t)t;
    }
    free(cursor);
    for (int64_t t = n; t < max_num_tokens; ++t) sorted_token_ids[t] = -1;
    return status;
}

/*
 * Shrink: u[s][t][r] = c(m[t]) * sum_h x[t][h] * A_s[m[t]][r][h]   (fp64)
 *   c(l)          scale, or scale * lora_scales[l] when lora_scales is given
 *                 (a per-adapter factor; the pages are silent on it)
 *   x             bf16 bits, row t at x + t * x_row_stride, hidden entries
 *   lora_a[s]     bf16 bits, [L][R][hidden] row-major
 *   u             double, [S][max_num_tokens][R]; only rows of tokens
 *                 t < n with 0 <= m[t] < L are written, all else untouched
 */
void oracle_shrink(const uint16_t *x, int64_t x_row_stride, int64_t hidden,
                   const uint16_t *const *lora_a, int64_t num_slices, int64_t rank,
                   double scale, const double *lora_scales, const int32_t *token_lora_mapping,
                   int64_t num_tokens, int64_t num_loras, double *u, int64_t max_num_tokens,
                   int f16, int num_threads)
{
    int64_t t;
#pragma omp parallel for schedule(dynamic, 4) num_threads(num_threads)
    for (t = 0; t < num_tokens; ++t) {
        int32_t id = token_lora_mapping[t];
        if (id < 0 || (int64_t)id >= num_loras) continue;
        const uint16_t *xrow = x + t * x_row_stride;
        const double c = lora_scales ? scale * lora_scales[id] : scale;
        for (int64_t s = 0; s < num_slices; ++s) {
            const uint16_t *a = lora_a[s] + (int64_t)id * rank * hidden;
            for (int64_t r = 0; r < rank; ++r) {
                double acc = 0.0;
                for (int64_t h = 0; h < hidden; ++h)
                    acc += bits_to_double(xrow[h], f16) * bits_to_double(a[r * hidden + h], f16);
                u[(s * max_num_tokens + t) * rank + r] = c * acc;
            }
        }
    }
}

/*
 * Expand: y_out[t][off_s + j] = y_in[t][off_s + j] + sum_r u[s][t][r] * B_s[m[t]][r][j]
 *   u             double, [S][max_num_tokens][R]
 *   lora_b[s]     bf16 bits, [L][R][slice_width[s]] row-major
 *   y_in          bf16 bits, row t at y_in + t * y_row_stride
 *   y_out         double, same indexing as y_in; every element of rows
 *                 0..max_num_tokens-1 (columns < y_row_stride) is written:
 *                 a copy of y_in, plus the LoRA term on adapter tokens t < n
 */
void oracle_expand(const double *u, const uint16_t *const *lora_b, const int64_t *slice_width,
                   int64_t num_slices, int64_t rank, const uint16_t *y_in, int64_t y_row_stride,
                   const int32_t *token_lora_mapping, int64_t num_tokens, int64_t num_loras,
                   double *y_out, int64_t max_num_tokens, int f16, int num_threads)
{
    int64_t t;
#pragma omp parallel for schedule(dynamic, 4) num_threads(num_threads)
    for (t = 0; t < max_num_tokens; ++t) {
        for (int64_t c = 0; c < y_row_stride; ++c)
            y_out[t * y_row_stride + c] = bits_to_double(y_in[t * y_row_stride + c], f16);
        if (t >= num_tokens) continue;
        int32_t id = token_lora_mapping[t];
        if (id < 0 || (int64_t)id >= num_loras) continue;
        int64_t offset = 0;
        for (int64_t s = 0; s < num_slices; ++s) {
            const uint16_t *b = lora_b[s] + (int64_t)id * rank * slice_width[s];
            for (int64_t j = 0; j < slice_width[s]; ++j) {
                double acc = 0.0;
                for (int64_t r = 0; r < rank; ++r)
                    acc += u[(s * max_num_tokens + t) * rank + r] *
                           bits_to_double(b[r * slice_width[s] + j], f16);
                y_out[t * y_row_stride + offset + j] += acc;
            }
            offset += slice_width[s];
        }
    }
}

/* Threads the OpenMP runtime would use (1 when built without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Decodes n 16-bit input words (fp16 when f16 is set, else bf16) to doubles;
 * lets the tests pin the two decoders against an independent float16. */
void oracle_decode_bits(const uint16_t *bits, int64_t n, int f16, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = bits_to_double(bits[i], f16);
}
