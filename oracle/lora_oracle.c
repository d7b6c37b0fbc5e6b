/*
 * lora_oracle.c -- plain, slow, fp64 CPU oracle for the multi-LoRA
 * shrink/expand path.  TEST INFRASTRUCTURE ONLY: the test suite, the smoke
 * check and the benchmark's CPU-baseline leg use it; the product path never
 * does.  It shares no code, header or table with the CUDA library.
 *
 * What it follows (API pages "vllm.lora.ops.triton_ops.lora_kernel_metadata",
 * "vllm.lora.punica_wrapper.punica_gpu" and
 * "vllm.lora.punica_wrapper.punica_tpu"):
 *   - oracle_meta_prepare:  LoRAKernelMeta._reset and
 *     LoRAKernelMeta.prepare_tensors (all(map == -1) flag, stable sort,
 *     sorted unique with counts, cumsum into start_loc[1:]).
 *   - oracle_shrink:        PunicaWrapperGPU.add_shrink docstring,
 *     y[i] += (x @ lora_a_stacked[i]) * scale, applied per token with the
 *     token's own LoRA id.
 *   - oracle_expand:        PunicaWrapperGPU.add_expand docstring,
 *     y[:, offset:offset+slice] += x[i] @ lora_b_stacked[i] + bias[i], and
 *     the bias handling of PunicaWrapperTPU._apply_bias (gather bias[id],
 *     zero where id == -1, shift to the slice's columns).
 *
 * Every token is computed on its own, straight from its id, as a dense dot
 * product in double; bf16 inputs are widened exactly.  Results are written
 * unrounded (double); callers round if they need the stored precision.
 *
 * Readings of points the pages leave open (each also listed in the design
 * notes):
 *   - ids outside [-1, L) are invalid: they are counted, treated as -1 by
 *     every step, and the count is returned.
 *   - T == 0 counts as "no LoRA" (all() of an empty tensor is true).
 *   - with no LoRA, only the reset values are written; the mapping copy and
 *     the permutation are left as they were.
 *   - shrink accumulates (+=) into the fp32 buffer.
 *   - add_inputs == 0 overwrites the slice columns of rows with a valid id;
 *     other rows are left untouched in both modes.
 *   - bias columns are shifted by offset_start like the product.
 */
#include <omp.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

/* Threads the OpenMP loops below run on (reported with CPU timings). */
int oracle_num_threads(void)
{
    return omp_get_max_threads();
}

/* bf16 is the upper 16 bits of an IEEE-754 binary32: widening is exact. */
static double bf16_to_f64(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Widen n bf16 values; exposed so the widening itself can be pinned. */
void oracle_bf16_to_f64(const uint16_t *src, int64_t n, double *dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = bf16_to_f64(src[i]);
}

static int valid_id(int32_t id, int32_t num_loras)
{
    return id >= 0 && id < num_loras;
}

/*
 * Metadata (page vllm.lora.ops.triton_ops.lora_kernel_metadata,
 * LoRAKernelMeta.make / _reset / prepare_tensors).
 *   map          [T]      per-token LoRA id, -1 = no LoRA
 *   mapping_copy [T]      receives a copy of map (not written if no LoRA)
 *   sorted_idx   [T]      stable argsort of map   (not written if no LoRA)
 *   active_ids   [L+1]    distinct ids ascending, padded with -1
 *   counts       [L+1]    tokens per active id, padded with 0
 *   start_loc    [L+2]    0, then running sums of counts; tail stays 0
 *   no_lora      [1]      1 if every id is -1 (or T == 0), else 0
 * Returns the number of invalid ids (treated as -1).
 *
 * The sort is written as a counting sort over the bins -1..L-1: a stable
 * sort of small integer keys, which is what torch.sort(stable=True)
 * produces for such keys.
 */
int64_t oracle_meta_prepare(const int32_t *map, int64_t T, int32_t num_loras,
                            int32_t *mapping_copy, int32_t *sorted_idx,
                            int32_t *active_ids, int32_t *counts,
                            int32_t *start_loc, int32_t *no_lora)
{
    const int32_t nbins = num_loras + 1;   /* bin 0 is id -1 */
    int64_t invalid = 0;

    /* _reset */
    for (int32_t k = 0; k < nbins; ++k) {
        active_ids[k] = -1;
        counts[k] = 0;
    }
    for (int32_t k = 0; k < nbins + 1; ++k)
        start_loc[k] = 0;
    no_lora[0] = 0;

    /* histogram over bins; invalid ids go to the -1 bin */
    int64_t bin_count[nbins];
    for (int32_t k = 0; k < nbins; ++k)
        bin_count[k] = 0;
    for (int64_t t = 0; t < T; ++t) {
        int32_t id = map[t];
        if (!valid_id(id, num_loras)) {
            if (id != -1)
                ++invalid;
            id = -1;
        }
        ++bin_count[id + 1];
    }

    /* no-LoRA test: every (sanitised) id is -1; true for T == 0 */
    if (bin_count[0] == T) {
        no_lora[0] = 1;
        return invalid;
    }

    for (int64_t t = 0; t < T; ++t)
        mapping_copy[t] = map[t];

    /* sorted unique with counts: bins with a non-zero count, ascending */
    int32_t n_active = 0;
    int64_t bin_start[nbins];
    int64_t running = 0;
    for (int32_t k = 0; k < nbins; ++k) {
        bin_start[k] = running;
        if (bin_count[k] > 0) {
            active_ids[n_active] = k - 1;
            counts[n_active] = (int32_t)bin_count[k];
            ++n_active;
        }
        running += bin_count[k];
    }

    /* cumsum written to start_loc[1 : 1 + n_active] */
    int64_t acc = 0;
    for (int32_t k = 0; k < n_active; ++k) {
        acc += counts[k];
        start_loc[k + 1] = (int32_t)acc;
    }

    /* stable placement: tokens in increasing index order within each bin */
    int64_t seen[nbins];
    for (int32_t k = 0; k < nbins; ++k)
        seen[k] = 0;
    for (int64_t t = 0; t < T; ++t) {
        int32_t id = map[t];
        if (!valid_id(id, num_loras))
            id = -1;
        int32_t b = id + 1;
        sorted_idx[bin_start[b] + seen[b]] = (int32_t)t;
        ++seen[b];
    }
    return invalid;
}

/*
 * Shrink (page vllm.lora.punica_wrapper.punica_gpu, PunicaWrapperGPU.add_shrink
 * semantics):
 *   for every token t with a valid id and every slice s < S,
 *   buf_out[s][t][i] = buf_in[s][t][i] + scale * sum_h x[t][h] * A_s[id][i][h]
 * and buf_out = buf_in for tokens without one.
 *   x       bf16 bits, row t at x + t * x_ld, H values
 *   A[s]    bf16 bits, [L][r][H] row-major
 *   buf_in  fp32 [S][T][r];  buf_out double [S][T][r]
 */
void oracle_shrink(const uint16_t *x, int64_t T, int64_t H, int64_t x_ld,
                   const uint16_t *const *A, int32_t S, int32_t r,
                   int32_t num_loras, const int32_t *map, double scale,
                   const float *buf_in, double *buf_out)
{
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t t = 0; t < T; ++t) {
        const int32_t id = map[t];
        for (int32_t s = 0; s < S; ++s) {
            for (int32_t i = 0; i < r; ++i) {
                const int64_t o = ((int64_t)s * T + t) * r + i;
                double v = (double)buf_in[o];
                if (valid_id(id, num_loras)) {
                    const uint16_t *arow = A[s] + ((int64_t)id * r + i) * H;
                    const uint16_t *xrow = x + t * x_ld;
                    double dot = 0.0;
                    for (int64_t h = 0; h < H; ++h)
                        dot += bf16_to_f64(xrow[h]) * bf16_to_f64(arow[h]);
                    v += scale * dot;
                }
                buf_out[o] = v;
            }
        }
    }
}

/*
 * Expand (page vllm.lora.punica_wrapper.punica_gpu, PunicaWrapperGPU.add_expand
 * semantics, with the bias of page vllm.lora.punica_wrapper.punica_tpu,
 * PunicaWrapperTPU._apply_bias):
 *   off_s = offset_start + sum_{j<s} n_j
 *   for every token t with a valid id, slice s, and column j < n_s:
 *     v = sum_k xin[s][t][k] * B_s[id][j][k] + (bias_s ? bias_s[id][j] : 0)
 *     y_out[t][off_s + j] = (add_inputs ? y_in[t][off_s + j] : 0) + v
 *   every other element of y_out equals y_in.
 *   xin     fp32 [S][T][r]
 *   B[s]    bf16 bits, [L][n_s][r] row-major
 *   bias    NULL, or S pointers (each NULL or bf16 bits [L][n_s])
 *   y_in    bf16 bits [T][y_ld];  y_out double [T][y_ld]
 */
void oracle_expand(const float *xin, int64_t T, int32_t r,
                   const uint16_t *const *B, const uint16_t *const *bias,
                   const int32_t *slice_sizes, int32_t S, int32_t num_loras,
                   const int32_t *map, const uint16_t *y_in, int64_t y_ld,
                   int64_t offset_start, int32_t add_inputs, double *y_out)
{
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t t = 0; t < T; ++t) {
        const int32_t id = map[t];
        for (int64_t c = 0; c < y_ld; ++c)
            y_out[t * y_ld + c] = bf16_to_f64(y_in[t * y_ld + c]);
        if (!valid_id(id, num_loras))
            continue;
        int64_t off = offset_start;
        for (int32_t s = 0; s < S; ++s) {
            const int32_t n = slice_sizes[s];
            const float *xrow = xin + ((int64_t)s * T + t) * r;
            for (int32_t j = 0; j < n; ++j) {
                const uint16_t *brow = B[s] + ((int64_t)id * n + j) * r;
                double v = 0.0;
                for (int32_t k = 0; k < r; ++k)
                    v += (double)xrow[k] * bf16_to_f64(brow[k]);
                if (bias != NULL && bias[s] != NULL)
                    v += bf16_to_f64(bias[s][(int64_t)id * n + j]);
                const int64_t o = t * y_ld + off + j;
                y_out[o] = (add_inputs ? y_out[o] : 0.0) + v;
            }
            off += n;
        }
    }
}
