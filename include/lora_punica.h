/*
 * lora_punica.h -- C ABI of the GB300 (sm_103a) multi-LoRA shrink/expand
 * library (liblora_punica.so).
 *
 * The three core entry points are the three steps of the Punica-style
 * batched LoRA apply described by vLLM's API pages:
 *
 *   lora_meta_prepare  page "vllm.lora.ops.triton_ops.lora_kernel_metadata",
 *                      class LoRAKernelMeta, methods make / _reset /
 *                      prepare_tensors / meta_args.
 *   lora_shrink        page "vllm.lora.punica_wrapper.punica_gpu", method
 *                      PunicaWrapperGPU.add_shrink and its lora_shrink call
 *                      (argument order x, lora_a_stacked, y, meta, scale).
 *   lora_expand        same page, method PunicaWrapperGPU.add_expand and its
 *                      lora_expand call (x, lora_b_stacked, y, meta,
 *                      offset_start, add_inputs); the bias step of
 *                      PunicaWrapperTPU._apply_bias (page
 *                      "vllm.lora.punica_wrapper.punica_tpu") is fused into
 *                      it.
 *
 * Conventions shared by every call:
 *   - Every data pointer is a DEVICE pointer owned by the caller; the
 *     library allocates nothing and keeps no pointer after a call returns.
 *     Arrays of per-slice pointers (lora_a, lora_b, lora_bias) and
 *     slice_sizes are HOST arrays, read during the call only.
 *   - bf16 tensors are passed as pointers to their raw 16-bit patterns
 *     (lora_bf16_t).  All tensors are row-major and dense unless a leading
 *     dimension argument says otherwise.
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t passed
 *     as void*; NULL is the legacy default stream).  Nothing is
 *     synchronised and nothing is read back to the host.
 *   - The device that owns `stream` and every tensor of a call must be the
 *     calling thread's current CUDA device (per-device launch settings are
 *     looked up for the current device).
 *   - Return value: 0 on success; a negative LORA_ERR_* code when an
 *     argument is rejected on the host (nothing is launched); a positive
 *     cudaError_t when a launch fails.  lora_status_string() names both.
 *   - Invalid LoRA ids (outside [-1, max_loras)) are not host errors: the
 *     metadata kernel counts them into meta->error_word and treats those
 *     tokens as having no LoRA, so shrink/expand skip them.
 *   - The no-LoRA early exit is taken on the device: shrink and expand read
 *     *meta->no_lora_flag and return at once when it is set, so a whole
 *     forward pass stays capturable in a CUDA graph with no host sync.
 */
#ifndef LORA_PUNICA_H
#define LORA_PUNICA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Raw bit pattern of one bfloat16 value. */
typedef uint16_t lora_bf16_t;

#define LORA_PUNICA_VERSION 1
#define LORA_MAX_SLICES 8      /* slices per shrink/expand call          */
#define LORA_MAX_LORAS 1024    /* max_loras accepted by the metadata step */
#define LORA_MAX_RANK 128      /* rank r: a multiple of 8, 8 <= r <= 128 */
#define LORA_NOALLOC_MAX_FLOATS (1 << 20)  /* lora_linear_noalloc buffer: 4 MiB */

enum lora_status {
    LORA_OK = 0,
    LORA_ERR_NULL = -1,        /* a required pointer is NULL               */
    LORA_ERR_SIZE = -2,        /* a size is negative or out of range       */
    LORA_ERR_ALIGN = -3,       /* a pointer / stride breaks an alignment rule */
    LORA_ERR_RANK = -4,        /* rank not a multiple of 8 in [8, 128]      */
    LORA_ERR_SLICES = -5,      /* num_slices not in [1, LORA_MAX_SLICES]    */
    LORA_ERR_TOKENS = -6,      /* num_tokens > meta->max_num_tokens         */
    LORA_ERR_WIDTH = -7,       /* offset_start + sum(slice_sizes) > y_ld    */
    LORA_ERR_DEVICE = -8,      /* no usable CUDA device / wrong architecture */
    LORA_ERR_SCRATCH = -9      /* num_slices * num_tokens * rank exceeds
                                  LORA_NOALLOC_MAX_FLOATS (lora_linear_noalloc) */
};

/*
 * Per-forward metadata, the device-side counterpart of LoRAKernelMeta
 * (page "vllm.lora.ops.triton_ops.lora_kernel_metadata", LoRAKernelMeta.make
 * gives the buffer sizes).  The caller allocates every buffer once (int32,
 * device memory) and may reuse them for every forward pass:
 *   token_lora_mapping                [max_num_tokens]  copy of the id map
 *   token_indices_sorted_by_lora_ids  [max_num_tokens]  stable argsort
 *   num_tokens_per_lora               [max_loras + 1]   tokens per active id
 *   lora_token_start_loc              [max_loras + 2]   0, running sums
 *   active_lora_ids                   [max_loras + 1]   ascending, pad -1
 *   no_lora_flag                      [1]               1 = every id is -1
 *   error_word                        [1]               invalid ids counted
 *   grid_sync                         [2]               zero-filled once by
 *       the caller; the grid barrier of lora_linear's single-kernel path
 *       (every call leaves it zero again).  May be NULL, which turns that
 *       path off.  Calls that share a struct must be stream-ordered.
 * The same struct (by pointer) is then handed to lora_shrink/lora_expand;
 * they read it on the device.  The struct itself is host memory and is only
 * read during each call.
 */
typedef struct lora_meta {
    int32_t *token_lora_mapping;
    int32_t *token_indices_sorted_by_lora_ids;
    int32_t *num_tokens_per_lora;
    int32_t *lora_token_start_loc;
    int32_t *active_lora_ids;
    int32_t *no_lora_flag;
    int32_t *error_word;
    int32_t max_loras;
    int32_t max_num_tokens;
    int32_t *grid_sync;
} lora_meta_t;

/*
 * lora_meta_prepare -- LoRAKernelMeta.prepare_tensors on the device.
 *
 *   token_lora_mapping  device int32 [num_tokens], LoRA id per token, -1 =
 *                       no LoRA.
 *   num_tokens          0 <= num_tokens <= meta->max_num_tokens.
 *   meta                buffers as described above; 1 <= max_loras <=
 *                       LORA_MAX_LORAS.
 *
 * Writes, in one kernel: the reset values (active ids -1, counts 0,
 * start_loc 0); no_lora_flag = all(ids == -1) (true for num_tokens == 0);
 * and, only when the flag is false: the mapping copy, the stable permutation
 * of tokens sorted by id (ties keep token order, so id -1 tokens come
 * first), the distinct ids in ascending order with their counts, and
 * start_loc[k + 1] = counts[0] + ... + counts[k].  error_word receives the
 * number of ids outside [-1, max_loras); those tokens are sorted as -1.
 * Result: bit-exact, deterministic.
 */
int lora_meta_prepare(const int32_t *token_lora_mapping, int32_t num_tokens,
                      const lora_meta_t *meta, void *stream);

/*
 * lora_meta_read_no_lora -- the host copy of the no-LoRA flag (page
 * "vllm.lora.ops.triton_ops.lora_kernel_metadata", LoRAKernelMeta field
 * no_lora_flag_cpu, set by prepare_tensors).
 *
 *   meta      the metadata a preceding lora_meta_prepare on `stream` wrote;
 *             only meta->no_lora_flag is read.
 *   stream    the stream that call was ordered on.
 *   no_lora   HOST int32, receives 1 when every id of that batch is -1 (or
 *             it had no tokens), else 0.
 *
 * Copies the 4-byte device flag to the host and synchronises `stream`, so
 * it cannot be captured in a CUDA graph.  No other call needs it: every
 * kernel reads the device flag itself and returns early.
 * Errors: LORA_ERR_NULL for a NULL meta, meta->no_lora_flag or no_lora (on
 * the host, before any CUDA call); a positive cudaError_t if the copy or the
 * synchronisation fails (then *no_lora is left unchanged).
 */
int lora_meta_read_no_lora(const lora_meta_t *meta, void *stream, int32_t *no_lora);

/*
 * lora_shrink -- y[s][t, :] += scale * x[t, :] @ lora_a[s][id(t)]^T for
 * every slice s and every token t whose id is not -1 (page
 * "vllm.lora.punica_wrapper.punica_gpu", PunicaWrapperGPU.add_shrink,
 * "Semantics").  Rows of tokens without a LoRA are not touched.
 *
 *   x           device bf16 [num_tokens, x_ld]; the first `hidden` values of
 *               each row are used.  16-byte aligned, x_ld % 8 == 0.
 *   num_tokens  rows of x, <= meta->max_num_tokens; the metadata must have
 *               been prepared for exactly these tokens.
 *   hidden      H, a multiple of 8.
 *   lora_a      host array of num_slices device pointers, each bf16
 *               [max_loras, rank, hidden] (a leading singleton layer
 *               dimension is the same layout), 16-byte aligned.
 *   rank        r, a multiple of 8 in [8, LORA_MAX_RANK].
 *   y           device fp32 [num_slices, num_tokens, rank], 16-byte
 *               aligned; accumulated into (the caller zeroes it first to
 *               get a plain product).
 *   scale       multiplies the product before it is added.
 *
 * Accumulation is fp32 on the tensor cores (mma.sync; tcgen05 with TMEM
 * accumulators for batches of >= 1024 tokens with num_slices * rank >=
 * 256, LORA_PUNICA_UMMA* in the environment); when the hidden dimension is
 * split across CTAs the partial sums are added with fp32 atomics, so the
 * rounding order is not fixed from run to run.  A bounded wait of the
 * tcgen05 path that runs out sets bit 30 of meta->error_word.
 */
int lora_shrink(const lora_bf16_t *x, int32_t num_tokens, int32_t hidden,
                int64_t x_ld, const lora_bf16_t *const *lora_a,
                int32_t num_slices, int32_t rank, float *y,
                const lora_meta_t *meta, float scale, void *stream);

/*
 * lora_expand -- for every slice s and token t whose id is not -1:
 *   v = x[s][t, :] @ lora_b[s][id(t)]^T + (bias ? lora_bias[s][id(t)] : 0)
 *   y[t, off_s : off_s + n_s] = (add_inputs ? y[t, off_s : off_s + n_s] : 0) + v
 * with off_s = offset_start + n_0 + ... + n_{s-1} (page
 * "vllm.lora.punica_wrapper.punica_gpu", PunicaWrapperGPU.add_expand,
 * "Semantics"; bias as PunicaWrapperTPU._apply_bias).  Rows of tokens
 * without a LoRA, and columns outside the slices, are not touched.
 *
 *   x            device fp32 [num_slices, num_tokens, rank], 16-byte aligned
 *                (the shrink output).
 *   lora_b       host array of num_slices device pointers, each bf16
 *                [max_loras, n_s, rank], 16-byte aligned.
 *   lora_bias    NULL, or a host array of num_slices entries, each NULL or
 *                a device pointer to bf16 [max_loras, n_s].
 *   slice_sizes  host int32 [num_slices], n_s >= 1.
 *   y            device bf16 [num_tokens, y_ld],
 *                offset_start + sum(n_s) <= y_ld.
 *   add_inputs   nonzero: add to y; zero: overwrite the slice columns.
 *
 * x is rounded to bf16 for the tensor cores (as the Triton kernel does when
 * it casts its input to the weight type); products accumulate in fp32
 * (tcgen05 with TMEM accumulators at rank >= 64 when y, y_ld and
 * offset_start are 32-byte aligned and every slice width is a multiple of
 * 64; mma.sync otherwise; LORA_PUNICA_EXPAND_TC* in the environment move
 * the boundary, and with LORA_PUNICA_EXPAND_TC=2 a call the tcgen05 path
 * does not take fails with LORA_ERR_ALIGN or LORA_ERR_SIZE); y, the bias
 * and the product are summed in fp32 and
 * rounded to bf16 once (round to nearest even).  Output: deterministic.  A
 * bounded wait of the tcgen05 path that runs out sets bit 30 of
 * meta->error_word.
 */
int lora_expand(const float *x, const lora_bf16_t *const *lora_b,
                const lora_bf16_t *const *lora_bias,
                const int32_t *slice_sizes, int32_t num_slices, int32_t rank,
                lora_bf16_t *y, int64_t y_ld, int32_t num_tokens,
                int32_t offset_start, int32_t add_inputs,
                const lora_meta_t *meta, void *stream);

/*
 * lora_expand_bf16 -- lora_expand over a bf16 input, for the embedding LoRA
 * (page "vllm.lora.punica_wrapper.punica_gpu",
 * PunicaWrapperGPU.add_lora_embedding: y (+)= x @ lora_b, where x holds the
 * rows of the embedding LoRA's A looked up for each token, and add_inputs
 * is passed through from the caller).
 *
 *   x   device bf16 [num_slices, num_tokens, rank], 16-byte aligned; the
 *       tensor cores take it as it is (no rounding of the input).
 * Every other argument, the results and the errors are those of
 * lora_expand.
 */
int lora_expand_bf16(const lora_bf16_t *x, const lora_bf16_t *const *lora_b,
                     const lora_bf16_t *const *lora_bias,
                     const int32_t *slice_sizes, int32_t num_slices, int32_t rank,
                     lora_bf16_t *y, int64_t y_ld, int32_t num_tokens,
                     int32_t offset_start, int32_t add_inputs,
                     const lora_meta_t *meta, void *stream);

/*
 * lora_linear -- one LoRA layer applied to a batch, metadata included: the
 * result of lora_meta_prepare(token_lora_mapping), then lora_shrink(x ->
 * buf, scale), then lora_expand(buf -> y, lora_bias, offset_start = 0,
 * add_inputs = 1) (page "vllm.lora.punica_wrapper.punica_gpu",
 * PunicaWrapperGPU.update_metadata + add_lora_linear: add_shrink into the
 * fp32 buffer, then add_expand).  Arguments mean what they mean in those
 * three calls; `buf` is accumulated into like lora_shrink's y, and every
 * metadata buffer of `meta` is written as lora_meta_prepare writes it.
 *
 * How the layer runs (every form gives the three calls' results; the
 * shrink's partial sums may be added in a different order):
 *   - one cooperative kernel, by default when num_tokens * num_slices <=
 *     256 (and num_tokens <= 512, max_loras <= 256, rank <= 64, 16-byte
 *     aligned rows): every CTA sorts the ids in shared memory, the shrink
 *     is spread over the grid, a grid barrier (meta->grid_sync; bounded,
 *     bit 30 of the error word on expiry) separates it from the expand;
 *   - one thread-block-cluster kernel for other batches of at most 128
 *     tokens (max_loras <= 256, num_slices * padded rank <= 128);
 *   - rank 128, at most three slices, slice widths multiples of 64, y
 *     32-byte aligned with y_ld a multiple of 16, x and buf 16-byte
 *     aligned, batches of at least 72 tokens per SM of the device
 *     (LORA_PUNICA_LINEAR_TC_MIN_TOKENS sets another threshold): the
 *     metadata kernel, then one tensor-core kernel that runs
 *     the shrink of a 128-token tile, adds its result into that tile's
 *     buffer rows and runs the tile's expand (one CTA per SM, tiles of one
 *     LoRA in turn);
 *   - otherwise three kernels with programmatic dependent launch: the
 *     metadata kernel, the shrink (sorting the ids itself and loading
 *     before its dependency wait, for <= 512 tokens) and the expand
 *     (fetching the metadata, y and B before its wait).
 * Environment (read once, see lora_reload_options): LORA_PUNICA_COOP=0/1
 * never / always (when the batch fits) the cooperative kernel;
 * LORA_PUNICA_FUSED=0/1 and LORA_PUNICA_FUSED_MAX_TOKENS the cluster
 * kernel; LORA_PUNICA_LINEAR_TC=0/1 never / for every call that fits (any
 * batch size) the rank-128 tensor-core kernel (=2 requires it: a call it
 * does not fit fails with LORA_ERR_SIZE), and
 * LORA_PUNICA_LINEAR_TC_MIN_TOKENS its threshold; LORA_PUNICA_SELF_META=1 two
 * kernels (the shrink writes the metadata), =0 the plain three calls.
 */
int lora_linear(const int32_t *token_lora_mapping, int32_t num_tokens,
                const lora_bf16_t *x, int32_t hidden, int64_t x_ld,
                const lora_bf16_t *const *lora_a, const lora_bf16_t *const *lora_b,
                const lora_bf16_t *const *lora_bias, const int32_t *slice_sizes,
                int32_t num_slices, int32_t rank, float scale, float *buf,
                lora_bf16_t *y, int64_t y_ld, const lora_meta_t *meta, void *stream);

/*
 * lora_linear_noalloc -- lora_linear for callers that cannot allocate
 * device memory (code running where cudaMalloc is unavailable or forbidden:
 * inside an allocator or memory-pool callback, a plugin whose host owns
 * every allocation, a process that must not grow after start-up).  The
 * pages have no counterpart: this is an addition of this library.
 *
 * Same arguments and results as lora_linear, without `buf`: the fp32
 * buffer between shrink and expand lives in a fixed array of
 * LORA_NOALLOC_MAX_FLOATS floats (4 MiB) that the library holds on every
 * GPU that loads it, until the process exits.  Each call clears the
 * num_slices * num_tokens * rank floats it uses, so the shrink starts from
 * zero (as add_lora_linear's own zeroed buffer does); larger calls return
 * LORA_ERR_SCRATCH.  No cudaMalloc, cudaFree or allocating library routine
 * is called.
 *
 * The first call on a device looks up the array's device address (with that
 * device current); make it before any stream capture.  `stream` must belong
 * to the current device, else LORA_ERR_DEVICE is returned before anything
 * runs.  All calls on a device share the array: calls that may overlap on
 * the GPU (other streams or threads) race on it and must be serialised by
 * the caller.
 */
int lora_linear_noalloc(const int32_t *token_lora_mapping, int32_t num_tokens,
                        const lora_bf16_t *x, int32_t hidden, int64_t x_ld,
                        const lora_bf16_t *const *lora_a, const lora_bf16_t *const *lora_b,
                        const lora_bf16_t *const *lora_bias, const int32_t *slice_sizes,
                        int32_t num_slices, int32_t rank, float scale, lora_bf16_t *y,
                        int64_t y_ld, const lora_meta_t *meta, void *stream);

/*
 * lora_reload_options -- re-reads the library's tuning variables
 * (LORA_PUNICA_*: which of lora_linear's launch paths a batch takes, which
 * batches the tensor-core kernels take, programmatic dependent launch).
 * The library reads them once, at its first call; no later call reads the
 * environment unless this is called.  It must not run while another thread
 * is inside the library.  The pages have no counterpart: this is a control
 * of this library's own launch choices.
 */
void lora_reload_options(void);

/* Human-readable name of a status (negative LORA_ERR_* or cudaError_t). */
const char *lora_status_string(int status);

/* LORA_PUNICA_VERSION of the loaded library. */
int lora_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LORA_PUNICA_H */
