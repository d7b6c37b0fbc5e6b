// lora_expand.cu -- y[t, off_s + j] (+)= x[s][t, :] @ B[s][id(t)][j, :] +
// bias[s][id(t)][j]  (page "vllm.lora.punica_wrapper.punica_gpu",
// PunicaWrapperGPU.add_expand; bias step of page
// "vllm.lora.punica_wrapper.punica_tpu", PunicaWrapperTPU._apply_bias).
//
// Work items are (token tile of one LoRA segment, BN-column chunk of one
// slice), numbered chunk-fastest.  The grid is persistent and every CTA
// takes one contiguous, balanced range of items, so a CTA walks the column
// chunks of one token tile in order: the tile's tokens and its x rows (the
// MMA's A operand, rounded to bf16) are fetched once and held in registers,
// while the y tile and the B tile of each chunk stream through a 3-stage
// cp.async ring.  CTAs that start at the same chunk index of different
// tiles of one segment share that chunk of B in L2; y, the dominant
// traffic, is read and written exactly once.
//
// Epilogue: the product (mma.sync m16n8k16, fp32 accumulate), the bias and
// the old y are summed in fp32, rounded once to bf16 in place in the shared
// y tile, and the tile leaves with 128-bit coalesced stores.  When y, its
// stride, the offsets or a slice width are not multiples of 8 elements, y
// is not prefetched and a scalar epilogue reads and writes it per element.
#include "lora_expand.cuh"

namespace lora {

template <int KT>
__global__ void __launch_bounds__(EX_THREADS, (KT <= 2) ? 3 : 2) expand_kernel(ExpandArgs p)
{
    using Cfg = ExpandTile<KT>;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_tok[EX_BM];

    // In early mode every CTA still passes the grid-dependency wait before it
    // exits (no tile, no item, or the no-LoRA batch), so the kernel completes
    // only after everything before it in the stream has.
    bool waited = false;
    auto wait_once = [&]() {
        if (!waited) {
            pdl_wait();
            pdl_launch_dependents();
            waited = true;
        }
    };
    if (!p.early) wait_once();

    uint8_t *sA = smem + Cfg::NST * Cfg::STAGE_BYTES;
    const SegTab tab = seg_tab(reinterpret_cast<int *>(sA + Cfg::A_BYTES), p.nbins);
    const int32_t *tokens = p.sorted;
    int total_tiles;
    if (p.num_tokens <= EX_TOKLIST_MAX) {
        // Small batches: the whole sorted token list is loaded together with
        // the segment table (the loads are in flight while the table is
        // read), then kept in shared memory, so no item waits on a token load.
        int pre[EX_TOKLIST_MAX / EX_THREADS];
#pragma unroll
        for (int j = 0; j < EX_TOKLIST_MAX / EX_THREADS; ++j) {
            const int i = threadIdx.x + j * EX_THREADS;
            pre[j] = (i < p.num_tokens) ? p.sorted[i] : 0;
        }
        total_tiles = load_segments(p.no_lora, p.active, p.counts, p.start_loc, p.nbins, EX_BM,
                                    tab, false, 0, p.num_tokens, p.error_word);
        int *s_list = reinterpret_cast<int *>(sA + Cfg::A_BYTES + seg_tab_bytes(p.nbins));
#pragma unroll
        for (int j = 0; j < EX_TOKLIST_MAX / EX_THREADS; ++j) {
            const int i = threadIdx.x + j * EX_THREADS;
            if (i < p.num_tokens) s_list[i] = pre[j];
        }
        __syncthreads();
        tokens = s_list;
    } else {
        total_tiles = load_segments(p.no_lora, p.active, p.counts, p.start_loc, p.nbins, EX_BM,
                                    tab, false, 0, p.num_tokens, p.error_word);
    }
    if (total_tiles == 0) {
        wait_once();
        return;
    }
    // early mode: the grid-dependency wait sits right before the first read
    // of the shrink output
    expand_items<KT, Cfg::NST>(p, tab, tokens, total_tiles, smem, s_tok, [&]() {
        wait_once();
        return true;
    });
    wait_once();                              // a CTA that had no item
}

template <int KT>
static int launch_expand_kt(const ExpandArgs &p, cudaStream_t stream)
{
    static int grid_cache[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return int(e);
    const size_t smem = expand_smem_bytes(KT, LORA_MAX_LORAS + 1) + EX_TOKLIST_MAX * sizeof(int);
    int grid = (dev < 64) ? grid_cache[dev] : 0;
    if (grid == 0) {
        e = cudaFuncSetAttribute(expand_kernel<KT>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return int(e);
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, expand_kernel<KT>, EX_THREADS,
                                                          expand_smem_bytes(KT, 65));
        if (e != cudaSuccess) return int(e);
        grid = device_sm_count() * max(occ, 1);
        if (dev < 64) grid_cache[dev] = grid;
    }
    const size_t used = expand_smem_bytes(KT, p.nbins) +
                        (p.num_tokens <= EX_TOKLIST_MAX ? size_t(p.num_tokens) * sizeof(int) : 0);
    e = launch_kernel(expand_kernel<KT>, dim3(grid), dim3(EX_THREADS), used, stream, p);
    return int(e);
}

static int slice_chunks(int n, int rank)
{
    const int bn = (rank <= 16) ? expand_bn<1>() : (rank <= 32) ? expand_bn<2>()
                 : (rank <= 64) ? expand_bn<4>() : expand_bn<8>();
    return (n + bn - 1) / bn;
}

}  // namespace lora

namespace lora {
int expand_dispatch(ExpandArgs &p, const lora_meta_t *meta, cudaStream_t st);
static int lora_expand_impl(const void *x, int x_bf16, const lora_bf16_t *const *lora_b,
                            const lora_bf16_t *const *lora_bias,
                            const int32_t *slice_sizes, int32_t num_slices, int32_t rank,
                            lora_bf16_t *y, int64_t y_ld, int32_t num_tokens,
                            int32_t offset_start, int32_t add_inputs,
                            const lora_meta_t *meta, cudaStream_t stream, int early);
}  // namespace lora

LORA_API int lora_expand(const float *x, const lora_bf16_t *const *lora_b,
                         const lora_bf16_t *const *lora_bias,
                         const int32_t *slice_sizes, int32_t num_slices, int32_t rank,
                         lora_bf16_t *y, int64_t y_ld, int32_t num_tokens,
                         int32_t offset_start, int32_t add_inputs,
                         const lora_meta_t *meta, void *stream)
{
    lora::NvtxRange nvtx_range("lora_expand");
    return lora::lora_expand_impl(x, 0, lora_b, lora_bias, slice_sizes, num_slices, rank, y,
                                  y_ld, num_tokens, offset_start, add_inputs, meta,
                                  static_cast<cudaStream_t>(stream), 0);
}

// The same product over a bf16 input, which the MMA takes as it is (page
// "vllm.lora.punica_wrapper.punica_gpu", PunicaWrapperGPU.add_lora_embedding:
// the expand of the looked-up rows of an embedding LoRA's A).
LORA_API int lora_expand_bf16(const lora_bf16_t *x, const lora_bf16_t *const *lora_b,
                              const lora_bf16_t *const *lora_bias,
                              const int32_t *slice_sizes, int32_t num_slices, int32_t rank,
                              lora_bf16_t *y, int64_t y_ld, int32_t num_tokens,
                              int32_t offset_start, int32_t add_inputs,
                              const lora_meta_t *meta, void *stream)
{
    lora::NvtxRange nvtx_range("lora_expand_bf16");
    return lora::lora_expand_impl(x, 1, lora_b, lora_bias, slice_sizes, num_slices, rank, y,
                                  y_ld, num_tokens, offset_start, add_inputs, meta,
                                  static_cast<cudaStream_t>(stream), 0);
}

int lora::expand_setup(ExpandArgs &p, const void *x, int x_bf16,
                       const lora_bf16_t *const *lora_b, const lora_bf16_t *const *lora_bias,
                       const int32_t *slice_sizes, int32_t num_slices, int32_t rank,
                       lora_bf16_t *y, int64_t y_ld, int32_t num_tokens, int32_t offset_start,
                       int32_t add_inputs, const lora_meta_t *meta)
{
    if (meta == nullptr || lora_b == nullptr || slice_sizes == nullptr) return LORA_ERR_NULL;
    if (num_slices < 1 || num_slices > LORA_MAX_SLICES) return LORA_ERR_SLICES;
    if (rank < 8 || rank > LORA_MAX_RANK || rank % 8 != 0) return LORA_ERR_RANK;
    if (num_tokens < 0 || offset_start < 0 || y_ld < 0) return LORA_ERR_SIZE;
    if (meta->max_loras < 1 || meta->max_loras > LORA_MAX_LORAS) return LORA_ERR_SIZE;
    if (num_tokens > meta->max_num_tokens) return LORA_ERR_TOKENS;

    int64_t col = offset_start;
    int chunks = 0;
    bool vec = ((reinterpret_cast<uintptr_t>(y) & 15u) == 0) && (y_ld % 8 == 0) &&
               (offset_start % 8 == 0);
    bool bias_vec = true;
    for (int s = 0; s < LORA_MAX_SLICES; ++s) {
        p.b[s] = nullptr;
        p.bias[s] = nullptr;
        p.n[s] = 0;
        p.col0[s] = 0;
        p.chunk0[s] = 0;
    }
    for (int s = 0; s < num_slices; ++s) {
        const int32_t n = slice_sizes[s];
        if (n < 0) return LORA_ERR_SIZE;
        if (lora_b[s] == nullptr) return LORA_ERR_NULL;
        if (reinterpret_cast<uintptr_t>(lora_b[s]) & 15u) return LORA_ERR_ALIGN;
        p.b[s] = lora_b[s];
        p.bias[s] = (lora_bias != nullptr) ? lora_bias[s] : nullptr;
        p.n[s] = n;
        p.col0[s] = int32_t(col);
        p.chunk0[s] = chunks;
        if (n % 8 != 0) vec = false;
        if (p.bias[s] != nullptr && (reinterpret_cast<uintptr_t>(p.bias[s]) & 15u)) bias_vec = false;
        chunks += lora::slice_chunks(n, rank);
        col += n;
        if (col > INT32_MAX) return LORA_ERR_SIZE;
    }
    p.chunk0[num_slices] = chunks;
    if (col > y_ld) return LORA_ERR_WIDTH;
    if (num_tokens == 0 || chunks == 0) return 1;
    if (!x || !y || !meta->token_indices_sorted_by_lora_ids || !meta->num_tokens_per_lora ||
        !meta->lora_token_start_loc || !meta->active_lora_ids || !meta->no_lora_flag)
        return LORA_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(x) & 15u) return LORA_ERR_ALIGN;

    p.x = x;
    p.x_bf16 = x_bf16 ? 1 : 0;
    p.num_slices = num_slices;
    p.rank = rank;
    p.y = y;
    p.y_ld = y_ld;
    p.num_tokens = num_tokens;
    p.add_inputs = add_inputs ? 1 : 0;
    p.vec = vec ? 1 : 0;
    p.bias_vec = (vec && bias_vec) ? 1 : 0;
    p.sorted = meta->token_indices_sorted_by_lora_ids;
    p.counts = meta->num_tokens_per_lora;
    p.start_loc = meta->lora_token_start_loc;
    p.active = meta->active_lora_ids;
    p.no_lora = meta->no_lora_flag;
    p.error_word = meta->error_word;
    p.nbins = meta->max_loras + 1;
    p.early = 0;
    return LORA_OK;
}

static int lora::lora_expand_impl(const void *x, int x_bf16, const lora_bf16_t *const *lora_b,
                                  const lora_bf16_t *const *lora_bias,
                                  const int32_t *slice_sizes, int32_t num_slices, int32_t rank,
                                  lora_bf16_t *y, int64_t y_ld, int32_t num_tokens,
                                  int32_t offset_start, int32_t add_inputs,
                                  const lora_meta_t *meta, cudaStream_t stream, int early)
{
    lora::ExpandArgs p;
    const int r = lora::expand_setup(p, x, x_bf16, lora_b, lora_bias, slice_sizes, num_slices,
                                     rank, y, y_ld, num_tokens, offset_start, add_inputs, meta);
    if (r == 1) return LORA_OK;              // nothing to do
    if (r != LORA_OK) return r;
    p.early = early;
    return lora::expand_dispatch(p, meta, stream);
}

namespace lora {

int expand_dispatch(ExpandArgs &p, const lora_meta_t *meta, cudaStream_t st)
{
    const int num_slices = p.num_slices, rank = p.rank, num_tokens = p.num_tokens;
    lora_bf16_t *y = p.y;
    const int64_t y_ld = p.y_ld;

    // Tensor-core path (tcgen05, TMEM accumulators; lora_expand_tc.cu) for
    // 32-byte-aligned outputs and slice widths that are multiples of 64.  By
    // default (LORA_PUNICA_EXPAND_TC=-1) it takes ranks of at least
    // LORA_PUNICA_EXPAND_TC_MIN_RANK (64): measured, large (rank 128, 16384
    // tokens) 131 against 216 us for the mma.sync kernel, prefill (rank 64)
    // 30.7 against 34.5 us; at lower ranks, with short segments, the
    // mma.sync kernel's 64-token tiles win (MLP, rank 32: 39.7 against
    // 46.1 us; decode, rank 16: 6.9 against 11.3 us).
    // =1 takes it wherever it fits, =0 never, =2 requires it (a call it does
    // not fit fails with LORA_ERR_ALIGN or LORA_ERR_SIZE).
    const int tc_mode = lora::knob_expand_tc();
    if (tc_mode == 2 && !p.vec) return LORA_ERR_ALIGN;
    if (tc_mode != 0 && p.vec &&
        (tc_mode != -1 || rank >= lora::knob_expand_tc_min_rank())) {
        lora::ExpandLaunch u;
        u.x = p.x;
        u.x_bf16 = p.x_bf16;
        u.early = p.early;
        for (int s = 0; s < LORA_MAX_SLICES; ++s) {
            u.b[s] = p.b[s];
            u.bias[s] = p.bias[s];
            u.n[s] = p.n[s];
            u.col0[s] = p.col0[s];
        }
        u.num_slices = num_slices;
        u.rank = rank;
        u.max_loras = meta->max_loras;
        u.y = y;
        u.y_ld = y_ld;
        u.num_tokens = num_tokens;
        u.add_inputs = p.add_inputs;
        u.vec = p.vec;
        u.bias_vec = p.bias_vec;
        u.sorted = p.sorted;
        u.counts = p.counts;
        u.start_loc = p.start_loc;
        u.active = p.active;
        u.no_lora = p.no_lora;
        u.error_word = meta->error_word;
        const int r = lora::launch_expand_tc(u, st);
        if (r == lora::TC_LAUNCHED) return LORA_OK;
        if (r > 0) return r;                                    // a CUDA error
        if (tc_mode == 2) return r == lora::TC_MISALIGNED ? LORA_ERR_ALIGN : LORA_ERR_SIZE;
    }

    if (rank <= 16) return lora::launch_expand_kt<1>(p, st);
    if (rank <= 32) return lora::launch_expand_kt<2>(p, st);
    if (rank <= 64) return lora::launch_expand_kt<4>(p, st);
    return lora::launch_expand_kt<8>(p, st);
}

// lora_expand for lora_linear: the same call in early mode (see ExpandArgs).
int expand_early(const float *x, const lora_bf16_t *const *lora_b,
                 const lora_bf16_t *const *lora_bias, const int32_t *slice_sizes,
                 int32_t num_slices, int32_t rank, lora_bf16_t *y, int64_t y_ld,
                 int32_t num_tokens, const lora_meta_t *meta, cudaStream_t st)
{
    return lora_expand_impl(x, 0, lora_b, lora_bias, slice_sizes, num_slices, rank, y, y_ld,
                            num_tokens, 0, 1, meta, st, 1);
}

}  // namespace lora
