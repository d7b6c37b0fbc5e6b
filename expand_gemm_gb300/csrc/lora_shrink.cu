// lora_shrink.cu -- y[s][t, :] += scale * x[t, :] @ A[s][id(t)]^T
// (page "vllm.lora.punica_wrapper.punica_gpu", PunicaWrapperGPU.add_shrink).
//
// Work item = (token tile of one LoRA segment, slice s, chunk of the hidden
// dimension).  The product is computed "swapped": the r rows of A[s][id]
// are the MMA's M side and the tile's tokens its N side, so a rank of 16
// fills a full m16 tile while a decode segment of ~30 tokens only needs
// n8 tiles.  x rows are gathered through the sorted token permutation with
// 16-byte cp.async into a 4-stage, XOR-swizzled shared-memory ring; A rows
// are contiguous.  mma.sync m16n8k16 (bf16 in, fp32 accumulate).
//
// The grid is persistent (SMs x resident CTAs); every CTA rebuilds the
// segment -> tile table from the metadata and walks items with a grid
// stride, so nothing is read back to the host.  When there are fewer
// (tile, slice) pairs than CTAs the hidden dimension is split into chunks.
// Results are added to y with float4 reductions (red.global.add) in both
// cases: without a split each element has one owner, and the reduction
// adds exactly what a read-modify-write would.
#include "lora_common.cuh"

namespace lora {

constexpr int SH_BN = 64;          // tokens per tile
constexpr int SH_BK = 64;          // hidden elements per stage (128 B rows)
constexpr int SH_STAGES = 4;
constexpr int SH_THREADS = 128;    // 4 warps, 16 tokens each
constexpr int SH_MIN_STEPS = 4;    // smallest hidden chunk, in stages

struct ShrinkArgs {
    const uint16_t *x;
    int64_t x_ld;
    int32_t hidden;
    int32_t num_tokens;
    const uint16_t *a[LORA_MAX_SLICES];
    int32_t num_slices;
    int32_t rank;
    float *y;
    float scale;
    const int32_t *sorted;
    const int32_t *counts;
    const int32_t *start_loc;
    const int32_t *active;
    const int32_t *no_lora;
    int32_t nbins;                 // max_loras + 1
    int32_t *error_word;           // debug checks report here
    int32_t skip_rows;             // rows per segment left to the tensor-core path
    // Self-built metadata (small batches, lora_linear): every CTA sorts the
    // raw id map in shared memory; CTA 0 also writes the metadata buffers.
    const int32_t *map;            // non-null selects this mode
    int32_t *mapping_copy;
    int32_t *sorted_out;
    int32_t *counts_out;
    int32_t *start_out;
    int32_t *active_out;
    int32_t *no_lora_out;
    int32_t *error_out;
    int32_t write_meta;            // CTA 0 writes the metadata buffers
    // Early mode (lora_linear, after its metadata kernel): the ids are sorted
    // and the first tile's loads issued before the grid-dependency wait.
    // Safe because the metadata kernel lets its dependents launch only after
    // its own wait (so the id map, x and A are final), and this kernel reads
    // nothing the metadata kernel writes; it lets its own dependents launch
    // only after that wait, which is what lora_linear's expand relies on.
    int32_t early;
};

constexpr int SH_SELF_META_MAX_TOKENS = 512;

// Extra shared memory of the self-built-metadata mode.
size_t shrink_self_meta_bytes(int nbins)
{
    return size_t(4 * nbins + 3 * nbins + 2 * SH_SELF_META_MAX_TOKENS + 4) * sizeof(int);
}

template <int MT>
struct ShrinkTile {
    static constexpr int RP = 16 * MT;                       // padded rank
    static constexpr int A_BYTES = RP * SH_BK * 2;
    static constexpr int X_BYTES = SH_BN * SH_BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + X_BYTES;
    static constexpr int RING_BYTES = SH_STAGES * STAGE_BYTES;
    static constexpr int OUT_LD = RP + 4;                     // fp32 staging row
    static_assert(SH_BN * OUT_LD * 4 <= RING_BYTES, "staging fits in the ring");
};

size_t shrink_smem_bytes(int mt, int nbins)
{
    size_t ring = 0;
    switch (mt) {
    case 1: ring = ShrinkTile<1>::RING_BYTES; break;
    case 2: ring = ShrinkTile<2>::RING_BYTES; break;
    case 4: ring = ShrinkTile<4>::RING_BYTES; break;
    default: ring = ShrinkTile<8>::RING_BYTES; break;
    }
    return ring + seg_tab_bytes(nbins);
}

template <int MT>
__global__ void __launch_bounds__(SH_THREADS) shrink_kernel(ShrinkArgs p)
{
    using Cfg = ShrinkTile<MT>;
    constexpr int RP = Cfg::RP;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_tok[SH_BN];

    bool waited = false;
    // Every CTA passes the grid-dependency wait before it exits, whichever
    // way it leaves: a kernel's completion then implies the completion of
    // everything before it in the stream, which the expand that follows (it
    // reads the metadata before its own wait) relies on.
    auto wait_once = [&]() {
        if (!waited) {
            pdl_wait();
            pdl_launch_dependents();
            waited = true;
        }
    };
    if (!p.early) wait_once();

    const SegTab tab = seg_tab(reinterpret_cast<int *>(smem + Cfg::RING_BYTES), p.nbins);
    const int32_t *tokens = p.sorted;
    int total_tiles;
    if (p.map != nullptr) {
        int *mm = reinterpret_cast<int *>(smem + Cfg::RING_BYTES + seg_tab_bytes(p.nbins));
        int *cnt = mm, *tot = cnt + 4 * p.nbins, *base = tot + p.nbins, *pos = base + p.nbins;
        int *srt = pos + p.nbins, *ids = srt + SH_SELF_META_MAX_TOKENS;
        int *misc = ids + SH_SELF_META_MAX_TOKENS;
        const bool nl = block_sort_ids<SH_THREADS / 32>(p.map, p.num_tokens, p.nbins - 1, cnt,
                                                        tot, base, pos, srt, misc, ids);
        if (blockIdx.x == 0 && p.write_meta)
            write_meta(p.map, p.num_tokens, p.nbins - 1, nl, tot, base, pos, srt, misc,
                       p.mapping_copy, p.sorted_out, p.counts_out, p.start_out, p.active_out,
                       p.no_lora_out, p.error_out);
        if (nl) {
            wait_once();
            return;
        }
        total_tiles = segments_from_sort(tot, base, p.nbins, SH_BN, tab);
        tokens = srt;
    } else {
        total_tiles = load_segments(p.no_lora, p.active, p.counts, p.start_loc,
                                    p.nbins, SH_BN, tab, false, p.skip_rows, p.num_tokens,
                                    p.error_word);
    }
    if (total_tiles == 0) {
        wait_once();
        return;
    }

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = p.num_slices, H = p.hidden, T = p.num_tokens, R = p.rank;
    const int nk = (H + SH_BK - 1) / SH_BK;

    // Split of the hidden dimension: as many chunks as keep every CTA busy,
    // but never shorter than SH_MIN_STEPS stages.
    const int pairs = total_tiles * S;
    int kchunks = 1;
    if (pairs < int(gridDim.x)) {
        kchunks = min(int(gridDim.x) / pairs, max(1, nk / SH_MIN_STEPS));
        kchunks = max(kchunks, 1);
    }
    const int steps_per_chunk = (nk + kchunks - 1) / kchunks;
    kchunks = (nk + steps_per_chunk - 1) / steps_per_chunk;
    const int total_items = pairs * kchunks;

    const uint32_t ring = smem_addr(smem);

    for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
        const int s = item % S;
        const int rest = item / S;
        const int tile = rest % total_tiles;
        const int kc = rest / total_tiles;

        const int seg = find_segment(tab.tile, p.nbins, tile);
        const int id = tab.id[seg];
        const int row0 = tab.start[seg] + (tile - tab.tile[seg]) * SH_BN;
        const int nrows = min(SH_BN, tab.start[seg] + tab.count[seg] - row0);
        if (tid < SH_BN)
            s_tok[tid] = (tid < nrows) ? checked_token(tokens[row0 + tid], T, p.error_word) : -1;
        __syncthreads();

        const int k_first = kc * steps_per_chunk;
        const int k_steps = min(steps_per_chunk, nk - k_first);

        // Per-thread load assignment (fixed for the item):
        //   x tile: 64 rows x 8 chunks = 512 chunks, 4 per thread, rows tid/8 + 16j
        //   A tile: RP rows x 8 chunks, MT*... chunks per thread
        const int xc = tid & 7;
        const uint16_t *xrow[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = (tid >> 3) + 16 * j;
            const int t = s_tok[r];
            xrow[j] = (t >= 0) ? p.x + int64_t(t) * p.x_ld : nullptr;
        }
        const uint16_t *abase = p.a[s] + int64_t(id) * R * H;

        auto load_stage = [&](int kstep, int slot) {
            const uint32_t sa = ring + slot * Cfg::STAGE_BYTES;
            const uint32_t sx = sa + Cfg::A_BYTES;
            const int k0 = kstep * SH_BK + xc * 8;
            const bool kin = k0 < H;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = (tid >> 3) + 16 * j;
                const bool ok = kin && xrow[j] != nullptr;
                cp_async16(sx + swz<8>(r, xc), ok ? xrow[j] + k0 : p.x, ok);
            }
#pragma unroll
            for (int j = 0; j < (RP * 8) / SH_THREADS; ++j) {
                const int r = (tid >> 3) + 16 * j;
                const bool ok = kin && r < R;
                cp_async16(sa + swz<8>(r, xc), ok ? abase + int64_t(r) * H + k0 : p.x, ok);
            }
        };

        float acc[MT][2][4];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[m][n][q] = 0.f;

#pragma unroll
        for (int st = 0; st < SH_STAGES - 1; ++st) {
            if (st < k_steps) load_stage(k_first + st, st);
            cp_async_commit();
        }

        wait_once();                          // y (the buffer) is written from here on
        for (int ks = 0; ks < k_steps; ++ks) {
            cp_async_wait<SH_STAGES - 2>();
            __syncthreads();
            {
                const int nxt = ks + SH_STAGES - 1;
                if (nxt < k_steps) load_stage(k_first + nxt, nxt % SH_STAGES);
                cp_async_commit();
            }
            const uint32_t sa = ring + (ks % SH_STAGES) * Cfg::STAGE_BYTES;
            const uint32_t sx = sa + Cfg::A_BYTES;
#pragma unroll
            for (int kk = 0; kk < SH_BK / 16; ++kk) {
                // B operand: this warp's 16 tokens x k16 (two n8 tiles).
                uint32_t b[4];
                {
                    const int q = lane >> 3;
                    const int n = warp * 16 + (q >> 1) * 8 + (lane & 7);
                    const int c = kk * 2 + (q & 1);
                    ldmatrix_x4(sx + swz<8>(n, c), b[0], b[1], b[2], b[3]);
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    uint32_t af[4];
                    const int r = m * 16 + (lane & 15);
                    const int c = kk * 2 + (lane >> 4);
                    ldmatrix_x4(sa + swz<8>(r, c), af[0], af[1], af[2], af[3]);
                    mma_bf16_16816(acc[m][0], af, b[0], b[1]);
                    mma_bf16_16816(acc[m][1], af, b[2], b[3]);
                }
            }
        }
        cp_async_wait<0>();
        __syncthreads();

        // Stage scale * acc as [token][rank] fp32, then write rows with float4.
        float *stage = reinterpret_cast<float *>(smem);
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const int r = m * 16 + (lane >> 2);
                const int t = warp * 16 + n * 8 + 2 * (lane & 3);
                stage[t * Cfg::OUT_LD + r] = acc[m][n][0] * p.scale;
                stage[(t + 1) * Cfg::OUT_LD + r] = acc[m][n][1] * p.scale;
                stage[t * Cfg::OUT_LD + r + 8] = acc[m][n][2] * p.scale;
                stage[(t + 1) * Cfg::OUT_LD + r + 8] = acc[m][n][3] * p.scale;
            }
        __syncthreads();

        const int r4n = R / 4;
        for (int i = tid; i < SH_BN * r4n; i += SH_THREADS) {
            const int t = i / r4n, c4 = i - t * r4n;
            const int tok = s_tok[t];
            if (tok < 0) continue;
            const float4 v = *reinterpret_cast<const float4 *>(&stage[t * Cfg::OUT_LD + 4 * c4]);
            float4 *dst = reinterpret_cast<float4 *>(p.y + (int64_t(s) * T + tok) * R) + c4;
            // a reduction (red.global.add), nothing read back: with one
            // owner per element (no split) it adds exactly what a
            // read-modify-write would, without the load's latency
            atomicAdd(dst, v);
        }
        __syncthreads();
    }
    wait_once();                              // a CTA that had no item
}

template <int MT>
static int launch_shrink_mt(const ShrinkArgs &p, cudaStream_t stream)
{
    static int grid_cache[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return int(e);
    const size_t smem = shrink_smem_bytes(MT, LORA_MAX_LORAS + 1) +
                        shrink_self_meta_bytes(LORA_MAX_LORAS + 1);
    int grid = (dev < 64) ? grid_cache[dev] : 0;
    if (grid == 0) {
        e = cudaFuncSetAttribute(shrink_kernel<MT>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return int(e);
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, shrink_kernel<MT>, SH_THREADS,
                                                          shrink_smem_bytes(MT, 65));
        if (e != cudaSuccess) return int(e);
        grid = device_sm_count() * max(occ, 1);
        if (dev < 64) grid_cache[dev] = grid;
    }
    const size_t used = shrink_smem_bytes(MT, p.nbins) +
                        (p.map != nullptr ? shrink_self_meta_bytes(p.nbins) : 0);
    // In early mode (small batches inside lora_linear) at most
    // LORA_PUNICA_EARLY_SHRINK_CTAS CTAs per SM, so that one CTA of the
    // expand that follows fits beside them and starts loading.  Two was
    // measured best on 256-token q/k/v decode (14.9 us a step, against 15.3
    // with one and 15.4 with three).
    if (p.early)
        grid = min(grid, max(1, knobs().early_shrink_ctas) * device_sm_count());
    e = launch_kernel(shrink_kernel<MT>, dim3(grid), dim3(SH_THREADS), used, stream, p);
    return int(e);
}

}  // namespace lora

LORA_API int lora_shrink(const lora_bf16_t *x, int32_t num_tokens, int32_t hidden,
                         int64_t x_ld, const lora_bf16_t *const *lora_a,
                         int32_t num_slices, int32_t rank, float *y,
                         const lora_meta_t *meta, float scale, void *stream)
{
    lora::NvtxRange nvtx_range("lora_shrink");
    if (meta == nullptr || lora_a == nullptr) return LORA_ERR_NULL;
    if (num_slices < 1 || num_slices > LORA_MAX_SLICES) return LORA_ERR_SLICES;
    if (rank < 8 || rank > LORA_MAX_RANK || rank % 8 != 0) return LORA_ERR_RANK;
    if (num_tokens < 0 || hidden < 0 || x_ld < hidden) return LORA_ERR_SIZE;
    if (meta->max_loras < 1 || meta->max_loras > LORA_MAX_LORAS) return LORA_ERR_SIZE;
    if (num_tokens > meta->max_num_tokens) return LORA_ERR_TOKENS;
    if (num_tokens == 0 || hidden == 0) return LORA_OK;
    if (!x || !y || !meta->token_indices_sorted_by_lora_ids || !meta->num_tokens_per_lora ||
        !meta->lora_token_start_loc || !meta->active_lora_ids || !meta->no_lora_flag)
        return LORA_ERR_NULL;
    if (hidden % 8 != 0 || x_ld % 8 != 0) return LORA_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u)
        return LORA_ERR_ALIGN;

    lora::ShrinkArgs p;
    lora::ShrinkLaunch u;
    for (int s = 0; s < LORA_MAX_SLICES; ++s) p.a[s] = u.a[s] = nullptr;
    for (int s = 0; s < num_slices; ++s) {
        if (lora_a[s] == nullptr) return LORA_ERR_NULL;
        if (reinterpret_cast<uintptr_t>(lora_a[s]) & 15u) return LORA_ERR_ALIGN;
        p.a[s] = u.a[s] = lora_a[s];
    }
    p.x = x;
    p.x_ld = x_ld;
    p.hidden = hidden;
    p.num_tokens = num_tokens;
    p.num_slices = num_slices;
    p.rank = rank;
    p.y = y;
    p.scale = scale;
    p.sorted = meta->token_indices_sorted_by_lora_ids;
    p.counts = meta->num_tokens_per_lora;
    p.start_loc = meta->lora_token_start_loc;
    p.active = meta->active_lora_ids;
    p.no_lora = meta->no_lora_flag;
    p.nbins = meta->max_loras + 1;
    p.error_word = meta->error_word;
    p.skip_rows = 0;
    p.map = nullptr;
    p.write_meta = 0;
    p.early = 0;

    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // Tensor-core path for the 128-token tiles of long segments.  It
    // pays where the contraction is dense enough to outrun mma.sync: a batch
    // large enough to hold long segments (LORA_PUNICA_UMMA_MIN_TOKENS,
    // default 1024) and at least LORA_PUNICA_UMMA_MIN_COLS output columns per
    // token over all slices (num_slices * rank, default 256).
    // LORA_PUNICA_UMMA=0 turns it off.  The variables are read at each call.
    const lora::Knobs &kn = lora::knobs();
    const int umma_on = kn.umma;
    const int umma_min_tokens = kn.umma_min_tokens;
    const int umma_min_cols = kn.umma_min_cols;
    if (umma_on && num_tokens >= umma_min_tokens && num_slices * rank >= umma_min_cols &&
        meta->error_word != nullptr) {
        u.x = x;
        u.x_ld = x_ld;
        u.hidden = hidden;
        u.num_tokens = num_tokens;
        u.num_slices = num_slices;
        u.rank = rank;
        u.max_loras = meta->max_loras;
        u.y = y;
        u.scale = scale;
        u.sorted = p.sorted;
        u.counts = p.counts;
        u.start_loc = p.start_loc;
        u.active = p.active;
        u.no_lora = p.no_lora;
        u.error_word = meta->error_word;
        // LORA_PUNICA_UMMA_PARTIAL=1 (default): the tensor-core kernel takes
        // the partial tile at the end of every segment too, and covers the
        // whole batch; =0: whole tiles only, the remainders on mma.sync.
        u.partial = kn.umma_partial ? 1 : 0;
        const int r = lora::launch_shrink_umma(u, st);
        if (r == 1 && u.partial) return LORA_OK;
        if (r == 1) p.skip_rows = 128;
        else if (r != 0) return r;
    }

    if (rank <= 16) return lora::launch_shrink_mt<1>(p, st);
    if (rank <= 32) return lora::launch_shrink_mt<2>(p, st);
    if (rank <= 64) return lora::launch_shrink_mt<4>(p, st);
    return lora::launch_shrink_mt<8>(p, st);
}

namespace lora {

// lora_shrink for lora_linear on small batches: the kernel sorts the raw id
// map itself.  early == 0: no separate metadata kernel runs and CTA 0 writes
// the metadata buffers exactly as lora_meta_prepare would.  early == 1: the
// metadata kernel runs just before and writes them; this kernel sorts and
// starts loading while it runs (see ShrinkArgs::early).  Returns 0 when it does not
// apply (the caller then runs the metadata kernel and lora_shrink), 1 when
// launched, or an error status.
int shrink_self_meta(const int32_t *map, const lora_bf16_t *x, int32_t num_tokens,
                     int32_t hidden, int64_t x_ld, const lora_bf16_t *const *lora_a,
                     int32_t num_slices, int32_t rank, float *y, const lora_meta_t *meta,
                     float scale, cudaStream_t st, int early)
{
    if (num_tokens < 1 || num_tokens > SH_SELF_META_MAX_TOKENS || meta->max_loras > 256)
        return 0;
    if (num_slices < 1 || num_slices > LORA_MAX_SLICES || rank < 8 || rank > LORA_MAX_RANK ||
        rank % 8 != 0 || hidden < 8 || hidden % 8 != 0 || x_ld % 8 != 0 || x_ld < hidden)
        return 0;
    if (!map || !x || !y || !meta->token_lora_mapping || !meta->token_indices_sorted_by_lora_ids ||
        !meta->num_tokens_per_lora || !meta->lora_token_start_loc || !meta->active_lora_ids ||
        !meta->no_lora_flag || !meta->error_word)
        return 0;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) return 0;
    ShrinkArgs p;
    for (int s = 0; s < LORA_MAX_SLICES; ++s) p.a[s] = nullptr;
    for (int s = 0; s < num_slices; ++s) {
        if (lora_a[s] == nullptr || (reinterpret_cast<uintptr_t>(lora_a[s]) & 15u)) return 0;
        p.a[s] = lora_a[s];
    }
    p.x = x;
    p.x_ld = x_ld;
    p.hidden = hidden;
    p.num_tokens = num_tokens;
    p.num_slices = num_slices;
    p.rank = rank;
    p.y = y;
    p.scale = scale;
    p.sorted = nullptr;
    p.counts = nullptr;
    p.start_loc = nullptr;
    p.active = nullptr;
    p.no_lora = nullptr;
    p.nbins = meta->max_loras + 1;
    p.error_word = meta->error_word;
    p.skip_rows = 0;
    p.map = map;
    p.mapping_copy = meta->token_lora_mapping;
    p.sorted_out = meta->token_indices_sorted_by_lora_ids;
    p.counts_out = meta->num_tokens_per_lora;
    p.start_out = meta->lora_token_start_loc;
    p.active_out = meta->active_lora_ids;
    p.no_lora_out = meta->no_lora_flag;
    p.error_out = meta->error_word;
    // early == 1: the metadata kernel writes the buffers, and the loads start
    // before the grid-dependency wait.  Otherwise CTA 0 writes them.
    p.write_meta = early == 1 ? 0 : 1;
    p.early = early == 1 ? 1 : 0;
    int r;
    if (rank <= 16) r = launch_shrink_mt<1>(p, st);
    else if (rank <= 32) r = launch_shrink_mt<2>(p, st);
    else if (rank <= 64) r = launch_shrink_mt<4>(p, st);
    else r = launch_shrink_mt<8>(p, st);
    return r == 0 ? 1 : r;
}

}  // namespace lora

