// lora_expand.cu -- y[t, off_s + j] (+)= x[s][t, :] @ B[s][id(t)][j, :] +
// bias[s][id(t)][j]  (page "vllm.lora.punica_wrapper.punica_gpu",
// PunicaWrapperGPU.add_expand; bias step of page
// "vllm.lora.punica_wrapper.punica_tpu", PunicaWrapperTPU._apply_bias).
//
// Work item = (token tile of one LoRA segment, 128-column chunk of one
// slice).  Items are numbered tile-fastest, so the CTAs resident at one
// time share the same B chunk (read once from HBM, then from L2) while the
// y rows, the dominant traffic, stream through exactly once.
//
// Per item: the y tile (64 rows x 128 columns, bf16) is fetched with
// 16-byte cp.async into shared memory at the start, overlapping the B tile
// and the fp32 x tile; x is rounded to bf16 while it is staged (the rank-r
// contraction then runs on mma.sync m16n8k16 with fp32 accumulation).  The
// epilogue adds bias and the old y in fp32, rounds once to bf16 in place in
// the shared y tile, and the tile leaves with 128-bit coalesced stores.
// When y, its stride, the offsets or a slice width are not multiples of 8
// elements, a scalar epilogue reads and writes y element by element.
#include "lora_common.cuh"

namespace lora {

constexpr int EX_BM = 64;          // tokens per tile
constexpr int EX_BN = 128;         // output columns per item
constexpr int EX_THREADS = 256;    // 8 warps: 2 (rows) x 4 (columns), 32x32 each
constexpr int EX_Y_LD = EX_BN * 2 + 16;   // bytes per shared y row (padded)

struct ExpandArgs {
    const float *x;
    const uint16_t *b[LORA_MAX_SLICES];
    const uint16_t *bias[LORA_MAX_SLICES];
    int32_t n[LORA_MAX_SLICES];          // slice widths
    int32_t col0[LORA_MAX_SLICES];       // off_s
    int32_t chunk0[LORA_MAX_SLICES + 1]; // first column chunk of each slice
    int32_t num_slices;
    int32_t rank;
    uint16_t *y;
    int64_t y_ld;
    int32_t num_tokens;
    int32_t add_inputs;
    int32_t vec;                         // 16-byte epilogue allowed
    const int32_t *sorted;
    const int32_t *counts;
    const int32_t *start_loc;
    const int32_t *active;
    const int32_t *no_lora;
    int32_t nbins;
};

template <int KT>
struct ExpandTile {
    static constexpr int RP = 16 * KT;                 // padded rank
    static constexpr int CPR = RP / 8;                 // 16-byte chunks per row
    static constexpr int A_BYTES = EX_BM * RP * 2;     // bf16 x tile
    static constexpr int B_BYTES = EX_BN * RP * 2;     // bf16 B tile
    static constexpr int Y_BYTES = EX_BM * EX_Y_LD;
    static constexpr int BIAS_BYTES = EX_BN * 4;
    static constexpr int BYTES = A_BYTES + B_BYTES + Y_BYTES + BIAS_BYTES;
};

size_t expand_smem_bytes(int kt, int nbins)
{
    size_t t = 0;
    switch (kt) {
    case 1: t = ExpandTile<1>::BYTES; break;
    case 2: t = ExpandTile<2>::BYTES; break;
    case 4: t = ExpandTile<4>::BYTES; break;
    default: t = ExpandTile<8>::BYTES; break;
    }
    return t + size_t(nbins + 1) * sizeof(int);
}

template <int KT>
__global__ void __launch_bounds__(EX_THREADS) expand_kernel(ExpandArgs p)
{
    using Cfg = ExpandTile<KT>;
    constexpr int CPR = Cfg::CPR;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_tok[EX_BM];

    if (*p.no_lora) return;

    uint8_t *sA = smem;
    uint8_t *sB = sA + Cfg::A_BYTES;
    uint8_t *sY = sB + Cfg::B_BYTES;
    float *sBias = reinterpret_cast<float *>(sY + Cfg::Y_BYTES);
    int *s_tile = reinterpret_cast<int *>(smem + Cfg::BYTES);

    const int total_tiles = build_tile_table(p.active, p.counts, p.nbins, EX_BM, s_tile);
    if (total_tiles == 0) return;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm = warp >> 2, wn = warp & 3;
    const int S = p.num_slices, R = p.rank, T = p.num_tokens;
    const int total_items = total_tiles * p.chunk0[S];
    const uint32_t aA = smem_addr(sA), aB = smem_addr(sB), aY = smem_addr(sY);

    for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
        const int tile = item % total_tiles;
        const int chunk = item / total_tiles;
        int s = 0;
        while (s + 1 < S && p.chunk0[s + 1] <= chunk) ++s;
        const int n_s = p.n[s];
        const int c0 = (chunk - p.chunk0[s]) * EX_BN;        // first column in the slice
        const int ncols = min(EX_BN, n_s - c0);

        const int seg = find_segment(s_tile, p.nbins, tile);
        const int id = p.active[seg];
        const int row0 = p.start_loc[seg] + (tile - s_tile[seg]) * EX_BM;
        const int nrows = min(EX_BM, p.start_loc[seg] + p.counts[seg] - row0);
        if (tid < EX_BM) s_tok[tid] = (tid < nrows) ? p.sorted[row0 + tid] : -1;
        if (tid < EX_BN) {
            const uint16_t *bb = p.bias[s];
            sBias[tid] = (bb != nullptr && tid < ncols)
                             ? bf16_to_f32(bb[int64_t(id) * n_s + c0 + tid]) : 0.f;
        }
        __syncthreads();

        uint16_t *ybase = p.y + p.col0[s] + c0;              // + tok * y_ld

        // (1) y tile -> shared (vector path, add_inputs only).
        if (p.vec && p.add_inputs) {
            for (int i = tid; i < EX_BM * (EX_BN / 8); i += EX_THREADS) {
                const int r = i >> 4, c = i & 15;
                const int tok = s_tok[r];
                const bool ok = tok >= 0 && c * 8 < ncols;
                cp_async16(aY + r * EX_Y_LD + c * 16,
                           ok ? ybase + int64_t(tok) * p.y_ld + c * 8 : p.y, ok);
            }
        }
        // (2) B tile: 128 rows (columns of the slice) x RP, zero past n_s / R.
        {
            const uint16_t *bbase = p.b[s] + (int64_t(id) * n_s + c0) * R;
            for (int i = tid; i < EX_BN * CPR; i += EX_THREADS) {
                const int r = i / CPR, c = i - r * CPR;
                const bool ok = r < ncols && c * 8 < R;
                cp_async16(aB + swz<CPR>(r, c), ok ? bbase + int64_t(r) * R + c * 8 : p.b[s], ok);
            }
        }
        cp_async_commit();
        // (3) x tile: fp32 rows of the shrink output, rounded to bf16.
        {
            const float *xs = p.x + int64_t(s) * T * R;
            for (int i = tid; i < EX_BM * CPR; i += EX_THREADS) {
                const int r = i / CPR, c = i - r * CPR;
                const int tok = s_tok[r];
                uint4 v = make_uint4(0, 0, 0, 0);
                if (tok >= 0 && c * 8 < R) {
                    const float4 *src = reinterpret_cast<const float4 *>(xs + int64_t(tok) * R + c * 8);
                    const float4 u = src[0], w = src[1];
                    v.x = pack_bf16x2(u.x, u.y);
                    v.y = pack_bf16x2(u.z, u.w);
                    v.z = pack_bf16x2(w.x, w.y);
                    v.w = pack_bf16x2(w.z, w.w);
                }
                *reinterpret_cast<uint4 *>(sA + swz<CPR>(r, c)) = v;
            }
        }
        cp_async_wait<0>();
        __syncthreads();

        // (4) 64 x 128 x RP on the tensor cores.
        float acc[2][4][4];
#pragma unroll
        for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[m][n][q] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KT; ++kk) {
            uint32_t af[2][4];
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                const int r = wm * 32 + m * 16 + (lane & 15);
                const int c = kk * 2 + (lane >> 4);
                ldmatrix_x4(aA + swz<CPR>(r, c), af[m][0], af[m][1], af[m][2], af[m][3]);
            }
#pragma unroll
            for (int n2 = 0; n2 < 2; ++n2) {
                uint32_t b[4];
                const int q = lane >> 3;
                const int r = wn * 32 + n2 * 16 + (q >> 1) * 8 + (lane & 7);
                const int c = kk * 2 + (q & 1);
                ldmatrix_x4(aB + swz<CPR>(r, c), b[0], b[1], b[2], b[3]);
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    mma_bf16_16816(acc[m][2 * n2], af[m], b[0], b[1]);
                    mma_bf16_16816(acc[m][2 * n2 + 1], af[m], b[2], b[3]);
                }
            }
        }

        // (5) epilogue.
        if (p.vec) {
            // Combine in place in the shared y tile, then 16-byte stores.
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int n = 0; n < 4; ++n)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int r = wm * 32 + m * 16 + (lane >> 2) + 8 * h;
                        const int c = wn * 32 + n * 8 + 2 * (lane & 3);
                        uint32_t *cell = reinterpret_cast<uint32_t *>(sY + r * EX_Y_LD + c * 2);
                        float v0 = acc[m][n][2 * h] + sBias[c];
                        float v1 = acc[m][n][2 * h + 1] + sBias[c + 1];
                        if (p.add_inputs) {
                            const uint32_t old = *cell;
                            v0 += bf16_lo(old);
                            v1 += bf16_hi(old);
                        }
                        *cell = pack_bf16x2(v0, v1);
                    }
            __syncthreads();
            for (int i = tid; i < EX_BM * (EX_BN / 8); i += EX_THREADS) {
                const int r = i >> 4, c = i & 15;
                const int tok = s_tok[r];
                if (tok < 0 || c * 8 >= ncols) continue;
                const uint4 v = *reinterpret_cast<const uint4 *>(sY + r * EX_Y_LD + c * 16);
                *reinterpret_cast<uint4 *>(ybase + int64_t(tok) * p.y_ld + c * 8) = v;
            }
        } else {
#pragma unroll
            for (int m = 0; m < 2; ++m)
#pragma unroll
                for (int n = 0; n < 4; ++n)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int r = wm * 32 + m * 16 + (lane >> 2) + 8 * (q >> 1);
                        const int c = wn * 32 + n * 8 + 2 * (lane & 3) + (q & 1);
                        const int tok = s_tok[r];
                        if (tok < 0 || c >= ncols) continue;
                        uint16_t *dst = ybase + int64_t(tok) * p.y_ld + c;
                        float v = acc[m][n][q] + sBias[c];
                        if (p.add_inputs) v += bf16_to_f32(*dst);
                        *dst = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu);
                    }
        }
        __syncthreads();
    }
}

template <int KT>
static int launch_expand_kt(const ExpandArgs &p, cudaStream_t stream)
{
    static int grid_cache[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return int(e);
    const size_t smem = expand_smem_bytes(KT, LORA_MAX_LORAS + 1);
    int grid = (dev < 64) ? grid_cache[dev] : 0;
    if (grid == 0) {
        e = cudaFuncSetAttribute(expand_kernel<KT>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return int(e);
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, expand_kernel<KT>,
                                                          EX_THREADS, smem);
        if (e != cudaSuccess) return int(e);
        grid = device_sm_count() * max(occ, 1);
        if (dev < 64) grid_cache[dev] = grid;
    }
    expand_kernel<KT><<<grid, EX_THREADS, expand_smem_bytes(KT, p.nbins), stream>>>(p);
    return int(cudaGetLastError());
}

}  // namespace lora

LORA_API int lora_expand(const float *x, const lora_bf16_t *const *lora_b,
                         const lora_bf16_t *const *lora_bias,
                         const int32_t *slice_sizes, int32_t num_slices, int32_t rank,
                         lora_bf16_t *y, int64_t y_ld, int32_t num_tokens,
                         int32_t offset_start, int32_t add_inputs,
                         const lora_meta_t *meta, void *stream)
{
    if (meta == nullptr || lora_b == nullptr || slice_sizes == nullptr) return LORA_ERR_NULL;
    if (num_slices < 1 || num_slices > LORA_MAX_SLICES) return LORA_ERR_SLICES;
    if (rank < 8 || rank > LORA_MAX_RANK || rank % 8 != 0) return LORA_ERR_RANK;
    if (num_tokens < 0 || offset_start < 0 || y_ld < 0) return LORA_ERR_SIZE;
    if (meta->max_loras < 1 || meta->max_loras > LORA_MAX_LORAS) return LORA_ERR_SIZE;
    if (num_tokens > meta->max_num_tokens) return LORA_ERR_TOKENS;

    lora::ExpandArgs p;
    int64_t col = offset_start;
    int chunks = 0;
    bool vec = ((reinterpret_cast<uintptr_t>(y) & 15u) == 0) && (y_ld % 8 == 0) &&
               (offset_start % 8 == 0);
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
        chunks += (n + lora::EX_BN - 1) / lora::EX_BN;
        col += n;
    }
    p.chunk0[num_slices] = chunks;
    if (col > y_ld) return LORA_ERR_WIDTH;
    if (num_tokens == 0 || chunks == 0) return LORA_OK;
    if (!x || !y || !meta->token_indices_sorted_by_lora_ids || !meta->num_tokens_per_lora ||
        !meta->lora_token_start_loc || !meta->active_lora_ids || !meta->no_lora_flag)
        return LORA_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(x) & 15u) return LORA_ERR_ALIGN;

    p.x = x;
    p.num_slices = num_slices;
    p.rank = rank;
    p.y = y;
    p.y_ld = y_ld;
    p.num_tokens = num_tokens;
    p.add_inputs = add_inputs ? 1 : 0;
    p.vec = vec ? 1 : 0;
    p.sorted = meta->token_indices_sorted_by_lora_ids;
    p.counts = meta->num_tokens_per_lora;
    p.start_loc = meta->lora_token_start_loc;
    p.active = meta->active_lora_ids;
    p.no_lora = meta->no_lora_flag;
    p.nbins = meta->max_loras + 1;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (rank <= 16) return lora::launch_expand_kt<1>(p, st);
    if (rank <= 32) return lora::launch_expand_kt<2>(p, st);
    if (rank <= 64) return lora::launch_expand_kt<4>(p, st);
    return lora::launch_expand_kt<8>(p, st);
}
