// lora_shrink_umma.cu -- tensor-core (tcgen05 / TMEM) path of lora_shrink
// for the 128-token tiles of long LoRA segments, the partial last tile of
// each segment included (page
// "vllm.lora.punica_wrapper.punica_gpu", PunicaWrapperGPU.add_shrink:
// y[s][t, :] += scale * x[t, :] @ A[s][id(t)]^T).
//
// One CTA per SM, persistent over (tile, hidden chunk) items: the hidden
// dimension is split when there are too few whole tiles to fill the GPU
// (see shrink_kchunks).  Warp-specialised:
//   warp 0      x producer: per 64-wide hidden block, the tile's 128 x rows
//               arrive by 2-D TMA: the tile's tokens (increasing, as the
//               sort is stable) are cut into runs of consecutive tokens and
//               each run into power-of-two pieces, one TMA box per piece
//               (a long prefill sequence makes the tile one 128-row box).
//   warps 6..8  A producers: one 2-D TMA box per slice brings the r rows of
//               A[s][id], slice s issued by warp 6 + s % 3.  Each producer
//               arrives on the stage's mbarrier with the bytes it loads, so
//               a stage completes when all of them have landed.  One thread
//               issuing every box was measured to hold the kernel at its TMA
//               issue rate (on this GPU about 1000 cycles of latency per box
//               for each issuing thread); several issuers overlap them.
//               (Per-row TMA tile::gather4 and an LSU cp.async gather were
//               both measured slower: they stay near 30 GB/s per SM.)
//   warp 1      allocates TMEM; lane 0 issues tcgen05.mma (M = 128 tokens,
//               N = padded rank, K = 16) for every slice into its own TMEM
//               columns, and commits to free each stage and, at the end of
//               a tile, to hand the accumulators to the epilogue.
//   warps 2..5  epilogue: tcgen05.ld of their 32 TMEM lanes (one token row
//               per thread), buf[s][t, :] += scale * acc with float4
//               reductions (red.global.add; see shrink_epilogue_row), also
//               when the tile's hidden dimension is split over several CTAs.
// x is read once per tile for all slices; the A block of a LoRA is shared in
// L2 by the CTAs working on tiles of the same segment.
//
// Every mbarrier wait is bounded (about one second); on expiry the kernel
// sets bit 30 of the metadata error word, stops issuing, waits (bounded)
// for its copies and MMAs in flight, frees TMEM and returns.
#include "lora_common.cuh"
#include "lora_umma.cuh"

namespace lora {

constexpr int UM_BM = 128;            // tokens per tile = UMMA M
constexpr int UM_BK = 64;             // hidden per stage (one 128-byte swizzle atom)
constexpr int UM_MMA_WARP = 1;        // warp 0: x producer; warp 1: TMEM owner, UMMA issue
constexpr int UM_APROD0 = 6;          // warps 2..5: epilogue; warps 6..8: A producers
constexpr int UM_APRODS = 3;
constexpr int UM_THREADS = 32 * (UM_APROD0 + UM_APRODS);
constexpr int UM_XMAPS = 8;           // x box heights 1, 2, 4, ..., 128
constexpr int UM_MAX_STAGES = 8;
constexpr int UM_SMEM_BUDGET = 200 * 1024;
constexpr long long UM_TIMEOUT_CYCLES = 2000000000ll;
constexpr int UM_ERROR_BIT = 1 << 30;
constexpr int UM_MIN_BLOCKS = 8;      // shortest hidden chunk of a split item

struct UmmaShrinkArgs {
    CUtensorMap map_x[UM_XMAPS];               // x: [T, H], box {64, 2^i rows}
    CUtensorMap map_a[LORA_MAX_SLICES];        // A[s]: [L * r, H], box {64, RP}
    float *y;
    float scale;
    int32_t num_tokens;
    int32_t hidden;
    int32_t num_slices;
    int32_t rank;
    int32_t rp;                                // padded rank (UMMA N), power of 2
    int32_t stages;
    int32_t tmem_cols;
    const int32_t *sorted;
    const int32_t *counts;
    const int32_t *start_loc;
    const int32_t *active;
    const int32_t *no_lora;
    int32_t *error_word;
    int32_t nbins;
    int32_t partial;                           // take partial tiles too (else whole ones only)
};

struct UmmaLayout {
    int x_bytes, a_bytes, stage_bytes, ring_bytes, bar_off, misc_off, piece_off, tab_off, total;
};

__host__ __device__ inline UmmaLayout umma_layout(int S, int rp, int stages, int nbins)
{
    UmmaLayout l;
    l.x_bytes = UM_BM * UM_BK * 2;                       // 16 KB
    l.a_bytes = rp * UM_BK * 2;                          // per slice
    l.stage_bytes = l.x_bytes + S * l.a_bytes;
    l.ring_bytes = stages * l.stage_bytes;
    l.bar_off = l.ring_bytes;                            // 2 * stages + 3 mbarriers
    l.misc_off = l.bar_off + (2 * UM_MAX_STAGES + 3) * 8; // tmem base, abort flag
    l.piece_off = l.misc_off + 16;                      // [UM_BM] (row, token, log2 rows)
    l.tab_off = l.piece_off + UM_BM * 4;
    l.total = l.tab_off + int(seg_tab_bytes(nbins)) + 1024;   // + alignment slack
    return l;
}

__global__ void __launch_bounds__(UM_THREADS, 1) shrink_umma_kernel(const __grid_constant__ UmmaShrinkArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms.
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.num_slices, RP = p.rp, STAGES = p.stages;
    const UmmaLayout L = umma_layout(S, RP, STAGES, p.nbins);
    const uint32_t base = smem_addr(smem);
    const uint32_t bar_full = base + L.bar_off;                 // [STAGES]
    const uint32_t bar_empty = bar_full + 8 * UM_MAX_STAGES;    // [STAGES]
    const uint32_t bar_acc_full = bar_empty + 8 * UM_MAX_STAGES;
    const uint32_t bar_acc_empty = bar_acc_full + 8;
    const uint32_t bar_drain = bar_acc_empty + 8;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + L.misc_off + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    pdl_wait();
    pdl_launch_dependents();

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            // one expect_tx arrival from the x producer and one from each A
            // producer that has a slice
            mbar_init(bar_full + 8 * i, 1 + min(S, UM_APRODS));
            mbar_init(bar_empty + 8 * i, 1);
        }
        mbar_init(bar_acc_full, 1);
        mbar_init(bar_acc_empty, 4);
        mbar_init(bar_drain, 1);
        mbar_fence_init();
        *s_abort = 0;
        for (int s = 0; s < S; ++s) tma_prefetch_map(&p.map_a[s]);
        for (int i = 0; i < UM_XMAPS; ++i) tma_prefetch_map(&p.map_x[i]);
    }
    const SegTab tab = seg_tab(reinterpret_cast<int *>(smem + L.tab_off), p.nbins);
    // Every tile of every segment (partial), or the whole 128-token tiles
    // only (a segment of c tokens then contributes c / 128).
    const int total_tiles = load_segments(p.no_lora, p.active, p.counts, p.start_loc,
                                          p.nbins, UM_BM, tab, /*full_tiles_only=*/!p.partial, 0,
                                          p.num_tokens, p.error_word);
    if (total_tiles == 0) return;
    const int H = p.hidden, R = p.rank, T = p.num_tokens;
    const int nk = (H + UM_BK - 1) / UM_BK;
    const int kchunks = shrink_kchunks(total_tiles, nk, int(gridDim.x), UM_MIN_BLOCKS);
    const int spc = (nk + kchunks - 1) / kchunks;
    // Items: item = kc * total_tiles + tile.  When every tile is one whole
    // item and some CTAs would have none, the first `extra` tiles are halved
    // along the hidden dimension instead (items 2j and 2j + 1 are the halves
    // of tile j < extra, item extra + t the whole tile t >= extra): the
    // idle SMs take half of those tiles, and the first tile (on a mixed
    // batch, the one whose tokens break into the most short runs, whose CTA
    // finished last) is one of them.
    const int extra = (kchunks == 1 && total_tiles < int(gridDim.x) && nk >= 2 * UM_MIN_BLOCKS)
                          ? min(int(gridDim.x) - total_tiles, total_tiles)
                          : 0;
    const int total_items = total_tiles * kchunks + extra;
    auto item_range = [&](int item, int &tile, int &kb0, int &kb1) {
        if (extra > 0) {
            if (item < 2 * extra) {
                tile = item >> 1;
                kb0 = (item & 1) ? nk / 2 : 0;
                kb1 = (item & 1) ? nk : nk / 2;
            } else {
                tile = item - extra;
                kb0 = 0;
                kb1 = nk;
            }
            return;
        }
        tile = item % total_tiles;
        const int kc = item / total_tiles;
        kb0 = kc * spc;
        kb1 = min(nk, kb0 + spc);
    };
    if (int(blockIdx.x) >= total_items) return;

    if (warp == UM_MMA_WARP) tmem_alloc(smem_addr(s_tmem), p.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    const long long deadline = clock64() + UM_TIMEOUT_CYCLES;

    if (warp == 0) {
        // ------------------------------------------------------ producer
        // Tokens of a tile are increasing (the sort is stable), so they
        // split into runs of consecutive tokens, cut into pieces whose
        // heights are powers of two (tile_pieces_warp); each piece is one 2-D
        // TMA box of the x map with that height, written at its row of the
        // 128-byte-swizzled tile.  Long prefill sequences make most tiles a
        // single 128-row box.
        uint32_t *pieces = reinterpret_cast<uint32_t *>(smem + L.piece_off);
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        for (int item = blockIdx.x; ok && item < total_items; item += gridDim.x) {
            int tile, kb0, kb1;
            item_range(item, tile, kb0, kb1);
            const int seg = find_segment(tab.tile, p.nbins, tile);
            const int row0 = tab.start[seg] + (tile - tab.tile[seg]) * UM_BM;
            // rows of this tile that belong to the segment (all 128 but in
            // the last, partial tile of a segment); only they are loaded, and
            // the stage's barrier expects exactly their bytes
            const int nrows = min(UM_BM, tab.start[seg] + tab.count[seg] - row0);
            const uint32_t tx = uint32_t(nrows * 128);
            const int npieces = tile_pieces_warp(p.sorted + row0, nrows, pieces);
            __syncwarp();
            for (int kb = kb0; kb < kb1; ++kb) {
                bool got = mbar_wait_bounded(bar_empty + 8 * stage, phase ^ 1u, s_abort, deadline);
                if (__all_sync(0xffffffffu, got) == 0) {
                    ok = false;
                    break;
                }
                const uint32_t sx = base + stage * L.stage_bytes;
                const uint32_t full = bar_full + 8 * stage;
                if (lane == 0) mbar_arrive_expect_tx(full, tx);
                __syncwarp();
                for (int i = lane; i < npieces; i += 32) {
                    const uint32_t pc = pieces[i];
                    const int r = int(pc & 0xFFu), lg = int((pc >> 8) & 7u), t0 = int(pc >> 11);
                    tma_load_2d(sx + r * 128, &p.map_x[lg], kb * UM_BK, t0, full);
                }
                ++issued;
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
        }
        // Every issued fill must land before the CTA may exit.
        if (lane == 0) {
            const long long drain_deadline = clock64() + UM_TIMEOUT_CYCLES;
            for (int i = max(0, issued - STAGES); i < issued; ++i) {
                const uint32_t ph = uint32_t(i / STAGES) & 1u;
                while (!mbar_try_wait(bar_full + 8 * (i % STAGES), ph) &&
                       clock64() < drain_deadline) {
                }
            }
        }
    } else if (warp >= UM_APROD0) {
        // ------------------------------------------------------ A producers
        // Producer j loads the A blocks of slices j, j + 3, ... into every
        // stage, in the same stage order as the x producer.
        const int j = warp - UM_APROD0;
        if (j < S && lane == 0) {
            int nsl = 0;
            for (int s = j; s < S; s += UM_APRODS) ++nsl;
            const uint32_t tx = uint32_t(nsl * L.a_bytes);
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int item = blockIdx.x; ok && item < total_items; item += gridDim.x) {
                int tile, kb0, kb1;
                item_range(item, tile, kb0, kb1);
                const int id = tab.id[find_segment(tab.tile, p.nbins, tile)];
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait_bounded(bar_empty + 8 * stage, phase ^ 1u, s_abort, deadline)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sx = base + stage * L.stage_bytes;
                    const uint32_t full = bar_full + 8 * stage;
                    mbar_arrive_expect_tx(full, tx);
                    for (int s = j; s < S; s += UM_APRODS)
                        tma_load_2d(sx + L.x_bytes + s * L.a_bytes, &p.map_a[s], kb * UM_BK,
                                    id * R, full);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            // Every issued fill must land before the CTA may exit.
            const long long drain_deadline = clock64() + UM_TIMEOUT_CYCLES;
            for (int i = max(0, issued - STAGES); i < issued; ++i) {
                const uint32_t ph = uint32_t(i / STAGES) & 1u;
                while (!mbar_try_wait(bar_full + 8 * (i % STAGES), ph) &&
                       clock64() < drain_deadline) {
                }
            }
        }
        __syncwarp();
    } else if (warp == UM_MMA_WARP) {
        // ------------------------------------------------------ MMA issue
        if (lane == 0) {
            // Consecutive slices share one UMMA of N = G * RP <= 256 (their
            // A blocks and TMEM columns are adjacent): x is read from shared
            // memory once per group instead of once per slice.
            const int G = 256 / RP < S ? 256 / RP : S;
            const uint32_t idesc_g = umma_idesc_bf16(UM_BM, G * RP);
            const uint32_t idesc_r = umma_idesc_bf16(UM_BM, (S % G == 0 ? G : S % G) * RP);
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int item = blockIdx.x; ok && item < total_items; item += gridDim.x) {
                int tile, kb0, kb1;
                item_range(item, tile, kb0, kb1);
                if (!mbar_wait_bounded(bar_acc_empty, acc_phase ^ 1, s_abort, deadline)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait_bounded(bar_full + 8 * stage, phase, s_abort, deadline)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sx = base + stage * L.stage_bytes;
#pragma unroll
                    for (int kk = 0; kk < UM_BK / 16; ++kk) {
                        const uint64_t adesc = umma_desc_sw128(sx + kk * 32);
                        for (int s = 0; s < S; s += G) {
                            const uint64_t bdesc = umma_desc_sw128(sx + L.x_bytes + s * L.a_bytes + kk * 32);
                            umma_bf16(tmem + s * RP, adesc, bdesc, s + G <= S ? idesc_g : idesc_r,
                                      kb != kb0 || kk != 0);
                        }
                    }
                    umma_commit(bar_empty + 8 * stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                umma_commit(bar_acc_full);
                acc_phase ^= 1;
            }
            // After an abort, wait (bounded) until every MMA issued so far
            // has completed before TMEM is released.
            if (!ok || *s_abort) {
                umma_commit(bar_drain);
                const long long drain_deadline = clock64() + UM_TIMEOUT_CYCLES;
                while (!mbar_try_wait(bar_drain, 0) && clock64() < drain_deadline) {
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        const int row = q * 32 + lane;          // token row inside the tile
        uint32_t acc_phase = 0;
        for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
            int tile, kb0, kb1;
            item_range(item, tile, kb0, kb1);
            const int seg = find_segment(tab.tile, p.nbins, tile);
            const int row0 = tab.start[seg] + (tile - tab.tile[seg]) * UM_BM;
            // rows past the segment's end hold stale shared data: their
            // accumulators are read (the load is warp-wide) but not stored
            const int nrows = min(UM_BM, tab.start[seg] + tab.count[seg] - row0);
            const int tok =
                row < nrows ? checked_token(p.sorted[row0 + row], T, p.error_word) : -1;
            bool got = mbar_wait_bounded(bar_acc_full, acc_phase, s_abort, deadline);
            if (__all_sync(0xffffffffu, got) == 0) break;       // warp-uniform exit
            tc_fence_after();
            shrink_epilogue_row(tmem + (uint32_t(q * 32) << 16), p.y, tok, T, R, RP,
                                S, p.scale);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_acc_empty);
            acc_phase ^= 1;
        }
    }

    if (tid == 0 && *s_abort) atomicOr(p.error_word, UM_ERROR_BIT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == UM_MMA_WARP) tmem_dealloc(tmem, p.tmem_cols);
}


// ------------------------------------------------------------------ host

// Launches the UMMA path if the shapes allow it; returns 1 if launched, 0
// if not applicable (caller then covers every row with the mma.sync path),
// or a negative value / cudaError_t on failure.
int launch_shrink_umma(const ShrinkLaunch &a, cudaStream_t stream)
{
    // The CTA-pair kernel (lora_shrink_pair.cu) is opt-in: measured slower.
    if (knobs().umma_pair != 0) {
        const int r = launch_shrink_pair(a, stream);
        if (r != 0) return r;
    }
    int rp = 16;
    while (rp < a.rank) rp <<= 1;
    const int S = a.num_slices;
    // Token indices travel in 21 bits of a piece descriptor.
    if (S * rp > 512 || a.hidden < UM_BK || a.num_tokens < UM_BM || a.num_tokens >= (1 << 21))
        return 0;
    int cols = 32;
    while (cols < S * rp) cols <<= 1;
    const int nbins = a.max_loras + 1;
    int stages = UM_MAX_STAGES;
    while (stages > 2 && umma_layout(S, rp, stages, nbins).total > UM_SMEM_BUDGET) --stages;
    const UmmaLayout L = umma_layout(S, rp, stages, nbins);
    if (L.total > 227 * 1024) return 0;

    static UmmaShrinkArgs p;      // large (>1 KB): keep off the stack
    for (int i = 0; i < UM_XMAPS; ++i)
        if (!encode_tile_map(&p.map_x[i], a.x, uint64_t(a.num_tokens), uint64_t(a.hidden),
                             uint64_t(a.x_ld), UM_BK, 1u << i, CU_TENSOR_MAP_SWIZZLE_128B))
            return 0;
    for (int s = 0; s < S; ++s) {
        if (!encode_tile_map(&p.map_a[s], a.a[s], uint64_t(a.max_loras) * a.rank, uint64_t(a.hidden),
                             uint64_t(a.hidden), UM_BK, uint32_t(rp), CU_TENSOR_MAP_SWIZZLE_128B))
            return 0;
    }
    p.y = a.y;
    p.scale = a.scale;
    p.num_tokens = a.num_tokens;
    p.hidden = a.hidden;
    p.num_slices = S;
    p.rank = a.rank;
    p.rp = rp;
    p.stages = stages;
    p.tmem_cols = cols;
    p.sorted = a.sorted;
    p.counts = a.counts;
    p.start_loc = a.start_loc;
    p.active = a.active;
    p.no_lora = a.no_lora;
    p.error_word = a.error_word;
    p.nbins = nbins;
    p.partial = a.partial;

    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return int(e);
    if (dev < 64 && configured[dev] == 0) {
        e = cudaFuncSetAttribute(shrink_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 227 * 1024);
        if (e != cudaSuccess) return int(e);
        configured[dev] = 1;
    }
    const int grid = device_sm_count();
    e = launch_kernel(shrink_umma_kernel, dim3(grid), dim3(UM_THREADS), size_t(L.total), stream, p);
    return e == cudaSuccess ? 1 : int(e);
}

}  // namespace lora
