// lora_shrink_pair.cu -- tensor-core path of lora_shrink on CTA pairs (page
// "vllm.lora.punica_wrapper.punica_gpu", PunicaWrapperGPU.add_shrink:
// y[s][t, :] += scale * x[t, :] @ A[s][id(t)]^T).
//
// The same product as shrink_umma_kernel, computed by clusters of two CTAs
// on neighbouring SMs that drive one tcgen05 MMA with M = 256
// (cta_group::2): a work item is a 256-token tile of one LoRA segment (and
// a chunk of the hidden dimension); the even CTA of the pair holds tokens
// 0..127 of the tile, the odd CTA tokens 128..255.  Each CTA loads its own
// x rows and HALF of the A rows of every stage; the pair's tensor cores
// exchange the halves.  Against one CTA per 128-token tile this halves the
// A bytes each SM moves through TMA and reads from shared memory, which
// bound the single-CTA kernel (its UMMAs read both operands from shared
// memory while TMA fills it, on this GPU about 128 bytes per clock per SM).
//
// Opt-in (LORA_PUNICA_UMMA_PAIR=1): measured on the large workload (16384
// tokens, hidden 8192, rank 128, three slices) it takes 238 us against
// 138 us for the single-CTA kernel.  Per-chunk clock64 stamps put the pair's
// UMMAs at about half the per-SM rate of the single-CTA kernel's (about
// 1700 cycles to issue one stage's eight UMMAs, against 1050), and the
// relay of each odd-CTA stage to the even CTA (a cluster-scope release
// arrive) at about 1300 cycles; the hidden split that balances 256-token
// tiles over 76 pairs also multiplies the epilogues.
//
// Slices are grouped as in the single-CTA kernel: a group of G consecutive
// slices is one UMMA of N = G * RP.  In the M = 256 form each CTA holds N/2
// of the group's B rows: a group of an even number of slices gives each CTA
// whole slices (the even CTA the first half); a group of one slice gives
// each CTA half of its rows.
//
// Warps of each CTA:
//   warp 0      x producer: the CTA's 128 x rows per 64-wide hidden block,
//               by 2-D TMA boxes over runs of consecutive tokens.
//   warps 6..8  A producers: the CTA's half of each group's B rows, group g
//               issued by warp 6 + g % 3.
//   warp 1      allocates the pair's TMEM (both CTAs, together).  In the even
//               CTA lane 0 issues the pair's UMMAs once both CTAs' stage has
//               landed and commits to the stage's empty barrier in both CTAs
//               and, at the end of an item, to both accumulator barriers.
//               In the odd CTA lane 0 relays "stage landed" to the even CTA.
//   warps 2..5  epilogue: tcgen05.ld of the CTA's own 128 TMEM lanes (one
//               token row per thread), buf += scale * acc (float4
//               reductions); then they release the accumulators to the even
//               CTA.
//
// Every mbarrier wait is bounded (about one second); on expiry a CTA sets
// bit 30 of the metadata error word, stops issuing, waits (bounded) for its
// copies and MMAs in flight and for the commits aimed at its barriers, then
// meets its peer at the final cluster barrier, frees TMEM and returns.
#include "lora_common.cuh"
#include "lora_umma.cuh"

namespace lora {

constexpr int PR_BM = 128;            // tokens per CTA = UMMA M / 2
constexpr int PR_TILE = 2 * PR_BM;    // tokens per pair tile
constexpr int PR_BK = 64;             // hidden per stage (one 128-byte swizzle atom)
constexpr int PR_MMA_WARP = 1;
constexpr int PR_APROD0 = 6;
constexpr int PR_APRODS = 3;
constexpr int PR_THREADS = 32 * (PR_APROD0 + PR_APRODS);
constexpr int PR_XMAPS = 8;           // x box heights 1, 2, 4, ..., 128
constexpr int PR_MAX_STAGES = 8;
constexpr int PR_MAX_GROUPS = LORA_MAX_SLICES;
constexpr int PR_SMEM_BUDGET = 200 * 1024;
constexpr long long PR_TIMEOUT_CYCLES = 2000000000ll;
constexpr int PR_ERROR_BIT = 1 << 30;
constexpr int PR_MIN_BLOCKS = 8;      // shortest hidden chunk of a split item

struct PairShrinkArgs {
    CUtensorMap map_x[PR_XMAPS];               // x: [T, H], box {64, 2^i rows}
    CUtensorMap map_a[LORA_MAX_SLICES];        // A[s]: [L * r, H], box {64, RP}
    CUtensorMap map_ah[LORA_MAX_SLICES];       // A[s]: box {64, RP / 2}
    float *y;
    float scale;
    int32_t num_tokens;
    int32_t hidden;
    int32_t num_slices;
    int32_t rank;
    int32_t rp;                                // padded rank, 64 or 128
    int32_t stages;
    int32_t tmem_cols;
    int32_t num_groups;
    int32_t group_first[PR_MAX_GROUPS];        // first slice of group g
    int32_t group_size[PR_MAX_GROUPS];         // slices in group g (even, or 1)
    int32_t group_off[PR_MAX_GROUPS];          // byte offset of the CTA's B half in a stage
    int32_t stage_bytes;
    const int32_t *sorted;
    const int32_t *counts;
    const int32_t *start_loc;
    const int32_t *active;
    const int32_t *no_lora;
    int32_t *error_word;
    int32_t nbins;
};

// Shared-memory layout of one CTA (offsets from the 1024-byte-aligned base).
struct PairLayout {
    int ring_bytes, bar_off, misc_off, piece_off, tab_off, total;
};

__host__ __device__ inline PairLayout pair_layout(int stage_bytes, int stages, int nbins)
{
    PairLayout l;
    l.ring_bytes = stages * stage_bytes;
    l.bar_off = l.ring_bytes;                             // full, empty, pfull; acc x2; drain
    l.misc_off = l.bar_off + (3 * PR_MAX_STAGES + 3) * 8; // tmem base, abort flag
    l.piece_off = l.misc_off + 16;                        // [PR_BM] x pieces
    l.tab_off = l.piece_off + PR_BM * 4;
    l.total = l.tab_off + int(seg_tab_bytes(nbins)) + 1024;    // + alignment slack
    return l;
}

__global__ void __launch_bounds__(PR_THREADS, 1) shrink_pair_kernel(const __grid_constant__ PairShrinkArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms; the same offsets
    // in both CTAs of the pair (the UMMA descriptors address both).
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int RP = p.rp, STAGES = p.stages, NG = p.num_groups;
    const PairLayout L = pair_layout(p.stage_bytes, STAGES, p.nbins);
    const uint32_t base = smem_addr(smem);
    const uint32_t bar_full = base + L.bar_off;                 // [STAGES] this CTA's fills
    const uint32_t bar_empty = bar_full + 8 * PR_MAX_STAGES;    // [STAGES] the pair's MMAs
    const uint32_t bar_pfull = bar_empty + 8 * PR_MAX_STAGES;   // [STAGES] odd CTA's fills
    const uint32_t bar_acc_full = bar_pfull + 8 * PR_MAX_STAGES;
    const uint32_t bar_acc_empty = bar_acc_full + 8;            // both CTAs' epilogues
    const uint32_t bar_drain = bar_acc_empty + 8;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + L.misc_off + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();                    // 0 issues the MMAs
    const int cluster = int(blockIdx.x >> 1), nclusters = int(gridDim.x >> 1);

    pdl_wait();
    pdl_launch_dependents();

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            // one expect_tx arrival from the x producer and one from each A
            // producer that has a group
            mbar_init(bar_full + 8 * i, 1 + min(NG, PR_APRODS));
            mbar_init(bar_empty + 8 * i, 1);
            mbar_init(bar_pfull + 8 * i, 1);
        }
        mbar_init(bar_acc_full, 1);
        mbar_init(bar_acc_empty, 8);
        mbar_init(bar_drain, 1);
        mbar_fence_init();
        *s_abort = 0;
        for (int s = 0; s < p.num_slices; ++s) {
            tma_prefetch_map(&p.map_a[s]);
            tma_prefetch_map(&p.map_ah[s]);
        }
        for (int i = 0; i < PR_XMAPS; ++i) tma_prefetch_map(&p.map_x[i]);
    }
    const SegTab tab = seg_tab(reinterpret_cast<int *>(smem + L.tab_off), p.nbins);
    // Both CTAs of a pair read the same metadata, so every exit below is
    // taken by both (neither then waits at a cluster barrier).
    const int total_tiles = load_segments(p.no_lora, p.active, p.counts, p.start_loc, p.nbins,
                                          PR_TILE, tab, false, 0, p.num_tokens, p.error_word);
    if (total_tiles == 0) return;
    const int H = p.hidden, R = p.rank, T = p.num_tokens;
    const int nk = (H + PR_BK - 1) / PR_BK;
    const int kchunks = shrink_kchunks(total_tiles, nk, nclusters, PR_MIN_BLOCKS);
    const int spc = (nk + kchunks - 1) / kchunks;
    const int total_items = total_tiles * kchunks;      // item = kc * total_tiles + tile
    if (cluster >= total_items) return;

    if (warp == PR_MMA_WARP) tmem_alloc_pair(smem_addr(s_tmem), p.tmem_cols);
    tc_fence_before();
    cluster_sync_all();       // barriers of both CTAs initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const long long deadline = clock64() + PR_TIMEOUT_CYCLES;

    // The CTA's rows of a pair tile: [row0, row0 + nrows) of the sorted list.
    auto cta_rows = [&](int tile, int &row0, int &nrows) {
        const int seg = find_segment(tab.tile, p.nbins, tile);
        row0 = tab.start[seg] + (tile - tab.tile[seg]) * PR_TILE + int(rank) * PR_BM;
        nrows = min(PR_BM, max(0, tab.start[seg] + tab.count[seg] - row0));
        return seg;
    };
    // After its last fill, a producer waits (bounded) until the fills of the
    // last STAGES stages have landed and the pair's MMAs that read them have
    // committed to this CTA's empty barriers: no copy and no commit may
    // still target this CTA's shared memory when it exits.
    auto drain_fills = [&](int issued) {
        const long long dd = clock64() + PR_TIMEOUT_CYCLES;
        for (int i = max(0, issued - STAGES); i < issued; ++i) {
            const uint32_t ph = uint32_t(i / STAGES) & 1u;
            while (!mbar_try_wait(bar_full + 8 * (i % STAGES), ph) && clock64() < dd) {
            }
            while (!mbar_try_wait_cluster(bar_empty + 8 * (i % STAGES), ph) && clock64() < dd) {
            }
        }
    };

    if (warp == 0) {
        // ------------------------------------------------------ x producer
        // The CTA's tokens of a tile are increasing (the sort is stable), so
        // they split into runs of consecutive tokens; lane 0 cuts them into
        // pieces whose heights are powers of two, one TMA box each, written
        // at their row of the 128-byte-swizzled x tile.
        uint32_t *pieces = reinterpret_cast<uint32_t *>(smem + L.piece_off);
        int stage = 0, issued = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int item = cluster; ok && item < total_items; item += nclusters) {
            const int tile = item % total_tiles, kc = item / total_tiles;
            const int kb0 = kc * spc, kb1 = min(nk, kb0 + spc);
            int row0, nrows;
            cta_rows(tile, row0, nrows);
            const uint32_t tx = uint32_t(nrows * 128);
            int npieces = 0;
            if (lane == 0) {
                const int32_t *tk = p.sorted + row0;
                int j = 0;
                while (j < nrows) {
                    int lg = 7;
                    while ((1 << lg) > nrows - j || (j & ((1 << lg) - 1)) != 0 ||
                           tk[j + (1 << lg) - 1] - tk[j] != (1 << lg) - 1)
                        --lg;
                    pieces[npieces++] = uint32_t(j) | (uint32_t(lg) << 8) |
                                        (uint32_t(tk[j]) << 11);
                    j += 1 << lg;
                }
            }
            npieces = __shfl_sync(0xffffffffu, npieces, 0);
            __syncwarp();
            for (int kb = kb0; kb < kb1; ++kb) {
                const bool got = mbar_wait_bounded_cluster(bar_empty + 8 * stage, phase ^ 1u,
                                                           s_abort, deadline);
                if (__all_sync(0xffffffffu, got) == 0) {
                    ok = false;
                    break;
                }
                const uint32_t sx = base + stage * p.stage_bytes;
                const uint32_t full = bar_full + 8 * stage;
                if (lane == 0) mbar_arrive_expect_tx(full, tx);
                __syncwarp();
                for (int i = lane; i < npieces; i += 32) {
                    const uint32_t pc = pieces[i];
                    const int r = int(pc & 0xFFu), lg = int((pc >> 8) & 7u), t0 = int(pc >> 11);
                    tma_load_2d(sx + r * 128, &p.map_x[lg], kb * PR_BK, t0, full);
                }
                ++issued;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (lane == 0) drain_fills(issued);
        __syncwarp();
    } else if (warp >= PR_APROD0) {
        // ------------------------------------------------------ A producers
        // Producer j loads this CTA's half of the B rows of groups j, j + 3,
        // ... into every stage, in the x producer's stage order.
        const int j = warp - PR_APROD0;
        if (j < NG && lane == 0) {
            uint32_t tx = 0;
            for (int g = j; g < NG; g += PR_APRODS)
                tx += uint32_t(p.group_size[g] >= 2 ? p.group_size[g] / 2 * RP : RP / 2) * 128u;
            int stage = 0, issued = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int item = cluster; ok && item < total_items; item += nclusters) {
                const int tile = item % total_tiles, kc = item / total_tiles;
                const int kb0 = kc * spc, kb1 = min(nk, kb0 + spc);
                const int id = tab.id[find_segment(tab.tile, p.nbins, tile)];
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait_bounded_cluster(bar_empty + 8 * stage, phase ^ 1u, s_abort,
                                                   deadline)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sx = base + stage * p.stage_bytes;
                    const uint32_t full = bar_full + 8 * stage;
                    mbar_arrive_expect_tx(full, tx);
                    for (int g = j; g < NG; g += PR_APRODS) {
                        const int gs = p.group_size[g], s0 = p.group_first[g];
                        const uint32_t dst = sx + uint32_t(p.group_off[g]);
                        if (gs >= 2) {
                            // whole slices: the even CTA the group's first half
                            for (int q = 0; q < gs / 2; ++q)
                                tma_load_2d(dst + uint32_t(q * RP * 128),
                                            &p.map_a[s0 + int(rank) * (gs / 2) + q], kb * PR_BK,
                                            id * R, full);
                        } else {
                            // one slice: the even CTA its first RP/2 rows
                            tma_load_2d(dst, &p.map_ah[s0], kb * PR_BK,
                                        id * R + int(rank) * (RP / 2), full);
                        }
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            drain_fills(issued);
        }
        __syncwarp();
    } else if (warp == PR_MMA_WARP) {
        if (lane == 0 && rank == 0) {
            // -------------------------------------------------- pair MMA issue
            const uint32_t empty_me = cluster_map(bar_empty, 0), empty_peer = cluster_map(bar_empty, 1);
            const uint32_t accf_me = cluster_map(bar_acc_full, 0);
            const uint32_t accf_peer = cluster_map(bar_acc_full, 1);
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int item = cluster; ok && item < total_items; item += nclusters) {
                const int kc = item / total_tiles;
                const int kb0 = kc * spc, kb1 = min(nk, kb0 + spc);
                if (!mbar_wait_bounded_cluster(bar_acc_empty, acc_phase ^ 1u, s_abort, deadline)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait_bounded(bar_full + 8 * stage, phase, s_abort, deadline) ||
                        !mbar_wait_bounded_cluster(bar_pfull + 8 * stage, phase, s_abort,
                                                   deadline)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sx = base + stage * p.stage_bytes;
#pragma unroll
                    for (int kk = 0; kk < PR_BK / 16; ++kk) {
                        const uint64_t adesc = umma_desc_sw128(sx + kk * 32);
                        for (int g = 0; g < NG; ++g) {
                            const uint64_t bdesc =
                                umma_desc_sw128(sx + uint32_t(p.group_off[g]) + kk * 32);
                            umma_bf16_pair(tmem + uint32_t(p.group_first[g] * RP), adesc, bdesc,
                                           umma_idesc_bf16(2 * PR_BM, p.group_size[g] * RP),
                                           kb != kb0 || kk != 0);
                        }
                    }
                    umma_commit_pair(empty_me + 8 * stage);
                    umma_commit_pair(empty_peer + 8 * stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair(accf_me);
                umma_commit_pair(accf_peer);
                acc_phase ^= 1u;
            }
            // After an abort, wait (bounded) until every MMA issued so far
            // has completed before TMEM is released.
            if (!ok || *s_abort) {
                umma_commit_pair(cluster_map(bar_drain, 0));
                const long long dd = clock64() + PR_TIMEOUT_CYCLES;
                while (!mbar_try_wait_cluster(bar_drain, 0) && clock64() < dd) {
                }
            }
        } else if (lane == 0) {
            // -------------------------------------------------- relay (odd CTA)
            const uint32_t pfull_leader = cluster_map(bar_pfull, 0);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int item = cluster; ok && item < total_items; item += nclusters) {
                const int kc = item / total_tiles;
                const int kb0 = kc * spc, kb1 = min(nk, kb0 + spc);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait_bounded(bar_full + 8 * stage, phase, s_abort, deadline)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_cluster(pfull_leader + 8 * stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        const int row = q * 32 + lane;          // token row of this CTA's half tile
        const uint32_t acce_leader = cluster_map(bar_acc_empty, 0);
        uint32_t acc_phase = 0;
        for (int item = cluster; item < total_items; item += nclusters) {
            const int tile = item % total_tiles;
            int row0, nrows;
            cta_rows(tile, row0, nrows);
            // rows past the segment's end hold stale shared data: their
            // accumulators are read (the load is warp-wide) but not stored
            const int tok =
                row < nrows ? checked_token(p.sorted[row0 + row], T, p.error_word) : -1;
            const bool got = mbar_wait_bounded_cluster(bar_acc_full, acc_phase, s_abort, deadline);
            if (__all_sync(0xffffffffu, got) == 0) break;       // warp-uniform exit
            tc_fence_after();
            shrink_epilogue_row(tmem + (uint32_t(q * 32) << 16), p.y, tok, T, R, RP,
                                p.num_slices, p.scale);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acce_leader);
            acc_phase ^= 1u;
        }
    }

    if (tid == 0 && *s_abort) atomicOr(p.error_word, PR_ERROR_BIT);
    tc_fence_before();
    cluster_sync_all();       // both CTAs done: no MMA, copy or arrive in flight
    tc_fence_after();
    if (warp == PR_MMA_WARP) tmem_dealloc_pair(tmem, uint32_t(p.tmem_cols));
}

// ------------------------------------------------------------------ host

// Launches the CTA-pair kernel if the shapes allow it: returns 1 if
// launched, 0 if not applicable (the caller then runs the single-CTA
// tensor-core kernel), or a cudaError_t.
int launch_shrink_pair(const ShrinkLaunch &a, cudaStream_t stream)
{
    int rp = 16;
    while (rp < a.rank) rp <<= 1;
    const int S = a.num_slices;
    // Token indices travel in 21 bits of a piece descriptor.
    if ((rp != 64 && rp != 128) || !a.partial || S * rp > 512 || a.hidden < PR_BK ||
        a.num_tokens < 1 || a.num_tokens >= (1 << 21))
        return 0;
    const int grid = device_sm_count() & ~1;
    if (grid < 2) return 0;

    static thread_local PairShrinkArgs p;       // large (> 3 KB): keep off the stack
    // Groups of consecutive slices, one UMMA of N = size * rp each: the
    // largest power of two of slices that fits N <= 256 and what is left.
    const int gmax = 256 / rp;
    int ng = 0, off = PR_BM * PR_BK * 2;            // the x tile comes first
    for (int s = 0; s < S;) {
        int gs = gmax;
        while (gs > S - s) gs >>= 1;
        p.group_first[ng] = s;
        p.group_size[ng] = gs;
        p.group_off[ng] = off;
        off += (gs >= 2 ? gs / 2 * rp : rp / 2) * PR_BK * 2;
        s += gs;
        ++ng;
    }
    p.num_groups = ng;
    p.stage_bytes = off;                            // a multiple of 4096
    const int nbins = a.max_loras + 1;
    int stages = PR_MAX_STAGES;
    while (stages > 2 && pair_layout(off, stages, nbins).total > PR_SMEM_BUDGET) --stages;
    const PairLayout L = pair_layout(off, stages, nbins);
    if (L.total > 227 * 1024) return 0;
    int cols = 32;
    while (cols < S * rp) cols <<= 1;

    for (int i = 0; i < PR_XMAPS; ++i)
        if (!encode_tile_map(&p.map_x[i], a.x, uint64_t(a.num_tokens), uint64_t(a.hidden),
                             uint64_t(a.x_ld), PR_BK, 1u << i, CU_TENSOR_MAP_SWIZZLE_128B))
            return 0;
    for (int s = 0; s < S; ++s) {
        const uint64_t rows = uint64_t(a.max_loras) * uint64_t(a.rank);
        if (!encode_tile_map(&p.map_a[s], a.a[s], rows, uint64_t(a.hidden), uint64_t(a.hidden),
                             PR_BK, uint32_t(rp), CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tile_map(&p.map_ah[s], a.a[s], rows, uint64_t(a.hidden), uint64_t(a.hidden),
                             PR_BK, uint32_t(rp / 2), CU_TENSOR_MAP_SWIZZLE_128B))
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

    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return int(e);
    if (dev < 64 && configured[dev] == 0) {
        e = cudaFuncSetAttribute(shrink_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 227 * 1024);
        if (e != cudaSuccess) return int(e);
        configured[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(PR_THREADS);
    cfg.dynamicSmemBytes = size_t(L.total);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, shrink_pair_kernel, p);
    return e == cudaSuccess ? 1 : int(e);
}

}  // namespace lora
