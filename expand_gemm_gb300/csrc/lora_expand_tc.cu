// lora_expand_tc.cu -- tensor-core (tcgen05 / TMEM) path of lora_expand
// (page "vllm.lora.punica_wrapper.punica_gpu", PunicaWrapperGPU.add_expand;
// bias step of page "vllm.lora.punica_wrapper.punica_tpu",
// PunicaWrapperTPU._apply_bias):
//   y[t, off_s + j] (+)= x[s][t, :] @ B[s][id(t)][j, :] + bias[s][id(t)][j]
//
// Work items are (128-token tile of one LoRA segment, 128-column chunk of
// one slice), numbered chunk-fastest; one persistent CTA per SM takes a
// contiguous, balanced range of them, so it walks the chunks of one tile
// with the tile's x rows (the MMA's A operand) resident in tensor memory.
// Chunks stream through a ring of DEPTH slots in shared memory, each
// holding the chunk's B tile (swizzled K-major, as UMMA reads it) and its
// old y rows.
//
// A sits in TMEM, not shared memory: a UMMA that reads both operands from
// shared memory is bound by its operand reads (measured on this GPU: 48
// cycles for M = 128, N = 64, K = 16, against 32 for the math), and A is
// a large share of those bytes; from TMEM, each chunk reads only its B tile
// from shared memory.
//
// One job per warp (rank 128: fourteen warps; lower ranks: twelve, with two
// y loader warps and more registers for the epilogue):
//   warp 0       owns TMEM (two 128-column fp32 accumulators and the A
//                operand); lane 0 issues tcgen05.mma (M = 128 tokens,
//                N = 128 columns, K = 16 steps over the rank) and commits
//                each chunk's accumulator and the release of its slot's B.
//   warp 1       lane 0 loads each chunk's B tile with TMA through a 5-D
//                tensor map that permutes its rows (below).
//   warps 2..    y loaders: the chunk's 128 old y rows, gathered through the
//                permutation with 16-byte cp.async (four whole 128-byte lines
//                per instruction); each thread's copies arrive on the slot's
//                y barrier when they land, so the loaders never wait for
//                their own copies and run up to DEPTH chunks ahead.
//   last 8 warps epilogue.  Warp (q, h) = (warp % 4, (warp - first) / 4) owns
//                tile rows 32q + 16h .. 32q + 16h + 15 (TMEM lane quarter q,
//                as tcgen05.ld requires).  It reads their accumulators one
//                64-column half at a time in the 16x256b shape, in which
//                thread (g, t) = (lane / 4, lane % 4) holds columns 8i + 2t,
//                8i + 2t + 1 (i < 8) of rows g and g + 8.  B's rows were
//                loaded permuted so that, in each 64-column half, accumulator
//                column 8i + 2t + e is output column 16t + 2i + e: each
//                thread then holds 16 consecutive output columns of each of
//                its rows, adds old y (from the slot) and bias in fp32,
//                rounds once, and writes them with one 32-byte store (8 whole
//                128-byte rows per warp instruction), straight from
//                registers.  When the next chunk opens a new tile or slice,
//                it rounds that item's x rows to bf16 and stores them into
//                the A operand's TMEM columns right after reading the current
//                accumulator.
//
// Measured on the large workload (16384 tokens, rank 128, 10240 columns):
// 132 us against the mma.sync kernel's 216 us (149 us with 64-column
// chunks).  Designs that added old y on the tensor core (one more UMMA pass
// with a permutation matrix), split the epilogue into two groups taking
// alternate chunks, or suspended the waiting warps in hardware were slower.
//
// Every mbarrier wait is bounded (about one second); on expiry the kernel
// sets bit 30 of the metadata error word, drains its copies and MMAs, frees
// TMEM and returns.
#include "lora_common.cuh"
#include "lora_umma.cuh"

namespace lora {

constexpr int TC_BM = 128;                    // tokens per tile (UMMA M, TMEM lanes)
constexpr int TC_BN = 128;                    // columns per chunk (UMMA N)
constexpr int TC_HALVES = TC_BN / 64;         // 64-column blocks per chunk
constexpr int TC_EPI = 8;                     // epilogue warps
constexpr int TC_NACC = 2;                    // TMEM accumulators (chunk g uses g % TC_NACC)
constexpr int TC_A_COL = TC_NACC * TC_BN;    // TMEM column of the first A operand
// A operands held at once: row item j (a tile and slice) uses buffer
// j % TC_NXB.  The epilogue writes the first TC_NXB items' A operands when
// the CTA starts, so that no item boundary waits for x (the shrink output)
// while the y stream keeps HBM busy: there, x loads took 5-7 us a round
// trip, and a boundary held the MMA and the epilogue for 4-10 us.  Items
// past the first TC_NXB (CTAs with many short items) are written at their
// boundary, into the buffer item - TC_NXB used.
constexpr int TC_NXB = 4;
constexpr int TC_TMEM_COLS = 512;             // accumulators + TC_NXB A operands
static_assert(TC_BN == 64 || TC_BN == 128, "chunk width");
constexpr long long TC_TIMEOUT_CYCLES = 2000000000ll;
constexpr uint32_t TC_BACKOFF_NS = 200;       // loaders' sleep between polls of a full ring
constexpr int TC_ERROR_BIT = 1 << 30;

struct TcArgs {
    CUtensorMap bmap[LORA_MAX_SLICES];        // B[s] rows, permuted (encode_perm_rows_map)
    const void *x;                            // [S, T, r]: fp32, or bf16 when x_bf16
    int32_t x_bf16;
    const uint16_t *b[LORA_MAX_SLICES];       // [L, n_s, r]
    const uint16_t *bias[LORA_MAX_SLICES];    // [L, n_s] or null
    int32_t n[LORA_MAX_SLICES];
    int32_t col0[LORA_MAX_SLICES];
    int32_t chunk0[LORA_MAX_SLICES + 1];      // first chunk of each slice
    int32_t num_slices;
    int32_t rank;
    uint16_t *y;
    int64_t y_ld;
    int32_t num_tokens;
    int32_t add_inputs;
    int32_t bias_vec;
    int32_t early;                            // lora_linear's early mode (see ExpandArgs)
    const int32_t *sorted;
    const int32_t *counts;
    const int32_t *start_loc;
    const int32_t *active;
    const int32_t *no_lora;
    int32_t *error_word;
    int32_t nbins;
};

template <int KT>
struct TcCfg {
    static constexpr int RP = 16 * KT;                     // padded rank
    static constexpr int CPR = RP / 8;                     // 16-byte pieces per operand row
    static constexpr int BOX_K = RP < 64 ? RP : 64;        // B box width (elements)
    static constexpr int NBOX = RP / BOX_K;                // B boxes per chunk
    static constexpr int A_COLS = RP / 2;                  // TMEM columns of the A operand
    static constexpr int B_BYTES = TC_BN * RP * 2;
    static constexpr int Y_BYTES = TC_BM * TC_BN * 2;      // 128 rows x TC_BN columns
    static constexpr int SLOT_BYTES = B_BYTES + Y_BYTES;   // a multiple of 1024
    static constexpr int DEPTH = 196608 / SLOT_BYTES < 8 ? 196608 / SLOT_BYTES : 8;
    static constexpr int RING_OFF = 0;
    static constexpr int BAR_OFF = RING_OFF + DEPTH * SLOT_BYTES;
    static constexpr int MISC_OFF = BAR_OFF + (3 * DEPTH + 2 * TC_NACC + TC_NXB + 1) * 8;
    static_assert(TC_A_COL + TC_NXB * A_COLS <= TC_TMEM_COLS, "TMEM: accumulators + A buffers");
    static constexpr int TAB_OFF = MISC_OFF + 16;
    // Rank 128 keeps four y loader warps (its chunks carry the most bytes)
    // and reads each accumulator half right before finishing it; lower ranks
    // take two loader warps, which leaves the epilogue enough registers
    // (twelve warps: up to 168 per thread) to request both halves'
    // accumulators and old y before waiting for any of them.
    static constexpr int YLOADERS = KT >= 8 ? 4 : 2;
    static constexpr bool OVERLAP = KT < 8;
    // B issuer warps (1 .. BISSUE), each with its share of the chunk's
    // boxes: one thread streams about 15 bytes a clock by TMA, and the
    // rank-128 chunk's 32 KB of B then set the chunk period (chunks of
    // tiles with a handful of rows took nearly as long as full ones).
    static constexpr int BISSUE = KT >= 8 ? 2 : 1;
    static constexpr int YL0 = 1 + BISSUE;                 // first y loader warp
    static constexpr int EPI0 = YL0 + YLOADERS;            // first epilogue warp
    static constexpr int THREADS = 32 * (EPI0 + TC_EPI);
    static constexpr int LT = 32 * YLOADERS;               // y loader threads
    static constexpr int PPR = TC_BN / 8;                  // 16-byte y pieces per row
    static constexpr int Y_PER_T = TC_BM * PPR / LT;       // y pieces per loader thread
    static_assert(SLOT_BYTES % 1024 == 0, "1024-byte aligned operands");
    static_assert(NBOX % BISSUE == 0, "each B issuer takes the same number of boxes");
    static_assert(LT % PPR == 0, "whole y rows per loader pass");
};

// Byte offset of 16-byte piece `pc` (columns 8pc .. 8pc+7) of row `r` of a
// slot's y rows (128-byte-swizzled, so that the epilogue's reads, two rows
// x four 32-byte pieces per 8-thread phase, hit all 32 banks).
__device__ __forceinline__ uint32_t tc_y_off(int r, int pc)
{
    return uint32_t((pc >> 3) * (TC_BM * 128) + r * 128 + (((pc & 7) ^ (r & 7)) << 4));
}



template <int KT>
inline size_t tc_smem_bytes(int nbins)
{
    return size_t(TcCfg<KT>::TAB_OFF) + seg_tab_bytes(nbins) + 1024;     // + alignment slack
}

// Shared-memory descriptor of K step kk (16 columns) of such a tile.
__device__ __forceinline__ uint64_t tc_kmajor_desc(int rp, int rows, uint32_t tile, int kk)
{
    uint32_t addr, sbo, layout;
    switch (rp) {
    case 16: addr = tile; sbo = 256; layout = 6; break;                         // 32-byte swizzle
    case 32: addr = tile + kk * 32; sbo = 512; layout = 4; break;               // 64-byte swizzle
    case 64: addr = tile + kk * 32; sbo = 1024; layout = 2; break;              // 128-byte swizzle
    default: addr = tile + (kk >> 2) * rows * 128 + (kk & 3) * 32; sbo = 1024; layout = 2; break;
    }
    uint64_t d = 0;
    d |= uint64_t((addr & 0x3FFFFu) >> 4);
    d |= uint64_t(1) << 16;
    d |= uint64_t(sbo >> 4) << 32;
    d |= uint64_t(1) << 46;
    d |= uint64_t(layout) << 61;
    return d;
}

// A walk over the CTA's chunks (tile-major, chunk-fastest) that yields, per
// chunk, its tile, slice, first column and width, and whether it opens a new
// row item (a new tile or slice, or the CTA's first chunk).  One division at
// the start; every step after it is a compare and an add.
struct TcCursor {
    int tile, c, s;                 // tile, chunk within the tile's chunk list, slice
    bool first;

    __device__ __forceinline__ void start(const TcArgs &p, int64_t w, int nchunks)
    {
        tile = int(w / nchunks);
        c = int(w - int64_t(tile) * nchunks);
        s = 0;
        while (s + 1 < p.num_slices && p.chunk0[s + 1] <= c) ++s;
        first = true;
    }
    __device__ __forceinline__ void next(const TcArgs &p, int nchunks)
    {
        if (++c == nchunks) {
            c = 0;
            ++tile;
            s = 0;
            first = true;
        } else if (c == p.chunk0[s + 1]) {
            ++s;
            first = true;
        } else {
            first = false;
        }
    }
    __device__ __forceinline__ int c0(const TcArgs &p) const { return (c - p.chunk0[s]) * TC_BN; }
    // Moves to the first chunk of the next row item; returns the chunks passed.
    __device__ __forceinline__ int skip_item(const TcArgs &p, int nchunks)
    {
        const int n = p.chunk0[s + 1] - c;
        c += n;
        if (c == nchunks) {
            c = 0;
            ++tile;
            s = 0;
        } else {
            ++s;
        }
        first = true;
        return n;
    }
};

// BIAS: some slice has a bias.  Without one the epilogue keeps fewer
// registers live, which lets rank 128 request both accumulator halves
// before finishing either (with the bias path compiled in, that spilled).
template <int KT, bool BIAS>
__global__ void __launch_bounds__(TcCfg<KT>::THREADS, 1) expand_tc_kernel(const __grid_constant__ TcArgs p)
{
    using C = TcCfg<KT>;
    constexpr bool OVERLAP = C::OVERLAP;
    constexpr bool ACC_BOTH = !C::OVERLAP && !BIAS;     // both halves' accumulators, then y
    constexpr int RP = C::RP, CPR = C::CPR, DEPTH = C::DEPTH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t base = smem_addr(smem);
    const uint32_t bar_bfull = base + C::BAR_OFF;          // [DEPTH]: B TMA bytes
    const uint32_t bar_yfull = bar_bfull + 8 * DEPTH;      // [DEPTH]: y loader threads
    const uint32_t bar_empty = bar_yfull + 8 * DEPTH;      // [DEPTH]: MMA + epilogue warps
    const uint32_t bar_accf = bar_empty + 8 * DEPTH;       // [TC_NACC]: MMA commit
    const uint32_t bar_acce = bar_accf + 8 * TC_NACC;      // [TC_NACC]: epilogue warps
    const uint32_t bar_x = bar_acce + 8 * TC_NACC;         // [TC_NXB] A operand ready: epilogue
    const uint32_t bar_drain = bar_x + 8 * TC_NXB;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // Every thread passes the grid-dependency wait before it exits; in early
    // mode the wait sits right before the first read of x (the shrink
    // output): the metadata, y, B and bias are final before this kernel
    // starts (see ExpandArgs::early).
    bool waited = false;
    auto wait_once = [&]() {
        if (!waited) {
            pdl_wait();
            pdl_launch_dependents();
            waited = true;
        }
    };
    if (!p.early) wait_once();

    if (tid == 0) {
        for (int i = 0; i < DEPTH; ++i) {
            mbar_init(bar_bfull + 8 * i, C::BISSUE);
            mbar_init(bar_yfull + 8 * i, C::LT);
            mbar_init(bar_empty + 8 * i, 1 + TC_EPI);
        }
        for (int i = 0; i < TC_NACC; ++i) {
            mbar_init(bar_accf + 8 * i, 1);
            mbar_init(bar_acce + 8 * i, TC_EPI);
        }
        for (int i = 0; i < TC_NXB; ++i) mbar_init(bar_x + 8 * i, TC_EPI);
        mbar_init(bar_drain, 1);
        mbar_fence_init();
        *s_abort = 0;
    }
    if (tid == 32)
        for (int s = 0; s < p.num_slices; ++s) tma_prefetch_map(&p.bmap[s]);
    const SegTab tab = seg_tab(reinterpret_cast<int *>(smem + C::TAB_OFF), p.nbins);
    const int total_tiles = load_segments(p.no_lora, p.active, p.counts, p.start_loc, p.nbins,
                                          TC_BM, tab, false, 0, p.num_tokens, p.error_word);
    const int S = p.num_slices;
    const int nchunks = p.chunk0[S];
    const int64_t total = int64_t(total_tiles) * nchunks;
    const int64_t w_begin = int64_t(blockIdx.x) * total / gridDim.x;
    const int64_t w_end = int64_t(blockIdx.x + 1) * total / gridDim.x;
    if (w_begin >= w_end) {                 // no tile, or no chunk for this CTA
        wait_once();
        return;
    }

    if (warp == 0) tmem_alloc(smem_addr(s_tmem), TC_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const long long deadline = clock64() + TC_TIMEOUT_CYCLES;
    const int R = p.rank, T = p.num_tokens;

    if (warp == 0) {
        // ------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_bf16(TC_BM, TC_BN);
            int g = 0, item = -1;
            uint32_t a_col = TC_A_COL;
            bool ok = true;
            TcCursor k;
            k.start(p, w_begin, nchunks);
            for (int64_t w = w_begin; w < w_end; ++w, ++g, k.next(p, nchunks)) {
                if (k.first) {
                    ++item;
                    if (!mbar_wait_bounded(bar_x + 8 * (item % TC_NXB),
                                           uint32_t(item / TC_NXB) & 1u, s_abort, deadline)) {
                        ok = false;
                        break;
                    }
                    a_col = TC_A_COL + uint32_t((item % TC_NXB) * C::A_COLS);
                }
                const int slot = g % DEPTH, ab = g % TC_NACC;
                if (!mbar_wait_bounded(bar_bfull + 8 * slot, uint32_t(g / DEPTH) & 1u, s_abort,
                                       deadline) ||
                    !mbar_wait_bounded(bar_acce + 8 * ab, (uint32_t(g / TC_NACC) & 1u) ^ 1u,
                                       s_abort, deadline)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t bt = base + C::RING_OFF + slot * C::SLOT_BYTES;
#pragma unroll
                for (int kk = 0; kk < KT; ++kk)
                    umma_bf16_tmem_a(tmem + ab * TC_BN, tmem + a_col + kk * 8,
                                     tc_kmajor_desc(RP, TC_BN, bt, kk), idesc, kk != 0);
                umma_commit(bar_empty + 8 * slot);           // B read
                umma_commit(bar_accf + 8 * ab);
            }
            // After an abort, wait (bounded) for every MMA issued so far
            // before TMEM is released.
            if (!ok || *s_abort) {
                umma_commit(bar_drain);
                const long long dd = clock64() + TC_TIMEOUT_CYCLES;
                while (!mbar_try_wait(bar_drain, 0) && clock64() < dd) {
                }
            }
        }
        __syncwarp();
    } else if (warp <= C::BISSUE) {
        // ------------------------------------------------------ B by TMA
        if (lane == 0) {
            int cur_tile = -1, l_id = 0, g = 0;
            TcCursor k;
            k.start(p, w_begin, nchunks);
            for (int64_t w = w_begin; w < w_end; ++w, ++g, k.next(p, nchunks)) {
                const int slot = g % DEPTH;
                if (!mbar_wait_backoff(bar_empty + 8 * slot, (uint32_t(g / DEPTH) & 1u) ^ 1u,
                                       s_abort, deadline, TC_BACKOFF_NS))
                    break;
                if (k.tile != cur_tile) {
                    cur_tile = k.tile;
                    l_id = tab.id[find_segment(tab.tile, p.nbins, cur_tile)];
                }
                // 64-row block of the chunk's first B row (n_s and c0 are
                // multiples of 64)
                const int blk = (l_id * p.n[k.s] + k.c0(p)) >> 6;
                const uint32_t bt = base + C::RING_OFF + slot * C::SLOT_BYTES;
                mbar_arrive_expect_tx(bar_bfull + 8 * slot, C::B_BYTES / C::BISSUE);
#pragma unroll
                for (int b = warp - 1; b < C::NBOX; b += C::BISSUE)
                    tma_load_5d(bt + b * TC_BN * 128, &p.bmap[k.s], b * C::BOX_K, 0, 0, 0, blk,
                                bar_bfull + 8 * slot);
            }
            // Before the CTA may exit, every issued load has landed: wait
            // (bounded) for the last phase of each slot in use.
            const int first = g > DEPTH ? g - DEPTH : 0;
            const long long dd = clock64() + TC_TIMEOUT_CYCLES;
            for (int j = first; j < g; ++j)
                while (!mbar_try_wait(bar_bfull + 8 * (j % DEPTH), uint32_t(j / DEPTH) & 1u) &&
                       clock64() < dd) {
                }
        }
        __syncwarp();
    } else if (warp < C::EPI0) {
        // ------------------------------------------------------ y loaders
        const int lt = tid - 32 * C::YL0;                  // 0 .. C::LT - 1
        const uint16_t *const ydummy = p.y;
        int cur_tile = -1;
        int ltok[C::Y_PER_T];                              // rows i * (LT / PPR) + lt / PPR
        int g = 0;
        TcCursor k;
        k.start(p, w_begin, nchunks);
        for (int64_t w = w_begin; w < w_end; ++w, ++g, k.next(p, nchunks)) {
            const int slot = g % DEPTH;
            const bool got = mbar_wait_backoff(bar_empty + 8 * slot,
                                               (uint32_t(g / DEPTH) & 1u) ^ 1u, s_abort, deadline,
                                               TC_BACKOFF_NS);
            if (__all_sync(0xffffffffu, got) == 0) break;
            if (p.add_inputs) {
                if (k.tile != cur_tile) {
                    cur_tile = k.tile;
                    const int seg = find_segment(tab.tile, p.nbins, cur_tile);
                    const int row0 = tab.start[seg] + (cur_tile - tab.tile[seg]) * TC_BM;
                    const int nrows = min(TC_BM, tab.start[seg] + tab.count[seg] - row0);
#pragma unroll
                    for (int i = 0; i < C::Y_PER_T; ++i) {
                        const int r = i * (C::LT / C::PPR) + lt / C::PPR;
                        ltok[i] = (r < nrows) ? checked_token(p.sorted[row0 + r], T, p.error_word)
                                              : -1;
                    }
                }
                const int c0 = k.c0(p), ncols = min(TC_BN, p.n[k.s] - c0);
                const int pc = lt % C::PPR;
                const bool cin = pc * 8 < ncols;
                const uint16_t *ycol = p.y + p.col0[k.s] + c0 + pc * 8;
                const uint32_t yt = base + C::RING_OFF + slot * C::SLOT_BYTES + C::B_BYTES;
#pragma unroll
                for (int i = 0; i < C::Y_PER_T; ++i) {
                    const int r = i * (C::LT / C::PPR) + lt / C::PPR;
                    const bool ld = cin && ltok[i] >= 0;
                    cp_async16(yt + tc_y_off(r, pc), ld ? ycol + int64_t(ltok[i]) * p.y_ld : ydummy,
                               ld);
                }
            }
            cp_async_mbar_arrive_noinc(bar_yfull + 8 * slot);
        }
        cp_async_wait<0>();
    } else {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3, h = (warp - C::EPI0) >> 2;
        const int my_row = q * 32 + lane;                  // TMEM lane (A operand row)
        const int qg = lane >> 2, qt = lane & 3;           // 16x256b fragment coordinates
        const int qrow = q * 32 + h * 16 + qg;             // this thread's rows: qrow, qrow + 8
        int ct = -1, c_id = 0, ctok = -1;
        int qtok[2];
        auto tile_rows = [&](int tile) {
            if (tile != ct) {
                ct = tile;
                const int seg = find_segment(tab.tile, p.nbins, ct);
                c_id = tab.id[seg];
                const int row0 = tab.start[seg] + (ct - tab.tile[seg]) * TC_BM;
                const int nrows = min(TC_BM, tab.start[seg] + tab.count[seg] - row0);
                ctok = (my_row < nrows) ? checked_token(p.sorted[row0 + my_row], T, p.error_word)
                                        : -1;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int r = qrow + 8 * u;
                    qtok[u] = (r < nrows) ? checked_token(p.sorted[row0 + r], T, p.error_word)
                                          : -1;
                }
            }
        };
        // this warp's row of x (slice s), half h of the rank, rounded to bf16
        // into A buffer buf's TMEM columns
        auto convert_x = [&](int s, int buf) {
            wait_once();                                   // x is the shrink output
            const int64_t xrow = (int64_t(s) * T + (ctok >= 0 ? ctok : 0)) * R;
            uint32_t wv[RP / 4];
#pragma unroll
            for (int j = 0; j < CPR / 2; ++j) {
                const int c = h * (CPR / 2) + j;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (ctok >= 0 && c * 8 < R) {
                    if (p.x_bf16) {
                        v = __ldcg(reinterpret_cast<const uint4 *>(
                            static_cast<const uint16_t *>(p.x) + xrow + c * 8));
                    } else {
                        const float4 *src = reinterpret_cast<const float4 *>(
                            static_cast<const float *>(p.x) + xrow + c * 8);
                        const float4 u = __ldcg(src), t = __ldcg(src + 1);
                        v.x = pack_bf16x2(u.x, u.y);
                        v.y = pack_bf16x2(u.z, u.w);
                        v.z = pack_bf16x2(t.x, t.y);
                        v.w = pack_bf16x2(t.z, t.w);
                    }
                }
                wv[4 * j] = v.x;
                wv[4 * j + 1] = v.y;
                wv[4 * j + 2] = v.z;
                wv[4 * j + 3] = v.w;
            }
            tmem_st<RP / 4>(tmem + (uint32_t(q * 32) << 16) +
                                uint32_t(TC_A_COL + buf * C::A_COLS + h * (RP / 4)),
                            wv);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_x + 8 * buf);
        };

        TcCursor k;
        k.start(p, w_begin, nchunks);
        {
            // the first TC_NXB row items' A operands, before the first chunk
            TcCursor kc = k;
            int64_t wc = w_begin;
            for (int n = 0; n < TC_NXB && wc < w_end; ++n) {
                tile_rows(kc.tile);
                convert_x(kc.s, n);
                wc += kc.skip_item(p, nchunks);
            }
        }
        int item = 0;                                  // row item of the current chunk

        int g = 0;
#pragma unroll 1
        for (int64_t w = w_begin; w < w_end; ++w, ++g) {
            tile_rows(k.tile);
            const int kc0 = k.c0(p), ks = k.s;
            const int ncols = min(TC_BN, p.n[ks] - kc0);
            const uint16_t *bias_row = (BIAS && p.bias[ks]) ? p.bias[ks] + int64_t(c_id) * p.n[ks] + kc0
                                                            : nullptr;
            const int ab = g % TC_NACC;
            const int slot = g % DEPTH;
            bool got = mbar_wait_bounded(bar_accf + 8 * ab, uint32_t(g / TC_NACC) & 1u, s_abort,
                                         deadline);
            got = got && mbar_wait_bounded(bar_yfull + 8 * slot, uint32_t(g / DEPTH) & 1u, s_abort,
                                           deadline);
            if (__all_sync(0xffffffffu, got) == 0) break;
            tc_fence_after();
            const int tok[2] = {qtok[0], qtok[1]};
            const uint8_t *yt = smem + C::RING_OFF + slot * C::SLOT_BYTES + C::B_BYTES;
            const bool has_bias = BIAS && bias_row != nullptr;
            // x B + old y + bias, rounded once, straight to y: output columns
            // 64 hf + 16 qt + 2j + e of the chunk are accumulator columns
            // 64 hf + 8j + 2 qt + e, registers acc[4j + e] (row qrow) and
            // acc[4j + 2 + e] (row qrow + 8); one 32-byte store per row.
            auto finish_half = [&](int hf, const uint32_t (&acc)[32], const uint4 (&yh)[2][2]) {
                const int cb = hf * 64 + qt * 16;
                const bool cin = cb < ncols;
                uint32_t bw[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                if (has_bias && cin) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint16_t *bq = bias_row + cb + j * 8;
                        uint4 v;
                        if (p.bias_vec) {
                            v = __ldg(reinterpret_cast<const uint4 *>(bq));
                        } else {
                            v.x = uint32_t(bq[0]) | (uint32_t(bq[1]) << 16);
                            v.y = uint32_t(bq[2]) | (uint32_t(bq[3]) << 16);
                            v.z = uint32_t(bq[4]) | (uint32_t(bq[5]) << 16);
                            v.w = uint32_t(bq[6]) | (uint32_t(bq[7]) << 16);
                        }
                        bw[4 * j] = v.x;
                        bw[4 * j + 1] = v.y;
                        bw[4 * j + 2] = v.z;
                        bw[4 * j + 3] = v.w;
                    }
                }
                uint16_t *ycol = p.y + p.col0[ks] + kc0 + cb;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (cin && tok[u] >= 0) {
                        const uint32_t yw[8] = {yh[u][0].x, yh[u][0].y, yh[u][0].z, yh[u][0].w,
                                                yh[u][1].x, yh[u][1].y, yh[u][1].z, yh[u][1].w};
                        uint32_t o[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float a0 = __uint_as_float(acc[4 * j + 2 * u]);
                            float a1 = __uint_as_float(acc[4 * j + 2 * u + 1]);
                            a0 += bf16_lo(yw[j]);
                            a1 += bf16_hi(yw[j]);
                            if (has_bias) {
                                a0 += bf16_lo(bw[j]);
                                a1 += bf16_hi(bw[j]);
                            }
                            o[j] = pack_bf16x2(a0, a1);
                        }
                        st_global_v8(ycol + int64_t(tok[u]) * p.y_ld, o);
                    }
                }
            };
            // this thread's old y of half hf (both rows, 32 bytes each)
            auto load_y = [&](int hf, uint4 (&yh)[2][2]) {
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        yh[u][e] = make_uint4(0u, 0u, 0u, 0u);
                        if (p.add_inputs)
                            yh[u][e] = *reinterpret_cast<const uint4 *>(
                                yt + tc_y_off(qrow + 8 * u, hf * 8 + 2 * qt + e));
                    }
            };
            // The accumulator goes back to the MMA once it is in registers;
            // when the next chunk opens a new tile or slice, its A operand is
            // written right then (the MMAs up to chunk g are done; that of
            // chunk g + 1 waits for it).
            auto release_acc = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_acce + 8 * ab);
                k.next(p, nchunks);
                if (w + 1 < w_end && k.first && ++item >= TC_NXB) {
                    tile_rows(k.tile);
                    convert_x(k.s, item % TC_NXB);
                }
            };
            const uint32_t tl = tmem + (uint32_t(q * 32 + h * 16) << 16) + uint32_t(ab * TC_BN);
            if constexpr (OVERLAP) {
                // both halves' accumulators and old y requested before any
                // is waited for: the chunk's latencies overlap
                uint32_t va[TC_HALVES][32];
                uint4 yv[TC_HALVES][2][2];
#pragma unroll
                for (int hf = 0; hf < TC_HALVES; ++hf)
                    tmem_ld16x256b_x8_nowait(tl + uint32_t(hf * 64), va[hf]);
#pragma unroll
                for (int hf = 0; hf < TC_HALVES; ++hf) load_y(hf, yv[hf]);
                tmem_wait_ld();
                release_acc();
#pragma unroll
                for (int hf = 0; hf < TC_HALVES; ++hf) finish_half(hf, va[hf], yv[hf]);
            } else if constexpr (ACC_BOTH) {
                // both halves' accumulators requested together (one TMEM
                // latency a chunk), old y read half by half
                uint32_t va[TC_HALVES][32];
#pragma unroll
                for (int hf = 0; hf < TC_HALVES; ++hf)
                    tmem_ld16x256b_x8_nowait(tl + uint32_t(hf * 64), va[hf]);
                tmem_wait_ld();
                release_acc();
#pragma unroll
                for (int hf = 0; hf < TC_HALVES; ++hf) {
                    uint4 yv[2][2];
                    load_y(hf, yv);
                    finish_half(hf, va[hf], yv);
                }
            } else {
#pragma unroll
                for (int hf = 0; hf < TC_HALVES; ++hf) {
                    uint32_t va[32];
                    uint4 yv[2][2];
                    tmem_ld16x256b_x8_nowait(tl + uint32_t(hf * 64), va);
                    tmem_wait_ld();
                    if (hf == TC_HALVES - 1) release_acc();
                    load_y(hf, yv);
                    finish_half(hf, va, yv);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * slot);   // done with the slot's y
        }
    }

    wait_once();
    if (tid == 0 && *s_abort) atomicOr(p.error_word, TC_ERROR_BIT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TC_TMEM_COLS);
}

template <int KT>
static int launch_tc_kt(const TcArgs &p, cudaStream_t stream)
{
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return int(e);
    const size_t smem = tc_smem_bytes<KT>(p.nbins);
    if (smem > 227 * 1024) return TC_NO_FIT;
    if (dev < 64 && configured[dev] == 0) {
        e = cudaFuncSetAttribute(expand_tc_kernel<KT, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return int(e);
        e = cudaFuncSetAttribute(expand_tc_kernel<KT, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return int(e);
        configured[dev] = 1;
    }
    bool bias = false;
    for (int s = 0; s < p.num_slices; ++s) bias = bias || p.bias[s] != nullptr;
    e = launch_kernel(bias ? expand_tc_kernel<KT, true> : expand_tc_kernel<KT, false>,
                      dim3(device_sm_count()), dim3(TcCfg<KT>::THREADS), smem, stream, p);
    return e == cudaSuccess ? int(TC_LAUNCHED) : int(e);
}

// Launches the tensor-core expand: returns TC_LAUNCHED, TC_NO_FIT or
// TC_MISALIGNED if the call does not fit it (the caller then runs the
// mma.sync kernel), or a cudaError_t.
int launch_expand_tc(const ExpandLaunch &a, cudaStream_t stream)
{
    if (!a.vec) return TC_MISALIGNED;
    if (a.error_word == nullptr) return TC_NO_FIT;
    TcArgs p;
    p.x = a.x;
    p.x_bf16 = a.x_bf16;
    int chunks = 0;
    for (int s = 0; s < LORA_MAX_SLICES; ++s) {
        p.b[s] = a.b[s];
        p.bias[s] = a.bias[s];
        p.n[s] = a.n[s];
        p.col0[s] = a.col0[s];
        p.chunk0[s] = 0;
    }
    for (int s = 0; s < a.num_slices; ++s) {
        p.chunk0[s] = chunks;
        chunks += (a.n[s] + TC_BN - 1) / TC_BN;
    }
    p.chunk0[a.num_slices] = chunks;
    // B by TMA through the row-permuting map: every slice's width must be a
    // multiple of 64 (each LoRA's rows start a 64-row block); y's rows are
    // written with 32-byte stores: y, its row stride and every slice's first
    // column 32-byte aligned
    const uint32_t rp = a.rank <= 16 ? 16u : a.rank <= 32 ? 32u : a.rank <= 64 ? 64u : 128u;
    const CUtensorMapSwizzle sw = rp == 16 ? CU_TENSOR_MAP_SWIZZLE_32B
                                  : rp == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_128B;
    if (reinterpret_cast<uintptr_t>(a.y) % 32 != 0 || a.y_ld % 16 != 0) return TC_MISALIGNED;
    for (int s = 0; s < a.num_slices; ++s) {
        if (a.col0[s] % 16 != 0) return TC_MISALIGNED;
        if (a.n[s] % 64 != 0) return TC_NO_FIT;
    }
    for (int s = 0; s < a.num_slices; ++s)
        if (!encode_perm_rows_map(&p.bmap[s], a.b[s], uint64_t(a.max_loras) * uint64_t(a.n[s]),
                                  uint32_t(a.rank), rp < 64 ? rp : 64u, uint32_t(TC_HALVES), sw))
            return int(cudaErrorInvalidValue);
    for (int s = a.num_slices; s < LORA_MAX_SLICES; ++s) p.bmap[s] = p.bmap[0];
    p.num_slices = a.num_slices;
    p.rank = a.rank;
    p.y = a.y;
    p.y_ld = a.y_ld;
    p.num_tokens = a.num_tokens;
    p.add_inputs = a.add_inputs;
    p.bias_vec = a.bias_vec;
    p.early = a.early;
    p.sorted = a.sorted;
    p.counts = a.counts;
    p.start_loc = a.start_loc;
    p.active = a.active;
    p.no_lora = a.no_lora;
    p.error_word = a.error_word;
    p.nbins = a.max_loras + 1;
    if (a.rank <= 16) return launch_tc_kt<1>(p, stream);
    if (a.rank <= 32) return launch_tc_kt<2>(p, stream);
    if (a.rank <= 64) return launch_tc_kt<4>(p, stream);
    return launch_tc_kt<8>(p, stream);
}

}  // namespace lora
