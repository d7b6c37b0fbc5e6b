// lora_linear_tc.cu -- the shrink and the expand of one LoRA layer in one
// tensor-core kernel, tile by tile (page "vllm.lora.punica_wrapper.
// punica_gpu", PunicaWrapperGPU.add_lora_linear: add_shrink into the fp32
// buffer, then add_expand of that buffer into y; bias step of page
// "vllm.lora.punica_wrapper.punica_tpu", PunicaWrapperTPU._apply_bias).
//
// For rank 128 and at most three slices, one persistent CTA per SM takes
// one 128-token tile of one LoRA segment at a time and runs, on its SM:
//   phase 1  the shrink of the tile: x rows and A blocks by TMA, tcgen05
//            UMMAs (M = 128 tokens, slices 0 and 1 in one N = 256 UMMA)
//            into a TMEM accumulator of S x 128 fp32 columns, as in
//            lora_shrink_umma.cu;
//   phase 2  buf[s][t, :] = old + scale * acc for the tile's tokens (the
//            old rows by TMA into the freed ring, the new ones written over
//            them there and stored by TMA: the tile's CTA is their only
//            writer), and the same values rounded to bf16 into TMEM as the
//            expand's A operands;
//   phase 3  the expand of the tile over every 128-column chunk of every
//            slice: B by TMA, old y by cp.async, UMMAs with A from TMEM,
//            32-byte stores, as in lora_expand_tc.cu.
// Against the shrink kernel followed by the expand kernel this drops the
// buffer's reductions and its reread, the expand's conversion of x at the
// start of its row items, and the tail of one kernel before the next.
//
// The phases of a tile are separated by CTA-wide barriers, so the ring of
// three 64 KB slots (a shrink stage: x 16 KB + 3 A blocks; an expand slot:
// B 32 KB + y 32 KB; in phase 2 one slice's old buffer rows) and the TMEM
// columns change hands only when nothing is in flight on them.
//
// TMEM (512 columns): phase 1 accumulates slice s at columns 128 s; phase 2
// writes the A operands of slices 0 and 1 at columns 384 and 448 (free in
// phase 1) and that of slice 2 at column 0 (after every conversion warp has
// read the accumulator there); phase 3 alternates two accumulators at
// columns 128 and 256.
//
// Every mbarrier wait is bounded (about one second); on expiry the kernel
// sets bit 30 of the metadata error word, every role stops issuing, and the
// CTA waits (bounded) for its copies and MMAs in flight before it frees
// TMEM and returns.
#include "lora_common.cuh"
#include "lora_umma.cuh"

namespace lora {

constexpr int LT_BM = 128;            // tokens per tile (UMMA M)
constexpr int LT_R = 128;             // rank (the only one this kernel takes)
constexpr int LT_BK = 64;             // hidden per shrink stage
constexpr int LT_BN = 128;            // columns per expand chunk (UMMA N)
constexpr int LT_MAXS = 3;            // slices
constexpr int LT_SLOTS = 3;           // ring slots, both phases
constexpr int LT_SLOT = 65536;        // bytes per slot
constexpr int LT_XMAPS = 8;           // box heights 1, 2, 4, ..., 128
constexpr int LT_EPI = 8;             // conversion / epilogue warps
constexpr int LT_ST_ISSUERS = 6;      // warps moving a tile's buffer rows by TMA (phase 2)
constexpr int LT_W_X = 0;             // x producer; old-buffer loads; B issuer 0
constexpr int LT_W_MMA = 1;           // TMEM owner, UMMA issue
constexpr int LT_W_B1 = 2;            // A producer of slice 0; B issuer 1
constexpr int LT_W_YL0 = 3;           // A producers of slices 1, 2; y loaders 3..6
constexpr int LT_YL = 4;              // y loader warps
constexpr int LT_W_EPI0 = LT_W_YL0 + LT_YL;
constexpr int LT_THREADS = 32 * (LT_W_EPI0 + LT_EPI);
static_assert(LT_ST_ISSUERS == 2 + LT_YL, "buffer-row issuers: the x producer, B issuer 1, the y loaders");
constexpr int LT_ACC_A01 = 384;       // TMEM columns of the A operands of slices 0, 1 (+64)
constexpr int LT_ACC3 = 128;          // phase-3 accumulators at 128 and 256
constexpr long long LT_TIMEOUT_CYCLES = 2000000000ll;
constexpr uint32_t LT_BACKOFF_NS = 200;
constexpr int LT_ERROR_BIT = 1 << 30;

struct LinearTcArgs {
    CUtensorMap map_x[LT_XMAPS];              // x: [T, H] bf16, box {64, 2^i}, 128B swizzle
    CUtensorMap map_a[LT_MAXS];               // A[s]: [L * 128, H] bf16, box {64, 128}
    CUtensorMap map_buf[LT_XMAPS];            // buf: [S * T, 128] fp32, box {32, 2^i}
    CUtensorMap map_b[LT_MAXS];               // B[s] rows, permuted (encode_perm_rows_map)
    const uint16_t *bias[LT_MAXS];            // [L, n_s] or null
    int32_t n[LT_MAXS];                       // slice widths (multiples of 64)
    int32_t col0[LT_MAXS];                    // first y column of each slice
    int32_t chunk0[LT_MAXS + 1];              // first chunk of each slice
    int32_t num_slices;
    int32_t hidden;
    int32_t num_tokens;
    float scale;
    float *buf;                               // [S, T, 128] fp32
    uint16_t *y;
    int64_t y_ld;
    int32_t bias_vec;
    const int32_t *sorted;
    const int32_t *counts;
    const int32_t *start_loc;
    const int32_t *active;
    const int32_t *no_lora;
    int32_t *error_word;
    int32_t nbins;
};

// Shared memory: the ring, then the barriers, the piece list and the
// segment table.
struct LtLayout {
    static constexpr int RING = LT_SLOTS * LT_SLOT;
    // full1, empty1 [3]; accf1; bufb; bfull, yfull, empty3 [3]; accf, acce [2]; drain
    static constexpr int NBARS = 3 + 3 + 1 + 1 + 3 + 3 + 3 + 2 + 2 + 1;
    static constexpr int BAR = RING;
    static constexpr int MISC = BAR + NBARS * 8;          // tmem base, abort flag
    static constexpr int PIECES = MISC + 16;              // [LT_BM] (row, token, log2 rows)
    static constexpr int TAB = PIECES + LT_BM * 4;
};

inline size_t linear_tc_smem_bytes(int nbins)
{
    return size_t(LtLayout::TAB) + seg_tab_bytes(nbins) + 1024;      // + alignment slack
}

// Byte offset of 16-byte piece `pc` (columns 8 pc .. 8 pc + 7) of row `r` of
// a slot's old y rows (two 64-column halves, 128-byte swizzled).
__device__ __forceinline__ uint32_t lt_y_off(int r, int pc)
{
    return uint32_t((pc >> 3) * (LT_BM * 128) + r * 128 + (((pc & 7) ^ (r & 7)) << 4));
}

// Descriptor of K step kk (16 bf16) of a slot's B tile: two boxes of 64
// rank elements (128-byte rows, 128-byte swizzle), 128 rows each.
__device__ __forceinline__ uint64_t lt_b_desc(uint32_t tile, int kk)
{
    return umma_desc_sw128(tile + uint32_t((kk >> 2) * LT_BN * 128 + (kk & 3) * 32));
}

// TMEM column of slice s's A operand in phase 3.
__device__ __forceinline__ uint32_t lt_a_col(int s)
{
    return s == 2 ? 0u : uint32_t(LT_ACC_A01 + 64 * s);
}

// Cuts a tile's tokens (increasing: the sort is stable) into pieces of
// consecutive tokens whose heights are powers of two, each starting at a
// row that is a multiple of its height: one TMA box per piece.
__device__ __forceinline__ int lt_pieces(const int32_t *tk, int nrows, uint32_t *pieces)
{
    int n = 0, j = 0;
    while (j < nrows) {
        int lg = 7;
        while ((1 << lg) > nrows - j || (j & ((1 << lg) - 1)) != 0 ||
               tk[j + (1 << lg) - 1] - tk[j] != (1 << lg) - 1)
            --lg;
        pieces[n++] = uint32_t(j) | (uint32_t(lg) << 8) | (uint32_t(tk[j]) << 11);
        j += 1 << lg;
    }
    return n;
}

template <bool BIAS>
__global__ void __launch_bounds__(LT_THREADS, 1) linear_tc_kernel(const __grid_constant__ LinearTcArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t base = smem_addr(smem);
    const uint32_t full1 = base + LtLayout::BAR;            // [3] shrink stage landed
    const uint32_t empty1 = full1 + 24;                     // [3] shrink stage read (MMA commit)
    const uint32_t accf1 = empty1 + 24;                     // shrink accumulator complete
    const uint32_t bufb = accf1 + 8;                        // old buffer rows landed
    const uint32_t bfull = bufb + 8;                        // [3] B landed (two issuers)
    const uint32_t yfull = bfull + 24;                      // [3] old y landed (loader threads)
    const uint32_t empty3 = yfull + 24;                     // [3] slot read (MMA + epilogue warps)
    const uint32_t accf = empty3 + 24;                      // [2] expand accumulator complete
    const uint32_t acce = accf + 16;                        // [2] expand accumulator read
    const uint32_t drain = acce + 16;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + LtLayout::MISC);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + LtLayout::MISC + 4);
    volatile int *s_np = reinterpret_cast<volatile int *>(smem + LtLayout::MISC + 8);
    uint32_t *pieces = reinterpret_cast<uint32_t *>(smem + LtLayout::PIECES);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.num_slices, T = p.num_tokens, H = p.hidden;

    if (tid == 0) {
        for (int i = 0; i < LT_SLOTS; ++i) {
            mbar_init(full1 + 8 * i, 1 + S);
            mbar_init(empty1 + 8 * i, 1);
            mbar_init(bfull + 8 * i, 2);
            mbar_init(yfull + 8 * i, 32 * LT_YL);
            mbar_init(empty3 + 8 * i, 1 + LT_EPI);
        }
        mbar_init(accf1, 1);
        mbar_init(bufb, LT_ST_ISSUERS);
        for (int i = 0; i < 2; ++i) {
            mbar_init(accf + 8 * i, 1);
            mbar_init(acce + 8 * i, LT_EPI);
        }
        mbar_init(drain, 1);
        mbar_fence_init();
        *s_abort = 0;
    }
    if (tid == 32) {
        for (int i = 0; i < LT_XMAPS; ++i) {
            tma_prefetch_map(&p.map_x[i]);
            tma_prefetch_map(&p.map_buf[i]);
        }
        for (int s = 0; s < S; ++s) {
            tma_prefetch_map(&p.map_a[s]);
            tma_prefetch_map(&p.map_b[s]);
        }
    }
    // (barriers and tensor maps above need nothing from the metadata kernel:
    // they are set up while it runs)
    pdl_wait();
    pdl_launch_dependents();
    const SegTab tab = seg_tab(reinterpret_cast<int *>(smem + LtLayout::TAB), p.nbins);
    const int total_tiles = load_segments(p.no_lora, p.active, p.counts, p.start_loc, p.nbins,
                                          LT_BM, tab, false, 0, T, p.error_word);
    // Items: when the tiles are fewer than the CTAs, the first `extra` tiles
    // are cut into two 64-row halves (items 2j and 2j + 1), the others are
    // whole (item extra + t): the idle SMs take half of those tiles, and the
    // first one (on a mixed batch, the one whose tokens break into the most
    // runs, whose CTA finished 18 us after the next) is among them.
    const int extra = total_tiles < int(gridDim.x) ? min(int(gridDim.x) - total_tiles, total_tiles)
                                                   : 0;
    const int total_items = total_tiles + extra;
    if (int(blockIdx.x) >= total_items) return;             // (the same in every thread)

    if (warp == LT_W_MMA) tmem_alloc(smem_addr(s_tmem), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const long long deadline = clock64() + LT_TIMEOUT_CYCLES;
    const int nk = (H + LT_BK - 1) / LT_BK;
    const int nchunks = p.chunk0[S];
    int n1 = 0;                  // shrink stages so far (stage n1 % 3)
    int g3 = 0;                  // expand chunks so far (slot g3 % 3, accumulator g3 % 2)
    int it = 0;                  // tiles so far

    for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
        const int tile = item < 2 * extra ? item >> 1 : item - extra;
        const int half = item < 2 * extra ? (item & 1) : -1;
        const int seg = find_segment(tab.tile, p.nbins, tile);
        const int l_id = tab.id[seg];
        int row0 = tab.start[seg] + (tile - tab.tile[seg]) * LT_BM;
        int nrows = min(LT_BM, tab.start[seg] + tab.count[seg] - row0);
        if (half >= 0) {
            row0 += 64 * half;
            nrows = min(64, nrows - 64 * half);
        }
        if (nrows <= 0) continue;            // (an empty second half: the same in every thread)
        int npieces = 0;         // (lane 0 of the x producer)

        // ============================================================ phase 1: shrink
        if (warp == LT_W_X) {
            if (lane == 0) {
                npieces = lt_pieces(p.sorted + row0, nrows, pieces);
                *s_np = npieces;             // for the buffer-row issuers of phase 2
            }
            const int np = __shfl_sync(0xffffffffu, npieces, 0);
            __syncwarp();
            int issued = 0;
            for (int kb = 0; kb < nk; ++kb) {
                const int n = n1 + kb, stage = n % LT_SLOTS;
                const bool got = mbar_wait_bounded(empty1 + 8 * stage,
                                                   (uint32_t(n / LT_SLOTS) & 1u) ^ 1u, s_abort,
                                                   deadline);
                if (__all_sync(0xffffffffu, got) == 0) break;
                const uint32_t sx = base + stage * LT_SLOT;
                if (lane == 0) mbar_arrive_expect_tx(full1 + 8 * stage, uint32_t(nrows * 128));
                __syncwarp();
                for (int i = lane; i < np; i += 32) {
                    const uint32_t pc = pieces[i];
                    const int r = int(pc & 0xFFu), lg = int((pc >> 8) & 7u), t0 = int(pc >> 11);
                    tma_load_2d(sx + r * 128, &p.map_x[lg], kb * LT_BK, t0, full1 + 8 * stage);
                }
                ++issued;
            }
            if (lane == 0) {                 // every issued fill lands before the ring is reused
                const long long dd = clock64() + LT_TIMEOUT_CYCLES;
                for (int i = max(0, issued - LT_SLOTS); i < issued; ++i) {
                    const int n = n1 + i;
                    while (!mbar_try_wait(full1 + 8 * (n % LT_SLOTS), uint32_t(n / LT_SLOTS) & 1u) &&
                           clock64() < dd) {
                    }
                }
            }
            __syncwarp();
        } else if (warp == LT_W_B1 || warp == LT_W_YL0 || warp == LT_W_YL0 + 1) {
            // A producer of slice sa: its block of 128 rows per stage
            const int sa = warp == LT_W_B1 ? 0 : warp - LT_W_YL0 + 1;
            if (sa < S && lane == 0) {
                int issued = 0;
                for (int kb = 0; kb < nk; ++kb) {
                    const int n = n1 + kb, stage = n % LT_SLOTS;
                    if (!mbar_wait_bounded(empty1 + 8 * stage, (uint32_t(n / LT_SLOTS) & 1u) ^ 1u,
                                           s_abort, deadline))
                        break;
                    mbar_arrive_expect_tx(full1 + 8 * stage, uint32_t(LT_R * LT_BK * 2));
                    tma_load_2d(base + stage * LT_SLOT + (1 + sa) * (LT_R * LT_BK * 2), &p.map_a[sa],
                                kb * LT_BK, l_id * LT_R, full1 + 8 * stage);
                    ++issued;
                }
                const long long dd = clock64() + LT_TIMEOUT_CYCLES;
                for (int i = max(0, issued - LT_SLOTS); i < issued; ++i) {
                    const int n = n1 + i;
                    while (!mbar_try_wait(full1 + 8 * (n % LT_SLOTS), uint32_t(n / LT_SLOTS) & 1u) &&
                           clock64() < dd) {
                    }
                }
            }
            __syncwarp();
        } else if (warp == LT_W_MMA) {
            if (lane == 0) {
                // slices 0 and 1 in one UMMA of N = 256 (adjacent A blocks and
                // TMEM columns), slice 2 alone
                const int G = S < 2 ? S : 2;
                const uint32_t idesc_g = umma_idesc_bf16(LT_BM, G * LT_R);
                const uint32_t idesc_1 = umma_idesc_bf16(LT_BM, LT_R);
                bool ok = true;
                for (int kb = 0; kb < nk; ++kb) {
                    const int n = n1 + kb, stage = n % LT_SLOTS;
                    if (!mbar_wait_bounded(full1 + 8 * stage, uint32_t(n / LT_SLOTS) & 1u, s_abort,
                                           deadline)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sx = base + stage * LT_SLOT;
#pragma unroll
                    for (int kk = 0; kk < LT_BK / 16; ++kk) {
                        const uint64_t adesc = umma_desc_sw128(sx + kk * 32);
                        const uint32_t acc_on = (kb != 0 || kk != 0) ? 1u : 0u;
                        umma_bf16(tmem, adesc, umma_desc_sw128(sx + LT_R * LT_BK * 2 + kk * 32),
                                  idesc_g, acc_on);
                        if (S == 3)
                            umma_bf16(tmem + 2 * LT_R, adesc,
                                      umma_desc_sw128(sx + 3 * LT_R * LT_BK * 2 + kk * 32), idesc_1,
                                      acc_on);
                    }
                    umma_commit(empty1 + 8 * stage);
                }
                if (ok) umma_commit(accf1);
            }
            __syncwarp();
        } else if (warp >= LT_W_EPI0) {
            // idle in this phase: bring the tile's old buffer rows into L2
            // (three 512-byte rows a token), which phase 2 reads.  Read there
            // from HBM by every CTA at once, they took 11-17 us.
            const int nl = S * nrows * 4;                    // 128-byte lines
            for (int i = tid - 32 * LT_W_EPI0; i < nl; i += 32 * LT_EPI) {
                const int sb = i / (nrows * 4), rem = i - sb * nrows * 4;
                const int rr = rem >> 2, j = rem & 3;
                const int tk = p.sorted[row0 + rr];
                if (tk >= 0 && tk < T)
                    prefetch_l2(p.buf + (int64_t(sb) * T + tk) * LT_R + 32 * j);
            }
        }
        n1 += nk;
        fence_proxy_async_smem();
        if (__syncthreads_or(*s_abort != 0)) break;      // (one answer for the whole CTA)

        // ============================================================ phase 2: buffer, A operands
        if (warp == LT_W_X || warp == LT_W_B1 || (warp >= LT_W_YL0 && warp < LT_W_EPI0)) {
            // LT_ST_ISSUERS warps (the x producer, B issuer 1 and the y
            // loaders; idle here) move the tile's buffer rows, one box per
            // (slice, run, 32-column block), box i by warp i / 32 mod
            // LT_ST_ISSUERS.  Slot s receives slice s's old rows: four
            // 32-column blocks of 128 rows x 128 bytes, 128-byte swizzled.
            // Issued by one warp, the stores' reads of the ring took 6 us
            // (every CTA storing at once); a thread's 16-byte stores of its
            // own row (32 lines a warp store) 9 us; 512-byte rows by warp
            // stores 8 us.
            const int k = warp == LT_W_X ? 0 : warp == LT_W_B1 ? 1 : 2 + warp - LT_W_YL0;
            const int np = *s_np;
            const int nbox = S * np * 4;
            bool go = true;
            if (lane == 0) {
                // the ring is free once the shrink's last UMMAs have completed
                go = mbar_wait_bounded(accf1, uint32_t(it) & 1u, s_abort, deadline);
                uint32_t bytes = 0;
                for (int i = 32 * k; i < nbox; i += 32 * LT_ST_ISSUERS)
                    for (int l = i; l < min(i + 32, nbox); ++l)
                        bytes += (128u << ((pieces[(l % (np * 4)) >> 2] >> 8) & 7u));
                if (go) mbar_arrive_expect_tx(bufb, bytes);
            }
            go = __shfl_sync(0xffffffffu, go ? 1 : 0, 0) != 0;
            if (go)
                for (int i = 32 * k + lane; i < nbox; i += 32 * LT_ST_ISSUERS) {
                    const int sb = i / (np * 4), rem = i - sb * np * 4, pi = rem >> 2, j = rem & 3;
                    const uint32_t pc = pieces[pi];
                    const int r = int(pc & 0xFFu), lg = int((pc >> 8) & 7u), t0 = int(pc >> 11);
                    tma_load_2d(base + sb * LT_SLOT + j * (LT_BM * 128) + r * 128, &p.map_buf[lg],
                                32 * j, sb * T + t0, bufb);
                }
            if (lane == 0 && go) {               // they land before the ring changes hands
                const long long dd = clock64() + LT_TIMEOUT_CYCLES;
                while (!mbar_try_wait(bufb, uint32_t(it) & 1u) && clock64() < dd) {
                }
            }
            __syncwarp();
            // the conversion warps have written the new rows over the old
            // ones in shared memory: they leave with the same boxes
            asm volatile("bar.sync 1, %0;\n" :: "n"(32 * (LT_EPI + LT_ST_ISSUERS)) : "memory");
            if (__shfl_sync(0xffffffffu, *s_abort == 0 ? 1 : 0, 0) != 0) {
                for (int i = 32 * k + lane; i < nbox; i += 32 * LT_ST_ISSUERS) {
                    const int sb = i / (np * 4), rem = i - sb * np * 4, pi = rem >> 2, j = rem & 3;
                    const uint32_t pc = pieces[pi];
                    const int r = int(pc & 0xFFu), lg = int((pc >> 8) & 7u), t0 = int(pc >> 11);
                    tma_store_2d(&p.map_buf[lg], 32 * j, sb * T + t0,
                                 base + sb * LT_SLOT + j * (LT_BM * 128) + r * 128);
                }
                bulk_commit_group();
                bulk_wait_group_read0();             // the ring is read before it changes hands
            }
            __syncwarp();
        } else if (warp >= LT_W_EPI0) {
            // thread = TMEM lane (token row r), half h of each slice's 128 columns
            const int q = warp & 3, h = (warp - LT_W_EPI0) >> 2;
            const int r = q * 32 + lane;
            bool ok = mbar_wait_bounded(accf1, uint32_t(it) & 1u, s_abort, deadline);
            ok = ok && mbar_wait_bounded(bufb, uint32_t(it) & 1u, s_abort, deadline);
            ok = __all_sync(0xffffffffu, ok) != 0;
            const uint32_t tl = tmem + (uint32_t(q * 32) << 16);
            uint32_t w2[2][16];                     // slice 2's A words (written last)
            if (ok) {
                tc_fence_after();
                for (int sb = 0; sb < S; ++sb) {
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int c0 = 64 * h + 32 * u;              // column of the slice
                        uint32_t a[32];
                        tmem_ld32_nowait(tl + uint32_t(sb * LT_R + c0), a);
                        tmem_wait_ld();
                        uint8_t *blk = smem + sb * LT_SLOT + (2 * h + u) * (LT_BM * 128) + r * 128;
                        float v[32];
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            float4 *cell = reinterpret_cast<float4 *>(blk + ((c ^ (r & 7)) << 4));
                            const float4 o = *cell;
                            v[4 * c] = o.x + p.scale * __uint_as_float(a[4 * c]);
                            v[4 * c + 1] = o.y + p.scale * __uint_as_float(a[4 * c + 1]);
                            v[4 * c + 2] = o.z + p.scale * __uint_as_float(a[4 * c + 2]);
                            v[4 * c + 3] = o.w + p.scale * __uint_as_float(a[4 * c + 3]);
                            // the new row over the old one (stored by TMA: rows past
                            // the segment are not)
                            *cell = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                        }
                        uint32_t wv[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k) wv[k] = pack_bf16x2(v[2 * k], v[2 * k + 1]);
                        if (sb < 2) {
                            tmem_st<16>(tl + lt_a_col(sb) + uint32_t(c0 / 2), wv);
                        } else {
#pragma unroll
                            for (int k = 0; k < 16; ++k) w2[u][k] = wv[k];
                        }
                    }
                }
            }
            // slice 2's A operand goes over the accumulator of slice 0: only
            // once every conversion warp has read it; the new rows go out
            // once all are in shared memory (the barrier is taken by the
            // eight conversion warps and the LT_ST_ISSUERS issuers, whatever
            // happened above)
            fence_proxy_async_smem();
            asm volatile("bar.sync 1, %0;\n" :: "n"(32 * (LT_EPI + LT_ST_ISSUERS)) : "memory");
            if (ok && S == 3) {
#pragma unroll
                for (int u = 0; u < 2; ++u)
                    tmem_st<16>(tl + lt_a_col(2) + uint32_t((64 * h + 32 * u) / 2), w2[u]);
            }
            tmem_wait_st();
        }
        tc_fence_before();
        fence_proxy_async_smem();
        const bool stop = __syncthreads_or(*s_abort != 0) != 0;
        tc_fence_after();
        if (stop) break;

        // ============================================================ phase 3: expand
        if (warp == LT_W_X || warp == LT_W_B1) {
            // B issuers: one 64-rank box of the chunk's B tile each
            if (lane == 0) {
                const int b = warp == LT_W_X ? 0 : 1;
                int sc = 0, issued = 0;
                for (int c = 0; c < nchunks; ++c) {
                    while (sc + 1 < S && p.chunk0[sc + 1] <= c) ++sc;
                    const int g = g3 + c, slot = g % LT_SLOTS;
                    if (!mbar_wait_backoff(empty3 + 8 * slot, (uint32_t(g / LT_SLOTS) & 1u) ^ 1u,
                                           s_abort, deadline, LT_BACKOFF_NS))
                        break;
                    // 64-row block of the chunk's first B row (n_s and the
                    // chunk's first column are multiples of 64)
                    const int blk = (l_id * p.n[sc] + (c - p.chunk0[sc]) * LT_BN) >> 6;
                    mbar_arrive_expect_tx(bfull + 8 * slot, uint32_t(LT_BN * 64 * 2));
                    tma_load_5d(base + slot * LT_SLOT + b * (LT_BN * 128), &p.map_b[sc], b * 64, 0,
                                0, 0, blk, bfull + 8 * slot);
                    ++issued;
                }
                const long long dd = clock64() + LT_TIMEOUT_CYCLES;
                for (int i = max(0, issued - LT_SLOTS); i < issued; ++i) {
                    const int g = g3 + i;
                    while (!mbar_try_wait(bfull + 8 * (g % LT_SLOTS), uint32_t(g / LT_SLOTS) & 1u) &&
                           clock64() < dd) {
                    }
                }
            }
            __syncwarp();
        } else if (warp >= LT_W_YL0 && warp < LT_W_EPI0) {
            // old y loaders: 16-byte pieces; thread lt takes piece lt % 16 of
            // rows i * 8 + lt / 16 (i < 16) of every chunk
            const int lt = tid - 32 * LT_W_YL0;
            int ltok[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int rr = i * 8 + lt / 16;
                ltok[i] = rr < nrows ? checked_token(p.sorted[row0 + rr], T, p.error_word) : -1;
            }
            const int pc = lt % 16;
            int sc = 0;
            for (int c = 0; c < nchunks; ++c) {
                while (sc + 1 < S && p.chunk0[sc + 1] <= c) ++sc;
                const int g = g3 + c, slot = g % LT_SLOTS;
                const bool got = mbar_wait_backoff(empty3 + 8 * slot,
                                                   (uint32_t(g / LT_SLOTS) & 1u) ^ 1u, s_abort,
                                                   deadline, LT_BACKOFF_NS);
                if (__all_sync(0xffffffffu, got) == 0) break;
                const int c0 = (c - p.chunk0[sc]) * LT_BN;
                const bool cin = pc * 8 < min(LT_BN, p.n[sc] - c0);
                const uint16_t *ycol = p.y + p.col0[sc] + c0 + pc * 8;
                const uint32_t yt = base + slot * LT_SLOT + LT_BN * LT_R * 2;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const bool ld = cin && ltok[i] >= 0;
                    cp_async16(yt + lt_y_off(i * 8 + lt / 16, pc),
                               ld ? ycol + int64_t(ltok[i]) * p.y_ld : p.y, ld);
                }
                cp_async_mbar_arrive_noinc(yfull + 8 * slot);
            }
            cp_async_wait<0>();
        } else if (warp == LT_W_MMA) {
            if (lane == 0) {
                const uint32_t idesc = umma_idesc_bf16(LT_BM, LT_BN);
                int sc = 0;
                for (int c = 0; c < nchunks; ++c) {
                    while (sc + 1 < S && p.chunk0[sc + 1] <= c) ++sc;
                    const int g = g3 + c, slot = g % LT_SLOTS, ab = g % 2;
                    if (!mbar_wait_bounded(bfull + 8 * slot, uint32_t(g / LT_SLOTS) & 1u, s_abort,
                                           deadline) ||
                        !mbar_wait_bounded(acce + 8 * ab, (uint32_t(g / 2) & 1u) ^ 1u, s_abort,
                                           deadline))
                        break;
                    tc_fence_after();
                    const uint32_t bt = base + slot * LT_SLOT;
#pragma unroll
                    for (int kk = 0; kk < LT_R / 16; ++kk)
                        umma_bf16_tmem_a(tmem + uint32_t(LT_ACC3 + LT_BN * ab),
                                         tmem + lt_a_col(sc) + uint32_t(kk * 8), lt_b_desc(bt, kk),
                                         idesc, kk != 0);
                    umma_commit(empty3 + 8 * slot);             // B read
                    umma_commit(accf + 8 * ab);
                }
            }
            __syncwarp();
        } else if (warp >= LT_W_EPI0) {
            // epilogue: warp (q, h) takes rows q * 32 + h * 16 .. + 15 with the
            // 16x256b shape; thread (qg, qt) holds rows qrow and qrow + 8 and,
            // through the B-row permutation, 16 consecutive output columns of
            // each 64-column half
            const int q = warp & 3, h = (warp - LT_W_EPI0) >> 2;
            const int qg = lane >> 2, qt = lane & 3;
            const int qrow = q * 32 + h * 16 + qg;
            int tok[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int rr = qrow + 8 * u;
                tok[u] = rr < nrows ? checked_token(p.sorted[row0 + rr], T, p.error_word) : -1;
            }
            int sc = 0;
            for (int c = 0; c < nchunks; ++c) {
                while (sc + 1 < S && p.chunk0[sc + 1] <= c) ++sc;
                const int g = g3 + c, slot = g % LT_SLOTS, ab = g % 2;
                bool got = mbar_wait_bounded(accf + 8 * ab, uint32_t(g / 2) & 1u, s_abort, deadline);
                got = got && mbar_wait_bounded(yfull + 8 * slot, uint32_t(g / LT_SLOTS) & 1u,
                                               s_abort, deadline);
                if (__all_sync(0xffffffffu, got) == 0) break;
                tc_fence_after();
                const int kc0 = (c - p.chunk0[sc]) * LT_BN;
                const int ncols = min(LT_BN, p.n[sc] - kc0);
                const uint16_t *bias_row =
                    (BIAS && p.bias[sc] != nullptr) ? p.bias[sc] + int64_t(l_id) * p.n[sc] + kc0
                                                    : nullptr;
                const uint8_t *yt = smem + slot * LT_SLOT + LT_BN * LT_R * 2;
                uint16_t *ybase = p.y + p.col0[sc] + kc0;
                // x B + old y (+ bias), rounded once: output columns
                // 64 hf + 16 qt + 2j + e of the chunk are accumulator columns
                // 64 hf + 8j + 2 qt + e, registers acc[4j + e] (row qrow) and
                // acc[4j + 2 + e] (row qrow + 8)
                auto finish_half = [&](int hf, const uint32_t (&acc)[32]) {
                    const int cb = hf * 64 + qt * 16;
                    if (cb >= ncols) return;
                    uint32_t bw[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                    if (BIAS && bias_row != nullptr) {
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const uint16_t *bq = bias_row + cb + j * 8;
                            uint4 bv;
                            if (p.bias_vec) {
                                bv = __ldg(reinterpret_cast<const uint4 *>(bq));
                            } else {
                                bv.x = uint32_t(bq[0]) | (uint32_t(bq[1]) << 16);
                                bv.y = uint32_t(bq[2]) | (uint32_t(bq[3]) << 16);
                                bv.z = uint32_t(bq[4]) | (uint32_t(bq[5]) << 16);
                                bv.w = uint32_t(bq[6]) | (uint32_t(bq[7]) << 16);
                            }
                            bw[4 * j] = bv.x;
                            bw[4 * j + 1] = bv.y;
                            bw[4 * j + 2] = bv.z;
                            bw[4 * j + 3] = bv.w;
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        if (tok[u] < 0) continue;
                        const uint4 y0 = *reinterpret_cast<const uint4 *>(
                            yt + lt_y_off(qrow + 8 * u, hf * 8 + 2 * qt));
                        const uint4 y1 = *reinterpret_cast<const uint4 *>(
                            yt + lt_y_off(qrow + 8 * u, hf * 8 + 2 * qt + 1));
                        const uint32_t yw[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
                        uint32_t o[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float a0 = __uint_as_float(acc[4 * j + 2 * u]);
                            float a1 = __uint_as_float(acc[4 * j + 2 * u + 1]);
                            a0 += bf16_lo(yw[j]);
                            a1 += bf16_hi(yw[j]);
                            if (BIAS) {
                                a0 += bf16_lo(bw[j]);
                                a1 += bf16_hi(bw[j]);
                            }
                            o[j] = pack_bf16x2(a0, a1);
                        }
                        st_global_v8(ybase + cb + int64_t(tok[u]) * p.y_ld, o);
                    }
                };
                const uint32_t tl = tmem + (uint32_t(q * 32 + h * 16) << 16) +
                                    uint32_t(LT_ACC3 + LT_BN * ab);
                auto release_acc = [&]() {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acce + 8 * ab);
                };
                // the two 64-column halves one after the other (requesting
                // both before finishing either, as the expand kernel does
                // without a bias, measured 4.9 us slower here on the large
                // workload, 223.3 against 218.4 us)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t va[32];
                    tmem_ld16x256b_x8_nowait(tl + uint32_t(hf * 64), va);
                    tmem_wait_ld();
                    if (hf == 1) release_acc();
                    finish_half(hf, va);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty3 + 8 * slot);   // done with the slot's y
            }
        }
        g3 += nchunks;
        ++it;
        tc_fence_before();
        fence_proxy_async_smem();
        const bool stop3 = __syncthreads_or(*s_abort != 0) != 0;
        tc_fence_after();
        if (stop3) break;
    }

    // After an abort, every UMMA issued so far completes (bounded) before
    // TMEM is released.
    if (warp == LT_W_MMA && lane == 0 && *s_abort) {
        umma_commit(drain);
        const long long dd = clock64() + LT_TIMEOUT_CYCLES;
        while (!mbar_try_wait(drain, 0) && clock64() < dd) {
        }
    }
    if (tid == 0 && *s_abort) atomicOr(p.error_word, LT_ERROR_BIT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == LT_W_MMA) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ host

bool linear_tc_fits(const LinearTcLaunch &a)
{
    const int S = a.num_slices;
    if (a.rank != LT_R || S < 1 || S > LT_MAXS) return false;
    if (a.num_tokens < 1 || a.num_tokens >= (1 << 21)) return false;   // 21-bit piece tokens
    if (a.hidden < LT_BK || a.hidden % 8 != 0 || a.x_ld % 8 != 0) return false;
    if (!a.x || !a.buf || !a.y || !a.error_word || !a.sorted || !a.counts || !a.start_loc ||
        !a.active || !a.no_lora)
        return false;
    if ((reinterpret_cast<uintptr_t>(a.x) | reinterpret_cast<uintptr_t>(a.buf)) & 15u) return false;
    // y rows leave with 32-byte stores
    if ((reinterpret_cast<uintptr_t>(a.y) & 31u) || a.y_ld % 16 != 0) return false;
    for (int s = 0; s < S; ++s) {
        if (!a.a[s] || !a.b[s] || a.n[s] <= 0 || a.n[s] % 64 != 0) return false;
        if ((reinterpret_cast<uintptr_t>(a.a[s]) | reinterpret_cast<uintptr_t>(a.b[s])) & 15u)
            return false;
    }
    return linear_tc_smem_bytes(a.max_loras + 1) <= 227 * 1024;
}

int launch_linear_tc(const LinearTcLaunch &a, cudaStream_t stream)
{
    const int S = a.num_slices, T = a.num_tokens;
    static thread_local LinearTcArgs p;       // large (> 3 KB): keep off the stack
    for (int i = 0; i < LT_XMAPS; ++i) {
        if (!encode_tile_map(&p.map_x[i], a.x, uint64_t(T), uint64_t(a.hidden), uint64_t(a.x_ld),
                             LT_BK, 1u << i, CU_TENSOR_MAP_SWIZZLE_128B))
            return int(cudaErrorInvalidValue);
        if (!encode_tile_map_f32(&p.map_buf[i], a.buf, uint64_t(S) * T, uint64_t(LT_R),
                                 uint64_t(LT_R), 32, 1u << i, CU_TENSOR_MAP_SWIZZLE_128B))
            return int(cudaErrorInvalidValue);
    }
    bool bias = false, bias_vec = true;
    int chunks = 0, col = 0;
    for (int s = 0; s < LT_MAXS; ++s) {
        if (s >= S) {
            p.map_a[s] = p.map_a[0];
            p.map_b[s] = p.map_b[0];
            p.bias[s] = nullptr;
            p.n[s] = p.col0[s] = 0;
            continue;
        }
        if (!encode_tile_map(&p.map_a[s], a.a[s], uint64_t(a.max_loras) * LT_R,
                             uint64_t(a.hidden), uint64_t(a.hidden), LT_BK, LT_R,
                             CU_TENSOR_MAP_SWIZZLE_128B))
            return int(cudaErrorInvalidValue);
        if (!encode_perm_rows_map(&p.map_b[s], a.b[s], uint64_t(a.max_loras) * uint64_t(a.n[s]),
                                  uint32_t(LT_R), 64u, 2u, CU_TENSOR_MAP_SWIZZLE_128B))
            return int(cudaErrorInvalidValue);
        p.bias[s] = a.bias[s];
        if (a.bias[s] != nullptr) {
            bias = true;
            if (reinterpret_cast<uintptr_t>(a.bias[s]) & 15u) bias_vec = false;
        }
        p.n[s] = a.n[s];
        p.col0[s] = col;
        p.chunk0[s] = chunks;
        col += a.n[s];
        chunks += (a.n[s] + LT_BN - 1) / LT_BN;
    }
    p.chunk0[S] = chunks;
    for (int s = S + 1; s <= LT_MAXS; ++s) p.chunk0[s] = chunks;
    p.num_slices = S;
    p.hidden = a.hidden;
    p.num_tokens = T;
    p.scale = a.scale;
    p.buf = a.buf;
    p.y = a.y;
    p.y_ld = a.y_ld;
    p.bias_vec = bias_vec ? 1 : 0;
    p.sorted = a.sorted;
    p.counts = a.counts;
    p.start_loc = a.start_loc;
    p.active = a.active;
    p.no_lora = a.no_lora;
    p.error_word = a.error_word;
    p.nbins = a.max_loras + 1;

    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return int(e);
    if (dev < 64 && configured[dev] == 0) {
        e = cudaFuncSetAttribute(linear_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 227 * 1024);
        if (e != cudaSuccess) return int(e);
        e = cudaFuncSetAttribute(linear_tc_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return int(e);
        configured[dev] = 1;
    }
    return int(launch_kernel(bias ? linear_tc_kernel<true> : linear_tc_kernel<false>,
                             dim3(device_sm_count()), dim3(LT_THREADS),
                             linear_tc_smem_bytes(a.max_loras + 1), stream, p));
}

}  // namespace lora
