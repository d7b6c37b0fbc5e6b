// lora_expand_tc.cu -- tensor-core (tcgen05 / TMEM) path of lora_expand
// (page "vllm.lora.punica_wrapper.punica_gpu", PunicaWrapperGPU.add_expand;
// bias step of page "vllm.lora.punica_wrapper.punica_tpu",
// PunicaWrapperTPU._apply_bias):
//   y[t, off_s + j] (+)= x[s][t, :] @ B[s][id(t)][j, :] + bias[s][id(t)][j]
//
// Work items are (128-token tile of one LoRA segment, 64-column chunk of one
// slice), numbered chunk-fastest; one persistent CTA per SM takes a
// contiguous, balanced range of them, so it walks the chunks of one tile
// with the tile's x rows (the MMA's A operand) resident in shared memory.
// Chunks stream through a ring of DEPTH slots, each holding the chunk's B
// tile (swizzled K-major, as UMMA reads it) and its old y rows.
//
// Thirteen warps, one job each:
//   warp 0       owns TMEM (two 64-column fp32 accumulators); lane 0 issues
//                tcgen05.mma (M = 128 tokens, N = 64 columns, K = 16 steps
//                over the rank) and commits each chunk's accumulator and
//                the release of its slot's B.
//   warps 1..4   loaders.  They fill slots with coalesced 16-byte cp.async
//                (four whole 128-byte lines per instruction): the chunk's
//                128 old y rows and its B tile.  Up to DEPTH - 1 chunks are
//                in flight; as each one lands, the loaders fence it for the
//                tensor core and signal the slot's mbarrier.
//   warps 5..12  epilogue.  Warp (q, h) = (warp % 4, (warp - 5) / 4) owns
//                the tile rows of TMEM lane quarter q and column half h.
//                Per chunk it reads its accumulators with tcgen05.ld (one
//                token row per thread), adds bias and old y in fp32, rounds
//                once to bf16 into the slot and writes its rows back with
//                coalesced 16-byte stores (8 rows x 64 bytes per
//                instruction), then releases the slot.  When the next chunk
//                opens a new tile or slice, it rounds that item's x rows to
//                bf16 into the A operand right after reading the current
//                accumulator.
// Splitting loading from the epilogue keeps each warp on one latency chain:
// a version in which every warp did both ran at half the rate.
//
// The ring is fed by the load/store units, not TMA: measured on this GPU,
// a TMA box costs about 1000 cycles of latency per issuing thread and the
// engine tops out near 50 bytes per clock per SM, and the old y rows of a
// tile cut into several boxes wherever its token runs break.
//
// Every mbarrier wait is bounded (about one second); on expiry the kernel
// sets bit 30 of the metadata error word, drains its copies and MMAs, frees
// TMEM and returns.
#include "lora_common.cuh"
#include "lora_umma.cuh"

namespace lora {

constexpr int TC_BM = 128;                    // tokens per tile (UMMA M, TMEM lanes)
constexpr int TC_BN = 64;                     // columns per chunk (UMMA N)
constexpr int TC_LOADERS = 4;
constexpr int TC_EPI = 8;
constexpr int TC_EPI0 = 1 + TC_LOADERS;       // first epilogue warp
constexpr int TC_THREADS = 32 * (TC_EPI0 + TC_EPI);
constexpr int TC_LT = 32 * TC_LOADERS;        // loader threads
constexpr long long TC_TIMEOUT_CYCLES = 2000000000ll;
constexpr int TC_ERROR_BIT = 1 << 30;

struct TcArgs {
    const void *x;                            // [S, T, r]: fp32, or bf16 when x_bf16
    int32_t x_bf16;
    const uint16_t *b[LORA_MAX_SLICES];       // [L, n_s, r]
    const uint16_t *bias[LORA_MAX_SLICES];    // [L, n_s] or null
    int32_t n[LORA_MAX_SLICES];
    int32_t col0[LORA_MAX_SLICES];
    int32_t chunk0[LORA_MAX_SLICES + 1];      // first 64-column chunk of each slice
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
    static constexpr int A_BYTES = TC_BM * RP * 2;
    static constexpr int B_BYTES = TC_BN * RP * 2;
    static constexpr int Y_BYTES = TC_BM * TC_BN * 2;      // 128 rows x 128 bytes
    static constexpr int SLOT_BYTES = B_BYTES + Y_BYTES;   // a multiple of 1024
    static constexpr int DEPTH = (KT >= 8) ? 5 : 8;
    static constexpr int RING_OFF = A_BYTES;
    static constexpr int BAR_OFF = RING_OFF + DEPTH * SLOT_BYTES;
    static constexpr int MISC_OFF = BAR_OFF + (2 * DEPTH + 6) * 8;
    static constexpr int TAB_OFF = MISC_OFF + 16;
    static constexpr int Y_PER_T = TC_BM * 8 / TC_LT;      // y pieces per loader thread (8)
    static constexpr int B_PER_T = (TC_BN * CPR + TC_LT - 1) / TC_LT;
    static_assert(SLOT_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "1024-byte aligned operands");
};

template <int KT>
inline size_t tc_smem_bytes(int nbins)
{
    return size_t(TcCfg<KT>::TAB_OFF) + seg_tab_bytes(nbins) + 1024;     // + alignment slack
}

// Byte offset of 16-byte piece `c` of row `r` in a K-major operand tile of
// `rows` rows and rp bf16 columns, in the swizzled layout UMMA reads (32-,
// 64- or 128-byte swizzle; rank 128 = two 64-column blocks).
__device__ __forceinline__ uint32_t tc_kmajor_off(int rp, int rows, int r, int c)
{
    switch (rp) {
    case 16: return uint32_t(r * 32 + ((c ^ ((r >> 2) & 1)) << 4));
    case 32: return uint32_t(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
    case 64: return uint32_t(r * 128 + ((c ^ (r & 7)) << 4));
    default: return uint32_t((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    }
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
};

template <int KT>
__global__ void __launch_bounds__(TC_THREADS, 1) expand_tc_kernel(const __grid_constant__ TcArgs p)
{
    using C = TcCfg<KT>;
    constexpr int RP = C::RP, CPR = C::CPR, DEPTH = C::DEPTH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t base = smem_addr(smem);
    const uint32_t bar_full = base + C::BAR_OFF;           // [DEPTH]: 4 loader warps
    const uint32_t bar_empty = bar_full + 8 * DEPTH;       // [DEPTH]: MMA + 8 epilogue warps
    const uint32_t bar_accf = bar_empty + 8 * DEPTH;       // [2]: MMA commit
    const uint32_t bar_acce = bar_accf + 16;               // [2]: 8 epilogue warps
    const uint32_t bar_x = bar_acce + 16;                  // A operand ready: 8 epilogue warps
    const uint32_t bar_drain = bar_x + 8;
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
            mbar_init(bar_full + 8 * i, TC_LOADERS);
            mbar_init(bar_empty + 8 * i, 1 + TC_EPI);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_accf + 8 * i, 1);
            mbar_init(bar_acce + 8 * i, TC_EPI);
        }
        mbar_init(bar_x, TC_EPI);
        mbar_init(bar_drain, 1);
        mbar_fence_init();
        *s_abort = 0;
    }
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

    if (warp == 0) tmem_alloc(smem_addr(s_tmem), 2 * TC_BN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const long long deadline = clock64() + TC_TIMEOUT_CYCLES;
    const int R = p.rank, T = p.num_tokens;
    const uint32_t a_tile = base;

    if (warp == 0) {
        // ------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_bf16(TC_BM, TC_BN);
            int g = 0, items = 0;
            bool ok = true;
            TcCursor k;
            k.start(p, w_begin, nchunks);
            for (int64_t w = w_begin; w < w_end; ++w, ++g, k.next(p, nchunks)) {
                if (k.first) {
                    if (!mbar_wait_bounded(bar_x, uint32_t(items) & 1u, s_abort, deadline)) {
                        ok = false;
                        break;
                    }
                    ++items;
                }
                const int slot = g % DEPTH, ab = g & 1;
                if (!mbar_wait_bounded(bar_full + 8 * slot, uint32_t(g / DEPTH) & 1u, s_abort,
                                       deadline) ||
                    !mbar_wait_bounded(bar_acce + 8 * ab, (uint32_t(g >> 1) & 1u) ^ 1u, s_abort,
                                       deadline)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t bt = base + C::RING_OFF + slot * C::SLOT_BYTES;
#pragma unroll
                for (int kk = 0; kk < KT; ++kk)
                    umma_bf16(tmem + ab * TC_BN, tc_kmajor_desc(RP, TC_BM, a_tile, kk),
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
    } else if (warp < TC_EPI0) {
        // ------------------------------------------------------ loaders
        const int lt = tid - 32;                           // 0 .. TC_LT - 1
        const uint16_t *const ydummy = p.y;
        int cur_tile = -1, l_id = 0;
        int ltok[C::Y_PER_T];                              // rows i * 16 + lt / 8
        int issued = 0, signalled = 0;
        bool ok = true;
        // Hands the oldest chunk in flight to the MMA and the epilogue.
        auto signal_oldest = [&]() {
            fence_proxy_async_smem();                      // B is read by the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_full + 8 * (signalled % DEPTH));
            ++signalled;
        };
        TcCursor k;
        k.start(p, w_begin, nchunks);
        for (int64_t w = w_begin; w < w_end; ++w, k.next(p, nchunks)) {
            const int g = issued, slot = g % DEPTH;
            const bool got = mbar_wait_bounded(bar_empty + 8 * slot,
                                               (uint32_t(g / DEPTH) & 1u) ^ 1u, s_abort, deadline);
            if (__all_sync(0xffffffffu, got) == 0) {
                ok = false;
                break;
            }
            if (k.tile != cur_tile) {
                cur_tile = k.tile;
                const int seg = find_segment(tab.tile, p.nbins, cur_tile);
                l_id = tab.id[seg];
                const int row0 = tab.start[seg] + (cur_tile - tab.tile[seg]) * TC_BM;
                const int nrows = min(TC_BM, tab.start[seg] + tab.count[seg] - row0);
#pragma unroll
                for (int i = 0; i < C::Y_PER_T; ++i) {
                    const int r = i * (TC_LT / 8) + lt / 8;
                    ltok[i] = (r < nrows) ? checked_token(p.sorted[row0 + r], T, p.error_word)
                                          : -1;
                }
            }
            const int c0 = k.c0(p), ncols = min(TC_BN, p.n[k.s] - c0);
            const uint32_t st = base + C::RING_OFF + slot * C::SLOT_BYTES;
            if (p.add_inputs) {
                const int piece = lt % 8;
                const bool cin = piece * 8 < ncols;
                const uint16_t *ycol = p.y + p.col0[k.s] + c0 + piece * 8;
#pragma unroll
                for (int i = 0; i < C::Y_PER_T; ++i) {
                    const int r = i * (TC_LT / 8) + lt / 8;
                    const bool ld = cin && ltok[i] >= 0;
                    cp_async16(st + C::B_BYTES + r * 128 + ((piece ^ (r & 7)) << 4),
                               ld ? ycol + int64_t(ltok[i]) * p.y_ld : ydummy, ld);
                }
            }
            const int n_s = p.n[k.s];
            const uint16_t *brows = p.b[k.s] + (int64_t(l_id) * n_s + c0) * R;
#pragma unroll
            for (int i = 0; i < C::B_PER_T; ++i) {
                const int j = i * TC_LT + lt;
                if (TC_BN * CPR % TC_LT != 0 && j >= TC_BN * CPR) break;
                const int r = j / CPR, c = j % CPR;
                const bool ld = r < ncols && c * 8 < R;
                cp_async16(st + tc_kmajor_off(RP, TC_BN, r, c),
                           ld ? brows + int64_t(r) * R + c * 8 : p.b[k.s], ld);
            }
            cp_async_commit();
            ++issued;
            if (issued - signalled == DEPTH - 1) {         // the oldest must land now
                cp_async_wait<DEPTH - 2>();
                signal_oldest();
            }
        }
        cp_async_wait<0>();
        if (ok)
            while (signalled < issued) signal_oldest();
    } else {
        // ------------------------------------------------------ epilogue
        const int ew = warp - TC_EPI0, q = warp & 3, h = ew >> 2;
        const int my_row = q * 32 + lane;                  // TMEM lane
        int ct = -1, c_id = 0, ctok = -1;
        auto tile_rows = [&](int tile) {
            if (tile != ct) {
                ct = tile;
                const int seg = find_segment(tab.tile, p.nbins, ct);
                c_id = tab.id[seg];
                const int row0 = tab.start[seg] + (ct - tab.tile[seg]) * TC_BM;
                const int nrows = min(TC_BM, tab.start[seg] + tab.count[seg] - row0);
                ctok = (my_row < nrows) ? checked_token(p.sorted[row0 + my_row], T, p.error_word)
                                        : -1;
            }
        };
        // this warp's rows of x (slice s), rounded to bf16, into the A operand
        auto convert_x = [&](int s) {
            wait_once();                                   // x is the shrink output
            const int64_t xrow = (int64_t(s) * T + (ctok >= 0 ? ctok : 0)) * R;
#pragma unroll
            for (int c = h * (CPR / 2); c < (h + 1) * (CPR / 2); ++c) {
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
                *reinterpret_cast<uint4 *>(smem + tc_kmajor_off(RP, TC_BM, my_row, c)) = v;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_x);
        };

        TcCursor k;
        k.start(p, w_begin, nchunks);
        tile_rows(k.tile);
        convert_x(k.s);

        int g = 0;
#pragma unroll 1
        for (int64_t w = w_begin; w < w_end; ++w, ++g) {
            tile_rows(k.tile);
            const int kc0 = k.c0(p), kncols = min(TC_BN, p.n[k.s] - kc0), ks = k.s;
            // bias of this warp's 32 columns, fetched before the waits
            uint4 bpre[4];
            const uint16_t *bias_row = p.bias[ks] ? p.bias[ks] + int64_t(c_id) * p.n[ks] + kc0
                                                  : nullptr;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int piece = 4 * h + j;
                bpre[j] = make_uint4(0u, 0u, 0u, 0u);
                if (bias_row != nullptr && p.bias_vec && piece * 8 < kncols)
                    bpre[j] = __ldg(reinterpret_cast<const uint4 *>(bias_row + piece * 8));
            }
            const int ab = g & 1, slot = g % DEPTH;
            bool got = mbar_wait_bounded(bar_accf + 8 * ab, uint32_t(g >> 1) & 1u, s_abort,
                                         deadline);
            got = got && mbar_wait_bounded(bar_full + 8 * slot, uint32_t(g / DEPTH) & 1u, s_abort,
                                           deadline);
            if (__all_sync(0xffffffffu, got) == 0) break;
            tc_fence_after();
            uint32_t va[32];
            tmem_ld32_nowait(tmem + (uint32_t(q * 32) << 16) + uint32_t(ab * TC_BN + h * 32), va);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_acce + 8 * ab);
            const int tok_g = ctok;
            // the next chunk opens a new tile or slice: its A operand now (the
            // MMA of chunk g is done; that of chunk g + 1 waits for it)
            k.next(p, nchunks);
            if (w + 1 < w_end && k.first) {
                tile_rows(k.tile);
                convert_x(k.s);
            }
            // + bias + old y, rounded once, back into the slot (own row)
            uint8_t *yt = smem + C::RING_OFF + slot * C::SLOT_BYTES + C::B_BYTES;
            if (tok_g >= 0) {
                uint4 yv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int piece = 4 * h + j;
                    yv[j] = make_uint4(0u, 0u, 0u, 0u);
                    if (p.add_inputs)
                        yv[j] = *reinterpret_cast<const uint4 *>(
                            yt + my_row * 128 + ((piece ^ (my_row & 7)) << 4));
                }
                if (bias_row != nullptr && !p.bias_vec) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int piece = 4 * h + j;
                        if (piece * 8 < kncols) {
                            const uint16_t *bq = bias_row + piece * 8;
                            bpre[j].x = uint32_t(bq[0]) | (uint32_t(bq[1]) << 16);
                            bpre[j].y = uint32_t(bq[2]) | (uint32_t(bq[3]) << 16);
                            bpre[j].z = uint32_t(bq[4]) | (uint32_t(bq[5]) << 16);
                            bpre[j].w = uint32_t(bq[6]) | (uint32_t(bq[7]) << 16);
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int piece = 4 * h + j;
                    const uint32_t yw[4] = {yv[j].x, yv[j].y, yv[j].z, yv[j].w};
                    const uint32_t bw[4] = {bpre[j].x, bpre[j].y, bpre[j].z, bpre[j].w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float a0 = __uint_as_float(va[j * 8 + 2 * e]) + bf16_lo(bw[e]) +
                                         bf16_lo(yw[e]);
                        const float a1 = __uint_as_float(va[j * 8 + 2 * e + 1]) + bf16_hi(bw[e]) +
                                         bf16_hi(yw[e]);
                        o[e] = pack_bf16x2(a0, a1);
                    }
                    // columns past the slice are never stored
                    *reinterpret_cast<uint4 *>(yt + my_row * 128 + ((piece ^ (my_row & 7)) << 4)) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            __syncwarp();
            // this warp's rows out: 8 rows x 64 bytes per store instruction
            {
                const int piece = 4 * h + (lane & 3);
                const bool cin = piece * 8 < kncols;
                uint16_t *ycol = p.y + p.col0[ks] + kc0 + piece * 8;
                int tok[4];
                uint4 v[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int rl = i * 8 + (lane >> 2);
                    const int r = q * 32 + rl;
                    tok[i] = __shfl_sync(0xffffffffu, tok_g, rl);
                    v[i] = *reinterpret_cast<const uint4 *>(yt + r * 128 + ((piece ^ (r & 7)) << 4));
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (cin && tok[i] >= 0)
                        *reinterpret_cast<uint4 *>(ycol + int64_t(tok[i]) * p.y_ld) = v[i];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * slot);   // this warp is done with the slot
        }
    }

    wait_once();
    if (tid == 0 && *s_abort) atomicOr(p.error_word, TC_ERROR_BIT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 2 * TC_BN);
}

template <int KT>
static int launch_tc_kt(const TcArgs &p, cudaStream_t stream)
{
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return int(e);
    const size_t smem = tc_smem_bytes<KT>(p.nbins);
    if (smem > 227 * 1024) return 0;
    if (dev < 64 && configured[dev] == 0) {
        e = cudaFuncSetAttribute(expand_tc_kernel<KT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 227 * 1024);
        if (e != cudaSuccess) return int(e);
        configured[dev] = 1;
    }
    e = launch_kernel(expand_tc_kernel<KT>, dim3(device_sm_count()), dim3(TC_THREADS), smem,
                      stream, p);
    return e == cudaSuccess ? 1 : int(e);
}

// Launches the tensor-core expand: returns 1 if launched, 0 if the call does
// not fit it (the caller then runs the mma.sync kernel), or a cudaError_t.
int launch_expand_tc(const ExpandLaunch &a, cudaStream_t stream)
{
    if (!a.vec || a.error_word == nullptr) return 0;
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
