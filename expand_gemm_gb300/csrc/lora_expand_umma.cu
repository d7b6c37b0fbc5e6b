// lora_expand_umma.cu -- tensor-core (tcgen05 / TMEM) path of lora_expand
// (page "vllm.lora.punica_wrapper.punica_gpu", PunicaWrapperGPU.add_expand;
// bias step of page "vllm.lora.punica_wrapper.punica_tpu",
// PunicaWrapperTPU._apply_bias):
//   y[t, off_s + j] (+)= x[s][t, :] @ B[s][id(t)][j, :] + bias[s][id(t)][j]
//
// Work items are (token tile of 128 tokens of one LoRA segment, 64-column
// chunk of one slice), numbered chunk-fastest; one persistent CTA per SM
// takes a contiguous, balanced range of them.  Ten warps, specialised:
//   warp 0      producer, all TMA: per chunk one 2-D box of B[s][id] (two
//               for rank 128) in the swizzled K-major layout UMMA reads; the
//               tile's old y rows as 2-D boxes over runs of consecutive
//               tokens (power-of-two heights, 128-byte swizzle; the runs are
//               found once per tile from its token list staged in shared
//               memory); the bias chunk as one 1-D bulk copy.
//   warp 1      owns TMEM (two 64-column fp32 accumulators); lane 0 issues
//               tcgen05.mma (M = 128 tokens, N = 64 columns, K = 16 steps
//               over the rank) and commits.
//   warps 2..9  epilogue, one token row per thread (its TMEM lane), two
//               warps per lane quarter splitting the columns: at each new
//               tile the fp32 x rows are rounded to bf16 into the A operand;
//               per chunk the accumulators are read with tcgen05.ld, bias
//               and old y added in fp32, rounded once to bf16 and written
//               with 16-byte stores straight to the thread's own y row.
// The accumulators are double-buffered so the MMA of chunk i + 1 runs while
// the epilogue drains chunk i.  B, old y and bias stream through a ring of
// up to six stages; a stage is refilled once the MMA has read its B and
// every epilogue warp its y and bias, so the loads run several chunks ahead
// of the epilogue.  The epilogue warps never wait for one another.
//
// Used when y rows, offsets and slice widths are 16-byte aligned (the same
// condition as the vector path of the mma.sync kernel).  Every mbarrier
// wait is bounded; on expiry the kernel sets bit 30 of the metadata error
// word, drains its copies and MMAs, frees TMEM and returns.
#include "lora_common.cuh"
#include "lora_umma.cuh"

namespace lora {

constexpr int XU_BM = 128;              // tokens per tile (UMMA M, TMEM lanes)
constexpr int XU_BN = 64;               // columns per chunk (UMMA N; one 128-byte y row)
constexpr int XU_EPI_WARPS = 8;         // two per TMEM lane quarter (column halves)
constexpr int XU_THREADS = 64 + 32 * XU_EPI_WARPS;
constexpr int XU_MAX_STAGES = 6;
constexpr int XU_SMEM_BUDGET = 224 * 1024;
constexpr int XU_YMAPS = 8;             // y box heights 1, 2, 4, ..., 128
constexpr long long XU_TIMEOUT_CYCLES = 2000000000ll;
constexpr int XU_ERROR_BIT = 1 << 30;

struct ExpandUmmaArgs {
    CUtensorMap map_b[LORA_MAX_SLICES];      // B[s]: [L * n_s rows, r cols], box {min(rp, 64), 128}
    CUtensorMap map_y[XU_YMAPS];             // y: [T rows, y_ld cols], box {64, 2^i}, 128-byte swizzle
    const float *x;
    uint16_t *y;
    int64_t y_ld;
    const uint16_t *bias[LORA_MAX_SLICES];
    int32_t n[LORA_MAX_SLICES];
    int32_t col0[LORA_MAX_SLICES];
    int32_t chunk0[LORA_MAX_SLICES + 1];
    int32_t num_slices;
    int32_t rank;
    int32_t rp;                              // padded rank: 16, 32, 64 or 128
    int32_t num_tokens;
    int32_t add_inputs;
    int32_t bias_vec;
    int32_t stages;
    const int32_t *sorted;
    const int32_t *counts;
    const int32_t *start_loc;
    const int32_t *active;
    const int32_t *no_lora;
    int32_t *error_word;
    int32_t nbins;
};

struct XuLayout {
    int a_bytes, b_bytes, y_off, bias_off, stage_bytes, ring_off, bar_off, misc_off, ppc_off,
        ptok_off, tab_off, total;
};

// Stage: B tile | old y tile (128 rows x 128 bytes, 128-byte swizzle) |
// bias chunk.
__host__ __device__ inline XuLayout xu_layout(int rp, int stages, int nbins)
{
    XuLayout l;
    l.a_bytes = XU_BM * rp * 2;
    l.b_bytes = XU_BN * rp * 2;
    l.y_off = l.b_bytes;
    l.bias_off = l.y_off + XU_BM * 128;
    l.stage_bytes = ((l.bias_off + XU_BN * 2) + 1023) & ~1023;
    l.ring_off = l.a_bytes;
    l.bar_off = l.ring_off + stages * l.stage_bytes;
    l.misc_off = l.bar_off + (2 * XU_MAX_STAGES + 6) * 8;
    l.ppc_off = l.misc_off + 16;                         // producer pieces [128]
    l.ptok_off = l.ppc_off + XU_BM * 4;                  // producer's token list [128]
    l.tab_off = l.ptok_off + XU_BM * 4;
    l.total = l.tab_off + int(seg_tab_bytes(nbins)) + 1024;
    return l;
}

// Byte offset of 16-byte chunk `c` of row `r` in a K-major operand tile of
// `rows` rows and rp bf16 columns, in the swizzled layout TMA writes and
// UMMA reads (32-, 64- or 128-byte swizzle; rank 128 = two 64-column blocks).
__device__ __forceinline__ uint32_t kmajor_off(int rp, int rows, int r, int c)
{
    switch (rp) {
    case 16: return uint32_t(r * 32 + ((c ^ ((r >> 2) & 1)) << 4));
    case 32: return uint32_t(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
    case 64: return uint32_t(r * 128 + ((c ^ (r & 7)) << 4));
    default: return uint32_t((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    }
}

// Descriptor of K step kk (16 columns) of such a tile starting at `tile`.
__device__ __forceinline__ uint64_t kmajor_desc(int rp, int rows, uint32_t tile, int kk)
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

// Cuts the increasing token list tk[0..n) into pieces of consecutive
// tokens whose heights are powers of two aligned to their row; each piece
// is (row | log2 height << 8 | first token << 11).  Returns the count.
__device__ __forceinline__ int token_pieces(const int32_t *tk, int n, uint32_t *pieces)
{
    int np = 0, j = 0;
    while (j < n) {
        int lg = 7;
        while ((1 << lg) > n - j || (j & ((1 << lg) - 1)) != 0 ||
               tk[j + (1 << lg) - 1] - tk[j] != (1 << lg) - 1)
            --lg;
        pieces[np++] = uint32_t(j) | (uint32_t(lg) << 8) | (uint32_t(tk[j]) << 11);
        j += 1 << lg;
    }
    return np;
}

__global__ void __launch_bounds__(XU_THREADS, 1) expand_umma_kernel(const __grid_constant__ ExpandUmmaArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int RP = p.rp, STAGES = p.stages, S = p.num_slices, R = p.rank;
    const XuLayout L = xu_layout(RP, STAGES, p.nbins);
    const uint32_t base = smem_addr(smem);
    const uint32_t bar_full = base + L.bar_off;                   // [STAGES] B + y + bias (TMA)
    const uint32_t bar_empty = bar_full + 8 * XU_MAX_STAGES;      // [STAGES] MMA + epilogue warps
    const uint32_t bar_acc_full = bar_empty + 8 * XU_MAX_STAGES;  // [2]
    const uint32_t bar_acc_empty = bar_acc_full + 16;             // [2]
    const uint32_t bar_x_ready = bar_acc_empty + 16;
    const uint32_t bar_drain = bar_x_ready + 8;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + L.misc_off + 4);
    uint32_t *s_ppieces = reinterpret_cast<uint32_t *>(smem + L.ppc_off);
    int32_t *s_ptok = reinterpret_cast<int32_t *>(smem + L.ptok_off);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    pdl_wait();
    pdl_launch_dependents();

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, 1 + XU_EPI_WARPS);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_acc_full + 8 * i, 1);
            mbar_init(bar_acc_empty + 8 * i, XU_EPI_WARPS);
        }
        mbar_init(bar_x_ready, XU_EPI_WARPS);
        mbar_init(bar_drain, 1);
        mbar_fence_init();
        *s_abort = 0;
        for (int s = 0; s < S; ++s) tma_prefetch_map(&p.map_b[s]);
        for (int i = 0; i < XU_YMAPS; ++i) tma_prefetch_map(&p.map_y[i]);
    }
    const SegTab tab = seg_tab(reinterpret_cast<int *>(smem + L.tab_off), p.nbins);
    const int total_tiles = load_segments(p.no_lora, p.active, p.counts, p.start_loc,
                                          p.nbins, XU_BM, tab);
    if (total_tiles == 0) return;
    const int nchunks = p.chunk0[S];
    const int64_t total = int64_t(total_tiles) * nchunks;
    const int64_t w_begin = int64_t(blockIdx.x) * total / gridDim.x;
    const int64_t w_end = int64_t(blockIdx.x + 1) * total / gridDim.x;
    if (w_begin >= w_end) return;

    if (warp == 1) tmem_alloc(smem_addr(s_tmem), 2 * XU_BN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const long long deadline = clock64() + XU_TIMEOUT_CYCLES;
    const uint32_t a_tile = base;                                  // x tile at offset 0
    const int b_boxes = (RP > 64) ? 2 : 1;

    // Row items: token tile `tile`, slice s, chunks [cb, ce) of that slice.
    auto row_item = [&](int64_t w, int &tile, int &s, int &cb, int &ce) {
        tile = int(w / nchunks);
        cb = int(w - int64_t(tile) * nchunks);
        s = 0;
        while (s + 1 < S && p.chunk0[s + 1] <= cb) ++s;
        ce = int(min(int64_t(p.chunk0[s + 1]), int64_t(cb) + (w_end - w)));
    };
    auto tile_rows = [&](int tile, int &id, int &row0, int &nrows) {
        const int seg = find_segment(tab.tile, p.nbins, tile);
        id = tab.id[seg];
        row0 = tab.start[seg] + (tile - tab.tile[seg]) * XU_BM;
        nrows = min(XU_BM, tab.start[seg] + tab.count[seg] - row0);
    };

    if (warp == 0) {
        // ------------------------------------------ producer: TMA for B, y, bias
        int g = 0;
        bool ok = true;
        for (int64_t w = w_begin; ok && w < w_end;) {
            int tile, s, cb, ce, id, row0, nrows;
            row_item(w, tile, s, cb, ce);
            tile_rows(tile, id, row0, nrows);
            int np = 0;
            if (p.add_inputs) {
                // the tile's tokens in one coalesced read, then the runs
                for (int i = lane; i < nrows; i += 32) s_ptok[i] = p.sorted[row0 + i];
                __syncwarp();
                if (lane == 0) np = token_pieces(s_ptok, nrows, s_ppieces);
                np = __shfl_sync(0xffffffffu, np, 0);
                __syncwarp();
            }
            const int n_s = p.n[s];
            const uint16_t *bias_row = p.bias[s] ? p.bias[s] + int64_t(id) * n_s : nullptr;
            for (int c = cb; c < ce; ++c, ++g) {
                const int stage = g % STAGES;
                const uint32_t ph = uint32_t(g / STAGES) & 1u;
                bool got = mbar_wait_bounded(bar_empty + 8 * stage, ph ^ 1u, s_abort, deadline);
                if (__all_sync(0xffffffffu, got) == 0) {
                    ok = false;
                    break;
                }
                const uint32_t st = base + L.ring_off + stage * L.stage_bytes;
                const uint32_t full = bar_full + 8 * stage;
                const int c0 = (c - p.chunk0[s]) * XU_BN;
                const int ncols = min(XU_BN, n_s - c0);
                const bool with_bias = bias_row != nullptr && p.bias_vec;
                if (lane == 0) {
                    const uint32_t tx = uint32_t(L.b_bytes) +
                                        (p.add_inputs ? uint32_t(nrows) * 128u : 0u) +
                                        (with_bias ? uint32_t(ncols) * 2u : 0u);
                    mbar_arrive_expect_tx(full, tx);
                }
                __syncwarp();
                if (p.add_inputs) {
                    const int col = p.col0[s] + c0;
                    for (int i = lane; i < np; i += 32) {
                        const uint32_t pc = s_ppieces[i];
                        const int r = int(pc & 0xFFu), lg = int((pc >> 8) & 7u), t0 = int(pc >> 11);
                        tma_load_2d(st + L.y_off + r * 128, &p.map_y[lg], col, t0, full);
                    }
                }
                if (lane == 0) {
                    const int brow = id * n_s + c0;
                    for (int k = 0; k < b_boxes; ++k)
                        tma_load_2d(st + k * XU_BN * 128, &p.map_b[s], k * 64, brow, full);
                    if (with_bias) bulk_load_1d(st + L.bias_off, bias_row + c0, uint32_t(ncols) * 2u, full);
                }
            }
            w += ce - cb;
        }
        // every issued fill must land before the CTA may exit
        if (lane == 0) {
            const long long dd = clock64() + XU_TIMEOUT_CYCLES;
            for (int i = max(0, g - STAGES); i < g; ++i)
                while (!mbar_try_wait(bar_full + 8 * (i % STAGES), uint32_t(i / STAGES) & 1u) &&
                       clock64() < dd) {
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_bf16(XU_BM, XU_BN);
            int g = 0, items = 0;
            bool ok = true;
            for (int64_t w = w_begin; ok && w < w_end; ++items) {
                int tile, s, cb, ce;
                row_item(w, tile, s, cb, ce);
                if (!mbar_wait_bounded(bar_x_ready, uint32_t(items) & 1u, s_abort, deadline)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int c = cb; c < ce; ++c, ++g) {
                    const int stage = g % STAGES, ab = g & 1;
                    if (!mbar_wait_bounded(bar_full + 8 * stage, uint32_t(g / STAGES) & 1u, s_abort, deadline) ||
                        !mbar_wait_bounded(bar_acc_empty + 8 * ab, (uint32_t(g >> 1) & 1u) ^ 1u, s_abort, deadline)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sb = base + L.ring_off + stage * L.stage_bytes;
                    for (int kk = 0; kk < RP / 16; ++kk)
                        umma_bf16(tmem + ab * XU_BN, kmajor_desc(RP, XU_BM, a_tile, kk),
                                  kmajor_desc(RP, XU_BN, sb, kk), idesc, kk != 0);
                    umma_commit(bar_empty + 8 * stage);
                    umma_commit(bar_acc_full + 8 * ab);
                }
                w += ce - cb;
            }
            if (!ok || *s_abort) {
                umma_commit(bar_drain);
                const long long dd = clock64() + XU_TIMEOUT_CYCLES;
                while (!mbar_try_wait(bar_drain, 0) && clock64() < dd) {
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------ epilogue (8 warps)
        // Warp e = warp - 2: TMEM lane quarter q = warp % 4 (one token row per
        // thread), column half hf = e / 4 (32 of the chunk's 64 columns).
        const int e = warp - 2;
        const int q = warp & 3;
        const int hf = e >> 2;
        const int row = q * 32 + lane;
        int g = 0;
        bool ok = true;
        for (int64_t w = w_begin; ok && w < w_end;) {
            int tile, s, cb, ce, id, row0, nrows;
            row_item(w, tile, s, cb, ce);
            tile_rows(tile, id, row0, nrows);
            const int tok = (row < nrows) ? p.sorted[row0 + row] : -1;
            // x row -> bf16 A operand row; each half converts half of the
            // 16-byte pieces.  A is free: this warp has seen the accumulator
            // of the previous item's last chunk, committed after its MMAs.
            {
                const float *xr = p.x + (int64_t(s) * p.num_tokens + (tok >= 0 ? tok : 0)) * R;
                const int nch = RP / 8;
                for (int c = hf * (nch / 2); c < (hf + 1) * (nch / 2) + (nch & 1) * hf; ++c) {
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (tok >= 0 && c * 8 < R) {
                        const float4 u = reinterpret_cast<const float4 *>(xr + c * 8)[0];
                        const float4 t = reinterpret_cast<const float4 *>(xr + c * 8)[1];
                        v.x = pack_bf16x2(u.x, u.y);
                        v.y = pack_bf16x2(u.z, u.w);
                        v.z = pack_bf16x2(t.x, t.y);
                        v.w = pack_bf16x2(t.z, t.w);
                    }
                    *reinterpret_cast<uint4 *>(smem + kmajor_off(RP, XU_BM, row, c)) = v;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_x_ready);
            }
            const int n_s = p.n[s];
            const uint16_t *bias_row = p.bias[s] ? p.bias[s] + int64_t(id) * n_s : nullptr;
            uint16_t *yrow = (tok >= 0) ? p.y + int64_t(tok) * p.y_ld + p.col0[s] : nullptr;
            for (int c = cb; c < ce; ++c, ++g) {
                const int stage = g % STAGES, ab = g & 1;
                const bool got =
                    mbar_wait_bounded(bar_acc_full + 8 * ab, uint32_t(g >> 1) & 1u, s_abort, deadline) &&
                    mbar_wait_bounded(bar_full + 8 * stage, uint32_t(g / STAGES) & 1u, s_abort, deadline);
                if (__all_sync(0xffffffffu, got) == 0) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int c0 = (c - p.chunk0[s]) * XU_BN;
                const int ncols = min(XU_BN, n_s - c0);         // a multiple of 8
                const uint8_t *ysm = smem + L.ring_off + stage * L.stage_bytes + L.y_off + row * 128;
                const uint16_t *sbias = reinterpret_cast<const uint16_t *>(
                    smem + L.ring_off + stage * L.stage_bytes + L.bias_off);
                uint32_t va[32];
                tmem_ld32_nowait(tmem + ab * XU_BN + hf * 32 + (uint32_t(q * 32) << 16), va);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_acc_empty + 8 * ab);   // TMEM buffer free
                if (yrow != nullptr) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int cl = hf * 32 + j * 8;                 // 8 columns, one 16-byte piece
                        if (cl >= ncols) break;
                        uint32_t yw[4] = {0u, 0u, 0u, 0u}, bw[4] = {0u, 0u, 0u, 0u};
                        if (p.add_inputs) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(
                                ysm + ((((hf * 4 + j) ^ (row & 7))) << 4));
                            yw[0] = v.x; yw[1] = v.y; yw[2] = v.z; yw[3] = v.w;
                        }
                        if (bias_row != nullptr && p.bias_vec) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(sbias + cl);
                            bw[0] = v.x; bw[1] = v.y; bw[2] = v.z; bw[3] = v.w;
                        } else if (bias_row != nullptr) {
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                bw[k] = uint32_t(bias_row[c0 + cl + 2 * k]) |
                                        (uint32_t(bias_row[c0 + cl + 2 * k + 1]) << 16);
                        }
                        uint32_t o[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float a0 = __uint_as_float(va[j * 8 + 2 * k]) + bf16_lo(bw[k]) + bf16_lo(yw[k]);
                            const float a1 = __uint_as_float(va[j * 8 + 2 * k + 1]) + bf16_hi(bw[k]) + bf16_hi(yw[k]);
                            o[k] = pack_bf16x2(a0, a1);
                        }
                        *reinterpret_cast<uint4 *>(yrow + c0 + cl) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * stage);    // this warp is done with the stage
            }
            w += ce - cb;
        }
    }

    if (tid == 0 && *s_abort) atomicOr(p.error_word, XU_ERROR_BIT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 2 * XU_BN);
}

// ------------------------------------------------------------------ host

typedef CUresult (*XuEncodeFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                               const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                               const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static XuEncodeFn xu_encode_fn()
{
    static XuEncodeFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<XuEncodeFn>(ptr);
    }
    return fn;
}

static bool xu_encode(XuEncodeFn fn, CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols,
                      uint64_t row_stride, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw)
{
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_stride * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launches the tensor-core expand if the shapes allow it: returns 1 if
// launched, 0 if not applicable, or a cudaError_t on a launch failure.
int launch_expand_umma(const ExpandLaunch &a, cudaStream_t stream)
{
    if (!a.vec || a.error_word == nullptr) return 0;
    // Token indices travel in 21 bits of a piece descriptor.
    if (a.num_tokens >= (1 << 21)) return 0;
    int rp = 16;
    while (rp < a.rank) rp <<= 1;
    if (rp > 128) return 0;
    XuEncodeFn fn = xu_encode_fn();
    if (fn == nullptr) return 0;
    const int nbins = a.max_loras + 1;
    int stages = XU_MAX_STAGES;
    while (stages > 2 && xu_layout(rp, stages, nbins).total > XU_SMEM_BUDGET) --stages;
    const XuLayout L = xu_layout(rp, stages, nbins);
    if (L.total > 227 * 1024) return 0;

    static ExpandUmmaArgs p;      // > 2 KB: keep off the stack
    const CUtensorMapSwizzle sw = (rp == 16) ? CU_TENSOR_MAP_SWIZZLE_32B
                                : (rp == 32) ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_128B;
    for (int s = 0; s < a.num_slices; ++s) {
        if (a.n[s] == 0) continue;
        if (!xu_encode(fn, &p.map_b[s], a.b[s], uint64_t(a.max_loras) * uint64_t(a.n[s]),
                       uint64_t(a.rank), uint64_t(a.rank), uint32_t(rp > 64 ? 64 : rp), XU_BN, sw))
            return 0;
    }
    for (int i = 0; i < XU_YMAPS; ++i)
        if (!xu_encode(fn, &p.map_y[i], a.y, uint64_t(a.num_tokens), uint64_t(a.y_ld),
                       uint64_t(a.y_ld), 64u, 1u << i, CU_TENSOR_MAP_SWIZZLE_128B))
            return 0;
    p.x = a.x;
    p.y = a.y;
    p.y_ld = a.y_ld;
    for (int s = 0; s < LORA_MAX_SLICES; ++s) {
        p.bias[s] = a.bias[s];
        p.n[s] = a.n[s];
        p.col0[s] = a.col0[s];
    }
    int chunks = 0;
    for (int s = 0; s < a.num_slices; ++s) {
        p.chunk0[s] = chunks;
        chunks += (a.n[s] + XU_BN - 1) / XU_BN;
    }
    p.chunk0[a.num_slices] = chunks;
    p.num_slices = a.num_slices;
    p.rank = a.rank;
    p.rp = rp;
    p.num_tokens = a.num_tokens;
    p.add_inputs = a.add_inputs;
    p.bias_vec = a.bias_vec;
    p.stages = stages;
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
        e = cudaFuncSetAttribute(expand_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 227 * 1024);
        if (e != cudaSuccess) return int(e);
        configured[dev] = 1;
    }
    e = launch_kernel(expand_umma_kernel, dim3(device_sm_count()), dim3(XU_THREADS),
                      size_t(L.total), stream, p);
    if (e != cudaSuccess) return int(e);
    return 1;
}

}  // namespace lora
