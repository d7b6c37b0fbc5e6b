// lora_expand_umma.cu -- tensor-core (tcgen05 / TMEM) path of lora_expand
// (page "vllm.lora.punica_wrapper.punica_gpu", PunicaWrapperGPU.add_expand;
// bias step of page "vllm.lora.punica_wrapper.punica_tpu",
// PunicaWrapperTPU._apply_bias):
//   y[t, off_s + j] (+)= x[s][t, :] @ B[s][id(t)][j, :] + bias[s][id(t)][j]
//
// Work items are (token tile of 128 tokens of one LoRA segment, 128-column
// chunk of one slice), numbered chunk-fastest; one persistent CTA per SM
// takes a contiguous, balanced range of them.  Eight warps, specialised:
//   warp 0      B producer: one 2-D TMA box per chunk (two for rank 128)
//               brings B[s][id][c0 : c0 + 128, :] in the swizzled K-major
//               layout UMMA reads.
//   warp 1      owns TMEM (two 128-column fp32 accumulators); lane 0 issues
//               tcgen05.mma (M = 128 tokens, N = 128 columns, K = 16 steps
//               over the rank) and commits.
//   warps 2, 3  y producers: coalesced 16-byte cp.async of the tile's y rows
//               (two rows of 256 bytes per warp instruction) and of the bias
//               chunk into the stage; each thread's copies arrive on the
//               stage's mbarrier when they land.
//   warps 4..7  epilogue, one token row per thread (its TMEM lane): at each
//               new tile, the fp32 x rows are rounded to bf16 into the A
//               operand tile; per chunk, tcgen05.ld 16 columns at a time,
//               add bias and old y in fp32, round once to bf16 in place in
//               the shared y row, then the four warps store the tile back
//               with coalesced 16-byte stores.
// The accumulators are double-buffered so the MMA of chunk i + 1 runs while
// the epilogue drains chunk i; y and B stream through a ring of stages.
//
// Used when y rows, offsets and slice widths are 16-byte aligned (the same
// condition as the vector path of the mma.sync kernel).  Every mbarrier
// wait is bounded; on expiry the kernel sets bit 30 of the metadata error
// word, drains its copies and MMAs, frees TMEM and returns.
#include "lora_common.cuh"
#include "lora_umma.cuh"

namespace lora {

constexpr int XU_BM = 128;              // tokens per tile (UMMA M, TMEM lanes)
constexpr int XU_BN = 128;              // columns per chunk (UMMA N)
constexpr int XU_THREADS = 256;
constexpr int XU_MAX_STAGES = 4;
constexpr int XU_SMEM_BUDGET = 200 * 1024;
constexpr int XU_Y_LD = XU_BN * 2 + 16;  // padded shared y row (bytes)
constexpr long long XU_TIMEOUT_CYCLES = 2000000000ll;
constexpr int XU_ERROR_BIT = 1 << 30;

struct ExpandUmmaArgs {
    CUtensorMap map_b[LORA_MAX_SLICES];      // B[s]: [L * n_s rows, r cols], box {min(rp, 64), 128}
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
    int a_bytes, y_bytes, b_bytes, bias_off, stage_bytes, ring_off, bar_off, misc_off, tok_off,
        etok_off, tab_off, total;
};

__host__ __device__ inline XuLayout xu_layout(int rp, int stages, int nbins)
{
    XuLayout l;
    l.a_bytes = XU_BM * rp * 2;                          // x tile, bf16
    l.y_bytes = XU_BM * XU_Y_LD;
    l.b_bytes = XU_BN * rp * 2;
    l.bias_off = l.b_bytes + l.y_bytes;                  // within the stage
    l.stage_bytes = ((l.bias_off + XU_BN * 2) + 1023) & ~1023;
    l.ring_off = l.a_bytes;                              // stage: B tile | y tile | bias
    l.bar_off = l.ring_off + stages * l.stage_bytes;
    l.misc_off = l.bar_off + (3 * XU_MAX_STAGES + 6) * 8;  // + acc[2] x2, x_ready, drain
    l.tok_off = l.misc_off + 16;                         // producer-side token rows
    l.etok_off = l.tok_off + XU_BM * 4;                  // epilogue-side token rows
    l.tab_off = l.etok_off + XU_BM * 4;
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

__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void named_barrier(int id, int count)
{
    asm volatile("bar.sync %0, %1;\n" :: "r"(id), "r"(count) : "memory");
}

__global__ void __launch_bounds__(XU_THREADS, 1) expand_umma_kernel(const __grid_constant__ ExpandUmmaArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int RP = p.rp, STAGES = p.stages, S = p.num_slices, R = p.rank;
    const XuLayout L = xu_layout(RP, STAGES, p.nbins);
    const uint32_t base = smem_addr(smem);
    const uint32_t bar_full_b = base + L.bar_off;                 // [STAGES] TMA (B)
    const uint32_t bar_full_y = bar_full_b + 8 * XU_MAX_STAGES;    // [STAGES] 64 y producers
    const uint32_t bar_empty = bar_full_y + 8 * XU_MAX_STAGES;     // [STAGES] MMA + 4 epilogue warps
    const uint32_t bar_acc_full = bar_empty + 8 * XU_MAX_STAGES;   // [2]
    const uint32_t bar_acc_empty = bar_acc_full + 16;              // [2]
    const uint32_t bar_x_ready = bar_acc_empty + 16;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + L.misc_off);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + L.misc_off + 4);
    int *s_tok = reinterpret_cast<int *>(smem + L.tok_off);
    int *s_etok = reinterpret_cast<int *>(smem + L.etok_off);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    pdl_wait();
    pdl_launch_dependents();

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(bar_full_b + 8 * i, 1);
            mbar_init(bar_full_y + 8 * i, 64);
            mbar_init(bar_empty + 8 * i, 5);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_acc_full + 8 * i, 1);
            mbar_init(bar_acc_empty + 8 * i, 4);
        }
        mbar_init(bar_x_ready, 4);
        mbar_fence_init();
        *s_abort = 0;
        for (int s = 0; s < S; ++s) tma_prefetch_map(&p.map_b[s]);
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
    const uint32_t b_tx = uint32_t(L.b_bytes);

    // Row-item decoding shared by all roles.
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
        // -------------------------------------------------- B producer (TMA)
        if (lane == 0) {
            int g = 0;
            bool ok = true;
            for (int64_t w = w_begin; ok && w < w_end;) {
                int tile, s, cb, ce, id, row0, nrows;
                row_item(w, tile, s, cb, ce);
                tile_rows(tile, id, row0, nrows);
                for (int c = cb; c < ce; ++c, ++g) {
                    const int stage = g % STAGES;
                    const uint32_t ph = uint32_t(g / STAGES) & 1u;
                    if (!mbar_wait_bounded(bar_empty + 8 * stage, ph ^ 1u, s_abort, deadline)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sb = base + L.ring_off + stage * L.stage_bytes;
                    const uint32_t full = bar_full_b + 8 * stage;
                    mbar_arrive_expect_tx(full, b_tx);
                    const int brow = id * p.n[s] + (c - p.chunk0[s]) * XU_BN;
                    for (int k = 0; k < b_boxes; ++k)
                        tma_load_2d(sb + k * XU_BN * 128, &p.map_b[s], k * 64, brow, full);
                }
                w += ce - cb;
            }
            // every issued box must land before the CTA may exit
            const long long dd = clock64() + XU_TIMEOUT_CYCLES;
            for (int i = max(0, g - STAGES); i < g; ++i)
                while (!mbar_try_wait(bar_full_b + 8 * (i % STAGES), uint32_t(i / STAGES) & 1u) &&
                       clock64() < dd) {
                }
        }
        __syncwarp();
    } else if (warp == 1) {
        // -------------------------------------------------- MMA issue
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
                    if (!mbar_wait_bounded(bar_full_b + 8 * stage, uint32_t(g / STAGES) & 1u, s_abort, deadline) ||
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
                const uint32_t bar_drain = bar_x_ready + 8;
                mbar_init(bar_drain, 1);
                asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
                umma_commit(bar_drain);
                const long long dd = clock64() + XU_TIMEOUT_CYCLES;
                while (!mbar_try_wait(bar_drain, 0) && clock64() < dd) {
                }
            }
        }
        __syncwarp();
    } else if (warp < 4) {
        // -------------------------------------------------- y producers
        // After an abort the threads keep walking the items (skipping the
        // work) so that the named barriers stay matched.
        const int ptid = tid - 64;                       // 0..63
        const int pw = warp - 2;                         // 0..1
        int g = 0;
        bool ok = true;
        for (int64_t w = w_begin; w < w_end;) {
            int tile, s, cb, ce, id, row0, nrows;
            row_item(w, tile, s, cb, ce);
            tile_rows(tile, id, row0, nrows);
            named_barrier(1, 64);                        // previous item fully issued
            for (int r = ptid; r < XU_BM; r += 64) s_tok[r] = (r < nrows) ? p.sorted[row0 + r] : -1;
            named_barrier(1, 64);
            const int n_s = p.n[s];
            const uint16_t *bias_row = p.bias[s] ? p.bias[s] + int64_t(id) * n_s : nullptr;
            uint16_t *yslice = p.y + p.col0[s];
            for (int c = cb; c < ce; ++c, ++g) {
                const int stage = g % STAGES;
                const uint32_t ph = uint32_t(g / STAGES) & 1u;
                if (ok) ok = mbar_wait_bounded(bar_empty + 8 * stage, ph ^ 1u, s_abort, deadline);
                if (!ok) continue;
                const uint32_t st = base + L.ring_off + stage * L.stage_bytes;
                const int c0 = (c - p.chunk0[s]) * XU_BN;
                const int ncols = min(XU_BN, n_s - c0);
                if (p.add_inputs) {
                    // warp pw covers row pairs pw, pw + 2, ...: lanes 0..15 one row, 16..31 the next
                    const int cc = lane & 15;
                    for (int pr = pw; pr < XU_BM / 2; pr += 2) {
                        const int r = 2 * pr + (lane >> 4);
                        const int tok = s_tok[r];
                        if (tok >= 0 && cc * 8 < ncols)
                            cp_async16(st + L.b_bytes + r * XU_Y_LD + cc * 16,
                                       yslice + int64_t(tok) * p.y_ld + c0 + cc * 8, true);
                    }
                }
                if (bias_row != nullptr && p.bias_vec && ptid < XU_BN / 8 && ptid * 8 < ncols)
                    cp_async16(st + L.bias_off + ptid * 16, bias_row + c0 + ptid * 8, true);
                cp_async_mbar_arrive_noinc(bar_full_y + 8 * stage);
            }
            w += ce - cb;
        }
        cp_async_wait<0>();
    } else {
        // -------------------------------------------------- epilogue
        // After an abort the warps keep walking the items (skipping the
        // work) so that the named barriers stay matched.
        const int q = warp & 3;                          // TMEM lane quarter
        const int row = q * 32 + lane;
        const int etid = tid - 128;                      // 0..127
        int g = 0, items = 0;
        bool ok = true;
        for (int64_t w = w_begin; w < w_end; ++items) {
            int tile, s, cb, ce, id, row0, nrows;
            row_item(w, tile, s, cb, ce);
            tile_rows(tile, id, row0, nrows);
            const int tok = (row < nrows) ? p.sorted[row0 + row] : -1;
            named_barrier(2, 128);                       // previous item's stores done
            s_etok[row] = tok;
            // x row of this token -> bf16 A operand row (zeros past the rank / rows)
            {
                const float *xr = p.x + (int64_t(s) * p.num_tokens + (tok >= 0 ? tok : 0)) * R;
                for (int c = 0; c < RP / 8; ++c) {
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
                asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_x_ready);
            }
            named_barrier(2, 128);                       // s_etok visible
            const int n_s = p.n[s];
            const uint16_t *bias_row = p.bias[s] ? p.bias[s] + int64_t(id) * n_s : nullptr;
            uint16_t *yslice = p.y + p.col0[s];
            for (int c = cb; c < ce; ++c, ++g) {
                const int stage = g % STAGES, ab = g & 1;
                if (ok) {
                    bool got = mbar_wait_bounded(bar_acc_full + 8 * ab, uint32_t(g >> 1) & 1u, s_abort, deadline) &&
                               mbar_wait_bounded(bar_full_y + 8 * stage, uint32_t(g / STAGES) & 1u, s_abort, deadline);
                    ok = __all_sync(0xffffffffu, got) != 0;
                }
                const int c0 = (c - p.chunk0[s]) * XU_BN;
                const int ncols = min(XU_BN, n_s - c0);
                if (ok) {
                    tc_fence_after();
                    uint8_t *sy = smem + L.ring_off + stage * L.stage_bytes + L.b_bytes + row * XU_Y_LD;
                    const uint16_t *sbias = reinterpret_cast<const uint16_t *>(
                        smem + L.ring_off + stage * L.stage_bytes + L.bias_off);
                    // 64 columns per round: two 32-column TMEM loads in flight, one wait
                    for (int h = 0; h < XU_BN / 64; ++h) {
                        uint32_t va[32], vb[32];
                        const uint32_t ta = tmem + ab * XU_BN + h * 64 + (uint32_t(q * 32) << 16);
                        tmem_ld32_nowait(ta, va);
                        tmem_ld32_nowait(ta + 32, vb);
                        tmem_wait_ld();
                        if (tok < 0) continue;
#pragma unroll
                        for (int j4 = 0; j4 < 4; ++j4) {
                            const int j = h * 4 + j4;
                            if (j * 16 >= ncols) continue;
                            float v[16];
#pragma unroll
                            for (int k = 0; k < 16; ++k)
                                v[k] = __uint_as_float(j4 < 2 ? va[(j4 & 1) * 16 + k] : vb[(j4 & 1) * 16 + k]);
                            uint4 *yp = reinterpret_cast<uint4 *>(sy + j * 32);
                            uint32_t yw[8], bw[8];
                            if (p.add_inputs) {
                                const uint4 y0 = yp[0], y1 = yp[1];
                                yw[0] = y0.x; yw[1] = y0.y; yw[2] = y0.z; yw[3] = y0.w;
                                yw[4] = y1.x; yw[5] = y1.y; yw[6] = y1.z; yw[7] = y1.w;
                            } else {
#pragma unroll
                                for (int k = 0; k < 8; ++k) yw[k] = 0u;
                            }
                            if (bias_row != nullptr && p.bias_vec) {
                                const uint4 b0 = reinterpret_cast<const uint4 *>(sbias + j * 16)[0];
                                const uint4 b1 = reinterpret_cast<const uint4 *>(sbias + j * 16)[1];
                                bw[0] = b0.x; bw[1] = b0.y; bw[2] = b0.z; bw[3] = b0.w;
                                bw[4] = b1.x; bw[5] = b1.y; bw[6] = b1.z; bw[7] = b1.w;
                            } else if (bias_row != nullptr) {
#pragma unroll
                                for (int k = 0; k < 8; ++k) {
                                    const int cc = j * 16 + 2 * k;
                                    const uint32_t lo = cc < ncols ? bias_row[c0 + cc] : 0u;
                                    const uint32_t hi = cc + 1 < ncols ? bias_row[c0 + cc + 1] : 0u;
                                    bw[k] = lo | (hi << 16);
                                }
                            } else {
#pragma unroll
                                for (int k = 0; k < 8; ++k) bw[k] = 0u;
                            }
                            uint32_t o[8];
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const float a0 = v[2 * k] + bf16_lo(bw[k]) + bf16_lo(yw[k]);
                                const float a1 = v[2 * k + 1] + bf16_hi(bw[k]) + bf16_hi(yw[k]);
                                o[k] = pack_bf16x2(a0, a1);
                            }
                            yp[0] = make_uint4(o[0], o[1], o[2], o[3]);
                            yp[1] = make_uint4(o[4], o[5], o[6], o[7]);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_acc_empty + 8 * ab);
                }
                named_barrier(2, 128);                   // every row of the tile combined
                if (ok) {
                    // coalesced store: two rows of 256 bytes per warp instruction
                    const int cc = lane & 15;
                    const uint8_t *ys = smem + L.ring_off + stage * L.stage_bytes + L.b_bytes;
                    for (int pr = etid >> 5; pr < XU_BM / 2; pr += 4) {
                        const int r = 2 * pr + (lane >> 4);
                        const int t = s_etok[r];
                        if (t >= 0 && cc * 8 < ncols) {
                            const uint4 val = *reinterpret_cast<const uint4 *>(ys + r * XU_Y_LD + cc * 16);
                            *reinterpret_cast<uint4 *>(yslice + int64_t(t) * p.y_ld + c0 + cc * 8) = val;
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_empty + 8 * stage);
                }
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

// Launches the tensor-core expand if the shapes allow it: returns 1 if
// launched, 0 if not applicable, or a cudaError_t on a launch failure.
int launch_expand_umma(const ExpandLaunch &a, cudaStream_t stream)
{
    if (!a.vec || a.error_word == nullptr) return 0;
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

    static ExpandUmmaArgs p;      // > 1 KB: keep off the stack
    const CUtensorMapSwizzle sw = (rp == 16) ? CU_TENSOR_MAP_SWIZZLE_32B
                                : (rp == 32) ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_128B;
    for (int s = 0; s < a.num_slices; ++s) {
        if (a.n[s] == 0) continue;
        const cuuint64_t dims[2] = {cuuint64_t(a.rank), cuuint64_t(a.max_loras) * cuuint64_t(a.n[s])};
        const cuuint64_t strides[1] = {cuuint64_t(a.rank) * 2};
        const cuuint32_t box[2] = {cuuint32_t(rp > 64 ? 64 : rp), cuuint32_t(XU_BN)};
        const cuuint32_t estr[2] = {1, 1};
        if (fn(&p.map_b[s], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(a.b[s]),
               dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return 0;
    }
    p.x = a.x;
    p.y = a.y;
    p.y_ld = a.y_ld;
    for (int s = 0; s < LORA_MAX_SLICES; ++s) {
        p.bias[s] = a.bias[s];
        p.n[s] = a.n[s];
        p.col0[s] = a.col0[s];
    }
    for (int s = 0; s <= a.num_slices; ++s) p.chunk0[s] = 0;
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
