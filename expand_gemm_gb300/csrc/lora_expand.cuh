// lora_expand.cuh -- tile shapes, arguments and the per-CTA item loop of
// the expand (page "vllm.lora.punica_wrapper.punica_gpu",
// PunicaWrapperGPU.add_expand; bias step of page
// "vllm.lora.punica_wrapper.punica_tpu", PunicaWrapperTPU._apply_bias),
// shared by the expand kernel and the single-kernel lora_linear.
#pragma once

#include "lora_common.cuh"

namespace lora {

constexpr int EX_BM = 64;          // tokens per tile
constexpr int EX_THREADS = 256;    // 8 warps
constexpr int EX_STAGES = 3;

struct ExpandArgs {
    const void *x;                       // [S, T, r]: fp32, or bf16 when x_bf16
    int32_t x_bf16;
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
    int32_t vec;                         // 16-byte y path allowed
    int32_t bias_vec;                    // 16-byte bias loads allowed (every bias)
    const int32_t *sorted;
    const int32_t *counts;
    const int32_t *start_loc;
    const int32_t *active;
    const int32_t *no_lora;
    int32_t *error_word;                 // debug checks report here
    int32_t nbins;
    // Early mode (set only by lora_linear, whose preceding kernel is its own
    // shrink): the segment table, the token list and the y / B / bias loads
    // of the first tile are issued before the grid-dependency wait; only the
    // shrink output (x) is read after it.  Safe because the shrink lets its
    // dependents launch only after its own wait, i.e. once the metadata
    // kernel and everything before it in the stream have completed, and the
    // shrink writes neither the metadata, y, B nor bias.
    int32_t early;
};

// Batches of up to this many tokens keep the whole sorted token list in
// shared memory (4 bytes a token).
constexpr int EX_TOKLIST_MAX = 1024;

template <int KT>
struct ExpandTile {
    static constexpr int RP = 16 * KT;                 // padded rank
    static constexpr int CPR = RP / 8;                 // 16-byte chunks per row
    static constexpr int BN = (KT >= 8) ? 64 : 128;    // columns per chunk
    static constexpr int WARPS_M = (BN == 128) ? 2 : 4;
    static constexpr int WARPS_N = 8 / WARPS_M;
    static constexpr int WM = EX_BM / WARPS_M;         // rows per warp
    static constexpr int WN = BN / WARPS_N;            // columns per warp (32)
    static constexpr int MI = WM / 16;
    static constexpr int NI = WN / 8;
    static constexpr int YCH = BN / 8;                 // 16-byte chunks per y row
    // DIRECT epilogue (128-column chunks): each thread's accumulators cover 8
    // contiguous columns (B rows stored permuted, see b_slot) and leave with
    // 16-byte stores straight to global memory.  Otherwise (64-column chunks,
    // rank 128, measured faster): the tile is rounded in place in shared
    // memory and written back row by row.
    static constexpr bool DIRECT = (BN == 128);
    static constexpr int Y_LD = DIRECT ? BN * 2 : BN * 2 + 16;   // shared y row (bytes)
    static constexpr int Y_BYTES = EX_BM * Y_LD;
    static constexpr int B_BYTES = BN * RP * 2;
    static constexpr int BIAS_BYTES = BN * 2;                // bf16 bias chunk
    static constexpr int STAGE_BYTES = Y_BYTES + B_BYTES + BIAS_BYTES;
    static constexpr int A_BYTES = EX_BM * RP * 2;
    // ring stages of the expand kernel: rank 32 takes two, which leaves room
    // (shared memory and, at 80 registers, the register file) for three
    // CTAs per SM instead of two
    static constexpr int NST = (KT == 2) ? 2 : EX_STAGES;
    static constexpr int BYTES = NST * STAGE_BYTES + A_BYTES;
    // Copy shapes: y pieces (16 bytes) of one row are taken by YCH
    // consecutive threads, so one pass covers Y_RPP rows and every thread
    // keeps the same Y_PASSES rows for a whole tile; B likewise with CPR
    // threads per row and B_RPP rows per pass.
    static constexpr int Y_RPP = EX_THREADS / YCH;
    static constexpr int Y_PASSES = EX_BM / Y_RPP;
    static constexpr int B_RPP = EX_THREADS / CPR;
    static constexpr int B_PASSES = (BN + B_RPP - 1) / B_RPP;
    static_assert(WN == 32 && NI == 4 && MI >= 1, "warp tile: 8 output columns per thread");
    static_assert(EX_THREADS % YCH == 0 && EX_BM % Y_RPP == 0, "y copy shape");
    static_assert(EX_THREADS % CPR == 0 && B_RPP % 8 == 0, "B copy shape (swizzle period)");
};

template <int KT>
constexpr int expand_bn() { return ExpandTile<KT>::BN; }

inline size_t expand_smem_bytes(int kt, int nbins)
{
    size_t t = 0;
    switch (kt) {
    case 1: t = ExpandTile<1>::BYTES; break;
    case 2: t = ExpandTile<2>::BYTES; break;
    case 4: t = ExpandTile<4>::BYTES; break;
    default: t = ExpandTile<8>::BYTES; break;
    }
    return t + seg_tab_bytes(nbins);
}

// 16-byte piece `chunk` of shared y-tile row `row`: odd rows swap the two
// halves of every 8-piece group, so the two rows a quarter-warp reads with
// 16-byte loads fall in disjoint banks.
__device__ __forceinline__ int ysw(int row, int chunk)
{
    return chunk ^ ((row & 1) << 2);
}

// Shared row of B row (output column) r of a chunk.  Within each 32-column
// warp block, column q * 8 + 2n + e (q, n < 4, e < 2) goes to row
// n * 8 + 2q + e: the MMA's n-tile n then reads, as its columns 2q + e, the
// output columns q * 8 + 2n + e, so each thread's accumulators cover 8
// contiguous columns.  The reads stay on 8 consecutive rows (conflict-free
// under swz).
__device__ __forceinline__ int b_slot(int r)
{
    const int l = r & 31;
    return (r & ~31) | (((l >> 1) & 3) << 3) | ((l >> 3) << 1) | (l & 1);
}

// Host: checks the arguments of an expand call and fills `p` (the layout
// rules and the slice table); returns LORA_OK, 1 when there is nothing to
// do (no tokens or no columns), or a negative status.
int expand_setup(ExpandArgs &p, const void *x, int x_bf16, const lora_bf16_t *const *lora_b,
                 const lora_bf16_t *const *lora_bias, const int32_t *slice_sizes,
                 int32_t num_slices, int32_t rank, lora_bf16_t *y, int64_t y_ld,
                 int32_t num_tokens, int32_t offset_start, int32_t add_inputs,
                 const lora_meta_t *meta);

// The expand work of one CTA: items are (token tile of one LoRA segment,
// BN-column chunk of one slice), numbered chunk-fastest; the CTA takes one
// contiguous, balanced range of them (by blockIdx.x / gridDim.x).  The
// segment table `tab` and the sorted token list `tokens` are already known.
// The y / B / bias copies stream through a ring of NST stages.  `gate()` is
// called once by all threads, right before the first read of x (the shrink
// output), with the copies of the first NST - 1 chunks already in flight.  When it returns false the CTA drains its copies and
// stops.  x is read with L2-only loads, so rows that other CTAs of the same
// grid accumulated are never served from a stale L1 line.
template <int KT, int NST = EX_STAGES, class Gate>
__device__ __forceinline__ void expand_items(const ExpandArgs &p, SegTab tab,
                                             const int32_t *tokens, int total_tiles,
                                             uint8_t *smem, int *s_tok, Gate gate)
{
    using Cfg = ExpandTile<KT>;
    constexpr int CPR = Cfg::CPR, BN = Cfg::BN, MI = Cfg::MI, NI = Cfg::NI, YCH = Cfg::YCH;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm = warp / Cfg::WARPS_N, wn = warp % Cfg::WARPS_N;
    const int S = p.num_slices, R = p.rank, T = p.num_tokens;
    uint8_t *sA = smem + NST * Cfg::STAGE_BYTES;
    bool gated = false;
    const int nchunks = p.chunk0[S];
    const int64_t total = int64_t(total_tiles) * nchunks;
    // Balanced contiguous ranges: the last `rem` CTAs take one item more
    // (in the single-kernel lora_linear the first CTAs also carry the
    // shrink items).  32-bit arithmetic whenever the item count allows.
    const bool small = total < int64_t(INT32_MAX);
    int64_t w, w_end;
    if (small) {
        const uint32_t g = gridDim.x, b = blockIdx.x, t32 = uint32_t(total);
        const uint32_t base = t32 / g, rem = t32 - base * g, first_extra = g - rem;
        w = int64_t(b * base + (b > first_extra ? b - first_extra : 0u));
        w_end = w + base + (b >= first_extra ? 1 : 0);
    } else {
        w = int64_t(blockIdx.x) * total / gridDim.x;
        w_end = int64_t(blockIdx.x + 1) * total / gridDim.x;
    }
    const uint32_t ring = smem_addr(smem), aA = smem_addr(sA);
    const bool prefetch_y = p.vec && p.add_inputs;

    while (w < w_end) {
        // ---- one row item: token tile `tile`, slice s, chunks [cb, ce)
        const int tile = small ? int(uint32_t(w) / uint32_t(nchunks)) : int(w / nchunks);
        const int cb = int(w - int64_t(tile) * nchunks);
        int s = 0;
        while (s + 1 < S && p.chunk0[s + 1] <= cb) ++s;
        const int ce = int(min(int64_t(p.chunk0[s + 1]), int64_t(cb) + (w_end - w)));
        w += ce - cb;

        const int seg = find_segment(tab.tile, p.nbins, tile);
        const int id = tab.id[seg];
        const int row0 = tab.start[seg] + (tile - tab.tile[seg]) * EX_BM;
        const int nrows = min(EX_BM, tab.start[seg] + tab.count[seg] - row0);
        const int n_s = p.n[s];
        const uint16_t *bslice = p.b[s] + int64_t(id) * n_s * R;
        const uint16_t *bias_row = p.bias[s] ? p.bias[s] + int64_t(id) * n_s : nullptr;
        uint16_t *yslice = p.y + p.col0[s];

        if (tid < EX_BM)
            s_tok[tid] = (tid < nrows) ? checked_token(tokens[row0 + tid], T, p.error_word) : -1;
        __syncthreads();

        // This thread's y rows for the whole tile (piece ycc of rows
        // yr0 + j * Y_RPP), and its B row / piece of every chunk.
        const int ycc = tid % YCH, yr0 = tid / YCH;
        int ytok[Cfg::Y_PASSES];
#pragma unroll
        for (int j = 0; j < Cfg::Y_PASSES; ++j) ytok[j] = s_tok[yr0 + j * Cfg::Y_RPP];
        uint16_t *const ybase = yslice + ycc * 8;
        const uint32_t y_soff = yr0 * Cfg::Y_LD + (Cfg::DIRECT ? ysw(yr0, ycc) : ycc) * 16;
        const int bcc = tid % CPR, br0 = tid / CPR;
        const bool b_kin = bcc * 8 < R;
        const uint16_t *brow = bslice + int64_t(br0) * R + bcc * 8;

        auto load_chunk = [&](int slot, int c) {
            const int c0 = (c - p.chunk0[s]) * BN;
            const int ncols = min(BN, n_s - c0);
            const uint32_t sy = ring + slot * Cfg::STAGE_BYTES;
            const uint32_t sb = sy + Cfg::Y_BYTES;
            if (prefetch_y) {
                const bool cin = ycc * 8 < ncols;
#pragma unroll
                for (int j = 0; j < Cfg::Y_PASSES; ++j) {
                    const bool ok = cin && ytok[j] >= 0;
                    cp_async16(sy + y_soff + j * Cfg::Y_RPP * Cfg::Y_LD,
                               ok ? ybase + (int64_t(ytok[j]) * p.y_ld + c0) : p.y, ok);
                }
            }
            const uint16_t *bc = brow + int64_t(c0) * R;
#pragma unroll
            for (int j = 0; j < Cfg::B_PASSES; ++j) {
                const int r = br0 + j * Cfg::B_RPP;
                if (Cfg::B_PASSES * Cfg::B_RPP > BN && r >= BN) break;
                const bool ok = b_kin && r < ncols;
                cp_async16(sb + swz<CPR>(Cfg::DIRECT ? b_slot(r) : r, bcc),
                           ok ? bc + int64_t(j) * Cfg::B_RPP * R : p.b[s], ok);
            }
            if (bias_row != nullptr && p.bias_vec && tid < BN / 8) {
                const bool ok = tid * 8 < ncols;
                cp_async16(sb + Cfg::B_BYTES + tid * 16, ok ? bias_row + c0 + tid * 8 : bias_row, ok);
            }
        };

#pragma unroll
        for (int st = 0; st < NST - 1; ++st) {
            if (cb + st < ce) load_chunk(st, cb + st);
            cp_async_commit();
        }

        if (!gated) {                         // the shrink output is read from here on
            gated = true;
            if (!gate()) {
                cp_async_wait<0>();
                __syncthreads();
                return;
            }
        }
        // x rows of this tile and slice -> bf16 A operand (overlaps the ring
        // fill): fp32 rows are rounded to bf16, bf16 rows are copied as they are
        {
            const int64_t xoff = int64_t(s) * T * R;
            for (int i = tid; i < EX_BM * CPR; i += EX_THREADS) {
                const int r = i / CPR, cc = i - r * CPR;
                const int tok = s_tok[r];
                uint4 v = make_uint4(0, 0, 0, 0);
                if (tok >= 0 && cc * 8 < R) {
                    const int64_t e = xoff + int64_t(tok) * R + cc * 8;
                    if (p.x_bf16) {
                        v = __ldcg(reinterpret_cast<const uint4 *>(
                            static_cast<const uint16_t *>(p.x) + e));
                    } else {
                        const float4 *src = reinterpret_cast<const float4 *>(
                            static_cast<const float *>(p.x) + e);
                        const float4 u = __ldcg(src), q = __ldcg(src + 1);
                        v.x = pack_bf16x2(u.x, u.y);
                        v.y = pack_bf16x2(u.z, u.w);
                        v.z = pack_bf16x2(q.x, q.y);
                        v.w = pack_bf16x2(q.z, q.w);
                    }
                }
                *reinterpret_cast<uint4 *>(sA + swz<CPR>(r, cc)) = v;
            }
        }
        __syncthreads();
        uint32_t af[MI][KT][4];
#pragma unroll
        for (int m = 0; m < MI; ++m)
#pragma unroll
            for (int kk = 0; kk < KT; ++kk) {
                const int r = wm * Cfg::WM + m * 16 + (lane & 15);
                const int c = kk * 2 + (lane >> 4);
                ldmatrix_x4(aA + swz<CPR>(r, c), af[m][kk][0], af[m][kk][1], af[m][kk][2],
                            af[m][kk][3]);
            }

        for (int i = 0; cb + i < ce; ++i) {
            cp_async_wait<NST - 2>();
            __syncthreads();
            {
                const int nxt = i + NST - 1;
                if (cb + nxt < ce) load_chunk(nxt % NST, cb + nxt);
                cp_async_commit();
            }
            const int slot = i % NST;
            const int c0 = (cb + i - p.chunk0[s]) * BN;
            const int ncols = min(BN, n_s - c0);
            uint8_t *sy = smem + slot * Cfg::STAGE_BYTES;
            const uint32_t sb = ring + slot * Cfg::STAGE_BYTES + Cfg::Y_BYTES;

            // This thread's output column for n-tile n, pair element e: in the
            // DIRECT layout colw + 2n + e (8 contiguous ones), else the MMA's
            // own n * 8 + 2 (lane % 4) + e.
            const int colw = wn * Cfg::WN + (lane & 3) * 8;
            auto out_col = [&](int n, int e) {
                return Cfg::DIRECT ? colw + 2 * n + e : wn * Cfg::WN + n * 8 + 2 * (lane & 3) + e;
            };

            // bias of this chunk: staged with the chunk when aligned, else read here
            float bv[NI][2];
            const uint16_t *sbias = reinterpret_cast<const uint16_t *>(
                smem + slot * Cfg::STAGE_BYTES + Cfg::Y_BYTES + Cfg::B_BYTES);
#pragma unroll
            for (int n = 0; n < NI; ++n)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c = out_col(n, h);
                    float b = 0.f;
                    if (bias_row != nullptr && c < ncols)
                        b = bf16_to_f32(p.bias_vec ? sbias[c] : bias_row[c0 + c]);
                    bv[n][h] = b;
                }

            // the accumulators start at the bias, so the product lands on it
            float acc[MI][NI][4];
#pragma unroll
            for (int m = 0; m < MI; ++m)
#pragma unroll
                for (int n = 0; n < NI; ++n)
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[m][n][q] = bv[n][q & 1];
            // B operand (DIRECT: shared row j of n-tile n holds the B row that
            // b_slot maps there, so the thread that gets C columns 2q, 2q + 1
            // of every n-tile holds the output columns colw .. colw + 7).
#pragma unroll
            for (int kk = 0; kk < KT; ++kk)
#pragma unroll
                for (int n2 = 0; n2 < NI / 2; ++n2) {
                    uint32_t b[4];
                    const int q = lane >> 3;
                    const int r = wn * Cfg::WN + n2 * 16 + (q >> 1) * 8 + (lane & 7);
                    const int c = kk * 2 + (q & 1);
                    ldmatrix_x4(sb + swz<CPR>(r, c), b[0], b[1], b[2], b[3]);
#pragma unroll
                    for (int m = 0; m < MI; ++m) {
                        mma_bf16_16816(acc[m][2 * n2], af[m][kk], b[0], b[1]);
                        mma_bf16_16816(acc[m][2 * n2 + 1], af[m][kk], b[2], b[3]);
                    }
                }

            if (Cfg::DIRECT && p.vec) {
                // per row: old y (one 16-byte shared load) + product + bias,
                // rounded once, one 16-byte store straight to global memory
                if (colw < ncols) {
#pragma unroll
                    for (int m = 0; m < MI; ++m)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int r = wm * Cfg::WM + m * 16 + (lane >> 2) + 8 * h;
                            const int tok = s_tok[r];
                            if (tok < 0) continue;
                            float v[2 * NI];
#pragma unroll
                            for (int n = 0; n < NI; ++n) {
                                v[2 * n] = acc[m][n][2 * h];
                                v[2 * n + 1] = acc[m][n][2 * h + 1];
                            }
                            if (p.add_inputs) {
                                const uint4 old = *reinterpret_cast<const uint4 *>(
                                    sy + r * Cfg::Y_LD + ysw(r, colw >> 3) * 16);
                                v[0] += bf16_lo(old.x);
                                v[1] += bf16_hi(old.x);
                                v[2] += bf16_lo(old.y);
                                v[3] += bf16_hi(old.y);
                                v[4] += bf16_lo(old.z);
                                v[5] += bf16_hi(old.z);
                                v[6] += bf16_lo(old.w);
                                v[7] += bf16_hi(old.w);
                            }
                            uint4 out;
                            out.x = pack_bf16x2(v[0], v[1]);
                            out.y = pack_bf16x2(v[2], v[3]);
                            out.z = pack_bf16x2(v[4], v[5]);
                            out.w = pack_bf16x2(v[6], v[7]);
                            *reinterpret_cast<uint4 *>(yslice + int64_t(tok) * p.y_ld + c0 + colw) =
                                out;
                        }
                }
            } else if (p.vec) {
                // round in place in the shared tile, then whole rows out
#pragma unroll
                for (int m = 0; m < MI; ++m)
#pragma unroll
                    for (int n = 0; n < NI; ++n)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int r = wm * Cfg::WM + m * 16 + (lane >> 2) + 8 * h;
                            uint32_t *cell = reinterpret_cast<uint32_t *>(
                                sy + r * Cfg::Y_LD + out_col(n, 0) * 2);
                            float v0 = acc[m][n][2 * h];
                            float v1 = acc[m][n][2 * h + 1];
                            if (p.add_inputs) {
                                const uint32_t old = *cell;
                                v0 += bf16_lo(old);
                                v1 += bf16_hi(old);
                            }
                            *cell = pack_bf16x2(v0, v1);
                        }
                __syncthreads();
                if (ycc * 8 < ncols) {
#pragma unroll
                    for (int j = 0; j < Cfg::Y_PASSES; ++j) {
                        if (ytok[j] < 0) continue;
                        const uint4 v = *reinterpret_cast<const uint4 *>(
                            sy + y_soff + j * Cfg::Y_RPP * Cfg::Y_LD);
                        *reinterpret_cast<uint4 *>(ybase + (int64_t(ytok[j]) * p.y_ld + c0)) = v;
                    }
                }
            } else {
#pragma unroll
                for (int m = 0; m < MI; ++m)
#pragma unroll
                    for (int n = 0; n < NI; ++n)
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int r = wm * Cfg::WM + m * 16 + (lane >> 2) + 8 * (q >> 1);
                            const int c = out_col(n, q & 1);
                            const int tok = s_tok[r];
                            if (tok < 0 || c >= ncols) continue;
                            uint16_t *dst = yslice + int64_t(tok) * p.y_ld + c0 + c;
                            float v = acc[m][n][q];
                            if (p.add_inputs) v += bf16_to_f32(*dst);
                            *dst = static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu);
                        }
            }
        }
        cp_async_wait<0>();
        __syncthreads();
    }
}

}  // namespace lora
