// lora_common.cuh -- device helpers shared by the metadata, shrink and
// expand kernels: inline-PTX wrappers (cp.async, ldmatrix, mma.sync), the
// shared-memory swizzle, and the segment -> tile schedule that both GEMM
// kernels walk.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "lora_punica.h"

#define LORA_API extern "C" __attribute__((visibility("default")))

namespace lora {

// ------------------------------------------------------------------ PTX

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy, cached in L2 only.  When `valid` is false
// nothing is read and the 16 destination bytes are zero-filled; `src` must
// still be a mapped address, so callers pass a known-good base pointer.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid)
{
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n"
                 :: "r"(dst), "l"(src), "r"(n) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" :: "n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                            uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t v) { return __uint_as_float(uint32_t(v) << 16); }

// ------------------------------------------------------------ swizzle
//
// A K-contiguous bf16 tile is stored as rows of CPR 16-byte chunks.  ldmatrix
// reads one 16-byte chunk from each of 8 consecutive rows; the XOR below
// spreads those 8 chunks over all 32 banks for every CPR used here (2, 4, 8,
// 16), which makes both the cp.async writes and the ldmatrix reads
// conflict-free.
template <int CPR>
__device__ __forceinline__ uint32_t swz(int row, int chunk)
{
    static_assert(CPR == 2 || CPR == 4 || CPR >= 8, "chunks per row");
    int phys;
    if constexpr (CPR >= 8) {
        phys = (chunk & ~7) | ((chunk ^ row) & 7);
    } else {
        constexpr int SHIFT = (CPR == 4) ? 1 : 2;      // rows that share a bank line
        phys = chunk ^ ((row >> SHIFT) & (CPR - 1));
    }
    return static_cast<uint32_t>(row * CPR * 16 + phys * 16);
}

// Programmatic dependent launch.  Every kernel waits for the grids it
// depends on before its first global read, then lets the next kernel in the
// stream begin its launch (which overlaps that kernel's launch latency with
// this kernel's work).  Both are no-ops when the launch carried no
// programmatic dependency.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// ------------------------------------------------------- debug checks
//
// A build with LORA_PUNICA_DEBUG_CHECKS defined checks every LoRA id, token
// index and segment bound a kernel takes from the metadata before it
// indexes x, y, A, B or the buffer with it.  A value out of range sets bit
// 29 of the metadata error word and the access is skipped (the token or
// segment is treated as having no LoRA); nothing traps.  The normal build
// compiles the checks away.
#ifdef LORA_PUNICA_DEBUG_CHECKS
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif
constexpr int LORA_DEBUG_BIT = 1 << 29;

__device__ __forceinline__ void debug_flag(int32_t *err)
{
    if (err != nullptr) atomicOr(err, LORA_DEBUG_BIT);
}

// A token index read from the sorted list: itself, or -1 (no LoRA) when a
// debug build finds it outside [0, T).
__device__ __forceinline__ int checked_token(int tok, int T, int32_t *err)
{
    if constexpr (kDebugChecks) {
        if (tok >= T || tok < -1) {
            debug_flag(err);
            return -1;
        }
    }
    return tok;
}

// ----------------------------------------------------------- schedule
//
// Segment table held in shared memory (4 * nbins + 2 ints):
//   tile[k]  (k <= nbins)  tiles in segments before k (tile[nbins] = total)
//   id[k], start[k], count[k]  copies of active_lora_ids, lora_token_start_loc
//                              and num_tokens_per_lora
struct SegTab {
    int *tile, *id, *start, *count;
};

__device__ __forceinline__ SegTab seg_tab(int *base, int nbins)
{
    SegTab t;
    t.tile = base;
    t.id = base + nbins + 1;
    t.start = t.id + nbins;
    t.count = t.start + nbins;
    return t;
}

__host__ __device__ constexpr size_t seg_tab_bytes(int nbins)
{
    return size_t(4 * nbins + 2) * sizeof(int);
}

// Reads the no-LoRA flag and the whole segment table with one round of
// independent loads, then scans tile counts.  Returns 0 (no work) when the
// flag is set; otherwise the total number of tiles of `tile_rows` tokens.
// Every thread of the block gets the result.
//   full_tiles_only: each segment contributes only its whole tiles
//                    (count / tile_rows of them).
//   skip_rows:       when nonzero, the first (count / skip_rows) * skip_rows
//                    tokens of every segment are left out (another kernel
//                    covers them) and only the rest is tiled.
//   num_tokens, err: a debug build drops (and reports in err) segments
//                    whose id is outside [-1, nbins - 1) or whose tokens
//                    leave [0, num_tokens).
__device__ __forceinline__ int load_segments(const int32_t *no_lora, const int32_t *active,
                                             const int32_t *counts, const int32_t *start_loc,
                                             int nbins, int tile_rows, SegTab t,
                                             bool full_tiles_only = false, int skip_rows = 0,
                                             int num_tokens = 0, int32_t *err = nullptr)
{
    int *s_flag = t.count + nbins;
    for (int k = threadIdx.x; k < nbins; k += blockDim.x) {
        int id = active[k];
        int c = counts[k];
        int st = start_loc[k];
        if constexpr (kDebugChecks) {
            if (id < -1 || id >= nbins - 1 ||
                (id >= 0 && c > 0 && (st < 0 || c > num_tokens || st > num_tokens - c))) {
                debug_flag(err);
                id = -1;
                c = 0;
            }
        }
        if (skip_rows > 0) {
            const int skip = (c / skip_rows) * skip_rows;
            st += skip;
            c -= skip;
        }
        if (full_tiles_only) c = (c / tile_rows) * tile_rows;
        t.id[k] = id;
        t.count[k] = c;
        t.start[k] = st;
    }
    if (threadIdx.x == 0) *s_flag = *no_lora;
    __syncthreads();
    if (*s_flag) return 0;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int carry = 0;
        for (int b0 = 0; b0 < nbins; b0 += 32) {
            const int k = b0 + lane;
            int n = 0;
            if (k < nbins) {
                const int c = t.count[k];
                n = (t.id[k] >= 0 && c > 0) ? (c + tile_rows - 1) / tile_rows : 0;
            }
            int v = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (k < nbins) t.tile[k] = carry + v - n;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) t.tile[nbins] = carry;
    }
    __syncthreads();
    return t.tile[nbins];
}

// Per bin b: the exclusive scan of cnt[w * nb + b] over the W warps (warp
// order is token order), in place, and tot[b] = the bin's total (plus
// bef[b] + aft[b] when given: tokens counted outside the warps' run).
// With 32 warps, three threads share a bin, each summing 11 warps' counts
// with independent loads and taking the others' sums by shuffle, instead
// of one thread walking all 32 (a chain of dependent loads).  Banks: word
// w * nb + b with nb = L + 1; with three threads per bin the lanes' words
// differ mod 32 when nb = 257 (11 j + g for j < 3, g < 10).
template <int NT, int W>
__device__ __forceinline__ void scan_bins_over_warps(int32_t *cnt, int32_t *tot,
                                                     const int32_t *bef, const int32_t *aft,
                                                     int nb)
{
    constexpr int Q = W >= 24 ? 3 : 1;          // threads per bin
    constexpr int SPAN = (W + Q - 1) / Q;       // warps per thread
    constexpr int G = 32 / Q;                   // bins per warp and pass
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane / Q, j = lane - g * Q;
    for (int b0 = warp * G; b0 < nb; b0 += (NT / 32) * G) {   // the same in every lane
        const int b = b0 + g;
        const bool act = g < G && b < nb;
        int c[SPAN];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < SPAN; ++i) {
            const int w = j * SPAN + i;
            c[i] = (act && w < W) ? cnt[w * nb + b] : 0;
            sum += c[i];
        }
        int run = 0;                            // sums of the bin's earlier threads
#pragma unroll
        for (int d = 1; d < Q; ++d) {
            const int u = __shfl_up_sync(0xffffffffu, sum, d);
            if (j >= d) run += u;
        }
#pragma unroll
        for (int i = 0; i < SPAN; ++i) {
            const int w = j * SPAN + i;
            if (act && w < W) cnt[w * nb + b] = run;
            run += c[i];
        }
        if (act && j == Q - 1) tot[b] = run + (bef != nullptr ? bef[b] + aft[b] : 0);
    }
}

// Exclusive scans over the bins of tot: base[b] = tokens in bins before b,
// pos[b] = non-empty bins before b (the torch.unique(sorted=True) order),
// *nactive = non-empty bins.  One warp per 32 bins: each first sums every
// earlier bin itself (up to eight independent loads a lane and one warp
// reduction), then scans its own 32; no warp waits for another.  Token
// counts and non-empty flags travel packed in one 64-bit value.
template <int NT>
__device__ __forceinline__ void scan_over_bins(const int32_t *tot, int32_t *base, int32_t *pos,
                                               int32_t *nactive, int nb)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nchunk = (nb + 31) >> 5;
    auto pack = [](int32_t v) {
        return uint64_t(uint32_t(v)) | (uint64_t(v > 0 ? 1u : 0u) << 32);
    };
    for (int c = warp; c < nchunk; c += NT / 32) {
        uint64_t before = 0;
        for (int k = 0; k < c; ++k) before += pack(tot[k * 32 + lane]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
        const int b = c * 32 + lane;
        const uint64_t pv = b < nb ? pack(tot[b]) : 0ull;
        uint64_t incl = pv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        const uint64_t excl = before + incl - pv;
        if (b < nb) {
            base[b] = int32_t(uint32_t(excl));
            pos[b] = int32_t(excl >> 32);
        }
        if (c == nchunk - 1 && lane == 31) *nactive = int32_t((before + incl) >> 32);
    }
}

// Stable counting sort of a small batch's LoRA ids inside one CTA of NW
// warps (the metadata step of LoRAKernelMeta.prepare_tensors, computed in
// shared memory).  Bin 0 holds id -1 and invalid ids, bin b holds id b - 1.
// Shared arrays: cnt[NW * nbins], tot[nbins], base[nbins], pos[nbins],
// srt[T] (the permutation), misc[2] (invalid ids, number of non-empty bins).
// Each warp owns a contiguous run of tokens, so warp order, group order and
// lane order together give token order inside every bin.  Returns the
// no-LoRA flag to every thread; srt is only filled when it is false.
//
// The id map is first copied into shared memory (ids[T], one round of
// independent global loads), so both passes read shared memory.
template <int NW>
__device__ __forceinline__ bool block_sort_ids(const int32_t *map_g, int T, int max_loras,
                                               int *cnt, int *tot, int *base, int *pos,
                                               int *srt, int *misc, int *ids)
{
    const int nbins = max_loras + 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int t = tid; t < T; t += NW * 32) ids[t] = map_g[t];
    for (int i = tid; i < NW * nbins; i += NW * 32) cnt[i] = 0;
    if (tid == 0) misc[0] = 0;
    __syncthreads();
    const int32_t *map = ids;
    const int per_warp = ((T + NW * 32 - 1) / (NW * 32)) * 32;
    const int t0 = min(T, warp * per_warp), t1 = min(T, t0 + per_warp);
    int bad = 0;
    for (int g = t0; g < t1; g += 32) {
        const int t = g + lane;
        const bool has = t < t1;
        int b = -1;
        if (has) {
            const int32_t id = map[t];
            if (id >= 0 && id < max_loras) b = id + 1;
            else { b = 0; if (id != -1) ++bad; }
        }
        if (has) atomicAdd(&cnt[warp * nbins + b], 1);          // counts only
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if (lane == 0 && bad) atomicAdd(&misc[0], bad);
    __syncthreads();
    scan_bins_over_warps<NW * 32, NW>(cnt, tot, nullptr, nullptr, nbins);
    __syncthreads();
    scan_over_bins<NW * 32>(tot, base, pos, &misc[1], nbins);
    __syncthreads();
    const bool no_lora = (tot[0] == T);
    if (!no_lora) {
        for (int g = t0; g < t1; g += 32) {
            const int t = g + lane;
            const bool has = t < t1;
            int b = -1;
            if (has) {
                const int32_t id = map[t];
                b = (id >= 0 && id < max_loras) ? id + 1 : 0;
            }
            const unsigned grp = __match_any_sync(0xffffffffu, b);
            const int rk = __popc(grp & ((1u << lane) - 1u));
            if (has) srt[base[b] + cnt[warp * nbins + b] + rk] = t;
            __syncwarp();
            if (has && rk == 0) cnt[warp * nbins + b] += __popc(grp);
            __syncwarp();
        }
    }
    __syncthreads();
    return no_lora;
}

// Writes the metadata buffers from a block_sort_ids result (one CTA calls it).
__device__ __forceinline__ void write_meta(const int32_t *map, int T, int max_loras, bool no_lora,
                                           const int *tot, const int *base, const int *pos,
                                           const int *srt, const int *misc,
                                           int32_t *mapping_copy, int32_t *sorted, int32_t *counts,
                                           int32_t *start_loc, int32_t *active, int32_t *flag,
                                           int32_t *error_word)
{
    const int nbins = max_loras + 1;
    const int nact = no_lora ? 0 : misc[1];
    for (int k = threadIdx.x; k < nbins; k += blockDim.x)
        if (k >= nact) { active[k] = -1; counts[k] = 0; start_loc[k + 1] = 0; }
    if (threadIdx.x == 0) {
        start_loc[0] = 0;
        *flag = no_lora ? 1 : 0;
        *error_word = misc[0];
    }
    if (no_lora) return;
    for (int b = threadIdx.x; b < nbins; b += blockDim.x) {
        const int c = tot[b];
        if (c > 0) {
            const int k = pos[b];
            active[k] = b - 1;
            counts[k] = c;
            start_loc[k + 1] = base[b] + c;
        }
    }
    for (int t = threadIdx.x; t < T; t += blockDim.x) {
        sorted[t] = srt[t];
        mapping_copy[t] = map[t];
    }
}

// Fills a segment table from a block_sort_ids result (segment k = bin k)
// and scans it into tiles of `tile_rows`; returns the total tile count.
__device__ __forceinline__ int segments_from_sort(const int *tot, const int *base, int nbins,
                                                  int tile_rows, SegTab t)
{
    for (int k = threadIdx.x; k < nbins; k += blockDim.x) {
        t.id[k] = (k >= 1 && tot[k] > 0) ? k - 1 : -1;
        t.count[k] = tot[k];
        t.start[k] = base[k];
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int carry = 0;
        for (int b0 = 0; b0 < nbins; b0 += 32) {
            const int k = b0 + lane;
            int n = 0;
            if (k < nbins) {
                const int c = t.count[k];
                n = (t.id[k] >= 0 && c > 0) ? (c + tile_rows - 1) / tile_rows : 0;
            }
            int v = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (k < nbins) t.tile[k] = carry + v - n;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) t.tile[nbins] = carry;
    }
    __syncthreads();
    return t.tile[nbins];
}

// Segment that holds global tile `tile`: the last k with s_tile[k] <= tile.
// Segments with no tiles (id -1, or no tokens) share their successor's
// prefix value and are skipped by the search.
__device__ __forceinline__ int find_segment(const int *s_tile, int nbins, int tile)
{
    int lo = 0, hi = nbins;          // answer in [lo, hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_tile[mid] <= tile) lo = mid; else hi = mid;
    }
    return lo;
}

}  // namespace lora

// Host-side launch helpers (lora_api.cu).
namespace lora {
int device_sm_count();

// Tuning knobs: the LORA_PUNICA_* environment variables, read once (at the
// first library call) into this process-wide struct; lora_reload_options()
// reads them again.  No call reads the environment after that.
struct Knobs {
    int pdl;                  // LORA_PUNICA_PDL: programmatic dependent launch (1)
    int coop;                 // LORA_PUNICA_COOP: single cooperative kernel (-1 auto, 0, 1)
    int fused;                // LORA_PUNICA_FUSED: cluster kernel (-1 auto, 0, 1)
    int fused_max_tokens;     // LORA_PUNICA_FUSED_MAX_TOKENS (128)
    int self_meta;            // LORA_PUNICA_SELF_META (-1 early mode, 0 three calls, 1 two kernels)
    int umma;                 // LORA_PUNICA_UMMA: tcgen05 shrink (1)
    int umma_min_tokens;      // LORA_PUNICA_UMMA_MIN_TOKENS (1024)
    int umma_min_cols;        // LORA_PUNICA_UMMA_MIN_COLS (256)
    int umma_partial;         // LORA_PUNICA_UMMA_PARTIAL (1)
    int umma_pair;            // LORA_PUNICA_UMMA_PAIR: CTA-pair (M = 256) tensor-core shrink
    int nvtx;                 // LORA_PUNICA_NVTX: NVTX ranges around the C-ABI calls (1)
    int early_shrink_ctas;    // LORA_PUNICA_EARLY_SHRINK_CTAS (2)
    int expand_tc;            // LORA_PUNICA_EXPAND_TC: tcgen05 expand (0 off, -1 ranks >= min, 1 where it fits, 2 required)
    int expand_tc_min_rank;   // LORA_PUNICA_EXPAND_TC_MIN_RANK (64)
    int meta_small;           // LORA_PUNICA_META_SMALL (1)
    int meta_multi;           // LORA_PUNICA_META_MULTI: multi-CTA metadata kernel (1)
    int meta_cluster;         // LORA_PUNICA_META_CLUSTER: its thread-block-cluster form (1)
    int linear_tc;            // LORA_PUNICA_LINEAR_TC: lora_linear's one-kernel tensor-core path (-1)
    int linear_tc_min_tokens; // LORA_PUNICA_LINEAR_TC_MIN_TOKENS: its batch threshold (0: 72 x SMs)
    int coop_test_extra;      // LORA_PUNICA_COOP_TEST_EXTRA_ARRIVALS (0, tests only)
    int coop_test_timeout;    // LORA_PUNICA_COOP_TEST_TIMEOUT_CYCLES (0, tests only)
};
const Knobs &knobs();
inline bool pdl_enabled() { return knobs().pdl != 0; }
inline int knob_expand_tc() { return knobs().expand_tc; }

// An NVTX range around one C-ABI call, so that a profiler's timeline shows
// the library's calls (LORA_PUNICA_NVTX=0 turns them off; without a tool
// attached a push and a pop cost a few nanoseconds).
struct NvtxRange {
    bool on;
    explicit NvtxRange(const char *name) : on(knobs().nvtx != 0)
    {
        if (on) nvtxRangePushA(name);
    }
    ~NvtxRange()
    {
        if (on) nvtxRangePop();
    }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
inline int knob_expand_tc_min_rank() { return knobs().expand_tc_min_rank; }

// Host-side description of one lora_shrink call, shared by its two paths.
struct ShrinkLaunch {
    const uint16_t *x;
    int64_t x_ld;
    int32_t hidden;
    int32_t num_tokens;
    const uint16_t *a[LORA_MAX_SLICES];
    int32_t num_slices;
    int32_t rank;
    int32_t max_loras;
    float *y;
    float scale;
    const int32_t *sorted;
    const int32_t *counts;
    const int32_t *start_loc;
    const int32_t *active;
    const int32_t *no_lora;
    int32_t *error_word;
    int32_t partial;      // the tensor-core path takes partial tiles too
};
int launch_shrink_umma(const ShrinkLaunch &a, cudaStream_t stream);
int launch_shrink_pair(const ShrinkLaunch &a, cudaStream_t stream);
int shrink_self_meta(const int32_t *map, const lora_bf16_t *x, int32_t num_tokens,
                     int32_t hidden, int64_t x_ld, const lora_bf16_t *const *lora_a,
                     int32_t num_slices, int32_t rank, float *y, const lora_meta_t *meta,
                     float scale, cudaStream_t st, int early);
int expand_early(const float *x, const lora_bf16_t *const *lora_b,
                 const lora_bf16_t *const *lora_bias, const int32_t *slice_sizes,
                 int32_t num_slices, int32_t rank, lora_bf16_t *y, int64_t y_ld,
                 int32_t num_tokens, const lora_meta_t *meta, cudaStream_t st);
// lora_linear as one cooperative kernel (small batches).  Returns 1 when
// launched, 0 when the batch or its layout does not fit that path.
int linear_coop(const int32_t *map, int32_t num_tokens, const lora_bf16_t *x, int32_t hidden,
                int64_t x_ld, const lora_bf16_t *const *lora_a,
                const lora_bf16_t *const *lora_b, const lora_bf16_t *const *lora_bias,
                const int32_t *slice_sizes, int32_t num_slices, int32_t rank, float scale,
                float *buf, lora_bf16_t *y, int64_t y_ld, const lora_meta_t *meta,
                cudaStream_t st);

// Host-side description of one lora_expand call for its tensor-core path.
struct ExpandLaunch {
    const void *x;                 // fp32, or bf16 when x_bf16
    int32_t x_bf16;
    int32_t early;                 // lora_linear's early mode
    const uint16_t *b[LORA_MAX_SLICES];
    const uint16_t *bias[LORA_MAX_SLICES];
    int32_t n[LORA_MAX_SLICES];
    int32_t col0[LORA_MAX_SLICES];
    int32_t num_slices;
    int32_t rank;
    int32_t max_loras;
    uint16_t *y;
    int64_t y_ld;
    int32_t num_tokens;
    int32_t add_inputs;
    int32_t vec;
    int32_t bias_vec;
    const int32_t *sorted;
    const int32_t *counts;
    const int32_t *start_loc;
    const int32_t *active;
    const int32_t *no_lora;
    int32_t *error_word;
};
// The shrink and expand of one lora_linear call in one tensor-core kernel
// (lora_linear_tc.cu): rank 128, up to three slices.  linear_tc_fits says
// whether a call fits it; launch_linear_tc returns 0 when launched or a
// cudaError_t.
struct LinearTcLaunch {
    const uint16_t *x;
    int64_t x_ld;
    int32_t hidden;
    int32_t num_tokens;
    const uint16_t *a[LORA_MAX_SLICES];
    const uint16_t *b[LORA_MAX_SLICES];
    const uint16_t *bias[LORA_MAX_SLICES];
    int32_t n[LORA_MAX_SLICES];
    int32_t num_slices;
    int32_t rank;
    int32_t max_loras;
    float scale;
    float *buf;
    uint16_t *y;
    int64_t y_ld;
    const int32_t *sorted;
    const int32_t *counts;
    const int32_t *start_loc;
    const int32_t *active;
    const int32_t *no_lora;
    int32_t *error_word;
};
bool linear_tc_fits(const LinearTcLaunch &a);
int launch_linear_tc(const LinearTcLaunch &a, cudaStream_t stream);

// launch_expand_tc's results besides a cudaError_t (positive).
enum : int { TC_LAUNCHED = 0, TC_NO_FIT = -1, TC_MISALIGNED = -2 };
int launch_expand_tc(const ExpandLaunch &a, cudaStream_t stream);

// Launch with the programmatic-stream-serialization attribute (when
// enabled), so the kernel may start while its predecessor drains; the
// kernel itself calls pdl_wait() before touching memory.
template <typename Kern, typename Arg>
cudaError_t launch_kernel(Kern kernel, dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, const Arg &arg)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, arg);
}
}
