// lora_linear_coop.cu -- lora_linear for small batches as one cooperative
// kernel: metadata, shrink and expand with fused bias in a single launch
// (page "vllm.lora.ops.triton_ops.lora_kernel_metadata",
// LoRAKernelMeta.prepare_tensors; page "vllm.lora.punica_wrapper.punica_gpu",
// PunicaWrapperGPU.add_lora_linear = add_shrink into an fp32 buffer, then
// add_expand).
//
// A small batch is a chain of short dependent phases: every extra launch and
// every re-read of the metadata costs more than the bytes it moves.  Here one
// persistent grid, every CTA resident (a cooperative launch guarantees it),
// runs the whole chain:
//   1. every CTA sorts the batch's ids in shared memory (the stable counting
//      sort of the metadata kernel); CTA 0 also writes the metadata buffers;
//   2. shrink: (64-token tile, slice, hidden chunk) items spread over all
//      CTAs; mma.sync with the r rows of A as M and the tile's tokens as N,
//      through a 4-stage cp.async ring; the partial sums are added into the
//      fp32 buffer with float4 reductions (red.global.add, also when the
//      hidden dimension is not split: no load latency);
//   3. each CTA announces its arrival at a grid-wide barrier, starts the
//      copies of y, B and bias for its first expand chunks, then waits for
//      every other arrival;
//   4. the expand items of the expand kernel, reading the finished buffer.
// The barrier uses two counters of the caller's metadata (arrivals, exits):
// CTAs poll the arrival count, and the last CTA to leave the kernel puts
// both back to zero, so they are zero whenever the kernel is not running,
// on every path.  A poll gives up after a bounded time: it sets bit 30 of
// the metadata error word and the CTA skips its expand work.
#include "lora_expand.cuh"

namespace lora {

constexpr int CO_THREADS = EX_THREADS;      // 8 warps: the expand's tile layout
constexpr int CO_BN = EX_BM;                // shrink tokens per item (64)
constexpr int CO_BK = 64;                   // hidden per stage (128-byte rows)
constexpr int CO_STAGES = 4;                // shrink pipeline depth (hidden blocks)
constexpr int CO_MIN_STEPS = 2;             // shortest hidden chunk, in blocks
constexpr int CO_MAX_TOKENS = 512;
constexpr int CO_MAX_LORAS = 256;
constexpr int CO_MAX_MT = 4;                // rank <= 64
constexpr long long CO_TIMEOUT_CYCLES = 2000000000ll;   // about one second
constexpr int CO_ERROR_BIT = 1 << 30;

struct CoopArgs {
    ExpandArgs ex;                  // the expand part: x = buf, add_inputs = 1
    const int32_t *map;
    const uint16_t *x;
    int64_t x_ld;
    int32_t hidden;
    const uint16_t *a[LORA_MAX_SLICES];
    float scale;
    float *buf;
    int32_t *mapping_copy, *sorted, *counts, *start_loc, *active, *no_lora, *error_word;
    uint32_t *sync;                 // [0] arrivals at the barrier, [1] exits
    uint32_t expect;                // arrivals that open the barrier (= grid size)
    long long timeout;              // poll limit, clock cycles
};

template <int MT>
struct CoopTile {
    static constexpr int RP = 16 * MT;
    static constexpr int A_BYTES = RP * CO_BK * 2;
    static constexpr int X_BYTES = CO_BN * CO_BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + X_BYTES;
    static constexpr int SHRINK_BYTES = CO_STAGES * STAGE_BYTES;
    static constexpr int OUT_LD = RP + 4;                   // fp32 staging row
    static constexpr int EXPAND_BYTES =
        EX_STAGES * ExpandTile<MT>::STAGE_BYTES + ExpandTile<MT>::A_BYTES;
    // the shrink ring and its staging reuse the expand's ring
    static constexpr int RING_BYTES = SHRINK_BYTES > EXPAND_BYTES ? SHRINK_BYTES : EXPAND_BYTES;
    static_assert(CO_BN * OUT_LD * 4 <= SHRINK_BYTES, "staging fits in the shrink ring");
    static_assert(RING_BYTES % 16 == 0, "int region alignment");
};

// Shared memory of the metadata part (segment table + sort arrays), ints.
__host__ __device__ constexpr int coop_int_words(int nbins)
{
    return (4 * nbins + 2) + 8 * nbins + 3 * nbins + 2 * CO_MAX_TOKENS + 2;
}

inline size_t coop_smem_bytes(int mt, int nbins)
{
    int ring = 0;
    switch (mt) {
    case 1: ring = CoopTile<1>::RING_BYTES; break;
    case 2: ring = CoopTile<2>::RING_BYTES; break;
    default: ring = CoopTile<4>::RING_BYTES; break;
    }
    return size_t(ring) + size_t(coop_int_words(nbins)) * sizeof(int);
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t &r0, uint32_t &r1)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];\n"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *a)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(a) : "memory");
    return v;
}

// Grid barrier in two halves.  Arrival (after the CTA's shrink, before it
// issues any expand copy, so the fence waits only for the shrink's buffer
// updates): every thread, then one fence and one increment.
__device__ __forceinline__ void coop_arrive(const CoopArgs &p)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(&p.sync[0], 1u);
    }
}

// Wait (right before the first read of the buffer): polls the arrival count
// with a time limit.  Returns false when it ran out (bit 30 of the error
// word is then set).
__device__ __forceinline__ bool coop_wait(const CoopArgs &p)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        const long long t0 = clock64();
        while (ld_acquire_u32(&p.sync[0]) < p.expect) {
            if (clock64() - t0 > p.timeout) {
                ok = 0;
                atomicOr(p.error_word, CO_ERROR_BIT);
                break;
            }
            __nanosleep(64);
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// Every CTA that passed the sort calls this last: the final one resets both
// counters (no CTA polls any more at that point).
__device__ __forceinline__ void coop_exit(const CoopArgs &p)
{
    __syncthreads();
    if (threadIdx.x == 0 && atomicAdd(&p.sync[1], 1u) == gridDim.x - 1) {
        atomicExch(&p.sync[0], 0u);
        atomicExch(&p.sync[1], 0u);
    }
}

// Shrink items of this CTA: buf[s][t, :] += scale * x[t, :] @ A[s][id]^T
// over one hidden chunk of one 64-token tile.
template <int MT>
__device__ __forceinline__ void coop_shrink(const CoopArgs &p, SegTab tab, const int *tokens, int total_tiles, uint8_t *smem, int *s_tok) {
    using Cfg = CoopTile<MT>; constexpr int RP = Cfg::RP;
    constexpr int A_PASSES = (RP * 8 + CO_THREADS - 1) / CO_THREADS;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = p.ex.num_slices, H = p.hidden, T = p.ex.num_tokens, R = p.ex.rank, nbins = p.ex.nbins;
    const int nk = (H + CO_BK - 1) / CO_BK;
    const int pairs = total_tiles * S; int kchunks = 1;
    if (pairs < int(gridDim.x)) kchunks = max(1, min(int(gridDim.x) / pairs, max(1, nk / CO_MIN_STEPS)));
    const int spc = (nk + kchunks - 1) / kchunks; kchunks = (nk + spc - 1) / spc;
    const int total_items = pairs * kchunks;
    const uint32_t ring = smem_addr(smem); const int xc = tid & 7, xr = tid >> 3;
    for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
        const int s = item % S, rest = item / S, tile = rest % total_tiles, kc = rest / total_tiles;
        const int seg = find_segment(tab.tile, nbins, tile); const int id = tab.id[seg];
        const int row0 = tab.start[seg] + (tile - tab.tile[seg]) * CO_BN;
        const int nrows = min(CO_BN, tab.start[seg] + tab.count[seg] - row0);
        __syncthreads(); if (tid < CO_BN) s_tok[tid] = (tid < nrows) ? tokens[row0 + tid] : -1; __syncthreads();
        const int k_first = kc * spc, k_steps = min(spc, nk - k_first);
        const uint16_t *xrow[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) { const int t = s_tok[xr + 32 * j]; xrow[j] = (t >= 0) ? p.x + int64_t(t) * p.x_ld : nullptr; }
        const uint16_t *abase = p.a[s] + int64_t(id) * R * H;
        auto load_stage = [&](int kstep, int slot) {
            const uint32_t sa = ring + slot * Cfg::STAGE_BYTES, sx = sa + Cfg::A_BYTES;
            const int k0 = kstep * CO_BK + xc * 8; const bool kin = k0 < H;
#pragma unroll
            for (int j = 0; j < 2; ++j) { const bool ok = kin && xrow[j] != nullptr; cp_async16(sx + swz<8>(xr + 32 * j, xc), ok ? xrow[j] + k0 : p.x, ok); }
#pragma unroll
            for (int j = 0; j < A_PASSES; ++j) { const int r = xr + 32 * j; if (r < RP) { const bool ok = kin && r < R; cp_async16(sa + swz<8>(r, xc), ok ? abase + int64_t(r) * H + k0 : p.x, ok); } }
        };
        float acc[MT][4];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[m][q] = 0.f;
#pragma unroll
        for (int st = 0; st < CO_STAGES - 1; ++st) { if (st < k_steps) load_stage(k_first + st, st); cp_async_commit(); }
        for (int ks = 0; ks < k_steps; ++ks) {
            cp_async_wait<CO_STAGES - 2>(); __syncthreads();
            { const int nxt = ks + CO_STAGES - 1; if (nxt < k_steps) load_stage(k_first + nxt, nxt % CO_STAGES); cp_async_commit(); }
            const uint32_t sa = ring + (ks % CO_STAGES) * Cfg::STAGE_BYTES, sx = sa + Cfg::A_BYTES;
#pragma unroll
            for (int kk = 0; kk < CO_BK / 16; ++kk) {
                uint32_t b0, b1; ldmatrix_x2(sx + swz<8>(warp * 8 + (lane & 7), kk * 2 + ((lane >> 3) & 1)), b0, b1);
#pragma unroll
                for (int m = 0; m < MT; ++m) { uint32_t af[4]; ldmatrix_x4(sa + swz<8>(m * 16 + (lane & 15), kk * 2 + (lane >> 4)), af[0], af[1], af[2], af[3]); mma_bf16_16816(acc[m], af, b0, b1); }
            }
        }
        cp_async_wait<0>(); __syncthreads();
        float *stage = reinterpret_cast<float *>(smem);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const int r = m * 16 + (lane >> 2), t = warp * 8 + 2 * (lane & 3);
            stage[t * Cfg::OUT_LD + r] = acc[m][0] * p.scale; stage[(t + 1) * Cfg::OUT_LD + r] = acc[m][1] * p.scale;
            stage[t * Cfg::OUT_LD + r + 8] = acc[m][2] * p.scale; stage[(t + 1) * Cfg::OUT_LD + r + 8] = acc[m][3] * p.scale;
        }
        __syncthreads();
        const int r4n = R / 4;
        for (int i = tid; i < CO_BN * r4n; i += CO_THREADS) {
            const int t = i / r4n, c4 = i - t * r4n; const int tok = s_tok[t]; if (tok < 0) continue;
            const float4 v = *reinterpret_cast<const float4 *>(&stage[t * Cfg::OUT_LD + 4 * c4]);
            float4 *dst = reinterpret_cast<float4 *>(p.buf + (int64_t(s) * T + tok) * R) + c4;
            atomicAdd(dst, v);                // a reduction: no load latency
        }
    }
    __syncthreads();
}
template <int MT>
__global__ void __launch_bounds__(CO_THREADS, 2) linear_coop_kernel(CoopArgs p)
{
    using Cfg = CoopTile<MT>;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_tok[CO_BN];
    const int nbins = p.ex.nbins, T = p.ex.num_tokens;

    int *ib = reinterpret_cast<int *>(smem + Cfg::RING_BYTES);
    const SegTab tab = seg_tab(ib, nbins);
    int *cnt = ib + 4 * nbins + 2, *tot = cnt + 8 * nbins, *base = tot + nbins;
    int *pos = base + nbins, *srt = pos + nbins, *ids = srt + CO_MAX_TOKENS;
    int *misc = ids + CO_MAX_TOKENS;
    const bool nl = block_sort_ids<CO_THREADS / 32>(p.map, T, nbins - 1, cnt, tot, base, pos,
                                                    srt, misc, ids);
    if (blockIdx.x == 0)
        write_meta(ids, T, nbins - 1, nl, tot, base, pos, srt, misc, p.mapping_copy, p.sorted,
                   p.counts, p.start_loc, p.active, p.no_lora, p.error_word);
    if (nl) return;                               // every CTA sees the same map
    const int total_tiles = segments_from_sort(tot, base, nbins, CO_BN, tab);

    coop_shrink<MT>(p, tab, srt, total_tiles, smem, s_tok);
    coop_arrive(p);
    expand_items<MT>(p.ex, tab, srt, total_tiles, smem, s_tok, [&]() { return coop_wait(p); });
    coop_exit(p);
}

// Returns 1 when launched, 0 when the batch does not fit this path (the
// caller takes another), a status otherwise.
int launch_linear_coop(CoopArgs &p, cudaStream_t st)
{
    const int R = p.ex.rank;
    const int mt = (R <= 16) ? 1 : (R <= 32) ? 2 : 4;
    if (R > 16 * CO_MAX_MT || p.ex.num_tokens > CO_MAX_TOKENS || p.ex.nbins - 1 > CO_MAX_LORAS)
        return 0;
    static int grid_cache[64][3] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return int(e);
    if (dev >= 64) return 0;
    const int ti = (mt == 1) ? 0 : (mt == 2) ? 1 : 2;
    const size_t smem = coop_smem_bytes(mt, CO_MAX_LORAS + 1);
    auto kern = (mt == 1) ? linear_coop_kernel<1> : (mt == 2) ? linear_coop_kernel<2>
                                                              : linear_coop_kernel<4>;
    int grid = grid_cache[dev][ti];
    if (grid == 0) {
        int coop = 0;
        e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
        if (e != cudaSuccess) return int(e);
        if (!coop) {
            grid_cache[dev][ti] = -1;
            return 0;
        }
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return int(e);
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, CO_THREADS, smem);
        if (e != cudaSuccess) return int(e);
        grid = (occ >= 1) ? device_sm_count() * min(occ, 2) : -1;
        grid_cache[dev][ti] = grid;
    }
    if (grid < 0) return 0;
    p.expect = uint32_t(grid) + uint32_t(max(0, knobs().coop_test_extra));
    const long long tmo = knobs().coop_test_timeout;
    p.timeout = (tmo > 0) ? tmo : CO_TIMEOUT_CYCLES;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(CO_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    return e == cudaSuccess ? 1 : int(e);
}

int linear_coop(const int32_t *map, int32_t num_tokens, const lora_bf16_t *x, int32_t hidden,
                int64_t x_ld, const lora_bf16_t *const *lora_a,
                const lora_bf16_t *const *lora_b, const lora_bf16_t *const *lora_bias,
                const int32_t *slice_sizes, int32_t num_slices, int32_t rank, float scale,
                float *buf, lora_bf16_t *y, int64_t y_ld, const lora_meta_t *meta,
                cudaStream_t st)
{
    if (meta->grid_sync == nullptr || meta->token_lora_mapping == nullptr ||
        meta->error_word == nullptr || map == nullptr || num_tokens < 1 ||
        num_tokens > CO_MAX_TOKENS || meta->max_loras > CO_MAX_LORAS || rank > 16 * CO_MAX_MT)
        return 0;
    if (x == nullptr || buf == nullptr || hidden < 1 || hidden % 8 != 0 || x_ld % 8 != 0 ||
        ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(buf)) & 15u) != 0)
        return 0;
    CoopArgs p;
    for (int s = 0; s < LORA_MAX_SLICES; ++s) p.a[s] = nullptr;
    for (int s = 0; s < num_slices; ++s) {
        if (lora_a[s] == nullptr || (reinterpret_cast<uintptr_t>(lora_a[s]) & 15u)) return 0;
        p.a[s] = lora_a[s];
    }
    const int r = expand_setup(p.ex, buf, 0, lora_b, lora_bias, slice_sizes, num_slices, rank, y,
                               y_ld, num_tokens, 0, 1, meta);
    if (r != LORA_OK) return r == 1 ? 0 : r;
    p.map = map;
    p.x = x;
    p.x_ld = x_ld;
    p.hidden = hidden;
    p.scale = scale;
    p.buf = buf;
    p.mapping_copy = meta->token_lora_mapping;
    p.sorted = meta->token_indices_sorted_by_lora_ids;
    p.counts = meta->num_tokens_per_lora;
    p.start_loc = meta->lora_token_start_loc;
    p.active = meta->active_lora_ids;
    p.no_lora = meta->no_lora_flag;
    p.error_word = meta->error_word;
    p.sync = reinterpret_cast<uint32_t *>(meta->grid_sync);
    return launch_linear_coop(p, st);
}

}  // namespace lora
