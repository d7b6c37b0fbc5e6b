// lora_fused.cu -- the whole per-layer LoRA apply for small batches in one
// launch: metadata (page "vllm.lora.ops.triton_ops.lora_kernel_metadata",
// LoRAKernelMeta.prepare_tensors), shrink and expand with fused bias (page
// "vllm.lora.punica_wrapper.punica_gpu", PunicaWrapperGPU.add_lora_linear =
// add_shrink into an fp32 buffer, then add_expand).
//
// Decode batches are latency-bound: three dependent kernels cost more than
// the bytes they move.  Here one thread-block cluster of CL CTAs (one CTA
// per SM) takes one unit = (LoRA segment, tile of up to 64 of its tokens):
//   1. every CTA rebuilds the metadata of the (small) batch in shared memory
//      with the same stable counting sort as the metadata kernel; cluster 0
//      writes it out;
//   2. CTA j computes the shrink partial over its 1/CL of the hidden
//      dimension for all slices (mma.sync, A rows stacked over slices);
//   3. the partials are summed across the cluster through distributed
//      shared memory (each CTA reduces 1/CL of the elements, adds them into
//      the fp32 buffer it owns, then every CTA gathers the full result);
//   4. CTA j expands its 1/CL of the output column chunks for the unit's
//      tokens (mma.sync; bias and old y added in fp32, one bf16 rounding)
//      with a two-stage cp.async ring for y and B.
// Clusters are persistent over units.  The buffer and y receive exactly
// what lora_meta_prepare + lora_shrink + lora_expand (add_inputs = 1,
// offset_start = 0) would write.
#include "lora_common.cuh"

namespace lora {

constexpr int FU_THREADS = 256;         // 8 warps
constexpr int FU_WARPS = FU_THREADS / 32;
constexpr int FU_TT = 64;               // tokens per unit
constexpr int FU_TMAX = 512;            // largest batch the fused path takes
constexpr int FU_MAX_LORAS = 256;
constexpr int FU_HK = 64;               // hidden block (128-byte rows)
constexpr int FU_BN = 128;              // expand columns per chunk
constexpr int FU_Y_LD = FU_BN * 2 + 16;

struct FusedArgs {
    const int32_t *map;
    int32_t num_tokens;
    int32_t max_loras;
    const uint16_t *x;
    int64_t x_ld;
    int32_t hidden;
    const uint16_t *a[LORA_MAX_SLICES];
    const uint16_t *b[LORA_MAX_SLICES];
    const uint16_t *bias[LORA_MAX_SLICES];
    int32_t n[LORA_MAX_SLICES];
    int32_t col0[LORA_MAX_SLICES];
    int32_t chunk0[LORA_MAX_SLICES + 1];
    int32_t num_slices;
    int32_t rank;
    int32_t rp;                          // padded rank (16, 32, 64), S * rp <= 128
    float scale;
    float *buf;
    uint16_t *y;
    int64_t y_ld;
    int32_t hper;                        // hidden elements per CTA (multiple of 64)
    int32_t nst;                         // expand stages (1..8)
    // metadata outputs
    int32_t *mapping_copy;
    int32_t *sorted;
    int32_t *counts;
    int32_t *start_loc;
    int32_t *active;
    int32_t *no_lora;
    int32_t *error_word;
};

struct FuLayout {
    int meta_off, p_off, red_off, work_off, total;
    // meta region
    int cnt_off, tot_off, base_off, pos_off, srt_off, misc_off;
    // phase 2 (shrink) inside work
    int xs_off, as_off;
    // phase 4 (expand) inside work
    int aop_off, stage_off, stage_bytes;
};

__host__ __device__ inline FuLayout fu_layout(int S, int rp, int nbins, int hper, int nst)
{
    FuLayout l;
    const int M = S * rp;                                   // stacked A rows
    l.meta_off = 0;
    l.cnt_off = 0;                                          // [FU_WARPS][nbins]
    l.tot_off = l.cnt_off + FU_WARPS * nbins * 4;           // [nbins]
    l.base_off = l.tot_off + nbins * 4;
    l.pos_off = l.base_off + nbins * 4;
    l.srt_off = l.pos_off + nbins * 4;                      // sorted tokens [FU_TMAX]
    l.misc_off = l.srt_off + FU_TMAX * 4;                   // small scalars
    int end = l.misc_off + 64;
    l.p_off = (end + 127) & ~127;                           // partial [M][FU_TT] fp32
    l.red_off = l.p_off + M * FU_TT * 4;                    // reduced [M][FU_TT] fp32
    l.work_off = ((l.red_off + M * FU_TT * 4) + 1023) & ~1023;
    // shrink: x tile [FU_TT][hper] and A tile [M][hper], 64-column blocks
    l.xs_off = l.work_off;
    l.as_off = l.xs_off + FU_TT * hper * 2;
    // expand (its own region, so its loads can fly during the shrink):
    // A operand [FU_TT][rp] bf16, then nst stages of y tile + B tile + bias
    l.aop_off = (l.as_off + M * hper * 2 + 127) & ~127;
    l.stage_bytes = (FU_TT * FU_Y_LD + FU_BN * rp * 2 + FU_BN * 2 + 127) & ~127;
    l.stage_off = (l.aop_off + FU_TT * rp * 2 + 127) & ~127;
    l.total = l.stage_off + nst * l.stage_bytes + 128;
    return l;
}

__device__ __forceinline__ void cp_async_wait_dyn(int n)
{
    switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    case 7: cp_async_wait<7>(); break;
    default: cp_async_wait<8>(); break;
    }
}

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_peer(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_peer_f4(uint32_t addr)
{
    float4 v;
    asm("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

template <int CL>
__global__ void __launch_bounds__(FU_THREADS, 1) fused_kernel(FusedArgs p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int S = p.num_slices, RP = p.rp, R = p.rank, T = p.num_tokens;
    const int M = S * RP, MT = M / 16;
    const int nbins = p.max_loras + 1;
    const FuLayout Ly = fu_layout(S, RP, nbins, p.hper, p.nst);
    int32_t *cnt = reinterpret_cast<int32_t *>(smem + Ly.cnt_off);
    int32_t *tot = reinterpret_cast<int32_t *>(smem + Ly.tot_off);
    int32_t *basev = reinterpret_cast<int32_t *>(smem + Ly.base_off);
    int32_t *pos = reinterpret_cast<int32_t *>(smem + Ly.pos_off);
    int32_t *srt = reinterpret_cast<int32_t *>(smem + Ly.srt_off);
    int32_t *misc = reinterpret_cast<int32_t *>(smem + Ly.misc_off);
    float *P = reinterpret_cast<float *>(smem + Ly.p_off);
    float *RED = reinterpret_cast<float *>(smem + Ly.red_off);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cluster_ctarank();
    const int cluster = blockIdx.x / CL, nclusters = gridDim.x / CL;

    pdl_wait();
    pdl_launch_dependents();

    // ---------------------------------------------------- 1. metadata
    for (int i = tid; i < FU_WARPS * nbins; i += FU_THREADS) cnt[i] = 0;
    if (tid == 0) misc[0] = 0;                              // invalid ids
    __syncthreads();
    const int per_warp = FU_TMAX / FU_WARPS;                // 64 tokens per warp
    const int t0w = min(T, warp * per_warp), t1w = min(T, t0w + per_warp);
    int bad = 0;
    for (int g = t0w; g < t1w; g += 32) {
        const int t = g + lane;
        const bool has = t < t1w;
        int b = -1;
        if (has) {
            const int32_t id = p.map[t];
            if (id >= 0 && id < p.max_loras) b = id + 1;
            else { b = 0; if (id != -1) ++bad; }
        }
        if (has) atomicAdd(&cnt[warp * nbins + b], 1);          // counts only
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if (lane == 0 && bad) atomicAdd(&misc[0], bad);
    __syncthreads();
    for (int b = tid; b < nbins; b += FU_THREADS) {
        int run = 0;
        for (int w = 0; w < FU_WARPS; ++w) {
            const int c = cnt[w * nbins + b];
            cnt[w * nbins + b] = run;
            run += c;
        }
        tot[b] = run;
    }
    __syncthreads();
    if (warp == 0) {
        int ct = 0, cp = 0;
        for (int b0 = 0; b0 < nbins; b0 += 32) {
            const int b = b0 + lane;
            const int v = (b < nbins) ? tot[b] : 0;
            const int f = v > 0 ? 1 : 0;
            int iv = v, jf = f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, iv, o);
                const int w = __shfl_up_sync(0xffffffffu, jf, o);
                if (lane >= o) { iv += u; jf += w; }
            }
            if (b < nbins) { basev[b] = ct + iv - v; pos[b] = cp + jf - f; }
            ct += __shfl_sync(0xffffffffu, iv, 31);
            cp += __shfl_sync(0xffffffffu, jf, 31);
        }
        if (lane == 0) misc[1] = cp;                         // active entries
    }
    __syncthreads();
    const bool no_lora = (tot[0] == T);
    // stable scatter into the shared sorted list
    if (!no_lora) {
        for (int g = t0w; g < t1w; g += 32) {
            const int t = g + lane;
            const bool has = t < t1w;
            int b = -1;
            if (has) {
                const int32_t id = p.map[t];
                b = (id >= 0 && id < p.max_loras) ? id + 1 : 0;
            }
            const unsigned grp = __match_any_sync(0xffffffffu, b);
            const int rk = __popc(grp & ((1u << lane) - 1u));
            if (has) srt[basev[b] + cnt[warp * nbins + b] + rk] = t;
            __syncwarp();
            if (has && rk == 0) cnt[warp * nbins + b] += __popc(grp);
            __syncwarp();
        }
    }
    __syncthreads();
    // cluster 0 / CTA 0 writes the metadata outputs
    if (cluster == 0 && rank == 0) {
        const int nact = no_lora ? 0 : misc[1];
        for (int k = tid; k < nbins; k += FU_THREADS)
            if (k >= nact) { p.active[k] = -1; p.counts[k] = 0; p.start_loc[k + 1] = 0; }
        if (tid == 0) {
            p.start_loc[0] = 0;
            *p.no_lora = no_lora ? 1 : 0;
            *p.error_word = misc[0];
        }
        if (!no_lora) {
            for (int b = tid; b < nbins; b += FU_THREADS) {
                const int c = tot[b];
                if (c > 0) {
                    const int k = pos[b];
                    p.active[k] = b - 1;
                    p.counts[k] = c;
                    p.start_loc[k + 1] = basev[b] + c;
                }
            }
            for (int t = tid; t < T; t += FU_THREADS) {
                p.sorted[t] = srt[t];
                p.mapping_copy[t] = p.map[t];
            }
        }
    }
    if (no_lora) return;                                     // uniform across the grid

    // units: (bin b with a valid id, tile i of ceil(tot[b] / FU_TT))
    int total_units = 0;
    for (int b = 1; b < nbins; ++b) total_units += (tot[b] + FU_TT - 1) / FU_TT;

    const int hper = p.hper;
    const int h0 = int(rank) * hper;
    const int nkb = max(0, min(hper, p.hidden - h0) + FU_HK - 1) / FU_HK;   // hidden blocks of this CTA
    const int nchunks = p.chunk0[S];
    const int cper = (nchunks + CL - 1) / CL;
    const int cb = int(rank) * cper, ce = min(nchunks, cb + cper);

    for (int unit = cluster; unit < total_units; unit += nclusters) {
        // locate the unit
        int b = 1, u = unit;
        while (b < nbins) {
            const int nt = (tot[b] + FU_TT - 1) / FU_TT;
            if (u < nt) break;
            u -= nt;
            ++b;
        }
        const int id = b - 1;
        const int r0 = basev[b] + u * FU_TT;
        const int nt = min(FU_TT, basev[b] + tot[b] - r0);
        const int32_t *tok = srt + r0;                        // nt tokens (shared)
        const int CPR = RP / 8;
        const int nmine = max(0, ce - cb);                    // expand chunks of this CTA
        int issued = 0;
        auto load_chunk = [&](int slot, int c) {
            int s = 0;
            while (s + 1 < S && p.chunk0[s + 1] <= c) ++s;
            const int n_s = p.n[s];
            const int c0 = (c - p.chunk0[s]) * FU_BN;
            const int ncols = min(FU_BN, n_s - c0);
            const uint32_t sy = smem_addr(smem + Ly.stage_off + slot * Ly.stage_bytes);
            const uint32_t sb = sy + FU_TT * FU_Y_LD;
            const uint32_t sbias = sb + FU_BN * RP * 2;
            uint16_t *yslice = p.y + p.col0[s];
            for (int i = tid; i < FU_TT * (FU_BN / 8); i += FU_THREADS) {
                const int r = i >> 4, cc = i & 15;
                const bool ok = r < nt && cc * 8 < ncols;
                cp_async16(sy + r * FU_Y_LD + cc * 16,
                           ok ? yslice + int64_t(tok[r]) * p.y_ld + c0 + cc * 8 : p.y, ok);
            }
            const uint16_t *bbase = p.b[s] + (int64_t(id) * n_s + c0) * R;
            for (int i = tid; i < FU_BN * CPR; i += FU_THREADS) {
                const int r = i / CPR, cc = i - r * CPR;
                const bool ok = r < ncols && cc * 8 < R;
                const uint32_t dst = (RP == 16) ? sb + swz<2>(r, cc)
                                   : (RP == 32) ? sb + swz<4>(r, cc) : sb + swz<8>(r, cc);
                cp_async16(dst, ok ? bbase + int64_t(r) * R + cc * 8 : p.b[s], ok);
            }
            const uint16_t *bias_row = p.bias[s] ? p.bias[s] + int64_t(id) * n_s + c0 : nullptr;
            if (bias_row != nullptr && tid < FU_BN / 8 && tid * 8 < ncols)
                cp_async16(sbias + tid * 16, bias_row + tid * 8, true);
        };

        // ------------------------------------------------ 2. shrink partial
        {
            const uint32_t xs = smem_addr(smem + Ly.xs_off), as = smem_addr(smem + Ly.as_off);
            // x: FU_TT rows x nkb blocks of 64; A: M rows x nkb blocks (rows past r zero)
            for (int i = tid; i < FU_TT * nkb * 8; i += FU_THREADS) {
                const int row = i / (nkb * 8), rem = i - row * nkb * 8;
                const int kb = rem >> 3, c = rem & 7;
                const int h = h0 + kb * FU_HK + c * 8;
                const bool ok = row < nt && h < p.hidden;
                cp_async16(xs + kb * (FU_TT * 128) + swz<8>(row, c),
                           ok ? p.x + int64_t(tok[row]) * p.x_ld + h : p.x, ok);
            }
            for (int i = tid; i < M * nkb * 8; i += FU_THREADS) {
                const int row = i / (nkb * 8), rem = i - row * nkb * 8;
                const int kb = rem >> 3, c = rem & 7;
                const int s = row / RP, ri = row - s * RP;
                const int h = h0 + kb * FU_HK + c * 8;
                const bool ok = ri < R && h < p.hidden;
                cp_async16(as + kb * (M * 128) + swz<8>(row, c),
                           ok ? p.a[s] + (int64_t(id) * R + ri) * p.hidden + h : p.x, ok);
            }
            cp_async_commit();                                // group: shrink tiles
            // prefetch the first expand chunks (they need only tokens and id)
            for (; issued < nmine && issued < p.nst; ++issued) {
                load_chunk(issued % p.nst, cb + issued);
                cp_async_commit();
            }
            cp_async_wait_dyn(issued);                         // shrink tiles landed
            __syncthreads();
            // warp w: tokens [8w, 8w + 8), all MT row tiles
            float acc[8][4];
#pragma unroll
            for (int m = 0; m < 8; ++m)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[m][q] = 0.f;
            for (int kb = 0; kb < nkb; ++kb) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    uint32_t bfr[2];
                    {
                        // x^T as the col-major B operand: 8 tokens x k16 (x2 load)
                        const int n = warp * 8 + (lane & 7);
                        const int c = kk * 2 + ((lane >> 3) & 1);
                        asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];\n"
                                     : "=r"(bfr[0]), "=r"(bfr[1])
                                     : "r"(xs + kb * (FU_TT * 128) + swz<8>(n, c)));
                    }
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        if (m < MT) {
                            uint32_t af[4];
                            const int r = m * 16 + (lane & 15);
                            const int c = kk * 2 + (lane >> 4);
                            ldmatrix_x4(as + kb * (M * 128) + swz<8>(r, c), af[0], af[1], af[2], af[3]);
                            mma_bf16_16816(acc[m], af, bfr[0], bfr[1]);
                        }
                    }
                }
            }
            // partial P[m][n]
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                if (m < MT) {
                    const int r = m * 16 + (lane >> 2);
                    const int n = warp * 8 + 2 * (lane & 3);
                    P[r * FU_TT + n] = acc[m][0];
                    P[r * FU_TT + n + 1] = acc[m][1];
                    P[(r + 8) * FU_TT + n] = acc[m][2];
                    P[(r + 8) * FU_TT + n + 1] = acc[m][3];
                }
            }
        }
        cluster_sync_all();                                   // all partials written

        // ------------------------------------------------ 3. all-reduce (DSMEM)
        {
            const int E = M * FU_TT;                          // floats, multiple of 4
            const int per = ((E / 4 + CL - 1) / CL) * 4;
            const int e0 = int(rank) * per, e1 = min(E, e0 + per);
            const uint32_t pa = smem_addr(P);
            for (int e = e0 + tid * 4; e < e1; e += FU_THREADS * 4) {
                // all CL remote loads in flight before the first add
                float4 v[CL];
#pragma unroll
                for (int j = 0; j < CL; ++j) v[j] = ld_peer_f4(map_peer(pa + e * 4, uint32_t(j)));
                float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int j = 0; j < CL; ++j) {
                    s4.x += v[j].x; s4.y += v[j].y; s4.z += v[j].z; s4.w += v[j].w;
                }
                // the owner updates the fp32 buffer (buf += scale * sum) and keeps
                // the updated value: that is what expand reads from the buffer
                const float sums[4] = {s4.x, s4.y, s4.z, s4.w};
                float outv[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int el = e + k, mrow = el / FU_TT, n = el - mrow * FU_TT;
                    const int s = mrow / RP, ri = mrow - s * RP;
                    outv[k] = 0.f;
                    if (n < nt && ri < R) {
                        float *bp = p.buf + (int64_t(s) * T + tok[n]) * R + ri;
                        const float v = *bp + p.scale * sums[k];
                        *bp = v;
                        outv[k] = v;
                    }
                }
                *reinterpret_cast<float4 *>(&RED[e]) = make_float4(outv[0], outv[1], outv[2], outv[3]);
            }
        }
        cluster_sync_all();                                   // reduced shares ready
        {
            // gather every share into RED, for the expand of this CTA
            const int E = M * FU_TT;
            const int per = ((E / 4 + CL - 1) / CL) * 4;
            const uint32_t ra = smem_addr(RED);
            for (int e = tid * 4; e < E; e += FU_THREADS * 4) {
                const int owner = e / per;
                if (owner != int(rank)) {
                    const float4 v = ld_peer_f4(map_peer(ra + e * 4, uint32_t(owner)));
                    *reinterpret_cast<float4 *>(&RED[e]) = v;
                }
            }
        }
        cluster_sync_all();                                   // peers done reading P / RED

        // ------------------------------------------------ 4. expand
        if (nmine > 0) {
            uint8_t *aop = smem + Ly.aop_off;
            const uint32_t aopa = smem_addr(aop);
            int cur_s = -1;
            const int wm = warp >> 2, wn = warp & 3;         // 2 x 4 warps, 32 x 32 each
            for (int i = 0; i < nmine; ++i) {
                const int c = cb + i, slot = i % p.nst;
                int s = 0;
                while (s + 1 < S && p.chunk0[s + 1] <= c) ++s;
                if (s != cur_s) {
                    // A operand: reduced rank vectors of slice s for the unit's tokens, bf16
                    __syncthreads();
                    for (int i = tid; i < FU_TT * CPR; i += FU_THREADS) {
                        const int r = i / CPR, cc = i - r * CPR;
                        uint32_t w4[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int c2 = cc * 8 + 2 * k;
                            const float lo = RED[(s * RP + c2) * FU_TT + r];
                            const float hi = RED[(s * RP + c2 + 1) * FU_TT + r];
                            w4[k] = pack_bf16x2(lo, hi);
                        }
                        const uint32_t off = (RP == 16) ? swz<2>(r, cc) : (RP == 32) ? swz<4>(r, cc) : swz<8>(r, cc);
                        *reinterpret_cast<uint4 *>(aop + off) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                    cur_s = s;
                }
                cp_async_wait_dyn(issued - (i + 1));          // chunk i landed
                __syncthreads();
                const int n_s = p.n[s];
                const int c0 = (c - p.chunk0[s]) * FU_BN;
                const int ncols = min(FU_BN, n_s - c0);
                uint8_t *sy = smem + Ly.stage_off + slot * Ly.stage_bytes;
                const uint32_t sb = smem_addr(sy) + FU_TT * FU_Y_LD;
                const uint16_t *sbias = reinterpret_cast<const uint16_t *>(sy + FU_TT * FU_Y_LD + FU_BN * RP * 2);
                const bool has_bias = p.bias[s] != nullptr;
                float acc[2][4][4];
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int n = 0; n < 4; ++n)
#pragma unroll
                        for (int q = 0; q < 4; ++q) acc[m][n][q] = 0.f;
                for (int kk = 0; kk < RP / 16; ++kk) {
                    uint32_t af[2][4];
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const int r = wm * 32 + m * 16 + (lane & 15);
                        const int cc = kk * 2 + (lane >> 4);
                        const uint32_t off = (RP == 16) ? swz<2>(r, cc) : (RP == 32) ? swz<4>(r, cc) : swz<8>(r, cc);
                        ldmatrix_x4(aopa + off, af[m][0], af[m][1], af[m][2], af[m][3]);
                    }
#pragma unroll
                    for (int n2 = 0; n2 < 2; ++n2) {
                        uint32_t bq[4];
                        const int q = lane >> 3;
                        const int r = wn * 32 + n2 * 16 + (q >> 1) * 8 + (lane & 7);
                        const int cc = kk * 2 + (q & 1);
                        const uint32_t off = (RP == 16) ? swz<2>(r, cc) : (RP == 32) ? swz<4>(r, cc) : swz<8>(r, cc);
                        ldmatrix_x4(sb + off, bq[0], bq[1], bq[2], bq[3]);
#pragma unroll
                        for (int m = 0; m < 2; ++m) {
                            mma_bf16_16816(acc[m][2 * n2], af[m], bq[0], bq[1]);
                            mma_bf16_16816(acc[m][2 * n2 + 1], af[m], bq[2], bq[3]);
                        }
                    }
                }
#pragma unroll
                for (int m = 0; m < 2; ++m)
#pragma unroll
                    for (int n = 0; n < 4; ++n)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int r = wm * 32 + m * 16 + (lane >> 2) + 8 * h;
                            const int cl = wn * 32 + n * 8 + 2 * (lane & 3);
                            uint32_t *cell = reinterpret_cast<uint32_t *>(sy + r * FU_Y_LD + cl * 2);
                            float v0 = acc[m][n][2 * h], v1 = acc[m][n][2 * h + 1];
                            if (has_bias && cl < ncols) {
                                v0 += bf16_to_f32(sbias[cl]);
                                v1 += bf16_to_f32(sbias[cl + 1]);
                            }
                            const uint32_t old = *cell;
                            *cell = pack_bf16x2(v0 + bf16_lo(old), v1 + bf16_hi(old));
                        }
                __syncthreads();
                uint16_t *yslice = p.y + p.col0[s];
                for (int i = tid; i < FU_TT * (FU_BN / 8); i += FU_THREADS) {
                    const int r = i >> 4, cc = i & 15;
                    if (r >= nt || cc * 8 >= ncols) continue;
                    const uint4 v = *reinterpret_cast<const uint4 *>(sy + r * FU_Y_LD + cc * 16);
                    *reinterpret_cast<uint4 *>(yslice + int64_t(tok[r]) * p.y_ld + c0 + cc * 8) = v;
                }
                __syncthreads();
                if (issued < nmine) {                          // refill the slot just used
                    load_chunk(issued % p.nst, cb + issued);
                    cp_async_commit();
                    ++issued;
                }
            }
        }
        cp_async_wait<0>();
        __syncthreads();
    }
}

// Cluster size chosen once per device: 16 when the device can co-schedule
// it, else 8; 0 if neither fits (the caller then uses the three kernels).
template <int CL>
static int fused_fits(size_t smem)
{
    if (cudaFuncSetAttribute(fused_kernel<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(smem)) != cudaSuccess)
        return 0;
    if (CL > 8 && cudaFuncSetAttribute(fused_kernel<CL>,
                                       cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL);
    cfg.blockDim = dim3(FU_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fused_kernel<CL>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <int CL>
static int launch_fused_cl(const FusedArgs &p, size_t smem, int clusters, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(clusters * CL);
    cfg.blockDim = dim3(FU_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    return int(cudaLaunchKernelEx(&cfg, fused_kernel<CL>, p));
}

// Returns 1 if the fused kernel was launched, 0 if the call does not fit it,
// or a cudaError_t.
int launch_fused(FusedArgs &p, cudaStream_t stream)
{
    if (p.num_tokens > FU_TMAX || p.max_loras > FU_MAX_LORAS) return 0;
    int rp = 16;
    while (rp < p.rank) rp <<= 1;
    if (rp > 64 || p.num_slices * rp > 128) return 0;
    p.rp = rp;
    static int cl_cache[64] = {0};
    static int nclu_cache[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return int(e);
    const int nbins = p.max_loras + 1;
    // hidden share per CTA, for the largest cluster that fits
    auto hper_for = [&](int cl) {
        return ((p.hidden + cl * FU_HK - 1) / (cl * FU_HK)) * FU_HK;
    };
    if (dev >= 64) return 0;
    if (cl_cache[dev] == 0) {
        // probe with a generous layout (the largest smem this path may use)
        const size_t probe = 227 * 1024;
        int n16 = fused_fits<16>(probe);
        if (n16 > 0) { cl_cache[dev] = 16; nclu_cache[dev] = n16; }
        else {
            int n8 = fused_fits<8>(probe);
            if (n8 > 0) { cl_cache[dev] = 8; nclu_cache[dev] = n8; }
            else cl_cache[dev] = -1;
        }
    }
    const int cl = cl_cache[dev];
    if (cl <= 0) return 0;
    p.hper = hper_for(cl);
    int chunks_total = p.chunk0[p.num_slices];
    const int cper = (chunks_total + cl - 1) / cl;
    p.nst = 8;
    if (p.nst > cper) p.nst = max(1, cper);
    while (p.nst > 1 && fu_layout(p.num_slices, rp, nbins, p.hper, p.nst).total > 227 * 1024) --p.nst;
    const FuLayout L = fu_layout(p.num_slices, rp, nbins, p.hper, p.nst);
    if (L.total > 227 * 1024) return 0;
    // units: at most ceil(T / 64) + (number of distinct ids)
    const int units_max = (p.num_tokens + FU_TT - 1) / FU_TT + min(p.max_loras, p.num_tokens);
    const int clusters = max(1, min(units_max, nclu_cache[dev]));
    const int err = (cl == 16) ? launch_fused_cl<16>(p, size_t(L.total), clusters, stream)
                               : launch_fused_cl<8>(p, size_t(L.total), clusters, stream);
    return err == 0 ? 1 : err;
}

}  // namespace lora

LORA_API int lora_linear(const int32_t *token_lora_mapping, int32_t num_tokens,
                         const lora_bf16_t *x, int32_t hidden, int64_t x_ld,
                         const lora_bf16_t *const *lora_a, const lora_bf16_t *const *lora_b,
                         const lora_bf16_t *const *lora_bias, const int32_t *slice_sizes,
                         int32_t num_slices, int32_t rank, float scale, float *buf,
                         lora_bf16_t *y, int64_t y_ld, const lora_meta_t *meta, void *stream)
{
    lora::NvtxRange nvtx_range("lora_linear");
    if (meta == nullptr || lora_a == nullptr || lora_b == nullptr || slice_sizes == nullptr)
        return LORA_ERR_NULL;
    if (num_slices < 1 || num_slices > LORA_MAX_SLICES) return LORA_ERR_SLICES;
    if (rank < 8 || rank > LORA_MAX_RANK || rank % 8 != 0) return LORA_ERR_RANK;
    if (num_tokens < 0 || hidden < 0 || x_ld < hidden || y_ld < 0) return LORA_ERR_SIZE;
    if (num_tokens > meta->max_num_tokens) return LORA_ERR_TOKENS;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // Small batches as one cooperative kernel (metadata, shrink, grid
    // barrier, expand), when the layout fits it (lora_linear_coop.cu).  By
    // default it takes batches with num_tokens * num_slices <= 256 (the
    // shrink rows): measured faster than the other paths on 64 tokens x 1
    // slice and on 256 x 1 (logits-like), slower on 256 x 3 (q/k/v decode),
    // where the shrink phase and the barrier cost more than the launches
    // they replace.  LORA_PUNICA_COOP=1 takes it for every batch that fits
    // (up to 512 tokens), LORA_PUNICA_COOP=0 never.
    const lora::Knobs &kn = lora::knobs();
    const int coop_mode = kn.coop;
    if (kn.linear_tc != 2 && (coop_mode == 1 ||
                              (coop_mode != 0 && int64_t(num_tokens) * num_slices <= 256))) {
        const int r = lora::linear_coop(token_lora_mapping, num_tokens, x, hidden, x_ld, lora_a,
                                        lora_b, lora_bias, slice_sizes, num_slices, rank, scale,
                                        buf, y, y_ld, meta, st);
        if (r == 1) return LORA_OK;
        if (r != 0) return r;
    }

    // One fused kernel for small batches when every layout rule of the
    // vector paths holds.  By default it is taken for batches of at most
    // LORA_PUNICA_FUSED_MAX_TOKENS (128) tokens: measured on decode-sized
    // batches (256 tokens, 8 LoRAs) the per-unit chain of cluster syncs and
    // shared-memory reductions made it slower than the three kernels, on 64
    // tokens faster.  LORA_PUNICA_FUSED=1 takes it up to 512 tokens,
    // LORA_PUNICA_FUSED=0 never.
    const int fused_mode = kn.fused;
    const int fused_max = fused_mode == 1 ? lora::FU_TMAX : kn.fused_max_tokens;
    bool fused = fused_mode != 0 && kn.linear_tc != 2 && num_tokens > 0 && num_tokens <= fused_max &&
                 token_lora_mapping != nullptr && x != nullptr && buf != nullptr && y != nullptr &&
                 hidden > 0 && hidden % 8 == 0 && x_ld % 8 == 0 && y_ld % 8 == 0 &&
                 meta->max_loras >= 1 && meta->max_loras <= lora::FU_MAX_LORAS &&
                 meta->token_lora_mapping && meta->token_indices_sorted_by_lora_ids &&
                 meta->num_tokens_per_lora && meta->lora_token_start_loc &&
                 meta->active_lora_ids && meta->no_lora_flag && meta->error_word &&
                 ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y) |
                   reinterpret_cast<uintptr_t>(buf)) & 15u) == 0;
    lora::FusedArgs p;
    if (fused) {
        int64_t col = 0;
        int chunks = 0;
        for (int s = 0; s < LORA_MAX_SLICES; ++s) {
            p.a[s] = p.b[s] = p.bias[s] = nullptr;
            p.n[s] = p.col0[s] = p.chunk0[s] = 0;
        }
        for (int s = 0; s < num_slices && fused; ++s) {
            const int32_t n = slice_sizes[s];
            const lora_bf16_t *bb = lora_bias ? lora_bias[s] : nullptr;
            if (n < 0 || n % 8 != 0 || !lora_a[s] || !lora_b[s] ||
                ((reinterpret_cast<uintptr_t>(lora_a[s]) | reinterpret_cast<uintptr_t>(lora_b[s]) |
                  reinterpret_cast<uintptr_t>(bb)) & 15u)) {
                fused = false;
                break;
            }
            p.a[s] = lora_a[s];
            p.b[s] = lora_b[s];
            p.bias[s] = bb;
            p.n[s] = n;
            p.col0[s] = int32_t(col);
            p.chunk0[s] = chunks;
            chunks += (n + lora::FU_BN - 1) / lora::FU_BN;
            col += n;
        }
        p.chunk0[num_slices] = chunks;
        if (col > y_ld) return LORA_ERR_WIDTH;
        if (fused) {
            p.map = token_lora_mapping;
            p.num_tokens = num_tokens;
            p.max_loras = meta->max_loras;
            p.x = x;
            p.x_ld = x_ld;
            p.hidden = hidden;
            p.num_slices = num_slices;
            p.rank = rank;
            p.scale = scale;
            p.buf = buf;
            p.y = y;
            p.y_ld = y_ld;
            p.mapping_copy = meta->token_lora_mapping;
            p.sorted = meta->token_indices_sorted_by_lora_ids;
            p.counts = meta->num_tokens_per_lora;
            p.start_loc = meta->lora_token_start_loc;
            p.active = meta->active_lora_ids;
            p.no_lora = meta->no_lora_flag;
            p.error_word = meta->error_word;
            const int r = lora::launch_fused(p, st);
            if (r == 1) return LORA_OK;
            if (r != 0) return r;
        }
    }
    // Rank 128, up to three slices, batches of at least 72 tokens per SM
    // (LORA_PUNICA_LINEAR_TC_MIN_TOKENS): the metadata kernel, then the
    // shrink and the expand of every 128-token tile in one tensor-core
    // kernel (lora_linear_tc.cu).  A CTA takes a whole tile through both,
    // about 180 us at hidden 8192 and 10240 output columns whatever its
    // rows, so the kernel pays when the tiles fill the SMs.  Measured on the
    // large workload's shapes (hidden 8192, slices 8192/1024/1024), step
    // time, separate kernels against this one: 140 / 181 us at 8192 tokens,
    // 211 / 195 at 11264, 239 / 214.5 at 16384, 339 / 351 at 17408 (past one
    // tile per SM both take two rounds of tiles), 415 / 398 at 24576, 461 /
    // 409 at 32768.  LORA_PUNICA_LINEAR_TC=0 keeps the separate kernels; =1
    // takes it for every call it fits; =2 requires it (a call it does not
    // fit fails with LORA_ERR_SIZE: for tests that must not pass on the
    // separate kernels).
    const int64_t tc_min = kn.linear_tc_min_tokens > 0 ? int64_t(kn.linear_tc_min_tokens)
                                                       : int64_t(72) * lora::device_sm_count();
    const bool tc_req = kn.linear_tc == 2;
    if (tc_req && (token_lora_mapping == nullptr || meta->error_word == nullptr || rank != 128 ||
                   num_slices > 3))
        return LORA_ERR_SIZE;
    if (kn.linear_tc != 0 && token_lora_mapping != nullptr && meta->error_word != nullptr &&
        (kn.linear_tc >= 1 || num_tokens >= tc_min) && rank == 128 && num_slices <= 3) {
        lora::LinearTcLaunch u;
        int64_t width = 0;
        for (int s = 0; s < LORA_MAX_SLICES; ++s) u.a[s] = u.b[s] = u.bias[s] = nullptr;
        for (int s = 0; s < num_slices; ++s) {
            u.a[s] = lora_a[s];
            u.b[s] = lora_b[s];
            u.bias[s] = lora_bias ? lora_bias[s] : nullptr;
            u.n[s] = slice_sizes[s];
            width += slice_sizes[s];
        }
        u.x = x;
        u.x_ld = x_ld;
        u.hidden = hidden;
        u.num_tokens = num_tokens;
        u.num_slices = num_slices;
        u.rank = rank;
        u.max_loras = meta->max_loras;
        u.scale = scale;
        u.buf = buf;
        u.y = y;
        u.y_ld = y_ld;
        u.sorted = meta->token_indices_sorted_by_lora_ids;
        u.counts = meta->num_tokens_per_lora;
        u.start_loc = meta->lora_token_start_loc;
        u.active = meta->active_lora_ids;
        u.no_lora = meta->no_lora_flag;
        u.error_word = meta->error_word;
        if (width <= y_ld && lora::linear_tc_fits(u)) {
            int r = lora_meta_prepare(token_lora_mapping, num_tokens, meta, stream);
            if (r != 0) return r;
            r = lora::launch_linear_tc(u, st);
            return r == 0 ? LORA_OK : r;
        }
        if (tc_req) return LORA_ERR_SIZE;
    }

    // The metadata kernel, then the shrink in early mode (for batches of up
    // to 512 tokens it sorts the ids itself and starts its loads while the
    // metadata kernel runs), then the expand in early mode (it fetches the
    // metadata, y and B while the shrink runs).  LORA_PUNICA_SELF_META=1
    // instead drops the metadata kernel (the shrink writes the metadata);
    // =0 runs the plain three calls.
    const int self_meta = kn.self_meta;
    int r = 0;
    bool early = false;
    if (self_meta == 1) {
        r = lora::shrink_self_meta(token_lora_mapping, x, num_tokens, hidden, x_ld, lora_a,
                                   num_slices, rank, buf, meta, scale, st, 0);
        if (r < 0 || r > 1) return r;
    } else if (self_meta == -1) {
        r = lora_meta_prepare(token_lora_mapping, num_tokens, meta, stream);
        if (r != 0) return r;
        r = lora::shrink_self_meta(token_lora_mapping, x, num_tokens, hidden, x_ld, lora_a,
                                   num_slices, rank, buf, meta, scale, st, 1);
        if (r < 0 || r > 1) return r;
        if (r == 0) {
            r = lora_shrink(x, num_tokens, hidden, x_ld, lora_a, num_slices, rank, buf, meta,
                            scale, stream);
            if (r != 0) return r;
        }
        early = true;
        r = 1;
    }
    if (r == 0) {
        r = lora_meta_prepare(token_lora_mapping, num_tokens, meta, stream);
        if (r != 0) return r;
        r = lora_shrink(x, num_tokens, hidden, x_ld, lora_a, num_slices, rank, buf, meta, scale,
                        stream);
        if (r != 0) return r;
    }
    if (early)
        return lora::expand_early(buf, lora_b, lora_bias, slice_sizes, num_slices, rank, y, y_ld,
                                  num_tokens, meta, st);
    return lora_expand(buf, lora_b, lora_bias, slice_sizes, num_slices, rank, y, y_ld, num_tokens,
                       0, 1, meta, stream);
}
