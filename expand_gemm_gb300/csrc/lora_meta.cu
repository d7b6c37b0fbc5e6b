// lora_meta.cu -- metadata step (page "vllm.lora.ops.triton_ops.
// lora_kernel_metadata", LoRAKernelMeta._reset + prepare_tensors): a
// stable counting sort by LoRA id.  Per-warp bin histograms (shared-memory
// atomic adds), a warp-shuffle scan over (bin, warp), and a stable scatter
// (lanes of one bin ranked with __match_any_sync).
//
// Two kernels compute it:
//   - meta_prepare_kernel: one CTA, the id map staged in shared memory;
//     batches of up to META_MULTI_MIN tokens.
//   - meta_multi_kernel<NT>: one CTA per run of NT tokens (256 up to
//     META_MULTI_BIG tokens, 1024 above), one 32-token group per warp.  Every
//     CTA counts the whole map itself (its run one 32-token group per warp,
//     the rest 128 tokens per 16-byte warp load with one vote; the map is
//     read from L2), keeping apart the tokens before its run, those of its
//     run (per warp) and those after it.  That gives
//     it the bin totals and its own start inside every bin without any
//     exchange between CTAs, and it scatters the tokens of its run.
//
// Bins: bin 0 holds id -1 (and every invalid id), bin b > 0 holds id b - 1.
// Token order inside a bin is preserved because (1) each warp owns one
// contiguous run of tokens, (2) warps are ranked in token order inside a
// bin by the scan, and (3) inside a warp, 32-token groups are visited in
// order and lanes are ranked by lane index.  So the permutation equals a
// stable sort by id, which is what torch.sort(stable=True) returns.
#include "lora_common.cuh"

namespace lora {

constexpr int META_THREADS = 1024;       // the largest block (big batches)
constexpr int META_SMALL_THREADS = 256;  // batches of up to META_SMALL_MAX tokens
constexpr int META_SMALL_MAX = 512;
// Batches up to this many tokens are first copied into shared memory with
// one block-wide load (all of it in flight at once); both passes then read
// shared memory.  Larger batches read the map from global memory.
constexpr int META_STAGE_MAX = 16384;
// Batches above this many tokens take the multi-CTA kernel: runs of 256
// tokens up to META_MULTI_BIG tokens (8 to 16 CTAs), runs of 1024 above.
// One SM sorting 2048 tokens was issue-bound (4.4 us in the kernel).
constexpr int META_MULTI_MIN = 512;
constexpr int META_MULTI_BIG = 4096;
constexpr int META_MULTI_SMALL_THREADS = 256;
constexpr int META_MULTI_THREADS = 1024;

struct MetaArgs {
    const int32_t *map;
    int32_t num_tokens;
    int32_t max_loras;
    int32_t *mapping_copy;
    int32_t *sorted;
    int32_t *counts;
    int32_t *start_loc;
    int32_t *active;
    int32_t *no_lora;
    int32_t *error_word;
};

// Batches up to this many tokens also build the permutation in shared
// memory (written out in order at the end).  With 1025 bins and the map
// staged, 4096 more ints is what still fits in one CTA's shared memory.
constexpr int META_PERM_STAGE_MAX = 4096;

// Ints of shared memory for the staged map and the staged permutation,
// each rounded up to 16 bytes (0 when not staged).
__host__ __device__ __forceinline__ int meta_staged_ints(int num_tokens)
{
    return num_tokens <= META_STAGE_MAX ? (num_tokens + 3) & ~3 : 0;
}
__host__ __device__ __forceinline__ int meta_perm_ints(int num_tokens)
{
    return num_tokens <= META_PERM_STAGE_MAX ? (num_tokens + 3) & ~3 : 0;
}

size_t meta_smem_bytes(int warps, int max_loras, int num_tokens)
{
    const size_t nb = size_t(max_loras) + 1;
    return (size_t(warps) * nb + 3 * nb + size_t(meta_staged_ints(num_tokens)) +
            size_t(meta_perm_ints(num_tokens))) * sizeof(int32_t);
}

// Bin of one token; counts an invalid id into `bad`.
__device__ __forceinline__ int token_bin(int32_t id, int32_t max_loras, int &bad)
{
    if (id >= 0 && id < max_loras) return id + 1;
    if (id != -1) ++bad;
    return 0;
}

// Pass 1 for one 32-token group: adds the group's tokens to this warp's bin
// counts.  A group whose tokens all fall in one bin (runs of one sequence,
// the all -1 batch) takes one add instead of 32 conflicting ones.
__device__ __forceinline__ void count_group(int32_t *cnt_w, int b, bool has, int lane)
{
    const int b0 = __shfl_sync(0xffffffffu, b, 0);
    if (__all_sync(0xffffffffu, has && b == b0)) {
        if (lane == 0) atomicAdd(&cnt_w[b0], 32);
    } else if (has) {
        atomicAdd(&cnt_w[b], 1);
    }
}

// Pass 2 for one 32-token group: each token's rank among the group's tokens
// of its bin, and the number of those tokens (returned to rank 0 of each
// bin).  Lane order is token order, so the ranks keep the sort stable.
__device__ __forceinline__ int rank_in_group(int b, bool has, int lane, int &group_count)
{
    const int b0 = __shfl_sync(0xffffffffu, b, 0);
    if (__all_sync(0xffffffffu, has && b == b0)) {
        group_count = 32;
        return lane;
    }
    const unsigned grp = __match_any_sync(0xffffffffu, b);
    group_count = __popc(grp);
    return __popc(grp & ((1u << lane) - 1u));
}

template <int NT>
__global__ void __launch_bounds__(NT, 1) meta_prepare_kernel(MetaArgs a)
{
    constexpr int META_WARPS = NT / 32;
    extern __shared__ int4 sm4[];
    const int nb = a.max_loras + 1;
    const int T = a.num_tokens;
    const int TS = meta_staged_ints(T);         // 0 when not staged
    const int TP = meta_perm_ints(T);
    int32_t *ids_s = reinterpret_cast<int32_t *>(sm4);  // [TS] the map, when staged
    int32_t *perm_s = ids_s + TS;               // [TP] the permutation, when staged
    int32_t *cnt = perm_s + TP;                 // [META_WARPS][nb]: count, then offset
    int32_t *tot = cnt + META_WARPS * nb;       // [nb] tokens per bin
    int32_t *base = tot + nb;                   // [nb] first sorted slot of the bin
    int32_t *pos = base + nb;                   // [nb] index among non-empty bins
    __shared__ int32_t s_invalid, s_nactive;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    pdl_wait();
    pdl_launch_dependents();

    // Stage the map with one 16-byte load per thread and pass where it is
    // aligned (all of it in flight at once).
    const bool staged = TS > 0;
    if (staged) {
        const bool vec = (reinterpret_cast<uintptr_t>(a.map) & 15u) == 0;
        const int nv = vec ? T >> 2 : 0;
        for (int i = tid; i < nv; i += NT)
            reinterpret_cast<int4 *>(ids_s)[i] = reinterpret_cast<const int4 *>(a.map)[i];
        for (int t = nv * 4 + tid; t < T; t += NT) ids_s[t] = a.map[t];
    }
    const int32_t *ids = staged ? ids_s : a.map;
    for (int i = tid; i < META_WARPS * nb; i += NT) cnt[i] = 0;
    if (tid == 0) s_invalid = 0;
    __syncthreads();

    // Each warp owns tokens [t0, t1), a multiple of 32 long (the last may be short).
    const int per_warp = ((T + NT - 1) / NT) * 32;
    const int t0 = min(T, warp * per_warp);
    const int t1 = min(T, t0 + per_warp);

    // Pass 1: per-warp histogram, one shared-memory atomic add per token,
    // or one per group of 32 tokens of one bin (counts only: pass 2 keeps
    // the order).  Per-token adds were measured faster than grouping lanes
    // (with __match_any_sync, or with one ballot per bit of the bin).
    int bad = 0;
    for (int g = t0; g < t1; g += 32) {
        const int t = g + lane;
        const bool has = t < t1;
        const int b = has ? token_bin(ids[t], a.max_loras, bad) : -1;
        count_group(cnt + warp * nb, b, has, lane);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if (lane == 0 && bad) atomicAdd(&s_invalid, bad);
    __syncthreads();

    scan_bins_over_warps<NT, META_WARPS>(cnt, tot, nullptr, nullptr, nb);
    __syncthreads();
    scan_over_bins<NT>(tot, base, pos, &s_nactive, nb);
    __syncthreads();

    const bool no_lora = (tot[0] == T);         // also true for T == 0
    const int nact = no_lora ? 0 : s_nactive;

    // _reset values for every slot that no active id fills.
    for (int k = tid; k < nb; k += NT) {
        if (k >= nact) {
            a.active[k] = -1;
            a.counts[k] = 0;
            a.start_loc[k + 1] = 0;
        }
    }
    if (tid == 0) {
        a.start_loc[0] = 0;
        *a.no_lora = no_lora ? 1 : 0;
        *a.error_word = s_invalid;
    }
    if (no_lora) return;                        // early exit: nothing else written

    // unique(sorted=True, return_counts=True) and cumsum into start_loc[1:].
    for (int b = tid; b < nb; b += NT) {
        const int c = tot[b];
        if (c > 0) {
            const int k = pos[b];
            a.active[k] = b - 1;
            a.counts[k] = c;
            a.start_loc[k + 1] = base[b] + c;
        }
    }

    // Pass 2: stable scatter + mapping copy.  A batch of up to
    // META_PERM_STAGE_MAX tokens is scattered in shared memory and written
    // out in order afterwards: scattered 4-byte stores from one SM (one L2
    // request each) were the slowest phase with per-token ids.
    const bool perm_staged = TP > 0;
    int32_t *perm = perm_staged ? perm_s : a.sorted;
    int unused = 0;
    for (int g = t0; g < t1; g += 32) {
        const int t = g + lane;
        const bool has = t < t1;
        const int32_t id = has ? ids[t] : -1;
        const int b = has ? token_bin(id, a.max_loras, unused) : -1;
        int n = 0;
        const int rank = rank_in_group(b, has, lane, n);
        if (has) {
            perm[base[b] + cnt[warp * nb + b] + rank] = t;
            a.mapping_copy[t] = id;
        }
        __syncwarp();
        if (has && rank == 0) cnt[warp * nb + b] += n;
        __syncwarp();
    }
    if (perm_staged) {
        __syncthreads();
        const bool vec = (reinterpret_cast<uintptr_t>(a.sorted) & 15u) == 0;
        const int nv = vec ? T >> 2 : 0;
        for (int i = tid; i < nv; i += NT)
            reinterpret_cast<int4 *>(a.sorted)[i] = reinterpret_cast<const int4 *>(perm_s)[i];
        for (int t = nv * 4 + tid; t < T; t += NT) a.sorted[t] = perm_s[t];
    }
}

template <int NT>
__global__ void __launch_bounds__(NT) meta_multi_kernel(MetaArgs a)
{
    constexpr int NW = NT / 32;                 // the run: one 32-token group per warp
    static_assert(NT % 128 == 0, "the run is whole 128-token blocks");
    extern __shared__ int32_t sm[];
    const int nb = a.max_loras + 1;
    int32_t *own = sm;                          // [NW][nb]: run counts per warp, then offsets
    int32_t *bef = own + NW * nb;               // [nb] tokens before the run
    int32_t *aft = bef + nb;                    // [nb] tokens after the run
    int32_t *tot = aft + nb;                    // [nb] all tokens
    int32_t *base = tot + nb;                   // [nb] first sorted slot of the bin
    int32_t *pos = base + nb;                   // [nb] index among non-empty bins
    __shared__ int32_t s_invalid, s_nactive;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = a.num_tokens, cta = int(blockIdx.x);
    const int g_run = cta * NW;                 // first 32-token group of the run

    pdl_wait();
    pdl_launch_dependents();

    for (int i = tid; i < (NW + 2) * nb; i += NT) sm[i] = 0;
    if (tid == 0) s_invalid = 0;
    __syncthreads();

    // Pass 1.  The CTA's own run: warp w counts the run's 32-token group w
    // into own[w] (pass 2 needs the per-warp offsets).  The rest of the map
    // only needs its totals before and after the run: it is read in blocks
    // of 128 tokens, four ids per lane from one 16-byte load, four blocks
    // per warp at a time so that their latencies overlap, and a block whose
    // ids all fall in one bin (runs of one sequence, the all -1 batch) takes
    // a single add.
    int bad = 0;
    // The run's id is loaded first and counted after the rest, so that all
    // of this warp's loads are in flight together (one round trip, not two).
    const int t_own = (g_run + warp) * 32 + lane;
    const int32_t id_own = t_own < T ? a.map[t_own] : -1;
    const bool vec = (reinterpret_cast<uintptr_t>(a.map) & 15u) == 0;
    const int nblk = (T + 127) / 128, rb0 = cta * (NW / 4), rb1 = rb0 + NW / 4;
    constexpr int UB = 4;
    for (int k0 = warp; k0 < nblk; k0 += NW * UB) {
        int4 v[UB];
#pragma unroll
        for (int u = 0; u < UB; ++u) {
            const int k = k0 + u * NW, t0 = k * 128 + lane * 4;
            v[u] = make_int4(-1, -1, -1, -1);
            if (k < nblk && (k < rb0 || k >= rb1)) {
                if (vec && t0 + 3 < T) {
                    v[u] = *reinterpret_cast<const int4 *>(a.map + t0);
                } else {
                    if (t0 < T) v[u].x = a.map[t0];
                    if (t0 + 1 < T) v[u].y = a.map[t0 + 1];
                    if (t0 + 2 < T) v[u].z = a.map[t0 + 2];
                    if (t0 + 3 < T) v[u].w = a.map[t0 + 3];
                }
            }
        }
#pragma unroll
        for (int u = 0; u < UB; ++u) {
            const int k = k0 + u * NW, t0 = k * 128 + lane * 4;     // k: the same in every lane
            if (k >= nblk) break;
            if (k >= rb0 && k < rb1) continue;                       // the run: counted above
            int32_t *dst = k < rb0 ? bef : aft;
            const int ids[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            int bs[4];
            bool all_in = true;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool has = t0 + j < T;
                bs[j] = has ? token_bin(ids[j], a.max_loras, bad) : -1;
                all_in = all_in && has;
            }
            const int b0 = __shfl_sync(0xffffffffu, bs[0], 0);
            const bool same = all_in && bs[0] == b0 && bs[1] == b0 && bs[2] == b0 && bs[3] == b0;
            if (__all_sync(0xffffffffu, same)) {
                if (lane == 0) atomicAdd(&dst[b0], 128);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (bs[j] >= 0) atomicAdd(&dst[bs[j]], 1);
            }
        }
    }
    {
        const bool has = t_own < T;
        const int b = has ? token_bin(id_own, a.max_loras, bad) : -1;
        count_group(own + warp * nb, b, has, lane);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if (lane == 0 && bad) atomicAdd(&s_invalid, bad);
    __syncthreads();
    // Per bin: the run's warps scanned in token order, and the totals; then
    // the scans over bins.
    scan_bins_over_warps<NT, NW>(own, tot, bef, aft, nb);
    __syncthreads();
    scan_over_bins<NT>(tot, base, pos, &s_nactive, nb);
    __syncthreads();

    const bool no_lora = (tot[0] == T);
    const int nact = no_lora ? 0 : s_nactive;
    if (cta == 0) {
        for (int k = tid; k < nb; k += NT) {
            if (k >= nact) {
                a.active[k] = -1;
                a.counts[k] = 0;
                a.start_loc[k + 1] = 0;
            }
        }
        if (tid == 0) {
            a.start_loc[0] = 0;
            *a.no_lora = no_lora ? 1 : 0;
            *a.error_word = s_invalid;
        }
        if (!no_lora) {
            for (int b = tid; b < nb; b += NT) {
                const int c = tot[b];
                if (c > 0) {
                    const int k = pos[b];
                    a.active[k] = b - 1;
                    a.counts[k] = c;
                    a.start_loc[k + 1] = base[b] + c;
                }
            }
        }
    }
    if (no_lora) return;                        // early exit: nothing else written
    // Pass 2: stable scatter of this warp's group of the run + mapping copy.
    const bool has = t_own < T;
    int unused = 0;
    const int b = has ? token_bin(id_own, a.max_loras, unused) : -1;
    int n = 0;
    const int rank = rank_in_group(b, has, lane, n);
    if (has) {
        a.sorted[base[b] + bef[b] + own[warp * nb + b] + rank] = t_own;
        a.mapping_copy[t_own] = id_own;
    }
}

// ------------------------------------------------------------------------
// Thread-block-cluster form (one cluster of C <= 8 CTAs is the whole grid,
// batches of META_MULTI_BIG + 1 .. META_CLUSTER_MAX tokens): CTA c owns the
// run of GW * NT tokens starting at c * GW * NT (GW 32-token groups per
// warp) and counts only that run.  Its bin totals and its start inside
// every bin come from the other CTAs' run counts, read from their shared
// memory after a cluster barrier, instead of every CTA reading the whole
// map (2.6 us of the 4 us kernel at 16384 tokens).  Every thread passes
// both cluster barriers on one straight path (no early return), so neither
// can be left waiting.
constexpr int META_CLUSTER_MAX = 8 * 4 * 1024;

__device__ __forceinline__ uint32_t meta_cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ int32_t meta_ld_cluster(const int32_t *local, uint32_t rank)
{
    uint32_t a, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(a) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];\n" : "=r"(v) : "r"(a) : "memory");
    return int32_t(v);
}
// (.aligned: the warp reaches them converged)
__device__ __forceinline__ void meta_cluster_arrive()
{
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void meta_cluster_wait()
{
    __syncwarp();
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

template <int NT, int GW>
__global__ void __launch_bounds__(NT) meta_cluster_kernel(MetaArgs a)
{
    constexpr int NW = NT / 32;
    extern __shared__ int32_t sm[];
    const int nb = a.max_loras + 1;
    int32_t *own = sm;                          // [NW][nb]: run counts per warp, then offsets
    int32_t *run = own + NW * nb;               // [nb] this CTA's run (read by the others)
    int32_t *bef = run + nb;                    // [nb] tokens of the CTAs before this one
    int32_t *tot = bef + nb;                    // [nb] all tokens
    int32_t *base = tot + nb;                   // [nb] first sorted slot of the bin
    int32_t *pos = base + nb;                   // [nb] index among non-empty bins
    __shared__ int32_t s_invalid, s_nactive, s_bad_all;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = a.num_tokens;
    const uint32_t crank = meta_cluster_rank();     // == blockIdx.x: one cluster per grid
    const int nctas = int(gridDim.x);
    const int tw0 = int(crank) * (NT * GW) + warp * (32 * GW);   // this warp's run

    pdl_wait();
    pdl_launch_dependents();

    int32_t idv[GW];
#pragma unroll
    for (int j = 0; j < GW; ++j) {
        const int t = tw0 + 32 * j + lane;
        idv[j] = t < T ? a.map[t] : -1;
    }
    for (int i = tid; i < NW * nb; i += NT) own[i] = 0;
    if (tid == 0) s_invalid = 0;
    __syncthreads();
    int bad = 0;
#pragma unroll
    for (int j = 0; j < GW; ++j) {
        const int t = tw0 + 32 * j + lane;
        const bool has = t < T;
        const int b = has ? token_bin(idv[j], a.max_loras, bad) : -1;
        count_group(own + warp * nb, b, has, lane);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if (lane == 0 && bad) atomicAdd(&s_invalid, bad);
    __syncthreads();
    scan_bins_over_warps<NT, NW>(own, run, nullptr, nullptr, nb);

    meta_cluster_arrive();                      // every CTA's run counts are final
    meta_cluster_wait();
    // eight lanes per bin, one CTA's count each (one remote load a thread,
    // all in flight together), summed by shuffles
    for (int i0 = 0; i0 < nb * 8; i0 += NT) {      // the same in every thread
        const int i = i0 + tid, b = i >> 3, c = i & 7;
        const int v = (b < nb && c < nctas) ? meta_ld_cluster(run + b, uint32_t(c)) : 0;
        int st = v, sb = c < int(crank) ? v : 0;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            st += __shfl_xor_sync(0xffffffffu, st, o);
            sb += __shfl_xor_sync(0xffffffffu, sb, o);
        }
        if (b < nb && c == 0) {
            bef[b] = sb;
            tot[b] = st;
        }
    }
    if (crank == 0 && tid == 0) {
        int sbad = 0;
        for (int c = 0; c < nctas; ++c) sbad += meta_ld_cluster(&s_invalid, uint32_t(c));
        s_bad_all = sbad;
    }
    meta_cluster_arrive();                      // done reading the others' shared memory
    __syncthreads();
    scan_over_bins<NT>(tot, base, pos, &s_nactive, nb);
    __syncthreads();

    const bool no_lora = (tot[0] == T);
    const int nact = no_lora ? 0 : s_nactive;
    if (crank == 0) {
        for (int k = tid; k < nb; k += NT) {
            if (k >= nact) {
                a.active[k] = -1;
                a.counts[k] = 0;
                a.start_loc[k + 1] = 0;
            }
        }
        if (tid == 0) {
            a.start_loc[0] = 0;
            *a.no_lora = no_lora ? 1 : 0;
            *a.error_word = s_bad_all;
        }
        if (!no_lora) {
            for (int b = tid; b < nb; b += NT) {
                const int c = tot[b];
                if (c > 0) {
                    const int k = pos[b];
                    a.active[k] = b - 1;
                    a.counts[k] = c;
                    a.start_loc[k + 1] = base[b] + c;
                }
            }
        }
    }
    if (!no_lora) {                             // stable scatter of this warp's run
        int unused = 0;
#pragma unroll
        for (int j = 0; j < GW; ++j) {
            const int t = tw0 + 32 * j + lane;
            const bool has = t < T;
            const int b = has ? token_bin(idv[j], a.max_loras, unused) : -1;
            int n = 0;
            const int rank = rank_in_group(b, has, lane, n);
            if (has) {
                a.sorted[base[b] + bef[b] + own[warp * nb + b] + rank] = t;
                a.mapping_copy[t] = idv[j];
            }
            __syncwarp();
            if (has && rank == 0) own[warp * nb + b] += n;
            __syncwarp();
        }
    }
    meta_cluster_wait();                        // no CTA leaves while another reads it
}

size_t meta_cluster_smem_bytes(int max_loras)
{
    const size_t nb = size_t(max_loras) + 1;
    return (size_t(META_MULTI_THREADS / 32) * nb + 5 * nb) * sizeof(int32_t);
}

template <int GW>
static cudaError_t launch_meta_cluster(const MetaArgs &a, cudaStream_t stream)
{
    constexpr int NT = META_MULTI_THREADS;
    const int grid = (a.num_tokens + NT * GW - 1) / (NT * GW);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = meta_cluster_smem_bytes(a.max_loras);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(grid);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, meta_cluster_kernel<NT, GW>, a);
}

size_t meta_multi_smem_bytes(int warps, int max_loras)
{
    const size_t nb = size_t(max_loras) + 1;
    return (size_t(warps) * nb + 5 * nb) * sizeof(int32_t);
}

int launch_meta_prepare(const MetaArgs &a, cudaStream_t stream)
{
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return int(e);
    if (dev < 64 && configured[dev] == 0) {
        e = cudaFuncSetAttribute(meta_prepare_kernel<META_THREADS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(meta_smem_bytes(META_THREADS / 32, LORA_MAX_LORAS,
                                                     META_STAGE_MAX)));
        if (e != cudaSuccess) return int(e);
        e = cudaFuncSetAttribute(meta_prepare_kernel<META_SMALL_THREADS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(meta_smem_bytes(META_SMALL_THREADS / 32, LORA_MAX_LORAS,
                                                     META_SMALL_MAX)));
        if (e != cudaSuccess) return int(e);
        e = cudaFuncSetAttribute(meta_multi_kernel<META_MULTI_THREADS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(meta_multi_smem_bytes(META_MULTI_THREADS / 32,
                                                           LORA_MAX_LORAS)));
        if (e != cudaSuccess) return int(e);
        e = cudaFuncSetAttribute(meta_multi_kernel<META_MULTI_SMALL_THREADS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(meta_multi_smem_bytes(META_MULTI_SMALL_THREADS / 32,
                                                           LORA_MAX_LORAS)));
        if (e != cudaSuccess) return int(e);
        const int csm = int(meta_cluster_smem_bytes(LORA_MAX_LORAS));
        e = cudaFuncSetAttribute(meta_cluster_kernel<META_MULTI_THREADS, 1>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, csm);
        if (e != cudaSuccess) return int(e);
        e = cudaFuncSetAttribute(meta_cluster_kernel<META_MULTI_THREADS, 2>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, csm);
        if (e != cudaSuccess) return int(e);
        e = cudaFuncSetAttribute(meta_cluster_kernel<META_MULTI_THREADS, 4>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, csm);
        if (e != cudaSuccess) return int(e);
        configured[dev] = 1;
    }
    // Batches above META_MULTI_MIN tokens on one CTA per run of 256 or 1024
    // tokens (LORA_PUNICA_META_MULTI=0 turns it off).
    if (a.num_tokens > META_MULTI_MIN && knobs().meta_multi) {
        if (a.num_tokens <= META_MULTI_BIG) {
            constexpr int NT = META_MULTI_SMALL_THREADS;
            return int(launch_kernel(meta_multi_kernel<NT>, dim3((a.num_tokens + NT - 1) / NT),
                                     dim3(NT), meta_multi_smem_bytes(NT / 32, a.max_loras),
                                     stream, a));
        }
        // up to META_CLUSTER_MAX tokens: one cluster of at most 8 CTAs
        // (LORA_PUNICA_META_CLUSTER=0 keeps the plain multi-CTA kernel)
        if (a.num_tokens <= META_CLUSTER_MAX && knobs().meta_cluster) {
            const int t = a.num_tokens;
            e = t <= 8 * 1024    ? launch_meta_cluster<1>(a, stream)
                : t <= 16 * 1024 ? launch_meta_cluster<2>(a, stream)
                                 : launch_meta_cluster<4>(a, stream);
            if (e == cudaSuccess) return 0;
            (void)cudaGetLastError();          // a cluster that cannot be placed: plain kernel
        }
        constexpr int NT = META_MULTI_THREADS;
        return int(launch_kernel(meta_multi_kernel<NT>, dim3((a.num_tokens + NT - 1) / NT),
                                 dim3(NT), meta_multi_smem_bytes(NT / 32, a.max_loras), stream,
                                 a));
    }
    // Small batches on 8 warps (fewer warps to pass each barrier), the rest
    // on 32.  LORA_PUNICA_META_SMALL=0 always takes 32 warps.
    if (a.num_tokens <= META_SMALL_MAX && knobs().meta_small) {
        const size_t smem = meta_smem_bytes(META_SMALL_THREADS / 32, a.max_loras, a.num_tokens);
        return int(launch_kernel(meta_prepare_kernel<META_SMALL_THREADS>, dim3(1),
                                 dim3(META_SMALL_THREADS), smem, stream, a));
    }
    const size_t smem = meta_smem_bytes(META_THREADS / 32, a.max_loras, a.num_tokens);
    return int(launch_kernel(meta_prepare_kernel<META_THREADS>, dim3(1), dim3(META_THREADS), smem,
                             stream, a));
}

}  // namespace lora

LORA_API int lora_meta_prepare(const int32_t *token_lora_mapping, int32_t num_tokens,
                               const lora_meta_t *meta, void *stream)
{
    lora::NvtxRange nvtx_range("lora_meta_prepare");
    if (meta == nullptr) return LORA_ERR_NULL;
    if (!meta->token_lora_mapping || !meta->token_indices_sorted_by_lora_ids ||
        !meta->num_tokens_per_lora || !meta->lora_token_start_loc ||
        !meta->active_lora_ids || !meta->no_lora_flag || !meta->error_word)
        return LORA_ERR_NULL;
    if (meta->max_loras < 1 || meta->max_loras > LORA_MAX_LORAS) return LORA_ERR_SIZE;
    if (meta->max_num_tokens < 0 || num_tokens < 0) return LORA_ERR_SIZE;
    if (num_tokens > meta->max_num_tokens) return LORA_ERR_TOKENS;
    if (num_tokens > 0 && token_lora_mapping == nullptr) return LORA_ERR_NULL;

    lora::MetaArgs a;
    a.map = token_lora_mapping;
    a.num_tokens = num_tokens;
    a.max_loras = meta->max_loras;
    a.mapping_copy = meta->token_lora_mapping;
    a.sorted = meta->token_indices_sorted_by_lora_ids;
    a.counts = meta->num_tokens_per_lora;
    a.start_loc = meta->lora_token_start_loc;
    a.active = meta->active_lora_ids;
    a.no_lora = meta->no_lora_flag;
    a.error_word = meta->error_word;
    return lora::launch_meta_prepare(a, static_cast<cudaStream_t>(stream));
}
