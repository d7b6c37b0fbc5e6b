// lora_meta.cu -- metadata step (page "vllm.lora.ops.triton_ops.
// lora_kernel_metadata", LoRAKernelMeta._reset + prepare_tensors) as one
// single-CTA kernel: the id map staged in shared memory, per-warp bin
// histograms (shared-memory atomic adds), a warp-shuffle scan over
// (bin, warp), and a stable counting-sort scatter (lanes of one bin ranked
// with __match_any_sync).
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

size_t meta_smem_bytes(int warps, int max_loras, int num_tokens)
{
    const size_t nb = size_t(max_loras) + 1;
    const size_t staged = num_tokens <= META_STAGE_MAX ? size_t(num_tokens) : 0;
    return (size_t(warps) * nb + 3 * nb + staged) * sizeof(int32_t);
}

// Bin of one token; counts an invalid id into `bad`.
__device__ __forceinline__ int token_bin(int32_t id, int32_t max_loras, int &bad)
{
    if (id >= 0 && id < max_loras) return id + 1;
    if (id != -1) ++bad;
    return 0;
}

template <int NT>
__global__ void __launch_bounds__(NT, 1) meta_prepare_kernel(MetaArgs a)
{
    constexpr int META_WARPS = NT / 32;
    extern __shared__ int32_t sm[];
    const int nb = a.max_loras + 1;
    int32_t *cnt = sm;                          // [META_WARPS][nb]: count, then offset
    int32_t *tot = cnt + META_WARPS * nb;       // [nb] tokens per bin
    int32_t *base = tot + nb;                   // [nb] first sorted slot of the bin
    int32_t *pos = base + nb;                   // [nb] index among non-empty bins
    int32_t *ids_s = pos + nb;                  // [T] the map, when staged
    __shared__ int32_t s_invalid, s_nactive;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int T = a.num_tokens;

    pdl_wait();
    pdl_launch_dependents();

    const bool staged = T <= META_STAGE_MAX;
    if (staged)
        for (int t = tid; t < T; t += NT) ids_s[t] = a.map[t];
    const int32_t *ids = staged ? ids_s : a.map;
    for (int i = tid; i < META_WARPS * nb; i += NT) cnt[i] = 0;
    if (tid == 0) s_invalid = 0;
    __syncthreads();

    // Each warp owns tokens [t0, t1), a multiple of 32 long (the last may be short).
    const int per_warp = ((T + NT - 1) / NT) * 32;
    const int t0 = min(T, warp * per_warp);
    const int t1 = min(T, t0 + per_warp);

    // Pass 1: per-warp histogram, one shared-memory atomic add per token
    // (counts only: pass 2 keeps the order).  Measured faster than grouping
    // lanes with __match_any_sync, whose cost grows with the number of
    // distinct ids in a warp.
    int bad = 0;
    for (int g = t0; g < t1; g += 32) {
        const int t = g + lane;
        const bool has = t < t1;
        const int b = has ? token_bin(ids[t], a.max_loras, bad) : -1;
        if (has) atomicAdd(&cnt[warp * nb + b], 1);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if (lane == 0 && bad) atomicAdd(&s_invalid, bad);
    __syncthreads();

    // Per bin, exclusive scan over warps (warp order = token order).
    for (int b = tid; b < nb; b += NT) {
        int run = 0;
        for (int w = 0; w < META_WARPS; ++w) {
            const int c = cnt[w * nb + b];
            cnt[w * nb + b] = run;
            run += c;
        }
        tot[b] = run;
    }
    __syncthreads();

    // Exclusive scans over bins: first sorted slot, and rank among the
    // non-empty bins (torch.unique(sorted=True) order).
    if (warp == 0) {
        int carry_t = 0, carry_p = 0;
        for (int b0 = 0; b0 < nb; b0 += 32) {
            const int b = b0 + lane;
            const int v = (b < nb) ? tot[b] : 0;
            const int f = v > 0 ? 1 : 0;
            int iv = v, jf = f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, iv, o);
                const int w = __shfl_up_sync(0xffffffffu, jf, o);
                if (lane >= o) { iv += u; jf += w; }
            }
            if (b < nb) {
                base[b] = carry_t + iv - v;
                pos[b] = carry_p + jf - f;
            }
            carry_t += __shfl_sync(0xffffffffu, iv, 31);
            carry_p += __shfl_sync(0xffffffffu, jf, 31);
        }
        if (lane == 0) s_nactive = carry_p;
    }
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

    // Pass 2: stable scatter + mapping copy.
    int unused = 0;
    for (int g = t0; g < t1; g += 32) {
        const int t = g + lane;
        const bool has = t < t1;
        const int32_t id = has ? ids[t] : -1;
        const int b = has ? token_bin(id, a.max_loras, unused) : -1;
        const unsigned grp = __match_any_sync(0xffffffffu, b);
        const int rank = __popc(grp & ((1u << lane) - 1u));
        if (has) {
            a.sorted[base[b] + cnt[warp * nb + b] + rank] = t;
            a.mapping_copy[t] = id;
        }
        __syncwarp();
        if (has && rank == 0) cnt[warp * nb + b] += __popc(grp);
        __syncwarp();
    }
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
        configured[dev] = 1;
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
