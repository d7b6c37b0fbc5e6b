// lora_api.cu -- library-wide C entry points (status names, version, the
// host read of the no-LoRA flag) and the host helpers the launchers share.
#include <stdlib.h>

#include <mutex>

#include "lora_common.cuh"
#include "lora_umma.cuh"

namespace lora {

int device_sm_count()
{
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        n = 1;
    if (dev < 64) cache[dev] = n;
    return n;
}

static int env_int(const char *name, int fallback)
{
    const char *v = getenv(name);
    if (v == nullptr || *v == 0) return fallback;
    return atoi(v);
}

static Knobs read_knobs()
{
    Knobs k;
    k.pdl = env_int("LORA_PUNICA_PDL", 1);
    k.coop = env_int("LORA_PUNICA_COOP", -1);
    k.fused = env_int("LORA_PUNICA_FUSED", -1);
    k.fused_max_tokens = env_int("LORA_PUNICA_FUSED_MAX_TOKENS", 128);
    k.self_meta = env_int("LORA_PUNICA_SELF_META", -1);
    k.umma = env_int("LORA_PUNICA_UMMA", 1);
    k.umma_min_tokens = env_int("LORA_PUNICA_UMMA_MIN_TOKENS", 1024);
    k.umma_min_cols = env_int("LORA_PUNICA_UMMA_MIN_COLS", 256);
    k.umma_partial = env_int("LORA_PUNICA_UMMA_PARTIAL", 1);
    k.umma_pair = env_int("LORA_PUNICA_UMMA_PAIR", 0);
    k.nvtx = env_int("LORA_PUNICA_NVTX", 1);
    k.early_shrink_ctas = env_int("LORA_PUNICA_EARLY_SHRINK_CTAS", 2);
    k.expand_tc = env_int("LORA_PUNICA_EXPAND_TC", -1);
    k.expand_tc_min_rank = env_int("LORA_PUNICA_EXPAND_TC_MIN_RANK", 64);
    k.meta_small = env_int("LORA_PUNICA_META_SMALL", 1);
    k.meta_multi = env_int("LORA_PUNICA_META_MULTI", 1);
    k.meta_cluster = env_int("LORA_PUNICA_META_CLUSTER", 1);
    k.linear_tc = env_int("LORA_PUNICA_LINEAR_TC", -1);
    k.linear_tc_min_tokens = env_int("LORA_PUNICA_LINEAR_TC_MIN_TOKENS", 0);
    k.coop_test_extra = env_int("LORA_PUNICA_COOP_TEST_EXTRA_ARRIVALS", 0);
    k.coop_test_timeout = env_int("LORA_PUNICA_COOP_TEST_TIMEOUT_CYCLES", 0);
    return k;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

bool encode_tile_map(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols,
                     uint64_t row_stride, uint32_t box_cols, uint32_t box_rows,
                     CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_stride * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tile_map_f32(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols,
                         uint64_t row_stride, uint32_t box_cols, uint32_t box_rows,
                         CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_stride * 4};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_perm_rows_map(CUtensorMap *m, const void *ptr, uint64_t rows, uint32_t rank,
                          uint32_t box_k, uint32_t blocks, CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr || rows % 64 != 0) return false;
    // dims (innermost first): k, e, t, i, 64-row block; global row
    // 64 * blk + 16 * t + 2 * i + e; the box's shared-memory image takes the
    // dims in order, so shared row 64 * blk + 8 * i + 2 * t + e.
    const cuuint64_t row = uint64_t(rank) * 2;
    const cuuint64_t dims[5] = {rank, 2, 4, 8, rows / 64};
    const cuuint64_t strides[4] = {row, 16 * row, 2 * row, 64 * row};
    const cuuint32_t box[5] = {box_k, 2, 4, 8, blocks};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static Knobs g_knobs;
static std::once_flag g_knobs_once;

const Knobs &knobs()
{
    std::call_once(g_knobs_once, [] { g_knobs = read_knobs(); });
    return g_knobs;
}

}  // namespace lora

LORA_API const char *lora_status_string(int status)
{
    switch (status) {
    case LORA_OK: return "ok";
    case LORA_ERR_NULL: return "a required pointer is NULL";
    case LORA_ERR_SIZE: return "a size is negative or out of range";
    case LORA_ERR_ALIGN: return "a pointer or stride breaks the 16-byte alignment rule";
    case LORA_ERR_RANK: return "rank must be a multiple of 8 in [8, 128]";
    case LORA_ERR_SLICES: return "num_slices must be in [1, 8]";
    case LORA_ERR_TOKENS: return "num_tokens exceeds meta->max_num_tokens";
    case LORA_ERR_WIDTH: return "offset_start + sum(slice_sizes) exceeds y_ld";
    case LORA_ERR_DEVICE: return "no usable CUDA device";
    case LORA_ERR_SCRATCH: return "num_slices * num_tokens * rank exceeds the fixed buffer of lora_linear_noalloc";
    default: break;
    }
    if (status > 0) return cudaGetErrorString(static_cast<cudaError_t>(status));
    return "unknown status";
}

LORA_API int lora_version(void) { return LORA_PUNICA_VERSION; }

// Host copy of the flag, as LoRAKernelMeta.no_lora_flag_cpu on the page
// "vllm.lora.ops.triton_ops.lora_kernel_metadata": one 4-byte copy ordered
// after the metadata step on `stream`, then a synchronisation.
LORA_API int lora_meta_read_no_lora(const lora_meta_t *meta, void *stream, int32_t *no_lora)
{
    if (meta == nullptr || meta->no_lora_flag == nullptr || no_lora == nullptr)
        return LORA_ERR_NULL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, meta->no_lora_flag, sizeof(v), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return int(e);
    *no_lora = v != 0 ? 1 : 0;
    return LORA_OK;
}

// Re-reads the LORA_PUNICA_* tuning variables (otherwise read once, at the
// first call).  Not to be called while another thread calls the library.
LORA_API void lora_reload_options(void)
{
    lora::knobs();
    lora::g_knobs = lora::read_knobs();
}
