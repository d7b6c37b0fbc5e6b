// lora_api.cu -- library-wide C entry points (status names, version, the
// host read of the no-LoRA flag) and the host helpers the launchers share.
#include <stdlib.h>

#include "lora_common.cuh"

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

// Programmatic dependent launch is on unless LORA_PUNICA_PDL=0 is set in
// the environment (read once).
bool pdl_enabled()
{
    static int cached = -1;
    if (cached < 0) {
        const char *v = getenv("LORA_PUNICA_PDL");
        cached = (v != nullptr && v[0] == '0') ? 0 : 1;
    }
    return cached == 1;
}

// Integer tuning knob from the environment (read at every call; the
// callers cache what they need).
int env_int(const char *name, int fallback)
{
    const char *v = getenv(name);
    if (v == nullptr || *v == 0) return fallback;
    return atoi(v);
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
