// lora_noalloc.cu -- lora_linear for callers that cannot allocate device
// memory.
//
// lora_linear needs an fp32 buffer of num_slices x num_tokens x rank floats
// between its shrink and its expand.  Some callers cannot provide one: code
// that runs where cudaMalloc is unavailable or forbidden (inside a custom
// allocator or memory-pool callback, in a plugin whose host framework owns
// every allocation, or in a process that must not grow its footprint after
// start-up).  lora_linear_noalloc keeps that buffer in a fixed array of
// device memory that belongs to this library: it calls no allocator, and the
// caller passes only its inputs and outputs.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (LORA_NOALLOC_MAX_FLOATS floats) until the process exits.
// Host code cannot use the array's name as a device address; the first call
// on each device looks the address up with cudaGetSymbolAddress while that
// device is current (so make that first call before any stream capture), and
// later calls reuse it.  Every call on a device shares the one array: calls
// that overlap on the GPU (other streams, other threads) race on it and must
// be serialised by the caller.  Each call clears the part it uses before the
// shrink accumulates into it.
#include <atomic>

#include "lora_common.cuh"

namespace lora {

static __device__ __align__(256) float g_noalloc_buf[LORA_NOALLOC_MAX_FLOATS];

// Per-device address of g_noalloc_buf (host threads may race to fill an
// entry; they all store the same value).
static std::atomic<float *> noalloc_ptr[64];

}  // namespace lora

LORA_API int lora_linear_noalloc(const int32_t *token_lora_mapping, int32_t num_tokens,
                                 const lora_bf16_t *x, int32_t hidden, int64_t x_ld,
                                 const lora_bf16_t *const *lora_a,
                                 const lora_bf16_t *const *lora_b,
                                 const lora_bf16_t *const *lora_bias,
                                 const int32_t *slice_sizes, int32_t num_slices, int32_t rank,
                                 float scale, lora_bf16_t *y, int64_t y_ld,
                                 const lora_meta_t *meta, void *stream)
{
    lora::NvtxRange nvtx_range("lora_linear_noalloc");
    if (num_slices < 1 || num_slices > LORA_MAX_SLICES) return LORA_ERR_SLICES;
    if (rank < 8 || rank > LORA_MAX_RANK || rank % 8 != 0) return LORA_ERR_RANK;
    if (num_tokens < 0) return LORA_ERR_SIZE;
    const int64_t floats = int64_t(num_slices) * num_tokens * rank;
    if (floats > LORA_NOALLOC_MAX_FLOATS) return LORA_ERR_SCRATCH;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return int(e);
    if (dev < 0 || dev >= 64) return LORA_ERR_DEVICE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The array is looked up for the current device, so the stream must
    // belong to it (a stream of another GPU would be handed this GPU's array).
    if (st != nullptr) {
        int sdev = -1;
        e = cudaStreamGetDevice(st, &sdev);
        if (e != cudaSuccess) return int(e);
        if (sdev != dev) return LORA_ERR_DEVICE;
    }
    float *buf = lora::noalloc_ptr[dev].load(std::memory_order_acquire);
    if (buf == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, lora::g_noalloc_buf);
        if (e != cudaSuccess) return int(e);
        buf = static_cast<float *>(p);
        lora::noalloc_ptr[dev].store(buf, std::memory_order_release);
    }
    if (floats > 0) {
        e = cudaMemsetAsync(buf, 0, size_t(floats) * sizeof(float), st);
        if (e != cudaSuccess) return int(e);
    }
    return lora_linear(token_lora_mapping, num_tokens, x, hidden, x_ld, lora_a, lora_b, lora_bias,
                       slice_sizes, num_slices, rank, scale, buf, y, y_ld, meta, stream);
}
