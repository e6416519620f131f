// noalloc.cu -- decode attention for callers that cannot allocate device memory.
//
// kv_attn_decode needs scratch space for its split-T partial states, and the
// caller normally allocates it (kv_attn_workspace_size bytes).  Some callers
// cannot: code that runs while a stream is being captured into a CUDA graph
// (an allocation there is not recorded and cudaMalloc synchronizes the
// device), plugins hosted by an engine that owns every device allocation, or
// real-time loops that must never block in the allocator.  For them this file
// provides kv_attn_decode_noalloc, which keeps the scratch in a fixed array
// that lives in the library's own device memory.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes.  Every
// GPU on which the library's module is loaded holds it until the process
// exits.  Host code cannot use the array's name as a device address; the
// device address is looked up once per device with cudaGetSymbolAddress, with
// that device current, and passed to the kernels as their workspace.
#include "kvq_internal.cuh"

#include <mutex>

// 32 MiB.  The tensor-core decode balances a batch over whole waves of CTAs,
// each wave 76 * ceil(batch / 76) work items for KV8 (38 * ceil(batch / 38)
// for TQ4), each item keeping heads x 514 floats; this entry takes as many
// waves (up to the regular entry's 4) as fit, so at 128 heads it covers
// batches of up to 76 sequences (KV8) or 114 (TQ4) whatever their lengths.
static constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices];

// Device address of g_decode_scratch on the current device (set up on first use).
kvq_status scratch_on_current_device(void** addr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KVQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return KVQ_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kv_attn_decode_noalloc(kvq_format fmt, const kvq_mla_layout* layout, const void* q,
                                             kvq_dtype q_dtype, int32_t batch, int32_t n_heads, const uint8_t* codes,
                                             const float* scales, const int64_t* cu_seqlens, int64_t max_total_rows,
                                             float sm_scale, float* out, kvq_path path, void* stream) {
    if (batch < 0 || n_heads < 0 || max_total_rows < 0) return KVQ_ERR_ARG;
    if (batch == 0 || n_heads == 0) return KVQ_OK;
    // the largest wave budget whose workspace fits the scratch
    int waves = kvq::kDecodeWaves;
    size_t need = kvq::attn_workspace_size_waves(fmt, layout, batch, n_heads, max_total_rows, path, waves);
    while (need > kNoAllocScratchBytes && waves > 1)
        need = kvq::attn_workspace_size_waves(fmt, layout, batch, n_heads, max_total_rows, path, --waves);
    if (need == 0) {
        // invalid or unsupported arguments: let the regular entry point name the
        // reason without touching any memory (its checks run before the workspace check)
        return kv_attn_decode(fmt, layout, q, q_dtype, batch, n_heads, codes, scales, cu_seqlens, max_total_rows,
                              sm_scale, out, nullptr, 0, path, stream);
    }
    if (need > kNoAllocScratchBytes) return KVQ_ERR_WORKSPACE;
    void* scratch = nullptr;
    const kvq_status s = scratch_on_current_device(&scratch);
    if (s != KVQ_OK) return s;
    return kvq::attn_decode_waves(fmt, layout, q, q_dtype, batch, n_heads, codes, scales, cu_seqlens, max_total_rows,
                                  sm_scale, out, scratch, kNoAllocScratchBytes, path, stream, waves);
}
