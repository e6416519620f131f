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
// device address is looked up with cudaGetSymbolAddress, with the device
// current, once per device context (a context re-created after a device reset
// loads the module again, so the address is looked up again), and passed to
// the kernels as their workspace.
#include <cuda.h>

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
unsigned long long g_scratch_ctx[kMaxDevices];   // id of the context the address belongs to

// The two driver calls that identify the current context, taken through the
// runtime's entry-point query so that the library does not link the driver
// (it loads on machines without one; nothing here runs there).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// Id of the current context, creating the device's primary context when this
// thread has none yet.  Called with g_scratch_mutex held.
kvq_status current_context_id(unsigned long long* id) {
    if (!g_ctx_get_current || !g_ctx_get_id) {
        void* f0 = nullptr;
        void* f1 = nullptr;
        cudaDriverEntryPointQueryResult q0{}, q1{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 12000, cudaEnableDefault, &q0) != cudaSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
            q0 != cudaDriverEntryPointSuccess || q1 != cudaDriverEntryPointSuccess || !f0 || !f1)
            return KVQ_ERR_CUDA;
        g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f0);
        g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f1);
    }
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return KVQ_ERR_CUDA;
    if (ctx == nullptr) {
        // no context on this thread yet: the lookup makes the device's primary context current
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return KVQ_ERR_CUDA;
        if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return KVQ_ERR_CUDA;
    }
    return g_ctx_get_id(ctx, id) == CUDA_SUCCESS ? KVQ_OK : KVQ_ERR_CUDA;
}

// Device address of g_decode_scratch on the current device (looked up on first
// use in each context of the device).
kvq_status scratch_on_current_device(void** addr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KVQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    unsigned long long id = 0;
    const kvq_status cs = current_context_id(&id);
    if (cs != KVQ_OK) return cs;
    if (g_scratch_addr[dev] == nullptr || g_scratch_ctx[dev] != id) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return KVQ_ERR_CUDA;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = id;
    }
    *addr = g_scratch_addr[dev];
    return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kv_attn_decode_noalloc(kvq_format fmt, const kvq_mla_layout* layout, const void* q,
                                             kvq_dtype q_dtype, int32_t batch, int32_t n_heads, const uint8_t* codes,
                                             const float* scales, const int64_t* cu_seqlens, int64_t max_total_rows,
                                             float sm_scale, float* out, kvq_path path, void* stream) {
    // the regular entry point's argument checks, in its order: without a
    // workspace it returns KVQ_ERR_WORKSPACE exactly when every argument is
    // valid (and KVQ_OK for an empty batch), launching nothing either way
    const kvq_status pre = kvq::attn_decode_waves(fmt, layout, q, q_dtype, batch, n_heads, codes, scales, cu_seqlens,
                                                  max_total_rows, sm_scale, out, nullptr, 0, path, stream,
                                                  kvq::decode_waves(fmt));
    if (pre != KVQ_ERR_WORKSPACE) return pre;
    // the largest wave budget whose workspace fits the scratch
    int waves = kvq::decode_waves(fmt);
    size_t need = kvq::attn_workspace_size_waves(fmt, layout, batch, n_heads, max_total_rows, path, waves);
    while (need > kNoAllocScratchBytes && waves > 1)
        need = kvq::attn_workspace_size_waves(fmt, layout, batch, n_heads, max_total_rows, path, --waves);
    if (need == 0 || need > kNoAllocScratchBytes) return KVQ_ERR_WORKSPACE;
    void* scratch = nullptr;
    const kvq_status s = scratch_on_current_device(&scratch);
    if (s != KVQ_OK) return s;
    return kvq::attn_decode_waves(fmt, layout, q, q_dtype, batch, n_heads, codes, scales, cu_seqlens, max_total_rows,
                                  sm_scale, out, scratch, kNoAllocScratchBytes, path, stream, waves);
}
