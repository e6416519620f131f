// abi.cu -- the extern "C" entry points declared in include/kvq.h.
//
// Every call validates its arguments on the host and only then launches; a
// failed check returns a status and launches nothing.  No call allocates or
// frees device memory.
#include "kvq_internal.cuh"
#include "pq_common.cuh"

#include <algorithm>
#include <math.h>

using namespace kvq;

namespace {

constexpr int kMaxD = 4096;

bool is_pow2_ge2(int n) { return n >= 2 && (n & (n - 1)) == 0; }

kvq_status check_layout(const kvq_mla_layout* L) {
    if (!L) return KVQ_ERR_ARG;
    if (L->n_blocks < 1 || L->n_blocks > 2) return KVQ_ERR_ARG;
    for (int b = 0; b < L->n_blocks; ++b)
        if (L->block_dim[b] <= 0) return KVQ_ERR_ARG;
    const int D = L->block_dim[0] + (L->n_blocks > 1 ? L->block_dim[1] : 0);
    if (D > kMaxD) return KVQ_ERR_UNSUPPORTED;
    return KVQ_OK;
}

int row_dim(const kvq_mla_layout* L) { return L->block_dim[0] + (L->n_blocks > 1 ? L->block_dim[1] : 0); }

kvq_status check_tq4_layout(const kvq_mla_layout* L) {
    kvq_status s = check_layout(L);
    if (s != KVQ_OK) return s;
    for (int b = 0; b < L->n_blocks; ++b)
        if (!is_pow2_ge2(L->block_dim[b])) return KVQ_ERR_SHAPE;
    for (int b = 0; b < L->n_blocks; ++b)
        if (L->block_dim[b] > 1024) return KVQ_ERR_UNSUPPORTED;
    if (row_dim(L) > 1024) return KVQ_ERR_UNSUPPORTED;   // 16 sign words
    return KVQ_OK;
}

// The attention kernels are written for the 576-dim MLA latent row.
// Vector widths the attention kernels read and write with: the code pool in
// 32-byte pieces (every row of a 32-byte aligned pool is, as 576 and 288 are
// multiples of 32), queries, outputs and new rows in 16 bytes, scales and the
// int64 arrays in 8.
static bool aligned(const void* p, uintptr_t n) { return ((uintptr_t)p & (n - 1)) == 0; }
static bool attn_pointers_aligned(const void* q, const uint8_t* codes, const float* scales, const int64_t* cu,
                                  const float* out) {
    return aligned(q, 16) && aligned(codes, 32) && aligned(scales, 8) && aligned(cu, 8) && aligned(out, 16);
}

bool is_tq(kvq_format fmt) { return fmt == KVQ_TQ4 || is_pq(fmt); }

kvq_status check_attn_layout(kvq_format fmt, const kvq_mla_layout* L) {
    kvq_status s = is_tq(fmt) ? check_tq4_layout(L) : (fmt == KVQ_KV8 ? check_layout(L) : KVQ_ERR_ARG);
    if (s != KVQ_OK) return s;
    if (L->v_dim != 512) return KVQ_ERR_UNSUPPORTED;
    const bool two = L->n_blocks == 2 && L->block_dim[0] == 512 && L->block_dim[1] == 64;
    const bool one = L->n_blocks == 1 && L->block_dim[0] == 576;
    if (is_tq(fmt) ? !two : !(two || one)) return KVQ_ERR_UNSUPPORTED;
    return KVQ_OK;
}

// The encoder of a format (err: the error word a non-finite row sets).
cudaError_t launch_encode(kvq_format fmt, const float* x, int64_t n_rows, const kvq_mla_layout& L,
                          const int64_t* dst_rows, uint8_t* codes, float* scales, int32_t* err, cudaStream_t st) {
    if (fmt == KVQ_KV8) return launch_kv8_encode(x, n_rows, L, dst_rows, codes, scales, err, st);
    if (fmt == KVQ_TQ4) return launch_tq4_encode(x, n_rows, L, dst_rows, codes, scales, err, st);
    return launch_pq_encode(pq_bits_of(fmt), x, n_rows, L, dst_rows, codes, scales, err, st);
}

int64_t format_row_bytes(kvq_format fmt, const kvq_mla_layout& L) {
    const int D = L.block_dim[0] + (L.n_blocks > 1 ? L.block_dim[1] : 0);
    if (fmt == KVQ_KV8) return D;
    if (fmt == KVQ_TQ4) return D / 2;
    return pq_row_bytes(pq_bits_of(fmt), L);
}

kvq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

kvq_status check_path(kvq_path path) {
    if (path != KVQ_PATH_AUTO && path != KVQ_PATH_SIMT && path != KVQ_PATH_TENSOR) return KVQ_ERR_ARG;
    return KVQ_OK;
}

// The attention family that runs: AUTO takes the tensor-core kernel when it
// supports the format and head count, else the SIMT kernel.  PolarQuant runs
// on the SIMT kernel unless the tensor path is asked for, which serves 4-bit
// rows (its f16 leaves carry a looser bound than the other tensor paths).
kvq_status resolve_path(kvq_format fmt, kvq_path path, const kvq_mla_layout* L, int32_t n_heads, kvq_path* out) {
    if (path == KVQ_PATH_SIMT || (path == KVQ_PATH_AUTO && is_pq(fmt))) {
        *out = KVQ_PATH_SIMT;
        return KVQ_OK;
    }
    const bool tc = (!is_pq(fmt) || fmt == KVQ_PQ4) && tc_supported(*L, n_heads);
    if (path == KVQ_PATH_TENSOR && !tc) return KVQ_ERR_UNSUPPORTED;
    *out = tc ? KVQ_PATH_TENSOR : KVQ_PATH_SIMT;
    return KVQ_OK;
}

// K2/V4 paths: the tensor-core kernel serves head_dim 128 and 256 (AUTO takes
// it there), the fp32 kernel every supported layout.
kvq_status check_k2v4_path(kvq_path path) { return check_path(path); }
static kvq_status resolve_k2v4_path(kvq_path path, const kvq_k2v4_layout* L, bool* tensor) {
    const bool tc = k2v4_tc_supported(*L);
    if (path == KVQ_PATH_TENSOR && !tc) return KVQ_ERR_UNSUPPORTED;
    *tensor = path == KVQ_PATH_SIMT ? false : tc;
    return KVQ_OK;
}

AttnPlan plan_decode(kvq_format fmt, kvq_path resolved, int32_t batch, int32_t n_heads, int64_t max_total_rows,
                     int waves) {
    return resolved == KVQ_PATH_TENSOR ? plan_decode_tc(fmt, batch, n_heads, max_total_rows, waves)
                                       : plan_decode_simt(batch, n_heads, max_total_rows);
}

kvq_status check_k2v4(const kvq_k2v4_layout* L) {
    if (!L) return KVQ_ERR_ARG;
    if (L->n_kv_heads <= 0 || L->head_dim <= 0 || L->n_sink < 0 || L->n_window < 0 || L->n_slack < 0)
        return KVQ_ERR_ARG;
    if (L->group != 32) return KVQ_ERR_UNSUPPORTED;
    if (L->head_dim % 32 != 0 || L->head_dim > 512) return KVQ_ERR_UNSUPPORTED;
    if (!(L->k_gain > 0.0f) || !isfinite(L->k_gain)) return KVQ_ERR_ARG;
    return KVQ_OK;
}

}  // namespace

extern "C" {

const char* kvq_status_string(kvq_status s) {
    switch (s) {
        case KVQ_OK: return "ok";
        case KVQ_ERR_ARG: return "invalid argument";
        case KVQ_ERR_SHAPE: return "TQ4 block width is not a power of two >= 2 (rows would all be inert)";
        case KVQ_ERR_WORKSPACE: return "workspace missing or too small";
        case KVQ_ERR_CUDA: return "CUDA launch or runtime error";
        case KVQ_ERR_UNSUPPORTED: return "arguments valid but not supported by this build";
        case KVQ_ERR_DEVICE: return "device error word set";
        case KVQ_ERR_MISMATCH: return "cache file of another tier, codec, bit width or layout: refused";
        case KVQ_ERR_IO: return "cache file missing, unreadable, corrupt or of the wrong size";
        case KVQ_ERR_NONFINITE: return "an encoder met a NaN or infinite value (device error word)";
        case KVQ_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out (device error word)";
    }
    return "unknown status";
}

const char* kvq_version(void) { return "0.1.0"; }

kvq_status kvq_codebook(int32_t which, float* levels, float* thresholds) {
    if (!levels || !thresholds) return KVQ_ERR_ARG;
    if (which == 16) {
        const Codebook16 c = tq4_codebook();
        for (int k = 0; k < 16; ++k) levels[k] = c.lv[k];
        for (int k = 0; k < 15; ++k) thresholds[k] = c.th[k];
        return KVQ_OK;
    }
    if (which == 4) {
        const Codebook4 c = k2_codebook();
        for (int k = 0; k < 4; ++k) levels[k] = c.lv[k];
        for (int k = 0; k < 3; ++k) thresholds[k] = c.th[k];
        return KVQ_OK;
    }
    return KVQ_ERR_ARG;
}

kvq_status kv8_encode(const float* x, int64_t n_rows, const kvq_mla_layout* layout, const int64_t* dst_rows,
                      uint8_t* codes, float* scales, int32_t* err_word, void* stream) {
    kvq_status s = check_layout(layout);
    if (s != KVQ_OK) return s;
    if (n_rows < 0) return KVQ_ERR_ARG;
    if (n_rows == 0) return KVQ_OK;
    if (!x || !codes || !scales) return KVQ_ERR_ARG;
    return cuda_status(launch_kv8_encode(x, n_rows, *layout, dst_rows, codes, scales, err_word, (cudaStream_t)stream));
}

kvq_status tq4_encode(const float* x, int64_t n_rows, const kvq_mla_layout* layout, const int64_t* dst_rows,
                      uint8_t* packed, float* scales, int32_t* err_word, void* stream) {
    kvq_status s = check_tq4_layout(layout);
    if (s != KVQ_OK) return s;
    if (n_rows < 0) return KVQ_ERR_ARG;
    if (n_rows == 0) return KVQ_OK;
    if (!x || !packed || !scales) return KVQ_ERR_ARG;
    return cuda_status(
        launch_tq4_encode(x, n_rows, *layout, dst_rows, packed, scales, err_word, (cudaStream_t)stream));
}

kvq_status pq_encode(kvq_format fmt, const float* x, int64_t n_rows, const kvq_mla_layout* layout,
                     const int64_t* dst_rows, uint8_t* codes, float* radii, int32_t* err_word, void* stream) {
    if (!is_pq(fmt)) return KVQ_ERR_ARG;
    kvq_status s = check_tq4_layout(layout);
    if (s != KVQ_OK) return s;
    if (n_rows < 0) return KVQ_ERR_ARG;
    if (n_rows == 0) return KVQ_OK;
    if (!x || !codes || !radii) return KVQ_ERR_ARG;
    return cuda_status(launch_pq_encode(pq_bits_of(fmt), x, n_rows, *layout, dst_rows, codes, radii, err_word,
                                        (cudaStream_t)stream));
}

kvq_status pq_decode(kvq_format fmt, const uint8_t* codes, const float* radii, int64_t n_rows,
                     const kvq_mla_layout* layout, int32_t rotated, float* out, void* stream) {
    if (!is_pq(fmt)) return KVQ_ERR_ARG;
    kvq_status s = check_tq4_layout(layout);
    if (s != KVQ_OK) return s;
    if (n_rows < 0) return KVQ_ERR_ARG;
    if (n_rows == 0) return KVQ_OK;
    if (!codes || !radii || !out) return KVQ_ERR_ARG;
    return cuda_status(
        launch_pq_decode(pq_bits_of(fmt), codes, radii, n_rows, *layout, rotated != 0, out, (cudaStream_t)stream));
}

int64_t kvq_row_bytes(kvq_format fmt, const kvq_mla_layout* layout) {
    if (fmt == KVQ_KV8) {
        if (check_layout(layout) != KVQ_OK) return 0;
    } else if (is_tq(fmt)) {
        if (check_tq4_layout(layout) != KVQ_OK) return 0;
    } else {
        return 0;
    }
    return format_row_bytes(fmt, *layout);
}

kvq_status kvq_pq_codebook(int32_t bits, int32_t level, float* centroids, float* thresholds) {
    if (!centroids || !thresholds) return KVQ_ERR_ARG;
    return pq_host_codebook(bits, level, centroids, thresholds) ? KVQ_OK : KVQ_ERR_ARG;
}

kvq_status tq4_rotate(const void* in, kvq_dtype in_dtype, int64_t n_vecs, const kvq_mla_layout* layout,
                      int32_t inverse, float* out, void* stream) {
    kvq_status s = check_tq4_layout(layout);
    if (s != KVQ_OK) return s;
    if (n_vecs < 0 || (in_dtype != KVQ_F32 && in_dtype != KVQ_BF16)) return KVQ_ERR_ARG;
    if (n_vecs == 0) return KVQ_OK;
    if (!in || !out) return KVQ_ERR_ARG;
    return cuda_status(launch_tq4_rotate(in, in_dtype, n_vecs, *layout, inverse, out, (cudaStream_t)stream));
}

}  // extern "C"

namespace kvq {

size_t attn_workspace_size_waves(kvq_format fmt, const kvq_mla_layout* layout, int32_t batch, int32_t n_heads,
                                 int64_t max_total_rows, kvq_path path, int waves) {
    if (check_attn_layout(fmt, layout) != KVQ_OK || check_path(path) != KVQ_OK) return 0;
    if (batch < 0 || n_heads < 0 || max_total_rows < 0) return 0;
    kvq_path rp;
    if (resolve_path(fmt, path, layout, n_heads, &rp) != KVQ_OK) return 0;
    const AttnPlan pl = plan_decode(fmt, rp, batch, n_heads, max_total_rows, waves);
    return kWsHeader + partial_bytes(pl.max_items, n_heads, layout->v_dim);
}

kvq_status attn_decode_waves(kvq_format fmt, const kvq_mla_layout* layout, const void* q, kvq_dtype q_dtype,
                             int32_t batch, int32_t n_heads, const uint8_t* codes, const float* scales,
                             const int64_t* cu_seqlens, int64_t max_total_rows, float sm_scale, float* out,
                             void* workspace, size_t workspace_bytes, kvq_path path, void* stream, int waves) {
    kvq_status s = check_attn_layout(fmt, layout);
    if (s != KVQ_OK) return s;
    if ((s = check_path(path)) != KVQ_OK) return s;
    if (batch < 0 || n_heads < 0 || max_total_rows < 0 || (q_dtype != KVQ_F32 && q_dtype != KVQ_BF16))
        return KVQ_ERR_ARG;
    if (batch > 65535 || n_heads > 65535) return KVQ_ERR_UNSUPPORTED;
    if (batch == 0 || n_heads == 0) return KVQ_OK;
    kvq_path rp;
    if ((s = resolve_path(fmt, path, layout, n_heads, &rp)) != KVQ_OK) return s;
    if (!q || !cu_seqlens || !out) return KVQ_ERR_ARG;
    if (max_total_rows > 0 && (!codes || !scales)) return KVQ_ERR_ARG;
    if (!attn_pointers_aligned(q, codes, scales, cu_seqlens, out)) return KVQ_ERR_ARG;
    if (!isfinite(sm_scale)) return KVQ_ERR_ARG;
    const size_t need = attn_workspace_size_waves(fmt, layout, batch, n_heads, max_total_rows, path, waves);
    if (!workspace || workspace_bytes < need) return KVQ_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const AttnPlan pl = plan_decode(fmt, rp, batch, n_heads, max_total_rows, waves);
    if (rp == KVQ_PATH_TENSOR)
        return cuda_status(launch_attn_tc(fmt, *layout, q, q_dtype, batch, n_heads, codes, scales, cu_seqlens, -1, pl,
                                          sm_scale, out, workspace, st));
    return cuda_status(launch_attn_simt(fmt, *layout, q, q_dtype, batch, n_heads, codes, scales, cu_seqlens, -1, pl,
                                        sm_scale, out, workspace, st));
}

}  // namespace kvq

extern "C" {

size_t kv_attn_workspace_size(kvq_format fmt, const kvq_mla_layout* layout, int32_t batch, int32_t n_heads,
                              int64_t max_total_rows, kvq_path path) {
    return attn_workspace_size_waves(fmt, layout, batch, n_heads, max_total_rows, path, decode_waves(fmt));
}

kvq_status kv_attn_decode(kvq_format fmt, const kvq_mla_layout* layout, const void* q, kvq_dtype q_dtype,
                          int32_t batch, int32_t n_heads, const uint8_t* codes, const float* scales,
                          const int64_t* cu_seqlens, int64_t max_total_rows, float sm_scale, float* out,
                          void* workspace, size_t workspace_bytes, kvq_path path, void* stream) {
    return attn_decode_waves(fmt, layout, q, q_dtype, batch, n_heads, codes, scales, cu_seqlens, max_total_rows,
                             sm_scale, out, workspace, workspace_bytes, path, stream, decode_waves(fmt));
}

kvq_status kv_attn_decode_append(kvq_format fmt, const kvq_mla_layout* layout, const float* x_new,
                                 const int64_t* dst_rows, const void* q, kvq_dtype q_dtype, int32_t batch,
                                 int32_t n_heads, uint8_t* codes, float* scales, const int64_t* cu_seqlens,
                                 int64_t max_total_rows, float sm_scale, float* out, void* workspace,
                                 size_t workspace_bytes, kvq_path path, void* stream) {
    kvq_status s = check_attn_layout(fmt, layout);
    if (s != KVQ_OK) return s;
    if ((s = check_path(path)) != KVQ_OK) return s;
    if (batch < 0 || n_heads < 0 || max_total_rows < 0 || (q_dtype != KVQ_F32 && q_dtype != KVQ_BF16))
        return KVQ_ERR_ARG;
    if (batch > 65535 || n_heads > 65535) return KVQ_ERR_UNSUPPORTED;
    if (batch == 0 || n_heads == 0) return KVQ_OK;
    kvq_path rp;
    if ((s = resolve_path(fmt, path, layout, n_heads, &rp)) != KVQ_OK) return s;
    if (!x_new || !dst_rows || !q || !cu_seqlens || !out || !codes || !scales) return KVQ_ERR_ARG;
    if (!attn_pointers_aligned(q, codes, scales, cu_seqlens, out) || !aligned(x_new, 16) || !aligned(dst_rows, 8))
        return KVQ_ERR_ARG;
    if (max_total_rows < batch) return KVQ_ERR_ARG;   // every sequence holds at least its new row
    if (!isfinite(sm_scale)) return KVQ_ERR_ARG;
    const size_t need = kv_attn_workspace_size(fmt, layout, batch, n_heads, max_total_rows, path);
    if (!workspace || workspace_bytes < need) return KVQ_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    if (rp == KVQ_PATH_TENSOR && fmt == KVQ_KV8 && q_dtype == KVQ_BF16) {
        const AttnPlan pl = plan_decode(fmt, rp, batch, n_heads, max_total_rows, decode_waves(fmt));
        return cuda_status(launch_attn_tc_kv8_append(*layout, x_new, dst_rows, q, batch, n_heads, codes, scales,
                                                     cu_seqlens, pl, sm_scale, out, workspace, st));
    }
    // other formats and paths: the encoder launch, then the decode
    int32_t* err = static_cast<int32_t*>(workspace);
    const cudaError_t e = launch_encode(fmt, x_new, batch, *layout, dst_rows, codes, scales, err, st);
    if (e != cudaSuccess) return KVQ_ERR_CUDA;
    return kv_attn_decode(fmt, layout, q, q_dtype, batch, n_heads, codes, scales, cu_seqlens, max_total_rows,
                          sm_scale, out, workspace, workspace_bytes, path, stream);
}

// Gather decode: the tensor-core kernel reads rows through an index table for
// KV8 with bf16 queries; every other combination runs on the fp32 kernels.
static kvq_status resolve_gather_path(kvq_format fmt, kvq_dtype qdt, kvq_path path, const kvq_mla_layout* L,
                                      int32_t n_heads, kvq_path* out) {
    const bool tc_ok = fmt == KVQ_KV8 && qdt == KVQ_BF16 && tc_supported(*L, n_heads);
    if (path == KVQ_PATH_TENSOR && !tc_ok) return KVQ_ERR_UNSUPPORTED;
    *out = path == KVQ_PATH_SIMT ? KVQ_PATH_SIMT : (tc_ok ? KVQ_PATH_TENSOR : KVQ_PATH_SIMT);
    return KVQ_OK;
}

size_t kv_attn_gather_workspace_size(kvq_format fmt, const kvq_mla_layout* layout, kvq_dtype q_dtype, int32_t batch,
                                     int32_t n_heads, int64_t max_total_selected, kvq_path path) {
    if (check_attn_layout(fmt, layout) != KVQ_OK || check_path(path) != KVQ_OK) return 0;
    if (batch < 0 || n_heads < 0 || max_total_selected < 0 || (q_dtype != KVQ_F32 && q_dtype != KVQ_BF16)) return 0;
    kvq_path rp;
    if (resolve_gather_path(fmt, q_dtype, path, layout, n_heads, &rp) != KVQ_OK) return 0;
    const AttnPlan pl = plan_decode(fmt, rp, batch, n_heads, max_total_selected, decode_waves(fmt));
    return kWsHeader + partial_bytes(pl.max_items, n_heads, layout->v_dim);
}

kvq_status kv_attn_decode_gather(kvq_format fmt, const kvq_mla_layout* layout, const void* q, kvq_dtype q_dtype,
                                 int32_t batch, int32_t n_heads, const uint8_t* codes, const float* scales,
                                 int64_t pool_rows, const int64_t* sel_rows, const int64_t* cu_sel,
                                 int64_t max_total_selected, float sm_scale, float* out, void* workspace,
                                 size_t workspace_bytes, kvq_path path, void* stream) {
    kvq_status s = check_attn_layout(fmt, layout);
    if (s != KVQ_OK) return s;
    if ((s = check_path(path)) != KVQ_OK) return s;
    if (batch < 0 || n_heads < 0 || max_total_selected < 0 || pool_rows < 0 ||
        (q_dtype != KVQ_F32 && q_dtype != KVQ_BF16))
        return KVQ_ERR_ARG;
    if (batch > 65535 || n_heads > 65535) return KVQ_ERR_UNSUPPORTED;
    if (batch == 0 || n_heads == 0) return KVQ_OK;
    kvq_path rp;
    if ((s = resolve_gather_path(fmt, q_dtype, path, layout, n_heads, &rp)) != KVQ_OK) return s;
    if (!q || !cu_sel || !out) return KVQ_ERR_ARG;
    if (max_total_selected > 0 && (!codes || !scales || !sel_rows || pool_rows == 0)) return KVQ_ERR_ARG;
    if (!attn_pointers_aligned(q, codes, scales, cu_sel, out) || !aligned(sel_rows, 8)) return KVQ_ERR_ARG;
    if (!isfinite(sm_scale)) return KVQ_ERR_ARG;
    const size_t need = kv_attn_gather_workspace_size(fmt, layout, q_dtype, batch, n_heads, max_total_selected, path);
    if (!workspace || workspace_bytes < need) return KVQ_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const AttnPlan pl = plan_decode(fmt, rp, batch, n_heads, max_total_selected, decode_waves(fmt));
    if (rp == KVQ_PATH_TENSOR)
        return cuda_status(launch_attn_tc(fmt, *layout, q, q_dtype, batch, n_heads, codes, scales, cu_sel, -1, pl,
                                          sm_scale, out, workspace, st, sel_rows, pool_rows));
    return cuda_status(launch_attn_simt(fmt, *layout, q, q_dtype, batch, n_heads, codes, scales, cu_sel, -1, pl,
                                        sm_scale, out, workspace, st, sel_rows, pool_rows));
}

static AttnPlan plan_prefill(int64_t n_past, int64_t n_new) {
    AttnPlan pl{};
    pl.chunk = std::max<int64_t>(1, n_past + n_new);
    pl.max_items = n_new;
    return pl;
}

size_t kv_attn_prefill_workspace_size(kvq_format fmt, const kvq_mla_layout* layout, int32_t n_heads, int64_t n_past,
                                      int64_t n_new, kvq_path path) {
    if (check_attn_layout(fmt, layout) != KVQ_OK || check_path(path) != KVQ_OK) return 0;
    if (n_heads < 0 || n_past < 0 || n_new < 0) return 0;
    const AttnPlan pl = plan_prefill(n_past, n_new);
    return kWsHeader + partial_bytes(pl.max_items, n_heads, layout->v_dim);
}

kvq_status kv_attn_prefill(kvq_format fmt, const kvq_mla_layout* layout, const float* x_new, const void* q,
                           kvq_dtype q_dtype, int64_t n_past, int64_t n_new, int32_t n_heads, uint8_t* codes,
                           float* scales, float sm_scale, float* out, void* workspace, size_t workspace_bytes,
                           kvq_path path, void* stream) {
    kvq_status s = check_attn_layout(fmt, layout);
    if (s != KVQ_OK) return s;
    if ((s = check_path(path)) != KVQ_OK) return s;
    if (n_past < 0 || n_new < 0 || n_heads < 0 || (q_dtype != KVQ_F32 && q_dtype != KVQ_BF16)) return KVQ_ERR_ARG;
    if (n_new > 65535 || n_heads > 65535) return KVQ_ERR_UNSUPPORTED;
    if (n_new == 0 || n_heads == 0) return KVQ_OK;
    kvq_path rp;
    if ((s = resolve_path(fmt, path, layout, n_heads, &rp)) != KVQ_OK) return s;
    if (!x_new || !q || !codes || !scales || !out) return KVQ_ERR_ARG;
    if (!attn_pointers_aligned(q, codes, scales, nullptr, out) || !aligned(x_new, 16)) return KVQ_ERR_ARG;
    if (!isfinite(sm_scale)) return KVQ_ERR_ARG;
    const size_t need = kv_attn_prefill_workspace_size(fmt, layout, n_heads, n_past, n_new, path);
    if (!workspace || workspace_bytes < need) return KVQ_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t row_bytes = format_row_bytes(fmt, *layout);
    const cudaError_t e = launch_encode(fmt, x_new, n_new, *layout, nullptr, codes + n_past * row_bytes,
                                        scales + n_past * layout->n_blocks, static_cast<int32_t*>(workspace), st);
    if (e != cudaSuccess) return KVQ_ERR_CUDA;
    const AttnPlan pl = plan_prefill(n_past, n_new);
    if (rp == KVQ_PATH_TENSOR)
        return cuda_status(launch_attn_tc(fmt, *layout, q, q_dtype, (int32_t)n_new, n_heads, codes, scales, nullptr,
                                          n_past, pl, sm_scale, out, workspace, st));
    return cuda_status(launch_attn_simt(fmt, *layout, q, q_dtype, (int32_t)n_new, n_heads, codes, scales, nullptr,
                                        n_past, pl, sm_scale, out, workspace, st));
}

int32_t kvq_read_device_error(void* workspace, int32_t clear, void* stream) {
    if (!workspace) return KVQ_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess) return KVQ_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KVQ_ERR_CUDA;
    if (clear && v != 0) {
        if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), st) != cudaSuccess) return KVQ_ERR_CUDA;
    }
    return v;
}

kvq_status kvq_test_stall_waits(int64_t polls) {
    if (polls < 0) return KVQ_ERR_ARG;
    kvq::set_test_stall_polls(polls);
    return KVQ_OK;
}

int64_t kvq_read_exact_rescales(void* workspace, int32_t clear, void* stream) {
    if (!workspace) return -1;
    cudaStream_t st = (cudaStream_t)stream;
    uint32_t* counter = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + 16);
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, counter, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess) return -1;
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
    if (clear && v != 0 && cudaMemsetAsync(counter, 0, sizeof v, st) != cudaSuccess) return -1;
    return (int64_t)v;
}

kvq_status k2v4_encode(const kvq_k2v4_layout* layout, const float* k, const float* v, int32_t batch,
                       int64_t n_cells, int64_t capacity, uint8_t* k_codes, uint16_t* k_scales, uint8_t* v_blocks,
                       uint16_t* k_win, uint16_t* v_win, int32_t* err_word, void* stream) {
    kvq_status s = check_k2v4(layout);
    if (s != KVQ_OK) return s;
    if (batch < 0 || n_cells < 0 || capacity < n_cells) return KVQ_ERR_ARG;
    if (n_cells % 32 != 0 || capacity % 32 != 0) return KVQ_ERR_UNSUPPORTED;
    if (batch > 65535 || layout->n_kv_heads > 65535 || n_cells / 32 > 0x7fffffff) return KVQ_ERR_UNSUPPORTED;
    if (batch == 0 || n_cells == 0) return KVQ_OK;
    if (!k || !v || !k_codes || !k_scales || !v_blocks) return KVQ_ERR_ARG;
    if ((layout->n_sink + layout->n_window) > 0 && (!k_win || !v_win)) return KVQ_ERR_ARG;
    return cuda_status(launch_k2v4_encode(*layout, k, v, batch, n_cells, capacity, k_codes, k_scales, v_blocks, k_win,
                                          v_win, err_word, (cudaStream_t)stream));
}

kvq_status k2v4_append(const kvq_k2v4_layout* layout, const float* k_new, const float* v_new, int32_t batch,
                       int64_t n_past, int64_t n_new, int64_t capacity, uint8_t* k_codes, uint16_t* k_scales,
                       uint8_t* v_blocks, uint16_t* k_win, uint16_t* v_win, int32_t* err_word, void* stream) {
    kvq_status s = check_k2v4(layout);
    if (s != KVQ_OK) return s;
    if (batch < 0 || n_past < 0 || n_new < 0 || capacity < 0 || n_past > capacity - n_new) return KVQ_ERR_ARG;
    if (capacity % 32 != 0) return KVQ_ERR_UNSUPPORTED;
    if (batch > 65535 || layout->n_kv_heads > 65535 || n_new > 0x7fffffff) return KVQ_ERR_UNSUPPORTED;
    if (batch == 0 || n_new == 0) return KVQ_OK;
    if (!k_new || !v_new || !k_codes || !k_scales || !v_blocks) return KVQ_ERR_ARG;
    if ((layout->n_sink + layout->n_window) > 0 && (!k_win || !v_win)) return KVQ_ERR_ARG;
    return cuda_status(launch_k2v4_append(*layout, k_new, v_new, batch, n_past, n_new, capacity, k_codes, k_scales,
                                          v_blocks, k_win, v_win, err_word, (cudaStream_t)stream));
}

size_t kv_attn_decode_k2v4_workspace_size(const kvq_k2v4_layout* layout, int32_t batch, int32_t n_q_heads,
                                          int64_t n_cells, kvq_path path) {
    if (check_k2v4(layout) != KVQ_OK || check_k2v4_path(path) != KVQ_OK) return 0;
    if (batch < 0 || n_q_heads < 0 || n_cells < 0) return 0;
    bool tensor;
    if (resolve_k2v4_path(path, layout, &tensor) != KVQ_OK) return 0;
    const K2V4Plan pl = plan_k2v4(*layout, batch, n_q_heads, n_cells, tensor);
    return kWsHeader + k2v4_partial_bytes(*layout, batch, n_q_heads, pl);
}

kvq_status kv_attn_decode_k2v4(const kvq_k2v4_layout* layout, const float* q, int32_t batch, int32_t n_q_heads,
                               int64_t n_cells, int64_t capacity, const uint8_t* k_codes, const uint16_t* k_scales,
                               const uint8_t* v_blocks, const uint16_t* k_win, const uint16_t* v_win, float sm_scale,
                               float* out, void* workspace, size_t workspace_bytes, kvq_path path, void* stream) {
    kvq_status s = check_k2v4(layout);
    if (s != KVQ_OK) return s;
    if ((s = check_k2v4_path(path)) != KVQ_OK) return s;
    if (batch < 0 || n_q_heads < 0 || n_cells < 0 || capacity < n_cells) return KVQ_ERR_ARG;
    if (n_q_heads % layout->n_kv_heads != 0) return KVQ_ERR_ARG;
    if (n_q_heads / layout->n_kv_heads > 8) return KVQ_ERR_UNSUPPORTED;
    if (capacity % 32 != 0) return KVQ_ERR_UNSUPPORTED;   // n_cells may end inside a group
    const int D = layout->head_dim;
    if (D != 128 && D != 256 && D != 512) return KVQ_ERR_UNSUPPORTED;
    if (batch > 65535) return KVQ_ERR_UNSUPPORTED;
    if (batch == 0 || n_q_heads == 0) return KVQ_OK;
    if (!q || !out || (n_cells > 0 && (!k_codes || !k_scales || !v_blocks))) return KVQ_ERR_ARG;
    if ((layout->n_sink + layout->n_window) > 0 && (!k_win || !v_win)) return KVQ_ERR_ARG;
    // the tile staging copies whole 32-cell groups of each pool in 16-byte units
    if (n_cells > 0 && (!aligned(k_codes, 16) || !aligned(k_scales, 16) || !aligned(v_blocks, 16)))
        return KVQ_ERR_ARG;
    if (!isfinite(sm_scale)) return KVQ_ERR_ARG;
    const size_t need = kv_attn_decode_k2v4_workspace_size(layout, batch, n_q_heads, n_cells, path);
    if (!workspace || workspace_bytes < need) return KVQ_ERR_WORKSPACE;
    bool tensor;
    if ((s = resolve_k2v4_path(path, layout, &tensor)) != KVQ_OK) return s;
    const K2V4Plan pl = plan_k2v4(*layout, batch, n_q_heads, n_cells, tensor);
    return cuda_status(launch_k2v4_decode(*layout, q, batch, n_q_heads, n_cells, capacity, k_codes, k_scales,
                                          v_blocks, k_win, v_win, sm_scale, out, workspace, pl,
                                          (cudaStream_t)stream));
}

}  // extern "C"
