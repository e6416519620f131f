// attn_common.cuh -- pieces shared by the SIMT and tensor-core attention paths:
// the parameter block, the device-side enumeration of split-T work items from
// cu_seqlens, and the partial-state format the merge kernel consumes.
//
// Partial state of one work item (a chunk of rows of one sequence) and head h,
// in natural-log units: m = max_t z_t over the chunk, l = sum_t exp(z_t - m),
// o[d] = sum_t exp(z_t - m) * x_hat_t[d] (TQ4: in the rotated domain).
#pragma once

#include "kvq_internal.cuh"

namespace kvq {

constexpr int kMlaD = 576, kMlaDL = 512, kMlaDR = 64, kMlaDV = 512;

struct AttnParams {
    int32_t n_blocks;
    int32_t n_seq, n_heads;
    const void* q;
    const uint8_t* codes;
    const float* scales;
    const int64_t* cu;      // decode: ragged row offsets
    int64_t prefill_past;   // prefill: >= 0; token b attends rows [0, past + b]
    int64_t chunk, max_items;
    float sm_scale;
    float* ws_o;            // [max_items][n_heads][512]
    float* ws_ml;           // [max_items][n_heads][2]
    int32_t* err;
    SignWords signs;
    float kn[2];
    float lv[16];
    // decode with rows appended in the same launch (tensor-core KV8 kernel):
    // x_new[b] is encoded into pool row dst_rows[b], inside [cu[b], cu[b+1])
    const float* x_new;
    const int64_t* dst_rows;
    uint8_t* codes_out;
    float* scales_out;
    int32_t bd0, bd1;
    // decode over selected rows: the rows of sequence b are the pool rows
    // sel[cu[b]] .. sel[cu[b+1] - 1] (absolute indices, each < pool_rows)
    const int64_t* sel;
    int64_t pool_rows;
};

// Pool row of logical row r of a gather decode; an index outside the pool sets
// the error word and is clamped so that nothing outside the pool is read.
__device__ __forceinline__ int64_t gather_row(const AttnParams& p, int64_t r) {
    int64_t pr = p.sel[r];
    if (pr < 0 || pr >= p.pool_rows) {
        atomicCAS(p.err, 0, KVQ_ERR_ARG);
        pr = pr < 0 ? 0 : p.pool_rows - 1;
    }
    return pr;
}

__device__ __forceinline__ void set_err(int32_t* err, int32_t code) { atomicCAS(err, 0, code); }

// Programmatic dependent launch: a partial kernel lets the dependent merge grid
// be scheduled early; the merge waits for the partial grid's completion (and
// the visibility of its writes) before it reads the partial state.  Both are
// no-ops when the launch carries no programmatic dependency.
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Number of chunks of sequence b (0 for an empty or malformed range).
__device__ __forceinline__ int64_t n_chunks_of(const int64_t* cu, int b, int64_t chunk, int32_t* err) {
    const int64_t len = cu[b + 1] - cu[b];
    if (len < 0) {
        set_err(err, KVQ_ERR_ARG);
        return 0;
    }
    return (len + chunk - 1) / chunk;
}

// Warp-cooperative search for the sequence owning work item `item`.
// Returns b (or -1), the chunk index within b and, from the bounds the search
// has already read, the chunk's row range [row0, row1).
__device__ __forceinline__ int find_item(const int64_t* cu, int n_seq, int64_t chunk, int64_t item, int lane,
                                         int64_t* ch_out, int32_t* err, int64_t* row0 = nullptr,
                                         int64_t* row1 = nullptr) {
    int64_t base = 0;
    for (int b0 = 0; b0 < n_seq; b0 += 32) {
        const int b = b0 + lane;
        int64_t s = 0, e = 0, n = 0;
        if (b < n_seq) {
            s = cu[b];
            e = cu[b + 1];
            if (e < s) set_err(err, KVQ_ERR_ARG);
            else n = (e - s + chunk - 1) / chunk;
        }
        int64_t incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t t = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += t;
        }
        const int64_t total = __shfl_sync(kFull, incl, 31);
        if (item < base + total) {
            const int64_t excl = incl - n;
            const bool mine = b < n_seq && item >= base + excl && item < base + incl;
            const unsigned mask = __ballot_sync(kFull, mine);
            const int src = __ffs(mask) - 1;
            const int64_t ch = item - base - __shfl_sync(kFull, excl, src);
            const int64_t ss = __shfl_sync(kFull, s, src), ee = __shfl_sync(kFull, e, src);
            *ch_out = ch;
            if (row0) {
                *row0 = ss + ch * chunk;
                *row1 = min(*row0 + chunk, ee);
            }
            return b0 + src;
        }
        base += total;
    }
    return -1;
}

// First work item of sequence b and its chunk count.
__device__ __forceinline__ void seq_items(const int64_t* cu, int b, int64_t chunk, int lane, int64_t* first,
                                          int64_t* count, int32_t* err) {
    int64_t acc = 0;
    for (int b0 = 0; b0 < b; b0 += 32) {
        const int bb = b0 + lane;
        int64_t n = bb < b ? n_chunks_of(cu, bb, chunk, err) : 0;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) n += __shfl_xor_sync(kFull, n, o);
        acc += n;
    }
    *first = acc;
    *count = n_chunks_of(cu, b, chunk, err);
}

// Locates this CTA's work item (warp 0 calls it); returns the sequence (or -1)
// and the row range [row0, row1) of the chunk.
__device__ __forceinline__ int locate_item(const AttnParams& p, int64_t item, int lane, int64_t* row0,
                                           int64_t* row1) {
    int b = -1;
    int64_t ch = 0;
    if (p.prefill_past >= 0) {
        if (item < p.n_seq) {
            b = (int)item;
            *row0 = 0;
            *row1 = p.prefill_past + b + 1;
        }
    } else {
        b = find_item(p.cu, p.n_seq, p.chunk, item, lane, &ch, p.err, row0, row1);
    }
    return b;
}

template <bool QBF16>
__device__ __forceinline__ float load_q(const void* q, int64_t idx) {
    if (QBF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(q)[idx]);
    return reinterpret_cast<const float*>(q)[idx];
}

AttnParams make_attn_params(kvq_format fmt, const kvq_mla_layout& L, const void* q, int32_t n_seq, int32_t n_heads,
                            const uint8_t* codes, const float* scales, const int64_t* cu_seqlens,
                            int64_t prefill_past, const AttnPlan& plan, float sm_scale, void* workspace);

// Tensor-core partial kernel for KV8 rows with bf16 queries (every chunk of a
// tile decoded once); grid = work items x head groups of 64.
cudaError_t launch_attn_tc_kv8_bf16(const AttnParams& p, int64_t grid_x, int groups, cudaStream_t stream);
// The same kernel with the per-sequence new rows (p.x_new, p.dst_rows) encoded
// into the pool and substituted into the tiles that hold them.
cudaError_t launch_attn_tc_kv8_bf16_append(const AttnParams& p, int64_t grid_x, int groups, cudaStream_t stream);

// LSE merge of the chunk partials into out[n_seq][n_heads][512] (TQ4: unrotated).
cudaError_t launch_attn_merge(kvq_format fmt, const AttnParams& p, float* out, cudaStream_t stream);

}  // namespace kvq
