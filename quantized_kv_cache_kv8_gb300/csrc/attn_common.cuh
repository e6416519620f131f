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
    // tensor-core decode: > 0 = items per wave of CTAs; the chunk is then
    // chosen on the device from the actual lengths (balanced_tiles) and kept
    // in the workspace header for the merge
    int64_t wave_items;
    int32_t max_waves;      // waves of items the workspace holds (>= 1 when wave_items > 0)
    int64_t max_rows;       // host bound on cu[n_seq] the launch was sized for
    int64_t* ws_chunk;
    float sm_scale;
    float* ws_o;            // [max_items][n_heads][512]
    float* ws_ml;           // [max_items][n_heads][2]
    int32_t* err;
    // tensor-core kernels: tiles after a chunk's first that took the exact
    // rescale path of the lagged running maxima (a diagnostic counter in the
    // workspace header)
    uint32_t* exact_count;
    // bounded waits: the tile-loop limit (try_wait polls) and the testing
    // hook's stall (> 0: first wait on a barrier nothing arrives on)
    int64_t wait_limit;
    int64_t stall_polls;
    SignWords signs;
    float kn[2];
    float lv[16];
    // PolarQuant rows (fp32 consumer): width, row bytes, byte offset of the
    // rope block's stream, device centroids of the width ([level 1..10][2^b])
    int32_t pq_bits, pq_row_bytes, pq_boff1;
    const float2* pq_cent;
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

// Rows per work item of a tensor-core decode, chosen from the actual lengths
// T_b (R rows in all, n non-empty sequences, S = wave_items items per wave of
// CTAs).  For k = 1 .. max_waves waves the chunk C_k is the smallest multiple
// of 128 rows (one tile) whose item count sum_b ceil(T_b / C) fits
// W_k = k * S * ceil(n / S); C_k is found by bisection over
// [ceil(R / W_k), ceil(R / (W_k - n))] tiles (sum_b ceil(T_b / C) <= R / C + n)
// or up to the longest sequence.  The chunk kept minimises the wave estimate
// waves(C) * (C + kItemOverhead); the loop stops once no larger k can win
// (every k' waves cost at least R / S + k' * kItemOverhead).  Equal lengths
// end at k = 1: 8 sequences of 4096 rows at 38 items per wave take 1024-row
// chunks (32 items, one wave) where a chunk from the total alone (896) gives
// 40 items and two waves.  Ragged lengths take more, shorter items: a
// 131072-row sequence among short ones is not left to one CTA.  Every CTA
// computes the same value (warp-cooperative; lanes converged).  More than
// kBalanceSeqs sequences keep the host's chunk.
constexpr int kBalanceSeqs = 1024;
constexpr int64_t kBalanceGranule = 128;
constexpr int64_t kItemOverhead = 2;   // tiles' worth of a CTA's prologue and epilogue

// What the balanced split reads of the call: the ragged bounds and the wave
// budget.
struct BatchView {
    const int64_t* cu;
    int32_t n_seq;
    int32_t wave_items;   // items per wave of CTAs
    int32_t max_waves;    // waves the workspace holds
    int64_t max_rows;     // host bound on cu[n_seq]
    int32_t* err;
};

// The batch's lengths in tiles of kBalanceGranule rows as the warp sees them:
// one per lane, read once, for batches of at most 32 sequences; re-read from
// cu_seqlens on every pass for larger ones.
struct WarpTiles {
    bool small;
    int32_t tiles;   // small: this lane's sequence (0 past the batch)
    int64_t len;     // small: its rows
};

__device__ __forceinline__ int32_t warp_sum32(int32_t v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ int64_t seq_len(const BatchView& bv, int b) {
    return b < bv.n_seq ? max((int64_t)0, bv.cu[b + 1] - bv.cu[b]) : 0;
}

// sum_b ceil(tiles_b / k): the item count at a chunk of k tiles
__device__ __forceinline__ int32_t count_items(const BatchView& bv, const WarpTiles& wt, int32_t k, int lane) {
    if (wt.small) return warp_sum32((wt.tiles + k - 1) / k);
    int32_t cnt = 0;
    for (int b0 = 0; b0 < bv.n_seq; b0 += 32) {
        const int32_t t = (int32_t)((seq_len(bv, b0 + lane) + kBalanceGranule - 1) / kBalanceGranule);
        cnt += warp_sum32((t + k - 1) / k);
    }
    return cnt;
}

// Chunk (in tiles) of a tensor-core decode, chosen from the actual lengths
// (R tiles in all, n non-empty sequences, S = wave_items items per wave of
// CTAs).  For k = 1 .. max_waves waves the chunk C_k is the smallest whose
// item count sum_b ceil(T_b / C) fits W_k = k * S * ceil(n / S), found by
// bisection over [ceil(R / W_k), ceil(R / (W_k - n))] (the count is at most
// R / C + n) or up to the longest sequence.  The chunk kept minimises the
// wave estimate waves(C) * (C + kItemOverhead); the loop stops once no larger
// k can win (k' waves cost at least R / S + k' * kItemOverhead).  Equal
// lengths end at k = 1: 8 sequences of 32 tiles at 38 items per wave take
// 8-tile chunks (32 items, one wave) where a chunk from the total alone (7)
// gives 40 items and two waves.  Ragged lengths take more, shorter items: a
// long sequence among short ones is not left to one CTA.  Every CTA computes
// the same value (warp-cooperative; lanes converged).
__device__ __forceinline__ int32_t balanced_tiles(const BatchView& bv, const WarpTiles& wt, int lane) {
    int64_t rows = 0;
    int32_t tiles = 0, tmax = 0, n = 0;
    for (int b0 = 0; b0 < (wt.small ? 1 : bv.n_seq); b0 += 32) {
        int64_t len = wt.small ? wt.len : seq_len(bv, b0 + lane);
        const int32_t t = wt.small ? wt.tiles : (int32_t)((len + kBalanceGranule - 1) / kBalanceGranule);
        int32_t m = t, c = t > 0, ts = t;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            len += __shfl_xor_sync(kFull, len, o);
            m = max(m, __shfl_xor_sync(kFull, m, o));
            c += __shfl_xor_sync(kFull, c, o);
            ts += __shfl_xor_sync(kFull, ts, o);
        }
        rows += len;
        tiles += ts;
        tmax = max(tmax, m);
        n += c;
    }
    if (rows > bv.max_rows && lane == 0) set_err(bv.err, KVQ_ERR_DEVICE);
    if (n == 0) return 1;
    const int32_t S = bv.wave_items;
    const int32_t base = S * ((n + S - 1) / S);
    int32_t best_c = tmax, best_e = 0;
    for (int k = 1; k <= bv.max_waves; ++k) {
        const int32_t W = k * base;
        int32_t lo = max(1, (tiles + W - 1) / W);
        int32_t hi = tmax;
        if (W > n) hi = min(hi, (tiles + (W - n) - 1) / (W - n));
        lo = min(lo, hi);
        while (lo < hi) {
            const int32_t mid = (lo + hi) / 2;
            if (count_items(bv, wt, mid, lane) <= W) hi = mid;
            else lo = mid + 1;
        }
        const int32_t e = (count_items(bv, wt, lo, lane) + S - 1) / S * (lo + (int32_t)kItemOverhead);
        if (k == 1 || e < best_e) {
            best_e = e;
            best_c = lo;
        }
        if (best_e <= (tiles + S - 1) / S + (k + 1) * (int32_t)kItemOverhead) break;
    }
    return best_c;
}

struct ItemRange {
    int64_t row0, row1;
    int b;
};

// The balanced split's item lookup for the tensor-core decode: the chunk, the
// sequence of `item` (or -1) and its rows.  Not inlined: the kernels that call
// it run at their register cap, and keeping this search out of their bodies
// keeps it out of their register allocation.
static __device__ __noinline__ ItemRange locate_balanced(BatchView bv, int64_t item, int lane, int64_t* ws_chunk,
                                                         bool store_chunk) {
    ItemRange r{0, 0, -1};
    if (bv.n_seq <= 32) {
        // one read of the batch's bounds; chunk choice and lookup in registers
        int64_t s = 0, e = 0;
        if (lane < bv.n_seq) {
            s = bv.cu[lane];
            e = bv.cu[lane + 1];
            if (e < s) set_err(bv.err, KVQ_ERR_ARG);
        }
        const int64_t len = max((int64_t)0, e - s);
        const WarpTiles wt{true, (int32_t)((len + kBalanceGranule - 1) / kBalanceGranule), len};
        const int32_t kc = balanced_tiles(bv, wt, lane);
        const int64_t chunk = (int64_t)kc * kBalanceGranule;
        if (store_chunk && lane == 0) *ws_chunk = chunk;
        const int32_t nb = (wt.tiles + kc - 1) / kc;
        int32_t incl = nb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t t = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += t;
        }
        const unsigned mask = __ballot_sync(kFull, item >= incl - nb && item < incl);
        if (mask) {
            const int src = __ffs(mask) - 1;
            const int64_t c = item - (__shfl_sync(kFull, incl, src) - __shfl_sync(kFull, nb, src));
            const int64_t ss = __shfl_sync(kFull, s, src), ee = __shfl_sync(kFull, e, src);
            r.row0 = ss + c * chunk;
            r.row1 = min(r.row0 + chunk, ee);
            r.b = src;
        }
        return r;
    }
    const int64_t chunk = (int64_t)balanced_tiles(bv, WarpTiles{false, 0, 0}, lane) * kBalanceGranule;
    if (store_chunk && lane == 0) *ws_chunk = chunk;
    int64_t ch = 0;
    r.b = find_item(bv.cu, bv.n_seq, chunk, item, lane, &ch, bv.err, &r.row0, &r.row1);
    return r;
}

// Locates this CTA's work item (warp 0 calls it); returns the sequence (or -1)
// and the row range [row0, row1) of the chunk.  Tensor-core decodes of up to
// kBalanceSeqs sequences take the balanced split; the chunk then goes to the
// workspace header for the merge.
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
    } else if (p.wave_items > 0 && p.n_seq <= kBalanceSeqs) {
        const BatchView bv{p.cu, p.n_seq, (int32_t)p.wave_items, p.max_waves, p.max_rows, p.err};
        const ItemRange r = locate_balanced(bv, item, lane, p.ws_chunk, blockIdx.x == 0);
        *row0 = r.row0;
        *row1 = r.row1;
        b = r.b;
    } else {
        if (p.wave_items > 0 && blockIdx.x == 0 && lane == 0) *p.ws_chunk = p.chunk;
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
// Tensor-core partial kernel for TQ4 rows (bf16 or f32 queries, rotated in the
// kernel); grid = work items x head groups of 32.
// TQ4 rows, or (pq) PolarQuant rows at 4 bits
cudaError_t launch_attn_tc_tq4(const AttnParams& p, bool q_bf16, bool pq, int64_t grid_x, int n_heads,
                               cudaStream_t stream);

// LSE merge of the chunk partials into out[n_seq][n_heads][512] (TQ4: unrotated).
cudaError_t launch_attn_merge(kvq_format fmt, const AttnParams& p, float* out, cudaStream_t stream);

}  // namespace kvq
