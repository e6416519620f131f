// k2v4.cu -- the 2-bit-K / 4-bit-V GQA cache with an exact FP16 window ([P3]).
//
// Encode: K per (kv head, channel, 32-cell group) -- one thread per channel
// walks its 32 cells, forms the sum of squares in a fixed pairwise order,
// s = sqrt(ss/32), picks the nearest of 4 Lloyd-Max levels for x/s and stores
// fp16(k_gain * s) ([P3] Summary item 3: codes against the un-gained scale).
// V per cell and 32-dim block (q4_0) -- one warp per block.  Cells inside the
// sink/window overlay also get exact fp16 copies.
//
// Decode, fp32 CUDA cores: one CTA per (sequence, kv head, chunk of cells)
// serves the kv head's query heads; tiles of 32 cells are staged, dequantized
// to f32 in shared memory (overlay cells take their fp16 copy), then scores,
// online softmax and the context follow as in the MLA path.
// Decode, tensor cores (head_dim 128 or 256): tiles of 128 cells are
// dequantized to f16 in shared memory and both products run as tcgen05 MMAs
// with the cells on M: S^T = K Q^T (N = 16: the query heads as f16 and as
// their f16 residuals) and O^T += V^T P^T (N = 16, heads past the group are
// zero).  A CTA runs two such pipelines, each on its own chunk.  Both paths
// write the same chunk partials; a merge kernel combines them by
// log-sum-exp.
#include "tc_common.cuh"

#include <algorithm>
#include <math.h>

namespace kvq {
namespace {

constexpr int kG = 32;          // cells per K scale group
constexpr int kMaxD = 512;
constexpr int kTC = 32;         // cells per tile
constexpr int kNT = 256;
constexpr int kSmSMs = 152;

struct K2V4Params {
    int32_t H, D, slots, n_sink, n_window, n_slack;
    int64_t T, cap;
    float k_gain;
    float lv[4], th[4];
};

__device__ __forceinline__ int64_t overlay_slot(int64_t c, const K2V4Params& p) {
    if (c < p.n_sink) return c;
    if (c >= p.T - p.n_window) return p.n_sink + c % (p.n_window + p.n_slack);
    return -1;
}

// grid: (groups, H, batch), block: D threads (one per channel)
__global__ void __launch_bounds__(kMaxD) k2_encode_kernel(const float* __restrict__ k, K2V4Params p,
                                                          uint8_t* __restrict__ k_codes,
                                                          uint16_t* __restrict__ k_scales, int32_t* err) {
    const int d = threadIdx.x;
    const int64_t gi = blockIdx.x;
    const int g = blockIdx.y, b = blockIdx.z;
    const int64_t seq = (int64_t)b * p.H + g;
    const float* col = k + (seq * p.T + gi * kG) * p.D + d;
    float x[kG], ps[kG];
#pragma unroll
    for (int j = 0; j < kG; ++j) {
        x[j] = __ldg(col + (int64_t)j * p.D);
        ps[j] = __fmaf_rn(x[j], x[j], 0.0f);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
        for (int j = 0; j < off; ++j) ps[j] = __fadd_rn(ps[j], ps[j + off]);
    // a NaN or infinite K value (or squares past the f32 range): no code exists
    if (!(ps[0] <= 3.402823466e38f) && err) atomicCAS(err, 0, (int32_t)KVQ_ERR_NONFINITE);
    const float s_rule = __fsqrt_rn(__fdiv_rn(ps[0], 32.0f));
    k_scales[(seq * (p.cap / kG) + gi) * p.D + d] = __half_as_ushort(__float2half_rn(__fmul_rn(p.k_gain, s_rule)));
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < kG; ++j) {
        int c = 0;
        if (s_rule != 0.0f) {
            const float u = __fdiv_rn(x[j], s_rule);
            c = (u > p.th[0]) + (u > p.th[1]) + (u > p.th[2]);
        }
        // dims d..d+3 share a byte: lane d%4 == 0 gathers its three neighbours
        const int c1 = __shfl_down_sync(kFull, c, 1);
        const int c2 = __shfl_down_sync(kFull, c, 2);
        const int c3 = __shfl_down_sync(kFull, c, 3);
        if ((lane & 3) == 0)
            k_codes[(seq * p.cap + gi * kG + j) * (p.D / 4) + d / 4] = (uint8_t)(c | (c1 << 2) | (c2 << 4) | (c3 << 6));
    }
}

// Append of n_new cells at t_old .. t_old + n_new - 1 (k_new is [batch][H]
// [n_new][D]): one block per (touched group, kv head, sequence), one thread
// per channel.  A group first written here takes, with all 32 cells present,
// the encoder's rule; with n < 32 cells, sqrt((ss + (32 - n) prev^2) / 32)
// ([P3] "Review fixes": the previous group's mean square stands in for the
// cells not yet written), prev = f16(stored scale of the previous group) /
// k_gain -- recomputed here from the new cells when that group is written in
// this launch (it is then whole), read from the pool otherwise, the same bits
// either way; group 0 with n < 32 cells takes the RMS of the cells present.
// A group that already holds cells keeps its scale and codes the new cells
// against f16(stored) / k_gain.
__global__ void __launch_bounds__(kMaxD) k2_append_kernel(const float* __restrict__ k_new, K2V4Params p,
                                                          int64_t t_old, int64_t n_new,
                                                          uint8_t* __restrict__ k_codes,
                                                          uint16_t* __restrict__ k_scales, int32_t* err) {
    const int d = threadIdx.x, lane = threadIdx.x & 31;
    const int64_t gi = t_old / kG + blockIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    const int64_t seq = (int64_t)b * p.H + h;
    const int64_t g0 = gi * kG;
    const bool fresh = g0 >= t_old;
    const int64_t c0 = fresh ? g0 : t_old;
    const int n = (int)(min(g0 + kG, t_old + n_new) - c0);            // new cells of the group
    const float* col = k_new + (seq * n_new + (c0 - t_old)) * p.D + d;
    uint16_t* sc = k_scales + (seq * (p.cap / kG) + gi) * p.D + d;
    float x[kG];
#pragma unroll
    for (int j = 0; j < kG; ++j) x[j] = j < n ? __ldg(col + (int64_t)j * p.D) : 0.0f;
    {
        bool bad = false;
#pragma unroll
        for (int j = 0; j < kG; ++j) bad |= !(fabsf(x[j]) <= 3.402823466e38f);
        if (bad && err) atomicCAS(err, 0, (int32_t)KVQ_ERR_NONFINITE);
    }
    float s_rule;
    if (fresh) {
        float ps[kG];
#pragma unroll
        for (int j = 0; j < kG; ++j) ps[j] = __fmaf_rn(x[j], x[j], 0.0f);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
            for (int j = 0; j < off; ++j) ps[j] = __fadd_rn(ps[j], ps[j + off]);
        if (n == kG) {
            s_rule = __fsqrt_rn(__fdiv_rn(ps[0], 32.0f));
        } else if (gi == 0) {
            s_rule = __fsqrt_rn(__fdiv_rn(ps[0], (float)n));
        } else {
            uint16_t prev_bits;
            if ((gi - 1) * kG >= t_old) {
                // the previous group is written by this launch, whole: its stored
                // scale is recomputed here in the encoder's order
                const float* pc = col - (int64_t)kG * p.D;
                float pp[kG];
#pragma unroll
                for (int j = 0; j < kG; ++j) {
                    const float y = __ldg(pc + (int64_t)j * p.D);
                    pp[j] = __fmaf_rn(y, y, 0.0f);
                }
#pragma unroll
                for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
                    for (int j = 0; j < off; ++j) pp[j] = __fadd_rn(pp[j], pp[j + off]);
                const float s_prev = __fsqrt_rn(__fdiv_rn(pp[0], 32.0f));
                prev_bits = __half_as_ushort(__float2half_rn(__fmul_rn(p.k_gain, s_prev)));
            } else {
                prev_bits = sc[-p.D];   // stored by an earlier call
            }
            const float prev = __fdiv_rn(__half2float(__ushort_as_half(prev_bits)), p.k_gain);
            const float add = __fmul_rn((float)(kG - n), __fmul_rn(prev, prev));
            s_rule = __fsqrt_rn(__fdiv_rn(__fadd_rn(ps[0], add), 32.0f));
        }
        *sc = __half_as_ushort(__float2half_rn(__fmul_rn(p.k_gain, s_rule)));
    } else {
        s_rule = __fdiv_rn(__half2float(__ushort_as_half(*sc)), p.k_gain);
    }
#pragma unroll
    for (int j = 0; j < kG; ++j) {
        if (j >= n) break;   // n is the same for the whole block
        int c = 0;
        if (s_rule != 0.0f) {
            const float u = __fdiv_rn(x[j], s_rule);
            c = (u > p.th[0]) + (u > p.th[1]) + (u > p.th[2]);
        }
        const int c1 = __shfl_down_sync(kFull, c, 1);
        const int c2 = __shfl_down_sync(kFull, c, 2);
        const int c3 = __shfl_down_sync(kFull, c, 3);
        if ((lane & 3) == 0)
            k_codes[(seq * p.cap + c0 + j) * (p.D / 4) + d / 4] = (uint8_t)(c | (c1 << 2) | (c2 << 4) | (c3 << 6));
    }
}

// grid: (cells written, H, batch), block: D threads; warp w encodes 32-dim
// block w of cell cell0 + blockIdx.x, read from row blockIdx.x of a source of
// src_cells rows per sequence (the whole sequence for the encoder, the new
// cells for an append); the overlay window is taken at p.T
__global__ void __launch_bounds__(kMaxD) v4_encode_kernel(const float* __restrict__ k, const float* __restrict__ v,
                                                          K2V4Params p, int64_t src_cells, int64_t cell0,
                                                          uint8_t* __restrict__ v_blocks,
                                                          uint16_t* __restrict__ k_win, uint16_t* __restrict__ v_win,
                                                          int32_t* err) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int64_t cell = cell0 + blockIdx.x;
    const int g = blockIdx.y, b = blockIdx.z;
    const int64_t seq = (int64_t)b * p.H + g;
    const int64_t src = (seq * src_cells + blockIdx.x) * p.D + tid;
    const float x = __ldg(v + src);
    const float ax = fabsf(x);
    const float amax = warp_max(ax);
    // a NaN or infinite V value (a vote: the max above passes over NaNs)
    if (__any_sync(kFull, !(ax <= 3.402823466e38f)) && lane == 0 && err)
        atomicCAS(err, 0, (int32_t)KVQ_ERR_NONFINITE);
    float m = 0.0f;
    const unsigned at = __ballot_sync(kFull, ax == amax);
    if (amax > 0.0f) m = __shfl_sync(kFull, x, __ffs(at) - 1);   // first element of largest magnitude
    const float dd = __fdiv_rn(m, -8.0f);
    int c = 8;
    if (dd != 0.0f) c = min(15, __float2int_rz(__fadd_rn(__fdiv_rn(x, dd), 8.5f)));
    const int hi = __shfl_down_sync(kFull, c, 16);
    uint8_t* blk = v_blocks + ((seq * p.cap + cell) * (p.D / 32) + w) * 18;
    // one byte per lane: lanes 0..15 the packed codes, lanes 16/17 the two
    // bytes of the little-endian fp16 d
    const uint16_t hb = __half_as_ushort(__float2half_rn(dd));
    uint8_t byte = 0;
    int at_off = -1;
    if (lane < 16) {
        byte = (uint8_t)(c | (hi << 4));
        at_off = 2 + lane;
    } else if (lane == 16) {
        byte = (uint8_t)(hb & 0xffu);
        at_off = 0;
    } else if (lane == 17) {
        byte = (uint8_t)(hb >> 8);
        at_off = 1;
    }
    if (at_off >= 0) blk[at_off] = byte;
    const int64_t slot = overlay_slot(cell, p);
    if (slot >= 0) {
        const int64_t o = (seq * p.slots + slot) * p.D + tid;
        k_win[o] = __half_as_ushort(__float2half_rn(__ldg(k + src)));
        v_win[o] = __half_as_ushort(__float2half_rn(x));
    }
}

// ---------------------------------------------------------------------------
// SIMT decode
// ---------------------------------------------------------------------------
struct K2V4DecodeParams {
    K2V4Params c;
    int32_t batch, Hq, grp;   // grp = query heads per kv head (<= 8)
    int64_t chunk;
    int32_t n_chunks;
    float sm_scale;
    const float* q;
    const uint8_t* k_codes;
    const uint16_t* k_scales;
    const uint8_t* v_blocks;
    const uint16_t* k_win;
    const uint16_t* v_win;
    float* ws_o;   // [batch][Hq][n_chunks][D]
    float* ws_ml;  // [batch][Hq][n_chunks][2]
    int32_t* err;  // the workspace's error word
    int64_t wait_limit;   // try_wait polls of the tensor-core kernel's tile-loop waits
};

constexpr int kHQ = 8;   // query heads per CTA (one kv group)

// Raw bytes of one 32-cell tile of one kv head, staged in shared memory with
// 16-byte loads: K codes (32 x D/4), the group's K scales (D fp16), V blocks
// (32 x D/32 x 18).  Each piece is contiguous in the cache, and as tiles start
// on a multiple of 32 cells (and cell counts and capacities are multiples of
// 32), each starts 16-byte aligned and lies inside the allocation.
template <int D>
struct RawTileBytes {
    static constexpr int kKc = kTC * D / 4, kKs = 2 * D, kVb = kTC * (D / 32) * 18;
    static constexpr int kTotal = kKc + kKs + kVb;
};

template <int D>
__global__ void __launch_bounds__(kNT) k2v4_partial_kernel(K2V4DecodeParams p) {
    launch_dependents();
    constexpr int XS = D + 4;
    using RB = RawTileBytes<D>;
    extern __shared__ float4 smem4[];
    float* qs = reinterpret_cast<float*>(smem4);   // [8][XS]
    float* ks = qs + kHQ * XS;                      // [32][XS]
    float* vs = ks + kTC * XS;                      // [32][XS]
    float* P = vs + kTC * XS;                       // [32][8]
    float* alpha = P + kTC * kHQ;                   // [8]
    unsigned char* raw = reinterpret_cast<unsigned char*>(alpha + 8);   // RB::kTotal bytes
    const unsigned char* raw_kc = raw;
    const uint16_t* raw_ks = reinterpret_cast<const uint16_t*>(raw + RB::kKc);
    const unsigned char* raw_vb = raw + RB::kKc + RB::kKs;
    const int tid = threadIdx.x;
    const int chunk_id = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int64_t seq = (int64_t)b * p.c.H + g;
    const int64_t c0 = (int64_t)chunk_id * p.chunk;
    const int64_t c1 = min(c0 + p.chunk, p.c.T);
    for (int i = tid; i < kHQ * D; i += kNT) {
        const int h = i / D, d = i - h * D;
        qs[h * XS + d] = h < p.grp ? p.q[((int64_t)b * p.Hq + g * p.grp + h) * D + d] : 0.0f;
    }
    const int sh = tid >> 5, st = tid & 31;          // score: head, cell
    float m_run = -INFINITY, l_run = 0.0f;
    const int ch = tid >> 5, cl = tid & 31;          // context: head, dims 128i + 4cl
    constexpr int NG = D / 128;                      // float4 groups per lane: dims 128i + 4cl .. +3
    float o[NG][4];
#pragma unroll
    for (int i = 0; i < NG; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    __syncthreads();

    for (int64_t t0 = c0; t0 < c1; t0 += kTC) {
        const int nt = (int)min((int64_t)kTC, c1 - t0);
        // stage the tile's raw bytes (a whole 32-cell group)
        const int64_t grp_idx = t0 / kG;
        {
            const uint4* kc_src = reinterpret_cast<const uint4*>(p.k_codes + (seq * p.c.cap + t0) * (D / 4));
            const uint4* ks_src = reinterpret_cast<const uint4*>(p.k_scales + (seq * (p.c.cap / kG) + grp_idx) * D);
            const uint4* vb_src = reinterpret_cast<const uint4*>(p.v_blocks + (seq * p.c.cap + t0) * (D / 32) * 18);
            for (int i = tid; i < RB::kTotal / 16; i += kNT) {
                uint4 w;
                if (i < RB::kKc / 16)
                    w = __ldg(kc_src + i);
                else if (i < (RB::kKc + RB::kKs) / 16)
                    w = __ldg(ks_src + (i - RB::kKc / 16));
                else
                    w = __ldg(vb_src + (i - (RB::kKc + RB::kKs) / 16));
                reinterpret_cast<uint4*>(raw)[i] = w;
            }
        }
        __syncthreads();
        // dequantize K and V of the tile (overlay cells read their fp16 copy)
        for (int i = tid; i < kTC * D; i += kNT) {
            const int r = i / D, d = i - r * D;
            float kv = 0.0f, vv = 0.0f;
            if (r < nt) {
                const int64_t cell = t0 + r;
                const int64_t slot = overlay_slot(cell, p.c);
                if (slot >= 0) {
                    const int64_t o2 = (seq * p.c.slots + slot) * D + d;
                    kv = __half2float(__ushort_as_half(p.k_win[o2]));
                    vv = __half2float(__ushort_as_half(p.v_win[o2]));
                } else {
                    const uint8_t kb = raw_kc[r * (D / 4) + d / 4];
                    const float ksc = __half2float(__ushort_as_half(raw_ks[d]));
                    kv = p.c.lv[(kb >> (2 * (d & 3))) & 3] * ksc;
                    const unsigned char* blk = raw_vb + (r * (D / 32) + d / 32) * 18;
                    const float dd = __half2float(__ushort_as_half((uint16_t)(blk[0] | (blk[1] << 8))));
                    const int j = d & 31;
                    const int code = j < 16 ? (blk[2 + j] & 15) : (blk[2 + j - 16] >> 4);
                    vv = (float)(code - 8) * dd;
                }
            }
            ks[r * XS + d] = kv;
            vs[r * XS + d] = vv;
        }
        __syncthreads();
        {
            const float* qh = qs + sh * XS;
            const float* kr = ks + st * XS;
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
            for (int d = 0; d < D; d += 4) {
                const float4 a = *reinterpret_cast<const float4*>(qh + d);
                const float4 x = *reinterpret_cast<const float4*>(kr + d);
                a0 = fmaf(a.x, x.x, a0);
                a1 = fmaf(a.y, x.y, a1);
                a2 = fmaf(a.z, x.z, a2);
                a3 = fmaf(a.w, x.w, a3);
            }
            const float z = st < nt ? p.sm_scale * ((a0 + a1) + (a2 + a3)) : -INFINITY;
            const float tmax = warp_max(z);
            const float m_new = fmaxf(m_run, tmax);
            const float a = m_run == -INFINITY ? 0.0f : expf(m_run - m_new);
            const float pz = expf(z - m_new);
            float psum = pz;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) psum += __shfl_xor_sync(kFull, psum, off);
            l_run = l_run * a + psum;
            m_run = m_new;
            P[st * kHQ + sh] = pz;
            if (st == 0) alpha[sh] = a;
        }
        __syncthreads();
        {
            const float al = alpha[ch];
#pragma unroll
            for (int i = 0; i < NG; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) o[i][j] *= al;
            for (int t = 0; t < nt; ++t) {
                const float pw = P[t * kHQ + ch];
#pragma unroll
                for (int i = 0; i < NG; ++i) {
                    const float4 x = *reinterpret_cast<const float4*>(vs + t * XS + 128 * i + 4 * cl);
                    o[i][0] = fmaf(pw, x.x, o[i][0]);
                    o[i][1] = fmaf(pw, x.y, o[i][1]);
                    o[i][2] = fmaf(pw, x.z, o[i][2]);
                    o[i][3] = fmaf(pw, x.w, o[i][3]);
                }
            }
        }
        __syncthreads();
    }
    if (ch < p.grp) {
        const int hq = g * p.grp + ch;
        const int64_t slot = (((int64_t)b * p.Hq + hq) * p.n_chunks + chunk_id);
        float* dst = p.ws_o + slot * D;
#pragma unroll
        for (int i = 0; i < NG; ++i)
            *reinterpret_cast<float4*>(dst + 128 * i + 4 * cl) = make_float4(o[i][0], o[i][1], o[i][2], o[i][3]);
        if (cl == 0) {
            p.ws_ml[slot * 2] = m_run;
            p.ws_ml[slot * 2 + 1] = l_run;
        }
    }
}

// Combines the chunk partials of (sequence, query head) by log-sum-exp;
// launched as a programmatic dependent of the partial kernel.  The chunk
// weights exp(m_c - M) and the total L = sum_c w_c l_c are formed once, in
// shared memory; then 1024 threads take the D dims 1024 / D ways over the
// chunks, each with its loads in flight together, and one shared-memory pass
// adds the ways.
constexpr int kMergeThreads = 1024;
__global__ void __launch_bounds__(kMergeThreads) k2v4_merge_kernel(K2V4DecodeParams p, float* __restrict__ out) {
    grid_dependency_wait();
    extern __shared__ float smw[];   // [n_chunks] weights
    __shared__ float red[kMergeThreads];
    __shared__ float wred[32];
    const int hq = blockIdx.x, b = blockIdx.y, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int D = p.c.D, n = p.n_chunks;
    const int64_t base = ((int64_t)b * p.Hq + hq) * n;
    float mloc = -INFINITY;
    for (int c = t; c < n; c += kMergeThreads) mloc = fmaxf(mloc, p.ws_ml[(base + c) * 2]);
    mloc = warp_max(mloc);
    if (lane == 0) wred[warp] = mloc;
    __syncthreads();
    float M = -INFINITY;
    for (int i = 0; i < kMergeThreads / 32; ++i) M = fmaxf(M, wred[i]);
    float lloc = 0.0f;
    for (int c = t; c < n; c += kMergeThreads) {
        const float2 ml = *reinterpret_cast<const float2*>(p.ws_ml + (base + c) * 2);
        const float w = ml.x == -INFINITY ? 0.0f : expf(ml.x - M);
        smw[c] = w;
        lloc = fmaf(w, ml.y, lloc);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) lloc += __shfl_xor_sync(0xffffffffu, lloc, o);
    __syncthreads();   // every warp has read wred; the weights are stored
    if (lane == 0) wred[warp] = lloc;
    __syncthreads();
    float L = 0.0f;
    for (int i = 0; i < kMergeThreads / 32; ++i) L += wred[i];
    const int ways = kMergeThreads / D, d = t % D, way = t / D;
    float acc = 0.0f;
    if (way < ways) {
#pragma unroll 16
        for (int c = way; c < n; c += ways) acc = fmaf(smw[c], p.ws_o[(base + c) * D + d], acc);
    }
    red[t] = acc;
    __syncthreads();
    if (t < D) {
        float sum = 0.0f;
        for (int k = 0; k < ways; ++k) sum += red[k * D + t];
        out[((int64_t)b * p.Hq + hq) * D + t] = L > 0.0f ? sum / L : 0.0f;
    }
}

cudaError_t launch_k2v4_merge(const K2V4DecodeParams& p, float* out, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.Hq, (unsigned)p.batch);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = (size_t)p.n_chunks * sizeof(float);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    timing_mark(stream, 1);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k2v4_merge_kernel, p, out);
    timing_mark(stream, 2);
    return e;
}

// ---------------------------------------------------------------------------
// Tensor-core decode
// ---------------------------------------------------------------------------
using namespace tc;
constexpr int kRowsT = 128;     // cells per tile: the MMA M
constexpr int kNq = 16;         // MMA N: 8 heads as f16 + their residuals (score), heads (context)
constexpr int kThreadsT = 256;
constexpr uint32_t kChunkT = kRowsT * 128;   // 128 cells x 64 dims f16, 128-byte swizzle

template <int D>
struct SmemT {
    static constexpr int kChunks = D / 64;
    // one f16 operand region: K for the score, then (once the score MMAs have
    // read it) V for the context; at about 105 KB in all for D = 256, two
    // pipelines share a CTA (and an SM), each one's serial steps hiding
    // behind the other's
    static constexpr uint32_t kOffK = 0;
    static constexpr uint32_t kOffV = kOffK;
    static constexpr uint32_t kOffQ = kOffK + kChunks * kChunkT;     // kChunks x (16 rows x 128 B)
    static constexpr uint32_t kOffP = kOffQ + kChunks * kNq * 128;    // 2 x (16 rows x 128 B): P^T by 64 cells
    static constexpr uint32_t kOffRed = kOffP + 2 * kNq * 128;        // [4 warps][8] max, [4][8] sums
    static constexpr uint32_t kOffState = kOffRed + 2 * 4 * 8 * 4;    // running max, sum, qmax (8 each), levels (4)
    static constexpr uint32_t kOffBar = kOffState + 3 * 8 * 4 + 16;
    static constexpr uint32_t kOffMisc = kOffBar + 4 * 8;             // abort flag, TMEM base
    // raw bytes of a tile: K codes (128 x D/4) and the 4 groups' K scales
    // (4 x D fp16) in one buffer, V blocks (128 x D/32 x 18) in another, each
    // refilled for the next tile as soon as its own dequantization is done
    static constexpr uint32_t kRawKc = kRowsT * D / 4, kRawKs = 4 * 2 * D, kRawVb = kRowsT * (D / 32) * 18;
    static constexpr uint32_t kOffRawK = (kOffMisc + 16 + 127) / 128 * 128;
    static constexpr uint32_t kOffRawV = kOffRawK + kRawKc + kRawKs;
    static constexpr uint32_t kBytes = kOffRawV + kRawVb;
    static constexpr uint32_t kStride = (kBytes + 1023) / 1024 * 1024;   // one pipeline's region
};
static_assert(2 * SmemT<256>::kStride <= 232448, "two pipelines per CTA");

constexpr uint32_t kColS = 0, kColO = 32, kTmemColsT = 64;
constexpr uint32_t kIdescK2Score = idesc_f16(128, kNq, false, false);
constexpr uint32_t kIdescK2Ctx = idesc_f16(128, kNq, true, false);

// Bulk K values enter the f16 operand scaled by kK2Gamma: the two level
// magnitudes times it round to f16 within 1.6e-5 relative (2.4e-4 unscaled;
// gen_codebook.py --k2-level-scale), so a K value is one correctly rounded f16
// product of (level, scale).  Overlay rows keep their exact fp16 K; the
// softmax divides the scores of bulk rows by the scale.
constexpr float kK2Gamma = 1.126953125f;

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
    const __half2 z = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&z);
}
__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
    const __half2 z = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&z);
}
// Two q4_0 codes (each 0..15 in the low 4 bits of a 16-bit half) -> half2
// (code - 8) * d, one correctly rounded f16 multiply: 0x6400 | c is 1024 + c
// in f16 and 0x6408 is 1032, so the subtraction is exact.
__device__ __forceinline__ uint32_t q4_pair(uint32_t codes2, uint32_t d2) {
    return hmul2_bits(hsub2_bits(codes2 | 0x64006400u, 0x64086408u), d2);
}

// Stages the raw bytes of the tile at cells [t0, t0 + nt), rounded up to
// whole 32-cell groups (t0 a multiple of 32): the K codes and K scales (two
// bulk copies into the K buffer) or the V blocks (one into the V buffer), each
// contiguous in the cache, issued by one thread on the TMA engine and
// completing on the buffer's mbarrier.  A sequence may end inside its last
// group (after appends); the cells past its end lie inside the pool
// (capacities are multiples of 32, every size and source offset a multiple of
// 16 bytes) and are masked by the caller.
template <int D, bool V>
__device__ __forceinline__ void stage_tile(const K2V4DecodeParams& p, int64_t seq, int64_t t0, int nt,
                                           unsigned char* dst, uint64_t* bar) {
    const int ns = (nt + kG - 1) / kG * kG;
    const uint32_t mb = smem_u32(bar);
    const unsigned char* src[2];
    uint32_t off[2], bytes[2];
    int n;
    if (V) {
        src[0] = p.v_blocks + (seq * p.c.cap + t0) * (D / 32) * 18;
        off[0] = 0;
        bytes[0] = ns * (D / 32) * 18;
        n = 1;
    } else {
        src[0] = p.k_codes + (seq * p.c.cap + t0) * (D / 4);
        src[1] = reinterpret_cast<const unsigned char*>(p.k_scales + (seq * (p.c.cap / kG) + t0 / kG) * D);
        off[0] = 0;
        off[1] = SmemT<D>::kRawKc;
        bytes[0] = ns * (D / 4);
        bytes[1] = (ns / kG) * 2 * D;
        n = 2;
    }
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb),
                 "r"(n == 1 ? bytes[0] : bytes[0] + bytes[1])
                 : "memory");
    for (int i = 0; i < n; ++i)
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(smem_u32(dst + off[i])), "l"(src[i]), "r"(bytes[i]), "r"(mb)
                     : "memory");
}

// Named barrier `id` of pipeline `half` (ids 1-3 and 4-6; 0 is the CTA's).
__device__ __forceinline__ void pipe_bar(int half, int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(3 * half + id), "r"(n) : "memory");
}

// One decode pipeline: 256 threads (local `tid`) over chunk `chunk_id` with
// their own shared-memory region, TMEM columns, mbarriers and named barriers.
template <int D>
__device__ __forceinline__ void k2v4_tc_pipe(const K2V4DecodeParams& p, unsigned char* smem_raw, uint32_t tmem,
                                             int tid, int half, int chunk_id) {
    using SM = SmemT<D>;
    unsigned char* sK = smem_raw + SM::kOffK;
    unsigned char* sV = smem_raw + SM::kOffV;
    unsigned char* sQ = smem_raw + SM::kOffQ;
    unsigned char* sP = smem_raw + SM::kOffP;
    float* sRedM = reinterpret_cast<float*>(smem_raw + SM::kOffRed);
    float* sRedL = sRedM + 32;
    float* sM = reinterpret_cast<float*>(smem_raw + SM::kOffState);
    float* sL = sM + 8;
    float* sQmax = sL + 8;
    float* sLv = sQmax + 8;   // the 4 K levels
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + SM::kOffBar);   // 0 score, 1 context, 2 raw K, 3 raw V
    volatile int* sAbort = reinterpret_cast<volatile int*>(smem_raw + SM::kOffMisc);
    unsigned char* sRawK = smem_raw + SM::kOffRawK;
    unsigned char* sRawV = smem_raw + SM::kOffRawV;

    const int lane = tid & 31, warp = tid >> 5;
    const int g = blockIdx.y, b = blockIdx.z;
    const int64_t seq = (int64_t)b * p.c.H + g;
    const int64_t c0 = (int64_t)chunk_id * p.chunk;
    const int64_t c1 = min(c0 + p.chunk, p.c.T);
    const int n_tiles = (int)((c1 - c0 + kRowsT - 1) / kRowsT);
    const int grp = p.grp;

    if (tid == 32) {
        for (int i = 0; i < 4; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&bars[i])), "r"(1u));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // the swizzled operands need a 1024-byte base (2: refused; a wait that
        // runs out raises the flag to 1)
        *sAbort = smem_u32(smem_raw) & 1023u ? 2 : 0;
        if (n_tiles > 0) {
            stage_tile<D, false>(p, seq, c0, (int)min((int64_t)kRowsT, c1 - c0), sRawK, &bars[2]);
            stage_tile<D, true>(p, seq, c0, (int)min((int64_t)kRowsT, c1 - c0), sRawV, &bars[3]);
        }
    }
    if (tid < 8) {
        sM[tid] = -INFINITY;
        sL[tid] = 0.0f;
    }
    if (tid < 4) sLv[tid] = p.c.lv[tid];
    // P^T rows 8..15 (no head) stay zero; rows of heads past the group too
    for (int i = tid; i < 2 * kNq * 128 / 16; i += kThreadsT) reinterpret_cast<uint4*>(sP)[i] = make_uint4(0, 0, 0, 0);

    // ---- query: the group's heads as an f16 pair (value, residual), scaled
    // by a power of two so that every element stays below 2^14 ----
    const float* qg = p.q + ((int64_t)b * p.Hq + (int64_t)g * grp) * D;
    float qmax = 0.0f;
    for (int i = tid; i < grp * D; i += kThreadsT) qmax = fmaxf(qmax, fabsf(qg[i]));
    qmax = warp_max(qmax);
    if (lane == 0) sQmax[warp] = qmax;
    pipe_bar(half, 1, kThreadsT);
    float q_max = 0.0f;
    for (int i = 0; i < 8; ++i) q_max = fmaxf(q_max, sQmax[i]);
    int e_q = 0;
    if (q_max > 0.0f) frexpf(q_max, &e_q);
    const float q_scale = q_max > 0.0f ? ldexpf(1.0f, 14 - e_q) : 1.0f;
    const float cz = p.sm_scale * kLog2e * (q_max > 0.0f ? ldexpf(1.0f, e_q - 14) : 1.0f);
    // the 4 scaled K levels as f16, bytes 0..7 of (lv01, lv23) for byte_perm lookups
    uint32_t lv01, lv23;
    {
        const __half2 a = __floats2half2_rn(sLv[0] * kK2Gamma, sLv[1] * kK2Gamma);
        const __half2 c = __floats2half2_rn(sLv[2] * kK2Gamma, sLv[3] * kK2Gamma);
        lv01 = *reinterpret_cast<const uint32_t*>(&a);
        lv23 = *reinterpret_cast<const uint32_t*>(&c);
    }

    for (int i = tid; i < 8 * D; i += kThreadsT) {
        const int h = i / D, d = i - h * D;
        const float x = h < grp ? qg[h * D + d] * q_scale : 0.0f;
        const __half hi = __float2half_rn(x);
        const __half lo = __float2half_rn(x - __half2float(hi));
        unsigned char* chunk = sQ + (d >> 6) * (kNq * 128);
        *reinterpret_cast<__half*>(chunk + sw128(h, (d & 63) * 2)) = hi;
        *reinterpret_cast<__half*>(chunk + sw128(8 + h, (d & 63) * 2)) = lo;
    }
    tc_before();
    pipe_bar(half, 1, kThreadsT);
    tc_after();

    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    // the raw copy of each buffer that its issuing thread (0 for K, 128 for
    // V) has not yet seen land: copy t is waited for before copy t + 1 is
    // issued into the same buffer, and one still pending when the loop ends
    // (after an abort) is waited for before the CTA leaves
    int pend_k = n_tiles > 0 ? 0 : -1, pend_v = pend_k;
    for (int t = 0; t < n_tiles; ++t) {
        const int64_t t0 = c0 + (int64_t)t * kRowsT;
        const int nt = (int)min((int64_t)kRowsT, c1 - t0);
        if (mbar_wait(&bars[2], (uint32_t)t & 1u, sAbort, p.wait_limit) && pend_k == t) pend_k = -1;
        // the f16 region holds the previous tile's V until its context MMAs
        // have read it
        if (t > 0) mbar_wait(&bars[1], (uint32_t)(t - 1) & 1u, sAbort, p.wait_limit);
        const unsigned char* raw_kc = sRawK;
        const uint16_t* raw_ks = reinterpret_cast<const uint16_t*>(sRawK + SM::kRawKc);
        const unsigned char* raw_vb = sRawV;
        // ---- K of the tile to f16 (cells on rows, 64 dims per chunk), all
        // warps.  A whole tile of bulk cells (no sink or window cell, the
        // usual case) takes a branch-free loop whose unrolled iterations
        // interleave.
        const bool plain = nt == kRowsT && t0 >= p.c.n_sink && t0 + kRowsT <= p.c.T - p.c.n_window;
        // the fp16 scales of dims 32j .. 32j + 31 in the K scale group g
        auto k_scales = [&](int g, int j, uint32_t (&scw)[16]) {
            const uint4* scq = reinterpret_cast<const uint4*>(raw_ks + g * D + 32 * j);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 w = scq[i];
                scw[4 * i] = w.x; scw[4 * i + 1] = w.y; scw[4 * i + 2] = w.z; scw[4 * i + 3] = w.w;
            }
        };
        // 2-bit codes (32 dims = 8 bytes; dims 2m, 2m+1 in bits 4m..4m+3)
        // times the group's per-dim fp16 scales, pairwise in f16.  A code
        // byte (dims 4q .. 4q+3) is spread to one code per byte by two masked
        // multiplies (even codes, odd codes: no carries cross a byte), then
        // x * 0x22 + 0x10 turns each code c into the byte-permute selector
        // nibbles (2c, 2c + 1) of its f16 level: the low half selects the pair
        // of dims 4q, 4q+1, the high half the pair 4q+2, 4q+3
        auto k_dec = [&](int r, int j, const uint32_t (&scw)[16], uint32_t (&kw)[16]) {
            const uint2 kc = *reinterpret_cast<const uint2*>(raw_kc + r * (D / 4) + 8 * j);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint32_t t = (q < 4 ? kc.x : kc.y) >> (8 * (q & 3));
                const uint32_t x = (((t & 0x33u) * 0x1001u) | ((t & 0xCCu) * 0x40040u)) & 0x03030303u;
                const uint32_t sel = x * 0x22u + 0x10101010u;
                kw[2 * q] = hmul2_bits(__byte_perm(lv01, lv23, sel), scw[2 * q]);
                kw[2 * q + 1] = hmul2_bits(__byte_perm(lv01, lv23, sel >> 16), scw[2 * q + 1]);
            }
        };
        auto k_bulk = [&](int r, int j, uint32_t (&kw)[16]) {
            uint32_t scw[16];
            k_scales(r / kG, j, scw);
            k_dec(r, j, scw, kw);
        };
        auto k_store = [&](int r, int j, const uint32_t (&kw)[16]) {
            unsigned char* kdst = sK + (j >> 1) * kChunkT;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<uint4*>(kdst + sw128(r, (j & 1) * 64 + 16 * i)) =
                    make_uint4(kw[4 * i], kw[4 * i + 1], kw[4 * i + 2], kw[4 * i + 3]);
        };
        if (plain) {
            // warp w takes cells 16w .. 16w + 15 (one scale group) and every
            // 32-dim slice; a thread keeps one slice, so its scales load once
            // A 16-byte store is served 8 lanes at a time, and the lanes of
            // one such phase must cover the 8 swizzled 16-byte units of a
            // row: lanes 8p .. 8p + 7 take kQ consecutive cells (distinct
            // swizzle phases) and 8 / kQ slices (the two halves of a chunk
            // row when kQ = 4), where one cell and 8 slices hit 2 units 4 ways
            constexpr int kS = D / 32, kQ = 32 / kS;
            const int q = lane % kQ, j = lane / kQ;
            uint32_t scw[16];
            k_scales((16 * warp) / kG, j, scw);
#pragma unroll
            for (int k = 0; k < 16 / kQ; ++k) {
                const int r = 16 * warp + q + kQ * k;
                uint32_t kw[16];
                k_dec(r, j, scw, kw);
                k_store(r, j, kw);
            }
        } else {
            for (int it = tid; it < kRowsT * (D / 32); it += kThreadsT) {
                const int r = it / (D / 32), j = it - r * (D / 32);
                uint32_t kw[16];
                if (r < nt) {
                    const int64_t slot = overlay_slot(t0 + r, p.c);
                    if (slot >= 0) {
                        // exact fp16 copy
                        const uint4* kwin =
                            reinterpret_cast<const uint4*>(p.k_win + (seq * p.c.slots + slot) * D + 32 * j);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint4 a = __ldg(kwin + i);
                            kw[4 * i] = a.x; kw[4 * i + 1] = a.y; kw[4 * i + 2] = a.z; kw[4 * i + 3] = a.w;
                        }
                    } else {
                        k_bulk(r, j, kw);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) kw[i] = 0u;
                }
                k_store(r, j, kw);
            }
        }
        fence_async_smem();
        tc_before();
        pipe_bar(half, 1, kThreadsT);
        tc_after();
        // ---- score MMAs (issued after the previous context MMAs: its commit
        // covers both) ----
        if (tid == 0 && !*sAbort) {
            const uint64_t dk = umma_desc(smem_u32(sK), 16, 1024), dq = umma_desc(smem_u32(sQ), 16, 1024);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    umma_f16(tmem + kColS, dk + c * (kChunkT >> 4) + 2 * ks, dq + c * (kNq * 128 >> 4) + 2 * ks,
                             kIdescK2Score, (c | ks) ? 1u : 0u);
            umma_commit(&bars[0]);
        }
        // the raw K buffer is free (every thread fenced its reads before the
        // barrier): the next tile's K streams in during this one
        if (tid == 0 && pend_k < 0 && t + 1 < n_tiles && !*sAbort) {
            stage_tile<D, false>(p, seq, t0 + kRowsT, (int)min((int64_t)kRowsT, c1 - t0 - kRowsT), sRawK, &bars[2]);
            pend_k = t + 1;
        }
        if (warp >= 4) {
            // ---- V of the tile to f16, warps 4-7, alongside the softmax, once
            // the score MMAs have read K out of the shared f16 region ----
            mbar_wait(&bars[0], (uint32_t)t & 1u, sAbort, p.wait_limit);
            if (mbar_wait(&bars[3], (uint32_t)t & 1u, sAbort, p.wait_limit) && pend_v == t) pend_v = -1;
            auto v_bulk = [&](int r, int j, uint32_t (&vw)[16]) {
                // q4_0 block (d, then 16 bytes: element e in the low nibble of
                // byte e, e + 16 in the high nibble)
                const uint16_t* blk = reinterpret_cast<const uint16_t*>(raw_vb + (r * (D / 32) + j) * 18);
                const uint32_t d2 = (uint32_t)blk[0] * 0x10001u;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t w = (uint32_t)blk[1 + 2 * m] | ((uint32_t)blk[2 + 2 * m] << 16);
                    const uint32_t p01 = __byte_perm(w, 0u, 0x4140u), p23 = __byte_perm(w, 0u, 0x4342u);
                    vw[2 * m] = q4_pair(p01 & 0x000F000Fu, d2);
                    vw[2 * m + 1] = q4_pair(p23 & 0x000F000Fu, d2);
                    vw[8 + 2 * m] = q4_pair((p01 >> 4) & 0x000F000Fu, d2);
                    vw[9 + 2 * m] = q4_pair((p23 >> 4) & 0x000F000Fu, d2);
                }
            };
            // four consecutive q4_0 blocks (72 bytes, 8-byte aligned: a cell's
            // blocks are contiguous and D / 32 of them take 9 D / 16 bytes)
            // read as nine 8-byte words; block jj's scale and nibbles sit at
            // byte 18 jj and 18 jj + 2
            auto v_quad = [&](int r, int u, auto&& emit) {
                const uint2* src = reinterpret_cast<const uint2*>(raw_vb + (r * (D / 32) + 4 * u) * 18);
                uint32_t w[18];
#pragma unroll
                for (int i = 0; i < 9; ++i) {
                    const uint2 x = src[i];
                    w[2 * i] = x.x;
                    w[2 * i + 1] = x.y;
                }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int b = 9 * jj / 2;   // first word of the block (18 jj / 4)
                    uint32_t d16, nb[4];
                    if ((jj & 1) == 0) {
                        d16 = w[b] & 0xffffu;
#pragma unroll
                        for (int m = 0; m < 4; ++m) nb[m] = __funnelshift_r(w[b + m], w[b + m + 1], 16);
                    } else {
                        d16 = w[b] >> 16;
#pragma unroll
                        for (int m = 0; m < 4; ++m) nb[m] = w[b + 1 + m];
                    }
                    const uint32_t d2 = d16 * 0x10001u;
                    uint32_t vw[16];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const uint32_t p01 = __byte_perm(nb[m], 0u, 0x4140u), p23 = __byte_perm(nb[m], 0u, 0x4342u);
                        vw[2 * m] = q4_pair(p01 & 0x000F000Fu, d2);
                        vw[2 * m + 1] = q4_pair(p23 & 0x000F000Fu, d2);
                        vw[8 + 2 * m] = q4_pair((p01 >> 4) & 0x000F000Fu, d2);
                        vw[9 + 2 * m] = q4_pair((p23 >> 4) & 0x000F000Fu, d2);
                    }
                    emit(4 * u + jj, vw);
                }
            };
            auto v_store = [&](int r, int j, const uint32_t (&vw)[16]) {
                unsigned char* vdst = sV + (j >> 1) * kChunkT;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    *reinterpret_cast<uint4*>(vdst + sw128(r, (j & 1) * 64 + 16 * i)) =
                        make_uint4(vw[4 * i], vw[4 * i + 1], vw[4 * i + 2], vw[4 * i + 3]);
            };
            if (plain) {
#pragma unroll
                for (int it = tid - 128; it < kRowsT * (D / 128); it += kThreadsT - 128) {
                    // cell and run of 4 blocks: each 8-lane store phase takes 8
                    // consecutive cells (8 distinct swizzle phases) of one run
                    const int r = D == 256 ? (it & 7) + 8 * (it >> 4) : it;
                    const int u = D == 256 ? (it >> 3) & 1 : 0;
                    v_quad(r, u, [&](int j, const uint32_t (&vw)[16]) { v_store(r, j, vw); });
                }
            } else {
                for (int it = tid - 128; it < kRowsT * (D / 32); it += kThreadsT - 128) {
                    const int r = it / (D / 32), j = it - r * (D / 32);
                    uint32_t vw[16];
                    if (r < nt) {
                        const int64_t slot = overlay_slot(t0 + r, p.c);
                        if (slot >= 0) {
                            const uint4* vwin =
                                reinterpret_cast<const uint4*>(p.v_win + (seq * p.c.slots + slot) * D + 32 * j);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const uint4 c = __ldg(vwin + i);
                                vw[4 * i] = c.x; vw[4 * i + 1] = c.y; vw[4 * i + 2] = c.z; vw[4 * i + 3] = c.w;
                            }
                        } else {
                            v_bulk(r, j, vw);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) vw[i] = 0u;
                    }
                    v_store(r, j, vw);
                }
            }
            // the raw V buffer is free once warps 4-7 have fenced their reads
            fence_async_smem();
            pipe_bar(half, 3, 128);
            if (tid == 128 && pend_v < 0 && t + 1 < n_tiles && !*sAbort) {
                stage_tile<D, true>(p, seq, t0 + kRowsT, (int)min((int64_t)kRowsT, c1 - t0 - kRowsT), sRawV,
                                    &bars[3]);
                pend_v = t + 1;
            }
        } else {
            // ---- softmax: warps 0-3, thread = cell (TMEM lane), the group's
            // heads.  The score commit covers the previous context MMAs too, so
            // P^T and O^T are free once it has arrived.
            mbar_wait(&bars[0], (uint32_t)t & 1u, sAbort, p.wait_limit);
            tc_after();
            uint32_t sv[16];
            tmem_ld16(tmem + lane_base + kColS, sv);
            tmem_wait_ld();
            const int r = 32 * warp + lane;
            // bulk rows carry K scaled by kK2Gamma, overlay rows do not
            const float rz = overlay_slot(t0 + r, p.c) >= 0 ? cz : cz * (1.0f / kK2Gamma);
            float z[8];
#pragma unroll
            for (int h = 0; h < 8; ++h)
                z[h] = (r < nt && h < grp) ? (__uint_as_float(sv[h]) + __uint_as_float(sv[8 + h])) * rz : -INFINITY;
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const float m = warp_max(z[h]);
                if (lane == 0) sRedM[warp * 8 + h] = m;
            }
            pipe_bar(half, 2, 128);
            float mnew[8], alpha[8], pv[8];
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const float mt = fmaxf(fmaxf(sRedM[h], sRedM[8 + h]), fmaxf(sRedM[16 + h], sRedM[24 + h]));
                mnew[h] = fmaxf(sM[h], mt);
                alpha[h] = (sM[h] == -INFINITY) ? 0.0f : ex2(sM[h] - mnew[h]);
                pv[h] = mnew[h] == -INFINITY ? 0.0f : ex2(z[h] - mnew[h]);
            }
            unsigned char* pc = sP + (r >> 6) * (kNq * 128);
#pragma unroll
            for (int h = 0; h < 8; ++h) *reinterpret_cast<__half*>(pc + sw128(h, (r & 63) * 2)) = __float2half_rn(pv[h]);
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                float l = pv[h];
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(kFull, l, o);
                if (lane == 0) sRedL[warp * 8 + h] = l;
            }
            if (t > 0) {
                // rescale O^T (its lanes are dims, its first 8 columns heads)
#pragma unroll
                for (int m = 0; m < D / 128; ++m) {
                    uint32_t ov[16];
                    tmem_ld16(tmem + lane_base + kColO + 16 * m, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < 8; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
                    tmem_st16(tmem + lane_base + kColO + 16 * m, ov);
                }
                tmem_wait_st();
            }
            pipe_bar(half, 2, 128);
            if (tid < 8) {
                float a = 0.0f, mn = 0.0f;
#pragma unroll
                for (int h = 0; h < 8; ++h)
                    if (h == tid) {
                        a = alpha[h];
                        mn = mnew[h];
                    }
                sL[tid] = sL[tid] * a + ((sRedL[tid] + sRedL[8 + tid]) + (sRedL[16 + tid] + sRedL[24 + tid]));
                sM[tid] = mn;
            }
        }
        fence_async_smem();
        tc_before();
        pipe_bar(half, 1, kThreadsT);
        tc_after();
        // ---- context MMAs ----
        if (tid == 0 && !*sAbort) {
            const uint64_t dv = umma_desc(smem_u32(sV), kChunkT, 1024), dp = umma_desc(smem_u32(sP), 16, 1024);
#pragma unroll
            for (int m = 0; m < D / 128; ++m)
#pragma unroll
                for (int ks = 0; ks < kRowsT / 16; ++ks)
                    umma_f16(tmem + kColO + 16 * m, dv + 2 * m * (kChunkT >> 4) + 128 * ks,
                             dp + (ks >> 2) * (kNq * 128 >> 4) + 2 * (ks & 3), kIdescK2Ctx, (t > 0 || ks > 0) ? 1u : 0u);
            umma_commit(&bars[1]);
        }
    }
    // ---- epilogue: O^T -> chunk partials (natural-log max, sum) ----
    if (n_tiles > 0) {
        volatile int never = 0;
        if (!mbar_wait(&bars[1], (uint32_t)(n_tiles - 1) & 1u, &never)) *sAbort = 1;
        // after an abort the loop stopped waiting for its raw tiles: a bulk
        // copy still in flight lands before the CTA leaves
        if (tid == 0 && pend_k >= 0 && !mbar_wait(&bars[2], (uint32_t)pend_k & 1u, &never)) *sAbort = 1;
        if (tid == 128 && pend_v >= 0 && !mbar_wait(&bars[3], (uint32_t)pend_v & 1u, &never)) *sAbort = 1;
    }
    tc_after();
    if (*sAbort) {
        if (tid == 0) atomicCAS(p.err, 0, *sAbort == 2 ? (int32_t)KVQ_ERR_DEVICE : (int32_t)KVQ_ERR_TIMEOUT);
    } else if (warp < 4) {
#pragma unroll
        for (int m = 0; m < D / 128; ++m) {
            uint32_t ov[16];
            tmem_ld16(tmem + lane_base + kColO + 16 * m, ov);
            tmem_wait_ld();
            const int d = 128 * m + 32 * warp + lane;
#pragma unroll
            for (int h = 0; h < 8; ++h)
                if (h < grp) {
                    const int64_t slot = ((int64_t)b * p.Hq + (int64_t)g * grp + h) * p.n_chunks + chunk_id;
                    p.ws_o[slot * D + d] = n_tiles > 0 ? __uint_as_float(ov[h]) : 0.0f;
                }
        }
        if (tid < grp) {
            const int64_t slot = ((int64_t)b * p.Hq + (int64_t)g * grp + tid) * p.n_chunks + chunk_id;
            p.ws_ml[slot * 2] = sM[tid] * kLn2;
            p.ws_ml[slot * 2 + 1] = sL[tid];
        }
    }
}

// Two pipelines per CTA, each on its own chunk: a kernel that allocates TMEM
// runs one CTA per SM, and one pipeline's serial steps (dequantization, MMA
// waits, softmax) leave most of the SM idle; the second fills it.
template <int D>
__global__ void __launch_bounds__(2 * kThreadsT, 1) k2v4_tc_kernel(K2V4DecodeParams p) {
    launch_dependents();
    extern __shared__ __align__(1024) unsigned char smem_all[];
    const int half = threadIdx.x / kThreadsT;
    // the TMEM base goes to a word of pipeline 0's region that it never uses
    uint32_t* slot = reinterpret_cast<uint32_t*>(smem_all + SmemT<D>::kOffMisc + 4);
    if (threadIdx.x < 32) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                     "r"(2 * kTmemColsT));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t base = *slot;
    const int chunk_id = 2 * (int)blockIdx.x + half;
    if (chunk_id < p.n_chunks)
        k2v4_tc_pipe<D>(p, smem_all + half * SmemT<D>::kStride, base + half * kTmemColsT, (int)threadIdx.x % kThreadsT,
                        half, chunk_id);
    tc_before();
    __syncthreads();
    tc_after();
    if (threadIdx.x < 32)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(2 * kTmemColsT));
}

K2V4Params make_params(const kvq_k2v4_layout& L, int64_t T, int64_t cap) {
    K2V4Params p{};
    p.H = L.n_kv_heads;
    p.D = L.head_dim;
    p.n_sink = L.n_sink;
    p.n_window = L.n_window;
    p.n_slack = L.n_slack;
    p.slots = L.n_sink + L.n_window + L.n_slack;
    p.T = T;
    p.cap = cap;
    p.k_gain = L.k_gain;
    const Codebook4 cb = k2_codebook();
    for (int i = 0; i < 4; ++i) {
        p.lv[i] = cb.lv[i];
        p.th[i] = cb.th[i];
    }
    return p;
}

}  // namespace

cudaError_t launch_k2v4_encode(const kvq_k2v4_layout& L, const float* k, const float* v, int32_t batch,
                               int64_t n_cells, int64_t cap, uint8_t* k_codes, uint16_t* k_scales,
                               uint8_t* v_blocks, uint16_t* k_win, uint16_t* v_win, int32_t* err,
                               cudaStream_t stream) {
    if (batch == 0 || n_cells == 0) return cudaSuccess;
    const K2V4Params p = make_params(L, n_cells, cap);
    k2_encode_kernel<<<dim3((unsigned)(n_cells / kG), p.H, batch), p.D, 0, stream>>>(k, p, k_codes, k_scales, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    v4_encode_kernel<<<dim3((unsigned)n_cells, p.H, batch), p.D, 0, stream>>>(k, v, p, n_cells, 0, v_blocks, k_win,
                                                                              v_win, err);
    return cudaGetLastError();
}

cudaError_t launch_k2v4_append(const kvq_k2v4_layout& L, const float* k_new, const float* v_new, int32_t batch,
                               int64_t n_past, int64_t n_new, int64_t cap, uint8_t* k_codes, uint16_t* k_scales,
                               uint8_t* v_blocks, uint16_t* k_win, uint16_t* v_win, int32_t* err,
                               cudaStream_t stream) {
    if (batch == 0 || n_new == 0) return cudaSuccess;
    const K2V4Params p = make_params(L, n_past + n_new, cap);   // overlay window at the new length
    const int64_t groups = (n_past + n_new - 1) / kG - n_past / kG + 1;
    k2_append_kernel<<<dim3((unsigned)groups, p.H, batch), p.D, 0, stream>>>(k_new, p, n_past, n_new, k_codes,
                                                                            k_scales, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    v4_encode_kernel<<<dim3((unsigned)n_new, p.H, batch), p.D, 0, stream>>>(k_new, v_new, p, n_new, n_past,
                                                                            v_blocks, k_win, v_win, err);
    return cudaGetLastError();
}

bool k2v4_tc_supported(const kvq_k2v4_layout& L) { return L.head_dim == 128 || L.head_dim == 256; }

K2V4Plan plan_k2v4(const kvq_k2v4_layout& L, int32_t batch, int32_t, int64_t n_cells, bool tensor) {
    K2V4Plan pl{};
    pl.tensor = tensor;
    if (tensor) {
        // about one CTA (two pipelines, a chunk each) per SM, chunks of whole
        // 128-cell tiles
        const int64_t per = std::max<int64_t>(1, (int64_t)batch * L.n_kv_heads);
        const int64_t target = std::max<int64_t>(1, (int64_t)kSmSMs * 2 / per);
        int64_t chunk = (std::max<int64_t>(n_cells, 1) + target - 1) / target;
        chunk = std::max<int64_t>(kRowsT, (chunk + kRowsT - 1) / kRowsT * kRowsT);
        pl.chunk = chunk;
        pl.n_chunks = (int32_t)((n_cells + chunk - 1) / chunk);
        return pl;
    }
    const int64_t per = std::max<int64_t>(1, (int64_t)batch * L.n_kv_heads);
    const int64_t target = std::max<int64_t>(1, (int64_t)kSmSMs * 4 / per);
    int64_t chunk = (std::max<int64_t>(n_cells, 1) + target - 1) / target;
    chunk = std::max<int64_t>(kTC, (chunk + kTC - 1) / kTC * kTC);
    pl.chunk = chunk;
    pl.n_chunks = (int32_t)((n_cells + chunk - 1) / chunk);
    return pl;
}

size_t k2v4_partial_bytes(const kvq_k2v4_layout& L, int32_t batch, int32_t n_q_heads, const K2V4Plan& pl) {
    return (size_t)batch * n_q_heads * pl.n_chunks * (L.head_dim + 2) * sizeof(float);
}

cudaError_t launch_k2v4_decode(const kvq_k2v4_layout& L, const float* q, int32_t batch, int32_t n_q_heads,
                               int64_t n_cells, int64_t cap, const uint8_t* k_codes, const uint16_t* k_scales,
                               const uint8_t* v_blocks, const uint16_t* k_win, const uint16_t* v_win,
                               float sm_scale, float* out, void* workspace, const K2V4Plan& plan,
                               cudaStream_t stream) {
    if (batch == 0 || n_q_heads == 0) return cudaSuccess;
    K2V4DecodeParams p{};
    p.c = make_params(L, n_cells, cap);
    p.batch = batch;
    p.Hq = n_q_heads;
    p.grp = n_q_heads / L.n_kv_heads;
    p.chunk = plan.chunk;
    p.n_chunks = plan.n_chunks;
    p.sm_scale = sm_scale;
    p.q = q;
    p.k_codes = k_codes;
    p.k_scales = k_scales;
    p.v_blocks = v_blocks;
    p.k_win = k_win;
    p.v_win = v_win;
    p.err = static_cast<int32_t*>(workspace);
    p.wait_limit = kWaitLimit;
    char* ws = static_cast<char*>(workspace) + kWsHeader;
    p.ws_o = reinterpret_cast<float*>(ws);
    p.ws_ml = p.ws_o + (size_t)batch * n_q_heads * plan.n_chunks * L.head_dim;
    const dim3 grid(plan.n_chunks, L.n_kv_heads, batch);
    cudaError_t e = cudaSuccess;
    timing_mark(stream, 0);
    if (plan.tensor) {
        switch (L.head_dim) {
#define KVQ_TC_CASE(DD)                                                                                 \
    case DD: {                                                                                          \
        e = cudaFuncSetAttribute(k2v4_tc_kernel<DD>, cudaFuncAttributeMaxDynamicSharedMemorySize,      \
                                 (int)(2 * SmemT<DD>::kStride));                                       \
        if (e != cudaSuccess) return e;                                                                 \
        k2v4_tc_kernel<DD><<<dim3((plan.n_chunks + 1) / 2, L.n_kv_heads, batch), 2 * kThreadsT,        \
                             2 * SmemT<DD>::kStride, stream>>>(p);                                      \
        break;                                                                                          \
    }
            KVQ_TC_CASE(128)
            KVQ_TC_CASE(256)
#undef KVQ_TC_CASE
            default: return cudaErrorInvalidValue;
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        return launch_k2v4_merge(p, out, stream);
    }
    switch (L.head_dim) {
#define KVQ_D_CASE(DD)                                                                                  \
    case DD: {                                                                                          \
        const size_t smem = ((size_t)(kHQ + 2 * kTC) * (DD + 4) + kTC * kHQ + 8) * sizeof(float) +     \
                            RawTileBytes<DD>::kTotal;                                                  \
        e = cudaFuncSetAttribute(k2v4_partial_kernel<DD>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                 (int)smem);                                                            \
        if (e != cudaSuccess) return e;                                                                 \
        k2v4_partial_kernel<DD><<<grid, kNT, smem, stream>>>(p);                                        \
        break;                                                                                          \
    }
        KVQ_D_CASE(128)
        KVQ_D_CASE(256)
        KVQ_D_CASE(512)
#undef KVQ_D_CASE
        default: return cudaErrorInvalidValue;
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_k2v4_merge(p, out, stream);
}

}  // namespace kvq
