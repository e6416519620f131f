// k2v4.cu -- the 2-bit-K / 4-bit-V GQA cache with an exact FP16 window ([P3]).
//
// Encode: K per (kv head, channel, 32-cell group) -- one thread per channel
// walks its 32 cells, forms the sum of squares in a fixed pairwise order,
// s = sqrt(ss/32), picks the nearest of 4 Lloyd-Max levels for x/s and stores
// fp16(k_gain * s) ([P3] Summary item 3: codes against the un-gained scale).
// V per cell and 32-dim block (q4_0) -- one warp per block.  Cells inside the
// sink/window overlay also get exact fp16 copies.
//
// Decode (fp32 CUDA cores): one CTA per (sequence, kv head, chunk of cells)
// serves the kv head's 8 query heads; tiles of 32 cells are dequantized to f32
// in shared memory (overlay cells take their fp16 copy), then scores, online
// softmax and the context follow as in the MLA path; a merge kernel combines
// the chunks by log-sum-exp.
#include "kvq_internal.cuh"

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
                                                          uint16_t* __restrict__ k_scales) {
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

// grid: (T, H, batch), block: D threads; warp w encodes 32-dim block w of the cell
__global__ void __launch_bounds__(kMaxD) v4_encode_kernel(const float* __restrict__ k, const float* __restrict__ v,
                                                          K2V4Params p, uint8_t* __restrict__ v_blocks,
                                                          uint16_t* __restrict__ k_win, uint16_t* __restrict__ v_win) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int64_t cell = blockIdx.x;
    const int g = blockIdx.y, b = blockIdx.z;
    const int64_t seq = (int64_t)b * p.H + g;
    const int64_t src = (seq * p.T + cell) * p.D + tid;
    const float x = __ldg(v + src);
    const float ax = fabsf(x);
    const float amax = warp_max(ax);
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
};

constexpr int kHQ = 8;   // query heads per CTA (one kv group)

template <int D>
__global__ void __launch_bounds__(kNT) k2v4_partial_kernel(K2V4DecodeParams p) {
    constexpr int XS = D + 4;
    extern __shared__ float4 smem4[];
    float* qs = reinterpret_cast<float*>(smem4);   // [8][XS]
    float* ks = qs + kHQ * XS;                      // [32][XS]
    float* vs = ks + kTC * XS;                      // [32][XS]
    float* P = vs + kTC * XS;                       // [32][8]
    float* alpha = P + kTC * kHQ;                   // [8]
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
        // dequantize K and V of the tile (overlay cells read their fp16 copy)
        const int64_t grp_idx = t0 / kG;
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
                    const uint8_t kb = p.k_codes[(seq * p.c.cap + cell) * (D / 4) + d / 4];
                    const float ksc = __half2float(__ushort_as_half(p.k_scales[(seq * (p.c.cap / kG) + grp_idx) * D + d]));
                    kv = p.c.lv[(kb >> (2 * (d & 3))) & 3] * ksc;
                    const uint8_t* blk = p.v_blocks + ((seq * p.c.cap + cell) * (D / 32) + d / 32) * 18;
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

__global__ void k2v4_merge_kernel(K2V4DecodeParams p, float* __restrict__ out) {
    const int hq = blockIdx.x, b = blockIdx.y;
    const int D = p.c.D;
    const int64_t base = ((int64_t)b * p.Hq + hq) * p.n_chunks;
    float M = -INFINITY;
    for (int c = 0; c < p.n_chunks; ++c) M = fmaxf(M, p.ws_ml[(base + c) * 2]);
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float L = 0.0f, acc = 0.0f;
        for (int c = 0; c < p.n_chunks; ++c) {
            const float w = M == -INFINITY ? 0.0f : expf(p.ws_ml[(base + c) * 2] - M);
            L += w * p.ws_ml[(base + c) * 2 + 1];
            acc = fmaf(w, p.ws_o[(base + c) * D + d], acc);
        }
        out[((int64_t)b * p.Hq + hq) * D + d] = L > 0.0f ? acc / L : 0.0f;
    }
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
                               uint8_t* v_blocks, uint16_t* k_win, uint16_t* v_win, cudaStream_t stream) {
    if (batch == 0 || n_cells == 0) return cudaSuccess;
    const K2V4Params p = make_params(L, n_cells, cap);
    k2_encode_kernel<<<dim3((unsigned)(n_cells / kG), p.H, batch), p.D, 0, stream>>>(k, p, k_codes, k_scales);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    v4_encode_kernel<<<dim3((unsigned)n_cells, p.H, batch), p.D, 0, stream>>>(k, v, p, v_blocks, k_win, v_win);
    return cudaGetLastError();
}

K2V4Plan plan_k2v4(const kvq_k2v4_layout& L, int32_t batch, int32_t, int64_t n_cells) {
    K2V4Plan pl{};
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
    char* ws = static_cast<char*>(workspace) + kWsHeader;
    p.ws_o = reinterpret_cast<float*>(ws);
    p.ws_ml = p.ws_o + (size_t)batch * n_q_heads * plan.n_chunks * L.head_dim;
    const dim3 grid(plan.n_chunks, L.n_kv_heads, batch);
    cudaError_t e = cudaSuccess;
    switch (L.head_dim) {
#define KVQ_D_CASE(DD)                                                                                  \
    case DD: {                                                                                          \
        const size_t smem = ((size_t)(kHQ + 2 * kTC) * (DD + 4) + kTC * kHQ + kHQ) * sizeof(float);    \
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
    k2v4_merge_kernel<<<dim3(n_q_heads, batch), 256, 0, stream>>>(p, out);
    return cudaGetLastError();
}

}  // namespace kvq
