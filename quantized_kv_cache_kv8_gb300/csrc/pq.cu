// pq.cu -- PolarQuant (codec 0 of the TQ tier): the row encoder and the
// dequantizing decoder.
//
// The codec follows the published method (Han et al., "PolarQuant: Quantizing
// KV Caches with Polar Transformation", 2025), named by the KV cache
// quantization pages ([P1] Summary: "PolarQuant ... variable 2-6 bit"; [P1]
// Commits item 6: "randomized-Hadamard rotation + recursive polar"): the block
// is rotated as for TQ4, turned into a tree of (radius, angle) pairs down to
// one radius, and every angle is coded with b bits by its level's codebook
// (level 1 uniform on the circle, level l >= 2 the Lloyd-Max quantizer of the
// density sin(2 psi)^(2^(l-1) - 1)).
//
// One warp per row.  The rotation is the TQ4 encoder's (lane j holds elements
// j, j+32, ...; warp FWHT); the rotated block goes to shared memory, where the
// tree is built level by level with __syncwarp between levels.  Decisions
// compare f32 products with the tables' f32 cos and sin (psi > t when
// hi * cos t > lo * sin t), so no angle is computed and the codes are
// bit-identical to the plain definition.
#include "pq_common.cuh"

#include <math.h>

namespace kvq {

namespace {

#include "pq_codebook.inc"

__device__ const uint32_t g_pq_cent[kPqCentWords] = {KVQ_PQ_CENT_WORDS};
__device__ const uint32_t g_pq_thresh[kPqThreshWords] = {KVQ_PQ_THRESH_WORDS};
constexpr uint32_t kPqCentHost[kPqCentWords] = {KVQ_PQ_CENT_WORDS};
constexpr uint32_t kPqThreshHost[kPqThreshWords] = {KVQ_PQ_THRESH_WORDS};

constexpr int kWarps = 4;

struct PqParams {
    int32_t D, n_blocks, bd[2], bits, row_bytes, boff[2], maxn;
    float kn[2];   // (float)(1/sqrt(n)) per block
    SignWords signs;
};

// number of thresholds t (ascending) below the angle of (lo, hi), lo, hi >= 0:
// the predicate hi*cos t > lo*sin t holds for a prefix of the thresholds (the
// f32 cos fall and the sin rise with t, and rounding keeps the order), so a
// binary search counts it
__device__ __forceinline__ int pq_count(float lo, float hi, const float2* t, int n) {
    int a = 0, z = n;
    while (a < z) {
        const int mid = (a + z) >> 1;
        const float2 cs = t[mid];
        if (__fmul_rn(hi, cs.x) > __fmul_rn(lo, cs.y)) a = mid + 1;
        else z = mid;
    }
    return a;
}

// level-1 code of the pair (a, c): the quadrant by exact sign swaps, then the
// cell inside it; a zero pair is code 0
__device__ __forceinline__ int pq_code1(float a, float c, int b, const float2* t, int n_th) {
    int q;
    float u, w;
    if (a > 0.0f && c >= 0.0f) { q = 0; u = a; w = c; }
    else if (a <= 0.0f && c > 0.0f) { q = 1; u = c; w = -a; }
    else if (a < 0.0f && c <= 0.0f) { q = 2; u = -a; w = -c; }
    else if (a >= 0.0f && c < 0.0f) { q = 3; u = -c; w = a; }
    else return 0;
    return (q << (b - 2)) + pq_count(u, w, t, n_th);
}

__device__ __forceinline__ float pq_radius(float lo, float hi) {
    return __fsqrt_rn(__fadd_rn(__fmul_rn(lo, lo), __fmul_rn(hi, hi)));
}

template <int N>
__device__ __forceinline__ void pq_encode_block(const float* __restrict__ xb, int lane, const PqParams& p, int blk,
                                                const float2* th, float* y, uint8_t* cd, uint8_t* __restrict__ out,
                                                float* radius_out, int32_t* err) {
    constexpr int K = N >= 32 ? N / 32 : 1;
    constexpr int L = N >= 1024 ? 10 : N >= 512 ? 9 : N >= 256 ? 8 : N >= 128 ? 7 : N >= 64 ? 6 : N >= 32 ? 5
                    : N >= 16 ? 4 : N >= 8 ? 3 : N >= 4 ? 2 : 1;
    constexpr int R = (N / 2 + 31) / 32;   // pairs of level 1 per lane
    const bool active = (N >= 32) || (lane < N);
    float v[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int i = lane + 32 * k;
        const float x = active ? __ldg(xb + i) : 0.0f;
        v[k] = (active && sign_neg(p.signs, blk, i)) ? -x : x;
    }
    warp_fwht<N>(v, lane);
#pragma unroll
    for (int k = 0; k < K; ++k)
        if (active) y[lane + 32 * k] = __fmul_rn(v[k], p.kn[blk]);
    __syncwarp();
    const int b = p.bits, nth = (1 << b) - 1;
    float rr[R];
    // level 1: pairs of rotated values
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int j = lane + 32 * i;
        if (j < N / 2) {
            const float a = y[2 * j], c = y[2 * j + 1];
            cd[j] = (uint8_t)pq_code1(a, c, b, th + 9 * nth, (1 << (b - 2)) - 1);
            rr[i] = pq_radius(a, c);
        }
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < R; ++i)
        if (lane + 32 * i < N / 2) y[lane + 32 * i] = rr[i];
    __syncwarp();
    // levels 2 .. L: pairs of radii
    int first = N / 2;
#pragma unroll
    for (int l = 2; l <= L; ++l) {
        const int m = N >> l;
        const float2* tl = th + (l - 2) * nth;
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int j = lane + 32 * i;
            if (j < m) {
                const float lo = y[2 * j], hi = y[2 * j + 1];
                cd[first + j] = (uint8_t)pq_count(lo, hi, tl, nth);
                rr[i] = pq_radius(lo, hi);
            }
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < R; ++i)
            if (lane + 32 * i < m) y[lane + 32 * i] = rr[i];
        __syncwarp();
        first += m;
    }
    const float r = y[0];
    if (lane == 0) {
        *radius_out = r;
        if (!(r <= 3.402823466e38f) && err) atomicCAS(err, 0, (int32_t)KVQ_ERR_NONFINITE);
    }
    // pack the N - 1 codes, b bits each, least significant bit first
    const int nb = (N * b + 7) / 8;
    for (int k = lane; k < nb; k += 32) {
        unsigned w = 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int pos = 8 * k + t, a = pos / b;
            if (a < N - 1) w |= ((unsigned)(cd[a] >> (pos - a * b)) & 1u) << t;
        }
        out[k] = (uint8_t)w;
    }
    __syncwarp();
}

#define KVQ_POW2_CASES(MACRO) \
    MACRO(2) MACRO(4) MACRO(8) MACRO(16) MACRO(32) MACRO(64) MACRO(128) MACRO(256) MACRO(512) MACRO(1024)

// thresholds of width b in shared memory: [level 2..10][2^b - 1], then level 1's
__global__ void __launch_bounds__(kWarps * 32) pq_encode_kernel(const float* __restrict__ x, int64_t n_rows,
                                                                PqParams p, const float2* __restrict__ th_g,
                                                                const int64_t* __restrict__ dst_rows,
                                                                uint8_t* __restrict__ codes,
                                                                float* __restrict__ radii, int32_t* err) {
    extern __shared__ float4 smem4[];
    float2* th = reinterpret_cast<float2*>(smem4);
    const int nth_all = 9 * ((1 << p.bits) - 1) + (1 << (p.bits - 2)) - 1;
    float* ybase = reinterpret_cast<float*>(th + 9 * 63 + 15 + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* y = ybase + warp * p.maxn;
    uint8_t* cd = reinterpret_cast<uint8_t*>(ybase + kWarps * p.maxn) + warp * p.maxn;
    for (int i = threadIdx.x; i < nth_all; i += blockDim.x) th[i] = th_g[i];
    __syncthreads();
    const int64_t src = (int64_t)blockIdx.x * kWarps + warp;
    if (src >= n_rows) return;
    const int64_t row = dst_rows ? dst_rows[src] : src;
    int off = 0;
    for (int b = 0; b < p.n_blocks; ++b) {
        const float* xb = x + src * p.D + off;
        uint8_t* ob = codes + row * p.row_bytes + p.boff[b];
        float* ro = radii + row * p.n_blocks + b;
        switch (p.bd[b]) {
#define KVQ_CASE(n) \
    case n: pq_encode_block<n>(xb, lane, p, b, th, y, cd, ob, ro, err); break;
            KVQ_POW2_CASES(KVQ_CASE)
#undef KVQ_CASE
            default: break;
        }
        off += p.bd[b];
    }
}

template <int N>
__device__ __forceinline__ void pq_unrotate_store(const float* y, int lane, const PqParams& p, int blk,
                                                  float* __restrict__ out) {
    constexpr int K = N >= 32 ? N / 32 : 1;
    const bool active = (N >= 32) || (lane < N);
    float v[K];
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] = active ? y[lane + 32 * k] : 0.0f;
    warp_fwht<N>(v, lane);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int i = lane + 32 * k;
        const float t = __fmul_rn(v[k], p.kn[blk]);
        if (active) out[i] = sign_neg(p.signs, blk, i) ? -t : t;
    }
}

// centroids of width b in shared memory: [level 1..10][2^b]
__global__ void __launch_bounds__(kWarps * 32) pq_decode_kernel(const uint8_t* __restrict__ codes,
                                                                const float* __restrict__ radii, int64_t n_rows,
                                                                PqParams p, const float2* __restrict__ cent_g,
                                                                int rotated, float* __restrict__ out) {
    extern __shared__ float4 smem4[];
    float2* cent = reinterpret_cast<float2*>(smem4);
    float* ybase = reinterpret_cast<float*>(cent + (kPqMaxLevel << 6));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* y = ybase + warp * p.maxn;
    for (int i = threadIdx.x; i < (kPqMaxLevel << p.bits); i += blockDim.x) cent[i] = cent_g[i];
    __syncthreads();
    const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
    if (row >= n_rows) return;
    int off = 0;
    for (int b = 0; b < p.n_blocks; ++b) {
        const int n = p.bd[b];
        const int L = 31 - __clz(n);
        pq_expand_block(codes + row * p.row_bytes + p.boff[b], n, L, p.bits, radii[row * p.n_blocks + b], cent, y,
                        lane);
        float* ob = out + row * p.D + off;
        if (rotated) {
            for (int i = lane; i < n; i += 32) ob[i] = y[i];
        } else {
            switch (n) {
#define KVQ_CASE(nn) \
    case nn: pq_unrotate_store<nn>(y, lane, p, b, ob); break;
                KVQ_POW2_CASES(KVQ_CASE)
#undef KVQ_CASE
                default: break;
            }
        }
        __syncwarp();
        off += n;
    }
}

PqParams make_pq_params(int bits, const kvq_mla_layout& L) {
    PqParams p{};
    p.bits = bits;
    p.n_blocks = L.n_blocks;
    p.bd[0] = L.block_dim[0];
    p.bd[1] = L.n_blocks > 1 ? L.block_dim[1] : 0;
    p.D = p.bd[0] + p.bd[1];
    p.boff[0] = 0;
    p.boff[1] = (int32_t)pq_block_bytes(p.bd[0], bits);
    p.row_bytes = (int32_t)(p.boff[1] + (L.n_blocks > 1 ? pq_block_bytes(p.bd[1], bits) : 0));
    p.maxn = p.bd[0] > p.bd[1] ? p.bd[0] : p.bd[1];
    for (int b = 0; b < L.n_blocks; ++b) p.kn[b] = (float)(1.0 / sqrt((double)p.bd[b]));
    p.signs = tq4_sign_words(L);
    return p;
}

const float2* symbol_base(const void* sym) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, sym) != cudaSuccess) return nullptr;
    return static_cast<const float2*>(ptr);
}

}  // namespace

const float2* pq_device_centroids(int bits) {
    const float2* base = symbol_base(g_pq_cent);
    return base ? base + kPqCentOff[bits] : nullptr;
}

const float2* pq_device_thresholds(int bits) {
    const float2* base = symbol_base(g_pq_thresh);
    return base ? base + kPqThreshOff[bits] : nullptr;
}

bool pq_host_codebook(int bits, int level, float* centroids, float* thresholds) {
    if (bits < 2 || bits > 6 || level < 1 || level > kPqMaxLevel) return false;
    const int n = 1 << bits;
    const uint32_t* c = kPqCentHost + 2 * (kPqCentOff[bits] + (level - 1) * n);
    for (int i = 0; i < 2 * n; ++i) centroids[i] = host_bits_to_float(c[i]);
    const int nt = level == 1 ? n / 4 - 1 : n - 1;
    const uint32_t* t = kPqThreshHost + 2 * (kPqThreshOff[bits] + (level == 1 ? 9 * (n - 1) : (level - 2) * (n - 1)));
    for (int i = 0; i < 2 * nt; ++i) thresholds[i] = host_bits_to_float(t[i]);
    return true;
}

int64_t pq_row_bytes(int bits, const kvq_mla_layout& L) {
    int64_t s = 0;
    for (int b = 0; b < L.n_blocks; ++b) s += pq_block_bytes(L.block_dim[b], bits);
    return s;
}

cudaError_t launch_pq_encode(int bits, const float* x, int64_t n_rows, const kvq_mla_layout& L,
                             const int64_t* dst_rows, uint8_t* codes, float* radii, int32_t* err,
                             cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    const PqParams p = make_pq_params(bits, L);
    const float2* th = pq_device_thresholds(bits);
    if (!th) return cudaErrorInvalidSymbol;
    const size_t smem = sizeof(float2) * (9 * 63 + 16) + (size_t)kWarps * p.maxn * (sizeof(float) + 1);
    const int64_t grid = (n_rows + kWarps - 1) / kWarps;
    pq_encode_kernel<<<(unsigned)grid, kWarps * 32, smem, stream>>>(x, n_rows, p, th, dst_rows, codes, radii, err);
    return cudaGetLastError();
}

cudaError_t launch_pq_decode(int bits, const uint8_t* codes, const float* radii, int64_t n_rows,
                             const kvq_mla_layout& L, int rotated, float* out, cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    const PqParams p = make_pq_params(bits, L);
    const float2* cent = pq_device_centroids(bits);
    if (!cent) return cudaErrorInvalidSymbol;
    const size_t smem = sizeof(float2) * (kPqMaxLevel << 6) + (size_t)kWarps * p.maxn * sizeof(float);
    const int64_t grid = (n_rows + kWarps - 1) / kWarps;
    pq_decode_kernel<<<(unsigned)grid, kWarps * 32, smem, stream>>>(codes, radii, n_rows, p, cent, rotated, out);
    return cudaGetLastError();
}

}  // namespace kvq
