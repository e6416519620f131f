// encode.cu -- the producers: KV8 and TQ4 row encoders and the TQ4 rotation.
//
// One warp per row.  Lane j owns elements j, j+32, j+64, ... of each scale
// block, so global loads and code stores are coalesced 128-byte runs, the warp
// reductions are exact (max) or in a fixed order (sum of squares), and the
// FWHT of a 512-block is 5 shuffle stages plus 4 in-register stages.  All
// arithmetic is IEEE f32 with explicit _rn intrinsics, so nvcc cannot fuse or
// reorder it: the codes and scales are bit-identical to the plain definition.
#include "kvq_internal.cuh"

#include <math.h>

namespace kvq {

Codebook16 tq4_codebook() {
    Codebook16 c;
    for (int k = 0; k < 16; ++k) c.lv[k] = host_bits_to_float(kTq4LevelBits[k]);
    for (int k = 0; k < 15; ++k) c.th[k] = host_bits_to_float(kTq4ThreshBits[k]);
    c.th[15] = INFINITY;
    return c;
}

Codebook4 k2_codebook() {
    Codebook4 c;
    for (int k = 0; k < 4; ++k) c.lv[k] = host_bits_to_float(kK2LevelBits[k]);
    for (int k = 0; k < 3; ++k) c.th[k] = host_bits_to_float(kK2ThreshBits[k]);
    c.th[3] = INFINITY;
    return c;
}

static uint64_t splitmix64_next(uint64_t* state) {
    uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

SignWords tq4_sign_words(const kvq_mla_layout& L) {
    SignWords s{};
    uint64_t state = L.seed;
    int w = 0;
    for (int b = 0; b < L.n_blocks; ++b) {
        s.block_word[b] = w;
        int words = (L.block_dim[b] + 63) / 64;
        for (int i = 0; i < words && w < 16; ++i) s.w[w++] = splitmix64_next(&state);
    }
    return s;
}

// ---------------------------------------------------------------------------
// KV8: s = amax / 448, code = e4m3_rn_satfinite(x / s)
// ---------------------------------------------------------------------------
struct Kv8Params {
    int32_t D, n_blocks, bd[2];
};

__global__ void __launch_bounds__(256) kv8_encode_kernel(const float* __restrict__ x, int64_t n_rows, Kv8Params p,
                                                         const int64_t* __restrict__ dst_rows,
                                                         uint8_t* __restrict__ codes, float* __restrict__ scales,
                                                         int32_t* err) {
    const int lane = threadIdx.x & 31;
    const int64_t src = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (src >= n_rows) return;
    const int64_t row = dst_rows ? dst_rows[src] : src;
    kv8_encode_row_warp(x + src * p.D, p.n_blocks, p.bd[0], p.bd[1], codes + row * p.D, scales + row * p.n_blocks,
                        lane, err);
}

cudaError_t launch_kv8_encode(const float* x, int64_t n_rows, const kvq_mla_layout& L, const int64_t* dst_rows,
                              uint8_t* codes, float* scales, int32_t* err, cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    Kv8Params p{};
    p.n_blocks = L.n_blocks;
    p.bd[0] = L.block_dim[0];
    p.bd[1] = L.n_blocks > 1 ? L.block_dim[1] : 0;
    p.D = p.bd[0] + p.bd[1];
    const int warps = 8;
    const int64_t grid = (n_rows + warps - 1) / warps;
    kv8_encode_kernel<<<(unsigned)grid, warps * 32, 0, stream>>>(x, n_rows, p, dst_rows, codes, scales, err);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// TQ4: rotate, radius, nearest codebook level, nibble pack
// ---------------------------------------------------------------------------
struct Tq4Params {
    int32_t D, n_blocks, bd[2];
    float kn[2];      // (float)(1/sqrt(n)) per block
    float sqrtn[2];   // sqrtf((float)n) per block
    SignWords signs;
    Codebook16 cb;
};

template <int N>
__device__ __forceinline__ void tq4_encode_block(const float* __restrict__ xb, int lane, const Tq4Params& p, int blk,
                                                 const float* th, uint8_t* __restrict__ out, float* scale_out,
                                                 int32_t* err) {
    constexpr int K = N >= 32 ? N / 32 : 1;
    const bool active = (N >= 32) || (lane < N);
    float x[K], v[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int i = lane + 32 * k;
        x[k] = active ? __ldg(xb + i) : 0.0f;
        v[k] = (active && sign_neg(p.signs, blk, i)) ? -x[k] : x[k];
    }
    // sum of squares: per-lane fma chain over ascending elements, then halving
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < K; ++k) ss = __fmaf_rn(x[k], x[k], ss);
    ss = warp_sum(ss);
    // a NaN or infinite input, or a radius past the f32 range: no code exists
    if (!(ss <= 3.402823466e38f) && lane == 0 && err) atomicCAS(err, 0, (int32_t)KVQ_ERR_NONFINITE);
    const float s = __fdiv_rn(__fsqrt_rn(ss), p.sqrtn[blk]);
    warp_fwht<N>(v, lane);
    const float kn = p.kn[blk];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        int c = 0;
        if (s != 0.0f) c = code16(__fdiv_rn(__fmul_rn(v[k], kn), s), th);
        const int hi = __shfl_down_sync(kFull, c, 1);
        if (active && (lane & 1) == 0) out[(lane + 32 * k) >> 1] = (uint8_t)(c | (hi << 4));
    }
    if (lane == 0) *scale_out = s;
}

template <int N>
__device__ __forceinline__ void tq4_rotate_block(float* v, int lane, const Tq4Params& p, int blk, bool inverse) {
    constexpr int K = N >= 32 ? N / 32 : 1;
    const bool active = (N >= 32) || (lane < N);
    if (!inverse) {
#pragma unroll
        for (int k = 0; k < K; ++k)
            if (active && sign_neg(p.signs, blk, lane + 32 * k)) v[k] = -v[k];
    }
    warp_fwht<N>(v, lane);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        v[k] = __fmul_rn(v[k], p.kn[blk]);
        if (inverse && active && sign_neg(p.signs, blk, lane + 32 * k)) v[k] = -v[k];
    }
}

#define KVQ_POW2_CASES(MACRO) \
    MACRO(2) MACRO(4) MACRO(8) MACRO(16) MACRO(32) MACRO(64) MACRO(128) MACRO(256) MACRO(512) MACRO(1024)

__global__ void __launch_bounds__(256) tq4_encode_kernel(const float* __restrict__ x, int64_t n_rows, Tq4Params p,
                                                         const int64_t* __restrict__ dst_rows,
                                                         uint8_t* __restrict__ packed, float* __restrict__ scales,
                                                         int32_t* err) {
    __shared__ float th[16];
    if (threadIdx.x < 16) th[threadIdx.x] = p.cb.th[threadIdx.x];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t src = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (src >= n_rows) return;
    const int64_t row = dst_rows ? dst_rows[src] : src;
    int off = 0;
    for (int b = 0; b < p.n_blocks; ++b) {
        const float* xb = x + src * p.D + off;
        uint8_t* ob = packed + row * (p.D / 2) + off / 2;
        float* so = scales + row * p.n_blocks + b;
        switch (p.bd[b]) {
#define KVQ_CASE(n) \
    case n: tq4_encode_block<n>(xb, lane, p, b, th, ob, so, err); break;
            KVQ_POW2_CASES(KVQ_CASE)
#undef KVQ_CASE
            default: break;
        }
        off += p.bd[b];
    }
}

template <typename T>
__device__ __forceinline__ float load_as_float(const T* p);
template <>
__device__ __forceinline__ float load_as_float<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load_as_float<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}

template <typename T, int N>
__device__ __forceinline__ void rotate_vec_block(const T* __restrict__ in, float* __restrict__ out, int lane,
                                                 const Tq4Params& p, int blk, bool inverse) {
    constexpr int K = N >= 32 ? N / 32 : 1;
    const bool active = (N >= 32) || (lane < N);
    float v[K];
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] = active ? load_as_float<T>(in + lane + 32 * k) : 0.0f;
    tq4_rotate_block<N>(v, lane, p, blk, inverse);
#pragma unroll
    for (int k = 0; k < K; ++k)
        if (active) out[lane + 32 * k] = v[k];
}

template <typename T>
__global__ void __launch_bounds__(256) tq4_rotate_kernel(const T* __restrict__ in, int64_t n_vecs, Tq4Params p,
                                                         int inverse, float* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t vec = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (vec >= n_vecs) return;
    int off = 0;
    for (int b = 0; b < p.n_blocks; ++b) {
        const T* ib = in + vec * p.D + off;
        float* ob = out + vec * p.D + off;
        switch (p.bd[b]) {
#define KVQ_CASE(n) \
    case n: rotate_vec_block<T, n>(ib, ob, lane, p, b, inverse != 0); break;
            KVQ_POW2_CASES(KVQ_CASE)
#undef KVQ_CASE
            default: break;
        }
        off += p.bd[b];
    }
}

static Tq4Params make_tq4_params(const kvq_mla_layout& L) {
    Tq4Params p{};
    p.n_blocks = L.n_blocks;
    p.bd[0] = L.block_dim[0];
    p.bd[1] = L.n_blocks > 1 ? L.block_dim[1] : 0;
    p.D = p.bd[0] + p.bd[1];
    for (int b = 0; b < L.n_blocks; ++b) {
        p.kn[b] = (float)(1.0 / sqrt((double)p.bd[b]));
        p.sqrtn[b] = sqrtf((float)p.bd[b]);
    }
    p.signs = tq4_sign_words(L);
    p.cb = tq4_codebook();
    return p;
}

cudaError_t launch_tq4_encode(const float* x, int64_t n_rows, const kvq_mla_layout& L, const int64_t* dst_rows,
                              uint8_t* packed, float* scales, int32_t* err, cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    const Tq4Params p = make_tq4_params(L);
    const int warps = 8;
    const int64_t grid = (n_rows + warps - 1) / warps;
    tq4_encode_kernel<<<(unsigned)grid, warps * 32, 0, stream>>>(x, n_rows, p, dst_rows, packed, scales, err);
    return cudaGetLastError();
}

cudaError_t launch_tq4_rotate(const void* in, kvq_dtype dt, int64_t n_vecs, const kvq_mla_layout& L, int inverse,
                              float* out, cudaStream_t stream) {
    if (n_vecs == 0) return cudaSuccess;
    const Tq4Params p = make_tq4_params(L);
    const int warps = 8;
    const int64_t grid = (n_vecs + warps - 1) / warps;
    if (dt == KVQ_BF16)
        tq4_rotate_kernel<__nv_bfloat16><<<(unsigned)grid, warps * 32, 0, stream>>>(
            (const __nv_bfloat16*)in, n_vecs, p, inverse, out);
    else
        tq4_rotate_kernel<float><<<(unsigned)grid, warps * 32, 0, stream>>>((const float*)in, n_vecs, p, inverse, out);
    return cudaGetLastError();
}

}  // namespace kvq
