// kvq_internal.cuh -- shared device helpers and the launchers behind the C ABI.
//
// Page titles cited as in kvq.h: [P1] KV cache quantization: fp8 (KV8) + 4-bit
// TurboQuant (KV_TQ) on CPU, CUDA, and Metal; [P2] CPU: KV cache quantization
// -- KV8 (fp8 e4m3) + KV_TQ (rotated-int4 / PolarQuant); [P3] KV cache: FP16
// sliding window + attention sinks, and an optional 2-bit K / 4-bit V cache
// scheme (--kv q2k).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "kvq.h"

namespace kvq {

constexpr unsigned kFull = 0xffffffffu;

// Opt-in launch timing (timing.cu): phase 0 before a call's partial kernel,
// 1 before its merge, 2 after it; a no-op unless kvq_timing_enable is on.
void timing_mark(cudaStream_t stream, int phase);

// Bounded waits of the tensor-core kernels: try_wait polls before a wait
// gives up, and the testing hook's stall (kvq_test_stall_waits; 0 = off).
constexpr long long kWaitLimit = 1ll << 22;
int64_t test_stall_polls();
void set_test_stall_polls(int64_t polls);

// N(0,1) Lloyd-Max codebooks as f32 bit patterns (levels ascending, then the
// decision thresholds = f64 midpoints of adjacent levels rounded to f32).
// Derived by gen_codebook.py (root finding on the centroid and midpoint
// conditions); the test suite checks them against an independent solver.
constexpr uint32_t kTq4LevelBits[16] = {
    0xc02ee2bfu, 0xc0046ac7u, 0xbfcf1c25u, 0xbfa0cc2fu, 0xbf713d39u, 0xbf28215eu, 0xbec6ae44u, 0xbe0379fdu,
    0x3e0379fdu, 0x3ec6ae44u, 0x3f28215eu, 0x3f713d39u, 0x3fa0cc2fu, 0x3fcf1c25u, 0x40046ac7u, 0x402ee2bfu};
constexpr uint32_t kTq4ThreshBits[15] = {
    0xc019a6c3u, 0xbfebf8dau, 0xbfb7f42au, 0xbf8cb566u, 0xbf4caf4bu, 0xbf05bc40u, 0xbe8435a1u, 0x00000000u,
    0x3e8435a1u, 0x3f05bc40u, 0x3f4caf4bu, 0x3f8cb566u, 0x3fb7f42au, 0x3febf8dau, 0x4019a6c3u};
constexpr uint32_t kK2LevelBits[4] = {0xbfc1555du, 0xbee7d2c9u, 0x3ee7d2c9u, 0x3fc1555du};
constexpr uint32_t kK2ThreshBits[3] = {0xbf7b4a0fu, 0x00000000u, 0x3f7b4a0fu};

inline float host_bits_to_float(uint32_t b) {
    float f;
    memcpy(&f, &b, sizeof f);
    return f;
}

struct Codebook16 {
    float lv[16];
    float th[16];   // 15 used; th[15] = +inf pads the branchless search
};
struct Codebook4 {
    float lv[4];
    float th[4];    // 3 used
};

Codebook16 tq4_codebook();
Codebook4 k2_codebook();

// Rotation signs of one TQ4 row: bit i of the D-bit mask (-1 where set).  The
// words are splitmix64 outputs from state = seed, block b starting at a fresh
// word ([P1] Commits, item 6: seeded randomized-Hadamard rotation).
struct SignWords {
    uint64_t w[16];        // up to 1024 dims
    int32_t block_word[2]; // first word of each block
};
SignWords tq4_sign_words(const kvq_mla_layout& L);

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// KV8 encoding of one row by one warp ([P1] Commits item 1): per scale block,
// s = amax / 448 (f32 division, round to nearest) and code =
// e4m3_rn_satfinite(x / s); a block with s == 0 stores s = 0 and codes 0.
// Lane 0 writes the block scales to sr[0 .. n_blocks).  The encoder kernel and
// the decode kernel that appends rows both call this, so their bytes agree.
// With CHECK, a NaN or an infinity in the row sets *err (if given and still
// 0) to KVQ_ERR_NONFINITE; the pages define no code for such values.
template <bool CHECK = true>
__device__ __forceinline__ void kv8_encode_row_warp(const float* __restrict__ xr, int n_blocks, int bd0, int bd1,
                                                    uint8_t* cr, float* sr, int lane, int32_t* err) {
    int off = 0;
    bool bad = false;
    for (int b = 0; b < n_blocks; ++b) {
        const int n = b == 0 ? bd0 : bd1;
        float amax = 0.0f;
        for (int i = lane; i < n; i += 32) {
            const float a = fabsf(__ldg(xr + off + i));
            if (CHECK) bad |= !(a <= 3.402823466e38f);
            amax = fmaxf(amax, a);
        }
        amax = warp_max(amax);
        const float s = __fdiv_rn(amax, 448.0f);
        if (lane == 0) sr[b] = s;
        for (int i = lane; i < n; i += 32) {
            uint8_t c = 0;
            if (s != 0.0f)
                c = (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(__ldg(xr + off + i), s), __NV_SATFINITE, __NV_E4M3);
            cr[off + i] = c;
        }
        off += n;
    }
    if (CHECK && __any_sync(kFull, bad) && lane == 0 && err) atomicCAS(err, 0, (int32_t)KVQ_ERR_NONFINITE);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// Number of thresholds strictly below u (a sorted list of 15, th[15] = +inf).
__device__ __forceinline__ int code16(float u, const float* th) {
    int c = (u > th[7]) ? 8 : 0;
    c += (u > th[c + 3]) ? 4 : 0;
    c += (u > th[c + 1]) ? 2 : 0;
    c += (u > th[c]) ? 1 : 0;
    return c;
}

// 4 e4m3 codes (one word, code k in byte k) -> their f16 values (exact) as two
// f16x2 words (codes 0, 1 and 2, 3): each 16-bit half of the word feeds one
// pair conversion in place, with no unpacking or repacking around it.  The
// NaN pattern S.1111.111 is never stored by the encoder; it would read back
// as NaN.
__device__ __forceinline__ void e4m3x4_to_half2x2(uint32_t in, uint32_t& w0, uint32_t& w1) {
    asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n"
        " cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}\n"
        : "=r"(w0), "=r"(w1)
        : "r"(in));
}
// The same 4 codes as f32 (exact).
__device__ __forceinline__ float4 e4m3x4_to_float4(uint32_t in) {
    uint32_t w0, w1;
    e4m3x4_to_half2x2(in, w0, w1);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w0));
    const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&w1));
    return make_float4(a.x, a.y, c.x, c.y);
}

// Warp-held radix-2 FWHT of an n-point block (n a power of two, 2..1024).
// Lane j holds elements j + 32k in v[k], k < K = max(n/32, 1); for n < 32
// only lanes j < n hold data.  Stages run in ascending h = 1, 2, 4, ..., n/2,
// each butterfly mapping (a, b) to (a+b, a-b) in f32 -- the same additions as
// the plain loop, so the result is bit-identical to it.
template <int N>
__device__ __forceinline__ void warp_fwht(float* v, int lane) {
    constexpr int K = N >= 32 ? N / 32 : 1;
#pragma unroll
    for (int h = 1; h < 32 && h < N; h <<= 1) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            float other = __shfl_xor_sync(kFull, v[k], h);
            v[k] = (lane & h) ? __fsub_rn(other, v[k]) : __fadd_rn(v[k], other);
        }
    }
#pragma unroll
    for (int hs = 1; hs < K; hs <<= 1) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            if ((k & hs) == 0) {
                float a = v[k], b = v[k + hs];
                v[k] = __fadd_rn(a, b);
                v[k + hs] = __fsub_rn(a, b);
            }
        }
    }
}

__device__ __forceinline__ bool sign_neg(const SignWords& s, int block, int i) {
    uint64_t w = s.w[s.block_word[block] + (i >> 6)];
    return (w >> (i & 63)) & 1ull;
}

// ---------------------------------------------------------------------------
// Launchers (all asynchronous on `stream`; return cudaGetLastError()).
// ---------------------------------------------------------------------------
// dst_rows (device, may be null): input row i goes to pool row dst_rows[i].
// err (device, may be null): the error word a non-finite row sets.
cudaError_t launch_kv8_encode(const float* x, int64_t n_rows, const kvq_mla_layout& L, const int64_t* dst_rows,
                              uint8_t* codes, float* scales, int32_t* err, cudaStream_t stream);
cudaError_t launch_tq4_encode(const float* x, int64_t n_rows, const kvq_mla_layout& L, const int64_t* dst_rows,
                              uint8_t* packed, float* scales, int32_t* err, cudaStream_t stream);
cudaError_t launch_tq4_rotate(const void* in, kvq_dtype dt, int64_t n_vecs, const kvq_mla_layout& L, int inverse,
                              float* out, cudaStream_t stream);
// PolarQuant (pq.cu): b = bits per angle; codes [*][pq_row_bytes], radii [*][n_blocks]
cudaError_t launch_pq_encode(int bits, const float* x, int64_t n_rows, const kvq_mla_layout& L,
                             const int64_t* dst_rows, uint8_t* codes, float* radii, int32_t* err,
                             cudaStream_t stream);
cudaError_t launch_pq_decode(int bits, const uint8_t* codes, const float* radii, int64_t n_rows,
                             const kvq_mla_layout& L, int rotated, float* out, cudaStream_t stream);
int64_t pq_row_bytes(int bits, const kvq_mla_layout& L);
bool pq_host_codebook(int bits, int level, float* centroids, float* thresholds);

// SIMT attention over the 576 = 512 + 64 latent layout.
struct AttnPlan {
    int64_t chunk;        // rows per work item
    int64_t max_items;    // grid bound
    int32_t heads_per_cta;
    int64_t wave_items;   // > 0: the chunk is balanced on the device (items per wave of CTAs)
    int32_t max_waves;    // waves of items the workspace holds
    int64_t max_rows;     // host bound on the total rows
};
AttnPlan plan_decode_simt(int32_t batch, int32_t n_heads, int64_t max_total_rows);
size_t partial_bytes(int64_t max_items, int32_t n_heads, int32_t v_dim);
// error word (bytes 0..3), device-chosen chunk (8..15), exact-path counter (16..19), padding
constexpr size_t kWsHeader = 256;

cudaError_t launch_attn_simt(kvq_format fmt, const kvq_mla_layout& L, const void* q, kvq_dtype qdt, int32_t n_seq,
                             int32_t n_heads, const uint8_t* codes, const float* scales, const int64_t* cu_seqlens,
                             int64_t prefill_past, const AttnPlan& plan, float sm_scale, float* out,
                             void* workspace, cudaStream_t stream, const int64_t* sel = nullptr,
                             int64_t pool_rows = 0);

// Tensor-core attention (tcgen05; 64 heads per CTA for KV8, 32 for TQ4).
bool tc_supported(const kvq_mla_layout& L, int32_t n_heads);
// Waves of work items a decode workspace is sized for (the device picks
// 1 .. waves from the actual lengths): 4 for KV8's 64-head CTAs, 6 for the
// 32-head CTAs of TQ4 and PolarQuant (on the 32-sequence ragged decode KV8
// took 1.003 ms at 4 waves and 1.007 ms at 6, TQ4 2.442 ms and 2.399 ms).
constexpr int decode_waves(kvq_format fmt) { return fmt == KVQ_KV8 ? 4 : 6; }
AttnPlan plan_decode_tc(kvq_format fmt, int32_t batch, int32_t n_heads, int64_t max_total_rows, int waves);
// kv_attn_workspace_size / kv_attn_decode with a given wave budget (the
// no-allocation entry takes fewer waves to fit its fixed scratch).
size_t attn_workspace_size_waves(kvq_format fmt, const kvq_mla_layout* layout, int32_t batch, int32_t n_heads,
                                 int64_t max_total_rows, kvq_path path, int waves);
kvq_status attn_decode_waves(kvq_format fmt, const kvq_mla_layout* layout, const void* q, kvq_dtype q_dtype,
                             int32_t batch, int32_t n_heads, const uint8_t* codes, const float* scales,
                             const int64_t* cu_seqlens, int64_t max_total_rows, float sm_scale, float* out,
                             void* workspace, size_t workspace_bytes, kvq_path path, void* stream, int waves);
// KV8 decode with bf16 queries on the tensor cores, the step's new rows
// encoded in the same launch (row x_new[b] -> pool row dst_rows[b]).
cudaError_t launch_attn_tc_kv8_append(const kvq_mla_layout& L, const float* x_new, const int64_t* dst_rows,
                                      const void* q, int32_t n_seq, int32_t n_heads, uint8_t* codes, float* scales,
                                      const int64_t* cu_seqlens, const AttnPlan& plan, float sm_scale, float* out,
                                      void* workspace, cudaStream_t stream);
cudaError_t launch_attn_tc(kvq_format fmt, const kvq_mla_layout& L, const void* q, kvq_dtype qdt, int32_t n_seq,
                           int32_t n_heads, const uint8_t* codes, const float* scales, const int64_t* cu_seqlens,
                           int64_t prefill_past, const AttnPlan& plan, float sm_scale, float* out, void* workspace,
                           cudaStream_t stream, const int64_t* sel = nullptr, int64_t pool_rows = 0);

// K2/V4
cudaError_t launch_k2v4_encode(const kvq_k2v4_layout& L, const float* k, const float* v, int32_t batch,
                               int64_t n_cells, int64_t cap, uint8_t* k_codes, uint16_t* k_scales,
                               uint8_t* v_blocks, uint16_t* k_win, uint16_t* v_win, int32_t* err,
                               cudaStream_t stream);
// n_new cells per sequence appended at cells n_past .. n_past + n_new - 1
// (k_new, v_new [batch][Hkv][n_new][D]), with the partial-group scale rule.
cudaError_t launch_k2v4_append(const kvq_k2v4_layout& L, const float* k_new, const float* v_new, int32_t batch,
                               int64_t n_past, int64_t n_new, int64_t cap, uint8_t* k_codes, uint16_t* k_scales,
                               uint8_t* v_blocks, uint16_t* k_win, uint16_t* v_win, int32_t* err,
                               cudaStream_t stream);
struct K2V4Plan {
    int64_t chunk;
    int32_t n_chunks;
    bool tensor;   // tensor-core kernel (head_dim 128 or 256), else fp32
};
bool k2v4_tc_supported(const kvq_k2v4_layout& L);
K2V4Plan plan_k2v4(const kvq_k2v4_layout& L, int32_t batch, int32_t n_q_heads, int64_t n_cells, bool tensor);
size_t k2v4_partial_bytes(const kvq_k2v4_layout& L, int32_t batch, int32_t n_q_heads, const K2V4Plan& p);
cudaError_t launch_k2v4_decode(const kvq_k2v4_layout& L, const float* q, int32_t batch, int32_t n_q_heads,
                               int64_t n_cells, int64_t cap, const uint8_t* k_codes, const uint16_t* k_scales,
                               const uint8_t* v_blocks, const uint16_t* k_win, const uint16_t* v_win,
                               float sm_scale, float* out, void* workspace, const K2V4Plan& plan,
                               cudaStream_t stream);

}  // namespace kvq
