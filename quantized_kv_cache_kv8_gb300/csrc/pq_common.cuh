// pq_common.cuh -- PolarQuant (codec 0 of the TQ tier) pieces shared by its
// encoder and dequantizer (pq.cu) and by the fp32 attention consumer.
//
// A block of n = 2^L rotated values is a tree: level 1 pairs consecutive
// values into (radius, angle), level l pairs the level-(l-1) radii, and one
// radius is left.  The n - 1 angle codes are stored level by level (level 1
// first, in pair order), b bits each, least significant bit first.
#pragma once

#include "kvq_internal.cuh"

namespace kvq {

// template id of the PolarQuant consumer in the attention kernels (the width
// is a runtime value there)
constexpr int kFmtPolar = 3;
constexpr int kPqMaxLevel = 10;

inline bool is_pq(kvq_format f) { return f >= KVQ_PQ2 && f <= KVQ_PQ6; }
inline int pq_bits_of(kvq_format f) { return (int)f - 10; }
inline int64_t pq_block_bytes(int n, int bits) { return ((int64_t)n * bits + 7) / 8; }

// Device tables of width b (pq.cu): centroids [level 1..10][2^b] and
// thresholds [level 2..10][2^b - 1] then level 1's in-quadrant [2^(b-2) - 1],
// each as (cos, sin).  Host functions returning device pointers of the
// current device.
const float2* pq_device_centroids(int bits);
const float2* pq_device_thresholds(int bits);

// Angle code at stream bit `pos`: b bits, least significant first; the second
// byte is read only when the code crosses into it, so nothing past the
// stream's last byte is touched.
__device__ __forceinline__ unsigned pq_get_bits(const uint8_t* __restrict__ s, int64_t pos, int b) {
    const uint8_t* q = s + (pos >> 3);
    const int sh = (int)(pos & 7);
    unsigned v = (unsigned)__ldg(q) >> sh;
    if (sh + b > 8) v |= (unsigned)__ldg(q + 1) << (8 - sh);
    return v & ((1u << b) - 1u);
}

// Rebuilds one block's leaves into y[0 .. n) from the top radius r0, in
// place: the radius of node j of level l sits at y[j << l] (its first leaf),
// so a node writes its two children at y[j << l] and y[(j << l) + 2^(l-1)] and
// no two nodes touch the same word.  cent: centroids of width b, levels 1..L
// ([level - 1][2^b] (cos, sin)).  One warp; f32 products rounded once each.
__device__ __forceinline__ void pq_expand_block(const uint8_t* __restrict__ stream, int n, int L, int b, float r0,
                                                const float2* cent, float* y, int lane) {
    if (lane == 0) y[0] = r0;
    __syncwarp();
    for (int l = L; l >= 1; --l) {
        const int m = n >> l;
        const int first = n - (n >> (l - 1));   // stream index of the level's first angle
        const float2* c = cent + ((l - 1) << b);
        for (int j = lane; j < m; j += 32) {
            const int at = j << l;
            const float r = y[at];
            const float2 cs = c[pq_get_bits(stream, (int64_t)(first + j) * b, b)];
            y[at] = __fmul_rn(r, cs.x);
            y[at + (1 << (l - 1))] = __fmul_rn(r, cs.y);
        }
        __syncwarp();
    }
}

}  // namespace kvq
