// attn_tc_tq4.cu -- tensor-core attention over TQ4 rows with every chunk of a
// tile decoded once.
//
// The structure of the KV8 kernel (attn_tc_kv8.cu): one chunk of rows per CTA,
// 128-row tiles whose 9 f16 chunks stay resident for both products, decode in
// three groups overlapping the previous tile's context MMAs, a single MMA
// issuer, a lagged running max.  What differs for TQ4 ([P1] "Ready for review"
// comment, finding 2: rotate the query once per head, dot it with the
// codebook levels, unrotate the context once):
//   - the rotated query is not exact in f16, so each query chunk holds the f16
//     value and the f16 residual of every head; to leave room for the retained
//     chunks a CTA serves 32 heads: the score runs with N = 64 (32 values + 32
//     residuals), the context with N = 32;
//   - codes are nibbles: byte permutes over the 16 f16 levels (store32) turn
//     them into f16 operands, the levels scaled by kTq4Gamma (within 9.3e-5
//     of f16; divided out of scores and context);
//   - P is stored K-major (heads on rows) so that N = 32 needs no padding.
// The context accumulates in the rotated domain; the merge unrotates it.
// The same kernel serves PolarQuant rows at 4 bits (PQ = true; codec 0 of the
// TQ tier, 288 code bytes per row like TQ4): each row's tree is rebuilt from
// a unit top radius, the block radius riding the row scale as TQ4's does; two
// threads rebuild a row, one per half of its latent and rope blocks, with the
// level centroids' (cos, sin) in shared memory and the leaves written as f16.
// Softmax weights as in the KV8 kernel: the row sums take p = 2^(z - m) (m a
// lagged running maximum of the scores), the context the f16 weight
// w = p s_L E with E = 2^(m - R - 3) per head, R the largest z + log2 s_L of
// the tiles that set the references, so that the context weights are relative
// to the largest p * s_L of the chunk (which weighs 2^-3); the exact path runs
// when a score passes m by 2^14 or a latent scale passes 3.5 / max_h E; the
// partial state is (m, sum p, O^T / E).
#include "tc_common.cuh"

#include <math.h>

namespace kvq {
namespace {
using namespace tc;

constexpr int kRows = 128;      // rows per tile
constexpr int kHC = 32;         // heads per CTA
constexpr int kWorkers = 256;
// warpgroup 2 (the MMA-issuing warp and three idle warps) gives its registers
// to the eight worker warps after the prologue (setmaxnreg)
constexpr int kThreads = kWorkers + 128;
constexpr int kRegsLaunch = 168, kRegsWorker = 232, kRegsMma = 40;
static_assert(kWorkers * kRegsWorker + 128 * kRegsMma <= kThreads * kRegsLaunch, "register split");
constexpr int kChunks = 9;      // 64-dim chunks: 8 latent + 1 rope
constexpr int kRope = 8;
constexpr int kRowBytes = kMlaD / 2;                // 288 code bytes per row
constexpr uint32_t kSlotBytes = kRows * 128;       // 128 rows x 64 f16
constexpr uint32_t kQChunkBytes = 2 * kHC * 128;   // 32 heads (f16) + 32 residual rows
constexpr uint32_t kPChunkBytes = kHC * 128;       // P: 32 head rows x 64 cells
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffSlot = kOffQ + kChunks * kQChunkBytes;
constexpr uint32_t kOffLevels = kOffSlot + kChunks * kSlotBytes;   // LevelBytes: 32 bytes
constexpr uint32_t kOffM = kOffLevels + 32;             // m: running max of z per head
constexpr uint32_t kOffR = kOffM + kHC * 4;              // R: reference of z + log2 s_L
constexpr uint32_t kOffE = kOffR + kHC * 4;              // E = 2^(m - R - kHeadroom)
constexpr uint32_t kOffF = kOffE + kHC * 4;              // 1 / E
constexpr uint32_t kOffAlpha = kOffF + kHC * 4;          // O^T rescale
constexpr uint32_t kOffAlphaM = kOffAlpha + kHC * 4;     // row-sum rescale 2^(m_old - m_new)
constexpr uint32_t kOffEmax = kOffAlphaM + kHC * 4;      // max E over the heads
constexpr uint32_t kOffRed = kOffEmax + 16;          // 2 x 4 quadrants x 32 heads
constexpr uint32_t kOffBar = kOffRed + 2 * 4 * kHC * 4;
constexpr uint32_t kOffMisc = kOffBar + 16 * 8;
constexpr uint32_t kOffCent = kOffMisc + 32;             // PolarQuant: [level 1..9][16] (cos, sin)
constexpr uint32_t kSmemUsed = kOffCent + 9 * 16 * 8;
static_assert(kOffSlot % 1024 == 0, "swizzled operands need 1024-byte alignment");
static_assert(kSmemUsed <= 232448, "shared memory budget");

// TMEM: O^T 4 blocks x 32 columns, S_L^T and S_R^T 64 columns each (values, residuals)
constexpr uint32_t kColO = 0, kColSL = 128, kColSR = 192, kTmemCols = 256;

// (the same barriers as the KV8 kernel, the last one for the testing hook's stall)
enum { kBarFull0 = 0, kBarFree0 = 3, kBarScore = 7, kBarP = 8, kBarDone = 9, kBarNever = 10, kNumBars = 11 };

constexpr float kLagLog2 = 14.0f;   // p <= 2^14, w <= 3.5 * 2^14 without the exact path
constexpr float kHeadroom = 3.0f;   // the largest p * s_L of a reference tile weighs 2^-3
constexpr float kLogEmax = 120.0f;  // cap of log2 E (E and 1 / E finite in f32)
// TQ4 levels in f16: the 16 Lloyd-Max levels times kTq4Gamma round to f16 with
// a relative error of at most 9.3e-5 (2^-13.4), against 3.2e-4 unscaled; the
// value comes from a search over scales in [1, 2) (csrc/gen_codebook.py
// --level-scale).  Scores and context are divided by it in f32.
constexpr float kTq4Gamma = 1.3338516f;
constexpr float kTq4InvGamma = 1.0f / 1.3338516f;
constexpr uint32_t kIdescScore = idesc_f16(128, 2 * kHC, false, false);
constexpr uint32_t kIdescCtx = idesc_f16(128, kHC, true, false);

// A worker's raw share of a tile.  Groups A and B (code bytes 128 g .. + 127):
// 4 pieces, piece i at row 4 (warp + 8 i) + (lane / 2) % 4, bytes
// 32 (lane / 8) + 16 (lane % 2) of the group -- chunk 4 g + lane / 8, dims
// 32 (lane % 2) of it.  A 16-byte shared-memory store is served 8 lanes at a
// time: lanes 8p .. 8p + 7 write 4 rows x 2 halves of one chunk, and 4
// consecutive rows' 128-byte swizzle phases map a half's units {i, 4 + i} onto
// 8 distinct 16-byte units (one row across four chunks hit 2 units 4 ways).
// Group C (the rope chunk, bytes 256..287): 1 piece at row 16 warp + lane / 2,
// bytes 16 (lane % 2).
struct RawGroup {
    uint4 v[4];
};

__device__ __forceinline__ void load_group(RawGroup& r, const uint8_t* __restrict__ codes, int64_t t0, int nt, int g,
                                           int warp, int lane) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = 4 * (warp + 8 * i) + ((lane >> 1) & 3);
        r.v[i] = row < nt ? __ldg(reinterpret_cast<const uint4*>(codes + (t0 + row) * kRowBytes + 128 * g +
                                                                 32 * (lane >> 3) + 16 * (lane & 1)))
                          : make_uint4(0u, 0u, 0u, 0u);
    }
}
__device__ __forceinline__ uint4 load_rope(const uint8_t* __restrict__ codes, int64_t t0, int nt, int warp, int lane) {
    const int row = 16 * warp + (lane >> 1);
    return row < nt ? __ldg(reinterpret_cast<const uint4*>(codes + (t0 + row) * kRowBytes + 256 + 16 * (lane & 1)))
                    : make_uint4(0u, 0u, 0u, 0u);
}

// The 16 f16 levels (x kTq4Gamma) as byte planes, four levels per word:
// lo[k] holds the low bytes of levels 4k .. 4k+3, hi[k] their high bytes.
struct LevelBytes {
    uint32_t lo[4], hi[4];
};


// PolarQuant, 4 bits: a worker's raw share of a tile is half of one row --
// row 32 (warp / 2) + lane, half h = warp % 2 -- as the byte ranges holding the
// angles of that half: latent level 1 (bytes 64 h .. + 63), level 2
// (128 + 32 h .. + 31), level 3 (192 + 16 h .. + 15), levels 4-9 of both halves
// (bytes 224 .. 255) and the whole rope block (256 .. 287).  Angle a of a
// block is nibble a of its stream (level 1 first); level l starts at angle
// n - n / 2^(l-1).
struct RawPQ {
    uint4 l1[4], l2[2], l3, tail[2], rope[2];
};

__device__ __forceinline__ void load_pq(RawPQ& r, const uint8_t* __restrict__ codes, int64_t t0, int nt, int warp,
                                        int lane) {
    const int row = 32 * (warp >> 1) + lane, h = warp & 1;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const uint4* base = reinterpret_cast<const uint4*>(codes + (t0 + row) * kRowBytes);
    const bool ok = row < nt;
#pragma unroll
    for (int i = 0; i < 4; ++i) r.l1[i] = ok ? __ldg(base + 4 * h + i) : z;
#pragma unroll
    for (int i = 0; i < 2; ++i) r.l2[i] = ok ? __ldg(base + 8 + 2 * h + i) : z;
    r.l3 = ok ? __ldg(base + 12 + h) : z;
#pragma unroll
    for (int i = 0; i < 2; ++i) r.tail[i] = ok ? __ldg(base + 14 + i) : z;
#pragma unroll
    for (int i = 0; i < 2; ++i) r.rope[i] = ok ? __ldg(base + 16 + i) : z;
}

template <int N>
__device__ __forceinline__ void words_of(const uint4 (&v)[N], uint32_t (&w)[4 * N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
        w[4 * i] = v[i].x;
        w[4 * i + 1] = v[i].y;
        w[4 * i + 2] = v[i].z;
        w[4 * i + 3] = v[i].w;
    }
}

// nibble i of a word array (i a compile-time index after unrolling)
template <int W>
__device__ __forceinline__ uint32_t nib(const uint32_t (&w)[W], int i) {
    return (w[i >> 3] >> (4 * (i & 7))) & 15u;
}

// children of node radius r under the angle with code c at level l: (r cos, r sin)
__device__ __forceinline__ void split(const float2* cent, int level, uint32_t c, float r, float& a, float& b) {
    const float2 cs = cent[(level - 1) * 16 + c];
    a = __fmul_rn(r, cs.x);
    b = __fmul_rn(r, cs.y);
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    const __half2 h2 = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h2);
}

// Latent half h of a row: its 256 leaves (unit top radius) as f16 into
// chunks 4 h .. 4 h + 3 of swizzled row `row`.  h is a template argument so
// that every nibble index is a constant (the code words stay in registers).
template <int h>
__device__ __forceinline__ void pq_latent_half(const RawPQ& r, int row, const float2* cent, unsigned char* sSlot) {
    uint32_t T[8], L3[4], L2[8], L1[16];
    words_of(r.tail, T);
    L3[0] = r.l3.x; L3[1] = r.l3.y; L3[2] = r.l3.z; L3[3] = r.l3.w;
    words_of(r.l2, L2);
    words_of(r.l1, L1);
    // levels 9 .. 5: angles 510, 508 + h, 504 + 2h + j, 496 + 4h + j, 480 + 8h + j
    // (tail nibbles 62, 60 + h, 56 + 2h + j, 48 + 4h + j, 32 + 8h + j)
    float a9, b9;
    split(cent, 9, nib(T, 62), 1.0f, a9, b9);
    const float r8 = h ? b9 : a9;
    float r7[2], r6[4], r5[8], r4[16];
    split(cent, 8, nib(T, 60 + h), r8, r7[0], r7[1]);
#pragma unroll
    for (int j = 0; j < 2; ++j) split(cent, 7, nib(T, 56 + 2 * h + j), r7[j], r6[2 * j], r6[2 * j + 1]);
#pragma unroll
    for (int j = 0; j < 4; ++j) split(cent, 6, nib(T, 48 + 4 * h + j), r6[j], r5[2 * j], r5[2 * j + 1]);
#pragma unroll
    for (int j = 0; j < 8; ++j) split(cent, 5, nib(T, 32 + 8 * h + j), r5[j], r4[2 * j], r4[2 * j + 1]);
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        // the 16-leaf subtree k: level 4 (tail nibble 16 h + k), level 3 (l3
        // nibbles 2k, 2k + 1), level 2 (l2 nibbles 4k ..), level 1 (l1 nibbles 8k ..)
        float r3[2], r2[4], r1[8], x[16];
        split(cent, 4, nib(T, 16 * h + k), r4[k], r3[0], r3[1]);
#pragma unroll
        for (int i = 0; i < 2; ++i) split(cent, 3, nib(L3, 2 * k + i), r3[i], r2[2 * i], r2[2 * i + 1]);
#pragma unroll
        for (int i = 0; i < 4; ++i) split(cent, 2, nib(L2, 4 * k + i), r2[i], r1[2 * i], r1[2 * i + 1]);
#pragma unroll
        for (int i = 0; i < 8; ++i) split(cent, 1, nib(L1, 8 * k + i), r1[i], x[2 * i], x[2 * i + 1]);
        unsigned char* slot = sSlot + (4 * h + (k >> 2)) * kSlotBytes;
#pragma unroll
        for (int q = 0; q < 2; ++q)
            *reinterpret_cast<uint4*>(slot + sw128(row, 32 * (k & 3) + 16 * q)) =
                make_uint4(pack_h2(x[8 * q], x[8 * q + 1]), pack_h2(x[8 * q + 2], x[8 * q + 3]),
                           pack_h2(x[8 * q + 4], x[8 * q + 5]), pack_h2(x[8 * q + 6], x[8 * q + 7]));
    }
}

// Rope half h of a row (64 dims, 6 levels): leaves 32 h .. 32 h + 31 into the
// rope chunk's slot, bytes 64 h .. 64 h + 63 of swizzled row `row`.
template <int h>
__device__ __forceinline__ void pq_rope_half(const RawPQ& r, int row, const float2* cent, unsigned char* sRopeSlot) {
    uint32_t R[8];
    words_of(r.rope, R);
    // levels 6 .. 1 of the rope block start at angles 62, 60, 56, 48, 32, 0
    float a6, b6;
    split(cent, 6, nib(R, 62), 1.0f, a6, b6);
    const float r5 = h ? b6 : a6;
    float r4[2], r3[4], r2[8], r1[16], x[32];
    split(cent, 5, nib(R, 60 + h), r5, r4[0], r4[1]);
#pragma unroll
    for (int j = 0; j < 2; ++j) split(cent, 4, nib(R, 56 + 2 * h + j), r4[j], r3[2 * j], r3[2 * j + 1]);
#pragma unroll
    for (int j = 0; j < 4; ++j) split(cent, 3, nib(R, 48 + 4 * h + j), r3[j], r2[2 * j], r2[2 * j + 1]);
#pragma unroll
    for (int j = 0; j < 8; ++j) split(cent, 2, nib(R, 32 + 8 * h + j), r2[j], r1[2 * j], r1[2 * j + 1]);
#pragma unroll
    for (int j = 0; j < 16; ++j) split(cent, 1, nib(R, 16 * h + j), r1[j], x[2 * j], x[2 * j + 1]);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(sRopeSlot + sw128(row, 64 * h + 16 * q)) =
            make_uint4(pack_h2(x[8 * q], x[8 * q + 1]), pack_h2(x[8 * q + 2], x[8 * q + 3]),
                       pack_h2(x[8 * q + 4], x[8 * q + 5]), pack_h2(x[8 * q + 6], x[8 * q + 7]));
}

// 16 code bytes (32 codes, one per nibble, dims in order) -> 32 f16 levels at
// byte offset `b` (64 bytes) of swizzled row `row`, by byte permutes: the low
// 3 bits of each code pick a byte from levels 0-7 and from levels 8-15, bit 3
// picks between the two, then the low and high byte planes are interleaved.
// The selector and pick words are formed once per code word (8 codes) and
// shifted for its upper four codes (a byte permute reads only the low 16 bits
// of its selector).  No shared memory access (a 256-entry table in shared
// memory took ~4k bank-conflicted wavefronts per tile on the port the MMAs
// read their operands through).
__device__ __forceinline__ void store32(unsigned char* slot, const uint4& c, int row, int b, const LevelBytes& t) {
    const uint32_t in[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t sel = in[i] & 0x77777777u;
        const uint32_t pick = ((in[i] >> 1) & 0x44444444u) | 0x32103210u;
        uint32_t w[4];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const uint32_t sl = hh ? sel >> 16 : sel, pk = hh ? pick >> 16 : pick;
            const uint32_t l = __byte_perm(__byte_perm(t.lo[0], t.lo[1], sl), __byte_perm(t.lo[2], t.lo[3], sl), pk);
            const uint32_t h = __byte_perm(__byte_perm(t.hi[0], t.hi[1], sl), __byte_perm(t.hi[2], t.hi[3], sl), pk);
            w[2 * hh] = __byte_perm(l, h, 0x5140u);
            w[2 * hh + 1] = __byte_perm(l, h, 0x7362u);
        }
        *reinterpret_cast<uint4*>(slot + sw128(row, b + 16 * i)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <bool QBF16, bool PQ>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_tq4_kernel(AttnParams p) {
    launch_dependents();
    const int64_t w = blockIdx.x;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = smem_raw;
    unsigned char* sQ = sm + kOffQ;
    unsigned char* sSlot = sm + kOffSlot;
    unsigned char* sP = sSlot + kRope * kSlotBytes;
    unsigned char* sLevels = sm + kOffLevels;
    float2* sCent = reinterpret_cast<float2*>(sm + kOffCent);
    float* sM = reinterpret_cast<float*>(sm + kOffM);
    float* sR = reinterpret_cast<float*>(sm + kOffR);
    float* sE = reinterpret_cast<float*>(sm + kOffE);
    float* sF = reinterpret_cast<float*>(sm + kOffF);
    float* sEmax = reinterpret_cast<float*>(sm + kOffEmax);
    float* sAlpha = reinterpret_cast<float*>(sm + kOffAlpha);
    float* sAlphaM = reinterpret_cast<float*>(sm + kOffAlphaM);
    float* sRed = reinterpret_cast<float*>(sm + kOffRed);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
    volatile int* sAbort = reinterpret_cast<volatile int*>(sm + kOffMisc);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + kOffMisc + 4);
    int64_t* sInfo = reinterpret_cast<int64_t*>(sm + kOffMisc + 8);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // item-major linear grid: the CTAs of the first items (the ones with work)
    // are dispatched first; item and head group are re-derived where the
    // epilogue needs them, so that they hold no register over the tile loop
    const int64_t item = w / (p.n_heads / kHC);
    const int group = (int)(w % (p.n_heads / kHC));
    const int hbase = group * kHC;

    if (tid == 32 && p.prefill_past < 0) {
        // a decode batch's queries into L2, a slice per CTA, while warp 0
        // looks up the item (not for prefill, whose CTAs each read one
        // token's query, nor for batches whose queries would crowd the cache)
        const uint64_t total = (uint64_t)p.n_seq * p.n_heads * kMlaD * (QBF16 ? 2 : 4);   // a multiple of 16
        const uint64_t per = (total / gridDim.x + 15) & ~(uint64_t)15;
        const uint64_t off = per * blockIdx.x;
        if (total <= (32ull << 20) && off < total)
            prefetch_l2(reinterpret_cast<const char*>(p.q) + off, (uint32_t)min(per, total - off));
    }
    if (warp == 0) {
        int64_t r0 = 0, r1 = 0;
        int b = locate_item(p, item, lane, &r0, &r1);
        if (smem_u32(smem_raw) & 1023u) {
            if (lane == 0) set_err(p.err, KVQ_ERR_DEVICE);
            b = -1;
        }
        if (lane == 0) {
            sInfo[0] = b;
            sInfo[1] = r0;
            sInfo[2] = r1;
        }
    }
    __syncthreads();
    const int b = (int)sInfo[0];
    if (b < 0) return;
    const int64_t row0 = sInfo[1], row1 = sInfo[2];
    const int n_tiles = (int)((row1 - row0 + kRows - 1) / kRows);

    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(sTmem)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 64) {
        for (int i = 0; i < kNumBars; ++i) {
            // PolarQuant: each latent group comes from the 128 threads of one half
            const uint32_t count = (i < kBarFree0 || i == kBarP)
                                       ? ((PQ && i < kBarFull0 + 2) ? (uint32_t)kWorkers / 2 : (uint32_t)kWorkers)
                                       : 1u;
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&bars[i])), "r"(count));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *sAbort = 0;
    }
    if (tid < kHC) {
        sM[tid] = -INFINITY;
        sR[tid] = -INFINITY;
        sE[tid] = 0.0f;
        sF[tid] = 0.0f;
    }
    if (PQ)
        for (int i = tid; i < 9 * 16; i += kThreads) sCent[i] = p.pq_cent[i];
    if (!PQ && tid == 0) {
        // one thread builds both planes in registers and stores each as one
        // 16-byte word, so no word of them is written by two threads; the
        // barrier after the prologue orders these stores before every reader
        uint32_t lo[4] = {0u, 0u, 0u, 0u}, hi[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const uint32_t h = __half_as_ushort(__float2half_rn(__fmul_rn(p.lv[k], kTq4Gamma)));
            lo[k >> 2] |= (h & 0xffu) << (8 * (k & 3));
            hi[k >> 2] |= (h >> 8) << (8 * (k & 3));
        }
        *reinterpret_cast<uint4*>(sLevels) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        *reinterpret_cast<uint4*>(sLevels + 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    }
    if (tid == 0) {
        const int64_t n = min((int64_t)kRows, row1 - row0);
        prefetch_l2(p.codes + row0 * kRowBytes, (uint32_t)(n * kRowBytes));
        // the second tile too: the loop keeps the L2 prefetch two tiles ahead
        if (row0 + kRows < row1)
            prefetch_l2(p.codes + (row0 + kRows) * kRowBytes, (uint32_t)(min((int64_t)kRows, row1 - row0 - kRows) * kRowBytes));
    }

    // ---- query: 32 heads, 4 per worker warp, rotated once (sign flip, FWHT of
    // the 512 and 64 blocks, 1/sqrt(n)), then stored as an f16 pair scaled by a
    // power of two that keeps every element below 2^14 ----
    const int64_t qbase = ((int64_t)b * p.n_heads + hbase) * kMlaD;
    float qv[4][18];
    if (tid < kWorkers) {
        float qmax = 0.0f;
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
            const int64_t base = qbase + (int64_t)(4 * warp + hh) * kMlaD;
#pragma unroll
            for (int k = 0; k < 18; ++k) {
                const int64_t idx = base + lane + 32 * k;
                qv[hh][k] = QBF16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.q)[idx])
                                  : reinterpret_cast<const float*>(p.q)[idx];
                qmax = fmaxf(qmax, fabsf(qv[hh][k]));
            }
        }
        qmax = warp_max(qmax);
        if (lane == 0) sRed[warp] = qmax;
    }
    __syncthreads();
    float q_max = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) q_max = fmaxf(q_max, sRed[i]);
    // |q'_i| <= ||q|| <= 24 max|q| for the rotated query
    const float q_bound = 24.0f * q_max;
    int e_q = 0;
    if (q_bound > 0.0f) frexpf(q_bound, &e_q);
    const float q_scale = q_bound > 0.0f ? ldexpf(1.0f, 14 - e_q) : 1.0f;
    const float cz = p.sm_scale * kLog2e * (q_bound > 0.0f ? ldexpf(1.0f, e_q - 14) : 1.0f) * (PQ ? 1.0f : kTq4InvGamma);
    if (tid < kWorkers) {
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
            float (&v)[18] = qv[hh];
#pragma unroll
            for (int k = 0; k < 16; ++k)
                if (sign_neg(p.signs, 0, lane + 32 * k)) v[k] = -v[k];
            warp_fwht<512>(v, lane);
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = __fmul_rn(v[k], p.kn[0]);
#pragma unroll
            for (int k = 16; k < 18; ++k)
                if (sign_neg(p.signs, 1, lane + 32 * (k - 16))) v[k] = -v[k];
            warp_fwht<64>(v + 16, lane);
#pragma unroll
            for (int k = 16; k < 18; ++k) v[k] = __fmul_rn(v[k], p.kn[1]);
            const int h = 4 * warp + hh;
#pragma unroll
            for (int k = 0; k < 18; ++k) {
                const int d = lane + 32 * k;
                const float x = v[k] * q_scale;
                const __half hi = __float2half_rn(x);
                const __half lo = __float2half_rn(x - __half2float(hi));
                unsigned char* chunk = sQ + (d >> 6) * kQChunkBytes;
                *reinterpret_cast<__half*>(chunk + sw128(h, (d & 63) * 2)) = hi;
                *reinterpret_cast<__half*>(chunk + sw128(kHC + h, (d & 63) * 2)) = lo;
            }
        }
    }
    fence_async_smem();
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem = *sTmem;

    if (warp >= kWorkers / 32) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsMma));
        // ================= MMA warp: lane 0 issues =================
        if (warp == kWorkers / 32 && lane == 0) {
            const uint64_t dq0 = umma_desc(smem_u32(sQ), 16, 1024);
            const uint64_t dslot0 = umma_desc(smem_u32(sSlot), 16, 1024);
            const uint64_t dpair0 = umma_desc(smem_u32(sSlot), kSlotBytes, 1024);
            const uint64_t dp = umma_desc(smem_u32(sP), 16, 1024);
            constexpr uint64_t kQStep = kQChunkBytes >> 4, kSlotStep = kSlotBytes >> 4, kPStep = kPChunkBytes >> 4;
            bool ok = true;
            if (p.stall_polls > 0) ok = mbar_wait(&bars[kBarNever], 0u, sAbort, p.stall_polls);
            for (int t = 0; t < n_tiles && ok; ++t) {
                const uint32_t par = (uint32_t)t & 1u;
#pragma unroll 1
                for (int kc = 0; kc < kChunks && ok; ++kc) {
                    if ((kc & 3) == 0) {
                        ok = mbar_wait(&bars[kBarFull0 + (kc >> 2)], par, sAbort, p.wait_limit);
                        tc_after();
                    }
                    const uint32_t d = tmem + (kc < kRope ? kColSL : kColSR);
                    const uint64_t a = dslot0 + kc * kSlotStep, bq = dq0 + kc * kQStep;
                    const bool first = kc == 0 || kc == kRope;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        umma_f16(d, a + 2 * ks, bq + 2 * ks, kIdescScore, (first && ks == 0) ? 0u : 1u);
                }
                umma_commit(&bars[kBarScore]);
                ok = ok && mbar_wait(&bars[kBarP], par, sAbort, p.wait_limit);
                tc_after();
#pragma unroll 1
                for (int db = 0; db < 4 && ok; ++db) {
                    const uint32_t d = tmem + kColO + kHC * db;
                    const uint64_t a = dpair0 + 2 * db * kSlotStep;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        umma_f16(d, a + 128 * ks, dp + (ks >> 2) * kPStep + 2 * (ks & 3), kIdescCtx,
                                 (t > 0 || ks > 0) ? 1u : 0u);
                    umma_commit(&bars[kBarFree0 + db]);
                }
            }
            umma_commit(&bars[kBarDone]);
        }
        return;
    }

    // ================= workers =================
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsWorker));
    const int srow = 32 * (warp & 3) + lane;            // softmax: TMEM lane / row
    const int hq = warp >> 2;                            // softmax: heads 16 hq .. 16 hq + 15
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    // this thread's row: sums of p for its 16 heads over every tile so far
    // (reduced over the rows once, in the epilogue); m and E of its heads,
    // refreshed after each exact path
    float lsum[16], mreg[16], ereg[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) lsum[j] = 0.0f;
    auto load_state = [&]() {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            mreg[j] = sM[16 * hq + j];
            ereg[j] = sE[16 * hq + j];
        }
    };
    load_state();
    float s_lim = 0.0f;  // latent scales above this take the exact path (3.5 / max_h E)

    float sl_next = 0.0f, sr_next = 0.0f;
    auto load_scales = [&](int64_t t0n, int ntn) {
        sl_next = sr_next = 0.0f;
        if (srow < ntn) {
            const int64_t r = t0n + srow;
            sl_next = p.scales[r * p.n_blocks];
            sr_next = p.scales[r * p.n_blocks + (p.n_blocks - 1)];
        }
    };
    RawGroup rawA, rawB;
    uint4 rawC;
    RawPQ rawP;
    auto load_tile = [&](int64_t t0n, int ntn) {
        if constexpr (PQ) {
            load_pq(rawP, p.codes, t0n, ntn, warp, lane);
        } else {
            load_group(rawA, p.codes, t0n, ntn, 0, warp, lane);
            load_group(rawB, p.codes, t0n, ntn, 1, warp, lane);
            rawC = load_rope(p.codes, t0n, ntn, warp, lane);
        }
        load_scales(t0n, ntn);
    };
    load_tile(row0, (int)min((int64_t)kRows, row1 - row0));
    int t = 0;
    for (; t < n_tiles; ++t) {
        const int64_t t0 = row0 + (int64_t)t * kRows;
        const int nt = (int)min((int64_t)kRows, row1 - t0);
        if (tid == 0 && t0 + 2 * kRows < row1) {
            const int64_t n = min((int64_t)kRows, row1 - (t0 + 2 * kRows));
            prefetch_l2(p.codes + (t0 + 2 * kRows) * kRowBytes, (uint32_t)(n * kRowBytes));
        }
        const float my_sl = sl_next, my_sr = sr_next;
        // ---- decode the tile: groups A (chunks 0-3), B (4-7), C (rope) ----
        const uint32_t prev = (uint32_t)(t - 1) & 1u;
        if constexpr (PQ) {
            // half h of row 32 (warp / 2) + lane: latent chunks 4h .. 4h + 3
            // (group A or B), then half of the rope chunk (group C)
            const int h = warp & 1, row = 32 * (warp >> 1) + lane;
            if (t > 0) {
                mbar_wait(&bars[kBarFree0 + 2 * h], prev, sAbort, p.wait_limit);
                mbar_wait(&bars[kBarFree0 + 2 * h + 1], prev, sAbort, p.wait_limit);
            }
            if (h) pq_latent_half<1>(rawP, row, sCent, sSlot);
            else pq_latent_half<0>(rawP, row, sCent, sSlot);
            fence_async_smem();
            mbar_arrive(&bars[kBarFull0 + h]);
            if (t > 0 && h == 0) mbar_wait(&bars[kBarFree0 + 3], prev, sAbort, p.wait_limit);
            if (h) pq_rope_half<1>(rawP, row, sCent, sSlot + kRope * kSlotBytes);
            else pq_rope_half<0>(rawP, row, sCent, sSlot + kRope * kSlotBytes);
            fence_async_smem();
            mbar_arrive(&bars[kBarFull0 + 2]);
        } else {
            // the level byte planes, re-read per tile (asm volatile: not kept
            // in registers across the softmax)
            LevelBytes lvb;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(lvb.lo[0]), "=r"(lvb.lo[1]), "=r"(lvb.lo[2]), "=r"(lvb.lo[3])
                         : "r"(smem_u32(sLevels))
                         : "memory");
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(lvb.hi[0]), "=r"(lvb.hi[1]), "=r"(lvb.hi[2]), "=r"(lvb.hi[3])
                         : "r"(smem_u32(sLevels + 16))
                         : "memory");
            const int half = lane & 1, cg = lane >> 3;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                if (t > 0) {
                    mbar_wait(&bars[kBarFree0 + 2 * g], prev, sAbort, p.wait_limit);
                    mbar_wait(&bars[kBarFree0 + 2 * g + 1], prev, sAbort, p.wait_limit);
                }
                unsigned char* slot = sSlot + (4 * g + cg) * kSlotBytes;
                const RawGroup& rg = g == 0 ? rawA : rawB;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    store32(slot, rg.v[i], 4 * (warp + 8 * i) + ((lane >> 1) & 3), 64 * half, lvb);
                fence_async_smem();
                mbar_arrive(&bars[kBarFull0 + g]);
            }
            store32(sSlot + kRope * kSlotBytes, rawC, 16 * warp + (lane >> 1), 64 * half, lvb);
            fence_async_smem();
            mbar_arrive(&bars[kBarFull0 + 2]);
        }
        const int64_t t1 = t0 + kRows;
        const int nt1 = (int)min((int64_t)kRows, row1 - t1);
        // all of tile t+1 is requested before the softmax (the raw codes stay in
        // registers across it: the workers' share of the register split)
        if (t + 1 < n_tiles) load_tile(t1, nt1);

        // ---- softmax of the tile: thread = row srow, 16 heads ----
        // one warp polls; the others wait on the named barrier, issuing nothing
        if (warp == 1) mbar_wait(&bars[kBarScore], (uint32_t)t & 1u, sAbort, p.wait_limit);
        worker_sync();
        tc_after();
        float z[16];
        const float za = my_sl * cz, zb = my_sr * cz;
        const bool row_ok = srow < nt;
        auto load_z = [&]() {
            // the four 16-column loads go out together, then one wait
            uint32_t a[16], c[16], e[16], f[16];
            tmem_ld16(tmem + lane_base + kColSR + 16 * hq, a);            // rope, values
            tmem_ld16(tmem + lane_base + kColSR + kHC + 16 * hq, c);      // rope, residuals
            tmem_ld16(tmem + lane_base + kColSL + 16 * hq, e);
            tmem_ld16(tmem + lane_base + kColSL + kHC + 16 * hq, f);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j)
                z[j] = row_ok ? fmaf(__uint_as_float(e[j]) + __uint_as_float(f[j]), za,
                                     (__uint_as_float(a[j]) + __uint_as_float(c[j])) * zb)
                              : -INFINITY;
        };
        // d = z - m: the lag test and the weights 2^d (m = -inf before the first
        // exact path: d = +inf on every row of the tile)
        auto load_d = [&]() {
            uint32_t a[16], c[16], e[16], f[16];
            tmem_ld16(tmem + lane_base + kColSR + 16 * hq, a);
            tmem_ld16(tmem + lane_base + kColSR + kHC + 16 * hq, c);
            tmem_ld16(tmem + lane_base + kColSL + 16 * hq, e);
            tmem_ld16(tmem + lane_base + kColSL + kHC + 16 * hq, f);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j)
                z[j] = row_ok ? fmaf(__uint_as_float(e[j]) + __uint_as_float(f[j]), za,
                                     fmaf(__uint_as_float(a[j]) + __uint_as_float(c[j]), zb, -mreg[j]))
                              : -INFINITY;
        };
        load_d();
        // one maximum over the heads, then one test
        float dm[4] = {z[0], z[1], z[2], z[3]};
#pragma unroll
        for (int j = 4; j < 16; ++j) dm[j & 3] = fmaxf(dm[j & 3], z[j]);
        const float dmax = fmaxf(fmaxf(dm[0], dm[1]), fmaxf(dm[2], dm[3]));
        const bool flag = (*sAbort != 0) | (my_sl > s_lim) | (dmax > kLagLog2);
        if (worker_any(flag)) {
            if (worker_any(*sAbort != 0)) break;
            // exact column maxima of z and of y = z + log2 s_L, new running
            // maxima, rescale factors
            load_z();
            {
                const float cm = warp_columns16<true>(z, lane);
                if (lane < 16) sRed[(warp & 3) * kHC + 16 * hq + lane] = cm;
            }
            load_z();
            const float ls = my_sl > 0.0f ? __log2f(my_sl) : -INFINITY;   // -inf: an inert latent block
#pragma unroll
            for (int j = 0; j < 16; ++j) z[j] += ls;
            {
                const float cm = warp_columns16<true>(z, lane);
                if (lane < 16) sRed[4 * kHC + (warp & 3) * kHC + 16 * hq + lane] = cm;
            }
            worker_sync();
            if (tid < kHC) {
                const float* rz = sRed;
                const float* ry = sRed + 4 * kHC;
                const float cz4 = fmaxf(fmaxf(rz[tid], rz[kHC + tid]), fmaxf(rz[2 * kHC + tid], rz[3 * kHC + tid]));
                const float cy4 = fmaxf(fmaxf(ry[tid], ry[kHC + tid]), fmaxf(ry[2 * kHC + tid], ry[3 * kHC + tid]));
                const float mo = sM[tid], mn = fmaxf(mo, cz4);
                const float ro = sR[tid], rn = fmaxf(ro, cy4);
                const float dn = fminf(mn - rn - kHeadroom, kLogEmax), d_old = fminf(mo - ro - kHeadroom, kLogEmax);
                sAlphaM[tid] = mo == -INFINITY ? 0.0f : ex2(mo - mn);
                sAlpha[tid] = ro == -INFINITY ? 0.0f : ex2(dn - d_old + (mo - mn));   // E_new / E_old x 2^(m_old - m_new)
                sM[tid] = mn;
                sR[tid] = rn;
                const float e = rn == -INFINITY ? 0.0f : ex2(dn);   // R = -inf: only inert latent blocks so far
                sE[tid] = e;
                sF[tid] = rn == -INFINITY ? 0.0f : ex2(-dn);
                const float em = warp_max(e);
                if (tid == 0) {
                    sEmax[0] = em;
                    if (t > 0) atomicAdd(p.exact_count, 1u);
                }
            }
            worker_sync();
            s_lim = sEmax[0] > 0.0f ? 3.5f / sEmax[0] : 0.0f;
            if (t > 0) {
                // O^T (lanes = dims, columns = heads) is stable: the score commit
                // of this tile follows every context MMA of the previous one
                const uint32_t ta = tmem + lane_base + kColO + kHC * (2 * hq);
#pragma unroll 1
                for (int bi = 0; bi < 2; ++bi) {
                    uint32_t o[32];
                    tmem_ld32(ta + kHC * bi, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * sAlpha[j]);
                    tmem_st32(ta + kHC * bi, o);
                }
                tmem_wait_st();
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) lsum[j] *= sAlphaM[16 * hq + j];
            load_state();
            load_d();
        }
        {
            // row-sum weights p = 2^(z - m), f16 context weights w = p s_L E
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int h = 16 * hq + j;
                z[j] = ex2(z[j]);
                *reinterpret_cast<__half*>(sP + (srow >> 6) * kPChunkBytes + sw128(h, (srow & 63) * 2)) =
                    __float2half_rn(z[j] * ereg[j] * my_sl);
            }
        }
        fence_async_smem();
        tc_before();
        mbar_arrive(&bars[kBarP]);
#pragma unroll
        for (int j = 0; j < 16; ++j) lsum[j] += z[j];
    }

    // ---- epilogue: wait for every MMA, row sums, O^T -> partial state ----
    {
        volatile int never = 0;
        if (!mbar_wait(&bars[kBarDone], 0u, &never)) *sAbort = 1;
    }
    tc_after();
    const bool aborted = worker_any(*sAbort != 0 || t < n_tiles);
    {
        worker_sync();
        const float lcol = warp_columns16<false>(lsum, lane);
        if (lane < 16) sRed[(warp & 3) * kHC + 16 * hq + lane] = lcol;
        worker_sync();
        if (tid < kHC) sAlpha[tid] = (sRed[tid] + sRed[kHC + tid]) + (sRed[2 * kHC + tid] + sRed[3 * kHC + tid]);
        worker_sync();
    }
    if (aborted) {
        if (tid == 0) set_err(p.err, KVQ_ERR_TIMEOUT);
    } else {
        const int64_t unit = blockIdx.x;
        const int64_t item = unit / (p.n_heads / kHC);
        const int hbase = (int)(unit % (p.n_heads / kHC)) * kHC;
        const float o_scale = PQ ? 1.0f : kTq4InvGamma;
#pragma unroll
        for (int bi = 0; bi < 2; ++bi) {
            const int db = 2 * hq + bi;
            const int dim = 128 * db + 32 * (warp & 3) + lane;
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + kColO + kHC * db, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int h = hbase + j;
                p.ws_o[(item * p.n_heads + h) * kMlaDV + dim] =
                    n_tiles > 0 ? __uint_as_float(v[j]) * (sF[j] * o_scale) : 0.0f;
            }
        }
        if (tid < kHC) {
            float* ml = p.ws_ml + (item * p.n_heads + hbase + tid) * 2;
            ml[0] = sM[tid] * kLn2;
            ml[1] = sAlpha[tid];
        }
    }
    tc_before();
    worker_sync();
    tc_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

template <bool QBF16, bool PQ>
cudaError_t launch_tq4(const AttnParams& p, int64_t grid_x, int groups, cudaStream_t stream) {
    // the workers' setmaxnreg.inc waits for registers the other warpgroup
    // released: launch only if the split adds up against the launch's count
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, attn_tc_tq4_kernel<QBF16, PQ>);
    if (e != cudaSuccess) return e;
    if (kWorkers * kRegsWorker + 128 * kRegsMma > kThreads * fa.numRegs) return cudaErrorInvalidConfiguration;
    if (PQ && !p.pq_cent) return cudaErrorInvalidSymbol;
    e = cudaFuncSetAttribute(attn_tc_tq4_kernel<QBF16, PQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemUsed);
    if (e != cudaSuccess) return e;
    attn_tc_tq4_kernel<QBF16, PQ><<<dim3((unsigned)(grid_x * groups)), kThreads, kSmemUsed, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_tc_tq4(const AttnParams& p, bool q_bf16, bool pq, int64_t grid_x, int n_heads,
                               cudaStream_t stream) {
    const int g = n_heads / kHC;
    if (pq) return q_bf16 ? launch_tq4<true, true>(p, grid_x, g, stream) : launch_tq4<false, true>(p, grid_x, g, stream);
    return q_bf16 ? launch_tq4<true, false>(p, grid_x, g, stream) : launch_tq4<false, false>(p, grid_x, g, stream);
}

}  // namespace kvq
