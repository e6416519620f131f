// attn_tc.cu -- tensor-core (tcgen05 / TMEM) attention over quantized MLA rows.
//
// All heads share one latent cache, so per tile of rows the score (heads x
// rows x 576) and the context (heads x 512 x rows) are dense contractions.
// They run on the 5th-generation tensor cores with f16 operands decoded from
// the quantized rows in shared memory; accumulators live in tensor memory.
//
// Formulation (transposed, per CTA: one chunk of rows x 64 heads):
//   S_L^T[t][h] = sum_{d<512} c[t][d] q[h][d]     M = 128 rows, N = 64 heads
//   S_R^T[t][h] = sum_{d>=512} c[t][d] q[h][d]    (the rope block, own scale)
//   O^T[d][h]  += sum_t c[t][d] * P^T[t][h]        M = 128 dims (x4), K = rows
// c are the codes' values (e4m3 value, or TQ4 codebook level against the
// rotated query), exact in f16 for KV8.  The per-row scales stay outside the
// products and are applied by the thread that owns the row: z = sm*(s_L*S_L +
// s_R*S_R), and the context weight is p*s_L ([P2] "What's in it": the row
// scale factors out of both sums; [P1] "Ready for review" comment, finding 2:
// TQ4 dots the rotated query with codebook levels and unrotates once).
//
// TMEM (512 columns x 128 lanes of f32): O^T = 4 blocks x 64 columns, S_L^T and
// S_R^T 64 columns each.  A full O for 128 heads x 512 dims would fill all of
// TMEM, which is why a CTA serves 64 heads and two CTAs share each chunk.
//
// Softmax in this layout: a thread owns one row (a TMEM lane) and 32 heads.
// The running max per head is lagged: rows are exponentiated against the max
// of the previous tiles and a tile takes an exact slow path (column max over
// the tile, rescale of O^T in TMEM) only when some score exceeds that max by
// more than 2^8.  Row sums are accumulated per thread and reduced across the
// 128 rows once per chunk.  The partial state written for the merge is the
// same as the SIMT path's, in natural-log units.
#include "attn_common.cuh"

#include <algorithm>
#include <math.h>

namespace kvq {
namespace {

constexpr int kRows = 128;      // rows per tile: the score's M, the context's K
constexpr int kHC = 64;         // heads per CTA: the MMA N
constexpr int kThreads = 256;
constexpr int kSlots = 4;       // f16 staging slots of 128 rows x 64 dims
constexpr uint32_t kSlotBytes = kRows * 128;
// query chunk kc (64 dims): rows 0..63 = f16(q) of the 64 heads, rows 64..127 =
// f16(q - f16(q)), the residual that makes the pair exact to ~22 bits
constexpr uint32_t kQChunkBytes = 2 * kHC * 128;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffSlot = kOffQ + 9 * kQChunkBytes;
constexpr uint32_t kOffP = kOffSlot + kSlots * kSlotBytes;
constexpr uint32_t kOffScale = kOffP + kRows * 128;
constexpr uint32_t kOffM = kOffScale + kRows * 8;
constexpr uint32_t kOffAlpha = kOffM + kHC * 4;
constexpr uint32_t kOffLut = kOffAlpha + kHC * 4;
constexpr uint32_t kOffBar = kOffLut + 256 * 4;
constexpr uint32_t kOffMisc = kOffBar + 8 * 8;   // abort flag, TMEM base, item info, reductions
constexpr uint32_t kSmemUsed = kOffMisc + 128;
constexpr size_t kSmemAlloc = kSmemUsed;          // the base is 1024-aligned (checked at run time)
static_assert(kSmemAlloc <= 232448, "shared memory budget");

// TMEM columns: O^T blocks 0..255; S_L^T 256..383 and S_R^T 384..511, each as
// 64 columns for the f16 query and 64 for its residual
constexpr uint32_t kColO = 0, kColSL = 256, kColSR = 384, kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr long long kWaitLimit = 1ll << 24;

enum { kBarSlot0 = 0, kBarScore = 4, kBarCtx = 5 };

__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn, bool b_mn) {
    // D f32 (bit 4), A and B f16 (format 0), operand majors, N>>3 at 17, M>>4 at 24
    return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kIdescScore = idesc_f16(128, kHC, false, false);
constexpr uint32_t kIdescScore2 = idesc_f16(128, 2 * kHC, false, false);
constexpr uint32_t kIdescCtx = idesc_f16(128, kHC, true, true);

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Byte offset of (row r, byte b) in a region of 128-byte rows laid out in the
// 128-byte swizzle (16-byte chunk index XOR row index within 8-row atoms).
__device__ __forceinline__ uint32_t sw128(int r, int b) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((b >> 4) ^ r) & 7) << 4) + (b & 15));
}

// Shared-memory matrix descriptor: start, leading and stride byte offsets,
// descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void umma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Bounded wait on an mbarrier phase.  Returns false (and raises the CTA's
// abort flag) when the limit is reached; later waits then return at once.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    if (*abort_flag) return false;
    const uint32_t a = smem_u32(bar);
    for (long long i = 0; i < kWaitLimit; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(a), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    *abort_flag = 1;
    return false;
}

#define KVQ_R32(v) \
    "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), \
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),   \
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), \
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
#define KVQ_W32(v)                                                                                                \
    "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), \
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),          \
        "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]),           \
        "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])

// 32 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : KVQ_R32(v)
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        KVQ_W32(v));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t e4m3x2_to_half2_bits(uint32_t two) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
    return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// Decodes dims [64 kc, 64 kc + 64) of the tile's 128 rows to f16 code values in
// a staging slot (row r = one 128-byte swizzled row).  Rows past the end are 0.
template <int FMT>
__device__ __forceinline__ void decode_chunk(const uint8_t* __restrict__ codes, int64_t t0, int nt, int kc,
                                             unsigned char* slot, const uint32_t* lut, int tid) {
    const int r = tid >> 1, half = tid & 1;
    uint32_t w[16];
    if (r < nt) {
        if (FMT == KVQ_KV8) {
            const uint4* src = reinterpret_cast<const uint4*>(codes + (t0 + r) * kMlaD + kc * 64 + half * 32);
            const uint4 a = __ldg(src), b = __ldg(src + 1);
            const uint32_t in[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                w[2 * i] = e4m3x2_to_half2_bits(in[i] & 0xffffu);
                w[2 * i + 1] = e4m3x2_to_half2_bits(in[i] >> 16);
            }
        } else {
            const uint4 a = __ldg(reinterpret_cast<const uint4*>(codes + (t0 + r) * (kMlaD / 2) + kc * 32 + half * 16));
            const uint32_t in[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) w[4 * i + j] = lut[(in[i] >> (8 * j)) & 0xffu];
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = 0u;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(slot + sw128(r, half * 64 + 16 * j)) =
            make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
}

// TQ4: the f16 rounding residual of each code's level (level - f16(level)),
// same layout as decode_chunk.  Residuals are below 4e-4 of the level.
__device__ __forceinline__ void decode_delta_chunk(const uint8_t* __restrict__ codes, int64_t t0, int nt, int kc,
                                                   unsigned char* slot, const __half* delta, int tid) {
    const int r = tid >> 1, half = tid & 1;
    uint32_t w[16];
    if (r < nt) {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(codes + (t0 + r) * (kMlaD / 2) + kc * 32 + half * 16));
        const uint32_t in[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t byte = (in[i] >> (8 * j)) & 0xffu;
                w[4 * i + j] = (uint32_t)__half_as_ushort(delta[byte & 15u]) |
                               ((uint32_t)__half_as_ushort(delta[byte >> 4]) << 16);
            }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = 0u;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(slot + sw128(r, half * 64 + 16 * j)) =
            make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
}

template <int FMT, bool QBF16>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(AttnParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = smem_raw;
    unsigned char* sQ = sm + kOffQ;
    unsigned char* sSlot = sm + kOffSlot;
    unsigned char* sP = sm + kOffP;
    float2* sScale = reinterpret_cast<float2*>(sm + kOffScale);
    float* sM = reinterpret_cast<float*>(sm + kOffM);
    float* sAlpha = reinterpret_cast<float*>(sm + kOffAlpha);
    uint32_t* sLut = reinterpret_cast<uint32_t*>(sm + kOffLut);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
    volatile int* sAbort = reinterpret_cast<volatile int*>(sm + kOffMisc);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + kOffMisc + 4);
    int* sHasLo = reinterpret_cast<int*>(sm + kOffMisc + 8);
    int64_t* sInfo = reinterpret_cast<int64_t*>(sm + kOffMisc + 16);
    float* sRed = reinterpret_cast<float*>(sm + kOffMisc + 48);
    __half* sDelta = reinterpret_cast<__half*>(sm + kOffMisc + 80);   // TQ4: level - f16(level)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t item = blockIdx.x;
    const int hbase = blockIdx.y * kHC;

    if (warp == 0) {
        int64_t r0 = 0, r1 = 0;
        int b = locate_item(p, item, lane, &r0, &r1);
        if (smem_u32(smem_raw) & 1023u) {          // the swizzled layouts need a 1024-byte aligned base
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
    if (b < 0) return;   // past the last work item: nothing allocated yet
    const int64_t row0 = sInfo[1], row1 = sInfo[2];

    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(sTmem)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 64) {
        for (int i = 0; i < 6; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bars[i])));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *sAbort = 0;
        *sHasLo = 0;
    }
    if (tid < kHC) sM[tid] = -INFINITY;
    if (FMT == KVQ_TQ4) {
        const int lo = tid & 15, hi = tid >> 4;
        const __half2 h2 = __halves2half2(__float2half_rn(p.lv[lo]), __float2half_rn(p.lv[hi]));
        sLut[tid] = *reinterpret_cast<const uint32_t*>(&h2);
        if (tid < 16) sDelta[tid] = __float2half_rn(p.lv[tid] - __half2float(__float2half_rn(p.lv[tid])));
    }

    // reference scale of the chunk: a power of two >= every latent scale, so
    // that the context weights p * s_L / S_ref stay within f16 range
    float smax = 0.0f;
    for (int64_t r = row0 + tid; r < row1; r += kThreads) smax = fmaxf(smax, p.scales[r * p.n_blocks]);
    smax = warp_max(smax);
    if (lane == 0) sRed[warp] = smax;
    // query norm bound of the CTA's heads: fixes one power-of-two prescale
    // keeping every f16 query element below 2^14
    float qn = 0.0f;
    for (int h = warp; h < kHC; h += kThreads / 32) {
        float ss = 0.0f;
        for (int d = lane; d < kMlaD; d += 32) {
            const float v = load_q<QBF16>(p.q, ((int64_t)b * p.n_heads + hbase + h) * kMlaD + d);
            ss = fmaf(v, v, ss);
        }
        qn = fmaxf(qn, sqrtf(warp_sum(ss)));
    }
    tc_before();
    __syncthreads();
    tc_after();
    float s_max = 0.0f;
    for (int i = 0; i < 8; ++i) s_max = fmaxf(s_max, sRed[i]);
    __syncthreads();
    if (lane == 0) sRed[warp] = qn;
    __syncthreads();
    float q_bound = 0.0f;
    for (int i = 0; i < 8; ++i) q_bound = fmaxf(q_bound, sRed[i]);
    int e_s = 0, e_q = 0;
    if (s_max > 0.0f) frexpf(s_max, &e_s);
    if (q_bound > 0.0f) frexpf(q_bound, &e_q);
    const float s_ref = s_max > 0.0f ? ldexpf(1.0f, e_s) : 1.0f;
    const float inv_s_ref = s_max > 0.0f ? ldexpf(1.0f, -e_s) : 1.0f;
    const float q_scale = q_bound > 0.0f ? ldexpf(1.0f, 14 - e_q) : 1.0f;
    const float cz = p.sm_scale * kLog2e * (q_bound > 0.0f ? ldexpf(1.0f, e_q - 14) : 1.0f);
    const uint32_t tmem = *sTmem;

    // queries -> f16 pair (value, residual) in the score's B layout (K-major,
    // 9 chunks of 64 dims x 128 rows)
    int any_lo = 0;
    for (int h = warp; h < kHC; h += kThreads / 32) {
        float v[18];
        const int64_t qoff = ((int64_t)b * p.n_heads + hbase + h) * kMlaD;
#pragma unroll
        for (int k = 0; k < 18; ++k) v[k] = load_q<QBF16>(p.q, qoff + lane + 32 * k);
        if (FMT == KVQ_TQ4) {
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
        }
#pragma unroll
        for (int k = 0; k < 18; ++k) {
            const int d = lane + 32 * k;
            const float x = v[k] * q_scale;
            const __half hi = __float2half_rn(x);
            const __half lo = __float2half_rn(x - __half2float(hi));
            any_lo |= __half_as_ushort(lo) & 0x7fff;
            unsigned char* chunk = sQ + (d >> 6) * kQChunkBytes;
            *reinterpret_cast<__half*>(chunk + sw128(h, (d & 63) * 2)) = hi;
            *reinterpret_cast<__half*>(chunk + sw128(kHC + h, (d & 63) * 2)) = lo;
        }
    }
    if (any_lo) atomicOr(sHasLo, 1);
    fence_async_smem();
    tc_before();
    __syncthreads();
    tc_after();
    // a query exact in f16 (bf16 input) needs only the first 64 rows
    const bool has_lo = *sHasLo != 0;

    const int srow = 32 * (warp & 3) + lane;   // TMEM lane owned in the softmax
    const int hq = warp >> 2;                   // heads 32 hq .. 32 hq + 31
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    float lsum[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) lsum[j] = 0.0f;
    uint32_t uses[kSlots] = {0u, 0u, 0u, 0u};
    bool o_init = false;
    int tile = 0;

    for (int64_t t0 = row0; t0 < row1 && !*sAbort; t0 += kRows, ++tile) {
        const int nt = (int)min((int64_t)kRows, row1 - t0);
        if (tid < kRows) {
            float2 s2 = make_float2(0.0f, 0.0f);
            if (tid < nt) {
                const int64_t r = t0 + tid;
                s2 = p.n_blocks == 2 ? make_float2(p.scales[r * 2], p.scales[r * 2 + 1])
                                     : make_float2(p.scales[r], p.scales[r]);
            }
            sScale[tid] = s2;
        }
        // ---- scores: 9 chunks of 64 dims (8 latent, 1 rope) ----
        for (int kc = 0; kc < 9; ++kc) {
            // KV8: one slot per chunk (codes are exact in f16).  TQ4: a slot pair,
            // the f16 levels and their rounding residuals, both multiplied by the
            // query into the same accumulator so the score sees the f32 levels.
            const int s = FMT == KVQ_KV8 ? (kc & 3) : (kc & 1) * 2;
            if (uses[s] > 0) mbar_wait(&bars[kBarSlot0 + s], (uses[s] - 1) & 1, sAbort);
            if (FMT == KVQ_TQ4 && uses[s + 1] > 0) mbar_wait(&bars[kBarSlot0 + s + 1], (uses[s + 1] - 1) & 1, sAbort);
            decode_chunk<FMT>(p.codes, t0, nt, kc, sSlot + s * kSlotBytes, sLut, tid);
            if (FMT == KVQ_TQ4) decode_delta_chunk(p.codes, t0, nt, kc, sSlot + (s + 1) * kSlotBytes, sDelta, tid);
            fence_async_smem();
            tc_before();
            __syncthreads();
            if (tid == 0) {
                tc_after();
                const uint32_t d = tmem + (kc < 8 ? kColSL : kColSR);
                const uint32_t a0 = smem_u32(sSlot + s * kSlotBytes), b0 = smem_u32(sQ + kc * kQChunkBytes);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    umma_f16(d, umma_desc(a0 + ks * 32, 16, 1024), umma_desc(b0 + ks * 32, 16, 1024),
                             has_lo ? kIdescScore2 : kIdescScore, (kc == 0 || kc == 8) ? (ks > 0 ? 1u : 0u) : 1u);
                if (FMT == KVQ_TQ4) {
                    const uint32_t a1 = smem_u32(sSlot + (s + 1) * kSlotBytes);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        umma_f16(d, umma_desc(a1 + ks * 32, 16, 1024), umma_desc(b0 + ks * 32, 16, 1024), kIdescScore,
                                 1u);
                }
                umma_commit(&bars[kBarSlot0 + s]);
                if (FMT == KVQ_TQ4) umma_commit(&bars[kBarSlot0 + s + 1]);
                if (kc == 8) umma_commit(&bars[kBarScore]);
            }
            ++uses[s];
            if (FMT == KVQ_TQ4) ++uses[s + 1];
        }
        // ---- softmax of the tile (thread = row, 32 heads) ----
        mbar_wait(&bars[kBarScore], tile & 1, sAbort);
        if (tile > 0) mbar_wait(&bars[kBarCtx], (tile - 1) & 1, sAbort);
        tc_after();
        float z[32];
        {
            uint32_t sl[32], sr[32];
            tmem_ld32(tmem + lane_base + kColSL + 32 * hq, sl);
            tmem_ld32(tmem + lane_base + kColSR + 32 * hq, sr);
            tmem_wait_ld();
            float fl[32], fr[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                fl[j] = __uint_as_float(sl[j]);
                fr[j] = __uint_as_float(sr[j]);
            }
            if (has_lo) {
                tmem_ld32(tmem + lane_base + kColSL + kHC + 32 * hq, sl);
                tmem_ld32(tmem + lane_base + kColSR + kHC + 32 * hq, sr);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    fl[j] += __uint_as_float(sl[j]);
                    fr[j] += __uint_as_float(sr[j]);
                }
            }
            const float2 sc = sScale[srow];
            const float a = sc.x * cz, bb = sc.y * cz;
            const bool valid = srow < nt;
#pragma unroll
            for (int j = 0; j < 32; ++j) z[j] = valid ? fmaf(fl[j], a, fr[j] * bb) : -INFINITY;
        }
        bool flag = false;
#pragma unroll
        for (int j = 0; j < 32; ++j) flag |= z[j] > sM[32 * hq + j] + 8.0f;
        if (__syncthreads_or(flag)) {
            // exact column max of the tile, new running max, rescale factors
            float* zbuf = reinterpret_cast<float*>(sSlot);   // 128 x 64 f32 over slots 0-1 (idle now)
#pragma unroll
            for (int j = 0; j < 32; ++j) zbuf[srow * kHC + 32 * hq + j] = z[j];
            __syncthreads();
            if (tid < kHC) {
                float cm = -INFINITY;
                for (int r = 0; r < kRows; ++r) cm = fmaxf(cm, zbuf[r * kHC + tid]);
                const float mo = sM[tid], mn = fmaxf(mo, cm);
                sAlpha[tid] = mo == -INFINITY ? 0.0f : exp2f(mo - mn);
                sM[tid] = mn;
            }
            __syncthreads();
            if (o_init) {
#pragma unroll
                for (int bi = 0; bi < 2; ++bi)
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint32_t ta = tmem + lane_base + kColO + 64 * (2 * hq + bi) + 32 * c;
                        uint32_t v[32];
                        tmem_ld32(ta, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * sAlpha[32 * c + j]);
                        tmem_st32(ta, v);
                    }
                tmem_wait_st();
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) lsum[j] *= sAlpha[32 * hq + j];
            tc_before();
            __syncthreads();
            tc_after();
        }
        {
            const float wrow = sScale[srow].x * inv_s_ref;
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float p0 = exp2f(z[j] - sM[32 * hq + j]);
                const float p1 = exp2f(z[j + 1] - sM[32 * hq + j + 1]);
                lsum[j] += p0;
                lsum[j + 1] += p1;
                const __half2 h2 = __floats2half2_rn(p0 * wrow, p1 * wrow);
                pk[j / 2] = *reinterpret_cast<const uint32_t*>(&h2);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<uint4*>(sP + sw128(srow, 64 * hq + 16 * i)) =
                    make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
        // ---- context: 4 blocks of 128 dims, K = the tile's 128 rows ----
        for (int db = 0; db < 4; ++db) {
            const int s0 = (db & 1) * 2;
            if (uses[s0] > 0) mbar_wait(&bars[kBarSlot0 + s0], (uses[s0] - 1) & 1, sAbort);
            if (uses[s0 + 1] > 0) mbar_wait(&bars[kBarSlot0 + s0 + 1], (uses[s0 + 1] - 1) & 1, sAbort);
            decode_chunk<FMT>(p.codes, t0, nt, 2 * db, sSlot + s0 * kSlotBytes, sLut, tid);
            decode_chunk<FMT>(p.codes, t0, nt, 2 * db + 1, sSlot + (s0 + 1) * kSlotBytes, sLut, tid);
            fence_async_smem();
            tc_before();
            __syncthreads();
            if (tid == 0) {
                tc_after();
                const uint32_t d = tmem + kColO + 64 * db;
                const uint32_t a0 = smem_u32(sSlot + s0 * kSlotBytes), b0 = smem_u32(sP);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    umma_f16(d, umma_desc(a0 + ks * 2048, kSlotBytes, 1024), umma_desc(b0 + ks * 2048, kSlotBytes, 1024),
                             kIdescCtx, (o_init || ks > 0) ? 1u : 0u);
                umma_commit(&bars[kBarSlot0 + s0]);
                umma_commit(&bars[kBarSlot0 + s0 + 1]);
                if (db == 3) umma_commit(&bars[kBarCtx]);
            }
            ++uses[s0];
            ++uses[s0 + 1];
        }
        o_init = true;
    }

    // ---- epilogue: row sums, O^T -> partial state ----
    if (tile > 0) mbar_wait(&bars[kBarCtx], (tile - 1) & 1, sAbort);
    tc_after();
    {
        float* lbuf = reinterpret_cast<float*>(sSlot);
#pragma unroll
        for (int j = 0; j < 32; ++j) lbuf[srow * kHC + 32 * hq + j] = lsum[j];
        __syncthreads();
        if (tid < kHC) {
            float l = 0.0f;
            for (int r = 0; r < kRows; ++r) l += lbuf[r * kHC + tid];
            sAlpha[tid] = l;
        }
        __syncthreads();
    }
    if (*sAbort) {
        if (tid == 0) set_err(p.err, KVQ_ERR_DEVICE);
    } else {
#pragma unroll
        for (int bi = 0; bi < 2; ++bi) {
            const int db = 2 * hq + bi;
            const int dim = 128 * db + 32 * (warp & 3) + lane;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + kColO + 64 * db + 32 * c, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int h = hbase + 32 * c + j;
                    p.ws_o[(item * p.n_heads + h) * kMlaDV + dim] = o_init ? __uint_as_float(v[j]) * s_ref : 0.0f;
                }
            }
        }
        if (tid < kHC) {
            float* ml = p.ws_ml + (item * p.n_heads + hbase + tid) * 2;
            ml[0] = sM[tid] * kLn2;
            ml[1] = sAlpha[tid];
        }
    }
    tc_before();
    __syncthreads();
    tc_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

template <int FMT, bool QBF16>
cudaError_t launch_tc(const AttnParams& p, int64_t grid_x, int groups, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<FMT, QBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemAlloc);
    if (e != cudaSuccess) return e;
    attn_tc_kernel<FMT, QBF16><<<dim3((unsigned)grid_x, (unsigned)groups), kThreads, kSmemAlloc, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(const kvq_mla_layout& L, int32_t n_heads) {
    (void)L;
    return n_heads > 0 && n_heads % kHC == 0;
}

AttnPlan plan_decode_tc(int32_t batch, int32_t n_heads, int64_t max_total_rows) {
    AttnPlan pl{};
    pl.heads_per_cta = kHC;
    const int64_t groups = std::max<int64_t>(1, n_heads / kHC);
    const int64_t target_items = std::max<int64_t>(1, 152 / groups);
    int64_t chunk = (std::max<int64_t>(max_total_rows, 1) + target_items - 1) / target_items;
    chunk = std::max<int64_t>(kRows, (chunk + kRows - 1) / kRows * kRows);
    pl.chunk = chunk;
    pl.max_items = (max_total_rows + chunk - 1) / chunk + batch;
    return pl;
}

cudaError_t launch_attn_tc(kvq_format fmt, const kvq_mla_layout& L, const void* q, kvq_dtype qdt, int32_t n_seq,
                           int32_t n_heads, const uint8_t* codes, const float* scales, const int64_t* cu_seqlens,
                           int64_t prefill_past, const AttnPlan& plan, float sm_scale, float* out, void* workspace,
                           cudaStream_t stream) {
    if (n_seq == 0 || n_heads == 0) return cudaSuccess;
    const AttnParams p = make_attn_params(fmt, L, q, n_seq, n_heads, codes, scales, cu_seqlens, prefill_past, plan,
                                          sm_scale, workspace);
    const int groups = n_heads / kHC;
    cudaError_t e;
    if (fmt == KVQ_KV8)
        e = qdt == KVQ_BF16 ? launch_tc<KVQ_KV8, true>(p, plan.max_items, groups, stream)
                            : launch_tc<KVQ_KV8, false>(p, plan.max_items, groups, stream);
    else
        e = qdt == KVQ_BF16 ? launch_tc<KVQ_TQ4, true>(p, plan.max_items, groups, stream)
                            : launch_tc<KVQ_TQ4, false>(p, plan.max_items, groups, stream);
    if (e != cudaSuccess) return e;
    return launch_attn_merge(fmt, p, out, stream);
}

}  // namespace kvq
