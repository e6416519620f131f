// attn_tc.cu -- tensor-core (tcgen05 / TMEM) attention over KV8 rows with f32
// queries, the planning of the tensor-core split and the dispatch to the
// kernels of each format (attn_tc_kv8.cu: KV8 with bf16 queries; attn_tc_tq4.cu:
// TQ4).
//
// All heads share one latent cache, so per tile of rows the score (heads x
// rows x 576) and the context (heads x 512 x rows) are dense contractions.
// They run on the 5th-generation tensor cores with f16 operands decoded from
// the quantized rows in shared memory; accumulators live in tensor memory.
// An f32 query is not exact in f16: it enters as an f16 value and an f16
// residual (rows 64..127 of each query chunk), which leaves room for a 4-slot
// ring of decoded chunks only, each chunk decoded once for the score and once
// for the context.
//
// Formulation (transposed, per CTA: one chunk of rows x 64 heads):
//   S_L^T[t][h] = sum_{d<512} c[t][d] q[h][d]     M = 128 rows, N = 64 heads
//   S_R^T[t][h] = sum_{d>=512} c[t][d] q[h][d]    (the rope block, own scale)
//   O^T[d][h]  += sum_t c[t][d] * P^T[t][h]        M = 128 dims (x4), K = rows
// c are the codes' e4m3 values, exact in f16.  The per-row scales stay outside
// the products and are applied by the thread that owns the row: z = sm*(s_L*S_L
// + s_R*S_R), and the context weight is p*s_L ([P2] "What's in it": the row
// scale factors out of both sums).
//
// TMEM (512 columns x 128 lanes of f32): O^T = 4 blocks x 64 columns, S_L^T and
// S_R^T 64 columns each.  A full O for 128 heads x 512 dims would fill all of
// TMEM, which is why a CTA serves 64 heads and two CTAs share each chunk.
//
// Softmax in this layout: a thread owns one row (a TMEM lane) and 32 heads.
// In log2 units, per head: m is a lagged running maximum of the scores z and
// the row sums take p = 2^(z - m); R is the largest y = z + log2 s_L of the
// tiles that set the references, and the context takes the f16 weight
// w = p s_L E with E = 2^(m - R - 3) -- relative to the largest p * s_L of the
// chunk (which weighs 2^-3), so a row whose latent scale is small keeps f16
// precision when it carries the attention.  A tile takes an exact slow path
// (column maxima of z and y over the tile, new m, R, E, rescale of O^T in TMEM
// by (E_new / E_old) 2^(m_old - m_new) and of the row sums by
// 2^(m_old - m_new)) only when some z exceeds m by more than 2^14 or a row's
// latent scale exceeds 3.5 / max_h E (then p <= 2^14, w <= 3.5 * 2^14).  Row sums are accumulated per thread
// and reduced across the 128 rows once per chunk.  The partial state written
// for the merge is the SIMT path's, in natural-log units: (m, sum p, O^T / E).
#include "tc_common.cuh"

#include <algorithm>
#include <math.h>

namespace kvq {
namespace {

constexpr int kRows = 128;      // rows per tile: the score's M, the context's K
constexpr int kHC = 64;         // heads per CTA: the MMA N
constexpr int kWorkers = 256;   // 8 warps: conversion, softmax, epilogue
// + warpgroup 2: one warp whose lane 0 issues every MMA and three idle warps;
// after the prologue it gives its registers to the workers (setmaxnreg)
constexpr int kThreads = kWorkers + 128;
constexpr int kRegsLaunch = 168, kRegsWorker = 232, kRegsMma = 40;
static_assert(kWorkers * kRegsWorker + 128 * kRegsMma <= kThreads * kRegsLaunch, "register split");
constexpr int kSlots = 4;       // f16 staging slots of 128 rows x 64 dims
constexpr uint32_t kSlotBytes = kRows * 128;
// query chunk kc (64 dims): rows 0..63 = f16(q) of the 64 heads, rows 64..127 =
// f16(q - f16(q)), the residual that makes the pair exact to ~22 bits
constexpr uint32_t kQChunkBytes = 2 * kHC * 128;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffSlot = kOffQ + 9 * kQChunkBytes;
constexpr uint32_t kOffP = kOffSlot + kSlots * kSlotBytes;
constexpr uint32_t kOffM = kOffP + kRows * 128;          // m: running max of z per head
constexpr uint32_t kOffR = kOffM + kHC * 4;               // R: reference of z + log2 s_L
constexpr uint32_t kOffE = kOffR + kHC * 4;               // E = 2^(m - R - 3)
constexpr uint32_t kOffF = kOffE + kHC * 4;               // 1 / E
constexpr uint32_t kOffAlpha = kOffF + kHC * 4;           // O^T rescale, then the row sums
constexpr uint32_t kOffAlphaM = kOffAlpha + kHC * 4;      // row-sum rescale
constexpr uint32_t kOffEmax = kOffAlphaM + kHC * 4;       // max E of each 32 heads
constexpr uint32_t kOffBar = kOffEmax + 16;
constexpr uint32_t kOffMisc = kOffBar + 16 * 8;   // abort flag, TMEM base, residual flag, item info, reductions
constexpr uint32_t kSmemUsed = kOffMisc + 160;
constexpr size_t kSmemAlloc = kSmemUsed;          // the base is 1024-aligned (checked at run time)
static_assert(kSmemAlloc <= 232448, "shared memory budget");

// TMEM columns: O^T blocks 0..255; S_L^T 256..383 and S_R^T 384..511, each as
// 64 columns for the f16 query and 64 for its residual
constexpr uint32_t kColO = 0, kColSL = 256, kColSR = 384, kTmemCols = 512;

// mbarriers: slot full (256 worker arrivals), slot empty (MMA commit), score
// done, context done (MMA commits), P^T ready (256 worker arrivals), every MMA
// of the CTA complete (the MMA warp's last commit, also after an abort), and
// one that nothing arrives on (the testing hook's stall)
enum { kBarFull0 = 0, kBarEmpty0 = 4, kBarScore = 8, kBarCtx = 9, kBarP = 10, kBarDone = 11, kBarNever = 12,
       kNumBars = 13 };

using namespace tc;
constexpr uint32_t kIdescScore = idesc_f16(128, kHC, false, false);
constexpr uint32_t kIdescScore2 = idesc_f16(128, 2 * kHC, false, false);
constexpr uint32_t kIdescCtx = idesc_f16(128, kHC, true, true);

// The raw bytes one thread converts for one chunk: dims [64 kc, 64 kc + 64) of
// row (tid / 2), half (tid % 2) of them: 32 bytes (a, b).
struct RawChunk {
    uint4 a, b;
};

// Each tile is consumed as a fixed stream of 17 chunk steps: the 9 score
// chunks (dims 0..575), then the 8 context chunks (dims 0..511).  Loads are
// issued several steps ahead of their use so that DRAM latency overlaps the
// conversion and the MMAs of the steps in between.
constexpr int kStepsPerTile = 17;

__device__ __forceinline__ RawChunk load_step(const uint8_t* __restrict__ codes, int64_t row0, int64_t row1,
                                              int64_t step, int tid) {
    const int64_t tile = step / kStepsPerTile;
    const int j = (int)(step - tile * kStepsPerTile);
    const int kc = j < 9 ? j : j - 9;
    const int64_t row = row0 + tile * kRows + (tid >> 1);
    const int half = tid & 1;
    RawChunk c;
    c.a = c.b = make_uint4(0u, 0u, 0u, 0u);
    if (row < row1) {
        const uint4* src = reinterpret_cast<const uint4*>(codes + row * kMlaD + kc * 64 + half * 32);
        c.a = __ldg(src);
        c.b = __ldg(src + 1);
    }
    return c;
}

// Converts a thread's raw chunk to f16 code values (e4m3 values) in a staging
// slot: row r = one 128-byte swizzled row.  Rows past the tile's end are
// written as zeros.
__device__ __forceinline__ void store_chunk(const RawChunk& c, bool valid, unsigned char* slot, int tid) {
    const int r = tid >> 1, half = tid & 1;
    uint32_t w[16];
    if (valid) {
        const uint32_t in[8] = {c.a.x, c.a.y, c.a.z, c.a.w, c.b.x, c.b.y, c.b.z, c.b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) e4m3x4_to_half2x2(in[i], w[2 * i], w[2 * i + 1]);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = 0u;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(slot + sw128(r, half * 64 + 16 * j)) =
            make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
}

__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(AttnParams p) {
    launch_dependents();
    const int64_t w = blockIdx.x;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = smem_raw;
    unsigned char* sQ = sm + kOffQ;
    unsigned char* sSlot = sm + kOffSlot;
    unsigned char* sP = sm + kOffP;
    float* sM = reinterpret_cast<float*>(sm + kOffM);
    float* sR = reinterpret_cast<float*>(sm + kOffR);
    float* sE = reinterpret_cast<float*>(sm + kOffE);
    float* sF = reinterpret_cast<float*>(sm + kOffF);
    float* sEmax = reinterpret_cast<float*>(sm + kOffEmax);
    float* sAlpha = reinterpret_cast<float*>(sm + kOffAlpha);
    float* sAlphaM = reinterpret_cast<float*>(sm + kOffAlphaM);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
    volatile int* sAbort = reinterpret_cast<volatile int*>(sm + kOffMisc);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + kOffMisc + 4);
    int* sHasLo = reinterpret_cast<int*>(sm + kOffMisc + 8);
    int64_t* sInfo = reinterpret_cast<int64_t*>(sm + kOffMisc + 16);
    float* sRed = reinterpret_cast<float*>(sm + kOffMisc + 48);       // 16 floats

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // item-major linear grid: the CTAs of the first items (the ones with work)
    // are dispatched first; item and head group are re-derived where the
    // epilogue needs them, so that they hold no register over the tile loop
    const int64_t item = w / (p.n_heads / kHC);
    const int group = (int)(w % (p.n_heads / kHC));
    const int hbase = group * kHC;

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
    if (b < 0) return;   // past the last work item
    const int64_t row0 = sInfo[1], row1 = sInfo[2];
    const int n_tiles = (int)((row1 - row0 + kRows - 1) / kRows);

    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(sTmem)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 64) {
        for (int i = 0; i < kNumBars; ++i) {
            const uint32_t count = (i < kBarEmpty0 || i == kBarP) ? (uint32_t)kWorkers : 1u;
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&bars[i])), "r"(count));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *sAbort = 0;
        *sHasLo = 0;
    }
    if (tid < kHC) {
        sM[tid] = -INFINITY;
        sR[tid] = -INFINITY;
        sE[tid] = 0.0f;
        sF[tid] = 0.0f;
    }

    const int wt = tid < kWorkers ? tid : 0;
    int64_t step = 0;
    if (tid == 0) {
        // the first tile's bytes (contiguous rows) into L2
        const int64_t n = min((int64_t)kRows, row1 - row0);
        prefetch_l2(p.codes + row0 * kMlaD, (uint32_t)(n * kMlaD));
    }
    // the raw chunk of step `step`, straight from global memory (L2-prefetched
    // one tile ahead)
#define KVQ_NEXT_CHUNK(dst)                                    \
    do {                                                       \
        dst = load_step(p.codes, row0, row1, step, wt);        \
        ++step;                                                \
    } while (0)

    // The 64 heads of this CTA are 64 x 576 contiguous query values.
    const int64_t qbase = ((int64_t)b * p.n_heads + hbase) * kMlaD;
    constexpr int kQVec = 4;                               // f32 values per 16-byte load
    constexpr int kQLoads = kHC * kMlaD / kQVec;           // 16-byte loads covering the 64 heads
    // largest |q| (with the bound 24 max|q| >= ||q|| that the other kernels
    // use for rotated queries)
    float qmax = 0.0f;
    if (tid < kWorkers) {
        const uint4* qv = reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(p.q) + qbase);
        constexpr int kPer = kQLoads / kWorkers;           // 36: all in flight at once
        static_assert(kQLoads % kWorkers == 0, "query loads per worker");
#pragma unroll 6
        for (int i0 = 0; i0 < kPer; i0 += 6) {
            uint4 w[6];
#pragma unroll
            for (int i = 0; i < 6; ++i) w[i] = __ldg(qv + tid + (i0 + i) * kWorkers);
#pragma unroll
            for (int i = 0; i < 6; ++i) {
                const uint32_t in[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) qmax = fmaxf(qmax, fabsf(__uint_as_float(in[k])));
            }
        }
        qmax = warp_max(qmax);
        if (lane == 0) sRed[warp] = qmax;
    }
    tc_before();
    __syncthreads();
    tc_after();
    float q_max = 0.0f;
    for (int i = 0; i < 8; ++i) q_max = fmaxf(q_max, sRed[i]);
    const float q_bound = 24.0f * q_max;
    int e_q = 0;
    if (q_bound > 0.0f) frexpf(q_bound, &e_q);
    // queries scaled so every f16 element stays below 2^14
    const float q_scale = q_bound > 0.0f ? ldexpf(1.0f, 14 - e_q) : 1.0f;
    const float cz = p.sm_scale * kLog2e * (q_bound > 0.0f ? ldexpf(1.0f, e_q - 14) : 1.0f);
    const uint32_t tmem = *sTmem;

    // queries -> f16 pair (value, residual) in the score's B layout (K-major,
    // 9 chunks of 64 dims x 128 rows)
    int any_lo = 0;
    if (tid < kWorkers) {
        // 8 consecutive dims of one head per step: one 16-byte store of each half
        const uint4* qv = reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(p.q) + qbase);
#pragma unroll 3
        for (int u = tid; u < kHC * kMlaD / 8; u += kWorkers) {
            const uint4 w0 = __ldg(qv + 2 * u), w1 = __ldg(qv + 2 * u + 1);
            const float x[8] = {__uint_as_float(w0.x), __uint_as_float(w0.y), __uint_as_float(w0.z),
                                __uint_as_float(w0.w), __uint_as_float(w1.x), __uint_as_float(w1.y),
                                __uint_as_float(w1.z), __uint_as_float(w1.w)};
            const int e = u * 8, h = e / kMlaD, d = e - h * kMlaD;
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float a0 = x[2 * i] * q_scale, a1 = x[2 * i + 1] * q_scale;
                const __half h0 = __float2half_rn(a0), h1 = __float2half_rn(a1);
                const __half l0 = __float2half_rn(a0 - __half2float(h0));
                const __half l1 = __float2half_rn(a1 - __half2float(h1));
                any_lo |= (__half_as_ushort(l0) | __half_as_ushort(l1)) & 0x7fff;
                hw[i] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
                lw[i] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
            }
            unsigned char* chunk = sQ + (d >> 6) * kQChunkBytes;
            *reinterpret_cast<uint4*>(chunk + sw128(h, (d & 63) * 2)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(chunk + sw128(kHC + h, (d & 63) * 2)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
    }
    if (any_lo) atomicOr(sHasLo, 1);
    fence_async_smem();
    tc_before();
    __syncthreads();
    tc_after();
    // a query exact in f16 needs only the first 64 rows
    const bool has_lo = *sHasLo != 0;

    if (warp >= kWorkers / 32) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsMma));
        // ================= MMA warp: lane 0 issues, the rest idle =================
        if (warp == kWorkers / 32 && lane == 0) {
            const uint32_t id_score = has_lo ? kIdescScore2 : kIdescScore;
            const uint64_t dq0 = umma_desc(smem_u32(sQ), 16, 1024);
            const uint64_t dslot0 = umma_desc(smem_u32(sSlot), 16, 1024);
            const uint64_t dpair0 = umma_desc(smem_u32(sSlot), kSlotBytes, 1024);
            const uint64_t dp = umma_desc(smem_u32(sP), kSlotBytes, 1024);
            constexpr uint64_t kQStep = kQChunkBytes >> 4, kSlotStep = kSlotBytes >> 4;
            uint32_t fills[kSlots] = {0u, 0u, 0u, 0u};
            bool o_init = false, ok = true;
            if (p.stall_polls > 0) ok = mbar_wait(&bars[kBarNever], 0u, sAbort, p.stall_polls);
            for (int tile = 0; tile < n_tiles && ok; ++tile) {
                for (int kc = 0; kc < 9 && ok; ++kc) {
                    const int s = kc & 3;
                    ok = mbar_wait(&bars[kBarFull0 + s], fills[s] & 1, sAbort, p.wait_limit);
                    ++fills[s];
                    tc_after();
                    const uint32_t d = tmem + (kc < 8 ? kColSL : kColSR);
                    const uint64_t a = dslot0 + s * kSlotStep, bq = dq0 + kc * kQStep;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        umma_f16(d, a + 2 * ks, bq + 2 * ks, id_score, (kc == 0 || kc == 8) ? (ks > 0 ? 1u : 0u) : 1u);
                    umma_commit(&bars[kBarEmpty0 + s]);
                    if (kc == 8) umma_commit(&bars[kBarScore]);
                }
                ok = ok && mbar_wait(&bars[kBarP], tile & 1, sAbort, p.wait_limit);
                tc_after();
                for (int db = 0; db < 4 && ok; ++db) {
                    const int s0 = (db & 1) * 2;
                    ok = mbar_wait(&bars[kBarFull0 + s0], fills[s0] & 1, sAbort, p.wait_limit) &&
                         mbar_wait(&bars[kBarFull0 + s0 + 1], fills[s0 + 1] & 1, sAbort, p.wait_limit);
                    ++fills[s0];
                    ++fills[s0 + 1];
                    tc_after();
                    const uint32_t d = tmem + kColO + 64 * db;
                    const uint64_t a = dpair0 + s0 * kSlotStep;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        umma_f16(d, a + 128 * ks, dp + 128 * ks, kIdescCtx, (o_init || ks > 0) ? 1u : 0u);
                    umma_commit(&bars[kBarEmpty0 + s0]);
                    umma_commit(&bars[kBarEmpty0 + s0 + 1]);
                    if (db == 3) umma_commit(&bars[kBarCtx]);
                }
                o_init = true;
            }
            umma_commit(&bars[kBarDone]);
        }
        return;
    }

    // ================= workers: conversion, softmax, epilogue =================
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsWorker));
    const int srow = 32 * (warp & 3) + lane;   // TMEM lane owned in the softmax
    const int hq = warp >> 2;                   // heads 32 hq .. 32 hq + 31
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    float lsum[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) lsum[j] = 0.0f;
    uint32_t uses[kSlots] = {0u, 0u, 0u, 0u};
    bool o_init = false;
    int tile = 0;
    float s_lim = 0.0f;   // latent scales above this take the exact path (3.5 / max_h E)

    for (; tile < n_tiles; ++tile) {
        if (worker_any(*sAbort != 0)) break;
        const int64_t t0 = row0 + (int64_t)tile * kRows;
        const int nt = (int)min((int64_t)kRows, row1 - t0);
        const bool valid = (tid >> 1) < nt;
        if (tid == 0 && t0 + kRows < row1) {
            const int64_t n = min((int64_t)kRows, row1 - (t0 + kRows));
            prefetch_l2(p.codes + (t0 + kRows) * kMlaD, (uint32_t)(n * kMlaD));
        }
        // this thread's softmax row scales (used after the score chunks)
        float my_sl = 0.0f, my_sr = 0.0f;
        if (srow < nt) {
            const int64_t r = t0 + srow;
            my_sl = p.scales[r * p.n_blocks];
            my_sr = p.scales[r * p.n_blocks + (p.n_blocks - 1)];
        }
        // ---- score chunks: 9 chunks of 64 dims (8 latent, 1 rope) ----
        for (int kc = 0; kc < 9; ++kc) {
            const int s = kc & 3;
            if (uses[s] > 0) mbar_wait(&bars[kBarEmpty0 + s], (uses[s] - 1) & 1, sAbort, p.wait_limit);
            RawChunk rc;
            KVQ_NEXT_CHUNK(rc);
            store_chunk(rc, valid, sSlot + s * kSlotBytes, tid);
            fence_async_smem();
            mbar_arrive(&bars[kBarFull0 + s]);
            ++uses[s];
        }
        // ---- softmax of the tile (thread = row, 32 heads) ----
        mbar_wait(&bars[kBarScore], tile & 1, sAbort, p.wait_limit);
        if (tile > 0) mbar_wait(&bars[kBarCtx], (tile - 1) & 1, sAbort, p.wait_limit);
        tc_after();
        float z[32];
        {
            const float a = my_sl * cz, bb = my_sr * cz;
            const bool row_ok = srow < nt;
            // 16 columns at a time keeps the peak register count under the cap
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t sl[16], sr[16];
                tmem_ld16(tmem + lane_base + kColSL + 32 * hq + 16 * c, sl);
                tmem_ld16(tmem + lane_base + kColSR + 32 * hq + 16 * c, sr);
                tmem_wait_ld();
                float fl[16], fr[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    fl[j] = __uint_as_float(sl[j]);
                    fr[j] = __uint_as_float(sr[j]);
                }
                if (has_lo) {
                    tmem_ld16(tmem + lane_base + kColSL + kHC + 32 * hq + 16 * c, sl);
                    tmem_ld16(tmem + lane_base + kColSR + kHC + 32 * hq + 16 * c, sr);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        fl[j] += __uint_as_float(sl[j]);
                        fr[j] += __uint_as_float(sr[j]);
                    }
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) z[16 * c + j] = row_ok ? fmaf(fl[j], a, fr[j] * bb) : -INFINITY;
            }
        }
        bool flag = my_sl > s_lim;
#pragma unroll
        for (int j = 0; j < 32; ++j) flag |= z[j] > sM[32 * hq + j] + 14.0f;
        if (worker_any(flag)) {
            const float ls = my_sl > 0.0f ? __log2f(my_sl) : -INFINITY;   // -inf: an inert latent block
            // exact column maxima of z and of y = z + log2 s_L over the tile,
            // new running maxima, rescale factors
            float* zbuf = reinterpret_cast<float*>(sSlot);                   // 128 x 64 f32, slots 0-1
            float* ybuf = reinterpret_cast<float*>(sSlot + 2 * kSlotBytes);  // slots 2-3 (all idle now)
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                zbuf[srow * kHC + 32 * hq + j] = z[j];
                ybuf[srow * kHC + 32 * hq + j] = z[j] + ls;
            }
            worker_sync();
            {
                const int col = tid & (kHC - 1), quarter = tid >> 6;
                float cm = -INFINITY, cy = -INFINITY;
#pragma unroll 8
                for (int r = 32 * quarter; r < 32 * quarter + 32; ++r) {
                    cm = fmaxf(cm, zbuf[r * kHC + col]);
                    cy = fmaxf(cy, ybuf[r * kHC + col]);
                }
                float* part = reinterpret_cast<float*>(sP);   // P^T is rewritten after this
                part[quarter * kHC + col] = cm;
                part[4 * kHC + quarter * kHC + col] = cy;
                worker_sync();
                if (tid < kHC) {
                    const float* py = part + 4 * kHC;
                    const float c4 = fmaxf(fmaxf(part[tid], part[kHC + tid]), fmaxf(part[2 * kHC + tid], part[3 * kHC + tid]));
                    const float y4 = fmaxf(fmaxf(py[tid], py[kHC + tid]), fmaxf(py[2 * kHC + tid], py[3 * kHC + tid]));
                    const float mo = sM[tid], mn = fmaxf(mo, c4);
                    const float ro = sR[tid], rn = fmaxf(ro, y4);
                    const float dn = fminf(mn - rn - 3.0f, 120.0f), d_old = fminf(mo - ro - 3.0f, 120.0f);
                    sAlphaM[tid] = mo == -INFINITY ? 0.0f : exp2f(mo - mn);
                    sAlpha[tid] = ro == -INFINITY ? 0.0f : exp2f(dn - d_old + (mo - mn));
                    sM[tid] = mn;
                    sR[tid] = rn;
                    const float e = rn == -INFINITY ? 0.0f : exp2f(dn);   // R = -inf: only inert latent blocks
                    sE[tid] = e;
                    sF[tid] = rn == -INFINITY ? 0.0f : exp2f(-dn);
                    const float em = warp_max(e);
                    if ((tid & 31) == 0) sEmax[tid >> 5] = em;
                    if (tile > 0 && tid == 0) atomicAdd(p.exact_count, 1u);
                }
            }
            worker_sync();
            {
                const float em = fmaxf(sEmax[0], sEmax[1]);
                s_lim = em > 0.0f ? 3.5f / em : 0.0f;
            }
            if (o_init) {
#pragma unroll 1
                for (int bi = 0; bi < 2; ++bi)
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t ta = tmem + lane_base + kColO + 64 * (2 * hq + bi) + 16 * c;
                        uint32_t v[16];
                        tmem_ld16(ta, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * sAlpha[16 * c + j]);
                        tmem_st16(ta, v);
                    }
                tmem_wait_st();
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) lsum[j] *= sAlphaM[32 * hq + j];
        }
        {
            // row-sum weights p = 2^(z - m), f16 context weights w = p s_L E
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float p0 = exp2f(z[j] - sM[32 * hq + j]);
                const float p1 = exp2f(z[j + 1] - sM[32 * hq + j + 1]);
                lsum[j] += p0;
                lsum[j + 1] += p1;
                const __half2 h2 = __floats2half2_rn(p0 * sE[32 * hq + j] * my_sl, p1 * sE[32 * hq + j + 1] * my_sl);
                pk[j / 2] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            // slow path: every column max must be read before P^T overwrites the partials
            worker_sync();
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<uint4*>(sP + sw128(srow, 64 * hq + 16 * i)) =
                    make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
        fence_async_smem();
        tc_before();
        mbar_arrive(&bars[kBarP]);
        // ---- context chunks: 4 blocks of 128 dims (2 chunks each) ----
        for (int db = 0; db < 4; ++db) {
            const int s0 = (db & 1) * 2;
            if (uses[s0] > 0) mbar_wait(&bars[kBarEmpty0 + s0], (uses[s0] - 1) & 1, sAbort, p.wait_limit);
            if (uses[s0 + 1] > 0) mbar_wait(&bars[kBarEmpty0 + s0 + 1], (uses[s0 + 1] - 1) & 1, sAbort, p.wait_limit);
            RawChunk r0c, r1c;
            KVQ_NEXT_CHUNK(r0c);
            KVQ_NEXT_CHUNK(r1c);
            store_chunk(r0c, valid, sSlot + s0 * kSlotBytes, tid);
            store_chunk(r1c, valid, sSlot + (s0 + 1) * kSlotBytes, tid);
            fence_async_smem();
            mbar_arrive(&bars[kBarFull0 + s0]);
            mbar_arrive(&bars[kBarFull0 + s0 + 1]);
            ++uses[s0];
            ++uses[s0 + 1];
        }
        o_init = true;
    }
#undef KVQ_NEXT_CHUNK

    // ---- epilogue: row sums, O^T -> partial state ----
    {
        // bounded, and not cut short by the abort flag: TMEM is released only
        // after the MMAs in flight have completed
        volatile int never = 0;
        if (!mbar_wait(&bars[kBarDone], 0u, &never)) *sAbort = 1;
    }
    tc_after();
    {
        float* lbuf = reinterpret_cast<float*>(sSlot);
        worker_sync();   // every worker is past its last slot use
#pragma unroll
        for (int j = 0; j < 32; ++j) lbuf[srow * kHC + 32 * hq + j] = lsum[j];
        worker_sync();
        const int col = tid & (kHC - 1), quarter = tid >> 6;
        float l = 0.0f;
#pragma unroll 8
        for (int r = 32 * quarter; r < 32 * quarter + 32; ++r) l += lbuf[r * kHC + col];
        float* part = reinterpret_cast<float*>(sP);
        part[quarter * kHC + col] = l;
        worker_sync();
        if (tid < kHC) sAlpha[tid] = (part[tid] + part[kHC + tid]) + (part[2 * kHC + tid] + part[3 * kHC + tid]);
        worker_sync();
    }
    const bool aborted = worker_any(*sAbort != 0 || tile < n_tiles);
    if (aborted) {
        if (tid == 0) set_err(p.err, KVQ_ERR_TIMEOUT);
    } else {
        const int64_t unit = blockIdx.x;
        const int64_t item = unit / (p.n_heads / kHC);
        const int hbase = (int)(unit % (p.n_heads / kHC)) * kHC;
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
                    p.ws_o[(item * p.n_heads + h) * kMlaDV + dim] =
                        o_init ? __uint_as_float(v[j]) * sF[32 * c + j] : 0.0f;
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
    worker_sync();
    tc_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

cudaError_t launch_tc_kv8_f32(const AttnParams& p, int64_t grid_x, int groups, cudaStream_t stream) {
    // the workers' setmaxnreg.inc waits for registers the other warpgroup
    // released: launch only if the split adds up against the launch's count
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, attn_tc_kernel);
    if (e != cudaSuccess) return e;
    if (kWorkers * kRegsWorker + 128 * kRegsMma > kThreads * fa.numRegs) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
    if (e != cudaSuccess) return e;
    attn_tc_kernel<<<dim3((unsigned)(grid_x * groups)), kThreads, kSmemAlloc, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(const kvq_mla_layout& L, int32_t n_heads) {
    (void)L;
    return n_heads > 0 && n_heads % kHC == 0;
}

AttnPlan plan_decode_tc(kvq_format fmt, int32_t batch, int32_t n_heads, int64_t max_total_rows, int waves) {
    AttnPlan pl{};
    pl.heads_per_cta = (fmt == KVQ_TQ4 || fmt == KVQ_PQ4) ? kHC / 2 : kHC;
    const int64_t groups = std::max<int64_t>(1, n_heads / pl.heads_per_cta);
    const int64_t target_items = std::max<int64_t>(1, 152 / groups);
    int64_t chunk = (std::max<int64_t>(max_total_rows, 1) + target_items - 1) / target_items;
    chunk = std::max<int64_t>(kRows, (chunk + kRows - 1) / kRows * kRows);
    pl.chunk = chunk;   // used as is for more than kBalanceSeqs sequences
    pl.max_rows = max_total_rows;
    // A chunk fixed here is enough when it guarantees one wave whatever the
    // split of the rows into `batch` sequences (at most R / C + batch items)
    // at little more than the ideal R / S rows per item: the CTAs then skip
    // the device-side search (8 x 4096 KV8 rows: 512 either way).
    if (target_items > batch) {
        int64_t c1 = (std::max<int64_t>(max_total_rows, 1) + (target_items - batch) - 1) / (target_items - batch);
        c1 = std::max<int64_t>(kRows, (c1 + kRows - 1) / kRows * kRows);
        if (c1 <= chunk + chunk / 4) {
            pl.chunk = c1;
            pl.wave_items = 0;
            pl.max_waves = 1;
            pl.max_items = (max_total_rows + c1 - 1) / c1 + batch;
            return pl;
        }
    }
    pl.wave_items = target_items;
    pl.max_waves = std::max(1, waves);
    if (batch <= kBalanceSeqs) {
        // the balanced chunk yields at most max_waves * target * ceil(n / target)
        // items, and at most one per tile plus one per sequence
        const int64_t per_wave = target_items * std::max<int64_t>(1, (batch + target_items - 1) / target_items);
        pl.max_items = std::min<int64_t>(pl.max_waves * per_wave,
                                         (max_total_rows + kBalanceGranule - 1) / kBalanceGranule + batch);
    } else {
        pl.max_items = (max_total_rows + chunk - 1) / chunk + batch;
    }
    return pl;
}

cudaError_t launch_attn_tc(kvq_format fmt, const kvq_mla_layout& L, const void* q, kvq_dtype qdt, int32_t n_seq,
                           int32_t n_heads, const uint8_t* codes, const float* scales, const int64_t* cu_seqlens,
                           int64_t prefill_past, const AttnPlan& plan, float sm_scale, float* out, void* workspace,
                           cudaStream_t stream, const int64_t* sel, int64_t pool_rows) {
    if (n_seq == 0 || n_heads == 0) return cudaSuccess;
    AttnParams p = make_attn_params(fmt, L, q, n_seq, n_heads, codes, scales, cu_seqlens, prefill_past, plan,
                                    sm_scale, workspace);
    p.sel = sel;
    p.pool_rows = pool_rows;
    // only the KV8 / bf16-query kernel reads rows through an index table
    if (sel && !(fmt == KVQ_KV8 && qdt == KVQ_BF16)) return cudaErrorNotSupported;
    const int groups = n_heads / kHC;
    timing_mark(stream, 0);
    cudaError_t e;
    if (fmt == KVQ_KV8)
        e = qdt == KVQ_BF16 ? launch_attn_tc_kv8_bf16(p, plan.max_items, groups, stream)
                            : launch_tc_kv8_f32(p, plan.max_items, groups, stream);
    else
        e = launch_attn_tc_tq4(p, qdt == KVQ_BF16, fmt == KVQ_PQ4, plan.max_items, n_heads, stream);
    if (e != cudaSuccess) return e;
    return launch_attn_merge(fmt, p, out, stream);
}

cudaError_t launch_attn_tc_kv8_append(const kvq_mla_layout& L, const float* x_new, const int64_t* dst_rows,
                                      const void* q, int32_t n_seq, int32_t n_heads, uint8_t* codes, float* scales,
                                      const int64_t* cu_seqlens, const AttnPlan& plan, float sm_scale, float* out,
                                      void* workspace, cudaStream_t stream) {
    if (n_seq == 0 || n_heads == 0) return cudaSuccess;
    AttnParams p = make_attn_params(KVQ_KV8, L, q, n_seq, n_heads, codes, scales, cu_seqlens, -1, plan, sm_scale,
                                    workspace);
    p.x_new = x_new;
    p.dst_rows = dst_rows;
    p.codes_out = codes;
    p.scales_out = scales;
    p.bd0 = L.block_dim[0];
    p.bd1 = L.n_blocks > 1 ? L.block_dim[1] : 0;
    timing_mark(stream, 0);
    const cudaError_t e = launch_attn_tc_kv8_bf16_append(p, plan.max_items, n_heads / kHC, stream);
    if (e != cudaSuccess) return e;
    return launch_attn_merge(KVQ_KV8, p, out, stream);
}

}  // namespace kvq
