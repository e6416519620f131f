// attn_tc_kv8.cu -- tensor-core attention over KV8 rows for bf16 queries, with
// every quantized chunk decoded once per tile.
//
// Same transposed formulation as the general tensor-core kernel (one chunk of
// rows x 64 heads per CTA; S^T = C Q^T with M = 128 rows, N = 64 heads;
// O^T += C^T P^T with M = 128 dims, K = rows), specialised for the case the
// decode benchmark runs: e4m3 codes and a bf16 query.
//
// A bf16 query times a power of two is exact in f16 (over the range that can
// matter), so each 64-dim query chunk needs only its 64 head rows: the query
// takes 72 KB of shared memory.  That leaves room for all 9 f16 chunks of a
// 128-row tile (144 KB).  Each chunk is decoded once and read twice by the
// tensor cores: as the K-major A operand of the score and, for the 8 latent
// chunks, as the MN-major A operand of the context.  P^T takes the rope
// chunk's slot once the score of the tile has completed.
//
// Pipeline per tile t (8 worker warps, 1 MMA warp; the MMA warp's warpgroup,
// padded with three idle warps, hands its registers to the workers):
//   workers: decode the tile in three groups -- chunks 0-3 (row bytes
//            0..255), chunks 4-7 (256..511), the rope chunk 8 (512..575) --
//            each as soon as the context of tile t-1 has released its slots,
//            then the softmax of tile t (thread = row, 32 heads), then P^T.
//            The raw bytes of tile t+1 are loaded into registers during tile t,
//            all three groups before the softmax (they stay live across it in
//            the workers' 232 registers).
//   MMA:     score of tile t group by group, commit; once P^T(t) is written,
//            the 4 context blocks, each committed to its slot pair's barrier.
// The decode of tile t+1 thus overlaps the context MMAs of tile t, and the
// score MMAs of tile t+1 follow the decode group by group.
//
// Loads are laid out so that each warp instruction reads whole rows: in groups
// A and B the 256 contiguous bytes of two rows (lanes alternate between them
// in fours), in group C 8 rows of 64 bytes.
//
// Reductions over the 128 rows of a tile (column max in the softmax's exact
// path, the row sums at the end) run as a 31-shuffle transpose-reduce within
// each warp plus one 4-way combine in shared memory.
//
// The row scales factor out of both sums ([P2] "What's in it"; [P1] "Ready for
// review" comment, finding 2): z = sm * (s_L * S_L + s_R * S_R), and the
// context weight of row t is p_t * s_L,t.  In log2 units, per head: m is a
// lagged running maximum of the scores and the row sums take p = 2^(z - m);
// R is the largest y = z + log2 s_L of the tiles that set the references, and
// the context takes the f16 weight w = p * s_L * E with E = 2^(m - R - 3):
// weights relative to the largest p * s_L (which weighs 2^-3), so rows whose
// latent scale is small keep f16 precision whenever they carry the attention.
// A tile takes the exact path when a score passes m by more than 2^14 or a
// row's latent scale passes 3.5 / max_h E (about 28 times the scale of the
// row that set a head's reference); below both, p <= 2^14 and
// w <= 3.5 * 2^14 < 65504, the f16 maximum.  The exact path takes the column
// maxima of z and y over the tile, sets m, R and E, and rescales O^T in TMEM
// by (E_new / E_old) 2^(m_old - m_new) and the row sums by 2^(m_old - m_new).
// The partial state is (m, sum p, O^T / E).
#include "tc_common.cuh"

#include <math.h>

namespace kvq {
namespace {
using namespace tc;

constexpr int kRows = 128;      // rows per tile
constexpr int kHC = 64;         // heads per CTA
constexpr int kWorkers = 256;
// warpgroup 2 holds the MMA-issuing warp and three idle warps: after the
// prologue it gives its registers to the eight worker warps (setmaxnreg), so
// the tile loop runs with kRegsWorker registers per thread instead of the
// 168 a 384-thread launch allows
constexpr int kThreads = kWorkers + 128;
constexpr int kRegsLaunch = 168, kRegsWorker = 232, kRegsMma = 40;
static_assert(kWorkers * kRegsWorker + 128 * kRegsMma <= kThreads * kRegsLaunch, "register split");
constexpr int kChunks = 9;      // 64-dim chunks of a row: 8 latent + 1 rope
constexpr int kRope = 8;        // the rope chunk's slot, reused for P^T
constexpr uint32_t kSlotBytes = kRows * 128;       // 128 rows x 64 f16
constexpr uint32_t kQChunkBytes = kHC * 128;       // 64 heads x 64 f16
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffSlot = kOffQ + kChunks * kQChunkBytes;
constexpr uint32_t kOffM = kOffSlot + kChunks * kSlotBytes;   // m: running max of z per head
constexpr uint32_t kOffR = kOffM + kHC * 4;                    // R: reference of z + log2 s_L
constexpr uint32_t kOffE = kOffR + kHC * 4;                    // E = 2^(m - R - kHeadroom)
constexpr uint32_t kOffF = kOffE + kHC * 4;                    // 1 / E
constexpr uint32_t kOffAlpha = kOffF + kHC * 4;                // O^T rescale, then the row sums
constexpr uint32_t kOffAlphaM = kOffAlpha + kHC * 4;           // row-sum rescale 2^(m_old - m_new)
constexpr uint32_t kOffEmax = kOffAlphaM + kHC * 4;            // max E of each 32 heads
constexpr uint32_t kOffRed = kOffEmax + 16;   // 2 x 4 quadrants x 64 heads of f32
constexpr uint32_t kOffBar = kOffRed + 2 * 4 * kHC * 4;
constexpr uint32_t kOffMisc = kOffBar + 16 * 8;      // abort flag, TMEM base, item info
constexpr uint32_t kOffNew = kOffMisc + 32;          // appended row: 576 codes, 2 scales, row index
constexpr uint32_t kOffRowIdx = kOffNew + 576 + 16;   // gather: pool rows of 2 tiles (int64)
constexpr uint32_t kSmemUsed = kOffRowIdx + 2 * kRows * 8;
static_assert(kOffSlot % 1024 == 0, "swizzled operands need 1024-byte alignment");
static_assert(kSmemUsed <= 232448, "shared memory budget");

// TMEM columns: O^T blocks 0..255, S_L^T 256..319, S_R^T 320..383
constexpr uint32_t kColO = 0, kColSL = 256, kColSR = 320, kTmemCols = 512;

// mbarriers: decode group g stored (256 arrivals; A = chunks 0-3, B = 4-7,
// C = the rope chunk), slot pair db released by the context (MMA commit; the
// last pair also releases the rope/P^T slot), score complete (MMA commit), P^T
// written (256 arrivals), every MMA of the CTA complete (the MMA warp's last
// commit, also after an abort), and one that nothing arrives on (the testing
// hook's stall)
enum { kBarFull0 = 0, kBarFree0 = 3, kBarScore = 7, kBarP = 8, kBarDone = 9, kBarNever = 10, kNumBars = 11 };

// A score may pass m by up to 2^14 without the exact path (p <= 2^14), a
// latent scale up to 3.5 / max_h E (w <= 3.5 * 2^14); the largest p * s_L of a
// reference tile weighs 2^-kHeadroom; log2 E is capped so that E and 1 / E
// stay finite in f32 (any E is exact: the epilogue divides it out).
constexpr float kLagLog2 = 14.0f;
constexpr float kScaleLim = 3.5f;
constexpr float kHeadroom = 3.0f;
constexpr float kLogEmax = 120.0f;

constexpr uint32_t kIdescScore = idesc_f16(128, kHC, false, false);
constexpr uint32_t kIdescCtx = idesc_f16(128, kHC, true, true);

// A worker's raw share of a tile.  Groups A and B: 8 pieces of 16 bytes, piece
// i at row 2 (warp + 8 i) + (lane / 4) % 2, bytes 64 (lane / 8) + 16 (lane % 4)
// of the group's 256 (so the thread always serves chunk 4 g + lane / 8, 16
// dims at 16 (lane % 4)).  A 16-byte shared-memory store is served 8 lanes at
// a time: lanes 8p .. 8p + 3 and 8p + 4 .. 8p + 7 write the same chunk of two
// adjacent rows, whose 128-byte swizzle phases differ in their low bit, so the
// 8 lanes cover 8 distinct 16-byte units (one row across two chunks hit 4
// units twice).  Group C: 2 pieces, piece i at row (tid + 256 i) / 4, bytes
// 16 (tid % 4) of the rope chunk.
struct RawGroup {
    uint4 v[8];
};
struct RawRope {
    uint4 v[2];
};

// Pool row `rn` (an appended row, or -1) is read from its shared-memory copy
// `snew` instead of global memory.
template <bool APPEND>
__device__ __forceinline__ uint4 load16(const uint8_t* __restrict__ codes, int64_t row, int byte, int64_t rn,
                                        const unsigned char* snew) {
    if (APPEND && row == rn) return *reinterpret_cast<const uint4*>(snew + byte);
    return __ldg(reinterpret_cast<const uint4*>(codes + row * kMlaD + byte));
}
// Pool row of tile row `row`: contiguous rows, or (gather) the tile's index table.
template <bool GATHER>
__device__ __forceinline__ int64_t pool_row(int64_t t0, int row, const int64_t* prow) {
    return GATHER ? prow[row] : t0 + row;
}
template <bool APPEND, bool GATHER>
__device__ __forceinline__ void load_group(RawGroup& r, const uint8_t* __restrict__ codes, int64_t t0, int nt, int g,
                                           int warp, int lane, int64_t rn, const unsigned char* snew,
                                           const int64_t* prow) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = 2 * (warp + 8 * i) + ((lane >> 2) & 1);
        r.v[i] = row < nt ? load16<APPEND>(codes, pool_row<GATHER>(t0, row, prow),
                                           256 * g + 64 * (lane >> 3) + 16 * (lane & 3), rn, snew)
                          : make_uint4(0u, 0u, 0u, 0u);
    }
}
template <bool APPEND, bool GATHER>
__device__ __forceinline__ void load_rope(RawRope& r, const uint8_t* __restrict__ codes, int64_t t0, int nt, int tid,
                                          int64_t rn, const unsigned char* snew, const int64_t* prow) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int u = tid + kWorkers * i, row = u >> 2;
        r.v[i] = row < nt ? load16<APPEND>(codes, pool_row<GATHER>(t0, row, prow), 512 + 16 * (u & 3), rn, snew)
                          : make_uint4(0u, 0u, 0u, 0u);
    }
}
// The same three groups for a full tile of contiguous rows that does not hold
// the appended row: no per-piece row tests, one base address per group.
__device__ __forceinline__ void load_tile_full(RawGroup& a, RawGroup& b, RawRope& c,
                                               const uint8_t* __restrict__ codes, int64_t t0, int warp, int lane,
                                               int tid) {
    const uint8_t* ga = codes + (t0 + 2 * warp + ((lane >> 2) & 1)) * kMlaD + 64 * (lane >> 3) + 16 * (lane & 3);
#pragma unroll
    for (int i = 0; i < 8; ++i) a.v[i] = __ldg(reinterpret_cast<const uint4*>(ga + i * 16 * kMlaD));
#pragma unroll
    for (int i = 0; i < 8; ++i) b.v[i] = __ldg(reinterpret_cast<const uint4*>(ga + i * 16 * kMlaD + 256));
    const uint8_t* gc = codes + (t0 + (tid >> 2)) * kMlaD + 512 + 16 * (tid & 3);
#pragma unroll
    for (int i = 0; i < 2; ++i) c.v[i] = __ldg(reinterpret_cast<const uint4*>(gc + i * (kWorkers / 4) * kMlaD));
}

// 16 e4m3 codes -> 16 f16 values (exact) at byte offset `b` of swizzled row `row`.
__device__ __forceinline__ void store16(unsigned char* slot, const uint4& c, int row, int b) {
    const uint32_t in[4] = {c.x, c.y, c.z, c.w};
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) e4m3x4_to_half2x2(in[i], w[2 * i], w[2 * i + 1]);
    *reinterpret_cast<uint4*>(slot + sw128(row, b)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(slot + sw128(row, b + 16)) = make_uint4(w[4], w[5], w[6], w[7]);
}

// In-warp transpose-reduce: on entry each lane holds 32 values (columns
// 0..31 of its row); on return lane j's v[0] is the reduction of column j over
// the 32 lanes.  31 shuffles.
template <bool MAX>
__device__ __forceinline__ float warp_columns(float (&v)[32], int lane) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = upper ? v[i] : v[i + s];
            const float keep = upper ? v[i + s] : v[i];
            const float got = __shfl_xor_sync(kFull, send, s);
            v[i] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
    return v[0];
}

// The exact path of a tile (see the top of the file), by every worker thread
// with its row's scores in TMEM: column maxima of z and of y = z + log2 s_L
// over the tile (16 heads at a time, straight from TMEM), new m, R and E per
// head (sAlphaM: the row-sum rescale), the rescale of O^T in TMEM after the
// first tile.  Out of line: the path is rare, and kept out of the tile loop it
// leaves the loop's registers alone.
__device__ __noinline__ void exact_path(unsigned char* sm, uint32_t tmem, uint32_t lane_base, int hq, bool row_ok,
                                        float za, float zb, float my_sl, int lane, int warp, int tid, int t,
                                        uint32_t* exact_count) {
    float* sM = reinterpret_cast<float*>(sm + kOffM);
    float* sR = reinterpret_cast<float*>(sm + kOffR);
    float* sE = reinterpret_cast<float*>(sm + kOffE);
    float* sF = reinterpret_cast<float*>(sm + kOffF);
    float* sAlpha = reinterpret_cast<float*>(sm + kOffAlpha);
    float* sAlphaM = reinterpret_cast<float*>(sm + kOffAlphaM);
    float* sEmax = reinterpret_cast<float*>(sm + kOffEmax);
    float* sRed = reinterpret_cast<float*>(sm + kOffRed);
            // exact column maxima of z and of y = z + log2 s_L over the tile
            {
                float v[32];
                auto load_v = [&](float add) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t s16[16];
                        tmem_ld16(tmem + lane_base + kColSR + 32 * hq + 16 * c, s16);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[16 * c + j] = __uint_as_float(s16[j]) * zb;
                        tmem_ld16(tmem + lane_base + kColSL + 32 * hq + 16 * c, s16);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            v[16 * c + j] = row_ok ? fmaf(__uint_as_float(s16[j]), za, v[16 * c + j]) + add : -INFINITY;
                    }
                };
                load_v(0.0f);
                sRed[(warp & 3) * kHC + 32 * hq + lane] = warp_columns<true>(v, lane);
                load_v(my_sl > 0.0f ? __log2f(my_sl) : -INFINITY);   // -inf: an inert latent block
                sRed[4 * kHC + (warp & 3) * kHC + 32 * hq + lane] = warp_columns<true>(v, lane);
            }
            worker_sync();
            if (tid < kHC) {
                const float* ry = sRed + 4 * kHC;
                const float c4 = fmaxf(fmaxf(sRed[tid], sRed[kHC + tid]), fmaxf(sRed[2 * kHC + tid], sRed[3 * kHC + tid]));
                const float y4 = fmaxf(fmaxf(ry[tid], ry[kHC + tid]), fmaxf(ry[2 * kHC + tid], ry[3 * kHC + tid]));
                const float mo = sM[tid], mn = fmaxf(mo, c4);
                const float ro = sR[tid], rn2 = fmaxf(ro, y4);
                // log2 E = m - R - kHeadroom (capped); R = -inf: every row so far
                // has an inert latent block (E = 0 keeps their weights 0 and
                // makes any later latent scale take this path)
                const float dn = fminf(mn - rn2 - kHeadroom, kLogEmax), d_old = fminf(mo - ro - kHeadroom, kLogEmax);
                sAlphaM[tid] = mo == -INFINITY ? 0.0f : ex2(mo - mn);
                // O^T holds sum p s_L E c: rescaled by (E_new / E_old) 2^(m_old - m_new)
                sAlpha[tid] = ro == -INFINITY ? 0.0f : ex2(dn - d_old + (mo - mn));
                sM[tid] = mn;
                sR[tid] = rn2;
                const float e = rn2 == -INFINITY ? 0.0f : ex2(dn);
                sE[tid] = e;
                sF[tid] = rn2 == -INFINITY ? 0.0f : ex2(-dn);
                const float em = warp_max(rn2 == -INFINITY ? INFINITY : e);
                if (lane == 0) sEmax[tid >> 5] = em;
                if (t > 0 && tid == 0) atomicAdd(exact_count, 1u);
            }
            worker_sync();
            if (t > 0) {
                // O^T is stable: the score commit of this tile follows every
                // context MMA of the previous one
#pragma unroll 1
                for (int bi = 0; bi < 2; ++bi)
#pragma unroll 1
                    for (int c = 0; c < 2; ++c) {
                        const uint32_t ta = tmem + lane_base + kColO + 64 * (2 * hq + bi) + 32 * c;
                        uint32_t o[32];
                        tmem_ld32(ta, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * sAlpha[32 * c + j]);
                        tmem_st32(ta, o);
                    }
                tmem_wait_st();
            }
}

template <bool APPEND, bool GATHER>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kv8_kernel(AttnParams p) {
    const int64_t wl = p.wait_limit;
    launch_dependents();
    const int64_t w = blockIdx.x;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = smem_raw;
    unsigned char* sQ = sm + kOffQ;
    unsigned char* sSlot = sm + kOffSlot;
    unsigned char* sP = sSlot + kRope * kSlotBytes;
    float* sM = reinterpret_cast<float*>(sm + kOffM);
    float* sR = reinterpret_cast<float*>(sm + kOffR);
    float* sE = reinterpret_cast<float*>(sm + kOffE);
    float* sF = reinterpret_cast<float*>(sm + kOffF);
    float* sAlpha = reinterpret_cast<float*>(sm + kOffAlpha);
    float* sAlphaM = reinterpret_cast<float*>(sm + kOffAlphaM);
    float* sEmax = reinterpret_cast<float*>(sm + kOffEmax);
    float* sRed = reinterpret_cast<float*>(sm + kOffRed);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
    volatile int* sAbort = reinterpret_cast<volatile int*>(sm + kOffMisc);
    uint32_t* sTmem = reinterpret_cast<uint32_t*>(sm + kOffMisc + 4);
    int64_t* sInfo = reinterpret_cast<int64_t*>(sm + kOffMisc + 8);
    unsigned char* sNew = sm + kOffNew;                       // appended row's codes
    float* sNewScale = reinterpret_cast<float*>(sm + kOffNew + 576);
    int64_t* sNewRow = reinterpret_cast<int64_t*>(sm + kOffNew + 584);
    int64_t* sRowIdx = reinterpret_cast<int64_t*>(sm + kOffRowIdx);   // gather: [2][kRows]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // item-major linear grid: the CTAs of the first items (the ones with work)
    // are dispatched first; item and head group are re-derived where the
    // epilogue needs them, so that they hold no register over the tile loop
    const int64_t item = w / (p.n_heads / kHC);
    const int group = (int)(w % (p.n_heads / kHC));
    const int hbase = group * kHC;

    if (tid == 32 && p.prefill_past < 0) {
        // a decode batch's queries into L2, a slice per CTA, while warp 0
        // looks up the item: the query loads after the lookup then hit L2
        // (not for prefill, whose CTAs each read one token's query, nor for
        // batches whose queries would crowd the cache)
        const uint64_t total = (uint64_t)p.n_seq * p.n_heads * kMlaD * 2;   // bf16, a multiple of 16
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
            const uint32_t count = (i < kBarFree0 || i == kBarP) ? (uint32_t)kWorkers : 1u;
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
        if (tid < kHC / 32) sEmax[tid] = INFINITY;
    }
    if (!GATHER && tid == 0) {
        const int64_t n = min((int64_t)kRows, row1 - row0);
        prefetch_l2(p.codes + row0 * kMlaD, (uint32_t)(n * kMlaD));
        // the second tile too: the loop keeps the L2 prefetch two tiles ahead
        if (row0 + kRows < row1)
            prefetch_l2(p.codes + (row0 + kRows) * kMlaD, (uint32_t)(min((int64_t)kRows, row1 - row0 - kRows) * kMlaD));
    }
    if (GATHER && tid < kRows) sRowIdx[tid] = row0 + tid < row1 ? gather_row(p, row0 + tid) : 0;

    // ---- appended row: the MMA warp (idle until the first score) encodes it
    // into shared memory; the group-0 CTA of the chunk also writes it to the
    // pool.  Workers learn its index from dst_rows directly. ----
    int64_t rn = -1;
    if (APPEND) {
        const int64_t d = p.dst_rows[b];
        rn = (d >= row0 && d < row1) ? d : -1;
        if (warp == kWorkers / 32) {
            if (lane == 0) {
                *sNewRow = rn;
                const int64_t s0 = p.cu[b], s1 = p.cu[b + 1];
                if ((d < s0 || d >= s1) && row0 == s0 && group == 0) set_err(p.err, KVQ_ERR_ARG);
            }
            if (rn >= 0) {
                kv8_encode_row_warp(p.x_new + (int64_t)b * kMlaD, p.n_blocks, p.bd0, p.bd1, sNew, sNewScale, lane,
                                    group == 0 ? p.err : nullptr);
                __syncwarp();
                if (group == 0) {
                    for (int i = lane; i < kMlaD / 16; i += 32)
                        reinterpret_cast<uint4*>(p.codes_out + rn * kMlaD)[i] = reinterpret_cast<const uint4*>(sNew)[i];
                    if (lane < p.n_blocks) p.scales_out[rn * p.n_blocks + lane] = sNewScale[lane];
                }
            }
        }
    }

    // ---- query: 64 heads x 576 bf16, 18 16-byte loads per worker held in
    // registers; largest |q| ----
    const int64_t qbase = ((int64_t)b * p.n_heads + hbase) * kMlaD;
    constexpr int kQPer = kHC * kMlaD / 8 / kWorkers;   // 18
    static_assert(kHC * kMlaD / 8 == kQPer * kWorkers, "query loads per worker");
    uint4 qraw[kQPer];
    if (tid < kWorkers) {
        const uint4* qv = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) + qbase);
        float qmax = 0.0f;
#pragma unroll
        for (int i = 0; i < kQPer; ++i) qraw[i] = __ldg(qv + tid + i * kWorkers);
#pragma unroll
        for (int i = 0; i < kQPer; ++i) {
            const uint32_t in[4] = {qraw[i].x, qraw[i].y, qraw[i].z, qraw[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                qmax = fmaxf(qmax, fabsf(__uint_as_float(in[k] << 16)));
                qmax = fmaxf(qmax, fabsf(__uint_as_float(in[k] & 0xffff0000u)));
            }
        }
        qmax = warp_max(qmax);
        if (lane == 0) sRed[warp] = qmax;
    }
    __syncthreads();
    float q_max = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) q_max = fmaxf(q_max, sRed[i]);
    int e_q = 0;
    if (q_max > 0.0f) frexpf(q_max, &e_q);
    // |q| * q_scale < 2^14: every product with a code (|c| <= 448) and every
    // 576-term sum stays finite in f32, and a bf16 value scaled by a power of
    // two is exact in f16 unless it is below 2^-17 of the scaled maximum range
    // (its residual, under 2^-24 after scaling, is dropped)
    const float q_scale = q_max > 0.0f ? ldexpf(1.0f, 14 - e_q) : 1.0f;
    const float cz = p.sm_scale * kLog2e * (q_max > 0.0f ? ldexpf(1.0f, e_q - 14) : 1.0f);

    if (tid < kWorkers) {
#pragma unroll
        for (int i = 0; i < kQPer; ++i) {
            const int u = tid + i * kWorkers;
            const int e = u * 8, h = e / kMlaD, d = e - h * kMlaD;
            const uint32_t in[4] = {qraw[i].x, qraw[i].y, qraw[i].z, qraw[i].w};
            uint32_t hw[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const __half2 h2 = __floats2half2_rn(__uint_as_float(in[k] << 16) * q_scale,
                                                     __uint_as_float(in[k] & 0xffff0000u) * q_scale);
                hw[k] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(sQ + (d >> 6) * kQChunkBytes + sw128(h, (d & 63) * 2)) =
                make_uint4(hw[0], hw[1], hw[2], hw[3]);
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
            const uint64_t dp = umma_desc(smem_u32(sP), kSlotBytes, 1024);
            constexpr uint64_t kQStep = kQChunkBytes >> 4, kSlotStep = kSlotBytes >> 4;
            bool ok = true;
            if (p.stall_polls > 0) ok = mbar_wait(&bars[kBarNever], 0u, sAbort, p.stall_polls);
            for (int t = 0; t < n_tiles && ok; ++t) {
                const uint32_t par = (uint32_t)t & 1u;
#pragma unroll 1
                for (int kc = 0; kc < kChunks && ok; ++kc) {
                    if ((kc & 3) == 0) {
                        ok = mbar_wait(&bars[kBarFull0 + (kc >> 2)], par, sAbort, wl);
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
                ok = ok && mbar_wait(&bars[kBarP], par, sAbort, wl);
                tc_after();
#pragma unroll 1
                for (int db = 0; db < 4 && ok; ++db) {
                    const uint32_t d = tmem + kColO + 64 * db;
                    const uint64_t a = dpair0 + 2 * db * kSlotStep;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        umma_f16(d, a + 128 * ks, dp + 128 * ks, kIdescCtx, (t > 0 || ks > 0) ? 1u : 0u);
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
    const int hq = warp >> 2;                            // softmax: heads 32 hq .. 32 hq + 31
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    // running row sum of head 32 hq + lane over the rows of quadrant (warp & 3)
    // this thread's row: sums of p for its 32 heads, over every tile so far
    // (reduced over the rows once, in the epilogue); m and E of its heads,
    // refreshed after each exact path
    float lsum[32], mreg[32], ereg[32], emax = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; ++j) lsum[j] = 0.0f;
    auto load_state = [&]() {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            mreg[j] = sM[32 * hq + j];
            ereg[j] = sE[32 * hq + j];
        }
        emax = fmaxf(sEmax[0], sEmax[1]);
    };
    load_state();

    // this thread's softmax row scales, one tile ahead
    float sl_next = 0.0f, sr_next = 0.0f;
    auto load_scales = [&](int64_t t0n, int ntn) {
        sl_next = sr_next = 0.0f;
        if (srow < ntn) {
            const int64_t r = GATHER ? sRowIdx[(((t0n - row0) / kRows) & 1) * kRows + srow] : t0n + srow;
            if (APPEND && r == rn) {
                sl_next = sNewScale[0];
                sr_next = sNewScale[p.n_blocks - 1];
            } else {
                sl_next = p.scales[r * p.n_blocks];
                sr_next = p.scales[r * p.n_blocks + (p.n_blocks - 1)];
            }
        }
    };
    RawGroup rawA, rawB;
    RawRope rawC;
    {
        const int nt0 = (int)min((int64_t)kRows, row1 - row0);
        load_group<APPEND, GATHER>(rawA, p.codes, row0, nt0, 0, warp, lane, rn, sNew, sRowIdx);
        load_group<APPEND, GATHER>(rawB, p.codes, row0, nt0, 1, warp, lane, rn, sNew, sRowIdx);
        load_rope<APPEND, GATHER>(rawC, p.codes, row0, nt0, tid, rn, sNew, sRowIdx);
        load_scales(row0, nt0);
    }
    int t = 0;
    for (; t < n_tiles; ++t) {
        const int64_t t0 = row0 + (int64_t)t * kRows;
        const int nt = (int)min((int64_t)kRows, row1 - t0);
        if (!GATHER && tid == 0 && t0 + 2 * kRows < row1) {
            const int64_t n = min((int64_t)kRows, row1 - (t0 + 2 * kRows));
            prefetch_l2(p.codes + (t0 + 2 * kRows) * kMlaD, (uint32_t)(n * kMlaD));
        }
        // gather: the next tile's pool rows, read after the softmax's first barrier
        if (GATHER && tid < kRows && t0 + kRows < row1)
            sRowIdx[((t + 1) & 1) * kRows + tid] = t0 + kRows + tid < row1 ? gather_row(p, t0 + kRows + tid) : 0;
        const float my_sl = sl_next, my_sr = sr_next;
        // ---- decode the tile: groups A (chunks 0-3), B (4-7), C (rope) ----
        const uint32_t prev = (uint32_t)(t - 1) & 1u;
        {
            const int q4 = lane & 3, cg = lane >> 3;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                if (t > 0) {
                    if (!APPEND && (warp & 3) == 0) {
                        // warps 0 and 4 share a scheduler with the MMA-issuing
                        // warp: here they wait on named barrier 2 + g, which
                        // warp 1 releases once it has seen both slots free.
                        // Warp 1 arrives there again only after the next
                        // tile's context, which needs these warps' P^T, so
                        // each barrier instance completes before the next one
                        // starts.  (Measured faster on the prefill's long
                        // items, not on the appending decode.)
                        asm volatile("bar.sync %0, 96;" ::"r"(2 + g) : "memory");
                    } else {
                        mbar_wait(&bars[kBarFree0 + 2 * g], prev, sAbort, wl);
                        mbar_wait(&bars[kBarFree0 + 2 * g + 1], prev, sAbort, wl);
                        if (!APPEND && warp == 1) asm volatile("bar.arrive %0, 96;" ::"r"(2 + g) : "memory");
                    }
                }
                unsigned char* slot = sSlot + (4 * g + cg) * kSlotBytes;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    store16(slot, g == 0 ? rawA.v[i] : rawB.v[i], 2 * (warp + 8 * i) + ((lane >> 2) & 1), 32 * q4);
                fence_async_smem();
                mbar_arrive(&bars[kBarFull0 + g]);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int u = tid + kWorkers * i;
                store16(sSlot + kRope * kSlotBytes, rawC.v[i], u >> 2, 32 * (u & 3));
            }
            fence_async_smem();
            mbar_arrive(&bars[kBarFull0 + 2]);
        }
        const int64_t t1 = t0 + kRows;
        const int nt1 = (int)min((int64_t)kRows, row1 - t1);
        // all of tile t+1 is requested before the softmax (its raw codes stay in
        // registers across it: the worker warps' share of the register split)
        if (!GATHER && t + 1 < n_tiles) {
            if (nt1 == kRows && !(APPEND && rn >= t1 && rn < t1 + kRows)) {
                load_tile_full(rawA, rawB, rawC, p.codes, t1, warp, lane, tid);
            } else {
                load_group<APPEND, GATHER>(rawA, p.codes, t1, nt1, 0, warp, lane, rn, sNew, nullptr);
                load_group<APPEND, GATHER>(rawB, p.codes, t1, nt1, 1, warp, lane, rn, sNew, nullptr);
                load_rope<APPEND, GATHER>(rawC, p.codes, t1, nt1, tid, rn, sNew, nullptr);
            }
            load_scales(t1, nt1);
        }

        // ---- softmax of the tile: thread = row srow, 32 heads ----
        // one warp polls; the others wait on the named barrier, issuing nothing
        if (warp == 1) mbar_wait(&bars[kBarScore], (uint32_t)t & 1u, sAbort, wl);
        worker_sync();
        tc_after();
        // d = z - m with z = sm log2(e) (s_L S_L + s_R S_R), for this row's 32
        // heads read from TMEM: the lag test below and the weights 2^d after it
        float z[32];
        const float za = my_sl * cz, zb = my_sr * cz;
        const bool row_ok = srow < nt;
        auto load_d = [&]() {
            // 16 heads at a time: their rope and latent columns go out together,
            // then one wait (all four at once made the appending kernel spill)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t r[16], l[16];
                tmem_ld16(tmem + lane_base + kColSR + 32 * hq + 16 * c, r);
                tmem_ld16(tmem + lane_base + kColSL + 32 * hq + 16 * c, l);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    z[16 * c + j] = row_ok ? fmaf(__uint_as_float(l[j]), za,
                                                  fmaf(__uint_as_float(r[j]), zb, -mreg[16 * c + j]))
                                           : -INFINITY;
            }
        };
        load_d();
        // a latent scale with s_L max_h E > kScaleLim takes the exact path
        // (max_h E is +inf while only inert latent blocks have been met); so
        // does a score past m by more than the lag (m = -inf before the first
        // exact path: d = +inf on every row of the tile)
        // one maximum over the heads, then one test
        float dm[4] = {z[0], z[1], z[2], z[3]};
#pragma unroll
        for (int j = 4; j < 32; ++j) dm[j & 3] = fmaxf(dm[j & 3], z[j]);
        const float dmax = fmaxf(fmaxf(dm[0], dm[1]), fmaxf(dm[2], dm[3]));
        const bool flag = (*sAbort != 0) | (my_sl * emax > kScaleLim) | (dmax > kLagLog2);
        const bool any_flag = worker_any(flag);
        if (GATHER && t + 1 < n_tiles) {
            // the barrier above made the next tile's index table visible
            const int64_t* prow = sRowIdx + ((t + 1) & 1) * kRows;
            load_group<APPEND, GATHER>(rawA, p.codes, t1, nt1, 0, warp, lane, rn, sNew, prow);
            load_group<APPEND, GATHER>(rawB, p.codes, t1, nt1, 1, warp, lane, rn, sNew, prow);
            load_rope<APPEND, GATHER>(rawC, p.codes, t1, nt1, tid, rn, sNew, prow);
            load_scales(t1, nt1);
        }
        if (any_flag) {
            if (worker_any(*sAbort != 0)) break;
            exact_path(sm, tmem, lane_base, hq, row_ok, za, zb, my_sl, lane, warp, tid, t, p.exact_count);
#pragma unroll
            for (int j = 0; j < 32; ++j) lsum[j] *= sAlphaM[32 * hq + j];
            load_state();
            load_d();   // refreshed after the rescale path
        }
        {
            // row-sum weights p = 2^(z - m), f16 context weights w = p s_L E
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                z[j] = ex2(z[j]);
                z[j + 1] = ex2(z[j + 1]);
                const __half2 h2 = __floats2half2_rn(z[j] * ereg[j] * my_sl, z[j + 1] * ereg[j + 1] * my_sl);
                pk[j / 2] = *reinterpret_cast<const uint32_t*>(&h2);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<uint4*>(sP + sw128(srow, 64 * hq + 16 * i)) =
                    make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
        fence_async_smem();
        tc_before();
        mbar_arrive(&bars[kBarP]);
#pragma unroll
        for (int j = 0; j < 32; ++j) lsum[j] += z[j];
    }

    // ---- epilogue: wait for every MMA, row sums, O^T -> partial state ----
    {
        // bounded, and not cut short by the abort flag: TMEM is released only
        // after the MMAs in flight have completed
        volatile int never = 0;
        if (!mbar_wait(&bars[kBarDone], 0u, &never)) *sAbort = 1;
    }
    tc_after();
    const bool aborted = worker_any(*sAbort != 0 || t < n_tiles);
    {
        worker_sync();   // sRed may still be read by the last exact-max pass
        sRed[(warp & 3) * kHC + 32 * hq + lane] = warp_columns<false>(lsum, lane);
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
                        n_tiles > 0 ? __uint_as_float(v[j]) * sF[32 * c + j] : 0.0f;
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

}  // namespace

namespace {
template <bool APPEND, bool GATHER>
cudaError_t launch_kv8(const AttnParams& p, int64_t grid_x, int groups, cudaStream_t stream) {
    // the worker warps' setmaxnreg.inc waits for registers the other warpgroup
    // released: launch only if the split adds up against the launch's own count
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, attn_tc_kv8_kernel<APPEND, GATHER>);
    if (e != cudaSuccess) return e;
    if (kWorkers * kRegsWorker + 128 * kRegsMma > kThreads * fa.numRegs) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(attn_tc_kv8_kernel<APPEND, GATHER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemUsed);
    if (e != cudaSuccess) return e;
    attn_tc_kv8_kernel<APPEND, GATHER><<<dim3((unsigned)(grid_x * groups)), kThreads, kSmemUsed, stream>>>(p);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_attn_tc_kv8_bf16(const AttnParams& p, int64_t grid_x, int groups, cudaStream_t stream) {
    return p.sel ? launch_kv8<false, true>(p, grid_x, groups, stream) : launch_kv8<false, false>(p, grid_x, groups, stream);
}

cudaError_t launch_attn_tc_kv8_bf16_append(const AttnParams& p, int64_t grid_x, int groups, cudaStream_t stream) {
    return launch_kv8<true, false>(p, grid_x, groups, stream);
}

}  // namespace kvq
