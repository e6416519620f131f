// attn_simt.cu -- fp32 CUDA-core attention over quantized MLA rows (the
// parity path: outputs within 1e-5 of exact attention).
//
// Work decomposition (split-T, [P1] Commits item 2: split-T kernels): the rows
// of every sequence are cut into chunks of `chunk` rows; one CTA handles one
// (chunk, group of 32 heads) and leaves a partial softmax state (running max
// m, running sum l, unnormalized context o[512]) per head in the workspace.  A
// second kernel merges the chunks of each (sequence, head) by log-sum-exp and,
// for TQ4, unrotates the context once.  Ragged sequences are found on the
// device from cu_seqlens, so nothing is synchronized with the host.
//
// Inside a CTA the consumer never reconstructs a row ([P2] "What's in it"):
// a tile of 16 rows is decoded to the codes' values only (e4m3 value, TQ4
// codebook level, or the PolarQuant tree's leaves under a unit radius) and the
// per-row scales (radii) stay separate.  The score of head h
// and row t is sm_scale * (s_L * (q_L . c_L) + s_R * (q_R . c_R)) and the
// context weight of row t is p_t * s_L: the scale is factored out of both sums.
// For TQ4 and PolarQuant the query is rotated in shared memory first ([P1]
// "Ready for review" comment, finding 2: the rotation is orthogonal, so
// q . x_hat = rotate(q) . y_hat and the context unrotates once).
#include "attn_common.cuh"
#include "pq_common.cuh"

#include <algorithm>
#include <math.h>

namespace kvq {
namespace {

constexpr int kD = kMlaD, kDL = kMlaDL, kDV = kMlaDV;
constexpr int kHG = 32;   // heads per CTA: each tile is decoded (a PolarQuant row rebuilt) once for them
constexpr int kTR = 16;   // rows per tile
constexpr int kFlushTiles = 64;   // tiles per block sum (1024 rows)
constexpr int kNT = 512;  // threads per CTA: a score (head, row) and a 4-head x 8-dim context share each
constexpr int kXS = 580;  // shared-memory row stride in floats (bank spread)
constexpr int kSmSMs = 152;

// shared floats: queries, tile, row scales, weights, rescale factors, TQ4 levels (16),
// item info (4 int64), the pool rows of a gather tile (kTR int64), the
// PolarQuant centroids of levels 1..9 (up to 64 (cos, sin) pairs each)
constexpr int kPqCentPairs = 9 * 64;
constexpr size_t kSmemFloats =
    (size_t)kHG * kXS + (size_t)kTR * kXS + kTR * 2 + kTR * kHG + kHG + 16 + 8 + 2 * kTR + 2 * kPqCentPairs;

// One PolarQuant block of n = 32 Q leaves (2^L, unit top radius) rebuilt by
// one warp in registers and stored to y[0 .. n).  Lane k owns the subtree of
// node k at level log2(Q): its radius is the product of the factors on its
// path from the root (each lane reads the top L - log2(Q) angles of that
// path), then the lane expands its Q leaves level by level.  Node j of level
// l is the right child (factor sin) when j is odd.  The products are taken in
// the in-place expansion's order (root to leaf, each rounded once), so the
// leaves are bit-identical to it, without its strided shared-memory accesses
// (2- to 16-way bank conflicts at every level).
template <int Q, int L>
__device__ __forceinline__ void pq_expand_regs(const uint8_t* __restrict__ stream, int b, const float2* cent, float* y,
                                               int lane) {
    constexpr int n = 32 * Q;
    constexpr int Lb = Q == 16 ? 4 : Q == 8 ? 3 : Q == 4 ? 2 : Q == 2 ? 1 : 0;
    static_assert((1 << Lb) == Q && n == (1 << L), "block shape");
    float v = 1.0f;
#pragma unroll
    for (int l = L; l > Lb; --l) {
        const int j = lane >> (l - Lb);            // the path's node at level l
        const int first = n - (n >> (l - 1));      // stream index of level l's first angle
        const float2 cs = cent[((l - 1) << b) + pq_get_bits(stream, (int64_t)(first + j) * b, b)];
        v = __fmul_rn(v, ((lane >> (l - 1 - Lb)) & 1) ? cs.y : cs.x);
    }
    float t[Q];
    t[0] = v;
#pragma unroll
    for (int l = Lb; l >= 1; --l) {
        const int first = n - (n >> (l - 1));
#pragma unroll
        for (int jj = 0; jj < (Q >> l); ++jj) {
            const int j = (lane << (Lb - l)) + jj;
            const float2 cs = cent[((l - 1) << b) + pq_get_bits(stream, (int64_t)(first + j) * b, b)];
            const float r = t[jj << l];
            t[jj << l] = __fmul_rn(r, cs.x);
            t[(jj << l) + (1 << (l - 1))] = __fmul_rn(r, cs.y);
        }
    }
    if constexpr (Q % 4 == 0) {
#pragma unroll
        for (int i = 0; i < Q; i += 4)
            *reinterpret_cast<float4*>(y + Q * lane + i) = make_float4(t[i], t[i + 1], t[i + 2], t[i + 3]);
    } else {
        static_assert(Q == 2, "leaves per lane");
        *reinterpret_cast<float2*>(y + 2 * lane) = make_float2(t[0], t[1]);
    }
}

template <int FMT, bool QBF16, bool GATHER>
__global__ void __launch_bounds__(kNT, 1) attn_partial_kernel(AttnParams p) {
    launch_dependents();
    extern __shared__ float4 smem4[];
    float* qs = reinterpret_cast<float*>(smem4);
    float* xs = qs + kHG * kXS;
    float* sc = xs + kTR * kXS;
    float* P = sc + kTR * 2;
    float* alpha = P + kTR * kHG;
    float* lvs = alpha + kHG;
    int64_t* info = reinterpret_cast<int64_t*>(lvs + 16);
    int64_t* prow = info + 4;   // gather: the pool rows of the tile
    float2* pqc = reinterpret_cast<float2*>(prow + kTR);   // PolarQuant centroids

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t item = blockIdx.x;
    const int h0 = blockIdx.y * kHG;
    if (warp == 0) {
        int64_t r0 = 0, r1 = 0;
        const int b = locate_item(p, item, lane, &r0, &r1);
        if (lane == 0) {
            info[0] = b;
            info[1] = r0;
            info[2] = r1;
        }
    }
    if (tid < 16) lvs[tid] = p.lv[tid];
    if (FMT == kFmtPolar)
        for (int i = tid; i < (9 << p.pq_bits); i += kNT) pqc[i] = p.pq_cent[i];
    __syncthreads();
    const int b = (int)info[0];
    if (b < 0) return;
    const int64_t row0 = info[1], row1 = info[2];

    // queries of this head group -> shared memory, f32
    for (int i = tid; i < kHG * kD; i += kNT) {
        const int h = i / kD, d = i - h * kD;
        float v = 0.0f;
        if (h0 + h < p.n_heads) v = load_q<QBF16>(p.q, ((int64_t)b * p.n_heads + h0 + h) * kD + d);
        qs[h * kXS + d] = v;
    }
    __syncthreads();
    if (FMT != KVQ_KV8) {
        // rotate each head's query once: latent block (512) and rope block (64)
        for (int hh = warp; hh < kHG; hh += kNT / 32) {
            float* qh = qs + hh * kXS;
            float v[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int i = lane + 32 * k;
                v[k] = sign_neg(p.signs, 0, i) ? -qh[i] : qh[i];
            }
            warp_fwht<512>(v, lane);
#pragma unroll
            for (int k = 0; k < 16; ++k) qh[lane + 32 * k] = __fmul_rn(v[k], p.kn[0]);
            float r[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int i = lane + 32 * k;
                r[k] = sign_neg(p.signs, 1, i) ? -qh[kDL + i] : qh[kDL + i];
            }
            warp_fwht<64>(r, lane);
#pragma unroll
            for (int k = 0; k < 2; ++k) qh[kDL + lane + 32 * k] = __fmul_rn(r[k], p.kn[1]);
        }
        __syncthreads();
    }

    const int sh = tid >> 4;   // score: head of this thread
    const int st = tid & 15;   // score: row of this thread
    // Two-level sums: the block sums (o, l_blk) take at most kFlushTiles tiles
    // and are then added into the totals (o_tot, l_run), so that f32 rounding
    // grows with sqrt(rows / 1024) + sqrt(1024) rather than sqrt(rows) over
    // chunks of 10^5 rows.
    float m_run = -INFINITY, l_run = 0.0f, l_blk = 0.0f;
    const int cq = tid >> 6;   // context: head quad
    const int cc = tid & 63;   // context: dims 4cc..4cc+3 and 256+4cc..+3
    float o[4][8], o_tot[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) o[i][j] = o_tot[i][j] = 0.0f;
    int blk_tiles = 0;

    for (int64_t t0 = row0; t0 < row1; t0 += kTR) {
        const int nt = (int)min((int64_t)kTR, row1 - t0);
        if (GATHER) {
            if (tid < kTR) prow[tid] = tid < nt ? gather_row(p, t0 + tid) : 0;
            __syncthreads();
        }
        // decode the tile to code values (no scale applied)
        if (FMT == KVQ_KV8) {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(p.codes + t0 * kD);
            for (int w = tid; w < kTR * (kD / 4); w += kNT) {
                const int r = w / (kD / 4), c4 = (w - r * (kD / 4)) * 4;
                float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
                if (r < nt) {
                    const uint32_t u = GATHER ? __ldg(reinterpret_cast<const uint32_t*>(p.codes + prow[r] * kD) + c4 / 4)
                                              : __ldg(src + w);
                    f = e4m3x4_to_float4(u);
                }
                *reinterpret_cast<float4*>(xs + r * kXS + c4) = f;
            }
        } else if (FMT == kFmtPolar) {
            // each warp rebuilds whole rows: the latent and rope trees with unit
            // top radius, in the rotated domain (the radii stay in sc)
            for (int r = warp; r < kTR; r += kNT / 32) {
                float* xr = xs + r * kXS;
                if (r < nt) {
                    const uint8_t* cr = p.codes + (GATHER ? prow[r] : t0 + r) * p.pq_row_bytes;
                    pq_expand_regs<kDL / 32, 9>(cr, p.pq_bits, pqc, xr, lane);
                    pq_expand_regs<kMlaDR / 32, 6>(cr + p.pq_boff1, p.pq_bits, pqc, xr + kDL, lane);
                } else {
                    for (int i = lane; i < kD; i += 32) xr[i] = 0.0f;
                }
            }
        } else {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(p.codes + t0 * (kD / 2));
            for (int w = tid; w < kTR * (kD / 8); w += kNT) {
                const int r = w / (kD / 8), c8 = (w - r * (kD / 8)) * 8;
                float f[8];
                if (r < nt) {
                    const uint32_t u = GATHER ? __ldg(reinterpret_cast<const uint32_t*>(p.codes + prow[r] * (kD / 2)) + c8 / 8)
                                              : __ldg(src + w);
#pragma unroll
                    for (int j = 0; j < 8; ++j) f[j] = lvs[(u >> (4 * j)) & 15u];
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) f[j] = 0.0f;
                }
                *reinterpret_cast<float4*>(xs + r * kXS + c8) = make_float4(f[0], f[1], f[2], f[3]);
                *reinterpret_cast<float4*>(xs + r * kXS + c8 + 4) = make_float4(f[4], f[5], f[6], f[7]);
            }
        }
        if (tid < kTR) {
            float sL = 0.0f, sR = 0.0f;
            if (tid < nt) {
                const int64_t row = GATHER ? prow[tid] : t0 + tid;
                if (p.n_blocks == 2) {
                    sL = p.scales[row * 2];
                    sR = p.scales[row * 2 + 1];
                } else {
                    sL = sR = p.scales[row];
                }
            }
            sc[tid * 2] = sL;
            sc[tid * 2 + 1] = sR;
        }
        __syncthreads();

        // scores and the online softmax of this tile (16 lanes share a head)
        {
            const float* qh = qs + sh * kXS;
            const float* xr = xs + st * kXS;
            float aL0 = 0.f, aL1 = 0.f, aL2 = 0.f, aL3 = 0.f;
#pragma unroll 8
            for (int d = 0; d < kDL; d += 4) {
                const float4 a = *reinterpret_cast<const float4*>(qh + d);
                const float4 x = *reinterpret_cast<const float4*>(xr + d);
                aL0 = fmaf(a.x, x.x, aL0);
                aL1 = fmaf(a.y, x.y, aL1);
                aL2 = fmaf(a.z, x.z, aL2);
                aL3 = fmaf(a.w, x.w, aL3);
            }
            float aR0 = 0.f, aR1 = 0.f, aR2 = 0.f, aR3 = 0.f;
#pragma unroll
            for (int d = kDL; d < kD; d += 4) {
                const float4 a = *reinterpret_cast<const float4*>(qh + d);
                const float4 x = *reinterpret_cast<const float4*>(xr + d);
                aR0 = fmaf(a.x, x.x, aR0);
                aR1 = fmaf(a.y, x.y, aR1);
                aR2 = fmaf(a.z, x.z, aR2);
                aR3 = fmaf(a.w, x.w, aR3);
            }
            const float dotL = (aL0 + aL1) + (aL2 + aL3);
            const float dotR = (aR0 + aR1) + (aR2 + aR3);
            const float z = st < nt ? p.sm_scale * (sc[st * 2] * dotL + sc[st * 2 + 1] * dotR) : -INFINITY;
            float tmax = z;
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, off));
            const float m_new = fmaxf(m_run, tmax);
            const float a = m_run == -INFINITY ? 0.0f : expf(m_run - m_new);
            const float pz = expf(z - m_new);
            float psum = pz;
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) psum += __shfl_xor_sync(kFull, psum, off);
            l_blk = l_blk * a + psum;
            l_run = l_run * a;
            m_run = m_new;
            P[st * kHG + sh] = pz * sc[st * 2];
            if (st == 0) alpha[sh] = a;
        }
        __syncthreads();

        // context: o[h][d] = alpha_h * o[h][d] + sum_t P[t][h] * c[t][d]
        {
            float al[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) al[i] = alpha[cq * 4 + i];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    o[i][j] *= al[i];
                    o_tot[i][j] *= al[i];
                }
            for (int t = 0; t < nt; ++t) {
                const float4 xa = *reinterpret_cast<const float4*>(xs + t * kXS + 4 * cc);
                const float4 xb = *reinterpret_cast<const float4*>(xs + t * kXS + 256 + 4 * cc);
                const float4 pw = *reinterpret_cast<const float4*>(P + t * kHG + 4 * cq);
                const float pv[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    o[i][0] = fmaf(pv[i], xa.x, o[i][0]);
                    o[i][1] = fmaf(pv[i], xa.y, o[i][1]);
                    o[i][2] = fmaf(pv[i], xa.z, o[i][2]);
                    o[i][3] = fmaf(pv[i], xa.w, o[i][3]);
                    o[i][4] = fmaf(pv[i], xb.x, o[i][4]);
                    o[i][5] = fmaf(pv[i], xb.y, o[i][5]);
                    o[i][6] = fmaf(pv[i], xb.z, o[i][6]);
                    o[i][7] = fmaf(pv[i], xb.w, o[i][7]);
                }
            }
        }
        if (++blk_tiles == kFlushTiles) {
            blk_tiles = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    o_tot[i][j] += o[i][j];
                    o[i][j] = 0.0f;
                }
            l_run += l_blk;
            l_blk = 0.0f;
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) o[i][j] += o_tot[i][j];
    l_run += l_blk;

    // partial state of this chunk
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int h = h0 + cq * 4 + i;
        if (h < p.n_heads) {
            float* dst = p.ws_o + (item * p.n_heads + h) * kDV;
            *reinterpret_cast<float4*>(dst + 4 * cc) = make_float4(o[i][0], o[i][1], o[i][2], o[i][3]);
            *reinterpret_cast<float4*>(dst + 256 + 4 * cc) = make_float4(o[i][4], o[i][5], o[i][6], o[i][7]);
        }
    }
    if (st == 0 && h0 + sh < p.n_heads) {
        float* ml = p.ws_ml + (item * p.n_heads + h0 + sh) * 2;
        ml[0] = m_run;
        ml[1] = l_run;
    }
}

template <int FMT>
__global__ void __launch_bounds__(128) attn_merge_kernel(AttnParams p, float* __restrict__ out) {
    __shared__ int64_t info[2];
    __shared__ float ov[kDV];
    const int h = blockIdx.x, b = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31;
    const bool prefill = p.prefill_past >= 0;
    // a chunk the partial kernel chose on the device is read after the wait
    const bool dev_chunk = !prefill && p.wave_items > 0;
    if (dev_chunk) grid_dependency_wait();
    if (tid < 32) {
        int64_t first = b, count = 1;
        if (!prefill) seq_items(p.cu, b, dev_chunk ? *p.ws_chunk : p.chunk, lane, &first, &count, p.err);
        if (lane == 0) {
            info[0] = first;
            info[1] = count;
        }
    }
    __syncthreads();
    if (!dev_chunk) grid_dependency_wait();   // the partial state is complete and visible past this point
    const int64_t first = info[0];
    int64_t count = info[1];
    if (first + count > p.max_items) {
        if (tid == 0) set_err(p.err, KVQ_ERR_DEVICE);
        count = 0;
    }
    // one pass over the chunks, 8 at a time: their loads go out together, then
    // an online log-sum-exp combine (running max M, sum L, weighted context)
    float M = -INFINITY, L = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    constexpr int kBatch = 8;
    for (int64_t c0 = 0; c0 < count; c0 += kBatch) {
        float mv[kBatch], lw[kBatch];
        float4 ov[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            mv[k] = -INFINITY;
            lw[k] = 0.0f;
            ov[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c0 + k < count) {
                const int64_t row = (first + c0 + k) * p.n_heads + h;
                const float2 ml = *reinterpret_cast<const float2*>(p.ws_ml + row * 2);
                mv[k] = ml.x;
                lw[k] = ml.y;
                ov[k] = *reinterpret_cast<const float4*>(p.ws_o + row * kDV + 4 * tid);
            }
        }
        float mb = M;
#pragma unroll
        for (int k = 0; k < kBatch; ++k) mb = fmaxf(mb, mv[k]);
        if (mb == -INFINITY) continue;   // nothing but empty partials so far
        const float keep = M == -INFINITY ? 0.0f : expf(M - mb);
        L *= keep;
        acc = make_float4(acc.x * keep, acc.y * keep, acc.z * keep, acc.w * keep);
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const float w = mv[k] == -INFINITY ? 0.0f : expf(mv[k] - mb);
            L = fmaf(w, lw[k], L);
            acc.x = fmaf(w, ov[k].x, acc.x);
            acc.y = fmaf(w, ov[k].y, acc.y);
            acc.z = fmaf(w, ov[k].z, acc.z);
            acc.w = fmaf(w, ov[k].w, acc.w);
        }
        M = mb;
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    acc = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    float* dst = out + ((int64_t)b * p.n_heads + h) * kDV;
    if (FMT == KVQ_KV8) {
        *reinterpret_cast<float4*>(dst + 4 * tid) = acc;
        return;
    }
    *reinterpret_cast<float4*>(ov + 4 * tid) = acc;
    __syncthreads();
    if (tid < 32) {
        // context was accumulated in the rotated domain: unrotate once
        float v[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = ov[lane + 32 * k];
        warp_fwht<512>(v, lane);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int i = lane + 32 * k;
            const float y = __fmul_rn(v[k], p.kn[0]);
            dst[i] = sign_neg(p.signs, 0, i) ? -y : y;
        }
    }
}

template <int FMT, bool QBF16>
cudaError_t launch_partial(const AttnParams& p, int64_t grid_x, int groups, cudaStream_t stream) {
    const size_t smem = kSmemFloats * sizeof(float);
    auto kernel = p.sel ? attn_partial_kernel<FMT, QBF16, true> : attn_partial_kernel<FMT, QBF16, false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<dim3((unsigned)grid_x, (unsigned)groups), kNT, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

AttnPlan plan_decode_simt(int32_t batch, int32_t n_heads, int64_t max_total_rows) {
    AttnPlan pl{};
    pl.heads_per_cta = kHG;
    const int64_t groups = (n_heads + kHG - 1) / kHG;
    const int64_t target_items = std::max<int64_t>(1, (int64_t)kSmSMs * 4 / groups);
    int64_t chunk = (std::max<int64_t>(max_total_rows, 1) + target_items - 1) / target_items;
    chunk = std::max<int64_t>(kTR, (chunk + kTR - 1) / kTR * kTR);
    pl.chunk = chunk;
    pl.max_items = (max_total_rows + chunk - 1) / chunk + batch;
    return pl;
}

AttnParams make_attn_params(kvq_format fmt, const kvq_mla_layout& L, const void* q, int32_t n_seq, int32_t n_heads,
                            const uint8_t* codes, const float* scales, const int64_t* cu_seqlens,
                            int64_t prefill_past, const AttnPlan& plan, float sm_scale, void* workspace) {
    AttnParams p{};
    p.n_blocks = L.n_blocks;
    p.n_seq = n_seq;
    p.n_heads = n_heads;
    p.q = q;
    p.codes = codes;
    p.scales = scales;
    p.cu = cu_seqlens;
    p.prefill_past = prefill_past;
    p.chunk = plan.chunk;
    p.max_items = plan.max_items;
    p.wave_items = plan.wave_items;
    p.max_waves = plan.max_waves;
    p.max_rows = plan.max_rows;
    p.sm_scale = sm_scale;
    char* ws = static_cast<char*>(workspace);
    p.err = reinterpret_cast<int32_t*>(ws);
    p.ws_chunk = reinterpret_cast<int64_t*>(ws + 8);
    p.exact_count = reinterpret_cast<uint32_t*>(ws + 16);
    p.stall_polls = test_stall_polls();
    p.wait_limit = p.stall_polls > 0 ? p.stall_polls : kWaitLimit;
    p.ws_o = reinterpret_cast<float*>(ws + kWsHeader);
    p.ws_ml = p.ws_o + (size_t)plan.max_items * n_heads * kMlaDV;
    if (fmt != KVQ_KV8) {
        p.signs = tq4_sign_words(L);
        p.kn[0] = (float)(1.0 / sqrt((double)L.block_dim[0]));
        p.kn[1] = (float)(1.0 / sqrt((double)L.block_dim[1]));
        const Codebook16 cb = tq4_codebook();
        for (int k = 0; k < 16; ++k) p.lv[k] = cb.lv[k];
    }
    if (is_pq(fmt)) {
        p.pq_bits = pq_bits_of(fmt);
        p.pq_boff1 = (int32_t)pq_block_bytes(L.block_dim[0], p.pq_bits);
        p.pq_row_bytes = (int32_t)pq_row_bytes(p.pq_bits, L);
        p.pq_cent = pq_device_centroids(p.pq_bits);
    }
    return p;
}

size_t partial_bytes(int64_t max_items, int32_t n_heads, int32_t v_dim) {
    return (size_t)max_items * n_heads * (v_dim + 2) * sizeof(float);
}

cudaError_t launch_attn_simt(kvq_format fmt, const kvq_mla_layout& L, const void* q, kvq_dtype qdt, int32_t n_seq,
                             int32_t n_heads, const uint8_t* codes, const float* scales, const int64_t* cu_seqlens,
                             int64_t prefill_past, const AttnPlan& plan, float sm_scale, float* out,
                             void* workspace, cudaStream_t stream, const int64_t* sel, int64_t pool_rows) {
    if (n_seq == 0 || n_heads == 0) return cudaSuccess;
    AttnParams p = make_attn_params(fmt, L, q, n_seq, n_heads, codes, scales, cu_seqlens, prefill_past, plan,
                                    sm_scale, workspace);
    p.sel = sel;
    p.pool_rows = pool_rows;
    const int groups = (n_heads + kHG - 1) / kHG;
    timing_mark(stream, 0);
    cudaError_t e;
    if (fmt == KVQ_KV8)
        e = qdt == KVQ_BF16 ? launch_partial<KVQ_KV8, true>(p, plan.max_items, groups, stream)
                            : launch_partial<KVQ_KV8, false>(p, plan.max_items, groups, stream);
    else if (is_pq(fmt))
        e = !p.pq_cent ? cudaErrorInvalidSymbol
            : qdt == KVQ_BF16 ? launch_partial<kFmtPolar, true>(p, plan.max_items, groups, stream)
                              : launch_partial<kFmtPolar, false>(p, plan.max_items, groups, stream);
    else
        e = qdt == KVQ_BF16 ? launch_partial<KVQ_TQ4, true>(p, plan.max_items, groups, stream)
                            : launch_partial<KVQ_TQ4, false>(p, plan.max_items, groups, stream);
    if (e != cudaSuccess) return e;
    return launch_attn_merge(fmt, p, out, stream);
}

// The merge is launched as a programmatic dependent of the partial kernel: its
// CTAs may start (and find their chunks) while the partial kernel drains, and
// wait for its completion before reading the partial state.
cudaError_t launch_attn_merge(kvq_format fmt, const AttnParams& p, float* out, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.n_heads, (unsigned)p.n_seq);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    timing_mark(stream, 1);
    const cudaError_t e = fmt == KVQ_KV8 ? cudaLaunchKernelEx(&cfg, attn_merge_kernel<KVQ_KV8>, p, out)
                                         : cudaLaunchKernelEx(&cfg, attn_merge_kernel<KVQ_TQ4>, p, out);
    timing_mark(stream, 2);
    return e;
}

}  // namespace kvq
