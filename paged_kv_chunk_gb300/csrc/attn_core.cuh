// Per-warp attention units of the streaming (paged) bf16 kernel: 16 query rows of one head
// against one stage of 64 keys, or against a 16-key slice of it.
//
// A CTA has kConsumerWarps consumer warps and one producer warp.  The producer streams
// stages of 64 keys (K rows, V rows and, without the position table, the rel band they
// need) into a ring of smem slots with TMA, completing a `full` mbarrier per slot;
// consumers release a slot by arriving on its `empty` mbarrier.  Consumer warp w owns
// m-tile (w % MT) of the CTA's Tp = 16*MT query rows and the stages s with
// s % KG == w / MT (KG = 4/MT), so each warp works on whole stages (warp_stage); with one
// m-tile the four warps instead split every stage into 16-key slices (warp_slice16, or
// warp_slice16_gt when the CTA has built its whole position term as a pre-skewed table,
// PosTable).  Per unit of work (the band form; with the table, G is read from it):
//
//   S  = bf16(q+u) . K^T                       mma.sync m16n8k16, fp32 accumulators
//   G  = bf16(q+v) . Rband^T                   80 band columns for the 64 keys
//   S += G[i][j + 15 - i]                      rel_shift skew through a smem tile
//   S  = S * scale * log2(e), keys past the end -> -inf
//   online softmax (running max/sum per row, fp32, exp2)
//   O += P . V                                 P rounded to bf16; V rows past the end
//                                              are zeroed in registers
//
// Score (Scheduler page, section 4.3; Model Layer page, fixed_attention_window row and
// Nemotron ASR section): s_ij = scale * ((q_i+u).k_j + (q_i+v).rel[rho]), rho = off + j - i
// with `off` chosen by the kernel's mode.  For keys [j0, j0+64) and query rows [i0, i0+Tp)
// a stage's band is rel rows [off + j0 - i0 - (Tp-1), +64+Tp); warp m-tile mt reads band rows
// from o = Tp - 16 - 16*mt, and element (i', j) of its tile uses band column j + 15 - i'.
#pragma once

#include "ptx.cuh"

namespace oasr {

constexpr int kHeadDim = 64;               // head dimension of the tensor-core path
constexpr int kStageKeys = 64;             // keys per stage
constexpr int kRowBytes = 128;             // one bf16 row of kHeadDim
constexpr int kConsumerWarps = 4;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kBandCols = kStageKeys + 16; // band columns one warp computes per stage
constexpr int kGW = kBandCols + 4;         // skew scratch row stride (floats)
constexpr int kGBytes = 16 * kGW * 4;      // skew scratch of one warp
constexpr int kOW = kHeadDim + 4;          // combine scratch row stride (floats)

template <int MT_>
struct Tile {
    static constexpr int MT = MT_;                  // 16-row m-tiles of the CTA
    static constexpr int KG = kConsumerWarps / MT;  // stage groups
    static constexpr int Tp = 16 * MT;              // padded query rows
    static constexpr int RB = kStageKeys + Tp;      // band rows per stage
};

struct WarpAcc {
    float o[8][4];  // 16 rows x 64 dims: n-tile dt holds dims [8dt, 8dt+8)
    float m[2];     // running max (log2 units) of rows g and g+8
    float l[2];     // running sum over this thread's columns
};

__device__ __forceinline__ void acc_init(WarpAcc& a)
{
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) a.o[i][e] = 0.f;
    a.m[0] = a.m[1] = -INFINITY;
    a.l[0] = a.l[1] = 0.f;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ uint16_t bf16_bits(float x)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// A fragments of bf16(q + u) and bf16(q + v) for the warp's 16 query rows (rows 16*mt..)
// of a swizzled Q tile; u, v are fp32 in smem.  Rounding q + u to bf16 changes a score
// by ~2^-9 of one term, far below the bf16 output rounding.
__device__ __forceinline__ void make_q_frags(uint32_t q_s, const float* u, const float* v, int mt,
                                             int lane, uint32_t (&qu)[4][4], uint32_t (&qv)[4][4])
{
    const int t4 = lane & 3;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        uint32_t r[4];
        ldsm_x4(q_s + swz128(16 * mt + (lane & 15), 2 * ks + (lane >> 4)), r[0], r[1], r[2], r[3]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = 16 * ks + ((i >> 1) << 3) + 2 * t4;   // r0,r1: cols 2t; r2,r3: 8+2t
            const float lo = bf16_lo(r[i]), hi = bf16_hi(r[i]);
            qu[ks][i] = pack_bf16(lo + u[c], hi + u[c + 1]);
            qv[ks][i] = pack_bf16(lo + v[c], hi + v[c + 1]);
        }
    }
}

// One warp, one stage.  k_s, v_s: shared addresses of the stage's 64 K and V rows;
// band_s: shared address of the stage's band tile, band_o: first band row this warp uses;
// g: this warp's skew scratch [16][kGW] floats (may alias the band tile once the band
// MMAs are done); kvalid: keys [0, kvalid) of the stage exist.
__device__ __forceinline__ void warp_stage(WarpAcc& acc, const uint32_t (&qu)[4][4],
                                           const uint32_t (&qv)[4][4], uint32_t k_s, uint32_t v_s,
                                           uint32_t band_s, int band_o, float* g, int kvalid,
                                           float scale_log2, int lane)
{
    const int g4 = lane >> 2, t4 = lane & 3, mi = lane >> 3;
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(k_s + swz128(16 * np + ((mi >> 1) << 3) + (lane & 7), 2 * ks + (mi & 1)), b0,
                    b1, b2, b3);
            mma_bf16_16816(s[2 * np], qu[ks], b0, b1);
            mma_bf16_16816(s[2 * np + 1], qu[ks], b2, b3);
        }
    }
    {
        float gacc[kBandCols / 8][4];
#pragma unroll
        for (int nb = 0; nb < kBandCols / 8; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e) gacc[nb][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int np = 0; np < kBandCols / 16; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(band_s + swz128(band_o + 16 * np + ((mi >> 1) << 3) + (lane & 7),
                                        2 * ks + (mi & 1)),
                        b0, b1, b2, b3);
                mma_bf16_16816(gacc[2 * np], qv[ks], b0, b1);
                mma_bf16_16816(gacc[2 * np + 1], qv[ks], b2, b3);
            }
        }
        __syncwarp();   // every lane's band reads are done before the scratch (maybe aliasing) is written
#pragma unroll
        for (int nb = 0; nb < kBandCols / 8; ++nb) {
            *reinterpret_cast<float2*>(g + g4 * kGW + 8 * nb + 2 * t4) =
                make_float2(gacc[nb][0], gacc[nb][1]);
            *reinterpret_cast<float2*>(g + (g4 + 8) * kGW + 8 * nb + 2 * t4) =
                make_float2(gacc[nb][2], gacc[nb][3]);
        }
    }
    __syncwarp();
    float mx0 = acc.m[0], mx1 = acc.m[1];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int j = 8 * nt + 2 * t4 + e;
            const bool ok = j < kvalid;
            const float b0 = g[g4 * kGW + j + 15 - g4];
            const float b1 = g[(g4 + 8) * kGW + j + 7 - g4];
            s[nt][e] = ok ? (s[nt][e] + b0) * scale_log2 : -INFINITY;
            s[nt][2 + e] = ok ? (s[nt][2 + e] + b1) * scale_log2 : -INFINITY;
        }
        mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float base0 = (mx0 == -INFINITY) ? 0.f : mx0;
    const float base1 = (mx1 == -INFINITY) ? 0.f : mx1;
    if (mx0 != acc.m[0] || mx1 != acc.m[1]) {
        const float alpha0 = ex2_approx(acc.m[0] - base0);
        const float alpha1 = ex2_approx(acc.m[1] - base1);
        acc.l[0] *= alpha0;
        acc.l[1] *= alpha1;
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) {
            acc.o[dt][0] *= alpha0;
            acc.o[dt][1] *= alpha0;
            acc.o[dt][2] *= alpha1;
            acc.o[dt][3] *= alpha1;
        }
        acc.m[0] = mx0;
        acc.m[1] = mx1;
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        s[nt][0] = ex2_approx(s[nt][0] - base0);
        s[nt][1] = ex2_approx(s[nt][1] - base0);
        s[nt][2] = ex2_approx(s[nt][2] - base1);
        s[nt][3] = ex2_approx(s[nt][3] - base1);
        acc.l[0] += s[nt][0] + s[nt][1];
        acc.l[1] += s[nt][2] + s[nt][3];
    }
    const bool tail = kvalid < kStageKeys;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint32_t pa[4] = {pack_bf16(s[2 * kk][0], s[2 * kk][1]),
                                pack_bf16(s[2 * kk][2], s[2 * kk][3]),
                                pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                                pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3])};
        const int row = 16 * kk + ((mi & 1) << 3) + (lane & 7);
        // keys held by this lane's B fragments: b0,b2 -> 16kk+2t(+1), b1,b3 -> 16kk+8+2t(+1)
        const int k0 = 16 * kk + 2 * t4;
#pragma unroll
        for (int dp = 0; dp < 4; ++dp) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(v_s + swz128(row, 2 * dp + (mi >> 1)), b0, b1, b2, b3);
            if (tail) {   // V rows past the last key may hold anything (0 * NaN is NaN)
                const uint32_t m0 = (k0 < kvalid ? 0xffffu : 0u) | (k0 + 1 < kvalid ? 0xffff0000u : 0u);
                const uint32_t m1 =
                    (k0 + 8 < kvalid ? 0xffffu : 0u) | (k0 + 9 < kvalid ? 0xffff0000u : 0u);
                b0 &= m0;
                b2 &= m0;
                b1 &= m1;
                b3 &= m1;
            }
            mma_bf16_16816(acc.o[2 * dp], pa, b0, b1);
            mma_bf16_16816(acc.o[2 * dp + 1], pa, b2, b3);
        }
    }
}

// The rest of a 16-key slice once its scaled scores s (log2 units, masked keys -inf) and the
// running maxima folded with this thread's scores (mx0, mx1) are known: quad max, online
// softmax update, P rounded to bf16, O += P . V (vf: the slice's V fragments).
__device__ __forceinline__ void softmax_pv16(WarpAcc& acc, float (&s)[2][4], const uint32_t (&vf)[4][4],
                                             float mx0, float mx1, int kvalid, int lane)
{
    const int t4 = lane & 3;
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float base0 = (mx0 == -INFINITY) ? 0.f : mx0;
    const float base1 = (mx1 == -INFINITY) ? 0.f : mx1;
    if (mx0 != acc.m[0] || mx1 != acc.m[1]) {
        const float alpha0 = ex2_approx(acc.m[0] - base0);
        const float alpha1 = ex2_approx(acc.m[1] - base1);
        acc.l[0] *= alpha0;
        acc.l[1] *= alpha1;
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) {
            acc.o[dt][0] *= alpha0;
            acc.o[dt][1] *= alpha0;
            acc.o[dt][2] *= alpha1;
            acc.o[dt][3] *= alpha1;
        }
        acc.m[0] = mx0;
        acc.m[1] = mx1;
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        s[nt][0] = ex2_approx(s[nt][0] - base0);
        s[nt][1] = ex2_approx(s[nt][1] - base0);
        s[nt][2] = ex2_approx(s[nt][2] - base1);
        s[nt][3] = ex2_approx(s[nt][3] - base1);
        acc.l[0] += s[nt][0] + s[nt][1];
        acc.l[1] += s[nt][2] + s[nt][3];
    }
    const uint32_t pa[4] = {pack_bf16(s[0][0], s[0][1]), pack_bf16(s[0][2], s[0][3]),
                            pack_bf16(s[1][0], s[1][1]), pack_bf16(s[1][2], s[1][3])};
    const int k0 = 2 * t4;   // keys of this lane's B fragments: b0,b2 -> 2t(+1), b1,b3 -> 8+2t(+1)
    const bool tail = kvalid < 16;
    const uint32_t m0 = (k0 < kvalid ? 0xffffu : 0u) | (k0 + 1 < kvalid ? 0xffff0000u : 0u);
    const uint32_t m1 = (k0 + 8 < kvalid ? 0xffffu : 0u) | (k0 + 9 < kvalid ? 0xffff0000u : 0u);
#pragma unroll
    for (int dp = 0; dp < 4; ++dp) {
        uint32_t b0 = vf[dp][0], b1 = vf[dp][1], b2 = vf[dp][2], b3 = vf[dp][3];
        if (tail) {   // V rows past the last key may hold anything (0 * NaN is NaN)
            b0 &= m0;
            b2 &= m0;
            b1 &= m1;
            b3 &= m1;
        }
        mma_bf16_16816(acc.o[2 * dp], pa, b0, b1);
        mma_bf16_16816(acc.o[2 * dp + 1], pa, b2, b3);
    }
}

// One warp, 16 query rows, one 16-key slice of a stage (the four consumer warps of a
// one-m-tile CTA split every stage this way, so a stage is consumed in a quarter of the
// latency).  k_s, v_s: shared addresses of the slice's first K and V rows; band_s: the
// slice's first band row (32 band rows: element (i, j) of the slice uses band row
// j + 15 - i); g: 16 x 32 floats of skew scratch, which may alias the slice's K rows (they
// are dead once S is formed); kvalid: keys [0, kvalid) of the slice exist (kvalid > 0).
// Scratch column c of row r is stored at c ^ (8 * (r & 3)): the fragment stores are
// conflict-free, the skewed reads at most 2-way.
__device__ __forceinline__ void warp_slice16(WarpAcc& acc, const uint32_t (&qu)[4][4],
                                             const uint32_t (&qv)[4][4], uint32_t k_s, uint32_t v_s,
                                             uint32_t band_s, float* g, int kvalid, float scale_log2,
                                             int lane)
{
    const int g4 = lane >> 2, t4 = lane & 3, mi = lane >> 3;
    uint32_t vf[4][4];   // V fragments of the slice
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(k_s + swz128(((mi >> 1) << 3) + (lane & 7), 2 * ks + (mi & 1)), b0, b1, b2, b3);
        mma_bf16_16816(s[0], qu[ks], b0, b1);
        mma_bf16_16816(s[1], qu[ks], b2, b3);
    }
    {
        float gacc[4][4];
#pragma unroll
        for (int nb = 0; nb < 4; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e) gacc[nb][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(band_s + swz128(16 * np + ((mi >> 1) << 3) + (lane & 7), 2 * ks + (mi & 1)),
                        b0, b1, b2, b3);
                mma_bf16_16816(gacc[2 * np], qv[ks], b0, b1);
                mma_bf16_16816(gacc[2 * np + 1], qv[ks], b2, b3);
            }
        }
        __syncwarp();   // every lane's K reads are done before the scratch (aliasing them) is written
        // the slice's V fragments now, so their shared-memory latency hides behind the skew
        // and the softmax
        const int vrow = ((mi & 1) << 3) + (lane & 7);
#pragma unroll
        for (int dp = 0; dp < 4; ++dp)
            ldsm_x4_t(v_s + swz128(vrow, 2 * dp + (mi >> 1)), vf[dp][0], vf[dp][1], vf[dp][2], vf[dp][3]);
        const int sw0 = 8 * (g4 & 3);   // rows g4 and g4 + 8 share the swizzle
#pragma unroll
        for (int nb = 0; nb < 4; ++nb) {
            *reinterpret_cast<float2*>(g + g4 * 32 + ((8 * nb + 2 * t4) ^ sw0)) =
                make_float2(gacc[nb][0], gacc[nb][1]);
            *reinterpret_cast<float2*>(g + (g4 + 8) * 32 + ((8 * nb + 2 * t4) ^ sw0)) =
                make_float2(gacc[nb][2], gacc[nb][3]);
        }
    }
    __syncwarp();
    const int sw0 = 8 * (g4 & 3);
    float mx0 = acc.m[0], mx1 = acc.m[1];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int j = 8 * nt + 2 * t4 + e;
            const bool ok = j < kvalid;
            const float b0 = g[g4 * 32 + ((j + 15 - g4) ^ sw0)];
            const float b1 = g[(g4 + 8) * 32 + ((j + 7 - g4) ^ sw0)];
            s[nt][e] = ok ? (s[nt][e] + b0) * scale_log2 : -INFINITY;
            s[nt][2 + e] = ok ? (s[nt][2 + e] + b1) * scale_log2 : -INFINITY;
        }
        mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    softmax_pv16(acc, s, vf, mx0, mx1, kvalid, lane);
}

// Position table of one CTA (Tp = 16 MT query rows of one head), built once before the key
// loop: G[i][c] = bf16(q_i + v) . rel[rho0 + c] for c in [0, ncols), rel rows outside [0, R)
// taken as zero, accumulated in fp32 and stored rounded to bf16 (a relative 2^-9 of the
// position term, the order of the bf16 rounding of P; half the shared memory of fp32, which
// lets four CTAs share an SM on short histories and five stages fit on long ones).  It is
// stored pre-skewed, G[i][c] at gs[i*W + c + i + 1], so that query i and key j
// (c = j + Tp - 1 - i) read gs[i*W + j + Tp]: one row of a slice's scores is one contiguous run.
// Warp `warp` of `nw` computes column tiles warp, warp + nw, ...  The head dimension is
// contracted in a permuted order: lane quad position t4 holds dims [16 t4, 16 t4 + 16) of
// both operands, so a lane's B fragments for one rel row are two 16-byte loads (rel is read
// from global memory; the table is the same for every stream and stays in L2).
// The rel rows of the first BATCH tiles are requested by load() (once the caller has the
// cache length), the rest by build() itself.  BATCH: column tiles of one warp whose rel
// rows are in flight together (10; 5 for the lighter three-CTAs-per-SM kernel).
template <int BATCH, int MT = 1>
struct PosTable {
    const uint16_t* rel_h;   // rel + h * 64
    long long stride;        // elements between rel rows
    int R, rho0, ncols, warp, nw, lane;
    uint4 bl[BATCH], bh[BATCH];

    __device__ __forceinline__ int ntiles() const { return (ncols + 7) >> 3; }

    __device__ __forceinline__ void load(int nb0)
    {
        const int g4 = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int rho = rho0 + 8 * (nb0 + u * nw) + g4;
            bl[u] = bh[u] = make_uint4(0u, 0u, 0u, 0u);
            if (nb0 + u * nw < ntiles() && rho >= 0 && rho < R) {
                const uint4* src = reinterpret_cast<const uint4*>(rel_h + rho * stride + 16 * t4);
                bl[u] = __ldg(src);
                bh[u] = __ldg(src + 1);
            }
        }
    }

    // A fragments of bf16(q + v) for m-tile mt (rows 16 mt ..), head dimension permuted
    __device__ __forceinline__ void make_a(uint32_t (&qa)[4][4], const uint8_t* q_tile,
                                           const float* v, int mt) const
    {
        const int g4 = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int row = 16 * mt + g4 + 8 * half;
            const uint4 c0 = *reinterpret_cast<const uint4*>(q_tile + swz128(row, 2 * t4));
            const uint4 c1 = *reinterpret_cast<const uint4*>(q_tile + swz128(row, 2 * t4 + 1));
            const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int d = 16 * t4 + 2 * m;
                // word m holds dims d, d+1: k-step m/2, k pair m%2 (a0/a1 pair 0, a2/a3 pair 1)
                qa[m >> 1][half + 2 * (m & 1)] =
                    pack_bf16(bf16_lo(w[m]) + v[d], bf16_hi(w[m]) + v[d + 1]);
            }
        }
    }

    // q_tile: the 128-byte-swizzled Q tile; v: the bias v in fp32 (smem).  load(warp) must
    // have been called.  Every m-tile's rows of a batch's columns use the batch's rel rows.
    __device__ __forceinline__ void build(uint16_t* gs, int W, const uint8_t* q_tile, const float* v)
    {
        uint32_t qa[MT][4][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) make_a(qa[mt], q_tile, v, mt);
        for (int nb0 = warp;;) {
            // the batch's tiles as independent MMA chains (tiles past the table have zero rel
            // rows and store nothing); a short batch runs the half-size version
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                if (nb0 + (BATCH / 2) * nw < ntiles())
                    tiles<BATCH>(gs, W, qa[mt], nb0, mt);
                else
                    tiles<BATCH / 2>(gs, W, qa[mt], nb0, mt);
            }
            nb0 += BATCH * nw;
            if (nb0 >= ntiles()) break;
            load(nb0);
        }
    }

    template <int N>
    __device__ __forceinline__ void tiles(uint16_t* gs, int W, const uint32_t (&qa)[4][4], int nb0,
                                          int mt)
    {
        const int g4 = lane >> 2, t4 = lane & 3;
        float c[N][4];
#pragma unroll
        for (int u = 0; u < N; ++u) {
            c[u][0] = c[u][1] = c[u][2] = c[u][3] = 0.f;
            mma_bf16_16816(c[u], qa[0], bl[u].x, bl[u].y);
        }
#pragma unroll
        for (int u = 0; u < N; ++u) mma_bf16_16816(c[u], qa[1], bl[u].z, bl[u].w);
#pragma unroll
        for (int u = 0; u < N; ++u) mma_bf16_16816(c[u], qa[2], bh[u].x, bh[u].y);
#pragma unroll
        for (int u = 0; u < N; ++u) mma_bf16_16816(c[u], qa[3], bh[u].z, bh[u].w);
#pragma unroll
        for (int u = 0; u < N; ++u) {
            const int col = 8 * (nb0 + u * nw) + 2 * t4;
            const int i = 16 * mt + g4;   // query row of c[u][0..1]; c[u][2..3] is row i + 8
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                if (col + e < ncols) {
                    gs[i * W + col + e + i + 1] = bf16_bits(c[u][e]);
                    gs[(i + 8) * W + col + e + i + 9] = bf16_bits(c[u][2 + e]);
                }
            }
        }
    }
};

// One warp, one 16-key slice, with the position term read from the CTA's pre-skewed table:
// gq points at gs + js + 16 for the slice's first key js, so key jl of query row i uses
// gq[i*W + jl].  k_s, v_s: the slice's 16 K and V rows (128-byte swizzled); keys
// [0, kvalid) of the slice exist.
// release_bar (non-zero): an mbarrier every lane arrives on as soon as its last read of the
// slice's K and V rows is done (the V fragments are in registers), so the slot can be refilled
// while the position term, softmax and P.V run.
__device__ __forceinline__ void warp_slice16_gt(WarpAcc& acc, const uint32_t (&qu)[4][4],
                                                uint32_t k_s, uint32_t v_s, const uint16_t* gq,
                                                int W, bool even, int kvalid, float scale_log2,
                                                int lane, uint32_t release_bar = 0)
{
    const int g4 = lane >> 2, t4 = lane & 3, mi = lane >> 3;
    float gb[2][4];   // [nt][row g4 cols 2t4, 2t4+1 | row g4+8 cols 2t4, 2t4+1]
    {
        const uint16_t* r0 = gq + g4 * W + 2 * t4;
        const uint16_t* r1 = r0 + 8 * W;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            if (even) {
                const uint32_t x = *reinterpret_cast<const uint32_t*>(r0 + 8 * nt);
                const uint32_t y = *reinterpret_cast<const uint32_t*>(r1 + 8 * nt);
                gb[nt][0] = bf16_lo(x);
                gb[nt][1] = bf16_hi(x);
                gb[nt][2] = bf16_lo(y);
                gb[nt][3] = bf16_hi(y);
            } else {
                gb[nt][0] = bf16_lo(r0[8 * nt]);
                gb[nt][1] = bf16_lo(r0[8 * nt + 1]);
                gb[nt][2] = bf16_lo(r1[8 * nt]);
                gb[nt][3] = bf16_lo(r1[8 * nt + 1]);
            }
        }
    }
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(k_s + swz128(((mi >> 1) << 3) + (lane & 7), 2 * ks + (mi & 1)), b0, b1, b2, b3);
        mma_bf16_16816(s[0], qu[ks], b0, b1);
        mma_bf16_16816(s[1], qu[ks], b2, b3);
    }
    uint32_t vf[4][4];
    const int vrow = ((mi & 1) << 3) + (lane & 7);
#pragma unroll
    for (int dp = 0; dp < 4; ++dp)
        ldsm_x4_t(v_s + swz128(vrow, 2 * dp + (mi >> 1)), vf[dp][0], vf[dp][1], vf[dp][2], vf[dp][3]);
    if (release_bar) mbar_arrive_release(release_bar);
    float mx0 = acc.m[0], mx1 = acc.m[1];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const bool ok = 8 * nt + 2 * t4 + e < kvalid;
            s[nt][e] = ok ? (s[nt][e] + gb[nt][e]) * scale_log2 : -INFINITY;
            s[nt][2 + e] = ok ? (s[nt][2 + e] + gb[nt][2 + e]) * scale_log2 : -INFINITY;
        }
        mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    softmax_pv16(acc, s, vf, mx0, mx1, kvalid, lane);
}

// Quad-reduce the row sums (each thread held its own columns' share).
__device__ __forceinline__ void acc_reduce_l(WarpAcc& acc)
{
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        acc.l[r] += __shfl_xor_sync(0xffffffffu, acc.l[r], 1);
        acc.l[r] += __shfl_xor_sync(0xffffffffu, acc.l[r], 2);
    }
}

// Write the warp's partial (O, m, l) of its 16 rows into comb_o [.][kOW], comb_m, comb_l at
// row offset r0 (call acc_reduce_l first).
__device__ __forceinline__ void write_partial(const WarpAcc& acc, float* comb_o, float* comb_m,
                                              float* comb_l, int r0, int lane)
{
    const int g4 = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int dt = 0; dt < 8; ++dt) {
        *reinterpret_cast<float2*>(comb_o + (r0 + g4) * kOW + 8 * dt + 2 * t4) =
            make_float2(acc.o[dt][0], acc.o[dt][1]);
        *reinterpret_cast<float2*>(comb_o + (r0 + g4 + 8) * kOW + 8 * dt + 2 * t4) =
            make_float2(acc.o[dt][2], acc.o[dt][3]);
    }
    if (t4 == 0) {
        comb_m[r0 + g4] = acc.m[0];
        comb_m[r0 + g4 + 8] = acc.m[1];
        comb_l[r0 + g4] = acc.l[0];
        comb_l[r0 + g4 + 8] = acc.l[1];
    }
}

// Merge the nparts partials of query row `row` (stride `pstride` rows between partials),
// dims [d0, d0+8), and return them as 8 bf16.
__device__ __forceinline__ uint4 combine_row8(const float* comb_o, const float* comb_m,
                                              const float* comb_l, int nparts, int pstride,
                                              int row, int d0)
{
    float mstar = -INFINITY;
    for (int k = 0; k < nparts; ++k) mstar = fmaxf(mstar, comb_m[k * pstride + row]);
    float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float L = 0.f;
    for (int k = 0; k < nparts; ++k) {
        const float mk = comb_m[k * pstride + row];
        const float w = (mk == -INFINITY) ? 0.f : ex2_approx(mk - mstar);
        L += w * comb_l[k * pstride + row];
        const float* src = comb_o + (k * pstride + row) * kOW + d0;
#pragma unroll
        for (int d = 0; d < 8; ++d) o[d] += w * src[d];
    }
    const float inv = 1.f / L;
    return make_uint4(pack_bf16(o[0] * inv, o[1] * inv), pack_bf16(o[2] * inv, o[3] * inv),
                      pack_bf16(o[4] * inv, o[5] * inv), pack_bf16(o[6] * inv, o[7] * inv));
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Arrive on named barrier `id` without waiting: the shared-memory writes this thread made
// before are visible to the threads that wait on it with named_bar_sync.
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

}  // namespace oasr
