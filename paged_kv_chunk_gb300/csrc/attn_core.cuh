// Per-stage warp compute shared by the streaming (paged) and packed (varlen) bf16
// attention kernels.
//
// A CTA of 4 warps owns one query tile of Tp = 16*MT rows of one head and walks the keys
// in stages of 64.  Warp w takes m-tile (w % MT) and the key slice (w / MT) of each stage
// (KG = 4/MT slices of NK = 64/KG keys).  Per stage and warp:
//
//   S  = Q . K^T + (u . k_j)                  mma.sync m16n8k16 bf16, fp32 accumulators
//                                              seeded with the per-key u.k_j (fp32)
//   G  = Q . Rband^T + (v . r_m)               the same for the rel rows of the band
//   S += G[i][j + 15 - i]                      rel_shift skew through a per-warp smem tile
//   S  = S * scale * log2(e), keys past the end masked to -inf
//   online softmax (running max/sum per row, fp32, exp2)
//   O += P . V                                 P rounded to bf16 in registers
//
// Score convention (Scheduler page, section 4.3; Model Layer page, fixed_attention_window
// row and Nemotron ASR section): s_ij = scale * ((q_i+u).k_j + (q_i+v).rel[rho]),
// rho = off + j - i, where the kernel chooses `off` for its mode.  The band loaded for a
// stage of keys [j0, j0+64) and query rows [i0, i0+Tp) is rel rows
// [off + j0 - i0 - (Tp-1), +64+Tp); warp (mt, kg) reads band columns starting at
// o_w = Tp - 16 - 16*mt + kg*NK, and element (i', jl) of its tile uses column jl + 15 - i'.
#pragma once

#include "ptx.cuh"

namespace oasr {

constexpr int kHeadDim = 64;    // head dimension of the tensor-core path
constexpr int kStageKeys = 64;  // keys per pipeline stage
constexpr int kRowBytes = 128;  // one bf16 row of kHeadDim
constexpr int kThreads = 128;   // 4 warps per CTA

template <int MT_>
struct Tile {
    static constexpr int MT = MT_;                // 16-row m-tiles per CTA
    static constexpr int KG = 4 / MT;             // key slices per stage
    static constexpr int NK = kStageKeys / KG;    // keys per warp per stage
    static constexpr int Tp = 16 * MT;            // padded query rows
    static constexpr int RB = kStageKeys + Tp;    // rel band rows per stage
    static constexpr int NBAND = NK + 16;         // band columns per warp
    static constexpr int GW = NBAND + 4;          // skew scratch row stride (floats)
    static constexpr int OW = kHeadDim + 4;       // combine scratch row stride (floats)
};

// Shared-memory plan (byte offsets from a 1024-byte aligned base).  K/V/R/Q tiles are
// written by TMA with 128-byte swizzling.  After the key loop the K/V stage area is
// reused for the cross-warp combine.
template <int MT, int NS, int EXTRA = 0>
struct SmemPlan {
    using TL = Tile<MT>;
    static constexpr int kKV = kStageKeys * kRowBytes;
    static constexpr int kR = TL::RB * kRowBytes;
    static constexpr int off_k = 0;
    static constexpr int off_v = off_k + NS * kKV;
    static constexpr int off_r = off_v + NS * kKV;
    static constexpr int off_q = off_r + NS * kR;
    static constexpr int off_g = off_q + TL::Tp * kRowBytes;
    static constexpr int off_uk = off_g + 4 * 16 * TL::GW * 4;
    static constexpr int off_vr = off_uk + NS * kStageKeys * 4;
    static constexpr int off_u = off_vr + NS * TL::RB * 4;
    static constexpr int off_vb = off_u + kHeadDim * 4;
    static constexpr int off_bar = off_vb + kHeadDim * 4;
    static constexpr int off_extra = off_bar + (NS + 1) * 8;
    static constexpr int bytes = off_extra + EXTRA + 1024;
    static constexpr int off_comb_o = off_k;
    static constexpr int off_comb_ml = off_k + TL::KG * TL::Tp * TL::OW * 4;
    static_assert(off_r % 1024 == 0 && off_q % 1024 == 0 && kR % 1024 == 0, "TMA tiles");
    static_assert(off_comb_ml + 2 * TL::KG * TL::Tp * 4 <= off_r, "combine area");
};

struct WarpAcc {
    float o[8][4];  // 16 rows x 64 dims: n-tile dt holds dims [8dt, 8dt+8)
    float m[2];     // running max (log2 units) of rows g and g+8
    float l[2];     // running sum (this thread's columns only)
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

// A fragments of the warp's 16 query rows (4 k-steps of 16 dims) from a swizzled Q tile.
__device__ __forceinline__ void load_q_frags(uint32_t q_s, int mt, int lane, uint32_t (&qa)[4][4])
{
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
        ldsm_x4(q_s + swz128(16 * mt + (lane & 15), 2 * ks + (lane >> 4)), qa[ks][0], qa[ks][1],
                qa[ks][2], qa[ks][3]);
}

// fp32 dot product of the 64-wide bf16 row `r` of a swizzled tile with vec (fp32, smem).
__device__ __forceinline__ float dot_row_bf16(const uint8_t* tile, int r, const float* vec)
{
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 raw = *reinterpret_cast<const uint4*>(tile + swz128(r, c));
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float lo = __uint_as_float(w[e] << 16);
            const float hi = __uint_as_float(w[e] & 0xffff0000u);
            acc = fmaf(lo, vec[8 * c + 2 * e], acc);
            acc = fmaf(hi, vec[8 * c + 2 * e + 1], acc);
        }
    }
    return acc;
}

// Cooperative per-stage prologue (all 128 threads): u.k for the stage's keys, v.r for its
// band rows, and zeroed V rows past the last valid key (their p is 0, but 0 * NaN is not).
template <int MT>
__device__ __forceinline__ void stage_prologue(const uint8_t* k_tile, uint8_t* v_tile,
                                               const uint8_t* r_tile, const float* s_u,
                                               const float* s_vb, float* uk, float* vr,
                                               int kvalid, int tid)
{
    using TL = Tile<MT>;
    if (tid < kStageKeys) {
        uk[tid] = (tid < kvalid) ? dot_row_bf16(k_tile, tid, s_u) : 0.f;
    } else {
        for (int r = tid - kStageKeys; r < TL::RB; r += kThreads - kStageKeys)
            vr[r] = dot_row_bf16(r_tile, r, s_vb);
    }
    if (kvalid < kStageKeys) {
        const int n16 = (kStageKeys - kvalid) * (kRowBytes / 16);
        uint4* base = reinterpret_cast<uint4*>(v_tile + kvalid * kRowBytes);
        for (int i = tid; i < n16; i += kThreads) base[i] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// One stage of one warp; see the file comment.  k_s, v_s, r_s: shared addresses of the
// stage's K (64 rows), V (64 rows) and band (RB rows) tiles.  gw: this warp's skew scratch.
template <int MT>
__device__ __forceinline__ void stage_compute(WarpAcc& acc, const uint32_t (&qa)[4][4],
                                              uint32_t k_s, uint32_t v_s, uint32_t r_s,
                                              const float* uk, const float* vr, float* gw,
                                              int kvalid, float scale_log2, int mt, int kg,
                                              int lane)
{
    using TL = Tile<MT>;
    constexpr int NK = TL::NK;
    constexpr int NT = NK / 8;            // key n-tiles
    constexpr int NB = TL::NBAND / 8;     // band n-tiles
    constexpr int GW = TL::GW;
    const int g4 = lane >> 2, t4 = lane & 3, mi = lane >> 3;
    const int kb = kg * NK;

    // ---- content scores, accumulators seeded with u.k_j
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const float2 ukv = *reinterpret_cast<const float2*>(uk + kb + 8 * nt + 2 * t4);
        s[nt][0] = ukv.x;
        s[nt][1] = ukv.y;
        s[nt][2] = ukv.x;
        s[nt][3] = ukv.y;
    }
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
            const int row = kb + 16 * np + ((mi >> 1) << 3) + (lane & 7);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(k_s + swz128(row, 2 * ks + (mi & 1)), b0, b1, b2, b3);
            mma_bf16_16816(s[2 * np], qa[ks], b0, b1);
            mma_bf16_16816(s[2 * np + 1], qa[ks], b2, b3);
        }
    }

    // ---- position scores on the band, seeded with v.r_m, staged for the skew
    const int ow = TL::Tp - 16 - 16 * mt + kb;
    {
        float gacc[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const float2 vv = *reinterpret_cast<const float2*>(vr + ow + 8 * nb + 2 * t4);
            gacc[nb][0] = vv.x;
            gacc[nb][1] = vv.y;
            gacc[nb][2] = vv.x;
            gacc[nb][3] = vv.y;
        }
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int np = 0; np < NB / 2; ++np) {
                const int row = ow + 16 * np + ((mi >> 1) << 3) + (lane & 7);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(r_s + swz128(row, 2 * ks + (mi & 1)), b0, b1, b2, b3);
                mma_bf16_16816(gacc[2 * np], qa[ks], b0, b1);
                mma_bf16_16816(gacc[2 * np + 1], qa[ks], b2, b3);
            }
        }
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            *reinterpret_cast<float2*>(gw + g4 * GW + 8 * nb + 2 * t4) =
                make_float2(gacc[nb][0], gacc[nb][1]);
            *reinterpret_cast<float2*>(gw + (g4 + 8) * GW + 8 * nb + 2 * t4) =
                make_float2(gacc[nb][2], gacc[nb][3]);
        }
    }
    __syncwarp();
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int jl = 8 * nt + 2 * t4 + e;
            s[nt][e] += gw[g4 * GW + jl + 15 - g4];
            s[nt][2 + e] += gw[(g4 + 8) * GW + jl + 7 - g4];
        }
    }
    __syncwarp();

    // ---- scale, mask, online softmax
    float mx0 = acc.m[0], mx1 = acc.m[1];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const bool ok = (kb + 8 * nt + 2 * t4 + e) < kvalid;
            s[nt][e] = ok ? s[nt][e] * scale_log2 : -INFINITY;
            s[nt][2 + e] = ok ? s[nt][2 + e] * scale_log2 : -INFINITY;
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
    const float alpha0 = exp2f(acc.m[0] - base0);
    const float alpha1 = exp2f(acc.m[1] - base1);
    acc.m[0] = mx0;
    acc.m[1] = mx1;
    acc.l[0] *= alpha0;
    acc.l[1] *= alpha1;
#pragma unroll
    for (int dt = 0; dt < 8; ++dt) {
        acc.o[dt][0] *= alpha0;
        acc.o[dt][1] *= alpha0;
        acc.o[dt][2] *= alpha1;
        acc.o[dt][3] *= alpha1;
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        s[nt][0] = exp2f(s[nt][0] - base0);
        s[nt][1] = exp2f(s[nt][1] - base0);
        s[nt][2] = exp2f(s[nt][2] - base1);
        s[nt][3] = exp2f(s[nt][3] - base1);
        acc.l[0] += s[nt][0] + s[nt][1];
        acc.l[1] += s[nt][2] + s[nt][3];
    }

    // ---- O += P . V
#pragma unroll
    for (int kk = 0; kk < NK / 16; ++kk) {
        const uint32_t pa[4] = {pack_bf16(s[2 * kk][0], s[2 * kk][1]),
                                pack_bf16(s[2 * kk][2], s[2 * kk][3]),
                                pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                                pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3])};
        const int row = kb + 16 * kk + ((mi & 1) << 3) + (lane & 7);
#pragma unroll
        for (int dp = 0; dp < 4; ++dp) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(v_s + swz128(row, 2 * dp + (mi >> 1)), b0, b1, b2, b3);
            mma_bf16_16816(acc.o[2 * dp], pa, b0, b1);
            mma_bf16_16816(acc.o[2 * dp + 1], pa, b2, b3);
        }
    }
}

// Write the warp's partial (O, m, l) into the combine area: comb_o [KG][Tp][OW],
// comb_m / comb_l [KG][Tp].  Call after the key loop's last __syncthreads.
template <int MT>
__device__ __forceinline__ void write_partial(WarpAcc& acc, float* comb_o, float* comb_m,
                                              float* comb_l, int mt, int kg, int lane)
{
    using TL = Tile<MT>;
    acc.l[0] += __shfl_xor_sync(0xffffffffu, acc.l[0], 1);
    acc.l[0] += __shfl_xor_sync(0xffffffffu, acc.l[0], 2);
    acc.l[1] += __shfl_xor_sync(0xffffffffu, acc.l[1], 1);
    acc.l[1] += __shfl_xor_sync(0xffffffffu, acc.l[1], 2);
    const int g4 = lane >> 2, t4 = lane & 3;
    const int r0 = kg * TL::Tp + 16 * mt + g4;
#pragma unroll
    for (int dt = 0; dt < 8; ++dt) {
        *reinterpret_cast<float2*>(comb_o + r0 * TL::OW + 8 * dt + 2 * t4) =
            make_float2(acc.o[dt][0], acc.o[dt][1]);
        *reinterpret_cast<float2*>(comb_o + (r0 + 8) * TL::OW + 8 * dt + 2 * t4) =
            make_float2(acc.o[dt][2], acc.o[dt][3]);
    }
    if (t4 == 0) {
        comb_m[r0] = acc.m[0];
        comb_m[r0 + 8] = acc.m[1];
        comb_l[r0] = acc.l[0];
        comb_l[r0 + 8] = acc.l[1];
    }
}

// Merge the KG partials of query row `row` (dims [d0, d0+8)) and return 8 bf16 packed.
template <int MT>
__device__ __forceinline__ uint4 combine_row8(const float* comb_o, const float* comb_m,
                                              const float* comb_l, int row, int d0)
{
    using TL = Tile<MT>;
    float mstar = -INFINITY;
#pragma unroll
    for (int k = 0; k < TL::KG; ++k) mstar = fmaxf(mstar, comb_m[k * TL::Tp + row]);
    float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float L = 0.f;
#pragma unroll
    for (int k = 0; k < TL::KG; ++k) {
        const float mk = comb_m[k * TL::Tp + row];
        const float w = (mk == -INFINITY) ? 0.f : exp2f(mk - mstar);
        L += w * comb_l[k * TL::Tp + row];
        const float* src = comb_o + (k * TL::Tp + row) * TL::OW + d0;
#pragma unroll
        for (int d = 0; d < 8; ++d) o[d] += w * src[d];
    }
    const float inv = 1.f / L;
    return make_uint4(pack_bf16(o[0] * inv, o[1] * inv), pack_bf16(o[2] * inv, o[3] * inv),
                      pack_bf16(o[4] * inv, o[5] * inv), pack_bf16(o[6] * inv, o[7] * inv));
}

}  // namespace oasr
