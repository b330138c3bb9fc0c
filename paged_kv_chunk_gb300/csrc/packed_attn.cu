// Packed varlen bidirectional attention with the Transformer-XL relative-position term
// (oasr_packed_relattn_varlen).
//
// ASR Engine page, section 4.1: with sequence packing an offline micro-batch is one
// gapless varlen-attention row; Model Layer page, engine-facing surface table,
// forward_offline_packed.  Segment s owns rows [cu[s], cu[s+1]); query i and key j of
// the same segment score ((q_i+u).k_j + (q_i+v).rel[z + j - i]) * scale with
// z = (R - 1) / 2 (rel_shift order, Model Layer page, Nemotron ASR section).
//
// bf16 path: a persistent kernel.  Work items are (query tile of 64 rows, head) over all
// segments; each CTA builds the per-segment tile prefix in shared memory from cu_seqlens
// and walks items blockIdx.x, blockIdx.x + gridDim.x, ...  An item streams its segment's
// keys in stages of 64 (one TMA box each for K, V and the rel band) through the same
// per-stage warp compute as the streaming kernel (attn_core.cuh) with four m-tiles.
//
// f32 path: a SIMT kernel (one warp per query row).
#include "attn_core.cuh"
#include "host_common.h"

namespace oasr {
namespace {

constexpr int kMaxSeqs = 1024;
constexpr int kPackedNS = 2;
constexpr int kPackedExtra = 2 * (kMaxSeqs + 1) * 4 + 64;

struct PackedArgs {
    const int32_t* cu_seqlens;
    const uint16_t* pos_bias_u;
    const uint16_t* pos_bias_v;
    uint16_t* out;
    unsigned* status;
    int num_seqs, total, H, z;
    float scale_log2;
};

template <int NS>
__global__ void __launch_bounds__(kThreads) packed_attn_bf16_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_r,
    const PackedArgs a)
{
    constexpr int MT = 4;
    using TL = Tile<MT>;
    using SP = SmemPlan<MT, NS, kPackedExtra>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned err = 0;
    int* s_cu = reinterpret_cast<int*>(sm + SP::off_extra);       // [num_seqs + 1]
    int* s_tile = s_cu + (kMaxSeqs + 1);                          // [num_seqs + 1] tile prefix
    int* s_wsum = s_tile + (kMaxSeqs + 1);                        // [4] warp totals
    float* s_u = reinterpret_cast<float*>(sm + SP::off_u);
    float* s_vb = reinterpret_cast<float*>(sm + SP::off_vb);
    const uint32_t bar_full = sb + SP::off_bar;
    const uint32_t bar_q = bar_full + NS * 8;
    const int ns = a.num_seqs;

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) mbar_init(bar_full + 8 * i, 1);
        mbar_init(bar_q, 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        prefetch_tensormap(&tm_r);
    }
    // Segment starts, clamped into [0, total] and made non-decreasing.
    for (int i = tid; i <= ns; i += kThreads) {
        int c = __ldg(a.cu_seqlens + i);
        if (c < 0 || c > a.total) { err |= kErrBounds; c = c < 0 ? 0 : a.total; }
        s_cu[i] = c;
    }
    __syncthreads();
    // Exclusive prefix of per-segment tile counts: thread tid owns segments
    // [tid*per, tid*per + per).
    const int per = (ns + kThreads - 1) / kThreads;
    int mine = 0;
    for (int k = 0; k < per; ++k) {
        const int sidx = tid * per + k;
        if (sidx < ns) {
            const int L = s_cu[sidx + 1] - s_cu[sidx];
            if (L < 0) err |= kErrBounds;
            mine += L > 0 ? (L + 63) / 64 : 0;
        }
    }
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int base = incl - mine;
    for (int w = 0; w < warp; ++w) base += s_wsum[w];
    for (int k = 0; k < per; ++k) {
        const int sidx = tid * per + k;
        if (sidx < ns) {
            s_tile[sidx] = base;
            const int L = s_cu[sidx + 1] - s_cu[sidx];
            base += L > 0 ? (L + 63) / 64 : 0;
        }
    }
    if (tid == kThreads - 1) s_tile[ns] = s_wsum[0] + s_wsum[1] + s_wsum[2] + s_wsum[3];
    __syncthreads();
    const int n_tiles = s_tile[ns];
    const long long n_items = static_cast<long long>(n_tiles) * a.H;

    const int mt = warp;   // KG = 1
    float* gw = reinterpret_cast<float*>(sm + SP::off_g) + warp * 16 * TL::GW;
    float* comb_o = reinterpret_cast<float*>(sm + SP::off_comb_o);
    float* comb_m = reinterpret_cast<float*>(sm + SP::off_comb_ml);
    float* comb_l = comb_m + TL::Tp;
    int gs = 0;        // stages consumed by this CTA so far (barrier phase bookkeeping)
    int items_done = 0;
    bool failed = false;

    for (long long item = blockIdx.x; item < n_items && !failed; item += gridDim.x, ++items_done) {
        const int tile = static_cast<int>(item / a.H);
        const int h = static_cast<int>(item - static_cast<long long>(tile) * a.H);
        // segment holding `tile`: last s with s_tile[s] <= tile (skips empty segments)
        int lo = 0, hi = ns - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_tile[mid] <= tile) lo = mid; else hi = mid - 1;
        }
        const int seg = lo;
        const int start = s_cu[seg];
        const int L = s_cu[seg + 1] - start;
        const int i0 = (tile - s_tile[seg]) * 64;
        const int n_stages = (L + kStageKeys - 1) / kStageKeys;
        const int off = a.z - i0;   // rho = off + j - i'   (i' local to the tile)

        auto issue = [&](int s, int g) {   // stage s of this item into buffer g % NS
            const int buf = g % NS;
            const uint32_t bar = bar_full + 8 * buf;
            const int j0 = s * kStageKeys;
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>((2 * kStageKeys + TL::RB) * kRowBytes));
            tma_load_3d(sb + SP::off_k + buf * SP::kKV, &tm_k, bar, 0, h, start + j0);
            tma_load_3d(sb + SP::off_v + buf * SP::kKV, &tm_v, bar, 0, h, start + j0);
            tma_load_3d(sb + SP::off_r + buf * SP::kR, &tm_r, bar, 0, h, off + j0 - (TL::Tp - 1));
        };
        const int pre = n_stages < NS ? n_stages : NS;
        if (tid == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bar_q, TL::Tp * kRowBytes);
            tma_load_3d(sb + SP::off_q, &tm_q, bar_q, 0, h, start + i0);
            for (int s = 0; s < pre; ++s) issue(s, gs + s);
        }
        if (tid < kHeadDim)
            s_u[tid] = __uint_as_float(static_cast<uint32_t>(__ldg(a.pos_bias_u + h * kHeadDim + tid)) << 16);
        else
            s_vb[tid - kHeadDim] = __uint_as_float(
                static_cast<uint32_t>(__ldg(a.pos_bias_v + h * kHeadDim + tid - kHeadDim)) << 16);
        uint32_t qa[4][4];
        WarpAcc acc;
        acc_init(acc);
        int s = 0;
        failed = __syncthreads_or(!mbar_wait(bar_q, items_done & 1));
        if (!failed) load_q_frags(sb + SP::off_q, mt, lane, qa);
        for (; s < n_stages && !failed; ++s) {
            const int g = gs + s;
            const int buf = g % NS;
            const bool ok = mbar_wait(bar_full + 8 * buf, (g / NS) & 1);
            const int kvalid = min(kStageKeys, L - s * kStageKeys);
            float* uk = reinterpret_cast<float*>(sm + SP::off_uk) + buf * kStageKeys;
            float* vr = reinterpret_cast<float*>(sm + SP::off_vr) + buf * TL::RB;
            if (ok)
                stage_prologue<MT>(sm + SP::off_k + buf * SP::kKV, sm + SP::off_v + buf * SP::kKV,
                                   sm + SP::off_r + buf * SP::kR, s_u, s_vb, uk, vr, kvalid, tid);
            if (__syncthreads_or(!ok)) { failed = true; break; }
            stage_compute<MT>(acc, qa, sb + SP::off_k + buf * SP::kKV,
                              sb + SP::off_v + buf * SP::kKV, sb + SP::off_r + buf * SP::kR, uk,
                              vr, gw, kvalid, a.scale_log2, mt, 0, lane);
            __syncthreads();
            if (tid == 0 && s + NS < n_stages) {
                fence_proxy_async_smem();
                issue(s + NS, g + NS);
            }
        }
        if (failed) {
            if (tid == 0) {
                const int issued = min(n_stages, s + NS);
                for (int s2 = s; s2 < issued; ++s2)
                    mbar_wait(bar_full + 8 * ((gs + s2) % NS), ((gs + s2) / NS) & 1, 100000000ull);
                err |= kErrTimeout;
            }
            break;
        }
        gs += n_stages;
        write_partial<MT>(acc, comb_o, comb_m, comb_l, mt, 0, lane);
        __syncthreads();
        const int rows = min(64, L - i0);
        for (int idx = tid; idx < rows * 8; idx += kThreads) {
            const int row = idx >> 3, d0 = (idx & 7) * 8;
            const uint4 v = combine_row8<MT>(comb_o, comb_m, comb_l, row, d0);
            *reinterpret_cast<uint4*>(a.out + (static_cast<long long>(start + i0 + row) * a.H + h) *
                                                  kHeadDim + d0) = v;
        }
        fence_proxy_async_smem();   // the next item's TMA overwrites the combine area
        __syncthreads();            // combine area and s_u reused by the next item
    }
    if (err) atomicOr(a.status, err);
}

// ----------------------------------------------------------------------------- fp32

__global__ void __launch_bounds__(128) packed_attn_f32_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const int32_t* __restrict__ cu, int num_seqs, int total, const float* __restrict__ u,
    const float* __restrict__ vb, const float* __restrict__ rel, int R, int z,
    float* __restrict__ out, int H, float scale, unsigned* status)
{
    __shared__ float s_qu[4][kHeadDim];
    __shared__ float s_qv[4][kHeadDim];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 4 + warp;
    const int h = blockIdx.y;
    if (t >= total) return;   // no block-wide barrier below
    // segment of token t: last s with cu[s] <= t
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int start = cu[lo];
    int end = cu[lo + 1];
    unsigned err = 0;
    if (end > total) { end = total; err |= kErrBounds; }
    if (t < start || t >= end) {   // token in no segment
        if (lane == 0) atomicOr(status, kErrBounds);
        return;
    }
    const int L = end - start, i = t - start;
    const long long qo = (static_cast<long long>(t) * H + h) * kHeadDim;
    for (int d = lane; d < kHeadDim; d += 32) {
        s_qu[warp][d] = q[qo + d] + u[h * kHeadDim + d];
        s_qv[warp][d] = q[qo + d] + vb[h * kHeadDim + d];
    }
    __syncwarp();
    float m = -INFINITY, l = 0.f, o0 = 0.f, o1 = 0.f;
    for (int j0 = 0; j0 < L; j0 += 32) {
        const int j = j0 + lane;
        float sc = -INFINITY;
        if (j < L) {
            const float4* kr =
                reinterpret_cast<const float4*>(k + (static_cast<long long>(start + j) * H + h) * kHeadDim);
            float acc = 0.f;
#pragma unroll 4
            for (int d4 = 0; d4 < kHeadDim / 4; ++d4) {
                const float4 kk = kr[d4];
                acc = fmaf(s_qu[warp][4 * d4], kk.x, acc);
                acc = fmaf(s_qu[warp][4 * d4 + 1], kk.y, acc);
                acc = fmaf(s_qu[warp][4 * d4 + 2], kk.z, acc);
                acc = fmaf(s_qu[warp][4 * d4 + 3], kk.w, acc);
            }
            const int rho = z + j - i;
            if (rho >= 0 && rho < R) {
                const float4* rr =
                    reinterpret_cast<const float4*>(rel + (static_cast<long long>(rho) * H + h) * kHeadDim);
#pragma unroll 4
                for (int d4 = 0; d4 < kHeadDim / 4; ++d4) {
                    const float4 r4 = rr[d4];
                    acc = fmaf(s_qv[warp][4 * d4], r4.x, acc);
                    acc = fmaf(s_qv[warp][4 * d4 + 1], r4.y, acc);
                    acc = fmaf(s_qv[warp][4 * d4 + 2], r4.z, acc);
                    acc = fmaf(s_qv[warp][4 * d4 + 3], r4.w, acc);
                }
            } else {
                err |= kErrBounds;
            }
            sc = acc * scale;
        }
        float mx = sc;
#pragma unroll
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_new = fmaxf(m, mx);
        const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
        const float p = (j < L) ? expf(sc - m_new) : 0.f;
        float psum = p;
#pragma unroll
        for (int o = 16; o; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
        l = l * alpha + psum;
        o0 *= alpha;
        o1 *= alpha;
        const int nj = min(32, L - j0);
        for (int jj = 0; jj < nj; ++jj) {
            const float pj = __shfl_sync(0xffffffffu, p, jj);
            const float* vr = v + (static_cast<long long>(start + j0 + jj) * H + h) * kHeadDim;
            o0 = fmaf(pj, vr[lane], o0);
            o1 = fmaf(pj, vr[lane + 32], o1);
        }
        m = m_new;
    }
    out[qo + lane] = o0 / l;
    out[qo + lane + 32] = o1 / l;
    if (err) atomicOr(status, err);
}

int g_smem_done_packed[64];

}  // namespace
}  // namespace oasr

extern "C" oasr_status oasr_packed_relattn_varlen(const void* q, const void* k, const void* v,
                                                  const int32_t* cu_seqlens, int num_seqs,
                                                  int max_seqlen, int total,
                                                  const void* pos_bias_u, const void* pos_bias_v,
                                                  const void* rel, int R, void* out, int H, int D,
                                                  float scale, oasr_dtype dt, cudaStream_t stream)
{
    using namespace oasr;
    if (!q || !k || !v || !cu_seqlens || !pos_bias_u || !pos_bias_v || !rel || !out)
        return OASR_ERR_INVALID_ARG;
    if (num_seqs <= 0 || max_seqlen <= 0 || total <= 0 || R <= 0 || H <= 0 || D <= 0)
        return OASR_ERR_INVALID_ARG;
    if (dt != OASR_F32 && dt != OASR_BF16) return OASR_ERR_UNSUPPORTED;
    if (D != kHeadDim || num_seqs > kMaxSeqs) return OASR_ERR_UNSUPPORTED;
    const void* ptrs[] = {q, k, v, pos_bias_u, pos_bias_v, rel, out};
    for (const void* p : ptrs)
        if (!aligned16(p)) return OASR_ERR_INVALID_ARG;
    unsigned* status = status_word();
    const int sms = sm_count();
    if (!status || !sms) return OASR_ERR_CUDA;
    const int z = (R - 1) / 2;
    if (dt == OASR_F32) {
        dim3 grid((total + 3) / 4, H);
        packed_attn_f32_kernel<<<grid, 128, 0, stream>>>(
            static_cast<const float*>(q), static_cast<const float*>(k),
            static_cast<const float*>(v), cu_seqlens, num_seqs, total,
            static_cast<const float*>(pos_bias_u), static_cast<const float*>(pos_bias_v),
            static_cast<const float*>(rel), R, z, static_cast<float*>(out), H, scale, status);
        return launch_status();
    }
    CUtensorMap tm_q, tm_k, tm_v, tm_r;
    if (!encode_rows_bf16(&tm_q, q, total, H, 64) || !encode_rows_bf16(&tm_k, k, total, H, 64) ||
        !encode_rows_bf16(&tm_v, v, total, H, 64) ||
        !encode_rows_bf16(&tm_r, rel, R, H, Tile<4>::RB))
        return OASR_ERR_INVALID_ARG;
    auto kern = packed_attn_bf16_kernel<kPackedNS>;
    constexpr int smem = SmemPlan<4, kPackedNS, kPackedExtra>::bytes;
    if (!ensure_smem(kern, smem, g_smem_done_packed)) return OASR_ERR_CUDA;
    PackedArgs a;
    a.cu_seqlens = cu_seqlens;
    a.pos_bias_u = static_cast<const uint16_t*>(pos_bias_u);
    a.pos_bias_v = static_cast<const uint16_t*>(pos_bias_v);
    a.out = static_cast<uint16_t*>(out);
    a.status = status;
    a.num_seqs = num_seqs;
    a.total = total;
    a.H = H;
    a.z = z;
    a.scale_log2 = scale * 1.4426950408889634f;
    const long long tiles_bound = (static_cast<long long>(total) + 63) / 64 + num_seqs;
    long long grid = tiles_bound * H;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    if (grid > static_cast<long long>(sms) * per_sm) grid = static_cast<long long>(sms) * per_sm;
    kern<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(tm_q, tm_k, tm_v, tm_r, a);
    return launch_status();
}
