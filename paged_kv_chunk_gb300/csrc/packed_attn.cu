// Packed varlen bidirectional attention with the Transformer-XL relative-position term
// (oasr_packed_relattn_varlen).
//
// ASR Engine page, section 4.1: with sequence packing an offline micro-batch is one
// gapless varlen-attention row; Model Layer page, engine-facing surface table,
// forward_offline_packed.  Segment s owns rows [cu[s], cu[s+1]); query i and key j of
// the same segment score ((q_i+u).k_j + (q_i+v).rel[z + j - i]) * scale with
// z = (R - 1) / 2 (rel_shift order, Model Layer page, Nemotron ASR section).
//
// bf16 path: the persistent tcgen05/TMEM kernel of packed_tc.cu; with the chunked-limited
// window (an even head count, up to 511 segments), the packed mode of chunk_tc.cu.
// f32 path: a SIMT kernel here (one warp per query row).
#include "attn_core.cuh"
#include "host_common.h"

namespace oasr {
namespace {

constexpr int kMaxSeqs = 1024;
// ----------------------------------------------------------------------------- fp32

__global__ void __launch_bounds__(128) packed_attn_f32_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const int32_t* __restrict__ cu, int num_seqs, int total, const float* __restrict__ u,
    const float* __restrict__ vb, const float* __restrict__ rel, int R, int z,
    float* __restrict__ out, int H, float scale, int cs, int left, unsigned* status)
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
    // keys this query sees: the whole segment, or (cs > 0) its own chunk and `left` earlier ones
    const int kl = cs > 0 ? max(0, (i / cs - left) * cs) : 0;
    const int kh = cs > 0 ? min(L, (i / cs + 1) * cs) : L;
    const long long qo = (static_cast<long long>(t) * H + h) * kHeadDim;
    for (int d = lane; d < kHeadDim; d += 32) {
        s_qu[warp][d] = q[qo + d] + u[h * kHeadDim + d];
        s_qv[warp][d] = q[qo + d] + vb[h * kHeadDim + d];
    }
    __syncwarp();
    float m = -INFINITY, l = 0.f, o0 = 0.f, o1 = 0.f;
    for (int j0 = kl; j0 < kh; j0 += 32) {
        const int j = j0 + lane;
        float sc = -INFINITY;
        if (j < kh) {
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
        const float p = (j < kh) ? expf(sc - m_new) : 0.f;
        float psum = p;
#pragma unroll
        for (int o = 16; o; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
        l = l * alpha + psum;
        o0 *= alpha;
        o1 *= alpha;
        const int nj = min(32, kh - j0);
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

}  // namespace

oasr_status launch_packed_tc(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                             int num_seqs, int total, const void* pos_bias_u,
                             const void* pos_bias_v, const void* rel, int R, void* out, int H,
                             float scale, int cs, int left, cudaStream_t stream);
oasr_status launch_chunk_tc_packed(const void* q, const void* k, const void* v,
                                   const int32_t* cu_seqlens, int num_seqs, int total,
                                   const void* pos_bias_u, const void* pos_bias_v, const void* rel,
                                   int R, void* out, int H, float scale, int cs, int left,
                                   cudaStream_t stream);
}  // namespace oasr

namespace oasr {
namespace {

oasr_status packed_impl(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                        int num_seqs, int max_seqlen, int total, const void* pos_bias_u,
                        const void* pos_bias_v, const void* rel, int R, void* out, int H, int D,
                        float scale, int cs, int left, oasr_dtype dt, cudaStream_t stream)
{
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
            static_cast<const float*>(rel), R, z, static_cast<float*>(out), H, scale, cs, left,
            status);
        return launch_status();
    }
    if (cs > 0) {
        // the chunked-limited window: 64-query blocks of a head pair on the streaming tensor-core
        // kernel, whose stages cover the window's keys (about two per block); shapes it does not
        // take go to the packed kernel below
        const oasr_status st = launch_chunk_tc_packed(q, k, v, cu_seqlens, num_seqs, total,
                                                      pos_bias_u, pos_bias_v, rel, R, out, H,
                                                      scale, cs, left, stream);
        if (st != OASR_ERR_UNSUPPORTED) return st;
    }
    return launch_packed_tc(q, k, v, cu_seqlens, num_seqs, total, pos_bias_u, pos_bias_v, rel, R,
                            out, H, scale, cs, left, stream);
}

}  // namespace
}  // namespace oasr

extern "C" oasr_status oasr_packed_relattn_varlen(const void* q, const void* k, const void* v,
                                                  const int32_t* cu_seqlens, int num_seqs,
                                                  int max_seqlen, int total,
                                                  const void* pos_bias_u, const void* pos_bias_v,
                                                  const void* rel, int R, void* out, int H, int D,
                                                  float scale, oasr_dtype dt, cudaStream_t stream)
{
    return oasr::packed_impl(q, k, v, cu_seqlens, num_seqs, max_seqlen, total, pos_bias_u,
                             pos_bias_v, rel, R, out, H, D, scale, 0, 0, dt, stream);
}

extern "C" oasr_status oasr_packed_relattn_chunked(const void* q, const void* k, const void* v,
                                                   const int32_t* cu_seqlens, int num_seqs,
                                                   int max_seqlen, int total,
                                                   const void* pos_bias_u, const void* pos_bias_v,
                                                   const void* rel, int R, void* out, int H, int D,
                                                   float scale, int chunk_size, int left_chunks,
                                                   oasr_dtype dt, cudaStream_t stream)
{
    if (chunk_size < 1 || left_chunks < 0) return OASR_ERR_INVALID_ARG;
    return oasr::packed_impl(q, k, v, cu_seqlens, num_seqs, max_seqlen, total, pos_bias_u,
                             pos_bias_v, rel, R, out, H, D, scale, chunk_size, left_chunks, dt,
                             stream);
}
