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
// and walks items blockIdx.x, blockIdx.x + gridDim.x, ...  A producer warp streams each
// item's query tile (double-buffered) and its segment's keys in stages of 64 (one TMA box
// each for K, V and the rel band) into a ring of slots, running ahead across items; four
// consumer warps each own 16 query rows and run the per-warp unit of attn_core.cuh.
//
// f32 path: a SIMT kernel (one warp per query row).
#include "attn_core.cuh"
#include "host_common.h"

namespace oasr {
namespace {

constexpr int kMaxSeqs = 1024;
constexpr int kPackedNS = 2;

struct PackedArgs {
    const int32_t* cu_seqlens;
    const uint16_t* pos_bias_u;
    const uint16_t* pos_bias_v;
    uint16_t* out;
    unsigned* status;
    int num_seqs, total, H, z;
    float scale_log2;
};

// Shared-memory plan (byte offsets from a 1024-aligned base).  Slots as in the streaming
// kernel (K, V, rel band of one stage); two Q buffers (Q tile + that head's u and v, bf16)
// so the producer fetches the next work item's query tile while the current one runs.
template <int NS>
struct PackedSmem {
    using TL = Tile<4>;
    static constexpr int kBand = TL::RB * kRowBytes;
    static constexpr int kSlot = 2 * kStageKeys * kRowBytes + kBand;
    static constexpr int kQ = TL::Tp * kRowBytes;
    static constexpr int kQBuf = kQ + 2 * kHeadDim * 2 + 768;   // keep 1024 alignment
    static constexpr int off_slots = 0;
    static constexpr int off_q = NS * kSlot;
    static constexpr int off_g = off_q + 2 * kQBuf;
    static constexpr int off_cu = off_g + kConsumerWarps * kGBytes;
    static constexpr int off_tile = off_cu + (kMaxSeqs + 1) * 4;
    static constexpr int off_wsum = off_tile + (kMaxSeqs + 1) * 4;
    static constexpr int off_bar = off_wsum + 64;   // full[NS], empty[NS], qfull[2], qempty[2]
    static constexpr int bytes = off_bar + (2 * NS + 4) * 8 + 1024;
    static_assert(kSlot % 1024 == 0 && off_q % 1024 == 0 && kQBuf % 1024 == 0, "TMA tiles");
};

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

template <int NS>
__global__ void __launch_bounds__(kThreads, 2) packed_attn_bf16_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_r,
    const PackedArgs a)
{
    using TL = Tile<4>;
    using SP = PackedSmem<NS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned err = 0;
    int* s_cu = reinterpret_cast<int*>(sm + SP::off_cu);       // [num_seqs + 1]
    int* s_tile = reinterpret_cast<int*>(sm + SP::off_tile);   // [num_seqs + 1] tile prefix
    int* s_wsum = reinterpret_cast<int*>(sm + SP::off_wsum);
    const uint32_t bar_full = sb + SP::off_bar;
    const uint32_t bar_empty = bar_full + NS * 8;
    const uint32_t bar_qfull = bar_empty + NS * 8;
    const uint32_t bar_qempty = bar_qfull + 16;
    const int ns = a.num_seqs;

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, kConsumerWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_qfull + 8 * i, 1);
            mbar_init(bar_qempty + 8 * i, kConsumerWarps);
        }
        fence_mbar_init();
    }
    // Segment starts, clamped into [0, total].
    for (int i = tid; i <= ns; i += kThreads) {
        int c = __ldg(a.cu_seqlens + i);
        if (c < 0 || c > a.total) { err |= kErrBounds; c = c < 0 ? 0 : a.total; }
        s_cu[i] = c;
    }
    __syncthreads();
    // Exclusive prefix of per-segment 64-row tile counts (thread tid owns a run of segments).
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
    if (tid == kThreads - 1) {
        int t = 0;
        for (int w = 0; w < kThreads / 32; ++w) t += s_wsum[w];
        s_tile[ns] = t;
    }
    __syncthreads();
    const long long n_items = static_cast<long long>(s_tile[ns]) * a.H;

    // Work item -> (segment start, length, first query row, head).
    auto decode = [&](long long item, int& start, int& L, int& i0, int& h) {
        const int tile = static_cast<int>(item / a.H);
        h = static_cast<int>(item - static_cast<long long>(tile) * a.H);
        int lo = 0, hi = ns - 1;   // last segment with s_tile[s] <= tile
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_tile[mid] <= tile) lo = mid; else hi = mid - 1;
        }
        start = s_cu[lo];
        L = s_cu[lo + 1] - start;
        i0 = (tile - s_tile[lo]) * 64;
    };

    if (warp == kConsumerWarps) {
        // ---------------- producer
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            prefetch_tensormap(&tm_r);
            int gs = 0, it = 0;
            bool ok = true;
            for (long long item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
                int start, L, i0, h;
                decode(item, start, L, i0, h);
                const int qb = it & 1;
                if (it >= 2 && !mbar_wait(bar_qempty + 8 * qb, ((it >> 1) - 1) & 1)) { ok = false; break; }
                const uint32_t qbuf = sb + SP::off_q + qb * SP::kQBuf;
                mbar_arrive_expect_tx(bar_qfull + 8 * qb, SP::kQ + 2 * kHeadDim * 2);
                tma_load_3d(qbuf, &tm_q, bar_qfull + 8 * qb, 0, h, start + i0);
                bulk_load(qbuf + SP::kQ, a.pos_bias_u + h * kHeadDim, kHeadDim * 2, bar_qfull + 8 * qb);
                bulk_load(qbuf + SP::kQ + kHeadDim * 2, a.pos_bias_v + h * kHeadDim, kHeadDim * 2,
                          bar_qfull + 8 * qb);
                const int n_stages = (L + kStageKeys - 1) / kStageKeys;
                const int off = a.z - i0;
                for (int s = 0; s < n_stages; ++s, ++gs) {
                    const int slot = gs % NS;
                    if (gs >= NS && !mbar_wait(bar_empty + 8 * slot, ((gs / NS) - 1) & 1)) { ok = false; break; }
                    const uint32_t bar = bar_full + 8 * slot;
                    const uint32_t sbase = sb + SP::off_slots + slot * SP::kSlot;
                    const int j0 = s * kStageKeys;
                    mbar_arrive_expect_tx(bar, static_cast<uint32_t>((2 * kStageKeys + TL::RB) * kRowBytes));
                    tma_load_3d(sbase, &tm_k, bar, 0, h, start + j0);
                    tma_load_3d(sbase + kStageKeys * kRowBytes, &tm_v, bar, 0, h, start + j0);
                    tma_load_3d(sbase + 2 * kStageKeys * kRowBytes, &tm_r, bar, 0, h,
                                off + j0 - (TL::Tp - 1));
                }
            }
            if (!ok) err |= kErrTimeout;
        }
        if (err) atomicOr(a.status, err);
        return;
    }

    // -------------------- consumers: warp w owns query rows [16w, 16w+16) of every item
    float* gw = reinterpret_cast<float*>(sm + SP::off_g) + warp * (kGBytes / 4);
    int gs = 0, it = 0;
    bool failed = false;
    for (long long item = blockIdx.x; item < n_items; item += gridDim.x, ++it) {
        int start, L, i0, h;
        decode(item, start, L, i0, h);
        const int qb = it & 1;
        const uint32_t qbuf = sb + SP::off_q + qb * SP::kQBuf;
        if (!mbar_wait(bar_qfull + 8 * qb, (it >> 1) & 1)) { failed = true; break; }
        uint32_t qu[4][4], qv[4][4];
        {
            const uint16_t* uv = reinterpret_cast<const uint16_t*>(sm + SP::off_q + qb * SP::kQBuf + SP::kQ);
            float* u = gw;                 // scratch is free between items
            float* v = gw + kHeadDim;
            u[lane] = bf16_lo(uv[lane]);
            u[lane + 32] = bf16_lo(uv[lane + 32]);
            v[lane] = bf16_lo(uv[kHeadDim + lane]);
            v[lane + 32] = bf16_lo(uv[kHeadDim + lane + 32]);
            __syncwarp();
            make_q_frags(qbuf, u, v, warp, lane, qu, qv);
            __syncwarp();
        }
        if (lane == 0) mbar_arrive(bar_qempty + 8 * qb);
        WarpAcc acc;
        acc_init(acc);
        const int n_stages = (L + kStageKeys - 1) / kStageKeys;
        for (int s = 0; s < n_stages; ++s, ++gs) {
            const int slot = gs % NS;
            if (!mbar_wait(bar_full + 8 * slot, (gs / NS) & 1)) { failed = true; break; }
            const uint32_t sbase = sb + SP::off_slots + slot * SP::kSlot;
            warp_stage(acc, qu, qv, sbase, sbase + kStageKeys * kRowBytes,
                       sbase + 2 * kStageKeys * kRowBytes, TL::Tp - 16 - 16 * warp, gw,
                       min(kStageKeys, L - s * kStageKeys), a.scale_log2, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
        }
        if (failed) break;
        // normalise this warp's 16 rows, stage them as bf16 in the scratch, store 16 B per lane
        acc_reduce_l(acc);
        {
            const int g4 = lane >> 2, t4 = lane & 3;
            uint32_t* st = reinterpret_cast<uint32_t*>(gw);   // [16][32] words = 16 rows x 64 bf16
            const float i0l = 1.f / acc.l[0], i1l = 1.f / acc.l[1];
#pragma unroll
            for (int dt = 0; dt < 8; ++dt) {
                st[g4 * 32 + 4 * dt + t4] = pack_bf16(acc.o[dt][0] * i0l, acc.o[dt][1] * i0l);
                st[(g4 + 8) * 32 + 4 * dt + t4] = pack_bf16(acc.o[dt][2] * i1l, acc.o[dt][3] * i1l);
            }
            __syncwarp();
            const int row0 = i0 + 16 * warp;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int idx = lane + 32 * k;
                const int r = idx >> 3, c = idx & 7;
                if (row0 + r < L) {
                    const uint4 v = reinterpret_cast<const uint4*>(st)[r * 8 + c];
                    *reinterpret_cast<uint4*>(a.out + (static_cast<long long>(start + row0 + r) * a.H + h) *
                                                          kHeadDim + c * 8) = v;
                }
            }
            __syncwarp();
        }
    }
    if (failed) err |= kErrTimeout;
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
    constexpr int smem = PackedSmem<kPackedNS>::bytes;
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
