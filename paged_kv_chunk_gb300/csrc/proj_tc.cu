// The projections that feed the path, in one launch (oasr_project_qkv_pos):
//   q | k | v = x . W_qkv^T + b_qkv      ([M, 3 d] -> three [M, H, 64] tensors)
//   rel       = pos_emb . W_pos^T        ([R, d]   -> [R, H, 64])
// Model Layer page, fixed_attention_window row: one positional projection per step serves
// the whole cohort; the Conformer rel-pos attention's linear_q / linear_k / linear_v carry
// a bias and linear_pos does not.
//
// A grouped bf16 GEMM on the 5th-generation tensor cores.  Persistent CTAs (one per SM) walk
// one list of 128 x 128 output tiles (128 x 64 when the wide ones would occupy at most half
// the SMs): those of the q/k/v problem, then those of the positional one.  Warp 5 feeds a ring of {A tile, W tile} stages (64-wide K steps, TMA,
// 128-byte swizzle; the row-major inputs are viewed as [rows, K/64, 64]); one thread of warp 4
// issues tcgen05.mma M128 N128 K16 into one of two TMEM accumulators, so the epilogue of a
// tile overlaps the products of the next; warps 0-3 (one TMEM lane quadrant each, thread =
// output row) add the bias, round to bf16 and store their row's 128 columns straight into
// q, k, v or rel.  Every wait is bounded; a wait that runs out aborts the CTA's remaining
// work and raises the timeout bit, after which the CTA drains and frees its TMEM.
#include "attn_core.cuh"
#include "host_common.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace oasr {
namespace {

constexpr int kPM = 128, kPK = 64;   // output tile rows, K step (the tile's width PN is 128 or 64)
constexpr int kPStages = 4;
constexpr int kPThreads = 192;       // warps 0-3 epilogue, 4 MMA, 5 TMA

template <int PN>
struct ProjSmem {
    static constexpr int tile = kPM * kRowBytes;            // A: 16 KB (128 rows x 64 bf16)
    static constexpr int tile_w = PN * kRowBytes;           // W: PN rows x 64 bf16
    static constexpr int stage = tile + tile_w;
    static constexpr int off_ring = 0;
    static constexpr int off_misc = kPStages * stage;       // tmem base, abort flag
    static constexpr int off_bias = off_misc + 64;          // [4 warps][PN] fp32 tile bias
    static constexpr int off_bar = off_bias + 4 * PN * 4;
    static constexpr int n_bars = 2 * kPStages + 2 + 2 + 1;
    static constexpr int bytes = off_bar + n_bars * 8 + 1024;
    static constexpr int tmem_cols = 2 * PN;                // two accumulators
    static_assert(tile % 1024 == 0 && tile_w % 1024 == 0, "TMA tiles need 1024-byte alignment");
};

struct ProjArgs {
    const uint16_t* bias;   // [3 d] for the q/k/v problem
    uint16_t* out[4];       // q, k, v ([M0, d] each), rel ([M1, d])
    int M0, M1, d;          // rows of x, rows of pos_emb, d_model (the K of both problems)
    int nt0, nt1;           // n-tiles per row tile: 3 d / PN, d / PN
    int tiles0, tiles;      // tiles of the q/k/v problem, of both
    unsigned* status;
};

template <int PN>
__global__ void __launch_bounds__(kPThreads, 1) project_tc_kernel(
    const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wqkv,
    const __grid_constant__ CUtensorMap tm_pos, const __grid_constant__ CUtensorMap tm_wpos,
    const ProjArgs a)
{
    using SP = ProjSmem<PN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + SP::off_misc);
    volatile int* s_abort = reinterpret_cast<volatile int*>(sm + SP::off_misc + 4);
    const uint32_t bar_full = sb + SP::off_bar;                  // [kPStages] stage landed
    const uint32_t bar_empty = bar_full + 8 * kPStages;          // [kPStages] stage consumed
    const uint32_t bar_acc_full = bar_empty + 8 * kPStages;      // [2] accumulator ready
    const uint32_t bar_acc_free = bar_acc_full + 16;             // [2] accumulator read out
    const uint32_t bar_drain = bar_acc_free + 16;                // issuer's MMAs all finished
    const int ksteps = a.d / kPK;

    if (warp == 5 && lane == 0) {   // launch parameters: fetched before the previous grid ends
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_wqkv);
        prefetch_tensormap(&tm_pos);
        prefetch_tensormap(&tm_wpos);
    }
    if (tid == 0) {
        for (int i = 0; i < kPStages; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_acc_full + 8 * i, 1);
            mbar_init(bar_acc_free + 8 * i, 4);
        }
        mbar_init(bar_drain, 1);
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(s_tmem)),
                     "r"(SP::tmem_cols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    // the setup above overlaps the previous grid on the stream; inputs and outputs are
    // touched only after it has finished
    grid_dep_wait();

    // tile t -> problem, row tile, column tile
    auto decode = [&](int t, int& g, int& mt, int& nt) {
        if (t < a.tiles0) {
            g = 0;
            mt = t / a.nt0;
            nt = t - mt * a.nt0;
        } else {
            g = 1;
            t -= a.tiles0;
            mt = t / a.nt1;
            nt = t - mt * a.nt1;
        }
    };

    if (warp == 5) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int i = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < a.tiles && ok; t += gridDim.x) {
                int g, mt, nt;
                decode(t, g, mt, nt);
                for (int kb = 0; kb < ksteps; ++kb, ++i) {
                    const int slot = i % kPStages;
                    if (i >= kPStages &&
                        !wait_or_abort(bar_empty + 8 * slot, ((i / kPStages) - 1) & 1, s_abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t base = sb + SP::off_ring + slot * SP::stage;
                    const uint32_t bar = bar_full + 8 * slot;
                    mbar_arrive_expect_tx(bar, SP::stage);
                    tma_load_3d(base, g ? &tm_pos : &tm_x, bar, 0, kb, mt * kPM);
                    tma_load_3d(base + SP::tile, g ? &tm_wpos : &tm_wqkv, bar, 0, kb, nt * PN);
                }
            }
            // no copy may still be landing when the CTA exits
            for (int u = i - kPStages; u < i; ++u)
                if (u >= 0 && !mbar_wait(bar_full + 8 * (u % kPStages), (u / kPStages) & 1)) *s_abort = 1;
        }
    } else if (warp == 4) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t id = idesc(kPM, PN, 0);
            int i = 0, lt = 0, nacc = 0, nfree = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < a.tiles && ok; t += gridDim.x, ++lt) {
                const int buf = lt & 1;
                // the accumulator's previous tile has been read out
                if (lt >= 2 && !wait_or_abort(bar_acc_free + 8 * buf, ((lt >> 1) - 1) & 1, s_abort)) break;
                for (int kb = 0; kb < ksteps; ++kb, ++i) {
                    const int slot = i % kPStages;
                    if (!wait_or_abort(bar_full + 8 * slot, (i / kPStages) & 1, s_abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t base = sb + SP::off_ring + slot * SP::stage;
#pragma unroll
                    for (int k = 0; k < kPK / 16; ++k)
                        umma_ss(tmem + buf * PN, sdesc(base + 32 * k), sdesc(base + SP::tile + 32 * k), id,
                                (kb > 0 || k > 0) ? 1 : 0);
                    umma_commit(bar_empty + 8 * slot);
                    ++nfree;
                }
                if (!ok) break;
                umma_commit(bar_acc_full + 8 * buf);
                ++nacc;
            }
            // drain: every MMA issued has finished and every arrival it owes has landed
            umma_commit(bar_drain);
            bool drained = mbar_wait(bar_drain, 0);
            for (int u = nacc - 2; u < nacc; ++u)
                if (u >= 0) drained = mbar_wait(bar_acc_full + 8 * (u & 1), (u >> 1) & 1) && drained;
            for (int u = nfree - kPStages; u < nfree; ++u)
                if (u >= 0) drained = mbar_wait(bar_empty + 8 * (u % kPStages), (u / kPStages) & 1) && drained;
            if (!drained) *s_abort = 1;
        }
    } else {
        // --------------------------------------------------------------- epilogue
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * warp) << 16);
        float* s_bias = reinterpret_cast<float*>(sm + SP::off_bias) + warp * PN;   // this warp's
        int lt = 0;
        for (int t = blockIdx.x; t < a.tiles; t += gridDim.x, ++lt) {
            int g, mt, nt;
            decode(t, g, mt, nt);
            const int buf = lt & 1;
            // the tile's PN bias values, PN / 32 per lane, requested before the accumulator is
            // waited for (the previous tile's reads of them are this warp's own, done)
            if constexpr (PN == 128) {
                float4 b4 = make_float4(0.f, 0.f, 0.f, 0.f);
                if (g == 0) {
                    const uint2 w = __ldg(reinterpret_cast<const uint2*>(a.bias + nt * PN) + lane);
                    b4 = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
                }
                *reinterpret_cast<float4*>(s_bias + 4 * lane) = b4;
            } else {
                float2 b2 = make_float2(0.f, 0.f);
                if (g == 0) {
                    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(a.bias + nt * PN) + lane);
                    b2 = make_float2(bf16_lo(w), bf16_hi(w));
                }
                *reinterpret_cast<float2*>(s_bias + 2 * lane) = b2;
            }
            __syncwarp();
            const bool ok = __all_sync(0xffffffffu, wait_or_abort(bar_acc_full + 8 * buf, (lt >> 1) & 1, s_abort));
            if (!ok) break;
            tc_fence_after();
            const int row = mt * kPM + 32 * warp + lane;
            const int M = g ? a.M1 : a.M0;
#pragma unroll
            for (int c = 0; c < PN / 32; ++c) {
                uint32_t r[32];
                OASR_TMEM_LD32(tl + buf * PN + 32 * c, r);
                tmem_wait_ld();
                const int col = nt * PN + 32 * c;     // column of the problem's output
                float bias[32];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 b4 = *reinterpret_cast<const float4*>(s_bias + 32 * c + j);
                    bias[j] = b4.x;
                    bias[j + 1] = b4.y;
                    bias[j + 2] = b4.z;
                    bias[j + 3] = b4.w;
                }
                if (row < M) {
                    // q, k or v by the column's third (d is a multiple of 128, so a tile
                    // never straddles two of them); rel for the positional problem
                    const int which = g ? 3 : col / a.d;
                    const int cw = g ? col : col - which * a.d;
                    // a select rather than an indexed read keeps the parameter array out of
                    // local memory
                    uint16_t* ob = which == 0 ? a.out[0] : which == 1 ? a.out[1] : which == 2 ? a.out[2] : a.out[3];
                    uint4* dst = reinterpret_cast<uint4*>(ob + static_cast<long long>(row) * a.d + cw);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t p[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 8 * q4 + 2 * e;
                            p[e] = pack_bf16(__uint_as_float(r[j]) + bias[j], __uint_as_float(r[j + 1]) + bias[j + 1]);
                        }
                        dst[q4] = make_uint4(p[0], p[1], p[2], p[3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_acc_free + 8 * buf);
        }
    }
    grid_dep_trigger();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(SP::tmem_cols));
    }
    if (tid == 0 && *s_abort) atomicOr(a.status, kErrTimeout);
}

int g_smem_done_proj[2][64];

template <int PN>
oasr_status launch_proj(const void* x, const void* w_qkv, const void* b_qkv, const void* pos_emb,
                        const void* w_pos, void* q, void* k, void* v, void* rel, int M, int R,
                        int d_model, int sms, unsigned* status, cudaStream_t stream)
{
    CUtensorMap tm_x, tm_wqkv, tm_pos, tm_wpos;
    const int kb = d_model / kPK;   // the inputs as [rows, d/64, 64]
    if (!encode_rows_bf16(&tm_x, x, M, kb, kPM) || !encode_rows_bf16(&tm_wqkv, w_qkv, 3LL * d_model, kb, PN) ||
        !encode_rows_bf16(&tm_pos, pos_emb, R, kb, kPM) || !encode_rows_bf16(&tm_wpos, w_pos, d_model, kb, PN))
        return OASR_ERR_INVALID_ARG;
    constexpr int smem = ProjSmem<PN>::bytes;
    if (!ensure_smem(project_tc_kernel<PN>, smem, g_smem_done_proj[PN == 64])) return OASR_ERR_CUDA;
    ProjArgs a;
    a.bias = static_cast<const uint16_t*>(b_qkv);
    a.out[0] = static_cast<uint16_t*>(q);
    a.out[1] = static_cast<uint16_t*>(k);
    a.out[2] = static_cast<uint16_t*>(v);
    a.out[3] = static_cast<uint16_t*>(rel);
    a.M0 = M;
    a.M1 = R;
    a.d = d_model;
    a.nt0 = 3 * d_model / PN;
    a.nt1 = d_model / PN;
    a.tiles0 = ((M + kPM - 1) / kPM) * a.nt0;
    a.tiles = a.tiles0 + ((R + kPM - 1) / kPM) * a.nt1;
    a.status = status;
    const int grid = a.tiles < sms ? a.tiles : sms;
    return launch_pdl(project_tc_kernel<PN>, dim3(grid), dim3(kPThreads), smem, stream, tm_x,
                      tm_wqkv, tm_pos, tm_wpos, a);
}

}  // namespace
}  // namespace oasr

extern "C" oasr_status oasr_project_qkv_pos(const void* x, const void* w_qkv, const void* b_qkv,
                                            const void* pos_emb, const void* w_pos, void* q,
                                            void* k, void* v, void* rel, int M, int R,
                                            int d_model, int H, oasr_dtype dt, cudaStream_t stream)
{
    using namespace oasr;
    if (!x || !w_qkv || !b_qkv || !pos_emb || !w_pos || !q || !k || !v || !rel)
        return OASR_ERR_INVALID_ARG;
    if (M <= 0 || R <= 0 || d_model <= 0 || H <= 0) return OASR_ERR_INVALID_ARG;
    if (dt != OASR_BF16) return OASR_ERR_UNSUPPORTED;
    if (d_model != H * kHeadDim || d_model % 128) return OASR_ERR_UNSUPPORTED;
    const void* ptrs[] = {x, w_qkv, b_qkv, pos_emb, w_pos, q, k, v, rel};
    for (const void* p : ptrs)
        if (!aligned16(p)) return OASR_ERR_INVALID_ARG;
    unsigned* status = status_word();
    const int sms = sm_count();
    if (!status || !sms) return OASR_ERR_CUDA;
    // 128 x 128 output tiles, or 128 x 64 when the wide ones would leave most SMs idle (a
    // small step is latency bound: twice the tiles at half the work each)
    const long long tiles128 = ((M + kPM - 1LL) / kPM) * (3LL * d_model / 128) +
                               ((R + kPM - 1LL) / kPM) * (d_model / 128LL);
    if (2 * tiles128 <= sms)
        return launch_proj<64>(x, w_qkv, b_qkv, pos_emb, w_pos, q, k, v, rel, M, R, d_model, sms,
                               status, stream);
    return launch_proj<128>(x, w_qkv, b_qkv, pos_emb, w_pos, q, k, v, rel, M, R, d_model, sms,
                            status, stream);
}
