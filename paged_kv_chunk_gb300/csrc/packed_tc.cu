// Packed varlen bidirectional rel-pos attention on the 5th-generation tensor cores
// (tcgen05 + TMEM), bf16.  Used by oasr_packed_relattn_varlen for bf16 inputs.
//
// ASR Engine page, section 4.1 (sequence packing: one gapless varlen row); Model Layer
// page, engine-facing surface table (forward_offline_packed) and Nemotron ASR section
// (Transformer-XL rel_shift).  Segment s owns rows [cu[s], cu[s+1]); query i and key j of
// one segment score s_ij = scale * ((q_i+u).k_j + (q_i+v).rel[z - (i - j)]), z = (R-1)/2.
//
// Persistent CTAs (one per SM) walk work items (128-query tile of a segment, head).  For a
// tile of 128 queries against a stage of 128 keys, in tensor memory (TMEM lane = query row):
//   S [128 x 128] = bf16(q+u) . K^T     columns [0,128)    tcgen05.mma M128 N128, A and B in smem
//   G [128 x 256] = bf16(q+v) . Band^T  columns [128,384)  M128 N256; the band is the 256 rel
//                   rows z - i0 + j0 - 127 ... the tile reaches, and row i, key j uses band
//                   row 127 - i + j
//   O [128 x 64] += P . V               columns [384,448)  M128 N64, A = P from TMEM, B = V
//                                                          as an MN-major smem operand
//   P [128 x 128] bf16                  columns [448,512)
// Warp roles (384 threads):
//   warps 0-7  softmax.  Warps w and w+4 share TMEM lane quadrant w and the 32 query rows in
//              it; warp w takes keys 0-63 of each stage, warp w+4 keys 64-127, and the pair
//              swaps row maxima and sums through shared memory.  Each thread loads its S half
//              row and the G columns its row reaches, releases S and G to the issuer, then
//              takes its skewed half row of G (rounded to bf16) through its own shared staging
//              tile;
//              masks keys past the segment; keeps the running max (O is rescaled in TMEM only
//              when the max grows by more than 2^8) and sum; writes its half row of bf16 P to TMEM; at
//              the end of the tile normalises and stores its half of the O row.
//   warp 8     S/G issuer (one thread): S and G of stage s+1 as soon as the softmax warps have
//              read stage s's.
//   warp 9     TMA producer of the q rows and of the K and band tiles of a two-slot ring: a
//              slot's K and band are refilled as soon as the S and G products that read them
//              have finished.
//   warp 10    TMA producer of the ring's V tiles: a slot's V is refilled once its last P.V has
//              finished.  With V on a thread of its own, the next K and band never wait behind
//              a V copy; S and G of a stage wait for K and band alone.
//   warp 11    P.V issuer (one thread): P.V of stage s once the softmax warps have written P.
// Every wait is bounded; a wait that runs out raises the timeout bit and aborts the CTA's
// remaining work, after which the CTA still drains its copies and tensor-core work and frees
// its TMEM.
#include "attn_core.cuh"
#include "host_common.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace oasr {
namespace {

constexpr int kTcMaxSeqs = 1024;
constexpr int kSoftmaxWarps = 8;
constexpr int kTcThreads = 32 * (kSoftmaxWarps + 4);
constexpr int kMmaWarp = kSoftmaxWarps, kTmaWarp = kSoftmaxWarps + 1, kVWarp = kSoftmaxWarps + 2,
              kPvWarp = kSoftmaxWarps + 3;
constexpr int kBM = 128;                 // queries per tile
constexpr int kBN = 128;                 // keys per stage
constexpr int kBand = 256;               // band rows per stage
constexpr int kTmemCols = 512;
constexpr int kColS = 0, kColG = 128, kColO = 384, kColP = 448;
constexpr int kStgWarpBytes = 4704;     // one warp's bf16 staging: 32 rows of 9 16-byte chunks

struct TcSmem {
    static constexpr int k_tile = kBN * kRowBytes;               // 16 KB
    static constexpr int band_tile = kBand * kRowBytes;          // 32 KB
    static constexpr int v_tile = kBN * kRowBytes;               // 16 KB
    static constexpr int slot = k_tile + band_tile + v_tile;     // 64 KB: K | band | V
    static constexpr int off_band = k_tile;
    static constexpr int off_v = k_tile + band_tile;
    static constexpr int off_slot = 0;                           // 2 slots
    static constexpr int off_qu = 2 * slot;                      // 16 KB
    static constexpr int off_qv = off_qu + kBM * kRowBytes;      // 16 KB
    static constexpr int off_qbuf = off_qv + kBM * kRowBytes;    // 16 KB: next item's q rows (TMA)
    static constexpr int off_stg = off_qbuf + kBM * kRowBytes;   // the softmax warps' staging
    static constexpr int off_xm = off_stg + kSoftmaxWarps * kStgWarpBytes;
    static constexpr int off_cu = off_xm + 2 * 2 * kBM * 4;      // [exchange parity][half][row]
    static constexpr int off_tile = off_cu + (kTcMaxSeqs + 1) * 4;
    static constexpr int off_misc = (off_tile + (kTcMaxSeqs + 1) * 4 + 15) & ~15;   // wsum[16], tmem, abort
    static constexpr int off_bar = (off_misc + 128 + 7) & ~7;
    static constexpr int n_bars = 2 + 2 + 8 + 4 + 2 + 2 + 2;
    static constexpr int bytes = off_bar + n_bars * 8 + 1024;
    static_assert(bytes <= 232448, "dynamic shared memory of one CTA");
};

struct TcArgs {
    const uint16_t* q;
    const int32_t* cu_seqlens;
    const uint16_t* pos_bias_u;
    const uint16_t* pos_bias_v;
    uint16_t* out;
    unsigned* status;
    int num_seqs, total, H, z;
    int cs, left;            // chunked-limited window (MASKED kernel): chunk frames, earlier chunks
    uint32_t sign;           // 0x80008000 when the scale is negative (q+u, q+v are negated)
    float scale_log2;        // |scale| * log2(e)
};

// lo += bf16 low half of pair, hi += bf16 high half, each rounded once in fp32 (a bf16 value
// widens to fp32 exactly, so this equals widening first and adding in fp32)
__device__ __forceinline__ void add_bf16x2_f32(float& lo, float& hi, uint32_t pair)
{
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "r"(pair));
}

// ------------------------------------------------------------------------ kernel

// A bounded wait: the first poll inline, the rest (sleeping polls, the abort flag, the time
// limit) out of line, so that the many wait sites cost a few instructions of code each (the
// kernel's roles run different code at once, and instruction fetch stalls them otherwise).
__device__ __noinline__ bool pt_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort)
{
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        // suspended until the phase completes, for 20 us at most between the checks below
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            return false;
        }
    }
}
__device__ __forceinline__ bool pt_wait(uint32_t bar, uint32_t parity, volatile int* abort)
{
    return mbar_try_wait(bar, parity) || pt_wait_slow(bar, parity, abort);
}
// The bounded waits of the CTA's final drain, out of line.
__device__ __noinline__ bool pt_drain_wait(uint32_t bar, uint32_t parity) { return mbar_wait(bar, parity); }

template <bool MASKED>
__global__ void __launch_bounds__(kTcThreads, 1) packed_attn_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_r, const TcArgs a)
{
    using SP = TcSmem;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived from the __shared__ array itself so that every access
    // through it stays a shared-space access
    uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned err = 0;
    int* s_cu = reinterpret_cast<int*>(sm + SP::off_cu);
    int* s_tile = reinterpret_cast<int*>(sm + SP::off_tile);
    int* s_wsum = reinterpret_cast<int*>(sm + SP::off_misc);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + SP::off_misc + 64);
    volatile int* s_abort = reinterpret_cast<volatile int*>(sm + SP::off_misc + 68);
    const uint32_t bar_full = sb + SP::off_bar;        // [2] the stage's K and band tiles landed
    const uint32_t bar_empty = bar_full + 16;          // [2] the slot's V tile free (after P.V)
    const uint32_t bar_sg_full = bar_empty + 16;       // S and G in TMEM
    const uint32_t bar_sg_free = bar_sg_full + 8;      // softmax warps have read S and G
    const uint32_t bar_p_full = bar_sg_free + 8;       // P written to TMEM
    const uint32_t bar_pv_done = bar_p_full + 8;       // P.V finished
    const uint32_t bar_q_ready = bar_pv_done + 8;      // bf16(q+u), bf16(q+v) written
    const uint32_t bar_q_free = bar_q_ready + 8;       // last S/G MMA of an item finished
    const uint32_t bar_drain = bar_q_free + 8;         // everything the S/G issuer issued finished
    const uint32_t bar_drain2 = bar_drain + 8;         // everything the P.V issuer issued finished
    const uint32_t bar_pair = bar_drain2 + 8;          // [4] softmax warp pair exchanged a value
    const uint32_t bar_qb_full = bar_pair + 32;        // q rows of the next item landed
    const uint32_t bar_qb_free = bar_qb_full + 8;      // softmax warps have read the q rows
    const uint32_t bar_kb_empty = bar_qb_free + 8;     // [2] the slot's K and band tiles read
    const uint32_t bar_v_full = bar_kb_empty + 16;     // [2] the stage's V tile landed
    const int ns = a.num_seqs;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_full + 8 * i, 1);
            mbar_init(bar_empty + 8 * i, 1);
        }
        mbar_init(bar_sg_full, 1);
        mbar_init(bar_sg_free, kSoftmaxWarps);
        mbar_init(bar_p_full, kSoftmaxWarps);
        mbar_init(bar_pv_done, 1);
        mbar_init(bar_q_ready, kSoftmaxWarps);
        mbar_init(bar_q_free, 1);
        mbar_init(bar_drain, 1);
        mbar_init(bar_drain2, 1);
        for (int i = 0; i < 4; ++i) mbar_init(bar_pair + 8 * i, 64);
        mbar_init(bar_qb_full, 1);
        mbar_init(bar_qb_free, kSoftmaxWarps);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_kb_empty + 8 * i, 1);
            mbar_init(bar_v_full + 8 * i, 1);
        }
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(s_tmem)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // segment starts and the exclusive prefix of per-segment 128-row tile counts
    for (int i = tid; i <= ns; i += kTcThreads) {
        int c = __ldg(a.cu_seqlens + i);
        if (c < 0 || c > a.total) { err |= kErrBounds; c = c < 0 ? 0 : a.total; }
        s_cu[i] = c;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    {
        const int per = (ns + kTcThreads - 1) / kTcThreads;
        int mine = 0;
        for (int k = 0; k < per; ++k) {
            const int s = tid * per + k;
            if (s < ns) {
                const int L = s_cu[s + 1] - s_cu[s];
                if (L < 0) err |= kErrBounds;
                mine += L > 0 ? (L + kBM - 1) / kBM : 0;
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
            const int s = tid * per + k;
            if (s < ns) {
                s_tile[s] = base;
                const int L = s_cu[s + 1] - s_cu[s];
                base += L > 0 ? (L + kBM - 1) / kBM : 0;
            }
        }
        if (tid == kTcThreads - 1) {
            int t = 0;
            for (int w = 0; w < kTcThreads / 32; ++w) t += s_wsum[w];
            s_tile[ns] = t;
        }
        __syncthreads();
    }
    const long long n_items = static_cast<long long>(s_tile[ns]) * a.H;
    // item -> segment start and length, first query of the tile, head, and the keys
    // [kl, kh) the tile's queries can see (the whole segment, or with the chunked-limited
    // window the chunks from the first query's window start to the last query's chunk)
    // The unmasked kernel finds the segment by scanning on from the caller's previous one
    // (`seg`, starting at 0: each role visits its items in increasing order); the masked one,
    // whose softmax warps have no register to spare for it, by binary search.
    auto decode = [&](long long item, int& seg, int& start, int& L, int& i0, int& h, int& kl,
                      int& kh) {
        const int tile = static_cast<int>(item / a.H);
        h = static_cast<int>(item - static_cast<long long>(tile) * a.H);
        int lo = 0;
        if (!MASKED) {
            while (seg + 1 < ns && s_tile[seg + 1] <= tile) ++seg;
            lo = seg;
        } else {
            int hi = ns - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_tile[mid] <= tile) lo = mid; else hi = mid - 1;
            }
        }
        start = s_cu[lo];
        L = s_cu[lo + 1] - start;
        i0 = (tile - s_tile[lo]) * kBM;
        kl = 0;
        kh = L;
        if (MASKED) {
            const int ilast = (i0 + kBM < L ? i0 + kBM : L) - 1;
            kl = (i0 / a.cs - a.left) * a.cs;
            kl = kl > 0 ? kl : 0;
            kh = (ilast / a.cs + 1) * a.cs;
            kh = kh < L ? kh : L;
        }
    };

    // The TMA producers wait on the barrier itself (suspended until its phase completes), so
    // that they react at once and take no issue slots from the softmax warps meanwhile.
    auto prod_wait = [&](uint32_t bar, uint32_t parity, volatile int* abort) {
        return pt_wait(bar, parity, abort);
    };
    // Softmax warps take every wait together: a warp-wide vote keeps the warp converged for
    // the .sync.aligned tensor-memory instructions even if one lane's wait runs out.
    auto warp_wait = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xffffffffu, pt_wait(bar, parity, s_abort)) != 0;
    };

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            prefetch_tensormap(&tm_r);
            const uint64_t pol = policy_evict_last();   // K/V tiles are re-read by every query tile
            int g = 0, itp = 0;
            bool ok = true;
            int seg = 0;
            for (long long item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++itp) {
                int start, L, i0, h, kl, kh;
                decode(item, seg, start, L, i0, h, kl, kh);
                const int n_st = (kh - kl + kBN - 1) / kBN;
                // the item's 128 q rows, once the softmax warps have read the previous ones
                if (itp > 0 && !prod_wait(bar_qb_free, (itp - 1) & 1, s_abort)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar_qb_full, kBM * kRowBytes);
                tma_load_3d(sb + SP::off_qbuf, &tm_q, bar_qb_full, 0, h, start + i0);
                for (int s = 0; s < n_st; ++s, ++g) {
                    // K and band as soon as the S and G products that read the slot's last ones
                    // have finished
                    const int slot = g & 1;
                    if (g >= 2 && !prod_wait(bar_kb_empty + 8 * slot, ((g >> 1) - 1) & 1, s_abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t base = sb + SP::off_slot + slot * SP::slot;
                    const uint32_t bar = bar_full + 8 * slot;
                    mbar_arrive_expect_tx(bar, SP::k_tile + SP::band_tile);
                    const int js = kl + s * kBN;   // first key of the stage
                    tma_load_3d_hint(base, &tm_k, bar, 0, h, start + js, pol);
                    tma_load_3d(base + SP::off_band, &tm_r, bar, 0, h, a.z - i0 + js - (kBM - 1));
                }
            }
            // no copy may still be landing when the CTA exits
            for (int u = g - 2; u < g; ++u)
                if (u >= 0 && !pt_drain_wait(bar_full + 8 * (u & 1), (u >> 1) & 1)) *s_abort = 1;
            if (itp > 0 && !pt_drain_wait(bar_qb_full, (itp - 1) & 1)) *s_abort = 1;
        }
    } else if (warp == kVWarp) {
        // ---------------------------------------------------------- V producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            int g = 0, seg = 0;
            bool ok = true;
            for (long long item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
                int start, L, i0, h, kl, kh;
                decode(item, seg, start, L, i0, h, kl, kh);
                const int n_st = (kh - kl + kBN - 1) / kBN;
                for (int s = 0; s < n_st; ++s, ++g) {
                    const int slot = g & 1;
                    if (g >= 2 && !prod_wait(bar_empty + 8 * slot, ((g >> 1) - 1) & 1, s_abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar_v_full + 8 * slot, SP::v_tile);
                    tma_load_3d_hint(sb + SP::off_slot + slot * SP::slot + SP::off_v, &tm_v,
                                     bar_v_full + 8 * slot, 0, h, start + kl + s * kBN, pol);
                }
            }
            for (int u = g - 2; u < g; ++u)
                if (u >= 0 && !pt_drain_wait(bar_v_full + 8 * (u & 1), (u >> 1) & 1)) *s_abort = 1;
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ S/G issuer
        // Each tcgen05.mma holds its issuing thread until the tensor pipe takes it, so S/G and
        // P.V are issued from two threads: while one waits on a barrier the other's products run.
        // S and G of a stage (possibly the next item's first) go as soon as the previous stage's
        // have been read, so they overlap that stage's softmax and, across items, the previous
        // tile's last stage and epilogue.
        if (lane == 0) {
            constexpr uint32_t id_s = idesc(kBM, kBN, 0), id_g = idesc(kBM, kBand, 0);
            int x = 0, nq = 0, it = 0, seg = 0;   // x: stages issued
            int kbn[2] = {0, 0};                  // commits to each slot's K-and-band barrier
            bool ok = true;
            for (long long item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++it) {
                int start, L, i0, h, kl, kh;
                decode(item, seg, start, L, i0, h, kl, kh);
                const int n_st = (kh - kl + kBN - 1) / kBN;
                for (int s = 0; s < n_st; ++s, ++x) {
                    ok = (s > 0 || pt_wait(bar_q_ready, it & 1, s_abort)) &&
                         pt_wait(bar_full + 8 * (x & 1), (x >> 1) & 1, s_abort) &&
                         (x == 0 || pt_wait(bar_sg_free, (x - 1) & 1, s_abort));
                    if (!ok) break;
                    const int slot = x & 1;
                    const uint32_t base = sb + SP::off_slot + slot * SP::slot;
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_ss(tmem + kColS, sdesc(sb + SP::off_qu + 32 * k), sdesc(base + 32 * k), id_s, k > 0);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_ss(tmem + kColG, sdesc(sb + SP::off_qv + 32 * k),
                                sdesc(base + SP::off_band + 32 * k), id_g, k > 0);
                    umma_commit(bar_sg_full);
                    umma_commit(bar_kb_empty + 8 * slot);   // the slot's K and band may be refilled
                    ++kbn[slot];
                    if (s + 1 == n_st) { umma_commit(bar_q_free); ++nq; }   // the Qu/Qv tiles are free
                }
            }
            // drain: every product issued here has finished and every arrival it owes has landed
            umma_commit(bar_drain);
            bool drained = pt_drain_wait(bar_drain, 0);
            if (nq > 0) drained = pt_drain_wait(bar_q_free, (nq - 1) & 1) && drained;
            if (x > 0) drained = pt_drain_wait(bar_sg_full, (x - 1) & 1) && drained;
            for (int sl = 0; sl < 2; ++sl)
                if (kbn[sl] > 0) drained = pt_drain_wait(bar_kb_empty + 8 * sl, (kbn[sl] - 1) & 1) && drained;
            if (!drained) *s_abort = 1;
        }
    } else if (warp == kPvWarp) {
        // ------------------------------------------------------------ P.V issuer
        if (lane == 0) {
            constexpr uint32_t id_o = idesc(kBM, 64, 1);
            int g = 0, seg = 0;
            bool ok = true;
            for (long long item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
                int start, L, i0, h, kl, kh;
                decode(item, seg, start, L, i0, h, kl, kh);
                const int n_keys = kh - kl;
                const int n_st = (n_keys + kBN - 1) / kBN;
                for (int s = 0; s < n_st; ++s, ++g) {
                    ok = pt_wait(bar_p_full, g & 1, s_abort) &&
                         pt_wait(bar_v_full + 8 * (g & 1), (g >> 1) & 1, s_abort);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t vbase = sb + SP::off_slot + (g & 1) * SP::slot + SP::off_v;
                    // only the 16-key steps that hold keys of the segment (a partial last stage
                    // stops early, so V rows past them are never read)
                    const int kst = n_keys - s * kBN;
                    const int ksteps = kst < kBN ? (kst + 15) >> 4 : kBN / 16;
#pragma unroll
                    for (int k = 0; k < kBN / 16; ++k)
                        if (k < ksteps)
                            umma_ts(tmem + kColO, tmem + kColP + 8 * k, sdesc(vbase + 2048 * k), id_o,
                                    (s > 0 || k > 0) ? 1 : 0);
                    umma_commit(bar_pv_done);
                    umma_commit(bar_empty + 8 * (g & 1));
                }
            }
            umma_commit(bar_drain2);
            bool drained = pt_drain_wait(bar_drain2, 0);
            if (g > 0) drained = pt_drain_wait(bar_pv_done, (g - 1) & 1) && drained;
            for (int u = g - 2; u < g; ++u)
                if (u >= 0) drained = pt_drain_wait(bar_empty + 8 * (u & 1), (u >> 1) & 1) && drained;
            if (!drained) *s_abort = 1;
        }
    } else if (warp < kSoftmaxWarps) {
        // ----------------------------------------------------------------- softmax
        const int quad = warp & 3, hf = warp >> 2;
        const int r = 32 * quad + lane;         // query row within the tile == TMEM lane
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * quad) << 16);
        // The two warps of a quadrant swap one value per row through shared memory; the
        // pair's mbarrier phase k completes when both have written exchange k.
        float* xm = reinterpret_cast<float*>(sm + SP::off_xm);   // [exchange parity][half][row]
        const uint32_t pbar = bar_pair + 8 * quad;
        int nx = 0;
        auto pair_post = [&](float mine) {
            xm[(nx & 1) * (2 * kBM) + hf * kBM + r] = mine;
            mbar_arrive(pbar);
        };
        auto pair_collect = [&](float& theirs) {
            if (!warp_wait(pbar, nx & 1)) return false;
            theirs = xm[(nx & 1) * (2 * kBM) + (1 - hf) * kBM + r];
            ++nx;
            return true;
        };
        // bf16(q+u) and bf16(q+v) of item number itq (head hq): this thread's half row, from
        // the q rows the TMA warp staged; the caller has made sure the MMAs of the previous
        // item no longer read the Qu/Qv tiles
        auto prep_q = [&](int itq, int hq) {
            if (!warp_wait(bar_qb_full, itq & 1)) return false;
            const uint4* up = reinterpret_cast<const uint4*>(a.pos_bias_u + hq * kHeadDim);
            const uint4* vp = reinterpret_cast<const uint4*>(a.pos_bias_v + hq * kHeadDim);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int c = 4 * hf + cc;
                const uint32_t offs = static_cast<uint32_t>(r * kRowBytes + ((c ^ (r & 7)) << 4));
                const uint4 qc = *reinterpret_cast<const uint4*>(sm + SP::off_qbuf + offs);
                const uint4 uc = __ldg(up + c);
                const uint4 vc = __ldg(vp + c);
                const uint32_t w[4] = {qc.x, qc.y, qc.z, qc.w};
                const uint32_t wu[4] = {uc.x, uc.y, uc.z, uc.w};
                const uint32_t wv[4] = {vc.x, vc.y, vc.z, vc.w};
                uint32_t ou[4], ov[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
                    ou[e] = pack_bf16(lo + __uint_as_float(wu[e] << 16), hi + __uint_as_float(wu[e] & 0xffff0000u));
                    ov[e] = pack_bf16(lo + __uint_as_float(wv[e] << 16), hi + __uint_as_float(wv[e] & 0xffff0000u));
                    ou[e] ^= a.sign;   // a negative scale: negate q+u and q+v (exact in bf16)
                    ov[e] ^= a.sign;
                }
                *reinterpret_cast<uint4*>(sm + SP::off_qu + offs) = make_uint4(ou[0], ou[1], ou[2], ou[3]);
                *reinterpret_cast<uint4*>(sm + SP::off_qv + offs) = make_uint4(ov[0], ov[1], ov[2], ov[3]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_qb_free);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_q_ready);
            return true;
        };
        int g = 0, it = 0, sg = 0, seg = 0;
        if (static_cast<long long>(blockIdx.x) < n_items) {
            int st0, L0, i00, h0, kl0, kh0;
            decode(blockIdx.x, seg, st0, L0, i00, h0, kl0, kh0);
            if (!prep_q(0, h0)) *s_abort = 1;
        }
        // O rows of a finished item: wait for its last P.V, combine the pair's sums, store.
        // It runs inside the next item's first stage, after that stage's S/G have been read,
        // so the wait for the last P.V overlaps useful work.
        auto epilogue = [&](int e_start, int e_L, int e_i0, int e_h, float e_l) {
            if (!warp_wait(bar_pv_done, (g - 1) & 1)) return false;
            float l_other;
            pair_post(e_l);
            if (!pair_collect(l_other)) return false;
            const float l_row = e_l + l_other;
            tc_fence_after();
            uint32_t oo[32];
            OASR_TMEM_LD32(tl + kColO + 32 * hf, oo);
            tmem_wait_ld();
            const int row = e_i0 + r;
            if (row < e_L) {
                const float inv = 1.f / l_row;
                uint4* dst = reinterpret_cast<uint4*>(
                                 a.out + (static_cast<long long>(e_start + row) * a.H + e_h) * kHeadDim) + 4 * hf;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    dst[c] = make_uint4(
                        pack_bf16(__uint_as_float(oo[8 * c]) * inv, __uint_as_float(oo[8 * c + 1]) * inv),
                        pack_bf16(__uint_as_float(oo[8 * c + 2]) * inv, __uint_as_float(oo[8 * c + 3]) * inv),
                        pack_bf16(__uint_as_float(oo[8 * c + 4]) * inv, __uint_as_float(oo[8 * c + 5]) * inv),
                        pack_bf16(__uint_as_float(oo[8 * c + 6]) * inv, __uint_as_float(oo[8 * c + 7]) * inv));
            }
            tc_fence_before();
            return true;
        };
        int p_start = 0, p_L = 0, p_i0 = 0, p_h = 0;
        float p_l = 0.f;
        bool have_prev = false, all_ok = true;
        for (long long item = blockIdx.x; item < n_items && !*s_abort; item += gridDim.x, ++it) {
            int start, L, i0, h, kl, kh;
            decode(item, seg, start, L, i0, h, kl, kh);
            const int n_st = (kh - kl + kBN - 1) / kBN;
            float m_used = -INFINITY, l_sum = 0.f;
            bool ok = true;
            for (int s = 0; s < n_st; ++s, ++g) {
                if (!warp_wait(bar_sg_full, sg & 1)) { ok = false; break; }
                ++sg;
                tc_fence_after();
                uint8_t* slot_p = sm + SP::off_slot + (g & 1) * SP::slot;
                // the half holds keys jh .. jh+63; row r sees [ka, kb) of them.  Under the
                // chunked-limited window a warp whose rows see none of them skips the half (it
                // still releases S/G, exchanges -inf and writes P = 0)
                const int jh = kl + s * kBN + 64 * hf;
                int ka = 0, kb = kh - jh;
                if (MASKED) {
                    const int ci = (i0 + r) / a.cs;
                    const int lo = (ci - a.left) * a.cs - jh, hi = (ci + 1) * a.cs - jh;
                    ka = lo > 0 ? lo : 0;
                    kb = hi < kb ? hi : kb;
                }
                const bool live = !MASKED || __any_sync(0xffffffffu, ka < kb && ka < 64 && kb > 0);
                float sc[64];
                // position term, skewed: row r needs G[r][127 - r + j].  This warp's rows reach
                // 95 columns of G for this half (row r, key j of the half: window column
                // 31 - lane + j), which go through this warp's shared staging tile as bf16 pairs.
                // Lane reads words w0 .. w0+32 (w0 = (31 - lane) / 2), so it stores only the
                // 16-byte chunks q0 .. q0+8 (q0 = w0 / 4) of the window, from a row base of
                // 4 (9 lane + 2 (lane / 8)) words: the eight lanes of a store phase share q0 and
                // land in distinct bank quads, and the lane-shifted 4-byte loads hit 32 distinct
                // banks.  An even lane's window starts on the odd half of word w0, so its pairs
                // are realigned with a byte permute.
                const int w0 = (31 - lane) >> 1;
                const int q0 = w0 >> 2;
                uint32_t* stg = reinterpret_cast<uint32_t*>(sm + SP::off_stg + warp * kStgWarpBytes) +
                                4 * (9 * lane + 2 * (lane >> 3));
                if (live) {
                    uint32_t gr[96];
                    const uint32_t colg = kColG + static_cast<uint32_t>(96 - 32 * quad + 64 * hf);
                    OASR_TMEM_LD32(tl + colg, gr);
                    OASR_TMEM_LD32(tl + colg + 32, (gr + 32));
                    OASR_TMEM_LD32(tl + colg + 64, (gr + 64));
                    tmem_wait_ld();
#pragma unroll
                    for (int pc = 0; pc < 12; ++pc)
                        if (pc >= q0 && pc <= q0 + 8) {
                            uint32_t gw[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                gw[e] = pack_bf16(__uint_as_float(gr[8 * pc + 2 * e]),
                                                  __uint_as_float(gr[8 * pc + 2 * e + 1]));
                            *reinterpret_cast<uint4*>(stg + 4 * (pc - q0)) = make_uint4(gw[0], gw[1], gw[2], gw[3]);
                        }
                    uint32_t sr[64];
                    OASR_TMEM_LD32(tl + kColS + 64 * hf, sr);
                    OASR_TMEM_LD32(tl + kColS + 64 * hf + 32, (sr + 32));
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 64; ++j) sc[j] = __uint_as_float(sr[j]);
                }
                // S and G are read: the issuer may compute the next stage's into the same
                // columns while this warp adds the position term and exponentiates
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_sg_free);
                if (live) {
                    const uint32_t sel = (lane & 1) ? 0x3210u : 0x5432u;
                    const uint32_t* rd = stg + (w0 & 3);
                    uint32_t wa = rd[0];
#pragma unroll
                    for (int m = 0; m < 32; ++m) {
                        const uint32_t wb = rd[m + 1];
                        add_bf16x2_f32(sc[2 * m], sc[2 * m + 1], __byte_perm(wa, wb, sel));
                        wa = wb;
                    }
                }
                // last stage of the item: the next item's Qu/Qv, so that its first S/G can be
                // issued while this stage's softmax and the epilogue run
                if (s + 1 == n_st && item + gridDim.x < n_items) {
                    int ns1, nL, ni0, nh, nkl, nkh;
                    decode(item + gridDim.x, seg, ns1, nL, ni0, nh, nkl, nkh);
                    if (!warp_wait(bar_q_free, it & 1) || !prep_q(it + 1, nh)) { ok = false; break; }
                }
                // the previous item's O, now that this first stage's S/G are read
                if (s == 0 && have_prev) {
                    if (!epilogue(p_start, p_L, p_i0, p_h, p_l)) { ok = false; break; }
                    have_prev = false;
                }
                // scale (log2 domain), mask keys this row does not see, this half's max
                // scores stay unscaled here: the scale (> 0, its sign is folded into q+u and
                // q+v) is applied to the row max and inside the exponent's FFMA
                // (three-input max: two scores per instruction)
                float mx0 = -INFINITY, mx1 = -INFINITY;
                if (!live) {
                } else if (ka <= 0 && kb >= 64) {
#pragma unroll
                    for (int j = 0; j < 64; j += 4) {
                        mx0 = fmax3(mx0, sc[j], sc[j + 1]);
                        mx1 = fmax3(mx1, sc[j + 2], sc[j + 3]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 64; j += 4) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            sc[j + e] = (j + e >= ka && j + e < kb) ? sc[j + e] : -INFINITY;
                        mx0 = fmax3(mx0, sc[j], sc[j + 1]);
                        mx1 = fmax3(mx1, sc[j + 2], sc[j + 3]);
                    }
                }
                float mx = fmaxf(mx0, mx1) * a.scale_log2, mx_other;
                pair_post(mx);
                // P.V of the previous stage must be done before P and O are touched
                if (s > 0 && !warp_wait(bar_pv_done, (g - 1) & 1)) { ok = false; break; }
                if (!pair_collect(mx_other)) { ok = false; break; }
                mx = fmaxf(mx, mx_other);
                const bool rescale = mx > m_used + 8.f;   // keeps every P <= 2^8 between rescales
                const float m_new = rescale ? mx : m_used;
                if (s > 0 && __any_sync(0xffffffffu, rescale)) {
                    const float alpha = ex2_approx(m_used - m_new);
                    l_sum *= alpha;
                    tc_fence_after();
                    uint32_t oo[32];
                    OASR_TMEM_LD32(tl + kColO + 32 * hf, oo);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) oo[j] = __float_as_uint(__uint_as_float(oo[j]) * alpha);
                    OASR_TMEM_ST32(tl + kColO + 32 * hf, oo);
                }
                m_used = m_new;
                // a row that has seen no key yet has max -inf: its P is 0, not NaN
                const float mref = m_used == -INFINITY ? 0.f : m_used;
                if (!live) {
                    uint32_t zero[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) zero[j] = 0u;
                    OASR_TMEM_ST16(tl + kColP + 32 * hf, zero);
                    OASR_TMEM_ST16(tl + kColP + 32 * hf + 16, zero);
                } else {
                    float2 ps = make_float2(0.f, 0.f);
                    const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
                    const float2 nm2 = make_float2(-mref, -mref);
#pragma unroll
                    for (int q2 = 0; q2 < 2; ++q2) {
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            // the exponents' scale-and-shift and the row sums two at a time
                            const float2 e2 = __ffma2_rn(
                                make_float2(sc[32 * q2 + 2 * j], sc[32 * q2 + 2 * j + 1]), sc2, nm2);
                            const float2 p2 = make_float2(ex2_approx(e2.x), ex2_approx(e2.y));
                            ps = __fadd2_rn(ps, p2);
                            pk[j] = pack_bf16(p2.x, p2.y);
                        }
                        OASR_TMEM_ST16(tl + kColP + 32 * hf + 16 * q2, pk);
                    }
                    l_sum += ps.x + ps.y;
                }
                // V rows past the segment belong to the next one.  P.V stops at the 16-key
                // step holding the segment's last key; that step's rows past it are zeroed so
                // that P = 0 there never meets a non-finite value (only the warps whose rows
                // fall there take part)
                const int kstage = kh - (kl + s * kBN);   // keys of this stage that exist
                const int k16 = (kstage + 15) & ~15;
                if (kstage < k16 && 32 * quad < k16 && 32 * quad + 32 > kstage) {
                    if (!warp_wait(bar_v_full + 8 * (g & 1), (g >> 1) & 1)) { ok = false; break; }
                    if (r >= kstage && r < k16) {
                        uint4* vrow = reinterpret_cast<uint4*>(slot_p + SP::off_v + r * kRowBytes) + 4 * hf;
#pragma unroll
                        for (int c = 0; c < 4; ++c) vrow[c] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_p_full);
            }
            if (!ok) { all_ok = false; break; }
            p_start = start;
            p_L = L;
            p_i0 = i0;
            p_h = h;
            p_l = l_sum;
            have_prev = true;
        }
        if (all_ok && have_prev && !*s_abort) epilogue(p_start, p_L, p_i0, p_h, p_l);
    }
    // every role has stopped issuing and the MMA issuer has drained the tensor pipe
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
    if (tid == 0 && *s_abort) err |= kErrTimeout;
    if (err) atomicOr(a.status, err);
}

int g_smem_done_tc[2][64];

}  // namespace

// Host launcher used by oasr_packed_relattn_varlen and oasr_packed_relattn_chunked (bf16);
// cs > 0 selects the chunked-limited window (own chunk of cs frames and `left` earlier ones).
oasr_status launch_packed_tc(const void* q, const void* k, const void* v, const int32_t* cu_seqlens,
                             int num_seqs, int total, const void* pos_bias_u,
                             const void* pos_bias_v, const void* rel, int R, void* out, int H,
                             float scale, int cs, int left, cudaStream_t stream)
{
    if (num_seqs > kTcMaxSeqs) return OASR_ERR_UNSUPPORTED;
    if ((static_cast<long long>(total) / kBM + num_seqs) * H >= 0x7fffffffLL) return OASR_ERR_UNSUPPORTED;
    CUtensorMap tm_q, tm_k, tm_v, tm_r;
    if (!encode_rows_bf16(&tm_q, q, total, H, kBM) || !encode_rows_bf16(&tm_k, k, total, H, kBN) ||
        !encode_rows_bf16(&tm_v, v, total, H, kBN) ||
        !encode_rows_bf16(&tm_r, rel, R, H, kBand))
        return OASR_ERR_INVALID_ARG;
    unsigned* status = status_word();
    const int sms = sm_count();
    if (!status || !sms) return OASR_ERR_CUDA;
    constexpr int smem = TcSmem::bytes;
    const bool masked = cs > 0;
    auto kern = masked ? packed_attn_tc_kernel<true> : packed_attn_tc_kernel<false>;
    if (!ensure_smem(kern, smem, g_smem_done_tc[masked ? 1 : 0])) return OASR_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTcThreads, smem) != cudaSuccess ||
        per_sm < 1)
        return OASR_ERR_CUDA;
    TcArgs a;
    a.q = static_cast<const uint16_t*>(q);
    a.cu_seqlens = cu_seqlens;
    a.pos_bias_u = static_cast<const uint16_t*>(pos_bias_u);
    a.pos_bias_v = static_cast<const uint16_t*>(pos_bias_v);
    a.out = static_cast<uint16_t*>(out);
    a.status = status;
    a.num_seqs = num_seqs;
    a.total = total;
    a.H = H;
    a.z = (R - 1) / 2;
    a.cs = masked ? cs : 1;
    a.left = masked ? left : 0;
    a.sign = scale < 0.f ? 0x80008000u : 0u;
    // > 0 even for a zero scale, so that a masked score (-inf) times it stays -inf; at 1e-30
    // every finite score's contribution to ex2 rounds away in fp32, as with a zero scale
    a.scale_log2 = fmaxf(fabsf(scale) * 1.4426950408889634f, 1e-30f);
    const long long items_bound = ((static_cast<long long>(total) + kBM - 1) / kBM + num_seqs) * H;
    const int grid = static_cast<int>(items_bound < sms ? items_bound : sms);
    kern<<<grid, kTcThreads, smem, stream>>>(tm_q, tm_k, tm_v, tm_r, a);
    return launch_status();
}

}  // namespace oasr
