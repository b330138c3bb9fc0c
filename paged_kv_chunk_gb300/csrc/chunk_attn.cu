// Streaming chunk attention over the block-paged pool, with the shared Transformer-XL
// relative-position term (oasr_chunk_relattn_paged), and the fused append + attention
// step (oasr_chunk_step_paged).
//
// Scheduler page, section 4.3 "Heterogeneous-offset batching": each stream's keys are
// masked by its cache_seqlens and the rel-pos bias matrix_bd / sqrt(d_k) is added to the
// content score.  Model Layer page, fixed_attention_window row: with uniform cache length
// one table serves the cohort, distances cache + i - j; Nemotron ASR section: rel_shift
// order, so the row for query i and key j is rho = (R - T - C) + j - i.
//
// bf16 path (the hot path): one CTA per (stream, head), 4 consumer warps and a TMA
// producer warp.  Keys are streamed in stages of 64 through a TMA pipeline: each stage is
// one box per block-table page for K and for V (the page's rows of this head, 128 B each,
// 128-byte swizzled), all arriving on one mbarrier.  The position term comes one of two
// ways.  Position table (GT; T <= 16 and a history that fits): the consumer warps compute
// the CTA's whole term once, from rel rows read from L2, into a pre-skewed bf16 table in
// shared memory while the first pages are in flight, and every 16-key slice reads it back.
// Band (otherwise): each stage also carries a box of the rel band, and each slice or stage
// multiplies it and skews the product through shared memory.  The per-slice and per-stage
// math is in attn_core.cuh.
// Fused variant (append + attention): when every page the chunk lands in is a valid block
// of the table ("direct" mode) the chunk is read by TMA straight from k_new / v_new (with
// the position table into a region of its own at kernel start, else as stage 0), the pool
// stages cover only the cached keys [0, C), and the chunk is written into the pool
// meanwhile, a side effect no stage of this launch reads.  Otherwise (a chunk past the
// table or in an invalid block) the stages cover [0, C + T) from the pool and those holding
// the chunk are issued only after the consumers' 16-byte stores of it are fenced against
// the async proxy, so the error handling of the append applies unchanged.
//
// f32 path: a SIMT kernel (one warp per query row, lanes over keys, fp32 FMA and expf).
#include "attn_core.cuh"
#include "host_common.h"

namespace oasr {

// A pipeline wait: the first poll inline, the polling loop with its time limit out of line,
// so that each wait site costs a few instructions of code.
__device__ __noinline__ bool ca_wait_slow(uint32_t bar, uint32_t parity) { return mbar_wait(bar, parity); }
__device__ __forceinline__ bool ca_wait(uint32_t bar, uint32_t parity)
{
    return mbar_try_wait(bar, parity) || ca_wait_slow(bar, parity);
}

// The tensor-core kernel for 33 <= T <= 64 (chunk_tc.cu).
bool chunk_tc_takes(int B, int T, int H, int mbps, int num_blocks, int block_size, int R);
oasr_status launch_chunk_tc(const void* q, const void* k_pool, const void* v_pool, int num_blocks,
                            int block_size, const int32_t* bt, int mbps, const int32_t* cs,
                            const void* u, const void* vb, const void* rel, int R, void* out,
                            int B, int T, int H, int k_max, float scale, cudaStream_t stream);

namespace {

struct ChunkArgs {
    const uint16_t* k_new;   // fused only
    const uint16_t* v_new;   // fused only
    uint16_t* k_pool;        // fused only
    uint16_t* v_pool;        // fused only
    const int32_t* block_table;
    const int32_t* cache_seqlens;
    const uint16_t* pos_bias_u;
    const uint16_t* pos_bias_v;
    const uint16_t* rel;     // position-table variant: rel rows [R][H][64]
    uint16_t* out;
    unsigned* status;
    int num_blocks, block_size, mbps, T, H, R;
    int box_rows;            // rows of one K/V TMA box = min(block_size, 64)
    int bs_shift;            // log2(block_size)
    int gt_w;                // position-table variant: row stride of the table (bf16 elements)
    int k_max;               // keys a stream may have: the table's pages and the keys the rel
                             // table serves (R - T + 1); the position table is sized for them
    int bt_pages;            // block-table entries a CTA reads: ceil(k_max / block_size)
    float scale_log2;        // scale * log2(e)
};

// Shared-memory plan of the streaming kernel (byte offsets from a 1024-aligned base).
// Slot i holds one stage: K rows [64][128 B], V rows [64][128 B] and, for the band, rel
// band rows [RB][128 B], all 128-byte swizzled by TMA.  With one m-tile a warp's skew
// scratch overlays its own K rows of the slot (dead once its scores are formed); with 2 or
// 4 m-tiles each consumer warp has its own scratch.  After the key loop the slots hold the
// cross-warp combine.  Position-table variant (GT, one m-tile): no band in the slots, a
// 4 KB region for the chunk's rows, and the CTA's whole position term, 16 rows of gt_w
// floats, after the barriers (its size is set at launch).
// Block-table entries a CTA caches in shared memory.
constexpr int kMaxPages = 512;

template <int MT, int NS, bool GT>
struct ChunkSmem {
    using TL = Tile<MT>;
    static_assert(!GT || MT <= 2, "the position table serves one or two m-tiles");
    static constexpr int kBand = GT ? 0 : TL::RB * kRowBytes;
    static constexpr int kSlot = 2 * kStageKeys * kRowBytes + kBand;
    static constexpr int off_slots = 0;
    static constexpr int off_q = NS * kSlot;
    static constexpr int off_ck = off_q + TL::Tp * kRowBytes;   // GT: the chunk's K|V rows
    static constexpr int off_g = off_ck + (GT ? 2 * TL::Tp * kRowBytes : 0);
    static constexpr int off_u = off_g + ((MT == 1 || GT) ? 0 : kConsumerWarps * kGBytes);
    static constexpr int off_vb = off_u + kHeadDim * 4;
    static constexpr int off_bt = off_vb + kHeadDim * 4;    // the stream's block-table row
    static constexpr int off_bar = off_bt + kMaxPages * 4;  // full[NS], empty[NS], q, written, chunk
    static constexpr int off_gt = (off_bar + (2 * NS + 3) * 8 + 15) & ~15;
    static constexpr int bytes = off_gt + 1024;   // + 16 * gt_w * 2 with GT
    static constexpr int comb_o = 0;
    static constexpr int comb_m = comb_o + TL::KG * TL::Tp * kOW * 4;
    static constexpr int comb_l = comb_m + TL::KG * TL::Tp * 4;
    static_assert(kSlot % 1024 == 0 && off_q % 1024 == 0 && off_ck % 1024 == 0,
                  "TMA tiles need 1024-byte alignment");
    static_assert(comb_l + TL::KG * TL::Tp * 4 <= NS * kSlot, "combine area");
};

// Two CTAs per SM; the position-table kernel with a two-stage ring (short histories on grids
// of several waves) is built for four (96 registers), with lighter batches of rel loads.
template <int MT, int NS, bool FUSED, bool GT>
__global__ void __launch_bounds__(kThreads, (GT && NS == 2) ? 4 : 2) chunk_attn_bf16_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_r,
    const __grid_constant__ CUtensorMap tm_kn, const __grid_constant__ CUtensorMap tm_vn,
    const ChunkArgs a)
{
    using TL = Tile<MT>;
    using SP = ChunkSmem<MT, NS, GT>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived from the __shared__ array itself so that every access
    // through it stays a shared-space access
    uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x / a.H, h = blockIdx.x - (blockIdx.x / a.H) * a.H;
    const int T = a.T;
    unsigned err = 0;

    // The tensor maps are launch parameters no grid writes: their descriptors are fetched
    // while the previous grid on the stream drains.
    if (tid == 0) prefetch_tensormap(&tm_q);
    if (warp == kConsumerWarps && lane == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
        if (!GT) prefetch_tensormap(&tm_r);
        if (FUSED) {
            prefetch_tensormap(&tm_kn);
            prefetch_tensormap(&tm_vn);
        }
    }
    // Launched with programmatic stream serialization: everything the previous grid on the
    // stream wrote is visible once this returns, and nothing global is read before it.
    grid_dep_wait();
    const uint32_t bar_full = sb + SP::off_bar;
    const uint32_t bar_empty = bar_full + NS * 8;
    const uint32_t bar_q = bar_empty + NS * 8;
    const uint32_t bar_written = bar_q + 8;   // fused: the chunk is in the pool and fenced
    const uint32_t bar_chunk = bar_written + 8;   // GT, fused: the chunk rows have landed
    float* s_u = reinterpret_cast<float*>(sm + SP::off_u);
    float* s_vb = reinterpret_cast<float*>(sm + SP::off_vb);
    __shared__ int s_failed;

    // The producer warp sets up the barriers, requests Q (and the chunk's rows), loads the
    // block-table row and starts issuing stages without waiting for the consumers: named
    // barrier 2 (producer arrives, consumers wait) hands them the initialised barriers and the
    // row in shared memory.
    int* s_bt = reinterpret_cast<int*>(sm + SP::off_bt);
    const bool producer = warp == kConsumerWarps;
    int C = __ldg(a.cache_seqlens + b);
    if (producer) {
        // the block-table entries of every key a stream may have (bt_pages <= mbps <=
        // kMaxPages, host check), not just the pages of this stream's K keys: their loads go
        // out beside the cache length's instead of after it (the first 128 held in registers
        // meanwhile, the rest of a longer row copied after)
        constexpr int kRowRegs = 4;
        const int32_t* bt_row = a.block_table + static_cast<long long>(b) * a.mbps;
        int row[kRowRegs];
#pragma unroll
        for (int k = 0; k < kRowRegs; ++k) {
            const int i = lane + 32 * k;
            if (i < a.bt_pages) row[k] = __ldg(bt_row + i);
        }
        if (lane == 0) {
            for (int i = 0; i < NS; ++i) {
                mbar_init(bar_full + 8 * i, 1);
                // one m-tile or the position table: all consumer warps read every stage (with
                // the table and one m-tile every lane arrives, as soon as its reads are done)
                mbar_init(bar_empty + 8 * i, (GT && MT == 1) ? 32 * kConsumerWarps
                                             : (MT == 1 || GT) ? kConsumerWarps : MT);
            }
            mbar_init(bar_q, 1);
            mbar_init(bar_written, 32 * kConsumerWarps);
            mbar_init(bar_chunk, 1);
            fence_mbar_init();
            s_failed = 0;
            // the Q tile needs neither the cache length nor the block table: it is requested
            // before either is read
            mbar_arrive_expect_tx(bar_q, TL::Tp * kRowBytes);
            tma_load_3d(sb + SP::off_q, &tm_q, bar_q, 0, h, b * T);
            if (GT && FUSED) {
                // nor do the chunk's rows (T <= Tp: one Tp-row box each for K and V)
                mbar_arrive_expect_tx(bar_chunk, 2 * TL::Tp * kRowBytes);
                tma_load_3d(sb + SP::off_ck, &tm_kn, bar_chunk, 0, h, b * T);
                tma_load_3d(sb + SP::off_ck + TL::Tp * kRowBytes, &tm_vn, bar_chunk, 0, h, b * T);
            }
        }
#pragma unroll
        for (int k = 0; k < kRowRegs; ++k) {
            const int i = lane + 32 * k;
            if (i < a.bt_pages) s_bt[i] = row[k];
        }
        for (int i = lane + 32 * kRowRegs; i < a.bt_pages; i += 32) s_bt[i] = __ldg(bt_row + i);
        __syncwarp();
        named_bar_arrive(2, kThreads);
    } else {
        // u, v go out beside the block-table row (the position table's rel rows are requested
        // only once the row is in: issued earlier they delay it and the first stages behind
        // them)
        if (tid < kHeadDim)
            s_u[tid] = bf16_lo(__ldg(a.pos_bias_u + h * kHeadDim + tid));
        else
            s_vb[tid - kHeadDim] = bf16_lo(__ldg(a.pos_bias_v + h * kHeadDim + tid - kHeadDim));
        named_bar_sync(2, kThreads);
    }
    if (C < 0) { C = 0; err |= kErrBounds; }
    int K = C + T;
    // keys past the table's pages (or past the keys the position table was sized for, which
    // only a rel table shorter than C + 2T - 1 rows allows) are dropped
    const int cap = a.k_max;
    if (K > cap) { K = cap; err |= kErrBounds; }
    if (C + 2 * T - 1 > a.R) err |= kErrBounds;   // distances the rel table does not hold
    const int off = a.R - T - C;   // rho = off + j - i
    const int sh = a.bs_shift;

    // Stage plan (every thread derives the same one from the cached table row).
    bool direct = false;
    if (FUSED && C + T <= cap) {
        direct = true;
        for (int pg = C >> sh; pg <= (C + T - 1) >> sh; ++pg) {
            const int blk = s_bt[pg];
            if (blk < 0 || blk >= a.num_blocks) direct = false;
        }
    }
    const int kc = direct ? C : K;                        // keys served from the pool
    const int n_pool = (kc + kStageKeys - 1) / kStageKeys;
    // direct: the chunk is stage 0 of the ring, or (GT) a region of its own loaded at the start
    const bool chunk_stage = direct && !GT;
    const int n_stages = n_pool + (chunk_stage ? 1 : 0);
    // stage s: first key and number of valid keys
    auto stage_j0 = [&](int s) {
        return chunk_stage ? (s == 0 ? C : kStageKeys * (s - 1)) : kStageKeys * s;
    };
    auto stage_valid = [&](int s) {
        if (chunk_stage && s == 0) return T;
        const int left = kc - stage_j0(s);
        return left < kStageKeys ? left : kStageKeys;
    };

    // Stage s into slot s % NS, by the whole producer warp: lane q issues the K box of the
    // stage's q-th page (or 16-row piece of the chunk) and lane 16 + q its V box, lane 31 the
    // band box, so a stage's boxes go out in one instruction rather than one after another.
    auto issue = [&](int s, uint64_t pol) {
        const int slot = s % NS;
        const uint32_t bar = bar_full + 8 * slot;
        const uint32_t base = sb + SP::off_slots + slot * SP::kSlot;
        const int j0 = stage_j0(s);
        const bool chunk = chunk_stage && s == 0;
        const int box = chunk ? 16 : a.box_rows;
        const int nbox = chunk ? (T + 15) / 16
                               : min(kStageKeys / box, (kc - j0 + box - 1) / box);
        if (lane == 0)
            mbar_arrive_expect_tx(
                bar, static_cast<uint32_t>((2 * nbox * box + (GT ? 0 : TL::RB)) * kRowBytes));
        __syncwarp();
        const int q = lane & 15;
        const bool is_v = lane >= 16;
        if (q < nbox) {
            const uint32_t dst = base + (q * box + (is_v ? kStageKeys : 0)) * kRowBytes;
            if (chunk) {
                tma_load_3d(dst, is_v ? &tm_vn : &tm_kn, bar, 0, h, b * T + 16 * q);
            } else {
                const int j = j0 + q * box;
                const int lb = j >> sh;
                const int blk = s_bt[lb];
                int row;
                if (blk < 0 || blk >= a.num_blocks) {
                    err |= kErrBounds;
                    row = -2 * box;   // outside the pool: the box reads zeros
                } else {
                    row = (blk << sh) + (j - (lb << sh));
                }
                tma_load_3d_hint(dst, is_v ? &tm_v : &tm_k, bar, 0, h, row, pol);
            }
        }
        if (!GT && lane == 31)
            tma_load_3d(base + 2 * kStageKeys * kRowBytes, &tm_r, bar, 0, h, off + j0 - (TL::Tp - 1));
    };

    if (producer) {
        // The producer warp only issues copies: no other work shares its warp.
        const uint64_t pol = policy_evict_first();
        // without the direct chunk stage, stages from this one on hold chunk rows
        const int first_chunk_stage = (FUSED && !direct) ? C / kStageKeys : n_stages;
        int n_issued = 0;
        for (int issued = 0; issued < n_stages; ++issued) {
            const int slot = issued % NS;
            bool ok = issued < NS || ca_wait(bar_empty + 8 * slot, ((issued / NS) - 1) & 1);
            if (ok && issued == first_chunk_stage) ok = ca_wait(bar_written, 0);
            if (!__all_sync(0xffffffffu, ok)) {
                err |= kErrTimeout;
                break;
            }
            issue(issued, pol);
            n_issued = issued + 1;
        }
        if (GT && FUSED && direct) {
            // with every stage out, the chunk's rows (in their own region) go into the pool;
            // every chunk page is a valid block: that is what selected direct mode
            if (ca_wait(bar_chunk, 0)) {
                for (int idx = lane; idx < 2 * T * 8; idx += 32) {
                    const int kv = idx >= T * 8;
                    const int rem = idx - kv * T * 8;
                    const int t = rem >> 3, c = rem & 7;
                    const int p = C + t;
                    const int lb = p / a.block_size;
                    const uint4 val = *reinterpret_cast<const uint4*>(
                        sm + SP::off_ck + kv * TL::Tp * kRowBytes + swz128(t, c));
                    *reinterpret_cast<uint4*>(
                        (kv ? a.v_pool : a.k_pool) +
                        ((static_cast<long long>(s_bt[lb]) * a.block_size + (p - lb * a.block_size)) *
                             a.H + h) * kHeadDim + c * 8) = val;
                }
            } else {
                err |= kErrTimeout;
            }
        }
        // Every copy this CTA requested lands before the CTA can end, also when a consumer's
        // wait ran out and it left early (bounded waits: the last stage of each slot, Q).
        for (int x = n_issued > NS ? n_issued - NS : 0; x < n_issued; ++x)
            if (!mbar_wait_idle(bar_full + 8 * (x % NS), (x / NS) & 1)) err |= kErrTimeout;
        if (!mbar_wait_idle(bar_q, 0)) err |= kErrTimeout;
        if (err) atomicOr(a.status, err);
        return;
    }

    // ---- consumers: u, v; the chunk into the pool (fused); then the stages
    const int mt = warp % MT, kg = warp / MT;
    bool failed = false;
    uint32_t qu[4][4], qv[4][4];
    WarpAcc acc;
    acc_init(acc);
    // fused, without the direct chunk stage: this head's slice of the chunk into the pool
    // (T rows x 8 vectors of 16 B, for K and for V), fenced for the stages that read it back
    auto copy_chunk_global = [&]() {
        for (int idx = tid; idx < 2 * T * 8; idx += 32 * kConsumerWarps) {
            const int kv = idx >= T * 8;
            const int rem = idx - kv * T * 8;
            const int t = rem >> 3, c = rem & 7;
            const int p = C + t;
            const int lb = p / a.block_size;
            if (lb >= a.mbps || p >= K) { err |= kErrBounds; continue; }
            const int slot = p - lb * a.block_size;
            const int blk = s_bt[lb];
            if (blk < 0 || blk >= a.num_blocks) { err |= kErrBounds; continue; }
            const uint16_t* src = (kv ? a.v_new : a.k_new) +
                                  ((static_cast<long long>(b) * T + t) * a.H + h) * kHeadDim + c * 8;
            uint16_t* dst = (kv ? a.v_pool : a.k_pool) +
                            ((static_cast<long long>(blk) * a.block_size + slot) * a.H + h) * kHeadDim +
                            c * 8;
            *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
        }
        fence_proxy_async_global();
        mbar_arrive(bar_written);
    };
    if constexpr (GT) {
        PosTable<NS == 2 ? 5 : 10, MT> pt;
        pt.rel_h = a.rel + h * kHeadDim;
        pt.stride = static_cast<long long>(a.H) * kHeadDim;
        pt.R = a.R;
        pt.rho0 = off - (TL::Tp - 1);
        pt.ncols = K + TL::Tp - 1;
        pt.warp = warp;
        pt.nw = kConsumerWarps;
        pt.lane = lane;
        pt.load(warp);
        if (FUSED && !direct) copy_chunk_global();
        // the whole position term of the CTA (its rel rows are in flight or in), while the
        // first pages land
        failed = !ca_wait(bar_q, 0);
        if (!failed)
            pt.build(reinterpret_cast<uint16_t*>(sm + SP::off_gt), a.gt_w, sm + SP::off_q, s_vb);
        // fused: the chunk's rows (requested at the start; they must land before the CTA
        // ends even when the stages do not use them)
        if (FUSED && !ca_wait(bar_chunk, 0)) failed = true;
        named_bar_sync(1, 32 * kConsumerWarps);   // the table is complete
        if (!failed) make_q_frags(sb + SP::off_q, s_u, s_vb, mt, lane, qu, qv);
    } else {
        if constexpr (FUSED) copy_chunk_global();
        named_bar_sync(1, 32 * kConsumerWarps);
        failed = !ca_wait(bar_q, 0);
        if (!failed) make_q_frags(sb + SP::off_q, s_u, s_vb, mt, lane, qu, qv);
    }
    if (!failed) {
        float* gw = reinterpret_cast<float*>(sm + SP::off_g) + warp * (kGBytes / 4);
        if constexpr (GT) {
            const uint16_t* gs = reinterpret_cast<const uint16_t*>(sm + SP::off_gt);
            // warp w: m-tile w % MT (its 16 query rows of the table at gm) and, of every stage,
            // the MT 16-key slices from key 16 MT (w / MT); query i, key j read table position
            // j + Tp
            const int kh = warp / MT;
            const uint16_t* gm = gs + 16 * mt * a.gt_w;
            if (FUSED && direct) {
                // the chunk, landed long before the first pool stage: its 16-key slice kh (the
                // producer warp writes its rows into the pool)
                const int kvc = T - 16 * kh;
                if (kvc > 0) {
                    const int x0 = C + 16 * kh + TL::Tp;
                    warp_slice16_gt(acc, qu, sb + SP::off_ck + 16 * kh * kRowBytes,
                                    sb + SP::off_ck + (TL::Tp + 16 * kh) * kRowBytes, gm + x0,
                                    a.gt_w, (x0 & 1) == 0, kvc, a.scale_log2, lane);
                }
            }
            for (int s = 0; s < n_stages; ++s) {
                const int slot = s % NS;
                if (!ca_wait(bar_full + 8 * slot, (s / NS) & 1)) { failed = true; break; }
                const uint32_t base = sb + SP::off_slots + slot * SP::kSlot;
                // one m-tile: every lane releases the slot as soon as its slice's K and V rows
                // are read (before the position term, softmax and P.V), so the producer can
                // refill it earlier; two m-tiles: lane 0 after both slices
                const uint32_t rel_bar = MT == 1 ? bar_empty + 8 * slot : 0u;
#pragma unroll
                for (int u = 0; u < MT; ++u) {
                    const int jl = 16 * (MT * kh + u);   // the slice's first key in the stage
                    const int kv = stage_valid(s) - jl;
                    if (kv > 0) {
                        const int x0 = stage_j0(s) + jl + TL::Tp;   // table position of the slice
                        warp_slice16_gt(acc, qu, base + jl * kRowBytes,
                                        base + (kStageKeys + jl) * kRowBytes, gm + x0, a.gt_w,
                                        (x0 & 1) == 0, kv, a.scale_log2, lane, rel_bar);
                    } else if (MT == 1) {
                        mbar_arrive_release(rel_bar);
                    }
                }
                if (MT != 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
                }
            }
        } else if constexpr (MT == 1) {
            // every stage: this warp's 16-key slice; its skew scratch overlays its K rows
            for (int s = 0; s < n_stages; ++s) {
                const int slot = s % NS;
                if (!ca_wait(bar_full + 8 * slot, (s / NS) & 1)) { failed = true; break; }
                const uint32_t base = sb + SP::off_slots + slot * SP::kSlot;
                const int kv = stage_valid(s) - 16 * warp;
                if (kv > 0) {
                    warp_slice16(acc, qu, qv, base + 16 * warp * kRowBytes,
                                 base + (kStageKeys + 16 * warp) * kRowBytes,
                                 base + (2 * kStageKeys + 16 * warp) * kRowBytes,
                                 reinterpret_cast<float*>(sm + SP::off_slots + slot * SP::kSlot +
                                                          16 * warp * kRowBytes),
                                 kv, a.scale_log2, lane);
                    fence_proxy_async_smem();   // the next TMA into this slot
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
            }
        } else
        for (int s = kg; s < n_stages; s += TL::KG) {
            const int slot = s % NS;
            if (!ca_wait(bar_full + 8 * slot, (s / NS) & 1)) { failed = true; break; }
            const uint32_t base = sb + SP::off_slots + slot * SP::kSlot;
            const uint32_t band = base + 2 * kStageKeys * kRowBytes;
            warp_stage(acc, qu, qv, base, base + kStageKeys * kRowBytes, band,
                       TL::Tp - 16 - 16 * mt, gw, stage_valid(s), a.scale_log2, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
        }
    }
    if (failed) s_failed = 1;
    // the stage loop is done: the next grid on the stream may start launching its CTAs (they
    // wait for this grid to finish before reading anything)
    grid_dep_trigger();
    named_bar_sync(1, 32 * kConsumerWarps);
    if (s_failed) {
        if (tid == 0) atomicOr(a.status, err | kErrTimeout);
        return;
    }
    float* comb_o = reinterpret_cast<float*>(sm + SP::comb_o);
    float* comb_m = reinterpret_cast<float*>(sm + SP::comb_m);
    float* comb_l = reinterpret_cast<float*>(sm + SP::comb_l);
    acc_reduce_l(acc);
    write_partial(acc, comb_o, comb_m, comb_l, kg * TL::Tp + 16 * mt, lane);
    named_bar_sync(1, 32 * kConsumerWarps);
    for (int idx = tid; idx < T * 8; idx += 32 * kConsumerWarps) {
        const int row = idx >> 3, d0 = (idx & 7) * 8;
        const uint4 v = combine_row8(comb_o, comb_m, comb_l, TL::KG, TL::Tp, row, d0);
        *reinterpret_cast<uint4*>(a.out + ((static_cast<long long>(b) * T + row) * a.H + h) *
                                              kHeadDim + d0) = v;
    }
    if (err) atomicOr(a.status, err);
}

// ----------------------------------------------------------------------------- fp32

template <bool FUSED>
__global__ void __launch_bounds__(128) chunk_attn_f32_kernel(
    const float* __restrict__ q, const float* __restrict__ k_new, const float* __restrict__ v_new,
    float* k_pool, float* v_pool, int num_blocks, int block_size,
    const int32_t* __restrict__ block_table, int mbps, const int32_t* __restrict__ cache_seqlens,
    const float* __restrict__ u, const float* __restrict__ vb, const float* __restrict__ rel,
    int R, float* __restrict__ out, int T, int H, float scale, unsigned* status)
{
    __shared__ float s_qu[64][kHeadDim];
    __shared__ float s_qv[64][kHeadDim];
    const int b = blockIdx.x / H, h = blockIdx.x % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned err = 0;
    int C = cache_seqlens[b];
    if (C < 0) { C = 0; err |= kErrBounds; }
    int K = C + T;
    const int cap = mbps * block_size;
    if (K > cap) { K = cap; err |= kErrBounds; }
    if (C + 2 * T - 1 > R) err |= kErrBounds;   // distances the rel table does not hold
    const int off = R - T - C;

    if (FUSED) {
        for (int idx = tid; idx < 2 * T * kHeadDim; idx += blockDim.x) {
            const int kv = idx >= T * kHeadDim;
            const int rem = idx - kv * T * kHeadDim;
            const int t = rem / kHeadDim, d = rem % kHeadDim;
            const int p = C + t;
            const int lb = p / block_size;
            if (lb >= mbps) { err |= kErrBounds; continue; }
            const int blk = block_table[static_cast<long long>(b) * mbps + lb];
            if (blk < 0 || blk >= num_blocks) { err |= kErrBounds; continue; }
            const long long dst =
                ((static_cast<long long>(blk) * block_size + (p - lb * block_size)) * H + h) * kHeadDim + d;
            const long long src = ((static_cast<long long>(b) * T + t) * H + h) * kHeadDim + d;
            (kv ? v_pool : k_pool)[dst] = (kv ? v_new : k_new)[src];
        }
    }
    for (int idx = tid; idx < T * kHeadDim; idx += blockDim.x) {
        const int t = idx / kHeadDim, d = idx % kHeadDim;
        const float qq = q[((static_cast<long long>(b) * T + t) * H + h) * kHeadDim + d];
        s_qu[t][d] = qq + u[h * kHeadDim + d];
        s_qv[t][d] = qq + vb[h * kHeadDim + d];
    }
    __syncthreads();

    for (int i = warp; i < T; i += 4) {
        float m = -INFINITY, l = 0.f, o0 = 0.f, o1 = 0.f;
        for (int j0 = 0; j0 < K; j0 += 32) {
            const int j = j0 + lane;
            float sc = -INFINITY;
            long long row_off = -1;   // element offset of key j's row in the pools
            if (j < K) {
                const int lb = j / block_size;
                const int blk = block_table[static_cast<long long>(b) * mbps + lb];
                float acc = 0.f;
                if (blk >= 0 && blk < num_blocks) {
                    row_off = ((static_cast<long long>(blk) * block_size + (j - lb * block_size)) * H + h) *
                              kHeadDim;
                    const float4* kr = reinterpret_cast<const float4*>(k_pool + row_off);
#pragma unroll 4
                    for (int d4 = 0; d4 < kHeadDim / 4; ++d4) {
                        const float4 kk = kr[d4];
                        acc = fmaf(s_qu[i][4 * d4], kk.x, acc);
                        acc = fmaf(s_qu[i][4 * d4 + 1], kk.y, acc);
                        acc = fmaf(s_qu[i][4 * d4 + 2], kk.z, acc);
                        acc = fmaf(s_qu[i][4 * d4 + 3], kk.w, acc);
                    }
                } else {
                    err |= kErrBounds;
                }
                const int rho = off + j - i;
                if (rho >= 0 && rho < R) {
                    const float4* rr =
                        reinterpret_cast<const float4*>(rel + (static_cast<long long>(rho) * H + h) * kHeadDim);
#pragma unroll 4
                    for (int d4 = 0; d4 < kHeadDim / 4; ++d4) {
                        const float4 r4 = rr[d4];
                        acc = fmaf(s_qv[i][4 * d4], r4.x, acc);
                        acc = fmaf(s_qv[i][4 * d4 + 1], r4.y, acc);
                        acc = fmaf(s_qv[i][4 * d4 + 2], r4.z, acc);
                        acc = fmaf(s_qv[i][4 * d4 + 3], r4.w, acc);
                    }
                }
                sc = acc * scale;
            }
            float mx = sc;
#pragma unroll
            for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float m_new = fmaxf(m, mx);
            const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
            const float p = (j < K) ? expf(sc - m_new) : 0.f;
            float psum = p;
#pragma unroll
            for (int o = 16; o; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
            l = l * alpha + psum;
            o0 *= alpha;
            o1 *= alpha;
            const int nj = min(32, K - j0);
            for (int jj = 0; jj < nj; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, p, jj);
                const long long ro = __shfl_sync(0xffffffffu, row_off, jj);
                if (ro >= 0) {
                    o0 = fmaf(pj, v_pool[ro + lane], o0);
                    o1 = fmaf(pj, v_pool[ro + 32 + lane], o1);
                }
            }
            m = m_new;
        }
        float* dst = out + ((static_cast<long long>(b) * T + i) * H + h) * kHeadDim;
        dst[lane] = o0 / l;
        dst[lane + 32] = o1 / l;
    }
    if (err) atomicOr(status, err);
}

// --------------------------------------------------------------------------- host

int g_smem_done[16][64];

// Dynamic shared memory of one CTA that still lets two (four) CTAs share an SM.
constexpr int kTwoCtaSmem = 112 * 1024;
constexpr int kFourCtaSmem = 56 * 1024;

// Row stride (bf16 elements) of the position table of Tp query rows for keys up to `cap`:
// every read and write stays below cap + 2 Tp, and a stride of 16 mod 64 elements (8 mod 32
// words) keeps the 4-byte reads of a slice conflict-free.
inline int pos_table_stride(int cap, int Tp = 16) { return ((cap + 2 * Tp + 63) & ~63) + 16; }

// Shared memory of the position table of Tp query rows (bf16).
inline int pos_table_bytes(long long cap, int Tp)
{
    return Tp * pos_table_stride(static_cast<int>(cap), Tp) * 2;
}

// Keys a stream of a call may have, as the host knows them: the table's pages, and the
// R - T + 1 keys a rel table of R rows serves (R >= C + 2T - 1 is required).
inline int key_bound(int mbps, int block_size, int R, int T)
{
    const long long pages = static_cast<long long>(mbps) * block_size;
    const long long rel = static_cast<long long>(R) - T + 1;
    const long long k = pages < rel ? pages : rel;
    return static_cast<int>(k < T ? T : k);
}

template <int MT, int NS, bool FUSED, bool GT>
oasr_status launch_bf16(const void* q, const void* k_new, const void* v_new, void* k_pool,
                        void* v_pool, int num_blocks, int block_size, const int32_t* bt,
                        int mbps, const int32_t* cs, const void* u, const void* vb,
                        const void* rel, int R, void* out, int B, int T, int H, float scale,
                        cudaStream_t stream, int slot)
{
    CUtensorMap tm_q, tm_k, tm_v, tm_r, tm_kn, tm_vn;
    const int box = block_size < kStageKeys ? block_size : kStageKeys;
    if (!encode_rows_bf16(&tm_q, q, static_cast<long long>(B) * T, H, Tile<MT>::Tp) ||
        !encode_rows_bf16(&tm_k, k_pool, static_cast<long long>(num_blocks) * block_size, H, box) ||
        !encode_rows_bf16(&tm_v, v_pool, static_cast<long long>(num_blocks) * block_size, H, box))
        return OASR_ERR_INVALID_ARG;
    if (GT)
        tm_r = tm_k;   // unused: the table reads rel directly
    else if (!encode_rows_bf16(&tm_r, rel, R, H, Tile<MT>::RB))
        return OASR_ERR_INVALID_ARG;
    if (FUSED) {
        // the chunk's rows as TMA sources for the direct chunk stage (16-row boxes) or the
        // position-table kernel's chunk region (Tp rows)
        const int cbox = GT ? Tile<MT>::Tp : 16;
        if (!encode_rows_bf16(&tm_kn, k_new, static_cast<long long>(B) * T, H, cbox) ||
            !encode_rows_bf16(&tm_vn, v_new, static_cast<long long>(B) * T, H, cbox))
            return OASR_ERR_INVALID_ARG;
    } else {
        tm_kn = tm_k;
        tm_vn = tm_v;
    }
    unsigned* status = status_word();
    if (!status) return OASR_ERR_CUDA;
    auto kern = chunk_attn_bf16_kernel<MT, NS, FUSED, GT>;
    // the keys the host can bound (the position table is sized for them); a stream with more
    // (a rel table shorter than the precondition allows) is clamped to them and flagged
    const int k_max = key_bound(mbps, block_size, R, T);
    const int gt_w = GT ? pos_table_stride(k_max, Tile<MT>::Tp) : 0;
    const int smem = ChunkSmem<MT, NS, GT>::bytes + Tile<MT>::Tp * gt_w * 2;
    if (!ensure_smem(kern, smem, g_smem_done[slot])) return OASR_ERR_CUDA;
    ChunkArgs a;
    a.k_new = static_cast<const uint16_t*>(k_new);
    a.v_new = static_cast<const uint16_t*>(v_new);
    a.k_pool = static_cast<uint16_t*>(k_pool);
    a.v_pool = static_cast<uint16_t*>(v_pool);
    a.block_table = bt;
    a.cache_seqlens = cs;
    a.pos_bias_u = static_cast<const uint16_t*>(u);
    a.pos_bias_v = static_cast<const uint16_t*>(vb);
    a.rel = static_cast<const uint16_t*>(rel);
    a.out = static_cast<uint16_t*>(out);
    a.status = status;
    a.num_blocks = num_blocks;
    a.block_size = block_size;
    a.mbps = mbps;
    a.T = T;
    a.H = H;
    a.R = R;
    a.box_rows = box;
    a.bs_shift = __builtin_ctz(static_cast<unsigned>(block_size));
    a.gt_w = gt_w;
    a.k_max = k_max;
    a.bt_pages = (k_max + block_size - 1) / block_size;
    a.scale_log2 = scale * 1.4426950408889634f;
    return launch_pdl(kern, dim3(static_cast<unsigned>(B) * H), dim3(kThreads), smem, stream, tm_q,
                      tm_k, tm_v, tm_r, tm_kn, tm_vn, a);
}

template <bool FUSED>
oasr_status dispatch(const void* q, const void* k_new, const void* v_new, void* k_pool,
                     void* v_pool, int num_blocks, int block_size, const int32_t* bt, int mbps,
                     const int32_t* cs, const void* u, const void* vb, const void* rel, int R,
                     void* out, int B, int T, int H, int D, float scale, oasr_dtype dt,
                     cudaStream_t stream)
{
    if (!q || !k_pool || !v_pool || !bt || !cs || !u || !vb || !rel || !out)
        return OASR_ERR_INVALID_ARG;
    if (FUSED && (!k_new || !v_new)) return OASR_ERR_INVALID_ARG;
    if (num_blocks <= 0 || block_size <= 0 || mbps <= 0 || R <= 0 || B <= 0 || T <= 0 ||
        H <= 0 || D <= 0)
        return OASR_ERR_INVALID_ARG;
    if (dt != OASR_F32 && dt != OASR_BF16) return OASR_ERR_UNSUPPORTED;
    if (D != kHeadDim || T > 64) return OASR_ERR_UNSUPPORTED;
    if (block_size < 8 || block_size > 256 || (block_size & (block_size - 1)))
        return OASR_ERR_UNSUPPORTED;
    if (dt == OASR_BF16 && mbps > kMaxPages) return OASR_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * H > 0x7fffffffLL) return OASR_ERR_UNSUPPORTED;
    const void* ptrs[] = {q, k_pool, v_pool, u, vb, rel, out, FUSED ? k_new : q,
                          FUSED ? v_new : q};
    for (const void* p : ptrs)
        if (!aligned16(p)) return OASR_ERR_INVALID_ARG;
    if (dt == OASR_F32) {
        unsigned* status = status_word();
        if (!status) return OASR_ERR_CUDA;
        chunk_attn_f32_kernel<FUSED><<<static_cast<unsigned>(B) * H, 128, 0, stream>>>(
            static_cast<const float*>(q), static_cast<const float*>(k_new),
            static_cast<const float*>(v_new), static_cast<float*>(k_pool),
            static_cast<float*>(v_pool), num_blocks, block_size, bt, mbps, cs,
            static_cast<const float*>(u), static_cast<const float*>(vb),
            static_cast<const float*>(rel), R, static_cast<float*>(out), T, H, scale, status);
        return launch_status();
    }
    // 33 <= T <= 64 with an even head count: the tensor-core kernel (two heads of a stream per
    // 128-row tile); the fused step appends the chunk first, on the same stream
    if (T > 32 && chunk_tc_takes(B, T, H, mbps, num_blocks, block_size, R)) {
        if (FUSED) {
            const oasr_status st = oasr_paged_append(k_new, v_new, k_pool, v_pool, num_blocks,
                                                     block_size, bt, mbps, cs, B, T, H, D, dt,
                                                     stream);
            if (st != OASR_OK) return st;
        }
        return launch_chunk_tc(q, k_pool, v_pool, num_blocks, block_size, bt, mbps, cs, u, vb,
                               rel, R, out, B, T, H, key_bound(mbps, block_size, R, T), scale,
                               stream);
    }
    const int f = FUSED ? 8 : 0;
    // One m-tile (T <= 16): the position table when it fits beside the ring, else the
    // per-stage band.  The table is sized for the keys the host can bound (the table's pages,
    // and the keys the rel table serves), so an engine-sized block table keeps the table form.
    // Grids of several waves at two CTAs per SM: four CTAs per SM with a two-stage ring when
    // their shared memory allows it (short histories: more CTAs resident beat stages in flight,
    // T = 16 24.3 -> 21.3 us, T = 4 and T = 8 15-18 % each), else two with five stages
    // (Conformer-large 63.4 -> 62.6 us); one wave: two CTAs with four stages.
    const long long cap = key_bound(mbps, block_size, R, T);
    const int sms = sm_count();
    const bool waves = sms > 0 && static_cast<long long>(B) * H > 2LL * sms;
    if (T <= 16 && cap <= 4096) {
        const int tb = pos_table_bytes(cap, 16);
        if (waves && ChunkSmem<1, 2, true>::bytes + tb <= kFourCtaSmem)
            return launch_bf16<1, 2, FUSED, true>(q, k_new, v_new, k_pool, v_pool, num_blocks,
                                                  block_size, bt, mbps, cs, u, vb, rel, R, out, B,
                                                  T, H, scale, stream, f + 4);
        if (waves && ChunkSmem<1, 5, true>::bytes + tb <= kTwoCtaSmem)
            return launch_bf16<1, 5, FUSED, true>(q, k_new, v_new, k_pool, v_pool, num_blocks,
                                                  block_size, bt, mbps, cs, u, vb, rel, R, out, B,
                                                  T, H, scale, stream, f + 5);
        if (ChunkSmem<1, 4, true>::bytes + tb <= kTwoCtaSmem)
            return launch_bf16<1, 4, FUSED, true>(q, k_new, v_new, k_pool, v_pool, num_blocks,
                                                  block_size, bt, mbps, cs, u, vb, rel, R, out, B,
                                                  T, H, scale, stream, f + 3);
    }
    // T = 17 .. 32: the position table of two m-tiles when it fits beside three stages
    if (T > 16 && T <= 32 && cap <= 4096 &&
        ChunkSmem<2, 3, true>::bytes + pos_table_bytes(cap, 32) <= kTwoCtaSmem)
        return launch_bf16<2, 3, FUSED, true>(q, k_new, v_new, k_pool, v_pool, num_blocks,
                                              block_size, bt, mbps, cs, u, vb, rel, R, out, B, T,
                                              H, scale, stream, f + 6);
    if (T <= 16)
        return launch_bf16<1, 4, FUSED, false>(q, k_new, v_new, k_pool, v_pool, num_blocks,
                                               block_size, bt, mbps, cs, u, vb, rel, R, out, B, T,
                                               H, scale, stream, f + 0);
    if (T <= 32)
        return launch_bf16<2, 3, FUSED, false>(q, k_new, v_new, k_pool, v_pool, num_blocks, block_size,
                                        bt, mbps, cs, u, vb, rel, R, out, B, T, H, scale, stream,
                                        f + 1);
    return launch_bf16<4, 2, FUSED, false>(q, k_new, v_new, k_pool, v_pool, num_blocks, block_size, bt,
                                    mbps, cs, u, vb, rel, R, out, B, T, H, scale, stream, f + 2);
}

}  // namespace
}  // namespace oasr

extern "C" oasr_status oasr_chunk_relattn_paged(
    const void* q, const void* k_pool, const void* v_pool, int num_blocks, int block_size,
    const int32_t* block_table, int max_blocks_per_seq, const int32_t* cache_seqlens,
    const void* pos_bias_u, const void* pos_bias_v, const void* rel, int R, void* out, int B,
    int T, int H, int D, float scale, oasr_dtype dt, cudaStream_t stream)
{
    return oasr::dispatch<false>(q, nullptr, nullptr, const_cast<void*>(k_pool),
                                 const_cast<void*>(v_pool), num_blocks, block_size, block_table,
                                 max_blocks_per_seq, cache_seqlens, pos_bias_u, pos_bias_v, rel,
                                 R, out, B, T, H, D, scale, dt, stream);
}

extern "C" oasr_status oasr_chunk_step_paged(
    const void* q, const void* k_new, const void* v_new, void* k_pool, void* v_pool,
    int num_blocks, int block_size, const int32_t* block_table, int max_blocks_per_seq,
    const int32_t* cache_seqlens, const void* pos_bias_u, const void* pos_bias_v, const void* rel,
    int R, void* out, int B, int T, int H, int D, float scale, oasr_dtype dt, cudaStream_t stream)
{
    return oasr::dispatch<true>(q, k_new, v_new, k_pool, v_pool, num_blocks, block_size,
                                block_table, max_blocks_per_seq, cache_seqlens, pos_bias_u,
                                pos_bias_v, rel, R, out, B, T, H, D, scale, dt, stream);
}
