// Streaming chunk attention over the block-paged pool on the 5th-generation tensor cores
// (tcgen05 + TMEM), bf16, for chunks of 33 to 64 frames.  Used by oasr_chunk_relattn_paged
// and oasr_chunk_step_paged (after the append) for those chunk lengths when H is even.
// A second mode (PK) serves the chunked-limited packed attention of oasr_packed_relattn_chunked
// (Model Layer page, Nemotron ASR section: a query sees its own chunk and `left` earlier ones):
// a work item is 64 queries of a segment for a head pair, its keys the window those queries
// reach (for chunks of 8 frames and 7 earlier ones, 120 keys: two stages), read from the packed K/V.
//
// Scheduler page, section 4.3 "Heterogeneous-offset batching": each stream's keys are its
// cache_seqlens cached frames and the chunk, and the rel-pos term matrix_bd / sqrt(d_k) is
// added to the content score.  Model Layer page, fixed_attention_window row (one rel table
// serves the cohort, distances cache + i - j) and Nemotron ASR section (rel_shift order):
// query i and key j of stream b use rel row rho = (R - T - C_b) - i + j.
//
// A chunk of T <= 64 queries fills half of a 128-row tensor-core tile, so one work item is a
// stream and a pair of its heads (h0 = 2 hp, h0 + 1): TMEM lanes 0-63 hold the chunk's queries
// for head h0 and lanes 64-127 for head h0 + 1 (rows T..63 of each half are padding).  A
// tcgen05.mma of M128 K16 costs about the same up to N = 128, so each product spans both heads
// at N = 128 and each row keeps the half that belongs to its head.  Per stage of 64 keys:
//   S [128 x 128] = bf16(q+u) . Kpair^T                  columns [0, 128)    M128 N128; Kpair holds
//                   the stage's keys of both heads in groups of 8 (column 16 (j / 8) + 8 hd +
//                   j % 8 is key j of head hd), and each row keeps its own head's columns
//   G [128 x 128] = A0 . Band_h0^T + A1 . Band_h1^T      columns [128, 256)  M128 N128, block-
//                   diagonal: A0 = [bf16(q+v) of h0 ; 0], A1 = [0 ; bf16(q+v) of h0+1] (one 8 KB
//                   zero block shared between them); the band is the 128 rel rows rho_min ..
//                   rho_min + 127 the stage reaches (rho_min = R - T - C - 63 + 64 s), and row i,
//                   key j of the stage uses band row 63 - i + j
//   O [128 x 128] += P . [V_h0 | V_h1]                   columns [256, 384)  M128 N128 (V of both
//                   heads as one MN-major operand); rows of head h0 keep columns 0-63, rows of
//                   h0 + 1 columns 64-127
//   P [128 x 64] bf16                                    columns [384, 416)
// The packed mode reads each stage's K and V rows of a head as one 64-row box, so there S
// column 64 hd + j is key j of head hd and P.V takes V_h0 and V_h1 as two 8 KB tiles.
// Warp roles (416 threads; 480 in the packed mode), one persistent CTA per SM walking work items:
//   warps 0-7  softmax.  Warps w and w+4 share TMEM lane quadrant w (rows 32w .. 32w+31); warp
//              w takes keys 0-31 of each stage, w+4 keys 32-63, and the pair swaps row maxima
//              and sums through shared memory.  Each thread reads its S half row and the G
//              columns its row reaches, releases S and G to the issuer, takes its skewed half
//              row of G (rounded to bf16) through its own shared staging tile, masks keys past
//              the stream's history, keeps the running max (O is rescaled in TMEM only when
//              the max grows by more than 2^8) and sum, and writes its half row of bf16 P to
//              TMEM; at the end of the item it normalises and stores its half of the O row.
//   warp 8     S/G issuer (one thread).
//   warp 9     TMA producer of the q rows and of the stage's K page boxes.
//   warp 10    TMA producer of the stage's V page boxes.
//   warp 11    TMA producer of the stage's rel band.
//   warp 12    P.V issuer (one thread).
//   warps 13-14 (packed mode) the A tiles of the coming items, one warp per head: q rows by TMA
//              into the item's A set (two sets, items alternating), then bf16(q+u) and bf16(q+v)
//              in place; the streaming mode's softmax warps do this between items instead.
// K and V (read from HBM) run through three-slot rings (two in the packed mode), a slot's K
// refilled as soon as the S and G products that read it have finished and its V once its P.V
// has; the band (rel rows, resident in L2) runs through a two-slot ring, because the softmax
// warps stage the skewed position term in the band tile of the stage they process (free once
// G is computed) and release it when their skewed reads are done.
// K and V arrive as one box per block-table page holding both heads (the pool viewed as
// {64, key % 8, head, key / 8}, so that each head's 8 consecutive keys form one 128-byte-
// swizzled 1 KB atom; one box per page instead of one per page and head halves the copies the
// SM's TMA unit issues); a block id outside the pool reads as zero rows.
// Streaming items that leave at most half a wave over the SMs are split: the leftover items
// run by key stages on the two CTAs of a cluster (the even one the first half of the stages),
// each CTA finishing one head of the item.  The warps of the other head hand their normalised
// rows over through that head's output rows (which the partner then overwrites) and their
// row weights log2(l) + m through the partner's shared memory, signalling an mbarrier there;
// the partner merges the two halves as two softmax blocks of the same row.
// Every wait is bounded; a wait that runs out raises the timeout bit and aborts the CTA's
// remaining work, after which the CTA still drains its copies and tensor-core work and frees
// its TMEM.
#include <mutex>

#include "attn_core.cuh"
#include "host_common.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace oasr {
namespace {

constexpr int kCtSoftmaxWarps = 8;
constexpr int kCtMmaWarp = 8, kCtKWarp = 9, kCtVWarp = 10, kCtBandWarp = 11, kCtPvWarp = 12;
constexpr int kCtPrepWarp = 13;           // packed mode: the A tiles of the coming items, one
                                          // warp per head (13, 14)
// threads of a CTA: the streaming mode has no A-tile warps
template <bool PK>
__host__ __device__ constexpr int ct_threads() { return 32 * (kCtSoftmaxWarps + (PK ? 7 : 5)); }
constexpr int kBandSlots = 2;             // depth of the band ring
constexpr int kCtBN = 64;                 // keys per stage
constexpr int kCtBand = 128;              // band rows per stage and head
constexpr int kCtTq = 64;                 // query rows of one head in the tile
constexpr int kCtTmemCols = 512;
constexpr int kCtColS = 0, kCtColG = 128, kCtColO = 256, kCtColP = 384;
constexpr int kCtStg = 2656;              // one softmax warp's bf16 staging: 32 rows of 5 chunks
constexpr int kCtMaxPages = 512;          // block-table entries a producer caches
constexpr int kCtMaxItems = 128;          // work items of one CTA whose keys are cached
constexpr int kCtMaxSeqs = 511;           // segments of the packed mode (offsets and tile prefix)

// Shared memory of one CTA.  The streaming mode (items of many stages) keeps three-deep K and V
// rings and one set of A tiles, refilled between items; the packed mode (items of about two
// stages) trades a ring slot for a second A set, so that the next item's tiles are ready before
// the current one ends.
template <bool PK>
struct CtSmem {
    static constexpr int kv_slots = PK ? 2 : 3;                   // depth of the K and V rings
    static constexpr int a_sets = PK ? 2 : 1;                     // sets of A tiles
    static constexpr int kv_tile = 2 * kCtBN * kRowBytes;         // 16 KB: two heads' 64 key rows
    static constexpr int head_band = kCtBand * kRowBytes;         // 16 KB
    static constexpr int band_tile = 2 * head_band;               // band h0 | band h1
    static constexpr int off_k = 0;                               // kv_slots K tiles
    static constexpr int off_v = off_k + kv_slots * kv_tile;      // kv_slots V tiles
    static constexpr int off_band = off_v + kv_slots * kv_tile;   // kBandSlots band tiles
    static_assert(kCtSoftmaxWarps * kCtStg <= band_tile, "staging overlays a band tile");
    static constexpr int q_tile = kCtTq * kRowBytes;              // 8 KB: 64 rows of one head
    // A set: bf16(q+u) in one tile [h0 rows | h0+1 rows] (the packed mode's q rows land there
    // and are converted in place), then bf16(q+v) in [h0 rows | zero | h0+1 rows], A0 starting
    // at 0 and A1 at q_tile
    static constexpr int a_set = 5 * q_tile;
    static constexpr int off_qu = off_band + kBandSlots * band_tile;   // set j at + j a_set
    static constexpr int off_qv = off_qu + 2 * q_tile;
    // streaming: the next item's q rows (TMA), 2 heads
    static constexpr int off_qbuf = off_qu + a_sets * a_set;
    static constexpr int off_xm = off_qbuf + (PK ? 0 : 2 * q_tile);   // [parity][half][row]
    static constexpr int off_btk = off_xm + 2 * 2 * 128 * 4;
    static constexpr int off_btv = off_btk + kCtMaxPages * 4;
    // per item 4 ints: streaming C, N; packed segment, first query, first and last key + 1
    static constexpr int off_len = off_btv + kCtMaxPages * 4;
    static constexpr int off_misc = off_len + 4 * kCtMaxItems * 4;   // tmem, abort
    // packed mode: segment offsets in the K producer's block-table cache, the per-segment
    // prefix of 64-query blocks in the V producer's
    static_assert(kCtMaxSeqs + 1 <= kCtMaxPages, "packed offsets fit a block-table cache");
    static constexpr int off_bar = off_misc + 64;
    static constexpr int n_bars = 4 * kv_slots + 2 * kBandSlots + 10 + 4 + 3 * 2 + 1;
    // streaming, an item split over a CTA pair: the partner's row weights for this CTA's head,
    // and each softmax thread's running max at the end of its last item
    static constexpr int off_xw = (off_bar + n_bars * 8 + 15) & ~15;
    static constexpr int off_mlast = off_xw + kCtTq * 4;
    static constexpr int bytes = off_mlast + (PK ? 0 : 32 * kCtSoftmaxWarps * 4) + 1024;
    static_assert(bytes <= 232448, "dynamic shared memory of one CTA");
    static_assert(kv_tile % 1024 == 0 && off_band % 1024 == 0 && off_qu % 1024 == 0 &&
                  off_qv % 1024 == 0 && off_qbuf % 1024 == 0 && a_set % 1024 == 0,
                  "TMA and MMA tiles need 1024-byte alignment");
};

struct CtArgs {
    const int32_t* block_table;
    const int32_t* cache_seqlens;
    const uint16_t* pos_bias_u;
    const uint16_t* pos_bias_v;
    uint16_t* out;
    unsigned* status;
    int B, T, H, R, num_blocks, block_size, bs_shift, box_rows, mbps;
    int k_max;               // keys a stream may have (the table's pages, the rel table's reach)
    uint32_t sign;           // 0x80008000 when the scale is negative (q+u, q+v are negated)
    float scale_log2;        // |scale| * log2(e)
    // packed mode
    const int32_t* cu_seqlens;
    int num_seqs, total, z, cs, left;
    // streaming, launched as CTA pairs: each CTA takes n_full items (c + k grid), and pair p <
    // n_split also splits item split_base + p by its key stages (0 = no split, no pairs)
    int n_full, n_split, split_base;
};

// One work item, as every role sees it: the global rows of its 64 query slots (nq of them real)
// and of its first key (packed mode), its heads h0 and h0 + 1, the keys [key0, key0 + nkeys) in
// the stream's or segment's own numbering, and the rel row of query slot 63 and key key0.
struct CtItem {
    int q_row0, nq, h0, key0, nkeys, kv_row0, rho_base;
    int b, seg_start, seg_len, i0;   // streaming: b; packed: the segment and first query
    int s_lo, s_hi;                  // the key stages this CTA runs
    bool xchg;                       // the other stages run on the pair's other CTA
};

// lo += bf16 low half of pair, hi += bf16 high half, each rounded once in fp32 (a bf16 value
// widens to fp32 exactly, so this equals widening first and adding in fp32)
__device__ __forceinline__ void ct_add_bf16x2(float& lo, float& hi, uint32_t pair)
{
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "add.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "r"(pair));
}

// A bounded wait: the first poll inline, the rest (sleeping polls, the abort flag, the time
// limit) out of line, so that the many wait sites cost a few instructions of code each (the
// kernel's roles run different code at once, and instruction fetch had become a stall).
__device__ __noinline__ bool ct_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort)
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
__device__ __forceinline__ bool ct_wait(uint32_t bar, uint32_t parity, volatile int* abort)
{
    return mbar_try_wait(bar, parity) || ct_wait_slow(bar, parity, abort);
}
// The bounded waits of the CTA's final drain, out of line.
__device__ __noinline__ bool ct_drain_wait(uint32_t bar, uint32_t parity) { return mbar_wait(bar, parity); }

// CTA pairs (a cluster of two): the partner's address of a shared variable, a store and an
// mbarrier arrival there (release at cluster scope), a bounded wait on this CTA's mbarrier that
// acquires at cluster scope, and the pair-wide barrier.
__device__ __forceinline__ uint32_t ct_mapa(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void ct_st_cluster_f32(uint32_t addr, float v)
{
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void ct_arrive_cluster(uint32_t remote_bar)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}
__device__ __noinline__ bool ct_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort)
{
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done)
                     : "r"(bar), "r"(parity)
                     : "memory");
        if (done) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            return false;
        }
    }
}
__device__ __forceinline__ void ct_cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// bf16(a + b) of two bf16 pairs, each rounded once: the same value as the fp32 sum rounded to
// bf16, since fp32 (24 bits) holds more than twice bf16's 8 bits plus two, where rounding twice
// cannot differ from rounding once
__device__ __forceinline__ uint32_t ct_bf16x2_add(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

template <bool PK>
__global__ void __launch_bounds__(ct_threads<PK>(), 1) chunk_attn_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_r, const CtArgs a)
{
    using SP = CtSmem<PK>;
    constexpr int kKvSlots = SP::kv_slots;
    constexpr int kCtThreads = ct_threads<PK>();
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived from the __shared__ array itself so that every access
    // through it stays a shared-space access
    uint8_t* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    unsigned err = 0;
    int* s_len = reinterpret_cast<int*>(sm + SP::off_len);        // [item][4]
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + SP::off_misc);
    volatile int* s_abort = reinterpret_cast<volatile int*>(sm + SP::off_misc + 4);
    const uint32_t bar_kfull = sb + SP::off_bar;             // [3] the stage's K landed
    const uint32_t bar_kempty = bar_kfull + 8 * kKvSlots;    // [3] the slot's K read (S/G done)
    const uint32_t bar_vfull = bar_kempty + 8 * kKvSlots;    // [3] the stage's V landed
    const uint32_t bar_vempty = bar_vfull + 8 * kKvSlots;    // [3] the slot's V read (P.V done)
    const uint32_t bar_bfull = bar_vempty + 8 * kKvSlots;    // [2] the stage's band landed
    const uint32_t bar_bempty = bar_bfull + 8 * kBandSlots;  // [2] the band tile (and staging) free
    const uint32_t bar_sg_full = bar_bempty + 8 * kBandSlots;  // S and G in TMEM
    const uint32_t bar_sg_free = bar_sg_full + 8;      // softmax warps have read S and G
    const uint32_t bar_p_full = bar_sg_free + 8;       // P written to TMEM
    const uint32_t bar_pv_done = bar_p_full + 8;       // P.V finished
    const uint32_t bar_q_ready = bar_pv_done + 8;      // bf16(q+u), bf16(q+v) written
    const uint32_t bar_q_free = bar_q_ready + 8;       // last S/G MMA of an item finished
    const uint32_t bar_drain = bar_q_free + 8;         // everything the S/G issuer issued finished
    const uint32_t bar_drain2 = bar_drain + 8;         // everything the P.V issuer issued finished
    const uint32_t bar_qb_full = bar_drain2 + 8;       // q rows of the next item landed
    const uint32_t bar_qb_free = bar_qb_full + 8;      // softmax warps have read the q rows
    const uint32_t bar_pair = bar_qb_free + 8;         // [4] softmax warp pair exchanged a value
    // packed mode, per A set: its q rows landed, its A tiles written, its last S/G MMA finished
    const uint32_t bar_afull = bar_pair + 8 * 4;       // [2]
    const uint32_t bar_aready = bar_afull + 8 * 2;     // [2]
    const uint32_t bar_afree = bar_aready + 8 * 2;     // [2]
    const uint32_t bar_xchg = bar_afree + 8 * 2;       // the pair's partial of this CTA's head landed
    const int Hp = a.H >> 1;
    __shared__ int s_my_items;

    if (warp == kCtKWarp && lane == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
    }
    if (warp == kCtVWarp && lane == 0) prefetch_tensormap(&tm_v);
    if (warp == kCtBandWarp && lane == 0) prefetch_tensormap(&tm_r);
    if (tid == 0) {
        for (int i = 0; i < kKvSlots; ++i) {
            mbar_init(bar_kfull + 8 * i, 1);
            mbar_init(bar_kempty + 8 * i, 1);
            mbar_init(bar_vfull + 8 * i, 1);
            mbar_init(bar_vempty + 8 * i, 1);
        }
        for (int i = 0; i < kBandSlots; ++i) {
            mbar_init(bar_bfull + 8 * i, 1);
            mbar_init(bar_bempty + 8 * i, kCtSoftmaxWarps);
        }
        mbar_init(bar_sg_full, 1);
        mbar_init(bar_sg_free, kCtSoftmaxWarps);
        mbar_init(bar_p_full, kCtSoftmaxWarps);
        mbar_init(bar_pv_done, 1);
        mbar_init(bar_q_ready, kCtSoftmaxWarps);
        mbar_init(bar_q_free, 1);
        mbar_init(bar_drain, 1);
        mbar_init(bar_drain2, 1);
        mbar_init(bar_qb_full, 1);
        mbar_init(bar_qb_free, kCtSoftmaxWarps);
        for (int i = 0; i < 4; ++i) mbar_init(bar_pair + 8 * i, 64);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_afull + 8 * i, 1);
            mbar_init(bar_aready + 8 * i, 2);
            mbar_init(bar_afree + 8 * i, 1);
        }
        mbar_init(bar_xchg, 4 * 32);   // every lane of the partner's four warps of the other head
        fence_mbar_init();
        *s_abort = 0;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(s_tmem)),
                     "r"(kCtTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // each set's zero block, shared by its two block-diagonal A tiles of G
    for (int i = tid; i < SP::a_sets * SP::q_tile / 16; i += kCtThreads)
        reinterpret_cast<uint4*>(sm + SP::off_qv + SP::q_tile + (i / (SP::q_tile / 16)) * SP::a_set)
            [i % (SP::q_tile / 16)] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    // Launched with programmatic stream serialization: everything the previous grid on the
    // stream wrote (the append of this step's chunk) is visible once this returns.
    grid_dep_wait();
    int* s_cu = reinterpret_cast<int*>(sm + SP::off_btk);     // packed: segment offsets
    int* s_pre = reinterpret_cast<int*>(sm + SP::off_btv);    // packed: blocks before segment s
    long long n_items;
    if constexpr (PK) {
        const int ns = a.num_seqs;
        for (int i = tid; i <= ns; i += kCtThreads) {
            int c = __ldg(a.cu_seqlens + i);
            if (c < 0 || c > a.total) { err |= kErrBounds; c = c < 0 ? 0 : a.total; }
            s_cu[i] = c;
        }
        __syncthreads();
        if (warp == 0) {
            // the exclusive prefix of each segment's 64-query blocks (lane l takes `per`
            // consecutive segments)
            const int per = (ns + 31) / 32;
            int mine = 0;
            for (int q = 0; q < per; ++q) {
                const int sg = lane * per + q;
                if (sg < ns) {
                    const int L = s_cu[sg + 1] - s_cu[sg];
                    if (L < 0) err |= kErrBounds;
                    mine += L > 0 ? (L + kCtTq - 1) / kCtTq : 0;
                }
            }
            int incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            int base = incl - mine;
            for (int q = 0; q < per; ++q) {
                const int sg = lane * per + q;
                if (sg < ns) {
                    s_pre[sg] = base;
                    const int L = s_cu[sg + 1] - s_cu[sg];
                    base += L > 0 ? (L + kCtTq - 1) / kCtTq : 0;
                }
            }
            if (lane == 31) s_pre[ns] = incl;
        }
        __syncthreads();
        n_items = static_cast<long long>(s_pre[ns]) * Hp;
    } else {
        n_items = static_cast<long long>(a.B) * Hp;
    }
    // Streaming on CTA pairs: the items c + k grid (k < n_full), then, for pair p < n_split, item
    // split_base + p split by key stages (the even CTA the first half, the odd one the rest; an
    // item of one stage stays whole on the even CTA).
    __shared__ int s_split_k;   // the split item's place in this CTA's list, or -1
    const bool pairs = !PK && a.n_split > 0;
    const long long split_item = a.split_base + static_cast<long long>(blockIdx.x >> 1);
    auto stages_of = [&](long long item, int& c, int& n) {
        c = __ldg(a.cache_seqlens + item / Hp);
        if (c < 0) { err |= kErrBounds; c = 0; }
        long long nn = static_cast<long long>(c) + a.T;
        if (nn > a.k_max) { err |= kErrBounds; nn = a.k_max; }
        n = static_cast<int>(nn);
        return (n + kCtBN - 1) / kCtBN;
    };
    if (tid == 0) {
        long long m;
        int sk = -1;
        if (pairs) {
            m = a.n_full;
            if ((blockIdx.x >> 1) < a.n_split) {
                int c, n;
                if ((blockIdx.x & 1) == 0 || stages_of(split_item, c, n) >= 2) sk = static_cast<int>(m++);
            }
        } else {
            m = n_items > blockIdx.x ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
        }
        if (m > kCtMaxItems) { err |= kErrBounds; m = kCtMaxItems; sk = -1; }   // the host bounds it
        s_my_items = static_cast<int>(m);
        s_split_k = sk;
    }
    __syncthreads();
    // the partner's mbarriers are initialised before any arrival from this CTA can reach them
    if (pairs) ct_cluster_sync();
    const int my_items = s_my_items;
    const int split_k = s_split_k;
    // every item's keys.  Streaming: the cache length and key count (keys past what the host
    // can bound are dropped and flagged, as is a negative cache length).  Packed: the segment,
    // the first query and the keys the block's queries see (from the first query's window start
    // to the last query's chunk end).
    for (int k = tid; k < my_items; k += kCtThreads) {
        const long long item = blockIdx.x + static_cast<long long>(k) * gridDim.x;
        if constexpr (PK) {
            const int blk = static_cast<int>(item / Hp);
            int lo = 0, hi = a.num_seqs - 1;   // the last segment whose blocks start at or before blk
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_pre[mid] <= blk) lo = mid; else hi = mid - 1;
            }
            const int i0 = (blk - s_pre[lo]) * kCtTq;
            const int L = s_cu[lo + 1] - s_cu[lo];
            const int ilast = (i0 + kCtTq < L ? i0 + kCtTq : L) - 1;
            int kl = (i0 / a.cs - a.left) * a.cs;
            kl = kl > 0 ? kl : 0;
            int kh = (ilast / a.cs + 1) * a.cs;
            kh = kh < L ? kh : L;
            s_len[4 * k] = lo;
            s_len[4 * k + 1] = i0;
            s_len[4 * k + 2] = kl;
            s_len[4 * k + 3] = kh;
        } else {
            int c, n;
            const int n_st = stages_of(k == split_k ? split_item : item, c, n);
            // the stages [lo, hi) this CTA runs: all of them, or its half of a split item
            int lo = 0, hi = n_st;
            if (k == split_k && n_st >= 2) {
                const int h = (n_st + 1) / 2;
                if (blockIdx.x & 1) lo = h; else hi = h;
            }
            s_len[4 * k] = c;
            s_len[4 * k + 1] = n;
            s_len[4 * k + 2] = lo;
            s_len[4 * k + 3] = hi;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;
    auto item_info = [&](int k) {
        CtItem it;
        const long long item = (!PK && k == split_k) ? split_item : blockIdx.x + static_cast<long long>(k) * gridDim.x;
        it.h0 = 2 * static_cast<int>(item % Hp);
        if constexpr (PK) {
            const int sg = s_len[4 * k];
            it.seg_start = s_cu[sg];
            it.seg_len = s_cu[sg + 1] - it.seg_start;
            it.i0 = s_len[4 * k + 1];
            it.key0 = s_len[4 * k + 2];
            it.nkeys = s_len[4 * k + 3] - it.key0;
            it.q_row0 = it.seg_start + it.i0;
            it.nq = it.seg_len - it.i0 < kCtTq ? it.seg_len - it.i0 : kCtTq;
            it.kv_row0 = it.seg_start + it.key0;
            it.rho_base = a.z - (it.i0 + kCtTq - 1) + it.key0;
            it.b = 0;
            it.s_lo = 0;
            it.s_hi = (it.nkeys + kCtBN - 1) / kCtBN;
            it.xchg = false;
        } else {
            it.b = static_cast<int>(item / Hp);
            const int C = s_len[4 * k];
            it.nkeys = s_len[4 * k + 1];
            it.key0 = 0;
            it.q_row0 = it.b * a.T;
            it.nq = a.T;
            it.kv_row0 = 0;
            it.rho_base = a.R - a.T - C - (kCtTq - 1);
            it.seg_start = it.seg_len = it.i0 = 0;
            it.s_lo = s_len[4 * k + 2];
            it.s_hi = s_len[4 * k + 3];
            it.xchg = k == split_k && (it.nkeys + kCtBN - 1) / kCtBN >= 2;
        }
        return it;
    };

    // The producers wait on the barrier itself (suspended until its phase completes), so that
    // they react at once and take no issue slots from the softmax warps meanwhile.
    auto prod_wait = [&](uint32_t bar, uint32_t parity) { return ct_wait(bar, parity, s_abort); };
    // Softmax warps take every wait together: a warp-wide vote keeps the warp converged for
    // the .sync.aligned tensor-memory instructions even if one lane's wait runs out.
    auto warp_wait = [&](uint32_t bar, uint32_t parity) {
        return __all_sync(0xffffffffu, ct_wait(bar, parity, s_abort)) != 0;
    };

    // One producer warp's page boxes of a stage: box q (one page, both heads) goes from lane q.
    // Returns the bytes the stage's boxes bring.
    auto page_boxes = [&](const CUtensorMap* map, const int* bt_row, int s, int N, int h0,
                          uint32_t dst0, uint32_t bar, uint64_t pol, bool issue) {
        const int j0 = s * kCtBN;
        const int jn = N - j0 < kCtBN ? N - j0 : kCtBN;
        const int nbox = a.box_rows == kCtBN ? 1 : (jn + a.box_rows - 1) >> a.bs_shift;
        if (issue && lane < nbox) {
            const int key = j0 + lane * a.box_rows;               // first key of the box
            const int blk = bt_row[key >> a.bs_shift];
            int row;
            if (blk >= 0 && blk < a.num_blocks) {
                row = (blk << a.bs_shift) + (key & (a.block_size - 1));
            } else {
                err |= kErrBounds;
                row = a.num_blocks << a.bs_shift;                 // past the pool: zero rows
            }
            tma_load_4d_hint(dst0 + lane * a.box_rows * 2 * kRowBytes, map, bar, 0, 0, h0, row >> 3, pol);
        }
        return nbox * a.box_rows * 2 * kRowBytes;
    };
    // the block-table row of stream b, pages [0, ceil(N / block_size)), into a producer's cache
    auto load_bt = [&](int* bt_row, int b, int N) {
        const int np = (N + a.block_size - 1) >> a.bs_shift;
        const int32_t* src = a.block_table + static_cast<long long>(b) * a.mbps;
        for (int p = lane; p < np; p += 32) bt_row[p] = __ldg(src + p);
        __syncwarp();
    };

    if (warp == kCtKWarp) {
        // --------------------------------------------------------- q rows and K producer
        int* bt_row = reinterpret_cast<int*>(sm + SP::off_btk);
        const uint64_t pol = policy_evict_first();   // every K and V row is read once
        int g = 0, itp = 0;
        bool ok = true;
        for (int k = 0; k < my_items && ok; ++k, ++itp) {
            const CtItem it = item_info(k);
            if (!PK) load_bt(bt_row, it.b, it.nkeys);
            // streaming: the item's q rows of both heads, once the softmax warps have read the
            // previous ones (the packed mode's go to the A-tile warp)
            if (!PK && lane == 0) {
                if (itp > 0 && !prod_wait(bar_qb_free, (itp - 1) & 1)) ok = false;
                if (ok) {
                    mbar_arrive_expect_tx(bar_qb_full, 2 * SP::q_tile);
                    tma_load_3d(sb + SP::off_qbuf, &tm_q, bar_qb_full, 0, it.h0, it.q_row0);
                    tma_load_3d(sb + SP::off_qbuf + SP::q_tile, &tm_q, bar_qb_full, 0, it.h0 + 1, it.q_row0);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            for (int s = it.s_lo; s < it.s_hi && ok; ++s, ++g) {
                const int u = g % kKvSlots, n = g / kKvSlots;
                if (lane == 0 && n > 0 && !prod_wait(bar_kempty + 8 * u, (n - 1) & 1)) ok = false;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                const uint32_t dst = sb + SP::off_k + u * SP::kv_tile;
                const uint32_t bar = bar_kfull + 8 * u;
                if constexpr (PK) {
                    // the stage's 64 key rows of each head (rows past the arrays read as zeros)
                    if (lane == 0) mbar_arrive_expect_tx(bar, SP::kv_tile);
                    __syncwarp();
                    if (lane < 2)
                        tma_load_3d_hint(dst + lane * (SP::kv_tile / 2), &tm_k, bar, 0, it.h0 + lane,
                                         it.kv_row0 + s * kCtBN, pol);
                } else {
                    const int kbytes = page_boxes(&tm_k, bt_row, s, it.nkeys, it.h0, dst, bar, pol, false);
                    if (lane == 0) mbar_arrive_expect_tx(bar, kbytes);
                    __syncwarp();
                    page_boxes(&tm_k, bt_row, s, it.nkeys, it.h0, dst, bar, pol, true);
                }
            }
        }
        // no copy may still be landing when the CTA exits
        if (lane == 0) {
            for (int x = g - kKvSlots; x < g; ++x)
                if (x >= 0 && !ct_drain_wait(bar_kfull + 8 * (x % kKvSlots), (x / kKvSlots) & 1)) *s_abort = 1;
            if (!PK && itp > 0 && !ct_drain_wait(bar_qb_full, (itp - 1) & 1)) *s_abort = 1;
        }
    } else if (warp == kCtVWarp) {
        // ---------------------------------------------------------------- V producer
        int* bt_row = reinterpret_cast<int*>(sm + SP::off_btv);
        const uint64_t pol = policy_evict_first();
        int g = 0;
        bool ok = true;
        for (int k = 0; k < my_items && ok; ++k) {
            const CtItem it = item_info(k);
            if (!PK) load_bt(bt_row, it.b, it.nkeys);
            for (int s = it.s_lo; s < it.s_hi && ok; ++s, ++g) {
                const int u = g % kKvSlots, n = g / kKvSlots;
                if (lane == 0 && n > 0 && !prod_wait(bar_vempty + 8 * u, (n - 1) & 1)) ok = false;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                const uint32_t dst = sb + SP::off_v + u * SP::kv_tile;
                const uint32_t bar = bar_vfull + 8 * u;
                if constexpr (PK) {
                    if (lane == 0) mbar_arrive_expect_tx(bar, SP::kv_tile);
                    __syncwarp();
                    if (lane < 2)
                        tma_load_3d_hint(dst + lane * (SP::kv_tile / 2), &tm_v, bar, 0, it.h0 + lane,
                                         it.kv_row0 + s * kCtBN, pol);
                } else {
                    const int vbytes = page_boxes(&tm_v, bt_row, s, it.nkeys, it.h0, dst, bar, pol, false);
                    if (lane == 0) mbar_arrive_expect_tx(bar, vbytes);
                    __syncwarp();
                    page_boxes(&tm_v, bt_row, s, it.nkeys, it.h0, dst, bar, pol, true);
                }
            }
        }
        if (lane == 0)
            for (int x = g - kKvSlots; x < g; ++x)
                if (x >= 0 && !ct_drain_wait(bar_vfull + 8 * (x % kKvSlots), (x / kKvSlots) & 1)) *s_abort = 1;
    } else if (warp == kCtBandWarp) {
        // ------------------------------------------------------------- band producer
        if (lane == 0) {
            int g = 0;
            bool ok = true;
            for (int k = 0; k < my_items && ok; ++k) {
                const CtItem it = item_info(k);
                for (int s = it.s_lo; s < it.s_hi; ++s, ++g) {
                    const int slot = g & 1;
                    if (g >= kBandSlots && !prod_wait(bar_bempty + 8 * slot, ((g >> 1) - 1) & 1)) { ok = false; break; }
                    // rel rows rho_min .. rho_min + 127 of both heads (rows outside the table
                    // read as zeros)
                    const int rho_min = it.rho_base + s * kCtBN;
                    const uint32_t dst = sb + SP::off_band + slot * SP::band_tile;
                    mbar_arrive_expect_tx(bar_bfull + 8 * slot, SP::band_tile);
                    tma_load_3d(dst, &tm_r, bar_bfull + 8 * slot, 0, it.h0, rho_min);
                    tma_load_3d(dst + SP::head_band, &tm_r, bar_bfull + 8 * slot, 0, it.h0 + 1, rho_min);
                }
            }
            for (int x = g - kBandSlots; x < g; ++x)
                if (x >= 0 && !ct_drain_wait(bar_bfull + 8 * (x & 1), (x >> 1) & 1)) *s_abort = 1;
        }
    } else if (warp == kCtMmaWarp) {
        // ------------------------------------------------------------ S/G issuer
        // Each tcgen05.mma holds its issuing thread until the tensor pipe takes it, so S/G and
        // P.V are issued from two threads: while one waits on a barrier the other's products run.
        if (lane == 0) {
            constexpr uint32_t id_s = idesc(128, 2 * kCtBN, 0), id_g = idesc(128, kCtBand, 0);
            int x = 0, nq = 0;   // stages issued
            bool ok = true;
            for (int k = 0; k < my_items && ok; ++k) {
                const CtItem itk = item_info(k);
                for (int s = itk.s_lo; s < itk.s_hi; ++s, ++x) {
                    // the item's A tiles (first stage), the stage's K and band, and the previous
                    // stage's S and G read by the softmax warps
                    ok = (s > itk.s_lo || (PK ? ct_wait(bar_aready + 8 * (k & 1), (k >> 1) & 1, s_abort)
                                       : ct_wait(bar_q_ready, k & 1, s_abort))) &&
                         ct_wait(bar_kfull + 8 * (x % kKvSlots), (x / kKvSlots) & 1, s_abort) &&
                         ct_wait(bar_bfull + 8 * (x & 1), (x >> 1) & 1, s_abort) &&
                         (x == 0 || ct_wait(bar_sg_free, (x - 1) & 1, s_abort));
                    if (!ok) break;
                    const uint32_t kbase = sb + SP::off_k + (x % kKvSlots) * SP::kv_tile;
                    const uint32_t bbase = sb + SP::off_band + (x & 1) * SP::band_tile;
                    const uint32_t aset = sb + (PK ? (k & 1) * SP::a_set : 0);
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_ss(tmem + kCtColS, sdesc(aset + SP::off_qu + 32 * kk), sdesc(kbase + 32 * kk), id_s, kk > 0);
#pragma unroll
                    for (int hd = 0; hd < 2; ++hd)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_ss(tmem + kCtColG, sdesc(aset + SP::off_qv + hd * SP::q_tile + 32 * kk),
                                    sdesc(bbase + hd * SP::head_band + 32 * kk), id_g, (hd | kk) ? 1 : 0);
                    umma_commit(bar_sg_full);
                    umma_commit(bar_kempty + 8 * (x % kKvSlots));   // the slot's K may be refilled
                    if (s + 1 == itk.s_hi) {   // the A tiles are free
                        umma_commit(PK ? bar_afree + 8 * (k & 1) : bar_q_free);
                        ++nq;
                    }
                }
            }
            // drain: every product issued here has finished and every arrival it owes has landed
            umma_commit(bar_drain);
            bool drained = ct_drain_wait(bar_drain, 0);
            if constexpr (PK) {
                for (int y = nq - 2; y < nq; ++y)
                    if (y >= 0) drained = ct_drain_wait(bar_afree + 8 * (y & 1), (y >> 1) & 1) && drained;
            } else if (nq > 0) {
                drained = ct_drain_wait(bar_q_free, (nq - 1) & 1) && drained;
            }
            if (x > 0) drained = ct_drain_wait(bar_sg_full, (x - 1) & 1) && drained;
            for (int y = x - kKvSlots; y < x; ++y)    // the last commits to each K slot
                if (y >= 0) drained = ct_drain_wait(bar_kempty + 8 * (y % kKvSlots), (y / kKvSlots) & 1) && drained;
            if (!drained) *s_abort = 1;
        }
    } else if (warp == kCtPvWarp) {
        // ------------------------------------------------------------ P.V issuer
        if (lane == 0) {
            constexpr uint32_t id_o = idesc(128, 128, 1);
            int g = 0;
            bool ok = true;
            for (int k = 0; k < my_items && ok; ++k) {
                const CtItem itk = item_info(k);
                const int n_keys = itk.nkeys;
                for (int s = itk.s_lo; s < itk.s_hi; ++s, ++g) {
                    ok = ct_wait(bar_p_full, g & 1, s_abort) &&
                         ct_wait(bar_vfull + 8 * (g % kKvSlots), (g / kKvSlots) & 1, s_abort);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t vbase = sb + SP::off_v + (g % kKvSlots) * SP::kv_tile;
                    // only over the 16-key steps that hold keys of the stream
                    const int kst = n_keys - s * kCtBN;
                    const int ksteps = kst < kCtBN ? (kst + 15) >> 4 : kCtBN / 16;
                    // B = [V_h0 | V_h1], MN-major.  Pool head pairs: a step's 16 keys are two 8-key
                    // groups 2 KB apart, and within a group head h0 + 1's atom follows h0's (1 KB);
                    // packed: each head's 64 rows in a tile of their own (8 KB apart)
#pragma unroll
                    for (int kk = 0; kk < kCtBN / 16; ++kk)
                        if (kk < ksteps)
                            umma_ts(tmem + kCtColO, tmem + kCtColP + 8 * kk,
                                    PK ? sdesc_mn(vbase + 2048 * kk, SP::kv_tile / 2, 1024)
                                       : sdesc_mn(vbase + 4096 * kk, 1024, 2048),
                                    id_o, (s > itk.s_lo || kk > 0) ? 1 : 0);
                    umma_commit(bar_pv_done);
                    umma_commit(bar_vempty + 8 * (g % kKvSlots));
                }
            }
            umma_commit(bar_drain2);
            bool drained = ct_drain_wait(bar_drain2, 0);
            if (g > 0) drained = ct_drain_wait(bar_pv_done, (g - 1) & 1) && drained;
            for (int y = g - kKvSlots; y < g; ++y)    // and to each V slot
                if (y >= 0) drained = ct_drain_wait(bar_vempty + 8 * (y % kKvSlots), (y / kKvSlots) & 1) && drained;
            if (!drained) *s_abort = 1;
        }
    } else if (PK && warp >= kCtPrepWarp) {
        // ------------------------------------------------------------- A tiles (packed)
        // Item k uses set k % 2: once the S/G MMAs of item k - 2 are done with it, its q rows of
        // both heads land in the set's q+u tile and become bf16(q+u) there and bf16(q+v) beside
        // it (rows past the segment zero).  Warp 13 + hd takes head h0 + hd; lane l takes
        // 16-byte chunk l % 8 of rows l / 8 + 4 j.
        const int hd = warp - kCtPrepWarp, c = lane & 7;
        bool ok = true;
        for (int k = 0; k < my_items && ok; ++k) {
            const CtItem it = item_info(k);
            const int set = k & 1;
            const uint32_t bar = bar_afull + 8 * set;
            uint8_t* qu = sm + SP::off_qu + set * SP::a_set + hd * SP::q_tile;
            uint8_t* qv = sm + SP::off_qv + set * SP::a_set + 2 * hd * SP::q_tile;
            if (hd == 0 && lane == 0) {
                if (k >= 2 && !prod_wait(bar_afree + 8 * set, ((k >> 1) - 1) & 1)) ok = false;
                if (ok) {
                    mbar_arrive_expect_tx(bar, 2 * SP::q_tile);
                    tma_load_3d(smem_addr(qu), &tm_q, bar, 0, it.h0, it.q_row0);
                    tma_load_3d(smem_addr(qu) + SP::q_tile, &tm_q, bar, 0, it.h0 + 1, it.q_row0);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            const uint4 uc = __ldg(reinterpret_cast<const uint4*>(a.pos_bias_u + (it.h0 + hd) * kHeadDim) + c);
            const uint4 vc = __ldg(reinterpret_cast<const uint4*>(a.pos_bias_v + (it.h0 + hd) * kHeadDim) + c);
            const uint32_t wu[4] = {uc.x, uc.y, uc.z, uc.w};
            const uint32_t wv[4] = {vc.x, vc.y, vc.z, vc.w};
            if (!ok || !warp_wait(bar, (k >> 1) & 1)) { ok = false; break; }
#pragma unroll 4
            for (int j = 0; j < kCtTq / 4; ++j) {
                const int row = (lane >> 3) + 4 * j;
                const uint32_t offs = swz128(row, c);
                uint4 ou4 = make_uint4(0u, 0u, 0u, 0u), ov4 = ou4;
                if (row < it.nq) {
                    const uint4 qc = *reinterpret_cast<const uint4*>(qu + offs);
                    const uint32_t w[4] = {qc.x, qc.y, qc.z, qc.w};
                    uint32_t ou[4], ov[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        ou[e] = ct_bf16x2_add(w[e], wu[e]) ^ a.sign;
                        ov[e] = ct_bf16x2_add(w[e], wv[e]) ^ a.sign;
                    }
                    ou4 = make_uint4(ou[0], ou[1], ou[2], ou[3]);
                    ov4 = make_uint4(ov[0], ov[1], ov[2], ov[3]);
                }
                *reinterpret_cast<uint4*>(qu + offs) = ou4;
                *reinterpret_cast<uint4*>(qv + offs) = ov4;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_aready + 8 * set);
        }
    } else if (warp < kCtSoftmaxWarps) {
        // ----------------------------------------------------------------- softmax
        const int quad = warp & 3, hf = warp >> 2;
        const int r = 32 * quad + lane;         // tile row == TMEM lane
        const int hd = quad >> 1;               // head of the pair
        const int i = r & (kCtTq - 1);          // query row of the chunk (padding when >= T)
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * quad) << 16);
        float* xm = reinterpret_cast<float*>(sm + SP::off_xm);   // [exchange parity][half][row]
        const uint32_t pbar = bar_pair + 8 * quad;
        int nx = 0;
        auto pair_post = [&](float mine) {
            xm[(nx & 1) * 256 + hf * 128 + r] = mine;
            mbar_arrive(pbar);
        };
        auto pair_collect = [&](float& theirs) {
            if (!warp_wait(pbar, nx & 1)) return false;
            theirs = xm[(nx & 1) * 256 + (1 - hf) * 128 + r];
            ++nx;
            return true;
        };
        // bf16(q+u) and bf16(q+v) of item number itq (heads h0, h0+1): this thread's half row,
        // from the q rows the producer staged; padding rows are zero.  The caller has made sure
        // the MMAs of the previous item no longer read the tiles.
        auto prep_q = [&](int itq, int h0, int nq) {
            if (!warp_wait(bar_qb_full, itq & 1)) return false;
            const uint4* up = reinterpret_cast<const uint4*>(a.pos_bias_u + (h0 + hd) * kHeadDim);
            const uint4* vp = reinterpret_cast<const uint4*>(a.pos_bias_v + (h0 + hd) * kHeadDim);
            const uint32_t dst_u = hd * SP::q_tile, dst_v = hd ? 2 * SP::q_tile : 0;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int c = 4 * hf + cc;
                const uint32_t offs = swz128(i, c);
                uint4 ou4 = make_uint4(0u, 0u, 0u, 0u), ov4 = ou4;
                if (i < nq) {
                    const uint4 qc = *reinterpret_cast<const uint4*>(sm + SP::off_qbuf + hd * SP::q_tile + offs);
                    const uint4 uc = __ldg(up + c);
                    const uint4 vc = __ldg(vp + c);
                    const uint32_t w[4] = {qc.x, qc.y, qc.z, qc.w};
                    const uint32_t wu[4] = {uc.x, uc.y, uc.z, uc.w};
                    const uint32_t wv[4] = {vc.x, vc.y, vc.z, vc.w};
                    uint32_t ou[4], ov[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        // a negative scale: negate q+u and q+v (exact in bf16)
                        ou[e] = ct_bf16x2_add(w[e], wu[e]) ^ a.sign;
                        ov[e] = ct_bf16x2_add(w[e], wv[e]) ^ a.sign;
                    }
                    ou4 = make_uint4(ou[0], ou[1], ou[2], ou[3]);
                    ov4 = make_uint4(ov[0], ov[1], ov[2], ov[3]);
                }
                *reinterpret_cast<uint4*>(sm + SP::off_qu + dst_u + offs) = ou4;
                *reinterpret_cast<uint4*>(sm + SP::off_qv + dst_v + offs) = ov4;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_qb_free);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_q_ready);
            return true;
        };
        int g = 0, it = 0, sg = 0;
        if (!PK && my_items > 0) {
            const CtItem it0 = item_info(0);
            if (!prep_q(0, it0.h0, it0.nq)) *s_abort = 1;
        }
        // O rows of a finished item: wait for its last P.V, combine the pair's sums, store.
        // It runs inside the next item's first stage, after that stage's S/G have been read.
        // An item split over the CTA pair: each CTA finishes one head (its rank's), so the warps
        // of the other head hand their normalised half of the rows to the partner (O through the
        // output rows the partner then overwrites, the row weight log2(l) + m into its shared
        // memory), and the warps of this CTA's head wait for the partner's half and merge.
        auto epilogue = [&](int e_row0, int e_nq, int e_h0, float e_l) {
            if (!warp_wait(bar_pv_done, (g - 1) & 1)) return false;
            float l_other;   // posted by the partner when its item ended
            if (!pair_collect(l_other)) return false;
            tc_fence_after();
            uint32_t oo[32];
            OASR_TMEM_LD32(tl + kCtColO + 64 * hd + 32 * hf, oo);
            tmem_wait_ld();
            if (i < e_nq) {
                const float inv = 1.f / (e_l + l_other);
                uint4* dst = reinterpret_cast<uint4*>(
                                 a.out + ((static_cast<long long>(e_row0) + i) * a.H + e_h0 + hd) * kHeadDim) + 4 * hf;
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
        // The same for the CTA's last item, which may be split over the pair (a split item is
        // always the last of its CTAs, so only this form carries the exchange).
        auto epilogue_last = [&](int e_row0, int e_nq, int e_h0, float e_l, float e_m, bool e_x) {
            if (!warp_wait(bar_pv_done, (g - 1) & 1)) return false;
            float l_other;   // posted by the partner when its item ended
            if (!pair_collect(l_other)) return false;
            tc_fence_after();
            uint32_t oo[32];
            OASR_TMEM_LD32(tl + kCtColO + 64 * hd + 32 * hf, oo);
            tmem_wait_ld();
            const float l_row = e_l + l_other;
            uint4* dst = reinterpret_cast<uint4*>(
                             a.out + ((static_cast<long long>(e_row0) + i) * a.H + e_h0 + hd) * kHeadDim) + 4 * hf;
            float co = 1.f / l_row, cp = 0.f;   // weights of this CTA's O and of the partner's
            const uint32_t rank = blockIdx.x & 1;
            if (e_x && hd == static_cast<int>(rank)) {
                if (!__all_sync(0xffffffffu, ct_wait_cluster(bar_xchg, 0, s_abort))) return false;
                if (i < e_nq) {
                    const float w_own = e_m + __log2f(l_row);
                    const float w_p = reinterpret_cast<const float*>(sm + SP::off_xw)[i];
                    const float mw = fmaxf(w_own, w_p);
                    const float ea = ex2_approx(w_own - mw), eb = ex2_approx(w_p - mw);
                    const float inv = 1.f / (ea + eb);
                    co = ea * inv / l_row;
                    cp = eb * inv;
                }
            }
            if (i < e_nq) {
                uint32_t w[16];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 part = cp != 0.f ? __ldcg(dst + c) : make_uint4(0u, 0u, 0u, 0u);
                    const uint32_t pw[4] = {part.x, part.y, part.z, part.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float lo = __uint_as_float(oo[8 * c + 2 * e]) * co;
                        float hi = __uint_as_float(oo[8 * c + 2 * e + 1]) * co;
                        if (cp != 0.f) {
                            lo += __uint_as_float(pw[e] << 16) * cp;
                            hi += __uint_as_float(pw[e] & 0xffff0000u) * cp;
                        }
                        w[4 * c + e] = pack_bf16(lo, hi);
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                if (e_x && hd != static_cast<int>(rank) && hf == 0)
                    ct_st_cluster_f32(ct_mapa(smem_addr(sm + SP::off_xw) + 4 * i, rank ^ 1u), e_m + __log2f(l_row));
            }
            // the half of the rows handed over: every lane of these warps signals the partner
            if (e_x && hd != static_cast<int>(rank)) ct_arrive_cluster(ct_mapa(bar_xchg, rank ^ 1u));
            tc_fence_before();
            return true;
        };
        // This warp's bf16 staging of the position term: row `lane` holds the 16-byte chunks
        // q0 .. q0+4 of its window (q0 = w0 / 4, w0 = (31 - lane) / 2 the first word it reads)
        // at 4 (5 lane + 2 (lane / 8)) words, so that both the chunk stores (the eight lanes of
        // a store phase share q0 and land in distinct bank quads) and the lane-shifted 4-byte
        // loads (32 distinct banks) are free of conflicts.
        const int w0 = (31 - lane) >> 1;
        const int q0 = w0 >> 2;
        const int stg_off = warp * kCtStg + 16 * (5 * lane + 2 * (lane >> 3));   // bytes
        int p_row0 = 0, p_nq = 0, p_h0 = 0;
        float p_l = 0.f;
        bool have_prev = false, all_ok = true;
        for (int k = 0; k < my_items && !*s_abort; ++k, ++it) {
            const CtItem itm = item_info(k);
            const int N = itm.nkeys;
            // packed: the keys this row sees, in the item's key numbering (none for padding rows)
            int win_lo = 0, win_hi = N;
            if constexpr (PK) {
                const int qi = itm.i0 + i;   // query index in the segment
                if (qi < itm.seg_len) {
                    const int ci = qi / a.cs;
                    int lo = (ci - a.left) * a.cs, hi = (ci + 1) * a.cs;
                    lo = lo > 0 ? lo : 0;
                    hi = hi < itm.seg_len ? hi : itm.seg_len;
                    win_lo = lo - itm.key0;
                    win_hi = hi - itm.key0;
                } else {
                    win_lo = win_hi = 0;
                }
            }
            float m_used = -INFINITY, l_sum = 0.f;
            bool ok = true;
            for (int s = itm.s_lo; s < itm.s_hi; ++s, ++g) {
                if (!warp_wait(bar_sg_full, sg & 1)) { ok = false; break; }
                ++sg;
                tc_fence_after();
                // the half holds keys jh .. jh+31 of the item; this row sees [ka, kb) of them
                const int jh = s * kCtBN + 32 * hf;
                const int ka = win_lo - jh;
                const int kb = win_hi - jh;
                // the staging tile overlays this stage's band tile (G has been computed from it)
                uint32_t* stg = reinterpret_cast<uint32_t*>(sm + SP::off_band + (g & 1) * SP::band_tile + stg_off);
                float sc[32];
                {
                    // position term, skewed: row i needs G[r][63 - i + j] (j the key of the
                    // stage); this warp's rows reach 63 columns for its half (window column
                    // 31 - lane + j), which go through the staging tile as bf16 pairs
                    uint32_t gr[64];
                    const uint32_t colg = kCtColG + static_cast<uint32_t>(32 * hf + 32 - 32 * (quad & 1));
                    OASR_TMEM_LD32(tl + colg, gr);
                    OASR_TMEM_LD32(tl + colg + 32, (gr + 32));
                    tmem_wait_ld();
#pragma unroll
                    for (int pc = 0; pc < 8; ++pc)
                        if (pc >= q0 && pc <= q0 + 4) {
                            uint32_t gw[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                gw[e] = pack_bf16(__uint_as_float(gr[8 * pc + 2 * e]),
                                                  __uint_as_float(gr[8 * pc + 2 * e + 1]));
                            *reinterpret_cast<uint4*>(stg + 4 * (pc - q0)) = make_uint4(gw[0], gw[1], gw[2], gw[3]);
                        }
                    uint32_t sr[32];
                    if constexpr (PK) {
                        // head-major keys: column 64 hd + key
                        OASR_TMEM_LD32(tl + kCtColS + 64 * hd + 32 * hf, sr);
                    } else {
                        // S columns of this half's keys 8 gg + e: 16 (4 hf + gg) + 8 hd + e
                        OASR_TMEM_LD8(tl + kCtColS + 64 * hf + 8 * hd, sr);
                        OASR_TMEM_LD8(tl + kCtColS + 64 * hf + 16 + 8 * hd, (sr + 8));
                        OASR_TMEM_LD8(tl + kCtColS + 64 * hf + 32 + 8 * hd, (sr + 16));
                        OASR_TMEM_LD8(tl + kCtColS + 64 * hf + 48 + 8 * hd, (sr + 24));
                    }
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) sc[j] = __uint_as_float(sr[j]);
                }
                // S and G are read: the issuer may compute the next stage's into the same columns
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_sg_free);
                {
                    // an even lane's window starts on the odd half of word w0: its pairs are
                    // realigned with a byte permute
                    const uint32_t sel = (lane & 1) ? 0x3210u : 0x5432u;
                    const uint32_t* rd = stg + (w0 & 3);
                    uint32_t wa = rd[0];
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        const uint32_t wb = rd[m + 1];
                        ct_add_bf16x2(sc[2 * m], sc[2 * m + 1], __byte_perm(wa, wb, sel));
                        wa = wb;
                    }
                }
                // the band tile (staging included) is no longer read: its next stage may land
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_bempty + 8 * (g & 1));
                // last stage of the item: the next item's A tiles, so that its first S/G can be
                // issued while this stage's softmax and the epilogue run
                if (!PK && s + 1 == itm.s_hi && k + 1 < my_items) {
                    const CtItem nx1 = item_info(k + 1);
                    if (!warp_wait(bar_q_free, it & 1) || !prep_q(it + 1, nx1.h0, nx1.nq)) { ok = false; break; }
                }
                // the previous item's O, now that this first stage's S/G are read
                if (s == itm.s_lo && have_prev) {
                    if (!epilogue(p_row0, p_nq, p_h0, p_l)) { ok = false; break; }
                    have_prev = false;
                }
                // mask keys past the stream's history; this half's max (scores unscaled: the
                // scale, > 0 with its sign folded into q+u and q+v, is applied to the row max
                // and inside the exponent's FFMA)
                float mx0 = -INFINITY, mx1 = -INFINITY;
                if (ka <= 0 && kb >= 32) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        mx0 = fmax3(mx0, sc[j], sc[j + 1]);
                        mx1 = fmax3(mx1, sc[j + 2], sc[j + 3]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) sc[j + e] = (j + e >= ka && j + e < kb) ? sc[j + e] : -INFINITY;
                        mx0 = fmax3(mx0, sc[j], sc[j + 1]);
                        mx1 = fmax3(mx1, sc[j + 2], sc[j + 3]);
                    }
                }
                float mx = fmaxf(mx0, mx1) * a.scale_log2, mx_other;
                pair_post(mx);
                // P.V of the previous stage must be done before P and O are touched
                if (s > itm.s_lo && !warp_wait(bar_pv_done, (g - 1) & 1)) { ok = false; break; }
                if (!pair_collect(mx_other)) { ok = false; break; }
                mx = fmaxf(mx, mx_other);
                const bool rescale = mx > m_used + 8.f;   // keeps every P <= 2^8 between rescales
                const float m_new = rescale ? mx : m_used;
                if (s > itm.s_lo && __any_sync(0xffffffffu, rescale)) {
                    const float alpha = ex2_approx(m_used - m_new);
                    l_sum *= alpha;
                    tc_fence_after();
                    uint32_t oo[32];
                    OASR_TMEM_LD32(tl + kCtColO + 64 * hd + 32 * hf, oo);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) oo[j] = __float_as_uint(__uint_as_float(oo[j]) * alpha);
                    OASR_TMEM_ST32(tl + kCtColO + 64 * hd + 32 * hf, oo);
                }
                m_used = m_new;
                // a row that has seen no key yet (a packed window that starts later, a padding
                // row) has max -inf: its P is 0, not NaN
                {
                    const float mref = m_used == -INFINITY ? 0.f : m_used;
                    float2 ps = make_float2(0.f, 0.f);
                    const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
                    const float2 nm2 = make_float2(-mref, -mref);
                    uint32_t pk[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float2 e2 = __ffma2_rn(make_float2(sc[2 * j], sc[2 * j + 1]), sc2, nm2);
                        const float2 p2 = make_float2(ex2_approx(e2.x), ex2_approx(e2.y));
                        ps = __fadd2_rn(ps, p2);
                        pk[j] = pack_bf16(p2.x, p2.y);
                    }
                    OASR_TMEM_ST16(tl + kCtColP + 16 * hf, pk);
                    l_sum += ps.x + ps.y;
                }
                // V rows past the history: P.V stops at the 16-key step holding the last key;
                // that step's rows past it (stale pool rows, possibly non-finite) are zeroed so
                // that P = 0 there never meets a non-finite value.  Rows 0-63 of the tile are the
                // stage's keys: warps of quadrants 0 and 1 zero them in head hf's V tile.
                const int kstage = N - s * kCtBN;
                const int k16 = (kstage + 15) & ~15;
                if (kstage < k16 && quad < 2 && 32 * quad < k16 && 32 * quad + 32 > kstage) {
                    if (!warp_wait(bar_vfull + 8 * (g % kKvSlots), (g / kKvSlots) & 1)) { ok = false; break; }
                    if (r >= kstage && r < k16) {
                        uint4* vrow = reinterpret_cast<uint4*>(
                            sm + SP::off_v + (g % kKvSlots) * SP::kv_tile +
                            (PK ? hf * (SP::kv_tile / 2) + r * kRowBytes : ((r >> 3) * 2 + hf) * 1024 + (r & 7) * kRowBytes));
#pragma unroll
                        for (int c = 0; c < 8; ++c) vrow[c] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_p_full);
            }
            if (!ok) { all_ok = false; break; }
            pair_post(l_sum);   // this half's sum, for the pair's epilogue
            p_row0 = itm.q_row0;
            p_nq = itm.nq;
            p_h0 = itm.h0;
            p_l = l_sum;
            if (!PK && k + 1 == my_items) reinterpret_cast<float*>(sm + SP::off_mlast)[tid] = m_used;
            have_prev = true;
        }
        // the last item's O
        if (all_ok && have_prev && !*s_abort) {
            if constexpr (PK)
                epilogue(p_row0, p_nq, p_h0, p_l);
            else
                epilogue_last(p_row0, p_nq, p_h0, p_l, reinterpret_cast<const float*>(sm + SP::off_mlast)[tid],
                              item_info(my_items - 1).xchg);
        }
    }
    grid_dep_trigger();
    // every role has stopped issuing and the MMA issuer has drained the tensor pipe
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCtTmemCols));
    }
    // a CTA of a pair stays until its partner no longer writes into its shared memory
    if (pairs) ct_cluster_sync();
    if (tid == 0 && *s_abort) err |= kErrTimeout;
    if (err) atomicOr(a.status, err);
}

int g_smem_done_ct[2][64];

// How many CTA pairs (clusters of two) of the streaming kernel the current device holds at
// once; 0 if it cannot tell.  Looked up once per device.
int ct_pair_capacity(int threads, int smem)
{
    static std::mutex mu;
    static int cap[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (cap[dev] == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = static_cast<size_t>(smem);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, chunk_attn_tc_kernel<false>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        cap[dev] = n > 0 ? n : -1;
    }
    return cap[dev] > 0 ? cap[dev] : 0;
}

}  // namespace

// Whether the tensor-core kernel takes a bf16 streaming call of this shape: 33 <= T <= 64, an
// even head count, and coordinates and per-CTA work items within its limits.
bool chunk_tc_takes(int B, int T, int H, int mbps, int num_blocks, int block_size, int R)
{
    if (T < 33 || T > kCtTq || (H & 1) || mbps > kCtMaxPages) return false;
    if (static_cast<long long>(num_blocks) * block_size + kCtBN >= 0x7fffffffLL ||
        static_cast<long long>(B) * T + kCtTq >= 0x7fffffffLL ||
        static_cast<long long>(R) + kCtBand >= 0x7fffffffLL)
        return false;
    const int sms = sm_count();
    if (!sms) return false;
    const long long n_items = static_cast<long long>(B) * (H / 2);
    const long long grid = n_items < sms ? n_items : sms;
    return (n_items + grid - 1) / grid <= kCtMaxItems;
}

// Host launcher used by the streaming entry points for the shapes chunk_tc_takes accepts
// (bf16; the caller has validated the arguments).
oasr_status launch_chunk_tc(const void* q, const void* k_pool, const void* v_pool, int num_blocks,
                            int block_size, const int32_t* bt, int mbps, const int32_t* cs,
                            const void* u, const void* vb, const void* rel, int R, void* out,
                            int B, int T, int H, int k_max, float scale, cudaStream_t stream)
{
    if (!chunk_tc_takes(B, T, H, mbps, num_blocks, block_size, R)) return OASR_ERR_UNSUPPORTED;
    const int sms = sm_count();
    const long long n_items = static_cast<long long>(B) * (H / 2);
    int grid = static_cast<int>(n_items < sms ? n_items : sms);
    const int box = block_size < kCtBN ? block_size : kCtBN;
    CUtensorMap tm_q, tm_k, tm_v, tm_r;
    if (!encode_rows_bf16(&tm_q, q, static_cast<long long>(B) * T, H, kCtTq) ||
        !encode_head_pairs_bf16(&tm_k, k_pool, static_cast<long long>(num_blocks) * block_size, H, box) ||
        !encode_head_pairs_bf16(&tm_v, v_pool, static_cast<long long>(num_blocks) * block_size, H, box) ||
        !encode_rows_bf16(&tm_r, rel, R, H, kCtBand))
        return OASR_ERR_INVALID_ARG;
    unsigned* status = status_word();
    if (!status) return OASR_ERR_CUDA;
    constexpr int smem = CtSmem<false>::bytes;
    if (!ensure_smem(chunk_attn_tc_kernel<false>, smem, g_smem_done_ct[0])) return OASR_ERR_CUDA;
    CtArgs a;
    a.block_table = bt;
    a.cache_seqlens = cs;
    a.pos_bias_u = static_cast<const uint16_t*>(u);
    a.pos_bias_v = static_cast<const uint16_t*>(vb);
    a.out = static_cast<uint16_t*>(out);
    a.status = status;
    a.B = B;
    a.T = T;
    a.H = H;
    a.R = R;
    a.num_blocks = num_blocks;
    a.block_size = block_size;
    a.bs_shift = __builtin_ctz(static_cast<unsigned>(block_size));
    a.box_rows = box;
    a.mbps = mbps;
    a.k_max = k_max;
    a.sign = scale < 0.f ? 0x80008000u : 0u;
    // > 0 even for a zero scale, so that a masked score (-inf) times it stays -inf
    a.scale_log2 = fmaxf(fabsf(scale) * 1.4426950408889634f, 1e-30f);
    // Items do not divide evenly over the SMs (at most half a wave left over): the leftover
    // items are split by key stages over CTA pairs, so that no CTA runs a whole extra item.
    a.n_full = a.n_split = a.split_base = 0;
    const int pairs = ct_pair_capacity(ct_threads<false>(), smem);
    if (pairs > 0) {
        const long long g2 = (2LL * pairs < sms ? 2LL * pairs : sms) & ~1LL;
        const long long full = g2 > 0 ? n_items / g2 : 0, extra = n_items - full * g2;
        if (g2 >= 2 && extra > 0 && extra <= g2 / 2 && full + 1 <= kCtMaxItems) {
            grid = static_cast<int>(full > 0 ? g2 : 2 * extra);
            a.n_full = static_cast<int>(full);
            a.n_split = static_cast<int>(extra);
            a.split_base = static_cast<int>(full * g2);
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(ct_threads<false>());
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.n_split > 0 ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, chunk_attn_tc_kernel<false>, tm_q, tm_k, tm_v, tm_r, a) != cudaSuccess)
        return OASR_ERR_CUDA;
    return launch_status();
}

// Host launcher of the packed mode (oasr_packed_relattn_chunked, bf16, chunk_size >= 1): returns
// OASR_ERR_UNSUPPORTED (nothing launched) for an odd head count, more than kCtMaxSeqs segments
// or more work items per CTA than it caches, so that the caller falls back to its other kernel.
oasr_status launch_chunk_tc_packed(const void* q, const void* k, const void* v,
                                   const int32_t* cu_seqlens, int num_seqs, int total,
                                   const void* pos_bias_u, const void* pos_bias_v, const void* rel,
                                   int R, void* out, int H, float scale, int cs, int left,
                                   cudaStream_t stream)
{
    if ((H & 1) || num_seqs < 1 || num_seqs > kCtMaxSeqs || cs < 1 || left < 0)
        return OASR_ERR_UNSUPPORTED;
    if (static_cast<long long>(total) + 2 * kCtTq >= 0x7fffffffLL ||
        static_cast<long long>(R) + kCtBand >= 0x7fffffffLL)
        return OASR_ERR_UNSUPPORTED;
    const int sms = sm_count();
    if (!sms) return OASR_ERR_CUDA;
    // work items: at most one 64-query block per 64 frames plus one per segment, per head pair
    const long long items_bound = (static_cast<long long>(total) / kCtTq + num_seqs) * (H / 2);
    const int grid = static_cast<int>(items_bound < sms ? items_bound : sms);
    if ((items_bound + grid - 1) / grid > kCtMaxItems) return OASR_ERR_UNSUPPORTED;
    CUtensorMap tm_q, tm_k, tm_v, tm_r;
    if (!encode_rows_bf16(&tm_q, q, total, H, kCtTq) || !encode_rows_bf16(&tm_k, k, total, H, kCtBN) ||
        !encode_rows_bf16(&tm_v, v, total, H, kCtBN) || !encode_rows_bf16(&tm_r, rel, R, H, kCtBand))
        return OASR_ERR_INVALID_ARG;
    unsigned* status = status_word();
    if (!status) return OASR_ERR_CUDA;
    constexpr int smem = CtSmem<true>::bytes;
    if (!ensure_smem(chunk_attn_tc_kernel<true>, smem, g_smem_done_ct[1])) return OASR_ERR_CUDA;
    CtArgs a = {};
    a.pos_bias_u = static_cast<const uint16_t*>(pos_bias_u);
    a.pos_bias_v = static_cast<const uint16_t*>(pos_bias_v);
    a.out = static_cast<uint16_t*>(out);
    a.status = status;
    a.H = H;
    a.R = R;
    a.sign = scale < 0.f ? 0x80008000u : 0u;
    a.scale_log2 = fmaxf(fabsf(scale) * 1.4426950408889634f, 1e-30f);
    a.cu_seqlens = cu_seqlens;
    a.num_seqs = num_seqs;
    a.total = total;
    a.z = (R - 1) / 2;
    a.cs = cs;
    a.left = left;
    return launch_pdl(chunk_attn_tc_kernel<true>, dim3(grid), dim3(ct_threads<true>()), smem, stream, tm_q,
                      tm_k, tm_v, tm_r, a);
}

}  // namespace oasr
