// oasr_paged_append: scatter the chunk's K/V rows into the block-paged pools.
//
// ASR Engine page, section 4.3 "Batched paged forward", step 1: the new chunk is written
// into each stream's pool blocks through its block_table; the caller advances
// cache_seqlens afterwards.  Row t of stream b lands at logical position
// p = cache_seqlens[b] + t: block block_table[b][p / block_size], slot p % block_size.
//
// One warp moves one frame of one tensor: its H heads are contiguous both in the chunk and
// in the pool row, so the reads and the writes are coalesced H * 128-byte (bf16) or
// H * 256-byte (fp32) rows.
#include "host_common.h"
#include "ptx.cuh"

namespace oasr {
namespace {

// One warp per (K or V, stream b, frame t): it reads the frame's H heads (H * vpr 16-byte
// vectors, contiguous in k_new / v_new) and writes them into the pool row of position
// cache_seqlens[b] + t (also contiguous: a pool row holds all heads of one frame).
__global__ void __launch_bounds__(256) paged_append_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, uint4* __restrict__ k_pool,
    uint4* __restrict__ v_pool, int num_blocks, int block_size,
    const int32_t* __restrict__ block_table, int mbps, const int32_t* __restrict__ cache_seqlens,
    int B, int T, int row_vecs, unsigned* status)
{
    grid_dep_wait();     // the previous grid on the stream has finished (programmatic launch)
    const int rows = B * T;   // per tensor (host check: 2 * rows fits an int)
    const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    unsigned err = 0;
    if (w < 2 * rows) {
        const bool is_v = w >= rows;
        const int r = is_v ? w - rows : w;   // b * T + t
        const int b = r / T, t = r - (r / T) * T;
        const long long src = static_cast<long long>(r) * row_vecs;
        const uint4* in = is_v ? v_new : k_new;
        // the frame's first 4 * 32 vectors are requested before the cache length and the
        // table entry (they do not depend on them), so the three loads overlap
        uint4 pre[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (lane + 32 * u < row_vecs) pre[u] = __ldg(in + src + lane + 32 * u);
        const long long p = static_cast<long long>(__ldg(cache_seqlens + b)) + t;
        const long long lb = p / block_size;
        int blk = -1;
        if (p < 0 || lb >= mbps) {
            err = kErrBounds;
        } else {
            blk = __ldg(block_table + static_cast<long long>(b) * mbps + lb);
            if (blk < 0 || blk >= num_blocks) err = kErrBounds;
        }
        if (!err) {
            const long long dst = (static_cast<long long>(blk) * block_size + (p - lb * block_size)) * row_vecs;
            uint4* out = is_v ? v_pool : k_pool;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (lane + 32 * u < row_vecs) out[dst + lane + 32 * u] = pre[u];
            for (int c = lane + 128; c < row_vecs; c += 32) out[dst + c] = __ldg(in + src + c);
        }
    }
    // this thread's copies are issued: the next grid may schedule (it waits for this one)
    grid_dep_trigger();
    if (err && lane == 0) atomicOr(status, err);
}

}  // namespace
}  // namespace oasr

extern "C" oasr_status oasr_paged_append(const void* k_new, const void* v_new, void* k_pool,
                                         void* v_pool, int num_blocks, int block_size,
                                         const int32_t* block_table, int max_blocks_per_seq,
                                         const int32_t* cache_seqlens, int B, int T, int H, int D,
                                         oasr_dtype dt, cudaStream_t stream)
{
    using namespace oasr;
    if (!k_new || !v_new || !k_pool || !v_pool || !block_table || !cache_seqlens)
        return OASR_ERR_INVALID_ARG;
    if (num_blocks <= 0 || block_size <= 0 || max_blocks_per_seq <= 0 || B <= 0 || T <= 0 ||
        H <= 0 || D <= 0)
        return OASR_ERR_INVALID_ARG;
    if (dt != OASR_F32 && dt != OASR_BF16) return OASR_ERR_UNSUPPORTED;
    const int es = dt == OASR_F32 ? 4 : 2;
    if ((D * es) % 16 != 0) return OASR_ERR_UNSUPPORTED;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
        return OASR_ERR_INVALID_ARG;
    if (2LL * B * T > 0x7fffffffLL / 32) return OASR_ERR_UNSUPPORTED;
    unsigned* status = status_word();
    if (!status) return OASR_ERR_CUDA;
    const int row_vecs = H * D * es / 16;   // 16-byte vectors of one frame (all heads)
    const int warps = 2 * B * T;
    return launch_pdl(paged_append_kernel, dim3(static_cast<unsigned>((warps + 7) / 8)), dim3(256), 0,
                      stream, static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                      static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), num_blocks,
                      block_size, block_table, max_blocks_per_seq, cache_seqlens, B, T, row_vecs,
                      status);
}
