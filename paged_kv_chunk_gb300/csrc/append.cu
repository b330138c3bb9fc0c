// oasr_paged_append: scatter the chunk's K/V rows into the block-paged pools.
//
// ASR Engine page, section 4.3 "Batched paged forward", step 1: the new chunk is written
// into each stream's pool blocks through its block_table; the caller advances
// cache_seqlens afterwards.  Row t of stream b lands at logical position
// p = cache_seqlens[b] + t: block block_table[b][p / block_size], slot p % block_size.
//
// One thread moves one 16-byte vector; consecutive threads cover consecutive vectors of
// a head row, so both the chunk reads and the pool writes are coalesced 128-byte (bf16)
// or 256-byte (fp32) row segments.
#include "host_common.h"
#include "ptx.cuh"

namespace oasr {
namespace {

__global__ void __launch_bounds__(256) paged_append_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, uint4* __restrict__ k_pool,
    uint4* __restrict__ v_pool, int num_blocks, int block_size,
    const int32_t* __restrict__ block_table, int mbps, const int32_t* __restrict__ cache_seqlens,
    int T, int H, int vpr, long long n_vec, unsigned* status)
{
    grid_dep_wait();     // the previous grid on the stream has finished (programmatic launch)
    unsigned err = 0;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
         idx < 2 * n_vec; idx += stride) {
        const bool is_v = idx >= n_vec;
        const long long e = is_v ? idx - n_vec : idx;       // vector index in [B,T,H,vpr]
        const long long row = e / vpr;                     // (b*T + t)*H + h
        const int c = static_cast<int>(e - row * vpr);
        const int h = static_cast<int>(row % H);
        const long long bt_ = row / H;
        const int t = static_cast<int>(bt_ % T);
        const int b = static_cast<int>(bt_ / T);
        const long long p = static_cast<long long>(__ldg(cache_seqlens + b)) + t;
        const long long lb = p / block_size;
        if (p < 0 || lb >= mbps) { err |= kErrBounds; continue; }
        const int slot = static_cast<int>(p - lb * block_size);
        const int blk = __ldg(block_table + static_cast<long long>(b) * mbps + lb);
        if (blk < 0 || blk >= num_blocks) { err |= kErrBounds; continue; }
        const long long dst =
            ((static_cast<long long>(blk) * block_size + slot) * H + h) * vpr + c;
        if (is_v)
            v_pool[dst] = __ldg(v_new + e);
        else
            k_pool[dst] = __ldg(k_new + e);
    }
    // this thread's copies are issued: the next grid may schedule (it waits for this one)
    grid_dep_trigger();
    if (err) atomicOr(status, err);
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
    unsigned* status = status_word();
    const int sms = sm_count();
    if (!status || !sms) return OASR_ERR_CUDA;
    const int vpr = D * es / 16;
    const long long n_vec = static_cast<long long>(B) * T * H * vpr;
    long long blocks = (2 * n_vec + 255) / 256;
    if (blocks > 16LL * sms) blocks = 16LL * sms;
    return launch_pdl(paged_append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                      static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), num_blocks,
                      block_size, block_table, max_blocks_per_seq, cache_seqlens, T, H, vpr, n_vec,
                      status);
}
