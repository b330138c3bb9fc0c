// Fixed-window history eviction (oasr_window_commit): the commit that follows a streaming
// step when the encoder has a trained attention window.
//
// ASR Engine page, KV-pool sizing paragraphs: an encoder with a trained window pages by
// chunk and retains ceil(window / chunk) + 1 pages per stream, and with history eviction the
// cached length is held at the window; section 4.3 "Batched paged forward": the caller
// commits the cache length after the step.  Per stream, after a chunk of T frames the
// stream holds n = C + T frames in its first P = ceil(n / block_size) pages; beyond the
// window the oldest d = ceil((n - window) / block_size) pages are dropped by rotating those
// P entries left by d (the dropped blocks become the next pages to be written) and the
// cached length becomes n - d * block_size, else n.  Eviction moves whole pages, so d never
// exceeds the floor(n / block_size) full ones: a window shorter than a page keeps the partly
// written newest page rather than a negative length.  Relative positions make the shift of
// every remaining frame's page index invisible to the attention.
//
// One warp per stream: the lanes gather the row's first P entries into registers, then
// write them back rotated.
#include "host_common.h"
#include "ptx.cuh"

namespace oasr {
namespace {

constexpr int kWinMaxPages = 512;

__global__ void __launch_bounds__(128) window_commit_kernel(int32_t* __restrict__ bt,
                                                            int32_t* __restrict__ cs, int B,
                                                            int mbps, int bs, int T, int window,
                                                            unsigned* status)
{
    grid_dep_wait();     // the previous grid on the stream has finished (programmatic launch)
    grid_dep_trigger();
    const int b = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (b >= B) return;
    unsigned err = 0;
    const int C = cs[b];
    long long n = static_cast<long long>(C) + T;
    if (C < 0) {
        err = kErrBounds;
        n = T;
    }
    int P = static_cast<int>((n + bs - 1) / bs);
    if (P > mbps) {   // the append dropped the rows past the table
        err = kErrBounds;
        P = mbps;
        n = static_cast<long long>(mbps) * bs;
    }
    int d = 0;
    if (n > window) {
        const long long want = (n - window + bs - 1) / bs, full = n / bs;
        d = static_cast<int>(want < full ? want : full);
    }
    int32_t* row = bt + static_cast<long long>(b) * mbps;
    int32_t vals[kWinMaxPages / 32];
#pragma unroll
    for (int k = 0; k < kWinMaxPages / 32; ++k) {
        const int i = lane + 32 * k;
        vals[k] = i < P ? row[i] : 0;
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < kWinMaxPages / 32; ++k) {
        const int i = lane + 32 * k;
        if (i < P) row[i >= d ? i - d : i - d + P] = vals[k];
    }
    if (lane == 0) {
        cs[b] = static_cast<int32_t>(n - static_cast<long long>(d) * bs);
        if (err) atomicOr(status, err);
    }
}

}  // namespace
}  // namespace oasr

extern "C" oasr_status oasr_window_commit(int32_t* block_table, int32_t* cache_seqlens, int B,
                                          int max_blocks_per_seq, int block_size, int T,
                                          int window_frames, cudaStream_t stream)
{
    using namespace oasr;
    if (!block_table || !cache_seqlens || B <= 0 || max_blocks_per_seq <= 0 || block_size <= 0 ||
        T < 0 || window_frames < 0)
        return OASR_ERR_INVALID_ARG;
    if (max_blocks_per_seq > kWinMaxPages) return OASR_ERR_UNSUPPORTED;
    unsigned* status = status_word();
    if (!status) return OASR_ERR_CUDA;
    return launch_pdl(window_commit_kernel, dim3((B + 3) / 4), dim3(128), 0, stream, block_table,
                      cache_seqlens, B, max_blocks_per_seq, block_size, T, window_frames, status);
}
