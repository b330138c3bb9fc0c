// Host-side helpers shared by the entry points: argument checks, the device status word
// and TMA tensor-map encoding.  No allocation; the only state is a per-device cache of
// the status word's address and of kernel attributes.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "oasr_attn.h"

namespace oasr {

// Device address of the status word on the current device (nullptr on failure).
unsigned* status_word();

// Number of SMs of the current device (cached; 0 on failure).
int sm_count();

// Encode a 3-D bf16 tensor map over rows of [rows, H, 64] with a box of box_rows rows of
// one head, 128-byte swizzled.  Returns false if the driver rejects it.
bool encode_rows_bf16(CUtensorMap* map, const void* base, long long rows, int H, int box_rows);

// Encode a 4-D bf16 tensor map over the rows of [rows, H, 64] (rows a multiple of 8) viewed as
// {64, row % 8, head, row / 8}, with a box of two adjacent heads and box_rows rows (a multiple
// of 8), 128-byte swizzled: in shared memory a box is [row / 8][head][row % 8][64], so every
// 8 rows of one head form one 1 KB swizzle atom.  Returns false if the driver rejects it.
bool encode_head_pairs_bf16(CUtensorMap* map, const void* base, long long rows, int H, int box_rows);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline oasr_status launch_status()
{
    return cudaGetLastError() == cudaSuccess ? OASR_OK : OASR_ERR_CUDA;
}

// Launch with programmatic stream serialization: the grid's CTAs may be scheduled while the
// previous grid on the stream drains.  Every kernel launched this way executes
// griddepcontrol.wait before its first global access, so it still sees all of the previous
// grid's writes.
template <typename... KArgs, typename... Args>
oasr_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, int smem,
                       cudaStream_t stream, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...) != cudaSuccess)
        return OASR_ERR_CUDA;
    return launch_status();
}

// Raise the dynamic shared-memory limit of `func` once per device.
template <typename F>
bool ensure_smem(F* func, int bytes, int (&done)[64])
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (done[dev] >= bytes) return true;
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(func),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return false;
    done[dev] = bytes;
    return true;
}

}  // namespace oasr
