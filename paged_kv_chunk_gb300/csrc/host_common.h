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

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline oasr_status launch_status()
{
    return cudaGetLastError() == cudaSuccess ? OASR_OK : OASR_ERR_CUDA;
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
