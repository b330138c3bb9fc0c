// Library-wide entry points (status strings, device status word, version) and the host
// helpers declared in host_common.h.
#include <mutex>

#include "host_common.h"
#include "ptx.cuh"

namespace oasr {

// OR of kErrBounds / kErrTimeout raised by any kernel of this library on this device.
__device__ unsigned g_status_word;

namespace {
// Signature of the driver's cuTensorMapEncodeTiled (resolved at run time, so the library
// links against the CUDA runtime only).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::mutex g_mu;
unsigned* g_status_ptr[64];
int g_sms[64];

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}
}  // namespace

unsigned* status_word()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<unsigned*>(p);
    }
    return g_status_ptr[dev];
}

int sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

bool encode_rows_bf16(CUtensorMap* map, const void* base, long long rows, int H, int box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn || rows < 1 || H < 1 || box_rows < 1 || box_rows > 256 || !aligned16(base))
        return false;
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[2] = {64 * 2, static_cast<cuuint64_t>(H) * 64 * 2};
    const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_head_pairs_bf16(CUtensorMap* map, const void* base, long long rows, int H, int box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn || rows < 8 || (rows & 7) || H < 2 || box_rows < 8 || box_rows > 256 || (box_rows & 7) ||
        !aligned16(base))
        return false;
    const cuuint64_t dims[4] = {64, 8, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows / 8)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(H) * 64 * 2, 64 * 2,
                                   static_cast<cuuint64_t>(H) * 64 * 2 * 8};
    const cuuint32_t box[4] = {64, 8, 2, static_cast<cuuint32_t>(box_rows / 8)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
// A wait on a barrier that no thread or copy ever signals: it runs out after limit_ns and
// takes the path every pipeline wait of the library takes when it runs out.
__global__ void __launch_bounds__(32) selftest_wait_kernel(uint64_t limit_ns, unsigned* status)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const bool ok = mbar_wait(b, 0, limit_ns);
    if (threadIdx.x == 0 && !ok) atomicOr(status, kErrTimeout);
}
}  // namespace

}  // namespace oasr

extern "C" oasr_status oasr_selftest_wait(unsigned limit_us, cudaStream_t stream)
{
    using namespace oasr;
    if (limit_us < 1 || limit_us > 2000000) return OASR_ERR_INVALID_ARG;
    unsigned* status = status_word();
    if (!status) return OASR_ERR_CUDA;
    selftest_wait_kernel<<<1, 32, 0, stream>>>(static_cast<uint64_t>(limit_us) * 1000ull, status);
    return launch_status();
}

extern "C" const char* oasr_status_string(oasr_status s)
{
    switch (s) {
    case OASR_OK: return "ok";
    case OASR_ERR_INVALID_ARG: return "invalid argument";
    case OASR_ERR_UNSUPPORTED: return "unsupported size or dtype";
    case OASR_ERR_CUDA: return "CUDA error";
    case OASR_ERR_BOUNDS: return "device index out of range";
    case OASR_ERR_TIMEOUT: return "kernel wait timed out";
    }
    return "unknown status";
}

extern "C" oasr_status oasr_device_status(unsigned* flags, int clear)
{
    if (!flags) return OASR_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return OASR_ERR_CUDA;
    if (cudaMemcpyFromSymbol(flags, oasr::g_status_word, sizeof(unsigned)) != cudaSuccess)
        return OASR_ERR_CUDA;
    if (clear) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(oasr::g_status_word, &zero, sizeof(unsigned)) != cudaSuccess)
            return OASR_ERR_CUDA;
    }
    return OASR_OK;
}

extern "C" int oasr_version(void) { return 100; }
