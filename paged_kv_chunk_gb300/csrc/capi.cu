// Library-wide entry points (status strings, device status word, version) and the host
// helpers declared in host_common.h.
#include <mutex>

#include "host_common.h"

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

}  // namespace oasr

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
