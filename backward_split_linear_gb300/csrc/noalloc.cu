// RMSNorm gamma-gradient reduction for callers that cannot allocate device
// memory: the float32 partial sums live in a fixed array inside this library
// instead of in caller scratch.
//
// Who needs it: code that receives only its input and output tensors from a
// host framework (a plugin or custom-op interface that offers no workspace),
// and code whose device memory is owned entirely by another allocator, where
// a cudaMalloc of its own would fail or would synchronise the device.
//
// The array below is a file-scope __device__ variable: every GPU that loads
// the library holds it until the process exits.  Host code cannot use its
// name as a device address (there it names a host-side stand-in), so the
// device address is looked up once per device with cudaGetSymbolAddress and
// passed to the kernels like any other pointer.
#include <mutex>

#include "../../include/zb.h"
#include "launch.h"

namespace {

// 512 KiB of float32 partial sums: the most the reduction's partition takes
// for any hidden <= 131072, at any token count.
constexpr size_t kStaticScratchFloats = static_cast<size_t>(zbk::kGammaMaxPartialFloats);

__device__ __align__(256) float g_gamma_scratch[kStaticScratchFloats];

// Device address of g_gamma_scratch on the current device, looked up on the
// first call for that device (with that device current) and kept for the
// process.  cudaDeviceReset() on a device invalidates the kept address, so the
// library must not be used on that device again afterwards.  nullptr on
// failure.
float* static_scratch() {
    static float* ptrs[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gamma_scratch) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<float*>(p);
    }
    return ptrs[dev];
}

}  // namespace

extern "C" size_t zb_op_rmsnorm_backward_gamma_noalloc_max_floats(void) { return kStaticScratchFloats; }

extern "C" zb_status zb_op_rmsnorm_backward_gamma_noalloc(const void* dn, const void* x, const float* rstd,
                                                          float* dgamma, int32_t tokens, int32_t hidden,
                                                          void* stream) {
    auto rows_ok = [tokens](const void* p) {
        return tokens == 0 ? (p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0)
                           : (p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0);
    };
    if (tokens < 0 || tokens > (1 << 24) || hidden <= 0 || hidden > (1 << 20) || hidden % 64 != 0)
        return ZB_ERR_SHAPE;
    if (!rows_ok(dn) || !rows_ok(x) || !rows_ok(rstd) || !dgamma ||
        (reinterpret_cast<uintptr_t>(dgamma) & 15u) != 0)
        return ZB_ERR_ARG;
    // The partial sums must fit the fixed array: they take exactly the bytes
    // zb_op_rmsnorm_backward_gamma_scratch_bytes(T, H) reports (the partition's
    // parts * H floats), which fit for every T when H <= 131072.
    if (zbk::rmsnorm_gamma_scratch_bytes(tokens, hidden) > kStaticScratchFloats * sizeof(float))
        return ZB_ERR_SHAPE;
    if (zbk::device_arch() != 103) return zbk::device_arch() < 0 ? ZB_ERR_CUDA : ZB_ERR_DEVICE;
    float* scratch = static_scratch();
    if (!scratch) return ZB_ERR_CUDA;
    const cudaError_t e = zbk::launch_rmsnorm_backward_gamma(dn, x, rstd, dgamma, tokens, hidden, scratch,
                                                              static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ZB_OK : ZB_ERR_CUDA;
}
