// Library-wide host entry points: device check, status text, device status word.
#include <mutex>

#include "common.cuh"

namespace tern {

namespace {
constexpr int kMaxDevices = 64;
struct DevInfo {
    std::once_flag once;
    int status = TERN_ERR_CUDA;
    int num_sms = 0;
};
DevInfo g_dev[kMaxDevices];
}  // namespace

// The kernels are built for sm_103a only: accept compute capability 10.3.
int check_device(int* num_sms) {
    int dev = 0;
    TERN_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return TERN_ERR_DEVICE;
    DevInfo& d = g_dev[dev];
    std::call_once(d.once, [&] {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            d.status = TERN_ERR_CUDA;
            return;
        }
        d.num_sms = sms;
        d.status = (major == 10 && minor == 3) ? TERN_OK : TERN_ERR_DEVICE;
    });
    if (num_sms) *num_sms = d.num_sms;
    return d.status;
}

}  // namespace tern

extern "C" const char* tern_strerror(int status) {
    switch (status) {
    case TERN_OK: return "ok";
    case TERN_ERR_ARG: return "invalid argument (null pointer, size, theta or clamp)";
    case TERN_ERR_ALIGN: return "alignment: K and N must be multiples of 16 and pointers 16-byte aligned";
    case TERN_ERR_CUDA: return "a CUDA runtime or driver call failed";
    case TERN_ERR_TIMEOUT: return "a bounded device-side wait gave up";
    case TERN_ERR_WORKSPACE: return "workspace too small";
    case TERN_ERR_DEVICE: return "current device is not an sm_103 (GB300) GPU";
    case TERN_ERR_SCRATCH_LIMIT:
        return "problem too large for the built-in scratch of tern_linear_bwd_noalloc (use tern_linear_bwd)";
    default: return "unknown status";
    }
}

extern "C" int tern_device_status(void* stream, int clear) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TERN_ERR_CUDA;
    return tern::gemm_status_read(clear);
}
