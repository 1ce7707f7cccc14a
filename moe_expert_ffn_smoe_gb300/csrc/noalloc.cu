// ffn_batch_q4_noalloc: the token-batch FFN with its workspace in a static
// device array, for callers that must not allocate device memory (see
// include/smoe.h).  It checks the sizes against the array and then calls the
// ordinary ffn_batch_q4 with the array's device address as the workspace.
#include <mutex>

#include "internal.h"
#include "smoe.h"

namespace {

// The workspace of every ffn_batch_q4_noalloc call on this device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SMOE_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (in host code the symbol itself is only a host-side stand-in).
// A cudaDeviceReset() unloads the module, so the library is not used again
// on a device after one (include/smoe.h, "Devices").
void *scratch_device_address()
{
    constexpr int kMaxDevices = 64;
    static void *addr[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace

extern "C" int ffn_batch_q4_noalloc(const uint8_t *gate_codes, const float *gate_scales,
                                    const uint8_t *up_codes, const float *up_scales,
                                    const uint8_t *down_codes, const float *down_scales,
                                    const float *X, float *Y, int T, int d_model, int d_ff,
                                    int group, void *stream)
{
    if (T < 0) return SMOE_ERR_SHAPE;
    // the shape is checked for every T (T == 0 included), as ffn_batch_q4 does
    const size_t need = smoe_ffn_batch_workspace_bytes(T, d_model, d_ff, group);
    if (need == static_cast<size_t>(-1)) return SMOE_ERR_SHAPE;
    if (need > SMOE_NOALLOC_SCRATCH_BYTES) return SMOE_ERR_SHAPE;
    if (T == 0 || d_model == 0) return SMOE_OK;
    void *scratch = scratch_device_address();
    if (!scratch) return SMOE_ERR_LAUNCH;
    return ffn_batch_q4(gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, X,
                        Y, T, d_model, d_ff, group, scratch, SMOE_NOALLOC_SCRATCH_BYTES, stream);
}
