// noalloc.cu -- decode attention for callers that cannot allocate device memory: the scratch
// lives in a fixed array of this module instead of a caller-provided workspace.
#include <mutex>

#include "../../include/oscar_kv.h"
#include "internal.h"

namespace {

constexpr size_t kFixedScratchBytes = (size_t)16 << 20;   // 16 MiB, held by every GPU that loads us

// The device array.  In host code its name is only a stand-in for the device address, which
// cudaGetSymbolAddress resolves per device below.
static __device__ __align__(256) unsigned char g_fixed_scratch[kFixedScratchBytes];

std::mutex g_mu;
void* g_addr[oscar::kMaxDevices] = {nullptr};

// Device address of the array on the current device (looked up once per device).
int fixed_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return OSCAR_ECUDA;
    if (dev < 0 || dev >= oscar::kMaxDevices) return OSCAR_EINVAL;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fixed_scratch);
        if (e != cudaSuccess || !p) return OSCAR_ECUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return OSCAR_OK;
}

}  // namespace

extern "C" int oscar_decode_attention_noalloc(oscar_cache* c, const void* q, int32_t q_dtype, const float* rk,
                                              void* out, int32_t out_dtype, void* stream) {
    void* scratch = nullptr;
    int rc = fixed_scratch(&scratch);
    if (rc != OSCAR_OK) return rc;
    oscar::DecodeParams p;
    rc = oscar::noalloc_decode_params(c, q, q_dtype, rk, out, out_dtype, scratch, kFixedScratchBytes, &p,
                                      (cudaStream_t)stream);
    if (rc != OSCAR_OK) return rc;
    cudaError_t e = oscar::launch_decode(p, (cudaStream_t)stream);
    return e == cudaSuccess ? OSCAR_OK : OSCAR_ECUDA;
}

// The error word sits at a fixed offset of the array, so it can be read without knowing the
// layout the last call used.  Reading it allocates nothing: the copy goes to a host variable.
extern "C" int oscar_decode_status_noalloc(void* stream) {
    void* scratch = nullptr;
    int rc = fixed_scratch(&scratch);
    if (rc != OSCAR_OK) return rc;
    int32_t err = 0;
    cudaError_t e = cudaMemcpyAsync(&err, (const unsigned char*)scratch + oscar::kNoallocErrOffset, sizeof(err),
                                    cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return OSCAR_ECUDA;
    return err ? OSCAR_ETIMEOUT : OSCAR_OK;
}
