// static_scratch.cu -- gdn_chunk_fwd_staged_static: the staged prefill with
// its scratch in one fixed device array, for callers that cannot allocate
// device memory (see gdn.h for the contract).
#include <cuda_runtime.h>

#include <mutex>

#include "gdn.h"

namespace {

// The scratch: one array per device, created when the library's module is
// loaded on that device and held until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[GDN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the array on the current device, looked up once per
// device.  In host code the array's name is only a host-side stand-in, so
// kernels must be given this address, never the name.
cudaError_t scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" gdn_status gdn_chunk_fwd_staged_static(const void* q, const void* k, const void* v,
                                                  const float* log_alpha, const float* beta,
                                                  const float* h0, const int32_t* cu_seqlens,
                                                  int n_seqs, int64_t T_total, int H, int dk,
                                                  int dv, gdn_dtype io_dtype, int delta_rule,
                                                  void* o, float* h_T, int* device_status,
                                                  void* stream) {
    const size_t need = gdn_staged_workspace_size(T_total, H, dk, dv, n_seqs, io_dtype);
    if (need > GDN_STATIC_SCRATCH_BYTES) return GDN_ERR_WORKSPACE;
    void* ws = nullptr;
    if (need > 0) {  // need == 0: bad sizes, reported by the staged call below
        if (scratch_address(&ws) != cudaSuccess) {
            cudaGetLastError();
            return GDN_ERR_CUDA;
        }
    }
    gdn_status s = gdn_chunk_fwd_staged(q, k, v, log_alpha, beta, h0, cu_seqlens, n_seqs, T_total,
                                        H, dk, dv, io_dtype, delta_rule, o, h_T, ws,
                                        GDN_STATIC_SCRATCH_BYTES, stream);
    if (s == GDN_OK && device_status != nullptr) {
        // the status word is the first int of the scratch (written by the call's plan kernel)
        if (cudaMemcpyAsync(device_status, ws, sizeof(int), cudaMemcpyDeviceToDevice,
                            (cudaStream_t)stream) != cudaSuccess) {
            cudaGetLastError();
            return GDN_ERR_CUDA;
        }
    }
    return s;
}
