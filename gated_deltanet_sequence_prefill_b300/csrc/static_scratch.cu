// static_scratch.cu -- gdn_chunk_fwd_staged_static: the staged prefill with
// its scratch in one fixed device array, for callers that cannot allocate
// device memory (see gdn.h for the contract).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gdn.h"

namespace {

// The scratch: one array per device, created when the library's module is
// loaded on that device and held until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[GDN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;

// Device address of the array, per device, together with the identity of the
// context it was looked up in.  A device reset (cudaDeviceReset) destroys the
// primary context and the library's module with it; the next context loads
// the module again, possibly at another address, and has a new context id,
// so the address is looked up again.
struct ScratchSlot {
    bool valid;
    unsigned long long ctx_id;
    void* addr;
};
ScratchSlot g_slots[kMaxDevices];
std::mutex g_scratch_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (false if there is none
// or the driver cannot tell).
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the array in the current device's context.  In host code
// the array's name is only a host-side stand-in, so kernels must be given
// this address, never the name.  The lookup (cudaGetSymbolAddress, with the
// device current) runs once per device and context; later calls reuse it.
cudaError_t scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchSlot& slot = g_slots[dev];
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    if (!slot.valid || !have_id || slot.ctx_id != id) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);  // also creates the context if needed
        if (e != cudaSuccess) return e;
        const bool known = current_context_id(&id);
        slot.valid = known;  // without a context id, look it up on every call
        slot.ctx_id = id;
        slot.addr = p;
        *out = p;
        return cudaSuccess;
    }
    *out = slot.addr;
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
