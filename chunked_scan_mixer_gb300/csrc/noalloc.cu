// Forward entry point for callers that cannot allocate device memory.
//
// hla2_forward takes its scratch space from the caller.  Some callers have no way to get
// device memory for it: plug-in hosts that hand out only the input and output buffers, or
// programs without a device allocator of their own.  hla2_forward_noalloc serves them: its
// scratch is a fixed array in the library's device memory (kScratchBytes on every GPU on
// which the library's kernels are loaded, held until the process exits), and it calls no
// allocation routine of CUDA, of any library or of PyTorch.
#include <mutex>

#include "kernels.h"

namespace hla2 {
int set_last_error(int code, const char* fmt, ...);
}

extern "C" int hla2_workspace_status(const void* workspace, hla2_stream_t stream);
extern "C" int hla2_selftest_wait_timeout(void* workspace, hla2_stream_t stream);

namespace {

constexpr size_t kScratchBytes = 32u << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of g_scratch on the current device, looked up once per device (with that
// device current).  In host code the name g_scratch is only a host-side stand-in.
int scratch_pointer(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return hla2::set_last_error(HLA2_ERR_CUDA, "hla2_forward_noalloc: no usable current device");
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return hla2::set_last_error(HLA2_ERR_CUDA, "hla2_forward_noalloc: scratch address lookup failed: %s",
                                        cudaGetErrorString(e));
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return HLA2_OK;
}

}  // namespace

extern "C" int hla2_forward_noalloc(const void* q, const void* k, const void* v, void* out, int B, int H, int n,
                                    int d, int dv, const float* gamma, int normalize, int chunk, int dtype,
                                    float eps, hla2_stream_t stream) {
    const size_t need = hla2_forward_workspace_bytes(B, H, n, d, dv, chunk, dtype, normalize, 0);
    if (need != (size_t)-1 && need > kScratchBytes)
        return hla2::set_last_error(HLA2_ERR_WORKSPACE,
                                    "hla2_forward_noalloc: these sizes need %zu bytes of scratch; the "
                                    "allocation-free entry point has %zu (use hla2_forward with a workspace)",
                                    need, kScratchBytes);
    void* scratch = nullptr;
    if (need != (size_t)-1 && need > 0) {
        const int rc = scratch_pointer(&scratch);
        if (rc != HLA2_OK) return rc;
    }
    hla2_opts o{};
    o.dtype = dtype;
    o.eps = eps;
    o.workspace = scratch;
    o.workspace_bytes = scratch ? kScratchBytes : 0;
    return hla2_forward(q, k, v, out, B, H, n, d, dv, gamma, normalize, chunk, stream, &o);
}

// The scratch array starts with the same status word as a caller's workspace; a caller of
// this entry point has no address for it, so these two read it and run the wait self-test
// on it for them.
extern "C" int hla2_noalloc_status(hla2_stream_t stream) {
    void* scratch = nullptr;
    const int rc = scratch_pointer(&scratch);
    if (rc != HLA2_OK) return rc;
    return hla2_workspace_status(scratch, stream);
}

extern "C" int hla2_noalloc_selftest_wait_timeout(hla2_stream_t stream) {
    void* scratch = nullptr;
    const int rc = scratch_pointer(&scratch);
    if (rc != HLA2_OK) return rc;
    return hla2_selftest_wait_timeout(scratch, stream);
}
