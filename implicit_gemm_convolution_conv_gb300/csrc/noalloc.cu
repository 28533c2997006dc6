// Forward convolution without any allocation by the caller or the library.
//
// The CUDA-core implicit-GEMM path needs one piece of scratch: the weights
// re-laid out as [tap][C][OCp]. gbconv_conv_fwd_noalloc keeps that scratch in
// a fixed array compiled into the library instead of in a caller workspace.
// It exists for callers that cannot obtain device memory themselves: code
// running inside a region where cudaMalloc is forbidden or would block (for
// example a stream being captured into a CUDA graph, or a real-time loop
// that must not enter the driver's allocator), and plain-C hosts that have no
// caching allocator and do not want to manage a workspace buffer.
//
// Costs and rules, for a user of this entry point:
//  - Every GPU that loads the library holds kNoallocScratchBytes of device
//    memory for this array until the process exits.
//  - All calls on a device share the one array. Calls whose kernels overlap
//    on that GPU (different streams, or host threads racing) overwrite each
//    other's packed weights; serialise them on one stream.
//  - The array keeps whatever the last call wrote. Nothing in it has to start
//    at zero: each call rewrites every byte it reads, zero padding included.
//  - The first call on a device looks up the array's device address with
//    cudaGetSymbolAddress (with that device current) and caches it; make that
//    first call before any stream capture begins. The cached address belongs
//    to the device's primary context: after cudaDeviceReset (or anything
//    else that destroys that context) it is stale, so such a process must
//    not call this entry point again.
//  - The fused max pool (flags bit 2) lives only in the direct kernel, so a
//    descriptor that asks for it is rejected with GBCONV_ERR_ALGO.
#include <mutex>

#include "internal.h"

namespace gbconv {
// Defined in api.cu.
gbconv_status make_problem(const gbconv_desc *d, int ndim, Problem *p);
}

namespace {

constexpr size_t kNoallocScratchBytes = GBCONV_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself. In host code this name is only a host-side handle of
// the symbol, not a device address; host code must pass the address returned
// by cudaGetSymbolAddress to kernels.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_addr_mutex;
void *g_addr[kMaxDevices] = {};

// Device address of the scratch on the current device (looked up once per
// device, with that device current).
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_addr_mutex);
    if (!g_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return cudaSuccess;
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }
bool overlap(const void *a, size_t an, const void *b, size_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + bn && b0 < a0 + an;
}

}  // namespace

extern "C" gbconv_status gbconv_conv_fwd_noalloc(const gbconv_desc *desc, int ndim,
                                                 const void *x, const void *w,
                                                 const float *b, void *y,
                                                 cudaStream_t stream) {
    using namespace gbconv;
    if (!desc) return GBCONV_ERR_NULL;
    if (desc->algo != GBCONV_ALGO_AUTO && desc->algo != GBCONV_ALGO_IGEMM_FFMA)
        return GBCONV_ERR_ALGO;
    if (desc->w_layout != GBCONV_W_OIHW) return GBCONV_ERR_LAYOUT;
    gbconv_desc d = *desc;
    d.algo = GBCONV_ALGO_IGEMM_FFMA;
    d.workspace = nullptr;
    d.workspace_bytes = 0;
    Problem p;
    gbconv_status st = make_problem(&d, ndim, &p);
    if (st != GBCONV_OK) return st;
    const size_t wp_bytes = packed_weight_bytes(p);
    if (wp_bytes > kNoallocScratchBytes) return GBCONV_ERR_TOO_LARGE;
    if (!x || !w || !y) return GBCONV_ERR_NULL;
    if (!aligned(x, p.elt) || !aligned(w, p.elt) || !aligned(y, p.elt) || (b && !aligned(b, 4)))
        return GBCONV_ERR_ALIGN;
    const size_t yb = (size_t)p.y_elems * p.elt;
    if (overlap(y, yb, x, (size_t)p.x_elems * p.elt) ||
        overlap(y, yb, w, (size_t)p.w_elems * p.elt) ||
        overlap(y, yb, b, b ? (size_t)p.OC * 4 : 0))
        return GBCONV_ERR_OVERLAP;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || !gbconv_device_supported(dev)) {
        cudaGetLastError();
        return GBCONV_ERR_UNSUPPORTED_DEVICE;
    }
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) {
        cudaGetLastError();
        return GBCONV_ERR_CUDA;
    }
    if (overlap(y, yb, scratch, wp_bytes)) return GBCONV_ERR_OVERLAP;
    cudaError_t e = launch_pack_ffma(p, w, scratch, stream);
    // no workspace: no split-K partial sums either
    if (e == cudaSuccess) e = launch_igemm_ffma(p, x, scratch, b, y, nullptr, 0, stream);
    return launch_status(e);   // the same mapping as the regular forward call
}
