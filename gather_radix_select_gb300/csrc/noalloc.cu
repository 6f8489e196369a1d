// noalloc.cu -- sel_topk for callers that cannot allocate device memory.
//
// sel_topk needs a caller-owned workspace when it splits a few wide rows over
// several CTAs.  Some callers have no way to provide one: code that runs while
// a framework owns the whole device pool (a serving engine that reserves all
// free HBM for its caches at start-up), code inside an allocator callback that
// must not re-enter the allocator, or plain C callers without a device
// allocator of their own.  sel_topk_noalloc gives them the same results with
// the scratch taken from a fixed array that lives in this library's device
// image instead.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/sel.h"
#include "sel_internal.h"

namespace {

// The scratch itself: SEL_NOALLOC_SCRATCH_BYTES of device memory in this module.  Every GPU
// that loads the library holds one copy until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SEL_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};  // device address of g_noalloc_scratch, per device

// In host code the array's name is only a host-side stand-in; the device address comes from
// cudaGetSymbolAddress, with the device current (the caller's).  The address belongs to the
// current context: a device reset (or another context made current) can move the array.  So it
// is looked up again on every call whose stream is not capturing a graph; a capturing call uses
// the address the last non-capturing call on this device found (or looks it up if there was none).
int scratch_address(cudaStream_t stream, void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SEL_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return SEL_EUNSUPPORTED;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return SEL_ECUDA;
    std::lock_guard<std::mutex> g(g_mu);
    if (cs == cudaStreamCaptureStatusNone || !g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SEL_ECUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SEL_OK;
}

}  // namespace

extern "C" {

int sel_topk_noalloc(const void *x, int dtype, int64_t rows, int64_t cols, int64_t stride, const int32_t *row_end,
                     int k, int sorted_index, int idx_dtype, int want_values, void *out_idx, int64_t out_idx_stride,
                     void *out_val, int64_t out_val_stride, int32_t *nan_flag, int32_t *err_flag, void *stream)
{
    // sel_topk's own argument errors come first, then the scratch limit
    const int chk = sel::check_topk_call(x, dtype, rows, cols, stride, k, sorted_index, idx_dtype, want_values, out_idx,
                                         out_idx_stride, out_val, out_val_stride);
    if (chk != SEL_OK || rows == 0) return chk;
    const size_t need = sel_topk_workspace_size(dtype, rows, cols, k);
    if (need > static_cast<size_t>(SEL_NOALLOC_SCRATCH_BYTES)) return SEL_ESCRATCH;
    void *ws = nullptr;
    if (need > 0) {
        const int st = scratch_address(static_cast<cudaStream_t>(stream), &ws);
        if (st != SEL_OK) return st;
    }
    return sel_topk(x, dtype, rows, cols, stride, row_end, k, sorted_index, idx_dtype, want_values, out_idx,
                    out_idx_stride, out_val, out_val_stride, ws, need > 0 ? SEL_NOALLOC_SCRATCH_BYTES : 0, nan_flag,
                    err_flag, stream);
}

}  // extern "C"
