// noalloc.cu -- a forward entry point that allocates nothing.
//
// rdot_forward asks the caller for a small device workspace (the status word the kernels
// report into). Some callers cannot provide one: a plugin running inside a host framework whose
// memory manager owns the whole device heap (a serving engine that reserves nearly all HBM for
// weights and KV cache up front), code on a latency-critical path where cudaMalloc's implicit
// device synchronisation would stall other streams, and systems certified to allocate nothing
// after initialisation. rdot_forward_no_alloc serves them: it runs the same forward kernels with
// the workspace placed in a fixed-size array in the library's own device memory, and
// rdot_no_alloc_read_status reads back the status word the kernels left there.
//
// The array below is a file-scope __device__ object: every GPU on which the library is loaded
// holds these RDOT_NO_ALLOC_SCRATCH_BYTES bytes until the process exits. Host code must not
// pass the symbol itself to a kernel (on the host it names a host-side shadow, not device
// memory); the device address is looked up once per device with cudaGetSymbolAddress.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>
#include <string>

#include "kernels.h"
#include "rdot.h"

namespace {

static __device__ __align__(256) unsigned char g_no_alloc_scratch[RDOT_NO_ALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the static scratch on `device` (which must be current). Set up once per
// device; returns nullptr with the CUDA error text recorded if the lookup fails.
void* scratch_address(int device) {
    if (device < 0 || device >= kMaxDevices) {
        rdot::set_last_error("rdot_forward_no_alloc: device index out of range");
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[device]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
        if (e != cudaSuccess || !p) {
            rdot::set_last_error(std::string("cudaGetSymbolAddress(static scratch): ") + cudaGetErrorString(e));
            return nullptr;
        }
        g_scratch_ptr[device] = p;
    }
    return g_scratch_ptr[device];
}

// Makes `device` current for the lifetime of the object and puts the caller's device back
// afterwards. Failures are recorded for rdot_last_cuda_error.
struct CurrentDevice {
    int prev = -1;
    bool ok = false;
    explicit CurrentDevice(int device) {
        cudaError_t e = cudaGetDevice(&prev);
        if (e == cudaSuccess && prev != device) e = cudaSetDevice(device);
        if (e != cudaSuccess) {
            rdot::set_last_error(std::string("rdot no-alloc path: selecting the plan's device: ") +
                                 cudaGetErrorString(e));
            return;
        }
        ok = true;
    }
    // Restores the caller's device; false (with the error recorded) if that failed.
    bool restore() {
        if (prev < 0) return true;
        int cur = -1;
        cudaError_t e = cudaGetDevice(&cur);
        if (e == cudaSuccess && cur != prev) e = cudaSetDevice(prev);
        prev = -1;
        if (e != cudaSuccess) {
            rdot::set_last_error(std::string("rdot no-alloc path: restoring the caller's device: ") +
                                 cudaGetErrorString(e));
            return false;
        }
        return true;
    }
    ~CurrentDevice() { (void)restore(); }
};

}  // namespace

extern "C" RDOT_API rdot_status rdot_forward_no_alloc(rdot_plan_t plan, const void* lhs, const void* rhs,
                                                      const int32_t* group_sizes, void* out, void* stream) {
    if (!plan) return RDOT_ERR_INVALID_ARG;
    size_t need = 0;
    rdot_status st = rdot_workspace_size(plan, &need);
    if (st != RDOT_OK) return st;
    if (need > RDOT_NO_ALLOC_SCRATCH_BYTES) {
        char buf[160];
        std::snprintf(buf, sizeof buf,
                      "rdot_forward_no_alloc: the plan needs %zu bytes of workspace, more than the %d-byte "
                      "static scratch",
                      need, RDOT_NO_ALLOC_SCRATCH_BYTES);
        rdot::set_last_error(buf);
        return RDOT_ERR_UNSUPPORTED;
    }
    CurrentDevice cd(rdot::plan_device(plan));
    if (!cd.ok) return RDOT_ERR_CUDA;
    void* scratch = scratch_address(rdot::plan_device(plan));
    rdot_status result = RDOT_ERR_CUDA;
    if (scratch) {
        // the previous call's status bits are cleared: this call starts from a zero status word
        cudaError_t e = cudaMemsetAsync(scratch, 0, RDOT_NO_ALLOC_SCRATCH_BYTES, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) {
            rdot::set_last_error(std::string("rdot_forward_no_alloc: ") + cudaGetErrorString(e));
        } else {
            result = rdot_forward(plan, lhs, rhs, group_sizes, out, scratch, stream);
        }
    }
    if (!cd.restore() && result == RDOT_OK) result = RDOT_ERR_CUDA;
    return result;
}

extern "C" RDOT_API rdot_status rdot_no_alloc_read_status(rdot_plan_t plan, int32_t* flags, void* stream) {
    if (!plan || !flags) return RDOT_ERR_INVALID_ARG;
    CurrentDevice cd(rdot::plan_device(plan));
    if (!cd.ok) return RDOT_ERR_CUDA;
    void* scratch = scratch_address(rdot::plan_device(plan));
    if (!scratch) return RDOT_ERR_CUDA;
    // the status word sits where rdot_read_status expects it in a workspace: read it the same way
    rdot_status st = rdot_read_status(plan, scratch, flags, stream);
    if (!cd.restore() && (st == RDOT_OK || st == RDOT_WARN_GROUP_SIZES || st == RDOT_ERR_DEVICE_TIMEOUT))
        st = RDOT_ERR_CUDA;
    return st;
}
