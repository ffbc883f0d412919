// noalloc.cu -- ssm_scan_fwd_lookback_static: the look-back scan with its scratch
// in a fixed device array that the library owns, for callers that cannot
// allocate device memory (see include/ssm_scan.h for who and why).
//
// The look-back scan needs scratch beyond its inputs and outputs: a status word,
// a ticket counter and one published descriptor per (channel, time segment).
// Here that scratch is g_scratch, a file-scope __device__ array of
// SSM_STATIC_SCRATCH_BYTES. Every device that loads this library holds it until
// the process exits, and all calls on a device share it.
//
// In host code the name g_scratch is only a host-side stand-in for the array,
// not a device address: passing it to a kernel would fault (or, where the GPU can
// reach host memory, silently use the wrong memory). The device address is looked
// up once per device with cudaGetSymbolAddress, with that device current, on the
// first call made on it, and reused afterwards.
#include <mutex>

#include "launch.h"
#include "ssm_scan.h"

namespace {

constexpr size_t kScratchBytes = SSM_STATIC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_dev[kMaxDevices];   // device address of g_scratch per device (set on first use)

// Device address of g_scratch on the current device (looked up on first use).
int scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSM_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_dev[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return SSM_ERR_LAUNCH;
        g_scratch_dev[dev] = p;
    }
    *out = g_scratch_dev[dev];
    return SSM_OK;
}

}  // namespace

extern "C" int ssm_scan_fwd_lookback_static(const void* u, const void* delta, const float* A,
                                            const void* B, const void* C, const float* D,
                                            const void* z, const float* delta_bias, int softplus,
                                            const float* h0, void* y, float* h_last,
                                            int64_t batch, int64_t dim, int64_t seqlen,
                                            int64_t dstate, int in_dtype, int out_dtype,
                                            void* stream) {
    // the look-back's scratch for these sizes (status word, ticket, descriptors);
    // invalid sizes report 16 here and are rejected below by the scan's own checks
    if (ssm_scan_workspace_size(batch, dim, seqlen, dstate) > kScratchBytes) return SSM_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != SSM_OK) return st;
    // validates the arguments, zeroes the part of the scratch the scan uses (on
    // `stream`) and launches the look-back scan on `stream`
    return ssm_scan_fwd_algo(u, delta, A, B, C, D, z, delta_bias, softplus, h0, y, h_last, batch, dim,
                             seqlen, dstate, in_dtype, out_dtype, scratch, kScratchBytes,
                             SSM_ALGO_LOOKBACK, stream);
}
