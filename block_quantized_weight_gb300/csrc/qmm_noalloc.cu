// qmm_noalloc.cu -- the small-M tensor-core product with its split-K scratch in
// a fixed, statically sized device array, for callers that cannot hand the
// library a workspace.
//
// Some callers own no device allocator at the point of the call: a decode
// engine that carves all of HBM into weights and KV cache at start-up and
// forbids allocation afterwards, a host program written against the plain C
// ABI with no memory pool of its own, or a loop where a cudaMalloc (which can
// synchronize the whole device) would stall the pipeline.  For them this entry
// point takes no workspace argument and allocates nothing: the scratch is one
// module-level array, located on the current device with cudaGetSymbolAddress.
//
// The arithmetic, the split-K plan and the kernel are exactly those of
// qmm_q4_0_smallM: this file only supplies the scratch and forwards the call.

#include <cuda_runtime.h>

#include <mutex>

#include "qbw.h"
#include "qbw_internal.h"

namespace {

constexpr size_t kScratchBytes = QBW_QMM_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Split-K partial sums followed by one arrival counter per 128-row tile.  Only
// the counters must be zero before a call; every completed call leaves them
// zero again.  The array is zero-filled explicitly on first use per device.
static __device__ __align__(256) unsigned char g_qmm_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};
bool g_scratch_dirty[kMaxDevices] = {};

// The array's address on the current device, looked up on every call (cheap;
// a device reset or a new context moves it).  When the address is new, or a
// fault was reported since the last call (a call that gave up may have left
// counters nonzero), the array is zero-filled on the caller's stream first,
// so the kernel that follows sees zero counters.
qbw_status scratch_for_current_device(cudaStream_t s, void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QBW_ECUDA;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_qmm_scratch) != cudaSuccess || !addr) return QBW_ECUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_addr[dev] != addr || g_scratch_dirty[dev]) {
        if (cudaMemsetAsync(addr, 0, kScratchBytes, s) != cudaSuccess) return QBW_ECUDA;
        g_scratch_addr[dev] = addr;
        g_scratch_dirty[dev] = false;
    }
    *out = addr;
    return QBW_OK;
}

}  // namespace

namespace qbw {

void noalloc_scratch_mark_dirty(int device) {
    if (device < 0 || device >= kMaxDevices) return;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    g_scratch_dirty[device] = true;
}

}  // namespace qbw

extern "C" {

qbw_status qmm_q4_0_smallM_noalloc(const void* w, const void* X, qbw_dtype xt, void* Y, qbw_dtype yt, int64_t M,
                                   int64_t N, int64_t K, void* stream) {
    // A shape that needs no scratch (one split, or the CUDA-core path) goes
    // straight through; qmm_q4_0_smallM validates every argument.
    const size_t need = qmm_q4_0_smallM_workspace_bytes(M, N, K);
    if (need == 0) return qmm_q4_0_smallM(w, X, xt, Y, yt, M, N, K, nullptr, 0, stream);
    if (need > kScratchBytes) return QBW_EWORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* scratch = nullptr;
    qbw_status st = scratch_for_current_device(s, &scratch);
    if (st != QBW_OK) return st;
    return qmm_q4_0_smallM(w, X, xt, Y, yt, M, N, K, scratch, kScratchBytes, stream);
}

}  // extern "C"
