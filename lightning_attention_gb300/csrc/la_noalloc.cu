// la_noalloc.cu -- la_extend_noalloc: the extend entry point for callers that cannot allocate
// device memory.
//
// la_extend splits long requests of small batches into segments, plans skewed batches on the
// device and keeps request records for large ones, and needs scratch memory for it, which the
// caller passes in (la_extend_workspace_size says how much).  Some callers have no way to
// obtain that buffer at the point where they run the extend step: a plugin inside a host framework
// that owns the device's whole memory budget and hands the plugin nothing but its input and output
// tensors, or a latency-critical loop in which cudaMalloc (with the implicit synchronisation it can
// bring) is not acceptable.  For them this file keeps the scratch in a fixed, module-scope device
// array instead.
//
// Facts a caller needs:
//   * The array is kNoAllocScratchBytes (16 MiB) on every device that loads this library, held
//     until the process exits.  The split planner asks for at most 1.5 x (number of SMs) fp32
//     128 x 128 matrices of 64 KiB (one request whose head count is half the SM count), i.e.
//     14.25 MiB on a 152-SM GB300, so every plan fits on any device of up to 170 SMs.  A plan
//     that needs more is rejected with LA_ERR_UNSUPPORTED and nothing is launched.
//   * The first call on a device looks the array's device address up (cudaGetSymbolAddress, with
//     that device current) and caches it; make that first call before any stream capture.  The
//     cached address belongs to the device's current context: after cudaDeviceReset the module is
//     loaded anew, so do not call this entry point again in that process.
//   * Every call on a device shares the one array, and it keeps the last call's contents.  Nothing
//     in it has to start at zero: each call writes every value it later reads (the initial-state
//     copy and the block states, the records, the balanced plan and its read counters) before
//     reading it.  Calls that overlap on the GPU (for example on
//     two streams at once) race on the array and give wrong results; serialise them.
//   * The entry point calls no cudaMalloc, cudaFree or other allocating routine.
#include <mutex>

#include "la.h"
#include "la_internal.h"

#define LA_NOALLOC_SCRATCH_BYTES (size_t(16) << 20)

// The scratch itself: file scope, device memory, 256-byte aligned.  Host code must not pass
// `g_noalloc_scratch` to a kernel (on the host it only names a stand-in); it passes the device
// address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr size_t kNoAllocScratchBytes = LA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once per device.
la_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return LA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return LA_OK;
}

}  // namespace

extern "C" la_status la_extend_noalloc(const la_bf16 *q, const la_bf16 *k, const la_bf16 *v,
                                       const float *slopes, float *state_pool, int num_slots,
                                       const int32_t *state_idx, const int32_t *cu_seqlens,
                                       const uint8_t *prefix_mask, la_bf16 *out, int B, int T,
                                       int H, int D, int max_seqlen, la_stream stream) {
    size_t need = 0;
    la_status st = la_extend_workspace_size(B, T, H, D, max_seqlen, &need);
    if (st != LA_OK) return st;
    if (need > kNoAllocScratchBytes) return LA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (need > 0 && (st = scratch_address(&scratch)) != LA_OK) return st;
    return la_extend(q, k, v, slopes, state_pool, num_slots, state_idx, cu_seqlens, prefix_mask,
                     out, B, T, H, D, max_seqlen, scratch, need > 0 ? kNoAllocScratchBytes : 0,
                     stream);
}
