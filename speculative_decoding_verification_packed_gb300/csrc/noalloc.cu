// noalloc.cu -- svp_margin_accept_noalloc: the fused row-margin + greedy-accept step
// for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hold a workspace of their own: code that runs
// inside a memory pool whose owner forbids foreign allocations, plug-ins loaded into a
// host process that manages all device memory itself, or latency-critical paths where an
// allocation (and the implicit synchronisation it can cause) is not acceptable.  For
// them this entry point runs the same kernel as svp_margin_accept, with its scratch in a
// fixed array that the library owns.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes bytes.  Every GPU
// that loads the library holds it until the process exits.  Host code cannot use the
// array's name as a device address, so on the first call on each device (with that
// device current) the library asks the runtime for the array's device address with
// cudaGetSymbolAddress, checks the result, and clears the array once: a cudaMemsetAsync on
// the caller's stream, then a wait for that stream, so the clear is complete before any
// kernel on any stream uses the array (neither call allocates).  After that the kernel
// leaves the scratch all zero at the end of every call, as the fused kernel always does
// with its workspace.
#include <mutex>

#include "svp_device.cuh"

namespace svp {

svp_status margin_workspace(int32_t rows, int32_t vocab, int32_t n, size_t *bytes);
svp_status margin_launch(const void *logits, int64_t row_stride, int32_t rows, int32_t vocab,
                         svp_dtype dtype, int32_t *top1_idx, float *top1, float *top2,
                         float *margin, const int32_t *tokens, const int32_t *cu_slots,
                         int32_t n, int32_t *accept_len, int32_t *next_token, void *ws,
                         size_t ws_bytes, cudaStream_t stream);

// 2 MiB: e.g. 4096 rows of a 262144-entry vocabulary with 4096 requests fit.
constexpr size_t kNoAllocScratchBytes = 2u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {nullptr};
}  // namespace

// Device address of this device's scratch, set up on first use (nullptr on failure).  The
// first use clears the array on `stream` and waits for it before the address is handed
// out, so a first call made on a non-blocking stream cannot race the clear.
static void *noalloc_scratch_for_current_device(cudaStream_t stream, svp_status *err)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = SVP_ECUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
            *err = SVP_ECUDA;
            return nullptr;
        }
        if (cudaMemsetAsync(ptr, 0, kNoAllocScratchBytes, stream) != cudaSuccess ||
            cudaStreamSynchronize(stream) != cudaSuccess) {
            *err = SVP_ECUDA;
            return nullptr;
        }
        g_scratch_addr[dev] = ptr;
    }
    return g_scratch_addr[dev];
}

}  // namespace svp

extern "C" svp_status svp_margin_accept_noalloc(const void *logits, int64_t row_stride,
                                                int32_t m_cap, int32_t vocab, svp_dtype dtype,
                                                const int32_t *tokens, const int32_t *cu_slots,
                                                int32_t n, int32_t *top1_idx, float *top1,
                                                float *top2, float *margin,
                                                int32_t *accept_len, int32_t *next_token,
                                                void *stream)
{
    using namespace svp;
    if (!cu_slots)
        return SVP_EINVAL;
    size_t need = 0;
    const svp_status st = margin_workspace(m_cap, vocab, n, &need);
    if (st != SVP_OK)
        return st;
    if (need > kNoAllocScratchBytes)
        return SVP_EWORKSPACE;   // sizes beyond the fixed scratch: use svp_margin_accept
    svp_status err = SVP_OK;
    void *scratch = noalloc_scratch_for_current_device((cudaStream_t)stream, &err);
    if (!scratch)
        return err;
    return margin_launch(logits, row_stride, m_cap, vocab, dtype, top1_idx, top1, top2, margin,
                         tokens, cu_slots, n, accept_len, next_token, scratch,
                         kNoAllocScratchBytes, (cudaStream_t)stream);
}
