// gather.cu -- row-mapped packing of wide per-row fields.
//
// "DScale: Scaling Block-Diffusion Speculative Decoding with Adaptive Verification",
// SIII-C (Flat-buffer packer: every field is packed with the same row mapping) and SIII-D
// (fixed-address workspace): rows of a wide field (query / key / value rows, logit rows)
// are copied to the packed buffer by the row ids that the packer wrote, so that every
// per-row buffer of a step shares one row map.  Rows whose id is out of range are
// zero-filled.  16-byte vector copies, grid-stride over (row, vector) pairs.
#include <cstdint>
#include <cuda_runtime.h>

#include "svp_device.cuh"

namespace svp {

__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4 *__restrict__ src,
                                                          int64_t src_rows, int64_t vecs_per_row,
                                                          const int32_t *__restrict__ idx,
                                                          int32_t rows, uint4 *__restrict__ dst)
{
    const int64_t total = (int64_t)rows * vecs_per_row;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = e / vecs_per_row, v = e - r * vecs_per_row;
        const int32_t s = __ldg(idx + r);
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (s >= 0 && s < src_rows)
            x = __ldg(src + (int64_t)s * vecs_per_row + v);
        dst[e] = x;
    }
}

}  // namespace svp

extern "C" svp_status svp_gather_rows(const void *src, int64_t src_rows, int64_t row_bytes,
                                      const int32_t *idx, int32_t rows, void *dst, void *stream)
{
    using namespace svp;
    if (!src || !idx || !dst || src_rows < 0 || row_bytes < 16 || rows < 0)
        return SVP_EINVAL;
    if ((row_bytes & 15) || (reinterpret_cast<uintptr_t>(src) & 15) ||
        (reinterpret_cast<uintptr_t>(dst) & 15))
        return SVP_EUNSUPPORTED;
    if (rows == 0)
        return SVP_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SVP_ECUDA;
    const int64_t vecs = row_bytes / 16, total = (int64_t)rows * vecs;
    int64_t grid = (total + 255) / 256;
    if (grid > (int64_t)sms * 16)
        grid = (int64_t)sms * 16;
    gather_rows_kernel<<<(unsigned)grid, 256, 0, (cudaStream_t)stream>>>(
        static_cast<const uint4 *>(src), src_rows, vecs, idx, rows, static_cast<uint4 *>(dst));
    return cudaGetLastError() == cudaSuccess ? SVP_OK : SVP_ECUDA;
}
