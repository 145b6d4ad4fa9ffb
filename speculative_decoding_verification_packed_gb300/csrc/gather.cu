// gather.cu -- row-mapped packing of wide per-row fields.
//
// "DScale: Scaling Block-Diffusion Speculative Decoding with Adaptive Verification",
// SIII-C (Flat-buffer packer: every field is packed with the same row mapping) and SIII-D
// (fixed-address workspace): rows of a wide field (query / key / value rows, logit rows)
// are copied to the packed buffer by the row ids that the packer wrote, so that every
// per-row buffer of a step shares one row map.  Rows whose id is out of range are
// zero-filled.  16-byte vector copies, grid-stride over (row, vector) pairs; the multi-field
// entry covers several fields of one row map in one launch.
#include <cstdint>
#include <cuda_runtime.h>

#include "svp_device.cuh"

namespace svp {

__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4 *__restrict__ src,
                                                          int64_t src_rows, int64_t vecs_per_row,
                                                          const int32_t *__restrict__ idx,
                                                          int32_t rows, uint4 *__restrict__ dst)
{
    griddep_launch_dependents();
    griddep_wait();
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

// All fields of one row map in one launch: grid-stride over the concatenated
// (field, row, vector) index space.
struct GatherMulti {
    const uint4 *src[SVP_GATHER_MAX_FIELDS];
    uint4 *dst[SVP_GATHER_MAX_FIELDS];
    int64_t src_rows[SVP_GATHER_MAX_FIELDS];
    int64_t vecs[SVP_GATHER_MAX_FIELDS];
    int64_t start[SVP_GATHER_MAX_FIELDS + 1];   // first index of each field
    const int32_t *idx;
    int32_t n_fields;
};

__global__ void __launch_bounds__(256) gather_rows_multi_kernel(const __grid_constant__ GatherMulti g)
{
    griddep_launch_dependents();
    griddep_wait();
    const int64_t total = g.start[g.n_fields];
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        int f = 0;
        while (f + 1 < g.n_fields && e >= g.start[f + 1])
            ++f;
        const int64_t l = e - g.start[f];
        const int64_t r = l / g.vecs[f], v = l - r * g.vecs[f];
        const int32_t s = __ldg(g.idx + r);
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (s >= 0 && s < g.src_rows[f])
            x = __ldg(g.src[f] + s * g.vecs[f] + v);
        g.dst[f][l] = x;
    }
}

static svp_status gather_grid(int64_t total, int64_t &grid)
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SVP_ECUDA;
    grid = (total + 255) / 256;
    if (grid > (int64_t)sms * 16)
        grid = (int64_t)sms * 16;
    return SVP_OK;
}

}  // namespace svp

extern "C" svp_status svp_gather_rows_multi(const svp_gather_field *fields, int32_t n_fields,
                                            const int32_t *idx, int32_t rows, void *stream)
{
    using namespace svp;
    if (!fields || !idx || n_fields < 1 || n_fields > SVP_GATHER_MAX_FIELDS || rows < 0)
        return SVP_EINVAL;
    GatherMulti g = {};
    g.idx = idx;
    g.n_fields = n_fields;
    g.start[0] = 0;
    for (int f = 0; f < n_fields; ++f) {
        const svp_gather_field &x = fields[f];
        if (!x.src || !x.dst || x.src_rows < 0 || x.row_bytes < 16)
            return SVP_EINVAL;
        if ((x.row_bytes & 15) || (reinterpret_cast<uintptr_t>(x.src) & 15) ||
            (reinterpret_cast<uintptr_t>(x.dst) & 15))
            return SVP_EUNSUPPORTED;
        g.src[f] = static_cast<const uint4 *>(x.src);
        g.dst[f] = static_cast<uint4 *>(x.dst);
        g.src_rows[f] = x.src_rows;
        g.vecs[f] = x.row_bytes / 16;
        g.start[f + 1] = g.start[f] + (int64_t)rows * g.vecs[f];
    }
    if (rows == 0)
        return SVP_OK;
    int64_t grid = 0;
    const svp_status st = gather_grid(g.start[n_fields], grid);
    if (st != SVP_OK)
        return st;
    return launch_pdl(gather_rows_multi_kernel, dim3((unsigned)grid), dim3(256), 0, (cudaStream_t)stream, g) ==
                   cudaSuccess
               ? SVP_OK
               : SVP_ECUDA;
}

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
    const int64_t vecs = row_bytes / 16, total = (int64_t)rows * vecs;
    int64_t grid = 0;
    const svp_status st = gather_grid(total, grid);
    if (st != SVP_OK)
        return st;
    return launch_pdl(gather_rows_kernel, dim3((unsigned)grid), dim3(256), 0, (cudaStream_t)stream,
                      static_cast<const uint4 *>(src), src_rows, vecs, idx, rows,
                      static_cast<uint4 *>(dst)) == cudaSuccess
               ? SVP_OK
               : SVP_ECUDA;
}
