// attn_simt.cu -- fp32 verification attention on CUDA cores (FFMA, fp32 accumulate).
//
// Same definition as the tensor-core path (DScale SIII-D: row j of request i attends to
// the request's context and then to its own candidates 0..j; query head h reads KV head
// h / G), for fp32 inputs, where tf32 tensor cores would miss a 1e-4 bound.
//
// One CTA of 128 threads per (packed candidate row, query head).  Keys stream in tiles
// of 128: each thread scores one key against the query row held in shared memory, the
// tile maximum / sum update the running softmax state, and each thread accumulates
// d / 128 output columns from coalesced value-row reads.
#include <cfloat>

#include "svp_params.cuh"

namespace svp {

constexpr int kSimtThreads = 128;

__device__ __forceinline__ const float *ctx_row(const SimtParams &p, int32_t i, int32_t g,
                                                int32_t t, const float *base, bool &ok)
{
    ok = true;
    if (!p.paged)
        return base + ((__ldg(p.cu_ctx + i) + t) * (int64_t)p.hkv + g) * p.d;
    const int32_t page = __ldg(p.block_table + (int64_t)i * p.max_pages + t / 16);
    if (page < 0 || page >= p.num_pages) {
        ok = false;
        return base;
    }
    return base + page * p.s_page + g * p.s_head + (t % 16) * p.s_tok;
}

__global__ void __launch_bounds__(kSimtThreads) attn_simt_kernel(SimtParams p)
{
    __shared__ float qs[256];
    __shared__ float ps[kSimtThreads];
    __shared__ float red[kSimtThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t i = blockIdx.x / p.w;
    const int32_t j = blockIdx.x % p.w;
    const int32_t h = blockIdx.y;
    const int32_t off = __ldg(p.cu_slots + i);
    const int32_t end = __ldg(p.cu_slots + i + 1);
    if (off < 0 || end < off || end - off > p.w || end > p.m_cap) {
        if (tid == 0 && j == 0 && h == 0)
            set_status(p.status, SVP_DEV_BAD_SLOTS);
        return;
    }
    if (j >= end - off)
        return;
    const int32_t L = p.ctx_len ? __ldg(p.ctx_len + i) : 0;
    bool ctx_ok = L >= 0;
    if (ctx_ok && L > 0) {
        if (p.paged)
            ctx_ok = (L + 15) / 16 <= p.max_pages;
        else
            ctx_ok = __ldg(p.cu_ctx + i) >= 0 && __ldg(p.cu_ctx + i) + L <= p.total_tokens;
    }
    if (!ctx_ok) {
        if (tid == 0 && j == 0 && h == 0)
            set_status(p.status, SVP_DEV_BAD_CONTEXT);
        return;
    }
    const int32_t G = p.hq / p.hkv, g = h / G;
    const int32_t D = p.d;
    const int64_t qrow = ((int64_t)(off + j) * p.hq + h) * D;
    for (int e = tid; e < D; e += kSimtThreads)
        qs[e] = p.q[qrow + e];
    __syncthreads();

    const int32_t nkeys = L + j + 1;
    float m_run = -INFINITY, l_run = 0.0f;
    float acc0 = 0.0f, acc1 = 0.0f;           // columns tid and tid + 128
    bool bad_page = false;
    for (int32_t t0 = 0; t0 < nkeys; t0 += kSimtThreads) {
        const int32_t t = t0 + tid;
        float s = -INFINITY;
        if (t < nkeys) {
            const float *kr;
            bool ok = true;
            if (t < L)
                kr = ctx_row(p, i, g, t, p.k, ok);
            else
                kr = p.k_new + ((int64_t)(off + t - L) * p.hkv + g) * D;
            if (ok) {
                float dot = 0.0f;
                for (int e = 0; e < D; ++e)
                    dot = fmaf(qs[e], __ldg(kr + e), dot);
                s = dot * p.scale;
            } else {
                bad_page = true;
            }
        }
        // tile maximum
        float mt = s;
        for (int o = 16; o > 0; o >>= 1)
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
        if (lane == 0)
            red[warp] = mt;
        __syncthreads();
        mt = red[0];
        for (int w2 = 1; w2 < kSimtThreads / 32; ++w2)
            mt = fmaxf(mt, red[w2]);
        __syncthreads();
        const float m_new = fmaxf(m_run, mt);
        const float alpha = (m_run == -INFINITY) ? 0.0f : expf(m_run - m_new);
        const float pk = (s == -INFINITY) ? 0.0f : expf(s - m_new);
        ps[tid] = pk;
        float sum = pk;
        for (int o = 16; o > 0; o >>= 1)
            sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0)
            red[warp] = sum;
        __syncthreads();
        float tsum = 0.0f;
        for (int w2 = 0; w2 < kSimtThreads / 32; ++w2)
            tsum += red[w2];
        l_run = l_run * alpha + tsum;
        m_run = m_new;
        acc0 *= alpha;
        acc1 *= alpha;
        const int32_t cnt = min(kSimtThreads, nkeys - t0);
        for (int32_t kk = 0; kk < cnt; ++kk) {
            const int32_t tt = t0 + kk;
            const float *vr;
            bool ok = true;
            if (tt < L)
                vr = ctx_row(p, i, g, tt, p.v, ok);
            else
                vr = p.v_new + ((int64_t)(off + tt - L) * p.hkv + g) * D;
            if (!ok)
                continue;
            const float pw = ps[kk];
            if (tid < D)
                acc0 = fmaf(pw, __ldg(vr + tid), acc0);
            if (tid + kSimtThreads < D)
                acc1 = fmaf(pw, __ldg(vr + tid + kSimtThreads), acc1);
        }
        __syncthreads();
    }
    if (bad_page)
        set_status(p.status, SVP_DEV_BAD_CONTEXT);
    const float inv = 1.0f / l_run;
    if (tid < D)
        p.out[qrow + tid] = acc0 * inv;
    if (tid + kSimtThreads < D)
        p.out[qrow + tid + kSimtThreads] = acc1 * inv;
    if (tid == 0 && p.lse)
        p.lse[(int64_t)(off + j) * p.hq + h] = m_run + logf(l_run);
}

svp_status attn_simt_launch(const SimtParams &p, cudaStream_t stream)
{
    if (p.n == 0)
        return SVP_OK;
    dim3 grid((unsigned)(p.n * p.w), (unsigned)p.hq);
    attn_simt_kernel<<<grid, kSimtThreads, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? SVP_OK : SVP_ECUDA;
}

}  // namespace svp
