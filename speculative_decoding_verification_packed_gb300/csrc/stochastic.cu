// stochastic.cu -- stochastic prefix verifier (temperature > 0).
//
// "DScale: Scaling Block-Diffusion Speculative Decoding with Adaptive Verification", SIII-D
// (Prefix verifier): P_r = softmax(z_r / T) of packed target-logit row r; the deterministic
// draft candidate x_j = tokens[off_i + j] is accepted with probability P_{off_i+j-1}(x_j)
// (u_accept[off_i + j] < P), in order, until the first rejection; the successor is drawn
// from P_{off_i+a} with the rejected candidate removed and the rest renormalised, or from
// the unmodified P_{off_i+k_i-1} when every candidate passes.  accept_len = 1 + a,
// next_token = the successor (inverse-CDF draw with u_next[i] in token order).
//
// Two launches: (1) per-row softmax statistics (max, sum of 2^((z - max) log2(e) / T)) over
// (row, chunk) units with a per-row ticket merge, HBM-bound over the live logit rows;
// (2) one block per request: the acceptance chain from the row statistics, then the
// successor draw over one row (block prefix sum of per-thread chunk weights).
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "svp_device.cuh"

namespace svp {

constexpr int kStChunk = 8192;          // vocabulary elements per (row, chunk) unit
constexpr int kStThreads1 = 256;
constexpr int kStThreads2 = 512;

struct StParams {
    const void *logits;
    int64_t row_stride;
    int32_t m_cap, vocab, dtype, n, chunks;
    float c;                            // log2(e) / T
    const int32_t *tokens, *cu_slots;
    const float *u_accept, *u_next;
    int32_t *accept_len, *next_token;
    float *p_draft;
    int32_t *status;
    float2 *row_stat;                   // [m_cap]: (max, sum of 2^((z - max) c))
    int32_t *tickets;                   // [m_cap]
    float2 *partial;                    // [m_cap * chunks]
};

template <int DT>
__device__ __forceinline__ float st_load(const void *base, int64_t idx)
{
    if (DT == 1) {
        const uint16_t b = __ldg(reinterpret_cast<const uint16_t *>(base) + idx);
        return __uint_as_float((uint32_t)b << 16);
    }
    return __ldg(reinterpret_cast<const float *>(base) + idx);
}

// Merge (m, s) pairs: s is relative to its own max.
__device__ __forceinline__ float2 st_merge(float2 a, float2 b, float c)
{
    if (a.x < b.x) {
        const float2 t = a;
        a = b;
        b = t;
    }
    if (b.x == -INFINITY)
        return a;
    return make_float2(a.x, a.y + b.y * exp2f((b.x - a.x) * c));
}

template <int DT>
__global__ void __launch_bounds__(kStThreads1) st_rowstat_kernel(const StParams p)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp_g = ((int64_t)blockIdx.x * kStThreads1 + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kStThreads1) >> 5;
    int32_t live = __ldg(p.cu_slots + p.n);
    live = live < 0 ? 0 : (live > p.m_cap ? p.m_cap : live);
    const int64_t units = (int64_t)live * p.chunks;
    for (int64_t u = warp_g; u < units; u += nwarps) {
        const int32_t r = (int32_t)(u / p.chunks), ch = (int32_t)(u - (int64_t)r * p.chunks);
        const int64_t lo = (int64_t)ch * kStChunk;
        const int64_t hi = lo + kStChunk < p.vocab ? lo + kStChunk : p.vocab;
        const int64_t rowb = (int64_t)r * p.row_stride;
        float m = -INFINITY, s = 0.0f;
        // one 16-byte vector per lane per step when the rows are aligned: rescale once to
        // the vector maximum, then one ex2 per value
        constexpr int VEC = DT == 1 ? 8 : 4;
        int64_t e0 = lo;
        if (((p.row_stride * (DT == 1 ? 2 : 4)) & 15) == 0 &&
            (reinterpret_cast<uintptr_t>(p.logits) & 15) == 0) {
            const int64_t nv = (hi - lo) / VEC;
            const uint4 *src = reinterpret_cast<const uint4 *>(
                static_cast<const uint8_t *>(p.logits) + (rowb + lo) * (DT == 1 ? 2 : 4));
            for (int64_t v0 = lane; v0 < nv; v0 += 64) {
                uint4 x[2];
#pragma unroll
                for (int q = 0; q < 2; ++q)
                    if (v0 + q * 32 < nv)
                        x[q] = __ldg(src + v0 + q * 32);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    if (v0 + q * 32 >= nv)
                        continue;
                    const uint32_t w[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
                    float f[VEC];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        if (DT == 1) {
                            f[2 * h] = __uint_as_float(w[h] << 16);
                            f[2 * h + 1] = __uint_as_float(w[h] & 0xffff0000u);
                        } else {
                            f[h] = __uint_as_float(w[h]);
                        }
                    }
                    float vmax = f[0];
#pragma unroll
                    for (int h = 1; h < VEC; ++h)
                        vmax = fmaxf(vmax, f[h]);
                    if (vmax > m) {
                        s = m == -INFINITY ? 0.0f : s * fast_exp2((m - vmax) * p.c);
                        m = vmax;
                    }
                    if (m != -INFINITY) {
#pragma unroll
                        for (int h = 0; h < VEC; ++h)
                            s += fast_exp2((f[h] - m) * p.c);
                    }
                }
            }
            e0 = lo + nv * VEC;
        }
        for (int64_t e = e0 + lane; e < hi; e += 32) {
            const float v = st_load<DT>(p.logits, rowb + e);
            if (v > m) {
                s = s * exp2f((m - v) * p.c) + 1.0f;
                m = v;
            } else {
                s += exp2f((v - m) * p.c);
            }
        }
        float2 a = make_float2(m, m == -INFINITY ? 0.0f : s);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float2 b;
            b.x = __shfl_xor_sync(0xffffffffu, a.x, o);
            b.y = __shfl_xor_sync(0xffffffffu, a.y, o);
            a = st_merge(a, b, p.c);
        }
        if (p.chunks == 1) {
            if (lane == 0)
                p.row_stat[r] = a;
            continue;
        }
        int last = 0;
        if (lane == 0) {
            p.partial[u] = a;
            __threadfence();
            last = atomicAdd(p.tickets + r, 1) == p.chunks - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence();
            float2 t = make_float2(-INFINITY, 0.0f);
            for (int q = lane; q < p.chunks; q += 32)
                t = st_merge(t, __ldcg(p.partial + (int64_t)r * p.chunks + q), p.c);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                float2 b;
                b.x = __shfl_xor_sync(0xffffffffu, t.x, o);
                b.y = __shfl_xor_sync(0xffffffffu, t.y, o);
                t = st_merge(t, b, p.c);
            }
            if (lane == 0) {
                p.row_stat[r] = t;
                p.tickets[r] = 0;
            }
        }
    }
}

template <int DT>
__global__ void __launch_bounds__(kStThreads2) st_accept_kernel(const StParams p)
{
    __shared__ float sh_sum[kStThreads2 / 32];
    __shared__ float sh_total;
    __shared__ int32_t sh_row, sh_excl, sh_claim;
    const int i = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t off = __ldg(p.cu_slots + i), end = __ldg(p.cu_slots + i + 1);
    const int32_t live = __ldg(p.cu_slots + p.n);
    if (off < 0 || end < off || end > p.m_cap || live > p.m_cap) {
        if (tid == 0) {
            set_status(p.status, SVP_DEV_BAD_SLOTS);
            p.accept_len[i] = 0;
            p.next_token[i] = -1;
        }
        return;
    }
    const int32_t k = end - off;
    if (k == 0) {
        if (tid == 0) {
            p.accept_len[i] = 0;
            p.next_token[i] = -1;
        }
        return;
    }
    if (tid == 0) {
        // acceptance chain: candidate j against row off + j - 1
        int32_t a = 0, excl = -1;
        for (int32_t j = 1; j < k; ++j) {
            const int32_t r = off + j - 1;
            const int32_t x = __ldg(p.tokens + off + j);
            const float2 st = p.row_stat[r];
            float pr = 0.0f;
            if (x >= 0 && x < p.vocab)
                pr = exp2f((st_load<DT>(p.logits, (int64_t)r * p.row_stride + x) - st.x) * p.c) / st.y;
            if (p.p_draft)
                p.p_draft[off + j] = pr;
            if (__ldg(p.u_accept + off + j) < pr) {
                ++a;
            } else {
                excl = x;
                break;
            }
        }
        p.accept_len[i] = 1 + a;
        sh_row = off + a;
        sh_excl = excl;
        sh_claim = kStThreads2;
    }
    __syncthreads();
    // successor: inverse-CDF draw over row sh_row without token sh_excl, in token order
    const int32_t r = sh_row, excl = sh_excl;
    const float m = p.row_stat[r].x;
    const int64_t rowb = (int64_t)r * p.row_stride;
    const int64_t per = ((int64_t)p.vocab + kStThreads2 - 1) / kStThreads2;
    const int64_t lo = (int64_t)tid * per;
    const int64_t hi = lo + per < p.vocab ? lo + per : p.vocab;
    float own = 0.0f;
    for (int64_t e = lo; e < hi; ++e)
        if (e != excl)
            own += exp2f((st_load<DT>(p.logits, rowb + e) - m) * p.c);
    // block exclusive scan of the chunk weights
    float incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        sh_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        float t = lane < kStThreads2 / 32 ? sh_sum[lane] : 0.0f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o)
                t += y;
        }
        if (lane < kStThreads2 / 32)
            sh_sum[lane] = t;
        if (lane == kStThreads2 / 32 - 1)
            sh_total = t;
    }
    __syncthreads();
    const float before = (warp > 0 ? sh_sum[warp - 1] : 0.0f) + incl - own;
    const float target = __ldg(p.u_next + i) * sh_total;
    // the lowest chunk whose interval [before, before + own) holds the target (rounding
    // may let two intervals touch it; the lower one is the smaller token)
    const bool mine = own > 0.0f && before <= target &&
                      (target < before + own || before + own >= sh_total);
    if (mine)
        atomicMin(&sh_claim, tid);
    __syncthreads();
    if (tid == sh_claim) {
        float cum = before;
        int32_t y = -1, last_nz = -1;
        for (int64_t e = lo; e < hi; ++e) {
            if (e == excl)
                continue;
            const float w = exp2f((st_load<DT>(p.logits, rowb + e) - m) * p.c);
            if (w > 0.0f)
                last_nz = (int32_t)e;
            cum += w;
            if (cum > target && w > 0.0f) {
                y = (int32_t)e;
                break;
            }
        }
        p.next_token[i] = y >= 0 ? y : last_nz;
    }
    if (tid == 0 && sh_claim == kStThreads2) {
        // rounding left the target past every chunk: the last token with weight
        int32_t y = -1;
        for (int64_t e = p.vocab - 1; e >= 0 && y < 0; --e)
            if (e != excl && exp2f((st_load<DT>(p.logits, rowb + e) - m) * p.c) > 0.0f)
                y = (int32_t)e;
        p.next_token[i] = y;
    }
}

static void st_plan(int32_t m_cap, int32_t vocab, int32_t &chunks, size_t &off_stat,
                    size_t &off_tk, size_t &off_part, size_t &bytes)
{
    chunks = (vocab + kStChunk - 1) / kStChunk;
    off_stat = kWsHeader;
    off_tk = off_stat + (size_t)m_cap * sizeof(float2);
    off_part = (off_tk + (size_t)m_cap * 4 + 255) / 256 * 256;
    bytes = off_part + (size_t)m_cap * chunks * sizeof(float2);
}

}  // namespace svp

extern "C" svp_status svp_stochastic_accept_workspace_size(int32_t m_cap, int32_t vocab,
                                                           size_t *bytes)
{
    using namespace svp;
    if (!bytes || m_cap < 0 || vocab < 2)
        return SVP_EINVAL;
    int32_t chunks;
    size_t a, b, c;
    st_plan(m_cap, vocab, chunks, a, b, c, *bytes);
    return SVP_OK;
}

extern "C" svp_status svp_stochastic_accept(const void *logits, int64_t row_stride,
                                            int32_t m_cap, int32_t vocab, svp_dtype dtype,
                                            const int32_t *tokens, const int32_t *cu_slots,
                                            int32_t n, float temperature,
                                            const float *u_accept, const float *u_next,
                                            int32_t *accept_len, int32_t *next_token,
                                            float *p_draft, void *ws, size_t ws_bytes,
                                            void *stream)
{
    using namespace svp;
    if (!logits || !tokens || !cu_slots || !u_accept || !u_next || !accept_len ||
        !next_token || !ws || n < 0 || m_cap < 0 || vocab < 2 || row_stride < vocab ||
        !(temperature > 0.0f))
        return SVP_EINVAL;
    if (dtype != SVP_BF16 && dtype != SVP_F32)
        return SVP_EUNSUPPORTED;
    StParams p;
    size_t off_stat, off_tk, off_part, need;
    st_plan(m_cap, vocab, p.chunks, off_stat, off_tk, off_part, need);
    if (ws_bytes < need)
        return SVP_EWORKSPACE;
    if (n == 0)
        return SVP_OK;
    uint8_t *w = static_cast<uint8_t *>(ws);
    p.logits = logits;
    p.row_stride = row_stride;
    p.m_cap = m_cap;
    p.vocab = vocab;
    p.dtype = dtype;
    p.n = n;
    p.c = 1.4426950408889634f / temperature;
    p.tokens = tokens;
    p.cu_slots = cu_slots;
    p.u_accept = u_accept;
    p.u_next = u_next;
    p.accept_len = accept_len;
    p.next_token = next_token;
    p.p_draft = p_draft;
    p.status = reinterpret_cast<int32_t *>(w);
    p.row_stat = reinterpret_cast<float2 *>(w + off_stat);
    p.tickets = reinterpret_cast<int32_t *>(w + off_tk);
    p.partial = reinterpret_cast<float2 *>(w + off_part);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SVP_ECUDA;
    const int64_t units = (int64_t)m_cap * p.chunks;
    int64_t grid1 = (units + (kStThreads1 / 32) - 1) / (kStThreads1 / 32);
    if (grid1 > (int64_t)sms * 8)
        grid1 = (int64_t)sms * 8;
    if (grid1 < 1)
        grid1 = 1;
    cudaStream_t s = (cudaStream_t)stream;
    if (dtype == SVP_BF16) {
        st_rowstat_kernel<1><<<(unsigned)grid1, kStThreads1, 0, s>>>(p);
        st_accept_kernel<1><<<n, kStThreads2, 0, s>>>(p);
    } else {
        st_rowstat_kernel<0><<<(unsigned)grid1, kStThreads1, 0, s>>>(p);
        st_accept_kernel<0><<<n, kStThreads2, 0, s>>>(p);
    }
    return cudaGetLastError() == cudaSuccess ? SVP_OK : SVP_ECUDA;
}
