// features.cu -- draft-signal features per draft-logit row, and ACT truncation.
//
// "DScale: Scaling Block-Diffusion Speculative Decoding with Adaptive Verification", SIII-C
// (Acceptance predictor): each draft position contributes its highest logit, the gaps to
// ranks 2..16, the top token's log-probability and the distribution entropy (18 values).
// DFlash-Mini-Lab README (DFlash7-ACT): a draft suffix is cut before the first position
// whose top-1/top-2 margin is below a calibrated threshold (0 keeps the full block).
//
// Row reduction over (row, chunk of 8192 elements) units, one warp per unit: per lane a
// sorted top-16 register list (bubble insertion, taken only by values that beat its tail)
// and the online (max m, s = sum e^(z-m), t = sum e^(z-m) (z-m)); warp merge by 16 rounds
// of warp max extraction; chunks of a row merged by the last warp to take the row's ticket.
// entropy = ln s - t / s; log-sum-exp = m + ln s.  HBM-bound over rows x vocab.
#include <cstdint>
#include <cuda_runtime.h>

#include "svp_device.cuh"

namespace svp {

constexpr int kFtChunk = 8192;
constexpr int kFtThreads = 256;
constexpr int kFtTop = 16;
constexpr int kFtPart = 20;   // 16 values, m, s, t, pad

struct FtParams {
    const void *logits;
    int64_t row_stride;
    int32_t rows, vocab, chunks;
    float *feat;                // [rows, 18]
    int32_t *tickets;           // [rows]
    float *partial;             // [rows * chunks, kFtPart]
};

struct FtState {
    float top[kFtTop];
    float m, s, t;
};

__device__ __forceinline__ void ft_init(FtState &st)
{
#pragma unroll
    for (int i = 0; i < kFtTop; ++i)
        st.top[i] = -INFINITY;
    st.m = -INFINITY;
    st.s = 0.0f;
    st.t = 0.0f;
}

__device__ __forceinline__ void ft_insert(FtState &st, float v)
{
    if (v > st.top[kFtTop - 1]) {
        float x = v;
#pragma unroll
        for (int i = 0; i < kFtTop; ++i) {
            const float hi = fmaxf(st.top[i], x);
            x = fminf(st.top[i], x);
            st.top[i] = hi;
        }
    }
}

// Fold one value into (m, s, t).
__device__ __forceinline__ void ft_acc(FtState &st, float v)
{
    constexpr float kL2e = 1.4426950408889634f;
    if (v > st.m) {
        if (st.m == -INFINITY) {
            st.m = v;
            st.s = 1.0f;
            st.t = 0.0f;
        } else {
            const float d = st.m - v;                  // < 0
            const float a = exp2f(d * kL2e);
            st.t = a * (st.t + st.s * d);
            st.s = a * st.s + 1.0f;
            st.m = v;
        }
    } else if (v != -INFINITY) {
        const float d = v - st.m;
        const float w = exp2f(d * kL2e);
        st.s += w;
        st.t += w * d;
    }
}

// Fold a vector of values: one rescale to the vector maximum, then one ex2 per value
// (ex2.approx: relative error ~2^-22, well inside the fp32 sums' own rounding).
template <int N>
__device__ __forceinline__ void ft_acc_vec(FtState &st, const float (&f)[N])
{
    constexpr float kL2e = 1.4426950408889634f;
    float vmax = f[0];
#pragma unroll
    for (int h = 1; h < N; ++h)
        vmax = fmaxf(vmax, f[h]);
    if (vmax == -INFINITY)
        return;
    if (vmax > st.m) {
        if (st.m == -INFINITY) {
            st.s = 0.0f;
            st.t = 0.0f;
        } else {
            const float d = st.m - vmax;
            const float a = fast_exp2(d * kL2e);
            st.t = a * (st.t + st.s * d);
            st.s = a * st.s;
        }
        st.m = vmax;
    }
    if (vmax > st.top[kFtTop - 1]) {
#pragma unroll
        for (int h = 0; h < N; ++h)
            ft_insert(st, f[h]);
    }
#pragma unroll
    for (int h = 0; h < N; ++h) {
        const float d = fmaxf(f[h] - st.m, -1e30f);   // -inf entries: weight 0, no 0 * inf
        const float w = fast_exp2(d * kL2e);
        st.s += w;
        st.t = fmaf(w, d, st.t);
    }
}

// Merge another (m, s, t) into st.
__device__ __forceinline__ void ft_merge_mst(FtState &st, float m2, float s2, float t2)
{
    constexpr float kL2e = 1.4426950408889634f;
    if (m2 == -INFINITY)
        return;
    if (st.m == -INFINITY) {
        st.m = m2;
        st.s = s2;
        st.t = t2;
        return;
    }
    const float M = fmaxf(st.m, m2);
    const float d1 = st.m - M, d2 = m2 - M;
    const float a1 = exp2f(d1 * kL2e), a2 = exp2f(d2 * kL2e);
    st.t = a1 * (st.t + st.s * d1) + a2 * (t2 + s2 * d2);
    st.s = a1 * st.s + a2 * s2;
    st.m = M;
}

// Warp-wide merge: every lane ends with the warp's top-16 in out[] and the merged m, s, t.
__device__ __forceinline__ void ft_warp_merge(FtState &st, float (&out)[kFtTop], int lane)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, st.m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, st.s, o);
        const float t2 = __shfl_xor_sync(0xffffffffu, st.t, o);
        ft_merge_mst(st, m2, s2, t2);
    }
#pragma unroll
    for (int k = 0; k < kFtTop; ++k) {
        float best = st.top[0];
        int who = lane;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
            const int w2 = __shfl_xor_sync(0xffffffffu, who, o);
            if (b2 > best || (b2 == best && w2 < who)) {
                best = b2;
                who = w2;
            }
        }
        out[k] = best;
        if (who == lane) {
#pragma unroll
            for (int i = 0; i < kFtTop - 1; ++i)
                st.top[i] = st.top[i + 1];
            st.top[kFtTop - 1] = -INFINITY;
        }
    }
}

__device__ __forceinline__ void ft_write(const FtParams &p, int32_t r, const float (&out)[kFtTop],
                                         float m, float s, float t)
{
    float *f = p.feat + (int64_t)r * 18;
    f[0] = out[0];
#pragma unroll
    for (int k = 1; k < kFtTop; ++k)
        f[k] = out[0] - out[k];
    const float ls = logf(s);
    f[16] = out[0] - (m + ls);
    f[17] = ls - t / s;
}

template <int DT>
__device__ __forceinline__ float ft_load(const void *base, int64_t idx)
{
    if (DT == 1)
        return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const uint16_t *>(base) + idx) << 16);
    return __ldg(reinterpret_cast<const float *>(base) + idx);
}

template <int DT>
__global__ void __launch_bounds__(kFtThreads) features_kernel(const FtParams p)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp_g = ((int64_t)blockIdx.x * kFtThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kFtThreads) >> 5;
    const int64_t units = (int64_t)p.rows * p.chunks;
    // 16-byte vectors: 8 bf16 or 4 fp32 values
    constexpr int VEC = DT == 1 ? 8 : 4;
    const bool vec_ok = ((p.row_stride * (DT == 1 ? 2 : 4)) & 15) == 0 &&
                        (reinterpret_cast<uintptr_t>(p.logits) & 15) == 0;
    for (int64_t u = warp_g; u < units; u += nwarps) {
        const int32_t r = (int32_t)(u / p.chunks), ch = (int32_t)(u - (int64_t)r * p.chunks);
        const int64_t lo = (int64_t)ch * kFtChunk;
        const int64_t hi = lo + kFtChunk < p.vocab ? lo + kFtChunk : p.vocab;
        const int64_t rowb = (int64_t)r * p.row_stride;
        FtState st;
        ft_init(st);
        int64_t e0 = lo;
        if (vec_ok) {
            const int64_t nv = (hi - lo) / VEC;
            const uint4 *src = reinterpret_cast<const uint4 *>(
                static_cast<const uint8_t *>(p.logits) + (rowb + lo) * (DT == 1 ? 2 : 4));
            for (int64_t v0 = lane; v0 < nv; v0 += 4 * 32) {
                uint4 x[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    x[q] = v0 + q * 32 < nv ? __ldg(src + v0 + q * 32)
                                            : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
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
                    ft_acc_vec<VEC>(st, f);
                }
            }
            e0 = lo + nv * VEC;
        }
        for (int64_t e = e0 + lane; e < hi; e += 32) {
            const float a = ft_load<DT>(p.logits, rowb + e);
            ft_insert(st, a);
            ft_acc(st, a);
        }
        float out[kFtTop];
        ft_warp_merge(st, out, lane);
        if (p.chunks == 1) {
            if (lane == 0)
                ft_write(p, r, out, st.m, st.s, st.t);
            continue;
        }
        int last = 0;
        if (lane == 0) {
            float *pp = p.partial + u * kFtPart;
#pragma unroll
            for (int k = 0; k < kFtTop; ++k)
                pp[k] = out[k];
            pp[16] = st.m;
            pp[17] = st.s;
            pp[18] = st.t;
            __threadfence();
            last = atomicAdd(p.tickets + r, 1) == p.chunks - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence();
            FtState mg;
            ft_init(mg);
            for (int q = lane; q < p.chunks; q += 32) {
                const float *pp = p.partial + ((int64_t)r * p.chunks + q) * kFtPart;
#pragma unroll
                for (int k = 0; k < kFtTop; ++k)
                    ft_insert(mg, __ldcg(pp + k));
                ft_merge_mst(mg, __ldcg(pp + 16), __ldcg(pp + 17), __ldcg(pp + 18));
            }
            float fin[kFtTop];
            ft_warp_merge(mg, fin, lane);
            if (lane == 0) {
                ft_write(p, r, fin, mg.m, mg.s, mg.t);
                p.tickets[r] = 0;
            }
        }
    }
}

__global__ void act_truncate_kernel(const float *margins, int64_t stride, int32_t n, int32_t w,
                                    float threshold, int32_t *k_out)
{
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n)
        return;
    int32_t k = 1;
    for (int32_t j = 1; j < w; ++j) {
        const float mg = __ldg(margins + ((int64_t)i * (w - 1) + (j - 1)) * stride);
        if (!(mg >= threshold))
            break;
        ++k;
    }
    k_out[i] = k;
}

static void ft_plan(int32_t rows, int32_t vocab, int32_t &chunks, size_t &off_tk,
                    size_t &off_part, size_t &bytes)
{
    chunks = (vocab + kFtChunk - 1) / kFtChunk;
    off_tk = kWsHeader;
    off_part = (off_tk + (size_t)rows * 4 + 255) / 256 * 256;
    bytes = off_part + (size_t)rows * chunks * kFtPart * sizeof(float);
}

}  // namespace svp

extern "C" svp_status svp_draft_features_workspace_size(int32_t rows, int32_t vocab,
                                                        size_t *bytes)
{
    using namespace svp;
    if (!bytes || rows < 0 || vocab < kFtTop)
        return SVP_EINVAL;
    int32_t chunks;
    size_t a, b;
    ft_plan(rows, vocab, chunks, a, b, *bytes);
    return SVP_OK;
}

extern "C" svp_status svp_draft_features(const void *logits, int64_t row_stride, int32_t rows,
                                         int32_t vocab, svp_dtype dtype, float *features,
                                         void *ws, size_t ws_bytes, void *stream)
{
    using namespace svp;
    if (!logits || !features || !ws || rows < 0 || vocab < kFtTop || row_stride < vocab)
        return SVP_EINVAL;
    if (dtype != SVP_BF16 && dtype != SVP_F32)
        return SVP_EUNSUPPORTED;
    FtParams p;
    size_t off_tk, off_part, need;
    ft_plan(rows, vocab, p.chunks, off_tk, off_part, need);
    if (ws_bytes < need)
        return SVP_EWORKSPACE;
    if (rows == 0)
        return SVP_OK;
    uint8_t *w = static_cast<uint8_t *>(ws);
    p.logits = logits;
    p.row_stride = row_stride;
    p.rows = rows;
    p.vocab = vocab;
    p.feat = features;
    p.tickets = reinterpret_cast<int32_t *>(w + off_tk);
    p.partial = reinterpret_cast<float *>(w + off_part);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SVP_ECUDA;
    const int64_t units = (int64_t)rows * p.chunks;
    int64_t grid = (units + (kFtThreads / 32) - 1) / (kFtThreads / 32);
    if (grid > (int64_t)sms * 8)
        grid = (int64_t)sms * 8;
    if (dtype == SVP_BF16)
        features_kernel<1><<<(unsigned)grid, kFtThreads, 0, (cudaStream_t)stream>>>(p);
    else
        features_kernel<0><<<(unsigned)grid, kFtThreads, 0, (cudaStream_t)stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? SVP_OK : SVP_ECUDA;
}

extern "C" svp_status svp_act_truncate(const float *margins, int64_t stride, int32_t n,
                                       int32_t w, float threshold, int32_t *k_out, void *stream)
{
    if (!margins || !k_out || n < 0 || w < 1 || stride < 1)
        return SVP_EINVAL;
    if (n == 0)
        return SVP_OK;
    svp::act_truncate_kernel<<<(n + 127) / 128, 128, 0, (cudaStream_t)stream>>>(
        margins, stride, n, w, threshold, k_out);
    return cudaGetLastError() == cudaSuccess ? SVP_OK : SVP_ECUDA;
}
