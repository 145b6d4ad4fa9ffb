// margin_accept.cu -- row top-1/top-2/margin over vocabulary logits, fused with greedy
// prefix acceptance.
//
// Definitions: DFlash-Mini-Lab README (DFlash7-ACT uses the top-1/top-2 draft-logit
// margin; one verifier call on [anchor + draft suffix], accept the exact prefix) and
// DScale SIII-D (Prefix verifier: after a_i accepted candidates, row offset_i + a_i
// supplies the successor).
//
// Design (HBM-bound stream, no tensor cores):
//   * Each logits row is cut into equal chunks of <= 16384 elements; a persistent grid
//     (a multiple of the SM count) strides over all (row, chunk) pairs.
//   * Each thread keeps a (top1, top1_idx, top2) triple over 16-byte vector loads that
//     are all issued before use; a vector whose maximum cannot beat the current top-2
//     is skipped after one packed max.
//   * Triples merge by warp shuffles and shared memory; the merge is commutative and
//     associative (ties: lowest index), so results do not depend on arrival order.
//   * The CTA that finishes the last chunk of a row (atomic ticket, no waiting)
//     finalises the row; in the fused kernel the CTA that finalises the last row of a
//     request then runs the greedy acceptance for that request.  Tickets, partials and
//     per-row argmaxes are cleared by their last reader, so the workspace is all zero
//     again after every call and can serve calls of any size.
#include <cfloat>
#include <climits>
#include <cuda_bf16.h>

#include "svp_device.cuh"

namespace svp {

struct Top2 {
    float v1;
    float v2;
    int32_t i1;
};

__device__ __forceinline__ Top2 top2_identity() { return Top2{-INFINITY, -INFINITY, INT_MAX}; }

// Insert element (x, idx); indices reach a given triple in increasing order.
__device__ __forceinline__ void top2_push(Top2 &t, float x, int32_t idx)
{
    if (x > t.v1 || (x == t.v1 && idx < t.i1)) {
        t.v2 = t.v1;
        t.v1 = x;
        t.i1 = idx;
    } else if (x > t.v2) {
        t.v2 = x;
    }
}

// Merge two triples over disjoint index sets.
__device__ __forceinline__ Top2 top2_merge(Top2 a, Top2 b)
{
    const bool b_wins = (b.v1 > a.v1) || (b.v1 == a.v1 && b.i1 < a.i1);
    Top2 w = b_wins ? b : a;
    Top2 l = b_wins ? a : b;
    w.v2 = fmaxf(w.v2, l.v1);
    return w;
}

__device__ __forceinline__ Top2 top2_warp_merge(Top2 t)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Top2 u;
        u.v1 = __shfl_xor_sync(0xffffffffu, t.v1, o);
        u.v2 = __shfl_xor_sync(0xffffffffu, t.v2, o);
        u.i1 = __shfl_xor_sync(0xffffffffu, t.i1, o);
        t = top2_merge(t, u);
    }
    return t;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b)
{
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162 *>(&a);
    __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162 *>(&b);
    __nv_bfloat162 z = __hmax2(x, y);
    return *reinterpret_cast<uint32_t *>(&z);
}

struct MarginArgs {
    const void *logits;
    int64_t row_stride;      // elements
    int32_t rows;            // rows of the logits buffer (m_cap for the fused kernel)
    int32_t vocab;
    int32_t chunk;           // elements per chunk (multiple of the vector width)
    int32_t chunks_per_row;
    int32_t vec_ok;          // rows start 16-byte aligned
    int32_t *top1_idx;       // outputs, each nullable
    float *top1;
    float *top2;
    float *margin;
    // workspace
    int32_t *status;
    int32_t *row_ticket;     // [rows]
    int32_t *row_argmax;     // [rows]
    Top2 *partial;           // [rows * chunks_per_row]
    // fused acceptance (cu_slots == nullptr: margin only)
    const int32_t *tokens;
    const int32_t *cu_slots;
    int32_t n;
    int32_t *req_ticket;     // [n]
    int32_t *accept_len;
    int32_t *next_token;
};

constexpr int kMarginThreads = 256;
constexpr int kMarginUnroll = 8;

// Which request owns packed row r (cu_slots non-decreasing, validated by the caller).
__device__ __forceinline__ int32_t owner_of_row(const int32_t *cu, int32_t n, int32_t r)
{
    int32_t lo = 0, hi = n;   // find the largest i with cu[i] <= r, among i < n
    while (hi - lo > 1) {
        int32_t mid = (lo + hi) >> 1;
        if (__ldg(cu + mid) <= r)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

template <bool kBf16>
__device__ __forceinline__ Top2 scan_chunk(const MarginArgs &a, int64_t row, int32_t c0, int32_t c1)
{
    Top2 t = top2_identity();
    const int tid = threadIdx.x;
    constexpr int VW = kBf16 ? 8 : 4;        // elements per 16-byte vector
    if (a.vec_ok) {
        const int32_t nvec = (c1 - c0) / VW;
        const uint8_t *base = reinterpret_cast<const uint8_t *>(a.logits) +
                              (row * a.row_stride + c0) * (kBf16 ? 2 : 4);
        const uint4 *vp = reinterpret_cast<const uint4 *>(base);
        for (int32_t v0 = 0; v0 < nvec; v0 += kMarginThreads * kMarginUnroll) {
            uint4 buf[kMarginUnroll];
#pragma unroll
            for (int u = 0; u < kMarginUnroll; ++u) {
                const int32_t v = v0 + u * kMarginThreads + tid;
                if (v < nvec)
                    buf[u] = __ldcs(vp + v);
                else
                    buf[u] = make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kMarginUnroll; ++u) {
                const int32_t v = v0 + u * kMarginThreads + tid;
                if (v >= nvec)
                    break;
                const int32_t e0 = c0 + v * VW;
                if (kBf16) {
                    const uint32_t m4 = bf16x2_max(bf16x2_max(buf[u].x, buf[u].y),
                                                   bf16x2_max(buf[u].z, buf[u].w));
                    const float m8 = fmaxf(bf16_lo(m4), bf16_hi(m4));
                    if (m8 > t.v2 || t.i1 == INT_MAX) {
                        top2_push(t, bf16_lo(buf[u].x), e0 + 0);
                        top2_push(t, bf16_hi(buf[u].x), e0 + 1);
                        top2_push(t, bf16_lo(buf[u].y), e0 + 2);
                        top2_push(t, bf16_hi(buf[u].y), e0 + 3);
                        top2_push(t, bf16_lo(buf[u].z), e0 + 4);
                        top2_push(t, bf16_hi(buf[u].z), e0 + 5);
                        top2_push(t, bf16_lo(buf[u].w), e0 + 6);
                        top2_push(t, bf16_hi(buf[u].w), e0 + 7);
                    }
                } else {
                    const float x0 = __uint_as_float(buf[u].x), x1 = __uint_as_float(buf[u].y);
                    const float x2 = __uint_as_float(buf[u].z), x3 = __uint_as_float(buf[u].w);
                    const float m4 = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
                    if (m4 > t.v2 || t.i1 == INT_MAX) {
                        top2_push(t, x0, e0 + 0);
                        top2_push(t, x1, e0 + 1);
                        top2_push(t, x2, e0 + 2);
                        top2_push(t, x3, e0 + 3);
                    }
                }
            }
        }
        // ragged tail of the chunk (only the row's last chunk can have one)
        for (int32_t e = c0 + nvec * VW + tid; e < c1; e += kMarginThreads) {
            float x;
            if (kBf16)
                x = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(a.logits)[row * a.row_stride + e] << 16);
            else
                x = reinterpret_cast<const float *>(a.logits)[row * a.row_stride + e];
            top2_push(t, x, e);
        }
    } else {
        for (int32_t e = c0 + tid; e < c1; e += kMarginThreads) {
            float x;
            if (kBf16)
                x = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(a.logits)[row * a.row_stride + e] << 16);
            else
                x = reinterpret_cast<const float *>(a.logits)[row * a.row_stride + e];
            top2_push(t, x, e);
        }
    }
    return t;
}

__device__ void finish_request(const MarginArgs &a, int32_t i)
{
    const int32_t off = __ldcg(a.cu_slots + i);
    const int32_t k = __ldcg(a.cu_slots + i + 1) - off;
    int32_t acc = 0;
    while (acc + 1 < k && __ldg(a.tokens + off + acc + 1) == __ldcg(a.row_argmax + off + acc))
        ++acc;
    a.accept_len[i] = 1 + acc;
    a.next_token[i] = __ldcg(a.row_argmax + off + acc);
    for (int32_t j = 0; j < k; ++j)      // the workspace returns to zero
        a.row_argmax[off + j] = 0;
}

template <bool kBf16>
__global__ void __launch_bounds__(kMarginThreads) margin_kernel(MarginArgs a)
{
    __shared__ Top2 warp_part[kMarginThreads / 32];
    __shared__ int s_flag;
    __shared__ int32_t s_live_rows;
    __shared__ int s_valid;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;

    // Fused mode: validate cu_slots once per CTA; rows >= cu[n] are not read.
    if (tid == 0) {
        int32_t live = a.rows;
        int valid = 1;
        if (a.cu_slots) {
            int bad = (__ldg(a.cu_slots) != 0);
            for (int32_t i = 0; i < a.n && !bad; ++i)
                bad = __ldg(a.cu_slots + i + 1) < __ldg(a.cu_slots + i);
            live = __ldg(a.cu_slots + a.n);
            if (bad || live > a.rows || live < 0) {
                live = 0;
                valid = 0;
                if (blockIdx.x == 0)
                    set_status(a.status, SVP_DEV_BAD_SLOTS);
            }
        }
        s_live_rows = live;
        s_valid = valid;
    }
    __syncthreads();
    const int32_t live_rows = s_live_rows;
    const int64_t total = (int64_t)live_rows * a.chunks_per_row;

    for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
        const int64_t row = w / a.chunks_per_row;
        const int32_t ch = (int32_t)(w % a.chunks_per_row);
        const int32_t c0 = ch * a.chunk;
        const int32_t c1 = min(a.vocab, c0 + a.chunk);
        Top2 t = scan_chunk<kBf16>(a, row, c0, c1);
        t = top2_warp_merge(t);
        if (lane == 0)
            warp_part[warp] = t;
        __syncthreads();
        if (tid == 0) {
            Top2 r = warp_part[0];
            for (int k = 1; k < kMarginThreads / 32; ++k)
                r = top2_merge(r, warp_part[k]);
            a.partial[row * a.chunks_per_row + ch] = r;
            __threadfence();
            const int prev = atomicAdd(a.row_ticket + row, 1);
            s_flag = (prev == a.chunks_per_row - 1);
        }
        __syncthreads();
        if (s_flag && tid == 0) {
            // last chunk of this row: merge the row's partials in chunk order
            __threadfence();
            Top2 *pp = a.partial + row * a.chunks_per_row;
            Top2 r = top2_identity();
            for (int k = 0; k < a.chunks_per_row; ++k) {
                Top2 u;
                u.v1 = __ldcg(&pp[k].v1);
                u.v2 = __ldcg(&pp[k].v2);
                u.i1 = __ldcg(&pp[k].i1);
                r = top2_merge(r, u);
                pp[k] = Top2{0.0f, 0.0f, 0};   // the workspace returns to zero
            }
            a.row_ticket[row] = 0;
            if (a.top1_idx) a.top1_idx[row] = r.i1;
            if (a.top1) a.top1[row] = r.v1;
            if (a.top2) a.top2[row] = r.v2;
            if (a.margin) a.margin[row] = __fsub_rn(r.v1, r.v2);
            if (a.cu_slots) {
                a.row_argmax[row] = r.i1;
                __threadfence();
                const int32_t i = owner_of_row(a.cu_slots, a.n, (int32_t)row);
                const int32_t k = __ldg(a.cu_slots + i + 1) - __ldg(a.cu_slots + i);
                const int prev = atomicAdd(a.req_ticket + i, 1);
                if (prev == k - 1) {
                    __threadfence();
                    a.req_ticket[i] = 0;
                    finish_request(a, i);
                }
            }
        }
        __syncthreads();
    }

    // Inactive requests (k_i = 0) have no rows: block 0 writes their results.
    if (a.cu_slots && blockIdx.x == 0 && s_valid) {
        for (int32_t i = tid; i < a.n; i += kMarginThreads) {
            if (__ldg(a.cu_slots + i + 1) == __ldg(a.cu_slots + i)) {
                a.accept_len[i] = 0;
                a.next_token[i] = -1;
            }
        }
    }
}

__global__ void greedy_accept_kernel(const int32_t *target_argmax, const int32_t *tokens,
                                     const int32_t *cu_slots, int32_t n, int32_t m_cap,
                                     int32_t *accept_len, int32_t *next_token, int32_t *status)
{
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n)
        return;
    const int32_t off = __ldg(cu_slots + i);
    const int32_t end = __ldg(cu_slots + i + 1);
    if (off < 0 || end < off || end > m_cap) {
        set_status(status, SVP_DEV_BAD_SLOTS);
        accept_len[i] = 0;
        next_token[i] = -1;
        return;
    }
    const int32_t k = end - off;
    if (k == 0) {
        accept_len[i] = 0;
        next_token[i] = -1;
        return;
    }
    int32_t acc = 0;
    while (acc + 1 < k && __ldg(tokens + off + acc + 1) == __ldg(target_argmax + off + acc))
        ++acc;
    accept_len[i] = 1 + acc;
    next_token[i] = __ldg(target_argmax + off + acc);
}

// ------------------------------------------------------------------ host side
struct MarginPlan {
    int32_t chunk, chunks_per_row;
    size_t off_row_ticket, off_row_argmax, off_req_ticket, off_partial, bytes;
};

static MarginPlan margin_plan(int32_t rows, int32_t vocab, int32_t n)
{
    MarginPlan p{};
    const int32_t target = 16384;
    p.chunks_per_row = (vocab + target - 1) / target;
    if (p.chunks_per_row < 1)
        p.chunks_per_row = 1;
    int32_t c = (vocab + p.chunks_per_row - 1) / p.chunks_per_row;
    c = (c + 7) / 8 * 8;
    p.chunk = c;
    p.chunks_per_row = (vocab + c - 1) / c;
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    size_t o = kWsHeader;
    p.off_row_ticket = o; o = al(o + sizeof(int32_t) * (size_t)rows);
    p.off_row_argmax = o; o = al(o + sizeof(int32_t) * (size_t)rows);
    p.off_req_ticket = o; o = al(o + sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    p.off_partial = o; o = al(o + sizeof(Top2) * (size_t)rows * p.chunks_per_row);
    p.bytes = o;
    return p;
}

int sm_count();   // defined in api.cu

svp_status margin_workspace(int32_t rows, int32_t vocab, int32_t n, size_t *bytes)
{
    if (!bytes || rows < 0 || vocab < 2 || n < 0)
        return SVP_EINVAL;
    *bytes = margin_plan(rows, vocab, n).bytes;
    return SVP_OK;
}

svp_status margin_launch(const void *logits, int64_t row_stride, int32_t rows, int32_t vocab,
                         svp_dtype dtype, int32_t *top1_idx, float *top1, float *top2,
                         float *margin, const int32_t *tokens, const int32_t *cu_slots,
                         int32_t n, int32_t *accept_len, int32_t *next_token, void *ws,
                         size_t ws_bytes, cudaStream_t stream)
{
    if (rows < 0 || vocab < 2 || row_stride < vocab || n < 0)
        return SVP_EINVAL;
    if (dtype != SVP_F32 && dtype != SVP_BF16)
        return SVP_EUNSUPPORTED;
    if ((rows > 0 && !logits) || !ws)
        return ws ? SVP_EINVAL : SVP_EWORKSPACE;
    const bool fused = cu_slots != nullptr;
    if (fused && (!tokens || !accept_len || !next_token))
        return SVP_EINVAL;
    const MarginPlan p = margin_plan(rows, vocab, fused ? n : 0);
    if (ws_bytes < p.bytes)
        return SVP_EWORKSPACE;
    if (rows == 0 && !(fused && n > 0))
        return SVP_OK;
    MarginArgs a{};
    a.logits = logits;
    a.row_stride = row_stride;
    a.rows = rows;
    a.vocab = vocab;
    a.chunk = p.chunk;
    a.chunks_per_row = p.chunks_per_row;
    const int esz = dtype == SVP_BF16 ? 2 : 4;
    a.vec_ok = ((reinterpret_cast<uintptr_t>(logits) & 15) == 0) &&
               ((row_stride * esz) % 16 == 0) && ((p.chunk * esz) % 16 == 0);
    a.top1_idx = top1_idx;
    a.top1 = top1;
    a.top2 = top2;
    a.margin = margin;
    uint8_t *w = static_cast<uint8_t *>(ws);
    a.status = reinterpret_cast<int32_t *>(w);
    a.row_ticket = reinterpret_cast<int32_t *>(w + p.off_row_ticket);
    a.row_argmax = reinterpret_cast<int32_t *>(w + p.off_row_argmax);
    a.req_ticket = reinterpret_cast<int32_t *>(w + p.off_req_ticket);
    a.partial = reinterpret_cast<Top2 *>(w + p.off_partial);
    a.tokens = tokens;
    a.cu_slots = cu_slots;
    a.n = n;
    a.accept_len = accept_len;
    a.next_token = next_token;
    const int64_t work = (int64_t)rows * p.chunks_per_row;
    int64_t grid = (int64_t)sm_count() * 4;
    if (grid > work)
        grid = work;
    if (grid < 1)
        grid = 1;
    if (dtype == SVP_BF16)
        margin_kernel<true><<<(unsigned)grid, kMarginThreads, 0, stream>>>(a);
    else
        margin_kernel<false><<<(unsigned)grid, kMarginThreads, 0, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? SVP_OK : SVP_ECUDA;
}

svp_status accept_launch(const int32_t *target_argmax, const int32_t *tokens,
                         const int32_t *cu_slots, int32_t n, int32_t m_cap,
                         int32_t *accept_len, int32_t *next_token, cudaStream_t stream)
{
    if (n < 0 || m_cap < 0)
        return SVP_EINVAL;
    if (n == 0)
        return SVP_OK;
    if (!target_argmax || !tokens || !cu_slots || !accept_len || !next_token)
        return SVP_EINVAL;
    const int threads = 128;
    greedy_accept_kernel<<<(n + threads - 1) / threads, threads, 0, stream>>>(
        target_argmax, tokens, cu_slots, n, m_cap, accept_len, next_token, nullptr);
    return cudaGetLastError() == cudaSuccess ? SVP_OK : SVP_ECUDA;
}

}  // namespace svp
