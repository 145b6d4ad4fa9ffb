// margin_accept.cu -- row top-1/top-2/margin over vocabulary logits, fused with greedy
// prefix acceptance.
//
// Definitions: DFlash-Mini-Lab README (DFlash7-ACT uses the top-1/top-2 draft-logit
// margin; one verifier call on [anchor + draft suffix], accept the exact prefix) and
// DScale SIII-D (Prefix verifier: after a_i accepted candidates, row offset_i + a_i
// supplies the successor).
//
// Design (HBM-bound stream, no tensor cores):
//   * Each logits row is cut into equal chunks of <= 16384 elements, more of them when the
//     batch is short, so that the units fill the resident warps once; every warp is an
//     independent worker on one (row, chunk) unit at a time (no CTA barriers).
//   * Each lane keeps a (top1, top1_idx, top2) triple over 16-byte vector loads, eight
//     in flight at once, updated without branches (a skip test on the lane's own top-2
//     diverges across the warp on nearly every vector of a chunk).  bf16 rows: packed
//     bf16x2 min/max over two interleaved streams, the lane maximum per vector with the
//     first vector that reached it, whose element index is recovered at the end; fp32
//     rows: top2 = max(top2, min(top1, x)), top1 = max(top1, x), the index moving only
//     on a strictly larger value (the lane's first occurrence of its maximum).
//   * Triples merge by warp shuffles; the merge is commutative and associative (ties:
//     lowest index), so results do not depend on arrival order.
//   * The warp that finishes the last chunk of a row (acquire-release ticket, no waiting)
//     finalises the row; in the fused kernel the warp that finalises the last row of a
//     request then runs the greedy acceptance for that request, all candidates at once
//     (lane l compares candidate l, the first mismatch by ballot).  Tickets, partials and
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

// Insert element (x, idx) without branches; indices reach a triple in increasing order,
// so the first occurrence of the maximum keeps its index.
__device__ __forceinline__ void top2_push_nb(Top2 &t, float x, int32_t idx)
{
    t.v2 = fmaxf(t.v2, fminf(t.v1, x));
    t.i1 = (x > t.v1 || t.i1 == INT_MAX) ? idx : t.i1;   // the lane's first element seeds it
    t.v1 = fmaxf(t.v1, x);
}

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

constexpr int kMarginThreads = 256;      // 8 independent warps per CTA
constexpr int kMarginBatch = 8;          // 16-byte loads in flight per lane

// Which request owns packed row r (cu_slots non-decreasing, validated by the caller).
__device__ __forceinline__ int32_t owner_of_row(const int32_t *cu, int32_t n, int32_t r)
{
    int32_t lo = 0, hi = n;   // the largest i < n with cu[i] <= r
    while (hi - lo > 1) {
        const int32_t mid = (lo + hi) >> 1;
        if (__ldg(cu + mid) <= r)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

template <bool kBf16>
__device__ __forceinline__ float load_elem(const MarginArgs &a, int64_t row, int32_t e)
{
    if (kBf16)
        return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(a.logits)[row * a.row_stride + e] << 16);
    return reinterpret_cast<const float *>(a.logits)[row * a.row_stride + e];
}

// One warp scans elements [c0, c1) of a row; lane-local triples, indices increasing.
template <bool kBf16>
__device__ __forceinline__ Top2 scan_chunk_warp(const MarginArgs &a, int64_t row, int32_t c0,
                                                int32_t c1, int lane)
{
    Top2 t = top2_identity();
    constexpr int VW = kBf16 ? 8 : 4;        // elements per 16-byte vector
    int32_t done = c0;
    if (a.vec_ok) {
        const int32_t nvec = (c1 - c0) / VW;
        const uint4 *vp = reinterpret_cast<const uint4 *>(
            reinterpret_cast<const uint8_t *>(a.logits) + (row * a.row_stride + c0) * (kBf16 ? 2 : 4));
        if (kBf16) {
            // two interleaved streams per lane (even / odd elements of each bf16 pair), each
            // with a packed (top1, top2): 3 bf16x2 min/max per pair of elements.  The lane's
            // maximum is tracked per vector with the first vector that reached it; the
            // element index is recovered from that vector at the end.
            uint32_t p1 = 0xff80ff80u, p2 = 0xff80ff80u;
            float vmax = -INFINITY;
            int32_t pos = -1;
            // each lane loads its own vectors v = lane, lane + 32, ..., eight in flight
            for (int32_t v0 = 0; v0 < nvec; v0 += 32 * kMarginBatch) {
                uint4 buf[kMarginBatch];
#pragma unroll
                for (int u = 0; u < kMarginBatch; ++u) {
                    const int32_t v = v0 + u * 32 + lane;
                    buf[u] = (v < nvec) ? __ldcs(vp + v) : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int32_t v = v0 + u * 32 + lane;
                    if (v >= nvec)
                        break;
                    const uint32_t w[4] = {buf[u].x, buf[u].y, buf[u].z, buf[u].w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        p2 = bf16x2_max(p2, bf16x2_min(p1, w[h]));
                        p1 = bf16x2_max(p1, w[h]);
                    }
                    const uint32_t m4 = bf16x2_max(bf16x2_max(w[0], w[1]), bf16x2_max(w[2], w[3]));
                    const float m8 = fmaxf(bf16_lo(m4), bf16_hi(m4));
                    const bool take = m8 > vmax || pos < 0;
                    pos = take ? v : pos;
                    vmax = take ? fmaxf(vmax, m8) : vmax;
                }
            }
            if (pos >= 0) {
                const float a1 = bf16_lo(p1), b1 = bf16_hi(p1);
                t.v1 = fmaxf(a1, b1);
                t.v2 = fmaxf(fminf(a1, b1), fmaxf(bf16_lo(p2), bf16_hi(p2)));
                const uint4 x = __ldg(vp + pos);
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
                int32_t j = 7;
#pragma unroll
                for (int h = 3; h >= 0; --h) {
                    j = bf16_hi(w[h]) == t.v1 ? 2 * h + 1 : j;
                    j = bf16_lo(w[h]) == t.v1 ? 2 * h : j;
                }
                t.i1 = c0 + pos * VW + j;
            }
        } else {
            for (int32_t v0 = 0; v0 < nvec; v0 += 32 * kMarginBatch) {
                uint4 buf[kMarginBatch];
#pragma unroll
                for (int u = 0; u < kMarginBatch; ++u) {
                    const int32_t v = v0 + u * 32 + lane;
                    buf[u] = (v < nvec) ? __ldcs(vp + v) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < kMarginBatch; ++u) {
                    const int32_t v = v0 + u * 32 + lane;
                    if (v >= nvec)
                        break;
                    const int32_t e0 = c0 + v * VW;
                    top2_push_nb(t, __uint_as_float(buf[u].x), e0 + 0);
                    top2_push_nb(t, __uint_as_float(buf[u].y), e0 + 1);
                    top2_push_nb(t, __uint_as_float(buf[u].z), e0 + 2);
                    top2_push_nb(t, __uint_as_float(buf[u].w), e0 + 3);
                }
            }
        }
        done = c0 + nvec * VW;
    }
    for (int32_t e = done + lane; e < c1; e += 32)      // ragged tail / unaligned rows
        top2_push(t, load_elem<kBf16>(a, row, e), e);
    return t;
}

// Greedy acceptance of request i by one warp, once every row argmax is in: lane l compares
// candidate j0 + l with the argmax of the row before it, and the first mismatch (ballot)
// ends the accepted prefix.
__device__ void finish_request(const MarginArgs &a, int32_t i, int lane)
{
    const int32_t off = __ldcg(a.cu_slots + i);
    const int32_t k = __ldcg(a.cu_slots + i + 1) - off;
    int32_t acc = k - 1;
    for (int32_t j0 = 1; j0 < k; j0 += 32) {
        const int32_t j = j0 + lane;
        const bool miss = j < k && __ldg(a.tokens + off + j) != __ldcg(a.row_argmax + off + j - 1);
        const uint32_t m = __ballot_sync(0xffffffffu, miss);
        if (m) {
            acc = j0 + __ffs(m) - 2;
            break;
        }
    }
    if (lane == 0) {
        a.accept_len[i] = 1 + acc;
        a.next_token[i] = __ldcg(a.row_argmax + off + acc);
    }
    __syncwarp();
    for (int32_t j = lane; j < k; j += 32)   // the workspace returns to zero
        a.row_argmax[off + j] = 0;
}

template <bool kBf16>
__global__ void __launch_bounds__(kMarginThreads, 4) margin_kernel(MarginArgs a)
{
    const int lane = threadIdx.x & 31;
    const int64_t gwarp = ((int64_t)blockIdx.x * kMarginThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kMarginThreads) >> 5;

    // fused mode: rows >= cu[n] are not read; invalid cu_slots -> nothing is read
    int32_t live_rows = a.rows;
    bool valid = true;
    if (a.cu_slots) {
        bool bad = (lane == 0) && (__ldg(a.cu_slots) != 0);
        for (int32_t i = lane; i < a.n; i += 32)
            bad |= __ldg(a.cu_slots + i + 1) < __ldg(a.cu_slots + i);
        live_rows = __ldg(a.cu_slots + a.n);
        bad |= live_rows > a.rows || live_rows < 0;
        valid = !__any_sync(0xffffffffu, bad);
        if (!valid) {
            live_rows = 0;
            if (gwarp == 0 && lane == 0)
                set_status(a.status, SVP_DEV_BAD_SLOTS);
        }
    }
    const int64_t units = (int64_t)live_rows * a.chunks_per_row;

    for (int64_t w = gwarp; w < units; w += nwarps) {
        const int64_t row = w / a.chunks_per_row;
        const int32_t ch = (int32_t)(w % a.chunks_per_row);
        const int32_t c0 = ch * a.chunk;
        const int32_t c1 = min(a.vocab, c0 + a.chunk);
        Top2 t = top2_warp_merge(scan_chunk_warp<kBf16>(a, row, c0, c1, lane));
        int last = 0;
        if (lane == 0) {
            a.partial[row * a.chunks_per_row + ch] = t;
            last = ticket_add_acq_rel(a.row_ticket + row, 1) == a.chunks_per_row - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last)
            continue;
        // last chunk of this row: merge its partials (lane-parallel) and clear them; lane 0's
        // acquire orders the other lanes' reads through the warp barrier
        __syncwarp();
        Top2 *pp = a.partial + row * a.chunks_per_row;
        Top2 r = top2_identity();
        for (int32_t k = lane; k < a.chunks_per_row; k += 32) {
            Top2 u;
            u.v1 = __ldcg(&pp[k].v1);
            u.v2 = __ldcg(&pp[k].v2);
            u.i1 = __ldcg(&pp[k].i1);
            r = top2_merge(r, u);
            pp[k] = Top2{0.0f, 0.0f, 0};
        }
        r = top2_warp_merge(r);
        int32_t fin = -1;   // request whose last row this is
        if (lane == 0) {
            a.row_ticket[row] = 0;
            if (a.top1_idx) a.top1_idx[row] = r.i1;
            if (a.top1) a.top1[row] = r.v1;
            if (a.top2) a.top2[row] = r.v2;
            if (a.margin) a.margin[row] = __fsub_rn(r.v1, r.v2);
            if (a.cu_slots) {
                a.row_argmax[row] = r.i1;
                const int32_t i = owner_of_row(a.cu_slots, a.n, (int32_t)row);
                const int32_t k = __ldg(a.cu_slots + i + 1) - __ldg(a.cu_slots + i);
                if (ticket_add_acq_rel(a.req_ticket + i, 1) == k - 1) {
                    a.req_ticket[i] = 0;
                    fin = i;
                }
            }
        }
        fin = __shfl_sync(0xffffffffu, fin, 0);
        if (fin >= 0) {
            __syncwarp();   // lane 0's acquire on the request ticket orders the other lanes' reads
            finish_request(a, fin, lane);
        }
    }

    // inactive requests (k_i = 0) have no rows: the first warp writes their results
    if (a.cu_slots && gwarp == 0 && valid) {
        for (int32_t i = lane; i < a.n; i += 32) {
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

int sm_count();   // defined in api.cu

// Chunks per row: at least enough for units of at most 16384 elements (32 KB of bf16), and
// as many as fill the resident warps once (4 CTAs of 8 warps per SM at 64 registers), so
// that every warp gets one unit of about the same size; at most 64.
static MarginPlan margin_plan(int32_t rows, int32_t vocab, int32_t n)
{
    MarginPlan p{};
    const int32_t target = 16384;
    const int64_t warps = (int64_t)sm_count() * 4 * (kMarginThreads / 32);
    int64_t per_row = (vocab + target - 1) / target;
    const int64_t fill = rows > 0 ? warps / rows : 1;
    per_row = per_row > fill ? per_row : (fill > 64 ? 64 : fill);
    p.chunks_per_row = per_row < 1 ? 1 : (int32_t)per_row;
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
    // one unit per warp, capped at eight resident CTAs of 8 warps per SM (grid-stride)
    const int64_t work = (int64_t)rows * p.chunks_per_row;
    int64_t grid = (work + kMarginThreads / 32 - 1) / (kMarginThreads / 32);
    if (grid > (int64_t)sm_count() * 8)
        grid = (int64_t)sm_count() * 8;
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
