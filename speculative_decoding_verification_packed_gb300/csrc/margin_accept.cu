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
//   * Draft rows (no acceptance): the warp that delivers the last chunk of a row (one
//     acquire-release ticket per row, no waiting) merges the row's chunk triples.
//   * Fused margin + accept: the ticket is per request and counts the chunks of all its
//     rows, so the warp that delivers the request's last chunk merges every row of the
//     request (four lanes per row, eight rows per pass), writes the row outputs and runs
//     the greedy acceptance on the row argmaxes it holds: one ticket and one read-back on
//     the tail instead of a row level and a request level.  Tickets and triples are
//     cleared by their last reader, so the workspace is all zero again after every call
//     and can serve calls of any size.
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

// A chunk's triple as stored in the workspace: 16 bytes, read back with one vector load.
struct alignas(16) Top2Part {
    float v1;
    float v2;
    int32_t i1;
    int32_t pad;
};

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
    Top2Part *partial;       // [rows * chunks_per_row]
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

__device__ __forceinline__ Top2 load_part(const Top2Part *p)
{
    const int4 q = __ldcg(reinterpret_cast<const int4 *>(p));
    return Top2{__int_as_float(q.x), __int_as_float(q.y), q.z};
}

// Request i (packed rows off .. off + k - 1) once the chunks of all its rows are in: one warp
// merges every row's chunk triples (four lanes per row, eight rows per pass, each lane's
// triples loaded together), writes the row outputs, and runs the greedy acceptance on the
// row argmaxes as they come: row j's argmax is compared with draft token j + 1, and the
// first mismatch ends the accepted prefix.  The triples it read are cleared.
__device__ void finish_request(const MarginArgs &a, int32_t i, int32_t off, int32_t k, int lane)
{
    const int32_t cpr = a.chunks_per_row;
    const int sub = lane & 3, g = lane >> 2;     // quarter and row of this lane within a pass
    int32_t acc = -1, nxt = -1;                   // decided: accepted drafts, successor token
    for (int32_t j0 = 0; j0 < k; j0 += 8) {
        const int32_t j = j0 + g;                 // request row of this lane
        const bool live = j < k;
        const int32_t tok = live && j + 1 < k ? __ldg(a.tokens + off + j + 1) : 0;
        Top2 r = top2_identity();
        if (live) {
            Top2Part *pp = a.partial + (int64_t)(off + j) * cpr;
            for (int32_t c0 = sub; c0 < cpr; c0 += 32) {       // one pass while cpr <= 32
                Top2 u[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    u[q] = c0 + 4 * q < cpr ? load_part(pp + c0 + 4 * q) : top2_identity();
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    // chunks in increasing order within the lane: ties keep the lowest index
                    r = top2_merge(r, u[q]);
                    if (c0 + 4 * q < cpr)
                        *reinterpret_cast<int4 *>(pp + c0 + 4 * q) = make_int4(0, 0, 0, 0);
                }
            }
        }
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {       // the row's four lanes
            Top2 v;
            v.v1 = __shfl_xor_sync(0xffffffffu, r.v1, o);
            v.v2 = __shfl_xor_sync(0xffffffffu, r.v2, o);
            v.i1 = __shfl_xor_sync(0xffffffffu, r.i1, o);
            r = top2_merge(r, v);
        }
        const int64_t row = off + j;
        if (live && sub == 0) {
            if (a.top1_idx) a.top1_idx[row] = r.i1;
            if (a.top1) a.top1[row] = r.v1;
            if (a.top2) a.top2[row] = r.v2;
            if (a.margin) a.margin[row] = __fsub_rn(r.v1, r.v2);
        }
        if (acc < 0) {
            // row j ends the prefix when it is the last row or draft j + 1 differs
            const bool stop = live && (j + 1 == k || tok != r.i1);
            const uint32_t m = __ballot_sync(0xffffffffu, stop && sub == 0);
            if (m) {
                const int src = __ffs(m) - 1;
                acc = j0 + (src >> 2);
                nxt = __shfl_sync(0xffffffffu, r.i1, src);
            }
        }
    }
    if (lane == 0) {
        a.accept_len[i] = 1 + acc;
        a.next_token[i] = nxt;
    }
}

// Which request owns packed row r: cu_slots non-decreasing (validated), so it is the number
// of requests 1 .. n-1 that start at or before r (empty requests own no rows).
__device__ __forceinline__ int32_t owner_of_row_warp(const int32_t *cu, int32_t n, int32_t r, int lane)
{
    int32_t cnt = 0;
    for (int32_t l0 = 1; l0 < n; l0 += 32) {
        const int32_t l = l0 + lane;
        cnt += __popc(__ballot_sync(0xffffffffu, l < n && __ldg(cu + l) <= r));
    }
    return cnt;
}

template <bool kBf16>
__global__ void __launch_bounds__(kMarginThreads, 4) margin_kernel(MarginArgs a)
{
    griddep_launch_dependents();
    griddep_wait();
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
        if (a.cu_slots) {
            // fused: the warp that delivers the last chunk of the last row of a request
            // finishes the whole request (acquire-release ticket over its chunks)
            const int32_t i = owner_of_row_warp(a.cu_slots, a.n, (int32_t)row, lane);
            const int32_t off = __ldg(a.cu_slots + i);
            const int32_t k = __ldg(a.cu_slots + i + 1) - off;
            int last = 0;
            if (lane == 0) {
                a.partial[row * a.chunks_per_row + ch] = Top2Part{t.v1, t.v2, t.i1, 0};
                last = ticket_add_acq_rel(a.req_ticket + i, 1) == k * a.chunks_per_row - 1;
                if (last)
                    a.req_ticket[i] = 0;
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __syncwarp();   // lane 0's acquire orders the other lanes' reads
                finish_request(a, i, off, k, lane);
            }
            continue;
        }
        int last = 0;
        if (lane == 0) {
            a.partial[row * a.chunks_per_row + ch] = Top2Part{t.v1, t.v2, t.i1, 0};
            last = ticket_add_acq_rel(a.row_ticket + row, 1) == a.chunks_per_row - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last)
            continue;
        // last chunk of this row: merge its partials (lane-parallel) and clear them; lane 0's
        // acquire orders the other lanes' reads through the warp barrier
        __syncwarp();
        Top2Part *pp = a.partial + row * a.chunks_per_row;
        Top2 r = top2_identity();
        for (int32_t k = lane; k < a.chunks_per_row; k += 32) {
            r = top2_merge(r, load_part(pp + k));
            *reinterpret_cast<int4 *>(pp + k) = make_int4(0, 0, 0, 0);
        }
        r = top2_warp_merge(r);
        if (lane == 0) {
            a.row_ticket[row] = 0;
            if (a.top1_idx) a.top1_idx[row] = r.i1;
            if (a.top1) a.top1[row] = r.v1;
            if (a.top2) a.top2[row] = r.v2;
            if (a.margin) a.margin[row] = __fsub_rn(r.v1, r.v2);
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
    griddep_launch_dependents();
    griddep_wait();
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
    p.off_partial = o; o = al(o + sizeof(Top2Part) * (size_t)rows * p.chunks_per_row);
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
    a.partial = reinterpret_cast<Top2Part *>(w + p.off_partial);
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
    const cudaError_t e = dtype == SVP_BF16
                              ? launch_pdl(margin_kernel<true>, dim3((unsigned)grid), dim3(kMarginThreads), 0, stream, a)
                              : launch_pdl(margin_kernel<false>, dim3((unsigned)grid), dim3(kMarginThreads), 0, stream, a);
    return e == cudaSuccess ? SVP_OK : SVP_ECUDA;
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
    return launch_pdl(greedy_accept_kernel, dim3((unsigned)((n + threads - 1) / threads)), dim3(threads), 0,
                      stream, target_argmax, tokens, cu_slots, n, m_cap, accept_len, next_token,
                      static_cast<int32_t *>(nullptr)) == cudaSuccess
               ? SVP_OK
               : SVP_ECUDA;
}

}  // namespace svp
