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
// Two launches.  (1) Softmax statistics over (row, chunk) units, one warp per unit with
// eight 16-byte loads in flight per lane, the chunk sized so that the units of m_cap rows
// fill the GPU's resident warps once: the chunk's (max, sum of
// 2^((z - max) log2(e) / T)) is kept per chunk and merged per row by the last warp to take
// the row's ticket; bf16 batches take their maximum by packed max and rebase the sum once.
// HBM-bound over the live logit rows.  (2) One block per request: warp 0 tests every
// candidate at once (probabilities from the row statistics, first rejection by ballot)
// while the other warps bring the chunk statistics of the request's rows into shared
// memory, then walks the chunk masses of the successor row in token order to the chunk
// that holds the draw; the block rescans only that chunk (block prefix sum of per-thread
// masses, then one thread's elements in order).  (2) is a programmatic dependent launch of
// (1): its blocks start on SMs that (1) has left, load their input-only operands, and wait
// on the device before reading the statistics; each block returns its request's row and
// chunk statistics to zero once read, so the workspace is all zero after every call.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "svp_device.cuh"

namespace svp {

constexpr int kStChunkMin = 256;        // chunk sizes are multiples of this (one bf16 vector per lane)
constexpr int kStWarpsPerSm = 32;       // resident pass-1 warps per SM (4 CTAs of 8 warps at 64 registers)
constexpr int kStMaxChunks = 64;        // chunks per row at most
constexpr int kStThreads1 = 256;
constexpr int kStThreads2 = 512;
constexpr uint32_t kStNegInf2 = 0xff80ff80u;   // packed bf16 (-inf, -inf)
constexpr int kStPrefRows = 16;        // rows of a request whose chunk statistics pass 2 prefetches
constexpr int kStLoads = 8;             // pass 1: 16-byte loads in flight per lane

struct StParams {
    const void *logits;
    int64_t row_stride;
    int32_t m_cap, vocab, dtype, n, chunks, chunk;   // chunk: elements per (row, chunk) unit
    float c;                            // log2(e) / T
    const int32_t *tokens, *cu_slots;
    const float *u_accept, *u_next;
    int32_t *accept_len, *next_token;
    float *p_draft;
    int32_t *status;
    float2 *row_stat;                   // [m_cap]: (max, sum of 2^((z - max) c))
    int32_t *tickets;                   // [m_cap]
    float2 *partial;                    // [m_cap * chunks]: the same per chunk
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

__device__ __forceinline__ float2 st_warp_merge(float2 a, float c)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float2 b;
        b.x = __shfl_xor_sync(0xffffffffu, a.x, o);
        b.y = __shfl_xor_sync(0xffffffffu, a.y, o);
        a = st_merge(a, b, c);
    }
    return a;
}

// Fold N values of one lane into (m, s): one rescale to the vector maximum.  The exponent
// of each value is one fma against mc = m c rounded to fp32: the rounding shifts every
// exponent of this lane's (m, s) by the same amount (|m c| 2^-24), a common factor of the
// chunk's weights that is far below the probabilities' tolerance.
template <int N>
__device__ __forceinline__ void st_acc(float &m, float &mc, float &s, const float (&f)[N], float c)
{
    float vmax = f[0];
#pragma unroll
    for (int h = 1; h < N; ++h)
        vmax = fmaxf(vmax, f[h]);
    if (vmax == -INFINITY)
        return;
    if (vmax > m) {
        s = m == -INFINITY ? 0.0f : s * fast_exp2((m - vmax) * c);
        m = vmax;
        mc = m * c;
    }
#pragma unroll
    for (int h = 0; h < N; ++h)
        s += fast_exp2(fmaf(f[h], c, -mc));
}

template <int DT>
__global__ void __launch_bounds__(kStThreads1, 4) st_rowstat_kernel(const StParams p)
{
    // the grid always fits in one wave (at most 4 CTAs per SM): the acceptance pass may be
    // scheduled as soon as every CTA has started, onto SMs as this pass frees them
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warp_g = ((int64_t)blockIdx.x * kStThreads1 + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kStThreads1) >> 5;
    // cu_slots must start at 0, never decrease and end within m_cap; otherwise no row is read
    // and the second pass gives every request 0 / -1
    bool bad = (lane == 0) && (__ldg(p.cu_slots) != 0);
    for (int32_t i = lane; i < p.n; i += 32)
        bad |= __ldg(p.cu_slots + i + 1) < __ldg(p.cu_slots + i);
    int32_t live = __ldg(p.cu_slots + p.n);
    bad |= live > p.m_cap || live < 0;
    const bool valid = !__any_sync(0xffffffffu, bad);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        p.status[2] = valid ? 0 : 1;
        if (!valid)
            set_status(p.status, SVP_DEV_BAD_SLOTS);
    }
    if (!valid)
        live = 0;
    const int64_t units = (int64_t)live * p.chunks;
    constexpr int VEC = DT == 1 ? 8 : 4;
    const bool vec_ok = ((p.row_stride * (DT == 1 ? 2 : 4)) & 15) == 0 &&
                        (reinterpret_cast<uintptr_t>(p.logits) & 15) == 0;
    for (int64_t u = warp_g; u < units; u += nwarps) {
        const int32_t r = (int32_t)(u / p.chunks), ch = (int32_t)(u - (int64_t)r * p.chunks);
        const int64_t lo = (int64_t)ch * p.chunk;
        const int64_t hi = lo + p.chunk < p.vocab ? lo + p.chunk : p.vocab;
        const int64_t rowb = (int64_t)r * p.row_stride;
        float m = -INFINITY, mc = 0.0f, s = 0.0f;
        int64_t e0 = lo;
        if (vec_ok) {
            const int64_t nv = (hi - lo) / VEC;
            const uint4 *src = reinterpret_cast<const uint4 *>(
                static_cast<const uint8_t *>(p.logits) + (rowb + lo) * (DT == 1 ? 2 : 4));
            for (int64_t v0 = 0; v0 < nv; v0 += kStLoads * 32) {
                uint4 x[kStLoads];
#pragma unroll
                for (int q = 0; q < kStLoads; ++q) {
                    const int64_t v = v0 + q * 32 + lane;
                    x[q] = v < nv ? __ldg(src + v) : make_uint4(kStNegInf2, kStNegInf2, kStNegInf2, kStNegInf2);
                }
                if constexpr (DT == 1) {
                    // bf16: the batch maximum by packed max (vectors past the end hold -inf),
                    // one rescale, then every value of the batch
                    uint32_t b2 = kStNegInf2;
#pragma unroll
                    for (int q = 0; q < kStLoads; ++q)
                        b2 = bf16x2_max(bf16x2_max(b2, bf16x2_max(x[q].x, x[q].y)), bf16x2_max(x[q].z, x[q].w));
                    const float bmax = fmaxf(bf16_lo(b2), bf16_hi(b2));
                    if (bmax == -INFINITY)
                        continue;
                    if (bmax > m) {
                        s = m == -INFINITY ? 0.0f : s * fast_exp2((m - bmax) * p.c);
                        m = bmax;
                        mc = m * p.c;
                    }
                    float s0 = 0.0f, s1 = 0.0f;   // two chains of adds
#pragma unroll
                    for (int q = 0; q < kStLoads; ++q) {
                        const uint32_t w[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            s0 += fast_exp2(fmaf(bf16_lo(w[h]), p.c, -mc));
                            s1 += fast_exp2(fmaf(bf16_hi(w[h]), p.c, -mc));
                        }
                    }
                    s += s0 + s1;
                } else {
#pragma unroll
                    for (int q = 0; q < kStLoads; ++q) {
                        if (v0 + q * 32 + lane >= nv)
                            continue;
                        float f[VEC];
                        f[0] = __uint_as_float(x[q].x);
                        f[1] = __uint_as_float(x[q].y);
                        f[2] = __uint_as_float(x[q].z);
                        f[3] = __uint_as_float(x[q].w);
                        st_acc<VEC>(m, mc, s, f, p.c);
                    }
                }
            }
            e0 = lo + nv * VEC;
        }
        for (int64_t e = e0 + lane; e < hi; e += 32) {
            float f[1];
            f[0] = st_load<DT>(p.logits, rowb + e);
            st_acc<1>(m, mc, s, f, p.c);
        }
        float2 a = st_warp_merge(make_float2(m, m == -INFINITY ? 0.0f : s), p.c);
        // the successor draw walks the chunk masses, so every chunk's pair is kept
        if (lane == 0)
            p.partial[u] = a;
        if (p.chunks == 1) {
            if (lane == 0)
                p.row_stat[r] = a;
            continue;
        }
        int last = 0;
        if (lane == 0)
            last = ticket_add_acq_rel(p.tickets + r, 1) == p.chunks - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __syncwarp();   // lane 0's acquire orders the other lanes' reads of the partials
            float2 t = make_float2(-INFINITY, 0.0f);
            for (int q = lane; q < p.chunks; q += 32)
                t = st_merge(t, __ldcg(p.partial + (int64_t)r * p.chunks + q), p.c);
            t = st_warp_merge(t, p.c);
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
    constexpr int NW = kStThreads2 / 32;
    __shared__ float2 sh_part[kStPrefRows * kStMaxChunks];   // chunk statistics of the first rows
    __shared__ float sh_sum[NW];
    __shared__ float sh_target, sh_m;
    __shared__ int32_t sh_row, sh_excl, sh_chunk, sh_claim, sh_lastnz;
    const int i = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t off = __ldg(p.cu_slots + i), end = __ldg(p.cu_slots + i + 1);
    const bool meta_ok = off >= 0 && end >= off && end <= p.m_cap;
    // before the wait for the statistics pass: what depends on the inputs only.  Warp 0
    // brings the first 32 candidates' tokens, their logits on the rows they are tested on
    // and their acceptance draws.
    int32_t x_pre = -1;
    float z_pre = -INFINITY, u_pre = 0.0f;
    if (warp == 0 && meta_ok && 1 + lane < end - off) {
        const int32_t j = 1 + lane;
        x_pre = __ldg(p.tokens + off + j);
        if (x_pre >= 0 && x_pre < p.vocab)
            z_pre = st_load<DT>(p.logits, (int64_t)(off + j - 1) * p.row_stride + x_pre);
        u_pre = __ldg(p.u_accept + off + j);
    }
    griddep_wait();
    // the first pass found cu_slots invalid (it set the status bit): nothing was read
    if (*reinterpret_cast<volatile int32_t *>(p.status + 2) != 0 || !meta_ok) {
        if (tid == 0) {
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
    // the other warps bring the chunk statistics of the request's first rows (any of them
    // may be the successor row) into shared memory while warp 0 runs the acceptance chain
    const int32_t npre = k < kStPrefRows ? k : kStPrefRows;
    if (warp > 0) {
        for (int32_t x = tid - 32; x < npre * p.chunks; x += kStThreads2 - 32)
            sh_part[x] = __ldcg(p.partial + (int64_t)off * p.chunks + x);
        named_bar_arrive(1, kStThreads2);
    }
    if (warp == 0) {
        // ---- acceptance chain: lane l tests candidate j0 + l (row off + j - 1); the first
        // rejection, found by ballot, ends the prefix.  Probabilities are written for the
        // candidates tested in order (up to and including the first rejection).
        // the last row's maximum, in case every candidate is accepted
        const float m_last = lane == 0 ? __ldcg(p.row_stat + off + k - 1).x : 0.0f;
        int32_t a = 0, excl = -1;
        float M = 0.0f, zx = -INFINITY;   // successor row maximum; rejected token's logit
        bool rejected = false;
        for (int32_t j0 = 1; j0 < k; j0 += 32) {
            const int32_t j = j0 + lane;
            float pr = 0.0f, z = -INFINITY, mr = 0.0f;
            int32_t x = -1;
            bool pass = true;
            if (j < k) {
                const int32_t r = off + j - 1;
                float u;
                if (j0 == 1) {   // brought before the wait
                    x = x_pre;
                    z = z_pre;
                    u = u_pre;
                } else {
                    x = __ldg(p.tokens + off + j);
                    if (x >= 0 && x < p.vocab)
                        z = st_load<DT>(p.logits, (int64_t)r * p.row_stride + x);
                    u = __ldg(p.u_accept + off + j);
                }
                const float2 st = __ldcg(p.row_stat + r);
                mr = st.x;
                if (x >= 0 && x < p.vocab)
                    pr = exp2f((z - st.x) * p.c) / st.y;
                pass = u < pr;
            }
            const uint32_t rej = __ballot_sync(0xffffffffu, !pass);
            const int first = rej ? __ffs(rej) - 1 : 32;
            if (p.p_draft && j < k && lane <= first)
                p.p_draft[off + j] = pr;
            if (rej) {
                // the successor row is the row the rejected candidate was tested on
                a += first;
                excl = __shfl_sync(0xffffffffu, x, first);
                zx = __shfl_sync(0xffffffffu, z, first);
                M = __shfl_sync(0xffffffffu, mr, first);
                rejected = true;
                break;
            }
            a += min(32, k - j0);
        }
        if (!rejected)
            M = __shfl_sync(0xffffffffu, m_last, 0);
        // ---- successor row r = off + a: chunk masses relative to the row max, the rejected
        // token's mass taken out of its chunk; walk them in token order to the draw.
        const int32_t r = off + a;
        float wx = 0.0f;
        int32_t cx = -1;
        if (excl >= 0 && excl < p.vocab) {
            wx = exp2f((zx - M) * p.c);
            cx = excl / p.chunk;
        }
        named_bar_sync(1, kStThreads2);   // the prefetched chunk statistics are in
        const float2 *prow = a < npre ? sh_part + a * p.chunks : p.partial + (int64_t)r * p.chunks;
        auto chunk_mass = [&](int32_t ch) -> float {
            if (ch >= p.chunks)
                return 0.0f;
            const float2 pc = a < npre ? prow[ch] : __ldcg(prow + ch);
            float w = pc.x == -INFINITY ? 0.0f : pc.y * exp2f((pc.x - M) * p.c);
            if (ch == cx)   // what is left within rounding of the removed token counts as none
                w = w - wx > w * 0x1p-20f ? w - wx : 0.0f;
            return w;
        };
        float tot = 0.0f;
        for (int32_t c0 = 0; c0 < p.chunks; c0 += 32)
            tot += chunk_mass(c0 + lane);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            tot += __shfl_xor_sync(0xffffffffu, tot, o);
        const float target = __ldg(p.u_next + i) * tot;
        int32_t sel = -1, last_nz = -1;
        float sel_before = 0.0f, carry = 0.0f;
        for (int32_t c0 = 0; c0 < p.chunks; c0 += 32) {
            const float w = chunk_mass(c0 + lane);
            float incl = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += y;
            }
            incl += carry;
            const float before = incl - w;
            const uint32_t nz = __ballot_sync(0xffffffffu, w > 0.0f);
            if (nz)
                last_nz = c0 + 31 - __clz(nz);
            const uint32_t hit = __ballot_sync(0xffffffffu, w > 0.0f && before <= target && target < incl);
            if (hit) {
                const int l = __ffs(hit) - 1;
                sel = c0 + l;
                sel_before = __shfl_sync(0xffffffffu, before, l);
                break;
            }
            carry = __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            p.accept_len[i] = 1 + a;
            sh_row = r;
            sh_excl = excl;
            sh_m = M;
            // rounding left the draw past every chunk: the last chunk with mass, whose last
            // token with weight is taken below
            sh_chunk = sel >= 0 ? sel : last_nz;
            sh_target = sel >= 0 ? target - sel_before : INFINITY;
            sh_claim = kStThreads2;
            sh_lastnz = -1;
        }
    }
    __syncthreads();
    // the request's rows are done with their statistics: back to zero, so that the workspace
    // is all zero after every call and serves later calls with other m_cap and vocabularies
    for (int32_t x = tid; x < k * (1 + p.chunks); x += kStThreads2) {
        if (x < k)
            p.row_stat[off + x] = make_float2(0.0f, 0.0f);
        else
            p.partial[(int64_t)off * p.chunks + (x - k)] = make_float2(0.0f, 0.0f);
    }
    const int32_t r = sh_row, excl = sh_excl, ch = sh_chunk;
    if (ch < 0) {   // no token with weight at all (every other token underflowed)
        if (tid == 0)
            p.next_token[i] = -1;
        return;
    }
    const float m = sh_m, target = sh_target;
    const int64_t rowb = (int64_t)r * p.row_stride;
    const int64_t clo = (int64_t)ch * p.chunk;
    const int64_t chi = clo + p.chunk < p.vocab ? clo + p.chunk : p.vocab;
    // per thread a contiguous run of whole 16-byte vectors (the chunk starts on one); each
    // weight is one ex2.approx (relative error ~2^-22), the same expression in the sum below
    // and in the claiming thread's scan, so that the scan reproduces the sum exactly
    constexpr int VEC = DT == 1 ? 8 : 4;
    const int64_t per = ((chi - clo + kStThreads2 - 1) / kStThreads2 + VEC - 1) / VEC * VEC;
    const int64_t lo = clo + (int64_t)tid * per;
    const int64_t hi = lo + per < chi ? lo + per : chi;
    const bool vec_ok = ((p.row_stride * (DT == 1 ? 2 : 4)) & 15) == 0 &&
                        (reinterpret_cast<uintptr_t>(p.logits) & 15) == 0;
    float own = 0.0f;
    int64_t e = lo;
    uint4 xb[8];   // the last batch of vectors; with at most eight it is the thread's whole run
    if (vec_ok) {
        const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(p.logits) +
                                                           (rowb + lo) * (DT == 1 ? 2 : 4));
        const int64_t nv = hi > lo ? (hi - lo) / VEC : 0;
        for (int64_t v0 = 0; v0 < nv; v0 += 8) {   // eight vectors in flight, summed in order
#pragma unroll
            for (int q = 0; q < 8; ++q)
                xb[q] = v0 + q < nv ? __ldg(src + v0 + q) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (v0 + q >= nv)
                    break;
                const int64_t v = v0 + q;
                const uint32_t w[4] = {xb[q].x, xb[q].y, xb[q].z, xb[q].w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    if (DT == 1) {
                        const int64_t e2 = lo + v * VEC + 2 * h;
                        own += e2 != excl ? fast_exp2((bf16_lo(w[h]) - m) * p.c) : 0.0f;
                        own += e2 + 1 != excl ? fast_exp2((bf16_hi(w[h]) - m) * p.c) : 0.0f;
                    } else {
                        own += lo + v * VEC + h != excl ? fast_exp2((__uint_as_float(w[h]) - m) * p.c) : 0.0f;
                    }
                }
            }
        }
        e = lo + nv * VEC;
    }
    for (; e < hi; ++e)
        if (e != excl)
            own += fast_exp2((st_load<DT>(p.logits, rowb + e) - m) * p.c);
    // block exclusive scan of the per-thread masses
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
        float t = lane < NW ? sh_sum[lane] : 0.0f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o)
                t += y;
        }
        if (lane < NW)
            sh_sum[lane] = t;
    }
    __syncthreads();
    const float before = (warp > 0 ? sh_sum[warp - 1] : 0.0f) + incl - own;
    // the lowest thread whose interval [before, before + own) holds the draw
    if (own > 0.0f && before <= target && target < before + own)
        atomicMin(&sh_claim, tid);
    if (own > 0.0f)
        atomicMax(&sh_lastnz, tid);
    __syncthreads();
    const int claim = sh_claim;
    // no claim (the draw lies past the recomputed masses by rounding): the chunk's last token
    // with weight
    const int who = claim < kStThreads2 ? claim : sh_lastnz;
    if (tid == who) {
        // the same weights in the same order as the sum above; the thread's 16-byte vectors
        // come eight at a time (one round trip per batch, none when the run fits one batch)
        float cum = before;
        int32_t y = -1, lnz = -1;
        bool found = false;
        const bool want = claim < kStThreads2;
        auto take = [&](int64_t e2, float v) {
            if (found || e2 == excl)
                return;
            const float w = fast_exp2((v - m) * p.c);
            if (w > 0.0f)
                lnz = (int32_t)e2;
            cum += w;
            if (want && cum > target && w > 0.0f) {
                y = (int32_t)e2;
                found = true;
            }
        };
        int64_t e3 = lo;
        if (vec_ok) {
            const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(p.logits) +
                                                               (rowb + lo) * (DT == 1 ? 2 : 4));
            const int64_t nv = hi > lo ? (hi - lo) / VEC : 0;
            for (int64_t v0 = 0; v0 < nv && !found; v0 += 8) {
                if (nv > 8) {   // otherwise the vectors summed above are still in xb
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        xb[q] = v0 + q < nv ? __ldg(src + v0 + q) : make_uint4(0u, 0u, 0u, 0u);
                }
                for (int q = 0; q < 8 && v0 + q < nv && !found; ++q) {
                    const uint32_t w4[4] = {xb[q].x, xb[q].y, xb[q].z, xb[q].w};
                    const int64_t eb = lo + (v0 + q) * VEC;
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        if (DT == 1) {
                            take(eb + 2 * h, bf16_lo(w4[h]));
                            take(eb + 2 * h + 1, bf16_hi(w4[h]));
                        } else {
                            take(eb + h, __uint_as_float(w4[h]));
                        }
                    }
                }
            }
            e3 = lo + nv * VEC;
        }
        for (; e3 < hi && !found; ++e3)
            take(e3, st_load<DT>(p.logits, rowb + e3));
        p.next_token[i] = y >= 0 ? y : lnz;
    }
    if (tid == 0 && who < 0)
        p.next_token[i] = -1;
}

// Chunk size: the rows of m_cap get floor(resident pass-1 warps / m_cap) chunks each (at
// least one, at most kStMaxChunks), so that the units fill the resident warps at most once;
// chunks are multiples of kStChunkMin.
static int32_t st_chunk(int32_t m_cap, int32_t vocab, int sms)
{
    const int64_t warps = (int64_t)sms * kStWarpsPerSm;
    int64_t per_row = m_cap > 0 ? warps / m_cap : 1;
    per_row = per_row < 1 ? 1 : (per_row > kStMaxChunks ? kStMaxChunks : per_row);
    int64_t c = ((int64_t)vocab + per_row - 1) / per_row;
    c = (c + kStChunkMin - 1) / kStChunkMin * kStChunkMin;
    return (int32_t)c;
}

static void st_plan(int32_t m_cap, int32_t vocab, size_t &off_stat, size_t &off_tk,
                    size_t &off_part, size_t &bytes)
{
    const int64_t mc = ((int64_t)vocab + kStChunkMin - 1) / kStChunkMin;
    off_stat = kWsHeader;
    off_tk = off_stat + (size_t)m_cap * sizeof(float2);
    off_part = (off_tk + (size_t)m_cap * 4 + 255) / 256 * 256;
    bytes = off_part + (size_t)m_cap * (mc < kStMaxChunks ? mc : kStMaxChunks) * sizeof(float2);
}

}  // namespace svp

extern "C" svp_status svp_stochastic_accept_workspace_size(int32_t m_cap, int32_t vocab,
                                                           size_t *bytes)
{
    using namespace svp;
    if (!bytes || m_cap < 0 || vocab < 2)
        return SVP_EINVAL;
    size_t a, b, c;
    st_plan(m_cap, vocab, a, b, c, *bytes);
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
        !next_token || n < 0 || m_cap < 0 || vocab < 2 || row_stride < vocab ||
        !(temperature > 0.0f))
        return SVP_EINVAL;
    if (dtype != SVP_BF16 && dtype != SVP_F32)
        return SVP_EUNSUPPORTED;
    StParams p;
    size_t off_stat, off_tk, off_part, need;
    st_plan(m_cap, vocab, off_stat, off_tk, off_part, need);
    if (!ws || ws_bytes < need)
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
    p.chunk = st_chunk(m_cap, vocab, sms);
    p.chunks = (vocab + p.chunk - 1) / p.chunk;
    const int64_t units = (int64_t)m_cap * p.chunks;
    int64_t grid1 = (units + (kStThreads1 / 32) - 1) / (kStThreads1 / 32);
    if (grid1 > (int64_t)sms * (kStWarpsPerSm * 32 / kStThreads1))
        grid1 = (int64_t)sms * (kStWarpsPerSm * 32 / kStThreads1);
    if (grid1 < 1)
        grid1 = 1;
    cudaStream_t s = (cudaStream_t)stream;
    // the acceptance pass is a programmatic dependent of the statistics pass: its CTAs start
    // on SMs the first pass has left and wait on the device before reading its results
    cudaError_t e;
    if (dtype == SVP_BF16) {
        st_rowstat_kernel<1><<<(unsigned)grid1, kStThreads1, 0, s>>>(p);
        e = cudaGetLastError();
        if (e == cudaSuccess)
            e = launch_pdl(st_accept_kernel<1>, dim3((unsigned)n), dim3(kStThreads2), 0, s, p);
    } else {
        st_rowstat_kernel<0><<<(unsigned)grid1, kStThreads1, 0, s>>>(p);
        e = cudaGetLastError();
        if (e == cudaSuccess)
            e = launch_pdl(st_accept_kernel<0>, dim3((unsigned)n), dim3(kStThreads2), 0, s, p);
    }
    return e == cudaSuccess ? SVP_OK : SVP_ECUDA;
}
