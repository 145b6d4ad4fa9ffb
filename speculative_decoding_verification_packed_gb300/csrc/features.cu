// features.cu -- draft-signal features per draft-logit row, and ACT truncation.
//
// "DScale: Scaling Block-Diffusion Speculative Decoding with Adaptive Verification", SIII-C
// (Acceptance predictor): each draft position contributes its highest logit, the gaps to
// ranks 2..16, the top token's log-probability and the distribution entropy (18 values).
// DFlash-Mini-Lab README (DFlash7-ACT): a draft suffix is cut before the first position
// whose top-1/top-2 margin is below a calibrated threshold (0 keeps the full block).
//
// Row reduction over (row, chunk) units, one warp per unit, the chunk sized so that the
// units fill the GPU's resident warps once; the chunks of a row are merged by the last warp
// to take the row's acquire-release ticket, which also returns the row's partial lists and
// ticket to zero (the workspace is all zero after every call).
//  * Softmax statistics per lane: an online (max m, s = sum 2^d, t = sum 2^d d) with
//    d = (z - m) log2 e; entropy = ln s - t ln2 / s, log-sum-exp = m + ln s.  bf16 rows:
//    a batch of eight 16-byte vectors is summed in packed f32x2 arithmetic against the
//    running reference m, which then moves to the batch maximum; a batch whose sums
//    overflow or turn NaN (a -inf logit) is redone with the reference moved first and -inf
//    read as -9.97e37.  A warp's (m, s, t) fold: the warp maximum by one redux, one rescale
//    per lane, a butterfly sum.
//  * Top-16, bf16 rows: each lane's 8 streams (packed word k of its 16-byte vectors, low or
//    high half) keep their top 4; a selection network on the packed words merges each
//    batch's 8 values per stream (and yields the batch maximum).  16 rounds of redux on
//    unique order-preserving keys draw the chunk's top-16 from those entries.  Exact unless
//    a stream's fourth value reaches the 16th drawn value; then (rarely) the chunk is
//    rescanned taking only values at or above it.
//  * Top-16, fp32 rows and the rescan: the warp's top-16 so far sorted across lanes 0..15
//    with the 16th value as a warp-uniform threshold; a vector is offered only when its
//    maximum beats the threshold, and an insertion is a ballot, a popcount and a lane shift.
// HBM-bound over rows x vocab (issue-bound in practice for bf16: packed min / max and one
// exponential per value).
#include <cstdint>
#include <cuda_runtime.h>

#include "svp_device.cuh"

namespace svp {

constexpr int kFtChunkMin = 256;    // chunk sizes are multiples of this (one 16-byte bf16 vector per lane)
constexpr int kFtWarpsPerSm = 24;   // resident warps per SM the chunk size is planned for
constexpr int kFtMaxChunks = 64;
constexpr int kFtThreads = 256;
constexpr int kFtTop = 16;
constexpr int kFtPart = 20;   // 16 values, m, s, t, pad
constexpr int kFtLoads = 8;   // 16-byte loads in flight per lane
constexpr float kFtL2e = 1.4426950408889634f;
constexpr float kFtLn2 = 0.69314718055994531f;
constexpr uint32_t kFtNegInf2 = 0xff80ff80u;   // packed bf16 (-inf, -inf)
constexpr uint32_t kFtLow2 = 0xfe96fe96u;      // packed bf16 (-9.97e37, -9.97e37)

struct FtParams {
    const void *logits;
    int64_t row_stride;
    int32_t rows, vocab, chunks, chunk;   // chunk: elements per (row, chunk) unit
    float *feat;                // [rows, 18]
    int32_t *tickets;           // [rows]
    float *partial;             // [rows * chunks, kFtPart]
};

// Warp-distributed sorted top-16: lane j < 16 holds the j-th largest value so far
// (-inf when fewer were seen); tau = lane 15's value, the same in every lane.
struct FtTop {
    float slot, tau, floor;   // floor: values at or below it are never taken
};

__device__ __forceinline__ void ft_top_init(FtTop &w)
{
    w.slot = -INFINITY;
    w.tau = -INFINITY;
    w.floor = -INFINITY;
}

// Insert v (warp-uniform, v > tau): the slots >= v are a prefix of length pos <= 15; the
// ones after it move down one lane.
__device__ __forceinline__ void ft_top_insert(FtTop &w, float v, int lane)
{
    const uint32_t ge = __ballot_sync(0xffffffffu, lane < kFtTop && w.slot >= v);
    const int pos = __popc(ge);
    const float prev = __shfl_up_sync(0xffffffffu, w.slot, 1);
    if (lane < kFtTop && lane >= pos)
        w.slot = lane == pos ? v : prev;
    w.tau = fmaxf(__shfl_sync(0xffffffffu, w.slot, kFtTop - 1), w.floor);
}

// Offer the N values of every lane in `cand` (lanes whose vector maximum beat tau), lane by
// lane in lane order.
template <int N>
__device__ __forceinline__ void ft_top_offer(FtTop &w, const float (&f)[N], uint32_t cand,
                                             int lane)
{
    while (cand) {
        const int src = __ffs(cand) - 1;
        cand &= cand - 1;
#pragma unroll
        for (int h = 0; h < N; ++h) {
            const float v = __shfl_sync(0xffffffffu, f[h], src);
            if (v > w.tau)
                ft_top_insert(w, v, lane);
        }
    }
}

// Online softmax statistics of one lane, base 2: m is the natural-unit maximum.
struct FtStat {
    float m, s, t;
};

__device__ __forceinline__ void ft_stat_init(FtStat &st)
{
    st.m = -INFINITY;
    st.s = 0.0f;
    st.t = 0.0f;
}

// Fold N values: one rescale to the vector maximum, then one ex2 per value (ex2.approx:
// relative error ~2^-22, well inside the fp32 sums' own rounding).  The exponent is one fma
// against the rounded m log2 e: at T = 1 its absolute error (~1e-6 for |m| < 50) is far
// below the sums' tolerance.  CLAMP: the values may hold -inf (weight 0, and no 0 * inf).
// Move the reference of (m, s, t) up to vmax when vmax exceeds it.
__device__ __forceinline__ void ft_stat_rebase(FtStat &st, float vmax)
{
    if (vmax > st.m) {
        if (st.m == -INFINITY) {
            st.s = 0.0f;
            st.t = 0.0f;
        } else {
            const float d = (st.m - vmax) * kFtL2e;
            const float a = fast_exp2(d);
            st.t = a > 0.0f ? a * (st.t + st.s * d) : 0.0f;   // d may be huge: no 0 * inf
            st.s = a * st.s;
        }
        st.m = vmax;
    }
}

template <int N, bool CLAMP>
__device__ __forceinline__ void ft_stat_acc(FtStat &st, const float (&f)[N], float vmax)
{
    if (vmax == -INFINITY)
        return;
    ft_stat_rebase(st, vmax);
    const float ml = st.m * kFtL2e;
#pragma unroll
    for (int h = 0; h < N; ++h) {
        float d = fmaf(f[h], kFtL2e, -ml);
        if (CLAMP)
            d = fmaxf(d, -1e30f);
        const float w = fast_exp2(d);
        st.s += w;
        st.t = fmaf(w, d, st.t);
    }
}

__device__ __forceinline__ void ft_stat_merge(FtStat &st, float m2, float s2, float t2)
{
    if (m2 == -INFINITY)
        return;
    if (st.m == -INFINITY) {
        st.m = m2;
        st.s = s2;
        st.t = t2;
        return;
    }
    const float M = fmaxf(st.m, m2);
    const float d1 = (st.m - M) * kFtL2e, d2 = (m2 - M) * kFtL2e;
    const float a1 = exp2f(d1), a2 = exp2f(d2);
    st.t = (a1 > 0.0f ? a1 * (st.t + st.s * d1) : 0.0f) + (a2 > 0.0f ? a2 * (t2 + s2 * d2) : 0.0f);
    st.s = a1 * st.s + a2 * s2;
    st.m = M;
}

// Order-preserving 32-bit code of a float (unsigned order of the codes = order of the
// values, -0 just below +0; no NaN) and its inverse.
__device__ __forceinline__ uint32_t ft_ord32(float f)
{
    const uint32_t u = __float_as_uint(f);
    return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

__device__ __forceinline__ float ft_unord32(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// Fold the 32 lanes' (m, s, t): the warp maximum M by one redux, each lane's sums moved to
// M, then a butterfly sum.  Every lane ends with the warp's (M, s, t).
__device__ __forceinline__ void ft_stat_warp(FtStat &st)
{
    const float M = ft_unord32(__reduce_max_sync(0xffffffffu, ft_ord32(st.m)));
    if (M == -INFINITY)   // warp-uniform: no lane saw a value
        return;
    float s = 0.0f, t = 0.0f;
    if (st.m != -INFINITY) {
        const float d = (st.m - M) * kFtL2e;
        const float a = exp2f(d);
        s = a * st.s;
        t = a > 0.0f ? a * (st.t + st.s * d) : 0.0f;   // d may be huge: no 0 * inf
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        s += __shfl_xor_sync(0xffffffffu, s, o);
        t += __shfl_xor_sync(0xffffffffu, t, o);
    }
    st.m = M;
    st.s = s;
    st.t = t;
}

// Lane 0 writes the 18 features of row r (top values gathered from lanes 0..15).
__device__ __forceinline__ void ft_write(const FtParams &p, int32_t r, const FtTop &w,
                                         const FtStat &st, int lane)
{
    const float top0 = __shfl_sync(0xffffffffu, w.slot, 0);
    float *f = p.feat + (int64_t)r * 18;
    if (lane == 0)
        f[0] = top0;
    else if (lane < kFtTop)
        f[lane] = top0 - w.slot;
    if (lane == 0) {
        const float ls = logf(st.s);
        f[16] = top0 - (st.m + ls);
        f[17] = ls - st.t * kFtLn2 / st.s;
    }
}

template <int DT>
__device__ __forceinline__ float ft_load(const void *base, int64_t idx)
{
    if (DT == 1)
        return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const uint16_t *>(base) + idx) << 16);
    return __ldg(reinterpret_cast<const float *>(base) + idx);
}

template <int DT>
__device__ __forceinline__ void ft_unpack(const uint4 &x, float (&f)[DT == 1 ? 8 : 4])
{
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        if (DT == 1) {
            f[2 * h] = bf16_lo(w[h]);
            f[2 * h + 1] = bf16_hi(w[h]);
        } else {
            f[h] = __uint_as_float(w[h]);
        }
    }
}

// Any dtype, any alignment: the warp-shared top-16 takes a vector only when its maximum
// beats the threshold; WITH_STAT also folds every value into st (with -inf handling).
template <int DT, bool WITH_STAT>
__device__ __forceinline__ void ft_scan_generic(const FtParams &p, int64_t rowb, int64_t lo,
                                                int64_t hi, bool vec_ok, int lane, FtTop &top,
                                                FtStat &st)
{
    constexpr int VEC = DT == 1 ? 8 : 4;
    int64_t e0 = lo;
    if (vec_ok) {
        const int64_t nv = (hi - lo) / VEC;
        const uint4 *src = reinterpret_cast<const uint4 *>(
            static_cast<const uint8_t *>(p.logits) + (rowb + lo) * (DT == 1 ? 2 : 4));
        for (int64_t v0 = 0; v0 < nv; v0 += kFtLoads * 32) {
            uint4 x[kFtLoads];
#pragma unroll
            for (int q = 0; q < kFtLoads; ++q) {
                const int64_t v = v0 + q * 32 + lane;
                x[q] = v < nv ? __ldg(src + v) : make_uint4(kFtNegInf2, kFtNegInf2, kFtNegInf2, kFtNegInf2);
            }
#pragma unroll
            for (int q = 0; q < kFtLoads; ++q) {
                if (v0 + q * 32 >= nv)   // warp-uniform
                    break;
                float f[VEC];
                if (v0 + q * 32 + lane < nv) {
                    ft_unpack<DT>(x[q], f);
                } else {
#pragma unroll
                    for (int h = 0; h < VEC; ++h)
                        f[h] = -INFINITY;
                }
                float vmax = f[0];
#pragma unroll
                for (int h = 1; h < VEC; ++h)
                    vmax = fmaxf(vmax, f[h]);
                if (WITH_STAT)
                    ft_stat_acc<VEC, true>(st, f, vmax);
                const uint32_t cand = __ballot_sync(0xffffffffu, vmax > top.tau);
                if (cand)
                    ft_top_offer<VEC>(top, f, cand, lane);
            }
        }
        e0 = lo + nv * VEC;
    }
    // ragged tail (or rows without 16-byte alignment): one value per lane per step
    for (int64_t e0b = e0; e0b < hi; e0b += 32) {
        float f[1];
        f[0] = e0b + lane < hi ? ft_load<DT>(p.logits, rowb + e0b + lane) : -INFINITY;
        if (WITH_STAT)
            ft_stat_acc<1, true>(st, f, f[0]);
        const uint32_t cand = __ballot_sync(0xffffffffu, f[0] > top.tau);
        if (cand)
            ft_top_offer<1>(top, f, cand, lane);
    }
}

// Per-stream top 4 of packed bf16 pairs (t0 >= t1 >= t2 >= t3 in each half).
__device__ __forceinline__ void ft_top4(uint32_t &t0, uint32_t &t1, uint32_t &t2, uint32_t &t3,
                                        uint32_t x)
{
    const uint32_t y1 = bf16x2_min(t0, x);
    t0 = bf16x2_max(t0, x);
    const uint32_t y2 = bf16x2_min(t1, y1);
    t1 = bf16x2_max(t1, y1);
    t3 = bf16x2_max(t3, bf16x2_min(t2, y2));
    t2 = bf16x2_max(t2, y2);
}

// Compare-exchange of packed pairs: a takes the larger, b the smaller value of each half.
__device__ __forceinline__ void ft_cx(uint32_t &a, uint32_t &b)
{
    const uint32_t h = bf16x2_max(a, b);
    b = bf16x2_min(a, b);
    a = h;
}

// Per-stream top 4 after one batch of 8 new packed pairs v[0..7] (one per vector): the
// pairs are sorted, merged into two sorted quadruples (odd-even merge), the top 4 of both
// taken as a bitonic half and sorted; that list is merged into (t0 >= t1 >= t2 >= t3) the
// same way.  44 packed min / max against 56 for eight single insertions.  Returns the
// batch maximum of each half.
__device__ __forceinline__ uint32_t ft_top4_batch(uint32_t &t0, uint32_t &t1, uint32_t &t2,
                                                  uint32_t &t3, uint32_t (&v)[8])
{
    ft_cx(v[0], v[1]);
    ft_cx(v[2], v[3]);
    ft_cx(v[4], v[5]);
    ft_cx(v[6], v[7]);
    ft_cx(v[0], v[2]);
    ft_cx(v[1], v[3]);
    ft_cx(v[1], v[2]);
    ft_cx(v[4], v[6]);
    ft_cx(v[5], v[7]);
    ft_cx(v[5], v[6]);
    uint32_t c0 = bf16x2_max(v[0], v[7]), c1 = bf16x2_max(v[1], v[6]);
    uint32_t c2 = bf16x2_max(v[2], v[5]), c3 = bf16x2_max(v[3], v[4]);
    ft_cx(c0, c2);
    ft_cx(c1, c3);
    ft_cx(c0, c1);
    ft_cx(c2, c3);
    uint32_t u0 = bf16x2_max(t0, c3), u1 = bf16x2_max(t1, c2);
    uint32_t u2 = bf16x2_max(t2, c1), u3 = bf16x2_max(t3, c0);
    ft_cx(u0, u2);
    ft_cx(u1, u3);
    ft_cx(u0, u1);
    ft_cx(u2, u3);
    t0 = u0;
    t1 = u1;
    t2 = u2;
    t3 = u3;
    return c0;
}

// Sums (s, t) of one lane's batch against the reference ml = m log2 e: both values of a
// packed pair at once (d = z log2 e - ml by one packed fma, the sum and the weighted sum by
// one packed add and one packed fma).  CLAMP reads -inf as -9.97e37 (weight 0, finite d);
// without it a -inf value makes t NaN (0 * -inf).
template <bool CLAMP>
__device__ __forceinline__ void ft_batch_sums(const uint4 (&x)[kFtLoads], float ml, float &s,
                                              float &t)
{
    const uint64_t l2e2 = f32x2_pack(kFtL2e, kFtL2e), nml2 = f32x2_pack(-ml, -ml);
    uint64_t s2 = f32x2_pack(0.0f, 0.0f), t2 = s2;
#pragma unroll
    for (int q = 0; q < kFtLoads; ++q) {
        const uint32_t w[4] = {x[q].x, x[q].y, x[q].z, x[q].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t c = CLAMP ? bf16x2_max(w[k], kFtLow2) : w[k];
            const uint64_t d2 = f32x2_fma(f32x2_pack(bf16_lo(c), bf16_hi(c)), l2e2, nml2);
            float d0, d1;
            f32x2_unpack(d2, d0, d1);
            const uint64_t e2 = f32x2_pack(fast_exp2(d0), fast_exp2(d1));
            s2 = f32x2_add(s2, e2);
            t2 = f32x2_fma(e2, d2, t2);
        }
    }
    float a0, a1, b0, b1;
    f32x2_unpack(s2, a0, a1);
    f32x2_unpack(t2, b0, b1);
    s = a0 + a1;
    t = b0 + b1;
}

// Order-preserving codes of both bf16 halves of w (unsigned order of the codes = order of
// the values; -0 sits just below +0): a set sign bit flips all 16 bits, a clear one only
// the sign bit.
__device__ __forceinline__ uint32_t ft_ord2(uint32_t w)
{
    const uint32_t sg = (w >> 15) & 0x00010001u;
    return w ^ (sg * 0x7fffu + 0x80008000u);
}

// The value of a draw key (its code in the high half).
__device__ __forceinline__ float ft_unord(uint32_t key)
{
    const uint32_t o = key >> 16;
    return __uint_as_float((o ^ ((o & 0x8000u) ? 0x8000u : 0xffffu)) << 16);
}

__device__ __forceinline__ uint32_t ft_max8(const uint32_t (&k)[8])
{
    return max(max(max(k[0], k[1]), max(k[2], k[3])), max(max(k[4], k[5]), max(k[6], k[7])));
}

__device__ __forceinline__ float ft_hmax(uint32_t w) { return fmaxf(bf16_lo(w), bf16_hi(w)); }


// bf16 rows with 16-byte alignment.  Every lane has 8 streams (packed word k of its vectors,
// low or high half); each stream keeps its top 4 with packed bf16 min / max, branch-free.
// The chunk's top-16 is then drawn from the 1024 stream entries by 16 rounds of warp
// maximum.  It is the exact top-16 unless some stream's fourth value reaches the 16th value
// drawn (that stream may have dropped a fifth one above it): false is returned and the
// caller rescans the chunk for the top-16.  The statistics see -inf as the bf16 value
// -9.97e37 (weight 0 next to any finite maximum; the product with log2 e stays finite).
__device__ __forceinline__ bool ft_scan_bf16(const FtParams &p, int64_t rowb, int64_t lo,
                                             int64_t hi, int lane, FtTop &top, FtStat &st)
{
    uint32_t T0[4], T1[4], T2[4], T3[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        T0[k] = T1[k] = T2[k] = T3[k] = kFtNegInf2;
    const int64_t nv = (hi - lo) / 8;
    const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(p.logits) +
                                                       (rowb + lo) * 2);
    for (int64_t v0 = 0; v0 < nv; v0 += kFtLoads * 32) {
        uint4 x[kFtLoads];
#pragma unroll
        for (int q = 0; q < kFtLoads; ++q) {
            const int64_t v = v0 + q * 32 + lane;
            x[q] = v < nv ? __ldg(src + v) : make_uint4(kFtNegInf2, kFtNegInf2, kFtNegInf2, kFtNegInf2);
        }
        // the statistics of the lane's 64 values against the running reference st.m (the
        // first batch of a chunk takes its reference from the lane's first vector), then the
        // top-4 network of each word in place, whose batch maximum moves the reference
        if (st.m == -INFINITY)
            st.m = ft_hmax(bf16x2_max(bf16x2_max(bf16x2_max(x[0].x, x[0].y), bf16x2_max(x[0].z, x[0].w)),
                                      kFtLow2));
        float bs, bt;
        const bool full = v0 + kFtLoads * 32 <= nv;   // warp-uniform; a partial batch holds -inf
        if (full)
            ft_batch_sums<false>(x, st.m * kFtL2e, bs, bt);
        if (!full || !(bs <= 1e37f && fabsf(bt) <= 1e37f)) {
            // a -inf value (t is NaN) or values far above the reference: move the reference
            // to the batch maximum first and read -inf as -9.97e37
            uint32_t b2 = kFtLow2;
#pragma unroll
            for (int q = 0; q < kFtLoads; ++q)
                b2 = bf16x2_max(b2, bf16x2_max(bf16x2_max(x[q].x, x[q].y), bf16x2_max(x[q].z, x[q].w)));
            ft_stat_rebase(st, ft_hmax(b2));
            ft_batch_sums<true>(x, st.m * kFtL2e, bs, bt);
        }
        st.s += bs;
        st.t += bt;
        uint32_t b2 = kFtLow2;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t v[8];
#pragma unroll
            for (int q = 0; q < kFtLoads; ++q)
                v[q] = k == 0 ? x[q].x : k == 1 ? x[q].y : k == 2 ? x[q].z : x[q].w;
            b2 = bf16x2_max(b2, ft_top4_batch(T0[k], T1[k], T2[k], T3[k], v));
        }
        ft_stat_rebase(st, ft_hmax(b2));
    }
    for (int64_t e = lo + nv * 8 + lane; e < hi; e += 32) {   // fewer than 8 values
        const uint32_t b = __ldg(reinterpret_cast<const uint16_t *>(p.logits) + rowb + e);
        const uint32_t w = b | 0xff800000u;                    // (value, -inf)
        ft_top4(T0[0], T1[0], T2[0], T3[0], w);
        float f[1];
        f[0] = bf16_lo(bf16x2_max(w, kFtLow2));
        ft_stat_acc<1, false>(st, f, f[0]);
    }
    // the draw, on 32-bit keys: the order-preserving code of the value in the high half,
    // then (31 - lane, 7 - stream) so that every entry's key is unique; K0[j] is the key of
    // stream j's head (stream j = half j & 1 of word j >> 1)
    uint32_t K0[8], K1[8], K2[8], K3[8];
    const uint32_t ltag = (uint32_t)(31 - lane) << 3;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t tlo = ltag | (uint32_t)(7 - 2 * k), thi = ltag | (uint32_t)(6 - 2 * k);
        const uint32_t o0 = ft_ord2(T0[k]), o1 = ft_ord2(T1[k]), o2 = ft_ord2(T2[k]), o3 = ft_ord2(T3[k]);
        K0[2 * k] = (o0 << 16) | tlo;
        K0[2 * k + 1] = (o0 & 0xffff0000u) | thi;
        K1[2 * k] = (o1 << 16) | tlo;
        K1[2 * k + 1] = (o1 & 0xffff0000u) | thi;
        K2[2 * k] = (o2 << 16) | tlo;
        K2[2 * k + 1] = (o2 & 0xffff0000u) | thi;
        K3[2 * k] = (o3 << 16) | tlo;
        K3[2 * k + 1] = (o3 & 0xffff0000u) | thi;
    }
    const uint32_t fourth = ft_max8(K3);   // before any entry is drawn
    uint32_t head = ft_max8(K0), kmax = 0, slot = 0;
#pragma unroll 1
    for (int rnd = 0; rnd < kFtTop; ++rnd) {
        kmax = __reduce_max_sync(0xffffffffu, head);
        if (lane == rnd)
            slot = kmax;
        if (head == kmax) {   // the one lane holding the drawn entry: its stream moves up
            switch (7 - (int)(kmax & 7u)) {
#define FT_POP(J)                                                                          \
    case J:                                                                                \
        K0[J] = K1[J];                                                                     \
        K1[J] = K2[J];                                                                     \
        K2[J] = K3[J];                                                                     \
        K3[J] = 0u;                                                                        \
        break;
                FT_POP(0) FT_POP(1) FT_POP(2) FT_POP(3) FT_POP(4) FT_POP(5) FT_POP(6) FT_POP(7)
#undef FT_POP
            }
            head = ft_max8(K0);
        }
    }
    if (lane < kFtTop)
        top.slot = ft_unord(slot);
    top.tau = ft_unord(kmax);
    // exact unless a stream's fourth entry reaches the 16th drawn value
    return __ballot_sync(0xffffffffu, (fourth >> 16) >= (kmax >> 16)) == 0;
}

// Top-16 of a row from its chunks' sorted top-16 lists (kFtPart floats apart): lane l holds
// list l of a batch of 31 (lane 31 the top-16 so far), and 16 rounds of warp maximum (one
// redux on the heads' order codes) draw the next batch top-16; the lowest lane holding the
// maximum gives up its head.
__device__ __forceinline__ void ft_merge_lists(const float *lists, int32_t nl, int lane, FtTop &top)
{
    for (int32_t b0 = 0; b0 < nl; b0 += 31) {
        float l[kFtTop];
        const int32_t q = b0 + lane;
#pragma unroll
        for (int k = 0; k < kFtTop; ++k) {
            const float run = __shfl_sync(0xffffffffu, top.slot, k);
            l[k] = lane == 31 ? run : (lane < 31 && q < nl ? __ldcg(lists + (int64_t)q * kFtPart + k) : -INFINITY);
        }
        uint32_t kmax = 0;
#pragma unroll 1
        for (int rnd = 0; rnd < kFtTop; ++rnd) {
            const uint32_t key = ft_ord32(l[0]);
            kmax = __reduce_max_sync(0xffffffffu, key);
            if (lane == rnd)
                top.slot = ft_unord32(kmax);
            const uint32_t win = __ballot_sync(0xffffffffu, key == kmax);
            if (lane == __ffs(win) - 1) {
#pragma unroll
                for (int k = 0; k < kFtTop - 1; ++k)
                    l[k] = l[k + 1];
                l[kFtTop - 1] = -INFINITY;
            }
        }
        top.tau = ft_unord32(kmax);
    }
}

template <int DT>
__global__ void __launch_bounds__(kFtThreads, 3) features_kernel(const FtParams p)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp_g = ((int64_t)blockIdx.x * kFtThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kFtThreads) >> 5;
    const int64_t units = (int64_t)p.rows * p.chunks;
    const bool vec_ok = ((p.row_stride * (DT == 1 ? 2 : 4)) & 15) == 0 &&
                        (reinterpret_cast<uintptr_t>(p.logits) & 15) == 0;
    for (int64_t u = warp_g; u < units; u += nwarps) {
        const int32_t r = (int32_t)(u / p.chunks), ch = (int32_t)(u - (int64_t)r * p.chunks);
        const int64_t lo = (int64_t)ch * p.chunk;
        const int64_t hi = lo + p.chunk < p.vocab ? lo + p.chunk : p.vocab;
        const int64_t rowb = (int64_t)r * p.row_stride;
        FtTop top;
        ft_top_init(top);
        FtStat st;
        ft_stat_init(st);
        if (DT == 1 && vec_ok) {
            if (!ft_scan_bf16(p, rowb, lo, hi, lane, top, st)) {
                // rare: rescan the chunk for its exact top-16, taking only values at or
                // above the 16th drawn one (a lower bound of the true 16th)
                const float v16 = top.tau;
                ft_top_init(top);
                if (v16 != -INFINITY)
                    top.floor = top.tau = nextafterf(v16, -INFINITY);
                ft_scan_generic<DT, false>(p, rowb, lo, hi, vec_ok, lane, top, st);
            }
        } else {
            ft_scan_generic<DT, true>(p, rowb, lo, hi, vec_ok, lane, top, st);
        }
        ft_stat_warp(st);
        if (p.chunks == 1) {
            ft_write(p, r, top, st, lane);
            continue;
        }
        int last = 0;
        {
            float *pp = p.partial + u * kFtPart;
            if (lane < kFtTop)
                pp[lane] = top.slot;
            if (lane == 0) {
                pp[16] = st.m;
                pp[17] = st.s;
                pp[18] = st.t;
            }
            __syncwarp();   // every lane's partial stores before lane 0's release
            if (lane == 0)
                last = ticket_add_acq_rel(p.tickets + r, 1) == p.chunks - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __syncwarp();   // lane 0's acquire orders the other lanes' reads
            FtTop mg;
            ft_top_init(mg);
            ft_merge_lists(p.partial + (int64_t)r * p.chunks * kFtPart, p.chunks, lane, mg);
            FtStat ms;
            ft_stat_init(ms);
            for (int32_t q = lane; q < p.chunks; q += 32) {
                const float *pp = p.partial + ((int64_t)r * p.chunks + q) * kFtPart;
                ft_stat_merge(ms, __ldcg(pp + 16), __ldcg(pp + 17), __ldcg(pp + 18));
            }
            ft_stat_warp(ms);
            ft_write(p, r, mg, ms, lane);
            // the row's partials go back to zero with its ticket: the workspace is all zero
            // after every call, so it can serve later calls with other row counts and vocabularies
            __syncwarp();   // every lane's reads of them first
            float *rp = p.partial + (int64_t)r * p.chunks * kFtPart;
            for (int32_t x = lane; x < p.chunks * kFtPart; x += 32)
                rp[x] = 0.0f;
            if (lane == 0)
                p.tickets[r] = 0;
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

// Chunk size: every row gets floor(resident warps / rows) chunks (at least one, at most
// kFtMaxChunks), so that the units fill the resident warps at most once; chunks are
// multiples of kFtChunkMin.
static int32_t ft_chunk(int32_t rows, int32_t vocab, int sms)
{
    const int64_t warps = (int64_t)sms * kFtWarpsPerSm;
    int64_t per_row = rows > 0 ? warps / rows : 1;
    per_row = per_row < 1 ? 1 : (per_row > kFtMaxChunks ? kFtMaxChunks : per_row);
    int64_t c = ((int64_t)vocab + per_row - 1) / per_row;
    c = (c + kFtChunkMin - 1) / kFtChunkMin * kFtChunkMin;
    return (int32_t)c;
}

static void ft_plan(int32_t rows, int32_t vocab, size_t &off_tk, size_t &off_part, size_t &bytes)
{
    const int64_t max_chunks = ((int64_t)vocab + kFtChunkMin - 1) / kFtChunkMin;
    off_tk = kWsHeader;
    off_part = (off_tk + (size_t)rows * 4 + 255) / 256 * 256;
    bytes = off_part + (size_t)rows * (max_chunks < kFtMaxChunks ? max_chunks : kFtMaxChunks) *
                           kFtPart * sizeof(float);
}

}  // namespace svp

extern "C" svp_status svp_draft_features_workspace_size(int32_t rows, int32_t vocab,
                                                        size_t *bytes)
{
    using namespace svp;
    if (!bytes || rows < 0 || vocab < kFtTop)
        return SVP_EINVAL;
    size_t a, b;
    ft_plan(rows, vocab, a, b, *bytes);
    return SVP_OK;
}

extern "C" svp_status svp_draft_features(const void *logits, int64_t row_stride, int32_t rows,
                                         int32_t vocab, svp_dtype dtype, float *features,
                                         void *ws, size_t ws_bytes, void *stream)
{
    using namespace svp;
    if (!logits || !features || rows < 0 || vocab < kFtTop || row_stride < vocab)
        return SVP_EINVAL;
    if (dtype != SVP_BF16 && dtype != SVP_F32)
        return SVP_EUNSUPPORTED;
    FtParams p;
    size_t off_tk, off_part, need;
    ft_plan(rows, vocab, off_tk, off_part, need);
    if (!ws || ws_bytes < need)
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
    p.chunk = ft_chunk(rows, vocab, sms);
    p.chunks = (vocab + p.chunk - 1) / p.chunk;
    const int64_t units = (int64_t)rows * p.chunks;
    int64_t grid = (units + (kFtThreads / 32) - 1) / (kFtThreads / 32);
    if (grid > (int64_t)sms * (kFtWarpsPerSm * 32 / kFtThreads))
        grid = (int64_t)sms * (kFtWarpsPerSm * 32 / kFtThreads);
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
