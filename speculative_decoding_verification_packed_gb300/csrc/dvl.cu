// dvl.cu -- DVL budget allocator and flat-buffer packer in one thread block.
//
// "DScale: Scaling Block-Diffusion Speculative Decoding with Adaptive Verification",
// SIII-C (Budget allocator, Flat-buffer packer, Algorithm 1, Fig. 6): the slot counts k_i
// of a batch of requests are adjusted to a shared budget from per-position acceptance
// scores, then token ids, positions and KV references are packed at prefix-sum offsets.
// The page runs the adjustment as one block, without host round trips or grid-wide
// synchronisation; so does this kernel.
//
// The page's loop adds the best next slot (or drops the worst last slot) one at a time.
// Prefix scores are non-increasing along a request, so that loop takes the |delta| best
// next slots (worst last slots) of the whole batch in the order (score, request, slot):
// this kernel finds the |delta|-th key of that order with a byte-wise radix selection over
// the score bits and gives every request its share, with ties at the threshold going to
// the lowest request index, which is the loop's tie rule.
#include <cstdint>
#include <cuda_runtime.h>

#include "svp_device.cuh"

namespace svp {

constexpr int kDvlThreads = 1024;
constexpr int kDvlMaxRequests = 2048;
constexpr int kDvlMaxW = 16;
constexpr int kDvlRow = kDvlMaxW + 1;   // row stride of the score table: one request per bank step

struct DvlParams {
    const float *scores;        // [n_bs, w-1]
    const int32_t *n_live;      // device scalar or nullptr (all live)
    const int32_t *tokens, *positions, *kv_refs;    // [n_bs, w] or nullptr
    int32_t n_bs, w, budget_per_req, m_cap;
    int32_t fill_token, fill_pos, fill_ref;
    int32_t *k_init, *k_out, *cu_slots;             // [n_bs], [n_bs], [n_bs + 1]
    int32_t *tokens_packed, *pos_packed, *ref_packed;   // [m_cap] or nullptr
    int32_t *n_adjust;          // device scalar or nullptr
    int32_t *status;
};

// Order-preserving map of a float to uint32 (-0 is folded into +0 first).
__device__ __forceinline__ uint32_t dvl_key(float v)
{
    const uint32_t b = __float_as_uint(v + 0.0f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct DvlShared {
    int32_t k0[kDvlMaxRequests];
    int32_t cnt[kDvlMaxRequests];     // slots strictly beyond the threshold key, per request
    int32_t eq[kDvlMaxRequests];      // slots equal to the threshold key, per request
    int32_t cu[kDvlMaxRequests + 1];
    int32_t hist[256];
    int32_t warp_tot[32];
    int32_t bcast[4];
    float q[kDvlMaxRequests * kDvlRow];    // prefix scores, row stride kDvlRow (no bank conflicts
                                           // when threads walk one request each)
};

// Sum over the block (every thread gets the result).
__device__ int32_t dvl_block_sum(int32_t v, DvlShared &sh)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if (lane == 0)
        sh.warp_tot[warp] = v;
    __syncthreads();
    int32_t t = lane < (int)(blockDim.x >> 5) ? sh.warp_tot[lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

// Exclusive prefix sum of a[0..n) in place (n <= 2 * blockDim.x); returns the total.
__device__ int32_t dvl_block_scan(int32_t *a, int n, DvlShared &sh)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int i0 = 2 * threadIdx.x;
    const int32_t x0 = i0 < n ? a[i0] : 0, x1 = i0 + 1 < n ? a[i0 + 1] : 0;
    int32_t incl = x0 + x1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    __syncthreads();
    if (lane == 31)
        sh.warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int32_t t = lane < (int)(blockDim.x >> 5) ? sh.warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o)
                t += y;
        }
        sh.warp_tot[lane] = t;   // inclusive over warps
    }
    __syncthreads();
    const int32_t before = (warp > 0 ? sh.warp_tot[warp - 1] : 0) + incl - x0 - x1;
    const int32_t total = sh.warp_tot[31];
    if (i0 < n)
        a[i0] = before;
    if (i0 + 1 < n)
        a[i0 + 1] = before + x0;
    __syncthreads();
    return total;
}

// Slots j in [lo_i, hi_i) of live request i are the candidates; `grow` selects the `need`
// largest keys (score, then lowest request, then lowest slot), otherwise the `need`
// smallest scores (lowest request first, then highest slot).  Leaves per request the
// count of selected slots in sh.cnt.
__device__ void dvl_select(DvlShared &sh, int n_live, int w, bool grow, int32_t need)
{
    const int tid = threadIdx.x;
    auto lo = [&](int i) { return grow ? sh.k0[i] : 1; };
    auto hi = [&](int i) { return grow ? w : sh.k0[i]; };
    auto key = [&](int i, int j) {
        const uint32_t k = dvl_key(sh.q[i * kDvlRow + j]);
        return grow ? k : ~k;                   // selection of the largest keys
    };
    uint32_t prefix = 0, mask = 0;
    int32_t m = need;                           // rank of the threshold key, from the top
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = tid; b < 256; b += blockDim.x)
            sh.hist[b] = 0;
        __syncthreads();
        if (n_live * w > 2 * (int)blockDim.x) {
            // many requests: one request per thread
            for (int i = tid; i < n_live; i += blockDim.x)
                for (int j = lo(i); j < hi(i); ++j) {
                    const uint32_t k = key(i, j);
                    if ((k & mask) == prefix)
                        atomicAdd(&sh.hist[(k >> shift) & 255u], 1);
                }
        } else
        // few requests: one (request, slot) pair per thread, and lanes that hit the same
        // bucket add together (keys crowd into a few buckets; same-address atomics serialise)
        for (int c = tid; c < n_live * w; c += blockDim.x) {
            const int i = c / w, j = c - i * w;
            bool hit = false;
            uint32_t bucket = 0;
            if (j >= lo(i) && j < hi(i)) {
                const uint32_t k = key(i, j);
                hit = (k & mask) == prefix;
                bucket = (k >> shift) & 255u;
            }
            const uint32_t act = __ballot_sync(__activemask(), hit);
            if (hit) {
                const uint32_t peers = __match_any_sync(act, bucket);
                if ((tid & 31) == __ffs(peers) - 1)
                    atomicAdd(&sh.hist[bucket], __popc(peers));
            }
        }
        __syncthreads();
        if (tid < 32) {
            // lane L owns buckets 255-8L .. 248-8L, scanned from the top
            int32_t c[8], s = 0;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                c[e] = sh.hist[255 - 8 * tid - e];
                s += c[e];
            }
            int32_t incl = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o)
                    incl += y;
            }
            const bool here = incl >= m && incl - s < m;
            if (here) {
                int32_t acc = incl - s;
                int e = 0;
                while (e < 7 && acc + c[e] < m) {
                    acc += c[e];
                    ++e;
                }
                sh.bcast[0] = 255 - 8 * tid - e;   // digit of the threshold key
                sh.bcast[1] = m - acc;             // its rank among keys with that digit
            }
        }
        __syncthreads();
        prefix |= (uint32_t)sh.bcast[0] << shift;
        mask |= 255u << shift;
        m = sh.bcast[1];
        __syncthreads();
    }
    // per request: keys above the threshold, and keys equal to it
    for (int i = tid; i < n_live; i += blockDim.x) {
        int32_t gt = 0, eq = 0;
        for (int j = lo(i); j < hi(i); ++j) {
            const uint32_t k = key(i, j);
            gt += k > prefix;
            eq += k == prefix;
        }
        sh.cnt[i] = gt;
        sh.eq[i] = eq;
    }
    __syncthreads();
    int32_t my_gt = 0;
    for (int i = tid; i < n_live; i += blockDim.x)
        my_gt += sh.cnt[i];
    const int32_t g_total = dvl_block_sum(my_gt, sh);
    dvl_block_scan(sh.eq, n_live, sh);          // equal keys in earlier requests
    const int32_t ties = need - g_total;       // taken from the lowest requests
    for (int i = tid; i < n_live; i += blockDim.x) {
        int32_t e_i = 0;
        for (int j = lo(i); j < hi(i); ++j)
            e_i += key(i, j) == prefix;
        const int32_t share = min(max(ties - sh.eq[i], 0), e_i);
        sh.cnt[i] += share;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kDvlThreads, 1) dvl_kernel(const DvlParams p)
{
    griddep_launch_dependents();
    griddep_wait();
    extern __shared__ __align__(16) uint8_t dvl_smem[];
    DvlShared &sh = *reinterpret_cast<DvlShared *>(dvl_smem);
    const int tid = threadIdx.x;
    const int n_bs = p.n_bs, w = p.w;
    int32_t n_live = p.n_live ? *p.n_live : n_bs;
    const int64_t budget64 = (int64_t)p.budget_per_req * n_live;
    const bool bad = n_live < 0 || n_live > n_bs || budget64 > p.m_cap;
    if (bad) {
        if (tid == 0)
            set_status(p.status, SVP_DEV_BAD_SLOTS);
        n_live = 0;
    }
    const int32_t budget = bad ? 0 : (int32_t)budget64;

    // the scores, staged with coalesced loads (one memory round trip, not w - 1 of them)
    for (int e = tid; e < n_bs * (w - 1); e += blockDim.x) {
        const int i = e / (w - 1), j = e - i * (w - 1) + 1;
        sh.q[i * kDvlRow + j] = __ldg(p.scores + e);
    }
    __syncthreads();
    // prefix scores (cumulative minimum after the anchor's 1) and initial lengths
    for (int i = tid; i < n_bs; i += blockDim.x) {
        float qv = 1.0f, acc = 0.0f;
        sh.q[i * kDvlRow] = 1.0f;
        for (int j = 1; j < w; ++j) {
            qv = fminf(qv, sh.q[i * kDvlRow + j]);
            sh.q[i * kDvlRow + j] = qv;
            acc = __fadd_rn(acc, qv);
        }
        int32_t k0 = 0;
        if (i < n_live)
            k0 = min(max((int32_t)rintf(acc), 1), w);
        sh.k0[i] = k0;
        if (p.k_init)
            p.k_init[i] = k0;
    }
    __syncthreads();
    int32_t my = 0;
    for (int i = tid; i < n_live; i += blockDim.x)
        my += sh.k0[i];
    const int32_t delta = budget - dvl_block_sum(my, sh);

    // grow (delta > 0) or shrink (delta < 0) to the budget
    const bool grow = delta > 0;
    int32_t cand = 0;
    for (int i = tid; i < n_live; i += blockDim.x)
        cand += grow ? w - sh.k0[i] : sh.k0[i] - 1;
    const int32_t avail = dvl_block_sum(cand, sh);
    const int32_t need = min(grow ? delta : -delta, avail);
    for (int i = tid; i < n_bs; i += blockDim.x)
        sh.cnt[i] = 0;
    __syncthreads();
    if (need > 0)
        dvl_select(sh, n_live, w, grow, need);
    for (int i = tid; i < n_bs; i += blockDim.x) {
        const int32_t k = i < n_live ? sh.k0[i] + (grow ? sh.cnt[i] : -sh.cnt[i]) : 0;
        sh.cu[i] = k;
        p.k_out[i] = k;
    }
    if (tid == 0 && p.n_adjust)
        *p.n_adjust = need;
    __syncthreads();

    // offsets, then the row-mapped fields and the tail placeholders
    const int32_t end = dvl_block_scan(sh.cu, n_bs, sh);
    if (tid == 0)
        sh.cu[n_bs] = end;
    __syncthreads();
    for (int i = tid; i <= n_bs; i += blockDim.x)
        p.cu_slots[i] = sh.cu[i];
    for (int r = tid; r < p.m_cap; r += blockDim.x) {
        int32_t t = p.fill_token, po = p.fill_pos, rf = p.fill_ref;
        if (r < end) {
            int lo = 0, hi = n_bs;   // cu[lo] <= r < cu[hi]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (sh.cu[mid] <= r)
                    lo = mid;
                else
                    hi = mid;
            }
            const int64_t src = (int64_t)lo * w + (r - sh.cu[lo]);
            if (p.tokens)
                t = __ldg(p.tokens + src);
            if (p.positions)
                po = __ldg(p.positions + src);
            if (p.kv_refs)
                rf = __ldg(p.kv_refs + src);
        }
        if (p.tokens_packed)
            p.tokens_packed[r] = t;
        if (p.pos_packed)
            p.pos_packed[r] = po;
        if (p.ref_packed)
            p.ref_packed[r] = rf;
    }
}

}  // namespace svp

extern "C" svp_status svp_dvl_allocate_pack(const float *scores, int32_t n_bs, int32_t w,
                                            const int32_t *n_live, int32_t budget_per_req,
                                            const int32_t *tokens, const int32_t *positions,
                                            const int32_t *kv_refs, int32_t m_cap,
                                            int32_t fill_token, int32_t fill_pos,
                                            int32_t fill_ref, int32_t *k_init, int32_t *k_out,
                                            int32_t *cu_slots, int32_t *tokens_packed,
                                            int32_t *pos_packed, int32_t *ref_packed,
                                            int32_t *n_adjust, void *ws, size_t ws_bytes,
                                            void *stream)
{
    using namespace svp;
    if (!scores || !k_out || !cu_slots || n_bs < 1 || w < 2 || m_cap < 1 ||
        budget_per_req < 1 || budget_per_req > w)
        return SVP_EINVAL;
    if (n_bs > kDvlMaxRequests || w > kDvlMaxW)
        return SVP_EUNSUPPORTED;
    if (!ws || ws_bytes < kWsHeader)
        return SVP_EWORKSPACE;
    static std::atomic<uint64_t> configured{0};
    if (set_smem_limit_once(dvl_kernel, (int)sizeof(DvlShared), configured) != cudaSuccess)
        return SVP_ECUDA;
    DvlParams p;
    p.scores = scores;
    p.n_live = n_live;
    p.tokens = tokens;
    p.positions = positions;
    p.kv_refs = kv_refs;
    p.n_bs = n_bs;
    p.w = w;
    p.budget_per_req = budget_per_req;
    p.m_cap = m_cap;
    p.fill_token = fill_token;
    p.fill_pos = fill_pos;
    p.fill_ref = fill_ref;
    p.k_init = k_init;
    p.k_out = k_out;
    p.cu_slots = cu_slots;
    p.tokens_packed = tokens_packed;
    p.pos_packed = pos_packed;
    p.ref_packed = ref_packed;
    p.n_adjust = n_adjust;
    p.status = static_cast<int32_t *>(ws);
    // small batches (at most one candidate slot per thread of a quarter block) run a quarter
    // block: every loop of the kernel strides by the block size, and fewer warps meet at
    // each of its barriers
    const int threads = (int64_t)n_bs * w <= kDvlThreads / 4 ? kDvlThreads / 4 : kDvlThreads;
    return launch_pdl(dvl_kernel, dim3(1), dim3(threads), sizeof(DvlShared), (cudaStream_t)stream, p) ==
                   cudaSuccess
               ? SVP_OK
               : SVP_ECUDA;
}
