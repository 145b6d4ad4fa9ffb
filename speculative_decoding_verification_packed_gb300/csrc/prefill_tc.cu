// prefill_tc.cu -- causal prefill attention on tcgen05: the WIDE tile's contrast workload
// (DScale SIII-B: prefill keeps the 128-row hardware tile, which it fills).
//
// What it computes: for each packed sequence i (rows cu_seqlens[i] .. cu_seqlens[i+1]-1)
// and query head h, row r attends to keys 0..r of the same sequence through KV head h / G,
// softmax scale `scale`; out = softmax(q k^T) v, lse = log-sum-exp of the scaled scores.
//
// Design (head_dim 128, bf16, an even number G of query heads per KV head):
//   * A work item is one 128-row query tile of two query heads that share a KV head; both
//     tiles need the same causal KV range (tiles 0..j), so one K/V stream feeds two
//     independent 128-row problems.  Items are handed out heaviest first (largest j), in a
//     snake order over the persistent CTAs (one per SM), which evens out the causal costs.
//   * Per CTA: warp 0 streams Q (two tiles per item) and 128-key K / V tiles through TMA
//     into a five-slot ring; warp 1 owns TMEM and issues the MMAs; warps 2-5 and 6-9 are the
//     softmax warpgroups of the two query tiles, one thread per query row (TMEM lane).
//   * S_a = Q_a K^T (M = 128 rows, N = 128 keys, K = 128) lands in TMEM; the softmax writes
//     P_a in bf16 over the first 64 columns of S_a, and O_a += P_a V takes P_a straight from
//     TMEM as the A operand (no shared-memory round trip).  MMAs from one thread run in
//     order, so S_a(t+1), issued after PV_a(t), overwrites S_a only once P_a(t) has been read.
//   * Issue order per KV tile t: PV_0(t), S_0(t+1), PV_1(t), S_1(t+1): the softmax of one
//     query tile runs while the tensor pipe works on the other.
//   * The exponent reference of a row is its maximum over the item's first KV tile; it is
//     moved (and O_a rescaled in TMEM by its own thread) only when a later tile's row sum of
//     2^(s - reference) exceeds 2^32, so ordinary tiles need no maximum.  The commit that
//     signals S_a(t) also covers PV_a(t-1), so O_a is stable while its thread rescales it.
//   TMEM: S_0 / P_0 [0, 128), S_1 / P_1 [128, 256), O_0 [256, 384), O_1 [384, 512).
#include <algorithm>
#include <cfloat>
#include <cstring>

#include "svp_params.cuh"

namespace svp {

constexpr int kPfThreads = 320;      // producer, MMA issuer, two softmax warpgroups
constexpr int kPfSub = 16384;        // [128 rows][64 d] bf16, 128-byte swizzled
constexpr int kPfTile = 2 * kPfSub;  // [128][128] bf16
constexpr int kPfSlots = 5;          // K / V ring slots, one tile each
constexpr int kPfMaxSeq = 16;        // sequences per launch (tables in shared memory)
constexpr int kPfMaxTiles = 256;     // query tiles per sequence (32K rows)
constexpr float kPfSumLimit = 4294967296.0f;   // 2^32: a tile row sum above it moves the reference
constexpr int kPfOffRing = 2 * kPfTile;
constexpr int kPfOffMisc = kPfOffRing + kPfSlots * kPfTile;
constexpr int kPfSmem = kPfOffMisc + 1536 + 1024;   // misc region + alignment slack

struct PfParams {
    CUtensorMap tm_q, tm_k, tm_v;    // {d, heads, total_s}, box {64, 1, 128}
    const int32_t *cu_seqlens;       // [n + 1] (device)
    int32_t n, hq, hkv, G, pairs, max_tiles;
    int32_t total_s;                 // rows of q / k / v / out
    float scale_log2;
    void *out;                       // [total_s, hq, 128] bf16
    float *lse;                      // [total_s, hq] or nullptr
    int32_t *status;
};

struct PfMisc {
    uint64_t bars[24];
    uint32_t tmem;
    int32_t abort_flag;
    int32_t nitems;
    int32_t seq_start[kPfMaxSeq];
    int32_t seq_len[kPfMaxSeq];
    int32_t jpref[kPfMaxTiles + 1];  // items with a query-tile index of j or above, j descending
    int32_t warp_tot[kPfThreads / 32];
};
static_assert(sizeof(PfMisc) <= 1536, "misc region");

struct PfItem {
    int32_t j, g, h0, row0, kv0, len;   // query tile j of rows [row0, row0 + 128), keys from kv0
};

// D[tmem] (+)= A[tmem] * B[smem], bf16 inputs, fp32 accumulate (A from tensor memory).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Largest raw score of this thread's row in one S tile (TMEM columns ts .. ts + 127); with
// kMasked, keys past kmax are hidden.
template <bool kMasked>
__device__ __forceinline__ float pf_row_max(uint32_t ts, int32_t kmax)
{
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint32_t sa[32], sb[32];
        tmem_ld32(ts + half * 64, sa);
        tmem_ld32(ts + half * 64 + 32, sb);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 64; ++e) {
            const float v = __uint_as_float(e < 32 ? sa[e] : sb[e - 32]);
            mx[e & 3] = fmaxf(mx[e & 3], (!kMasked || half * 64 + e <= kmax) ? v : -INFINITY);
        }
    }
    return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
}

// P = 2^(s * cl2 - m_ref) of this thread's row in one S tile, as 64 bf16 pairs (keys 2e and
// 2e + 1 in pk[e]), and the sum of the 128 values in fp32.
template <bool kMasked>
__device__ __forceinline__ float pf_row_exp(uint32_t ts, int32_t kmax, float cl2, float m_ref,
                                            uint32_t (&pk)[64])
{
    const uint64_t c2 = f32x2_pack(cl2, cl2), nm2 = f32x2_pack(-m_ref, -m_ref);
    uint64_t acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        acc[i] = f32x2_pack(0.0f, 0.0f);
    // all 128 scores in one round trip; each register dies as its P value is packed
    uint32_t sv[4][32];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        tmem_ld32(ts + q * 32, sv[q]);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 64; ++e) {
        const int k0 = 2 * e;
        float s0 = __uint_as_float(sv[k0 >> 5][k0 & 31]);
        float s1 = __uint_as_float(sv[k0 >> 5][(k0 & 31) + 1]);
        if (kMasked) {
            s0 = k0 <= kmax ? s0 : -INFINITY;
            s1 = k0 + 1 <= kmax ? s1 : -INFINITY;
        }
        float y0, y1;
        f32x2_unpack(f32x2_fma(f32x2_pack(s0, s1), c2, nm2), y0, y1);
        const float p0 = fast_exp2(y0), p1 = fast_exp2(y1);
        pk[e] = pack_bf16x2(p0, p1);
        acc[e & 3] = f32x2_add(acc[e & 3], f32x2_pack(p0, p1));
    }
    float a0, a1, b0, b1, c0, c1, d0, d1;
    f32x2_unpack(acc[0], a0, a1);
    f32x2_unpack(acc[1], b0, b1);
    f32x2_unpack(acc[2], c0, c1);
    f32x2_unpack(acc[3], d0, d1);
    return ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (d0 + d1));
}

// Item idx (in heaviest-first order) -> query tile, sequence, head pair.
__device__ __forceinline__ bool pf_item(const PfParams &p, const PfMisc *m, int32_t idx, PfItem &it)
{
    const int32_t nj = p.max_tiles;
    if (idx >= m->jpref[nj])
        return false;
    int32_t lo = 0, hi = nj;   // largest jj with jpref[jj] <= idx
    while (hi - lo > 1) {
        const int32_t mid = (lo + hi) >> 1;
        if (m->jpref[mid] <= idx)
            lo = mid;
        else
            hi = mid;
    }
    const int32_t j = nj - 1 - lo;
    int32_t r = idx - m->jpref[lo];
    const int32_t per_seq = p.hkv * p.pairs;
    int32_t k = r / per_seq;
    r -= k * per_seq;
    const int32_t g = r / p.pairs, pair = r - g * p.pairs;
    int32_t i = 0;
    for (; i < p.n; ++i) {
        if (m->seq_len[i] > j * 128) {
            if (k == 0)
                break;
            --k;
        }
    }
    it.j = j;
    it.g = g;
    it.h0 = g * p.G + 2 * pair;
    it.kv0 = m->seq_start[i];
    it.row0 = it.kv0 + j * 128;
    it.len = m->seq_len[i];
    return true;
}

// The idx-th item of CTA c: rounds of C items, snake order across the CTAs.
__device__ __forceinline__ int32_t pf_index(int32_t round, int32_t c, int32_t C)
{
    return round * C + ((round & 1) ? (C - 1 - c) : c);
}

__global__ void __launch_bounds__(kPfThreads, 1) prefill_tc_kernel(const __grid_constant__ PfParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    PfMisc *m = reinterpret_cast<PfMisc *>(smem + kPfOffMisc);
    const uint32_t bar0 = smem_u32(m->bars);
    auto bar_kfull = [&](int s) { return bar0 + 8u * s; };
    auto bar_kempty = [&](int s) { return bar0 + 8u * (kPfSlots + s); };
    const uint32_t bar_qfull = bar0 + 8u * 10, bar_qempty = bar0 + 8u * 11;
    auto bar_sfull = [&](int a) { return bar0 + 8u * (12 + a); };
    auto bar_pfull = [&](int a) { return bar0 + 8u * (14 + a); };
    auto bar_oready = [&](int a) { return bar0 + 8u * (16 + a); };
    auto bar_ofree = [&](int a) { return bar0 + 8u * (18 + a); };
    const uint32_t bar_drain = bar0 + 8u * 20;
    volatile int *abort_flag = &m->abort_flag;

    if (tid == 0) {
        for (int s = 0; s < kPfSlots; ++s) {
            mbar_init(bar_kfull(s), 1);
            mbar_init(bar_kempty(s), 1);
        }
        mbar_init(bar_qfull, 1);
        mbar_init(bar_qempty, 1);
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_sfull(a), 1);
            mbar_init(bar_pfull(a), 4);
            mbar_init(bar_oready(a), 1);
            mbar_init(bar_ofree(a), 4);
        }
        mbar_init(bar_drain, 1);
        mbar_fence_init();
        m->abort_flag = 0;
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&m->tmem), 512);
        tmem_relinquish();
    }
    // sequences (n <= kPfMaxSeq, host-checked); a sequence that starts before row 0, runs
    // backwards, ends past the buffer or is longer than max_s is skipped (status bit)
    if (tid < p.n) {
        const int32_t s0 = __ldg(p.cu_seqlens + tid), s1 = __ldg(p.cu_seqlens + tid + 1);
        const bool bad = s0 < 0 || s1 < s0 || s1 > p.total_s || s1 - s0 > p.max_tiles * 128;
        m->seq_start[tid] = bad ? 0 : s0;
        m->seq_len[tid] = bad ? 0 : s1 - s0;
        if (bad && blockIdx.x == 0)
            set_status(p.status, SVP_DEV_BAD_SLOTS);
    }
    __syncthreads();
    // items per query-tile index, heaviest (largest j) first: count per index, then an
    // exclusive scan (max_tiles <= 256 < the block size)
    {
        int32_t cnt = 0;
        if (tid < p.max_tiles) {
            const int32_t j = p.max_tiles - 1 - tid;
            for (int32_t i = 0; i < p.n; ++i)
                cnt += m->seq_len[i] > j * 128 ? 1 : 0;
            cnt *= p.hkv * p.pairs;
        }
        int32_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += v;
        }
        if (lane == 31)
            m->warp_tot[warp] = incl;
        __syncthreads();
        int32_t before = 0;
        for (int w2 = 0; w2 < warp; ++w2)
            before += m->warp_tot[w2];
        if (tid < p.max_tiles)
            m->jpref[tid] = before + incl - cnt;
        if (tid == p.max_tiles - 1) {
            m->jpref[p.max_tiles] = before + incl;
            m->nitems = before + incl;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = m->tmem;
    const int32_t C = (int32_t)gridDim.x, c = (int32_t)blockIdx.x;

    if (warp == 0) {
        // ============================================================ TMA producer
        if (lane == 0) {
            uint32_t kvs = 0, nitem = 0;
            bool ok = true;
            const uint64_t pol = l2_policy_evict_last();   // K / V are re-read by later items
            PfItem it;
            for (int32_t round = 0; ok && pf_item(p, m, pf_index(round, c, C), it); ++round, ++nitem) {
                if (nitem > 0 && !(ok = mbar_wait(bar_qempty, (nitem - 1) & 1u, abort_flag)))
                    break;
                mbar_arrive_expect_tx(bar_qfull, 2u * kPfTile);
                for (int a = 0; a < 2; ++a)
                    for (int cc = 0; cc < 2; ++cc)
                        tma_load_3d(sbase + a * kPfTile + cc * kPfSub, &p.tm_q, bar_qfull, cc * 64,
                                    it.h0 + a, it.row0);
                for (int32_t t = 0; t <= it.j && ok; ++t) {
                    for (int kv = 0; kv < 2; ++kv, ++kvs) {
                        const int sl = (int)(kvs % kPfSlots);
                        if (!(ok = mbar_wait(bar_kempty(sl), ((kvs / kPfSlots) & 1u) ^ 1u, abort_flag)))
                            break;
                        mbar_arrive_expect_tx(bar_kfull(sl), (uint32_t)kPfTile);
                        const CUtensorMap *tm = kv ? &p.tm_v : &p.tm_k;
                        for (int cc = 0; cc < 2; ++cc)
                            tma_load_3d_hint(sbase + kPfOffRing + sl * kPfTile + cc * kPfSub, tm,
                                             bar_kfull(sl), cc * 64, it.g, it.kv0 + t * 128, pol);
                    }
                }
            }
            volatile int drain = 0;
            const uint32_t first = kvs > (uint32_t)kPfSlots ? kvs - kPfSlots : 0u;
            if (!ok) {
                // the loads already issued land before the CTA exits
                for (uint32_t k = first; k < kvs; ++k)
                    mbar_wait(bar_kfull((int)(k % kPfSlots)), (k / kPfSlots) & 1u, &drain);
                if (nitem > 0)
                    mbar_wait(bar_qfull, (nitem - 1) & 1u, &drain);
            } else {
                // tail: the releases of the last slots and of Q have landed
                for (uint32_t k = first; k < kvs; ++k)
                    mbar_wait(bar_kempty((int)(k % kPfSlots)), (k / kPfSlots) & 1u, abort_flag);
                if (nitem > 0)
                    mbar_wait(bar_qempty, (nitem - 1) & 1u, abort_flag);
            }
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
            const uint32_t idesc_o = idesc_bf16_f32(128, 128, false, true);
            uint32_t kvs = 0, nitem = 0, it_g = 0;
            bool ok = true;
            PfItem it;
            auto slot_addr = [&](uint32_t pos) { return sbase + kPfOffRing + (pos % kPfSlots) * kPfTile; };
            auto wait_full = [&](uint32_t pos) {
                return mbar_wait(bar_kfull((int)(pos % kPfSlots)), (pos / kPfSlots) & 1u, abort_flag);
            };
            auto issue_s = [&](int a, uint32_t kpos) {
                const uint64_t qd = sw128_desc(sbase + a * kPfTile, 16, 1024);
                const uint64_t kd = sw128_desc(slot_addr(kpos), 16, 1024);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    tc_mma_ss(tmem + a * 128,
                              qd + (uint64_t)((ks >> 2) * (kPfSub >> 4) + (ks & 3) * 2),
                              kd + (uint64_t)((ks >> 2) * (kPfSub >> 4) + (ks & 3) * 2), idesc_s,
                              ks ? 1u : 0u);
                tc_commit(bar_sfull(a));
            };
            for (int32_t round = 0; ok && pf_item(p, m, pf_index(round, c, C), it); ++round, ++nitem) {
                if (!(ok = mbar_wait(bar_qfull, nitem & 1u, abort_flag)))
                    break;
                if (!(ok = wait_full(kvs)))
                    break;
                tc_fence_after();
                issue_s(0, kvs);
                issue_s(1, kvs);
                tc_commit(bar_kempty((int)(kvs % kPfSlots)));   // K(0) read by both
                if (it.j == 0)
                    tc_commit(bar_qempty);
                for (int32_t t = 0; t <= it.j && ok; ++t, ++it_g) {
                    const uint32_t kpos = kvs + 2u * t, vpos = kpos + 1u;
                    for (int a = 0; a < 2 && ok; ++a) {
                        if (!(ok = mbar_wait(bar_pfull(a), it_g & 1u, abort_flag)))
                            break;
                        if (t == 0 && nitem > 0 && !(ok = mbar_wait(bar_ofree(a), (nitem - 1) & 1u, abort_flag)))
                            break;
                        if (a == 0 && !(ok = wait_full(vpos)))
                            break;
                        tc_fence_after();
                        const uint64_t vd = sw128_desc(slot_addr(vpos), kPfSub, 1024);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)   // 16 keys = 8 TMEM columns of P per MMA
                            tc_mma_ts(tmem + 256 + a * 128, tmem + a * 128 + ks * 8,
                                      vd + (uint64_t)(ks * 128), idesc_o, (t | ks) ? 1u : 0u);
                        if (t == it.j)
                            tc_commit(bar_oready(a));
                        if (a == 1)
                            tc_commit(bar_kempty((int)(vpos % kPfSlots)));   // V(t) read by both
                        if (t < it.j) {
                            if (a == 0 && !(ok = wait_full(kpos + 2u)))
                                break;
                            tc_fence_after();
                            issue_s(a, kpos + 2u);
                            if (a == 1) {
                                tc_commit(bar_kempty((int)((kpos + 2u) % kPfSlots)));
                                if (t + 1 == it.j)
                                    tc_commit(bar_qempty);
                            }
                        }
                    }
                }
                kvs += 2u * (uint32_t)(it.j + 1);
            }
            tc_commit(bar_drain);
            volatile int drain = 0;
            mbar_wait(bar_drain, 0, &drain);
        }
    } else {
        // ============================================================ softmax warpgroups
        const int a = (warp - 2) >> 2;                   // query tile of this warpgroup
        const int quarter = warp & 3;                     // TMEM lane quarter of this warp
        const int r = quarter * 32 + lane;                // query row within the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t ts = tmem + lane_off + a * 128;           // S_a / P_a
        const uint32_t to = tmem + lane_off + 256 + a * 128;     // O_a
        const float cl2 = p.scale_log2;
        uint32_t it_g = 0, nitem = 0;
        bool ok = true;
        PfItem it;
        for (int32_t round = 0; ok && pf_item(p, m, pf_index(round, c, C), it); ++round, ++nitem) {
            const int32_t qrow = it.j * 128 + r;               // row index within the sequence
            float m_ref = -INFINITY, l = 0.0f;
            for (int32_t t = 0; t <= it.j; ++t, ++it_g) {
                // warp-uniform outcome: the TMEM accesses below are warp-collective
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_sfull(a), it_g & 1u, abort_flag))))
                    break;
                tc_fence_after();
                // Keys hidden from this row (past it, or past the sequence) only occur in the
                // diagonal tile and in the sequence's last tile; elsewhere the scores are used as
                // they are.  Raw scores are used: the scale is positive, so the maximum of the
                // scaled scores is the scaled maximum, and 2^(s c - m) is one fma.  P is taken
                // against the reference m_ref in one pass over the scores; the reference is set to
                // the row maximum on the item's first tile, and moved later only when a tile's row
                // sum exceeds 2^32 (some score then lies more than 2^25 above it): O_a and l are
                // rescaled and the tile is recomputed against the larger of the two.
                const bool masked = !(t < it.j && (t + 1) * 128 <= it.len);
                const int32_t kmax = masked ? min(qrow, it.len - 1) - t * 128 : 127;   // last visible key
                uint32_t pk[64];
                float tsum;
                bool move = (t == 0);
#pragma unroll 1
                for (;;) {
                    if (move) {
                        // (m_ref is -inf on the first tile; later it only grows)
                        const float tmax = fmaxf(m_ref, (masked ? pf_row_max<true>(ts, kmax)
                                                                : pf_row_max<false>(ts, kmax)) * cl2);
                        if (t > 0) {
                            const float alpha = fast_exp2(m_ref - tmax);
#pragma unroll 1
                            for (int cc = 0; cc < 4; ++cc) {
                                uint32_t ov[32];
                                tmem_ld32(to + cc * 32, ov);
                                tmem_wait_ld();
#pragma unroll
                                for (int e = 0; e < 32; ++e)
                                    ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                                tmem_st32(to + cc * 32, ov);
                            }
                            l *= alpha;
                        }
                        m_ref = tmax;
                    }
                    tsum = masked ? pf_row_exp<true>(ts, kmax, cl2, m_ref, pk)
                                  : pf_row_exp<false>(ts, kmax, cl2, m_ref, pk);
                    // tcgen05.ld / st are warp-collective (.sync.aligned): the warp takes the
                    // move together when any of its rows needs it (NaN sums included)
                    if (move || !__any_sync(0xffffffffu, !(tsum <= kPfSumLimit)))
                        break;
                    move = true;
                }
                // P over columns [0, 64) of S_a, in bf16 (the scores there have been read)
                tmem_st32(ts, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
                tmem_st32(ts + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
                l += tsum;
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar_pfull(a));
            }
            if (!ok)
                break;
            // ---- epilogue: O_a complete after the item's last PV_a
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar_oready(a), nitem & 1u, abort_flag))))
                break;
            tc_fence_after();
            const float inv = 1.0f / l;
            const bool live = qrow < it.len;
            const int32_t h = it.h0 + a;
            uint16_t *orow = reinterpret_cast<uint16_t *>(p.out) +
                             ((int64_t)(it.row0 + r) * p.hq + h) * 128;
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t ov[32];
                tmem_ld32(to + cc * 32, ov);
                tmem_wait_ld();
                if (live) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
            if (live && p.lse)
                p.lse[(int64_t)(it.row0 + r) * p.hq + h] = (m_ref + __log2f(l)) * 0.69314718055994531f;
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar_ofree(a));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // read once every role has finished, so that a wait given up late is reported too
    if (*abort_flag && tid == 0)
        set_status(p.status, SVP_DEV_TIMEOUT);
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------------ host side
bool prefill_tc_supported(int32_t n, int32_t max_s, int32_t hq, int32_t hkv, int32_t d)
{
    return d == 128 && hkv > 0 && hq % hkv == 0 && (hq / hkv) % 2 == 0 && n >= 1 &&
           n <= kPfMaxSeq && max_s >= 1 && (max_s + 127) / 128 <= kPfMaxTiles;
}

svp_status prefill_tc_launch(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                             const int32_t *cu_seqlens, int32_t n, int32_t max_s, int32_t total_s,
                             int32_t hq, int32_t hkv, float scale_log2, void *out, float *lse,
                             int32_t *status, int grid, cudaStream_t stream)
{
    PfParams p;
    std::memset(&p, 0, sizeof p);
    p.tm_q = tm_q;
    p.tm_k = tm_k;
    p.tm_v = tm_v;
    p.cu_seqlens = cu_seqlens;
    p.n = n;
    p.hq = hq;
    p.hkv = hkv;
    p.G = hq / hkv;
    p.pairs = p.G / 2;
    p.max_tiles = (max_s + 127) / 128;
    p.total_s = total_s;
    p.scale_log2 = scale_log2;
    p.out = out;
    p.lse = lse;
    p.status = status;
    static std::atomic<uint64_t> configured{0};
    if (set_smem_limit_once(prefill_tc_kernel, kPfSmem, configured) != cudaSuccess)
        return SVP_ECUDA;
    const int64_t items = (int64_t)p.max_tiles * n * hkv * p.pairs;   // an upper bound
    const int g = (int)std::min<int64_t>(grid, std::max<int64_t>(items, 1));
    prefill_tc_kernel<<<g, kPfThreads, kPfSmem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? SVP_OK : SVP_ECUDA;
}

}  // namespace svp
