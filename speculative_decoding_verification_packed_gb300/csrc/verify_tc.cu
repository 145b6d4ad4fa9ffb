// verify_tc.cu -- GQA-packed short-tile verification attention on tcgen05, in the
// transposed ("keys on lanes") form.
//
// What it computes is the same as attn_tc.cu (DScale SIII-D: row j of request i sees
// the request's context, then its own candidates 0..j; query head h reads KV head
// h / G), for the SHORT tile: the G query heads of one KV head and R candidate rows
// each form one query tile of G*R <= 128 rows (DScale SIII-B: the tile follows the
// candidate width, here times the GQA group).
//
// Why transposed: a verification tile has only G*k live rows (32..96 in the target
// workloads).  With rows on TMEM lanes most lanes idle and each softmax thread walks
// every key of a tile.  Here the 128 keys of a KV tile are the MMA M dimension:
//   S^T  = K Q^T     M=128 keys, N=rows, K=d            (TMEM, double buffered)
//   O^T += V^T P^T   M=128 d,    N=rows, K=keys         (TMEM, one per 128 columns of d)
//   l^T += 1 P^T     M=128,      N=rows, K=keys         (row sums on the tensor core)
// Every softmax thread owns one key and touches only the live rows.  The running
// maximum of each row is a stale reference m_ref: P = 2^(s*c - m_ref) is used while
// no visible score exceeds m_ref + 8; only then (and on the first tile of a piece) the
// softmax warps reduce the row maxima across keys, move m_ref, and rescale O^T and l^T
// in TMEM.  Inactive rows carry m_ref = +inf, so their P is 0 without per-element
// masks.
//
// Pipeline: warp 0 issues TMA into a ring of 32 KB slots ([128 keys][128 d] halves of
// K, then of V), warp 1 owns TMEM and issues tcgen05.mma from one thread, warps 2..5
// (one per TMEM lane quarter) run the softmax and the epilogue.  K slots are released
// as soon as S^T is done, V slots after PV.  Work split, partials and the last-arrival
// combine are as in attn_tc.cu (stream-K over KV tiles, tickets, no waiting).
#include <cfloat>
#include <climits>

#include "svp_params.cuh"

namespace svp {

constexpr int kVK = 128;            // keys per KV tile
constexpr int kVThreads = 192;
constexpr int kSlotBytes = 32768;   // [128 keys][128 d] bf16 = 2 x [128][64] SW128
constexpr int kSubBytes = 16384;    // [128 keys][64 d]
constexpr float kSlack = 8.0f;      // P <= 2^8

// Shared per-row softmax state (in the misc region).
struct VtRows {
    float m_ref[128];
    float alpha[128];
    float red[4][128];
    int32_t jr[128];     // candidate index of the row (INT_MAX for padding rows)
    float lrow[128];
    int32_t flag[2];
    int32_t rescale;
    int32_t last;
    int32_t abort_flag;
    uint32_t tmem;
    int32_t warp_sums[8];
};

__device__ __forceinline__ int64_t vt_cta_start(int64_t total, int32_t c, int32_t C)
{
    return (int64_t)c * total / C;
}

__device__ __forceinline__ int32_t vt_cta_of_unit(int64_t u, int64_t total, int32_t C)
{
    return (int32_t)(((u + 1) * C + total - 1) / total - 1);
}

struct VtSeg {
    int32_t i, rb, hg, t0, t1, n_ctx, n_tiles, first_of_cta, single, pair;
    int64_t u_pair0;
};

// KV tiles of (request i, row block rb): context tiles of 128 keys, then candidate
// tiles of CB keys up to the last candidate this row block needs.
__device__ __forceinline__ void vt_units(const TcParams &p, int32_t i, int32_t rb,
                                         int32_t &n_tiles, int32_t &bad)
{
    n_tiles = 0;
    bad = 0;
    const int32_t off = __ldg(p.cu_slots + i);
    const int32_t end = __ldg(p.cu_slots + i + 1);
    const int32_t k = end - off;
    if (off < 0 || end < off || k > p.w || end > p.m_cap) {
        bad = SVP_DEV_BAD_SLOTS;
        return;
    }
    const int32_t L = p.ctx_len ? __ldg(p.ctx_len + i) : 0;
    if (L < 0) {
        bad = SVP_DEV_BAD_CONTEXT;
        return;
    }
    if (L > 0) {
        if (p.paged) {
            if ((int64_t)(L + 15) / 16 > p.max_pages) {
                bad = SVP_DEV_BAD_CONTEXT;
                return;
            }
        } else {
            const int64_t c0 = __ldg(p.cu_ctx + i);
            if (c0 < 0 || c0 + L > p.total_tokens) {
                bad = SVP_DEV_BAD_CONTEXT;
                return;
            }
        }
    }
    const int32_t r0 = rb * p.R;
    if (r0 >= k)
        return;
    const int32_t cmax = min(k, r0 + p.R);
    n_tiles = (L + kVK - 1) / kVK + (cmax + p.CB - 1) / p.CB;
}

__device__ __forceinline__ void vt_seg(const TcParams &p, const int32_t *prefix, int32_t nq,
                                       int64_t u, int64_t ue, int64_t cta_s, VtSeg &s)
{
    int32_t lo = 0, hi = nq;
    while (hi - lo > 1) {
        const int32_t mid = (lo + hi) >> 1;
        if (prefix[mid] <= u)
            lo = mid;
        else
            hi = mid;
    }
    while (prefix[lo + 1] <= u)
        ++lo;
    const int32_t q = lo;
    const int32_t per = (prefix[q + 1] - prefix[q]) / p.HG;
    const int64_t local = u - prefix[q];
    s.i = q / p.RB;
    s.rb = q % p.RB;
    s.hg = (int32_t)(local / per);
    s.t0 = (int32_t)(local % per);
    s.n_tiles = per;
    s.u_pair0 = prefix[q] + (int64_t)s.hg * per;
    const int64_t seg_end = min(ue, s.u_pair0 + per);
    s.t1 = s.t0 + (int32_t)(seg_end - u);
    const int32_t L = p.ctx_len ? __ldg(p.ctx_len + s.i) : 0;
    s.n_ctx = (L + kVK - 1) / kVK;
    s.first_of_cta = (u == cta_s);
    s.single = (s.t0 == 0 && s.t1 == per);
    s.pair = q * p.HG + s.hg;
}

// Keys of tile t that hold data of this request (rows >= kvalid are zeroed in V).
__device__ __forceinline__ int32_t vt_kvalid(const TcParams &p, const VtSeg &s, int32_t t,
                                             int32_t L, int32_t k_i)
{
    if (t < s.n_ctx)
        return min(kVK, L - t * kVK);
    return max(0, min(p.CB, min(k_i, (s.rb + 1) * p.R) - (t - s.n_ctx) * p.CB));
}

// Transpose-reduce of 32 values across the warp: lane l ends with max over lanes of v[l].
__device__ __forceinline__ float warp_transpose_max32(float (&v)[32], int lane)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = upper ? v[i] : v[i + o];
            const float keep = upper ? v[i + o] : v[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, o);
            v[i] = fmaxf(keep, recv);
        }
    }
    return v[0];
}

template <int D>
__global__ void __launch_bounds__(kVThreads, 1) verify_tc_kernel(const __grid_constant__ TcParams p)
{
    constexpr int DH = D / 128;           // 128-column halves of d
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NR = p.NR;                  // rows of the query tile (multiple of 32)
    const int nslot = p.nslot;
    const uint32_t QSUB = (uint32_t)NR * 128u;   // [NR rows][64 d] sub-tile

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    const uint32_t bar0 = smem_u32(bars);
    auto bar_full = [&](int s) { return bar0 + 8u * s; };
    auto bar_empty = [&](int s) { return bar0 + 8u * (8 + s); };
    const uint32_t bar_qfull = bar0 + 8u * 16, bar_qempty = bar0 + 8u * 17;
    auto bar_sfull = [&](int b) { return bar0 + 8u * (18 + b); };
    auto bar_sfree = [&](int b) { return bar0 + 8u * (20 + b); };
    const uint32_t bar_pfull = bar0 + 8u * 22, bar_pvdone = bar0 + 8u * 23;
    const uint32_t bar_ofree = bar0 + 8u * 24, bar_drain = bar0 + 8u * 25;

    VtRows *rs = reinterpret_cast<VtRows *>(smem + p.off_misc);
    volatile int *abort_flag = &rs->abort_flag;
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + p.off_pref);
    const int32_t NQ = p.n * p.RB;

    if (tid == 0) {
        for (int s = 0; s < nslot; ++s) {
            mbar_init(bar_full(s), 1);
            mbar_init(bar_empty(s), 1);
        }
        mbar_init(bar_qfull, 1);
        mbar_init(bar_qempty, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_sfull(b), 1);
            mbar_init(bar_sfree(b), 4);
        }
        mbar_init(bar_pfull, 4);
        mbar_init(bar_pvdone, 1);
        mbar_init(bar_ofree, 4);
        mbar_init(bar_drain, 1);
        mbar_fence_init();
        rs->abort_flag = 0;
        rs->flag[0] = rs->flag[1] = 0;
        rs->rescale = 0;
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_kc);
        tma_prefetch_desc(&p.tm_vc);
        tma_prefetch_desc(&p.tm_kn);
        tma_prefetch_desc(&p.tm_vn);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&rs->tmem), (uint32_t)p.tmem_cols);
        tmem_relinquish();
    }
    // Q rows beyond the TMA box stay zero; the ones block feeds the row-sum MMA.
    for (int x = tid; x < (int)(QSUB * (D / 64) / 16); x += kVThreads)
        st_shared_v4(sbase + p.off_q + x * 16, 0u, 0u, 0u, 0u);
    for (int x = tid; x < 1024 / 16; x += kVThreads)
        st_shared_v4(sbase + p.off_ones + x * 16, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u,
                     0x3f803f80u);
    fence_proxy_async_smem();

    // prefix sums of KV tiles over (request, row block)
    int32_t bad_bits = 0;
    if (tid == 0)
        prefix[0] = 0;
    int32_t running = 0;
    for (int32_t base = 0; base < NQ; base += kVThreads) {
        const int32_t q = base + tid;
        int32_t units = 0;
        if (q < NQ) {
            int32_t nt, bad;
            vt_units(p, q / p.RB, q % p.RB, nt, bad);
            bad_bits |= bad;
            units = nt * p.HG;
        }
        int32_t incl = units;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += v;
        }
        __syncthreads();
        if (lane == 31)
            rs->warp_sums[warp] = incl;
        __syncthreads();
        int32_t before = running;
        for (int w2 = 0; w2 < warp; ++w2)
            before += rs->warp_sums[w2];
        if (q < NQ)
            prefix[q + 1] = before + incl;
        for (int w2 = 0; w2 < kVThreads / 32; ++w2)
            running += rs->warp_sums[w2];
    }
    if (bad_bits && blockIdx.x == 0)
        set_status(p.status, bad_bits);
    if (tid == 0) {
        // the workspace layout must match this call's (head_dim, tile mode)
        const int32_t seen = *reinterpret_cast<volatile int32_t *>(p.status + 1);
        rs->last = (seen != 0 && seen != p.sig) ? 1 : 0;
        if (rs->last && blockIdx.x == 0)
            set_status(p.status, SVP_DEV_WORKSPACE);
        if (seen == 0 && blockIdx.x == 0)
            p.status[1] = p.sig;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = rs->tmem;
    const int64_t total = rs->last ? 0 : prefix[NQ];
    const int32_t ncta = (int32_t)((int64_t)gridDim.x < total ? (int64_t)gridDim.x : total);
    int64_t cta_s = 0, cta_e = 0;
    if ((int32_t)blockIdx.x < ncta) {
        cta_s = vt_cta_start(total, blockIdx.x, ncta);
        cta_e = vt_cta_start(total, blockIdx.x + 1, ncta);
    }
    const uint32_t TM_S = 0, TM_O = 2u * NR, TM_L = (2u + DH) * NR;

    if (warp == 0) {
        // ================================================================ producer
        if (lane == 0) {
            uint32_t it = 0, nseg = 0, seq = 0;
            bool ok = true;
            for (int64_t u = cta_s; u < cta_e && ok;) {
                VtSeg s;
                vt_seg(p, prefix, NQ, u, cta_e, cta_s, s);
                const int32_t off = __ldg(p.cu_slots + s.i);
                const int32_t L = p.ctx_len ? __ldg(p.ctx_len + s.i) : 0;
                const int32_t g = (s.hg * p.HP) / p.G;
                if (nseg > 0 && !(ok = mbar_wait(bar_qempty, (nseg - 1) & 1, abort_flag)))
                    break;
                mbar_arrive_expect_tx(bar_qfull, (uint32_t)((D / 64) * 64 * p.HP * p.R * 2));
                for (int dc = 0; dc < D / 64; ++dc)
                    tma_load_3d(sbase + p.off_q + dc * QSUB, &p.tm_q, bar_qfull, dc * 64,
                                s.hg * p.HP, off + s.rb * p.R);
                ++nseg;
                const int64_t cctx = (!p.paged && L > 0) ? __ldg(p.cu_ctx + s.i) : 0;
                for (int32_t t = s.t0; t < s.t1 && ok; ++t, ++it) {
                    // K halves then V halves of this tile, one ring slot each
                    for (int kv = 0; kv < 2 && ok; ++kv) {
                        const CUtensorMap *mc = kv ? &p.tm_vc : &p.tm_kc;
                        const CUtensorMap *mn = kv ? &p.tm_vn : &p.tm_kn;
                        for (int h = 0; h < DH; ++h, ++seq) {
                            const int sl = seq % nslot;
                            if (!(ok = mbar_wait(bar_empty(sl), ((seq / nslot) & 1) ^ 1, abort_flag)))
                                break;
                            const uint32_t dst = sbase + p.off_ring + sl * kSlotBytes;
                            if (t < s.n_ctx) {
                                if (!p.paged) {
                                    mbar_arrive_expect_tx(bar_full(sl), (uint32_t)kSlotBytes);
                                    const int32_t row = (int32_t)(cctx + (int64_t)t * kVK);
                                    for (int c = 0; c < 2; ++c)
                                        tma_load_3d(dst + c * kSubBytes, mc, bar_full(sl),
                                                    h * 128 + c * 64, g, row);
                                } else {
                                    const int32_t pg0 = t * (kVK / 16);
                                    const int32_t npg = min(kVK / 16, (L + 15) / 16 - pg0);
                                    int32_t ids[kVK / 16];
                                    int32_t nv = 0;
                                    for (int pp = 0; pp < kVK / 16; ++pp) {
                                        ids[pp] = -1;
                                        if (pp < npg) {
                                            const int32_t id = __ldg(p.block_table +
                                                                     (int64_t)s.i * p.max_pages + pg0 + pp);
                                            if (id >= 0 && id < p.num_pages) {
                                                ids[pp] = id;
                                                ++nv;
                                            } else {
                                                set_status(p.status, SVP_DEV_BAD_CONTEXT);
                                            }
                                        }
                                    }
                                    mbar_arrive_expect_tx(bar_full(sl), (uint32_t)(nv * 2 * 2048));
                                    for (int pp = 0; pp < kVK / 16; ++pp) {
                                        if (ids[pp] < 0)
                                            continue;
                                        for (int c = 0; c < 2; ++c)
                                            tma_load_4d(dst + c * kSubBytes + pp * 2048, mc,
                                                        bar_full(sl), h * 128 + c * 64, 0, g, ids[pp]);
                                    }
                                }
                            } else {
                                const int32_t ct = t - s.n_ctx;
                                mbar_arrive_expect_tx(bar_full(sl), (uint32_t)(2 * p.CB * 128));
                                for (int c = 0; c < 2; ++c)
                                    tma_load_3d(dst + c * kSubBytes, mn, bar_full(sl),
                                                h * 128 + c * 64, g, off + ct * p.CB);
                            }
                        }
                    }
                }
                u += (s.t1 - s.t0);
            }
            if (!ok) {
                volatile int drain_abort = 0;
                const uint32_t first = seq > (uint32_t)nslot ? seq - nslot : 0;
                for (uint32_t k = first; k < seq; ++k)
                    mbar_wait(bar_full(k % nslot), (k / nslot) & 1, &drain_abort);
                if (nseg > 0)
                    mbar_wait(bar_qfull, (nseg - 1) & 1, &drain_abort);
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, nseg = 0;
            bool ok = true;
            for (int64_t u = cta_s; u < cta_e && ok;) {
                VtSeg s;
                vt_seg(p, prefix, NQ, u, cta_e, cta_s, s);
                const int32_t off = __ldg(p.cu_slots + s.i);
                const int32_t k_i = __ldg(p.cu_slots + s.i + 1) - off;
                const int32_t L = p.ctx_len ? __ldg(p.ctx_len + s.i) : 0;
                const int32_t kk = min(k_i - s.rb * p.R, p.R);
                const uint32_t NRs = (uint32_t)((p.HP * kk + 31) / 32 * 32);
                const uint32_t idesc_s = idesc_bf16_f32(128, NRs, false, false);
                const uint32_t idesc_o = idesc_bf16_f32(128, NRs, true, true);
                const uint32_t idesc_l = idesc_bf16_f32(128, NRs, false, true);
                if (!(ok = mbar_wait(bar_qfull, nseg & 1, abort_flag)))
                    break;
                tc_fence_after();
                const int32_t nt = s.t1 - s.t0;
                for (int32_t k = 0; k <= nt && ok; ++k) {
                    if (k < nt) {
                        const uint32_t itk = it + k;
                        const int b = itk & 1;
                        if (!(ok = mbar_wait(bar_sfree(b), ((itk >> 1) & 1) ^ 1, abort_flag)))
                            break;
                        for (int h = 0; h < DH && ok; ++h) {
                            const uint32_t sq = itk * 2 * DH + h;
                            ok = mbar_wait(bar_full(sq % nslot), (sq / nslot) & 1, abort_flag);
                        }
                        if (!ok)
                            break;
                        tc_fence_after();
                        for (int h = 0; h < DH; ++h) {
                            const uint32_t ka = sbase + p.off_ring + ((itk * 2 * DH + h) % nslot) * kSlotBytes;
                            for (int ks = 0; ks < 8; ++ks) {
                                const uint32_t a = ka + (ks >> 2) * kSubBytes + (ks & 3) * 32;
                                const uint32_t bq = sbase + p.off_q + (2 * h + (ks >> 2)) * QSUB + (ks & 3) * 32;
                                tc_mma_ss(tmem + TM_S + b * NR, sw128_desc(a, 16, 1024),
                                          sw128_desc(bq, 16, 1024), idesc_s, (h | ks) ? 1u : 0u);
                            }
                        }
                        tc_commit(bar_sfull(b));
                        for (int h = 0; h < DH; ++h)
                            tc_commit(bar_empty((itk * 2 * DH + h) % nslot));
                        if (k == nt - 1)
                            tc_commit(bar_qempty);
                    }
                    if (k > 0) {
                        const uint32_t itp = it + k - 1;
                        const int32_t t = s.t0 + k - 1;
                        const int32_t kv = vt_kvalid(p, s, t, L, k_i);
                        const int32_t k16 = (kv + 15) / 16;
                        if (k == 1 && nseg > 0 &&
                            !(ok = mbar_wait(bar_ofree, (nseg - 1) & 1, abort_flag)))
                            break;
                        if (!(ok = mbar_wait(bar_pfull, itp & 1, abort_flag)))
                            break;
                        for (int h = 0; h < DH && ok; ++h) {
                            const uint32_t sq = itp * 2 * DH + DH + h;
                            ok = mbar_wait(bar_full(sq % nslot), (sq / nslot) & 1, abort_flag);
                        }
                        if (!ok)
                            break;
                        tc_fence_after();
                        const uint32_t pb = sbase + p.off_p;
                        for (int h = 0; h < DH; ++h) {
                            const uint32_t va = sbase + p.off_ring + ((itp * 2 * DH + DH + h) % nslot) * kSlotBytes;
                            for (int ks = 0; ks < k16; ++ks)
                                tc_mma_ss(tmem + TM_O + h * NR, sw128_desc(va + ks * 2048, kSubBytes, 1024),
                                          sw128_desc(pb + ks * 2048, 16384, 1024), idesc_o,
                                          (k == 1 && ks == 0) ? 0u : 1u);
                        }
                        for (int ks = 0; ks < k16; ++ks)
                            tc_mma_ss(tmem + TM_L, sw128_desc(sbase + p.off_ones, 16, 0),
                                      sw128_desc(pb + ks * 2048, 16384, 1024), idesc_l,
                                      (k == 1 && ks == 0) ? 0u : 1u);
                        tc_commit(bar_pvdone);
                        for (int h = 0; h < DH; ++h)
                            tc_commit(bar_empty((itp * 2 * DH + DH + h) % nslot));
                    }
                }
                it += nt;
                ++nseg;
                u += nt;
            }
            tc_commit(bar_drain);
            volatile int drain_abort = 0;
            mbar_wait(bar_drain, 0, &drain_abort);
        }
    } else {
        // ================================================================ softmax
        const int quarter = warp & 3;
        const int t = quarter * 32 + lane;            // key of the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int stid = tid - 64;                    // 0..127
        const float cl2 = p.scale_log2;
        uint32_t it = 0, nseg = 0;
        bool ok = true;
        for (int64_t u = cta_s; u < cta_e && ok;) {
            VtSeg s;
            vt_seg(p, prefix, NQ, u, cta_e, cta_s, s);
            const int32_t off = __ldg(p.cu_slots + s.i);
            const int32_t k_i = __ldg(p.cu_slots + s.i + 1) - off;
            const int32_t L = p.ctx_len ? __ldg(p.ctx_len + s.i) : 0;
            const int32_t kk = min(k_i - s.rb * p.R, p.R);
            const int NRs = (p.HP * kk + 31) / 32 * 32;
            const int nch = NRs / 32;
            // per-row state: active rows start at m_ref = -inf, the others at +inf
            if (stid < NR) {
                const int r = stid;
                const bool act = r < p.HP * kk;
                rs->m_ref[r] = act ? -INFINITY : INFINITY;
                rs->jr[r] = act ? s.rb * p.R + r / p.HP : INT_MAX;
            }
            named_bar_sync(1, 128);
            const int32_t nt = s.t1 - s.t0;
            for (int32_t k = 0; k < nt; ++k, ++it) {
                const int32_t tt = s.t0 + k;
                const int b = it & 1;
                const bool is_ctx = tt < s.n_ctx;
                const int32_t kvalid = vt_kvalid(p, s, tt, L, k_i);
                const int32_t cbase = is_ctx ? 0 : (tt - s.n_ctx) * p.CB;   // candidate index of key 0
                const bool key_ok = t < kvalid;
                if (!(ok = mbar_wait(bar_sfull(b), (it >> 1) & 1, abort_flag)))
                    break;
                tc_fence_after();
                // P^T (shared) is read by PV of the previous tile
                if (it > 0 && !(ok = mbar_wait(bar_pvdone, (it - 1) & 1, abort_flag)))
                    break;
                const uint32_t sa = tmem + lane_off + TM_S + b * NR;
                const uint32_t pline = sbase + p.off_p + t * 128;
                bool hit = false;
                for (int c = 0; c < nch; ++c) {
                    uint32_t sr[32];
                    tmem_ld32(sa + c * 32, sr);
                    tmem_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int e2 = 0; e2 < 16; ++e2) {
                        float pv[2];
#pragma unroll
                        for (int q2 = 0; q2 < 2; ++q2) {
                            const int r = c * 32 + e2 * 2 + q2;
                            const float y = fmaf(__uint_as_float(sr[e2 * 2 + q2]), cl2, -rs->m_ref[r]);
                            const bool vis = key_ok && (is_ctx || cbase + t <= rs->jr[r]);
                            hit |= vis && (y > kSlack);
                            pv[q2] = vis ? fast_exp2(y) : 0.0f;
                        }
                        pk[e2] = pack_bf16x2(pv[0], pv[1]);
                    }
                    const int blk = c >> 1, c0 = (c & 1) * 4;
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        st_shared_v4(pline + blk * 16384 + (((c0 + v) ^ (t & 7)) << 4),
                                     pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
                if (__any_sync(0xffffffffu, hit) && lane == 0)
                    rs->flag[it & 1] = 1;
                named_bar_sync(1, 128);
                const bool need = rs->flag[it & 1] != 0;
                if (stid == 0)
                    rs->flag[(it + 1) & 1] = 0;
                if (need) {
                    // ---- rare path: row maxima across keys, move m_ref, rescale O^T, l^T
                    for (int c = 0; c < nch; ++c) {
                        uint32_t sr[32];
                        tmem_ld32(sa + c * 32, sr);
                        tmem_wait_ld();
                        float v[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int r = c * 32 + e;
                            const bool vis = key_ok && (is_ctx || cbase + t <= rs->jr[r]);
                            v[e] = vis ? __uint_as_float(sr[e]) * cl2 : -INFINITY;
                        }
                        rs->red[quarter][c * 32 + lane] = warp_transpose_max32(v, lane);
                    }
                    named_bar_sync(1, 128);
                    if (stid < NRs) {
                        const int r = stid;
                        const float mo = rs->m_ref[r];
                        float a = 1.0f;
                        if (mo != INFINITY) {
                            const float mt = fmaxf(fmaxf(rs->red[0][r], rs->red[1][r]),
                                                   fmaxf(rs->red[2][r], rs->red[3][r]));
                            const float mn = fmaxf(mo, mt);
                            if (mn > mo + kSlack || (mo == -INFINITY && mn != -INFINITY)) {
                                a = (mo == -INFINITY) ? 0.0f : fast_exp2(mo - mn);
                                rs->m_ref[r] = mn;
                                if (k > 0)
                                    rs->rescale = 1;
                            }
                        }
                        rs->alpha[r] = a;
                    }
                    named_bar_sync(1, 128);
                    if (rs->rescale) {
                        // O^T halves and l^T: column r scaled by alpha[r] (PV of the
                        // previous tile is complete: waited above)
                        for (int m = 0; m <= DH; ++m) {
                            const uint32_t base = tmem + lane_off + (m < DH ? TM_O + m * NR : TM_L);
                            for (int c = 0; c < nch; ++c) {
                                uint32_t ro[32];
                                tmem_ld32(base + c * 32, ro);
                                tmem_wait_ld();
#pragma unroll
                                for (int e = 0; e < 32; ++e)
                                    ro[e] = __float_as_uint(__uint_as_float(ro[e]) * rs->alpha[c * 32 + e]);
                                tmem_st32(base + c * 32, ro);
                            }
                        }
                        tmem_wait_st();
                    }
                    // P with the new reference
                    for (int c = 0; c < nch; ++c) {
                        uint32_t sr[32];
                        tmem_ld32(sa + c * 32, sr);
                        tmem_wait_ld();
                        uint32_t pk[16];
#pragma unroll
                        for (int e2 = 0; e2 < 16; ++e2) {
                            float pv[2];
#pragma unroll
                            for (int q2 = 0; q2 < 2; ++q2) {
                                const int r = c * 32 + e2 * 2 + q2;
                                const float y = fmaf(__uint_as_float(sr[e2 * 2 + q2]), cl2, -rs->m_ref[r]);
                                const bool vis = key_ok && (is_ctx || cbase + t <= rs->jr[r]);
                                pv[q2] = vis ? fast_exp2(y) : 0.0f;
                            }
                            pk[e2] = pack_bf16x2(pv[0], pv[1]);
                        }
                        const int blk = c >> 1, c0 = (c & 1) * 4;
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            st_shared_v4(pline + blk * 16384 + (((c0 + v) ^ (t & 7)) << 4),
                                         pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    }
                    named_bar_sync(1, 128);
                    if (stid == 0)
                        rs->rescale = 0;
                }
                // S buffer b is free for the next S^T
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar_sfree(b));
                // zero V rows of keys without data that PV reads (NaN-safe)
                const int32_t k16 = (kvalid + 15) / 16 * 16;
                if (kvalid < k16 && t >= kvalid && t < k16) {
                    for (int h = 0; h < DH; ++h) {
                        const uint32_t sq = it * 2 * DH + DH + h;
                        if (!mbar_wait(bar_full(sq % nslot), (sq / nslot) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        const uint32_t vrow = sbase + p.off_ring + (sq % nslot) * kSlotBytes + t * 128;
                        for (int c = 0; c < 2; ++c)
                            for (int v = 0; v < 8; ++v)
                                st_shared_v4(vrow + c * kSubBytes + v * 16, 0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar_pfull);
                if (!ok)
                    break;
            }
            if (!ok)
                break;
            // ---- epilogue: O^T, l^T complete after the last PV of the segment
            if (!(ok = mbar_wait(bar_pvdone, (it - 1) & 1, abort_flag)))
                break;
            tc_fence_after();
            // row sums: every lane of l^T holds l for each column
            for (int c = 0; c < nch; ++c) {
                uint32_t lr[32];
                tmem_ld32(tmem + lane_off + TM_L + c * 32, lr);
                tmem_wait_ld();
                if (quarter == 0 && lane == 0) {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        rs->lrow[c * 32 + e] = __uint_as_float(lr[e]);
                }
            }
            named_bar_sync(1, 128);
            const int32_t out_row0 = off + s.rb * p.R;
            const int nact = p.HP * kk;                // active rows of this tile
            if (s.single) {
                for (int h = 0; h < DH; ++h) {
                    for (int c = 0; c < nch; ++c) {
                        uint32_t ro[32];
                        tmem_ld32(tmem + lane_off + TM_O + h * NR + c * 32, ro);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int r = c * 32 + e;
                            if (r < nact) {
                                const int64_t orow = (int64_t)(out_row0 + r / p.HP) * p.hq + s.hg * p.HP + r % p.HP;
                                reinterpret_cast<uint16_t *>(p.out)[orow * D + h * 128 + t] =
                                    (uint16_t)(pack_bf16x2(__uint_as_float(ro[e]) / rs->lrow[r], 0.0f) & 0xffffu);
                            }
                        }
                    }
                }
                if (stid < nact && p.lse) {
                    const int r = stid;
                    const int64_t orow = (int64_t)(out_row0 + r / p.HP) * p.hq + s.hg * p.HP + r % p.HP;
                    p.lse[orow] = (rs->m_ref[r] + __log2f(rs->lrow[r])) * 0.69314718055994531f;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar_ofree);
            } else {
                const int32_t slot = 2 * blockIdx.x + (s.first_of_cta ? 0 : 1);
                for (int h = 0; h < DH; ++h) {
                    for (int c = 0; c < nch; ++c) {
                        uint32_t ro[32];
                        tmem_ld32(tmem + lane_off + TM_O + h * NR + c * 32, ro);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int r = c * 32 + e;
                            if (r < nact)
                                __stcg(p.part_o + ((int64_t)slot * kRows + r) * D + h * 128 + t,
                                       __uint_as_float(ro[e]));
                        }
                    }
                }
                if (stid < nact)
                    __stcg(p.part_ml + (int64_t)slot * kRows + stid,
                           make_float2(rs->m_ref[stid], rs->lrow[stid]));
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar_ofree);
                __threadfence();
                named_bar_sync(1, 128);
                const int32_t cf = vt_cta_of_unit(s.u_pair0, total, ncta);
                const int32_t cl = vt_cta_of_unit(s.u_pair0 + s.n_tiles - 1, total, ncta);
                if (stid == 0) {
                    const int prev = atomicAdd(p.tickets + s.pair, 1);
                    rs->last = (prev == cl - cf) ? 1 : 0;
                }
                named_bar_sync(1, 128);
                if (rs->last) {
                    __threadfence();
                    // per row: global max and sum over the pieces (threads r < nact)
                    if (stid < nact) {
                        const int r = stid;
                        float M = -INFINITY;
                        for (int32_t c = cf; c <= cl; ++c) {
                            const int64_t cs = vt_cta_start(total, c, ncta);
                            const int32_t sl = 2 * c + ((c == cf && cs < s.u_pair0) ? 1 : 0);
                            M = fmaxf(M, __ldcg(p.part_ml + (int64_t)sl * kRows + r).x);
                        }
                        float Ls = 0.0f;
                        for (int32_t c = cf; c <= cl; ++c) {
                            const int64_t cs = vt_cta_start(total, c, ncta);
                            const int32_t sl = 2 * c + ((c == cf && cs < s.u_pair0) ? 1 : 0);
                            const float2 ml = __ldcg(p.part_ml + (int64_t)sl * kRows + r);
                            Ls += ml.y * fast_exp2(ml.x - M);
                        }
                        rs->m_ref[r] = M;          // reused as the merged max
                        rs->lrow[r] = Ls;
                        if (p.lse) {
                            const int64_t orow = (int64_t)(out_row0 + r / p.HP) * p.hq + s.hg * p.HP + r % p.HP;
                            p.lse[orow] = (M + __log2f(Ls)) * 0.69314718055994531f;
                        }
                    }
                    named_bar_sync(1, 128);
                    // thread = column of d; rows in order, pieces in order
                    for (int r = 0; r < nact; ++r) {
                        const float M = rs->m_ref[r], inv = 1.0f / rs->lrow[r];
                        float acc[DH];
#pragma unroll
                        for (int h = 0; h < DH; ++h)
                            acc[h] = 0.0f;
                        for (int32_t c = cf; c <= cl; ++c) {
                            const int64_t cs = vt_cta_start(total, c, ncta);
                            const int32_t sl = 2 * c + ((c == cf && cs < s.u_pair0) ? 1 : 0);
                            const float wgt = fast_exp2(__ldcg(p.part_ml + (int64_t)sl * kRows + r).x - M);
#pragma unroll
                            for (int h = 0; h < DH; ++h)
                                acc[h] += wgt * __ldcg(p.part_o + ((int64_t)sl * kRows + r) * D + h * 128 + t);
                        }
                        const int64_t orow = (int64_t)(out_row0 + r / p.HP) * p.hq + s.hg * p.HP + r % p.HP;
#pragma unroll
                        for (int h = 0; h < DH; ++h)
                            reinterpret_cast<uint16_t *>(p.out)[orow * D + h * 128 + t] =
                                (uint16_t)(pack_bf16x2(acc[h] * inv, 0.0f) & 0xffffu);
                    }
                    named_bar_sync(1, 128);
                    if (stid == 0)
                        p.tickets[s.pair] = 0;
                }
            }
            named_bar_sync(1, 128);
            ++nseg;
            u += nt;
        }
    }

    if (*abort_flag && tid == 0)
        set_status(p.status, SVP_DEV_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
}

template <int D>
static svp_status vt_launch_d(const TcParams &p, int grid, cudaStream_t stream)
{
    static bool configured = false;
    if (!configured) {
        if (cudaFuncSetAttribute(verify_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 227 * 1024) != cudaSuccess)
            return SVP_ECUDA;
        configured = true;
    }
    verify_tc_kernel<D><<<grid, kVThreads, p.smem_bytes, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? SVP_OK : SVP_ECUDA;
}

svp_status verify_tc_launch(const TcParams &p, int d, int grid, cudaStream_t stream)
{
    switch (d) {
    case 128: return vt_launch_d<128>(p, grid, stream);
    case 256: return vt_launch_d<256>(p, grid, stream);
    default: return SVP_EUNSUPPORTED;
    }
}

// Shared-memory layout of verify_tc_kernel for a tile of NR rows (host helper).
bool verify_tc_layout(int d, int NR, TcParams &p)
{
    const int budget = 227 * 1024;
    const int q = (d / 64) * NR * 128;
    const int pt = ((NR + 63) / 64) * 16384;
    int off = 0;
    p.off_q = off; off += q;
    p.off_p = off; off += pt;
    p.off_ones = off; off += 1024;
    p.off_bar = off; off += 26 * 8;
    off = (off + 15) / 16 * 16;
    p.off_misc = off; off += (int)sizeof(VtRows);
    off = (off + 15) / 16 * 16;
    p.off_pref = off; off += (kMaxPrefix + 1) * 4;
    off = (off + 1023) / 1024 * 1024;
    p.off_ring = off;
    const int slots = (budget - 1024 - off) / kSlotBytes;
    p.nslot = slots > 8 ? 8 : slots;
    if (p.nslot < 2 * (d / 128))
        return false;
    p.smem_bytes = off + p.nslot * kSlotBytes + 1024;
    const int cols = (3 + d / 128) * NR;
    int tc = 32;
    while (tc < cols)
        tc <<= 1;
    if (tc > 512)
        return false;
    p.tmem_cols = tc;
    p.NR = NR;
    return true;
}

}  // namespace svp
