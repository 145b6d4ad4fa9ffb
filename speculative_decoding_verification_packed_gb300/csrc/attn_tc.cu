// attn_tc.cu -- verification / prefill attention on tcgen05 tensor cores (bf16 in,
// fp32 accumulate), fed by TMA.
//
// What it computes (DScale, SIII-B path-aware tile router, SIII-C packed rows, SIII-D
// request-local causal masking): for request i, every packed candidate row j in
// [0, k_i) of every query head h attends to the ctx_len[i] context tokens of KV head
// h / G and then to the request's own candidates 0..j, with softmax scale `scale`.
//
// Tile shapes (host-chosen, one kernel):
//   SHORT     the G query heads that share one KV head are packed into one query tile
//             of G x R rows (R = min(w, 128 / G) candidate rows per head), so one pass
//             over a KV tile serves all of them; the tile height follows the candidate
//             width instead of a fixed 128.
//   FIXED128  one query head per 128-row tile, one CTA per (request, head), no split:
//             the prior-art native tile, kept only as a contrast.
//   WIDE      one query head, 128 candidate rows per tile, causal over the candidates
//             (prefill and verification blocks longer than 16).
//
// Per CTA (one per SM, persistent): warp 0 issues TMA loads (Q tile once per work
// segment, then K/V tiles of 64 keys into a ring of shared-memory stages), warp 1
// allocates tensor memory and issues tcgen05.mma from one thread, warps 2..5 run the
// online softmax and the epilogue with one thread per query row (TMEM lane).
//   S  = Q K^T  : M=128 query rows, N=64 keys, K=d      -> TMEM (double buffered)
//   O += P V    : M=128 query rows, N=d,       K=64 keys -> TMEM (fp32 accumulator)
// P is written to shared memory in bf16 by the softmax warps.  The running maximum is
// only moved (and O rescaled in TMEM) when it grows by more than 2^8, so P <= 256.
//
// Work split (stream-K): the KV tiles of all (request, row block, head group) pairs form
// one sequence of work units that is cut into gridDim.x equal ranges.  A pair covered
// by one CTA is finished in place; otherwise every CTA writes an unnormalised partial
// (O, running max, sum) and the CTA that arrives last at the pair's ticket merges the
// partials in order (no waiting on other CTAs) and resets the ticket.
#include <cfloat>
#include <climits>

#include "svp_params.cuh"

namespace svp {

template <int D>
struct TcCfg {
    static constexpr int DC = D / 64;                         // 64-column chunks of d
    static constexpr int STAGES = (D == 64) ? 8 : (D == 128 ? 4 : 2);
    static constexpr int SUB = kBN * 128;                     // [64 keys][64 d] bf16
    static constexpr int KV_BYTES = DC * SUB;                 // one K (or V) tile
    static constexpr int STAGE = 2 * KV_BYTES;
    static constexpr int QSUB = kRows * 128;                  // [128 rows][64 d] bf16
    static constexpr int Q_BYTES = DC * QSUB;
    static constexpr int P_BYTES = kRows * 128;               // [128 rows][64 keys] bf16
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_P = OFF_Q + Q_BYTES;
    static constexpr int OFF_KV = OFF_P + P_BYTES;
    static constexpr int OFF_BAR = OFF_KV + STAGES * STAGE;
    static constexpr int NBAR = 2 * STAGES + 10;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int OFF_PREFIX = OFF_MISC + 64;
    static constexpr int SMEM = OFF_PREFIX + (kMaxPrefix + 1) * 4 + 1024;  // + align slack
    static constexpr int TMEM_O = 0;
    static constexpr int TMEM_S = D;                          // two buffers of 64 columns
    static constexpr int TMEM_COLS = (D + 2 * kBN) <= 256 ? 256 : 512;
};

// Work description shared by all roles (computed identically by each).
struct Seg {
    int32_t i, rb, hg;        // request, row block, head group
    int32_t t0, t1;           // tile range of the pair covered by this segment
    int32_t n_ctx, n_tiles;   // context tiles, all tiles of the pair
    int64_t u_pair0;          // first unit of the pair
    int32_t first_of_cta;     // the CTA's first segment
    int32_t single;           // the whole pair is in this segment
    int32_t pair;             // ticket index
};

struct Shared {
    int32_t *prefix;          // [NQ+1] cumulative units over (request, row block)
    int32_t nq;
    int64_t total;
};

__device__ __forceinline__ int64_t cta_start(int64_t total, int32_t c, int32_t C)
{
    return (int64_t)c * total / C;
}

// CTA that owns unit u (the largest c with cta_start(c) <= u).
__device__ __forceinline__ int32_t cta_of_unit(int64_t u, int64_t total, int32_t C)
{
    return (int32_t)(((u + 1) * C + total - 1) / total - 1);
}

// Units (KV tiles) of every head group of (request i, row block rb).
__device__ __forceinline__ void pair_units(const TcParams &p, int32_t i, int32_t rb,
                                           int32_t &n_ctx, int32_t &n_tiles, int32_t &bad)
{
    n_ctx = 0;
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
    n_ctx = (L + kBN - 1) / kBN;
    n_tiles = n_ctx + (cmax + p.CB - 1) / p.CB;
}

// Decode the segment that starts at unit u (u < CTA end ue).
__device__ __forceinline__ void make_seg(const TcParams &p, const Shared &sh, int64_t u,
                                         int64_t ue, int64_t cta_s, Seg &s)
{
    // binary search: largest q with prefix[q] <= u
    int32_t lo = 0, hi = sh.nq;
    while (hi - lo > 1) {
        const int32_t mid = (lo + hi) >> 1;
        if (sh.prefix[mid] <= u)
            lo = mid;
        else
            hi = mid;
    }
    // skip empty entries (prefix[q] == prefix[q+1])
    while (sh.prefix[lo + 1] <= u)
        ++lo;
    const int32_t q = lo;
    const int32_t per = (sh.prefix[q + 1] - sh.prefix[q]) / p.HG;
    const int64_t local = u - sh.prefix[q];
    s.i = q / p.RB;
    s.rb = q % p.RB;
    s.hg = (int32_t)(local / per);
    s.t0 = (int32_t)(local % per);
    s.n_tiles = per;
    s.u_pair0 = sh.prefix[q] + (int64_t)s.hg * per;
    const int64_t pair_end = s.u_pair0 + per;
    const int64_t seg_end = min(ue, pair_end);
    s.t1 = s.t0 + (int32_t)(seg_end - u);
    const int32_t L = p.ctx_len ? __ldg(p.ctx_len + s.i) : 0;
    s.n_ctx = (L + kBN - 1) / kBN;
    s.first_of_cta = (u == cta_s);
    s.single = (s.t0 == 0 && s.t1 == per);
    s.pair = q * p.HG + s.hg;
}

// ------------------------------------------------------------------------------ kernel
template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ TcParams p)
{
    using C = TcCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    const uint32_t bar0 = smem_u32(bars);
    auto bar_full = [&](int s) { return bar0 + 8u * s; };
    auto bar_empty = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    const uint32_t bar_qfull = bar0 + 8u * (2 * C::STAGES + 0);
    const uint32_t bar_qempty = bar0 + 8u * (2 * C::STAGES + 1);
    auto bar_sfull = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 + b); };
    auto bar_sfree = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 4 + b); };
    const uint32_t bar_pfull = bar0 + 8u * (2 * C::STAGES + 6);
    const uint32_t bar_pvdone = bar0 + 8u * (2 * C::STAGES + 7);
    const uint32_t bar_ofree = bar0 + 8u * (2 * C::STAGES + 8);
    const uint32_t bar_drain = bar0 + 8u * (2 * C::STAGES + 9);

    int32_t *misc = reinterpret_cast<int32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 0);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc + 1);
    int32_t *flag_last = misc + 2;
    int32_t *warp_sums = misc + 4;   // 6 entries
    Shared sh;
    sh.prefix = reinterpret_cast<int32_t *>(smem + C::OFF_PREFIX);
    const int32_t NQ = p.n * p.RB;
    sh.nq = NQ;

    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
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
        *abort_flag = 0;
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_kc);
        tma_prefetch_desc(&p.tm_vc);
        tma_prefetch_desc(&p.tm_kn);
        tma_prefetch_desc(&p.tm_vn);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }

    // Prefix sums of units over (request, row block), computed by every CTA.
    int32_t bad_bits = 0;
    if (tid == 0)
        sh.prefix[0] = 0;
    int32_t running = 0;
    for (int32_t base = 0; base < NQ; base += kThreads) {
        const int32_t q = base + tid;
        int32_t units = 0;
        if (q < NQ) {
            int32_t n_ctx, n_tiles, bad;
            pair_units(p, q / p.RB, q % p.RB, n_ctx, n_tiles, bad);
            bad_bits |= bad;
            units = n_tiles * p.HG;
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
            warp_sums[warp] = incl;
        __syncthreads();
        int32_t before = running;
        for (int w2 = 0; w2 < warp; ++w2)
            before += warp_sums[w2];
        if (q < NQ)
            sh.prefix[q + 1] = before + incl;
        for (int w2 = 0; w2 < kThreads / 32; ++w2)
            running += warp_sums[w2];
    }
    if (bad_bits && blockIdx.x == 0)
        set_status(p.status, bad_bits);
    if (tid == 0) {
        // the workspace layout must match this call's (head_dim, tile mode)
        const int32_t seen = *reinterpret_cast<volatile int32_t *>(p.status + 1);
        const int32_t poisoned = *reinterpret_cast<volatile int32_t *>(p.status + kWsPoisonWord);
        *flag_last = ((seen != 0 && seen != p.sig) || poisoned != 0) ? 1 : 0;
        if (*flag_last && blockIdx.x == 0)
            set_status(p.status, SVP_DEV_WORKSPACE);
        if (seen == 0 && blockIdx.x == 0)
            p.status[1] = p.sig;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const bool ws_bad = *flag_last != 0;
    sh.total = ws_bad ? 0 : sh.prefix[NQ];

    // This CTA's unit range.  The units are cut into ncta = min(grid, units) ranges so
    // that every range is non-empty (a pair's pieces are then consecutive CTAs).
    const int32_t ncta = (int32_t)((int64_t)gridDim.x < sh.total ? (int64_t)gridDim.x : sh.total);
    int64_t cta_s, cta_e;
    if (p.split) {
        if ((int32_t)blockIdx.x < ncta) {
            cta_s = cta_start(sh.total, blockIdx.x, ncta);
            cta_e = cta_start(sh.total, blockIdx.x + 1, ncta);
        } else {
            cta_s = cta_e = 0;
        }
    } else if (ws_bad) {
        cta_s = cta_e = 0;
    } else {
        // one (request, row block, head group) pair per CTA
        const int32_t pair = blockIdx.x;
        const int32_t q = pair / p.HG, hg = pair % p.HG;
        const int32_t per = (sh.prefix[q + 1] - sh.prefix[q]) / p.HG;
        cta_s = sh.prefix[q] + (int64_t)hg * per;
        cta_e = cta_s + per;
    }

    const int32_t CB = p.CB;
    const int32_t DCn = C::DC;

    if (warp == 0) {
        // ============================================================ TMA producer
        if (lane == 0) {
            uint32_t it = 0, nseg = 0;
            bool ok = true;
            for (int64_t u = cta_s; u < cta_e && ok;) {
                Seg s;
                make_seg(p, sh, u, cta_e, cta_s, s);
                const int32_t off = __ldg(p.cu_slots + s.i);
                const int32_t L = p.ctx_len ? __ldg(p.ctx_len + s.i) : 0;
                const int32_t g = (s.hg * p.HP) / p.G;
                // Q tile
                if (nseg > 0 && !(ok = mbar_wait(bar_qempty, (nseg - 1) & 1, abort_flag)))
                    break;
                mbar_arrive_expect_tx(bar_qfull, (uint32_t)(DCn * 64 * p.HP * p.R * 2));
                for (int dc = 0; dc < DCn; ++dc)
                    tma_load_3d(sbase + C::OFF_Q + dc * C::QSUB, &p.tm_q, bar_qfull, dc * 64,
                                s.hg * p.HP, off + s.rb * p.R);
                ++nseg;
                // K/V tiles
                const int64_t cctx = (!p.paged && L > 0) ? __ldg(p.cu_ctx + s.i) : 0;
                for (int32_t t = s.t0; t < s.t1; ++t, ++it) {
                    const int st = it % C::STAGES;
                    const uint32_t round = it / C::STAGES;
                    if (!(ok = mbar_wait(bar_empty(st), (round & 1) ^ 1, abort_flag)))
                        break;
                    const uint32_t kdst = sbase + C::OFF_KV + st * C::STAGE;
                    const uint32_t vdst = kdst + C::KV_BYTES;
                    if (t < s.n_ctx) {
                        if (!p.paged) {
                            mbar_arrive_expect_tx(bar_full(st), (uint32_t)(2 * C::KV_BYTES));
                            const int32_t row = (int32_t)(cctx + (int64_t)t * kBN);
                            for (int dc = 0; dc < DCn; ++dc) {
                                tma_load_3d(kdst + dc * C::SUB, &p.tm_kc, bar_full(st), dc * 64, g, row);
                                tma_load_3d(vdst + dc * C::SUB, &p.tm_vc, bar_full(st), dc * 64, g, row);
                            }
                        } else {
                            const int32_t pg0 = t * (kBN / 16);
                            const int32_t npg = min(kBN / 16, (L + 15) / 16 - pg0);
                            int32_t ids[kBN / 16];
                            int32_t nvalid = 0;
                            for (int pp = 0; pp < kBN / 16; ++pp) {
                                ids[pp] = -1;
                                if (pp < npg) {
                                    const int32_t id = __ldg(p.block_table + (int64_t)s.i * p.max_pages + pg0 + pp);
                                    if (id >= 0 && id < p.num_pages) {
                                        ids[pp] = id;
                                        ++nvalid;
                                    } else {
                                        set_status(p.status, SVP_DEV_BAD_CONTEXT);
                                    }
                                }
                            }
                            mbar_arrive_expect_tx(bar_full(st), (uint32_t)(nvalid * 2 * DCn * 16 * 128));
                            for (int pp = 0; pp < kBN / 16; ++pp) {
                                if (ids[pp] < 0)
                                    continue;
                                for (int dc = 0; dc < DCn; ++dc) {
                                    tma_load_4d(kdst + dc * C::SUB + pp * 2048, &p.tm_kc, bar_full(st), dc * 64, 0, g, ids[pp]);
                                    tma_load_4d(vdst + dc * C::SUB + pp * 2048, &p.tm_vc, bar_full(st), dc * 64, 0, g, ids[pp]);
                                }
                            }
                        }
                    } else {
                        const int32_t ct = t - s.n_ctx;
                        mbar_arrive_expect_tx(bar_full(st), (uint32_t)(2 * DCn * CB * 128));
                        const int32_t row = off + ct * CB;
                        for (int dc = 0; dc < DCn; ++dc) {
                            tma_load_3d(kdst + dc * C::SUB, &p.tm_kn, bar_full(st), dc * 64, g, row);
                            tma_load_3d(vdst + dc * C::SUB, &p.tm_vn, bar_full(st), dc * 64, g, row);
                        }
                    }
                }
                u += (s.t1 - s.t0);
            }
            const uint32_t first = it > (uint32_t)C::STAGES ? it - C::STAGES : 0;
            if (!ok) {
                // drain: wait (bounded) for every stage armed but not yet consumed
                volatile int drain_abort = 0;
                for (uint32_t k = first; k < it; ++k)
                    mbar_wait(bar_full(k % C::STAGES), (k / C::STAGES) & 1, &drain_abort);
            } else {
                // tail: the release of every stage (a tensor-core commit on bar_empty) has
                // landed before the CTA exits
                for (uint32_t k = first; k < it; ++k)
                    mbar_wait(bar_empty(k % C::STAGES), (k / C::STAGES) & 1, abort_flag);
            }
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            const uint32_t idesc_pv = idesc_bf16_f32(kRows, D, false, true);
            uint32_t it = 0, nseg = 0;
            bool ok = true;
            for (int64_t u = cta_s; u < cta_e && ok;) {
                Seg s;
                make_seg(p, sh, u, cta_e, cta_s, s);
                if (!(ok = mbar_wait(bar_qfull, nseg & 1, abort_flag)))
                    break;
                tc_fence_after();
                const int32_t nt = s.t1 - s.t0;
                for (int32_t k = 0; k <= nt && ok; ++k) {
                    // S for tile k (if any), then PV for tile k-1
                    if (k < nt) {
                        const uint32_t itk = it + k;
                        const int st = itk % C::STAGES;
                        const int b = itk & 1;
                        const int32_t t = s.t0 + k;
                        const int32_t keys = (t < s.n_ctx) ? kBN : CB;
                        if (!(ok = mbar_wait(bar_full(st), (itk / C::STAGES) & 1, abort_flag)))
                            break;
                        if (!(ok = mbar_wait(bar_sfree(b), ((itk >> 1) & 1) ^ 1, abort_flag)))
                            break;
                        tc_fence_after();
                        const uint32_t idesc_s = idesc_bf16_f32(kRows, keys, false, false);
                        const uint32_t kbase = sbase + C::OFF_KV + st * C::STAGE;
                        // descriptors formed once; a 16-byte step is +1 in the address field
                        const uint64_t qd = sw128_desc(sbase + C::OFF_Q, 16, 1024);
                        const uint64_t kd = sw128_desc(kbase, 16, 1024);
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks)
                            tc_mma_ss(tmem + C::TMEM_S + b * kBN,
                                      qd + (uint64_t)((ks >> 2) * (C::QSUB >> 4) + (ks & 3) * 2),
                                      kd + (uint64_t)((ks >> 2) * (C::SUB >> 4) + (ks & 3) * 2), idesc_s,
                                      ks > 0 ? 1u : 0u);
                        tc_commit(bar_sfull(b));
                        if (k == nt - 1)
                            tc_commit(bar_qempty);   // Q no longer read by this segment
                    }
                    if (k > 0) {
                        const uint32_t itp = it + k - 1;
                        const int st = itp % C::STAGES;
                        const int32_t t = s.t0 + k - 1;
                        const int32_t keys = (t < s.n_ctx) ? kBN : CB;
                        if (k == 1 && nseg > 0 &&
                            !(ok = mbar_wait(bar_ofree, (nseg - 1) & 1, abort_flag)))
                            break;
                        if (!(ok = mbar_wait(bar_pfull, itp & 1, abort_flag)))
                            break;
                        tc_fence_after();
                        const uint32_t vbase = sbase + C::OFF_KV + st * C::STAGE + C::KV_BYTES;
                        const uint64_t pd = sw128_desc(sbase + C::OFF_P, 16, 1024);
                        const uint64_t vd = sw128_desc(vbase, C::SUB, 1024);
                        const uint32_t acc0 = k == 1 ? 0u : 1u;
                        const int nks = keys / 16;
#pragma unroll
                        for (int ks = 0; ks < kBN / 16; ++ks)
                            if (ks < nks)
                                tc_mma_ss(tmem + C::TMEM_O, pd + (uint64_t)(ks * 2), vd + (uint64_t)(ks * 128),
                                          idesc_pv, ks ? 1u : acc0);
                        tc_commit(bar_pvdone);
                        tc_commit(bar_empty(st));
                    }
                }
                it += nt;
                ++nseg;
                u += nt;
            }
            // make sure no MMA is still running before TMEM is released
            tc_commit(bar_drain);
            volatile int drain_abort = 0;
            mbar_wait(bar_drain, 0, &drain_abort);
            // tail: the arrives of the last Q-release and S-buffer commits have landed
            if (ok && nseg > 0)
                mbar_wait(bar_qempty, (nseg - 1) & 1, abort_flag);
            for (uint32_t back = 1; ok && back <= 2 && back <= it; ++back)
                mbar_wait(bar_sfull((it - back) & 1), ((it - back) >> 1) & 1, abort_flag);
        }
    } else {
        // ============================================================ softmax / epilogue
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;                // query row of the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int stid = tid - kSoftmaxWarp0 * 32;        // 0..127
        uint32_t it = 0, nseg = 0;
        bool ok = true;
        // A wait that gives up does not leave the loops: the thread runs on (later waits
        // return at once) and the four warps leave together at the next barrier they share.
        for (int64_t u = cta_s; u < cta_e;) {
            Seg s;
            make_seg(p, sh, u, cta_e, cta_s, s);
            const int32_t off = __ldg(p.cu_slots + s.i);
            const int32_t k_i = __ldg(p.cu_slots + s.i + 1) - off;
            const int32_t L = p.ctx_len ? __ldg(p.ctx_len + s.i) : 0;
            const int32_t j = s.rb * p.R + r / p.HP;      // candidate row of this thread
            const int32_t hh = r % p.HP;
            const bool active = (r < p.HP * p.R) && (j < k_i);
            const bool warp_active = __any_sync(0xffffffffu, active) != 0;
            float m_run = -INFINITY, l_run = 0.0f;
            const int32_t nt = s.t1 - s.t0;
            for (int32_t k = 0; k < nt; ++k, ++it) {
                const int32_t t = s.t0 + k;
                const int b = it & 1;
                const bool is_ctx = t < s.n_ctx;
                const int32_t keys = is_ctx ? kBN : CB;
                // keys of this tile visible to this row: always a prefix [0, nvis)
                int32_t nvis;
                if (is_ctx)
                    nvis = min(kBN, L - t * kBN);
                else
                    nvis = max(0, min(CB, j - (t - s.n_ctx) * CB + 1));
                if (!active)
                    nvis = 0;
                // keys of this tile that hold real data (rows >= kvalid are zeroed in V)
                int32_t kvalid;
                if (is_ctx)
                    kvalid = min(kBN, L - t * kBN);
                else
                    kvalid = max(0, min(CB, min(k_i, (s.rb + 1) * p.R) - (t - s.n_ctx) * CB));
                ok &= mbar_wait(bar_sfull(b), (it >> 1) & 1, abort_flag);
                __syncwarp();
                tc_fence_after();
                float sv[kBN];
                if (warp_active) {
                    const uint32_t sa = tmem + lane_off + C::TMEM_S + b * kBN;
                    if (keys == kBN) {
                        uint32_t ra[32], rb2[32];
                        tmem_ld32(sa, ra);
                        tmem_ld32(sa + 32, rb2);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            sv[e] = __uint_as_float(ra[e]);
                            sv[e + 32] = __uint_as_float(rb2[e]);
                        }
                    } else {
                        uint32_t ra[16];
                        tmem_ld16(sa, ra);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            sv[e] = __uint_as_float(ra[e]);
#pragma unroll
                        for (int e = 16; e < kBN; ++e)
                            sv[e] = 0.0f;
                    }
                }
                // S buffer b may now be overwritten by the next S MMA
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar_sfree(b));

                float mt = -INFINITY;
#pragma unroll
                for (int e = 0; e < kBN; ++e)
                    if (e < nvis)
                        mt = fmaxf(mt, sv[e] * p.scale_log2);
                const float m_new = fmaxf(m_run, mt);
                const bool grow = m_new > m_run + kRescaleLog2;   // also m_run == -inf
                const float alpha = grow ? fast_exp2(m_run - m_new) : 1.0f;
                if (grow) {
                    l_run *= alpha;
                    m_run = m_new;
                }
                // P (shared) and O (TMEM) are in use by PV of the previous tile
                if (it > 0)
                    ok &= mbar_wait(bar_pvdone, (it - 1) & 1, abort_flag);
                __syncwarp();
                tc_fence_after();
                if (k > 0 && __any_sync(0xffffffffu, grow && active)) {
                    // rescale this warp's rows of O
                    const float a = (grow && active) ? alpha : 1.0f;
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t ro[32];
                        const uint32_t oa = tmem + lane_off + C::TMEM_O + c * 32;
                        tmem_ld32(oa, ro);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            ro[e] = __float_as_uint(__uint_as_float(ro[e]) * a);
                        tmem_st32(oa, ro);
                    }
                    tmem_wait_st();
                }
                // P row of this thread: 64 keys = 8 swizzled 16-byte chunks
                const uint32_t prow = sbase + C::OFF_P + r * 128;
                float lsum = 0.0f;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint32_t w4[4];
#pragma unroll
                    for (int h2 = 0; h2 < 4; ++h2) {
                        const int e = c * 8 + h2 * 2;
                        const float p0 = (e < nvis) ? fast_exp2(fmaf(sv[e], p.scale_log2, -m_run)) : 0.0f;
                        const float p1 = (e + 1 < nvis) ? fast_exp2(fmaf(sv[e + 1], p.scale_log2, -m_run)) : 0.0f;
                        lsum += p0 + p1;
                        w4[h2] = pack_bf16x2(p0, p1);
                    }
                    st_shared_v4(prow + ((c ^ (r & 7)) << 4), w4[0], w4[1], w4[2], w4[3]);
                }
                l_run += lsum;
                // zero V rows that hold no data of this request (NaN-safe PV)
                if (kvalid < keys) {
                    const uint32_t vbase = sbase + C::OFF_KV + (it % C::STAGES) * C::STAGE + C::KV_BYTES;
                    const int32_t chunks = (keys - kvalid) * 8 * DCn;
                    for (int32_t x = stid; x < chunks; x += 128) {
                        const int32_t row = kvalid + x / (8 * DCn);
                        const int32_t rem = x % (8 * DCn);
                        const int32_t dc = rem / 8, c16 = rem % 8;
                        st_shared_v4(vbase + dc * C::SUB + row * 128 + c16 * 16, 0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar_pfull);
            }
            // ---- epilogue: O of this segment is complete after the last PV
            ok &= mbar_wait(bar_pvdone, (it - 1) & 1, abort_flag);
            __syncwarp();
            tc_fence_after();
            const int32_t h = s.hg * p.HP + hh;
            const int64_t orow = (int64_t)(off + j) * p.hq + h;
            if (s.single) {
                const float inv = 1.0f / l_run;
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t ro[32];
                    if (warp_active) {
                        tmem_ld32(tmem + lane_off + C::TMEM_O + c * 32, ro);
                        tmem_wait_ld();
                    }
                    if (active) {
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            pk[e] = pack_bf16x2(__uint_as_float(ro[2 * e]) * inv,
                                                __uint_as_float(ro[2 * e + 1]) * inv);
                        uint4 *dst = reinterpret_cast<uint4 *>(
                            reinterpret_cast<uint16_t *>(p.out) + orow * D + c * 32);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    }
                }
                if (active && p.lse)
                    p.lse[orow] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar_ofree);
            } else {
                // unnormalised partial of this piece
                const int32_t slot = 2 * blockIdx.x + (s.first_of_cta ? 0 : 1);
                float *po = p.part_o + ((int64_t)slot * kRows + r) * D;
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t ro[32];
                    if (warp_active) {
                        tmem_ld32(tmem + lane_off + C::TMEM_O + c * 32, ro);
                        tmem_wait_ld();
                    }
                    if (active) {
                        float4 *dst = reinterpret_cast<float4 *>(po + c * 32);
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            __stcg(dst + v, make_float4(__uint_as_float(ro[4 * v]), __uint_as_float(ro[4 * v + 1]),
                                                        __uint_as_float(ro[4 * v + 2]), __uint_as_float(ro[4 * v + 3])));
                    }
                }
                if (active)
                    __stcg(p.part_ml + (int64_t)slot * kRows + r, make_float2(m_run, l_run));
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar_ofree);
                __threadfence();
                if (named_bar_any(1, 128, !ok))
                    break;   // all four warps leave here together
                if (stid == 0) {
                    const int32_t C0 = ncta;
                    const int32_t cf = cta_of_unit(s.u_pair0, sh.total, C0);
                    const int32_t cl = cta_of_unit(s.u_pair0 + s.n_tiles - 1, sh.total, C0);
                    const int prev = atomicAdd(p.tickets + s.pair, 1);
                    *flag_last = (prev == cl - cf) ? 1 : 0;
                }
                named_bar_sync(1, 128);
                if (*flag_last) {
                    __threadfence();
                    const int32_t C0 = ncta;
                    const int32_t cf = cta_of_unit(s.u_pair0, sh.total, C0);
                    const int32_t cl = cta_of_unit(s.u_pair0 + s.n_tiles - 1, sh.total, C0);
                    if (active) {
                        float M = -INFINITY;
                        for (int32_t c = cf; c <= cl; ++c) {
                            const int64_t cs = cta_start(sh.total, c, C0);
                            const int32_t sl = 2 * c + ((c == cf && cs < s.u_pair0) ? 1 : 0);
                            M = fmaxf(M, __ldcg(p.part_ml + (int64_t)sl * kRows + r).x);
                        }
                        float Lsum = 0.0f;
                        for (int32_t c = cf; c <= cl; ++c) {
                            const int64_t cs = cta_start(sh.total, c, C0);
                            const int32_t sl = 2 * c + ((c == cf && cs < s.u_pair0) ? 1 : 0);
                            const float2 ml = __ldcg(p.part_ml + (int64_t)sl * kRows + r);
                            Lsum += ml.y * fast_exp2(ml.x - M);
                        }
                        const float inv = 1.0f / Lsum;
                        for (int c32 = 0; c32 < D / 32; ++c32) {
                            float acc[32];
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                acc[e] = 0.0f;
                            for (int32_t c = cf; c <= cl; ++c) {
                                const int64_t cs = cta_start(sh.total, c, C0);
                                const int32_t sl = 2 * c + ((c == cf && cs < s.u_pair0) ? 1 : 0);
                                const float wgt = fast_exp2(__ldcg(p.part_ml + (int64_t)sl * kRows + r).x - M);
                                const float4 *src = reinterpret_cast<const float4 *>(
                                    p.part_o + ((int64_t)sl * kRows + r) * D + c32 * 32);
#pragma unroll
                                for (int v = 0; v < 8; ++v) {
                                    const float4 x = __ldcg(src + v);
                                    acc[4 * v + 0] += wgt * x.x;
                                    acc[4 * v + 1] += wgt * x.y;
                                    acc[4 * v + 2] += wgt * x.z;
                                    acc[4 * v + 3] += wgt * x.w;
                                }
                            }
                            uint32_t pk[16];
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                pk[e] = pack_bf16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv);
                            uint4 *dst = reinterpret_cast<uint4 *>(
                                reinterpret_cast<uint16_t *>(p.out) + orow * D + c32 * 32);
#pragma unroll
                            for (int v = 0; v < 4; ++v)
                                dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                        }
                        if (p.lse)
                            p.lse[orow] = (M + __log2f(Lsum)) * 0.69314718055994531f;
                    }
                    named_bar_sync(1, 128);
                    if (stid == 0)
                        p.tickets[s.pair] = 0;
                }
            }
            ++nseg;
            u += nt;
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // read once every role has finished, so that a wait given up late is reported too
    if (*abort_flag && tid == 0) {
        set_status(p.status, SVP_DEV_TIMEOUT);
        *reinterpret_cast<volatile int32_t *>(p.status + kWsPoisonWord) = 1;
    }
    if (warp == 1)
        tmem_dealloc(tmem, C::TMEM_COLS);
}

// ------------------------------------------------------------------------ host side
template <int D>
static svp_status launch_d(const TcParams &p, int grid, cudaStream_t stream)
{
    using C = TcCfg<D>;
    static std::atomic<uint64_t> configured{0};
    if (set_smem_limit_once(attn_tc_kernel<D>, C::SMEM, configured) != cudaSuccess)
        return SVP_ECUDA;
    attn_tc_kernel<D><<<grid, kThreads, C::SMEM, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? SVP_OK : SVP_ECUDA;
}

svp_status attn_tc_launch(const TcParams &p, int d, int grid, cudaStream_t stream)
{
    switch (d) {
    case 64: return launch_d<64>(p, grid, stream);
    case 128: return launch_d<128>(p, grid, stream);
    case 256: return launch_d<256>(p, grid, stream);
    default: return SVP_EUNSUPPORTED;
    }
}

int attn_tc_max_prefix() { return kMaxPrefix; }
int attn_tc_block_keys() { return kBN; }

}  // namespace svp
