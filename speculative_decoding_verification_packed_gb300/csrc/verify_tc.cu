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
// maximum of each row is a stale reference m_ref, seeded on the first tile of a piece
// with the score of its first key: P = 2^(s*c - m_ref) is used while no visible score
// exceeds m_ref + 32 (bf16 P and the fp32 accumulators hold 2^32 exactly in relative
// terms); only then the softmax warps reduce the row maxima across keys, move m_ref,
// and rescale O^T and l^T in TMEM.  Inactive rows carry m_ref = +inf, so their P is 0
// without per-element masks.
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
constexpr int kVThreads = 224;   // producer, S issuer, 4 softmax warps, PV issuer
constexpr int kSlotBytes = 32768;   // [128 keys][128 d] bf16 = 2 x [128][64] SW128
constexpr int kSubBytes = 16384;    // [128 keys][64 d]
constexpr float kSlack = 32.0f;     // P <= 2^32 (exact in bf16 / fp32 accumulation)

// Shared per-row softmax state (in the misc region).
constexpr int kReqCache = 256;      // requests whose (offset, context length) sit in smem
constexpr int kPairCost = 4;        // partition cost of starting a pair (segment switch + merge), in tiles

struct VtRows {
    float m_ref[128];
    float alpha[128];
    union {
        float red[4][128];   // rare path: per-quarter row maxima
        float wts[8][128];   // merge: per-piece weight of each row
    };
    int32_t jr[128];     // candidate index of the row (INT_MAX for padding rows)
    float lrow[128];
    int64_t orow[128];   // epilogue: output element offset of row r (-1: not a live row)
    float linv[128];     // epilogue: 1 / l of row r
    int32_t flag[2];
    int32_t rescale;
    int32_t last;
    int32_t abort_flag;
    uint32_t tmem;
    int32_t warp_sums[8];
    int32_t warp_costs[8];
    int32_t req_off[kReqCache];
    int32_t req_len[kReqCache];
    int32_t req_ctx[kReqCache];   // contiguous context: first token row (< 2^31, host-checked)
    int32_t pslot[256];   // merge: partial slot of each piece (pieces <= CTAs <= 256)
    int32_t npend;        // merges this CTA owes (it delivered the last piece of a pair)
    uint32_t v_seen;      // tiles whose V fill the PV issuer has seen land (S issuer reads it)
    int32_t pend[2][8];   // pair, cf, cl, nact, out_row0, hg, u_pair0 (lo, hi)
};

__device__ __forceinline__ int32_t rs_req_off(const VtRows *rs, const TcParams &p, int32_t i)
{
    return i < kReqCache ? rs->req_off[i] : __ldg(p.cu_slots + i);
}

__device__ __forceinline__ int32_t rs_req_len(const VtRows *rs, const TcParams &p, int32_t i)
{
    if (i < kReqCache)
        return rs->req_len[i];
    return p.ctx_len ? __ldg(p.ctx_len + i) : 0;
}

__device__ __forceinline__ int32_t rs_req_ctx(const VtRows *rs, const TcParams &p, int32_t i)
{
    return i < kReqCache ? rs->req_ctx[i] : (int32_t)__ldg(p.cu_ctx + i);
}

// The CTAs split the KV tiles of all (request, row block, head group) pairs in order, in
// equal shares of a cost that charges every pair cost0 tiles at its start: the CTA that
// starts a pair also pays the segment switch into it and, as a rule, the pair's merge.
// prefix[q] / cprefix[q]: tiles / cost before (request, row block) q (each of its HG pairs
// has nt tiles and costs nt + cost0, or nothing when nt = 0).
// First tile at or after cost unit v (v <= ctot).
__device__ __forceinline__ int32_t vt_tile_of_cost(const int32_t *prefix, const int32_t *cprefix,
                                                   int32_t nq, int32_t hg_n, int32_t cost0,
                                                   int32_t v)
{
    if (v >= cprefix[nq])
        return prefix[nq];
    int32_t lo = 0, hi = nq;
    while (hi - lo > 1) {
        const int32_t mid = (lo + hi) >> 1;
        if (cprefix[mid] <= v)
            lo = mid;
        else
            hi = mid;
    }
    while (cprefix[lo + 1] <= v)
        ++lo;
    const int32_t pc = (cprefix[lo + 1] - cprefix[lo]) / hg_n;   // nt + cost0
    const int32_t nt = pc - cost0;
    const int32_t lc = v - cprefix[lo];
    const int32_t hg = lc / pc;
    const int32_t loc = lc - hg * pc;
    return prefix[lo] + hg * nt + (loc > cost0 ? loc - cost0 : 0);
}

// CTA c owns tiles [ctile[c], ctile[c+1]); the owner of tile u is the last c with
// ctile[c] <= u (CTAs with an empty range never own a tile inside a pair).
__device__ __forceinline__ int32_t vt_cta_of_unit(const int32_t *ctile, int32_t ncta, int64_t u)
{
    int32_t lo = 0, hi = ncta;   // ctile[lo] <= u < ctile[hi]
    while (hi - lo > 1) {
        const int32_t mid = (lo + hi) >> 1;
        if (ctile[mid] <= u)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

struct VtSeg {
    int32_t i, rb, hg, t0, t1, n_ctx, n_tiles, first_of_cta, single, pair;
    int64_t u_pair0;
};

// Per-request inputs, read together (one memory round trip in the prologue).
struct VtReq {
    int32_t off, end, L;
    int64_t c0;
};

__device__ __forceinline__ VtReq vt_req_load(const TcParams &p, int32_t i)
{
    VtReq r;
    r.off = __ldg(p.cu_slots + i);
    r.end = __ldg(p.cu_slots + i + 1);
    r.L = p.ctx_len ? __ldg(p.ctx_len + i) : 0;
    r.c0 = (!p.paged && p.cu_ctx) ? __ldg(p.cu_ctx + i) : 0;
    return r;
}

// KV tiles of (request, row block rb): context tiles of 128 keys, then candidate
// tiles of CB keys up to the last candidate this row block needs.
__device__ __forceinline__ void vt_units(const TcParams &p, const VtReq &q, int32_t rb,
                                         int32_t &n_tiles, int32_t &bad)
{
    n_tiles = 0;
    bad = 0;
    const int32_t k = q.end - q.off;
    if (q.off < 0 || q.end < q.off || k > p.w || q.end > p.m_cap) {
        bad = SVP_DEV_BAD_SLOTS;
        return;
    }
    const int32_t L = q.L;
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
        } else if (q.c0 < 0 || q.c0 + L > p.total_tokens) {
            bad = SVP_DEV_BAD_CONTEXT;
            return;
        }
    }
    const int32_t r0 = rb * p.R;
    if (r0 >= k)
        return;
    const int32_t cmax = min(k, r0 + p.R);
    n_tiles = (L + kVK - 1) / kVK + (cmax + p.CB - 1) / p.CB;
}

__device__ __forceinline__ void vt_seg(const TcParams &p, const VtRows *rs, const int32_t *prefix,
                                       int32_t nq, int64_t u, int64_t ue, int64_t cta_s, VtSeg &s)
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
    const int32_t local = (int32_t)(u - prefix[q]);   // < per * HG: fits 32 bits
    s.i = q / p.RB;
    s.rb = q - s.i * p.RB;
    s.hg = local / per;
    s.t0 = local - s.hg * per;
    s.n_tiles = per;
    s.u_pair0 = prefix[q] + (int64_t)s.hg * per;
    const int64_t seg_end = min(ue, s.u_pair0 + per);
    s.t1 = s.t0 + (int32_t)(seg_end - u);
    const int32_t L = rs_req_len(rs, p, s.i);
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

// P for one 32-row chunk of this thread's key: y = s*c - m_ref, P = 2^y (0 where the
// key is not visible).  ymax collects the largest visible y (the hit test).
// cand: candidate tile, key index ckey must be <= the row's candidate index.
__device__ __forceinline__ void vt_chunk(const uint32_t (&sr)[32], uint32_t mref_addr,
                                         uint32_t jr_addr, bool key_ok, bool cand, int ckey,
                                         float cl2, uint32_t *pk, float &ymax)
{
    float y[32];
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        const float4 m = ld_shared_f4(mref_addr + 16 * v);
        y[4 * v + 0] = fmaf(__uint_as_float(sr[4 * v + 0]), cl2, -m.x);
        y[4 * v + 1] = fmaf(__uint_as_float(sr[4 * v + 1]), cl2, -m.y);
        y[4 * v + 2] = fmaf(__uint_as_float(sr[4 * v + 2]), cl2, -m.z);
        y[4 * v + 3] = fmaf(__uint_as_float(sr[4 * v + 3]), cl2, -m.w);
    }
    if (cand) {
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            const int4 j = ld_shared_i4(jr_addr + 16 * v);
            if (ckey > j.x) y[4 * v + 0] = -INFINITY;
            if (ckey > j.y) y[4 * v + 1] = -INFINITY;
            if (ckey > j.z) y[4 * v + 2] = -INFINITY;
            if (ckey > j.w) y[4 * v + 3] = -INFINITY;
        }
    }
    if (!key_ok) {
#pragma unroll
        for (int e = 0; e < 16; ++e)
            pk[e] = 0u;
        return;
    }
    float t16[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
        t16[e] = fmaxf(y[2 * e], y[2 * e + 1]);
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int e = 0; e < w; ++e)
            t16[e] = fmaxf(t16[e], t16[e + w]);
    ymax = fmaxf(ymax, t16[0]);
#pragma unroll
    for (int e = 0; e < 16; ++e)
        pk[e] = pack_bf16x2(fast_exp2(y[2 * e]), fast_exp2(y[2 * e + 1]));
}

// One contiguous global -> shared copy on the async proxy, completing on an mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// A position in the TMA ring: slot index and the parity of that slot's current use.
// Tracked incrementally so that no role divides by the (runtime) slot count on its loop.
struct RingPos {
    uint32_t slot, phase;
};

__device__ __forceinline__ RingPos ring_add(RingPos r, uint32_t n, uint32_t nslot)
{
    r.slot += n;
    while (nslot != 0 && r.slot >= nslot) {   // (a ring always has slots; never spin on 0)
        r.slot -= nslot;
        r.phase ^= 1u;
    }
    return r;
}

// Bounded wait until a shared-memory counter that another warp of the CTA advances reaches
// need; the fences pair with the writer's, so what the writer had observed before its store
// (here: an mbarrier phase that completed) is observed by the caller after it returns.
__device__ __forceinline__ bool vt_wait_count(const uint32_t *cnt, uint32_t need,
                                              volatile int *abort_flag)
{
    const volatile uint32_t *c = cnt;
    if (*c >= need) {
        __threadfence_block();
        return true;
    }
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        __nanosleep(64);
        if (*c >= need) {
            __threadfence_block();
            return true;
        }
        if ((i & 15u) == 0) {
            if (*abort_flag)
                return false;
            if ((int64_t)(global_ns() - t0) > (int64_t)kWaitLimitNs) {
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// One merge pass over NB partial slabs staged in shared memory: column block h (128 columns
// of d) of each piece, row-major [nact][128] fp32 at ring + q * slab.  acc_r = run_r +
// sum_q w_q[r] * slab_q[r]; the last pass of the block scales by 1/L and writes bf16
// output, earlier ones keep the running sum in the first piece's slot.  Each of the 128
// threads owns four columns and takes eight rows at once so that the shared-memory reads of
// all NB x 8 operands are in flight together.
template <int NB, int D>
__device__ __forceinline__ void vt_merge_pass(const TcParams &p, const VtRows *rs, uint32_t ring,
                                              uint32_t slab, int32_t wq0, int32_t nact, int32_t slot0,
                                              int h, bool first_pass, bool last_pass, int stid)
{
    constexpr int C4 = 128 / 4;
    constexpr int RGS = 128 / C4;
    constexpr int RU = 8;
    const int col4 = stid % C4, rg = stid / C4;
    float4 *run = reinterpret_cast<float4 *>(p.part_o + ((int64_t)slot0 * (D / 128) + h) * kRows * 128) + col4;
    uint16_t *out = reinterpret_cast<uint16_t *>(p.out) + h * 128 + col4 * 4;
    const uint32_t col_b = (uint32_t)col4 * 16u;
    for (int r0 = rg; r0 < nact; r0 += RU * RGS) {
        float4 acc[RU];
        int rr[RU];
#pragma unroll
        for (int k = 0; k < RU; ++k) {
            rr[k] = min(r0 + k * RGS, nact - 1);   // padded lanes recompute the last row
            acc[k] = first_pass ? make_float4(0.f, 0.f, 0.f, 0.f) : __ldcg(run + (int64_t)rr[k] * C4);
        }
#pragma unroll
        for (int q = 0; q < NB; ++q) {
            float4 x[RU];
            float w[RU];
#pragma unroll
            for (int k = 0; k < RU; ++k) {
                x[k] = ld_shared_f4(ring + q * slab + (uint32_t)rr[k] * (128 * 4) + col_b);
                w[k] = rs->wts[wq0 + q][rr[k]];
            }
#pragma unroll
            for (int k = 0; k < RU; ++k) {
                acc[k].x += w[k] * x[k].x;
                acc[k].y += w[k] * x[k].y;
                acc[k].z += w[k] * x[k].z;
                acc[k].w += w[k] * x[k].w;
            }
        }
#pragma unroll
        for (int k = 0; k < RU; ++k) {
            const int r = r0 + k * RGS;
            if (r >= nact)
                break;
            if (!last_pass) {
                __stcg(run + (int64_t)r * C4, acc[k]);
            } else {
                const float inv = rs->linv[r];
                uint2 pk2;
                pk2.x = pack_bf16x2(acc[k].x * inv, acc[k].y * inv);
                pk2.y = pack_bf16x2(acc[k].z * inv, acc[k].w * inv);
                *reinterpret_cast<uint2 *>(out + rs->orow[r]) = pk2;
            }
        }
    }
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
    auto bar_pfull = [&](int b) { return bar0 + 8u * (22 + b); };    // per P buffer
    auto bar_pvdone = [&](int b) { return bar0 + 8u * (24 + b); };   // per P buffer
    const uint32_t bar_ofree = bar0 + 8u * 26, bar_drain = bar0 + 8u * 27;
    const uint32_t bar_merge = bar0 + 8u * 28;
    const uint32_t bar_tick = bar0 + 8u * 29;   // merges owed by this CTA are known
    const int nP = p.nP;                                          // P buffers (1 or 2)
    auto pbuf = [&](uint32_t x) -> int { return nP == 2 ? (int)(x & 1u) : 0; };
    auto ppar = [&](uint32_t x) -> uint32_t { return (nP == 2 ? (x >> 1) : x) & 1u; };
    const uint32_t PBYTES = (uint32_t)((NR + 63) / 64) * 16384u;

    VtRows *rs = reinterpret_cast<VtRows *>(smem + p.off_misc);
    volatile int *abort_flag = &rs->abort_flag;
    const int32_t NQ = p.n * p.RB;
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + p.off_pref);   // [NQ + 1]
    int32_t *cprefix = prefix + (NQ + 1);                                 // [NQ + 1]
    int32_t *ctile = cprefix + (NQ + 1);                                  // [gridDim.x + 1]
    // a chained launch: the next kernel may be scheduled from here on; this one reads
    // nothing before the previous kernel on the stream has completed
    griddep_launch_dependents();
    griddep_wait();
    // start the workspace-signature load early; it is checked after the prologue
    const int32_t sig_seen = (tid == 0) ? *reinterpret_cast<volatile int32_t *>(p.status + 1) : 0;
    const int32_t poison_seen =
        (tid == 0) ? *reinterpret_cast<volatile int32_t *>(p.status + kWsPoisonWord) : 0;

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
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_pfull(b), 4);
            mbar_init(bar_pvdone(b), 1);
        }
        mbar_init(bar_ofree, 4);
        mbar_init(bar_drain, 2);   // one commit from each MMA issuer
        mbar_init(bar_merge, 1);
        mbar_init(bar_tick, 1);
        mbar_fence_init();
        rs->abort_flag = 0;
        rs->flag[0] = rs->flag[1] = 0;
        rs->rescale = 0;
        rs->npend = 0;
        rs->v_seen = 0;
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

    // prefix sums of KV tiles and of partition cost over (request, row block)
    int32_t bad_bits = 0;
    if (tid == 0) {
        prefix[0] = 0;
        cprefix[0] = 0;
    }
    int32_t running = 0, crunning = 0;
    for (int32_t base = 0; base < NQ; base += kVThreads) {
        const int32_t q = base + tid;
        int32_t units = 0, costs = 0;
        if (q < NQ) {
            const int32_t i = q / p.RB, rb = q - i * p.RB;
            const VtReq rq = vt_req_load(p, i);
            int32_t nt, bad;
            vt_units(p, rq, rb, nt, bad);
            bad_bits |= bad;
            units = nt * p.HG;
            costs = nt > 0 ? (nt + p.cost0) * p.HG : 0;
            if (rb == 0 && i < kReqCache) {
                rs->req_off[i] = rq.off;
                rs->req_len[i] = rq.L;
                rs->req_ctx[i] = (p.total_tokens > 0) ? (int32_t)rq.c0 : 0;
            }
        }
        int32_t incl = units, cincl = costs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
            const int32_t cv = __shfl_up_sync(0xffffffffu, cincl, o);
            if (lane >= o) {
                incl += v;
                cincl += cv;
            }
        }
        __syncthreads();
        if (lane == 31) {
            rs->warp_sums[warp] = incl;
            rs->warp_costs[warp] = cincl;
        }
        __syncthreads();
        int32_t before = running, cbefore = crunning;
        for (int w2 = 0; w2 < warp; ++w2) {
            before += rs->warp_sums[w2];
            cbefore += rs->warp_costs[w2];
        }
        if (q < NQ) {
            prefix[q + 1] = before + incl;
            cprefix[q + 1] = cbefore + cincl;
        }
        for (int w2 = 0; w2 < kVThreads / 32; ++w2) {
            running += rs->warp_sums[w2];
            crunning += rs->warp_costs[w2];
        }
    }
    if (bad_bits && blockIdx.x == 0)
        set_status(p.status, bad_bits);
    if (tid == 0) {
        // the workspace layout must match this call's (head_dim, tile mode), and no earlier
        // launch may have given up mid-flight (its tickets would be stale)
        const int32_t seen = sig_seen;
        rs->last = ((seen != 0 && seen != p.sig) || poison_seen != 0) ? 1 : 0;
        if (rs->last && blockIdx.x == 0)
            set_status(p.status, SVP_DEV_WORKSPACE);
        if (seen == 0 && blockIdx.x == 0)
            p.status[1] = p.sig;
    }
    __syncthreads();
    // tile range of every CTA: equal shares of the partition cost
    const int64_t total = rs->last ? 0 : prefix[NQ];
    const int32_t ctot = cprefix[NQ];
    const int32_t ncta = total > 0 ? (int32_t)((int64_t)gridDim.x < (int64_t)ctot ? gridDim.x : ctot) : 0;
    for (int32_t c = tid; c <= ncta; c += kVThreads)
        ctile[c] = vt_tile_of_cost(prefix, cprefix, NQ, p.HG, p.cost0,
                                   (int32_t)((int64_t)c * ctot / (ncta > 0 ? ncta : 1)));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = rs->tmem;
    int64_t cta_s = 0, cta_e = 0;
    if ((int32_t)blockIdx.x < ncta) {
        cta_s = ctile[blockIdx.x];
        cta_e = ctile[blockIdx.x + 1];
    }
    const uint32_t TM_S = 0, TM_O = 2u * NR, TM_L = (2u + DH) * NR;

    if (warp == 0) {
        // ================================================================ producer
        // The whole warp runs the loop; lane 0 issues TMA.  For paged context the lanes
        // fetch a tile's page ids in parallel (shared by its K and V), one tile ahead.
        uint32_t it = 0, nseg = 0, seq = 0;
        RingPos wp = {0u, 0u};
        bool ok = true;
        const uint64_t pol_stream = l2_policy_evict_first();   // each KV byte is read once
        for (int64_t u = cta_s; u < cta_e && ok;) {
            VtSeg s;
            vt_seg(p, rs, prefix, NQ, u, cta_e, cta_s, s);
            const int32_t off = rs_req_off(rs, p, s.i);
            const int32_t L = rs_req_len(rs, p, s.i);
            const int32_t g = (s.hg * p.HP) / p.G;
            const int32_t npages = (L + 15) / 16;
            const int32_t *bt_row = p.paged ? p.block_table + (int64_t)s.i * p.max_pages : nullptr;
            ++nseg;
            const int32_t cctx = (!p.paged && L > 0) ? rs_req_ctx(rs, p, s.i) : 0;
            // page id of lane pp (< 8) for context tile t
            auto page_id = [&](int32_t t) -> int32_t {
                const int32_t pg = t * (kVK / 16) + lane;
                if (!p.paged || lane >= kVK / 16 || t >= s.n_ctx || pg >= npages)
                    return -1;
                return __ldg(bt_row + pg);
            };
            int32_t id_next = page_id(s.t0);
            for (int32_t t = s.t0; t < s.t1 && ok; ++t, ++it) {
                int32_t id = id_next;
                id_next = page_id(t + 1);                // prefetch the next tile's ids
                if (id >= p.num_pages || (id < 0 && p.paged && t < s.n_ctx &&
                                          lane < kVK / 16 && t * (kVK / 16) + lane < npages)) {
                    set_status(p.status, SVP_DEV_BAD_CONTEXT);
                    id = -1;
                }
                const uint32_t vmask = __ballot_sync(0xffffffffu, id >= 0);
                const int32_t nv = __popc(vmask);
                // K halves then V halves of this tile, one ring slot each
                for (int kv = 0; kv < 2 && ok; ++kv) {
                    const CUtensorMap *mc = kv ? &p.tm_vc : &p.tm_kc;
                    const CUtensorMap *mn = kv ? &p.tm_vn : &p.tm_kn;
                    for (int h = 0; h < DH; ++h, ++seq) {
                        const int sl = (int)wp.slot;
                        int w_ok = 1;
                        if (lane == 0)
                            w_ok = mbar_wait(bar_empty(sl), wp.phase ^ 1u, abort_flag);
                        wp = ring_add(wp, 1u, (uint32_t)nslot);
                        if (!(ok = __shfl_sync(0xffffffffu, w_ok, 0) != 0))
                            break;
                        const uint32_t dst = sbase + p.off_ring + sl * kSlotBytes;
                        if (t < s.n_ctx && p.paged) {
                            if (lane == 0)
                                mbar_arrive_expect_tx(bar_full(sl), (uint32_t)(nv * 2 * 2048));
                            __syncwarp();
                            if (id >= 0) {      // lane pp issues page pp
                                for (int c = 0; c < 2; ++c)
                                    tma_load_4d_hint(dst + c * kSubBytes + lane * 2048, mc, bar_full(sl),
                                                     h * 128 + c * 64, 0, g, id, pol_stream);
                            }
                        } else if (lane == 0) {
                            if (t < s.n_ctx) {
                                mbar_arrive_expect_tx(bar_full(sl), (uint32_t)kSlotBytes);
                                const int32_t row = cctx + t * kVK;
                                for (int c = 0; c < 2; ++c)
                                    tma_load_3d_hint(dst + c * kSubBytes, mc, bar_full(sl),
                                                     h * 128 + c * 64, g, row, pol_stream);
                            } else {
                                const int32_t ct = t - s.n_ctx;
                                mbar_arrive_expect_tx(bar_full(sl), (uint32_t)(2 * p.CB * 128));
                                for (int c = 0; c < 2; ++c)
                                    tma_load_3d(dst + c * kSubBytes, mn, bar_full(sl),
                                                h * 128 + c * 64, g, off + ct * p.CB);
                            }
                        }
                        __syncwarp();
                    }
                }
            }
            u += (s.t1 - s.t0);
        }
        if (lane == 0) {
            const uint32_t first = seq > (uint32_t)nslot ? seq - nslot : 0;
            if (!ok) {
                // the loads already issued land before the CTA exits
                volatile int drain_abort = 0;
                for (uint32_t k = first; k < seq; ++k)
                    mbar_wait(bar_full(k % nslot), (k / nslot) & 1, &drain_abort);
            } else {
                // tail: the release of every fill (a tensor-core commit arriving on
                // bar_empty) has landed before the CTA exits, so no asynchronous arrive
                // reaches this shared memory after it is handed to another CTA
                for (uint32_t k = first; k < seq; ++k)
                    mbar_wait(bar_empty(k % nslot), (k / nslot) & 1, abort_flag);
            }
        }
    } else if (warp == 1) {
        // ================================================================ S^T issuer
        // S^T = K Q^T of each tile into S buffer it & 1.  The tensor pipe accepts one MMA at
        // a time and a thread's later shared-memory operations queue behind its MMAs, so S
        // and PV are issued by two warps: each one blocks only on its own inputs and the
        // pipe always has the other's work queued.
        if (lane == 0) {
            uint32_t it = 0, nseg = 0;
            RingPos kpos = {0u, 0u};                     // ring position of K(it)
            bool ok = true;
            for (int64_t u = cta_s; u < cta_e && ok;) {
                VtSeg s;
                vt_seg(p, rs, prefix, NQ, u, cta_e, cta_s, s);
                const int32_t off = rs_req_off(rs, p, s.i);
                const int32_t k_i = (s.i + 1 < kReqCache && s.i + 1 < p.n ? rs->req_off[s.i + 1]
                                                                          : __ldg(p.cu_slots + s.i + 1)) - off;
                const int32_t kk = min(k_i - s.rb * p.R, p.R);
                const uint32_t NRs = (uint32_t)((p.HP * kk + 31) / 32 * 32);
                const uint32_t idesc_s = idesc_bf16_f32(128, NRs, false, false);
                const uint32_t qsub16 = QSUB >> 4;
                // Q of this segment replaces the previous one once its last S^T is done;
                // the KV stream of this segment is already under way meanwhile
                if (nseg > 0 && !(ok = mbar_wait(bar_qempty, (nseg - 1) & 1, abort_flag)))
                    break;
                mbar_arrive_expect_tx(bar_qfull, (uint32_t)((D / 64) * 64 * p.HP * p.R * 2));
                for (int dc = 0; dc < D / 64; ++dc)
                    tma_load_3d(sbase + p.off_q + dc * QSUB, &p.tm_q, bar_qfull, dc * 64,
                                s.hg * p.HP, off + s.rb * p.R);
                if (!(ok = mbar_wait(bar_qfull, nseg & 1, abort_flag))) {
                    volatile int drain_abort = 0;   // the Q copy lands before the CTA exits
                    mbar_wait(bar_qfull, nseg & 1, &drain_abort);
                    break;
                }
                const int32_t nt = s.t1 - s.t0;
                for (int32_t k = 0; k < nt; ++k, ++it) {
                    const int b = it & 1;
                    if (!(ok = mbar_wait(bar_sfree(b), ((it >> 1) & 1) ^ 1, abort_flag)))
                        break;
                    // K(it) half h goes into the slot whose previous fill was ring position
                    // pos - nslot.  When that fill was a V half (an odd slot count at
                    // d = 128), only the PV issuer has waited on it, and a parity wait here
                    // cannot tell "that V fill still in flight" from "this K fill landed"
                    // (both leave the barrier one phase short of, or at, the same parity).
                    // So first wait until the PV issuer has seen that V fill land; in the
                    // steady state it has (S(it) follows the softmax of it - 2, which
                    // follows PV's wait for the earlier tile's V).
                    uint32_t need = 0;
                    for (int h = 0; h < DH; ++h) {
                        const uint32_t pos = it * 2u * DH + (uint32_t)h;
                        if (pos >= (uint32_t)nslot) {
                            const uint32_t prev = pos - (uint32_t)nslot;
                            if (prev % (2u * DH) >= (uint32_t)DH)
                                need = max(need, prev / (2u * DH) + 1u);
                        }
                    }
                    if (need > 0 && !(ok = vt_wait_count(&rs->v_seen, need, abort_flag)))
                        break;
                    for (int h = 0; h < DH && ok; ++h) {
                        const RingPos q = ring_add(kpos, (uint32_t)h, (uint32_t)nslot);
                        ok = mbar_wait(bar_full(q.slot), q.phase, abort_flag);
                    }
                    if (!ok)
                        break;
                    tc_fence_after();
                    // descriptors formed up front, MMAs back to back (a 16-byte step in
                    // shared memory is +1 in a descriptor's address field)
                    for (int h = 0; h < DH; ++h) {
                        const uint64_t ad = sw128_desc(
                            sbase + p.off_ring + ring_add(kpos, (uint32_t)h, (uint32_t)nslot).slot * kSlotBytes,
                            16, 1024);
                        const uint64_t bd = sw128_desc(sbase + p.off_q + 2 * h * QSUB, 16, 1024);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            tc_mma_ss(tmem + TM_S + b * NR,
                                      ad + (uint64_t)((ks >> 2) * (kSubBytes >> 4) + (ks & 3) * 2),
                                      bd + (uint64_t)((ks >> 2) * qsub16 + (ks & 3) * 2), idesc_s,
                                      (h | ks) ? 1u : 0u);
                        // this half's slot is free once its MMAs are done
                        tc_commit(bar_empty(ring_add(kpos, (uint32_t)h, (uint32_t)nslot).slot));
                    }
                    tc_commit(bar_sfull(b));
                    if (k == nt - 1)
                        tc_commit(bar_qempty);   // Q no longer read by this segment
                    kpos = ring_add(kpos, 2u * DH, (uint32_t)nslot);
                }
                ++nseg;
                u += nt;
            }
            tc_commit(bar_drain);
            volatile int drain_abort = 0;
            mbar_wait(bar_drain, 0, &drain_abort);
            // tail: the arrives of this thread's last commits (Q released, last two S
            // buffers full) have landed before the CTA exits
            if (ok && nseg > 0)
                mbar_wait(bar_qempty, (nseg - 1) & 1, abort_flag);
            for (uint32_t back = 1; ok && back <= 2 && back <= it; ++back)
                mbar_wait(bar_sfull((it - back) & 1), ((it - back) >> 1) & 1, abort_flag);
        }
    } else if (warp == 6) {
        // ================================================================ PV issuer
        // O^T += V^T P^T and l^T += 1 P^T of each tile, from P buffer pbuf(it).
        if (lane == 0) {
            uint32_t it = 0, nseg = 0;
            RingPos ppos = {0u, 0u};                     // ring position of K(it)
            bool ok = true;
            // A segment that holds part of a (request, row block, head group) pair leaves
            // a partial result; its pair ticket is taken here, while this warp waits for
            // the epilogue anyway.  The partial stores precede the epilogue's arrive on
            // ofree (release), this thread's wait acquires them, and the gpu-scope fence
            // below is cumulative over them.  The ticket values are read at the end only.
            VtSeg sp = {};
            int32_t sp_nact = 0, sp_row0 = 0;
            int32_t ntk = 0, tk0 = 0, tk1 = 0;
            VtSeg tks0 = {}, tks1 = {};
            int32_t tkn0 = 0, tkr0 = 0, tkn1 = 0, tkr1 = 0;
            auto take_ticket = [&]() {
                if (sp.single)
                    return;
                __threadfence();
                if (ntk == 0) {
                    tk0 = atomicAdd(p.tickets + sp.pair, 1);
                    tks0 = sp; tkn0 = sp_nact; tkr0 = sp_row0;
                } else {
                    tk1 = atomicAdd(p.tickets + sp.pair, 1);
                    tks1 = sp; tkn1 = sp_nact; tkr1 = sp_row0;
                }
                ++ntk;
            };
            for (int64_t u = cta_s; u < cta_e && ok;) {
                VtSeg s;
                vt_seg(p, rs, prefix, NQ, u, cta_e, cta_s, s);
                const int32_t off = rs_req_off(rs, p, s.i);
                const int32_t k_i = (s.i + 1 < kReqCache && s.i + 1 < p.n ? rs->req_off[s.i + 1]
                                                                          : __ldg(p.cu_slots + s.i + 1)) - off;
                const int32_t L = rs_req_len(rs, p, s.i);
                const int32_t kk = min(k_i - s.rb * p.R, p.R);
                const uint32_t NRs = (uint32_t)((p.HP * kk + 31) / 32 * 32);
                const uint32_t idesc_o = idesc_bf16_f32(128, NRs, true, true);
                const uint32_t idesc_l = idesc_bf16_f32(128, NRs, false, true);
                const uint64_t ao = sw128_desc(sbase + p.off_ones, 16, 0);
                const int32_t nt = s.t1 - s.t0;
                // O^T of this segment may be written once the previous epilogue read it
                if (nseg > 0) {
                    if (!(ok = mbar_wait(bar_ofree, (nseg - 1) & 1, abort_flag)))
                        break;
                    take_ticket();
                }
                sp = s;
                sp_nact = p.HP * kk;
                sp_row0 = off + s.rb * p.R;
                for (int32_t k = 0; k < nt; ++k, ++it) {
                    const int pb = pbuf(it);
                    if (!(ok = mbar_wait(bar_pfull(pb), ppar(it), abort_flag)))
                        break;
                    for (int h = 0; h < DH && ok; ++h) {
                        const RingPos q = ring_add(ppos, (uint32_t)(DH + h), (uint32_t)nslot);
                        ok = mbar_wait(bar_full(q.slot), q.phase, abort_flag);
                    }
                    if (!ok)
                        break;
                    // V(it) has landed: the S issuer may reuse the parity of its slots
                    __threadfence_block();
                    *reinterpret_cast<volatile uint32_t *>(&rs->v_seen) = it + 1u;
                    tc_fence_after();
                    const int32_t kv = vt_kvalid(p, s, s.t0 + k, L, k_i);
                    const int32_t k16 = (kv + 15) / 16;
                    const uint64_t bp = sw128_desc(sbase + p.off_p + pb * PBYTES, 16384, 1024);
                    const uint32_t acc0 = k == 0 ? 0u : 1u;
                    for (int h = 0; h < DH; ++h) {
                        const uint64_t av = sw128_desc(
                            sbase + p.off_ring + ring_add(ppos, (uint32_t)(DH + h), (uint32_t)nslot).slot * kSlotBytes,
                            kSubBytes, 1024);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            if (ks < k16)   // 16 keys (2048 bytes) per MMA
                                tc_mma_ss(tmem + TM_O + h * NR, av + (uint64_t)(ks * 128),
                                          bp + (uint64_t)(ks * 128), idesc_o, ks ? 1u : acc0);
                        // this half's V slot is free once its MMAs are done
                        tc_commit(bar_empty(ring_add(ppos, (uint32_t)(DH + h), (uint32_t)nslot).slot));
                    }
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        if (ks < k16)
                            tc_mma_ss(tmem + TM_L, ao, bp + (uint64_t)(ks * 128), idesc_l, ks ? 1u : acc0);
                    tc_commit(bar_pvdone(pb));
                    ppos = ring_add(ppos, 2u * DH, (uint32_t)nslot);
                }
                ++nseg;
                u += nt;
            }
            if (ok && nseg > 0 && (ok = mbar_wait(bar_ofree, (nseg - 1) & 1, abort_flag)))
                take_ticket();
            if (ok) {
                // the pair's last arrival merges it after this CTA's range
                int32_t npend = 0;
                for (int q = 0; q < ntk; ++q) {
                    const VtSeg &e = q ? tks1 : tks0;
                    const int32_t cf = vt_cta_of_unit(ctile, ncta, e.u_pair0);
                    const int32_t cl = vt_cta_of_unit(ctile, ncta, e.u_pair0 + e.n_tiles - 1);
                    if ((q ? tk1 : tk0) == cl - cf) {
                        int32_t *d = rs->pend[npend++];
                        d[0] = e.pair; d[1] = cf; d[2] = cl; d[3] = q ? tkn1 : tkn0;
                        d[4] = q ? tkr1 : tkr0; d[5] = e.hg;
                        d[6] = (int32_t)(e.u_pair0 & 0xffffffff); d[7] = (int32_t)(e.u_pair0 >> 32);
                    }
                }
                rs->npend = npend;
                if (npend)
                    __threadfence();   // acquire side: the other pieces' partials are visible
            }
            mbar_arrive(bar_tick);
            tc_commit(bar_drain);
            volatile int drain_abort = 0;
            mbar_wait(bar_drain, 0, &drain_abort);
            // tail: the last pvdone commit of each P buffer has landed
            for (uint32_t back = 1; ok && back <= (uint32_t)nP && back <= it; ++back)
                mbar_wait(bar_pvdone(pbuf(it - back)), ppar(it - back), abort_flag);
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
            vt_seg(p, rs, prefix, NQ, u, cta_e, cta_s, s);
            const int32_t off = rs_req_off(rs, p, s.i);
            const int32_t k_i = (s.i + 1 < kReqCache && s.i + 1 < p.n ? rs->req_off[s.i + 1]
                                                                      : __ldg(p.cu_slots + s.i + 1)) - off;
            const int32_t L = rs_req_len(rs, p, s.i);
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
                // A wait that gives up does not leave the loop here: the thread runs on to
                // the next barrier of the four warps, where all of them leave together.
                ok &= mbar_wait(bar_sfull(b), (it >> 1) & 1, abort_flag);
                __syncwarp();
                tc_fence_after();
                const uint32_t sa = tmem + lane_off + TM_S + b * NR;
                const uint32_t pline = sbase + p.off_p + pbuf(it) * PBYTES + t * 128;
                const uint32_t mref_a = smem_u32(rs->m_ref), jr_a = smem_u32(rs->jr);
                if (k == 0) {
                    // seed the reference of every live row with the score of key 0 of
                    // this piece's first tile (lane 0 of the first lane quarter)
                    if (quarter == 0) {
                        for (int c = 0; c < nch; ++c) {
                            uint32_t sr[32];
                            tmem_ld32(sa + c * 32, sr);
                            tmem_wait_ld();
                            // lane e takes key 0's score of row 32c + e
                            float mine = 0.0f;
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const float v = __shfl_sync(0xffffffffu, __uint_as_float(sr[e]), 0);
                                if (lane == e)
                                    mine = v;
                            }
                            const int r = c * 32 + lane;
                            if (rs->m_ref[r] != INFINITY && (is_ctx || cbase <= rs->jr[r]))
                                rs->m_ref[r] = mine * cl2;
                        }
                    }
                    if (named_bar_any(1, 128, !ok)) {
                        ok = false;
                        break;
                    }
                }
                // P of all chunks into registers while PV of the previous tile runs
                uint32_t pk[4][16];
                float ymax = -INFINITY;
#pragma unroll
                for (int c = 0; c < 4; c += 2) {
                    if (c < nch) {
                        uint32_t sr0[32], sr1[32];
                        tmem_ld32(sa + c * 32, sr0);
                        if (c + 1 < nch)
                            tmem_ld32(sa + (c + 1) * 32, sr1);
                        tmem_wait_ld();
                        vt_chunk(sr0, mref_a + c * 128, jr_a + c * 128, key_ok, !is_ctx, cbase + t,
                                 cl2, pk[c], ymax);
                        if (c + 1 < nch)
                            vt_chunk(sr1, mref_a + (c + 1) * 128, jr_a + (c + 1) * 128, key_ok, !is_ctx,
                                     cbase + t, cl2, pk[c + 1], ymax);
                    }
                }
                const bool hit = ymax > kSlack;
                // this P buffer is read by PV of tile it - nP
                if (it >= (uint32_t)nP)
                    ok &= mbar_wait(bar_pvdone(pbuf(it)), ppar(it - nP), abort_flag);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (c < nch) {
                        const int blk = c >> 1, c0 = (c & 1) * 4;
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            st_shared_v4(pline + blk * 16384 + (((c0 + v) ^ (t & 7)) << 4),
                                         pk[c][4 * v], pk[c][4 * v + 1], pk[c][4 * v + 2], pk[c][4 * v + 3]);
                    }
                }
                if (__any_sync(0xffffffffu, hit) && lane == 0)
                    rs->flag[it & 1] = 1;
                if (named_bar_any(1, 128, !ok)) {
                    ok = false;
                    break;
                }
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
                    if (named_bar_any(1, 128, !ok)) {
                        ok = false;
                        break;
                    }
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
                    if (named_bar_any(1, 128, !ok)) {
                        ok = false;
                        break;
                    }
                    if (rs->rescale) {
                        // O^T halves and l^T: column r scaled by alpha[r], once PV of the
                        // previous tile is complete
                        ok &= mbar_wait(bar_pvdone(pbuf(it - 1)), ppar(it - 1), abort_flag);
                        __syncwarp();
                        tc_fence_after();
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
                        uint32_t pq[16];
                        float dummy = -INFINITY;
                        vt_chunk(sr, mref_a + c * 128, jr_a + c * 128, key_ok, !is_ctx, cbase + t,
                                 cl2, pq, dummy);
                        const int blk = c >> 1, c0 = (c & 1) * 4;
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            st_shared_v4(pline + blk * 16384 + (((c0 + v) ^ (t & 7)) << 4),
                                         pq[4 * v], pq[4 * v + 1], pq[4 * v + 2], pq[4 * v + 3]);
                    }
                    if (named_bar_any(1, 128, !ok)) {
                        ok = false;
                        break;
                    }
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
                        // only some threads wait here, after the tile's last collective
                        // decision: a failed wait (the abort flag is set by then) does not
                        // touch ok, so the four warps still leave the loops together; the
                        // other roles give up at their next wait and the launch reports it
                        if (!mbar_wait(bar_full(sq % nslot), (sq / nslot) & 1, abort_flag))
                            break;
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
                    mbar_arrive(bar_pfull(pbuf(it)));
            }
            if (!ok)
                break;   // only ever reached by all four warps together (a barrier decided it)
            // ---- epilogue: O^T, l^T complete after the last PV of the segment
            ok &= mbar_wait(bar_pvdone(pbuf(it - 1)), ppar(it - 1), abort_flag);
            __syncwarp();
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
            const int32_t out_row0 = off + s.rb * p.R;
            const int nact = p.HP * kk;                // active rows of this tile
            if (stid < nact) {
                const int r = stid;
                rs->orow[r] = ((int64_t)(out_row0 + r / p.HP) * p.hq + s.hg * p.HP + r % p.HP) * D;
            }
            if (named_bar_any(1, 128, !ok)) {
                ok = false;
                break;
            }
            if (stid < nact)
                rs->linv[stid] = 1.0f / rs->lrow[stid];
            named_bar_sync(1, 128);
            if (s.single) {
                for (int h = 0; h < DH; ++h) {
                    for (int c = 0; c < nch; ++c) {
                        uint32_t ro[32];
                        tmem_ld32(tmem + lane_off + TM_O + h * NR + c * 32, ro);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int r = c * 32 + e;
                            if (r < nact)
                                reinterpret_cast<uint16_t *>(p.out)[rs->orow[r] + h * 128 + t] =
                                    (uint16_t)(pack_bf16x2(__uint_as_float(ro[e]) * rs->linv[r], 0.0f) & 0xffffu);
                        }
                    }
                }
                if (stid < nact && p.lse)
                    p.lse[rs->orow[stid] / D] = (rs->m_ref[stid] + __log2f(rs->lrow[stid])) * 0.69314718055994531f;
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar_ofree);
            } else {
                const int32_t slot = 2 * blockIdx.x + (s.first_of_cta ? 0 : 1);
                const uint64_t pol_keep = l2_policy_evict_last();   // read back by the merge
                for (int h = 0; h < DH; ++h) {
                    for (int c = 0; c < nch; ++c) {
                        uint32_t ro[32];
                        tmem_ld32(tmem + lane_off + TM_O + h * NR + c * 32, ro);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int r = c * 32 + e;
                            if (r < nact)
                                st_global_f32_hint(p.part_o + (((int64_t)slot * DH + h) * kRows + r) * 128 + t,
                                                   __uint_as_float(ro[e]), pol_keep);
                        }
                    }
                }
                if (stid < nact)
                    st_global_f2_hint(p.part_ml + (int64_t)slot * kRows + stid,
                                      make_float2(rs->m_ref[stid], rs->lrow[stid]), pol_keep);
                // the partial stores of this warp precede its arrive (the PV issuer takes
                // the pair's ticket after it)
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar_ofree);
            }
            named_bar_sync(1, 128);
            ++nseg;
            u += nt;
        }
        // ---- merges owed by this CTA (it delivered the pair's last piece): partial slabs
        // -> TMA ring (one bulk copy per piece), then weights x slabs from shared memory;
        // pieces in order.
        if (ok)
            ok = mbar_wait(bar_tick, 0, abort_flag);
        if (named_bar_any(1, 128, !ok))
            ok = false;
        const int npend = ok ? rs->npend : 0;
        if (npend)
            __threadfence();   // acquire: the other pieces' partials, read below by this thread
        uint32_t merge_phase = 0;
        for (int pi = 0; pi < npend && ok; ++pi) {
            const int32_t *e = rs->pend[pi];
            const int32_t pair = e[0], cf = e[1], cl = e[2], nact = e[3], out_row0 = e[4], hg = e[5];
            const int64_t u_pair0 = (int64_t)(uint32_t)e[6] | ((int64_t)e[7] << 32);
            const int32_t np = cl - cf + 1;
            for (int32_t q = stid; q < np; q += 128) {
                const int32_t c = cf + q;
                const int64_t cs = ctile[c];
                rs->pslot[q] = 2 * c + ((q == 0 && cs < u_pair0) ? 1 : 0);
            }
            if (stid < nact) {
                const int r = stid;
                rs->orow[r] = ((int64_t)(out_row0 + r / p.HP) * p.hq + hg * p.HP + r % p.HP) * D;
            }
            named_bar_sync(1, 128);
            // a slab is one 128-column block (d-half) of one piece's partial, contiguous in
            // the [slot][d / 128][row][128] layout; the merge runs block by block
            const uint32_t slab = (uint32_t)nact * 128u * 4u;
            const int32_t cap_ring = (int32_t)((uint32_t)(nslot * kSlotBytes) / slab);
            const int32_t cap = cap_ring < 8 ? cap_ring : 8;
            // the first pass's slabs are on their way while the row statistics are formed
            auto issue_pass = [&](int h, int32_t c0) {
                const int32_t nb = min(cap, np - c0);
                asm volatile("fence.proxy.async.global;" ::: "memory");
                mbar_arrive_expect_tx(bar_merge, (uint32_t)nb * slab);
                for (int q = 0; q < nb; ++q)
                    bulk_g2s(sbase + p.off_ring + q * slab,
                             p.part_o + ((int64_t)rs->pslot[c0 + q] * DH + h) * kRows * 128, slab, bar_merge);
            };
            if (stid == 0)
                issue_pass(0, 0);
            // per row: merged max M and sum L over the pieces, one online pass; with at
            // most 8 pieces the weights 2^(m_q - M) come out of the same pass
            const bool one_block = np <= 8;
            if (stid < nact) {
                const int r = stid;
                float M = -INFINITY, Ls = 0.0f;
                for (int32_t c0 = 0; c0 < np; c0 += 8) {
                    float2 ml[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        ml[q] = (c0 + q < np) ? __ldcg(p.part_ml + (int64_t)rs->pslot[c0 + q] * kRows + r)
                                              : make_float2(-INFINITY, 0.0f);
                    float Mb = M;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        Mb = fmaxf(Mb, ml[q].x);
                    float Lb = (M == -INFINITY) ? 0.0f : Ls * fast_exp2(M - Mb);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (c0 + q < np)
                            Lb += ml[q].y * fast_exp2(ml[q].x - Mb);
                    M = Mb;
                    Ls = Lb;
                    if (one_block) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            if (q < np)
                                rs->wts[q][r] = fast_exp2(ml[q].x - M);
                    }
                }
                rs->m_ref[r] = M;
                rs->linv[r] = 1.0f / Ls;
                if (p.lse)
                    p.lse[rs->orow[r] / D] = (M + __log2f(Ls)) * 0.69314718055994531f;
            }
            const int32_t slot0 = rs->pslot[0];
            int32_t npass = 0;
            for (int h = 0; h < DH && ok; ++h) {
                for (int32_t c0 = 0; c0 < np; c0 += cap, ++npass) {
                    const int32_t nb = min(cap, np - c0);
                    const int32_t wq0 = one_block ? c0 : 0;   // weights of this pass: wts[wq0 + q]
                    if (npass > 0) {
                        if (named_bar_any(1, 128, !ok)) {    // the ring was read by the last pass
                            ok = false;
                            break;
                        }
                        if (stid == 0)
                            issue_pass(h, c0);
                    }
                    if (!one_block && stid < nact) {
                        const int r = stid;
                        for (int q = 0; q < nb; ++q)
                            rs->wts[q][r] = fast_exp2(__ldcg(p.part_ml + (int64_t)rs->pslot[c0 + q] * kRows + r).x -
                                                      rs->m_ref[r]);
                    }
                    named_bar_sync(1, 128);
                    const bool landed = mbar_wait(bar_merge, merge_phase & 1, abort_flag);
                    if (!landed && stid == 0) {
                        volatile int drain_abort = 0;   // the slabs land before the CTA exits
                        mbar_wait(bar_merge, merge_phase & 1, &drain_abort);
                    }
                    ok &= landed;
                    ++merge_phase;
                    const bool last_pass = c0 + cap >= np;
                    const uint32_t ring = sbase + p.off_ring;
                    switch (nb) {
#define SVP_MERGE_CASE(K)                                                                          \
    case K:                                                                                        \
        vt_merge_pass<K, D>(p, rs, ring, slab, wq0, nact, slot0, h, c0 == 0, last_pass, stid);     \
        break;
                        SVP_MERGE_CASE(1)
                        SVP_MERGE_CASE(2)
                        SVP_MERGE_CASE(3)
                        SVP_MERGE_CASE(4)
                        SVP_MERGE_CASE(5)
                        SVP_MERGE_CASE(6)
                        SVP_MERGE_CASE(7)
                        default:
                            vt_merge_pass<8, D>(p, rs, ring, slab, wq0, nact, slot0, h, c0 == 0, last_pass, stid);
                            break;
#undef SVP_MERGE_CASE
                    }
                    if (!last_pass)
                        __threadfence_block();
                }
                // landed is per thread (with the abort flag set, a thread may see the slabs
                // land or give up): decide together, so that the loop test below is the
                // same in all four warps
                if (named_bar_any(1, 128, !ok))
                    ok = false;
            }
            if (named_bar_any(1, 128, !ok)) {
                ok = false;
                break;
            }
            if (stid == 0)
                p.tickets[pair] = 0;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // read once every role has finished, so that a wait given up late (in a merge, say) is
    // reported too and the workspace is marked for clearing
    if (*abort_flag && tid == 0) {
        set_status(p.status, SVP_DEV_TIMEOUT);
        *reinterpret_cast<volatile int32_t *>(p.status + kWsPoisonWord) = 1;
    }
    if (warp == 1)
        tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
}

template <int D>
static svp_status vt_launch_d(const TcParams &p, int grid, cudaStream_t stream)
{
    static std::atomic<uint64_t> configured{0};
    if (set_smem_limit_once(verify_tc_kernel<D>, 227 * 1024, configured) != cudaSuccess)
        return SVP_ECUDA;
    return launch_pdl(verify_tc_kernel<D>, dim3(grid), dim3(kVThreads), (size_t)p.smem_bytes, stream, p) ==
                   cudaSuccess
               ? SVP_OK
               : SVP_ECUDA;
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
static bool verify_tc_layout_np(int d, int NR, int nP, int grid, TcParams &p);

bool verify_tc_layout(int d, int NR, int grid, TcParams &p)
{
    p.cost0 = kPairCost;
    // two P buffers when the ring keeps enough slots, else one
    if (verify_tc_layout_np(d, NR, 2, grid, p) && p.nslot >= (d == 128 ? 5 : 4))
        return true;
    return verify_tc_layout_np(d, NR, 1, grid, p);
}

static bool verify_tc_layout_np(int d, int NR, int nP, int grid, TcParams &p)
{
    const int budget = 227 * 1024;
    const int q = (d / 64) * NR * 128;
    const int pt = nP * ((NR + 63) / 64) * 16384;
    p.nP = nP;
    int off = 0;
    p.off_q = off; off += q;
    p.off_p = off; off += pt;
    p.off_ones = off; off += 1024;
    p.off_bar = off; off += 30 * 8;
    off = (off + 15) / 16 * 16;
    p.off_misc = off; off += (int)sizeof(VtRows);
    off = (off + 15) / 16 * 16;
    p.off_pref = off; off += (2 * (p.n * p.RB + 1) + grid + 1) * 4;   // prefix, cprefix, ctile
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
