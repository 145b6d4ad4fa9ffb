// api.cu -- the C ABI of include/svp.h: argument checks, launch planning (tile router,
// work split, workspace layout), TMA tensor-map encoding and kernel launches.
#include <cmath>
#include <cstring>
#include <mutex>

#include <algorithm>

#include "svp_params.cuh"

namespace svp {

// ---- kernels defined in the other translation units
svp_status attn_tc_launch(const TcParams &p, int d, int grid, cudaStream_t stream);
svp_status verify_tc_launch(const TcParams &p, int d, int grid, cudaStream_t stream);
bool verify_tc_layout(int d, int NR, int grid, TcParams &p);
int attn_tc_max_prefix();
int attn_tc_block_keys();
svp_status attn_simt_launch(const SimtParams &p, cudaStream_t stream);
svp_status margin_workspace(int32_t rows, int32_t vocab, int32_t n, size_t *bytes);
svp_status margin_launch(const void *logits, int64_t row_stride, int32_t rows, int32_t vocab,
                         svp_dtype dtype, int32_t *top1_idx, float *top1, float *top2,
                         float *margin, const int32_t *tokens, const int32_t *cu_slots,
                         int32_t n, int32_t *accept_len, int32_t *next_token, void *ws,
                         size_t ws_bytes, cudaStream_t stream);
bool prefill_tc_supported(int32_t n, int32_t max_s, int32_t hq, int32_t hkv, int32_t d);
svp_status prefill_tc_launch(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                             const int32_t *cu_seqlens, int32_t n, int32_t max_s, int32_t total_s,
                             int32_t hq, int32_t hkv, float scale_log2, void *out, float *lse,
                             int32_t *status, int grid, cudaStream_t stream);
svp_status accept_launch(const int32_t *target_argmax, const int32_t *tokens,
                         const int32_t *cu_slots, int32_t n, int32_t m_cap,
                         int32_t *accept_len, int32_t *next_token, cudaStream_t stream);

int sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 148;
    if (cached[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        cached[dev] = v;
    }
    return cached[dev];
}

// ---- TMA tensor-map encoding through the driver entry point (no libcuda link)
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

static bool encode_bf16(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
                        const uint64_t *strides_bytes, const uint32_t *box)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    for (int r = 0; r < rank; ++r) {
        gd[r] = dims[r];
        bx[r] = box[r];
        es[r] = 1;
        if (r + 1 < rank)
            gs[r] = strides_bytes[r];
    }
    CUresult rc = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base),
                     gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return rc == CUDA_SUCCESS;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
static size_t al256(size_t x) { return (x + 255) / 256 * 256; }

// ---- tensor-core attention plan (tile router + work split + workspace layout)
struct AttnPlan {
    int mode, HP, R, RB, HG, CB, split, grid, transposed, NR;
    size_t off_part_ml, off_part_o, off_tickets, bytes;
};

static svp_status attn_plan(int32_t n, int32_t w, int32_t hq, int32_t hkv, int32_t d,
                            int32_t tile_mode, AttnPlan &pl)
{
    if (n < 0 || w < 1 || hq <= 0 || hkv <= 0 || hq % hkv)
        return SVP_EINVAL;
    if (d != 64 && d != 128 && d != 256)
        return SVP_EUNSUPPORTED;
    const int G = hq / hkv;
    int mode = tile_mode;
    if (mode == SVP_TILE_AUTO)
        mode = (w <= 16) ? SVP_TILE_SHORT : SVP_TILE_WIDE;   // DScale SIII-B router
    pl = AttnPlan{};
    pl.mode = mode;
    switch (mode) {
    case SVP_TILE_SHORT: {
        // transposed kernel: G*R rows of the tile on the MMA N dimension; TMEM holds two
        // S^T buffers, O^T (d/128 of them) and l^T, each NR columns wide.
        const int nr_cap = (d == 256) ? 96 : 128;
        if (d != 64 && G <= nr_cap) {
            pl.transposed = 1;
            pl.HP = G;
            pl.R = std::min(w, nr_cap / G);
            pl.NR = (G * pl.R + 31) / 32 * 32;
        } else {
            if (G > 128)
                return SVP_EUNSUPPORTED;
            pl.HP = G;
            pl.R = std::min(w, 128 / G);
        }
        pl.HG = hkv;
        pl.CB = 16;
        pl.split = 1;
        break;
    }
    case SVP_TILE_SHORT_UNPACKED: {
        // contrast: the same transposed kernel with one query head per tile, so every query
        // head streams its KV head itself (G times the KV bytes of the packed tile)
        if (d == 64)
            return SVP_EUNSUPPORTED;
        const int nr_cap = (d == 256) ? 96 : 128;
        pl.transposed = 1;
        pl.HP = 1;
        pl.R = std::min(w, nr_cap);
        pl.NR = (pl.R + 31) / 32 * 32;
        pl.HG = hq;
        pl.CB = 16;
        pl.split = 1;
        break;
    }
    case SVP_TILE_FIXED128:
        pl.HP = 1;
        pl.R = std::min(w, 128);
        pl.HG = hq;
        pl.CB = 16;
        pl.split = 0;
        break;
    case SVP_TILE_WIDE:
        pl.HP = 1;
        pl.R = 128;
        pl.HG = hq;
        pl.CB = attn_tc_block_keys();
        pl.split = 1;
        break;
    default:
        return SVP_EUNSUPPORTED;
    }
    pl.RB = (w + pl.R - 1) / pl.R;
    if ((int64_t)n * pl.RB > attn_tc_max_prefix())
        return SVP_EUNSUPPORTED;
    const int64_t pairs = (int64_t)n * pl.RB * pl.HG;
    if (pl.split)
        pl.grid = sm_count();
    else
        pl.grid = (int)std::max<int64_t>(pairs, 1);
    // header | partial (max, sum) | partial O | tickets: the partial regions depend only
    // on the device and head_dim, so a workspace can serve calls with different n.
    const size_t slots = pl.split ? 2 * (size_t)sm_count() : 0;
    size_t o = kWsHeader;
    pl.off_part_ml = o;
    o = al256(o + slots * 128 * 2 * sizeof(float));
    pl.off_part_o = o;
    o = al256(o + slots * 128 * (size_t)d * sizeof(float));
    pl.off_tickets = o;
    o = al256(o + sizeof(int32_t) * (size_t)std::max<int64_t>(pairs, 1));
    pl.bytes = o;
    return SVP_OK;
}

}  // namespace svp

using namespace svp;

extern "C" {

int32_t svp_version(void) { return SVP_VERSION; }

const char *svp_status_string(svp_status s)
{
    switch (s) {
    case SVP_OK: return "ok";
    case SVP_EINVAL: return "invalid argument";
    case SVP_EUNSUPPORTED: return "unsupported configuration";
    case SVP_EWORKSPACE: return "workspace missing or too small";
    case SVP_ECUDA: return "CUDA error";
    default: return "unknown status";
    }
}

svp_status svp_workspace_init(void *ws, size_t ws_bytes, void *stream)
{
    if (!ws || ws_bytes < kWsHeader)
        return SVP_EWORKSPACE;
    return cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream) == cudaSuccess ? SVP_OK : SVP_ECUDA;
}

svp_status svp_read_status(void *ws, void *stream, int32_t *status)
{
    if (!ws || !status)
        return SVP_EINVAL;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t host = 0;
    if (cudaMemcpyAsync(&host, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SVP_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return SVP_ECUDA;
    if (cudaMemsetAsync(ws, 0, sizeof(int32_t), s) != cudaSuccess)
        return SVP_ECUDA;
    *status = host;
    return SVP_OK;
}

svp_status svp_verify_attn_workspace_size(int32_t n, int32_t m_cap, int32_t w,
                                          const svp_heads *heads, svp_dtype dtype,
                                          int32_t tile_mode, size_t *bytes)
{
    if (!heads || !bytes || m_cap < 0)
        return SVP_EINVAL;
    if (dtype == SVP_F32) {
        if (n < 0 || w < 1 || heads->hq <= 0 || heads->hkv <= 0 || heads->hq % heads->hkv)
            return SVP_EINVAL;
        *bytes = kWsHeader;
        return SVP_OK;
    }
    if (dtype != SVP_BF16)
        return SVP_EUNSUPPORTED;
    AttnPlan pl;
    svp_status st = attn_plan(n, w, heads->hq, heads->hkv, heads->d, tile_mode, pl);
    if (st != SVP_OK)
        return st;
    *bytes = pl.bytes;
    return SVP_OK;
}

static svp_status verify_impl(const void *q, const void *k_new, const void *v_new,
                              const svp_kv *kv, const int32_t *ctx_len, const int32_t *cu_slots,
                              int32_t n, int32_t m_cap, int32_t w, const svp_heads *heads,
                              svp_dtype dtype, int32_t tile_mode, void *out, float *lse,
                              void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (!heads || !kv)
        return SVP_EINVAL;
    if (n < 0 || m_cap < 0 || w < 1)
        return SVP_EINVAL;
    const int32_t hq = heads->hq, hkv = heads->hkv, d = heads->d;
    if (hq <= 0 || hkv <= 0 || hq % hkv)
        return SVP_EINVAL;
    if (d != 64 && d != 128 && d != 256)
        return SVP_EUNSUPPORTED;
    if (dtype != SVP_F32 && dtype != SVP_BF16)
        return SVP_EUNSUPPORTED;
    if (!ws)
        return SVP_EWORKSPACE;
    if (n == 0 || m_cap == 0)
        return SVP_OK;
    if (!q || !k_new || !v_new || !cu_slots || !out)
        return SVP_EINVAL;
    const bool has_ctx = kv->paged ? kv->num_pages > 0 : kv->total_tokens > 0;
    if (has_ctx && !ctx_len)
        return SVP_EINVAL;
    if (kv->paged) {
        if (kv->page_size != 16)
            return SVP_EUNSUPPORTED;
        if (!kv->k || !kv->v || !kv->block_table || kv->max_pages < 0 || kv->num_pages < 0)
            return SVP_EINVAL;
        if (kv->stride_page <= 0 || kv->stride_head <= 0 || kv->stride_tok <= 0)
            return SVP_EINVAL;
    } else {
        if (kv->total_tokens < 0 || kv->total_tokens >= (int64_t)INT32_MAX)
            return SVP_EINVAL;
        if (kv->total_tokens > 0 && (!kv->k || !kv->v || !kv->cu_ctx))
            return SVP_EINVAL;
    }
    const float scale = heads->scale != 0.0f ? heads->scale : 1.0f / std::sqrt((float)d);

    if (dtype == SVP_F32) {
        if (tile_mode != SVP_TILE_AUTO)
            return SVP_EUNSUPPORTED;
        if (ws_bytes < kWsHeader)
            return SVP_EWORKSPACE;
        SimtParams p{};
        p.q = static_cast<const float *>(q);
        p.k_new = static_cast<const float *>(k_new);
        p.v_new = static_cast<const float *>(v_new);
        p.k = static_cast<const float *>(kv->k);
        p.v = static_cast<const float *>(kv->v);
        p.cu_ctx = kv->cu_ctx;
        p.block_table = kv->block_table;
        p.ctx_len = ctx_len;
        p.cu_slots = cu_slots;
        p.n = n; p.m_cap = m_cap; p.w = w; p.hq = hq; p.hkv = hkv; p.d = d;
        p.paged = kv->paged; p.max_pages = kv->max_pages;
        p.num_pages = kv->num_pages; p.total_tokens = kv->total_tokens;
        p.s_page = kv->stride_page; p.s_head = kv->stride_head; p.s_tok = kv->stride_tok;
        p.scale = scale;
        p.out = static_cast<float *>(out);
        p.lse = lse;
        p.status = static_cast<int32_t *>(ws);
        return attn_simt_launch(p, stream);
    }

    AttnPlan pl;
    svp_status st = attn_plan(n, w, hq, hkv, d, tile_mode, pl);
    if (st != SVP_OK)
        return st;
    if (ws_bytes < pl.bytes)
        return SVP_EWORKSPACE;
    if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(out))
        return SVP_EINVAL;
    if (kv->k && (!aligned16(kv->k) || !aligned16(kv->v)))
        return SVP_EINVAL;

    TcParams p;
    std::memset(&p, 0, sizeof p);
    const uint64_t esz = 2;
    // q: {d, hq, m_cap}, box {64, HP, R}
    {
        const uint64_t dims[3] = {(uint64_t)d, (uint64_t)hq, (uint64_t)m_cap};
        const uint64_t str[2] = {d * esz, (uint64_t)hq * d * esz};
        const uint32_t box[3] = {64, (uint32_t)pl.HP, (uint32_t)pl.R};
        if (!encode_bf16(&p.tm_q, q, 3, dims, str, box))
            return SVP_EUNSUPPORTED;
    }
    // candidates: {d, hkv, m_cap}, box {64, 1, CB}
    {
        const uint64_t dims[3] = {(uint64_t)d, (uint64_t)hkv, (uint64_t)m_cap};
        const uint64_t str[2] = {d * esz, (uint64_t)hkv * d * esz};
        const uint32_t box[3] = {64, 1, (uint32_t)pl.CB};
        if (!encode_bf16(&p.tm_kn, k_new, 3, dims, str, box) ||
            !encode_bf16(&p.tm_vn, v_new, 3, dims, str, box))
            return SVP_EUNSUPPORTED;
    }
    // context
    const int BK = pl.transposed ? 128 : attn_tc_block_keys();
    if (kv->paged && kv->num_pages > 0) {
        const uint64_t dims[4] = {(uint64_t)d, 16, (uint64_t)hkv, (uint64_t)kv->num_pages};
        const uint64_t str[3] = {(uint64_t)kv->stride_tok * esz, (uint64_t)kv->stride_head * esz,
                                 (uint64_t)kv->stride_page * esz};
        const uint32_t box[4] = {64, 16, 1, 1};   // one 16-token page of one head
        if (!encode_bf16(&p.tm_kc, kv->k, 4, dims, str, box) ||
            !encode_bf16(&p.tm_vc, kv->v, 4, dims, str, box))
            return SVP_EUNSUPPORTED;
    } else if (!kv->paged && kv->total_tokens > 0) {
        const uint64_t dims[3] = {(uint64_t)d, (uint64_t)hkv, (uint64_t)kv->total_tokens};
        const uint64_t str[2] = {d * esz, (uint64_t)hkv * d * esz};
        const uint32_t box[3] = {64, 1, (uint32_t)BK};
        if (!encode_bf16(&p.tm_kc, kv->k, 3, dims, str, box) ||
            !encode_bf16(&p.tm_vc, kv->v, 3, dims, str, box))
            return SVP_EUNSUPPORTED;
    } else {
        p.tm_kc = p.tm_kn;   // no context storage: never read
        p.tm_vc = p.tm_vn;
    }
    p.ctx_len = ctx_len;
    p.cu_slots = cu_slots;
    p.cu_ctx = kv->cu_ctx;
    p.block_table = kv->block_table;
    p.n = n; p.m_cap = m_cap; p.w = w; p.hq = hq; p.hkv = hkv; p.G = hq / hkv;
    p.HP = pl.HP; p.R = pl.R; p.RB = pl.RB; p.HG = pl.HG; p.CB = pl.CB;
    p.paged = kv->paged; p.max_pages = kv->max_pages; p.mode = pl.mode; p.split = pl.split;
    p.num_pages = kv->paged ? kv->num_pages : 0;
    p.total_tokens = kv->paged ? 0 : kv->total_tokens;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out = out;
    p.lse = lse;
    uint8_t *wsb = static_cast<uint8_t *>(ws);
    p.status = reinterpret_cast<int32_t *>(wsb);
    p.tickets = reinterpret_cast<int32_t *>(wsb + pl.off_tickets);
    p.part_o = reinterpret_cast<float *>(wsb + pl.off_part_o);
    p.part_ml = reinterpret_cast<float2 *>(wsb + pl.off_part_ml);
    p.sig = (pl.transposed << 20) | (pl.mode << 12) | d;
    if (pl.transposed) {
        if (!verify_tc_layout(d, pl.NR, pl.grid, p))
            return SVP_EUNSUPPORTED;
        return verify_tc_launch(p, d, pl.grid, stream);
    }
    return attn_tc_launch(p, d, pl.grid, stream);
}

svp_status svp_verify_attn_packed(const void *q, const void *k_new, const void *v_new,
                                  const svp_kv *kv, const int32_t *ctx_len,
                                  const int32_t *cu_slots, int32_t n, int32_t m_cap, int32_t w,
                                  const svp_heads *heads, svp_dtype dtype, void *out,
                                  float *lse, void *ws, size_t ws_bytes, void *stream)
{
    return verify_impl(q, k_new, v_new, kv, ctx_len, cu_slots, n, m_cap, w, heads, dtype,
                       SVP_TILE_AUTO, out, lse, ws, ws_bytes, (cudaStream_t)stream);
}

svp_status svp_verify_attn_packed_ex(const void *q, const void *k_new, const void *v_new,
                                     const svp_kv *kv, const int32_t *ctx_len,
                                     const int32_t *cu_slots, int32_t n, int32_t m_cap,
                                     int32_t w, const svp_heads *heads, svp_dtype dtype,
                                     int32_t tile_mode, void *out, float *lse, void *ws,
                                     size_t ws_bytes, void *stream)
{
    return verify_impl(q, k_new, v_new, kv, ctx_len, cu_slots, n, m_cap, w, heads, dtype,
                       tile_mode, out, lse, ws, ws_bytes, (cudaStream_t)stream);
}

svp_status svp_prefill_attn_workspace_size(int32_t n, int32_t max_s, const svp_heads *heads,
                                           svp_dtype dtype, size_t *bytes)
{
    if (!heads || !bytes || n < 0 || max_s < 1)
        return SVP_EINVAL;
    if (dtype != SVP_BF16)
        return SVP_EUNSUPPORTED;
    AttnPlan pl;
    svp_status st = attn_plan(n, max_s, heads->hq, heads->hkv, heads->d, SVP_TILE_WIDE, pl);
    if (st != SVP_OK)
        return st;
    *bytes = pl.bytes;
    return SVP_OK;
}

svp_status svp_prefill_attn(const void *q, const void *k, const void *v,
                            const int32_t *cu_seqlens, int32_t n, int32_t max_s,
                            int64_t total_s, int32_t causal, const svp_heads *heads,
                            svp_dtype dtype, void *out, float *lse, void *ws, size_t ws_bytes,
                            void *stream)
{
    if (causal != 1)
        return SVP_EUNSUPPORTED;
    if (dtype != SVP_BF16)
        return SVP_EUNSUPPORTED;
    if (total_s < 0 || total_s >= (int64_t)INT32_MAX || max_s < 1)
        return SVP_EINVAL;
    if (heads && prefill_tc_supported(n, max_s, heads->hq, heads->hkv, heads->d)) {
        // the dedicated kernel: head_dim 128, an even number of query heads per KV head
        if (!ws)
            return SVP_EWORKSPACE;
        size_t need = 0;
        const svp_status st = svp_prefill_attn_workspace_size(n, max_s, heads, dtype, &need);
        if (st != SVP_OK)
            return st;
        if (ws_bytes < need)
            return SVP_EWORKSPACE;
        if (n == 0 || total_s == 0)
            return SVP_OK;
        if (!q || !k || !v || !cu_seqlens || !out)
            return SVP_EINVAL;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
            return SVP_EINVAL;
        const int32_t hq = heads->hq, hkv = heads->hkv, d = heads->d;
        CUtensorMap tq, tk, tv;
        const uint64_t esz = 2;
        const uint32_t box[3] = {64, 1, 128};
        const uint64_t dq[3] = {(uint64_t)d, (uint64_t)hq, (uint64_t)total_s};
        const uint64_t sq[2] = {d * esz, (uint64_t)hq * d * esz};
        const uint64_t dk[3] = {(uint64_t)d, (uint64_t)hkv, (uint64_t)total_s};
        const uint64_t sk[2] = {d * esz, (uint64_t)hkv * d * esz};
        if (!encode_bf16(&tq, q, 3, dq, sq, box) || !encode_bf16(&tk, k, 3, dk, sk, box) ||
            !encode_bf16(&tv, v, 3, dk, sk, box))
            return SVP_EUNSUPPORTED;
        const float scale = heads->scale != 0.0f ? heads->scale : 1.0f / std::sqrt((float)d);
        return prefill_tc_launch(tq, tk, tv, cu_seqlens, n, max_s, (int32_t)total_s, hq, hkv,
                                 scale * 1.4426950408889634f, out, lse,
                                 static_cast<int32_t *>(ws), sm_count(), (cudaStream_t)stream);
    }
    svp_kv kv;
    std::memset(&kv, 0, sizeof kv);   // no committed context
    return verify_impl(q, k, v, &kv, nullptr, cu_seqlens, n, (int32_t)total_s, max_s, heads,
                       dtype, SVP_TILE_WIDE, out, lse, ws, ws_bytes, (cudaStream_t)stream);
}

svp_status svp_draft_margin_workspace_size(int32_t rows, int32_t vocab, size_t *bytes)
{
    return margin_workspace(rows, vocab, 0, bytes);
}

svp_status svp_draft_margin(const void *logits, int64_t row_stride, int32_t rows, int32_t vocab,
                            svp_dtype dtype, int32_t *top1_idx, float *top1, float *top2,
                            float *margin, void *ws, size_t ws_bytes, void *stream)
{
    return margin_launch(logits, row_stride, rows, vocab, dtype, top1_idx, top1, top2, margin,
                         nullptr, nullptr, 0, nullptr, nullptr, ws, ws_bytes,
                         (cudaStream_t)stream);
}

svp_status svp_greedy_accept(const int32_t *target_argmax, const int32_t *tokens,
                             const int32_t *cu_slots, int32_t n, int32_t m_cap,
                             int32_t *accept_len, int32_t *next_token, void *stream)
{
    return accept_launch(target_argmax, tokens, cu_slots, n, m_cap, accept_len, next_token,
                         (cudaStream_t)stream);
}

svp_status svp_margin_accept_workspace_size(int32_t n, int32_t m_cap, int32_t vocab,
                                            size_t *bytes)
{
    return margin_workspace(m_cap, vocab, n, bytes);
}

svp_status svp_margin_accept(const void *logits, int64_t row_stride, int32_t m_cap,
                             int32_t vocab, svp_dtype dtype, const int32_t *tokens,
                             const int32_t *cu_slots, int32_t n, int32_t *top1_idx,
                             float *top1, float *top2, float *margin, int32_t *accept_len,
                             int32_t *next_token, void *ws, size_t ws_bytes, void *stream)
{
    if (!cu_slots)
        return SVP_EINVAL;
    return margin_launch(logits, row_stride, m_cap, vocab, dtype, top1_idx, top1, top2, margin,
                         tokens, cu_slots, n, accept_len, next_token, ws, ws_bytes,
                         (cudaStream_t)stream);
}

}  // extern "C"
