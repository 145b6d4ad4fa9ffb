// svp_params.cuh -- launch parameter blocks shared by the attention kernels and the
// host-side planner.
#pragma once

#include "svp_device.cuh"

namespace svp {

constexpr int kBN = 64;               // keys per KV tile
constexpr int kRows = 128;            // query rows per tile (MMA M)
constexpr int kThreads = 192;         // 6 warps
constexpr int kSoftmaxWarp0 = 2;
constexpr int kMaxPrefix = 1024;      // (request, row block) entries held in shared memory
constexpr float kRescaleLog2 = 8.0f;  // move the running max only when it grows by > 2^8

enum { kModeShort = 1, kModeFixed128 = 2, kModeWide = 3 };

struct TcParams {
    CUtensorMap tm_q;     // q:     dims {d, hq, rows}, box {64, HP, R}
    CUtensorMap tm_kc;    // ctx K: contiguous dims {d, hkv, tokens} box {64, 1, 64};
                          //        paged dims {d, 16, hkv, pages} box {64, 16, 1, 1}
    CUtensorMap tm_vc;
    CUtensorMap tm_kn;    // candidate K: dims {d, hkv, rows}, box {64, 1, CB}
    CUtensorMap tm_vn;
    const int32_t *ctx_len;      // [n] (nullptr: all zero)
    const int32_t *cu_slots;     // [n+1]
    const int64_t *cu_ctx;       // [n]
    const int32_t *block_table;  // [n, max_pages]
    int32_t n, m_cap, w, hq, hkv, G;
    int32_t HP, R, RB, HG, CB;
    int32_t paged, max_pages, mode, split;
    int64_t num_pages, total_tokens;
    float scale_log2;
    void *out;                   // [m_cap, hq, d] bf16
    float *lse;                  // [m_cap, hq] or nullptr
    int32_t *status;
    int32_t *tickets;            // [n * RB * HG]
    float *part_o;               // verify_tc: [2 * gridDim.x][d / 128][128][128]; attn_tc: [2 * gridDim.x][128][d]
    float2 *part_ml;             // [2 * gridDim.x][128]
    int32_t sig;                 // workspace layout signature (header word 1)
    // transposed short-tile kernel only: tile rows and shared-memory layout
    int32_t NR, nslot, tmem_cols, smem_bytes, nP;
    int32_t cost0;               // partition cost of starting a pair, in KV tiles
    int32_t off_q, off_p, off_ones, off_ring, off_bar, off_misc, off_pref;
};

struct SimtParams {
    const float *q, *k_new, *v_new;
    const float *k, *v;               // context storage (contiguous or paged pool)
    const int64_t *cu_ctx;
    const int32_t *block_table;
    const int32_t *ctx_len, *cu_slots;
    int32_t n, m_cap, w, hq, hkv, d, paged, max_pages;
    int64_t num_pages, total_tokens, s_page, s_head, s_tok;
    float scale;
    float *out, *lse;
    int32_t *status;
};

}  // namespace svp
