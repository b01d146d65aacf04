// Decode-attention plan and workspace layout shared by the decode kernels.
#pragma once

#include <stdint.h>
#include <stddef.h>

#include <algorithm>

#include "oscar_internal.h"

namespace oscar {

// The history of each request is cut into chunks of `chunk` tokens.  A
// persistent history grid of at most `max_ctas` CTAs splits the flattened
// chunk list into contiguous runs (CTA i owns [i·N/n, (i+1)·N/n)), and each
// CTA writes one (m, l, o) partial per request it touches and per stage parity
// π < par (par = 1 or 2 warp sets consuming alternate stages), at partial slot
// (i + b)·par + π.  i + b is unique: if CTAs i < i' both touch requests b and b'
// with i + b = i' + b', then b' < b, but runs are ordered so b' >= b.  The
// CUDA-core grid has up to max_ctas = 4·n_sm CTAs and par = 1; the tensor-core
// grid has at most n_sm CTAs and par <= 2.  So max(max_ctas + batch,
// 2·(n_sm + batch)) slots suffice, whatever the lengths.
// A combine block takes at most kCombHeads query heads of one KV head; larger
// query groups (up to 16) take ceil(g / kCombHeads) blocks per KV head.
constexpr int kCombHeads = 8;
constexpr int kCombGroups = 2;   // combine blocks per KV head at g = 16

struct DecodePlan {
    int chunk;        // tokens per chunk (multiple of 32)
    int max_ctas;     // upper bound of the history grid
    int part_slots;   // max(max_ctas + batch, 2 * (n_sm + batch))
    int n_frag_tiles; // n-tiles of 8 columns for the fragment-packed queries
    int n_win_tiles;  // 64-token tiles of the BF16 sink + recent windows
    // workspace offsets (bytes, 256-aligned)
    size_t off_len, off_req, off_cprefix, off_qt, off_qsum, off_qfrag, off_ml, off_o, off_wml, off_wo, off_cnt, total;
};

inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

inline DecodePlan make_plan(const oscar_config* cfg, int batch, int max_seq_len, int n_sm) {
    DecodePlan p;
    const int d = cfg->head_dim, Hq = cfg->num_q_heads, Hkv = cfg->num_kv_heads;
    const int g = Hq / Hkv, ng = d / cfg->group_size;
    const int64_t max_hist = std::max<int64_t>(0, (int64_t)max_seq_len - cfg->sink - cfg->recent);
    // ~64 chunks per SM of work for balance, 32..1024 tokens each
    const int64_t target = (int64_t)std::max(1, n_sm) * 64;
    int64_t c = ((int64_t)batch * max_hist + target - 1) / target;
    c = (c + 31) / 32 * 32;
    if (c < 32) c = 32;
    if (c > 1024) c = 1024;
    p.chunk = (int)c;
    p.max_ctas = std::max(1, n_sm) * 4;
    p.part_slots = std::max(p.max_ctas + batch, 2 * (std::max(1, n_sm) + batch));
    p.n_frag_tiles = (2 * g + 7) / 8;
    p.n_win_tiles = (cfg->sink + cfg->recent + 63) / 64;
    size_t off = 0;
    p.off_len = off;      off = align256(off + (size_t)batch * 4);
    p.off_req = off;      off = align256(off + (size_t)batch * 4);
    p.off_cprefix = off;  off = align256(off + (size_t)(batch + 1) * 4);
    p.off_qt = off;       off = align256(off + (size_t)batch * Hq * d * 4);
    p.off_qsum = off;     off = align256(off + (size_t)batch * Hq * ng * 8);
    p.off_qfrag = off;    off = align256(off + (size_t)batch * Hkv * p.n_frag_tiles * (d / 16) * 32 * 8);
    p.off_ml = off;       off = align256(off + (size_t)p.part_slots * Hq * 8);
    p.off_o = off;        off = align256(off + (size_t)p.part_slots * Hq * d * 4);
    p.off_cnt = off;      off = align256(off + (size_t)batch * Hkv * kCombGroups * 4);
    p.off_wml = off;      off = align256(off + (size_t)batch * Hq * p.n_win_tiles * 8);
    p.off_wo = off;       off = align256(off + (size_t)batch * Hq * p.n_win_tiles * d * 4);
    p.total = off;
    return p;
}

// Device view of the decode arguments.
struct DecodeParams {
    const void* q;
    int q_dtype;
    const int32_t* page_table;
    int64_t pt_stride;
    const int32_t* seq_lens;
    const int32_t* req_idx;
    int batch, max_seq_len;
    float* out;
    const uint8_t* records;
    const uint16_t* sink;
    const uint16_t* recent;
    const float* rot_k;
    const float* rot_v;
    int64_t num_slots;
    int max_reqs;
    int Hq, Hkv, g, S, W, G, ng, rec_bytes;
    int64_t slot_bytes;  // pool stride of one slot (all KV heads)
    int fp8;           // (s, z) stored as E4M3 pairs (else fp16 pairs)
    int chunk, n_frag_tiles, n_win_tiles;
    int n_ctas;        // history grid actually launched (<= plan.max_ctas)
    int par;           // partial slots per (CTA, request): stage parities of the history kernel
    float qscale;      // log2(e) / sqrt(d)
    // workspace
    int32_t* len;      // effective L per request (0 when invalid)
    int32_t* req;      // window row per request
    int32_t* cprefix;  // exclusive prefix of history chunk counts, [batch + 1]
    float* qt;         // q·R_K·qscale, [batch][Hq][d]
    float2* qsum;      // per group of the fp16 hi+lo parts of q̃: (Σ q̃, Σ q̃/α) with α the
                       // per-channel code weight of the MMA path, [batch][Hq][ng]
    uint2* qfrag;      // fp16 hi/lo B fragments, [batch][Hkv][n_tiles][d/16][32]
    float2* ml;        // (m, l) per partial slot, [part_slots][Hq]
    float* po;         // unnormalised o per partial slot, [part_slots][Hq][d]
    int* comb_count;   // combine: merged slices per (request, KV head, head group), [batch][Hkv][kCombGroups]; zeroed by prep
    float2* wml;       // (m, l) per BF16 window tile, [batch][Hq][n_win_tiles]
    float* wo;         // unnormalised o per BF16 window tile, [batch][Hq][n_win_tiles][d]
    int* status;
};

}  // namespace oscar

namespace oscar {

// Tensor-core code encoding for group sizes >= 64.  A code at position p of a
// 32-bit word of 16 codes (bits 2p, 2p+1 of each 16-bit half) enters the MMA as
// the exact fp16 subnormal c·2^(bit - 24) after one AND, on the word itself for
// p <= 4 (bit = 2p) or on the word >> 6 for p = 5, 6, 7 (bit = 2p - 6).
__host__ __device__ constexpr int sub_bit(int p) { return p <= 4 ? 2 * p : 2 * p - 6; }
// The four register slots of a word: (first, second) position of slot s.
__host__ __device__ constexpr int slot_pos(int s, int second) {
    return s == 0 ? (second ? 4 : 3) : s == 1 ? (second ? 5 : 2) : s == 2 ? (second ? 7 : 6) : (second ? 1 : 0);
}
// The query operand of channel at position p is q̃·2^(kQkExp - bit) (at most 256·q̃,
// inside the fp16 range), so a QK product is q̃·c·2^(kQkExp - 24).
constexpr int kQkExp = 8;

// CTA of the history grid that owns flattened chunk f (N chunks over n CTAs).
__host__ __device__ __forceinline__ int64_t chunk_owner(int64_t f, int64_t N, int64_t n) {
    return ((f + 1) * n - 1) / N;
}

}  // namespace oscar
