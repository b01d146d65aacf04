// Decode-attention plan and workspace layout shared by the decode kernels.
#pragma once

#include <stdint.h>
#include <stddef.h>

#include "oscar_internal.h"

namespace oscar {

// The history of each request is cut into chunks of `chunk` tokens; a
// persistent history grid takes contiguous runs of the flattened chunk list,
// and each run inside one request produces one (m, l, o) partial, stored at
// the slot of its first chunk (the other chunks of the run get a marker).
struct DecodePlan {
    int chunk;        // tokens per chunk (multiple of 32)
    int max_chunks;   // chunk slots per request
    int n_frag_tiles; // n-tiles of 8 columns for the fragment-packed queries
    // workspace offsets (bytes, 256-aligned)
    size_t off_len, off_req, off_cprefix, off_qt, off_qsum, off_qfrag, off_ml, off_o, total;
};

inline size_t align256(size_t x) { return (x + 255) / 256 * 256; }

inline DecodePlan make_plan(const oscar_config* cfg, int batch, int max_seq_len, int n_sm) {
    DecodePlan p;
    const int d = cfg->head_dim, Hq = cfg->num_q_heads, Hkv = cfg->num_kv_heads;
    const int g = Hq / Hkv, ng = d / cfg->group_size;
    const int64_t max_hist = std::max<int64_t>(0, (int64_t)max_seq_len - cfg->sink - cfg->recent);
    // aim for ~16 chunks per CTA-slot of a 2-per-SM grid, 32..1024 tokens each
    const int64_t target = (int64_t)std::max(1, n_sm) * 32;
    int64_t c = ((int64_t)batch * max_hist + target - 1) / target;
    c = (c + 31) / 32 * 32;
    if (c < 32) c = 32;
    if (c > 1024) c = 1024;
    p.chunk = (int)c;
    p.max_chunks = (int)std::max<int64_t>(1, (max_hist + c - 1) / c);
    p.n_frag_tiles = (2 * g + 7) / 8;
    size_t off = 0;
    p.off_len = off;      off = align256(off + (size_t)batch * 4);
    p.off_req = off;      off = align256(off + (size_t)batch * 4);
    p.off_cprefix = off;  off = align256(off + (size_t)(batch + 1) * 4);
    p.off_qt = off;       off = align256(off + (size_t)batch * Hq * d * 4);
    p.off_qsum = off;     off = align256(off + (size_t)batch * Hq * ng * 4);
    p.off_qfrag = off;    off = align256(off + (size_t)batch * Hkv * p.n_frag_tiles * (d / 16) * 32 * 8);
    p.off_ml = off;       off = align256(off + (size_t)batch * p.max_chunks * Hq * 8);
    p.off_o = off;        off = align256(off + (size_t)batch * p.max_chunks * Hq * d * 4);
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
    int chunk, max_chunks, n_frag_tiles;
    float qscale;      // log2(e) / sqrt(d)
    // workspace
    int32_t* len;      // effective L per request (0 when invalid)
    int32_t* req;      // window row per request
    int32_t* cprefix;  // exclusive prefix of history chunk counts, [batch + 1]
    float* qt;         // q·R_K·qscale, [batch][Hq][d]
    float* qsum;       // per-group sums of the fragment-packed q̃, [batch][Hq][ng]
    uint2* qfrag;      // fp16 hi/lo B fragments, [batch][Hkv][n_tiles][d/16][32]
    float2* ml;        // (m, l) per chunk slot, [batch][max_chunks][Hq]
    float* po;         // unnormalised o per chunk slot, [batch][max_chunks][Hq][d]
    int* status;
};

}  // namespace oscar
