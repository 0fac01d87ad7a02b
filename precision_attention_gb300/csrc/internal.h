// internal.h -- layouts shared by the host launchers and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>

namespace pa {

// Device status word bits (bit e = attn_status e), OR-ed by kernels.
constexpr uint32_t ST_TIMEOUT = 1u << 4;
constexpr uint32_t ST_NONFINITE = 1u << 5;
constexpr uint32_t ST_BAD_SEQLENS = 1u << 7;

// Largest document count the quantiser keeps its document table for in shared
// memory (built by every CTA); larger batches get the table in the workspace,
// written by one extra launch before the quantiser.
constexpr int MAX_DOCS = 1024;

// One document of the packed batch, as the forward reads it.
struct DocEntry {
    int32_t start;    // first token
    int32_t len;      // tokens
    int32_t toff;     // first 128-token tile (prefix of ceil(L / 128))
    int32_t boff_q;   // first scale block of Q (prefix of ceil(L / block_q))
    int32_t boff_k;
    int32_t boff_v;
    int32_t poff;     // first query-tile pair (prefix of ceil(ceil(L / 128) / 2))
    int32_t pad1;
};

// One unit of forward work: the 128-row query tile `qtile` of (doc, head), or,
// in pair mode, the query tiles 2 * qtile and 2 * qtile + 1.
struct WorkItem {
    int32_t doc;
    int32_t head;
    int32_t qtile;
    int32_t ntiles;   // key tiles to visit
};

// Workspace layout: [header 256 B][docs][items][vref][tile multipliers][quantiser
// document table: start, tile prefix, block prefix, each num_docs + 1 ints]
struct WsLayout {
    size_t docs_off, items_off, vref_off, tsc_off, qtab_off, total;
    int64_t items_cap, vref_cap, tsc_cap;   // tsc_cap: 128-token tiles per head (bound)
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WsLayout ws_layout(int64_t T, int64_t H, int64_t nd) {
    WsLayout w;
    w.items_cap = H * ((T + 127) / 128 + nd);
    w.vref_cap = H * (T > nd ? T : nd);
    w.docs_off = 256;
    w.items_off = align_up(w.docs_off + sizeof(DocEntry) * static_cast<size_t>(nd), 256);
    w.vref_off = align_up(w.items_off + sizeof(WorkItem) * static_cast<size_t>(w.items_cap), 256);
    w.tsc_cap = (T + 127) / 128 + nd;
    w.tsc_off = align_up(w.vref_off + sizeof(float) * static_cast<size_t>(w.vref_cap), 256);
    w.qtab_off = align_up(w.tsc_off + 4 * sizeof(float) * static_cast<size_t>(H * w.tsc_cap), 256);
    w.total = align_up(w.qtab_off + 3 * sizeof(int32_t) * static_cast<size_t>(nd + 1), 256);
    return w;
}

// NVFP4 scales array: fp32 block scales [H][nt_cap], then the 1024-byte scale-factor
// tiles [H][nt_cap] from this byte offset
inline size_t nvfp4_sf_offset(int64_t H, int64_t nt_cap) { return align_up(static_cast<size_t>(H * nt_cap) * 4, 1024); }

// Header at the start of the workspace.
struct WsHeader {
    uint32_t status;
    int32_t n_items;
    int32_t n_tiles;
    int32_t ticket;      // next item of the just-in-time schedule (written by the work-list pass)
    int32_t pad[60];
};

}  // namespace pa
