// common.cuh -- workspace layout, entry kinds, tile geometry and the rail
// decode shared by the host library and the kernels.
//
// A rail is the ordered list of entries of one queue.  Entries are never
// stored: a claimed ticket t is decoded arithmetically into its entry
// ("the order of the rail is the schedule", KOSMOS explainer, paragraph
// "Role switching only works").
#pragma once
#include <cstddef>
#include <cstdint>

#include "../../include/kosmos.h"

#ifdef __CUDACC__
#define KOS_HD __host__ __device__ __forceinline__
#else
#define KOS_HD inline
#endif

namespace kosmos {

// ---------------------------------------------------------------- tiles
constexpr int BM = 128;            // tile rows (= tcgen05 M, = TMEM lanes)
constexpr int BN = 256;            // tile columns (= tcgen05 N)
constexpr int BK = 64;             // K per pipeline stage (bf16: 128 bytes = one swizzle row)
constexpr int UMMA_K = 16;         // K per tcgen05.mma (kind::f16)
constexpr int NSTAGE = 4;          // shared-memory pipeline depth
constexpr int A_STAGE_BYTES = BM * BK * 2;
constexpr int B_STAGE_BYTES = BK * BN * 2;
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int PBM = 256;           // tile rows of an SM pair (tcgen05 cta_group::2, M = 256)
constexpr int PIECE_ROWS = BM;     // all-gather piece height (one tile row): the unit a tile waits for
constexpr int PART_ROWS = 32;      // all-gather transfer entry height: a piece arrives in PIECE_PARTS parts
constexpr int PIECE_PARTS = PIECE_ROWS / PART_ROWS;
constexpr int NSCHED = 4;          // depth of the in-CTA entry ring
constexpr int NUM_THREADS = 192;   // warp 0 scheduler/producer, warp 1 MMA, warps 2-5 epilogue
constexpr int NUM_EPI_THREADS = 128;
constexpr int TMEM_COLS = 512;     // two 128x256 fp32 accumulators
constexpr int RED_ROWS = 8;        // rows of one reduce stage (P x 8 x 256 bf16 <= 32 KB)
constexpr int SF_ATOM_ROWS = 4;    // an MXFP8 scale atom (512 bytes) as tensor-map rows of 128 bytes
constexpr int MAX_CTAS = 256;
constexpr int TRACE_CAP = 1024;    // trace records per CTA

enum EntryKind : int32_t {
    K_NONE = 0,
    K_TRANSFER = 1,
    K_TILE = 2,
    K_REDUCE = 3,
    K_ROUTE = 4,
    K_DISPATCH = 5,
    K_TILE_GU = 6,
    K_TILE_D = 7,
    K_PUSH = 8,
    K_FOLD = 9,
    K_TILE_HALF = 10,  // rail decode only: a tile's column half (the kernels run it as a K_TILE of BN/2 columns)
    K_DONE = 15
};

// ---------------------------------------------------------------- workspace
// Offset 0 of every workspace.  Tickets and done_ctas are returned to zero by
// the last CTA of every successful launch; epoch then advances, so readiness
// flags written as (epoch + 1) need no clearing between calls.
struct WsHeader {
    uint32_t epoch;
    uint32_t status;       // kosmos_status of the device side (0 = OK)
    uint32_t done_ctas;
    uint32_t pad0;
    int64_t fail_entry;    // ticket (or encoded entry) that failed, -1 none
    uint32_t tickets[40];  // rail counters
    uint32_t aux[4];
    uint64_t link_t0;      // emulated link: globaltimer of the launch's first reservation (0 = none yet)
    uint64_t link_bytes;   // emulated link: bytes reserved so far in this launch
};
static_assert(sizeof(WsHeader) <= 256, "header must fit its 256-byte slot");

struct TraceRec {
    int64_t t_claim, t_ready, t_done;
    int32_t kind, ticket, cta, pad;
};
static_assert(sizeof(TraceRec) == sizeof(kosmos_trace_rec), "trace record layout");

KOS_HD int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
KOS_HD int64_t align_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }

// ---------------------------------------------------------------- AG geometry / rails
struct AgGeom {
    int P;
    int64_t m, k, n;
    int pieces;      // 128-row pieces per shard (one readiness flag each)
    int parts;       // transfer entries per piece (PART_ROWS rows each)
    int tile_rows;   // 128 (one SM per tile) or 256 (an SM pair per tile)
    int tiles_m;     // tile rows per shard
    int tiles_n;
    int n_transfer;  // P * pieces * parts: remote shards first, the local shard's copies last
    int n_full;      // P * tiles_m * tiles_n whole tiles
    int n_split;     // the last n_split of them run as two column halves each
    int n_tile;      // tile rail length: n_full + n_split
};
KOS_HD AgGeom ag_geom(int P, int64_t m, int64_t k, int64_t n, int tile_rows = BM, int64_t n_split = 0) {
    AgGeom g;
    g.P = P; g.m = m; g.k = k; g.n = n;
    g.pieces = static_cast<int>(cdiv(m, PIECE_ROWS));
    g.parts = PIECE_PARTS;
    g.tile_rows = tile_rows;
    g.tiles_m = static_cast<int>(cdiv(m, tile_rows));
    g.tiles_n = static_cast<int>(cdiv(n, BN));
    g.n_transfer = P * g.pieces * g.parts;
    g.n_full = P * g.tiles_m * g.tiles_n;
    g.n_split = static_cast<int>(n_split < 0 ? 0 : (n_split > g.n_full ? g.n_full : n_split));
    g.n_tile = g.n_full + g.n_split;
    return g;
}
// Transfer rail: shards 1..P-1 in the order the tiles consume them, then
// shard 0; inside a shard, pieces in row order, each as `parts` row-ordered
// parts.  A piece's flag reaches (epoch + 1) * parts when all its parts have
// landed.
KOS_HD void ag_decode_transfer(const AgGeom &g, int t, int &shard, int &piece, int &part) {
    const int per_shard = g.pieces * g.parts;
    const int sidx = t / per_shard;
    const int r = t - sidx * per_shard;
    piece = r / g.parts;
    part = r - piece * g.parts;
    shard = (sidx + 1 < g.P) ? sidx + 1 : 0;
}
// Rows [row0, row0 + rows) of a shard carried by transfer part (piece, part); rows may be 0.
KOS_HD void ag_part_rows(const AgGeom &g, int piece, int part, int64_t &row0, int64_t &rows) {
    row0 = static_cast<int64_t>(piece) * PIECE_ROWS + static_cast<int64_t>(part) * PART_ROWS;
    const int64_t left = g.m - row0;
    rows = left <= 0 ? 0 : (left < PART_ROWS ? left : PART_ROWS);
}
KOS_HD uint32_t ag_piece_ready(const AgGeom &g, uint32_t epoch) {
    return (epoch + 1u) * static_cast<uint32_t>(g.parts);
}
// Tile rail: shard-major (local shard 0 first), tile rows, then tile columns;
// the last n_split tiles of that order appear as their two column halves,
// left half first.  Returns K_TILE (tcol counts BN columns) or K_TILE_HALF
// (tcol counts BN / 2 columns).
KOS_HD int ag_decode_tile(const AgGeom &g, int t, int &shard, int &trow, int &tcol) {
    const int keep = g.n_full - g.n_split;
    int f = t, half = -1;
    if (t >= keep) {
        const int h = t - keep;
        f = keep + h / 2;
        half = h - (h / 2) * 2;
    }
    const int per_shard = g.tiles_m * g.tiles_n;
    shard = f / per_shard;
    const int r = f - shard * per_shard;
    trow = r / g.tiles_n;
    tcol = r - trow * g.tiles_n;
    if (half < 0) return K_TILE;
    tcol = 2 * tcol + half;
    return K_TILE_HALF;
}

// ---------------------------------------------------------------- RS geometry / rails
struct RsGeom {
    int P;
    int64_t m, k, n;
    int64_t mc;       // rows per chunk = m / P
    int band_rows;    // 128 (one SM per tile) or 256 (an SM pair per tile)
    int bands;        // tile rows per chunk
    int tiles_n;
    int n_tile;       // one rail for all ranks: P * P * bands * tiles_n
    int n_reduce;     // per rank: bands * tiles_n
};
KOS_HD RsGeom rs_geom(int P, int64_t m, int64_t k, int64_t n, int band_rows = BM) {
    RsGeom g;
    g.P = P; g.m = m; g.k = k; g.n = n;
    g.mc = m / P;
    g.band_rows = band_rows;
    g.bands = static_cast<int>(cdiv(g.mc, band_rows));
    g.tiles_n = static_cast<int>(cdiv(n, BN));
    g.n_tile = P * P * g.bands * g.tiles_n;
    g.n_reduce = g.bands * g.tiles_n;
    return g;
}
// Tile rail shared by all ranks: TILE(rank, chunk, band, column) of the
// rank's partial.  Band order: band, rank, column, chunk (one rank's band at a
// time, the P tiles that share one W_rank column slice adjacent: the tiles in
// flight read one band of X_rank and a few W_rank slices, which stay in L2).
// Row order: chunk, band, rank, column.
KOS_HD void rs_decode_tile(const RsGeom &g, int order, int t, int &rank, int &chunk, int &band, int &tcol) {
    if (order == KOSMOS_ORDER_BAND) {
        const int per_rank = g.P * g.tiles_n;
        const int per_band = g.P * per_rank;
        band = t / per_band;
        int r = t - band * per_band;
        rank = r / per_rank;
        r -= rank * per_rank;
        tcol = r / g.P;
        chunk = r - tcol * g.P;
    } else {
        const int per_rank = g.tiles_n;
        const int per_band = g.P * per_rank;
        const int per_chunk = g.bands * per_band;
        chunk = t / per_chunk;
        int r = t - chunk * per_chunk;
        band = r / per_band;
        r -= band * per_band;
        rank = r / per_rank;
        tcol = r - rank * per_rank;
    }
}
// Reduce rail of rank r (its own chunk): band, then column.
KOS_HD void rs_decode_reduce(const RsGeom &g, int t, int &band, int &tcol) {
    band = t / g.tiles_n;
    tcol = t - band * g.tiles_n;
}

// ---------------------------------------------------------------- workspace layouts
// K-split tail tiles: each split tile owns a slot with, per CTA of the tile
// engine (two for an SM pair), an arrival counter, a ready flag and an fp32
// partial of 128 rows x 256 columns, stored as [64 column quads][128 rows] of float4.
constexpr int MAX_SPLIT_SLOTS = 256;
constexpr size_t KPART_CTA_BYTES = static_cast<size_t>(BM) * BN * 4;
struct AgWsLayout {
    size_t flags_off, ksync_off, kpart_off, trace_off, ext_off, total;
};
// Host-input flow: a shard arrives from the host in at most AG_HOST_CHUNKS
// chunks of whole 128-row pieces, each with an arrival word, and its output
// rows go back in at most AG_HOST_GROUPS groups of whole tile rows, each with
// an output-tile count (the last shard, whose tiles and output copies end the
// call, in at most AG_HOST_LAST_CHUNKS and AG_HOST_LAST_GROUPS).  Region:
// [KOSMOS_MAX_P][AG_EXT_STRIDE] arrival words, the same for the counts, then
// three stream-join words.
constexpr int AG_HOST_CHUNKS = 1;
constexpr int AG_HOST_GROUPS = 2;
constexpr int AG_HOST_LAST_CHUNKS = 2;
constexpr int AG_HOST_LAST_GROUPS = 2;
constexpr int AG_EXT_STRIDE = 8;                              // words per shard in each array
constexpr int AG_EXT_WORDS = KOSMOS_MAX_P * AG_EXT_STRIDE;    // words of each of the two arrays
constexpr int AG_EXT_BYTES = 1024;
static_assert(AG_HOST_CHUNKS <= AG_EXT_STRIDE && AG_HOST_GROUPS <= AG_EXT_STRIDE &&
                  AG_HOST_LAST_CHUNKS <= AG_EXT_STRIDE && AG_HOST_LAST_GROUPS <= AG_EXT_STRIDE,
              "host-flow words per shard");
static_assert(2 * AG_EXT_WORDS * 4 + 3 * 4 <= AG_EXT_BYTES, "host-flow words exceed their region");
// pieces per arrival chunk and tile rows per output group of shard s
KOS_HD int ag_host_cpp(const AgGeom &g, int s) {
    return static_cast<int>(cdiv(g.pieces, s == g.P - 1 ? AG_HOST_LAST_CHUNKS : AG_HOST_CHUNKS));
}
KOS_HD int ag_host_tpg(const AgGeom &g, int s) {
    return static_cast<int>(cdiv(g.tiles_m, s == g.P - 1 ? AG_HOST_LAST_GROUPS : AG_HOST_GROUPS));
}
// Written to the output-done counters when a launch fails or never starts: a
// stream wait "value >= target" compares (int32_t)(word - target) >= 0, so the
// release value must stay below 2^31 above any target.
constexpr uint32_t AG_YDONE_RELEASE = 0x40000000u;
inline AgWsLayout ag_ws_layout(const AgGeom &g, bool trace, int n_slots = 0) {
    AgWsLayout L;
    L.flags_off = 256;
    size_t off = L.flags_off + static_cast<size_t>(align_up(static_cast<int64_t>(g.P) * g.pieces * 4, 256));
    L.ksync_off = off;
    off += static_cast<size_t>(align_up(static_cast<int64_t>(n_slots) * 2 * 2 * 4, 256));
    L.kpart_off = off;
    off += static_cast<size_t>(n_slots) * 2 * KPART_CTA_BYTES;
    L.trace_off = off;
    if (trace) off += static_cast<size_t>(MAX_CTAS) * TRACE_CAP * sizeof(TraceRec);
    L.ext_off = off;
    off += AG_EXT_BYTES;
    L.total = off;
    return L;
}
struct RsWsLayout {
    size_t arrive_off, partial_off, trace_off, total;
};
inline RsWsLayout rs_ws_layout(const RsGeom &g, bool trace) {
    RsWsLayout L;
    L.arrive_off = 256;
    size_t off = L.arrive_off + static_cast<size_t>(align_up(static_cast<int64_t>(g.P) * g.bands * g.tiles_n * 4, 1024));
    L.partial_off = off;
    off += static_cast<size_t>(align_up(static_cast<int64_t>(g.P) * g.m * g.n * 2, 1024));
    L.trace_off = off;
    if (trace) off += static_cast<size_t>(MAX_CTAS) * TRACE_CAP * sizeof(TraceRec);
    L.total = off;
    return L;
}

}  // namespace kosmos
