// moe_common.cuh -- pieces shared by the MoE forward and backward kernels:
// the layer geometry, the forward workspace layout (the backward reads the
// forward's saved tensors from it), ready-queue primitives and small helpers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "mxfp8.cuh"

namespace kosmos {

constexpr int MOE_MAXK = 8;
constexpr int MOE_SCRATCH = 12288;          // epilogue 8 KB + producer 4 KB
constexpr int MOE_SF_BYTES = 3 * 512;       // MXFP8: per stage, SFA atom + two SFB atoms
constexpr int MOE_STG_BYTES = 2048;         // per epilogue warp: one 32 x 32 bf16 box of a D tile
constexpr int MOE_SMEM_BYTES = SMEM_BYTES + MOE_SCRATCH + NSTAGE * MOE_SF_BYTES + 4 * MOE_STG_BYTES;
static_assert(MOE_SMEM_BYTES <= 232448, "MoE forward exceeds 227 KB of shared memory per CTA");
static_assert(MOE_SMEM_BYTES <= 232448, "MoE kernel exceeds 227 KB of shared memory per CTA");
constexpr int MOE_QR = 16;                  // MXFP8: token rows per QUANT entry
// aux[2] of a forward workspace after a complete bf16 forward: its saved
// context (g, u, h, slots, logits, tables) is what the backward reads
constexpr uint32_t MOE_BF16_CTX = 0x4B4D4642u;
constexpr int K_QUANT = 11;                 // rail kind of a QUANT entry

struct MoeGeom {
    bool mx;         // MXFP8 expert GEMMs
    int P, E, Eq, K;
    int64_t T, Tq, H, I;
    int RB;          // route blocks per rank
    int NB;          // route blocks in total
    int NGU;         // TILE_GU column blocks (I / 128)
    int ND;          // TILE_D column blocks = push / fold column tiles (H / 256)
    int MAXRB;       // row blocks an expert can need (ceil(T / 128))
    int64_t rows_cap;
    int push_cap;    // per rank
    int fold_cap;    // per rank
    int NQ;          // QUANT entries per rank (MXFP8; else 0)
    int n_head;      // RB + NQ + RB*K main-rail entries before the tiles
    int nkb_r;       // router K blocks: H / 64
    int nkb_h;       // GU K stages: H / 64 (bf16) or H / 128 (MXFP8)
    int nkb_i;       // D K stages: I / 64 or I / 128
};

inline MoeGeom moe_geom(int P, int64_t T, int64_t H, int E, int K, int64_t I, bool mx) {
    MoeGeom g;
    g.mx = mx;
    g.P = P; g.E = E; g.Eq = E / P; g.K = K;
    g.T = T; g.Tq = T / P; g.H = H; g.I = I;
    g.RB = static_cast<int>(cdiv(g.Tq, BM));
    g.NB = P * g.RB;
    g.NGU = static_cast<int>(I / 128);
    g.ND = static_cast<int>(H / BN);
    g.MAXRB = static_cast<int>(cdiv(T, BM));
    // MXFP8: every expert's rows start on a 128-row boundary (at most E * 127
    // padding rows), and the buffer is whole 128-row scale atoms
    g.rows_cap = mx ? align_up(T * K + static_cast<int64_t>(E + 1) * BM, BM) : T * K + BM;
    g.push_cap = static_cast<int>((g.Eq + cdiv(T * K, BM)) * g.ND);
    g.fold_cap = g.RB * g.ND;
    g.NQ = mx ? static_cast<int>(cdiv(g.Tq, MOE_QR)) : 0;
    g.n_head = g.RB + g.NQ + g.RB * K;
    const int kst = mx ? FBK : BK;
    g.nkb_r = static_cast<int>(H / BK);
    g.nkb_h = static_cast<int>(H / kst);
    g.nkb_i = static_cast<int>(I / kst);
    return g;
}

struct MoeWsLayout {
    size_t ctr, ctr_bytes, disp_cnt, gu_cnt, fold_cnt, quant_cnt, qctl, route_done;
    size_t blk_counts, rank_in_blk, base, offsets, offl, counts, unit_start, inv_pos;
    size_t push_items, push_flags, fold_items, fold_flags;
    size_t logits, xq, xs, recv, recv_sf, h, h_sf, ybuf, slot, gsave, usave, trace, total;
};

inline MoeWsLayout moe_ws_layout(const MoeGeom &g, bool trace) {
    MoeWsLayout L;
    size_t off = 256;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = static_cast<size_t>(align_up(static_cast<int64_t>(off + bytes), 256));
        return at;
    };
    // counters returned to zero by the last CTA of every launch
    L.ctr = off;
    size_t c = off;
    L.disp_cnt = c; c += 4ull * g.E * g.MAXRB;
    L.gu_cnt = c; c += 4ull * g.E * g.MAXRB;
    L.fold_cnt = c; c += 4ull * g.NB * g.ND;
    L.quant_cnt = c; c += 4ull * g.NB;
    L.qctl = c; c += 4ull * 4 * g.P;
    L.route_done = c; c += 4;
    L.ctr_bytes = static_cast<size_t>(align_up(static_cast<int64_t>(c - L.ctr), 16));
    off = L.ctr;
    take(L.ctr_bytes);
    L.blk_counts = take(4ull * g.NB * g.E);
    L.rank_in_blk = take(4ull * g.T * g.K);
    L.base = take(4ull * g.NB * g.E);
    L.offsets = take(4ull * (g.E + 1));
    L.offl = take(4ull * (g.E + 1));
    L.counts = take(4ull * g.E);
    L.unit_start = take(4ull * g.P * (g.Eq + 1));
    L.inv_pos = take(4ull * g.rows_cap);
    L.push_items = take(4ull * g.P * g.push_cap);
    L.push_flags = take(4ull * g.P * g.push_cap);
    L.fold_items = take(4ull * g.P * g.fold_cap);
    L.fold_flags = take(4ull * g.P * g.fold_cap);
    L.logits = take(4ull * g.T * g.E);
    const size_t esz = g.mx ? 1 : 2;
    L.xq = g.mx ? take(static_cast<size_t>(g.T * g.H)) : 0;
    L.xs = g.mx ? take(static_cast<size_t>(g.T * g.H / 32)) : 0;
    L.recv = take(esz * g.rows_cap * g.H);
    L.recv_sf = g.mx ? take(static_cast<size_t>(g.rows_cap * g.H / 32)) : 0;
    L.h = take(esz * g.rows_cap * g.I);
    L.h_sf = g.mx ? take(static_cast<size_t>(g.rows_cap * g.I / 32)) : 0;
    L.ybuf = take(2ull * g.rows_cap * g.H);
    L.slot = take(2ull * g.T * g.K * g.H);
    // bf16 layer: the SwiGLU inputs g = x W_gate and u = x W_up of every
    // receive row, kept for the backward
    L.gsave = g.mx ? 0 : take(2ull * g.rows_cap * g.I);
    L.usave = g.mx ? 0 : take(2ull * g.rows_cap * g.I);
    L.trace = off;
    if (trace) take(static_cast<size_t>(MAX_CTAS) * TRACE_CAP * sizeof(TraceRec));
    L.total = off;
    return L;
}

// Data written earlier in the same launch by other CTAs is read through L2
// only (ld.global.cg): an L1 line filled before the writer finished would be
// stale.
__device__ __forceinline__ int32_t ldcg_i32(const int32_t *p) { return __ldcg(p); }
__device__ __forceinline__ float ldcg_f32(const float *p) { return __ldcg(p); }
__device__ __forceinline__ uint4 ldcg_u4(const void *p) { return __ldcg(reinterpret_cast<const uint4 *>(p)); }

__device__ __forceinline__ void red_relaxed_add_gpu(uint32_t *p, uint32_t v) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acqrel_gpu(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Publish one item into a ready queue: reserve an index, write the item, then
// release its per-item flag (epoch-tagged).
__device__ __forceinline__ void queue_put(uint32_t *tail, int32_t *items, uint32_t *flags, int cap, int32_t code,
                                          uint32_t epoch, WsHeader *ws) {
    const uint32_t idx = atomicAdd(tail, 1u);
    if (idx >= static_cast<uint32_t>(cap)) {
        set_error(ws, KOSMOS_ERR_DEVICE, -20);
        return;
    }
    items[idx] = code;
    st_release_gpu(&flags[idx], epoch + 1u);
}

// Take the next item if one has been published; non-blocking except for the
// few cycles between a publisher's reservation and its flag release.
__device__ __forceinline__ bool queue_try_take(uint32_t *head, uint32_t *tail, const int32_t *items,
                                               const uint32_t *flags, uint32_t epoch, int32_t &code,
                                               WsHeader *ws) {
    const uint32_t h = ld_relaxed_gpu(head);
    if (h >= ld_acquire_gpu(tail)) return false;
    if (atomicCAS(head, h, h + 1u) != h) return false;
    if (!wait_flag_eq(ws, &flags[h], epoch + 1u, PIPE_LIMIT_NS, -21)) return false;
    code = *reinterpret_cast<const volatile int32_t *>(&items[h]);
    return true;
}

__device__ __forceinline__ int32_t push_code(int e, int rb, int dn) { return e | (rb << 9) | (dn << 20); }
__device__ __forceinline__ void push_decode(int32_t c, int &e, int &rb, int &dn) {
    e = c & 511; rb = (c >> 9) & 2047; dn = (c >> 20) & 4095;
}

__device__ __forceinline__ void fill_entry(SchedEntry &e, int kind, int a, int b, int c, int nstage, int ticket,
                                           int slot) {
    e.kind = kind; e.a = a; e.b = b; e.c = c; e.d = 0; e.nstage = nstage; e.ticket = ticket; e.slot = slot;
    e.nmma = 0; e.x0 = e.x1 = e.x2 = 0;
}

// Exclusive prefix sum of n values by one warp (lane l takes a run of
// consecutive values); with div > 0 each value v counts as ceil(v / div).
// Returns the total.
__device__ __forceinline__ int warp_excl_scan(const int32_t *in, int32_t *out, int n, int lane, int div) {
    const int per = (n + 31) / 32;
    const int i0 = lane * per;
    int loc = 0;
    for (int i = i0; i < i0 + per && i < n; ++i) loc += div > 0 ? (in[i] + div - 1) / div : in[i];
    int incl = loc;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += v;
    }
    int run = incl - loc;
    for (int i = i0; i < i0 + per && i < n; ++i) {
        out[i] = run;
        run += div > 0 ? (in[i] + div - 1) / div : in[i];
    }
    return __shfl_sync(0xFFFFFFFFu, incl, 31);
}

// fp32 silu through the fast exponential and the approximate division (a
// few ulp; h is rounded to bf16 or quantised to E4M3 after it): the
// correctly rounded division took a large share of the SwiGLU epilogue
__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

}  // namespace kosmos
