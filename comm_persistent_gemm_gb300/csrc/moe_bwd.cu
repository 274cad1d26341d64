// moe_bwd.cu -- MoE expert layer backward, fold back to router, in ONE
// persistent launch (KOSMOS abstract: "one launch per direction").
//
// Gradients of the bf16 forward layer with its top-K routing held fixed.  The
// forward's workspace is the saved context: expert-ordered token rows, the
// SwiGLU inputs g and u, h, the per-slot expert outputs, the router logits
// and the dispatch tables.  CTA c plays EP rank q = c mod P, as in the
// forward.  Rail of rank q (claimed in ticket order by rank q's CTAs):
//   ZPAD            zero rows that pad each of rank q's experts to 16 rows
//                   in the backward's expert-ordered buffers;
//   GRADIN(b, k)    the combine's backward = a dispatch: slot k of the 128
//                   tokens of block b: dgate = <dout, y_slot>, and the row
//                   dy = gate * dout goes to the expert-ordered buffer;
//   RBWD(b)         router backward of the block once its K slots are in:
//                   dl = softmax' of the renormalised top-K gates;
//   RDX(b, hc)      dx_router = dl . W_router^T (256 columns of hidden);
//   expert tiles    per expert j, grouped like the forward with a lag of one
//                   expert:
//                   DH(j) | DWD(j) | DGU(j-1) | DWGU(j-1)
//                   DH:   dh = dy . W_down^T (256 columns of inter) with the
//                         SwiGLU backward in the epilogue: dg, du;
//                   DWD:  dW_down = h^T . dy over the expert's rows;
//                   DGU:  dx_e = dg . W_gate^T + du . W_up^T;
//                   DWGU: dW_gate, dW_up = x^T . [dg | du];
//   DWR(hb)         dW_router rows = x^T . dl over every token (after all
//                   RBWD entries).
// Ready queues as in the forward: PUSH(e, rb, hc) when a DGU tile finishes
// (dx_e rows back to their token slots), FOLD(g, hc) when all K slots and
// the router part of a token block's column tile are in:
// dx = sum_k dx_slot[t][k] (k order) + dx_router, one rounding to bf16.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>

#include "moe_common.cuh"
#include "launch.h"

namespace kosmos {

enum BwdKind : int {
    KB_ZPAD = 16, KB_GRADIN = 17, KB_RBWD = 18, KB_RDX = 19, KB_DH = 20, KB_DGU = 21, KB_DWD = 22, KB_DWGU = 23,
    KB_DWR = 24
};
__device__ __forceinline__ bool bwd_is_mma(int k) {
    return k == KB_RDX || k == KB_DH || k == KB_DGU || k == KB_DWD || k == KB_DWGU || k == KB_DWR;
}
constexpr int BWD_LAG = 1;  // experts between an expert's DH tiles and its DWGU tiles (DGU: always 1)
constexpr int BWD_GROUP = 4;  // weight-gradient tiles per rail ticket (at most)
// A DH tile's SwiGLU inputs g and u reach its epilogue through three more
// pipeline stages after its K loop: per 32-column chunk of the tile, the
// 128 rows of g then of u (8 KB each, 64-byte swizzled), three chunks to a
// stage (3 + 3 + 2 of the tile's 8).
constexpr int DH_EPI_STAGES = 3;
constexpr int DH_CH_BYTES = 2 * BM * 32 * 2;
// shared memory: the engine's stages and control, the per-CTA tables, and
// per epilogue warp a 4 KB staging buffer for the dW and the dg / du stores
constexpr int BWD_TABLE_BYTES = 5120;
constexpr int BWD_STAGE_OUT = 2048;
constexpr int BWD_SMEM_BYTES = SMEM_BYTES + BWD_TABLE_BYTES + 4 * 2 * BWD_STAGE_OUT;
static_assert(BWD_SMEM_BYTES <= 232448, "MoE backward exceeds 227 KB of shared memory per CTA");

struct BwdGeom {
    MoeGeom f;
    int NIC;        // DH column blocks: I / 256
    int NHC;        // DGU / RDX / fold column tiles: H / 256
    int NWI;        // I / 128
    int NWH;        // H / 128
    int W1;         // DWD tiles per expert: NWI * NHC
    int W2;         // DWGU tiles per expert: NWH * NWI
    int G1, G2;     // DWD / DWGU tiles per rail ticket (4, 2 or 1: divides W1 / W2)
    int T1, T2;     // DWD / DWGU tickets per expert: W1 / G1, W2 / G2
    int64_t rows16; // rows of the 16-row-padded expert-ordered buffers
    int push_cap, fold_cap;
    int n_head;     // 1 + RB*K + RB + RB*NHC
    int nkb_h, nkb_gu, nkb_e;  // K stages: H/64, 2I/64, E/64
    int fold_tps;
    int rbwd_tps;   // RBWD: tokens' fp32 logit rows per 32 KB stage
};

inline BwdGeom bwd_geom(int P, int64_t T, int64_t H, int E, int K, int64_t I) {
    BwdGeom b;
    b.f = moe_geom(P, T, H, E, K, I, false);
    b.NIC = static_cast<int>(I / 256);
    b.NHC = static_cast<int>(H / 256);
    b.NWI = static_cast<int>(I / 128);
    b.NWH = static_cast<int>(H / 128);
    b.W1 = b.NWI * b.NHC;
    b.W2 = b.NWH * b.NWI;
    b.G1 = b.W1 % BWD_GROUP == 0 ? BWD_GROUP : (b.W1 % 2 == 0 ? 2 : 1);
    b.G2 = b.W2 % BWD_GROUP == 0 ? BWD_GROUP : (b.W2 % 2 == 0 ? 2 : 1);
    b.T1 = b.W1 / b.G1;
    b.T2 = b.W2 / b.G2;
    b.rows16 = align_up(T * K + static_cast<int64_t>(E) * 16, BM) + BM;
    b.push_cap = static_cast<int>((b.f.Eq + cdiv(T * K, BM)) * b.NHC);
    b.fold_cap = b.f.RB * b.NHC;
    b.n_head = 1 + b.f.RB * K + b.f.RB + b.f.RB * b.NHC;
    b.nkb_h = static_cast<int>(H / BK);
    b.nkb_gu = static_cast<int>(2 * I / BK);
    b.nkb_e = E / BK;
    b.fold_tps = 64 / K < 16 ? 64 / K : 16;
    b.rbwd_tps = 32768 / (E * 4);  // a stage: tps x K slot rows (bf16) + tps router rows (fp32)
    return b;
}

struct BwdWsLayout {
    size_t ctr, ctr_bytes, dy_cnt, dh_cnt, dgate_cnt, rbwd_flag, rbwd_done, fold_cnt, qctl;
    size_t push_items, push_flags, fold_items, fold_flags;
    size_t dgate, dl, dxr, dy, dg, du, dxb, dslot, trace, total;
};

inline BwdWsLayout bwd_ws_layout(const BwdGeom &b, bool trace) {
    const MoeGeom &g = b.f;
    BwdWsLayout L;
    size_t off = 256;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = static_cast<size_t>(align_up(static_cast<int64_t>(off + bytes), 256));
        return at;
    };
    L.ctr = off;
    size_t c = off;
    L.dy_cnt = c; c += 4ull * g.E * g.MAXRB;
    L.dh_cnt = c; c += 4ull * g.E * g.MAXRB;
    L.dgate_cnt = c; c += 4ull * g.NB;
    L.rbwd_flag = c; c += 4ull * g.NB;
    L.rbwd_done = c; c += 4;
    L.fold_cnt = c; c += 4ull * g.NB * b.NHC;
    L.qctl = c; c += 4ull * 4 * g.P;
    L.ctr_bytes = static_cast<size_t>(align_up(static_cast<int64_t>(c - L.ctr), 16));
    take(L.ctr_bytes);
    L.push_items = take(4ull * g.P * b.push_cap);
    L.push_flags = take(4ull * g.P * b.push_cap);
    L.fold_items = take(4ull * g.P * b.fold_cap);
    L.fold_flags = take(4ull * g.P * b.fold_cap);
    L.dgate = take(4ull * g.T * g.K);
    L.dl = take(2ull * g.T * g.E);
    L.dxr = take(4ull * g.T * g.H);
    L.dy = take(2ull * b.rows16 * g.H);
    L.dg = take(2ull * b.rows16 * g.I);
    L.du = take(2ull * b.rows16 * g.I);
    L.dxb = take(2ull * b.rows16 * g.H);
    L.dslot = take(2ull * g.T * g.K * g.H);
    L.trace = off;
    if (trace) take(static_cast<size_t>(MAX_CTAS) * TRACE_CAP * sizeof(TraceRec));
    L.total = off;
    return L;
}

struct BwdParams {
    CUtensorMap tmDyA;               // dy [rows16, H]: A of DH, box {64, 128}
    CUtensorMap tmDyB;               // dy as B of DWD: box {64, 64}
    CUtensorMap tmDgA, tmDuA;        // dg, du [rows16, I]: A of DGU, box {64, 128}
    CUtensorMap tmDgB, tmDuB;        // dg, du as B of DWGU: box {64, 64}
    CUtensorMap tmH;                 // forward h [T*K, I]: MN-major A of DWD, box {64, 64}
    CUtensorMap tmGs, tmUs;          // forward g, u [T*K, I]: DH epilogue chunks, box {32, 128}, 64-byte swizzle
    CUtensorMap tmDgS, tmDuS;        // dg, du [rows16, I] (3-d, depth 1): DH epilogue stores, box {32, 16, 1}, 64-byte swizzle
    CUtensorMap tmX;                 // forward receive rows [T*K, H]: MN-major A of DWGU, box {64, 64}
    CUtensorMap tmDlA;               // dl [T, E]: A of RDX, box {64, 128}
    CUtensorMap tmDlB;               // dl as B of DWR: box {64, 64}
    CUtensorMap tmWrT;               // W_router [H, E] as K-major B of RDX: dims {E, H}, box {64, 256}
    CUtensorMap tmDslot;             // dx slots [T*K, H]: FOLD, box {256, fold_tps*K}, no swizzle
    CUtensorMap tmDxr;               // dx router part [T, H] fp32: FOLD, box {256, fold_tps}, no swizzle
    CUtensorMap tmDxbP;              // dx_e rows [rows16, H]: PUSH, box {256, 64}, no swizzle
    CUtensorMap tmLogits;            // forward logits [T, E] fp32: RBWD, box {E, rbwd_tps}, no swizzle
    CUtensorMap tmDxbS;              // dx_e rows (3-d, depth 1): DGU epilogue stores, box {32, 16, 1}, 64-byte swizzle
    CUtensorMap tmWdT[KOSMOS_MAX_P]; // W_down[q] [Eq, I, H] as K-major B of DH: dims {H, I, Eq}, box {64, 256, 1}
    CUtensorMap tmWgT[KOSMOS_MAX_P]; // W_gate[q] [Eq, H, I] as K-major B of DGU: dims {I, H, Eq}, box {64, 256, 1}
    CUtensorMap tmWuT[KOSMOS_MAX_P];
    CUtensorMap tmXs[KOSMOS_MAX_P];  // x_shards[q] [Tq, H]: MN-major A of DWR, box {64, 64}
    CUtensorMap tmDout[KOSMOS_MAX_P];  // dout[q] [Tq, H]: GRADIN, box {256, 32}, no swizzle
    CUtensorMap tmYslot;             // forward slot outputs [T, K, H]: GRADIN, box {256, 1, 32}, no swizzle
    // weight-gradient outputs, stored from shared memory in 32 x 32 blocks (no swizzle)
    CUtensorMap tmDwg[KOSMOS_MAX_P]; // dims {I, H, Eq}
    CUtensorMap tmDwu[KOSMOS_MAX_P];
    CUtensorMap tmDwd[KOSMOS_MAX_P]; // dims {H, I, Eq}
    // forward context
    const WsHeader *fwd_hdr;
    const int32_t *counts, *offl, *unit_start, *base, *rank_in_blk, *inv_pos;
    const float *logits;
    const __nv_bfloat16 *yslot, *gsave, *usave;
    // user tensors
    const int32_t *topk_idx;
    const float *topk_gate;
    const __nv_bfloat16 *dout[KOSMOS_MAX_P];
    __nv_bfloat16 *dx[KOSMOS_MAX_P];
    float *dwr;
    __nv_bfloat16 *dwg[KOSMOS_MAX_P], *dwu[KOSMOS_MAX_P], *dwd[KOSMOS_MAX_P];
    // backward workspace
    WsHeader *ws;
    uint8_t *ctr;
    int ctr_bytes;
    uint32_t *dy_cnt, *dh_cnt, *dgate_cnt, *rbwd_flag, *rbwd_done, *fold_cnt, *qctl;
    int32_t *push_items, *fold_items;
    uint32_t *push_flags, *fold_flags;
    float *dgate, *dxr;
    __nv_bfloat16 *dl, *dy, *dg, *du, *dxb, *dslot;
    TraceRec *trace;
    BwdGeom b;
    uint64_t wait_limit_ns;
    int phase;  // 0: the whole backward in this launch; 1-7: one phase of the unfused baseline
};

// Per-CTA tables in shared memory (producer scratch), filled once at the
// start from the forward's counts: 16-row-padded offsets of every expert
// (E + 1), then this rank's unit prefix (Eq + 1), counts (Eq) and unpadded
// offsets (Eq).
struct BwdTables {
    int32_t *offp;  // [E + 1]
    int32_t *us;    // [Eq + 1]
    int32_t *cnt;   // [Eq]
    int32_t *offl;  // [Eq]
};

__device__ __forceinline__ void bwd_load_tables(const BwdParams &p, const BwdTables &tb, int lane) {
    const MoeGeom &g = p.b.f;
    const int q = blockIdx.x % g.P;
    // padded offsets: exclusive scan of ceil(cnt / 16), times 16
    const int per = (g.E + 31) / 32;
    int loc = 0;
    for (int i = lane * per; i < lane * per + per && i < g.E; ++i) loc += (__ldg(&p.counts[i]) + 15) / 16;
    int incl = loc;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += v;
    }
    int run = incl - loc;
    for (int i = lane * per; i < lane * per + per && i < g.E; ++i) {
        tb.offp[i] = run * 16;
        run += (__ldg(&p.counts[i]) + 15) / 16;
    }
    if (lane == 31) tb.offp[g.E] = incl * 16;
    for (int j = lane; j <= g.Eq; j += 32) tb.us[j] = __ldg(&p.unit_start[q * (g.Eq + 1) + j]);
    for (int j = lane; j < g.Eq; j += 32) {
        tb.cnt[j] = __ldg(&p.counts[q * g.Eq + j]);
        tb.offl[j] = __ldg(&p.offl[q * g.Eq + j]);
    }
    __syncwarp();
}

// Expert-tile rail of rank q (tt = ticket - n_head).  Group j holds
//   DH(j): NIC x u_j (column block outer, row block inner), DWD(j): T1
//   (j < Eq), DGU(j-1): NHC x u_{j-1}, DWGU(j-1): T2 (0 <= j-1 < Eq)
// with u_j the row blocks of expert j and U(j) their prefix.  A DH or DGU
// ticket is one tile; a DWD / DWGU ticket is G1 / G2 consecutive tiles
// (cnt), taken by one CTA: these tiles are short, and one atomic claim per
// group saves round trips.  The long data-gradient tiles are claimed one by
// one, so that the tiles of an expert's row blocks that read the same weight
// block run side by side on different CTAs and the weights come from HBM
// once.
__device__ __forceinline__ void bwd_decode_tile(const BwdGeom &b, const int32_t *us, int tt, int &kind, int &le,
                                                int &x, int &y, int &cnt, int &hint) {
    const MoeGeom &g = b.f;
    auto U = [&](int j) { return j <= 0 ? 0 : us[j < g.Eq ? j : g.Eq]; };
    auto clampEq = [&](int v) { return v < 0 ? 0 : (v > g.Eq ? g.Eq : v); };
    auto gstart = [&](int j) { return b.NIC * U(j) + b.T1 * clampEq(j) + b.NHC * U(j - 1) + b.T2 * clampEq(j - BWD_LAG); };
    kind = 0;
    cnt = 1;
    if (tt < 0) return;
    // a CTA's tickets increase: start from the group of its previous tile
    int j0 = (hint > 0 && hint < g.Eq + BWD_LAG && gstart(hint) <= tt) ? hint : 0;
    for (int j = j0; j < g.Eq + BWD_LAG; ++j) {
        hint = j;
        const int uj = j < g.Eq ? U(j + 1) - U(j) : 0;
        const int n_dh = b.NIC * uj;
        const int n_dwd = j < g.Eq ? b.T1 : 0;
        const int uj1 = (j >= 1 && j - 1 < g.Eq) ? U(j) - U(j - 1) : 0;
        const int n_dgu = b.NHC * uj1;
        const int n_dwgu = (j >= BWD_LAG && j - BWD_LAG < g.Eq) ? b.T2 : 0;
        const int start = gstart(j);
        int r = tt - start;
        if (r < 0) return;
        if (r < n_dh) { kind = KB_DH; le = j; x = r / uj; y = r % uj; return; }  // x = ic, y = rb
        r -= n_dh;
        if (r < n_dwd) {  // first tile of the group: x = ib, y = hc
            const int t0 = r * b.G1;
            kind = KB_DWD; le = j; x = t0 / b.NHC; y = t0 % b.NHC; cnt = b.G1;
            return;
        }
        r -= n_dwd;
        if (r < n_dgu) { kind = KB_DGU; le = j - 1; x = r / uj1; y = r % uj1; return; }  // x = hc, y = rb
        r -= n_dgu;
        if (r < n_dwgu) {  // first tile of the group: x = hb, y = ib
            const int t0 = r * b.G2;
            kind = KB_DWGU; le = j - BWD_LAG; x = t0 / b.NWI; y = t0 % b.NWI; cnt = b.G2;
            return;
        }
    }
}

__device__ __forceinline__ int bwd_expert_tickets(const BwdGeom &b, const int32_t *us) {
    return (b.NIC + b.NHC) * us[b.f.Eq] + (b.T1 + b.T2) * b.f.Eq;
}

// Rows of unit (expert j of this rank, row block rb): real rows and rows
// including the 16-row padding.
__device__ __forceinline__ void unit_rows(const BwdTables &tb, int le, int rb, int &real, int &r16) {
    const int c = tb.cnt[le];
    const int c16 = (c + 15) / 16 * 16;
    real = c - rb * BM; real = real < 0 ? 0 : (real > BM ? BM : real);
    r16 = c16 - rb * BM; r16 = r16 < 0 ? 0 : (r16 > BM ? BM : r16);
}

struct BwdProdState {
    PipeState ps;
    RingState rs;
    int nrec = 0;
    bool main_done = false;
    uint64_t idle_t0 = 0;
    int hint = 0;      // tile-rail group of the previous tile
    uint32_t polls = 0;  // decide calls: the push queue is polled on every fourth while the rail lasts
    uint32_t calls = 0;
    int ready_dwd = -1, ready_dwgu = -1;  // the expert whose inputs were last confirmed complete
};

__device__ __forceinline__ int bwd_trace_open(const BwdParams &p, BwdProdState &st, int kind, int ticket) {
    int slot = -1;
    if (TraceRec *r = trace_rec(p.trace, blockIdx.x, st.nrec)) {
        const int64_t now = static_cast<int64_t>(globaltimer());
        r->t_claim = now; r->t_ready = now; r->t_done = 0;
        r->kind = kind; r->ticket = ticket; r->cta = blockIdx.x;
        slot = st.nrec;
    }
    ++st.nrec;
    return slot;
}

// Operand layouts follow the kind: the data gradients (RDX, DH, DGU) read
// both operands K-major, the weight gradients (DWD, DWGU, DWR) read both
// MN-major (the reduction runs over rows).  DWD / DWGU entries carry in x1
// the K steps of 16 of their last stage (0 = all four).
__device__ __forceinline__ bool bwd_is_wgrad(int k) { return k == KB_DWD || k == KB_DWGU || k == KB_DWR; }

__device__ __forceinline__ bool bwd_wait_stage(const BwdParams &p, const Smem &sm, PipeState &ps, int64_t entry) {
    if (!mbar_wait(&sm.empty[ps.stage], ps.phase ^ 1u, PIPE_LIMIT_NS)) {
        set_error(p.ws, KOSMOS_ERR_DEVICE, entry);
        return false;
    }
    return true;
}

// Lane 0 of the producer warp: one piece of work per call.  Returns false
// when this CTA is finished.  Inlined into the producer loop so that its
// state stays in registers: as a called function the state lived in local
// memory, and the short weight-gradient tiles waited on those round trips.
__device__ __forceinline__ bool bwd_decide(const BwdParams &p, const Smem &sm, BwdProdState &st, const BwdTables &tb,
                                        uint32_t epoch) {
    const BwdGeom &b = p.b;
    const MoeGeom &g = b.f;
    const int q = blockIdx.x % g.P;
    uint32_t *qc = p.qctl + 4 * q;
    // the status word is a round trip to L2: read on every eighth call (the
    // waits below read it as well)
    if ((st.calls++ & 7u) == 0 && failed(p.ws)) return false;
    // unfused baseline: phase 1 the head (ZPAD, GRADIN, RBWD, RDX), 2 DH,
    // 3 DWD, 4 DGU, 5 DWGU, 6 DWR, 7 PUSH + FOLD; 0 = everything in one launch
    const int ph = p.phase;
    const bool combine = ph == 0 || ph == 7;
    if (ph == 7) st.main_done = true;
    // 1) a ready PUSH (polled on every fourth call while rail entries remain:
    //    each poll is a round trip to L2, and the short weight-gradient
    //    tiles would otherwise wait on it)
    if (combine && (st.main_done || (st.polls++ & 3u) == 0)) {
        int32_t code;
        if (queue_try_take(&qc[1], &qc[0], p.push_items + q * b.push_cap, p.push_flags + q * b.push_cap, epoch, code,
                           p.ws)) {
            int e, rb, hc;
            push_decode(code, e, rb, hc);
            SchedEntry en;
            int real, r16;
            unit_rows(tb, e - q * g.Eq, rb, real, r16);
            // the unit's dx_e rows come by TMA, 64 rows (32 KB) per stage
            const int nst = (real + 63) / 64;
            fill_entry(en, K_PUSH, e, rb, hc, nst, code, bwd_trace_open(p, st, K_PUSH, code));
            en.x0 = tb.offp[e] + rb * BM;
            en.x1 = real;
            en.x2 = tb.offl[e - q * g.Eq] + rb * BM;  // logical receive row of the unit's first row
            if (!ring_push(sm, st.rs, en, p.ws)) return false;
            for (int s = 0; s < nst; ++s) {
                if (!bwd_wait_stage(p, sm, st.ps, code)) return false;
                uint64_t *bar = &sm.full[st.ps.stage];
                mbar_arrive_expect_tx(bar, 64 * 512);
                tma_load_2d(sm.stages + st.ps.stage * STAGE_BYTES, &p.tmDxbP, bar, hc * 256, en.x0 + s * 64);
                st.ps.advance();
            }
            st.idle_t0 = 0;
            return true;
        }
        if (failed(p.ws)) return false;
    }
    // 2) the next entry of this rank's rail
    if (!st.main_done) {
        const int nh = b.n_head;
        const int RB = g.RB, K = g.K;
        // a phase of the unfused baseline counts from its own first ticket
        const uint32_t base = ph <= 1 ? 0u
                                      : static_cast<uint32_t>(nh + (ph == 6 ? bwd_expert_tickets(b, tb.us) : 0));
        const uint32_t t = base + atomicAdd(&p.ws->tickets[q], 1u);
        if (ph == 1 && t >= static_cast<uint32_t>(nh)) return false;  // the head is done
        if (ph >= 2 && ph <= 5 && t - static_cast<uint32_t>(nh) >= static_cast<uint32_t>(bwd_expert_tickets(b, tb.us)))
            return false;  // the expert tiles are done
        if (t == 0) {  // ZPAD
            SchedEntry en;
            fill_entry(en, KB_ZPAD, q, 0, 0, 0, t, bwd_trace_open(p, st, KB_ZPAD, t));
            ring_push(sm, st.rs, en, p.ws);
            st.idle_t0 = 0;
            return true;
        }
        if (t < static_cast<uint32_t>(1 + RB * K)) {  // GRADIN(b, k)
            const int i = static_cast<int>(t) - 1;
            const int bb = i / K, kk = i % K;
            const int64_t left = g.Tq - static_cast<int64_t>(bb) * BM;
            const int ntok = static_cast<int>(left < BM ? left : BM);
            // per stage 32 tokens x 256 columns of dout and of the slot
            // outputs (16 KB each), token groups outer
            const int nch = b.NHC, nst = (ntok + 31) / 32 * nch;
            SchedEntry en;
            fill_entry(en, KB_GRADIN, q, bb, kk, nst, t, bwd_trace_open(p, st, KB_GRADIN, t));
            if (!ring_push(sm, st.rs, en, p.ws)) return false;
            for (int s = 0; s < nst; ++s) {
                const int r0 = bb * BM + (s / nch) * 32, c0 = (s % nch) * 256;
                if (!bwd_wait_stage(p, sm, st.ps, t)) return false;
                uint8_t *sa = sm.stages + st.ps.stage * STAGE_BYTES;
                uint64_t *bar = &sm.full[st.ps.stage];
                mbar_arrive_expect_tx(bar, 2 * 32 * 512);
                tma_load_2d(sa, &p.tmDout[q], bar, c0, r0);
                tma_load_3d(sa + 32 * 512, &p.tmYslot, bar, c0, kk, static_cast<int32_t>(q * g.Tq + r0));
                st.ps.advance();
            }
            st.idle_t0 = 0;
            return true;
        }
        if (t < static_cast<uint32_t>(1 + RB * K + RB)) {  // RBWD(b)
            const int bb = static_cast<int>(t) - 1 - RB * K;
            if (!wait_flag_eq(p.ws, &p.dgate_cnt[q * RB + bb], static_cast<uint32_t>(K), p.wait_limit_ns, t))
                return false;
            // the block's fp32 logits come by TMA, rbwd_tps tokens per stage
            const int64_t left = g.Tq - static_cast<int64_t>(bb) * BM;
            const int ntok = static_cast<int>(left < BM ? left : BM);
            const int nst = (ntok + b.rbwd_tps - 1) / b.rbwd_tps;
            SchedEntry en;
            fill_entry(en, KB_RBWD, q, bb, 0, nst, t, bwd_trace_open(p, st, KB_RBWD, t));
            if (!ring_push(sm, st.rs, en, p.ws)) return false;
            const int32_t tok0 = static_cast<int32_t>(q * g.Tq + static_cast<int64_t>(bb) * BM);
            for (int s2 = 0; s2 < nst; ++s2) {
                if (!bwd_wait_stage(p, sm, st.ps, t)) return false;
                uint64_t *bar = &sm.full[st.ps.stage];
                mbar_arrive_expect_tx(bar, static_cast<uint32_t>(b.rbwd_tps * g.E * 4));
                tma_load_2d(sm.stages + st.ps.stage * STAGE_BYTES, &p.tmLogits, bar, 0, tok0 + s2 * b.rbwd_tps);
                st.ps.advance();
            }
            st.idle_t0 = 0;
            return true;
        }
        if (t < static_cast<uint32_t>(nh)) {  // RDX(b, hc)
            const int i = static_cast<int>(t) - 1 - RB * K - RB;
            const int bb = i / b.NHC, hc = i % b.NHC;
            if (!wait_flag_eq(p.ws, &p.rbwd_flag[q * RB + bb], 1u, p.wait_limit_ns, t)) return false;
            SchedEntry en;
            fill_entry(en, KB_RDX, q, bb, hc, b.nkb_e, t, bwd_trace_open(p, st, KB_RDX, t));
            if (!ring_push(sm, st.rs, en, p.ws)) return false;
            const int32_t tok0 = static_cast<int32_t>(q * g.Tq + static_cast<int64_t>(bb) * BM);
            for (int kb = 0; kb < b.nkb_e; ++kb) {
                if (!bwd_wait_stage(p, sm, st.ps, t)) return false;
                uint8_t *sa = sm.stages + st.ps.stage * STAGE_BYTES;
                uint64_t *bar = &sm.full[st.ps.stage];
                mbar_arrive_expect_tx(bar, STAGE_BYTES);
                tma_load_2d(sa, &p.tmDlA, bar, kb * BK, tok0);
                tma_load_2d(sa + A_STAGE_BYTES, &p.tmWrT, bar, kb * BK, hc * 256);
                st.ps.advance();
            }
            st.idle_t0 = 0;
            return true;
        }
        const int ntile = bwd_expert_tickets(b, tb.us);
        const int tt = static_cast<int>(t) - nh;
        if (tt >= ntile) {  // DWR tiles of this rank, then done
            const int hb = q + (tt - ntile) * g.P;
            if (hb >= b.NWH) {
                st.main_done = true;
                if (ph != 0) return false;
            } else {
                if (!wait_flag_eq(p.ws, p.rbwd_done, static_cast<uint32_t>(g.NB), p.wait_limit_ns, t)) return false;
                SchedEntry en;
                const int nkb = static_cast<int>(g.T / BK);
                fill_entry(en, KB_DWR, hb, 0, 0, nkb, t, bwd_trace_open(p, st, KB_DWR, t));
                en.nmma = g.E;
                if (!ring_push(sm, st.rs, en, p.ws)) return false;
                const uint32_t bytes = A_STAGE_BYTES + (g.E / 64) * 8192;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!bwd_wait_stage(p, sm, st.ps, t)) return false;
                    uint8_t *sa = sm.stages + st.ps.stage * STAGE_BYTES;
                    uint8_t *sb = sa + A_STAGE_BYTES;
                    uint64_t *bar = &sm.full[st.ps.stage];
                    mbar_arrive_expect_tx(bar, bytes);
                    const int64_t t0 = static_cast<int64_t>(kb) * BK;
                    const int qs = static_cast<int>(t0 / g.Tq);
                    const int32_t tl = static_cast<int32_t>(t0 - static_cast<int64_t>(qs) * g.Tq);
                    tma_load_2d(sa, &p.tmXs[qs], bar, hb * 128, tl);
                    tma_load_2d(sa + 8192, &p.tmXs[qs], bar, hb * 128 + 64, tl);
                    for (int j = 0; j < g.E / 64; ++j)
                        tma_load_2d(sb + j * 8192, &p.tmDlB, bar, j * 64, static_cast<int32_t>(t0));
                    st.ps.advance();
                }
                st.idle_t0 = 0;
                return true;
            }
        } else {
            int kind = 0, le = 0, x = 0, y = 0, cnt = 1;
            bwd_decode_tile(b, tb.us, tt, kind, le, x, y, cnt, st.hint);
            if (kind == 0) {
                set_error(p.ws, KOSMOS_ERR_DEVICE, -30);
                return false;
            }
            if (ph >= 2 && ph <= 5 && kind != (ph == 2 ? KB_DH : ph == 3 ? KB_DWD : ph == 4 ? KB_DGU : KB_DWGU))
                return true;  // another phase's tile
            const int e = q * g.Eq + le;
            const int c = tb.cnt[le];
            const int c16 = (c + 15) / 16 * 16;
            const int units = tb.us[le + 1] - tb.us[le];
            SchedEntry en;
            if (kind == KB_DH || kind == KB_DGU) {
                const int rb = y, col = x;
                int real, r16;
                unit_rows(tb, le, rb, real, r16);
                const int ci = e * g.MAXRB + rb;
                if (kind == KB_DH) {
                    if (!wait_flag_eq(p.ws, &p.dy_cnt[ci], static_cast<uint32_t>(r16), p.wait_limit_ns, t))
                        return false;
                } else {
                    if (!wait_flag_eq(p.ws, &p.dh_cnt[ci], static_cast<uint32_t>(b.NIC), p.wait_limit_ns, t))
                        return false;
                }
                const int nst = kind == KB_DH ? b.nkb_h : b.nkb_gu;
                fill_entry(en, kind, e, rb, col, nst, t, bwd_trace_open(p, st, kind, t));
                en.d = le;
                en.x0 = tb.offp[e] + rb * BM;   // padded row of the unit
                en.x1 = real | (r16 << 16);
                en.x2 = tb.offl[le] + rb * BM;   // forward (unpadded) row of the unit
                if (!ring_push(sm, st.rs, en, p.ws)) return false;
                for (int kb = 0; kb < nst; ++kb) {
                    if (!bwd_wait_stage(p, sm, st.ps, t)) return false;
                    uint8_t *sa = sm.stages + st.ps.stage * STAGE_BYTES;
                    uint8_t *sb = sa + A_STAGE_BYTES;
                    uint64_t *bar = &sm.full[st.ps.stage];
                    mbar_arrive_expect_tx(bar, STAGE_BYTES);
                    if (kind == KB_DH) {
                        tma_load_2d(sa, &p.tmDyA, bar, kb * BK, en.x0);
                        tma_load_3d(sb, &p.tmWdT[q], bar, kb * BK, col * 256, le);
                    } else {
                        const int half = b.nkb_gu / 2;
                        const int kk = kb < half ? kb : kb - half;
                        tma_load_2d(sa, kb < half ? &p.tmDgA : &p.tmDuA, bar, kk * BK, en.x0);
                        tma_load_3d(sb, kb < half ? &p.tmWgT[q] : &p.tmWuT[q], bar, kk * BK, col * 256, le);
                    }
                    st.ps.advance();
                }
                for (int s = 0; kind == KB_DH && s < DH_EPI_STAGES; ++s) {  // the epilogue's g / u chunks
                    if (!bwd_wait_stage(p, sm, st.ps, t)) return false;
                    uint8_t *sa = sm.stages + st.ps.stage * STAGE_BYTES;
                    uint64_t *bar = &sm.full[st.ps.stage];
                    const int c0 = s * 3, nch = 8 - c0 < 3 ? 8 - c0 : 3;
                    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nch * DH_CH_BYTES));
                    for (int j = 0; j < nch; ++j) {
                        const int32_t xc = col * 256 + (c0 + j) * 32;
                        tma_load_2d(sa + j * DH_CH_BYTES, &p.tmGs, bar, xc, en.x2);
                        tma_load_2d(sa + j * DH_CH_BYTES + DH_CH_BYTES / 2, &p.tmUs, bar, xc, en.x2);
                    }
                    st.ps.advance();
                }
            } else {
                // weight gradients over the expert's rows: the K loop covers
                // the 16-row-padded rows; the last stage issues only its
                // K steps of 16
                int &ready = kind == KB_DWD ? st.ready_dwd : st.ready_dwgu;
                if (ready != e) {
                    for (int u = 0; u < units; ++u) {
                        const int ci = e * g.MAXRB + u;
                        if (kind == KB_DWD) {
                            int real, r16;
                            unit_rows(tb, le, u, real, r16);
                            if (!wait_flag_eq(p.ws, &p.dy_cnt[ci], static_cast<uint32_t>(r16), p.wait_limit_ns, t))
                                return false;
                        } else {
                            if (!wait_flag_eq(p.ws, &p.dh_cnt[ci], static_cast<uint32_t>(b.NIC), p.wait_limit_ns, t))
                                return false;
                        }
                    }
                    ready = e;
                }
                const int nst = (c16 + BK - 1) / BK;
                const int last = (c16 - (nst - 1) * BK) / 16;  // 1..4 when nst > 0
                const int32_t rl = tb.offl[le], rp = tb.offp[e];
                const int ny = kind == KB_DWD ? b.NHC : b.NWI;  // tiles of the group: y fastest
                for (int gi = 0; gi < cnt; ++gi) {
                    const int xi = x + (y + gi) / ny, yi = (y + gi) % ny;
                    fill_entry(en, kind, e, xi, yi, nst, t, bwd_trace_open(p, st, kind, t));
                    en.d = le;
                    en.x1 = last & 3;
                    if (!ring_push(sm, st.rs, en, p.ws)) return false;
                    for (int kb = 0; kb < nst; ++kb) {
                        if (!bwd_wait_stage(p, sm, st.ps, t)) return false;
                        uint8_t *sa = sm.stages + st.ps.stage * STAGE_BYTES;
                        uint8_t *sb = sa + A_STAGE_BYTES;
                        uint64_t *bar = &sm.full[st.ps.stage];
                        mbar_arrive_expect_tx(bar, STAGE_BYTES);
                        if (kind == KB_DWD) {  // A = h^T (I block xi), B = dy (256 columns yi)
                            tma_load_2d(sa, &p.tmH, bar, xi * 128, rl + kb * BK);
                            tma_load_2d(sa + 8192, &p.tmH, bar, xi * 128 + 64, rl + kb * BK);
                            for (int j = 0; j < 4; ++j)
                                tma_load_2d(sb + j * 8192, &p.tmDyB, bar, yi * 256 + j * 64, rp + kb * BK);
                        } else {  // A = x^T (hidden block xi), B = [dg | du] (inter block yi)
                            tma_load_2d(sa, &p.tmX, bar, xi * 128, rl + kb * BK);
                            tma_load_2d(sa + 8192, &p.tmX, bar, xi * 128 + 64, rl + kb * BK);
                            tma_load_2d(sb, &p.tmDgB, bar, yi * 128, rp + kb * BK);
                            tma_load_2d(sb + 8192, &p.tmDgB, bar, yi * 128 + 64, rp + kb * BK);
                            tma_load_2d(sb + 16384, &p.tmDuB, bar, yi * 128, rp + kb * BK);
                            tma_load_2d(sb + 24576, &p.tmDuB, bar, yi * 128 + 64, rp + kb * BK);
                        }
                        st.ps.advance();
                    }
                }
            }

            st.idle_t0 = 0;
            return true;
        }
    }
    // 3) a ready FOLD of this rank's tokens
    if (combine) {
        int32_t code;
        if (queue_try_take(&qc[3], &qc[2], p.fold_items + q * b.fold_cap, p.fold_flags + q * b.fold_cap, epoch, code,
                           p.ws)) {
            const int gb = code & 0xFFFF, hc = (code >> 16) & 0xFFFF;
            const int qs = gb / g.RB, bq = gb % g.RB;
            const int64_t left = g.Tq - static_cast<int64_t>(bq) * BM;
            const int ntok = static_cast<int>(left < BM ? left : BM);
            const int nst = (ntok + b.fold_tps - 1) / b.fold_tps;
            const int64_t row0 = (static_cast<int64_t>(qs) * g.Tq + static_cast<int64_t>(bq) * BM) * g.K;
            SchedEntry en;
            fill_entry(en, K_FOLD, gb, 0, hc, nst, code, bwd_trace_open(p, st, K_FOLD, code));
            if (!ring_push(sm, st.rs, en, p.ws)) return false;
            const uint32_t slot_bytes = static_cast<uint32_t>(256 * 2 * b.fold_tps * g.K);
            const uint32_t bytes = slot_bytes + static_cast<uint32_t>(256 * 4 * b.fold_tps);
            for (int s = 0; s < nst; ++s) {
                if (!bwd_wait_stage(p, sm, st.ps, code)) return false;
                uint64_t *bar = &sm.full[st.ps.stage];
                uint8_t *sa = sm.stages + st.ps.stage * STAGE_BYTES;
                mbar_arrive_expect_tx(bar, bytes);
                tma_load_2d(sa, &p.tmDslot, bar, hc * 256,
                            static_cast<int32_t>(row0 + static_cast<int64_t>(s) * b.fold_tps * g.K));
                tma_load_2d(sa + slot_bytes, &p.tmDxr, bar, hc * 256,
                            static_cast<int32_t>(row0 / g.K + static_cast<int64_t>(s) * b.fold_tps));
                st.ps.advance();
            }
            st.idle_t0 = 0;
            return true;
        }
        if (failed(p.ws)) return false;
    }
    // 4) finished when the rail and both queues of this rank are drained
    if (st.main_done) {
        const uint32_t push_total = static_cast<uint32_t>(tb.us[g.Eq]) * b.NHC;
        const uint32_t fold_total = static_cast<uint32_t>(b.fold_cap);
        if (ld_relaxed_gpu(&qc[1]) >= push_total && ld_relaxed_gpu(&qc[3]) >= fold_total) return false;
    }
    const uint64_t now = globaltimer();
    if (st.idle_t0 == 0) {
        st.idle_t0 = now;
    } else if (now - st.idle_t0 > p.wait_limit_ns) {
        set_error(p.ws, KOSMOS_ERR_TIMEOUT, -31);
        return false;
    }
    return true;
}

__device__ __forceinline__ void bwd_producer(const BwdParams &p, const Smem &sm, const BwdTables &tb,
                                             uint32_t epoch) {
    BwdProdState st;
    while (bwd_decide(p, sm, st, tb, epoch)) {
    }
    SchedEntry done;
    fill_entry(done, K_DONE, 0, 0, 0, 0, -1, -1);
    ring_push(sm, st.rs, done, p.ws);
}

// ---------------------------------------------------------------- MMA warp
// One accumulator pair as in the forward (two alternating 128 x 256 fp32
// accumulators).  Per entry: operand majors and the K steps of its last stage
// from x2, N from nmma (0 = 256).
__device__ __forceinline__ void bwd_mma_loop(const BwdParams &p, const Smem &sm, uint32_t tmem_base) {
    PipeState ps;
    RingState rs;
    uint32_t acc = 0, acc_phase = 0;
    while (true) {
        if (!mbar_wait(&sm.sfull[rs.idx], rs.phase, PIPE_LIMIT_NS)) {
            set_error(p.ws, KOSMOS_ERR_DEVICE, -3);
            break;
        }
        const SchedEntry e = sm.sched[rs.idx];
        mbar_arrive(&sm.sempty[rs.idx]);
        rs.advance();
        if (e.kind == K_DONE) break;
        if (!bwd_is_mma(e.kind)) {
            ps.advance(e.nstage);
            continue;
        }
        const bool mn = bwd_is_wgrad(e.kind);
        const bool amn = mn, bmn = mn;
        const int last = (e.kind == KB_DWD || e.kind == KB_DWGU) ? (e.x1 & 3) : 0;
        const int N = (e.nmma > 0 && e.nmma < BN) ? e.nmma : BN;
        const uint32_t idesc = idesc_bf16_f32(BM, N, amn, bmn);
        if (!mbar_wait(&sm.tempty[acc], acc_phase ^ 1u, PIPE_LIMIT_NS)) {
            set_error(p.ws, KOSMOS_ERR_DEVICE, -4);
            break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < e.nstage; ++kb) {
            if (!mbar_wait(&sm.full[ps.stage], ps.phase, PIPE_LIMIT_NS)) {
                set_error(p.ws, KOSMOS_ERR_DEVICE, -5);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sm.stages + ps.stage * STAGE_BYTES);
            const uint32_t b_addr = a_addr + A_STAGE_BYTES;
            const int nk = (kb == e.nstage - 1 && last != 0) ? last : BK / UMMA_K;
            for (int k = 0; k < nk; ++k) {
                const uint64_t ad = amn ? sdesc_sw128(a_addr + k * (UMMA_K * 128), 8192, 1024)
                                        : sdesc_sw128(a_addr + k * (UMMA_K * 2), 16, 1024);
                const uint64_t bd = bmn ? sdesc_sw128(b_addr + k * (UMMA_K * 128), 8192, 1024)
                                        : sdesc_sw128(b_addr + k * (UMMA_K * 2), 16, 1024);
                mma_bf16_ss(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            }
            mma_commit(&sm.empty[ps.stage]);
            ps.advance();
        }
        if (!ok) break;
        if (e.kind == KB_DH) ps.advance(DH_EPI_STAGES);  // consumed by the epilogue
        if (e.nstage == 0) {
            mbar_arrive(&sm.tfull[acc]);  // nothing to multiply: the epilogue writes zeros
        } else {
            mma_commit(&sm.tfull[acc]);
        }
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
}

// ---------------------------------------------------------------- epilogue helpers
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// 32 fp32 accumulator columns of this thread's row (zeros when `zero`).
__device__ __forceinline__ void acc_chunk(uint32_t taddr, bool zero, float (&v)[32]) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = zero ? 0.f : __uint_as_float(r[j]);
}

// ZPAD: zero the padding rows [cnt, ceil16(cnt)) of each of rank q's experts
// in dy, then count them as arrived rows of the expert's last unit.
__device__ __noinline__ void bwd_zpad(const BwdParams &p, const BwdTables &tb, int q, int et) {
    const MoeGeom &g = p.b.f;
    const int H8 = static_cast<int>(g.H / 8);  // 16-byte words per row
    for (int le = 0; le < g.Eq; ++le) {
        const int c = tb.cnt[le];
        const int pad = (c + 15) / 16 * 16 - c;
        const int e = q * g.Eq + le;
        for (int i = et; i < pad * H8; i += NUM_EPI_THREADS) {
            const int64_t row = tb.offp[e] + c + i / H8;
            reinterpret_cast<uint4 *>(p.dy + row * g.H)[i % H8] = make_uint4(0, 0, 0, 0);
        }
    }
    fence_proxy_async_global();  // generic stores, read by the tiles' tensor copies
    __threadfence();
    named_bar_sync(1, NUM_EPI_THREADS);
    if (et < g.Eq) {
        const int c = tb.cnt[et];
        const int pad = (c + 15) / 16 * 16 - c;
        if (pad > 0) red_release_add_gpu(&p.dy_cnt[(q * g.Eq + et) * g.MAXRB + (c - 1) / BM], static_cast<uint32_t>(pad));
    }
}

// GRADIN(b, k): the combine's backward for slot k of the block's tokens,
// dgate = <dout, y_slot> in fp32 and dy = bf16(gate * dout) to the token's
// expert-ordered row.  dout and the slot outputs arrive by TMA, 32 tokens x
// 256 columns per stage; thread et takes token et / 4 of the group and
// columns (et % 4) * 64 .. + 63, writes its dy values over its dout in the
// stage, and the token's dy segment leaves with one 512-byte bulk copy.  The
// 16-byte pieces are visited in a lane-rotated order so that the lanes of a
// quarter-warp (two tokens, four segments each) hit distinct banks.
__device__ __noinline__ bool bwd_gradin(const BwdParams &p, const Smem &sm, PipeState &ps, const BwdTables &tb,
                                        const SchedEntry &e, int lane, int et) {
    const MoeGeom &g = p.b.f;
    const int q = e.a, bb = e.b, k = e.c;
    const int gblk = q * g.RB + bb;
    const int64_t left = g.Tq - static_cast<int64_t>(bb) * BM;
    const int ntok = static_cast<int>(left < BM ? left : BM);
    const int nch = p.b.NHC;
    const int seg = et & 3, tl = et >> 2;
    float dot = 0.f, gk = 0.f;
    int64_t t = 0, prow = 0;
    bool real = false, sent = false;
    for (int s = 0; s < e.nstage; ++s) {
        const int cc = s % nch;
        if (cc == 0) {  // a new group of 32 tokens
            const int r = (s / nch) * 32 + tl;
            real = r < ntok;
            dot = 0.f;
            if (real) {
                t = static_cast<int64_t>(q) * g.Tq + static_cast<int64_t>(bb) * BM + r;
                const int ex = __ldg(&p.topk_idx[t * g.K + k]);
                gk = __ldg(&p.topk_gate[t * g.K + k]);
                const int pos = ldcg_i32(&p.base[gblk * g.E + ex]) + ldcg_i32(&p.rank_in_blk[t * g.K + k]);
                prow = static_cast<int64_t>(pos) - __ldg(&p.offl[ex]) + tb.offp[ex];
            }
        }
        // a thread whose wait runs out skips the stage's work and still takes
        // the stage's barrier, which makes the decision to stop for all
        const bool ok = mbar_wait(&sm.full[ps.stage], ps.phase, PIPE_LIMIT_NS);
        if (!ok) set_error(p.ws, KOSMOS_ERR_DEVICE, -34);
        uint8_t *drow = sm.stages + ps.stage * STAGE_BYTES + tl * 512;
        const uint8_t *yrow = drow + 32 * 512;
        if (ok && real) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int off = seg * 128 + ((i + lane) & 7) * 16;
                const uint4 dv = *reinterpret_cast<const uint4 *>(drow + off);
                const uint4 yv = *reinterpret_cast<const uint4 *>(yrow + off);
                const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w}, yw[4] = {yv.x, yv.y, yv.z, yv.w};
                uint32_t ow[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    dot = __fmaf_rn(bf_lo(dw[j]), bf_lo(yw[j]), dot);
                    dot = __fmaf_rn(bf_hi(dw[j]), bf_hi(yw[j]), dot);
                    ow[j] = pack_bf16x2(gk * bf_lo(dw[j]), gk * bf_hi(dw[j]));
                }
                *reinterpret_cast<uint4 *>(drow + off) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
            }
        }
        fence_proxy_async_smem();  // the dy values in the stage, for the bulk copy
        __syncwarp();              // the token's four threads are lanes of one warp
        if (ok && seg == 0 && real) {
            bulk_s2g(p.dy + prow * g.H + cc * 256, drow, 512);
            bulk_commit();
            bulk_wait_read<0>();
            sent = true;
        }
        if (!named_bar_and(1, NUM_EPI_THREADS, ok)) {
            if (sent) bulk_wait<0>();
            return false;
        }
        if (et == 0) mbar_arrive(&sm.empty[ps.stage]);
        ps.advance();
        if (cc == nch - 1) {  // the token's dot product: its four threads' parts
            dot += __shfl_xor_sync(0xFFFFFFFFu, dot, 1);
            dot += __shfl_xor_sync(0xFFFFFFFFu, dot, 2);
            if (seg == 0 && real) p.dgate[t * g.K + k] = dot;
        }
    }
    if (sent) {
        bulk_wait<0>();  // this thread's dy segments have landed
        fence_proxy_async_global();
    }
    __threadfence();
    named_bar_sync(1, NUM_EPI_THREADS);
    // one arrival per row on its unit; then the block's slot-k count.  The
    // thread that counts token et's row is not the one that copied it: a
    // release add carries the copier's writes (ordered before the barrier)
    // to the tile that acquires the count.
    if (et < ntok) {
        const int64_t tt = static_cast<int64_t>(q) * g.Tq + static_cast<int64_t>(bb) * BM + et;
        const int ex = __ldg(&p.topk_idx[tt * g.K + k]);
        const int pos = ldcg_i32(&p.base[gblk * g.E + ex]) + ldcg_i32(&p.rank_in_blk[tt * g.K + k]);
        const int rb = (pos - __ldg(&p.offl[ex])) / BM;
        red_release_add_gpu(&p.dy_cnt[ex * g.MAXRB + rb], 1u);
    }
    named_bar_sync(1, NUM_EPI_THREADS);
    if (et == 0) red_release_add_gpu(&p.dgate_cnt[gblk], 1u);
    return true;
}

// RBWD(b): one token per thread.  p = softmax(l) (fp32, the forward's
// logits), S = sum over the top-K of p; dp_j = (dgate_k - sum_k dgate_k
// gate_k) / S for j = e_k; dl = p * (dp - <p, dp>), written as bf16.
__device__ __noinline__ bool bwd_rbwd(const BwdParams &p, const Smem &sm, PipeState &ps, const SchedEntry &e, int et) {
    const MoeGeom &g = p.b.f;
    const int q = e.a, bb = e.b;
    const int64_t left = g.Tq - static_cast<int64_t>(bb) * BM;
    const int ntok = static_cast<int>(left < BM ? left : BM);
    const int tps = p.b.rbwd_tps;
    // the block's logits arrive by TMA, tps tokens per stage; all of them are
    // held until the block is done
    PipeState s0 = ps;
    bool ok = true;
    for (int s2 = 0; s2 < e.nstage; ++s2) {
        if (ok && !mbar_wait(&sm.full[ps.stage], ps.phase, PIPE_LIMIT_NS)) {
            set_error(p.ws, KOSMOS_ERR_DEVICE, -35);
            ok = false;
        }
        ps.advance();
    }
    if (!named_bar_and(1, NUM_EPI_THREADS, ok)) return false;  // one decision for all threads
    if (et < ntok) {
        const int64_t t = static_cast<int64_t>(q) * g.Tq + static_cast<int64_t>(bb) * BM + et;
        PipeState sp = s0;
        sp.advance(et / tps);
        const float *l = reinterpret_cast<const float *>(sm.stages + sp.stage * STAGE_BYTES) +
                         static_cast<int64_t>(et % tps) * g.E;
        const float4 *l4 = reinterpret_cast<const float4 *>(l);
        float mx = -INFINITY;
#pragma unroll 4
        for (int i = 0; i < g.E / 4; ++i) {
            const float4 v = l4[i];
            mx = fmaxf(fmaxf(fmaxf(fmaxf(mx, v.x), v.y), v.z), v.w);
        }
        float z = 0.f;  // ascending expert order, as the forward's softmax
#pragma unroll 4
        for (int i = 0; i < g.E / 4; ++i) {
            const float4 v = l4[i];
            z += expf(v.x - mx);
            z += expf(v.y - mx);
            z += expf(v.z - mx);
            z += expf(v.w - mx);
        }
        int ix[MOE_MAXK];
        float pk[MOE_MAXK], dgk[MOE_MAXK];
        float S = 0.f;
#pragma unroll
        for (int k = 0; k < MOE_MAXK; ++k) {
            if (k < g.K) {
                ix[k] = __ldg(&p.topk_idx[t * g.K + k]);
                pk[k] = expf(l[ix[k]] - mx) / z;
                dgk[k] = __ldcg(&p.dgate[t * g.K + k]);
                S += pk[k];
            }
        }
        float sdg = 0.f;
#pragma unroll
        for (int k = 0; k < MOE_MAXK; ++k)
            if (k < g.K) sdg += dgk[k] * (pk[k] / S);
        float pdp = 0.f;
        float dpk[MOE_MAXK];
#pragma unroll
        for (int k = 0; k < MOE_MAXK; ++k) {
            if (k < g.K) {
                dpk[k] = (dgk[k] - sdg) / S;
                pdp += pk[k] * dpk[k];
            }
        }
        // dl_j = p_j (dp_j - <p, dp>) with dp_j = 0 off the top-K: every
        // expert is written as -p_j <p, dp> first, then the K selected ones
        // are rewritten with their dp
        __nv_bfloat16 *out = p.dl + t * g.E;
        const float inv_z = 1.0f / z;
#pragma unroll 1
        for (int c = 0; c < g.E / 32; ++c) {
            uint32_t o[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 v = l4[c * 8 + i];
                o[2 * i] = pack_bf16x2((expf(v.x - mx) * inv_z) * -pdp, (expf(v.y - mx) * inv_z) * -pdp);
                o[2 * i + 1] = pack_bf16x2((expf(v.z - mx) * inv_z) * -pdp, (expf(v.w - mx) * inv_z) * -pdp);
            }
            uint4 *o4 = reinterpret_cast<uint4 *>(out + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) o4[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
#pragma unroll
        for (int k = 0; k < MOE_MAXK; ++k)
            if (k < g.K) out[ix[k]] = __float2bfloat16_rn((expf(l[ix[k]] - mx) * inv_z) * (dpk[k] - pdp));
    }
    fence_proxy_async_global();  // dl is read by tensor copies (RDX, DWR)
    __threadfence();
    named_bar_sync(1, NUM_EPI_THREADS);
    if (et == 0) {
        PipeState sp = s0;
        for (int s2 = 0; s2 < e.nstage; ++s2) {  // the logits' stages go back to the producer
            mbar_arrive(&sm.empty[sp.stage]);
            sp.advance();
        }
        st_release_gpu(&p.rbwd_flag[q * g.RB + bb], 1u);
        red_release_add_gpu(p.rbwd_done, 1u);
    }
    return true;
}

// One arrival on the fold counter of (token block gb, column tile hc); the
// arrival that completes it (all K slot rows of the block's tokens plus the
// router part) queues the FOLD on the block's rank.
__device__ __forceinline__ void bwd_fold_arrive(const BwdParams &p, int gb, int hc, uint32_t cnt, uint32_t epoch) {
    const MoeGeom &g = p.b.f;
    const int bq = gb % g.RB;
    const int64_t left = g.Tq - static_cast<int64_t>(bq) * BM;
    const uint32_t target = static_cast<uint32_t>((left < BM ? left : BM) * g.K + 1);
    if (atom_add_acqrel_gpu(&p.fold_cnt[gb * p.b.NHC + hc], cnt) + cnt == target) {
        const int qs = gb / g.RB;
        queue_put(&p.qctl[4 * qs + 2], p.fold_items + qs * p.b.fold_cap, p.fold_flags + qs * p.b.fold_cap,
                  p.b.fold_cap, gb | (hc << 16), epoch, p.ws);
    }
}

// PUSH(e, rb, hc): the 256-column slice of each of the unit's rows of dx_e
// goes to its token slot.
__device__ __noinline__ bool bwd_push(const BwdParams &p, const Smem &sm, PipeState &ps, const SchedEntry &e, int et,
                                      int lane, uint32_t epoch) {
    const MoeGeom &g = p.b.f;
    const int hc = e.c;
    const int rows = e.x1, lrow0 = e.x2;
    const int32_t my_sl = (et < rows) ? ldcg_i32(&p.inv_pos[lrow0 + et]) : -1;  // this thread's row
    // the rows arrive by TMA, 64 to a stage; thread et sends row et with one
    // 512-byte bulk copy to its token slot
    for (int s = 0; s < e.nstage; ++s) {
        const bool ok = mbar_wait(&sm.full[ps.stage], ps.phase, PIPE_LIMIT_NS);
        if (!ok) set_error(p.ws, KOSMOS_ERR_DEVICE, -33);
        if (ok && (et >> 6) == s && my_sl >= 0) {
            bulk_s2g(p.dslot + static_cast<int64_t>(my_sl) * g.H + hc * 256,
                     sm.stages + ps.stage * STAGE_BYTES + (et & 63) * 512, 512);
            bulk_commit();
            bulk_wait_read<0>();
        }
        if (!named_bar_and(1, NUM_EPI_THREADS, ok)) {  // one decision for all threads
            bulk_wait<0>();
            return false;
        }
        if (et == 0) mbar_arrive(&sm.empty[ps.stage]);
        ps.advance();
    }
    if (my_sl >= 0) {
        bulk_wait<0>();  // the row has landed; order it before the release below
        fence_proxy_async_global();
    }
    __threadfence();
    __syncwarp();
    int gb = -1;
    if (my_sl >= 0) {
        const int64_t t = my_sl / g.K;
        const int qs = static_cast<int>(t / g.Tq);
        const int bq = static_cast<int>((t - static_cast<int64_t>(qs) * g.Tq) / BM);
        gb = qs * g.RB + bq;
    }
    const uint32_t grp = __match_any_sync(0xFFFFFFFFu, gb);
    if (gb >= 0 && (__ffs(grp) - 1) == lane) bwd_fold_arrive(p, gb, hc, __popc(grp), epoch);
    __syncwarp();
    return true;
}

// FOLD(gb, hc): dx[t] = sum_k slot[t][k] (fp32, k order) + dx_router[t], one
// rounding to bf16.  Slot rows and the tokens' router rows arrive through the
// stage ring, fold_tps tokens per stage; thread et takes token et / 16 (and
// every 8th after it) and 16 of the 256 columns.
__device__ __noinline__ bool bwd_fold(const BwdParams &p, const Smem &sm, PipeState &ps, const SchedEntry &e, int et) {
    const MoeGeom &g = p.b.f;
    const int gb = e.a, hc = e.c;
    const int q = gb / g.RB, bq = gb % g.RB;
    const int K = g.K;
    const int tps = p.b.fold_tps;
    const int64_t left = g.Tq - static_cast<int64_t>(bq) * BM;
    const int ntok = static_cast<int>(left < BM ? left : BM);
    const int c0 = (et & 15) * 16;
    for (int s = 0; s < e.nstage; ++s) {
        const bool ok = mbar_wait(&sm.full[ps.stage], ps.phase, PIPE_LIMIT_NS);
        if (!ok) set_error(p.ws, KOSMOS_ERR_DEVICE, -32);
        const uint8_t *buf = sm.stages + ps.stage * STAGE_BYTES;
        for (int u = et >> 4; ok && u < tps; u += NUM_EPI_THREADS / 16) {
            const int r = s * tps + u;
            if (r >= ntok) break;
            float acc[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = 0.f;
            for (int k = 0; k < K; ++k) {
                const uint4 *src = reinterpret_cast<const uint4 *>(buf + ((u * K + k) * 256 + c0) * 2);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 v = src[h];
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[h * 8 + 2 * j] = __fadd_rn(acc[h * 8 + 2 * j], bf_lo(w[j]));
                        acc[h * 8 + 2 * j + 1] = __fadd_rn(acc[h * 8 + 2 * j + 1], bf_hi(w[j]));
                    }
                }
            }
            // the router part came with the stage (fp32 rows after the slot rows)
            const float4 *xr = reinterpret_cast<const float4 *>(buf + 512 * tps * K + (u * 256 + c0) * 4);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 a = xr[j];
                acc[4 * j + 0] = __fadd_rn(acc[4 * j + 0], a.x);
                acc[4 * j + 1] = __fadd_rn(acc[4 * j + 1], a.y);
                acc[4 * j + 2] = __fadd_rn(acc[4 * j + 2], a.z);
                acc[4 * j + 3] = __fadd_rn(acc[4 * j + 3], a.w);
            }
            uint4 o[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                o[h].x = pack_bf16x2(acc[h * 8 + 0], acc[h * 8 + 1]);
                o[h].y = pack_bf16x2(acc[h * 8 + 2], acc[h * 8 + 3]);
                o[h].z = pack_bf16x2(acc[h * 8 + 4], acc[h * 8 + 5]);
                o[h].w = pack_bf16x2(acc[h * 8 + 6], acc[h * 8 + 7]);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(p.dx[q] + (static_cast<int64_t>(bq) * BM + r) * g.H + hc * 256 + c0);
            dst[0] = o[0];
            dst[1] = o[1];
        }
        if (!named_bar_and(1, NUM_EPI_THREADS, ok)) return false;  // one decision for all threads
        if (et == 0) mbar_arrive(&sm.empty[ps.stage]);
        ps.advance();
    }
    return true;
}

// fp32 sigmoid through the fast exponential and the approximate division (a
// few ulp; the results are rounded to bf16)
__device__ __forceinline__ float sigmoid_f(float a) { return __fdividef(1.0f, 1.0f + __expf(-a)); }

// 32 fp32 accumulator columns of this thread's row as bf16 into pieces
// p0 .. p0 + 3 (16 bytes each) of its 128-byte row of a staging box in the
// 128-byte swizzled layout of the store's tensor map (piece p of row r at
// p ^ (r & 7)): the 32 lanes' row writes spread over all banks.
__device__ __forceinline__ void bwd_stage_cols(uint8_t *box, int lane, const uint32_t (&r)[32], int p0) {
    uint4 *row = reinterpret_cast<uint4 *>(box + lane * 128);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
        const uint32_t *w = r + q4 * 8;
        row[(p0 + q4) ^ (lane & 7)] =
            make_uint4(pack_bf16x2(__uint_as_float(w[0]), __uint_as_float(w[1])),
                       pack_bf16x2(__uint_as_float(w[2]), __uint_as_float(w[3])),
                       pack_bf16x2(__uint_as_float(w[4]), __uint_as_float(w[5])),
                       pack_bf16x2(__uint_as_float(w[6]), __uint_as_float(w[7])));
    }
}

__device__ __forceinline__ void bwd_epilogue(const BwdParams &p, const Smem &sm, const BwdTables &tb,
                                             uint32_t tmem_base, uint8_t *stg, int warp, int lane, uint32_t epoch) {
    const BwdGeom &b = p.b;
    const MoeGeom &g = b.f;
    const int grp = warp & 3;
    const int row = grp * 32 + lane;
    const int ew = warp - 2;
    const int et = ew * 32 + lane;
    RingState rs;
    PipeState ps;
    uint32_t acc = 0, acc_phase = 0;
    while (true) {
        if (!mbar_wait(&sm.sfull[rs.idx], rs.phase, PIPE_LIMIT_NS)) {
            set_error(p.ws, KOSMOS_ERR_DEVICE, -6);
            break;
        }
        const SchedEntry e = sm.sched[rs.idx];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.sempty[rs.idx]);
        rs.advance();
        if (e.kind == K_DONE) break;
        if (bwd_is_mma(e.kind)) {
            ps.advance(e.nstage);
            if (e.kind == KB_DH && row < (e.x1 & 0xFFFF)) {
                // the SwiGLU inputs of this thread's row come from HBM: start
                // them towards L2 while the tile's K loop (the whole of H) runs
                const int64_t off = (static_cast<int64_t>(e.x2) + row) * g.I + static_cast<int64_t>(e.c) * 256;
                bulk_prefetch_l2(p.gsave + off, 512);
                bulk_prefetch_l2(p.usave + off, 512);
            }
            if (!mbar_wait(&sm.tfull[acc], acc_phase, PIPE_LIMIT_NS)) {
                set_error(p.ws, KOSMOS_ERR_DEVICE, -7);
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(grp * 32) << 16) + acc * BN;
            const bool zero = e.nstage == 0;
            if (e.kind == KB_DH) {
                const int real = e.x1 & 0xFFFF, r16 = e.x1 >> 16;
                const bool is_real = row < real;
                const int sw = (row >> 1) & 3;  // 64-byte swizzle of this row's 16-byte pieces
                bool ok = true;
#pragma unroll 1
                for (int ch = 0; ch < 8; ++ch) {
                    const int j = ch % 3;
                    // a thread whose wait runs out computes zeros up to the
                    // stage's barrier, which makes the decision to stop for all
                    if (j == 0 && ok && !mbar_wait(&sm.full[ps.stage], ps.phase, PIPE_LIMIT_NS)) {
                        set_error(p.ws, KOSMOS_ERR_DEVICE, -8);
                        ok = false;
                    }
                    const uint8_t *cs = sm.stages + ps.stage * STAGE_BYTES + j * DH_CH_BYTES + row * 64;
                    float dh[32];
                    acc_chunk(taddr + ch * 32, false, dh);
                    uint32_t dgp[16], dup[16];  // bf16 pairs of dg, du
                    if (ok && is_real) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const uint4 gv = *reinterpret_cast<const uint4 *>(cs + (q4 ^ sw) * 16);
                            const uint4 uv = *reinterpret_cast<const uint4 *>(cs + DH_CH_BYTES / 2 + (q4 ^ sw) * 16);
                            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
                            for (int w = 0; w < 4; ++w) {
                                float dgo[2], duo[2];
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    const float gg = h ? bf_hi(gw[w]) : bf_lo(gw[w]);
                                    const float uu = h ? bf_hi(uw[w]) : bf_lo(uw[w]);
                                    const float sg = sigmoid_f(gg);
                                    const float d = dh[q4 * 8 + 2 * w + h];
                                    dgo[h] = d * uu * (sg * (1.0f + gg * (1.0f - sg)));
                                    duo[h] = d * (gg * sg);
                                }
                                dgp[q4 * 4 + w] = pack_bf16x2(dgo[0], dgo[1]);
                                dup[q4 * 4 + w] = pack_bf16x2(duo[0], duo[1]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int w = 0; w < 16; ++w) { dgp[w] = 0u; dup[w] = 0u; }
                    }
                    if (j == 2 || ch == 7) {  // every epilogue warp has read its rows of the stage
                        if (!named_bar_and(1, NUM_EPI_THREADS, ok)) {
                            ok = false;
                            break;
                        }
                        if (et == 0) mbar_arrive(&sm.empty[ps.stage]);
                        ps.advance();
                    }
                    // dg and du leave through the warp's staging buffer as 16-row
                    // boxes (64-byte swizzle: piece c of row r at c ^ ((r >> 1) & 3));
                    // boxes past the unit's 16-row-padded end are not stored,
                    // those rows belong to the next expert
                    if (lane == 0) bulk_wait_read<0>();
                    __syncwarp();
                    {
                        uint4 *gr = reinterpret_cast<uint4 *>(stg + lane * 64);
                        uint4 *ur = reinterpret_cast<uint4 *>(stg + 2048 + lane * 64);
                        const int swz = (lane >> 1) & 3;
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            gr[q4 ^ swz] = make_uint4(dgp[q4 * 4], dgp[q4 * 4 + 1], dgp[q4 * 4 + 2], dgp[q4 * 4 + 3]);
                            ur[q4 ^ swz] = make_uint4(dup[q4 * 4], dup[q4 * 4 + 1], dup[q4 * 4 + 2], dup[q4 * 4 + 3]);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int32_t col = e.c * 256 + ch * 32;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            if (grp * 32 + h * 16 < r16) {
                                const int32_t r0 = e.x0 + grp * 32 + h * 16;
                                tma_store_3d(&p.tmDgS, stg + h * 1024, col, r0, 0);
                                tma_store_3d(&p.tmDuS, stg + 2048 + h * 1024, col, r0, 0);
                            }
                        }
                        bulk_commit();
                    }
                }
                if (lane == 0) {  // the boxes have landed; ordered before the release below
                    bulk_wait<0>();
                    fence_proxy_async_global();
                }
                __syncwarp();
                if (!ok) break;
            } else if (e.kind == KB_DGU) {
                // dx_e rows as 16-row TMA boxes through the two halves of the
                // warp's staging buffer (64-byte swizzle); boxes past the unit's
                // 16-row-padded end are not stored (the next expert's rows), the
                // padding rows below it are never read
                const int r16 = e.x1 >> 16;
                const int swz = (lane >> 1) & 3;
#pragma unroll 1
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + ch * 32, r);
                    tmem_ld_wait();
                    uint8_t *buf = stg + (ch & 1) * 2048;
                    if (lane == 0) {
                        if (ch == 0)
                            bulk_wait_read<0>();  // the previous entry's boxes may span both halves
                        else
                            bulk_wait_read<1>();
                    }
                    __syncwarp();
                    uint4 *srow = reinterpret_cast<uint4 *>(buf + lane * 64);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const uint32_t *w = r + q4 * 8;
                        srow[q4 ^ swz] = make_uint4(pack_bf16x2(__uint_as_float(w[0]), __uint_as_float(w[1])),
                                                    pack_bf16x2(__uint_as_float(w[2]), __uint_as_float(w[3])),
                                                    pack_bf16x2(__uint_as_float(w[4]), __uint_as_float(w[5])),
                                                    pack_bf16x2(__uint_as_float(w[6]), __uint_as_float(w[7])));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            if (grp * 32 + h * 16 < r16)
                                tma_store_3d(&p.tmDxbS, buf + h * 1024, e.c * 256 + ch * 32, e.x0 + grp * 32 + h * 16, 0);
                        bulk_commit();
                    }
                }
                if (lane == 0) {  // landed, and ordered before the PUSH release below
                    bulk_wait<0>();
                    fence_proxy_async_global();
                }
                __syncwarp();
            } else if (e.kind == KB_DWD || e.kind == KB_DWGU) {
                // DWD: dW_down[e] rows (inter) x * 128 + row, columns (hidden) y * 256 ..
                // DWGU: columns 0-127 dW_gate[e] (hidden row x * 128 + row, inter y * 128 ..), 128-255 dW_up
                // Per iteration 64 columns (two tensor-memory loads) go out as
                // one 32 x 64 box through the warp's 4 KB staging buffer: the
                // tensor-copy unit also serves the operand loads of the next
                // tiles, and its cost goes with the number of boxes and rows.
                const int q = e.a / g.Eq;
                const int32_t r0 = e.b * 128 + grp * 32;
                uint32_t ra[32], rb[32];
                tmem_ld_32x32b_x32(taddr, ra);
                tmem_ld_32x32b_x32(taddr + 32, rb);
#pragma unroll 1
                for (int pr = 0; pr < 4; ++pr) {
                    tmem_ld_wait_regs(ra);
                    tmem_ld_wait_regs(rb);
                    if (zero) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) { ra[j] = 0u; rb[j] = 0u; }
                    }
                    if (lane == 0) bulk_wait_read<0>();  // the previous box has been read
                    __syncwarp();
                    bwd_stage_cols(stg, lane, ra, 0);
                    bwd_stage_cols(stg, lane, rb, 4);
                    if (pr + 1 < 4) {  // the next 64 columns load while this box is stored
                        tmem_ld_32x32b_x32(taddr + pr * 64 + 64, ra);
                        tmem_ld_32x32b_x32(taddr + pr * 64 + 96, rb);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (e.kind == KB_DWD)
                            tma_store_3d(&p.tmDwd[q], stg, e.c * 256 + pr * 64, r0, e.d);
                        else  // columns 0-127 dW_gate, 128-255 dW_up
                            tma_store_3d(pr < 2 ? &p.tmDwg[q] : &p.tmDwu[q], stg, e.c * 128 + (pr & 1) * 64, r0, e.d);
                        bulk_commit();
                    }
                }
            } else if (e.kind == KB_RDX) {
                const int q = e.a, bb = e.b;
                const int64_t left = g.Tq - static_cast<int64_t>(bb) * BM;
                const int ntok = static_cast<int>(left < BM ? left : BM);
                const int64_t t = static_cast<int64_t>(q) * g.Tq + static_cast<int64_t>(bb) * BM + row;
#pragma unroll 1
                for (int ch = 0; ch < 8; ++ch) {
                    float v[32];
                    acc_chunk(taddr + ch * 32, false, v);
                    if (row < ntok) {
                        float4 *dst = reinterpret_cast<float4 *>(p.dxr + t * g.H + e.c * 256 + ch * 32);
#pragma unroll
                        for (int j = 0; j < 8; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    }
                }
            } else {  // KB_DWR: dW_router rows (hidden) a * 128 + row, all E columns, fp32
                float *dst = p.dwr + (static_cast<int64_t>(e.a) * 128 + row) * g.E;
#pragma unroll 1
                for (int ch = 0; ch < g.E / 32; ++ch) {
                    float v[32];
                    acc_chunk(taddr + ch * 32, false, v);
                    float4 *d4 = reinterpret_cast<float4 *>(dst + ch * 32);
#pragma unroll
                    for (int j = 0; j < 8; ++j) d4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.tempty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            if (e.kind == KB_DH || e.kind == KB_DGU || e.kind == KB_RDX) {
                if (e.kind == KB_RDX) fence_proxy_async_global();  // dxr: generic stores, read by FOLD's tensor copies
                __threadfence();
                named_bar_sync(1, NUM_EPI_THREADS);
                if (et == 0) {
                    if (e.kind == KB_DH) {
                        red_release_add_gpu(&p.dh_cnt[e.a * g.MAXRB + e.b], 1u);
                    } else if (e.kind == KB_DGU) {
                        const int qe = e.a / g.Eq;
                        queue_put(&p.qctl[4 * qe + 0], p.push_items + qe * b.push_cap, p.push_flags + qe * b.push_cap,
                                  b.push_cap, push_code(e.a, e.b, e.c), epoch, p.ws);
                    } else {
                        bwd_fold_arrive(p, e.a * g.RB + e.b, e.c, 1u, epoch);
                    }
                }
            }
        } else if (e.kind == KB_ZPAD) {
            bwd_zpad(p, tb, e.a, et);
        } else if (e.kind == KB_GRADIN) {
            if (!bwd_gradin(p, sm, ps, tb, e, lane, et)) break;
        } else if (e.kind == KB_RBWD) {
            if (!bwd_rbwd(p, sm, ps, e, et)) break;
        } else if (e.kind == K_PUSH) {
            if (!bwd_push(p, sm, ps, e, et, lane, epoch)) break;
        } else if (e.kind == K_FOLD) {
            if (!bwd_fold(p, sm, ps, e, et)) break;
        }
        if (e.slot >= 0 && et == 0) {
            if (TraceRec *r = trace_rec(p.trace, blockIdx.x, e.slot)) r->t_done = static_cast<int64_t>(globaltimer());
        }
    }
    if (lane == 0) bulk_wait<0>();  // this warp's block stores have landed
    __syncwarp();
}

__global__ void __launch_bounds__(NUM_THREADS, 1) moe_bwd_kernel(const __grid_constant__ BwdParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const Smem sm = carve_smem(smem_raw);
    uint8_t *scratch = sm.stages + NSTAGE * STAGE_BYTES + SMEM_CTRL_BYTES;
    const MoeGeom &g = p.b.f;
    BwdTables tb;
    tb.offp = reinterpret_cast<int32_t *>(scratch);
    tb.us = tb.offp + g.E + 1;
    tb.cnt = tb.us + g.Eq + 1;
    tb.offl = tb.cnt + g.Eq;
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t epoch = *reinterpret_cast<volatile uint32_t *>(&p.ws->epoch);
    if (threadIdx.x == 0) {
        // the forward's context must come from a complete bf16 forward call
        const volatile WsHeader *fh = p.fwd_hdr;
        if (fh->status != KOSMOS_OK || fh->aux[2] != MOE_BF16_CTX) set_error(p.ws, KOSMOS_ERR_INVALID_ARG, -50);
    }
    if (warp == 0) bwd_load_tables(p, tb, lane);  // before the setup barrier: every warp reads them after it
    engine_setup(sm, warp);
    const uint32_t tmem_base = *sm.tmem_slot;
    if (warp == 0) {
        if (lane == 0) bwd_producer(p, sm, tb, epoch);
    } else if (warp == 1) {
        if (lane == 0) bwd_mma_loop(p, sm, tmem_base);
    } else {
        bwd_epilogue(p, sm, tb, tmem_base, scratch + BWD_TABLE_BYTES + (warp - 2) * 2 * BWD_STAGE_OUT, warp, lane,
                     epoch);
    }
    engine_teardown(sm, warp, tmem_base);
    __shared__ int s_last;
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = (atomicAdd(&p.ws->done_ctas, 1u) == gridDim.x - 1) ? 1 : 0;
    }
    __syncthreads();
    if (s_last && p.phase >= 1 && p.phase <= 6) {
        // a phase of the unfused baseline: the next launch goes on with the
        // counters and flags as they are, from fresh tickets
        if (threadIdx.x == 0) {
            volatile uint32_t *t = p.ws->tickets;
            for (int i = 0; i < KOSMOS_MAX_P; ++i) t[i] = 0u;
            *reinterpret_cast<volatile uint32_t *>(&p.ws->done_ctas) = 0u;
            __threadfence();
        }
    } else if (s_last) {
        __threadfence();
        uint4 *c = reinterpret_cast<uint4 *>(p.ctr);
        const int n16 = p.ctr_bytes / 16;
        for (int i = threadIdx.x; i < n16; i += blockDim.x) c[i] = make_uint4(0, 0, 0, 0);
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            volatile uint32_t *t = p.ws->tickets;
            for (int i = 0; i < KOSMOS_MAX_P; ++i) t[i] = 0u;
            *reinterpret_cast<volatile uint32_t *>(&p.ws->done_ctas) = 0u;
            __threadfence();
            *reinterpret_cast<volatile uint32_t *>(&p.ws->epoch) = epoch + 1u;
            __threadfence();
        }
    }
}

// ---------------------------------------------------------------- host side
size_t moe_bwd_workspace_bytes(int P, int64_t T, int64_t H, int E, int K, int64_t I, bool trace) {
    return bwd_ws_layout(bwd_geom(P, T, H, E, K, I), trace).total;
}

bool moe_bwd_debug_view(int what, int P, int64_t T, int64_t H, int E, int K, int64_t I, void *ws, void **ptr,
                        int64_t *bytes) {
    const BwdGeom b = bwd_geom(P, T, H, E, K, I);
    const BwdWsLayout L = bwd_ws_layout(b, what == 8);
    size_t off = 0, n = 0;
    switch (what) {
        case 0: off = L.dy; n = 2ull * b.rows16 * H; break;
        case 1: off = L.dg; n = 2ull * b.rows16 * I; break;
        case 2: off = L.du; n = 2ull * b.rows16 * I; break;
        case 3: off = L.dxb; n = 2ull * b.rows16 * H; break;
        case 4: off = L.dslot; n = 2ull * T * K * H; break;
        case 5: off = L.dgate; n = 4ull * T * K; break;
        case 6: off = L.dl; n = 2ull * T * E; break;
        case 7: off = L.dxr; n = 4ull * T * H; break;
        case 8: off = L.trace; n = static_cast<size_t>(MAX_CTAS) * TRACE_CAP * sizeof(TraceRec); break;
        default: return false;
    }
    *ptr = static_cast<uint8_t *>(ws) + off;
    *bytes = static_cast<int64_t>(n);
    return true;
}

kosmos_status launch_moe_bwd(const MoeBwdLaunch &Lc, cudaStream_t stream) {
    BwdParams p;
    memset(&p, 0, sizeof(p));
    p.b = bwd_geom(Lc.P, Lc.T, Lc.H, Lc.E, Lc.K, Lc.I);
    const BwdGeom &b = p.b;
    const MoeGeom &g = b.f;
    const BwdWsLayout L = bwd_ws_layout(b, Lc.trace != 0);
    const MoeWsLayout F = moe_ws_layout(g, false);
    const uint8_t *fw = static_cast<const uint8_t *>(Lc.fwd_ws);
    uint8_t *ws = static_cast<uint8_t *>(Lc.ws);
    p.fwd_hdr = reinterpret_cast<const WsHeader *>(fw);
    p.counts = reinterpret_cast<const int32_t *>(fw + F.counts);
    p.offl = reinterpret_cast<const int32_t *>(fw + F.offsets);
    p.unit_start = reinterpret_cast<const int32_t *>(fw + F.unit_start);
    p.base = reinterpret_cast<const int32_t *>(fw + F.base);
    p.rank_in_blk = reinterpret_cast<const int32_t *>(fw + F.rank_in_blk);
    p.inv_pos = reinterpret_cast<const int32_t *>(fw + F.inv_pos);
    p.logits = reinterpret_cast<const float *>(fw + F.logits);
    p.yslot = reinterpret_cast<const __nv_bfloat16 *>(fw + F.slot);
    p.gsave = reinterpret_cast<const __nv_bfloat16 *>(fw + F.gsave);
    p.usave = reinterpret_cast<const __nv_bfloat16 *>(fw + F.usave);
    p.topk_idx = Lc.topk_idx;
    p.topk_gate = Lc.topk_gate;
    p.dwr = Lc.dwr;
    p.ws = reinterpret_cast<WsHeader *>(ws);
    p.ctr = ws + L.ctr;
    p.ctr_bytes = static_cast<int>(L.ctr_bytes);
    p.dy_cnt = reinterpret_cast<uint32_t *>(ws + L.dy_cnt);
    p.dh_cnt = reinterpret_cast<uint32_t *>(ws + L.dh_cnt);
    p.dgate_cnt = reinterpret_cast<uint32_t *>(ws + L.dgate_cnt);
    p.rbwd_flag = reinterpret_cast<uint32_t *>(ws + L.rbwd_flag);
    p.rbwd_done = reinterpret_cast<uint32_t *>(ws + L.rbwd_done);
    p.fold_cnt = reinterpret_cast<uint32_t *>(ws + L.fold_cnt);
    p.qctl = reinterpret_cast<uint32_t *>(ws + L.qctl);
    p.push_items = reinterpret_cast<int32_t *>(ws + L.push_items);
    p.push_flags = reinterpret_cast<uint32_t *>(ws + L.push_flags);
    p.fold_items = reinterpret_cast<int32_t *>(ws + L.fold_items);
    p.fold_flags = reinterpret_cast<uint32_t *>(ws + L.fold_flags);
    p.dgate = reinterpret_cast<float *>(ws + L.dgate);
    p.dl = reinterpret_cast<__nv_bfloat16 *>(ws + L.dl);
    p.dxr = reinterpret_cast<float *>(ws + L.dxr);
    p.dy = reinterpret_cast<__nv_bfloat16 *>(ws + L.dy);
    p.dg = reinterpret_cast<__nv_bfloat16 *>(ws + L.dg);
    p.du = reinterpret_cast<__nv_bfloat16 *>(ws + L.du);
    p.dxb = reinterpret_cast<__nv_bfloat16 *>(ws + L.dxb);
    p.dslot = reinterpret_cast<__nv_bfloat16 *>(ws + L.dslot);
    p.trace = Lc.trace ? reinterpret_cast<TraceRec *>(ws + L.trace) : nullptr;
    p.wait_limit_ns = Lc.wait_limit_ns;
    const uint64_t H = static_cast<uint64_t>(g.H), I = static_cast<uint64_t>(g.I), E = static_cast<uint64_t>(g.E);
    const uint64_t Eq = static_cast<uint64_t>(g.Eq), Tq = static_cast<uint64_t>(g.Tq), T = static_cast<uint64_t>(g.T);
    const uint64_t TK = static_cast<uint64_t>(g.T * g.K), R16 = static_cast<uint64_t>(b.rows16);
    const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto SW = CU_TENSOR_MAP_SWIZZLE_128B;
    auto map2 = [&](CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer, uint32_t b0, uint32_t b1) {
        const uint64_t dims[2] = {inner, outer};
        const uint64_t st[1] = {inner * 2};
        const uint32_t box[2] = {b0, b1};
        return encode_tmap(m, BF, 2, const_cast<void *>(ptr), dims, st, box, SW);
    };
    auto mapgu = [&](CUtensorMap *m, const void *ptr) {
        const uint64_t dims[2] = {static_cast<uint64_t>(I), static_cast<uint64_t>(TK)};
        const uint64_t st[1] = {static_cast<uint64_t>(I) * 2};
        const uint32_t box[2] = {32, BM};
        return encode_tmap(m, BF, 2, const_cast<void *>(ptr), dims, st, box, CU_TENSOR_MAP_SWIZZLE_64B);
    };
    auto map3 = [&](CUtensorMap *m, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1) {
        const uint64_t dims[3] = {d0, d1, d2};
        const uint64_t st[2] = {d0 * 2, d0 * d1 * 2};
        const uint32_t box[3] = {b0, b1, 1};
        return encode_tmap(m, BF, 3, const_cast<void *>(ptr), dims, st, box, SW);
    };
    bool ok = map2(&p.tmDyA, p.dy, H, R16, BK, BM) && map2(&p.tmDyB, p.dy, H, R16, 64, BK) &&
              map2(&p.tmDgA, p.dg, I, R16, BK, BM) && map2(&p.tmDuA, p.du, I, R16, BK, BM) &&
              map2(&p.tmDgB, p.dg, I, R16, 64, BK) && map2(&p.tmDuB, p.du, I, R16, 64, BK) &&
              map2(&p.tmH, fw + F.h, I, TK, 64, BK) && map2(&p.tmX, fw + F.recv, H, TK, 64, BK) &&
              mapgu(&p.tmGs, fw + F.gsave) && mapgu(&p.tmUs, fw + F.usave) &&
              map2(&p.tmDlA, p.dl, E, T, BK, BM) && map2(&p.tmDlB, p.dl, E, T, 64, BK) &&
              map2(&p.tmWrT, Lc.wr, E, H, BK, 256);
    for (int q = 0; ok && q < g.P; ++q) {
        p.dout[q] = static_cast<const __nv_bfloat16 *>(Lc.dout[q]);
        p.dx[q] = static_cast<__nv_bfloat16 *>(Lc.dx[q]);
        p.dwg[q] = static_cast<__nv_bfloat16 *>(Lc.dwg[q]);
        p.dwu[q] = static_cast<__nv_bfloat16 *>(Lc.dwu[q]);
        p.dwd[q] = static_cast<__nv_bfloat16 *>(Lc.dwd[q]);
        {
            const uint64_t dims[2] = {H, static_cast<uint64_t>(g.Tq)};
            const uint64_t st[1] = {H * 2};
            const uint32_t box[2] = {256, 32};
            ok = encode_tmap(&p.tmDout[q], BF, 2, const_cast<void *>(Lc.dout[q]), dims, st, box,
                             CU_TENSOR_MAP_SWIZZLE_NONE);
        }
        ok = ok && map3(&p.tmWdT[q], Lc.wd[q], H, I, Eq, BK, 256) && map3(&p.tmWgT[q], Lc.wg[q], I, H, Eq, BK, 256) &&
             map3(&p.tmWuT[q], Lc.wu[q], I, H, Eq, BK, 256) && map2(&p.tmXs[q], Lc.x[q], H, Tq, 64, BK);
        auto out3 = [&](CUtensorMap *m, void *ptr, uint64_t d0, uint64_t d1) {
            const uint64_t dims[3] = {d0, d1, Eq};
            const uint64_t st[2] = {d0 * 2, d0 * d1 * 2};
            const uint32_t box[3] = {64, 32, 1};
            return encode_tmap(m, BF, 3, ptr, dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B);
        };
        ok = ok && out3(&p.tmDwg[q], Lc.dwg[q], I, H) && out3(&p.tmDwu[q], Lc.dwu[q], I, H) &&
             out3(&p.tmDwd[q], Lc.dwd[q], H, I);
    }
    if (ok) {
        const uint64_t dims[2] = {H, TK};
        const uint64_t st[1] = {H * 2};
        const uint32_t box[2] = {256, static_cast<uint32_t>(b.fold_tps * g.K)};
        ok = encode_tmap(&p.tmDslot, BF, 2, p.dslot, dims, st, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (ok) {
        const uint64_t dims[3] = {H, static_cast<uint64_t>(g.K), static_cast<uint64_t>(g.T)};
        const uint64_t st[2] = {H * 2, H * 2 * static_cast<uint64_t>(g.K)};
        const uint32_t box[3] = {256, 1, 32};
        ok = encode_tmap(&p.tmYslot, BF, 3, const_cast<__nv_bfloat16 *>(p.yslot), dims, st, box,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (ok) {
        const uint64_t dims[3] = {I, R16, 1};
        const uint64_t st[2] = {I * 2, I * 2 * R16};
        const uint32_t box[3] = {32, 16, 1};
        ok = encode_tmap(&p.tmDgS, BF, 3, p.dg, dims, st, box, CU_TENSOR_MAP_SWIZZLE_64B) &&
             encode_tmap(&p.tmDuS, BF, 3, p.du, dims, st, box, CU_TENSOR_MAP_SWIZZLE_64B);
    }
    if (ok) {
        const uint64_t dims[2] = {E, T};
        const uint64_t st[1] = {E * 4};
        const uint32_t box[2] = {static_cast<uint32_t>(E), static_cast<uint32_t>(b.rbwd_tps)};
        ok = encode_tmap(&p.tmLogits, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(p.logits), dims, st, box,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (ok) {
        const uint64_t dims[3] = {H, R16, 1};
        const uint64_t st[2] = {H * 2, H * 2 * R16};
        const uint32_t box[3] = {32, 16, 1};
        ok = encode_tmap(&p.tmDxbS, BF, 3, p.dxb, dims, st, box, CU_TENSOR_MAP_SWIZZLE_64B);
    }
    if (ok) {
        const uint64_t dims[2] = {H, R16};
        const uint64_t st[1] = {H * 2};
        const uint32_t box[2] = {256, 64};
        ok = encode_tmap(&p.tmDxbP, BF, 2, p.dxb, dims, st, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (ok) {
        const uint64_t dims[2] = {H, static_cast<uint64_t>(g.T)};
        const uint64_t st[1] = {H * 4};
        const uint32_t box[2] = {256, static_cast<uint32_t>(b.fold_tps)};
        ok = encode_tmap(&p.tmDxr, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.dxr, dims, st, box,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (!ok) return KOSMOS_ERR_CUDA;
    if (Lc.sched != KOSMOS_SCHED_UNFUSED)
        return launch_persistent(reinterpret_cast<const void *>(&moe_bwd_kernel), &p, Lc.grid, BWD_SMEM_BYTES, stream,
                                 Lc.plain_launch != 0);
    // unfused baseline: the same kernel once per phase, each launch running
    // only its phase's entries to completion before the next starts
    for (int ph = 1; ph <= 7; ++ph) {
        p.phase = ph;
        const kosmos_status st = launch_persistent(reinterpret_cast<const void *>(&moe_bwd_kernel), &p, Lc.grid,
                                                   BWD_SMEM_BYTES, stream, Lc.plain_launch != 0);
        if (st != KOSMOS_OK) return st;
    }
    return KOSMOS_OK;
}

}  // namespace kosmos
