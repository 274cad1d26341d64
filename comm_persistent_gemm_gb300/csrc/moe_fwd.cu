// moe_fwd.cu -- MoE expert layer forward, router to fold, in ONE persistent
// launch (KOSMOS abstract: "runs an entire expert layer, from router to fold,
// in one launch per direction").
//
// P emulated expert-parallel ranks; CTA c plays rank q = c mod P.  Rank q owns
// tokens [q*Tq, (q+1)*Tq) and experts [q*Eq, (q+1)*Eq).
//
// Main rail of rank q (claimed in ticket order by rank q's CTAs):
//   ROUTE(b)        router GEMM of 128 tokens x W_router (tcgen05), epilogue:
//                   fp32 softmax, top-k (ties to the lower expert), gates
//                   renormalised over the top-k, per-block expert counts and
//                   each slot's rank inside its block.  The CTA that finishes
//                   the last ROUTE of all ranks runs PLAN: expert counts,
//                   exclusive offsets (receive order expert-major, then
//                   token), per-block bases, per-rank row-block units.
//   DISPATCH(b, k)  the all-to-all to the expert ranks: slot k of 128 tokens is
//                   copied (bulk async copies) to row pos = base + rank of the
//                   expert-ordered receive buffer; per (expert, row block)
//                   arrival counters are released.
//   TILE_GU / TILE_D  per unit u = (expert, 128-row block), consumer-ordered
//                   with a lag of two experts: GU(e0) | GU(e1) | GU(e2) D(e0) | ...
//                   GU: [rows x H] . [W_gate | W_up] (128 + 128 columns) with a
//                   SwiGLU epilogue h = silu(gate) * up; D: [rows x I] . W_down.
// Ready queues of rank q (the combine step, two-way role switching; explainer
// paragraph "KOSMOS removes the manager": push any ready result, otherwise
// build a tile):
//   PUSH(e, rb, dn) queued when a TILE_D finishes; copies the 256-column
//                   slice of each row back to its source slot[t][k];
//   FOLD(g, dn)     queued when all k slots of token block g have arrived for
//                   column tile dn; out[t] = sum_k gate[t][k] * slot[t][k] in
//                   fp32, k in emission order, one rounding to bf16.
// A CTA takes a ready PUSH first, else its next main-rail entry, else a ready
// FOLD, and exits when its rank's rail and queues are drained.
//
// MXFP8 variant (E4M3 elements, one E8M0 scale per 32 K-elements, on every
// operand of the expert GEMMs): between ROUTE and DISPATCH the rail holds
//   QUANT(j)        16 token rows of the rank quantised along the hidden
//                   dimension (bf16 rows staged through the pipeline; scales
//                   row-major); DISPATCH then moves E4M3 rows and their scales;
// each expert's receive rows start on a 128-row boundary (the scale atoms of
// the block-scaled MMA cover 128 aligned rows); the GU epilogue quantises h
// along the intermediate dimension for TILE_D.  The router stays bf16.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>

#include "moe_common.cuh"
#include "launch.h"

namespace kosmos {

struct MoeParams {
    CUtensorMap tmX[KOSMOS_MAX_P];   // x_shards[q]: dims {H, Tq}, box {64, 128}
    CUtensorMap tmWr;                // w_router: dims {E, H}, box {64, 64}
    CUtensorMap tmRecv;              // receive buffer: dims {H, rows_cap}, box {64, 128}
    CUtensorMap tmH;                 // SwiGLU output: dims {I, rows_cap}, box {64, 128}
    CUtensorMap tmYbuf;              // D output rows: dims {H, rows_cap, 1}, box {32, 32, 1}, 64-byte swizzle
    CUtensorMap tmWg[KOSMOS_MAX_P];  // w_gate[q]: dims {I, H, Eq}, box {64, 64, 1}
    CUtensorMap tmWu[KOSMOS_MAX_P];  // w_up[q]:   dims {I, H, Eq}, box {64, 64, 1}
    CUtensorMap tmWd[KOSMOS_MAX_P];  // w_down[q]: dims {H, I, Eq}, box {64, 64, 1}
    CUtensorMap tmSlot;              // slot buffer: dims {H, T*K}, box {256, fold_tps*K}, no swizzle
    // MXFP8 (the maps above then hold E4M3 bytes: tmRecv, tmH box {128, 128};
    // tmWg, tmWu, tmWd box {128, 128, 1}): tiled scales as rows of 16 bytes,
    // one 512-byte atom per box (encode_sf_tmap)
    CUtensorMap tmSRecv;             // receive-row scales, K = H
    CUtensorMap tmSH;                // h scales, K = I
    CUtensorMap tmSWg[KOSMOS_MAX_P]; // per expert: I/128 column atoms x H/128 K atoms
    CUtensorMap tmSWu[KOSMOS_MAX_P];
    CUtensorMap tmSWd[KOSMOS_MAX_P]; // per expert: H/128 column atoms x I/128 K atoms
    const __nv_bfloat16 *x[KOSMOS_MAX_P];
    __nv_bfloat16 *y[KOSMOS_MAX_P];
    int32_t *topk_idx;
    float *topk_gate;
    int32_t *counts_out;
    int32_t *pos_out;
    WsHeader *ws;
    uint8_t *ctr;
    int ctr_bytes;
    int identity;
    uint32_t *disp_cnt, *gu_cnt, *fold_cnt, *qctl, *route_done;
    int32_t *blk_counts, *rank_in_blk, *base, *offsets, *counts, *unit_start, *inv_pos;
    int32_t *offl;                   // receive offsets without padding (dispatch_pos is reported in these)
    uint32_t *quant_cnt;             // MXFP8: quantised rows per route block
    uint8_t *xq, *xs;                // MXFP8: quantised tokens [T, H], scales [T, H/32] row-major
    uint8_t *recv8, *recv_sf, *h8, *h_sf;
    int32_t *push_items, *fold_items;
    uint32_t *push_flags, *fold_flags;
    float *logits;
    __nv_bfloat16 *recv, *h, *ybuf, *slot;
    __nv_bfloat16 *gsave, *usave;    // bf16: g and u of every receive row (saved for the backward)
    TraceRec *trace;
    MoeGeom g;
    int fold_tps;                    // FOLD: tokens per pipeline stage (64 / K)
    int phase;                       // 0: the whole layer in this launch; 1-5: one phase of the unfused
                                     // baseline (ROUTE+PLAN[+QUANT] | DISPATCH | TILE_GU | TILE_D | PUSH+FOLD)
    uint64_t wait_limit_ns;
    uint64_t inject;
};

// ---------------------------------------------------------------- producer (warp 0)
enum MoeAct : int { ACT_NONE = 0, ACT_DISPATCH = 1, ACT_EXIT = 2, ACT_PLAN = 3 };

struct MoeProdState {
    PipeState ps;
    RingState rs;
    uint32_t cphase = 0;
    int nrec = 0;
    bool main_done = false;
    bool plan_seen = false;
    uint64_t idle_t0 = 0;
    // this rank's plan, copied to shared memory once it is published:
    // us[Eq + 1] row-block prefix, off[Eq] receive offsets, cnt[Eq] row counts
    int32_t *us = nullptr, *off = nullptr, *cnt = nullptr;
    uint8_t *sf = nullptr;  // MXFP8: per-stage scale atoms
    int64_t pending = -1;  // a claimed main-rail ticket waiting for the plan table
    int64_t ahead = -1;    // the next main-rail ticket, claimed early so its latency overlaps the current entry
};


__device__ __forceinline__ int trace_open(const MoeParams &p, MoeProdState &st, int kind, int ticket, int64_t tc) {
    int slot = -1;
    if (TraceRec *r = trace_rec(p.trace, blockIdx.x, st.nrec)) {
        r->t_claim = tc; r->t_ready = static_cast<int64_t>(globaltimer()); r->t_done = 0;
        r->kind = kind; r->ticket = ticket; r->cta = blockIdx.x;
        slot = st.nrec;
    }
    ++st.nrec;
    return slot;
}

// The whole producer warp, once the plan is published (lane 0 acquired its
// flag): copies this rank's plan into the shared-memory table.
__device__ __forceinline__ void load_plan_table(const MoeParams &p, MoeProdState &st, int lane) {
    const MoeGeom &g = p.g;
    const int q = blockIdx.x % g.P;
    __syncwarp();  // orders lane 0's acquire of the plan before the other lanes' reads
    for (int j = lane; j <= g.Eq; j += 32) st.us[j] = ldcg_i32(&p.unit_start[q * (g.Eq + 1) + j]);
    for (int j = lane; j < g.Eq; j += 32) {
        st.off[j] = ldcg_i32(&p.offsets[q * g.Eq + j]);
        st.cnt[j] = ldcg_i32(&p.counts[q * g.Eq + j]);
    }
    __syncwarp();
    st.plan_seen = true;
}

// Waits until every pipeline stage is free (all earlier MMAs have read their
// operands), so the stage buffers can serve as copy buffers.
__device__ __forceinline__ bool drain_pipeline(const MoeParams &p, const Smem &sm, const PipeState &ps) {
    for (int i = 0; i < NSTAGE; ++i) {
        uint32_t s = ps.stage + i, ph = ps.phase;
        if (s >= NSTAGE) { s -= NSTAGE; ph ^= 1u; }
        if (!mbar_wait(&sm.empty[s], ph ^ 1u, PIPE_LIMIT_NS)) {
            set_error(p.ws, KOSMOS_ERR_DEVICE, -11);
            return false;
        }
    }
    return true;
}

// Expert tile rail of rank q, grouped by expert with a lag of MOE_LAG experts:
//   GU(e0) | GU(e1) | GU(e2) D(e0) | GU(e3) D(e1) | ... | D(e_last)
// so that a D tile, which needs every GU column block of its rows, is claimed
// well after them.  GU(e): column block outer, row block inner (the row
// blocks of one weight slice are adjacent, so the slice is read from DRAM
// once); D(e) likewise.  With U(j) = row blocks of the rank's experts before
// expert j (clamped to [0, Eq]), group j starts at NGU U(j) + ND U(j - LAG).
constexpr int MOE_LAG = 2;
__device__ __forceinline__ void moe_decode_tile(const MoeParams &p, const int32_t *us, int tt, int &kind, int &le,
                                                int &rb, int &col) {
    const MoeGeom &g = p.g;
    auto U = [&](int j) { return j <= 0 ? 0 : us[j < g.Eq ? j : g.Eq]; };
    kind = 0;
    const int total = U(g.Eq);
    if (tt < 0 || tt >= total * (g.NGU + g.ND)) return;
    for (int j = 0; j < g.Eq + MOE_LAG; ++j) {
        const int ngu = j < g.Eq ? U(j + 1) - U(j) : 0;                        // row blocks of expert j
        const int nd = j >= MOE_LAG ? U(j - MOE_LAG + 1) - U(j - MOE_LAG) : 0;  // of expert j - LAG
        const int start = g.NGU * U(j) + g.ND * U(j - MOE_LAG);
        if (tt < start + g.NGU * ngu + g.ND * nd) {
            const int r = tt - start;
            if (r < g.NGU * ngu) {
                kind = K_TILE_GU; le = j; col = r / ngu; rb = r % ngu;
            } else {
                const int r2 = r - g.NGU * ngu;
                kind = K_TILE_D; le = j - MOE_LAG; col = r2 / nd; rb = r2 % nd;
            }
            return;
        }
    }
}

// Lane 0 of the producer warp: claims and issues one piece of work.  Returns
// ACT_DISPATCH (with v0 = b, v1 = k, v2 = ticket) when the whole warp must
// help, ACT_EXIT when this CTA is finished.
__device__ __forceinline__ int moe_decide(const MoeParams &p, const Smem &sm, MoeProdState &st, uint32_t epoch, int &v0,
                                       int &v1, int &v2) {
    const MoeGeom &g = p.g;
    const int q = blockIdx.x % g.P;
    uint32_t *qc = p.qctl + 4 * q;
    if (failed(p.ws)) return ACT_EXIT;
    const int ph = p.phase;
    if (ph == 5 && !st.plan_seen) {  // the combine alone: the plan of the earlier launches, no main rail
        if (!wait_flag_eq(p.ws, &p.ws->aux[1], epoch + 1u, p.wait_limit_ns, -10)) return ACT_EXIT;
        st.main_done = true;
        return ACT_PLAN;
    }
    // main-rail tickets: one counter per rank; a phase of the unfused baseline
    // counts from its own first ticket (the counters start from zero in
    // every launch)
    const uint32_t base = ph == 2 ? static_cast<uint32_t>(g.RB + g.NQ) : (ph >= 3 ? static_cast<uint32_t>(g.n_head) : 0u);
    uint32_t *tctr = &p.ws->tickets[q];
    // 1) a ready result to push back to its source rank
    if (st.plan_seen && (ph == 0 || ph == 5)) {
        int32_t code;
        if (queue_try_take(&qc[1], &qc[0], p.push_items + q * g.push_cap, p.push_flags + q * g.push_cap, epoch,
                           code, p.ws)) {
            int e, rb, dn;
            push_decode(code, e, rb, dn);
            SchedEntry en;
            fill_entry(en, K_PUSH, e, rb, dn, 0, code,
                       trace_open(p, st, K_PUSH, code, p.trace ? static_cast<int64_t>(globaltimer()) : 0));
            en.x0 = st.off[e - q * g.Eq] + rb * BM;
            const int rows = st.cnt[e - q * g.Eq] - rb * BM;
            en.x1 = rows < BM ? rows : BM;
            ring_push(sm, st.rs, en, p.ws);
            st.idle_t0 = 0;
            return ACT_NONE;
        }
        if (failed(p.ws)) return ACT_EXIT;
    }
    // 2) the next entry of this rank's main rail
    if (!st.main_done) {
        uint32_t t;
        if (st.pending >= 0) {
            t = static_cast<uint32_t>(st.pending);
        } else if (st.ahead >= 0) {
            t = static_cast<uint32_t>(st.ahead);
        } else {
            t = base + atomicAdd(tctr, 1u);
        }
        st.pending = -1;
        st.ahead = -1;
        if ((ph == 1 && t >= static_cast<uint32_t>(g.RB + g.NQ)) || (ph == 2 && t >= static_cast<uint32_t>(g.n_head)))
            return ACT_EXIT;  // this launch's phase of the rail is done
        const int64_t tc = p.trace ? static_cast<int64_t>(globaltimer()) : 0;
        if (t < static_cast<uint32_t>(g.RB)) {  // ROUTE(b)
            const int b = static_cast<int>(t);
            SchedEntry en;
            fill_entry(en, K_ROUTE, q, b, q * g.RB + b, g.nkb_r, t, trace_open(p, st, K_ROUTE, t, tc));
            en.nmma = g.E;
            if (!ring_push(sm, st.rs, en, p.ws)) return ACT_EXIT;
            const uint32_t bytes = A_STAGE_BYTES + (g.E / 64) * (64 * BK * 2);
            for (int kb = 0; kb < g.nkb_r; ++kb) {
                if (!mbar_wait(&sm.empty[st.ps.stage], st.ps.phase ^ 1u, PIPE_LIMIT_NS)) {
                    set_error(p.ws, KOSMOS_ERR_DEVICE, t);
                    return ACT_EXIT;
                }
                uint8_t *sa = sm.stages + st.ps.stage * STAGE_BYTES;
                uint8_t *sb = sa + A_STAGE_BYTES;
                uint64_t *bar = &sm.full[st.ps.stage];
                mbar_arrive_expect_tx(bar, bytes);
                tma_load_2d(sa, &p.tmX[q], bar, kb * BK, b * BM);
                for (int j = 0; j < g.E / 64; ++j) tma_load_2d(sb + j * (64 * BK * 2), &p.tmWr, bar, j * 64, kb * BK);
                st.ps.advance();
            }
            st.idle_t0 = 0;
            return ACT_NONE;
        }
        if (t < static_cast<uint32_t>(g.RB + g.NQ)) {  // QUANT(j): bf16 token rows through the stages
            const int j = static_cast<int>(t) - g.RB;
            const int64_t r0 = static_cast<int64_t>(j) * MOE_QR;
            const int rows = static_cast<int>((g.Tq - r0) < MOE_QR ? (g.Tq - r0) : MOE_QR);
            const uint32_t rbytes = static_cast<uint32_t>(g.H * 2);
            const int rps = STAGE_BYTES / static_cast<int>(rbytes);
            SchedEntry en;
            fill_entry(en, K_QUANT, q, j, rows, (rows + rps - 1) / rps, t, trace_open(p, st, K_QUANT, t, tc));
            if (!ring_push(sm, st.rs, en, p.ws)) return ACT_EXIT;
            const uint8_t *src = reinterpret_cast<const uint8_t *>(p.x[q] + r0 * g.H);
            for (int s0 = 0; s0 < rows; s0 += rps) {
                if (!mbar_wait(&sm.empty[st.ps.stage], st.ps.phase ^ 1u, PIPE_LIMIT_NS)) {
                    set_error(p.ws, KOSMOS_ERR_DEVICE, t);
                    return ACT_EXIT;
                }
                const int n = (rows - s0) < rps ? (rows - s0) : rps;
                uint64_t *bar = &sm.full[st.ps.stage];
                mbar_arrive_expect_tx(bar, n * rbytes);
                for (int i = 0; i < n; ++i)
                    bulk_g2s(sm.stages + st.ps.stage * STAGE_BYTES + i * rbytes, src + (s0 + i) * static_cast<int64_t>(rbytes),
                             rbytes, bar);
                st.ps.advance();
            }
            st.idle_t0 = 0;
            return ACT_NONE;
        }
        if (!st.plan_seen) {  // every later entry needs the plan: wait for it, then the warp loads the table
            if (!wait_flag_eq(p.ws, &p.ws->aux[1], epoch + 1u, p.wait_limit_ns, -10)) return ACT_EXIT;
            st.pending = t;
            return ACT_PLAN;
        }
        if (t < static_cast<uint32_t>(g.n_head)) {  // DISPATCH(b, k)
            const int i = static_cast<int>(t) - g.RB - g.NQ;
            v0 = i / g.K;
            v1 = i % g.K;
            v2 = static_cast<int>(t);
            st.idle_t0 = 0;
            return ACT_DISPATCH;
        }
        const int tt = static_cast<int>(t) - g.n_head;
        int kind = 0, le = 0, rb = 0, col = 0;
        moe_decode_tile(p, st.us, tt, kind, le, rb, col);
        if (kind == 0) {
            st.main_done = true;
            if (ph != 0) return ACT_EXIT;
        } else if ((ph == 3 && kind != K_TILE_GU) || (ph == 4 && kind != K_TILE_D)) {
            st.ahead = base + atomicAdd(tctr, 1u);  // another phase's tile: take the next ticket
            return ACT_NONE;
        } else {
            // claim the next tile ticket now; its value is first needed after this
            // entry's loads are issued, so the atomic's round trip overlaps them
            const uint32_t nxt = base + atomicAdd(tctr, 1u);
            const int e = q * g.Eq + le;
            const int row0 = st.off[le] + rb * BM;
            const int left = st.cnt[le] - rb * BM;
            const int rows = left < BM ? left : BM;
            const int ci = e * g.MAXRB + rb;
            if (kind == K_TILE_GU) {
                if (!wait_flag_eq(p.ws, &p.disp_cnt[ci], static_cast<uint32_t>(rows), p.wait_limit_ns, t))
                    return ACT_EXIT;
            } else {
                if (!wait_flag_eq(p.ws, &p.gu_cnt[ci], static_cast<uint32_t>(g.NGU), p.wait_limit_ns, t))
                    return ACT_EXIT;
            }
            const int slot = trace_open(p, st, kind, t, tc);
            if (p.identity) {
                // identity experts: no GEMMs; keep the dependency chain and the push
                if (kind == K_TILE_GU) {
                    __threadfence();
                    red_release_add_gpu(&p.gu_cnt[ci], 1u);
                } else {
                    const int qe = e / g.Eq;
                    queue_put(&p.qctl[4 * qe + 0], p.push_items + qe * g.push_cap, p.push_flags + qe * g.push_cap,
                              g.push_cap, push_code(e, rb, col), epoch, p.ws);
                }
                if (TraceRec *r = trace_rec(p.trace, blockIdx.x, slot)) r->t_done = static_cast<int64_t>(globaltimer());
                st.idle_t0 = 0;
                st.ahead = nxt;
                return ACT_NONE;
            }
            SchedEntry en;
            fill_entry(en, kind, e, rb, col, kind == K_TILE_GU ? g.nkb_h : g.nkb_i, t, slot);
            en.x0 = row0;
            en.x1 = rows;
            en.d = le;
            if (!ring_push(sm, st.rs, en, p.ws)) return ACT_EXIT;
            for (int kb = 0; kb < en.nstage; ++kb) {
                if (!mbar_wait(&sm.empty[st.ps.stage], st.ps.phase ^ 1u, PIPE_LIMIT_NS)) {
                    set_error(p.ws, KOSMOS_ERR_DEVICE, t);
                    return ACT_EXIT;
                }
                uint8_t *sa = sm.stages + st.ps.stage * STAGE_BYTES;
                uint8_t *sb = sa + A_STAGE_BYTES;
                uint64_t *bar = &sm.full[st.ps.stage];
                if (g.mx) {
                    // A 128 rows x 128 bytes, B two 128-column slabs of 16 KB, three scale atoms
                    uint8_t *sfs = st.sf + st.ps.stage * MOE_SF_BYTES;
                    mbar_arrive_expect_tx(bar, STAGE_BYTES + MOE_SF_BYTES);
                    if (kind == K_TILE_GU) {
                        const int wa = (le * g.NGU + col) * g.nkb_h + kb;  // weight atom (gate and up alike)
                        tma_load_2d(sa, &p.tmRecv, bar, kb * FBK, row0);
                        tma_load_3d(sb, &p.tmWg[q], bar, col * 128, kb * FBK, le);
                        tma_load_3d(sb + 16384, &p.tmWu[q], bar, col * 128, kb * FBK, le);
                        tma_load_2d(sfs, &p.tmSRecv, bar, 0, ((row0 / BM) * g.nkb_h + kb) * SF_ATOM_ROWS);
                        tma_load_2d(sfs + 512, &p.tmSWg[q], bar, 0, wa * SF_ATOM_ROWS);
                        tma_load_2d(sfs + 1024, &p.tmSWu[q], bar, 0, wa * SF_ATOM_ROWS);
                    } else {
                        const int wa = (le * 2 * g.ND + 2 * col) * g.nkb_i + kb;  // down atoms of columns 2col, 2col+1
                        tma_load_2d(sa, &p.tmH, bar, kb * FBK, row0);
                        tma_load_3d(sb, &p.tmWd[q], bar, col * BN, kb * FBK, le);
                        tma_load_3d(sb + 16384, &p.tmWd[q], bar, col * BN + 128, kb * FBK, le);
                        tma_load_2d(sfs, &p.tmSH, bar, 0, ((row0 / BM) * g.nkb_i + kb) * SF_ATOM_ROWS);
                        tma_load_2d(sfs + 512, &p.tmSWd[q], bar, 0, wa * SF_ATOM_ROWS);
                        tma_load_2d(sfs + 1024, &p.tmSWd[q], bar, 0, (wa + g.nkb_i) * SF_ATOM_ROWS);
                    }
                    st.ps.advance();
                    continue;
                }
                mbar_arrive_expect_tx(bar, STAGE_BYTES);
                if (kind == K_TILE_GU) {
                    tma_load_2d(sa, &p.tmRecv, bar, kb * BK, row0);
                    tma_load_3d(sb + 0 * 8192, &p.tmWg[q], bar, col * 128 + 0, kb * BK, le);
                    tma_load_3d(sb + 1 * 8192, &p.tmWg[q], bar, col * 128 + 64, kb * BK, le);
                    tma_load_3d(sb + 2 * 8192, &p.tmWu[q], bar, col * 128 + 0, kb * BK, le);
                    tma_load_3d(sb + 3 * 8192, &p.tmWu[q], bar, col * 128 + 64, kb * BK, le);
                } else {
                    tma_load_2d(sa, &p.tmH, bar, kb * BK, row0);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        tma_load_3d(sb + j * 8192, &p.tmWd[q], bar, col * BN + j * 64, kb * BK, le);
                }
                st.ps.advance();
            }
            st.idle_t0 = 0;
            st.ahead = nxt;
            return ACT_NONE;
        }
    }
    // 3) a ready fold of this rank's tokens
    if (st.plan_seen && (ph == 0 || ph == 5)) {
        int32_t code;
        if (queue_try_take(&qc[3], &qc[2], p.fold_items + q * g.fold_cap, p.fold_flags + q * g.fold_cap, epoch, code,
                           p.ws)) {
            // the block's K slot rows of every token, column tile dn, through the
            // stage ring: fold_tps tokens (fold_tps * K rows x 256 columns) per stage
            const int gb = code & 0xFFFF, dn = (code >> 16) & 0xFFFF;
            const int qs = gb / g.RB, bq = gb % g.RB;
            const int64_t left = g.Tq - static_cast<int64_t>(bq) * BM;
            const int ntok = static_cast<int>(left < BM ? left : BM);
            const int nst = (ntok + p.fold_tps - 1) / p.fold_tps;
            const int64_t row0 = (static_cast<int64_t>(qs) * g.Tq + static_cast<int64_t>(bq) * BM) * g.K;
            SchedEntry en;
            fill_entry(en, K_FOLD, gb, 0, dn, nst, code,
                       trace_open(p, st, K_FOLD, code, p.trace ? static_cast<int64_t>(globaltimer()) : 0));
            if (!ring_push(sm, st.rs, en, p.ws)) return ACT_EXIT;
            const uint32_t bytes = static_cast<uint32_t>(BN * 2 * p.fold_tps * g.K);
            for (int s = 0; s < nst; ++s) {
                if (!mbar_wait(&sm.empty[st.ps.stage], st.ps.phase ^ 1u, PIPE_LIMIT_NS)) {
                    set_error(p.ws, KOSMOS_ERR_DEVICE, code);
                    return ACT_EXIT;
                }
                uint64_t *bar = &sm.full[st.ps.stage];
                mbar_arrive_expect_tx(bar, bytes);
                tma_load_2d(sm.stages + st.ps.stage * STAGE_BYTES, &p.tmSlot, bar, dn * BN,
                            static_cast<int32_t>(row0 + static_cast<int64_t>(s) * p.fold_tps * g.K));
                st.ps.advance();
            }
            st.idle_t0 = 0;
            return ACT_NONE;
        }
        if (failed(p.ws)) return ACT_EXIT;
    }
    // 4) finished when the rail and both queues of this rank are drained
    if (st.main_done && st.plan_seen) {
        const uint32_t push_total = static_cast<uint32_t>(st.us[g.Eq]) * g.ND;
        const uint32_t fold_total = static_cast<uint32_t>(g.fold_cap);
        if (ld_relaxed_gpu(&qc[1]) >= push_total && ld_relaxed_gpu(&qc[3]) >= fold_total) return ACT_EXIT;
    }
    const uint64_t now = globaltimer();
    if (st.idle_t0 == 0) {
        st.idle_t0 = now;
    } else if (now - st.idle_t0 > p.wait_limit_ns) {
        set_error(p.ws, KOSMOS_ERR_TIMEOUT, -12);
        return ACT_EXIT;
    }
    return ACT_NONE;
}

// The whole producer warp: slot k of the 128 tokens of block b goes to the
// receive buffer of its expert's rank.  Lanes compute the destination rows;
// lane 0 moves the rows with bulk async copies through the stage buffers and
// then releases the per-(expert, row block) arrival counters.  MXFP8: the
// rows are the block's quantised rows (once its QUANT entries are done), and
// the lanes first copy each row's scale words (4 K-blocks each) into the
// tiled scale atoms of the destination row.
__device__ __noinline__ MoeProdState moe_dispatch(const MoeParams &p, const Smem &sm, MoeProdState st, uint8_t *pscr,
                                          int lane, int b, int k, int ticket, uint32_t epoch) {
    const MoeGeom &g = p.g;
    const int q = blockIdx.x % g.P;
    const int gblk = q * g.RB + b;
    const int64_t left = g.Tq - static_cast<int64_t>(b) * BM;
    const int nrows = static_cast<int>(left < BM ? left : BM);
    int32_t *s_pos = reinterpret_cast<int32_t *>(pscr);
    int32_t *s_ci = s_pos + BM;
    __syncwarp();  // orders lane 0's acquire of the plan before the other lanes' reads
    int slot = -1;
    if (lane == 0) slot = trace_open(p, st, K_DISPATCH, ticket, p.trace ? static_cast<int64_t>(globaltimer()) : 0);
    const int64_t tok0 = static_cast<int64_t>(q) * g.Tq + static_cast<int64_t>(b) * BM;
    for (int r = lane; r < nrows; r += 32) {
        const int64_t t = tok0 + r;
        const int e = ldcg_i32(&p.topk_idx[t * g.K + k]);
        const int pos = ldcg_i32(&p.base[gblk * g.E + e]) + ldcg_i32(&p.rank_in_blk[t * g.K + k]);
        const int oe = ldcg_i32(&p.offsets[e]);
        p.pos_out[t * g.K + k] = g.mx ? pos - oe + ldcg_i32(&p.offl[e]) : pos;  // reported without padding
        p.inv_pos[pos] = static_cast<int32_t>(t * g.K + k);
        s_pos[r] = pos;
        s_ci[r] = e * g.MAXRB + (pos - oe) / BM;
    }
    bool qok = true;
    if (g.mx) {
        if (lane == 0) qok = wait_flag_eq(p.ws, &p.quant_cnt[gblk], static_cast<uint32_t>(nrows), p.wait_limit_ns, ticket);
        qok = __shfl_sync(0xFFFFFFFFu, qok ? 1 : 0, 0) != 0;
        __syncwarp();
        if (qok) {
            // the block's scale words into the receive rows' tiled atoms: word c
            // of a row (K-blocks 4c .. 4c+3) goes to atom (pos / 128, c) at the
            // row's place inside it; 32 rows in flight per lane, one row's words
            // across the lanes (coalesced loads)
            const int W = static_cast<int>(g.H / 128);  // scale words per row
            const uint32_t *xs = reinterpret_cast<const uint32_t *>(p.xs) + tok0 * W;
            constexpr int R = 32;
            for (int r0 = 0; r0 < nrows; r0 += R) {
                for (int c0 = 0; c0 < W; c0 += 32) {
                    const int c = c0 + lane;
                    uint32_t v[R];
#pragma unroll
                    for (int u = 0; u < R; ++u)
                        if (r0 + u < nrows && c < W) v[u] = __ldcg(xs + (r0 + u) * W + c);
#pragma unroll
                    for (int u = 0; u < R; ++u)
                        if (r0 + u < nrows && c < W) {
                            const int pos = s_pos[r0 + u];
                            const int64_t off = (static_cast<int64_t>(pos >> 7) * W + c) * 512 + (pos & 31) * 16 +
                                                ((pos >> 5) & 3) * 4;
                            *reinterpret_cast<uint32_t *>(p.recv_sf + off) = v[u];
                        }
                }
            }
            __threadfence();
        }
    }
    __syncwarp();
    if (lane == 0) {
        bool ok = qok && drain_pipeline(p, sm, st.ps);
        const uint32_t rbytes = static_cast<uint32_t>(g.mx ? g.H : g.H * 2);
        const int per = STAGE_BYTES / static_cast<int>(rbytes);
        const int nch = (nrows + per - 1) / per;
        const uint8_t *src0 = g.mx ? p.xq + tok0 * g.H
                                   : reinterpret_cast<const uint8_t *>(p.x[q] + static_cast<int64_t>(b) * BM * g.H);
        uint8_t *recv = g.mx ? p.recv8 : reinterpret_cast<uint8_t *>(p.recv);
        auto issue = [&](int c) {
            const int bi = c % NSTAGE;
            const int r0 = c * per;
            const int n = (nrows - r0) < per ? (nrows - r0) : per;
            mbar_arrive_expect_tx(&sm.cbar[bi], n * rbytes);
            for (int i = 0; i < n; ++i)
                bulk_g2s(sm.stages + bi * STAGE_BYTES + i * rbytes, src0 + static_cast<int64_t>(r0 + i) * rbytes,
                         rbytes, &sm.cbar[bi]);
        };
        for (int c = 0; ok && c < nch && c < NSTAGE; ++c) issue(c);
        for (int c = 0; ok && c < nch; ++c) {
            const int bi = c % NSTAGE;
            if (!mbar_wait(&sm.cbar[bi], (st.cphase >> bi) & 1u, PIPE_LIMIT_NS)) {
                set_error(p.ws, KOSMOS_ERR_DEVICE, ticket);
                ok = false;
                break;
            }
            st.cphase ^= (1u << bi);
            const int r0 = c * per;
            const int n = (nrows - r0) < per ? (nrows - r0) : per;
            for (int i = 0; i < n; ++i)
                bulk_s2g(recv + static_cast<int64_t>(s_pos[r0 + i]) * rbytes, sm.stages + bi * STAGE_BYTES + i * rbytes,
                         rbytes);
            bulk_commit();
            if (c >= 1 && c - 1 + NSTAGE < nch) {
                bulk_wait_read<1>();
                issue(c - 1 + NSTAGE);
            }
        }
        bulk_wait<0>();
        fence_proxy_async_global();
        __threadfence();  // orders the row copies before the relaxed arrival adds below
        const bool drop = (p.inject & KOSMOS_INJECT_DROP_DISPATCH) && static_cast<int64_t>(p.inject >> 32) == ticket;
        if (ok && !drop)
            for (int r = 0; r < nrows; ++r) red_relaxed_add_gpu(&p.disp_cnt[s_ci[r]], 1u);
        if (TraceRec *rec = trace_rec(p.trace, blockIdx.x, slot)) rec->t_done = static_cast<int64_t>(globaltimer());
    }
    __syncwarp();
    return st;
}

__device__ __forceinline__ void moe_producer(const MoeParams &p, const Smem &sm, uint8_t *pscr, uint8_t *sf,
                                             uint32_t epoch, int lane) {
    MoeProdState st;
    st.sf = sf;
    // producer scratch: [0, 1 KB) dispatch rows, then the plan table (3 Eq + 1 words <= 3 KB)
    st.us = reinterpret_cast<int32_t *>(pscr + 1024);
    st.off = st.us + p.g.Eq + 1;
    st.cnt = st.off + p.g.Eq;
    while (true) {
        int act = ACT_NONE, v0 = 0, v1 = 0, v2 = 0;
        if (lane == 0) act = moe_decide(p, sm, st, epoch, v0, v1, v2);
        act = __shfl_sync(0xFFFFFFFFu, act, 0);
        v0 = __shfl_sync(0xFFFFFFFFu, v0, 0);
        v1 = __shfl_sync(0xFFFFFFFFu, v1, 0);
        v2 = __shfl_sync(0xFFFFFFFFu, v2, 0);
        if (act == ACT_EXIT) break;
        if (act == ACT_PLAN) load_plan_table(p, st, lane);
        if (act == ACT_DISPATCH) st = moe_dispatch(p, sm, st, pscr, lane, v0, v1, v2, epoch);
    }
    if (lane == 0) {
        SchedEntry done;
        fill_entry(done, K_DONE, 0, 0, 0, 0, -1, -1);
        ring_push(sm, st.rs, done, p.ws);
    }
}

// ---------------------------------------------------------------- epilogue (warps 2-5)
// ROUTE epilogue for one block of 128 tokens (one token per thread).
__device__ __noinline__ void moe_route_epilogue(const MoeParams &p, const SchedEntry &e, uint32_t taddr, int row,
                                                int et, uint8_t *escr, uint32_t epoch) {
    const MoeGeom &g = p.g;
    const int q = e.a, b = e.b, gblk = e.c;
    const int K = g.K, E = g.E;
    const int64_t tl = static_cast<int64_t>(b) * BM + row;
    const bool valid = tl < g.Tq;
    const int64_t t = static_cast<int64_t>(q) * g.Tq + (valid ? tl : 0);
    // Top-k by k rounds of selection: round s takes the largest logit not
    // taken yet, ties to the lower expert (the scan runs in ascending expert
    // order and only a strictly larger value replaces the best so far).
    // Round 0 also writes the logits out.  The logits are re-read from TMEM
    // in every round, which keeps the code and the registers small.
    float tv[MOE_MAXK];
    int ti[MOE_MAXK];
    uint32_t taken[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};  // one bit per expert (E <= 256)
#pragma unroll 1
    for (int s = 0; s < K; ++s) {
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
#pragma unroll 1
        for (int ch = 0; ch < E / 32; ++ch) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + ch * 32, r);
            tmem_ld_wait();
            if (s == 0 && valid) {
                float4 *dump = reinterpret_cast<float4 *>(p.logits + t * E + ch * 32);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    dump[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                          __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            }
            uint32_t tk = 0u;
#pragma unroll
            for (int w = 0; w < 8; ++w)
                if (w == ch) tk = taken[w];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float l = __uint_as_float(r[j]);
                if (!((tk >> j) & 1u) && l > bv) { bv = l; bi = ch * 32 + j; }
            }
        }
#pragma unroll
        for (int w = 0; w < 8; ++w)
            if (w == (bi >> 5)) taken[w] |= 1u << (bi & 31);
#pragma unroll
        for (int u = 0; u < MOE_MAXK; ++u)
            if (u == s) { tv[u] = bv; ti[u] = bi; }
    }
    const float lmax = tv[0];
    // softmax denominator over all experts (ascending expert order)
    float z = 0.f;
#pragma unroll 1
    for (int ch = 0; ch < E / 32; ++ch) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + ch * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) z += expf(__uint_as_float(r[j]) - lmax);
    }
    float pk[MOE_MAXK];
    float ps = 0.f;
#pragma unroll
    for (int s = 0; s < MOE_MAXK; ++s) {
        pk[s] = (s < K) ? expf(tv[s] - lmax) / z : 0.f;
        if (s < K) ps += pk[s];
    }
    // Rank of each slot among the block's tokens routed to the same expert:
    // a 128-bit membership mask per expert (token r sets bit r), then a
    // popcount of the bits below this token.
    uint32_t *s_bits = reinterpret_cast<uint32_t *>(escr);         // [E][4]
    int32_t *s_hist = reinterpret_cast<int32_t *>(escr + 4096);    // [E]
    for (int i = et; i < E; i += NUM_EPI_THREADS) {
        s_hist[i] = 0;
        s_bits[4 * i + 0] = s_bits[4 * i + 1] = s_bits[4 * i + 2] = s_bits[4 * i + 3] = 0u;
    }
    named_bar_sync(1, NUM_EPI_THREADS);
#pragma unroll
    for (int s = 0; s < MOE_MAXK; ++s) {
        if (s < K && valid) {
            p.topk_idx[t * K + s] = ti[s];
            p.topk_gate[t * K + s] = pk[s] / ps;
            atomicOr(&s_bits[4 * ti[s] + (row >> 5)], 1u << (row & 31));
            atomicAdd(&s_hist[ti[s]], 1);
        }
    }
    named_bar_sync(1, NUM_EPI_THREADS);
    if (valid) {
#pragma unroll
        for (int s = 0; s < MOE_MAXK; ++s) {
            if (s < K) {
                const uint32_t *b4 = s_bits + 4 * ti[s];
                int rk = 0;
                for (int w = 0; w < (row >> 5); ++w) rk += __popc(b4[w]);
                rk += __popc(b4[row >> 5] & ((1u << (row & 31)) - 1u));
                p.rank_in_blk[t * K + s] = rk;
            }
        }
    }
    named_bar_sync(1, NUM_EPI_THREADS);
    for (int i = et; i < E; i += NUM_EPI_THREADS) p.blk_counts[gblk * E + i] = s_hist[i];
    __threadfence();
    named_bar_sync(1, NUM_EPI_THREADS);
    int32_t *s_last = reinterpret_cast<int32_t *>(escr + 8188);
    if (et == 0) *s_last = (atom_add_acqrel_gpu(p.route_done, 1u) == static_cast<uint32_t>(g.NB - 1)) ? 1 : 0;
    named_bar_sync(1, NUM_EPI_THREADS);
    if (*s_last == 0) return;
    // PLAN: every route block has published its counts
    __threadfence();
    int32_t *s_cnt = reinterpret_cast<int32_t *>(escr + 5120);
    int32_t *s_off = reinterpret_cast<int32_t *>(escr + 6144);
    for (int i = et; i < E; i += NUM_EPI_THREADS) {
        int c = 0;
#pragma unroll 8
        for (int gb = 0; gb < g.NB; ++gb) c += ldcg_i32(&p.blk_counts[gb * E + i]);
        s_cnt[i] = c;
        p.counts[i] = c;
        p.counts_out[i] = c;
    }
    named_bar_sync(1, NUM_EPI_THREADS);
    // exclusive prefix sums by warp scans (a serial loop interleaving shared
    // and global accesses cost tens of microseconds here): warp 0 scans the
    // expert counts into the receive offsets, warps 1.. scan each rank's
    // row-block units
    int32_t *s_us = reinterpret_cast<int32_t *>(escr);           // [P][Eq + 1] <= 264 words, over s_bits (done with)
    int32_t *s_offl = reinterpret_cast<int32_t *>(escr + 2048);  // [E + 1], MXFP8 only, over s_bits
    const int ew = et / 32, lane = et % 32;
    if (ew == 0) {
        if (g.mx) {
            // receive offsets without padding (reported), and with every expert
            // starting on a 128-row boundary (the layout of the buffers)
            const int tl = warp_excl_scan(s_cnt, s_offl, E, lane, 0);
            if (lane == 0) s_offl[E] = tl;
            const int tu = warp_excl_scan(s_cnt, s_off, E, lane, BM);
            __syncwarp();
            for (int i = lane; i < E; i += 32) s_off[i] *= BM;
            if (lane == 0) s_off[E] = tu * BM;
        } else {
            const int total = warp_excl_scan(s_cnt, s_off, E, lane, 0);
            if (lane == 0) s_off[E] = total;
        }
    } else {
        for (int qq = ew - 1; qq < g.P; qq += NUM_EPI_THREADS / 32 - 1) {
            const int total = warp_excl_scan(s_cnt + qq * g.Eq, s_us + qq * (g.Eq + 1), g.Eq, lane, BM);
            if (lane == 0) s_us[qq * (g.Eq + 1) + g.Eq] = total;
        }
    }
    named_bar_sync(1, NUM_EPI_THREADS);
    for (int i = et; i <= E; i += NUM_EPI_THREADS) {
        p.offsets[i] = s_off[i];
        p.offl[i] = g.mx ? s_offl[i] : s_off[i];
    }
    for (int i = et; i < g.P * (g.Eq + 1); i += NUM_EPI_THREADS) p.unit_start[i] = s_us[i];
    for (int i = et; i < E; i += NUM_EPI_THREADS) {
        int run = s_off[i];
#pragma unroll 8
        for (int gb = 0; gb < g.NB; ++gb) {
            p.base[gb * E + i] = run;
            run += ldcg_i32(&p.blk_counts[gb * E + i]);
        }
    }
    __threadfence();
    named_bar_sync(1, NUM_EPI_THREADS);
    if (et == 0) st_release_gpu(&p.ws->aux[1], epoch + 1u);
}


// Copies the dn-th 256-column slice of each row of one unit back to the
// source slot[t][k] (warp w: rows 32w..32w+31, lane: 16 bytes of the slice),
// then counts the arrivals per (token block, dn); the arrival that completes a
// block queues its FOLD on the block's rank.
__device__ __noinline__ void moe_push(const MoeParams &p, const SchedEntry &e, int ew, int lane, uint32_t epoch) {
    const MoeGeom &g = p.g;
    const int dn = e.c;
    const int row0 = e.x0, rows = e.x1;
    const __nv_bfloat16 *srcb = p.identity ? p.recv : p.ybuf;
    const int rbase = ew * 32;
    const int my = rbase + lane;                       // the row this lane accounts for
    const int32_t my_sl = (my < rows) ? ldcg_i32(&p.inv_pos[row0 + my]) : -1;
    const int n = (rows - rbase) < 32 ? (rows - rbase) : 32;
    constexpr int RU = 16;
    for (int i0 = 0; i0 < n; i0 += RU) {
        int32_t sl[RU];
        uint4 v[RU];
#pragma unroll
        for (int i = 0; i < RU; ++i) sl[i] = __shfl_sync(0xFFFFFFFFu, my_sl, (i0 + i) & 31);
#pragma unroll
        for (int i = 0; i < RU; ++i)
            if (i0 + i < n)
                v[i] = ldcg_u4(srcb + static_cast<int64_t>(row0 + rbase + i0 + i) * g.H + dn * BN + lane * 8);
#pragma unroll
        for (int i = 0; i < RU; ++i)
            if (i0 + i < n)
                *reinterpret_cast<uint4 *>(p.slot + static_cast<int64_t>(sl[i]) * g.H + dn * BN + lane * 8) = v[i];
    }
    __threadfence();
    __syncwarp();
    // one release-add per distinct token block among this warp's rows
    int gb = -1;
    uint32_t target = 0;
    if (my_sl >= 0) {
        const int64_t t = my_sl / g.K;
        const int qs = static_cast<int>(t / g.Tq);
        const int bq = static_cast<int>((t - static_cast<int64_t>(qs) * g.Tq) / BM);
        gb = qs * g.RB + bq;
        const int64_t left = g.Tq - static_cast<int64_t>(bq) * BM;
        target = static_cast<uint32_t>((left < BM ? left : BM) * g.K);
    }
    const uint32_t grp = __match_any_sync(0xFFFFFFFFu, gb);
    if (gb >= 0 && (__ffs(grp) - 1) == lane) {
        const uint32_t cnt = __popc(grp);
        if (atom_add_acqrel_gpu(&p.fold_cnt[gb * g.ND + dn], cnt) + cnt == target) {
            const int qs = gb / g.RB;
            queue_put(&p.qctl[4 * qs + 2], p.fold_items + qs * g.fold_cap, p.fold_flags + qs * g.fold_cap, g.fold_cap,
                      gb | (dn << 16), epoch, p.ws);
        }
    }
    __syncwarp();
}

// out[t] = sum_k gate[t][k] * slot[t][k] (fp32 multiply, then add, k in
// emission order), one rounding to bf16.  The slot rows arrive through the
// stage ring, fold_tps tokens per stage; thread et takes token et / 16 (and
// every 8th after it) and 16 of the 256 columns.  Returns false after a
// device error.
__device__ __noinline__ bool moe_fold(const MoeParams &p, const Smem &sm, PipeState &ps, const SchedEntry &e, int et,
                                      uint8_t *escr) {
    const MoeGeom &g = p.g;
    const int gb = e.a, dn = e.c;
    const int q = gb / g.RB, b = gb % g.RB;
    const int K = g.K;
    const int64_t left = g.Tq - static_cast<int64_t>(b) * BM;
    const int ntok = static_cast<int>(left < BM ? left : BM);
    const int64_t t0 = static_cast<int64_t>(q) * g.Tq + static_cast<int64_t>(b) * BM;
    // the block's gates, once
    float *s_gate = reinterpret_cast<float *>(escr);  // [BM * K] <= 4 KB
    for (int i = et; i < ntok * K; i += NUM_EPI_THREADS) s_gate[i] = ldcg_f32(&p.topk_gate[t0 * K + i]);
    named_bar_sync(1, NUM_EPI_THREADS);
    const int c0 = (et & 15) * 16;
    for (int s = 0; s < e.nstage; ++s) {
        // a thread whose wait runs out skips the stage and still takes its
        // barrier, which makes the decision to stop for all threads
        const bool ok = mbar_wait(&sm.full[ps.stage], ps.phase, PIPE_LIMIT_NS);
        if (!ok) set_error(p.ws, KOSMOS_ERR_DEVICE, -9);
        const uint8_t *buf = sm.stages + ps.stage * STAGE_BYTES;
        for (int u = et >> 4; ok && u < p.fold_tps; u += NUM_EPI_THREADS / 16) {
            const int r = s * p.fold_tps + u;  // token within the block
            if (r >= ntok) break;
            float acc[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = 0.f;
            for (int k = 0; k < K; ++k) {
                const float gk = s_gate[r * K + k];
                const uint4 *src = reinterpret_cast<const uint4 *>(buf + ((u * K + k) * BN + c0) * 2);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 v = src[h];
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[h * 8 + 2 * j] = __fadd_rn(acc[h * 8 + 2 * j], __fmul_rn(gk, __uint_as_float(w[j] << 16)));
                        acc[h * 8 + 2 * j + 1] =
                            __fadd_rn(acc[h * 8 + 2 * j + 1], __fmul_rn(gk, __uint_as_float(w[j] & 0xFFFF0000u)));
                    }
                }
            }
            uint4 o[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                o[h].x = pack_bf16x2(acc[h * 8 + 0], acc[h * 8 + 1]);
                o[h].y = pack_bf16x2(acc[h * 8 + 2], acc[h * 8 + 3]);
                o[h].z = pack_bf16x2(acc[h * 8 + 4], acc[h * 8 + 5]);
                o[h].w = pack_bf16x2(acc[h * 8 + 6], acc[h * 8 + 7]);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(p.y[q] + (static_cast<int64_t>(b) * BM + r) * g.H + dn * BN + c0);
            dst[0] = o[0];
            dst[1] = o[1];
        }
        if (!named_bar_and(1, NUM_EPI_THREADS, ok)) return false;
        if (et == 0) mbar_arrive(&sm.empty[ps.stage]);
        ps.advance();
    }
    return true;
}

// QUANT(j): the entry's bf16 token rows arrive through the stage ring; each
// thread quantises 32-element blocks (E4M3 bytes to xq, the E8M0 byte to the
// row-major xs), then the block's quantised-row counter is released.
__device__ __noinline__ bool moe_quant(const MoeParams &p, const Smem &sm, PipeState &ps, const SchedEntry &e,
                                       int et) {
    const MoeGeom &g = p.g;
    const int q = e.a, j = e.b, rows = e.c;
    const int64_t t0 = static_cast<int64_t>(q) * g.Tq + static_cast<int64_t>(j) * MOE_QR;
    const int rbytes = static_cast<int>(g.H * 2);
    const int rps = STAGE_BYTES / rbytes;
    const int HB = static_cast<int>(g.H / 32);
    for (int s = 0; s < e.nstage; ++s) {
        const bool ok = mbar_wait(&sm.full[ps.stage], ps.phase, PIPE_LIMIT_NS);
        if (!ok) set_error(p.ws, KOSMOS_ERR_DEVICE, -13);
        const uint8_t *buf = sm.stages + ps.stage * STAGE_BYTES;
        const int n = (rows - s * rps) < rps ? (rows - s * rps) : rps;
        for (int bi = et; ok && bi < n * HB; bi += NUM_EPI_THREADS) {
            const int r = bi / HB, kb = bi % HB;
            const uint4 *src = reinterpret_cast<const uint4 *>(buf + r * rbytes + kb * 64);
            float v[32];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const uint4 w4 = src[h];
                const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[h * 8 + 2 * i] = __uint_as_float(w[i] << 16);
                    v[h * 8 + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
                }
            }
            uint32_t o[8];
            const uint32_t sc = mx_quant32(v, o);
            const int64_t t = t0 + static_cast<int64_t>(s) * rps + r;
            uint4 *dst = reinterpret_cast<uint4 *>(p.xq + t * g.H + kb * 32);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
            p.xs[t * HB + kb] = static_cast<uint8_t>(sc);
        }
        if (!named_bar_and(1, NUM_EPI_THREADS, ok)) return false;  // one decision for all threads
        if (et == 0) mbar_arrive(&sm.empty[ps.stage]);
        ps.advance();
    }
    fence_proxy_async_global();  // xq: generic stores, copied by DISPATCH's bulk copies
    __threadfence();
    named_bar_sync(1, NUM_EPI_THREADS);
    if (et == 0) red_release_add_gpu(&p.quant_cnt[q * g.RB + (j * MOE_QR) / BM], static_cast<uint32_t>(rows));
    return true;
}

__device__ __forceinline__ void moe_epilogue(const MoeParams &p, const Smem &sm, uint32_t tmem_base, uint8_t *escr,
                                             uint8_t *stg,
                                             int warp, int lane, uint32_t epoch) {
    const MoeGeom &g = p.g;
    const int grp = warp & 3;
    const int row = grp * 32 + lane;
    const int ew = warp - 2;
    const int et = ew * 32 + lane;
    RingState rs;
    PipeState ps;  // stages of the ring: MMA entries are skipped, FOLD and QUANT stages consumed here
    uint32_t acc = 0, acc_phase = 0;
    const uint32_t nacc = g.mx ? 1u : 2u;  // MXFP8: the scale atoms take the second accumulator's columns
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
        if (is_mma_kind(e.kind)) {
            ps.advance(e.nstage);
            if (!mbar_wait(&sm.tfull[acc], acc_phase, PIPE_LIMIT_NS)) {
                set_error(p.ws, KOSMOS_ERR_DEVICE, -7);
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(grp * 32) << 16) + acc * BN;
            if (e.kind == K_ROUTE) {
                moe_route_epilogue(p, e, taddr, row, et, escr, epoch);
            } else if (e.kind == K_TILE_GU && g.mx) {
                // h = silu(gate) * up per 32 columns, quantised: E4M3 bytes to h8,
                // the four E8M0 bytes of this row (K-blocks 4c .. 4c+3) as one word
                const bool valid = row < e.x1;
                const int64_t r = e.x0 + row;  // e.x0 is a multiple of 128
                uint8_t *dst = p.h8 + r * g.I + e.c * 128;
                uint32_t sw = 0;
#pragma unroll 1
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t gr[32], ur[32];
                    tmem_ld_32x32b_x32(taddr + ch * 32, gr);
                    tmem_ld_32x32b_x32(taddr + 128 + ch * 32, ur);
                    tmem_ld_wait();
                    float hv[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) hv[j] = silu_f(__uint_as_float(gr[j])) * __uint_as_float(ur[j]);
                    uint32_t o[8];
                    sw |= mx_quant32(hv, o) << (8 * ch);
                    if (valid) {
                        uint4 *d = reinterpret_cast<uint4 *>(dst + ch * 32);
                        d[0] = make_uint4(o[0], o[1], o[2], o[3]);
                        d[1] = make_uint4(o[4], o[5], o[6], o[7]);
                    }
                }
                if (valid) *reinterpret_cast<uint32_t *>(p.h_sf + sf_tiled_offset(r, 4 * e.c, g.I / 32)) = sw;
            } else if (e.kind == K_TILE_GU) {
                // h = silu(gate) * up, and gate and up saved for the backward, as
                // bf16 rows of 128 columns; each 64-column block of each output
                // leaves through the lane transpose (whole 128-byte row segments
                // per store instruction), gate and up re-read from tensor memory
                const int rows_w = e.x1 - grp * 32 <= 0 ? 0 : (e.x1 - grp * 32 >= 32 ? 32 : e.x1 - grp * 32);
                const int64_t off = static_cast<int64_t>(e.x0 + (rows_w > 0 ? grp * 32 : 0)) * g.I + e.c * 128;
#pragma unroll 1
                for (int b = 0; b < 2; ++b) {
#pragma unroll
                    for (int gu = 0; gu < 2; ++gu) {  // gate, then up
                        uint32_t vk[32];
                        uint32_t r0[32], r1[32];
                        tmem_ld_32x32b_x32(taddr + gu * 128 + b * 64, r0);
                        tmem_ld_32x32b_x32(taddr + gu * 128 + b * 64 + 32, r1);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            vk[j] = pack_bf16x2(__uint_as_float(r0[2 * j]), __uint_as_float(r0[2 * j + 1]));
                            vk[16 + j] = pack_bf16x2(__uint_as_float(r1[2 * j]), __uint_as_float(r1[2 * j + 1]));
                        }
                        lane_transpose8_16B(vk, lane);
                        store_row_lines(vk, (gu == 0 ? p.gsave : p.usave) + off + b * 64, g.I, rows_w, 64, lane);
                    }
                    uint32_t hk[32];
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t gr[32], ur[32];
                        tmem_ld_32x32b_x32(taddr + b * 64 + hh * 32, gr);
                        tmem_ld_32x32b_x32(taddr + 128 + b * 64 + hh * 32, ur);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            hk[hh * 16 + j] =
                                pack_bf16x2(silu_f(__uint_as_float(gr[2 * j])) * __uint_as_float(ur[2 * j]),
                                            silu_f(__uint_as_float(gr[2 * j + 1])) * __uint_as_float(ur[2 * j + 1]));
                    }
                    lane_transpose8_16B(hk, lane);
                    store_row_lines(hk, p.h + off + b * 64, g.I, rows_w, 64, lane);
                }
            } else if (!g.mx && grp * 32 + 32 > e.x1) {  // K_TILE_D, bf16, a warp with rows past the
                // unit's end: plain stores of its real rows (in the bf16 layout the
                // next rows belong to the next expert; MXFP8 pads every expert to
                // whole 128-row blocks, never read)
                const bool valid = row < e.x1;
                __nv_bfloat16 *dst = p.ybuf + static_cast<int64_t>(e.x0 + (valid ? row : 0)) * g.H + e.c * BN;
#pragma unroll 1
                for (int ch = 0; ch < BN / 32; ++ch) tmem_row_chunk_to_bf16(taddr + ch * 32, valid, dst + ch * 32, 32);
            } else {  // K_TILE_D: 32 x 32 boxes through the warp's staging buffer
                // (64-byte swizzle: piece c of row r at c ^ ((r >> 1) & 3))
                const int swz = (lane >> 1) & 3;
                uint4 *srow = reinterpret_cast<uint4 *>(stg + lane * 64);
#pragma unroll 1
                for (int ch = 0; ch < BN / 32; ++ch) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + ch * 32, r);
                    tmem_ld_wait();
                    if (lane == 0) bulk_wait_read<0>();
                    __syncwarp();
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
                        tma_store_3d(&p.tmYbuf, stg, e.c * BN + ch * 32, e.x0 + grp * 32, 0);
                        bulk_commit();
                    }
                }
                if (lane == 0) {  // landed, and ordered before the PUSH release below
                    bulk_wait<0>();
                    fence_proxy_async_global();
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.tempty[acc]);
            if (++acc == nacc) { acc = 0; acc_phase ^= 1u; }
            if (e.kind == K_TILE_GU || e.kind == K_TILE_D) {
                __threadfence();
                named_bar_sync(1, NUM_EPI_THREADS);
                if (et == 0) {
                    if (e.kind == K_TILE_GU) {
                        red_release_add_gpu(&p.gu_cnt[e.a * g.MAXRB + e.b], 1u);
                    } else {
                        const int qe = e.a / g.Eq;
                        queue_put(&p.qctl[4 * qe + 0], p.push_items + qe * g.push_cap, p.push_flags + qe * g.push_cap,
                                  g.push_cap, push_code(e.a, e.b, e.c), epoch, p.ws);
                    }
                }
            }
        } else if (e.kind == K_PUSH) {
            moe_push(p, e, ew, lane, epoch);
        } else if (e.kind == K_FOLD) {
            if (!moe_fold(p, sm, ps, e, et, escr)) break;
        } else if (e.kind == K_QUANT) {
            if (!moe_quant(p, sm, ps, e, et)) break;
        }
        if (e.slot >= 0 && et == 0) {
            if (TraceRec *r = trace_rec(p.trace, blockIdx.x, e.slot)) r->t_done = static_cast<int64_t>(globaltimer());
        }
    }
}

// MMA warp (one thread): ROUTE entries as bf16 MMAs with N = E; GU / D tiles
// as bf16 MMAs into two alternating accumulators, or (MXFP8) as block-scaled
// MMAs into one accumulator with the stage's scale atoms copied to tensor
// memory columns 256 + 16 * stage.
__device__ __forceinline__ void moe_mma_loop(const MoeParams &p, const Smem &sm, const uint8_t *sf,
                                             uint32_t tmem_base) {
    constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, false, true);
    const bool mx = p.g.mx;
    const uint32_t nacc = mx ? 1u : 2u;
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
        if (!is_mma_kind(e.kind)) {
            ps.advance(e.nstage);
            continue;
        }
        const uint32_t idesc = (e.nmma > 0 && e.nmma < BN) ? idesc_bf16_f32(BM, e.nmma, false, true) : IDESC;
        const bool blk = mx && e.kind != K_ROUTE;
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
            if (blk) {
                mx_stage_mma(d_tmem, a_addr, b_addr, 16384, smem_u32(sf + ps.stage * MOE_SF_BYTES),
                             tmem_base + F_TMEM_SF + ps.stage * F_TMEM_SF_STRIDE, kb == 0);
            } else {
#pragma unroll
                for (int k = 0; k < BK / UMMA_K; ++k) {
                    const uint64_t ad = sdesc_sw128(a_addr + k * (UMMA_K * 2), 16, 1024);
                    const uint64_t bd = sdesc_sw128(b_addr + k * (UMMA_K * 128), 64 * 128, 1024);
                    mma_bf16_ss(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                }
            }
            mma_commit(&sm.empty[ps.stage]);
            ps.advance();
        }
        if (!ok) break;
        mma_commit(&sm.tfull[acc]);
        if (++acc == nacc) { acc = 0; acc_phase ^= 1u; }
    }
}

__global__ void __launch_bounds__(NUM_THREADS, 1) moe_fwd_kernel(const __grid_constant__ MoeParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const Smem sm = carve_smem(smem_raw);
    uint8_t *scratch = sm.stages + NSTAGE * STAGE_BYTES + SMEM_CTRL_BYTES;
    uint8_t *escr = scratch;          // epilogue: 8 KB
    uint8_t *pscr = scratch + 8192;   // producer: 4 KB
    uint8_t *sf = scratch + MOE_SCRATCH;  // MXFP8 scale atoms: NSTAGE x 1.5 KB
    uint8_t *stg = sf + NSTAGE * MOE_SF_BYTES;  // epilogue warps' D-tile store boxes: 4 x 2 KB
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t epoch = *reinterpret_cast<volatile uint32_t *>(&p.ws->epoch);
    engine_setup(sm, warp);
    const uint32_t tmem_base = *sm.tmem_slot;
    if (warp == 0) {
        moe_producer(p, sm, pscr, sf, epoch, lane);
    } else if (warp == 1) {
        if (lane == 0) moe_mma_loop(p, sm, sf, tmem_base);
    } else {
        moe_epilogue(p, sm, tmem_base, escr, stg + (warp - 2) * MOE_STG_BYTES, warp, lane, epoch);
    }
    engine_teardown(sm, warp, tmem_base);
    // The last CTA returns every counter to zero, then the rail tickets and epoch.
    __shared__ int s_last;
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = (atomicAdd(&p.ws->done_ctas, 1u) == gridDim.x - 1) ? 1 : 0;
    }
    __syncthreads();
    if (s_last && p.phase >= 1 && p.phase <= 4) {
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
            *reinterpret_cast<volatile uint32_t *>(&p.ws->aux[2]) = p.g.mx ? 0u : MOE_BF16_CTX;
            *reinterpret_cast<volatile uint32_t *>(&p.ws->done_ctas) = 0u;
            __threadfence();
            *reinterpret_cast<volatile uint32_t *>(&p.ws->epoch) = epoch + 1u;
            __threadfence();
        }
    }
}

size_t moe_workspace_bytes(int P, int64_t T, int64_t H, int E, int K, int64_t I, bool mx, bool trace) {
    return moe_ws_layout(moe_geom(P, T, H, E, K, I, mx), trace).total;
}

bool moe_debug_view(int what, int P, int64_t T, int64_t H, int E, int K, int64_t I, bool mx, void *ws, void **ptr,
                    int64_t *bytes) {
    const MoeGeom g = moe_geom(P, T, H, E, K, I, mx);
    const MoeWsLayout L = moe_ws_layout(g, what == 6);
    const size_t esz = mx ? 1 : 2;
    const size_t rows = mx ? static_cast<size_t>(g.rows_cap) : static_cast<size_t>(g.T * g.K);
    size_t off = 0, n = 0;
    switch (what) {
        case 0: off = L.logits; n = 4ull * g.T * g.E; break;
        case 1: off = L.recv; n = esz * rows * g.H; break;
        case 2: off = L.h; n = esz * rows * g.I; break;
        case 3: off = L.ybuf; n = 2ull * rows * g.H; break;
        case 4: off = L.slot; n = 2ull * g.T * g.K * g.H; break;
        case 5: off = L.offsets; n = 4ull * (g.E + 1); break;
        case 6: off = L.trace; n = static_cast<size_t>(MAX_CTAS) * TRACE_CAP * sizeof(TraceRec); break;
        case 7: if (!mx) return false; off = L.recv_sf; n = static_cast<size_t>(g.rows_cap * g.H / 32); break;
        case 8: if (!mx) return false; off = L.xq; n = static_cast<size_t>(g.T * g.H); break;
        case 9: if (!mx) return false; off = L.xs; n = static_cast<size_t>(g.T * g.H / 32); break;
        default: return false;
    }
    *ptr = static_cast<uint8_t *>(ws) + off;
    *bytes = static_cast<int64_t>(n);
    return true;
}

kosmos_status launch_moe_fwd(const MoeLaunch &Lc, cudaStream_t stream) {
    MoeParams p;
    memset(&p, 0, sizeof(p));
    const bool mx = Lc.dtype == KOSMOS_MXFP8_E4M3;
    p.g = moe_geom(Lc.P, Lc.T, Lc.H, Lc.E, Lc.K, Lc.I, mx);
    const MoeGeom &g = p.g;
    const MoeWsLayout L = moe_ws_layout(g, Lc.trace != 0);
    uint8_t *ws = static_cast<uint8_t *>(Lc.ws);
    p.ws = reinterpret_cast<WsHeader *>(ws);
    p.ctr = ws + L.ctr;
    p.ctr_bytes = static_cast<int>(L.ctr_bytes);
    p.disp_cnt = reinterpret_cast<uint32_t *>(ws + L.disp_cnt);
    p.gu_cnt = reinterpret_cast<uint32_t *>(ws + L.gu_cnt);
    p.fold_cnt = reinterpret_cast<uint32_t *>(ws + L.fold_cnt);
    p.qctl = reinterpret_cast<uint32_t *>(ws + L.qctl);
    p.route_done = reinterpret_cast<uint32_t *>(ws + L.route_done);
    p.blk_counts = reinterpret_cast<int32_t *>(ws + L.blk_counts);
    p.rank_in_blk = reinterpret_cast<int32_t *>(ws + L.rank_in_blk);
    p.base = reinterpret_cast<int32_t *>(ws + L.base);
    p.offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    p.offl = reinterpret_cast<int32_t *>(ws + L.offl);
    p.quant_cnt = reinterpret_cast<uint32_t *>(ws + L.quant_cnt);
    if (mx) {
        p.xq = ws + L.xq;
        p.xs = ws + L.xs;
        p.recv8 = ws + L.recv;
        p.recv_sf = ws + L.recv_sf;
        p.h8 = ws + L.h;
        p.h_sf = ws + L.h_sf;
    }
    p.counts = reinterpret_cast<int32_t *>(ws + L.counts);
    p.unit_start = reinterpret_cast<int32_t *>(ws + L.unit_start);
    p.inv_pos = reinterpret_cast<int32_t *>(ws + L.inv_pos);
    p.push_items = reinterpret_cast<int32_t *>(ws + L.push_items);
    p.push_flags = reinterpret_cast<uint32_t *>(ws + L.push_flags);
    p.fold_items = reinterpret_cast<int32_t *>(ws + L.fold_items);
    p.fold_flags = reinterpret_cast<uint32_t *>(ws + L.fold_flags);
    p.logits = reinterpret_cast<float *>(ws + L.logits);
    p.recv = reinterpret_cast<__nv_bfloat16 *>(ws + L.recv);
    p.h = reinterpret_cast<__nv_bfloat16 *>(ws + L.h);
    p.ybuf = reinterpret_cast<__nv_bfloat16 *>(ws + L.ybuf);
    p.slot = reinterpret_cast<__nv_bfloat16 *>(ws + L.slot);
    if (!mx) {
        p.gsave = reinterpret_cast<__nv_bfloat16 *>(ws + L.gsave);
        p.usave = reinterpret_cast<__nv_bfloat16 *>(ws + L.usave);
    }
    p.trace = Lc.trace ? reinterpret_cast<TraceRec *>(ws + L.trace) : nullptr;
    p.topk_idx = Lc.topk_idx;
    p.topk_gate = Lc.topk_gate;
    p.counts_out = Lc.counts;
    p.pos_out = Lc.pos;
    p.identity = (Lc.inject & KOSMOS_INJECT_IDENTITY_EXPERTS) ? 1 : 0;
    p.wait_limit_ns = Lc.wait_limit_ns;
    p.inject = Lc.inject;
    const uint64_t H = static_cast<uint64_t>(g.H), I = static_cast<uint64_t>(g.I), E = static_cast<uint64_t>(g.E);
    const uint64_t Eq = static_cast<uint64_t>(g.Eq), Tq = static_cast<uint64_t>(g.Tq);
    const uint64_t RC = static_cast<uint64_t>(g.rows_cap);
    for (int q = 0; q < g.P; ++q) {
        p.x[q] = static_cast<const __nv_bfloat16 *>(Lc.x[q]);
        p.y[q] = static_cast<__nv_bfloat16 *>(Lc.y[q]);
        {
            const uint64_t dims[2] = {H, Tq};
            const uint64_t st[1] = {H * 2};
            const uint32_t box[2] = {BK, BM};
            if (!encode_tmap(&p.tmX[q], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(Lc.x[q]), dims, st, box,
                             CU_TENSOR_MAP_SWIZZLE_128B))
                return KOSMOS_ERR_CUDA;
        }
        // weights: bf16 boxes of 64 columns x 64 K, or E4M3 boxes of 128 x 128
        const CUtensorMapDataType wdt = mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const uint64_t esz = mx ? 1 : 2;
        const uint32_t bw = mx ? 128u : 64u, bk = mx ? static_cast<uint32_t>(FBK) : static_cast<uint32_t>(BK);
        {
            const uint64_t dims[3] = {I, H, Eq};
            const uint64_t st[2] = {I * esz, H * I * esz};
            const uint32_t box[3] = {bw, bk, 1};
            if (!encode_tmap(&p.tmWg[q], wdt, 3, const_cast<void *>(Lc.wg[q]), dims, st, box,
                             CU_TENSOR_MAP_SWIZZLE_128B) ||
                !encode_tmap(&p.tmWu[q], wdt, 3, const_cast<void *>(Lc.wu[q]), dims, st, box,
                             CU_TENSOR_MAP_SWIZZLE_128B))
                return KOSMOS_ERR_CUDA;
        }
        {
            const uint64_t dims[3] = {H, I, Eq};
            const uint64_t st[2] = {H * esz, H * I * esz};
            const uint32_t box[3] = {bw, bk, 1};
            if (!encode_tmap(&p.tmWd[q], wdt, 3, const_cast<void *>(Lc.wd[q]), dims, st, box,
                             CU_TENSOR_MAP_SWIZZLE_128B))
                return KOSMOS_ERR_CUDA;
        }
        if (mx) {
            // tiled weight scales, experts one after the other: I*H/32 bytes each
            const uint64_t atoms = Eq * I * H / 32 / 512;
            if (!encode_sf_tmap(&p.tmSWg[q], const_cast<void *>(Lc.wgs[q]), atoms) ||
                !encode_sf_tmap(&p.tmSWu[q], const_cast<void *>(Lc.wus[q]), atoms) ||
                !encode_sf_tmap(&p.tmSWd[q], const_cast<void *>(Lc.wds[q]), atoms))
                return KOSMOS_ERR_CUDA;
        }
    }
    {
        const uint64_t dims[2] = {E, H};
        const uint64_t st[1] = {E * 2};
        const uint32_t box[2] = {64, BK};
        if (!encode_tmap(&p.tmWr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(Lc.wr), dims, st, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return KOSMOS_ERR_CUDA;
    }
    {
        // receive rows and h: bf16 boxes of 64 K x 128 rows, or E4M3 boxes of 128 x 128
        const CUtensorMapDataType adt = mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const uint64_t esz = mx ? 1 : 2;
        const uint32_t bk = mx ? static_cast<uint32_t>(FBK) : static_cast<uint32_t>(BK);
        const uint64_t dr[2] = {H, RC}, sr[1] = {H * esz};
        const uint64_t dh[2] = {I, RC}, sh[1] = {I * esz};
        const uint32_t box[2] = {bk, BM};
        if (!encode_tmap(&p.tmRecv, adt, 2, p.recv, dr, sr, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tmap(&p.tmH, adt, 2, p.h, dh, sh, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return KOSMOS_ERR_CUDA;
        if (mx) {
            if (!encode_sf_tmap(&p.tmSRecv, p.recv_sf, RC * H / 32 / 512) ||
                !encode_sf_tmap(&p.tmSH, p.h_sf, RC * I / 32 / 512))
                return KOSMOS_ERR_CUDA;
        }
    }
    {
        // D tile output rows (ybuf), stored as 32 x 32 boxes
        const uint64_t dy[3] = {H, RC, 1}, sy[2] = {H * 2, H * 2 * RC};
        const uint32_t ybox[3] = {32, 32, 1};
        if (!encode_tmap(&p.tmYbuf, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.ybuf, dy, sy, ybox,
                         CU_TENSOR_MAP_SWIZZLE_64B))
            return KOSMOS_ERR_CUDA;
    }
    {
        // FOLD: fold_tps tokens x K slot rows x 256 columns per stage (<= 32 KB)
        p.fold_tps = 64 / g.K;
        const uint64_t dims[2] = {static_cast<uint64_t>(g.H), static_cast<uint64_t>(g.T * g.K)};
        const uint64_t st[1] = {static_cast<uint64_t>(g.H) * 2};
        const uint32_t box[2] = {BN, static_cast<uint32_t>(p.fold_tps * g.K)};
        if (!encode_tmap(&p.tmSlot, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.slot, dims, st, box,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
            return KOSMOS_ERR_CUDA;
    }
    if (Lc.sched != KOSMOS_SCHED_UNFUSED)
        return launch_persistent(reinterpret_cast<const void *>(&moe_fwd_kernel), &p, Lc.grid, MOE_SMEM_BYTES, stream,
                                 Lc.plain_launch != 0);
    // unfused baseline: the same kernel once per phase, each launch running
    // only its phase's entries to completion before the next starts
    for (int ph = 1; ph <= 5; ++ph) {
        p.phase = ph;
        const kosmos_status st = launch_persistent(reinterpret_cast<const void *>(&moe_fwd_kernel), &p, Lc.grid,
                                                   MOE_SMEM_BYTES, stream, Lc.plain_launch != 0);
        if (st != KOSMOS_OK) return st;
    }
    return KOSMOS_OK;
}

}  // namespace kosmos
