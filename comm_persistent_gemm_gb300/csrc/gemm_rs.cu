// gemm_rs.cu -- GEMM + reduce-scatter as one self-scheduling persistent launch.
//
// Y = sum_r X_r . W_r, scattered as P row chunks (KOSMOS explainer, paragraph
// "Start with the problem": scatter and add the partial results).  All P
// emulated ranks run in one launch.  Rails:
//   tile rail    TILE(rank q, chunk, band, col), one rail for all ranks: the
//                partial X_q . W_q on one tile, rounded to bf16 into rank q's
//                partial buffer, then one release-increment of that output
//                tile's arrival counter; band order (band, rank, col, chunk)
//                or the row-order ablation (chunk, band, rank, col)
//                (explainer, "Role switching only works");
//   reduce rail  REDUCE(band, col) of rank r's own chunk, one per rank:
//                acquire counter == P arrivals, sum the P partials in rank
//                order 0..P-1 in fp32, round once to bf16 into y_chunks[r].
// CTA c reduces for rank c mod P.  Builders whose tile rail runs out join
// that rank's reduction (one-way, explainer "KOSMOS removes the manager").
// n_comm CTAs per rank are the rank's first reducers: with self-scheduling
// they build until the rank's next reduce entry has all its arrivals and
// then switch (data readiness, not a start-up split); in the fixed split
// they reduce from the start.
#include <cuda.h>
#include <cuda_runtime.h>

#include "mxfp8.cuh"
#include "launch.h"

namespace kosmos {

enum RsMode : int { RS_FUSED = 0, RS_TILES_ONLY = 1, RS_REDUCE_ONLY = 2 };

struct RsParams {
    CUtensorMap tmX[KOSMOS_MAX_P];  // X_r viewed [P chunks][mc][k]: dims {k, mc, P}, box {64, 128, 1}, 128B swizzle
    CUtensorMap tmW[KOSMOS_MAX_P];  // W_r: dims {n, k}, box {64, 64}, 128B swizzle
    CUtensorMap tmPart;             // partials [rank][chunk][mc][n]: dims {n, mc, P, P}, box {256, 8, 1, P}
    // MXFP8 (SM pairs): tmX/tmW hold E4M3 bytes (boxes {128, 128, 1} / {128, 128}) and these the
    // tiled scales, one 512-byte atom per box (encode_sf_tmap)
    CUtensorMap tmSX[KOSMOS_MAX_P]; // X_r scales: (m / 128) * nkb atoms
    CUtensorMap tmSW[KOSMOS_MAX_P]; // W_r scales: ceil(n / 128) * nkb atoms
    __nv_bfloat16 *part;            // [P ranks][m][n]
    __nv_bfloat16 *y[KOSMOS_MAX_P]; // chunk c: [mc][n]
    WsHeader *ws;
    uint32_t *arrive;               // [chunk][band][col] arrival counters
    TraceRec *trace;
    RsGeom g;
    int nkb;                        // K stages: k / 64 (bf16) or k / 128 (MXFP8)
    int sched;
    int n_red;
    int order;
    int mode;
    int pad;
    uint64_t wait_limit_ns;
    uint64_t inject;
    int64_t link_gbs;               // emulated link for other ranks' partial tiles; 0 = uncapped
};

// Bytes of partial tile (band, tcol) rows [r0, r0 + nr) that exist.
__device__ __forceinline__ uint64_t rs_tile_bytes(const RsParams &p, int64_t r0, int64_t nr, int tcol) {
    int64_t rows = p.g.mc - r0;
    rows = rows < 0 ? 0 : (rows > nr ? nr : rows);
    int64_t cols = p.g.n - static_cast<int64_t>(tcol) * BN;
    cols = cols > BN ? BN : cols;
    return static_cast<uint64_t>(rows * cols * 2);
}

// True when the next unclaimed entry of rank r's reduce rail has `need`
// arrivals (relaxed reads: a hint for the switch; the reducer acquires the
// counter itself before it reads the partials).
__device__ __forceinline__ bool rs_reduce_ready(const RsParams &p, int r, uint32_t need) {
    const uint32_t t = ld_relaxed_gpu(&p.ws->tickets[KOSMOS_MAX_P + r]);
    if (t >= static_cast<uint32_t>(p.g.n_reduce)) return false;
    int band, tcol;
    rs_decode_reduce(p.g, static_cast<int>(t), band, tcol);
    return ld_relaxed_gpu(&p.arrive[(static_cast<int64_t>(r) * p.g.bands + band) * p.g.tiles_n + tcol]) >= need;
}

__device__ __forceinline__ void rs_producer(const RsParams &p, const Smem &sm) {
    const int cta = blockIdx.x;
    const int P = p.g.P;
    const int rank = cta % P;
    const int local = cta / P;
    // first reducers: from the start in the fixed split, on the first ready entry when self-scheduled
    const bool first = p.mode == RS_FUSED && local < p.n_red;
    const bool on_ready = first && p.sched == KOSMOS_SCHED_SELF;
    bool reducer = (p.mode == RS_REDUCE_ONLY) || (first && !on_ready);
    PipeState ps;
    RingState rs;
    int nrec = 0;
    const uint32_t red_bytes = static_cast<uint32_t>(BN * RED_ROWS * 2 * P);
    while (true) {
        if (failed(p.ws)) break;
        if (!reducer && on_ready && rs_reduce_ready(p, rank, static_cast<uint32_t>(P))) reducer = true;
        if (!reducer) {
            const uint32_t t = atomicAdd(&p.ws->tickets[0], 1u);
            if (t < static_cast<uint32_t>(p.g.n_tile)) {
                int q, chunk, band, tcol;
                rs_decode_tile(p.g, p.order, static_cast<int>(t), q, chunk, band, tcol);
                int slot = -1;
                if (TraceRec *r = trace_rec(p.trace, cta, nrec)) {
                    const int64_t now = static_cast<int64_t>(globaltimer());
                    r->t_claim = now; r->t_ready = now; r->t_done = 0;
                    r->kind = K_TILE; r->ticket = static_cast<int32_t>(t); r->cta = cta;
                    slot = nrec;
                }
                ++nrec;
                SchedEntry e;
                e.kind = K_TILE; e.a = chunk; e.b = band; e.c = tcol; e.d = q; e.nstage = p.nkb;
                e.ticket = static_cast<int32_t>(t); e.slot = slot; e.nmma = 0; e.x0 = e.x1 = e.x2 = 0;
                if (!ring_push(sm, rs, e, p.ws)) break;
                bool ok = true;
                for (int kb = 0; kb < p.nkb; ++kb) {
                    if (!mbar_wait(&sm.empty[ps.stage], ps.phase ^ 1u, PIPE_LIMIT_NS)) {
                        set_error(p.ws, KOSMOS_ERR_DEVICE, t);
                        ok = false;
                        break;
                    }
                    uint8_t *sa = sm.stages + ps.stage * STAGE_BYTES;
                    uint8_t *sb = sa + A_STAGE_BYTES;
                    uint64_t *bar = &sm.full[ps.stage];
                    mbar_arrive_expect_tx(bar, STAGE_BYTES);
                    tma_load_3d(sa, &p.tmX[q], bar, kb * BK, band * BM, chunk);
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        tma_load_2d(sb + j * (64 * BK * 2), &p.tmW[q], bar, tcol * BN + j * 64, kb * BK);
                    ps.advance();
                }
                if (!ok) break;
                continue;
            }
            if (p.mode == RS_TILES_ONLY || p.sched == KOSMOS_SCHED_FIXED) break;
            reducer = true;  // one-way switch: builder -> reducer
        }
        const uint32_t t = atomicAdd(&p.ws->tickets[KOSMOS_MAX_P + rank], 1u);
        if (t >= static_cast<uint32_t>(p.g.n_reduce)) break;
        int band, tcol;
        rs_decode_reduce(p.g, static_cast<int>(t), band, tcol);
        const int64_t tc = p.trace ? static_cast<int64_t>(globaltimer()) : 0;
        if (p.mode == RS_FUSED) {
            uint32_t *ctr = &p.arrive[(static_cast<int64_t>(rank) * p.g.bands + band) * p.g.tiles_n + tcol];
            if (!wait_flag_eq(p.ws, ctr, static_cast<uint32_t>(P), p.wait_limit_ns,
                              (static_cast<int64_t>(1) << 40) | (static_cast<int64_t>(rank) << 32) | t))
                break;
            st_relaxed_gpu(ctr, 0u);  // sole consumer: return the counter to zero for the next call
        } else if (p.link_gbs > 0 && P > 1) {
            // unfused: the other ranks' partials of this tile cross the link now
            link_wait(link_reserve(p.ws, (P - 1) * rs_tile_bytes(p, static_cast<int64_t>(band) * BM, BM, tcol),
                                   p.link_gbs));
        }
        int slot = -1;
        if (TraceRec *r = trace_rec(p.trace, cta, nrec)) {
            r->t_claim = tc; r->t_ready = static_cast<int64_t>(globaltimer()); r->t_done = 0;
            r->kind = K_REDUCE; r->ticket = static_cast<int32_t>(t); r->cta = cta;
            slot = nrec;
        }
        ++nrec;
        const int64_t rows = (p.g.mc - static_cast<int64_t>(band) * BM) < BM ? (p.g.mc - static_cast<int64_t>(band) * BM) : BM;
        const int nsub = static_cast<int>(cdiv(rows, RED_ROWS));
        SchedEntry e;
        e.kind = K_REDUCE; e.a = rank; e.b = band; e.c = tcol; e.d = rank; e.nstage = nsub;
        e.ticket = static_cast<int32_t>(t); e.slot = slot; e.nmma = 0; e.x0 = e.x1 = e.x2 = 0;
        if (!ring_push(sm, rs, e, p.ws)) break;
        bool ok = true;
        for (int s = 0; s < nsub; ++s) {
            if (!mbar_wait(&sm.empty[ps.stage], ps.phase ^ 1u, PIPE_LIMIT_NS)) {
                set_error(p.ws, KOSMOS_ERR_DEVICE, t);
                ok = false;
                break;
            }
            uint64_t *bar = &sm.full[ps.stage];
            mbar_arrive_expect_tx(bar, red_bytes);
            tma_load_4d(sm.stages + ps.stage * STAGE_BYTES, &p.tmPart, bar, tcol * BN, band * BM + s * RED_ROWS,
                        rank, 0);
            ps.advance();
        }
        if (!ok) break;
    }
    SchedEntry done;
    done.kind = K_DONE; done.a = done.b = done.c = done.d = 0; done.nstage = 0; done.ticket = -1; done.slot = -1;
    done.nmma = 0; done.x0 = done.x1 = done.x2 = 0;
    ring_push(sm, rs, done, p.ws);
}

__device__ __forceinline__ void rs_epilogue(const RsParams &p, const Smem &sm, uint32_t tmem_base, int warp,
                                            int lane) {
    const int grp = warp & 3;              // TMEM lanes 32 grp .. 32 grp + 31 (accumulator rows)
    const int et = (warp - 2) * 32 + lane; // 0..127 within the epilogue warps
    const int P = p.g.P;
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
        if (e.kind == K_TILE) {
            if (!mbar_wait(&sm.tfull[acc], acc_phase, PIPE_LIMIT_NS)) {
                set_error(p.ws, KOSMOS_ERR_DEVICE, -7);
                break;
            }
            tc_fence_after();
            const int chunk = e.a, band = e.b, tcol = e.c, rank = e.d;
            const int64_t rw = static_cast<int64_t>(band) * BM + grp * 32;  // the warp's first row
            const int64_t rleft = p.g.mc - rw;
            const int rows_w = rleft <= 0 ? 0 : (rleft >= 32 ? 32 : static_cast<int>(rleft));
            __nv_bfloat16 *base = p.part + (static_cast<int64_t>(rank) * p.g.m + static_cast<int64_t>(chunk) * p.g.mc +
                                            (rows_w > 0 ? rw : 0)) * p.g.n;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(grp * 32) << 16) + acc * BN;
#pragma unroll 1
            for (int c64 = 0; c64 < BN / 64; ++c64) {
                const int64_t col0 = static_cast<int64_t>(tcol) * BN + c64 * 64;
                if (col0 >= p.g.n) break;
                const int64_t left = p.g.n - col0;
                tmem_rows64_to_bf16_lines(taddr + c64 * 64, base + col0, p.g.n, rows_w,
                                          left < 64 ? static_cast<int>(left) : 64, lane);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.tempty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            ps.advance(e.nstage);
            if (p.mode == RS_FUSED) {
                __threadfence();
                named_bar_sync(1, NUM_EPI_THREADS);
                const bool drop = (p.inject & KOSMOS_INJECT_DROP_PARTIAL) && static_cast<int>(p.inject >> 32) == rank;
                if (et == 0 && !drop) {
                    if (p.link_gbs > 0 && rank != chunk)  // another rank's partial crosses the link
                        link_wait(link_reserve(p.ws, rs_tile_bytes(p, static_cast<int64_t>(band) * BM, BM, tcol),
                                               p.link_gbs));
                    red_release_add_gpu(&p.arrive[(static_cast<int64_t>(chunk) * p.g.bands + band) * p.g.tiles_n + tcol], 1u);
                }
            }
            if (e.slot >= 0 && et == 0) {
                if (TraceRec *r = trace_rec(p.trace, blockIdx.x, e.slot)) r->t_done = static_cast<int64_t>(globaltimer());
            }
        } else if (e.kind == K_REDUCE) {
            const int chunk = e.a, band = e.b, tcol = e.c;
            const int cg = et & 31;           // 16-byte column group of the 256-wide tile
            const int64_t col = static_cast<int64_t>(tcol) * BN + cg * 8;
            bool ok = true;
            for (int s = 0; s < e.nstage; ++s) {
                // a thread whose wait runs out skips the stage and still takes
                // its barrier, which makes the decision to stop for all threads
                const bool got = mbar_wait(&sm.full[ps.stage], ps.phase, PIPE_LIMIT_NS);
                if (!got) set_error(p.ws, KOSMOS_ERR_DEVICE, -8);
                const uint8_t *buf = sm.stages + ps.stage * STAGE_BYTES;
#pragma unroll
                for (int rr = 0; got && rr < 2; ++rr) {
                    const int r8 = (et >> 5) * 2 + rr;  // row within the 8-row stage
                    float a[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) a[q] = 0.f;
                    for (int rk = 0; rk < P; ++rk) {    // fixed rank order 0..P-1
                        const uint4 v = *reinterpret_cast<const uint4 *>(buf + ((rk * RED_ROWS + r8) * BN + cg * 8) * 2);
                        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            a[2 * q] += __uint_as_float(w[q] << 16);
                            a[2 * q + 1] += __uint_as_float(w[q] & 0xFFFF0000u);
                        }
                    }
                    const int64_t grow = static_cast<int64_t>(band) * BM + s * RED_ROWS + r8;
                    if (grow < p.g.mc && col < p.g.n) {
                        uint4 o;
                        o.x = pack_bf16x2(a[0], a[1]);
                        o.y = pack_bf16x2(a[2], a[3]);
                        o.z = pack_bf16x2(a[4], a[5]);
                        o.w = pack_bf16x2(a[6], a[7]);
                        *reinterpret_cast<uint4 *>(p.y[chunk] + grow * p.g.n + col) = o;
                    }
                }
                if (!named_bar_and(1, NUM_EPI_THREADS, got)) {
                    ok = false;
                    break;
                }
                if (et == 0) mbar_arrive(&sm.empty[ps.stage]);
                ps.advance();
            }
            if (!ok) break;
            if (e.slot >= 0 && et == 0) {
                if (TraceRec *r = trace_rec(p.trace, blockIdx.x, e.slot)) r->t_done = static_cast<int64_t>(globaltimer());
            }
        } else {
            ps.advance(e.nstage);
        }
    }
}

__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_rs_kernel(const __grid_constant__ RsParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const Smem sm = carve_smem(smem_raw);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t epoch = *reinterpret_cast<volatile uint32_t *>(&p.ws->epoch);
    engine_setup(sm, warp);
    const uint32_t tmem_base = *sm.tmem_slot;
    if (warp == 0) {
        if (lane == 0) rs_producer(p, sm);
    } else if (warp == 1) {
        if (lane == 0) mma_loop(sm, tmem_base, p.ws);
    } else {
        rs_epilogue(p, sm, tmem_base, warp, lane);
    }
    engine_teardown(sm, warp, tmem_base);
    if (threadIdx.x == 0) engine_finish(p.ws, epoch, 2 * KOSMOS_MAX_P);
}

// ============================================================== SM-pair variant
// Builder pairs compute 256 x 256 partial tiles (bands of 256 rows); each CTA
// stores its 128 rows and adds one arrival, so an output tile is complete at
// 2P arrivals.  When the pair's tile rail runs out (one-way switch), or from
// the start for reducer pairs, each CTA reduces on its own through a local
// reduce ring with its own stage barriers.

struct RedRing {
    uint64_t *rfull;    // [NSTAGE2]
    uint64_t *rempty;   // [NSTAGE2]
    uint64_t *rsfull;   // [NSCHED]
    uint64_t *rsempty;  // [NSCHED] 4 epilogue warps
    SchedEntry *rsched; // [NSCHED]
};

__device__ __forceinline__ RedRing carve_red(const Smem2 &sm) {
    RedRing r;
    uint64_t *b = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(sm.tmem_slot) + 16);
    r.rfull = b; b += NSTAGE2;
    r.rempty = b; b += NSTAGE2;
    r.rsfull = b; b += NSCHED;
    r.rsempty = b; b += NSCHED;
    r.rsched = reinterpret_cast<SchedEntry *>(b);
    return r;
}

__device__ __forceinline__ bool red_push(const RedRing &rr, RingState &rs, const SchedEntry &e, WsHeader *ws) {
    if (!mbar_wait(&rr.rsempty[rs.idx], rs.phase ^ 1u, PIPE_LIMIT_NS)) {
        set_error(ws, KOSMOS_ERR_DEVICE, -2);
        return false;
    }
    rr.rsched[rs.idx] = e;
    mbar_arrive(&rr.rsfull[rs.idx]);
    rs.advance();
    return true;
}

// Stage geometry of the two pair engines: bf16 (7 stages, two accumulators)
// and MXFP8 (6 stages + scale atoms, one accumulator); both stages are 32 KB,
// which the reduce phase reuses.
template <bool MX>
struct RsPairCfg {
    static constexpr int NS = MX ? F2_NSTAGE : NSTAGE2;
    static constexpr int SMEM = MX ? F2_SMEM_BYTES : SMEM2_BYTES;
    static constexpr int NACC = MX ? 1 : 2;
};
static_assert(F2_STAGE == STAGE2_BYTES, "both pair engines reuse 32 KB stages for the reduce phase");

// One CTA's half of one K stage of tile (q, chunk, band, tcol): A rows
// [row0, row0 + 128) of chunk `chunk` of X_q, B columns [col0, col0 + 128) of
// W_q; MXFP8 adds the rows' scale atom and the tile's two W scale atoms.
template <bool MX>
__device__ __forceinline__ void rs2_load_half(const RsParams &p, const Smem2 &sm, uint8_t *sf, uint32_t stage, int q,
                                              int chunk, int row0, int col0, int tile_c, int kb, uint32_t fb) {
    uint8_t *sa = sm.stages + stage * STAGE2_BYTES;
    if (MX) {
        uint8_t *sb = sa + F2_A_BYTES;
        uint8_t *sfs = sf + stage * F2_SF;
        const int rb = static_cast<int>((static_cast<int64_t>(chunk) * p.g.mc + row0) / BM);  // 128-row scale block
        tma_load_3d_pair(sa, &p.tmX[q], fb, kb * FBK, row0, chunk);
        tma_load_2d_pair(sb, &p.tmW[q], fb, col0, kb * FBK);
        tma_load_2d_pair(sfs, &p.tmSX[q], fb, 0, (rb * p.nkb + kb) * SF_ATOM_ROWS);
        tma_load_2d_pair(sfs + 512, &p.tmSW[q], fb, 0, ((2 * tile_c) * p.nkb + kb) * SF_ATOM_ROWS);
        tma_load_2d_pair(sfs + 1024, &p.tmSW[q], fb, 0, ((2 * tile_c + 1) * p.nkb + kb) * SF_ATOM_ROWS);
    } else {
        uint8_t *sb = sa + A2_BYTES;
        tma_load_3d_pair(sa, &p.tmX[q], fb, kb * BK, row0, chunk);
        tma_load_2d_pair(sb, &p.tmW[q], fb, col0, kb * BK);
        tma_load_2d_pair(sb + 64 * BK * 2, &p.tmW[q], fb, col0 + 64, kb * BK);
    }
}

template <bool MX>
__device__ __forceinline__ void rs2_producer(const RsParams &p, const Smem2 &sm, uint8_t *sf, const RedRing &rr,
                                             uint32_t crank) {
    using Cfg = RsPairCfg<MX>;
    const int P = p.g.P;
    const int pair = blockIdx.x / 2;
    const bool leader = crank == 0;
    // the first n_red pairs are the first reducers, each of their CTAs for rank (CTA index mod P):
    // from the start in the fixed split; self-scheduled, they build until either CTA's rank has a
    // ready reduce entry.  Builder pairs build tiles of any rank and reduce for rank (pair index
    // mod P) after the switch.
    const bool first = p.mode == RS_FUSED && pair < p.n_red;
    const bool on_ready = first && p.sched == KOSMOS_SCHED_SELF;
    const bool reducer_pair = (p.mode == RS_REDUCE_ONLY) || first;
    const int rank = (reducer_pair && p.mode == RS_FUSED) ? static_cast<int>(blockIdx.x) % P : pair % P;
    PipeStateN<Cfg::NS> ps;
    RingPair rs;
    int nrec = 0;
    // ---- tile phase (pair)
    if (leader) {
        const uint32_t my_full0 = mapa_u32(smem_u32(&sm.full[0]), 0);
        const int r_peer = static_cast<int>(blockIdx.x + 1) % P;
        while ((!reducer_pair || on_ready) && !failed(p.ws)) {
            if (on_ready && (rs_reduce_ready(p, rank, static_cast<uint32_t>(2 * P)) ||
                             rs_reduce_ready(p, r_peer, static_cast<uint32_t>(2 * P))))
                break;
            const uint32_t t = atomicAdd(&p.ws->tickets[0], 1u);
            if (t >= static_cast<uint32_t>(p.g.n_tile)) break;
            int q, chunk, band, tcol;
            rs_decode_tile(p.g, p.order, static_cast<int>(t), q, chunk, band, tcol);
            int slot = -1;
            if (TraceRec *r = trace_rec(p.trace, blockIdx.x, nrec)) {
                const int64_t now = static_cast<int64_t>(globaltimer());
                r->t_claim = now; r->t_ready = now; r->t_done = 0;
                r->kind = K_TILE; r->ticket = static_cast<int32_t>(t); r->cta = blockIdx.x;
                slot = nrec;
            }
            ++nrec;
            SchedEntry e;
            fill_done(e);
            e.kind = K_TILE; e.a = chunk; e.b = band; e.c = tcol; e.d = q; e.nstage = p.nkb;
            e.ticket = static_cast<int32_t>(t); e.slot = slot;
            if (!ring2_push(sm, rs, e, p.ws)) break;
            bool ok = true;
            for (int kb = 0; kb < p.nkb; ++kb) {
                if (!mbar_wait(&sm.empty[ps.stage], ps.phase ^ 1u, PIPE_LIMIT_NS)) {
                    set_error(p.ws, KOSMOS_ERR_DEVICE, t);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&sm.full[ps.stage], MX ? 2 * (F2_STAGE + F2_SF) : 2 * STAGE2_BYTES);
                rs2_load_half<MX>(p, sm, sf, ps.stage, q, chunk, band * PBM, tcol * BN, tcol, kb,
                                  my_full0 + ps.stage * 8);
                ps.advance();
            }
            if (!ok) break;
        }
        SchedEntry done;
        fill_done(done);
        ring2_push(sm, rs, done, p.ws);
    } else {
        const uint32_t leader_full0 = mapa_u32(smem_u32(&sm.full[0]), 0);
        while (true) {
            SchedEntry e;
            if (!ring2_take(sm, rs, false, e, p.ws, false)) break;
            if (e.kind == K_DONE) break;
            const int chunk = e.a, band = e.b, tcol = e.c, q = e.d;
            bool ok = true;
            for (int kb = 0; kb < e.nstage; ++kb) {
                if (!mbar_wait(&sm.empty[ps.stage], ps.phase ^ 1u, PIPE_LIMIT_NS)) {
                    set_error(p.ws, KOSMOS_ERR_DEVICE, e.ticket);
                    ok = false;
                    break;
                }
                rs2_load_half<MX>(p, sm, sf, ps.stage, q, chunk, band * PBM + HBM_ROWS, tcol * BN + HBN, tcol, kb,
                                  leader_full0 + ps.stage * 8);
                ps.advance();
            }
            if (!ok) break;
        }
    }
    // ---- reduce phase (this CTA alone): one-way switch after the tiles, or a reducer pair
    RingState rrs;
    const bool reduce = reducer_pair || (p.mode == RS_FUSED && p.sched == KOSMOS_SCHED_SELF);
    if (reduce && drain_stages2(sm, ps, p.ws)) {
        PipeStateN<Cfg::NS> rp;
        const uint32_t red_bytes = static_cast<uint32_t>(BN * RED_ROWS * 2 * P);
        while (!failed(p.ws)) {
            const uint32_t t = atomicAdd(&p.ws->tickets[KOSMOS_MAX_P + rank], 1u);
            if (t >= static_cast<uint32_t>(p.g.n_reduce)) break;
            int band, tcol;
            rs_decode_reduce(p.g, static_cast<int>(t), band, tcol);
            const int64_t tc = p.trace ? static_cast<int64_t>(globaltimer()) : 0;
            if (p.mode == RS_FUSED) {
                uint32_t *ctr = &p.arrive[(static_cast<int64_t>(rank) * p.g.bands + band) * p.g.tiles_n + tcol];
                if (!wait_flag_eq(p.ws, ctr, static_cast<uint32_t>(2 * P), p.wait_limit_ns,
                                  (static_cast<int64_t>(1) << 40) | (static_cast<int64_t>(rank) << 32) | t))
                    break;
                st_relaxed_gpu(ctr, 0u);
            } else if (p.link_gbs > 0 && P > 1) {
                link_wait(link_reserve(p.ws, (P - 1) * rs_tile_bytes(p, static_cast<int64_t>(band) * PBM, PBM, tcol),
                                       p.link_gbs));
            }
            int slot = -1;
            if (TraceRec *r = trace_rec(p.trace, blockIdx.x, nrec)) {
                r->t_claim = tc; r->t_ready = static_cast<int64_t>(globaltimer()); r->t_done = 0;
                r->kind = K_REDUCE; r->ticket = static_cast<int32_t>(t); r->cta = blockIdx.x;
                slot = nrec;
            }
            ++nrec;
            const int64_t left = p.g.mc - static_cast<int64_t>(band) * PBM;
            const int64_t rows = left < PBM ? left : PBM;
            const int nsub = static_cast<int>(cdiv(rows, RED_ROWS));
            SchedEntry e;
            fill_done(e);
            e.kind = K_REDUCE; e.a = rank; e.b = band; e.c = tcol; e.d = rank; e.nstage = nsub;
            e.ticket = static_cast<int32_t>(t); e.slot = slot;
            if (!red_push(rr, rrs, e, p.ws)) break;
            bool ok = true;
            for (int sidx = 0; sidx < nsub; ++sidx) {
                if (!mbar_wait(&rr.rempty[rp.stage], rp.phase ^ 1u, PIPE_LIMIT_NS)) {
                    set_error(p.ws, KOSMOS_ERR_DEVICE, t);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&rr.rfull[rp.stage], red_bytes);
                tma_load_4d(sm.stages + rp.stage * STAGE2_BYTES, &p.tmPart, &rr.rfull[rp.stage], tcol * BN,
                            band * PBM + sidx * RED_ROWS, rank, 0);
                rp.advance();
            }
            if (!ok) break;
        }
    }
    SchedEntry done;
    fill_done(done);
    red_push(rr, rrs, done, p.ws);
}

template <bool MX>
__device__ __forceinline__ void rs2_epilogue(const RsParams &p, const Smem2 &sm, const RedRing &rr, uint32_t tmem_base,
                                             int warp, int lane, uint32_t crank) {
    using Cfg = RsPairCfg<MX>;
    const bool leader = crank == 0;
    const int grp = warp & 3;  // TMEM lanes (accumulator rows) 32 grp .. 32 grp + 31
    const int et = (warp - 2) * 32 + lane;
    const int P = p.g.P;
    RingPair rs;
    uint32_t acc = 0, acc_phase = 0;
    // ---- pair tiles
    while (true) {
        SchedEntry e;
        if (!ring2_take(sm, rs, leader, e, p.ws, true)) break;
        if (e.kind == K_DONE) break;
        if (e.kind != K_TILE) continue;
        if (!mbar_wait(&sm.tfull[acc], acc_phase, PIPE_LIMIT_NS)) {
            set_error(p.ws, KOSMOS_ERR_DEVICE, -7);
            break;
        }
        tc_fence_after();
        const int chunk = e.a, band = e.b, tcol = e.c, rank = e.d;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(grp * 32) << 16) + acc * BN;
        if constexpr (Cfg::NACC == 1) {
            // One accumulator (the scale atoms take the other's columns): the
            // row is copied into registers as bf16 and the accumulator released
            // before the global stores, so the next tile's MMAs run under them.
            uint32_t pk[BN / 64][32];
#pragma unroll
            for (int ch = 0; ch < BN / 32; ++ch) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(taddr + ch * 32, r);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    pk[ch / 2][(ch % 2) * 16 + j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
            }
            acc_release(sm, acc, leader, lane);
            if (++acc == Cfg::NACC) { acc = 0; acc_phase ^= 1u; }
            const int64_t rw = static_cast<int64_t>(band) * PBM + crank * HBM_ROWS + grp * 32;  // the warp's first row
            const int64_t rleft = p.g.mc - rw;
            const int rows_w = rleft <= 0 ? 0 : (rleft >= 32 ? 32 : static_cast<int>(rleft));
            __nv_bfloat16 *base = p.part + (static_cast<int64_t>(rank) * p.g.m + static_cast<int64_t>(chunk) * p.g.mc +
                                            (rows_w > 0 ? rw : 0)) * p.g.n;
#pragma unroll
            for (int c64 = 0; c64 < BN / 64; ++c64) {
                const int64_t col0 = static_cast<int64_t>(tcol) * BN + c64 * 64;
                const int64_t left = p.g.n - col0;
                if (left > 0) {  // warp-uniform
                    lane_transpose8_16B(pk[c64], lane);
                    store_row_lines(pk[c64], base + col0, p.g.n, rows_w, left < 64 ? static_cast<int>(left) : 64, lane);
                }
            }
        } else {
            const int64_t rw = static_cast<int64_t>(band) * PBM + crank * HBM_ROWS + grp * 32;  // the warp's first row
            const int64_t rleft = p.g.mc - rw;
            const int rows_w = rleft <= 0 ? 0 : (rleft >= 32 ? 32 : static_cast<int>(rleft));
            __nv_bfloat16 *base = p.part + (static_cast<int64_t>(rank) * p.g.m + static_cast<int64_t>(chunk) * p.g.mc +
                                            (rows_w > 0 ? rw : 0)) * p.g.n;
#pragma unroll 1
            for (int c64 = 0; c64 < BN / 64; ++c64) {
                const int64_t col0 = static_cast<int64_t>(tcol) * BN + c64 * 64;
                if (col0 >= p.g.n) break;
                const int64_t left = p.g.n - col0;
                tmem_rows64_to_bf16_lines(taddr + c64 * 64, base + col0, p.g.n, rows_w,
                                          left < 64 ? static_cast<int>(left) : 64, lane);
            }
            acc_release(sm, acc, leader, lane);
            if (++acc == Cfg::NACC) { acc = 0; acc_phase ^= 1u; }
        }
        if (p.mode == RS_FUSED) {
            __threadfence();
            named_bar_sync(1, NUM_EPI_THREADS);
            const bool drop = (p.inject & KOSMOS_INJECT_DROP_PARTIAL) && static_cast<int>(p.inject >> 32) == rank;
            if (et == 0 && !drop) {
                if (p.link_gbs > 0 && rank != chunk)  // this CTA's half of another rank's partial
                    link_wait(link_reserve(
                        p.ws, rs_tile_bytes(p, static_cast<int64_t>(band) * PBM + crank * HBM_ROWS, HBM_ROWS, tcol),
                        p.link_gbs));
                red_release_add_gpu(&p.arrive[(static_cast<int64_t>(chunk) * p.g.bands + band) * p.g.tiles_n + tcol], 1u);
            }
        }
        if (leader && e.slot >= 0 && et == 0) {
            if (TraceRec *r = trace_rec(p.trace, blockIdx.x, e.slot)) r->t_done = static_cast<int64_t>(globaltimer());
        }
    }
    // ---- this CTA's reductions
    RingState rrs;
    PipeStateN<Cfg::NS> rp;
    const int cg = et & 31;
    while (true) {
        if (!mbar_wait(&rr.rsfull[rrs.idx], rrs.phase, PIPE_LIMIT_NS)) {
            set_error(p.ws, KOSMOS_ERR_DEVICE, -9);
            break;
        }
        const SchedEntry e = rr.rsched[rrs.idx];
        __syncwarp();
        if (lane == 0) mbar_arrive(&rr.rsempty[rrs.idx]);
        rrs.advance();
        if (e.kind == K_DONE) break;
        const int chunk = e.a, band = e.b, tcol = e.c;
        const int64_t col = static_cast<int64_t>(tcol) * BN + cg * 8;
        bool ok = true;
        for (int sidx = 0; sidx < e.nstage; ++sidx) {
            // each warp releases the stage once its lanes have read it (no
            // group barrier per stage); a wait that runs out stops the warp
            const bool got = __all_sync(0xFFFFFFFFu, mbar_wait(&rr.rfull[rp.stage], rp.phase, PIPE_LIMIT_NS));
            if (!got) {
                set_error(p.ws, KOSMOS_ERR_DEVICE, -8);
                ok = false;
                break;
            }
            const uint8_t *buf = sm.stages + rp.stage * STAGE2_BYTES;
#pragma unroll
            for (int r2 = 0; got && r2 < 2; ++r2) {
                const int r8 = (et >> 5) * 2 + r2;
                float a[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) a[q] = 0.f;
                for (int rk = 0; rk < P; ++rk) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(buf + ((rk * RED_ROWS + r8) * BN + cg * 8) * 2);
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        a[2 * q] += __uint_as_float(w[q] << 16);
                        a[2 * q + 1] += __uint_as_float(w[q] & 0xFFFF0000u);
                    }
                }
                const int64_t grow = static_cast<int64_t>(band) * PBM + sidx * RED_ROWS + r8;
                if (grow < p.g.mc && col < p.g.n) {
                    uint4 o;
                    o.x = pack_bf16x2(a[0], a[1]);
                    o.y = pack_bf16x2(a[2], a[3]);
                    o.z = pack_bf16x2(a[4], a[5]);
                    o.w = pack_bf16x2(a[6], a[7]);
                    *reinterpret_cast<uint4 *>(p.y[chunk] + grow * p.g.n + col) = o;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&rr.rempty[rp.stage]);
            rp.advance();
        }
        if (!ok) break;
        if (e.slot >= 0 && et == 0) {
            if (TraceRec *r = trace_rec(p.trace, blockIdx.x, e.slot)) r->t_done = static_cast<int64_t>(globaltimer());
        }
    }
}

template <bool MX>
__device__ __forceinline__ void rs_pair_body(const RsParams &p, uint8_t *smem_raw) {
    using Cfg = RsPairCfg<MX>;
    Smem2 sm;
    uint8_t *sf = nullptr;
    if (MX) {
        const F2Smem fs = carve_f2(smem_raw);
        sm = fs.base;
        sf = fs.sf;
    } else {
        sm = carve_smem2(smem_raw);
    }
    const RedRing rr = carve_red(sm);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t crank = cluster_rank();
    const uint32_t epoch = *reinterpret_cast<volatile uint32_t *>(&p.ws->epoch);
    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::NS; ++i) {
            mbar_init(&rr.rfull[i], 1);
            mbar_init(&rr.rempty[i], NUM_EPI_THREADS / 32);  // each epilogue warp releases the stage
        }
        for (int i = 0; i < NSCHED; ++i) {
            mbar_init(&rr.rsfull[i], 1);
            mbar_init(&rr.rsempty[i], 4);
        }
    }
    engine2_setup(sm, warp, Cfg::NS);
    const uint32_t tmem_base = *sm.tmem_slot;
    if (warp == 0) {
        if (lane == 0) rs2_producer<MX>(p, sm, sf, rr, crank);
    } else if (warp == 1) {
        if (lane == 0 && crank == 0) {
            if (MX) {
                F2Smem fs;
                fs.base = sm;
                fs.sf = sf;
                f2_mma_loop(fs, tmem_base, p.ws);
            } else {
                mma2_loop(sm, tmem_base, p.ws);
            }
        }
    } else {
        rs2_epilogue<MX>(p, sm, rr, tmem_base, warp, lane, crank);
    }
    engine2_teardown(sm, warp, tmem_base);
    if (threadIdx.x == 0) engine_finish(p.ws, epoch, 2 * KOSMOS_MAX_P);
}

__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_rs_pair_kernel(const __grid_constant__ RsParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    rs_pair_body<false>(p, smem_raw);
}

// MXFP8 operands (E4M3 + E8M0 per 32 K), block-scaled pair MMAs; bf16 partials.
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_rs_mx_pair_kernel(const __grid_constant__ RsParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    rs_pair_body<true>(p, smem_raw);
}

int rs_pair_grid_limit(bool mx) {
    return mx ? max_pair_ctas(reinterpret_cast<const void *>(&gemm_rs_mx_pair_kernel), F2_SMEM_BYTES)
              : max_pair_ctas(reinterpret_cast<const void *>(&gemm_rs_pair_kernel), SMEM2_BYTES);
}

kosmos_status launch_rs_bf16(const RsLaunch &L, cudaStream_t stream) {
    RsParams p;
    memset(&p, 0, sizeof(p));
    p.g = rs_geom(L.P, L.m, L.k, L.n);
    const int64_t mc = p.g.mc;
    const bool mx = L.dtype == KOSMOS_MXFP8_E4M3;
    const uint64_t esz = mx ? 1 : 2;  // element bytes
    const CUtensorMapDataType dt = mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int kstage = mx ? FBK : BK;  // K elements per stage
    for (int r = 0; r < L.P; ++r) {
        {
            const uint64_t dims[3] = {static_cast<uint64_t>(L.k), static_cast<uint64_t>(mc), static_cast<uint64_t>(L.P)};
            const uint64_t strides[2] = {static_cast<uint64_t>(L.k) * esz, static_cast<uint64_t>(mc * L.k) * esz};
            const uint32_t box[3] = {static_cast<uint32_t>(kstage), BM, 1};
            if (!encode_tmap(&p.tmX[r], dt, 3, const_cast<void *>(L.x[r]), dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B))
                return KOSMOS_ERR_CUDA;
        }
        {
            const uint64_t dims[2] = {static_cast<uint64_t>(L.n), static_cast<uint64_t>(L.k)};
            const uint64_t strides[1] = {static_cast<uint64_t>(L.n) * esz};
            const uint32_t box[2] = {mx ? 128u : 64u, static_cast<uint32_t>(kstage)};
            if (!encode_tmap(&p.tmW[r], dt, 2, const_cast<void *>(L.w[r]), dims, strides, box,
                             CU_TENSOR_MAP_SWIZZLE_128B))
                return KOSMOS_ERR_CUDA;
        }
        if (mx) {
            const uint64_t nkb = static_cast<uint64_t>(L.k / FBK);
            if (!encode_sf_tmap(&p.tmSX[r], const_cast<void *>(L.xs[r]), static_cast<uint64_t>(L.m / BM) * nkb) ||
                !encode_sf_tmap(&p.tmSW[r], const_cast<void *>(L.ws_[r]), static_cast<uint64_t>(cdiv(L.n, 128)) * nkb))
                return KOSMOS_ERR_CUDA;
        }
        p.y[r] = static_cast<__nv_bfloat16 *>(L.y[r]);
    }
    const RsWsLayout W = rs_ws_layout(p.g, L.trace != 0);
    uint8_t *ws = static_cast<uint8_t *>(L.ws);
    p.ws = reinterpret_cast<WsHeader *>(ws);
    p.arrive = reinterpret_cast<uint32_t *>(ws + W.arrive_off);
    p.part = reinterpret_cast<__nv_bfloat16 *>(ws + W.partial_off);
    p.trace = L.trace ? reinterpret_cast<TraceRec *>(ws + W.trace_off) : nullptr;
    {
        const uint64_t dims[4] = {static_cast<uint64_t>(L.n), static_cast<uint64_t>(mc), static_cast<uint64_t>(L.P),
                                  static_cast<uint64_t>(L.P)};
        const uint64_t strides[3] = {static_cast<uint64_t>(L.n) * 2, static_cast<uint64_t>(mc * L.n) * 2,
                                     static_cast<uint64_t>(L.m * L.n) * 2};
        const uint32_t box[4] = {BN, RED_ROWS, 1, static_cast<uint32_t>(L.P)};
        if (!encode_tmap(&p.tmPart, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.part, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
            return KOSMOS_ERR_CUDA;
    }
    p.nkb = static_cast<int>(L.k / kstage);
    p.sched = L.sched;
    p.n_red = L.pair ? (L.n_comm * L.P + 1) / 2 : L.n_comm;  // pair kernel: reducer pairs
    p.order = L.order;
    p.wait_limit_ns = L.wait_limit_ns;
    p.inject = L.inject;
    p.link_gbs = L.link_gbs;
    const void *fn = mx       ? reinterpret_cast<const void *>(&gemm_rs_mx_pair_kernel)
                     : L.pair ? reinterpret_cast<const void *>(&gemm_rs_pair_kernel)
                              : reinterpret_cast<const void *>(&gemm_rs_kernel);
    const int smem = mx ? F2_SMEM_BYTES : (L.pair ? SMEM2_BYTES : SMEM_BYTES);
    if (mx && !L.pair) return KOSMOS_ERR_UNSUPPORTED;
    if (L.pair) p.g = rs_geom(L.P, L.m, L.k, L.n, PBM);
    auto go = [&]() {
        return L.pair ? launch_persistent_pairs(fn, &p, L.grid, smem, stream, L.plain_launch != 0)
                      : launch_persistent(fn, &p, L.grid, smem, stream, L.plain_launch != 0);
    };
    if (L.sched == KOSMOS_SCHED_UNFUSED) {
        p.mode = RS_TILES_ONLY;
        const kosmos_status s1 = go();
        if (s1 != KOSMOS_OK) return s1;
        p.mode = RS_REDUCE_ONLY;
        return go();
    }
    p.mode = RS_FUSED;
    return go();
}

}  // namespace kosmos
