// ag_gemm.cu -- all-gather + GEMM as one self-scheduling persistent launch.
//
// Y = concat_r(X_r) . W from rank 0's view (KOSMOS explainer, paragraph
// "Start with the problem").  Two rails:
//   transfer rail  TRANSFER(shard, piece): copy 128 rows of a remote shard
//                  into the gathered buffer, then release that piece's flag;
//                  remote shards in the order the tiles consume them, the
//                  local shard's own copy last (explainer, "Role switching
//                  only works");
//   tile rail      TILE(shard, tile_row, tile_col), local shard first.
// The first n_comm CTAs start as movers and become builders when the
// transfer rail runs out (one-way, explainer "KOSMOS removes the manager");
// the others are builders from the start.  A builder acquires the flag of
// the piece its tile reads before loading it.
#include <cuda.h>
#include <cuda_runtime.h>

#include "engine2.cuh"
#include "launch.h"

namespace kosmos {

struct AgParams {
    CUtensorMap tmA_local;  // x_shards[0]: dims {k, m}, box {64, 128}, 128B swizzle
    CUtensorMap tmA_gath;   // x_gathered: dims {k, m, P}, box {64, 128, 1}, 128B swizzle
    CUtensorMap tmB;        // W: dims {n, k}, box {64, 64}, 128B swizzle
    const uint8_t *x_src[KOSMOS_MAX_P];
    uint8_t *x_gath;
    __nv_bfloat16 *y;
    WsHeader *ws;
    uint32_t *flags;
    uint32_t *ksync;  // K-split slots: [slot][cta of the engine][counter, flag]
    float4 *kpart;    // K-split slots: [slot][cta of the engine] fp32 partials
    TraceRec *trace;
    AgGeom g;
    int nkb;
    int sched;
    int n_comm;
    int pad;
    uint64_t wait_limit_ns;
    uint64_t inject;
    int64_t link_gbs;  // emulated link for the remote pieces; 0 = uncapped
    // host-input flow (null otherwise): ext_ready[s * AG_EXT_STRIDE + c] becomes
    // 1 once chunk c of shard s (ag_host_cpp(g, s) pieces) has been copied into its
    // slot of x_gathered (by a copy stream); ydone[s * AG_EXT_STRIDE + j]
    // counts the output tiles of tile-row group j of shard s written (per CTA
    // of a tile engine).  In this flow the tiles read every shard from
    // x_gathered once its chunk has arrived, and the transfers run the other
    // way: each copies its part from x_gathered into the shard's device
    // buffer (x_src), beside the tiles rather than ahead of them.
    const uint32_t *ext_ready;
    uint32_t *ydone;
};

// Host-input flow: waits until the chunk holding piece `piece` of shard s is
// on the device.
__device__ __forceinline__ bool ag_ext_wait(const AgParams &p, int s, int piece, int64_t entry) {
    if (p.ext_ready == nullptr) return true;
    const int c = piece / ag_host_cpp(p.g, s);
    return wait_flag_eq(p.ws, const_cast<uint32_t *>(&p.ext_ready[s * AG_EXT_STRIDE + c]), 1u, p.wait_limit_ns,
                        entry);
}

// Whether tiles of shard s read A from the local shard buffer (tmA_local)
// rather than from x_gathered: the local shard of a fused call on device
// inputs.  The unfused baseline gathers first; the host-input flow lands
// every shard in x_gathered.
__device__ __forceinline__ bool ag_reads_local(const AgParams &p, int s) {
    return s == 0 && p.sched != KOSMOS_SCHED_UNFUSED && p.ext_ready == nullptr;
}

// Whether a tile of shard s waits for its pieces' flags (released by the
// transfers into x_gathered): remote shards of a fused call on device inputs.
__device__ __forceinline__ bool ag_waits_flags(const AgParams &p, int s) {
    return s != 0 && p.sched != KOSMOS_SCHED_UNFUSED && p.ext_ready == nullptr;
}

// Whether a tile of shard s waits for its chunk's arrival word: every shard
// of a fused host-input call (the unfused baseline's gather waits instead).
__device__ __forceinline__ bool ag_waits_arrival(const AgParams &p) {
    return p.ext_ready != nullptr && p.sched != KOSMOS_SCHED_UNFUSED;
}

// Host-input flow: one output tile of tile row `trow` of shard s written by
// this CTA's epilogue warps.
__device__ __forceinline__ void ag_ydone(const AgParams &p, int s, int trow, int grp, int lane) {
    if (p.ydone == nullptr) return;
    __threadfence();
    named_bar_sync(1, NUM_EPI_THREADS);
    if (grp == 0 && lane == 0) red_release_add_gpu(&p.ydone[s * AG_EXT_STRIDE + trow / ag_host_tpg(p.g, s)], 1u);
}

// Host-input flow: a failed launch releases every output wait of the host.
__device__ __forceinline__ void ag_ydone_release(const AgParams &p) {
    if (p.ydone == nullptr || !failed(p.ws)) return;
    for (int i = 0; i < p.g.P * AG_EXT_STRIDE; ++i) st_release_gpu(&p.ydone[i], AG_YDONE_RELEASE);
}

// Tile-rail entry -> what the engine runs: output columns [col0, col0 + BN)
// and K blocks [kb0, kb0 + nk); slot >= 0 marks one K half of a split tile.
struct AgTileWork {
    int s, i, col0, kb0, nk, slot;
};
__device__ __forceinline__ AgTileWork ag_tile_work(const AgParams &p, int t) {
    AgTileWork w;
    int c;
    const int kind = ag_decode_tile(p.g, t, w.s, w.i, c);
    w.kb0 = 0;
    w.nk = p.nkb;
    w.slot = -1;
    if (kind == K_TILE_HALF) {
        const int h = c & 1;
        c >>= 1;
        w.kb0 = h ? p.nkb / 2 : 0;
        w.nk = h ? p.nkb - p.nkb / 2 : p.nkb / 2;
        w.slot = (t - (p.g.n_full - p.g.n_split)) >> 1;
    }
    w.col0 = c * BN;
    return w;
}

// Mover side of the all-gather: claims transfer entries (one part of one
// piece: <= 32 rows of one shard, contiguous in both the shard and the
// gathered buffer) and streams them through the stage buffers; each landed
// part adds one arrival to its piece's flag.
__device__ __forceinline__ bool ag_claim_transfer(const AgParams &p, MoveEntry &e) {
    if (failed(p.ws)) return false;
    const uint32_t t = atomicAdd(&p.ws->tickets[0], 1u);
    if (t >= static_cast<uint32_t>(p.g.n_transfer)) return false;
    int shard, piece, part;
    ag_decode_transfer(p.g, static_cast<int>(t), shard, piece, part);
    if (!ag_ext_wait(p, shard, piece, t)) return false;
    int64_t row0, rows;
    ag_part_rows(p.g, piece, part, row0, rows);
    const int64_t row_bytes = p.g.k * 2;
    uint8_t *gath = p.x_gath + (static_cast<int64_t>(shard) * p.g.m + row0) * row_bytes;
    uint8_t *shard_buf = const_cast<uint8_t *>(p.x_src[shard]) + row0 * row_bytes;
    const bool to_shard = p.ext_ready != nullptr;  // host-input flow: x_gathered -> the shard's device buffer
    e.src[0] = to_shard ? gath : shard_buf;
    e.dst[0] = to_shard ? shard_buf : gath;
    e.bytes[0] = rows * row_bytes;
    e.src[1] = nullptr; e.dst[1] = nullptr; e.bytes[1] = 0;
    const bool drop = (p.inject & KOSMOS_INJECT_DROP_TRANSFER) && static_cast<int64_t>(p.inject >> 32) == t;
    e.flag = drop ? nullptr : &p.flags[shard * p.g.pieces + piece];
    e.ticket = static_cast<int32_t>(t);
    e.t_claim = p.trace ? static_cast<int64_t>(globaltimer()) : 0;
    // a remote piece crosses the emulated link; the local shard's own copy does not
    e.deadline = (p.link_gbs > 0 && shard != 0) ? link_reserve(p.ws, static_cast<uint64_t>(e.bytes[0]), p.link_gbs) : 0;
    return true;
}

// Runs this CTA's mover role until the transfer rail is exhausted; false after a device error.
template <int NS, int CH>
__device__ __forceinline__ bool ag_mover_phase(const AgParams &p, uint8_t *stages, uint64_t *cbar, uint32_t &cphase,
                                               int &nrec) {
    auto claim = [&](MoveEntry &e) { return ag_claim_transfer(p, e); };
    auto done = [&](int32_t ticket, int64_t t_claim) {
        if (TraceRec *r = trace_rec(p.trace, blockIdx.x, nrec)) {
            r->t_claim = t_claim; r->t_ready = t_claim; r->t_done = static_cast<int64_t>(globaltimer());
            r->kind = K_TRANSFER; r->ticket = ticket; r->cta = blockIdx.x;
        }
        ++nrec;
    };
    return stream_mover<NS, CH, 2>(stages, cbar, cphase, p.ws, claim, done) && !failed(p.ws);
}

// Readiness-driven role switching on the builder side (self-scheduling only):
// a builder whose next tile waits for a piece that has not arrived takes the
// transfer rail's next unclaimed part -- a piece some tile waits for, its own
// or a later one -- instead of spinning, one part at a time, re-checking its
// piece after each, while its piece is missing and parts remain.  One part at
// a time: claiming several in a row (or streaming the next part ahead of the
// current one) made a helper copy its own piece part after part, later than
// the movers would have delivered it.  It does not claim while the emulated
// link is backlogged beyond one part's copy time: then the link, not the
// number of movers, sets the pace, and a part claimed now would only wait in
// the link's queue.  Its stage buffers carry the copies: drain() first waits
// until the tile pipeline has consumed every stage it loaded (the previous
// tiles' MMAs keep running meanwhile).  Returns false after a device error.
constexpr uint64_t HELP_LINK_SLACK_NS = 16000;  // about one 32-row part's copy time by one SM
template <int NS, int CH, class Drain>
__device__ __forceinline__ bool ag_help_until_ready(const AgParams &p, uint8_t *stages, uint64_t *cbar,
                                                    uint32_t &cphase, int &nrec, int s, int pc, uint32_t target,
                                                    Drain &&drain) {
    if (p.sched != KOSMOS_SCHED_SELF || p.ext_ready != nullptr || s == 0) return true;
    const uint32_t *flag = &p.flags[s * p.g.pieces + pc];
    auto link_free = [&] {
        if (p.link_gbs <= 0) return true;
        const uint64_t t0 = *reinterpret_cast<const volatile uint64_t *>(&p.ws->link_t0);
        if (t0 == 0) return true;
        const uint64_t queued = *reinterpret_cast<const volatile uint64_t *>(&p.ws->link_bytes);
        return t0 + queued / static_cast<uint64_t>(p.link_gbs) <= globaltimer() + HELP_LINK_SLACK_NS;
    };
    auto wanted = [&] {
        return ld_acquire_gpu(flag) != target &&
               ld_relaxed_gpu(&p.ws->tickets[0]) < static_cast<uint32_t>(p.g.n_transfer) && link_free();
    };
    if (!wanted()) return true;
    if (!drain()) return false;
    auto done = [&](int32_t ticket, int64_t t_claim) {
        if (TraceRec *r = trace_rec(p.trace, blockIdx.x, nrec)) {
            r->t_claim = t_claim; r->t_ready = t_claim; r->t_done = static_cast<int64_t>(globaltimer());
            r->kind = K_TRANSFER; r->ticket = ticket; r->cta = blockIdx.x;
        }
        ++nrec;
    };
    while (wanted()) {
        bool taken = false;
        auto claim = [&](MoveEntry &e) {
            if (taken) return false;
            taken = true;
            return ag_claim_transfer(p, e);
        };
        if (!stream_mover<NS, CH, 2>(stages, cbar, cphase, p.ws, claim, done) || failed(p.ws)) return false;
    }
    return true;
}

// Waits until every stage of the one-SM pipeline has been consumed.
__device__ __forceinline__ bool drain_stages1(const Smem &sm, const PipeState &ps, WsHeader *ws) {
    for (int i = 0; i < NSTAGE; ++i) {
        uint32_t st = ps.stage + i, ph = ps.phase;
        if (st >= NSTAGE) { st -= NSTAGE; ph ^= 1u; }
        if (!mbar_wait(&sm.empty[st], ph ^ 1u, PIPE_LIMIT_NS)) {
            set_error(ws, KOSMOS_ERR_DEVICE, -11);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void ag_producer(const AgParams &p, const Smem &sm, uint32_t epoch) {
    const int cta = blockIdx.x;
    bool mover = (p.sched != KOSMOS_SCHED_UNFUSED) && cta < p.n_comm;
    uint32_t cphase = 0;
    PipeState ps;
    RingState rs;
    int nrec = 0;
    while (true) {
        if (failed(p.ws)) break;
        if (mover) {
            if (!ag_mover_phase<NSTAGE, STAGE_BYTES>(p, sm.stages, sm.cbar, cphase, nrec)) break;
            if (p.sched == KOSMOS_SCHED_FIXED) break;  // a fixed crew never builds
            mover = false;                             // one-way switch: mover -> builder
        }
        const uint32_t t = atomicAdd(&p.ws->tickets[1], 1u);
        if (t >= static_cast<uint32_t>(p.g.n_tile)) break;
        const AgTileWork w = ag_tile_work(p, static_cast<int>(t));
        const int s = w.s, i = w.i;
        const int64_t tc = p.trace ? static_cast<int64_t>(globaltimer()) : 0;
        if (ag_waits_flags(p, s)) {
            if (!ag_help_until_ready<NSTAGE, STAGE_BYTES>(p, sm.stages, sm.cbar, cphase, nrec, s, i,
                                                          ag_piece_ready(p.g, epoch),
                                                          [&] { return drain_stages1(sm, ps, p.ws); }))
                break;
            if (!wait_flag_eq(p.ws, &p.flags[s * p.g.pieces + i], ag_piece_ready(p.g, epoch), p.wait_limit_ns, t))
                break;
        }
        if (ag_waits_arrival(p) && !ag_ext_wait(p, s, i, t)) break;  // host-input flow
        int slot = -1;
        if (TraceRec *r = trace_rec(p.trace, cta, nrec)) {
            r->t_claim = tc; r->t_ready = static_cast<int64_t>(globaltimer()); r->t_done = 0;
            r->kind = K_TILE; r->ticket = static_cast<int32_t>(t); r->cta = cta;
            slot = nrec;
        }
        ++nrec;
        SchedEntry e;
        fill_done(e);
        e.kind = K_TILE; e.a = s; e.b = i; e.c = w.col0; e.d = w.kb0; e.nstage = w.nk;
        e.ticket = static_cast<int32_t>(t); e.slot = slot; e.x1 = w.slot;
        if (!ring_push(sm, rs, e, p.ws)) break;
        const bool local = ag_reads_local(p, s);
        bool ok = true;
        for (int kk = 0; kk < w.nk; ++kk) {
            const int kb = w.kb0 + kk;
            if (!mbar_wait(&sm.empty[ps.stage], ps.phase ^ 1u, PIPE_LIMIT_NS)) {
                set_error(p.ws, KOSMOS_ERR_DEVICE, t);
                ok = false;
                break;
            }
            uint8_t *sa = sm.stages + ps.stage * STAGE_BYTES;
            uint8_t *sb = sa + A_STAGE_BYTES;
            uint64_t *bar = &sm.full[ps.stage];
            mbar_arrive_expect_tx(bar, STAGE_BYTES);
            if (local)
                tma_load_2d(sa, &p.tmA_local, bar, kb * BK, i * BM);
            else
                tma_load_3d(sa, &p.tmA_gath, bar, kb * BK, i * BM, s);
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
                tma_load_2d(sb + j * (64 * BK * 2), &p.tmB, bar, w.col0 + j * 64, kb * BK);
            ps.advance();
        }
        if (!ok) break;
    }
    SchedEntry done;
    done.kind = K_DONE; done.a = done.b = done.c = 0; done.nstage = 0; done.ticket = -1; done.slot = -1; done.d = 0;
    done.nmma = 0; done.x0 = done.x1 = done.x2 = 0;
    ring_push(sm, rs, done, p.ws);
}

__device__ __forceinline__ void ag_epilogue(const AgParams &p, const Smem &sm, uint32_t tmem_base, int warp,
                                            int lane, uint32_t epoch) {
    const int grp = warp & 3;  // TMEM lane group this warp may access
    const int row = grp * 32 + lane;
    RingState rs;
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
        if (e.kind != K_TILE) continue;
        if (!mbar_wait(&sm.tfull[acc], acc_phase, PIPE_LIMIT_NS)) {
            set_error(p.ws, KOSMOS_ERR_DEVICE, -7);
            break;
        }
        tc_fence_after();
        const int s = e.a, i = e.b;
        const int64_t rloc = static_cast<int64_t>(i) * BM + row;
        const bool valid = rloc < p.g.m;
        __nv_bfloat16 *yrow = p.y + (static_cast<int64_t>(s) * p.g.m + (valid ? rloc : 0)) * p.g.n;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(grp * 32) << 16) + acc * BN;
        if (e.x1 >= 0) {  // one K half of a split tile
            const int64_t cs = static_cast<int64_t>(e.x1) * 2;  // slot, CTA 0 of the engine
            khalf_epilogue(taddr, valid, yrow, e.c, p.g.n, p.kpart + cs * (BM * BN / 4), &p.ksync[cs * 2],
                           &p.ksync[cs * 2 + 1], epoch, p.ws, p.wait_limit_ns, e.ticket, row, sm.tmem_slot + 1);
        } else {
            const int64_t rw = static_cast<int64_t>(i) * BM + grp * 32;  // the warp's first row
            const int64_t rleft = p.g.m - rw;
            const int rows_w = rleft <= 0 ? 0 : (rleft >= 32 ? 32 : static_cast<int>(rleft));
            __nv_bfloat16 *base = p.y + (static_cast<int64_t>(s) * p.g.m + (rows_w > 0 ? rw : 0)) * p.g.n;
#pragma unroll 1
            for (int c64 = 0; c64 < BN / 64; ++c64) {
                const int64_t col0 = static_cast<int64_t>(e.c) + c64 * 64;
                if (col0 >= p.g.n) break;
                const int64_t left = p.g.n - col0;
                tmem_rows64_to_bf16_lines(taddr + c64 * 64, base + col0, p.g.n, rows_w,
                                          left < 64 ? static_cast<int>(left) : 64, lane);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.tempty[acc]);
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        ag_ydone(p, s, i, grp, lane);
        if (e.slot >= 0 && lane == 0 && grp == 0) {
            if (TraceRec *r = trace_rec(p.trace, blockIdx.x, e.slot)) r->t_done = static_cast<int64_t>(globaltimer());
        }
    }
}

__global__ void __launch_bounds__(NUM_THREADS, 1) ag_gemm_kernel(const __grid_constant__ AgParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const Smem sm = carve_smem(smem_raw);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        prefetch_tmap(&p.tmA_local);
        prefetch_tmap(&p.tmA_gath);
        prefetch_tmap(&p.tmB);
    }
    const uint32_t epoch = *reinterpret_cast<volatile uint32_t *>(&p.ws->epoch);
    engine_setup(sm, warp);
    const uint32_t tmem_base = *sm.tmem_slot;
    if (warp == 0) {
        if (lane == 0) ag_producer(p, sm, epoch);
    } else if (warp == 1) {
        if (lane == 0) mma_loop(sm, tmem_base, p.ws);
    } else {
        ag_epilogue(p, sm, tmem_base, warp, lane, epoch);
    }
    engine_teardown(sm, warp, tmem_base);
    if (threadIdx.x == 0) ag_ydone_release(p);
    if (threadIdx.x == 0) engine_finish(p.ws, epoch, 3);
}

// ============================================================== SM-pair variant
// Same rails and roles; tiles are 256 x 256 and belong to an SM pair (a
// cluster of two CTAs).  Transfer pieces stay 128 rows: the leader's half of a
// tile waits for piece 2i, the peer's half for piece 2i + 1.  Movers are whole
// pairs (both CTAs copy, then both build).

constexpr bool AG_KEEP_W_IN_L2 = true;

// Loads this CTA's half of one stage: A rows [row0, row0+128) of shard s and
// B columns [col0, col0+128) of K block kb, completing on the leader's full
// barrier.  W is read by every tile row: its loads ask L2 to keep it (wpol).
__device__ __forceinline__ void ag2_load_half(const AgParams &p, const Smem2 &sm, const PipeState2 &ps, bool local,
                                              int s, int64_t row0, int64_t col0, int kb, uint32_t leader_full,
                                              uint64_t wpol) {
    uint8_t *sa = sm.stages + ps.stage * STAGE2_BYTES;
    uint8_t *sb = sa + A2_BYTES;
    if (local)
        tma_load_2d_pair(sa, &p.tmA_local, leader_full, kb * BK, static_cast<int32_t>(row0));
    else
        tma_load_3d_pair(sa, &p.tmA_gath, leader_full, kb * BK, static_cast<int32_t>(row0), s);
    if (AG_KEEP_W_IN_L2) {
        tma_load_2d_pair_hint(sb, &p.tmB, leader_full, static_cast<int32_t>(col0), kb * BK, wpol);
        tma_load_2d_pair_hint(sb + 64 * BK * 2, &p.tmB, leader_full, static_cast<int32_t>(col0 + 64), kb * BK, wpol);
    } else {
        tma_load_2d_pair(sb, &p.tmB, leader_full, static_cast<int32_t>(col0), kb * BK);
        tma_load_2d_pair(sb + 64 * BK * 2, &p.tmB, leader_full, static_cast<int32_t>(col0 + 64), kb * BK);
    }
}

__device__ __forceinline__ void ag2_producer(const AgParams &p, const Smem2 &sm, uint32_t epoch, uint32_t rank) {
    const int pair = blockIdx.x / 2;
    const bool leader = rank == 0;
    const bool mover = (p.sched != KOSMOS_SCHED_UNFUSED) && pair < p.n_comm;
    uint32_t cphase = 0;
    PipeState2 ps;
    RingPair rs;
    int nrec = 0;
    const uint64_t wpol = AG_KEEP_W_IN_L2 ? l2_policy_evict_last() : 0;
    if (mover) {
        if (!ag_mover_phase<NSTAGE2, STAGE2_BYTES>(p, sm.stages, sm.cbar, cphase, nrec) ||
            p.sched == KOSMOS_SCHED_FIXED) {
            if (leader) {
                SchedEntry done;
                fill_done(done);
                ring2_push(sm, rs, done, p.ws);
            } else {
                SchedEntry e;
                while (ring2_take(sm, rs, false, e, p.ws, false) && e.kind != K_DONE) {
                }
            }
            return;
        }
    }
    if (leader) {
        const uint32_t my_full0 = mapa_u32(smem_u32(&sm.full[0]), 0);
        while (true) {
            if (failed(p.ws)) break;
            const uint32_t t = atomicAdd(&p.ws->tickets[1], 1u);
            if (t >= static_cast<uint32_t>(p.g.n_tile)) break;
            const AgTileWork w = ag_tile_work(p, static_cast<int>(t));
            const int s = w.s, i2 = w.i;
            const int64_t tc = p.trace ? static_cast<int64_t>(globaltimer()) : 0;
            const int pc = 2 * i2;  // the leader's 128-row piece
            const bool remote = ag_waits_flags(p, s) && pc < p.g.pieces;
            // the entry is published before the readiness wait, so that the
            // peer can take transfer parts (or wait for the arrival of its
            // own piece) meanwhile
            int slot = -1;
            TraceRec *rec = trace_rec(p.trace, blockIdx.x, nrec);
            if (rec) {
                rec->t_claim = tc; rec->t_ready = tc; rec->t_done = 0;
                rec->kind = K_TILE; rec->ticket = static_cast<int32_t>(t); rec->cta = blockIdx.x;
                slot = nrec;
            }
            ++nrec;
            SchedEntry e;
            fill_done(e);
            e.kind = K_TILE; e.a = s; e.b = i2; e.c = w.col0; e.d = w.kb0; e.nstage = w.nk;
            e.ticket = static_cast<int32_t>(t); e.slot = slot; e.x1 = w.slot;
            if (!ring2_push(sm, rs, e, p.ws)) break;
            if (remote) {
                if (!ag_help_until_ready<NSTAGE2, STAGE2_BYTES>(p, sm.stages, sm.cbar, cphase, nrec, s, pc,
                                                                ag_piece_ready(p.g, epoch),
                                                                [&] { return drain_stages2(sm, ps, p.ws); }))
                    break;
                if (!wait_flag_eq(p.ws, &p.flags[s * p.g.pieces + pc], ag_piece_ready(p.g, epoch),
                                  p.wait_limit_ns, t))
                    break;
            }
            if (ag_waits_arrival(p) && !ag_ext_wait(p, s, pc, t)) break;  // host-input flow
            if (rec) rec->t_ready = static_cast<int64_t>(globaltimer());
            const bool local = ag_reads_local(p, s);
            bool ok = true;
            for (int kk = 0; kk < w.nk; ++kk) {
                if (!mbar_wait(&sm.empty[ps.stage], ps.phase ^ 1u, PIPE_LIMIT_NS)) {
                    set_error(p.ws, KOSMOS_ERR_DEVICE, t);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&sm.full[ps.stage], 2 * STAGE2_BYTES);
                ag2_load_half(p, sm, ps, local, s, static_cast<int64_t>(i2) * PBM, w.col0, w.kb0 + kk,
                              my_full0 + ps.stage * 8, wpol);
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
            const int s = e.a, i2 = e.b;
            const int pc = 2 * i2 + 1;  // the peer's 128-row piece
            if (ag_waits_flags(p, s) && pc < p.g.pieces) {
                if (!ag_help_until_ready<NSTAGE2, STAGE2_BYTES>(p, sm.stages, sm.cbar, cphase, nrec, s, pc,
                                                                ag_piece_ready(p.g, epoch),
                                                                [&] { return drain_stages2(sm, ps, p.ws); }))
                    break;
                if (!wait_flag_eq(p.ws, &p.flags[s * p.g.pieces + pc], ag_piece_ready(p.g, epoch),
                                  p.wait_limit_ns, e.ticket))
                    break;
            }
            if (ag_waits_arrival(p) && pc < p.g.pieces && !ag_ext_wait(p, s, pc, e.ticket)) break;
            const bool local = ag_reads_local(p, s);
            bool ok = true;
            for (int kb = 0; kb < e.nstage; ++kb) {
                if (!mbar_wait(&sm.empty[ps.stage], ps.phase ^ 1u, PIPE_LIMIT_NS)) {
                    set_error(p.ws, KOSMOS_ERR_DEVICE, e.ticket);
                    ok = false;
                    break;
                }
                ag2_load_half(p, sm, ps, local, s, static_cast<int64_t>(i2) * PBM + HBM_ROWS,
                              static_cast<int64_t>(e.c) + HBN, e.d + kb, leader_full0 + ps.stage * 8, wpol);
                ps.advance();
            }
            if (!ok) break;
        }
    }
}

__device__ __forceinline__ void ag2_epilogue(const AgParams &p, const Smem2 &sm, uint32_t tmem_base, int warp, int lane,
                                             uint32_t rank, uint32_t epoch) {
    const bool leader = rank == 0;
    const int grp = warp & 3;
    const int row = grp * 32 + lane;
    RingPair rs;
    uint32_t acc = 0, acc_phase = 0;
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
        const int s = e.a, i2 = e.b;
        const int64_t rloc = static_cast<int64_t>(i2) * PBM + rank * HBM_ROWS + row;
        const bool valid = rloc < p.g.m;
        __nv_bfloat16 *yrow = p.y + (static_cast<int64_t>(s) * p.g.m + (valid ? rloc : 0)) * p.g.n;
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(grp * 32) << 16) + acc * BN;
        if (e.x1 >= 0) {  // one K half of a split tile: this CTA's 128 rows
            const int64_t cs = static_cast<int64_t>(e.x1) * 2 + rank;
            khalf_epilogue(taddr, valid, yrow, e.c, p.g.n, p.kpart + cs * (BM * BN / 4), &p.ksync[cs * 2],
                           &p.ksync[cs * 2 + 1], epoch, p.ws, p.wait_limit_ns, e.ticket, row, sm.tmem_slot + 1);
        } else {
            const int64_t rw = static_cast<int64_t>(i2) * PBM + rank * HBM_ROWS + grp * 32;  // the warp's first row
            const int64_t rleft = p.g.m - rw;
            const int rows_w = rleft <= 0 ? 0 : (rleft >= 32 ? 32 : static_cast<int>(rleft));
            __nv_bfloat16 *base = p.y + (static_cast<int64_t>(s) * p.g.m + (rows_w > 0 ? rw : 0)) * p.g.n;
#pragma unroll 1
            for (int c64 = 0; c64 < BN / 64; ++c64) {
                const int64_t col0 = static_cast<int64_t>(e.c) + c64 * 64;
                if (col0 >= p.g.n) break;
                const int64_t left = p.g.n - col0;
                tmem_rows64_to_bf16_lines(taddr + c64 * 64, base + col0, p.g.n, rows_w,
                                          left < 64 ? static_cast<int>(left) : 64, lane);
            }
        }
        acc_release(sm, acc, leader, lane);
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        ag_ydone(p, s, i2, grp, lane);
        if (leader && e.slot >= 0 && lane == 0 && grp == 0) {
            if (TraceRec *r = trace_rec(p.trace, blockIdx.x, e.slot)) r->t_done = static_cast<int64_t>(globaltimer());
        }
    }
}

__global__ void __launch_bounds__(NUM_THREADS, 1) ag_gemm_pair_kernel(const __grid_constant__ AgParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const Smem2 sm = carve_smem2(smem_raw);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = cluster_rank();
    if (threadIdx.x == 0) {
        prefetch_tmap(&p.tmA_local);
        prefetch_tmap(&p.tmA_gath);
        prefetch_tmap(&p.tmB);
    }
    const uint32_t epoch = *reinterpret_cast<volatile uint32_t *>(&p.ws->epoch);
    engine2_setup(sm, warp);
    const uint32_t tmem_base = *sm.tmem_slot;
    if (warp == 0) {
        if (lane == 0) ag2_producer(p, sm, epoch, rank);
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) mma2_loop(sm, tmem_base, p.ws);
    } else {
        ag2_epilogue(p, sm, tmem_base, warp, lane, rank, epoch);
    }
    engine2_teardown(sm, warp, tmem_base);
    if (threadIdx.x == 0) ag_ydone_release(p);
    if (threadIdx.x == 0) engine_finish(p.ws, epoch, 3);
}

// Unfused baseline, first launch: gather every shard into x_gathered with
// plain 16-byte vector copies over all SMs (in the host-input flow, where the
// shards land in x_gathered, copy each on into its device buffer instead).
__global__ void __launch_bounds__(256) ag_gather_copy_kernel(const AgParams p) {
    if (p.ext_ready != nullptr) {  // host-input flow: every shard must be on the device
        if (threadIdx.x == 0)
            for (int s = 0; s < p.g.P; ++s)
                for (int pc = 0; pc < p.g.pieces; pc += ag_host_cpp(p.g, s)) ag_ext_wait(p, s, pc, -40);
        __syncthreads();
        if (failed(p.ws)) return;
    }
    const int64_t shard_bytes = p.g.m * p.g.k * 2;
    const int64_t per = shard_bytes / 16;
    const int64_t total = per * p.g.P;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const bool to_shard = p.ext_ready != nullptr;  // host-input flow: x_gathered -> the shard buffers
    for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < total; v += stride) {
        const int64_t s = v / per;
        const int64_t o = v - s * per;
        uint4 *gath = reinterpret_cast<uint4 *>(p.x_gath + s * shard_bytes) + o;
        uint4 *shard = reinterpret_cast<uint4 *>(const_cast<uint8_t *>(p.x_src[s])) + o;
        if (to_shard)
            *shard = *gath;
        else
            *gath = *shard;
    }
    if (p.link_gbs > 0) ag_copy_link_pace(p.ws, per, total, p.link_gbs);
}

// ---------------------------------------------------------------- host launcher
int ag_pair_grid_limit() { return max_pair_ctas(reinterpret_cast<const void *>(&ag_gemm_pair_kernel), SMEM2_BYTES); }

kosmos_status launch_ag_bf16(const AgLaunch &L, cudaStream_t stream) {
    AgParams p;
    memset(&p, 0, sizeof(p));
    p.g = ag_geom(L.P, L.m, L.k, L.n, L.pair ? PBM : BM, L.n_split);
    // tensor maps
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(L.k), static_cast<uint64_t>(L.m)};
        const uint64_t strides[1] = {static_cast<uint64_t>(L.k) * 2};
        const uint32_t box[2] = {BK, BM};
        if (!encode_tmap(&p.tmA_local, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(L.x[0]), dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return KOSMOS_ERR_CUDA;
    }
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(L.k), static_cast<uint64_t>(L.m), static_cast<uint64_t>(L.P)};
        const uint64_t strides[2] = {static_cast<uint64_t>(L.k) * 2, static_cast<uint64_t>(L.m * L.k) * 2};
        const uint32_t box[3] = {BK, BM, 1};
        if (!encode_tmap(&p.tmA_gath, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, L.x_gathered, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return KOSMOS_ERR_CUDA;
    }
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(L.n), static_cast<uint64_t>(L.k)};
        const uint64_t strides[1] = {static_cast<uint64_t>(L.n) * 2};
        const uint32_t box[2] = {64, BK};
        if (!encode_tmap(&p.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(L.w), dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return KOSMOS_ERR_CUDA;
    }
    for (int r = 0; r < L.P; ++r) p.x_src[r] = static_cast<const uint8_t *>(L.x[r]);
    p.x_gath = static_cast<uint8_t *>(L.x_gathered);
    p.y = static_cast<__nv_bfloat16 *>(L.y);
    const AgWsLayout W = ag_ws_layout(p.g, L.trace != 0, L.n_slots);
    uint8_t *ws = static_cast<uint8_t *>(L.ws);
    p.ws = reinterpret_cast<WsHeader *>(ws);
    p.flags = reinterpret_cast<uint32_t *>(ws + W.flags_off);
    p.ksync = reinterpret_cast<uint32_t *>(ws + W.ksync_off);
    p.kpart = reinterpret_cast<float4 *>(ws + W.kpart_off);
    p.trace = L.trace ? reinterpret_cast<TraceRec *>(ws + W.trace_off) : nullptr;
    if (L.host_flow) {
        p.ext_ready = reinterpret_cast<const uint32_t *>(ws + W.ext_off);
        p.ydone = reinterpret_cast<uint32_t *>(ws + W.ext_off) + AG_EXT_WORDS;
    }
    p.nkb = static_cast<int>(L.k / BK);
    p.sched = L.sched;
    p.n_comm = L.n_comm;
    p.wait_limit_ns = L.wait_limit_ns;
    p.inject = L.inject;
    p.link_gbs = L.link_gbs;

    if (L.pair) p.n_comm = (L.n_comm + 1) / 2;  // mover pairs
    if (L.sched == KOSMOS_SCHED_UNFUSED) {
        const int sms = L.grid;
        ag_gather_copy_kernel<<<sms * 4, 256, 0, stream>>>(p);
        if (cudaGetLastError() != cudaSuccess) return KOSMOS_ERR_CUDA;
    }
    if (L.pair)
        return launch_persistent_pairs(reinterpret_cast<const void *>(&ag_gemm_pair_kernel), &p, L.grid, SMEM2_BYTES,
                                       stream, L.plain_launch != 0);
    return launch_persistent(reinterpret_cast<const void *>(&ag_gemm_kernel), &p, L.grid, SMEM_BYTES, stream,
                             L.plain_launch != 0);
}

}  // namespace kosmos
