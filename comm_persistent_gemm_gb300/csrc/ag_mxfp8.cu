// ag_mxfp8.cu -- all-gather + GEMM with MXFP8 operands (E4M3 elements, one E8M0
// scale per 32 consecutive K-elements), one self-scheduling persistent launch
// (KOSMOS abstract: TP+SP training "1.10-1.25x in MXFP8").
//
// Same rails and roles as the bf16 kernel (ag_gemm.cu): movers copy remote
// shard pieces (elements and their scale blocks) into the gathered buffers and
// release per-piece flags; builders start on the local shard.  The product uses
// tcgen05.mma kind::mxf8f6f4.block_scale: per 128-wide K stage the MMA warp
// copies the stage's scale factors from shared memory into tensor memory with
// tcgen05.cp, then issues four K=32 MMAs, each selecting its scale byte.
//
// Scale layout (MMA-tiled, produced by kosmos_mxfp8_quantize): for an operand
// with R scale rows (rows of X, columns of W) and K, the scale of (row r,
// K-block b) is at byte ((r/128)*(K/128) + b/4)*512 + (r%32)*16 + ((r/32)%4)*4
// + b%4.  One 512-byte atom covers 128 rows x 4 K-blocks; copied with
// tcgen05.cp 32x128b.warpx4 it lands in four TMEM columns, lane r%32 of every
// 32-lane group holding rows r%32 + 32c in column c, one byte per K-block.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>

#include "mxfp8.cuh"
#include "launch.h"

namespace kosmos {

constexpr int F_A_BYTES = BM * FBK;            // 16 KB
constexpr int F_B_SLAB = 128 * FBK;            // one 128-column slab of B: 16 KB
constexpr int F_B_BYTES = 2 * F_B_SLAB;        // 32 KB
constexpr int F_SF_BYTES = 3 * 512;            // SFA atom + two SFB atoms
constexpr int F_SMEM_BYTES = SMEM_BYTES + NSTAGE * F_SF_BYTES;

struct AgF8Params {
    CUtensorMap tmA_local;  // x_shards[0]: dims {k, m} (bytes), box {128, 128}, 128B swizzle
    CUtensorMap tmA_gath;   // x_gathered: dims {k, m, P}, box {128, 128, 1}
    CUtensorMap tmB;        // W: dims {n, k}, box {128, 128}
    // SM-pair kernel only: the tiled scales as rows of 16 bytes, one 512-byte atom per box
    CUtensorMap tmSA_local; // x_scales[0]: pieces * nkb atoms (encode_sf_tmap)
    CUtensorMap tmSA_gath;  // gathered scales: P * pieces * nkb atoms
    CUtensorMap tmSW;       // W scales: nb_w * nkb atoms
    const uint8_t *x_src[KOSMOS_MAX_P];
    const uint8_t *sx_src[KOSMOS_MAX_P];  // tiled scales of each shard
    const uint8_t *sw;                    // tiled scales of W
    uint8_t *x_gath;
    uint8_t *sx_gath;                     // tiled scales, gathered [P][pieces][k/128][512]
    __nv_bfloat16 *y;
    WsHeader *ws;
    uint32_t *flags;
    TraceRec *trace;
    AgGeom g;
    int nkb;          // k / 128
    int nb_w;         // 128-column scale blocks of W
    int sched;
    int n_comm;
    uint64_t wait_limit_ns;
    uint64_t inject;
    int64_t link_gbs;  // emulated link for the remote pieces; 0 = uncapped
};

struct F8Smem {
    Smem base;
    uint8_t *sf;  // [NSTAGE][F_SF_BYTES]
};

__device__ __forceinline__ F8Smem carve_f8(uint8_t *raw) {
    F8Smem s;
    s.base = carve_smem(raw);
    s.sf = s.base.stages + NSTAGE * STAGE_BYTES + SMEM_CTRL_BYTES;
    return s;
}

// Transfer entry of the MXFP8 all-gather: one part (<= 32 rows of E4M3
// bytes) of one piece; part 0 also carries the piece's scale block (the
// E8M0 scales are tiled per 128 rows).
__device__ __forceinline__ bool f8_claim_transfer(const AgF8Params &p, MoveEntry &e) {
    if (failed(p.ws)) return false;
    const uint32_t t = atomicAdd(&p.ws->tickets[0], 1u);
    if (t >= static_cast<uint32_t>(p.g.n_transfer)) return false;
    int shard, piece, part;
    ag_decode_transfer(p.g, static_cast<int>(t), shard, piece, part);
    int64_t row0, rows;
    ag_part_rows(p.g, piece, part, row0, rows);
    const int64_t row_bytes = p.g.k;
    e.src[0] = p.x_src[shard] + row0 * row_bytes;
    e.dst[0] = p.x_gath + (static_cast<int64_t>(shard) * p.g.m + row0) * row_bytes;
    e.bytes[0] = rows * row_bytes;
    const int64_t sblk = static_cast<int64_t>(p.nkb) * 512;  // scale bytes of one 128-row block
    e.src[1] = p.sx_src[shard] + piece * sblk;
    e.dst[1] = p.sx_gath + (static_cast<int64_t>(shard) * p.g.pieces + piece) * sblk;
    e.bytes[1] = part == 0 ? sblk : 0;
    const bool drop = (p.inject & KOSMOS_INJECT_DROP_TRANSFER) && static_cast<int64_t>(p.inject >> 32) == t;
    e.flag = drop ? nullptr : &p.flags[shard * p.g.pieces + piece];
    e.ticket = static_cast<int32_t>(t);
    e.t_claim = p.trace ? static_cast<int64_t>(globaltimer()) : 0;
    e.deadline = (p.link_gbs > 0 && shard != 0)
                     ? link_reserve(p.ws, static_cast<uint64_t>(e.bytes[0] + e.bytes[1]), p.link_gbs)
                     : 0;
    return true;
}

__device__ __forceinline__ void f8_producer(const AgF8Params &p, const F8Smem &fs, uint32_t epoch) {
    const Smem &sm = fs.base;
    const int cta = blockIdx.x;
    bool mover = (p.sched != KOSMOS_SCHED_UNFUSED) && cta < p.n_comm;
    uint32_t cphase = 0;
    PipeState ps;
    RingState rs;
    int nrec = 0;
    const int64_t sblk = static_cast<int64_t>(p.nkb) * 512;
    while (true) {
        if (failed(p.ws)) break;
        if (mover) {
            auto claim = [&](MoveEntry &e) { return f8_claim_transfer(p, e); };
            auto done = [&](int32_t ticket, int64_t t_claim) {
                if (TraceRec *r = trace_rec(p.trace, cta, nrec)) {
                    r->t_claim = t_claim; r->t_ready = t_claim; r->t_done = static_cast<int64_t>(globaltimer());
                    r->kind = K_TRANSFER; r->ticket = ticket; r->cta = cta;
                }
                ++nrec;
            };
            if (!stream_mover<NSTAGE, STAGE_BYTES, 2>(sm.stages, sm.cbar, cphase, p.ws, claim, done) || failed(p.ws))
                break;
            if (p.sched == KOSMOS_SCHED_FIXED) break;
            mover = false;
        }
        const uint32_t t = atomicAdd(&p.ws->tickets[1], 1u);
        if (t >= static_cast<uint32_t>(p.g.n_tile)) break;
        int s, i, c;
        ag_decode_tile(p.g, static_cast<int>(t), s, i, c);
        const int64_t tc = p.trace ? static_cast<int64_t>(globaltimer()) : 0;
        if (p.sched != KOSMOS_SCHED_UNFUSED && s != 0) {
            if (!wait_flag_eq(p.ws, &p.flags[s * p.g.pieces + i], ag_piece_ready(p.g, epoch), p.wait_limit_ns, t))
                break;
        }
        int slot = -1;
        if (TraceRec *r = trace_rec(p.trace, cta, nrec)) {
            r->t_claim = tc; r->t_ready = static_cast<int64_t>(globaltimer()); r->t_done = 0;
            r->kind = K_TILE; r->ticket = static_cast<int32_t>(t); r->cta = cta;
            slot = nrec;
        }
        ++nrec;
        SchedEntry e;
        e.kind = K_TILE; e.a = s; e.b = i; e.c = c; e.d = 0; e.nstage = p.nkb; e.ticket = static_cast<int32_t>(t);
        e.slot = slot; e.nmma = 0; e.x0 = e.x1 = e.x2 = 0;
        if (!ring_push(sm, rs, e, p.ws)) break;
        const bool local = (s == 0) && p.sched != KOSMOS_SCHED_UNFUSED;
        const uint8_t *sfa_base = local ? (p.sx_src[0] + static_cast<int64_t>(i) * sblk)
                                        : (p.sx_gath + (static_cast<int64_t>(s) * p.g.pieces + i) * sblk);
        const int nb0 = c * 2, nb1 = c * 2 + 1;
        const bool has_b1 = nb1 < p.nb_w;
        const uint32_t bytes = F_A_BYTES + F_B_BYTES + 512u * (has_b1 ? 3u : 2u);
        bool ok = true;
        for (int kb = 0; kb < p.nkb; ++kb) {
            if (!mbar_wait(&sm.empty[ps.stage], ps.phase ^ 1u, PIPE_LIMIT_NS)) {
                set_error(p.ws, KOSMOS_ERR_DEVICE, t);
                ok = false;
                break;
            }
            uint8_t *sa = sm.stages + ps.stage * STAGE_BYTES;
            uint8_t *sb = sa + F_A_BYTES;
            uint8_t *sf = fs.sf + ps.stage * F_SF_BYTES;
            uint64_t *bar = &sm.full[ps.stage];
            mbar_arrive_expect_tx(bar, bytes);
            if (local)
                tma_load_2d(sa, &p.tmA_local, bar, kb * FBK, i * BM);
            else
                tma_load_3d(sa, &p.tmA_gath, bar, kb * FBK, i * BM, s);
            tma_load_2d(sb, &p.tmB, bar, c * BN, kb * FBK);
            tma_load_2d(sb + F_B_SLAB, &p.tmB, bar, c * BN + 128, kb * FBK);
            bulk_g2s(sf, sfa_base + static_cast<int64_t>(kb) * 512, 512, bar);
            bulk_g2s(sf + 512, p.sw + (static_cast<int64_t>(nb0) * p.nkb + kb) * 512, 512, bar);
            if (has_b1) bulk_g2s(sf + 1024, p.sw + (static_cast<int64_t>(nb1) * p.nkb + kb) * 512, 512, bar);
            ps.advance();
        }
        if (!ok) break;
    }
    SchedEntry done;
    done.kind = K_DONE; done.a = done.b = done.c = done.d = 0; done.nstage = 0; done.ticket = -1; done.slot = -1;
    done.nmma = 0; done.x0 = done.x1 = done.x2 = 0;
    ring_push(sm, rs, done, p.ws);
}

// One accumulator (TMEM columns 0..255); the scale buffers use 256 + 16*stage.
__device__ __forceinline__ void f8_mma_loop(const F8Smem &fs, uint32_t tmem_base, WsHeader *ws) {
    const Smem &sm = fs.base;
    PipeState ps;
    RingState rs;
    uint32_t acc_phase = 0;
    while (true) {
        if (!mbar_wait(&sm.sfull[rs.idx], rs.phase, PIPE_LIMIT_NS)) {
            set_error(ws, KOSMOS_ERR_DEVICE, -3);
            break;
        }
        const SchedEntry e = sm.sched[rs.idx];
        mbar_arrive(&sm.sempty[rs.idx]);
        rs.advance();
        if (e.kind == K_DONE) break;
        if (e.kind != K_TILE) {
            ps.advance(e.nstage);
            continue;
        }
        if (!mbar_wait(&sm.tempty[0], acc_phase ^ 1u, PIPE_LIMIT_NS)) {
            set_error(ws, KOSMOS_ERR_DEVICE, -4);
            break;
        }
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < e.nstage; ++kb) {
            if (!mbar_wait(&sm.full[ps.stage], ps.phase, PIPE_LIMIT_NS)) {
                set_error(ws, KOSMOS_ERR_DEVICE, -5);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sm.stages + ps.stage * STAGE_BYTES);
            const uint32_t b_addr = a_addr + F_A_BYTES;
            const uint32_t sf_addr = smem_u32(fs.sf + ps.stage * F_SF_BYTES);
            const uint32_t sfa_t = tmem_base + F_TMEM_SF + ps.stage * F_TMEM_SF_STRIDE;
            mx_stage_mma(tmem_base, a_addr, b_addr, F_B_SLAB, sf_addr, sfa_t, kb == 0);
            mma_commit(&sm.empty[ps.stage]);
            ps.advance();
        }
        if (!ok) break;
        mma_commit(&sm.tfull[0]);
        acc_phase ^= 1u;
    }
}

// A warp's 32 drained rows (row-per-lane, four 64-column blocks of bf16
// pairs) stored as 128-byte row segments of Y: shard s, the warp's first
// row rw, column tile c.  All 32 lanes call it.
__device__ __forceinline__ void ag_f8_store_rows(const AgF8Params &p, uint32_t (&packed)[BN / 64][32], int s,
                                                 int64_t rw, int c, int lane) {
    const int64_t rleft = p.g.m - rw;
    const int rows_w = rleft <= 0 ? 0 : (rleft >= 32 ? 32 : static_cast<int>(rleft));
    __nv_bfloat16 *base = p.y + (static_cast<int64_t>(s) * p.g.m + (rows_w > 0 ? rw : 0)) * p.g.n;
#pragma unroll
    for (int c64 = 0; c64 < BN / 64; ++c64) {
        const int64_t col0 = static_cast<int64_t>(c) * BN + c64 * 64;
        const int64_t left = p.g.n - col0;
        if (left > 0) {  // warp-uniform
            lane_transpose8_16B(packed[c64], lane);
            store_row_lines(packed[c64], base + col0, p.g.n, rows_w, left < 64 ? static_cast<int>(left) : 64, lane);
        }
    }
}

// Drains the accumulator into registers (bf16-packed), releases it, then stores.
__device__ __forceinline__ void f8_epilogue(const AgF8Params &p, const Smem &sm, uint32_t tmem_base, int warp,
                                            int lane) {
    const int grp = warp & 3;  // TMEM lanes (accumulator rows) 32 grp .. 32 grp + 31
    RingState rs;
    uint32_t acc_phase = 0;
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
        if (!mbar_wait(&sm.tfull[0], acc_phase, PIPE_LIMIT_NS)) {
            set_error(p.ws, KOSMOS_ERR_DEVICE, -7);
            break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(grp * 32) << 16);
        uint32_t packed[BN / 64][32];
#pragma unroll
        for (int ch = 0; ch < BN / 32; ++ch) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + ch * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j)
                packed[ch / 2][(ch % 2) * 16 + j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.tempty[0]);
        acc_phase ^= 1u;
        const int s = e.a, i = e.b, c = e.c;
        ag_f8_store_rows(p, packed, s, static_cast<int64_t>(i) * BM + grp * 32, c, lane);
        if (e.slot >= 0 && lane == 0 && grp == 0) {
            if (TraceRec *r = trace_rec(p.trace, blockIdx.x, e.slot)) r->t_done = static_cast<int64_t>(globaltimer());
        }
    }
}

__global__ void __launch_bounds__(NUM_THREADS, 1) ag_mxfp8_kernel(const __grid_constant__ AgF8Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const F8Smem fs = carve_f8(smem_raw);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t epoch = *reinterpret_cast<volatile uint32_t *>(&p.ws->epoch);
    engine_setup(fs.base, warp);
    const uint32_t tmem_base = *fs.base.tmem_slot;
    if (warp == 0) {
        if (lane == 0) f8_producer(p, fs, epoch);
    } else if (warp == 1) {
        if (lane == 0) f8_mma_loop(fs, tmem_base, p.ws);
    } else {
        f8_epilogue(p, fs.base, tmem_base, warp, lane);
    }
    engine_teardown(fs.base, warp, tmem_base);
    if (threadIdx.x == 0) engine_finish(p.ws, epoch, 3);
}

// ============================================================== SM-pair variant
// Tiles of 256 x 256 on an SM pair (tcgen05.mma.cta_group::2, block-scaled).
// Each CTA stages its 128 rows of A, its 128 columns of B, the scale atom of
// its rows (SFA) and the scale atoms of all 256 columns (SFB); the leader's
// tcgen05.cp.cta_group::2 copies every CTA's atoms into that CTA's tensor
// memory, where the pair MMA reads SFA of the CTA's rows and SFB of the whole
// tile (the placement was checked on the GB300 against exact results); the
// stage layout and MMA loop are in mxfp8.cuh.

// This CTA's half of one K stage of tile (s, i2, c): A rows of piece pc, B
// columns [col0, col0 + 128), the piece's scale atom and the tile's two W
// scale atoms; everything completes on the leader's full barrier.
__device__ __forceinline__ void f2_load_half(const AgF8Params &p, const F2Smem &fs, uint32_t stage, bool local, int s,
                                             int pc, int64_t col0, int tile_c, int kb, uint32_t leader_full) {
    uint8_t *sa = fs.base.stages + stage * F2_STAGE;
    uint8_t *sb = sa + F2_A_BYTES;
    uint8_t *sf = fs.sf + stage * F2_SF;
    const int32_t row0 = pc * BM;
    if (local) {
        tma_load_2d_pair(sa, &p.tmA_local, leader_full, kb * FBK, row0);
        tma_load_2d_pair(sf, &p.tmSA_local, leader_full, 0, (pc * p.nkb + kb) * SF_ATOM_ROWS);
    } else {
        tma_load_3d_pair(sa, &p.tmA_gath, leader_full, kb * FBK, row0, s);
        tma_load_2d_pair(sf, &p.tmSA_gath, leader_full, 0, ((s * p.g.pieces + pc) * p.nkb + kb) * SF_ATOM_ROWS);
    }
    tma_load_2d_pair(sb, &p.tmB, leader_full, static_cast<int32_t>(col0), kb * FBK);
    tma_load_2d_pair(sf + 512, &p.tmSW, leader_full, 0, ((2 * tile_c) * p.nkb + kb) * SF_ATOM_ROWS);
    tma_load_2d_pair(sf + 1024, &p.tmSW, leader_full, 0, ((2 * tile_c + 1) * p.nkb + kb) * SF_ATOM_ROWS);
}

__device__ __forceinline__ void f2_producer(const AgF8Params &p, const F2Smem &fs, uint32_t epoch, uint32_t rank) {
    const Smem2 &sm = fs.base;
    const int pair = blockIdx.x / 2;
    const bool leader = rank == 0;
    const bool mover = (p.sched != KOSMOS_SCHED_UNFUSED) && pair < p.n_comm;
    uint32_t cphase = 0;
    PipeF2 ps;
    RingPair rs;
    int nrec = 0;
    if (mover) {
        auto claim = [&](MoveEntry &e) { return f8_claim_transfer(p, e); };
        auto done = [&](int32_t ticket, int64_t t_claim) {
            if (TraceRec *r = trace_rec(p.trace, blockIdx.x, nrec)) {
                r->t_claim = t_claim; r->t_ready = t_claim; r->t_done = static_cast<int64_t>(globaltimer());
                r->kind = K_TRANSFER; r->ticket = ticket; r->cta = blockIdx.x;
            }
            ++nrec;
        };
        if (!stream_mover<F2_NSTAGE, F2_STAGE, 2>(sm.stages, sm.cbar, cphase, p.ws, claim, done) || failed(p.ws) ||
            p.sched == KOSMOS_SCHED_FIXED) {
            if (leader) {
                SchedEntry d;
                fill_done(d);
                ring2_push(sm, rs, d, p.ws);
            } else {
                SchedEntry e;
                while (ring2_take(sm, rs, false, e, p.ws, false) && e.kind != K_DONE) {
                }
            }
            return;
        }
    }
    const uint32_t leader_full0 = mapa_u32(smem_u32(&sm.full[0]), 0);
    if (leader) {
        while (true) {
            if (failed(p.ws)) break;
            const uint32_t t = atomicAdd(&p.ws->tickets[1], 1u);
            if (t >= static_cast<uint32_t>(p.g.n_tile)) break;
            int s, i2, c;
            ag_decode_tile(p.g, static_cast<int>(t), s, i2, c);
            const int64_t tc = p.trace ? static_cast<int64_t>(globaltimer()) : 0;
            const int pc = 2 * i2;  // the leader's 128-row piece
            if (p.sched != KOSMOS_SCHED_UNFUSED && s != 0 && pc < p.g.pieces) {
                if (!wait_flag_eq(p.ws, &p.flags[s * p.g.pieces + pc], ag_piece_ready(p.g, epoch), p.wait_limit_ns,
                                  t))
                    break;
            }
            int slot = -1;
            if (TraceRec *r = trace_rec(p.trace, blockIdx.x, nrec)) {
                r->t_claim = tc; r->t_ready = static_cast<int64_t>(globaltimer()); r->t_done = 0;
                r->kind = K_TILE; r->ticket = static_cast<int32_t>(t); r->cta = blockIdx.x;
                slot = nrec;
            }
            ++nrec;
            SchedEntry e;
            fill_done(e);
            e.kind = K_TILE; e.a = s; e.b = i2; e.c = c; e.nstage = p.nkb; e.ticket = static_cast<int32_t>(t);
            e.slot = slot;
            if (!ring2_push(sm, rs, e, p.ws)) break;
            const bool local = (s == 0) && p.sched != KOSMOS_SCHED_UNFUSED;
            bool ok = true;
            for (int kb = 0; kb < p.nkb; ++kb) {
                if (!mbar_wait(&sm.empty[ps.stage], ps.phase ^ 1u, PIPE_LIMIT_NS)) {
                    set_error(p.ws, KOSMOS_ERR_DEVICE, t);
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&sm.full[ps.stage], 2 * (F2_STAGE + F2_SF));
                f2_load_half(p, fs, ps.stage, local, s, pc, static_cast<int64_t>(c) * BN, c, kb,
                             leader_full0 + ps.stage * 8);
                ps.advance();
            }
            if (!ok) break;
        }
        SchedEntry d;
        fill_done(d);
        ring2_push(sm, rs, d, p.ws);
    } else {
        while (true) {
            SchedEntry e;
            if (!ring2_take(sm, rs, false, e, p.ws, false)) break;
            if (e.kind == K_DONE) break;
            const int s = e.a, i2 = e.b, c = e.c;
            const int pc = 2 * i2 + 1;  // the peer's 128-row piece
            if (p.sched != KOSMOS_SCHED_UNFUSED && s != 0 && pc < p.g.pieces) {
                if (!wait_flag_eq(p.ws, &p.flags[s * p.g.pieces + pc], ag_piece_ready(p.g, epoch), p.wait_limit_ns,
                                  e.ticket))
                    break;
            }
            const bool local = (s == 0) && p.sched != KOSMOS_SCHED_UNFUSED;
            bool ok = true;
            for (int kb = 0; kb < e.nstage; ++kb) {
                if (!mbar_wait(&sm.empty[ps.stage], ps.phase ^ 1u, PIPE_LIMIT_NS)) {
                    set_error(p.ws, KOSMOS_ERR_DEVICE, e.ticket);
                    ok = false;
                    break;
                }
                f2_load_half(p, fs, ps.stage, local, s, pc, static_cast<int64_t>(c) * BN + HBN, c, kb,
                             leader_full0 + ps.stage * 8);
                ps.advance();
            }
            if (!ok) break;
        }
    }
}

// Both CTAs: drain this CTA's 128 rows into registers (bf16-packed), release
// the accumulator (local or remote arrive), then store.
__device__ __forceinline__ void f2_epilogue(const AgF8Params &p, const Smem2 &sm, uint32_t tmem_base, int warp, int lane,
                                            uint32_t rank) {
    const bool leader = rank == 0;
    const int grp = warp & 3;  // TMEM lanes (accumulator rows) 32 grp .. 32 grp + 31
    RingPair rs;
    uint32_t acc_phase = 0;
    while (true) {
        SchedEntry e;
        if (!ring2_take(sm, rs, leader, e, p.ws, true)) break;
        if (e.kind == K_DONE) break;
        if (e.kind != K_TILE) continue;
        if (!mbar_wait(&sm.tfull[0], acc_phase, PIPE_LIMIT_NS)) {
            set_error(p.ws, KOSMOS_ERR_DEVICE, -7);
            break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(grp * 32) << 16);
        uint32_t packed[BN / 64][32];
#pragma unroll
        for (int ch = 0; ch < BN / 32; ++ch) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + ch * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j)
                packed[ch / 2][(ch % 2) * 16 + j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
        }
        acc_release(sm, 0, leader, lane);
        acc_phase ^= 1u;
        const int s = e.a, i2 = e.b, c = e.c;
        ag_f8_store_rows(p, packed, s, static_cast<int64_t>(i2) * PBM + rank * HBM_ROWS + grp * 32, c, lane);
        if (leader && e.slot >= 0 && lane == 0 && grp == 0) {
            if (TraceRec *r = trace_rec(p.trace, blockIdx.x, e.slot)) r->t_done = static_cast<int64_t>(globaltimer());
        }
    }
}

__global__ void __launch_bounds__(NUM_THREADS, 1) ag_mxfp8_pair_kernel(const __grid_constant__ AgF8Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const F2Smem fs = carve_f2(smem_raw);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = cluster_rank();
    if (threadIdx.x == 0) {
        prefetch_tmap(&p.tmA_local);
        prefetch_tmap(&p.tmA_gath);
        prefetch_tmap(&p.tmB);
        prefetch_tmap(&p.tmSA_local);
        prefetch_tmap(&p.tmSA_gath);
        prefetch_tmap(&p.tmSW);
    }
    const uint32_t epoch = *reinterpret_cast<volatile uint32_t *>(&p.ws->epoch);
    engine2_setup(fs.base, warp, F2_NSTAGE);
    const uint32_t tmem_base = *fs.base.tmem_slot;
    if (warp == 0) {
        if (lane == 0) f2_producer(p, fs, epoch, rank);
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) f2_mma_loop(fs, tmem_base, p.ws);
    } else {
        f2_epilogue(p, fs.base, tmem_base, warp, lane, rank);
    }
    engine2_teardown(fs.base, warp, tmem_base);
    if (threadIdx.x == 0) engine_finish(p.ws, epoch, 3);
}

int ag_mxfp8_pair_grid_limit() {
    return max_pair_ctas(reinterpret_cast<const void *>(&ag_mxfp8_pair_kernel), F2_SMEM_BYTES);
}

// Unfused baseline, first launch: gather elements and scale blocks of every shard.
__global__ void __launch_bounds__(256) ag_f8_gather_copy_kernel(const AgF8Params p) {
    const int64_t shard_bytes = p.g.m * p.g.k;
    const int64_t sblk = static_cast<int64_t>(p.nkb) * 512 * p.g.pieces;
    const int64_t per = shard_bytes / 16, sper = sblk / 16;
    const int64_t total = (per + sper) * p.g.P;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < total; v += stride) {
        const int64_t s = v / (per + sper);
        const int64_t o = v - s * (per + sper);
        if (o < per)
            reinterpret_cast<uint4 *>(p.x_gath + s * shard_bytes)[o] = reinterpret_cast<const uint4 *>(p.x_src[s])[o];
        else
            reinterpret_cast<uint4 *>(p.sx_gath + s * sblk)[o - per] =
                reinterpret_cast<const uint4 *>(p.sx_src[s])[o - per];
    }
    if (p.link_gbs > 0) ag_copy_link_pace(p.ws, per + sper, total, p.link_gbs);
}

size_t ag_mxfp8_scale_bytes(int P, int64_t m, int64_t k) {
    return static_cast<size_t>(P) * static_cast<size_t>(cdiv(m, BM)) * static_cast<size_t>(k / FBK) * 512;
}

kosmos_status launch_ag_mxfp8(const AgLaunch &L, cudaStream_t stream) {
    AgF8Params p;
    memset(&p, 0, sizeof(p));
    p.g = ag_geom(L.P, L.m, L.k, L.n);
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(L.k), static_cast<uint64_t>(L.m)};
        const uint64_t strides[1] = {static_cast<uint64_t>(L.k)};
        const uint32_t box[2] = {FBK, BM};
        if (!encode_tmap(&p.tmA_local, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(L.x[0]), dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return KOSMOS_ERR_CUDA;
    }
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(L.k), static_cast<uint64_t>(L.m), static_cast<uint64_t>(L.P)};
        const uint64_t strides[2] = {static_cast<uint64_t>(L.k), static_cast<uint64_t>(L.m * L.k)};
        const uint32_t box[3] = {FBK, BM, 1};
        if (!encode_tmap(&p.tmA_gath, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, L.x_gathered, dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return KOSMOS_ERR_CUDA;
    }
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(L.n), static_cast<uint64_t>(L.k)};
        const uint64_t strides[1] = {static_cast<uint64_t>(L.n)};
        const uint32_t box[2] = {128, FBK};
        if (!encode_tmap(&p.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(L.w), dims, strides, box,
                         CU_TENSOR_MAP_SWIZZLE_128B))
            return KOSMOS_ERR_CUDA;
    }
    for (int r = 0; r < L.P; ++r) {
        p.x_src[r] = static_cast<const uint8_t *>(L.x[r]);
        p.sx_src[r] = static_cast<const uint8_t *>(L.xs[r]);
    }
    p.sw = static_cast<const uint8_t *>(L.wsc);
    p.x_gath = static_cast<uint8_t *>(L.x_gathered);
    p.y = static_cast<__nv_bfloat16 *>(L.y);
    const AgWsLayout W = ag_ws_layout(p.g, L.trace != 0);
    uint8_t *ws = static_cast<uint8_t *>(L.ws);
    p.ws = reinterpret_cast<WsHeader *>(ws);
    p.flags = reinterpret_cast<uint32_t *>(ws + W.flags_off);
    p.trace = L.trace ? reinterpret_cast<TraceRec *>(ws + W.trace_off) : nullptr;
    p.sx_gath = ws + W.total;  // gathered scale blocks follow the bf16 layout (see kosmos_workspace_bytes)
    p.nkb = static_cast<int>(L.k / FBK);
    p.nb_w = static_cast<int>(cdiv(L.n, 128));
    p.sched = L.sched;
    p.n_comm = L.n_comm;
    p.wait_limit_ns = L.wait_limit_ns;
    p.inject = L.inject;
    p.link_gbs = L.link_gbs;
    if (L.pair) {
        p.g = ag_geom(L.P, L.m, L.k, L.n, PBM);
        p.n_comm = (L.n_comm + 1) / 2;  // mover pairs
        if (!encode_sf_tmap(&p.tmSA_local, const_cast<void *>(L.xs[0]), static_cast<uint64_t>(p.g.pieces) * p.nkb) ||
            !encode_sf_tmap(&p.tmSA_gath, p.sx_gath, static_cast<uint64_t>(L.P) * p.g.pieces * p.nkb) ||
            !encode_sf_tmap(&p.tmSW, const_cast<void *>(L.wsc), static_cast<uint64_t>(p.nb_w) * p.nkb))
            return KOSMOS_ERR_CUDA;
    }
    if (L.sched == KOSMOS_SCHED_UNFUSED) {
        ag_f8_gather_copy_kernel<<<L.grid * 4, 256, 0, stream>>>(p);
        if (cudaGetLastError() != cudaSuccess) return KOSMOS_ERR_CUDA;
    }
    if (L.pair)
        return launch_persistent_pairs(reinterpret_cast<const void *>(&ag_mxfp8_pair_kernel), &p, L.grid,
                                       F2_SMEM_BYTES, stream, L.plain_launch != 0);
    return launch_persistent(reinterpret_cast<const void *>(&ag_mxfp8_kernel), &p, L.grid, F_SMEM_BYTES, stream,
                             L.plain_launch != 0);
}

}  // namespace kosmos
