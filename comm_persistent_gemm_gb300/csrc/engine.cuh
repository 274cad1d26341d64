// engine.cuh -- the persistent CTA engine shared by the fused operators.
//
// One CTA per SM, 192 threads, warp-specialised:
//   warp 0 (lane 0)  scheduler + producer: claims tickets from the rails,
//                    performs mover transfers itself, waits for readiness
//                    flags, pushes TILE/REDUCE entries into an in-CTA ring and
//                    streams their operands into the shared-memory pipeline
//                    with TMA;
//   warp 1 (lane 0)  MMA issuer: tcgen05.mma over the staged K blocks into one
//                    of two TMEM accumulators (double-buffered);
//   warps 2..5       epilogue: tcgen05.ld of the accumulator (one row per
//                    thread), conversion and stores; reduction entries are
//                    summed here from the staged partial tiles.
// Every wait is bounded: on expiry the CTA records an error in the workspace
// header and leaves its loops; nothing traps.
#pragma once
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace kosmos {

struct SchedEntry {
    int32_t kind;     // EntryKind (K_DONE ends the CTA's loops)
    int32_t a, b, c;  // decoded entry fields
    int32_t nstage;   // pipeline stages the entry occupies
    int32_t ticket;
    int32_t slot;     // trace record index of this CTA, -1 when untraced
    int32_t d;        // extra field (op specific)
    int32_t nmma;     // N of the MMA (0 = BN)
    int32_t x0, x1, x2;  // extra fields (op specific)
};

__device__ __forceinline__ void fill_done(SchedEntry &e) {
    e.kind = K_DONE; e.a = e.b = e.c = e.d = 0; e.nstage = 0; e.ticket = -1; e.slot = -1;
    e.nmma = 0; e.x0 = e.x1 = e.x2 = 0;
}

__host__ __device__ __forceinline__ bool is_mma_kind(int32_t k) {
    return k == K_TILE || k == K_ROUTE || k == K_TILE_GU || k == K_TILE_D;
}

struct Smem {
    uint8_t *stages;   // NSTAGE * STAGE_BYTES, 1024-byte aligned
    uint64_t *full;    // [NSTAGE] operands landed (TMA complete_tx)
    uint64_t *empty;   // [NSTAGE] stage consumed (tcgen05.commit or epilogue)
    uint64_t *cbar;    // [NSTAGE] mover copy buffers landed
    uint64_t *tfull;   // [2] accumulator ready (tcgen05.commit)
    uint64_t *tempty;  // [2] accumulator drained (4 epilogue warps)
    uint64_t *sfull;   // [NSCHED] entry published
    uint64_t *sempty;  // [NSCHED] entry read by MMA + 4 epilogue warps
    SchedEntry *sched; // [NSCHED]
    uint32_t *tmem_slot;
};
constexpr int SMEM_CTRL_BYTES = 1024;  // barriers, entry ring, TMEM slot
constexpr int SMEM_BYTES = NSTAGE * STAGE_BYTES + SMEM_CTRL_BYTES + 1024;
constexpr uint64_t PIPE_LIMIT_NS = 4000000000ull;  // internal pipeline waits: 4 s

__device__ __forceinline__ Smem carve_smem(uint8_t *raw) {
    const uintptr_t base = (reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023);
    uint8_t *p = reinterpret_cast<uint8_t *>(base);
    Smem s;
    s.stages = p;
    p += NSTAGE * STAGE_BYTES;
    uint64_t *b = reinterpret_cast<uint64_t *>(p);
    s.full = b; b += NSTAGE;
    s.empty = b; b += NSTAGE;
    s.cbar = b; b += NSTAGE;
    s.tfull = b; b += 2;
    s.tempty = b; b += 2;
    s.sfull = b; b += NSCHED;
    s.sempty = b; b += NSCHED;
    s.sched = reinterpret_cast<SchedEntry *>(b);
    s.tmem_slot = reinterpret_cast<uint32_t *>(s.sched + NSCHED);
    return s;
}

struct PipeState {
    uint32_t stage = 0, phase = 0;
    __device__ __forceinline__ void advance() {
        if (++stage == NSTAGE) { stage = 0; phase ^= 1; }
    }
    __device__ __forceinline__ void advance(int n) {
        for (int i = 0; i < n; ++i) advance();
    }
};

struct RingState {
    uint32_t idx = 0, phase = 0;
    __device__ __forceinline__ void advance() {
        if (++idx == NSCHED) { idx = 0; phase ^= 1; }
    }
};

// ---------------------------------------------------------------- status
__device__ __forceinline__ void set_error(WsHeader *ws, uint32_t code, int64_t entry) {
    if (atomicCAS(&ws->status, 0u, code) == 0u) {
        ws->fail_entry = entry;
        __threadfence();
    }
}
__device__ __forceinline__ bool failed(WsHeader *ws) { return ld_relaxed_gpu(&ws->status) != 0u; }

// Bounded acquire-wait until *flag == target.  On success the caller may read
// the guarded data with TMA (the proxy fence orders the async-proxy reads
// after the acquire).  On expiry: status = TIMEOUT, fail_entry = entry.
__device__ __forceinline__ bool wait_flag_eq(WsHeader *ws, const uint32_t *flag, uint32_t target,
                                             uint64_t limit_ns, int64_t entry) {
    uint32_t it = 0;
    uint64_t t0 = 0;
    while (ld_acquire_gpu(flag) != target) {
        if ((++it & 15u) == 0u) {
            if (failed(ws)) return false;
            const uint64_t now = globaltimer();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > limit_ns) {
                set_error(ws, KOSMOS_ERR_TIMEOUT, entry);
                return false;
            }
        }
    }
    fence_proxy_async_global();
    return true;
}

// ---------------------------------------------------------------- streaming mover
// One transfer entry: up to two contiguous segments, copied global -> shared
// -> global with bulk async copies, then one release-add on *flag.
struct MoveEntry {
    const uint8_t *src[2];
    uint8_t *dst[2];
    int64_t bytes[2];
    uint32_t *flag;  // nullptr: no release (a transfer dropped by fault injection)
    int32_t ticket;
    int64_t t_claim;
    uint64_t deadline = 0;  // emulated link: release no earlier than this globaltimer value (0 = none)
};

struct MoveChunk {
    uint8_t *dst;
    uint32_t *flag;
    int64_t t_claim;
    int32_t ticket;
    uint32_t bytes;
    int32_t last;  // the entry's final chunk
    uint64_t deadline;
};

// ---------------------------------------------------------------- emulated link
// A pipe of gbs bytes per ns that never idles once the launch first uses it:
// the transfer that brings the reserved total to B bytes is delivered at
// t0 + B / gbs, t0 = the launch's first reservation.  While the link is
// backlogged (the case the cap exists for) this is a first-come-first-served
// server; when it would idle, later transfers catch up on the unused time.
// One atomic add per transfer (a compare-and-swap server serialised the
// reservations of 150 CTAs and cost more than the link itself).
__device__ __forceinline__ uint64_t link_reserve(WsHeader *ws, uint64_t bytes, int64_t gbs) {
    unsigned long long *t0p = reinterpret_cast<unsigned long long *>(&ws->link_t0);
    unsigned long long t0 = *reinterpret_cast<volatile unsigned long long *>(t0p);
    if (t0 == 0) {
        const unsigned long long now = globaltimer();
        const unsigned long long seen = atomicCAS(t0p, 0ull, now);
        t0 = seen == 0 ? now : seen;
    }
    const unsigned long long c =
        atomicAdd(reinterpret_cast<unsigned long long *>(&ws->link_bytes), static_cast<unsigned long long>(bytes));
    return t0 + (c + bytes) / static_cast<uint64_t>(gbs);
}

// Spins until globaltimer reaches deadline (at most 4 s: the host bounds the
// total link time of a call well below that).
__device__ __forceinline__ void link_wait(uint64_t deadline) {
    if (deadline == 0) return;
    const uint64_t t0 = globaltimer();
    while (true) {
        const uint64_t now = globaltimer();
        if (now >= deadline || now - t0 > PIPE_LIMIT_NS) return;
    }
}

// Publishes a transfer whose stores have completed: order the async-proxy
// writes before the generic release, then add one arrival to its flag.
template <class Done>
__device__ __forceinline__ void move_release(const MoveChunk &c, Done &done) {
    link_wait(c.deadline);
    fence_proxy_async_global();
    __threadfence();
    if (c.flag) red_release_add_gpu(c.flag, 1u);
    done(c.ticket, c.t_claim);
}

// Single-thread mover loop over consecutive transfer entries.  Chunks of CH
// bytes flow through NS stage buffers (stage b completes on cbar[b]); loads of
// the next entry are issued while the current one drains, so the pipeline
// does not empty between entries.  An entry is released once its last store
// is DEFER bulk groups old (cp.async.bulk.wait_group DEFER).
//   claim(MoveEntry &) -> bool : claim and describe the next entry; false when
//                                the rail is exhausted.
//   done(ticket, t_claim)      : called after each release (role trace).
// Returns false after a device error (a copy that never landed).
template <int NS, int CH, int DEFER, class Claim, class Done>
__device__ __noinline__ bool stream_mover(uint8_t *stages, uint64_t *cbar, uint32_t &cphase, WsHeader *ws,
                                          Claim &claim, Done &done) {
    static_assert(NS >= 2 && DEFER >= 0 && DEFER < 4, "stream_mover parameters");
    MoveChunk meta[NS];
    MoveChunk pend[4];  // entries whose last store is in flight, oldest first
    int64_t pend_at[4];
    int npend = 0;
    MoveEntry cur;
    int seg = 0;
    int64_t off = 0;
    bool have = false, more = true;

    auto next_chunk = [&](MoveChunk &out, const uint8_t *&src) -> bool {
        while (true) {
            if (!have) {
                if (!more || !claim(cur)) {
                    more = false;
                    return false;
                }
                seg = 0;
                off = 0;
                have = true;
                if (cur.bytes[0] + cur.bytes[1] == 0) {  // an empty part: nothing to copy
                    MoveChunk e;
                    e.flag = cur.flag; e.ticket = cur.ticket; e.t_claim = cur.t_claim; e.deadline = cur.deadline;
                    move_release(e, done);
                    have = false;
                    continue;
                }
            }
            if (off >= cur.bytes[seg]) {
                if (++seg >= 2) {
                    have = false;
                } else {
                    off = 0;
                }
                continue;
            }
            const int64_t rem = cur.bytes[seg] - off;
            const uint32_t nb = static_cast<uint32_t>(rem < CH ? rem : CH);
            src = cur.src[seg] + off;
            out.dst = cur.dst[seg] + off;
            out.bytes = nb;
            out.flag = cur.flag;
            out.ticket = cur.ticket;
            out.t_claim = cur.t_claim;
            out.deadline = cur.deadline;
            off += nb;
            out.last = (off >= cur.bytes[seg]) && (seg == 1 || cur.bytes[1] == 0);
            if (out.last) have = false;
            return true;
        }
    };

    // sources are read once: let them leave L2 first
    const uint64_t pol = l2_policy_evict_first();
    int64_t issued = 0, stored = 0;
    for (int b = 0; b < NS; ++b) {
        const uint8_t *src;
        if (!next_chunk(meta[b], src)) break;
        mbar_arrive_expect_tx(&cbar[b], meta[b].bytes);
        bulk_g2s_hint(stages + b * CH, src, meta[b].bytes, &cbar[b], pol);
        ++issued;
    }
    while (stored < issued) {
        const int b = static_cast<int>(stored % NS);
        if (!mbar_wait(&cbar[b], (cphase >> b) & 1u, PIPE_LIMIT_NS)) {
            bulk_wait<0>();
            set_error(ws, KOSMOS_ERR_DEVICE, meta[b].ticket);
            return false;
        }
        cphase ^= (1u << b);
        bulk_s2g(meta[b].dst, stages + b * CH, meta[b].bytes);
        bulk_commit();
        if (meta[b].last) {
            pend[npend] = meta[b];
            pend_at[npend] = stored;
            ++npend;
        }
        if (npend > 0 && pend_at[0] + DEFER <= stored) {
            bulk_wait<DEFER>();
            int k = 0;
            while (k < npend && pend_at[k] + DEFER <= stored) move_release(pend[k++], done);
            for (int j = k; j < npend; ++j) {
                pend[j - k] = pend[j];
                pend_at[j - k] = pend_at[j];
            }
            npend -= k;
        }
        // refill the previous chunk's stage once its store has read it
        if (stored >= 1) {
            MoveChunk nc;
            const uint8_t *src;
            if (next_chunk(nc, src)) {
                bulk_wait_read<1>();
                const int rb = static_cast<int>((stored - 1) % NS);
                meta[rb] = nc;
                mbar_arrive_expect_tx(&cbar[rb], nc.bytes);
                bulk_g2s_hint(stages + rb * CH, src, nc.bytes, &cbar[rb], pol);
                ++issued;
            }
        }
        ++stored;
    }
    bulk_wait<0>();
    for (int k = 0; k < npend; ++k) move_release(pend[k], done);
    return true;
}

// Unfused all-gather copy kernels (grid-stride over 16-byte words, the first
// `local` words being the local shard's): once a block has copied its words,
// it reserves the link for the remote ones and waits until they would have
// crossed it.
__device__ __forceinline__ void ag_copy_link_pace(WsHeader *ws, int64_t local, int64_t total, int64_t gbs) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t mine = 0;  // remote words of this thread
    for (int64_t v = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < total; v += stride)
        mine += v >= local ? 1 : 0;
    __shared__ unsigned long long s_words;
    if (threadIdx.x == 0) s_words = 0;
    __syncthreads();
    atomicAdd(&s_words, static_cast<unsigned long long>(mine));
    __syncthreads();
    if (threadIdx.x == 0 && s_words > 0) link_wait(link_reserve(ws, s_words * 16ull, gbs));
    __syncthreads();
}

// ---------------------------------------------------------------- setup / teardown
__device__ __forceinline__ void engine_setup(const Smem &sm, int warp) {
    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
            mbar_init(&sm.cbar[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.tfull[i], 1);
            mbar_init(&sm.tempty[i], 4);
        }
        for (int i = 0; i < NSCHED; ++i) {
            mbar_init(&sm.sfull[i], 1);
            mbar_init(&sm.sempty[i], 5);
        }
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(sm.tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// The last CTA to finish returns the rail counters to zero and advances the
// epoch, leaving the workspace ready for the next stream-ordered call.
__device__ __forceinline__ void engine_finish(WsHeader *ws, uint32_t epoch, int n_tickets) {
    __threadfence();
    const uint32_t prev = atomicAdd(&ws->done_ctas, 1u);
    if (prev == gridDim.x - 1) {
        __threadfence();
        volatile uint32_t *t = ws->tickets;
        for (int i = 0; i < n_tickets; ++i) t[i] = 0u;
        *reinterpret_cast<volatile uint64_t *>(&ws->link_t0) = 0ull;
        *reinterpret_cast<volatile uint64_t *>(&ws->link_bytes) = 0ull;
        *reinterpret_cast<volatile uint32_t *>(&ws->done_ctas) = 0u;
        __threadfence();
        *reinterpret_cast<volatile uint32_t *>(&ws->epoch) = epoch + 1u;
        __threadfence();
    }
}

__device__ __forceinline__ void engine_teardown(const Smem &sm, int warp, uint32_t tmem_base) {
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- ring (producer side)
__device__ __forceinline__ bool ring_push(const Smem &sm, RingState &rs, const SchedEntry &e, WsHeader *ws) {
    if (!mbar_wait(&sm.sempty[rs.idx], rs.phase ^ 1u, PIPE_LIMIT_NS)) {
        set_error(ws, KOSMOS_ERR_DEVICE, -2);
        return false;
    }
    sm.sched[rs.idx] = e;
    mbar_arrive(&sm.sfull[rs.idx]);
    rs.advance();
    return true;
}

// ---------------------------------------------------------------- MMA warp
// Issues, for each TILE entry, nstage K blocks of BM x BN x BK into accumulator
// acc (TMEM columns acc*BN .. acc*BN+BN-1).  A: K-major, 128-byte swizzle
// (rows of 128 bytes, 8-row atoms of 1024 bytes).  B: N-major, 128-byte
// swizzle, four 64-column slabs of 8 KB (LBO = 8 KB between slabs,
// SBO = 1 KB between 8-row K groups).
__device__ __forceinline__ void mma_loop(const Smem &sm, uint32_t tmem_base, WsHeader *ws) {
    constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, false, true);
    PipeState ps;
    RingState rs;
    uint32_t acc = 0, acc_phase = 0;
    while (true) {
        if (!mbar_wait(&sm.sfull[rs.idx], rs.phase, PIPE_LIMIT_NS)) {
            set_error(ws, KOSMOS_ERR_DEVICE, -3);
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
        // N of this entry's MMA: a multiple of 16 in [16, 256] (0 selects BN)
        const uint32_t idesc = (e.nmma > 0 && e.nmma < BN) ? idesc_bf16_f32(BM, e.nmma, false, true) : IDESC;
        if (!mbar_wait(&sm.tempty[acc], acc_phase ^ 1u, PIPE_LIMIT_NS)) {
            set_error(ws, KOSMOS_ERR_DEVICE, -4);
            break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < e.nstage; ++kb) {
            if (!mbar_wait(&sm.full[ps.stage], ps.phase, PIPE_LIMIT_NS)) {
                set_error(ws, KOSMOS_ERR_DEVICE, -5);
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sm.stages + ps.stage * STAGE_BYTES);
            const uint32_t b_addr = a_addr + A_STAGE_BYTES;
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k) {
                const uint64_t ad = sdesc_sw128(a_addr + k * (UMMA_K * 2), 16, 1024);
                const uint64_t bd = sdesc_sw128(b_addr + k * (UMMA_K * 128), 64 * 128, 1024);
                mma_bf16_ss(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            }
            mma_commit(&sm.empty[ps.stage]);
            ps.advance();
        }
        if (!ok) break;
        mma_commit(&sm.tfull[acc]);
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
}

// ---------------------------------------------------------------- epilogue helpers
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Reads 32 fp32 columns of this thread's accumulator row and stores them as
// bf16 at dst (16-byte stores; columns >= ncols_valid are skipped in groups
// of 8).  tcgen05.ld is warp-collective: every lane calls this.
__device__ __forceinline__ void tmem_row_chunk_to_bf16(uint32_t taddr, bool row_valid, __nv_bfloat16 *dst,
                                                       int ncols_valid) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr, r);
    tmem_ld_wait();
    if (row_valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (q * 8 < ncols_valid) {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(r[q * 8 + 0]), __uint_as_float(r[q * 8 + 1]));
                v.y = pack_bf16x2(__uint_as_float(r[q * 8 + 2]), __uint_as_float(r[q * 8 + 3]));
                v.z = pack_bf16x2(__uint_as_float(r[q * 8 + 4]), __uint_as_float(r[q * 8 + 5]));
                v.w = pack_bf16x2(__uint_as_float(r[q * 8 + 6]), __uint_as_float(r[q * 8 + 7]));
                *reinterpret_cast<uint4 *>(dst + q * 8) = v;
            }
        }
    }
}

// Row-segment stores from the epilogue's row-per-lane layout.  Each
// epilogue thread holds one accumulator row (lane = row of the warp's 32).
// v holds eight 16-byte units (4 words each: 8 bf16 columns) of this lane's
// row; after an 8 x 8 transpose of units among lanes 8g..8g+7 (three
// butterfly stages of shuffles) lane 8g+i holds unit i of rows 8g..8g+7, so
// each warp store instruction writes four whole 128-byte row segments
// instead of 16 bytes of 32 rows.  All 32 lanes must call it (shuffles).
__device__ __forceinline__ void lane_transpose8_16B(uint32_t (&v)[32], int lane) {
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {
        const bool up = (lane & m) != 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j & m) continue;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t send = up ? v[4 * j + w] : v[4 * (j + m) + w];
                const uint32_t recv = __shfl_xor_sync(0xFFFFFFFFu, send, m);
                if (up) v[4 * j + w] = recv;
                else v[4 * (j + m) + w] = recv;
            }
        }
    }
}
// Stores the transposed block: dst0 = the warp's first row at the block's
// first column, ld = row stride, rows / ncols = valid rows of the warp's 32
// and valid columns of the 64 (a multiple of 8).
__device__ __forceinline__ void store_row_lines(const uint32_t (&v)[32], __nv_bfloat16 *dst0, int64_t ld, int rows,
                                                int ncols, int lane) {
    const int g = lane >> 3, i = lane & 7;
    if (8 * i < ncols) {
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int r = 8 * g + s;
            if (r < rows)
                *reinterpret_cast<uint4 *>(dst0 + r * ld + 8 * i) =
                    make_uint4(v[4 * s], v[4 * s + 1], v[4 * s + 2], v[4 * s + 3]);
        }
    }
}
// 64 accumulator columns of this thread's row to bf16, stored as row
// segments (arguments as for store_row_lines).
__device__ __forceinline__ void tmem_rows64_to_bf16_lines(uint32_t taddr, __nv_bfloat16 *dst0, int64_t ld, int rows,
                                                          int ncols, int lane) {
    uint32_t pk[32];
    {
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32(taddr, r0);
        tmem_ld_32x32b_x32(taddr + 32, r1);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            pk[j] = pack_bf16x2(__uint_as_float(r0[2 * j]), __uint_as_float(r0[2 * j + 1]));
            pk[16 + j] = pack_bf16x2(__uint_as_float(r1[2 * j]), __uint_as_float(r1[2 * j + 1]));
        }
    }
    lane_transpose8_16B(pk, lane);
    store_row_lines(pk, dst0, ld, rows, ncols, lane);
}

// Epilogue of one CTA's 128 x 256 accumulator for a tile computed as two K
// halves by two entries (possibly on two engines).  The first of the two to
// arrive stores its fp32 partial in the slot and releases the slot's flag;
// the second waits for the flag, adds the partial to its own accumulator
// (fp32 addition is commutative, so the result does not depend on which half
// finished first), writes Y and returns the slot's counter to zero.  Called
// by all 128 epilogue threads; thread `row` owns accumulator row `row`;
// xword points to two shared-memory words.  Returns false after a device error.
__device__ __forceinline__ bool khalf_epilogue(uint32_t taddr, bool row_valid, __nv_bfloat16 *yrow, int64_t col0,
                                               int64_t n, float4 *part, uint32_t *cnt, uint32_t *flag,
                                               uint32_t epoch, WsHeader *ws, uint64_t limit_ns, int64_t entry,
                                               int row, uint32_t *xword) {
    const bool lead = row == 0;
    if (lead) xword[0] = atomicAdd(cnt, 1u);
    named_bar_sync(1, NUM_EPI_THREADS);
    const uint32_t order = *reinterpret_cast<volatile uint32_t *>(&xword[0]);
    if (order == 0) {
#pragma unroll 1
        for (int ch = 0; ch < BN / 32; ++ch) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + ch * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int v = 0; v < 8; ++v)
                part[(ch * 8 + v) * BM + row] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                                            __uint_as_float(r[4 * v + 2]),
                                                            __uint_as_float(r[4 * v + 3]));
        }
        __threadfence();
        named_bar_sync(1, NUM_EPI_THREADS);
        if (lead) st_release_gpu(flag, epoch + 1u);
        return true;
    }
    if (lead) {
        const bool ok = wait_flag_eq(ws, flag, epoch + 1u, limit_ns, entry);
        st_relaxed_gpu(cnt, 0u);
        xword[1] = ok ? 1u : 0u;
    }
    named_bar_sync(1, NUM_EPI_THREADS);
    if (*reinterpret_cast<volatile uint32_t *>(&xword[1]) == 0u) return false;
    // 64 columns (16 float4 of the partner's partial) per pass; the next
    // pass's loads are in flight while this one is combined
    float4 pv[2][16];
#pragma unroll
    for (int v = 0; v < 16; ++v) pv[0][v] = __ldcg(&part[v * BM + row]);
#pragma unroll
    for (int ps = 0; ps < BN / 64; ++ps) {
        if (ps + 1 < BN / 64) {
#pragma unroll
            for (int v = 0; v < 16; ++v) pv[(ps + 1) & 1][v] = __ldcg(&part[((ps + 1) * 16 + v) * BM + row]);
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int ch = ps * 2 + cc;
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + ch * 32, r);
            tmem_ld_wait();
            const int64_t c0 = col0 + ch * 32;
            if (!row_valid || c0 >= n) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (c0 + q * 8 >= n) break;
                const float4 a = pv[ps & 1][cc * 8 + 2 * q];
                const float4 b = pv[ps & 1][cc * 8 + 2 * q + 1];
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(r[q * 8 + 0]) + a.x, __uint_as_float(r[q * 8 + 1]) + a.y);
                v.y = pack_bf16x2(__uint_as_float(r[q * 8 + 2]) + a.z, __uint_as_float(r[q * 8 + 3]) + a.w);
                v.z = pack_bf16x2(__uint_as_float(r[q * 8 + 4]) + b.x, __uint_as_float(r[q * 8 + 5]) + b.y);
                v.w = pack_bf16x2(__uint_as_float(r[q * 8 + 6]) + b.z, __uint_as_float(r[q * 8 + 7]) + b.w);
                *reinterpret_cast<uint4 *>(yrow + c0 + q * 8) = v;
            }
        }
    }
    return true;
}

__device__ __forceinline__ TraceRec *trace_rec(TraceRec *base, int cta, int slot) {
    return (base != nullptr && slot >= 0 && slot < TRACE_CAP) ? base + static_cast<int64_t>(cta) * TRACE_CAP + slot
                                                              : nullptr;
}

}  // namespace kosmos
