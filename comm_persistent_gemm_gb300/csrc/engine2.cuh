// engine2.cuh -- the SM-pair persistent engine (tcgen05 cta_group::2).
//
// CTAs run in clusters of two on the two SMs of a TPC.  A pair computes one
// 256 x 256 output tile per entry: each CTA stages its own 128 rows of A and
// its own 128 columns of B (so each SM's shared memory supplies half of B and
// the B operand's shared-memory traffic per SM halves), the leader (cluster
// rank 0) issues tcgen05.mma.cta_group::2 with M = 256, and each CTA's TMEM
// receives its 128 rows x 256 fp32 columns.
//
// Per CTA: warp 0 producer, warp 1 MMA issuer (leader only), warps 2-5
// epilogue.  The leader's producer claims entries and mirrors each one into
// the peer's entry ring over distributed shared memory; both producers stream
// their halves with TMA .cta_group::2 into their own stages, completing on the
// leader's "full" barriers; the leader's commits multicast to both CTAs'
// "empty" and "accumulator full" barriers; the peer's epilogue warps arrive
// remotely on the leader's "accumulator empty" barriers.  All waits bounded.
#pragma once
#include "engine.cuh"

namespace kosmos {

constexpr int HBM_ROWS = 128;                   // rows per CTA
constexpr int HBN = 128;                        // B columns per CTA
constexpr int NSTAGE2 = 7;                      // 224 KB of stages: loads are latency-bound below ~7
constexpr int A2_BYTES = HBM_ROWS * BK * 2;     // 16 KB
constexpr int B2_BYTES = BK * HBN * 2;          // 16 KB (two 64-column slabs)
constexpr int STAGE2_BYTES = A2_BYTES + B2_BYTES;
constexpr int SMEM2_CTRL = 2048;
constexpr int SMEM2_BYTES = NSTAGE2 * STAGE2_BYTES + SMEM2_CTRL + 1024;
static_assert(SMEM2_BYTES <= 232448, "pair engine exceeds 227 KB of shared memory per CTA");

// ---------------------------------------------------------------- cluster helpers
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t mapa_u32(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (globaltimer() - t0 > limit_ns) return false;
    }
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *m, uint32_t leader_bar, int32_t c0,
                                                 int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(leader_bar), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair_hint(void *dst, const CUtensorMap *m, uint32_t leader_bar, int32_t c0,
                                                      int32_t c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(leader_bar), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void *dst, const CUtensorMap *m, uint32_t leader_bar, int32_t c0,
                                                 int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(leader_bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc2(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma2_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the barrier at this shared-memory offset in both CTAs of the
// pair when every tcgen05 op issued so far by this thread has completed.
__device__ __forceinline__ void mma2_commit_both(uint64_t *bar) {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}

// ---------------------------------------------------------------- shared memory
struct Smem2 {
    uint8_t *stages;    // NSTAGE2 * STAGE2_BYTES
    uint64_t *full;     // [NSTAGE2] leader only: both halves landed (count 1 + tx)
    uint64_t *empty;    // [NSTAGE2] each CTA: stage consumed (multicast commit)
    uint64_t *cbar;     // [NSTAGE2] mover copies
    uint64_t *tfull;    // [2] each CTA: accumulator ready (multicast commit)
    uint64_t *tempty;   // [2] leader: accumulator drained (4 local + 4 remote epilogue warps)
    uint64_t *sfull;    // [NSCHED] each CTA: entry published (by the leader's producer)
    uint64_t *sempty;   // [NSCHED] leader: entry read by its MMA + 4 epilogue warps
    uint64_t *pempty;   // [NSCHED] leader: entry read by the peer's producer + 4 epilogue warps
    SchedEntry *sched;  // [NSCHED]
    uint32_t *tmem_slot;
};

__device__ __forceinline__ Smem2 carve_smem2(uint8_t *raw) {
    const uintptr_t base = (reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023);
    uint8_t *p = reinterpret_cast<uint8_t *>(base);
    Smem2 s;
    s.stages = p;
    p += NSTAGE2 * STAGE2_BYTES;
    uint64_t *b = reinterpret_cast<uint64_t *>(p);
    s.full = b; b += NSTAGE2;
    s.empty = b; b += NSTAGE2;
    s.cbar = b; b += NSTAGE2;
    s.tfull = b; b += 2;
    s.tempty = b; b += 2;
    s.sfull = b; b += NSCHED;
    s.sempty = b; b += NSCHED;
    s.pempty = b; b += NSCHED;
    s.sched = reinterpret_cast<SchedEntry *>(b);
    s.tmem_slot = reinterpret_cast<uint32_t *>(s.sched + NSCHED);
    return s;
}

template <int NS>
struct PipeStateN {
    uint32_t stage = 0, phase = 0;
    __device__ __forceinline__ void advance() {
        if (++stage == NS) { stage = 0; phase ^= 1; }
    }
    __device__ __forceinline__ void advance(int n) {
        for (int i = 0; i < n; ++i) advance();
    }
};
using PipeState2 = PipeStateN<NSTAGE2>;

__device__ __forceinline__ void engine2_setup(const Smem2 &sm, int warp, int nstage = NSTAGE2) {
    if (threadIdx.x == 0) {
        for (int i = 0; i < nstage; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
            mbar_init(&sm.cbar[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.tfull[i], 1);
            mbar_init(&sm.tempty[i], 8);
        }
        for (int i = 0; i < NSCHED; ++i) {
            mbar_init(&sm.sfull[i], 1);
            mbar_init(&sm.sempty[i], 5);
            mbar_init(&sm.pempty[i], 5);
        }
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc2(sm.tmem_slot, TMEM_COLS);
        tmem_relinquish2();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // the peer's barriers are initialised before any remote arrive
    tc_fence_after();
}

__device__ __forceinline__ void engine2_teardown(const Smem2 &sm, int warp, uint32_t tmem_base) {
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc2(tmem_base, TMEM_COLS);
    }
}

// Leader: publish an entry into both CTAs' rings.
struct RingPair {
    uint32_t idx = 0, phase = 0;
    __device__ __forceinline__ void advance() {
        if (++idx == NSCHED) { idx = 0; phase ^= 1; }
    }
};
__device__ __forceinline__ bool ring2_push(const Smem2 &sm, RingPair &rs, const SchedEntry &e, WsHeader *ws) {
    if (!mbar_wait(&sm.sempty[rs.idx], rs.phase ^ 1u, PIPE_LIMIT_NS) ||
        !mbar_wait_cluster(&sm.pempty[rs.idx], rs.phase ^ 1u, PIPE_LIMIT_NS)) {
        set_error(ws, KOSMOS_ERR_DEVICE, -2);
        return false;
    }
    sm.sched[rs.idx] = e;
    const uint32_t remote = mapa_u32(smem_u32(&sm.sched[rs.idx]), 1);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(&e);
#pragma unroll
    for (int i = 0; i < static_cast<int>(sizeof(SchedEntry) / 4); ++i) st_cluster_u32(remote + 4 * i, w[i]);
    mbar_arrive(&sm.sfull[rs.idx]);
    mbar_arrive_remote(mapa_u32(smem_u32(&sm.sfull[rs.idx]), 1));
    rs.advance();
    return true;
}

// Consumer side (either CTA): take the next entry.  is_leader selects which
// "entry read" barrier to arrive on (the leader's local sempty, or the
// leader's pempty from the peer).  whole_warp: the caller is a full warp and
// only lane 0 arrives; otherwise the caller is a single thread.
__device__ __forceinline__ bool ring2_take(const Smem2 &sm, RingPair &rs, bool is_leader, SchedEntry &e, WsHeader *ws,
                                           bool whole_warp) {
    const bool ok = is_leader ? mbar_wait(&sm.sfull[rs.idx], rs.phase, PIPE_LIMIT_NS)
                              : mbar_wait_cluster(&sm.sfull[rs.idx], rs.phase, PIPE_LIMIT_NS);
    if (!ok) {
        set_error(ws, KOSMOS_ERR_DEVICE, -6);
        return false;
    }
    e = sm.sched[rs.idx];
    bool arrive = true;
    if (whole_warp) {
        __syncwarp();
        arrive = (threadIdx.x % 32) == 0;
    }
    if (arrive) {
        if (is_leader)
            mbar_arrive(&sm.sempty[rs.idx]);
        else
            mbar_arrive_remote(mapa_u32(smem_u32(&sm.pempty[rs.idx]), 0));
    }
    rs.advance();
    return true;
}

// Leader MMA warp: for each MMA entry, nstage K blocks of a 256 x 256 x 64
// pair tile into accumulator acc of both CTAs.  Per CTA: A 128 rows K-major
// 128B-swizzled, B 128 columns N-major 128B-swizzled in two 8 KB slabs.
__device__ __forceinline__ void mma2_loop(const Smem2 &sm, uint32_t tmem_base, WsHeader *ws) {
    constexpr uint32_t IDESC = idesc_bf16_f32(PBM, BN, false, true);
    PipeState2 ps;
    RingPair rs;
    uint32_t acc = 0, acc_phase = 0;
    while (true) {
        SchedEntry e;
        if (!ring2_take(sm, rs, true, e, ws, false)) break;
        if (e.kind == K_DONE) break;
        if (!is_mma_kind(e.kind)) {
            ps.advance(e.nstage);
            continue;
        }
        // N of this entry's MMA (both CTAs' columns): a multiple of 32 in [32, 256] (0 selects BN)
        const uint32_t idesc = (e.nmma > 0 && e.nmma < BN) ? idesc_bf16_f32(PBM, e.nmma, false, true) : IDESC;
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
            const uint32_t a_addr = smem_u32(sm.stages + ps.stage * STAGE2_BYTES);
            const uint32_t b_addr = a_addr + A2_BYTES;
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k) {
                const uint64_t ad = sdesc_sw128(a_addr + k * (UMMA_K * 2), 16, 1024);
                const uint64_t bd = sdesc_sw128(b_addr + k * (UMMA_K * 128), 64 * 128, 1024);
                mma2_bf16_ss(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            }
            mma2_commit_both(&sm.empty[ps.stage]);
            ps.advance();
        }
        if (!ok) break;
        mma2_commit_both(&sm.tfull[acc]);
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
}

// Releases accumulator acc after this warp's tcgen05.ld's completed: local
// arrive in the leader, remote arrive from the peer.
__device__ __forceinline__ void acc_release(const Smem2 &sm, uint32_t acc, bool is_leader, int lane) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
        if (is_leader)
            mbar_arrive(&sm.tempty[acc]);
        else
            mbar_arrive_remote(mapa_u32(smem_u32(&sm.tempty[acc]), 0));
    }
}

// Waits until every stage is free again (both CTAs' stages are released by the
// leader's multicast commits), so the stage buffers can serve as copy buffers.
template <int NS>
__device__ __forceinline__ bool drain_stages2(const Smem2 &sm, const PipeStateN<NS> &ps, WsHeader *ws) {
    for (int i = 0; i < NS; ++i) {
        uint32_t s = ps.stage + i, ph = ps.phase;
        if (s >= NS) { s -= NS; ph ^= 1u; }
        if (!mbar_wait(&sm.empty[s], ph ^ 1u, PIPE_LIMIT_NS)) {
            set_error(ws, KOSMOS_ERR_DEVICE, -11);
            return false;
        }
    }
    return true;
}

// The last CTA to finish (grid-wide) resets the rail counters and the epoch.
__device__ __forceinline__ void engine2_finish(WsHeader *ws, uint32_t epoch, int n_tickets) {
    engine_finish(ws, epoch, n_tickets);
}

}  // namespace kosmos
