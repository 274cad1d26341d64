// mxfp8.cuh -- shared pieces of the MXFP8 (E4M3 + E8M0 per 32 K) tensor-core
// paths: shared-memory descriptors of the scale atoms, the block-scaled
// instruction descriptor, and the SM-pair block-scaled engine (stage layout,
// MMA issue loop) used by the all-gather + GEMM and the GEMM +
// reduce-scatter kernels.
//
// Scale layout (MMA-tiled, produced by kosmos_mxfp8_quantize): for an operand
// with R scale rows (rows of X, columns of W) and K, the scale of (row r,
// K-block b) is at byte ((r/128)*(K/128) + b/4)*512 + (r%32)*16 + ((r/32)%4)*4
// + b%4.  One 512-byte atom covers 128 rows x 4 K-blocks; copied with
// tcgen05.cp 32x128b.warpx4 it lands in four TMEM columns, lane r%32 of every
// 32-lane group holding rows r%32 + 32c in column c, one byte per K-block.
#pragma once
#include <cuda_fp8.h>

#include "engine2.cuh"

namespace kosmos {

constexpr int FBK = 128;                       // K elements (bytes) per stage
constexpr int F_TMEM_SF = 256;                 // first TMEM column of the scale buffers
constexpr int F_TMEM_SF_STRIDE = 16;           // columns per stage: SFA 4, SFB 8 (+4 spare)


// Descriptor of a 32-row x 16-byte matrix stored contiguously (rows 16 bytes
// apart; 8-row core matrices 128 bytes apart), no swizzle.
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(128 >> 4) << 16;  // leading byte offset (one 16-byte column: unused)
    d |= static_cast<uint64_t>(128 >> 4) << 32;  // stride byte offset between 8-row core matrices
    d |= static_cast<uint64_t>(1) << 46;
    return d;
}

// Instruction descriptor, kind::mxf8f6f4 block-scaled: A/B E4M3 (format 0),
// A K-major, B MN-major, scale type E8M0 (bit 23), N >> 3 at bits 17-22,
// M >> 4 at bits 24-28, B scale byte at bits 4-5, A scale byte at bits 29-30.
__device__ __forceinline__ uint32_t idesc_mxf8(int M, int N, int sf_id) {
    return (static_cast<uint32_t>(sf_id) << 4) | (1u << 16) | (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
           (static_cast<uint32_t>(M >> 4) << 24) | (static_cast<uint32_t>(sf_id) << 29);
}

// ---------------------------------------------------------------- codec
// Shared exponent of one block: the smallest integer e with
// blockmax <= 448 * 2^e, clamped to [-127, 127]; 0 for an all-zero block.
// Write blockmax (a finite float) as f * 2^E with f in [1, 2); 448 = 1.75 * 2^8,
// so e = E - 8 when f <= 1.75 and E - 7 otherwise.
__device__ __forceinline__ int mx_block_exp(float blockmax) {
    const uint32_t b = __float_as_uint(blockmax);
    const int ex = static_cast<int>((b >> 23) & 0xFF);
    const uint32_t man = b & 0x7FFFFFu;
    if (ex == 0) return man == 0 ? 0 : -127;  // zero, or below 2^-126: clamped
    const int E = ex - 127;
    int e = (man <= 0x600000u) ? E - 8 : E - 7;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

// Byte offset of the scale of (scale row r, K-block b) in the MMA-tiled layout:
// 512-byte atoms of 128 scale rows x 4 K-blocks, atoms ordered by row block,
// then K; inside an atom row r sits at (r % 32) * 16 + ((r / 32) % 4) * 4.
__host__ __device__ __forceinline__ int64_t sf_tiled_offset(int64_t r, int64_t b, int64_t kblocks) {
    return ((r / 128) * (kblocks / 4) + b / 4) * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + (b % 4);
}

// One MXFP8 block of 32 values: the E4M3 bytes of v / 2^e (round to nearest
// even, saturating; exact scaling by a power of two) packed four to a word in
// element order, and the E8M0 byte e + 127 as the return value.
__device__ __forceinline__ uint32_t mx_quant32(const float (&v)[32], uint32_t (&w)[8]) {
    float mx = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) mx = fmaxf(mx, fabsf(v[j]));
    const int e = mx_block_exp(mx);
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e (e <= 126 for finite input)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            word |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(v[4 * i + j] * inv, __NV_SATFINITE, __NV_E4M3))
                    << (8 * j);
        w[i] = word;
    }
    return static_cast<uint32_t>(e + 127);
}

// ---------------------------------------------------------------- single-SM pieces
__device__ __forceinline__ void mma_mxf8_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// 32 rows x 16 bytes from shared memory into TMEM lanes 0-31 of four columns,
// replicated to the four 32-lane groups.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// One 128-wide K stage of a 128 x 256 block-scaled tile on one SM: copy the
// stage's three scale atoms (SFA, SFB columns 0-127, SFB 128-255) into tensor
// memory at sfa_t, then four K = 32 MMAs.  A: 128 rows x 128 bytes, B: two
// 128-column slabs of b_slab bytes, both with the 128-byte swizzle.
__device__ __forceinline__ void mx_stage_mma(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr, uint32_t b_slab,
                                             uint32_t sf_addr, uint32_t sfa_t, bool first) {
    const uint32_t sfb_t = sfa_t + 4;
    tmem_cp_32x128b_x4(sfa_t, sdesc_sf(sf_addr));
    tmem_cp_32x128b_x4(sfb_t, sdesc_sf(sf_addr + 512));
    tmem_cp_32x128b_x4(sfb_t + 4, sdesc_sf(sf_addr + 1024));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint64_t ad = sdesc_sw128(a_addr + j * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(b_addr + j * (32 * 128), b_slab, 1024);
        mma_mxf8_ss(d_tmem, ad, bd, idesc_mxf8(BM, BN, j), sfa_t, sfb_t, (!first || j != 0) ? 1u : 0u);
    }
}

// ---------------------------------------------------------------- SM-pair engine
// Tiles of 256 x 256 on an SM pair (tcgen05.mma.cta_group::2, block-scaled).
// Each CTA stages its 128 rows of A, its 128 columns of B, the scale atom of
// its rows (SFA) and the scale atoms of all 256 columns (SFB); the leader's
// tcgen05.cp.cta_group::2 copies every CTA's atoms into that CTA's tensor
// memory, where the pair MMA reads SFA of the CTA's rows and SFB of the whole
// tile (the placement was checked on the GB300 against exact results).
constexpr int F2_NSTAGE = 6;
constexpr int F2_A_BYTES = HBM_ROWS * FBK;             // 16 KB
constexpr int F2_B_BYTES = HBN * FBK;                  // 16 KB
constexpr int F2_STAGE = F2_A_BYTES + F2_B_BYTES;
constexpr int F2_SF = 3 * 512;                         // SFA atom + two SFB atoms
constexpr int F2_SMEM_BYTES = F2_NSTAGE * (F2_STAGE + F2_SF) + SMEM2_CTRL + 1024;
static_assert(F2_SMEM_BYTES <= 232448, "MXFP8 pair engine exceeds 227 KB of shared memory per CTA");
using PipeF2 = PipeStateN<F2_NSTAGE>;

struct F2Smem {
    Smem2 base;
    uint8_t *sf;  // [F2_NSTAGE][F2_SF]
};

__device__ __forceinline__ F2Smem carve_f2(uint8_t *raw) {
    const uintptr_t b0 = (reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023);
    uint8_t *p = reinterpret_cast<uint8_t *>(b0);
    F2Smem f;
    Smem2 &s = f.base;
    s.stages = p;
    p += F2_NSTAGE * F2_STAGE;
    f.sf = p;
    p += F2_NSTAGE * F2_SF;
    uint64_t *b = reinterpret_cast<uint64_t *>(p);
    s.full = b; b += F2_NSTAGE;
    s.empty = b; b += F2_NSTAGE;
    s.cbar = b; b += F2_NSTAGE;
    s.tfull = b; b += 2;
    s.tempty = b; b += 2;
    s.sfull = b; b += NSCHED;
    s.sempty = b; b += NSCHED;
    s.pempty = b; b += NSCHED;
    s.sched = reinterpret_cast<SchedEntry *>(b);
    s.tmem_slot = reinterpret_cast<uint32_t *>(s.sched + NSCHED);
    return f;
}

__device__ __forceinline__ void mma2_mxf8_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}
// Issued by the leader: each CTA of the pair copies its own shared-memory
// atom into its own tensor memory.
__device__ __forceinline__ void tmem_cp2_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Leader only: per stage, copy the pair's scale atoms into tensor memory, then
// four K = 32 block-scaled MMAs into the single accumulator (columns 0-255).
__device__ __forceinline__ void f2_mma_loop(const F2Smem &fs, uint32_t tmem_base, WsHeader *ws) {
    const Smem2 &sm = fs.base;
    PipeF2 ps;
    RingPair rs;
    uint32_t acc_phase = 0;
    while (true) {
        SchedEntry e;
        if (!ring2_take(sm, rs, true, e, ws, false)) break;
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
            const uint32_t a_addr = smem_u32(sm.stages + ps.stage * F2_STAGE);
            const uint32_t b_addr = a_addr + F2_A_BYTES;
            const uint32_t sf_addr = smem_u32(fs.sf + ps.stage * F2_SF);
            const uint32_t sfa_t = tmem_base + F_TMEM_SF + ps.stage * F_TMEM_SF_STRIDE;
            const uint32_t sfb_t = sfa_t + 4;
            tmem_cp2_32x128b_x4(sfa_t, sdesc_sf(sf_addr));
            tmem_cp2_32x128b_x4(sfb_t, sdesc_sf(sf_addr + 512));
            tmem_cp2_32x128b_x4(sfb_t + 4, sdesc_sf(sf_addr + 1024));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint64_t ad = sdesc_sw128(a_addr + j * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(b_addr + j * (32 * 128), F2_B_BYTES, 1024);
                mma2_mxf8_ss(tmem_base, ad, bd, idesc_mxf8(PBM, BN, j), sfa_t, sfb_t, (kb | j) != 0 ? 1u : 0u);
            }
            mma2_commit_both(&sm.empty[ps.stage]);
            ps.advance();
        }
        if (!ok) break;
        mma2_commit_both(&sm.tfull[0]);
        acc_phase ^= 1u;
    }
}

}  // namespace kosmos
