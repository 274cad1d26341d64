// launch.h -- host-side interfaces between the C ABI (host.cu) and the
// per-operator launchers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/kosmos.h"

namespace kosmos {

struct AgLaunch {
    int P;
    int64_t m, k, n;
    const void *x[KOSMOS_MAX_P];
    const void *xs[KOSMOS_MAX_P];  // MXFP8 scales
    const void *w;
    const void *wsc;               // MXFP8 scales
    void *x_gathered;
    void *y;
    void *ws;
    int dtype;
    int sched;
    int n_comm;
    int trace;
    int grid;
    int pair;       // 1: SM-pair (cta_group::2) tiles, grid = 2 x clusters
    int plain_launch;
    int64_t n_split;  // trailing tiles of the tile rail run as two K halves
    int n_slots;      // K-split slots in the workspace (>= n_split)
    uint64_t wait_limit_ns;
    uint64_t inject;
    int64_t link_gbs;
    int host_flow;    // bf16: shards arrive through copy streams (arrival and output-done words in the workspace)
};

struct RsLaunch {
    int P;
    int64_t m, k, n;
    const void *x[KOSMOS_MAX_P];
    const void *w[KOSMOS_MAX_P];
    const void *xs[KOSMOS_MAX_P];   // MXFP8 scales of X_r
    const void *ws_[KOSMOS_MAX_P];  // MXFP8 scales of W_r
    void *y[KOSMOS_MAX_P];
    void *ws;
    int dtype;
    int sched;
    int n_comm;
    int order;
    int trace;
    int grid;
    int pair;
    int plain_launch;
    uint64_t wait_limit_ns;
    uint64_t inject;
    int64_t link_gbs;
};

struct MoeLaunch {
    int P;
    int64_t T, H, I;
    int E, K;
    const void *x[KOSMOS_MAX_P];
    const void *wr;
    const void *wg[KOSMOS_MAX_P];
    const void *wu[KOSMOS_MAX_P];
    const void *wd[KOSMOS_MAX_P];
    const void *wgs[KOSMOS_MAX_P];  // MXFP8: tiled scales of the gate / up / down weights
    const void *wus[KOSMOS_MAX_P];
    const void *wds[KOSMOS_MAX_P];
    int dtype;
    void *y[KOSMOS_MAX_P];
    int32_t *topk_idx;
    float *topk_gate;
    int32_t *counts;
    int32_t *pos;
    void *ws;
    int sched;
    int n_comm;
    int trace;
    int grid;
    int plain_launch;
    uint64_t wait_limit_ns;
    uint64_t inject;
};

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
bool encode_tmap(CUtensorMap *map, CUtensorMapDataType dt, int rank, void *base, const uint64_t *dims,
                 const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swizzle);

// Tensor map over `atoms` MXFP8 scale atoms stored one after another from
// `base` (512 contiguous bytes each): four rows of 128 bytes per atom, box
// = one atom.  The copy unit's cost follows the rows of a box, so an atom
// costs four rows here instead of the 32 of its 16-byte scale rows.  Atom a
// starts at row a * SF_ATOM_ROWS.
bool encode_sf_tmap(CUtensorMap *map, void *base, uint64_t atoms);

// Cooperative launch of a persistent kernel whose only argument is *params
// (plain = true: the same grid without the cooperative attribute).
kosmos_status launch_persistent(const void *func, void *params, int grid, int smem_bytes, cudaStream_t stream,
                                bool plain = false);
// The same with clusters of two CTAs (SM pairs); grid must be even.
kosmos_status launch_persistent_pairs(const void *func, void *params, int grid, int smem_bytes, cudaStream_t stream,
                                      bool plain = false);
// Number of CTAs a pair-kernel grid may have on the current device (2 x the
// co-resident clusters of two at ~200 KB of shared memory), or -1.
int max_pair_ctas(const void *func, int smem_bytes);

kosmos_status launch_ag_bf16(const AgLaunch &L, cudaStream_t stream);
// K-split slots a workspace holds for these sizes and options (0 without a tail split).
int ag_split_slots(int P, int64_t m, int64_t n, int dtype, const kosmos_opts &o);
kosmos_status launch_ag_mxfp8(const AgLaunch &L, cudaStream_t stream);
size_t ag_mxfp8_scale_bytes(int P, int64_t m, int64_t k);
kosmos_status launch_rs_bf16(const RsLaunch &L, cudaStream_t stream);
kosmos_status launch_moe_fwd(const MoeLaunch &L, cudaStream_t stream);

struct MoeBwdLaunch {
    int P;
    int64_t T, H, I;
    int E, K;
    const void *x[KOSMOS_MAX_P];
    const void *wr;
    const void *wg[KOSMOS_MAX_P];
    const void *wu[KOSMOS_MAX_P];
    const void *wd[KOSMOS_MAX_P];
    const int32_t *topk_idx;
    const float *topk_gate;
    const void *fwd_ws;
    const void *dout[KOSMOS_MAX_P];
    void *dx[KOSMOS_MAX_P];
    float *dwr;
    void *dwg[KOSMOS_MAX_P];
    void *dwu[KOSMOS_MAX_P];
    void *dwd[KOSMOS_MAX_P];
    void *ws;
    int sched;   // KOSMOS_SCHED_SELF (one launch) or KOSMOS_SCHED_UNFUSED (one launch per phase)
    int trace;
    int grid;
    int plain_launch;
    uint64_t wait_limit_ns;
};
kosmos_status launch_moe_bwd(const MoeBwdLaunch &L, cudaStream_t stream);
size_t moe_bwd_workspace_bytes(int P, int64_t T, int64_t H, int E, int K, int64_t I, bool trace);
bool moe_bwd_debug_view(int what, int P, int64_t T, int64_t H, int E, int K, int64_t I, void *ws, void **ptr,
                        int64_t *bytes);
size_t moe_workspace_bytes(int P, int64_t T, int64_t H, int E, int K, int64_t I, bool mx, bool trace);
bool moe_debug_view(int what, int P, int64_t T, int64_t H, int E, int K, int64_t I, bool mx, void *ws, void **ptr,
                    int64_t *bytes);
kosmos_status launch_mxfp8_quantize(const void *x, int64_t rows, int64_t cols, int along_cols, void *q,
                                    void *scales, cudaStream_t stream);
kosmos_status launch_rail_decode(int op, int P, int64_t m, int64_t n, int order, int rank, int rail, int tile_m,
                                 int64_t split,
                                 int32_t *out, int64_t count, cudaStream_t stream);
int ag_pair_grid_limit();
int ag_mxfp8_pair_grid_limit();
int rs_pair_grid_limit(bool mx = false);

}  // namespace kosmos
