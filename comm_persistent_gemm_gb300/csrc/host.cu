// host.cu -- the C ABI: argument validation, workspace sizing, status
// read-back, rail decode, and dispatch to the operator launchers.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>

#include "common.cuh"
#include "launch.h"

using namespace kosmos;

namespace kosmos {

typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                      const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                      CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                      CUtensorMapFloatOOBfill);

static PFN_encodeTiled_t get_encode_fn() {
    static PFN_encodeTiled_t fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_encodeTiled_t>(p);
    }
    return fn;
}

// Tokens of the host-input all-gather calls: the value its streams exchange
// through the workspace's join words, distinct from the previous call's.
static std::atomic<uint32_t> g_host_flow_token{0};

// The arrival words of the host-input all-gather are set by a 4-byte copy of
// this pinned word (value 1) after each chunk's copy on the same stream: the
// copy starts once the chunk's copy has completed, and costs the copy engine
// less than a stream write operation.  Allocated once, never freed.
static const uint32_t *host_one_word() {
    static std::atomic<uint32_t *> word{nullptr};
    uint32_t *w = word.load(std::memory_order_acquire);
    if (w == nullptr) {
        void *p = nullptr;
        if (cudaHostAlloc(&p, 16, cudaHostAllocPortable) != cudaSuccess) return nullptr;
        static_cast<uint32_t *>(p)[0] = 1u;
        uint32_t *expected = nullptr;
        if (!word.compare_exchange_strong(expected, static_cast<uint32_t *>(p), std::memory_order_acq_rel)) {
            cudaFreeHost(p);  // another thread installed its word first
            return expected;
        }
        w = static_cast<uint32_t *>(p);
    }
    return w;
}

// Stream memory operations (write / wait on a 32-bit word in device memory).
typedef CUresult (*PFN_streamValue32_t)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
static PFN_streamValue32_t get_stream_value_fn(bool wait) {
    static PFN_streamValue32_t fw = nullptr, fr = nullptr;
    PFN_streamValue32_t &fn = wait ? fr : fw;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion(wait ? "cuStreamWaitValue32" : "cuStreamWriteValue32", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_streamValue32_t>(p);
    }
    return fn;
}

bool encode_tmap(CUtensorMap *map, CUtensorMapDataType dt, int rank, void *base, const uint64_t *dims,
                 const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swizzle) {
    PFN_encodeTiled_t fn = get_encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) s[i] = strides_bytes[i];
    }
    const CUresult r = fn(map, dt, static_cast<cuuint32_t>(rank), base, d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_sf_tmap(CUtensorMap *map, void *base, uint64_t atoms) {
    const uint64_t dims[2] = {128, atoms * SF_ATOM_ROWS};
    const uint64_t st[1] = {128};
    const uint32_t box[2] = {128, SF_ATOM_ROWS};
    return encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, st, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

kosmos_status launch_persistent(const void *func, void *params, int grid, int smem_bytes, cudaStream_t stream,
                                bool plain) {
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess)
        return KOSMOS_ERR_CUDA;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = plain ? 0 : 1;
    void *args[1] = {params};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, func, args);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return KOSMOS_ERR_CUDA;
    }
    return KOSMOS_OK;
}

kosmos_status launch_persistent_pairs(const void *func, void *params, int grid, int smem_bytes, cudaStream_t stream,
                                      bool plain) {
    if ((grid & 1) != 0 || grid < 2) return KOSMOS_ERR_INVALID_ARG;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess)
        return KOSMOS_ERR_CUDA;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = plain ? 1 : 2;
    void *args[1] = {params};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, func, args);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return KOSMOS_ERR_CUDA;
    }
    return KOSMOS_OK;
}

int max_pair_ctas(const void *func, int smem_bytes) {
    static const void *cached_func[8] = {};
    static int cached_dev[8] = {-1, -1, -1, -1, -1, -1, -1, -1};
    static int cached_val[8] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    for (int i = 0; i < 8; ++i)
        if (cached_func[i] == func && cached_dev[i] == dev) return cached_val[i];
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess) return -1;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, func, &cfg) != cudaSuccess || clusters < 1) {
        (void)cudaGetLastError();
        return -1;
    }
    for (int i = 0; i < 8; ++i)
        if (cached_func[i] == nullptr) {
            cached_func[i] = func;
            cached_dev[i] = dev;
            cached_val[i] = 2 * clusters;
            break;
        }
    return 2 * clusters;
}

}  // namespace kosmos

namespace {

int device_sms() {
    static int cached_dev = -1;
    static int cached_sms = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (dev != cached_dev) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
        cached_dev = dev;
        cached_sms = sms;
    }
    return cached_sms;
}

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The emulated link: 0 (off) or 1..1e6 GB/s, and the call's whole link
// traffic must cross it within half the wait bound (every wait stays bounded).
static bool link_ok(const kosmos_opts &o, uint64_t link_bytes) {
    if (o.link_gbs == 0) return true;
    if (o.link_gbs < 1 || o.link_gbs > 1000000) return false;
    return link_bytes / static_cast<uint64_t>(o.link_gbs) < o.wait_limit_ns / 2;
}

kosmos_opts resolve_opts(const kosmos_opts *o) {
    kosmos_opts r;
    kosmos_default_opts(&r);
    if (o) r = *o;
    if (r.wait_limit_ns == 0) r.wait_limit_ns = 2000000000ull;
    return r;
}

int grid_for(const kosmos_opts &o) {
    const int sms = device_sms();
    if (sms <= 0) return -1;
    int g = (o.num_ctas > 0 && o.num_ctas < sms) ? o.num_ctas : sms;
    if (g > MAX_CTAS) g = MAX_CTAS;
    return g;
}

// Movers at start (SELF) or the fixed crew size (FIXED): ceil(S/P) by default,
// kept within [1, grid-1] so at least one builder exists.
int resolve_comm(const kosmos_opts &o, int grid, int P, bool fixed) {
    int n = o.n_comm0 >= 0 ? o.n_comm0 : static_cast<int>((grid + P - 1) / P);
    if (fixed && o.fixed_comm_ctas >= 0) n = o.fixed_comm_ctas;
    if (n < 1) n = 1;
    if (grid > 1 && n > grid - 1) n = grid - 1;
    return n;
}

}  // namespace

int kosmos::ag_split_slots(int P, int64_t m, int64_t n, int dtype, const kosmos_opts &o) {
    if (dtype != KOSMOS_BF16 || o.tail_split == 0) return 0;
    int64_t s = ag_geom(P, m, 64, n, BM).n_full;  // 128-row tiles: the most tiles either engine has
    if (s > MAX_SPLIT_SLOTS) s = MAX_SPLIT_SLOTS;
    if (o.tail_split > 0 && o.tail_split < s) s = o.tail_split;
    return static_cast<int>(s);
}

namespace {

// Launch shape of one all-gather + GEMM call: grid, tile engine, initial
// movers (CTAs) and the tile-rail split.
struct AgPlan {
    int grid;
    int pair;
    int n_comm;
    int64_t n_split;
};

kosmos_status ag_plan(int P, int64_t m, int64_t k, int64_t n, int dtype, const kosmos_opts &o, AgPlan &pl) {
    int grid = grid_for(o);
    if (grid < 1) return KOSMOS_ERR_CUDA;
    int pair = o.cta_pair != 0 ? 1 : 0;
    if (pair) {
        const int lim = dtype == KOSMOS_BF16 ? ag_pair_grid_limit() : ag_mxfp8_pair_grid_limit();
        int g2 = grid & ~1;
        if (lim >= 2 && g2 > lim) g2 = lim;
        if (lim < 2 || g2 < 2) {
            if (o.cta_pair == 1) return KOSMOS_ERR_UNSUPPORTED;
            pair = 0;
        } else {
            grid = g2;
        }
    }
    if (o.sched == KOSMOS_SCHED_FIXED && grid < (pair ? 4 : 2)) return KOSMOS_ERR_INVALID_ARG;
    int n_comm = resolve_comm(o, grid, P, o.sched == KOSMOS_SCHED_FIXED);
    if (pair && n_comm > grid - 2) n_comm = grid - 2;  // keep a builder pair
    int64_t split = 0;
    if (dtype == KOSMOS_BF16 && k >= 2 * BK) {  // both K halves need at least one K block
        if (o.tail_split >= 0) {
            split = o.tail_split;
        } else {  // one wave: every tile engine that builds
            split = pair ? grid / 2 : grid;
            if (o.sched == KOSMOS_SCHED_FIXED) split -= pair ? (n_comm + 1) / 2 : n_comm;
        }
        const int64_t n_full = ag_geom(P, m, 64, n, pair ? PBM : BM).n_full;
        if (split > n_full) split = n_full;
        if (split > ag_split_slots(P, m, n, dtype, o)) split = ag_split_slots(P, m, n, dtype, o);
        if (split < 0) split = 0;
    }
    pl.grid = grid;
    pl.pair = pair;
    pl.n_comm = n_comm;
    pl.n_split = split;
    return KOSMOS_OK;
}

}  // namespace

extern "C" {

void kosmos_default_opts(kosmos_opts *opts) {
    if (!opts) return;
    memset(opts, 0, sizeof(*opts));
    opts->sched = KOSMOS_SCHED_SELF;
    opts->n_comm0 = -1;
    opts->fixed_comm_ctas = -1;
    opts->order = KOSMOS_ORDER_BAND;
    opts->num_ctas = -1;
    opts->trace = 0;
    opts->cta_pair = -1;
    opts->plain_launch = 0;
    opts->tail_split = 0;
    opts->link_gbs = 0;
    opts->wait_limit_ns = 0;
    opts->inject = 0;
}

int kosmos_num_sms(void) { return device_sms(); }

size_t kosmos_workspace_bytes(int op, int P, int64_t m, int64_t n, int64_t k, int dtype, const kosmos_opts *opts) {
    const kosmos_opts o = resolve_opts(opts);
    if (P < 1 || P > KOSMOS_MAX_P || m < 1 || n < 1 || k < 1) return 0;
    if (op == KOSMOS_OP_AG_GEMM) {
        size_t total = ag_ws_layout(ag_geom(P, m, k, n), o.trace != 0, ag_split_slots(P, m, n, dtype, o)).total;
        if (dtype == KOSMOS_MXFP8_E4M3) {
            if (k % 128) return 0;
            total += ag_mxfp8_scale_bytes(P, m, k);  // gathered scale blocks
        }
        return total;
    }
    if (op == KOSMOS_OP_GEMM_RS) {
        if (m % P) return 0;
        return rs_ws_layout(rs_geom(P, m, k, n), o.trace != 0).total;
    }
    return 0;
}

kosmos_status kosmos_workspace_init(void *ws, size_t ws_bytes, void *stream) {
    if (!aligned16(ws) || ws_bytes < 256) return KOSMOS_ERR_INVALID_ARG;
    if (cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KOSMOS_ERR_CUDA;
    return KOSMOS_OK;
}

kosmos_status kosmos_ag_gemm(const void *const *x_shards, const void *const *x_scales, int P, int64_t m_per_shard,
                             int64_t k, int64_t n, const void *w, const void *w_scales, int dtype, void *x_gathered,
                             void *y, void *ws, size_t ws_bytes, const kosmos_opts *opts, void *stream) {
    if (P < 1 || P > KOSMOS_MAX_P || x_shards == nullptr) return KOSMOS_ERR_INVALID_ARG;
    if (m_per_shard < 1 || k < BK || n < 8 || n % 8 != 0) return KOSMOS_ERR_INVALID_ARG;
    if (m_per_shard > (1ll << 30) || k > (1ll << 24) || n > (1ll << 24)) return KOSMOS_ERR_INVALID_ARG;
    if (dtype != KOSMOS_BF16 && dtype != KOSMOS_MXFP8_E4M3) return KOSMOS_ERR_INVALID_ARG;
    if (dtype == KOSMOS_BF16 && k % BK != 0) return KOSMOS_ERR_INVALID_ARG;
    if (dtype == KOSMOS_MXFP8_E4M3 && (k % 128 != 0 || n % 16 != 0)) return KOSMOS_ERR_INVALID_ARG;
    for (int r = 0; r < P; ++r) {
        if (!aligned16(x_shards[r])) return KOSMOS_ERR_INVALID_ARG;
        if (dtype == KOSMOS_MXFP8_E4M3 && (x_scales == nullptr || !aligned16(x_scales[r])))
            return KOSMOS_ERR_INVALID_ARG;
    }
    if (!aligned16(w) || !aligned16(x_gathered) || !aligned16(y)) return KOSMOS_ERR_INVALID_ARG;
    if (dtype == KOSMOS_MXFP8_E4M3 && !aligned16(w_scales)) return KOSMOS_ERR_INVALID_ARG;
    if (!aligned16(ws)) return KOSMOS_ERR_WORKSPACE;
    const kosmos_opts o = resolve_opts(opts);
    if (o.sched < KOSMOS_SCHED_SELF || o.sched > KOSMOS_SCHED_UNFUSED) return KOSMOS_ERR_INVALID_ARG;
    if (!link_ok(o, static_cast<uint64_t>(P - 1) * static_cast<uint64_t>(m_per_shard) * static_cast<uint64_t>(k) *
                        (dtype == KOSMOS_BF16 ? 2u : 1u)))
        return KOSMOS_ERR_INVALID_ARG;
    if (ws_bytes < kosmos_workspace_bytes(KOSMOS_OP_AG_GEMM, P, m_per_shard, n, k, dtype, &o))
        return KOSMOS_ERR_WORKSPACE;
    AgPlan pl;
    const kosmos_status ps = ag_plan(P, m_per_shard, k, n, dtype, o, pl);
    if (ps != KOSMOS_OK) return ps;
    AgLaunch L;
    memset(&L, 0, sizeof(L));
    L.P = P; L.m = m_per_shard; L.k = k; L.n = n;
    for (int r = 0; r < P; ++r) {
        L.x[r] = x_shards[r];
        L.xs[r] = x_scales ? x_scales[r] : nullptr;
    }
    L.w = w; L.wsc = w_scales; L.x_gathered = x_gathered; L.y = y; L.ws = ws;
    L.dtype = dtype; L.sched = o.sched;
    L.n_comm = pl.n_comm;
    L.pair = pl.pair;
    L.n_split = pl.n_split;
    L.n_slots = ag_split_slots(P, m_per_shard, n, dtype, o);
    L.trace = o.trace; L.grid = pl.grid; L.wait_limit_ns = o.wait_limit_ns; L.inject = o.inject;
    L.plain_launch = o.plain_launch;
    L.link_gbs = o.link_gbs;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dtype == KOSMOS_BF16 ? launch_ag_bf16(L, s) : launch_ag_mxfp8(L, s);
}

kosmos_status kosmos_ag_gemm_host(const void *const *x_host, void *const *x_dev, int P, int64_t m_per_shard,
                                  int64_t k, int64_t n, const void *w, void *x_gathered, void *y_dev, void *y_host,
                                  void *ws, size_t ws_bytes, const kosmos_opts *opts, void *stream, void *h2d_stream,
                                  void *d2h_stream) {
    if (P < 1 || P > KOSMOS_MAX_P || x_host == nullptr || x_dev == nullptr || y_host == nullptr) return KOSMOS_ERR_INVALID_ARG;
    if (m_per_shard < 1 || k < BK || k % BK != 0 || n < 8 || n % 8 != 0) return KOSMOS_ERR_INVALID_ARG;
    if (m_per_shard > (1ll << 30) || k > (1ll << 24) || n > (1ll << 24)) return KOSMOS_ERR_INVALID_ARG;
    if (h2d_stream == nullptr || d2h_stream == nullptr || h2d_stream == stream || d2h_stream == stream)
        return KOSMOS_ERR_INVALID_ARG;
    for (int r = 0; r < P; ++r)
        if (x_host[r] == nullptr || !aligned16(x_dev[r])) return KOSMOS_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(x_gathered) || !aligned16(y_dev)) return KOSMOS_ERR_INVALID_ARG;
    if (!aligned16(ws)) return KOSMOS_ERR_WORKSPACE;
    kosmos_opts o = resolve_opts(opts);
    o.tail_split = 0;  // every tile writes its output once: the per-shard output counts stay exact
    if (o.sched < KOSMOS_SCHED_SELF || o.sched > KOSMOS_SCHED_UNFUSED) return KOSMOS_ERR_INVALID_ARG;
    if (!link_ok(o, static_cast<uint64_t>(P - 1) * static_cast<uint64_t>(m_per_shard) * static_cast<uint64_t>(k) * 2u))
        return KOSMOS_ERR_INVALID_ARG;
    if (ws_bytes < kosmos_workspace_bytes(KOSMOS_OP_AG_GEMM, P, m_per_shard, n, k, KOSMOS_BF16, &o))
        return KOSMOS_ERR_WORKSPACE;
    PFN_streamValue32_t wr = get_stream_value_fn(false), wt = get_stream_value_fn(true);
    if (wr == nullptr || wt == nullptr) return KOSMOS_ERR_CUDA;
    AgPlan pl;
    const kosmos_status ps = ag_plan(P, m_per_shard, k, n, KOSMOS_BF16, o, pl);
    if (ps != KOSMOS_OK) return ps;
    AgLaunch L;
    memset(&L, 0, sizeof(L));
    L.P = P; L.m = m_per_shard; L.k = k; L.n = n;
    for (int r = 0; r < P; ++r) L.x[r] = x_dev[r];
    L.w = w; L.x_gathered = x_gathered; L.y = y_dev; L.ws = ws;
    L.dtype = KOSMOS_BF16; L.sched = o.sched; L.n_comm = pl.n_comm; L.pair = pl.pair; L.n_split = 0; L.n_slots = 0;
    L.trace = o.trace; L.grid = pl.grid; L.wait_limit_ns = o.wait_limit_ns; L.inject = o.inject;
    L.plain_launch = o.plain_launch; L.link_gbs = o.link_gbs; L.host_flow = 1;
    const AgWsLayout W = ag_ws_layout(ag_geom(P, m_per_shard, k, n), o.trace != 0, 0);
    uint8_t *ext = static_cast<uint8_t *>(ws) + W.ext_off;
    const CUdeviceptr ready = reinterpret_cast<CUdeviceptr>(ext);
    const CUdeviceptr done = ready + 4 * AG_EXT_WORDS;
    // A shard arrives in chunks of whole 128-row pieces and its output rows go
    // back in groups of whole tile rows (ag_host_cpp / ag_host_tpg: the same
    // geometry as the kernel's), so that the kernel starts on a shard's first
    // rows before the rest are in and the host receives a shard's first
    // output rows while its other tile rows are still being built.
    const AgGeom tg = ag_geom(P, m_per_shard, k, n, pl.pair ? PBM : BM);
    cudaStream_t s = static_cast<cudaStream_t>(stream), h = static_cast<cudaStream_t>(h2d_stream),
                 d = static_cast<cudaStream_t>(d2h_stream);
    CUstream cs = reinterpret_cast<CUstream>(s), ch = reinterpret_cast<CUstream>(h), cd = reinterpret_cast<CUstream>(d);
    // The three streams join through three words of the workspace (no CUDA
    // events to create per call): `stream` publishes this call's token once
    // its earlier work (a previous call's kernel, which reads x_gathered and
    // writes x_dev) is done and the arrival and output words are zeroed; the
    // copy streams wait for it before they overwrite x_gathered or y_host; at
    // the end each copy stream publishes the token and `stream` waits for both.
    const CUdeviceptr sync = done + 4 * AG_EXT_WORDS;  // [0] stream ready, [1] h2d done, [2] d2h done
    uint32_t tok = g_host_flow_token.fetch_add(1u, std::memory_order_relaxed) + 1u;
    if (tok == 0u) tok = g_host_flow_token.fetch_add(1u, std::memory_order_relaxed) + 1u;
    bool ok = cudaMemsetAsync(ext, 0, 2 * 4 * AG_EXT_WORDS, s) == cudaSuccess &&
              wr(cs, sync, tok, CU_STREAM_WRITE_VALUE_DEFAULT) == CUDA_SUCCESS &&
              wt(ch, sync, tok, CU_STREAM_WAIT_VALUE_EQ) == CUDA_SUCCESS &&
              wt(cd, sync, tok, CU_STREAM_WAIT_VALUE_EQ) == CUDA_SUCCESS;
    // The kernel is enqueued first: its tiles and movers wait for the
    // arrival words, so it starts on the first chunks while the host
    // is still enqueueing the later ones.  If an enqueue below fails, the
    // kernel's bounded waits end it with a status and it releases the
    // output waits.
    kosmos_status st = ok ? launch_ag_bf16(L, s) : KOSMOS_ERR_CUDA;
    if (st != KOSMOS_OK) {
        // no kernel: release the output waits below so that no stream blocks
        for (int i = 0; i < P * AG_EXT_STRIDE; ++i)
            wr(ch, done + 4 * i, AG_YDONE_RELEASE, CU_STREAM_WRITE_VALUE_DEFAULT);
    }
    // shard r into its slot of x_gathered chunk by chunk, each followed by its
    // arrival word (the local shard first); the kernel's tiles read the slot
    // as soon as the word is set, and its movers copy the slot on into x_dev[r]
    const int64_t xrow = k * 2, yrow = n * 2;
    const bool drop = (o.inject & KOSMOS_INJECT_DROP_ARRIVAL) != 0;
    const uint32_t *one = host_one_word();
    for (int r = 0; ok && r < P; ++r) {
        const int cpp = ag_host_cpp(tg, r), nch = static_cast<int>(cdiv(tg.pieces, cpp));
        for (int c = 0; ok && c < nch; ++c) {
            const int64_t r0 = static_cast<int64_t>(c) * cpp * PIECE_ROWS;
            const int64_t r1 = std::min<int64_t>(m_per_shard, r0 + static_cast<int64_t>(cpp) * PIECE_ROWS);
            ok = cudaMemcpyAsync(static_cast<uint8_t *>(x_gathered) + (static_cast<int64_t>(r) * m_per_shard + r0) * xrow,
                                 static_cast<const uint8_t *>(x_host[r]) + r0 * xrow, static_cast<size_t>((r1 - r0) * xrow),
                                 cudaMemcpyHostToDevice, h) == cudaSuccess;
            if (ok && !(drop && static_cast<int64_t>(o.inject >> 32) == r)) {
                const CUdeviceptr word = ready + 4 * (r * AG_EXT_STRIDE + c);
                ok = one != nullptr ? cudaMemcpyAsync(reinterpret_cast<void *>(word), one, 4, cudaMemcpyHostToDevice,
                                                      h) == cudaSuccess
                                    : wr(ch, word, 1u, CU_STREAM_WRITE_VALUE_DEFAULT) == CUDA_SUCCESS;
            }
        }
    }
    // each group of shard r's output rows back to the host once all its tiles
    // are written (output tiles counted per CTA of a tile engine)
    const int64_t tr = pl.pair ? PBM : BM;
    const uint32_t per_row = static_cast<uint32_t>(cdiv(n, BN) * (pl.pair ? 2 : 1));
    for (int r = 0; ok && r < P; ++r) {
        const int tpg = ag_host_tpg(tg, r), ngr = static_cast<int>(cdiv(tg.tiles_m, tpg));
        for (int j = 0; ok && j < ngr; ++j) {
            const int t0 = j * tpg, t1 = std::min(tg.tiles_m, t0 + tpg);
            const int64_t r0 = t0 * tr, r1 = std::min<int64_t>(m_per_shard, t1 * tr);
            const size_t off = static_cast<size_t>((static_cast<int64_t>(r) * m_per_shard + r0) * yrow);
            ok = wt(cd, done + 4 * (r * AG_EXT_STRIDE + j), static_cast<uint32_t>(t1 - t0) * per_row,
                    CU_STREAM_WAIT_VALUE_GEQ) == CUDA_SUCCESS &&
                 cudaMemcpyAsync(static_cast<uint8_t *>(y_host) + off, static_cast<uint8_t *>(y_dev) + off,
                                 static_cast<size_t>((r1 - r0) * yrow), cudaMemcpyDeviceToHost, d) == cudaSuccess;
        }
    }
    ok = ok && wr(ch, sync + 4, tok, CU_STREAM_WRITE_VALUE_DEFAULT) == CUDA_SUCCESS &&
         wr(cd, sync + 8, tok, CU_STREAM_WRITE_VALUE_DEFAULT) == CUDA_SUCCESS &&
         wt(cs, sync + 4, tok, CU_STREAM_WAIT_VALUE_EQ) == CUDA_SUCCESS &&
         wt(cs, sync + 8, tok, CU_STREAM_WAIT_VALUE_EQ) == CUDA_SUCCESS;
    if (st != KOSMOS_OK) return st;
    return ok ? KOSMOS_OK : KOSMOS_ERR_CUDA;
}

int kosmos_ag_tile_plan(int P, int64_t m_per_shard, int64_t k, int64_t n, int dtype, const kosmos_opts *opts,
                        int64_t *tail_split, int *tile_m) {
    if (P < 1 || P > KOSMOS_MAX_P || m_per_shard < 1 || n < 8 || k < BK) return -1;
    if (dtype != KOSMOS_BF16 && dtype != KOSMOS_MXFP8_E4M3) return -1;
    const kosmos_opts o = resolve_opts(opts);
    AgPlan pl;
    if (ag_plan(P, m_per_shard, k, n, dtype, o, pl) != KOSMOS_OK) return -1;
    if (tail_split) *tail_split = pl.n_split;
    if (tile_m) *tile_m = pl.pair ? PBM : BM;
    return 0;
}

kosmos_status kosmos_gemm_rs(const void *const *x_shards, const void *const *x_scales, const void *const *w_shards,
                             const void *const *w_scales, int P, int64_t m, int64_t k_per_rank, int64_t n, int dtype,
                             void *const *y_chunks, void *ws, size_t ws_bytes, const kosmos_opts *opts,
                             void *stream) {
    if (P < 1 || P > KOSMOS_MAX_P || x_shards == nullptr || w_shards == nullptr || y_chunks == nullptr)
        return KOSMOS_ERR_INVALID_ARG;
    if (m < P || m % P != 0 || k_per_rank < BK || k_per_rank % BK != 0 || n < 8 || n % 8 != 0)
        return KOSMOS_ERR_INVALID_ARG;
    if (m > (1ll << 30) || k_per_rank > (1ll << 24) || n > (1ll << 24)) return KOSMOS_ERR_INVALID_ARG;
    if (dtype != KOSMOS_BF16 && dtype != KOSMOS_MXFP8_E4M3) return KOSMOS_ERR_INVALID_ARG;
    const bool mx = dtype == KOSMOS_MXFP8_E4M3;
    if (mx && ((m / P) % 128 != 0 || k_per_rank % 128 != 0 || n % 16 != 0 || x_scales == nullptr ||
               w_scales == nullptr))
        return KOSMOS_ERR_INVALID_ARG;
    for (int r = 0; r < P; ++r) {
        if (!aligned16(x_shards[r]) || !aligned16(w_shards[r]) || !aligned16(y_chunks[r]))
            return KOSMOS_ERR_INVALID_ARG;
        if (mx && (!aligned16(x_scales[r]) || !aligned16(w_scales[r]))) return KOSMOS_ERR_INVALID_ARG;
    }
    if (!aligned16(ws)) return KOSMOS_ERR_WORKSPACE;
    const kosmos_opts o = resolve_opts(opts);
    if (o.sched < KOSMOS_SCHED_SELF || o.sched > KOSMOS_SCHED_UNFUSED) return KOSMOS_ERR_INVALID_ARG;
    if (o.order != KOSMOS_ORDER_BAND && o.order != KOSMOS_ORDER_ROW) return KOSMOS_ERR_INVALID_ARG;
    if (!link_ok(o, static_cast<uint64_t>(P - 1) * static_cast<uint64_t>(m) * static_cast<uint64_t>(n) * 2u))
        return KOSMOS_ERR_INVALID_ARG;
    if (ws_bytes < kosmos_workspace_bytes(KOSMOS_OP_GEMM_RS, P, m, n, k_per_rank, dtype, &o))
        return KOSMOS_ERR_WORKSPACE;
    int grid = grid_for(o);
    if (grid < 1) return KOSMOS_ERR_CUDA;
    int pair = o.cta_pair != 0 ? 1 : 0;
    if (mx && !pair) return KOSMOS_ERR_UNSUPPORTED;  // MXFP8 runs on SM pairs only
    if (pair) {
        const int lim = rs_pair_grid_limit(mx);
        int g2 = grid & ~1;
        if (lim >= 2 && g2 > lim) g2 = lim;
        // every emulated rank needs a builder pair; a fixed reducer crew needs at least one
        // reducer CTA per rank on top (two ranks per reducer pair)
        const int need = (o.sched == KOSMOS_SCHED_FIXED) ? 2 * P + 2 * ((P + 1) / 2) : 2 * P;
        if (lim < 2 || g2 < need) {
            if (o.cta_pair == 1 || mx) return KOSMOS_ERR_UNSUPPORTED;
            pair = 0;
        } else {
            grid = g2;
        }
    }
    if (grid < P) return KOSMOS_ERR_INVALID_ARG;  // every emulated rank needs a CTA
    RsLaunch L;
    memset(&L, 0, sizeof(L));
    L.P = P; L.m = m; L.k = k_per_rank; L.n = n;
    for (int r = 0; r < P; ++r) {
        L.x[r] = x_shards[r];
        L.w[r] = w_shards[r];
        L.y[r] = y_chunks[r];
        L.xs[r] = mx ? x_scales[r] : nullptr;
        L.ws_[r] = mx ? w_scales[r] : nullptr;
    }
    L.ws = ws;
    L.dtype = dtype;
    L.sched = o.sched;
    L.pair = pair;
    {
        // reducer CTAs per emulated rank; SM pairs host two ranks' reducers each
        const int max_red = pair ? (2 * (grid / 2 - P)) / P : grid / P - 1;  // keep a builder on every rank
        int n_red = o.n_comm0 >= 0 ? o.n_comm0 : 1;
        if (o.sched == KOSMOS_SCHED_FIXED && o.fixed_comm_ctas >= 0) n_red = o.fixed_comm_ctas;
        if (n_red < 1) n_red = 1;
        if (n_red > max_red) n_red = max_red;
        if (n_red < 1 && o.sched == KOSMOS_SCHED_FIXED) return KOSMOS_ERR_INVALID_ARG;
        L.n_comm = n_red;
    }
    L.order = o.order; L.trace = o.trace; L.grid = grid; L.plain_launch = o.plain_launch;
    L.link_gbs = o.link_gbs;
    L.wait_limit_ns = o.wait_limit_ns; L.inject = o.inject;
    return launch_rs_bf16(L, static_cast<cudaStream_t>(stream));
}

static bool moe_sizes_ok(int P, int64_t tokens, int64_t hidden, int n_experts, int topk, int64_t inter) {
    if (P < 1 || P > KOSMOS_MAX_P) return false;
    if (n_experts < 1 || n_experts > 256 || n_experts % 64 != 0 || n_experts % P != 0) return false;
    if (topk < 1 || topk > 8 || topk > n_experts) return false;
    if (tokens < P || tokens % P != 0 || tokens > (1ll << 24)) return false;
    if (hidden < 256 || hidden % 256 != 0 || hidden > 24576) return false;
    if (inter < 128 || inter % 128 != 0 || inter > (1ll << 16)) return false;
    return true;
}

size_t kosmos_moe_workspace_bytes(int P, int64_t tokens, int64_t hidden, int n_experts, int topk, int64_t inter,
                                  int dtype, const kosmos_opts *opts) {
    const kosmos_opts o = resolve_opts(opts);
    if (!moe_sizes_ok(P, tokens, hidden, n_experts, topk, inter)) return 0;
    if (dtype != KOSMOS_BF16 && dtype != KOSMOS_MXFP8_E4M3) return 0;
    return moe_workspace_bytes(P, tokens, hidden, n_experts, topk, inter, dtype == KOSMOS_MXFP8_E4M3, o.trace != 0);
}

kosmos_status kosmos_moe_debug_view(int what, int P, int64_t tokens, int64_t hidden, int n_experts, int topk,
                                    int64_t inter, int dtype, void *ws, void **ptr, int64_t *bytes) {
    if (!moe_sizes_ok(P, tokens, hidden, n_experts, topk, inter) || ws == nullptr || ptr == nullptr ||
        bytes == nullptr || (dtype != KOSMOS_BF16 && dtype != KOSMOS_MXFP8_E4M3))
        return KOSMOS_ERR_INVALID_ARG;
    return moe_debug_view(what, P, tokens, hidden, n_experts, topk, inter, dtype == KOSMOS_MXFP8_E4M3, ws, ptr, bytes)
               ? KOSMOS_OK
               : KOSMOS_ERR_INVALID_ARG;
}

kosmos_status kosmos_moe_fwd(const void *const *x_shards, const void *w_router, int P, int64_t tokens, int64_t hidden,
                             int n_experts, int topk, int64_t inter, const void *const *w_gate,
                             const void *const *w_gate_scales, const void *const *w_up,
                             const void *const *w_up_scales, const void *const *w_down,
                             const void *const *w_down_scales, int dtype, void *const *y_shards, int32_t *topk_idx,
                             float *topk_gate, int32_t *expert_counts, int32_t *dispatch_pos, void *ws,
                             size_t ws_bytes, const kosmos_opts *opts, void *stream) {
    if (!moe_sizes_ok(P, tokens, hidden, n_experts, topk, inter)) return KOSMOS_ERR_INVALID_ARG;
    if (x_shards == nullptr || w_gate == nullptr || w_up == nullptr || w_down == nullptr || y_shards == nullptr)
        return KOSMOS_ERR_INVALID_ARG;
    if (dtype != KOSMOS_BF16 && dtype != KOSMOS_MXFP8_E4M3) return KOSMOS_ERR_INVALID_ARG;
    const bool mx = dtype == KOSMOS_MXFP8_E4M3;
    if (mx && (w_gate_scales == nullptr || w_up_scales == nullptr || w_down_scales == nullptr))
        return KOSMOS_ERR_INVALID_ARG;
    for (int q = 0; q < P; ++q) {
        if (!aligned16(x_shards[q]) || !aligned16(w_gate[q]) || !aligned16(w_up[q]) || !aligned16(w_down[q]) ||
            !aligned16(y_shards[q]))
            return KOSMOS_ERR_INVALID_ARG;
        if (mx && (!aligned16(w_gate_scales[q]) || !aligned16(w_up_scales[q]) || !aligned16(w_down_scales[q])))
            return KOSMOS_ERR_INVALID_ARG;
    }
    if (!aligned16(w_router) || !aligned16(topk_idx) || !aligned16(topk_gate) || !aligned16(expert_counts) ||
        !aligned16(dispatch_pos))
        return KOSMOS_ERR_INVALID_ARG;
    if (!aligned16(ws)) return KOSMOS_ERR_WORKSPACE;
    const kosmos_opts o = resolve_opts(opts);
    // SELF: one launch; UNFUSED: the baseline of one launch per phase (no role trace: each launch would
    // overwrite the previous one's records)
    if (o.sched == KOSMOS_SCHED_FIXED || (o.sched == KOSMOS_SCHED_UNFUSED && o.trace)) return KOSMOS_ERR_UNSUPPORTED;
    if (o.link_gbs != 0) return KOSMOS_ERR_UNSUPPORTED;
    if (mx && (o.inject & KOSMOS_INJECT_IDENTITY_EXPERTS)) return KOSMOS_ERR_UNSUPPORTED;
    if (ws_bytes < kosmos_moe_workspace_bytes(P, tokens, hidden, n_experts, topk, inter, dtype, &o))
        return KOSMOS_ERR_WORKSPACE;
    const int grid = grid_for(o);
    if (grid < 1) return KOSMOS_ERR_CUDA;
    if (grid < P) return KOSMOS_ERR_INVALID_ARG;  // every emulated rank needs a CTA
    MoeLaunch L;
    memset(&L, 0, sizeof(L));
    L.P = P; L.T = tokens; L.H = hidden; L.I = inter; L.E = n_experts; L.K = topk;
    for (int q = 0; q < P; ++q) {
        L.x[q] = x_shards[q];
        L.wg[q] = w_gate[q];
        L.wu[q] = w_up[q];
        L.wd[q] = w_down[q];
        L.wgs[q] = mx ? w_gate_scales[q] : nullptr;
        L.wus[q] = mx ? w_up_scales[q] : nullptr;
        L.wds[q] = mx ? w_down_scales[q] : nullptr;
        L.y[q] = y_shards[q];
    }
    L.dtype = dtype;
    L.wr = w_router;
    L.topk_idx = topk_idx; L.topk_gate = topk_gate; L.counts = expert_counts; L.pos = dispatch_pos;
    L.ws = ws; L.sched = o.sched; L.n_comm = 0; L.trace = o.trace; L.grid = grid; L.plain_launch = o.plain_launch;
    L.wait_limit_ns = o.wait_limit_ns; L.inject = o.inject;
    return launch_moe_fwd(L, static_cast<cudaStream_t>(stream));
}

static bool moe_bwd_sizes_ok(int P, int64_t tokens, int64_t hidden, int n_experts, int topk, int64_t inter) {
    if (!moe_sizes_ok(P, tokens, hidden, n_experts, topk, inter)) return false;
    return inter % 256 == 0 && (tokens / P) % 64 == 0;
}

size_t kosmos_moe_bwd_workspace_bytes(int P, int64_t tokens, int64_t hidden, int n_experts, int topk, int64_t inter,
                                      const kosmos_opts *opts) {
    const kosmos_opts o = resolve_opts(opts);
    if (!moe_bwd_sizes_ok(P, tokens, hidden, n_experts, topk, inter)) return 0;
    return moe_bwd_workspace_bytes(P, tokens, hidden, n_experts, topk, inter, o.trace != 0);
}

kosmos_status kosmos_moe_bwd_debug_view(int what, int P, int64_t tokens, int64_t hidden, int n_experts, int topk,
                                        int64_t inter, void *ws, void **ptr, int64_t *bytes) {
    if (!moe_bwd_sizes_ok(P, tokens, hidden, n_experts, topk, inter) || ws == nullptr || ptr == nullptr ||
        bytes == nullptr)
        return KOSMOS_ERR_INVALID_ARG;
    return moe_bwd_debug_view(what, P, tokens, hidden, n_experts, topk, inter, ws, ptr, bytes)
               ? KOSMOS_OK
               : KOSMOS_ERR_INVALID_ARG;
}

kosmos_status kosmos_moe_bwd(const void *const *x_shards, const void *w_router, int P, int64_t tokens, int64_t hidden,
                             int n_experts, int topk, int64_t inter, const void *const *w_gate,
                             const void *const *w_up, const void *const *w_down, const int32_t *topk_idx,
                             const float *topk_gate, const void *fwd_ws, size_t fwd_ws_bytes,
                             const void *const *dy_shards, void *const *dx_shards, float *dw_router,
                             void *const *dw_gate, void *const *dw_up, void *const *dw_down, void *ws,
                             size_t ws_bytes, const kosmos_opts *opts, void *stream) {
    if (!moe_bwd_sizes_ok(P, tokens, hidden, n_experts, topk, inter)) return KOSMOS_ERR_INVALID_ARG;
    if (x_shards == nullptr || w_gate == nullptr || w_up == nullptr || w_down == nullptr || dy_shards == nullptr ||
        dx_shards == nullptr || dw_gate == nullptr || dw_up == nullptr || dw_down == nullptr)
        return KOSMOS_ERR_INVALID_ARG;
    for (int q = 0; q < P; ++q)
        if (!aligned16(x_shards[q]) || !aligned16(w_gate[q]) || !aligned16(w_up[q]) || !aligned16(w_down[q]) ||
            !aligned16(dy_shards[q]) || !aligned16(dx_shards[q]) || !aligned16(dw_gate[q]) || !aligned16(dw_up[q]) ||
            !aligned16(dw_down[q]))
            return KOSMOS_ERR_INVALID_ARG;
    if (!aligned16(w_router) || !aligned16(topk_idx) || !aligned16(topk_gate) || !aligned16(dw_router) ||
        !aligned16(fwd_ws))
        return KOSMOS_ERR_INVALID_ARG;
    if (!aligned16(ws)) return KOSMOS_ERR_WORKSPACE;
    const kosmos_opts o = resolve_opts(opts);
    // SELF: one launch; UNFUSED: the baseline of one launch per phase (no role trace)
    if (o.sched == KOSMOS_SCHED_FIXED || (o.sched == KOSMOS_SCHED_UNFUSED && o.trace) || o.link_gbs != 0 ||
        o.inject != 0)
        return KOSMOS_ERR_UNSUPPORTED;
    if (fwd_ws_bytes < moe_workspace_bytes(P, tokens, hidden, n_experts, topk, inter, false, false))
        return KOSMOS_ERR_WORKSPACE;
    if (ws_bytes < kosmos_moe_bwd_workspace_bytes(P, tokens, hidden, n_experts, topk, inter, &o))
        return KOSMOS_ERR_WORKSPACE;
    const int grid = grid_for(o);
    if (grid < 1) return KOSMOS_ERR_CUDA;
    if (grid < P) return KOSMOS_ERR_INVALID_ARG;
    MoeBwdLaunch L;
    memset(&L, 0, sizeof(L));
    L.P = P; L.T = tokens; L.H = hidden; L.I = inter; L.E = n_experts; L.K = topk;
    for (int q = 0; q < P; ++q) {
        L.x[q] = x_shards[q];
        L.wg[q] = w_gate[q];
        L.wu[q] = w_up[q];
        L.wd[q] = w_down[q];
        L.dout[q] = dy_shards[q];
        L.dx[q] = dx_shards[q];
        L.dwg[q] = dw_gate[q];
        L.dwu[q] = dw_up[q];
        L.dwd[q] = dw_down[q];
    }
    L.wr = w_router;
    L.topk_idx = topk_idx; L.topk_gate = topk_gate; L.fwd_ws = fwd_ws; L.dwr = dw_router;
    L.ws = ws; L.trace = o.trace; L.grid = grid; L.plain_launch = o.plain_launch; L.wait_limit_ns = o.wait_limit_ns;
    L.sched = o.sched;
    return launch_moe_bwd(L, static_cast<cudaStream_t>(stream));
}

kosmos_status kosmos_mxfp8_quantize(const void *x, int64_t rows, int64_t cols, int along_cols, void *q, void *scales,
                                    void *stream) {
    if (!aligned16(x) || !aligned16(q) || !aligned16(scales) || rows < 1 || cols < 1) return KOSMOS_ERR_INVALID_ARG;
    if (along_cols ? (cols % 128 != 0) : (rows % 128 != 0)) return KOSMOS_ERR_INVALID_ARG;
    return launch_mxfp8_quantize(x, rows, cols, along_cols, q, scales, static_cast<cudaStream_t>(stream));
}

kosmos_status kosmos_status_sync(void *ws, void *stream, int64_t *failing_entry) {
    if (!aligned16(ws)) return KOSMOS_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KOSMOS_ERR_CUDA;
    WsHeader h;
    if (cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return KOSMOS_ERR_CUDA;
    if (failing_entry) *failing_entry = h.status ? h.fail_entry : -1;
    return static_cast<kosmos_status>(h.status);
}

kosmos_status kosmos_trace_info(int op, int P, int64_t m, int64_t n, int64_t k, int dtype, const kosmos_opts *opts,
                                void *ws, void **records, int32_t *per_cta_capacity, int32_t *num_ctas) {
    const kosmos_opts o = resolve_opts(opts);
    if (!o.trace || ws == nullptr) return KOSMOS_ERR_INVALID_ARG;
    size_t off = 0;
    if (op == KOSMOS_OP_AG_GEMM)
        off = ag_ws_layout(ag_geom(P, m, k, n), true, ag_split_slots(P, m, n, dtype, o)).trace_off;
    else if (op == KOSMOS_OP_GEMM_RS)
        off = rs_ws_layout(rs_geom(P, m, k, n), true).trace_off;
    else
        return KOSMOS_ERR_UNSUPPORTED;
    if (records) *records = static_cast<uint8_t *>(ws) + off;
    if (per_cta_capacity) *per_cta_capacity = TRACE_CAP;
    if (num_ctas) *num_ctas = grid_for(o);
    return KOSMOS_OK;
}

int64_t kosmos_rail_decode(int op, int P, int64_t m, int64_t n, int order, int rank, int rail, int tile_m,
                           int64_t split, int32_t *out, int64_t max_entries) {
    if (P < 1 || P > KOSMOS_MAX_P || m < 1 || n < 1 || (tile_m != 128 && tile_m != 256) || split < 0) return -1;
    if (op == KOSMOS_OP_AG_GEMM) {
        const AgGeom g = ag_geom(P, m, 64, n, tile_m, split);
        const int64_t len = rail == 0 ? g.n_transfer : g.n_tile;
        if (out) {
            for (int64_t t = 0; t < len && t < max_entries; ++t) {
                int32_t *e = out + 4 * t;
                if (rail == 0) {
                    int s, j, q;
                    ag_decode_transfer(g, static_cast<int>(t), s, j, q);
                    e[0] = K_TRANSFER; e[1] = s; e[2] = j; e[3] = q;
                } else {
                    int s, i, c;
                    const int kind = ag_decode_tile(g, static_cast<int>(t), s, i, c);
                    e[0] = kind; e[1] = s; e[2] = i; e[3] = c;
                }
            }
        }
        return len;
    }
    if (op == KOSMOS_OP_GEMM_RS) {
        if (m % P || rank < 0 || rank >= P) return -1;
        const RsGeom g = rs_geom(P, m, 64, n, tile_m);
        const int64_t len = rail == 0 ? g.n_tile : g.n_reduce;
        if (out) {
            for (int64_t t = 0; t < len && t < max_entries; ++t) {
                int32_t *e = out + 4 * t;
                if (rail == 0) {
                    int q, c, b, j;
                    rs_decode_tile(g, order, static_cast<int>(t), q, c, b, j);
                    e[0] = K_TILE; e[1] = q * P + c; e[2] = b; e[3] = j;
                } else {
                    int b, j;
                    rs_decode_reduce(g, static_cast<int>(t), b, j);
                    e[0] = K_REDUCE; e[1] = rank; e[2] = b; e[3] = j;
                }
            }
        }
        return len;
    }
    return -1;
}

int64_t kosmos_rail_decode_device(int op, int P, int64_t m, int64_t n, int order, int rank, int rail, int tile_m,
                                  int64_t split, int32_t *out, int64_t max_entries, void *stream) {
    const int64_t len = kosmos_rail_decode(op, P, m, n, order, rank, rail, tile_m, split, nullptr, 0);
    if (len < 0 || out == nullptr) return len;
    const int64_t cnt = len < max_entries ? len : max_entries;
    if (launch_rail_decode(op, P, m, n, order, rank, rail, tile_m, split, out, cnt,
                           static_cast<cudaStream_t>(stream)) != KOSMOS_OK)
        return -1;
    return len;
}

}  // extern "C"
