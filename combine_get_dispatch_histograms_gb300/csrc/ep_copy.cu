// ep_copy.cu -- the row-copy steps of the normal path, on one bulk-copy engine:
//
//  * dispatch scatter (page "DeepEP 学习笔记", sections "dispatch 过程" and
//    "DeepEP v2 / direct 模式": one copy of a token per destination RANK, with
//    its metadata x, src_idx, topk_idx, topk_weights);
//  * local permute (page "事件驱动 EP 内核的调度策略与零拷贝通信", section "高吞吐量
//    模式": received rows regrouped into contiguous per-expert blocks for the
//    grouped GEMM);
//  * fused dispatch (same pages, v2 direct mode's dispatch straight into the
//    tensors the experts consume): each token written once per valid top-k
//    entry into the expert-major layout, without the per-rank receive buffer;
//  * hierarchical staging (page "DeepEP 学习笔记", section "hybrid 模式"; home
//    rank rule from "零拷贝通信"): stage A one copy per destination node to the
//    home rank, stage B forward inside the node.
//
// Every step reads each source row ONCE and writes it to 0..F destination rows
// whose indices the notify pass fixed.  The engine is a persistent CTA with
//  - warp 0, lane 0: the issuer.  It streams source rows global -> shared with
//    cp.async.bulk (completion on an mbarrier per stage, S stages in flight) and
//    writes each staged row to all its destinations with cp.async.bulk
//    shared -> global (bulk groups, reuse of a stage after wait_group.read);
//  - warps 1..3: the builders.  They compute the destination rows of the next
//    batch of units into a double-buffered shared table and write the small
//    per-row metadata with plain stores.
// Data never passes through registers; every wait is bounded and a wait that
// runs out sets FLAG_TIMEOUT and stops the CTA's copies.
#include "ep_internal.cuh"

namespace ep {

constexpr int kCopyThreads = 128;
constexpr int kBuilderThreads = kCopyThreads - 32;
constexpr int kBatch = 32;      // units per table batch
constexpr int kMaxStages = 16;

struct CopyGeom {
    int64_t n_units;               // units, or the most units when n_units_dev is given
    const int32_t* n_units_dev;    // nullable: actual count on the device (clamped to n_units)
    int64_t row_bytes;
    int32_t chunk_bytes;
    int32_t nchunks;
    int32_t stages;
    int32_t fanout;  // candidates examined per unit (<= kMaxFanout)
    int64_t timeout_ns;
    uint32_t* status;
};

// ---- routes: where a unit comes from and where its copies go ----------------

// dispatch scatter: unit = source token g = s*T + t, candidates = receivers d
struct ScatterRoute {
    const uint8_t* x;
    uint8_t* recv_x;
    const int64_t* topk_idx;
    const float* w;
    const int32_t* send_pos;
    const int32_t* rank_base;
    int32_t* recv_src_rank;
    int32_t* recv_src_idx;
    int32_t* recv_topk_idx;
    float* recv_topk_w;
    int R, K, T, L;
    int64_t row_bytes;
    int64_t recv_rows;  // rows the recv buffers hold
    uint32_t* status;
    __device__ const uint8_t* src(int64_t u) const { return x + u * row_bytes; }
    __device__ uint8_t* dst(int64_t row) const { return recv_x + row * row_bytes; }
    __device__ bool candidate(int64_t u, int d, int64_t* row) const {
        const int32_t sp = send_pos[u * R + d];
        if (sp < 0) return false;
        const int64_t r = (int64_t)rank_base[d] + sp;
        if (r >= recv_rows) {  // more rows than the caller's buffers hold
            flag(status, FLAG_CAPACITY);
            return false;
        }
        *row = r;
        const int s = (int)(u / T), t = (int)(u % T);
        recv_src_rank[r] = s;
        recv_src_idx[r] = t;
        for (int k = 0; k < K; ++k) {
            const int64_t e = topk_idx[u * K + k];
            const bool on = e >= 0 && e / L == d;
            recv_topk_idx[r * K + k] = on ? (int32_t)(e - (int64_t)d * L) : -1;
            recv_topk_w[r * K + k] = on ? w[u * K + k] : 0.0f;
        }
        return true;
    }
};

// local permute: unit = received row r, candidates = its K local top-k slots
struct PermuteRoute {
    const uint8_t* recv_x;
    uint8_t* permuted_x;
    const int32_t* recv_src_rank;
    const int32_t* recv_src_idx;
    const int32_t* recv_topk_idx;
    const int32_t* perm_pos;
    int32_t* perm_src_row;
    int K, T;
    int64_t row_bytes;
    int64_t perm_rows;
    uint32_t* status;
    __device__ const uint8_t* src(int64_t u) const { return recv_x + u * row_bytes; }
    __device__ uint8_t* dst(int64_t row) const { return permuted_x + row * row_bytes; }
    __device__ bool candidate(int64_t u, int k, int64_t* row) const {
        if (recv_topk_idx[u * K + k] < 0) return false;
        const int64_t g = (int64_t)recv_src_rank[u] * T + recv_src_idx[u];
        const int32_t p = perm_pos[g * K + k];
        if (p < 0 || p >= perm_rows) {
            flag(status, p < 0 ? FLAG_BOUNDS : FLAG_CAPACITY);
            return false;
        }
        perm_src_row[p] = (int32_t)u;
        *row = p;
        return true;
    }
};

// fused dispatch: unit = source token g, candidates = its K top-k entries; the
// row goes straight to its permuted rows (no receive buffer in between)
struct PermutedScatterRoute {
    const uint8_t* x;
    uint8_t* permuted_x;
    const int64_t* topk_idx;
    const float* w;
    const int32_t* perm_pos;
    int32_t* perm_src_token;  // [P] s * T + t of each permuted row
    float* perm_weight;       // [P] the entry's weight (nullable)
    int K, E;
    int64_t row_bytes;
    int64_t perm_rows;
    uint32_t* status;
    __device__ const uint8_t* src(int64_t u) const { return x + u * row_bytes; }
    __device__ uint8_t* dst(int64_t row) const { return permuted_x + row * row_bytes; }
    __device__ bool candidate(int64_t u, int k, int64_t* row) const {
        const int64_t e = topk_idx[u * K + k];
        if (e < 0 || e >= E) return false;
        const int32_t p = perm_pos[u * K + k];
        if (p < 0 || p >= perm_rows) {
            flag(status, p < 0 ? FLAG_BOUNDS : FLAG_CAPACITY);
            return false;
        }
        perm_src_token[p] = (int32_t)u;
        if (perm_weight) perm_weight[p] = w[u * K + k];
        *row = p;
        return true;
    }
};

// hierarchical stage A: unit = source token, candidates = nodes
struct StageARoute {
    const uint8_t* x;
    uint8_t* staging;
    const int32_t* stage_pos;
    int32_t* stage_src_rank;
    int32_t* stage_src_idx;
    int N, T;
    int64_t row_bytes;
    int64_t stage_rows;  // rows the staging buffers hold
    uint32_t* status;
    __device__ const uint8_t* src(int64_t u) const { return x + u * row_bytes; }
    __device__ uint8_t* dst(int64_t row) const { return staging + row * row_bytes; }
    __device__ bool candidate(int64_t u, int n, int64_t* row) const {
        const int32_t p = stage_pos[u * N + n];
        if (p < 0) return false;
        if (p >= stage_rows) {
            flag(status, FLAG_CAPACITY);
            return false;
        }
        stage_src_rank[p] = (int32_t)(u / T);
        stage_src_idx[p] = (int32_t)(u % T);
        *row = p;
        return true;
    }
};

// hierarchical stage B: unit = staged row, candidates = the G ranks of its node
struct StageBRoute {
    const uint8_t* staging;
    uint8_t* recv_x;
    const int32_t* stage_base;  // [R+1]
    const int32_t* stage_src_rank;
    const int32_t* stage_src_idx;
    const int64_t* topk_idx;
    const float* w;
    const int32_t* send_pos;
    const int32_t* rank_base;
    int32_t* recv_src_rank;
    int32_t* recv_src_idx;
    int32_t* recv_topk_idx;
    float* recv_topk_w;
    int R, K, T, L, G;
    int64_t row_bytes;
    int64_t recv_rows;
    uint32_t* status;
    __device__ const uint8_t* src(int64_t u) const { return staging + u * row_bytes; }
    __device__ uint8_t* dst(int64_t row) const { return recv_x + row * row_bytes; }
    __device__ bool candidate(int64_t u, int j, int64_t* row) const {
        // home rank h of staged row u: the last h with stage_base[h] <= u
        int lo = 0, hi = R;  // invariant: stage_base[lo] <= u < stage_base[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (stage_base[mid] <= u) lo = mid;
            else hi = mid;
        }
        const int n = lo / G;
        const int d = n * G + j;
        const int s = stage_src_rank[u], t = stage_src_idx[u];
        const int64_t g = (int64_t)s * T + t;
        const int32_t sp = send_pos[g * R + d];
        if (sp < 0) return false;
        const int64_t r = (int64_t)rank_base[d] + sp;
        if (r >= recv_rows) {
            flag(status, FLAG_CAPACITY);
            return false;
        }
        *row = r;
        recv_src_rank[r] = s;
        recv_src_idx[r] = t;
        for (int k = 0; k < K; ++k) {
            const int64_t e = topk_idx[g * K + k];
            const bool on = e >= 0 && e / L == d;
            recv_topk_idx[r * K + k] = on ? (int32_t)(e - (int64_t)d * L) : -1;
            recv_topk_w[r * K + k] = on ? w[g * K + k] : 0.0f;
        }
        return true;
    }
};

// ---- the engine -------------------------------------------------------------

struct EngineSmem {
    uint64_t* bar;    // [stages]
    int32_t* cnt;     // [2][kBatch]
    int64_t* rows;    // [2][kBatch][fanout]
    uint8_t* stage;   // [stages][chunk_bytes]
};

__host__ __device__ inline size_t engine_table_bytes(int fanout) {
    return 2 * kBatch * sizeof(int32_t) + 2 * (size_t)kBatch * fanout * sizeof(int64_t);
}
__host__ __device__ inline size_t engine_stage_offset(int fanout) {
    size_t off = kMaxStages * sizeof(uint64_t) + engine_table_bytes(fanout);
    return (off + 127) & ~size_t(127);
}

template <class Route>
__device__ void build_batch(const Route& route, const CopyGeom& g, const EngineSmem& sm, int buf, int64_t u0,
                            int nunits) {
    const int bt = threadIdx.x - 32;  // 0 .. kBuilderThreads-1
    int32_t* cnt = sm.cnt + buf * kBatch;
    int64_t* rows = sm.rows + (size_t)buf * kBatch * g.fanout;
    for (int i = bt; i < kBatch; i += kBuilderThreads) cnt[i] = 0;
    asm volatile("bar.sync 1, %0;" ::"n"(kBuilderThreads) : "memory");
    const int pairs = nunits * g.fanout;
    for (int p = bt; p < pairs; p += kBuilderThreads) {
        const int i = p / g.fanout, j = p % g.fanout;
        int64_t row;
        if (route.candidate(u0 + i, j, &row)) {
            const int slot = atomicAdd(&cnt[i], 1);
            rows[(size_t)i * g.fanout + slot] = row;
        }
    }
}

template <class Route, int DEPTH>
__global__ void __launch_bounds__(kCopyThreads) copy_engine_kernel(Route route, CopyGeom g) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    EngineSmem sm;
    sm.bar = reinterpret_cast<uint64_t*>(smem_raw);
    sm.cnt = reinterpret_cast<int32_t*>(smem_raw + kMaxStages * sizeof(uint64_t));
    sm.rows = reinterpret_cast<int64_t*>(smem_raw + kMaxStages * sizeof(uint64_t) + 2 * kBatch * sizeof(int32_t));
    sm.stage = smem_raw + engine_stage_offset(g.fanout);

    int64_t total = g.n_units;
    if (g.n_units_dev) {
        const int64_t dv = *g.n_units_dev;
        if (dv > total && threadIdx.x == 0 && blockIdx.x == 0) flag(g.status, FLAG_CAPACITY);
        total = dv < total ? (dv > 0 ? dv : 0) : total;
    }
    const int64_t u_begin = total * blockIdx.x / gridDim.x;
    const int64_t u_end = total * (blockIdx.x + 1) / gridDim.x;
    const int64_t n_units = u_end - u_begin;
    const int nbatches = (int)((n_units + kBatch - 1) / kBatch);
    const int64_t J = n_units * g.nchunks;  // jobs of this CTA
    const bool issuer = threadIdx.x == 0;
    const bool builder = threadIdx.x >= 32;
    const int S = g.stages;

    auto job_bytes = [&](int64_t j) -> uint32_t {
        const int c = (int)(j % g.nchunks);
        const int64_t rem = g.row_bytes - (int64_t)c * g.chunk_bytes;
        return (uint32_t)(rem < g.chunk_bytes ? rem : g.chunk_bytes);
    };
    auto issue_load = [&](int64_t j) {
        const int st = (int)(j % S);
        const int64_t u = u_begin + j / g.nchunks;
        const int c = (int)(j % g.nchunks);
        const uint32_t bytes = job_bytes(j);
        mbar_arrive_expect_tx(&sm.bar[st], bytes);
        bulk_g2s(sm.stage + (size_t)st * g.chunk_bytes, route.src(u) + (int64_t)c * g.chunk_bytes, bytes,
                 &sm.bar[st]);
    };

    int64_t issued = 0;  // jobs whose load has been issued (issuer only)
    bool aborted = false;
    if (issuer) {
        for (int st = 0; st < S; ++st) mbar_init(&sm.bar[st], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
        for (; issued < J && issued < S; ++issued) issue_load(issued);
    }
    if (builder && nbatches > 0) build_batch(route, g, sm, 0, u_begin, (int)(n_units < kBatch ? n_units : kBatch));
    __syncthreads();

    for (int b = 0; b < nbatches; ++b) {
        const int64_t ub = (int64_t)b * kBatch;
        const int nb = (int)(n_units - ub < kBatch ? n_units - ub : kBatch);
        if (issuer) {
            const int32_t* cnt = sm.cnt + (b & 1) * kBatch;
            const int64_t* rows = sm.rows + (size_t)(b & 1) * kBatch * g.fanout;
            const int64_t j0 = ub * g.nchunks, j1 = (ub + nb) * g.nchunks;
            for (int64_t j = j0; j < j1 && !aborted; ++j) {
                const int st = (int)(j % S);
                const uint32_t parity = (uint32_t)((j / S) & 1);
                if (!mbar_wait_bounded(&sm.bar[st], parity, g.timeout_ns)) {
                    flag(g.status, FLAG_TIMEOUT);
                    aborted = true;
                    break;
                }
                const int i = (int)(j / g.nchunks - ub);
                const int c = (int)(j % g.nchunks);
                const uint32_t bytes = job_bytes(j);
                const uint8_t* sbuf = sm.stage + (size_t)st * g.chunk_bytes;
                const int n = cnt[i];
                for (int q = 0; q < n; ++q)
                    bulk_s2g(route.dst(rows[(size_t)i * g.fanout + q]) + (int64_t)c * g.chunk_bytes, sbuf, bytes);
                bulk_commit();
                // the groups up to job j-DEPTH have finished reading their stages:
                // refill the stage of job j-DEPTH
                bulk_wait_read<DEPTH>();
                if (j >= DEPTH && issued < J) {
                    issue_load(issued);
                    ++issued;
                }
            }
        } else if (builder && b + 1 < nbatches) {
            const int64_t un = (int64_t)(b + 1) * kBatch;
            build_batch(route, g, sm, (b + 1) & 1, u_begin + un, (int)(n_units - un < kBatch ? n_units - un : kBatch));
        }
        __syncthreads();
    }
    if (issuer) {
        bulk_wait_all();
        if (aborted) {
            // let every load still in flight land before the CTA leaves
            for (int64_t j = issued - S > 0 ? issued - S : 0; j < issued; ++j)
                mbar_wait_bounded(&sm.bar[j % S], (uint32_t)((j / S) & 1), g.timeout_ns);
        }
    }
}

// ---- host launch ----------------------------------------------------------------

struct EngineLaunch {
    CopyGeom g;
    int grid;
    int depth;  // bulk store groups allowed to be reading shared memory
    size_t smem;
};

static EngineLaunch plan_engine(const ep_ctx* c, int64_t n_units, int64_t row_bytes, int fanout, CopyKind kind,
                                bool more_issuers = false) {
    EngineLaunch p;
    p.g.n_units = n_units;
    p.g.n_units_dev = nullptr;
    p.g.row_bytes = row_bytes;
    p.g.fanout = fanout;
    p.g.timeout_ns = c->wait_timeout_ns;
    p.g.status = c->status;
    p.depth = c->copy_read_depth;
    // copy_ctas_per_sm persistent CTAs per SM, each with copy_stage_bytes of
    // staging; `more_issuers`: four CTAs per SM with 48 KB each (see permute_rows)
    int ctas_per_sm = c->copy_ctas_per_sm[kind];
    size_t budget = (size_t)c->copy_stage_bytes[kind];
    if (more_issuers && !c->copy_shape_forced[kind]) {
        ctas_per_sm = 4;
        budget = 48 * 1024;
    }
    const size_t fixed = engine_stage_offset(fanout);
    const size_t stage_room = budget > fixed ? budget - fixed : 16 * 1024;
    int64_t chunk = row_bytes;
    if (chunk * 4 > (int64_t)stage_room) chunk = (int64_t)(stage_room / 4) & ~int64_t(15);
    if (chunk < 16) chunk = 16;
    p.g.chunk_bytes = (int32_t)chunk;
    p.g.nchunks = (int32_t)((row_bytes + chunk - 1) / chunk);
    int stages = (int)(stage_room / (size_t)chunk);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < p.depth + 1) stages = p.depth + 1;
    p.g.stages = stages;
    p.smem = fixed + (size_t)stages * chunk;
    const int64_t max_grid = (int64_t)c->num_sms * ctas_per_sm;
    const int64_t want = (n_units + 7) / 8;  // at least 8 units per CTA
    p.grid = (int)(want < max_grid ? (want < 1 ? 1 : want) : max_grid);
    return p;
}

template <class Route, int DEPTH>
static ep_status launch_depth(const Route& r, const EngineLaunch& p, int device, cudaStream_t s, const char* what) {
    // the dynamic shared-memory limit is raised once per device and size
    static int raised[kMaxDevicesTracked] = {};
    if (device < 0 || device >= kMaxDevicesTracked || raised[device] < (int)p.smem) {
        cudaError_t e = cudaFuncSetAttribute(copy_engine_kernel<Route, DEPTH>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
        if (e != cudaSuccess) return cuda_error(e, what);
        if (device >= 0 && device < kMaxDevicesTracked) raised[device] = (int)p.smem;
    }
    copy_engine_kernel<Route, DEPTH><<<p.grid, kCopyThreads, p.smem, s>>>(r, p.g);
    EP_CHECK_LAUNCH(what);
    return EP_OK;
}

template <class Route>
static ep_status launch_engine(const ep_ctx* c, const Route& r, const EngineLaunch& p, cudaStream_t s,
                               const char* what) {
    if (p.g.n_units <= 0) return EP_OK;
    switch (p.depth) {
        case 1: return launch_depth<Route, 1>(r, p, c->device, s, what);
        case 2: return launch_depth<Route, 2>(r, p, c->device, s, what);
        default: return launch_depth<Route, 3>(r, p, c->device, s, what);
    }
}

}  // namespace ep

using namespace ep;

static ep_status check_rows(const void* p, const char* name) {
    if (!p) return set_error(EP_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned16(p)) return set_error(EP_ERR_INVALID_ARG, "%s must be 16-byte aligned", name);
    return EP_OK;
}

namespace ep {

ep_status dispatch_rows(ep_ctx* c, const void* x, int64_t row_bytes, const int64_t* topk_idx, const float* topk_weights,
                        const ep_dispatch_handle* h, void* recv_x, int32_t* recv_src_rank, int32_t* recv_src_idx,
                        int32_t* recv_topk_idx, float* recv_topk_weights, int64_t recv_capacity_rows, void* stream) {
    if (!c || !h) return set_error(EP_ERR_INVALID_ARG, "ctx or handle is NULL");
    c->last_launches = 0;
    const ep_config& f = c->cfg;
    if (f.num_tokens == 0 || (c->totals_known && c->last_total_recv == 0) || recv_capacity_rows == 0) return EP_OK;
    ep_status st;
    if ((st = check_rows(x, "x")) != EP_OK || (st = check_rows(recv_x, "recv_x")) != EP_OK) return st;
    if (!topk_idx || !topk_weights || !h->send_pos || !h->rank_base || !recv_src_rank || !recv_src_idx ||
        !recv_topk_idx || !recv_topk_weights)
        return set_error(EP_ERR_INVALID_ARG, "NULL dispatch argument");
    if (c->totals_known && recv_capacity_rows < c->last_total_recv)
        return set_error(EP_ERR_CAPACITY, "recv buffers hold %lld rows, notify counted %lld",
                         (long long)recv_capacity_rows, (long long)c->last_total_recv);
    ScatterRoute r;
    r.x = static_cast<const uint8_t*>(x);
    r.recv_x = static_cast<uint8_t*>(recv_x);
    r.topk_idx = topk_idx;
    r.w = topk_weights;
    r.send_pos = h->send_pos;
    r.rank_base = h->rank_base;
    r.recv_src_rank = recv_src_rank;
    r.recv_src_idx = recv_src_idx;
    r.recv_topk_idx = recv_topk_idx;
    r.recv_topk_w = recv_topk_weights;
    r.R = f.num_ranks;
    r.K = f.num_topk;
    r.T = f.num_tokens;
    r.L = c->L;
    r.row_bytes = row_bytes;
    r.recv_rows = recv_capacity_rows;
    r.status = c->status;
    EngineLaunch p = plan_engine(c, (int64_t)f.num_ranks * f.num_tokens, r.row_bytes, f.num_ranks, COPY_SCATTER);
    st = launch_engine(c, r, p, as_stream(stream), "dispatch scatter");
    if (st == EP_OK) c->last_launches = 1;
    return st;
}

ep_status permute_rows(ep_ctx* c, const ep_dispatch_handle* h, const void* recv_x, int64_t row_bytes,
                       const int32_t* recv_src_rank, const int32_t* recv_src_idx, const int32_t* recv_topk_idx,
                       int64_t num_recv_rows, void* permuted_x, int32_t* perm_src_row, int64_t perm_capacity_rows,
                       void* stream) {
    if (!c || !h) return set_error(EP_ERR_INVALID_ARG, "ctx or handle is NULL");
    c->last_launches = 0;
    const ep_config& f = c->cfg;
    if (num_recv_rows < 0) return set_error(EP_ERR_INVALID_ARG, "num_recv_rows < 0");
    if (num_recv_rows == 0 || (c->totals_known && c->last_total_recv == 0)) return EP_OK;
    ep_status st;
    if ((st = check_rows(recv_x, "recv_x")) != EP_OK || (st = check_rows(permuted_x, "permuted_x")) != EP_OK)
        return st;
    if (!recv_src_rank || !recv_src_idx || !recv_topk_idx || !perm_src_row || !h->perm_pos || !h->rank_base)
        return set_error(EP_ERR_INVALID_ARG, "NULL permute argument");
    if (c->totals_known && perm_capacity_rows < c->last_total_perm)
        return set_error(EP_ERR_CAPACITY, "permuted buffers hold %lld rows, notify counted %lld",
                         (long long)perm_capacity_rows, (long long)c->last_total_perm);
    PermuteRoute r;
    r.recv_x = static_cast<const uint8_t*>(recv_x);
    r.permuted_x = static_cast<uint8_t*>(permuted_x);
    r.recv_src_rank = recv_src_rank;
    r.recv_src_idx = recv_src_idx;
    r.recv_topk_idx = recv_topk_idx;
    r.perm_pos = h->perm_pos;
    r.perm_src_row = perm_src_row;
    r.K = f.num_topk;
    r.T = f.num_tokens;
    r.row_bytes = row_bytes;
    r.perm_rows = perm_capacity_rows;
    r.status = c->status;
    // Rows of at most 8 KB that mostly go to one local expert (fewer than 1.25
    // permuted rows per received row, known after a waiting notify) move
    // faster with four issuing CTAs per SM: one row load then about one store
    // each, so the bytes in flight per SM set the rate (skewed permute, 8 KB
    // rows, 1.09 rows out per row in: 1299 -> 1219-1230 us).  Larger rows
    // (prefill and hierarchical, 14 KB) and higher fan-out (prefill FP8 rows,
    // 7.4 KB, 1.5 rows out per row in: 511 against 529 us) keep two.
    const bool more_issuers = r.row_bytes <= 8192 && c->totals_known && c->last_total_recv > 0 &&
                              c->last_total_perm * 4 < c->last_total_recv * 5;
    EngineLaunch p = plan_engine(c, num_recv_rows, r.row_bytes, f.num_topk, COPY_PERMUTE, more_issuers);
    p.g.n_units_dev = h->rank_base + f.num_ranks;  // rows actually received, at most num_recv_rows
    st = launch_engine(c, r, p, as_stream(stream), "local permute");
    if (st == EP_OK) c->last_launches = 1;
    return st;
}

ep_status dispatch_permuted_rows(ep_ctx* c, const void* x, int64_t row_bytes, const int64_t* topk_idx,
                                 const float* topk_weights, const ep_dispatch_handle* h, void* permuted_x,
                                 int32_t* perm_src_token, float* perm_weight, int64_t perm_capacity_rows,
                                 void* stream) {
    if (!c || !h) return set_error(EP_ERR_INVALID_ARG, "ctx or handle is NULL");
    c->last_launches = 0;
    const ep_config& f = c->cfg;
    if (f.num_tokens == 0 || (c->totals_known && c->last_total_perm == 0) || perm_capacity_rows == 0) return EP_OK;
    ep_status st;
    if ((st = check_rows(x, "x")) != EP_OK || (st = check_rows(permuted_x, "permuted_x")) != EP_OK) return st;
    if (!topk_idx || !h->perm_pos || !perm_src_token || (perm_weight && !topk_weights))
        return set_error(EP_ERR_INVALID_ARG, "NULL fused dispatch argument");
    if (c->totals_known && perm_capacity_rows < c->last_total_perm)
        return set_error(EP_ERR_CAPACITY, "permuted buffers hold %lld rows, notify counted %lld",
                         (long long)perm_capacity_rows, (long long)c->last_total_perm);
    PermutedScatterRoute r;
    r.x = static_cast<const uint8_t*>(x);
    r.permuted_x = static_cast<uint8_t*>(permuted_x);
    r.topk_idx = topk_idx;
    r.w = topk_weights;
    r.perm_pos = h->perm_pos;
    r.perm_src_token = perm_src_token;
    r.perm_weight = perm_weight;
    r.K = f.num_topk;
    r.E = f.num_experts;
    r.row_bytes = row_bytes;
    r.perm_rows = perm_capacity_rows;
    r.status = c->status;
    EngineLaunch p = plan_engine(c, (int64_t)f.num_ranks * f.num_tokens, r.row_bytes, f.num_topk, COPY_FUSED);
    st = launch_engine(c, r, p, as_stream(stream), "fused dispatch");
    if (st == EP_OK) c->last_launches = 1;
    return st;
}

}  // namespace ep

extern "C" ep_status ep_dispatch(ep_ctx* c, const void* x, const int64_t* topk_idx, const float* topk_weights,
                                 const ep_dispatch_handle* h, void* recv_x, int32_t* recv_src_rank,
                                 int32_t* recv_src_idx, int32_t* recv_topk_idx, float* recv_topk_weights,
                                 int64_t recv_capacity_rows, void* stream) {
    if (!c) return set_error(EP_ERR_INVALID_ARG, "ctx is NULL");
    return dispatch_rows(c, x, (int64_t)c->cfg.hidden * 2, topk_idx, topk_weights, h, recv_x, recv_src_rank,
                         recv_src_idx, recv_topk_idx, recv_topk_weights, recv_capacity_rows, stream);
}

extern "C" ep_status ep_permute(ep_ctx* c, const ep_dispatch_handle* h, const void* recv_x,
                                const int32_t* recv_src_rank, const int32_t* recv_src_idx,
                                const int32_t* recv_topk_idx, int64_t num_recv_rows, void* permuted_x,
                                int32_t* perm_src_row, int64_t perm_capacity_rows, void* stream) {
    if (!c) return set_error(EP_ERR_INVALID_ARG, "ctx is NULL");
    return permute_rows(c, h, recv_x, (int64_t)c->cfg.hidden * 2, recv_src_rank, recv_src_idx, recv_topk_idx,
                        num_recv_rows, permuted_x, perm_src_row, perm_capacity_rows, stream);
}

extern "C" ep_status ep_dispatch_permuted(ep_ctx* c, const void* x, const int64_t* topk_idx,
                                          const float* topk_weights, const ep_dispatch_handle* h, void* permuted_x,
                                          int32_t* perm_src_token, float* perm_weight, int64_t perm_capacity_rows,
                                          void* stream) {
    if (!c) return set_error(EP_ERR_INVALID_ARG, "ctx is NULL");
    return dispatch_permuted_rows(c, x, (int64_t)c->cfg.hidden * 2, topk_idx, topk_weights, h, permuted_x,
                                  perm_src_token, perm_weight, perm_capacity_rows, stream);
}

extern "C" ep_status ep_dispatch_hier(ep_ctx* c, const void* x, const int64_t* topk_idx,
                                      const float* topk_weights, const ep_dispatch_handle* h, void* staging,
                                      int32_t* stage_src_rank, int32_t* stage_src_idx,
                                      int64_t stage_capacity_rows, void* recv_x, int32_t* recv_src_rank,
                                      int32_t* recv_src_idx, int32_t* recv_topk_idx, float* recv_topk_weights,
                                      int64_t recv_capacity_rows, void* stream) {
    if (!c || !h) return set_error(EP_ERR_INVALID_ARG, "ctx or handle is NULL");
    c->last_launches = 0;
    const ep_config& f = c->cfg;
    if (f.num_nodes < 2) return set_error(EP_ERR_INVALID_ARG, "ep_dispatch_hier needs num_nodes > 1");
    if (f.num_tokens == 0 || (c->totals_known && c->last_total_recv == 0) || recv_capacity_rows == 0 ||
        stage_capacity_rows == 0)
        return EP_OK;
    ep_status st;
    if ((st = check_rows(x, "x")) != EP_OK || (st = check_rows(recv_x, "recv_x")) != EP_OK ||
        (st = check_rows(staging, "staging")) != EP_OK)
        return st;
    if (!topk_idx || !topk_weights || !h->send_pos || !h->rank_base || !h->stage_base || !h->stage_pos ||
        !stage_src_rank || !stage_src_idx || !recv_src_rank || !recv_src_idx || !recv_topk_idx ||
        !recv_topk_weights)
        return set_error(EP_ERR_INVALID_ARG, "NULL hierarchical dispatch argument");
    if (c->totals_known && (stage_capacity_rows < c->last_total_stage || recv_capacity_rows < c->last_total_recv))
        return set_error(EP_ERR_CAPACITY, "staging / recv buffers smaller than notify's counts");
    const int64_t row_bytes = (int64_t)f.hidden * 2;
    StageARoute a;
    a.x = static_cast<const uint8_t*>(x);
    a.staging = static_cast<uint8_t*>(staging);
    a.stage_pos = h->stage_pos;
    a.stage_src_rank = stage_src_rank;
    a.stage_src_idx = stage_src_idx;
    a.N = f.num_nodes;
    a.T = f.num_tokens;
    a.row_bytes = row_bytes;
    a.stage_rows = stage_capacity_rows;
    a.status = c->status;
    EngineLaunch pa = plan_engine(c, (int64_t)f.num_ranks * f.num_tokens, row_bytes, f.num_nodes, COPY_STAGE);
    st = launch_engine(c, a, pa, as_stream(stream), "hierarchical stage A");
    if (st != EP_OK) return st;
    StageBRoute b;
    b.staging = static_cast<const uint8_t*>(staging);
    b.recv_x = static_cast<uint8_t*>(recv_x);
    b.stage_base = h->stage_base;
    b.stage_src_rank = stage_src_rank;
    b.stage_src_idx = stage_src_idx;
    b.topk_idx = topk_idx;
    b.w = topk_weights;
    b.send_pos = h->send_pos;
    b.rank_base = h->rank_base;
    b.recv_src_rank = recv_src_rank;
    b.recv_src_idx = recv_src_idx;
    b.recv_topk_idx = recv_topk_idx;
    b.recv_topk_w = recv_topk_weights;
    b.R = f.num_ranks;
    b.K = f.num_topk;
    b.T = f.num_tokens;
    b.L = c->L;
    b.G = c->G;
    b.row_bytes = row_bytes;
    b.recv_rows = recv_capacity_rows;
    b.status = c->status;
    EngineLaunch pb = plan_engine(c, c->totals_known ? c->last_total_stage : stage_capacity_rows, row_bytes, c->G, COPY_STAGE);
    pb.g.n_units_dev = h->stage_base + f.num_ranks;  // rows actually staged
    st = launch_engine(c, b, pb, as_stream(stream), "hierarchical stage B");
    if (st == EP_OK) c->last_launches = 2;
    return st;
}
