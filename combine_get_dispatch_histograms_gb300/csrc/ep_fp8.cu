// ep_fp8.cu -- FP8 rows for the normal (high-throughput) path.
//
// Page "DeepEP 学习笔记", section "内存布局": a token's message carries x and its
// scales (the RDMA channel data holds "x, scales, SourceMeta, topk_idx,
// topk_weights"); page "事件驱动 EP 内核的调度策略与零拷贝通信", section "低延迟模式":
// hidden states travel as FP8 and combine stays BF16.  Here each token is
// quantised once into an FP8 row -- H e4m3 codes followed by H/128 fp32 scales,
// padded to 16 bytes -- with the same codec as the low-latency send, and the
// scatter / permute / fused-dispatch row movers carry those rows instead of the
// 2H-byte bf16 rows.
#include <cstdlib>

#include "ep_fp8.cuh"

namespace ep {

__host__ __device__ inline int64_t fp8_row_bytes(int H) { return ((int64_t)H + H / 32 + 15) / 16 * 16; }

// Items are (token, 16-channel group) pairs in row-major order; thread i of
// the grid takes items i, i + S, ... (S = grid threads), kU of them per round
// with all their loads issued before the first is quantised, so that each
// warp keeps kU KB of x in flight.  S and each block's first item are
// multiples of 8, and so is the number of groups per row, so an aligned group
// of 8 lanes always holds one whole 128-channel block (or none).
constexpr int kQuantU = 2;

template <typename Idx>
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint16_t* __restrict__ x, uint8_t* __restrict__ xq,
                                                            int64_t tokens, int H) {
    const int64_t row_q = fp8_row_bytes(H);
    const Idx ng = (Idx)(H / 16);
    const Idx total = (Idx)tokens * ng;
    const Idx S = (Idx)gridDim.x * blockDim.x;
    for (Idx r0 = (Idx)blockIdx.x * blockDim.x; r0 < total; r0 += S * kQuantU) {
        int4 p[kQuantU][2];
        Idx g[kQuantU], gi[kQuantU];
        bool act[kQuantU];
#pragma unroll
        for (int u = 0; u < kQuantU; ++u) {
            const Idx i = r0 + (Idx)u * S + threadIdx.x;
            act[u] = i < total;
            g[u] = i / ng;
            gi[u] = i - g[u] * ng;
            if (act[u]) {
                const uint16_t* src = x + (int64_t)g[u] * H + (int64_t)gi[u] * 16;
                p[u][0] = ld_nc_na_v4(src);
                p[u][1] = ld_nc_na_v4(src + 8);
            }
        }
#pragma unroll
        for (int u = 0; u < kQuantU; ++u) {
            float v[16];
            if (act[u]) {
                bf16x16_to_f32(p[u][0], p[u][1], v);
            } else {
#pragma unroll
                for (int k = 0; k < 16; ++k) v[k] = 0.0f;
            }
            float scale;
            const int4 codes = quantize16(v, &scale);
            if (act[u]) {
                uint8_t* q = xq + (int64_t)g[u] * row_q;
                st_na_v4(q + (int64_t)gi[u] * 16, codes);
                if ((gi[u] & 7) == 0) reinterpret_cast<float*>(q + H)[gi[u] >> 3] = scale;
            }
        }
    }
}

// Quantise-and-scatter: the fused dispatch of FP8 rows straight from the bf16
// tokens (one pass instead of ep_quantize_fp8 followed by
// ep_dispatch_permuted_fp8; the same bytes come out).  Persistent CTAs own
// contiguous token ranges; thread 0 streams the x rows global -> shared with
// cp.async.bulk a few tokens ahead (one mbarrier per stage); all threads
// quantise the staged row into an FP8 row in shared memory (two buffers);
// thread 0 then writes that row to each of the token's permuted rows with
// cp.async.bulk shared -> global, with the row's source token and weight.
constexpr int kQsMaxStages = 8;

struct QuantScatterArgs {
    const uint16_t* x;         // [tokens][H] bf16
    const int64_t* topk_idx;   // [tokens][K]
    const float* w;            // [tokens][K]
    // permuted destinations
    const int32_t* perm_pos;   // [tokens][K]
    int32_t* perm_src_token;   // [rows]
    float* perm_weight;        // [rows] or NULL
    // per-rank destinations (the dispatch scatter's receive layout)
    const int32_t* send_pos;   // [tokens][R]
    const int32_t* rank_base;  // [R+1]
    int32_t* recv_src_rank;    // [rows]
    int32_t* recv_src_idx;     // [rows]
    int32_t* recv_topk_idx;    // [rows][K]
    float* recv_topk_w;        // [rows][K]
    uint8_t* out;              // [rows][row_q]
    int64_t tokens, rows, row_q;
    int K, H, R, T, L;
    uint32_t* status;
};

__host__ __device__ inline size_t qs_fixed_smem() { return 128; }  // the stage mbarriers, padded

template <bool kRecv>
__global__ void __launch_bounds__(256) quant_scatter_kernel(QuantScatterArgs a, int stages, int64_t timeout_ns) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    const int H = a.H, K = a.K;
    const int64_t row_bytes = (int64_t)H * 2;
    uint8_t* xs = smem + qs_fixed_smem();                  // [stages][row_bytes]
    uint8_t* rows = xs + (size_t)stages * row_bytes;       // [2][row_q]
    __shared__ int sh_abort;
    __shared__ int64_t sh_dst[kRecv ? kMaxRanks : kMaxTopk];  // row per destination, -1 if none
    __shared__ int64_t sh_e[kMaxTopk];                             // the token's top-k entries
    __shared__ float sh_w[kMaxTopk];
    const int64_t q0 = a.tokens * blockIdx.x / gridDim.x, q1 = a.tokens * (blockIdx.x + 1) / gridDim.x;
    const int tid = threadIdx.x;
    auto issue_load = [&](int64_t q) {
        const int st = (int)((q - q0) % stages);
        mbar_arrive_expect_tx(&bar[st], (uint32_t)row_bytes);
        bulk_g2s(xs + (size_t)st * row_bytes, a.x + q * H, (uint32_t)row_bytes, &bar[st]);
    };
    int64_t next_load = q0;  // thread 0: first token whose load is not issued
    if (tid == 0) {
        for (int st = 0; st < stages; ++st) mbar_init(&bar[st], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
        for (; next_load < q1 && next_load < q0 + stages; ++next_load) issue_load(next_load);
        sh_abort = 0;
    }
    int64_t q_stop = q1;
    const int ngroups = H / 16;
    for (int64_t q = q0; q < q1; ++q) {
        const int64_t i = q - q0;
        const int st = (int)(i % stages);
        __syncthreads();  // thread 0 has seen the row buffer of token q-2 read out
        if (!mbar_wait_bounded(&bar[st], (uint32_t)((i / stages) & 1), timeout_ns)) {
            flag(a.status, FLAG_TIMEOUT);
            atomicExch(&sh_abort, 1);
        }
        __syncthreads();
        if (sh_abort) {
            q_stop = q;
            break;
        }
        uint8_t* row = rows + (size_t)(i & 1) * a.row_q;
        const uint8_t* xrow = xs + (size_t)st * row_bytes;
        // this token's routing, loaded now and kept until after the quantisation
        // (the loads' latency hides behind it)
        int64_t my_e = -1;
        float my_w = 0.0f;
        int32_t my_pos = -1;
        if (tid < K) {
            my_e = a.topk_idx[q * K + tid];
            my_w = a.w[q * K + tid];
            if constexpr (!kRecv) my_pos = a.perm_pos[q * K + tid];
        }
        if constexpr (kRecv) {
            if (tid >= 32 && tid - 32 < a.R) my_pos = a.send_pos[q * a.R + (tid - 32)];
        }
        for (int gi0 = 0; gi0 < ngroups; gi0 += blockDim.x) {
            const int gi = gi0 + tid;
            const bool act = gi < ngroups;
            float v[16];
            if (act) {
                const int4 p0 = *reinterpret_cast<const int4*>(xrow + (size_t)gi * 32);
                const int4 p1 = *reinterpret_cast<const int4*>(xrow + (size_t)gi * 32 + 16);
                bf16x16_to_f32(p0, p1, v);
            } else {
#pragma unroll
                for (int u = 0; u < 16; ++u) v[u] = 0.0f;
            }
            float scale;
            const int4 codes = quantize16(v, &scale);  // every lane takes part (shuffles)
            if (act) {
                *reinterpret_cast<int4*>(row + (size_t)gi * 16) = codes;
                if ((gi & 7) == 0) *reinterpret_cast<float*>(row + H + (gi >> 3) * 4) = scale;
            }
        }
        if (tid < K) {
            sh_e[tid] = my_e;
            sh_w[tid] = my_w;
        }
        if constexpr (kRecv) {
            // threads 32..32+R-1: one destination rank each, its receive row
            if (tid >= 32 && tid - 32 < a.R) {
                int64_t r = -1;
                if (my_pos >= 0) {
                    r = (int64_t)a.rank_base[tid - 32] + my_pos;
                    if (r >= a.rows) {
                        flag(a.status, FLAG_CAPACITY);
                        r = -1;
                    }
                }
                sh_dst[tid - 32] = r;
            }
        } else {
            // threads 0..K-1: one top-k entry each, its permuted row and metadata
            if (tid < K) {
                int64_t p = my_pos;
                if (p >= a.rows) {
                    flag(a.status, FLAG_CAPACITY);
                    p = -1;
                }
                if (p >= 0) {
                    a.perm_src_token[p] = (int32_t)q;
                    if (a.perm_weight) a.perm_weight[p] = my_w;
                }
                sh_dst[tid] = p;
            }
        }
        fence_proxy_async_smem();  // the row is read by the bulk copies below
        __syncthreads();
        if constexpr (kRecv) {
            // the receive rows' metadata: thread 32 + d for destination d
            if (tid >= 32 && tid - 32 < a.R) {
                const int d = tid - 32;
                const int64_t r = sh_dst[d];
                if (r >= 0) {
                    a.recv_src_rank[r] = (int32_t)(q / a.T);
                    a.recv_src_idx[r] = (int32_t)(q % a.T);
                    for (int k = 0; k < K; ++k) {
                        const int64_t e = sh_e[k];
                        const bool on = e >= 0 && e / a.L == d;
                        a.recv_topk_idx[r * K + k] = on ? (int32_t)(e - (int64_t)d * a.L) : -1;
                        a.recv_topk_w[r * K + k] = on ? sh_w[k] : 0.0f;
                    }
                }
            }
        }
        if (tid == 0) {
            const int nd = kRecv ? a.R : K;
            for (int j = 0; j < nd; ++j)
                if (sh_dst[j] >= 0) bulk_s2g(a.out + sh_dst[j] * a.row_q, row, (uint32_t)a.row_q);
            bulk_commit();
            // the x stage of this token is free: stream the token `stages` ahead
            if (next_load < q1) {
                fence_proxy_async_smem();
                issue_load(next_load);
                ++next_load;
            }
            // the row buffer of the previous token must be read out before reuse
            bulk_wait_read<1>();
        }
    }
    if (tid == 0) {
        bulk_wait_all();
        // after an aborted wait, let the loads still in flight land before leaving
        for (int64_t qq = q_stop; qq < next_load; ++qq)
            mbar_wait_bounded(&bar[(qq - q0) % stages], (uint32_t)(((qq - q0) / stages) & 1), timeout_ns);
    }
}

}  // namespace ep

using namespace ep;

extern "C" int64_t ep_fp8_row_bytes(int hidden) { return hidden > 0 ? fp8_row_bytes(hidden) : 0; }

static ep_status fp8_ok(const ep_ctx* c) {
    if (!c) return set_error(EP_ERR_INVALID_ARG, "ctx is NULL");
    if (c->cfg.hidden % 128) return set_error(EP_ERR_INVALID_ARG, "FP8 rows need hidden %% 128 == 0");
    return EP_OK;
}

extern "C" ep_status ep_quantize_fp8(ep_ctx* c, const void* x, uint8_t* xq, void* stream) {
    ep_status st = fp8_ok(c);
    if (st != EP_OK) return st;
    c->last_launches = 0;
    const int64_t tokens = (int64_t)c->cfg.num_ranks * c->cfg.num_tokens;
    if (tokens == 0) return EP_OK;
    if (!x || !xq || !aligned16(x) || !aligned16(xq)) return set_error(EP_ERR_INVALID_ARG, "x and xq must be 16-byte aligned");
    // one wave of resident CTAs
    const int64_t total = tokens * (c->cfg.hidden / 16);
    const bool narrow = total <= (int64_t)UINT32_MAX - 2 * kQuantU * 256 * (int64_t)c->num_sms * 8;
    // resident CTAs per SM, queried once per device and index width
    static int cached[kMaxDevicesTracked][2] = {};
    const bool cacheable = c->device >= 0 && c->device < kMaxDevicesTracked;
    int per_sm = cacheable ? cached[c->device][narrow] : 0;
    if (per_sm == 0) {
        EP_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, narrow ? quantize_rows_kernel<uint32_t> : quantize_rows_kernel<uint64_t>, 256, 0));
        if (per_sm < 1) per_sm = 1;
        if (per_sm > 8) per_sm = 8;
        if (cacheable) cached[c->device][narrow] = per_sm;
    }
    int64_t grid = (int64_t)c->num_sms * per_sm;
    if (grid > (total + 255) / 256) grid = (total + 255) / 256;
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    if (narrow)
        quantize_rows_kernel<uint32_t><<<(int)grid, 256, 0, as_stream(stream)>>>(xb, xq, tokens, c->cfg.hidden);
    else
        quantize_rows_kernel<uint64_t><<<(int)grid, 256, 0, as_stream(stream)>>>(xb, xq, tokens, c->cfg.hidden);
    EP_CHECK_LAUNCH("quantize_rows_kernel");
    c->last_launches = 1;
    return EP_OK;
}

extern "C" ep_status ep_dispatch_fp8(ep_ctx* c, const uint8_t* xq, const int64_t* topk_idx, const float* topk_weights,
                                     const ep_dispatch_handle* h, uint8_t* recv_xq, int32_t* recv_src_rank,
                                     int32_t* recv_src_idx, int32_t* recv_topk_idx, float* recv_topk_weights,
                                     int64_t recv_capacity_rows, void* stream) {
    ep_status st = fp8_ok(c);
    if (st != EP_OK) return st;
    return dispatch_rows(c, xq, fp8_row_bytes(c->cfg.hidden), topk_idx, topk_weights, h, recv_xq, recv_src_rank,
                         recv_src_idx, recv_topk_idx, recv_topk_weights, recv_capacity_rows, stream);
}

extern "C" ep_status ep_permute_fp8(ep_ctx* c, const ep_dispatch_handle* h, const uint8_t* recv_xq,
                                    const int32_t* recv_src_rank, const int32_t* recv_src_idx,
                                    const int32_t* recv_topk_idx, int64_t num_recv_rows, uint8_t* permuted_xq,
                                    int32_t* perm_src_row, int64_t perm_capacity_rows, void* stream) {
    ep_status st = fp8_ok(c);
    if (st != EP_OK) return st;
    return permute_rows(c, h, recv_xq, fp8_row_bytes(c->cfg.hidden), recv_src_rank, recv_src_idx, recv_topk_idx,
                        num_recv_rows, permuted_xq, perm_src_row, perm_capacity_rows, stream);
}

extern "C" ep_status ep_dispatch_permuted_fp8(ep_ctx* c, const uint8_t* xq, const int64_t* topk_idx,
                                              const float* topk_weights, const ep_dispatch_handle* h,
                                              uint8_t* permuted_xq, int32_t* perm_src_token, float* perm_weight,
                                              int64_t perm_capacity_rows, void* stream) {
    ep_status st = fp8_ok(c);
    if (st != EP_OK) return st;
    return dispatch_permuted_rows(c, xq, fp8_row_bytes(c->cfg.hidden), topk_idx, topk_weights, h, permuted_xq,
                                  perm_src_token, perm_weight, perm_capacity_rows, stream);
}

template <bool kRecv>
static ep_status launch_quant_scatter(ep_ctx* c, const QuantScatterArgs& a, void* stream) {
    // three CTAs per SM, ~72 KB each: two FP8 row buffers and as many staged x
    // rows as fit (EP_QS_CTAS_PER_SM and EP_QS_STAGE_KB override the shape)
    static const int qs_ctas = [] {
        const char* v = getenv("EP_QS_CTAS_PER_SM");
        const int x = v ? atoi(v) : 3;
        return x < 1 ? 1 : (x > 8 ? 8 : x);
    }();
    static const int qs_kb = [] {
        const char* v = getenv("EP_QS_STAGE_KB");
        const int x = v ? atoi(v) : 72;
        return x < 32 ? 32 : (x > 220 ? 220 : x);
    }();
    const int64_t row_bytes = (int64_t)a.H * 2;
    const size_t budget = (size_t)qs_kb * 1024;
    int stages = (int)((budget - qs_fixed_smem() - 2 * (size_t)a.row_q) / (size_t)row_bytes);
    if (stages > kQsMaxStages) stages = kQsMaxStages;
    if (stages < 2) stages = 2;
    const size_t smem = qs_fixed_smem() + (size_t)stages * row_bytes + 2 * (size_t)a.row_q;
    static int raised[kMaxDevicesTracked] = {};
    if (c->device < 0 || c->device >= kMaxDevicesTracked || raised[c->device] < (int)smem) {
        EP_CUDA(cudaFuncSetAttribute(quant_scatter_kernel<kRecv>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem));
        if (c->device >= 0 && c->device < kMaxDevicesTracked) raised[c->device] = (int)smem;
    }
    int64_t grid = (int64_t)c->num_sms * qs_ctas;
    if (grid > a.tokens) grid = a.tokens;
    quant_scatter_kernel<kRecv><<<(int)grid, 256, smem, as_stream(stream)>>>(a, stages, c->wait_timeout_ns);
    EP_CHECK_LAUNCH("quant_scatter_kernel");
    c->last_launches = 1;
    return EP_OK;
}

static QuantScatterArgs quant_args(const ep_ctx* c, const void* x, const int64_t* topk_idx, const float* w,
                                   uint8_t* out, int64_t rows) {
    const ep_config& f = c->cfg;
    QuantScatterArgs a{};
    a.x = static_cast<const uint16_t*>(x);
    a.topk_idx = topk_idx;
    a.w = w;
    a.out = out;
    a.tokens = (int64_t)f.num_ranks * f.num_tokens;
    a.rows = rows;
    a.row_q = fp8_row_bytes(f.hidden);
    a.K = f.num_topk;
    a.H = f.hidden;
    a.R = f.num_ranks;
    a.T = f.num_tokens;
    a.L = c->L;
    a.status = c->status;
    return a;
}

extern "C" ep_status ep_dispatch_permuted_quant(ep_ctx* c, const void* x, const int64_t* topk_idx,
                                                const float* topk_weights, const ep_dispatch_handle* h,
                                                uint8_t* permuted_xq, int32_t* perm_src_token, float* perm_weight,
                                                int64_t perm_capacity_rows, void* stream) {
    ep_status st = fp8_ok(c);
    if (st != EP_OK) return st;
    if (!h) return set_error(EP_ERR_INVALID_ARG, "handle is NULL");
    c->last_launches = 0;
    const ep_config& f = c->cfg;
    if (f.num_tokens == 0 || (c->totals_known && c->last_total_perm == 0) || perm_capacity_rows == 0) return EP_OK;
    if (!x || !aligned16(x) || !permuted_xq || !aligned16(permuted_xq))
        return set_error(EP_ERR_INVALID_ARG, "x and permuted_xq must be 16-byte aligned");
    if (!topk_idx || !h->perm_pos || !perm_src_token || (perm_weight && !topk_weights))
        return set_error(EP_ERR_INVALID_ARG, "NULL fused dispatch argument");
    if (c->totals_known && perm_capacity_rows < c->last_total_perm)
        return set_error(EP_ERR_CAPACITY, "permuted buffers hold %lld rows, notify counted %lld",
                         (long long)perm_capacity_rows, (long long)c->last_total_perm);
    QuantScatterArgs a = quant_args(c, x, topk_idx, topk_weights, permuted_xq, perm_capacity_rows);
    a.perm_pos = h->perm_pos;
    a.perm_src_token = perm_src_token;
    a.perm_weight = perm_weight;
    return launch_quant_scatter<false>(c, a, stream);
}

extern "C" ep_status ep_dispatch_quant(ep_ctx* c, const void* x, const int64_t* topk_idx, const float* topk_weights,
                                       const ep_dispatch_handle* h, uint8_t* recv_xq, int32_t* recv_src_rank,
                                       int32_t* recv_src_idx, int32_t* recv_topk_idx, float* recv_topk_weights,
                                       int64_t recv_capacity_rows, void* stream) {
    ep_status st = fp8_ok(c);
    if (st != EP_OK) return st;
    if (!h) return set_error(EP_ERR_INVALID_ARG, "handle is NULL");
    c->last_launches = 0;
    const ep_config& f = c->cfg;
    if (f.num_tokens == 0 || (c->totals_known && c->last_total_recv == 0) || recv_capacity_rows == 0) return EP_OK;
    if (!x || !aligned16(x) || !recv_xq || !aligned16(recv_xq))
        return set_error(EP_ERR_INVALID_ARG, "x and recv_xq must be 16-byte aligned");
    if (!topk_idx || !topk_weights || !h->send_pos || !h->rank_base || !recv_src_rank || !recv_src_idx ||
        !recv_topk_idx || !recv_topk_weights)
        return set_error(EP_ERR_INVALID_ARG, "NULL dispatch argument");
    if (c->totals_known && recv_capacity_rows < c->last_total_recv)
        return set_error(EP_ERR_CAPACITY, "recv buffers hold %lld rows, notify counted %lld",
                         (long long)recv_capacity_rows, (long long)c->last_total_recv);
    QuantScatterArgs a = quant_args(c, x, topk_idx, topk_weights, recv_xq, recv_capacity_rows);
    a.send_pos = h->send_pos;
    a.rank_base = h->rank_base;
    a.recv_src_rank = recv_src_rank;
    a.recv_src_idx = recv_src_idx;
    a.recv_topk_idx = recv_topk_idx;
    a.recv_topk_w = recv_topk_weights;
    return launch_quant_scatter<true>(c, a, stream);
}
