// ep_combine.cu -- the weighted reductions back to the original token order:
//
//  * combine (page "DeepEP 学习笔记", sections "combine 过程" and "DeepEP v2 /
//    direct 模式": the rank-level partial result of a token is reduced inside
//    the rank that holds its experts, the epilogue reduces over destination
//    ranks);
//  * hierarchical combine (same page, section "hybrid 模式": local reduce inside
//    the node, then the final reduce at the source);
//  * low-latency BF16 combine (page "事件驱动 EP 内核的调度策略与零拷贝通信", section
//    "低延迟模式": combine stays in BF16).
//
// One warp owns one token (or a channel slice of it).  Lanes 0..K-1 read the
// token's top-k entries and order them by (rank, k) (or by k for the
// low-latency mode); every lane then owns U vectors of 8 channels per step,
// loads them from each of the token's rows before accumulating (up to U*K
// 16-byte loads in flight per lane), and reduces in fp32 with explicit fused
// multiply-adds in the defined order.  The partial sums are never materialised: on one GPU a
// "partial" is the grouping of the sum.  Output: bf16, round to nearest even.
#include <climits>
#include <cstdlib>

#include "ep_internal.cuh"
#include "ep_combine.cuh"

namespace ep {

constexpr int kCombineThreads = 128;  // 4 warps: the grid spreads more evenly over the SMs than with 8
constexpr int kCombineWarps = kCombineThreads / 32;

__device__ __forceinline__ void bf16x8_to_f32(const int4& v, float* f) {
    const uint32_t u[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ int4 f32x8_to_bf16(const float* f) {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        u[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    return make_int4((int)u[0], (int)u[1], (int)u[2], (int)u[3]);
}

// MODE 0: flat (rank partials), 1: hierarchical (rank, node, final), 2: low-latency (k order)
template <int KMAX, int MODE, int U>
__global__ void __launch_bounds__(kCombineThreads, (KMAX <= 8 ? (U == 2 ? 2 : 3) : 1) * (256 / kCombineThreads)) combine_kernel(CombineArgs a) {
    __shared__ int64_t sh_row[kCombineWarps][KMAX];
    __shared__ float sh_w[kCombineWarps][KMAX];
    __shared__ uint8_t sh_brk[kCombineWarps][KMAX];  // bit0: new rank group, bit1: new node group
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = a.K;
    const int64_t n_tok = (int64_t)a.R * a.n;
    const int nvec = a.H / 8;
    const int64_t row_bytes = (int64_t)a.H * 2;
    // a work item is (token, channel slice); small batches use several slices
    // per token so that enough loads are in flight
    const int per = (nvec + a.splits - 1) / a.splits;
    const int64_t n_items = n_tok * a.splits;
    const int64_t stride = (int64_t)gridDim.x * kCombineWarps;
    // The entry loads of a warp's next item are issued before the current
    // item's row loads, so that they arrive while the rows stream in (otherwise
    // every item would start with idle dependent loads).
    auto token_of = [&](int64_t q) -> int64_t {
        const int64_t tok = q / a.splits;
        return (int64_t)(tok / a.n) * a.T + a.t0 + (int)(tok % a.n);
    };
    int64_t nx_e = -1, nx_aux = -1;  // topk_idx and perm_pos / slot of the next item's entry `lane`
    float nx_w = 0.0f;
    int64_t q = (int64_t)blockIdx.x * kCombineWarps + warp;
    if (q < n_items && lane < K) {
        const int64_t g = token_of(q);
        nx_e = a.topk_idx[g * K + lane];
        nx_w = a.w[g * K + lane];
        nx_aux = MODE == 2 ? a.slot[g * K + lane] : a.perm_pos[g * K + lane];
    }
    // launched as a programmatic dependent (low-latency mode): the entries above
    // (inputs the previous kernel does not write) load before its completion;
    // the rows and the receive layout only after.  Without that launch
    // attribute the wait returns at once.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (; q < n_items; q += stride) {
        const int64_t tok = q / a.splits;
        const int c_lo = (int)(q % a.splits) * per;
        const int c_hi = min(nvec, c_lo + per);
        const int s = (int)(tok / a.n);
        const int t = a.t0 + (int)(tok % a.n);
        const int64_t g = (int64_t)s * a.T + t;
        // ---- entries of this token -------------------------------------------------
        bool valid = false;
        int d = INT_MAX;
        int64_t row = 0;
        float wk = 0.0f;
        if (lane < K) {
            const int64_t e = nx_e;
            if (e >= 0 && e < a.E) {
                d = (int)(e / a.L);
                if (MODE == 2) {
                    const int l = (int)(e % a.L);
                    const int32_t sl = (int32_t)nx_aux;
                    const int32_t begin = a.layout_range[(((int64_t)d * a.L + l) * a.R + s) * 2];
                    row = ((int64_t)d * a.L + l) * a.rows_per_expert + begin + sl;
                    valid = sl >= 0 && row >= 0 && row < a.y_rows;
                } else {
                    row = nx_aux;
                    valid = row >= 0 && row < a.y_rows;
                }
                if (!valid) flag(a.status, FLAG_BOUNDS);
                wk = nx_w;
            }
        }
        if (q + stride < n_items && lane < K) {  // the next item's entries, in flight from here on
            const int64_t gn = token_of(q + stride);
            nx_e = a.topk_idx[gn * K + lane];
            nx_w = a.w[gn * K + lane];
            nx_aux = MODE == 2 ? a.slot[gn * K + lane] : a.perm_pos[gn * K + lane];
        }
        const int key = valid ? (MODE == 2 ? lane : d * 32 + lane) : INT_MAX;
        int rank = 0;
        bool new_rank = true, new_node = true;
        for (int j = 0; j < K; ++j) {
            const int kj = __shfl_sync(0xffffffffu, key, j);
            const int dj = __shfl_sync(0xffffffffu, d, j);
            if (kj < key) {
                ++rank;
                if (dj == d) new_rank = false;
                if (dj / a.G == d / a.G) new_node = false;
            }
        }
        const int nvalid = __popc(__ballot_sync(0xffffffffu, valid));
        if (valid) {
            sh_row[warp][rank] = row;
            sh_w[warp][rank] = wk;
            sh_brk[warp][rank] = (uint8_t)((new_rank ? 1 : 0) | (new_node ? 2 : 0));
        }
        __syncwarp();
        int64_t roff[KMAX];
        float wr[KMAX];
        uint8_t br[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            roff[j] = j < nvalid ? sh_row[warp][j] * row_bytes : 0;
            wr[j] = j < nvalid ? sh_w[warp][j] : 0.0f;
            br[j] = j < nvalid ? sh_brk[warp][j] : 0;
        }
        __syncwarp();
        const uint8_t* y = static_cast<const uint8_t*>(a.y);
        int4* out = reinterpret_cast<int4*>(static_cast<uint8_t*>(a.out) + g * row_bytes);
        // ---- channels: U vectors of 8 channels per lane per step, every load of
        // the step issued before the first is used ----------------------------------
        for (int c = c_lo + lane; c < c_hi; c += 32 * U) {
            int4 v[U][KMAX];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int cu = c + 32 * u;
#pragma unroll
                for (int j = 0; j < KMAX; ++j)
                    if (j < nvalid && cu < c_hi) v[u][j] = ld_nc_na_v4(y + roff[j] + (int64_t)cu * 16);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int cu = c + 32 * u;
                if (cu >= c_hi) break;
                float fin[8], nod[8], par[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) fin[i] = nod[i] = par[i] = 0.0f;
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    if (j < nvalid) {
                        if (MODE != 2 && j > 0 && (br[j] & 1)) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                if (MODE == 1) {
                                    nod[i] = __fadd_rn(nod[i], par[i]);
                                    if (br[j] & 2) {
                                        fin[i] = __fadd_rn(fin[i], nod[i]);
                                        nod[i] = 0.0f;
                                    }
                                } else {
                                    fin[i] = __fadd_rn(fin[i], par[i]);
                                }
                                par[i] = 0.0f;
                            }
                        }
                        float yv[8];
                        bf16x8_to_f32(v[u][j], yv);
#pragma unroll
                        for (int i = 0; i < 8; ++i) par[i] = __fmaf_rn(wr[j], yv[i], par[i]);
                    }
                }
                if (nvalid > 0) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (MODE == 1) {
                            nod[i] = __fadd_rn(nod[i], par[i]);
                            fin[i] = __fadd_rn(fin[i], nod[i]);
                        } else if (MODE == 0) {
                            fin[i] = __fadd_rn(fin[i], par[i]);
                        } else {
                            fin[i] = par[i];
                        }
                    }
                }
                st_na_v4(out + cu, f32x8_to_bf16(fin));
            }
        }
    }
}

// vectors per lane per step for K <= 8: 2 (16 loads of 16 B in flight per
// lane at 16 warps/SM of registers) beat 1 (8 loads at 24 warps/SM) on GB300:
// prefill combine 673 -> 649 us, hierarchical 2713 -> 2647 us.  Larger K
// keeps 1 (the row arrays take the registers).
static int combine_vectors(int mode) {
    static const int forced = [] {  // EP_COMBINE_VEC: 1 or 2, for sweeps of the flat and staged modes
        const char* v = getenv("EP_COMBINE_VEC");
        return v ? atoi(v) : 0;
    }();
    if (mode != 2 && (forced == 1 || forced == 2)) return forced;
    return 2;
}

// pdl: programmatic stream serialisation, so that the kernel may start while
// the previous one on the stream finishes (it waits for it before reading rows)
template <class Kern>
static cudaError_t launch_combine_kernel(Kern kern, int grid, cudaStream_t s, const CombineArgs& a, bool pdl) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3(kCombineThreads);
    lc.dynamicSmemBytes = 0;
    lc.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&lc, kern, a);
}

// The low-latency combine is launched this way: it starts as the receive's
// CTAs exit (their exit is the trigger), with its launch and first entry loads
// overlapping the receive's completion: eager decode layer 111.7-113.7 ->
// 109.6 us; a CUDA graph of the layer (111.1 us) and two overlapped
// microbatches (105.5 us/layer) are unchanged.
template <int MODE>
static cudaError_t launch_mode(const CombineArgs& a, int grid, int vec, cudaStream_t s) {
    const bool pdl = MODE == 2;
    if (a.K <= 8) {
        if (vec == 2) return launch_combine_kernel(combine_kernel<8, MODE, 2>, grid, s, a, pdl);
        return launch_combine_kernel(combine_kernel<8, MODE, 1>, grid, s, a, pdl);
    }
    if (a.K <= 16) return launch_combine_kernel(combine_kernel<16, MODE, 1>, grid, s, a, pdl);
    return launch_combine_kernel(combine_kernel<32, MODE, 1>, grid, s, a, pdl);
}

ep_status launch_combine(const CombineArgs& a, int mode, int num_sms, cudaStream_t s) {
    const int64_t n_tok = (int64_t)a.R * a.n;
    if (n_tok <= 0) return EP_OK;
    CombineArgs b = a;
    // Work items are (token, channel slice).  A slice reloads the token's
    // entries, so use the fewest slices per token that still give about three
    // quarters of the resident warps an item (measured on the decode batch:
    // 1-2 slices 49 us, 7 slices 53 us, 8 slices 57 us).
    const int nvec = a.H / 8;
    const int vec = a.K <= 8 ? combine_vectors(mode) : 1;
    const int64_t conc = (int64_t)num_sms * (vec == 2 ? 2 : 3) * (256 / kCombineThreads) * kCombineWarps;  // resident warps
    int max_splits = nvec / 32 < 8 ? nvec / 32 : 8;
    if (max_splits < 1) max_splits = 1;
    int splits = max_splits;
    for (int sp = 1; sp <= max_splits; ++sp) {
        if (n_tok * sp * 4 >= conc * 3) {
            splits = sp;
            break;
        }
    }
    static const int forced = [] {  // EP_COMBINE_SPLITS: launch-shape override for sweeps
        const char* v = getenv("EP_COMBINE_SPLITS");
        return v ? atoi(v) : 0;
    }();
    if (forced >= 1 && forced <= max_splits) splits = forced;
    b.splits = splits;
    const int64_t items = n_tok * splits;
    int64_t want = (items + kCombineWarps - 1) / kCombineWarps;
    const int64_t cap = (int64_t)num_sms * 16 * (256 / kCombineThreads);
    const int grid = (int)(want < cap ? want : cap);
    cudaError_t e = mode == 0   ? launch_mode<0>(b, grid, vec, s)
                    : mode == 1 ? launch_mode<1>(b, grid, vec, s)
                                : launch_mode<2>(b, grid, vec, s);
    if (e != cudaSuccess) return cuda_error(e, "combine kernel");
    return EP_OK;
}

}  // namespace ep

using namespace ep;

static ep_status combine_common(ep_ctx* c, const ep_dispatch_handle* h, const void* y, int64_t perm_rows,
                                const int64_t* topk_idx, const float* w, void* out, void* stream, int mode) {
    if (!c || !h) return set_error(EP_ERR_INVALID_ARG, "ctx or handle is NULL");
    c->last_launches = 0;
    const ep_config& f = c->cfg;
    if (f.num_tokens == 0) return EP_OK;
    if (!out || !aligned16(out)) return set_error(EP_ERR_INVALID_ARG, "out must be a 16-byte aligned pointer");
    if (perm_rows > 0 && (!y || !aligned16(y))) return set_error(EP_ERR_INVALID_ARG, "expert_out must be 16-byte aligned");
    if (!topk_idx || !w || !h->perm_pos) return set_error(EP_ERR_INVALID_ARG, "NULL combine argument");
    CombineArgs a{};
    a.y = y;
    a.y_rows = perm_rows;
    a.topk_idx = topk_idx;
    a.w = w;
    a.perm_pos = h->perm_pos;
    a.out = out;
    a.R = f.num_ranks;
    a.E = f.num_experts;
    a.L = c->L;
    a.K = f.num_topk;
    a.T = f.num_tokens;
    a.H = f.hidden;
    a.G = mode == 1 ? c->G : f.num_ranks;
    a.t0 = 0;
    a.n = f.num_tokens;
    a.status = c->status;
    ep_status st = launch_combine(a, mode, c->num_sms, as_stream(stream));
    if (st == EP_OK) c->last_launches = 1;
    return st;
}

extern "C" ep_status ep_combine(ep_ctx* c, const ep_dispatch_handle* h, const void* expert_out, int64_t num_perm_rows,
                                const int64_t* topk_idx, const float* topk_weights, void* out, void* stream) {
    return combine_common(c, h, expert_out, num_perm_rows, topk_idx, topk_weights, out, stream, 0);
}

extern "C" ep_status ep_combine_hier(ep_ctx* c, const ep_dispatch_handle* h, const void* expert_out,
                                     int64_t num_perm_rows, const int64_t* topk_idx, const float* topk_weights,
                                     void* out, void* stream) {
    if (c && c->cfg.num_nodes < 2) return set_error(EP_ERR_INVALID_ARG, "ep_combine_hier needs num_nodes > 1");
    return combine_common(c, h, expert_out, num_perm_rows, topk_idx, topk_weights, out, stream, 1);
}
