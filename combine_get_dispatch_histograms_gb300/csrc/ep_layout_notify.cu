// ep_layout_notify.cu -- context, error plumbing, and the two small integer
// steps of the normal path:
//
//  * get_dispatch_layout (page "DeepEP 学习笔记", section "dispatch 前：全局布局与
//    通知"): per source rank, the histograms num_tokens_per_expert,
//    num_tokens_per_rank and the lookup table is_token_in_rank (plus the node
//    versions for the hierarchical mode).
//  * notify_dispatch (same section, notify steps 1-3; page "事件驱动 EP 内核的调度
//    策略与零拷贝通信", section "事件驱动调度的本质": count, exchange, prefix-sum to
//    the write offset of each source): receiver totals, ragged offsets,
//    channel_prefix_matrix, and every token's destination row (send_pos,
//    perm_pos, stage_pos) so that the copy kernels need no atomics and the
//    order of the result is fixed.
//
// All R virtual ranks are handled by one launch.  The exchange of counts
// between ranks is a transpose read of the [R][R] matrix and the barrier of
// the original design is stream order.
#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "ep_internal.cuh"

namespace ep {

static thread_local std::string g_last_error;

ep_status set_error(ep_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

ep_status cuda_error(cudaError_t e, const char* what) {
    return set_error(EP_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

ep_status status_from_flags(uint32_t flags) {
    if (flags & FLAG_INVALID_TOPK) return set_error(EP_ERR_INVALID_INPUT, "topk_idx holds a value outside [-1, E)");
    if (flags & FLAG_TIMEOUT) return set_error(EP_ERR_TIMEOUT, "a bounded device wait ran out");
    if (flags & FLAG_CAPACITY) return set_error(EP_ERR_CAPACITY, "a device-side capacity check failed");
    if (flags & FLAG_BOUNDS) return set_error(EP_ERR_INVALID_INPUT, "a device-side index check failed");
    return EP_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ============================================================================
// Layout kernel
// ============================================================================
// grid = (tiles_per_src, R), block = kTileTokens threads, one token per thread.
// Each CTA histograms its tile in shared memory and stores the partial counts;
// the last CTA of a source (completion counter) sums the partials of that
// source into the outputs and re-arms the counter.  Integer sums do not
// depend on the order, so the result is deterministic.
// Returns true in the CTA that completed source s (it wrote the sums).
__device__ bool layout_tile(const int64_t* __restrict__ topk_idx, int R, int E, int K, int T, int L, int N, int G,
                            TileGeom geom, int32_t* __restrict__ ntpe, int32_t* __restrict__ ntpr,
                            uint8_t* __restrict__ itir, int32_t* __restrict__ ntpn, uint8_t* __restrict__ itin,
                            int32_t* __restrict__ part, uint32_t* __restrict__ done, uint32_t* __restrict__ status,
                            int s, int tile) {
    extern __shared__ int32_t sh_cnt[];  // [E + R + N]
    __shared__ bool is_last;
    const int W = E + R + N;
    const int lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < W; i += blockDim.x) sh_cnt[i] = 0;
    __syncthreads();

    int lo, hi;
    tile_range(geom, tile, &lo, &hi);
    const int t = lo + threadIdx.x;
    uint64_t mask = 0;
    if (t < hi) {
        const int64_t* row = topk_idx + ((int64_t)s * T + t) * K;
        for (int k = 0; k < K; ++k) {
            const int64_t e = row[k];
            if (e == -1) continue;
            if (e < -1 || e >= E) {
                flag(status, FLAG_INVALID_TOPK);
                continue;
            }
            atomicAdd(&sh_cnt[e], 1);
            mask |= 1ull << (int)(e / L);
        }
        uint8_t* out = itir + ((int64_t)s * T + t) * R;
        if ((R & 3) == 0 && ((reinterpret_cast<uintptr_t>(out) & 3u) == 0)) {
            for (int d = 0; d < R; d += 4) {
                uint32_t wv = (uint32_t)((mask >> d) & 1) | ((uint32_t)((mask >> (d + 1)) & 1) << 8) |
                              ((uint32_t)((mask >> (d + 2)) & 1) << 16) | ((uint32_t)((mask >> (d + 3)) & 1) << 24);
                *reinterpret_cast<uint32_t*>(out + d) = wv;
            }
        } else {
            for (int d = 0; d < R; ++d) out[d] = (uint8_t)((mask >> d) & 1);
        }
        if (N > 0) {
            uint8_t* on = itin + ((int64_t)s * T + t) * N;
            for (int n = 0; n < N; ++n) {
                const uint64_t node_bits = (G >= 64) ? ~0ull : (((1ull << G) - 1) << (n * G));
                on[n] = (mask & node_bits) ? 1 : 0;
            }
        }
    }
    // per-rank and per-node counts, one shared atomic per warp and bin
    for (int d = 0; d < R; ++d) {
        const uint32_t b = __ballot_sync(0xffffffffu, (mask >> d) & 1);
        if (lane == 0 && b) atomicAdd(&sh_cnt[E + d], __popc(b));
    }
    for (int n = 0; n < N; ++n) {
        const uint64_t node_bits = (G >= 64) ? ~0ull : (((1ull << G) - 1) << (n * G));
        const uint32_t b = __ballot_sync(0xffffffffu, (mask & node_bits) != 0);
        if (lane == 0 && b) atomicAdd(&sh_cnt[E + R + n], __popc(b));
    }
    __syncthreads();
    int32_t* mine = part + ((int64_t)s * geom.tiles_per_src + tile) * W;
    for (int i = threadIdx.x; i < W; i += blockDim.x) mine[i] = sh_cnt[i];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = (atomicAdd(&done[s], 1u) == (uint32_t)(geom.tiles_per_src - 1));
    __syncthreads();
    if (!is_last) return false;
    __threadfence();
    const int32_t* first = part + (int64_t)s * geom.tiles_per_src * W;
    for (int i = threadIdx.x; i < W; i += blockDim.x) {
        int32_t acc = 0;
        for (int j = 0; j < geom.tiles_per_src; ++j) acc += __ldcg(first + (int64_t)j * W + i);
        if (i < E) ntpe[(int64_t)s * E + i] = acc;
        else if (i < E + R) ntpr[(int64_t)s * R + (i - E)] = acc;
        else ntpn[(int64_t)s * N + (i - E - R)] = acc;
    }
    if (threadIdx.x == 0) done[s] = 0;  // re-arm for the next call (stream ordered)
    return true;
}

__global__ void __launch_bounds__(kTileTokens)
layout_kernel(const int64_t* __restrict__ topk_idx, int R, int E, int K, int T, int L, int N, int G,
              TileGeom geom, int32_t* __restrict__ ntpe, int32_t* __restrict__ ntpr,
              uint8_t* __restrict__ itir, int32_t* __restrict__ ntpn, uint8_t* __restrict__ itin,
              int32_t* __restrict__ part, uint32_t* __restrict__ done, uint32_t* __restrict__ status) {
    layout_tile(topk_idx, R, E, K, T, L, N, G, geom, ntpe, ntpr, itir, ntpn, itin, part, done, status, blockIdx.y,
                blockIdx.x);
}

// ============================================================================
// Notify, pass 1: per-tile partial counts + (one extra CTA) the global scans
// ============================================================================
// Linear grid of R * tiles_per_src + 1 CTAs.  CTA b < R*tiles counts tile
// (b % tiles) of source (b / tiles): per receiver d (is_token_in_rank), per
// expert e (topk_idx) and per node n.  The extra CTA performs the small scans
// over the layout histograms, which need no tile data:
//   recv_count, recv_offsets, num_recv_tokens, rank_base,
//   num_recv_per_expert, expert_offsets, perm_rank_base,
//   ebase[s][e] = first permuted row of (source s, expert e),
//   stage_base and sbase[s][n] (hierarchical),
// and writes the receive counts to the CPU-mapped block.
struct NotifyArgs {
    const int64_t* topk_idx;
    const int32_t* ntpe;
    const int32_t* ntpr;
    const uint8_t* itir;
    const int32_t* ntpn;
    const uint8_t* itin;
    ep_dispatch_handle h;
    int R, E, K, T, L, N, G;
    int align;       // expert alignment of the permuted blocks (1 = none)
    TileGeom geom;
    int32_t* part;   // [R][tiles][E + R + N]
    int32_t* ebase;  // [R][E]
    int32_t* sbase;  // [R][N]
    int32_t* host;   // mapped: [R] num_recv, [R*L] per expert, [3] totals, [1] status, [1] epoch
    uint32_t* status;
    int32_t epoch;   // sequence number of this notify call
};

// Exclusive prefix sum over the block's threads (blockDim.x a multiple of 32,
// at most 1024): warp shuffles, then the warp totals scanned by warp 0.
__device__ int32_t block_exclusive_scan(int32_t v, int32_t* sh_tmp /* >= 32 ints */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    __syncthreads();
    if (lane == 31) sh_tmp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int32_t t = lane < nw ? sh_tmp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < nw) sh_tmp[lane] = t - (lane < nw ? sh_tmp[lane] : 0);  // exclusive warp offsets
    }
    __syncthreads();
    return sh_tmp[warp] + inc - v;
}

__device__ void notify_global_scan(const NotifyArgs& a, int32_t* sh /* >= 2E + 3R + 98 ints */) {
    const int R = a.R, E = a.E, L = a.L, N = a.N, G = a.G;
    int32_t* tot = sh;              // [E]  pairs per expert (over sources)
    int32_t* off = tot + E;         // [E]  first permuted row of each expert
    int32_t* nrecv = off + E;       // [R]  rows per receiver
    int32_t* rbase = nrecv + R;     // [R+1]
    int32_t* scan_tmp = rbase + R + 1;  // [32]
    int32_t* hcnt = scan_tmp + 32;      // [R+1] staged rows per home rank
    __shared__ int32_t sh_total_recv, sh_total_perm;
    // (a) per receiver: the transpose of the count matrix and its exclusive
    // prefix over sources; (b) per expert: totals over sources.  All loads of
    // a thread are independent, so each phase costs one memory round trip.
    for (int d = threadIdx.x; d < R; d += blockDim.x) {
        int32_t acc = 0;
        for (int s0 = 0; s0 < R; s0 += 16) {  // loads first: the stores may alias them
            int32_t c[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) c[u] = s0 + u < R ? a.ntpr[(s0 + u) * R + d] : 0;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                if (s0 + u >= R) break;
                a.h.recv_count[d * R + s0 + u] = c[u];
                a.h.recv_offsets[d * R + s0 + u] = acc;
                acc += c[u];
            }
        }
        a.h.num_recv_tokens[d] = acc;
        a.host[d] = acc;
        nrecv[d] = acc;
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int32_t acc = 0;
#pragma unroll 16
        for (int s = 0; s < R; ++s) acc += a.ntpe[(int64_t)s * E + e];
        tot[e] = acc;
        a.h.num_recv_per_expert[e] = acc;  // [d][l] flattened == e
        a.host[R + e] = acc;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t acc = 0;
        for (int d = 0; d < R; ++d) {
            rbase[d] = acc;
            acc += nrecv[d];
        }
        rbase[R] = acc;
        sh_total_recv = acc;
    }
    // (c) exclusive scan over experts in (d, l) order: contiguous chunk per
    // thread; each expert's block takes its count rounded up to the alignment
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = threadIdx.x * per;
    const int al = a.align > 1 ? a.align : 1;
    auto rows_of = [al](int32_t n) -> int32_t { return (n + al - 1) / al * al; };
    int32_t local = 0;
    for (int e = e0; e < e0 + per && e < E; ++e) local += rows_of(tot[e]);
    int32_t run = block_exclusive_scan(local, scan_tmp);
    for (int e = e0; e < e0 + per && e < E; ++e) {
        off[e] = run;
        run += rows_of(tot[e]);
    }
    __syncthreads();
    const int32_t total_perm = off[E - 1] + rows_of(tot[E - 1]);
    if (threadIdx.x == 0) sh_total_perm = total_perm;
    for (int d = threadIdx.x; d <= R; d += blockDim.x) {
        a.h.rank_base[d] = rbase[d];
        a.h.perm_rank_base[d] = d < R ? off[d * L] : total_perm;
    }
    // (d) per expert: offsets inside the rank, and the first permuted row of
    // every (source, expert) = the expert's first row + earlier sources' pairs
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int32_t o = off[e];
        a.h.expert_offsets[e] = o - off[(e / L) * L];
        int32_t acc = o;
        for (int s0 = 0; s0 < R; s0 += 16) {  // loads first: the stores may alias them
            int32_t c[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) c[u] = s0 + u < R ? a.ntpe[(int64_t)(s0 + u) * E + e] : 0;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                if (s0 + u >= R) break;
                a.ebase[(int64_t)(s0 + u) * E + e] = acc;
                acc += c[u];
            }
        }
    }
    // (e) hierarchical staging bases: home rank h of node n = h / G receives
    // from the sources s with s % G == h % G, in ascending s
    if (N > 1) {
        __syncthreads();
        for (int h = threadIdx.x; h < R; h += blockDim.x) {
            const int n = h / G;
            int32_t acc = 0;
            for (int s = h % G; s < R; s += G) acc += a.ntpn[s * N + n];
            hcnt[h] = acc;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int32_t acc = 0;
            for (int h = 0; h < R; ++h) {
                const int32_t c = hcnt[h];
                hcnt[h] = acc;
                acc += c;
            }
            hcnt[R] = acc;
            a.host[R + E + 2] = acc;
        }
        __syncthreads();
        for (int h = threadIdx.x; h <= R; h += blockDim.x) a.h.stage_base[h] = hcnt[h];
        for (int h = threadIdx.x; h < R; h += blockDim.x) {
            const int n = h / G;
            int32_t acc = hcnt[h];
            for (int s = h % G; s < R; s += G) {
                a.sbase[s * N + n] = acc;
                acc += a.ntpn[s * N + n];
            }
        }
    } else if (threadIdx.x == 0) {
        a.host[R + E + 2] = 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        a.host[R + E + 0] = sh_total_recv;
        a.host[R + E + 1] = sh_total_perm;
        a.host[R + E + 3] = (int32_t)atomicOr(a.status, 0u);
        __threadfence_system();
        // the host polls this word: it is written after every count above
        *reinterpret_cast<volatile int32_t*>(a.host + R + E + 4) = a.epoch;
        __threadfence_system();
    }
}

__global__ void __launch_bounds__(kTileTokens) notify_count_kernel(NotifyArgs a) {
    const int tiles = a.geom.tiles_per_src;
    extern __shared__ int32_t sh_cnt[];  // [max(E + R + N, 2E + 3R + 98)]
    if ((int)blockIdx.x == a.R * tiles) {
        notify_global_scan(a, sh_cnt);
        return;
    }
    const int s = blockIdx.x / tiles, tile = blockIdx.x % tiles;
    const int E = a.E, R = a.R, N = a.N, K = a.K, T = a.T;
    const int W = E + R + N;
    const int lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < W; i += blockDim.x) sh_cnt[i] = 0;
    __syncthreads();
    int lo, hi;
    tile_range(a.geom, tile, &lo, &hi);
    const int t = lo + threadIdx.x;
    const bool active = t < hi;
    // experts: entries of the tile, flattened, coalesced
    const int64_t* ent = a.topk_idx + ((int64_t)s * T + lo) * K;
    for (int i = threadIdx.x; i < (hi - lo) * K; i += blockDim.x) {
        const int64_t e = ent[i];
        if (e >= 0 && e < E) atomicAdd(&sh_cnt[e], 1);
    }
    // receivers and nodes: one ballot per bin and warp
    for (int d = 0; d < R; ++d) {
        const bool b = active && a.itir[((int64_t)s * T + t) * R + d];
        const uint32_t m = __ballot_sync(0xffffffffu, b);
        if (lane == 0 && m) atomicAdd(&sh_cnt[E + d], __popc(m));
    }
    for (int n = 0; n < N; ++n) {
        const bool b = active && a.itin[((int64_t)s * T + t) * N + n];
        const uint32_t m = __ballot_sync(0xffffffffu, b);
        if (lane == 0 && m) atomicAdd(&sh_cnt[E + R + n], __popc(m));
    }
    __syncthreads();
    int32_t* mine = a.part + ((int64_t)s * tiles + tile) * W;
    for (int i = threadIdx.x; i < W; i += blockDim.x) mine[i] = sh_cnt[i];
}

// ============================================================================
// Layout fused with notify pass 1
// ============================================================================
// grid = (tiles_per_src, R).  Each CTA is a layout tile whose per-tile counts
// (experts, receivers, nodes) are also notify's tile partials; the CTA that
// completes a source writes the source's histograms, and the CTA that
// completes the last source (a second completion counter) runs the global
// scans.  One launch instead of layout + notify pass 1, nothing waits.
__global__ void __launch_bounds__(kTileTokens) layout_notify_kernel(NotifyArgs a, int32_t* ntpe, int32_t* ntpr,
                                                                   uint8_t* itir, int32_t* ntpn, uint8_t* itin,
                                                                   uint32_t* done_src, uint32_t* done_all) {
    extern __shared__ int32_t sh_dyn[];
    __shared__ bool last_all;
    if (!layout_tile(a.topk_idx, a.R, a.E, a.K, a.T, a.L, a.N, a.G, a.geom, ntpe, ntpr, itir, ntpn, itin, a.part,
                     done_src, a.status, blockIdx.y, blockIdx.x))
        return;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();  // this source's sums before the count
        last_all = atomicAdd(done_all, 1u) == (uint32_t)(a.R - 1);
    }
    __syncthreads();
    if (!last_all) return;
    __threadfence();  // every source's sums are visible from here on
    notify_global_scan(a, sh_dyn);
    if (threadIdx.x == 0) *done_all = 0;  // re-arm for the next call (stream ordered)
}

// ============================================================================
// Notify, pass 2: per-token destination rows
// ============================================================================
// grid = (tiles_per_src, R), block = kTileTokens (8 warps, one token per thread).
//  send_pos[s][t][d]  = recv_offsets[d][s] + #{t' < t of s bound to d}
//  perm_pos[s][t][k]  = ebase[s][e] + #{(t', k') < (t, k) of s with expert e}
//  stage_pos[s][t][n] = sbase[s][n] + #{t' < t of s bound to node n}
//  channel_prefix_matrix[s][d][c] by the CTA holding channel c's last tile.
// Tile bases come from the partial counts of the tiles before this one; the
// rank inside the tile comes from warp ballots (receivers, nodes) and from
// __match_any_sync over 32 consecutive (t, k) entries (experts), walked in
// (t, k) order, so positions are a pure function of the input.
constexpr int kWarps = kTileTokens / 32;

__global__ void __launch_bounds__(kTileTokens) notify_position_kernel(NotifyArgs a) {
    extern __shared__ int32_t sh[];
    const int E = a.E, R = a.R, N = a.N, K = a.K, T = a.T;
    const int W = E + R + N;
    const int tiles = a.geom.tiles_per_src;
    const int s = blockIdx.y, tile = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* base = sh;                       // [W]   tile base per column
    int32_t* srcrel_d = base + W;             // [R]   source-relative prefix per receiver
    int32_t* wcnt = srcrel_d + R;             // [kWarps][E]  per-warp expert counters
    uint32_t* ball = reinterpret_cast<uint32_t*>(wcnt + kWarps * E);  // [kWarps][R + N]

    int lo, hi;
    tile_range(a.geom, tile, &lo, &hi);
    // 1. tile bases
    const int32_t* prev = a.part + (int64_t)s * tiles * W;
    for (int c = threadIdx.x; c < W; c += blockDim.x) {
        int32_t acc = 0;
        for (int j = 0; j < tile; ++j) acc += prev[(int64_t)j * W + c];
        if (c < E) {
            base[c] = a.ebase[(int64_t)s * E + c] + acc;
        } else if (c < E + R) {
            const int d = c - E;
            srcrel_d[d] = acc;
            base[c] = a.h.recv_offsets[d * R + s] + acc;
        } else {
            base[c] = a.sbase[s * N + (c - E - R)] + acc;
        }
    }
    for (int i = threadIdx.x; i < kWarps * E; i += blockDim.x) wcnt[i] = 0;
    __syncthreads();

    const int t = lo + threadIdx.x;
    const bool active = t < hi;
    // 2. receivers and nodes: ballots
    const uint8_t* in_rank = a.itir + ((int64_t)s * T + t) * R;
    for (int d = 0; d < R; ++d) {
        const uint32_t m = __ballot_sync(0xffffffffu, active && in_rank[d]);
        if (lane == 0) ball[warp * (R + N) + d] = m;
    }
    for (int n = 0; n < N; ++n) {
        const uint32_t m = __ballot_sync(0xffffffffu, active && a.itin[((int64_t)s * T + t) * N + n]);
        if (lane == 0) ball[warp * (R + N) + R + n] = m;
    }
    // 3. experts, pass 1: per-warp counts over the warp's 32 tokens
    const int wt0 = lo + warp * 32;                    // first token of this warp
    const int wtok = max(0, min(32, hi - wt0));        // tokens this warp holds
    const int64_t* went = a.topk_idx + ((int64_t)s * T + wt0) * K;
    for (int i = lane; i < wtok * K; i += 32) {
        const int64_t e = went[i];
        if (e >= 0 && e < E) atomicAdd(&wcnt[warp * E + e], 1);
    }
    __syncthreads();
    // exclusive scan over warps, per expert, seeded with the tile base
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int32_t run = base[e];
        for (int w = 0; w < kWarps; ++w) {
            const int32_t v = wcnt[w * E + e];
            wcnt[w * E + e] = run;
            run += v;
        }
    }
    __syncthreads();
    // 4. send_pos / stage_pos of this thread's token
    const uint32_t lt = lanemask_lt();
    if (active) {
        int32_t* sp = a.h.send_pos + ((int64_t)s * T + t) * R;
        for (int d = 0; d < R; ++d) {
            const uint32_t m = ball[warp * (R + N) + d];
            int32_t v = -1;
            if ((m >> lane) & 1) {
                int32_t acc = base[E + d];
                for (int w = 0; w < warp; ++w) acc += __popc(ball[w * (R + N) + d]);
                v = acc + __popc(m & lt);
            }
            sp[d] = v;
        }
        if (N > 1) {
            int32_t* stp = a.h.stage_pos + ((int64_t)s * T + t) * N;
            for (int n = 0; n < N; ++n) {
                const uint32_t m = ball[warp * (R + N) + R + n];
                int32_t v = -1;
                if ((m >> lane) & 1) {
                    int32_t acc = base[E + R + n];
                    for (int w = 0; w < warp; ++w) acc += __popc(ball[w * (R + N) + R + n]);
                    v = acc + __popc(m & lt);
                }
                stp[n] = v;
            }
        }
    }
    // 5. experts, pass 2: walk the warp's entries 32 at a time in (t, k) order
    int32_t* pp = a.h.perm_pos + ((int64_t)s * T + wt0) * K;
    const int nent = wtok * K;
    for (int c0 = 0; c0 < nent; c0 += 32) {
        const int i = c0 + lane;
        int64_t e64 = (i < nent) ? went[i] : -1;
        const int key = (e64 >= 0 && e64 < E) ? (int)e64 : -1;
        const uint32_t peers = __match_any_sync(0xffffffffu, key);
        int32_t pos = -1;
        if (key >= 0) pos = wcnt[warp * E + key] + __popc(peers & lt);
        __syncwarp();
        if (key >= 0 && lane == __ffs(peers) - 1) wcnt[warp * E + key] += __popc(peers);
        __syncwarp();
        if (i < nent) pp[i] = pos;
    }
    // 6. channel_prefix_matrix: the last tile of each channel writes it
    if (tile % a.geom.tiles_per_channel == a.geom.tiles_per_channel - 1) {
        const int c = tile / a.geom.tiles_per_channel;
        const int C = a.geom.C;
        for (int d = threadIdx.x; d < R; d += blockDim.x) {
            int32_t own = 0;
            for (int w = 0; w < kWarps; ++w) own += __popc(ball[w * (R + N) + d]);
            a.h.channel_prefix_matrix[((int64_t)s * R + d) * C + c] = srcrel_d[d] + own;
        }
    }
}

}  // namespace ep

using namespace ep;

// ============================================================================
// C ABI: context
// ============================================================================

extern "C" const char* ep_last_error(void) { return ep::g_last_error.c_str(); }

extern "C" const char* ep_status_name(int st) {
    switch (st) {
        case EP_OK: return "EP_OK";
        case EP_ERR_INVALID_ARG: return "EP_ERR_INVALID_ARG";
        case EP_ERR_INVALID_INPUT: return "EP_ERR_INVALID_INPUT";
        case EP_ERR_CAPACITY: return "EP_ERR_CAPACITY";
        case EP_ERR_TIMEOUT: return "EP_ERR_TIMEOUT";
        case EP_ERR_CUDA: return "EP_ERR_CUDA";
        default: return "EP_ERR_UNKNOWN";
    }
}

extern "C" const char* ep_version(void) { return "ep_gb300 0.1 (sm_103a)"; }

static ep_status validate_config(const ep_config* c) {
    if (!c) return set_error(EP_ERR_INVALID_ARG, "config is NULL");
    if (c->num_ranks < 1 || c->num_ranks > kMaxRanks)
        return set_error(EP_ERR_INVALID_ARG, "num_ranks %d outside [1, %d]", c->num_ranks, kMaxRanks);
    if (c->num_experts < 1 || c->num_experts > kMaxExperts || c->num_experts % c->num_ranks)
        return set_error(EP_ERR_INVALID_ARG, "num_experts %d must be a multiple of num_ranks and <= %d",
                         c->num_experts, kMaxExperts);
    if (c->num_experts / c->num_ranks > kMaxLocalExperts)
        return set_error(EP_ERR_INVALID_ARG, "more than %d experts per rank", kMaxLocalExperts);
    if (c->num_topk < 1 || c->num_topk > kMaxTopk)
        return set_error(EP_ERR_INVALID_ARG, "num_topk %d outside [1, %d]", c->num_topk, kMaxTopk);
    if (c->num_tokens < 0) return set_error(EP_ERR_INVALID_ARG, "num_tokens < 0");
    if (c->hidden < 8 || c->hidden % 8)
        return set_error(EP_ERR_INVALID_ARG, "hidden %d must be a positive multiple of 8", c->hidden);
    if (c->num_channels < 1 || c->num_channels > 1024)
        return set_error(EP_ERR_INVALID_ARG, "num_channels %d outside [1, 1024]", c->num_channels);
    if (c->num_nodes < 1 || c->num_nodes > c->num_ranks || c->num_ranks % c->num_nodes)
        return set_error(EP_ERR_INVALID_ARG, "num_nodes %d must divide num_ranks %d", c->num_nodes,
                         c->num_ranks);
    const int64_t R = c->num_ranks, T = c->num_tokens, K = c->num_topk;
    if (R * T * (K > R ? K : R) >= (1ll << 31) || R * T * c->num_nodes >= (1ll << 31))
        return set_error(EP_ERR_INVALID_ARG, "R*T*max(K,R) must stay below 2^31");
    return EP_OK;
}

static int env_int(const char* name, int dflt, int lo, int hi) {
    const char* v = getenv(name);
    if (!v || !*v) return dflt;
    int x = atoi(v);
    return x < lo ? lo : (x > hi ? hi : x);
}

static size_t notify_position_smem(const ep_ctx* c) {
    const int R = c->cfg.num_ranks, E = c->cfg.num_experts, N = c->cfg.num_nodes > 1 ? c->cfg.num_nodes : 0;
    return sizeof(int32_t) * (size_t)(E + R + N + R + kWarps * E + kWarps * (R + N));
}

extern "C" ep_status ep_ctx_create(const ep_config* cfg, ep_ctx** out) {
    if (!out) return set_error(EP_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    ep_status st = validate_config(cfg);
    if (st != EP_OK) return st;
    ep_ctx* c = new ep_ctx();  // value-initialised: every member starts at zero
    c->totals_known = true;      // nothing notified yet: zero rows, so a copy launched now does nothing
    c->expert_alignment = 1;
    c->cfg = *cfg;
    c->L = cfg->num_experts / cfg->num_ranks;
    c->G = cfg->num_ranks / cfg->num_nodes;
    c->tiles = make_tiles(cfg->num_tokens, cfg->num_channels);
    c->wait_timeout_ns = 2000000000ll;
    {
        // launch shape per copy route kind (measured on GB300): two CTAs per SM
        // with 64 KB of staging each, except the dispatch scatter, whose row
        // fans out to every destination rank: one CTA per SM with 160 KB
        // (skewed 803 -> 757 us, prefill unchanged; the permute and the
        // staging kernels are slower that way).  EP_COPY_CTAS_PER_SM and
        // EP_COPY_STAGE_KB set every kind, EP_<KIND>_CTAS_PER_SM and
        // EP_<KIND>_STAGE_KB one kind (PERMUTE, SCATTER, FUSED, STAGE).
        static const char* const kinds[4] = {"PERMUTE", "SCATTER", "FUSED", "STAGE"};
        static const int dflt_ctas[4] = {2, 1, 2, 2};
        static const int dflt_kb[4] = {64, 160, 64, 64};
        for (int k = 0; k < 4; ++k) {
            char n1[48], n2[48];
            snprintf(n1, sizeof n1, "EP_%s_CTAS_PER_SM", kinds[k]);
            snprintf(n2, sizeof n2, "EP_%s_STAGE_KB", kinds[k]);
            c->copy_ctas_per_sm[k] = env_int(n1, env_int("EP_COPY_CTAS_PER_SM", dflt_ctas[k], 1, 8), 1, 8);
            c->copy_stage_bytes[k] = env_int(n2, env_int("EP_COPY_STAGE_KB", dflt_kb[k], 16, 220), 16, 220) * 1024;
            c->copy_shape_forced[k] = getenv(n1) || getenv(n2) || getenv("EP_COPY_CTAS_PER_SM") ||
                                      getenv("EP_COPY_STAGE_KB");
        }
    }
    c->copy_read_depth = env_int("EP_COPY_READ_DEPTH", 2, 1, 3);
    cudaError_t e = cudaGetDevice(&c->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e != cudaSuccess) {
        delete c;
        return cuda_error(e, "cudaGetDevice");
    }
    const int R = cfg->num_ranks, E = cfg->num_experts, N = cfg->num_nodes;
    const int W = E + R + N;
    const size_t part = sizeof(int32_t) * (size_t)R * c->tiles.tiles_per_src * W;
    size_t off = 0;
    auto carve = [&](size_t bytes) {
        size_t o = off;
        off += (bytes + 255) & ~size_t(255);
        return o;
    };
    const size_t o_lp = carve(part), o_np = carve(part), o_eb = carve(sizeof(int32_t) * (size_t)R * E),
                 o_sb = carve(sizeof(int32_t) * (size_t)R * N), o_ld = carve(sizeof(uint32_t) * R),
                 o_nd = carve(sizeof(uint32_t)), o_st = carve(sizeof(uint32_t));
    c->ws_bytes = off;
    e = cudaMalloc(&c->ws, c->ws_bytes);
    if (e != cudaSuccess) {
        delete c;
        return cuda_error(e, "cudaMalloc(workspace)");
    }
    char* b = static_cast<char*>(c->ws);
    c->ws_layout_part = reinterpret_cast<int32_t*>(b + o_lp);
    c->ws_notify_part = reinterpret_cast<int32_t*>(b + o_np);
    c->ws_ebase = reinterpret_cast<int32_t*>(b + o_eb);
    c->ws_sbase = reinterpret_cast<int32_t*>(b + o_sb);
    c->ws_layout_done = reinterpret_cast<uint32_t*>(b + o_ld);
    c->ws_notify_done = reinterpret_cast<uint32_t*>(b + o_nd);
    c->status = reinterpret_cast<uint32_t*>(b + o_st);
    e = cudaMemset(c->ws, 0, c->ws_bytes);
    const size_t hb = sizeof(int32_t) * (size_t)(R + E + 8);
    if (e == cudaSuccess) e = cudaHostAlloc(reinterpret_cast<void**>(&c->host_block), hb, cudaHostAllocMapped);
    if (e == cudaSuccess) e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&c->host_block_dev), c->host_block, 0);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->ev_counts, cudaEventDisableTiming);
    const size_t smem = notify_position_smem(c);
    if (e == cudaSuccess && smem > 48 * 1024)
        e = cudaFuncSetAttribute(notify_position_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
        ep_ctx_destroy(c);
        return cuda_error(e, "ep_ctx_create");
    }
    std::memset(c->host_block, 0, hb);
    *out = c;
    return EP_OK;
}

extern "C" void ep_ctx_destroy(ep_ctx* c) {
    if (!c) return;
    if (c->ev_counts) cudaEventDestroy(c->ev_counts);
    if (c->host_block) cudaFreeHost(c->host_block);
    if (c->ws) cudaFree(c->ws);
    delete c;
}

extern "C" ep_status ep_ctx_check(ep_ctx* c, void* stream) {
    if (!c) return set_error(EP_ERR_INVALID_ARG, "ctx is NULL");
    uint32_t flags = 0;
    EP_CUDA(cudaStreamSynchronize(as_stream(stream)));
    EP_CUDA(cudaMemcpy(&flags, c->status, sizeof(flags), cudaMemcpyDeviceToHost));
    if (flags) EP_CUDA(cudaMemset(c->status, 0, sizeof(uint32_t)));
    return status_from_flags(flags);
}

extern "C" ep_status ep_ctx_set_wait_timeout_us(ep_ctx* c, int64_t us) {
    if (!c || us <= 0) return set_error(EP_ERR_INVALID_ARG, "bad context or timeout");
    c->wait_timeout_ns = us * 1000;
    return EP_OK;
}

extern "C" ep_status ep_ctx_set_expert_alignment(ep_ctx* c, int32_t alignment) {
    if (!c || alignment < 1 || alignment > (1 << 16)) return set_error(EP_ERR_INVALID_ARG, "bad context or alignment");
    // permuted rows (int32 positions) are at most R*T*K plus E*(alignment-1) of padding
    const ep_config& f = c->cfg;
    const int64_t worst = (int64_t)f.num_ranks * f.num_tokens * f.num_topk + (int64_t)f.num_experts * (alignment - 1);
    if (worst >= (1ll << 31))
        return set_error(EP_ERR_INVALID_ARG, "alignment %d: R*T*K + E*(alignment-1) = %lld must stay below 2^31",
                         alignment, (long long)worst);
    c->expert_alignment = alignment;
    return EP_OK;
}

extern "C" int32_t ep_ctx_expert_alignment(const ep_ctx* c) { return c ? c->expert_alignment : 0; }

extern "C" int32_t ep_ctx_last_launches(const ep_ctx* c) { return c ? c->last_launches : 0; }

// ============================================================================
// C ABI: layout and notify
// ============================================================================

extern "C" ep_status ep_get_dispatch_layout(ep_ctx* c, const int64_t* topk_idx, int32_t* ntpe,
                                            int32_t* ntpr, uint8_t* itir, int32_t* ntpn, uint8_t* itin,
                                            void* stream) {
    if (!c) return set_error(EP_ERR_INVALID_ARG, "ctx is NULL");
    c->last_launches = 0;
    const ep_config& f = c->cfg;
    // node outputs: num_tokens_per_node selects the hierarchical layout;
    // is_token_in_node may be NULL only when there are no tokens
    const bool nodes = ntpn != nullptr;
    if (!nodes && itin) return set_error(EP_ERR_INVALID_ARG, "is_token_in_node given without num_tokens_per_node");
    if (nodes && !itin && f.num_tokens > 0) return set_error(EP_ERR_INVALID_ARG, "is_token_in_node is NULL");
    if (!ntpe || !ntpr || (!itir && f.num_tokens > 0) || (!topk_idx && f.num_tokens > 0))
        return set_error(EP_ERR_INVALID_ARG, "NULL layout pointer");
    const int N = nodes ? f.num_nodes : 0;
    const int W = f.num_experts + f.num_ranks + N;
    dim3 grid(c->tiles.tiles_per_src, f.num_ranks);
    layout_kernel<<<grid, kTileTokens, sizeof(int32_t) * W, as_stream(stream)>>>(
        topk_idx, f.num_ranks, f.num_experts, f.num_topk, f.num_tokens, c->L, N, c->G, c->tiles, ntpe, ntpr,
        itir, ntpn, itin, c->ws_layout_part, c->ws_layout_done, c->status);
    EP_CHECK_LAUNCH("layout_kernel");
    c->last_launches = 1;
    return EP_OK;
}

// ============================================================================
// Allocation-free layout (see ep.h): the same layout kernel, with its scratch
// in a fixed device array of this library instead of a context's workspace.
// ============================================================================
namespace {
constexpr size_t kNoAllocScratchInts = EP_LAYOUT_NOALLOC_SCRATCH_BYTES / sizeof(int32_t);
constexpr size_t kNoAllocHeaderInts = 128;  // [0, 64) completion counters, [64] status
constexpr int kNoAllocMaxDevices = 64;
static __device__ __align__(256) int32_t g_noalloc_layout_scratch[kNoAllocScratchInts];
std::mutex g_noalloc_mu;
int32_t* g_noalloc_scratch_dev[kNoAllocMaxDevices];  // device address of the array, per device
}  // namespace

extern "C" ep_status ep_get_dispatch_layout_noalloc(int32_t R, int32_t E, int32_t K, int32_t T, int32_t num_nodes,
                                                    const int64_t* topk_idx, int32_t* ntpe, int32_t* ntpr,
                                                    uint8_t* itir, int32_t* ntpn, uint8_t* itin,
                                                    uint32_t* status_out, void* stream) {
    if (R < 1 || R > kMaxRanks || E < 1 || E > kMaxExperts || E % R || E / R > kMaxLocalExperts || K < 1 ||
        K > kMaxTopk || T < 0 || num_nodes < 1 || num_nodes > R || R % num_nodes)
        return set_error(EP_ERR_INVALID_ARG, "bad sizes (R %d, E %d, K %d, T %d, nodes %d)", R, E, K, T, num_nodes);
    if ((int64_t)R * T * (K > R ? K : R) >= (1ll << 31)) return set_error(EP_ERR_INVALID_ARG, "R*T*max(K,R) >= 2^31");
    const bool nodes = ntpn != nullptr;
    if (!nodes && itin) return set_error(EP_ERR_INVALID_ARG, "is_token_in_node given without num_tokens_per_node");
    if (!ntpe || !ntpr || (T > 0 && (!itir || !topk_idx || (nodes && !itin))))
        return set_error(EP_ERR_INVALID_ARG, "NULL layout pointer");
    const int N = nodes ? num_nodes : 0;
    const TileGeom geom = make_tiles(T, 1);
    const int W = E + R + N;
    const size_t need = kNoAllocHeaderInts + (size_t)R * geom.tiles_per_src * W;
    if (need > kNoAllocScratchInts)
        return set_error(EP_ERR_CAPACITY,
                         "the allocation-free layout needs %zu bytes of scratch, it has %u; use ep_get_dispatch_layout",
                         need * sizeof(int32_t), (unsigned)EP_LAYOUT_NOALLOC_SCRATCH_BYTES);
    int dev = 0;
    EP_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kNoAllocMaxDevices) return set_error(EP_ERR_INVALID_ARG, "device index %d not supported", dev);
    int32_t* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_scratch_dev[dev]) {
            void* p = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_layout_scratch);
            if (e != cudaSuccess) return cuda_error(e, "cudaGetSymbolAddress(layout scratch)");
            g_noalloc_scratch_dev[dev] = static_cast<int32_t*>(p);
        }
        scratch = g_noalloc_scratch_dev[dev];
    }
    cudaStream_t s = as_stream(stream);
    // completion counters and the status word must start at zero
    EP_CUDA(cudaMemsetAsync(scratch, 0, kNoAllocHeaderInts * sizeof(int32_t), s));
    uint32_t* done = reinterpret_cast<uint32_t*>(scratch);
    uint32_t* status = status_out ? status_out : reinterpret_cast<uint32_t*>(scratch + 64);
    dim3 grid(geom.tiles_per_src, R);
    layout_kernel<<<grid, kTileTokens, sizeof(int32_t) * W, s>>>(topk_idx, R, E, K, T, E / R, N, R / num_nodes, geom,
                                                                 ntpe, ntpr, itir, ntpn, itin,
                                                                 scratch + kNoAllocHeaderInts, done, status);
    EP_CHECK_LAUNCH("layout_kernel (allocation-free)");
    return EP_OK;
}

// Notify (and, with `fused`, the layout in the same launch as notify's first
// pass: the layout pointers are then outputs).
static ep_status notify_impl(ep_ctx* c, const int64_t* topk_idx, int32_t* ntpe, int32_t* ntpr, uint8_t* itir,
                             int32_t* ntpn, uint8_t* itin, const ep_dispatch_handle* h, int32_t* host_num_recv,
                             int32_t* host_num_recv_per_expert, int32_t* host_totals, void* stream, bool fused) {
    if (!c || !h) return set_error(EP_ERR_INVALID_ARG, "ctx or handle is NULL");
    c->last_launches = 0;
    const ep_config& f = c->cfg;
    const bool hier = f.num_nodes > 1;
    if (!ntpe || !ntpr || (f.num_tokens > 0 && (!itir || !topk_idx)))
        return set_error(EP_ERR_INVALID_ARG, "NULL notify input");
    const bool wait = host_num_recv != nullptr;
    if (!wait && (host_num_recv_per_expert || host_totals))
        return set_error(EP_ERR_INVALID_ARG, "host count arrays need host_num_recv_tokens (the waiting form)");
    if (hier && (!ntpn || !h->stage_base || (f.num_tokens > 0 && (!itin || !h->stage_pos))))
        return set_error(EP_ERR_INVALID_ARG, "hierarchical mode needs node layout and stage_* handle arrays");
    if (!h->recv_count || !h->recv_offsets || !h->num_recv_tokens || !h->rank_base || !h->num_recv_per_expert ||
        !h->expert_offsets || !h->perm_rank_base || !h->channel_prefix_matrix ||
        (f.num_tokens > 0 && (!h->send_pos || !h->perm_pos)))
        return set_error(EP_ERR_INVALID_ARG, "NULL handle array");
    NotifyArgs a;
    a.topk_idx = topk_idx;
    a.ntpe = ntpe;
    a.ntpr = ntpr;
    a.itir = itir;
    a.ntpn = hier ? ntpn : nullptr;
    a.itin = hier ? itin : nullptr;
    a.h = *h;
    a.R = f.num_ranks;
    a.E = f.num_experts;
    a.K = f.num_topk;
    a.T = f.num_tokens;
    a.L = c->L;
    a.N = hier ? f.num_nodes : 0;
    a.G = c->G;
    a.align = c->expert_alignment;
    a.geom = c->tiles;
    a.part = c->ws_notify_part;
    a.ebase = c->ws_ebase;
    a.sbase = c->ws_sbase;
    a.host = c->host_block_dev;
    a.status = c->status;
    a.epoch = ++c->notify_epoch;
    const int W = a.E + a.R + a.N;
    cudaStream_t s = as_stream(stream);
    const int Wscan = 2 * a.E + 3 * a.R + 98;
    const size_t scan_smem = sizeof(int32_t) * (W > Wscan ? W : Wscan);
    if (fused) {
        dim3 lgrid(c->tiles.tiles_per_src, a.R);
        layout_notify_kernel<<<lgrid, kTileTokens, scan_smem, s>>>(a, ntpe, ntpr, itir, hier ? ntpn : nullptr,
                                                                   hier ? itin : nullptr, c->ws_layout_done,
                                                                   c->ws_notify_done);
        EP_CHECK_LAUNCH("layout_notify_kernel");
    } else {
        const int nblk = a.R * c->tiles.tiles_per_src + 1;
        notify_count_kernel<<<nblk, kTileTokens, scan_smem, s>>>(a);
        EP_CHECK_LAUNCH("notify_count_kernel");
    }
    if (wait) EP_CUDA(cudaEventRecord(c->ev_counts, s));
    dim3 grid(c->tiles.tiles_per_src, a.R);
    notify_position_kernel<<<grid, kTileTokens, notify_position_smem(c), s>>>(a);
    EP_CHECK_LAUNCH("notify_position_kernel");
    c->last_launches = 2;
    if (!wait) {
        // no host synchronisation: later calls size their grids from their
        // capacity arguments and read the row counts from the handle on the device
        c->totals_known = false;
        return EP_OK;
    }
    // the one host synchronisation of the normal path: the receive counts.
    // Poll the CPU-mapped sequence word the count kernel writes last (cheaper
    // than an event wake-up); the event bounds the poll and reports errors.
    volatile int32_t* hb = c->host_block;
    const int R = a.R, E = a.E;
    {
        const auto t0 = std::chrono::steady_clock::now();
        unsigned spins = 0;
        while (hb[R + E + 4] != a.epoch) {
            if ((++spins & 1023u) == 0) {
                const cudaError_t q = cudaEventQuery(c->ev_counts);
                if (q == cudaSuccess) {
                    if (hb[R + E + 4] != a.epoch) return set_error(EP_ERR_CUDA, "notify counts were not published");
                    break;
                }
                if (q != cudaErrorNotReady) return cuda_error(q, "notify_count_kernel");
                if (std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(2)) {
                    EP_CUDA(cudaEventSynchronize(c->ev_counts));  // long wait: block instead of spinning
                    if (hb[R + E + 4] != a.epoch) return set_error(EP_ERR_CUDA, "notify counts were not published");
                    break;
                }
            }
        }
    }
    for (int d = 0; d < R; ++d) host_num_recv[d] = hb[d];
    if (host_num_recv_per_expert)
        for (int e = 0; e < E; ++e) host_num_recv_per_expert[e] = hb[R + e];
    c->last_total_recv = hb[R + E + 0];
    c->last_total_perm = hb[R + E + 1];
    c->last_total_stage = hb[R + E + 2];
    c->totals_known = true;
    if (host_totals) {
        host_totals[0] = (int32_t)c->last_total_recv;
        host_totals[1] = (int32_t)c->last_total_perm;
        host_totals[2] = (int32_t)c->last_total_stage;
    }
    const uint32_t flags = (uint32_t)hb[R + E + 3];
    if (flags & FLAG_INVALID_TOPK) return status_from_flags(flags);
    return EP_OK;
}

extern "C" ep_status ep_notify_dispatch(ep_ctx* c, const int64_t* topk_idx, const int32_t* ntpe,
                                        const int32_t* ntpr, const uint8_t* itir, const int32_t* ntpn,
                                        const uint8_t* itin, const ep_dispatch_handle* h,
                                        int32_t* host_num_recv, int32_t* host_num_recv_per_expert,
                                        int32_t* host_totals, void* stream) {
    // the layout arrays are only read on this path
    return notify_impl(c, topk_idx, const_cast<int32_t*>(ntpe), const_cast<int32_t*>(ntpr),
                       const_cast<uint8_t*>(itir), const_cast<int32_t*>(ntpn), const_cast<uint8_t*>(itin), h,
                       host_num_recv, host_num_recv_per_expert, host_totals, stream, false);
}

extern "C" ep_status ep_layout_notify(ep_ctx* c, const int64_t* topk_idx, int32_t* ntpe, int32_t* ntpr,
                                      uint8_t* itir, int32_t* ntpn, uint8_t* itin, const ep_dispatch_handle* h,
                                      int32_t* host_num_recv, int32_t* host_num_recv_per_expert,
                                      int32_t* host_totals, void* stream) {
    if (c && c->cfg.num_nodes > 1 && c->cfg.num_tokens > 0 && (!ntpn || !itin))
        return set_error(EP_ERR_INVALID_ARG, "hierarchical mode needs the node layout outputs");
    if (c && c->cfg.num_nodes == 1 && (ntpn || itin))
        return set_error(EP_ERR_INVALID_ARG, "node layout outputs need num_nodes > 1");
    return notify_impl(c, topk_idx, ntpe, ntpr, itir, ntpn, itin, h, host_num_recv, host_num_recv_per_expert,
                       host_totals, stream, true);
}
