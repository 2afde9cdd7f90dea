// ep_ll.cu -- low-latency mode ("send without asking").
//
// Page "事件驱动 EP 内核的调度策略与零拷贝通信", section "低延迟模式": every receiver
// keeps a private region per (source rank, expert); the sender computes the
// address base + (expert*num_ranks + src_rank)*chunk + slot itself, writes
// the data, then writes the real count into the region's count slot, whose
// initial value is an empty sentinel; dispatch data is FP8, combine BF16.
// Page "DeepEP 学习笔记": two buffers used in turn (XOR flip), no allocation and
// no CPU synchronisation per call; counters start at -1.
// Page "DeepSeek DeepEP探索：低延迟分发", sections 2.2 (worst-case buffer size
// hint) and 4.2 (receiver: acquire-load the count of (local expert, source),
// then copy to the contiguous per-expert tensor using per-expert begin
// indices).
//
// GB300 design on one GPU: the R ranks' regions are one allocation; the send
// kernel quantises each token once (per-128-channel amax, IEEE division,
// cvt.rn.satfinite.e4m3x2) and stores the message to its K regions; slots are
// the deterministic (t, k)-order rank of the entry among the source's entries
// for the same expert (no atomic slot claims); the last CTA of a source
// (completion counter) publishes all counts of that source with st.release
// after the data, 0 included.  The receive kernel polls each count with
// ld.acquire under a time limit and packs the messages.
#include <cuda_fp8.h>

#include "ep_internal.cuh"
#include "ep_combine.cuh"

struct ep_ll_buffer {
    ep_config cfg;
    int cap, L, device, num_sms;
    int64_t msg_bytes;
    void* mem;
    size_t bytes;
    uint8_t* regions[2];
    int32_t* counts[2];
    uint32_t* done[2];
    uint32_t* status;
    int cur;
    int64_t wait_timeout_ns;
};

namespace ep {

constexpr int kSendThreads = 1024;
constexpr int kRecvThreads = 128;

struct LLSendArgs {
    const uint16_t* x;  // bf16 bits [R][T][H]
    const int64_t* topk_idx;
    int32_t* slot_out;
    uint8_t* regions;
    int32_t* counts;       // [E][R] of the buffer in use
    uint32_t* done;        // [R]
    int32_t* other_counts; // [E][R] of the other buffer
    int R, E, K, T, H, cap, t0, n, nblk;
    int64_t msg_bytes;
    uint32_t* status;
};

__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    // low byte <- a, high byte <- b
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// grid = (n tokens, R sources), one CTA per token.  All loads of the CTA (its
// own top-k entries, the source's earlier entries of the microbatch, the x row)
// are issued before the first barrier; the slots come from shared-memory
// counts; the token is quantised once and stored to its K regions.  No fence
// or atomic on global memory: the counts are published by ll_publish_kernel.
constexpr int kPriorPerThread = 8;

__global__ void __launch_bounds__(1024) ll_send_kernel(LLSendArgs a) {
    __shared__ int sh_e[kMaxTopk];
    __shared__ int sh_cnt[kMaxTopk];
    __shared__ int sh_slot[kMaxTopk];
    const int s = blockIdx.y, j = blockIdx.x;  // j-th token of the microbatch
    const int K = a.K, R = a.R, E = a.E, H = a.H;
    // let the publish kernel start its own (independent) work early
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int t = a.t0 + j;
    const int64_t g = (int64_t)s * a.T + t;
    const int64_t* first = a.topk_idx + ((int64_t)s * a.T + a.t0) * K;
    const int prior = j * K;
    // ---- loads ---------------------------------------------------------------------
    if (threadIdx.x < K) {
        const int64_t e = a.topk_idx[g * K + threadIdx.x];
        int ev = -1;
        if (e >= 0 && e < E) ev = (int)e;
        else if (e != -1) flag(a.status, FLAG_INVALID_TOPK);
        sh_e[threadIdx.x] = ev;
        sh_cnt[threadIdx.x] = 0;
    }
    int pe[kPriorPerThread];
#pragma unroll
    for (int u = 0; u < kPriorPerThread; ++u) {
        const int i = threadIdx.x + u * blockDim.x;
        const int64_t e = i < prior ? first[i] : -1;
        pe[u] = (e >= 0 && e < E) ? (int)e : -1;
    }
    const int ngroups = H / 16;  // 16 channels per thread per pass; 8 groups per scale block
    const uint16_t* xr = a.x + g * H;
    int4 p0 = make_int4(0, 0, 0, 0), p1 = make_int4(0, 0, 0, 0);
    if ((int)threadIdx.x < ngroups) {
        p0 = ld_nc_na_v4(xr + threadIdx.x * 16);
        p1 = ld_nc_na_v4(xr + threadIdx.x * 16 + 8);
    }
    __syncthreads();
    // ---- slots: earlier entries of this source with the same expert ----------------
#pragma unroll
    for (int u = 0; u < kPriorPerThread; ++u)
        if (pe[u] >= 0)
            for (int k = 0; k < K; ++k)
                if (sh_e[k] == pe[u]) atomicAdd(&sh_cnt[k], 1);
    for (int i = threadIdx.x + kPriorPerThread * blockDim.x; i < prior; i += blockDim.x) {
        const int64_t e = first[i];
        if (e < 0 || e >= E) continue;
        for (int k = 0; k < K; ++k)
            if (sh_e[k] == (int)e) atomicAdd(&sh_cnt[k], 1);
    }
    __syncthreads();
    if (threadIdx.x < K) {
        const int k = threadIdx.x;
        const int ev = sh_e[k];
        int sl = -1;
        if (ev >= 0) {
            sl = sh_cnt[k];
            for (int k2 = 0; k2 < k; ++k2) sl += (sh_e[k2] == ev);
            if (sl >= a.cap) {
                flag(a.status, FLAG_CAPACITY);
                sl = -1;
            }
        }
        sh_slot[k] = sl;
        a.slot_out[g * K + k] = sl;
        if (sl >= 0) {
            uint8_t* msg = a.regions + (((int64_t)ev * R + s) * a.cap + sl) * a.msg_bytes;
            *reinterpret_cast<int4*>(msg) = make_int4(t, 0, 0, 0);
        }
    }
    __syncthreads();
    // ---- quantise once, store to every destination region ----------------------
    for (int gi0 = 0; gi0 < ngroups; gi0 += blockDim.x) {
        const int gi = gi0 + threadIdx.x;
        const bool act = gi < ngroups;
        if (gi0 > 0 && act) {  // later passes (H > 16 * blockDim)
            p0 = ld_nc_na_v4(xr + gi * 16);
            p1 = ld_nc_na_v4(xr + gi * 16 + 8);
        }
        float v[16];
        const uint32_t uu[8] = {(uint32_t)p0.x, (uint32_t)p0.y, (uint32_t)p0.z, (uint32_t)p0.w,
                                (uint32_t)p1.x, (uint32_t)p1.y, (uint32_t)p1.z, (uint32_t)p1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = __uint_as_float(uu[i] << 16);
            v[2 * i + 1] = __uint_as_float(uu[i] & 0xffff0000u);
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
        // max over the 8 lanes holding one 128-channel block
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float scale = __fdiv_rn(amax, 448.0f);
        uint32_t w4[4];
        if (scale == 0.0f) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t c = 0;
#pragma unroll
                for (int b = 0; b < 4; ++b) c |= ((__float_as_uint(v[4 * i + b]) >> 31) ? 0x80u : 0u) << (8 * b);
                w4[i] = c;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t lo = e4m3x2(__fdiv_rn(v[4 * i], scale), __fdiv_rn(v[4 * i + 1], scale));
                const uint32_t hi = e4m3x2(__fdiv_rn(v[4 * i + 2], scale), __fdiv_rn(v[4 * i + 3], scale));
                w4[i] = (lo & 0xffffu) | (hi << 16);
            }
        }
        if (act) {
            const int4 codes = make_int4((int)w4[0], (int)w4[1], (int)w4[2], (int)w4[3]);
            for (int k = 0; k < K; ++k) {
                const int sl = sh_slot[k];
                if (sl < 0) continue;
                uint8_t* msg = a.regions + (((int64_t)sh_e[k] * R + s) * a.cap + sl) * a.msg_bytes;
                st_na_v4(msg + 16 + (int64_t)gi * 16, codes);
                if ((gi & 7) == 0) *reinterpret_cast<float*>(msg + 16 + H + (gi >> 3) * 4) = scale;
            }
        }
    }
}

// grid = R sources (launched as a programmatic dependent of ll_send_kernel).
// Counts the source's entries per expert while the send runs, then waits for
// the send grid to complete (griddepcontrol.wait: its writes are visible) and
// publishes every count slot of the source, 0 included, with release stores.
// Also re-arms the other ping-pong buffer's count slots of this source.
__global__ void __launch_bounds__(256) ll_publish_kernel(LLSendArgs a) {
    extern __shared__ int32_t sh_hist[];  // [E]
    const int s = blockIdx.x;
    const int E = a.E, R = a.R, K = a.K;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        sh_hist[e] = 0;
        st_relaxed_gpu(a.other_counts + (int64_t)e * R + s, -1);
    }
    __syncthreads();
    const int64_t* first = a.topk_idx + ((int64_t)s * a.T + a.t0) * K;
    for (int i = threadIdx.x; i < a.n * K; i += blockDim.x) {
        const int64_t e = first[i];
        if (e >= 0 && e < E) atomicAdd(&sh_hist[e], 1);
    }
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int c = sh_hist[e];
        st_release_gpu(a.counts + (int64_t)e * R + s, c < a.cap ? c : a.cap);
    }
}

struct LLRecvArgs {
    const uint8_t* regions;
    const int32_t* counts;
    uint8_t* packed_x;
    float* packed_scales;
    int32_t* packed_src_info;
    int32_t* packed_recv_count;
    int32_t* layout_range;
    int R, E, L, H, cap;
    int64_t msg_bytes;
    int64_t timeout_ns;
    uint32_t* status;
};

// Bounded poll of one count slot: the sentinel -1 means "not written yet".
__device__ int wait_count(const int32_t* p, int64_t limit_ns, uint32_t* status) {
    int v = ld_acquire_gpu(p);
    if (v >= 0) return v;
    const uint64_t t0 = globaltimer_ns();
    unsigned ns = 32;
    while (true) {
        __nanosleep(ns);
        if (ns < 1024) ns <<= 1;
        v = ld_acquire_gpu(p);
        if (v >= 0) return v;
        if ((int64_t)(globaltimer_ns() - t0) > limit_ns) {
            flag(status, FLAG_TIMEOUT);
            return 0;
        }
    }
}


// grid = (R sources, E experts): CTA (s, e) waits for the counts of sources
// 0..s of expert e (begin = exclusive prefix), then copies its messages.
__global__ void __launch_bounds__(kRecvThreads) ll_recv_kernel(LLRecvArgs a) {
    __shared__ int sh_begin, sh_count;
    const int s = blockIdx.x, e = blockIdx.y;
    // launched as a programmatic dependent of the count publisher: start once
    // its grid (and every write before it) is complete
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int R = a.R, L = a.L, H = a.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        int before = 0, mine = 0;
        for (int s2 = lane; s2 <= s; s2 += 32) {
            const int v = wait_count(a.counts + (int64_t)e * R + s2, a.timeout_ns, a.status);
            if (s2 < s) before += v;
            else mine = v;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            before += __shfl_xor_sync(0xffffffffu, before, o);
            mine += __shfl_xor_sync(0xffffffffu, mine, o);
        }
        if (lane == 0) {
            if (mine > a.cap) {
                flag(a.status, FLAG_CAPACITY);
                mine = a.cap;
            }
            sh_begin = before;
            sh_count = mine;
        }
    }
    __syncthreads();
    const int begin = sh_begin, count = sh_count;
    const int d = e / L, l = e % L;
    if (threadIdx.x == 0) {
        int32_t* lr = a.layout_range + (((int64_t)d * L + l) * R + s) * 2;
        lr[0] = begin;
        lr[1] = count;
        if (s == R - 1) a.packed_recv_count[(int64_t)d * L + l] = begin + count;
    }
    const int S = H / 128;
    const int64_t rows_per_expert = (int64_t)R * a.cap;
    const int nwarps = blockDim.x / 32;
    const int nv = H / 16;
    for (int i = warp; i < count; i += nwarps) {
        const uint8_t* msg = a.regions + (((int64_t)e * R + s) * a.cap + i) * a.msg_bytes;
        const int64_t p = ((int64_t)d * L + l) * rows_per_expert + begin + i;
        const int4* src = reinterpret_cast<const int4*>(msg + 16);
        int4* dx = reinterpret_cast<int4*>(a.packed_x + p * H);
        // issue a batch of loads before the stores that consume them
        for (int v0 = 0; v0 < nv; v0 += 8 * 32) {
            int4 buf[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < nv) buf[u] = __ldcg(src + v);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < nv) __stcs(dx + v, buf[u]);
            }
        }
        const float* sc = reinterpret_cast<const float*>(msg + 16 + H);
        for (int v = lane; v < S; v += 32) __stcs(a.packed_scales + p * S + v, __ldcg(sc + v));
        if (lane == 0) {
            a.packed_src_info[p * 2] = s;
            a.packed_src_info[p * 2 + 1] = __ldcg(reinterpret_cast<const int32_t*>(msg));
        }
    }
}

}  // namespace ep

using namespace ep;

extern "C" int64_t ep_ll_message_bytes(int hidden) {
    if (hidden <= 0) return 0;
    const int64_t b = 16 + (int64_t)hidden + (int64_t)(hidden / 128) * 4;
    return (b + 15) / 16 * 16;
}

static int64_t ll_one_buffer_bytes(int cap, int H, int R, int E) {
    const int64_t counts = ((int64_t)E * R * 4 + 15) / 16 * 16;
    const int64_t done = ((int64_t)R * 4 + 15) / 16 * 16;
    int64_t one = (int64_t)E * R * cap * ep_ll_message_bytes(H) + counts + done;
    return (one + 127) / 128 * 128;
}

extern "C" int64_t ep_ll_size_hint(int cap, int hidden, int num_ranks, int num_experts) {
    if (cap <= 0 || hidden <= 0 || num_ranks <= 0 || num_experts <= 0) return 0;
    return 2 * ll_one_buffer_bytes(cap, hidden, num_ranks, num_experts);
}

extern "C" ep_status ep_ll_buffer_create(const ep_config* cfg, int cap, ep_ll_buffer** out) {
    if (!out || !cfg) return set_error(EP_ERR_INVALID_ARG, "NULL argument");
    *out = nullptr;
    const int R = cfg->num_ranks, E = cfg->num_experts, H = cfg->hidden, K = cfg->num_topk;
    if (R < 1 || R > kMaxRanks || E < 1 || E > kMaxExperts || E % R || K < 1 || K > kMaxTopk || cfg->num_tokens < 0)
        return set_error(EP_ERR_INVALID_ARG, "bad low-latency configuration (R %d, E %d, K %d)", R, E, K);
    if (H < 128 || H % 128) return set_error(EP_ERR_INVALID_ARG, "hidden %d must be a positive multiple of 128", H);
    if (cap < 1 || cap > 4096) return set_error(EP_ERR_INVALID_ARG, "cap %d outside [1, 4096]", cap);
    ep_ll_buffer* b = new ep_ll_buffer();
    b->cfg = *cfg;
    b->cap = cap;
    b->L = E / R;
    b->msg_bytes = ep_ll_message_bytes(H);
    b->cur = 1;  // the first send flips to buffer 0
    b->wait_timeout_ns = 100000000ll;
    cudaError_t e = cudaGetDevice(&b->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&b->num_sms, cudaDevAttrMultiProcessorCount, b->device);
    const int64_t one = ll_one_buffer_bytes(cap, H, R, E);
    b->bytes = (size_t)(2 * one + 256);
    if (e == cudaSuccess) e = cudaMalloc(&b->mem, b->bytes);
    if (e != cudaSuccess) {
        delete b;
        return cuda_error(e, "ep_ll_buffer_create");
    }
    uint8_t* base = static_cast<uint8_t*>(b->mem);
    const int64_t reg = (int64_t)E * R * cap * b->msg_bytes;
    const int64_t counts = ((int64_t)E * R * 4 + 15) / 16 * 16;
    for (int i = 0; i < 2; ++i) {
        uint8_t* p = base + i * one;
        b->regions[i] = p;
        b->counts[i] = reinterpret_cast<int32_t*>(p + reg);
        b->done[i] = reinterpret_cast<uint32_t*>(p + reg + counts);
    }
    b->status = reinterpret_cast<uint32_t*>(base + 2 * one);
    // counts start at the empty sentinel; completion counters and status at 0
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
        e = cudaMemset(b->counts[i], 0xff, (size_t)E * R * 4);
        if (e == cudaSuccess) e = cudaMemset(b->done[i], 0, (size_t)R * 4);
    }
    if (e == cudaSuccess) e = cudaMemset(b->status, 0, 4);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        ep_ll_buffer_destroy(b);
        return cuda_error(e, "ep_ll_buffer_create");
    }
    *out = b;
    return EP_OK;
}

extern "C" void ep_ll_buffer_destroy(ep_ll_buffer* b) {
    if (!b) return;
    if (b->mem) cudaFree(b->mem);
    delete b;
}

extern "C" ep_status ep_ll_set_wait_timeout_us(ep_ll_buffer* b, int64_t us) {
    if (!b || us <= 0) return set_error(EP_ERR_INVALID_ARG, "bad buffer or timeout");
    b->wait_timeout_ns = us * 1000;
    return EP_OK;
}

extern "C" ep_status ep_ll_check(ep_ll_buffer* b, void* stream) {
    if (!b) return set_error(EP_ERR_INVALID_ARG, "buffer is NULL");
    uint32_t flags = 0;
    EP_CUDA(cudaStreamSynchronize(as_stream(stream)));
    EP_CUDA(cudaMemcpy(&flags, b->status, 4, cudaMemcpyDeviceToHost));
    if (flags) EP_CUDA(cudaMemset(b->status, 0, 4));
    return status_from_flags(flags);
}

extern "C" int32_t* ep_ll_count_slots(ep_ll_buffer* b, int which) {
    if (!b || which < 0 || which > 1) return nullptr;
    return b->counts[which];
}

extern "C" int ep_ll_current_buffer(const ep_ll_buffer* b) { return b ? b->cur : -1; }

extern "C" ep_status ep_ll_send(ep_ll_buffer* b, const void* x, const int64_t* topk_idx, int t0, int n,
                                int32_t* slot_out, void* stream) {
    if (!b) return set_error(EP_ERR_INVALID_ARG, "buffer is NULL");
    const ep_config& f = b->cfg;
    if (t0 < 0 || n < 0 || t0 + n > f.num_tokens) return set_error(EP_ERR_INVALID_ARG, "tokens [%d, %d) outside [0, %d)", t0, t0 + n, f.num_tokens);
    if (n > b->cap) return set_error(EP_ERR_CAPACITY, "microbatch of %d tokens exceeds the region cap %d", n, b->cap);
    if (n > 0 && (!x || !aligned16(x) || !topk_idx || !slot_out))
        return set_error(EP_ERR_INVALID_ARG, "x (16-byte aligned), topk_idx and slot_out are required");
    b->cur ^= 1;
    LLSendArgs a;
    a.x = static_cast<const uint16_t*>(x);
    a.topk_idx = topk_idx;
    a.slot_out = slot_out;
    a.regions = b->regions[b->cur];
    a.counts = b->counts[b->cur];
    a.done = b->done[b->cur];
    a.other_counts = b->counts[b->cur ^ 1];
    a.R = f.num_ranks;
    a.E = f.num_experts;
    a.K = f.num_topk;
    a.T = f.num_tokens;
    a.H = f.hidden;
    a.cap = b->cap;
    a.t0 = t0;
    a.n = n;
    a.nblk = n;
    a.msg_bytes = b->msg_bytes;
    a.status = b->status;
    cudaStream_t s = as_stream(stream);
    if (n > 0) {
        // one thread per 16 channels (one pass) up to 1024 threads, whole warps
        int threads = ((a.H / 16 + 31) / 32) * 32;
        if (threads < 64) threads = 64;
        if (threads > kSendThreads) threads = kSendThreads;
        ll_send_kernel<<<dim3(n, a.R), threads, 0, s>>>(a);
        EP_CHECK_LAUNCH("ll_send_kernel");
    }
    // counts after the data: a programmatic dependent launch overlaps the
    // publisher's histogram with the send; its griddepcontrol.wait orders the
    // count stores after every data store of the send grid
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(a.R);
    lc.blockDim = dim3(256);
    lc.dynamicSmemBytes = sizeof(int32_t) * (size_t)a.E;
    lc.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    EP_CUDA(cudaLaunchKernelEx(&lc, ll_publish_kernel, a));
    return EP_OK;
}

extern "C" ep_status ep_ll_recv(ep_ll_buffer* b, uint8_t* packed_x, float* packed_scales, int32_t* packed_src_info,
                                int32_t* packed_recv_count, int32_t* layout_range, void* stream) {
    if (!b) return set_error(EP_ERR_INVALID_ARG, "buffer is NULL");
    if (!packed_x || !aligned16(packed_x) || !packed_scales || !packed_src_info || !packed_recv_count || !layout_range)
        return set_error(EP_ERR_INVALID_ARG, "NULL or misaligned receive output");
    const ep_config& f = b->cfg;
    LLRecvArgs a;
    a.regions = b->regions[b->cur];
    a.counts = b->counts[b->cur];
    a.packed_x = packed_x;
    a.packed_scales = packed_scales;
    a.packed_src_info = packed_src_info;
    a.packed_recv_count = packed_recv_count;
    a.layout_range = layout_range;
    a.R = f.num_ranks;
    a.E = f.num_experts;
    a.L = b->L;
    a.H = f.hidden;
    a.cap = b->cap;
    a.msg_bytes = b->msg_bytes;
    a.timeout_ns = b->wait_timeout_ns;
    a.status = b->status;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(a.R, a.E);
    lc.blockDim = dim3(kRecvThreads);
    lc.dynamicSmemBytes = 0;
    lc.stream = as_stream(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    EP_CUDA(cudaLaunchKernelEx(&lc, ll_recv_kernel, a));
    return EP_OK;
}

extern "C" ep_status ep_ll_dispatch(ep_ll_buffer* b, const void* x, const int64_t* topk_idx, int t0, int n,
                                    uint8_t* packed_x, float* packed_scales, int32_t* packed_src_info,
                                    int32_t* packed_recv_count, int32_t* layout_range, int32_t* slot_out, void* stream) {
    ep_status st = ep_ll_send(b, x, topk_idx, t0, n, slot_out, stream);
    if (st != EP_OK) return st;
    return ep_ll_recv(b, packed_x, packed_scales, packed_src_info, packed_recv_count, layout_range, stream);
}

extern "C" ep_status ep_ll_combine(ep_ll_buffer* b, const void* y_ll, const int64_t* topk_idx, const float* topk_weights,
                                   const int32_t* slot, const int32_t* layout_range, int t0, int n, void* out,
                                   void* stream) {
    if (!b) return set_error(EP_ERR_INVALID_ARG, "buffer is NULL");
    const ep_config& f = b->cfg;
    if (t0 < 0 || n < 0 || t0 + n > f.num_tokens) return set_error(EP_ERR_INVALID_ARG, "token range outside [0, T)");
    if (n == 0) return EP_OK;
    if (!y_ll || !aligned16(y_ll) || !out || !aligned16(out) || !topk_idx || !topk_weights || !slot || !layout_range)
        return set_error(EP_ERR_INVALID_ARG, "NULL or misaligned combine argument");
    CombineArgs a{};
    a.y = y_ll;
    a.rows_per_expert = (int64_t)f.num_ranks * b->cap;
    a.y_rows = (int64_t)f.num_experts * a.rows_per_expert;
    a.topk_idx = topk_idx;
    a.w = topk_weights;
    a.slot = slot;
    a.layout_range = layout_range;
    a.out = out;
    a.R = f.num_ranks;
    a.E = f.num_experts;
    a.L = b->L;
    a.K = f.num_topk;
    a.T = f.num_tokens;
    a.H = f.hidden;
    a.G = f.num_ranks;
    a.t0 = t0;
    a.n = n;
    a.status = b->status;
    return launch_combine(a, 2, b->num_sms, as_stream(stream));
}
