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
// kernel quantises each token once (per-128-channel amax, the e4m3 code of the
// IEEE quotient x / scale, ep_fp8.cuh) and stores the message to its K regions; slots are
// the deterministic (t, k)-order rank of the entry among the source's entries
// for the same expert (no atomic slot claims); a publisher kernel, launched as
// a programmatic dependent of the send, stores every count of every source
// with st.release once the send grid has completed, 0 included.  The receive
// kernel polls each count with ld.acquire under a time limit and packs the
// messages.
#include <cuda_fp8.h>
#include <cstdlib>

#include "ep_internal.cuh"
#include "ep_combine.cuh"
#include "ep_fp8.cuh"

struct ep_ll_buffer {
    ep_config cfg;
    int cap, L, device, num_sms;
    int64_t msg_bytes;
    void* mem;
    size_t bytes;
    uint8_t* regions[2];
    int32_t* counts[2];
    uint32_t* status;
    int cur;
    int64_t wait_timeout_ns;
    int send_ctas_per_sm;    // send kernel launch shape
    size_t send_smem_bytes;
    int recv_split;          // CTAs per (source, expert) region of the receive; 0 = from the last send
    int last_send_n;         // tokens per source of the last send (sizes the receive's split)
    int64_t* wait_trace;     // nullable device [E][R]: receive signal waits (ns)
};

namespace ep {

constexpr int kRecvThreads = 128;

struct LLSendArgs {
    const uint16_t* x;  // bf16 bits [R][T][H]
    const int64_t* topk_idx;
    int32_t* slot_out;
    uint8_t* regions;
    int32_t* counts;       // [E][R] of the buffer in use
    int32_t* other_counts; // [E][R] of the other buffer
    int R, E, K, T, H, cap, t0, n;
    int64_t msg_bytes;
    uint32_t* status;
};


// Persistent send: CTA c owns the contiguous tokens [q0, q1) of the flattened
// (source, token) order.  Thread 0 streams their x rows global -> shared with
// cp.async.bulk, `stages` tokens ahead (one mbarrier per stage).  A running
// per-expert count of the current source in shared memory gives each entry's
// slot (initialised once from the source's earlier tokens).  All threads
// quantise the staged row into a message in shared memory (header, e4m3
// codes, fp32 scales); thread 0 then writes that message to each of the
// token's K regions with cp.async.bulk shared -> global.  The counts are
// published afterwards by ll_publish_kernel.
constexpr int kSendMaxStages = 8;

__host__ __device__ inline size_t ll_send_fixed_smem(int E) {
    size_t off = kSendMaxStages * sizeof(uint64_t) + sizeof(int32_t) * ((size_t)E + 4 * kMaxTopk + 4);
    return (off + 127) & ~size_t(127);
}

__global__ void __launch_bounds__(256, 3) ll_send_kernel(LLSendArgs a, int stages, int64_t timeout_ns) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int32_t* cnt = reinterpret_cast<int32_t*>(bar + kSendMaxStages);  // [E]
    int32_t* sh_e2 = cnt + a.E;                                         // [2][kMaxTopk] by token parity
    int32_t* sh_slot2 = sh_e2 + 2 * kMaxTopk;                           // [2][kMaxTopk]
    int32_t* sh_flag = sh_slot2 + 2 * kMaxTopk;                         // [1] abort
    const int R = a.R, E = a.E, K = a.K, H = a.H, n = a.n;
    const int64_t row_bytes = (int64_t)H * 2;
    uint8_t* xs = smem + ll_send_fixed_smem(E);                        // [stages][row_bytes]
    uint8_t* msgs = xs + (size_t)stages * row_bytes;                    // [2][msg_bytes]
    const int64_t total = (int64_t)R * n;
    const int64_t q0 = total * blockIdx.x / gridDim.x, q1 = total * (blockIdx.x + 1) / gridDim.x;
    const int tid = threadIdx.x;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    auto token_g = [&](int64_t q) -> int64_t { return (int64_t)(q / n) * a.T + a.t0 + (int)(q % n); };
    auto issue_load = [&](int64_t q) {
        const int st = (int)((q - q0) % stages);
        mbar_arrive_expect_tx(&bar[st], (uint32_t)row_bytes);
        bulk_g2s(xs + (size_t)st * row_bytes, a.x + token_g(q) * H, (uint32_t)row_bytes, &bar[st]);
    };
    if (tid == 0) {
        for (int st = 0; st < stages; ++st) mbar_init(&bar[st], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
        for (int64_t q = q0; q < q1 && q < q0 + stages; ++q) issue_load(q);
        sh_flag[0] = 0;
    }
    int cur_s = -1;
    int64_t nx_e = -1;  // next token's entry (threads < K), loaded one token ahead
    if (q0 < q1 && tid < K) nx_e = a.topk_idx[token_g(q0) * K + tid];
    int64_t next_load = q0 + stages < q1 ? q0 + stages : q1;  // thread 0: first token not yet loaded
    int64_t q_stop = q1;
    for (int64_t q = q0; q < q1; ++q) {
        const int64_t i = q - q0;
        // entries and slots of this token live in the buffer of its parity, so
        // that thread 0 can still read the previous token's while the others
        // move on
        int32_t* sh_e = sh_e2 + (i & 1) * kMaxTopk;
        int32_t* sh_slot = sh_slot2 + (i & 1) * kMaxTopk;
        const int s = (int)(q / n), j = (int)(q % n), t = a.t0 + j;
        const int64_t g = (int64_t)s * a.T + t;
        const int64_t my_e = nx_e;
        if (q + 1 < q1 && tid < K) nx_e = a.topk_idx[token_g(q + 1) * K + tid];
        // A new source: its per-expert counts restart from the source's tokens
        // before this one (only the CTA's first token can have any; a later
        // source change starts at token 0).  Their loads are issued now and
        // consumed after the quantisation, which hides their latency.
        constexpr int kScanU = 8;
        int64_t ee[kScanU];
        int before = 0;
        const bool scan = s != cur_s;
        const int64_t* first = a.topk_idx + ((int64_t)s * a.T + a.t0) * K;
        if (scan) {
            __syncthreads();  // thread 0 is done with the previous token's counts
            for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
            before = j * K;
#pragma unroll
            for (int u = 0; u < kScanU; ++u) {
                const int p = tid + u * (int)blockDim.x;
                ee[u] = p < before ? first[p] : -1;
            }
            cur_s = s;
        }
        if (tid < K) {
            int ev = -1;
            if (my_e >= 0 && my_e < E) ev = (int)my_e;
            else if (my_e != -1) flag(a.status, FLAG_INVALID_TOPK);
            sh_e[tid] = ev;
        }
        // the staged x row of this token
        const int st = (int)(i % stages);
        if (!mbar_wait_bounded(&bar[st], (uint32_t)((i / stages) & 1), timeout_ns)) {
            flag(a.status, FLAG_TIMEOUT);
            atomicExch(sh_flag, 1);
        }
        __syncthreads();
        if (sh_flag[0]) {
            q_stop = q;
            break;
        }
        // ---- quantise into the message buffer ----------------------------------
        uint8_t* msg = msgs + (size_t)(i & 1) * a.msg_bytes;
        const uint8_t* xrow = xs + (size_t)st * row_bytes;
        const int ngroups = H / 16;
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
            const int4 codes = quantize16(v, &scale);
            if (act) {
                *reinterpret_cast<int4*>(msg + 16 + (size_t)gi * 16) = codes;
                if ((gi & 7) == 0) *reinterpret_cast<float*>(msg + 16 + H + (gi >> 3) * 4) = scale;
            }
        }
        if (scan) {
#pragma unroll
            for (int u = 0; u < kScanU; ++u)
                if (ee[u] >= 0 && ee[u] < E) atomicAdd(&cnt[ee[u]], 1);
            for (int p = tid + kScanU * (int)blockDim.x; p < before; p += blockDim.x) {
                const int64_t e = first[p];
                if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
            }
        }
        if (tid == 0) *reinterpret_cast<int4*>(msg) = make_int4(t, 0, 0, 0);
        fence_proxy_async_smem();  // the message is read by the bulk copies below
        __syncthreads();
        if (tid == 0) {
            // slots: the running per-expert counts of this source, (t, k) order
            for (int k = 0; k < K; ++k) {
                const int ev = sh_e[k];
                int sl = -1;
                if (ev >= 0) {
                    sl = cnt[ev];
                    cnt[ev] = sl + 1;
                    if (sl >= a.cap) {
                        flag(a.status, FLAG_CAPACITY);
                        sl = -1;
                    }
                }
                sh_slot[k] = sl;
                a.slot_out[g * K + k] = sl;
                if (sl >= 0)
                    bulk_s2g(a.regions + (((int64_t)ev * R + s) * a.cap + sl) * a.msg_bytes, msg,
                             (uint32_t)a.msg_bytes);
            }
            bulk_commit();
            // the x stage of this token is free again: stream the token `stages` ahead
            if (q + stages < q1) {
                fence_proxy_async_smem();
                issue_load(q + stages);
                next_load = q + stages + 1;
            }
            // the message buffer of the previous token must be read out before reuse
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
    int64_t* wait_trace;  // nullable [E][R]: ns from the CTA's start until its counts were read
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


// grid = (R sources, E experts, Z): CTA (s, e, z) waits for the counts of
// sources 0..s of expert e (begin = exclusive prefix), then copies its share
// (every Z-th group of 4 messages) of region (e, s).
__global__ void __launch_bounds__(kRecvThreads) ll_recv_kernel(LLRecvArgs a) {
    __shared__ int sh_begin, sh_count;
    const int s = blockIdx.x, e = blockIdx.y;
    const int z = blockIdx.z, Z = gridDim.z;  // this CTA's share of the region's messages
    const uint64_t t_start = a.wait_trace ? globaltimer_ns() : 0;
    // launched as a programmatic dependent of the count publisher: start once
    // its grid (and every write before it) is complete.  No early trigger for
    // the combine that follows: its CTAs would sit resident through this
    // grid's last wave (two overlapped microbatches: 105.5 -> 106.5 us/layer)
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
            // the signal wait: from this CTA's start until its counts were read
            if (a.wait_trace && z == 0) a.wait_trace[(int64_t)e * R + s] = (int64_t)(globaltimer_ns() - t_start);
        }
    }
    __syncthreads();
    const int begin = sh_begin, count = sh_count;
    const int d = e / L, l = e % L;
    if (threadIdx.x == 0 && z == 0) {
        int32_t* lr = a.layout_range + (((int64_t)d * L + l) * R + s) * 2;
        lr[0] = begin;
        lr[1] = count;
        if (s == R - 1) a.packed_recv_count[(int64_t)d * L + l] = begin + count;
    }
    const int S = H / 128;
    const int64_t rows_per_expert = (int64_t)R * a.cap;
    const int nwarps = blockDim.x / 32;
    const int nv = H / 16;
    for (int i = z * nwarps + warp; i < count; i += nwarps * Z) {
        const uint8_t* msg = a.regions + (((int64_t)e * R + s) * a.cap + i) * a.msg_bytes;
        const int64_t p = ((int64_t)d * L + l) * rows_per_expert + begin + i;
        const int4* src = reinterpret_cast<const int4*>(msg + 16);
        int4* dx = reinterpret_cast<int4*>(a.packed_x + p * H);
        // the message's vectors in batches of eight per lane, each batch's
        // loads before its stores; the scales ride along
        const float* sc = reinterpret_cast<const float*>(msg + 16 + H);
        float scv = lane < S ? __ldcg(sc + lane) : 0.0f;
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
        if (lane < S) __stcs(a.packed_scales + p * S + lane, scv);
        for (int v = lane + 32; v < S; v += 32) __stcs(a.packed_scales + p * S + v, __ldcg(sc + v));
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
    int64_t one = (int64_t)E * R * cap * ep_ll_message_bytes(H) + counts;
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
    if (H < 128 || H % 128 || H > 16384)
        return set_error(EP_ERR_INVALID_ARG, "hidden %d must be a multiple of 128 in [128, 16384]", H);
    if (cap < 1 || cap > 4096) return set_error(EP_ERR_INVALID_ARG, "cap %d outside [1, 4096]", cap);
    ep_ll_buffer* b = new ep_ll_buffer();
    b->cfg = *cfg;
    b->cap = cap;
    b->L = E / R;
    b->msg_bytes = ep_ll_message_bytes(H);
    b->cur = 1;  // the first send flips to buffer 0
    b->wait_timeout_ns = 100000000ll;
    b->send_ctas_per_sm = 3;
    b->send_smem_bytes = 72 * 1024;
    if (const char* v = getenv("EP_LL_SEND_CTAS_PER_SM")) b->send_ctas_per_sm = atoi(v) > 0 ? atoi(v) : 3;
    if (const char* v = getenv("EP_LL_SEND_SMEM_KB")) b->send_smem_bytes = (size_t)(atoi(v) > 16 ? atoi(v) : 72) * 1024;
    b->recv_split = 0;
    b->last_send_n = cap;
    if (const char* v = getenv("EP_LL_RECV_SPLIT")) b->recv_split = atoi(v);
    {
        // room for two messages, the fixed part and at least two staged rows
        const size_t need = ll_send_fixed_smem(E) + 2 * (size_t)ep_ll_message_bytes(H) + 2 * (size_t)H * 2;
        if (b->send_smem_bytes < need) b->send_smem_bytes = need;
    }
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
    for (int i = 0; i < 2; ++i) {
        uint8_t* p = base + i * one;
        b->regions[i] = p;
        b->counts[i] = reinterpret_cast<int32_t*>(p + reg);
    }
    b->status = reinterpret_cast<uint32_t*>(base + 2 * one);
    // counts start at the empty sentinel, the status word at 0
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaMemset(b->counts[i], 0xff, (size_t)E * R * 4);
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

extern "C" ep_status ep_ll_set_wait_trace(ep_ll_buffer* b, int64_t* wait_ns) {
    if (!b) return set_error(EP_ERR_INVALID_ARG, "buffer is NULL");
    b->wait_trace = wait_ns;
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
    a.other_counts = b->counts[b->cur ^ 1];
    a.R = f.num_ranks;
    a.E = f.num_experts;
    a.K = f.num_topk;
    a.T = f.num_tokens;
    a.H = f.hidden;
    a.cap = b->cap;
    a.t0 = t0;
    a.n = n;
    b->last_send_n = n;
    a.msg_bytes = b->msg_bytes;
    a.status = b->status;
    cudaStream_t s = as_stream(stream);
    if (n > 0) {
        const int64_t row_bytes = (int64_t)a.H * 2;
        const size_t fixed = ll_send_fixed_smem(a.E) + 2 * (size_t)a.msg_bytes;
        int stages = (int)((b->send_smem_bytes - fixed) / row_bytes);
        if (stages > kSendMaxStages) stages = kSendMaxStages;
        if (stages < 2) stages = 2;
        const size_t smem = fixed + (size_t)stages * row_bytes;
        int64_t grid = (int64_t)b->num_sms * b->send_ctas_per_sm;
        if (grid > (int64_t)a.R * n) grid = (int64_t)a.R * n;
        static int raised[kMaxDevicesTracked] = {};
        if (b->device < 0 || b->device >= kMaxDevicesTracked || raised[b->device] < (int)smem) {
            EP_CUDA(cudaFuncSetAttribute(ll_send_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
            if (b->device >= 0 && b->device < kMaxDevicesTracked) raised[b->device] = (int)smem;
        }
        ll_send_kernel<<<(int)grid, 256, smem, s>>>(a, stages, 2000000000ll);
        EP_CHECK_LAUNCH("ll_send_kernel");
    }
    // counts after the data: a programmatic dependent launch overlaps the
    // publisher's histogram with the send; its griddepcontrol.wait orders the
    // count stores after every data store of the send grid
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(a.R);
    // 128 threads: four warps of 32 registers fit in the registers the send's
    // three CTAs per SM leave free, so the publisher's histogram runs beside
    // the send instead of after it (eager decode layer 111.0 -> 109.8 us,
    // skewed send 65.5 -> 63.5 us per microbatch; two microbatches overlapped
    // on two streams 105.5 -> 107.5 us per layer).  EP_LL_PUB_THREADS (32..256)
    // overrides it.
    static const int pub_threads = [] {
        const char* v = getenv("EP_LL_PUB_THREADS");
        const int x = v ? atoi(v) / 32 * 32 : 128;
        return x < 32 ? 32 : (x > 256 ? 256 : x);
    }();
    lc.blockDim = dim3(pub_threads);
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
    a.wait_trace = b->wait_trace;
    cudaLaunchConfig_t lc = {};
    // split each region's messages over Z CTAs, Z = half the average messages
    // per region of the last send (ceil(n*K/E)), rounded up: the measured best
    // on the decode batch (4 messages per region on average: Z = 2) and on the
    // Zipf-skewed microbatches (8 on average, hot regions near cap: Z = 4)
    const int64_t avg = ((int64_t)b->last_send_n * f.num_topk + f.num_experts - 1) / f.num_experts;
    int Z = (int)((avg + 1) / 2);
    if (b->recv_split > 0) Z = b->recv_split;
    if (Z < 1) Z = 1;
    if (Z > 8) Z = 8;
    lc.gridDim = dim3(a.R, a.E, Z);
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
