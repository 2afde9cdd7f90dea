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
#include "ep_fp8.cuh"

namespace ep {

__host__ __device__ inline int64_t fp8_row_bytes(int H) { return ((int64_t)H + H / 32 + 15) / 16 * 16; }

// grid-stride over tokens; one thread per 16 channels, 8 lanes per 128-channel block
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint16_t* __restrict__ x, uint8_t* __restrict__ xq,
                                                            int64_t tokens, int H) {
    const int64_t row_q = fp8_row_bytes(H);
    const int ngroups = H / 16;
    for (int64_t g = blockIdx.x; g < tokens; g += gridDim.x) {
        const uint16_t* xr = x + g * H;
        uint8_t* q = xq + g * row_q;
        for (int gi0 = 0; gi0 < ngroups; gi0 += blockDim.x) {
            const int gi = gi0 + threadIdx.x;
            const bool act = gi < ngroups;
            float v[16];
            if (act) {
                bf16x16_to_f32(ld_nc_na_v4(xr + gi * 16), ld_nc_na_v4(xr + gi * 16 + 8), v);
            } else {
#pragma unroll
                for (int u = 0; u < 16; ++u) v[u] = 0.0f;
            }
            float scale;
            const int4 codes = quantize16(v, &scale);
            if (act) {
                st_na_v4(q + (size_t)gi * 16, codes);
                if ((gi & 7) == 0) reinterpret_cast<float*>(q + H)[gi >> 3] = scale;
            }
        }
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
    int64_t grid = (int64_t)c->num_sms * 8;
    if (grid > tokens) grid = tokens;
    int threads = ((c->cfg.hidden / 16 + 31) / 32) * 32;
    if (threads > 256) threads = 256;
    quantize_rows_kernel<<<(int)grid, threads, 0, as_stream(stream)>>>(static_cast<const uint16_t*>(x), xq, tokens,
                                                                       c->cfg.hidden);
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
