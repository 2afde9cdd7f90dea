// ep_combine.cuh -- arguments of the shared gather-reduce kernel (normal,
// hierarchical and low-latency combine).
#pragma once
#include "ep_internal.cuh"

namespace ep {

struct CombineArgs {
    const void* y;            // bf16 rows
    int64_t y_rows;           // rows y holds (bounds of every gathered row)
    const int64_t* topk_idx;  // [R][T][K]
    const float* w;           // [R][T][K]
    const int32_t* perm_pos;  // normal modes: [R][T][K]
    const int32_t* slot;      // low-latency: [R][T][K]
    const int32_t* layout_range;  // low-latency: [R][L][R][2]
    int64_t rows_per_expert;  // low-latency: R * cap
    void* out;                // bf16 [R][T][H]
    int R, E, L, K, T, H, G;
    int t0, n;                // tokens [t0, t0 + n) of every source rank
    int splits;               // channel slices per token (set by launch_combine)
    uint32_t* status;
};

// mode 0: flat, 1: hierarchical, 2: low-latency
ep_status launch_combine(const CombineArgs& a, int mode, int num_sms, cudaStream_t s);

}  // namespace ep
