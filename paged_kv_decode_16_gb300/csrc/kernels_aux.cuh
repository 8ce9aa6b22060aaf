// kernels_aux.cuh -- launchers of the plan / combine / append / gather kernels
// and the per-dtype decode instantiation tables.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace pkv {

struct PlanArgs {
    const int32_t* lens;   // [B] context lengths (caller)
    int batch;
    int units_per_b;       // Hkv * sub_groups
    long long cap;         // table_stride * page_size
    int workers_req;       // > 0: caller's worker count
    int workers_auto;      // automatic worker count of this kernel on this device
    int min_chunks;        // automatic mode: at least this many chunks per worker
    int32_t* lens_eff;     // [B] clamped lengths (workspace)
    int32_t* prefix;       // [B+1] chunk prefix sums (workspace)
    int32_t* wstart;       // [workers+1] sequence of each worker's first chunk
    WsHeader* hdr;
    int32_t* unit_done;    // [units] merge counters of the decode kernel (nullable), zeroed
    long long units;
    const int32_t* table;  // page table (nullable), prefetched into L2 for the decode kernel
    int table_stride;
    int page_size;
};

struct AppendArgs {
    const uint4* k_new;    // [B][Hkv][D] as 16-byte vectors
    const uint4* v_new;
    const int32_t* positions;
    const int32_t* table;
    int table_stride;
    uint4* k_pool;
    uint4* v_pool;
    int n_kv_heads, vecs, page_size, num_pages;  // vecs = D / 8
    // rotary embedding before the append (q_in null: plain append)
    const uint4* q_in;     // [B][Hq][D] queries of the step
    uint4* q_out;          // [B][Hq][D] rotated queries
    int n_q_heads;
    int bf16;              // element type of q / k / v: bf16, else fp16
    double inv_freq[64];   // theta^(-2i/D), i < D/2 (computed on the host)
};

// Rotary + append: sequences handled together by one CTA of 1024 threads
// (one angle per thread: 1024 / (D / 2)), and their cos / sin table.
constexpr int kRopeThreads = 1024;

// Plan, optionally with the append fused into the same launch.
cudaError_t launch_plan(const PlanArgs& pa, const AppendArgs* append, cudaStream_t stream);

cudaError_t launch_combine(pkv_dtype dtype, int head_dim, const float* partials,
                           const int32_t* prefix, const int32_t* lens_eff, const WsHeader* hdr,
                           void* out, int units, int units_per_b, int sub_groups, int gs,
                           int group, int n_q_heads, int merge_batch, cudaStream_t stream);

// batches up to this size keep their chunk prefix sums in the plan's shared memory
constexpr int kPlanSmemSeqs = 4096;

cudaError_t launch_append(const AppendArgs& a, int batch, uint32_t* status, cudaStream_t stream);

// Rotary embedding of q and k_new, then the append (stand-alone launch).
cudaError_t launch_rope_append(const AppendArgs& a, int batch, int head_dim, uint32_t* status,
                               cudaStream_t stream);

cudaError_t launch_gather(const void* k_pool, const void* v_pool, const int32_t* table,
                          int table_stride, const int32_t* lens, int batch, int n_kv_heads,
                          int head_dim, int page_size, int num_pages, int max_len, void* k_out,
                          void* v_out, uint32_t* status, cudaStream_t stream);

DecodeKernelInfo decode_info_bf16(int head_dim, int gs);
DecodeKernelInfo decode_info_f16(int head_dim, int gs);

// Tensor-core variant (decode_mma.cuh).
DecodeMmaInfo decode_mma_info_bf16_d64(int gs);
DecodeMmaInfo decode_mma_info_bf16_d128(int gs);
DecodeMmaInfo decode_mma_info_f16_d64(int gs);
DecodeMmaInfo decode_mma_info_f16_d128(int gs);

}  // namespace pkv
