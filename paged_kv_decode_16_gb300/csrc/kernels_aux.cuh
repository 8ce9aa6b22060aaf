// kernels_aux.cuh -- launchers of the plan / combine / append / gather kernels
// and the per-dtype decode instantiation tables.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace pkv {

cudaError_t launch_plan(const int32_t* lens, int batch, int units_per_b, long long cap,
                        int workers_req, int workers_auto, int min_chunks, int32_t* lens_eff,
                        int32_t* prefix, WsHeader* hdr, cudaStream_t stream);

cudaError_t launch_combine(pkv_dtype dtype, int head_dim, const float* partials,
                           const int32_t* prefix, const int32_t* lens_eff, const WsHeader* hdr,
                           void* out, int units, int units_per_b, int sub_groups, int gs,
                           int group, int n_q_heads, cudaStream_t stream);

cudaError_t launch_append(const void* k_new, const void* v_new, const int32_t* table,
                          int table_stride, const int32_t* positions, int batch, int n_kv_heads,
                          int head_dim, int page_size, int num_pages, void* k_pool, void* v_pool,
                          uint32_t* status, cudaStream_t stream);

cudaError_t launch_gather(const void* k_pool, const void* v_pool, const int32_t* table,
                          int table_stride, const int32_t* lens, int batch, int n_kv_heads,
                          int head_dim, int page_size, int num_pages, int max_len, void* k_out,
                          void* v_out, uint32_t* status, cudaStream_t stream);

DecodeKernelInfo decode_info_bf16(int head_dim, int gs);
DecodeKernelInfo decode_info_f16(int head_dim, int gs);

}  // namespace pkv
