// kernels_aux.cuh -- launchers of the plan / combine / append / gather kernels
// and the per-dtype decode instantiation tables.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace pkv {

struct PlanArgs {
    const int32_t* lens;   // [B] context lengths (caller)
    int len_offset;        // tokens before the decoded range (lengths below it are flagged)
    int uniform_len;       // >= 0: every sequence has this length and lens is not read
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
    int lens_host;         // lens in page-locked host memory (read with ld.global.cv)
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
    // per-head RMS norm before the rotation (null: none): weights [D] in the
    // element type, shared by all heads; x_d * w_d / sqrt(mean(x^2) + eps)
    const void* q_norm_w;
    const void* k_norm_w;
    float norm_eps;
    double inv_freq[64];   // theta^(-2i/D), i < D/2 (computed on the host)
    int host;              // k_new, v_new, positions, table in page-locked host memory
};

// Copies of host-resident step inputs into device memory, run by extra CTAs
// of the plan launch (a host-buffer step: the decode reads q and the page
// table from these copies, issued after the launch's dependency wait).
// Sources are page-locked host memory read with ld.global.cv; zero counts
// copy nothing.
struct StageArgs {
    const uint4* q_src;    // q as 16-byte vectors
    uint4* q_dst;
    long long q_vecs;
    const int32_t* t_src;  // page table as 4-byte words
    int32_t* t_dst;
    long long t_words;
    int ctas;              // CTAs of the launch doing the copies (set by launch_plan)
};
constexpr int kMaxStageCtas = 64;

// Shared memory of a rotary + append pass: the cos / sin table (one angle per
// thread) and the two norm weight rows.
constexpr int kRopeSmemFloats = 2 * 1024 + 2 * 128;

// Rotary + append: sequences handled together by one CTA of 1024 threads
// (one angle per thread: 1024 / (D / 2)), and their cos / sin table.
constexpr int kRopeThreads = 1024;

// Plan, optionally with the append and the staging copies fused into the
// same launch.
cudaError_t launch_plan(const PlanArgs& pa, const AppendArgs* append, cudaStream_t stream,
                        const StageArgs* stage = nullptr);

cudaError_t launch_combine(pkv_dtype dtype, int head_dim, const float* partials,
                           const int32_t* prefix, const int32_t* lens_eff, const WsHeader* hdr,
                           void* out, int units, int units_per_b, int sub_groups, int gs,
                           const RowShape& rs, int workers, cudaStream_t stream);

// batches up to this size keep their chunk prefix sums in the plan's shared memory
constexpr int kPlanSmemSeqs = 4096;

// Shared-prefix decode: the partial states of the prefix pass (virtual units
// of v_gs rows over the shared prefix, v_nch chunks each) and of the suffix
// pass (the usual units over each sequence's own tokens), merged into out.
struct CascadeArgs {
    const float* s_partials;  // suffix pass
    const int32_t* s_prefix;
    const int32_t* s_lens;
    const WsHeader* s_hdr;
    const float* v_partials;  // prefix pass
    const WsHeader* v_hdr;
    void* out;
    int units_per_b, sub_groups, gs, group, n_q_heads;  // real units
    int v_gs, v_sub, v_nch;                              // virtual units per KV head, chunks
    // prefix pass on the tensor-core tiles (prefix_umma.cu) instead: v_partials
    // holds its slots, v_tiles tiles of v_tile_rows rows per KV head, v_splits
    // slots per tile
    int umma, v_tile_rows, v_tiles, v_splits;
};

// Shared-prefix pass on the fifth-generation tensor cores (prefix_umma.cu):
// grid (splits, tiles, n_kv_heads); CTA (s, t, h) attends query rows
// [t * tile_rows, (t + 1) * tile_rows) of KV head h -- row b * G + g is
// q[b][h * G + g], read through a 3-D tensor map of q ([B][Hq][D], boxes of
// 64 x G x tile_rows / G) -- over its balanced range of the prefix's chunks
// and writes one partial
// state: o [128][D], then m [128], then l [128] -- 128 * D + 256 floats per
// slot, slot (h * tiles + t) * splits + s; o goes through `omap`, a 3-D fp32
// tensor map of the slots (D, 128, slots) with boxes of 32 x 128 x 1.
struct PrefixUmmaArgs {
    const int32_t* table;  // the prefix's page ids (row 0 of the page table)
    int num_pages, n_kv_heads, page_size;
    int chunks;            // 16-token chunks of the prefix
    int splits;            // ranges of chunks per (KV head, tile), 1 .. chunks
    int rows;              // query rows per KV head (B * G)
    int group;             // G
    int tile_rows;         // rows of a tile that belong to it: a multiple of G, <= 128
    int tiles;             // tiles per KV head
    float scale_log2;      // scale * log2(e)
    float* partials;
    uint32_t* status;
};

constexpr int kPrefixTileRows = 128;  // rows of one tensor-core tile (and of a partial slot)

cudaError_t launch_prefix_umma(pkv_dtype dtype, int head_dim, const PrefixUmmaArgs& a,
                               const CUtensorMap& qmap, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, const CUtensorMap& omap,
                               cudaStream_t stream);

// CTAs of the prefix kernel that fit on one SM (0 on an error).
int prefix_umma_ctas_per_sm(pkv_dtype dtype, int head_dim);

// The query gather and prefix check of the shared-prefix decode's plan launch.
struct CascadeGather {
    const uint4* q;        // [B][Hkv * G][D] as 16-byte vectors
    uint4* qv;             // [Hkv][B * G][D]: qv[h][b*G + g] = q[b][h*G + g]; null: no gather
    int batch, n_kv_heads, group, vecs;
    const int32_t* table;  // rows 1 .. B-1 must start with row 0's first share_cols ids
    int table_stride, share_cols;
    int plan_virtual;      // nonzero: CTA 1 plans the prefix pass's virtual decode
};

// One launch: the suffix pass's plan (ps, whose header receives the check's
// status slots), the prefix pass's plan (pv), and the gather + check.
cudaError_t launch_cascade_plan(const PlanArgs& ps, const PlanArgs& pv, const CascadeGather& g,
                                cudaStream_t stream);

cudaError_t launch_cascade_combine(pkv_dtype dtype, int head_dim, const CascadeArgs& c,
                                   int units, cudaStream_t stream);

cudaError_t launch_append(const AppendArgs& a, int batch, uint32_t* status, cudaStream_t stream);

// One bounded wait that never succeeds (see pkv_check_bounded_wait).
cudaError_t launch_wait_check(uint32_t tries, uint32_t* status, unsigned long long* elapsed_ns,
                              cudaStream_t stream);

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
DecodeUmmaInfo decode_umma_info(bool bf16, int head_dim, int rows);
DecodeMmaInfo decode_mma_info_f16_d64(int gs);
DecodeMmaInfo decode_mma_info_f16_d128(int gs);

}  // namespace pkv
