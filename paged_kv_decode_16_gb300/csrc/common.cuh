// common.cuh -- shared device helpers of the paged decode library (sm_103a).
//
// Inline PTX for the Blackwell async-copy path: mbarrier wait/arrive with a
// transaction count, and the bulk (TMA) global->shared copy that completes on
// an mbarrier.  Every wait is bounded: after kSpinLimit failed polls the caller
// gets `false` and reports PKV_DEV_TIMEOUT instead of spinning forever.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

constexpr int kChunk = 16;               // tokens per pipeline stage
constexpr unsigned kFull = 0xffffffffu;  // full-warp shuffle mask
constexpr uint32_t kSpinLimit = 1u << 22;
constexpr int kMaxAppendCtas = 32;       // CTAs of the append fused into the plan launch

// Workspace header (first 256 bytes of the decode workspace).
struct WsHeader {
    uint32_t status;         // PKV_DEV_* bits of the current call (plan, decode)
    int32_t total_chunks;    // chunks over all (sequence, KV head, sub-group) units
    int32_t num_workers;     // workers that received a non-empty range
    int32_t append_slots;    // append_status entries written by this call
    uint32_t append_status[kMaxAppendCtas];  // PKV_DEV_* bits of each fused-append CTA
    int32_t chunks_per_worker;  // sw: every worker's range holds sw or sw + 1 chunks
    int32_t extra_chunks;       // r: workers 0 .. r-1 hold sw + 1 chunks
    int32_t pad[64 - 6 - kMaxAppendCtas];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// First chunk of worker w's range (workers 0 .. r-1 hold sw + 1 chunks, the
// others sw), and the worker whose range holds chunk f.
__host__ __device__ __forceinline__ int range_begin(int w, int sw, int r) {
    return w * sw + (w < r ? w : r);
}
__host__ __device__ __forceinline__ int worker_of(int f, int sw, int r) {
    const int big = r * (sw + 1);
    return f < big ? f / (sw + 1) : r + (f - big) / sw;
}

// Query rows of the units.  Unit (b, KV head h, sub-group sg) holds rows
// r = 0 .. rows(sg) - 1; sub-group sg = tile * head_blocks + block picks one
// tile of queries_per_unit query tokens (the last tile may be shorter) and one
// block of heads_per_unit query heads of the GQA group; row r is token
// first_query(sg) + r / heads_per_unit of query head
// h * group + block * heads_per_unit + r % heads_per_unit.  One query per
// sequence: a single tile of one token, every row of a unit in use.
struct RowShape {
    int n_queries;         // query tokens per sequence: q, out [B][n_queries][Hq][D]
    int queries_per_unit;  // tokens of a full query tile
    int heads_per_unit;    // query heads of a head block
    int head_blocks;       // group / heads_per_unit
    int group, n_q_heads;

    __host__ __device__ __forceinline__ int first_query(int sg) const {
        return (sg / head_blocks) * queries_per_unit;
    }
    __host__ __device__ __forceinline__ int rows(int sg) const {
        const int n = n_queries - first_query(sg);
        return (n < queries_per_unit ? n : queries_per_unit) * heads_per_unit;
    }
    __host__ __device__ __forceinline__ int query(int sg, int r) const {
        return first_query(sg) + r / heads_per_unit;
    }
    // row r of unit (b, h, sg) as a row of q / out
    __host__ __device__ __forceinline__ long long row(int b, int h, int sg, int r) const {
        const int t = sg / head_blocks, blk = sg - t * head_blocks;
        const int jl = r / heads_per_unit, g = r - jl * heads_per_unit;
        return ((long long)b * n_queries + t * queries_per_unit + jl) * n_q_heads + h * group +
               blk * heads_per_unit + g;
    }
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order earlier generic-proxy shared-memory accesses before later async-proxy
// (bulk copy) writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete: false after
// `tries` failed polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t tries = kSpinLimit) {
    for (uint32_t it = 0; it < tries; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
    }
    return false;
}

// Bulk async copy global -> shared (no tensor map), completes `bytes` of
// transaction on `bar`.  dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tensor copy (cp.async.bulk.tensor) of one box at element coordinates
// (x, y) of `map` into shared memory, completing on `bar`.  x times the
// element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// The same for a 3-D tensor map, element coordinates (x, y, z).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y,
                                            int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// Tensor store (cp.async.bulk.tensor) of one box from shared memory to
// element coordinates (x, y, z) of `map`, tracked by the thread's bulk group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y,
                                             int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_group_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// An L2 policy that makes the lines a load brings in the first to be evicted:
// for data read once (the K/V stream of a decode), so that it does not push
// out what is read again (page tables, prefix sums, partial states).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// tma_load_2d with an L2 cache policy for the loaded lines.
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y,
                                                 uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 2^x with the hardware approximation (flushes subnormal results to zero).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// bulk_g2s with an L2 cache policy for the loaded lines.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while the previous kernel in the
// stream still runs; pdl_wait() blocks until that kernel has completed and its
// memory is visible (a no-op for a normal launch).  pdl_trigger() lets the
// next kernel in the stream be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
    if (status) atomicOr(status, bits);
}

// 16-bit storage types and their conversions.
template <typename T>
struct Cvt;

template <>
struct Cvt<__nv_bfloat16> {
    // 8 packed bf16 (one 16-byte vector) -> 8 floats
    static __device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
};

template <>
struct Cvt<__half> {
    static __device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
            float2 x = __half22float2(h);
            f[2 * i] = x.x;
            f[2 * i + 1] = x.y;
        }
    }
    static __device__ __forceinline__ uint32_t pack2(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
};

// P in two bf16 pieces: hi = bf16(p), lo = bf16(p - hi).  bf16 keeps 8
// significant bits, too few for P (an output that cancels would carry ~2^-9
// relative error); hi + lo carries ~16.  fp16 P (11 bits) is used as is.
__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = Cvt<__nv_bfloat16>::pack2(a, b);
    const float ha = __uint_as_float(hi << 16), hb = __uint_as_float(hi & 0xffff0000u);
    lo = Cvt<__nv_bfloat16>::pack2(a - ha, b - hb);
}

__host__ __device__ constexpr int next_pow2(int x) {
    return x <= 1 ? 1 : (x <= 2 ? 2 : (x <= 4 ? 4 : (x <= 8 ? 8 : 16)));
}

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// Floats in one partial-state slot: o [gs][D], then m [gs], then l [gs],
// padded to a multiple of 4 floats so every slot (and every o row) starts on
// a 16-byte boundary for the float4 stores.
__host__ __device__ constexpr int partial_slot_floats(int gs, int d) {
    return (gs * (d + 2) + 3) / 4 * 4;
}

// Parameters of the decode kernel (one struct, passed by value).
struct DecodeParams {
    const void* q;            // [B][Hq][D]
    const void* k_pool;       // [NP][Hkv][P][D]
    const void* v_pool;
    const int32_t* table;     // [B][stride]
    const int32_t* lens_eff;  // [B] lengths after the plan's clamp (workspace)
    const int32_t* prefix;    // [B+1] chunk prefix sums (workspace)
    const int32_t* wstart;    // [workers+1] sequence holding each worker's first chunk
    int units;                // U = batch * Hkv * sub_groups
    const WsHeader* hdr;      // total chunks, worker count
    uint32_t* status;
    float* partials;          // [slots][partial_slot_floats(GS, D)]
    int32_t* unit_done;       // [U] chunks finished per unit (zeroed by the plan); null: split
                              // units are left to the combine kernel
    int all_partials;         // nonzero: every segment leaves a partial state, out is not written
                              // (a later merge completes it)
    RowShape rows;            // the query rows of each unit
    void* out;                // [B][n_queries][Hq][D]
    int table_stride;
    int batch, n_q_heads, n_kv_heads, page_size, num_pages;
    int group;                // G = Hq / Hkv
    int sub_groups;           // units per KV head (query tiles x head blocks)
    float scale_log2;         // scale * log2(e)
};

// Launch a kernel on `stream` with programmatic stream serialization, so that
// it can be scheduled while the previous kernel of the stream finishes; every
// kernel of this library calls pdl_wait() before touching global memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Launch configuration of one tcgen05 decode instantiation (decode_umma.cu:
// one CTA per worker; the kernel also takes the q, K and V tensor maps).
struct DecodeUmmaInfo {
    void (*fn)(DecodeParams, CUtensorMap, CUtensorMap, CUtensorMap) = nullptr;
    int stages = 0;
    int smem_bytes = 0;
    int n = 0;        // query rows of the tile (a unit's rows rounded up)
    int threads = 0;  // threads of a CTA (consumer warps + the producer warp)
};

// Launch configuration of one tensor-core decode instantiation (the kernel
// also takes the K and V tensor maps).
struct DecodeMmaInfo {
    void (*fn)(DecodeParams, CUtensorMap, CUtensorMap);
    int warps;
    int stages;
    int smem_bytes;
    int gs;
};

// Launch configuration of one decode-kernel instantiation.
struct DecodeKernelInfo {
    void (*fn)(DecodeParams);
    int warps;       // warps (workers) per CTA
    int stages;      // chunk buffers per warp
    int smem_bytes;  // dynamic shared memory per CTA
    int gs;          // query heads served per unit
};

}  // namespace pkv
