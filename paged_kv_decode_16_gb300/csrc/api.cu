// api.cu -- the C ABI (include/pagedkv.h): host-side validation, workspace
// layout, tensor-map encoding, and the stream-ordered launches of the plan,
// decode and combine kernels, the KV append and the gather.
//
// Conventions follow Experimental LibTorch prefix cache, "Identity, ownership
// and output behavior": work is ordered on the caller's stream, the caller
// owns every buffer, the host validates shapes and rejects aliased output
// before anything is launched, and failures are reported, never thrown.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "common.cuh"
#include "kernels_aux.cuh"
#include "merge.cuh"
#include "pool_impl.hpp"

namespace {

using pkv::DecodeKernelInfo;
using pkv::DecodeMmaInfo;
using pkv::DecodeUmmaInfo;
using pkv::WsHeader;

constexpr int kMinChunksPerWorker = 4;  // automatic worker count: at least this many chunks each

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline pkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

// G = sub_groups * gs with gs <= max_gs (the widest group one warp serves):
// the smallest number of sub-groups that divides G.
inline bool split_group(int group, int max_gs, int* sub_groups, int* gs) {
    for (int ns = (group + max_gs - 1) / max_gs; ns <= group; ++ns) {
        if (group % ns == 0) {
            *sub_groups = ns;
            *gs = group / ns;
            return true;
        }
    }
    return false;
}

pkv_status check_shapes(int batch, int n_q_heads, int n_kv_heads, int head_dim, int page_size) {
    if (batch < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || page_size <= 0)
        return PKV_ERR_INVALID_ARG;
    if (n_q_heads % n_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (page_size % 16 != 0 || page_size > 256) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

inline bool valid_variant(int v) {
    return v == PKV_VARIANT_AUTO || v == PKV_VARIANT_CUDA_CORES ||
           v == PKV_VARIANT_TENSOR_CORES || v == PKV_VARIANT_TCGEN05;
}

// The decode kernel chosen for a call: an entry of one instantiation table.
// A worker is a warp, except on the tcgen05 kernel, where it is a CTA.
struct KernelPick {
    int variant = 0;  // PKV_VARIANT_CUDA_CORES, _TENSOR_CORES or _TCGEN05
    DecodeKernelInfo cc{};
    DecodeMmaInfo mma{};
    DecodeUmmaInfo um{};
    const void* fn() const {
        return variant == PKV_VARIANT_TCGEN05     ? reinterpret_cast<const void*>(um.fn)
               : variant == PKV_VARIANT_TENSOR_CORES ? reinterpret_cast<const void*>(mma.fn)
                                                     : reinterpret_cast<const void*>(cc.fn);
    }
    int threads() const {
        return variant == PKV_VARIANT_TCGEN05       ? um.threads
               : variant == PKV_VARIANT_TENSOR_CORES ? mma.warps * 32
                                                     : cc.warps * 32;
    }
    int warps() const {  // workers per CTA
        return variant == PKV_VARIANT_TCGEN05       ? 1
               : variant == PKV_VARIANT_TENSOR_CORES ? mma.warps
                                                     : cc.warps;
    }
    int smem() const {
        return variant == PKV_VARIANT_TCGEN05       ? um.smem_bytes
               : variant == PKV_VARIANT_TENSOR_CORES ? mma.smem_bytes
                                                     : cc.smem_bytes;
    }
};

KernelPick pick_kernel(pkv_dtype dtype, int head_dim, int variant, int gs) {
    KernelPick k;
    k.variant = variant;
    if (variant == PKV_VARIANT_TCGEN05) {
        k.um = pkv::decode_umma_info(dtype == PKV_BF16, head_dim, gs);
    } else if (variant == PKV_VARIANT_TENSOR_CORES) {
        if (dtype == PKV_BF16)
            k.mma = head_dim == 128 ? pkv::decode_mma_info_bf16_d128(gs)
                                    : pkv::decode_mma_info_bf16_d64(gs);
        else
            k.mma = head_dim == 128 ? pkv::decode_mma_info_f16_d128(gs)
                                    : pkv::decode_mma_info_f16_d64(gs);
    } else {
        k.cc = dtype == PKV_BF16 ? pkv::decode_info_bf16(head_dim, gs)
                                 : pkv::decode_info_f16(head_dim, gs);
    }
    return k;
}

// Per (device, kernel): dynamic shared memory opt-in done, and the automatic
// worker count = SMs x resident CTAs per SM x workers per CTA.
std::mutex g_mu;
std::map<std::pair<int, const void*>, int> g_auto_workers;

pkv_status prepare_kernel(const KernelPick& k, int* auto_workers) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    const auto key = std::make_pair(dev, k.fn());
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_auto_workers.find(key);
        if (it != g_auto_workers.end()) {
            *auto_workers = it->second;
            return PKV_OK;
        }
    }
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (cudaFuncSetAttribute(k.fn(), cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem()) !=
        cudaSuccess)
        return PKV_ERR_CUDA;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k.fn(), k.threads(),
                                                      k.smem()) != cudaSuccess)
        return PKV_ERR_CUDA;
    const int workers = sms * (per_sm > 0 ? per_sm : 1) * k.warps();
    std::lock_guard<std::mutex> lk(g_mu);
    g_auto_workers[key] = workers;
    *auto_workers = workers;
    return PKV_OK;
}

struct WsLayout {
    size_t lens_eff, prefix, wstart, unit_done, partials, total;
};

// Partial slots: the segment of unit u in worker w's range uses slot u + w < U + NW.
WsLayout ws_layout(int batch, long long units, int gs, int head_dim, int workers) {
    WsLayout w;
    size_t off = sizeof(WsHeader);
    w.lens_eff = off;
    off += align256((size_t)batch * 4);
    w.prefix = off;
    off += align256((size_t)(batch + 1) * 4);
    w.wstart = off;
    off += align256((size_t)(workers + 1) * 4);
    w.unit_done = off;
    off += align256((size_t)units * 4);
    w.partials = off;
    const size_t slots = (size_t)(units + workers);
    off += align256(slots * pkv::partial_slot_floats(gs, head_dim) * 4);
    w.total = off;
    return w;
}

// Everything the decode steps derive from the shapes and the variant.
struct DecodeSetup {
    int group, sub_groups, gs, units_per_b;
    long long units;
    int workers;       // launched workers (upper bound of the plan's count)
    int workers_auto;  // automatic count for this kernel on this device
    KernelPick kernel;
    WsLayout ws;
    pkv::RowShape rs{};  // the query rows of each unit
};

// Query tokens per sequence that paged_decode_attention_multi takes.
constexpr int kMaxQueries = 64;

// AUTO picks the tensor-core kernel; CUDA cores on request.
int resolve_variant(int variant) {
    return variant == PKV_VARIANT_AUTO ? PKV_VARIANT_TENSOR_CORES : variant;
}

pkv_status setup_decode(int batch, int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                        pkv_dtype dtype, int num_workers, int variant, DecodeSetup* s,
                        int force_gs = 0, int n_queries = 1) {
    pkv_status st = check_shapes(batch, n_q_heads, n_kv_heads, head_dim, page_size);
    if (st != PKV_OK) return st;
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if (num_workers < 0 || !valid_variant(variant)) return PKV_ERR_INVALID_ARG;
    const int v = resolve_variant(variant);
    s->group = n_q_heads / n_kv_heads;
    const int max_gs = v == PKV_VARIANT_TENSOR_CORES ? 16 : 8;
    if (n_queries > 1) {
        // rows of a unit (one warp: one m16 tile, or two): the queries split
        // into the fewest tiles of at most kUnitRows tokens, of equal size but
        // the last, times the most heads of the group that still fit kUnitRows
        // rows; units of more than 16 rows run on the two-tile kernel
        if ((v != PKV_VARIANT_TENSOR_CORES && v != PKV_VARIANT_TCGEN05) ||
            n_queries > kMaxQueries)
            return PKV_ERR_UNSUPPORTED;
        // tcgen05: one tile of up to 64 rows (N of the transposed products)
        const int kUnitRows = v == PKV_VARIANT_TCGEN05 ? 64 : 32;
        const int t0 = (n_queries + kUnitRows - 1) / kUnitRows;
        const int qpu = (n_queries + t0 - 1) / t0;
        const int tiles = (n_queries + qpu - 1) / qpu;
        int hpu = 1;
        for (int d = 1; d <= s->group; ++d)
            if (s->group % d == 0 && qpu * d <= kUnitRows) hpu = d;
        const int rows = qpu * hpu;
        if (v == PKV_VARIANT_TCGEN05)
            s->gs = rows <= 16 ? 16 : (rows <= 32 ? 32 : 64);  // N of the tile
        else
            s->gs = rows > 16 ? 32 : rows;
        s->sub_groups = (s->group / hpu) * tiles;
        s->rs = pkv::RowShape{n_queries, qpu, hpu, s->group / hpu, s->group, n_q_heads};
    } else if (v == PKV_VARIANT_TCGEN05) {
        return PKV_ERR_UNSUPPORTED;  // one query per sequence: the warp kernels
    } else if (force_gs > 0) {  // a sub-group size chosen by the caller (divides the group)
        if (force_gs > max_gs || s->group % force_gs) return PKV_ERR_UNSUPPORTED;
        s->gs = force_gs;
        s->sub_groups = s->group / force_gs;
    } else if (!split_group(s->group, max_gs, &s->sub_groups, &s->gs)) {
        return PKV_ERR_UNSUPPORTED;
    }
    if (n_queries <= 1) s->rs = pkv::RowShape{1, 1, s->gs, s->sub_groups, s->group, n_q_heads};
    s->units_per_b = n_kv_heads * s->sub_groups;
    s->units = (long long)batch * s->units_per_b;
    s->kernel = pick_kernel(dtype, head_dim, v, s->gs);
    if (!s->kernel.fn()) return PKV_ERR_UNSUPPORTED;
    st = prepare_kernel(s->kernel, &s->workers_auto);
    if (st != PKV_OK) return st;
    s->workers = num_workers > 0 ? num_workers : s->workers_auto;
    s->ws = ws_layout(batch, s->units, s->gs, head_dim, s->workers);
    return PKV_OK;
}

pkv_status check_workspace(const void* workspace, size_t ws_bytes, const DecodeSetup& s) {
    if (!workspace) return PKV_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PKV_ERR_WORKSPACE;
    if (ws_bytes < s.ws.total) return PKV_ERR_WORKSPACE;
    return PKV_OK;
}

// --- tensor maps of the pools (tensor-core variant) ------------------------
// A pool [NP][Hkv][P][D] is seen as a 2-D tensor of NP*Hkv*P rows of D
// elements; a box is 16 rows x 64 elements (128 bytes) with the 128-byte
// swizzle.  Encoded through the driver entry point (no libcuda link), cached
// per (address, rows, D, dtype).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

std::mutex g_map_mu;
std::map<std::tuple<const void*, long long, int, int, int>, CUtensorMap> g_maps;

// box_rows: rows of one box (16: a chunk of the pool; 128: a tensor-core row
// tile of gathered query rows)
pkv_status pool_map(const void* pool, long long rows, int head_dim, pkv_dtype dtype,
                    CUtensorMap* out, int box_rows = pkv::kChunk) {
    const auto key = std::make_tuple(pool, rows, head_dim, (int)dtype, box_rows);
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto it = g_maps.find(key);
        if (it != g_maps.end()) {
            *out = it->second;
            return PKV_OK;
        }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return PKV_ERR_CUDA;
    CUtensorMap m;
    memset(&m, 0, sizeof(m));
    const cuuint64_t dims[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)head_dim * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt =
        dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (fn(&m, dt, 2, const_cast<void*>(pool), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_maps.size() > 256) g_maps.clear();
    g_maps[key] = m;
    *out = m;
    return PKV_OK;
}

// q [B][Hq][D] as a 3-D tensor (D, Hq, B) whose box is 64 elements x `group`
// heads x tile_rows / group sequences: the rows of one shared-prefix tile of
// a KV head in sequence-major order (128-byte swizzle).  Cached like the
// pool maps.
std::map<std::tuple<const void*, int, int, int, int, int, int>, CUtensorMap> g_qmaps;

pkv_status q_tile_map(const void* q, int batch, int n_q_heads, int head_dim, pkv_dtype dtype,
                      int group, int tile_rows, CUtensorMap* out) {
    const auto key = std::make_tuple(q, batch, n_q_heads, head_dim, (int)dtype, group, tile_rows);
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto it = g_qmaps.find(key);
        if (it != g_qmaps.end()) {
            *out = it->second;
            return PKV_OK;
        }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return PKV_ERR_CUDA;
    CUtensorMap m;
    memset(&m, 0, sizeof(m));
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)n_q_heads, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)n_q_heads * head_dim * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)(tile_rows / group)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (fn(&m, dt, 3, const_cast<void*>(q), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_qmaps.size() > 256) g_qmaps.clear();
    g_qmaps[key] = m;
    *out = m;
    return PKV_OK;
}

// The shared-prefix pass's partial slots (128 * D + 256 floats each; o is the
// first 128 * D) as a 3-D fp32 tensor (D, 128 rows, slots) with boxes of 32
// floats x 128 rows x 1 slot (128-byte swizzle), for the pass's tensor stores.
std::map<std::tuple<const void*, int, long long>, CUtensorMap> g_omaps;

pkv_status prefix_slots_map(void* partials, int head_dim, long long slots, CUtensorMap* out) {
    const auto key = std::make_tuple((const void*)partials, head_dim, slots);
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto it = g_omaps.find(key);
        if (it != g_omaps.end()) {
            *out = it->second;
            return PKV_OK;
        }
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return PKV_ERR_CUDA;
    CUtensorMap m;
    memset(&m, 0, sizeof(m));
    const int rows = pkv::kPrefixTileRows;
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)rows, (cuuint64_t)slots};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 4,
                                   (cuuint64_t)(rows * (head_dim + 2)) * 4};
    const cuuint32_t box[3] = {32, (cuuint32_t)rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, partials, dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_omaps.size() > 256) g_omaps.clear();
    g_omaps[key] = m;
    *out = m;
    return PKV_OK;
}

// The plan inputs of one decode.  skip_cols: the decoded range starts
// skip_cols table columns into each row (table points at that column) and the
// lengths count from the row's start; uniform_len >= 0: every sequence has
// this length and context_lens is not read.
pkv::PlanArgs plan_args(const int32_t* context_lens, const int32_t* table, int batch,
                        int page_size, int table_stride, int num_workers, void* workspace,
                        const DecodeSetup& s, int skip_cols = 0, int uniform_len = -1) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    pkv::PlanArgs pa = {};  // lens_host = 0: device lengths
    pa.lens = context_lens;
    pa.len_offset = skip_cols * page_size;
    pa.uniform_len = uniform_len;
    pa.batch = batch;
    pa.units_per_b = s.units_per_b;
    pa.cap = (long long)(table_stride - skip_cols) * page_size;
    pa.workers_req = num_workers > 0 ? s.workers : 0;
    pa.workers_auto = s.workers_auto;
    pa.min_chunks = kMinChunksPerWorker;
    pa.lens_eff = reinterpret_cast<int32_t*>(ws + s.ws.lens_eff);
    pa.prefix = reinterpret_cast<int32_t*>(ws + s.ws.prefix);
    pa.wstart = reinterpret_cast<int32_t*>(ws + s.ws.wstart);
    pa.hdr = reinterpret_cast<WsHeader*>(ws);
    pa.unit_done = reinterpret_cast<int32_t*>(ws + s.ws.unit_done);
    pa.units = s.units;
    pa.table = table;
    pa.table_stride = table_stride;
    pa.page_size = page_size;
    return pa;
}

pkv_status do_plan(const int32_t* context_lens, const int32_t* table, int batch, int page_size,
                   int table_stride, int num_workers, void* workspace, const DecodeSetup& s,
                   const pkv::AppendArgs* append, cudaStream_t stream) {
    return cuda_status(pkv::launch_plan(plan_args(context_lens, table, batch, page_size,
                                                  table_stride, num_workers, workspace, s),
                                        append, stream));
}

pkv_status do_run(const void* q, const void* k_pool, const void* v_pool, const int32_t* table,
                  int table_stride, int batch, int n_q_heads, int n_kv_heads, int head_dim,
                  int page_size, int num_pages, pkv_dtype dtype, float scale, void* out,
                  void* workspace, const DecodeSetup& s, bool merge, cudaStream_t stream,
                  bool all_partials = false, uint32_t* status = nullptr) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    pkv::DecodeParams p;
    p.q = q;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.table = table;
    p.lens_eff = reinterpret_cast<const int32_t*>(ws + s.ws.lens_eff);
    p.prefix = reinterpret_cast<const int32_t*>(ws + s.ws.prefix);
    p.wstart = reinterpret_cast<const int32_t*>(ws + s.ws.wstart);
    p.units = (int)s.units;
    p.hdr = reinterpret_cast<const WsHeader*>(ws);
    p.status = status ? status : &reinterpret_cast<WsHeader*>(ws)->status;
    p.partials = reinterpret_cast<float*>(ws + s.ws.partials);
    p.unit_done = merge ? reinterpret_cast<int32_t*>(ws + s.ws.unit_done) : nullptr;
    p.all_partials = all_partials ? 1 : 0;
    p.rows = s.rs;
    p.out = out;
    p.table_stride = table_stride;
    p.batch = batch;
    p.n_q_heads = n_q_heads;
    p.n_kv_heads = n_kv_heads;
    p.page_size = page_size;
    p.num_pages = num_pages;
    p.group = s.group;
    p.sub_groups = s.sub_groups;
    p.scale_log2 = scale * 1.4426950408889634f;
    const int blocks = (s.workers + s.kernel.warps() - 1) / s.kernel.warps();
    if (s.kernel.variant == PKV_VARIANT_TCGEN05) {
        const long long rows = (long long)num_pages * n_kv_heads * page_size;
        if (rows > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;  // 32-bit tensor row coordinate
        const pkv::RowShape& rs = s.rs;
        if ((long long)batch * rs.n_queries > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
        // q [B * n_queries][Hq][D]: a box is one unit's rows (queries_per_unit
        // tokens x heads_per_unit heads, token-major)
        CUtensorMap qm, km, vm;
        pkv_status st = q_tile_map(q, batch * rs.n_queries, n_q_heads, head_dim, dtype,
                                   rs.heads_per_unit, rs.heads_per_unit * rs.queries_per_unit,
                                   &qm);
        if (st == PKV_OK) st = pool_map(k_pool, rows, head_dim, dtype, &km);
        if (st == PKV_OK) st = pool_map(v_pool, rows, head_dim, dtype, &vm);
        if (st != PKV_OK) return st;
        if (merge || all_partials) return PKV_ERR_UNSUPPORTED;  // the combine kernel merges
        return cuda_status(pkv::launch_pdl(s.kernel.um.fn, dim3(blocks), dim3(s.kernel.um.threads),
                                           s.kernel.um.smem_bytes, stream, p, qm, km, vm));
    }
    if (s.kernel.variant == PKV_VARIANT_TENSOR_CORES) {
        const long long rows = (long long)num_pages * n_kv_heads * page_size;
        if (rows > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;  // 32-bit tensor row coordinate
        CUtensorMap km, vm;
        pkv_status st = pool_map(k_pool, rows, head_dim, dtype, &km);
        if (st == PKV_OK) st = pool_map(v_pool, rows, head_dim, dtype, &vm);
        if (st != PKV_OK) return st;
        return cuda_status(pkv::launch_pdl(s.kernel.mma.fn, dim3(blocks),
                                           dim3(s.kernel.mma.warps * 32), s.kernel.mma.smem_bytes,
                                           stream, p, km, vm));
    }
    return cuda_status(pkv::launch_pdl(s.kernel.cc.fn, dim3(blocks), dim3(s.kernel.cc.warps * 32),
                                       s.kernel.cc.smem_bytes, stream, p));
}

pkv_status do_combine(int batch, int n_q_heads, int head_dim, pkv_dtype dtype, void* out,
                      void* workspace, const DecodeSetup& s, cudaStream_t stream) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (batch == 0) return PKV_OK;
    return cuda_status(pkv::launch_combine(
        dtype, head_dim, reinterpret_cast<const float*>(ws + s.ws.partials),
        reinterpret_cast<const int32_t*>(ws + s.ws.prefix),
        reinterpret_cast<const int32_t*>(ws + s.ws.lens_eff), reinterpret_cast<const WsHeader*>(ws),
        out, (int)s.units, s.units_per_b, s.sub_groups, s.gs, s.rs, s.workers, stream));
}

// --- fixed device scratch for paged_decode_attention_no_alloc -------------
// Callers that may not allocate device memory (see pagedkv.h) get the
// decode workspace from this file-scope array.  In host code the symbol is
// only a host-side stand-in, so its device address is looked up once per
// device with cudaGetSymbolAddress (with that device current) and cached.
static __device__ __align__(256) uint8_t g_no_alloc_scratch[PKV_NO_ALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

pkv_status no_alloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_no_alloc_scratch) != cudaSuccess || !p) return PKV_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return PKV_OK;
}

pkv::AppendArgs make_append(const void* k_new, const void* v_new, const int32_t* positions,
                            const int32_t* table, int table_stride, void* k_pool, void* v_pool,
                            int n_kv_heads, int head_dim, int page_size, int num_pages) {
    pkv::AppendArgs a = {};  // host = 0: device inputs
    a.k_new = static_cast<const uint4*>(k_new);
    a.v_new = static_cast<const uint4*>(v_new);
    a.positions = positions;
    a.table = table;
    a.table_stride = table_stride;
    a.k_pool = static_cast<uint4*>(k_pool);
    a.v_pool = static_cast<uint4*>(v_pool);
    a.n_kv_heads = n_kv_heads;
    a.vecs = head_dim / 8;
    a.page_size = page_size;
    a.num_pages = num_pages;
    a.q_in = nullptr;  // no rotary embedding unless the caller sets it up
    a.q_norm_w = nullptr;
    a.k_norm_w = nullptr;
    a.norm_eps = 0.f;
    a.q_out = nullptr;
    a.n_q_heads = 0;
    a.bf16 = 0;
    return a;
}

// The rotary angles per position unit, theta^(-2i/D) for i < D/2, in double
// (the kernel multiplies them by each token's position).
// Norm weights (nullable, 2-byte aligned, head_dim elements) and eps of the
// optional per-head RMS norm before the rotation.
bool norm_args_ok(const void* q_norm_weight, const void* k_norm_weight, float norm_eps) {
    if ((reinterpret_cast<uintptr_t>(q_norm_weight) & 1u) ||
        (reinterpret_cast<uintptr_t>(k_norm_weight) & 1u))
        return false;
    return !(q_norm_weight || k_norm_weight) || (norm_eps >= 0.f && isfinite(norm_eps));
}

pkv_status set_norm(pkv::AppendArgs* a, const void* q_norm_weight, const void* k_norm_weight,
                    float norm_eps) {
    if (!norm_args_ok(q_norm_weight, k_norm_weight, norm_eps)) return PKV_ERR_INVALID_ARG;
    a->q_norm_w = q_norm_weight;
    a->k_norm_w = k_norm_weight;
    a->norm_eps = norm_eps;
    return PKV_OK;
}

void set_inv_freq(pkv::AppendArgs* a, double theta, int head_dim) {
    for (int i = 0; i < 64; ++i)
        a->inv_freq[i] = i < head_dim / 2 ? pow(theta, -2.0 * i / head_dim) : 0.0;
}

// Host-only argument checks of a decode call (no CUDA call is made), in the
// order: shapes, scalars, pointers, alignment, aliasing of out.
pkv_status validate_decode_args(const void* q, const void* k_pool, const void* v_pool,
                                const int32_t* page_table, int table_stride,
                                const int32_t* context_lens, bool need_lens, int batch,
                                int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                                int num_pages, pkv_dtype dtype, float scale, const void* out,
                                const void* workspace, size_t ws_bytes, int num_workers,
                                int variant) {
    pkv_status st = check_shapes(batch, n_q_heads, n_kv_heads, head_dim, page_size);
    if (st != PKV_OK) return st;
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if (num_pages <= 0 || table_stride <= 0 || num_workers < 0 || !valid_variant(variant))
        return PKV_ERR_INVALID_ARG;
    if (!isfinite(scale)) return PKV_ERR_INVALID_ARG;
    if (batch == 0) return PKV_OK;
    if (!q || !k_pool || !v_pool || !page_table || !out || (need_lens && !context_lens))
        return PKV_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PKV_ERR_WORKSPACE;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return PKV_ERR_INVALID_ARG;
    const size_t qo_bytes = (size_t)batch * n_q_heads * head_dim * 2;
    const size_t pool_bytes = (size_t)num_pages * n_kv_heads * page_size * head_dim * 2;
    const size_t table_bytes = (size_t)batch * table_stride * 4;
    if (overlaps(out, qo_bytes, q, qo_bytes) || overlaps(out, qo_bytes, k_pool, pool_bytes) ||
        overlaps(out, qo_bytes, v_pool, pool_bytes) ||
        overlaps(out, qo_bytes, page_table, table_bytes) ||
        (need_lens && overlaps(out, qo_bytes, context_lens, (size_t)batch * 4)) ||
        overlaps(out, qo_bytes, workspace, ws_bytes))
        return PKV_ERR_ALIAS;
    return PKV_OK;
}

}  // namespace

extern "C" {

const char* pkv_status_string(pkv_status s) {
    switch (s) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PKV_ERR_ALIAS: return "output overlaps an input";
        case PKV_ERR_OUT_OF_PAGES: return "not enough free pages";
        case PKV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case PKV_ERR_CUDA: return "CUDA runtime error";
        case PKV_ERR_DEVICE_CHECK: return "device status reports skipped input";
        case PKV_ERR_REFCOUNT: return "page reference count error";
    }
    return "unknown status";
}

int pkv_version(void) { return 200; }

pkv_status pkv_check_bounded_wait(uint32_t tries, uint32_t* status, unsigned long long* elapsed_ns,
                                  pkv_stream stream) {
    if (!status || tries == 0) return PKV_ERR_INVALID_ARG;
    return cuda_status(pkv::launch_wait_check(tries, status, elapsed_ns,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status kv_append(const pkv_pool* pool, const void* k_new, const void* v_new,
                     const int32_t* page_table, int table_stride, const int32_t* positions,
                     int batch, uint32_t* dev_status, pkv_stream stream) {
    if (!pool || batch < 0 || table_stride <= 0) return PKV_ERR_INVALID_ARG;
    if (batch == 0) return PKV_OK;
    if (!k_new || !v_new || !page_table || !positions) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(pool->k) || !aligned16(pool->v))
        return PKV_ERR_INVALID_ARG;
    const size_t pool_bytes =
        (size_t)pool->num_pages * pool->n_kv_heads * pool->page_size * pool->head_dim * 2;
    const size_t row_bytes = (size_t)batch * pool->n_kv_heads * pool->head_dim * 2;
    if (overlaps(k_new, row_bytes, pool->k, pool_bytes) ||
        overlaps(k_new, row_bytes, pool->v, pool_bytes) ||
        overlaps(v_new, row_bytes, pool->k, pool_bytes) ||
        overlaps(v_new, row_bytes, pool->v, pool_bytes))
        return PKV_ERR_ALIAS;
    const pkv::AppendArgs a = make_append(k_new, v_new, positions, page_table, table_stride,
                                          pool->k, pool->v, pool->n_kv_heads, pool->head_dim,
                                          pool->page_size, pool->num_pages);
    return cuda_status(pkv::launch_append(a, batch, dev_status,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status kv_append_rope(const pkv_pool* pool, const void* q, const void* k_new,
                          const void* v_new, const int32_t* page_table, int table_stride,
                          const int32_t* positions, int batch, int n_q_heads, double rope_theta,
                          const void* q_norm_weight, const void* k_norm_weight, float norm_eps,
                          void* q_out, uint32_t* dev_status, pkv_stream stream) {
    if (!pool || batch < 0 || table_stride <= 0 || n_q_heads <= 0) return PKV_ERR_INVALID_ARG;
    if (!(rope_theta > 0.0 && isfinite(rope_theta))) return PKV_ERR_INVALID_ARG;
    if (!norm_args_ok(q_norm_weight, k_norm_weight, norm_eps)) return PKV_ERR_INVALID_ARG;
    if (batch == 0) return PKV_OK;
    if (!q || !q_out || !k_new || !v_new || !page_table || !positions) return PKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(q_out) || !aligned16(k_new) || !aligned16(v_new))
        return PKV_ERR_INVALID_ARG;
    const size_t pool_bytes =
        (size_t)pool->num_pages * pool->n_kv_heads * pool->page_size * pool->head_dim * 2;
    const size_t row_bytes = (size_t)batch * pool->n_kv_heads * pool->head_dim * 2;
    const size_t q_bytes = (size_t)batch * n_q_heads * pool->head_dim * 2;
    const void* ins[3] = {q, k_new, v_new};
    const size_t in_bytes[3] = {q_bytes, row_bytes, row_bytes};
    for (int i = 0; i < 3; ++i)
        if (overlaps(ins[i], in_bytes[i], pool->k, pool_bytes) ||
            overlaps(ins[i], in_bytes[i], pool->v, pool_bytes))
            return PKV_ERR_ALIAS;
    // q_out may be q itself (each element is read before it is written), but no
    // other overlap
    if ((q_out != q && overlaps(q_out, q_bytes, q, q_bytes)) ||
        overlaps(q_out, q_bytes, k_new, row_bytes) || overlaps(q_out, q_bytes, v_new, row_bytes) ||
        overlaps(q_out, q_bytes, pool->k, pool_bytes) ||
        overlaps(q_out, q_bytes, pool->v, pool_bytes))
        return PKV_ERR_ALIAS;
    pkv::AppendArgs a = make_append(k_new, v_new, positions, page_table, table_stride, pool->k,
                                    pool->v, pool->n_kv_heads, pool->head_dim, pool->page_size,
                                    pool->num_pages);
    a.q_in = static_cast<const uint4*>(q);
    a.q_out = static_cast<uint4*>(q_out);
    a.n_q_heads = n_q_heads;
    set_inv_freq(&a, rope_theta, pool->head_dim);
    a.bf16 = pool->dtype == PKV_BF16;
    if (set_norm(&a, q_norm_weight, k_norm_weight, norm_eps) != PKV_OK) return PKV_ERR_INVALID_ARG;
    return cuda_status(pkv::launch_rope_append(a, batch, pool->head_dim, dev_status,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status kv_gather(const pkv_pool* pool, const int32_t* page_table, int table_stride,
                     const int32_t* context_lens, int batch, int max_len, void* k_out,
                     void* v_out, uint32_t* dev_status, pkv_stream stream) {
    if (!pool || batch < 0 || max_len < 0 || table_stride <= 0) return PKV_ERR_INVALID_ARG;
    if (batch == 0 || max_len == 0) return PKV_OK;
    if (batch > 65535 || pool->n_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
    if (!page_table || !context_lens || !k_out || !v_out) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_out) || !aligned16(v_out)) return PKV_ERR_INVALID_ARG;
    const size_t pool_bytes =
        (size_t)pool->num_pages * pool->n_kv_heads * pool->page_size * pool->head_dim * 2;
    const size_t out_bytes = (size_t)batch * pool->n_kv_heads * max_len * pool->head_dim * 2;
    if (overlaps(k_out, out_bytes, pool->k, pool_bytes) ||
        overlaps(k_out, out_bytes, pool->v, pool_bytes) ||
        overlaps(v_out, out_bytes, pool->k, pool_bytes) ||
        overlaps(v_out, out_bytes, pool->v, pool_bytes) ||
        overlaps(k_out, out_bytes, v_out, out_bytes))
        return PKV_ERR_ALIAS;
    return cuda_status(pkv::launch_gather(pool->k, pool->v, page_table, table_stride, context_lens,
                                          batch, pool->n_kv_heads, pool->head_dim, pool->page_size,
                                          pool->num_pages, max_len, k_out, v_out, dev_status,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

pkv_status paged_decode_workspace_size(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                       int num_workers, pkv_decode_variant variant,
                                       size_t* bytes) {
    if (!bytes) return PKV_ERR_INVALID_ARG;
    *bytes = 0;
    pkv_status st = check_shapes(batch, n_q_heads, n_kv_heads, head_dim, 16);
    if (st != PKV_OK) return st;
    if (num_workers < 0 || !valid_variant(variant)) return PKV_ERR_INVALID_ARG;
    DecodeSetup s;
    if ((st = setup_decode(batch, n_q_heads, n_kv_heads, head_dim, 16, PKV_BF16, num_workers,
                           variant, &s)) != PKV_OK)
        return st;
    *bytes = s.ws.total;
    return PKV_OK;
}

pkv_status paged_decode_plan(const int32_t* context_lens, int batch, int n_q_heads,
                             int n_kv_heads, int head_dim, int page_size, int table_stride,
                             int num_workers, pkv_decode_variant variant, void* workspace,
                             size_t ws_bytes, pkv_stream stream) {
    pkv_status st = check_shapes(batch, n_q_heads, n_kv_heads, head_dim, page_size);
    if (st != PKV_OK) return st;
    if (table_stride <= 0 || num_workers < 0 || !valid_variant(variant))
        return PKV_ERR_INVALID_ARG;
    if (batch == 0) return PKV_OK;
    if (!context_lens) return PKV_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PKV_ERR_WORKSPACE;
    DecodeSetup s;
    if ((st = setup_decode(batch, n_q_heads, n_kv_heads, head_dim, page_size, PKV_BF16,
                           num_workers, variant, &s)) != PKV_OK)
        return st;
    if ((st = check_workspace(workspace, ws_bytes, s)) != PKV_OK) return st;
    return do_plan(context_lens, nullptr, batch, page_size, table_stride, num_workers,
                   workspace, s, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

pkv_status paged_decode_run(const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* page_table, int table_stride, int batch,
                            int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                            int num_pages, pkv_dtype dtype, float scale, void* out,
                            void* workspace, size_t ws_bytes, int num_workers,
                            pkv_decode_variant variant, int merge, pkv_stream stream) {
    pkv_status st = validate_decode_args(q, k_pool, v_pool, page_table, table_stride, nullptr,
                                         false, batch, n_q_heads, n_kv_heads, head_dim,
                                         page_size, num_pages, dtype, scale, out, workspace,
                                         ws_bytes, num_workers, variant);
    if (st != PKV_OK) return st;
    if (merge != 0 && merge != 1) return PKV_ERR_INVALID_ARG;
    if (batch == 0) return PKV_OK;
    DecodeSetup s;
    if ((st = setup_decode(batch, n_q_heads, n_kv_heads, head_dim, page_size, dtype, num_workers,
                           variant, &s)) != PKV_OK)
        return st;
    if ((st = check_workspace(workspace, ws_bytes, s)) != PKV_OK) return st;
    return do_run(q, k_pool, v_pool, page_table, table_stride, batch, n_q_heads, n_kv_heads,
                  head_dim, page_size, num_pages, dtype, scale, out, workspace, s, merge != 0,
                  reinterpret_cast<cudaStream_t>(stream));
}

pkv_status paged_decode_combine(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                pkv_dtype dtype, void* out, void* workspace, size_t ws_bytes,
                                int num_workers, pkv_decode_variant variant, pkv_stream stream) {
    pkv_status st = check_shapes(batch, n_q_heads, n_kv_heads, head_dim, 16);
    if (st != PKV_OK) return st;
    if ((dtype != PKV_F16 && dtype != PKV_BF16) || num_workers < 0 || !valid_variant(variant))
        return PKV_ERR_INVALID_ARG;
    if (batch == 0) return PKV_OK;
    if (!out || !aligned16(out)) return PKV_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PKV_ERR_WORKSPACE;
    if (overlaps(out, (size_t)batch * n_q_heads * head_dim * 2, workspace, ws_bytes))
        return PKV_ERR_ALIAS;
    DecodeSetup s;
    if ((st = setup_decode(batch, n_q_heads, n_kv_heads, head_dim, 16, dtype, num_workers,
                           variant, &s)) != PKV_OK)
        return st;
    if ((st = check_workspace(workspace, ws_bytes, s)) != PKV_OK) return st;
    return do_combine(batch, n_q_heads, head_dim, dtype, out, workspace, s,
                      reinterpret_cast<cudaStream_t>(stream));
}

pkv_status paged_decode_attention(const void* q, const void* k_pool, const void* v_pool,
                                  const int32_t* page_table, int table_stride,
                                  const int32_t* context_lens, int batch, int n_q_heads,
                                  int n_kv_heads, int head_dim, int page_size, int num_pages,
                                  pkv_dtype dtype, float scale, void* out, void* workspace,
                                  size_t ws_bytes, int num_workers, pkv_decode_variant variant,
                                  pkv_stream stream) {
    pkv_status st = validate_decode_args(q, k_pool, v_pool, page_table, table_stride,
                                         context_lens, true, batch, n_q_heads, n_kv_heads,
                                         head_dim, page_size, num_pages, dtype, scale, out,
                                         workspace, ws_bytes, num_workers, variant);
    if (st != PKV_OK || batch == 0) return st;
    DecodeSetup s;
    if ((st = setup_decode(batch, n_q_heads, n_kv_heads, head_dim, page_size, dtype, num_workers,
                           variant, &s)) != PKV_OK)
        return st;
    if ((st = check_workspace(workspace, ws_bytes, s)) != PKV_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if ((st = do_plan(context_lens, page_table, batch, page_size, table_stride, num_workers,
                      workspace, s, nullptr, cs)) != PKV_OK)
        return st;
    if ((st = do_run(q, k_pool, v_pool, page_table, table_stride, batch, n_q_heads, n_kv_heads,
                     head_dim, page_size, num_pages, dtype, scale, out, workspace, s, false, cs)) !=
        PKV_OK)
        return st;
    return do_combine(batch, n_q_heads, head_dim, dtype, out, workspace, s, cs);
}

}  // extern "C" (reopened below)

namespace {
// One decode step; rope: the rotary embedding of q and k_new (angle base
// rope_theta) runs in the append CTAs, and the rotated q goes through `out`.
pkv_status step_impl(const void* k_new, const void* v_new, const int32_t* positions,
                     const void* q, void* k_pool, void* v_pool, const int32_t* page_table,
                     int table_stride, const int32_t* context_lens, int batch, int n_q_heads,
                     int n_kv_heads, int head_dim, int page_size, int num_pages, pkv_dtype dtype,
                     float scale, bool rope, double rope_theta, const void* q_norm_weight,
                     const void* k_norm_weight, float norm_eps, void* out, void* workspace,
                     size_t ws_bytes, int num_workers, pkv_decode_variant variant,
                     pkv_stream stream) {
    if (rope && !(rope_theta > 0.0 && isfinite(rope_theta))) return PKV_ERR_INVALID_ARG;
    if (rope && !norm_args_ok(q_norm_weight, k_norm_weight, norm_eps)) return PKV_ERR_INVALID_ARG;
    pkv_status st = validate_decode_args(q, k_pool, v_pool, page_table, table_stride,
                                         context_lens, true, batch, n_q_heads, n_kv_heads,
                                         head_dim, page_size, num_pages, dtype, scale, out,
                                         workspace, ws_bytes, num_workers, variant);
    if (st != PKV_OK || batch == 0) return st;
    if (!k_new || !v_new || !positions) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_INVALID_ARG;
    const size_t pool_bytes = (size_t)num_pages * n_kv_heads * page_size * head_dim * 2;
    const size_t row_bytes = (size_t)batch * n_kv_heads * head_dim * 2;
    const size_t qo_bytes = (size_t)batch * n_q_heads * head_dim * 2;
    if (overlaps(k_new, row_bytes, k_pool, pool_bytes) ||
        overlaps(k_new, row_bytes, v_pool, pool_bytes) ||
        overlaps(v_new, row_bytes, k_pool, pool_bytes) ||
        overlaps(v_new, row_bytes, v_pool, pool_bytes) ||
        overlaps(out, qo_bytes, k_new, row_bytes) || overlaps(out, qo_bytes, v_new, row_bytes))
        return PKV_ERR_ALIAS;
    DecodeSetup s;
    if ((st = setup_decode(batch, n_q_heads, n_kv_heads, head_dim, page_size, dtype, num_workers,
                           variant, &s)) != PKV_OK)
        return st;
    if ((st = check_workspace(workspace, ws_bytes, s)) != PKV_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    pkv::AppendArgs a = make_append(k_new, v_new, positions, page_table, table_stride, k_pool,
                                    v_pool, n_kv_heads, head_dim, page_size, num_pages);
    if (rope) {
        a.q_in = static_cast<const uint4*>(q);
        a.q_out = static_cast<uint4*>(out);  // the decode reads the rotated q from here
        a.n_q_heads = n_q_heads;
        set_inv_freq(&a, rope_theta, head_dim);
        a.bf16 = dtype == PKV_BF16;
        if ((st = set_norm(&a, q_norm_weight, k_norm_weight, norm_eps)) != PKV_OK) return st;
    }
    if ((st = do_plan(context_lens, page_table, batch, page_size, table_stride, num_workers,
                      workspace, s, &a, cs)) != PKV_OK)
        return st;
    if ((st = do_run(rope ? out : q, k_pool, v_pool, page_table, table_stride, batch, n_q_heads,
                     n_kv_heads, head_dim, page_size, num_pages, dtype, scale, out, workspace, s,
                     false, cs)) != PKV_OK)
        return st;
    return do_combine(batch, n_q_heads, head_dim, dtype, out, workspace, s, cs);
}
}  // namespace

extern "C" {

pkv_status paged_decode_step(const void* k_new, const void* v_new, const int32_t* positions,
                             const void* q, void* k_pool, void* v_pool,
                             const int32_t* page_table, int table_stride,
                             const int32_t* context_lens, int batch, int n_q_heads,
                             int n_kv_heads, int head_dim, int page_size, int num_pages,
                             pkv_dtype dtype, float scale, void* out, void* workspace,
                             size_t ws_bytes, int num_workers, pkv_decode_variant variant,
                             pkv_stream stream) {
    return step_impl(k_new, v_new, positions, q, k_pool, v_pool, page_table, table_stride,
                     context_lens, batch, n_q_heads, n_kv_heads, head_dim, page_size, num_pages,
                     dtype, scale, false, 0.0, nullptr, nullptr, 0.f, out, workspace, ws_bytes,
                     num_workers, variant, stream);
}

pkv_status paged_decode_step_rope(const void* k_new, const void* v_new, const int32_t* positions,
                                  const void* q, void* k_pool, void* v_pool,
                                  const int32_t* page_table, int table_stride,
                                  const int32_t* context_lens, int batch, int n_q_heads,
                                  int n_kv_heads, int head_dim, int page_size, int num_pages,
                                  pkv_dtype dtype, float scale, double rope_theta,
                                  const void* q_norm_weight, const void* k_norm_weight,
                                  float norm_eps, void* out, void* workspace, size_t ws_bytes,
                                  int num_workers, pkv_decode_variant variant,
                                  pkv_stream stream) {
    return step_impl(k_new, v_new, positions, q, k_pool, v_pool, page_table, table_stride,
                     context_lens, batch, n_q_heads, n_kv_heads, head_dim, page_size, num_pages,
                     dtype, scale, true, rope_theta, q_norm_weight, k_norm_weight, norm_eps, out,
                     workspace, ws_bytes, num_workers, variant, stream);
}

}  // extern "C" (reopened below)

namespace {
// The device address of [p, p + bytes) in page-locked host memory (under
// unified addressing the same number).  Its first and its last byte must both
// be page-locked host memory mapped for the current device, the last at
// distance bytes - 1 from the first; else INVALID_ARG and nothing launches.
pkv_status host_range(const void* p, size_t bytes, const void** dev) {
    if (!p) return PKV_ERR_INVALID_ARG;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_INVALID_ARG;
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer) return PKV_ERR_INVALID_ARG;
    if (bytes > 1) {
        cudaPointerAttributes e;
        const char* last = static_cast<const char*>(p) + (bytes - 1);
        if (cudaPointerGetAttributes(&e, last) != cudaSuccess) {
            cudaGetLastError();
            return PKV_ERR_INVALID_ARG;
        }
        if (e.type != cudaMemoryTypeHost ||
            static_cast<const char*>(e.devicePointer) !=
                static_cast<const char*>(a.devicePointer) + (bytes - 1))
            return PKV_ERR_INVALID_ARG;
    }
    *dev = a.devicePointer;
    return PKV_OK;
}

// Workspace of a host-buffer step: the decode's own, then the device copies
// of q and of the page table (each from a 256-byte boundary).
struct HostStepLayout {
    size_t q, table, total;
};

HostStepLayout host_step_layout(const DecodeSetup& s, int batch, int n_q_heads, int head_dim,
                                int table_stride) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    HostStepLayout l;
    l.q = up(s.ws.total);
    l.table = l.q + up((size_t)batch * n_q_heads * head_dim * 2);
    l.total = l.table + up((size_t)batch * table_stride * 4);
    return l;
}
}  // namespace

extern "C" {

pkv_status paged_decode_step_host_workspace_size(int batch, int n_q_heads, int n_kv_heads,
                                                 int head_dim, int table_stride, int num_workers,
                                                 pkv_decode_variant variant, size_t* bytes) {
    if (!bytes) return PKV_ERR_INVALID_ARG;
    *bytes = 0;
    pkv_status st = check_shapes(batch, n_q_heads, n_kv_heads, head_dim, 16);
    if (st != PKV_OK) return st;
    if (table_stride <= 0 || num_workers < 0 || !valid_variant(variant))
        return PKV_ERR_INVALID_ARG;
    DecodeSetup s;
    if ((st = setup_decode(batch, n_q_heads, n_kv_heads, head_dim, 16, PKV_BF16, num_workers,
                           variant, &s)) != PKV_OK)
        return st;
    *bytes = host_step_layout(s, batch, n_q_heads, head_dim, table_stride).total;
    return PKV_OK;
}

pkv_status paged_decode_step_host(const void* k_new, const void* v_new, const int32_t* positions,
                                  const void* q, void* k_pool, void* v_pool,
                                  const int32_t* page_table, int table_stride,
                                  const int32_t* context_lens, int batch, int n_q_heads,
                                  int n_kv_heads, int head_dim, int page_size, int num_pages,
                                  pkv_dtype dtype, float scale, void* out, void* workspace,
                                  size_t ws_bytes, int num_workers, pkv_decode_variant variant,
                                  pkv_stream stream) {
    pkv_status st = validate_decode_args(q, k_pool, v_pool, page_table, table_stride,
                                         context_lens, true, batch, n_q_heads, n_kv_heads,
                                         head_dim, page_size, num_pages, dtype, scale, out,
                                         workspace, ws_bytes, num_workers, variant);
    if (st != PKV_OK || batch == 0) return st;
    if (!k_new || !v_new || !positions) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_INVALID_ARG;
    const size_t row_bytes = (size_t)batch * n_kv_heads * head_dim * 2;
    const size_t qo_bytes = (size_t)batch * n_q_heads * head_dim * 2;
    const size_t table_bytes = (size_t)batch * table_stride * 4;
    const size_t seq_bytes = (size_t)batch * 4;
    if (overlaps(out, qo_bytes, k_new, row_bytes) || overlaps(out, qo_bytes, v_new, row_bytes) ||
        overlaps(out, qo_bytes, positions, seq_bytes))
        return PKV_ERR_ALIAS;
    const void *q_h, *kn_h, *vn_h, *pos_h, *tab_h, *len_h, *out_h;
    if ((st = host_range(q, qo_bytes, &q_h)) != PKV_OK ||
        (st = host_range(k_new, row_bytes, &kn_h)) != PKV_OK ||
        (st = host_range(v_new, row_bytes, &vn_h)) != PKV_OK ||
        (st = host_range(positions, seq_bytes, &pos_h)) != PKV_OK ||
        (st = host_range(page_table, table_bytes, &tab_h)) != PKV_OK ||
        (st = host_range(context_lens, seq_bytes, &len_h)) != PKV_OK ||
        (st = host_range(out, qo_bytes, &out_h)) != PKV_OK)
        return st;
    DecodeSetup s;
    if ((st = setup_decode(batch, n_q_heads, n_kv_heads, head_dim, page_size, dtype, num_workers,
                           variant, &s)) != PKV_OK)
        return st;
    const HostStepLayout hl = host_step_layout(s, batch, n_q_heads, head_dim, table_stride);
    if (ws_bytes < hl.total) return PKV_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* q_dev = ws + hl.q;
    int32_t* table_dev = reinterpret_cast<int32_t*>(ws + hl.table);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // the append reads its inputs from host memory; the staging CTAs copy q
    // and the table next to the decode's workspace; the plan reads the lengths
    pkv::AppendArgs a = make_append(kn_h, vn_h, static_cast<const int32_t*>(pos_h),
                                    static_cast<const int32_t*>(tab_h), table_stride, k_pool,
                                    v_pool, n_kv_heads, head_dim, page_size, num_pages);
    a.host = 1;
    pkv::PlanArgs pa = plan_args(static_cast<const int32_t*>(len_h), nullptr, batch, page_size,
                                 table_stride, num_workers, workspace, s);
    pa.lens_host = 1;
    pkv::StageArgs sa = {};
    sa.q_src = static_cast<const uint4*>(q_h);
    sa.q_dst = static_cast<uint4*>(q_dev);
    sa.q_vecs = (long long)(qo_bytes / 16);
    sa.t_src = static_cast<const int32_t*>(tab_h);
    sa.t_dst = table_dev;
    sa.t_words = (long long)batch * table_stride;
    if ((st = cuda_status(pkv::launch_plan(pa, &a, cs, &sa))) != PKV_OK) return st;
    void* out_dev = const_cast<void*>(out_h);
    if ((st = do_run(q_dev, k_pool, v_pool, table_dev, table_stride, batch, n_q_heads, n_kv_heads,
                     head_dim, page_size, num_pages, dtype, scale, out_dev, workspace, s, false,
                     cs)) != PKV_OK)
        return st;
    return do_combine(batch, n_q_heads, head_dim, dtype, out_dev, workspace, s, cs);
}

pkv_status paged_decode_attention_no_alloc(const void* q, const void* k_pool, const void* v_pool,
                                           const int32_t* page_table, int table_stride,
                                           const int32_t* context_lens, int batch,
                                           int n_q_heads, int n_kv_heads, int head_dim,
                                           int page_size, int num_pages, pkv_dtype dtype,
                                           float scale, void* out, int num_workers,
                                           pkv_decode_variant variant, pkv_stream stream) {
    // shape / pointer / alias checks first (the scratch address is only needed
    // once the call is known to be well formed)
    pkv_status st = check_shapes(batch, n_q_heads, n_kv_heads, head_dim, page_size);
    if (st != PKV_OK) return st;
    if (batch == 0) return PKV_OK;
    void* scratch = nullptr;
    if ((st = no_alloc_scratch(&scratch)) != PKV_OK) return st;
    st = validate_decode_args(q, k_pool, v_pool, page_table, table_stride, context_lens, true,
                              batch, n_q_heads, n_kv_heads, head_dim, page_size, num_pages, dtype,
                              scale, out, scratch, PKV_NO_ALLOC_SCRATCH_BYTES, num_workers,
                              variant);
    if (st != PKV_OK) return st;
    DecodeSetup s;
    if ((st = setup_decode(batch, n_q_heads, n_kv_heads, head_dim, page_size, dtype, num_workers,
                           variant, &s)) != PKV_OK)
        return st;
    // the workspace these shapes need must fit the fixed array
    if (s.ws.total > (size_t)PKV_NO_ALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if ((st = do_plan(context_lens, page_table, batch, page_size, table_stride, num_workers,
                      scratch, s, nullptr, cs)) != PKV_OK)
        return st;
    if ((st = do_run(q, k_pool, v_pool, page_table, table_stride, batch, n_q_heads, n_kv_heads,
                     head_dim, page_size, num_pages, dtype, scale, out, scratch, s, false, cs)) !=
        PKV_OK)
        return st;
    return do_combine(batch, n_q_heads, head_dim, dtype, out, scratch, s, cs);
}

static pkv_status read_status(const void* workspace, uint32_t* status_out) {
    WsHeader h;
    if (cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
        return PKV_ERR_CUDA;
    uint32_t v = h.status;
    const int n = h.append_slots < 0 ? 0
                  : (h.append_slots > pkv::kMaxAppendCtas ? pkv::kMaxAppendCtas
                                                          : h.append_slots);
    for (int i = 0; i < n; ++i) v |= h.append_status[i];
    *status_out = v;
    return v ? PKV_ERR_DEVICE_CHECK : PKV_OK;
}

pkv_status pkv_read_device_status(const void* workspace, uint32_t* status_out) {
    if (!workspace || !status_out) return PKV_ERR_INVALID_ARG;
    return read_status(workspace, status_out);
}

pkv_status pkv_read_no_alloc_status(uint32_t* status_out) {
    if (!status_out) return PKV_ERR_INVALID_ARG;
    void* scratch = nullptr;
    const pkv_status st = no_alloc_scratch(&scratch);
    if (st != PKV_OK) return st;
    return read_status(scratch, status_out);
}

}  // extern "C"

// --- shared-prefix decode (cascade) ----------------------------------------
namespace {
struct PrefixSetup {
    DecodeSetup real, virt;  // suffix pass (real units), prefix pass (virtual units)
    // prefix pass on tensor-core row tiles (tensor-core variant): tiles of
    // tile_rows rows per KV head, up to max_splits ranges of the prefix each
    bool umma = false;
    int tile_rows = 0, tiles = 0, max_splits = 0;
    size_t qv_off, v_off, s_off, total;
};

constexpr int kMaxPrefixSplits = 64;

// Ranges of the prefix per (KV head, row tile): enough tensor-core CTAs for
// one wave over the GPU (dtype < 0: the larger of the two dtypes' counts,
// for sizing a workspace before the dtype is known).
pkv_status prefix_splits(int head_dim, int dtype, long long tiles_total, int* splits) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PKV_ERR_CUDA;
    int per_sm = 0;
    for (int dt = 0; dt < 2; ++dt)
        if (dtype < 0 || dtype == dt) {
            const int n = pkv::prefix_umma_ctas_per_sm((pkv_dtype)dt, head_dim);
            per_sm = n > per_sm ? n : per_sm;
        }
    if (per_sm <= 0) return PKV_ERR_CUDA;
    const long long s = (long long)sms * per_sm / (tiles_total > 0 ? tiles_total : 1);
    *splits = (int)(s < 1 ? 1 : (s > kMaxPrefixSplits ? kMaxPrefixSplits : s));
    return PKV_OK;
}

// The prefix pass: one sequence (the shared prefix) whose every KV head serves
// all B*G query rows of that head.  Tensor-core variant (G <= 128): row tiles
// of up to 128 rows, whole sequences each, on the fifth-generation tensor
// cores.  Otherwise a virtual decode in sub-groups of gs_v rows, gs_v a
// multiple of the real sub-group size.  dtype < 0: size for either dtype.
pkv_status setup_prefix(int batch, int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                        int dtype, int num_workers, int variant, PrefixSetup* ps) {
    pkv_status st = setup_decode(batch, n_q_heads, n_kv_heads, head_dim, page_size,
                                 dtype < 0 ? PKV_BF16 : (pkv_dtype)dtype, num_workers, variant,
                                 &ps->real);
    if (st != PKV_OK) return st;
    const long long group_v = (long long)batch * ps->real.group;
    if (group_v * n_kv_heads > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;
    size_t prefix_bytes = 0;
    if (resolve_variant(variant) == PKV_VARIANT_TENSOR_CORES &&
        ps->real.group <= pkv::kPrefixTileRows) {
        // a tile holds whole sequences (all G rows of each), so every real unit
        // lies in one tile and Q comes as one box of G heads x sequences
        ps->umma = true;
        ps->tile_rows = (pkv::kPrefixTileRows / ps->real.group) * ps->real.group;
        ps->tiles = (int)((group_v + ps->tile_rows - 1) / ps->tile_rows);
        if ((st = prefix_splits(head_dim, dtype, (long long)ps->tiles * n_kv_heads,
                                &ps->max_splits)) != PKV_OK)
            return st;
        prefix_bytes = (size_t)n_kv_heads * ps->tiles * ps->max_splits *
                       (size_t)(pkv::kPrefixTileRows * (head_dim + 2)) * 4;
    } else {
        const int max_gs = 8;  // virtual units of up to 8 rows on CUDA cores
        int gs_v = ps->real.gs;
        for (int k = max_gs / ps->real.gs; k >= 1; --k)
            if (group_v % (k * ps->real.gs) == 0) {
                gs_v = k * ps->real.gs;
                break;
            }
        if ((st = setup_decode(1, (int)(group_v * n_kv_heads), n_kv_heads, head_dim, page_size,
                               dtype < 0 ? PKV_BF16 : (pkv_dtype)dtype, num_workers, variant,
                               &ps->virt, gs_v)) != PKV_OK)
            return st;
        prefix_bytes = ps->virt.ws.total;
    }
    // the suffix pass's workspace first: its header is the call's status word;
    // the gathered query rows last (CUDA-core variant only)
    const size_t qv_bytes = ps->umma ? 0 : align256((size_t)batch * n_q_heads * head_dim * 2);
    ps->s_off = 0;
    ps->v_off = align256(ps->real.ws.total);
    ps->qv_off = ps->v_off + align256(prefix_bytes);
    ps->total = ps->qv_off + qv_bytes;
    return PKV_OK;
}
}  // namespace

extern "C" {

pkv_status paged_decode_prefix_workspace_size(int batch, int n_q_heads, int n_kv_heads,
                                              int head_dim, int num_workers,
                                              pkv_decode_variant variant, size_t* bytes) {
    if (!bytes) return PKV_ERR_INVALID_ARG;
    if (batch == 0) {
        *bytes = 0;
        return PKV_OK;
    }
    PrefixSetup ps;
    pkv_status st = setup_prefix(batch, n_q_heads, n_kv_heads, head_dim, 16, -1, num_workers,
                                 variant, &ps);
    if (st != PKV_OK) return st;
    *bytes = ps.total;
    return PKV_OK;
}

pkv_status paged_decode_attention_prefix(const void* q, const void* k_pool, const void* v_pool,
                                         const int32_t* page_table, int table_stride,
                                         const int32_t* context_lens, int batch, int n_q_heads,
                                         int n_kv_heads, int head_dim, int page_size,
                                         int num_pages, pkv_dtype dtype, float scale,
                                         int prefix_tokens, void* out, void* workspace,
                                         size_t ws_bytes, int num_workers,
                                         pkv_decode_variant variant, pkv_stream stream) {
    pkv_status st = validate_decode_args(q, k_pool, v_pool, page_table, table_stride,
                                         context_lens, true, batch, n_q_heads, n_kv_heads,
                                         head_dim, page_size, num_pages, dtype, scale, out,
                                         workspace, ws_bytes, num_workers, variant);
    if (st != PKV_OK || batch == 0) return st;
    if (prefix_tokens <= 0 || prefix_tokens % page_size ||
        prefix_tokens / page_size > table_stride)
        return PKV_ERR_INVALID_ARG;
    PrefixSetup ps;
    if ((st = setup_prefix(batch, n_q_heads, n_kv_heads, head_dim, page_size, dtype, num_workers,
                           variant, &ps)) != PKV_OK)
        return st;
    if (ws_bytes < ps.total) return PKV_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* qv = ws + ps.qv_off;
    void* ws_v = ws + ps.v_off;
    void* ws_s = ws + ps.s_off;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const int skip = prefix_tokens / page_size;
    const int hq_v = (int)((long long)batch * ps.real.group * n_kv_heads);
    // one launch: the plan of the suffixes (each row from column skip on,
    // lengths minus prefix_tokens), on CUDA cores the plan of the prefix's
    // virtual decode (one sequence of prefix_tokens read through row 0), the
    // gather of the query rows per KV head, and the check that every row starts
    // with row 0's prefix pages
    const pkv::PlanArgs pv = plan_args(nullptr, page_table, 1, page_size, table_stride,
                                       num_workers, ws_v, ps.umma ? ps.real : ps.virt, 0,
                                       prefix_tokens);
    const pkv::PlanArgs pss = plan_args(context_lens, page_table + skip, batch, page_size,
                                        table_stride, num_workers, ws_s, ps.real, skip);
    pkv::CascadeGather g;
    g.q = static_cast<const uint4*>(q);
    g.qv = ps.umma ? nullptr : static_cast<uint4*>(qv);
    g.batch = batch;
    g.n_kv_heads = n_kv_heads;
    g.group = ps.real.group;
    g.vecs = head_dim / 8;
    g.table = page_table;
    g.table_stride = table_stride;
    g.share_cols = skip;
    g.plan_virtual = ps.umma ? 0 : 1;
    uint32_t* call_status = &reinterpret_cast<WsHeader*>(ws_s)->status;
    uint8_t* wv = static_cast<uint8_t*>(ws_v);
    pkv::CascadeArgs c;
    int splits = 0;
    if (ps.umma) {
        // the tensor maps first: nothing is launched if one cannot be made
        const long long pool_rows = (long long)num_pages * n_kv_heads * page_size;
        if (pool_rows > 0x7fffffffLL) return PKV_ERR_UNSUPPORTED;  // 32-bit row coordinate
        CUtensorMap qm, km, vm, om;
        const long long slots = (long long)n_kv_heads * ps.tiles * ps.max_splits;
        if ((st = q_tile_map(q, batch, n_q_heads, head_dim, dtype, ps.real.group, ps.tile_rows,
                             &qm)) != PKV_OK ||
            (st = prefix_slots_map(wv, head_dim, slots, &om)) != PKV_OK ||
            (st = pool_map(k_pool, pool_rows, head_dim, dtype, &km)) != PKV_OK ||
            (st = pool_map(v_pool, pool_rows, head_dim, dtype, &vm)) != PKV_OK)
            return st;
        const int chunks = prefix_tokens / pkv::kChunk;
        splits = ps.max_splits < chunks ? ps.max_splits : chunks;
        // plan, then the suffixes, then the prefix pass: it needs nothing the
        // suffix pass writes, so its CTAs take the SMs the suffix pass's warps
        // leave, and its partial states are fresh in L2 for the merge
        if ((st = cuda_status(pkv::launch_cascade_plan(pss, pv, g, cs))) != PKV_OK) return st;
        if ((st = do_run(q, k_pool, v_pool, page_table + skip, table_stride, batch, n_q_heads,
                         n_kv_heads, head_dim, page_size, num_pages, dtype, scale, out, ws_s,
                         ps.real, false, cs, true)) != PKV_OK)
            return st;
        pkv::PrefixUmmaArgs pa;
        pa.table = page_table;
        pa.num_pages = num_pages;
        pa.n_kv_heads = n_kv_heads;
        pa.page_size = page_size;
        pa.chunks = chunks;
        pa.splits = splits;
        pa.rows = (int)((long long)batch * ps.real.group);
        pa.group = ps.real.group;
        pa.tile_rows = ps.tile_rows;
        pa.tiles = ps.tiles;
        pa.scale_log2 = scale * 1.4426950408889634f;
        pa.partials = reinterpret_cast<float*>(wv);
        pa.status = call_status;
        if ((st = cuda_status(pkv::launch_prefix_umma(dtype, head_dim, pa, qm, km, vm, om,
                                                      cs))) != PKV_OK)
            return st;
        c.v_partials = pa.partials;
        c.v_hdr = nullptr;
    } else {
        if ((st = cuda_status(pkv::launch_cascade_plan(pss, pv, g, cs))) != PKV_OK) return st;
        if ((st = do_run(qv, k_pool, v_pool, page_table, table_stride, 1, hq_v, n_kv_heads,
                         head_dim, page_size, num_pages, dtype, scale, out, ws_v, ps.virt, false,
                         cs, true, call_status)) != PKV_OK)
            return st;
        c.v_partials = reinterpret_cast<const float*>(wv + ps.virt.ws.partials);
        c.v_hdr = reinterpret_cast<const WsHeader*>(wv);
        if ((st = do_run(q, k_pool, v_pool, page_table + skip, table_stride, batch, n_q_heads,
                         n_kv_heads, head_dim, page_size, num_pages, dtype, scale, out, ws_s,
                         ps.real, false, cs, true)) != PKV_OK)
            return st;
    }
    uint8_t* wsu = static_cast<uint8_t*>(ws_s);
    c.s_partials = reinterpret_cast<const float*>(wsu + ps.real.ws.partials);
    c.s_prefix = reinterpret_cast<const int32_t*>(wsu + ps.real.ws.prefix);
    c.s_lens = reinterpret_cast<const int32_t*>(wsu + ps.real.ws.lens_eff);
    c.s_hdr = reinterpret_cast<const WsHeader*>(wsu);
    c.out = out;
    c.units_per_b = ps.real.units_per_b;
    c.sub_groups = ps.real.sub_groups;
    c.gs = ps.real.gs;
    c.group = ps.real.group;
    c.n_q_heads = n_q_heads;
    c.v_gs = ps.umma ? 0 : ps.virt.gs;
    c.v_sub = ps.umma ? 0 : ps.virt.sub_groups;
    c.v_nch = (prefix_tokens + 15) / 16;
    c.umma = ps.umma ? 1 : 0;
    c.v_tile_rows = ps.tile_rows;
    c.v_tiles = ps.tiles;
    c.v_splits = splits;
    return cuda_status(pkv::launch_cascade_combine(dtype, head_dim, c, (int)ps.real.units, cs));
}

}  // extern "C"

// --- several query tokens per sequence --------------------------------------
extern "C" {

pkv_status paged_decode_multi_workspace_size(int batch, int n_queries, int n_q_heads,
                                             int n_kv_heads, int head_dim, int num_workers,
                                             pkv_decode_variant variant, size_t* bytes) {
    if (!bytes) return PKV_ERR_INVALID_ARG;
    *bytes = 0;
    pkv_status st = check_shapes(batch, n_q_heads, n_kv_heads, head_dim, 16);
    if (st != PKV_OK) return st;
    if (num_workers < 0 || !valid_variant(variant) || n_queries < 1) return PKV_ERR_INVALID_ARG;
    DecodeSetup s;
    if ((st = setup_decode(batch, n_q_heads, n_kv_heads, head_dim, 16, PKV_BF16, num_workers,
                           variant, &s, 0, n_queries)) != PKV_OK)
        return st;
    *bytes = s.ws.total;
    return PKV_OK;
}

pkv_status paged_decode_attention_multi(const void* q, const void* k_pool, const void* v_pool,
                                        const int32_t* page_table, int table_stride,
                                        const int32_t* context_lens, int batch, int n_queries,
                                        int n_q_heads, int n_kv_heads, int head_dim,
                                        int page_size, int num_pages, pkv_dtype dtype,
                                        float scale, void* out, void* workspace, size_t ws_bytes,
                                        int num_workers, pkv_decode_variant variant,
                                        pkv_stream stream) {
    if (n_queries < 1) return PKV_ERR_INVALID_ARG;
    pkv_status st = validate_decode_args(q, k_pool, v_pool, page_table, table_stride,
                                         context_lens, true, batch, n_q_heads, n_kv_heads,
                                         head_dim, page_size, num_pages, dtype, scale, out,
                                         workspace, ws_bytes, num_workers, variant);
    if (st != PKV_OK || batch == 0) return st;
    // q and out hold n_queries rows per sequence: check the full extents
    const size_t qo = (size_t)batch * n_queries * n_q_heads * head_dim * 2;
    const size_t pool_bytes = (size_t)num_pages * n_kv_heads * page_size * head_dim * 2;
    if (overlaps(out, qo, q, qo) || overlaps(out, qo, k_pool, pool_bytes) ||
        overlaps(out, qo, v_pool, pool_bytes) || overlaps(out, qo, workspace, ws_bytes))
        return PKV_ERR_ALIAS;
    DecodeSetup s;
    if ((st = setup_decode(batch, n_q_heads, n_kv_heads, head_dim, page_size, dtype, num_workers,
                           variant, &s, 0, n_queries)) != PKV_OK)
        return st;
    if ((st = check_workspace(workspace, ws_bytes, s)) != PKV_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if ((st = do_plan(context_lens, page_table, batch, page_size, table_stride, num_workers,
                      workspace, s, nullptr, cs)) != PKV_OK)
        return st;
    if ((st = do_run(q, k_pool, v_pool, page_table, table_stride, batch, n_q_heads, n_kv_heads,
                     head_dim, page_size, num_pages, dtype, scale, out, workspace, s, false,
                     cs)) != PKV_OK)
        return st;
    return do_combine(batch, n_q_heads, head_dim, dtype, out, workspace, s, cs);
}

}  // extern "C"
