// prefix_umma.cu -- the shared-prefix pass of the cascade decode on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// When every sequence of a batch starts with the same pages (Experimental
// LibTorch prefix cache, "Combining persistence with RadixMLP": suffix
// attention over a shared prefix; CacheIR, "Current Capabilities": batched
// decode over shared page tables), the prefix's K/V serve the B*G query rows
// of each KV head at once.  That is a dense [rows x tokens] contraction per
// KV head -- the one step of this path with enough rows to fill a 128-row
// tensor-core tile.  CTA (split s, row tile t, KV head h) takes 128 query rows
// (tile_rows of them its own; tile_rows is a multiple of the sequence's row
// count, so no sequence straddles two tiles) and a balanced contiguous range
// of the prefix's 16-token chunks, and for each block of up to 128 tokens:
//
//   S  = Q K^T                tcgen05.mma M=128, N=block tokens, K=D
//   P  = 2^(S*scale*log2e - m)  one thread per row, read with tcgen05.ld
//   O  = O * 2^(m_old - m) + P V   tcgen05.mma M=128, N=D, K=block tokens
//
// with S and O in tensor memory (one lane per query row).  Q (a 3-D box of
// G heads x tile_rows / G sequences straight from q), K and V arrive by TMA
// (cp.async.bulk.tensor, 128-byte swizzle, 64-element inner boxes); P is
// written to shared memory in the same swizzled K-major layout (bf16 P as a
// high part plus a bf16 residual, two MMAs, as in the warp-level decode
// kernel), the high part over K and the residual over Q, both consumed by
// then -- so Q comes again with every block (from L2), and two CTAs fit on an
// SM at D = 128.  Each prefix chunk is read once per row tile -- the rows of 8 KV
// heads x 64 sequences x 4 heads of a group take two tiles per KV head --
// instead of once per 16-row warp tile.
//
// The CTA leaves one partial state of its 128 rows: o [128][D] (fp32, staged
// in swizzled shared memory and written by TMA tensor stores), then m [128]
// (base-2 units) and l [128].  The cascade's merge combines the splits with
// the suffix pass's partial states.
//
// The pass reads only the caller's inputs (q, row 0 of the page table, the
// pools) and writes only its own slots and the call's status word.  The
// kernel before it in the stream is the call's suffix pass, which writes
// neither inputs nor these slots and waited for every earlier kernel (the
// plan launch included) before this one could start; so the copies and
// products run before the programmatic-dependency wait -- the CTAs take the
// SMs that the suffix pass's warps leave -- and the results are written
// after it.  The wait also keeps the order for the merge that follows: this
// grid completes only after the suffix pass has.
//
// Every wait is bounded: on a timeout the CTA records PKV_DEV_TIMEOUT, waits
// (bounded) for its copies or MMAs still in flight, frees its tensor memory
// and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"
#include "kernels_aux.cuh"
#include "umma.cuh"

namespace pkv {

namespace {

constexpr int kTileRows = kPrefixTileRows;  // M of every MMA: one tensor-memory lane per row
constexpr int kBlockTok = 128;  // prefix tokens per block: N of S = Q K^T, K of O += P V
constexpr int kBlockChunks = kBlockTok / kChunk;
constexpr int kUmmaThreads = 128;

// Shared memory of one CTA (offsets from a 1 KiB aligned base).  A column
// block is 64 elements (128 bytes) wide; rows follow each other at 128 bytes,
// 8-row groups at 1 KiB.
template <int D, bool kSplitP>
struct PrefixLayout {
    static constexpr int kBoxes = D / 64;                  // column blocks of D
    static constexpr int kQBlock = kTileRows * 128;        // one column block of Q
    static constexpr int kKVBlock = kBlockTok * 128;       // ... of K or V (token rows)
    static constexpr int kPBlock = kTileRows * 128;        // 64 tokens of P
    static constexpr int kPBytes = kTileRows * kBlockTok * 2;
    static constexpr int kQBytes = kBoxes * kQBlock;
    static constexpr int kKBytes = kBoxes * kKVBlock;
    static constexpr int kOffQ = 0;                         // Q, then P's bf16 residual
    static constexpr int kOffPL = kOffQ;
    // K, then P (its high part)
    static constexpr int kOffKP = kOffQ + (kSplitP && kPBytes > kQBytes ? kPBytes : kQBytes);
    static constexpr int kOffV = kOffKP + (kKBytes > kPBytes ? kKBytes : kPBytes);
    static constexpr int kOffBar = kOffV + kKBytes;
    static constexpr int kColsS = kBlockTok;                // tensor memory: S, then O
    static constexpr int kTmemCols = kColsS + D <= 256 ? 256 : 512;
    // barriers and slots, alignment slack; at least 80 KiB, so that no more
    // CTAs share an SM than its 512 tensor-memory columns serve
    // o staged for the tensor stores: D / 32 column blocks of [128 rows x 128 B]
    // over the Q and K regions (free once the last product is done)
    static constexpr int kOutBlocks = D / 32;
    static_assert(kOutBlocks * kTileRows * 128 <= kOffV, "o fits the Q and K regions");
    static constexpr int kUsed = kOffBar + 64 + 1024;
    static constexpr int kBytes = kUsed > 80 * 1024 ? kUsed : 80 * 1024;
    static_assert(kTmemCols <= 256, "two CTAs per SM share the tensor memory");
};

template <typename T, int D>
__global__ void __launch_bounds__(kUmmaThreads, 1)
prefix_umma_kernel(const PrefixUmmaArgs a, const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap,
                   const __grid_constant__ CUtensorMap omap) {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr bool kSplitP = kBf16;
    using Lay = PrefixLayout<D, kSplitP>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    uint8_t* base = smem_raw + pad;
    const uint32_t sb = raw + pad;
    uint64_t* bar_load = reinterpret_cast<uint64_t*>(base + Lay::kOffBar);
    uint64_t* bar_mma = bar_load + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + Lay::kOffBar + 16);
    uint32_t* bad_slot = tmem_slot + 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == 0) tmem_alloc(tmem_slot, Lay::kTmemCols);
    if (tid == 32) {
        mbar_init(bar_load, 1);
        mbar_init(bar_mma, 1);
        fence_barrier_init();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&qmap))
                     : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap))
                     : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vmap))
                     : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&omap))
                     : "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // this thread's row: tensor-memory lane tid (warp w reaches lanes 32w..32w+31)
    const uint32_t row_s = tmem + ((uint32_t)(warp * 32) << 16);
    const uint32_t row_o = row_s + Lay::kColsS;
    pdl_trigger();  // the next kernel waits for this grid's completion itself

    const int split = blockIdx.x, tile = blockIdx.y, h = blockIdx.z;
    const int per = a.chunks / a.splits, ext = a.chunks - per * a.splits;
    const int c0 = split * per + min(split, ext);
    const int cn = per + (split < ext ? 1 : 0);
    const int qseq = tile * (a.tile_rows / a.group);  // the tile's first sequence
    const int nblk = (cn + kBlockChunks - 1) / kBlockChunks;
    const float sl2 = a.scale_log2;

    float m_run = -INFINITY, l_run = 0.f;
    uint32_t ph_load = 0, ph_mma = 0;
    uint32_t flags = 0;         // PKV_DEV_* bits, written after the dependency wait
    uint64_t* stuck = nullptr;  // a wait that gave up: its barrier (and phase below)
    uint32_t stuck_phase = 0;
    for (int blk = 0; blk < nblk; ++blk) {
        const int cb = c0 + blk * kBlockChunks;
        const int nch = min(kBlockChunks, c0 + cn - cb);  // 1 .. 8 chunks
        const int ntok = nch * kChunk;
        // ---- copies: Q, then the block's K and V chunks (lane c: chunk c; a
        // page id outside the pool skips its chunk)
        if (warp == 0) {
            bool good = false;
            int y = 0;
            if (lane < nch) {
                const int tok = (cb + lane) * kChunk;
                const int page = __ldg(a.table + tok / a.page_size);
                good = page >= 0 && page < a.num_pages;
                if (good) y = (page * a.n_kv_heads + h) * a.page_size + tok % a.page_size;
            }
            const uint32_t goodm = __ballot_sync(kFull, good);
            const uint32_t badm = __ballot_sync(kFull, lane < nch && !good);
            if (badm) flags |= PKV_DEV_BAD_PAGE;
            if (lane == 0) {
                *bad_slot = badm;
                // a Q box is tile_rows rows (rows past them keep stale data: their
                // results are never read)
                const uint32_t bytes = (uint32_t)(Lay::kBoxes * a.tile_rows * 128) +
                                       (uint32_t)__popc(goodm) * 2u * kChunk * D * 2u;
                mbar_arrive_expect_tx(bar_load, bytes);
                for (int bx = 0; bx < Lay::kBoxes; ++bx)
                    tma_load_3d(base + Lay::kOffQ + bx * Lay::kQBlock, &qmap, bx * 64,
                                h * a.group, qseq, bar_load);
            }
            __syncwarp();
            if (good)
                for (int bx = 0; bx < Lay::kBoxes; ++bx) {
                    const int off = bx * Lay::kKVBlock + lane * kChunk * 128;
                    tma_load_2d(base + Lay::kOffKP + off, &kmap, bx * 64, y, bar_load);
                    tma_load_2d(base + Lay::kOffV + off, &vmap, bx * 64, y, bar_load);
                }
        }
        if (__syncthreads_or(!mbar_wait_bounded(bar_load, ph_load))) {
            stuck = bar_load;
            stuck_phase = ph_load;
            break;
        }
        ph_load ^= 1u;
        const uint32_t badm = *bad_slot;
        if (badm) {
            // a skipped chunk's P is 0, but its V rows must be finite: zero them
            for (int c = 0; c < nch; ++c) {
                if (!((badm >> c) & 1u)) continue;
                for (int x = tid; x < Lay::kBoxes * kChunk * 8; x += kUmmaThreads) {
                    const int bx = x / (kChunk * 8), v = x - bx * kChunk * 8;
                    reinterpret_cast<uint4*>(base + Lay::kOffV + bx * Lay::kKVBlock +
                                             c * kChunk * 128)[v] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
        }

        // ---- S = Q K^T into tensor-memory columns [0, ntok)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc = umma_idesc(kTileRows, ntok, kBf16, false);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t kb = (uint32_t)((kk & 3) * 32);  // K step inside a column block
                const uint64_t ad =
                    umma_sdesc(sb + Lay::kOffQ + (kk >> 2) * Lay::kQBlock + kb, 16, 1024);
                const uint64_t bd =
                    umma_sdesc(sb + Lay::kOffKP + (kk >> 2) * Lay::kKVBlock + kb, 16, 1024);
                umma_f16(tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
            }
            umma_commit(bar_mma);
        }
        if (__syncthreads_or(!mbar_wait_bounded(bar_mma, ph_mma))) {
            stuck = bar_mma;
            stuck_phase = ph_mma;
            break;
        }
        ph_mma ^= 1u;
        tc_fence_after();

        // ---- online softmax of row tid over the block (base 2): the row's
        // scores come out of tensor memory once (the loads are warp-collective:
        // the block length is the same for every thread)
        uint32_t r[kBlockTok / 32][32];
#pragma unroll
        for (int jb = 0; jb < kBlockTok / 32; ++jb)
            if (jb * 32 < ntok) tmem_ld32(row_s + jb * 32, r[jb]);
        float mx = -INFINITY;
#pragma unroll
        for (int jb = 0; jb < kBlockTok / 32; ++jb)
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int t = jb * 32 + e;
                const bool ok = t < ntok && !((badm >> (t >> 4)) & 1u);
                mx = ok ? fmaxf(mx, __uint_as_float(r[jb][e]) * sl2) : mx;
            }
        const float m_new = fmaxf(m_run, mx);
        const float m_ref = m_new == -INFINITY ? 0.f : m_new;  // no token yet: weights 0
        const float alpha = fast_exp2(m_run - m_ref);
        float sum = 0.f;
#pragma unroll
        for (int jb = 0; jb < kBlockTok / 32; ++jb) {
            const int j = jb * 32;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int t0 = j + 8 * q;  // the 8-token piece t0 .. t0+7 of row tid
                float p[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int t = t0 + e;
                    const bool ok = t < ntok && !((badm >> (t >> 4)) & 1u);
                    p[e] = ok ? fast_exp2(__uint_as_float(r[jb][8 * q + e]) * sl2 - m_ref) : 0.f;
                    sum += p[e];
                }
                if (t0 < ntok) {
                    // swizzled K-major P: token block t0/64, piece (t0%64)/8 of row tid
                    const uint32_t off = (uint32_t)((t0 >> 6) * Lay::kPBlock + (tid >> 3) * 1024 +
                                                    (tid & 7) * 128 +
                                                    ((((t0 & 63) >> 3) ^ (tid & 7)) << 4));
                    uint4 hi, lo;
                    if constexpr (kSplitP) {
                        split_bf16x2(p[0], p[1], hi.x, lo.x);
                        split_bf16x2(p[2], p[3], hi.y, lo.y);
                        split_bf16x2(p[4], p[5], hi.z, lo.z);
                        split_bf16x2(p[6], p[7], hi.w, lo.w);
                        *reinterpret_cast<uint4*>(base + Lay::kOffPL + off) = lo;
                    } else {
                        hi.x = Cvt<T>::pack2(p[0], p[1]);
                        hi.y = Cvt<T>::pack2(p[2], p[3]);
                        hi.z = Cvt<T>::pack2(p[4], p[5]);
                        hi.w = Cvt<T>::pack2(p[6], p[7]);
                    }
                    *reinterpret_cast<uint4*>(base + Lay::kOffKP + off) = hi;
                }
            }
        }
        l_run = l_run * alpha + sum;
        m_run = m_new;
        // the earlier blocks' O, to the new maximum (warp-collective loads and stores)
        if (blk > 0 && __any_sync(kFull, alpha != 1.f)) {
#pragma unroll
            for (int j = 0; j < D; j += 32) {
                uint32_t r[32];
                tmem_ld32(row_o + j, r);
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                tmem_st32(row_o + j, r);
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();  // P (and zeroed V rows) before the tensor cores read them
        tc_fence_before();
        __syncthreads();

        // ---- O (+)= P V into tensor-memory columns [kColsS, kColsS + D)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc = umma_idesc(kTileRows, D, kBf16, true);
            for (int kt = 0; kt < nch; ++kt) {
                const uint32_t poff = (uint32_t)((kt >> 2) * Lay::kPBlock + (kt & 3) * 32);
                const uint64_t bd =
                    umma_sdesc(sb + Lay::kOffV + kt * kChunk * 128, Lay::kKVBlock, 1024);
                umma_f16(tmem + Lay::kColsS, umma_sdesc(sb + Lay::kOffKP + poff, 16, 1024), bd,
                         idesc, (blk > 0 || kt > 0) ? 1u : 0u);
                if constexpr (kSplitP)
                    umma_f16(tmem + Lay::kColsS, umma_sdesc(sb + Lay::kOffPL + poff, 16, 1024),
                             bd, idesc, 1u);
            }
            umma_commit(bar_mma);
        }
        if (__syncthreads_or(!mbar_wait_bounded(bar_mma, ph_mma))) {
            stuck = bar_mma;
            stuck_phase = ph_mma;
            break;
        }
        ph_mma ^= 1u;
        tc_fence_after();
    }

    pdl_wait();  // the suffix pass is complete (and the plan long before it)
    if (!stuck) {
        if (flags && lane == 0) set_status(a.status, flags);
        // the partial state of row tid: o staged in swizzled shared memory
        // (row tid, 16-byte piece c of column block jb at piece c ^ (tid & 7)),
        // then D / 32 tensor stores of [128 rows x 32 floats]; m and l stored
        // directly (coalesced)
        const long long slot = (long long)(h * a.tiles + tile) * a.splits + split;
#pragma unroll
        for (int jb = 0; jb < Lay::kOutBlocks; ++jb) {
            uint32_t o[32];
            tmem_ld32(row_o + jb * 32, o);
            uint8_t* row = base + jb * kTileRows * 128 + tid * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(row + ((c ^ (tid & 7)) << 4)) =
                    make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
        }
        float* ml = a.partials + slot * (long long)(kTileRows * D + 2 * kTileRows) + kTileRows * D;
        ml[tid] = m_run;
        ml[kTileRows + tid] = l_run;
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            for (int jb = 0; jb < Lay::kOutBlocks; ++jb)
                tma_store_3d(&omap, base + jb * kTileRows * 128, jb * 32, 0, (int)slot);
            bulk_commit_group();
            bulk_wait_group_all();  // the stores are done before the CTA leaves
        }
    } else {
        if (tid == 0) set_status(a.status, flags | PKV_DEV_TIMEOUT);
        mbar_wait_bounded(stuck, stuck_phase);  // what is still in flight lands first
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, Lay::kTmemCols);
}

// Dynamic shared memory opt-in and the largest shared-memory carveout (two
// CTAs of up to 113 KiB per SM), once per process and instantiation.
template <typename T, int D>
cudaError_t prepare_t() {
    using Lay = PrefixLayout<D, std::is_same<T, __nv_bfloat16>::value>;
    auto fn = prefix_umma_kernel<T, D>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::kBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    return e;
}

template <typename T, int D>
cudaError_t launch_t(const PrefixUmmaArgs& a, const CUtensorMap& qm, const CUtensorMap& km,
                     const CUtensorMap& vm, const CUtensorMap& om, cudaStream_t stream) {
    using Lay = PrefixLayout<D, std::is_same<T, __nv_bfloat16>::value>;
    const cudaError_t e = prepare_t<T, D>();
    if (e != cudaSuccess) return e;
    return launch_pdl(prefix_umma_kernel<T, D>, dim3(a.splits, a.tiles, a.n_kv_heads),
                      dim3(kUmmaThreads), (size_t)Lay::kBytes, stream, a, qm, km, vm, om);
}

// CTAs per SM: what the SM's shared memory holds (each CTA also reserves the
// driver's per-block share), at most two (tensor-memory columns).
template <typename T, int D>
int ctas_per_sm_t() {
    using Lay = PrefixLayout<D, std::is_same<T, __nv_bfloat16>::value>;
    int dev = 0, smem = 0, reserved = 0;
    if (prepare_t<T, D>() != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
            cudaSuccess)
        return 0;
    const int n = smem / (Lay::kBytes + reserved);
    const int by_tmem = 512 / Lay::kTmemCols;
    return n < by_tmem ? n : by_tmem;
}

}  // namespace

cudaError_t launch_prefix_umma(pkv_dtype dtype, int head_dim, const PrefixUmmaArgs& a,
                               const CUtensorMap& qmap, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, const CUtensorMap& omap,
                               cudaStream_t stream) {
    if (a.splits <= 0 || a.tiles <= 0) return cudaSuccess;
    if (dtype == PKV_BF16)
        return head_dim == 128 ? launch_t<__nv_bfloat16, 128>(a, qmap, kmap, vmap, omap, stream)
                               : launch_t<__nv_bfloat16, 64>(a, qmap, kmap, vmap, omap, stream);
    return head_dim == 128 ? launch_t<__half, 128>(a, qmap, kmap, vmap, omap, stream)
                           : launch_t<__half, 64>(a, qmap, kmap, vmap, omap, stream);
}

int prefix_umma_ctas_per_sm(pkv_dtype dtype, int head_dim) {
    if (dtype == PKV_BF16)
        return head_dim == 128 ? ctas_per_sm_t<__nv_bfloat16, 128>()
                               : ctas_per_sm_t<__nv_bfloat16, 64>();
    return head_dim == 128 ? ctas_per_sm_t<__half, 128>() : ctas_per_sm_t<__half, 64>();
}

}  // namespace pkv
