// decode_umma.cu -- paged GQA decode of several query tokens per sequence on
// the fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// A unit (sequence, KV head, query tile) holds R query rows -- query tokens x
// heads of the GQA group (Experimental LibTorch prefix cache, "Current
// execution limits": causal suffix queries of a request, up to 64) -- that
// share every K/V chunk of the sequence.  R is 16..64: too few rows for a
// 128-row tile, too many for the registers of one warp.  So the products are
// taken transposed, with the 128 tokens of a block as the tile's rows:
//
//   S^T = K Q^T             tcgen05.mma M=128 tokens, N=rows, K=D (K-major A, B)
//   P^T = 2^(S^T*scale*log2e - m)   one thread per token, a column per row
//   O^T = O^T * 2^(m_old - m) + V^T P^T   M=D=128, N=rows, K=tokens (V as an
//                                         MN-major A operand)
//
// with S^T and O^T in tensor memory.  Nothing of the tile is padding but the
// rows of a unit beyond R (N = R rounded up to 16).  The running maximum of a
// row is a reduction over the block's tokens, i.e. over the CTA's 128
// threads: a warp reduction, then four partial maxima through shared memory.
//
// One CTA of 4 warps per SM is one worker of the decode schedule: a
// contiguous range of the batch's 16-token chunks (schedule.cuh), consumed in
// blocks of at most 8 chunks of one unit.  Warp 0 describes each block (unit,
// chunks, page ids) and issues its copies -- K and V chunks by 2-D tensor
// copies (128-byte swizzle, L2 evict-first), and at a segment start the
// unit's q rows by a 3-D tensor copy straight out of q -- STAGES blocks ahead
// of the consumer.  P (bf16: a high part and a bf16 residual, two products)
// is written over the block's K, which the S product has consumed.  A
// segment that is a whole unit writes the output; any other leaves a partial
// state (o, m, l of its N rows) in slot u + w for the combine kernel.
//
// Every wait is bounded: on a timeout the CTA records PKV_DEV_TIMEOUT, waits
// (bounded) for the copies and products still in flight, frees its tensor
// memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "merge.cuh"
#include "schedule.cuh"
#include "umma.cuh"

namespace pkv {

namespace {

constexpr int kD = 128;                // head_dim of this kernel
constexpr int kBlkTok = 128;           // tokens of a block: M of S^T = K Q^T
constexpr int kBlkChunks = kBlkTok / kChunk;
constexpr int kThreads = 128;          // one thread per token of a block, per d of O^T
constexpr int kColO = 64;              // tensor memory: S^T in [0, N), O^T in [64, 64 + N)
constexpr int kTmemCols = 128;

// A block as warp 0 described it (shared memory, one per stage).
struct BlockDesc {
    int u;          // unit
    int k0;         // first chunk of the block within the unit
    int nch;        // chunks (1..8)
    int len;        // tokens of the sequence
    int ntok;       // tokens of the block inside the sequence (the last chunk may be short)
    uint32_t bad;   // chunks whose page id is outside the pool (not copied, not attended)
    int flags;      // kSegStart, kSegEnd, kUnitFirst, kUnitLast
    int qslot;      // slot of the q ring holding the segment's rows
};
constexpr int kSegStart = 1, kSegEnd = 2, kUnitFirst = 4, kUnitLast = 8, kLast = 16;

// Shared memory (offsets from a 1 KiB aligned base).  A column block is 64
// elements (128 bytes) of D, or 64 tokens of P; rows follow at 128 bytes,
// 8-row groups at 1 KiB.
template <int N, int STAGES>
struct UmmaLayout {
    static constexpr int kKVBlock = kBlkTok * 128;        // one column block of K or V
    static constexpr int kK = 0;                          // K: 2 column blocks
    static constexpr int kV = 2 * kKVBlock;               // V: 2 column blocks
    static constexpr int kStage = 4 * kKVBlock;           // 64 KiB
    static constexpr int kRowBlock = N * 128;             // one column block of N rows
    static constexpr int kPHi = 0;                        // P^T over the stage's K:
    static constexpr int kPLo = 2 * kRowBlock;            // 2 token blocks each
    static constexpr int kQSlots = STAGES + 1;            // segments alive at once
    static constexpr int kQ = STAGES * kStage;            // the q ring: 2 column blocks per slot
    static constexpr int kQSlot = 2 * kRowBlock;
    static constexpr int kDesc = kQ + kQSlots * kQSlot;
    static constexpr int kRed = kDesc + STAGES * (int)sizeof(BlockDesc);   // [4][N] floats
    static constexpr int kRowM = kRed + 4 * N * 4;        // running maximum per row
    static constexpr int kRowRef = kRowM + N * 4;         // the block's reference maximum
    static constexpr int kRowAlpha = kRowRef + N * 4;     // rescale factor of the block
    static constexpr int kBar = (kRowAlpha + N * 4 + 15) / 16 * 16;  // full[STAGES], mma
    static constexpr int kTmemSlot = kBar + (STAGES + 1) * 8;
    static constexpr int kBytes = kTmemSlot + 16 + 1024;  // + alignment slack
};

template <int N>
constexpr int umma_stages() {
    return UmmaLayout<N, 3>::kBytes <= 227 * 1024 ? 3 : 2;
}

// Monotone map of a float onto a signed int (for warp max by redux.sync).
__device__ __forceinline__ int ord_of(float x) {
    const int i = __float_as_int(x);
    return i >= 0 ? i : (i ^ 0x7FFFFFFF);
}
__device__ __forceinline__ float float_of(int i) {
    return __int_as_float(i >= 0 ? i : (i ^ 0x7FFFFFFF));
}
__device__ __forceinline__ int warp_max_i(int v) {
    int r;
    asm volatile("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
    return r;
}

// Byte offset of element (row r, column c) of a K-major 128-byte-swizzled
// operand whose column blocks of 64 elements are `block` bytes apart.
__device__ __forceinline__ uint32_t swz_elem(int r, int c, int block) {
    return (uint32_t)((c >> 6) * block + r * 128 + (((((c & 63) >> 3) ^ (r & 7))) << 4) +
                      (c & 7) * 2);
}

template <typename T, int N, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
decode_umma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap) {
    using Lay = UmmaLayout<N, STAGES>;
    static_assert(N % 16 == 0 && N >= 16 && N <= kColO, "rows of a unit: 16, 32, 48 or 64");
    static_assert(Lay::kPLo + 2 * Lay::kRowBlock <= 2 * Lay::kKVBlock, "P fits over K");
    static_assert(Lay::kBytes <= 227 * 1024, "one CTA per SM");
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr bool kSplitP = kBf16;
    constexpr int NL = N < 32 ? 32 : N;  // columns read per tensor-memory load sweep
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    uint8_t* base = smem_raw + pad;
    const uint32_t sb = raw + pad;
    BlockDesc* desc = reinterpret_cast<BlockDesc*>(base + Lay::kDesc);
    float* red = reinterpret_cast<float*>(base + Lay::kRed);
    float* row_m = reinterpret_cast<float*>(base + Lay::kRowM);
    float* row_ref = reinterpret_cast<float*>(base + Lay::kRowRef);
    float* row_alpha = reinterpret_cast<float*>(base + Lay::kRowAlpha);
    uint64_t* full = reinterpret_cast<uint64_t*>(base + Lay::kBar);
    uint64_t* mma_bar = full + STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + Lay::kTmemSlot);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
    if (tid == 32) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
        mbar_init(mma_bar, 1);
        fence_barrier_init();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&qmap))
                     : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap))
                     : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vmap))
                     : "memory");
    }
    // the q ring: rows of a slot past a unit's rows are never copied and stay zero
    for (int x = tid; x < Lay::kQSlots * Lay::kQSlot / 16; x += kThreads)
        reinterpret_cast<uint4*>(base + Lay::kQ)[x] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // this thread's tensor-memory lane: token tid of S^T, element d = tid of O^T
    const uint32_t lane_s = tmem + ((uint32_t)(warp * 32) << 16);
    const uint32_t lane_o = lane_s + kColO;

    pdl_wait();
    pdl_trigger();

    const int gw = blockIdx.x;
    const int units_per_b = p.n_kv_heads * p.sub_groups;
    const RowShape rs = p.rows;
    const int q_rows = rs.queries_per_unit * rs.heads_per_unit;  // rows of a q copy
    int stream_end = 0, range_f0 = 0, b_lo = 0, b_hi = 0;
    if (gw < p.hdr->num_workers) {
        const int sw = p.hdr->chunks_per_worker, r = p.hdr->extra_chunks;
        range_f0 = range_begin(gw, sw, r);
        stream_end = sw + (gw < r ? 1 : 0);
        b_lo = __ldg(p.wstart + gw);
        b_hi = min(p.batch, __ldg(p.wstart + gw + 1) + 1);
    }
    if (warp == 0) zero_empty_sequences(p, kD, gw, gridDim.x, lane);

    // ---- producer (warp 0): the next block of at most 8 chunks of one unit
    const uint64_t kv_policy = l2_evict_first_policy();
    int next_pos = 0, seg_count = 0, issued = 0;
    auto issue = [&](int i) -> bool {
        if (next_pos >= stream_end) return false;
        const int st = i % STAGES;
        uint8_t* stage = base + st * Lay::kStage;
        ChunkDesc d;
        d.u = -1;
        d.k = 0;
        d.nch = 1;
        d.nvalid = 0;
        d.len = 0;
        d.off = -1;
        const bool in = lane < kBlkChunks && next_pos + lane < stream_end;
        if (in) d = describe_chunk(p, range_f0 + next_pos + lane, units_per_b, b_lo, b_hi);
        const int u0 = __shfl_sync(kFull, d.u, 0);
        const uint32_t same = __ballot_sync(kFull, in && d.u == u0);
        const int nch = __ffs(~same) - 1;  // the chunks of unit u0 at the front: 1..8
        const uint32_t bad = __ballot_sync(kFull, lane < nch && d.off < 0);
        const int k0 = __shfl_sync(kFull, d.k, 0);
        const int nch_u = __shfl_sync(kFull, d.nch, 0);
        const int len = __shfl_sync(kFull, d.len, 0);
        const int nv_last = __shfl_sync(kFull, d.nvalid, nch - 1);
        const bool unit_last = k0 + nch == nch_u;
        const bool last = next_pos + nch >= stream_end;
        int flags = (k0 == 0 ? kUnitFirst : 0) | (unit_last ? kUnitLast : 0) |
                    (last ? kLast : 0);
        if (k0 == 0 || next_pos == 0) flags |= kSegStart;
        if (unit_last || last) flags |= kSegEnd;
        if (flags & kSegStart) ++seg_count;
        const int qslot = (seg_count - 1) % Lay::kQSlots;
        const int b = u0 / units_per_b;
        b_lo = b;  // later chunks of the range lie in this sequence or after it
        if (lane == 0) {
            desc[st] = BlockDesc{u0, k0, nch, len, (nch - 1) * kChunk + nv_last, bad, flags, qslot};
            const int good = __popc(~bad & ((1u << nch) - 1u));
            uint32_t bytes = (uint32_t)good * 2u * kChunk * kD * 2u;
            if (flags & kSegStart) bytes += 2u * (uint32_t)q_rows * 128u;
            mbar_arrive_expect_tx(&full[st], bytes);
            if (flags & kSegStart) {
                // the unit's rows: q_rows = tokens x heads of q, token-major
                const int uidx = u0 - b * units_per_b;
                const int h = uidx / p.sub_groups, sg = uidx - h * p.sub_groups;
                const int t = sg / rs.head_blocks, blk = sg - t * rs.head_blocks;
                const int y = h * rs.group + blk * rs.heads_per_unit;
                const int z = b * rs.n_queries + t * rs.queries_per_unit;
                uint8_t* qd = base + Lay::kQ + qslot * Lay::kQSlot;
                tma_load_3d(qd, &qmap, 0, y, z, &full[st]);
                tma_load_3d(qd + Lay::kRowBlock, &qmap, 64, y, z, &full[st]);
            }
        }
        __syncwarp();
        if (lane < nch && d.off >= 0) {
            const int y = (int)d.off;
#pragma unroll
            for (int bx = 0; bx < 2; ++bx) {
                const int off = bx * Lay::kKVBlock + lane * kChunk * 128;
                tma_load_2d_hint(stage + Lay::kK + off, &kmap, bx * 64, y, &full[st], kv_policy);
                tma_load_2d_hint(stage + Lay::kV + off, &vmap, bx * 64, y, &full[st], kv_policy);
            }
        }
        next_pos += nch;
        return true;
    };
    if (warp == 0)
        while (issued < STAGES && issue(issued)) ++issued;

    // ---- consumer (all threads): block i in stage i % STAGES
    const float sl2 = p.scale_log2;
    float lp[N];  // this thread's (token's) share of each row's sum of weights
#pragma unroll
    for (int c = 0; c < N; ++c) lp[c] = 0.f;
    uint32_t ph_mma = 0;
    uint64_t* stuck = nullptr;  // a wait that gave up (and its phase)
    uint32_t stuck_phase = 0;
    int fail_block = 0;
    bool first_block = true, seg_unit_first = false;
    int seg_b = 0, seg_h = 0, seg_sg = 0, seg_rows = 0, seg_slot = 0;
    for (int i = 0; stream_end > 0; ++i) {
        const int st = i % STAGES;
        const uint32_t ph = (uint32_t)((i / STAGES) & 1);
        if (__syncthreads_or(!mbar_wait_bounded(&full[st], ph))) {
            stuck = &full[st];
            stuck_phase = ph;
            fail_block = i;
            break;
        }
        const BlockDesc bd = desc[st];
        uint8_t* stage = base + st * Lay::kStage;
        const uint32_t sst = sb + st * Lay::kStage;
        if (bd.flags & kSegStart) {
            seg_b = bd.u / units_per_b;
            const int uidx = bd.u - seg_b * units_per_b;
            seg_h = uidx / p.sub_groups;
            seg_sg = uidx - seg_h * p.sub_groups;
            seg_rows = rs.rows(seg_sg);
            seg_slot = gw + bd.u;
            seg_unit_first = (bd.flags & kUnitFirst) != 0;
            first_block = true;
            if (tid < N) row_m[tid] = -INFINITY;
#pragma unroll
            for (int c = 0; c < N; ++c) lp[c] = 0.f;
        }
        // V rows the block does not attend (past the length in its last chunk,
        // or in a skipped chunk) must still be finite for the P V product
        if (bd.bad || bd.ntok < bd.nch * kChunk) {
            for (int x = tid; x < bd.nch * kChunk * 16; x += kThreads) {
                const int row = x >> 4, piece = x & 15;
                if (row >= bd.ntok || ((bd.bad >> (row >> 4)) & 1u))
                    *reinterpret_cast<uint4*>(stage + Lay::kV + (piece >> 3) * Lay::kKVBlock +
                                              row * 128 + ((piece & 7) << 4)) =
                        make_uint4(0u, 0u, 0u, 0u);
            }
        }

        // ---- S^T = K Q^T into tensor-memory columns [0, N)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc = umma_idesc(kBlkTok, N, kBf16, false);
            const uint32_t qs = sb + Lay::kQ + bd.qslot * Lay::kQSlot;
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
                const uint32_t kb = (uint32_t)((kk & 3) * 32);  // K step inside a column block
                const uint64_t ad = umma_sdesc(sst + Lay::kK + (kk >> 2) * Lay::kKVBlock + kb, 16,
                                               1024);
                const uint64_t bdsc = umma_sdesc(qs + (kk >> 2) * Lay::kRowBlock + kb, 16, 1024);
                umma_f16(tmem, ad, bdsc, idesc, kk > 0 ? 1u : 0u);
            }
            umma_commit(mma_bar);
        }
        if (__syncthreads_or(!mbar_wait_bounded(mma_bar, ph_mma))) {
            stuck = mma_bar;
            stuck_phase = ph_mma;
            fail_block = i + 1;  // block i's copies have landed
            break;
        }
        ph_mma ^= 1u;
        tc_fence_after();

        // ---- scores of token tid for every row, masked: past the length, a
        // skipped chunk, or (several queries) after the row's query token
        float v[N];
        {
            const int t = tid;
            const bool tok_ok = t < bd.ntok && !((bd.bad >> (t >> 4)) & 1u);
            // row c (query fq + c / hpu) sees position pos iff
            // pos <= len - n_queries + fq + c / hpu
            const int slack = bd.len - rs.n_queries + rs.first_query(seg_sg) -
                              (bd.k0 * kChunk + t);
            const int c_min = slack >= 0 ? 0 : -slack * rs.heads_per_unit;
#pragma unroll
            for (int c0 = 0; c0 < NL; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(lane_s + c0, r);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int c = c0 + e;
                    if (c < N)
                        v[c] = (tok_ok && c >= c_min) ? __uint_as_float(r[e]) * sl2 : -INFINITY;
                }
            }
        }
        // per-row maxima of the block: warp maxima, then the four warps'
#pragma unroll
        for (int c = 0; c < N; ++c) {
            const int mi = warp_max_i(ord_of(v[c]));
            if (lane == (c & 31)) red[warp * N + c] = float_of(mi);
        }
        __syncthreads();
        if (tid < N) {
            const int c = tid;
            const float bm = fmaxf(fmaxf(red[c], red[N + c]), fmaxf(red[2 * N + c], red[3 * N + c]));
            const float m_old = row_m[c];
            const float m_new = fmaxf(m_old, bm);
            const float m_ref = m_new == -INFINITY ? 0.f : m_new;  // no token yet: weights 0
            row_m[c] = m_new;
            row_ref[c] = m_ref;
            row_alpha[c] = fast_exp2(m_old - m_ref);
        }
        const bool rescale = __syncthreads_or(!first_block && tid < N && row_alpha[tid] != 1.f);

        // ---- P^T over the consumed K: row c, token tid (pairs of tokens per
        // 32-bit store: even lanes take row c, odd lanes row c + 1)
        {
            const bool odd = lane & 1;
            const int tok = tid & ~1;
#pragma unroll
            for (int c = 0; c < N; c += 2) {
                const float p0 = fast_exp2(v[c] - row_ref[c]);
                const float p1 = fast_exp2(v[c + 1] - row_ref[c + 1]);
                lp[c] = fmaf(lp[c], row_alpha[c], p0);
                lp[c + 1] = fmaf(lp[c + 1], row_alpha[c + 1], p1);
                const float got = __shfl_xor_sync(kFull, odd ? p0 : p1, 1);
                const float a = odd ? got : p0, bb = odd ? p1 : got;
                const uint32_t off = swz_elem(c + (odd ? 1 : 0), tok, Lay::kRowBlock);
                if constexpr (kSplitP) {
                    uint32_t hi, lo;
                    split_bf16x2(a, bb, hi, lo);
                    *reinterpret_cast<uint32_t*>(stage + Lay::kPHi + off) = hi;
                    *reinterpret_cast<uint32_t*>(stage + Lay::kPLo + off) = lo;
                } else {
                    *reinterpret_cast<uint32_t*>(stage + Lay::kPHi + off) = Cvt<T>::pack2(a, bb);
                }
            }
        }
        // ---- the earlier blocks' O^T, to the new maxima (element d = tid)
        if (rescale) {
#pragma unroll
            for (int c0 = 0; c0 < NL; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(lane_o + c0, r);
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (c0 + e < N) r[e] = __float_as_uint(__uint_as_float(r[e]) * row_alpha[c0 + e]);
                tmem_st32(lane_o + c0, r);
            }
            tmem_wait_st();
        }
        fence_proxy_async_smem();  // P^T and zeroed V rows before the tensor cores read them
        tc_fence_before();
        __syncthreads();

        // ---- O^T (+)= V^T P^T into tensor-memory columns [64, 64 + N)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc = umma_idesc(kD, N, kBf16, false, true);
            for (int kt = 0; kt < bd.nch; ++kt) {
                const uint64_t ad =
                    umma_sdesc(sst + Lay::kV + kt * kChunk * 128, Lay::kKVBlock, 1024);
                const uint32_t poff = (uint32_t)((kt >> 2) * Lay::kRowBlock + (kt & 3) * 32);
                const uint32_t acc = (!first_block || kt > 0) ? 1u : 0u;
                umma_f16(tmem + kColO, ad, umma_sdesc(sst + Lay::kPHi + poff, 16, 1024), idesc,
                         acc);
                if constexpr (kSplitP)
                    umma_f16(tmem + kColO, ad, umma_sdesc(sst + Lay::kPLo + poff, 16, 1024),
                             idesc, 1u);
            }
            umma_commit(mma_bar);
        }
        if (__syncthreads_or(!mbar_wait_bounded(mma_bar, ph_mma))) {
            stuck = mma_bar;
            stuck_phase = ph_mma;
            fail_block = i + 1;
            break;
        }
        ph_mma ^= 1u;
        tc_fence_after();
        first_block = false;

        if (bd.flags & kSegEnd) {
            // each row's sum of weights over the CTA's tokens, in a fixed order
#pragma unroll
            for (int c = 0; c < N; ++c) {
                float s = lp[c];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
                if (lane == (c & 31)) red[warp * N + c] = s;
            }
            __syncthreads();
            if (tid < N)
                row_alpha[tid] = (red[tid] + red[N + tid]) + (red[2 * N + tid] + red[3 * N + tid]);
            __syncthreads();
            // element d = tid of every row: the output of a whole unit, else a
            // partial state (o, m, l) in slot u + w
            const bool whole = seg_unit_first && (bd.flags & kUnitLast) && !p.all_partials;
            float* slot = p.partials + (long long)seg_slot * partial_slot_floats(N, kD);
            uint16_t* outp = static_cast<uint16_t*>(p.out);
#pragma unroll
            for (int c0 = 0; c0 < NL; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(lane_o + c0, r);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int c = c0 + e;
                    if (c < N && c < seg_rows) {
                        const float o = __uint_as_float(r[e]);
                        if (whole) {
                            const float l = row_alpha[c];
                            const float inv = l > 0.f ? 1.0f / l : 0.f;
                            outp[rs.row(seg_b, seg_h, seg_sg, c) * kD + tid] =
                                (uint16_t)(Cvt<T>::pack2(o * inv, 0.f) & 0xffffu);
                        } else {
                            slot[c * kD + tid] = o;
                        }
                    }
                }
            }
            if (!whole && tid < seg_rows) {
                slot[N * kD + tid] = row_m[tid];
                slot[N * kD + N + tid] = row_alpha[tid];
            }
        }
        // the stage is free again: block i + STAGES into it
        if (warp == 0)
            while (issued <= i + STAGES && issue(issued)) ++issued;
        if (bd.flags & kLast) break;
    }

    if (stuck) {
        // a copy or a product never completed: report it, then wait (bounded)
        // for what is still in flight into this CTA's memory
        if (tid == 0) {
            set_status(p.status, PKV_DEV_TIMEOUT);
            if (stuck == mma_bar) mbar_wait_bounded(mma_bar, stuck_phase);
            for (int j = fail_block; j < issued; ++j)
                mbar_wait_bounded(&full[j % STAGES], (uint32_t)((j / STAGES) & 1));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <typename T, int N>
DecodeUmmaInfo make_umma_info() {
    constexpr int S = umma_stages<N>();
    DecodeUmmaInfo info;
    info.fn = decode_umma_kernel<T, N, S>;
    info.stages = S;
    info.smem_bytes = UmmaLayout<N, S>::kBytes;
    info.n = N;
    return info;
}

}  // namespace

// The instantiation for units of `rows` query rows (16, 32 or 64 after
// rounding up), head_dim 128; fn null when there is none.
DecodeUmmaInfo decode_umma_info(bool bf16, int head_dim, int rows) {
    if (head_dim != kD || rows < 1 || rows > 64) return DecodeUmmaInfo{};
    if (bf16) {
        if (rows <= 16) return make_umma_info<__nv_bfloat16, 16>();
        if (rows <= 32) return make_umma_info<__nv_bfloat16, 32>();
        return make_umma_info<__nv_bfloat16, 64>();
    }
    if (rows <= 16) return make_umma_info<__half, 16>();
    if (rows <= 32) return make_umma_info<__half, 32>();
    return make_umma_info<__half, 64>();
}

}  // namespace pkv
