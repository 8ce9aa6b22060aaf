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
// with S^T (two buffers) and O^T in tensor memory.  Nothing of the tile is
// padding but the rows of a unit beyond R (N = R rounded up to 16).
//
// One CTA per SM is one worker of the decode schedule: a contiguous range of
// the batch's 16-token chunks (schedule.cuh), consumed in blocks of at most 8
// chunks of one unit.  Its warps:
//   producer   describes the next block's chunks (page lookups) while it
//              waits for a free stage, then issues the block's copies: K and V
//              chunks by 2-D tensor copies (128-byte swizzle, L2 evict-first)
//              and, at a segment start, the unit's q rows by a 3-D tensor copy
//              straight out of q, into a ring of STAGES + 1 slots;
//   MMA        one thread, two independent streams: S^T of the next block
//              once its copies have landed and its S buffer is read, P V of a
//              block once its P^T is written; each P V commit frees the stage;
//   consumers  8 warps, token quarter (warp % 4: the tensor-memory lanes it
//              reaches) x half of the rows: mask, exponentiate, write P^T (bf16:
//              a high part and a bf16 residual, two products) over the block's
//              consumed K, keep each row's sum of weights.
// A row keeps its reference maximum unless a score of the block exceeds it by
// more than 2^kLazyMax; only then is the exact maximum over the CTA's tokens
// taken (a warp reduction, then the four token quarters through shared
// memory) and O^T rescaled.  Output and merge use o, m, l relative to the same
// reference, so the result is the exact softmax either way.  A segment that is
// a whole unit writes the output; any other leaves a partial state (o, m, l of
// its N rows) in slot u + w for the combine kernel.
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
constexpr int kConsWarps = 8;          // consumers: token quarter (warp % 4) x row half
constexpr int kConsThreads = kConsWarps * 32;
constexpr int kThreads = kConsThreads + 64;  // + the producer warp + the MMA warp
constexpr float kLazyMax = 8.f;  // a block keeps the row's reference maximum unless a score
                                 // exceeds it by more than this (base 2: weights <= 2^8)
constexpr int kColS = 64;              // tensor memory: S^T of block i in [64 (i % 2), +N),
constexpr int kColO = 128;             // O^T in [128, 128 + N)
constexpr int kTmemCols = 256;

// A block as the producer warp described it (shared memory, one per stage).
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
    // each row's reference maximum (the running maximum of the blocks that moved it)
    static constexpr int kRowRef = kRed + 4 * N * 4;
    // each row's rescale factor in a block that moved the reference; at a
    // segment end, each row's sum of weights
    static constexpr int kRowAlpha = kRowRef + N * 4;
    // barriers: full[STAGES], empty[STAGES], S done[2], S read[2], P ready, P V done, drain
    static constexpr int kBar = (kRowAlpha + N * 4 + 15) / 16 * 16;
    static constexpr int kTmemSlot = kBar + (2 * STAGES + 7) * 8;  // then the issued count
    static constexpr int kBytes = kTmemSlot + 16 + 1024;  // + alignment slack
};

// Three stages when they fit beside the q ring (the sum of UmmaLayout's
// regions for STAGES = 3), else two.
template <int N>
constexpr int umma_stages() {
    return 3 * 4 * kBlkTok * 128 + 4 * 2 * N * 128 + 3 * (int)sizeof(BlockDesc) + 6 * N * 4 +
                       16 + 13 * 8 + 16 + 1024 <=
                   227 * 1024
               ? 3
               : 2;
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

// Named barrier 1 over the consumer warps (the producer warp runs its own loop).
__device__ __forceinline__ void cons_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsThreads) : "memory");
}
__device__ __forceinline__ bool cons_sync_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kConsThreads)
        : "memory");
    return r != 0;
}

template <typename T, int N, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
decode_umma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap) {
    using Lay = UmmaLayout<N, STAGES>;
    static_assert(N % 16 == 0 && N >= 16 && N <= kColS, "rows of a unit: 16, 32, 48 or 64");
    static_assert(Lay::kPLo + 2 * Lay::kRowBlock <= 2 * Lay::kKVBlock, "P fits over K");
    static_assert(Lay::kBytes <= 227 * 1024, "one CTA per SM");
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr bool kSplitP = kBf16;
    constexpr int NH = N / 2;  // rows (tensor-memory columns) of one consumer thread
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
    uint8_t* base = smem_raw + pad;
    const uint32_t sb = raw + pad;
    BlockDesc* desc = reinterpret_cast<BlockDesc*>(base + Lay::kDesc);
    float* red = reinterpret_cast<float*>(base + Lay::kRed);
    float* row_ref = reinterpret_cast<float*>(base + Lay::kRowRef);
    float* row_alpha = reinterpret_cast<float*>(base + Lay::kRowAlpha);
    uint64_t* full = reinterpret_cast<uint64_t*>(base + Lay::kBar);  // copies of a stage landed
    uint64_t* empty = full + STAGES;  // a stage's P V product done: the stage is free
    uint64_t* sbar = empty + STAGES;  // [2] S^T product of buffer b done
    uint64_t* sfree = sbar + 2;       // [2] S^T of buffer b read by the consumers
    uint64_t* pready = sfree + 2;     // P^T written (and O^T rescaled) by the consumers
    uint64_t* pvbar = pready + 1;     // P V product done
    uint64_t* drain = pvbar + 1;      // every product of the MMA warp done (before the exit)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + Lay::kTmemSlot);
    int* issued_slot = reinterpret_cast<int*>(base + Lay::kTmemSlot + 4);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
    if (tid == 32) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&sbar[0], 1);
        mbar_init(&sbar[1], 1);
        mbar_init(&sfree[0], kConsWarps);
        mbar_init(&sfree[1], kConsWarps);
        mbar_init(pready, kConsWarps);
        mbar_init(pvbar, 1);
        mbar_init(drain, 1);
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
    if (tid == 0) *issued_slot = 0;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    pdl_wait();

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

    // the S^T product of the block in stage st into S buffer bf (one thread)
    auto issue_s = [&](int st, int bf) {
        tc_fence_after();
        const uint32_t idesc = umma_idesc(kBlkTok, N, kBf16, false);
        const uint32_t sst = sb + st * Lay::kStage;
        const uint32_t qs = sb + Lay::kQ + desc[st].qslot * Lay::kQSlot;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t kb = (uint32_t)((kk & 3) * 32);  // K step inside a column block
            const uint64_t ad =
                umma_sdesc(sst + Lay::kK + (kk >> 2) * Lay::kKVBlock + kb, 16, 1024);
            const uint64_t bdsc = umma_sdesc(qs + (kk >> 2) * Lay::kRowBlock + kb, 16, 1024);
            umma_f16(tmem + kColS * bf, ad, bdsc, idesc, kk > 0 ? 1u : 0u);
        }
        umma_commit(&sbar[bf]);
    };

    if (warp == kConsWarps) {
        // ---- producer: blocks of at most 8 chunks of one unit, STAGES ahead
        zero_empty_sequences(p, kD, gw, gridDim.x, lane);
        const uint64_t kv_policy = l2_evict_first_policy();
        // A block's plan: lane c describes its chunk c (page lookups), the
        // warp agrees on the run of chunks of one unit at the front.
        struct Plan {
            ChunkDesc d;
            int u0, nch, k0, nch_u, len, nv_last;
            uint32_t bad;
        };
        auto plan_at = [&](int pos, int lo) -> Plan {
            Plan pl;
            pl.d.u = -1;
            pl.d.k = 0;
            pl.d.nch = 1;
            pl.d.nvalid = 0;
            pl.d.len = 0;
            pl.d.off = -1;
            const bool in = lane < kBlkChunks && pos + lane < stream_end;
            if (in) pl.d = describe_chunk(p, range_f0 + pos + lane, units_per_b, lo, b_hi);
            pl.u0 = __shfl_sync(kFull, pl.d.u, 0);
            const uint32_t same = __ballot_sync(kFull, in && pl.d.u == pl.u0);
            pl.nch = __ffs(~same) - 1;  // the chunks of unit u0 at the front: 1..8
            pl.bad = __ballot_sync(kFull, lane < pl.nch && pl.d.off < 0);
            pl.k0 = __shfl_sync(kFull, pl.d.k, 0);
            pl.nch_u = __shfl_sync(kFull, pl.d.nch, 0);
            pl.len = __shfl_sync(kFull, pl.d.len, 0);
            pl.nv_last = __shfl_sync(kFull, pl.d.nvalid, pl.nch - 1);
            return pl;
        };
        int next_pos = 0, seg_count = 0, j = 0;
        Plan cur;
        if (stream_end > 0) cur = plan_at(0, b_lo);
        while (next_pos < stream_end) {
            const int st = j % STAGES;
            const int b = cur.u0 / units_per_b;
            // the next block's page lookups go out before the wait for a free stage
            const int pos_next = next_pos + cur.nch;
            Plan nxt = cur;
            if (pos_next < stream_end) nxt = plan_at(pos_next, b);
            if (j >= STAGES) {
                // the stage is free once the P V product of block j - STAGES is done
                bool ok = lane == 0
                              ? mbar_wait_bounded(&empty[st], (uint32_t)(((j / STAGES) - 1) & 1))
                              : true;
                ok = __shfl_sync(kFull, ok, 0);
                if (!ok) {
                    if (lane == 0) set_status(p.status, PKV_DEV_TIMEOUT);
                    break;
                }
            }
            uint8_t* stage = base + st * Lay::kStage;
            const int nch = cur.nch, k0 = cur.k0;
            const bool unit_last = k0 + nch == cur.nch_u;
            const bool last = pos_next >= stream_end;
            int flags = (k0 == 0 ? kUnitFirst : 0) | (unit_last ? kUnitLast : 0) |
                        (last ? kLast : 0);
            if (k0 == 0 || next_pos == 0) flags |= kSegStart;
            if (unit_last || last) flags |= kSegEnd;
            if (flags & kSegStart) ++seg_count;
            const int qslot = (seg_count - 1) % Lay::kQSlots;
            if (lane == 0) {
                desc[st] = BlockDesc{cur.u0, k0, nch, cur.len, (nch - 1) * kChunk + cur.nv_last,
                                     cur.bad, flags, qslot};
                const int good = __popc(~cur.bad & ((1u << nch) - 1u));
                uint32_t bytes = (uint32_t)good * 2u * kChunk * kD * 2u;
                if (flags & kSegStart) bytes += 2u * (uint32_t)q_rows * 128u;
                mbar_arrive_expect_tx(&full[st], bytes);
                if (flags & kSegStart) {
                    // the unit's rows: q_rows = tokens x heads of q, token-major
                    const int uidx = cur.u0 - b * units_per_b;
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
            if (lane < nch && cur.d.off >= 0) {
                const int y = (int)cur.d.off;
#pragma unroll
                for (int bx = 0; bx < 2; ++bx) {
                    const int off = bx * Lay::kKVBlock + lane * kChunk * 128;
                    tma_load_2d_hint(stage + Lay::kK + off, &kmap, bx * 64, y, &full[st],
                                     kv_policy);
                    tma_load_2d_hint(stage + Lay::kV + off, &vmap, bx * 64, y, &full[st],
                                     kv_policy);
                }
            }
            next_pos = pos_next;
            ++j;
            cur = nxt;
        }
        if (lane == 0) *issued_slot = j;
    } else if (warp == kConsWarps + 1) {
        // ---- MMA warp (one thread): S^T of block i + 1 as soon as its copies
        // have landed and its S buffer is read, then P V of block i once the
        // consumers have written P^T
        if (lane == 0 && stream_end > 0) {
            // two independent streams of products, issued as their inputs become
            // ready: S^T of block si (its copies landed, its S buffer read by the
            // consumers two blocks ago), P V of block pi (P^T written)
            int si = 0, pi = 0;
            bool s_all = false, ok = true;
            uint32_t idle = 0;
            while (true) {
                bool progress = false;
                if (!s_all) {
                    const int st = si % STAGES, bf = si & 1;
                    if (mbar_test_wait(&full[st], (uint32_t)((si / STAGES) & 1)) &&
                        (si < 2 || mbar_test_wait(&sfree[bf], (uint32_t)(((si - 2) >> 1) & 1)))) {
                        issue_s(st, bf);
                        s_all = (desc[st].flags & kLast) != 0;
                        ++si;
                        progress = true;
                    }
                }
                if (pi < si && mbar_test_wait(pready, (uint32_t)(pi & 1))) {
                    tc_fence_after();
                    const int st = pi % STAGES;
                    const BlockDesc bd = desc[st];
                    const uint32_t sst = sb + st * Lay::kStage;
                    const uint32_t idesc = umma_idesc(kD, N, kBf16, false, true);
                    const bool first = (bd.flags & kSegStart) != 0;
                    for (int kt = 0; kt < bd.nch; ++kt) {
                        const uint64_t ad =
                            umma_sdesc(sst + Lay::kV + kt * kChunk * 128, Lay::kKVBlock, 1024);
                        const uint32_t poff =
                            (uint32_t)((kt >> 2) * Lay::kRowBlock + (kt & 3) * 32);
                        const uint32_t acc = (!first || kt > 0) ? 1u : 0u;
                        umma_f16(tmem + kColO, ad, umma_sdesc(sst + Lay::kPHi + poff, 16, 1024),
                                 idesc, acc);
                        if constexpr (kSplitP)
                            umma_f16(tmem + kColO, ad,
                                     umma_sdesc(sst + Lay::kPLo + poff, 16, 1024), idesc, 1u);
                    }
                    umma_commit(pvbar);
                    umma_commit(&empty[st]);  // the stage is free once this product is done
                    ++pi;
                    progress = true;
                    if (bd.flags & kLast) break;
                }
                if (progress) {
                    idle = 0;
                } else if (++idle > kSpinLimit) {
                    ok = false;
                    break;
                }
            }
            if (!ok) set_status(p.status, PKV_DEV_TIMEOUT);
            // nothing of this CTA's products may still run when it exits
            umma_commit(drain);
            mbar_wait_bounded(drain, 0);
        }
    } else {
        // ---- consumers: token tq * 32 + lane of a block (element d of O^T),
        // rows [hf * NH, hf * NH + NH) of the unit
        const int tq = warp & 3, hf = warp >> 2;
        const int t = tq * 32 + lane;
        const int cb = hf * NH;
        const uint32_t lane_q = tmem + ((uint32_t)(tq * 32) << 16) + (uint32_t)cb;
        const uint32_t lane_o = lane_q + kColO;
        const float sl2 = p.scale_log2;
        float lp[NH];  // this token's share of each row's sum of weights
#pragma unroll
        for (int c = 0; c < NH; ++c) lp[c] = 0.f;
        uint32_t ph_pv = 0;
        bool pv_pending = false, first_block = true, seg_unit_first = false, local_fail = false;
        int seg_b = 0, seg_h = 0, seg_sg = 0, seg_rows = 0, seg_slot = 0;
        int consumed = 0, failed = 0;
        for (int i = 0; stream_end > 0; ++i) {
            const int st = i % STAGES, bf = i & 1;
            uint8_t* stage = base + st * Lay::kStage;
            bool ok = !local_fail && mbar_wait_bounded(&full[st], (uint32_t)((i / STAGES) & 1));
            ok = ok && mbar_wait_bounded(&sbar[bf], (uint32_t)((i >> 1) & 1));
            if (cons_sync_or(!ok)) {
                failed = 1;
                consumed = i;
                break;
            }
            tc_fence_after();
            const BlockDesc bd = desc[st];
            if (bd.flags & kSegStart) {
                seg_b = bd.u / units_per_b;
                const int uidx = bd.u - seg_b * units_per_b;
                seg_h = uidx / p.sub_groups;
                seg_sg = uidx - seg_h * p.sub_groups;
                seg_rows = rs.rows(seg_sg);
                seg_slot = gw + bd.u;
                seg_unit_first = (bd.flags & kUnitFirst) != 0;
                first_block = true;
#pragma unroll
                for (int c = 0; c < NH; ++c) lp[c] = 0.f;
            }
            // V rows the block does not attend (past the length in its last
            // chunk, or in a skipped chunk) must still be finite for P V
            if (bd.bad || bd.ntok < bd.nch * kChunk) {
                for (int x = tid; x < bd.nch * kChunk * 16; x += kConsThreads) {
                    const int row = x >> 4, piece = x & 15;
                    if (row >= bd.ntok || ((bd.bad >> (row >> 4)) & 1u))
                        *reinterpret_cast<uint4*>(stage + Lay::kV + (piece >> 3) * Lay::kKVBlock +
                                                  row * 128 + ((piece & 7) << 4)) =
                            make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // ---- scores of token t for this thread's rows, masked: past the
            // length, a skipped chunk, or after the row's query token
            float v[NH];
            {
                const bool tok_ok = t < bd.ntok && !((bd.bad >> (t >> 4)) & 1u);
                // row c (query fq + c / hpu) sees position pos iff
                // pos <= len - n_queries + fq + c / hpu
                const int slack =
                    bd.len - rs.n_queries + rs.first_query(seg_sg) - (bd.k0 * kChunk + t);
                const int c_min = slack >= 0 ? 0 : -slack * rs.heads_per_unit;
                uint32_t r[NH];
                tmem_ld(lane_q + kColS * bf, r);
#pragma unroll
                for (int c = 0; c < NH; ++c)
                    v[c] = (tok_ok && cb + c >= c_min) ? __uint_as_float(r[c]) * sl2 : -INFINITY;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sfree[bf]);  // this warp has read S^T
            // ---- reference maxima: a row keeps its reference (the running
            // maximum of the blocks that moved it) unless a score of this block
            // exceeds it by more than 2^kLazyMax; the first block of a segment
            // always sets it
            bool exceed = first_block;
#pragma unroll
            for (int c = 0; c < NH; ++c) exceed |= v[c] > row_ref[cb + c] + kLazyMax;
            const bool exact = cons_sync_or(exceed);
            if (exact) {
#pragma unroll
                for (int c = 0; c < NH; ++c) {
                    const int mi = warp_max_i(ord_of(v[c]));
                    if (lane == (c & 31)) red[tq * N + cb + c] = float_of(mi);
                }
                cons_sync();
                if (tid < N) {
                    const int c = tid;
                    const float bm =
                        fmaxf(fmaxf(red[c], red[N + c]), fmaxf(red[2 * N + c], red[3 * N + c]));
                    const float m_old = first_block ? -INFINITY : row_ref[c];
                    const float m_new = fmaxf(m_old, bm);
                    row_ref[c] = m_new;
                    // weights so far, to the new reference (none yet: 0)
                    row_alpha[c] = m_old == -INFINITY ? 0.f : fast_exp2(m_old - m_new);
                }
                cons_sync();
#pragma unroll
                for (int c = 0; c < NH; ++c) lp[c] *= row_alpha[cb + c];
            }
            // ---- P^T over the consumed K: row cb + c, token t (pairs of tokens
            // per 32-bit store: even lanes take row c, odd lanes row c + 1)
            {
                const bool odd = lane & 1;
                const int tok = t & ~1;
#pragma unroll
                for (int c = 0; c < NH; c += 2) {
                    const float r0 = row_ref[cb + c], r1 = row_ref[cb + c + 1];
                    const float p0 = fast_exp2(v[c] - (r0 == -INFINITY ? 0.f : r0));
                    const float p1 = fast_exp2(v[c + 1] - (r1 == -INFINITY ? 0.f : r1));
                    lp[c] += p0;
                    lp[c + 1] += p1;
                    const float got = __shfl_xor_sync(kFull, odd ? p0 : p1, 1);
                    const float a = odd ? got : p0, bb = odd ? p1 : got;
                    const uint32_t off = swz_elem(cb + c + (odd ? 1 : 0), tok, Lay::kRowBlock);
                    if constexpr (kSplitP) {
                        uint32_t hi, lo;
                        split_bf16x2(a, bb, hi, lo);
                        *reinterpret_cast<uint32_t*>(stage + Lay::kPHi + off) = hi;
                        *reinterpret_cast<uint32_t*>(stage + Lay::kPLo + off) = lo;
                    } else {
                        *reinterpret_cast<uint32_t*>(stage + Lay::kPHi + off) =
                            Cvt<T>::pack2(a, bb);
                    }
                }
            }
            fence_proxy_async_smem();  // P^T and zeroed V rows before the tensor cores read them
            // ---- the previous block's P V product; O^T to a moved reference
            if (pv_pending) {
                if (!mbar_wait_bounded(pvbar, ph_pv)) local_fail = true;
                ph_pv ^= 1u;
                pv_pending = false;
                tc_fence_after();
            }
            if (exact && !first_block) {
                uint32_t r[NH];
                tmem_ld(lane_o, r);
#pragma unroll
                for (int c = 0; c < NH; ++c)
                    r[c] = __float_as_uint(__uint_as_float(r[c]) * row_alpha[cb + c]);
                tmem_st(lane_o, r);
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pready);  // the MMA warp issues P V of this block
            pv_pending = true;
            first_block = false;
            if (bd.flags & kSegEnd) {
                const bool okp = !local_fail && mbar_wait_bounded(pvbar, ph_pv);
                ph_pv ^= 1u;
                pv_pending = false;
                if (cons_sync_or(!okp)) {
                    failed = 1;
                    consumed = i + 1;
                    break;
                }
                tc_fence_after();
                // each row's sum of weights over the block's tokens, in a fixed order
#pragma unroll
                for (int c = 0; c < NH; ++c) {
                    float s = lp[c];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
                    if (lane == (c & 31)) red[tq * N + cb + c] = s;
                }
                cons_sync();
                if (tid < N)
                    row_alpha[tid] =
                        (red[tid] + red[N + tid]) + (red[2 * N + tid] + red[3 * N + tid]);
                cons_sync();
                // element d = t of this thread's rows: the output of a whole
                // unit, else a partial state (o, m, l) in slot u + w
                const bool whole = seg_unit_first && (bd.flags & kUnitLast) && !p.all_partials;
                float* slot = p.partials + (long long)seg_slot * partial_slot_floats(N, kD);
                uint16_t* outp = static_cast<uint16_t*>(p.out);
                uint32_t r[NH];
                tmem_ld(lane_o, r);
#pragma unroll
                for (int c = 0; c < NH; ++c) {
                    const int row = cb + c;
                    if (row < seg_rows) {
                        const float o = __uint_as_float(r[c]);
                        if (whole) {
                            const float l = row_alpha[row];
                            const float inv = l > 0.f ? 1.0f / l : 0.f;
                            outp[rs.row(seg_b, seg_h, seg_sg, row) * kD + t] =
                                (uint16_t)(Cvt<T>::pack2(o * inv, 0.f) & 0xffffu);
                        } else {
                            slot[row * kD + t] = o;
                        }
                    }
                }
                if (!whole && tid < seg_rows) {
                    // the row's reference maximum (no token seen: -inf, weights 0)
                    slot[N * kD + tid] = row_ref[tid];
                    slot[N * kD + N + tid] = row_alpha[tid];
                }
                tc_fence_before();
            }
            if (bd.flags & kLast) {
                consumed = i + 1;
                break;
            }
        }
        pdl_trigger();  // the combine may launch once every CTA's consumers are done
        if (cons_sync_or(local_fail)) failed = 1;
        if (failed && tid == 0) set_status(p.status, PKV_DEV_TIMEOUT);
        if (tid == 0) issued_slot[1] = failed ? consumed : -1;
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && issued_slot[1] >= 0) {
        // after a timeout: the copies still in flight into this CTA's memory
        for (int j = issued_slot[1]; j < issued_slot[0]; ++j)
            mbar_wait_bounded(&full[j % STAGES], (uint32_t)((j / STAGES) & 1));
    }
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
    info.threads = kThreads;
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
