// decode_mma.cuh -- tensor-core variant of the paged GQA decode kernel.
//
// Same operation, work split, partial-state format and chunk pipeline as
// decode.cuh (one warp per balanced range of 16-token chunks, a STAGES-deep
// ring of chunk buffers per warp, one mbarrier per stage), with the two
// contractions of a chunk done by warp-level tensor-core MMA
// (mma.sync m16n8k16, bf16/fp16 in, fp32 accumulate):
//
//   S[g][t]  = sum_d Q[g][d] K[t][d]      rows = the query group (padded to 16),
//                                          n = 16 tokens, k = D
//   O[g][d] += sum_t P[g][t] V[t][d]      P = exp2(S*scale*log2e - m) in the input
//                                          dtype (bf16: as hi + lo, two MMAs),
//                                          k = 16 tokens, n = D
//
// A unit of 17..32 query rows (several query tokens per sequence) runs as two
// m16 tiles in one warp: each chunk's K and V fragments are loaded once and
// used by both, and the q rows come from a per-warp buffer filled at each
// segment start.
//
// The S accumulator fragments are exactly the A fragments of the P.V product,
// so P never leaves registers.  K and V chunks are brought in by 2-D tensor
// copies (cp.async.bulk.tensor) of [16 rows x 64 elements] boxes with the
// 128-byte swizzle, which makes the ldmatrix reads of both operands free of
// bank conflicts.  A chunk costs ~32 MMAs + 16 ldmatrix + the softmax, about an
// eighth of the instructions of the CUDA-core kernel, so the warps stay far
// from issue-bound and the kernel is limited by HBM.
//
// Rows of a ragged last chunk past the context length are still copied (a box
// is always 16 rows, all inside the same page); their scores are masked to
// -inf and their V rows are zeroed in shared memory before the P.V product, so
// stale or NaN data there never reaches a result.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "decode.cuh"
#include "merge.cuh"
#include "schedule.cuh"

namespace pkv {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

template <typename T>
struct Mma;

template <>
struct Mma<__nv_bfloat16> {
    static __device__ __forceinline__ void run(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};

template <>
struct Mma<__half> {
    static __device__ __forceinline__ void run(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};

// Byte offset of (row r, 16-byte column j) inside one [16 x 128 B] box written
// by a 128-byte-swizzled tensor copy into a 1024-byte aligned buffer.
__device__ __forceinline__ uint32_t swz128(int r, int j) {
    return (uint32_t)(r * 128 + ((j ^ (r & 7)) << 4));
}

// Query rows of one warp: one m16 tile (GS <= 16), or two (GS = 32: units of
// 17..32 rows, each K/V chunk used by both tiles).
template <int GS>
constexpr int mma_tiles() {
    return GS > 16 ? 2 : 1;
}

// Shared memory of one CTA: every warp's ring of K/V stages first (each stage a
// multiple of 1 KiB, as the 128-byte swizzle needs), then every warp's q
// space -- one slot per stage, filled with the segment's first chunk (one
// tile), or one buffer filled at each segment start (two tiles) -- then the
// mbarriers (one per stage, plus the q buffer's).
template <int D, int GS, int STAGES, int WARPS>
struct MmaLayout {
    static constexpr int kTiles = mma_tiles<GS>();
    static constexpr int kBoxes = D / 64;                       // [16 x 64] boxes per K or V chunk
    static constexpr int kBoxBytes = kChunk * 128;              // 2 KiB
    static constexpr int kStageBytes = 2 * kBoxes * kBoxBytes;  // K boxes then V boxes
    static constexpr int kWarpKV = STAGES * kStageBytes;
    static constexpr int kQBytes = GS * D * 2;
    static constexpr int kQRowBytes = D * 2 + 16;  // two tiles: rows padded by 16 bytes
    static constexpr int kWarpQ = kTiles == 1 ? STAGES * kQBytes : GS * kQRowBytes;
    static constexpr int kWarpBars = STAGES + (kTiles == 1 ? 0 : 1);
    static constexpr int kOffQ = WARPS * kWarpKV;
    static constexpr int kOffBar = ((kOffQ + WARPS * kWarpQ) + 15) / 16 * 16;
    static constexpr int kBytes = kOffBar + WARPS * kWarpBars * 8 + 1024;  // + alignment slack
};

template <typename T, int D, int GS, int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32)
decode_mma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap) {
    using Lay = MmaLayout<D, GS, STAGES, WARPS>;
    constexpr int TILES = Lay::kTiles;
    constexpr int KSTEPS = D / 16;      // k-steps of the q.k product
    constexpr int NT = D / 8;           // n-tiles of the P.V product
    constexpr bool kTwoHalves = GS > 8; // query rows 8..15 of a tile in use
    constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;  // P as bf16 hi + lo
    static_assert(GS <= 16 || GS == 32, "one m16 tile of query rows, or two");
    constexpr int kQRowBytes = Lay::kQRowBytes;  // two tiles: padded q rows
    static_assert(STAGES <= 4, "tiles of the schedule are at least 4 chunks long");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;  // 1 KiB alignment for the swizzle
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t* base = smem_raw + pad;
    uint8_t* wsm = base + warp * Lay::kWarpKV;                 // this warp's K/V stages
    const uint32_t wsm_u32 = raw + pad + warp * Lay::kWarpKV;
    T* sq = reinterpret_cast<T*>(base + Lay::kOffQ + warp * Lay::kWarpQ);
    uint64_t* bar = reinterpret_cast<uint64_t*>(base + Lay::kOffBar + warp * Lay::kWarpBars * 8);
    uint64_t* qbar = bar + STAGES;  // two tiles: the q buffer's barrier

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < Lay::kWarpBars; ++s) mbar_init(&bar[s], 1);
        fence_barrier_init();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap))
                     : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vmap))
                     : "memory");
    }
    __syncwarp();
    pdl_wait();

    const int nw = p.hdr->num_workers;
    const int gw = blockIdx.x * WARPS + warp;
    const int all_warps = gridDim.x * WARPS;
    if (gw >= nw) {
        zero_empty_sequences(p, D, gw, all_warps, lane);
        return;
    }
    WorkStream ws;
    ws.init(p, lane, gw);
    if (ws.stream_end == 0) {
        zero_empty_sequences(p, D, gw, all_warps, lane);
        return;
    }

    const int units_per_b = ws.units_per_b;
    // K/V lines are read once per call: they go first, so that what is read
    // again (page table, schedule, partial states) stays in L2
    const uint64_t kv_policy = l2_evict_first_policy();
    const int g_lo = lane >> 2;          // query row of c0/c1 (c2/c3: g_lo + 8)
    const int tq = (lane & 3) * 2;       // first token (or d) column of this lane in a tile
    const T* __restrict__ qg = static_cast<const T*>(p.q);

    // Issue the copies of stream position j into stage j % STAGES; false past
    // the end of the stream.
    auto issue = [&](int j) -> bool {
        if (!ws.covered(p, j)) return false;
        const ChunkDesc d = ws.fetch(j);
        const bool seg_start = ws.seg_start(j, d);
        if (lane == 0) {
            const int st = j % STAGES;
            int b = 0, h = 0, sg = 0, nrows = 0;
            if (TILES == 1 && seg_start) {
                b = d.u / units_per_b;
                const int uidx = d.u - b * units_per_b;
                h = uidx / p.sub_groups;
                sg = uidx - h * p.sub_groups;
                nrows = p.rows.rows(sg);
            }
            const uint32_t kv_bytes = d.off >= 0 ? (uint32_t)Lay::kStageBytes : 0u;
            const uint32_t q_bytes = TILES == 1 && seg_start ? (uint32_t)(nrows * D * 2) : 0u;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bar[st], kv_bytes + q_bytes);
            if (kv_bytes) {
                uint8_t* stage = wsm + st * Lay::kStageBytes;
                const int y = (int)d.off;  // first pool row of the chunk
#pragma unroll
                for (int bx = 0; bx < Lay::kBoxes; ++bx) {
                    tma_load_2d_hint(stage + bx * Lay::kBoxBytes, &kmap, bx * 64, y, &bar[st],
                                     kv_policy);
                    tma_load_2d_hint(stage + (Lay::kBoxes + bx) * Lay::kBoxBytes, &vmap, bx * 64,
                                     y, &bar[st], kv_policy);
                }
            }
            if (q_bytes) {
                // the unit's rows: one block of heads_per_unit contiguous q rows per token
                const int hpu = p.rows.heads_per_unit;
                for (int r = 0; r < nrows; r += hpu)
                    bulk_g2s(sq + st * GS * D + r * D, qg + p.rows.row(b, h, sg, r) * D,
                             (uint32_t)(hpu * D * 2), &bar[st]);
            }
        }
        return true;
    };

    int issued = 0;
    while (issued < STAGES && issue(issued)) ++issued;
    zero_empty_sequences(p, D, gw, all_warps, lane);  // while the first copies are in flight

    uint32_t qa[TILES == 1 ? KSTEPS : 1][4];  // one tile: A fragments of Q (rows g_lo, g_lo+8)
    float o[TILES][NT][4];      // O accumulators (c0,c1: row g_lo; c2,c3: row g_lo+8 of a tile)
    float m_lo[TILES], l_lo[TILES], m_hi[TILES], l_hi[TILES];
    int jq_lo[TILES], jq_hi[TILES];  // query tokens of rows g_lo and g_lo + 8 of each tile
#pragma unroll
    for (int t = 0; t < TILES; ++t) {
        m_lo[t] = m_hi[t] = -INFINITY;
        l_lo[t] = l_hi[t] = 0.f;
        jq_lo[t] = jq_hi[t] = 0;
    }
    bool seg_whole_start = false;
    int seg_slot = 0, seg_first = 0;
    int seg_rows = GS;              // rows of the segment's unit in use
    uint32_t qphase = 0;            // two tiles: phase of the q buffer's barrier
    // split segments to report after the loop (at most two: the range's first and last)
    int npend = 0;
    PendingMerge pend0 = {0, 0, 0, 0}, pend1 = {0, 0, 0, 0};

    // A copy never landed: report it, wait (bounded) for the copies still in
    // flight into this warp's buffers (stream positions from .. issued-1).
    auto give_up = [&](int from) {
        if (lane == 0) set_status(p.status, PKV_DEV_TIMEOUT);
        for (int j = from; j < issued; ++j)
            mbar_wait_bounded(&bar[j % STAGES], (uint32_t)((j / STAGES) & 1));
    };

    for (int i = 0; i < ws.stream_end; ++i) {
        ws.consumer_at(p, i, STAGES + 1);
        const ChunkDesc d = ws.fetch(i);
        const int st = i % STAGES;
        const bool seg_start = ws.seg_start(i, d);
        if (seg_start) {
            const int b = d.u / units_per_b;
            const int uidx = d.u - b * units_per_b;
            const int h = uidx / p.sub_groups;
            const int sg = uidx - h * p.sub_groups;
            seg_rows = p.rows.rows(sg);
#pragma unroll
            for (int t = 0; t < TILES; ++t) {
                jq_lo[t] = p.rows.query(sg, 16 * t + g_lo);
                jq_hi[t] = p.rows.query(sg, 16 * t + g_lo + 8);
            }
            if constexpr (TILES > 1) {
                // the unit's q rows into this warp's buffer, one row per lane
                // (padded rows: conflict-free ldmatrix); the previous segment's
                // reads of the buffer precede these writes in program order
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(qbar, (uint32_t)(seg_rows * D * 2));
                __syncwarp();
                if (lane < seg_rows)
                    bulk_g2s(reinterpret_cast<uint8_t*>(sq) + lane * kQRowBytes,
                             qg + p.rows.row(b, h, sg, lane) * D, (uint32_t)(D * 2), qbar);
            }
        }
        if (!mbar_wait_bounded(&bar[st], (uint32_t)((i / STAGES) & 1))) {
            if (TILES > 1 && seg_start) mbar_wait_bounded(qbar, qphase);
            give_up(i + 1);
            return;
        }
        if (seg_start) {
            seg_slot = ws.slot_base + d.u;
            seg_first = i;
            if constexpr (TILES == 1) {
                // A fragments of Q: a0 (row g, k tq..tq+1), a1 (row g+8), a2 (k+8), a3
                const uint32_t* q32 = reinterpret_cast<const uint32_t*>(sq + st * GS * D);
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const int c0 = (kk * 16 + tq) / 2, c1 = (kk * 16 + 8 + tq) / 2;
                    qa[kk][0] = g_lo < seg_rows ? q32[g_lo * (D / 2) + c0] : 0u;
                    qa[kk][2] = g_lo < seg_rows ? q32[g_lo * (D / 2) + c1] : 0u;
                    if constexpr (kTwoHalves) {
                        qa[kk][1] = g_lo + 8 < seg_rows ? q32[(g_lo + 8) * (D / 2) + c0] : 0u;
                        qa[kk][3] = g_lo + 8 < seg_rows ? q32[(g_lo + 8) * (D / 2) + c1] : 0u;
                    } else {
                        qa[kk][1] = 0u;
                        qa[kk][3] = 0u;
                    }
                }
            } else {
                if (!mbar_wait_bounded(qbar, qphase)) {
                    give_up(i + 1);
                    return;
                }
                qphase ^= 1u;
            }
#pragma unroll
            for (int t = 0; t < TILES; ++t) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    o[t][nt][0] = o[t][nt][1] = o[t][nt][2] = o[t][nt][3] = 0.f;
                m_lo[t] = m_hi[t] = -INFINITY;
                l_lo[t] = l_hi[t] = 0.f;
            }
            seg_whole_start = (d.k == 0);
        }

        if (d.off >= 0) {
            const uint32_t kst = wsm_u32 + st * Lay::kStageBytes;
            const uint32_t vst = kst + Lay::kBoxes * Lay::kBoxBytes;
            const int nvalid = d.nvalid;
            if (nvalid < kChunk) {
                // zero the V rows past the context (stale or NaN page contents)
                uint4* vrows = reinterpret_cast<uint4*>(wsm + st * Lay::kStageBytes +
                                                        Lay::kBoxes * Lay::kBoxBytes);
                const int nz = (kChunk - nvalid) * 8 * Lay::kBoxes;  // 16-byte vectors
                for (int z = lane; z < nz; z += 32) {
                    const int bx = z / ((kChunk - nvalid) * 8);
                    const int rem = z - bx * (kChunk - nvalid) * 8;
                    const int row = nvalid + rem / 8;
                    vrows[(bx * Lay::kBoxBytes + row * 128) / 16 + (rem & 7)] =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
            // ---- S = Q K^T : two n-tiles (tokens 0-7, 8-15); one tile: even/odd k
            // chains, two tiles: the tiles' chains interleave (one chain each) ----
            constexpr int KCH = TILES == 1 ? 2 : 1;
            float s[TILES][2][KCH][4];
#pragma unroll
            for (int t = 0; t < TILES; ++t)
#pragma unroll
                for (int a = 0; a < 2; ++a)
#pragma unroll
                    for (int b = 0; b < KCH; ++b)
                        s[t][a][b][0] = s[t][a][b][1] = s[t][a][b][2] = s[t][a][b][3] = 0.f;
            // ldmatrix x4 rows: lane -> matrix mi = lane/8, row r = lane%8;
            // matrices: (tok 0-7, d+0..7), (tok 0-7, d+8..15), (tok 8-15, d+0..7), (tok 8-15, d+8..15)
            const int mi = lane >> 3, rr = lane & 7;
            const int k_tok = (mi >> 1) * 8 + rr;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                const int dcol = kk * 16 + (mi & 1) * 8;      // first element of the 16-byte row piece
                const int bx = dcol / 64;
                const uint32_t addr = kst + bx * Lay::kBoxBytes + swz128(k_tok, (dcol % 64) / 8);
                uint32_t kb[4];
                ldsm_x4(addr, kb);
                if constexpr (TILES == 1) {
                    Mma<T>::run(s[0][0][kk & 1], qa[kk], kb[0], kb[1]);
                    Mma<T>::run(s[0][1][kk & 1], qa[kk], kb[2], kb[3]);
                } else {
#pragma unroll
                    for (int t = 0; t < TILES; ++t) {
                        // A fragments of tile t: matrices (rows 0-7, k 0-7), (rows 8-15,
                        // k 0-7), (rows 0-7, k 8-15), (rows 8-15, k 8-15)
                        const int qrow = 16 * t + (mi & 1) * 8 + rr;
                        uint32_t qf[4];
                        ldsm_x4(smem_u32(sq) + qrow * kQRowBytes + (kk * 16 + (mi >> 1) * 8) * 2,
                                qf);
                        Mma<T>::run(s[t][0][kk % KCH], qf, kb[0], kb[1]);
                        Mma<T>::run(s[t][1][kk % KCH], qf, kb[2], kb[3]);
                    }
                }
            }
            // ---- online softmax (base 2) on rows g_lo (c0,c1) and g_lo+8 (c2,c3) ----
            uint32_t pa[TILES][4];        // A fragments of P (its bf16 high part when split)
            uint32_t pl[TILES][4];        // bf16 residual p - hi (split only)
#pragma unroll
            for (int t = 0; t < TILES; ++t) {
                pl[t][0] = pl[t][1] = pl[t][2] = pl[t][3] = 0u;
                // causal limit of several query tokens: query j of a unit row sees
                // tokens up to len - n_queries + j (no limit inside the chunk when 1)
                int lim_lo = kChunk, lim_hi = kChunk;
                if (p.rows.n_queries > 1) {
                    const int base_tok = d.len - p.rows.n_queries - d.k * kChunk;
                    lim_lo = base_tok + jq_lo[t];
                    lim_hi = base_tok + jq_hi[t];
                }
                float sc[2][4];
#pragma unroll
                for (int a = 0; a < 2; ++a)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int tt = a * 8 + tq + (e & 1);
                        const float v =
                            (KCH == 2 ? s[t][a][0][e] + s[t][a][KCH - 1][e] : s[t][a][0][e]) *
                            p.scale_log2;
                        sc[a][e] = (tt < nvalid && tt <= (e < 2 ? lim_lo : lim_hi)) ? v : -INFINITY;
                    }
                {
                    float mx = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
                    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
                    const float m_new = fmaxf(m_lo[t], mx);
                    // a causal row with no token yet (m_new = -inf) takes weights 0
                    const float m_ref = m_new == -INFINITY ? 0.f : m_new;
                    const float alpha = fast_exp2(m_lo[t] - m_ref);
                    const float p00 = fast_exp2(sc[0][0] - m_ref), p01 = fast_exp2(sc[0][1] - m_ref);
                    const float p10 = fast_exp2(sc[1][0] - m_ref), p11 = fast_exp2(sc[1][1] - m_ref);
                    float rs = (p00 + p01) + (p10 + p11);
                    rs += __shfl_xor_sync(kFull, rs, 1);
                    rs += __shfl_xor_sync(kFull, rs, 2);
                    l_lo[t] = l_lo[t] * alpha + rs;
                    m_lo[t] = m_new;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        o[t][nt][0] *= alpha;
                        o[t][nt][1] *= alpha;
                    }
                    if constexpr (kSplitP) {
                        split_bf16x2(p00, p01, pa[t][0], pl[t][0]);
                        split_bf16x2(p10, p11, pa[t][2], pl[t][2]);
                    } else {
                        pa[t][0] = Cvt<T>::pack2(p00, p01);
                        pa[t][2] = Cvt<T>::pack2(p10, p11);
                    }
                }
                if constexpr (kTwoHalves) {
                    float mx = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
                    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
                    const float m_new = fmaxf(m_hi[t], mx);
                    // a causal row with no token yet (m_new = -inf) takes weights 0
                    const float m_ref = m_new == -INFINITY ? 0.f : m_new;
                    const float alpha = fast_exp2(m_hi[t] - m_ref);
                    const float p00 = fast_exp2(sc[0][2] - m_ref), p01 = fast_exp2(sc[0][3] - m_ref);
                    const float p10 = fast_exp2(sc[1][2] - m_ref), p11 = fast_exp2(sc[1][3] - m_ref);
                    float rs = (p00 + p01) + (p10 + p11);
                    rs += __shfl_xor_sync(kFull, rs, 1);
                    rs += __shfl_xor_sync(kFull, rs, 2);
                    l_hi[t] = l_hi[t] * alpha + rs;
                    m_hi[t] = m_new;
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        o[t][nt][2] *= alpha;
                        o[t][nt][3] *= alpha;
                    }
                    if constexpr (kSplitP) {
                        split_bf16x2(p00, p01, pa[t][1], pl[t][1]);
                        split_bf16x2(p10, p11, pa[t][3], pl[t][3]);
                    } else {
                        pa[t][1] = Cvt<T>::pack2(p00, p01);
                        pa[t][3] = Cvt<T>::pack2(p10, p11);
                    }
                } else {
                    pa[t][1] = pa[t][3] = 0u;
                }
            }
            // ---- O += P V : ldmatrix.trans gives the V^T fragments ----
            // x4 matrices: (tok 0-7, d 8nt..), (tok 8-15, d 8nt..), (tok 0-7, d 8nt+8..), (tok 8-15, ..)
            const int v_tok = (mi & 1) * 8 + rr;
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                const int dcol = np * 16 + (mi >> 1) * 8;
                const int bx = dcol / 64;
                const uint32_t addr = vst + bx * Lay::kBoxBytes + swz128(v_tok, (dcol % 64) / 8);
                uint32_t vb[4];
                ldsm_x4_trans(addr, vb);
#pragma unroll
                for (int t = 0; t < TILES; ++t) {
                    Mma<T>::run(o[t][2 * np], pa[t], vb[0], vb[1]);
                    Mma<T>::run(o[t][2 * np + 1], pa[t], vb[2], vb[3]);
                    if constexpr (kSplitP) {
                        Mma<T>::run(o[t][2 * np], pl[t], vb[0], vb[1]);
                        Mma<T>::run(o[t][2 * np + 1], pl[t], vb[2], vb[3]);
                    }
                }
            }
        }

        const bool seg_end = ws.seg_end(i, d);
        if (seg_end) {
            const bool whole = seg_whole_start && (d.k == d.nch - 1) && !p.all_partials;
            const int b = d.u / units_per_b;
            const int uidx = d.u - b * units_per_b;
            const int h = uidx / p.sub_groups;
            const int sg = uidx - h * p.sub_groups;
#pragma unroll
            for (int t = 0; t < TILES; ++t)
#pragma unroll
            for (int half = 0; half < (kTwoHalves ? 2 : 1); ++half) {
                const int g = 16 * t + g_lo + half * 8;
                const float l = half ? l_hi[t] : l_lo[t];
                const float m = half ? m_hi[t] : m_lo[t];
                if (g < seg_rows) {
                    if (whole) {
                        T* outp = static_cast<T*>(p.out) + p.rows.row(b, h, sg, g) * D;
                        const float inv = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            *reinterpret_cast<uint32_t*>(outp + nt * 8 + tq) =
                                Cvt<T>::pack2(o[t][nt][2 * half] * inv,
                                              o[t][nt][2 * half + 1] * inv);
                        }
                    } else {
                        float* dst = p.partials + (long long)seg_slot * partial_slot_floats(GS, D);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            *reinterpret_cast<float2*>(dst + g * D + nt * 8 + tq) =
                                make_float2(o[t][nt][2 * half], o[t][nt][2 * half + 1]);
                        }
                        if ((lane & 3) == 0) {
                            dst[GS * D + g] = m;
                            dst[GS * D + GS + g] = l;
                        }
                    }
                }
            }
            if (!whole && p.unit_done) {
                const PendingMerge pmg = {d.u, ws.range_f0 + i - d.k, d.nch, i - seg_first + 1};
                if (npend == 0) pend0 = pmg; else pend1 = pmg;
                ++npend;
            }
        }
        __syncwarp();
        // refill: positions up to i + STAGES (stage i % STAGES is free again)
        while (issued <= i + STAGES && issue(issued)) ++issued;
    }
    // the next kernel (combine, or the prefix pass) may launch once every CTA
    // has a warp past its chunk stream: earlier, its CTAs only wait beside
    // these (measured slower, cold and warm)
    pdl_trigger();
    if (npend > 0)
        finish_pending<T, D, GS>(p, npend, pend0, pend1, ws.sw, ws.r, lane);
}

template <int D, int GS>
constexpr int pick_mma_stages() {
    // as many stages as keep a 4-warp CTA within 112 KiB (two CTAs per SM)
    return MmaLayout<D, GS, 4, 4>::kBytes <= 112 * 1024
               ? 4
               : (MmaLayout<D, GS, 3, 4>::kBytes <= 112 * 1024 ? 3 : 2);
}

template <typename T, int D, int GS>
DecodeMmaInfo make_decode_mma_info() {
    constexpr int W = 4;
    constexpr int S = pick_mma_stages<D, GS>();
    DecodeMmaInfo info;
    info.fn = decode_mma_kernel<T, D, GS, W, S>;
    info.warps = W;
    info.stages = S;
    info.smem_bytes = MmaLayout<D, GS, S, W>::kBytes;
    info.gs = GS;
    return info;
}

}  // namespace pkv
