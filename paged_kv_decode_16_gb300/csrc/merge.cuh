// merge.cuh -- merging the partial states of a unit that several workers
// processed (split-K reduction of flash-decoding), and the other writes that
// complete the output.
//
// A segment s of unit u leaves (o_s, m_s, l_s) per query row: o_s the
// unnormalised weighted sum of V rows, m_s the running maximum of the scores
// in base-2 units, l_s the sum of 2^(score - m_s).  The merged output is
//     out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,   M = max_s m_s.
//
// Two passes, in an order that depends on nothing but the segment count:
// a warp per row finds M and the denominator (lane t takes segments t, t+32,
// ... in order; the lane sums meet in a fixed butterfly), then each output
// vector sums its weighted o_s in segment order straight from the slots.  The
// stand-alone combine kernels (merge_rows, a warp per row) and the decode
// kernels (the warp that finishes the last segment of a unit merges it after
// its own chunk stream: merge_rows_warp, several rows per warp) do the same
// arithmetic in the same order, so the two paths give the same bits.
#pragma once

#include "common.cuh"

namespace pkv {

// The segments of unit u, whose chunks are [a, a + nch) of the flattened
// batch: one per worker whose range meets them, in slots u + w for w from the
// worker holding chunk a to the one holding chunk a + nch - 1 (schedule.cuh).
struct UnitSegments {
    int count_;
    long long base;
    __device__ __forceinline__ int count() const { return count_; }
    __device__ __forceinline__ long long slot(int s) const { return base + s; }
};

__device__ __forceinline__ UnitSegments unit_segments(int sw, int r, int u, int a, int nch) {
    const int w0 = worker_of(a, sw, r), w1 = worker_of(a + nch - 1, sw, r);
    UnitSegments sg;
    sg.count_ = w1 - w0 + 1;
    sg.base = (long long)u + w0;
    return sg;
}

// Segment s of a unit in the usual slot layout (stride floats per slot: o at
// [g*D], m at [gs*D + g], l at [gs*D + gs + g]), slots base, base + 1, ...
struct SlotSegs {
    const float* partials;
    long long base;
    int stride, gs, d;
    __device__ __forceinline__ const float* o(int s, int g) const {
        return partials + (base + s) * stride + (long long)g * d;
    }
    __device__ __forceinline__ const float* m(int s, int g) const {
        return partials + (base + s) * stride + (long long)gs * d + g;
    }
    __device__ __forceinline__ const float* l(int s, int g) const { return m(s, g) + gs; }
    // output vector v (floats 4v .. 4v+3) of row g
    __device__ __forceinline__ const float4* o4(int s, int g, int v) const {
        return reinterpret_cast<const float4*>(o(s, g)) + v;
    }
};

// Segment s of a shared-prefix row tile (prefix_umma.cu): slots base, base + 1,
// ... of 128 rows each: o [128][d], then m [128], then l [128].
struct TileSegs {
    static constexpr int kRows = 128;
    const float* partials;
    long long base;
    int d;
    __device__ __forceinline__ const float* slot(int s) const {
        return partials + (base + s) * (long long)(kRows * d + 2 * kRows);
    }
    __device__ __forceinline__ const float4* o4(int s, int g, int v) const {
        return reinterpret_cast<const float4*>(slot(s) + (long long)g * d) + v;
    }
    __device__ __forceinline__ const float* m(int s, int g) const { return slot(s) + kRows * d + g; }
    __device__ __forceinline__ const float* l(int s, int g) const { return m(s, g) + kRows; }
};

// Row r + off of Segs as row r (one row of a unit merged on its own).
template <class Segs>
struct RowShift {
    const Segs& sg;
    int off;
    __device__ __forceinline__ const float4* o4(int s, int g, int v) const {
        return sg.o4(s, g + off, v);
    }
    __device__ __forceinline__ const float* m(int s, int g) const { return sg.m(s, g + off); }
    __device__ __forceinline__ const float* l(int s, int g) const { return sg.l(s, g + off); }
};

constexpr int kMergeBlock = 8;  // segments whose loads are in flight together

struct MergeRow {
    float M, den;
    float w;  // ns <= 32: the weight of segment `lane` (0 past ns)
};

__device__ __forceinline__ float merge_weight(float m, float M) {
    // no finite score in the segment (m = -inf): weight 0
    return m == -INFINITY ? 0.f : exp2f(m - M);
}

// Pass 1 for row g of ns segments; one warp, every lane gets M and den.  Up
// to 32 segments lane t holds segment t's m and l (one round of loads) and
// keeps its weight for pass 2; beyond, lane t walks segments t, t+32, ...
// twice.  Both give the same sums: lane t adds its segments' w_s l_s in order.
template <bool kUnroll = true, class Segs>
__device__ __forceinline__ MergeRow merge_row(const Segs& sg, int ns, int g, int lane) {
    float M = -INFINITY, den = 0.f, wl = 0.f;
    if (ns <= 32) {
        const float m = lane < ns ? __ldcg(sg.m(lane, g)) : -INFINITY;
        const float l = lane < ns ? __ldcg(sg.l(lane, g)) : 0.f;
        M = m;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
        wl = merge_weight(m, M);
        den = fmaf(wl, l, 0.f);
    } else {
        // kUnroll: unrolled 8 times, so that the loads of several segments go
        // out before the first use; else the compiler's choice (measured 1 us
        // faster in the shared-prefix merge, whose rows rarely have more than
        // 32 segments).  Each lane's operations stay in segment order.
        if constexpr (kUnroll) {
#pragma unroll 8
            for (int s = lane; s < ns; s += 32) M = fmaxf(M, __ldcg(sg.m(s, g)));
        } else {
            for (int s = lane; s < ns; s += 32) M = fmaxf(M, __ldcg(sg.m(s, g)));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
        if constexpr (kUnroll) {
#pragma unroll 8
            for (int s = lane; s < ns; s += 32)
                den = fmaf(merge_weight(__ldcg(sg.m(s, g)), M), __ldcg(sg.l(s, g)), den);
        } else {
            for (int s = lane; s < ns; s += 32)
                den = fmaf(merge_weight(__ldcg(sg.m(s, g)), M), __ldcg(sg.l(s, g)), den);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(kFull, den, o);
    return MergeRow{M, den, wl};
}

// Outputs 4*d4 .. 4*d4+3 of a merged row (out_row: its first output).
template <typename T, int D>
__device__ __forceinline__ void merge_store(const float4& acc, float den, int d4, T* out_row) {
    const float inv = den > 0.f ? 1.0f / den : 0.f;
    uint2 w2;
    w2.x = Cvt<T>::pack2(acc.x * inv, acc.y * inv);
    w2.y = Cvt<T>::pack2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(out_row + d4 * 4) = w2;
}

// Rows of more than 32 segments (one sequence split over many workers): pass
// 2 sums the o vectors of groups of kMergeGroup segments -- each group in
// segment order -- and adds the groups into kMergeSlots slots (slot j takes
// groups j, j + kMergeSlots, ...), then the slots in order, starting from 0.
// A combine CTA of kMergeSlots warps gives each slot its own warp (a group's
// loads all in flight); a single warp walks the slots itself, in the same
// order, so both give the same bits.
constexpr int kMergeGroup = 16;
constexpr int kMergeSlots = 8;

// Slot j of row g: its groups' weighted sums, added in order.
template <int D, class Segs>
__device__ __forceinline__ float4 merge_slot(const Segs& sg, int ns, int g, float M, int slot,
                                             int lane) {
    const bool act = lane < D / 4;
    float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int grp = slot; grp * kMergeGroup < ns; grp += kMergeSlots) {
        const int s0 = grp * kMergeGroup;
        float4 v[kMergeGroup];
        float w[kMergeGroup];
#pragma unroll
        for (int j = 0; j < kMergeGroup; ++j) {
            const int s = s0 + j;
            v[j] = act && s < ns ? __ldcg(sg.o4(s, g, lane)) : make_float4(0.f, 0.f, 0.f, 0.f);
            w[j] = s < ns ? merge_weight(__ldcg(sg.m(s, g)), M) : 0.f;
        }
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < kMergeGroup; ++j) {
            if (s0 + j >= ns) break;
            acc.x = fmaf(w[j], v[j].x, acc.x);
            acc.y = fmaf(w[j], v[j].y, acc.y);
            acc.z = fmaf(w[j], v[j].z, acc.z);
            acc.w = fmaf(w[j], v[j].w, acc.w);
        }
        part.x += acc.x;
        part.y += acc.y;
        part.z += acc.z;
        part.w += acc.w;
    }
    return part;
}

// merge_slot with a group's loads in two halves (8 in flight): the same
// multiply-adds in the same order, so the same bits, with fewer registers
// (the combine kernels' occupancy).
template <int D, class Segs>
__device__ __forceinline__ float4 merge_slot_lean(const Segs& sg, int ns, int g, float M,
                                                  int slot, int lane) {
    constexpr int H = kMergeGroup / 2;
    const bool act = lane < D / 4;
    float4 part = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int grp = slot; grp * kMergeGroup < ns; grp += kMergeSlots) {
        const int s0 = grp * kMergeGroup;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float4 v[H];
            float w[H];
#pragma unroll
            for (int j = 0; j < H; ++j) {
                const int s = s0 + hh * H + j;
                v[j] = act && s < ns ? __ldcg(sg.o4(s, g, lane)) : make_float4(0.f, 0.f, 0.f, 0.f);
                w[j] = s < ns ? merge_weight(__ldcg(sg.m(s, g)), M) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < H; ++j) {
                if (s0 + hh * H + j >= ns) break;
                acc.x = fmaf(w[j], v[j].x, acc.x);
                acc.y = fmaf(w[j], v[j].y, acc.y);
                acc.z = fmaf(w[j], v[j].z, acc.z);
                acc.w = fmaf(w[j], v[j].w, acc.w);
            }
        }
        part.x += acc.x;
        part.y += acc.y;
        part.z += acc.z;
        part.w += acc.w;
    }
    return part;
}

// merge_rows' pass 2 for up to 32 segments: segment order, loads in blocks.
template <typename T, int D, class Segs, class RowOut>
__device__ __forceinline__ void merge_rows_upto32(const Segs& sg, int ns, int nrows, int warp,
                                                  int nwarps, int lane, const RowOut& out_rows) {
    constexpr int Q = D / 4;
    for (int g = warp; g < nrows; g += nwarps) {
        const MergeRow mr = merge_row(sg, ns, g, lane);
        const bool act = lane < Q;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        // blocks of kMergeBlock segments: every load of a block is issued
        // before the first multiply-add waits on one
        for (int s0 = 0; s0 < ns; s0 += kMergeBlock) {
            float4 v[kMergeBlock];
            float w[kMergeBlock];
#pragma unroll
            for (int j = 0; j < kMergeBlock; ++j) {
                const int s = s0 + j;
                v[j] = act && s < ns
                           ? __ldcg(sg.o4(s, g, lane))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
                w[j] = s >= ns ? 0.f : __shfl_sync(kFull, mr.w, s & 31);
            }
#pragma unroll
            for (int j = 0; j < kMergeBlock; ++j) {
                if (s0 + j >= ns) break;
                x.x = fmaf(w[j], v[j].x, x.x);
                x.y = fmaf(w[j], v[j].y, x.y);
                x.z = fmaf(w[j], v[j].z, x.z);
                x.w = fmaf(w[j], v[j].w, x.w);
            }
        }
        if (act) merge_store<T, D>(x, mr.den, lane, out_rows(g));
    }
}

// Merge rows [0, nrows) of a unit with the warps of a CTA (warp w of nwarps
// takes rows w, w + nwarps, ...); out_rows(g) gives row g's output.  Pass 2:
// lane t sums output vector t of the row, sum_s w_s o_s in segment order (up
// to 32 segments), or in the grouped order above, a warp walking the slots.
template <typename T, int D, class Segs, class RowOut>
__device__ __forceinline__ void merge_rows(const Segs& sg, int ns, int nrows, int warp, int nwarps,
                                           int lane, const RowOut& out_rows) {
    constexpr int Q = D / 4;  // output vectors per row
    static_assert(Q <= 32, "one vector per lane");
    if (ns > 32) {
        for (int g = warp; g < nrows; g += nwarps) {
            const MergeRow mr = merge_row(sg, ns, g, lane);
            float4 total = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j = 0; j < kMergeSlots; ++j) {
                const float4 q = merge_slot<D>(sg, ns, g, mr.M, j, lane);
                total.x += q.x;
                total.y += q.y;
                total.z += q.z;
                total.w += q.w;
            }
            if (lane < Q) merge_store<T, D>(total, mr.den, lane, out_rows(g));
        }
        return;
    }
    merge_rows_upto32<T, D>(sg, ns, nrows, warp, nwarps, lane, out_rows);
}

// Merge rows [0, nrows) in segment order for any segment count (warp w of
// nwarps takes rows w, w + nwarps, ...; beyond 32 segments each weight comes
// from its own load).  For a merge whose bits no other path has to match (the
// shared-prefix call's): it keeps that kernel's register count.
template <typename T, int D, class Segs, class RowOut>
__device__ __forceinline__ void merge_rows_seq(const Segs& sg, int ns, int nrows, int warp,
                                               int nwarps, int lane, const RowOut& out_rows) {
    constexpr int Q = D / 4;
    for (int g = warp; g < nrows; g += nwarps) {
        const MergeRow mr = merge_row<false>(sg, ns, g, lane);
        const bool act = lane < Q;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 0; s0 < ns; s0 += kMergeBlock) {
            float4 v[kMergeBlock];
            float w[kMergeBlock];
#pragma unroll
            for (int j = 0; j < kMergeBlock; ++j) {
                const int s = s0 + j;
                v[j] = act && s < ns ? __ldcg(sg.o4(s, g, lane)) : make_float4(0.f, 0.f, 0.f, 0.f);
                w[j] = s >= ns ? 0.f
                       : ns <= 32 ? __shfl_sync(kFull, mr.w, s & 31)
                                  : merge_weight(__ldcg(sg.m(s, g)), mr.M);
            }
#pragma unroll
            for (int j = 0; j < kMergeBlock; ++j) {
                if (s0 + j >= ns) break;
                x.x = fmaf(w[j], v[j].x, x.x);
                x.y = fmaf(w[j], v[j].y, x.y);
                x.z = fmaf(w[j], v[j].z, x.z);
                x.w = fmaf(w[j], v[j].w, x.w);
            }
        }
        if (act) merge_store<T, D>(x, mr.den, lane, out_rows(g));
    }
}

// merge_rows for a combine CTA of kMergeSlots warps (every warp calls it):
// rows of more than 32 segments are taken kCtaRows at a time -- warps
// 0 .. kCtaRows-1 find the rows' maxima and denominators, then every warp sums
// (row, slot) items (item i: row i / kMergeSlots, slot i % kMergeSlots), then
// warp r adds row r's slots in order -- merge_rows' bits.
template <typename T, int D, class Segs, class RowOut>
__device__ __forceinline__ void merge_rows_cta(const Segs& sg, int ns, int nrows, int warp,
                                               int lane, const RowOut& out_rows) {
    if (ns <= 32) {
        merge_rows_upto32<T, D>(sg, ns, nrows, warp, kMergeSlots, lane, out_rows);
        return;
    }
    constexpr int kCtaRows = 2;
    __shared__ float4 s_part[kCtaRows][kMergeSlots][32];
    __shared__ float s_M[kCtaRows], s_den[kCtaRows];
    for (int g0 = 0; g0 < nrows; g0 += kCtaRows) {
        const int rb = min(kCtaRows, nrows - g0);
        if (warp < rb) {
            const MergeRow mr = merge_row(sg, ns, g0 + warp, lane);
            if (lane == 0) {
                s_M[warp] = mr.M;
                s_den[warp] = mr.den;
            }
        }
        __syncthreads();
        for (int it = warp; it < rb * kMergeSlots; it += kMergeSlots) {
            const int r = it / kMergeSlots, j = it - r * kMergeSlots;
            s_part[r][j][lane] = merge_slot_lean<D>(sg, ns, g0 + r, s_M[r], j, lane);
        }
        __syncthreads();
        if (warp < rb) {
            float4 total = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < kMergeSlots; ++j) {
                const float4 q = s_part[warp][j][lane];
                total.x += q.x;
                total.y += q.y;
                total.z += q.z;
                total.w += q.w;
            }
            if (lane < D / 4) merge_store<T, D>(total, s_den[warp], lane, out_rows(g0 + warp));
        }
        __syncthreads();
    }
}

// merge_rows for one warp and up to 32 segments, kRowBatch rows at a time:
// the m / l loads of all the batch's rows go out together, then their o loads
// kWarpBlock segments at a time, so up to kWarpBlock segments cost the rows
// two rounds of loads instead of two each.  Every row's arithmetic is
// merge_row's and merge_rows' (the same butterflies, the same multiply-add
// order over the segments), so the results are the same bits.  (The decode
// kernel calls this; its loads in flight are sized to keep the kernel's
// register count.)
constexpr int kRowBatch = 4;
constexpr int kWarpBlock = 4;

template <typename T, int D, class Segs, class RowOut>
__device__ __forceinline__ void merge_rows_warp(const Segs& sg, int ns, int nrows, int lane,
                                                const RowOut& out_rows) {
    constexpr int Q = D / 4;
    static_assert(Q <= 32, "one vector per lane");
    if (ns > 32) {
        merge_rows<T, D>(sg, ns, nrows, 0, 1, lane, out_rows);
        return;
    }
    const bool act = lane < Q;
    for (int g0 = 0; g0 < nrows; g0 += kRowBatch) {
        float m[kRowBatch], l[kRowBatch], wl[kRowBatch], den[kRowBatch];
#pragma unroll
        for (int r = 0; r < kRowBatch; ++r) {
            const bool ok = lane < ns && g0 + r < nrows;
            m[r] = ok ? __ldcg(sg.m(lane, g0 + r)) : -INFINITY;
            l[r] = ok ? __ldcg(sg.l(lane, g0 + r)) : 0.f;
        }
#pragma unroll
        for (int r = 0; r < kRowBatch; ++r) {
            float M = m[r];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
            wl[r] = merge_weight(m[r], M);
            float d = fmaf(wl[r], l[r], 0.f);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(kFull, d, o);
            den[r] = d;
        }
        float4 x[kRowBatch];
#pragma unroll
        for (int r = 0; r < kRowBatch; ++r) x[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 0; s0 < ns; s0 += kWarpBlock) {
            float4 v[kRowBatch][kWarpBlock];
#pragma unroll
            for (int r = 0; r < kRowBatch; ++r)
#pragma unroll
                for (int j = 0; j < kWarpBlock; ++j) {
                    const int s = s0 + j;
                    v[r][j] = act && s < ns && g0 + r < nrows
                                  ? __ldcg(sg.o4(s, g0 + r, lane))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
            for (int r = 0; r < kRowBatch; ++r)
#pragma unroll
                for (int j = 0; j < kWarpBlock; ++j) {
                    const int s = s0 + j;
                    const float w = __shfl_sync(kFull, wl[r], s & 31);
                    if (s < ns) {
                        x[r].x = fmaf(w, v[r][j].x, x[r].x);
                        x[r].y = fmaf(w, v[r][j].y, x[r].y);
                        x[r].z = fmaf(w, v[r][j].z, x[r].z);
                        x[r].w = fmaf(w, v[r][j].w, x[r].w);
                    }
                }
        }
#pragma unroll
        for (int r = 0; r < kRowBatch; ++r)
            if (act && g0 + r < nrows) merge_store<T, D>(x[r], den[r], lane, out_rows(g0 + r));
    }
}

// A split segment whose arrival a decode warp reports after its main loop.
struct PendingMerge {
    int u;       // unit
    int a;       // the unit's first chunk in the flattened order
    int nch;     // chunks of the unit
    int chunks;  // chunks of this warp's segment
};

// Merge split unit `pm` in the decode warp that finished its last segment.
// Warp-collective.
template <typename T, int D, int GS>
__device__ __noinline__ void merge_unit(const DecodeParams& p, const PendingMerge& pm, int sw,
                                        int r, int lane) {
    const UnitSegments us = unit_segments(sw, r, pm.u, pm.a, pm.nch);
    const SlotSegs sg{p.partials, us.base, partial_slot_floats(GS, D), GS, D};
    const int units_per_b = p.n_kv_heads * p.sub_groups;
    const int b = pm.u / units_per_b;
    const int uidx = pm.u - b * units_per_b;
    const int h = uidx / p.sub_groups;
    const int sgi = uidx - h * p.sub_groups;
    T* out = static_cast<T*>(p.out);
    merge_rows_warp<T, D>(sg, us.count(), p.rows.rows(sgi), lane,
                          [&](int g) { return out + p.rows.row(b, h, sgi, g) * D; });
}

// After a decode warp's main loop: report its split segments (at most two,
// the range's first and last) to the units' counters and merge every unit
// whose count this completes.  Lane 0's acquire-release adds publish the
// warp's partial stores (ordered before them by the warp barrier) and, for
// the last arriver, make the other segments' stores visible.  Warp-collective.
template <typename T, int D, int GS>
__device__ __forceinline__ void finish_pending(const DecodeParams& p, int npend,
                                               const PendingMerge& p0, const PendingMerge& p1,
                                               int sw, int r, int lane) {
    __syncwarp();
    int old0 = 0, old1 = 0;
    if (lane == 0) {
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
                     : "=r"(old0)
                     : "l"(p.unit_done + p0.u), "r"(p0.chunks)
                     : "memory");
        if (npend > 1)
            asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
                         : "=r"(old1)
                         : "l"(p.unit_done + p1.u), "r"(p1.chunks)
                         : "memory");
    }
    old0 = __shfl_sync(kFull, old0, 0);
    old1 = __shfl_sync(kFull, old1, 0);
    __syncwarp();  // lane 0's acquire before the merges below
    if (old0 + p0.chunks == p0.nch) merge_unit<T, D, GS>(p, p0, sw, r, lane);
    if (npend > 1 && old1 + p1.chunks == p1.nch) merge_unit<T, D, GS>(p, p1, sw, r, lane);
}

// Output rows of sequences with no tokens are zeros (no worker visits them).
// Warp gw of nwarps checks 32 sequences at a time and clears the empty ones.
// Warp-collective.
__device__ __forceinline__ void zero_empty_sequences(const DecodeParams& p, int head_dim, int gw,
                                                     int nwarps, int lane) {
    const long long vecs = (long long)p.rows.n_queries * p.n_q_heads * head_dim * 2 / 16;  // per seq
    for (long long b0 = (long long)gw * 32; b0 < p.batch; b0 += (long long)nwarps * 32) {
        const long long b = b0 + lane;
        const bool empty = b < p.batch && __ldg(p.lens_eff + b) == 0;
        unsigned mask = __ballot_sync(kFull, empty);
        while (mask) {
            const int e = __ffs(mask) - 1;
            mask &= mask - 1;
            uint4* dst = reinterpret_cast<uint4*>(p.out) + (b0 + e) * vecs;
            for (long long x = lane; x < vecs; x += 32) dst[x] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

}  // namespace pkv
