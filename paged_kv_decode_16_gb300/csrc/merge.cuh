// merge.cuh -- merging the partial states of a unit that several workers
// processed (split-K reduction of flash-decoding), and the other writes that
// complete the output.
//
// A segment s of unit u leaves (o_s, m_s, l_s) per query head: o_s the
// unnormalised weighted sum of V rows, m_s the running maximum of the scores
// in base-2 units, l_s the sum of 2^(score - m_s).  The merged output is
//     out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,   M = max_s m_s.
//
// The stand-alone combine kernel and the decode kernels (the warp that
// finishes the last segment of a unit merges it, after its own chunk stream)
// fold the same batches of segments with merge_weights / merge_accumulate,
// so the two paths give the same bits.
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

// Per-head running state of a merge, kept in shared memory next to the
// staged slots: maximum so far (base 2), denominator so far, and the factor
// that rescales the numerators of earlier batches in this batch.
struct MergeHead {
    float M, den, a, pad;
};

// Step 1 of folding a batch of cnt <= 32 staged segments (slot stride
// `stride` floats: o at [g*D], m at [gs*D + g], l at [gs*D + gs + g]) into a
// unit's merge: per head, lane s owns segment s; the batch maximum joins the
// running one, lane s turns m_s into its weight 2^(m_s - M) in place, and the
// weighted l_s are summed into the denominator.  One warp; heads[] holds the
// running state (M = -inf, den = 0 before the first batch).
__device__ __forceinline__ void merge_weights(float* slots, int stride, int cnt, int gs, int D,
                                              MergeHead* heads, int lane) {
    const int n = gs * D;
    for (int g = 0; g < gs; ++g) {
        float* mp = slots + lane * stride + n + g;
        const float m = lane < cnt ? *mp : -INFINITY;
        float mb = m;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, o));
        const float m_old = heads[g].M;
        const float mn = fmaxf(m_old, mb);
        // no finite score yet (mn = -inf): every weight and factor is 0
        const float w = (m == -INFINITY) ? 0.f : exp2f(m - mn);
        const float a = (m_old == -INFINITY) ? 0.f : exp2f(m_old - mn);
        float dl = lane < cnt ? w * mp[gs] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dl += __shfl_xor_sync(kFull, dl, o);
        if (lane < cnt) *mp = w;
        __syncwarp();
        if (lane == 0) {
            heads[g].M = mn;
            heads[g].den = fmaf(heads[g].den, a, dl);
            heads[g].a = a;
        }
        __syncwarp();
    }
}

// Step 2: output vector (g, d4) (4 consecutive outputs of head g) folds the
// batch in, in segment order: acc = acc * a_g + sum_s w_s o_s.
template <int D>
__device__ __forceinline__ void merge_accumulate(const float* slots, int stride, int cnt, int gs,
                                                 const MergeHead* heads, int g, int d4,
                                                 float4& acc) {
    const int n = gs * D;
    const float a = heads[g].a;
    float4 x = make_float4(acc.x * a, acc.y * a, acc.z * a, acc.w * a);
    for (int s = 0; s < cnt; ++s) {
        const float* pp = slots + s * stride;
        const float w = pp[n + g];
        const float4 v = *reinterpret_cast<const float4*>(pp + g * D + d4 * 4);
        x.x = fmaf(w, v.x, x.x);
        x.y = fmaf(w, v.y, x.y);
        x.z = fmaf(w, v.z, x.z);
        x.w = fmaf(w, v.w, x.w);
    }
    acc = x;
}

// Outputs 4*d4 .. 4*d4+3 of unit row g, whose output row starts at out_row.
template <typename T, int D>
__device__ __forceinline__ void merge_store(const float4& acc, const MergeHead* heads, int g,
                                            int d4, T* out_row) {
    const float den = heads[g].den;
    const float inv = den > 0.f ? 1.0f / den : 0.f;
    uint2 w2;
    w2.x = Cvt<T>::pack2(acc.x * inv, acc.y * inv);
    w2.y = Cvt<T>::pack2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(out_row + d4 * 4) = w2;
}

// Bytes of shared memory a merge needs: merge_batch staged slots, then the
// per-head state (16 heads at most).
__host__ __device__ constexpr int merge_smem_bytes(int merge_batch, int gs, int d) {
    return merge_batch * partial_slot_floats(gs, d) * 4 + 16 * (int)sizeof(MergeHead);
}

// A split segment whose arrival a decode warp reports after its main loop.
struct PendingMerge {
    int u;       // unit
    int a;       // the unit's first chunk in the flattened order
    int nch;     // chunks of the unit
    int chunks;  // chunks of this warp's segment
};

// 16-byte asynchronous copy global -> shared through L2 (cp.async.cg), and
// the wait for every copy this thread issued.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Merge split unit `pm` in the decode warp that finished its last segment:
// copy the segments' partial states, merge_batch slots at a time, into the
// warp's stage buffers (idle once its chunk stream is done; `stage` holds
// merge_smem_bytes(merge_batch, GS, D)) and fold them there.  Warp-collective.
template <typename T, int D, int GS>
__device__ __noinline__ void merge_staged(const DecodeParams& p, const PendingMerge& pm, int sw,
                                          int r, uint8_t* stage, int lane) {
    constexpr int stride = partial_slot_floats(GS, D);
    constexpr int vps = stride / 4;  // 16-byte vectors per slot
    constexpr int Q = D / 4;
    constexpr int KPL = (GS * Q + 31) / 32;  // output vectors per lane
    const UnitSegments sg = unit_segments(sw, r, pm.u, pm.a, pm.nch);
    const int ns = sg.count();
    float* slots = reinterpret_cast<float*>(stage);
    MergeHead* heads = reinterpret_cast<MergeHead*>(stage + p.merge_batch * stride * 4);
    if (lane < GS) heads[lane] = MergeHead{-INFINITY, 0.f, 0.f, 0.f};
    float4 acc[KPL];
#pragma unroll
    for (int k = 0; k < KPL; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < ns; s0 += p.merge_batch) {
        const int cnt = min(p.merge_batch, ns - s0);
        __syncwarp();  // every lane is done with the previous batch
        fence_proxy_async_smem();  // after the stage buffers' tensor copies
        for (int v = lane; v < cnt * vps; v += 32) {
            const int s = v / vps;
            cp_async16(slots + v * 4, p.partials + sg.slot(s0 + s) * stride + (v - s * vps) * 4);
        }
        cp_async_wait_all();
        __syncwarp();
        merge_weights(slots, stride, cnt, GS, D, heads, lane);
#pragma unroll
        for (int k = 0; k < KPL; ++k) {
            const int it = k * 32 + lane;
            if (it < GS * Q)
                merge_accumulate<D>(slots, stride, cnt, GS, heads, it / Q, it % Q, acc[k]);
        }
    }
    const int units_per_b = p.n_kv_heads * p.sub_groups;
    const int b = pm.u / units_per_b;
    const int uidx = pm.u - b * units_per_b;
    const int h = uidx / p.sub_groups;
    const int sgi = uidx - h * p.sub_groups;
#pragma unroll
    for (int k = 0; k < KPL; ++k) {
        const int it = k * 32 + lane;
        if (it < GS * Q) {
            const int g = it / Q;
            if (g < p.rows.rows(sgi))
                merge_store<T, D>(acc[k], heads, g, it % Q,
                                  static_cast<T*>(p.out) + p.rows.row(b, h, sgi, g) * D);
        }
    }
}

// After a decode warp's main loop: report its split segments (at most two,
// the range's first and last) to the units' counters and merge every unit
// whose count this completes.  Lane 0's acquire-release adds publish the
// warp's partial stores (ordered before them by the warp barrier) and, for
// the last arriver, make the other segments' stores visible.  Warp-collective.
template <typename T, int D, int GS>
__device__ __forceinline__ void finish_pending(const DecodeParams& p, int npend,
                                               const PendingMerge& p0, const PendingMerge& p1,
                                               int sw, int r, uint8_t* stage, int lane) {
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
    if (old0 + p0.chunks == p0.nch) merge_staged<T, D, GS>(p, p0, sw, r, stage, lane);
    if (npend > 1 && old1 + p1.chunks == p1.nch) merge_staged<T, D, GS>(p, p1, sw, r, stage, lane);
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
