// decode.cuh -- single-query GQA decode attention over a paged KV cache.
//
// Operation (CacheIR, "Boundaries": multi-batch page-table decode attention
// with GQA mapping; TorchInferno, "Custom Kernels": paged_decode_attention):
// for each sequence b and query head hq = h*G + g,
//     out[b][hq] = softmax_t(scale * q[b][hq] . k_t) . v_t ,  t < L_b,
// with k_t / v_t read from page table[b][t / P], row t % P, KV head h.
//
// GB300 design
// ------------
// * Unit of work: a chunk = 16 consecutive tokens of one (sequence, KV head).
//   In the [page][kv_head][slot][dim] pool a chunk is one contiguous block of
//   16*D*2 bytes (4 KB at D=128), fetched by ONE bulk async copy (TMA engine,
//   cp.async.bulk) for K and one for V; ragged last chunks copy only their
//   valid rows.  Rows past the context length are never loaded nor touched.
// * Balanced split (flash-decoding split-K, stream-K style): all chunks of the
//   batch are laid end to end (sequence-major, then KV head, then chunk); each
//   worker -- one warp -- takes an equal contiguous static range of most of
//   them, then small dynamic tiles of the rest from a shared counter
//   (schedule.cuh).  Long contexts are split over many warps, short ones packed
//   into one.  A (sequence, KV head) inside one piece is finished in place; one
//   that straddles pieces leaves fp32 partial states (m, l, o), merged by the
//   combine kernel.
// * Warps never wait on each other: each owns a STAGES-deep ring of chunk
//   buffers in shared memory with one mbarrier per stage; lane 0 refills a
//   stage (K, V, and q when a new unit starts) right after the warp consumed
//   it, so STAGES chunks per warp are always in flight.
// * The whole GQA group is served by the warp from one read of each K/V row:
//   every K/V element is loaded into registers once and used by all G heads.
//   Lane (r, c): token r of each 2- or 4-token step, 8-element slice c of D.
//   q.k partial sums of the G heads are combined across the D/8 lanes of a
//   token with a reduce-scatter butterfly (each shuffle halves the values in
//   flight), leaving each lane one full score.  Online softmax in base 2
//   (q pre-scaled by scale*log2 e), fp32 accumulation of o.
#pragma once

#include "common.cuh"
#include "merge.cuh"
#include "schedule.cuh"

namespace pkv {

// Reduce-scatter of a[GP] across the lanes that share a token (lane bits
// below LPT).  Level with mask M halves the live values; the lane with bit M
// set keeps the upper half.  Returns the complete sum of value index
// gsel(lane) = sum_lvl bit_lvl(lane) * (GP >> (lvl + 1)).
template <int N, int MASK, int LPT>
struct ReduceScatter {
    template <int GP>
    static __device__ __forceinline__ float run(float (&a)[GP], int lane) {
        if constexpr (N == 1) {
            float x = a[0];
#pragma unroll
            for (int m = MASK; m < LPT; m <<= 1) x += __shfl_xor_sync(kFull, x, m);
            return x;
        } else {
            static_assert(MASK < LPT, "query group wider than the lanes of one token");
            const bool upper = (lane & MASK) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                const float send = upper ? a[i] : a[i + N / 2];
                const float keep = upper ? a[i + N / 2] : a[i];
                a[i] = keep + __shfl_xor_sync(kFull, send, MASK);
            }
            return ReduceScatter<N / 2, MASK * 2, LPT>::run(a, lane);
        }
    }
};

template <int D, int GS, int STAGES>
struct DecodeLayout {
    static constexpr int kGP = next_pow2(GS);
    static constexpr int kChunkBytes = kChunk * D * 2;  // one K (or V) chunk
    static constexpr int kQBytes = GS * D * 2;          // q rows of one unit
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + STAGES * kChunkBytes;
    static constexpr int kOffQ = kOffV + STAGES * kChunkBytes;
    static constexpr int kOffP = kOffQ + STAGES * kQBytes;        // float [16][GP]
    static constexpr int kOffA = kOffP + kChunk * kGP * 4;        // float [GP] alpha
    static constexpr int kOffL = kOffA + kGP * 4;                 // float [GP] l
    static constexpr int kOffM = kOffL + kGP * 4;                 // float [GP] m
    static constexpr int kOffBar = ((kOffM + kGP * 4) + 15) / 16 * 16;
    static constexpr int kWarpBytes = ((kOffBar + STAGES * 8) + 127) / 128 * 128;
    static_assert(kQBytes % 16 == 0 && kChunkBytes % 16 == 0, "bulk copies need 16 B sizes");
};

template <typename T, int D, int GS, int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32)
decode_kernel(const DecodeParams p) {
    using Lay = DecodeLayout<D, GS, STAGES>;
    constexpr int LPT = D / 8;          // lanes per token (8 elements each)
    constexpr int TPS = 32 / LPT;       // tokens per step
    constexpr int STEPS = kChunk / TPS; // steps per chunk
    constexpr int GP = Lay::kGP;
    constexpr int RLOG = ilog2(GP);
    static_assert(GP <= LPT, "group too large for this head dim");
    static_assert(STAGES <= 4, "tiles of the schedule are at least 4 chunks long");

    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t* wsm = smem + warp * Lay::kWarpBytes;
    T* sk = reinterpret_cast<T*>(wsm + Lay::kOffK);
    T* sv = reinterpret_cast<T*>(wsm + Lay::kOffV);
    T* sq = reinterpret_cast<T*>(wsm + Lay::kOffQ);
    float* ps = reinterpret_cast<float*>(wsm + Lay::kOffP);
    float* pa = reinterpret_cast<float*>(wsm + Lay::kOffA);
    float* pl = reinterpret_cast<float*>(wsm + Lay::kOffL);
    float* pm = reinterpret_cast<float*>(wsm + Lay::kOffM);
    uint64_t* bar = reinterpret_cast<uint64_t*>(wsm + Lay::kOffBar);

    const int c = lane & (LPT - 1);     // D slice
    const int r = lane / LPT;           // token within a step
    int gsel = 0;
#pragma unroll
    for (int lvl = 0; lvl < RLOG; ++lvl) gsel += ((c >> lvl) & 1) * (GP >> (lvl + 1));
    const bool writer = (c >> RLOG) == 0 && gsel < GS;  // one lane per (token, head)

    const T* __restrict__ kpool = static_cast<const T*>(p.k_pool);
    const T* __restrict__ vpool = static_cast<const T*>(p.v_pool);
    const T* __restrict__ qg = static_cast<const T*>(p.q);

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < STAGES; ++s) mbar_init(&bar[s], 1);
        fence_barrier_init();
    }
    __syncwarp();
    // the plan (previous kernel of the stream) must be complete from here on
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

    // Issue the copies of stream position j into stage j % STAGES; false past
    // the end of the stream.
    auto issue = [&](int j) -> bool {
        if (!ws.covered(p, j)) return false;
        const ChunkDesc d = ws.fetch(j);
        const bool seg_start = ws.seg_start(j, d);
        if (lane == 0) {
            const int st = j % STAGES;
            const uint32_t kv_bytes = d.off >= 0 ? (uint32_t)d.nvalid * D * 2 : 0u;
            const uint32_t q_bytes = seg_start ? (uint32_t)Lay::kQBytes : 0u;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bar[st], 2 * kv_bytes + q_bytes);
            if (kv_bytes) {
                bulk_g2s_hint(sk + st * kChunk * D, kpool + d.off * D, kv_bytes, &bar[st],
                              kv_policy);
                bulk_g2s_hint(sv + st * kChunk * D, vpool + d.off * D, kv_bytes, &bar[st],
                              kv_policy);
            }
            if (q_bytes) {
                const int b = d.u / units_per_b;
                const int uidx = d.u - b * units_per_b;
                const int h = uidx / p.sub_groups;
                const int sg = uidx - h * p.sub_groups;
                const long long qrow = (long long)b * p.n_q_heads + h * p.group + sg * GS;
                bulk_g2s(sq + st * GS * D, qg + qrow * D, q_bytes, &bar[st]);
            }
        }
        return true;
    };

    int issued = 0;
    while (issued < STAGES && issue(issued)) ++issued;
    zero_empty_sequences(p, D, gw, all_warps, lane);  // while the first copies are in flight

    float qf[GS][8];
    float o[GS][8];
    float m_run = -INFINITY, l_run = 0.f;
    bool seg_whole_start = false;
    int seg_slot = 0, seg_first = 0;
    // split segments to report after the loop (at most two: the range's first and last)
    int npend = 0;
    PendingMerge pend0 = {0, 0, 0, 0}, pend1 = {0, 0, 0, 0};

    for (int i = 0; i < ws.stream_end; ++i) {
        ws.consumer_at(p, i, STAGES + 1);
        const ChunkDesc d = ws.fetch(i);
        const int st = i % STAGES;
        if (!mbar_wait_bounded(&bar[st], (uint32_t)((i / STAGES) & 1))) {
            // A copy never landed.  Report it, wait (bounded) for the copies
            // still in flight into this warp's buffers, and stop.
            if (lane == 0) set_status(p.status, PKV_DEV_TIMEOUT);
            for (int j = i + 1; j < issued; ++j)
                mbar_wait_bounded(&bar[j % STAGES], (uint32_t)((j / STAGES) & 1));
            return;
        }
        const bool seg_start = ws.seg_start(i, d);
        if (seg_start) {
            seg_slot = ws.slot_base + d.u;
            seg_first = i;
            const T* qs = sq + st * GS * D;
#pragma unroll
            for (int g = 0; g < GS; ++g) {
                const uint4 raw = *reinterpret_cast<const uint4*>(qs + g * D + c * 8);
                float f[8];
                Cvt<T>::unpack8(raw, f);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    qf[g][j] = f[j] * p.scale_log2;
                    o[g][j] = 0.f;
                }
            }
            m_run = -INFINITY;
            l_run = 0.f;
            seg_whole_start = (d.k == 0);
        }

        if (d.off >= 0) {
            const T* kc = sk + st * kChunk * D;
            const T* vc = sv + st * kChunk * D;
            const int nvalid = d.nvalid;
            // ---- scores of this chunk: lane holds s[t = s*TPS + r][gsel] ----
            float sc[STEPS];
#pragma unroll
            for (int s = 0; s < STEPS; ++s) {
                const int t = s * TPS + r;
                const uint4 raw = *reinterpret_cast<const uint4*>(kc + t * D + c * 8);
                float kf[8];
                Cvt<T>::unpack8(raw, kf);
                float a[GP];
#pragma unroll
                for (int g = 0; g < GP; ++g) a[g] = 0.f;
#pragma unroll
                for (int g = 0; g < GS; ++g) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) a[g] = fmaf(qf[g][j], kf[j], a[g]);
                }
                const float sv_ = ReduceScatter<GP, 1, LPT>::run(a, lane);
                sc[s] = (t < nvalid) ? sv_ : -INFINITY;
            }
            // ---- online softmax (base 2) ----
            float cmax = sc[0];
#pragma unroll
            for (int s = 1; s < STEPS; ++s) cmax = fmaxf(cmax, sc[s]);
#pragma unroll
            for (int m = LPT; m < 32; m <<= 1) cmax = fmaxf(cmax, __shfl_xor_sync(kFull, cmax, m));
            const float m_new = fmaxf(m_run, cmax);
            const float alpha = fast_exp2(m_run - m_new);
            float psum = 0.f;
#pragma unroll
            for (int s = 0; s < STEPS; ++s) {
                sc[s] = fast_exp2(sc[s] - m_new);
                psum += sc[s];
            }
#pragma unroll
            for (int m = LPT; m < 32; m <<= 1) psum += __shfl_xor_sync(kFull, psum, m);
            l_run = l_run * alpha + psum;
            m_run = m_new;
            if (writer) {
#pragma unroll
                for (int s = 0; s < STEPS; ++s) ps[(s * TPS + r) * GP + gsel] = sc[s];
                if (r == 0) pa[gsel] = alpha;
            }
            __syncwarp();
            // ---- o = o * alpha + P V ----
#pragma unroll
            for (int g = 0; g < GS; ++g) {
                const float al = pa[g];
#pragma unroll
                for (int j = 0; j < 8; ++j) o[g][j] *= al;
            }
#pragma unroll
            for (int s = 0; s < STEPS; ++s) {
                const int t = s * TPS + r;
                if (t < nvalid) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(vc + t * D + c * 8);
                    float vf[8];
                    Cvt<T>::unpack8(raw, vf);
                    float pr[GP];
#pragma unroll
                    for (int g4 = 0; g4 < GP; g4 += 4) {
                        if constexpr (GP >= 4) {
                            const float4 x = *reinterpret_cast<const float4*>(ps + t * GP + g4);
                            pr[g4] = x.x; pr[g4 + 1] = x.y; pr[g4 + 2] = x.z; pr[g4 + 3] = x.w;
                        }
                    }
                    if constexpr (GP < 4) {
#pragma unroll
                        for (int g = 0; g < GP; ++g) pr[g] = ps[t * GP + g];
                    }
#pragma unroll
                    for (int g = 0; g < GS; ++g) {
#pragma unroll
                        for (int j = 0; j < 8; ++j) o[g][j] = fmaf(pr[g], vf[j], o[g][j]);
                    }
                }
            }
            __syncwarp();
        }

        const bool seg_end = ws.seg_end(i, d);
        if (seg_end) {
            const bool whole = seg_whole_start && (d.k == d.nch - 1) && !p.all_partials;
            // tokens were split over the r lanes: sum their o
#pragma unroll
            for (int g = 0; g < GS; ++g) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
#pragma unroll
                    for (int m = LPT; m < 32; m <<= 1)
                        o[g][j] += __shfl_xor_sync(kFull, o[g][j], m);
                }
            }
            if (writer && r == 0) {
                pl[gsel] = l_run;
                pm[gsel] = m_run;
            }
            __syncwarp();
            const int b = d.u / units_per_b;
            const int uidx = d.u - b * units_per_b;
            const int h = uidx / p.sub_groups;
            const int sg = uidx - h * p.sub_groups;
            const long long hq0 = (long long)b * p.n_q_heads + h * p.group + sg * GS;
            if (whole) {
                if (r == 0) {
                    T* outp = static_cast<T*>(p.out);
#pragma unroll
                    for (int g = 0; g < GS; ++g) {
                        const float l = pl[g];
                        const float inv = l > 0.f ? 1.0f / l : 0.f;
                        uint4 w;
                        w.x = Cvt<T>::pack2(o[g][0] * inv, o[g][1] * inv);
                        w.y = Cvt<T>::pack2(o[g][2] * inv, o[g][3] * inv);
                        w.z = Cvt<T>::pack2(o[g][4] * inv, o[g][5] * inv);
                        w.w = Cvt<T>::pack2(o[g][6] * inv, o[g][7] * inv);
                        *reinterpret_cast<uint4*>(outp + (hq0 + g) * D + c * 8) = w;
                    }
                }
            } else {
                float* dst = p.partials + (long long)seg_slot * partial_slot_floats(GS, D);
                if (r == 0) {
#pragma unroll
                    for (int g = 0; g < GS; ++g) {
                        float4* q4 = reinterpret_cast<float4*>(dst + g * D + c * 8);
                        q4[0] = make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
                        q4[1] = make_float4(o[g][4], o[g][5], o[g][6], o[g][7]);
                    }
                }
                if (lane < GS) {
                    dst[GS * D + lane] = pm[lane];
                    dst[GS * D + GS + lane] = pl[lane];
                }
                if (p.unit_done) {
                    const PendingMerge pmg = {d.u, ws.range_f0 + i - d.k, d.nch, i - seg_first + 1};
                    if (npend == 0) pend0 = pmg; else pend1 = pmg;
                    ++npend;
                }
            }
            __syncwarp();
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
constexpr int pick_stages() {
    // as many stages as keep 4 warps' buffers within ~112 KB (two CTAs per SM)
    return DecodeLayout<D, GS, 4>::kWarpBytes * 4 <= 112 * 1024
               ? 4
               : (DecodeLayout<D, GS, 3>::kWarpBytes * 4 <= 112 * 1024 ? 3 : 2);
}

template <typename T, int D, int GS>
DecodeKernelInfo make_decode_info() {
    constexpr int W = 4;
    constexpr int S = pick_stages<D, GS>();
    DecodeKernelInfo info;
    info.fn = decode_kernel<T, D, GS, W, S>;
    info.warps = W;
    info.stages = S;
    info.smem_bytes = DecodeLayout<D, GS, S>::kWarpBytes * W;
    info.gs = GS;
    return info;
}

}  // namespace pkv
