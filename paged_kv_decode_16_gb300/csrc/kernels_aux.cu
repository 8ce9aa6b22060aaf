// kernels_aux.cu -- the small kernels around the decode kernel: plan (with an
// optional fused KV append), combine, stand-alone KV append and gather.  They
// move kilobytes; their cost is latency, so each one issues its independent
// loads together and is launched with programmatic dependent launch so that
// its launch overlaps the previous kernel's tail.
#include <limits.h>

#include "common.cuh"
#include "kernels_aux.cuh"
#include "merge.cuh"

namespace pkv {

// ---------------------------------------------------------------------------
// KV append, one 16-byte vector per call (TorchInferno, "OpenAI-Compatible
// Serving" knob list: KV-append kernel).  Returns PKV_DEV_* bits for a
// skipped row (reported once per row, by its vector 0 of head 0).
// ---------------------------------------------------------------------------
// A caller input: from page-locked host memory with ld.global.cv (a line the
// GPU may hold is fetched again), else a plain load.
template <bool kHost, typename V>
__device__ __forceinline__ V ld_input(const V* p) {
    if constexpr (kHost) return __ldcv(p);
    else return *p;
}

template <bool kHost>
__device__ __forceinline__ uint32_t append_vec(const AppendArgs& a, long long idx) {
    const int vec = (int)(idx % a.vecs);
    const long long row = idx / a.vecs;  // b * Hkv + h
    const int b = (int)(row / a.n_kv_heads);
    const int h = (int)(row - (long long)b * a.n_kv_heads);
    // the new rows' loads go out with the position's (independent of it)
    const uint4 kv = ld_input<kHost>(a.k_new + row * a.vecs + vec);
    const uint4 vv = ld_input<kHost>(a.v_new + row * a.vecs + vec);
    const int p = ld_input<kHost>(a.positions + b);
    if (p < 0) return 0;  // padded batch slot: never writes
    const int pi = p / a.page_size;
    if (pi >= a.table_stride) return (vec == 0 && h == 0) ? PKV_DEV_BAD_LEN : 0u;
    const int page = ld_input<kHost>(a.table + (long long)b * a.table_stride + pi);
    if (page < 0 || page >= a.num_pages) return (vec == 0 && h == 0) ? PKV_DEV_BAD_PAGE : 0u;
    const long long dst =
        (((long long)page * a.n_kv_heads + h) * a.page_size + p % a.page_size) * a.vecs + vec;
    a.k_pool[dst] = kv;
    a.v_pool[dst] = vv;
    return 0;
}

// ---------------------------------------------------------------------------
// Rotary embedding before the append (CacheIR, "Compiler Example": rope(q, k)
// feeds attention; TorchInferno, "OpenAI-Compatible Serving" knob list: a
// fused decode rotary + KV append kernel).  Rotate-half pairing: element i of
// a head pairs with i + D/2 and turns by pos * theta^(-2i/D).  The angle is
// formed in double (pos times the host's theta^(-2i/D)) and reduced modulo
// 2 pi with fused multiply-adds, which keeps it exact to double precision for
// any int32 position; cos / sin of the reduced angle and the rotation itself
// run in fp32 (fused multiply-add) and are rounded once to the element type.
// ---------------------------------------------------------------------------
template <typename T>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float to(__nv_bfloat16 x) { return __bfloat162float(x); }
    static __device__ __forceinline__ __nv_bfloat16 from(float x) { return __float2bfloat16_rn(x); }
};
template <>
struct Elem<__half> {
    static __device__ __forceinline__ float to(__half x) { return __half2float(x); }
    static __device__ __forceinline__ __half from(float x) { return __float2half_rn(x); }
};

// cos and sin of pos * inv: the product in double, reduced by the nearest
// multiple of 2 pi (2 pi as a double plus its remainder), then fp32.
__device__ __forceinline__ void rope_cos_sin(int pos, double inv, float* c, float* s) {
    const double two_pi_hi = 6.283185307179586;       // 2 pi rounded to double
    const double two_pi_lo = 2.4492935982947064e-16;  // 2 pi - two_pi_hi
    const double ang = (double)pos * inv;
    const double k = rint(ang * (1.0 / two_pi_hi));
    double r = fma(-k, two_pi_hi, ang);
    r = fma(-k, two_pi_lo, r);
    sincosf((float)r, s, c);
}

// Rotate the 8 pairs held by lo (first-half elements 8j .. 8j+7) and hi (their
// partners), with cos / sin of those pairs' angles.
template <typename T>
__device__ __forceinline__ void rotate8(uint4& lo, uint4& hi, const float* c, const float* s) {
    T* a = reinterpret_cast<T*>(&lo);
    T* b = reinterpret_cast<T*>(&hi);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float x0 = Elem<T>::to(a[e]), x1 = Elem<T>::to(b[e]);
        a[e] = Elem<T>::from(fmaf(x0, c[e], -x1 * s[e]));
        b[e] = Elem<T>::from(fmaf(x1, c[e], x0 * s[e]));
    }
}

// 1 / rms of a row for the norm before the rotation: the row's hv lanes
// (consecutive, hv a power of two dividing 32) each hold 8 element pairs.  The
// square of a 16-bit value is exact in fp32 and each lane adds its 16 squares
// with a compensated (Kahan) sum; the lane sums meet in a butterfly; sqrt and
// the division are correctly rounded.  A few fp32 roundings in all, far below
// an ulp of the 16-bit result (fp64 would cost more on this part).
template <typename T>
__device__ __forceinline__ float row_inv_rms(const uint4& lo, const uint4& hi, int hv,
                                             int head_dim, float eps) {
    const T* a = reinterpret_cast<const T*>(&lo);
    const T* b = reinterpret_cast<const T*>(&hi);
    float sum = 0.f, comp = 0.f;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const float x = Elem<T>::to(e < 8 ? a[e] : b[e - 8]);
        const float y = x * x - comp;
        const float t = sum + y;
        comp = (t - sum) - y;
        sum = t;
    }
    const int lane = threadIdx.x & 31;
    const unsigned mask = ((1u << hv) - 1u) << (lane & ~(hv - 1));
    for (int o = hv / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(mask, sum, o);
    return 1.0f / sqrtf(sum / (float)head_dim + eps);
}

// Scale 8 element pairs by inv_rms and their weights, then rotate them as
// rotate8 does.
template <typename T>
__device__ __forceinline__ void norm_rotate8(uint4& lo, uint4& hi, const float* c, const float* s,
                                             const float* wlo, const float* whi, float inv_rms) {
    T* a = reinterpret_cast<T*>(&lo);
    T* b = reinterpret_cast<T*>(&hi);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float x0 = Elem<T>::to(a[e]) * inv_rms * wlo[e];
        const float x1 = Elem<T>::to(b[e]) * inv_rms * whi[e];
        a[e] = Elem<T>::from(fmaf(x0, c[e], -x1 * s[e]));
        b[e] = Elem<T>::from(fmaf(x1, c[e], x0 * s[e]));
    }
}

// One CTA pass over sequences [b0, b0 + nseq): the cos / sin table of their
// positions (one angle per thread) and the norm weights, then every 16-byte
// vector pair of their q rows (normalised when q_norm_w is set, rotated into
// q_out) and k rows (the same with k_norm_w, rotated into the pool), and their
// v rows (copied).  tbl: kRopeSmemFloats floats of shared memory.  Returns the
// PKV_DEV_* bits of skipped rows.  Block-collective.
template <typename T>
__device__ uint32_t rope_append_pass(const AppendArgs& a, int b0, int nseq, int batch,
                                     int head_dim, float* tbl) {
    const int half = head_dim / 2;
    const int hv = half / 8;  // 16-byte vectors per half row
    float* ctab = tbl;
    float* stab = tbl + nseq * half;
    float* wq = tbl + 2 * 1024;  // norm weights of q, then of k
    float* wk = wq + head_dim;
    for (int t = threadIdx.x; t < nseq * half; t += blockDim.x) {
        const int b = b0 + t / half, i = t % half;
        float cv = 1.f, sv = 0.f;
        if (b < batch) rope_cos_sin(a.positions[b], a.inv_freq[i], &cv, &sv);
        ctab[t] = cv;
        stab[t] = sv;
    }
    for (int t = threadIdx.x; t < head_dim; t += blockDim.x) {
        wq[t] = a.q_norm_w ? Elem<T>::to(static_cast<const T*>(a.q_norm_w)[t]) : 1.f;
        wk[t] = a.k_norm_w ? Elem<T>::to(static_cast<const T*>(a.k_norm_w)[t]) : 1.f;
    }
    __syncthreads();
    uint32_t flags = 0;
    const int qi = a.n_q_heads * hv, ki = a.n_kv_heads * hv, vi = a.n_kv_heads * a.vecs;
    const int per_seq = qi + ki + vi;
    for (int it = threadIdx.x; it < nseq * per_seq; it += blockDim.x) {
        const int sq = it / per_seq, r = it - sq * per_seq;
        const int b = b0 + sq;
        if (b >= batch) break;
        const float* c = ctab + sq * half;
        const float* sn = stab + sq * half;
        if (r < qi) {  // query row: rotate into q_out
            const int h = r / hv, j = r % hv;
            const long long row = ((long long)b * a.n_q_heads + h) * a.vecs;
            uint4 lo = a.q_in[row + j], hi = a.q_in[row + hv + j];
            if (a.q_norm_w)
                norm_rotate8<T>(lo, hi, c + 8 * j, sn + 8 * j, wq + 8 * j, wq + half + 8 * j,
                                row_inv_rms<T>(lo, hi, hv, head_dim, a.norm_eps));
            else
                rotate8<T>(lo, hi, c + 8 * j, sn + 8 * j);
            a.q_out[row + j] = lo;
            a.q_out[row + hv + j] = hi;
            continue;
        }
        const int p = a.positions[b];
        if (p < 0) continue;  // padded batch slot: never writes the pool
        const int pi = p / a.page_size;
        const int rr = r - qi;
        const bool first = rr == 0;  // reports a skipped row once
        if (pi >= a.table_stride) {
            if (first) flags |= PKV_DEV_BAD_LEN;
            continue;
        }
        const int page = a.table[(long long)b * a.table_stride + pi];
        if (page < 0 || page >= a.num_pages) {
            if (first) flags |= PKV_DEV_BAD_PAGE;
            continue;
        }
        const long long base =
            (((long long)page * a.n_kv_heads) * a.page_size + p % a.page_size) * a.vecs;
        if (rr < ki) {  // key row: rotate into the pool
            const int h = rr / hv, j = rr % hv;
            const long long src = ((long long)b * a.n_kv_heads + h) * a.vecs;
            const long long dst = base + (long long)h * a.page_size * a.vecs;
            uint4 lo = a.k_new[src + j], hi = a.k_new[src + hv + j];
            if (a.k_norm_w)
                norm_rotate8<T>(lo, hi, c + 8 * j, sn + 8 * j, wk + 8 * j, wk + half + 8 * j,
                                row_inv_rms<T>(lo, hi, hv, head_dim, a.norm_eps));
            else
                rotate8<T>(lo, hi, c + 8 * j, sn + 8 * j);
            a.k_pool[dst + j] = lo;
            a.k_pool[dst + hv + j] = hi;
        } else {  // value row: bit copy
            const int v = rr - ki;
            const int h = v / a.vecs, j = v % a.vecs;
            const long long src = ((long long)b * a.n_kv_heads + h) * a.vecs;
            const long long dst = base + (long long)h * a.page_size * a.vecs;
            a.v_pool[dst + j] = a.v_new[src + j];
        }
    }
    __syncthreads();  // the table is rewritten by the next pass
    return flags;
}

// Sequences per pass: enough CTAs for the batch (up to kMaxAppendCtas), at most
// one angle per thread.
__host__ __device__ inline int rope_seqs_per_pass(int batch, int head_dim) {
    const int cap = kRopeThreads / (head_dim / 2);
    int n = (batch + kMaxAppendCtas - 1) / kMaxAppendCtas;
    return n < 1 ? 1 : (n > cap ? cap : n);
}

// Every pass of one CTA (CTA cta of nctas), for either element type.
__device__ uint32_t rope_append_cta(const AppendArgs& a, int batch, int head_dim, int cta,
                                    int nctas, float* tbl) {
    const int seqs = rope_seqs_per_pass(batch, head_dim);
    uint32_t flags = 0;
    for (int b0 = cta * seqs; b0 < batch; b0 += nctas * seqs) {
        flags |= a.bf16 ? rope_append_pass<__nv_bfloat16>(a, b0, seqs, batch, head_dim, tbl)
                        : rope_append_pass<__half>(a, b0, seqs, batch, head_dim, tbl);
    }
    return flags;
}

// ---------------------------------------------------------------------------
// Plan (CTA 0) and fused append (CTAs 1 .. append_ctas).
// Plan: clamps each context length to [0, table_stride * P] (PKV_DEV_BAD_LEN
// when it had to), writes the per-sequence chunk prefix sums (chunks of every
// unit of the sequence), the total, the worker count, and this call's status.
// Append CTA k writes its own status slot, so no clearing race exists.
// ---------------------------------------------------------------------------
// The plan of one decode (one CTA of 1024 threads); status_slots: the number
// of append_status entries other CTAs of the launch write.
__device__ void plan_cta(const PlanArgs& pa, int status_slots) {
    __shared__ int warp_tot[32];
    __shared__ long long running;
    __shared__ uint32_t flags;
    // the prefix sums also go to shared memory (when they fit) for the searches below
    __shared__ int32_t s_prefix[kPlanSmemSeqs + 1];
    const bool prefix_smem = pa.batch <= kPlanSmemSeqs;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int append_ctas = status_slots;
    if (tid == 0) {
        running = 0;
        flags = 0;
    }
    __syncthreads();
    if (pa.unit_done)
        for (long long x = tid; x < pa.units; x += blockDim.x) pa.unit_done[x] = 0;
    for (int base = 0; base < pa.batch; base += blockDim.x) {
        const int b = base + tid;
        int cnt = 0;
        if (b < pa.batch) {
            const int len = pa.uniform_len >= 0 ? pa.uniform_len
                             : pa.lens_host         ? __ldcv(pa.lens + b)
                                                    : pa.lens[b];
            long long L = (long long)len - pa.len_offset;
            if (L < 0) { L = 0; atomicOr(&flags, PKV_DEV_BAD_LEN); }
            if (L > pa.cap) { L = pa.cap; atomicOr(&flags, PKV_DEV_BAD_LEN); }
            pa.lens_eff[b] = (int32_t)L;
            cnt = (int)((L + kChunk - 1) / kChunk) * pa.units_per_b;
            if (pa.table) {  // the decode kernel reads this row right away: bring it into L2
                const int pages = (int)((L + pa.page_size - 1) / pa.page_size);
                const int32_t* row = pa.table + (long long)b * pa.table_stride;
                for (int e = 0; e < pages; e += 32)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(row + e));
            }
        }
        int x = cnt;  // inclusive warp scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int t = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, t, o);
                if (lane >= o) t += y;
            }
            warp_tot[lane] = t;
        }
        __syncthreads();
        const int excl = x - cnt + (warp > 0 ? warp_tot[warp - 1] : 0);
        if (b < pa.batch) {
            pa.prefix[b] = (int32_t)(running + excl);
            if (prefix_smem) s_prefix[b] = (int32_t)(running + excl);
        }
        __syncthreads();
        if (tid == 0) running += warp_tot[nwarps - 1];
        __syncthreads();
    }
    __shared__ int s_total, s_nw, s_sw, s_r;
    if (tid == 0) {
        long long total = running;
        uint32_t f = flags;
        if (total > INT_MAX) {  // beyond the 32-bit chunk index: refuse the work
            total = 0;
            f |= PKV_DEV_BAD_LEN;
        }
        pa.prefix[pa.batch] = (int32_t)total;
        if (prefix_smem) s_prefix[pa.batch] = (int32_t)total;
        int nw = 0;
        if (total > 0) {
            if (pa.workers_req > 0) {
                nw = (int)min((long long)pa.workers_req, total);
            } else {
                const long long want = (total + pa.min_chunks - 1) / pa.min_chunks;
                nw = (int)min((long long)pa.workers_auto, want < 1 ? 1LL : want);
            }
        }
        // contiguous ranges, equal to within one chunk: sw each, one more for
        // the first r workers
        const int sw = nw > 0 ? (int)(total / nw) : 0;
        const int r = nw > 0 ? (int)(total - (long long)sw * nw) : 0;
        pa.hdr->total_chunks = (int32_t)total;
        pa.hdr->num_workers = nw;
        pa.hdr->chunks_per_worker = sw;
        pa.hdr->extra_chunks = r;
        pa.hdr->append_slots = append_ctas;
        pa.hdr->status = f;
        s_total = (int)total;
        s_nw = nw;
        s_sw = sw;
        s_r = r;
    }
    __syncthreads();
    // sequence holding each worker's first chunk (for w = NW: the last chunk),
    // so that a worker searches only the sequences of its range
    const int T = s_total, nw = s_nw, sw = s_sw, r = s_r;
    const int32_t* pre = prefix_smem ? s_prefix : pa.prefix;
    auto seq_of = [&](int f) {
        int lo = 0, hi = pa.batch;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pre[mid] <= f) lo = mid; else hi = mid;
        }
        return lo;
    };
    for (int w = tid; w <= nw && T > 0; w += blockDim.x)
        pa.wstart[w] = seq_of(w < nw ? range_begin(w, sw, r) : T - 1);
}

// Staging copies of a host-buffer step (StageArgs), CTA c of sa.ctas: each
// thread has kStageLoads loads from host memory in flight before it stores.
constexpr int kStageLoads = 1;

__device__ void stage_cta(const StageArgs& sa, int c) {
    const long long stride = (long long)sa.ctas * blockDim.x;
    const long long t0 = (long long)c * blockDim.x + threadIdx.x;
    for (long long i = t0; i < sa.q_vecs; i += kStageLoads * stride) {
        uint4 v[kStageLoads];
#pragma unroll
        for (int j = 0; j < kStageLoads; ++j)
            if (i + j * stride < sa.q_vecs) v[j] = __ldcv(sa.q_src + i + j * stride);
#pragma unroll
        for (int j = 0; j < kStageLoads; ++j)
            if (i + j * stride < sa.q_vecs) sa.q_dst[i + j * stride] = v[j];
    }
    for (long long i = t0; i < sa.t_words; i += kStageLoads * stride) {
        int32_t v[kStageLoads];
#pragma unroll
        for (int j = 0; j < kStageLoads; ++j)
            if (i + j * stride < sa.t_words) v[j] = __ldcv(sa.t_src + i + j * stride);
#pragma unroll
        for (int j = 0; j < kStageLoads; ++j)
            if (i + j * stride < sa.t_words) sa.t_dst[i + j * stride] = v[j];
    }
}

__global__ void __launch_bounds__(1024)
plan_kernel(PlanArgs pa, AppendArgs aa, int append_ctas, StageArgs sa) {
    // No early trigger: the decode grid launches as this grid completes.  Let
    // in early, its CTAs all leave their dependency wait in the same instant,
    // which measured 0.5 us slower back to back and 8 us slower after a large
    // foreign kernel (cold L2) on a Llama-3-8B-shaped step.
    pdl_wait();
    if (blockIdx.x == 0) {
        plan_cta(pa, append_ctas);
        return;
    }
    if ((int)blockIdx.x > append_ctas) {  // staging CTAs (host-buffer step)
        stage_cta(sa, blockIdx.x - 1 - append_ctas);
        return;
    }
    __shared__ uint32_t flags;
    if (threadIdx.x == 0) flags = 0;
    __syncthreads();
    uint32_t f = 0;
    if (aa.q_in) {  // rotary embedding, then the append
        __shared__ float s_rope[kRopeSmemFloats];
        f = rope_append_cta(aa, pa.batch, aa.vecs * 8, blockIdx.x - 1, append_ctas, s_rope);
    } else {
        const long long total = (long long)pa.batch * aa.n_kv_heads * aa.vecs;
        const long long i0 = (long long)(blockIdx.x - 1) * blockDim.x + threadIdx.x;
        const long long stride = (long long)append_ctas * blockDim.x;
        if (aa.host) {
            for (long long idx = i0; idx < total; idx += stride) f |= append_vec<true>(aa, idx);
        } else {
            for (long long idx = i0; idx < total; idx += stride) f |= append_vec<false>(aa, idx);
        }
    }
    if (f) atomicOr(&flags, f);
    __syncthreads();
    if (threadIdx.x == 0) pa.hdr->append_status[blockIdx.x - 1] = flags;
}

// Plan launch of the shared-prefix decode: CTA 0 plans the suffix pass, CTA 1
// the prefix pass's virtual decode (CUDA-core variant); CTAs 2 .. 2+k-1 gather
// the query rows of every KV head in sequence-major order (qv[h][b*G + g] =
// q[b][h*G + g]; CUDA-core variant, qv non-null) and check that every table
// row starts with row 0's prefix pages (PKV_DEV_BAD_PREFIX into the suffix
// header's status slot of the CTA).
__global__ void __launch_bounds__(1024)
cascade_plan_kernel(PlanArgs ps, PlanArgs pv, CascadeGather g, int k) {
    pdl_wait();  // no early trigger, as in plan_kernel
    if (blockIdx.x == 0) {
        plan_cta(ps, k);
        return;
    }
    if (blockIdx.x == 1) {
        if (g.plan_virtual) plan_cta(pv, 0);
        return;
    }
    const int c = blockIdx.x - 2;
    const long long stride = (long long)k * blockDim.x;
    const long long total = g.qv ? (long long)g.batch * g.n_kv_heads * g.group * g.vecs : 0;
    for (long long idx = (long long)c * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        const int vec = (int)(idx % g.vecs);
        const long long row = idx / g.vecs;  // (h * B + b) * G + gi in qv
        const int gi = (int)(row % g.group);
        const long long hb = row / g.group;
        const int b = (int)(hb % g.batch), h = (int)(hb / g.batch);
        g.qv[idx] = g.q[(((long long)b * g.n_kv_heads + h) * g.group + gi) * g.vecs + vec];
    }
    bool differs = false;
    const long long cells = (long long)(g.batch - 1) * g.share_cols;
    for (long long x = (long long)c * blockDim.x + threadIdx.x; x < cells; x += stride) {
        const long long r = 1 + x / g.share_cols, col = x - (r - 1) * g.share_cols;
        differs |= __ldg(g.table + r * g.table_stride + col) != __ldg(g.table + col);
    }
    __shared__ int any;
    if (threadIdx.x == 0) any = 0;
    __syncthreads();
    if (differs) any = 1;
    __syncthreads();
    if (threadIdx.x == 0) ps.hdr->append_status[c] = any ? PKV_DEV_BAD_PREFIX : 0u;
}

// ---------------------------------------------------------------------------
// Combine: one CTA per unit (sequence, KV head, sub-group), or per (unit,
// row) when units are few beside the workers (row_split > 1: a long sequence
// in a small batch, whose units have many segments); units finished by a
// single worker and empty sequences exit at once.  The warps merge the rows
// with merge_rows_cta (the decode kernels' own merge does the same arithmetic
// per row, whichever CTA takes the row).
// ---------------------------------------------------------------------------
constexpr int kCombineWarps = 8;
static_assert(kCombineWarps == kMergeSlots, "a combine warp per merge slot");

template <typename T, int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
combine_kernel(const float* __restrict__ partials, const int32_t* __restrict__ prefix,
               const int32_t* __restrict__ lens_eff, const WsHeader* __restrict__ hdr,
               T* __restrict__ out, int units_per_b, int sub_groups, int gs, RowShape rs,
               int row_split) {
    // Everything up to pdl_wait reads only what the plan wrote: the plan grid
    // completed before any decode CTA passed its own wait and let this
    // kernel launch.  The partial states are read after the wait.
    const int u = blockIdx.x / row_split;
    const int part = blockIdx.x - u * row_split;  // row_split > 1: this CTA's row
    const int b = u / units_per_b;
    const int uidx = u - b * units_per_b;
    const int h = uidx / sub_groups;
    const int sgi = uidx - h * sub_groups;
    const int L = lens_eff[b];
    const int nch = (L + kChunk - 1) / kChunk;
    if (nch == 0) return;  // the decode kernel zeroed the rows of empty sequences
    if (hdr->total_chunks <= 0 || hdr->num_workers <= 0) return;
    const UnitSegments segs =
        unit_segments(hdr->chunks_per_worker, hdr->extra_chunks, u, prefix[b] + uidx * nch, nch);
    const int ns = segs.count();
    if (ns <= 1) return;  // finished in place by its worker
    const int nrows = rs.rows(sgi);
    if (row_split > 1 && part >= nrows) return;
    pdl_wait();
    pdl_trigger();
    const SlotSegs sg{partials, segs.base, partial_slot_floats(gs, D), gs, D};
    if (row_split > 1) {
        const RowShift<SlotSegs> one{sg, part};
        merge_rows_cta<T, D>(one, ns, 1, threadIdx.x >> 5, threadIdx.x & 31,
                             [&](int) { return out + rs.row(b, h, sgi, part) * D; });
    } else {
        merge_rows_cta<T, D>(sg, ns, nrows, threadIdx.x >> 5, threadIdx.x & 31,
                             [&](int g) { return out + rs.row(b, h, sgi, g) * D; });
    }
}

// ---------------------------------------------------------------------------
// Cascade combine (shared-prefix decode).  The prefix pass ran the shared
// prefix once per KV head for all B*G query rows (rows in b-major, head-minor
// order): as 128-row tensor-core tiles split over ranges of the prefix
// (prefix_umma.cu), or as a virtual decode of gs_v-row units; the suffix pass
// ran each sequence's own tokens.  Both left only partial states.  One CTA per
// real unit (sequence, KV head, sub-group of gs rows): its rows sit at rows
// ro .. ro+gs-1 of one tile or virtual unit (gs divides both).  The prefix
// segments, then the suffix segments, are merged as one list with merge_rows_seq.
// ---------------------------------------------------------------------------
template <class Pre>
struct CascadeSegs {
    Pre pre;  // the prefix pass's segments (rows offset by ro)
    int ro, np;
    SlotSegs suf;  // the unit's own segments
    __device__ __forceinline__ const float4* o4(int s, int g, int v) const {
        return s < np ? pre.o4(s, ro + g, v) : suf.o4(s - np, g, v);
    }
    __device__ __forceinline__ const float* m(int s, int g) const {
        return s < np ? pre.m(s, ro + g) : suf.m(s - np, g);
    }
    __device__ __forceinline__ const float* l(int s, int g) const {
        return s < np ? pre.l(s, ro + g) : suf.l(s - np, g);
    }
};

// The shared-prefix merge of units of at most kCombineWarps / 2 rows and at
// most 2 * kPairBlock segments: two warps per row, warp w taking row
// w % nrows and half w / nrows of the segments (the first ceil(ns / 2), or
// the rest).  Each warp issues its half's o loads together with the row's m
// and l loads (lane s: segment s), forms the row's maximum and denominator
// (both warps of a row the same bits), and sums its half in segment order;
// the second half's sum is then added to the first's, through shared memory.
// One round of loads per row instead of one plus one per 8 segments.
constexpr int kPairBlock = 16;

template <typename T, int D, class Segs, class RowOut>
__device__ __forceinline__ void merge_rows_pair(const Segs& sg, int ns, int nrows, int warp,
                                                int lane, float4* s_half,
                                                const RowOut& out_rows) {
    constexpr int Q = D / 4;
    static_assert(Q <= 32, "one vector per lane");
    const bool active = warp < 2 * nrows;
    const int g = active ? warp % nrows : 0;
    const int half = active ? warp / nrows : 0;
    const int h0 = (ns + 1) >> 1;
    const int s0 = half ? h0 : 0, s1 = half ? ns : h0;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    if (active) {
        const float m = lane < ns ? __ldcg(sg.m(lane, g)) : -INFINITY;
        const float l = lane < ns ? __ldcg(sg.l(lane, g)) : 0.f;
        float4 v[kPairBlock];
#pragma unroll
        for (int j = 0; j < kPairBlock; ++j)
            v[j] = lane < Q && s0 + j < s1 ? __ldcg(sg.o4(s0 + j, g, lane))
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
        float M = m;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
        const float wl = merge_weight(m, M);
        den = fmaf(wl, l, 0.f);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(kFull, den, o);
#pragma unroll
        for (int j = 0; j < kPairBlock; ++j) {
            const float w = __shfl_sync(kFull, wl, (s0 + j) & 31);
            if (s0 + j < s1) {
                x.x = fmaf(w, v[j].x, x.x);
                x.y = fmaf(w, v[j].y, x.y);
                x.z = fmaf(w, v[j].z, x.z);
                x.w = fmaf(w, v[j].w, x.w);
            }
        }
        if (half == 1 && lane < Q) s_half[g * 32 + lane] = x;
    }
    __syncthreads();
    if (active && half == 0 && lane < Q) {
        const float4 y = s_half[g * 32 + lane];
        x.x += y.x;
        x.y += y.y;
        x.z += y.z;
        x.w += y.w;
        merge_store<T, D>(x, den, lane, out_rows(g));
    }
}

// kUmma: the prefix pass ran on the tensor-core row tiles (prefix_umma.cu);
// else as a virtual decode of gs_v-row units.
template <typename T, int D, bool kUmma>
__global__ void __launch_bounds__(kCombineWarps * 32)
cascade_combine_kernel(CascadeArgs c) {
    const int u = blockIdx.x;
    const int b = u / c.units_per_b;
    const int uidx = u - b * c.units_per_b;
    const int h = uidx / c.sub_groups;
    const int sgi = uidx - h * c.sub_groups;
    const int gs = c.gs;
    T* o = static_cast<T*>(c.out) + ((long long)b * c.n_q_heads + h * c.group + sgi * gs) * D;
    // the suffix side: this unit's own segments
    const int L = c.s_lens[b];
    const int nch = (L + kChunk - 1) / kChunk;
    UnitSegments sv{0, 0};
    if (nch > 0 && c.s_hdr->num_workers > 0)
        sv = unit_segments(c.s_hdr->chunks_per_worker, c.s_hdr->extra_chunks, u,
                           c.s_prefix[b] + uidx * nch, nch);
    const int ns = sv.count();
    const SlotSegs suf{c.s_partials, sv.base, partial_slot_floats(gs, D), gs, D};
    // the prefix side: the rows of this unit among head h's B*G rows
    const int r0 = b * c.group + sgi * gs;
    if constexpr (kUmma) {
        const int t = r0 / c.v_tile_rows, ro = r0 - t * c.v_tile_rows;
        pdl_wait();  // the partial states of both passes are complete from here on
        pdl_trigger();
        const CascadeSegs<TileSegs> sg{
            TileSegs{c.v_partials, (long long)(h * c.v_tiles + t) * c.v_splits, D}, ro,
            c.v_splits, suf};
        const int nseg = c.v_splits + ns;
        if (2 * gs <= kCombineWarps && nseg <= 2 * kPairBlock) {
            __shared__ float4 s_half[(kCombineWarps / 2) * 32];
            merge_rows_pair<T, D>(sg, nseg, gs, threadIdx.x >> 5, threadIdx.x & 31, s_half,
                                  [&](int g) { return o + (long long)g * D; });
        } else {
            merge_rows_seq<T, D>(sg, nseg, gs, threadIdx.x >> 5, kCombineWarps,
                                 threadIdx.x & 31, [&](int g) { return o + (long long)g * D; });
        }
    } else {
        // the virtual unit holding this unit's rows
        const int vu = h * c.v_sub + r0 / c.v_gs, ro = r0 % c.v_gs;
        const UnitSegments pv = unit_segments(c.v_hdr->chunks_per_worker,
                                              c.v_hdr->extra_chunks, vu, vu * c.v_nch, c.v_nch);
        const int np = c.v_nch > 0 && c.v_hdr->num_workers > 0 ? pv.count() : 0;
        pdl_wait();  // the partial states of both passes are complete from here on
        pdl_trigger();
        const CascadeSegs<SlotSegs> sg{
            SlotSegs{c.v_partials, pv.base, partial_slot_floats(c.v_gs, D), c.v_gs, D}, ro, np,
            suf};
        merge_rows_seq<T, D>(sg, np + ns, gs, threadIdx.x >> 5, kCombineWarps, threadIdx.x & 31,
                             [&](int g) { return o + (long long)g * D; });
    }
}

cudaError_t launch_cascade_combine(pkv_dtype dtype, int head_dim, const CascadeArgs& c,
                                   int units, cudaStream_t stream) {
    if (units <= 0) return cudaSuccess;
#define PKV_CASCADE(T, D)                                                                  \
    return c.umma ? launch_pdl(cascade_combine_kernel<T, D, true>, dim3(units),             \
                               dim3(kCombineWarps * 32), 0, stream, c)                      \
                  : launch_pdl(cascade_combine_kernel<T, D, false>, dim3(units),            \
                               dim3(kCombineWarps * 32), 0, stream, c)
    if (dtype == PKV_BF16) {
        if (head_dim == 128) PKV_CASCADE(__nv_bfloat16, 128);
        PKV_CASCADE(__nv_bfloat16, 64);
    }
    if (head_dim == 128) PKV_CASCADE(__half, 128);
    PKV_CASCADE(__half, 64);
#undef PKV_CASCADE
}

// ---------------------------------------------------------------------------
// Check of the give-up path of the copy waits: one warp waits, bounded, on an
// mbarrier that nothing ever completes; when the tries run out it records
// PKV_DEV_TIMEOUT and the elapsed time, and returns.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(32)
wait_check_kernel(uint32_t tries, uint32_t* status, unsigned long long* elapsed_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    unsigned long long t0, t1;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    const bool done = mbar_wait_bounded(&bar, 0u, tries);  // phase 0 never completes
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
    if (threadIdx.x == 0) {
        if (!done) set_status(status, PKV_DEV_TIMEOUT);
        if (elapsed_ns) *elapsed_ns = t1 - t0;
    }
}

cudaError_t launch_wait_check(uint32_t tries, uint32_t* status, unsigned long long* elapsed_ns,
                              cudaStream_t stream) {
    wait_check_kernel<<<1, 32, 0, stream>>>(tries, status, elapsed_ns);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Stand-alone append: one thread per 16-byte vector of the new rows.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
append_kernel(AppendArgs a, int batch, uint32_t* status) {
    pdl_wait();
    pdl_trigger();
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long total = (long long)batch * a.n_kv_heads * a.vecs;
    if (idx >= total) return;
    const uint32_t f = append_vec<false>(a, idx);
    if (f) set_status(status, f);
}

// ---------------------------------------------------------------------------
// Gather: grid (ceil(max_len * vecs / 256), Hkv, B), bit copy.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
gather_kernel(const uint4* __restrict__ k_pool, const uint4* __restrict__ v_pool,
              const int32_t* __restrict__ table, int table_stride,
              const int32_t* __restrict__ lens, int n_kv_heads, int vecs, int page_size,
              int num_pages, int max_len, uint4* __restrict__ k_out, uint4* __restrict__ v_out,
              uint32_t* status) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.z, h = blockIdx.y;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const int t = (int)(idx / vecs), vec = (int)(idx % vecs);
    long long L = lens[b];
    const long long cap = (long long)table_stride * page_size;
    if (L < 0 || L > cap) {
        if (idx == 0 && h == 0) set_status(status, PKV_DEV_BAD_LEN);
        L = L < 0 ? 0 : cap;
    }
    if (t >= L || t >= max_len) return;
    const int page = table[(long long)b * table_stride + t / page_size];
    if (page < 0 || page >= num_pages) {
        if (vec == 0) set_status(status, PKV_DEV_BAD_PAGE);
        return;
    }
    const long long src = (((long long)page * n_kv_heads + h) * page_size + t % page_size) * vecs + vec;
    const long long dst = (((long long)b * n_kv_heads + h) * max_len + t) * vecs + vec;
    k_out[dst] = k_pool[src];
    v_out[dst] = v_pool[src];
}

// ---------------------------------------------------------------------------
// host-side launchers (stream-ordered, no synchronisation)
// ---------------------------------------------------------------------------
cudaError_t launch_plan(const PlanArgs& pa, const AppendArgs* append, cudaStream_t stream,
                        const StageArgs* stage) {
    AppendArgs aa = {};
    int append_ctas = 0;
    if (append) {
        aa = *append;
        long long ctas;
        if (aa.q_in) {  // rotary + append: rope_seqs_per_pass sequences per CTA pass
            const int seqs = rope_seqs_per_pass(pa.batch, aa.vecs * 8);
            ctas = (pa.batch + seqs - 1) / seqs;
        } else {
            const long long vecs = (long long)pa.batch * aa.n_kv_heads * aa.vecs;
            ctas = (vecs + 1023) / 1024;
        }
        append_ctas = (int)(ctas < kMaxAppendCtas ? ctas : kMaxAppendCtas);
    }
    StageArgs sa = {};
    if (stage) {
        sa = *stage;
        // 16-byte units of the copies over kStageLoads loads per thread
        const long long units = sa.q_vecs + (sa.t_words + 3) / 4;
        const long long per_cta = 1024LL * kStageLoads;
        const long long ctas = (units + per_cta - 1) / per_cta;
        sa.ctas = (int)(ctas < 1 ? 1 : (ctas > kMaxStageCtas ? kMaxStageCtas : ctas));
    }
    return launch_pdl(plan_kernel, dim3(1 + append_ctas + sa.ctas), dim3(1024), 0, stream, pa, aa,
                      append_ctas, sa);
}

cudaError_t launch_cascade_plan(const PlanArgs& ps, const PlanArgs& pv, const CascadeGather& g,
                                cudaStream_t stream) {
    // gather + check CTAs: about 4 K vectors (64 KiB of q, or of table cells when
    // nothing is gathered) each, at most kMaxAppendCtas
    const long long total = g.qv ? (long long)g.batch * g.n_kv_heads * g.group * g.vecs
                                 : (long long)(g.batch - 1) * g.share_cols;
    int k = (int)((total + 4095) / 4096);
    k = k < 1 ? 1 : (k > kMaxAppendCtas ? kMaxAppendCtas : k);
    return launch_pdl(cascade_plan_kernel, dim3(2 + k), dim3(1024), 0, stream, ps, pv, g, k);
}

cudaError_t launch_combine(pkv_dtype dtype, int head_dim, const float* partials,
                           const int32_t* prefix, const int32_t* lens_eff, const WsHeader* hdr,
                           void* out, int units, int units_per_b, int sub_groups, int gs,
                           const RowShape& rs, int workers, cudaStream_t stream) {
    if (units <= 0) return cudaSuccess;
    // few units beside the workers: their rows have many segments each, so a
    // CTA per (unit, row)
    const int row_split = (long long)units * 32 < workers ? gs : 1;
#define PKV_COMBINE(T, D)                                                                   \
    return launch_pdl(combine_kernel<T, D>, dim3(units * row_split), dim3(kCombineWarps * 32), \
                      0, stream, partials, prefix, lens_eff, hdr, static_cast<T*>(out),     \
                      units_per_b, sub_groups, gs, rs, row_split)
    if (dtype == PKV_BF16) {
        if (head_dim == 128) PKV_COMBINE(__nv_bfloat16, 128);
        PKV_COMBINE(__nv_bfloat16, 64);
    }
    if (head_dim == 128) PKV_COMBINE(__half, 128);
    PKV_COMBINE(__half, 64);
#undef PKV_COMBINE
}

cudaError_t launch_append(const AppendArgs& a, int batch, uint32_t* status,
                          cudaStream_t stream) {
    const long long total = (long long)batch * a.n_kv_heads * a.vecs;
    if (total == 0) return cudaSuccess;
    const int blocks = (int)((total + 255) / 256);
    return launch_pdl(append_kernel, dim3(blocks), dim3(256), 0, stream, a, batch, status);
}

// Stand-alone rotary + append: each CTA ORs its skipped-row bits into status.
__global__ void __launch_bounds__(kRopeThreads)
rope_append_kernel(AppendArgs a, int batch, int head_dim, uint32_t* status) {
    __shared__ float s_rope[kRopeSmemFloats];
    __shared__ uint32_t flags;
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) flags = 0;
    __syncthreads();
    const uint32_t f = rope_append_cta(a, batch, head_dim, blockIdx.x, gridDim.x, s_rope);
    if (f) atomicOr(&flags, f);
    __syncthreads();
    if (threadIdx.x == 0 && flags) set_status(status, flags);
}

cudaError_t launch_rope_append(const AppendArgs& a, int batch, int head_dim, uint32_t* status,
                               cudaStream_t stream) {
    if (batch == 0) return cudaSuccess;
    const int seqs = rope_seqs_per_pass(batch, head_dim);
    const int ctas = (batch + seqs - 1) / seqs;
    return launch_pdl(rope_append_kernel, dim3(ctas), dim3(kRopeThreads), 0, stream, a, batch,
                      head_dim, status);
}

cudaError_t launch_gather(const void* k_pool, const void* v_pool, const int32_t* table,
                          int table_stride, const int32_t* lens, int batch, int n_kv_heads,
                          int head_dim, int page_size, int num_pages, int max_len, void* k_out,
                          void* v_out, uint32_t* status, cudaStream_t stream) {
    const int vecs = head_dim / 8;
    const long long per_head = (long long)max_len * vecs;
    if (batch == 0 || per_head == 0) return cudaSuccess;
    dim3 grid((unsigned)((per_head + 255) / 256), (unsigned)n_kv_heads, (unsigned)batch);
    return launch_pdl(gather_kernel, grid, dim3(256), 0, stream,
                      static_cast<const uint4*>(k_pool), static_cast<const uint4*>(v_pool),
                      table, table_stride, lens, n_kv_heads, vecs, page_size, num_pages, max_len,
                      static_cast<uint4*>(k_out), static_cast<uint4*>(v_out), status);
}

}  // namespace pkv
