// kernels_aux.cu -- the small kernels around the decode kernel: plan (with an
// optional fused KV append), combine, stand-alone KV append and gather.  They
// move kilobytes; their cost is latency, so each one issues its independent
// loads together and is launched with programmatic dependent launch so that
// its launch overlaps the previous kernel's tail.
#include <limits.h>

#include "common.cuh"
#include "kernels_aux.cuh"

namespace pkv {

// ---------------------------------------------------------------------------
// KV append, one 16-byte vector per call (TorchInferno, "OpenAI-Compatible
// Serving" knob list: KV-append kernel).  Returns PKV_DEV_* bits for a
// skipped row (reported once per row, by its vector 0 of head 0).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t append_vec(const AppendArgs& a, long long idx) {
    const int vec = (int)(idx % a.vecs);
    const long long row = idx / a.vecs;  // b * Hkv + h
    const int b = (int)(row / a.n_kv_heads);
    const int h = (int)(row - (long long)b * a.n_kv_heads);
    const int p = a.positions[b];
    if (p < 0) return 0;  // padded batch slot: never writes
    const int pi = p / a.page_size;
    if (pi >= a.table_stride) return (vec == 0 && h == 0) ? PKV_DEV_BAD_LEN : 0u;
    const int page = a.table[(long long)b * a.table_stride + pi];
    if (page < 0 || page >= a.num_pages) return (vec == 0 && h == 0) ? PKV_DEV_BAD_PAGE : 0u;
    const long long dst =
        (((long long)page * a.n_kv_heads + h) * a.page_size + p % a.page_size) * a.vecs + vec;
    a.k_pool[dst] = a.k_new[row * a.vecs + vec];
    a.v_pool[dst] = a.v_new[row * a.vecs + vec];
    return 0;
}

// ---------------------------------------------------------------------------
// Plan (CTA 0) and fused append (CTAs 1 .. append_ctas).
// Plan: clamps each context length to [0, table_stride * P] (PKV_DEV_BAD_LEN
// when it had to), writes the per-sequence chunk prefix sums (chunks of every
// unit of the sequence), the total, the worker count, and this call's status.
// Append CTA k writes its own status slot, so no clearing race exists.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
plan_kernel(PlanArgs pa, AppendArgs aa, int append_ctas) {
    pdl_wait();
    pdl_trigger();
    __shared__ int warp_tot[32];
    __shared__ long long running;
    __shared__ uint32_t flags;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    if (tid == 0) {
        running = 0;
        flags = 0;
    }
    __syncthreads();
    if (blockIdx.x > 0) {
        const long long total = (long long)pa.batch * aa.n_kv_heads * aa.vecs;
        uint32_t f = 0;
        for (long long idx = (long long)(blockIdx.x - 1) * blockDim.x + tid; idx < total;
             idx += (long long)append_ctas * blockDim.x)
            f |= append_vec(aa, idx);
        if (f) atomicOr(&flags, f);
        __syncthreads();
        if (tid == 0) pa.hdr->append_status[blockIdx.x - 1] = flags;
        return;
    }
    for (int base = 0; base < pa.batch; base += blockDim.x) {
        const int b = base + tid;
        int cnt = 0;
        if (b < pa.batch) {
            long long L = pa.lens[b];
            if (L < 0) { L = 0; atomicOr(&flags, PKV_DEV_BAD_LEN); }
            if (L > pa.cap) { L = pa.cap; atomicOr(&flags, PKV_DEV_BAD_LEN); }
            pa.lens_eff[b] = (int32_t)L;
            cnt = (int)((L + kChunk - 1) / kChunk) * pa.units_per_b;
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
        if (b < pa.batch) pa.prefix[b] = (int32_t)(running + excl);
        __syncthreads();
        if (tid == 0) running += warp_tot[nwarps - 1];
        __syncthreads();
    }
    if (tid == 0) {
        long long total = running;
        uint32_t f = flags;
        if (total > INT_MAX) {  // beyond the 32-bit chunk index: refuse the work
            total = 0;
            f |= PKV_DEV_BAD_LEN;
        }
        pa.prefix[pa.batch] = (int32_t)total;
        int nw = 0;
        if (total > 0) {
            if (pa.workers_req > 0) {
                nw = (int)min((long long)pa.workers_req, total);
            } else {
                const long long want = (total + pa.min_chunks - 1) / pa.min_chunks;
                nw = (int)min((long long)pa.workers_auto, want < 1 ? 1LL : want);
            }
        }
        pa.hdr->total_chunks = (int32_t)total;
        pa.hdr->num_workers = nw;
        pa.hdr->append_slots = append_ctas;
        pa.hdr->status = f;
    }
}

// ---------------------------------------------------------------------------
// Combine: one CTA per unit (sequence, KV head, sub-group); units finished by
// a single worker exit at once, empty sequences get zeros.  Partial m is in
// base-2 units: out = sum_i 2^(m_i-M) o_i / sum_i 2^(m_i-M) l_i, M = max_i m_i.
// Warp w reduces M and the denominator of heads w, w+8, ... over the splits;
// then every thread owns 4 consecutive output elements and streams the
// splits' o.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(256)
combine_kernel(const float* __restrict__ partials, const int32_t* __restrict__ prefix,
               const int32_t* __restrict__ lens_eff, const WsHeader* __restrict__ hdr,
               T* __restrict__ out, int units_per_b, int sub_groups, int gs, int group,
               int n_q_heads) {
    pdl_wait();
    pdl_trigger();
    __shared__ float sM[16], sInv[16];  // per query head of the unit (gs <= 16)
    const int u = blockIdx.x;
    const int b = u / units_per_b;
    const int uidx = u - b * units_per_b;
    const int h = uidx / sub_groups;
    const int sg = uidx - h * sub_groups;
    T* o = out + ((long long)b * n_q_heads + h * group + sg * gs) * D;
    const int L = lens_eff[b];
    const int nch = (L + kChunk - 1) / kChunk;
    const int n = gs * D;
    const int tid = threadIdx.x;
    if (nch == 0) {
        for (int idx = tid; idx < n; idx += blockDim.x) o[idx] = T(0.f);
        return;
    }
    const long long total = hdr->total_chunks;
    const long long nw = hdr->num_workers;
    if (total <= 0 || nw <= 0) return;
    const long long a = (long long)prefix[b] + (long long)uidx * nch;
    const long long e = a + nch;
    const int w_first = (int)(((a + 1) * nw - 1) / total);
    const int w_last = (int)((e * nw - 1) / total);
    if (w_first == w_last) return;
    const int ns = w_last - w_first + 1;
    const long long stride = partial_slot_floats(gs, D);
    const float* base = partials + (long long)(u + w_first) * stride;  // slots u+w_first..u+w_last
    const int warp = tid >> 5, lane = tid & 31;
    for (int g = warp; g < gs; g += (int)(blockDim.x >> 5)) {
        float M = -INFINITY;
        for (int s = lane; s < ns; s += 32) M = fmaxf(M, base[s * stride + n + g]);
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, m));
        float S = 0.f;
        if (M != -INFINITY) {
            for (int s = lane; s < ns; s += 32)
                S += exp2f(base[s * stride + n + g] - M) * base[s * stride + n + gs + g];
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) S += __shfl_xor_sync(kFull, S, m);
        if (lane == 0) {
            sM[g] = M;
            sInv[g] = S > 0.f ? 1.0f / S : 0.f;
        }
    }
    __syncthreads();
    constexpr int Q = D / 4;
    for (int it = tid; it < gs * Q; it += blockDim.x) {
        const int g = it / Q, d4 = it - g * Q;
        const float M = sM[g];
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
#pragma unroll 4
            for (int s = 0; s < ns; ++s) {
                const float* pp = base + s * stride;
                const float w = exp2f(pp[n + g] - M);
                const float4 v = *reinterpret_cast<const float4*>(pp + g * D + d4 * 4);
                acc.x = fmaf(w, v.x, acc.x);
                acc.y = fmaf(w, v.y, acc.y);
                acc.z = fmaf(w, v.z, acc.z);
                acc.w = fmaf(w, v.w, acc.w);
            }
        }
        const float inv = sInv[g];
        uint2 w2;
        w2.x = Cvt<T>::pack2(acc.x * inv, acc.y * inv);
        w2.y = Cvt<T>::pack2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(o + g * D + d4 * 4) = w2;
    }
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
    const uint32_t f = append_vec(a, idx);
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
cudaError_t launch_plan(const PlanArgs& pa, const AppendArgs* append, cudaStream_t stream) {
    AppendArgs aa = {};
    int append_ctas = 0;
    if (append) {
        aa = *append;
        const long long vecs = (long long)pa.batch * aa.n_kv_heads * aa.vecs;
        const long long ctas = (vecs + 1023) / 1024;
        append_ctas = (int)(ctas < kMaxAppendCtas ? ctas : kMaxAppendCtas);
    }
    return launch_pdl(plan_kernel, dim3(1 + append_ctas), dim3(1024), 0, stream, pa, aa,
                      append_ctas);
}

cudaError_t launch_combine(pkv_dtype dtype, int head_dim, const float* partials,
                           const int32_t* prefix, const int32_t* lens_eff, const WsHeader* hdr,
                           void* out, int units, int units_per_b, int sub_groups, int gs,
                           int group, int n_q_heads, cudaStream_t stream) {
    if (units <= 0) return cudaSuccess;
#define PKV_COMBINE(T, D)                                                                     \
    return launch_pdl(combine_kernel<T, D>, dim3(units), dim3(256), 0, stream, partials,      \
                      prefix, lens_eff, hdr, static_cast<T*>(out), units_per_b, sub_groups,   \
                      gs, group, n_q_heads)
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
