// kernels_aux.cu -- the small kernels around the decode kernel: plan, combine,
// KV append and gather.  All are bandwidth-trivial; their cost is launch and
// latency, so they stay simple.
#include <limits.h>

#include "common.cuh"
#include "kernels_aux.cuh"

namespace pkv {

// ---------------------------------------------------------------------------
// Plan: one CTA.  Clamps each context length to [0, table_stride * P] (flags
// PKV_DEV_BAD_LEN when it had to), writes the per-sequence chunk prefix sums
// (chunks of every unit of the sequence), the total and the worker count, and
// resets the status word for this call.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
plan_kernel(const int32_t* __restrict__ lens, int batch, int units_per_b, long long cap,
            int workers_req, int workers_auto, int min_chunks, int32_t* __restrict__ lens_eff,
            int32_t* __restrict__ prefix, WsHeader* __restrict__ hdr) {
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
    for (int base = 0; base < batch; base += blockDim.x) {
        const int b = base + tid;
        int cnt = 0;
        if (b < batch) {
            long long L = lens[b];
            if (L < 0) { L = 0; atomicOr(&flags, PKV_DEV_BAD_LEN); }
            if (L > cap) { L = cap; atomicOr(&flags, PKV_DEV_BAD_LEN); }
            lens_eff[b] = (int32_t)L;
            cnt = (int)((L + kChunk - 1) / kChunk) * units_per_b;
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
        if (b < batch) prefix[b] = (int32_t)(running + excl);
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
        prefix[batch] = (int32_t)total;
        int nw = 0;
        if (total > 0) {
            if (workers_req > 0) {
                nw = (int)min((long long)workers_req, total);
            } else {
                const long long want = (total + min_chunks - 1) / min_chunks;
                nw = (int)min((long long)workers_auto, want < 1 ? 1LL : want);
            }
        }
        hdr->total_chunks = (int32_t)total;
        hdr->num_workers = nw;
        hdr->status = f;
    }
}

// ---------------------------------------------------------------------------
// Combine: one CTA per unit (sequence, KV head, sub-group).  Units finished by
// a single worker are left alone; empty sequences get zeros.  Partial m is in
// base-2 units, so the weights are 2^(m_i - max m).
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(128)
combine_kernel(const float* __restrict__ partials, const int32_t* __restrict__ prefix,
               const int32_t* __restrict__ lens_eff, const WsHeader* __restrict__ hdr,
               T* __restrict__ out, int units_per_b, int sub_groups, int gs, int group,
               int n_q_heads) {
    const int u = blockIdx.x;
    const int b = u / units_per_b;
    const int uidx = u - b * units_per_b;
    const int h = uidx / sub_groups;
    const int sg = uidx - h * sub_groups;
    T* o = out + ((long long)b * n_q_heads + h * group + sg * gs) * D;
    const int L = lens_eff[b];
    const int nch = (L + kChunk - 1) / kChunk;
    const int n = gs * D;
    if (nch == 0) {
        for (int idx = threadIdx.x; idx < n; idx += blockDim.x) o[idx] = T(0.f);
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
    const long long stride = partial_slot_floats(gs, D);
    for (int idx = threadIdx.x; idx < n; idx += blockDim.x) {
        const int g = idx / D;
        float M = -INFINITY;
        for (int w = w_first; w <= w_last; ++w)
            M = fmaxf(M, partials[(u + w) * stride + n + g]);
        float S = 0.f, O = 0.f;
        if (M != -INFINITY) {
            for (int w = w_first; w <= w_last; ++w) {
                const float* pp = partials + (u + w) * stride;
                const float wt = exp2f(pp[n + g] - M);
                S += wt * pp[n + gs + g];
                O += wt * pp[idx];
            }
        }
        o[idx] = T(S > 0.f ? O / S : 0.f);
    }
}

// ---------------------------------------------------------------------------
// Append: one thread per 16-byte vector of the new rows (bit copy).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
              const int32_t* __restrict__ table, int table_stride,
              const int32_t* __restrict__ positions, int batch, int n_kv_heads, int vecs,
              int page_size, int num_pages, uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
              uint32_t* status) {
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long total = (long long)batch * n_kv_heads * vecs;
    if (idx >= total) return;
    const int vec = (int)(idx % vecs);
    const long long row = idx / vecs;  // b * Hkv + h
    const int b = (int)(row / n_kv_heads);
    const int h = (int)(row - (long long)b * n_kv_heads);
    const int p = positions[b];
    if (p < 0) return;
    const int pi = p / page_size;
    if (pi >= table_stride) {
        if (vec == 0 && h == 0) set_status(status, PKV_DEV_BAD_LEN);
        return;
    }
    const int page = table[(long long)b * table_stride + pi];
    if (page < 0 || page >= num_pages) {
        if (vec == 0 && h == 0) set_status(status, PKV_DEV_BAD_PAGE);
        return;
    }
    const long long dst = (((long long)page * n_kv_heads + h) * page_size + p % page_size) * vecs + vec;
    k_pool[dst] = k_new[row * vecs + vec];
    v_pool[dst] = v_new[row * vecs + vec];
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
cudaError_t launch_plan(const int32_t* lens, int batch, int units_per_b, long long cap,
                        int workers_req, int workers_auto, int min_chunks, int32_t* lens_eff,
                        int32_t* prefix, WsHeader* hdr, cudaStream_t stream) {
    plan_kernel<<<1, 1024, 0, stream>>>(lens, batch, units_per_b, cap, workers_req, workers_auto,
                                        min_chunks, lens_eff, prefix, hdr);
    return cudaGetLastError();
}

cudaError_t launch_combine(pkv_dtype dtype, int head_dim, const float* partials,
                           const int32_t* prefix, const int32_t* lens_eff, const WsHeader* hdr,
                           void* out, int units, int units_per_b, int sub_groups, int gs,
                           int group, int n_q_heads, cudaStream_t stream) {
    if (units <= 0) return cudaSuccess;
#define PKV_COMBINE(T, D)                                                                    \
    combine_kernel<T, D><<<units, 128, 0, stream>>>(partials, prefix, lens_eff, hdr,         \
                                                    static_cast<T*>(out), units_per_b,       \
                                                    sub_groups, gs, group, n_q_heads)
    if (dtype == PKV_BF16) {
        if (head_dim == 128) PKV_COMBINE(__nv_bfloat16, 128); else PKV_COMBINE(__nv_bfloat16, 64);
    } else {
        if (head_dim == 128) PKV_COMBINE(__half, 128); else PKV_COMBINE(__half, 64);
    }
#undef PKV_COMBINE
    return cudaGetLastError();
}

cudaError_t launch_append(const void* k_new, const void* v_new, const int32_t* table,
                          int table_stride, const int32_t* positions, int batch, int n_kv_heads,
                          int head_dim, int page_size, int num_pages, void* k_pool, void* v_pool,
                          uint32_t* status, cudaStream_t stream) {
    const int vecs = head_dim / 8;
    const long long total = (long long)batch * n_kv_heads * vecs;
    if (total == 0) return cudaSuccess;
    const int blocks = (int)((total + 255) / 256);
    append_kernel<<<blocks, 256, 0, stream>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), table, table_stride,
        positions, batch, n_kv_heads, vecs, page_size, num_pages, static_cast<uint4*>(k_pool),
        static_cast<uint4*>(v_pool), status);
    return cudaGetLastError();
}

cudaError_t launch_gather(const void* k_pool, const void* v_pool, const int32_t* table,
                          int table_stride, const int32_t* lens, int batch, int n_kv_heads,
                          int head_dim, int page_size, int num_pages, int max_len, void* k_out,
                          void* v_out, uint32_t* status, cudaStream_t stream) {
    const int vecs = head_dim / 8;
    const long long per_head = (long long)max_len * vecs;
    if (batch == 0 || per_head == 0) return cudaSuccess;
    dim3 grid((unsigned)((per_head + 255) / 256), (unsigned)n_kv_heads, (unsigned)batch);
    gather_kernel<<<grid, 256, 0, stream>>>(
        static_cast<const uint4*>(k_pool), static_cast<const uint4*>(v_pool), table, table_stride,
        lens, n_kv_heads, vecs, page_size, num_pages, max_len, static_cast<uint4*>(k_out),
        static_cast<uint4*>(v_out), status);
    return cudaGetLastError();
}

}  // namespace pkv
