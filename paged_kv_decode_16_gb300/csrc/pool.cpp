// pool.cpp -- page pool handle and host page allocator with reference counts.
//
// (CacheIR, "Current Capabilities": persistent shared CUDA page-backed KV
// pools; "Boundaries": shared CUDA KV page allocator accounting across forked
// request sessions.  TorchInferno, "Runtime Scaffolds": runtime.paged.)
// The allocator is host bookkeeping only: it hands out page ids that the
// caller writes into page-table rows; pages shared by several sequences (a
// common prefix) carry one reference per holder and return to the free list
// when the last holder releases them.  Every mutating call checks all its ids
// before changing anything, so a failed call leaves the state as it was.
#include <cuda_runtime.h>

#include <algorithm>
#include <new>

#include "pool_impl.hpp"

extern "C" {

pkv_status kv_pool_create(int num_pages, int page_size, int n_kv_heads, int head_dim,
                          pkv_dtype dtype, void* k_pool, void* v_pool, pkv_pool** out) {
    if (!out) return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    if (num_pages <= 0 || page_size <= 0 || n_kv_heads <= 0 || head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if ((k_pool == nullptr) != (v_pool == nullptr)) return PKV_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (page_size % 16 != 0 || page_size > 256) return PKV_ERR_UNSUPPORTED;
    if (k_pool && ((reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool)) & 15))
        return PKV_ERR_INVALID_ARG;
    pkv_pool* p = new (std::nothrow) pkv_pool();
    if (!p) return PKV_ERR_INVALID_ARG;
    p->num_pages = num_pages;
    p->page_size = page_size;
    p->n_kv_heads = n_kv_heads;
    p->head_dim = head_dim;
    p->dtype = dtype;
    if (k_pool) {
        p->k = k_pool;
        p->v = v_pool;
        p->owned = false;
    } else {
        const size_t bytes = (size_t)num_pages * n_kv_heads * page_size * head_dim * 2;
        if (cudaGetDevice(&p->device) != cudaSuccess || cudaMalloc(&p->k, bytes) != cudaSuccess) {
            delete p;
            return PKV_ERR_CUDA;
        }
        if (cudaMalloc(&p->v, bytes) != cudaSuccess) {
            cudaFree(p->k);
            delete p;
            return PKV_ERR_CUDA;
        }
        p->owned = true;
    }
    try {
        p->refcount.assign(num_pages, 0);
        p->free_list.resize(num_pages);
        for (int i = 0; i < num_pages; ++i) p->free_list[i] = num_pages - 1 - i;
    } catch (...) {
        if (p->owned) { cudaFree(p->k); cudaFree(p->v); }
        delete p;
        return PKV_ERR_INVALID_ARG;
    }
    *out = p;
    return PKV_OK;
}

pkv_status kv_pool_destroy(pkv_pool* pool) {
    if (!pool) return PKV_OK;
    pkv_status st = PKV_OK;
    if (pool->owned) {
        int prev = 0;
        cudaGetDevice(&prev);
        if (prev != pool->device) cudaSetDevice(pool->device);
        if (cudaFree(pool->k) != cudaSuccess) st = PKV_ERR_CUDA;
        if (cudaFree(pool->v) != cudaSuccess) st = PKV_ERR_CUDA;
        if (prev != pool->device) cudaSetDevice(prev);
    }
    delete pool;
    return st;
}

void* kv_pool_k(const pkv_pool* pool) { return pool ? pool->k : nullptr; }
void* kv_pool_v(const pkv_pool* pool) { return pool ? pool->v : nullptr; }

pkv_status kv_pool_info(const pkv_pool* pool, int* num_pages, int* page_size, int* n_kv_heads,
                        int* head_dim, pkv_dtype* dtype) {
    if (!pool) return PKV_ERR_INVALID_ARG;
    if (num_pages) *num_pages = pool->num_pages;
    if (page_size) *page_size = pool->page_size;
    if (n_kv_heads) *n_kv_heads = pool->n_kv_heads;
    if (head_dim) *head_dim = pool->head_dim;
    if (dtype) *dtype = pool->dtype;
    return PKV_OK;
}

pkv_status kv_pool_alloc_pages(pkv_pool* pool, int n, int32_t* ids_out) {
    if (!pool || n < 0 || (n > 0 && !ids_out)) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(pool->mu);
    if ((size_t)n > pool->free_list.size()) return PKV_ERR_OUT_OF_PAGES;
    for (int i = 0; i < n; ++i) {
        const int32_t id = pool->free_list.back();
        pool->free_list.pop_back();
        pool->refcount[id] = 1;
        ids_out[i] = id;
    }
    return PKV_OK;
}

pkv_status kv_pool_retain_pages(pkv_pool* pool, const int32_t* ids, int n) {
    if (!pool || n < 0 || (n > 0 && !ids)) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(pool->mu);
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= pool->num_pages) return PKV_ERR_INVALID_ARG;
        if (pool->refcount[ids[i]] <= 0) return PKV_ERR_REFCOUNT;
    }
    for (int i = 0; i < n; ++i) ++pool->refcount[ids[i]];
    return PKV_OK;
}

pkv_status kv_pool_release_pages(pkv_pool* pool, const int32_t* ids, int n) {
    if (!pool || n < 0 || (n > 0 && !ids)) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(pool->mu);
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= pool->num_pages) return PKV_ERR_INVALID_ARG;
    // an id may appear several times in one call: check the totals first
    std::vector<int32_t> sorted(ids, ids + n);
    std::sort(sorted.begin(), sorted.end());
    for (size_t i = 0; i < sorted.size();) {
        size_t j = i;
        while (j < sorted.size() && sorted[j] == sorted[i]) ++j;
        if ((int)(j - i) > pool->refcount[sorted[i]]) return PKV_ERR_REFCOUNT;
        i = j;
    }
    for (int i = 0; i < n; ++i) {
        if (--pool->refcount[ids[i]] == 0) pool->free_list.push_back(ids[i]);
    }
    return PKV_OK;
}

int kv_pool_free_count(const pkv_pool* pool) {
    if (!pool) return -1;
    std::lock_guard<std::mutex> lk(const_cast<pkv_pool*>(pool)->mu);
    return (int)pool->free_list.size();
}

int kv_pool_refcount(const pkv_pool* pool, int32_t page_id) {
    if (!pool || page_id < 0 || page_id >= pool->num_pages) return -1;
    std::lock_guard<std::mutex> lk(const_cast<pkv_pool*>(pool)->mu);
    return pool->refcount[page_id];
}

}  // extern "C"
