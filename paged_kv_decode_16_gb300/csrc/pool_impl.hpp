// pool_impl.hpp -- definition of the opaque pkv_pool handle (host only).
#pragma once

#include <mutex>
#include <vector>

#include "pagedkv.h"

struct pkv_pool {
    int num_pages = 0, page_size = 0, n_kv_heads = 0, head_dim = 0;
    pkv_dtype dtype = PKV_BF16;
    void* k = nullptr;
    void* v = nullptr;
    bool owned = false;   // k / v were allocated by kv_pool_create
    int device = 0;       // device of owned memory
    std::mutex mu;        // guards the allocator state below
    std::vector<int32_t> free_list;  // stack; back() is handed out next
    std::vector<int32_t> refcount;   // per page, 0 = free
};
