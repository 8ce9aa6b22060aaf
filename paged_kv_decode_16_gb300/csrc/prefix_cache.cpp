// prefix_cache.cpp -- host radix tree of cached prompt prefixes over the page
// pool (TorchInferno, "Runtime Scaffolds": runtime.prefix, a radix prefix tree
// with prefix-aware lookup, and runtime.prefix_cache, prefix-cache lookup for
// reusable entries; CacheIR, "Current Capabilities": shared KV page allocator
// accounting across forked request sessions).
//
// The tree is page-granular: below the root, a node stands for one full page
// of token ids (page_size of them) following its parent's tokens, and names the
// pool page that holds their K/V.  A node's children are kept in a hash map by
// a hash of their tokens, with the tokens compared in full on lookup, so a
// collision never merges two prefixes.  The cache owns one pool reference per
// node; a match hands the caller one more reference per matched page, so a
// page stays allocated while any sequence or the cache uses it.  Eviction
// removes least-recently-used leaves whose page only the cache still holds.
// Counters of lookups, hits, misses and pages moved in and out are kept under
// the same lock (CacheIR, "Current Capabilities": prefix-cache reuse with
// hit/miss counters).
#include <stdint.h>

#include <algorithm>
#include <functional>
#include <cstring>
#include <memory>
#include <new>
#include <queue>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"
#include "pool_impl.hpp"

namespace {

struct Node;
struct NodeFree {
    void operator()(Node* n) const;
};
using NodePtr = std::unique_ptr<Node, NodeFree>;

// One allocation per node: the node, then its page's token ids.
struct Node {
    int32_t page = -1;
    int ntok = 0;  // token ids of the page (0 at the root)
    Node* parent = nullptr;
    uint64_t last_use = 0;
    std::unordered_multimap<uint64_t, NodePtr> children;  // by hash_tokens of their ids

    const int32_t* tokens() const { return reinterpret_cast<const int32_t*>(this + 1); }
    int32_t* tokens() { return reinterpret_cast<int32_t*>(this + 1); }

    static NodePtr make(const int32_t* t, int n) {
        void* mem = ::operator new(sizeof(Node) + sizeof(int32_t) * (size_t)n);
        Node* node = new (mem) Node;
        node->ntok = n;
        std::memcpy(node->tokens(), t, sizeof(int32_t) * (size_t)n);
        return NodePtr(node);
    }
};
static_assert(alignof(Node) >= alignof(int32_t), "token ids follow the node");

void NodeFree::operator()(Node* n) const {
    n->~Node();
    ::operator delete(n);
}

// Hash of a page's token ids, two ids per step: h = (rotl(h, 23) ^ w) * K over
// 64-bit words w (K = 2^64 / golden ratio, odd), then the splitmix64 finaliser
// so that every input bit reaches the bucket index.  Only spreads the
// children over buckets: lookups compare the tokens in full.  (A byte-wise
// FNV-1a took ~8 us of a 96-page match.)
uint64_t hash_tokens(const int32_t* t, int n) {
    constexpr uint64_t K = 0x9e3779b97f4a7c15ull;
    uint64_t h = (uint64_t)n * K;
    int i = 0;
    for (; i + 1 < n; i += 2) {
        uint64_t w;
        std::memcpy(&w, t + i, sizeof(w));
        h = (((h << 23) | (h >> 41)) ^ w) * K;
    }
    if (i < n) h = (((h << 23) | (h >> 41)) ^ (uint64_t)(uint32_t)t[i]) * K;
    h ^= h >> 30;
    h *= 0xbf58476d1ce4e5b9ull;
    h ^= h >> 27;
    h *= 0x94d049bb133111ebull;
    h ^= h >> 31;
    return h;
}

Node* find_child(Node* n, const int32_t* t, int len, uint64_t h) {
    auto range = n->children.equal_range(h);
    for (auto it = range.first; it != range.second; ++it) {
        Node* c = it->second.get();
        if (c->ntok == len && std::equal(c->tokens(), c->tokens() + len, t)) return c;
    }
    return nullptr;
}

}  // namespace

struct pkv_prefix_cache {
    pkv_pool* pool = nullptr;
    int page_size = 0;
    std::mutex mu;  // guards the tree; taken before the pool's own lock
    Node root;  // no token ids follow it: tokens() of the root is never read
    uint64_t clock = 0;
    int pages = 0;  // nodes below the root
    pkv_prefix_cache_stats stats{};
};

namespace {

// Release every page below n (children first) and drop the nodes.
void release_subtree(pkv_prefix_cache* c, Node* n) {
    for (auto& kv : n->children) {
        Node* ch = kv.second.get();
        release_subtree(c, ch);
        kv_pool_release_pages(c->pool, &ch->page, 1);
        --c->pages;
    }
    n->children.clear();
}

// Leaves whose page only the cache references, by last use (oldest on top).
// Every insert or match stamps the nodes of one path with a fresh clock
// value, so no two leaves share a stamp and the order is total.
using LeafHeap = std::priority_queue<std::pair<uint64_t, Node*>,
                                     std::vector<std::pair<uint64_t, Node*>>,
                                     std::greater<std::pair<uint64_t, Node*>>>;

void collect_evictable_leaves(pkv_prefix_cache* c, Node* n, LeafHeap& heap) {
    for (auto& kv : n->children) {
        Node* x = kv.second.get();
        if (x->children.empty()) {
            if (kv_pool_refcount(c->pool, x->page) == 1) heap.emplace(x->last_use, x);
        } else {
            collect_evictable_leaves(c, x, heap);
        }
    }
}

void remove_leaf(Node* leaf) {
    Node* p = leaf->parent;
    auto range = p->children.equal_range(hash_tokens(leaf->tokens(), leaf->ntok));
    for (auto it = range.first; it != range.second; ++it)
        if (it->second.get() == leaf) {
            p->children.erase(it);
            return;
        }
}

}  // namespace

extern "C" {

pkv_status pkv_prefix_cache_create(pkv_pool* pool, pkv_prefix_cache** out) {
    if (!pool || !out) return PKV_ERR_INVALID_ARG;
    auto* c = new pkv_prefix_cache;
    c->pool = pool;
    c->page_size = pool->page_size;
    *out = c;
    return PKV_OK;
}

pkv_status pkv_prefix_cache_destroy(pkv_prefix_cache* cache) {
    if (!cache) return PKV_OK;
    {
        std::lock_guard<std::mutex> lk(cache->mu);
        release_subtree(cache, &cache->root);
    }
    delete cache;
    return PKV_OK;
}

pkv_status pkv_prefix_cache_insert(pkv_prefix_cache* cache, const int32_t* tokens, int n_tokens,
                                   const int32_t* pages, int* n_new) {
    if (!cache || n_tokens < 0 || (n_tokens > 0 && (!tokens || !pages)))
        return PKV_ERR_INVALID_ARG;
    const int P = cache->page_size;
    const int full = n_tokens / P;
    for (int i = 0; i < full; ++i)
        if (pages[i] < 0 || pages[i] >= cache->pool->num_pages) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(cache->mu);
    Node* n = &cache->root;
    const uint64_t now = ++cache->clock;
    // the part of the path already cached
    int i = 0;
    for (; i < full; ++i) {
        const int32_t* t = tokens + (long long)i * P;
        Node* c = find_child(n, t, P, hash_tokens(t, P));
        if (!c) break;
        c->last_use = now;
        n = c;
    }
    // pages i .. full-1 are new (nothing lies below a node that is missing):
    // the cache's references to all of them in one step, all or nothing (the
    // caller must hold each page), then the chain of nodes
    if (i < full) {
        const pkv_status st = kv_pool_retain_pages(cache->pool, pages + i, full - i);
        if (st != PKV_OK) return st;
    }
    for (int j = i; j < full; ++j) {
        const int32_t* t = tokens + (long long)j * P;
        NodePtr node = Node::make(t, P);
        node->page = pages[j];
        node->parent = n;
        node->last_use = now;
        Node* c = node.get();
        n->children.emplace(hash_tokens(t, P), std::move(node));
        n = c;
    }
    cache->pages += full - i;
    cache->stats.pages_inserted += (uint64_t)(full - i);
    if (n_new) *n_new = full - i;
    return PKV_OK;
}

pkv_status pkv_prefix_cache_match(pkv_prefix_cache* cache, const int32_t* tokens, int n_tokens,
                                  int32_t* pages_out, int max_pages, int* n_pages) {
    if (!cache || !n_pages || n_tokens < 0 || max_pages < 0 ||
        (n_tokens > 0 && !tokens) || (max_pages > 0 && !pages_out))
        return PKV_ERR_INVALID_ARG;
    const int P = cache->page_size;
    std::lock_guard<std::mutex> lk(cache->mu);
    Node* n = &cache->root;
    const uint64_t now = ++cache->clock;
    int k = 0;
    while (k < max_pages && (long long)(k + 1) * P <= n_tokens) {
        const int32_t* t = tokens + (long long)k * P;
        Node* c = find_child(n, t, P, hash_tokens(t, P));
        if (!c) break;
        c->last_use = now;
        pages_out[k++] = c->page;
        n = c;
    }
    // the caller's references to the matched pages
    const pkv_status st = kv_pool_retain_pages(cache->pool, pages_out, k);
    if (st != PKV_OK) return st;
    *n_pages = k;
    // whole pages the lookup could have served (at most max_pages)
    const long long asked = std::min<long long>(max_pages, n_tokens / P);
    pkv_prefix_cache_stats& s = cache->stats;
    ++s.lookups;
    if (k > 0) ++s.hits; else ++s.misses;
    s.pages_hit += (uint64_t)k;
    s.pages_missed += (uint64_t)(asked - k);
    return PKV_OK;
}

pkv_status pkv_prefix_cache_evict(pkv_prefix_cache* cache, int n_pages, int* n_freed) {
    if (!cache || n_pages < 0) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(cache->mu);
    // the least recently used evictable leaf, one at a time: a parent whose
    // last child goes becomes a leaf itself and joins the heap
    LeafHeap heap;
    if (n_pages > 0) collect_evictable_leaves(cache, &cache->root, heap);
    int freed = 0;
    while (freed < n_pages && !heap.empty()) {
        Node* leaf = heap.top().second;
        heap.pop();
        if (kv_pool_refcount(cache->pool, leaf->page) != 1) continue;  // retained meanwhile
        const pkv_status st = kv_pool_release_pages(cache->pool, &leaf->page, 1);
        if (st != PKV_OK) {
            cache->stats.pages_evicted += (uint64_t)freed;
            if (n_freed) *n_freed = freed;
            return st;
        }
        Node* parent = leaf->parent;
        remove_leaf(leaf);
        --cache->pages;
        ++freed;
        if (parent != &cache->root && parent->children.empty() &&
            kv_pool_refcount(cache->pool, parent->page) == 1)
            heap.emplace(parent->last_use, parent);
    }
    cache->stats.pages_evicted += (uint64_t)freed;
    if (n_freed) *n_freed = freed;
    return PKV_OK;
}

int pkv_prefix_cache_pages(const pkv_prefix_cache* cache) {
    if (!cache) return -1;
    std::lock_guard<std::mutex> lk(const_cast<pkv_prefix_cache*>(cache)->mu);
    return cache->pages;
}

pkv_status pkv_prefix_cache_get_stats(pkv_prefix_cache* cache, int reset,
                                      pkv_prefix_cache_stats* out) {
    if (!cache || !out) return PKV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(cache->mu);
    *out = cache->stats;
    if (reset) cache->stats = pkv_prefix_cache_stats{};
    return PKV_OK;
}

}  // extern "C"
