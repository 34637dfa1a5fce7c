// radix.cu -- a radix prefix cache over INT2 history pages ("卓绝TurboQuant：
// Together AI把2-bit KV Cache推向实在行状", serving-path text under figure
// "从离线校准到在线推理的 pipeline": the pool works with a radix prefix
// cache; section "小模子也能守住高难推理": the decode gain is largest at a full
// prefix hit).
//
// Host logic.  A context is cut into 64-token chunks: chunk 0 is the BF16
// sink (no page), chunk i >= 1 is history page i - 1.  Because a token's K/V
// depend on every token before it, a cached page is reusable only under the
// same chain of chunks from the root, so the tree's path is the token
// sequence and each node below the root's children holds the page of its
// chunk.  The tree keeps one page reference per node (oscar_pages_*); a
// match hands the caller one more reference per matched page.  Eviction
// removes least-recently-used leaves whose page nobody else holds.
#include <cstring>
#include <map>
#include <new>
#include <vector>

#include "oscar_common.cuh"

namespace {

constexpr int kChunk = 64;  // tokens per chunk (the page size)

struct RadixNode {
    std::vector<int32_t> key;  // the chunk's token ids
    int32_t page = -1;         // history page of the chunk (-1: the sink chunk)
    uint64_t stamp = 0;        // last match or insert touching the node
    RadixNode* parent = nullptr;
    std::map<std::vector<int32_t>, RadixNode*> child;
};

void free_tree(oscar_pages* pages, RadixNode* n) {
    for (auto& kv : n->child) free_tree(pages, kv.second);
    if (n->page >= 0) oscar_pages_release(pages, 1, &n->page);
    delete n;
}

}  // namespace

struct oscar_radix {
    oscar_pages* pages = nullptr;
    RadixNode root;
    uint64_t clock = 0;
    int32_t cached = 0;  // nodes holding a page
};

extern "C" {

oscar_status oscar_radix_create(oscar_pages* pages, oscar_radix** out) {
    if (!pages || !out) return OSCAR_ERR_INVALID_ARG;
    oscar_radix* r = new (std::nothrow) oscar_radix;
    if (!r) return OSCAR_ERR_OUT_OF_PAGES;
    r->pages = pages;
    *out = r;
    return OSCAR_OK;
}

void oscar_radix_destroy(oscar_radix* r) {
    if (!r) return;
    for (auto& kv : r->root.child) free_tree(r->pages, kv.second);
    delete r;
}

int32_t oscar_radix_cached_pages(const oscar_radix* r) { return r ? r->cached : -1; }

oscar_status oscar_radix_match(oscar_radix* r, const int32_t* tokens, int32_t n_tokens, int32_t max_pages,
                               int32_t* pages_out, int32_t* n_pages_out) try {
    if (!r || n_tokens < 0 || max_pages < 0 || !n_pages_out || (n_tokens > 0 && !tokens) ||
        (max_pages > 0 && !pages_out))
        return OSCAR_ERR_INVALID_ARG;
    *n_pages_out = 0;
    const uint64_t now = ++r->clock;
    RadixNode* n = &r->root;
    int32_t got = 0;
    for (int32_t c = 0; (c + 1) * kChunk <= n_tokens && got < max_pages + 1; ++c) {
        const std::vector<int32_t> key(tokens + c * kChunk, tokens + (c + 1) * kChunk);
        auto it = n->child.find(key);
        if (it == n->child.end()) break;
        n = it->second;
        n->stamp = now;
        if (c == 0) continue;  // the sink chunk has no page
        if (got == max_pages) break;
        pages_out[got++] = n->page;
    }
    if (got > 0 && oscar_pages_retain(r->pages, got, pages_out) != OSCAR_OK) return OSCAR_ERR_INVALID_ARG;
    *n_pages_out = got;
    return OSCAR_OK;
} catch (...) {
    return OSCAR_ERR_OUT_OF_PAGES;
}

oscar_status oscar_radix_insert(oscar_radix* r, const int32_t* tokens, int32_t n_tokens, const int32_t* pages,
                                int32_t n_pages) try {
    if (!r || n_pages < 0 || (n_pages > 0 && (!tokens || !pages))) return OSCAR_ERR_INVALID_ARG;
    if (n_pages == 0) return OSCAR_OK;
    if ((int64_t)n_tokens < (int64_t)kChunk * (1 + n_pages)) return OSCAR_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_pages; ++i)
        if (oscar_pages_refcount(r->pages, pages[i]) < 1) return OSCAR_ERR_INVALID_ARG;
    // the nodes to create: the chunks past the longest cached path
    const uint64_t now = ++r->clock;
    RadixNode* n = &r->root;
    int32_t c = 0;
    for (; c <= n_pages; ++c) {
        const std::vector<int32_t> key(tokens + c * kChunk, tokens + (c + 1) * kChunk);
        auto it = n->child.find(key);
        if (it == n->child.end()) break;
        n = it->second;
        n->stamp = now;
    }
    if (c > n_pages) return OSCAR_OK;  // everything cached already
    // one tree reference per new page node, taken before the tree changes
    if (oscar_pages_retain(r->pages, n_pages - (c == 0 ? 0 : c - 1), pages + (c == 0 ? 0 : c - 1)) != OSCAR_OK)
        return OSCAR_ERR_INVALID_ARG;
    for (; c <= n_pages; ++c) {
        RadixNode* m = new RadixNode;
        m->key.assign(tokens + c * kChunk, tokens + (c + 1) * kChunk);
        m->page = c == 0 ? -1 : pages[c - 1];
        m->stamp = now;
        m->parent = n;
        n->child.emplace(m->key, m);
        if (m->page >= 0) ++r->cached;
        n = m;
    }
    return OSCAR_OK;
} catch (...) {
    return OSCAR_ERR_OUT_OF_PAGES;
}

oscar_status oscar_radix_evict(oscar_radix* r, int32_t n_pages, int32_t* n_freed) try {
    if (!r || n_pages < 0 || !n_freed) return OSCAR_ERR_INVALID_ARG;
    int32_t freed = 0;
    while (freed < n_pages) {
        // the least recently used leaf whose page only the tree holds
        RadixNode* best = nullptr;
        std::vector<RadixNode*> stack;
        for (auto& kv : r->root.child) stack.push_back(kv.second);
        while (!stack.empty()) {
            RadixNode* n = stack.back();
            stack.pop_back();
            for (auto& kv : n->child) stack.push_back(kv.second);
            if (n->child.empty() && (n->page < 0 || oscar_pages_refcount(r->pages, n->page) == 1) &&
                (!best || n->stamp < best->stamp))
                best = n;
        }
        if (!best) break;
        if (best->page >= 0) {
            oscar_pages_release(r->pages, 1, &best->page);
            --r->cached;
            ++freed;
        }
        RadixNode* parent = best->parent ? best->parent : &r->root;
        parent->child.erase(best->key);
        delete best;
    }
    *n_freed = freed;
    return OSCAR_OK;
} catch (...) {
    return OSCAR_ERR_OUT_OF_PAGES;
}

}  // extern "C"
