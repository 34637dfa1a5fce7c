// pages.cu -- refcounted history pages with copy-on-write, for prefix
// sharing in the paged INT2 history ("卓绝TurboQuant：Together AI把2-bit KV
// Cache推向实在行状", the serving-path text under figure "从离线校准到在线推理的
// pipeline": the pool works with paged KV and a radix prefix cache).
//
// Host logic: a free list and one reference count per page.  Sequences that
// share a prefix hold the same page ids in their page-table rows (one
// reference each).  Before a write (the eviction of a token into a page),
// oscar_pages_prepare_write makes every target page private: a page with
// more than one reference is replaced in that row by a fresh page and the
// (old, new) pair is returned; oscar_pages_copy then copies the blocks on
// the device with one cudaMemcpyAsync per page.
#include <cstring>
#include <new>
#include <vector>

#include "oscar_common.cuh"

namespace oscar {
void set_last_cuda_error(int e);  // api.cu
}

struct oscar_pages {
    std::vector<int32_t> ref;   // references per page (0 = free)
    std::vector<int32_t> free;  // free page ids, the next one at the back
};

namespace {

bool valid_page(const oscar_pages* a, int32_t p) { return p >= 0 && p < (int32_t)a->ref.size(); }

int32_t take(oscar_pages* a) {
    const int32_t p = a->free.back();
    a->free.pop_back();
    a->ref[p] = 1;
    return p;
}

void drop(oscar_pages* a, int32_t p) {
    if (--a->ref[p] == 0) a->free.push_back(p);
}

}  // namespace

using namespace oscar;

extern "C" {

// No C++ exception leaves the C ABI: a failed host allocation is reported as
// OSCAR_ERR_OUT_OF_PAGES with nothing changed.
oscar_status oscar_pages_create(int32_t num_pages, oscar_pages** out) {
    if (!out || num_pages < 0) return OSCAR_ERR_INVALID_ARG;
    oscar_pages* a = new (std::nothrow) oscar_pages;
    if (!a) return OSCAR_ERR_OUT_OF_PAGES;
    try {
        a->ref.assign((size_t)num_pages, 0);
        a->free.resize((size_t)num_pages);
    } catch (...) {
        delete a;
        return OSCAR_ERR_OUT_OF_PAGES;
    }
    for (int32_t i = 0; i < num_pages; ++i) a->free[(size_t)i] = num_pages - 1 - i;  // lowest id first
    *out = a;
    return OSCAR_OK;
}

void oscar_pages_destroy(oscar_pages* a) { delete a; }

int32_t oscar_pages_free_count(const oscar_pages* a) { return a ? (int32_t)a->free.size() : -1; }

int32_t oscar_pages_refcount(const oscar_pages* a, int32_t page) {
    return (a && valid_page(a, page)) ? a->ref[(size_t)page] : -1;
}

oscar_status oscar_pages_alloc(oscar_pages* a, int32_t n, int32_t* pages_out) {
    if (!a || n < 0 || (n > 0 && !pages_out)) return OSCAR_ERR_INVALID_ARG;
    if ((size_t)n > a->free.size()) return OSCAR_ERR_OUT_OF_PAGES;
    for (int32_t i = 0; i < n; ++i) pages_out[i] = take(a);
    return OSCAR_OK;
}

oscar_status oscar_pages_retain(oscar_pages* a, int32_t n, const int32_t* pages) {
    if (!a || n < 0 || (n > 0 && !pages)) return OSCAR_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i)
        if (!valid_page(a, pages[i]) || a->ref[(size_t)pages[i]] < 1) return OSCAR_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) ++a->ref[(size_t)pages[i]];
    return OSCAR_OK;
}

oscar_status oscar_pages_release(oscar_pages* a, int32_t n, const int32_t* pages) try {
    if (!a || n < 0 || (n > 0 && !pages)) return OSCAR_ERR_INVALID_ARG;
    std::vector<int32_t> need(a->ref.size(), 0);  // references this call drops, per page
    for (int32_t i = 0; i < n; ++i) {
        if (!valid_page(a, pages[i])) return OSCAR_ERR_INVALID_ARG;
        if (++need[(size_t)pages[i]] > a->ref[(size_t)pages[i]]) return OSCAR_ERR_INVALID_ARG;
    }
    for (int32_t i = 0; i < n; ++i) drop(a, pages[i]);
    return OSCAR_OK;
} catch (...) {
    return OSCAR_ERR_OUT_OF_PAGES;
}

oscar_status oscar_pages_prepare_write(oscar_pages* a, int32_t n, const int32_t* seq, const int32_t* page_index,
                                       int32_t* page_table, int32_t batch, int32_t max_pages, int32_t* copy_src,
                                       int32_t* copy_dst, int32_t* n_copies) try {
    if (!a || n < 0 || !n_copies || batch < 0 || max_pages <= 0) return OSCAR_ERR_INVALID_ARG;
    if (n > 0 && (!seq || !page_index || !page_table || !copy_src || !copy_dst)) return OSCAR_ERR_INVALID_ARG;
    // validate and count the fresh pages needed before changing anything
    int64_t fresh = 0;
    std::vector<int32_t> drops(a->ref.size(), 0);  // references the shared targets lose
    std::vector<char> seen((size_t)n, 0);
    for (int32_t i = 0; i < n; ++i) {
        if (seq[i] < 0 || seq[i] >= batch || page_index[i] < 0 || page_index[i] >= max_pages)
            return OSCAR_ERR_INVALID_ARG;
        const int32_t p = page_table[(size_t)seq[i] * max_pages + page_index[i]];
        if (p >= 0 && (!valid_page(a, p) || a->ref[(size_t)p] < 1)) return OSCAR_ERR_INVALID_ARG;
        bool dup = false;  // the same (sequence, page) earlier in this call
        for (int32_t j = 0; j < i && !dup; ++j) dup = seq[j] == seq[i] && page_index[j] == page_index[i];
        if (dup) continue;
        seen[(size_t)i] = 1;
        if (p < 0) {
            ++fresh;
        } else if (a->ref[(size_t)p] - drops[(size_t)p] > 1) {
            ++fresh;
            ++drops[(size_t)p];
        }
    }
    if (fresh > (int64_t)a->free.size()) return OSCAR_ERR_OUT_OF_PAGES;
    int32_t c = 0;
    for (int32_t i = 0; i < n; ++i) {
        if (!seen[(size_t)i]) continue;
        int32_t& slot = page_table[(size_t)seq[i] * max_pages + page_index[i]];
        if (slot < 0) {
            slot = take(a);
        } else if (a->ref[(size_t)slot] > 1) {
            const int32_t q = take(a);
            copy_src[c] = slot;
            copy_dst[c] = q;
            ++c;
            drop(a, slot);
            slot = q;
        }
    }
    *n_copies = c;
    return OSCAR_OK;
} catch (...) {  // the scratch vectors: before any change
    return OSCAR_ERR_OUT_OF_PAGES;
}

oscar_status oscar_pages_copy(const oscar_shape* shape, int32_t n_copies, const int32_t* copy_src,
                              const int32_t* copy_dst, uint8_t* pool, uint8_t* boost, int32_t num_pages,
                              void* stream) {
    const size_t bb = oscar_block_bytes(shape);
    if (bb == 0) return OSCAR_ERR_UNSUPPORTED;
    if (n_copies < 0 || num_pages < 0) return OSCAR_ERR_INVALID_ARG;
    if (n_copies == 0) return OSCAR_OK;
    if (!copy_src || !copy_dst || !pool) return OSCAR_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_copies; ++i)
        if (copy_src[i] < 0 || copy_src[i] >= num_pages || copy_dst[i] < 0 || copy_dst[i] >= num_pages ||
            copy_src[i] == copy_dst[i])
            return OSCAR_ERR_INVALID_ARG;
    const size_t hk = (size_t)shape->num_kv_heads;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (int32_t i = 0; i < n_copies; ++i) {  // a page's Hk blocks are contiguous
        cudaError_t e = cudaMemcpyAsync(pool + (size_t)copy_dst[i] * hk * bb, pool + (size_t)copy_src[i] * hk * bb,
                                        hk * bb, cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess && boost)
            e = cudaMemcpyAsync(boost + (size_t)copy_dst[i] * hk * kBoostBlock,
                                boost + (size_t)copy_src[i] * hk * kBoostBlock, hk * kBoostBlock,
                                cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) {
            set_last_cuda_error((int)e);
            return OSCAR_ERR_CUDA;
        }
    }
    return OSCAR_OK;
}

}  // extern "C"
