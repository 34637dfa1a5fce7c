// api.cu -- the liboscar C ABI (include/oscar.h): argument checks, the
// workspace plan, the host page-table layout and kernel launches.
#include <cstdio>
#include <cstring>
#include <vector>

#include "oscar_common.cuh"

namespace oscar {

// Pages per split-K item: about 4096 items for the whole batch at most,
// 16-256 pages each (an item ends with a merge of the four consumer warps'
// states, so short items pay it per page or two; 16 pages is 4 per warp).
// Long items on large requests (batch 256 up to 128K tokens, batch 128 at
// 32K) measured 2-5 % faster steps than a 64-page cap; the short tail items
// keep the last wave balanced.
static int pages_per_split(int batch, int hk, int max_pages) {
    const int64_t cap = (int64_t)batch * hk * max_pages;
    int64_t pps = (cap + 4095) / 4096;
    if (pps < 16) pps = 16;
    if (pps > 256) pps = 256;
    return (int)pps;
}

static thread_local int g_last_cuda_error = 0;
static thread_local cudaEvent_t g_int2_ev_start = nullptr, g_int2_ev_stop = nullptr;

void set_last_cuda_error(int e) { g_last_cuda_error = e; }

static oscar_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return OSCAR_ERR_CUDA;
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

static size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// shape check shared by all calls: INVALID_ARG for impossible values,
// UNSUPPORTED for valid shapes this build has no kernels for
static oscar_status check_shape(const oscar_shape* s) {
    if (!s) return OSCAR_ERR_INVALID_ARG;
    if (s->head_dim <= 0 || s->quant_group <= 0 || s->page_size <= 0 || s->sink < 0 || s->recent < 0 ||
        s->num_q_heads <= 0 || s->num_kv_heads <= 0 || s->num_q_heads % s->num_kv_heads != 0 ||
        s->head_dim % s->quant_group != 0)
        return OSCAR_ERR_INVALID_ARG;
    const int G = s->num_q_heads / s->num_kv_heads;
    if (s->head_dim != kD || s->page_size != kPage) return OSCAR_ERR_UNSUPPORTED;
    if (s->quant_group != 32 && s->quant_group != 64 && s->quant_group != 128) return OSCAR_ERR_UNSUPPORTED;
    if (G != 1 && G != 2 && G != 4 && G != 8) return OSCAR_ERR_UNSUPPORTED;
    if (s->sink + s->recent > 320) return OSCAR_ERR_UNSUPPORTED;
    return OSCAR_OK;
}

static int bf16_items(const oscar_shape* s) { return (s->sink + s->recent + 63) / 64; }

// log2(quant_group / 32) and the (page, KV head) block size: K and V codes
// (2 x 2048 B) + K and V (s, z) pairs (2 x 64 tokens x d/g x 4 B)
static int gshift_of(const oscar_shape* s) { return s->quant_group == 32 ? 0 : (s->quant_group == 64 ? 1 : 2); }
static int block_bytes_of(const oscar_shape* s) { return 4096 + 512 * (kD / s->quant_group); }

// Pages at the end of each (sequence, KV head) that go to short items
// queued after all the long ones, so that the last waves of the persistent
// INT2 grid are short (used when long items are longer than short ones).
static int tail_pages_of(int pps) { return pps > kShortItemPages ? 2 * kShortItemPages : 0; }

struct WsLayout {
    size_t counter, item_start, item_start2, qfrag, qsum, qkinv, qrot, part, bf_part, total;
    int NT, pps, tail_pg, part_stride;
    int64_t max_items;   // split-K items at most (int64: batch x KV heads x splits can exceed int32)
};

static WsLayout ws_layout(const oscar_shape* s, int batch, int max_pages) {
    WsLayout w{};
    const int G = s->num_q_heads / s->num_kv_heads, hk = s->num_kv_heads;
    w.NT = (G + 3) / 4;
    w.pps = pages_per_split(batch, hk, max_pages);
    w.part_stride = (int)round_up((size_t)G * (kD + 2), 4);
    w.tail_pg = tail_pages_of(w.pps);
    w.max_items = (int64_t)batch * hk * ((max_pages + w.pps - 1) / w.pps + w.tail_pg / kShortItemPages);
    size_t off = 0;
    w.counter = off;
    off += 256;
    w.item_start = off;
    off = round_up(off + (size_t)(batch + 1) * 4, 256);
    w.item_start2 = off;
    off = round_up(off + (size_t)(batch + 1) * 4, 256);
    w.qfrag = off;
    off = round_up(off + (size_t)batch * hk * w.NT * 8 * 32 * 2 * 4, 256);
    w.qsum = off;
    off = round_up(off + (size_t)batch * hk * w.NT * 4 * 4 * 4, 256);
    w.qkinv = off;
    off = round_up(off + (size_t)batch * hk * 16, 256);
    w.qrot = off;
    off = round_up(off + (size_t)batch * hk * w.NT * 4 * kD * 4, 256);
    w.part = off;
    off = round_up(off + (size_t)w.max_items * w.part_stride * 4, 256);
    w.bf_part = off;
    off = round_up(off + (size_t)batch * hk * bf16_items(s) * w.part_stride * 4, 256);
    w.total = off;
    return w;
}

// ------------------------------------------------------------------
// page-table layout (host)
// ------------------------------------------------------------------
static uint64_t splitmix64(uint64_t& state) {
    uint64_t z = (state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

}  // namespace oscar

using namespace oscar;

extern "C" {

size_t oscar_block_bytes(const oscar_shape* shape) {
    if (check_shape(shape) != OSCAR_OK) return 0;
    return (size_t)block_bytes_of(shape);
}

const char* oscar_status_string(oscar_status st) {
    switch (st) {
        case OSCAR_OK: return "ok";
        case OSCAR_ERR_INVALID_ARG: return "invalid argument";
        case OSCAR_ERR_UNSUPPORTED: return "unsupported shape";
        case OSCAR_ERR_OUT_OF_PAGES: return "out of pages";
        case OSCAR_ERR_WORKSPACE: return "workspace too small";
        case OSCAR_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

int oscar_last_cuda_error(void) { return g_last_cuda_error; }

void oscar_time_next_int2(void* ev_start, void* ev_stop) {
    g_int2_ev_start = static_cast<cudaEvent_t>(ev_start);
    g_int2_ev_stop = static_cast<cudaEvent_t>(ev_stop);
}

oscar_status oscar_pool_layout(const oscar_shape* shape, int32_t batch, const int32_t* hist_capacity,
                               const int32_t* prefix_group, int32_t shared_hist_tokens, uint64_t perm_seed,
                               int32_t max_pages, int32_t* page_table, int32_t* num_pages_out,
                               uint64_t* pool_bytes_out) try {
    const oscar_status sst = check_shape(shape);
    if (sst != OSCAR_OK) return sst;
    if (batch < 0 || max_pages <= 0 || (batch > 0 && (!hist_capacity || !page_table)))
        return OSCAR_ERR_INVALID_ARG;
    const int P = shape->page_size;
    if (shared_hist_tokens < 0 || shared_hist_tokens % P != 0) return OSCAR_ERR_INVALID_ARG;
    const int n_shared = shared_hist_tokens / P;
    for (int b = 0; b < batch; ++b) {
        if (hist_capacity[b] < 0) return OSCAR_ERR_INVALID_ARG;
        if (((int64_t)hist_capacity[b] + P - 1) / P > max_pages) return OSCAR_ERR_OUT_OF_PAGES;
        if (prefix_group && prefix_group[b] >= 0 && hist_capacity[b] < shared_hist_tokens)
            return OSCAR_ERR_INVALID_ARG;
    }
    // page ids in allocation order: shared runs first (one per group, in
    // order of first appearance), then private pages sequence by sequence
    std::vector<int32_t> table((size_t)batch * max_pages, -1);
    std::vector<int> group_owner;  // owner sequence of each group id seen
    std::vector<int32_t> group_ids;
    int64_t next = 0;
    for (int b = 0; b < batch; ++b) {
        if (!prefix_group || prefix_group[b] < 0) continue;
        int owner = -1;
        for (size_t i = 0; i < group_ids.size(); ++i)
            if (group_ids[i] == prefix_group[b]) owner = group_owner[i];
        int32_t* row = &table[(size_t)b * max_pages];
        if (owner < 0) {
            group_ids.push_back(prefix_group[b]);
            group_owner.push_back(b);
            for (int pg = 0; pg < n_shared; ++pg) row[pg] = (int32_t)next++;
        } else {
            const int32_t* orow = &table[(size_t)owner * max_pages];
            for (int pg = 0; pg < n_shared; ++pg) row[pg] = orow[pg];
        }
    }
    for (int b = 0; b < batch; ++b) {
        const int need = (hist_capacity[b] + P - 1) / P;
        const int first = (prefix_group && prefix_group[b] >= 0) ? n_shared : 0;
        int32_t* row = &table[(size_t)b * max_pages];
        for (int pg = first; pg < need; ++pg) row[pg] = (int32_t)next++;
    }
    if (next > INT32_MAX) return OSCAR_ERR_INVALID_ARG;
    if (perm_seed != 0 && next > 1) {
        std::vector<int32_t> perm((size_t)next);
        for (int64_t i = 0; i < next; ++i) perm[(size_t)i] = (int32_t)i;
        uint64_t state = perm_seed;
        for (int64_t i = next - 1; i >= 1; --i) {
            const int64_t j = (int64_t)(splitmix64(state) % (uint64_t)(i + 1));
            std::swap(perm[(size_t)i], perm[(size_t)j]);
        }
        for (auto& v : table)
            if (v >= 0) v = perm[(size_t)v];
    }
    if (batch > 0) std::memcpy(page_table, table.data(), table.size() * sizeof(int32_t));
    if (num_pages_out) *num_pages_out = (int32_t)next;
    if (pool_bytes_out)
        *pool_bytes_out = (uint64_t)next * (uint64_t)shape->num_kv_heads * (uint64_t)block_bytes_of(shape);
    return OSCAR_OK;
} catch (...) {  // host scratch allocation: nothing was written
    return OSCAR_ERR_OUT_OF_PAGES;
}

static oscar_status evict_impl(const oscar_shape* shape, int32_t n_tok, const void* src_kv, int32_t src_rows,
                               const int32_t* src_row, const int32_t* dst_seq, const int32_t* dst_pos,
                               const void* new_kv, const float* U, const float* clip, const float* codebook,
                               uint8_t* pool, uint8_t* boost, const int32_t* page_table, int32_t batch,
                               int32_t max_pages, int32_t num_pages, int32_t* dev_status, void* stream) {
    const oscar_status sst = check_shape(shape);
    if (sst != OSCAR_OK) return sst;
    if (n_tok < 0 || src_rows < 0 || batch < 0 || max_pages <= 0 || num_pages < 0) return OSCAR_ERR_INVALID_ARG;
    if (n_tok == 0) return OSCAR_OK;
    if (!src_kv || !dst_seq || !dst_pos || !U || !clip || !pool || !page_table) return OSCAR_ERR_INVALID_ARG;
    if (!aligned(src_kv, 8) || (new_kv && !aligned(new_kv, 8)) || !aligned(U, 16) || !aligned(pool, 16) ||
        !aligned(clip, 4) || !aligned(dev_status, 4))
        return OSCAR_ERR_INVALID_ARG;
    if (!src_row && src_rows < n_tok) return OSCAR_ERR_INVALID_ARG;
    if ((int64_t)n_tok * shape->num_kv_heads * 2 > INT32_MAX) return OSCAR_ERR_INVALID_ARG;
    EvictParams p{};
    p.src_kv = static_cast<const __nv_bfloat16*>(src_kv);
    p.src_row = src_row;
    p.dst_seq = dst_seq;
    p.dst_pos = dst_pos;
    p.new_kv = static_cast<const __nv_bfloat16*>(new_kv);
    p.U = U;
    p.clip = clip;
    p.codebook = codebook;
    p.pool = pool;
    p.boost = boost;
    p.page_table = page_table;
    p.status = dev_status;
    p.n_tok = n_tok;
    p.hk = shape->num_kv_heads;
    p.src_rows = src_rows;
    p.batch = batch;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    p.gshift = gshift_of(shape);
    p.block_bytes = block_bytes_of(shape);
    const cudaError_t e = launch_evict(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e);
}

oscar_status oscar_evict_quantize(const oscar_shape* shape, int32_t n_tok, const void* src_kv,
                                  int32_t src_rows, const int32_t* src_row, const int32_t* dst_seq,
                                  const int32_t* dst_pos, const void* new_kv, const float* U,
                                  const float* clip, uint8_t* pool, const int32_t* page_table,
                                  int32_t batch, int32_t max_pages, int32_t num_pages,
                                  int32_t* dev_status, void* stream) {
    return evict_impl(shape, n_tok, src_kv, src_rows, src_row, dst_seq, dst_pos, new_kv, U, clip, nullptr, pool,
                      nullptr, page_table, batch, max_pages, num_pages, dev_status, stream);
}

oscar_status oscar_evict_quantize_boost(const oscar_shape* shape, int32_t n_tok, const void* src_kv,
                                        int32_t src_rows, const int32_t* src_row, const int32_t* dst_seq,
                                        const int32_t* dst_pos, const void* new_kv, const float* U,
                                        const float* clip, uint8_t* pool, uint8_t* boost,
                                        const int32_t* page_table, int32_t batch, int32_t max_pages,
                                        int32_t num_pages, int32_t* dev_status, void* stream) {
    if (n_tok > 0 && (!boost || !aligned(boost, 16))) return OSCAR_ERR_INVALID_ARG;
    return evict_impl(shape, n_tok, src_kv, src_rows, src_row, dst_seq, dst_pos, new_kv, U, clip, nullptr, pool,
                      boost, page_table, batch, max_pages, num_pages, dev_status, stream);
}

oscar_status oscar_evict_quantize_codebook(const oscar_shape* shape, int32_t n_tok, const void* src_kv,
                                           int32_t src_rows, const int32_t* src_row, const int32_t* dst_seq,
                                           const int32_t* dst_pos, const void* new_kv, const float* U,
                                           const float* clip, const float* codebook, uint8_t* pool,
                                           const int32_t* page_table, int32_t batch, int32_t max_pages,
                                           int32_t num_pages, int32_t* dev_status, void* stream) {
    if (!codebook || !aligned(codebook, 4)) return OSCAR_ERR_INVALID_ARG;
    return evict_impl(shape, n_tok, src_kv, src_rows, src_row, dst_seq, dst_pos, new_kv, U, clip, codebook, pool,
                      nullptr, page_table, batch, max_pages, num_pages, dev_status, stream);
}

static oscar_status decode_impl(const oscar_shape* shape, int32_t batch, const void* q, const void* bf16_kv,
                                const int32_t* bf16_len, const uint8_t* pool, const int32_t* page_table,
                                int32_t max_pages, int32_t num_pages, const int32_t* hist_len, const float* U,
                                const float* codebook, const uint8_t* boost, float sm_scale, float* out,
                                void* workspace, size_t* ws_bytes, int32_t* dev_status, void* stream) {
    const oscar_status sst = check_shape(shape);
    if (sst != OSCAR_OK) return sst;
    if (batch < 0 || max_pages <= 0 || num_pages < 0 || !ws_bytes) return OSCAR_ERR_INVALID_ARG;
    const WsLayout w = ws_layout(shape, batch, max_pages);
    // item counts, item offsets and partial indices are int32 on the device
    if (w.max_items > INT32_MAX || (double)w.max_items * w.part_stride > 4.0e9) return OSCAR_ERR_INVALID_ARG;
    if (!workspace) {
        *ws_bytes = w.total;
        return OSCAR_OK;
    }
    if (*ws_bytes < w.total) return OSCAR_ERR_WORKSPACE;
    if (batch == 0) return OSCAR_OK;
    if (!q || !bf16_kv || !bf16_len || !hist_len || !U || !out || !page_table) return OSCAR_ERR_INVALID_ARG;
    if (num_pages > 0 && !pool) return OSCAR_ERR_INVALID_ARG;
    if (!aligned(q, 8) || !aligned(bf16_kv, 16) || !aligned(U, 16) || !aligned(pool, 16) || !aligned(out, 16) ||
        !aligned(workspace, 16) || !aligned(dev_status, 4))
        return OSCAR_ERR_INVALID_ARG;
    if (!(sm_scale == sm_scale)) return OSCAR_ERR_INVALID_ARG;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    DecodeParams p{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.bf16_kv = static_cast<const __nv_bfloat16*>(bf16_kv);
    p.bf16_len = bf16_len;
    p.pool = pool;
    p.page_table = page_table;
    p.hist_len = hist_len;
    p.U = U;
    p.out = out;
    p.status = dev_status;
    p.counter = reinterpret_cast<int32_t*>(ws + w.counter);
    p.item_start = reinterpret_cast<int32_t*>(ws + w.item_start);
    p.item_start2 = reinterpret_cast<int32_t*>(ws + w.item_start2);
    p.qfrag = reinterpret_cast<uint32_t*>(ws + w.qfrag);
    p.qsum = reinterpret_cast<float*>(ws + w.qsum);
    p.qkinv = reinterpret_cast<float*>(ws + w.qkinv);
    p.qrot = reinterpret_cast<float*>(ws + w.qrot);
    p.part = reinterpret_cast<float*>(ws + w.part);
    p.bf_part = reinterpret_cast<float*>(ws + w.bf_part);
    p.B = batch;
    p.hq = shape->num_q_heads;
    p.hk = shape->num_kv_heads;
    p.G = shape->num_q_heads / shape->num_kv_heads;
    p.NT = w.NT;
    p.nslot = shape->sink + shape->recent;
    p.bf_items = bf16_items(shape);
    {   // merge warps per row: more when rows are few and split-K partials many
        const int splits = (max_pages + w.pps - 1) / w.pps + w.tail_pg / kShortItemPages;
        const int rows = batch * p.G;
        int wpr = 1;
        while (wpr < 8 && splits > 16 * wpr && rows * wpr < 4096) wpr *= 2;
        p.merge_wpr = wpr;
    }
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    p.gshift = gshift_of(shape);
    p.block_bytes = block_bytes_of(shape);
    p.pps = w.pps;
    p.tail_pg = w.tail_pg;
    p.part_stride = w.part_stride;
    p.qscale = sm_scale * kLog2e;
    p.codebook = codebook;
    p.boost = boost;
    cudaEvent_t ev0 = g_int2_ev_start, ev1 = g_int2_ev_stop;
    g_int2_ev_start = g_int2_ev_stop = nullptr;
    if (!ev0 || !ev1) ev0 = ev1 = nullptr;
    const cudaError_t e = launch_decode(p, static_cast<cudaStream_t>(stream), ev0, ev1);
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e);
}

oscar_status oscar_decode_attn(const oscar_shape* shape, int32_t batch, const void* q, const void* bf16_kv,
                               const int32_t* bf16_len, const uint8_t* pool, const int32_t* page_table,
                               int32_t max_pages, int32_t num_pages, const int32_t* hist_len, const float* U,
                               float sm_scale, float* out, void* workspace, size_t* ws_bytes,
                               int32_t* dev_status, void* stream) {
    return decode_impl(shape, batch, q, bf16_kv, bf16_len, pool, page_table, max_pages, num_pages, hist_len, U,
                       nullptr, nullptr, sm_scale, out, workspace, ws_bytes, dev_status, stream);
}

oscar_status oscar_decode_attn_boost(const oscar_shape* shape, int32_t batch, const void* q, const void* bf16_kv,
                                     const int32_t* bf16_len, const uint8_t* pool, const uint8_t* boost,
                                     const int32_t* page_table, int32_t max_pages, int32_t num_pages,
                                     const int32_t* hist_len, const float* U, float sm_scale, float* out,
                                     void* workspace, size_t* ws_bytes, int32_t* dev_status, void* stream) {
    const oscar_status sst = check_shape(shape);
    if (sst != OSCAR_OK) return sst;
    if (workspace && batch > 0 && num_pages > 0 && (!boost || !aligned(boost, 16))) return OSCAR_ERR_INVALID_ARG;
    return decode_impl(shape, batch, q, bf16_kv, bf16_len, pool, page_table, max_pages, num_pages, hist_len, U,
                       nullptr, boost, sm_scale, out, workspace, ws_bytes, dev_status, stream);
}

oscar_status oscar_decode_attn_codebook(const oscar_shape* shape, int32_t batch, const void* q, const void* bf16_kv,
                                        const int32_t* bf16_len, const uint8_t* pool, const int32_t* page_table,
                                        int32_t max_pages, int32_t num_pages, const int32_t* hist_len,
                                        const float* U, const float* codebook, float sm_scale, float* out,
                                        void* workspace, size_t* ws_bytes, int32_t* dev_status, void* stream) {
    const oscar_status sst = check_shape(shape);
    if (sst != OSCAR_OK) return sst;
    if (workspace && (!codebook || !aligned(codebook, 4))) return OSCAR_ERR_INVALID_ARG;
    return decode_impl(shape, batch, q, bf16_kv, bf16_len, pool, page_table, max_pages, num_pages, hist_len, U,
                       codebook, nullptr, sm_scale, out, workspace, ws_bytes, dev_status, stream);
}

oscar_status oscar_calibrate_rotation(const oscar_shape* shape, int32_t n_q, const void* q, int32_t n_t,
                                      const void* kv, float sm_scale, float* U, float* eigvals,
                                      void* workspace, size_t* ws_bytes, int32_t* dev_status, void* stream) {
    const oscar_status sst = check_shape(shape);
    if (sst != OSCAR_OK) return sst;
    if (n_q < 1 || n_t < 1 || !ws_bytes) return OSCAR_ERR_INVALID_ARG;
    const int hq = shape->num_q_heads, hk = shape->num_kv_heads;
    // covariance sums [2][Hk][d][d], then the attention outputs [n_q][Hq][d]
    const size_t c_bytes = round_up((size_t)2 * hk * kD * kD * 4, 256);
    const size_t total = c_bytes + round_up((size_t)n_q * hq * kD * 4, 256);
    if (!workspace) {
        *ws_bytes = total;
        return OSCAR_OK;
    }
    if (*ws_bytes < total) return OSCAR_ERR_WORKSPACE;
    if (!q || !kv || !U) return OSCAR_ERR_INVALID_ARG;
    if (!aligned(q, 8) || !aligned(kv, 16) || !aligned(U, 16) || !aligned(eigvals, 4) || !aligned(workspace, 16) ||
        !aligned(dev_status, 4))
        return OSCAR_ERR_INVALID_ARG;
    if (!(sm_scale > 0.f) || !(sm_scale < 3.0e38f)) return OSCAR_ERR_INVALID_ARG;
    if ((double)n_q * hq > 2.0e9 || (double)n_t * hk * 2 * kD > 2.0e9) return OSCAR_ERR_INVALID_ARG;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    CalibParams p{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.kv = static_cast<const __nv_bfloat16*>(kv);
    p.C = reinterpret_cast<float*>(ws);
    p.o = reinterpret_cast<float*>(ws + c_bytes);
    p.U = U;
    p.lam = eigvals;
    p.status = dev_status;
    p.n_q = n_q;
    p.n_t = n_t;
    p.hq = hq;
    p.hk = hk;
    p.sm_scale = sm_scale;
    const cudaError_t e = launch_calibrate(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e);
}

oscar_status oscar_calibrate_codebook(const oscar_shape* shape, int32_t n_t, const void* kv, const float* U,
                                      const float* clip, float* codebook, void* workspace, size_t* ws_bytes,
                                      void* stream) {
    const oscar_status sst = check_shape(shape);
    if (sst != OSCAR_OK) return sst;
    if (n_t < 1 || !ws_bytes) return OSCAR_ERR_INVALID_ARG;
    const int hk = shape->num_kv_heads;
    if ((double)n_t * hk * 2 * kD > 1.0e9) return OSCAR_ERR_INVALID_ARG;
    const size_t total = round_up((size_t)hk * 2 * n_t * kD * 4, 256);
    if (!workspace) {
        *ws_bytes = total;
        return OSCAR_OK;
    }
    if (*ws_bytes < total) return OSCAR_ERR_WORKSPACE;
    if (!kv || !U || !clip || !codebook) return OSCAR_ERR_INVALID_ARG;
    if (!aligned(kv, 16) || !aligned(U, 16) || !aligned(clip, 4) || !aligned(codebook, 4) || !aligned(workspace, 16))
        return OSCAR_ERR_INVALID_ARG;
    FitParams p{};
    p.kv = static_cast<const __nv_bfloat16*>(kv);
    p.U = U;
    p.clip = clip;
    p.v = static_cast<float*>(workspace);
    p.a = codebook;
    p.n_t = n_t;
    p.hk = hk;
    p.gshift = gshift_of(shape);
    const cudaError_t e = launch_calibrate_codebook(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e);
}

oscar_status oscar_calibrate_clip(const oscar_shape* shape, int32_t n_t, const void* kv, const float* U,
                                  const float* grid, int32_t n_grid, float* clip, float* mse, void* workspace,
                                  size_t* ws_bytes, void* stream) {
    const oscar_status sst = check_shape(shape);
    if (sst != OSCAR_OK) return sst;
    if (n_t < 1 || n_grid < 1 || n_grid > kMaxClipGrid || !ws_bytes) return OSCAR_ERR_INVALID_ARG;
    const int hk = shape->num_kv_heads;
    const size_t total = round_up((size_t)hk * 2 * kMaxClipGrid * sizeof(double), 256);
    if (!workspace) {
        *ws_bytes = total;
        return OSCAR_OK;
    }
    if (*ws_bytes < total) return OSCAR_ERR_WORKSPACE;
    if (!kv || !U || !grid || !clip) return OSCAR_ERR_INVALID_ARG;
    if (!aligned(kv, 16) || !aligned(U, 16) || !aligned(grid, 4) || !aligned(clip, 4) || !aligned(mse, 4) ||
        !aligned(workspace, 16))
        return OSCAR_ERR_INVALID_ARG;
    if ((double)n_t * hk * 2 * kD > 2.0e9) return OSCAR_ERR_INVALID_ARG;
    ClipParams p{};
    p.kv = static_cast<const __nv_bfloat16*>(kv);
    p.U = U;
    p.grid = grid;
    p.err = static_cast<double*>(workspace);
    p.clip = clip;
    p.mse = mse;
    p.n_t = n_t;
    p.hk = hk;
    p.n_grid = n_grid;
    p.gshift = gshift_of(shape);
    const cudaError_t e = launch_calibrate_clip(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e);
}

}  // extern "C"
