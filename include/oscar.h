/*
 * oscar.h -- C ABI of liboscar, the GB300 (sm_103a) hot path of OSCAR's
 * 2-bit KV-cache serving scheme.
 *
 * The method, as the pages describe it:
 *   [NEWS] "卓绝TurboQuant：Together AI把2-bit KV Cache推向实在行状"
 *          (www.sanyangsrq.com news article on OSCAR)
 *          sec. B "OSCAR 把旋转瞄准 attention": the rotation
 *                 R = U . Hadamard . bit-reversal, U per layer and KV head,
 *                 separately for K and V;
 *          sec. C figure "从离线校准到在线推理的 pipeline" and the text
 *                 under it: three-segment token pool (BF16 sink of 64 |
 *                 INT2 history | BF16 recent window of 256); the oldest
 *                 recent token is rotated, clipped, quantised and packed by
 *                 one fused kernel and moved into the history; four 2-bit
 *                 codes per byte; decode runs an INT2 kernel (unpack,
 *                 scale/zero dequantisation, float accumulation) and a BF16
 *                 kernel for sink/recent, merged by online softmax;
 *                 compatible with paged KV and prefix caching.
 *   [TALK] ml-summit.org speaker page, "Beyond the Paper: Engineering 2-Bit
 *          KV Cache for Real-World Deployment": mixed-precision data in a
 *          paged KV cache.
 *
 * Conventions for every call
 *   - Device pointers are caller-owned (allocate them with any allocator);
 *     the library never allocates or frees device memory, and keeps no state
 *     between calls except a per-device cache of kernel attributes (and the
 *     fixed scratch array of oscar_decode_attn_noalloc, below).
 *   - Device calls are asynchronous on the given stream (a cudaStream_t
 *     passed as void*; NULL = the legacy default stream).  They validate
 *     their host-visible arguments first and return an error before any
 *     launch; after launching they return OSCAR_ERR_CUDA if the launch
 *     failed (oscar_last_cuda_error() then holds the cudaError_t value).
 *   - Kernels never trap.  Out-of-range page ids or positions found on the
 *     device are skipped (a skipped history page contributes nothing) and
 *     reported by OR-ing bits into *dev_status when dev_status (a device
 *     int32) is not NULL: OSCAR_STATUS_BAD_PAGE, OSCAR_STATUS_BAD_POS.
 *   - Only head_dim 128, quant_group 32, 64 or 128, page_size 64 and
 *     query-per-KV-head groups G = Hq/Hk in {1, 2, 4, 8} are supported;
 *     other shapes return OSCAR_ERR_UNSUPPORTED.
 *   - The host-side page allocator and prefix cache (oscar_pages,
 *     oscar_radix) are opaque objects the caller creates and destroys; they
 *     hold host memory only.  No C++ exception crosses this interface.
 *
 * Calls, in the order of this header
 *   oscar_pool_layout                      static page layout (host)
 *   oscar_evict_quantize                   fused rotate/clip/quantise/pack
 *   oscar_decode_attn, _noalloc            decode attention over the pool
 *   oscar_evict_quantize_codebook,
 *   oscar_decode_attn_codebook             Lloyd-Max levels variant
 *   oscar_pages_*                          refcounted copy-on-write pages
 *   oscar_radix_*                          radix prefix cache over pages
 *   oscar_evict_quantize_boost,
 *   oscar_decode_attn_boost                K channel precision boost
 *   oscar_calibrate_codebook               offline fit of the Lloyd-Max levels
 *   oscar_calibrate_rotation               offline U_K, U_V
 *   oscar_calibrate_clip                   offline clip ratios
 *
 * Data layouts (row-major, little-endian)
 *   K/V token rows   bf16 [rows][Hk][2][d]           (index 0 = K, 1 = V)
 *   BF16 segments    bf16 [B][sink+recent][Hk][2][d] per layer; slots
 *                    [0, bf16_len[b]) are the valid sink + recent tokens
 *                    (their order does not matter to attention)
 *   U                fp32 [Hk][2][d][d]  (U_K, U_V); a row vector x is
 *                    rotated as y = x . U . H . P
 *   clip             fp32 [Hk][2]        clip ratio c in (0, 1]
 *   q                bf16 [B][Hq][d];  query head h reads KV head h / G
 *   out              fp32 [B][Hq][d]
 *   page_table       int32 [B][max_pages]: history position pos of sequence
 *                    b lives in page page_table[b*max_pages + pos/64],
 *                    slot pos % 64
 *   pool             num_pages * Hk blocks of oscar_block_bytes(shape) bytes
 *                    (OSCAR_BLOCK_BYTES = 6144 at g = 32; 5120 at g = 64,
 *                    4608 at g = 128); block (page, kv) starts at
 *                    (page*Hk + kv) * block_bytes and holds 64 token slots t;
 *                    with ng = 128 / g scale/zero pairs per vector:
 *       [0, 2048)     K codes, token-major: byte t*32 + j
 *       [2048, 4096)  V codes, byte-plane-major: byte 2048 + j*64 + t
 *       [4096, ...)   K scale/zero: at 4096 + t*4*ng + k*4, fp16 s then fp16 z
 *       [4096 + 256*ng, ...)  V scale/zero: at 4096 + 256*ng + t*4*ng + k*4
 *                    Group k is stored positions g*k .. g*k + g - 1; code byte j
 *                    (j = 0..31) holds in-group index j of each group: stored
 *                    position 32i + j in bits 2i..2i+1 (i = 0..3); stored
 *                    position p holds Hadamard output bitrev7(p) (the
 *                    bit-reversal of R, folded into addressing); value =
 *                    s*code + z in the rotated domain.
 */
#ifndef OSCAR_H
#define OSCAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    OSCAR_OK = 0,
    OSCAR_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or value */
    OSCAR_ERR_UNSUPPORTED = 2,  /* valid but unsupported shape */
    OSCAR_ERR_OUT_OF_PAGES = 3, /* a sequence needs more pages than max_pages */
    OSCAR_ERR_WORKSPACE = 4,    /* workspace smaller than oscar_decode_attn needs */
    OSCAR_ERR_CUDA = 5          /* a CUDA launch or query failed */
} oscar_status;

/* Device-side report bits (see dev_status). */
#define OSCAR_STATUS_BAD_PAGE 1 /* a page id outside [0, num_pages) */
#define OSCAR_STATUS_BAD_POS 2  /* a position, row or sequence index out of range */
#define OSCAR_STATUS_TIMEOUT 4  /* a bounded wait for a page copy gave up */
#define OSCAR_STATUS_NO_CONVERGENCE 8 /* the calibration eigensolver stopped before converging */

#define OSCAR_BLOCK_BYTES 6144  /* bytes per (page, KV head) block, d=128, g=32, page 64 */

typedef struct {
    int32_t head_dim;     /* d = 128 */
    int32_t quant_group;  /* g = 32, 64 or 128 elements per fp16 scale/zero */
    int32_t sink;         /* BF16 sink tokens (64) */
    int32_t recent;       /* BF16 recent-window tokens (256) */
    int32_t page_size;    /* tokens per history page (64) */
    int32_t num_q_heads;  /* Hq */
    int32_t num_kv_heads; /* Hk; Hq % Hk == 0 */
} oscar_shape;

/* Bytes of one (page, KV head) block for this shape, 0 if unsupported. */
size_t oscar_block_bytes(const oscar_shape* shape);

/* Human-readable name of a status code (static string). */
const char* oscar_status_string(oscar_status st);

/* cudaError_t of the last call that returned OSCAR_ERR_CUDA on this thread. */
int oscar_last_cuda_error(void);

/*
 * oscar_pool_layout -- paged-block allocation for the INT2 history
 * ([NEWS] sec. C: paged KV and radix-prefix-cache compatibility;
 * [TALK]: mixed-precision data in a paged KV cache).  Host only.
 *
 *   hist_capacity[batch]  (host) history tokens each sequence may hold.
 *   prefix_group[batch]   (host, nullable) sequences with the same group
 *                         id >= 0 share their first shared_hist_tokens/64
 *                         history pages (one physical copy, read-only by
 *                         convention); -1 = no sharing.
 *   shared_hist_tokens    multiple of 64, <= hist_capacity of every sharer.
 *   perm_seed             0: pages are numbered in allocation order; else
 *                         page L of that order becomes pi[L], pi a
 *                         Fisher-Yates shuffle of 0..N-1 driven by
 *                         SplitMix64 started at perm_seed (for i = N-1 down
 *                         to 1: j = next() mod (i+1), swap pi[i], pi[j]).
 *   Allocation order: the shared pages of each prefix group in order of
 *   first appearance, then each sequence's private pages in order.
 *   page_table[batch*max_pages] (host, out): page ids, -1 where unused.
 *   num_pages_out, pool_bytes_out (host, out, nullable): pages allocated and
 *   pool bytes (num_pages * Hk * block bytes).
 * Errors: INVALID_ARG for bad sizes/pointers/prefix settings, OUT_OF_PAGES
 * if a sequence needs more than max_pages pages.
 */
oscar_status oscar_pool_layout(const oscar_shape* shape, int32_t batch, const int32_t* hist_capacity,
                               const int32_t* prefix_group, int32_t shared_hist_tokens, uint64_t perm_seed,
                               int32_t max_pages, int32_t* page_table, int32_t* num_pages_out,
                               uint64_t* pool_bytes_out);

/*
 * oscar_evict_quantize -- the fused eviction kernel ([NEWS] sec. C): for
 * each of n_tok tokens and each KV head, rotate the K and V vectors by
 * R = U . H . P ([NEWS] sec. B), clip each group of quant_group (32, 64 or
 * 128) stored positions to
 * +-c*max|y|, quantise to 2-bit codes with fp16 scale s = (max-min)/3 and
 * zero z = min (codes from the stored fp16 s, z, round half to even,
 * clamped to 0..3; all codes 0 when s == 0), pack four codes per byte and
 * write codes and s/z into the pool slot of history position dst_pos[i] of
 * sequence dst_seq[i].
 *
 *   src_kv   (device) bf16 token rows [src_rows][Hk][2][d]; token i reads
 *            row src_row[i] (device int32, nullable: row i).
 *   new_kv   (device, nullable) bf16 [n_tok][Hk][2][d]: when given, row
 *            src_row[i] is overwritten with new_kv[i] after it was read (the
 *            ring-buffer append of a decode step fused into the eviction).
 *            Rows must then be distinct.
 *   dst_seq, dst_pos (device int32 [n_tok]); page_table (device int32
 *            [batch][max_pages]); num_pages = pool extent.  Rows, sequences,
 *            positions and page ids are bounds-checked on the device; a
 *            token with a bad index is skipped and reported in dev_status.
 *   U, clip  (device fp32) as in the layouts above.
 * Precision: no fp64 arithmetic runs on the GPU.  y = x.U is accumulated
 * with compensated fp32 products and sums (Dot2), the Hadamard transform
 * and the group statistics (max |y|, clamp, min, max) run on double-float
 * (hi, lo) pairs, s and z are rounded to fp16 from a value within 2^-23
 * (relative) of the exact one, and each code is decided from a u within
 * 4e-7 code units of a float64 evaluation.  Codes and fp16 s/z therefore
 * match a float64 evaluation except where u lies within 4e-7 of k + 0.5, or
 * a pre-rounding s or z within 2^-23 (relative) of an fp16 rounding
 * midpoint.
 */
oscar_status oscar_evict_quantize(const oscar_shape* shape, int32_t n_tok, const void* src_kv,
                                  int32_t src_rows, const int32_t* src_row, const int32_t* dst_seq,
                                  const int32_t* dst_pos, const void* new_kv, const float* U,
                                  const float* clip, uint8_t* pool, const int32_t* page_table,
                                  int32_t batch, int32_t max_pages, int32_t num_pages,
                                  int32_t* dev_status, void* stream);

/*
 * oscar_decode_attn -- one decode step of attention for every (sequence,
 * query head) over sink + INT2 history + recent window ([NEWS] sec. C):
 *   out[b,h] = softmax_t(sm_scale * q . k_t) . V
 * over the valid BF16 slots and the hist_len[b] history tokens, whose keys
 * and values are the dequantised stored vectors mapped back by R^T.  The
 * INT2 segment is attended in the rotated domain (q' = q . R_K; output
 * mapped back by R_V^T); segments and split-K partials are merged by their
 * log-sum-exp.  An empty context gives a zero output.
 *
 *   q        (device) bf16 [B][Hq][d], 8-byte aligned
 *   bf16_kv  (device) see layouts, 16-byte aligned
 *   bf16_len (device int32 [B], each in [0, sink+recent])
 *   pool, page_table (device), max_pages, num_pages (pool extent)
 *   hist_len (device int32 [B]) history tokens at positions [0, hist_len)
 *   U        (device fp32 [Hk][2][d][d]) same matrices as the eviction
 *   out      (device fp32 [B][Hq][d])
 *   workspace, *ws_bytes: caller-owned device scratch, 16-byte aligned.
 *            With workspace == NULL the call only stores the required size
 *            in *ws_bytes (it depends on shape, batch and max_pages) and
 *            launches nothing; with a smaller *ws_bytes it returns
 *            OSCAR_ERR_WORKSPACE.  The workspace holds the rotated queries,
 *            the work plan and the split-K partials of this call; calls that
 *            share a workspace must be ordered on one stream.
 */
oscar_status oscar_decode_attn(const oscar_shape* shape, int32_t batch, const void* q, const void* bf16_kv,
                               const int32_t* bf16_len, const uint8_t* pool, const int32_t* page_table,
                               int32_t max_pages, int32_t num_pages, const int32_t* hist_len, const float* U,
                               float sm_scale, float* out, void* workspace, size_t* ws_bytes,
                               int32_t* dev_status, void* stream);

/*
 * oscar_time_next_int2 -- measurement hook (no counterpart on the pages).
 * When ev_start and ev_stop are both non-NULL cudaEvent_t handles (passed as
 * void*), the next oscar_decode_attn call made by this host thread records
 * ev_start on its stream immediately before launching the INT2 split-K
 * kernel and ev_stop immediately after it; the hook then clears itself.
 * A benchmark uses it to time that kernel alone with CUDA events; it adds
 * two event records to the stream and changes nothing else.
 */
void oscar_time_next_int2(void* ev_start, void* ev_stop);

/* Size of the fixed device scratch array used by oscar_decode_attn_noalloc. */
#define OSCAR_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20) /* 64 MiB */

/*
 * oscar_decode_attn_noalloc -- oscar_decode_attn without a caller workspace.
 * The pages have no counterpart for this call: it exists for callers that
 * cannot allocate device memory (for instance code running inside a runtime
 * that owns all device memory and hands none out, or a plugin that may only
 * touch the buffers it is given).  Arguments and results are those of
 * oscar_decode_attn minus workspace/ws_bytes; the caller still owns every
 * input and output.  The scratch lives in a fixed 64 MiB array
 * (OSCAR_NOALLOC_SCRATCH_BYTES) in the library's device code, held by every
 * GPU that loads that code until the process exits; the call itself
 * allocates nothing.
 *   - A request needing more scratch than that (large batch x max_pages)
 *     returns OSCAR_ERR_WORKSPACE before any launch; use oscar_decode_attn
 *     with a workspace instead.  oscar_decode_attn with workspace == NULL
 *     reports the size a request needs.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.  The address is kept for the life of the
 *     process: after cudaDeviceReset (or anything else that destroys the
 *     device's primary context) it is stale, so this call must not be used
 *     on that device again in the same process.
 *   - All calls share the one array and it keeps the last call's contents;
 *     each call rebuilds what it reads, but calls that may overlap on the GPU
 *     (different streams, or different host threads) race on it: order them.
 */
oscar_status oscar_decode_attn_noalloc(const oscar_shape* shape, int32_t batch, const void* q, const void* bf16_kv,
                                       const int32_t* bf16_len, const uint8_t* pool, const int32_t* page_table,
                                       int32_t max_pages, int32_t num_pages, const int32_t* hist_len,
                                       const float* U, float sm_scale, float* out, int32_t* dev_status,
                                       void* stream);

/*
 * Lloyd-Max codebook variant ([NEWS] sec. E: OSCAR's code repository pairs
 * the rotation with a Lloyd-Max codebook; the pages give no format).
 * Reading: the stored format is unchanged (codes, fp16 scale s and zero z
 * per group, z = clipped minimum, s = range / 3) and only the four levels
 * move: in units of s above z they are {0, a, 3 - a, 3} instead of
 * {0, 1, 2, 3}, with one inner level a per (KV head, K/V), fixed offline
 * (oscar_calibrate_codebook).  A code is the nearest level to
 * u = (y_clipped - z) / s (u reaching a threshold a/2, 3/2 or 3 - a/2 moves
 * it up); a value dequantises to z + s * level[code].  a = 1 gives the
 * uniform levels; a <= 0 is read as 1.  The levels are in order for
 * a <= 3/2, and the decode's fp16 products are sized for that range (a
 * larger a can overflow them).
 *
 *   codebook (device) fp32 [Hk][2] the inner levels a (K, V of each KV head)
 *
 * oscar_evict_quantize_codebook: oscar_evict_quantize with the codebook's
 *   nearest-level codes.
 * oscar_decode_attn_codebook: oscar_decode_attn reading the history with
 *   the codebook's levels (every supported G).  About 1.6x the INT2
 *   instructions (and time) of the uniform levels at G <= 4: one more
 *   tensor-core product on the codes' high-bit plane for K and for V.
 */
oscar_status oscar_evict_quantize_codebook(const oscar_shape* shape, int32_t n_tok, const void* src_kv,
                                           int32_t src_rows, const int32_t* src_row, const int32_t* dst_seq,
                                           const int32_t* dst_pos, const void* new_kv, const float* U,
                                           const float* clip, const float* codebook, uint8_t* pool,
                                           const int32_t* page_table, int32_t batch, int32_t max_pages,
                                           int32_t num_pages, int32_t* dev_status, void* stream);
oscar_status oscar_decode_attn_codebook(const oscar_shape* shape, int32_t batch, const void* q, const void* bf16_kv,
                                        const int32_t* bf16_len, const uint8_t* pool, const int32_t* page_table,
                                        int32_t max_pages, int32_t num_pages, const int32_t* hist_len,
                                        const float* U, const float* codebook, float sm_scale, float* out,
                                        void* workspace, size_t* ws_bytes, int32_t* dev_status, void* stream);

/*
 * Refcounted history pages with copy-on-write (prefix sharing: [NEWS]
 * sec. C, the pool works with paged KV and a radix prefix cache).  Host
 * only, except oscar_pages_copy.  Not thread-safe: one host thread per
 * allocator.
 *
 * Sequences that share a prefix hold the same page ids in their rows of
 * the page table, one reference each (oscar_pages_retain when a sequence
 * adopts another's pages; oscar_pages_release when it drops them).  A
 * prefix need not end on a page boundary: before tokens are evicted into
 * pages, oscar_pages_prepare_write makes each target page private to its
 * row, and oscar_pages_copy copies the shared contents into the new pages;
 * then the caller uploads the changed table rows and evicts as usual.
 *
 * oscar_pages_create: num_pages free pages, handed out lowest id first
 *   (OSCAR_ERR_OUT_OF_PAGES if host memory for the counts runs out; the
 *   other calls report a failed host allocation the same way, unchanged).
 * oscar_pages_alloc: n fresh pages (one reference each) into pages_out;
 *   OSCAR_ERR_OUT_OF_PAGES (nothing taken) if fewer than n are free.
 * oscar_pages_retain / oscar_pages_release: one more / one less reference
 *   per listed page (duplicates count once each); a page whose count drops
 *   to 0 is free again.  OSCAR_ERR_INVALID_ARG (nothing changed) for a
 *   free or out-of-range page, or more releases than references.
 * oscar_pages_refcount: references of a page (-1 if out of range).
 * oscar_pages_prepare_write: for each of the n write targets (seq[i],
 *   page_index[i]) of page_table (host, [batch][max_pages], updated in
 *   place): an empty entry (-1) gets a fresh page; a page with more than
 *   one reference is replaced in that row by a fresh page, its reference
 *   moves there and (old, new) is appended to copy_src / copy_dst (host,
 *   room for n each; *n_copies = count); a private page is left as is.
 *   Repeated targets count once.  OSCAR_ERR_OUT_OF_PAGES or
 *   OSCAR_ERR_INVALID_ARG leave the allocator and the table unchanged.
 * oscar_pages_copy: for each pair, the Hk pool blocks of page copy_src[i]
 *   (and, when boost is not NULL, its Hk boost-record blocks) copied to
 *   page copy_dst[i] on the device, one cudaMemcpyAsync per page and array
 *   on `stream`; copy_src / copy_dst are host arrays.
 */
typedef struct oscar_pages oscar_pages;
oscar_status oscar_pages_create(int32_t num_pages, oscar_pages** out);
void oscar_pages_destroy(oscar_pages* pages);
oscar_status oscar_pages_alloc(oscar_pages* pages, int32_t n, int32_t* pages_out);
oscar_status oscar_pages_retain(oscar_pages* pages, int32_t n, const int32_t* page_ids);
oscar_status oscar_pages_release(oscar_pages* pages, int32_t n, const int32_t* page_ids);
int32_t oscar_pages_refcount(const oscar_pages* pages, int32_t page);
int32_t oscar_pages_free_count(const oscar_pages* pages);
oscar_status oscar_pages_prepare_write(oscar_pages* pages, int32_t n, const int32_t* seq, const int32_t* page_index,
                                       int32_t* page_table, int32_t batch, int32_t max_pages, int32_t* copy_src,
                                       int32_t* copy_dst, int32_t* n_copies);
oscar_status oscar_pages_copy(const oscar_shape* shape, int32_t n_copies, const int32_t* copy_src,
                              const int32_t* copy_dst, uint8_t* pool, uint8_t* boost, int32_t num_pages,
                              void* stream);

/*
 * Radix prefix cache over history pages ([NEWS] sec. C: the pool works with
 * a radix prefix cache; sec. D: the decode gain is largest at a full prefix
 * hit).  Host only, on top of an oscar_pages allocator (not owned; it must
 * outlive the cache).  Not thread-safe.
 *
 * A context (token ids) is cut into 64-token chunks: chunk 0 is the BF16
 * sink (no page), chunk i >= 1 is INT2 history page i - 1.  A token's K/V
 * depend on every token before it, so a page is reused only under the same
 * chain of chunks from the start: the tree's paths are token sequences and
 * each node below the sink level holds the page of its chunk, with one page
 * reference of its own.  Only whole chunks are cached.
 *
 * oscar_radix_insert: caches the first n_pages history pages of a context
 *   (tokens[n_tokens], n_tokens >= 64 * (1 + n_pages); pages[i] = the page
 *   holding history page i, allocated).  Chunks already cached keep their
 *   page; new nodes take one reference each.
 * oscar_radix_match: the longest cached prefix of tokens, in whole chunks:
 *   up to max_pages page ids of history pages 0, 1, ... into pages_out,
 *   *n_pages_out = count (0 if even the sink chunk differs); the caller
 *   receives one reference per returned page (release them when done).
 * oscar_radix_evict: removes least-recently-used leaves whose page nobody
 *   but the cache holds, freeing up to n_pages pages; *n_freed = count.
 * oscar_radix_cached_pages: pages held by the cache.
 * oscar_radix_destroy: drops the cache's references.
 */
typedef struct oscar_radix oscar_radix;
oscar_status oscar_radix_create(oscar_pages* pages, oscar_radix** out);
void oscar_radix_destroy(oscar_radix* radix);
oscar_status oscar_radix_insert(oscar_radix* radix, const int32_t* tokens, int32_t n_tokens, const int32_t* pages,
                                int32_t n_pages);
oscar_status oscar_radix_match(oscar_radix* radix, const int32_t* tokens, int32_t n_tokens, int32_t max_pages,
                               int32_t* pages_out, int32_t* n_pages_out);
oscar_status oscar_radix_evict(oscar_radix* radix, int32_t n_pages, int32_t* n_freed);
int32_t oscar_radix_cached_pages(const oscar_radix* radix);

/*
 * K channel precision boost (the "Zhongzhu (Charlie) Zhou" home page,
 * Featured Projects, entry "KITTY: Accurate and Efficient 2-bit KV Cache
 * Quantization with Dynamic Channel-wise Precision Boost": a small fraction
 * of the K cache's channels is kept at 4 bits, the rest at 2 bits; the
 * pages give no format).  Reading: the pool is written exactly as by
 * oscar_evict_quantize; in addition, for every stored K token-vector the
 * OSCAR_BOOST_N = 8 stored positions (rotated channels) with the largest
 * 2-bit rounding error |u - c| (ties to the lower position; error 0 where
 * s = 0) keep a 4-bit code q4 = clamp(rint(5 u), 0, 15) on the group's
 * range: the K value there is z + s * q4 / 5 instead of z + s * c.  V is
 * unchanged.
 *
 *   boost (device) uint8 [num_pages][Hk][OSCAR_BOOST_BLOCK_BYTES], 16-byte
 *          aligned; caller-owned, indexed by the same page ids as the pool.
 *          Token t of a page has its record at byte 16 t of the block:
 *          eight little-endian uint16 entries, stored position in bits 0-6,
 *          q4 in bits 8-11 and a copy of the position's 2-bit code c in
 *          bits 12-13 (other bits 0), in increasing position.  A
 *          record is written when its token is evicted; the decode reads
 *          the records of the history tokens only.
 *
 * oscar_evict_quantize_boost: oscar_evict_quantize plus the K records.
 * oscar_decode_attn_boost: oscar_decode_attn with the boosted K values
 *   (every supported G).  The corrections q'[pos] * s * (q4 / 5 - c) are
 *   added to the logits of the INT2 kernel; everything else is the uniform
 *   path.
 */
#define OSCAR_BOOST_N 8
#define OSCAR_BOOST_BLOCK_BYTES 1024 /* 64 tokens x 8 entries x 2 bytes */
oscar_status oscar_evict_quantize_boost(const oscar_shape* shape, int32_t n_tok, const void* src_kv,
                                        int32_t src_rows, const int32_t* src_row, const int32_t* dst_seq,
                                        const int32_t* dst_pos, const void* new_kv, const float* U,
                                        const float* clip, uint8_t* pool, uint8_t* boost,
                                        const int32_t* page_table, int32_t batch, int32_t max_pages,
                                        int32_t num_pages, int32_t* dev_status, void* stream);
oscar_status oscar_decode_attn_boost(const oscar_shape* shape, int32_t batch, const void* q, const void* bf16_kv,
                                     const int32_t* bf16_len, const uint8_t* pool, const uint8_t* boost,
                                     const int32_t* page_table, int32_t max_pages, int32_t num_pages,
                                     const int32_t* hist_len, const float* U, float sm_scale, float* out,
                                     void* workspace, size_t* ws_bytes, int32_t* dev_status, void* stream);

/*
 * oscar_calibrate_codebook -- offline Lloyd-Max fit of the inner level a of
 * each (KV head, K/V) codebook from calibration tokens: every element's
 * u = (y_clipped - z) / s under the eviction's quantiser (given U and clip,
 * rotation in fp32), folded by the symmetry to v = min(u, 3 - u) in
 * [0, 3/2]; Lloyd's iteration a <- mean{v : v >= a/2} from a = 1 until a
 * moves by less than 1e-6 (at most 200 rounds).  Groups with s = 0 give no
 * samples.
 *   kv (device) bf16 [n_t][Hk][2][d]; U fp32 [Hk][2][d][d]; clip fp32 [Hk][2]
 *   codebook (device) fp32 [Hk][2] out; workspace as oscar_decode_attn
 *   (workspace == NULL returns the size: 4 * Hk * 2 * n_t * d bytes).
 */
oscar_status oscar_calibrate_codebook(const oscar_shape* shape, int32_t n_t, const void* kv, const float* U,
                                      const float* clip, float* codebook, void* workspace, size_t* ws_bytes,
                                      void* stream);

/*
 * oscar_calibrate_rotation -- offline calibration of U ([NEWS] sec. B: U is
 * fixed offline per layer and KV head, for K from the covariance of the
 * queries that read the keys, for V from the covariance of the values as
 * weighted by the attention scores).  The pages give no formula; this call
 * takes the plainest reading:
 *   U_K[kv] = eigenvectors of mean(q q^T) over every calibration query token
 *             of every query head h with h / G = kv;
 *   U_V[kv] = eigenvectors of mean(o o^T) over the same samples, o the
 *             output of that query head's full (non-causal) softmax
 *             attention, scale sm_scale, over the calibration tokens:
 *             sum o o^T = V^T S^T S V with S the attention probabilities;
 * columns in order of decreasing eigenvalue, each column's entry of largest
 * magnitude positive; the result feeds oscar_evict_quantize and
 * oscar_decode_attn as U.  Arithmetic is fp32 (attention, covariance sums,
 * cyclic Jacobi eigensolver), so U is orthogonal to about 1e-6.  It runs
 * once per layer, offline; it is not part of a decode step.
 *
 *   q        (device) bf16 [n_q][Hq][d] calibration queries, 8-byte aligned
 *   kv       (device) bf16 [n_t][Hk][2][d] calibration keys and values,
 *            16-byte aligned
 *   U        (device) fp32 [Hk][2][d][d] out (layout of the U argument above)
 *   eigvals  (device) fp32 [Hk][2][d] out, the eigenvalues in U's column
 *            order, or NULL
 *   workspace, *ws_bytes: as oscar_decode_attn (workspace == NULL returns
 *            the size, which depends on shape and n_q); 16-byte aligned.
 *   dev_status: OSCAR_STATUS_NO_CONVERGENCE if a matrix's off-diagonal mass
 *            stayed above 1e-6 of its diagonal after the sweep limit (U is
 *            then the last iterate).
 * Errors: OSCAR_ERR_INVALID_ARG for n_q < 1, n_t < 1, null or misaligned
 * pointers, a non-finite or non-positive sm_scale; OSCAR_ERR_UNSUPPORTED as
 * for the other calls; OSCAR_ERR_WORKSPACE for a short workspace.
 */
oscar_status oscar_calibrate_rotation(const oscar_shape* shape, int32_t n_q, const void* q, int32_t n_t,
                                      const void* kv, float sm_scale, float* U, float* eigvals,
                                      void* workspace, size_t* ws_bytes, int32_t* dev_status, void* stream);

/*
 * oscar_calibrate_clip -- offline choice of the clip ratios ([NEWS] sec. B:
 * the clip thresholds are fixed offline together with U).  Reading: for each
 * (KV head, K/V) the ratio c of the candidate list with the least mean
 * squared error sum (y - y^)^2 / (n_t d) over the calibration tokens, y = x . R
 * the rotated vector and y^ its dequantised value under the eviction's
 * quantiser with clip ratio c (values clipped to +-c max|y| per group, the
 * error measured against the unclipped y); ties go to the larger ratio.
 * fp32 arithmetic (rotation x . U in fp32, not the eviction's compensated
 * form; the error totals in fp64).
 *
 *   kv       (device) bf16 [n_t][Hk][2][d] calibration tokens, 16-byte aligned
 *   U        (device) fp32 [Hk][2][d][d] (e.g. from oscar_calibrate_rotation)
 *   grid     (device) fp32 [n_grid] candidate ratios in (0, 1], 1 <= n_grid <= 32
 *   clip     (device) fp32 [Hk][2] out: the chosen ratios (the eviction's clip)
 *   mse      (device) fp32 [Hk][2][n_grid] out, the mean squared error of every
 *            candidate, or NULL
 *   workspace, *ws_bytes: as oscar_decode_attn (workspace == NULL returns the
 *            size), 16-byte aligned.
 */
oscar_status oscar_calibrate_clip(const oscar_shape* shape, int32_t n_t, const void* kv, const float* U,
                                  const float* grid, int32_t n_grid, float* clip, float* mse, void* workspace,
                                  size_t* ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* OSCAR_H */
