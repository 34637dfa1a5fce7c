// oscar_common.cuh -- device helpers shared by the liboscar kernels
// (sm_103a).  Library-internal.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/oscar.h"

namespace oscar {

constexpr int kD = 128;           // head_dim
constexpr int kGroup = 32;        // quantisation group
constexpr int kNumGroups = kD / kGroup;
constexpr int kPage = 64;         // tokens per page
constexpr int kBfCounter = 32;      // index of the BF16 item queue's counter
constexpr int kShortItemPages = 16; // pages per short split-K item (the queue's tail)
constexpr int kBlock = OSCAR_BLOCK_BYTES;
constexpr int kKCodes = 0;        // byte offsets inside a (page, kv) block
constexpr int kVCodes = 2048;
constexpr int kKScale = 4096;
constexpr int kVScale = 5120;
constexpr float kLog2e = 1.4426950408889634f;
// 1/sqrt(128) in double
constexpr double kInvSqrtD = 0.088388347648318440550105545263;

constexpr unsigned kFull = 0xffffffffu;

// bit reversal of the low 5 / 2 bits
__device__ __forceinline__ int bitrev5(int v) { return (int)(__brev((unsigned)v) >> 27); }
__device__ __forceinline__ int bitrev2(int v) { return ((v & 1) << 1) | ((v >> 1) & 1); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float half_lo(uint32_t w) {
    return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
}
__device__ __forceinline__ float half_hi(uint32_t w) {
    return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

// binary16 from binary64, one rounding (round to nearest even)
__device__ __forceinline__ unsigned short f64_to_f16_bits(double x) {
    unsigned short h;
    asm("cvt.rn.f16.f64 %0, %1;" : "=h"(h) : "d"(x));
    return h;
}

// Programmatic dependent launch: let the next kernel in the stream start
// launching now / wait until the kernels this one overlaps with are complete
// and their writes visible (a no-op without a programmatic dependency).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// bf16x2 with lo -> bits 0-15, hi -> bits 16-31, round to nearest even
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// f16x2 with lo -> bits 0-15, hi -> bits 16-31, round to nearest even
__device__ __forceinline__ uint32_t pack_f16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
// Split four fp32 values into two f16x2 pairs each: the values rounded to
// fp16 (high parts) and the rounded remainders (low parts); together they
// carry 22 significant bits of every value whose remainder is a normal fp16.
__device__ __forceinline__ void split_f16(const float (&v)[4], uint32_t& h01, uint32_t& h23, uint32_t& l01,
                                          uint32_t& l23) {
    h01 = pack_f16x2_rn(v[0], v[1]);
    h23 = pack_f16x2_rn(v[2], v[3]);
    l01 = pack_f16x2_rn(v[0] - half_lo(h01), v[1] - half_hi(h01));
    l23 = pack_f16x2_rn(v[2] - half_lo(h23), v[3] - half_hi(h23));
}

__device__ __forceinline__ uint32_t rotr(uint32_t x, uint32_t n) { return __funnelshift_r(x, x, n); }

// Code pairs -> f16x2 MMA operands, with no offset and no arithmetic.
// A 16-bit pattern below 0x0400 (exponent field 0 or 1) is an fp16 whose
// value is exactly pattern * 2^-24: the subnormals and the first normal
// binade join without a gap.  So a 2-bit code c left at bits P, P+1 of an
// otherwise clear half reads as c * 2^(P-24), and one AND turns a code word
// into an operand register.  The tensor core keeps the products of such
// subnormal operands to a fixed number of bits below their nominal (biased)
// exponent, so each leading zero of the pattern below bit 9 costs one bit
// of the product: codes at bits 8-9 and 6-7 lose nothing, at 4-5 two bits,
// at 2-3 four bits, at 0-1 six.  The codes of byte slot 0 of bytes 0 and 2
// (bits 0-1 of a half) are therefore taken at bits 8-9 from the word with
// the two bytes of each half swapped (code_swap), which also brings slots
// 1-3 of bytes 1 and 3 down to bits 2-7; slot 0 of bytes 1 and 3 sits at bits
// 8-9 already and slots 1-3 of bytes 0 and 2 at bits 2-7.  The power
// 2^(P-24) of each slot is folded into the scales.
//
// Slot k of a byte holds the code of stored position 32k + j of the byte's
// vector (j = byte index); slot_bit(k) is the bit of that code inside the
// operand half.
__host__ __device__ __forceinline__ constexpr int slot_bit(int k) { return k == 0 ? 8 : 2 * k; }

// A code word with the two bytes of each 16-bit half swapped (bytes 1, 0,
// 3, 2): slots 1-3 of bytes 1 and 3 land at bits 2-7 of the halves and slot
// 0 of bytes 0 and 2 at bits 8-9, so that with the word itself every code
// sits at bit 2, 4, 6 or 8 of a half in one of the two.
__device__ __forceinline__ uint32_t code_swap(uint32_t x) { return __byte_perm(x, 0u, 0x2301u); }
// Operand from the slot-k codes of bytes 0 and 2 of x (k-index 0 and 1 of
// the register); xs = code_swap(x).
template <int SLOT>
__device__ __forceinline__ uint32_t code_pair_lo(uint32_t x, uint32_t xs) {
    if constexpr (SLOT == 0) return xs & 0x03000300u;
    else return x & (0x00030003u << (2 * SLOT));
}
// Operand from the slot-k codes of bytes 1 and 3 of x; xs = code_swap(x).
template <int SLOT>
__device__ __forceinline__ uint32_t code_pair_hi(uint32_t x, uint32_t xs) {
    if constexpr (SLOT == 0) return x & 0x03000300u;
    else return xs & (0x00030003u << (2 * SLOT));
}

// Power-of-two scalings of the INT2 decode (all exact):
//   K products run in fp16 (mma kind f16): the same code bit pattern read
//   as fp16 is c * 2^(slot_bit(k) - 24) (fp16 subnormals join the first
//   normal binade without a gap as well), and q' enters as q' * 2^e, one e
//   per (sequence, KV head) chosen by prep so that the largest |q'| of the
//   KV group's heads (times the Lloyd-Max plane weight, where it is above
//   1) lies in [2^13, 2^14): the fp16 high and low parts then hold q' to 22
//   bits (to an absolute 2^-25 * 2^-e below 2^-3 * 2^-e);
//   the K scale s is stored as s * 2^(24 - slot_bit(k) - e), which gives the
//   logit's products their true scale;
//   the V products (fp16 too) use B = W = p * s (times the Lloyd-Max inner
//   level a and 1/2 for the Lloyd-Max kernels), split into fp16 high and low
//   parts, so the P.V accumulator of slot k holds 2^(slot_bit(k) - 24) *
//   sum(W c), and the item's output multiplies it by v_out_scale(k).
// Ranges: K operands are below 2^14 and K products above 2^-46 (normal
// fp32); p <= 1 and s <= 65504 keep W <= 65504, finite in fp16 (the
// Lloyd-Max levels' factors a <= 3/2 and kappa * a <= 3/2 are offset by the
// 1/2); a W below 2^-14 keeps an absolute error of at most 2^-25, and V
// products stay above 2^-46.
constexpr int kQTopExp = 13;  // prep puts each head's largest |q'| in [2^13, 2^14)
__host__ __device__ __forceinline__ constexpr float pow2f(int e) {
    float r = 1.f;
    for (int i = 0; i < e; ++i) r *= 2.f;
    for (int i = 0; i > e; --i) r *= 0.5f;
    return r;
}
__device__ __forceinline__ constexpr float k_scale_up(int slot) { return pow2f(24 - slot_bit(slot)); }
__device__ __forceinline__ constexpr float v_out_scale(int slot) { return pow2f(24 - slot_bit(slot)); }
constexpr float kLmVDown = 0.5f;  // extra V-scale factor of the Lloyd-Max kernels (fp16 range)

// ---- packed fp32x2 arithmetic (two lanes of fp32 per instruction) --------
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 r;
    asm("{.reg .b64 A, B, C; mov.b64 A, {%2, %3}; mov.b64 B, {%4, %5}; mul.rn.f32x2 C, A, B; mov.b64 {%0, %1}, C;}"
        : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    float2 r;
    asm("{.reg .b64 A, B, C; mov.b64 A, {%2, %3}; mov.b64 B, {%4, %5}; sub.rn.f32x2 C, A, B; mov.b64 {%0, %1}, C;}"
        : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 r;
    asm("{.reg .b64 A, B, C, D; mov.b64 A, {%2, %3}; mov.b64 B, {%4, %5}; mov.b64 C, {%6, %7}; "
        "fma.rn.f32x2 D, A, B, C; mov.b64 {%0, %1}, D;}"
        : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}

// (x & mask) ^ bits in one LOP3
__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t x, uint32_t mask, uint32_t bits) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(x), "r"(mask), "r"(bits));
    return r;
}

// Selector of the hi / lo splits below (bf16 for the BF16 segment kernel's
// P operand, fp16 for the INT2 kernel's P*s operand): a lane taking the hi
// parts uses (a, sign) = (0, 0), a lane taking the lo parts (1, 0x80000000).
struct SplitSel {
    float2 a;
    uint32_t sign;
};
__device__ __forceinline__ SplitSel split_sel(bool take_lo) {
    return take_lo ? SplitSel{make_float2(1.f, 1.f), 0x80000000u} : SplitSel{make_float2(0.f, 0.f), 0u};
}

// A bf16x2 MMA operand register from two fp32 values w, split into bf16
// hi + lo: hi = w with its low 16 bits cleared (exact in bf16), lo = w - hi
// (exact in fp32, then rounded).  Returns the hi pair or the rounded lo
// pair, chosen arithmetically so that hi and lo lanes run the same
// instructions: x = a * w + (hi with its sign flipped by `sign`).
// (hi is taken by masking, not by the rounding-based Veltkamp split: the
// packed c - (c - w) form is exposed to algebraic simplification.)
__device__ __forceinline__ uint32_t split_pair(float2 w, const SplitSel& sel) {
    const float2 hs = make_float2(__uint_as_float(lop3_and_xor(__float_as_uint(w.x), 0xffff0000u, sel.sign)),
                                  __uint_as_float(lop3_and_xor(__float_as_uint(w.y), 0xffff0000u, sel.sign)));
    const float2 x = fma2(sel.a, w, hs);  // hi, or w - hi
    return pack_bf16x2_rn(x.x, x.y);
}

// the same for the products w = p * s
__device__ __forceinline__ uint32_t split_w_pair(float2 p, float2 s, const SplitSel& sel) {
    return split_pair(mul2(p, s), sel);
}

// fp16 versions (the INT2 P.V products): hi = w with its low 13 bits
// cleared, exact in fp16 for 2^-14 <= |hi| <= 65504 (below, its fp16
// rounding moves the sum by at most 2^-25), lo = w - hi rounded to fp16.
__device__ __forceinline__ uint32_t split_pair_f16(float2 w, const SplitSel& sel) {
    const float2 hs = make_float2(__uint_as_float(lop3_and_xor(__float_as_uint(w.x), 0xffffe000u, sel.sign)),
                                  __uint_as_float(lop3_and_xor(__float_as_uint(w.y), 0xffffe000u, sel.sign)));
    const float2 x = fma2(sel.a, w, hs);  // hi, or w - hi
    return pack_f16x2_rn(x.x, x.y);
}
__device__ __forceinline__ uint32_t split_w_pair_f16(float2 p, float2 s, const SplitSel& sel) {
    return split_pair_f16(mul2(p, s), sel);
}

// Token order inside the shared probability / V-scale rows of a 16-token
// tile: bits 0 and 1 swapped, so tokens (4a, 4a+2) and (4a+1, 4a+3) are
// adjacent pairs (the two token pairs of a PV B-operand register).
__device__ __forceinline__ int pv_slot(int t) { return (t & ~3) | ((t & 1) << 1) | ((t >> 1) & 1); }

// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// The same product with fp16 operands (both products of the INT2 decode).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}


// ------------------------------------------------------------------
// mbarrier + bulk async copy (TMA, non-tensor), all waits bounded
// ------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the barrier, giving up after max_iter polls
// (each try_wait itself suspends for a hardware-defined time).  Returns
// false on timeout; callers then report and skip instead of hanging.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int max_iter) {
    for (int i = 0; i < max_iter; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Bulk prefetch of global memory into L2 (16-byte aligned address and size).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src_gmem, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src_gmem), "r"(bytes) : "memory");
}

__device__ __forceinline__ void report(int32_t* status, int32_t bits) {
    if (status) atomicOr(status, bits);
}


// ------------------------------------------------------------------
// launch parameters (host <-> kernels)
// ------------------------------------------------------------------
// Channel precision boost of the K history: per token vector the kBoostN
// stored positions with the largest 2-bit rounding error |u - c| also keep
// a 4-bit code q4 = clamp(rint(5u), 0, 15) (levels z + s q4 / 5).  Record =
// kBoostN 16-bit entries (position bits 0-6, q4 bits 8-11, a copy of the
// position's 2-bit code in bits 12-13) in increasing position; records of a
// (page, KV head) in one block, token t at 16 t.
constexpr int kBoostN = 8;
constexpr int kBoostRecord = 2 * kBoostN;
constexpr int kBoostBlock = 64 * kBoostRecord;

struct EvictParams {
    const __nv_bfloat16* src_kv;
    const int32_t* src_row;
    const int32_t* dst_seq;
    const int32_t* dst_pos;
    const __nv_bfloat16* new_kv;
    const float* U;
    const float* clip;
    const float* codebook;   // [hk][2] inner level a of the Lloyd-Max codebook, or null (uniform levels)
    uint8_t* pool;
    uint8_t* boost;          // K boost records [num_pages][hk][kBoostBlock], or null (no boost)
    const int32_t* page_table;
    int32_t* status;
    int n_tok, hk, src_rows, batch, max_pages, num_pages;
    int gshift;       // log2(quant_group / 32): 0, 1, 2
    int block_bytes;  // bytes per (page, KV head) block: 4096 + 512 * (4 >> gshift)
};

// Scale/zero pairs per token vector (4, 2 or 1) and the V scale/zero offset
// inside a block (the K pairs start at kKScale).
__host__ __device__ __forceinline__ int sz_pairs(int gshift) { return 4 >> gshift; }
__host__ __device__ __forceinline__ int v_scale_off(int gshift) { return kKScale + kPage * 4 * (4 >> gshift); }

struct DecodeParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* bf16_kv;
    const int32_t* bf16_len;
    const uint8_t* pool;
    const int32_t* page_table;
    const int32_t* hist_len;
    const float* U;
    float* out;
    int32_t* status;
    // workspace sections
    int32_t* counter;     // [64]: [0] INT2 item queue, [kBfCounter] BF16 item queue (separate 128-byte lines)
    int32_t* item_start;  // [B + 1] long items before sequence b (prefix sums)
    int32_t* item_start2; // [B + 1] short tail items before sequence b
    uint32_t* qfrag;      // [B*Hk][NT][8][32][2] fp16 q' fragments (times 2^e_h)
    float* qsum;          // [B*Hk][NT*4][4] group sums of q' (times 2^e_h)
    float* qkinv;         // [B*Hk][4] 2^-e of the (sequence, KV head)'s q' fragments (16-byte records, [0] used)
    float* qrot;          // [B*Hk][4][kD] q' in stored order (fp32), written when boost is set
    float* part;          // [max_items][part_stride]
    float* bf_part;       // [B*Hk][bf_items][part_stride]
    int B, hq, hk, G, NT, nslot, max_pages, num_pages, pps, part_stride;
    int tail_pg;   // last pages of each (sequence, KV head) in short items (0 or 2 * kShortItemPages)
    int bf_items;  // 64-token blocks of the BF16 segment: ceil(nslot / 64)
    int merge_wpr; // merge warps per output row (1, 2, 4, 8)
    int gshift;    // log2(quant_group / 32)
    int block_bytes;
    float qscale;  // sm_scale * log2(e)
    const float* codebook;  // [hk][2] Lloyd-Max inner level a, or null (uniform levels)
    const uint8_t* boost;   // K boost records [num_pages][hk][kBoostBlock], or null (no boost)
};

// Split-K geometry of one sequence with npg history pages: the last
// min(npg, tail_pg) pages go to short items of kShortItemPages, the rest to
// long items of pps pages.
struct SeqSplits {
    int long_pages, n_long, n_short;
};
__host__ __device__ __forceinline__ SeqSplits seq_splits(int npg, int pps, int tail_pg) {
    SeqSplits r;
    const int short_pages = npg < tail_pg ? npg : tail_pg;
    r.long_pages = npg - short_pages;
    r.n_long = (r.long_pages + pps - 1) / pps;
    r.n_short = (short_pages + kShortItemPages - 1) / kShortItemPages;
    return r;
}

// offline rotation calibration (calibrate.cu)
struct CalibParams {
    const __nv_bfloat16* q;    // [n_q][hq][kD] calibration queries
    const __nv_bfloat16* kv;   // [n_t][hk][2][kD] calibration tokens
    float* o;                  // [n_q][hq][kD] attention outputs (scratch)
    float* C;                  // [2][hk][kD][kD] covariance sums (scratch): K, then V
    float* U;                  // [hk][2][kD][kD] out
    float* lam;                // [hk][2][kD] out, nullable
    int* status;
    int n_q, n_t, hq, hk;
    float sm_scale;
};
cudaError_t launch_calibrate(const CalibParams& p, cudaStream_t st);

constexpr int kMaxClipGrid = 32;   // candidate clip ratios per search
struct ClipParams {
    const __nv_bfloat16* kv;   // [n_t][hk][2][kD] calibration tokens
    const float* U;            // [hk][2][kD][kD]
    const float* grid;         // [n_grid] candidate ratios (device)
    double* err;               // [hk * 2][kMaxClipGrid] squared-error sums (scratch)
    float* clip;               // [hk][2] out
    float* mse;                // [hk][2][n_grid] out, nullable
    int n_t, hk, n_grid, gshift;
};
cudaError_t launch_calibrate_clip(const ClipParams& p, cudaStream_t st);

struct FitParams {
    const __nv_bfloat16* kv;   // [n_t][hk][2][kD] calibration tokens
    const float* U;            // [hk][2][kD][kD]
    const float* clip;         // [hk][2]
    float* v;                  // [hk * 2][n_t][kD] folded code coordinates (scratch)
    float* a;                  // [hk][2] out: the inner level of each codebook
    int n_t, hk, gshift;
};
cudaError_t launch_calibrate_codebook(const FitParams& p, cudaStream_t st);

cudaError_t launch_evict(const EvictParams& p, cudaStream_t st);
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t st, cudaEvent_t ev_int2_start,
                          cudaEvent_t ev_int2_stop);

}  // namespace oscar
