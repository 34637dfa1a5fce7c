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

// (x & mask) | bits in one LOP3
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t x, uint32_t mask, uint32_t bits) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "r"(mask), "r"(bits));
    return r;
}

// Two 2-bit codes at bits 4-5 and 20-21 of x -> bf16x2 (8 + c_lo, 8 + c_hi):
// bf16 0x4100 is 8.0 with 7 mantissa bits, so code c placed in mantissa
// bits 4-5 reads as 8 + c exactly.
__device__ __forceinline__ uint32_t codes_to_bf16x2(uint32_t x) {
    return lop3_and_or(x, 0x00300030u, 0x41004100u);
}

// bf16x2 with lo -> bits 0-15, hi -> bits 16-31, round to nearest even
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t rotr(uint32_t x, uint32_t n) { return __funnelshift_r(x, x, n); }

// Code pairs -> bf16x2 MMA operands.  A code pair sits at bits (P, P+16) of
// a 32-bit word (P = 2 * group in bytes 0/2; bytes 1/3 are first shifted
// down by 8).  Placed in bf16 mantissa bits T..T+1 under the exponent of
// M = 2^(7-T), a code c reads as the exact value M + c, so a group whose
// codes already sit at T = P in {0, 2, 4} needs a single logic op; the
// offset M is removed afterwards with the zero point (z - M s).  Pairs are
// moved up by T - P bits with a multiply by 4 or 16, and pairs at P = 6 down
// to T = 4 by the high word of a multiply by 2^30.  K and V use M = 8 for
// every group: the tensor core's fp32 accumulation error scales with the
// magnitude M * (sum of the other operand) the accumulator carries, and a
// larger offset (128 for K, 32 for V) cost a factor two of the attention
// error budget on heavy-tailed data.
// The multipliers are held in registers made opaque by a warp shuffle, so
// the compiler keeps them as integer multiply-adds (FMA pipe) instead of
// shifts or constant loads.
struct CodeMul {
    uint32_t m4, m16, mh30;
};

__device__ __forceinline__ CodeMul code_mul_regs(const uint32_t* mul_param) {
    CodeMul c;
    c.m4 = __shfl_sync(kFull, mul_param[1], 0);
    c.m16 = __shfl_sync(kFull, mul_param[2], 0);
    c.mh30 = __shfl_sync(kFull, mul_param[3], 0);
    return c;
}

// bf16 exponent bits of M = 2^(7-T) in both halves
template <int T>
struct Magic {
    static constexpr uint32_t bits = T == 0 ? 0x43004300u : (T == 2 ? 0x42004200u : 0x41004100u);
};

// pair at bits (P, P+16) -> bf16x2 (M + c_lo, M + c_hi), M = 2^(7-T)
template <int P, int T>
__device__ __forceinline__ uint32_t unpack_pair(uint32_t x, const CodeMul& m) {
    constexpr uint32_t kMask = 0x00030003u << P;
    uint32_t r;
    if constexpr (P == T) {
        r = lop3_and_or(x, kMask, Magic<T>::bits);
    } else if constexpr (T - P == 2) {
        asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(x & kMask), "r"(m.m4), "r"(Magic<T>::bits));
    } else if constexpr (T - P == 4) {
        asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(x & kMask), "r"(m.m16), "r"(Magic<T>::bits));
    } else {
        static_assert(P == 6 && T == 4, "unsupported code move");
        asm("mad.hi.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(x & kMask), "r"(m.mh30), "r"(Magic<T>::bits));
    }
    return r;
}

// code offset M of each 32-position block: 8 for K and V
__device__ __forceinline__ constexpr float k_magic(int) { return 8.f; }
__device__ __forceinline__ constexpr float v_magic(int) { return 8.f; }

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

// Selector of the bf16 hi / lo split below: a lane taking the hi parts uses
// (a, sign) = (0, 0), a lane taking the lo parts (1, 0x80000000).
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

__device__ __forceinline__ void report(int32_t* status, int32_t bits) {
    if (status) atomicOr(status, bits);
}


// ------------------------------------------------------------------
// launch parameters (host <-> kernels)
// ------------------------------------------------------------------
struct EvictParams {
    const __nv_bfloat16* src_kv;
    const int32_t* src_row;
    const int32_t* dst_seq;
    const int32_t* dst_pos;
    const __nv_bfloat16* new_kv;
    const float* U;
    const float* clip;
    uint8_t* pool;
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
    int32_t* counter;     // [1]
    int32_t* item_start;  // [B + 1]
    uint32_t* qfrag;      // [B*Hk][NT][8][32][2]
    float* qsum;          // [B*Hk][NT*4][4]
    float* part;          // [max_items][part_stride]
    float* bf_part;       // [B*Hk][bf_items][part_stride]
    int B, hq, hk, G, NT, nslot, max_pages, num_pages, pps, part_stride;
    int bf_items;  // 64-token blocks of the BF16 segment: ceil(nslot / 64)
    int merge_wpr; // merge warps per output row (1, 2, 4, 8)
    int gshift;    // log2(quant_group / 32)
    int block_bytes;
    float qscale;  // sm_scale * log2(e)
    // multipliers that move a code pair from bits (P, P+16) to (T, T+16):
    // [1] = 4 and [2] = 16 (low product, T - P = 2 or 4), [3] = 2^30 (high
    // product, P = 6 to T = 4).  Passed at run time so the compiler keeps
    // them as integer multiply-adds (FMA pipe) instead of shifts.
    uint32_t code_mul[8];
};

cudaError_t launch_evict(const EvictParams& p, cudaStream_t st);
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t st, cudaEvent_t ev_int2_start,
                          cudaEvent_t ev_int2_stop);

}  // namespace oscar
