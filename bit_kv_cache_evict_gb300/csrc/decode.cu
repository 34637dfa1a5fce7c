// decode.cu -- decode attention over the three-segment pool (BF16 sink |
// INT2 history | BF16 recent), following the serving path of
// "卓绝TurboQuant：Together AI把2-bit KV Cache推向实在行状" (figure
// "从离线校准到在线推理的 pipeline": an INT2 kernel that unpacks,
// dequantises with scale/zero and accumulates in floating point, a BF16
// kernel for sink/recent, and an online-softmax merge).
//
// Kernels, in launch order:
//   prep_kernel       q' = q . U_K . H . P scaled by sm_scale*log2(e), split
//                     into fp16 hi+lo MMA fragments; work plan (split-K items).
//   int2_kernel<NT>   persistent warps; each takes split-K items (a run of
//                     history pages of one (sequence, KV head)), streams the
//                     6 KB page blocks into shared memory with bulk async
//                     copies, and runs both products on tensor cores
//                     (mma.sync m16n8k16 fp16 -> fp32) straight from the
//                     packed codes.
//   bf16_kernel       sink + recent window per (sequence, KV head).
//   merge_kernel      log-sum-exp merge of the INT2 splits, un-rotation by
//                     R_V^T (bit-reversal, Hadamard, U_V^T), merge with the
//                     BF16 partial.
//
// Exact factoring used by int2_kernel.  With codes c, per-(token, group)
// fp16 scale s and zero z, and the code left in an otherwise clear 16-bit
// pattern at bit P_b for the 32-position block b (see code_pair_lo), which
// reads c * 2^(P_b - 24) as fp16 and c * 2^(P_b - 133) as bf16:
//   logit_t = sum_b s~_tb * D_tb + z_tb * Q_b,
//       D_tb = sum_{j in b} c_tj 2^(P_b - 24) q'_j 2^e   (fp16 MMA, tokens x heads),
//       s~_tb = s_tb 2^(24 - P_b - e),  Q_b = sum_{j in b} q'_j,
//       e one power of two per (sequence, KV head) from prep;
//   o'_j   = 2^(24 - P_b) sum_t W_t,b(j) c_tj 2^(P_b - 24) + sum_t p_t z_tb,
//       W_tb = p_t s_tb                                  (fp16 MMA, dims x heads).
// q' 2^e and W are split into fp16 hi + lo (22 bits); codes are exact and
// carry no offset.
#include "oscar_common.cuh"

namespace oscar {


// ---------------------------------------------------------------------------
// prep: rotated query fragments + split-K plan
// ---------------------------------------------------------------------------
// Block (kv, chunk of kPrepSeqs sequences): U_K of that KV head is staged in
// shared memory once; warp w then handles (b, nt, hh) units: head
// h = kv*G + 4*nt + hh (hh >= G: zero padding columns).  Block (last x,
// y = 0) builds the plan.
constexpr int kPrepSeqs = 2;
constexpr int kPrepThreads = 256;
constexpr int kPrepUnits = kPrepSeqs * 2 * 4;  // (b, nt, hh) units of a block at most
constexpr int kPrepSmem = kD * kD * 4 + kPrepUnits * kD * 4 + kPrepUnits * 4;

__device__ __forceinline__ void prep_body(const DecodeParams& p);

// Launched as a programmatic dependent of the eviction (it reads neither the
// pool nor the BF16 segment), so the two overlap.  One block waits for the
// eviction's completion before it exits, which keeps this grid from
// completing earlier, so that everything launched after it sees the evicted
// tokens; the other blocks leave as soon as their work is done (their SM
// slots go to the rest of the grid and to the INT2 kernel's blocks).
// 40 registers, so that two blocks fit on an SM beside the eviction's blocks
// (the grid is one wave there).
__global__ void __launch_bounds__(kPrepThreads, 6) prep_kernel(DecodeParams p) {
    pdl_trigger();
    prep_body(p);
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) pdl_wait();
}

__device__ __forceinline__ void prep_body(const DecodeParams& p) {
    extern __shared__ __align__(16) float psm[];
    float* Us = psm;                       // [a][k] = U_K[a][k]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    if (blockIdx.x == gridDim.x - 1) {  // plan
        if (blockIdx.y != 0 || warp != 0) return;
        // long items of every sequence first, then the short tail items
        int run_long = 0, run_short = 0;
        if (lane == 0) {
            p.item_start[0] = 0;
            p.item_start2[0] = 0;
            p.counter[0] = 0;
            p.counter[kBfCounter] = 0;
        }
        for (int base = 0; base < p.B; base += 32) {
            const int b = base + lane;
            int n_long = 0, n_short = 0;
            if (b < p.B) {
                int h = p.hist_len[b];
                if (h < 0 || h > p.max_pages * kPage) {
                    report(p.status, OSCAR_STATUS_BAD_POS);
                    h = min(max(h, 0), p.max_pages * kPage);
                }
                const SeqSplits sp = seq_splits((h + kPage - 1) / kPage, p.pps, p.tail_pg);
                n_long = sp.n_long * p.hk;
                n_short = sp.n_short * p.hk;
            }
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                const int v = __shfl_up_sync(kFull, n_long, m), w = __shfl_up_sync(kFull, n_short, m);
                if (lane >= m) {
                    n_long += v;
                    n_short += w;
                }
            }
            if (b < p.B) {
                p.item_start[b + 1] = run_long + n_long;
                p.item_start2[b + 1] = run_short + n_short;
            }
            run_long += __shfl_sync(kFull, n_long, 31);
            run_short += __shfl_sync(kFull, n_short, 31);
        }
        return;
    }

    const int kv = blockIdx.y;
    const int b0 = blockIdx.x * kPrepSeqs;
    const int nseq = min(kPrepSeqs, p.B - b0);
    {   // U_K -> shared memory, all copies in flight at once
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.U + ((size_t)kv * 2 + 0) * kD * kD);
        uint8_t* dst = reinterpret_cast<uint8_t*>(Us);
        for (int i = threadIdx.x; i < kD * kD / 4; i += kPrepThreads)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst + 16 * i)), "l"(src + 16 * i)
                         : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
        asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();

    // Two passes over the block's (b, nt, hh) units.  Pass 1: q' of every
    // unit into shared memory and its largest |q'|.  Pass 2: one power of
    // two 2^e per (sequence, KV head), from the largest |q'| over the KV
    // group's heads (times the Lloyd-Max plane weight kappa when it is
    // above 1), put into [2^13, 2^14); the fp16 fragments of q' 2^e, the
    // group sums of q' and 2^-e (which int2_kernel folds into the K scales).
    const int units = nseq * p.NT * 4;
    float* qU = psm + kD * kD;               // [unit][kD] q' in stored order
    float* mxU = qU + kPrepUnits * kD;       // [unit] largest |q'| (0 for padding)
    for (int u = warp; u < units; u += kPrepThreads / 32) {
        const int hl = 4 * ((u >> 2) % p.NT) + (u & 3);  // head within the KV group
        const int b = b0 + (u >> 2) / p.NT;
        const int bk = b * p.hk + kv;
        float* qs = qU + u * kD;
        if (hl >= p.G) {  // padding column pair
            if (lane == 0) mxU[u] = 0.f;
            if (p.boost)
                *reinterpret_cast<float4*>(p.qrot + ((size_t)bk * p.NT * 4 + hl) * kD + 4 * lane) =
                    make_float4(0.f, 0.f, 0.f, 0.f);
            continue;
        }
        const int h = kv * p.G + hl;
        const uint2 qr = *reinterpret_cast<const uint2*>(p.q + ((size_t)b * p.hq + h) * kD + 4 * lane);
        const float x[4] = {bf16_lo(qr.x), bf16_hi(qr.x), bf16_lo(qr.y), bf16_hi(qr.y)};
        float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int a4 = 0; a4 < kD; a4 += 4) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float xa = __shfl_sync(kFull, x[i], a4 >> 2);
                const float4 uu = *reinterpret_cast<const float4*>(Us + (size_t)(a4 + i) * kD + 4 * lane);
                y[0] = fmaf(xa, uu.x, y[0]);
                y[1] = fmaf(xa, uu.y, y[1]);
                y[2] = fmaf(xa, uu.z, y[2]);
                y[3] = fmaf(xa, uu.w, y[3]);
            }
        }
        {  // Hadamard, in-lane stages
            const float t0 = y[0] + y[1], t1 = y[0] - y[1], t2 = y[2] + y[3], t3 = y[2] - y[3];
            y[0] = t0 + t2;
            y[2] = t0 - t2;
            y[1] = t1 + t3;
            y[3] = t1 - t3;
        }
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float o = __shfl_xor_sync(kFull, y[k], m);
                y[k] = upper ? o - y[k] : y[k] + o;
            }
        }
        const float scale = (float)kInvSqrtD * p.qscale;
        const int r5 = bitrev5(lane);
        float mx = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float v = y[k] * scale;
            qs[32 * bitrev2(k) + r5] = v;  // stored order
            mx = fmaxf(mx, fabsf(v));
        }
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, m));
        if (lane == 0) mxU[u] = mx;
        __syncwarp();
        if (p.boost)  // q' itself for the boost corrections
            *reinterpret_cast<float4*>(p.qrot + ((size_t)bk * p.NT * 4 + hl) * kD + 4 * lane) =
                *reinterpret_cast<const float4*>(qs + 4 * lane);
    }
    __syncthreads();

    float kappa = 1.f;  // Lloyd-Max plane weight bound of this KV head's K levels
    if (p.codebook) {
        const float a = __ldg(p.codebook + kv * 2);
        kappa = fmaxf(1.f, fabsf(a > 0.f ? (3.f - 3.f * a) / (2.f * a) : 0.f));
    }
    for (int u = warp; u < units; u += kPrepThreads / 32) {
        const int hh = u & 3;
        const int nt = (u >> 2) % p.NT;
        const int b = b0 + (u >> 2) / p.NT;
        const int bk = b * p.hk + kv;
        const int hl = 4 * nt + hh;
        const int u0 = u - (u % (p.NT * 4));     // first unit of this (sequence, KV head)
        float mx = mxU[u0];
        for (int i = 1; i < p.NT * 4; ++i) mx = fmaxf(mx, mxU[u0 + i]);
        mx *= kappa;
        const int ex = mx > 0.f ? (int)((__float_as_uint(mx) >> 23) & 0xffu) - 127 : 0;
        const int e = min(126, max(-126, kQTopExp - ex));
        const float up = __uint_as_float((uint32_t)(127 + e) << 23);
        if (u == u0 && lane < 4) p.qkinv[(size_t)bk * 4 + lane] = lane == 0 ? __uint_as_float((uint32_t)(127 - e) << 23) : 0.f;
        uint32_t* frag = p.qfrag + ((size_t)bk * p.NT + nt) * 8 * 32 * 2;
        float* qsum = p.qsum + ((size_t)bk * p.NT * 4 + hl) * 4;
        const int ks = lane >> 2, tq = lane & 3;
        if (hl >= p.G) {  // padding column pair: zeros
#pragma unroll
            for (int par = 0; par < 2; ++par) {
                const int L = (2 * hh + par) * 4 + tq;
                *reinterpret_cast<uint2*>(frag + ((size_t)ks * 32 + L) * 2) = make_uint2(0u, 0u);
            }
            if (lane < 4) qsum[lane] = 0.f;
            continue;
        }
        const float* qs = qU + u * kD;

        // group sums of q' (the two fp16 parts add up to q' 2^e within
        // 2^-22 relative)
        float gs = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) gs += qs[4 * lane + k];
#pragma unroll
        for (int m = 1; m < 8; m <<= 1) gs += __shfl_xor_sync(kFull, gs, m);
        if ((lane & 7) == 0) qsum[lane >> 3] = gs;

        // fragments: lane -> (ks, tq), k-step ks = (group g = ks/2, half h = ks%2)
        // covers in-group indices 8tq + 4h + {0,2} (b0) and + {1,3} (b1), the
        // four codes of bytes 4(2tq+h)..4(2tq+h)+3 of group g's slot; column
        // 2hh = hi, 2hh+1 = lo
        const int base = 32 * (ks >> 1) + 8 * tq + 4 * (ks & 1);
        const float v[4] = {qs[base] * up, qs[base + 2] * up, qs[base + 1] * up, qs[base + 3] * up};
        uint32_t h01, h23, l01, l23;
        split_f16(v, h01, h23, l01, l23);
        if (p.NT == 2) {
            // eight heads: column = head, hi and lo parts in two fragment sets
            uint32_t* fr = p.qfrag + (size_t)bk * 2 * 8 * 32 * 2;  // [part][ks][32] uint2
            *reinterpret_cast<uint2*>(fr + ((size_t)(0 * 8 + ks) * 32 + 4 * hl + tq) * 2) = make_uint2(h01, h23);
            *reinterpret_cast<uint2*>(fr + ((size_t)(1 * 8 + ks) * 32 + 4 * hl + tq) * 2) = make_uint2(l01, l23);
        } else {
            *reinterpret_cast<uint2*>(frag + ((size_t)ks * 32 + (2 * hh) * 4 + tq) * 2) = make_uint2(h01, h23);
            *reinterpret_cast<uint2*>(frag + ((size_t)ks * 32 + (2 * hh + 1) * 4 + tq) * 2) = make_uint2(l01, l23);
        }
    }
}

// ---------------------------------------------------------------------------
// INT2 split-K decode
// ---------------------------------------------------------------------------
// Block = 4 consumer warps + 1 producer warp.  The producer takes split-K
// items from a global counter and streams their 6 KB page blocks into a
// ring of 8 shared-memory stages with bulk async copies (completion on a
// "full" mbarrier).  Ring slot n goes to consumer warp n % 4, so each warp
// owns two stages and attends over whole 64-token pages: the pages of an
// item are dealt round-robin to the four warps (an item's slot count is
// padded to a multiple of four with empty slots, so that every warp sees
// every item).  Per page a warp converts the page's scales, computes the
// logits of its four 16-token tiles, updates its softmax state once, and
// runs the P.V products; it then releases the stage on an "empty"
// mbarrier.  At an item's end the four warps merge their partial states in
// shared memory and write one partial per item.  In the uniform four-head
// kernel the producer also copies each item's q' data (fragments, group
// sums, 2^-e) into one of two item buffers when it starts the item, so that
// the consumers find it in shared memory at the item's first page.  Every
// wait is bounded; on a timeout the block reports OSCAR_STATUS_TIMEOUT, lets
// its copies land and exits.
constexpr int kConsumerWarps = 4;
constexpr int kStages = 2 * kConsumerWarps;
// Poll budget of every bounded mbarrier wait: a try_wait suspends about 4 us
// when the phase is not complete (measured on GB300), so 2^18 polls give up
// after about a second, far beyond any legitimate wait (a page copy, or the
// other consumer warps finishing an item).
constexpr int kWaitPolls = 1 << 18;
constexpr int kInt2Threads = (kConsumerWarps + 1) * 32;
constexpr int kFlagFirst = 1, kFlagLast = 2, kFlagPad = 4;

struct StageInfo {
    int item, b, kv, valid_flags;  // valid tokens in bits 0-7, flags above
    int pid, pad[3];               // page id (read by the boost variant)
};

// Blocks per SM and ring stages of an int2_kernel instantiation: three
// blocks (128 registers) with eight stages for up to four heads; for eight
// heads three blocks with seven stages (the shared memory of three blocks),
// except the Lloyd-Max and boost kernels, which keep two blocks (168
// registers) and eight stages.
template <int NT, bool LM, bool BOOST>
__host__ __device__ constexpr int int2_blocks_per_sm() { return (NT == 1 || !(LM || BOOST)) ? 3 : 2; }
template <int NT, bool LM, bool BOOST>
__host__ __device__ constexpr int int2_stages() { return (NT == 2 && int2_blocks_per_sm<NT, LM, BOOST>() == 3) ? kStages - 1 : kStages; }
// Whether an instantiation prefetches each item's q' data into shared
// memory (the uniform four-head kernel; the others load it at the item's
// first page).
template <int NT, bool LM, bool BOOST>
__host__ __device__ constexpr bool int2_q_prefetch() { return NT == 1 && !LM && !BOOST; }

template <int NT, int NS = kStages>
struct Int2Smem {
    static constexpr int G4 = NT * 4;  // head columns (padded to 4 per n-tile)
    // per-warp scratch: K s [64] float4 | K z [64] float4 | V z [64]
    // float4 | V s [4][72] float (token order pv_pos) | P [G4][72] float
    // (same token order).  Reused at an item's end for
    // the warp's (o', m, l) state [G4][kD + 2].
    static constexpr int kWKs = 0, kWKz = 1024, kWVz = 2048, kWVs = 3072, kWP = 3072 + 4 * 72 * 4;
    static constexpr int kWarpBytes0 = kWP + G4 * 72 * 4;
    static constexpr int kMergeBytes = G4 * (kD + 2) * 4;
    static constexpr int kWarpBytes = kWarpBytes0 > kMergeBytes ? kWarpBytes0 : kMergeBytes;
    static constexpr int kStage = 0;
    static constexpr int kInfo = kStage + NS * kBlock;
    static constexpr int kBars = kInfo + NS * (int)sizeof(StageInfo);
    static constexpr int kWarp = kBars + (2 * NS + 2) * 8;
    // q' fragments of the current item, shared by the four consumer warps
    // (all four are inside the same item between two item-end merges)
    static constexpr int kQf = kWarp + kConsumerWarps * kWarpBytes;       // [NT][8][32] uint2
    static constexpr int kBytes = kQf + NT * 8 * 32 * 8;
    // Lloyd-Max levels: kappa q' fragments of the high-bit plane follow q';
    // channel boost: q' [kD] float4 (four heads) there instead
    static constexpr int kBytesLM = kBytes + NT * 8 * 32 * 8;
    static_assert(NT * 8 * 32 * 8 >= kD * NT * 16, "room for the boost's q'");
    // The uniform four-head kernel instead has two item buffers, filled by
    // the producer with bulk copies when it starts an item: q' fragments
    // [8][32] uint2, the group sums [4] float4, 2^-e (a 16-byte record);
    // then their "full" and "empty" barriers.
    static constexpr int kQbFrag = 0, kQbSum = 8 * 32 * 8, kQbKinv = kQbSum + 4 * 16, kQbBytes = kQbKinv + 16;
    static constexpr int kQb = kQf;                      // [2][kQbBytes]
    static constexpr int kQbBars = kQb + 2 * kQbBytes;   // qfull[2], qempty[2]
    static constexpr int kBytesQP = kQbBars + 4 * 8;
    static_assert(kQb % 16 == 0 && kQbBytes % 16 == 0, "bulk-copy destinations 16-byte aligned");
};

__device__ __forceinline__ int find_seq(const int32_t* item_start, int B, int item) {
    int lo = 0, hi = B;  // largest b with item_start[b] <= item
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(item_start + mid) <= item) lo = mid;
        else hi = mid;
    }
    return lo;
}

// A-operand registers of one K k-step (slot g, word half h) from the
// token-row words of rows gID and gID + 8 (w*) and their >> 8 copies (w*8).
template <int G>
__device__ __forceinline__ void k_operands(uint32_t wa, uint32_t wb, uint32_t was, uint32_t wbs, uint32_t& a0,
                                           uint32_t& a1, uint32_t& a2, uint32_t& a3) {
    a0 = code_pair_lo<G>(wa, was);
    a1 = code_pair_lo<G>(wb, wbs);
    a2 = code_pair_hi<G>(wa, was);
    a3 = code_pair_hi<G>(wb, wbs);
}

// A-operand registers of one V m-tile half (slot g): plane words r0, r1 and
// their >> 8 copies.
template <int G>
__device__ __forceinline__ void v_operands(uint32_t r0, uint32_t r1, uint32_t r0s, uint32_t r1s, uint32_t& a0,
                                           uint32_t& a1, uint32_t& a2, uint32_t& a3) {
    a0 = code_pair_lo<G>(r0, r0s);
    a1 = code_pair_lo<G>(r1, r1s);
    a2 = code_pair_hi<G>(r0, r0s);
    a3 = code_pair_hi<G>(r1, r1s);
}

// Position of token t (0..63) in the warp's probability and V-scale rows.
// The P.V products take the page's tokens in 16 groups of four: k-step m of
// lane quad tq covers group q = 4 tq + m (tokens 4q .. 4q+3, whose V codes
// are bytes 4q .. 4q+3 of every code plane, so one 16-byte load per plane
// serves all four k-steps).  Group q sits in 16-byte chunk 4 tq + (m ^ tq)
// of a row, which keeps the lanes of one shared-memory wavefront on
// distinct banks; inside a chunk the order is pv_slot (tokens 4q, 4q+2 |
// 4q+1, 4q+3 as the two B-operand pairs).
__device__ __forceinline__ int pv_pos(int t) {
    const int q = t >> 2, tq = q >> 2, m = q & 3;
    return 4 * (4 * tq + (m ^ tq)) + pv_slot(t & 3);
}
constexpr int kPvRow = 72;  // floats per probability / V-scale row (64 + 8: conflict-free stores)

// The page's scales into the warp's scratch: for each token row and each
// 32-position block b (quantisation group b >> GS), fp32 s scaled by the
// block's power of two (K: k_scale_up) and z; rows past the
// valid tokens are zero.  K rows: s~ and z as float4 per token; V rows: z per
// token, and s~ in the P.V token order (pv_pos).
template <bool FULL, int GS>
__device__ __forceinline__ void page_scales_g(const uint8_t* blk, int valid, float4* ksS, float4* kzS, float4* vzS,
                                              float* vsS, float kmul, float vmul) {
    constexpr int NG = 4 >> GS;  // (s, z) pairs per token vector
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int which = it >> 1, t = lane + 32 * (it & 1);
        float sv[4], zz[4];
        if (FULL || t < valid) {
            const uint8_t* base = blk + (which ? v_scale_off(GS) : kKScale) + t * 4 * NG;
            uint32_t w[NG];
            if constexpr (NG == 4) {
                const uint4 v = *reinterpret_cast<const uint4*>(base);
                w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
            } else if constexpr (NG == 2) {
                const uint2 v = *reinterpret_cast<const uint2*>(base);
                w[0] = v.x; w[1] = v.y;
            } else {
                w[0] = *reinterpret_cast<const uint32_t*>(base);
            }
            float s_g[NG], z_g[NG];
#pragma unroll
            for (int k = 0; k < NG; ++k) {
                s_g[k] = half_lo(w[k]);
                z_g[k] = half_hi(w[k]);
            }
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                sv[b] = s_g[b >> GS] * (which ? vmul : k_scale_up(b) * kmul);
                zz[b] = z_g[b >> GS];
            }
        } else {
#pragma unroll
            for (int b = 0; b < 4; ++b) sv[b] = zz[b] = 0.f;
        }
        if (which == 0) {
            ksS[t] = make_float4(sv[0], sv[1], sv[2], sv[3]);
            kzS[t] = make_float4(zz[0], zz[1], zz[2], zz[3]);
        } else {
            vzS[t] = make_float4(zz[0], zz[1], zz[2], zz[3]);
            const int ps = pv_pos(t);
#pragma unroll
            for (int b = 0; b < 4; ++b) vsS[b * kPvRow + ps] = sv[b];
        }
    }
}

// kmul / vmul multiply the K / V scales (K: the item's 2^-e, times the
// Lloyd-Max inner level a; V: a; 1 for the uniform levels)
template <bool FULL>
__device__ __forceinline__ void page_scales(const uint8_t* blk, int valid, int gshift, float4* ksS, float4* kzS,
                                            float4* vzS, float* vsS, float kmul = 1.f, float vmul = 1.f) {
    switch (gshift) {  // warp-uniform, once per page
        case 0: page_scales_g<FULL, 0>(blk, valid, ksS, kzS, vzS, vsS, kmul, vmul); break;
        case 1: page_scales_g<FULL, 1>(blk, valid, ksS, kzS, vzS, vsS, kmul, vmul); break;
        default: page_scales_g<FULL, 2>(blk, valid, ksS, kzS, vzS, vsS, kmul, vmul); break;
    }
}

// Lloyd-Max codebook of an item: levels {0, a, 3 - a, 3} in units of s above
// z.  With c = b0 + 2 b1 the level is a c + (3 - 3a) b1, so a codebook
// product is a times the code product plus (3 - 3a) / 2 times the product
// of the high-bit plane (the plane's operand reads 2 b1 in the code's units).
// The factor a goes into the scales, kappa = (3 - 3a) / (2a) weighs the
// plane.  a <= 0 selects the uniform levels (kappa = 0).
struct Codebook {
    float ka, va, kk, vk;  // a and kappa for K and V
};
__device__ __forceinline__ Codebook codebook_of(const float* cb, int kv) {
    float a[2];
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        const float x = cb ? __ldg(cb + kv * 2 + w) : 0.f;
        a[w] = x > 0.f ? x : 1.f;
    }
    return {a[0], a[1], (3.f - 3.f * a[0]) / (2.f * a[0]), (3.f - 3.f * a[1]) / (2.f * a[1])};
}
// high-bit plane of a code operand register (codes at bits P, P + 1 of each half)
template <int SLOT>
__device__ __forceinline__ uint32_t high_plane(uint32_t a) { return a & (0x00020002u << slot_bit(SLOT)); }
template <int SLOT>
__device__ __forceinline__ void high_planes(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t& c0,
                                            uint32_t& c1, uint32_t& c2, uint32_t& c3) {
    c0 = high_plane<SLOT>(a0);
    c1 = high_plane<SLOT>(a1);
    c2 = high_plane<SLOT>(a2);
    c3 = high_plane<SLOT>(a3);
}


// fp16 B fragment of kappa q' from one of q': column n of a head's column
// pair holds its hi (n even) or lo (n odd) part, the partner column sits in
// lane ^ 4.  q' = hi + lo is rebuilt, scaled and split again (prep's power
// of two leaves room for kappa).
__device__ __forceinline__ uint2 scaled_fragment(uint2 f, float kappa, int is_lo) {
    const uint32_t ox = __shfl_xor_sync(kFull, f.x, 4), oy = __shfl_xor_sync(kFull, f.y, 4);
    const uint32_t hx = is_lo ? ox : f.x, hy = is_lo ? oy : f.y, lx = is_lo ? f.x : ox, ly = is_lo ? f.y : oy;
    const float y[4] = {kappa * (half_lo(hx) + half_lo(lx)), kappa * (half_hi(hx) + half_hi(lx)),
                        kappa * (half_lo(hy) + half_lo(ly)), kappa * (half_hi(hy) + half_hi(ly))};
    uint32_t h01, h23, l01, l23;
    split_f16(y, h01, h23, l01, l23);
    return is_lo ? make_uint2(l01, l23) : make_uint2(h01, h23);
}

// One page of INT2 history for one consumer warp: the page's scales, the
// logits of its four 16-token tiles, one online-softmax update, and the P.V
// products.  FULL (all 64 tokens valid, the common case) removes the
// per-tile conditions of the logit phase so that the four tiles' work can
// interleave.
template <int NT, bool FULL, bool LM = false, bool BOOST = false>
__device__ __forceinline__ void attend_page(const uint8_t* blk, int valid, uint8_t* wbuf, const uint2* qfS,
                                            const float4 (&qsv)[NT], float kq, float (&m_run)[NT],
                                            float (&l_run)[NT], float (&zacc)[NT][4], float (&acc_o)[NT][8][4],
                                            const SplitSel& take_lo, int gshift, const Codebook& cbk = {},
                                            const float4* qbS = nullptr, const uint8_t* brec = nullptr) {
    using SM = Int2Smem<NT>;
    const int lane = threadIdx.x & 31, gID = lane >> 2, tq = lane & 3;
    if (FULL) valid = kPage;
    float4* ksS = reinterpret_cast<float4*>(wbuf + SM::kWKs);   // [64] K s
    float4* kzS = reinterpret_cast<float4*>(wbuf + SM::kWKz);   // [64] K z
    float4* vzS = reinterpret_cast<float4*>(wbuf + SM::kWVz);   // [64] V z
    float* vsS = reinterpret_cast<float*>(wbuf + SM::kWVs);     // [4][kPvRow] V s at pv_pos
    float* pS = reinterpret_cast<float*>(wbuf + SM::kWP);       // [G4][kPvRow] P at pv_pos
    const int ntile = FULL ? 4 : (valid + 15) >> 4;             // warp-uniform, 1..4
    uint4 br0 = make_uint4(0u, 0u, 0u, 0u), br1 = br0;         // boost records of tokens 2 lane, 2 lane + 1
    if constexpr (BOOST) {
        br0 = __ldg(reinterpret_cast<const uint4*>(brec) + 2 * lane);
        br1 = __ldg(reinterpret_cast<const uint4*>(brec) + 2 * lane + 1);
    }

    // K scales times 2^-e (the power of two of the q' fragments)
    if constexpr (LM) page_scales<FULL>(blk, valid, gshift, ksS, kzS, vzS, vsS, cbk.ka * kq, cbk.va * kLmVDown);
    else page_scales<FULL>(blk, valid, gshift, ksS, kzS, vzS, vsS, kq);
    __syncwarp();

    // -- logits of the page's tiles: A rows gID / gID+8 = tokens 16m+gID /
    //    16m+gID+8; k-step (g, h) takes slot g of words 2tq+h of each token
    float la[4][NT], lb[4][NT];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) la[m][nt] = lb[m][nt] = -INFINITY;
        if (m < ntile) {
            const int ta = 16 * m + gID;
            const uint2 x = *reinterpret_cast<const uint2*>(blk + kKCodes + ta * 32 + 8 * tq);
            const uint2 y = *reinterpret_cast<const uint2*>(blk + kKCodes + (ta + 8) * 32 + 8 * tq);
            const uint32_t wa[2] = {x.x, x.y}, wb[2] = {y.x, y.y};
            const uint32_t wa8[2] = {code_swap(wa[0]), code_swap(wa[1])}, wb8[2] = {code_swap(wb[0]), code_swap(wb[1])};
            float acc[4][NT][4];
#pragma unroll
            for (int g = 0; g < 4; ++g)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[g][nt][e] = 0.f;
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                // half-major order: the four groups' accumulation chains interleave
                const int h = it >> 2, g = it & 3, ks = 2 * g + h;
                uint32_t a0, a1, a2, a3, c0 = 0, c1 = 0, c2 = 0, c3 = 0;
                switch (g) {  // compile-time after unrolling
                    case 0:
                        k_operands<0>(wa[h], wb[h], wa8[h], wb8[h], a0, a1, a2, a3);
                        if (LM) high_planes<0>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                    case 1:
                        k_operands<1>(wa[h], wb[h], wa8[h], wb8[h], a0, a1, a2, a3);
                        if (LM) high_planes<1>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                    case 2:
                        k_operands<2>(wa[h], wb[h], wa8[h], wb8[h], a0, a1, a2, a3);
                        if (LM) high_planes<2>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                    default:
                        k_operands<3>(wa[h], wb[h], wa8[h], wb8[h], a0, a1, a2, a3);
                        if (LM) high_planes<3>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint2 qb = qfS[(nt * 8 + ks) * 32 + lane];
                    mma_f16_16816(acc[g][nt], a0, a1, a2, a3, qb.x, qb.y);
                    if (LM) {  // high-bit plane against kappa q'
                        const uint2 qk = qfS[((NT + nt) * 8 + ks) * 32 + lane];
                        mma_f16_16816(acc[g][nt], c0, c1, c2, c3, qk.x, qk.y);
                    }
                }
            }
            const float4 sA = ksS[ta], sB = ksS[ta + 8], zA = kzS[ta], zB = kzS[ta + 8];
            const float sa[4] = {sA.x, sA.y, sA.z, sA.w}, za[4] = {zA.x, zA.y, zA.z, zA.w};
            const float sb[4] = {sB.x, sB.y, sB.z, sB.w}, zb[4] = {zB.x, zB.y, zB.z, zB.w};
            const bool va = FULL || ta < valid, vb = FULL || ta + 8 < valid;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float qg[4] = {qsv[nt].x, qsv[nt].y, qsv[nt].z, qsv[nt].w};
                float xa = 0.f, xb = 0.f;
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const float da = acc[g][nt][0] + acc[g][nt][1], db = acc[g][nt][2] + acc[g][nt][3];
                    xa = fmaf(sa[g], da, xa);
                    xa = fmaf(za[g], qg[g], xa);
                    xb = fmaf(sb[g], db, xb);
                    xb = fmaf(zb[g], qg[g], xb);
                }
                la[m][nt] = va ? xa : -INFINITY;
                lb[m][nt] = vb ? xb : -INFINITY;
            }
        }
    }

    // -- channel boost: logit corrections q'[pos] s (q4 / 5 - c) of the
    //    boosted positions; lane l computes tokens 2l, 2l + 1 for the four
    //    heads into the P scratch (free until the softmax below)
    if constexpr (BOOST) {
        float4* cS = reinterpret_cast<float4*>(pS);
        const int ng = 4 >> gshift;
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
            const int t = 2 * lane + tt;
            const uint4 rr = tt ? br1 : br0;
            float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < valid) {
                const uint32_t* szw = reinterpret_cast<const uint32_t*>(blk + kKScale + t * 4 * ng);
                const uint32_t wv[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
                for (int e = 0; e < kBoostN; ++e) {
                    const uint32_t ent = wv[e >> 1] >> (16 * (e & 1));
                    const int pos = ent & 127;
                    const float sg = __half2float(__ushort_as_half((unsigned short)(szw[pos >> (5 + gshift)] & 0xffffu)));
                    const float d = sg * fmaf((float)((ent >> 8) & 15u), 0.2f, -(float)((ent >> 12) & 3u));
                    const float4 qv = qbS[pos];
                    c.x = fmaf(d, qv.x, c.x);
                    c.y = fmaf(d, qv.y, c.y);
                    c.z = fmaf(d, qv.z, c.z);
                    c.w = fmaf(d, qv.w, c.w);
                }
            }
            cS[t] = c;
        }
        __syncwarp();
        const float* cf = reinterpret_cast<const float*>(pS);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int ta = 16 * m + gID;
            la[m][0] += cf[ta * 4 + tq];
            lb[m][0] += cf[(ta + 8) * 4 + tq];
        }
        __syncwarp();
    }

    // -- online softmax (base 2), once per page; every token's p is written
    //    (0 for the invalid ones)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        float mx = fmaxf(la[0][nt], lb[0][nt]);
#pragma unroll
        for (int m = 1; m < 4; ++m) mx = fmaxf(mx, fmaxf(la[m][nt], lb[m][nt]));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
        const float m_new = fmaxf(m_run[nt], mx);
        if (__any_sync(kFull, m_new > m_run[nt])) {  // warp-uniform rescale
            const float alpha = (m_new > m_run[nt]) ? ex2(m_run[nt] - m_new) : 1.f;
            l_run[nt] *= alpha;
#pragma unroll
            for (int g = 0; g < 4; ++g) zacc[nt][g] *= alpha;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc_o[nt][mt][e] *= alpha;
            m_run[nt] = m_new;
        }
        const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int ta = 16 * m + gID;
            const float pa = ex2(la[m][nt] - m_sub), pb = ex2(lb[m][nt] - m_sub);
            if (FULL || m < ntile) {
                l_run[nt] += pa + pb;
                const float4 vzA = vzS[ta], vzB = vzS[ta + 8];
                zacc[nt][0] = fmaf(pa, vzA.x, fmaf(pb, vzB.x, zacc[nt][0]));
                zacc[nt][1] = fmaf(pa, vzA.y, fmaf(pb, vzB.y, zacc[nt][1]));
                zacc[nt][2] = fmaf(pa, vzA.z, fmaf(pb, vzB.z, zacc[nt][2]));
                zacc[nt][3] = fmaf(pa, vzA.w, fmaf(pb, vzB.w, zacc[nt][3]));
            }
            pS[(nt * 4 + tq) * kPvRow + pv_pos(ta)] = pa;
            pS[(nt * 4 + tq) * kPvRow + pv_pos(ta + 8)] = pb;
        }
    }
    __syncwarp();

    // -- values: A rows = dims (m-tile (g, half): in-group index 16 half +
    //    row, code plane 16 half + row, slot g), k = token group 4 tq + m
    //    (tokens 4q, 4q+2 | 4q+1, 4q+3), columns = heads (hi, lo)
    uint4 pv4[4];  // bytes 16 tq .. 16 tq + 15 of planes gID, 8 + gID, 16 + gID, 24 + gID
#pragma unroll
    for (int k = 0; k < 4; ++k)
        pv4[k] = *reinterpret_cast<const uint4*>(blk + kVCodes + (gID + 8 * k) * kPage + 16 * tq);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int chunk = 4 * (4 * tq + (m ^ tq));
        float4 pp[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            pp[nt] = *reinterpret_cast<const float4*>(pS + (nt * 4 + (gID >> 1)) * kPvRow + chunk);
        uint32_t pw[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) pw[k] = m == 0 ? pv4[k].x : m == 1 ? pv4[k].y : m == 2 ? pv4[k].z : pv4[k].w;
        const uint32_t pw8[4] = {code_swap(pw[0]), code_swap(pw[1]), code_swap(pw[2]), code_swap(pw[3])};
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const float4 sg = *reinterpret_cast<const float4*>(vsS + g * kPvRow + chunk);
            uint32_t bb0[NT], bb1[NT], cc0[LM ? NT : 1], cc1[LM ? NT : 1];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if constexpr (LM) {
                    const float2 w0 = mul2(make_float2(pp[nt].x, pp[nt].y), make_float2(sg.x, sg.y));
                    const float2 w1 = mul2(make_float2(pp[nt].z, pp[nt].w), make_float2(sg.z, sg.w));
                    bb0[nt] = split_pair_f16(w0, take_lo);
                    bb1[nt] = split_pair_f16(w1, take_lo);
                    // the high-bit plane's weights kappa * W
                    const float2 kv2 = make_float2(cbk.vk, cbk.vk);
                    cc0[nt] = split_pair_f16(mul2(w0, kv2), take_lo);
                    cc1[nt] = split_pair_f16(mul2(w1, kv2), take_lo);
                } else {
                    bb0[nt] = split_w_pair_f16(make_float2(pp[nt].x, pp[nt].y), make_float2(sg.x, sg.y), take_lo);
                    bb1[nt] = split_w_pair_f16(make_float2(pp[nt].z, pp[nt].w), make_float2(sg.z, sg.w), take_lo);
                }
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const uint32_t r0 = pw[2 * half], r1 = pw[2 * half + 1];
                const uint32_t r08 = pw8[2 * half], r18 = pw8[2 * half + 1];
                uint32_t a0, a1, a2, a3, c0 = 0, c1 = 0, c2 = 0, c3 = 0;
                switch (g) {
                    case 0:
                        v_operands<0>(r0, r1, r08, r18, a0, a1, a2, a3);
                        if (LM) high_planes<0>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                    case 1:
                        v_operands<1>(r0, r1, r08, r18, a0, a1, a2, a3);
                        if (LM) high_planes<1>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                    case 2:
                        v_operands<2>(r0, r1, r08, r18, a0, a1, a2, a3);
                        if (LM) high_planes<2>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                    default:
                        v_operands<3>(r0, r1, r08, r18, a0, a1, a2, a3);
                        if (LM) high_planes<3>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_f16_16816(acc_o[nt][2 * g + half], a0, a1, a2, a3, bb0[nt], bb1[nt]);
                    if (LM) mma_f16_16816(acc_o[nt][2 * g + half], c0, c1, c2, c3, cc0[LM ? nt : 0], cc1[LM ? nt : 0]);
                }
            }
        }
    }
}

// Split two fp32 values into f16x2 registers of their high parts (the
// values with the low 13 bits cleared, see split_pair_f16) and of the
// rounded remainders.
__device__ __forceinline__ void split_both(float2 w, uint32_t& hi, uint32_t& lo) {
    const float2 h = make_float2(__uint_as_float(__float_as_uint(w.x) & 0xffffe000u),
                                 __uint_as_float(__float_as_uint(w.y) & 0xffffe000u));
    hi = pack_f16x2_rn(h.x, h.y);
    const float2 r = sub2(w, h);
    lo = pack_f16x2_rn(r.x, r.y);
}

// attend_page for eight query heads per KV head: the MMA columns are the
// heads, and the hi / lo parts of q' and of P*s enter as two MMAs on the
// same A fragment (accumulating into the same registers).  Lane (gID, tq)
// holds heads 2tq and 2tq + 1.
template <bool FULL, bool BOOST = false, bool LM = false>
__device__ __forceinline__ void attend_page_g8(const uint8_t* blk, int valid, uint8_t* wbuf, const uint2* qfS,
                                               const float4 (&qsv)[2], float kq, float (&m_run)[2],
                                               float (&l_run)[2],
                                               float (&zacc)[2][4], float (&acc_o)[8][4],
                                               int gshift, const float4* qbS = nullptr,
                                               const uint8_t* brec = nullptr, const Codebook& cbk = {}) {
    using SM = Int2Smem<2>;
    const int lane = threadIdx.x & 31, gID = lane >> 2, tq = lane & 3;
    if (FULL) valid = kPage;
    float4* ksS = reinterpret_cast<float4*>(wbuf + SM::kWKs);
    float4* kzS = reinterpret_cast<float4*>(wbuf + SM::kWKz);
    float4* vzS = reinterpret_cast<float4*>(wbuf + SM::kWVz);
    float* vsS = reinterpret_cast<float*>(wbuf + SM::kWVs);
    float* pS = reinterpret_cast<float*>(wbuf + SM::kWP);       // [8 heads][kPvRow]
    const int ntile = FULL ? 4 : (valid + 15) >> 4;
    uint4 br0 = make_uint4(0u, 0u, 0u, 0u), br1 = br0;         // boost records of tokens 2 lane, 2 lane + 1
    if constexpr (BOOST) {
        br0 = __ldg(reinterpret_cast<const uint4*>(brec) + 2 * lane);
        br1 = __ldg(reinterpret_cast<const uint4*>(brec) + 2 * lane + 1);
    }

    // K scales times 2^-e (the power of two of the q' fragments)
    if constexpr (LM) page_scales<FULL>(blk, valid, gshift, ksS, kzS, vzS, vsS, cbk.ka * kq, cbk.va * kLmVDown);
    else page_scales<FULL>(blk, valid, gshift, ksS, kzS, vzS, vsS, kq);
    __syncwarp();

    // -- logits: lg[m] = (token a, head 2tq), (a, 2tq+1), (b, 2tq), (b, 2tq+1)
    //    with a = 16m + gID, b = a + 8
    float lg[4][4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
#pragma unroll
        for (int e = 0; e < 4; ++e) lg[m][e] = -INFINITY;
        if (m < ntile) {
            const int ta = 16 * m + gID;
            const uint2 x = *reinterpret_cast<const uint2*>(blk + kKCodes + ta * 32 + 8 * tq);
            const uint2 y = *reinterpret_cast<const uint2*>(blk + kKCodes + (ta + 8) * 32 + 8 * tq);
            const uint32_t wa[2] = {x.x, x.y}, wb[2] = {y.x, y.y};
            const uint32_t wa8[2] = {code_swap(wa[0]), code_swap(wa[1])}, wb8[2] = {code_swap(wb[0]), code_swap(wb[1])};
            float acc[4][4];
#pragma unroll
            for (int g = 0; g < 4; ++g)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[g][e] = 0.f;
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int h = it >> 2, g = it & 3, ks = 2 * g + h;
                uint32_t a0, a1, a2, a3, c0 = 0, c1 = 0, c2 = 0, c3 = 0;
                switch (g) {
                    case 0:
                        k_operands<0>(wa[h], wb[h], wa8[h], wb8[h], a0, a1, a2, a3);
                        if (LM) high_planes<0>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                    case 1:
                        k_operands<1>(wa[h], wb[h], wa8[h], wb8[h], a0, a1, a2, a3);
                        if (LM) high_planes<1>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                    case 2:
                        k_operands<2>(wa[h], wb[h], wa8[h], wb8[h], a0, a1, a2, a3);
                        if (LM) high_planes<2>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                    default:
                        k_operands<3>(wa[h], wb[h], wa8[h], wb8[h], a0, a1, a2, a3);
                        if (LM) high_planes<3>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                }
                const uint2 qh = qfS[(0 * 8 + ks) * 32 + lane], ql = qfS[(1 * 8 + ks) * 32 + lane];
                mma_f16_16816(acc[g], a0, a1, a2, a3, qh.x, qh.y);
                mma_f16_16816(acc[g], a0, a1, a2, a3, ql.x, ql.y);
                if (LM) {  // high-bit plane against kappa q' (parts 2, 3: hi, lo)
                    const uint2 kh = qfS[(2 * 8 + ks) * 32 + lane], kl = qfS[(3 * 8 + ks) * 32 + lane];
                    mma_f16_16816(acc[g], c0, c1, c2, c3, kh.x, kh.y);
                    mma_f16_16816(acc[g], c0, c1, c2, c3, kl.x, kl.y);
                }
            }
            const float4 sA = ksS[ta], sB = ksS[ta + 8], zA = kzS[ta], zB = kzS[ta + 8];
            const float sa[4] = {sA.x, sA.y, sA.z, sA.w}, za[4] = {zA.x, zA.y, zA.z, zA.w};
            const float sb[4] = {sB.x, sB.y, sB.z, sB.w}, zb[4] = {zB.x, zB.y, zB.z, zB.w};
            const float q0[4] = {qsv[0].x, qsv[0].y, qsv[0].z, qsv[0].w};
            const float q1[4] = {qsv[1].x, qsv[1].y, qsv[1].z, qsv[1].w};
            float xa0 = 0.f, xa1 = 0.f, xb0 = 0.f, xb1 = 0.f;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                xa0 = fmaf(sa[g], acc[g][0], fmaf(za[g], q0[g], xa0));
                xa1 = fmaf(sa[g], acc[g][1], fmaf(za[g], q1[g], xa1));
                xb0 = fmaf(sb[g], acc[g][2], fmaf(zb[g], q0[g], xb0));
                xb1 = fmaf(sb[g], acc[g][3], fmaf(zb[g], q1[g], xb1));
            }
            const bool va = FULL || ta < valid, vb = FULL || ta + 8 < valid;
            lg[m][0] = va ? xa0 : -INFINITY;
            lg[m][1] = va ? xa1 : -INFINITY;
            lg[m][2] = vb ? xb0 : -INFINITY;
            lg[m][3] = vb ? xb1 : -INFINITY;
        }
    }

    // -- channel boost: as attend_page, for eight heads (q' of a position is
    //    two float4); corrections [64][8] in the P scratch
    if constexpr (BOOST) {
        float4* cS = reinterpret_cast<float4*>(pS);
        const int ng = 4 >> gshift;
#pragma unroll
        for (int tt = 0; tt < 2; ++tt) {
            const int t = 2 * lane + tt;
            const uint4 rr = tt ? br1 : br0;
            float4 c0 = make_float4(0.f, 0.f, 0.f, 0.f), c1 = c0;
            if (t < valid) {
                const uint32_t* szw = reinterpret_cast<const uint32_t*>(blk + kKScale + t * 4 * ng);
                const uint32_t wv[4] = {rr.x, rr.y, rr.z, rr.w};
#pragma unroll
                for (int e = 0; e < kBoostN; ++e) {
                    const uint32_t ent = wv[e >> 1] >> (16 * (e & 1));
                    const int pos = ent & 127;
                    const float sg = __half2float(__ushort_as_half((unsigned short)(szw[pos >> (5 + gshift)] & 0xffffu)));
                    const float d = sg * fmaf((float)((ent >> 8) & 15u), 0.2f, -(float)((ent >> 12) & 3u));
                    const float4 qa = qbS[2 * pos], qb = qbS[2 * pos + 1];
                    c0.x = fmaf(d, qa.x, c0.x);
                    c0.y = fmaf(d, qa.y, c0.y);
                    c0.z = fmaf(d, qa.z, c0.z);
                    c0.w = fmaf(d, qa.w, c0.w);
                    c1.x = fmaf(d, qb.x, c1.x);
                    c1.y = fmaf(d, qb.y, c1.y);
                    c1.z = fmaf(d, qb.z, c1.z);
                    c1.w = fmaf(d, qb.w, c1.w);
                }
            }
            cS[2 * t] = c0;
            cS[2 * t + 1] = c1;
        }
        __syncwarp();
        const float2* cf = reinterpret_cast<const float2*>(pS);  // [64][4] pairs: heads (2tq, 2tq + 1) at index tq
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int ta = 16 * m + gID;
            const float2 ca = cf[ta * 4 + tq], cb = cf[(ta + 8) * 4 + tq];
            lg[m][0] += ca.x;
            lg[m][1] += ca.y;
            lg[m][2] += cb.x;
            lg[m][3] += cb.y;
        }
        __syncwarp();
    }

    // -- online softmax per head (j: head 2tq + j)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        float mx = fmaxf(lg[0][j], lg[0][2 + j]);
#pragma unroll
        for (int m = 1; m < 4; ++m) mx = fmaxf(mx, fmaxf(lg[m][j], lg[m][2 + j]));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
        const float m_new = fmaxf(m_run[j], mx);
        if (__any_sync(kFull, m_new > m_run[j])) {
            const float alpha = (m_new > m_run[j]) ? ex2(m_run[j] - m_new) : 1.f;
            l_run[j] *= alpha;
#pragma unroll
            for (int g = 0; g < 4; ++g) zacc[j][g] *= alpha;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                acc_o[mt][j] *= alpha;
                acc_o[mt][2 + j] *= alpha;
            }
            m_run[j] = m_new;
        }
        const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int ta = 16 * m + gID;
            const float pa = ex2(lg[m][j] - m_sub), pb = ex2(lg[m][2 + j] - m_sub);
            if (FULL || m < ntile) {
                l_run[j] += pa + pb;
                const float4 vzA = vzS[ta], vzB = vzS[ta + 8];
                zacc[j][0] = fmaf(pa, vzA.x, fmaf(pb, vzB.x, zacc[j][0]));
                zacc[j][1] = fmaf(pa, vzA.y, fmaf(pb, vzB.y, zacc[j][1]));
                zacc[j][2] = fmaf(pa, vzA.z, fmaf(pb, vzB.z, zacc[j][2]));
                zacc[j][3] = fmaf(pa, vzA.w, fmaf(pb, vzB.w, zacc[j][3]));
            }
            pS[(2 * tq + j) * kPvRow + pv_pos(ta)] = pa;
            pS[(2 * tq + j) * kPvRow + pv_pos(ta + 8)] = pb;
        }
    }
    __syncwarp();

    // -- values: as attend_page, with B column gID = head gID (hi, then lo)
    uint4 pv4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        pv4[k] = *reinterpret_cast<const uint4*>(blk + kVCodes + (gID + 8 * k) * kPage + 16 * tq);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int chunk = 4 * (4 * tq + (m ^ tq));
        const float4 pp = *reinterpret_cast<const float4*>(pS + gID * kPvRow + chunk);
        uint32_t pw[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) pw[k] = m == 0 ? pv4[k].x : m == 1 ? pv4[k].y : m == 2 ? pv4[k].z : pv4[k].w;
        const uint32_t pw8[4] = {code_swap(pw[0]), code_swap(pw[1]), code_swap(pw[2]), code_swap(pw[3])};
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const float4 sg = *reinterpret_cast<const float4*>(vsS + g * kPvRow + chunk);
            uint32_t bh0, bl0, bh1, bl1, ch0 = 0, cl0 = 0, ch1 = 0, cl1 = 0;
            const float2 w0 = mul2(make_float2(pp.x, pp.y), make_float2(sg.x, sg.y));
            const float2 w1 = mul2(make_float2(pp.z, pp.w), make_float2(sg.z, sg.w));
            split_both(w0, bh0, bl0);
            split_both(w1, bh1, bl1);
            if constexpr (LM) {  // the high-bit plane's weights kappa * W
                const float2 kv2 = make_float2(cbk.vk, cbk.vk);
                split_both(mul2(w0, kv2), ch0, cl0);
                split_both(mul2(w1, kv2), ch1, cl1);
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const uint32_t r0 = pw[2 * half], r1 = pw[2 * half + 1];
                const uint32_t r08 = pw8[2 * half], r18 = pw8[2 * half + 1];
                uint32_t a0, a1, a2, a3, c0 = 0, c1 = 0, c2 = 0, c3 = 0;
                switch (g) {
                    case 0:
                        v_operands<0>(r0, r1, r08, r18, a0, a1, a2, a3);
                        if (LM) high_planes<0>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                    case 1:
                        v_operands<1>(r0, r1, r08, r18, a0, a1, a2, a3);
                        if (LM) high_planes<1>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                    case 2:
                        v_operands<2>(r0, r1, r08, r18, a0, a1, a2, a3);
                        if (LM) high_planes<2>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                    default:
                        v_operands<3>(r0, r1, r08, r18, a0, a1, a2, a3);
                        if (LM) high_planes<3>(a0, a1, a2, a3, c0, c1, c2, c3);
                        break;
                }
                mma_f16_16816(acc_o[2 * g + half], a0, a1, a2, a3, bh0, bh1);
                mma_f16_16816(acc_o[2 * g + half], a0, a1, a2, a3, bl0, bl1);
                if (LM) {
                    mma_f16_16816(acc_o[2 * g + half], c0, c1, c2, c3, ch0, ch1);
                    mma_f16_16816(acc_o[2 * g + half], c0, c1, c2, c3, cl0, cl1);
                }
            }
        }
    }
}

template <int NT, bool LM = false, bool BOOST = false>
__global__ void __launch_bounds__(kInt2Threads, (int2_blocks_per_sm<NT, LM, BOOST>())) int2_kernel(DecodeParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int NS = int2_stages<NT, LM, BOOST>();  // ring stages
    using SM = Int2Smem<NT, NS>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t* stages = smem + SM::kStage;
    StageInfo* info = reinterpret_cast<StageInfo*>(smem + SM::kInfo);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kBars);
    uint64_t* empty = full + NS;
    uint64_t* merge_bar = empty + NS;  // consumer-warp rendezvous at item ends
    constexpr bool QP = int2_q_prefetch<NT, LM, BOOST>();
    uint64_t* qfull = reinterpret_cast<uint64_t*>(smem + SM::kQbBars);  // QP only: item buffers' barriers
    uint64_t* qempty = qfull + 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(merge_bar, kConsumerWarps);
        if constexpr (QP) {
            for (int s = 0; s < 2; ++s) {
                mbar_init(&qfull[s], 1);
                mbar_init(&qempty[s], kConsumerWarps);
            }
        }
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();     // q' fragments, plan and counter come from prep_kernel
    pdl_trigger();  // the BF16 segment kernel may take SMs as this grid retires

    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        const int total_long = __ldg(p.item_start + p.B);
        const int total = total_long + __ldg(p.item_start2 + p.B);
        uint32_t n = 0;      // slots issued so far (stage n % NS, warp n % 4)
        uint32_t pitem = 0;  // items started (QP: item k's q' data goes to buffer k % 2)
        bool ok = true;
        // one slot: wait for the stage, then publish its info (and copy)
        auto post = [&](int item, int b, int kv, int pid, int valid, int flags) -> bool {
            const uint32_t s = n % NS;
            if (n >= (uint32_t)NS) {
                const bool w = mbar_wait_bounded(&empty[s], ((n / NS) - 1) & 1u, kWaitPolls);
                if (!__all_sync(kFull, w)) return false;
            }
            if (lane == 0) {
                StageInfo& si = info[s];
                si.item = item;
                si.b = b;
                si.kv = kv;
                if (item >= 0 && !(flags & kFlagPad) && (pid < 0 || pid >= p.num_pages)) {
                    report(p.status, OSCAR_STATUS_BAD_PAGE);
                    flags |= kFlagPad;
                }
                si.valid_flags = valid | (flags << 8);
                si.pid = pid;
                if (item < 0 || (flags & kFlagPad)) {
                    mbar_arrive(&full[s]);
                } else {
                    mbar_arrive_expect_tx(&full[s], p.block_bytes);
                    bulk_g2s(stages + s * kBlock, p.pool + ((size_t)pid * p.hk + kv) * p.block_bytes,
                             p.block_bytes, &full[s]);
                    // the consumer loads the page's boost records itself: have them in L2
                    if constexpr (BOOST) bulk_prefetch_l2(p.boost + ((size_t)pid * p.hk + kv) * kBoostBlock, kBoostBlock);
                }
            }
            __syncwarp();
            ++n;
            return true;
        };
        for (;;) {
            int item = 0;
            if (lane == 0) item = atomicAdd(p.counter, 1);
            item = __shfl_sync(kFull, item, 0);
            if (item >= total) {  // one end marker per consumer warp
                for (int i = 0; i < kConsumerWarps && ok; ++i) ok = post(-1, 0, 0, 0, 0, 0);
                break;
            }
            const bool is_long = item < total_long;
            const int32_t* starts = is_long ? p.item_start : p.item_start2;
            const int rel = is_long ? item : item - total_long;
            const int b = find_seq(starts, p.B, rel);
            const int s0 = __ldg(starts + b);
            const int splits = (__ldg(starts + b + 1) - s0) / p.hk;
            const int kv = (rel - s0) / splits;
            const int split = (rel - s0) % splits;
            const int hist = min(max(__ldg(p.hist_len + b), 0), p.max_pages * kPage);
            const int seq_pages = (hist + kPage - 1) / kPage;
            const SeqSplits sp = seq_splits(seq_pages, p.pps, p.tail_pg);
            const int pg0 = is_long ? split * p.pps : sp.long_pages + split * kShortItemPages;
            const int npg = is_long ? min(p.pps, sp.long_pages - pg0) : min(kShortItemPages, seq_pages - pg0);
            const int nslots = (npg + kConsumerWarps - 1) / kConsumerWarps * kConsumerWarps;
            if constexpr (QP) {  // the item's q' data into its buffer, once item k - 2 has left it
                const uint32_t qs = pitem & 1u;
                if (pitem >= 2) {
                    const bool w = mbar_wait_bounded(&qempty[qs], ((pitem >> 1) - 1) & 1u, kWaitPolls);
                    if (!__all_sync(kFull, w)) {
                        ok = false;
                        break;
                    }
                }
                if (lane == 0) {
                    const size_t bk = (size_t)b * p.hk + kv;
                    uint8_t* qb = smem + SM::kQb + qs * SM::kQbBytes;
                    mbar_arrive_expect_tx(&qfull[qs], SM::kQbBytes);
                    bulk_g2s(qb + SM::kQbFrag, p.qfrag + bk * 8 * 32 * 2, 8 * 32 * 8, &qfull[qs]);
                    bulk_g2s(qb + SM::kQbSum, p.qsum + bk * 4 * 4, 4 * 16, &qfull[qs]);
                    bulk_g2s(qb + SM::kQbKinv, p.qkinv + bk * 4, 16, &qfull[qs]);
                }
                __syncwarp();
                ++pitem;
            }
            for (int c = 0; c < nslots && ok; c += 32) {
                // page ids of the next 32 slots, one per lane
                int pid = -1;
                if (c + lane < npg) pid = __ldg(p.page_table + (size_t)b * p.max_pages + pg0 + c + lane);
                const int cnt = min(32, nslots - c);
                for (int i = 0; i < cnt && ok; ++i) {
                    const int pl = c + i;
                    const int pi = __shfl_sync(kFull, pid, i);
                    const int flags = (pl < kConsumerWarps ? kFlagFirst : 0) |
                                      (pl >= nslots - kConsumerWarps ? kFlagLast : 0) | (pl >= npg ? kFlagPad : 0);
                    const int valid = pl < npg ? min(kPage, hist - (pg0 + pl) * kPage) : 0;
                    ok = post(item, b, kv, pi, valid, flags);
                }
            }
            if (!ok) break;
        }
        if (!ok) {
            if (lane == 0) report(p.status, OSCAR_STATUS_TIMEOUT);
            // let issued copies land before the block can exit
            const uint32_t first = n > (uint32_t)NS ? n - NS : 0;
            for (uint32_t k = first; k < n; ++k)
                (void)mbar_wait_bounded(&full[k % NS], (k / NS) & 1u, kWaitPolls);
            if constexpr (QP)
                for (uint32_t k = pitem > 2 ? pitem - 2 : 0; k < pitem; ++k)
                    (void)mbar_wait_bounded(&qfull[k & 1u], (k >> 1) & 1u, kWaitPolls);
        }
        return;
    }

    // ------------------------------- consumers ---------------------------------
    const int gID = lane >> 2, tq = lane & 3;
    uint8_t* wbuf = smem + SM::kWarp + warp * SM::kWarpBytes;
    const SplitSel take_lo = split_sel(gID & 1);  // PV column: hi / lo

    uint32_t merge_phase = 0;
    // bounded rendezvous of the four consumer warps (an mbarrier, so that a
    // warp that gave up on a page cannot leave the others waiting forever)
    auto consumer_sync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(merge_bar);
        const bool w = mbar_wait_bounded(merge_bar, merge_phase & 1u, kWaitPolls);
        ++merge_phase;
        return __all_sync(kFull, w);
    };

    uint2* qfS = reinterpret_cast<uint2*>(smem + SM::kQf);
    float4* qbS = reinterpret_cast<float4*>(smem + SM::kQf + NT * 8 * 32 * 8);  // boost: q' of the four heads
    float4 qsv[NT];
    float kq = 1.f;  // the item's 2^-e (prep's power of two of q'), folded into the K scales
    uint32_t citem = 0, cur_qs = 0;  // QP: items started by this warp, the current item's buffer
    const uint2* qcur = qfS;         // the current item's q' fragments
    float m_run[NT], l_run[NT], zacc[NT][4], acc_o[NT][8][4];
    Codebook cbk{1.f, 1.f, 0.f, 0.f};  // Lloyd-Max levels of the current item's KV head

    for (uint32_t n = warp;; n += kConsumerWarps) {
        const uint32_t s = n % NS;
        const bool w = mbar_wait_bounded(&full[s], (n / NS) & 1u, kWaitPolls);
        if (!__all_sync(kFull, w)) {
            if (lane == 0) report(p.status, OSCAR_STATUS_TIMEOUT);
            return;
        }
        const int4 sraw = *reinterpret_cast<const int4*>(&info[s]);
        if (sraw.x < 0) break;
        const int item = sraw.x, flags = sraw.w >> 8, valid = sraw.w & 0xff;
        const uint8_t* blk = stages + s * kBlock;

        if (QP && (flags & kFlagFirst)) {  // the producer prefetched the item's q' data
            cur_qs = citem & 1u;
            const bool wq = mbar_wait_bounded(&qfull[cur_qs], (citem >> 1) & 1u, kWaitPolls);
            if (!__all_sync(kFull, wq)) {
                if (lane == 0) report(p.status, OSCAR_STATUS_TIMEOUT);
                return;
            }
            ++citem;
            const uint8_t* qb = smem + SM::kQb + cur_qs * SM::kQbBytes;
            qcur = reinterpret_cast<const uint2*>(qb + SM::kQbFrag);
            kq = *reinterpret_cast<const float*>(qb + SM::kQbKinv);
            qsv[0] = reinterpret_cast<const float4*>(qb + SM::kQbSum)[tq];
            m_run[0] = -INFINITY;
            l_run[0] = 0.f;
#pragma unroll
            for (int g = 0; g < 4; ++g) zacc[0][g] = 0.f;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc_o[0][mt][e] = 0.f;
        } else if (flags & kFlagFirst) {
            const int bk = sraw.y * p.hk + sraw.z;
            if (LM) cbk = codebook_of(p.codebook, sraw.z);
            kq = p.qkinv[(size_t)bk * 4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint32_t* fr = p.qfrag + ((size_t)bk * NT + nt) * 8 * 32 * 2;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {  // every warp writes the same values
                    const uint2 f = *reinterpret_cast<const uint2*>(fr + ((size_t)ks * 32 + lane) * 2);
                    qfS[(nt * 8 + ks) * 32 + lane] = f;
                    if (LM && NT == 1) qfS[((NT + nt) * 8 + ks) * 32 + lane] = scaled_fragment(f, cbk.kk, (lane >> 2) & 1);
                }
                if constexpr (LM && NT == 2) {  // eight heads: parts 0, 1 are q' hi, lo; kappa q' into parts 2, 3
                    if (nt == 1) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint2 hh = qfS[(0 * 8 + ks) * 32 + lane], ll = qfS[(1 * 8 + ks) * 32 + lane];
                            const float y[4] = {cbk.kk * (half_lo(hh.x) + half_lo(ll.x)),
                                                cbk.kk * (half_hi(hh.x) + half_hi(ll.x)),
                                                cbk.kk * (half_lo(hh.y) + half_lo(ll.y)),
                                                cbk.kk * (half_hi(hh.y) + half_hi(ll.y))};
                            uint32_t h01, h23, l01, l23;
                            split_f16(y, h01, h23, l01, l23);
                            qfS[(2 * 8 + ks) * 32 + lane] = make_uint2(h01, h23);
                            qfS[(3 * 8 + ks) * 32 + lane] = make_uint2(l01, l23);
                        }
                    }
                }
                if constexpr (BOOST) {  // q'[j] of heads 4nt..4nt+3 as float4 NT * j + nt
                    const float* qr = p.qrot + ((size_t)bk * NT + nt) * 4 * kD + 4 * lane;
                    const float4 a0 = *reinterpret_cast<const float4*>(qr), a1 = *reinterpret_cast<const float4*>(qr + kD);
                    const float4 a2 = *reinterpret_cast<const float4*>(qr + 2 * kD);
                    const float4 a3 = *reinterpret_cast<const float4*>(qr + 3 * kD);
                    qbS[NT * (4 * lane + 0) + nt] = make_float4(a0.x, a1.x, a2.x, a3.x);
                    qbS[NT * (4 * lane + 1) + nt] = make_float4(a0.y, a1.y, a2.y, a3.y);
                    qbS[NT * (4 * lane + 2) + nt] = make_float4(a0.z, a1.z, a2.z, a3.z);
                    qbS[NT * (4 * lane + 3) + nt] = make_float4(a0.w, a1.w, a2.w, a3.w);
                }
                // head of the lane's column: 4nt + tq (up to four heads), 2tq + nt (eight)
                const int hq = (NT == 2) ? 2 * tq + nt : 4 * nt + tq;
                qsv[nt] = *reinterpret_cast<const float4*>(p.qsum + ((size_t)bk * NT * 4 + hq) * 4);
                m_run[nt] = -INFINITY;
                l_run[nt] = 0.f;
#pragma unroll
                for (int g = 0; g < 4; ++g) zacc[nt][g] = 0.f;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc_o[nt][mt][e] = 0.f;
            }
        }

        if (!(flags & kFlagPad)) {
            const uint8_t* brec = nullptr;
            if constexpr (BOOST) brec = p.boost + ((size_t)info[s].pid * p.hk + sraw.z) * kBoostBlock;
            if constexpr (NT == 2) {
                if (valid == kPage)
                    attend_page_g8<true, BOOST, LM>(blk, valid, wbuf, qfS, qsv, kq, m_run, l_run, zacc, acc_o[0],
                                                    p.gshift, qbS, brec, cbk);
                else
                    attend_page_g8<false, BOOST, LM>(blk, valid, wbuf, qfS, qsv, kq, m_run, l_run, zacc, acc_o[0],
                                                     p.gshift, qbS, brec, cbk);
            } else {
                if (valid == kPage)
                    attend_page<NT, true, LM, BOOST>(blk, valid, wbuf, qcur, qsv, kq, m_run, l_run, zacc, acc_o,
                                                     take_lo, p.gshift, cbk, qbS, brec);
                else
                    attend_page<NT, false, LM, BOOST>(blk, valid, wbuf, qcur, qsv, kq, m_run, l_run, zacc, acc_o,
                                                      take_lo, p.gshift, cbk, qbS, brec);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (QP && (flags & kFlagLast) && lane == 0) mbar_arrive(&qempty[cur_qs]);  // done with the item's q' data

        if (flags & kFlagLast) {
            // this warp's partial state -> its scratch (no longer needed)
            float* mw = reinterpret_cast<float*>(wbuf);
            // P.V accumulator scales of the four slots (see v_out_scale)
            constexpr float kLmUp = LM ? 1.f / kLmVDown : 1.f;
            const float vout[4] = {v_out_scale(0) * kLmUp, v_out_scale(1) * kLmUp, v_out_scale(2) * kLmUp,
                                   v_out_scale(3) * kLmUp};
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float l = l_run[nt];
                l += __shfl_xor_sync(kFull, l, 4);
                l += __shfl_xor_sync(kFull, l, 8);
                l += __shfl_xor_sync(kFull, l, 16);
                float z[4];
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    z[g] = zacc[nt][g];
                    z[g] += __shfl_xor_sync(kFull, z[g], 4);
                    z[g] += __shfl_xor_sync(kFull, z[g], 8);
                    z[g] += __shfl_xor_sync(kFull, z[g], 16);
                }
                if constexpr (NT == 2) {  // column = head 2tq + nt (hi and lo summed by the MMA)
                    float* o = mw + (size_t)(2 * tq + nt) * (kD + 2);
#pragma unroll
                    for (int g = 0; g < 4; ++g)
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            o[32 * g + 16 * half + gID] = fmaf(acc_o[0][2 * g + half][nt], vout[g], z[g]);
                            o[32 * g + 16 * half + 8 + gID] = fmaf(acc_o[0][2 * g + half][2 + nt], vout[g], z[g]);
                        }
                    if (gID == 0) {
                        o[kD] = m_run[nt];
                        o[kD + 1] = l;
                    }
                    continue;
                }
                float* o = mw + (size_t)(4 * nt + tq) * (kD + 2);
#pragma unroll
                for (int g = 0; g < 4; ++g)
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        o[32 * g + 16 * half + gID] =
                            fmaf(acc_o[nt][2 * g + half][0] + acc_o[nt][2 * g + half][1], vout[g], z[g]);
                        o[32 * g + 16 * half + 8 + gID] =
                            fmaf(acc_o[nt][2 * g + half][2] + acc_o[nt][2 * g + half][3], vout[g], z[g]);
                    }
                if (gID == 0) {
                    o[kD] = m_run[nt];
                    o[kD + 1] = l;
                }
            }
            if (!consumer_sync()) {
                if (lane == 0) report(p.status, OSCAR_STATUS_TIMEOUT);
                return;
            }
            // merge the four warps: thread -> dimension, all heads
            float* part = p.part + (size_t)item * p.part_stride;
            const int d = threadIdx.x;  // 0..127
            for (int hl = 0; hl < p.G; ++hl) {
                float M = -INFINITY;
#pragma unroll
                for (int ww = 0; ww < kConsumerWarps; ++ww)
                    M = fmaxf(M, reinterpret_cast<const float*>(smem + SM::kWarp + ww * SM::kWarpBytes)[hl * (kD + 2) + kD]);
                float acc = 0.f, L = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int ww = 0; ww < kConsumerWarps; ++ww) {
                        const float* src =
                            reinterpret_cast<const float*>(smem + SM::kWarp + ww * SM::kWarpBytes) + hl * (kD + 2);
                        const float sc = ex2(src[kD] - M);
                        acc = fmaf(sc, src[d], acc);
                        L = fmaf(sc, src[kD + 1], L);
                    }
                }
                part[(size_t)hl * kD + d] = acc;
                if (d == 0) {
                    part[(size_t)p.G * kD + hl] = M;
                    part[(size_t)p.G * kD + p.G + hl] = L;
                }
            }
            if (!consumer_sync()) {
                if (lane == 0) report(p.status, OSCAR_STATUS_TIMEOUT);
                return;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// BF16 sink + recent segment
// ---------------------------------------------------------------------------
// Block (item, (b, kv)) covers 64 consecutive slots of the 320-token BF16
// segment; warp w attends over 16 of them on tensor cores, FlashAttention
// style with the query heads as MMA rows: S = Q.K^T with A = the query rows
// (row 2h and 2h+1 both hold head h; K and q are bf16, so the products are
// exact), then O = P.V with A = P taken straight from S's accumulator layout
// (row 2h carries the bf16 high part of p, row 2h+1 the rounded remainder, so
// P keeps ~16 bits) and B = V via ldmatrix.trans.  The four warps' partial
// states are merged in shared memory into one partial per block.
constexpr int kBfWarps = 4;
constexpr int kBfThreads = 32 * kBfWarps;
constexpr int kBfItemTok = 16 * kBfWarps;          // tokens per block
constexpr int kBfPitch = 528;                      // bytes per staged token row (512 + 16)
constexpr int kBfWarpBytes = 16 * kBfPitch;        // also holds the warp's state [G][kD + 2] at the end
constexpr int kBfQBytes = 8 * kD * 2;                 // query rows of one KV group (up to 8 heads)
constexpr int kBfSmem = 2 * kBfWarps * kBfWarpBytes + 2 * kBfQBytes;  // two buffers
static_assert(8 * (kD + 2) * 4 <= kBfWarpBytes, "warp state must fit in the warp's row tile");

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

// Copy one 16-token tile of (b, kv)'s BF16 rows (K | V, 512 B each) into
// rows with cp.async and zero the rows past the valid tokens; the caller
// commits the group.
__device__ __forceinline__ void bf16_stage_rows(const DecodeParams& p, int b, int kv, int t0, int nvalid,
                                                uint8_t* rows) {
    if (nvalid <= 0) return;
    const int lane = threadIdx.x & 31;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(p.bf16_kv) +
                         (((size_t)b * p.nslot + t0) * p.hk + kv) * (2 * kD * 2);
    const size_t row_stride = (size_t)p.hk * 2 * kD * 2;
#pragma unroll 4
    for (int r = 0; r < 16; ++r) {
        if (r < nvalid) cp_async16(rows + r * kBfPitch + 16 * lane, src + r * row_stride + 16 * lane);
        else *reinterpret_cast<uint4*>(rows + r * kBfPitch + 16 * lane) = make_uint4(0u, 0u, 0u, 0u);
    }
}

// One warp's 16-token tile from staged rows and the staged query rows of
// its KV group (qsm: [G][kD] bf16); leaves the warp's state (o, m, l) per
// head in rows.  MMA row h holds head h (rows G..15 are zero): S = Q.K^T,
// then O += P.V twice into the same accumulators, with A = the bf16 high
// part of P (its low 16 bits cleared, exact) and A = the rounded remainder,
// so P keeps ~16 bits and each head's output is one accumulator row.
template <int G>
__device__ void bf16_tile(int nvalid, uint8_t* rows, const __nv_bfloat16* qsm, float qscale) {
    const int lane = threadIdx.x & 31, gID = lane >> 2, tq = lane & 3;
    float* st = reinterpret_cast<float*>(rows);  // [G][kD + 2] at the end
    if (nvalid <= 0) {
        for (int i = lane; i < G * (kD + 2); i += 32) {
            const int c = i % (kD + 2);
            st[i] = (c == kD) ? -INFINITY : 0.f;
        }
        return;
    }
    const bool row_on = gID < G;
    const __nv_bfloat16* qa = qsm + (row_on ? gID : 0) * kD;
    uint32_t qf[8][2];  // A fragments (rows gID: a0, a2; rows gID + 8 are zero)
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        const int d0 = 16 * ks + 2 * tq;
        qf[ks][0] = row_on ? *reinterpret_cast<const uint32_t*>(qa + d0) : 0u;
        qf[ks][1] = row_on ? *reinterpret_cast<const uint32_t*>(qa + d0 + 8) : 0u;
    }

    // S = Q.K^T for tokens 8nt .. 8nt+7 (B via ldmatrix: matrix i/8 = dims
    // 16ks + 8(i/8) of token row i%8, covering k-steps ks and ks+1)
    float sacc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
        const uint8_t* rb = rows + (8 * nt + (lane & 7)) * kBfPitch + 16 * (lane >> 3);
#pragma unroll
        for (int ks = 0; ks < 8; ks += 2) {
            uint32_t kb[4];
            ldsm_x4(kb, rb + 32 * ks);
            mma_bf16_16816(sacc[nt], qf[ks][0], 0u, qf[ks][1], 0u, kb[0], kb[1]);
            mma_bf16_16816(sacc[nt], qf[ks + 1][0], 0u, qf[ks + 1][1], 0u, kb[2], kb[3]);
        }
    }
    // scale to base 2, mask, row max / exp / sum (row gID: e 0, 1)
    float ma = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int tok = 8 * nt + 2 * tq + e;
            sacc[nt][e] = (tok < nvalid) ? sacc[nt][e] * qscale : -INFINITY;
            ma = fmaxf(ma, sacc[nt][e]);
        }
    ma = fmaxf(ma, __shfl_xor_sync(kFull, ma, 1));
    ma = fmaxf(ma, __shfl_xor_sync(kFull, ma, 2));
    float la = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            sacc[nt][e] = ex2(sacc[nt][e] - ma);
            la += sacc[nt][e];
        }
    la += __shfl_xor_sync(kFull, la, 1);
    la += __shfl_xor_sync(kFull, la, 2);

    // P as the A operand of O = P.V (k = the 16 tokens), high and low parts
    uint32_t ph[2], pl[2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const float w0 = sacc[nt][0], w1 = sacc[nt][1];
        const float h0 = __uint_as_float(__float_as_uint(w0) & 0xffff0000u);
        const float h1 = __uint_as_float(__float_as_uint(w1) & 0xffff0000u);
        ph[nt] = row_on ? pack_bf16x2_rn(h0, h1) : 0u;
        pl[nt] = row_on ? pack_bf16x2_rn(w0 - h0, w1 - h1) : 0u;
    }

    // O = P.V over dims 8j .. 8j+7 (B via ldmatrix.trans: matrix i/8 = tokens
    // 8((i/8)&1) + i%8, dims 16jp + 8(i/16))
    float o[16][4];
    const uint8_t* vb = rows + 256 + ((lane & 7) + 8 * ((lane >> 3) & 1)) * kBfPitch + 16 * (lane >> 4);
#pragma unroll
    for (int jp = 0; jp < 8; ++jp) {
        uint32_t vf[4];
        ldsm_x4_trans(vf, vb + 32 * jp);
#pragma unroll
        for (int e = 0; e < 4; ++e) o[2 * jp][e] = o[2 * jp + 1][e] = 0.f;
        mma_bf16_16816(o[2 * jp], ph[0], 0u, ph[1], 0u, vf[0], vf[1]);
        mma_bf16_16816(o[2 * jp], pl[0], 0u, pl[1], 0u, vf[0], vf[1]);
        mma_bf16_16816(o[2 * jp + 1], ph[0], 0u, ph[1], 0u, vf[2], vf[3]);
        mma_bf16_16816(o[2 * jp + 1], pl[0], 0u, pl[1], 0u, vf[2], vf[3]);
    }
    __syncwarp();  // all row reads done: the tile now holds the warp's state
    if (row_on) {  // head gID: accumulator row gID
#pragma unroll
        for (int j = 0; j < 16; ++j)
            *reinterpret_cast<float2*>(st + gID * (kD + 2) + 8 * j + 2 * tq) = make_float2(o[j][0], o[j][1]);
        if (tq == 0) {
            st[gID * (kD + 2) + kD] = ma;
            st[gID * (kD + 2) + kD + 1] = la;
        }
    }
}

// Persistent: 3 blocks per SM loop over the (sequence, KV head, 64-slot
// block) items with two buffers per warp, so that the next item's rows (and
// its query rows, staged by warp 0) are in flight while the current item is
// attended.  Launched as a programmatic dependent of int2_kernel, whose
// results it does not read; its block 0 waits for int2_kernel's completion
// before it exits (the others leave when their items are done), so this grid
// completes after int2_kernel and the merge after it sees both.
__global__ void __launch_bounds__(kBfThreads, 3) bf16_kernel(DecodeParams p) {
    extern __shared__ __align__(128) uint8_t bsm[];
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = p.bf_items * p.B * p.hk;
    auto rows_of = [&](int buf, int w) { return bsm + (buf * kBfWarps + w) * kBfWarpBytes; };
    auto q_of = [&](int buf) { return bsm + 2 * kBfWarps * kBfWarpBytes + buf * kBfQBytes; };
    auto stage = [&](int it, int buf) {
        if (it < total) {
            const int bk = it / p.bf_items, item = it % p.bf_items;
            const int b = bk / p.hk, kv = bk % p.hk;
            const int n = min(max(__ldg(p.bf16_len + b), 0), p.nslot);
            const int t0 = item * kBfItemTok + 16 * warp;
            bf16_stage_rows(p, b, kv, t0, n - t0, rows_of(buf, warp));
            if (warp == 0) {  // the KV group's query rows (the query is only 8-byte aligned)
                const uint8_t* qsrc = reinterpret_cast<const uint8_t*>(p.q + ((size_t)b * p.hq + kv * p.G) * kD);
                uint8_t* qdst = q_of(buf);
                for (int c = lane; c < p.G * (kD * 2 / 8); c += 32)
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(qdst + 8 * c)),
                                 "l"(qsrc + 8 * c)
                                 : "memory");
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    // Block i takes item i first; the items after the first gridDim.x come
    // from a work counter (blocks start as the INT2 grid retires, so a fixed
    // stride would leave the late ones the same share).  s_it[buf] is the
    // item staged into buffer buf next, each claimed an item ahead so that the
    // atomic's latency hides behind an item's work.
    __shared__ int s_it[2];
    int32_t* ctr = p.counter + kBfCounter;
    int pend = 0;  // thread 0: the item after the next one
    if (threadIdx.x == 0) {
        s_it[0] = blockIdx.x;
        s_it[1] = gridDim.x + atomicAdd(ctr, 1);
        pend = gridDim.x + atomicAdd(ctr, 1);
    }
    __syncthreads();
    int buf = 0;
    int it = s_it[0];
    stage(it, 0);
    for (; it < total; buf ^= 1) {
        const int nxt = s_it[buf ^ 1];
        stage(nxt, buf ^ 1);
        asm volatile("cp.async.wait_group 1;" ::: "memory");
        __syncthreads();  // this item's rows and query rows have landed
        const int bk = it / p.bf_items, item = it % p.bf_items;
        const int b = bk / p.hk;
        const int n = min(max(__ldg(p.bf16_len + b), 0), p.nslot);
        const int t0 = item * kBfItemTok + 16 * warp;
        uint8_t* rows = rows_of(buf, warp);
        const __nv_bfloat16* qsm = reinterpret_cast<const __nv_bfloat16*>(q_of(buf));
        switch (p.G) {
            case 1: bf16_tile<1>(n - t0, rows, qsm, p.qscale); break;
            case 2: bf16_tile<2>(n - t0, rows, qsm, p.qscale); break;
            case 4: bf16_tile<4>(n - t0, rows, qsm, p.qscale); break;
            default: bf16_tile<8>(n - t0, rows, qsm, p.qscale); break;
        }
        __syncthreads();
        // merge the four warps: thread -> dimension
        float* part = p.bf_part + ((size_t)bk * p.bf_items + item) * p.part_stride;
        const int d = threadIdx.x;
        for (int h = 0; h < p.G; ++h) {
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kBfWarps; ++w)
                M = fmaxf(M, reinterpret_cast<const float*>(rows_of(buf, w))[h * (kD + 2) + kD]);
            float acc = 0.f, L = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kBfWarps; ++w) {
                    const float* src = reinterpret_cast<const float*>(rows_of(buf, w)) + h * (kD + 2);
                    const float sc = ex2(src[kD] - M);
                    acc = fmaf(sc, src[d], acc);
                    L = fmaf(sc, src[kD + 1], L);
                }
            }
            part[(size_t)h * kD + d] = acc;
            if (d == 0) {
                part[(size_t)p.G * kD + h] = M;
                part[(size_t)p.G * kD + p.G + h] = L;
            }
        }
        if (threadIdx.x == 0) {  // the item staged into this buffer after nxt
            s_it[buf] = pend;
            pend = gridDim.x + atomicAdd(ctr, 1);
        }
        __syncthreads();  // states read before this buffer is refilled; s_it[buf] visible
        it = nxt;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    if (blockIdx.x == 0 && threadIdx.x == 0) pdl_wait();  // this grid completes after int2_kernel
}

// ---------------------------------------------------------------------------
// merge: INT2 splits -> un-rotate -> merge with the BF16 partial
// ---------------------------------------------------------------------------
// Block = 8 warps, block y = KV head.  Each output row (b, head) is served by
// p.merge_wpr warps (1, 2, 4 or 8: more when rows are few and splits many,
// e.g. one long sequence): the row's split-K partials are dealt round-robin
// to its warps, each warp merges its share (log-sum-exp in base 2), and the
// row's first warp combines the shares.  U_V is copied row-major into shared
// memory with cp.async meanwhile (rows padded to kURow floats).  The
// un-rotation o = w . U_V^T of the block's rows (at most eight) runs on
// tensor cores, shared by the eight warps: warp w computes outputs
// 16w .. 16w+15 of every row as D(16 x 8) += W(16 x 16) . U_V^T(16 x 8)
// over the 128 inputs, rows 8-15 of W zero, W and U_V each split into fp16
// high and rounded-remainder parts (22 significant bits) and the three
// products hi.hi + hi.lo + lo.hi accumulated in fp32 (the lo.lo term is
// below 2^-22 of the product).  U_V is read once per block instead of once
// per row.
constexpr int kMergeWarps = 8;
constexpr int kMergeThreads = 32 * kMergeWarps;
constexpr int kMergeRow = kD + 4;  // floats per warp row (y[128], M, L; a multiple of 4 for float4 access)
constexpr int kURow = kD + 8;      // floats per staged U_V row: fragment loads of 8 rows hit distinct banks
constexpr int kMergeSmem = (kD * kURow + 2 * kMergeWarps * kMergeRow) * 4;
constexpr int kMergeBatch = 12;   // split-K partials per batch of loads
constexpr int kMaxBfItems = 5;    // BF16 segment blocks per row: ceil(320 / 64)

__global__ void __launch_bounds__(kMergeThreads, 2) merge_kernel(DecodeParams p) {
    extern __shared__ __align__(16) float msm[];
    float* Us = msm;                  // [a][kURow] = U_V[a][j]
    float* Ws = msm + kD * kURow;     // [warp][kMergeRow]: a warp's share (y, M, L), then the row's w
    float* Ys = Ws + kMergeWarps * kMergeRow;  // [row][kMergeRow]: the block's un-rotated rows
    const int kv = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.U + ((size_t)kv * 2 + 1) * kD * kD);
        uint8_t* dst = reinterpret_cast<uint8_t*>(Us);
        for (int i = threadIdx.x; i < kD * kD / 4; i += kMergeThreads)  // 16-byte chunk i: row i / 32, chunk i % 32
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst + (i >> 5) * kURow * 4 + 16 * (i & 31))),
                         "l"(src + 16 * i)
                         : "memory");
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    const int wpr = p.merge_wpr, rpb = kMergeWarps / wpr;
    const int r = blockIdx.x * rpb + warp / wpr, sub = warp % wpr;
    const bool active = r < p.B * p.G;
    const int b = active ? r / p.G : 0, hh = active ? r % p.G : 0;
    // the (sequence, KV head)'s partials: n_long long items, then n_short
    // short ones.  The plan comes from prep_kernel, which completed before
    // int2_kernel passed its wait, i.e. before this grid could start: read it
    // before the wait, so that only the partials' loads follow it.
    int splits = 0, first = 0, first2 = 0, n_long = 0;
    if (active) {
        const int s0 = __ldg(p.item_start + b), t0 = __ldg(p.item_start2 + b);
        n_long = (__ldg(p.item_start + b + 1) - s0) / p.hk;
        const int n_short = (__ldg(p.item_start2 + b + 1) - t0) / p.hk;
        splits = n_long + n_short;
        first = s0 + kv * n_long;
        first2 = __ldg(p.item_start + p.B) + t0 + kv * n_short - n_long;
    }
    pdl_wait();  // partials of int2_kernel and bf16_kernel
    const int r5 = bitrev5(lane);
    // lane handles Hadamard indices j = 4 lane + k, stored at bitrev7(j)
    float M = -INFINITY, L = 0.f, y[4] = {0.f, 0.f, 0.f, 0.f};
    // the BF16 segment's partials of the row (unrotated domain), loaded now
    // so that their latency overlaps the split-K merge; used by the row's
    // first warp after the un-rotation
    float bm[kMaxBfItems], bl[kMaxBfItems], bo[kMaxBfItems][4];
    {
        const float* bp = p.bf_part + (size_t)(b * p.hk + kv) * p.bf_items * p.part_stride;
#pragma unroll
        for (int it = 0; it < kMaxBfItems; ++it) {
            bm[it] = -INFINITY;
            bl[it] = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) bo[it][c] = 0.f;
            if (active && sub == 0 && it < p.bf_items) {
                const float* pt = bp + (size_t)it * p.part_stride;
                bm[it] = pt[(size_t)p.G * kD + hh];
                bl[it] = pt[(size_t)p.G * kD + p.G + hh];
#pragma unroll
                for (int c = 0; c < 4; ++c) bo[it][c] = pt[(size_t)hh * kD + lane + 32 * c];
            }
        }
    }
    if (active) {
        // this warp's splits sub, sub + wpr, ..., merged by online log-sum-exp
        // in batches whose loads (statistics and this lane's four values of
        // each split) are all issued before any is used
        const int nmine = splits > sub ? (splits - sub + wpr - 1) / wpr : 0;
        for (int i0 = 0; i0 < nmine; i0 += kMergeBatch) {
            float ms[kMergeBatch], ls[kMergeBatch], ov[kMergeBatch][4];
#pragma unroll
            for (int i = 0; i < kMergeBatch; ++i) {
                ms[i] = -INFINITY;
                ls[i] = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) ov[i][k] = 0.f;
                if (i0 + i < nmine) {
                    const int sp = sub + wpr * (i0 + i);
                    const float* pt =
                        p.part + (size_t)(sp < n_long ? first + sp : first2 + sp) * p.part_stride;
                    ms[i] = pt[(size_t)p.G * kD + hh];
                    ls[i] = pt[(size_t)p.G * kD + p.G + hh];
#pragma unroll
                    for (int k = 0; k < 4; ++k) ov[i][k] = pt[(size_t)hh * kD + 32 * bitrev2(k) + r5];
                }
            }
            float mb = M;
#pragma unroll
            for (int i = 0; i < kMergeBatch; ++i)
                if (ls[i] > 0.f) mb = fmaxf(mb, ms[i]);
            if (mb != -INFINITY) {
                const float a = (M == -INFINITY) ? 0.f : ex2(M - mb);
                L *= a;
#pragma unroll
                for (int k = 0; k < 4; ++k) y[k] *= a;
#pragma unroll
                for (int i = 0; i < kMergeBatch; ++i) {
                    const float sc = (ls[i] > 0.f) ? ex2(ms[i] - mb) : 0.f;
                    L = fmaf(sc, ls[i], L);
#pragma unroll
                    for (int k = 0; k < 4; ++k) y[k] = fmaf(sc, ov[i][k], y[k]);
                }
                M = mb;
            }
        }
    }
    if (wpr > 1) {  // combine the row's shares in its first warp
        float* ws = Ws + (size_t)warp * kMergeRow;
        *reinterpret_cast<float4*>(ws + 4 * lane) = make_float4(y[0], y[1], y[2], y[3]);
        if (lane == 0) {
            ws[kD] = M;
            ws[kD + 1] = L;
        }
        __syncthreads();
        if (sub == 0 && active) {
            float Mt = -INFINITY;
            for (int i = 0; i < wpr; ++i) Mt = fmaxf(Mt, Ws[(size_t)(warp + i) * kMergeRow + kD]);
            float Lt = 0.f, yt[4] = {0.f, 0.f, 0.f, 0.f};
            if (Mt != -INFINITY) {
                for (int i = 0; i < wpr; ++i) {
                    const float* wi = Ws + (size_t)(warp + i) * kMergeRow;
                    if (wi[kD] == -INFINITY) continue;
                    const float sc = ex2(wi[kD] - Mt);
                    Lt = fmaf(sc, wi[kD + 1], Lt);
                    const float4 v = *reinterpret_cast<const float4*>(wi + 4 * lane);
                    yt[0] = fmaf(sc, v.x, yt[0]);
                    yt[1] = fmaf(sc, v.y, yt[1]);
                    yt[2] = fmaf(sc, v.z, yt[2]);
                    yt[3] = fmaf(sc, v.w, yt[3]);
                }
            }
            M = Mt;
            L = Lt;
#pragma unroll
            for (int k = 0; k < 4; ++k) y[k] = yt[k];
        }
        __syncthreads();  // shares read before the rows' w overwrite them
    }
    const bool lead = active && sub == 0;
    if (sub == 0) {  // the row's w (zero for rows past the batch)
        const float inv = (L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) y[k] = active ? y[k] * inv : 0.f;
        {
            const float t0 = y[0] + y[1], t1 = y[0] - y[1], t2 = y[2] + y[3], t3 = y[2] - y[3];
            y[0] = t0 + t2;
            y[2] = t0 - t2;
            y[1] = t1 + t3;
            y[3] = t1 - t3;
        }
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float o = __shfl_xor_sync(kFull, y[k], m);
                y[k] = upper ? o - y[k] : y[k] + o;
            }
        }
        *reinterpret_cast<float4*>(Ws + (size_t)warp * kMergeRow + 4 * lane) =
            make_float4(y[0] * (float)kInvSqrtD, y[1] * (float)kInvSqrtD, y[2] * (float)kInvSqrtD,
                        y[3] * (float)kInvSqrtD);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    {   // un-rotation on tensor cores: A row gID = block row gID (its w in Ws[gID * wpr]), B = U_V^T
        const int gID = lane >> 2, tq = lane & 3;
        const float* wrow = Ws + (size_t)(gID * wpr) * kMergeRow;
        const bool rowok = gID < rpb;
        float d[2][4] = {};
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
            const int k0 = 16 * ks + 2 * tq;
            float2 w0 = make_float2(0.f, 0.f), w1 = w0;
            if (rowok) {
                w0 = *reinterpret_cast<const float2*>(wrow + k0);
                w1 = *reinterpret_cast<const float2*>(wrow + k0 + 8);
            }
            uint32_t ah0, ah2, al0, al2;
            {
                const float v[4] = {w0.x, w0.y, w1.x, w1.y};
                split_f16(v, ah0, ah2, al0, al2);
            }
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int a = 16 * warp + 8 * t + gID;  // output (column n = gID of n-tile 2 warp + t)
                const float2 u0 = *reinterpret_cast<const float2*>(Us + (size_t)a * kURow + k0);
                const float2 u1 = *reinterpret_cast<const float2*>(Us + (size_t)a * kURow + k0 + 8);
                uint32_t bh0, bh1, bl0, bl1;
                const float v[4] = {u0.x, u0.y, u1.x, u1.y};
                split_f16(v, bh0, bh1, bl0, bl1);
                mma_f16_16816(d[t], ah0, 0u, ah2, 0u, bh0, bh1);
                mma_f16_16816(d[t], ah0, 0u, ah2, 0u, bl0, bl1);
                mma_f16_16816(d[t], al0, 0u, al2, 0u, bh0, bh1);
            }
        }
        if (rowok) {  // D rows 0-7 = block rows: outputs 16 warp + 8 t + 2 tq, + 1
#pragma unroll
            for (int t = 0; t < 2; ++t)
                *reinterpret_cast<float2*>(Ys + (size_t)gID * kMergeRow + 16 * warp + 8 * t + 2 * tq) =
                    make_float2(d[t][0], d[t][1]);
        }
    }
    __syncthreads();
    if (!lead) return;
    const float* yrow = Ys + (size_t)(warp / wpr) * kMergeRow;
    // BF16 segment: log-sum-exp merge of its item partials (unrotated domain)
    float mb = -INFINITY;
#pragma unroll
    for (int it = 0; it < kMaxBfItems; ++it)
        if (bl[it] > 0.f) mb = fmaxf(mb, bm[it]);
    float lb = 0.f, ob[4] = {0.f, 0.f, 0.f, 0.f};
    if (mb != -INFINITY) {
#pragma unroll
        for (int it = 0; it < kMaxBfItems; ++it) {
            if (bl[it] > 0.f) {
                const float sc = ex2(bm[it] - mb);
                lb = fmaf(sc, bl[it], lb);
#pragma unroll
                for (int c = 0; c < 4; ++c) ob[c] = fmaf(sc, bo[it][c], ob[c]);
            }
        }
    }
    const float Mx = fmaxf(L > 0.f ? M : -INFINITY, lb > 0.f ? mb : -INFINITY);
    const float wi = (L > 0.f) ? ex2(M - Mx) * L : 0.f;
    const float wb = (lb > 0.f) ? ex2(mb - Mx) : 0.f;
    const float den = wi + wb * lb;
    const float inv = (den > 0.f) ? 1.f / den : 0.f;
    float* o = p.out + ((size_t)b * p.hq + kv * p.G + hh) * kD;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int a2 = lane + 32 * c;
        o[a2] = (wi * yrow[a2] + wb * ob[c]) * inv;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
struct Int2Attr {
    int sms = 0;
    bool set1 = false, set2 = false, setl = false, setl2 = false, setk = false, setk2 = false, setm = false,
         setp = false, setb = false;
};

static Int2Attr& attr_for_device(int dev) {
    static Int2Attr attrs[64];
    return attrs[dev & 63];
}

// Dynamic shared memory of a kernel, and the largest L1 / shared carveout:
// an SM changes its split only when idle, so every kernel of the chain asks
// for the same split and a programmatically launched kernel can start on SMs
// where its predecessor still runs.  (Not for the eight-head Lloyd-Max INT2
// kernel: its register spills go through L1, which the largest split leaves
// at 28 KB; it took 9 % longer with it.)
template <typename... Args>
static cudaError_t set_smem(void (*kernel)(Args...), int bytes, bool max_carveout = true) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && max_carveout)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    return e;
}

template <int NT, bool LM = false, bool BOOST = false>
static cudaError_t launch_int2(const DecodeParams& p, cudaStream_t st, int sms, bool& attr_set) {
    using SM = Int2Smem<NT, int2_stages<NT, LM, BOOST>()>;
    constexpr int smem = int2_q_prefetch<NT, LM, BOOST>() ? SM::kBytesQP : ((LM || BOOST) ? SM::kBytesLM : SM::kBytes);
    // the blocks of one SM share its 228 KB (1 KB of it reserved per block)
    static_assert(int2_blocks_per_sm<NT, LM, BOOST>() * (smem + 1024) <= 228 * 1024, "blocks per SM must fit");
    if (!attr_set) {
        cudaError_t e = set_smem(int2_kernel<NT, LM, BOOST>, smem, !(NT == 2 && LM));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int per_sm = int2_blocks_per_sm<NT, LM, BOOST>();
    const int64_t max_items =
        (int64_t)p.B * p.hk * ((p.max_pages + p.pps - 1) / p.pps + p.tail_pg / kShortItemPages);
    int blocks = (int)std::min<int64_t>((int64_t)per_sm * sms, max_items);
    if (blocks < 1) blocks = 1;
    cudaError_t e = launch_pdl(int2_kernel<NT, LM, BOOST>, dim3(blocks), dim3(kInt2Threads), smem, st, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Launch with a programmatic dependency on the previous kernel in the stream
// (the kernel itself decides where it waits, see pdl_wait).
template <typename... Args>
static cudaError_t launch_pdl(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              const DecodeParams& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

cudaError_t launch_decode(const DecodeParams& pin, cudaStream_t st, cudaEvent_t ev_int2_start,
                          cudaEvent_t ev_int2_stop) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    Int2Attr& at = attr_for_device(dev);
    if (at.sms == 0) {
        e = cudaDeviceGetAttribute(&at.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    DecodeParams p = pin;
    {   // Fewer history pages (at most) than two waves of minimum items on
        // the INT2 grid (a batch of one or two long sequences): items of one
        // wave instead, so that no block takes a second item while others
        // idle.  Longer items only lower the item count the workspace was
        // sized for.
        const int per_sm = (p.NT == 1 || !(p.codebook || p.boost)) ? 3 : 2;  // as int2_blocks_per_sm
        const int64_t blocks = (int64_t)per_sm * at.sms;
        const int64_t line = (int64_t)p.B * p.hk * p.max_pages;
        if (p.pps == kShortItemPages && line < 2 * kShortItemPages * blocks) {
            const int pps = (int)std::min<int64_t>(256, ((line + blocks - 1) / blocks + 3) & ~3ll);
            if (pps > p.pps) {
                p.pps = pps;
                p.tail_pg = 2 * kShortItemPages;
            }
        }
    }
    if (!at.setp) {
        e = set_smem(prep_kernel, kPrepSmem);
        if (e != cudaSuccess) return e;
        at.setp = true;
    }
    dim3 pg((p.B + kPrepSeqs - 1) / kPrepSeqs + 1, p.hk);
    if ((e = launch_pdl(prep_kernel, pg, dim3(kPrepThreads), kPrepSmem, st, p)) != cudaSuccess) return e;
    if (ev_int2_start && (e = cudaEventRecord(ev_int2_start, st)) != cudaSuccess) return e;
    if (p.codebook)  // Lloyd-Max levels
        e = (p.NT == 1) ? launch_int2<1, true>(p, st, at.sms, at.setl) : launch_int2<2, true>(p, st, at.sms, at.setl2);
    else if (p.boost)  // K channel boost
        e = (p.NT == 1) ? launch_int2<1, false, true>(p, st, at.sms, at.setk)
                        : launch_int2<2, false, true>(p, st, at.sms, at.setk2);
    else
        e = (p.NT == 1) ? launch_int2<1>(p, st, at.sms, at.set1) : launch_int2<2>(p, st, at.sms, at.set2);
    if (e != cudaSuccess) return e;
    if (ev_int2_stop && (e = cudaEventRecord(ev_int2_stop, st)) != cudaSuccess) return e;
    if (!at.setb) {
        e = set_smem(bf16_kernel, kBfSmem);
        if (e != cudaSuccess) return e;
        at.setb = true;
    }
    const int bf_total = p.bf_items * p.B * p.hk;
    e = launch_pdl(bf16_kernel, dim3(min(bf_total, 3 * at.sms)), dim3(kBfThreads), kBfSmem, st, p);
    if (e != cudaSuccess) return e;
    if (!at.setm) {
        e = set_smem(merge_kernel, kMergeSmem);
        if (e != cudaSuccess) return e;
        at.setm = true;
    }
    const int rpb = kMergeWarps / p.merge_wpr;
    dim3 mg((p.B * p.G + rpb - 1) / rpb, p.hk);
    return launch_pdl(merge_kernel, mg, dim3(kMergeThreads), kMergeSmem, st, p);
}

}  // namespace oscar
