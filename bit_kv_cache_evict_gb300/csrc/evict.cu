// evict.cu -- fused rotate + clip + quantise + pack of evicted tokens into
// the paged INT2 history (the eviction kernel of the serving pipeline in
// "卓绝TurboQuant：Together AI把2-bit KV Cache推向实在行状", figure
// "从离线校准到在线推理的 pipeline"; rotation R = U.Hadamard.bit-reversal
// from section "OSCAR 把旋转瞄准 attention").
//
// One block of four warps per (token, KV head, K|V) vector; lane l owns
// Hadamard indices j = 4l..4l+3.  y = x.U is accumulated with error-free transformations
// (FMA-based exact products, TwoSum accumulation: the "Dot2" scheme of
// Ogita, Rump and Oishi, "Accurate sum and dot product", 2005), the fast
// Walsh-Hadamard transform runs on the (hi, lo) float pairs, and the group
// statistics stay on the pairs, so every code decision is taken from a value
// within 4e-7 code units of a float64 evaluation of the method (fp64
// arithmetic is avoided: GB300 runs it at a small fraction of the fp32 rate).  Stored position p = bitrev7(j) =
// 32*bitrev2(i) + bitrev5(l) for value i of lane l: each lane holds one
// element of every group (group reductions are warp reductions), and the
// four codes of one code byte (in-group index bitrev5(l) of groups 0..3).
#include "oscar_common.cuh"

namespace oscar {


struct df {  // unevaluated sum hi + lo
    float hi, lo;
};

__device__ __forceinline__ df two_sum(float a, float b) {
    float s = __fadd_rn(a, b);
    float bp = __fsub_rn(s, a);
    float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
    return {s, e};
}

__device__ __forceinline__ df fast_two_sum(float a, float b) {  // |a| >= |b|
    float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ df df_add(df a, df b) {
    df s = two_sum(a.hi, b.hi);
    float e = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
    return fast_two_sum(s.hi, e);
}

__device__ __forceinline__ df df_neg(df a) { return {-a.hi, -a.lo}; }

// exact order of normalised pairs: compare high parts, then low parts
__device__ __forceinline__ bool df_less(df a, df b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }

// merge two blocks' (max, min) into both: the extremes of their union
__device__ __forceinline__ void df_group_extremes(df& hi_a, df& hi_b, df& lo_a, df& lo_b) {
    const df h = df_less(hi_a, hi_b) ? hi_b : hi_a;
    const df l = df_less(lo_b, lo_a) ? lo_b : lo_a;
    hi_a = hi_b = h;
    lo_a = lo_b = l;
}

// Block = one (token, KV head, K|V) vector; warp w accumulates the terms
// a in [w*128/W, (w+1)*128/W) of y = x . U, warp 0 adds the W partial sums
// exactly and finishes the vector.  W = 8 when there are few vectors (a
// decode step at small batch: shorter dependent chains per warp), 4 when
// there are many.
template <int kEvictWarps>
__global__ void __launch_bounds__(32 * kEvictWarps) evict_kernel(EvictParams p) {
    constexpr int kEvictTerms = kD / kEvictWarps;
    __shared__ df part[kEvictWarps][kD];
    pdl_trigger();  // the decode's query preparation does not read what this kernel writes
    pdl_wait();     // launched early (programmatic serialization): the previous kernel's results first
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int vec = blockIdx.x;
    const int i = vec / (p.hk * 2);
    const int kv = (vec >> 1) % p.hk;
    const int which = vec & 1;

    const long row = p.src_row ? (long)__ldg(p.src_row + i) : (long)i;
    if (row < 0 || row >= p.src_rows) {
        if (threadIdx.x == 0) report(p.status, OSCAR_STATUS_BAD_POS);
        return;
    }
    // this warp's rows of U (kEvictTerms x 512 B) requested into L2 at once:
    // after a decode launch has streamed the history through L2 they come
    // from DRAM, and the term loop below reads them only a few rows ahead
    const float* Um = p.U + ((size_t)kv * 2 + which) * kD * kD;
    if (lane == 0) bulk_prefetch_l2(Um + (size_t)kEvictTerms * warp * kD, kEvictTerms * kD * 4);
    const size_t xoff = ((size_t)row * p.hk * 2 + (size_t)kv * 2 + which) * kD + 4 * lane;
    const uint2 xr = *reinterpret_cast<const uint2*>(p.src_kv + xoff);
    float x[4] = {bf16_lo(xr.x), bf16_hi(xr.x), bf16_lo(xr.y), bf16_hi(xr.y)};

    // ---- partial y = x . U over this warp's 32 terms, compensated -------------
    float s[4] = {0.f, 0.f, 0.f, 0.f}, c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int aa = 0; aa < kEvictTerms; ++aa) {
        const int a = kEvictTerms * warp + aa;
        const float xa = __shfl_sync(kFull, x[aa & 3], a >> 2);
        const float4 u = __ldg(reinterpret_cast<const float4*>(Um + (size_t)a * kD + 4 * lane));
        const float uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float pr = __fmul_rn(xa, uu[k]);
            const float pe = __fmaf_rn(xa, uu[k], -pr);  // exact product error
            const df t = two_sum(s[k], pr);
            s[k] = t.hi;
            c[k] = __fadd_rn(c[k], __fadd_rn(pe, t.lo));
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) part[warp][4 * lane + k] = two_sum(s[k], c[k]);
    __syncthreads();  // all warps have read the source row and written partials
    if (warp != 0) return;
    if (p.new_kv) {  // fused ring append: overwrite the row just read
        const size_t noff = ((size_t)i * p.hk * 2 + (size_t)kv * 2 + which) * kD + 4 * lane;
        *reinterpret_cast<uint2*>(const_cast<__nv_bfloat16*>(p.src_kv) + xoff) =
            *reinterpret_cast<const uint2*>(p.new_kv + noff);
    }
    df y[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        y[k] = part[0][4 * lane + k];
#pragma unroll
        for (int w = 1; w < kEvictWarps; ++w) y[k] = df_add(y[k], part[w][4 * lane + k]);
    }

    // ---- Walsh-Hadamard transform (unnormalised), Sylvester order ------------
    // in-lane stages (distance 1, 2)
    {
        df t0 = df_add(y[0], y[1]), t1 = df_add(y[0], df_neg(y[1]));
        df t2 = df_add(y[2], y[3]), t3 = df_add(y[2], df_neg(y[3]));
        y[0] = df_add(t0, t2);
        y[2] = df_add(t0, df_neg(t2));
        y[1] = df_add(t1, t3);
        y[3] = df_add(t1, df_neg(t3));
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {  // distance 4*m: partner lane l ^ m
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            df o{__shfl_xor_sync(kFull, y[k].hi, m), __shfl_xor_sync(kFull, y[k].lo, m)};
            y[k] = upper ? df_add(o, df_neg(y[k])) : df_add(y[k], o);
        }
    }

    // ---- per-group clip / scale / zero / codes ----------------------------------
    // Values stay double-float: y = Y / sqrt(d) with 1/sqrt(d) as a float
    // pair (0x3db504f3 + 0x30cfe77a).  Selections (max |y|, clamp, min, max)
    // are exact on the pairs; the scale and zero are rounded to fp16 from the
    // pair's fp32 value, and the code decision u = (y_c - z) / s is evaluated
    // from the exact pair difference, so its error is below 4e-7 code units.
    const float cr = __ldg(p.clip + kv * 2 + which);
    const float cb_a = p.codebook ? __ldg(p.codebook + kv * 2 + which) : 0.f;
    const float kc_hi = __uint_as_float(0x3db504f3u), kc_lo = __uint_as_float(0x30cfe77au);
    df yn[4];
    float amax[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float ph = __fmul_rn(y[k].hi, kc_hi);
        float e = __fmaf_rn(y[k].hi, kc_hi, -ph);
        e = __fmaf_rn(y[k].hi, kc_lo, e);
        e = __fmaf_rn(y[k].lo, kc_hi, e);
        yn[k] = fast_two_sum(ph, e);
        amax[k] = fabsf(yn[k].hi);
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1)
#pragma unroll
        for (int k = 0; k < 4; ++k) amax[k] = fmaxf(amax[k], __shfl_xor_sync(kFull, amax[k], m));
    // value k's 32-position block is bitrev2(k); a group of 64 (128) stored
    // positions is blocks {0,1}, {2,3} (all four): k = {0,2}, {1,3} (all)
    if (p.gshift >= 1) {
        amax[0] = amax[2] = fmaxf(amax[0], amax[2]);
        amax[1] = amax[3] = fmaxf(amax[1], amax[3]);
    }
    if (p.gshift >= 2) amax[0] = amax[1] = amax[2] = amax[3] = fmaxf(amax[0], amax[1]);
    // clamp to +-t, t = c * max|y| (fp32: an error of 1 ulp in t moves the
    // clipped values by 6e-8 relative)
    df lo[4], hi[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (cr < 1.f) {  // warp-uniform; c >= 1 clips nothing
            const float t = __fmul_rn(cr, amax[k]);
            if (yn[k].hi > t || (yn[k].hi == t && yn[k].lo > 0.f)) yn[k] = {t, 0.f};
            else if (yn[k].hi < -t || (yn[k].hi == -t && yn[k].lo < 0.f)) yn[k] = {-t, 0.f};
        }
        lo[k] = hi[k] = yn[k];
    }
    // exact min / max of the pairs: reduce the high parts, then the low parts
    // of the lanes that hold the extreme high part
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float mx = hi[k].hi, mn = lo[k].hi;
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, m));
            mn = fminf(mn, __shfl_xor_sync(kFull, mn, m));
        }
        float mxl = (hi[k].hi == mx) ? hi[k].lo : -INFINITY;
        float mnl = (lo[k].hi == mn) ? lo[k].lo : INFINITY;
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) {
            mxl = fmaxf(mxl, __shfl_xor_sync(kFull, mxl, m));
            mnl = fminf(mnl, __shfl_xor_sync(kFull, mnl, m));
        }
        hi[k] = {mx, mxl};
        lo[k] = {mn, mnl};
    }
    if (p.gshift >= 1) {
        df_group_extremes(hi[0], hi[2], lo[0], lo[2]);
        df_group_extremes(hi[1], hi[3], lo[1], lo[3]);
    }
    if (p.gshift >= 2) {
        df_group_extremes(hi[0], hi[1], lo[0], lo[1]);
        hi[2] = hi[3] = hi[0];
        lo[2] = lo[3] = lo[0];
    }
    unsigned short sb[4], zb[4];
    // value k of this lane is in-group index bitrev5(lane) of group bitrev2(k):
    // all four codes of code byte j = bitrev5(lane) are this lane's, group k in
    // bits 2k..2k+1
    uint32_t byte = 0;
    const bool boost = p.boost != nullptr && which == 0;
    float berr[4] = {0.f, 0.f, 0.f, 0.f};  // 2-bit rounding error (0 where s = 0)
    int bq4[4] = {0, 0, 0, 0};             // 4-bit code on the group range
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const df d = df_add(hi[k], df_neg(lo[k]));
        sb[k] = __half_as_ushort(__float2half_rn(__fdiv_rn(__fadd_rn(d.hi, d.lo), 3.0f)));
        zb[k] = __half_as_ushort(__float2half_rn(__fadd_rn(lo[k].hi, lo[k].lo)));
        const float sf = __half2float(__ushort_as_half(sb[k]));
        const float zf = __half2float(__ushort_as_half(zb[k]));
        int code = 0;
        if (sf != 0.f) {
            const df yz = df_add(yn[k], df{-zf, 0.f});
            const float u = __fdiv_rn(__fadd_rn(yz.hi, yz.lo), sf);
            if (cb_a > 0.f)  // Lloyd-Max levels {0, a, 3 - a, 3}: the nearest one
                code = (u >= 0.5f * cb_a) + (u >= 1.5f) + (u >= 3.f - 0.5f * cb_a);
            else
                code = (int)fminf(fmaxf(rintf(u), 0.f), 3.f);
            if (boost) {
                berr[k] = fabsf(u - (float)code);
                bq4[k] = (int)fminf(fmaxf(rintf(__fmul_rn(5.f, u)), 0.f), 15.f);
            }
        }
        byte |= (uint32_t)code << (2 * bitrev2(k));
    }

    // ---- store ---------------------------------------------------------------
    const int seq = __ldg(p.dst_seq + i);
    const int pos = __ldg(p.dst_pos + i);
    if (pos < 0 || pos >= p.max_pages * kPage || seq < 0 || seq >= p.batch) {
        if (lane == 0) report(p.status, OSCAR_STATUS_BAD_POS);
        return;
    }
    const int page = __ldg(p.page_table + (size_t)seq * p.max_pages + pos / kPage);
    if (page < 0 || page >= p.num_pages) {
        if (lane == 0) report(p.status, OSCAR_STATUS_BAD_PAGE);
        return;
    }
    const int slot = pos % kPage;
    uint8_t* blk = p.pool + ((size_t)page * p.hk + kv) * p.block_bytes;
    const int j = bitrev5(lane);
    if (which == 0) blk[kKCodes + slot * (kD / 4) + j] = (uint8_t)byte;
    else blk[kVCodes + j * kPage + slot] = (uint8_t)byte;
    if (lane == 0) {
        // group of value k is bitrev2(k) >> gshift; scale/zero words in group order
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) w[bitrev2(k) >> p.gshift] = (uint32_t)sb[k] | ((uint32_t)zb[k] << 16);
        const int ng = sz_pairs(p.gshift);
        uint8_t* sz = blk + (which == 0 ? kKScale : v_scale_off(p.gshift)) + slot * 4 * ng;
        if (ng == 4) *reinterpret_cast<uint4*>(sz) = make_uint4(w[0], w[1], w[2], w[3]);
        else if (ng == 2) *reinterpret_cast<uint2*>(sz) = make_uint2(w[0], w[1]);
        else *reinterpret_cast<uint32_t*>(sz) = w[0];
    }
    if (boost) {
        // kBoostN rounds of a warp arg-max over the 128 errors (ties to the
        // lower stored position); value k of this lane is position 32
        // bitrev2(k) + j
        uint32_t sel = 0;  // bit k: value k chosen
#pragma unroll 1
        for (int r = 0; r < kBoostN; ++r) {
            float be = -1.f;
            int bp = 1 << 30;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int pos_k = 32 * bitrev2(k) + j;
                if (!((sel >> k) & 1u) && (berr[k] > be || (berr[k] == be && pos_k < bp))) {
                    be = berr[k];
                    bp = pos_k;
                }
            }
            float me = be;
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) me = fmaxf(me, __shfl_xor_sync(kFull, me, m));
            int mp = (be == me) ? bp : (1 << 30);
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) mp = min(mp, __shfl_xor_sync(kFull, mp, m));
            if ((mp & 31) == j) sel |= 1u << bitrev2(mp >> 5);
        }
        // rank of a chosen position = chosen positions below it: per 32-position
        // block b, lane L gathers the flag of position 32 b + L (held by lane
        // bitrev5(L)) and a ballot gives the block's mask in position order
        uint32_t mask[4];
#pragma unroll
        for (int b = 0; b < 4; ++b)
            mask[b] = __ballot_sync(kFull, (__shfl_sync(kFull, sel, bitrev5(lane)) >> bitrev2(b)) & 1u);
        uint16_t* rec = reinterpret_cast<uint16_t*>(p.boost + ((size_t)page * p.hk + kv) * kBoostBlock +
                                                    slot * kBoostRecord);
        int below = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int k = bitrev2(b);
            if ((sel >> k) & 1u) {
                const int rank = below + __popc(mask[b] & ((1u << j) - 1u));
                rec[rank] = (uint16_t)((32 * b + j) | (bq4[k] << 8) | (((byte >> (2 * b)) & 3u) << 12));
            }
            below += __popc(mask[b]);
        }
    }
}

// Launched with programmatic stream serialization: the blocks may be
// scheduled while the previous kernel's last blocks finish, and wait
// (griddepcontrol.wait) for its completion before reading anything.  The
// kernel asks for the largest shared-memory carveout although it uses 8 KB:
// an SM can change its L1 / shared split only when idle, so with a small
// split the decode's kernels (up to 213 KB per SM), launched early by the
// programmatic dependency, could not start on an SM until its eviction
// blocks had drained.
cudaError_t launch_evict(const EvictParams& p, cudaStream_t st) {
    const int vecs = p.n_tok * p.hk * 2;
    if (vecs == 0) return cudaSuccess;
    static bool carveout_set[64] = {};
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return ce;
    if (!carveout_set[dev & 63]) {
        ce = cudaFuncSetAttribute(evict_kernel<8>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  (int)cudaSharedmemCarveoutMaxShared);
        if (ce == cudaSuccess)
            ce = cudaFuncSetAttribute(evict_kernel<4>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                      (int)cudaSharedmemCarveoutMaxShared);
        if (ce != cudaSuccess) return ce;
        carveout_set[dev & 63] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(vecs);
    cfg.blockDim = dim3(vecs < 512 ? 256 : 128);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = vecs < 512 ? cudaLaunchKernelEx(&cfg, evict_kernel<8>, p)
                                     : cudaLaunchKernelEx(&cfg, evict_kernel<4>, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace oscar
