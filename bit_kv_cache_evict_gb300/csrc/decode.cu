// decode.cu -- decode attention over the three-segment pool (BF16 sink |
// INT2 history | BF16 recent), following the serving path of
// "卓绝TurboQuant：Together AI把2-bit KV Cache推向实在行状" (figure
// "从离线校准到在线推理的 pipeline": an INT2 kernel that unpacks,
// dequantises with scale/zero and accumulates in floating point, a BF16
// kernel for sink/recent, and an online-softmax merge).
//
// Kernels, in launch order:
//   prep_kernel       q' = q . U_K . H . P scaled by sm_scale*log2(e), split
//                     into bf16 hi+lo MMA fragments; work plan (split-K items).
//   int2_kernel<NT>   persistent warps; each takes split-K items (a run of
//                     history pages of one (sequence, KV head)), streams the
//                     6 KB page blocks into shared memory with bulk async
//                     copies, and runs both products on tensor cores
//                     (mma.sync m16n8k16 bf16 -> fp32) straight from the
//                     packed codes.
//   bf16_kernel       sink + recent window per (sequence, KV head).
//   merge_kernel      log-sum-exp merge of the INT2 splits, un-rotation by
//                     R_V^T (bit-reversal, Hadamard, U_V^T), merge with the
//                     BF16 partial.
//
// Exact factoring used by int2_kernel.  With codes c, per-(token, group)
// fp16 scale s and zero z, and A-operand values 8 + c (the code placed in
// bf16 mantissa bits, see codes_to_bf16x2):
//   logit_t = sum_g s_tg * D_tg + (z_tg - 8 s_tg) * Q_g,
//       D_tg = sum_{j in g} (8 + c_tj) q'_j  (MMA, tokens x heads),
//       Q_g  = sum_{j in g} q'_j;
//   o'_j   = sum_t W_t,g(j) (8 + c_tj) + sum_t p_t (z_tg - 8 s_tg),
//       W_tg = p_t s_tg                     (MMA, dims x heads).
// q' and W are split into bf16 hi + lo (two MMA columns per head), so the
// products keep ~2^-17 relative precision; codes are exact in bf16.
#include "oscar_common.cuh"

namespace oscar {


// ---------------------------------------------------------------------------
// prep: rotated query fragments + split-K plan
// ---------------------------------------------------------------------------
// One warp per (b, kv, nt, hh): head h = kv*G + 4*nt + hh (hh >= G: zero
// padding columns).  The last block builds the plan.
__global__ void __launch_bounds__(128) prep_kernel(DecodeParams p) {
    __shared__ float qs[4][kD];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    if (blockIdx.x == gridDim.x - 1) {  // plan
        if (warp != 0) return;
        int running = 0;
        if (lane == 0) {
            p.item_start[0] = 0;
            *p.counter = 0;
        }
        for (int base = 0; base < p.B; base += 32) {
            const int b = base + lane;
            int items = 0;
            if (b < p.B) {
                int h = p.hist_len[b];
                if (h < 0 || h > p.max_pages * kPage) {
                    report(p.status, OSCAR_STATUS_BAD_POS);
                    h = min(max(h, 0), p.max_pages * kPage);
                }
                const int npg = (h + kPage - 1) / kPage;
                items = ((npg + p.pps - 1) / p.pps) * p.hk;
            }
            int incl = items;
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                const int v = __shfl_up_sync(kFull, incl, m);
                if (lane >= m) incl += v;
            }
            if (b < p.B) p.item_start[b + 1] = running + incl;
            running += __shfl_sync(kFull, incl, 31);
        }
        return;
    }

    const int wid = blockIdx.x * 4 + warp;  // = ((b*Hk + kv)*NT + nt)*4 + hh
    if (wid >= p.B * p.hk * p.NT * 4) return;
    const int hh = wid & 3;
    const int nt = (wid >> 2) % p.NT;
    const int bk = (wid >> 2) / p.NT;
    const int b = bk / p.hk, kv = bk % p.hk;
    const int hl = 4 * nt + hh;  // head within the KV group
    uint32_t* frag = p.qfrag + ((size_t)bk * p.NT + nt) * 8 * 32 * 2;
    float* qsum = p.qsum + ((size_t)bk * p.NT * 4 + hl) * 4;

    if (hl >= p.G) {  // padding column pair: zeros
        const int ks = lane >> 2, tq = lane & 3;
#pragma unroll
        for (int par = 0; par < 2; ++par) {
            const int L = (2 * hh + par) * 4 + tq;
            *reinterpret_cast<uint2*>(frag + ((size_t)ks * 32 + L) * 2) = make_uint2(0u, 0u);
        }
        if (lane < 4) qsum[lane] = 0.f;
        return;
    }
    const int h = kv * p.G + hl;
    const uint2 qr = *reinterpret_cast<const uint2*>(p.q + ((size_t)b * p.hq + h) * kD + 4 * lane);
    const float x[4] = {bf16_lo(qr.x), bf16_hi(qr.x), bf16_lo(qr.y), bf16_hi(qr.y)};
    const float* Uk = p.U + ((size_t)kv * 2 + 0) * kD * kD;
    float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int a = 0; a < kD; ++a) {
        const float xa = __shfl_sync(kFull, x[a & 3], a >> 2);
        const float4 u = __ldg(reinterpret_cast<const float4*>(Uk + (size_t)a * kD + 4 * lane));
        y[0] = fmaf(xa, u.x, y[0]);
        y[1] = fmaf(xa, u.y, y[1]);
        y[2] = fmaf(xa, u.z, y[2]);
        y[3] = fmaf(xa, u.w, y[3]);
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
#pragma unroll
    for (int k = 0; k < 4; ++k) qs[warp][32 * bitrev2(k) + r5] = y[k] * scale;  // stored order
    __syncwarp();

    // group sums of the split values (exactly what the MMA multiplies)
    float gs = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float v = qs[warp][4 * lane + k];
        const float hi = __bfloat162float(__float2bfloat16_rn(v));
        const float lo = __bfloat162float(__float2bfloat16_rn(v - hi));
        gs += hi + lo;
    }
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) gs += __shfl_xor_sync(kFull, gs, m);
    if ((lane & 7) == 0) qsum[lane >> 3] = gs;

    // fragments: lane -> (ks, tq); b0 = (q'[16ks+tq], q'[16ks+8+tq]),
    // b1 = (q'[16ks+4+tq], q'[16ks+12+tq]); column 2hh = hi, 2hh+1 = lo
    const int ks = lane >> 2, tq = lane & 3;
    const float v0 = qs[warp][16 * ks + tq], v1 = qs[warp][16 * ks + 8 + tq];
    const float v2 = qs[warp][16 * ks + 4 + tq], v3 = qs[warp][16 * ks + 12 + tq];
    const uint32_t h01 = pack_bf16x2_rn(v0, v1), h23 = pack_bf16x2_rn(v2, v3);
    const uint32_t l01 = pack_bf16x2_rn(v0 - bf16_lo(h01), v1 - bf16_hi(h01));
    const uint32_t l23 = pack_bf16x2_rn(v2 - bf16_lo(h23), v3 - bf16_hi(h23));
    *reinterpret_cast<uint2*>(frag + ((size_t)ks * 32 + (2 * hh) * 4 + tq) * 2) = make_uint2(h01, h23);
    *reinterpret_cast<uint2*>(frag + ((size_t)ks * 32 + (2 * hh + 1) * 4 + tq) * 2) = make_uint2(l01, l23);
}

// ---------------------------------------------------------------------------
// INT2 split-K decode
// ---------------------------------------------------------------------------
constexpr int kStages = 3;
constexpr int kWaitPolls = 1 << 22;

template <int NT>
struct Int2Smem {
    static constexpr int kStageBytes = kStages * kBlock;
    static constexpr int kScaleBytes = kPage * 4 * 16;  // per token: sK, zzK, sV, zzV (float4 each)
    static constexpr int kPBytes = NT * 4 * kPage * 4;
    static constexpr int kWarpBytes = kStageBytes + kScaleBytes + kPBytes + 64;
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

template <int NT>
__global__ void __launch_bounds__(128, 2) int2_kernel(DecodeParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    using SM = Int2Smem<NT>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gID = lane >> 2, tq = lane & 3;
    uint8_t* wsm = smem + warp * SM::kWarpBytes;
    uint8_t* stage_buf = wsm;
    float4* sc4 = reinterpret_cast<float4*>(wsm + SM::kStageBytes);
    float* pbuf = reinterpret_cast<float*>(wsm + SM::kStageBytes + SM::kScaleBytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(wsm + SM::kStageBytes + SM::kScaleBytes + SM::kPBytes);
    int* stage_valid = reinterpret_cast<int*>(bars + kStages);

    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    const int total = __ldg(p.item_start + p.B);
    // lane-dependent rotations for the K operand: codes at bits 2tq / 16+2tq
    // and 8+2tq / 24+2tq move to bits 4-5 / 20-21
    const uint32_t rotA = (uint32_t)(2 * tq + 28) & 31u, rotB = (uint32_t)(4 + 2 * tq);
    const bool lo_lane = (gID & 1) != 0;  // PV B-operand column parity: hi / lo
    uint32_t issued = 0, consumed = 0;    // page-stream counters (stage = n % kStages)

    for (;;) {
        int item = 0;
        if (lane == 0) item = atomicAdd(p.counter, 1);
        item = __shfl_sync(kFull, item, 0);
        if (item >= total) break;
        const int b = find_seq(p.item_start, p.B, item);
        const int s0 = __ldg(p.item_start + b);
        const int splits = (__ldg(p.item_start + b + 1) - s0) / p.hk;
        const int local = item - s0;
        const int kv = local / splits, split = local % splits;
        const int hist = min(max(__ldg(p.hist_len + b), 0), p.max_pages * kPage);
        const int npg_seq = (hist + kPage - 1) / kPage;
        const int pg0 = split * p.pps;
        const int npg = min(p.pps, npg_seq - pg0);
        const int bk = b * p.hk + kv;

        // rotated-query fragments and group sums for this (b, kv)
        uint32_t qf[NT][8][2];
        float4 qsv[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint32_t* fr = p.qfrag + ((size_t)bk * NT + nt) * 8 * 32 * 2;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint2 v = *reinterpret_cast<const uint2*>(fr + ((size_t)ks * 32 + lane) * 2);
                qf[nt][ks][0] = v.x;
                qf[nt][ks][1] = v.y;
            }
            qsv[nt] = *reinterpret_cast<const float4*>(p.qsum + ((size_t)bk * NT * 4 + 4 * nt + tq) * 4);
        }

        float m_run[NT], l_run[NT], zacc[NT][4], acc_o[NT][8][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m_run[nt] = -INFINITY;
            l_run[nt] = 0.f;
#pragma unroll
            for (int g = 0; g < 4; ++g) zacc[nt][g] = 0.f;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc_o[nt][mt][e] = 0.f;
        }

        auto issue = [&](int pi_local) {  // lane 0 only
            const int st = issued % kStages;
            const int pi = pg0 + pi_local;
            const int pid = __ldg(p.page_table + (size_t)b * p.max_pages + pi);
            if (pid < 0 || pid >= p.num_pages) {
                report(p.status, OSCAR_STATUS_BAD_PAGE);
                stage_valid[st] = 0;
                mbar_arrive(&bars[st]);
            } else {
                stage_valid[st] = min(kPage, hist - pi * kPage);
                mbar_arrive_expect_tx(&bars[st], kBlock);
                bulk_g2s(stage_buf + st * kBlock, p.pool + ((size_t)pid * p.hk + kv) * kBlock, kBlock, &bars[st]);
            }
            ++issued;
        };
        if (lane == 0)
            for (int i = 0; i < min(kStages, npg); ++i) issue(i);
        issued = __shfl_sync(kFull, issued, 0);
        __syncwarp();

        bool failed = false;
        for (int pl = 0; pl < npg; ++pl) {
            const int st = consumed % kStages;
            const uint32_t parity = (consumed / kStages) & 1u;
            const bool ok = __all_sync(kFull, mbar_wait_bounded(&bars[st], parity, kWaitPolls));
            if (!ok) {
                failed = true;
                break;
            }
            ++consumed;
            const uint8_t* blk = stage_buf + st * kBlock;
            const int valid = stage_valid[st];

            // -- scales: fp16 (s, z) -> fp32 (s, z - 8 s); zero for masked slots
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
                const int t = lane + 32 * tt;
                const uint4 kw = *reinterpret_cast<const uint4*>(blk + kKScale + t * 16);
                const uint4 vw = *reinterpret_cast<const uint4*>(blk + kVScale + t * 16);
                const bool on = t < valid;
                const uint32_t kk[4] = {kw.x, kw.y, kw.z, kw.w}, vv[4] = {vw.x, vw.y, vw.z, vw.w};
                float ks_[4], kz_[4], vs_[4], vz_[4];
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const float sk = half_lo(kk[g]), zk = half_hi(kk[g]);
                    const float sv = half_lo(vv[g]), zv = half_hi(vv[g]);
                    ks_[g] = on ? sk : 0.f;
                    kz_[g] = on ? fmaf(-8.f, sk, zk) : 0.f;
                    vs_[g] = on ? sv : 0.f;
                    vz_[g] = on ? fmaf(-8.f, sv, zv) : 0.f;
                }
                sc4[t * 4 + 0] = make_float4(ks_[0], ks_[1], ks_[2], ks_[3]);
                sc4[t * 4 + 1] = make_float4(kz_[0], kz_[1], kz_[2], kz_[3]);
                sc4[t * 4 + 2] = make_float4(vs_[0], vs_[1], vs_[2], vs_[3]);
                sc4[t * 4 + 3] = make_float4(vz_[0], vz_[1], vz_[2], vz_[3]);
            }
            __syncwarp();

            // -- logits: rows = tokens (2gID, 2gID+1 of each 16-token tile)
            float sv[4][NT][2];
#pragma unroll
            for (int tile = 0; tile < 4; ++tile) {
                const int tA = tile * 16 + 2 * gID;
                const uint4* kr = reinterpret_cast<const uint4*>(blk + kKCodes + tA * 32);
                const uint4 ka0 = kr[0], ka1 = kr[1], kb0 = kr[2], kb1 = kr[3];
                const uint32_t wa[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
                const uint32_t wb[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
                float acc[4][NT][4];
#pragma unroll
                for (int g = 0; g < 4; ++g)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[g][nt][e] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t a0 = codes_to_bf16x2(rotr(wa[ks], rotA));
                    const uint32_t a1 = codes_to_bf16x2(rotr(wb[ks], rotA));
                    const uint32_t a2 = codes_to_bf16x2(rotr(wa[ks], rotB));
                    const uint32_t a3 = codes_to_bf16x2(rotr(wb[ks], rotB));
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_bf16_16816(acc[ks >> 1][nt], a0, a1, a2, a3, qf[nt][ks][0], qf[nt][ks][1]);
                }
                const float4 sA = sc4[tA * 4 + 0], zA = sc4[tA * 4 + 1];
                const float4 sB = sc4[(tA + 1) * 4 + 0], zB = sc4[(tA + 1) * 4 + 1];
                const float sa[4] = {sA.x, sA.y, sA.z, sA.w}, za[4] = {zA.x, zA.y, zA.z, zA.w};
                const float sb[4] = {sB.x, sB.y, sB.z, sB.w}, zb[4] = {zB.x, zB.y, zB.z, zB.w};
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float qg[4] = {qsv[nt].x, qsv[nt].y, qsv[nt].z, qsv[nt].w};
                    float la = 0.f, lb = 0.f;
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        la = fmaf(sa[g], acc[g][nt][0] + acc[g][nt][1], la);
                        la = fmaf(za[g], qg[g], la);
                        lb = fmaf(sb[g], acc[g][nt][2] + acc[g][nt][3], lb);
                        lb = fmaf(zb[g], qg[g], lb);
                    }
                    sv[tile][nt][0] = (tA < valid) ? la : -INFINITY;
                    sv[tile][nt][1] = (tA + 1 < valid) ? lb : -INFINITY;
                }
            }

            // -- online softmax (base 2): page max per head, rescale, p
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float mx = -INFINITY;
#pragma unroll
                for (int tile = 0; tile < 4; ++tile) mx = fmaxf(mx, fmaxf(sv[tile][nt][0], sv[tile][nt][1]));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
                const float m_new = fmaxf(m_run[nt], mx);
                if (m_new > m_run[nt]) {  // uniform across the lanes of head tq
                    const float alpha = ex2(m_run[nt] - m_new);
                    l_run[nt] *= alpha;
#pragma unroll
                    for (int g = 0; g < 4; ++g) zacc[nt][g] *= alpha;
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc_o[nt][mt][e] *= alpha;
                    m_run[nt] = m_new;
                }
                // all tokens masked so far: subtract 0 so p = ex2(-inf) = 0
                const float m_sub = (m_new == -INFINITY) ? 0.f : m_new;
#pragma unroll
                for (int tile = 0; tile < 4; ++tile) {
                    const int tA = tile * 16 + 2 * gID;
                    const float pa = ex2(sv[tile][nt][0] - m_sub);
                    const float pb = ex2(sv[tile][nt][1] - m_sub);
                    l_run[nt] += pa + pb;
                    const float4 vzA = sc4[tA * 4 + 3], vzB = sc4[(tA + 1) * 4 + 3];
                    zacc[nt][0] = fmaf(pa, vzA.x, fmaf(pb, vzB.x, zacc[nt][0]));
                    zacc[nt][1] = fmaf(pa, vzA.y, fmaf(pb, vzB.y, zacc[nt][1]));
                    zacc[nt][2] = fmaf(pa, vzA.z, fmaf(pb, vzB.z, zacc[nt][2]));
                    zacc[nt][3] = fmaf(pa, vzA.w, fmaf(pb, vzB.w, zacc[nt][3]));
                    *reinterpret_cast<float2*>(pbuf + (nt * 4 + tq) * kPage + tA) = make_float2(pa, pb);
                }
            }
            __syncwarp();

            // -- values: rows = dims, columns = heads (hi, lo), k = tokens
#pragma unroll
            for (int tile = 0; tile < 4; ++tile) {
                const int t0 = tile * 16 + 4 * tq;
                float4 pp[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    pp[nt] = *reinterpret_cast<const float4*>(pbuf + (nt * 4 + (gID >> 1)) * kPage + t0);
                const float4 s0 = sc4[(t0 + 0) * 4 + 2], s1 = sc4[(t0 + 1) * 4 + 2];
                const float4 s2 = sc4[(t0 + 2) * 4 + 2], s3 = sc4[(t0 + 3) * 4 + 2];
                const float sv0[4] = {s0.x, s0.y, s0.z, s0.w}, sv1[4] = {s1.x, s1.y, s1.z, s1.w};
                const float sv2[4] = {s2.x, s2.y, s2.z, s2.w}, sv3[4] = {s3.x, s3.y, s3.z, s3.w};
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const uint32_t wv =
                        *reinterpret_cast<const uint32_t*>(blk + kVCodes + (8 * g + gID) * kPage + t0);
                    uint32_t bb0[NT], bb1[NT];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const float w0 = pp[nt].x * sv0[g], w1 = pp[nt].y * sv1[g];
                        const float w2 = pp[nt].z * sv2[g], w3 = pp[nt].w * sv3[g];
                        // hi lanes: bf16 truncation; lo lanes: rounded remainder
                        const uint32_t u0 = __float_as_uint(w0), u1 = __float_as_uint(w1);
                        const uint32_t u2 = __float_as_uint(w2), u3 = __float_as_uint(w3);
                        const uint32_t hi02 = __byte_perm(u0, u2, 0x7632), hi13 = __byte_perm(u1, u3, 0x7632);
                        const uint32_t lo02 = pack_bf16x2_rn(w0 - __uint_as_float(u0 & 0xffff0000u),
                                                             w2 - __uint_as_float(u2 & 0xffff0000u));
                        const uint32_t lo13 = pack_bf16x2_rn(w1 - __uint_as_float(u1 & 0xffff0000u),
                                                             w3 - __uint_as_float(u3 & 0xffff0000u));
                        bb0[nt] = lo_lane ? lo02 : hi02;
                        bb1[nt] = lo_lane ? lo13 : hi13;
                    }
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const uint32_t sa0 = (uint32_t)(4 * half + 28) & 31u;      // slot 2half, bytes 0/2
                        const uint32_t sa1 = (uint32_t)(4 * half + 30) & 31u;      // slot 2half+1
                        const uint32_t a0 = codes_to_bf16x2(rotr(wv, sa0));
                        const uint32_t a1 = codes_to_bf16x2(rotr(wv, sa1));
                        const uint32_t a2 = codes_to_bf16x2(rotr(wv, (uint32_t)(4 + 4 * half)));
                        const uint32_t a3 = codes_to_bf16x2(rotr(wv, (uint32_t)(6 + 4 * half)));
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma_bf16_16816(acc_o[nt][2 * g + half], a0, a1, a2, a3, bb0[nt], bb1[nt]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0 && pl + kStages < npg) issue(pl + kStages);
            issued = __shfl_sync(kFull, issued, 0);
            __syncwarp();
        }
        if (failed) {
            if (lane == 0) report(p.status, OSCAR_STATUS_TIMEOUT);
            // let copies still in flight land before the block can exit
            while (consumed < issued) {
                const int st = consumed % kStages;
                (void)mbar_wait_bounded(&bars[st], (consumed / kStages) & 1u, kWaitPolls);
                ++consumed;
            }
            return;
        }

        // -- partial (unnormalised o', base-2 max m, sum l) of this item
        float* part = p.part + (size_t)item * p.part_stride;
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
            const int hl = 4 * nt + tq;
            if (hl < p.G) {
                float* o = part + (size_t)hl * kD;
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    *reinterpret_cast<float4*>(o + 32 * g + 4 * gID) = make_float4(
                        acc_o[nt][2 * g][0] + acc_o[nt][2 * g][1] + z[g],
                        acc_o[nt][2 * g][2] + acc_o[nt][2 * g][3] + z[g],
                        acc_o[nt][2 * g + 1][0] + acc_o[nt][2 * g + 1][1] + z[g],
                        acc_o[nt][2 * g + 1][2] + acc_o[nt][2 * g + 1][3] + z[g]);
                if (gID == 0) {
                    part[(size_t)p.G * kD + hl] = m_run[nt];
                    part[(size_t)p.G * kD + p.G + hl] = l;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// BF16 sink + recent segment
// ---------------------------------------------------------------------------
// One block (4 warps) per (b, kv); warp w takes slots w, w+4, ...; lane l
// owns dims 4l..4l+3.  Logits in base 2 (q scaled by sm_scale*log2 e).
struct Bf16Red {
    float m[4][8], l[4][8];
    float o[4][8][kD];
};

template <int G>
__device__ void bf16_segment(const DecodeParams& p, int b, int kv, Bf16Red& red) {
    auto& red_m = red.m;
    auto& red_l = red.l;
    auto& red_o = red.o;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float qv[G][4], m[G], l[G], o[G][4];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        const uint2 qr = *reinterpret_cast<const uint2*>(p.q + ((size_t)b * p.hq + kv * G + hh) * kD + 4 * lane);
        qv[hh][0] = bf16_lo(qr.x) * p.qscale;
        qv[hh][1] = bf16_hi(qr.x) * p.qscale;
        qv[hh][2] = bf16_lo(qr.y) * p.qscale;
        qv[hh][3] = bf16_hi(qr.y) * p.qscale;
        m[hh] = -INFINITY;
        l[hh] = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) o[hh][e] = 0.f;
    }
    const int n = min(max(__ldg(p.bf16_len + b), 0), p.nslot);
    for (int t = warp; t < n; t += 4) {
        const __nv_bfloat16* row = p.bf16_kv + (((size_t)b * p.nslot + t) * p.hk + kv) * 2 * kD;
        const uint2 kr = *reinterpret_cast<const uint2*>(row + 4 * lane);
        const uint2 vr = *reinterpret_cast<const uint2*>(row + kD + 4 * lane);
        const float k4[4] = {bf16_lo(kr.x), bf16_hi(kr.x), bf16_lo(kr.y), bf16_hi(kr.y)};
        const float v4[4] = {bf16_lo(vr.x), bf16_hi(vr.x), bf16_lo(vr.y), bf16_hi(vr.y)};
        float s[G];
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            float d = qv[hh][0] * k4[0];
            d = fmaf(qv[hh][1], k4[1], d);
            d = fmaf(qv[hh][2], k4[2], d);
            d = fmaf(qv[hh][3], k4[3], d);
            s[hh] = d;
        }
#pragma unroll
        for (int mm = 16; mm > 0; mm >>= 1)
#pragma unroll
            for (int hh = 0; hh < G; ++hh) s[hh] += __shfl_xor_sync(kFull, s[hh], mm);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            const float mn = fmaxf(m[hh], s[hh]);
            const float alpha = ex2(m[hh] - mn);
            const float pr = ex2(s[hh] - mn);
            l[hh] = l[hh] * alpha + pr;
#pragma unroll
            for (int e = 0; e < 4; ++e) o[hh][e] = fmaf(pr, v4[e], o[hh][e] * alpha);
            m[hh] = mn;
        }
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        if (lane == 0) {
            red_m[warp][hh] = m[hh];
            red_l[warp][hh] = l[hh];
        }
        *reinterpret_cast<float4*>(&red_o[warp][hh][4 * lane]) = make_float4(o[hh][0], o[hh][1], o[hh][2], o[hh][3]);
    }
    __syncthreads();
    // merge the four warps: warp w handles heads w, w+4
    float* part = p.bf_part + (size_t)(b * p.hk + kv) * p.part_stride;
    for (int hh = warp; hh < G; hh += 4) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, red_m[w][hh]);
        float L = 0.f, oo[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float sc = (red_l[w][hh] > 0.f) ? ex2(red_m[w][hh] - M) : 0.f;
            L += sc * red_l[w][hh];
            const float4 v = *reinterpret_cast<const float4*>(&red_o[w][hh][4 * lane]);
            oo[0] += sc * v.x;
            oo[1] += sc * v.y;
            oo[2] += sc * v.z;
            oo[3] += sc * v.w;
        }
        *reinterpret_cast<float4*>(part + (size_t)hh * kD + 4 * lane) = make_float4(oo[0], oo[1], oo[2], oo[3]);
        if (lane == 0) {
            part[(size_t)G * kD + hh] = M;
            part[(size_t)G * kD + G + hh] = L;
        }
    }
}

__global__ void __launch_bounds__(128) bf16_kernel(DecodeParams p) {
    __shared__ __align__(16) Bf16Red red;
    const int b = blockIdx.x / p.hk, kv = blockIdx.x % p.hk;
    switch (p.G) {
        case 1: bf16_segment<1>(p, b, kv, red); break;
        case 2: bf16_segment<2>(p, b, kv, red); break;
        case 4: bf16_segment<4>(p, b, kv, red); break;
        default: bf16_segment<8>(p, b, kv, red); break;
    }
}

// ---------------------------------------------------------------------------
// merge: INT2 splits -> un-rotate -> merge with the BF16 partial
// ---------------------------------------------------------------------------
constexpr int kMergeSeqs = 4;     // sequences per block
constexpr int kUPitch = kD + 1;   // padded row pitch of U_V in shared memory
constexpr int kMergeSmem = (kD * kUPitch + kMergeSeqs * 8 * kD + kMergeSeqs * 8 * 4) * 4;

__global__ void __launch_bounds__(256) merge_kernel(DecodeParams p) {
    extern __shared__ __align__(16) float msm[];
    float* Us = msm;                                   // [d][kUPitch]: U_V[a][j]
    float* Wr = msm + kD * kUPitch;                    // [rows][d]: normalised o'.P.H (Hadamard domain)
    float* st = Wr + kMergeSeqs * 8 * kD;              // [rows][4]: M_i2, L_i2, m_bf, l_bf
    const int kv = blockIdx.y;
    const int b0 = blockIdx.x * kMergeSeqs;
    const int nseq = min(kMergeSeqs, p.B - b0);
    const int rows = nseq * p.G;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    const float* Uv = p.U + ((size_t)kv * 2 + 1) * kD * kD;
    for (int i = threadIdx.x; i < kD * kD / 4; i += blockDim.x) {
        const float4 u = __ldg(reinterpret_cast<const float4*>(Uv) + i);
        const int a = (4 * i) / kD, j = (4 * i) % kD;
        Us[a * kUPitch + j] = u.x;
        Us[a * kUPitch + j + 1] = u.y;
        Us[a * kUPitch + j + 2] = u.z;
        Us[a * kUPitch + j + 3] = u.w;
    }
    const int r5 = bitrev5(lane);
    for (int r = warp; r < rows; r += 8) {
        const int b = b0 + r / p.G, hh = r % p.G;
        const int s0 = __ldg(p.item_start + b);
        const int splits = (__ldg(p.item_start + b + 1) - s0) / p.hk;
        const int first = s0 + kv * splits;
        // lane handles Hadamard indices j = 4 lane + k, stored at bitrev7(j)
        float M = -INFINITY;
        for (int s = lane; s < splits; s += 32)
            M = fmaxf(M, p.part[(size_t)(first + s) * p.part_stride + (size_t)p.G * kD + hh]);
#pragma unroll
        for (int mm = 16; mm > 0; mm >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, mm));
        float L = 0.f, y[4] = {0.f, 0.f, 0.f, 0.f};
        for (int s = 0; s < splits; ++s) {
            const float* pt = p.part + (size_t)(first + s) * p.part_stride;
            const float ls = pt[(size_t)p.G * kD + p.G + hh];
            if (!(ls > 0.f)) continue;
            const float sc = ex2(pt[(size_t)p.G * kD + hh] - M);
            L += sc * ls;
#pragma unroll
            for (int k = 0; k < 4; ++k) y[k] = fmaf(sc, pt[(size_t)hh * kD + 32 * bitrev2(k) + r5], y[k]);
        }
        const float inv = (L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) y[k] *= inv;
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
        *reinterpret_cast<float4*>(Wr + (size_t)r * kD + 4 * lane) =
            make_float4(y[0] * (float)kInvSqrtD, y[1] * (float)kInvSqrtD, y[2] * (float)kInvSqrtD,
                        y[3] * (float)kInvSqrtD);
        if (lane == 0) {
            const float* bp = p.bf_part + (size_t)(b * p.hk + kv) * p.part_stride;
            st[r * 4 + 0] = M;
            st[r * 4 + 1] = L;
            st[r * 4 + 2] = bp[(size_t)p.G * kD + hh];
            st[r * 4 + 3] = bp[(size_t)p.G * kD + p.G + hh];
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < rows * kD; idx += blockDim.x) {
        const int r = idx / kD, a = idx % kD;
        const int b = b0 + r / p.G, hh = r % p.G;
        const float* w = Wr + (size_t)r * kD;
        const float* u = Us + a * kUPitch;
        float acc = 0.f;
#pragma unroll 8
        for (int j = 0; j < kD; ++j) acc = fmaf(w[j], u[j], acc);
        const float Mi = st[r * 4 + 0], Li = st[r * 4 + 1], mb = st[r * 4 + 2], lb = st[r * 4 + 3];
        const float Mx = fmaxf(Li > 0.f ? Mi : -INFINITY, lb > 0.f ? mb : -INFINITY);
        const float wi = (Li > 0.f) ? ex2(Mi - Mx) * Li : 0.f;
        const float wb = (lb > 0.f) ? ex2(mb - Mx) : 0.f;
        const float den = wi + wb * lb;
        const float ob = p.bf_part[(size_t)(b * p.hk + kv) * p.part_stride + (size_t)hh * kD + a];
        p.out[((size_t)b * p.hq + kv * p.G + hh) * kD + a] = (den > 0.f) ? (wi * acc + wb * ob) / den : 0.f;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
struct Int2Attr {
    int sms = 0;
    bool set1 = false, set2 = false, setm = false;
};

static Int2Attr& attr_for_device(int dev) {
    static Int2Attr attrs[64];
    return attrs[dev & 63];
}

template <int NT>
static cudaError_t launch_int2(const DecodeParams& p, cudaStream_t st, int sms, bool& attr_set) {
    const int smem = 4 * Int2Smem<NT>::kWarpBytes;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(int2_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int max_items = p.B * p.hk * ((p.max_pages + p.pps - 1) / p.pps);
    int blocks = min(2 * sms, (max_items + 3) / 4);
    if (blocks < 1) blocks = 1;
    int2_kernel<NT><<<blocks, 128, smem, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t st, cudaEvent_t ev_int2_start,
                          cudaEvent_t ev_int2_stop) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    Int2Attr& at = attr_for_device(dev);
    if (at.sms == 0) {
        e = cudaDeviceGetAttribute(&at.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    const int prep_warps = p.B * p.hk * p.NT * 4;
    prep_kernel<<<(prep_warps + 3) / 4 + 1, 128, 0, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (ev_int2_start && (e = cudaEventRecord(ev_int2_start, st)) != cudaSuccess) return e;
    e = (p.NT == 1) ? launch_int2<1>(p, st, at.sms, at.set1) : launch_int2<2>(p, st, at.sms, at.set2);
    if (e != cudaSuccess) return e;
    if (ev_int2_stop && (e = cudaEventRecord(ev_int2_stop, st)) != cudaSuccess) return e;
    bf16_kernel<<<p.B * p.hk, 128, 0, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (!at.setm) {
        e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMergeSmem);
        if (e != cudaSuccess) return e;
        at.setm = true;
    }
    dim3 mg((p.B + kMergeSeqs - 1) / kMergeSeqs, p.hk);
    merge_kernel<<<mg, 256, kMergeSmem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace oscar
