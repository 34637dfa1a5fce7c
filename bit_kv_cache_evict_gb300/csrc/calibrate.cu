// calibrate.cu -- offline calibration of the orthogonal factor U of the
// rotation R = U . Hadamard . bit-reversal, following
// "卓绝TurboQuant：Together AI把2-bit KV Cache推向实在行状", section
// "OSCAR 把旋转瞄准 attention": U is fixed offline per layer and KV head, for
// K from the covariance of the queries that read the keys, for V from the
// covariance of the values as weighted by the attention scores.  Reading
// (the pages give no formula): U_K = eigenvectors of the mean of q q^T over
// the calibration query tokens of every query head of the KV group; U_V =
// eigenvectors of the mean of o o^T, o = softmax(q K^T sm_scale) V the
// attention output of those heads over the calibration tokens (sum o o^T =
// V^T S^T S V); columns by decreasing eigenvalue, each with its entry of
// largest magnitude positive.
//
// Kernels, in launch order:
//   calib_attn_kernel   o for every (query token, query head): one warp, one
//                       lane per calibration token of a 32-token chunk for the
//                       logits, online softmax, lanes split the dimensions
//                       for the weighted sum (fp32).
//   calib_cov_kernel    sum of x x^T per KV head over the samples of a chunk
//                       (q as bf16, o as fp32), fp32 atomics into C.
//   calib_eig_kernel    one block per (KV head, K/V) matrix: cyclic Jacobi
//                       with the round-robin ordering (64 disjoint rotations
//                       per round, 127 rounds per sweep) on the matrix held in
//                       shared memory, off-diagonal updates in Rutishauser's
//                       form (a - s (b + tau a), tau = s / (1 + c)) and each
//                       rotated 2 x 2 block set exactly; then the eigenpairs
//                       sorted and signed.
#include "oscar_common.cuh"

namespace oscar {

// ---------------------------------------------------------------------------
// attention outputs
// ---------------------------------------------------------------------------
constexpr int kCalAttnWarps = 8;

__global__ void __launch_bounds__(32 * kCalAttnWarps) calib_attn_kernel(CalibParams p) {
    __shared__ float qs[kCalAttnWarps][kD];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row = blockIdx.x * kCalAttnWarps + warp;  // (query token, query head)
    if (row >= p.n_q * p.hq) return;
    const int h = row % p.hq, kv = h / (p.hq / p.hk);
    {
        const uint2 qr = *reinterpret_cast<const uint2*>(p.q + (size_t)row * kD + 4 * lane);
        qs[warp][4 * lane + 0] = bf16_lo(qr.x);
        qs[warp][4 * lane + 1] = bf16_hi(qr.x);
        qs[warp][4 * lane + 2] = bf16_lo(qr.y);
        qs[warp][4 * lane + 3] = bf16_hi(qr.y);
    }
    __syncwarp();
    const float scale = p.sm_scale * kLog2e;
    const size_t tok_stride = (size_t)p.hk * 2 * kD;  // bf16 elements per calibration token
    float m = -INFINITY, l = 0.f, o[4] = {0.f, 0.f, 0.f, 0.f};
    for (int t0 = 0; t0 < p.n_t; t0 += 32) {
        const int t = t0 + lane;
        float logit = -INFINITY;
        if (t < p.n_t) {
            const uint4* kr = reinterpret_cast<const uint4*>(p.kv + t * tok_stride + (size_t)kv * 2 * kD);
            float acc = 0.f;
#pragma unroll 4
            for (int c = 0; c < kD / 8; ++c) {
                const uint4 w = kr[c];
                const float* qq = qs[warp] + 8 * c;
                acc = fmaf(qq[0], bf16_lo(w.x), acc);
                acc = fmaf(qq[1], bf16_hi(w.x), acc);
                acc = fmaf(qq[2], bf16_lo(w.y), acc);
                acc = fmaf(qq[3], bf16_hi(w.y), acc);
                acc = fmaf(qq[4], bf16_lo(w.z), acc);
                acc = fmaf(qq[5], bf16_hi(w.z), acc);
                acc = fmaf(qq[6], bf16_lo(w.w), acc);
                acc = fmaf(qq[7], bf16_hi(w.w), acc);
            }
            logit = acc * scale;
        }
        float mx = logit;
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, s));
        const float m_new = fmaxf(m, mx);
        const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - m_new);
        const float pt = (t < p.n_t) ? exp2f(logit - m_new) : 0.f;
        float ps = pt;
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) ps += __shfl_xor_sync(kFull, ps, s);
        l = l * alpha + ps;
#pragma unroll
        for (int k = 0; k < 4; ++k) o[k] *= alpha;
        m = m_new;
        const int cnt = min(32, p.n_t - t0);
        for (int i = 0; i < cnt; ++i) {
            const float w = __shfl_sync(kFull, pt, i);
            const uint2 vr = *reinterpret_cast<const uint2*>(p.kv + (t0 + i) * tok_stride + (size_t)(kv * 2 + 1) * kD +
                                                             4 * lane);
            o[0] = fmaf(w, bf16_lo(vr.x), o[0]);
            o[1] = fmaf(w, bf16_hi(vr.x), o[1]);
            o[2] = fmaf(w, bf16_lo(vr.y), o[2]);
            o[3] = fmaf(w, bf16_hi(vr.y), o[3]);
        }
    }
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
    *reinterpret_cast<float4*>(p.o + (size_t)row * kD + 4 * lane) =
        make_float4(o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv);
}

// ---------------------------------------------------------------------------
// covariance: C[kv] += sum over a chunk of samples of x x^T
// ---------------------------------------------------------------------------
constexpr int kCovThreads = 256;     // thread (i, j) of a 16 x 16 grid: C[8i..8i+7][8j..8j+7]
constexpr int kCovStage = 32;        // samples staged in shared memory at a time
constexpr int kCovChunk = 512;       // samples per block

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }

// x: [n][hq][kD]; the samples of KV head kv are (token n, head kv*G + j)
template <typename T>
__global__ void __launch_bounds__(kCovThreads) calib_cov_kernel(const T* x, int n, int hq, int hk, float* C) {
    __shared__ float xs[kCovStage][kD];
    const int kv = blockIdx.y, g = hq / hk;
    const int total = n * g;
    const int s0 = blockIdx.x * kCovChunk, s1 = min(total, s0 + kCovChunk);
    const int ti = threadIdx.x >> 4, tj = threadIdx.x & 15;
    float acc[8][8];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = 0.f;
    for (int sb = s0; sb < s1; sb += kCovStage) {
        const int cnt = min(kCovStage, s1 - sb);
        __syncthreads();
        for (int e = threadIdx.x; e < kCovStage * kD; e += kCovThreads) {
            const int r = e / kD, c = e % kD;
            float v = 0.f;
            if (r < cnt) {
                const int s = sb + r, tok = s / g, hh = kv * g + s % g;
                v = to_f32<T>(x[((size_t)tok * hq + hh) * kD + c]);
            }
            xs[r][c] = v;
        }
        __syncthreads();
        for (int r = 0; r < cnt; ++r) {
            float xi[8], xj[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                xi[a] = xs[r][8 * ti + a];
                xj[a] = xs[r][8 * tj + a];
            }
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(xi[a], xj[b], acc[a][b]);
        }
    }
    float* Ck = C + (size_t)kv * kD * kD;
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) atomicAdd(Ck + (8 * ti + a) * kD + 8 * tj + b, acc[a][b]);
}

// ---------------------------------------------------------------------------
// symmetric eigensolver (cyclic Jacobi, round-robin ordering)
// ---------------------------------------------------------------------------
constexpr int kEigThreads = 512;
constexpr int kEigLd = kD + 1;       // padded row of the shared matrices
constexpr int kEigMaxSweeps = 24;    // fp32 converges in well under this
constexpr int kEigSmem = 2 * kD * kEigLd * 4 + 6 * 64 * 4 + 2 * kD * 4 + 64;

// Round r of the round-robin: pair k (0..63) = (0, 1 + r) for k = 0, else
// (1 + (r + k) mod 127, 1 + (r - k) mod 127).  Every pair of the 128 indices
// meets once in 127 rounds, and the 64 pairs of a round are disjoint.
__device__ __forceinline__ void rr_pair(int r, int k, int& pp, int& qq) {
    if (k == 0) {
        pp = 0;
        qq = 1 + r;
    } else {
        pp = 1 + (r + k) % 127;
        qq = 1 + (r - k + 127) % 127;
    }
}

// C: sums of kD x kD matrices, scaled by inv_count.  Block (x, y) takes
// matrix C + x * kD * kD + y * c_y; its eigenvectors go to U + x * ustride +
// y * u_y (column j = eigenvector j, row-major kD x kD) and its eigenvalues
// to lam + x * lstride + y * l_y (lam may be null).  One launch serves the K
// (y = 0) and V (y = 1) matrices of every KV head.
__global__ void __launch_bounds__(kEigThreads) calib_eig_kernel(const float* C, float inv_count, float* U,
                                                                size_t ustride, float* lam, size_t lstride,
                                                                int* status, size_t c_y, size_t u_y, size_t l_y) {
    extern __shared__ __align__(16) float esm[];
    float* A = esm;                      // [kD][kEigLd]
    float* V = A + kD * kEigLd;          // [kD][kEigLd]
    float* cs = V + kD * kEigLd;         // [64] c of the round's rotations
    float* sn = cs + 64;                 // [64] s
    float* tn = sn + 64;                 // [64] t = s / c
    float* d0 = tn + 64;                 // [64] a_pp, a_qq, a_pq before the round
    float* d1 = d0 + 64;
    float* d2 = d1 + 64;
    float* red = d2 + 64;                // [kD] reduction scratch
    int* rank = reinterpret_cast<int*>(red + kD);   // [kD]
    const int tid = threadIdx.x;
    const size_t mo = (size_t)blockIdx.x * kD * kD + blockIdx.y * c_y;
    for (int e = tid; e < kD * kD; e += kEigThreads) {
        const int i = e / kD, j = e % kD;
        // symmetrise the accumulated sums (the atomics add in any order)
        A[i * kEigLd + j] = 0.5f * (C[mo + (size_t)i * kD + j] + C[mo + (size_t)j * kD + i]) * inv_count;
        V[i * kEigLd + j] = (i == j) ? 1.f : 0.f;
    }
    __syncthreads();
    // scale of the matrix: the largest diagonal entry (positive semidefinite)
    if (tid < kD) red[tid] = fabsf(A[tid * kEigLd + tid]);
    __syncthreads();
    if (tid == 0) {
        float m = 0.f;
        for (int i = 0; i < kD; ++i) m = fmaxf(m, red[i]);
        red[0] = m;
    }
    __syncthreads();
    // a pair is left alone once |a_pq| is at rounding level: below 1e-7 of
    // sqrt(|a_pp a_qq|), or below 2e-8 of the matrix scale (fp32 rounding of
    // the rotations keeps off-diagonal entries near that level); a sweep that
    // rotates nothing ends the iteration
    const float floor_abs = 2e-8f * red[0];
    int* rotated = rank;   // reused as a flag until the sort
    bool converged = false;
    for (int sweep = 0; sweep < kEigMaxSweeps && !converged; ++sweep) {
        if (tid == 0) *rotated = 0;
        __syncthreads();
        for (int r = 0; r < 127; ++r) {
            if (tid < 64) {
                int pp, qq;
                rr_pair(r, tid, pp, qq);
                const float app = A[pp * kEigLd + pp], aqq = A[qq * kEigLd + qq], apq = A[pp * kEigLd + qq];
                float c = 1.f, s = 0.f, t = 0.f;
                if (fabsf(apq) > fmaxf(1e-7f * sqrtf(fabsf(app * aqq)), floor_abs)) {
                    const float th = (aqq - app) / (2.f * apq);
                    t = copysignf(1.f, th) / (fabsf(th) + sqrtf(1.f + th * th));
                    c = 1.f / sqrtf(1.f + t * t);
                    s = t * c;
                    *rotated = 1;
                }
                cs[tid] = c;
                sn[tid] = s;
                tn[tid] = t;
                d0[tid] = app;
                d1[tid] = aqq;
                d2[tid] = apq;
            }
            __syncthreads();
            // rows p, q <- J^T rows
            for (int e = tid; e < 64 * kD; e += kEigThreads) {
                const int k = e / kD, j = e % kD;
                const float s = sn[k];
                if (s == 0.f) continue;
                const float tau = s / (1.f + cs[k]);
                int pp, qq;
                rr_pair(r, k, pp, qq);
                const float ap = A[pp * kEigLd + j], aq = A[qq * kEigLd + j];
                A[pp * kEigLd + j] = ap - s * (aq + tau * ap);
                A[qq * kEigLd + j] = aq + s * (ap - tau * aq);
            }
            __syncthreads();
            // columns p, q <- columns J (A and V)
            for (int e = tid; e < 64 * kD; e += kEigThreads) {
                const int k = e / kD, i = e % kD;
                const float s = sn[k];
                if (s == 0.f) continue;
                const float tau = s / (1.f + cs[k]);
                int pp, qq;
                rr_pair(r, k, pp, qq);
                const float ap = A[i * kEigLd + pp], aq = A[i * kEigLd + qq];
                A[i * kEigLd + pp] = ap - s * (aq + tau * ap);
                A[i * kEigLd + qq] = aq + s * (ap - tau * aq);
                const float vp = V[i * kEigLd + pp], vq = V[i * kEigLd + qq];
                V[i * kEigLd + pp] = vp - s * (vq + tau * vp);
                V[i * kEigLd + qq] = vq + s * (vp - tau * vq);
            }
            __syncthreads();
            // the rotated pair's own 2 x 2 block, set exactly: the diagonal
            // moves by -/+ t a_pq and the off-diagonal entry is zero (the
            // row and column passes above would round it twice)
            if (tid < 64 && sn[tid] != 0.f) {
                int pp, qq;
                rr_pair(r, tid, pp, qq);
                A[pp * kEigLd + pp] = d0[tid] - tn[tid] * d2[tid];
                A[qq * kEigLd + qq] = d1[tid] + tn[tid] * d2[tid];
                A[pp * kEigLd + qq] = 0.f;
                A[qq * kEigLd + pp] = 0.f;
            }
            __syncthreads();
        }
        converged = (*rotated == 0);
        __syncthreads();  // every thread read the flag before the next sweep resets it
    }
    if (!converged && tid == 0) report(status, OSCAR_STATUS_NO_CONVERGENCE);
    // sort by decreasing eigenvalue (ties by index), sign each column
    if (tid < kD) {
        const float w = A[tid * kEigLd + tid];
        int rk = 0;
        for (int j = 0; j < kD; ++j) {
            const float wj = A[j * kEigLd + j];
            rk += (wj > w || (wj == w && j < tid)) ? 1 : 0;
        }
        rank[tid] = rk;
    }
    __syncthreads();
    if (tid < kD) {  // column tid of V -> column rank[tid] of U
        int imax = 0;
        float vmax = -1.f;
        for (int i = 0; i < kD; ++i) {
            const float a = fabsf(V[i * kEigLd + tid]);
            if (a > vmax) {
                vmax = a;
                imax = i;
            }
        }
        const float sg = V[imax * kEigLd + tid] < 0.f ? -1.f : 1.f;
        const int col = rank[tid];
        float* Um = U + blockIdx.x * ustride + blockIdx.y * u_y;
        for (int i = 0; i < kD; ++i) Um[(size_t)i * kD + col] = sg * V[i * kEigLd + tid];
        if (lam) lam[blockIdx.x * lstride + blockIdx.y * l_y + col] = A[tid * kEigLd + tid];
    }
}

// ---------------------------------------------------------------------------
// clip-threshold search
// ---------------------------------------------------------------------------
// Block = (chunk of calibration tokens, (KV head, K/V)): U of the matrix is
// staged in shared memory; each warp rotates one token at a time,
// y = x . U . H (fp32, Hadamard by warp shuffles, scaled 1/sqrt(d)), with
// lane l holding Hadamard outputs j = 4l + k whose stored positions
// bitrev7(j) put value k of every lane in 32-position block bitrev2(k) -- so
// a block's statistics are warp reductions, as in the eviction.  For every
// candidate ratio c the token is quantised as the eviction does (clip to
// +-c max|y| per group, fp16 s = (max - min) / 3 and z = min, codes from the
// stored s, z) and sum (y - y^)^2 is added to the candidate's total.
constexpr int kClipWarps = 8;
constexpr int kClipTokens = 64;       // tokens per block

__global__ void __launch_bounds__(32 * kClipWarps) calib_clip_kernel(ClipParams p) {
    extern __shared__ __align__(16) float csm[];
    float* Us = csm;                                   // [kD][kD]
    float* errs = Us + kD * kD;                        // [kMaxClipGrid]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int mat = blockIdx.y;                        // kv * 2 + which
    const int kv = mat >> 1, which = mat & 1;
    const float* Ug = p.U + (size_t)mat * kD * kD;
    for (int i = threadIdx.x; i < kD * kD / 4; i += 32 * kClipWarps)
        reinterpret_cast<float4*>(Us)[i] = reinterpret_cast<const float4*>(Ug)[i];
    if (threadIdx.x < kMaxClipGrid) errs[threadIdx.x] = 0.f;
    __syncthreads();
    const int gshift = p.gshift;
    const int t_end = min(p.n_t, (blockIdx.x + 1) * kClipTokens);
    for (int t = blockIdx.x * kClipTokens + warp; t < t_end; t += kClipWarps) {
        const uint2 xr = *reinterpret_cast<const uint2*>(p.kv + ((size_t)t * p.hk * 2 + mat) * kD + 4 * lane);
        const float x[4] = {bf16_lo(xr.x), bf16_hi(xr.x), bf16_lo(xr.y), bf16_hi(xr.y)};
        float y[4] = {0.f, 0.f, 0.f, 0.f};
        for (int a = 0; a < kD; ++a) {
            const float xa = __shfl_sync(kFull, x[a & 3], a >> 2);
            const float4 u = *reinterpret_cast<const float4*>(Us + a * kD + 4 * lane);
            y[0] = fmaf(xa, u.x, y[0]);
            y[1] = fmaf(xa, u.y, y[1]);
            y[2] = fmaf(xa, u.z, y[2]);
            y[3] = fmaf(xa, u.w, y[3]);
        }
        {  // Hadamard: in-lane stages, then lanes
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
        float amax[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            y[k] *= (float)kInvSqrtD;
            amax[k] = fabsf(y[k]);
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1)
#pragma unroll
            for (int k = 0; k < 4; ++k) amax[k] = fmaxf(amax[k], __shfl_xor_sync(kFull, amax[k], m));
        if (gshift >= 1) {  // groups of 64 (128) stored positions: values k = {0,2}, {1,3} (all)
            amax[0] = amax[2] = fmaxf(amax[0], amax[2]);
            amax[1] = amax[3] = fmaxf(amax[1], amax[3]);
        }
        if (gshift >= 2) amax[0] = amax[1] = amax[2] = amax[3] = fmaxf(amax[0], amax[1]);
        for (int c = 0; c < p.n_grid; ++c) {
            const float cr = p.grid[c];
            float yc[4], lo[4], hi[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float tt = cr * amax[k];
                yc[k] = cr < 1.f ? fminf(fmaxf(y[k], -tt), tt) : y[k];
                lo[k] = hi[k] = yc[k];
            }
#pragma unroll
            for (int m = 16; m > 0; m >>= 1)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    lo[k] = fminf(lo[k], __shfl_xor_sync(kFull, lo[k], m));
                    hi[k] = fmaxf(hi[k], __shfl_xor_sync(kFull, hi[k], m));
                }
            if (gshift >= 1) {
                lo[0] = lo[2] = fminf(lo[0], lo[2]);
                lo[1] = lo[3] = fminf(lo[1], lo[3]);
                hi[0] = hi[2] = fmaxf(hi[0], hi[2]);
                hi[1] = hi[3] = fmaxf(hi[1], hi[3]);
            }
            if (gshift >= 2) {
                lo[0] = lo[1] = lo[2] = lo[3] = fminf(lo[0], lo[1]);
                hi[0] = hi[1] = hi[2] = hi[3] = fmaxf(hi[0], hi[1]);
            }
            float e = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float sf = __half2float(__float2half_rn((hi[k] - lo[k]) / 3.f));
                const float zf = __half2float(__float2half_rn(lo[k]));
                float code = 0.f;
                if (sf != 0.f) code = fminf(fmaxf(rintf((yc[k] - zf) / sf), 0.f), 3.f);
                const float d = y[k] - fmaf(sf, code, zf);
                e = fmaf(d, d, e);
            }
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) e += __shfl_xor_sync(kFull, e, m);
            if (lane == 0) atomicAdd(&errs[c], e);
        }
    }
    __syncthreads();
    if (threadIdx.x < p.n_grid) atomicAdd(p.err + (size_t)mat * kMaxClipGrid + threadIdx.x, (double)errs[threadIdx.x]);
}

// the ratio with the least error per matrix (the larger ratio on ties)
__global__ void calib_clip_pick_kernel(ClipParams p) {
    const int mat = threadIdx.x;
    if (mat >= p.hk * 2) return;
    const double* e = p.err + (size_t)mat * kMaxClipGrid;
    const double denom = (double)p.n_t * kD;
    int best = 0;
    for (int c = 1; c < p.n_grid; ++c)
        if (e[c] < e[best] || (e[c] == e[best] && p.grid[c] > p.grid[best])) best = c;
    p.clip[mat] = p.grid[best];
    if (p.mse)
        for (int c = 0; c < p.n_grid; ++c) p.mse[(size_t)mat * p.n_grid + c] = (float)(e[c] / denom);
}

// ---------------------------------------------------------------------------
// Lloyd-Max codebook fit
// ---------------------------------------------------------------------------
// Folded code coordinates of the calibration tokens: for every element, u =
// (y_c - z) / s under the eviction's quantiser with the matrix's clip ratio
// (rotation in fp32 as in the clip search), folded to v = min(u, 3 - u)
// clamped to [0, 3/2] (the codebook is symmetric); groups with s = 0 give
// no samples (v = -1, skipped by the fit).
__global__ void __launch_bounds__(32 * kClipWarps) calib_fold_kernel(FitParams p) {
    extern __shared__ __align__(16) float fsm[];
    float* Us = fsm;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int mat = blockIdx.y;
    const float* Ug = p.U + (size_t)mat * kD * kD;
    for (int i = threadIdx.x; i < kD * kD / 4; i += 32 * kClipWarps)
        reinterpret_cast<float4*>(Us)[i] = reinterpret_cast<const float4*>(Ug)[i];
    __syncthreads();
    const float cr = p.clip[mat];
    const int gshift = p.gshift;
    const int t_end = min(p.n_t, (blockIdx.x + 1) * kClipTokens);
    for (int t = blockIdx.x * kClipTokens + warp; t < t_end; t += kClipWarps) {
        const uint2 xr = *reinterpret_cast<const uint2*>(p.kv + ((size_t)t * p.hk * 2 + mat) * kD + 4 * lane);
        const float x[4] = {bf16_lo(xr.x), bf16_hi(xr.x), bf16_lo(xr.y), bf16_hi(xr.y)};
        float y[4] = {0.f, 0.f, 0.f, 0.f};
        for (int a = 0; a < kD; ++a) {
            const float xa = __shfl_sync(kFull, x[a & 3], a >> 2);
            const float4 u = *reinterpret_cast<const float4*>(Us + a * kD + 4 * lane);
            y[0] = fmaf(xa, u.x, y[0]);
            y[1] = fmaf(xa, u.y, y[1]);
            y[2] = fmaf(xa, u.z, y[2]);
            y[3] = fmaf(xa, u.w, y[3]);
        }
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
        float amax[4], lo[4], hi[4], yc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            y[k] *= (float)kInvSqrtD;
            amax[k] = fabsf(y[k]);
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1)
#pragma unroll
            for (int k = 0; k < 4; ++k) amax[k] = fmaxf(amax[k], __shfl_xor_sync(kFull, amax[k], m));
        if (gshift >= 1) {
            amax[0] = amax[2] = fmaxf(amax[0], amax[2]);
            amax[1] = amax[3] = fmaxf(amax[1], amax[3]);
        }
        if (gshift >= 2) amax[0] = amax[1] = amax[2] = amax[3] = fmaxf(amax[0], amax[1]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float tt = cr * amax[k];
            yc[k] = cr < 1.f ? fminf(fmaxf(y[k], -tt), tt) : y[k];
            lo[k] = hi[k] = yc[k];
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                lo[k] = fminf(lo[k], __shfl_xor_sync(kFull, lo[k], m));
                hi[k] = fmaxf(hi[k], __shfl_xor_sync(kFull, hi[k], m));
            }
        if (gshift >= 1) {
            lo[0] = lo[2] = fminf(lo[0], lo[2]);
            lo[1] = lo[3] = fminf(lo[1], lo[3]);
            hi[0] = hi[2] = fmaxf(hi[0], hi[2]);
            hi[1] = hi[3] = fmaxf(hi[1], hi[3]);
        }
        if (gshift >= 2) {
            lo[0] = lo[1] = lo[2] = lo[3] = fminf(lo[0], lo[1]);
            hi[0] = hi[1] = hi[2] = hi[3] = fmaxf(hi[0], hi[1]);
        }
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float sf = __half2float(__float2half_rn((hi[k] - lo[k]) / 3.f));
            const float zf = __half2float(__float2half_rn(lo[k]));
            if (sf == 0.f) {
                v[k] = -1.f;
            } else {
                const float u = (yc[k] - zf) / sf;
                v[k] = fminf(fmaxf(fminf(u, 3.f - u), 0.f), 1.5f);
            }
        }
        *reinterpret_cast<float4*>(p.v + ((size_t)mat * p.n_t + t) * kD + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
    }
}

// One block per matrix: Lloyd's iteration a <- mean{v : v >= a/2} from a = 1
// until a moves by less than 1e-6 (at most kFitIters rounds).
constexpr int kFitThreads = 512, kFitIters = 200;
__global__ void __launch_bounds__(kFitThreads) calib_lloyd_kernel(FitParams p) {
    __shared__ float rs[kFitThreads / 32], rc[kFitThreads / 32];
    __shared__ float a_sh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, mat = blockIdx.x;
    const float* v = p.v + (size_t)mat * p.n_t * kD;
    const size_t n = (size_t)p.n_t * kD;
    float a = 1.f;
    for (int it = 0; it < kFitIters; ++it) {
        const float th = 0.5f * a;
        float sum = 0.f, cnt = 0.f;
        for (size_t i = tid; i < n; i += kFitThreads) {
            const float x = v[i];
            if (x >= th) {
                sum += x;
                cnt += 1.f;
            }
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) {
            sum += __shfl_xor_sync(kFull, sum, m);
            cnt += __shfl_xor_sync(kFull, cnt, m);
        }
        if (lane == 0) {
            rs[warp] = sum;
            rc[warp] = cnt;
        }
        __syncthreads();
        if (tid == 0) {
            float S = 0.f, C = 0.f;
            for (int w = 0; w < kFitThreads / 32; ++w) {
                S += rs[w];
                C += rc[w];
            }
            a_sh = C > 0.f ? S / C : a;
        }
        __syncthreads();
        const float a_new = a_sh;
        __syncthreads();
        const bool done = fabsf(a_new - a) < 1e-6f;
        a = a_new;
        if (done) break;
    }
    if (tid == 0) p.a[mat] = a;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
cudaError_t launch_calibrate_codebook(const FitParams& p, cudaStream_t st) {
    const int smem = kD * kD * 4;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool attr_set[64] = {};
    if (!attr_set[dev & 63]) {
        e = cudaFuncSetAttribute(calib_fold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set[dev & 63] = true;
    }
    dim3 grid((p.n_t + kClipTokens - 1) / kClipTokens, p.hk * 2);
    calib_fold_kernel<<<grid, 32 * kClipWarps, smem, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    calib_lloyd_kernel<<<p.hk * 2, kFitThreads, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_calibrate_clip(const ClipParams& p, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(p.err, 0, (size_t)p.hk * 2 * kMaxClipGrid * sizeof(double), st);
    if (e != cudaSuccess) return e;
    const int smem = (kD * kD + kMaxClipGrid) * 4;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    static bool attr_set[64] = {};
    if (!attr_set[dev & 63]) {
        e = cudaFuncSetAttribute(calib_clip_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set[dev & 63] = true;
    }
    dim3 grid((p.n_t + kClipTokens - 1) / kClipTokens, p.hk * 2);
    calib_clip_kernel<<<grid, 32 * kClipWarps, smem, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    calib_clip_pick_kernel<<<1, 32 * ((p.hk * 2 + 31) / 32), 0, st>>>(p);
    return cudaGetLastError();
}
cudaError_t launch_calibrate(const CalibParams& p, cudaStream_t st) {
    const size_t mat = (size_t)kD * kD;
    cudaError_t e = cudaMemsetAsync(p.C, 0, (size_t)p.hk * 2 * mat * sizeof(float), st);
    if (e != cudaSuccess) return e;
    const int rows = p.n_q * p.hq;
    calib_attn_kernel<<<(rows + kCalAttnWarps - 1) / kCalAttnWarps, 32 * kCalAttnWarps, 0, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // C_K of KV head kv at C + kv * mat, C_V at C + (hk + kv) * mat
    const int g = p.hq / p.hk;
    dim3 cg((p.n_q * g + kCovChunk - 1) / kCovChunk, p.hk);
    calib_cov_kernel<__nv_bfloat16><<<cg, kCovThreads, 0, st>>>(p.q, p.n_q, p.hq, p.hk, p.C);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    calib_cov_kernel<float><<<cg, kCovThreads, 0, st>>>(p.o, p.n_q, p.hq, p.hk, p.C + (size_t)p.hk * mat);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    static bool attr_set[64] = {};
    if (!attr_set[dev & 63]) {
        e = cudaFuncSetAttribute(calib_eig_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kEigSmem);
        if (e != cudaSuccess) return e;
        attr_set[dev & 63] = true;
    }
    // outputs in the [hk][2] (K, V) layout of U and lam
    const float inv = 1.f / (float)(p.n_q * g);
    calib_eig_kernel<<<dim3(p.hk, 2), kEigThreads, kEigSmem, st>>>(p.C, inv, p.U, 2 * mat, p.lam, 2 * kD, p.status,
                                                                   (size_t)p.hk * mat, mat, kD);
    return cudaGetLastError();
}

}  // namespace oscar
