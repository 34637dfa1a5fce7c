// decode_tc.cu -- the INT2 history segment of decode attention on the
// fifth-generation tensor cores (tcgen05 MMAs with operands and
// accumulators in tensor memory), for up to four query heads per KV head and
// the uniform code levels.  It computes what int2_kernel computes for that
// case (the INT2 kernel of the serving path in "卓绝TurboQuant：Together AI
// 把2-bit KV Cache推向实在行状", figure "从离线校准到在线推理的 pipeline":
// unpack, scale/zero-point dequantisation, floating-point accumulation),
// split-K over history pages, in the rotated domain.
//
// One persistent block per SM, 320 threads, warp-specialised so that the
// operand preparation of one 128-token chunk (two pages) overlaps the softmax
// of the previous one and the MMAs of both:
//   warps 0-3  unpack: the K codes (thread = token: A_K row in tensor
//              memory, 128 tokens x 128 stored positions) and the V codes
//              (thread = stored position: A_V row, 128 positions x 128
//              tokens) into bf16 operand patterns -- a 2-bit code left at
//              bits 2b, 2b + 1 of an otherwise clear bf16 half reads as
//              c 2^(2b - 133) (the subnormals and the first normal binade
//              join without a gap), one AND per register;
//   warps 4-7  softmax: after the logit MMAs (D_K = A_K . B_K: 128 tokens x
//              (block, part, head), q' = high + low + third bf16 part as
//              columns, one accumulator per block) each thread reads its token's
//              row, applies the per-(token, block) K scales and zero points,
//              runs a lazy online softmax (the reference maximum moves only
//              when a logit exceeds it by kTcTau, rescaling the accumulator
//              then), accumulates sum p and sum p z, and writes the P.V
//              weights p s~ (bf16 high part and remainder) of its token as
//              B_V rows for the value MMAs (D_V += A_V . B_V: 128 positions x
//              (block, head, part), accumulated over the split-K item); at an
//              item's last chunk it reads D_V (thread = stored position),
//              adds the zero-point term and writes the item's partial;
//   warp 8     producer: split-K items from the global work counter, bulk
//              async copies of the 6 KB page blocks into a ring of stages
//              and of the item's q' B-operand image;
//   warp 9     allocates the tensor memory; its lane 0 issues every MMA.
// Every wait is bounded; a timeout reports OSCAR_STATUS_TIMEOUT and the
// block still drains its copies and MMAs and frees the tensor memory.
#include "oscar_common.cuh"

namespace oscar {

namespace {

constexpr int kTcStages = 16;                  // page-block ring (6 KB each); the block then needs > 114 KB of shared memory: one block per SM
constexpr int kTcThreads = 10 * 32;
constexpr int kTcUnpackWarp0 = 0, kTcSoftWarp0 = 4, kTcProducerWarp = 8, kTcMmaWarp = 9;
constexpr float kTcTau = 8.f;                  // lazy-max threshold (base 2): weights stay <= 2^8
constexpr int kTcWaitPolls = 1 << 18;          // about one second per bounded wait
// fixed power-of-two scalings (exact): the K products of block b are
// c q' 2^(2b - 133 + kTcQUp); the V products use B = p s 2^(kTcVUp - 2b), so
// every P.V accumulator is 2^(kTcVUp - 133) sum(p s c)
constexpr int kTcQUp = 64, kTcVUp = 96;
constexpr float kTcVOut = 137438953472.f;     // 2^(133 - kTcVUp) = 2^37
__device__ __forceinline__ constexpr float tc_k_scale(int b) { return pow2f(133 - kTcQUp - 2 * b); }
__device__ __forceinline__ constexpr float tc_v_scale(int b) { return pow2f(kTcVUp - 2 * b); }

// tensor-memory columns (512 allocated: the whole of it, one block per SM).
// MMAs that accumulate into the same columns serialise, so the logits use
// one accumulator per 32-position block and the P.V products four
// accumulators (k-steps ks with ks % 4 = e go to accumulator e): chains of
// two MMAs that the tensor pipe overlaps.
constexpr uint32_t kTmCols = 512;
constexpr uint32_t kTmDK = 0;     // [2 chunk buffers][4 blocks][16 = 4 part + head]  logits, fp32
constexpr uint32_t kTmDV = 128;   // [4 accumulators][32 = 8 block + 2 head + part]   P.V, fp32
constexpr uint32_t kTmAK = 256;   // [2 chunk buffers][64]  K code operands, bf16 pairs
constexpr uint32_t kTmAV = 384;   // [2 chunk buffers][64]  V code operands, bf16 pairs

// stage flags of the first page slot of a chunk
constexpr int kTcFirst = 1, kTcLast = 2, kTcPadPage = 4;

struct TcInfo {
    int item, b, kv, valid_flags;   // valid tokens in bits 0-7, flags above
    int item_seq, pad[3];
};

struct TcSmem {
    static constexpr int kStage = 0;
    static constexpr int kInfo = kStage + kTcStages * kBlock;
    static constexpr int kBars = kInfo + kTcStages * (int)sizeof(TcInfo);
    // full[S], empty[S], a_ready[2], dk_ready[2], dk_free[2], w_ready[2], v_done[2], bk_full[2], bk_free[2],
    // idle, softmax-group rendezvous, softmax-group any-vote
    static constexpr int kNumBars = 2 * kTcStages + 14 + 1 + 2;
    static constexpr int kCInfo = ((kBars + kNumBars * 8 + 15) / 16) * 16;  // [2] int4: chunk records for the MMA issuer
    static constexpr int kTBase = kCInfo + 2 * 16;                 // tensor-memory base address
    static constexpr int kAny = kTBase + 16;                       // [3] int: any-vote flags
    static constexpr int kRedMax = ((kAny + 3 * 4 + 15) / 16) * 16;  // [4 warps][4 heads] float
    static constexpr int kRedSum = kRedMax + 4 * 4 * 4;            // [4 warps][20] float
    static constexpr int kBK = ((kRedSum + 4 * 20 * 4 + 1023) / 1024) * 1024;  // [2][kTcKImg]
    static constexpr int kBV = kBK + 2 * kTcKImg;                  // [2][128 tokens x 32] bf16, core-matrix layout
    static constexpr int kBytes = kBV + 2 * 8192;
};
static_assert(2 * (TcSmem::kBytes + 1024) > 228 * 1024 && TcSmem::kBytes <= 227 * 1024, "one block per SM");
static_assert(TcSmem::kInfo % 16 == 0 && TcSmem::kBars % 8 == 0 && TcSmem::kCInfo % 16 == 0 &&
                  TcSmem::kRedMax % 16 == 0 && TcSmem::kRedSum % 16 == 0 && TcSmem::kBK % 1024 == 0 &&
                  TcSmem::kBV % 1024 == 0 && sizeof(TcInfo) % 16 == 0,
              "vector and bulk-copy alignment of the shared-memory regions");

// ---- tcgen05 / tensor-memory helpers ---------------------------------------
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tm_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tm_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tm_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tm_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    tm_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tm_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
    tm_wait_ld();
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tm_st8(uint32_t taddr, const float (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                 "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
                 : "memory");
}

// Shared-memory matrix descriptor, no swizzle: start address, leading and
// stride byte offsets (the core-matrix strides along K and along N).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
           (1ull << 46);
}
// Instruction descriptor: D fp32, A and B bf16, A K-major (tensor memory),
// B MN-major, N x M = n x 128.
__device__ __forceinline__ constexpr uint32_t idesc_bf16(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{.reg .pred p; setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// B_V row of token t (0..127) of a chunk: the value operand pairs the code
// bytes 0, 2 and 1, 3 of a plane word, i.e. tokens 4a + {0, 2} and
// 4a + {1, 3}, so k = 4a + 2 (t & 1) + ((t >> 1) & 1).
__device__ __forceinline__ int tc_vrow(int t) { return (t & ~3) | ((t & 1) << 1) | ((t >> 1) & 1); }

}  // namespace

// largest b with item_start[b] <= item
__device__ __forceinline__ int find_seq_tc(const int32_t* item_start, int B, int item) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(item_start + mid) <= item) lo = mid;
        else hi = mid;
    }
    return lo;
}

template <int GS>
__device__ __forceinline__ void tc_load_row(const uint8_t* base, float (&sg)[4 >> GS], float (&zg)[4 >> GS]) {
    constexpr int NG = 4 >> GS;
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
#pragma unroll
    for (int k = 0; k < NG; ++k) {
        sg[k] = half_lo(w[k]);
        zg[k] = half_hi(w[k]);
    }
}

// The K and V scales / zero points of one token (zeros when invalid):
// sK[b] = s 2^(133 - kTcQUp - 2b), sV[b] = s 2^(kTcVUp - 2b) per 32-position
// block b (s, z of the block's group).
template <int GS>
__device__ __forceinline__ void tc_token_scales(const uint8_t* blk, int r, bool ok, float (&sK)[4], float (&zK)[4],
                                                float (&sV)[4], float (&zV)[4]) {
    constexpr int NG = 4 >> GS;
#pragma unroll
    for (int b = 0; b < 4; ++b) sK[b] = zK[b] = sV[b] = zV[b] = 0.f;
    if (!ok) return;
    float s[NG], z[NG];
    tc_load_row<GS>(blk + kKScale + r * 4 * NG, s, z);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        sK[b] = s[b >> GS] * tc_k_scale(b);
        zK[b] = z[b >> GS];
    }
    tc_load_row<GS>(blk + v_scale_off(GS) + r * 4 * NG, s, z);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        sV[b] = s[b >> GS] * tc_v_scale(b);
        zV[b] = z[b >> GS];
    }
}

__global__ void __launch_bounds__(kTcThreads, 1) int2_tc_kernel(DecodeParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    using SM = TcSmem;
    constexpr int NS = kTcStages;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t* stages = smem + SM::kStage;
    TcInfo* info = reinterpret_cast<TcInfo*>(smem + SM::kInfo);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kBars);
    uint64_t* full = bars;
    uint64_t* empty = bars + NS;
    uint64_t* a_ready = bars + 2 * NS;   // [2] unpack -> MMA: A_K, A_V of the chunk written
    uint64_t* dk_ready = a_ready + 2;    // [2] MMA -> softmax: D_K of the chunk complete
    uint64_t* dk_free = a_ready + 4;     // [2] softmax -> MMA: D_K of the chunk read
    uint64_t* w_ready = a_ready + 6;     // [2] softmax -> MMA: B_V of the chunk written
    uint64_t* v_done = a_ready + 8;      // [2] MMA -> unpack, softmax: value MMAs of the chunk complete
    uint64_t* bk_full = a_ready + 10;    // [2] producer -> MMA: the item's q' image landed
    uint64_t* bk_free = a_ready + 12;    // [2] MMA -> producer: the item's logit MMAs complete
    uint64_t* idle = a_ready + 14;
    uint64_t* grp_mb = a_ready + 15;     // rendezvous of the softmax warps
    uint64_t* any_mb = a_ready + 16;     // any-vote of the softmax warps
    int4* cinfo = reinterpret_cast<int4*>(smem + SM::kCInfo);
    uint32_t* tbase_s = reinterpret_cast<uint32_t*>(smem + SM::kTBase);
    int* any_flag = reinterpret_cast<int*>(smem + SM::kAny);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 8);          // the four unpack and the four softmax warps
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&a_ready[i], 4);
            mbar_init(&dk_ready[i], 1);
            mbar_init(&dk_free[i], 4);
            mbar_init(&w_ready[i], 4);
            mbar_init(&v_done[i], 1);
            mbar_init(&bk_full[i], 1);
            mbar_init(&bk_free[i], 1);
        }
        mbar_init(idle, 1);
        mbar_init(grp_mb, 4);
        mbar_init(any_mb, 4);
        for (int i = 0; i < 3; ++i) any_flag[i] = 0;
        fence_mbar_init();
    }
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tbase_s)),
                     "r"(kTmCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *tbase_s;
    pdl_wait();     // plan, counter, q' images and sums come from prep_kernel
    pdl_trigger();  // the BF16 segment kernel may take SMs as this grid retires

    if (warp == kTcProducerWarp) {
        // ------------------------------ producer ------------------------------
        const int total_long = __ldg(p.item_start + p.B);
        const int total = total_long + __ldg(p.item_start2 + p.B);
        uint32_t n = 0;          // page slots issued (stage n % NS)
        uint32_t item_seq = 0;   // items taken by this block
        bool ok = true;
        auto post = [&](int item, int b, int kv, int pid, int valid, int flags, int seq) -> bool {
            const uint32_t s = n % NS;
            if (n >= (uint32_t)NS) {
                const bool w = mbar_wait_bounded(&empty[s], ((n / NS) - 1) & 1u, kTcWaitPolls);
                if (!__all_sync(kFull, w)) return false;
            }
            if (lane == 0) {
                TcInfo& si = info[s];
                si.item = item;
                si.b = b;
                si.kv = kv;
                si.item_seq = seq;
                if (item >= 0 && !(flags & kTcPadPage) && (pid < 0 || pid >= p.num_pages)) {
                    report(p.status, OSCAR_STATUS_BAD_PAGE);
                    flags |= kTcPadPage;
                    valid = 0;
                }
                si.valid_flags = valid | (flags << 8);
                if (item < 0 || (flags & kTcPadPage)) {
                    mbar_arrive(&full[s]);
                } else {
                    mbar_arrive_expect_tx(&full[s], p.block_bytes);
                    bulk_g2s(stages + s * kBlock, p.pool + ((size_t)pid * p.hk + kv) * p.block_bytes, p.block_bytes,
                             &full[s]);
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
            if (item >= total) {   // one end chunk (two slots)
                for (int i = 0; i < 2 && ok; ++i) ok = post(-1, 0, 0, 0, 0, 0, 0);
                break;
            }
            const bool is_long = item < total_long;
            const int32_t* starts = is_long ? p.item_start : p.item_start2;
            const int rel = is_long ? item : item - total_long;
            const int b = find_seq_tc(starts, p.B, rel);
            const int s0 = __ldg(starts + b);
            const int splits = (__ldg(starts + b + 1) - s0) / p.hk;
            const int kv = (rel - s0) / splits;
            const int split = (rel - s0) % splits;
            const int hist = min(max(__ldg(p.hist_len + b), 0), p.max_pages * kPage);
            const int seq_pages = (hist + kPage - 1) / kPage;
            const SeqSplits sp = seq_splits(seq_pages, p.pps, p.tail_pg);
            const int pg0 = is_long ? split * p.pps : sp.long_pages + split * kShortItemPages;
            const int npg = is_long ? min(p.pps, sp.long_pages - pg0) : min(kShortItemPages, seq_pages - pg0);
            const int nslots = (npg + 1) / 2 * 2;   // whole two-page chunks
            const int nch = nslots / 2;
            // the item's q' image, once the buffer's previous item is done with it
            {
                const uint32_t ib = item_seq & 1u;
                bool w = true;
                if (item_seq >= 2) w = mbar_wait_bounded(&bk_free[ib], ((item_seq >> 1) - 1) & 1u, kTcWaitPolls);
                if (!__all_sync(kFull, w)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bk_full[ib], kTcKImg);
                    bulk_g2s(smem + SM::kBK + ib * kTcKImg, p.kimg + ((size_t)b * p.hk + kv) * kTcKImg, kTcKImg,
                             &bk_full[ib]);
                }
                __syncwarp();
            }
            for (int c = 0; c < nslots && ok; c += 32) {
                int pid = -1;
                if (c + lane < npg) pid = __ldg(p.page_table + (size_t)b * p.max_pages + pg0 + c + lane);
                const int cnt = min(32, nslots - c);
                for (int i = 0; i < cnt && ok; ++i) {
                    const int pl = c + i;
                    const int pi = __shfl_sync(kFull, pid, i);
                    const int ch = pl >> 1;
                    int flags = pl >= npg ? kTcPadPage : 0;
                    if ((pl & 1) == 0) flags |= (ch == 0 ? kTcFirst : 0) | (ch == nch - 1 ? kTcLast : 0);
                    const int valid = pl < npg ? min(kPage, hist - (pg0 + pl) * kPage) : 0;
                    ok = post(item, b, kv, pi, valid, flags, (int)item_seq);
                }
            }
            ++item_seq;
            if (!ok) break;
        }
        if (!ok) {
            if (lane == 0) report(p.status, OSCAR_STATUS_TIMEOUT);
            // let issued copies land before the block can exit
            const uint32_t first = n > (uint32_t)NS ? n - NS : 0;
            for (uint32_t k = first; k < n; ++k)
                (void)mbar_wait_bounded(&full[k % NS], (k / NS) & 1u, kTcWaitPolls);
            for (uint32_t i = item_seq > 2 ? item_seq - 2 : 0; i < item_seq; ++i)
                (void)mbar_wait_bounded(&bk_full[i & 1], (i >> 1) & 1u, kTcWaitPolls);
        }
    } else if (warp == kTcMmaWarp) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            int cur_seq = -1;
            bool pend_v = false;   // value MMAs of the previous chunk still to issue
            int4 prev = make_int4(0, 0, 0, 0);
            bool ok = true;
            auto issue_v = [&](uint32_t k, const int4& ci) -> bool {
                const uint32_t b = k & 1u;
                if (!mbar_wait_bounded(&w_ready[b], (k >> 1) & 1u, kTcWaitPolls)) return false;
                tc_fence_after();
                const uint32_t bv = smem_u32(smem + SM::kBV + b * 8192);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)   // four independent accumulation chains
                    tc_mma(tb + kTmDV + 32 * (ks & 3), tb + kTmAV + 64 * b + 8 * ks,
                           smem_desc(bv + 256 * ks, 128, 2048), idesc_bf16(32),
                           (ks >= 4 || !(ci.y & 1)) ? 1u : 0u);
                tc_commit(&v_done[b]);
                return true;
            };
            for (uint32_t k = 0;; ++k) {
                const uint32_t b = k & 1u;
                if (!mbar_wait_bounded(&a_ready[b], (k >> 1) & 1u, kTcWaitPolls)) {
                    ok = false;
                    break;
                }
                const int4 ci = cinfo[b];   // x: item_seq, y: bit 0 item's first chunk, bit 1 item's last, bit 2 end
                if (ci.y & 4) {
                    if (pend_v) ok = issue_v(k - 1, prev);
                    break;
                }
                if (ci.x != cur_seq) {
                    cur_seq = ci.x;
                    if (!mbar_wait_bounded(&bk_full[cur_seq & 1], (cur_seq >> 1) & 1, kTcWaitPolls)) {
                        ok = false;
                        break;
                    }
                }
                if (k >= 2 && !mbar_wait_bounded(&dk_free[b], ((k >> 1) - 1) & 1u, kTcWaitPolls)) {
                    ok = false;   // the softmax warps still read D_K of chunk k - 2
                    break;
                }
                tc_fence_after();
                {   // logits: eight k-steps of 16 stored positions, the two of block blk
                    // into that block's accumulator (columns: three parts of q' x heads)
                    const uint32_t bk = smem_u32(smem + SM::kBK + (cur_seq & 1) * kTcKImg);
#pragma unroll
                    for (int j = 0; j < 2; ++j)
#pragma unroll
                        for (int blk = 0; blk < 4; ++blk) {
                            const int ks = 2 * blk + j;
                            tc_mma(tb + kTmDK + 64 * b + 16 * blk, tb + kTmAK + 64 * b + 8 * ks,
                                   smem_desc(bk + kTcKStep * ks, 128, 256), idesc_bf16(16), (uint32_t)j);
                        }
                    tc_commit(&dk_ready[b]);
                    if (ci.y & 2) tc_commit(&bk_free[cur_seq & 1]);
                }
                if (pend_v && !(ok = issue_v(k - 1, prev))) break;
                pend_v = true;
                prev = ci;
            }
            if (!ok) report(p.status, OSCAR_STATUS_TIMEOUT);
            // every MMA issued so far has completed before the tensor memory is freed
            tc_commit(idle);
            (void)mbar_wait_bounded(idle, 0, kTcWaitPolls);
        }
        __syncwarp();
    } else if (warp < kTcSoftWarp0) {
        // ------------------------------ unpack ------------------------------
        const int wq = warp & 3;
        const int t = 32 * wq + lane;                      // token of the chunk (K), stored position (V)
        const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
        bool ok = true;
        for (uint32_t k = 0;; ++k) {
            const uint32_t b = k & 1u;
            const uint32_t n0 = 2 * k, s0 = n0 % NS, s1 = (n0 + 1) % NS, ph = (n0 / NS) & 1u;
            bool w = mbar_wait_bounded(&full[s0], ph, kTcWaitPolls) && mbar_wait_bounded(&full[s1], ph, kTcWaitPolls);
            if (!__all_sync(kFull, w)) {
                ok = false;
                break;
            }
            const int4 i0 = *reinterpret_cast<const int4*>(&info[s0]);
            if (i0.x < 0) {   // end of the stream
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&empty[s0]);
                    mbar_arrive(&empty[s1]);
                }
                if (t == 0) cinfo[b] = make_int4(0, 4, 0, 0);
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_ready[b]);
                break;
            }
            const int flags = i0.w >> 8, seq = info[s0].item_seq;
            const uint8_t* blk0 = stages + s0 * kBlock;
            const uint8_t* blk1 = stages + s1 * kBlock;
            // -- K codes of token t -> A_K row t (column 16b + 2i + s: word i of the token's
            //    32 code bytes, slot b, bytes 0, 2 (s = 0) or 1, 3 (s = 1))
            if (k >= 2) {   // the logit MMAs of chunk k - 2 have read A_K
                const bool wk = mbar_wait_bounded(&dk_ready[b], ((k >> 1) - 1) & 1u, kTcWaitPolls);
                if (!__all_sync(kFull, wk)) {
                    ok = false;
                    break;
                }
            }
            {
                const uint8_t* kc = ((t >> 6) ? blk1 : blk0) + kKCodes + (t & 63) * 32;
                const uint4 c0 = *reinterpret_cast<const uint4*>(kc);
                const uint4 c1 = *reinterpret_cast<const uint4*>(kc + 16);
                const uint32_t wd[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                uint32_t wd8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) wd8[i] = wd[i] >> 8;
#pragma unroll
                for (int half = 0; half < 2; ++half) {   // blocks 2 half, 2 half + 1 -> 32 columns
                    uint32_t a[32];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
#pragma unroll
                        for (int bb = 0; bb < 2; ++bb) {
                            const uint32_t mask = 0x00030003u << (2 * (2 * half + bb));
                            a[16 * bb + 2 * i] = wd[i] & mask;
                            a[16 * bb + 2 * i + 1] = wd8[i] & mask;
                        }
                    tm_st32(tb + lane_off + kTmAK + 64 * b + 32 * half, a);
                }
            }
            // -- V codes of stored position t (slot wq of plane lane) -> A_V row t (column 2u + s:
            //    word u of the chunk's 128 tokens, bytes 0, 2 (s = 0) or 1, 3 (s = 1))
            if (k >= 2) {   // the value MMAs of chunk k - 2 have read A_V
                const bool wv = mbar_wait_bounded(&v_done[b], ((k >> 1) - 1) & 1u, kTcWaitPolls);
                if (!__all_sync(kFull, wv)) {
                    ok = false;
                    break;
                }
            }
            {
                const uint32_t mask = 0x00030003u << (2 * wq);
#pragma unroll
                for (int pgv = 0; pgv < 2; ++pgv) {
                    const uint8_t* pl = (pgv ? blk1 : blk0) + kVCodes + lane * kPage;
                    uint32_t a[32];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const uint4 v = *reinterpret_cast<const uint4*>(pl + 16 * q4);
                        const uint32_t wv4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            a[2 * (4 * q4 + e)] = wv4[e] & mask;
                            a[2 * (4 * q4 + e) + 1] = (wv4[e] >> 8) & mask;
                        }
                    }
                    tm_st32(tb + lane_off + kTmAV + 64 * b + 32 * pgv, a);
                }
            }
            tm_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[s0]);   // the codes are no longer read
                mbar_arrive(&empty[s1]);
            }
            if (t == 0) cinfo[b] = make_int4(seq, ((flags & kTcFirst) ? 1 : 0) | ((flags & kTcLast) ? 2 : 0), 0, 0);
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_ready[b]);
        }
        if (!ok && lane == 0) report(p.status, OSCAR_STATUS_TIMEOUT);
    } else {
        // ------------------------------ softmax ------------------------------
        const int wq = warp & 3;
        const int t = 32 * wq + lane;                      // token of the chunk; stored position for D_V
        const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
        // bounded rendezvous and any-vote of the four softmax warps (mbarriers,
        // so that a warp that gave up on a wait cannot leave the others stuck)
        uint32_t gph = 0, gaph = 0;
        auto gsync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(grp_mb);
            const bool w = mbar_wait_bounded(grp_mb, gph & 1u, kTcWaitPolls);
            ++gph;
            return __all_sync(kFull, w);
        };
        auto gany = [&](bool pred, bool& res) -> bool {
            const bool wa = __any_sync(kFull, pred);
            const int slot = (int)(gaph % 3u);
            if (t == 0) any_flag[(gaph + 1) % 3u] = 0;   // the next call's flag, last read two calls ago
            if (lane == 0 && wa) any_flag[slot] = 1;
            __syncwarp();
            if (lane == 0) mbar_arrive(any_mb);
            const bool w = mbar_wait_bounded(any_mb, gaph & 1u, kTcWaitPolls);
            ++gaph;
            res = *reinterpret_cast<volatile int*>(any_flag + slot) != 0;
            return __all_sync(kFull, w);
        };
        float* red_max = reinterpret_cast<float*>(smem + SM::kRedMax);
        float* red_sum = reinterpret_cast<float*>(smem + SM::kRedSum);
        float Q[4][4];                                     // item constants: sum of q' per (block, head)
        float m_ref[4], l[4], zacc[4][4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            m_ref[h] = -INFINITY;
            l[h] = 0.f;
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) zacc[h][bb] = Q[bb][h] = 0.f;
        }
        bool ok = true;
        for (uint32_t k = 0;; ++k) {
            const uint32_t b = k & 1u;
            const uint32_t n0 = 2 * k, s0 = n0 % NS, s1 = (n0 + 1) % NS, ph = (n0 / NS) & 1u;
            bool w = mbar_wait_bounded(&full[s0], ph, kTcWaitPolls) && mbar_wait_bounded(&full[s1], ph, kTcWaitPolls);
            if (!__all_sync(kFull, w)) {
                ok = false;
                break;
            }
            const int4 i0 = *reinterpret_cast<const int4*>(&info[s0]);
            const int vf1 = info[s1].valid_flags;
            if (i0.x < 0) {   // end of the stream
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&empty[s0]);
                    mbar_arrive(&empty[s1]);
                }
                break;
            }
            const int item = i0.x, flags = i0.w >> 8;
            const int valid0 = (flags & kTcPadPage) ? 0 : (i0.w & 0xff);
            const int valid1 = ((vf1 >> 8) & kTcPadPage) ? 0 : (vf1 & 0xff);
            const bool first = (flags & kTcFirst) != 0;
            if (first) {   // a new item: its constants and a fresh state
                const int bkv = i0.y * p.hk + i0.z;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float4 qs = *reinterpret_cast<const float4*>(p.qsum + ((size_t)bkv * 4 + h) * 4);
                    Q[0][h] = qs.x;
                    Q[1][h] = qs.y;
                    Q[2][h] = qs.z;
                    Q[3][h] = qs.w;
                    m_ref[h] = -INFINITY;
                    l[h] = 0.f;
#pragma unroll
                    for (int bb = 0; bb < 4; ++bb) zacc[h][bb] = 0.f;
                }
            }
            // -- scales of token t (read from the stage before the logits arrive)
            const int r = t & 63;
            const uint8_t* tblk = stages + ((t >> 6) ? s1 : s0) * kBlock;
            const bool tok_ok = r < ((t >> 6) ? valid1 : valid0);
            float sK[4], zK[4], sV[4], zV[4];
            switch (p.gshift) {
                case 0: tc_token_scales<0>(tblk, r, tok_ok, sK, zK, sV, zV); break;
                case 1: tc_token_scales<1>(tblk, r, tok_ok, sK, zK, sV, zV); break;
                default: tc_token_scales<2>(tblk, r, tok_ok, sK, zK, sV, zV); break;
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[s0]);   // the scale rows are no longer read
                mbar_arrive(&empty[s1]);
            }
            // -- logits of token t (base 2) from D_K
            {
                const bool wk = mbar_wait_bounded(&dk_ready[b], (k >> 1) & 1u, kTcWaitPolls);
                if (!__all_sync(kFull, wk)) {
                    ok = false;
                    break;
                }
            }
            tc_fence_after();
            float lg[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {   // block bb: columns 4 part + head
                float dk[16];
                tm_ld16(tb + lane_off + kTmDK + 64 * b + 16 * bb, dk);
#pragma unroll
                for (int h = 0; h < 4; ++h)
                    lg[h] = fmaf(sK[bb], (dk[h] + dk[4 + h]) + dk[8 + h], fmaf(zK[bb], Q[bb][h], lg[h]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&dk_free[b]);
#pragma unroll
            for (int h = 0; h < 4; ++h) lg[h] = tok_ok ? lg[h] : -INFINITY;
            // -- lazy online softmax: the reference maximum moves only when a
            //    logit of the chunk exceeds it by kTcTau
            const bool need = lg[0] > m_ref[0] + kTcTau || lg[1] > m_ref[1] + kTcTau || lg[2] > m_ref[2] + kTcTau ||
                              lg[3] > m_ref[3] + kTcTau;
            bool any_need = false;
            if (!gany(need, any_need)) {
                ok = false;
                break;
            }
            if (any_need) {
                float mx[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    mx[h] = lg[h];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], o));
                }
                if (lane == 0)
                    *reinterpret_cast<float4*>(red_max + 4 * wq) = make_float4(mx[0], mx[1], mx[2], mx[3]);
                if (!gsync()) {
                    ok = false;
                    break;
                }
                float alpha[4];
                bool rescale = false;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    float M = m_ref[h];
#pragma unroll
                    for (int ww = 0; ww < 4; ++ww) M = fmaxf(M, red_max[4 * ww + h]);
                    alpha[h] = (m_ref[h] == -INFINITY) ? 0.f : ex2(m_ref[h] - M);
                    rescale |= (m_ref[h] != -INFINITY) && (M > m_ref[h]);
                    m_ref[h] = M;
                    l[h] *= alpha[h];
#pragma unroll
                    for (int bb = 0; bb < 4; ++bb) zacc[h][bb] *= alpha[h];
                }
                if (!gsync()) {   // the maxima are read before the next chunk writes them
                    ok = false;
                    break;
                }
                if (rescale && !first) {
                    // the accumulator holds the item's earlier chunks: rescale it once
                    // the value MMAs of chunk k - 1 (and so of all earlier chunks) completed
                    const bool wv = mbar_wait_bounded(&v_done[(k - 1) & 1u], ((k - 1) >> 1) & 1u, kTcWaitPolls);
                    if (!__all_sync(kFull, wv)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // only the columns of the thread's own block are ever read
                    const uint32_t dv = tb + lane_off + kTmDV + 8 * wq;
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) {
                        float v[8];
                        tm_ld8(dv + 32 * e4, v);
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] *= alpha[(e >> 1) & 3];
                        tm_st8(dv + 32 * e4, v);
                    }
                    tm_wait_st();
                }
            }
            float pr[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                pr[h] = (m_ref[h] == -INFINITY) ? 0.f : ex2(lg[h] - m_ref[h]);
                l[h] += pr[h];
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) zacc[h][bb] = fmaf(pr[h], zV[bb], zacc[h][bb]);
            }
            // -- P.V weights of token t: B_V row tc_vrow(t), columns (block, head, part)
            if (k >= 2) {   // the value MMAs of chunk k - 2 have read B_V
                const bool wv = mbar_wait_bounded(&v_done[b], ((k >> 1) - 1) & 1u, kTcWaitPolls);
                if (!__all_sync(kFull, wv)) {
                    ok = false;
                    break;
                }
            }
            {
                const int kr = tc_vrow(t);
                uint8_t* bv = smem + SM::kBV + b * 8192 + (kr & 7) * 16 + (kr >> 3) * 128;
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) {
                    uint32_t wv[4];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float x = pr[h] * sV[bb];
                        const float hi = __uint_as_float(__float_as_uint(x) & 0xffff0000u);
                        wv[h] = pack_bf16x2_rn(hi, x - hi);   // (high part, rounded remainder)
                    }
                    *reinterpret_cast<uint4*>(bv + bb * 2048) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&w_ready[b]);

            // -- the item's last chunk: its partial (o', m, l)
            if (flags & kTcLast) {
                const bool wv = mbar_wait_bounded(&v_done[b], (k >> 1) & 1u, kTcWaitPolls);
                if (!__all_sync(kFull, wv)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float dv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {   // the four accumulators; stored position t is in block wq
                    float d4[8];
                    tm_ld8(tb + lane_off + kTmDV + 32 * e4 + 8 * wq, d4);
#pragma unroll
                    for (int e = 0; e < 8; ++e) dv[e] += d4[e];
                }
                tc_fence_before();
                // sums of p and p z over the chunk tokens of all four warps
                float v[20];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    v[h] = l[h];
#pragma unroll
                    for (int bb = 0; bb < 4; ++bb) v[4 + 4 * h + bb] = zacc[h][bb];
                }
#pragma unroll
                for (int i = 0; i < 20; ++i)
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v[i] += __shfl_xor_sync(kFull, v[i], o);
                if (lane < 20) {
                    float x = v[0];
#pragma unroll
                    for (int i = 1; i < 20; ++i) x = (lane == i) ? v[i] : x;
                    red_sum[20 * wq + lane] = x;
                }
                if (!gsync()) {
                    ok = false;
                    break;
                }
                float L[4], Z[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    L[h] = red_sum[h] + red_sum[20 + h] + red_sum[40 + h] + red_sum[60 + h];
                    const int zi = 4 + 4 * h + wq;
                    Z[h] = red_sum[zi] + red_sum[20 + zi] + red_sum[40 + zi] + red_sum[60 + zi];
                }
                if (!gsync()) {   // sums read before the next item end writes them
                    ok = false;
                    break;
                }
                float* part = p.part + (size_t)item * p.part_stride;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    if (h < p.G) {
                        part[(size_t)h * kD + t] = fmaf(dv[2 * h] + dv[2 * h + 1], kTcVOut, Z[h]);
                        if (t == 0) {
                            part[(size_t)p.G * kD + h] = m_ref[h];
                            part[(size_t)p.G * kD + p.G + h] = L[h];
                        }
                    }
                }
            }
        }
        if (!ok && lane == 0) report(p.status, OSCAR_STATUS_TIMEOUT);
    }

    // teardown: every warp arrives here (all waits are bounded); the MMA
    // warp has seen its MMAs complete, the producer its copies land
    tc_fence_before();
    __syncthreads();
    if (warp == kTcMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tb), "r"(kTmCols));
    }
}

cudaError_t launch_int2_tc(const DecodeParams& p, cudaStream_t st, int sms) {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!attr_set[dev & 63]) {
        e = cudaFuncSetAttribute(int2_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem::kBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev & 63] = true;
    }
    const int64_t max_items =
        (int64_t)p.B * p.hk * ((p.max_pages + p.pps - 1) / p.pps + p.tail_pg / kShortItemPages);
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>(sms, max_items));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = TcSmem::kBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, int2_tc_kernel, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace oscar
