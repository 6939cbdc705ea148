// Tensor-core prefill path: W4A16 / W8A16 GEMM on tcgen05 (sm_103a).
//
// y[s,o] = scale[o] * sum_k deq(W[o,k]) * bf16(x[s,k])
//
// The colibri CUDA docs ("The GPU-resident pipeline" section) describe a
// Tensor-Core int4 x 16-bit dispatch for batched rows that pays from 16 rows;
// this is that contraction built for the 5th-generation tensor cores.
//
// 1. A pre-pass converts x (f32 [S, I]) to bf16 (round to nearest even) into a
//    stream-ordered workspace [S, k_pad], zero past I.  For int4 the eight
//    elements of every 8-group are stored in the order 0,4,1,5,2,6,3,7, the
//    order in which the dequantizer below produces them (the contraction
//    index may be permuted freely as long as both operands agree).
// 2. The GEMM, D[o, s] = sum_k A[o, k] B[s, k], M = weight rows (A = the
//    dequantized weights, K-major), N = tokens (B = x, K-major), K = I.
//    Persistent CTAs walk 128 x 176 output tiles (176 = 11 * 16 splits 1571
//    tokens into 9 tiles with 0.8% padding).  Warp roles:
//      warp 0     TMA producer: per 64-wide k-block, one 2-D load of the
//                 128-row code tile and one of the 176 x 64 bf16 x tile
//                 (128-byte swizzle), completion on an mbarrier;
//      warps 2-9  dequantizers, two threads per weight row (each half of
//                 the row's k-block): codes -> exact bf16 (int4: OR the
//                 nibble into the mantissa of 128.0 and subtract 136; int8:
//                 exact via f32), stored with tcgen05.st into one of four
//                 A buffers in tensor memory (lane = weight row, 32 columns
//                 = the k-block's 64 bf16); a warp owns the rows of its
//                 lane quarter (warp % 4).  With A out of shared memory a
//                 stage holds only codes and x, so the ring is 8 deep;
//      warp 1     MMA issuer (one thread): 4 x tcgen05.mma (kind::f16,
//                 bf16 in, f32 accumulate, 128 x 176 x 16, A from tensor
//                 memory) per k-block into one of two TMEM accumulators;
//                 tcgen05.commit releases the stage and the A buffer and,
//                 after the last k-block, hands the tile to ...
//      warps 10-13 epilogue: tcgen05.ld of its 32 TMEM lanes, times scale[o],
//                 coalesced f32 stores of y (32 consecutive o per store).
//    Integer codes are exact in bf16 and products are exact in f32, so the
//    only approximation is x's rounding to bf16 plus f32 accumulation.
// Every mbarrier wait is bounded; a wait that gives up records
// B200Q_ETIMEOUT (b200q_device_status) and the CTA winds down, draining its
// copies and freeing its TMEM.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstring>
#include <mutex>

#include "qwq_internal.h"

namespace qwq {
namespace {

constexpr int BM = 128, BN = 176, BK = 64;
// Pipeline stages (code tile + x tile; 26.5 KB for int4 at 176 tokens): as
// many as fit in 227 KB of shared memory, at most 10, since the stage ring has
// to cover a TMA round trip plus dequantization.  The dequantized A tile of a
// k-block (128 rows x 64 bf16) lives in tensor memory, in a ring of its own.
// Group-scale tile of a stage when the producer copies the scales (GSM = 2):
// 128 rows x 4 f32 from a 4-aligned first group.
constexpr int kScaleBox = 4;
constexpr int kScaleTile = BM * kScaleBox * 4;      // 2 KB

template <int FMT, int BNT, int GSM = 0>
constexpr int stages_for() {
    constexpr int per = BNT * BK * 2 + BM * (FMT == B200Q_I4 ? 32 : 64) + (GSM == 2 ? kScaleTile : 0);
    constexpr int n = (232448 - 1024 - 512) / per;
    return n > 10 ? 10 : n;
}
constexpr int kDeqWarps = 8;         // per group of dequantizing warps
// Groups of dequantizing warps (on alternate k-blocks): two where the
// dequantization carries group scales (measured +8 % at gs = 128), one with
// per-row scales (measured 2 % slower with two).
constexpr int deq_groups(int gsm) { return gsm ? 2 : 1; }
constexpr int threads_for(int gsm) { return (2 + deq_groups(gsm) * kDeqWarps + 4) * 32; }
// Tensor memory: kNumA A buffers of 32 columns (a k-block of 64 bf16 per
// lane = weight row) at columns 0.., then two accumulators of up to 192
// columns.
constexpr int kTmemCols = 512;
constexpr int kNumA = 4;
constexpr int kAccBase = kNumA * 32;   // 128
constexpr int kAccStride = 192;
constexpr unsigned long long kWaitNs = 2000000000ull;

__device__ unsigned int g_prefill_err = 0;

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    unsigned long long t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if (it == 0) t0 = global_ns();
        if ((it & 255) == 255 && global_ns() - t0 > kWaitNs) {
            atomicExch(&g_prefill_err, (unsigned)(-B200Q_ETIMEOUT));
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);      // start address
    d |= (uint64_t)1 << 16;                        // leading-dimension byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;              // stride-dimension byte offset
    d |= (uint64_t)1 << 46;                        // descriptor version
    d |= (uint64_t)2 << 61;                        // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: D f32, A and B bf16, both K-major,
// M = 128, N = bnt.
constexpr uint32_t idesc_for(int bnt) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(bnt >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

// D (tensor memory) += A (tensor memory, 128 lanes x 16 bf16) x B (shared memory)
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t magic) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(magic));
    return r;
}

__device__ __forceinline__ uint32_t bsub2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// One int4 code word (8 nibbles, k = 8m..8m+7) -> 8 exact bf16 in the order
// 0,4,1,5,2,6,3,7: 0x4300 | c is 128 + c in bf16, minus 136 is c - 8.
__device__ __forceinline__ uint4 deq_i4_word(uint32_t w) {
    uint4 o;
    o.x = bsub2(lop3_and_or(w, 0x000F000Fu, 0x43004300u), 0x43084308u);
    o.y = bsub2(lop3_and_or(w >> 4, 0x000F000Fu, 0x43004300u), 0x43084308u);
    o.z = bsub2(lop3_and_or(w >> 8, 0x000F000Fu, 0x43004300u), 0x43084308u);
    o.w = bsub2(lop3_and_or(w >> 12, 0x000F000Fu, 0x43004300u), 0x43084308u);
    return o;
}

// One int8 code word (4 bytes) -> 4 exact bf16 in natural order, through f32:
// the byte with its sign bit flipped is u = code + 128; 0x4B000000 | u is
// 2^23 + u, minus (2^23 + 128) is the code.
__device__ __forceinline__ uint2 deq_i8_word(uint32_t w) {
    const uint32_t u = w ^ 0x80808080u;
    const float f0 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - 8388736.0f;
    const float f1 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - 8388736.0f;
    const float f2 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - 8388736.0f;
    const float f3 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - 8388736.0f;
    return make_uint2(pack_bf16(f0, f1), pack_bf16(f2, f3));
}

// Group-wise scales.  The group scale s is split into bf16 parts s_hi =
// bf16(s), s_lo = bf16(s - s_hi) (together s to ~2^-17); a pair of exact bf16
// codes c becomes fma(c, s_hi, bf16(c * s_lo)), rounded once: the product
// c * s_hi is exact inside the FMA and the correction term carries an error
// of at most 2^-17 |c s|, so each weight is c * s rounded to bf16 (relative
// error 2^-9 + 2^-16), like the bf16 rounding of x.
struct ScalePair {
    uint32_t hi, lo;   // (s_hi, s_hi) and (s_lo, s_lo) as bf16x2
};

__device__ __forceinline__ ScalePair split_scale(float s) {
    const uint32_t h = pack_bf16(s, s);
    const float sh = __uint_as_float(h << 16);
    const float sl = s - sh;                        // exact in f32
    return ScalePair{h, pack_bf16(sl, sl)};
}

__device__ __forceinline__ uint32_t scale_pair(uint32_t b2, const ScalePair &sp) {
    uint32_t t, r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(t) : "r"(b2), "r"(sp.lo));
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(b2), "r"(sp.hi), "r"(t));
    return r;
}

__device__ __forceinline__ uint4 scale_word4(uint4 e, const ScalePair &sp) {
    return make_uint4(scale_pair(e.x, sp), scale_pair(e.y, sp), scale_pair(e.z, sp), scale_pair(e.w, sp));
}

// Division by the group size as a multiply and a shift (exact for
// 0 <= n < 2^31): m = ceil(2^(31+c) / gs), c = ceil(log2 gs).
struct GroupDiv {
    uint32_t m;
    int sh;
};

__device__ __forceinline__ int group_of(int n, const GroupDiv &d) {
    return (int)(((unsigned long long)(unsigned)n * d.m) >> d.sh);
}

struct GemmParams {
    const float *scales;
    const float2 *unscale;   // x pieces: per token, 2^-k as two exact factors
    float *y;
    int O, S;
    int m_tiles, n_tiles, nk;
    int code_bytes;      // bytes of one code tile row per k-block (32 int4, 64 int8)
    int g_ld;            // group-wise scales: row stride of scales (floats)
    int g_last;          // last group index a padded column may reach (clamp)
    int g_one;           // a thread's 32 columns of a k-block lie in one group (gs % 32 == 0)
    GroupDiv gdiv;       // by the group size
    int ksplit;          // > 1: CTA b takes tile b / ksplit over part (b % ksplit) of the k-blocks and
                         // writes its partial result to plane (b % ksplit) of y ([ksplit][S][O])
};

// BNT: columns of the B tile (tokens, or x pieces).  PIECES: B holds three
// bf16 pieces per token (rows 3s, 3s+1, 3s+2, summing to x exactly) and the
// epilogue adds each token's three columns.  GSM: 0 per-row scales; 1 / 2
// group-wise scales, which the dequantizers load themselves (1) or find in
// the stage, copied by the producer with the code tile (2: a k-block's groups
// lie within 4 floats from a 4-aligned first group).  Group-wise scales, applied
// by the dequantizers (A = bf16((code - zero point) * scale[o, group]), one
// rounding per weight, see scale_pair); the epilogue then applies no row
// scale.  An int4
// code word (8 columns) or an int8 16-byte chunk (16 columns) always lies in
// one group (gs is a multiple of 16 for int8, of 16 or 32 for int4).
template <int FMT, int BNT, bool PIECES, int GSM = 0>
__global__ void __launch_bounds__(threads_for(GSM), 1)
    qgemm_tc_kernel(const __grid_constant__ CUtensorMap map_codes, const __grid_constant__ CUtensorMap map_x,
                    const __grid_constant__ CUtensorMap map_sc, const GemmParams p) {
    constexpr bool GS = GSM != 0;
    constexpr int kDeqGroups = deq_groups(GSM);
    constexpr int kStages = stages_for<FMT, BNT, GSM>();
    constexpr uint32_t kIdesc = idesc_for(BNT);
    static_assert(BNT % 16 == 0 && BNT >= 16 && BNT <= kAccStride && (!PIECES || BNT <= 48), "token tile");
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled operand tiles
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    constexpr int B_BYTES = BNT * BK * 2;
    constexpr int C_BYTES = BM * (FMT == B200Q_I4 ? 32 : 64);
    uint8_t *b_s = smem;                                 // [kStages][B_BYTES]
    uint8_t *c_s = b_s + kStages * B_BYTES;              // [kStages][C_BYTES]
    constexpr int S_BYTES = GSM == 2 ? kScaleTile : 0;
    uint8_t *s_s = c_s + kStages * C_BYTES;              // [kStages][BM][kScaleBox] f32 (GSM = 2)
    uint64_t *bars = reinterpret_cast<uint64_t *>(s_s + kStages * S_BYTES);
    uint64_t *tma_full = bars, *empty = bars + kStages;
    uint64_t *a_full = bars + 2 * kStages, *a_empty = a_full + kNumA;   // tensor-memory A ring
    uint64_t *acc_full = a_empty + kNumA, *acc_empty = acc_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles_total = p.m_tiles * p.n_tiles;
    // this CTA's work, walked identically by every warp role: persistent over
    // tiles (each over all k-blocks), or with ksplit > 1 one tile over a
    // contiguous part of its k-blocks
    const bool split = PIECES && p.ksplit > 1;         // only the three-piece path splits (compile-time off otherwise)
    const int t_first = split ? (int)blockIdx.x / p.ksplit : (int)blockIdx.x;
    const int t_step = split ? n_tiles_total : (int)gridDim.x;
    const int kb0 = split ? ((int)blockIdx.x % p.ksplit) * p.nk / p.ksplit : 0;
    const int kb1 = split ? ((int)blockIdx.x % p.ksplit + 1) * p.nk / p.ksplit : p.nk;
    // Loop heads of every role.  Variants that cannot split use blockIdx /
    // gridDim / p.nk directly (unsigned stepping, as written before splitting
    // existed): the compiler then schedules them ~5% faster.
#define QWQ_TILE_FIRST (PIECES ? (unsigned)t_first : blockIdx.x)
#define QWQ_TILE_STEP (PIECES ? (unsigned)t_step : gridDim.x)
#define QWQ_KB_FIRST (PIECES ? kb0 : 0)
#define QWQ_KB_END (PIECES ? kb1 : p.nk)

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&tma_full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int s = 0; s < kNumA; ++s) {
            mbar_init(smem_u32(&a_full[s]), kDeqWarps);
            mbar_init(smem_u32(&a_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), 4);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int tile = QWQ_TILE_FIRST; tile < n_tiles_total && ok; tile += QWQ_TILE_STEP) {
                const int m0 = (tile / p.n_tiles) * BM, n0 = (tile % p.n_tiles) * BNT;
                for (int kb = QWQ_KB_FIRST; kb < QWQ_KB_END; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bar = smem_u32(&tma_full[stage]);
                    mbar_expect_tx(bar, (uint32_t)(C_BYTES + B_BYTES + S_BYTES));
                    tma_load_2d(smem_u32(c_s + stage * C_BYTES), &map_codes, kb * p.code_bytes, m0, bar);
                    tma_load_2d(smem_u32(b_s + stage * B_BYTES), &map_x, kb * BK, n0, bar);
                    if (GSM == 2)   // the k-block's group scales, from its first group rounded down to 16 bytes
                        tma_load_2d(smem_u32(s_s + stage * S_BYTES), &map_sc, group_of(kb * BK, p.gdiv) & ~3, m0,
                                    bar);
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // the copies of the last kStages loads must land before the CTA
            // may leave (earlier ones were consumed before their stage was
            // refilled); a phase that already completed returns at once
            for (long long i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i)
                mbar_wait(smem_u32(&tma_full[i % kStages]), (uint32_t)((i / kStages) & 1));
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            int stage = 0, abuf = 0;
            uint32_t phase = 0, aphase = 0;
            bool ok = true;
            int t = 0;
            for (int tile = QWQ_TILE_FIRST; tile < n_tiles_total && ok; tile += QWQ_TILE_STEP, ++t) {
                const int ab = t & 1;
                if (!mbar_wait(smem_u32(&acc_empty[ab]), ((t >> 1) & 1) ^ 1)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + kAccBase + ab * kAccStride;
                for (int kb = QWQ_KB_FIRST; kb < QWQ_KB_END; ++kb) {
                    // the dequantizers arrive on a_full only after the stage's
                    // copies (codes and the x tile B) have landed
                    if (!mbar_wait(smem_u32(&a_full[abuf]), aphase)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_tmem = tmem_base + abuf * 32;
                    const uint32_t b_addr = smem_u32(b_s + stage * B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        mma_bf16_ts(d_tmem, a_tmem + 8 * k, sw128_desc(b_addr + 32 * k), kIdesc,
                                    (kb > QWQ_KB_FIRST || k > 0) ? 1u : 0u);
                    mma_commit(smem_u32(&empty[stage]));
                    mma_commit(smem_u32(&a_empty[abuf]));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                    if (++abuf == kNumA) {
                        abuf = 0;
                        aphase ^= 1;
                    }
                }
                if (ok) mma_commit(smem_u32(&acc_full[ab]));
            }
        }
    } else if (warp >= 2 && warp < 2 + kDeqGroups * kDeqWarps) {
        // ---------------- dequantizers: thread (r, half) owns half of row r
        // of every A tile (tensor-memory columns 16 half .. 16 half + 15 of an
        // A buffer); a warp reaches only its own lane quarter (warp % 4), so
        // that quarter's 32 rows are its rows
        // With two groups of eight warps, they take alternate k-blocks of
        // the CTA's sequence (the k-th of all its (tile, k-block) steps goes
        // to group k % 2), so two k-blocks are dequantized at once: each step
        // waits on the stage's copy and on the A buffer.
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int grp = (warp - 2) / kDeqWarps;
        const int half = ((warp - 2) % kDeqWarps) >> 2;
        bool ok = true;
        // group-wise scales of the thread's 4 code words (int4) or 2 chunks
        // (int8) of k-block kb, loaded one k-block ahead
        constexpr int kGW = FMT == B200Q_I4 ? 4 : 2;
        constexpr int kGCols = FMT == B200Q_I4 ? 8 : 16;
        float gsn[kGW];
        ScalePair gsc[kGW];
        auto load_gs = [&](int tile, int kb, float(&dst)[kGW]) {
            const long long o = (long long)(tile / p.n_tiles) * BM + r;
            if (p.g_one) {                               // one group for all of the thread's columns
                dst[0] = __ldg(p.scales + o * p.g_ld + min(group_of(kb * BK + 32 * half, p.gdiv), p.g_last));
                return;
            }
#pragma unroll
            for (int i = 0; i < kGW; ++i) {
                const int g = min(group_of(kb * BK + 32 * half + kGCols * i, p.gdiv), p.g_last);
                dst[i] = __ldg(p.scales + o * p.g_ld + g);
            }
        };
        // the step after (tile, kb) in the CTA's sequence
        auto step = [&](int &tl, int &k) {
            if (++k == kb1) {
                k = kb0;
                tl += t_step;
            }
        };
        if (GSM == 1) {   // this group's first step
            int tl = t_first, k = kb0;
            for (int g = 0; g < grp; ++g) step(tl, k);
            if (tl < n_tiles_total) load_gs(tl, k, gsn);
        }
        unsigned seq = 0;                                // step index in the CTA's sequence
        for (int tile = QWQ_TILE_FIRST; tile < n_tiles_total && ok; tile += QWQ_TILE_STEP) {
            for (int kb = QWQ_KB_FIRST; kb < QWQ_KB_END; ++kb, ++seq) {
                if ((int)(seq % kDeqGroups) != grp) continue;
                const int stage = (int)(seq % kStages), abuf = (int)(seq % kNumA);
                const uint32_t phase = (seq / kStages) & 1, aphase = (seq / kNumA) & 1;
                if constexpr (GSM == 1) {
                    if (p.g_one) {
                        const ScalePair sp = split_scale(gsn[0]);
#pragma unroll
                        for (int i = 0; i < kGW; ++i) gsc[i] = sp;
                    } else {
#pragma unroll
                        for (int i = 0; i < kGW; ++i) gsc[i] = split_scale(gsn[i]);
                    }
                    int tl = tile, k = kb;                   // this group's next step
                    for (int g = 0; g < kDeqGroups; ++g) step(tl, k);
                    if (tl < n_tiles_total) load_gs(tl, k, gsn);
                }
                if (!mbar_wait(smem_u32(&tma_full[stage]), phase)) {
                    ok = false;
                    break;
                }
                if constexpr (GSM == 2) {
                    const float *srow = reinterpret_cast<const float *>(s_s + stage * S_BYTES) + r * kScaleBox;
                    const int g0 = group_of(kb * BK, p.gdiv) & ~3;
                    if (p.g_one) {
                        const ScalePair sp = split_scale(srow[group_of(kb * BK + 32 * half, p.gdiv) - g0]);
#pragma unroll
                        for (int i = 0; i < kGW; ++i) gsc[i] = sp;
                    } else {
#pragma unroll
                        for (int i = 0; i < kGW; ++i)
                            gsc[i] = split_scale(srow[group_of(kb * BK + 32 * half + kGCols * i, p.gdiv) - g0]);
                    }
                }
                const uint8_t *crow = c_s + stage * C_BYTES + r * (C_BYTES / BM);
                // the thread's 32 bf16 of the k-block (16 columns) in MMA K order
                uint32_t cols[16];
                if (FMT == B200Q_I4) {
                    const uint4 cw = *reinterpret_cast<const uint4 *>(crow + 16 * half);
                    const uint32_t wv[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint4 e = deq_i4_word(wv[i]);
                        if (GS) e = scale_word4(e, gsc[i]);
                        cols[4 * i] = e.x;
                        cols[4 * i + 1] = e.y;
                        cols[4 * i + 2] = e.z;
                        cols[4 * i + 3] = e.w;
                    }
                } else {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int h = 2 * half + hh;
                        const uint4 cw = *reinterpret_cast<const uint4 *>(crow + 16 * h);
                        const uint2 lo = deq_i8_word(cw.x), hi = deq_i8_word(cw.y);
                        const uint2 lo2 = deq_i8_word(cw.z), hi2 = deq_i8_word(cw.w);
                        uint4 e0 = make_uint4(lo.x, lo.y, hi.x, hi.y), e1 = make_uint4(lo2.x, lo2.y, hi2.x, hi2.y);
                        if (GS) {
                            e0 = scale_word4(e0, gsc[hh]);
                            e1 = scale_word4(e1, gsc[hh]);
                        }
                        cols[8 * hh] = e0.x;
                        cols[8 * hh + 1] = e0.y;
                        cols[8 * hh + 2] = e0.z;
                        cols[8 * hh + 3] = e0.w;
                        cols[8 * hh + 4] = e1.x;
                        cols[8 * hh + 5] = e1.y;
                        cols[8 * hh + 6] = e1.z;
                        cols[8 * hh + 7] = e1.w;
                    }
                }
                // the A buffer comes free when the MMAs that read it complete
                if (!mbar_wait(smem_u32(&a_empty[abuf]), aphase ^ 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_st16(tmem_base + ((uint32_t)(quarter * 32) << 16) + abuf * 32 + half * 16, cols);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&a_full[abuf]));
            }
        }
    } else {
        // ---------------- epilogue: TMEM lanes 32 * (warp % 4) ..
        const int quarter = warp & 3;
        float *yplane = split ? p.y + (long long)((int)blockIdx.x % p.ksplit) * p.S * p.O : p.y;
        int t = 0;
        for (int tile = QWQ_TILE_FIRST; tile < n_tiles_total; tile += QWQ_TILE_STEP, ++t) {
            const int ab = t & 1;
            if (!mbar_wait(smem_u32(&acc_full[ab]), (t >> 1) & 1)) break;
            tc_fence_after();
            const int m0 = (tile / p.n_tiles) * BM, n0 = (tile % p.n_tiles) * BNT;
            const int o = m0 + quarter * 32 + lane;
            const float sc = o < p.O ? (GS ? 1.f : p.scales[o]) : 0.f;
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + kAccBase + ab * kAccStride;
            if constexpr (PIECES) {
                float v[BNT];
#pragma unroll
                for (int c = 0; c < BNT / 16; ++c) {
                    float w16[16];
                    tmem_ld16(taddr + c * 16, w16);
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[c * 16 + j] = w16[j];
                }
                if (o < p.O) {
#pragma unroll
                    for (int s3 = 0; s3 < BNT / 3; ++s3)
                        if (s3 < p.S) {
                            const float2 u = p.unscale[s3];
                            if (split) {   // still in the pieces' scaled units; unscaled after the planes are added
                                yplane[(long long)s3 * p.O + o] = ((v[3 * s3] + v[3 * s3 + 1]) + v[3 * s3 + 2]) * sc;
                            } else {
                                const float dot = (((v[3 * s3] + v[3 * s3 + 1]) + v[3 * s3 + 2]) * u.x) * u.y;   // exact scaling
                                yplane[(long long)s3 * p.O + o] = dot * sc;
                            }
                        }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BNT / 16; ++c) {
                    float v[16];
                    tmem_ld16(taddr + c * 16, v);
                    const int s0 = n0 + c * 16;
                    if (o < p.O) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (s0 + j < p.S) yplane[(long long)(s0 + j) * p.O + o] = v[j] * sc;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acc_empty[ab]));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
#undef QWQ_TILE_FIRST
#undef QWQ_TILE_STEP
#undef QWQ_KB_FIRST
#undef QWQ_KB_END
}

// x f32 [S, I] -> bf16 [S, k_pad] (RNE, zero past I); int4 tensors get each
// 8-group in the order 0,4,1,5,2,6,3,7.
__global__ void x_to_bf16_kernel(const float *__restrict__ x, __nv_bfloat16 *__restrict__ xb, int S, int I,
                                 int k_pad, int permute8) {
    const long long total = (long long)S * k_pad / 8;
    for (long long g8 = (long long)blockIdx.x * blockDim.x + threadIdx.x; g8 < total;
         g8 += (long long)gridDim.x * blockDim.x) {
        const long long s = g8 / (k_pad / 8);
        const int k0 = (int)(g8 - s * (k_pad / 8)) * 8;
        const float *xr = x + s * I;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = (k0 + i < I) ? xr[k0 + i] : 0.f;
        uint4 o;
        if (permute8) {
            o.x = pack_bf16(v[0], v[4]);
            o.y = pack_bf16(v[1], v[5]);
            o.z = pack_bf16(v[2], v[6]);
            o.w = pack_bf16(v[3], v[7]);
        } else {
            o.x = pack_bf16(v[0], v[1]);
            o.y = pack_bf16(v[2], v[3]);
            o.z = pack_bf16(v[4], v[5]);
            o.w = pack_bf16(v[6], v[7]);
        }
        reinterpret_cast<uint4 *>(xb + s * k_pad)[k0 / 8] = o;
    }
}

// 2^k exactly for -149 <= k <= 127 (from the bits).
__device__ __forceinline__ float pow2_bits(int k) {
    return k >= -126 ? __int_as_float((k + 127) << 23) : __int_as_float(1 << (k + 149));
}

// x f32 [S, I] -> exact three-piece bf16 split, one block per token.  The
// row is first scaled by 2^k (k from its largest |x|, so the scaled row lies
// below 2 in magnitude; two factors when k > 127): with v = x 2^k,
// p0 = RN(v), p1 = RN(v - p0), p2 = v - p0 - p1, where both subtractions are
// exact (operands within a factor of two) and p2 has at most 8 significant
// bits, so p0 + p1 + p2 = v exactly.  Rows 3s, 3s+1, 3s+2 of xb [rows, k_pad]
// receive the pieces (int4 tensors: each 8-group in the order
// 0,4,1,5,2,6,3,7), unscale[s] = 2^-k as two factors; block S zeroes rows
// 3S .. rows-1.
constexpr int kPieceThreads = 512;
constexpr int kPieceGroups = 2;          // 8-groups per thread kept in registers

__global__ void __launch_bounds__(kPieceThreads)
    x_to_pieces_kernel(const float *__restrict__ x, __nv_bfloat16 *__restrict__ xb, float2 *__restrict__ unscale,
                       int S, int I, int k_pad, int rows, int permute8) {
    const int groups = k_pad / 8;
    const int tid = threadIdx.x;
    if ((int)blockIdx.x == S) {
        for (long long g = tid; g < (long long)(rows - 3 * S) * groups; g += kPieceThreads)
            reinterpret_cast<uint4 *>(xb + (long long)3 * S * k_pad)[g] = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    const int s = blockIdx.x;
    const float *xr = x + (long long)s * I;
    auto load8 = [&](int g, float (&v)[8]) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = g * 8 + i < I ? xr[g * 8 + i] : 0.f;
    };
    float held[kPieceGroups][8];
    float m = 0.f;
    for (int base = 0; base < groups; base += kPieceGroups * kPieceThreads) {
#pragma unroll
        for (int j = 0; j < kPieceGroups; ++j) {
            const int g = base + j * kPieceThreads + tid;
            if (g < groups) load8(g, held[j]);
            else
#pragma unroll
                for (int i = 0; i < 8; ++i) held[j][i] = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(held[j][i]));
        }
    }
    __shared__ float red[kPieceThreads / 32];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    m = 0.f;
#pragma unroll
    for (int w = 0; w < kPieceThreads / 32; ++w) m = fmaxf(m, red[w]);
    // k = -floor(log2 m) from the bits (subnormal m included); 0 for a zero row
    int k = 0;
    if (m > 0.f) {
        const int b = __float_as_int(m), e = (b >> 23) & 0xFF;
        k = -(e ? e - 127 : -118 - __clz(b));
    }
    const float s1 = k > 127 ? pow2_bits(64) : 1.f, s2 = pow2_bits(k > 127 ? k - 64 : k);
    const int ku = -k;                                         // 2^-k as u1 * u2
    const float u1 = ku > 127 ? pow2_bits(64) : 1.f, u2 = pow2_bits(ku > 127 ? ku - 64 : ku);
    if (tid == 0) unscale[s] = make_float2(u1, u2);
    __nv_bfloat16 *r0 = xb + (long long)3 * s * k_pad;
    auto emit = [&](int g, const float (&v)[8]) {
        float pc[3][8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float a = (v[i] * s1) * s2;
            const float p0 = __bfloat162float(__float2bfloat16_rn(a));
            const float r1 = a - p0;
            const float p1 = __bfloat162float(__float2bfloat16_rn(r1));
            pc[0][i] = p0;
            pc[1][i] = p1;
            pc[2][i] = r1 - p1;
        }
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            uint4 o;
            if (permute8) {
                o = make_uint4(pack_bf16(pc[j][0], pc[j][4]), pack_bf16(pc[j][1], pc[j][5]),
                               pack_bf16(pc[j][2], pc[j][6]), pack_bf16(pc[j][3], pc[j][7]));
            } else {
                o = make_uint4(pack_bf16(pc[j][0], pc[j][1]), pack_bf16(pc[j][2], pc[j][3]),
                               pack_bf16(pc[j][4], pc[j][5]), pack_bf16(pc[j][6], pc[j][7]));
            }
            reinterpret_cast<uint4 *>(r0 + (long long)j * k_pad)[g] = o;
        }
    };
    if (groups <= kPieceGroups * kPieceThreads) {
#pragma unroll
        for (int j = 0; j < kPieceGroups; ++j) {
            const int g = j * kPieceThreads + tid;
            if (g < groups) emit(g, held[j]);
        }
    } else {
        for (int g = tid; g < groups; g += kPieceThreads) {
            float v[8];
            load8(g, v);
            emit(g, v);
        }
    }
}

cudaMemPool_t g_pool[64] = {};
std::mutex g_pool_mu;

}  // namespace

cudaError_t workspace_alloc(void **ptr, size_t bytes, cudaStream_t st);
cudaError_t workspace_free(void *ptr, cudaStream_t st);

namespace {

cudaError_t get_pool(int dev, cudaMemPool_t *out) {
    std::lock_guard<std::mutex> lk(g_pool_mu);
    if (!g_pool[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaError_t e = cudaMemPoolCreate(&g_pool[dev], &props);
        if (e != cudaSuccess) return e;
        count_workspace_alloc();
        uint64_t keep = ~0ull;   // keep freed workspace cached in the pool
        cudaMemPoolSetAttribute(g_pool[dev], cudaMemPoolAttrReleaseThreshold, &keep);
    }
    *out = g_pool[dev];
    return cudaSuccess;
}

// b_rows: rows of the bf16 B operand (tokens, or the padded pieces rows).
template <int FMT, int BNT, bool PIECES, int GSM = 0>
cudaError_t run_gemm(const Tensor &t, const __nv_bfloat16 *xb, int b_rows, const float2 *unscale, float *y, int S,
                     cudaStream_t st, int ksplit = 1) {
    constexpr bool GS = GSM != 0;
    constexpr int code_bytes = FMT == B200Q_I4 ? 32 : 64;
    // the codes' and group scales' maps were encoded at upload; only x's
    // (a per-call workspace) is encoded here
    CUtensorMap map_x;
    if (!tmap_encode_2d(&map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (void *)xb, (uint64_t)t.k_pad, (uint64_t)b_rows,
                   (uint64_t)t.k_pad * 2, BK, BNT, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    GemmParams p{};
    p.scales = t.scales;
    p.unscale = unscale;
    p.y = y;
    p.O = t.O;
    p.S = S;
    p.m_tiles = t.o_pad / BM;
    p.n_tiles = PIECES ? 1 : (S + BNT - 1) / BNT;
    p.nk = (int)(t.k_pad / BK);
    p.code_bytes = code_bytes;
    p.ksplit = ksplit;
    if (GS) {
        int c = 0;
        while ((1ll << c) < t.gs) ++c;
        p.gdiv = GroupDiv{(uint32_t)(((1ull << (31 + c)) + t.gs - 1) / t.gs), 31 + c};
        p.g_ld = t.G_ld;
        p.g_last = t.G_ld - 1;
        p.g_one = t.gs % 32 == 0;
    }
    constexpr int C_BYTES = BM * code_bytes;
    constexpr int kStages = stages_for<FMT, BNT, GSM>();
    const size_t smem = 1024 + (size_t)kStages * (BNT * BK * 2 + C_BYTES + (GSM == 2 ? kScaleTile : 0)) +
                        (2 * kStages + 2 * kNumA + 4) * 8 + 16;
    cudaError_t e = allow_dynamic_smem((const void *)qgemm_tc_kernel<FMT, BNT, PIECES, GSM>, (int)smem);
    if (e != cudaSuccess) return e;
    const int n_sms = sm_count(t.device);
    const int tiles = p.m_tiles * p.n_tiles;
    const int grid = ksplit > 1 ? tiles * ksplit : tiles < n_sms ? tiles : n_sms;
    qgemm_tc_kernel<FMT, BNT, PIECES, GSM><<<grid, threads_for(GSM), smem, st>>>(t.gemm_map, map_x, t.gemm_sc_map, p);
    count_launch();
    return cudaGetLastError();
}

template <int FMT>
cudaError_t run_gemm_x(const Tensor &t, const __nv_bfloat16 *xb, float *y, int S, cudaStream_t st) {
    if (!t.gs) return run_gemm<FMT, BN, false, 0>(t, xb, S, nullptr, y, S, st);
    // the producer copies the scales when a k-block's groups fit 4 floats
    // from a 4-aligned first group: gs a multiple of 64, or 16 / 32
    const bool boxed = t.gs % BK == 0 || t.gs == 16 || t.gs == 32;
    return boxed ? run_gemm<FMT, BN, false, 2>(t, xb, S, nullptr, y, S, st)
                 : run_gemm<FMT, BN, false, 1>(t, xb, S, nullptr, y, S, st);
}

}  // namespace

cudaError_t launch_prefill_tc(const Tensor &t, const Tensor *tu, const float *x, float *y, float *yu, int S,
                              cudaStream_t st, bool *handled) {
    *handled = false;
    if (t.fmt != B200Q_I4 && t.fmt != B200Q_I8) return cudaSuccess;
    const int n_sms = sm_count(t.device);
    const size_t ws_bytes = (size_t)S * t.k_pad * 2;
    void *ws = nullptr;
    cudaError_t e = workspace_alloc(&ws, ws_bytes, st);
    if (e != cudaSuccess) return e;
    const long long groups = (long long)S * t.k_pad / 8;
    long long blocks = (groups + 255) / 256;
    if (blocks > (long long)n_sms * 16) blocks = (long long)n_sms * 16;
    x_to_bf16_kernel<<<(int)blocks, 256, 0, st>>>(x, (__nv_bfloat16 *)ws, S, t.I, (int)t.k_pad,
                                                   t.fmt == B200Q_I4 ? 1 : 0);
    count_launch();
    e = cudaGetLastError();
    if (e == cudaSuccess)
        e = t.fmt == B200Q_I4 ? run_gemm_x<B200Q_I4>(t, (__nv_bfloat16 *)ws, y, S, st)
                              : run_gemm_x<B200Q_I8>(t, (__nv_bfloat16 *)ws, y, S, st);
    if (e == cudaSuccess && tu)
        e = t.fmt == B200Q_I4 ? run_gemm_x<B200Q_I4>(*tu, (__nv_bfloat16 *)ws, yu, S, st)
                              : run_gemm_x<B200Q_I8>(*tu, (__nv_bfloat16 *)ws, yu, S, st);
    cudaError_t ef = cudaFreeAsync(ws, st);
    if (e == cudaSuccess) e = ef;
    *handled = (e == cudaSuccess);
    return e;
}

// f32-accurate tensor-core path (B200Q_PATH_TCX): x split into three exact
// bf16 pieces, at most 15 tokens (45 piece columns) per GEMM launch.  With tu
// the same pieces serve the second tensor.
// y[s, o] = (sum of the ks planes' partials, in plane order) * 2^-k(s): the
// split k-blocks' partials are kept in the pieces' scaled units so that the
// unscaling (exact powers of two) rounds once, after the sum.
__global__ void sum_planes_kernel(const float *__restrict__ planes, const float2 *__restrict__ unscale,
                                  float *__restrict__ y, long long n, int O, int ks) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        float v = planes[i];
        for (int k = 1; k < ks; ++k) v += planes[(long long)k * n + i];
        const float2 u = unscale[i / O];
        y[i] = (v * u.x) * u.y;
    }
}

template <int FMT>
cudaError_t run_tcx_chunk(const Tensor &t, const Tensor *tu, const __nv_bfloat16 *pc, int bnt,
                          const float2 *unscale, float *y, float *yu, int ns, cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    for (int k = 0; k < (tu ? 2 : 1) && e == cudaSuccess; ++k) {
        const Tensor &tt = k ? *tu : t;
        float *yy = k ? yu : y;
        // Split each tile's k-blocks over ks CTAs (one CTA per SM, each
        // keeping at least 4 k-blocks) when that shortens the call: the time
        // goes as (waves of CTAs) x (k-blocks per CTA), since each k-block
        // costs a fixed copy/barrier round trip.  The partials go to planes
        // of a workspace and are added in plane order.  (O = 8192: 64 tiles,
        // ks = 2; O = 12288: 96 tiles, ks = 3 in two waves.)
        const int tiles = tt.o_pad / BM, nk = (int)(tt.k_pad / BK);
        const int n_sms = sm_count(tt.device);
        int ks = 1;
        long long best = (long long)((tiles + n_sms - 1) / n_sms) * nk;
        for (int k = 2; k <= 6 && nk / k >= 4; ++k) {
            const long long cost = (long long)((tiles * k + n_sms - 1) / n_sms) * ((nk + k - 1) / k);
            if (cost < best) {
                best = cost;
                ks = k;
            }
        }
        float *dst = yy;
        const long long n = (long long)ns * tt.O;
        if (ks > 1) {
            e = workspace_alloc((void **)&dst, (size_t)ks * n * sizeof(float), st);
            if (e != cudaSuccess) break;
        }
        e = bnt == 16   ? run_gemm<FMT, 16, true>(tt, pc, bnt, unscale, dst, ns, st, ks)
            : bnt == 32 ? run_gemm<FMT, 32, true>(tt, pc, bnt, unscale, dst, ns, st, ks)
                        : run_gemm<FMT, 48, true>(tt, pc, bnt, unscale, dst, ns, st, ks);
        if (ks > 1) {
            if (e == cudaSuccess) {
                long long blocks = (n + 255) / 256;
                if (blocks > (long long)n_sms * 4) blocks = (long long)n_sms * 4;
                sum_planes_kernel<<<(int)blocks, 256, 0, st>>>(dst, unscale, yy, n, tt.O, ks);
                count_launch();
                e = cudaGetLastError();
            }
            cudaError_t ef = workspace_free(dst, st);
            if (e == cudaSuccess) e = ef;
        }
    }
    return e;
}

cudaError_t launch_tcx(const Tensor &t, const Tensor *tu, const float *x, float *y, float *yu, int S,
                       cudaStream_t st, bool *handled) {
    *handled = false;
    if (t.fmt != B200Q_I4 && t.fmt != B200Q_I8) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    for (int s0 = 0; s0 < S && e == cudaSuccess;) {
        const int ns = S - s0 < 15 ? S - s0 : 15;
        const int bnt = 3 * ns <= 16 ? 16 : 3 * ns <= 32 ? 32 : 48;
        void *ws = nullptr;
        e = workspace_alloc(&ws, 1024 + (size_t)bnt * t.k_pad * 2, st);
        if (e != cudaSuccess) return e;
        float2 *unscale = (float2 *)ws;
        __nv_bfloat16 *pc = (__nv_bfloat16 *)((uint8_t *)ws + 1024);
        x_to_pieces_kernel<<<ns + 1, kPieceThreads, 0, st>>>(x + (long long)s0 * t.I, pc, unscale, ns, t.I,
                                                             (int)t.k_pad, bnt, t.fmt == B200Q_I4 ? 1 : 0);
        count_launch();
        e = cudaGetLastError();
        if (e == cudaSuccess) {
            float *yc = y + (long long)s0 * t.O, *yuc = tu ? yu + (long long)s0 * tu->O : nullptr;
            e = t.fmt == B200Q_I4 ? run_tcx_chunk<B200Q_I4>(t, tu, pc, bnt, unscale, yc, yuc, ns, st)
                                  : run_tcx_chunk<B200Q_I8>(t, tu, pc, bnt, unscale, yc, yuc, ns, st);
        }
        cudaError_t ef = workspace_free(ws, st);
        if (e == cudaSuccess) e = ef;
        s0 += ns;
    }
    *handled = (e == cudaSuccess);
    return e;
}

// Stream-ordered workspace from the library's per-device pool (the one the
// tensor-core path uses for its bf16 copy of x).
cudaError_t workspace_alloc(void **ptr, size_t bytes, cudaStream_t st) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    cudaMemPool_t pool;
    e = get_pool(dev, &pool);
    if (e != cudaSuccess) return e;
    count_workspace_alloc();
    return cudaMallocFromPoolAsync(ptr, bytes, pool, st);
}

// Tensor maps of the GEMM over an uploaded tensor: the codes as bytes
// [o_pad, ld] with a box of 128 rows x one k-block's code bytes, and the
// group scales [o_pad, G_ld] f32 with a box of 128 rows x 4.
bool gemm_maps_encode(Tensor &t) {
    memset(&t.gemm_map, 0, sizeof t.gemm_map);
    memset(&t.gemm_sc_map, 0, sizeof t.gemm_sc_map);
    if (t.fmt != B200Q_I4 && t.fmt != B200Q_I8) return true;
    const uint32_t code_bytes = t.fmt == B200Q_I4 ? 32 : 64;
    if (!tmap_encode_2d(&t.gemm_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, t.codes, (uint64_t)t.ld, (uint64_t)t.o_pad,
                        (uint64_t)t.ld, code_bytes, BM, CU_TENSOR_MAP_SWIZZLE_NONE))
        return false;
    if (t.gs && !tmap_encode_2d(&t.gemm_sc_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, t.scales, (uint64_t)t.G_ld,
                                (uint64_t)t.o_pad, (uint64_t)t.G_ld * 4, kScaleBox, BM, CU_TENSOR_MAP_SWIZZLE_NONE))
        return false;
    return true;
}

cudaError_t workspace_free(void *ptr, cudaStream_t st) { return cudaFreeAsync(ptr, st); }

// ---------------------------------------------------------------------------
// Allocation-free variant of the tensor-core path (b200q_matmul_tc_noalloc).
//
// Some callers cannot allocate device memory while they run: their device
// memory is owned by another allocator (a framework's caching allocator or a
// pool that reserved the device), or they are latency-critical loops that
// must not wait on an allocator call that may synchronize or fail.  For them
// the bf16 copy of x lives in a fixed file-scope device array instead of a
// per-call workspace.  Every GPU that loads the library holds the array until
// the process exits.  All calls on a device share it and it keeps the last
// call's contents (the conversion kernel overwrites every element a call
// reads, so nothing needs clearing); calls that overlap in time on the GPU
// race on it.
constexpr size_t kNoAllocBytes = 24u << 20;   // 24 MiB: S * k_pad bf16 values
static __device__ __align__(256) uint8_t g_noalloc_ws[kNoAllocBytes];

size_t noalloc_capacity() { return kNoAllocBytes; }

// Device address of the array in the current device's context, looked up
// on every call (a host-side query, not a stream operation), so that a call
// after the context was reset or recreated gets the new address rather than
// a stale one.  The first lookup on a device may load the library's device
// code into that context, which is why the first call should come before
// any stream capture.
cudaError_t noalloc_workspace(void **out) {
    void *ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_ws);
    if (e != cudaSuccess) return e;
    *out = ptr;
    return cudaSuccess;
}

// x -> bf16 into the caller-independent array, then the same GEMM kernel as
// the tensor-core path.  The caller has checked fmt and that
// S * k_pad * 2 <= kNoAllocBytes.
cudaError_t launch_prefill_tc_noalloc(const Tensor &t, const float *x, float *y, int S, cudaStream_t st) {
    void *ws = nullptr;
    cudaError_t e = noalloc_workspace(&ws);
    if (e != cudaSuccess) return e;
    const int n_sms = sm_count(t.device);
    const long long groups = (long long)S * t.k_pad / 8;
    long long blocks = (groups + 255) / 256;
    if (blocks > (long long)n_sms * 16) blocks = (long long)n_sms * 16;
    x_to_bf16_kernel<<<(int)blocks, 256, 0, st>>>(x, (__nv_bfloat16 *)ws, S, t.I, (int)t.k_pad,
                                                   t.fmt == B200Q_I4 ? 1 : 0);
    count_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return t.fmt == B200Q_I4 ? run_gemm_x<B200Q_I4>(t, (__nv_bfloat16 *)ws, y, S, st)
                             : run_gemm_x<B200Q_I8>(t, (__nv_bfloat16 *)ws, y, S, st);
}

cudaError_t prefill_take_error(unsigned int *code) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_prefill_err, sizeof(unsigned int));
    if (e == cudaSuccess && *code) e = cudaMemcpyToSymbol(g_prefill_err, &zero, sizeof(unsigned int));
    return e;
}

}  // namespace qwq
