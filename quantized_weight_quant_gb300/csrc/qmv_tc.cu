// f32-accurate tensor-core matmul for few tokens (1 <= S <= 16), int8 / int4 /
// int2 weights with per-row scales:
//     y[s,o] = scale[o] * sum_i deq(W[o,i]) * x[s,i]
// ("CUDA 后端", section 1: weight_at / quant_matmul; three-backends chapter,
// section 四: qmatmul.comp, x loaded once and reused across the output rows).
//
// At decode the call streams every weight once, so the kernel's job is to
// retire weights at HBM rate with f32 accuracy.  The products go to the
// 5th-generation tensor cores instead of the FP32 pipe, which halves the
// integer work per weight and makes the cost independent of S:
//   * A (M = 128 weight rows, K-major) lives in tensor memory.  Dequantizing
//     warps turn each 32-bit code word into exact fp16 integers with one
//     LOP3 per two codes (the code ORed into the mantissa of 1024.0) and one
//     packed fp16 subtraction of the zero point (1024 + m*z), and store them
//     with tcgen05.st: int4 nibbles 0,4 and 1,5 of a word in place (the
//     second pair times 16), nibbles 2,6 and 3,7 after one shift; int8 bytes
//     0,2 in place and 1,3 after one shift; int2 fields at bits 0/2/4 of each
//     half word (times 1, 4, 16) in place and after shifts by 6 and 12.
//   * B holds x as two fp16 pieces per token (N = 2S columns, padded to 16 or
//     32): v = x * 2^k with 2^k a power of two that brings the largest |x| of
//     the CTA's columns to [2^14, 2^15), p0 = fp16(v), p1 = fp16(v - p0).
//     v - p0 is exact in f32 and p0 + p1 carries v to 2^-22 relative; the
//     powers of two the A entries carry (16, 4, 16) are divided out of B
//     exactly.  Codes and pieces are exact in fp16 and their products exact
//     in f32; tcgen05.mma.kind::f16 accumulates them in f32 in tensor memory.
//   * The work is (128-row tile, 128-byte k-block) items, numbered tile-major
//     and cut into equal contiguous runs, one per CTA (one CTA per SM), so
//     every SM streams the same number of weight bytes.  A CTA accumulates
//     each tile's run of k-blocks in one tensor-memory accumulator; a tile it
//     covers whole is written to y directly, a tile shared with its
//     neighbours is written as a partial plane (still in its scaled units,
//     with its exponent), and a small second kernel adds the planes of each
//     shared tile in CTA order and rounds once.
// Warp roles (26 warps): warp 0 issues the TMA copies of the code tiles
// (128 rows x 128 bytes, 128-byte swizzle) into a deep ring, starting before
// the dependency wait since weights are read-only; warp 1 allocates tensor
// memory and issues the MMAs; warps 2-5 read x, find the per-token exponent
// and build the B tiles, one B stage each; warps 6-21 dequantize, four per
// tensor-memory lane quarter, each a quarter of the columns; warps 22-25
// drain the accumulators.  Every mbarrier wait is bounded and a CTA that gives
// up records B200Q_ETIMEOUT (b200q_device_status) and winds down: an abort
// flag in shared memory releases the other roles' waits, the producer's
// copies in flight land, and tensor memory is freed.
#include <cuda.h>
#include <cuda_fp16.h>

#include <atomic>
#include <climits>
#include <cstring>

#include "qwq_internal.h"

namespace qwq {
namespace {

constexpr int kRowsT = 128;                 // rows per tile (M)
constexpr int kKbBytes = 128;               // code bytes per row per item
constexpr int kCodeTile = kRowsT * kKbBytes;   // 16 KB
constexpr int kNA = 3;                      // A buffers in tensor memory (128 columns each)
constexpr int kNB = 4;                      // B stages (one per converter warp)
constexpr int kDCol = 3 * 128;              // first accumulator column
constexpr int kConvWarps = 4, kDeqWarps = 16, kEpiWarps = 4;
constexpr int kWConv = 2, kWDeq = kWConv + kConvWarps, kWEpi = kWDeq + kDeqWarps;
constexpr int kThreads = (kWEpi + kEpiWarps) * 32;   // 832
constexpr unsigned long long kWaitNs = 2000000000ull;
constexpr int kSmemLimit = 232448;          // 227 KB
constexpr int kNoK = 1000;                  // exponent of a token whose columns here are all zero
constexpr int kPreStages = 4;               // code stages issued before x has been read

__device__ unsigned int g_tcs_err = 0;

// ---- per-format constants
// STEPS: A blocks (128 tensor-memory columns at most) per item; COLS: columns
// per step; XK: x elements per item; E: B entries (K) per step.
template <int FMT>
struct Fmt;
template <>
struct Fmt<B200Q_I4> {
    static constexpr int STEPS = 1, COLS = 128, XK = 256, E = 256;
};
template <>
struct Fmt<B200Q_I8> {
    static constexpr int STEPS = 1, COLS = 64, XK = 128, E = 128;
};
template <>
struct Fmt<B200Q_I2> {
    static constexpr int STEPS = 2, COLS = 128, XK = 512, E = 256;
};

// ---- PTX helpers (PTX ISA: mbarrier, cp.async.bulk.tensor, tcgen05)
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

// Bounded wait on a phase parity.  Gives up after kWaitNs, or at once when
// another role has already given up (*abort set); a wait that gives up first
// records the timeout and raises the abort flag.  Waiters other than the MMA
// issuer pass a nonzero sleep_ns: between polls they sleep instead of
// spinning, so that the one thread issuing the MMAs is not starved of issue
// slots by two dozen polling warps.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort, int sleep_ns = 512) {
    unsigned long long t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if (sleep_ns) __nanosleep(sleep_ns);
        if ((it & 63) == 63) {
            if (*abort) return false;
            if (t0 == 0) t0 = global_ns();
            else if (global_ns() - t0 > kWaitNs) {
                atomicExch(&g_tcs_err, (unsigned)(-B200Q_ETIMEOUT));
                *abort = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: D f32, A and B fp16, both K-major,
// M = 128, N = nb.
constexpr uint32_t idesc_f16(int nb) { return (1u << 4) | ((uint32_t)(nb >> 3) << 17) | ((uint32_t)(128 >> 4) << 24); }

// D (tensor memory) += A (tensor memory) x B (shared memory descriptor)
__device__ __forceinline__ void mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
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

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
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

// (a & mask) ^ c: the code field(s) selected by mask, ORed into the fp16
// bits of c (c's bits outside mask; an XOR inside mask flips sign bits).
__device__ __forceinline__ uint32_t lop_and_xor(uint32_t a, uint32_t mask, uint32_t c) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(a), "r"(mask), "r"(c));
    return r;
}

// Packed fp16 subtraction (round to nearest; exact for the small integers here).
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// One 32-bit code word -> exact fp16 pairs (one tensor-memory column each),
// in the order the B entries follow (see entry_src below).
//   int4: 4 columns: (n0,n4) (16 n1,16 n5) (n2,n6) (16 n3,16 n7), minus 8 each
//   int8: 2 columns: (c0,c2) (c1,c3); u = c + 128 is the byte with its sign
//         bit flipped (1024 + u, minus 1152)
//   int2: 8 columns: fields (0,8) (1,9)x4 (2,10)x16 from the word, (3,11)
//         (4,12)x4 (5,13)x16 after >> 6, (6,14) (7,15)x4 after >> 12, minus 2
template <int FMT>
__device__ __forceinline__ void word_cols(uint32_t w, uint32_t *c) {
    if (FMT == B200Q_I4) {
        const uint32_t w8 = w >> 8;
        c[0] = hsub2(lop_and_xor(w, 0x000F000Fu, 0x64006400u), 0x64086408u);    // 1024 + n - 1032
        c[1] = hsub2(lop_and_xor(w, 0x00F000F0u, 0x64006400u), 0x64806480u);    // 1024 + 16 n - 1152
        c[2] = hsub2(lop_and_xor(w8, 0x000F000Fu, 0x64006400u), 0x64086408u);
        c[3] = hsub2(lop_and_xor(w8, 0x00F000F0u, 0x64006400u), 0x64806480u);
    } else if (FMT == B200Q_I8) {
        const uint32_t w8 = w >> 8;
        c[0] = hsub2(lop_and_xor(w, 0x00FF00FFu, 0x64806480u), 0x64806480u);    // 1024 + u - 1152
        c[1] = hsub2(lop_and_xor(w8, 0x00FF00FFu, 0x64806480u), 0x64806480u);
    } else {
        const uint32_t w6 = w >> 6, w12 = w >> 12;
        c[0] = hsub2(lop_and_xor(w, 0x00030003u, 0x64006400u), 0x64026402u);    // 1024 + c - 1026
        c[1] = hsub2(lop_and_xor(w, 0x000C000Cu, 0x64006400u), 0x64086408u);    // 1024 + 4c - 1032
        c[2] = hsub2(lop_and_xor(w, 0x00300030u, 0x64006400u), 0x64206420u);    // 1024 + 16c - 1056
        c[3] = hsub2(lop_and_xor(w6, 0x00030003u, 0x64006400u), 0x64026402u);
        c[4] = hsub2(lop_and_xor(w6, 0x000C000Cu, 0x64006400u), 0x64086408u);
        c[5] = hsub2(lop_and_xor(w6, 0x00300030u, 0x64006400u), 0x64206420u);
        c[6] = hsub2(lop_and_xor(w12, 0x00030003u, 0x64006400u), 0x64026402u);
        c[7] = hsub2(lop_and_xor(w12, 0x000C000Cu, 0x64006400u), 0x64086408u);
    }
}

// B entry e of chunk position p (e = 8 * chunk + p) of a step: the x element
// it multiplies (offset from the chunk's first x element) and the power of
// two divided out of it.
//   int4: a chunk is one code word (8 x): order 0,4,1,5,2,6,3,7, 1/16 on 1,5,3,7
//   int8: a chunk is two words (8 x): order 0,2,1,3,4,6,5,7
//   int2: a chunk is half a word (16 x per word): half 0 takes 0,8,1,9,2,10,3,11,
//         half 1 takes 4,12,5,13,6,14,7,15; powers 1,1,1/4,1/4,1/16,1/16,1,1 and
//         1/4,1/4,1/16,1/16,1,1,1/4,1/4
template <int FMT>
__device__ __forceinline__ void chunk_src(int chunk, int p, int &off, float &mult) {
    if (FMT == B200Q_I4) {
        off = 8 * chunk + (p >> 1) + 4 * (p & 1);
        mult = (p & 2) ? 0.0625f : 1.f;
    } else if (FMT == B200Q_I8) {
        off = 8 * chunk + (p & 4) + ((p >> 1) & 1) + 2 * (p & 1);
        mult = 1.f;
    } else {
        const int f = (p >> 1) + 4 * (chunk & 1);          // field of the low half word; +8 in the high half
        const int r = f % 3;                                // position within its shift group: x1, x4, x16
        off = 16 * (chunk >> 1) + f + 8 * (p & 1);
        mult = r == 0 ? 1.f : r == 1 ? 0.25f : 0.0625f;
    }
}

// Which of the chunk's 8 loaded x values B entry p multiplies (the loads of
// chunk_src's offsets, relative to the chunk's first group of four).
template <int FMT>
__device__ __forceinline__ constexpr int chunk_xv(int p) {
    return FMT == B200Q_I4   ? (p >> 1) + 4 * (p & 1)
           : FMT == B200Q_I8 ? (p & 4) + ((p >> 1) & 1) + 2 * (p & 1)
                             : (p >> 1) + 4 * (p & 1);
}

// 2^k as two factors f1 * f2 (each a normal float) for -252 <= k <= 252.
__device__ __forceinline__ float2 pow2_pair(int k) {
    const int a = k > 126 ? 64 : k < -126 ? -64 : 0;      // first factor's exponent
    return make_float2(__int_as_float((a + 127) << 23), __int_as_float((k - a + 127) << 23));
}

// Flag publication between CTAs (PTX memory model: release / acquire at
// GPU scope).
__device__ __forceinline__ void flag_release(unsigned long long *f, unsigned long long v) {
    asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(f), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long flag_acquire(const unsigned long long *f) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
    return v;
}

// The power of two a token is scaled by (none for an all-zero token).
__device__ __forceinline__ int kscale(int k) { return k == kNoK ? 0 : k; }

// floor(log2 m) for finite m > 0, subnormals included.
__device__ __forceinline__ int ilog2_bits(float m) {
    const int b = __float_as_int(m);
    const int e = (b >> 23) & 0xFF;
    return e ? e - 127 : -118 - __clz(b);
}

struct TcsParams {
    const float *x;        // [S, I]
    const float *scales;   // [o_pad]
    float *y;              // [S, O]
    float *part;           // [2 * grid][S][128] partial planes of shared tiles (scaled units)
    int *part_k;           // [2 * grid][S] the exponent k of each plane's pieces
    unsigned long long *flag;   // [2 * grid][4] per plane and lane quarter: token once published
    unsigned long long token;   // this call's value of a published flag
    int O, I, S;
    int nkb;               // items per tile (k-blocks of 128 code bytes)
    int n_items;           // tiles * nkb
    int dc;                // code ring stages
};

// The CTA whose run of items holds item i (runs are [b n / G, (b+1) n / G)).
__device__ __forceinline__ int cta_of(const TcsParams &p, long long i) {
    return (int)(((i + 1) * gridDim.x - 1) / p.n_items);
}

template <int FMT, int NB>
__global__ void __launch_bounds__(kThreads, 1)
    qmv_tc_kernel(const __grid_constant__ CUtensorMap map_codes, const TcsParams p) {
    using F = Fmt<FMT>;
    constexpr int kBStage = NB * F::E * 2;      // bytes of one B stage
    constexpr uint32_t kIdesc = idesc_f16(NB);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int DC = p.dc;
    uint8_t *code_s = smem;                                  // [DC][16 KB]
    uint8_t *b_s = code_s + (size_t)DC * kCodeTile;           // [kNB][kBStage]
    uint64_t *bars = reinterpret_cast<uint64_t *>(b_s + kNB * kBStage);
    uint64_t *code_full = bars, *code_empty = bars + DC;
    uint64_t *a_full = bars + 2 * DC, *a_empty = a_full + kNA;
    uint64_t *b_full = a_empty + kNA, *b_empty = b_full + kNB;
    uint64_t *d_full = b_empty + kNB, *d_empty = d_full + 2;
    uint64_t *x_ready = d_empty + 2;
    int *kexp = reinterpret_cast<int *>(x_ready + 1);        // [16] per-token exponent k
    float *red = reinterpret_cast<float *>(kexp + 16);        // [kConvWarps][16] per-warp maxima
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(red + kConvWarps * 16);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.S, nkb = p.nkb;
    const int G = gridDim.x;
    const int i0 = (int)((long long)blockIdx.x * p.n_items / G);
    const int i1 = (int)((long long)(blockIdx.x + 1) * p.n_items / G);
    const int n_steps = (i1 - i0) * F::STEPS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < DC; ++s) {
            mbar_init(smem_u32(&code_full[s]), 1);
            mbar_init(smem_u32(&code_empty[s]), kDeqWarps);
        }
        for (int s = 0; s < kNA; ++s) {
            mbar_init(smem_u32(&a_full[s]), kDeqWarps);
            mbar_init(smem_u32(&a_empty[s]), 1);
        }
        for (int s = 0; s < kNB; ++s) {
            mbar_init(smem_u32(&b_full[s]), 1);
            mbar_init(smem_u32(&b_empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&d_full[s]), 1);
            mbar_init(smem_u32(&d_empty[s]), kEpiWarps);
        }
        mbar_init(smem_u32(x_ready), 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_codes)) : "memory");
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------- producer: code tiles, read-only, so no dependency wait
        if (lane == 0) {
            const uint64_t policy = evict_first_policy();
            int st = 0;
            uint32_t ph = 0;
            long long issued = 0;
            int kb = i0 % nkb, tile = i0 / nkb;
            for (int i = i0; i < i1; ++i) {
                // a few stages go out before the dependency wait; the rest
                // once the converters have read x, whose loads would
                // otherwise return behind this CTA's whole prefetch
                if (i - i0 == kPreStages && !mbar_wait(smem_u32(x_ready), 0, abort)) break;
                if (!mbar_wait(smem_u32(&code_empty[st]), ph ^ 1, abort)) break;
                const uint32_t bar = smem_u32(&code_full[st]);
                mbar_expect_tx(bar, kCodeTile);
                tma_load_2d(smem_u32(code_s + (size_t)st * kCodeTile), &map_codes, kb * kKbBytes, tile * kRowsT,
                            bar, policy);
                ++issued;
                if (++st == DC) {
                    st = 0;
                    ph ^= 1;
                }
                if (++kb == nkb) {
                    kb = 0;
                    ++tile;
                }
            }
            // copies still in flight must land before the CTA leaves (those of
            // stages already released were consumed)
            for (long long k = issued - DC < 0 ? 0 : issued - DC; k < issued; ++k) {
                uint32_t done = 0;
                const uint32_t bar = smem_u32(&code_full[k % DC]);
                const unsigned long long t0 = global_ns();
                while (!done && global_ns() - t0 < kWaitNs / 4)
                    asm volatile(
                        "{ .reg .pred q; mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2; selp.u32 %0, 1, 0, q; "
                        "}"
                        : "=r"(done)
                        : "r"(bar), "r"((uint32_t)((k / DC) & 1))
                        : "memory");
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            // The issuing thread shares its scheduler with busy dequantizing
            // warps, so every instruction here is costly: the k-block index
            // advances without divisions, descriptors step by constants, and
            // the one MMA that starts an accumulator is peeled off.
            int ab = 0, bs = 0, db = 0;
            uint32_t aph = 0, bph = 0, dph = 0;
            bool ok = true;
            const uint64_t bdesc0 = sw128_desc(smem_u32(b_s));   // start-address field + offset >> 4 stays < 2^14
            int kb = i0 % nkb;
            for (int i = i0; i < i1 && ok; ++i) {
                const bool seg_first = i == i0 || kb == 0;
                const bool seg_last = i == i1 - 1 || kb == nkb - 1;
                if (++kb == nkb) kb = 0;
                if (seg_first) {
                    if (!mbar_wait(smem_u32(&d_empty[db]), dph ^ 1, abort, 0)) break;
                    tc_fence_after();
                }
                const uint32_t d_tmem = tmem_base + kDCol + db * 64;
                for (int h = 0; h < F::STEPS && ok; ++h) {
                    if (!mbar_wait(smem_u32(&a_full[ab]), aph, abort, 0) ||
                        !mbar_wait(smem_u32(&b_full[bs]), bph, abort, 0)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bd = bdesc0 + (uint64_t)((bs * kBStage) >> 4);
                    const uint32_t at = tmem_base + ab * 128;
                    mma_tmem_a(d_tmem, at, bd, kIdesc, (seg_first && h == 0) ? 0u : 1u);
#pragma unroll
                    for (int j = 1; j < F::E / 16; ++j)
                        mma_tmem_a(d_tmem, at + j * 8, bd + (uint64_t)((((j >> 2) * (NB * 128)) + (j & 3) * 32) >> 4),
                                   kIdesc, 1u);
                    mma_commit(smem_u32(&a_empty[ab]));
                    mma_commit(smem_u32(&b_empty[bs]));
                    if (++ab == kNA) {
                        ab = 0;
                        aph ^= 1;
                    }
                    if (++bs == kNB) {
                        bs = 0;
                        bph ^= 1;
                    }
                }
                if (ok && seg_last) {
                    mma_commit(smem_u32(&d_full[db]));
                    if (++db == 2) {
                        db = 0;
                        dph ^= 1;
                    }
                }
            }
        }
    } else if (warp < kWDeq) {
        // ---------------- converters: x -> B (two fp16 pieces per token)
        const int cw = warp - kWConv;
        const int tid = cw * 32 + lane;                       // 0..127
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        // four consecutive x of a row from k0 (a multiple of 4): one 16-byte
        // load when rows are 16-byte aligned and k0 + 3 < I, else element
        // loads with zeros past I (no branch: predicated selects)
        const bool vec = (p.I & 3) == 0;
        auto ld4 = [&](const float *r, int k0) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (vec) {
                if (k0 < p.I) v = *reinterpret_cast<const float4 *>(r + k0);
            } else {
                v.x = k0 < p.I ? *(r + k0) : 0.f;
                v.y = k0 + 1 < p.I ? *(r + k0 + 1) : 0.f;
                v.z = k0 + 2 < p.I ? *(r + k0 + 2) : 0.f;
                v.w = k0 + 3 < p.I ? *(r + k0 + 3) : 0.f;
            }
            return v;
        };
        // largest |x| per token over the x columns of this CTA's items (the
        // first nkb items cover every k-block the CTA touches).  Loads go out
        // eight at a time with no branch between them (out-of-range lanes
        // read zeros), so each batch costs one round trip.
        const int n_kb = (i1 - i0) < nkb ? (i1 - i0) : nkb;
        const int n4 = n_kb * (F::XK / 4);                    // float4 groups per token
        {
            float m[16];
#pragma unroll
            for (int s = 0; s < 16; ++s) m[s] = 0.f;
            // (token, group) pairs flattened, eight loads of a thread per batch
            for (int base = 0; base < S * n4; base += 8 * kConvWarps * 32) {
                float4 v[8];
                int sv[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int t = base + j * kConvWarps * 32 + tid;
                    const int s = t / n4, g = t - s * n4;
                    const int kb = (i0 + g / (F::XK / 4)) % nkb;
                    sv[j] = s;
                    v[j] = t < S * n4 ? ld4(p.x + (long long)s * p.I, kb * F::XK + (g % (F::XK / 4)) * 4)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float a = fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w)));
#pragma unroll
                    for (int s = 0; s < 16; ++s)
                        if (s == sv[j]) m[s] = fmaxf(m[s], a);
                }
            }
#pragma unroll
            for (int s = 0; s < 16; ++s)
                if (s < S) {
                    float mm = m[s];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, off));
                    if (lane == 0) red[cw * 16 + s] = mm;
                }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kConvWarps * 32) : "memory");
        // k per token: the scaled largest |x| lies in [2^14, 2^15); 0 for an
        // all-zero token.  Written once by thread 0 for the epilogue; every
        // converter reads its tokens' k back from the maxima below.
        if (tid < S) {
            const float m = fmaxf(fmaxf(red[tid], red[16 + tid]), fmaxf(red[32 + tid], red[48 + tid]));
            kexp[tid] = m > 0.f ? 14 - ilog2_bits(m) : kNoK;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kConvWarps * 32) : "memory");
        if (tid == 0) mbar_arrive(smem_u32(x_ready));
        // B stages: converter warp cw builds steps cw, cw + 4, ... into stage cw
        constexpr int CH = F::E / 8;                          // 16-byte chunks per B row
        // Units (token s, 16-byte chunk c of a B row) are converted four per
        // lane at a time: the eight 16-byte x loads of a batch go out together,
        // and the first batch's loads are issued before waiting for the stage
        // to come free, so their latency overlaps the wait.
        constexpr int kBatch = 4;
        for (int st = cw, r = 0; st < n_steps; st += kConvWarps, ++r) {
            const int item = i0 + st / F::STEPS, h = st % F::STEPS;
            const int kb = item % nkb;
            const int xbase = kb * F::XK + h * (F::XK / F::STEPS);
            uint8_t *bst = b_s + (size_t)cw * kBStage;
            bool ok = true;
            for (int ub = lane; ub < S * CH; ub += kBatch * 32) {
                float4 xa[kBatch], xb[kBatch];
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    const int u = ub + 32 * k;
                    const int s = u / CH, c = u - s * CH;
                    // the chunk's 8 x values, two aligned groups of four: int4 /
                    // int8 x[8c .. 8c+7]; int2 (half h of word m) x[16m+4h ..] and
                    // x[16m+8+4h ..], so that entry p reads xv[(p >> 1) + 4 (p & 1)]
                    const int g0 = FMT == B200Q_I2 ? xbase + 16 * (c >> 1) + 4 * (c & 1) : xbase + 8 * c;
                    const int g1 = FMT == B200Q_I2 ? g0 + 8 : g0 + 4;
                    const float *xr = p.x + (long long)(u < S * CH ? s : 0) * p.I;
                    xa[k] = u < S * CH ? ld4(xr, g0) : make_float4(0.f, 0.f, 0.f, 0.f);
                    xb[k] = u < S * CH ? ld4(xr, g1) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if (ub == lane && !mbar_wait(smem_u32(&b_empty[cw]), (r & 1) ^ 1, abort)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    const int u = ub + 32 * k;
                    if (u >= S * CH) break;
                    const int s = u / CH, c = u - s * CH;
                    const float2 sc = pow2_pair(kscale(kexp[s]));
                    const float xv[8] = {xa[k].x, xa[k].y, xa[k].z, xa[k].w, xb[k].x, xb[k].y, xb[k].z, xb[k].w};
                    uint32_t p0[4], p1[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float v[2], lo[2];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            int off;
                            float mult;
                            const int pe = 2 * q + hh;
                            chunk_src<FMT>(c, pe, off, mult);
                            const float xs = ((xv[chunk_xv<FMT>(pe)] * sc.x) * sc.y) * mult;
                            const __half h0 = __float2half_rn(xs);
                            v[hh] = __half2float(h0);
                            lo[hh] = xs - v[hh];                      // exact in f32
                        }
                        const __half2 a0 = __floats2half2_rn(v[0], v[1]);
                        const __half2 a1 = __floats2half2_rn(lo[0], lo[1]);
                        p0[q] = *reinterpret_cast<const uint32_t *>(&a0);
                        p1[q] = *reinterpret_cast<const uint32_t *>(&a1);
                    }
                    // rows 2s (p0) and 2s + 1 (p1), 16-byte chunk c, 128-byte swizzle
                    const int atom = c >> 3, cc = c & 7;
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int n = 2 * s + j;
                        uint8_t *dst = bst + (size_t)atom * (NB * 128) + (n >> 3) * 1024 + (n & 7) * 128 +
                                       ((cc ^ (n & 7)) << 4);
                        const uint32_t *pp = j ? p1 : p0;
                        *reinterpret_cast<uint4 *>(dst) = make_uint4(pp[0], pp[1], pp[2], pp[3]);
                    }
                }
            }
            // lanes with no unit still wait for the stage before signalling it
            if (ok && lane >= S * CH && !mbar_wait(smem_u32(&b_empty[cw]), (r & 1) ^ 1, abort)) ok = false;
            if (!ok) break;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&b_full[cw]));
        }
    } else if (warp < kWEpi) {
        // ---------------- dequantizers: lane quarter q, column slice sl
        const int dw = warp - kWDeq;
        const int q = warp & 3;                              // tensor-memory lane quarter of this warp
        const int sl = dw >> 2;                              // 0..3
        const int row = q * 32 + lane;
        constexpr int SCOLS = F::COLS / 4;                   // columns per slice: 32 (int4, int2) or 16 (int8)
        constexpr int WORDS = FMT == B200Q_I2 ? 4 : 8;       // code words per slice
        int cs = 0, ab = 0;
        uint32_t cph = 0, aph = 0;
        for (int i = i0; i < i1; ++i) {
            if (!mbar_wait(smem_u32(&code_full[cs]), cph, abort)) break;
            const uint8_t *crow = code_s + (size_t)cs * kCodeTile + row * kKbBytes;
            bool ok = true;
#pragma unroll 1
            for (int h = 0; h < F::STEPS; ++h) {
                // this slice's code words (16-byte chunks, 128-byte swizzle)
                uint32_t wv[8];
                const int c0 = FMT == B200Q_I2 ? 4 * h + sl : 2 * sl;
                {
                    const uint4 a = *reinterpret_cast<const uint4 *>(crow + ((c0 ^ (row & 7)) << 4));
                    wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
                }
                if (WORDS == 8) {
                    const uint4 b = *reinterpret_cast<const uint4 *>(crow + (((c0 + 1) ^ (row & 7)) << 4));
                    wv[4] = b.x; wv[5] = b.y; wv[6] = b.z; wv[7] = b.w;
                }
                if (!mbar_wait(smem_u32(&a_empty[ab]), aph ^ 1, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + ab * 128 + sl * SCOLS;
                if constexpr (SCOLS == 32) {
                    uint32_t cols[32];
#pragma unroll
                    for (int w = 0; w < WORDS; ++w) word_cols<FMT>(wv[w], cols + w * (32 / WORDS));
                    tmem_st32(taddr, cols);
                } else {
                    uint32_t cols[16];
#pragma unroll
                    for (int w = 0; w < 8; ++w) word_cols<FMT>(wv[w], cols + 2 * w);
                    tmem_st16(taddr, cols);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&a_full[ab]));
                if (++ab == kNA) {
                    ab = 0;
                    aph ^= 1;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&code_empty[cs]));
            if (!ok) break;
            if (++cs == DC) {
                cs = 0;
                cph ^= 1;
            }
        }
    } else {
        // ---------------- epilogue: lane quarter q of each accumulator
        const int q = warp & 3;
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (mbar_wait(smem_u32(x_ready), 0, abort)) {
            int db = 0;
            uint32_t dph = 0;
            for (int i = i0; i < i1;) {
                const int tile = i / nkb;
                const int seg_end = (tile + 1) * nkb < i1 ? (tile + 1) * nkb : i1;
                const bool full = i == tile * nkb && seg_end == (tile + 1) * nkb;
                if (!mbar_wait(smem_u32(&d_full[db]), dph, abort)) break;
                tc_fence_after();
                float v[NB];
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + kDCol + db * 64;
#pragma unroll
                for (int c = 0; c < NB / 16; ++c) {
                    float w16[16];
                    tmem_ld16(taddr + c * 16, w16);
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[c * 16 + j] = w16[j];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&d_empty[db]));
                const int o = tile * kRowsT + q * 32 + lane;
                if (full) {
                    if (o < p.O) {
                        const float rs = p.scales[o];
#pragma unroll
                        for (int s = 0; s < NB / 2; ++s)
                            if (s < S) {
                                const float2 un = pow2_pair(-kscale(kexp[s]));
                                p.y[(long long)s * p.O + o] = (((v[2 * s] + v[2 * s + 1]) * rs) * un.x) * un.y;
                            }
                    }
                } else {
                    // partial plane: the CTA's first tile in slot 2b, its last in
                    // 2b + 1; published per lane quarter once its rows are stored
                    const int slot = 2 * (int)blockIdx.x + (i == i0 ? 0 : 1);
                    float *pl = p.part + (long long)slot * S * kRowsT;
#pragma unroll
                    for (int s = 0; s < NB / 2; ++s)
                        if (s < S) pl[s * kRowsT + q * 32 + lane] = v[2 * s] + v[2 * s + 1];
                    if (lane < S) p.part_k[slot * 64 + q * 16 + lane] = kexp[lane];
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) flag_release(p.flag + slot * 4 + q, p.token);
                }
                if (++db == 2) {
                    db = 0;
                    dph ^= 1;
                }
                i = seg_end;
            }
            // A tile shared with lower-numbered CTAs whose last k-block is
            // this CTA's first item: wait for their planes (this quarter's
            // rows), add all planes in CTA order in common units, round once.
            const int t = i0 / nkb;
            const int b = (int)blockIdx.x;
            const int b_lo = cta_of(p, (long long)t * nkb);
            const bool owner = i0 != t * nkb && cta_of(p, (long long)(t + 1) * nkb - 1) == b;
            if (owner && !*abort) {
                bool ok = true;
                for (int c = b_lo; c < b && ok; ++c) {
                    const int slot = 2 * c + ((long long)c * p.n_items / G >= (long long)t * nkb ? 0 : 1);
                    const unsigned long long t0 = global_ns();
                    while (flag_acquire(p.flag + slot * 4 + q) != p.token) {
                        if (*abort || global_ns() - t0 > kWaitNs) {
                            if (!*abort) atomicExch(&g_tcs_err, (unsigned)(-B200Q_ETIMEOUT));
                            *abort = 1;
                            ok = false;
                            break;
                        }
                        __nanosleep(256);
                    }
                }
                const int o = t * kRowsT + q * 32 + lane;
                if (ok && o < p.O) {
                    const float rs = p.scales[o];
                    for (int s = 0; s < S; ++s) {
                        int K = INT_MAX;
                        for (int c = b_lo; c <= b; ++c) {
                            const int slot = 2 * c + ((long long)c * p.n_items / G >= (long long)t * nkb ? 0 : 1);
                            const int k = __ldcg(p.part_k + slot * 64 + q * 16 + s);
                            if (k != kNoK && k < K) K = k;
                        }
                        float acc = 0.f;
                        if (K != INT_MAX) {
                            for (int c = b_lo; c <= b; ++c) {
                                const int slot = 2 * c + ((long long)c * p.n_items / G >= (long long)t * nkb ? 0 : 1);
                                const int k = __ldcg(p.part_k + slot * 64 + q * 16 + s);
                                if (k == kNoK || K - k < -250) continue;
                                const float2 f = pow2_pair(K - k);
                                acc += (__ldcg(p.part + ((long long)slot * S + s) * kRowsT + q * 32 + lane) * f.x) * f.y;
                            }
                        } else {
                            K = 0;
                        }
                        const float2 un = pow2_pair(-K);
                        p.y[(long long)s * p.O + o] = ((acc * rs) * un.x) * un.y;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512) : "memory");
}

// Tokens of the flags that publish partial planes: unique per call in this
// process (a 64-bit counter), so a flag left in reused memory by an earlier
// call never reads as published.
std::atomic<unsigned long long> g_token{0x5eed0000000001ull};

unsigned long long next_token() { return g_token.fetch_add(1, std::memory_order_relaxed); }

template <int FMT, int NB>
size_t smem_for(int dc) {
    return 1024 + (size_t)dc * kCodeTile + (size_t)kNB * NB * Fmt<FMT>::E * 2 + (2 * dc + 2 * kNA + 2 * kNB + 5) * 8 +
           16 * 4 + kConvWarps * 16 * 4 + 16;
}

template <int FMT, int NB>
cudaError_t launch_fmt(const Tensor &t, const float *x, float *y, int S, cudaStream_t st) {
    const int nkb = (int)(t.ld / kKbBytes);
    const int tiles = t.o_pad / kRowsT;
    const long long n_items = (long long)tiles * nkb;
    if (n_items >= (1ll << 31) / 160) return cudaErrorInvalidValue;   // item arithmetic is 32-bit
    const int n_sms = sm_count(t.device);
    const int G = (int)(n_items < n_sms ? n_items : n_sms);
    int dc = 16;
    while (dc > 2 && smem_for<FMT, NB>(dc) > (size_t)kSmemLimit) --dc;
    const size_t smem = smem_for<FMT, NB>(dc);
    if (smem > (size_t)kSmemLimit) return cudaErrorInvalidValue;
    // is any tile shared by two CTAs?
    bool shared = false;
    for (int b = 1; b < G && !shared; ++b) shared = ((long long)b * n_items / G) % nkb != 0;
    // shared tiles: partial planes [2G][S][128] f32, their exponents [2G][4][16]
    // int, and flags [2G][4] u64 (published with this call's token; stale
    // values from earlier use of the memory never equal a new token)
    float *part = nullptr;
    cudaError_t e = cudaSuccess;
    const size_t planes = (size_t)2 * G * S * kRowsT * sizeof(float);
    const size_t kbytes = (size_t)2 * G * 64 * sizeof(int);
    const size_t fbytes = (size_t)2 * G * 4 * sizeof(unsigned long long);
    if (shared) {
        e = workspace_alloc((void **)&part, planes + kbytes + fbytes + 256, st);
        if (e != cudaSuccess) return e;
    }
    e = allow_dynamic_smem((const void *)qmv_tc_kernel<FMT, NB>, (int)smem);
    TcsParams prm;
    prm.x = x;
    prm.scales = t.scales;
    prm.y = y;
    prm.part = part;
    prm.part_k = part ? reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(part) + planes) : nullptr;
    prm.flag = part ? reinterpret_cast<unsigned long long *>(
                          (reinterpret_cast<uintptr_t>(part) + planes + kbytes + 15) & ~(uintptr_t)15)
                    : nullptr;
    prm.token = next_token();
    prm.O = t.O;
    prm.I = t.I;
    prm.S = S;
    prm.nkb = nkb;
    prm.n_items = (int)n_items;
    prm.dc = dc;
    if (e == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(G);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, qmv_tc_kernel<FMT, NB>, t.tcs_map, prm);
        count_launch();
        if (e == cudaSuccess) e = cudaGetLastError();
    }
    if (part) {
        cudaError_t ef = workspace_free(part, st);
        if (e == cudaSuccess) e = ef;
    }
    return e;
}

template <int FMT>
cudaError_t launch_nb(const Tensor &t, const float *x, float *y, int S, cudaStream_t st) {
    return S <= 8 ? launch_fmt<FMT, 16>(t, x, y, S, st) : launch_fmt<FMT, 32>(t, x, y, S, st);
}

}  // namespace

// Tensor map of the codes for this path: bytes [o_pad, ld], box 128 rows x
// 128 bytes, 128-byte swizzle (int8 / int4 / int2 tensors).
bool tcs_map_encode(Tensor &t) {
    memset(&t.tcs_map, 0, sizeof t.tcs_map);
    if (t.fmt != B200Q_I4 && t.fmt != B200Q_I8 && t.fmt != B200Q_I2) return true;
    return tmap_encode_2d(&t.tcs_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, t.codes, (uint64_t)t.ld, (uint64_t)t.o_pad,
                          (uint64_t)t.ld, kKbBytes, kRowsT, CU_TENSOR_MAP_SWIZZLE_128B);
}

// The f32-accurate tensor-core path for 1 <= S <= 16: int8 / int4 / int2
// tensors with per-row scales.  *handled = false for anything else.
cudaError_t launch_tcs(const Tensor &t, const float *x, float *y, int S, cudaStream_t st, bool *handled) {
    *handled = false;
    if (S < 1 || S > 16 || t.gs) return cudaSuccess;
    cudaError_t e;
    switch (t.fmt) {
    case B200Q_I4: e = launch_nb<B200Q_I4>(t, x, y, S, st); break;
    case B200Q_I8: e = launch_nb<B200Q_I8>(t, x, y, S, st); break;
    case B200Q_I2: e = launch_nb<B200Q_I2>(t, x, y, S, st); break;
    default: return cudaSuccess;
    }
    if (e == cudaErrorInvalidValue) return cudaSuccess;
    *handled = e == cudaSuccess;
    return e;
}

cudaError_t tcs_take_error(unsigned int *code) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_tcs_err, sizeof(unsigned int));
    if (e == cudaSuccess && *code) e = cudaMemcpyToSymbol(g_tcs_err, &zero, sizeof(unsigned int));
    return e;
}

}  // namespace qwq
