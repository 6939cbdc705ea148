// f32-accurate tensor-core matmul for few tokens (1 <= S <= 8 per launch),
// int8 / int4 / int2 weights with per-row scales:
//     y[s,o] = scale[o] * sum_i deq(W[o,i]) * x[s,i]
// ("CUDA 后端", section 1: weight_at / quant_matmul; three-backends chapter,
// section 四: qmatmul.comp, x loaded once and reused across the output rows).
//
// At decode the call streams every weight once, so the job is to retire
// weights at HBM rate with f32 accuracy.  The products run on the
// 5th-generation tensor cores as an exact integer dot product in fp8:
//   * A 4-bit field u placed in the low bits of an E4M3 byte (exponent bias
//     7) is worth exactly u * 2^-9 for every u in 0..15: 0..7 are the
//     subnormals u * 2^-9, 8..15 have the exponent field 1 and the mantissa
//     u - 8, i.e. (1 + (u - 8) / 8) * 2^-6 = u * 2^-9.  So a code field
//     masked into a byte *is* its fp8 operand: int4 codes take one AND per
//     four codes (w & 0x0F0F0F0F, (w >> 4) & 0x0F0F0F0F), int2 codes one per
//     four codes after a shift, and int8 codes (with the sign bit flipped,
//     u = c + 128) split into a low and a high nibble.
//   * x is rounded per token to a signed fixed-point integer
//     n = rint(x * 2^T), |n| < 2^(4J-1), with 2^T a power of two that brings
//     the token's largest |x| in the CTA's columns to [2^(4J-2), 2^(4J-1)),
//     then offset to n'' = n + 2^(4J-1) in [0, 16^J) and cut into J 4-bit
//     digits, each again a nibble byte.  B has one row (N column of the MMA)
//     per token and digit, plus one row of ones.
//   * The MMA (kind::f8f6f4, E4M3 x E4M3, f32 accumulation in tensor
//     memory) then computes sum_k u_k * d_k * 2^-18: integers below 2^24, so
//     every accumulation is exact.  The epilogue recombines the digits in
//     64-bit integers, sum_k (u_k - z) n_k
//       = sum_j 16^j D_j - 2^(4J-1) D_ones - z sum_k n_k,
//     exactly, and rounds once: y = f32(scale * 2^-T * that).  The only
//     approximation is the rounding of x to 4J-2 bits below its token's
//     largest magnitude (J = 7 or 8: 26 or 30 bits).
// Work: (128-row tile, 128-byte k-block) items, cut into equal contiguous
// runs, one per CTA (one CTA per SM), in range-major order: K is split into
// ranges of R k-blocks, and the items of range r come before those of r + 1,
// tile-major inside a range.  R is the largest value for which every CTA's
// k-blocks (whose B tiles it builds once, in shared memory) fit; it is the
// whole row when they do.  A CTA accumulates each (range, tile) run of its
// items in one tensor-memory accumulator.  A tile that one CTA covers whole
// goes straight to y.  Otherwise every piece is written as an f64 plane and
// the CTA that brings the tile's arrival count (an atomic tagged with the
// call's token) to its number of pieces adds the planes in a fixed order and
// writes y.  No CTA waits on another, so calls on concurrent streams cannot
// hold each other up.  (A variant in which the CTA holding the tile's first
// item waited for the others' flags measured ~1 us faster per call; its
// wait needs every CTA of the launch resident, which concurrent launches
// can prevent.)
// Warp roles: warp 0 issues the TMA copies of the code tiles (128 rows x
// 128 bytes, 128-byte swizzle) into a ring, from the start, since the
// weights are read-only; warp 1 allocates tensor memory and issues the MMAs;
// NA groups of four warps dequantize (group g takes every NA-th item into A
// buffer g, one tensor-memory lane quarter per warp); four warps drain the
// accumulators.  The dequantizing and draining warps first build the B
// tiles (after the dependency wait), slot by slot, and the MMAs start as
// soon as the slot they need is built.  Hand-offs inside the CTA that no
// tensor-core commit is involved in go through shared-memory counters
// (release add, acquire load): an mbarrier test costs a few hundred cycles
// on this part even when its phase is complete.  Every wait is bounded; a
// CTA that gives up records B200Q_ETIMEOUT (b200q_device_status) and winds
// down: an abort flag in shared memory releases the other roles' waits, the
// producer's copies in flight land, the MMAs issued complete, and tensor
// memory is freed.
#include <cuda.h>

#include <atomic>
#include <climits>
#include <cstring>
#include <vector>

#include "qwq_internal.h"

namespace qwq {
namespace {

constexpr int kRowsT = 128;                    // rows per tile (M)
constexpr int kKbBytes = 128;                  // code bytes per row per item
constexpr int kCodeTile = kRowsT * kKbBytes;   // 16 KB
constexpr int kMaxS = 8;                       // tokens per launch
constexpr int kEpiWarps = 4;
constexpr int kWDeq = 2;                       // first dequantizing warp
constexpr int kSmemLimit = 232448;             // 227 KB
constexpr int kSmemFloor = 120 * 1024;         // keeps one CTA per SM (tensor memory is taken whole)
constexpr int kMiscBytes = 3072;               // barriers, exponents, maxima, counters, plane list (plus 72 bytes per B slot)
constexpr int kMaxPlanes = 256;                // pieces of one tile, at most (the count is 8 bits)
constexpr unsigned long long kWaitNs = 2000000000ull;

__device__ unsigned int g_tcs_err = 0;

// ---- per-format constants
// KPE: codes per k-block (128 bytes of a row); POS: fp8 A entries per
// k-block (K of its MMAs); COLS: tensor-memory columns of one A buffer;
// NA: A buffers; Z: zero point in the unsigned code the MMA sees; PAIR: int8
// splits each code into a low and a high nibble, accumulated apart.
template <int FMT>
struct Fmt;
template <>
struct Fmt<B200Q_I4> {
    static constexpr int KPE = 256, POS = 256, COLS = 64, NA = 4, Z = 8, UMAX = 15;
    static constexpr bool PAIR = false;
};
template <>
struct Fmt<B200Q_I8> {
    static constexpr int KPE = 128, POS = 256, COLS = 64, NA = 4, Z = 128, UMAX = 15;
    static constexpr bool PAIR = true;
};
template <>
struct Fmt<B200Q_I2> {
    static constexpr int KPE = 512, POS = 512, COLS = 128, NA = 3, Z = 2, UMAX = 3;
    static constexpr bool PAIR = false;
};

// Warp roles per format: warp 0 producer, warp 1 MMA issuer, then NA groups
// of four dequantizing warps (one per tensor-memory lane quarter; group g
// takes items g, g + NA, ... of the run into A buffer g), then four
// epilogue warps.  The dequantizing and epilogue warps build B first.
template <int FMT>
struct Roles {
    static constexpr int kDeq = 4 * Fmt<FMT>::NA;
    static constexpr int kWEpi = kWDeq + kDeq;
    static constexpr int kThreads = (kWEpi + kEpiWarps) * 32;
    static constexpr int kStageWarps = kDeq + kEpiWarps;
    static constexpr int kStagers = kStageWarps * 32;
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

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait on a phase parity.  Gives up after kWaitNs, or at once when
// another role has already given up (*abort set); a wait that gives up first
// records the timeout and raises the abort flag.  try_wait itself suspends
// the thread for a while when the phase is not complete, so polling costs
// few issue slots and no sleep is added (a sleep delays the wake-up).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    unsigned long long t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_test(bar, parity)) return true;
        if ((it & 15) == 15) {
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

// Two adjacent counters read at once (8-byte aligned pair): waits for the
// first to reach want and reports whether the second has too.
__device__ __forceinline__ bool cnt_wait2(uint32_t addr, uint32_t want, volatile int *abort, bool &second) {
    unsigned long long t0 = 0;
    for (uint32_t it = 0;; ++it) {
        unsigned long long v;
        asm volatile("ld.acquire.cta.shared::cta.b64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
        if ((int)((uint32_t)v - want) >= 0) {
            second = (int)((uint32_t)(v >> 32) - want) >= 0;
            return true;
        }
        if ((it & 255) == 255) {
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

// Compare-and-swap at GPU scope with acquire-release semantics: the release
// orders this thread's earlier writes (and, through a preceding barrier, its
// CTA's) before the swap; the acquire orders its later reads after it.
__device__ __forceinline__ unsigned long long cas_acq_rel(unsigned long long *a, unsigned long long cmp,
                                                          unsigned long long val) {
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.cas.b64 %0, [%1], %2, %3;" : "=l"(old) : "l"(a), "l"(cmp), "l"(val)
                 : "memory");
    return old;
}

// A wait that ignores the abort flag (winding down: copies or MMAs already
// issued must complete before the CTA leaves), bounded by a quarter of kWaitNs.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    while (!mbar_test(bar, parity) && global_ns() - t0 < kWaitNs / 4) {
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

// Instruction descriptor, kind::f8f6f4: D f32, A and B E4M3 (format 0), both
// K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_e4m3(int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// D (tensor memory) += A (tensor memory) x B (shared memory descriptor)
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p; }" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// One accumulator column of this warp's lane quarter (32x32b.x1), not yet waited for.
__device__ __forceinline__ void tmem_ld1(uint32_t taddr, uint32_t &r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// Counters in shared memory that hand work between roles of the CTA: an
// mbarrier test costs a few hundred cycles on this part even when the phase
// is complete, a shared load far less.  Release on the add, acquire on the
// read (PTX memory model, CTA scope).
__device__ __forceinline__ void cnt_add(uint32_t addr) {
    asm volatile("red.release.cta.shared::cta.add.u32 [%0], 1;" ::"r"(addr) : "memory");
}
__device__ __forceinline__ uint32_t cnt_read(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Bounded wait for a shared counter to reach want (see cnt_add).
__device__ __forceinline__ bool cnt_wait(uint32_t addr, uint32_t want, volatile int *abort) {
    unsigned long long t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if ((int)(cnt_read(addr) - want) >= 0) return true;
        if ((it & 255) == 255) {
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

// Named barrier that also ORs a predicate over its threads (a uniform decision).
__device__ __forceinline__ bool named_sync_or(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// 2^-k as a double, |k| <= 1000.
__device__ __forceinline__ double pow2_neg(int k) { return __longlong_as_double((long long)(1023 - k) << 52); }

// floor(log2 m) for finite m > 0, subnormals included.
__device__ __forceinline__ int ilog2_bits(float m) {
    const int b = __float_as_int(m);
    const int e = (b >> 23) & 0xFF;
    return e ? e - 127 : -118 - __clz(b);
}

// 2^k as two factors f1 * f2 (each a normal float) for -252 <= k <= 252.
__device__ __forceinline__ float2 pow2_pair(int k) {
    const int a = k > 126 ? 64 : k < -126 ? -64 : 0;
    return make_float2(__int_as_float((a + 127) << 23), __int_as_float((k - a + 127) << 23));
}

// ---- the run of items, in range-major order
struct TcsParams {
    const float *x;            // [S, I]
    const float *scales;       // [o_pad]
    float *y;                  // [S, O]
    double *plane;             // [grid * pmax][S][128] pieces of shared tiles (f64, unscaled by 2^-T)
    unsigned long long *cnt;   // [tiles] (token << 8) | arrivals
    unsigned long long token;  // this call's tag (56 bits)
    int O, I, S;
    int J, N;                  // digits per token; MMA N (rows of B)
    int nkb;                   // k-blocks per row
    int R, nr;                 // k-blocks per range; ranges
    int tiles, n_items;
    int nb;                    // B slots (k-blocks staged per CTA, at most)
    int dc;                    // code ring stages
    int pmax;                  // pieces per CTA, at most
};

struct Item {
    int r, t, kb;   // range, tile, k-block
    int seg;        // r * tiles + t: increases along the order
};

__device__ __forceinline__ int range_size(const TcsParams &p, int r) {
    const int s = p.nkb - r * p.R;
    return s < p.R ? s : p.R;
}

__device__ __forceinline__ Item item_of(const TcsParams &p, int i) {
    const int per = p.R * p.tiles;     // items of a full range
    int r = i / per;
    if (r >= p.nr) r = p.nr - 1;
    const int size = range_size(p, r);
    const int rest = i - r * per;
    Item it;
    it.r = r;
    it.t = rest / size;
    it.kb = r * p.R + (rest - it.t * size);
    it.seg = r * p.tiles + it.t;
    return it;
}

// Walks the items in order without divisions (item_of once, at the start).
struct Walk {
    int i, r, t, kb, rlo, rend;   // k-blocks of range r: [rlo, rend)
    __device__ __forceinline__ void init(const TcsParams &p, int i_) {
        const Item it = item_of(p, i_);
        i = i_;
        r = it.r;
        t = it.t;
        kb = it.kb;
        rlo = r * p.R;
        rend = rlo + range_size(p, r);
    }
    __device__ __forceinline__ void next(const TcsParams &p) {
        ++i;
        if (++kb == rend) {
            kb = rlo;
            if (++t == p.tiles) {
                t = 0;
                ++r;
                rlo = r * p.R;
                rend = rlo + range_size(p, r);
                kb = rlo;
            }
        }
    }
    __device__ __forceinline__ int seg(const TcsParams &p) const { return r * p.tiles + t; }
};

// First item of segment (r, t), and the CTA whose run holds item i (runs are
// [b n / G, (b + 1) n / G)).
__device__ __forceinline__ int seg_first(const TcsParams &p, int r, int t) {
    return r * p.R * p.tiles + t * range_size(p, r);
}
__device__ __forceinline__ int cta_of(const TcsParams &p, int i) {
    return (int)(((long long)(i + 1) * gridDim.x - 1) / p.n_items);
}
__device__ __forceinline__ int run_first(const TcsParams &p, int b) {
    return (int)((long long)b * p.n_items / gridDim.x);
}

// The B slots of a CTA: its items touch one or two ranges; in each, the
// k-blocks it covers form a cyclic interval of the range (tile-major order).
struct Slots {
    int r0, first0, size0, cnt0;   // range r0: slots [0, cnt0) hold k-blocks (first0 + s) % size0 of it
    int first1, size1, cnt1;       // range r0 + 1 (cnt1 = 0 when untouched): slots [cnt0, cnt0 + cnt1)
};

__device__ __forceinline__ Slots slots_of(const TcsParams &p, int i0, int i1) {
    Slots s;
    const int per = p.R * p.tiles;
    const Item a = item_of(p, i0), z = item_of(p, i1 - 1);
    s.r0 = a.r;
    s.size0 = range_size(p, a.r);
    const int end0 = a.r == z.r ? i1 : (a.r + 1) * per;
    s.first0 = a.kb - a.r * p.R;
    s.cnt0 = end0 - i0 < s.size0 ? end0 - i0 : s.size0;
    s.first1 = 0;
    s.size1 = 1;
    s.cnt1 = 0;
    if (z.r != a.r) {
        s.size1 = range_size(p, z.r);
        s.cnt1 = i1 - end0 < s.size1 ? i1 - end0 : s.size1;
    }
    return s;
}

__device__ __forceinline__ int slot_of(const TcsParams &p, const Slots &s, int kb) {
    if (kb < (s.r0 + 1) * p.R) {
        int off = kb - s.r0 * p.R - s.first0;
        if (off < 0) off += s.size0;
        return off;
    }
    return s.cnt0 + (kb - (s.r0 + 1) * p.R - s.first1);
}

__device__ __forceinline__ int kb_of_slot(const TcsParams &p, const Slots &s, int slot) {
    if (slot < s.cnt0) {
        int off = s.first0 + slot;
        if (off >= s.size0) off -= s.size0;
        return s.r0 * p.R + off;
    }
    return (s.r0 + 1) * p.R + s.first1 + (slot - s.cnt0);
}

// Byte offset of B entry (row, pos) in a slot: K-major, 128-byte swizzle,
// atoms of 128 positions x N rows.
__device__ __forceinline__ uint32_t b_off(int row, int pos, int N) {
    const int atom = pos >> 7, b = pos & 127;
    return (uint32_t)(atom * N * 128 + row * 128 + ((((b >> 4) ^ (row & 7))) << 4) + (b & 15));
}

// Four 32-bit values -> their bytes transposed: t[m] holds byte m of a, b, c, d.
__device__ __forceinline__ void bytes_t4(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t (&t)[4]) {
    const uint32_t ab_lo = __byte_perm(a, b, 0x5140), cd_lo = __byte_perm(c, d, 0x5140);
    const uint32_t ab_hi = __byte_perm(a, b, 0x7362), cd_hi = __byte_perm(c, d, 0x7362);
    t[0] = __byte_perm(ab_lo, cd_lo, 0x5410);
    t[1] = __byte_perm(ab_lo, cd_lo, 0x7632);
    t[2] = __byte_perm(ab_hi, cd_hi, 0x5410);
    t[3] = __byte_perm(ab_hi, cd_hi, 0x7632);
}

// Digit j of four offset integers, as a word of nibble bytes (byte e: digit j of value e).
__device__ __forceinline__ uint32_t digit_word(const uint32_t (&t)[4], int j) {
    const uint32_t w = t[j >> 1];
    return ((j & 1) ? (w >> 4) : w) & 0x0F0F0F0Fu;
}

template <int FMT>
__global__ void __launch_bounds__(Roles<FMT>::kThreads, 1)
    qmv_tc_kernel(const __grid_constant__ CUtensorMap map_codes, const TcsParams p) {
    using F = Fmt<FMT>;
    using RL = Roles<FMT>;
    constexpr int kMma = F::POS / 32;          // MMAs per item
    constexpr int kDStride = F::PAIR ? 128 : 64;
    constexpr int kDCol = F::NA * F::COLS;     // first accumulator column
    constexpr int kWEpi = RL::kWEpi, kStageWarps = RL::kStageWarps, kStagers = RL::kStagers;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int DC = p.dc, N = p.N, S = p.S, J = p.J;
    const int bslot = N * F::POS;
    uint8_t *code_s = smem;                                    // [DC][16 KB]
    uint8_t *b_s = code_s + (size_t)DC * kCodeTile;             // [nb][bslot]
    uint64_t *bars = reinterpret_cast<uint64_t *>(b_s + (size_t)p.nb * bslot);
    uint64_t *code_full = bars, *code_empty = bars + DC;
    uint64_t *a_empty = bars + 2 * DC;                         // [NA] MMAs done with A buffer g
    uint64_t *d_full = a_empty + F::NA, *d_empty = d_full + 2;
    uint64_t *mma_done = d_empty + 2;
    long long *nsum = reinterpret_cast<long long *>(mma_done + 1);   // [nb][kMaxS] sum of n per slot and token
    long long *npiece = nsum + (size_t)p.nb * kMaxS;                // [2][kMaxS] the same over a piece
    int *texp = reinterpret_cast<int *>(npiece + 2 * kMaxS);         // [kMaxS] shift T per token
    float *red = reinterpret_cast<float *>(texp + kMaxS);             // [kStageWarps][kMaxS] per-warp maxima
    uint32_t *a_cnt = reinterpret_cast<uint32_t *>(red + kStageWarps * kMaxS);  // [NA] warps done filling buffer g
    uint32_t *slot_cnt = a_cnt + F::NA;                               // [nb] units of slot k built
    uint32_t *tmem_slot = slot_cnt + p.nb;
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *last_flag = abort + 1;
    int *plist = const_cast<int *>(last_flag + 1);                    // [kMaxPlanes + 1] planes of a tile to add

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i0 = run_first(p, blockIdx.x), i1 = run_first(p, blockIdx.x + 1);
    const int n_items = i1 - i0;
    const Slots sl = slots_of(p, i0, i1);
    const int n_slots = sl.cnt0 + sl.cnt1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < DC; ++s) {
            mbar_init(smem_u32(&code_full[s]), 1);
            mbar_init(smem_u32(&code_empty[s]), 4);
        }
        for (int s = 0; s < F::NA; ++s) {
            mbar_init(smem_u32(&a_empty[s]), 1);
            a_cnt[s] = 0;
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&d_full[s]), 1);
            mbar_init(smem_u32(&d_empty[s]), kEpiWarps);
        }
        mbar_init(smem_u32(mma_done), 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int k = threadIdx.x; k < p.nb; k += blockDim.x) slot_cnt[k] = 0;
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
        // ---------------- producer: code tiles (read-only: no dependency wait)
        if (lane == 0) {
            const uint64_t policy = evict_first_policy();
            int st = 0;
            uint32_t ph = 0;
            long long issued = 0;
            Walk w;
            w.init(p, i0);
            for (int i = i0; i < i1; ++i, w.next(p)) {
                if (!mbar_wait(smem_u32(&code_empty[st]), ph ^ 1, abort)) break;
                const uint32_t bar = smem_u32(&code_full[st]);
                mbar_expect_tx(bar, kCodeTile);
                tma_load_2d(smem_u32(code_s + (size_t)st * kCodeTile), &map_codes, w.kb * kKbBytes, w.t * kRowsT,
                            bar, policy);
                ++issued;
                if (++st == DC) {
                    st = 0;
                    ph ^= 1;
                }
            }
            // copies still in flight land before the CTA leaves
            for (long long k = issued - DC < 0 ? 0 : issued - DC; k < issued; ++k)
                mbar_drain(smem_u32(&code_full[k % DC]), (uint32_t)((k / DC) & 1));
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_e4m3(N);
            int g = 0, db = 0;
            uint32_t fill = 0, dph = 0;          // fills of buffer g so far (per round of groups)
            unsigned long long ready = 0;        // B slots known to be built
            uint32_t known = 0;                  // A buffers known to be filled for the current round
            const uint64_t bdesc0 = sw128_desc(smem_u32(b_s));
            bool issued_any = false;
            Walk w;
            w.init(p, i0);
            for (int i = i0; i < i1; ++i, w.next(p)) {
                const bool first = i == i0 || w.kb == w.rlo;
                const bool last = i == i1 - 1 || w.kb + 1 == w.rend;
                if (first) {
                    if (!mbar_wait(smem_u32(&d_empty[db]), dph ^ 1, abort)) break;
                }
                const int slot = slot_of(p, sl, w.kb);
                if (!((ready >> slot) & 1)) {
                    if (!cnt_wait(smem_u32(&slot_cnt[slot]), (uint32_t)S, abort)) break;
                    ready |= 1ull << slot;
                }
                // buffer g filled for this round; an even g also tells about g + 1
                if (!((known >> g) & 1)) {
                    if (F::NA % 2 == 0 && (g & 1) == 0) {
                        bool next = false;
                        if (!cnt_wait2(smem_u32(&a_cnt[g]), 4u * (fill + 1), abort, next)) break;
                        if (next) known |= 2u << g;
                    } else if (!cnt_wait(smem_u32(&a_cnt[g]), 4u * (fill + 1), abort)) {
                        break;
                    }
                }
                known &= ~(1u << g);
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + kDCol + db * kDStride;
                const uint64_t bd = bdesc0 + (uint64_t)(((uint32_t)slot * bslot) >> 4);
                const uint32_t at = tmem_base + g * F::COLS;
#pragma unroll
                for (int m = 0; m < kMma; ++m) {
                    const bool hi = F::PAIR && m >= kMma / 2;
                    const uint32_t acc = (first && (m == 0 || (F::PAIR && m == kMma / 2))) ? 0u : 1u;
                    mma_f8(d_tmem + (hi ? 64 : 0), at + m * 8,
                           bd + (uint64_t)((uint32_t)((m >> 2) * N * 128 + (m & 3) * 32) >> 4), idesc, acc);
                }
                issued_any = true;
                mma_commit(smem_u32(&a_empty[g]));
                if (++g == F::NA) {
                    g = 0;
                    ++fill;
                }
                if (last) {
                    mma_commit(smem_u32(&d_full[db]));
                    if (++db == 2) {
                        db = 0;
                        dph ^= 1;
                    }
                }
            }
            // every MMA issued has completed before tensor memory is freed
            if (issued_any) {
                mma_commit(smem_u32(mma_done));
                mbar_drain(smem_u32(mma_done), 0);
            }
        }
    } else {
        // ---------------- dequantizing and epilogue warps: build B, then their loops
        const int sw = warp - kWDeq;                  // 0 .. kStageWarps - 1
        const int stid = sw * 32 + lane;
        // Dequantizing warps: group grp fills A buffer grp with items grp,
        // grp + NA, ... of the run (lane = row of the tile).  Item k, the
        // fill-th use of the buffer:
        const int grp = (warp - kWDeq) >> 2, quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t abase = tmem_base + ((uint32_t)(quarter * 32) << 16) + grp * F::COLS;
        auto deq_item = [&](int k, uint32_t fill) -> bool {
            const int st = k % DC;
            if (!mbar_wait(smem_u32(&code_full[st]), (uint32_t)((k / DC) & 1), abort)) return false;
            // row r's 128 code bytes: eight 16-byte chunks, swizzled; read
            // in two halves of 16 words, the stage released after the second
            const uint8_t *row = code_s + (size_t)st * kCodeTile + r * 128;
            uint32_t w[16], v[32];
            auto load_half = [&](int h) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 t = *reinterpret_cast<const uint4 *>(row + (((4 * h + c) ^ (r & 7)) << 4));
                    w[4 * c] = t.x;
                    w[4 * c + 1] = t.y;
                    w[4 * c + 2] = t.z;
                    w[4 * c + 3] = t.w;
                }
            };
            load_half(0);
            if (!mbar_wait(smem_u32(&a_empty[grp]), (fill & 1) ^ 1, abort)) return false;
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (h == 1) {
                    load_half(1);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&code_empty[st]));
                }
                if (FMT == B200Q_I4) {
                    // word q -> columns 2q (even codes) and 2q + 1 (odd codes)
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        v[2 * q] = w[q] & 0x0F0F0F0Fu;
                        v[2 * q + 1] = (w[q] >> 4) & 0x0F0F0F0Fu;
                    }
                    tmem_st32(abase + h * 32, v);
                } else if (FMT == B200Q_I8) {
                    // code + 128 = 16 hi + lo: low nibbles to columns q, high to 32 + q
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        v[q] = (w[q] ^ 0x80808080u) & 0x0F0F0F0Fu;
                        v[16 + q] = ((w[q] ^ 0x80808080u) >> 4) & 0x0F0F0F0Fu;
                    }
                    tmem_st16(abase + h * 16, v);
                    tmem_st16(abase + 32 + h * 16, v + 16);
                } else {
                    // word q -> columns 4q + i: fields i, i + 4, i + 8, i + 12
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
#pragma unroll
                            for (int i = 0; i < 4; ++i) v[4 * q + i] = (w[8 * e + q] >> (2 * i)) & 0x03030303u;
                        tmem_st32(abase + h * 64 + e * 32, v);
                    }
                }
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) cnt_add(smem_u32(&a_cnt[grp]));
            return true;
        };
        // the row of ones (each byte 0x01: 2^-9) and the unused rows (zero)
        // do not depend on x: written before the dependency wait
        {
            const int ones = S * J;
            const int rows_left = N - ones;
            const int chunks = n_slots * rows_left * (F::POS / 16);
            for (int c = stid; c < chunks; c += kStagers) {
                const int slot = c / (rows_left * (F::POS / 16));
                const int rest = c - slot * (rows_left * (F::POS / 16));
                const int row = ones + rest / (F::POS / 16), ch = rest % (F::POS / 16);
                const uint32_t v = row == ones ? 0x01010101u : 0u;
                *reinterpret_cast<uint4 *>(b_s + (size_t)slot * bslot + b_off(row, ch * 16, N)) = make_uint4(v, v, v, v);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        const bool vec = (p.I & 3) == 0 && (reinterpret_cast<uintptr_t>(p.x) & 15) == 0;
        // Units of B work: (slot, token) pairs, unit u = slot * S + s, warp
        // sw takes units sw, sw + kStageWarps, ...; lane q of a unit holds V
        // float4 of x: 8 (int4), 4 (int8) or 16 (int2) consecutive elements of
        // its k-block.  When every warp has at most kHold units, x is loaded
        // once and kept in registers across the exponent barrier; otherwise a
        // max-only pass runs first and the digit pass loads again.  Loads of
        // a batch all go out before any is used.  Units go in slot order, and
        // each unit's slot counter is raised as soon as its rows are written,
        // so the MMAs can start on the first slot while the rest are built.
        constexpr int V = F::KPE / 128;
        constexpr int kHold = 2;
        const int units = n_slots * S;
        const bool hold = (units + kStageWarps - 1) / kStageWarps <= kHold;
        auto load_unit = [&](int u, float4 (&v)[V]) {
            const int slot = u / S, s = u - slot * S;
            const int kb = kb_of_slot(p, sl, slot);
            const float *xr = p.x + (long long)s * p.I + (long long)kb * F::KPE;
            const int kleft = p.I - kb * F::KPE;      // x beyond I reads as zero
#pragma unroll
            for (int h = 0; h < V; ++h) {
                const int k0 = (lane * V + h) * 4;
                float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
                if (vec) {
                    if (k0 < kleft) t = *reinterpret_cast<const float4 *>(xr + k0);
                } else {
                    t.x = k0 < kleft ? xr[k0] : 0.f;
                    t.y = k0 + 1 < kleft ? xr[k0 + 1] : 0.f;
                    t.z = k0 + 2 < kleft ? xr[k0 + 2] : 0.f;
                    t.w = k0 + 3 < kleft ? xr[k0 + 3] : 0.f;
                }
                v[h] = t;
            }
        };
        float4 xv[kHold][V];
        float m[kMaxS];
#pragma unroll
        for (int t = 0; t < kMaxS; ++t) m[t] = 0.f;
        auto note = [&](int u, const float4 (&v)[V]) {
            const int s = u % S;
            float a = 0.f;
#pragma unroll
            for (int h = 0; h < V; ++h) a = fmaxf(a, fmaxf(fmaxf(fabsf(v[h].x), fabsf(v[h].y)), fmaxf(fabsf(v[h].z), fabsf(v[h].w))));
#pragma unroll
            for (int t = 0; t < kMaxS; ++t)
                if (t == s) m[t] = fmaxf(m[t], a);
        };
        // (1) largest |x| per token over the staged k-blocks
        for (int u0 = sw; u0 < units; u0 += kStageWarps * kHold) {
#pragma unroll
            for (int k = 0; k < kHold; ++k)
                if (u0 + kStageWarps * k < units) load_unit(u0 + kStageWarps * k, xv[k]);
#pragma unroll
            for (int k = 0; k < kHold; ++k)
                if (u0 + kStageWarps * k < units) note(u0 + kStageWarps * k, xv[k]);
            if (hold) break;
        }
#pragma unroll
        for (int t = 0; t < kMaxS; ++t) {
            if (t >= S) break;
            float a = m[t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            if (lane == 0) red[sw * kMaxS + t] = a;
        }
        named_sync(1, kStagers);
        if (stid < S) {
            float a = 0.f;
            for (int w = 0; w < kStageWarps; ++w) a = fmaxf(a, red[w * kMaxS + stid]);
            // T brings the largest |x| to [2^(4J-2), 2^(4J-1)); zero tokens keep T = 0
            texp[stid] = a > 0.f ? 4 * J - 2 - ilog2_bits(a) : 0;
        }
        named_sync(1, kStagers);
        // (2) digits of each unit's x into its B rows
        {
            const uint32_t off_n = 1u << (4 * J - 1);
            auto convert = [&](int u, const float4 (&v)[V]) {
                const int slot = u / S, s = u - slot * S;
                const float2 f = pow2_pair(texp[s]);
                uint8_t *bs = b_s + (size_t)slot * bslot;
                long long nsm = 0;
                auto conv = [&](float x) {
                    const int n = __float2int_rn((x * f.x) * f.y);
                    nsm += n;
                    return (uint32_t)n + off_n;
                };
                if (FMT == B200Q_I4) {
                    // positions 8q + i <- k = 8q + 2i, positions 8q + 4 + i <- k = 8q + 2i + 1
                    uint32_t te[4], to[4];
                    bytes_t4(conv(v[0].x), conv(v[0].z), conv(v[1].x), conv(v[1].z), te);
                    bytes_t4(conv(v[0].y), conv(v[0].w), conv(v[1].y), conv(v[1].w), to);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (j >= J) break;
                        *reinterpret_cast<uint2 *>(bs + b_off(s * J + j, 8 * lane, N)) =
                            make_uint2(digit_word(te, j), digit_word(to, j));
                    }
                } else if (FMT == B200Q_I8) {
                    // positions 4q + i (low nibbles) and 128 + 4q + i (high) <- k = 4q + i
                    uint32_t t4[4];
                    bytes_t4(conv(v[0].x), conv(v[0].y), conv(v[0].z), conv(v[0].w), t4);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (j >= J) break;
                        const uint32_t w = digit_word(t4, j);
                        *reinterpret_cast<uint32_t *>(bs + b_off(s * J + j, 4 * lane, N)) = w;
                        *reinterpret_cast<uint32_t *>(bs + b_off(s * J + j, 128 + 4 * lane, N)) = w;
                    }
                } else {
                    // positions 16q + 4i + e <- k = 16q + 4e + i
                    uint32_t t0[4], t1[4], t2[4], t3[4];
                    bytes_t4(conv(v[0].x), conv(v[1].x), conv(v[2].x), conv(v[3].x), t0);
                    bytes_t4(conv(v[0].y), conv(v[1].y), conv(v[2].y), conv(v[3].y), t1);
                    bytes_t4(conv(v[0].z), conv(v[1].z), conv(v[2].z), conv(v[3].z), t2);
                    bytes_t4(conv(v[0].w), conv(v[1].w), conv(v[2].w), conv(v[3].w), t3);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (j >= J) break;
                        *reinterpret_cast<uint4 *>(bs + b_off(s * J + j, 16 * lane, N)) =
                            make_uint4(digit_word(t0, j), digit_word(t1, j), digit_word(t2, j), digit_word(t3, j));
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) nsm += __shfl_xor_sync(0xffffffffu, nsm, o);
                // every lane's rows visible to the tensor cores before the count
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    nsum[slot * kMaxS + s] = nsm;
                    cnt_add(smem_u32(&slot_cnt[slot]));
                }
            };
            for (int u0 = sw; u0 < units; u0 += kStageWarps * kHold) {
                if (!hold) {
#pragma unroll
                    for (int k = 0; k < kHold; ++k)
                        if (u0 + kStageWarps * k < units) load_unit(u0 + kStageWarps * k, xv[k]);
                }
#pragma unroll
                for (int k = 0; k < kHold; ++k)
                    if (u0 + kStageWarps * k < units) convert(u0 + kStageWarps * k, xv[k]);
            }
        }

        if (warp < kWEpi) {
            // ---------------- dequantizers
            for (int k = grp, fill = 0; k < n_items; k += F::NA, ++fill)
                if (!deq_item(k, (uint32_t)fill)) break;
        } else {
            // ---------------- epilogue: one row per thread, one piece at a time
            const int quarter = warp & 3;
            const int r = quarter * 32 + lane;
            const int etid = (warp - kWEpi) * 32 + lane;          // 0..127
            const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
            const long long off_n = 1ll << (4 * J - 1);
            int db = 0, pc = 0;
            uint32_t dph = 0;
            Walk w;
            w.init(p, i0);
            const int seg_base = w.seg(p);
            while (w.i < i1) {
                // the piece: k-blocks [kb0, kb0 + len) of segment (w.r, w.t)
                const int kb0 = w.kb, pr = w.r, t = w.t, seg = w.seg(p);
                const int len = w.rend - w.kb < i1 - w.i ? w.rend - w.kb : i1 - w.i;
                // sum of n over the piece's k-blocks, per token
                long long *np = npiece + (pc & 1) * kMaxS;
                bool ok = true;
                if (etid < S) {
                    long long a = 0;
                    for (int kb = kb0; kb < kb0 + len && ok; ++kb) {
                        const int slot = slot_of(p, sl, kb);
                        ok = cnt_wait(smem_u32(&slot_cnt[slot]), (uint32_t)S, abort);   // its nsum is written
                        a += nsum[slot * kMaxS + etid];
                    }
                    np[etid] = a;
                }
                ok = mbar_wait(smem_u32(&d_full[db]), dph, abort) && ok;
                if (named_sync_or(2, kEpiWarps * 32, !ok)) break;     // np is visible too
                tc_fence_after();
                const uint32_t dt = lane_base + kDCol + db * kDStride;
                // 2^18 D: exact integers; int8 adds 16 times the high-nibble accumulator
                uint32_t one_lo, one_hi = 0;
                tmem_ld1(dt + S * J, one_lo);
                if (F::PAIR) tmem_ld1(dt + 64 + S * J, one_hi);
                tmem_wait_ld();
                const long long d_one = (long long)__float2int_rn(__uint_as_float(one_lo) * 262144.f) +
                                        (F::PAIR ? 16ll * __float2int_rn(__uint_as_float(one_hi) * 262144.f) : 0ll);
                double val[kMaxS];
#pragma unroll
                for (int s = 0; s < kMaxS; ++s) {
                    val[s] = 0.0;
                    if (s < S) {
                        uint32_t dl[8], dh[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            dl[j] = dh[j] = 0u;
                            if (j < J) {
                                tmem_ld1(dt + s * J + j, dl[j]);
                                if (F::PAIR) tmem_ld1(dt + 64 + s * J + j, dh[j]);
                            }
                        }
                        tmem_wait_ld();
                        long long acc = 0;
#pragma unroll
                        for (int j = 7; j >= 0; --j) {
                            if (j >= J) continue;
                            long long dj = __float2int_rn(__uint_as_float(dl[j]) * 262144.f);
                            if (F::PAIR) dj += 16ll * __float2int_rn(__uint_as_float(dh[j]) * 262144.f);
                            acc = acc * 16 + dj;
                        }
                        acc -= off_n * d_one + (long long)F::Z * np[s];
                        val[s] = (double)acc * pow2_neg(texp[s]);   // exact: |acc| < 2^53
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&d_empty[db]));
                if (++db == 2) {
                    db = 0;
                    dph ^= 1;
                }
                const int o = t * kRowsT + r;
                const double sc = (double)p.scales[o];
                // whole tile in this piece: one range, and no other CTA in the segment
                const int sf = seg_first(p, pr, t);
                const bool whole = p.nr == 1 && cta_of(p, sf) == cta_of(p, sf + range_size(p, pr) - 1);
                if (whole) {
                    if (o < p.O)
                        #pragma unroll
                        for (int s = 0; s < kMaxS; ++s)
                            if (s < S) p.y[(long long)s * p.O + o] = (float)(sc * val[s]);
                } else {
                    const int lp = seg - seg_base;
                    double *pl = p.plane + ((size_t)blockIdx.x * p.pmax + lp) * S * kRowsT;
                    #pragma unroll
                    for (int s = 0; s < kMaxS; ++s)
                        if (s < S) pl[s * kRowsT + r] = val[s];
                    // the barrier orders every thread's plane before thread 0's
                    // release (cumulative), part of the count's update
                    named_sync(2, kEpiWarps * 32);
                    if (etid == 0) {
                        // pieces of tile t: its segments' CTAs, range by range
                        int expect = 0;
                        for (int rr = 0; rr < p.nr; ++rr) {
                            const int f0 = seg_first(p, rr, t);
                            expect += cta_of(p, f0 + range_size(p, rr) - 1) - cta_of(p, f0) + 1;
                        }
                        const unsigned long long tag = p.token << 8;
                        // a word left by an earlier call (or any earlier use of the
                        // memory) does not carry this call's tag: the first
                        // arrival replaces it
                        unsigned long long old = *(volatile unsigned long long *)&p.cnt[t], nv = 0;
                        for (int k = 0; k < 4096; ++k) {
                            nv = (old & ~0xFFull) == tag ? old + 1 : tag | 1ull;
                            const unsigned long long prev = cas_acq_rel(&p.cnt[t], old, nv);
                            if (prev == old) break;
                            old = prev;
                            nv = 0;
                        }
                        const bool last = nv != 0 && (int)(nv & 0xFF) == expect;
                        if (last) {
                            // the tile's planes in (range, CTA) order
                            int n = 0;
                            for (int rr = 0; rr < p.nr; ++rr) {
                                const int f0 = seg_first(p, rr, t);
                                const int c0 = cta_of(p, f0), c1 = cta_of(p, f0 + range_size(p, rr) - 1);
                                for (int c = c0; c <= c1 && n < kMaxPlanes; ++c)
                                    plist[1 + n++] = c * p.pmax + rr * p.tiles + t - item_of(p, run_first(p, c)).seg;
                            }
                            plist[0] = n;
                        }
                        *last_flag = last;
                    }
                    named_sync(2, kEpiWarps * 32);
                    if (*last_flag) {
                        // loads of two planes go out together
                        double sum[kMaxS];
#pragma unroll
                        for (int s = 0; s < kMaxS; ++s) sum[s] = 0.0;
                        const int npl = plist[0];
                        for (int k0 = 0; k0 < npl; k0 += 2) {
                            double v[2][kMaxS];
#pragma unroll
                            for (int k = 0; k < 2; ++k) {
                                const double *q = p.plane + (size_t)plist[1 + (k0 + k < npl ? k0 + k : 0)] * S * kRowsT + r;
#pragma unroll
                                for (int s = 0; s < kMaxS; ++s) v[k][s] = k0 + k < npl && s < S ? __ldcg(q + s * kRowsT) : 0.0;
                            }
#pragma unroll
                            for (int k = 0; k < 2; ++k)
#pragma unroll
                                for (int s = 0; s < kMaxS; ++s) sum[s] += v[k][s];
                        }
                        if (o < p.O)
                            #pragma unroll
                            for (int s = 0; s < kMaxS; ++s)
                                if (s < S) p.y[(long long)s * p.O + o] = (float)(sc * sum[s]);
                    }
                    named_sync(2, kEpiWarps * 32);
                }
                ++pc;
                for (int k = 0; k < len; ++k) w.next(p);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512) : "memory");
}

// Tokens tagging the per-tile arrival counters: unique per call in this
// process, so a count left in reused memory by an earlier call never reads
// as this call's.
std::atomic<unsigned long long> g_token{0x5eed01ull};

unsigned long long next_token() { return g_token.fetch_add(1, std::memory_order_relaxed) & 0xFFFFFFFFFFFFFFull; }

// Launch plan for one tensor and S tokens.
struct Plan {
    int J, N, R, nr, nb, dc, pmax, G;
    bool shared;
    size_t smem;
};

template <int FMT>
bool make_plan(const Tensor &t, int S, int n_sms, Plan &pl) {
    using F = Fmt<FMT>;
    const int nkb = (int)(t.ld / kKbBytes), tiles = t.o_pad / kRowsT;
    const long long n = (long long)tiles * nkb;
    if (nkb < 1 || n < 1 || n >= (1ll << 31) / 256) return false;
    const int G = (int)(n < n_sms ? n : n_sms);
    pl.G = G;
    pl.N = 16 * ((7 * S + 1 + 15) / 16);
    pl.J = 8 * S + 1 <= pl.N ? 8 : 7;
    const int bslot = pl.N * F::POS;
    const int budget = kSmemLimit - 1024 - kMiscBytes;
    // every accumulation exact: per accumulator column and piece, the products
    // (at most UMAX * 15) summed over R k-blocks stay below 2^24
    const int kacc = F::PAIR ? F::POS / 2 : F::POS;
    const int rmax = (1 << 24) / (F::UMAX * 15 * kacc);
    auto range_size = [&](int R, int r) { return nkb - r * R < R ? nkb - r * R : R; };
    for (int R = nkb < rmax ? nkb : rmax; R >= 1; R = R == 1 ? 0 : (R + 1) / 2) {
        const int nr = (nkb + R - 1) / R;
        const long long per = (long long)R * tiles;
        auto range_of = [&](long long i) { long long r = i / per; return (int)(r >= nr ? nr - 1 : r); };
        auto seg_of = [&](long long i) {
            const int r = range_of(i);
            return (long long)r * tiles + (i - r * per) / range_size(R, r);
        };
        int need = 0, pmax = 1;
        bool ok = true;
        for (int b = 0; b < G && ok; ++b) {
            const long long i0 = (long long)b * n / G, i1 = (long long)(b + 1) * n / G;
            if (i1 <= i0) continue;
            const int ra = range_of(i0), rz = range_of(i1 - 1);
            if (rz > ra + 1) {
                ok = false;
                break;
            }
            const long long end0 = ra == rz ? i1 : (long long)(ra + 1) * per;
            int c = (int)(end0 - i0 < range_size(R, ra) ? end0 - i0 : range_size(R, ra));
            if (rz != ra) c += (int)(i1 - end0 < range_size(R, rz) ? i1 - end0 : range_size(R, rz));
            if (c > need) need = c;
            const long long pc = seg_of(i1 - 1) - seg_of(i0) + 1;
            if (pc > pmax) pmax = (int)pc;
        }
        if (!ok || need > 64 || (long long)need * (bslot + 72) + 4ll * kCodeTile > budget) continue;
        // arrival counts fit 8 bits
        int maxc = 0;
        for (int tt = 0; tt < tiles && nr > 1; ++tt) {
            int c = 0;
            for (int r = 0; r < nr; ++r) {
                const long long f0 = (long long)r * per + (long long)tt * range_size(R, r);
                const long long f1 = f0 + range_size(R, r) - 1;
                c += (int)(((f1 + 1) * G - 1) / n - ((f0 + 1) * G - 1) / n + 1);
            }
            if (c > maxc) maxc = c;
        }
        if (maxc > 250) continue;
        pl.R = R;
        pl.nr = nr;
        pl.nb = need;
        pl.pmax = pmax;
        int dc = (int)((budget - (long long)need * (bslot + 72)) / kCodeTile);
        pl.dc = dc > 16 ? 16 : dc;
        bool shared = nr > 1;
        for (int b = 1; b < G && !shared; ++b) shared = ((long long)b * n / G) % nkb != 0;
        pl.shared = shared;
        size_t smem = 1024 + (size_t)pl.dc * kCodeTile + (size_t)need * (bslot + 72) + kMiscBytes;
        pl.smem = smem < (size_t)kSmemFloor ? (size_t)kSmemFloor : smem;
        return true;
    }
    return false;
}

template <int FMT>
cudaError_t launch_fmt(const Tensor &t, const float *x, float *y, int S, cudaStream_t st) {
    Plan pl;
    if (!make_plan<FMT>(t, S, sm_count(t.device), pl)) return cudaErrorInvalidValue;
    const int nkb = (int)(t.ld / kKbBytes), tiles = t.o_pad / kRowsT;
    double *plane = nullptr;
    cudaError_t e = cudaSuccess;
    const size_t plane_bytes = (size_t)pl.G * pl.pmax * S * kRowsT * sizeof(double);
    if (pl.shared) {
        e = workspace_alloc((void **)&plane, plane_bytes + (size_t)tiles * 8 + 256, st);
        if (e != cudaSuccess) return e;
    }
    e = allow_dynamic_smem((const void *)qmv_tc_kernel<FMT>, (int)pl.smem);
    TcsParams prm;
    prm.x = x;
    prm.scales = t.scales;
    prm.y = y;
    prm.plane = plane;
    prm.cnt = plane ? reinterpret_cast<unsigned long long *>(
                          (reinterpret_cast<uintptr_t>(plane) + plane_bytes + 15) & ~(uintptr_t)15)
                    : nullptr;
    prm.token = next_token();
    prm.O = t.O;
    prm.I = t.I;
    prm.S = S;
    prm.J = pl.J;
    prm.N = pl.N;
    prm.nkb = nkb;
    prm.R = pl.R;
    prm.nr = pl.nr;
    prm.tiles = tiles;
    prm.n_items = tiles * nkb;
    prm.nb = pl.nb;
    prm.dc = pl.dc;
    prm.pmax = pl.pmax;
    if (e == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(pl.G);
        cfg.blockDim = dim3(Roles<FMT>::kThreads);
        cfg.dynamicSmemBytes = pl.smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, qmv_tc_kernel<FMT>, t.tcs_map, prm);
        count_launch();
        if (e == cudaSuccess) e = cudaGetLastError();
    }
    if (plane) {
        cudaError_t ef = workspace_free(plane, st);
        if (e == cudaSuccess) e = ef;
    }
    return e;
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

// The f32-accurate tensor-core path: int8 / int4 / int2 tensors with per-row
// scales, launched in chunks of at most 8 tokens.  *handled = false for
// anything else.
cudaError_t launch_tcs(const Tensor &t, const float *x, float *y, int S, cudaStream_t st, bool *handled) {
    *handled = false;
    if (S < 1 || t.gs) return cudaSuccess;
    if (t.fmt != B200Q_I4 && t.fmt != B200Q_I8 && t.fmt != B200Q_I2) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    for (int s0 = 0; s0 < S && e == cudaSuccess; s0 += kMaxS) {
        const int ns = S - s0 < kMaxS ? S - s0 : kMaxS;
        const float *xs = x + (long long)s0 * t.I;
        float *ys = y + (long long)s0 * t.O;
        switch (t.fmt) {
        case B200Q_I4: e = launch_fmt<B200Q_I4>(t, xs, ys, ns, st); break;
        case B200Q_I8: e = launch_fmt<B200Q_I8>(t, xs, ys, ns, st); break;
        default: e = launch_fmt<B200Q_I2>(t, xs, ys, ns, st); break;
        }
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
