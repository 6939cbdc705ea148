// Decode kernel, the f32-accurate path at small S for every format:
//     y[s,o] = scale[o] * sum_i deq(W[o,i]) * x[s,i]
// ("CUDA 后端", section 1: weight_at / quant_matmul; three-backends chapter,
// section 四: the qmatmul.comp header, x staged once and reused for every
// output row).
//
// Decode reads every weight once, so the kernel must retire weights at HBM
// rate: ~90 G int4 weights/s per SM on GB300.  Two facts set the design.
//   * mma.sync (the pre-Blackwell tensor-core path) runs at a small fraction
//     of the tcgen05 rate here and at S = 1 would waste 7/8 of every
//     fragment, so the products stay on the FP32 pipe.
//   * A conventional unpack (shift, mask, convert, subtract) costs 3-4 issue
//     slots per weight before the FMA.  Instead each code is ANDed in place
//     out of its 32-bit word: with the exponent field zero the result *is* an
//     f32 (a subnormal) whose value is code * 2^b * 2^-149, b = the code's bit
//     offset in the word, exactly.  x is staged in shared memory pre-scaled by
//     the matching power of two, so one FFMA forms code * x * 2^T exactly
//     (2^T a per-token power of two that keeps every value in range).  The
//     zero-point comes out per lane and unit: the lane also runs a row of
//     zero-point codes through the identical FFMA chain (its multipliers are
//     compile-time constants) and subtracts it, so a run of zero-point codes
//     cancels to exactly 0: sum (c - z) x = sum c x - sum z x.
//     int4: nibbles 0-4 of a word are masked in place, nibbles 5-7 after one
//     shift by 12; int8 (two's complement): the sign bits are flipped once per
//     word (c + 128), bytes 0-1 in place, bytes 2-3 after one shift; int2:
//     fields 0-10 in place, 11-15 after one shift; f32 weights FFMA directly.
//     That is one AND and one FFMA per weight, plus a shift per word.
//
// Data movement: a unit is 8 weight rows x 512 bytes.  Every consumer warp
// reads its units from its own ring of DEPTH shared-memory stages, each filled
// by one 2-D TMA copy (cp.async.bulk.tensor) with full / empty mbarrier
// pairs.  One extra producer warp issues all copies: its lane c feeds consumer
// warp c, first one unit per ring before the dependency wait (weights are
// read-only), the rest once x is staged, then a refill whenever a stage is
// handed back.  The consumers only wait, compute and release.
// In a unit, lane l takes 16-byte chunk l of all 8 rows (a warp-wide load
// reads one row's 512 contiguous bytes), so the x values it loads from shared
// memory serve 8 rows; x is staged lane-interleaved so those loads are
// conflict-free.  The units of a CTA are split into contiguous runs, one per
// warp, in row-group-major order (even shares per warp, or shares weighted by
// the warps on each scheduler for quantized four-token launches, whose 10 or
// 11 warps sit unevenly on the four schedulers); a warp keeps its sums in
// registers across the segments of a row group and combines its lanes (butterfly
// reduce-scatter) only when its row group changes.  The per-warp partial
// sums of each row group are added in warp order after the run, in rounds of
// at most 16 row groups.  Persistent CTAs own contiguous runs of row groups.
// Every mbarrier wait is bounded; a wait that gives up records
// B200Q_ETIMEOUT in a device word (b200q_device_status), drains the warp's
// copies in flight and returns.
//
// Accuracy: per lane and row group, f32 FFMA chains over the lane's chunks,
// then fixed-order f32 additions; with the zero point taken out by the
// identical chain the result stays within 1e-5 of sum |scale * deq * x| on
// the workloads' distributions and is exact where every code is the zero
// point.
#include <climits>
#include <cstring>

#include "qwq_internal.h"

namespace qwq {
namespace {

constexpr int kMaxWarps = 16;
// Consumer warps of a variant (measured on the format sweep):
//   * f32 and int8, one token: 16 (under the 120 registers 17 warps allow);
//     their rings drop to 2 stages to make room, which these formats
//     tolerate (more weight bytes per instruction);
//   * int4 and int2, one token: 15 with 3-stage rings (the integer-bound
//     formats lose more from the shallower ring than they gain from the
//     sixteenth warp);
//   * two tokens: 15, or 11 with group-wise scales (a second set of sums,
//     no spills); for int4 and int2 their larger staged x is paid for with a
//     ring stage, for f32 and int8 with warps.
//   * four tokens (per-row scales, f32 / int8 / int4): four sets of sums and
//     the staged x of four tokens per word; 11 warps (f32, int8), 10 (int4).
//     int2 keeps launches of two: its 16 codes per word spill at four.
template <int FMT, int NS, int GW>
constexpr int max_warps() {
    return NS == 4   ? (FMT == B200Q_I4 ? 10 : 11)
           : NS == 2 ? (GW ? 11 : 15)
                     : (FMT == B200Q_F32 || FMT == B200Q_I8) ? 16 : 15;
}
// Whether a launch that does not fit gives up a ring stage before a warp:
// one token for f32 / int8, two tokens for int4 / int2.
template <int FMT, int NS>
constexpr bool stage_before_warp() { return (NS == 1) == (FMT == B200Q_F32 || FMT == B200Q_I8); }
constexpr int kMaxSets = B200Q_GROUP_MAX;  // tensors per launch
constexpr int kSeg = 512;            // bytes per row per stage: 32 lanes x 16 B
constexpr int kStage = 8 * kSeg;     // one stage: 8 rows x 512 B (one TMA box)
constexpr int kRound = 16;           // row groups combined per round
constexpr int kXB = 16;              // x elements per thread per staging batch
constexpr size_t kSmemMax = 220 * 1024;
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s bound on any wait

__device__ unsigned int g_decode_err = 0;

template <int FMT>
struct F;
// E: elements per 16-byte chunk; ZW (quantized formats): a code word whose
// every code is the zero point (int8: the byte 0, i.e. 128 after the sign flip)
template <>
struct F<B200Q_F32> {
    static constexpr int E = 4;
};
template <>
struct F<B200Q_I8> {
    static constexpr int E = 16;
    static constexpr uint32_t ZW = 0x00000000u;
};
template <>
struct F<B200Q_I4> {
    static constexpr int E = 32;
    static constexpr uint32_t ZW = 0x88888888u;
};
template <>
struct F<B200Q_I2> {
    static constexpr int E = 64;
    static constexpr uint32_t ZW = 0xAAAAAAAAu;
};

// Bit offset b of element e (0 <= e < 32 / bits) inside its extracted word:
// the value of the masked code is code * 2^b * 2^-149.
template <int FMT>
__device__ __forceinline__ int bit_offset(int e);
template <>
__device__ __forceinline__ int bit_offset<B200Q_F32>(int) { return 0; }
template <>
__device__ __forceinline__ int bit_offset<B200Q_I8>(int e) { return 8 * (e & 1); }               // 2,3: >> 16
template <>
__device__ __forceinline__ int bit_offset<B200Q_I4>(int e) { return e < 5 ? 4 * e : 4 * (e - 3); }  // 5-7: >> 12
template <>
__device__ __forceinline__ int bit_offset<B200Q_I2>(int e) { return e < 11 ? 2 * e : 2 * (e - 11); }  // >> 22

// The EW codes of one 32-bit word as exact subnormal f32 (code * 2^b * 2^-149).
template <int FMT, int EW>
__device__ __forceinline__ void word_codes(uint32_t w, float (&d)[EW]) {
    if (FMT == B200Q_I8) {
        const uint32_t u = w ^ 0x80808080u;  // two's complement -> code + 128
        const uint32_t v = u >> 16;
        d[0] = __uint_as_float(u & 0xFFu);
        d[1] = __uint_as_float(u & 0xFF00u);
        d[2] = __uint_as_float(v & 0xFFu);
        d[3] = __uint_as_float(v & 0xFF00u);
    } else if (FMT == B200Q_I4) {
        const uint32_t v = w >> 12;
#pragma unroll
        for (int e = 0; e < 5; ++e) d[e] = __uint_as_float(w & (0xFu << (4 * e)));
#pragma unroll
        for (int e = 5; e < 8; ++e) d[e] = __uint_as_float(v & (0xFu << (4 * (e - 3))));
    } else if (FMT == B200Q_I2) {
        const uint32_t v = w >> 22;
#pragma unroll
        for (int e = 0; e < 11; ++e) d[e] = __uint_as_float(w & (0x3u << (2 * e)));
#pragma unroll
        for (int e = 11; e < 16; ++e) d[e] = __uint_as_float(v & (0x3u << (2 * (e - 11))));
    }
}

// acc[t] += codes of word w times the staged x pairs, two products per
// packed FP32x2 FMA (the even and odd elements of a pair accumulate in .x
// and .y).
template <int FMT, int NS, int EW>
__device__ __forceinline__ void word_fma2(uint32_t w, const float2 (&xv)[NS * EW / 2], float2 (&acc)[NS]) {
    float d[EW];
    word_codes<FMT, EW>(w, d);
#pragma unroll
    for (int t = 0; t < NS; ++t)
#pragma unroll
        for (int i = 0; i < EW / 2; ++i)
            acc[t] = __ffma2_rn(make_float2(d[2 * i], d[2 * i + 1]), xv[t * (EW / 2) + i], acc[t]);
}

// ---- mbarrier / bulk-copy helpers (PTX ISA: mbarrier, cp.async.bulk)

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
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

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
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
        if ((it & 255) == 255 && global_ns() - t0 > limit_ns) return false;
    }
}

// floor(log2 m) for finite m > 0, subnormals included (from the bits).
__device__ __forceinline__ int ilogb_bits(float m) {
    const int b = __float_as_int(m);
    const int e = (b >> 23) & 0xFF;
    return e ? e - 127 : -118 - __clz(b);
}

// 2^k exactly, for -149 <= k <= 127.
__device__ __forceinline__ float pow2i(int k) {
    return k >= -126 ? __int_as_float((k + 127) << 23) : __int_as_float(1 << (k + 149));
}

// Per-token power-of-two factors of the staged x (see the staging code).
struct TokScale {
    float s1, s2;        // x * 2^k = (x * s1) * s2
    float u1, u2;        // 2^-T = u1 * u2
};

// Non-blocking probe of a phase (true once it has completed).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Barrier among the first n threads of the block (the consumer warps),
// which leaves the producer warp out.
__device__ __forceinline__ void consumers_sync(int n) { asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory"); }

// Butterfly reduce-scatter of N values (N a power of two <= 32) over the 32
// lanes: afterwards every lane holds the full sum of value index
// lane >> (5 - log2 N) (lanes that differ only in the low bits hold the same).
template <int N>
__device__ __forceinline__ float reduce_scatter(float (&v)[N], int lane) {
    int n = N;
    int off = 16;
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        if (n > 1) {
            const int h = n / 2;
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                if (i < h) {
                    const float send = upper ? v[i] : v[i + h];
                    const float keep = upper ? v[i + h] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
            n = h;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
        }
        off >>= 1;
    }
    return v[0];
}

// Division by a launch constant d >= 1 as a multiply and a shift, exact for
// dividends 0 <= n < 2^31: with s = ceil(log2 d) and m = ceil(2^(31+s) / d),
// n m / 2^(31+s) = n / d + e with 0 <= e < n / 2^(31+s) < 2^-s <= 1/d, which
// is below the gap from n / d up to the next integer.
struct FastDiv {
    uint32_t m;
    int sh;                   // 31 + s
};

inline FastDiv make_fastdiv(uint32_t d) {
    int s = 0;
    while ((1ull << s) < d) ++s;
    return FastDiv{(uint32_t)(((1ull << (31 + s)) + d - 1) / d), 31 + s};
}

__device__ __forceinline__ int fdiv(int n, const FastDiv &f) {
    return (int)(((unsigned long long)(unsigned)n * f.m) >> f.sh);
}

// One launch: nsets weight tensors ("sets") of one format and one I.  The
// row groups of all sets are numbered consecutively (set j owns
// [rg_start[j], rg_start[j+1])); CTAs own contiguous runs of that numbering,
// so a CTA's rows may span several sets.  Sets that read the same x share an
// x slot: slots are numbered in set order, a new slot wherever a set's input
// differs from the previous set's, and a CTA stages the slots of its sets.
template <int MS>
struct DecParams {
    CUtensorMap map[MS];      // decode tensor map of each set
    CUtensorMap smap[MS];     // group-scale tensor map of each set (group-wise scales)
    const float *scales[MS];
    float *y[MS];             // [S, O[j]] per set, at this launch's first token
    const float *xa[MS];      // per x slot: x, or g when silu(g) * u is staged
    const float *xb[MS];      // per x slot: u when silu(g) * u is staged
    int rg_start[MS + 1];     // first row group of each set; rg_start[nsets] = n_rg
    int O[MS];
    int xslot[MS];            // x slot of each set, nondecreasing
    int nsets;
    int silu;                 // stage silu(xa) * xb instead of xa
    int I;                    // elements per x row (also the row stride of x)
    int ld;                   // device row stride in bytes
    int row_bytes;            // bytes per row per stage: min(512, ld)
    int k_pad;                // elements per padded row
    int n_rg;                 // total row groups
    int depth;                // stages per warp
    int round_rgs;            // row groups combined per round (partials buffer rows)
    int nx_max;               // most x slots any CTA stages (shared-memory layout)
    int gbox;                 // group scales per row in a stage (group-wise scales)
    FastDiv div_grid, div_nseg;   // by gridDim.x, the segments per row
    FastDiv div_gs;           // by the group size (group-wise scales)
};

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// GW = 0: one scale per row, applied once per output.  GW > 0: group-wise
// scales; a group spans GW 32-bit words of a 16-byte chunk (GW = 1 or 2), or
// whole chunks (GW = 4).  Each lane then sums every group's products on their
// own (zero point taken out as above), multiplies the group sum by the group's
// scale and adds it to the row's sum; the producer copies each stage's
// scales (8 rows x gbox, from a 4-aligned first group) next to its codes.
template <int FMT, int NS, int MS, int GW>
__global__ void __launch_bounds__((max_warps<FMT, NS, GW>() + 1) * 32, 1)
    qmv_decode_kernel(const __grid_constant__ DecParams<MS> p) {
    constexpr int E = F<FMT>::E;
    constexpr int SEGE = (kSeg / 16) * E;            // elements of a row in one stage
    constexpr int bits = FMT == B200Q_F32 ? 32 : FMT == B200Q_I8 ? 8 : FMT == B200Q_I4 ? 4 : 2;
    constexpr int EW = 32 / bits;                    // elements per 32-bit word
    // four tokens with per-row scales: the unrolled body of a stage outgrows
    // the instruction cache (no_instruction stalls led), so its four words
    // run as a loop (measured slower at one and two tokens)
    constexpr bool kRollQ = FMT != B200Q_F32 && NS >= 4 && GW == 0;
    constexpr int NV = 8 * NS;                       // partial sums per lane and row group
    extern __shared__ __align__(128) uint8_t smem[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nw = (blockDim.x >> 5) - 1;            // consumer warps; warp nw copies the weights
    const int nct = nw * 32;                          // consumer threads
    const int depth = p.depth;
    const int nseg = (p.ld + kSeg - 1) / kSeg;
    const int rb = p.row_bytes;                       // smem row pitch of a stage
    // elements staged per token: whole segments (the lane-interleaved layout
    // addresses every lane slot of a segment), or k_pad for f32
    const int k_alloc = FMT == B200Q_F32 ? p.k_pad : nseg * (kSeg / 4) * EW;
    const int nxr = p.nx_max * NS;                    // staged x rows (slot-major)
    const int scb = GW ? 32 * p.gbox : 0;             // group-scale bytes per stage (8 rows x gbox f32)
    const int stg = kStage + scb;                     // bytes per ring stage

    // shared memory: x' [nx_max][NS][k_alloc] | rings [nw][depth] | full and
    // empty mbarriers [2][nw][depth] + x-staged + x-issued | partials | per-row unscale
    // factors | max scratch | 16 spare bytes | row scales
    float *xs = reinterpret_cast<float *>(smem);
    uint8_t *ring = smem + (size_t)4 * nxr * k_alloc;
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + (size_t)nw * depth * stg);
    const int kR = p.round_rgs;
    float *part = reinterpret_cast<float *>(bars + 2 * nw * depth + 2);  // [kR][nw][NS][8]
    float *unscale = part + (size_t)kR * nw * NS * 8;                  // [nxr][2]: 2^-T as two factors
    float *red = unscale + 2 * nxr;                                    // [nxr][kMaxWarps]
    float *row_scale = red + nxr * kMaxWarps + 4;                     // [rows of this CTA]
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + nw * depth);
    const uint32_t x_ready = smem_u32(bars + 2 * nw * depth);   // completes once x is staged
    const uint32_t x_issued = smem_u32(bars + 2 * nw * depth + 1);  // once every consumer warp's x loads are out

    // (32-bit products: the host keeps grid * n_rg and nw * round units below 2^31)
    const int rg0 = fdiv(blockIdx.x * p.n_rg, p.div_grid);
    const int rg1 = fdiv((blockIdx.x + 1) * p.n_rg, p.div_grid);
    // set of row group rg, scanning forward from set s (rg never decreases
    // along a scan)
    auto set_of = [&](int rg, int s) {
        while (s + 1 < p.nsets && rg >= p.rg_start[s + 1]) ++s;
        return s;
    };
    const int s_lo = set_of(rg0, 0), s_hi = set_of(rg1 - 1, s_lo);
    const int slot_lo = p.xslot[s_lo];
    const int nx = p.xslot[s_hi] - slot_lo + 1;       // x slots this CTA stages

    // Consumer warp c's units: in round r (row groups [rg0 + kR r, ...)), a
    // contiguous run of the round's U = rows * nseg units, row-group-major
    // ([c U / nw, (c + 1) U / nw), or by scheduler weights, run_of below).
    // A cursor walks them in order across rounds.
    struct Cursor {
        int round_base, round_end;   // row groups of the current round
        int u, u_end;                // unit index within the round's run
        int rgl, sg;                 // u = rgl * nseg + sg
    };
    // Quantized four-token launches share a round's units out by the warps'
    // schedulers (warp % 4). Measured per-scheduler finish times fit a throughput of
    // n / (n + 1) for n consumer warps on a scheduler (3 warps: 0.94 and
    // 2 warps: 0.87 of a full scheduler's rate), so each warp's weight is
    // 60 / (n + 1). Even shares per warp left the 3-warp schedulers of a
    // 10-warp launch (3, 3, 2, 2) with 30% more work than the rest.
    // wcum(w): the weights of the warps below w.
    auto wcum = [&](int w) {
        int c = 0;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const int n_on = (nw - s + 3) >> 2;
            const int below = w > s ? (w - s + 3) >> 2 : 0;
            c += below * (n_on >= 4 ? 12 : n_on == 3 ? 15 : n_on == 2 ? 20 : 30);
        }
        return c;
    };
    auto run_of = [&](Cursor &c, int base, int w) {
        c.round_base = base;
        c.round_end = base + kR < rg1 ? base + kR : rg1;
        const int U = (c.round_end - c.round_base) * nseg;
        // only the quantized four-token launches (10 or 11 warps, bound by
        // the FMA pipe) take the scheduler weights; at 15 or 16 warps even
        // shares per warp measured 1-2% faster, f32 streams at a rate set by
        // each warp's ring (f32 8192^2 S = 8: 100 against 112 us weighted),
        // and the two-token group-scale builds (at the register limit) would
        // spill for them
        constexpr bool kEven = GW || NS < 4 || FMT == B200Q_F32;
        const int wtot = wcum(nw);   // recomputed here rather than held across the main loop
        c.u = kEven ? w * U / nw : U * wcum(w) / wtot;
        c.u_end = kEven ? (w + 1) * U / nw : U * wcum(w + 1) / wtot;
        c.rgl = fdiv(c.u, p.div_nseg);
        c.sg = c.u - c.rgl * nseg;
    };
    auto advance = [&](Cursor &c) {
        ++c.u;
        if (++c.sg == nseg) {
            c.sg = 0;
            ++c.rgl;
        }
    };

    if (tid <= s_hi - s_lo) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.map[s_lo + tid])) : "memory");
        if (GW)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.smap[s_lo + tid])) : "memory");
    }
    if (tid < nxr) reinterpret_cast<unsigned *>(red)[tid] = 0u;   // row maxima of x (atomicMax)
    if (warp == nw && lane < nw) {
        for (int b = 0; b < depth; ++b) {
            mbar_init(full0 + 8 * (lane * depth + b), 1);
            mbar_init(empty0 + 8 * (lane * depth + b), 1);
        }
        if (lane == 0) {
            mbar_init(x_ready, 1);
            mbar_init(x_issued, nw);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == nw) {
        // ---- producer: lane c keeps consumer warp c's ring full.  Weights
        // are read-only, so the first unit of every ring goes out at once,
        // before the dependency wait the consumers make; the rest of the
        // rings fill once x is staged (x's loads must not queue behind them).
        const unsigned pmask = __ballot_sync(0xffffffffu, lane < nw);
        if (lane >= nw) return;
        const uint64_t policy = evict_first_policy();
        Cursor pc;
        run_of(pc, rg0, lane);
        auto next = [&]() {          // skip empty runs; false when past the last round
            while (pc.u >= pc.u_end) {
                if (pc.round_end >= rg1) return false;
                run_of(pc, pc.round_end, lane);
            }
            return true;
        };
        int ps = 0, pset = s_lo;
        uint32_t eph = 0;
        const uint32_t my_full = full0 + 8 * lane * depth, my_empty = empty0 + 8 * lane * depth;
        auto issue = [&]() {
            const int rg = pc.round_base + pc.rgl;
            pset = set_of(rg, pset);
            const uint32_t bar = my_full + 8 * ps;
            const uint32_t dst = smem_u32(ring + ((size_t)lane * depth + ps) * stg);
            mbar_expect_tx(bar, (uint32_t)(8 * rb + scb));
            tma_load_2d(dst, &p.map[pset], pc.sg * (kSeg / 4), (rg - p.rg_start[pset]) * 8, bar, policy);
            if (GW)   // this stage's group scales, from the first group rounded down to 16 bytes
                tma_load_2d(dst + kStage, &p.smap[pset], fdiv(pc.sg * SEGE, p.div_gs) & ~3,
                            (rg - p.rg_start[pset]) * 8, bar, policy);
            advance(pc);
            if (++ps == depth) {
                ps = 0;
                eph ^= 1;
            }
        };
        bool more = next();
        if (more) {
            issue();
            more = next();
        }
        // the rest of the rings go out once the consumers' loads of x have
        // been issued, so that x does not return behind them; the weights
        // then stream while x is staged
        if (!mbar_wait(x_issued, 0, kWaitNs)) more = false;   // the consumers report the same timeout
        for (int k = 1; k < depth && more; ++k) {
            issue();
            more = next();
        }
        eph = 0;                     // the first refill of each stage waits for its first release
        unsigned long long t0 = global_ns();
        while (__any_sync(pmask, more)) {
            bool progressed = false;
            if (more && mbar_test(my_empty + 8 * ps, eph)) {
                issue();
                more = next();
                progressed = true;
            }
            if (__any_sync(pmask, progressed)) {
                t0 = global_ns();
                continue;
            }
            // nothing was released: back off; lane 0 decides, for all lanes,
            // when the consumers have stopped releasing stages
            const bool late = global_ns() - t0 > kWaitNs;
            if (__shfl_sync(pmask, late ? 1 : 0, 0)) {
                if (more) atomicExch(&g_decode_err, (unsigned)(-B200Q_ETIMEOUT));
                break;
            }
            __nanosleep(64);
        }
        return;
    }

    // ---- consumers
    // the row scales are read-only too: start loading this CTA's now (kept
    // in registers, written to shared memory once x is staged)
    auto scale_of = [&](int r) {
        const int rg = rg0 + (r >> 3);
        const int s = set_of(rg, s_lo);
        const int o = (rg - p.rg_start[s]) * 8 + (r & 7);
        return o < p.O[s] ? p.scales[s][o] : 0.f;
    };
    // a volatile load stays here, ahead of the dependency wait, instead of
    // being scheduled next to its use after x is staged
    auto scale_early = [&](int r) {
        const int rg = rg0 + (r >> 3);
        const int s = set_of(rg, s_lo);
        const int o = (rg - p.rg_start[s]) * 8 + (r & 7);
        float v = 0.f;
        if (o < p.O[s]) asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p.scales[s] + o));
        return v;
    };
    constexpr int kSc = 4;
    float sc_reg[kSc];
#pragma unroll
    for (int i = 0; i < kSc; ++i) {
        const int r = i * nct + tid;
        sc_reg[i] = !GW && r < (rg1 - rg0) * 8 ? scale_early(r) : 0.f;
    }

    // round-0 partials start at zero (warps that touch no unit of a row group
    // leave 0)
    for (int i = tid; i < kR * nw * NS * 8; i += nct) part[i] = 0.f;

    // Everything above touched only the weights, which no kernel writes; x
    // (and y) may be written (read) by the kernel before this one in the
    // stream, so wait for it here (programmatic dependent launch), and let
    // the next kernel in the stream start its own weight prefetch.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // one staged input value: x, or silu(g) * u
    auto xval = [&](int j, int t, int k) {
        const long long off = (long long)t * p.I + k;
        if (k >= p.I) return 0.f;
        const float a = p.xa[slot_lo + j][off];
        return p.silu ? silu_f(a) * p.xb[slot_lo + j][off] : a;
    };

    // ---- stage x.  Quantized formats: 16-byte slot d of the lane-interleaved
    // layout [seg][word q][quad e4][lane][4] holds elements (e4*4 .. e4*4+3) of
    // word q of chunk c = seg * 32 + lane, 4 consecutive elements of x, so each
    // thread gathers its slots' 16-byte groups of x into registers (one round
    // trip), the per-token max of |x| comes from them, and they are stored as
    //     x' = (x * 2^(T + 23)) * 2^(126 - b),  b = the code's bit offset,
    // two exact power-of-two products per element.  f32 weights: x as is.
    const int nthr = nct;
    constexpr int Q4 = EW >= 4 ? EW / 4 : 1;      // quads per word (quantized formats)
    const int n_chunks = p.ld / 16;
    const int n_slots = nseg * 4 * Q4 * 32;
    const bool vec = (p.I & 3) == 0;
    auto slot_src = [&](int d) {                  // first x element of slot d, or -1 past the row
        const int ln = d & 31, rest = d >> 5;
        const int e4 = rest % Q4, q = (rest / Q4) & 3, seg = (rest / Q4) >> 2;
        const int c = seg * 32 + ln;
        return c < n_chunks ? c * E + q * EW + e4 * 4 : -1;
    };
    auto ld4 = [&](const float *r, int k0) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (vec && k0 + 3 < p.I) return *reinterpret_cast<const float4 *>(r + k0);
        v.x = k0 < p.I ? r[k0] : 0.f;
        v.y = k0 + 1 < p.I ? r[k0 + 1] : 0.f;
        v.z = k0 + 2 < p.I ? r[k0 + 2] : 0.f;
        v.w = k0 + 3 < p.I ? r[k0 + 3] : 0.f;
        return v;
    };
    auto gather = [&](int j, int t, int k0) {
        if (k0 < 0) return make_float4(0.f, 0.f, 0.f, 0.f);
        const long long off = (long long)t * p.I;
        float4 v = ld4(p.xa[slot_lo + j] + off, k0);
        if (p.silu) {
            const float4 u = ld4(p.xb[slot_lo + j] + off, k0);
            v = make_float4(silu_f(v.x) * u.x, silu_f(v.y) * u.y, silu_f(v.z) * u.z, silu_f(v.w) * u.w);
        }
        return v;
    };
    auto absmax4 = [](float4 v) { return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))); };
    // 2^(126 - b) for element i of quad e4 (a constant once both are known)
    auto post = [](int e4, int i) { return __int_as_float((253 - bit_offset<FMT>(e4 * 4 + i)) << 23); };
    auto put = [&](float *dst, int d, float4 v, const TokScale &ts) {
        const int e4 = (d >> 5) % Q4;
        float4 f = make_float4(post(0, 0), post(0, 1), post(0, 2), post(0, 3));
#pragma unroll
        for (int qq = 1; qq < Q4; ++qq)
            if (e4 == qq) f = make_float4(post(qq, 0), post(qq, 1), post(qq, 2), post(qq, 3));
        if (ts.s1 != 1.f) {                       // largest |x| subnormal: 2^k in two factors
            v.x *= ts.s1;
            v.y *= ts.s1;
            v.z *= ts.s1;
            v.w *= ts.s1;
        }
        v.x = (v.x * ts.s2) * f.x;
        v.y = (v.y * ts.s2) * f.y;
        v.z = (v.z * ts.s2) * f.z;
        v.w = (v.w * ts.s2) * f.w;
        reinterpret_cast<float4 *>(dst)[d] = v;
    };
    // With max |x| in [2^E, 2^(E+1)) and k = -E, x * 2^k stays below 2 and
    // the products code * x * 2^T, T = k - 23, below 2^-14.  2^k needs two
    // factors when max |x| is subnormal (k up to 149), and so does 2^-T
    // when max |x| >= 2^105.  Every factor is an exact power of two.
    auto tok_scale_k = [](int k) {
        TokScale r;
        const int ku = 23 - k;
        r.u1 = ku > 127 ? pow2i(64) : 1.f;
        r.u2 = pow2i(ku > 127 ? ku - 64 : ku);
        r.s1 = k > 127 ? pow2i(64) : 1.f;
        r.s2 = pow2i(k > 127 ? k - 64 : k);
        return r;
    };
    auto tok_scale = [&](float mt) { return tok_scale_k(mt > 0.f ? -ilogb_bits(mt) : 0); };
    // x slots per thread per round trip of the batched staging below, and
    // whether x_issued is signalled as soon as x's loads are out: only on the
    // one-slot path of kXB / 4 slots per thread.  Elsewhere it comes with
    // x_ready: the rest of the weight rings then go out after x is staged,
    // which measured faster (int4 8192^2: 11.7 against 13.0 us).
    constexpr int kG = 5;
    const bool x_issued_early = FMT != B200Q_F32 && nx == 1 && n_slots <= (kXB / 4) * nthr;
    if constexpr (FMT == B200Q_F32) {
        for (int j = 0; j < nx; ++j)
            for (int base = 0; base < p.k_pad; base += kXB * nthr) {
                float v[NS][kXB];                     // all loads of a batch in flight at once
#pragma unroll
                for (int t = 0; t < NS; ++t)
#pragma unroll
                    for (int jj = 0; jj < kXB; ++jj) v[t][jj] = xval(j, t, base + jj * nthr + tid);
#pragma unroll
                for (int t = 0; t < NS; ++t)
#pragma unroll
                    for (int jj = 0; jj < kXB; ++jj) {
                        const int k = base + jj * nthr + tid;
                        if (k < p.k_pad) xs[(size_t)(j * NS + t) * k_alloc + k] = v[t][jj];
                    }
            }
        if (tid < 2 * nxr) unscale[tid] = 1.f;
    } else {
        // First pass: every row with the fixed exponent k = -20, exact for
        // rows whose largest |x| lies in [2^-20, 2^20) (or that are all zero);
        // the largest |x| of each row is gathered on the side (atomicMax on
        // the bits of non-negative floats) and checked after the barrier.
        constexpr int kFix = -20;
        const TokScale ts_fix = tok_scale_k(kFix);
        unsigned *tokmax = reinterpret_cast<unsigned *>(red);   // [nxr], zeroed before the first barrier
        auto note_max = [&](int row, float mt) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
            if (lane == 0) atomicMax(tokmax + row, __float_as_uint(mt));
        };
        constexpr int kG1 = kXB / 4;
        if (nx == 1 && n_slots <= kG1 * nthr) {
            // one x slot in one round trip of kG1 slots per thread: every load
            // of the thread in flight at once (measured 1% faster at one token
            // than the batched form below)
            float4 held[NS][kG1];
#pragma unroll
            for (int t = 0; t < NS; ++t)
#pragma unroll
                for (int g = 0; g < kG1; ++g) {
                    const int d = g * nthr + tid;
                    held[t][g] = d < n_slots ? gather(0, t, slot_src(d)) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            __syncwarp();
            if (lane == 0) mbar_arrive(x_issued);
#pragma unroll
            for (int t = 0; t < NS; ++t) {
                float mt = 0.f;
#pragma unroll
                for (int g = 0; g < kG1; ++g) {
                    const int d = g * nthr + tid;
                    mt = fmaxf(mt, absmax4(held[t][g]));
                    if (d < n_slots) put(xs + (size_t)t * k_alloc, d, held[t][g], ts_fix);
                }
                note_max(t, mt);
            }
        } else if constexpr (NS >= 2 && GW != 0) {
            // two tokens with group scales (no registers to spare): a loop
            // over each token's slots, four loads in flight
            for (int j = 0; j < nx; ++j)
#pragma unroll
                for (int t = 0; t < NS; ++t) {
                    float *dst = xs + (size_t)(j * NS + t) * k_alloc;
                    float mt = 0.f;
#pragma unroll 4
                    for (int d = tid; d < n_slots; d += nthr) {
                        const float4 v = gather(j, t, slot_src(d));
                        mt = fmaxf(mt, absmax4(v));
                        put(dst, d, v, ts_fix);
                    }
                    note_max(j * NS + t, mt);
                }
        } else
        // Batches of kG slots per thread and token, every load of a batch in
        // flight at once: one round trip to L2 per batch.
        for (int j = 0; j < nx; ++j) {
            float mt[NS];
#pragma unroll
            for (int t = 0; t < NS; ++t) mt[t] = 0.f;
            for (int b0 = 0; b0 < n_slots; b0 += kG * nthr) {
                float4 held[NS][kG];
#pragma unroll
                for (int t = 0; t < NS; ++t)
#pragma unroll
                    for (int g = 0; g < kG; ++g) {
                        const int d = b0 + g * nthr + tid;
                        held[t][g] = d < n_slots ? gather(j, t, slot_src(d)) : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                for (int t = 0; t < NS; ++t)
#pragma unroll
                    for (int g = 0; g < kG; ++g) {
                        const int d = b0 + g * nthr + tid;
                        mt[t] = fmaxf(mt[t], absmax4(held[t][g]));
                        if (d < n_slots) put(xs + (size_t)(j * NS + t) * k_alloc, d, held[t][g], ts_fix);
                    }
            }
#pragma unroll
            for (int t = 0; t < NS; ++t) note_max(j * NS + t, mt[t]);
        }
        if (tid < nxr) {
            unscale[2 * tid] = ts_fix.u1;
            unscale[2 * tid + 1] = ts_fix.u2;
        }
    }
#pragma unroll
    for (int i = 0; i < kSc; ++i)
        if (i * nct + tid < (rg1 - rg0) * 8) row_scale[i * nct + tid] = sc_reg[i];
    if (!GW)
        for (int r = kSc * nct + tid; r < (rg1 - rg0) * 8; r += nct) row_scale[r] = scale_of(r);  // tall CTAs
    consumers_sync(nct);
    if constexpr (FMT != B200Q_F32) {
        // rows outside the fixed exponent's range: staged again with their own
        // exponent (every thread reads the same maxima, so the branch is uniform)
        const unsigned *tokmax = reinterpret_cast<const unsigned *>(red);
        auto in_range = [](float mt) { return mt == 0.f || (mt >= 0x1p-20f && mt < 0x1p20f); };
        bool redo = false;
        for (int r = 0; r < nx * NS; ++r) redo |= !in_range(__uint_as_float(tokmax[r]));
        if (redo) {
            for (int j = 0; j < nx; ++j)
                for (int t = 0; t < NS; ++t) {
                    const int row = j * NS + t;
                    const float mt = __uint_as_float(tokmax[row]);
                    if (in_range(mt)) continue;
                    const TokScale ts = tok_scale(mt);
                    if (tid == 0) {
                        unscale[2 * row] = ts.u1;
                        unscale[2 * row + 1] = ts.u2;
                    }
                    float *dst = xs + (size_t)row * k_alloc;
                    for (int d = tid; d < n_slots; d += nct) put(dst, d, gather(j, t, slot_src(d)), ts);
                }
            consumers_sync(nct);
        }
    }
    if (tid == 0) mbar_arrive(x_ready);
    if (!x_issued_early && lane == 0) mbar_arrive(x_issued);

    // ---- main loop
    const uint32_t my_full = full0 + 8 * warp * depth, my_empty = empty0 + 8 * warp * depth;
    const uint8_t *my_ring = ring + (size_t)warp * depth * stg;
    Cursor cc;
    int c_stage = 0, cset = s_lo;
    uint32_t c_phase = 0;
    bool ok = true;
    const float *xsb = xs;                            // x' rows of the current set's slot
    // per-row scales: a2 / az run across the row group's units; group-wise
    // scales: a2 / az hold one group, a1 the row group's scaled group sums
    float2 a2[8][NS], az[NS];
    float a1[8][NS];
    auto clear_group = [&]() {
#pragma unroll
        for (int t = 0; t < NS; ++t) {
            az[t] = make_float2(0.f, 0.f);
#pragma unroll
            for (int r = 0; r < 8; ++r) a2[r][t] = make_float2(0.f, 0.f);
        }
    };
    auto clear_acc = [&]() {
        clear_group();
#pragma unroll
        for (int t = 0; t < NS; ++t)
#pragma unroll
            for (int r = 0; r < 8; ++r) a1[r][t] = 0.f;
    };
    // a group's sums, times its scales (ssc: the stage's scales at the group's column)
    auto fold_group = [&](const float *ssc) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const float g = ssc[r * p.gbox];
#pragma unroll
            for (int t = 0; t < NS; ++t)
                a1[r][t] = fmaf(g, FMT == B200Q_F32 ? a2[r][t].x + a2[r][t].y
                                                    : (a2[r][t].x - az[t].x) + (a2[r][t].y - az[t].y),
                                a1[r][t]);
        }
        clear_group();
    };
    // lane sums of the current row group -> part[rgl][warp]
    auto flush = [&](int rgl) {
        float v[NV];
#pragma unroll
        for (int t = 0; t < NS; ++t)
#pragma unroll
            for (int r = 0; r < 8; ++r)
                v[t * 8 + r] = GW ? a1[r][t]
                                  : FMT == B200Q_F32 ? a2[r][t].x + a2[r][t].y
                                                     : (a2[r][t].x - az[t].x) + (a2[r][t].y - az[t].y);
        const float sum = reduce_scatter<NV>(v, lane);
        constexpr int sh = NS == 4 ? 0 : NS == 2 ? 1 : 2;   // this lane holds value index lane >> sh
        const int idx = lane >> sh;
        if ((lane & ((1 << sh) - 1)) == 0) part[(((size_t)rgl * nw + warp) * NS + idx / 8) * 8 + (idx & 7)] = sum;
        clear_acc();
    };
    clear_acc();

    // A warp whose wait gave up keeps walking the rounds without work, so
    // that every consumer still reaches each round's barriers.
    for (int base = rg0; base < rg1; base += kR) {
        const int rend = base + kR < rg1 ? base + kR : rg1;
        const bool last_round = rend >= rg1;
        if (base != rg0) {
            // zero this round's partials (round 0 was zeroed in the prologue)
            for (int i = tid; i < kR * nw * NS * 8; i += nct) part[i] = 0.f;
            consumers_sync(nct);
        }
        run_of(cc, base, warp);
        int cur_rgl = -1;
        for (; ok && cc.u < cc.u_end; advance(cc)) {
            if (!mbar_wait(my_full + 8 * c_stage, c_phase, kWaitNs)) {
                ok = false;
                break;
            }
            const int rgl = cc.rgl, sg = cc.sg;
            if (rgl != cur_rgl) {
                if (cur_rgl >= 0) flush(cur_rgl);
                cur_rgl = rgl;
                cset = set_of(base + rgl, cset);
                xsb = xs + (size_t)(p.xslot[cset] - slot_lo) * NS * k_alloc;
            }
            const int chunks = (p.ld - sg * kSeg < kSeg ? p.ld - sg * kSeg : kSeg) / 16;
            if (lane < chunks) {
                const uint8_t *st = my_ring + (size_t)c_stage * stg + lane * 16;
                // group-wise scales: this lane's first group, as a column of the stage's scales
                const float *ssc = nullptr;
                if (GW)
                    ssc = reinterpret_cast<const float *>(my_ring + (size_t)c_stage * stg + kStage) +
                          (fdiv(sg * SEGE + lane * E, p.div_gs) - (fdiv(sg * SEGE, p.div_gs) & ~3));
                uint4 cw[8];
                if constexpr (!kRollQ) {
#pragma unroll
                    for (int r = 0; r < 8; ++r) cw[r] = *reinterpret_cast<const uint4 *>(st + r * rb);
                }
                if constexpr (FMT == B200Q_F32) {
                    const int k0 = (sg * (kSeg / 16) + lane) * E;
#pragma unroll
                    for (int t = 0; t < NS; ++t) {
                        const float4 xf = *reinterpret_cast<const float4 *>(xsb + (size_t)t * k_alloc + k0);
#pragma unroll
                        for (int r = 0; r < 8; ++r) {
                            a2[r][t] = __ffma2_rn(make_float2(__uint_as_float(cw[r].x), __uint_as_float(cw[r].y)),
                                                  make_float2(xf.x, xf.y), a2[r][t]);
                            a2[r][t] = __ffma2_rn(make_float2(__uint_as_float(cw[r].z), __uint_as_float(cw[r].w)),
                                                  make_float2(xf.z, xf.w), a2[r][t]);
                        }
                    }
                    if (GW) fold_group(ssc);     // a chunk lies in one group
                } else if constexpr (kRollQ) {
                    // the chunk's 4 words in a loop (a body the instruction
                    // cache holds); lane group lane / 8 starts at its own word,
                    // so the warp's 4-byte code loads fall in 32 distinct banks
#pragma unroll 1
                    for (int q = 0; q < 4; ++q) {
                        const int qq = (q + (lane >> 3)) & 3;
                        float2 xv[NS * EW / 2];
#pragma unroll
                        for (int t = 0; t < NS; ++t)
#pragma unroll
                            for (int e4 = 0; e4 < EW; e4 += 4) {
                                const float4 v4 = *reinterpret_cast<const float4 *>(
                                    xsb + (size_t)t * k_alloc +
                                    ((((size_t)sg * 4 + qq) * (EW / 4) + (e4 >> 2)) * 32 + lane) * 4);
                                xv[t * (EW / 2) + e4 / 2] = make_float2(v4.x, v4.y);
                                xv[t * (EW / 2) + e4 / 2 + 1] = make_float2(v4.z, v4.w);
                            }
#pragma unroll
                        for (int r = 0; r < 8; ++r)
                            word_fma2<FMT, NS, EW>(*reinterpret_cast<const uint32_t *>(st + r * rb + 4 * qq), xv, a2[r]);
                        word_fma2<FMT, NS, EW>(F<FMT>::ZW, xv, az);
                    }
                } else {
                    // one 16-byte chunk = 4 words; x' for one word at a time
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float2 xv[NS * EW / 2];
#pragma unroll
                        for (int t = 0; t < NS; ++t)
#pragma unroll
                            for (int e4 = 0; e4 < EW; e4 += 4) {
                                const float4 v4 = *reinterpret_cast<const float4 *>(
                                    xsb + (size_t)t * k_alloc +
                                    ((((size_t)sg * 4 + q) * (EW / 4) + (e4 >> 2)) * 32 + lane) * 4);
                                xv[t * (EW / 2) + e4 / 2] = make_float2(v4.x, v4.y);
                                xv[t * (EW / 2) + e4 / 2 + 1] = make_float2(v4.z, v4.w);
                            }
#pragma unroll
                        for (int r = 0; r < 8; ++r) {
                            const uint32_t w = q == 0 ? cw[r].x : q == 1 ? cw[r].y : q == 2 ? cw[r].z : cw[r].w;
                            word_fma2<FMT, NS, EW>(w, xv, a2[r]);
                        }
                        word_fma2<FMT, NS, EW>(F<FMT>::ZW, xv, az);
                        if constexpr (GW != 0) {
                            if ((q + 1) % GW == 0) fold_group(ssc + q / GW);
                        }
                    }
                }
            }
            __syncwarp();  // every lane is done with this stage: hand it back to the producer
            if (lane == 0) mbar_arrive(my_empty + 8 * c_stage);
            if (++c_stage == depth) {
                c_stage = 0;
                c_phase ^= 1;
            }
        }
        if (cur_rgl >= 0) flush(cur_rgl);
        // combine this round, all consumers after a barrier (a row per thread;
        // measured 0.4 us faster per call than the last warp alone): warps in
        // order, unscale, apply the row scale
        const int c_first = tid, c_step = nct;
        consumers_sync(nct);
        // partials added in warp order (warps that ran no unit of a row group
        // hold +0 there); the set's fields stay in registers until the row
        // groups move into the next set
        const int rows = (rend - base) * 8;
        for (int t = 0; t < NS; ++t) {
            int s = s_lo;
            int s_start = p.rg_start[s], s_next = s + 1 < p.nsets ? p.rg_start[s + 1] : INT_MAX, s_O = p.O[s];
            float *s_y = p.y[s];
            int s_xr = (p.xslot[s] - slot_lo) * NS + t;
            for (int r = c_first; r < rows; r += c_step) {
                const int rgl = r >> 3, rr = r & 7;
                const float *pp = part + ((size_t)rgl * nw * NS + t) * 8 + rr;
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < kMaxWarps; ++w)
                    if (w < nw) sum += pp[(size_t)w * NS * 8];
                const int rg = base + rgl;
                if (rg >= s_next) {
                    s = set_of(rg, s);
                    s_start = p.rg_start[s];
                    s_next = s + 1 < p.nsets ? p.rg_start[s + 1] : INT_MAX;
                    s_O = p.O[s];
                    s_y = p.y[s];
                    s_xr = (p.xslot[s] - slot_lo) * NS + t;
                }
                const int o = (rg - s_start) * 8 + rr;
                if (o < s_O) {
                    const float dot = (sum * unscale[2 * s_xr]) * unscale[2 * s_xr + 1];   // exact: powers of two
                    s_y[(long long)t * s_O + o] = GW ? dot : dot * row_scale[(rg - rg0) * 8 + rr];
                }
            }
        }
        if (!last_round) consumers_sync(nct);   // part is reused by the next round
    }
    if (!ok) {
        // give up: record the timeout and let the copies the producer issued
        // into this warp's ring land first (at most `depth` stages ahead)
        if (lane == 0) atomicExch(&g_decode_err, (unsigned)(-B200Q_ETIMEOUT));
        for (int k = 0; k < depth; ++k) {
            mbar_wait(my_full + 8 * c_stage, c_phase, kWaitNs / 4);
            if (++c_stage == depth) {
                c_stage = 0;
                c_phase ^= 1;
            }
        }
    }
}

// One group: n sets, each a tensor with its input(s) and output at token 0.
struct Group {
    const Tensor *t[kMaxSets];
    const float *xa[kMaxSets];
    const float *xb[kMaxSets];
    float *y[kMaxSets];
    int n;
    bool silu;
};

template <int FMT, int NS, int MS, int GW>
cudaError_t launch_ns(const DecParams<MS> &p, int grid, cudaStream_t st) {
    constexpr int EW = FMT == B200Q_F32 ? 1 : FMT == B200Q_I8 ? 4 : FMT == B200Q_I4 ? 8 : 16;
    const int nseg = (p.ld + kSeg - 1) / kSeg;
    const size_t k_alloc = FMT == B200Q_F32 ? (size_t)p.k_pad : (size_t)nseg * (kSeg / 4) * EW;
    // ring stage (codes, then group scales) + its full and empty mbarriers
    const size_t stage = (size_t)kStage + (GW ? (size_t)32 * p.gbox : 0) + 16;
    const int rg_cta = (p.n_rg + grid - 1) / grid;
    const size_t nxr = (size_t)p.nx_max * NS;
    auto fixed_for = [&](int nw, int rr) {
        return 4 * nxr * k_alloc + 16 + (size_t)rr * nw * NS * 8 * 4 + nxr * 8 + nxr * kMaxWarps * 4 + 16 +
               (size_t)rg_cta * 8 * 4;
    };
    // warps and depth first (round of kRound), then grow the round to all of
    // the CTA's row groups if the partials still fit (one round: no barrier)
    int depth = 3, nw = max_warps<FMT, NS, GW>();
    if (stage_before_warp<FMT, NS>() && fixed_for(nw, kRound) + (size_t)nw * depth * stage > kSmemMax) depth = 2;
    while (nw > 4 && fixed_for(nw, kRound) + (size_t)nw * depth * stage > kSmemMax) --nw;
    if (fixed_for(nw, kRound) + (size_t)nw * depth * stage > kSmemMax) depth = 2;
    while (nw > 4 && fixed_for(nw, kRound) + (size_t)nw * depth * stage > kSmemMax) --nw;
    if (fixed_for(nw, kRound) + (size_t)nw * depth * stage > kSmemMax) return cudaErrorInvalidValue;  // x too long
    int rr = kRound;
    if (rg_cta <= kRound) {
        rr = rg_cta;
    } else {
        int big = rg_cta;
        while (big > kRound && fixed_for(nw, big) + (size_t)nw * depth * stage > kSmemMax) big = (big + kRound) / 2;
        rr = big > kRound ? big : kRound;
    }
    // the kernel's row-group and unit arithmetic is 32-bit
    if ((long long)grid * p.n_rg >= (1ll << 31) || (long long)nw * rr * nseg >= (1ll << 31))
        return cudaErrorInvalidValue;
    cudaError_t e = allow_dynamic_smem((const void *)qmv_decode_kernel<FMT, NS, MS, GW>, (int)kSmemMax);
    if (e != cudaSuccess) return e;
    DecParams<MS> q = p;
    q.depth = depth;
    q.round_rgs = rr;
    q.div_grid = make_fastdiv((uint32_t)grid);
    q.div_nseg = make_fastdiv((uint32_t)nseg);
    // programmatic dependent launch: this grid may start while the previous
    // kernel in the stream drains; it waits (griddepcontrol.wait) before it
    // touches x or y
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((nw + 1) * 32);              // consumers + the producer warp
    cfg.dynamicSmemBytes = fixed_for(nw, rr) + (size_t)nw * depth * stage;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, qmv_decode_kernel<FMT, NS, MS, GW>, q);
    count_launch();
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int FMT, int MS, int GW>
cudaError_t launch_group_ms(const Group &g, int S, cudaStream_t st) {
    const Tensor &t0 = *g.t[0];
    const int n_sms = sm_count(t0.device);
    DecParams<MS> p;
    memset(&p, 0, sizeof p);
    p.nsets = g.n;
    p.silu = g.silu ? 1 : 0;
    p.I = t0.I;
    p.ld = (int)t0.ld;
    p.row_bytes = (int)(t0.ld < kSeg ? t0.ld : kSeg);
    p.k_pad = (int)t0.k_pad;
    int slot = -1, n_rg = 0;
    if (GW) {
        p.gbox = t0.sc_box;
        p.div_gs = make_fastdiv((uint32_t)t0.gs);
    }
    for (int j = 0; j < g.n; ++j) {
        p.map[j] = g.t[j]->dec_map;
        if (GW) p.smap[j] = g.t[j]->sc_map;
        p.scales[j] = g.t[j]->scales;
        p.O[j] = g.t[j]->O;
        p.rg_start[j] = n_rg;
        n_rg += (g.t[j]->O + 7) / 8;
        if (j == 0 || g.xa[j] != g.xa[j - 1] || g.xb[j] != g.xb[j - 1]) ++slot;
        p.xslot[j] = slot;
    }
    p.rg_start[g.n] = n_rg;
    p.n_rg = n_rg;
    const int grid = n_rg < n_sms ? n_rg : n_sms;
    // most x slots a CTA spans (the same partition as the kernel's)
    int nx_max = 1;
    for (int b = 0, s = 0; b < grid; ++b) {
        const int r0 = (int)((long long)b * n_rg / grid), r1 = (int)((long long)(b + 1) * n_rg / grid);
        while (s + 1 < g.n && r0 >= p.rg_start[s + 1]) ++s;
        int e = s;
        while (e + 1 < g.n && r1 - 1 >= p.rg_start[e + 1]) ++e;
        const int nx = p.xslot[e] - p.xslot[s] + 1;
        if (nx > nx_max) nx_max = nx;
    }
    p.nx_max = nx_max;
    for (int s0 = 0; s0 < S;) {
        // tokens per launch: four while at least four remain (per-row scales),
        // else two, else one
        const int ns = !GW && FMT != B200Q_I2 && S - s0 >= 4 ? 4 : S - s0 >= 2 ? 2 : 1;
        for (int j = 0; j < g.n; ++j) {
            p.xa[p.xslot[j]] = g.xa[j] + (long long)s0 * t0.I;
            p.xb[p.xslot[j]] = g.xb[j] ? g.xb[j] + (long long)s0 * t0.I : nullptr;
            p.y[j] = g.y[j] + (long long)s0 * g.t[j]->O;
        }
        cudaError_t e;
        if constexpr (GW == 0 && FMT != B200Q_I2)
            e = ns == 4   ? launch_ns<FMT, 4, MS, GW>(p, grid, st)
                : ns == 2 ? launch_ns<FMT, 2, MS, GW>(p, grid, st)
                          : launch_ns<FMT, 1, MS, GW>(p, grid, st);
        else
            e = ns == 2 ? launch_ns<FMT, 2, MS, GW>(p, grid, st) : launch_ns<FMT, 1, MS, GW>(p, grid, st);
        if (e != cudaSuccess) return e;
        s0 += ns;
    }
    return cudaSuccess;
}

// Group-wise scales take the kernel variant for the group's span in words
// of a chunk (every set of a launch has the same group size); one variant
// per format serves all set counts.
template <int FMT>
cudaError_t launch_group_fmt(const Group &g, int S, cudaStream_t st) {
    constexpr int E = F<FMT>::E, EW = FMT == B200Q_F32 ? 1 : E / 4;
    const int gs = g.t[0]->gs;
    if (gs == 0) return g.n <= 2 ? launch_group_ms<FMT, 2, 0>(g, S, st) : launch_group_ms<FMT, kMaxSets, 0>(g, S, st);
    if (gs % E == 0) return launch_group_ms<FMT, kMaxSets, 4>(g, S, st);
    if constexpr (FMT == B200Q_I4) {
        if (gs == 2 * EW) return launch_group_ms<FMT, kMaxSets, 2>(g, S, st);
    } else if constexpr (FMT == B200Q_I2) {
        if (gs == EW) return launch_group_ms<FMT, kMaxSets, 1>(g, S, st);
        if (gs == 2 * EW) return launch_group_ms<FMT, kMaxSets, 2>(g, S, st);
    }
    return cudaErrorInvalidValue;   // not a group size the decode kernel takes
}

cudaError_t launch_group(const Group &g, int S, cudaStream_t st, bool *handled) {
    *handled = false;
    if (S < 1 || S > 15 || g.n < 1 || g.n > kMaxSets) return cudaSuccess;
    for (int j = 1; j < g.n; ++j)
        if (g.t[j]->gs != g.t[0]->gs) return cudaSuccess;   // mixed scale layouts: one tensor at a time
    // the group arithmetic is 32-bit
    if (g.t[0]->gs && g.t[0]->k_pad + (long long)kSeg * 8 >= (1ll << 31)) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    switch (g.t[0]->fmt) {
    case B200Q_F32: e = launch_group_fmt<B200Q_F32>(g, S, st); break;
    case B200Q_I8: e = launch_group_fmt<B200Q_I8>(g, S, st); break;
    case B200Q_I4: e = launch_group_fmt<B200Q_I4>(g, S, st); break;
    case B200Q_I2: e = launch_group_fmt<B200Q_I2>(g, S, st); break;
    default: return cudaSuccess;
    }
    if (e == cudaErrorInvalidValue) return cudaSuccess;
    *handled = (e == cudaSuccess);
    return e;
}

}  // namespace

// Handles every format for 1 <= S < 16 (tokens in launches of four, two or
// one);
// *handled = false sends the call to the general SIMT kernel (x too long for
// shared memory).
cudaError_t launch_decode(const Tensor &t, const Tensor *tu, const float *x, float *y, float *yu, int S,
                          cudaStream_t st, bool *handled) {
    Group g{};
    g.n = tu ? 2 : 1;
    g.t[0] = &t;
    g.xa[0] = x;
    g.y[0] = y;
    if (tu) {
        g.t[1] = tu;
        g.xa[1] = x;
        g.y[1] = yu;
    }
    return launch_group(g, S, st, handled);
}

// n (<= 16) tensors of one format and I in one launch per four, two or one
// tokens; input
// j is xa[j], or silu(xa[j]) * xb[j] when silu is set.  *handled = false when
// the staged inputs do not fit in shared memory (the caller then runs the
// tensors one at a time).
cudaError_t launch_decode_group(const Tensor *const *ts, int n, const float *const *xa, const float *const *xb,
                                float *const *ys, bool silu, int S, cudaStream_t st, bool *handled) {
    *handled = false;
    if (n < 1 || n > kMaxSets) return cudaSuccess;
    Group g{};
    g.n = n;
    g.silu = silu;
    for (int j = 0; j < n; ++j) {
        g.t[j] = ts[j];
        g.xa[j] = xa[j];
        g.xb[j] = silu ? xb[j] : nullptr;
        g.y[j] = ys[j];
    }
    return launch_group(g, S, st, handled);
}

// Reads and clears the decode kernel's device error word.
cudaError_t decode_take_error(unsigned int *code) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_decode_err, sizeof(unsigned int));
    if (e == cudaSuccess && *code) e = cudaMemcpyToSymbol(g_decode_err, &zero, sizeof(unsigned int));
    return e;
}

}  // namespace qwq
