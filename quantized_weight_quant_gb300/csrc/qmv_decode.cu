// Decode kernel for int8 / int4 / int2 weights at small S (the f32-accurate
// path): y[s,o] = scale[o] * sum_i deq(W[o,i]) * x[s,i]   ("CUDA 后端",
// section 1, weight_at / quant_matmul; three-backends chapter, section 四,
// qmatmul.comp header: x staged once and reused for every output row).
//
// Why tensor cores here.  Decode streams every weight once (HBM-bound), but
// on the SIMT pipe each int4 weight costs an unpack, a convert and an FMA per
// token: 3-4 issue slots per weight, more than an SM can issue at HBM rate.
// So the FMAs go to mma.sync and the SIMT pipe only unpacks:
//
//   * codes -> exact fp16 in registers.  A code c is ORed into the mantissa
//     of 1024.0 (fp16 0x6400, whose mantissa LSB is 1), giving 1024 + c
//     exactly; one packed subtraction of 1024 + zero-point leaves deq(c)
//     exactly (|deq| <= 128 fits fp16's 11-bit significand).  Two codes per
//     instruction pair: lop3 (int4: nibbles i and i+4 of a word; int2: fields
//     t and t+8) or prmt (int8: adjacent bytes, after flipping the sign bit).
//   * x -> two fp16 terms.  Per token s, x is scaled by 2^e_s (exact) so that
//     max|x_s| lands in [2^14, 2^15), then split as hi = fp16(v),
//     lo = fp16(v - hi).  hi + lo carries 22 significant bits; the remainder
//     is below 2^-21 |x| or 2^-38 max|x_s|, far inside the 1e-5 tolerance.
//   * every product of an exact fp16 integer and an fp16 term is exact in
//     f32; the tensor core sums them in f32.  Four independent accumulators
//     take alternate MMAs and are folded into an f32 register sum after every
//     k-block, so no accumulation chain is longer than a few MMAs;
//     y = 2^-e_s * (hi + lo sums) * scale[o].
//
// MMA shape m16n8k16 (row.col, f16 in, f32 accumulate), weights as the B
// operand: n = 8 weight rows (a "row group"), m = 16 rows of x terms
// (m = s is token s's hi term, m = 8 + s its lo term, so S <= 8 per launch),
// k = 16 weights of a row.  The contraction index is reordered consistently
// on both operands: lane (g, q) reads the 16-byte chunk q of each 4-chunk
// k-block of weight row g, and MMA j of the chunk takes its code pairs 2j and
// 2j+1; the x terms are staged in shared memory in exactly that order, 16
// bytes per lane per MMA, so each A fragment is one conflict-free 16-byte
// shared load.
//
// Data movement.  Every warp owns whole row groups (no cross-warp sums) and
// streams them through its own ring of DEPTH shared-memory stages; a stage
// holds one segment (up to 1 KB) of each of the row group's 8 rows, fetched
// by 8 bulk async copies (cp.async.bulk, completion on an mbarrier) that
// lane 0 issues DEPTH-1 stages ahead.  With ~12 warps x 2 stages in flight an
// SM keeps ~100 KB of weights in flight, enough to cover HBM latency at full
// bandwidth without spending registers on it.  Rows are stored with a
// 16-byte pad so the 8 rows of a fragment load fall in different banks.  The
// first copies are issued before x is staged, so the x prologue hides under
// the first HBM trip.  Persistent CTAs, one per SM, own contiguous runs of
// row groups.  Every mbarrier wait is bounded in time; a wait that gives up
// records B200Q_ETIMEOUT in a device word (b200q_device_status), drains its
// own copies in flight and returns.
#include <cuda_fp16.h>

#include "qwq_internal.h"

namespace qwq {
namespace {

constexpr int kMaxWarps = 16;
constexpr int kMaxS = 8;           // tokens per launch (hi terms in m 0..7, lo in 8..15)
constexpr int kSegMax = 512;       // bytes per row per stage
constexpr size_t kSmemMax = 220 * 1024;
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s bound on any wait

__device__ unsigned int g_decode_err = 0;

template <int FMT>
struct F;  // E: elements per 16-byte chunk; J: MMAs per chunk
template <>
struct F<B200Q_I8> {
    static constexpr int E = 16, J = 4;
};
template <>
struct F<B200Q_I4> {
    static constexpr int E = 32, J = 8;
};
template <>
struct F<B200Q_I2> {
    static constexpr int E = 64, J = 16;
};

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t magic) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(magic));
    return r;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ void mma_16816(float (&c)[4], const uint4 &a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word(const uint4 &c, int m) {
    return m == 0 ? c.x : m == 1 ? c.y : m == 2 ? c.z : c.w;
}

// The two fp16x2 B registers of MMA j from one 16-byte chunk of codes:
// code pairs 2j and 2j+1 in the production order of the format.
template <int FMT>
__device__ __forceinline__ void b_regs(const uint4 &c, int j, uint32_t &b0, uint32_t &b1);

template <>
__device__ __forceinline__ void b_regs<B200Q_I4>(const uint4 &c, int j, uint32_t &b0, uint32_t &b1) {
    // pair p = 4m + h holds nibbles h and h + 4 of word m
    const uint32_t w = word(c, j >> 1);
    const int h = 2 * (j & 1);
    b0 = hsub2(lop3_and_or(w >> (4 * h), 0x000F000Fu, 0x64006400u), 0x64086408u);
    b1 = hsub2(lop3_and_or(w >> (4 * h + 4), 0x000F000Fu, 0x64006400u), 0x64086408u);
}

template <>
__device__ __forceinline__ void b_regs<B200Q_I8>(const uint4 &c, int j, uint32_t &b0, uint32_t &b1) {
    // pair p = 2m + h holds bytes 2h and 2h + 1 of word m; flipping the sign
    // bit turns the two's-complement code into code + 128 in 0..255
    const uint32_t w = word(c, j) ^ 0x80808080u;
    b0 = hsub2(__byte_perm(w, 0x64646464u, 0x4140), 0x64806480u);
    b1 = hsub2(__byte_perm(w, 0x64646464u, 0x4342), 0x64806480u);
}

template <>
__device__ __forceinline__ void b_regs<B200Q_I2>(const uint4 &c, int j, uint32_t &b0, uint32_t &b1) {
    // pair p = 8m + t holds 2-bit fields t and t + 8 of word m
    const uint32_t w = word(c, j >> 2);
    const int t = 2 * (j & 3);
    b0 = hsub2(lop3_and_or(w >> (2 * t), 0x00030003u, 0x64006400u), 0x64026402u);
    b1 = hsub2(lop3_and_or(w >> (2 * t + 2), 0x00030003u, 0x64006400u), 0x64026402u);
}

// Inverse of the pair order: element e of a chunk -> (pair, half).
template <int FMT>
__device__ __forceinline__ void elem_pos(int e, int &pair, int &half);

template <>
__device__ __forceinline__ void elem_pos<B200Q_I4>(int e, int &pair, int &half) {
    const int r = e & 7;
    pair = 4 * (e >> 3) + (r & 3);
    half = r >> 2;
}

template <>
__device__ __forceinline__ void elem_pos<B200Q_I8>(int e, int &pair, int &half) {
    const int r = e & 3;
    pair = 2 * (e >> 2) + (r >> 1);
    half = r & 1;
}

template <>
__device__ __forceinline__ void elem_pos<B200Q_I2>(int e, int &pair, int &half) {
    const int r = e & 15;
    pair = 8 * (e >> 4) + (r & 7);
    half = r >> 3;
}

// ---- mbarrier / bulk-copy helpers (PTX ISA: mbarrier, cp.async.bulk)

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
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

// Bounded wait for the phase with the given parity to complete.
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

struct DecParams {
    const uint8_t *codes[2];
    const float *scales[2];
    float *y[2];
    const float *x;      // [S, I] f32 (offset to this launch's first token)
    int x_ld;            // row stride of x in elements (I)
    int y_ld;            // row stride of y in elements (O)
    int O, I;
    long long ld;        // device row stride in bytes
    int k_pad;           // elements per padded row
    int S;               // tokens in this launch, 1..kMaxS
    int rg_per_set;      // ceil(O / 8)
    int n_rg;            // total row groups (sets * rg_per_set)
    int seg;             // bytes per row per stage (multiple of 128, <= kSegMax)
    int depth;           // stages per warp
    int max_units;       // bound on (row group, segment) units per CTA (partials buffer)
};

// Calls fn(k, v) for every k in [0, k_end) of x row s (v = 0 for k >= I),
// with up to 8 independent 16-byte loads in flight per thread.
template <typename Fn>
__device__ __forceinline__ void for_x_row(const DecParams &p, int s, int k_end, Fn fn) {
    const float *xr = p.x + (long long)s * p.x_ld;
    const int nthr = blockDim.x;
    if ((p.x_ld & 3) == 0) {
        const float4 *x4 = reinterpret_cast<const float4 *>(xr);
        const int n4 = k_end >> 2;               // k_end is a multiple of 4
        for (int base = 0; base < n4; base += 8 * nthr) {
            float4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k4 = base + i * nthr + threadIdx.x;
                v[i] = (k4 < n4 && 4 * k4 < p.I) ? x4[k4] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k4 = base + i * nthr + threadIdx.x;
                if (k4 < n4) {
                    fn(4 * k4, v[i].x);
                    fn(4 * k4 + 1, v[i].y);
                    fn(4 * k4 + 2, v[i].z);
                    fn(4 * k4 + 3, v[i].w);
                }
            }
        }
    } else {
        for (int base = 0; base < k_end; base += 8 * nthr) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = base + i * nthr + threadIdx.x;
                v[i] = k < p.I ? xr[k] : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int k = base + i * nthr + threadIdx.x;
                if (k < k_end) fn(k, v[i]);
            }
        }
    }
}

template <int FMT>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) qmv_decode_kernel(const DecParams p) {
    using Fm = F<FMT>;
    constexpr int E = Fm::E, J = Fm::J;
    extern __shared__ __align__(128) uint8_t smem[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nw = blockDim.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int S = p.S;
    const int depth = p.depth;
    const int rp = p.seg + 16;                       // smem row pitch
    const int stage_bytes = 8 * rp;
    const int nseg = (int)((p.ld + p.seg - 1) / p.seg);

    // shared memory: x terms | rings | mbarriers | partials | exps | max scratch
    uint8_t *a_s = smem;                                              // 4 * S * k_pad
    uint8_t *ring = smem + (size_t)4 * S * p.k_pad;                   // nw * depth * stage_bytes
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + (size_t)nw * depth * stage_bytes);
    float *part = reinterpret_cast<float *>(bars + nw * depth);      // [unit][S][8]
    int *exps = reinterpret_cast<int *>(part + (size_t)p.max_units * S * 8);
    float *red = reinterpret_cast<float *>(exps + kMaxS);            // [S][nw]

    // this CTA's row groups [rg0, rg1) and its units (row group, segment);
    // warp w takes units w, w + nw, ...
    const int rg0 = (int)((long long)blockIdx.x * p.n_rg / gridDim.x);
    const int rg1 = (int)((long long)(blockIdx.x + 1) * p.n_rg / gridDim.x);
    const int cta_units = (rg1 - rg0) * nseg;
    const int n_units = cta_units > warp ? (cta_units - warp + nw - 1) / nw : 0;

    uint8_t *my_ring = ring + (size_t)warp * depth * stage_bytes;
    const uint32_t my_bars = smem_u32(bars + warp * depth);
    uint64_t policy = 0;

    auto issue = [&](int i) {  // lane 0 only: this warp's i-th unit
        const int u = warp + i * nw;
        const int rgl = u / nseg, sg = u - rgl * nseg;
        const int rg = rg0 + rgl;
        const int set = rg >= p.rg_per_set;
        const uint8_t *base = (set ? p.codes[1] : p.codes[0]) +
                              (long long)((rg - set * p.rg_per_set) * 8) * p.ld + (long long)sg * p.seg;
        const long long left = p.ld - (long long)sg * p.seg;
        const uint32_t bytes = (uint32_t)(left < p.seg ? left : p.seg);
        const int b = i % depth;
        const uint32_t bar = my_bars + 8 * b;
        const uint32_t dst = smem_u32(my_ring + (size_t)b * stage_bytes);
        mbar_expect_tx(bar, 8 * bytes);
#pragma unroll
        for (int r = 0; r < 8; ++r) bulk_g2s(dst + r * rp, base + (long long)r * p.ld, bytes, bar, policy);
    };

    if (lane == 0) {
        for (int b = 0; b < depth; ++b) mbar_init(my_bars + 8 * b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        policy = evict_first_policy();
        for (int i = 0; i < depth - 1 && i < n_units; ++i) issue(i);
    }
    __syncwarp();

    // ---- stage x: per-token power-of-two scale, hi/lo fp16 split, MMA order
    for (int s = 0; s < S; ++s) {
        float m = 0.f;
        for_x_row(p, s, (p.I + 3) & ~3, [&](int, float v) { m = fmaxf(m, fabsf(v)); });
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) red[s * nw + warp] = m;
    }
    __syncthreads();
    if (tid < S) {
        float m = 0.f;
        for (int w = 0; w < nw; ++w) m = fmaxf(m, red[tid * nw + w]);
        exps[tid] = m > 0.f ? 14 - ilogbf(m) : 0;
    }
    __syncthreads();
    {
        __half *a_h = reinterpret_cast<__half *>(a_s);
        for (int s = 0; s < S; ++s) {
            const int ex = exps[s];
            for_x_row(p, s, p.k_pad, [&](int k, float xv) {
                const float v = ldexpf(xv, ex);
                const __half hi = __float2half_rn(v);
                const __half lo = __float2half_rn(v - __half2float(hi));
                const int c = k / E, e = k - c * E;
                int pair, half;
                elem_pos<FMT>(e, pair, half);
                const int j = pair >> 1, slot = pair & 1;
                // 16-byte group (kb, j, s, q): words {hi p0, lo p0, hi p1, lo p1}
                const size_t grp = (((size_t)(c >> 2) * J + j) * S + s) * 4 + (c & 3);
                const size_t hidx = grp * 8 + slot * 4 + half;  // in halves
                a_h[hidx] = hi;
                a_h[hidx + 2] = lo;
            });
        }
    }
    __syncthreads();

    // ---- main loop over this warp's (row group, segment) units
    const uint4 *a_v = reinterpret_cast<const uint4 *>(a_s);
    const bool has_tok = g < S;
    const int kb_per_seg = p.seg / 64;
    int i = 0;
    bool ok = true;
    for (; i < n_units; ++i) {
        if (lane == 0 && i + depth - 1 < n_units) issue(i + depth - 1);
        const int b = i % depth;
        if (!mbar_wait(my_bars + 8 * b, (uint32_t)((i / depth) & 1), kWaitNs)) {
            ok = false;
            break;
        }
        const int u = warp + i * nw;
        const int sg = u % nseg;
        const long long left = p.ld - (long long)sg * p.seg;
        const int n_kb = (int)((left < p.seg ? left : p.seg) / 64);
        const uint8_t *rowp = my_ring + (size_t)b * stage_bytes + g * rp + q * 16;
        const uint4 *ak = a_v + ((size_t)sg * kb_per_seg * J * S + g) * 4 + q;
        float c4[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int r = 0; r < 4; ++r) c4[a][r] = 0.f;
        for (int kb = 0; kb < n_kb; ++kb) {
            const uint4 codes = *reinterpret_cast<const uint4 *>(rowp + kb * 64);
#pragma unroll
            for (int j = 0; j < J; ++j) {
                uint4 a = make_uint4(0, 0, 0, 0);
                if (has_tok) a = ak[((size_t)kb * J + j) * S * 4];
                uint32_t b0, b1;
                b_regs<FMT>(codes, j, b0, b1);
                mma_16816(c4[j & 3], a, b0, b1);
            }
        }
        __syncwarp();  // every lane is done with stage b before lane 0 refills it
        if (has_tok) {
            // rows 2q, 2q+1 of token g: hi terms (m = g) + lo terms (m = g + 8)
            float2 v;
            v.x = (c4[0][0] + c4[1][0]) + (c4[2][0] + c4[3][0]) + (c4[0][2] + c4[1][2]) + (c4[2][2] + c4[3][2]);
            v.y = (c4[0][1] + c4[1][1]) + (c4[2][1] + c4[3][1]) + (c4[0][3] + c4[1][3]) + (c4[2][3] + c4[3][3]);
            *reinterpret_cast<float2 *>(part + ((size_t)u * S + g) * 8 + 2 * q) = v;
        }
    }
    if (!ok) {
        // give up: record the timeout, then let this warp's copies in flight
        // land before the CTA's shared memory goes away
        if (lane == 0) atomicExch(&g_decode_err, (unsigned)(-B200Q_ETIMEOUT));
        const int last = (i + depth - 1 < n_units ? i + depth - 1 : n_units - 1);
        for (int v = i; v <= last; ++v) mbar_wait(my_bars + 8 * (v % depth), (uint32_t)((v / depth) & 1), kWaitNs / 4);
    }
    __syncthreads();

    // ---- combine the segments of each row group in a fixed order
    const int rows = (rg1 - rg0) * 8;
    for (int idx = tid; idx < rows * S; idx += blockDim.x) {
        const int s = idx / rows, r = idx - s * rows;
        const int rgl = r >> 3, rr = r & 7;
        float sum = 0.f;
        for (int sg = 0; sg < nseg; ++sg) sum += part[((size_t)(rgl * nseg + sg) * S + s) * 8 + rr];
        const int rg = rg0 + rgl;
        const int set = rg >= p.rg_per_set;
        const int o = (rg - set * p.rg_per_set) * 8 + rr;
        if (o < p.O) {
            float *yb = set ? p.y[1] : p.y[0];
            const float *sb = set ? p.scales[1] : p.scales[0];
            yb[(long long)s * p.y_ld + o] = ldexpf(sum, -exps[s]) * sb[o];
        }
    }
}

int g_sms = 0;

template <int FMT>
cudaError_t launch_fmt(const Tensor &t, const Tensor *tu, const float *x, float *y, float *yu, int S,
                       cudaStream_t st) {
    if (!g_sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
    }
    DecParams p{};
    p.codes[0] = t.codes;
    p.scales[0] = t.scales;
    p.codes[1] = tu ? tu->codes : t.codes;
    p.scales[1] = tu ? tu->scales : t.scales;
    p.x_ld = t.I;
    p.y_ld = t.O;
    p.O = t.O;
    p.I = t.I;
    p.ld = t.ld;
    p.k_pad = (int)t.k_pad;
    p.rg_per_set = (t.O + 7) / 8;
    p.n_rg = p.rg_per_set * (tu ? 2 : 1);
    p.seg = (int)(t.ld < kSegMax ? t.ld : kSegMax);
    const int nseg = (int)((t.ld + p.seg - 1) / p.seg);

    // one CTA per SM unless the partial-sum buffer would grow too large
    int grid = p.n_rg < g_sms ? p.n_rg : g_sms;
    const int max_rg_cta = 64;
    const int need = (p.n_rg + max_rg_cta - 1) / max_rg_cta;
    if (grid < need) grid = need;
    p.max_units = ((p.n_rg + grid - 1) / grid) * nseg;

    // tokens per launch: at most 4 keeps the A-fragment shared-memory traffic
    // under the SM's bandwidth; fewer when x terms would crowd out the rings
    const size_t stage = (size_t)8 * (p.seg + 16) + 8;   // ring stage + its mbarrier
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(qmv_decode_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemMax);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    auto fixed_for = [&](int sc) {
        return (size_t)4 * sc * p.k_pad + (size_t)p.max_units * sc * 8 * 4 + kMaxS * 4 +
               (size_t)kMaxS * kMaxWarps * 4;
    };
    for (int s0 = 0; s0 < S;) {
        int sc = S - s0 < 4 ? S - s0 : 4;
        while (sc > 1 && fixed_for(sc) + (size_t)4 * 2 * stage > kSmemMax) --sc;
        const size_t fixed = fixed_for(sc);
        if (fixed + (size_t)4 * 2 * stage > kSmemMax) return cudaErrorInvalidValue;
        int depth = 3, nw = kMaxWarps;
        while (nw > 4 && fixed + (size_t)nw * depth * stage > kSmemMax) --nw;
        if (fixed + (size_t)nw * depth * stage > kSmemMax) depth = 2;
        while (nw > 4 && fixed + (size_t)nw * depth * stage > kSmemMax) --nw;
        p.depth = depth;
        p.S = sc;
        p.x = x + (long long)s0 * t.I;
        p.y[0] = y + (long long)s0 * t.O;
        p.y[1] = tu ? yu + (long long)s0 * t.O : p.y[0];
        const size_t smem = fixed + (size_t)nw * depth * stage;
        qmv_decode_kernel<FMT><<<grid, nw * 32, smem, st>>>(p);
        count_launch();
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        s0 += sc;
    }
    return cudaSuccess;
}

}  // namespace

// Handles int8 / int4 / int2 tensors for S below the tensor-core threshold;
// *handled = false sends the call to the general SIMT kernel.
cudaError_t launch_decode(const Tensor &t, const Tensor *tu, const float *x, float *y, float *yu, int S,
                          cudaStream_t st, bool *handled) {
    *handled = false;
    if (S < 1 || S > 15) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    switch (t.fmt) {
    case B200Q_I8: e = launch_fmt<B200Q_I8>(t, tu, x, y, yu, S, st); break;
    case B200Q_I4: e = launch_fmt<B200Q_I4>(t, tu, x, y, yu, S, st); break;
    case B200Q_I2: e = launch_fmt<B200Q_I2>(t, tu, x, y, yu, S, st); break;
    default: return cudaSuccess;
    }
    if (e == cudaErrorInvalidValue) return cudaSuccess;  // x too large for shared memory
    *handled = (e == cudaSuccess);
    return e;
}

// Reads and clears the decode kernel's device error word.
cudaError_t decode_take_error(unsigned int *code) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_decode_err, sizeof(unsigned int));
    if (e == cudaSuccess && *code) e = cudaMemcpyToSymbol(g_decode_err, &zero, sizeof(unsigned int));
    return e;
}

}  // namespace qwq
