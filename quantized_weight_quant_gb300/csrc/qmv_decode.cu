// Decode kernel for int8 / int4 / int2 weights at small S (the f32-accurate
// path): y[s,o] = scale[o] * sum_i deq(W[o,i]) * x[s,i]   ("CUDA 后端",
// section 1, weight_at / quant_matmul; three-backends chapter, section 四,
// qmatmul.comp header: x staged once and reused for every output row).
//
// Why tensor cores here.  Decode streams every weight once (HBM-bound), but
// on the SIMT pipe each int4 weight costs an unpack, a convert and an FMA per
// token: about 3-4 issue slots per weight, more than an SM can issue at HBM
// rate.  So the FMAs go to mma.sync and the SIMT pipe only unpacks:
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
//     f32; the tensor core sums them in f32.  The MMA accumulator is folded
//     into an f32 register sum after every k-block (at most 16 MMA steps per
//     chain), the K-slices of the 16 warps are summed in shared memory in a
//     fixed order, and y = 2^-e_s * (hi + lo sums) * scale[o].
//
// MMA shape m16n8k16 (row.col, f16 in, f32 accumulate), weights as the B
// operand: n = 8 weight rows (a "row group"), m = 16 rows of x terms
// (m = s is token s's hi term, m = 8 + s its lo term, so S <= 8 per launch),
// k = 16 weights of a row.  The contraction index is reordered consistently
// on both operands: lane (g, q) of the warp loads the 16-byte chunk q of
// each 4-chunk k-block of weight row g, and MMA j of the chunk takes its
// code pairs 2j and 2j+1; the x terms are staged in shared memory in exactly
// that order, 16 bytes per lane per MMA, so each A fragment is one
// conflict-free 16-byte shared load.
//
// Work split.  Persistent CTAs of 16 warps, one per SM: each CTA owns a
// contiguous run of row groups (at most 12); its warps split the K blocks
// (warp wk owns a contiguous K-slice) and walk the CTA's row groups four at
// a time, so one A fragment feeds four MMAs.  The weight loads of the next
// step are issued before the current step's MMAs, and the first loads go
// out before x is staged, so the x prologue hides under the first HBM trip.
#include <cuda_fp16.h>

#include "qwq_internal.h"

namespace qwq {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kT = 4;          // row groups per pass (share one A fragment)
constexpr int kMaxS = 8;       // tokens per launch (hi terms in m 0..7, lo in 8..15)
constexpr int kMaxRgPerCta = 12;
constexpr int kMaxPasses = (kMaxRgPerCta + kT - 1) / kT;
constexpr size_t kSmemBudget = 200 * 1024;

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

__device__ __forceinline__ uint4 ld_stream(const uint8_t *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

struct DecParams {
    const uint8_t *codes[2];
    const float *scales[2];
    float *y[2];
    const float *x;      // [S, I] f32 (already offset to this launch's first token)
    int x_ld;            // row stride of x in elements (I)
    int y_ld;            // row stride of y in elements (O)
    int O, I;
    long long ld;        // device row stride in bytes
    int k_pad;           // elements per padded row
    int nkb;             // k-blocks per row (k_pad / (4 E))
    int wk;              // warps along K (WK), wr = kWarps / WK warp rows
    int S;               // tokens in this launch, 1..kMaxS
    int rg_per_set;      // ceil(O / 8)
    int n_rg;            // total row groups (sets * rg_per_set)
};

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) qmv_mma_kernel(const DecParams p) {
    using Fm = F<FMT>;
    constexpr int E = Fm::E, J = Fm::J;
    extern __shared__ __align__(16) uint8_t smem[];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int S = p.S;
    const int WK = p.wk, WR = kWarps / p.wk;
    const int wk = warp % WK, wr = warp / WK;
    const bool active = wr < WR;

    // this CTA's row groups [rg0, rg1)
    const int rg0 = (int)((long long)blockIdx.x * p.n_rg / gridDim.x);
    const int rg1 = (int)((long long)(blockIdx.x + 1) * p.n_rg / gridDim.x);
    const int n_pass = (rg1 - rg0 + kT - 1) / kT;

    // this warp's k-blocks [kb0, kb1)
    const int kb0 = wk * p.nkb / WK, kb1 = (wk + 1) * p.nkb / WK;
    const int n_kb = kb1 - kb0;

    // shared memory: A terms | partial sums | per-token exponents + max scratch
    uint8_t *a_s = smem;                                             // 4 * S * k_pad bytes
    float *part = reinterpret_cast<float *>(smem + (size_t)4 * S * p.k_pad);  // [pass][WK][kT][S][8]
    float *red = part + (size_t)kMaxPasses * WK * kT * S * 8;        // [S][kWarps]
    int *exps = reinterpret_cast<int *>(red + kMaxS * kWarps);       // [S]

    // iteration it = pass * n_kb + kb (this warp's passes are wr, wr + WR, ...)
    const int my_passes = active ? (n_pass > wr ? (n_pass - wr + WR - 1) / WR : 0) : 0;
    const int n_it = my_passes * n_kb;

    auto load_it = [&](int it, uint4 (&buf)[kT]) {
        const int pass = wr + (it / n_kb) * WR;
        const int kb = kb0 + it % n_kb;
        const int rgb = rg0 + pass * kT;
#pragma unroll
        for (int t = 0; t < kT; ++t) {
            const int rg = rgb + t;
            if (rg < rg1) {
                const int set = rg >= p.rg_per_set;
                const int row = (rg - set * p.rg_per_set) * 8 + g;
                const uint8_t *base = set ? p.codes[1] : p.codes[0];
                buf[t] = ld_stream(base + (long long)row * p.ld + (long long)(kb * 4 + q) * 16);
            } else {
                buf[t] = make_uint4(0, 0, 0, 0);
            }
        }
    };

    uint4 cur[kT], nxt[kT];
    if (n_it > 0) load_it(0, cur);

    // ---- stage x: per-token power-of-two scale, hi/lo fp16 split, MMA order
    for (int s = 0; s < S; ++s) {
        float m = 0.f;
        for (int k = tid; k < p.I; k += kThreads) m = fmaxf(m, fabsf(__ldg(p.x + (long long)s * p.x_ld + k)));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) red[s * kWarps + warp] = m;
    }
    __syncthreads();
    if (tid < S) {
        float m = 0.f;
        for (int w = 0; w < kWarps; ++w) m = fmaxf(m, red[tid * kWarps + w]);
        exps[tid] = m > 0.f ? 14 - ilogbf(m) : 0;
    }
    __syncthreads();
    {
        const int total = S * p.k_pad;
        __half *a_h = reinterpret_cast<__half *>(a_s);
        for (int idx = tid; idx < total; idx += kThreads) {
            const int s = idx / p.k_pad, k = idx - s * p.k_pad;
            const float v = k < p.I ? ldexpf(__ldg(p.x + (long long)s * p.x_ld + k), exps[s]) : 0.f;
            const __half hi = __float2half_rn(v);
            const __half lo = __float2half_rn(v - __half2float(hi));
            const int c = k / E, e = k - c * E;
            int pair, half;
            elem_pos<FMT>(e, pair, half);
            const int j = pair >> 1, slot = pair & 1;
            // 16-byte group (kb, j, s, q): words {hi p0, lo p0, hi p1, lo p1}
            const size_t grp = (((size_t)(c >> 2) * J + j) * S + s) * 4 + (c & 3);
            const size_t hidx = grp * 8 + slot * 4 + half;     // in halves
            a_h[hidx] = hi;
            a_h[hidx + 2] = lo;
        }
    }
    __syncthreads();

    // ---- main loop
    float acc[kT][4];
    float cfr[kT][4];
#pragma unroll
    for (int t = 0; t < kT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;

    const uint4 *a_v = reinterpret_cast<const uint4 *>(a_s);
    for (int it = 0; it < n_it; ++it) {
        if (it + 1 < n_it) load_it(it + 1, nxt);
        const int pass_local = it / n_kb;
        const int kb = kb0 + it % n_kb;
#pragma unroll
        for (int t = 0; t < kT; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) cfr[t][i] = 0.f;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            uint4 a = make_uint4(0, 0, 0, 0);
            if (g < S) a = a_v[(((size_t)kb * J + j) * S + g) * 4 + q];
#pragma unroll
            for (int t = 0; t < kT; ++t) {
                uint32_t b0, b1;
                b_regs<FMT>(cur[t], j, b0, b1);
                mma_16816(cfr[t], a, b0, b1);
            }
        }
#pragma unroll
        for (int t = 0; t < kT; ++t)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[t][i] += cfr[t][i];

        if (it % n_kb == n_kb - 1) {
            // end of a pass: publish this warp's K-slice partials (hi + lo)
            if (g < S) {
                const int pass = wr + pass_local * WR;
#pragma unroll
                for (int t = 0; t < kT; ++t) {
                    float2 v = make_float2(acc[t][0] + acc[t][2], acc[t][1] + acc[t][3]);
                    float *dst = part + ((((size_t)pass * WK + wk) * kT + t) * S + g) * 8 + 2 * q;
                    *reinterpret_cast<float2 *>(dst) = v;
                }
            }
#pragma unroll
            for (int t = 0; t < kT; ++t)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;
        }
#pragma unroll
        for (int t = 0; t < kT; ++t) cur[t] = nxt[t];
    }
    __syncthreads();

    // ---- combine K-slices in a fixed order, unscale, apply the row scale
    const int rows = (rg1 - rg0) * 8;
    for (int idx = tid; idx < rows * S; idx += kThreads) {
        const int s = idx / rows, r = idx - s * rows;
        const int rgl = r >> 3, rr = r & 7;
        const int pass = rgl / kT, t = rgl % kT;
        float sum = 0.f;
        for (int w = 0; w < WK; ++w) sum += part[((((size_t)pass * WK + w) * kT + t) * S + s) * 8 + rr];
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
    constexpr int E = F<FMT>::E;
    if (!g_sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
    }
    const int k_pad = (int)t.k_pad;
    const int nkb = k_pad / (4 * E);
    const int WK = nkb < kWarps ? nkb : kWarps;
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
    p.k_pad = k_pad;
    p.nkb = nkb;
    p.wk = WK;
    p.rg_per_set = (t.O + 7) / 8;
    p.n_rg = p.rg_per_set * (tu ? 2 : 1);
    int grid = p.n_rg < g_sms ? p.n_rg : g_sms;
    const int need = (p.n_rg + kMaxRgPerCta - 1) / kMaxRgPerCta;
    if (grid < need) grid = need;

    // tokens per launch: the staged x and the partials must fit
    const size_t per_tok = (size_t)4 * k_pad + (size_t)kMaxPasses * WK * kT * 8 * 4;
    int s_chunk = (int)((kSmemBudget - (size_t)kMaxS * kWarps * 4 - kMaxS * 4) / per_tok);
    if (s_chunk > kMaxS) s_chunk = kMaxS;
    if (s_chunk < 1) return cudaErrorInvalidValue;  // caller takes the general path

    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(qmv_mma_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBudget);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    for (int s0 = 0; s0 < S; s0 += s_chunk) {
        const int sc = S - s0 < s_chunk ? S - s0 : s_chunk;
        p.S = sc;
        p.x = x + (long long)s0 * t.I;
        p.y[0] = y + (long long)s0 * t.O;
        p.y[1] = tu ? yu + (long long)s0 * t.O : p.y[0];
        const size_t smem = (size_t)sc * per_tok + (size_t)kMaxS * kWarps * 4 + kMaxS * 4;
        qmv_mma_kernel<FMT><<<grid, kThreads, smem, st>>>(p);
        count_launch();
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
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
    if (t.k_pad > 40960) return cudaSuccess;  // x terms of one token must fit in shared memory
    cudaError_t e = cudaSuccess;
    switch (t.fmt) {
    case B200Q_I8: e = launch_fmt<B200Q_I8>(t, tu, x, y, yu, S, st); break;
    case B200Q_I4: e = launch_fmt<B200Q_I4>(t, tu, x, y, yu, S, st); break;
    case B200Q_I2: e = launch_fmt<B200Q_I2>(t, tu, x, y, yu, S, st); break;
    default: return cudaSuccess;
    }
    if (e == cudaErrorInvalidValue) return cudaSuccess;
    *handled = (e == cudaSuccess);
    return e;
}

}  // namespace qwq
