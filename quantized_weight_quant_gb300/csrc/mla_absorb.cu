// MLA decode attention with weight absorption (three-backends chapter,
// section 四, the header of attention_absorb.comp, the Vulkan twin of
// coli_cuda_attention_absorb).  For each new token s and head h:
//     qabs[i]    = sum_d q_nope[s,h,d] * Wk[h,d,i]                (absorb)
//     score_t    = (qabs . L[t] + q_rope[s,h] . Rr[t]) * scale    t in [st0, T-S+s]
//     p          = softmax(score)
//     clat[i]    = sum_t p_t * L[t,i]                             (latent context)
//     ctx[s,h,v] = sum_i clat[i] * Wv[h,v,i]                      (value rows)
// Wk / Wv are the key and value rows of one quantized weight tensor
// [H*(Dn+Dv), K] (head h: key rows h*(Dn+Dv) + d, value rows after them),
// weight = scale * (code - zero point), one scale per row or per row and group
// of gs columns (a 32-bit code word always lies in one group).  L and Rr are the latent and rope
// caches, paged by 64 positions (the CUDA chapter's KV pages): page p holds
// positions 64p .. 64p+63 as [64, K] and [64, R] f32 rows.
//
// Four kernels.
//   1. absorb: one CTA per (head, 32 code words of a row, 4 tokens); its 16
//      warps take every 16th key row, each lane one 32-bit word of codes, and
//      the 16 partial sums are added in warp order.
//   2. attention partials, split over the cache (flash-decoding): a CTA owns
//      16 (head, token) rows and a contiguous run of 32-position tiles.  One
//      thread streams the tiles into a two-slot shared-memory ring with bulk
//      copies (cp.async.bulk, one per cache and tile, completing on the slot's
//      mbarrier; every wait bounded).  The 16 x 32 scores of a tile come from
//      a lane-split contraction over K + R: each warp keeps 4 query rows in
//      registers for the whole run (lane l holds the 4-float slices l, l + 32,
//      ...), takes 16 of the tile's positions in blocks of 4 (packed FP32x2
//      FMAs) and sums the lanes with a butterfly reduce-scatter;
//      an online softmax (running max and sum per row, f32 expf) turns them
//      into weights, and each thread adds p * L into its 4 rows x up to 12
//      columns of the latent context.  The CTA writes its rows' running max,
//      sum and unnormalised context.
//   3. combine: one CTA per (row, 128 latent columns) merges the splits
//      (weights exp(m_z - max), fixed split order) into clat.
//   4. value rows: one CTA per (head, 16 value rows, 4 tokens); each warp loads
//      all code words of its 4 rows at once and runs them against the tokens'
//      clat in shared memory.
// Positions of a tile outside [st0, T-1] are never read by the arithmetic
// (the copy may bring them in with the tile); positions past a token's causal
// limit get weight 0.  All sums are f32.
#include <math.h>

#include "qwq_internal.h"

namespace qwq {
namespace {

constexpr int kPage = B200Q_KV_PAGE_TOKENS;   // positions per cache page
constexpr int kTile = 32;                     // positions per tile (half a page)
constexpr int kRows = 16;                     // (head, token) rows per attention CTA
constexpr int kAttnThreads = 256;
constexpr int kQuads = 3;                     // latent column quads per thread: K <= 4 * 64 * kQuads
constexpr int kQG = 6;                        // float4 slices of K + R per lane: K + R <= 4 * 32 * kQG
constexpr int kTokBlock = 4;                  // tokens per absorb / value CTA
constexpr int kMaxSplit = 512;
constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s bound on any wait

__device__ unsigned int g_mla_err = 0;        // first error a kernel recorded (a B200Q_E* code, negated)

__device__ __forceinline__ void record_error(int code) { atomicCAS(&g_mla_err, 0u, (unsigned)(-code)); }

// Programmatic dependent launch: every kernel here is launched so that it may
// start while the previous kernel in the stream drains.  Each thread runs
// dependency_wait() before its first read of another kernel's output and
// before its first global write (the stream-ordered workspace may be memory a
// previous call still reads); work on the weights comes before it.
__device__ __forceinline__ void dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- 32-bit word of codes -> EW exact values (code - zero point), by the
// 2^23 + field trick: the field sits in the mantissa of 2^23, one subtraction.
template <int FMT>
struct Word;
template <>
struct Word<B200Q_F32> {
    static constexpr int EW = 1;
    static __device__ __forceinline__ void deq(uint32_t w, float (&v)[1]) { v[0] = __uint_as_float(w); }
};
template <>
struct Word<B200Q_I8> {
    static constexpr int EW = 4;
    static __device__ __forceinline__ void deq(uint32_t w, float (&v)[4]) {
        const uint32_t u = w ^ 0x80808080u;   // two's complement byte -> code + 128
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = __uint_as_float(0x4B000000u | ((u >> (8 * e)) & 0xFFu)) - 8388736.f;
    }
};
template <>
struct Word<B200Q_I4> {
    static constexpr int EW = 8;
    static __device__ __forceinline__ void deq(uint32_t w, float (&v)[8]) {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = __uint_as_float(0x4B000000u | ((w >> (4 * e)) & 0xFu)) - 8388616.f;
    }
};
template <>
struct Word<B200Q_I2> {
    static constexpr int EW = 16;
    static __device__ __forceinline__ void deq(uint32_t w, float (&v)[16]) {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(0x4B000000u | ((w >> (2 * e)) & 0x3u)) - 8388610.f;
    }
};

// ---------------------------------------------------------------- absorb
template <int FMT>
__global__ void __launch_bounds__(512) mla_absorb_kernel(const uint8_t *__restrict__ codes,
                                                         const float *__restrict__ scales, int gs, int g_ld,
                                                         long long ld, int H, int Dn, int Dv, int K,
                                                         const float *__restrict__ q_nope, int S,
                                                         float *__restrict__ qabs) {
    constexpr int EW = Word<FMT>::EW;
    constexpr int kPh = 16;                             // warps = row phases
    extern __shared__ float red[];                      // [kPh][kTokBlock][EW][32]
    const int h = blockIdx.x, s0 = blockIdx.z * kTokBlock;
    const int ns = min(kTokBlock, S - s0);
    const int lane = threadIdx.x & 31, ph = threadIdx.x >> 5;
    const int word = blockIdx.y * 32 + lane;
    const int nwords = (K + EW - 1) / EW;
    const long long key0 = (long long)h * (Dn + Dv);
    // scale of this thread's word in a row: scales[row] (gs = 0), or the
    // word's group column (a word lies in one group)
    const long long s_ld = gs ? g_ld : 1;
    const int s_col = gs ? (word * EW) / gs : 0;
    float acc[kTokBlock][EW];
#pragma unroll
    for (int t = 0; t < kTokBlock; ++t)
#pragma unroll
        for (int e = 0; e < EW; ++e) acc[t][e] = 0.f;
    bool waited = false;
    if (word < nwords) {
        constexpr int kB = EW >= 16 ? 2 : EW >= 8 ? 4 : 8;   // rows per batch: all their loads in flight
        for (int d0 = ph; d0 < Dn; d0 += kPh * kB) {
            uint32_t wb[kB];
            float sc[kB];
            float u[kB][kTokBlock];
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                const int d = d0 + b * kPh;
                wb[b] = 0u;
                sc[b] = 0.f;
                if (d < Dn) {
                    wb[b] = __ldg(reinterpret_cast<const uint32_t *>(codes + (key0 + d) * ld) + word);
                    sc[b] = __ldg(scales + (key0 + d) * s_ld + s_col);
                }
            }
            if (!waited) {                               // q_nope comes from the previous kernel
                dependency_wait();
                waited = true;
            }
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                const int d = d0 + b * kPh;
#pragma unroll
                for (int t = 0; t < kTokBlock; ++t)
                    u[b][t] = d < Dn && t < ns ? __ldg(q_nope + ((long long)(s0 + t) * H + h) * Dn + d) * sc[b] : 0.f;
            }
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                float v[EW];
                Word<FMT>::deq(wb[b], v);
#pragma unroll
                for (int t = 0; t < kTokBlock; ++t)
#pragma unroll
                    for (int e = 0; e < EW; ++e) acc[t][e] = fmaf(u[b][t], v[e], acc[t][e]);
            }
        }
    }
    if (!waited) dependency_wait();
#pragma unroll
    for (int t = 0; t < kTokBlock; ++t)
#pragma unroll
        for (int e = 0; e < EW; ++e) red[((ph * kTokBlock + t) * EW + e) * 32 + lane] = acc[t][e];
    __syncthreads();
    constexpr int kOut = kTokBlock * EW * 32;
    for (int o = threadIdx.x; o < kOut; o += blockDim.x) {
        float sum = 0.f;
#pragma unroll
        for (int p = 0; p < kPh; ++p) sum += red[p * kOut + o];
        const int t = o / (EW * 32), e = (o / 32) % EW, ln = o % 32;
        const int col = (blockIdx.y * 32 + ln) * EW + e;
        if (t < ns && col < K) qabs[((long long)(s0 + t) * H + h) * K + col] = sum;
    }
}

// ---------------------------------------------------------------- attention partials
struct AttnParams {
    const float *qabs;                 // [S, H, K]
    const float *q_rope;               // [S, H, R]
    const float *const *lat_pages;     // device array of page pointers, [64, K] f32 each
    const float *const *rope_pages;    // device array of page pointers, [64, R] f32 each
    float *part_m, *part_l;            // [n_split][H*S]
    float *part_c;                     // [n_split][H*S][K]
    int H, S, K, R, T, st0;
    float scale;
    int tile0, n_tiles, n_split;       // first tile (st0 / 32) and tiles of the window
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

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

// Butterfly reduce-scatter of 16 values over a warp: afterwards lane l holds
// the full sum of value index l >> 1.
__device__ __forceinline__ float reduce16(float (&v)[16], int lane) {
#pragma unroll
    for (int n = 16, off = 16; n > 1; n >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < n / 2) {
                const float send = upper ? v[i] : v[i + n / 2];
                const float keep = upper ? v[i + n / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// KT, RT > 0: latent and rope widths fixed at compile time (strides and
// loop bounds resolved by the compiler); 0: taken from p.
template <int KT, int RT>
__global__ void __launch_bounds__(kAttnThreads, 1) mla_attn_kernel(const __grid_constant__ AttnParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int K = KT ? KT : p.K, R = KT ? RT : p.R, KR = K + R, HS = p.H * p.S;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float *qs = reinterpret_cast<float *>(smem);       // [kRows][KR]: qabs | q_rope
    float *ls = qs + kRows * KR;                        // [2][kTile][K]
    float *rs = ls + 2 * kTile * K;                     // [2][kTile][R]
    float *ps = rs + 2 * kTile * R;                     // [kTile][kRows]: scores, then weights
    float *alpha = ps + kTile * kRows;                  // [kRows]
    uint64_t *bars = reinterpret_cast<uint64_t *>(alpha + kRows);   // [2]
    const uint32_t bar0 = smem_u32(bars);

    const int r0 = blockIdx.y * kRows;
    const int z = blockIdx.x;
    const int j0 = (int)((long long)z * p.n_tiles / p.n_split), j1 = (int)((long long)(z + 1) * p.n_tiles / p.n_split);
    const int nt = j1 - j0;                             // >= 1 (n_split <= n_tiles)

    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0 + 8) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    dependency_wait();   // qabs (and the cache rows appended before it) come from earlier kernels

    // thread 0: tile j of this CTA's run into slot j & 1
    auto issue = [&](int j) {
        const int pos0 = (p.tile0 + j0 + j) * kTile;
        const int page = pos0 / kPage, off = pos0 % kPage;
        const float *lp = p.lat_pages[page];
        const float *rp = R ? p.rope_pages[page] : nullptr;
        const bool ok = lp && ((uintptr_t)lp & 15u) == 0 && (!R || (rp && ((uintptr_t)rp & 15u) == 0));
        if (!ok) record_error(B200Q_EINVAL);
        const uint32_t lbytes = ok ? (uint32_t)(kTile * K * 4) : 0u, rbytes = ok ? (uint32_t)(kTile * R * 4) : 0u;
        const uint32_t bar = bar0 + 8 * (j & 1);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(lbytes + rbytes)
                     : "memory");
        if (ok) {
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(ls + (j & 1) * kTile * K)),
                "l"(lp + (size_t)off * K), "r"(lbytes), "r"(bar)
                : "memory");
            if (R)
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                        smem_u32(rs + (j & 1) * kTile * R)),
                    "l"(rp + (size_t)off * R), "r"(rbytes), "r"(bar)
                    : "memory");
        }
    };
    if (tid == 0) {
        issue(0);
        if (nt > 1) issue(1);
    }

    // the CTA's query rows (rows past H*S are zero), as float4 (K, R multiples
    // of 4), every load of a thread issued before the first store
    {
        const int n4 = kRows * KR / 4, kr4 = KR / 4;
        constexpr int kLd = (kRows * 716 / 4 + kAttnThreads - 1) / kAttnThreads;
        float4 v[kLd];
#pragma unroll
        for (int k = 0; k < kLd; ++k) {
            const int idx = tid + k * kAttnThreads;
            v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (idx < n4) {
                const int m = idx / kr4, i = 4 * (idx - m * kr4), r = r0 + m;
                if (r < HS) {
                    const int h = r / p.S, s = r - h * p.S;
                    v[k] = i < K ? *reinterpret_cast<const float4 *>(p.qabs + ((long long)s * p.H + h) * K + i)
                                 : *reinterpret_cast<const float4 *>(p.q_rope + ((long long)s * p.H + h) * R + (i - K));
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kLd; ++k) {
            const int idx = tid + k * kAttnThreads;
            if (idx < n4) reinterpret_cast<float4 *>(qs)[idx] = v[k];
        }
    }
    // per-warp running max / sum of its two rows (softmax phase)
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    int last_pos[2];
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
        const int r = r0 + warp * 2 + mi;
        last_pos[mi] = r < HS ? p.T - p.S + (r % p.S) : -1;
    }
    // latent context accumulators: rows 4 mg .. 4 mg + 3, column quads c + 64 q
    const int mg = tid >> 6, cq = tid & 63, nK4 = K / 4;
    float4 acc[4][kQuads];
#pragma unroll
    for (int mi = 0; mi < 4; ++mi)
#pragma unroll
        for (int q = 0; q < kQuads; ++q) acc[mi][q] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    // score operand: this warp's 4 query rows, lane slices g = lane + 32 k
    const int mb = warp & 3, th = warp >> 2;          // row block; position half of the tile
    const int ng = KR / 4;
    float4 qreg[4][kQG];
#pragma unroll
    for (int k = 0; k < kQG; ++k) {
        const int g = lane + 32 * k;
#pragma unroll
        for (int mi = 0; mi < 4; ++mi)
            qreg[mi][k] = g < ng ? *reinterpret_cast<const float4 *>(qs + (mb * 4 + mi) * KR + 4 * g)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    bool ok = true;
    for (int j = 0; j < nt; ++j) {
        const int slot = j & 1;
        const bool arrived = mbar_wait(bar0 + 8 * slot, (uint32_t)((j >> 1) & 1), kWaitNs);
        if (__syncthreads_or(!arrived)) {
            ok = false;
            break;
        }
        const float *lt = ls + slot * kTile * K;
        const float *rt = rs + slot * kTile * R;
        const int pos0 = (p.tile0 + j0 + j) * kTile;
        // positions of this tile the arithmetic reads: [st0, T-1]
        const int tv0 = max(p.st0 - pos0, 0), tv1 = min(p.T - pos0, kTile);

        // scores: each warp 4 rows (in registers) x its 16 positions in
        // blocks of 4, lanes over float4 slices of K + R
        for (int tb = th * 4; tb < th * 4 + 4; ++tb) {
            float2 a2[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) a2[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < kQG; ++k) {
                const int g = lane + 32 * k;
                if (g >= ng) break;
                float4 lv[4];
                if (g < nK4) {
#pragma unroll
                    for (int ti = 0; ti < 4; ++ti) lv[ti] = *reinterpret_cast<const float4 *>(lt + (tb * 4 + ti) * K + 4 * g);
                } else {
#pragma unroll
                    for (int ti = 0; ti < 4; ++ti)
                        lv[ti] = *reinterpret_cast<const float4 *>(rt + (tb * 4 + ti) * R + 4 * (g - nK4));
                }
#pragma unroll
                for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                    for (int ti = 0; ti < 4; ++ti) {
                        float2 &a = a2[mi * 4 + ti];
                        a = __ffma2_rn(make_float2(qreg[mi][k].x, qreg[mi][k].y), make_float2(lv[ti].x, lv[ti].y), a);
                        a = __ffma2_rn(make_float2(qreg[mi][k].z, qreg[mi][k].w), make_float2(lv[ti].z, lv[ti].w), a);
                    }
            }
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = a2[i].x + a2[i].y;
            const float sum = reduce16(v, lane);
            if ((lane & 1) == 0) {
                const int idx = lane >> 1, mi = idx >> 2, ti = idx & 3;
                ps[(tb * 4 + ti) * kRows + mb * 4 + mi] = sum * p.scale;
            }
        }
        __syncthreads();

        // online softmax: warp w owns rows 2w, 2w + 1; lane = position
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
            const int m = warp * 2 + mi;
            const int pos = pos0 + lane;
            const bool valid = lane >= tv0 && lane < tv1 && pos <= last_pos[mi];
            const float sc = valid ? ps[lane * kRows + m] : -INFINITY;
            float tmax = sc;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
            const float m_new = fmaxf(m_run[mi], tmax);
            const float a = m_new == -INFINITY ? 1.f : expf(m_run[mi] - m_new);
            const float pv = valid ? expf(sc - m_new) : 0.f;
            float psum = pv;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
            l_run[mi] = l_run[mi] * a + psum;
            m_run[mi] = m_new;
            ps[lane * kRows + m] = pv;
            if (lane == 0) alpha[m] = a;
        }
        __syncthreads();

        // latent context: acc = alpha * acc + sum_t p_t * L[t]
        {
            float al[4];
#pragma unroll
            for (int mi = 0; mi < 4; ++mi) al[mi] = alpha[mg * 4 + mi];
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int q = 0; q < kQuads; ++q) {
                    acc[mi][q].x *= al[mi];
                    acc[mi][q].y *= al[mi];
                    acc[mi][q].z *= al[mi];
                    acc[mi][q].w *= al[mi];
                }
            auto add_position = [&](int t) {
                const float4 pv = *reinterpret_cast<const float4 *>(ps + t * kRows + mg * 4);
                const float pm[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
                for (int q = 0; q < kQuads; ++q) {
                    const int c4 = cq + 64 * q;
                    if (c4 < nK4) {
                        const float4 lv = *reinterpret_cast<const float4 *>(lt + t * K + 4 * c4);
#pragma unroll
                        for (int mi = 0; mi < 4; ++mi) {
                            const float2 pp2 = make_float2(pm[mi], pm[mi]);
                            float2 lo = __ffma2_rn(pp2, make_float2(lv.x, lv.y), make_float2(acc[mi][q].x, acc[mi][q].y));
                            float2 hi = __ffma2_rn(pp2, make_float2(lv.z, lv.w), make_float2(acc[mi][q].z, acc[mi][q].w));
                            acc[mi][q] = make_float4(lo.x, lo.y, hi.x, hi.y);
                        }
                    }
                }
            };
            if (tv0 == 0 && tv1 == kTile) {           // a whole tile: fixed trip count
#pragma unroll 8
                for (int t = 0; t < kTile; ++t) add_position(t);
            } else {
                for (int t = tv0; t < tv1; ++t) add_position(t);
            }
        }
        __syncthreads();   // slot and weights free: refill the slot with tile j + 2
        if (tid == 0 && j + 2 < nt) issue(j + 2);
    }
    if (!ok) {
        // give up: record it and let the copies in flight land (bounded)
        if (tid == 0) {
            record_error(B200Q_ETIMEOUT);
            mbar_wait(bar0, 0, kWaitNs / 4);
            mbar_wait(bar0 + 8, 0, kWaitNs / 4);
        }
        __syncthreads();
        return;
    }

    // this split's running max, sum and unnormalised context per row
    if (lane == 0) {
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
            const int r = r0 + warp * 2 + mi;
            if (r < HS) {
                p.part_m[(long long)z * HS + r] = m_run[mi];
                p.part_l[(long long)z * HS + r] = l_run[mi];
            }
        }
    }
#pragma unroll
    for (int mi = 0; mi < 4; ++mi) {
        const int r = r0 + mg * 4 + mi;
        if (r >= HS) continue;
        float *dst = p.part_c + ((long long)z * HS + r) * K;
#pragma unroll
        for (int q = 0; q < kQuads; ++q) {
            const int c4 = cq + 64 * q;
            if (c4 < nK4) reinterpret_cast<float4 *>(dst)[c4] = acc[mi][q];
        }
    }
}

// ---------------------------------------------------------------- combine
// One CTA per (row, 128 latent columns): each thread issues the loads of its
// column's partials first (64 at a time), warp 0 meanwhile forms the split
// weights exp(m_z - max) in shared memory, then the column is summed over the
// splits in a fixed order.
constexpr int kCombThreads = 128;

__global__ void __launch_bounds__(kCombThreads) mla_combine_kernel(const float *__restrict__ part_m,
                                                                   const float *__restrict__ part_l,
                                                                   const float *__restrict__ part_c, int n_split,
                                                                   int HS, int K, float *__restrict__ clat) {
    __shared__ float wz[kMaxSplit];
    __shared__ float inv_l;
    const int r = blockIdx.x, i = blockIdx.y * kCombThreads + threadIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    dependency_wait();
    // the first kB partials of this column go out before the split weights are
    // formed (they do not depend on them)
    constexpr int kB = 64;
    float pv[kB];
#pragma unroll
    for (int b = 0; b < kB; ++b)
        pv[b] = i < K && b < n_split ? part_c[((long long)b * HS + r) * K + i] : 0.f;
    if (warp == 0) {
        float mx = -INFINITY;
        for (int z = lane; z < n_split; z += 32) mx = fmaxf(mx, part_m[(long long)z * HS + r]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float lsum = 0.f;
        for (int z = lane; z < n_split; z += 32) {
            const float mz = part_m[(long long)z * HS + r];
            const float w = mz == -INFINITY ? 0.f : expf(mz - mx);
            wz[z] = w;
            lsum += w * part_l[(long long)z * HS + r];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
        if (lane == 0) inv_l = 1.f / lsum;
    }
    __syncthreads();
    if (i >= K) return;
    float c = 0.f;
#pragma unroll
    for (int b = 0; b < kB; ++b)
        if (b < n_split) c = fmaf(wz[b], pv[b], c);
    for (int z0 = kB; z0 < n_split; z0 += kB) {      // more than kB splits: further batches
#pragma unroll
        for (int b = 0; b < kB; ++b) pv[b] = z0 + b < n_split ? part_c[((long long)(z0 + b) * HS + r) * K + i] : 0.f;
#pragma unroll
        for (int b = 0; b < kB; ++b)
            if (z0 + b < n_split) c = fmaf(wz[z0 + b], pv[b], c);
    }
    clat[(long long)r * K + i] = c * inv_l;
}

// ---------------------------------------------------------------- value rows
// One CTA per (head, 16 value rows, 4 tokens): the tokens' latent contexts in
// shared memory; each warp loads all code words of its 4 rows at once, lanes
// over words (a word's columns read as float4 from shared memory).
constexpr int kValThreads = 128;
constexpr int kValRows = 16;                     // per CTA: 4 warps x 4 rows

template <int FMT>
__global__ void __launch_bounds__(kValThreads) mla_value_kernel(const uint8_t *__restrict__ codes,
                                                                const float *__restrict__ scales, int gs, int g_ld,
                                                                long long ld, int H, int Dn, int Dv, int K, int S,
                                                                const float *__restrict__ clat_g,
                                                                float *__restrict__ ctx) {
    constexpr int EW = Word<FMT>::EW;
    constexpr int kWL = (768 / EW + 31) / 32;        // words of a row per lane (K <= 768)
    extern __shared__ __align__(16) float clat[];    // [kTokBlock][K]
    const int h = blockIdx.x, s0 = blockIdx.z * kTokBlock;
    const int ns = min(kTokBlock, S - s0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwords = (K + EW - 1) / EW;
    const long long val0 = (long long)h * (Dn + Dv) + Dn;
    const int v0 = blockIdx.y * kValRows + warp * 4;
    uint32_t cw[4][kWL];
    float sc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const bool live = v0 + k < Dv;
        const uint32_t *row = reinterpret_cast<const uint32_t *>(codes + (val0 + (live ? v0 + k : 0)) * ld);
        sc[k] = live && !gs ? __ldg(scales + val0 + v0 + k) : 1.f;
#pragma unroll
        for (int b = 0; b < kWL; ++b) cw[k][b] = live && lane + 32 * b < nwords ? __ldg(row + lane + 32 * b) : 0u;
    }
    dependency_wait();   // clat comes from the combine kernel
    for (int idx = threadIdx.x; idx < ns * K / 4; idx += blockDim.x) {
        const int t = idx / (K / 4), i4 = idx - t * (K / 4);
        reinterpret_cast<float4 *>(clat)[idx] =     // clat rows are (head, token), head-major
            reinterpret_cast<const float4 *>(clat_g + ((long long)h * S + s0 + t) * K)[i4];
    }
    __syncthreads();
    float a[4][kTokBlock];
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int t = 0; t < kTokBlock; ++t) a[k][t] = 0.f;
#pragma unroll
    for (int b = 0; b < kWL; ++b) {
        const int wd = lane + 32 * b;
        if (wd >= nwords) break;
#pragma unroll
        for (int t = 0; t < kTokBlock; ++t) {
            if (t >= ns) break;
            float cl[EW];
            if constexpr (EW >= 4) {
#pragma unroll
                for (int e4 = 0; e4 < EW; e4 += 4) {
                    const float4 c4 = *reinterpret_cast<const float4 *>(clat + t * K + wd * EW + e4);
                    cl[e4] = c4.x;
                    cl[e4 + 1] = c4.y;
                    cl[e4 + 2] = c4.z;
                    cl[e4 + 3] = c4.w;
                }
            } else {
                cl[0] = clat[t * K + wd];
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float wv[EW];
                Word<FMT>::deq(cw[k][b], wv);
                if (gs) {   // the word's partial sum times its group scale
                    float part = 0.f;
#pragma unroll
                    for (int e = 0; e < EW; ++e) part = fmaf(wv[e], cl[e], part);
                    const bool live = v0 + k < Dv;
                    const float g = live ? __ldg(scales + (val0 + v0 + k) * g_ld + (wd * EW) / gs) : 0.f;
                    a[k][t] = fmaf(g, part, a[k][t]);
                } else {
#pragma unroll
                    for (int e = 0; e < EW; ++e) a[k][t] = fmaf(wv[e], cl[e], a[k][t]);
                }
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int t = 0; t < kTokBlock; ++t)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) a[k][t] += __shfl_xor_sync(0xffffffffu, a[k][t], off);
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (v0 + k < Dv)
                for (int t = 0; t < ns; ++t) ctx[((long long)(s0 + t) * H + h) * Dv + v0 + k] = sc[k] * a[k][t];
    }
}

// ---------------------------------------------------------------- bounded-wait self test
// One thread waits, with the given limit, on an mbarrier that nothing
// arrives on: the wait gives up and records B200Q_ETIMEOUT exactly as a
// kernel whose copies never land would (b200q_selftest_timeout).
__global__ void wait_selftest_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!mbar_wait(b, 0, limit_ns)) record_error(B200Q_ETIMEOUT);
    }
}

// ---------------------------------------------------------------- cache append
__global__ void kv_append_kernel(float *const *lat_pages, float *const *rope_pages, int K, int R, int pos,
                                 const float *__restrict__ lat_rows, const float *__restrict__ rope_rows, int n) {
    const int i = blockIdx.x;
    if (i >= n) return;
    const int at = pos + i, page = at / kPage, off = at % kPage;
    float *lp = lat_pages[page];
    float *rp = R ? rope_pages[page] : nullptr;
    if (!lp || (R && !rp)) {
        if (threadIdx.x == 0) record_error(B200Q_EINVAL);
        return;
    }
    for (int k = threadIdx.x; k < K; k += blockDim.x) lp[(size_t)off * K + k] = lat_rows[(size_t)i * K + k];
    for (int k = threadIdx.x; k < R; k += blockDim.x) rp[(size_t)off * R + k] = rope_rows[(size_t)i * R + k];
}

template <class... P, class... A>
cudaError_t launch_pdl(void (*k)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, A... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k, args...);
    count_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <class Kern>
cudaError_t allow_smem(Kern k, size_t bytes) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    return allow_dynamic_smem((const void *)k, 227 * 1024);
}

template <int FMT>
cudaError_t run_absorb(const Tensor &w, int H, int Dn, int Dv, const float *q_nope, int S, float *qabs,
                       cudaStream_t st) {
    constexpr int EW = Word<FMT>::EW;
    const size_t smem = (size_t)16 * kTokBlock * EW * 32 * 4;   // int2: 128 KB
    cudaError_t e = allow_smem(mla_absorb_kernel<FMT>, smem);
    if (e != cudaSuccess) return e;
    const int K = w.I, nwords = (K + EW - 1) / EW;
    dim3 grid(H, (nwords + 31) / 32, (S + kTokBlock - 1) / kTokBlock);
    return launch_pdl(mla_absorb_kernel<FMT>, grid, dim3(512), smem, st, (const uint8_t *)w.codes,
                      (const float *)w.scales, w.gs, w.G_ld, (long long)w.ld, H, Dn, Dv, K, q_nope, S, qabs);
}

template <int FMT>
cudaError_t run_value(const Tensor &w, int H, int Dn, int Dv, int S, const float *clat, float *ctx,
                      cudaStream_t st) {
    const int K = w.I;
    const size_t smem = (size_t)kTokBlock * K * 4;     // <= 12 KB
    dim3 grid(H, (Dv + kValRows - 1) / kValRows, (S + kTokBlock - 1) / kTokBlock);
    return launch_pdl(mla_value_kernel<FMT>, grid, dim3(kValThreads), smem, st, (const uint8_t *)w.codes,
                      (const float *)w.scales, w.gs, w.G_ld, (long long)w.ld, H, Dn, Dv, K, S, (const float *)clat,
                      ctx);
}

}  // namespace

size_t mla_smem_bytes(int K, int R) {
    return ((size_t)kRows * (K + R) + (size_t)2 * kTile * (K + R) + (size_t)kTile * kRows + kRows) * 4 + 16;
}

int mla_max_latent() { return 4 * 64 * kQuads; }

// Workspace floats a call needs (qabs + split partials); n_split from the
// same rule the launcher uses.
static int mla_splits(int H, int S, int T, int st0) {
    int dev = 0;
    cudaGetDevice(&dev);
    const int n_sms = sm_count(dev);
    const int rb = (H * S + kRows - 1) / kRows;
    const int n_tiles = (T - 1) / kTile - st0 / kTile + 1;
    int n = (n_sms + rb - 1) / rb;
    if (n > n_tiles) n = n_tiles;
    if (n > kMaxSplit) n = kMaxSplit;
    return n < 1 ? 1 : n;
}

size_t mla_workspace_floats(int H, int S, int K, int T, int st0) {
    const int n = mla_splits(H, S, T, st0);
    const size_t hs = (size_t)H * S;
    return hs * K + 2 * (size_t)n * hs + (size_t)n * hs * K + 8;
}

cudaError_t launch_mla_absorb(const Tensor &w, int H, int Dn, int Dv, const float *q_nope, const float *q_rope,
                              const float *const *lat_pages, const float *const *rope_pages, int R, int T, int st0,
                              float scale, float *ctx, int S, float *ws, cudaStream_t st) {
    const int K = w.I, HS = H * S;
    const int n_split = mla_splits(H, S, T, st0);
    float *qabs = ws;
    float *pm = qabs + (size_t)HS * K;
    float *pl = pm + (size_t)n_split * HS;
    float *pc = pl + (size_t)n_split * HS;
    pc = reinterpret_cast<float *>(((uintptr_t)pc + 15) & ~(uintptr_t)15);
    cudaError_t e = cudaSuccess;
    switch (w.fmt) {
    case B200Q_F32: e = run_absorb<B200Q_F32>(w, H, Dn, Dv, q_nope, S, qabs, st); break;
    case B200Q_I8: e = run_absorb<B200Q_I8>(w, H, Dn, Dv, q_nope, S, qabs, st); break;
    case B200Q_I4: e = run_absorb<B200Q_I4>(w, H, Dn, Dv, q_nope, S, qabs, st); break;
    case B200Q_I2: e = run_absorb<B200Q_I2>(w, H, Dn, Dv, q_nope, S, qabs, st); break;
    default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;

    AttnParams p;
    p.qabs = qabs;
    p.q_rope = q_rope;
    p.lat_pages = lat_pages;
    p.rope_pages = rope_pages;
    p.part_m = pm;
    p.part_l = pl;
    p.part_c = pc;
    p.H = H;
    p.S = S;
    p.K = K;
    p.R = R;
    p.T = T;
    p.st0 = st0;
    p.scale = scale;
    p.tile0 = st0 / kTile;
    p.n_tiles = (T - 1) / kTile - p.tile0 + 1;
    p.n_split = n_split;
    const size_t smem = mla_smem_bytes(K, R);
    dim3 grid(n_split, (HS + kRows - 1) / kRows);
    if (K == 512 && R == 64) {      // the pages' model shape: widths fixed at compile time
        e = allow_smem(mla_attn_kernel<512, 64>, smem);
        if (e != cudaSuccess) return e;
        e = launch_pdl(mla_attn_kernel<512, 64>, grid, dim3(kAttnThreads), smem, st, p);
    } else {
        e = allow_smem(mla_attn_kernel<0, 0>, smem);
        if (e != cudaSuccess) return e;
        e = launch_pdl(mla_attn_kernel<0, 0>, grid, dim3(kAttnThreads), smem, st, p);
    }
    if (e != cudaSuccess) return e;

    // the splits merged into clat (the qabs buffer, which the attention
    // kernel has finished with), then the value rows
    float *clat = qabs;
    e = launch_pdl(mla_combine_kernel, dim3(HS, (K + kCombThreads - 1) / kCombThreads), dim3(kCombThreads), 0, st,
                   (const float *)pm, (const float *)pl, (const float *)pc, n_split, HS, K, clat);
    if (e != cudaSuccess) return e;
    switch (w.fmt) {
    case B200Q_F32: return run_value<B200Q_F32>(w, H, Dn, Dv, S, clat, ctx, st);
    case B200Q_I8: return run_value<B200Q_I8>(w, H, Dn, Dv, S, clat, ctx, st);
    case B200Q_I4: return run_value<B200Q_I4>(w, H, Dn, Dv, S, clat, ctx, st);
    default: return run_value<B200Q_I2>(w, H, Dn, Dv, S, clat, ctx, st);
    }
}

cudaError_t launch_kv_append(float *const *lat_pages, float *const *rope_pages, int K, int R, int pos,
                             const float *lat_rows, const float *rope_rows, int n, cudaStream_t st) {
    kv_append_kernel<<<n, 128, 0, st>>>(lat_pages, rope_pages, K, R, pos, lat_rows, rope_rows, n);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(limit_ns);
    count_launch();
    return cudaGetLastError();
}

// Reads and clears the MLA kernels' device error word (0: none).
cudaError_t mla_take_error(unsigned int *code) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_mla_err, sizeof(unsigned int));
    if (e == cudaSuccess && *code) e = cudaMemcpyToSymbol(g_mla_err, &zero, sizeof(unsigned int));
    return e;
}

}  // namespace qwq
