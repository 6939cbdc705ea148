// SIMT quantized matmul: the f32-accurate path for every format and any S.
//
// y[s,o] = scale[o] * sum_i deq(W[o,i]) * x[s,i]  ("CUDA 后端", section 1:
// weight_at / quant_matmul; three-backends chapter, section 四: qmatmul.comp).
//
// One warp owns one weight row at a time and reads it once per token block
// with 16-byte coalesced loads (lane l takes 16-byte chunks l, l+32, ...).
// Each chunk is dequantized in registers and multiplied against up to
// kTok tokens of x; a chunk's products are summed into a chunk-local
// register before they join the lane's running sum, so no f32 sum runs over
// more than (elements per chunk + chunks per lane) terms.  The 32 lane sums
// are combined with shuffles and the scale is applied once per row.
//
// Group-wise scales (one scale per row and group of gs columns, the group
// size of the Vulkan tensor in the three-backends chapter, section 三): the
// chunk-local sum is scaled by its group's scale before it joins the lane's
// sum (gs a multiple of the chunk's element count), or the chunk is split into
// groups of 16 or 32 elements, each summed and scaled on its own.
//
// This kernel is the general path (f32 weights, int2, every S, group-wise
// scales); the decode kernels and the tensor-core kernels are faster on their
// shapes.
#include "qwq_internal.h"

namespace qwq {
namespace {

constexpr int kTok = 4;          // tokens per pass over a row
constexpr int kWarps = 8;        // warps per CTA

template <int FMT>
struct Deq;

// Each specialization turns one 16-byte chunk (4 words) into its values.
template <>
struct Deq<B200Q_F32> {
    static constexpr int kPerChunk = 4;
    __device__ static void run(const uint4 &c, float *w) {
        w[0] = __uint_as_float(c.x);
        w[1] = __uint_as_float(c.y);
        w[2] = __uint_as_float(c.z);
        w[3] = __uint_as_float(c.w);
    }
};

template <>
struct Deq<B200Q_I8> {
    static constexpr int kPerChunk = 16;
    __device__ static void run(const uint4 &c, float *w) {
        const uint32_t v[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int b = 0; b < 4; ++b)
                w[4 * q + b] = (float)(int)(int8_t)((v[q] >> (8 * b)) & 0xFFu);
    }
};

template <>
struct Deq<B200Q_I4> {
    static constexpr int kPerChunk = 32;
    __device__ static void run(const uint4 &c, float *w) {
        const uint32_t v[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int n = 0; n < 8; ++n)
                w[8 * q + n] = (float)((int)((v[q] >> (4 * n)) & 0xFu) - 8);
    }
};

template <>
struct Deq<B200Q_I2> {
    static constexpr int kPerChunk = 64;
    __device__ static void run(const uint4 &c, float *w) {
        const uint32_t v[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int n = 0; n < 16; ++n)
                w[16 * q + n] = (float)((int)((v[q] >> (2 * n)) & 0x3u) - 2);
    }
};

struct RowSet {
    const uint8_t *codes;
    const float *scales;   // [O] per row, or [O, G] per row and group (row stride G)
    float *y;
    int gs;                // 0: per-row scales
    int G;                 // row stride of the group scales
};

// SUB = 0: per-row scales, or groups that are whole chunks (gs a multiple of
// the chunk's element count); SUB = 16 or 32: groups of SUB elements inside
// a chunk.
template <int FMT, int SUB>
__global__ void __launch_bounds__(kWarps * 32)
qmv_simt_kernel(RowSet a, RowSet b, int n_sets, int O, int I, long long ld, const float *__restrict__ x,
                int S) {
    using D = Deq<FMT>;
    static_assert(SUB == 0 || D::kPerChunk % SUB == 0, "groups inside a chunk");
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int s0 = blockIdx.y * kTok;
    const int ns = min(kTok, S - s0);
    const long long n_chunks = ld / 16;
    const long long rows_total = (long long)O * n_sets;

    for (long long r = (long long)blockIdx.x * kWarps + warp; r < rows_total;
         r += (long long)gridDim.x * kWarps) {
        const RowSet &rs = (r < O) ? a : b;
        const int o = (int)(r < O ? r : r - O);
        const uint4 *row = reinterpret_cast<const uint4 *>(rs.codes + (long long)o * ld);
        float acc[kTok];
#pragma unroll
        for (int t = 0; t < kTok; ++t) acc[t] = 0.f;

        for (long long c = lane; c < n_chunks; c += 32) {
            const long long k0 = c * D::kPerChunk;
            if (k0 >= I) break;                 // the rest of the row is padding
            uint4 raw = __ldg(row + c);
            float w[D::kPerChunk];
            D::run(raw, w);
            const int kn = (int)min((long long)D::kPerChunk, (long long)I - k0);
            if constexpr (SUB == 0) {
                // per-row scale (applied at the end), or the chunk's group scale
                const float gsc = rs.gs ? rs.scales[(long long)o * rs.G + k0 / rs.gs] : 1.f;
#pragma unroll
                for (int t = 0; t < kTok; ++t) {
                    if (t < ns) {
                        const float *xs = x + (long long)(s0 + t) * I + k0;
                        float part = 0.f;
                        if (kn == D::kPerChunk) {
#pragma unroll
                            for (int j = 0; j < D::kPerChunk; ++j) part = fmaf(w[j], __ldg(xs + j), part);
                        } else {
                            for (int j = 0; j < kn; ++j) part = fmaf(w[j], __ldg(xs + j), part);
                        }
                        acc[t] = rs.gs ? fmaf(part, gsc, acc[t]) : acc[t] + part;
                    }
                }
            } else {
                // groups of SUB elements: each summed, scaled and added on its own
                const float *gsc = rs.scales + (long long)o * rs.G + k0 / SUB;
#pragma unroll
                for (int t = 0; t < kTok; ++t) {
                    if (t < ns) {
                        const float *xs = x + (long long)(s0 + t) * I + k0;
#pragma unroll
                        for (int g = 0; g < D::kPerChunk / SUB; ++g) {
                            float part = 0.f;
                            if (kn == D::kPerChunk) {
#pragma unroll
                                for (int j = 0; j < SUB; ++j) part = fmaf(w[g * SUB + j], __ldg(xs + g * SUB + j), part);
                            } else {
#pragma unroll
                                for (int j = 0; j < SUB; ++j)
                                    if (g * SUB + j < kn) part = fmaf(w[g * SUB + j], __ldg(xs + g * SUB + j), part);
                            }
                            if (g * SUB < kn) acc[t] = fmaf(part, gsc[g], acc[t]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kTok; ++t) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
        }
        if (lane == 0) {
            const float sc = rs.gs ? 1.f : rs.scales[o];
#pragma unroll
            for (int t = 0; t < kTok; ++t)
                if (t < ns) rs.y[(long long)(s0 + t) * O + o] = rs.gs ? acc[t] : sc * acc[t];
        }
    }
}

__global__ void fix_row_tails_kernel(uint8_t *codes, int O, long long ld, long long rb, uint8_t keep_mask,
                                     uint8_t zero) {
    const int o = blockIdx.x * blockDim.x + threadIdx.x;
    if (o >= O) return;
    uint8_t *p = codes + (long long)o * ld + (rb - 1);
    *p = (uint8_t)((*p & keep_mask) | (zero & (uint8_t)~keep_mask));
}

__global__ void silu_mul_kernel(const float *__restrict__ g, const float *__restrict__ u, float *h, long n) {
    const long n4 = n / 4;
    const long stride = (long)gridDim.x * blockDim.x;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        float4 a = reinterpret_cast<const float4 *>(g)[i];
        float4 b = reinterpret_cast<const float4 *>(u)[i];
        float4 r;
        r.x = a.x / (1.f + expf(-a.x)) * b.x;
        r.y = a.y / (1.f + expf(-a.y)) * b.y;
        r.z = a.z / (1.f + expf(-a.z)) * b.z;
        r.w = a.w / (1.f + expf(-a.w)) * b.w;
        reinterpret_cast<float4 *>(h)[i] = r;
    }
    for (long i = n4 * 4 + (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        h[i] = g[i] / (1.f + expf(-g[i])) * u[i];
}

// Layer glue kept on the device (colibri CUDA docs, "The GPU-resident
// pipeline": the norms and residual adds run on the GPU).  Textbook RMSNorm
// with an optional residual, one block per row:
//     h = x + r (r may be NULL: h = x),  y = h * w / sqrt(mean(h^2) + eps)
// h is stored when h_out is given (it may be x or r itself: the residual
// stream updated in place).  Rows of up to kRmsHeld float4 per thread stay in
// registers between the two passes; longer rows are read again (from h_out
// when given).  1 / sqrt uses the correctly rounded square root and division.
constexpr int kRmsThreads = 256;
constexpr int kRmsHeld = 8;

__global__ void __launch_bounds__(kRmsThreads)
    rmsnorm_kernel(const float *x, const float *r, float *h_out, const float *__restrict__ w, float *y, int D,
                   float eps) {
    const long long off = (long long)blockIdx.x * D;
    const int tid = threadIdx.x;
    __shared__ float red[kRmsThreads / 32];
    float ss = 0.f;
    if ((D & 3) == 0) {
        const int D4 = D / 4;
        const float4 *x4 = reinterpret_cast<const float4 *>(x + off);
        const float4 *r4 = r ? reinterpret_cast<const float4 *>(r + off) : nullptr;
        float4 *h4 = h_out ? reinterpret_cast<float4 *>(h_out + off) : nullptr;
        auto hval = [&](int k) {
            float4 v = x4[k];
            if (r4) {
                const float4 b = r4[k];
                v = make_float4(v.x + b.x, v.y + b.y, v.z + b.z, v.w + b.w);
            }
            return v;
        };
        float4 held[kRmsHeld];
#pragma unroll
        for (int i = 0; i < kRmsHeld; ++i) {
            const int k = i * kRmsThreads + tid;
            held[i] = k < D4 ? hval(k) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kRmsHeld; ++i) {
            const int k = i * kRmsThreads + tid;
            if (k < D4 && h4) h4[k] = held[i];
            ss += held[i].x * held[i].x + held[i].y * held[i].y + held[i].z * held[i].z + held[i].w * held[i].w;
        }
        for (int k = kRmsHeld * kRmsThreads + tid; k < D4; k += kRmsThreads) {
            const float4 v = hval(k);
            if (h4) h4[k] = v;
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if ((tid & 31) == 0) red[tid >> 5] = ss;
        __syncthreads();
        ss = 0.f;
#pragma unroll
        for (int i = 0; i < kRmsThreads / 32; ++i) ss += red[i];
        const float inv = 1.f / sqrtf(ss / (float)D + eps);
        const float4 *w4 = reinterpret_cast<const float4 *>(w);
        float4 *y4 = reinterpret_cast<float4 *>(y + off);
#pragma unroll
        for (int i = 0; i < kRmsHeld; ++i) {
            const int k = i * kRmsThreads + tid;
            if (k < D4) {
                const float4 g = w4[k];
                const float4 v = held[i];
                y4[k] = make_float4(v.x * inv * g.x, v.y * inv * g.y, v.z * inv * g.z, v.w * inv * g.w);
            }
        }
        for (int k = kRmsHeld * kRmsThreads + tid; k < D4; k += kRmsThreads) {
            const float4 v = h4 ? h4[k] : hval(k);
            const float4 g = w4[k];
            y4[k] = make_float4(v.x * inv * g.x, v.y * inv * g.y, v.z * inv * g.z, v.w * inv * g.w);
        }
    } else {
        const float *xr = x + off, *rr = r ? r + off : nullptr;
        float *hr = h_out ? h_out + off : nullptr;
        for (int k = tid; k < D; k += kRmsThreads) {
            const float v = rr ? xr[k] + rr[k] : xr[k];
            if (hr) hr[k] = v;
            ss += v * v;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if ((tid & 31) == 0) red[tid >> 5] = ss;
        __syncthreads();
        ss = 0.f;
#pragma unroll
        for (int i = 0; i < kRmsThreads / 32; ++i) ss += red[i];
        const float inv = 1.f / sqrtf(ss / (float)D + eps);
        for (int k = tid; k < D; k += kRmsThreads) {
            const float v = hr ? hr[k] : (rr ? xr[k] + rr[k] : xr[k]);
            y[off + k] = v * inv * w[k];
        }
    }
}

int sm_count() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
    }
    return n;
}

}  // namespace

cudaError_t launch_fix_row_tails(const Tensor &t, long long rb, cudaStream_t st) {
    const int used_bits = (int)(((long long)t.I * fmt_bits(t.fmt)) % 8);
    if (used_bits == 0) return cudaSuccess;
    const uint8_t keep = (uint8_t)((1u << used_bits) - 1u);
    fix_row_tails_kernel<<<(t.O + 255) / 256, 256, 0, st>>>(t.codes, t.O, t.ld, rb, keep, zero_byte(t.fmt));
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_qmv_simt(const Tensor &t, const Tensor *tu, const float *x, float *y, float *yu, int S,
                            cudaStream_t st) {
    RowSet a{t.codes, t.scales, y, t.gs, t.G_ld};
    RowSet b = tu ? RowSet{tu->codes, tu->scales, yu, tu->gs, tu->G_ld} : a;
    const int n_sets = tu ? 2 : 1;
    const long long rows = (long long)t.O * n_sets;
    const int tok_blocks = (S + kTok - 1) / kTok;
    long long want = (rows + kWarps - 1) / kWarps;
    const long long cap = (long long)sm_count() * 8;
    const int gx = (int)(want < cap ? want : cap);
    if (tok_blocks > 65535) return cudaErrorInvalidConfiguration;
    dim3 grid(gx, tok_blocks);
    // groups smaller than a chunk (16 or 32 elements) take the split variant
    const int per_chunk = t.fmt == B200Q_F32 ? 4 : t.fmt == B200Q_I8 ? 16 : t.fmt == B200Q_I4 ? 32 : 64;
    const int sub = (t.gs && t.gs < per_chunk) ? t.gs : 0;
    if (sub != 0 && sub != 16 && sub != 32) return cudaErrorInvalidValue;
#define QWQ_SIMT(F, SB) qmv_simt_kernel<F, SB><<<grid, kWarps * 32, 0, st>>>(a, b, n_sets, t.O, t.I, t.ld, x, S)
    switch (t.fmt) {
    case B200Q_F32: QWQ_SIMT(B200Q_F32, 0); break;
    case B200Q_I8: QWQ_SIMT(B200Q_I8, 0); break;
    case B200Q_I4:
        if (sub == 16) QWQ_SIMT(B200Q_I4, 16);
        else QWQ_SIMT(B200Q_I4, 0);
        break;
    case B200Q_I2:
        if (sub == 16) QWQ_SIMT(B200Q_I2, 16);
        else if (sub == 32) QWQ_SIMT(B200Q_I2, 32);
        else QWQ_SIMT(B200Q_I2, 0);
        break;
    default: return cudaErrorInvalidValue;
    }
#undef QWQ_SIMT
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_silu_mul(const float *g, const float *u, float *h, long n, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    long blocks = (n / 4 + 255) / 256;
    const long cap = (long)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    silu_mul_kernel<<<(int)blocks, 256, 0, st>>>(g, u, h, n);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const float *x, const float *r, float *h, const float *w, float *y, int S, int D,
                           float eps, cudaStream_t st) {
    rmsnorm_kernel<<<S, kRmsThreads, 0, st>>>(x, r, h, w, y, D, eps);
    count_launch();
    return cudaGetLastError();
}

}  // namespace qwq
