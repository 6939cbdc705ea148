/*
 * b200q.h -- C ABI of the GB300 quantized-weight matmul library.
 *
 * The library holds quantized weight tensors resident in GPU memory and runs
 *
 *     y[s,o] = scale[o] * sum_i deq(W[o,i]) * x[s,i]
 *
 * against S activation rows, plus the calls built on it: the gate/up pair,
 * grouped expert calls, RMSNorm glue and MLA decode attention with weight
 * absorption over paged caches.  Sources for the operation: the page "CUDA 后端"
 * (colibri-analysis 09), section 1, "设备侧库 backend_cuda.cu" (the resident
 * tensor, `weight_at`, `quant_matmul` and the five extern "C" functions of the
 * backend), and the page "第 8 章 · 02 CUDA/Metal/Vulkan 三后端", section 四
 * (the qmatmul.comp and qmatmul_gate_up.comp shader headers).
 *
 * Formats and their codes (fmt numbering 0/1/2 as on the Vulkan tensor in the
 * three-backends chapter, section 三; int2 = 3 extends it):
 *   B200Q_F32  stored f32 weights, deq = the float
 *   B200Q_I8   one byte per weight, deq = two's-complement value (-128..127)
 *   B200Q_I4   two codes per byte, low nibble first, deq = code - 8
 *   B200Q_I2   four codes per byte, low bits first, deq = code - 2
 * Host layout of codes: row-major [O, rb] bytes with rb = ceil(I*bits/8)
 * (4*I for f32); the unused high bits of a row's last byte are ignored.
 *
 * Numerics.  Every path computes from exact dequantized integers (or the
 * stored floats) and accumulates in f32.  Three paths:
 *   f32 path        (S < b200q_tc_min_s(), every S for f32 and int2 tensors):
 *                   |y - y_exact| <= 1e-5 * |scale[o]| * sum_i |deq * x|;
 *                   int8 / int4 tensors from b200q_tcx_min_s() rows run it on
 *                   the tensor cores (B200Q_PATH_TCX): each row of x is scaled
 *                   by an exact power of two and split exactly into three
 *                   bf16 pieces, so every product is exact and only the f32
 *                   accumulation rounds; int2 tensors with per-row scales
 *                   at 3 to 15 rows run it on the fp8 tensor cores
 *                   (B200Q_PATH_TCS: exact products, x rounded to 26-30
 *                   bits); S = 1 and the other cases run SIMT kernels
 *                   (B200Q_PATH_F32)
 *   tensor-core path (int8 / int4 tensors at S >= b200q_tc_min_s()): x is
 *                   rounded to bf16 (nearest, ties to even) inside the call,
 *                   products and sums are f32 on the tensor cores:
 *                   |y - y_exact| <= 4e-3 * |scale[o]| * sum_i |deq * x|
 * Tensors with group-wise scales (b200q_tensor_upload_grouped) follow the same
 * bounds with the scale taken per group: on the tensor-core path each weight
 * is (code - zero point) * scale rounded to bf16 once; the three-piece path
 * refuses them.
 * NaN and Inf inputs are outside the contract, and so are f32-weight products
 * |w * x| below the f32 normal range (2^-126): f32 arithmetic rounds them on
 * the subnormal grid.  Quantized formats stage each row of x scaled by an
 * exact power of two taken from the row's largest |x|, so the bound also holds
 * for subnormal or very large x.  On the f32 path they accumulate code * x and
 * the zero point's z * x in f32 and subtract, so the rounding error follows
 * sum_i (|code| + z) |x| rather than sum_i |code - z| |x|: the bound holds
 * for rows whose largest |x| is up to ~1e5 times their typical |x| at
 * I = 6144 (less at smaller I); a larger isolated outlier that meets
 * zero-point codes can exceed it.
 *
 * Devices.  A tensor lives on the device that was current when it was
 * uploaded; every call on it must be made with that device current.
 *
 * Errors.  Calls return B200Q_OK (0) or a negative status; the text of the
 * last error of the calling thread is b200q_last_error().  No call falls back
 * to the CPU.  Kernel faults that happen after an asynchronous call returned
 * surface at the caller's next synchronization, as usual in CUDA.
 */
#ifndef B200Q_H
#define B200Q_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct b200q_tensor b200q_tensor;   /* opaque, immutable after upload */

enum { B200Q_F32 = 0, B200Q_I8 = 1, B200Q_I4 = 2, B200Q_I2 = 3 };

enum {
    B200Q_OK = 0,
    B200Q_EINVAL = -1,     /* bad argument: format, shape, pointer, alignment, device */
    B200Q_ENOMEM = -2,     /* device allocation failed */
    B200Q_ECUDA = -3,      /* a CUDA call or kernel launch failed */
    B200Q_ETIMEOUT = -4    /* a bounded device-side wait gave up (kernel returned early) */
};

/* Path selection for b200q_matmul_ex. */
enum { B200Q_PATH_AUTO = 0, B200Q_PATH_F32 = 1, B200Q_PATH_TC = 2, B200Q_PATH_TCX = 3, B200Q_PATH_TCS = 4 };

/*
 * Upload one weight tensor to the current device and keep it resident.
 * Counterpart of coli_cuda_tensor_upload ("CUDA 后端", section 1, public C ABI
 * table: uploads weights and scales once).
 *
 *   fmt     B200Q_F32 / I8 / I4 / I2
 *   O, I    output rows and input columns, both > 0
 *   codes   HOST pointer to the host layout above ([O, rb] bytes; f32: O*I
 *           floats).  Read during the call only; the caller keeps ownership.
 *   scales  HOST pointer to O floats, required for quantized formats; for f32
 *           it may be NULL, meaning 1.0 for every row.
 *
 * Copies synchronously and returns once the tensor is resident.  The library
 * owns the device memory until b200q_tensor_free.  Returns NULL (and sets the
 * last error) on a bad argument or when device memory runs out; with the
 * environment variable B200Q_FAULT_INJECT=alloc it fails with out-of-memory
 * before touching the GPU (for testing callers' error paths).
 */
b200q_tensor *b200q_tensor_upload(int fmt, int O, int I, const void *codes, const float *scales);

/*
 * As b200q_tensor_upload with group-wise scales: one scale per row and group
 * of gs consecutive columns, the group size the Vulkan tensor carries next to
 * fmt (three-backends chapter, section 三; the pages say nothing more, so this
 * is the plain reading):
 *     y[s,o] = sum_g scales[o, g] * sum_{i in group g} deq(W[o,i]) * x[s,i]
 *   gs      group size: a multiple of a 16-byte chunk's element count (4 f32,
 *           16 int8, 32 int4, 64 int2), or 16 or 32 where that divides it;
 *           B200Q_EINVAL otherwise
 *   scales  HOST pointer to [O, ceil(I / gs)] floats, row-major; the last
 *           group of a row may be short
 * Paths (the bound is taken with the group scales):
 *   - the f32 path: the decode kernel below 16 rows, the SIMT kernel beyond;
 *   - int8 / int4, the bf16 tensor-core path (AUTO from b200q_tc_min_s()
 *     rows, and b200q_matmul_tc_noalloc): the dequantizer forms
 *     bf16((code - zero point) * scale) with one rounding per weight, like
 *     the bf16 rounding of x, so that path's 4e-3 bar still holds;
 *   - the three-piece path (B200Q_PATH_TCX) refuses them (B200Q_EINVAL): a
 *     rounded weight would break its f32 accuracy.
 */
b200q_tensor *b200q_tensor_upload_grouped(int fmt, int O, int I, int gs, const void *codes, const float *scales);

/* Group size of a tensor's scales (0: one scale per row), or a negative status. */
int b200q_tensor_group_size(const b200q_tensor *t);

/*
 * Free a tensor (counterpart of coli_cuda_tensor_free).  NULL is a no-op.
 * The caller must make sure no queued kernel still reads the tensor.
 */
void b200q_tensor_free(b200q_tensor *t);

/*
 * y = matmul(t, x) on `stream` (counterpart of coli_cuda_matmul, "CUDA 后端"
 * section 1; the formula is the qmatmul.comp header, three-backends chapter
 * section 四).
 *
 *   x       DEVICE pointer, [S, I] f32 row-major, contiguous, 16-byte aligned
 *   y       DEVICE pointer, [S, O] f32 row-major, 16-byte aligned; fully
 *           overwritten; must not overlap x
 *   S       number of activation rows, >= 0 (0 is a no-op)
 *   stream  a cudaStream_t passed as void*; NULL is the legacy default stream
 *
 * Asynchronous: returns after the kernels are queued.  The caller owns x and y
 * and must keep them alive until the stream reaches this work.  Path: the f32
 * path for S < b200q_tc_min_s() or for f32 / int2 tensors, else the
 * tensor-core path.  Returns B200Q_OK, B200Q_EINVAL or B200Q_ECUDA.
 */
int b200q_matmul(const b200q_tensor *t, const float *x, float *y, int S, void *stream);

/*
 * As b200q_matmul with an explicit path: B200Q_PATH_AUTO (same as
 * b200q_matmul), B200Q_PATH_F32 (the f32-accurate SIMT kernels at any S, any
 * format), B200Q_PATH_TCX (the f32-accurate tensor-core path, x in three bf16
 * pieces, any S >= 1, at most 15 rows per launch), B200Q_PATH_TCS (the
 * f32-accurate tensor-core path with the weights in tensor memory, below) or
 * B200Q_PATH_TC (the bf16 tensor-core path at any S >= 1).  TCX and TC take
 * int8 and int4 tensors only, TCS int8, int4 and int2 tensors with per-row
 * scales (B200Q_EINVAL otherwise).
 *
 * B200Q_PATH_TCS: an exact integer dot product on the fp8 tensor cores.
 * A 4-bit field in the low bits of an E4M3 byte is worth field * 2^-9 for
 * every field value 0..15, so each 128-row tile of codes is masked straight
 * into fp8 bytes in tensor memory (tcgen05.st): int4 and int2 codes as they
 * are, int8 codes (sign bit flipped) as a low and a high nibble.  x is
 * rounded per token to a fixed-point integer n = rint(x 2^T), 2^T a power of
 * two that brings the largest |x| among the columns one CTA handles to
 * [2^(4J-2), 2^(4J-1)), J = 7 or 8, offset to a non-negative value and cut
 * into J 4-bit digits, which are fp8 bytes the same way.  tcgen05.mma
 * (kind::f8f6f4, A in tensor memory) then sums products of small integers,
 * exactly in its f32 accumulator; the digits are recombined in 64-bit
 * integers (with one extra row of ones for the offset, and the zero point
 * taken out), and each output is rounded once.  The only error is the
 * rounding of x to 26 (S even) or 30 (S odd) bits below its token's largest
 * magnitude in the CTA's columns: for every output, |y - y_exact| <=
 * |scale| * 2^-27 * max|x| * sum|deq| at J = 7.  At most 8 tokens per launch
 * (more are chunked); the work is split evenly over the SMs in (row tile,
 * 128-byte k-block) items.  A tile shared by several CTAs is added up in a
 * fixed order by the CTA that brings its arrival count to its number of
 * parts; no CTA waits on another.  Each call with shared tiles takes a
 * workspace from the library's pool.  AUTO takes this path for int2 tensors
 * with per-row scales at 3 to 15 rows.
 */
int b200q_matmul_ex(const b200q_tensor *t, const float *x, float *y, int S, int path,
                    void *stream);

/*
 * The path b200q_matmul takes for this tensor at this S: B200Q_PATH_F32,
 * B200Q_PATH_TCX or B200Q_PATH_TC, or a negative status for a bad argument.
 */
int b200q_matmul_path(const b200q_tensor *t, int S);

/*
 * Threshold S from which int8 / int4 tensors take the tensor-core path:
 * 16 by default (the colibri CUDA docs, "The GPU-resident pipeline" section:
 * the Tensor-Core W4A16 dispatch pays from 16 rows up), or the value of the
 * environment variable B200Q_TC_MIN_S (>= 1) read at the first call.
 */
int b200q_tc_min_s(void);

/*
 * Threshold S from which int8 / int4 tensors below b200q_tc_min_s() take the
 * f32-accurate tensor-core path (B200Q_PATH_TCX) instead of the SIMT decode
 * kernels; the environment variable B200Q_TCX_MIN_S (>= 1) overrides the
 * default, read at the first call.  A value >= b200q_tc_min_s() disables it.
 */
int b200q_tcx_min_s(void);

/*
 * Fused gate/up pair: yg = matmul(tg, x) and yu = matmul(tu, x) in one pass
 * that reads x once (qmatmul_gate_up.comp, three-backends chapter, section 四
 * list of shaders).  tg and tu must have the same fmt, O, I and device.  The
 * pointer rules of b200q_matmul hold for x, yg, yu; yg and yu must not
 * overlap each other or x.  Same numerics and path rule as b200q_matmul.
 */
int b200q_matmul_gate_up(const b200q_tensor *tg, const b200q_tensor *tu, const float *x,
                         float *yg, float *yu, int S, void *stream);

/* Most tensors one grouped call takes. */
enum { B200Q_GROUP_MAX = 16 };

/*
 * Grouped matmul: ys[j] = matmul(ts[j], xs[j]) for j < n, in one kernel
 * launch per pair of activation rows on the f32 path.  This is the decode step
 * of a mixture-of-experts layer: the gate and up tensors of k routed experts
 * (2k tensors on one x, the pairing of qmatmul_gate_up.comp in the
 * three-backends chapter, section 四, widened to several experts) or their k
 * down tensors (one input each).  The pages run one expert at a time ("The
 * GPU-resident pipeline" section of the colibri CUDA docs keeps the expert
 * loop and groups expert uploads at prefill); launching the experts of a
 * layer together is this library's own step.
 *
 *   ts      HOST array of n tensor handles, 1 <= n <= B200Q_GROUP_MAX; all of
 *           one format and one I, on the current device; O may differ
 *   xs      HOST array of n DEVICE pointers, xs[j] = [S, I] f32 as in
 *           b200q_matmul; entries may repeat (consecutive sets with the same
 *           x stage it once per block)
 *   ys      HOST array of n DEVICE pointers, ys[j] = [S, O_j] f32, fully
 *           overwritten; no ys[j] may overlap another ys[k] or any xs[k]
 *   S       activation rows, >= 0 (0 is a no-op)
 *
 * The host arrays are read during the call only.  Same numerics and path rule
 * as b200q_matmul: below b200q_tc_min_s() (or for f32 / int2 tensors) the
 * whole group is one launch per two rows; from the threshold on, int8 / int4
 * tensors run one tensor-core call each.  If the group's inputs do not fit
 * the kernel's shared memory the tensors run one call each.  Returns
 * B200Q_OK, B200Q_EINVAL or B200Q_ECUDA.
 */
int b200q_matmul_grouped(const b200q_tensor *const *ts, int n, const float *const *xs,
                         float *const *ys, int S, void *stream);

/*
 * As b200q_matmul_grouped with the expert glue fused into the input:
 * ys[j] = matmul(ts[j], silu(gs[j]) * us[j]), silu(z) = z / (1 + e^-z), the
 * product taken elementwise over [S, I] (the down projection of k experts on
 * their own gate and up outputs).  gs[j] and us[j] follow the rules of xs[j];
 * the gated input is formed while it is staged and never written to memory
 * on the f32 path.  From b200q_tc_min_s() rows on it is formed in a
 * stream-ordered workspace of the library's pool and the tensors run one
 * tensor-core call each.  The f32 path's bound is taken on the f32 value of
 * silu(g) * u, which lies within a few ulp of the exact one.
 */
int b200q_matmul_grouped_silu(const b200q_tensor *const *ts, int n, const float *const *gs,
                              const float *const *us, float *const *ys, int S, void *stream);

/*
 * Expert glue: h[k] = silu(g[k]) * u[k], silu(z) = z / (1 + e^-z), for
 * k < n, f32, on `stream`.  g, u, h are DEVICE pointers to n floats, 16-byte
 * aligned; h may equal g or u (in place) but must not partially overlap them.
 * The activation itself is not printed on the pages; this is the textbook
 * SiLU of a gated MoE expert.
 */
int b200q_silu_mul(const float *g, const float *u, float *h, long n, void *stream);

/*
 * Layer glue kept on the device ("The GPU-resident pipeline" section of the
 * colibri CUDA docs: norms and residual adds run on the GPU while the expert
 * loop runs).  The norm is not printed on the pages; this is the textbook
 * RMSNorm with an optional residual, per row s of S rows of D floats:
 *     h = x + r (r NULL: h = x),  y = h * w / sqrt(mean_d h^2 + eps)
 *   x, r, y   DEVICE pointers, [S, D] f32, 16-byte aligned
 *   h         DEVICE pointer [S, D] receiving h, or NULL; it may be x or r
 *             itself (the residual stream updated in place) but must not
 *             partially overlap them
 *   w         DEVICE pointer, D floats
 *   eps       >= 0 and finite
 * y must not overlap x, r, h or w.  f32 arithmetic (sum of squares, correctly
 * rounded square root and division): |y - y_exact| <= 1e-5 * |y_exact| on
 * rows whose h is not all zero.  S = 0 is a no-op.  One kernel launch.
 */
int b200q_rmsnorm(const float *x, const float *r, float *h, const float *w, float *y, int S, int D, float eps,
                  void *stream);

/*
 * Host-buffer call in the style of the reference backend ("CUDA 后端",
 * section 1: each matmul copies its input to the GPU, runs the kernel and
 * copies the result back, blocking): copies x_host ([S, I] f32) to a
 * library-owned device staging buffer on `stream`, runs b200q_matmul, copies
 * y back to y_host ([S, O] f32) and synchronizes `stream` before returning.
 * Pinned host memory gives the fastest copies; pageable memory works.  The
 * staging buffer belongs to the device and grows as needed (it is allocated
 * with cudaMalloc); calls on one device from several threads are serialized.
 */
int b200q_matmul_host(const b200q_tensor *t, const float *x_host, float *y_host, int S,
                      void *stream);

/*
 * Tensor-core matmul that allocates nothing.  The pages have no counterpart
 * of this call; it exists for callers that cannot allocate device memory
 * while they run: their device memory is owned by another allocator (a
 * framework's caching allocator or a pool that reserved the device), or they
 * are latency-critical loops that must not wait on an allocator call, which
 * may synchronize the device or fail.
 *
 * Same operation, arguments, numerics and tensor-core path as
 * b200q_matmul_ex(t, x, y, S, B200Q_PATH_TC, stream) for int8 and int4
 * tensors, but the bf16 copy of x is kept in a fixed device array of
 * b200q_tc_noalloc_capacity() bytes (24 MiB) that the library defines at file
 * scope: every GPU that loads the library holds it until the process exits.
 * A call needs S * padded_I * 2 bytes of it (padded_I = I rounded up to the
 * device row length, a multiple of 256 for int4 and 128 for int8) and returns
 * B200Q_EINVAL with a clear message when that exceeds the capacity.  It calls
 * no cudaMalloc, cudaFree or allocating library routine.
 *
 * All calls on a device share the array, which keeps the last call's
 * contents; calls whose work overlaps in time on the GPU (for instance on two
 * streams without ordering between them) race on it and must be serialized by
 * the caller.  Every call looks up the array's device address in the
 * current device's context (cudaGetSymbolAddress, a host-side query), so a
 * context that was reset and recreated gets its own address; the first
 * lookup on a device may load the library's device code into that context,
 * so make the first call on each device before any stream capture.
 */
int b200q_matmul_tc_noalloc(const b200q_tensor *t, const float *x, float *y, int S, void *stream);

/* Bytes of the fixed workspace behind b200q_matmul_tc_noalloc. */
long long b200q_tc_noalloc_capacity(void);

/*
 * Describe a tensor.  Any out pointer may be NULL.  device_bytes is the size of
 * the resident copy (codes with row padding plus scales).
 */
int b200q_tensor_info(const b200q_tensor *t, int *fmt, int *O, int *I, int *device,
                      long long *device_bytes);

/*
 * Synchronizes the current device and reports whether any kernel of the
 * library gave up on a bounded device-side wait since the last call
 * (B200Q_ETIMEOUT; such a kernel leaves its outputs incomplete), met a NULL or
 * unaligned KV-cache page (B200Q_EINVAL, b200q_mla_absorb and
 * b200q_kv_append; the call's outputs are then undefined), or a CUDA error
 * (B200Q_ECUDA).  Clears the record.  B200Q_OK otherwise.
 */
int b200q_device_status(void);

/*
 * Number of kernels this process has launched through the library so far (all
 * devices, all threads).  Lets a caller count the launches inside a timed
 * region.
 */
long long b200q_kernel_launches(void);

/*
 * Number of device workspace allocations the library has made on its
 * callers' behalf so far (all devices, all threads): the creation of a
 * device's stream-ordered memory pool, every allocation from it (the
 * tensor-core paths' converted copy of x, split-K partials, MLA and grouped
 * call scratch) and the host-buffer call's staging buffer.  Tensor uploads
 * (the tensors' own memory) are not counted.  A call that must not allocate,
 * such as b200q_matmul_tc_noalloc, leaves it unchanged.
 */
long long b200q_workspace_allocations(void);

/*
 * ---- MLA decode attention with weight absorption ----
 *
 * Source: the three-backends chapter ("第 8 章 · 02 CUDA/Metal/Vulkan 三后端"),
 * section 四, the header of attention_absorb.comp (the Vulkan form of
 * coli_cuda_attention_absorb); the KV pages of section 一 (COLI_KV_PAGE_TOKENS:
 * the latent and rope caches are allocated 64 positions to a page and rows are
 * appended at their absolute position).  For each new token s < S and head
 * h < H:
 *     qabs[i]    = sum_d q_nope[s,h,d] * Wk[h,d,i]               d < Dn, i < K
 *     score_t    = (qabs . L[t] + q_rope[s,h] . Rr[t]) * scale   t in [st0, T-S+s]
 *     p          = softmax(score)
 *     clat[i]    = sum_t p_t * L[t,i]
 *     ctx[s,h,v] = sum_i clat[i] * Wv[h,v,i]                     v < Dv
 * Wk and Wv are rows of one tensor wkv_b of H * (Dn + Dv) rows and K columns
 * (any format): head h's key rows are h * (Dn + Dv) + d, its value rows
 * h * (Dn + Dv) + Dn + v; each weight is scale * (code - zero point), the
 * scale of its row or of its row and group of gs columns.  The S new tokens occupy positions T-S .. T-1 of the caches (append
 * them first); token s sees positions st0 .. T-S+s.
 */
enum { B200Q_KV_PAGE_TOKENS = 64 };

/*
 *   wkv_b       tensor handle, O = H * (Dn + Dv), I = K; per-row or group-wise
 *               scales; K a multiple of 4, at most 768
 *   q_nope      device [S, H, Dn] f32, 16-byte aligned
 *   q_rope      device [S, H, R] f32, 16-byte aligned (unused when R = 0)
 *   lat_pages   DEVICE array of ceil(T / 64) device pointers; page p holds
 *               positions 64p .. 64p+63 as [64, K] f32 rows.  Every page must
 *               be a full 64-row allocation, 16-byte aligned, non-NULL
 *   rope_pages  the same for the rope cache, [64, R] f32 pages (unused when R = 0)
 *   R           rope width, a multiple of 4 (K + R at most 716)
 *   T           positions in the caches, S <= T <= 2^30 (and H * S <= 2^20,
 *               S <= 262140)
 *   st0         first position any token sees, 0 <= st0 <= T - S; pages
 *               wholly before st0 are never read
 *   scale       softmax scale, finite
 *   ctx         device [S, H, Dv] f32 output, 16-byte aligned, not
 *               overlapping q_nope or q_rope
 * Asynchronous on `stream`; four kernel launches; a stream-ordered workspace
 * of about 4 * H * S * K * (1 + splits) bytes, splits <= 512 (the cache is
 * split so that the attention kernel fills the GPU).  S = 0 is a no-op.
 * Numerics: f32 arithmetic throughout (absorb, scores, expf softmax, latent
 * context, value rows); within 1e-5 of the bound
 *     (1 + max_t |scale| (sum_i QA_i |L[t,i]| + sum_j |q_rope_j Rr[t,j]|))
 *       * sum_i |Wv[h,v,i]| * sum_t p_t |L[t,i]|,   QA_i = sum_d |q_nope_d Wk[h,d,i]|
 * of the exact result.  A NULL or unaligned page is reported by
 * b200q_device_status.
 */
int b200q_mla_absorb(const b200q_tensor *wkv_b, int H, int Dn, int Dv, const float *q_nope, const float *q_rope,
                     const float *const *lat_pages, const float *const *rope_pages, int R, int T, int st0,
                     float scale, float *ctx, int S, void *stream);

/*
 * Appends n rows to the paged caches at absolute positions pos .. pos+n-1
 * (device copies; one launch): lat_rows device [n, K] f32 into lat_pages,
 * rope_rows device [n, R] f32 into rope_pages (device page-pointer arrays as in
 * b200q_mla_absorb).  n = 0 is a no-op.  Asynchronous on `stream`.
 */
int b200q_kv_append(float *const *lat_pages, float *const *rope_pages, int K, int R, int pos, const float *lat_rows,
                    const float *rope_rows, int n, void *stream);

/*
 * Self test of the bounded waits: one kernel waits, at most wait_us
 * microseconds (1 .. 10^6), on an mbarrier that nothing arrives on, gives up
 * and records B200Q_ETIMEOUT the way a kernel whose copies never land does.
 * The next b200q_device_status reports it (and clears it); the context stays
 * usable.  Asynchronous on `stream`; one launch.
 */
int b200q_selftest_timeout(int wait_us, void *stream);

/* Text of the calling thread's last error ("" if none). */
const char *b200q_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* B200Q_H */
