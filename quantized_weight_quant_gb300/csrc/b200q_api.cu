// Host side of the b200q C ABI: argument checks, tensor upload / free, path
// selection, the host-staged call and error reporting.  Every computation is
// done by the kernels; nothing here runs on the CPU besides bookkeeping.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "qwq_internal.h"

namespace qwq {

// Kernels of the other translation units.
cudaError_t launch_decode(const Tensor &t, const Tensor *tu, const float *x, float *y, float *yu, int S,
                          cudaStream_t st, bool *handled);
cudaError_t launch_tcx(const Tensor &t, const Tensor *tu, const float *x, float *y, float *yu, int S,
                       cudaStream_t st, bool *handled);
cudaError_t launch_prefill_tc(const Tensor &t, const Tensor *tu, const float *x, float *y, float *yu,
                              int S, cudaStream_t st, bool *handled);
cudaError_t decode_take_error(unsigned int *code);
cudaError_t launch_tcs(const Tensor &t, const float *x, float *y, int S, cudaStream_t st, bool *handled);
cudaError_t tcs_take_error(unsigned int *code);
size_t noalloc_capacity();
cudaError_t launch_prefill_tc_noalloc(const Tensor &t, const float *x, float *y, int S, cudaStream_t st);
cudaError_t prefill_take_error(unsigned int *code);
cudaError_t launch_decode_group(const Tensor *const *ts, int n, const float *const *xa, const float *const *xb,
                                float *const *ys, bool silu, int S, cudaStream_t st, bool *handled);
cudaError_t workspace_alloc(void **ptr, size_t bytes, cudaStream_t st);
cudaError_t workspace_free(void *ptr, cudaStream_t st);
size_t mla_smem_bytes(int K, int R);
int mla_max_latent();
size_t mla_workspace_floats(int H, int S, int K, int T, int st0);
cudaError_t launch_mla_absorb(const Tensor &w, int H, int Dn, int Dv, const float *q_nope, const float *q_rope,
                              const float *const *lat_pages, const float *const *rope_pages, int R, int T, int st0,
                              float scale, float *ctx, int S, float *ws, cudaStream_t st);
cudaError_t launch_kv_append(float *const *lat_pages, float *const *rope_pages, int K, int R, int pos,
                             const float *lat_rows, const float *rope_rows, int n, cudaStream_t st);
cudaError_t mla_take_error(unsigned int *code);
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t st);

namespace {

thread_local std::string g_err;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(e == cudaErrorMemoryAllocation ? B200Q_ENOMEM : B200Q_ECUDA, "%s: %s (%s)", what,
                cudaGetErrorString(e), cudaGetErrorName(e));
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    const char *pa = (const char *)a, *pb = (const char *)b;
    return pa < pb + nb && pb < pa + na;
}

long long host_row_bytes(int fmt, long long I) { return (I * fmt_bits(fmt) + 7) / 8; }

int check_tensor(const b200q_tensor *h, const char *who) {
    if (!h) return fail(B200Q_EINVAL, "%s: tensor is NULL", who);
    const Tensor *t = reinterpret_cast<const Tensor *>(h);
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, who);
    if (dev != t->device)
        return fail(B200Q_EINVAL, "%s: tensor lives on device %d but device %d is current", who, t->device,
                    dev);
    return B200Q_OK;
}

int check_io(const Tensor &t, const float *x, const float *y, int S, const char *who) {
    if (!x || !y) return fail(B200Q_EINVAL, "%s: x and y must be device pointers, got NULL", who);
    if (!aligned16(x) || !aligned16(y)) return fail(B200Q_EINVAL, "%s: x and y must be 16-byte aligned", who);
    if (overlap(x, (size_t)S * t.I * 4, y, (size_t)S * t.O * 4))
        return fail(B200Q_EINVAL, "%s: x and y overlap", who);
    return B200Q_OK;
}

std::atomic<long long> g_launches{0};

int g_tc_min_s = 0, g_tcx_min_s = 0;
std::once_flag g_tc_once;

struct Staging {
    std::mutex m;
    void *buf = nullptr;
    size_t cap = 0;
};
Staging g_staging[64];

}  // namespace

void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

namespace {
std::atomic<long long> g_ws_allocs{0};
std::atomic<int> g_sm_count[64];
struct SmemAttr {
    const void *fn;
    int dev, bytes;
};
std::mutex g_attr_mu;
std::vector<SmemAttr> g_attr_done;
}  // namespace

void count_workspace_alloc() { g_ws_allocs.fetch_add(1, std::memory_order_relaxed); }

int sm_count(int dev) {
    if (dev < 0 || dev >= 64) return 1;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t allow_dynamic_smem(const void *fn, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    for (const SmemAttr &a : g_attr_done)
        if (a.fn == fn && a.dev == dev && a.bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) g_attr_done.push_back(SmemAttr{fn, dev, bytes});
    return e;
}

void read_thresholds() {
    std::call_once(g_tc_once, [] {
        auto env_int = [](const char *name, int dflt) {
            if (const char *s = std::getenv(name)) {
                int p = std::atoi(s);
                if (p >= 1) return p;
            }
            return dflt;
        };
        g_tc_min_s = env_int("B200Q_TC_MIN_S", 16);
        g_tcx_min_s = env_int("B200Q_TCX_MIN_S", kTcxMinS);
    });
}

int tc_min_s() {
    read_thresholds();
    return g_tc_min_s;
}

int tcx_min_s() {
    read_thresholds();
    return g_tcx_min_s;
}

// AUTO: int8 / int4 take the bf16 tensor-core path from tc_min_s() rows, the
// f32-accurate tensor-core path (x in three bf16 pieces; per-row scales only)
// from tcx_min_s() rows, the SIMT f32 path below.  int2 with per-row scales
// takes the exact fp8 tensor-core path from 3 to 15 rows (where the SIMT
// kernel needs two or more passes over the weights: 8192^2 at 3 / 4 / 8
// rows, 29.0 / 32.5 / 64.4 us against 23.5 / 24.1 / 42.8 us), the SIMT path
// otherwise; f32 tensors always the SIMT path.
int select_path(const Tensor &t, int S, int path) {
    if (path != B200Q_PATH_AUTO) return path;
    if (t.fmt == B200Q_I2) return !t.gs && S >= 3 && S < 16 ? B200Q_PATH_TCS : B200Q_PATH_F32;
    if (t.fmt != B200Q_I4 && t.fmt != B200Q_I8) return B200Q_PATH_F32;
    if (S >= tc_min_s()) return B200Q_PATH_TC;
    if (!t.gs && S >= tcx_min_s()) return B200Q_PATH_TCX;
    return B200Q_PATH_F32;
}

int run_matmul(const Tensor &t, const Tensor *tu, const float *x, float *y, float *yu, int S, int path,
               cudaStream_t st, const char *who) {
    if (S == 0) return B200Q_OK;
    path = select_path(t, S, path);
    cudaError_t e = cudaSuccess;
    bool handled = false;
    if (path == B200Q_PATH_TCS) {
        if (t.fmt != B200Q_I4 && t.fmt != B200Q_I8 && t.fmt != B200Q_I2)
            return fail(B200Q_EINVAL, "%s: the f32-accurate tensor-core path takes int8, int4 and int2 tensors only",
                        who);
        if (t.gs || (tu && tu->gs))
            return fail(B200Q_EINVAL, "%s: the f32-accurate tensor-core path takes per-row scales only", who);
        // 16 rows per call here (launch_tcs splits them further); the pair's second tensor runs after the first
        for (int k = 0; k < (tu ? 2 : 1) && e == cudaSuccess; ++k) {
            const Tensor &tt = k ? *tu : t;
            float *yy = k ? yu : y;
            for (int s0 = 0; s0 < S && e == cudaSuccess; s0 += 16) {
                const int ns = S - s0 < 16 ? S - s0 : 16;
                e = launch_tcs(tt, x + (long long)s0 * tt.I, yy + (long long)s0 * tt.O, ns, st, &handled);
                if (e == cudaSuccess && !handled)
                    return fail(B200Q_ECUDA, "%s: no f32-accurate tensor-core kernel for this shape", who);
            }
        }
    } else if (path == B200Q_PATH_TC || path == B200Q_PATH_TCX) {
        if (t.fmt != B200Q_I4 && t.fmt != B200Q_I8)
            return fail(B200Q_EINVAL, "%s: the tensor-core paths take int8 and int4 tensors only", who);
        if (path == B200Q_PATH_TCX && (t.gs || (tu && tu->gs)))
            return fail(B200Q_EINVAL,
                        "%s: tensors with group-wise scales take the f32 and the bf16 tensor-core paths only", who);
        e = path == B200Q_PATH_TC ? launch_prefill_tc(t, tu, x, y, yu, S, st, &handled)
                                  : launch_tcx(t, tu, x, y, yu, S, st, &handled);
        if (e == cudaSuccess && !handled)
            return fail(B200Q_ECUDA, "%s: no tensor-core kernel for this shape", who);
    } else {
        e = launch_decode(t, tu, x, y, yu, S, st, &handled);
        if (e == cudaSuccess && !handled) e = launch_qmv_simt(t, tu, x, y, yu, S, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, who);
    return B200Q_OK;
}

}  // namespace qwq

using namespace qwq;

extern "C" {

const char *b200q_last_error(void) { return g_err.c_str(); }

long long b200q_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

long long b200q_workspace_allocations(void) { return g_ws_allocs.load(std::memory_order_relaxed); }

int b200q_device_status(void) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "b200q_device_status");
    unsigned int a = 0, b = 0, m = 0, c = 0;
    e = decode_take_error(&a);
    if (e == cudaSuccess) e = prefill_take_error(&b);
    if (e == cudaSuccess) e = mla_take_error(&m);
    if (e == cudaSuccess) e = tcs_take_error(&c);
    if (e != cudaSuccess) return cuda_fail(e, "b200q_device_status");
    if (a || b || c || m == (unsigned)(-B200Q_ETIMEOUT))
        return fail(B200Q_ETIMEOUT, "b200q_device_status: a kernel gave up on a bounded wait");
    if (m) return fail(B200Q_EINVAL, "b200q_device_status: an MLA call met a NULL or unaligned cache page");
    return B200Q_OK;
}

int b200q_tc_min_s(void) { return tc_min_s(); }

int b200q_tcx_min_s(void) { return tcx_min_s(); }

}  // extern "C"

namespace {

// One upload for both scale layouts: gs = 0, one scale per row; gs >= 1, one
// per row and group of gs columns ([O, ceil(I / gs)] host floats).
b200q_tensor *upload_impl(int fmt, int O, int I, int gs, const void *codes, const float *scales, const char *who) {
    g_err.clear();
    if (fmt_bits(fmt) == 0) {
        fail(B200Q_EINVAL, "%s: unknown format %d", who, fmt);
        return nullptr;
    }
    if (O <= 0 || I <= 0) {
        fail(B200Q_EINVAL, "%s: O and I must be > 0 (got O=%d, I=%d)", who, O, I);
        return nullptr;
    }
    if (!codes) {
        fail(B200Q_EINVAL, "%s: codes is NULL", who);
        return nullptr;
    }
    if (!scales && (fmt != B200Q_F32 || gs)) {
        fail(B200Q_EINVAL, "%s: scales are required for quantized formats and group-wise scales", who);
        return nullptr;
    }
    if (gs && !group_size_ok(fmt, gs)) {
        fail(B200Q_EINVAL,
             "%s: group size %d not supported for this format (a multiple of %d elements, or 16 / 32 dividing it)",
             who, gs, fmt == B200Q_F32 ? 4 : fmt == B200Q_I8 ? 16 : fmt == B200Q_I4 ? 32 : 64);
        return nullptr;
    }
    if (const char *fi = std::getenv("B200Q_FAULT_INJECT")) {
        if (std::strcmp(fi, "alloc") == 0) {
            fail(B200Q_ENOMEM, "%s: out of device memory (injected by B200Q_FAULT_INJECT)", who);
            return nullptr;
        }
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cuda_fail(e, who);
        return nullptr;
    }
    Tensor *t = new (std::nothrow) Tensor();
    if (!t) {
        fail(B200Q_ENOMEM, "%s: out of host memory", who);
        return nullptr;
    }
    const long long rb = host_row_bytes(fmt, I);
    t->fmt = fmt;
    t->O = O;
    t->I = I;
    t->device = dev;
    t->o_pad = (O + kRowTile - 1) / kRowTile * kRowTile;
    t->ld = (rb + kRowAlign - 1) / kRowAlign * kRowAlign;
    t->k_pad = t->ld * 8 / fmt_bits(fmt);
    t->gs = gs;
    t->G = gs ? (I + gs - 1) / gs : 1;
    t->G_ld = 1;
    t->sc_box = 0;
    if (gs) {
        // a decode stage holds 32 chunks of a row (32 * per-chunk elements);
        // its group scales are copied from the first group rounded down to a
        // multiple of 4 (16 bytes), so take the widest such span over stages
        const long long seg_elems = 32LL * (128 / fmt_bits(fmt));
        const long long nseg = (t->ld + 511) / 512;
        long long span = 1;
        for (long long sg = 0; sg < nseg; ++sg) {
            const long long lo = (sg * seg_elems / gs) & ~3LL;
            const long long end = (sg + 1) * seg_elems < t->k_pad ? (sg + 1) * seg_elems : t->k_pad;
            const long long hi = (end - 1) / gs;
            if (hi - lo + 1 > span) span = hi - lo + 1;
        }
        t->sc_box = (int)((span + 3) & ~3LL);
        t->G_ld = (t->G + 3) & ~3;
        if (t->G_ld < t->sc_box) t->G_ld = t->sc_box;
    }
    const size_t code_bytes = (size_t)t->o_pad * t->ld;
    const size_t scale_bytes = (size_t)t->o_pad * t->G_ld * sizeof(float);
    t->bytes = code_bytes + scale_bytes;
    void *mem = nullptr;
    e = cudaMalloc(&mem, t->bytes);
    if (e != cudaSuccess) {
        cuda_fail(e, who);
        cudaGetLastError();
        delete t;
        return nullptr;
    }
    t->codes = (uint8_t *)mem;
    t->scales = (float *)((uint8_t *)mem + code_bytes);

    cudaStream_t st = nullptr;
    e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaMemsetAsync(t->codes, zero_byte(fmt), code_bytes, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(t->scales, 0, scale_bytes, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(t->codes, (size_t)t->ld, codes, (size_t)rb, (size_t)rb, (size_t)O,
                              cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = launch_fix_row_tails(*t, rb, st);
    if (e == cudaSuccess) {
        if (scales) {
            e = cudaMemcpy2DAsync(t->scales, (size_t)t->G_ld * sizeof(float), scales, (size_t)t->G * sizeof(float),
                                  (size_t)t->G * sizeof(float), (size_t)O, cudaMemcpyHostToDevice, st);
        } else {
            // f32 without scales: 1.0 for every real row (0x3f800000 as four bytes is not a
            // memset pattern, so copy from a host vector)
            float *ones = (float *)std::malloc((size_t)O * sizeof(float));
            if (!ones) {
                e = cudaErrorMemoryAllocation;
            } else {
                for (int i = 0; i < O; ++i) ones[i] = 1.0f;
                e = cudaMemcpyAsync(t->scales, ones, (size_t)O * sizeof(float), cudaMemcpyHostToDevice, st);
                if (e == cudaSuccess) e = cudaStreamSynchronize(st);
                std::free(ones);
            }
        }
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (st) cudaStreamDestroy(st);
    if (e == cudaSuccess &&
        !tmap_encode_2d(&t->dec_map, CU_TENSOR_MAP_DATA_TYPE_UINT32, t->codes, (uint64_t)(t->ld / 4),
                        (uint64_t)t->o_pad, (uint64_t)t->ld, (uint32_t)(t->ld < 512 ? t->ld / 4 : 128), 8,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
        e = cudaErrorNotSupported;
    if (e == cudaSuccess && gs &&
        !tmap_encode_2d(&t->sc_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, t->scales, (uint64_t)t->G_ld,
                        (uint64_t)t->o_pad, (uint64_t)t->G_ld * sizeof(float), (uint32_t)t->sc_box, 8,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
        e = cudaErrorNotSupported;
    if (e == cudaSuccess && !gemm_maps_encode(*t)) e = cudaErrorNotSupported;
    if (e == cudaSuccess && !tcs_map_encode(*t)) e = cudaErrorNotSupported;
    if (e != cudaSuccess) {
        cuda_fail(e, who);
        cudaGetLastError();
        cudaFree(mem);
        delete t;
        return nullptr;
    }
    return reinterpret_cast<b200q_tensor *>(t);
}

}  // namespace

extern "C" {

b200q_tensor *b200q_tensor_upload(int fmt, int O, int I, const void *codes, const float *scales) {
    return upload_impl(fmt, O, I, 0, codes, scales, "b200q_tensor_upload");
}

b200q_tensor *b200q_tensor_upload_grouped(int fmt, int O, int I, int gs, const void *codes, const float *scales) {
    if (gs < 1) {
        g_err.clear();
        fail(B200Q_EINVAL, "b200q_tensor_upload_grouped: group size must be >= 1 (got %d)", gs);
        return nullptr;
    }
    return upload_impl(fmt, O, I, gs, codes, scales, "b200q_tensor_upload_grouped");
}

int b200q_tensor_group_size(const b200q_tensor *h) {
    if (!h) return fail(B200Q_EINVAL, "b200q_tensor_group_size: tensor is NULL");
    return reinterpret_cast<const Tensor *>(h)->gs;
}

void b200q_tensor_free(b200q_tensor *h) {
    if (!h) return;
    Tensor *t = reinterpret_cast<Tensor *>(h);
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != t->device) cudaSetDevice(t->device);
    cudaFree(t->codes);
    if (cur != t->device && cur >= 0) cudaSetDevice(cur);
    delete t;
}

int b200q_tensor_info(const b200q_tensor *h, int *fmt, int *O, int *I, int *device, long long *device_bytes) {
    if (!h) return fail(B200Q_EINVAL, "b200q_tensor_info: tensor is NULL");
    const Tensor *t = reinterpret_cast<const Tensor *>(h);
    if (fmt) *fmt = t->fmt;
    if (O) *O = t->O;
    if (I) *I = t->I;
    if (device) *device = t->device;
    if (device_bytes) *device_bytes = (long long)t->bytes;
    return B200Q_OK;
}

int b200q_matmul_path(const b200q_tensor *h, int S) {
    if (!h) return fail(B200Q_EINVAL, "b200q_matmul_path: tensor is NULL");
    if (S < 0) return fail(B200Q_EINVAL, "b200q_matmul_path: S must be >= 0");
    return select_path(*reinterpret_cast<const Tensor *>(h), S, B200Q_PATH_AUTO);
}

int b200q_matmul_ex(const b200q_tensor *h, const float *x, float *y, int S, int path, void *stream) {
    int rc = check_tensor(h, "b200q_matmul");
    if (rc) return rc;
    const Tensor &t = *reinterpret_cast<const Tensor *>(h);
    if (S < 0) return fail(B200Q_EINVAL, "b200q_matmul: S must be >= 0 (got %d)", S);
    if (path != B200Q_PATH_AUTO && path != B200Q_PATH_F32 && path != B200Q_PATH_TC && path != B200Q_PATH_TCX &&
        path != B200Q_PATH_TCS)
        return fail(B200Q_EINVAL, "b200q_matmul: unknown path %d", path);
    if (S == 0) return B200Q_OK;
    rc = check_io(t, x, y, S, "b200q_matmul");
    if (rc) return rc;
    return run_matmul(t, nullptr, x, y, nullptr, S, path, (cudaStream_t)stream, "b200q_matmul");
}

int b200q_matmul(const b200q_tensor *t, const float *x, float *y, int S, void *stream) {
    return b200q_matmul_ex(t, x, y, S, B200Q_PATH_AUTO, stream);
}

int b200q_matmul_gate_up(const b200q_tensor *hg, const b200q_tensor *hu, const float *x, float *yg, float *yu,
                         int S, void *stream) {
    int rc = check_tensor(hg, "b200q_matmul_gate_up");
    if (rc) return rc;
    rc = check_tensor(hu, "b200q_matmul_gate_up");
    if (rc) return rc;
    const Tensor &tg = *reinterpret_cast<const Tensor *>(hg);
    const Tensor &tu = *reinterpret_cast<const Tensor *>(hu);
    if (tg.fmt != tu.fmt || tg.O != tu.O || tg.I != tu.I || tg.gs != tu.gs)
        return fail(B200Q_EINVAL, "b200q_matmul_gate_up: gate and up differ in format, shape or group size");
    if (S < 0) return fail(B200Q_EINVAL, "b200q_matmul_gate_up: S must be >= 0 (got %d)", S);
    if (S == 0) return B200Q_OK;
    rc = check_io(tg, x, yg, S, "b200q_matmul_gate_up");
    if (rc) return rc;
    rc = check_io(tu, x, yu, S, "b200q_matmul_gate_up");
    if (rc) return rc;
    if (overlap(yg, (size_t)S * tg.O * 4, yu, (size_t)S * tu.O * 4))
        return fail(B200Q_EINVAL, "b200q_matmul_gate_up: yg and yu overlap");
    return run_matmul(tg, &tu, x, yg, yu, S, B200Q_PATH_AUTO, (cudaStream_t)stream, "b200q_matmul_gate_up");
}

}  // extern "C"

namespace {

// Checks of a grouped call; on success ts[] holds the tensors.
int check_group(const b200q_tensor *const *hs, int n, const float *const *xa, const float *const *xb,
                float *const *ys, int S, const Tensor **ts, const char *who) {
    if (n < 1 || n > B200Q_GROUP_MAX)
        return fail(B200Q_EINVAL, "%s: n must be in [1, %d] (got %d)", who, B200Q_GROUP_MAX, n);
    if (!hs || !xa || !ys) return fail(B200Q_EINVAL, "%s: NULL host array", who);
    if (S < 0) return fail(B200Q_EINVAL, "%s: S must be >= 0 (got %d)", who, S);
    for (int j = 0; j < n; ++j) {
        int rc = check_tensor(hs[j], who);
        if (rc) return rc;
        ts[j] = reinterpret_cast<const Tensor *>(hs[j]);
        if (ts[j]->fmt != ts[0]->fmt || ts[j]->I != ts[0]->I)
            return fail(B200Q_EINVAL, "%s: tensor %d differs from tensor 0 in format or I", who, j);
    }
    if (S == 0) return B200Q_OK;
    const size_t xbytes = (size_t)S * ts[0]->I * 4;
    for (int j = 0; j < n; ++j) {
        const size_t yb = (size_t)S * ts[j]->O * 4;
        if (!xa[j] || !ys[j] || (xb && !xb[j]))
            return fail(B200Q_EINVAL, "%s: set %d: device pointers must not be NULL", who, j);
        if (!aligned16(xa[j]) || !aligned16(ys[j]) || (xb && !aligned16(xb[j])))
            return fail(B200Q_EINVAL, "%s: set %d: device pointers must be 16-byte aligned", who, j);
        for (int k = 0; k < n; ++k) {
            if (overlap(ys[j], yb, xa[k], xbytes) || (xb && overlap(ys[j], yb, xb[k], xbytes)))
                return fail(B200Q_EINVAL, "%s: output %d overlaps input %d", who, j, k);
            if (k != j && overlap(ys[j], yb, ys[k], (size_t)S * ts[k]->O * 4))
                return fail(B200Q_EINVAL, "%s: outputs %d and %d overlap", who, j, k);
        }
    }
    return B200Q_OK;
}

int run_group(const b200q_tensor *const *hs, int n, const float *const *xa, const float *const *xb,
              float *const *ys, int S, cudaStream_t st, const char *who) {
    const Tensor *ts[B200Q_GROUP_MAX];
    int rc = check_group(hs, n, xa, xb, ys, S, ts, who);
    if (rc || S == 0) return rc;
    const bool silu = xb != nullptr;
    // below the bf16 tensor-core threshold the whole group is one decode launch
    // per two rows; from it, each tensor runs its own tensor-core call
    if (select_path(*ts[0], S, B200Q_PATH_AUTO) != B200Q_PATH_TC) {
        bool handled = false;
        cudaError_t e = launch_decode_group(ts, n, xa, xb, ys, silu, S, st, &handled);
        if (e != cudaSuccess) return cuda_fail(e, who);
        if (handled) return B200Q_OK;
    }
    // one call per tensor; the gated inputs go through a workspace first
    float *h = nullptr;
    const size_t xn = (size_t)S * ts[0]->I;
    if (silu) {
        cudaError_t e = workspace_alloc((void **)&h, (size_t)n * xn * 4, st);
        if (e != cudaSuccess) return cuda_fail(e, who);
    }
    for (int j = 0; j < n && rc == B200Q_OK; ++j) {
        const float *x = xa[j];
        if (silu) {
            cudaError_t e = launch_silu_mul(xa[j], xb[j], h + j * xn, (long)xn, st);
            if (e != cudaSuccess) rc = cuda_fail(e, who);
            x = h + j * xn;
        }
        if (rc == B200Q_OK) rc = run_matmul(*ts[j], nullptr, x, ys[j], nullptr, S, B200Q_PATH_AUTO, st, who);
    }
    if (h) {
        cudaError_t e = workspace_free(h, st);
        if (rc == B200Q_OK && e != cudaSuccess) rc = cuda_fail(e, who);
    }
    return rc;
}

}  // namespace

extern "C" {

int b200q_matmul_grouped(const b200q_tensor *const *ts, int n, const float *const *xs, float *const *ys, int S,
                         void *stream) {
    return run_group(ts, n, xs, nullptr, ys, S, (cudaStream_t)stream, "b200q_matmul_grouped");
}

int b200q_matmul_grouped_silu(const b200q_tensor *const *ts, int n, const float *const *gs,
                              const float *const *us, float *const *ys, int S, void *stream) {
    if (!us) return fail(B200Q_EINVAL, "b200q_matmul_grouped_silu: NULL host array");
    return run_group(ts, n, gs, us, ys, S, (cudaStream_t)stream, "b200q_matmul_grouped_silu");
}

int b200q_matmul_tc_noalloc(const b200q_tensor *h, const float *x, float *y, int S, void *stream) {
    int rc = check_tensor(h, "b200q_matmul_tc_noalloc");
    if (rc) return rc;
    const Tensor &t = *reinterpret_cast<const Tensor *>(h);
    if (t.fmt != B200Q_I4 && t.fmt != B200Q_I8)
        return fail(B200Q_EINVAL, "b200q_matmul_tc_noalloc: takes int8 and int4 tensors only");
    if (S < 0) return fail(B200Q_EINVAL, "b200q_matmul_tc_noalloc: S must be >= 0 (got %d)", S);
    if (S == 0) return B200Q_OK;
    const size_t need = (size_t)S * (size_t)t.k_pad * 2;
    if (need > noalloc_capacity())
        return fail(B200Q_EINVAL,
                    "b200q_matmul_tc_noalloc: S=%d x %lld padded columns needs %zu bytes of workspace, more than "
                    "the fixed %zu bytes (use b200q_matmul or a smaller S)",
                    S, t.k_pad, need, noalloc_capacity());
    rc = check_io(t, x, y, S, "b200q_matmul_tc_noalloc");
    if (rc) return rc;
    cudaError_t e = launch_prefill_tc_noalloc(t, x, y, S, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "b200q_matmul_tc_noalloc");
    return B200Q_OK;
}

long long b200q_tc_noalloc_capacity(void) { return (long long)noalloc_capacity(); }

int b200q_silu_mul(const float *g, const float *u, float *h, long n, void *stream) {
    if (n < 0) return fail(B200Q_EINVAL, "b200q_silu_mul: n must be >= 0");
    if (n == 0) return B200Q_OK;
    if (!g || !u || !h) return fail(B200Q_EINVAL, "b200q_silu_mul: NULL pointer");
    if (!aligned16(g) || !aligned16(u) || !aligned16(h))
        return fail(B200Q_EINVAL, "b200q_silu_mul: pointers must be 16-byte aligned");
    const size_t nb = (size_t)n * 4;
    if ((h != g && overlap(h, nb, g, nb)) || (h != u && overlap(h, nb, u, nb)))
        return fail(B200Q_EINVAL, "b200q_silu_mul: h partially overlaps g or u");
    cudaError_t e = launch_silu_mul(g, u, h, n, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "b200q_silu_mul");
    return B200Q_OK;
}

int b200q_rmsnorm(const float *x, const float *r, float *h, const float *w, float *y, int S, int D, float eps,
                  void *stream) {
    if (S < 0 || D < 1) return fail(B200Q_EINVAL, "b200q_rmsnorm: need S >= 0 and D >= 1 (got S=%d, D=%d)", S, D);
    if (!(eps >= 0.f) || eps > 3.0e38f) return fail(B200Q_EINVAL, "b200q_rmsnorm: eps must be finite and >= 0");
    if (S == 0) return B200Q_OK;
    if (!x || !w || !y) return fail(B200Q_EINVAL, "b200q_rmsnorm: x, w and y must not be NULL");
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (r && !aligned16(r)) || (h && !aligned16(h)))
        return fail(B200Q_EINVAL, "b200q_rmsnorm: pointers must be 16-byte aligned");
    const size_t nb = (size_t)S * D * 4;
    if (overlap(y, nb, x, nb) || (r && overlap(y, nb, r, nb)) || (h && overlap(y, nb, h, nb)) ||
        overlap(y, nb, w, (size_t)D * 4))
        return fail(B200Q_EINVAL, "b200q_rmsnorm: y must not overlap x, r, h or w");
    if (h && ((h != x && overlap(h, nb, x, nb)) || (r && h != r && overlap(h, nb, r, nb))))
        return fail(B200Q_EINVAL, "b200q_rmsnorm: h may equal x or r but must not partially overlap them");
    cudaError_t e = launch_rmsnorm(x, r, h, w, y, S, D, eps, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "b200q_rmsnorm");
    return B200Q_OK;
}

int b200q_matmul_host(const b200q_tensor *h, const float *x_host, float *y_host, int S, void *stream) {
    int rc = check_tensor(h, "b200q_matmul_host");
    if (rc) return rc;
    const Tensor &t = *reinterpret_cast<const Tensor *>(h);
    if (S < 0) return fail(B200Q_EINVAL, "b200q_matmul_host: S must be >= 0 (got %d)", S);
    if (S == 0) return B200Q_OK;
    if (!x_host || !y_host) return fail(B200Q_EINVAL, "b200q_matmul_host: NULL host pointer");
    if (t.device < 0 || t.device >= 64) return fail(B200Q_EINVAL, "b200q_matmul_host: device index too large");
    const size_t xb = (size_t)S * t.I * 4, yb = (size_t)S * t.O * 4;
    const size_t xb_al = (xb + 255) / 256 * 256;
    cudaStream_t st = (cudaStream_t)stream;
    Staging &sg = g_staging[t.device];
    std::lock_guard<std::mutex> lock(sg.m);
    cudaError_t e = cudaSuccess;
    if (sg.cap < xb_al + yb) {
        if (sg.buf) {
            e = cudaStreamSynchronize(st);
            if (e == cudaSuccess) e = cudaFree(sg.buf);
            sg.buf = nullptr;
            sg.cap = 0;
            if (e != cudaSuccess) return cuda_fail(e, "b200q_matmul_host: free staging");
        }
        count_workspace_alloc();
        e = cudaMalloc(&sg.buf, xb_al + yb);
        if (e != cudaSuccess) {
            sg.buf = nullptr;
            cudaGetLastError();
            return cuda_fail(e, "b200q_matmul_host: staging allocation");
        }
        sg.cap = xb_al + yb;
    }
    float *xd = (float *)sg.buf;
    float *yd = (float *)((char *)sg.buf + xb_al);
    e = cudaMemcpyAsync(xd, x_host, xb, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "b200q_matmul_host: copy x to device");
    rc = run_matmul(t, nullptr, xd, yd, nullptr, S, B200Q_PATH_AUTO, st, "b200q_matmul_host");
    if (rc) return rc;
    e = cudaMemcpyAsync(y_host, yd, yb, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "b200q_matmul_host: copy y to host");
    return B200Q_OK;
}

}  // extern "C"

extern "C" {

int b200q_mla_absorb(const b200q_tensor *wkv_b, int H, int Dn, int Dv, const float *q_nope, const float *q_rope,
                     const float *const *lat_pages, const float *const *rope_pages, int R, int T, int st0,
                     float scale, float *ctx, int S, void *stream) {
    const char *who = "b200q_mla_absorb";
    int rc = check_tensor(wkv_b, who);
    if (rc) return rc;
    const Tensor &w = *reinterpret_cast<const Tensor *>(wkv_b);
    if (S < 0) return fail(B200Q_EINVAL, "%s: S must be >= 0 (got %d)", who, S);
    if (S == 0) return B200Q_OK;
    if (H < 1 || Dn < 1 || Dv < 1 || R < 0)
        return fail(B200Q_EINVAL, "%s: need H, Dn, Dv >= 1 and R >= 0 (got %d, %d, %d, %d)", who, H, Dn, Dv, R);
    if ((long long)H * (Dn + Dv) != w.O)
        return fail(B200Q_EINVAL, "%s: the tensor has %d rows, H * (Dn + Dv) = %lld", who, w.O,
                    (long long)H * (Dn + Dv));
    const int K = w.I;
    if (K % 4 || R % 4 || K > mla_max_latent())
        return fail(B200Q_EINVAL, "%s: need K and R multiples of 4 and K <= %d (got K=%d, R=%d)", who,
                    mla_max_latent(), K, R);
    if (mla_smem_bytes(K, R) > 227 * 1024)
        return fail(B200Q_EINVAL, "%s: K + R = %d is too wide for one tile in shared memory", who, K + R);
    if (T < S || st0 < 0 || st0 > T - S || T > (1 << 30))
        return fail(B200Q_EINVAL, "%s: need S <= T <= 2^30 and 0 <= st0 <= T - S (got T=%d, st0=%d, S=%d)", who, T,
                    st0, S);
    if ((long long)H * S > (1 << 20)) return fail(B200Q_EINVAL, "%s: H * S above 2^20", who);
    if (S > 4 * 65535) return fail(B200Q_EINVAL, "%s: S above %d (token blocks of 4 per grid row)", who, 4 * 65535);
    if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return fail(B200Q_EINVAL, "%s: scale must be finite", who);
    if (!q_nope || !ctx || !lat_pages || (R && (!q_rope || !rope_pages)))
        return fail(B200Q_EINVAL, "%s: device pointers must not be NULL", who);
    if (!aligned16(q_nope) || !aligned16(ctx) || (R && !aligned16(q_rope)) || ((uintptr_t)lat_pages & 7u) ||
        (R && ((uintptr_t)rope_pages & 7u)))
        return fail(B200Q_EINVAL, "%s: q_nope, q_rope and ctx must be 16-byte aligned, the page arrays 8-byte", who);
    const size_t cb = (size_t)S * H * Dv * 4;
    if (overlap(ctx, cb, q_nope, (size_t)S * H * Dn * 4) || (R && overlap(ctx, cb, q_rope, (size_t)S * H * R * 4)))
        return fail(B200Q_EINVAL, "%s: ctx must not overlap q_nope or q_rope", who);
    cudaStream_t st = (cudaStream_t)stream;
    float *ws = nullptr;
    cudaError_t e = workspace_alloc((void **)&ws, mla_workspace_floats(H, S, K, T, st0) * 4, st);
    if (e != cudaSuccess) return cuda_fail(e, who);
    e = launch_mla_absorb(w, H, Dn, Dv, q_nope, q_rope, lat_pages, rope_pages, R, T, st0, scale, ctx, S, ws, st);
    cudaError_t e2 = workspace_free(ws, st);
    if (e != cudaSuccess) return cuda_fail(e, who);
    if (e2 != cudaSuccess) return cuda_fail(e2, who);
    return B200Q_OK;
}

int b200q_kv_append(float *const *lat_pages, float *const *rope_pages, int K, int R, int pos, const float *lat_rows,
                    const float *rope_rows, int n, void *stream) {
    const char *who = "b200q_kv_append";
    if (n < 0 || K < 1 || R < 0 || pos < 0 || (long long)pos + n > (1ll << 30))
        return fail(B200Q_EINVAL, "%s: need n >= 0, K >= 1, R >= 0, 0 <= pos, pos + n <= 2^30", who);
    if (n == 0) return B200Q_OK;
    if (!lat_pages || !lat_rows || (R && (!rope_pages || !rope_rows)))
        return fail(B200Q_EINVAL, "%s: device pointers must not be NULL", who);
    cudaError_t e = launch_kv_append(lat_pages, rope_pages, K, R, pos, lat_rows, rope_rows, n, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, who);
    return B200Q_OK;
}

}  // extern "C"

extern "C" int b200q_selftest_timeout(int wait_us, void *stream) {
    if (wait_us < 1 || wait_us > 1000000)
        return fail(B200Q_EINVAL, "b200q_selftest_timeout: wait_us must be in [1, 1000000] (got %d)", wait_us);
    cudaError_t e = launch_wait_selftest((unsigned long long)wait_us * 1000ull, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "b200q_selftest_timeout");
    return B200Q_OK;
}
