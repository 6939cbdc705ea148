// Internal declarations of the b200q library (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "b200q.h"

namespace qwq {

// Device copy of one weight tensor.
//
// codes: [o_pad, ld] bytes, row-major.  A row holds the host row's bytes
//        followed by padding up to ld (a multiple of kRowAlign).  Padding
//        bytes, the unused high bits of a row's last byte, and the rows
//        o >= O all hold the format's zero-point code, so they decode to 0.
// scales: [o_pad] f32, or [o_pad, G_ld] with group-wise scales (G used, the
//        rest of a row 0); rows o >= O have scale 0.
struct Tensor {
    CUtensorMap dec_map;  // codes as uint32 [o_pad, ld / 4], box 8 rows x 512 bytes (decode stages)
    CUtensorMap sc_map;   // group scales as f32 [o_pad, G_ld], box 8 rows x sc_box (decode stages)
    CUtensorMap gemm_map;     // int8 / int4 codes as bytes [o_pad, ld], box 128 rows x one k-block (tensor-core GEMM)
    CUtensorMap gemm_sc_map;  // group scales as f32 [o_pad, G_ld], box 128 rows x 4 (tensor-core GEMM)
    CUtensorMap tcs_map;      // int8 / int4 / int2 codes as bytes [o_pad, ld], box 128 rows x 128 bytes,
                              // 128-byte swizzle (f32-accurate tensor-core path for few tokens)
    int fmt;
    int O, I;
    int device;
    int o_pad;        // O rounded up to kRowTile
    long long ld;     // device row stride in bytes
    long long k_pad;  // elements per padded row = ld * 8 / bits
    uint8_t *codes;
    float *scales;    // [o_pad] per row, or [o_pad, G] per row and group
    size_t bytes;     // one allocation: codes then scales
    int gs;           // group size of the scales; 0: one scale per row
    int G;            // scales per row (1, or ceil(I / gs))
    int G_ld;         // device row stride of the scales in floats (G rounded up to 4, >= sc_box)
    int sc_box;       // group scales one decode stage (8 rows x 512 code bytes) spans, from a
                      // 4-aligned first group, rounded up to 4
};

// Group sizes the kernels take: a multiple of a 16-byte chunk's element
// count (4 f32, 16 int8, 32 int4, 64 int2), or 16 or 32 dividing it.
inline bool group_size_ok(int fmt, int gs) {
    const int per = fmt == B200Q_F32 ? 4 : fmt == B200Q_I8 ? 16 : fmt == B200Q_I4 ? 32 : fmt == B200Q_I2 ? 64 : 0;
    if (per == 0 || gs < 1) return false;
    return gs % per == 0 || ((gs == 16 || gs == 32) && per % gs == 0);
}

constexpr int kRowAlign = 128;  // bytes; rows start on 128-byte boundaries
constexpr int kRowTile = 128;   // O is padded to a multiple of this
constexpr int kTcxMinS = 5;     // default first S of the three-piece tensor-core path (int8 / int4)

inline int fmt_bits(int fmt) {
    return fmt == B200Q_F32 ? 32 : fmt == B200Q_I8 ? 8 : fmt == B200Q_I4 ? 4 : fmt == B200Q_I2 ? 2 : 0;
}

// Zero-point code replicated over a byte: decodes to 0 in every position.
inline uint8_t zero_byte(int fmt) {
    return fmt == B200Q_I4 ? 0x88 : fmt == B200Q_I2 ? 0xAA : 0x00;
}

// 2-D tiled tensor map (cuTensorMapEncodeTiled through the runtime's driver
// entry point): inner extent `inner` elements, `outer` rows of `row_bytes`.
// Returns false if the driver entry point is missing or encoding fails.
bool tmap_encode_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

// Counts kernel launches made through the library (b200q_kernel_launches).
void count_launch(int n = 1);

// Counts device workspace allocations the library makes on a call's behalf
// (stream-ordered pool allocations, the pool's creation, the host-call
// staging buffer); b200q_workspace_allocations reports the total.
void count_workspace_alloc();

// Stream-ordered device workspace from the library's per-device pool
// (counted by count_workspace_alloc), and its release on the same stream.
cudaError_t workspace_alloc(void **ptr, size_t bytes, cudaStream_t st);
cudaError_t workspace_free(void *ptr, cudaStream_t st);

// Multiprocessor count of device dev, read once per device; safe when
// several host threads make their first calls at the same time.
int sm_count(int dev);

// Raises kernel fn's dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device, bytes); thread-safe.
cudaError_t allow_dynamic_smem(const void *fn, int bytes);

// ---- kernels (launchers return cudaGetLastError() after the launch) ----

// Tail fix after the upload copy: forces the unused high bits of every row's
// last host byte to the zero-point pattern.
cudaError_t launch_fix_row_tails(const Tensor &t, long long rb, cudaStream_t st);

// Encodes the tensor-core GEMM's tensor maps of an uploaded int8 / int4
// tensor (codes, and group scales when gs > 0); other formats need none.
bool gemm_maps_encode(Tensor &t);

// Encodes Tensor::tcs_map (int8 / int4 / int2 tensors; others need none).
bool tcs_map_encode(Tensor &t);

// f32-accurate SIMT path, any format, any S.  With tu != nullptr the launch
// also computes yu = matmul(tu, x) (gate/up pair, same shape as t).
cudaError_t launch_qmv_simt(const Tensor &t, const Tensor *tu, const float *x, float *y,
                            float *yu, int S, cudaStream_t st);

cudaError_t launch_silu_mul(const float *g, const float *u, float *h, long n, cudaStream_t st);

cudaError_t launch_rmsnorm(const float *x, const float *r, float *h, const float *w, float *y, int S, int D,
                           float eps, cudaStream_t st);

}  // namespace qwq
