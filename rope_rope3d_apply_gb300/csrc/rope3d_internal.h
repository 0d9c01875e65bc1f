// rope3d_internal.h -- shared between the host API (rope3d_api.cpp) and the
// kernels (rope3d_kernels.cu). Not part of the public ABI.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace rope3d {

// Unsigned division by a run-time constant, n / d for 0 <= n < 2^31 and
// 1 <= d < 2^31, by a multiply-high and a shift (Granlund and Montgomery,
// "Division by invariant integers using multiplication", PLDI 1994, the
// round-up multiplier): with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// n / d = (mulhi(n, m) + n) >> l. Because n < 2^31, the sum cannot overflow.
struct FastDiv {
    uint32_t d;
    uint32_t mul;
    uint32_t shift;
};

inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((uint64_t(1) << l) < d) ++l;
    const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
    return FastDiv{d, static_cast<uint32_t>(m), l};
}

inline uint32_t fastdiv_host(uint32_t n, const FastDiv &f) {
    const uint32_t hi = static_cast<uint32_t>((uint64_t(n) * f.mul) >> 32);
    return (hi + n) >> f.shift;
}

// Largest number of work units (16-byte vectors or pairs) one launch handles;
// keeps every in-kernel index below 2^31 with room for the unrolled stride.
constexpr uint32_t kMaxUnitsPerLaunch = 1u << 30;

// Tables up to this size are staged in shared memory; larger ones are read
// through the read-only data path.
constexpr uint32_t kMaxSmemTableBytes = 96 * 1024;

// Launch description. Device layout of the tables: one buffer of float2
// (cos, sin) entries, the T table [T][pT], then the H table [H][pH] at offH,
// then the W table [W][pW] at offW (each offset a multiple of 4 entries).
struct LaunchArgs {
    const void *q;
    const void *k;
    void *q_out;
    void *k_out;
    const float2 *tables;
    uint32_t table_len;     // float2 entries in the whole buffer
    uint32_t offH, offW;    // entry offsets of the H and W tables
    uint32_t pT, pH, pW;    // pairs per axis chunk (d_X / 2)
    uint32_t T, H, W;       // grid extents
    uint32_t heads, head_dim;
    uint64_t rows;          // (batch, token) rows in the buffers of this call
    uint64_t row0;          // global row index of the first row (host path chunks)
    int dtype;              // ROPE3D_BF16 / ROPE3D_F32 / ROPE3D_F16
    bool vec16;             // take the 16-byte vector kernel
    // Strided views: element strides of (batch, t, h, w, head) for Q, K,
    // Q_out, K_out (channels are contiguous). When `strided` is false the
    // buffers are contiguous and the strides are unused.
    bool strided;
    int64_t strides[4][5];
    // Launch with programmatic stream serialization (the kernel may start
    // while the previous kernel of the stream drains; it waits for it before
    // touching Q, K or the outputs). Only for launches whose preceding stream
    // work is kernels or already complete: not after an upload of the tables
    // or a cross-stream wait in the same call.
    bool pdl;
};

// Copy a strided view ([B, T, H, W, heads, head_dim], element strides of
// (batch, t, h, w, head), contiguous channels) into a contiguous buffer.
// elem_bytes is 2 or 4.
cudaError_t launch_gather(const void *src, const int64_t strides[5], void *dst, int elem_bytes,
                          uint64_t B, uint32_t T, uint32_t H, uint32_t W, uint32_t heads,
                          uint32_t head_dim, cudaStream_t stream);

struct LaunchInfo {
    int kernel;  // 1 = vector, 2 = per-pair
    int grid;
    int block;
};

// Test hook: lower the units-per-launch cap so that small inputs take the
// multi-launch path (0 restores kMaxUnitsPerLaunch).
void set_max_units_per_launch(uint32_t n);
// The same for the K pass of rope3d_na3d_rotate_once.
void na3d_set_max_units_per_launch(uint32_t n);

// Launch the rotation; splits into several launches when needed. Returns a
// cudaError_t from the launch.
cudaError_t launch_rope3d(const LaunchArgs &a, cudaStream_t stream, LaunchInfo *info);

// The argument checks of rope3d_apply_pair without a table handle (shape,
// dtype, alignment, overlap, device memory of the current device). Returns a
// ROPE3D_* status. Allocates nothing.
int check_call_without_tables(const void *q, const void *k, const void *q_out, const void *k_out,
                              int64_t B, int64_t T, int64_t H, int64_t W, int64_t heads,
                              int64_t head_dim, const int32_t split[3], int32_t dtype);

}  // namespace rope3d

// Debug builds compile every kernel with -DROPE3D_DEBUG_BOUNDS=1: each computed
// index is checked before the access it guards; a failed check counts in the
// kernel file's error word and skips the access.
#ifndef ROPE3D_DEBUG_BOUNDS
#define ROPE3D_DEBUG_BOUNDS 0
#endif

namespace rope3d {
// Per kernel file: the bound-check error count (0 without the checks), -1 on a
// CUDA error; reset clears it.
int64_t kernels_bound_errors(bool reset);
int64_t patchify_bound_errors(bool reset);
int64_t neox_bound_errors(bool reset);
int64_t na3d_bound_errors(bool reset);
}  // namespace rope3d

struct rope3d_tables;
namespace rope3d {
// The device layout of a table handle: the float2 (cos, sin) buffer, its
// length in entries, the entry offsets of the T, H and W tables, the key, the
// device it lives on, and whether it is the host-memory test mode.
int tables_layout(const rope3d_tables *t, const float2 **dev, uint32_t *len, uint32_t offsets[3],
                  int64_t dims[3], int32_t split[3], int *device, bool *host_backed);
// Record that work just enqueued on `stream` reads t's tables, so that t's
// memory outlives that work when its last reference is released. Returns a
// ROPE3D_* status.
// Return the memory the attention's scratch pools keep (rope3d_na3d's K
// scratch) to the device, except what is still in use.
void na3d_scratch_trim();
int tables_note_use(const rope3d_tables *t, cudaStream_t stream);
}  // namespace rope3d
