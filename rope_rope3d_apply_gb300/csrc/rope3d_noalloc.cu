// rope3d_noalloc.cu -- rope3d_apply_pair_noalloc: the rotation for callers
// that cannot allocate device memory.
//
// rope3d_apply_pair needs a table handle, and rope3d_build_tables allocates a
// device buffer for it with cudaMalloc. Some callers cannot do that: a process
// whose device memory is owned by another allocator (a framework's caching
// pool, a fixed memory budget carved out at start-up), or code that must not
// take cudaMalloc's implicit device synchronisation in the middle of a
// pipeline. This entry point needs no handle: it builds the three axis tables
// on the host and uploads them into a fixed table area that lives in this
// file's static device memory, then launches the same kernels on it. It calls
// no cudaMalloc, cudaFree, host heap allocation or other allocating routine.
//
// The table area (kStaticTableBytes, 64 KiB) is a file-scope __device__ array:
// every GPU that loads the library holds it until the process exits. In host
// code its name is only a host-side stand-in for the symbol, so the device
// address is looked up once per device with cudaGetSymbolAddress and that
// address is what the kernel receives. The address is kept for the life of
// the process: calls after a cudaDeviceReset of that device are unsupported.
//
// The upload comes from pageable host memory, which a stream in capture mode
// cannot record; a capturing stream is therefore refused before anything is
// enqueued, so that the caller's capture is not invalidated.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/rope3d.h"
#include "rope3d_internal.h"

namespace {

constexpr size_t kStaticTableBytes = 64 * 1024;
constexpr uint32_t kStaticTableEntries = kStaticTableBytes / sizeof(float2);
constexpr int kMaxDevices = 64;

// The scratch: (cos, sin) entries of the T, H and W tables, each table starting
// at a multiple of 4 entries. Every call overwrites the part it reads.
static __device__ __align__(256) float2 g_static_tables[kStaticTableEntries];

// Host staging of the table values (no heap), and the per-device addresses of
// g_static_tables. The mutex serialises calls on the host.
float2 g_host_tables[kStaticTableEntries];
void *g_table_addr[kMaxDevices] = {};
std::mutex g_mutex;

// Device address of g_static_tables on the current device (set up on the
// first call on each device).
int static_tables_address(int device, float2 **out) {
    if (device < 0 || device >= kMaxDevices) return ROPE3D_ERR_DEVICE;
    if (!g_table_addr[device]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_tables) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return ROPE3D_ERR_CUDA;
        }
        g_table_addr[device] = ptr;
    }
    *out = static_cast<float2 *>(g_table_addr[device]);
    return ROPE3D_OK;
}

// One axis table into g_host_tables at `offset`: entry (p, j) is
// (cos, sin) of p * base^(-2j/dim), in double, rounded once to float -- the
// same values rope3d_build_tables produces.
void fill_axis(int64_t length, int64_t dim, double base, uint32_t offset) {
    const int64_t half = dim / 2;
    for (int64_t p = 0; p < length; ++p) {
        for (int64_t j = 0; j < half; ++j) {
            const double inv_freq = std::pow(base, -(2.0 * static_cast<double>(j)) /
                                                       static_cast<double>(dim));
            const double angle = static_cast<double>(p) * inv_freq;
            g_host_tables[offset + p * half + j] =
                float2{static_cast<float>(std::cos(angle)), static_cast<float>(std::sin(angle))};
        }
    }
}

}  // namespace

extern "C" int rope3d_apply_pair_noalloc(const void *q, const void *k, void *q_out, void *k_out,
                                         int64_t B, int64_t T, int64_t H, int64_t W,
                                         int64_t heads, int64_t head_dim,
                                         const int32_t split[3], double base, int32_t dtype,
                                         void *stream) {
    int rc = rope3d::check_call_without_tables(q, k, q_out, k_out, B, T, H, W, heads, head_dim,
                                               split, dtype);
    if (rc != ROPE3D_OK) return rc;
    if (!(std::isfinite(base) && base > 0.0)) return ROPE3D_ERR_ARG;

    // table layout: T | H | W, each rounded up to a multiple of 4 entries
    const int64_t lengths[3] = {T, H, W};
    uint32_t offset[3];
    uint64_t total = 0;
    for (int a = 0; a < 3; ++a) {
        offset[a] = static_cast<uint32_t>(total);
        total += (static_cast<uint64_t>(lengths[a]) * (split[a] / 2) + 3) / 4 * 4;
        if (total > kStaticTableEntries) return ROPE3D_ERR_SCRATCH;
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &capture) != cudaSuccess) {
        cudaGetLastError();
        return ROPE3D_ERR_CUDA;
    }
    if (capture != cudaStreamCaptureStatusNone) return ROPE3D_ERR_ARG;

    std::lock_guard<std::mutex> lock(g_mutex);
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return ROPE3D_ERR_CUDA;
    float2 *tables = nullptr;
    rc = static_tables_address(device, &tables);
    if (rc != ROPE3D_OK) return rc;

    for (int a = 0; a < 3; ++a) fill_axis(lengths[a], split[a], base, offset[a]);
    // From pageable memory: returns once the values have been taken from
    // g_host_tables, so the next call may overwrite them.
    if (cudaMemcpyAsync(tables, g_host_tables, total * sizeof(float2), cudaMemcpyHostToDevice,
                        s) != cudaSuccess)
        return ROPE3D_ERR_CUDA;

    const int64_t vec = 16 / (dtype == ROPE3D_F32 ? 4 : 2);
    bool vec16 = head_dim % vec == 0;
    for (int a = 0; a < 3; ++a) vec16 = vec16 && split[a] % vec == 0;
    for (const void *p : {q, k, static_cast<const void *>(q_out), static_cast<const void *>(k_out)})
        vec16 = vec16 && reinterpret_cast<uintptr_t>(p) % 16 == 0;

    rope3d::LaunchArgs la{};
    la.q = q;
    la.k = k;
    la.q_out = q_out;
    la.k_out = k_out;
    la.tables = tables;
    la.table_len = static_cast<uint32_t>(total);
    la.offH = offset[1];
    la.offW = offset[2];
    la.pT = static_cast<uint32_t>(split[0] / 2);
    la.pH = static_cast<uint32_t>(split[1] / 2);
    la.pW = static_cast<uint32_t>(split[2] / 2);
    la.T = static_cast<uint32_t>(T);
    la.H = static_cast<uint32_t>(H);
    la.W = static_cast<uint32_t>(W);
    la.heads = static_cast<uint32_t>(heads);
    la.head_dim = static_cast<uint32_t>(head_dim);
    la.rows = static_cast<uint64_t>(B * T * H * W);
    la.row0 = 0;
    la.dtype = dtype;
    la.vec16 = vec16;
    rope3d::LaunchInfo info{};
    if (rope3d::launch_rope3d(la, s, &info) != cudaSuccess) return ROPE3D_ERR_CUDA;
    return ROPE3D_OK;
}
