// rope3d_patchify.cu -- space-to-depth layout kernels of the LTX-2.5 diffusion
// decoder: rope3d_patchify and rope3d_unpatchify.
//
// sglang PR #34471 review, "关键源码片段", _patchify in
// ltx_2_5_diffusion_decoder.py: x of shape (B, C, F, H, W) becomes
// y of shape (B, C*p*p, F, H/p, W/p) with the channels packed in the order
// (channel, width offset, height offset):
//     y[b, (c*p + pw)*p + ph, f, i, j] = x[b, c, f, i*p + ph, j*p + pw].
// _unpatchify (named there without code) is its exact inverse.
//
// The work is a pure permutation, bound by HBM bandwidth. One thread owns a
// run of V = 16 / elem_bytes consecutive output columns j of one input row
// (b, c, f, h): it loads the p*V input elements that feed them (p 16-byte
// loads, contiguous across the warp), de-interleaves them in registers by
// width offset, and stores p 16-byte vectors, one into each of the p output
// rows (c, pw, ph) -- also contiguous across the warp. Unpatchify runs the same
// loop backwards. Shapes whose rows are not a whole number of vectors, or
// patch sizes other than 1, 2, 4 and 8, take an element-per-thread kernel.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/rope3d.h"
#include "rope3d_internal.h"

namespace {

using rope3d::FastDiv;
using rope3d::make_fastdiv;

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) {
    return (__umulhi(n, f.mul) + n) >> f.shift;
}

template <int ES> struct ElemT;
template <> struct ElemT<1> { using T = uint8_t; };
template <> struct ElemT<2> { using T = uint16_t; };
template <> struct ElemT<4> { using T = uint32_t; };
template <> struct ElemT<8> { using T = uint64_t; };

struct PParams {
    const char *src;
    char *dst;
    uint32_t units;        // work units of this launch
    FastDiv per_row;       // units per input row (b, c, f, h)
    FastDiv Hd;            // H
    FastDiv CF, Fd;        // C*F, F
    FastDiv pd;            // p (scalar kernels)
    FastDiv Wd;            // W (scalar kernels)
    uint32_t bcf0;         // first (b, c, f) of this launch
    uint32_t C, F, H, W, p;
    uint32_t Hp, Wp;
    unsigned long long total;   // bytes of x (and of y), for the debug bound checks
};

// Debug builds (-DROPE3D_DEBUG_BOUNDS=1) check each computed byte offset
// before the access it guards: a failed check counts in this file's error word
// and skips the access (never a trap). Otherwise every check compiles away.
#if ROPE3D_DEBUG_BOUNDS
__device__ unsigned int g_bound_errors;
__device__ __forceinline__ bool bound_ok(unsigned long long off, unsigned long long len,
                                         unsigned long long lim) {
    if (off + len <= lim) return true;
    atomicAdd(&g_bound_errors, 1u);
    return false;
}
#else
__device__ __forceinline__ constexpr bool bound_ok(unsigned long long, unsigned long long,
                                                   unsigned long long) {
    return true;
}
#endif

// Decoded input row: global (b, c, f) index, and h split into (i, ph).
struct Row {
    uint32_t b, c, f, i, ph;
    uint64_t row;          // global row index (b, c, f, h)
};

__device__ __forceinline__ Row decode_row(const PParams &q, uint32_t row_local, uint32_t p) {
    Row r;
    const uint32_t bcf_local = fdiv(row_local, q.Hd);
    const uint32_t h = row_local - bcf_local * q.H;
    const uint32_t bcf = q.bcf0 + bcf_local;
    r.b = fdiv(bcf, q.CF);
    const uint32_t rem = bcf - r.b * q.CF.d;
    r.c = fdiv(rem, q.Fd);
    r.f = rem - r.c * q.F;
    r.i = h / p;
    r.ph = h - r.i * p;
    r.row = uint64_t(bcf) * q.H + h;
    return r;
}

// Element offset of output row (b, c, pw, ph, f, i) of the patchified tensor.
__device__ __forceinline__ uint64_t patched_row(const PParams &q, const Row &r, uint32_t pw,
                                                uint32_t p) {
    const uint64_t ch = (uint64_t(r.b) * q.C + r.c) * p * p + uint64_t(pw) * p + r.ph;
    return ((ch * q.F + r.f) * q.Hp + r.i) * q.Wp;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void *ptr) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::128B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(ptr));
    return v;
}

__device__ __forceinline__ void st_cs_v4(void *ptr, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};"
                 :
                 : "l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// ---- vector kernels ----------------------------------------------------------
// The x side of a warp's 32 units is one contiguous run of 32*P 16-byte chunks
// (units are consecutive runs of x rows, and x rows are contiguous). A unit
// owns P consecutive chunks, so if each lane moved its own chunks every warp
// access would touch every other 32-byte sector. Instead the warp moves the
// run chunk-by-chunk across lanes (lane t handles chunks t, t+32, ...), fully
// coalesced, and swaps it through shared memory into per-unit order. The y
// side is coalesced per width offset as it is. A warp whose 32 units are not
// all in range (the last one) moves its chunks lane by lane.

// Programmatic dependent launch: a kernel lets the next kernel of the stream
// start launching at once, and waits for the grids before it to complete (and
// their writes to become visible) before it touches memory, so back-to-back
// launches overlap one kernel's tail with the next one's launch. Launched
// without the attribute, both instructions return at once.
__device__ __forceinline__ void pdl_begin() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Shared-memory slot of chunk c of a warp's run: an XOR swizzle of the low three
// bits, so that both lane-contiguous and lane-strided (by P) accesses hit eight
// different 16-byte bank groups per quarter warp.
__device__ __forceinline__ uint32_t swz(uint32_t c) { return c ^ ((c >> 3) & 7u); }

template <int P, int ES, bool kForward>
__global__ void __launch_bounds__(kThreads)
patchify_vec_kernel(const PParams q) {
    using E = typename ElemT<ES>::T;
    constexpr int V = 16 / ES;  // output columns per thread and width offset
    __shared__ uint4 stage[kThreads / 32][32 * P];
    pdl_begin();
    const uint32_t lane = threadIdx.x & 31u;
    uint4 *ws = stage[threadIdx.x >> 5];
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t base = blockIdx.x * blockDim.x + (threadIdx.x & ~31u); base < q.units;
         base += stride) {
        const uint32_t u = base + lane;
        const bool whole = base + 31 < q.units;   // warp-uniform
        const bool active = u < q.units;
        const uint32_t row_local = fdiv(u, q.per_row);
        const uint32_t jv = u - row_local * q.per_row.d;
        const Row r = decode_row(q, row_local, P);
        const uint64_t col = uint64_t(jv) * V;                       // first output column
        // byte offset in x of the warp's first unit (units map to x contiguously)
        const uint32_t base_row = fdiv(base, q.per_row);
        const uint32_t base_jv = base - base_row * q.per_row.d;
        const uint64_t xb = ((uint64_t(q.bcf0) * q.H + base_row) * q.W + uint64_t(base_jv) * V * P) * ES;
        E e[V * P];
        uint4 raw[P];
        if constexpr (kForward) {
            if (whole) {
#pragma unroll
                for (int k = 0; k < P; ++k) {
                    const uint64_t o = xb + 16 * (k * 32 + lane);
                    ws[swz(k * 32 + lane)] = bound_ok(o, 16, q.total) ? ld_nc_v4(q.src + o) : make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
#pragma unroll
                for (int k = 0; k < P; ++k) raw[k] = ws[swz(lane * P + k)];
                __syncwarp();
            } else if (active) {
                const uint64_t x_off = r.row * q.W + uint64_t(jv) * V * P;
#pragma unroll
                for (int k = 0; k < P; ++k) {
                    const uint64_t o = x_off * ES + 16 * k;
                    raw[k] = bound_ok(o, 16, q.total) ? ld_nc_v4(q.src + o) : make_uint4(0, 0, 0, 0);
                }
            }
            if (active) {
                memcpy(e, raw, sizeof raw);
#pragma unroll
                for (int pw = 0; pw < P; ++pw) {
                    E o[V];
#pragma unroll
                    for (int t = 0; t < V; ++t) o[t] = e[t * P + pw];
                    uint4 ov;
                    memcpy(&ov, o, sizeof ov);
                    const uint64_t yo = (patched_row(q, r, pw, P) + col) * ES;
                    if (bound_ok(yo, 16, q.total)) st_cs_v4(q.dst + yo, ov);
                }
            }
        } else {
            if (active) {
#pragma unroll
                for (int pw = 0; pw < P; ++pw) {
                    const uint64_t o = (patched_row(q, r, pw, P) + col) * ES;
                    const uint4 iv = bound_ok(o, 16, q.total) ? ld_nc_v4(q.src + o) : make_uint4(0, 0, 0, 0);
                    E in[V];
                    memcpy(in, &iv, sizeof iv);
#pragma unroll
                    for (int t = 0; t < V; ++t) e[t * P + pw] = in[t];
                }
                memcpy(raw, e, sizeof raw);
            }
            if (whole) {
#pragma unroll
                for (int k = 0; k < P; ++k) ws[swz(lane * P + k)] = raw[k];
                __syncwarp();
#pragma unroll
                for (int k = 0; k < P; ++k) {
                    const uint64_t o = xb + 16 * (k * 32 + lane);
                    if (bound_ok(o, 16, q.total)) st_cs_v4(q.dst + o, ws[swz(k * 32 + lane)]);
                }
                __syncwarp();
            } else if (active) {
                const uint64_t x_off = r.row * q.W + uint64_t(jv) * V * P;
#pragma unroll
                for (int k = 0; k < P; ++k) {
                    const uint64_t o = x_off * ES + 16 * k;
                    if (bound_ok(o, 16, q.total)) st_cs_v4(q.dst + o, raw[k]);
                }
            }
        }
    }
}

// ---- element kernels (any patch size, any row length) ----------------------

template <int ES, bool kForward>
__global__ void __launch_bounds__(kThreads)
patchify_elem_kernel(const PParams q) {
    using E = typename ElemT<ES>::T;
    const E *src = reinterpret_cast<const E *>(q.src);
    E *dst = reinterpret_cast<E *>(q.dst);
    pdl_begin();
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < q.units; u += stride) {
        const uint32_t row_local = fdiv(u, q.Wd);
        const uint32_t w = u - row_local * q.W;
        const Row r = decode_row(q, row_local, q.p);
        const uint32_t j = fdiv(w, q.pd);
        const uint32_t pw = w - j * q.p;
        const uint64_t x_idx = r.row * q.W + w;
        const uint64_t y_idx = patched_row(q, r, pw, q.p) + j;
        if (!bound_ok(x_idx * ES, ES, q.total) || !bound_ok(y_idx * ES, ES, q.total)) continue;
        if constexpr (kForward) {
            dst[y_idx] = src[x_idx];
        } else {
            dst[x_idx] = src[y_idx];
        }
    }
}

using PFn = void (*)(PParams);

template <int ES, bool kForward>
PFn pick_vec(uint32_t p) {
    switch (p) {
        case 1: return patchify_vec_kernel<1, ES, kForward>;
        case 2: return patchify_vec_kernel<2, ES, kForward>;
        case 4: return patchify_vec_kernel<4, ES, kForward>;
        case 8: return patchify_vec_kernel<8, ES, kForward>;
        default: return nullptr;
    }
}

template <bool kForward>
PFn pick(int es, uint32_t p, bool vec) {
    if (vec) {
        switch (es) {
            case 1: return pick_vec<1, kForward>(p);
            case 2: return pick_vec<2, kForward>(p);
            case 4: return pick_vec<4, kForward>(p);
            case 8: return pick_vec<8, kForward>(p);
        }
        return nullptr;
    }
    switch (es) {
        case 1: return patchify_elem_kernel<1, kForward>;
        case 2: return patchify_elem_kernel<2, kForward>;
        case 4: return patchify_elem_kernel<4, kForward>;
        case 8: return patchify_elem_kernel<8, kForward>;
    }
    return nullptr;
}

bool device_ptr(const void *p, int device) {
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (attr.type == cudaMemoryTypeManaged) return true;
    return attr.type == cudaMemoryTypeDevice && attr.device == device;
}

thread_local int t_patch_kernel = 0;  // 1 vector, 2 element

int run(bool forward, const void *src, void *dst, int64_t B, int64_t C, int64_t F, int64_t H,
        int64_t W, int64_t p, int32_t elem_bytes, void *stream, bool check_device) {
    if (!src || !dst) return ROPE3D_ERR_NULL;
    if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
        return ROPE3D_ERR_DTYPE;
    if (B <= 0 || C <= 0 || F <= 0 || H <= 0 || W <= 0 || p <= 0) return ROPE3D_ERR_SHAPE;
    if (H % p != 0 || W % p != 0) return ROPE3D_ERR_SHAPE;
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (B * C > lim || B * C * F > lim || H > lim || W > lim || C * p * p > lim)
        return ROPE3D_ERR_SHAPE;
    const double total = double(B) * C * F * H * W * elem_bytes;
    if (total > 1.0e18) return ROPE3D_ERR_SHAPE;
    const uint64_t bytes = uint64_t(B) * C * F * H * W * elem_bytes;
    const uintptr_t s = reinterpret_cast<uintptr_t>(src), d = reinterpret_cast<uintptr_t>(dst);
    if (s % elem_bytes != 0 || d % elem_bytes != 0) return ROPE3D_ERR_ALIGN;
    if (s < d + bytes && d < s + bytes) return ROPE3D_ERR_ALIAS;
    const uint64_t units_per_plane_elem = uint64_t(H) * uint64_t(W);
    if (units_per_plane_elem > rope3d::kMaxUnitsPerLaunch) return ROPE3D_ERR_SHAPE;
    if (!check_device) return ROPE3D_OK;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return ROPE3D_ERR_CUDA;
    if (!device_ptr(src, device) || !device_ptr(dst, device)) return ROPE3D_ERR_DEVICE;

    const uint32_t V = 16 / elem_bytes;
    const uint32_t Wp = static_cast<uint32_t>(W / p);
    const bool vec = (p == 1 || p == 2 || p == 4 || p == 8) && Wp % V == 0 && s % 16 == 0 &&
                     d % 16 == 0;
    const PFn fn = forward ? pick<true>(elem_bytes, static_cast<uint32_t>(p), vec)
                           : pick<false>(elem_bytes, static_cast<uint32_t>(p), vec);
    if (!fn) return ROPE3D_ERR_ARG;
    const uint64_t units_per_row = vec ? Wp / V : uint64_t(W);

    PParams q{};
    q.src = static_cast<const char *>(src);
    q.dst = static_cast<char *>(dst);
    q.per_row = make_fastdiv(static_cast<uint32_t>(units_per_row));
    q.Hd = make_fastdiv(static_cast<uint32_t>(H));
    q.CF = make_fastdiv(static_cast<uint32_t>(C * F));
    q.Fd = make_fastdiv(static_cast<uint32_t>(F));
    q.pd = make_fastdiv(static_cast<uint32_t>(p));
    q.Wd = make_fastdiv(static_cast<uint32_t>(W));
    q.C = static_cast<uint32_t>(C);
    q.F = static_cast<uint32_t>(F);
    q.H = static_cast<uint32_t>(H);
    q.W = static_cast<uint32_t>(W);
    q.p = static_cast<uint32_t>(p);
    q.Hp = static_cast<uint32_t>(H / p);
    q.Wp = Wp;
    q.total = bytes;

    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return ROPE3D_ERR_CUDA;
    // launches cover whole (b, c, f) planes so that a launch's rows start at h = 0
    const uint64_t rows_per_plane = uint64_t(H);
    const uint64_t planes = uint64_t(B) * C * F;
    const uint64_t units_per_plane = rows_per_plane * units_per_row;
    // units_per_plane <= H * W <= 2^30 (checked above)
    const uint64_t planes_per_launch = rope3d::kMaxUnitsPerLaunch / units_per_plane;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (uint64_t p0 = 0; p0 < planes; p0 += planes_per_launch) {
        const uint64_t np = std::min(planes_per_launch, planes - p0);
        q.units = static_cast<uint32_t>(np * units_per_plane);
        q.bcf0 = static_cast<uint32_t>(p0);
        const uint64_t need = (uint64_t(q.units) + kThreads - 1) / kThreads;
        const int grid = static_cast<int>(std::min<uint64_t>(need, uint64_t(sms) * 8));
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kThreads);
        cfg.stream = st;
        cudaLaunchAttribute attr{};
        attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr.val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, fn, q) != cudaSuccess) {
            cudaGetLastError();
            return ROPE3D_ERR_CUDA;
        }
    }
    t_patch_kernel = vec ? 1 : 2;
    return ROPE3D_OK;
}

}  // namespace

namespace rope3d {

int64_t patchify_bound_errors(bool reset) {
#if ROPE3D_DEBUG_BOUNDS
    unsigned int n = 0;
    if (cudaMemcpyFromSymbol(&n, g_bound_errors, sizeof(n)) != cudaSuccess) return -1;
    if (reset) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_bound_errors, &zero, sizeof(zero)) != cudaSuccess) return -1;
    }
    return n;
#else
    (void)reset;
    return 0;
#endif
}

}  // namespace rope3d

extern "C" int rope3d_patchify(const void *x, void *y, int64_t B, int64_t C, int64_t F,
                               int64_t H, int64_t W, int64_t p, int32_t elem_bytes,
                               void *stream) {
    const int rc = run(true, x, y, B, C, F, H, W, p, elem_bytes, stream, false);
    if (rc != ROPE3D_OK) return rc;
    return run(true, x, y, B, C, F, H, W, p, elem_bytes, stream, true);
}

extern "C" int rope3d_unpatchify(const void *y, void *x, int64_t B, int64_t C, int64_t F,
                                 int64_t H, int64_t W, int64_t p, int32_t elem_bytes,
                                 void *stream) {
    const int rc = run(false, y, x, B, C, F, H, W, p, elem_bytes, stream, false);
    if (rc != ROPE3D_OK) return rc;
    return run(false, y, x, B, C, F, H, W, p, elem_bytes, stream, true);
}

extern "C" int rope3d_patchify_check(const void *src, const void *dst, int64_t B, int64_t C,
                                     int64_t F, int64_t H, int64_t W, int64_t p,
                                     int32_t elem_bytes) {
    return run(true, src, const_cast<void *>(dst), B, C, F, H, W, p, elem_bytes, nullptr, false);
}

extern "C" int rope3d_patchify_last_kernel(void) { return t_patch_kernel; }
