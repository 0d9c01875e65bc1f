// rope3d_neox.cu -- NeoX-style rotary embedding of the Gemma3 text encoder:
// rope3d_apply_neox and the cache builder rope3d_neox_cache_host.
//
// sglang PR #24660 review, "关键源码片段", gemma_3.py _apply_rotary_pos_emb:
// for each token, the row of a precomputed cos_sin_cache
// [max_position][rotary_dim] = [cos | sin] at the token's position is cast to
// the input dtype and duplicated over both halves of head_dim; then
//     q = q * cos + rotate_half(q) * sin,   rotate_half(x) = (-x2, x1)
// with x1, x2 the two halves of each head, evaluated as 16-bit tensor
// operations (every product rounded to the input dtype, every sum rounded to
// float and then to the input dtype). K takes the same rows; Q and K may have
// different head counts (grouped-query attention). rotary_dim = head_dim.
//
// One thread owns a 16-byte vector of channels j..j+V-1 in the first half of
// one head row and the matching vector j+d/2.. in the second half: two 16-byte
// loads, two 128-bit reads of the fp32 cache row (cos, sin), two 16-byte
// stores. Heads of one token are adjacent in the unit order, so the cache row
// (and the position) is read from L1 after the first head. Halves that are not
// a whole number of vectors take the per-pair kernel.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/rope3d.h"
#include "rope3d_internal.h"

namespace {

using rope3d::FastDiv;
using rope3d::make_fastdiv;

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) {
    return (__umulhi(n, f.mul) + n) >> f.shift;
}

struct NParams {
    const char *q;
    const char *k;
    char *q_out;
    char *k_out;
    const int64_t *positions;
    const float *cache;
    int *invalid;             // may be null
    uint64_t max_position;
    uint32_t units;           // work units of this launch
    uint32_t token0;          // first token of this launch
    FastDiv per_token;        // units per token: (q_heads + k_heads) * per_head
    FastDiv per_head;         // units per head row
    uint32_t q_heads, k_heads, head_dim, half;
    unsigned long long q_bytes, k_bytes;   // tensor sizes, for the debug bound checks
};

// Debug builds (-DROPE3D_DEBUG_BOUNDS=1) check each computed offset before the
// accesses it guards: a failed check counts in this file's error word and
// skips the unit (never a trap). Otherwise every check compiles away.
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

// ---- rounding to the storage type --------------------------------------------

template <int kType>
__device__ __forceinline__ float round_to(float f) {
    if constexpr (kType == ROPE3D_BF16) return __bfloat162float(__float2bfloat16_rn(f));
    else if constexpr (kType == ROPE3D_F16) return __half2float(__float2half_rn(f));
    else return f;
}

// (y1, y2) of one NeoX pair; c and s already cast to the storage type.
template <int kType>
__device__ __forceinline__ float2 neox_pair(float x1, float x2, float c, float s) {
    const float x1c = round_to<kType>(__fmul_rn(x1, c));
    const float x2c = round_to<kType>(__fmul_rn(x2, c));
    const float nx2s = round_to<kType>(__fmul_rn(-x2, s));
    const float x1s = round_to<kType>(__fmul_rn(x1, s));
    return make_float2(round_to<kType>(__fadd_rn(x1c, nx2s)), round_to<kType>(__fadd_rn(x2c, x1s)));
}

// 16-byte vector <-> floats
template <int kType>
__device__ __forceinline__ void unpack(const uint4 &v, float *f) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (kType == ROPE3D_F32) {
#pragma unroll
        for (int i = 0; i < 4; ++i) f[i] = __uint_as_float(w[i]);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (kType == ROPE3D_BF16) {
                f[2 * i] = __uint_as_float(w[i] << 16);
                f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            } else {
                __half2 h;
                memcpy(&h, &w[i], 4);
                const float2 t = __half22float2(h);
                f[2 * i] = t.x;
                f[2 * i + 1] = t.y;
            }
        }
    }
}

template <int kType>
__device__ __forceinline__ uint4 pack(const float *f) {
    uint32_t w[4];
    if constexpr (kType == ROPE3D_F32) {
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = __float_as_uint(f[i]);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (kType == ROPE3D_BF16) {
                const __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
                memcpy(&w[i], &b, 4);
            } else {
                const __half2 b = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
                memcpy(&w[i], &b, 4);
            }
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint4 ld_v4(const void *ptr) {
    uint4 r;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(ptr)
                 : "memory");
    return r;
}

__device__ __forceinline__ void st_v4(void *ptr, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};"
                 :
                 : "l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Locate unit u: token, head row (Q heads first, then K heads) and the first
// channel j of the unit in the first half. Returns 1 for an invalid position,
// 2 for an offset that fails a debug bound check, else 0.
struct Unit {
    const char *in;
    char *out;
    const float *row;   // cache row of the token's position
    uint32_t j;
};

template <int kElemBytes>
__device__ __forceinline__ int locate(const NParams &p, uint32_t u, uint32_t elems_per_unit,
                                      Unit *x) {
    const uint32_t tl = fdiv(u, p.per_token);
    const uint32_t r = u - tl * p.per_token.d;
    const uint32_t hrow = fdiv(r, p.per_head);
    const uint32_t g = r - hrow * p.per_head.d;
    const uint64_t token = uint64_t(p.token0) + tl;
    const int64_t pos = __ldg(p.positions + token);
    if (pos < 0 || uint64_t(pos) >= p.max_position) return 1;
    const bool is_q = hrow < p.q_heads;
    const uint32_t h = is_q ? hrow : hrow - p.q_heads;
    const uint64_t heads = is_q ? p.q_heads : p.k_heads;
    const uint64_t off = ((token * heads + h) * p.head_dim) * kElemBytes;
    if (!bound_ok(off, uint64_t(p.head_dim) * kElemBytes, is_q ? p.q_bytes : p.k_bytes) ||
        !bound_ok(uint64_t(pos) * p.head_dim * 4, uint64_t(p.head_dim) * 4,
                  p.max_position * p.head_dim * 4))
        return 2;
    x->in = (is_q ? p.q : p.k) + off;
    x->out = (is_q ? p.q_out : p.k_out) + off;
    x->row = p.cache + uint64_t(pos) * p.head_dim;
    x->j = g * elems_per_unit;
    return 0;
}

// Packed 16-bit form of neox_pair for two adjacent channels. Every operation
// is one correctly rounded 16-bit multiply or add; this equals the float
// evaluation above (product exact in float, then rounded; sum rounded to float
// and then to 16 bits) because float's 24-bit significand is at least
// 2p + 2 for p = 8 (bf16) and p = 11 (fp16), which makes the double rounding
// innocuous (Figueroa, "When is double rounding innocuous?", SIGNUM 1995).
template <typename T2>
__device__ __forceinline__ void neox_pair2(T2 x1, T2 x2, T2 c, T2 s, T2 *y1, T2 *y2) {
    const T2 x1c = __hmul2(x1, c);
    const T2 x2c = __hmul2(x2, c);
    const T2 nx2s = __hmul2(__hneg2(x2), s);
    const T2 x1s = __hmul2(x1, s);
    *y1 = __hadd2(x1c, nx2s);
    *y2 = __hadd2(x2c, x1s);
}

template <int kType>
struct Pack2;
template <>
struct Pack2<ROPE3D_BF16> {
    using T2 = __nv_bfloat162;
    static __device__ __forceinline__ T2 from_floats(float a, float b) { return __floats2bfloat162_rn(a, b); }
};
template <>
struct Pack2<ROPE3D_F16> {
    using T2 = __half2;
    static __device__ __forceinline__ T2 from_floats(float a, float b) { return __floats2half2_rn(a, b); }
};

// Programmatic dependent launch: a kernel lets the next kernel of the stream
// start launching at once, and waits for the grids before it to complete (and
// their writes to become visible) before it touches memory, so back-to-back
// launches overlap one kernel's tail with the next one's launch. Launched
// without the attribute, both instructions return at once.
__device__ __forceinline__ void pdl_begin() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int kType>
__global__ void __launch_bounds__(kThreads)
rope3d_neox_vec_kernel(const NParams p) {
    constexpr int kElemBytes = kType == ROPE3D_F32 ? 4 : 2;
    constexpr int V = 16 / kElemBytes;   // channels per vector
    pdl_begin();
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < p.units; u += stride) {
        Unit x;
        if (const int bad = locate<kElemBytes>(p, u, V, &x)) {
            if (bad == 1 && p.invalid) atomicAdd(p.invalid, 1);
            continue;
        }
        const uint4 a = ld_v4(x.in + size_t(x.j) * kElemBytes);
        const uint4 b = ld_v4(x.in + size_t(x.j + p.half) * kElemBytes);
        float c[V], s[V];
#pragma unroll
        for (int i = 0; i < V; i += 4) {
            const float4 cv = __ldg(reinterpret_cast<const float4 *>(x.row + x.j + i));
            const float4 sv = __ldg(reinterpret_cast<const float4 *>(x.row + p.half + x.j + i));
            c[i] = cv.x; c[i + 1] = cv.y; c[i + 2] = cv.z; c[i + 3] = cv.w;
            s[i] = sv.x; s[i + 1] = sv.y; s[i + 2] = sv.z; s[i + 3] = sv.w;
        }
        if constexpr (kType == ROPE3D_F32) {
            float x1[V], x2[V], y1[V], y2[V];
            unpack<kType>(a, x1);
            unpack<kType>(b, x2);
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const float2 y = neox_pair<kType>(x1[i], x2[i], c[i], s[i]);
                y1[i] = y.x;
                y2[i] = y.y;
            }
            st_v4(x.out + size_t(x.j) * kElemBytes, pack<kType>(y1));
            st_v4(x.out + size_t(x.j + p.half) * kElemBytes, pack<kType>(y2));
        } else {
            using T2 = typename Pack2<kType>::T2;
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
            const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
            uint32_t y1w[4], y2w[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                T2 x1, x2, y1, y2;
                memcpy(&x1, &aw[w], 4);
                memcpy(&x2, &bw[w], 4);
                // cos.to(dtype), sin.to(dtype): round to nearest, two at a time
                const T2 c2 = Pack2<kType>::from_floats(c[2 * w], c[2 * w + 1]);
                const T2 s2 = Pack2<kType>::from_floats(s[2 * w], s[2 * w + 1]);
                neox_pair2(x1, x2, c2, s2, &y1, &y2);
                memcpy(&y1w[w], &y1, 4);
                memcpy(&y2w[w], &y2, 4);
            }
            st_v4(x.out + size_t(x.j) * kElemBytes, make_uint4(y1w[0], y1w[1], y1w[2], y1w[3]));
            st_v4(x.out + size_t(x.j + p.half) * kElemBytes, make_uint4(y2w[0], y2w[1], y2w[2], y2w[3]));
        }
    }
}

template <int kType>
__global__ void __launch_bounds__(kThreads)
rope3d_neox_pair_kernel(const NParams p) {
    constexpr int kElemBytes = kType == ROPE3D_F32 ? 4 : 2;
    pdl_begin();
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < p.units; u += stride) {
        Unit x;
        if (const int bad = locate<kElemBytes>(p, u, 1, &x)) {
            if (bad == 1 && p.invalid) atomicAdd(p.invalid, 1);
            continue;
        }
        const char *a = x.in + size_t(x.j) * kElemBytes;
        const char *b = x.in + size_t(x.j + p.half) * kElemBytes;
        float x1, x2;
        if constexpr (kType == ROPE3D_F32) {
            x1 = *reinterpret_cast<const volatile float *>(a);
            x2 = *reinterpret_cast<const volatile float *>(b);
        } else {
            const uint16_t ha = *reinterpret_cast<const volatile uint16_t *>(a);
            const uint16_t hb = *reinterpret_cast<const volatile uint16_t *>(b);
            if constexpr (kType == ROPE3D_BF16) {
                x1 = __uint_as_float(uint32_t(ha) << 16);
                x2 = __uint_as_float(uint32_t(hb) << 16);
            } else {
                x1 = __half2float(__ushort_as_half(ha));
                x2 = __half2float(__ushort_as_half(hb));
            }
        }
        const float c = round_to<kType>(__ldg(x.row + x.j));
        const float s = round_to<kType>(__ldg(x.row + p.half + x.j));
        const float2 y = neox_pair<kType>(x1, x2, c, s);
        char *oa = x.out + size_t(x.j) * kElemBytes;
        char *ob = x.out + size_t(x.j + p.half) * kElemBytes;
        if constexpr (kType == ROPE3D_F32) {
            *reinterpret_cast<float *>(oa) = y.x;
            *reinterpret_cast<float *>(ob) = y.y;
        } else if constexpr (kType == ROPE3D_BF16) {
            *reinterpret_cast<uint16_t *>(oa) = __bfloat16_as_ushort(__float2bfloat16_rn(y.x));
            *reinterpret_cast<uint16_t *>(ob) = __bfloat16_as_ushort(__float2bfloat16_rn(y.y));
        } else {
            *reinterpret_cast<uint16_t *>(oa) = __half_as_ushort(__float2half_rn(y.x));
            *reinterpret_cast<uint16_t *>(ob) = __half_as_ushort(__float2half_rn(y.y));
        }
    }
}

using NFn = void (*)(NParams);

NFn pick(int dtype, bool vec) {
    switch (dtype) {
        case ROPE3D_BF16: return vec ? rope3d_neox_vec_kernel<ROPE3D_BF16> : rope3d_neox_pair_kernel<ROPE3D_BF16>;
        case ROPE3D_F16: return vec ? rope3d_neox_vec_kernel<ROPE3D_F16> : rope3d_neox_pair_kernel<ROPE3D_F16>;
        default: return vec ? rope3d_neox_vec_kernel<ROPE3D_F32> : rope3d_neox_pair_kernel<ROPE3D_F32>;
    }
}

bool on_device(const void *p, int device) {
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (attr.type == cudaMemoryTypeManaged) return true;
    return attr.type == cudaMemoryTypeDevice && attr.device == device;
}

bool overlap(uintptr_t a, uint64_t na, uintptr_t b, uint64_t nb) { return a < b + nb && b < a + na; }

thread_local int t_neox_kernel = 0;

int neox(const void *q, const void *k, void *q_out, void *k_out, const int64_t *positions,
         const float *cache, int64_t max_position, int64_t tokens, int64_t q_heads,
         int64_t k_heads, int64_t head_dim, int32_t dtype, int32_t *invalid, void *stream,
         bool launch) {
    if (!q || !k || !q_out || !k_out || !positions || !cache) return ROPE3D_ERR_NULL;
    if (dtype != ROPE3D_BF16 && dtype != ROPE3D_F16 && dtype != ROPE3D_F32) return ROPE3D_ERR_DTYPE;
    if (tokens <= 0 || q_heads <= 0 || k_heads <= 0 || head_dim <= 0 || max_position <= 0 ||
        head_dim % 2 != 0 || head_dim > ROPE3D_MAX_HEAD_DIM || q_heads > 65536 || k_heads > 65536 ||
        tokens > (int64_t(1) << 40) || max_position > (int64_t(1) << 40))
        return ROPE3D_ERR_SHAPE;
    const int64_t es = dtype == ROPE3D_F32 ? 4 : 2;
    const uintptr_t P[7] = {reinterpret_cast<uintptr_t>(q), reinterpret_cast<uintptr_t>(k),
                            reinterpret_cast<uintptr_t>(q_out), reinterpret_cast<uintptr_t>(k_out),
                            reinterpret_cast<uintptr_t>(positions), reinterpret_cast<uintptr_t>(cache),
                            reinterpret_cast<uintptr_t>(invalid)};
    for (int i = 0; i < 4; ++i)
        if (P[i] % 4 != 0) return ROPE3D_ERR_ALIGN;
    if (P[4] % 8 != 0 || P[5] % 4 != 0 || P[6] % 4 != 0) return ROPE3D_ERR_ALIGN;
    const uint64_t qb = uint64_t(tokens) * q_heads * head_dim * es;
    const uint64_t kb = uint64_t(tokens) * k_heads * head_dim * es;
    const uint64_t pb = uint64_t(tokens) * 8, cb = uint64_t(max_position) * head_dim * 4;
    // outputs: an output is its own input exactly (in place) or disjoint from
    // it, and never overlaps the other input or the other output (a Q output
    // written in place over K's memory would be read back by the K units)
    const bool q_in_place = P[2] == P[0], k_in_place = P[3] == P[1];
    if ((!q_in_place && overlap(P[2], qb, P[0], qb)) || overlap(P[2], qb, P[1], kb) ||
        (!k_in_place && overlap(P[3], kb, P[1], kb)) || overlap(P[3], kb, P[0], qb) ||
        overlap(P[2], qb, P[3], kb))
        return ROPE3D_ERR_ALIAS;
    for (int o = 2; o < 4; ++o) {
        const uint64_t ob = o == 2 ? qb : kb;
        if (overlap(P[o], ob, P[4], pb) || overlap(P[o], ob, P[5], cb) ||
            (invalid && overlap(P[o], ob, P[6], 4)))
            return ROPE3D_ERR_ALIAS;
    }
    if (!launch) return ROPE3D_OK;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return ROPE3D_ERR_CUDA;
    for (int i = 0; i < 6; ++i)
        if (!on_device(reinterpret_cast<const void *>(P[i]), device)) return ROPE3D_ERR_DEVICE;
    if (invalid && !on_device(invalid, device)) return ROPE3D_ERR_DEVICE;

    const uint32_t half = static_cast<uint32_t>(head_dim / 2);
    const uint32_t V = static_cast<uint32_t>(16 / es);
    // vectors: whole 16-byte runs in each half, and 16-byte aligned cache rows
    bool vec = half % V == 0 && P[5] % 16 == 0;
    for (int i = 0; i < 4; ++i) vec = vec && P[i] % 16 == 0;
    const uint32_t per_head = vec ? half / V : half;
    const uint64_t per_token = uint64_t(q_heads + k_heads) * per_head;
    if (per_token > rope3d::kMaxUnitsPerLaunch) return ROPE3D_ERR_SHAPE;
    NParams p{};
    p.q = static_cast<const char *>(q);
    p.k = static_cast<const char *>(k);
    p.q_out = static_cast<char *>(q_out);
    p.k_out = static_cast<char *>(k_out);
    p.positions = positions;
    p.cache = cache;
    p.invalid = invalid;
    p.max_position = static_cast<uint64_t>(max_position);
    p.per_token = make_fastdiv(static_cast<uint32_t>(per_token));
    p.per_head = make_fastdiv(per_head);
    p.q_heads = static_cast<uint32_t>(q_heads);
    p.k_heads = static_cast<uint32_t>(k_heads);
    p.head_dim = static_cast<uint32_t>(head_dim);
    p.half = half;
    p.q_bytes = static_cast<unsigned long long>(tokens) * q_heads * head_dim * es;
    p.k_bytes = static_cast<unsigned long long>(tokens) * k_heads * head_dim * es;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return ROPE3D_ERR_CUDA;
    const NFn fn = pick(dtype, vec);
    const uint64_t tokens_per_launch = rope3d::kMaxUnitsPerLaunch / per_token;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    for (uint64_t t0 = 0; t0 < uint64_t(tokens); t0 += tokens_per_launch) {
        const uint64_t nt = std::min<uint64_t>(tokens_per_launch, uint64_t(tokens) - t0);
        if (t0 > 0xffffffffull) return ROPE3D_ERR_SHAPE;
        p.token0 = static_cast<uint32_t>(t0);
        p.units = static_cast<uint32_t>(nt * per_token);
        const uint64_t need = (uint64_t(p.units) + kThreads - 1) / kThreads;
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
        if (cudaLaunchKernelEx(&cfg, fn, p) != cudaSuccess) {
            cudaGetLastError();
            return ROPE3D_ERR_CUDA;
        }
    }
    t_neox_kernel = vec ? 1 : 2;
    return ROPE3D_OK;
}

}  // namespace

namespace rope3d {

int64_t neox_bound_errors(bool reset) {
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

extern "C" int rope3d_apply_neox(const void *q, const void *k, void *q_out, void *k_out,
                                 const int64_t *positions, const float *cos_sin_cache,
                                 int64_t max_position, int64_t tokens, int64_t q_heads,
                                 int64_t k_heads, int64_t head_dim, int32_t dtype,
                                 int32_t *invalid_count, void *stream) {
    return neox(q, k, q_out, k_out, positions, cos_sin_cache, max_position, tokens, q_heads,
                k_heads, head_dim, dtype, invalid_count, stream, true);
}

extern "C" int rope3d_neox_check(const void *q, const void *k, const void *q_out,
                                 const void *k_out, const int64_t *positions,
                                 const float *cos_sin_cache, int64_t max_position, int64_t tokens,
                                 int64_t q_heads, int64_t k_heads, int64_t head_dim, int32_t dtype,
                                 const int32_t *invalid_count) {
    return neox(q, k, const_cast<void *>(q_out), const_cast<void *>(k_out), positions,
                cos_sin_cache, max_position, tokens, q_heads, k_heads, head_dim, dtype,
                const_cast<int32_t *>(invalid_count), nullptr, false);
}

extern "C" int rope3d_neox_cache_host(int64_t max_position, int64_t rotary_dim, double base,
                                      float *cache) {
    if (!cache) return ROPE3D_ERR_NULL;
    if (max_position <= 0 || rotary_dim <= 0 || rotary_dim % 2 != 0) return ROPE3D_ERR_SHAPE;
    if (!(std::isfinite(base) && base > 0.0)) return ROPE3D_ERR_ARG;
    const int64_t half = rotary_dim / 2;
    for (int64_t p = 0; p < max_position; ++p)
        for (int64_t j = 0; j < half; ++j) {
            const double inv_freq = std::pow(base, -(2.0 * static_cast<double>(j)) /
                                                       static_cast<double>(rotary_dim));
            const double angle = static_cast<double>(p) * inv_freq;
            cache[p * rotary_dim + j] = static_cast<float>(std::cos(angle));
            cache[p * rotary_dim + half + j] = static_cast<float>(std::sin(angle));
        }
    return ROPE3D_OK;
}

extern "C" int rope3d_neox_last_kernel(void) { return t_neox_kernel; }
