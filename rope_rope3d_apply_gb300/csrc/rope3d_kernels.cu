// rope3d_kernels.cu -- the sm_103a kernels of the fused paired 3D RoPE.
//
// The arithmetic follows the sglang PR #35698 review ("fused LTX-2.5 decoder
// 3D RoPE"), section "关键源码片段", the rotate_pair helper of
// ltx25_decoder_rope.cuh: each (even, odd) pair is widened to float32 and
// rotated with four separately rounded products, one rounded subtract and one
// rounded add (even*cos - odd*sin, even*sin + odd*cos), then cast back to the
// input type. __fmul_rn / __fsub_rn / __fadd_rn are never contracted into a
// fused multiply-add, which keeps the result bit-identical to the eager order.
//
// What differs from that kernel (which decodes one pair per thread with 64-bit
// division and reads cos/sin with __ldg):
//   * one thread owns a 16-byte vector of Q and the same vector of K (8 bf16 or
//     fp16 = 4 pairs, or 4 fp32 = 2 pairs), loaded with streaming 128-bit loads
//     that bypass L1, and stores the two results with evict-first 128-bit stores;
//   * the three axis tables are staged once per CTA into shared memory as
//     interleaved (cos, sin) float2 entries, so the 4 pairs of a vector read
//     their 4 table entries with two 128-bit shared loads;
//   * the grid is persistent (a multiple of the SM count times the resident
//     CTAs per SM) and strides over vectors, two vectors in flight per thread
//     and tensor;
//   * (row, head, vector-in-head) and the grid coordinates (t, h, w) come from
//     32-bit multiply-high divisions by precomputed constants.
// Inputs that cannot take 16-byte vectors (unaligned pointers, chunks that
// are not a multiple of the vector) run the per-pair kernel, same arithmetic.
// Strided views (Q and K taken straight out of a fused QKV buffer, a crop of a
// larger grid, or rotation in place) run the strided variants of both kernels:
// same arithmetic, addresses from per-tensor (batch, t, h, w, head) strides,
// and loads through the coherent path so that in-place rotation is safe.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "../../include/rope3d.h"
#include "rope3d_internal.h"

namespace rope3d {
namespace {

// Threads per CTA and vectors of Q (and of K) in flight per thread in the
// contiguous vector kernel (compile-time, overridable for tuning sweeps).
#ifndef ROPE3D_BLOCK
#define ROPE3D_BLOCK 512
#endif
#ifndef ROPE3D_UNROLL
#define ROPE3D_UNROLL 2
#endif
constexpr int kBlock = ROPE3D_BLOCK;
constexpr int kUnroll = ROPE3D_UNROLL;
#ifdef ROPE3D_MIN_CTAS
#define ROPE3D_VEC_BOUNDS __launch_bounds__(kBlock, ROPE3D_MIN_CTAS)
#else
#define ROPE3D_VEC_BOUNDS __launch_bounds__(kBlock)
#endif

// Strided vector kernel: threads per CTA, vectors per tensor in flight per
// thread, and the resident CTAs per SM its register budget is sized for. At
// its 43-44 registers, 384 threads fit three CTAs per SM (1,152 threads) where
// 512 fit two; measured on a fused QKV buffer rotated in place, 384 x 2 was
// the fastest of 256-1,024 threads and 2-4 vectors.
#ifndef ROPE3D_STRIDED_BLOCK
#define ROPE3D_STRIDED_BLOCK 384
#endif
#ifndef ROPE3D_STRIDED_UNROLL
#define ROPE3D_STRIDED_UNROLL 2
#endif
#ifndef ROPE3D_STRIDED_MIN_CTAS
#define ROPE3D_STRIDED_MIN_CTAS 0
#endif
constexpr int kStridedBlock = ROPE3D_STRIDED_BLOCK;
constexpr int kStridedUnroll = ROPE3D_STRIDED_UNROLL;
#if ROPE3D_STRIDED_MIN_CTAS > 0
#define ROPE3D_STRIDED_BOUNDS __launch_bounds__(kStridedBlock, ROPE3D_STRIDED_MIN_CTAS)
#else
#define ROPE3D_STRIDED_BOUNDS __launch_bounds__(kStridedBlock)
#endif

// Tables of the contiguous vector kernel up to this many bytes are staged in
// shared memory; larger ones are read through the read-only (L1) path.
#ifndef ROPE3D_VEC_SMEM_TABLE_MAX
#define ROPE3D_VEC_SMEM_TABLE_MAX (96 * 1024)
#endif
// Resident CTAs per SM the contiguous vector kernel's grid is sized for
// (0: as many as fit). Fewer than fit leave room for the next kernel of the
// stream to become resident while this one still runs.
#ifndef ROPE3D_VEC_GRID_CTAS
#define ROPE3D_VEC_GRID_CTAS 0
#endif
// 1: the contiguous vector kernel asks L2 for each thread's first vectors of
// Q and K before it waits for the previous grid of the stream.
#ifndef ROPE3D_PREFETCH_FIRST
#define ROPE3D_PREFETCH_FIRST 0
#endif

struct KParams {
    const void *q;
    const void *k;
    void *q_out;
    void *k_out;
    const float2 *tab;
    uint32_t tab_len;
    uint32_t offH, offW;
    uint32_t pT, pH, pW;
    uint32_t units;         // vectors (or pairs) in this launch
    FastDiv per_row;        // units per (batch, token) row
    FastDiv per_head;       // units per head
    FastDiv N, HW, Wd;      // T*H*W, H*W, W
    uint32_t row0_mod_N;    // first row of this launch, modulo N
};

// Element strides of (batch, t, h, w, head) for Q, K, Q_out, K_out, and the
// batch index of the launch's first row (strided kernels only); lim: the bytes
// each of the four buffers spans from its pointer, for the bounds checks of
// debug builds.
struct KStrides {
    long long s[4][5];
    uint32_t b0;
    unsigned long long lim[4];
};

// Debug builds (-DROPE3D_DEBUG_BOUNDS=1) check each computed index before the
// access it guards: a failed check adds one to this file's error word and
// skips the access (never a trap); rope3d_debug_bounds() reads the words.
// Without the flag every check is `true` and compiles away.
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

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) {
    return (__umulhi(n, f.mul) + n) >> f.shift;
}

// Grid coordinates of row `row` of the launch: token (t, h, w) and the batch
// offset from the launch's first batch.
struct GridPos {
    uint32_t t, h, w, db;
};

__device__ __forceinline__ GridPos grid_pos(const KParams &p, uint32_t row) {
    const uint32_t q = fdiv(row, p.N);
    uint32_t tok = row - q * p.N.d + p.row0_mod_N;
    const uint32_t carry = tok >= p.N.d ? 1u : 0u;
    tok -= carry * p.N.d;
    GridPos g;
    g.t = fdiv(tok, p.HW);
    const uint32_t rem = tok - g.t * p.HW.d;
    g.h = fdiv(rem, p.Wd);
    g.w = rem - g.h * p.Wd.d;
    g.db = q + carry;
    return g;
}

// Entry index of the table entry for pair `pair_in_head` at grid position g.
__device__ __forceinline__ uint32_t table_index(const KParams &p, const GridPos &g,
                                                uint32_t pair_in_head) {
    const uint32_t it = g.t * p.pT + pair_in_head;
    const uint32_t ih = p.offH + g.h * p.pH + (pair_in_head - p.pT);
    const uint32_t iw = p.offW + g.w * p.pW + (pair_in_head - p.pT - p.pH);
    return pair_in_head < p.pT ? it : (pair_in_head < p.pT + p.pH ? ih : iw);
}

// Element offset of (row at g, head, channel) in tensor i of a strided call.
__device__ __forceinline__ long long strided_offset(const KStrides &st, int i, const GridPos &g,
                                                    uint32_t head, uint32_t channel) {
    const long long *s = st.s[i];
    return (long long)(st.b0 + g.db) * s[0] + (long long)g.t * s[1] + (long long)g.h * s[2] +
           (long long)g.w * s[3] + (long long)head * s[4] + channel;
}

// ---- memory access ---------------------------------------------------------

// Read-only streaming load (inputs never alias outputs in contiguous calls).
__device__ __forceinline__ uint4 ld_stream_v4(const void *ptr) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::128B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(ptr));
    return r;
}

// Coherent streaming load (strided calls, which may rotate in place).
// The asm is volatile so that it is never moved past the stores of the
// previous iteration, which may write the same buffer (in place).
__device__ __forceinline__ uint4 ld_coherent_v4(const void *ptr) {
    uint4 r;
    asm volatile("ld.global.L1::no_allocate.L2::128B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(ptr)
                 : "memory");
    return r;
}

__device__ __forceinline__ void st_stream_v4(void *ptr, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};"
                 :
                 : "l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_nc_u32(const void *ptr) {
    uint32_t r;
    asm("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(ptr));
    return r;
}

// ---- the pair rotation (eager order, no fused multiply-add) ----------------

struct Rot {
    float y0, y1;
};

__device__ __forceinline__ Rot rotate(float even, float odd, float c, float s) {
    const float even_cos = __fmul_rn(even, c);
    const float odd_sin = __fmul_rn(odd, s);
    const float even_sin = __fmul_rn(even, s);
    const float odd_cos = __fmul_rn(odd, c);
    return Rot{__fsub_rn(even_cos, odd_sin), __fadd_rn(even_sin, odd_cos)};
}

// One 32-bit word holding a 16-bit pair: the even element is the low half
// (lower address). bf16 -> f32 widening is a 16-bit shift; binary16 is widened
// exactly by the conversion instruction. Both narrow to nearest, ties to even.
template <int kType>
__device__ __forceinline__ uint32_t rotate_word16(uint32_t word, float c, float s) {
    float even, odd;
    if constexpr (kType == ROPE3D_BF16) {
        even = __uint_as_float(word << 16);
        odd = __uint_as_float(word & 0xffff0000u);
    } else {
        __half2 h;
        memcpy(&h, &word, sizeof h);
        const float2 f = __half22float2(h);
        even = f.x;
        odd = f.y;
    }
    const Rot r = rotate(even, odd, c, s);
    uint32_t out;
    if constexpr (kType == ROPE3D_BF16) {
        const __nv_bfloat162 packed = __floats2bfloat162_rn(r.y0, r.y1);  // .x = y0 (low)
        memcpy(&out, &packed, sizeof out);
    } else {
        const __half2 packed = __floats2half2_rn(r.y0, r.y1);  // .x = y0 (low)
        memcpy(&out, &packed, sizeof out);
    }
    return out;
}

template <int kType>
__device__ __forceinline__ uint4 rotate_vec(const uint4 v, const float4 cs01, const float4 cs23) {
    uint4 o;
    if constexpr (kType != ROPE3D_F32) {
        // 8 16-bit elements = 4 pairs; entries (c0, s0, c1, s1) and (c2, s2, c3, s3)
        o.x = rotate_word16<kType>(v.x, cs01.x, cs01.y);
        o.y = rotate_word16<kType>(v.y, cs01.z, cs01.w);
        o.z = rotate_word16<kType>(v.z, cs23.x, cs23.y);
        o.w = rotate_word16<kType>(v.w, cs23.z, cs23.w);
    } else {
        // 4 fp32 = 2 pairs; entries (c0, s0, c1, s1)
        const Rot a = rotate(__uint_as_float(v.x), __uint_as_float(v.y), cs01.x, cs01.y);
        const Rot b = rotate(__uint_as_float(v.z), __uint_as_float(v.w), cs01.z, cs01.w);
        o.x = __float_as_uint(a.y0);
        o.y = __float_as_uint(a.y1);
        o.z = __float_as_uint(b.y0);
        o.w = __float_as_uint(b.y1);
        (void)cs23;
    }
    return o;
}

// Programmatic dependent launch. A kernel launched with programmatic stream
// serialization may start while the previous kernel in the stream finishes:
// it lets its own successor launch early, stages the tables (which no kernel
// writes), and only then waits until every earlier grid has completed and its
// writes are visible, before it touches Q, K or the outputs. Launched without
// that attribute, both instructions return at once.
__device__ __forceinline__ void allow_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void wait_for_prerequisite_grids() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Stages the tables (kSmem) and waits for the earlier grids; the caller has
// already let its successor launch.
template <bool kSmem>
__device__ __forceinline__ const float2 *stage_tables_then_wait(const KParams &p, float2 *smem) {
    if constexpr (kSmem) {
        for (uint32_t i = threadIdx.x; i < p.tab_len; i += blockDim.x) smem[i] = __ldg(p.tab + i);
        __syncthreads();
    }
    wait_for_prerequisite_grids();
    return kSmem ? smem : p.tab;
}

template <bool kSmem>
__device__ __forceinline__ const float2 *stage_tables(const KParams &p, float2 *smem) {
    allow_dependents_launch();
    return stage_tables_then_wait<kSmem>(p, smem);
}

// A hint that moves the 128-byte line holding ptr into L2. It carries no
// memory-model meaning: L2 is where every SM of the GPU sees global memory, so
// a line fetched before an earlier grid writes it is updated there by that
// write, and a load after griddepcontrol.wait reads the written value.
__device__ __forceinline__ void prefetch_l2(const void *ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

template <bool kSmem>
__device__ __forceinline__ float4 tab4(const float2 *tab, uint32_t idx, uint32_t len) {
    // idx is a multiple of 2 entries: one 16-byte load of two (cos, sin) entries
    if (!bound_ok(idx, 2, len)) return make_float4(0.f, 0.f, 0.f, 0.f);
    if constexpr (kSmem) {
        return *reinterpret_cast<const float4 *>(tab + idx);
    } else {
        return __ldg(reinterpret_cast<const float4 *>(tab + idx));
    }
}

template <bool kSmem>
__device__ __forceinline__ float2 tab1(const float2 *tab, uint32_t idx, uint32_t len) {
    if (!bound_ok(idx, 1, len)) return make_float2(0.f, 0.f);
    if constexpr (kSmem) {
        return tab[idx];
    } else {
        return __ldg(tab + idx);
    }
}

// ---- 16-byte vector kernel, contiguous buffers -----------------------------
// Requires: 16-byte aligned pointers, head_dim and each chunk a multiple of the
// vector's element count (so a vector never straddles a chunk, head or row, and
// the first table entry of a vector is a multiple of 4 (16-bit) or 2 (fp32)).

template <int kType, bool kSmem>
__global__ void ROPE3D_VEC_BOUNDS
rope3d_vec16_kernel(const KParams p, const KStrides) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr uint32_t kPairsPerVec = kType == ROPE3D_F32 ? 2 : 4;

    const uint4 *q = static_cast<const uint4 *>(p.q);
    const uint4 *k = static_cast<const uint4 *>(p.k);
    uint4 *qo = static_cast<uint4 *>(p.q_out);
    uint4 *ko = static_cast<uint4 *>(p.k_out);

    const uint32_t stride = gridDim.x * blockDim.x;
    uint32_t v = blockIdx.x * blockDim.x + threadIdx.x;

    allow_dependents_launch();
    if constexpr (ROPE3D_PREFETCH_FIRST != 0) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            if (v + u * stride < p.units) {
                prefetch_l2(q + v + u * stride);
                prefetch_l2(k + v + u * stride);
            }
        }
    }
    const float2 *tab = stage_tables_then_wait<kSmem>(p, reinterpret_cast<float2 *>(smem_raw));

    // main loop: kUnroll vectors of Q and of K in flight per thread
    for (; v + (kUnroll - 1) * stride < p.units; v += kUnroll * stride) {
        uint4 qv[kUnroll], kv[kUnroll];
        uint32_t idx[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            qv[u] = ld_stream_v4(q + v + u * stride);
            kv[u] = ld_stream_v4(k + v + u * stride);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint32_t vv = v + u * stride;
            const uint32_t row = fdiv(vv, p.per_row);
            const uint32_t r = vv - row * p.per_row.d;
            const uint32_t g = r - fdiv(r, p.per_head) * p.per_head.d;
            idx[u] = table_index(p, grid_pos(p, row), g * kPairsPerVec);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const float4 cs01 = tab4<kSmem>(tab, idx[u], p.tab_len);
            const float4 cs23 = kType != ROPE3D_F32 ? tab4<kSmem>(tab, idx[u] + 2, p.tab_len) : cs01;
            st_stream_v4(qo + v + u * stride, rotate_vec<kType>(qv[u], cs01, cs23));
            st_stream_v4(ko + v + u * stride, rotate_vec<kType>(kv[u], cs01, cs23));
        }
    }
    // ragged tail: at most kUnroll - 1 more vectors per thread
    for (; v < p.units; v += stride) {
        const uint4 qv = ld_stream_v4(q + v);
        const uint4 kv = ld_stream_v4(k + v);
        const uint32_t row = fdiv(v, p.per_row);
        const uint32_t r = v - row * p.per_row.d;
        const uint32_t g = r - fdiv(r, p.per_head) * p.per_head.d;
        const uint32_t i = table_index(p, grid_pos(p, row), g * kPairsPerVec);
        const float4 cs01 = tab4<kSmem>(tab, i, p.tab_len);
        const float4 cs23 = kType != ROPE3D_F32 ? tab4<kSmem>(tab, i + 2, p.tab_len) : cs01;
        st_stream_v4(qo + v, rotate_vec<kType>(qv, cs01, cs23));
        st_stream_v4(ko + v, rotate_vec<kType>(kv, cs01, cs23));
    }
}

// ---- 16-byte vector kernel, strided views ----------------------------------
// Requires, besides the contiguous kernel's conditions, every stride a multiple
// of the vector's element count.

template <int kType, bool kSmem, bool kSame>
__global__ void ROPE3D_STRIDED_BOUNDS
rope3d_vec16_strided_kernel(const KParams p, const KStrides st) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const float2 *tab = stage_tables<kSmem>(p, reinterpret_cast<float2 *>(smem_raw));
    constexpr uint32_t kPairsPerVec = kType == ROPE3D_F32 ? 2 : 4;
    constexpr uint32_t kElemsPerVec = 2 * kPairsPerVec;
    constexpr int kElemBytes = kType == ROPE3D_F32 ? 4 : 2;

    const char *q = static_cast<const char *>(p.q);
    const char *k = static_cast<const char *>(p.k);
    char *qo = static_cast<char *>(p.q_out);
    char *ko = static_cast<char *>(p.k_out);

    // kSame: the four views share one set of strides (e.g. Q and K of a fused
    // QKV buffer rotated in place), so one offset serves all four pointers
    auto off = [&](int i, const GridPos &pos, uint32_t head, uint32_t c) {
        return strided_offset(st, kSame ? 0 : i, pos, head, c) * kElemBytes;
    };

    // position of vector vv: grid coordinates, head, and its first channel
    struct Where {
        GridPos pos;
        uint32_t head, g;
    };
    auto where = [&](uint32_t vv) {
        Where x;
        const uint32_t row = fdiv(vv, p.per_row);
        const uint32_t r = vv - row * p.per_row.d;
        x.head = fdiv(r, p.per_head);
        x.g = r - x.head * p.per_head.d;
        x.pos = grid_pos(p, row);
        return x;
    };

    const uint32_t stride = gridDim.x * blockDim.x;
    uint32_t v = blockIdx.x * blockDim.x + threadIdx.x;
    // main loop: kStridedUnroll vectors of Q and of K in flight per thread; all loads
    // of an iteration come before its stores, and no two threads touch one
    // element, so rotating in place is safe
    for (; v + (kStridedUnroll - 1) * stride < p.units; v += kStridedUnroll * stride) {
        Where x[kStridedUnroll];
        uint4 qv[kStridedUnroll], kv[kStridedUnroll];
#pragma unroll
        for (int u = 0; u < kStridedUnroll; ++u) {
            x[u] = where(v + u * stride);
            const uint32_t c = x[u].g * kElemsPerVec;
            const long long oq = off(0, x[u].pos, x[u].head, c), ok = off(1, x[u].pos, x[u].head, c);
            qv[u] = bound_ok(oq, 16, st.lim[0]) ? ld_coherent_v4(q + oq) : make_uint4(0, 0, 0, 0);
            kv[u] = bound_ok(ok, 16, st.lim[1]) ? ld_coherent_v4(k + ok) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kStridedUnroll; ++u) {
            const uint32_t c = x[u].g * kElemsPerVec;
            const uint32_t i = table_index(p, x[u].pos, x[u].g * kPairsPerVec);
            const float4 cs01 = tab4<kSmem>(tab, i, p.tab_len);
            const float4 cs23 = kType != ROPE3D_F32 ? tab4<kSmem>(tab, i + 2, p.tab_len) : cs01;
            const long long o2 = off(2, x[u].pos, x[u].head, c), o3 = off(3, x[u].pos, x[u].head, c);
            if (bound_ok(o2, 16, st.lim[2])) st_stream_v4(qo + o2, rotate_vec<kType>(qv[u], cs01, cs23));
            if (bound_ok(o3, 16, st.lim[3])) st_stream_v4(ko + o3, rotate_vec<kType>(kv[u], cs01, cs23));
        }
    }
    for (; v < p.units; v += stride) {
        const Where x = where(v);
        const uint32_t c = x.g * kElemsPerVec;
        const long long oq = off(0, x.pos, x.head, c), ok = off(1, x.pos, x.head, c);
        const uint4 qv = bound_ok(oq, 16, st.lim[0]) ? ld_coherent_v4(q + oq) : make_uint4(0, 0, 0, 0);
        const uint4 kv = bound_ok(ok, 16, st.lim[1]) ? ld_coherent_v4(k + ok) : make_uint4(0, 0, 0, 0);
        const uint32_t i = table_index(p, x.pos, x.g * kPairsPerVec);
        const float4 cs01 = tab4<kSmem>(tab, i, p.tab_len);
        const float4 cs23 = kType != ROPE3D_F32 ? tab4<kSmem>(tab, i + 2, p.tab_len) : cs01;
        const long long o2 = off(2, x.pos, x.head, c), o3 = off(3, x.pos, x.head, c);
        if (bound_ok(o2, 16, st.lim[2])) st_stream_v4(qo + o2, rotate_vec<kType>(qv, cs01, cs23));
        if (bound_ok(o3, 16, st.lim[3])) st_stream_v4(ko + o3, rotate_vec<kType>(kv, cs01, cs23));
    }
}

// ---- per-pair kernels (any valid alignment and split) -----------------------

template <int kType>
__device__ __forceinline__ void rotate_pair_at(const char *q, const char *k, char *qo, char *ko,
                                               float2 cs, bool coherent) {
    if constexpr (kType != ROPE3D_F32) {
        // a 16-bit pair is one 4-byte aligned word
        const uint32_t qw = coherent ? *reinterpret_cast<const volatile uint32_t *>(q)
                                     : ld_nc_u32(q);
        const uint32_t kw = coherent ? *reinterpret_cast<const volatile uint32_t *>(k)
                                     : ld_nc_u32(k);
        *reinterpret_cast<uint32_t *>(qo) = rotate_word16<kType>(qw, cs.x, cs.y);
        *reinterpret_cast<uint32_t *>(ko) = rotate_word16<kType>(kw, cs.x, cs.y);
    } else {
        // an fp32 pair may be only 4-byte aligned: two scalar accesses
        const float *qf = reinterpret_cast<const float *>(q);
        const float *kf = reinterpret_cast<const float *>(k);
        float qe, qd, ke, kd;
        if (coherent) {
            qe = *reinterpret_cast<const volatile float *>(qf);
            qd = *reinterpret_cast<const volatile float *>(qf + 1);
            ke = *reinterpret_cast<const volatile float *>(kf);
            kd = *reinterpret_cast<const volatile float *>(kf + 1);
        } else {
            qe = __ldg(qf);
            qd = __ldg(qf + 1);
            ke = __ldg(kf);
            kd = __ldg(kf + 1);
        }
        const Rot a = rotate(qe, qd, cs.x, cs.y);
        const Rot b = rotate(ke, kd, cs.x, cs.y);
        float *qof = reinterpret_cast<float *>(qo);
        float *kof = reinterpret_cast<float *>(ko);
        qof[0] = a.y0;
        qof[1] = a.y1;
        kof[0] = b.y0;
        kof[1] = b.y1;
    }
}

template <int kType, bool kSmem>
__global__ void __launch_bounds__(kBlock)
rope3d_pair_kernel(const KParams p, const KStrides st) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const float2 *tab = stage_tables<kSmem>(p, reinterpret_cast<float2 *>(smem_raw));
    constexpr size_t kPairBytes = kType == ROPE3D_F32 ? 8 : 4;
    const char *q = static_cast<const char *>(p.q);
    const char *k = static_cast<const char *>(p.k);
    char *qo = static_cast<char *>(p.q_out);
    char *ko = static_cast<char *>(p.k_out);
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v < p.units; v += stride) {
        const uint32_t row = fdiv(v, p.per_row);
        const uint32_t r = v - row * p.per_row.d;
        const uint32_t pair = r - fdiv(r, p.per_head) * p.per_head.d;
        const float2 cs = tab1<kSmem>(tab, table_index(p, grid_pos(p, row), pair), p.tab_len);
        const size_t off = size_t(v) * kPairBytes;
        if (bound_ok(off, kPairBytes, st.lim[0]) && bound_ok(off, kPairBytes, st.lim[1]) &&
            bound_ok(off, kPairBytes, st.lim[2]) && bound_ok(off, kPairBytes, st.lim[3]))
            rotate_pair_at<kType>(q + off, k + off, qo + off, ko + off, cs, false);
    }
}

template <int kType, bool kSmem>
__global__ void __launch_bounds__(kBlock)
rope3d_pair_strided_kernel(const KParams p, const KStrides st) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const float2 *tab = stage_tables<kSmem>(p, reinterpret_cast<float2 *>(smem_raw));
    constexpr int kElemBytes = kType == ROPE3D_F32 ? 4 : 2;
    const char *q = static_cast<const char *>(p.q);
    const char *k = static_cast<const char *>(p.k);
    char *qo = static_cast<char *>(p.q_out);
    char *ko = static_cast<char *>(p.k_out);
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v < p.units; v += stride) {
        const uint32_t row = fdiv(v, p.per_row);
        const uint32_t r = v - row * p.per_row.d;
        const uint32_t head = fdiv(r, p.per_head);
        const uint32_t pair = r - head * p.per_head.d;
        const GridPos pos = grid_pos(p, row);
        const float2 cs = tab1<kSmem>(tab, table_index(p, pos, pair), p.tab_len);
        const uint32_t channel = 2 * pair;
        long long o[4];
        bool in = true;
        for (int i = 0; i < 4; ++i) {
            o[i] = strided_offset(st, i, pos, head, channel) * kElemBytes;
            in = bound_ok(o[i], 2 * kElemBytes, st.lim[i]) && in;
        }
        if (in) rotate_pair_at<kType>(q + o[0], k + o[1], qo + o[2], ko + o[3], cs, true);
    }
}

// ---- gather of a strided view into a contiguous buffer ----------------------

template <int kElemBytes>
__global__ void __launch_bounds__(kBlock)
rope3d_gather_kernel(const char *src, char *dst, const KParams p, const KStrides st) {
    // units = elements of this launch; per_row = heads * head_dim, per_head = head_dim
    using Word = typename std::conditional<kElemBytes == 2, uint16_t, uint32_t>::type;
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t e = blockIdx.x * blockDim.x + threadIdx.x; e < p.units; e += stride) {
        const uint32_t row = fdiv(e, p.per_row);
        const uint32_t r = e - row * p.per_row.d;
        const uint32_t head = fdiv(r, p.per_head);
        const uint32_t c = r - head * p.per_head.d;
        const GridPos pos = grid_pos(p, row);
        const long long o = strided_offset(st, 0, pos, head, c) * kElemBytes;
        if (bound_ok(o, kElemBytes, st.lim[0]) && bound_ok(size_t(e) * kElemBytes, kElemBytes, st.lim[1]))
            *reinterpret_cast<Word *>(dst + size_t(e) * kElemBytes) =
                *reinterpret_cast<const Word *>(src + o);
    }
}

// ---- launch ----------------------------------------------------------------

using KernelFn = void (*)(KParams, KStrides);

template <int kType>
KernelFn pick_type(bool vec16, bool strided, bool same, bool smem) {
    if (vec16 && !strided)
        return smem ? rope3d_vec16_kernel<kType, true> : rope3d_vec16_kernel<kType, false>;
    if (vec16 && same)
        return smem ? rope3d_vec16_strided_kernel<kType, true, true>
                    : rope3d_vec16_strided_kernel<kType, false, true>;
    if (vec16)
        return smem ? rope3d_vec16_strided_kernel<kType, true, false>
                    : rope3d_vec16_strided_kernel<kType, false, false>;
    if (!strided)
        return smem ? rope3d_pair_kernel<kType, true> : rope3d_pair_kernel<kType, false>;
    return smem ? rope3d_pair_strided_kernel<kType, true> : rope3d_pair_strided_kernel<kType, false>;
}

KernelFn pick(int dtype, bool vec16, bool strided, bool same, bool smem) {
    if (dtype == ROPE3D_BF16) return pick_type<ROPE3D_BF16>(vec16, strided, same, smem);
    if (dtype == ROPE3D_F16) return pick_type<ROPE3D_F16>(vec16, strided, same, smem);
    return pick_type<ROPE3D_F32>(vec16, strided, same, smem);
}

constexpr int kMaxDevices = 64;
constexpr int kNumVariants = 48;

struct DeviceCache {
    bool init = false;
    int sm_count = 0;
    bool attr_set[kNumVariants] = {};
    int occ[kNumVariants] = {};     // resident CTAs per SM at the smem size below
    size_t occ_smem[kNumVariants] = {};
};

std::mutex g_dev_mutex;
DeviceCache g_dev[kMaxDevices];

int variant_id(int dtype, bool vec16, bool strided, bool same, bool smem) {
    return (dtype << 4) | (vec16 ? 8 : 0) | (strided ? 4 : 0) | (same ? 2 : 0) | (smem ? 1 : 0);
}

// Grid size: enough CTAs to fill every SM at full residency, no more than
// the work needs.
cudaError_t grid_for(const void *fn, int vid, size_t smem, uint64_t units, int block, int *grid,
                     int max_ctas_per_sm = 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || vid < 0 || vid >= kNumVariants)
        return cudaErrorInvalidValue;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceCache &dc = g_dev[dev];
    if (!dc.init) {
        e = cudaDeviceGetAttribute(&dc.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        dc.init = true;
    }
    if (!dc.attr_set[vid]) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kMaxSmemTableBytes));
        if (e != cudaSuccess) return e;
        dc.attr_set[vid] = true;
    }
    if (dc.occ[vid] == 0 || dc.occ_smem[vid] != smem) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, block, smem);
        if (e != cudaSuccess) return e;
        dc.occ[vid] = n > 0 ? n : 1;
        dc.occ_smem[vid] = smem;
    }
    const int per_sm = max_ctas_per_sm > 0 ? std::min(max_ctas_per_sm, dc.occ[vid]) : dc.occ[vid];
    const uint64_t full = uint64_t(dc.sm_count) * per_sm;
    const uint64_t need = (units + block - 1) / block;
    *grid = static_cast<int>(need < full ? (need > 0 ? need : 1) : full);
    return cudaSuccess;
}

std::atomic<uint32_t> g_max_units{kMaxUnitsPerLaunch};

void fill_geometry(KParams &p, uint32_t units_per_row, uint32_t units_per_head, uint32_t T,
                   uint32_t H, uint32_t W) {
    p.per_row = make_fastdiv(units_per_row);
    p.per_head = make_fastdiv(units_per_head);
    p.N = make_fastdiv(T * H * W);
    p.HW = make_fastdiv(H * W);
    p.Wd = make_fastdiv(W);
}

}  // namespace

void set_max_units_per_launch(uint32_t n) {
    g_max_units.store(n == 0 || n > kMaxUnitsPerLaunch ? kMaxUnitsPerLaunch : n);
}

cudaError_t launch_rope3d(const LaunchArgs &a, cudaStream_t stream, LaunchInfo *info) {
    const uint32_t esize = a.dtype == ROPE3D_F32 ? 4 : 2;
    const uint32_t elems_per_unit = a.vec16 ? 16 / esize : 2;
    const uint64_t row_elems = uint64_t(a.heads) * a.head_dim;
    const uint32_t units_per_row = static_cast<uint32_t>(row_elems / elems_per_unit);
    const uint32_t units_per_head = a.head_dim / elems_per_unit;
    const uint32_t N = a.T * a.H * a.W;
    const size_t table_bytes = size_t(a.table_len) * sizeof(float2);
    const size_t smem_max = a.vec16 && !a.strided
                                ? std::min<size_t>(ROPE3D_VEC_SMEM_TABLE_MAX, kMaxSmemTableBytes)
                                : kMaxSmemTableBytes;
    const bool smem = table_bytes <= smem_max;
    const size_t smem_bytes = smem ? table_bytes : 0;
    bool same = a.strided;
    for (int i = 1; i < 4 && same; ++i)
        for (int j = 0; j < 5; ++j) same = same && a.strides[i][j] == a.strides[0][j];
    const KernelFn fn = pick(a.dtype, a.vec16, a.strided, same, smem);
    const int vid = variant_id(a.dtype, a.vec16, a.strided, same, smem);
    const int block = a.vec16 && a.strided ? kStridedBlock : kBlock;

    KParams p{};
    p.tab = a.tables;
    p.tab_len = a.table_len;
    p.offH = a.offH;
    p.offW = a.offW;
    p.pT = a.pT;
    p.pH = a.pH;
    p.pW = a.pW;
    fill_geometry(p, units_per_row, units_per_head, a.T, a.H, a.W);
    KStrides st{};
    if (a.strided) {
        // a view's span: its farthest element (strides are >= 0) plus a head row
        const uint64_t B = (a.row0 + a.rows + N - 1) / N;
        const uint64_t ext[5] = {B, a.T, a.H, a.W, a.heads};
        for (int i = 0; i < 4; ++i) {
            uint64_t far = a.head_dim;
            for (int j = 0; j < 5; ++j) {
                st.s[i][j] = a.strides[i][j];
                far += (ext[j] - 1) * uint64_t(a.strides[i][j]);
            }
            st.lim[i] = far * esize;
        }
    }

    const uint64_t cap = g_max_units.load(std::memory_order_relaxed);
    const uint64_t rows_per_launch = cap / units_per_row > 0 ? cap / units_per_row : 1;
    for (uint64_t r = 0; r < a.rows; r += rows_per_launch) {
        const uint64_t nrows = (a.rows - r) < rows_per_launch ? (a.rows - r) : rows_per_launch;
        if (a.strided) {
            // strided views address rows by (batch, t, h, w): pointers stay put
            p.q = a.q;
            p.k = a.k;
            p.q_out = a.q_out;
            p.k_out = a.k_out;
            st.b0 = static_cast<uint32_t>((a.row0 + r) / N);
        } else {
            const uint64_t elem_off = r * row_elems;
            p.q = static_cast<const char *>(a.q) + elem_off * esize;
            p.k = static_cast<const char *>(a.k) + elem_off * esize;
            p.q_out = static_cast<char *>(a.q_out) + elem_off * esize;
            p.k_out = static_cast<char *>(a.k_out) + elem_off * esize;
            for (int i = 0; i < 4; ++i) st.lim[i] = nrows * row_elems * esize;
        }
        p.units = static_cast<uint32_t>(nrows * units_per_row);
        p.row0_mod_N = static_cast<uint32_t>((a.row0 + r) % N);
        int grid = 0;
        cudaError_t e = grid_for(reinterpret_cast<const void *>(fn), vid, smem_bytes, p.units,
                                 block, &grid, a.vec16 && !a.strided ? ROPE3D_VEC_GRID_CTAS : 0);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(block);
        cfg.dynamicSmemBytes = smem_bytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = a.pdl ? attr : nullptr;
        cfg.numAttrs = a.pdl ? 1 : 0;
        e = cudaLaunchKernelEx(&cfg, fn, p, st);
        if (e != cudaSuccess) return e;
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (info) {
            info->kernel = a.vec16 ? 1 : 2;
            info->grid = grid;
            info->block = block;
        }
    }
    return cudaSuccess;
}

cudaError_t launch_gather(const void *src, const int64_t strides[5], void *dst, int elem_bytes,
                          uint64_t B, uint32_t T, uint32_t H, uint32_t W, uint32_t heads,
                          uint32_t head_dim, cudaStream_t stream) {
    const uint64_t row_elems = uint64_t(heads) * head_dim;
    const uint64_t rows = B * T * H * W;
    const uint32_t N = T * H * W;
    KParams p{};
    fill_geometry(p, static_cast<uint32_t>(row_elems), head_dim, T, H, W);
    KStrides st{};
    uint64_t far = head_dim;
    const uint64_t ext[5] = {B, T, H, W, heads};
    for (int j = 0; j < 5; ++j) {
        st.s[0][j] = strides[j];
        far += (ext[j] - 1) * uint64_t(strides[j]);
    }
    st.lim[0] = far * elem_bytes;   // the source view
    const uint64_t rows_per_launch = std::max<uint64_t>(1, kMaxUnitsPerLaunch / row_elems);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    for (uint64_t r = 0; r < rows; r += rows_per_launch) {
        const uint64_t nrows = std::min<uint64_t>(rows - r, rows_per_launch);
        p.units = static_cast<uint32_t>(nrows * row_elems);
        p.row0_mod_N = static_cast<uint32_t>(r % N);
        st.b0 = static_cast<uint32_t>(r / N);
        const uint64_t need = (uint64_t(p.units) + kBlock - 1) / kBlock;
        const int grid = static_cast<int>(std::min<uint64_t>(need, uint64_t(sms) * 4));
        char *d = static_cast<char *>(dst) + r * row_elems * elem_bytes;
        st.lim[1] = nrows * row_elems * elem_bytes;   // this launch's part of dst
        if (elem_bytes == 2)
            rope3d_gather_kernel<2><<<grid, kBlock, 0, stream>>>(static_cast<const char *>(src), d, p, st);
        else
            rope3d_gather_kernel<4><<<grid, kBlock, 0, stream>>>(static_cast<const char *>(src), d, p, st);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace rope3d

namespace rope3d {

// This file's bound-check error count (0 unless built with the checks);
// `reset` clears it. Synchronises the device when built with the checks.
int64_t kernels_bound_errors(bool reset) {
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
