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
//   * one thread owns a 16-byte vector of Q and the same vector of K (8 bf16 =
//     4 pairs, or 4 fp32 = 2 pairs), loaded with streaming 128-bit loads that
//     bypass L1, and stores the two results with evict-first 128-bit stores;
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
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/rope3d.h"
#include "rope3d_internal.h"

namespace rope3d {
namespace {

constexpr int kBlock = 512;
constexpr int kUnroll = 2;

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

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) {
    return (__umulhi(n, f.mul) + n) >> f.shift;
}

// Entry index of the table entry for pair `pair_in_head` of row `row`.
__device__ __forceinline__ uint32_t table_index(const KParams &p, uint32_t row,
                                                uint32_t pair_in_head) {
    uint32_t tok = row - fdiv(row, p.N) * p.N.d + p.row0_mod_N;
    tok = tok >= p.N.d ? tok - p.N.d : tok;
    const uint32_t t = fdiv(tok, p.HW);
    const uint32_t rem = tok - t * p.HW.d;
    const uint32_t h = fdiv(rem, p.Wd);
    const uint32_t w = rem - h * p.Wd.d;
    const uint32_t it = t * p.pT + pair_in_head;
    const uint32_t ih = p.offH + h * p.pH + (pair_in_head - p.pT);
    const uint32_t iw = p.offW + w * p.pW + (pair_in_head - p.pT - p.pH);
    return pair_in_head < p.pT ? it : (pair_in_head < p.pT + p.pH ? ih : iw);
}

// ---- memory access ---------------------------------------------------------

__device__ __forceinline__ uint4 ld_stream_v4(const void *ptr) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(ptr));
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

// One 32-bit word holding a bf16 pair: the even element is the low half
// (lower address). bf16 -> f32 widening is a 16-bit shift.
__device__ __forceinline__ uint32_t rotate_bf16_word(uint32_t word, float c, float s) {
    const float even = __uint_as_float(word << 16);
    const float odd = __uint_as_float(word & 0xffff0000u);
    const Rot r = rotate(even, odd, c, s);
    const __nv_bfloat162 packed = __floats2bfloat162_rn(r.y0, r.y1);  // .x = y0 (low)
    uint32_t out;
    memcpy(&out, &packed, sizeof out);
    return out;
}

template <bool kBf16>
__device__ __forceinline__ uint4 rotate_vec(const uint4 v, const float4 cs01, const float4 cs23) {
    uint4 o;
    if constexpr (kBf16) {
        // 8 bf16 = 4 pairs; entries (c0, s0, c1, s1) and (c2, s2, c3, s3)
        o.x = rotate_bf16_word(v.x, cs01.x, cs01.y);
        o.y = rotate_bf16_word(v.y, cs01.z, cs01.w);
        o.z = rotate_bf16_word(v.z, cs23.x, cs23.y);
        o.w = rotate_bf16_word(v.w, cs23.z, cs23.w);
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

template <bool kSmem>
__device__ __forceinline__ const float2 *stage_tables(const KParams &p, float2 *smem) {
    if constexpr (kSmem) {
        for (uint32_t i = threadIdx.x; i < p.tab_len; i += blockDim.x) smem[i] = __ldg(p.tab + i);
        __syncthreads();
        return smem;
    } else {
        return p.tab;
    }
}

template <bool kSmem>
__device__ __forceinline__ float4 tab4(const float2 *tab, uint32_t idx) {
    // idx is a multiple of 2 entries: one 16-byte load of two (cos, sin) entries
    if constexpr (kSmem) {
        return *reinterpret_cast<const float4 *>(tab + idx);
    } else {
        return __ldg(reinterpret_cast<const float4 *>(tab + idx));
    }
}

// ---- 16-byte vector kernel ---------------------------------------------------
// Requires: 16-byte aligned pointers, head_dim and each chunk a multiple of the
// vector's element count (so a vector never straddles a chunk, head or row, and
// the first table entry of a vector is a multiple of 4 (bf16) or 2 (fp32)).

template <bool kBf16, bool kSmem>
__global__ void __launch_bounds__(kBlock)
rope3d_vec16_kernel(const KParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const float2 *tab = stage_tables<kSmem>(p, reinterpret_cast<float2 *>(smem_raw));
    constexpr uint32_t kPairsPerVec = kBf16 ? 4 : 2;

    const uint4 *q = static_cast<const uint4 *>(p.q);
    const uint4 *k = static_cast<const uint4 *>(p.k);
    uint4 *qo = static_cast<uint4 *>(p.q_out);
    uint4 *ko = static_cast<uint4 *>(p.k_out);

    const uint32_t stride = gridDim.x * blockDim.x;
    uint32_t v = blockIdx.x * blockDim.x + threadIdx.x;

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
            idx[u] = table_index(p, row, g * kPairsPerVec);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const float4 cs01 = tab4<kSmem>(tab, idx[u]);
            const float4 cs23 = kBf16 ? tab4<kSmem>(tab, idx[u] + 2) : cs01;
            st_stream_v4(qo + v + u * stride, rotate_vec<kBf16>(qv[u], cs01, cs23));
            st_stream_v4(ko + v + u * stride, rotate_vec<kBf16>(kv[u], cs01, cs23));
        }
    }
    // ragged tail: at most kUnroll - 1 more vectors per thread
    for (; v < p.units; v += stride) {
        const uint4 qv = ld_stream_v4(q + v);
        const uint4 kv = ld_stream_v4(k + v);
        const uint32_t row = fdiv(v, p.per_row);
        const uint32_t r = v - row * p.per_row.d;
        const uint32_t g = r - fdiv(r, p.per_head) * p.per_head.d;
        const uint32_t i = table_index(p, row, g * kPairsPerVec);
        const float4 cs01 = tab4<kSmem>(tab, i);
        const float4 cs23 = kBf16 ? tab4<kSmem>(tab, i + 2) : cs01;
        st_stream_v4(qo + v, rotate_vec<kBf16>(qv, cs01, cs23));
        st_stream_v4(ko + v, rotate_vec<kBf16>(kv, cs01, cs23));
    }
}

// ---- per-pair kernel (any valid alignment and split) -------------------------

template <bool kBf16, bool kSmem>
__global__ void __launch_bounds__(kBlock)
rope3d_pair_kernel(const KParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const float2 *tab = stage_tables<kSmem>(p, reinterpret_cast<float2 *>(smem_raw));
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t v = blockIdx.x * blockDim.x + threadIdx.x; v < p.units; v += stride) {
        const uint32_t row = fdiv(v, p.per_row);
        const uint32_t r = v - row * p.per_row.d;
        const uint32_t pair = r - fdiv(r, p.per_head) * p.per_head.d;
        const float2 cs = kSmem ? tab[table_index(p, row, pair)]
                                : __ldg(tab + table_index(p, row, pair));
        if constexpr (kBf16) {
            // a bf16 pair is one 4-byte aligned word
            const uint32_t *q = static_cast<const uint32_t *>(p.q);
            const uint32_t *k = static_cast<const uint32_t *>(p.k);
            uint32_t *qo = static_cast<uint32_t *>(p.q_out);
            uint32_t *ko = static_cast<uint32_t *>(p.k_out);
            qo[v] = rotate_bf16_word(ld_nc_u32(q + v), cs.x, cs.y);
            ko[v] = rotate_bf16_word(ld_nc_u32(k + v), cs.x, cs.y);
        } else {
            // an fp32 pair may be only 4-byte aligned: two scalar accesses
            const float *q = static_cast<const float *>(p.q);
            const float *k = static_cast<const float *>(p.k);
            float *qo = static_cast<float *>(p.q_out);
            float *ko = static_cast<float *>(p.k_out);
            const Rot a = rotate(__ldg(q + 2 * size_t(v)), __ldg(q + 2 * size_t(v) + 1), cs.x, cs.y);
            const Rot b = rotate(__ldg(k + 2 * size_t(v)), __ldg(k + 2 * size_t(v) + 1), cs.x, cs.y);
            qo[2 * size_t(v)] = a.y0;
            qo[2 * size_t(v) + 1] = a.y1;
            ko[2 * size_t(v)] = b.y0;
            ko[2 * size_t(v) + 1] = b.y1;
        }
    }
}

// ---- launch ----------------------------------------------------------------

using KernelFn = void (*)(KParams);

KernelFn pick(bool vec16, bool bf16, bool smem) {
    if (vec16) {
        if (bf16) return smem ? rope3d_vec16_kernel<true, true> : rope3d_vec16_kernel<true, false>;
        return smem ? rope3d_vec16_kernel<false, true> : rope3d_vec16_kernel<false, false>;
    }
    if (bf16) return smem ? rope3d_pair_kernel<true, true> : rope3d_pair_kernel<true, false>;
    return smem ? rope3d_pair_kernel<false, true> : rope3d_pair_kernel<false, false>;
}

constexpr int kMaxDevices = 64;
constexpr int kNumVariants = 8;

struct DeviceCache {
    bool init = false;
    int sm_count = 0;
    bool attr_set[kNumVariants] = {};
    int occ[kNumVariants] = {};     // resident CTAs per SM at the smem size below
    size_t occ_smem[kNumVariants] = {};
};

std::mutex g_dev_mutex;
DeviceCache g_dev[kMaxDevices];

int variant_id(bool vec16, bool bf16, bool smem) {
    return (vec16 ? 4 : 0) | (bf16 ? 2 : 0) | (smem ? 1 : 0);
}

// Grid size: enough CTAs to fill every SM at full residency, no more than
// the work needs.
cudaError_t grid_for(KernelFn fn, int vid, size_t smem, uint64_t units, int *grid) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceCache &dc = g_dev[dev];
    if (!dc.init) {
        e = cudaDeviceGetAttribute(&dc.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        dc.init = true;
    }
    if (!dc.attr_set[vid]) {
        e = cudaFuncSetAttribute(reinterpret_cast<const void *>(fn),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kMaxSmemTableBytes));
        if (e != cudaSuccess) return e;
        dc.attr_set[vid] = true;
    }
    if (dc.occ[vid] == 0 || dc.occ_smem[vid] != smem) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kBlock, smem);
        if (e != cudaSuccess) return e;
        dc.occ[vid] = n > 0 ? n : 1;
        dc.occ_smem[vid] = smem;
    }
    const uint64_t full = uint64_t(dc.sm_count) * dc.occ[vid];
    const uint64_t need = (units + kBlock - 1) / kBlock;
    *grid = static_cast<int>(need < full ? (need > 0 ? need : 1) : full);
    return cudaSuccess;
}

std::atomic<uint32_t> g_max_units{kMaxUnitsPerLaunch};

}  // namespace

void set_max_units_per_launch(uint32_t n) {
    g_max_units.store(n == 0 || n > kMaxUnitsPerLaunch ? kMaxUnitsPerLaunch : n);
}

cudaError_t launch_rope3d(const LaunchArgs &a, cudaStream_t stream, LaunchInfo *info) {
    const bool bf16 = a.dtype == ROPE3D_BF16;
    const uint32_t esize = bf16 ? 2 : 4;
    const uint32_t elems_per_unit = a.vec16 ? 16 / esize : 2;
    const uint64_t row_elems = uint64_t(a.heads) * a.head_dim;
    const uint32_t units_per_row = static_cast<uint32_t>(row_elems / elems_per_unit);
    const uint32_t units_per_head = a.head_dim / elems_per_unit;
    const uint32_t N = a.T * a.H * a.W;
    const size_t table_bytes = size_t(a.table_len) * sizeof(float2);
    const bool smem = table_bytes <= kMaxSmemTableBytes;
    const size_t smem_bytes = smem ? table_bytes : 0;
    const KernelFn fn = pick(a.vec16, bf16, smem);
    const int vid = variant_id(a.vec16, bf16, smem);

    KParams p{};
    p.tab = a.tables;
    p.tab_len = a.table_len;
    p.offH = a.offH;
    p.offW = a.offW;
    p.pT = a.pT;
    p.pH = a.pH;
    p.pW = a.pW;
    p.per_row = make_fastdiv(units_per_row);
    p.per_head = make_fastdiv(units_per_head);
    p.N = make_fastdiv(N);
    p.HW = make_fastdiv(a.H * a.W);
    p.Wd = make_fastdiv(a.W);

    const uint64_t cap = g_max_units.load(std::memory_order_relaxed);
    const uint64_t rows_per_launch = cap / units_per_row > 0 ? cap / units_per_row : 1;
    for (uint64_t r = 0; r < a.rows; r += rows_per_launch) {
        const uint64_t nrows = (a.rows - r) < rows_per_launch ? (a.rows - r) : rows_per_launch;
        const uint64_t elem_off = r * row_elems;
        p.q = static_cast<const char *>(a.q) + elem_off * esize;
        p.k = static_cast<const char *>(a.k) + elem_off * esize;
        p.q_out = static_cast<char *>(a.q_out) + elem_off * esize;
        p.k_out = static_cast<char *>(a.k_out) + elem_off * esize;
        p.units = static_cast<uint32_t>(nrows * units_per_row);
        p.row0_mod_N = static_cast<uint32_t>((a.row0 + r) % N);
        int grid = 0;
        cudaError_t e = grid_for(fn, vid, smem_bytes, p.units, &grid);
        if (e != cudaSuccess) return e;
        fn<<<grid, kBlock, smem_bytes, stream>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (info) {
            info->kernel = a.vec16 ? 1 : 2;
            info->grid = grid;
            info->block = kBlock;
        }
    }
    return cudaSuccess;
}

}  // namespace rope3d
