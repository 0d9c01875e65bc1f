// rope3d_na3d.cu -- 3D neighbourhood attention with the decoder's RoPE fused
// into its prologue: rope3d_na3d.
//
// Before each attention block the LTX-2.5 diffusion decoder rotates Q and K
// (sglang PR #35698 review, "功能与动机" and "实现拆解"); its attention is
// NATTEN's 3D neighbourhood attention (sglang PR #34471 review, "关键源码片段",
// _na3d). Fusing the rotation into the attention kernel removes the round trip
// of Q_out and K_out through HBM: Q and K tiles are rotated while they are
// staged into shared memory, with exactly the arithmetic of rope3d_apply_pair
// (four rounded fp32 products, one subtract, one add, a nearest-even cast to
// bf16), so the rotated operands are bit-identical to the unfused path's.
//
// Neighbourhood attention as published (Hassani et al., "Neighborhood Attention
// Transformer", CVPR 2023): a query at (t, h, w) attends to the k_t x k_h x k_w
// window centred on it, shifted inside the grid at the borders (start
// min(max(i - k/2, 0), L - k) per axis), with softmax(q.k / sqrt(d)) weights.
//
// Work decomposition: a CTA of 4 warps owns one (batch, head) and a block of
// 1 x 8 x 8 query tokens; its key region is the union of their windows, visited
// in chunks of 64 keys. Each warp holds 16 query rows; S = Q K^T and O += P V
// run on the tensor cores as bf16 m16n8k16 MMAs with fp32 accumulators, with a
// flash-style online softmax in registers (running max and sum per row) and a
// per-element window mask. Tables (when rotating) sit in shared memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/rope3d.h"
#include "rope3d_internal.h"

namespace {

constexpr int kHD = 128;             // head_dim
constexpr int kQB = 64;              // queries per CTA (1 x 8 x 8)
constexpr int kQBH = 8, kQBW = 8;
constexpr int kKC = 64;              // keys per chunk
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRow = kHD + 8;        // padded smem row (bf16): 272 bytes
constexpr uint32_t kMaxTableBytes = 48 * 1024;

struct NAParams {
    const uint16_t *q, *k, *v;
    uint16_t *out;
    const float2 *tab;
    uint32_t tab_len, offH, offW, pT, pH, pW;
    int B, T, H, W, heads;
    int kt, kh, kw;
    int nbh, nbw;            // query blocks along H and W
    int rope;
    float scale_log2;        // log2(e) / sqrt(head_dim)
};

__device__ __forceinline__ int na_start(int i, int L, int k) {
    int s = i - k / 2;
    s = s < 0 ? 0 : s;
    return s + k > L ? L - k : s;
}

// Eager-order rotation of one bf16 pair word (as in rope3d_kernels.cu).
__device__ __forceinline__ uint32_t rot_word(uint32_t word, float c, float s) {
    const float even = __uint_as_float(word << 16);
    const float odd = __uint_as_float(word & 0xffff0000u);
    const float ec = __fmul_rn(even, c), os = __fmul_rn(odd, s);
    const float es = __fmul_rn(even, s), oc = __fmul_rn(odd, c);
    const __nv_bfloat162 r = __floats2bfloat162_rn(__fsub_rn(ec, os), __fadd_rn(es, oc));
    uint32_t out;
    memcpy(&out, &r, 4);
    return out;
}

// Rotate the 8 channels [ch, ch + 8) of a token at grid position (t, h, w).
// Every chunk of the split is a multiple of 8 channels, so the 4 pairs lie in
// one axis and read 4 consecutive (cos, sin) entries: two 16-byte loads (the
// entry index is a multiple of 4, so they are aligned).
__device__ __forceinline__ uint4 rot_vec(uint4 v, const float2 *tab, const NAParams &p, int t,
                                         int h, int w, int ch) {
    const uint32_t pair = ch / 2;
    uint32_t idx;
    if (pair < p.pT) idx = t * p.pT + pair;
    else if (pair < p.pT + p.pH) idx = p.offH + h * p.pH + (pair - p.pT);
    else idx = p.offW + w * p.pW + (pair - p.pT - p.pH);
    const float4 a = *reinterpret_cast<const float4 *>(tab + idx);
    const float4 b = *reinterpret_cast<const float4 *>(tab + idx + 2);
    return make_uint4(rot_word(v.x, a.x, a.y), rot_word(v.y, a.z, a.w), rot_word(v.z, b.x, b.y),
                      rot_word(v.w, b.z, b.w));
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous copy global -> shared (bypassing registers and L1).
__device__ __forceinline__ void cp_async16(void *dst_smem, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)), "l"(src)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A * B + D, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
    uint32_t u;
    memcpy(&u, &r, 4);
    return u;
}

__global__ void __launch_bounds__(kThreads)
rope3d_na3d_kernel(const NAParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    uint16_t *sQ = reinterpret_cast<uint16_t *>(smem);
    uint16_t *sK = sQ + kQB * kRow;
    uint16_t *sV = sK + kKC * kRow;
    int *sKey = reinterpret_cast<int *>(sV + kKC * kRow);          // packed key coordinates
    float2 *sTab = reinterpret_cast<float2 *>(sKey + kKC);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tq = lane & 3;

    // which (batch, head, query block)
    int blk = blockIdx.x;
    const int bw = blk % p.nbw; blk /= p.nbw;
    const int bh = blk % p.nbh; blk /= p.nbh;
    const int qt = blk % p.T; blk /= p.T;
    const int head = blk % p.heads;
    const int b = blk / p.heads;
    const int h0 = bh * kQBH, w0 = bw * kQBW;

    if (p.rope) {
        for (uint32_t i = tid; i < p.tab_len; i += kThreads) sTab[i] = p.tab[i];
        __syncthreads();
    }
    const size_t tok_stride = size_t(p.heads) * kHD;            // elements per token
    auto token_index = [&](int t, int h, int w) {
        return ((size_t(b) * p.T + t) * p.H + h) * p.W + w;
    };

    // ---- Q tile: 64 rows x 128 channels copied asynchronously, then rotated in
    // shared memory
    for (int i = tid; i < kQB * (kHD / 8); i += kThreads) {
        const int row = i / (kHD / 8), cv = i % (kHD / 8);
        const int h = h0 + row / kQBW, w = w0 + row % kQBW;
        uint16_t *dst = sQ + row * kRow + cv * 8;
        if (h < p.H && w < p.W)
            cp_async16(dst, p.q + token_index(qt, h, w) * tok_stride + size_t(head) * kHD + cv * 8);
        else
            *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
    cp_async_wait_all();
    __syncthreads();
    if (p.rope) {
        for (int i = tid; i < kQB * (kHD / 8); i += kThreads) {
            const int cv = i / kQB, row = i % kQB;   // one channel column per warp
            const int h = h0 + row / kQBW, w = w0 + row % kQBW;
            if (h < p.H && w < p.W) {
                uint4 *ptr = reinterpret_cast<uint4 *>(sQ + row * kRow + cv * 8);
                *ptr = rot_vec(*ptr, sTab, p, qt, h, w, cv * 8);
            }
        }
    }

    // key region: the union of the block's windows
    const int rt0 = na_start(qt, p.T, p.kt), rt1 = rt0 + p.kt;
    const int hl = min(h0 + kQBH, p.H) - 1, wl = min(w0 + kQBW, p.W) - 1;
    const int rh0 = na_start(h0, p.H, p.kh), rh1 = na_start(hl, p.H, p.kh) + p.kh;
    const int rw0 = na_start(w0, p.W, p.kw), rw1 = na_start(wl, p.W, p.kw) + p.kw;
    const int RH = rh1 - rh0, RW = rw1 - rw0;
    const int R = (rt1 - rt0) * RH * RW;

    // this thread's two query rows (g and g + 8 of its warp): window starts
    int wh[2], ww[2];   // window starts of the two rows in h and w (t: the region's)
    bool rvalid[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int row = warp * 16 + g + 8 * r;
        const int h = h0 + row / kQBW, w = w0 + row % kQBW;
        rvalid[r] = h < p.H && w < p.W;
        wh[r] = na_start(min(h, p.H - 1), p.H, p.kh);
        ww[r] = na_start(min(w, p.W - 1), p.W, p.kw);
    }
    // the box of this warp's windows in (h, w): chunks with no key inside it
    // are skipped by the whole warp
    int box_h0 = min(wh[0], wh[1]), box_h1 = max(wh[0], wh[1]) + p.kh;
    int box_w0 = min(ww[0], ww[1]), box_w1 = max(ww[0], ww[1]) + p.kw;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        box_h0 = min(box_h0, __shfl_xor_sync(0xffffffffu, box_h0, off));
        box_h1 = max(box_h1, __shfl_xor_sync(0xffffffffu, box_h1, off));
        box_w0 = min(box_w0, __shfl_xor_sync(0xffffffffu, box_w0, off));
        box_w1 = max(box_w1, __shfl_xor_sync(0xffffffffu, box_w1, off));
    }
    __syncthreads();

    // Q fragments of this warp's 16 rows, all 8 k-steps
    uint32_t qa[kHD / 16][4];
#pragma unroll
    for (int ks = 0; ks < kHD / 16; ++ks) {
        const uint16_t *a = sQ + (warp * 16 + (lane & 15)) * kRow + ks * 16 + (lane >> 4) * 8;
        ldsm_x4(smem_addr(a), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
    }

    float o[kHD / 8][4];
#pragma unroll
    for (int n = 0; n < kHD / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

    for (int c0 = 0; c0 < R; c0 += kKC) {
        __syncthreads();   // the previous chunk's K and V are no longer read
        // ---- K and V chunk copied asynchronously, key coordinates; then K is
        // rotated in shared memory
        for (int i = tid; i < kKC * (kHD / 8); i += kThreads) {
            const int row = i / (kHD / 8), cv = i % (kHD / 8);
            const int r = c0 + row;
            uint16_t *dk = sK + row * kRow + cv * 8;
            uint16_t *dv = sV + row * kRow + cv * 8;
            if (r < R) {
                const int dt = r / (RH * RW), rem = r - dt * RH * RW;
                const int dh = rem / RW, dw = rem - dh * RW;
                const int t = rt0 + dt, h = rh0 + dh, w = rw0 + dw;
                const size_t off = token_index(t, h, w) * tok_stride + size_t(head) * kHD + cv * 8;
                cp_async16(dk, p.k + off);
                cp_async16(dv, p.v + off);
                if (cv == 0) sKey[row] = (t << 20) | (h << 10) | w;
            } else {
                *reinterpret_cast<uint4 *>(dk) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(dv) = make_uint4(0, 0, 0, 0);
                if (cv == 0) sKey[row] = -1;
            }
        }
        cp_async_wait_all();
        __syncthreads();
        if (p.rope) {
            for (int i = tid; i < kKC * (kHD / 8); i += kThreads) {
                const int cv = i / kKC, row = i % kKC;   // one channel column per warp
                const int key = sKey[row];
                if (key >= 0) {
                    uint4 *ptr = reinterpret_cast<uint4 *>(sK + row * kRow + cv * 8);
                    *ptr = rot_vec(*ptr, sTab, p, key >> 20, (key >> 10) & 1023, key & 1023, cv * 8);
                }
            }
            __syncthreads();
        }

        // skip the chunk if none of its keys falls in this warp's window box
        {
            bool any = false;
#pragma unroll
            for (int j = 0; j < kKC / 32; ++j) {
                const int key = sKey[lane + 32 * j];
                if (key >= 0) {
                    const int kh_ = (key >> 10) & 1023, kw_ = key & 1023;
                    any |= kh_ >= box_h0 && kh_ < box_h1 && kw_ >= box_w0 && kw_ < box_w1;
                }
            }
            if (!__any_sync(0xffffffffu, any)) continue;
        }

        // ---- S = Q K^T for this warp's 16 rows x 64 keys
        float s[kKC / 8][4];
#pragma unroll
        for (int n = 0; n < kKC / 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int np = 0; np < kKC / 16; ++np) {
#pragma unroll
            for (int ks = 0; ks < kHD / 16; ++ks) {
                const int mi = lane >> 3, rr = lane & 7;
                const uint16_t *bp = sK + (np * 16 + rr + (mi >> 1) * 8) * kRow + ks * 16 + (mi & 1) * 8;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(smem_addr(bp), b0, b1, b2, b3);
                mma(s[2 * np], qa[ks], b0, b1);
                mma(s[2 * np + 1], qa[ks], b2, b3);
            }
        }

        // ---- mask, online softmax
        float cmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < kKC / 8; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = e >> 1;
                const int key = sKey[n * 8 + 2 * tq + (e & 1)];
                // every key of the region lies in each row's t window (the block
                // is one frame), so only h and w are tested
                const bool ok = key >= 0 && rvalid[r] &&
                                unsigned(((key >> 10) & 1023) - wh[r]) < unsigned(p.kh) &&
                                unsigned((key & 1023) - ww[r]) < unsigned(p.kw);
                s[n][e] = ok ? s[n][e] * p.scale_log2 : -INFINITY;
                cmax[r] = fmaxf(cmax[r], s[n][e]);
            }
        }
        float corr[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            cmax[r] = fmaxf(cmax[r], __shfl_xor_sync(0xffffffffu, cmax[r], 1));
            cmax[r] = fmaxf(cmax[r], __shfl_xor_sync(0xffffffffu, cmax[r], 2));
            const float mn = fmaxf(m[r], cmax[r]);
            corr[r] = (mn == -INFINITY) ? 1.f : exp2f(m[r] - mn);   // m = -inf -> 0 unless mn is -inf
            m[r] = mn;
            l[r] *= corr[r];
        }
        float psum[2] = {0.f, 0.f};
#pragma unroll
        for (int n = 0; n < kKC / 8; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = e >> 1;
                const float pv = (s[n][e] == -INFINITY) ? 0.f : exp2f(s[n][e] - m[r]);
                s[n][e] = pv;
                psum[r] += pv;
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            psum[r] += __shfl_xor_sync(0xffffffffu, psum[r], 1);
            psum[r] += __shfl_xor_sync(0xffffffffu, psum[r], 2);
            l[r] += psum[r];
        }
#pragma unroll
        for (int n = 0; n < kHD / 8; ++n) {
            o[n][0] *= corr[0];
            o[n][1] *= corr[0];
            o[n][2] *= corr[1];
            o[n][3] *= corr[1];
        }

        // ---- O += P V
#pragma unroll
        for (int kk = 0; kk < kKC / 16; ++kk) {
            uint32_t pa[4];
            pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
            pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
            pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
            for (int np = 0; np < kHD / 16; ++np) {
                const int mi = lane >> 3, rr = lane & 7;
                const uint16_t *bp = sV + (kk * 16 + rr + (mi & 1) * 8) * kRow + np * 16 + (mi >> 1) * 8;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(smem_addr(bp), b0, b1, b2, b3);
                mma(o[2 * np], pa, b0, b1);
                mma(o[2 * np + 1], pa, b2, b3);
            }
        }
    }

    // ---- normalise and store
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        if (!rvalid[r]) continue;
        const int row = warp * 16 + g + 8 * r;
        const int h = h0 + row / kQBW, w = w0 + row % kQBW;
        const float inv = l[r] > 0.f ? 1.f / l[r] : 0.f;
        uint16_t *dst = p.out + token_index(qt, h, w) * tok_stride + size_t(head) * kHD;
#pragma unroll
        for (int n = 0; n < kHD / 8; ++n) {
            const uint32_t pk = pack_bf16(o[n][2 * r] * inv, o[n][2 * r + 1] * inv);
            *reinterpret_cast<uint32_t *>(dst + n * 8 + 2 * tq) = pk;
        }
    }
}

bool on_device(const void *ptr, int device) {
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (attr.type == cudaMemoryTypeManaged) return true;
    return attr.type == cudaMemoryTypeDevice && attr.device == device;
}

}  // namespace

extern "C" int rope3d_na3d(const void *q, const void *k, const void *v, void *out,
                           const rope3d_tables *tables, int64_t B, int64_t T, int64_t H,
                           int64_t W, int64_t heads, int64_t head_dim, const int32_t split[3],
                           const int32_t kernel_size[3], int32_t apply_rope, void *stream) {
    if (!q || !k || !v || !out || !kernel_size || (apply_rope && (!tables || !split)))
        return ROPE3D_ERR_NULL;
    if (B <= 0 || T <= 0 || H <= 0 || W <= 0 || heads <= 0) return ROPE3D_ERR_SHAPE;
    if (head_dim != kHD) return ROPE3D_ERR_SHAPE;
    if (T >= 1024 || H >= 1024 || W >= 1024 || B * T * H * W * heads > (int64_t(1) << 40))
        return ROPE3D_ERR_SHAPE;
    const int kt = kernel_size[0], kh = kernel_size[1], kw = kernel_size[2];
    if (kt < 1 || kh < 1 || kw < 1 || kt % 2 == 0 || kh % 2 == 0 || kw % 2 == 0 || kt > T ||
        kh > H || kw > W)
        return ROPE3D_ERR_SHAPE;
    for (const void *ptr : {q, k, v, static_cast<const void *>(out)})
        if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return ROPE3D_ERR_ALIGN;
    const uint64_t bytes = uint64_t(B * T * H * W * heads) * kHD * 2;
    const uintptr_t o = reinterpret_cast<uintptr_t>(out);
    for (const void *ptr : {q, k, v}) {
        const uintptr_t x = reinterpret_cast<uintptr_t>(ptr);
        if (o < x + bytes && x < o + bytes) return ROPE3D_ERR_ALIAS;
    }
    NAParams p{};
    if (apply_rope) {
        const float2 *dev = nullptr;
        uint32_t len = 0, offs[3];
        int64_t dims[3];
        int32_t sp[3];
        int tdev = -1;
        bool host_backed = false;
        if (rope3d::tables_layout(tables, &dev, &len, offs, dims, sp, &tdev, &host_backed) != ROPE3D_OK)
            return ROPE3D_ERR_NULL;
        if (dims[0] != T || dims[1] != H || dims[2] != W || sp[0] != split[0] || sp[1] != split[1] ||
            sp[2] != split[2])
            return ROPE3D_ERR_TABLES;
        if (int64_t(split[0]) + split[1] + split[2] != head_dim || split[0] % 8 || split[1] % 8 ||
            split[2] % 8)
            return ROPE3D_ERR_SHAPE;
        if (len * sizeof(float2) > kMaxTableBytes) return ROPE3D_ERR_SHAPE;
        int cur = 0;
        if (cudaGetDevice(&cur) != cudaSuccess) return ROPE3D_ERR_CUDA;
        if (host_backed || tdev != cur) return ROPE3D_ERR_DEVICE;
        p.tab = dev;
        p.tab_len = len;
        p.offH = offs[1];
        p.offW = offs[2];
        p.pT = split[0] / 2;
        p.pH = split[1] / 2;
        p.pW = split[2] / 2;
    }
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return ROPE3D_ERR_CUDA;
    for (const void *ptr : {q, k, v, static_cast<const void *>(out)})
        if (!on_device(ptr, device)) return ROPE3D_ERR_DEVICE;

    p.q = static_cast<const uint16_t *>(q);
    p.k = static_cast<const uint16_t *>(k);
    p.v = static_cast<const uint16_t *>(v);
    p.out = static_cast<uint16_t *>(out);
    p.B = int(B);
    p.T = int(T);
    p.H = int(H);
    p.W = int(W);
    p.heads = int(heads);
    p.kt = kt;
    p.kh = kh;
    p.kw = kw;
    p.nbh = int((H + kQBH - 1) / kQBH);
    p.nbw = int((W + kQBW - 1) / kQBW);
    p.rope = apply_rope ? 1 : 0;
    p.scale_log2 = float(1.4426950408889634 / std::sqrt(double(kHD)));
    const uint64_t blocks = uint64_t(B) * heads * T * p.nbh * p.nbw;
    if (blocks > 0x7fffffffull) return ROPE3D_ERR_SHAPE;
    const size_t smem = size_t(kQB + 2 * kKC) * kRow * 2 + kKC * sizeof(int) +
                        (apply_rope ? size_t(p.tab_len) * sizeof(float2) : 0);
    static const cudaError_t attr_rc = cudaFuncSetAttribute(
        rope3d_na3d_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        int(size_t(kQB + 2 * kKC) * kRow * 2 + kKC * sizeof(int) + kMaxTableBytes));
    if (attr_rc != cudaSuccess) return ROPE3D_ERR_CUDA;
    rope3d_na3d_kernel<<<unsigned(blocks), kThreads, smem, static_cast<cudaStream_t>(stream)>>>(p);
    if (cudaGetLastError() != cudaSuccess) return ROPE3D_ERR_CUDA;
    return ROPE3D_OK;
}
