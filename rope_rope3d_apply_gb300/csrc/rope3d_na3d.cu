// rope3d_na3d.cu -- 3D neighbourhood attention with the decoder's RoPE fused
// into it: rope3d_na3d and rope3d_na3d_rotate_once.
//
// Before each attention block the LTX-2.5 diffusion decoder rotates Q and K
// (sglang PR #35698 review, "功能与动机" and "实现拆解"); its attention is
// NATTEN's 3D neighbourhood attention (sglang PR #34471 review, "关键源码片段",
// _na3d). Fusing the rotation into the attention removes HBM round trips of
// the rotated operands. The rotation is exactly rope3d_apply_pair's (four
// rounded fp32 products, one subtract, one add, a nearest-even cast to bf16),
// so the rotated operands are bit-identical to the unfused path's. Three
// forms of the attention kernel:
//  - kRotNone: Q and K come rotated (rope3d_apply_pair first; apply_rope = 0);
//  - kRotQK: Q and every K tile are rotated while staged into shared memory
//    (apply_rope = 1). Each key lies in the key regions of about ten CTAs and
//    is rotated by each of them, which costs more than the round trip saves;
//  - kRotQ: a first kernel rotates K once, 16-byte vector by vector, and the
//    attention rotates only its Q tile, which no other CTA reads
//    (rope3d_na3d_rotate_once). Every element is rotated once and Q_out is
//    never written: the fastest of the three.
//
// Neighbourhood attention as published (Hassani et al., "Neighborhood Attention
// Transformer", CVPR 2023): a query at (t, h, w) attends to the k_t x k_h x k_w
// window centred on it, shifted inside the grid at the borders (start
// min(max(i - k/2, 0), L - k) per axis), with softmax(q.k / sqrt(d)) weights.
//
// Work decomposition: a CTA of 4 warps owns one (batch, head) and a block of
// 1 x 8 x 8 query tokens; each warp holds 2 x 8 of them (16 MMA rows), so the
// union of its windows spans whole rows of the block's key region. The region
// (the union of the block's windows) is visited in chunks of region rows (at
// most 64 key slots, 16 per row); inside a chunk a warp's keys are one
// contiguous run of slots, and the warp runs its MMAs on that run only.
// S = Q K^T and O += P V run on the tensor cores as bf16 m16n8k16 MMAs with
// fp32 accumulators, with a flash-style online softmax in registers and a
// per-element window mask. Chunks are double-buffered: the next chunk's K and
// V are copied asynchronously while the current one is computed; when
// rotating, each thread then rotates the K vectors it copied, in place.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "../../include/rope3d.h"
#include "rope3d_internal.h"

// Tuning: resident CTAs per SM the register allocation aims at (the
// unrotated kernel fits three in shared memory; the rotating one, with its
// tables, two), and log2 of the largest softmax weight before a rescale.
#ifndef NA_MIN_CTAS
#define NA_MIN_CTAS 3
#endif
#ifndef NA_MIN_CTAS_ROPE
#define NA_MIN_CTAS_ROPE 2
#endif
#ifndef NA_TC_SUSPEND_NS   // time limit hint of the tensor-core kernel's mbarrier waits
#define NA_TC_SUSPEND_NS 1000
#endif
#ifndef NA_LAZY
#define NA_LAZY 8.0f
#endif

namespace {

constexpr int kHD = 128;             // head_dim
constexpr int kQB = 64;              // queries per CTA (1 x 8 x 8)
constexpr int kQBH = 8, kQBW = 8;
constexpr int kKC = 64;              // at most this many keys per chunk
constexpr int kWarps = 4;            // warp i: block rows 2i and 2i + 1
constexpr int kThreads = kWarps * 32;
constexpr int kRow = kHD + 8;        // padded smem row (bf16): 272 bytes
constexpr int kVecs = kKC * (kHD / 8) / kThreads;   // 16-byte vectors per thread per chunk
constexpr uint32_t kMaxTableBytes = 48 * 1024;
constexpr float kLazy = NA_LAZY;     // log2 of the largest weight before a rescale
constexpr size_t kFixedSmem = size_t(4) * kKC * kRow * 2;   // K and V, two buffers each
static_assert(kQB == kQBH * kQBW && kQB == kWarps * 16 && kQBW == 8,
              "a warp holds two 8-wide rows of the query block");
static_assert(kVecs * kThreads == kQB * (kHD / 8), "the Q tile and a K chunk move alike");

struct NAParams {
    const uint16_t *q, *k, *v;
    uint16_t *out;
    const float2 *tab;
    uint32_t tab_len, offH, offW, pT, pH, pW;
    int B, T, H, W, heads;
    int kt, kh, kw;
    int nbh, nbw;            // query blocks along H and W
    float scale_log2;        // log2(e) / sqrt(head_dim)
    unsigned long long total;   // elements of each of q, k, v, out (debug bound checks)
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

// The tables in shared memory. Each position's row of an axis holds its P
// (cos, sin) entries split in two halves: the first two entries of every
// group of four pairs, then the last two. A thread's group g of a row is
// then one 16-byte load at 2 g and one at P / 2 + 2 g, and the threads of a
// warp, which take consecutive groups, read consecutive 16-byte words
// (interleaved groups put their loads 32 bytes apart: bank conflicts).
//
// Where a thread's 8 channels [8 cv, 8 cv + 8) read: every chunk of the
// split is a multiple of 8 channels, so the 4 pairs (group g of its axis) lie
// in one axis; the row of position pos starts at off + pos * P.
struct TabSlot {
    uint32_t base, stride, half;   // off + 2 g, P, P / 2
    int axis;                      // 0: t, 1: h, 2: w
};

__device__ __forceinline__ TabSlot tab_slot(const NAParams &p, int cv) {
    const uint32_t pair = 4 * cv;
    if (pair < p.pT) return {pair / 2, p.pT, p.pT / 2, 0};
    if (pair < p.pT + p.pH) return {p.offH + (pair - p.pT) / 2, p.pH, p.pH / 2, 1};
    return {p.offW + (pair - p.pT - p.pH) / 2, p.pW, p.pW / 2, 2};
}

// The same for the tables as they lie in global memory: row pos of an axis
// holds its P entries in pair order, so the 4 pairs of channel block cv
// (pair index j of the axis) are the 16-byte words at off + pos P + j and
// 2 entries further.
__device__ __forceinline__ TabSlot tab_slot_global(uint32_t pT, uint32_t pH, uint32_t pW,
                                                   uint32_t offH, uint32_t offW, int cv) {
    const uint32_t pair = 4 * cv;
    if (pair < pT) return {pair, pT, 2, 0};
    if (pair < pT + pH) return {offH + (pair - pT), pH, 2, 1};
    return {offW + (pair - pT - pH), pW, 2, 2};
}

// Copy the tables into shared memory in the split layout above: one group
// of four pairs (two 16-byte words) per step.
__device__ __forceinline__ void stage_tables(const NAParams &p, float2 *dst, int tid, int nthreads) {
    const uint32_t groups = p.tab_len / 4;
    for (uint32_t gi = tid; gi < groups; gi += nthreads) {
        const uint32_t e = 4 * gi;   // first entry of the group
        uint32_t off, P;
        if (e < p.offH) off = 0, P = p.pT;
        else if (e < p.offW) off = p.offH, P = p.pH;
        else off = p.offW, P = p.pW;
        const uint32_t pos = (e - off) / P, pair = (e - off) - pos * P;
        const uint32_t row = off + pos * P;
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p.tab + e));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p.tab + e + 2));
        *reinterpret_cast<float4 *>(dst + row + pair / 2) = a;
        *reinterpret_cast<float4 *>(dst + row + P / 2 + pair / 2) = b;
    }
}

// Debug builds (-DROPE3D_DEBUG_BOUNDS=1) check each computed index before the
// access it guards: a failed check counts in this file's error word and skips
// the access (never a trap). Otherwise every check compiles away.
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

// Rotate the 8 channels of a TabSlot at position pos of its axis (tables of
// len entries; kGlobal: read through the read-only data path, else shared).
template <bool kGlobal>
__device__ __forceinline__ uint4 rot_vec_at(uint4 v, const float2 *tab, const TabSlot &ts,
                                            uint32_t pos, uint32_t len) {
    const uint32_t idx = ts.base + pos * ts.stride;
    if (!bound_ok(idx, 2, len) || !bound_ok(idx + ts.half, 2, len)) return v;
    float4 a, b;
    if constexpr (kGlobal) {
        a = __ldg(reinterpret_cast<const float4 *>(tab + idx));
        b = __ldg(reinterpret_cast<const float4 *>(tab + idx + ts.half));
    } else {
        a = *reinterpret_cast<const float4 *>(tab + idx);
        b = *reinterpret_cast<const float4 *>(tab + idx + ts.half);
    }
    return make_uint4(rot_word(v.x, a.x, a.y), rot_word(v.y, a.z, a.w), rot_word(v.z, b.x, b.y),
                      rot_word(v.w, b.z, b.w));
}

// The same for a token at grid position (t, h, w), tables in shared memory.
__device__ __forceinline__ uint4 rot_vec(uint4 v, const float2 *tab, const TabSlot &ts, int t,
                                         int h, int w, uint32_t len) {
    const int pos = ts.axis == 0 ? t : (ts.axis == 1 ? h : w);
    return rot_vec_at<false>(v, tab, ts, uint32_t(pos), len);
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous copy global -> shared (bypassing registers and L1).
__device__ __forceinline__ void cp_async16(void *dst_smem, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst_smem)), "l"(src)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
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

// 2^x on the special-function unit (relative error about 2^-22; results below
// the smallest normal flush to zero, far under the bf16 rounding of P).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The largest of three floats (one three-input max instruction).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float y;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
    return y;
}

// S = Q K^T over NQ 16-key steps (keys q * 16 .. q * 16 + 15 of the warp's
// run start at kaddr + q * 16 rows), software-pipelined: the B fragments of
// k-step ks + 1 are loaded while the MMAs of k-step ks issue.
template <int NQ>
__device__ __forceinline__ void qk_steps(float (&s)[kKC / 8][4], const uint32_t (&qa)[kHD / 16][4],
                                         uint32_t kaddr) {
    uint32_t bf[2][NQ][4];
#pragma unroll
    for (int q = 0; q < NQ; ++q)
        ldsm_x4(kaddr + q * 16 * kRow * 2, bf[0][q][0], bf[0][q][1], bf[0][q][2], bf[0][q][3]);
#pragma unroll
    for (int ks = 0; ks < kHD / 16; ++ks) {
        const int cb = ks & 1;
        if (ks + 1 < kHD / 16) {
#pragma unroll
            for (int q = 0; q < NQ; ++q)
                ldsm_x4(kaddr + q * 16 * kRow * 2 + (ks + 1) * 32, bf[cb ^ 1][q][0], bf[cb ^ 1][q][1],
                        bf[cb ^ 1][q][2], bf[cb ^ 1][q][3]);
        }
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            mma(s[2 * q], qa[ks], bf[cb][q][0], bf[cb][q][1]);
            mma(s[2 * q + 1], qa[ks], bf[cb][q][2], bf[cb][q][3]);
        }
    }
}

// O += P V over NQ 16-key steps (P from the S registers, rounded to bf16),
// software-pipelined over the 8 column blocks of V in the same way.
template <int NQ>
__device__ __forceinline__ void pv_steps(float (&o)[kHD / 8][4], const float (&s)[kKC / 8][4],
                                         uint32_t vaddr) {
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        uint32_t pa[4];
        pa[0] = pack_bf16(s[2 * q][0], s[2 * q][1]);
        pa[1] = pack_bf16(s[2 * q][2], s[2 * q][3]);
        pa[2] = pack_bf16(s[2 * q + 1][0], s[2 * q + 1][1]);
        pa[3] = pack_bf16(s[2 * q + 1][2], s[2 * q + 1][3]);
        uint32_t bf[2][4];
        ldsm_x4_t(vaddr + q * 16 * kRow * 2, bf[0][0], bf[0][1], bf[0][2], bf[0][3]);
#pragma unroll
        for (int np = 0; np < kHD / 16; ++np) {
            const int cb = np & 1;
            if (np + 1 < kHD / 16)
                ldsm_x4_t(vaddr + q * 16 * kRow * 2 + (np + 1) * 32, bf[cb ^ 1][0], bf[cb ^ 1][1],
                          bf[cb ^ 1][2], bf[cb ^ 1][3]);
            mma(o[2 * np], pa, bf[cb][0], bf[cb][1]);
            mma(o[2 * np + 1], pa, bf[cb][2], bf[cb][3]);
        }
    }
}

// A chunk of the key region: frame t, region rows rb + i S (i < nr; ri = rb
// minus the region's first row), columns [c0, c0 + cw), nseg 16-slot segments
// per row; key (i, j) sits in slot i * 16 nseg + j.
struct Chunk {
    int t, rb, ri, nr, c0, cw, nseg;
};

// What the attention kernel rotates: nothing (Q and K come rotated), Q and
// every K tile it copies, or Q alone (K was rotated once beforehand by
// rope3d_na3d_rotate_k_kernel; the launch then waits for that kernel before
// its first copy of K).
enum RotMode : int { kRotNone = 0, kRotQK = 1, kRotQ = 2 };

template <int kMode>
__global__ void __launch_bounds__(kThreads, kMode == kRotQK ? NA_MIN_CTAS_ROPE : NA_MIN_CTAS)
rope3d_na3d_kernel(const NAParams p) {
    constexpr bool kRotK = kMode == kRotQK;
    extern __shared__ __align__(16) unsigned char smem[];
    uint16_t *sK = reinterpret_cast<uint16_t *>(smem);        // [2][kKC][kRow]
    uint16_t *sV = sK + 2 * kKC * kRow;                        // [2][kKC][kRow]
    float2 *sTab = reinterpret_cast<float2 *>(sV + 2 * kKC * kRow);
    uint16_t *sQ = sV + kKC * kRow;   // the Q tile borrows V's second buffer

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

    // A thread moves channel block cv of tile slots slot0 + 8 m (16 threads
    // per 256-byte row: coalesced).
    const int cv = tid & 15, slot0 = tid >> 4;
    const TabSlot ts = tab_slot(p, cv);
    const float2 *tab = sTab;
    const long long tok = (long long)p.heads * kHD;             // elements per token
    const long long grid_row = (long long)p.W * tok, frame = (long long)p.H * grid_row;
    const long long batch0 = (long long)b * p.T * frame + (long long)head * kHD + cv * 8;

    // Key region: the union of the block's windows. It is visited in chunks of
    // at most kKC key slots; a region row takes 16 slots per 16 columns (the
    // slots past its last column hold zeros), so one k16 MMA step covers 16
    // columns of one row. Chunk ri of a frame holds the rows ri, ri + S,
    // ri + 2 S, ...: a warp's windows span consecutive rows, which meet every
    // chunk in about the same number of rows, so the warps share each chunk's
    // work evenly. A row wider than kKC columns is cut into column groups.
    const int rt0 = na_start(qt, p.T, p.kt);
    const int hl = min(h0 + kQBH, p.H) - 1, wl = min(w0 + kQBW, p.W) - 1;
    const int rh0 = na_start(h0, p.H, p.kh), rh1 = na_start(hl, p.H, p.kh) + p.kh;
    const int rw0 = na_start(w0, p.W, p.kw), rw1 = na_start(wl, p.W, p.kw) + p.kw;
    const int RH = rh1 - rh0, RW = rw1 - rw0;
    const int CW = min(RW, kKC);                                // columns per chunk row
    const int CH = min(RH, kKC / (16 * ((CW + 15) / 16)));       // rows per chunk (>= 1)
    const int S = (RH + CH - 1) / CH, ncc = (RW + CW - 1) / CW;
    const int n_chunks = p.kt * S * ncc;
    const int qR = RH / S, mR = RH - qR * S;   // chunk ri holds qR + (ri < mR) rows
    // chunks in order: column group fastest, then ri, then the frame
    int it_ci = 0, it_ri = 0, it_dt = 0;
    auto next_chunk = [&]() {
        Chunk k;
        k.t = rt0 + it_dt;
        k.ri = it_ri;
        k.rb = rh0 + it_ri;
        k.nr = qR + (it_ri < mR ? 1 : 0);
        k.c0 = rw0 + it_ci * CW;
        k.cw = min(CW, rw1 - k.c0);
        k.nseg = (k.cw + 15) >> 4;
        if (++it_ci == ncc) {
            it_ci = 0;
            if (++it_ri == S) {
                it_ri = 0;
                ++it_dt;
            }
        }
        return k;
    };

    // K and V of a chunk are copied asynchronously. Slots past a row's last
    // column get zeros, so every slot a warp reads holds finite values.
    int kpos[kVecs];   // packed (h, w) of a K vector to rotate, else -1
    auto issue = [&](const Chunk &k, int buf) {
        const int sw = 16 * k.nseg;
        long long off = batch0 + k.t * frame + k.rb * grid_row + (long long)(k.c0 + slot0) * tok;
        const long long wrap = S * grid_row - sw * tok;   // to the chunk's next row
        int i = 0, j = slot0;                               // slot0 < 8 < sw
#pragma unroll
        for (int m = 0; m < kVecs; ++m) {
            const int slot = slot0 + 8 * m;
            uint16_t *dk = sK + (buf * kKC + slot) * kRow + cv * 8;
            uint16_t *dv = sV + (buf * kKC + slot) * kRow + cv * 8;
            if (kRotK) kpos[m] = -1;
            if (i < k.nr) {
                if (j < k.cw) {
                    if (bound_ok(off, 8, p.total) && bound_ok(slot, 1, kKC)) {
                        cp_async16(dk, p.k + off);
                        cp_async16(dv, p.v + off);
                    }
                    if (kRotK) kpos[m] = ((k.rb + i * S) << 10) | (k.c0 + j);
                } else {
                    *reinterpret_cast<uint4 *>(dk) = make_uint4(0, 0, 0, 0);
                    *reinterpret_cast<uint4 *>(dv) = make_uint4(0, 0, 0, 0);
                }
            }
            j += 8;
            off += 8 * tok;
            if (j >= sw) {
                j -= sw;
                ++i;
                off += wrap;
            }
        }
    };
    // Rotating path: a thread waits for its own copies of K and rotates them
    // in place (no other thread touches those 16-byte vectors).
    auto rotate_k = [&](int t, int buf) {
        cp_async_wait_all();
#pragma unroll
        for (int m = 0; m < kVecs; ++m) {
            const int pos = kpos[m];
            if (pos >= 0) {
                uint4 *ptr = reinterpret_cast<uint4 *>(sK + (buf * kKC + slot0 + 8 * m) * kRow + cv * 8);
                *ptr = rot_vec(*ptr, tab, ts, t, pos >> 10, pos & 1023, p.tab_len);
            }
        }
    };

    // ---- prologue: tables, the Q tile, the first chunk
    if (kRotK) stage_tables(p, sTab, tid, kThreads);
    uint4 qreg[kVecs];
    // Q rotated here (kRotQ): a thread's vectors are the block rows m of one
    // column, (h0 + m, w0 + slot0), so its T or W table words are the same for
    // all of them and are loaded once; H words are loaded per row.
    const TabSlot tsg = tab_slot_global(p.pT, p.pH, p.pW, p.offH, p.offW, cv);
    const bool col_ok = w0 + slot0 < p.W;
    float4 qta[kMode == kRotQ ? kVecs : 1], qtb[kMode == kRotQ ? kVecs : 1];
    if constexpr (kMode == kRotQ) {
        qta[0] = qtb[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (tsg.axis != 1 && col_ok) {
            const uint32_t idx = tsg.base + uint32_t(tsg.axis == 0 ? qt : w0 + slot0) * tsg.stride;
            if (bound_ok(idx, 4, p.tab_len)) {
                qta[0] = __ldg(reinterpret_cast<const float4 *>(p.tab + idx));
                qtb[0] = __ldg(reinterpret_cast<const float4 *>(p.tab + idx + 2));
            }
        }
    }
#pragma unroll
    for (int m = 0; m < kVecs; ++m) {
        const int r = slot0 + 8 * m;   // block row r: (h0 + r / 8, w0 + r % 8)
        const int h = h0 + r / kQBW, w = w0 + r % kQBW;
        qreg[m] = make_uint4(0, 0, 0, 0);
        const long long qo = batch0 + qt * frame + h * grid_row + (long long)w * tok;
        if (h < p.H && w < p.W && bound_ok(qo, 8, p.total))
            qreg[m] = __ldg(reinterpret_cast<const uint4 *>(p.q + qo));
        if constexpr (kMode == kRotQ) {
            if (tsg.axis == 1) {
                const uint32_t idx = tsg.base + uint32_t(h) * tsg.stride;
                qta[m] = qtb[m] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (h < p.H && col_ok && bound_ok(idx, 4, p.tab_len)) {
                    qta[m] = __ldg(reinterpret_cast<const float4 *>(p.tab + idx));
                    qtb[m] = __ldg(reinterpret_cast<const float4 *>(p.tab + idx + 2));
                }
            } else if (m > 0) {
                qta[m] = qta[0];
                qtb[m] = qtb[0];
            }
        }
    }
    // K comes from the kernel before this one in the stream (launched with
    // programmatic serialization): wait for it before the first copy.
    if (kMode == kRotQ) asm volatile("griddepcontrol.wait;" ::: "memory");
    Chunk cur = next_chunk();
    issue(cur, 0);
    cp_async_commit();
    if (kRotK) __syncthreads();   // tables staged
#pragma unroll
    for (int m = 0; m < kVecs; ++m) {
        const int r = slot0 + 8 * m;
        const int h = h0 + r / kQBW, w = w0 + r % kQBW;
        uint4 v = qreg[m];
        if (h < p.H && w < p.W) {
            if constexpr (kMode == kRotQK) v = rot_vec(v, tab, ts, qt, h, w, p.tab_len);
            if constexpr (kMode == kRotQ) {
                const float4 a = qta[m], b = qtb[m];
                v = make_uint4(rot_word(v.x, a.x, a.y), rot_word(v.y, a.z, a.w),
                               rot_word(v.z, b.x, b.y), rot_word(v.w, b.z, b.w));
            }
        }
        *reinterpret_cast<uint4 *>(sQ + r * kRow + cv * 8) = v;
    }
    if (kRotK) rotate_k(cur.t, 0);
    __syncthreads();

    // Q fragments of this warp's 16 rows, all 8 k-steps
    uint32_t qa[kHD / 16][4];
#pragma unroll
    for (int ks = 0; ks < kHD / 16; ++ks) {
        const uint16_t *a = sQ + (warp * 16 + (lane & 15)) * kRow + ks * 16 + (lane >> 4) * 8;
        ldsm_x4(smem_addr(a), qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
    }

    // this thread's two query rows: block rows 2 warp (MMA row g) and
    // 2 warp + 1 (MMA row g + 8), both in column w0 + g
    const int hq = h0 + 2 * warp, wq = w0 + g;
    const int ww = na_start(min(wq, p.W - 1), p.W, p.kw);
    const int wh0 = na_start(min(hq, p.H - 1), p.H, p.kh);
    const int wh1 = na_start(min(hq + 1, p.H - 1), p.H, p.kh);
    const bool cvalid = wq < p.W;
    const bool rvalid0 = hq < p.H && cvalid, rvalid1 = hq + 1 < p.H && cvalid;
    // The warp's windows span region rows [box_h0, box_h1) and every column;
    // chunk ri meets them in its rows [qb + (ri < mb), qu + (ri < mu)).
    const int bl = wh0 - rh0, bu = (hq < p.H ? wh1 + p.kh : wh0) - rh0;
    const int qb = bl / S, mb = bl - qb * S, qu = bu / S, mu = bu - qu * S;
    // column tests of this lane's keys: bit 4 seg + 2 half + kq for column
    // 16 seg + 8 half + 2 tq + kq of a chunk row; recomputed per column group
    uint32_t colbits = 0;
    int colbits_c0 = -1;

    float o[kHD / 8][4];
#pragma unroll
    for (int n = 0; n < kHD / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const int mi = lane >> 3, rr = lane & 7;

    for (int c = 0; c < n_chunks; ++c) {
        const int buf = c & 1;
        cp_async_wait_all();   // this thread's copies of chunk c
        __syncthreads();       // everyone's, K stored, chunk c - 1 no longer read
        Chunk nxt{};
        if (c + 1 < n_chunks) {
            nxt = next_chunk();
            issue(nxt, buf ^ 1);
        }
        cp_async_commit();

        const int ilo = qb + (cur.ri < mb ? 1 : 0), ihi = qu + (cur.ri < mu ? 1 : 0);
        const int nq = (ihi - ilo) * cur.nseg;   // k16 steps of this warp (<= kKC / 16)
        // (debug builds: the warp's slots [16 nseg ilo, + 16 nq) lie in the buffer)
        if (nq > 0 && bound_ok(ilo * 16 * cur.nseg, 16 * nq, kKC)) {
            if (cur.c0 != colbits_c0) {
                colbits_c0 = cur.c0;
                colbits = 0;
#pragma unroll
                for (int bit = 0; bit < 16; ++bit) {
                    const int j = (bit >> 2) * 16 + ((bit >> 1) & 1) * 8 + 2 * tq + (bit & 1);
                    if (j < cur.cw && unsigned(cur.c0 + j - ww) < unsigned(p.kw)) colbits |= 1u << bit;
                }
            }
            const int j0 = ilo * 16 * cur.nseg;   // first slot
            const uint16_t *Kb = sK + (buf * kKC + j0) * kRow;
            const uint16_t *Vb = sV + (buf * kKC + j0) * kRow;

            const uint32_t kaddr = smem_addr(Kb + ((mi >> 1) * 8 + rr) * kRow + (mi & 1) * 8);
            const uint32_t vaddr = smem_addr(Vb + (rr + (mi & 1) * 8) * kRow + (mi >> 1) * 8);
            // the chunk's work for NQ 16-key steps (compiled for 1 to kKC / 16;
            // two in most chunks), step q covering slots [16 q, 16 q + 16)
            auto steps = [&](auto nq_const) {
                constexpr int NQ = decltype(nq_const)::value;
                // ---- S = Q K^T
                float s[kKC / 8][4];
#pragma unroll
                for (int n = 0; n < 2 * NQ; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
                qk_steps<NQ>(s, qa, kaddr);

                // ---- mask, online softmax. Every key of the region lies in
                // each row's t window (the block is one frame): only h and w
                // are tested.
                int hk = cur.rb + ilo * S, seg = 0;
                float cmax0 = -INFINITY, cmax1 = -INFINITY;
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    const bool row0 = rvalid0 && unsigned(hk - wh0) < unsigned(p.kh);
                    const bool row1 = rvalid1 && unsigned(hk - wh1) < unsigned(p.kh);
                    const uint32_t cb = colbits >> (4 * seg);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {   // half = e >> 2, row = (e >> 1) & 1, kq = e & 1
                        const bool col = (cb >> (((e >> 2) << 1) | (e & 1))) & 1u;
                        float &x = s[2 * q + (e >> 2)][e & 3];
                        const bool ok = col && (((e >> 1) & 1) ? row1 : row0);
                        x = ok ? x * p.scale_log2 : -INFINITY;
                    }
                    cmax0 = fmaxf(cmax0, fmaxf(fmaxf(s[2 * q][0], s[2 * q][1]),
                                               fmaxf(s[2 * q + 1][0], s[2 * q + 1][1])));
                    cmax1 = fmaxf(cmax1, fmaxf(fmaxf(s[2 * q][2], s[2 * q][3]),
                                               fmaxf(s[2 * q + 1][2], s[2 * q + 1][3])));
                    if (++seg == cur.nseg) {
                        seg = 0;
                        hk += S;
                    }
                }
                cmax0 = fmaxf(cmax0, __shfl_xor_sync(0xffffffffu, cmax0, 1));
                cmax0 = fmaxf(cmax0, __shfl_xor_sync(0xffffffffu, cmax0, 2));
                cmax1 = fmaxf(cmax1, __shfl_xor_sync(0xffffffffu, cmax1, 1));
                cmax1 = fmaxf(cmax1, __shfl_xor_sync(0xffffffffu, cmax1, 2));
                // Weights are exp2(score - ref) with ref a running reference
                // per row. The reference moves up to the row's maximum (and O
                // and l are rescaled) only when the maximum exceeds it by more
                // than kLazy, so weights stay below 2^kLazy; a row with no key
                // yet has reference -inf and subtracts 0 (every score is -inf
                // there).
                const float mn0 = fmaxf(m0, cmax0), mn1 = fmaxf(m1, cmax1);
                if (__any_sync(0xffffffffu, mn0 > m0 + kLazy || mn1 > m1 + kLazy)) {
                    const float corr0 = m0 == -INFINITY ? 0.f : ex2(m0 - mn0);
                    const float corr1 = m1 == -INFINITY ? 0.f : ex2(m1 - mn1);
                    m0 = mn0;
                    m1 = mn1;
                    l0 *= corr0;
                    l1 *= corr1;
#pragma unroll
                    for (int n = 0; n < kHD / 8; ++n) {
                        o[n][0] *= corr0;
                        o[n][1] *= corr0;
                        o[n][2] *= corr1;
                        o[n][3] *= corr1;
                    }
                }
                const float ms0 = m0 == -INFINITY ? 0.f : m0, ms1 = m1 == -INFINITY ? 0.f : m1;
                float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
#pragma unroll
                    for (int n = 2 * q; n < 2 * q + 2; ++n) {
                        s[n][0] = ex2(s[n][0] - ms0);
                        s[n][1] = ex2(s[n][1] - ms0);
                        s[n][2] = ex2(s[n][2] - ms1);
                        s[n][3] = ex2(s[n][3] - ms1);
                    }
                    ps0 += (s[2 * q][0] + s[2 * q][1]) + (s[2 * q + 1][0] + s[2 * q + 1][1]);
                    ps1 += (s[2 * q][2] + s[2 * q][3]) + (s[2 * q + 1][2] + s[2 * q + 1][3]);
                }
                ps0 += __shfl_xor_sync(0xffffffffu, ps0, 1);
                ps0 += __shfl_xor_sync(0xffffffffu, ps0, 2);
                ps1 += __shfl_xor_sync(0xffffffffu, ps1, 1);
                ps1 += __shfl_xor_sync(0xffffffffu, ps1, 2);
                l0 += ps0;
                l1 += ps1;

                // ---- O += P V
                pv_steps<NQ>(o, s, vaddr);
            };
            switch (nq) {
                case 1: steps(std::integral_constant<int, 1>{}); break;
                case 2: steps(std::integral_constant<int, 2>{}); break;
                case 3: steps(std::integral_constant<int, 3>{}); break;
                default: steps(std::integral_constant<int, 4>{}); break;
            }
        }
        if (kRotK && c + 1 < n_chunks) rotate_k(nxt.t, buf ^ 1);
        cur = nxt;
    }

    // ---- normalise into a shared-memory tile (over K's first buffer, free
    // once every warp is past the last chunk), then store it as coalesced
    // 16-byte vectors, 16 threads per 256-byte row
    __syncthreads();
    uint16_t *sO = sK;   // [kQB][kRow]; block row r = warp 16 + 8 half + g
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const float l = r == 0 ? l0 : l1;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint16_t *row = sO + (warp * 16 + 8 * r + g) * kRow + 2 * tq;
#pragma unroll
        for (int n = 0; n < kHD / 8; ++n)
            *reinterpret_cast<uint32_t *>(row + n * 8) =
                pack_bf16(o[n][2 * r] * inv, o[n][2 * r + 1] * inv);
    }
    __syncthreads();
    // (not unrolled: unrolled, this loop made ptxas spill 96 bytes and the
    // kernel 16 % slower)
    const int hb = hq - 2 * warp, wb = wq - g;   // the block's first row and column
#pragma unroll 1
    for (int m = 0; m < kVecs; ++m) {
        const int r = slot0 + 8 * m;
        const int h = hb + r / kQBW, w = wb + r % kQBW;
        const long long oo = batch0 + qt * frame + h * grid_row + (long long)w * tok;
        if (h < p.H && w < p.W && bound_ok(oo, 8, p.total))
            *reinterpret_cast<uint4 *>(p.out + oo) =
                *reinterpret_cast<const uint4 *>(sO + r * kRow + cv * 8);
    }
}

// ---- K rotated once, before the attention (rope3d_na3d_rotate_once) -------
// K [tokens, heads, 128] bf16 is rotated vector by vector into k_rot with the
// eager arithmetic above; one launch covers a whole number of tokens.
struct RKParams {
    const uint4 *k;
    uint4 *k_rot;
    const float2 *tab;
    uint32_t tab_len, offH, offW, pT, pH, pW;
    uint32_t units;                  // 16-byte vectors of this launch (< 2^30)
    uint32_t tok0;                   // grid index (t H + h) W + w of the first token
    rope3d::FastDiv heads, Wd, Hd, HWd, Td;
};

constexpr int kRotThreads = 512, kRotUnroll = 4;
static_assert(kRotThreads % (kHD / 8) == 0, "a thread keeps one channel block");

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const rope3d::FastDiv &f) {
    return (__umulhi(n, f.mul) + n) >> f.shift;
}

// Plain (coherent) loads: k_rot may be k itself.
__device__ __forceinline__ uint4 ld_v4(const uint4 *ptr) {
    uint4 r;
    asm volatile("ld.global.L1::no_allocate.L2::128B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(ptr)
                 : "memory");
    return r;
}

// Grid coordinate on `axis` of the token of vector vv.
__device__ __forceinline__ uint32_t axis_pos(const RKParams &p, uint32_t vv, int axis) {
    const uint32_t gt = p.tok0 + fdiv(vv >> 4, p.heads);   // < 2^31
    if (axis == 2) return gt - fdiv(gt, p.Wd) * p.Wd.d;
    if (axis == 1) {
        const uint32_t r = fdiv(gt, p.Wd);
        return r - fdiv(r, p.Hd) * p.Hd.d;
    }
    const uint32_t r = fdiv(gt, p.HWd);
    return r - fdiv(r, p.Td) * p.Td.d;
}

__global__ void __launch_bounds__(kRotThreads, 3) rope3d_na3d_rotate_k_kernel(const RKParams p) {
    // The attention kernel may launch now; it waits for this grid to finish
    // before it reads K.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint32_t stride = gridDim.x * kRotThreads;   // a multiple of 16
    uint32_t v = blockIdx.x * kRotThreads + threadIdx.x;
    const TabSlot ts = tab_slot_global(p.pT, p.pH, p.pW, p.offH, p.offW, int(v & 15));
    for (; v + (kRotUnroll - 1) * stride < p.units; v += kRotUnroll * stride) {
        uint4 x[kRotUnroll];
#pragma unroll
        for (int u = 0; u < kRotUnroll; ++u)
            if (bound_ok(v + u * stride, 1, p.units)) x[u] = ld_v4(p.k + v + u * stride);
#pragma unroll
        for (int u = 0; u < kRotUnroll; ++u) {
            const uint32_t vv = v + u * stride;
            if (!bound_ok(vv, 1, p.units)) continue;
            p.k_rot[vv] = rot_vec_at<true>(x[u], p.tab, ts, axis_pos(p, vv, ts.axis), p.tab_len);
        }
    }
    for (; v < p.units; v += stride)
        p.k_rot[v] = rot_vec_at<true>(ld_v4(p.k + v), p.tab, ts, axis_pos(p, v, ts.axis), p.tab_len);
}

// ---- the attention on the fifth-generation tensor cores -------------------
// A query block is one (batch, head) and 2 x 8 x 8 queries: the 128 rows of a
// tcgen05 MMA (M = 128). The union of the block's windows (its key region) is
// streamed in chunks of whole region rows of one frame, at most kTcN keys
// each. One persistent CTA per SM walks the blocks blockIdx.x, + gridDim.x,
// ...; its warps have one job each and hand work over through mbarriers
// (counted over the CTA's whole sequence of chunks and blocks), so that the
// tensor cores, the copies and the softmax overlap, also across blocks:
//   warps 0 and 3 (one thread each): TMA copies of each chunk's K (warp 0)
//     and V (warp 3), two boxes each, one per 64 channels, with the 128-byte
//     swizzle, into two-slot rings;
//   warp 1 (one thread): the P V MMAs, O += P(c) V(c) (V read as an MN-major
//     operand), once the softmax has written P(c);
//   warp 2 (one thread): the S MMAs, S(c) = Q K(c)^T into one of three S
//     buffers in tensor memory (eight k16 steps), as soon as K(c) has landed
//     and P V has read the weights of chunk c - 3 out of that buffer. Two
//     issuing threads keep either kind of product from waiting behind the
//     other's inputs; S(c + 1) and S(c + 2) run while the softmax of chunk c
//     does;
//   warps 4-7: each query block's Q tile, copied by TMA into its Q buffer
//     while the previous block still uses the other (and rotated in place in
//     the rotating modes); each block's descriptor for the softmax, a block
//     ahead; each block's O, normalised, through its spent Q buffer and two
//     TMA stores; in the mode that rotates K per CTA, each K tile too, in
//     place once it lands;
//   warps 8-15: the softmax. Each query row's S is read back from tensor
//     memory by two threads (half of the chunk's columns each, in one batch of
//     loads: warps w and w + 4 share the 32 lanes of tensor memory that warp w
//     reaches), masked to the query's window (a 64-bit mask from the region
//     rows the half spans; a warp none of whose rows has a key in the chunk
//     skips it), scaled, and turned into weights with the same online
//     softmax as the warp-MMA kernel (the reference moves only when a row maximum passes it
//     by more than 2^kLazy; O in tensor memory is rescaled then); the bf16
//     weights are written back into the S buffer they came from (over the S
//     values, as bf16 pairs), where the P V MMA reads them as its A operand.
// Q stays in shared memory for every chunk of its block; the next block's Q
// is written into the other buffer meanwhile.
// Shared memory (bytes; every tile 1024-aligned, the swizzle's period):
//   Q  [2 buffers][2 column blocks][128 rows][128 B]    65,536
//   K  [2 slots][2 column blocks][kTcN rows][128 B]     57,344
//   V  [2 slots][2 column blocks][kTcN rows][128 B]     57,344
//   row maxima and sums of the row's two threads, the softmax threads' window
//   masks (3 sets of 4 KB per chunk row offset, up to 4 offsets), two block
//   descriptors, 36 mbarriers, the TMEM address.
// Tensor memory (512 columns): three S buffers at columns 0, 128 and 256 (S,
// then P in their first 56 columns), so that the S products run up to two
// chunks ahead of the softmax while P V reads the third; O at 384 (a block's
// first P V waits for the Q warps to have read the previous block's O out).
constexpr int kTcParts = 2;                  // softmax threads per query row
constexpr int kTcQBar = 5;                   // named barrier of the Q warps (1-4: softmax pairs)
constexpr int kTcSoftWarp0 = 8;              // first softmax warp
constexpr int kTcRotThreads = 128;           // warps 4-7
constexpr int kTcSoftThreads = 128 * kTcParts;
// 16 warps: K TMA, P V MMA, S MMA, V TMA, 4 Q warps, 8 softmax warps
constexpr int kTcThreads = 256 + kTcSoftThreads;
constexpr int kTcM = 128;                    // queries per CTA: 2 x 8 x 8
constexpr int kTcQT = 2, kTcQH = 8, kTcQW = 8;
constexpr int kTcN = 112;                    // keys per chunk at most
constexpr int kTcHalf = kTcN / kTcParts;     // columns of a chunk a softmax thread takes
constexpr uint32_t kTcQCb = kTcM * 128;      // bytes of a column block of Q or P
constexpr uint32_t kTcKvCb = kTcN * 128;     // bytes of a column block of K or V
constexpr uint32_t kTcKvSlot = 2 * kTcKvCb;  // bytes of a K or V slot
constexpr uint32_t kTcOffQ = 0;
constexpr uint32_t kTcOffK = kTcOffQ + 4 * kTcQCb;        // two Q buffers (block parity)
constexpr uint32_t kTcOffV = kTcOffK + 2 * kTcKvSlot;
// float row maxima [chunk parity][part][128], row sums [block parity][part][128]
constexpr uint32_t kTcOffRed = kTcOffV + 2 * kTcKvSlot;
// the softmax threads' window masks of a block's chunk row offsets (frames
// share them): [set][offset][part][128] 64-bit words, each thread its own;
// a set per window geometry the thread has met lately
constexpr int kTcMaxPF = 4;                                 // offsets kept; more: made per chunk
constexpr int kTcMaskSets = 3;
constexpr uint32_t kTcOffMask = kTcOffRed + 4 * kTcParts * kTcM * 4;
// block descriptors for the softmax threads, written by the Q warps a block
// ahead: [block parity] {first region frame, region rows, chunks per frame,
// chunks}, then per query row {in the grid, first window frame, window's first
// region row, window columns [lo, hi) packed}
constexpr uint32_t kTcDescSlot = 16 + kTcM * 16;
constexpr uint32_t kTcOffDesc = kTcOffMask + kTcMaskSets * kTcMaxPF * kTcSoftThreads * 8;
constexpr int kTcBars = 36;                                 // mbarriers, then the TMEM address
constexpr uint32_t kTcOffBar = kTcOffDesc + 2 * kTcDescSlot;
constexpr uint32_t kTcSmem = kTcOffBar + kTcBars * 8 + 16 + 1024;   // + room to align to 1024
#ifndef NA_TC_SBUFS   // S buffers in tensor memory: 3 (O single) or 2 (O double-buffered)
#define NA_TC_SBUFS 3
#endif
constexpr int kTcSBufs = NA_TC_SBUFS;
constexpr int kTcOBufs = kTcSBufs == 3 ? 1 : 2;             // O buffers
constexpr uint32_t kTcColS = 128;                           // S buffer b at column b * 128
constexpr uint32_t kTcColO = kTcSBufs * kTcColS;            // O buffer b at kTcColO + 128 b
constexpr uint32_t kTcTmemCols = 512;
constexpr int kTcMaxRW = kTcN;                              // a region row must fit a chunk
static_assert(kTcKvCb % 1024 == 0 && kTcOffK % 1024 == 0 && kTcOffV % 1024 == 0 &&
              kTcOffRed % 1024 == 0, "1024-aligned tiles");
static_assert(kTcN % 16 == 0 && kTcN <= int(kTcColS), "an S buffer holds a chunk");
static_assert(kTcColO + 128 * kTcOBufs <= kTcTmemCols, "S and O fit the allocation");
static_assert(kTcSmem + 1024 <= 228 * 1024, "one CTA per SM");
static_assert((128 / kTcParts) % 16 == 0, "O columns per thread");
static_assert(kTcParts == 2 && kTcHalf == 56, "a half row: 32 + 16 + 8 columns, a 64-bit mask");

// Waits that gave up (a bounded wait on an MMA completion ran out); they are
// counted here and reported by rope3d_testing_na3d_wait_timeouts.
__device__ unsigned int g_na3d_wait_timeouts;

// Shared-memory matrix descriptor of a tcgen05 operand: start address, the
// leading and stride byte offsets (all in 16-byte units, 14 bits), the fixed
// 0b001 at bits 46-48, and the 128-byte swizzle (2) in bits 61-63.
__device__ __forceinline__ uint64_t tc_sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t((lbo & 0x3FFFFu) >> 4) << 16) |
           (uint64_t((sbo & 0x3FFFFu) >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of a kind::f16 MMA: fp32 accumulators (bits 4-5 =
// 1), bf16 A and B (bits 7-9, 10-12 = 1), B read MN-major when b_mn (bit 16),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__device__ __forceinline__ uint32_t tc_idesc(uint32_t m, uint32_t n, uint32_t b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn << 16) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}

// The same with A (M x 16, K-major, two bf16 per 32-bit column) read from
// tensor memory at a_tmem.
__device__ __forceinline__ void tc_mma_ta(uint32_t tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory writes of this thread (plain stores and completed cp.async
// copies) become visible to the tensor cores' reads.
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The mbarrier's next phase completes once this arrival has happened and
// `bytes` have been written by the copies that name it.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    uint64_t state;
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 %0, [%1], %2;"
                 : "=l"(state) : "r"(bar), "r"(bytes) : "memory");
    asm volatile("" ::"l"(state));   // the arrival state is not needed
}

// One arrival on an mbarrier (release semantics at CTA scope: this thread's
// earlier writes are visible to whoever waits for the phase).
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    uint64_t state;
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 %0, [%1];" : "=l"(state) : "r"(bar) : "memory");
    asm volatile("" ::"l"(state));
}

// One TMA tile of a 5-D tensor map (channels, head, w, h, frame) into shared
// memory, completing on `bar`. The channel coordinate is 0 or 64: 0 or 128
// bytes, a multiple of 16 as TMA requires.
__device__ __forceinline__ void tma_load5(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                          int c2, int c3, int c4, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
          "r"(c4), "r"(bar)
        : "memory");
}

// A 5-D tile store from shared memory (a bulk group of this thread), its
// commit, and the waits for the group's shared-memory reads or its completion.
__device__ __forceinline__ void tma_store5(const CUtensorMap *map, uint32_t src, int c0, int c1,
                                           int c2, int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4, %5}], [%6];"
        ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(src)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Whether phase `parity` of an mbarrier has completed (no waiting).
__device__ __forceinline__ bool mbar_done(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    return done != 0;
}

// Wait for phase `parity` of an mbarrier for at most ~0.1 s of SM clocks.
// Returns false (and counts) when it gave up; `dead` then skips every later
// wait of this thread, so a CTA whose MMAs never complete still ends.
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, bool &dead) {
    if (dead) return false;
    {
        uint32_t done;   // the phase has usually completed already
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done) : "r"(bar), "r"(parity) : "memory");
        if (done) return true;
    }
    const long long t0 = clock64();
    while (true) {
        uint32_t done;
#if NA_TC_SUSPEND_NS > 0
        // the thread may be suspended for up to this long while it waits
        // (fewer issue slots spent spinning)
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done) : "r"(bar), "r"(parity), "n"(NA_TC_SUSPEND_NS) : "memory");
#else
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done) : "r"(bar), "r"(parity) : "memory");
#endif
        if (done) return true;
        if (clock64() - t0 > 200000000ll) {
            atomicAdd(&g_na3d_wait_timeouts, 1u);
            dead = true;
            return false;
        }
    }
}

// 16 consecutive fp32 columns of this warp's 32 lanes of tensor memory (lane
// = thread), read and waited for.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 and 8 consecutive fp32 columns, not waited for (tc_ld_wait_hold follows).
__device__ __forceinline__ void tc_ld32_async(uint32_t taddr, float *v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
        "%29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_ld8_async(uint32_t taddr, float *v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_ld16_async(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}


// Wait for this thread's tensor-memory loads; the n registers of v pass
// through the asm so that no use of them moves above the wait.
template <int n>
__device__ __forceinline__ void tc_ld_wait_hold(float *v) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < n; ++i) asm volatile("" : "+f"(v[i]));
}

__device__ __forceinline__ void tc_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};"
        ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
          "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])),
          "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
          "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
          "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
          "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
        : "memory");
}

// 16, 8 or 4 consecutive 32-bit columns of this warp's 32 lanes of tensor
// memory (lane = thread), from registers; tcgen05.wait::st completes them.
__device__ __forceinline__ void tc_st16w(uint32_t taddr, const uint32_t *w) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};"
        ::"r"(taddr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
          "r"(w[7]), "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]),
          "r"(w[15])
        : "memory");
}
__device__ __forceinline__ void tc_st8w(uint32_t taddr, const uint32_t *w) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 ::"r"(taddr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),
                   "r"(w[6]), "r"(w[7])
                 : "memory");
}
__device__ __forceinline__ void tc_st4w(uint32_t taddr, const uint32_t *w) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};"
                 ::"r"(taddr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                 : "memory");
}

// Byte offset of 16-byte chunk c (0..15: 8 elements each) of row `row` in a
// K-major tile with the 128-byte swizzle: chunk c lies in column block c / 8,
// and inside a 128-byte row the chunk index is XORed with row mod 8.
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t c, uint32_t cb_bytes) {
    return (c >> 3) * cb_bytes + row * 128 + (((c & 7) ^ (row & 7)) << 4);
}

// n / d by the multiply-high method of rope3d::FastDiv, its constants made on
// the device (the region row width differs between border and inner blocks).
__device__ __forceinline__ rope3d::FastDiv fastdiv_make_dev(uint32_t d) {
    const uint32_t l = 32u - __clz(d - 1u);   // ceil(log2 d); 0 for d = 1
    const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
    return rope3d::FastDiv{d, uint32_t(m), l};
}


// The launch-wide shape of a chunk: every TMA box is (64 channels, 1 head,
// rwb columns, chb rows, 1 frame) with rwb = min(W, kw + 7), the widest key
// region row of any block, and chb = kTcN / rwb rows; a block whose region
// is narrower masks the extra columns. Key j of a chunk is tile row j: region
// row j / rwb, column j % rwb of the box.
struct TcShape {
    int nbt;     // query blocks along T (2 frames each)
    int rwb;     // box width (columns)
    int chb;     // box height (rows per chunk)
    int total;   // query blocks of the launch
};

// One query block: its place and its key region (frames [rt0, rt0 + frames),
// rows [rh0, rh0 + RH), columns [rw0, rw0 + RW)), cut into per_frame chunks
// of chb region rows per frame.
struct TcBlock {
    int b, head, t0, h0, w0;
    int rt0, rh0, RH, rw0, RW;
    int per_frame, n_chunks;
};

// The block index's divisors (blocks along W, H, T, heads) as multiply-high
// constants, made once per thread: every role walks the blocks.
struct TcDivs {
    rope3d::FastDiv nbw, nbh, nbt, heads;
};

__device__ __forceinline__ TcBlock tc_block(const NAParams &p, const TcShape &shp, const TcDivs &dv,
                                            int blk) {
    TcBlock g;
    uint32_t b = uint32_t(blk), q = fdiv(b, dv.nbw);
    g.w0 = int(b - q * dv.nbw.d) * kTcQW;
    b = q;
    q = fdiv(b, dv.nbh);
    g.h0 = int(b - q * dv.nbh.d) * kTcQH;
    b = q;
    q = fdiv(b, dv.nbt);
    g.t0 = int(b - q * dv.nbt.d) * kTcQT;
    b = q;
    q = fdiv(b, dv.heads);
    g.head = int(b - q * dv.heads.d);
    g.b = int(q);
    g.rt0 = na_start(g.t0, p.T, p.kt);
    const int rt1 = na_start(min(g.t0 + 1, p.T - 1), p.T, p.kt) + p.kt;
    g.rh0 = na_start(g.h0, p.H, p.kh);
    g.RH = na_start(min(g.h0 + kTcQH - 1, p.H - 1), p.H, p.kh) + p.kh - g.rh0;
    g.rw0 = na_start(g.w0, p.W, p.kw);
    g.RW = na_start(min(g.w0 + kTcQW - 1, p.W - 1), p.W, p.kw) + p.kw - g.rw0;
    g.per_frame = (g.RH + shp.chb - 1) / shp.chb;
    g.n_chunks = (rt1 - g.rt0) * g.per_frame;
    return g;
}

// 128 registers a thread: the four warps a sub-partition holds fill its
// quarter of the register file
// 128 registers a thread: the four warps a sub-partition holds fill its
// quarter of the register file
template <int kMode>
__global__ void __launch_bounds__(kTcThreads, 1)
rope3d_na3d_tc_kernel(const NAParams p, const TcShape shp, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                      const __grid_constant__ CUtensorMap tmQ) {
    extern __shared__ unsigned char tc_raw[];
    unsigned char *sm = tc_raw + ((1024u - (smem_addr(tc_raw) & 1023u)) & 1023u);
    const uint32_t sQ = smem_addr(sm + kTcOffQ), sK = smem_addr(sm + kTcOffK);
    const uint32_t sV = smem_addr(sm + kTcOffV);
    float *red_max = reinterpret_cast<float *>(sm + kTcOffRed);   // [chunk parity][part][128]
    float *red_sum = red_max + 2 * kTcParts * kTcM;                 // [block parity][part][128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kTcOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + kTcOffBar + kTcBars * 8);
    // mbarriers, counted over the CTA's whole sequence of chunks. One per K or
    // V ring slot (chunk & 1):
    //   kFull  K landed (TMA)          kReady  K rotated (kRotQK; 128 arrivals)
    //   kEmpty S MMAs done with K      vFull   V landed (TMA)
    //   vEmpty P V MMAs done with V
    // one per S buffer (chunk % kTcSBufs):
    //   sFull  S written (MMA)         sEmpty  P V done with the P in it (commit)
    //   pFull  P written (256 arrivals) pEmpty  P V done (O updated)
    // per Q buffer (block parity): qFull (the Q tile landed, TMA), qReady (the
    // tile rotated, in the rotating modes; 128 arrivals), qEmpty (the block's
    // S MMAs done with Q);
    // per O buffer b: oReady[b] the block's last P V done (commit), oEmpty[b]
    // O read out (Q warps), so the next block using b may overwrite it; and
    // oFull[block parity] the block's row sums written (softmax threads);
    // per block descriptor (block parity): dFull (written, 128 arrivals of the
    // Q warps), dEmpty (read, 256 arrivals of the softmax threads).
    enum { kFull, kReady, kEmpty, vFull, vEmpty };
    enum { sFull, sEmpty, pFull, pEmpty };
    auto bar = [&](int kind, int slot) { return smem_addr(&bars[2 * kind + slot]); };
    auto sbar = [&](int kind, int b) { return smem_addr(&bars[10 + kTcSBufs * kind + b]); };
    constexpr int kQb = 10 + 4 * kTcSBufs;
    auto qReady = [&](int b) { return smem_addr(&bars[kQb + b]); };
    auto qEmpty = [&](int b) { return smem_addr(&bars[kQb + 2 + b]); };
    auto oReady = [&](int b) { return smem_addr(&bars[kQb + 4 + b]); };
    auto oEmpty = [&](int b) { return smem_addr(&bars[kQb + 4 + kTcOBufs + b]); };
    auto oFull = [&](int b) { return smem_addr(&bars[kQb + 4 + 2 * kTcOBufs + b]); };
    auto qFull = [&](int b) { return smem_addr(&bars[kQb + 6 + 2 * kTcOBufs + b]); };
    auto dFull = [&](int b) { return smem_addr(&bars[kQb + 8 + 2 * kTcOBufs + b]); };
    auto dEmpty = [&](int b) { return smem_addr(&bars[kQb + 10 + 2 * kTcOBufs + b]); };
    static_assert(kQb + 10 + 2 * kTcOBufs + 2 <= kTcBars, "mbarriers");

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long tok = (long long)p.heads * kHD;   // elements per token
    const int rwb = shp.rwb, chb = shp.chb;          // RW <= rwb, chb * rwb <= kTcN
    const rope3d::FastDiv rwd = fastdiv_make_dev(uint32_t(rwb));
    const TcDivs dv{fastdiv_make_dev(uint32_t(p.nbw)), fastdiv_make_dev(uint32_t(p.nbh)),
                    fastdiv_make_dev(uint32_t(shp.nbt)), fastdiv_make_dev(uint32_t(p.heads))};
    const uint32_t box_bytes = uint32_t(2 * 128 * rwb * chb);   // both column blocks

    // The chunks of block g in order: frame f, region rows [r0, r0 + nr);
    // r0 steps by chb through the block's RH region rows, then the next frame.
    struct ChunkPos {
        int f, r0, nr, pf;   // pf: the chunk's index within its frame
    };
    auto chunk_start = [&](const TcBlock &g) { return ChunkPos{g.rt0, 0, min(chb, g.RH), 0}; };
    auto chunk_advance = [&](const TcBlock &g, ChunkPos &cp) {
        cp.r0 += chb;
        ++cp.pf;
        if (cp.r0 >= g.RH) {
            cp.r0 = 0;
            cp.pf = 0;
            ++cp.f;
        }
        cp.nr = min(chb, g.RH - cp.r0);
    };
    auto chunk_n = [&](const ChunkPos &cp) { return (cp.nr * rwb + 15) & ~15; };   // MMA width
    // TMA copies of a chunk's K or V (both column blocks) into ring slot s
    auto tma_chunk = [&](const TcBlock &g, const ChunkPos &cp, int s, bool v) {
        const int f = cp.f, r0 = cp.r0;
        const int frame = g.b * p.T + f;
        const uint32_t full = bar(v ? vFull : kFull, s), dst = (v ? sV : sK) + s * kTcKvSlot;
        const CUtensorMap *map = v ? &tmV : &tmK;
        mbar_expect_tx(full, box_bytes);
        tma_load5(dst, map, 0, g.head, g.rw0, g.rh0 + r0, frame, full);
        tma_load5(dst + kTcKvCb, map, 64, g.head, g.rw0, g.rh0 + r0, frame, full);
    };

    // ---- set-up: barriers, tensor memory, zeroed pad rows
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            const int counts[5] = {1, kTcRotThreads, 1, 1, 1};
            for (int kind = 0; kind < 5; ++kind)
                asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar(kind, s)),
                             "r"(counts[kind]) : "memory");
        }
        for (int b = 0; b < kTcSBufs; ++b) {
            const int counts[4] = {1, 1, kTcSoftThreads, 1};
            for (int kind = 0; kind < 4; ++kind)
                asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sbar(kind, b)),
                             "r"(counts[kind]) : "memory");
        }
        for (int b = 0; b < 2; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(qReady(b)), "r"(kTcRotThreads) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(qEmpty(b)) : "memory");
        }
        for (int b = 0; b < kTcOBufs; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(oReady(b)) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(oEmpty(b)), "r"(kTcRotThreads) : "memory");
        }
        for (int b = 0; b < 2; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(oFull(b)), "r"(kTcSoftThreads) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(qFull(b)) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(dFull(b)), "r"(kTcRotThreads) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(dEmpty(b)), "r"(kTcSoftThreads) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmK)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmV)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmO)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmQ)) : "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_addr(tmem_slot)), "r"(kTcTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // Tile rows past a box (up to the MMA's next multiple of 16) are never
    // written by TMA: zero them once (finite, with weight 0).
    {
        const int box_rows = rwb * chb, pad = ((box_rows + 15) & ~15) - box_rows;
        for (int i = tid; i < 4 * 2 * pad * 8; i += kTcThreads) {   // 4 tiles x 2 column blocks x pad rows x 8 chunks
            const int tile = i / (2 * pad * 8), rest = i % (2 * pad * 8);
            const int cb = rest / (pad * 8), rr = (rest / 8) % pad, ch = rest % 8;
            const uint32_t r = uint32_t(box_rows + rr);
            *reinterpret_cast<uint4 *>(sm + kTcOffK + tile * kTcKvSlot + cb * kTcKvCb + r * 128 +
                                       (((uint32_t(ch)) ^ (r & 7)) << 4)) = make_uint4(0, 0, 0, 0);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool dead = false;

    if (warp == 0 || warp == 3) {
        // ---- TMA producers: each block's chunks' K (warp 0) or V (warp 3) into
        // their ring, each slot once the MMAs of the chunk two before are done
        // with it (two threads, so that K never waits for a V slot)
        if (lane == 0) {
            const bool v = warp == 3;
            // K of the rotate-once form comes from the kernel before this one in
            // the stream (programmatic serialization): wait for it first
            if constexpr (kMode == kRotQ)
                if (!v) asm volatile("griddepcontrol.wait;" ::: "memory");
            int gc = 0;   // chunks of the CTA so far
            for (int blk = blockIdx.x, k = 0; blk < shp.total; blk += gridDim.x, ++k) {
                const TcBlock g = tc_block(p, shp, dv, blk);
                ChunkPos cp = chunk_start(g);
                for (int c = 0; c < g.n_chunks; ++c, ++gc, chunk_advance(g, cp)) {
                    const int s = gc & 1;
                    const uint32_t use = uint32_t(gc >> 1);
                    if (gc >= 2) tc_wait(bar(v ? vEmpty : kEmpty, s), (use - 1) & 1u, dead);
                    tma_chunk(g, cp, s, v);
                }
            }
        }
    } else if (warp == 1) {
        // ---- P V issuer: O += P(c) V(c) for every chunk once the softmax has
        // written its weights (its own thread, so that these MMAs never wait
        // behind an S product that waits for its K tile, nor the reverse)
        if (lane == 0) {
            int gc = 0;
            const uint32_t id = tc_idesc(kTcM, kHD, 1);
            for (int blk = blockIdx.x, k = 0; blk < shp.total; blk += gridDim.x, ++k) {
                const TcBlock g = tc_block(p, shp, dv, blk);
                const int ob = k % kTcOBufs;
                const uint32_t o_col = tmem + kTcColO + uint32_t(ob) * 128;
                // O buffer ob once the Q warps have read the previous result in it
                if (k >= kTcOBufs) tc_wait(oEmpty(ob), uint32_t(k / kTcOBufs - 1) & 1u, dead);
                ChunkPos cp = chunk_start(g);
                for (int c = 0; c < g.n_chunks; ++c, ++gc, chunk_advance(g, cp)) {
                    const int s = gc & 1, sb = gc % kTcSBufs;   // V slot, S buffer
                    const uint32_t use = uint32_t(gc >> 1), suse = uint32_t(gc / kTcSBufs);
                    tc_wait(sbar(pFull, sb), suse & 1u, dead);
                    tc_wait(bar(vFull, s), use & 1u, dead);
                    tc_fence_after();
                    const int ngrp = chunk_n(cp) >> 4;
                    // P(c) is in S buffer sb: 16 keys = 8 columns of bf16 pairs a step
                    const uint32_t pa = tmem + sb * kTcColS, vt = sV + s * kTcKvSlot;
                    for (int j = 0; j < ngrp; ++j)
                        tc_mma_ta(o_col, pa + uint32_t(8 * j), tc_sdesc(vt + j * 2048, kTcKvCb, 1024), id,
                                  (j > 0 || c > 0) ? 1u : 0u);
                    tc_commit(bar(vEmpty, s));
                    tc_commit(sbar(pEmpty, sb));
                    tc_commit(sbar(sEmpty, sb));   // S buffer sb (and P in it) free again
                    if (c == g.n_chunks - 1) tc_commit(oReady(ob));
                }
            }
        }
    } else if (warp == 2) {
        // ---- S issuer: S(c) = Q K(c)^T into S buffer c % kTcSBufs as soon as
        // K(c) has landed (rotated, in the per-CTA mode) and P V has read the
        // P of the chunk kTcSBufs before from that buffer
        if (lane == 0) {
            int gc = 0;
            for (int blk = blockIdx.x, k = 0; blk < shp.total; blk += gridDim.x, ++k) {
                const TcBlock g = tc_block(p, shp, dv, blk);
                // this block's Q: landed (TMA), or landed and rotated
                tc_wait(kMode == kRotNone ? qFull(k & 1) : qReady(k & 1), uint32_t(k >> 1) & 1u, dead);
                const uint32_t sQk = sQ + uint32_t(k & 1) * 2 * kTcQCb;   // this block's Q buffer
                ChunkPos cp = chunk_start(g);
                for (int c = 0; c < g.n_chunks; ++c, ++gc, chunk_advance(g, cp)) {
                    const int s = gc & 1, sb = gc % kTcSBufs;   // K slot, S buffer
                    const uint32_t use = uint32_t(gc >> 1), suse = uint32_t(gc / kTcSBufs);
                    tc_wait(bar(kMode == kRotQK ? kReady : kFull, s), use & 1u, dead);
                    if (gc >= kTcSBufs) tc_wait(sbar(sEmpty, sb), (suse - 1) & 1u, dead);
                    tc_fence_after();
                    const uint32_t id = tc_idesc(kTcM, uint32_t(chunk_n(cp)), 0);
                    const uint32_t kt = sK + s * kTcKvSlot;
#pragma unroll
                    for (int ks = 0; ks < kHD / 16; ++ks) {
                        const uint32_t koff = (ks & 3) * 32;   // 16 channels = 32 bytes
                        tc_mma(tmem + sb * kTcColS, tc_sdesc(sQk + (ks >> 2) * kTcQCb + koff, 16, 1024),
                               tc_sdesc(kt + (ks >> 2) * kTcKvCb + koff, 16, 1024), id, ks > 0);
                    }
                    tc_commit(bar(kEmpty, s));
                    tc_commit(sbar(sFull, sb));
                    if (c == g.n_chunks - 1) tc_commit(qEmpty(k & 1));
                }
            }
        }
    } else if (warp < kTcSoftWarp0) {   // warps 4-7
        // ---- Q warps: each block's Q tile copied by TMA into Q buffer k & 1
        // (128-byte-swizzled box layout) while the previous block still runs on
        // the other buffer, and in the rotating modes rotated there in place;
        // each block's descriptor for the softmax threads, a block ahead; in the
        // mode that rotates K per CTA, each K tile too, in place once it lands.
        // For the rotation, thread rt holds 16-byte vector cv = rt % 16 of query
        // rows rt / 16 + 8 i, i = 0 .. 15: a row is (t, h, w) = (i / 8, i % 8,
        // rt / 16) from the block's corner.
        // They also write each block's result: once its last P V is done and
        // the softmax threads have left their row sums, each thread takes the
        // row of tensor memory lane 32 (warp % 4) + lane (the lanes its warp
        // reaches) and normalises its 128 channels, while the softmax threads
        // already work on the next block. The rows go into the block's own Q
        // buffer (its S products are done) in the TMA box layout, O is handed
        // back, and two TMA stores write the tile; the buffer takes the block
        // after next's Q once the stores have read it. A block whose frame pair
        // passes the grid's last frame (odd T) is stored row by row instead:
        // the tensor map's frame axis runs on into the next batch.
        {
            const int rt = tid - 128;   // 0 .. kTcRotThreads - 1
            const int cv = rt & 15, qw_off = rt >> 4;
            [[maybe_unused]] const TabSlot tsg = tab_slot_global(p.pT, p.pH, p.pW, p.offH, p.offW, cv);
            [[maybe_unused]] int gc = 0;
            const int orow = 32 * (warp & 3) + lane;   // the O row this thread stores
            bool o_pending = false;   // a TMA store of O may still read a Q buffer
            auto store_o = [&](const TcBlock &g, int k) {
                const int b = k & 1, ob = k % kTcOBufs;   // row-sum and O buffers
                tc_wait(oReady(ob), uint32_t(k / kTcOBufs) & 1u, dead);
                tc_wait(oFull(b), uint32_t(k >> 1) & 1u, dead);
                tc_fence_after();
                float l = 0.f;
#pragma unroll
                for (int i = 0; i < kTcParts; ++i) l += red_sum[(b * kTcParts + i) * kTcM + orow];
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const int qt = g.t0 + (orow >> 6), qh = g.h0 + ((orow >> 3) & 7), qw = g.w0 + (orow & 7);
                const bool ok = qt < p.T && qh < p.H && qw < p.W;
                const long long base = ((((long long)g.b * p.T + qt) * p.H + qh) * p.W + qw) * tok +
                                       (long long)g.head * kHD;
                const uint32_t tO = tmem + kTcColO + uint32_t(ob) * 128 + (uint32_t(32 * (warp & 3)) << 16);
                const bool tma_o = g.t0 + kTcQT <= p.T;
                unsigned char *stg = sm + kTcOffQ + (k & 1) * 2 * kTcQCb;
                // 64 columns per tensor-memory wait
#pragma unroll 1
                for (int hh = 0; hh < kHD / 64; ++hh) {
                    float o[64];
                    tc_ld32_async(tO + uint32_t(64 * hh), o);
                    tc_ld32_async(tO + uint32_t(64 * hh + 32), o + 32);
                    tc_ld_wait_hold<64>(o);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        const int h2 = 4 * hh + q4;   // 16 columns: vectors 2 h2 and 2 h2 + 1
                        uint32_t packed[8];
                        const float2 inv2 = make_float2(inv, inv);
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {   // packed multiplies: two channels each
                            const float2 y = __fmul2_rn(make_float2(o[16 * q4 + i], o[16 * q4 + i + 1]), inv2);
                            packed[i / 2] = pack_bf16(y.x, y.y);
                        }
                        if (tma_o) {
                            *reinterpret_cast<uint4 *>(stg + sw128(uint32_t(orow), uint32_t(2 * h2), kTcQCb)) =
                                make_uint4(packed[0], packed[1], packed[2], packed[3]);
                            *reinterpret_cast<uint4 *>(stg + sw128(uint32_t(orow), uint32_t(2 * h2 + 1), kTcQCb)) =
                                make_uint4(packed[4], packed[5], packed[6], packed[7]);
                        } else if (ok && bound_ok(base + 16 * h2, 16, p.total)) {
                            uint4 *dst = reinterpret_cast<uint4 *>(p.out + base + 16 * h2);
                            dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                            dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                        }
                    }
                }
                tc_fence_before();   // the reads of O, before the buffer is handed back
                mbar_arrive(oEmpty(ob));
                if (tma_o) {
                    fence_async_smem();   // the staged rows, to the tensor copies
                    asm volatile("bar.sync %0, %1;" ::"n"(kTcQBar), "n"(kTcRotThreads) : "memory");
                    if (rt == 0) {
                        const uint32_t src = smem_addr(stg);
                        const int frame = g.b * p.T + g.t0;
                        tma_store5(&tmO, src, 0, g.head, g.w0, g.h0, frame);
                        tma_store5(&tmO, src + kTcQCb, 64, g.head, g.w0, g.h0, frame);
                        bulk_commit();
                    }
                    o_pending = true;
                }
            };
            // before a Q buffer is written: the TMA stores that read it are done
            auto o_reads_done = [&]() {
                if (o_pending) {
                    if (rt == 0) bulk_wait_read_all();
                    asm volatile("bar.sync %0, %1;" ::"n"(kTcQBar), "n"(kTcRotThreads) : "memory");
                    o_pending = false;
                }
            };
            TcBlock g_prev{};
            for (int blk = blockIdx.x, k = 0; blk < shp.total; blk += gridDim.x, ++k) {
                const TcBlock g = tc_block(p, shp, dv, blk);
                const int w = g.w0 + qw_off;
                // the softmax threads' descriptor of this block, into slot k & 1
                // once they have read the one of block k - 2
                if (k >= 2) tc_wait(dEmpty(k & 1), uint32_t((k - 2) >> 1) & 1u, dead);
                {
                    unsigned char *ds = sm + kTcOffDesc + (k & 1) * kTcDescSlot;
                    if (rt == 0) *reinterpret_cast<int4 *>(ds) = make_int4(g.rt0, g.RH, g.per_frame, g.n_chunks);
                    const int qt = g.t0 + (orow >> 6), qh = g.h0 + ((orow >> 3) & 7), qw = g.w0 + (orow & 7);
                    const int aw = na_start(min(qw, p.W - 1), p.W, p.kw) - g.rw0;
                    const int clo = max(aw, 0), chi = min(aw + p.kw, g.RW);   // window columns of a region row
                    reinterpret_cast<int4 *>(ds + 16)[orow] =
                        make_int4(qt < p.T && qh < p.H && qw < p.W, na_start(min(qt, p.T - 1), p.T, p.kt),
                                  na_start(min(qh, p.H - 1), p.H, p.kh) - g.rh0, clo | chi << 16);
                    mbar_arrive(dFull(k & 1));
                }
                // Q buffer k & 1, once block k - 2's S MMAs are done with it
                // and the TMA stores of block k - 2's O have read it
                if (k >= 2) tc_wait(qEmpty(k & 1), uint32_t((k - 2) >> 1) & 1u, dead);
                o_reads_done();
                unsigned char *qbuf = sm + kTcOffQ + (k & 1) * 2 * kTcQCb;
                // the tile by two TMA box loads (64 channels each); rows past the
                // grid read zeros (or, past an odd last frame, the next batch's
                // first frame): their queries are masked
                if (rt == 0) {
                    const uint32_t dst = smem_addr(qbuf), full = qFull(k & 1);
                    const int frame = g.b * p.T + g.t0;
                    mbar_expect_tx(full, 2 * kTcQCb);
                    tma_load5(dst, &tmQ, 0, g.head, g.w0, g.h0, frame, full);
                    tma_load5(dst + kTcQCb, &tmQ, 64, g.head, g.w0, g.h0, frame, full);
                }
                if constexpr (kMode != kRotNone) {
                    // rotated in place, each thread its 16 vectors
                    tc_wait(qFull(k & 1), uint32_t(k >> 1) & 1u, dead);
#pragma unroll 4
                    for (int i = 0; i < 16; ++i) {
                        const int t = g.t0 + (i >> 3), h = g.h0 + (i & 7);
                        if (t < p.T && h < p.H && w < p.W) {
                            uint4 *ptr = reinterpret_cast<uint4 *>(
                                qbuf + sw128(uint32_t(qw_off + 8 * i), uint32_t(cv), kTcQCb));
                            const int pos = tsg.axis == 0 ? t : (tsg.axis == 1 ? h : w);
                            *ptr = rot_vec_at<true>(*ptr, p.tab, tsg, uint32_t(pos), p.tab_len);
                        }
                    }
                    fence_async_smem();
                    mbar_arrive(qReady(k & 1));
                }
                // the previous block's result: before this block's K tiles, whose
                // S products may wait for the O buffer through P V
                if (k >= 1) store_o(g_prev, k - 1);
                g_prev = g;
                if constexpr (kMode == kRotQK) {
                    ChunkPos cp = chunk_start(g);
                    for (int c = 0; c < g.n_chunks; ++c, ++gc, chunk_advance(g, cp)) {
                        const int s = gc & 1;
                        const uint32_t use = uint32_t(gc >> 1);
                        const int f = cp.f, r0 = cp.r0, nr = cp.nr;
                        tc_wait(bar(kFull, s), use & 1u, dead);
                        const int nvec = nr * rwb * 16;
                        for (int u = rt; u < nvec; u += kTcRotThreads) {
                            const uint32_t j = uint32_t(u) >> 4, cv = uint32_t(u) & 15;
                            const uint32_t rr = fdiv(j, rwd);
                            const int cc = int(j - rr * uint32_t(rwb));
                            if (cc >= g.RW) continue;   // outside the region: masked
                            const int pos = tsg.axis == 0 ? f : (tsg.axis == 1 ? g.rh0 + r0 + int(rr) : g.rw0 + cc);
                            uint4 *ptr = reinterpret_cast<uint4 *>(sm + kTcOffK + s * kTcKvSlot + sw128(j, cv, kTcKvCb));
                            *ptr = rot_vec_at<true>(*ptr, p.tab, tsg, uint32_t(pos), p.tab_len);
                        }
                        fence_async_smem();
                        mbar_arrive(bar(kReady, s));
                    }
                }
            }
            const int nblk = shp.total > int(blockIdx.x)
                                 ? (shp.total - int(blockIdx.x) + int(gridDim.x) - 1) / int(gridDim.x) : 0;
            if (nblk >= 1) store_o(g_prev, nblk - 1);
            if (rt == 0) bulk_wait_all();   // the last stores, before the CTA ends
        }
    } else {
        // ---- softmax warps: this thread's query row and column part
        const int lg = warp & 3, qq = (warp - kTcSoftWarp0) >> 2;
        const int row = 32 * lg + lane;
        const uint32_t lanes = uint32_t(32 * lg) << 16;
        int gc = 0;
        bool s_seen = false;   // the next chunk's S seen complete already (the whole warp)
        // the window geometries (packed) the mask sets were made for; the
        // set made longest ago is replaced first
        uint32_t mk0 = ~0u, mk1 = ~0u, mk2 = ~0u;
        int mk_next = 0;
        for (int blk = blockIdx.x, k = 0; blk < shp.total; blk += gridDim.x, ++k) {
            // the block's chunk geometry and this row's window, from the Q warps
            tc_wait(dFull(k & 1), uint32_t(k >> 1) & 1u, dead);
            const unsigned char *ds = sm + kTcOffDesc + (k & 1) * kTcDescSlot;
            const int4 bd = *reinterpret_cast<const int4 *>(ds);
            const int4 rd = reinterpret_cast<const int4 *>(ds + 16)[row];
            mbar_arrive(dEmpty(k & 1));
            TcBlock g{};
            g.rt0 = bd.x;
            g.RH = bd.y;
            g.per_frame = bd.z;
            g.n_chunks = bd.w;
            const bool row_ok = rd.x != 0;
            const int st_q = rd.y, ah = rd.z;
            const int clo = rd.w & 0xffff, chi = rd.w >> 16;   // window columns of a region row
            const uint32_t tO = tmem + kTcColO + uint32_t(k % kTcOBufs) * 128 + lanes;
            float m_ref = -INFINITY, l_part = 0.f;   // running reference and this part's sum
            const int cb0 = qq * kTcHalf;   // this thread's columns of a chunk: [cb0, cb0 + 56)
            // Window mask of the chunk at region rows [r0, r0 + nr): bit k stands
            // for column cb0 + k; each chunk row the part spans that lies in the
            // window contributes its columns [clo, chi). It depends on the row
            // offset only (every frame's chunks share it).
            auto window_mask = [&](int r0, int nr) {
                uint64_t m = 0;
                const int rr0 = int(fdiv(uint32_t(cb0), rwd));
                for (int rr = rr0, js = rr0 * rwb - cb0; js < kTcHalf && rr < nr; ++rr, js += rwb) {
                    if (unsigned(r0 + rr - ah) < unsigned(p.kh)) {
                        const int a = max(js + clo, 0), b2 = min(js + chi, kTcHalf);
                        if (a < b2) m |= (~0ull >> (64 - (b2 - a))) << a;
                    }
                }
                return m;
            };
            // A mask depends on the row's window in the region and the region's
            // height only (every interior block of the grid has the same), so
            // the sets made for recent blocks are kept and looked up.
            const bool kept = g.per_frame <= kTcMaxPF;
            const uint32_t key = g.RH < 256 ? uint32_t(ah) | uint32_t(clo) << 8 | uint32_t(chi) << 16 |
                                                  uint32_t(g.RH) << 24
                                            : ~0u;   // not kept across blocks
            int set = key == ~0u ? -1 : key == mk0 ? 0 : key == mk1 ? 1 : key == mk2 ? 2 : -1;
            if (kept && set < 0) {
                set = mk_next;
                mk_next = mk_next == kTcMaskSets - 1 ? 0 : mk_next + 1;
                mk0 = set == 0 ? key : mk0;
                mk1 = set == 1 ? key : mk1;
                mk2 = set == 2 ? key : mk2;
                uint64_t *wm = reinterpret_cast<uint64_t *>(sm + kTcOffMask) +
                               (set * kTcMaxPF * kTcSoftThreads + qq * kTcM + row);
                for (int pf = 0, r0 = 0; pf < g.per_frame; ++pf, r0 += chb)
                    wm[pf * kTcSoftThreads] = window_mask(r0, min(chb, g.RH - r0));
            }
            const uint64_t *wmask = reinterpret_cast<const uint64_t *>(sm + kTcOffMask) +
                                    (max(set, 0) * kTcMaxPF * kTcSoftThreads + qq * kTcM + row);

            ChunkPos cp = chunk_start(g);
            for (int c = 0; c < g.n_chunks; ++c, ++gc, chunk_advance(g, cp)) {
                const int s = gc & 1;   // parity of the row-maximum exchange buffer
                const int f = cp.f, r0 = cp.r0, nr = cp.nr;
                const int sb = gc % kTcSBufs;   // S buffer
                const uint32_t suse = uint32_t(gc / kTcSBufs);
                const uint32_t tS = tmem + sb * kTcColS + lanes;
                // this thread's half of the chunk's columns, [cb0, cb0 + 56), loaded
                // at once as 32 + 16 + 8 columns. Columns past the chunk's keys are
                // masked (their S values are stale or zero-row products) and their
                // weights, written as zeros, lie past the P V MMA's width.
                // A warp's rows share their frame (lanes 0-63 of tensor memory are
                // the block's first frame, 64-127 its second), so a frame outside
                // the warp's time window is skipped by the whole warp: zero weights.
                const bool frame_ok = row_ok && unsigned(f - st_q) < unsigned(p.kt);
                // the window mask (geometry only, so read before S is waited for)
                uint64_t win = 0;
                if (frame_ok) win = kept ? wmask[cp.pf * kTcSoftThreads] : window_mask(r0, nr);
                // A warp none of whose rows has a key of its window here reads no
                // S. The others treat every group alike: straight-line code (the
                // groups' work interleaves) beats skipping groups by branches.
                const bool any = __any_sync(0xffffffffu, win != 0);
                if (!s_seen) tc_wait(sbar(sFull, sb), suse & 1u, dead);
                tc_fence_after();
                float x[kTcHalf];
                if (any) {
                    tc_ld32_async(tS + uint32_t(cb0), x);
                    tc_ld16_async(tS + uint32_t(cb0 + 32), x + 32);
                    tc_ld8_async(tS + uint32_t(cb0 + 48), x + 48);
                    tc_ld_wait_hold<kTcHalf>(x);
                }
                // the masked maximum, as four independent partial maxima taken two
                // values at a time
                float cmax = -INFINITY;
                if (any) {
                    float pm[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) pm[e] = -INFINITY;
#pragma unroll
                    for (int k8 = 0; k8 < kTcHalf / 8; ++k8) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int kk = 8 * k8 + e;
                            x[kk] = (win >> kk) & 1u ? x[kk] : -INFINITY;   // outside: weight 0
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            pm[e] = fmax3(pm[e], x[8 * k8 + 2 * e], x[8 * k8 + 2 * e + 1]);
                    }
                    cmax = fmax3(pm[0], pm[1], fmaxf(pm[2], pm[3]));
                }
                cmax *= p.scale_log2;   // a positive scale: the maximum of the scaled scores
                float *rm = red_max + (s * kTcParts) * kTcM;   // this chunk parity's [part][128]
                rm[qq * kTcM + row] = cmax;
                // the row's two threads (warps w and w + 4): a named barrier per pair
                asm volatile("bar.sync %0, %1;" ::"r"(1 + lg), "n"(32 * kTcParts) : "memory");
                float rmax = rm[row];
#pragma unroll
                for (int i = 1; i < kTcParts; ++i) rmax = fmaxf(rmax, rm[i * kTcM + row]);
                const float mn = fmaxf(m_ref, rmax);
                // The decisions are the same for the row's threads (the same
                // inputs); tensor-memory accesses are made by whole warps. A row
                // without a key so far has O = 0 and l = 0: nothing to rescale.
                const bool move = mn > m_ref + kLazy;
                const bool rescale = move && m_ref != -INFINITY;
                float corr = 1.f;
                if (move) {
                    corr = m_ref == -INFINITY ? 0.f : ex2(m_ref - mn);
                    m_ref = mn;
                    l_part *= corr;
                }
                // The weights, as bf16 pairs, into this S buffer's first 56 columns
                // (this part's 28 from column cb0 / 2) over the S values both
                // threads of the row have read (the exchange above came after
                // their loads); the P V MMA reads them from there.
                const float ms = m_ref == -INFINITY ? 0.f : m_ref;
                // exponent arguments and the row sum in packed pairs (two sums)
                const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(-ms, -ms);
                float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                uint32_t pw[kTcHalf / 2];
#pragma unroll
                for (int k8 = 0; k8 < kTcHalf / 8; ++k8) {
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        uint32_t w = 0u;
                        if (any) {
                            const float2 t = __ffma2_rn(make_float2(x[8 * k8 + e], x[8 * k8 + e + 1]), sc2, nm2);
                            const float a0 = ex2(t.x), a1 = ex2(t.y);
                            sum2[(e >> 1) & 1] = __fadd2_rn(sum2[(e >> 1) & 1], make_float2(a0, a1));
                            w = pack_bf16(a0, a1);
                        }
                        pw[4 * k8 + (e >> 1)] = w;
                    }
                }
                l_part += (sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y);
                const uint32_t tP = tS + uint32_t(cb0 >> 1);
                tc_st16w(tP, pw);
                tc_st8w(tP + 16, pw + 16);
                tc_st4w(tP + 24, pw + 24);
                // O rescaled after the weights are out (the row's S values are
                // no longer held), before P V of this chunk adds to it
                if (__any_sync(0xffffffffu, rescale)) {
                    // O must hold chunk c - 1's P V first (the same block)
                    tc_wait(sbar(pEmpty, (gc - 1) % kTcSBufs), uint32_t((gc - 1) / kTcSBufs) & 1u, dead);
                    tc_fence_after();
                    float o[16];
#pragma unroll 1   // (unrolled, the loads are hoisted and registers spill)
                    for (int h2 = 0; h2 < 128 / kTcParts / 16; ++h2) {
                        const uint32_t ta = tO + uint32_t(128 / kTcParts * qq + 16 * h2);
                        tc_ld16(ta, o);
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] *= corr;
                        tc_st16(ta, o);
                    }
                }
                // the next chunk's S buffer, tested without waiting while this
                // chunk's weights are handed over (a phase not yet complete is
                // waited for at the next chunk as before)
                s_seen = __all_sync(0xffffffffu, mbar_done(sbar(sFull, (gc + 1) % kTcSBufs),
                                                           uint32_t((gc + 1) / kTcSBufs) & 1u));
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");   // P (and O) written
                tc_fence_before();    // the tensor-memory accesses, before the hand-over
                mbar_arrive(sbar(pFull, sb));
            }

            // ---- this part's row sum for the Q warps, which normalise and store
            // the block's O while this thread goes on to the next block
            red_sum[((k & 1) * kTcParts + qq) * kTcM + row] = l_part;
            mbar_arrive(oFull(k & 1));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTcTmemCols) : "memory");
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

namespace rope3d {

// Vectors per launch of the K pass (rope3d_testing_max_units_per_launch
// lowers it so that small inputs take several launches).
static std::atomic<uint32_t> g_na3d_max_units{kMaxUnitsPerLaunch};

void na3d_set_max_units_per_launch(uint32_t n) {
    g_na3d_max_units.store(n == 0 || n > kMaxUnitsPerLaunch ? kMaxUnitsPerLaunch : n);
}

int64_t na3d_bound_errors(bool reset) {
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

namespace {

// The checks and kernel arguments shared by rope3d_na3d and
// rope3d_na3d_rotate_once (apply_rope: the tables are used; with_k_rot: the
// k_rot buffer of rope3d_na3d_rotate_once). The pointer, size, overlap and
// table-key checks make no CUDA call; check_device adds the device queries.
int na3d_setup(const void *q, const void *k, const void *v, const void *out, const void *k_rot,
               bool with_k_rot, const rope3d_tables *tables, int64_t B, int64_t T, int64_t H,
               int64_t W, int64_t heads, int64_t head_dim, const int32_t split[3],
               const int32_t kernel_size[3], bool apply_rope, bool check_device, NAParams &p) {
    if (!q || !k || !v || !out || !kernel_size || (apply_rope && (!tables || !split)) ||
        (with_k_rot && !k_rot))
        return ROPE3D_ERR_NULL;
    if (B <= 0 || T <= 0 || H <= 0 || W <= 0 || heads <= 0) return ROPE3D_ERR_SHAPE;
    if (head_dim != kHD) return ROPE3D_ERR_SHAPE;
    if (T >= 1024 || H >= 1024 || W >= 1024 || B * T * H * W * heads > (int64_t(1) << 40))
        return ROPE3D_ERR_SHAPE;
    const int kt = kernel_size[0], kh = kernel_size[1], kw = kernel_size[2];
    if (kt < 1 || kh < 1 || kw < 1 || kt % 2 == 0 || kh % 2 == 0 || kw % 2 == 0 || kt > T ||
        kh > H || kw > W)
        return ROPE3D_ERR_SHAPE;
    for (const void *ptr : {q, k, v, out, with_k_rot ? k_rot : q})
        if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return ROPE3D_ERR_ALIGN;
    const uint64_t bytes = uint64_t(B * T * H * W * heads) * kHD * 2;
    auto overlap = [bytes](const void *a, const void *b) {
        const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
        return x < y + bytes && y < x + bytes;
    };
    for (const void *ptr : {q, k, v})
        if (overlap(out, ptr)) return ROPE3D_ERR_ALIAS;
    // k_rot is k itself (rotation in place) or overlaps nothing; either way it
    // overlaps none of q, v and out (when K is rotated in place, Q may not
    // share its memory: the attention reads Q while the K pass may still run)
    if (with_k_rot) {
        for (const void *ptr : {q, v, out})
            if (overlap(k_rot, ptr)) return ROPE3D_ERR_ALIAS;
        if (k_rot != k && overlap(k_rot, k)) return ROPE3D_ERR_ALIAS;
    }
    p = NAParams{};
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
        if (check_device) {
            int cur = 0;
            if (cudaGetDevice(&cur) != cudaSuccess) return ROPE3D_ERR_CUDA;
            if (host_backed || tdev != cur) return ROPE3D_ERR_DEVICE;
        }
        p.tab = dev;
        p.tab_len = len;
        p.offH = offs[1];
        p.offW = offs[2];
        p.pT = split[0] / 2;
        p.pH = split[1] / 2;
        p.pW = split[2] / 2;
    }
    if (with_k_rot && uint64_t(heads) * (kHD / 8) > rope3d::kMaxUnitsPerLaunch)
        return ROPE3D_ERR_SHAPE;
    const uint64_t blocks = uint64_t(B) * heads * T * ((H + kQBH - 1) / kQBH) * ((W + kQBW - 1) / kQBW);
    if (blocks > 0x7fffffffull) return ROPE3D_ERR_SHAPE;
    if (check_device) {
        int device = 0;
        if (cudaGetDevice(&device) != cudaSuccess) return ROPE3D_ERR_CUDA;
        for (const void *ptr : {q, k, v, out, with_k_rot ? k_rot : q})
            if (!on_device(ptr, device)) return ROPE3D_ERR_DEVICE;
    }

    p.q = static_cast<const uint16_t *>(q);
    p.k = static_cast<const uint16_t *>(k);
    p.v = static_cast<const uint16_t *>(v);
    p.out = static_cast<uint16_t *>(const_cast<void *>(out));
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
    p.scale_log2 = float(1.4426950408889634 / std::sqrt(double(kHD)));
    p.total = static_cast<unsigned long long>(B * T * H * W * heads) * kHD;
    return ROPE3D_OK;
}

uint32_t na3d_blocks(const NAParams &p) {
    return uint32_t(uint64_t(p.B) * p.heads * p.T * p.nbh * p.nbw);
}

// The tensor-core (tcgen05) kernel: 2 x 8 x 8 query blocks; it needs a key
// region row (at most kw + 7 columns, or W) to fit one chunk of kTcN keys.
TcShape na3d_tc_shape(const NAParams &p) {
    TcShape shp;
    shp.nbt = (p.T + kTcQT - 1) / kTcQT;
    shp.rwb = std::min(p.W, p.kw + kTcQW - 1);
    shp.chb = kTcN / shp.rwb;
    shp.total = int(uint64_t(p.B) * p.heads * shp.nbt * p.nbh * p.nbw);
    return shp;
}

// The persistent grid: one CTA per SM (each walks blocks blockIdx.x,
// blockIdx.x + gridDim.x, ...), no more CTAs than blocks.
uint32_t na3d_tc_grid(const TcShape &shp) {
    static const int sms = [] {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 1;
        return n > 0 ? n : 1;
    }();
    return uint32_t(std::min(shp.total, sms));
}

// cuTensorMapEncodeTiled, from the driver through the runtime's entry-point
// query (the library does not link the driver library itself).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return EncodeTiledFn(nullptr);
        }
        return reinterpret_cast<EncodeTiledFn>(ptr);
    }();
    return fn;
}

// A tensor map of K or V for the tensor-core kernel: a 5-D view
// (128 channels, heads, W, H, B * T frames) of the [B, T, H, W, heads, 128]
// buffer, boxes of (64 channels, 1 head, bw columns, bh rows, bt frames) with
// the 128-byte swizzle; coordinates past the view read zeros. A chunk is a
// (rwb, chb, 1) box.
bool na3d_tc_map(CUtensorMap *map, const void *base, const NAParams &p, int bw, int bh, int bt) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t tok = cuuint64_t(p.heads) * kHD * 2;   // bytes per token
    const cuuint64_t dims[5] = {cuuint64_t(kHD), cuuint64_t(p.heads), cuuint64_t(p.W),
                                cuuint64_t(p.H), cuuint64_t(p.B) * cuuint64_t(p.T)};
    const cuuint64_t strides[4] = {cuuint64_t(kHD) * 2, tok, tok * cuuint64_t(p.W),
                                   tok * cuuint64_t(p.W) * cuuint64_t(p.H)};
    const cuuint32_t box[5] = {64, 1, cuuint32_t(bw), cuuint32_t(bh), cuuint32_t(bt)};
    const cuuint32_t elem[5] = {1, 1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box,
              elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Which attention kernel runs: 0 = the library's default and 1 = the
// tensor-core kernel wherever the geometry allows it (the faster of the two
// in every rotation mode on the 16 x 64 x 64, 16-head, 3 x 7 x 7 workload),
// else the warp-MMA kernel; 2 = always the warp-MMA kernel
// (rope3d_testing_na3d_kernel).
std::atomic<int> g_na3d_kernel{0};
thread_local int g_na3d_last_kernel = 0;   // 1 tensor-core, 2 warp-MMA kernel

bool na3d_use_tc(const NAParams &p) {
    if (g_na3d_kernel.load(std::memory_order_relaxed) == 2) return false;
    return std::min(p.W, p.kw + kTcQW - 1) <= kTcMaxRW;
}

template <int kMode>
bool na3d_tc_attribute() {
    static const bool ok = cudaFuncSetAttribute(rope3d_na3d_tc_kernel<kMode>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                int(kTcSmem)) == cudaSuccess;
    return ok;
}

// Dynamic shared memory limits of the three instances, set once.
bool na3d_attributes() {
    static const bool ok = [] {
        const cudaError_t rc[3] = {
            cudaFuncSetAttribute(rope3d_na3d_kernel<kRotNone>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(kFixedSmem)),
            cudaFuncSetAttribute(rope3d_na3d_kernel<kRotQK>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(kFixedSmem + kMaxTableBytes)),
            cudaFuncSetAttribute(rope3d_na3d_kernel<kRotQ>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(kFixedSmem))};
        return rc[0] == cudaSuccess && rc[1] == cudaSuccess && rc[2] == cudaSuccess;
    }();
    return ok;
}

}  // namespace

namespace {

// The rotate-once form on checked arguments (na3d_setup with the tables):
// K rotated into k_rot by the K pass, then the attention on k_rot rotating
// its Q tiles.
int na3d_launch_rotate_once(NAParams &p, const void *k, void *k_rot, const rope3d_tables *tables,
                            int64_t B, int64_t T, int64_t H, int64_t W, int64_t heads,
                            cudaStream_t st) {
    if (!na3d_attributes()) return ROPE3D_ERR_CUDA;
    static const int sms = [] {
        int dev = 0, n = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        return n;
    }();
    if (sms <= 0) return ROPE3D_ERR_CUDA;

    // 1. K -> k_rot, in launches of whole tokens below 2^30 vectors each
    RKParams rp{};
    rp.tab = p.tab;
    rp.tab_len = p.tab_len;
    rp.offH = p.offH;
    rp.offW = p.offW;
    rp.pT = p.pT;
    rp.pH = p.pH;
    rp.pW = p.pW;
    const uint32_t vec_per_tok = uint32_t(heads) * (kHD / 8);
    rp.heads = rope3d::make_fastdiv(uint32_t(heads));
    rp.Wd = rope3d::make_fastdiv(uint32_t(W));
    rp.Hd = rope3d::make_fastdiv(uint32_t(H));
    rp.HWd = rope3d::make_fastdiv(uint32_t(H * W));
    rp.Td = rope3d::make_fastdiv(uint32_t(T));
    const uint64_t tokens = uint64_t(B) * T * H * W, grid_tokens = uint64_t(T) * H * W;
    const uint64_t cap = rope3d::g_na3d_max_units.load(std::memory_order_relaxed);
    const uint64_t per_launch = cap / vec_per_tok > 0 ? cap / vec_per_tok : 1;
    for (uint64_t t0 = 0; t0 < tokens; t0 += per_launch) {
        const uint64_t n = tokens - t0 < per_launch ? tokens - t0 : per_launch;
        rp.k = static_cast<const uint4 *>(k) + t0 * vec_per_tok;
        rp.k_rot = static_cast<uint4 *>(k_rot) + t0 * vec_per_tok;
        rp.units = uint32_t(n * vec_per_tok);
        rp.tok0 = uint32_t(t0 % grid_tokens);
        const uint64_t want = (uint64_t(rp.units) + kRotThreads - 1) / kRotThreads;
        const uint32_t grid = uint32_t(want < uint64_t(3) * sms ? want : uint64_t(3) * sms);
        rope3d_na3d_rotate_k_kernel<<<grid, kRotThreads, 0, st>>>(rp);
        if (cudaGetLastError() != cudaSuccess) return ROPE3D_ERR_CUDA;
    }

    // 2. the attention on k_rot, rotating its Q tiles; launched with
    // programmatic serialization, it waits for step 1 before reading K
    p.k = static_cast<const uint16_t *>(k_rot);
    const bool tc = na3d_use_tc(p);
    g_na3d_last_kernel = tc ? 1 : 2;
    const TcShape shp = na3d_tc_shape(p);
    CUtensorMap mk{}, mv{}, mo{}, mq{};
    if (tc && (!na3d_tc_attribute<kRotQ>() || !na3d_tc_map(&mk, p.k, p, shp.rwb, shp.chb, 1) ||
               !na3d_tc_map(&mv, p.v, p, shp.rwb, shp.chb, 1) ||
               !na3d_tc_map(&mo, p.out, p, kTcQW, kTcQH, kTcQT) ||
               !na3d_tc_map(&mq, p.q, p, kTcQW, kTcQH, kTcQT)))
        return ROPE3D_ERR_CUDA;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(tc ? na3d_tc_grid(shp) : na3d_blocks(p));
    cfg.blockDim = dim3(tc ? kTcThreads : kThreads);
    cfg.dynamicSmemBytes = tc ? kTcSmem : kFixedSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t le = tc ? cudaLaunchKernelEx(&cfg, rope3d_na3d_tc_kernel<kRotQ>, p, shp, mk, mv, mo, mq)
                              : cudaLaunchKernelEx(&cfg, rope3d_na3d_kernel<kRotQ>, p);
    if (le != cudaSuccess) {
        cudaGetLastError();
        return ROPE3D_ERR_CUDA;
    }
    if (rope3d::tables_note_use(tables, st) != ROPE3D_OK) return ROPE3D_ERR_CUDA;
    return ROPE3D_OK;
}

// The pools rope3d_na3d takes its K scratch from: one per device, made on
// first use, keeping freed memory for later calls (no release threshold)
// until rope3d_cache_clear trims them.
std::mutex g_pool_mutex;
constexpr int kMaxDevices = 64;
cudaMemPool_t g_pools[kMaxDevices] = {};

cudaMemPool_t scratch_pool(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_pool_mutex);
    if (!g_pools[dev]) {
        cudaMemPoolProps props{};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        uint64_t keep = ~uint64_t(0);
        if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) {
            cudaGetLastError();
            cudaMemPoolDestroy(pool);
            return nullptr;
        }
        g_pools[dev] = pool;
    }
    return g_pools[dev];
}

// 1: rope3d_na3d with the RoPE runs the kernel that rotates Q and every K
// tile per CTA (rope3d_testing_na3d_per_cta).
std::atomic<int> g_na3d_per_cta{0};

}  // namespace

namespace rope3d {

void na3d_scratch_trim() {
    std::lock_guard<std::mutex> lock(g_pool_mutex);
    for (cudaMemPool_t pool : g_pools)
        if (pool && cudaMemPoolTrimTo(pool, 0) != cudaSuccess) cudaGetLastError();
}

}  // namespace rope3d

extern "C" int rope3d_na3d(const void *q, const void *k, const void *v, void *out,
                           const rope3d_tables *tables, int64_t B, int64_t T, int64_t H,
                           int64_t W, int64_t heads, int64_t head_dim, const int32_t split[3],
                           const int32_t kernel_size[3], int32_t apply_rope, void *stream) {
    NAParams p;
    const int rc = na3d_setup(q, k, v, out, nullptr, false, tables, B, T, H, W, heads, head_dim,
                              split, kernel_size, apply_rope != 0, true, p);
    if (rc != ROPE3D_OK) return rc;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (apply_rope && g_na3d_per_cta.load(std::memory_order_relaxed) == 0) {
        // K rotated once into scratch of K's size, taken from and returned to
        // the pool in stream order around the two launches
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) {
            cudaGetLastError();
            return ROPE3D_ERR_CUDA;
        }
        const cudaMemPool_t pool = scratch_pool(dev);
        void *k_rot = nullptr;
        if (!pool || cudaMallocFromPoolAsync(&k_rot, p.total * 2, pool, st) != cudaSuccess) {
            cudaGetLastError();
            return ROPE3D_ERR_CUDA;
        }
        const int lrc = na3d_launch_rotate_once(p, k, k_rot, tables, B, T, H, W, heads, st);
        if (cudaFreeAsync(k_rot, st) != cudaSuccess) {
            cudaGetLastError();
            return ROPE3D_ERR_CUDA;
        }
        return lrc;
    }
    g_na3d_last_kernel = na3d_use_tc(p) ? 1 : 2;
    if (na3d_use_tc(p)) {
        const TcShape shp = na3d_tc_shape(p);
        CUtensorMap mk, mv, mo, mq;
        if (!na3d_tc_map(&mk, p.k, p, shp.rwb, shp.chb, 1) || !na3d_tc_map(&mv, p.v, p, shp.rwb, shp.chb, 1) ||
            !na3d_tc_map(&mo, p.out, p, kTcQW, kTcQH, kTcQT) || !na3d_tc_map(&mq, p.q, p, kTcQW, kTcQH, kTcQT))
            return ROPE3D_ERR_CUDA;
        if (apply_rope) {
            if (!na3d_tc_attribute<kRotQK>()) return ROPE3D_ERR_CUDA;
            rope3d_na3d_tc_kernel<kRotQK><<<na3d_tc_grid(shp), kTcThreads, kTcSmem, st>>>(p, shp, mk, mv, mo, mq);
        } else {
            if (!na3d_tc_attribute<kRotNone>()) return ROPE3D_ERR_CUDA;
            rope3d_na3d_tc_kernel<kRotNone><<<na3d_tc_grid(shp), kTcThreads, kTcSmem, st>>>(p, shp, mk, mv, mo, mq);
        }
    } else {
        if (!na3d_attributes()) return ROPE3D_ERR_CUDA;
        const size_t smem = kFixedSmem + (apply_rope ? size_t(p.tab_len) * sizeof(float2) : 0);
        if (apply_rope)
            rope3d_na3d_kernel<kRotQK><<<na3d_blocks(p), kThreads, smem, st>>>(p);
        else
            rope3d_na3d_kernel<kRotNone><<<na3d_blocks(p), kThreads, smem, st>>>(p);
    }
    if (cudaGetLastError() != cudaSuccess) return ROPE3D_ERR_CUDA;
    if (apply_rope && rope3d::tables_note_use(tables, st) != ROPE3D_OK) return ROPE3D_ERR_CUDA;
    return ROPE3D_OK;
}

extern "C" int rope3d_na3d_rotate_once(const void *q, const void *k, const void *v, void *k_rot,
                                       void *out, const rope3d_tables *tables, int64_t B,
                                       int64_t T, int64_t H, int64_t W, int64_t heads,
                                       int64_t head_dim, const int32_t split[3],
                                       const int32_t kernel_size[3], void *stream) {
    NAParams p;
    const int rc = na3d_setup(q, k, v, out, k_rot, true, tables, B, T, H, W, heads, head_dim,
                              split, kernel_size, true, true, p);
    if (rc != ROPE3D_OK) return rc;
    return na3d_launch_rotate_once(p, k, k_rot, tables, B, T, H, W, heads,
                                   static_cast<cudaStream_t>(stream));
}

extern "C" int rope3d_testing_na3d_kernel(int32_t which) {
    if (which < 0 || which > 2) return ROPE3D_ERR_ARG;
    g_na3d_kernel.store(which);
    return ROPE3D_OK;
}

extern "C" int rope3d_testing_na3d_last_kernel(void) { return g_na3d_last_kernel; }

extern "C" int rope3d_testing_na3d_per_cta(int32_t on) {
    if (on != 0 && on != 1) return ROPE3D_ERR_ARG;
    g_na3d_per_cta.store(on);
    return ROPE3D_OK;
}

extern "C" int rope3d_testing_na3d_wait_timeouts(int64_t *count, int32_t reset) {
    if (!count) return ROPE3D_ERR_NULL;
    unsigned int n = 0;
    if (cudaMemcpyFromSymbol(&n, g_na3d_wait_timeouts, sizeof(n)) != cudaSuccess) {
        cudaGetLastError();
        return ROPE3D_ERR_CUDA;
    }
    if (reset) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_na3d_wait_timeouts, &zero, sizeof(zero)) != cudaSuccess) {
            cudaGetLastError();
            return ROPE3D_ERR_CUDA;
        }
    }
    *count = n;
    return ROPE3D_OK;
}

extern "C" int rope3d_na3d_preflight(const void *q, const void *k, const void *v, const void *k_rot,
                                     const void *out, const rope3d_tables *tables, int64_t B,
                                     int64_t T, int64_t H, int64_t W, int64_t heads,
                                     int64_t head_dim, const int32_t split[3],
                                     const int32_t kernel_size[3], int32_t apply_rope,
                                     int32_t check_device) {
    NAParams p;
    return na3d_setup(q, k, v, out, k_rot, k_rot != nullptr, tables, B, T, H, W, heads, head_dim,
                      split, kernel_size, apply_rope != 0 || k_rot != nullptr, check_device != 0,
                      p);
}
