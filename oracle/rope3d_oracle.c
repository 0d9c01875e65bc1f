/*
 * rope3d_oracle.c -- plain, slow, CPU oracle for the paired 3D rotary
 * position embedding (RoPE) that the LTX-2.5 diffusion video decoder applies
 * to Q and K before each attention block.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load this file. The product library never links, loads or
 * calls it, and it shares no source with the CUDA path.
 *
 * Sources (sglang PR #35698 review, "fused LTX-2.5 decoder 3D RoPE", prhub.com.cn):
 *   - "实现拆解" (implementation breakdown) step 1: one (cos, sin) table per
 *     axis, built by _axis_tables(length, dim) from (length, dim, base);
 *   - "实现拆解" step 2: the eager _apply_rope -- each of T, H, W takes its own
 *     chunk of head_dim, the chunk is viewed as (even, odd) pairs, rotated in
 *     float32 and cast back to the input dtype;
 *   - "关键源码片段" (key source snippets), the CUDA listing ltx25_decoder_rope.cuh:
 *     the eager order is four separately rounded fp32 products, then one
 *     rounded subtract (even*cos - odd*sin) and one rounded add
 *     (even*sin + odd*cos), no fused multiply-add; the pair index is decoded as
 *     (token, head, pair in head), tokens row-major over (frame, y, x), and the
 *     table row is the integer grid coordinate of the token on that axis;
 *   - same snippets, the JIT wrapper's preflight: table shapes are
 *     (T, dim_t/2), (H, dim_h/2), (W, dim_w/2).
 *
 * Readings where the pages are silent:
 *   - the table formula is not printed. We take standard per-axis RoPE,
 *     inv_freq_j = base^(-2j/d), angle = pos * inv_freq_j for integer pos,
 *     evaluated in double with the host libm and rounded once to float;
 *   - bf16 output uses round-to-nearest-even (the behaviour of a PyTorch
 *     float32 -> bfloat16 cast); a NaN stays a quiet NaN (payload unspecified);
 *   - fp32 inputs take the same steps with an identity cast.
 *
 * Build: plain C99, -O2 -ffp-contract=off -fno-fast-math. The contraction flag
 * is essential: every product and sum below must be rounded on its own.
 * Every intermediate is a named float so that a reader can check the order.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* bfloat16 <-> binary32, from the bit layouts: bfloat16 is the upper half   */
/* of a binary32 (1 sign, 8 exponent, 7 fraction bits).                      */
/* ------------------------------------------------------------------------- */

float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    if ((bits & 0x7fffffffu) > 0x7f800000u) {
        /* NaN: keep sign and the top payload bits, force the quiet bit. */
        return (uint16_t)((bits >> 16) | 0x0040u);
    }
    /* Round to nearest, ties to even, on the 16 discarded bits. A carry out of
     * the fraction bumps the exponent, which also gives +-inf on overflow. */
    uint32_t kept_lsb = (bits >> 16) & 1u;
    uint32_t rounded = bits + 0x7fffu + kept_lsb;
    return (uint16_t)(rounded >> 16);
}

/* ------------------------------------------------------------------------- */
/* IEEE binary16 <-> binary32 (1 sign, 5 exponent bits biased by 15, 10      */
/* fraction bits; subnormals are fraction * 2^-24).                          */
/* ------------------------------------------------------------------------- */

float oracle_f16_to_f32(uint16_t h)
{
    const uint32_t sign = (uint32_t)(h >> 15);
    const uint32_t exponent = (uint32_t)(h >> 10) & 0x1fu;
    const uint32_t fraction = (uint32_t)h & 0x3ffu;
    double magnitude;
    if (exponent == 0x1fu) {
        if (fraction == 0) {
            magnitude = INFINITY;
        } else {
            /* NaN: widen the payload into the binary32 fraction, quiet bit set */
            uint32_t bits = (sign << 31) | 0x7fc00000u | (fraction << 13);
            float f;
            memcpy(&f, &bits, sizeof f);
            return f;
        }
    } else if (exponent == 0) {
        magnitude = ldexp((double)fraction, -24);           /* subnormal or zero */
    } else {
        magnitude = ldexp((double)(fraction | 0x400u), (int)exponent - 25);
    }
    float f = (float)magnitude;                              /* exact */
    return sign ? -f : f;
}

uint16_t oracle_f32_to_f16(float f)
{
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    const uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    const uint32_t mag = bits & 0x7fffffffu;
    if (mag > 0x7f800000u)                                   /* NaN stays a quiet NaN */
        return (uint16_t)(sign | 0x7e00u | ((mag >> 13) & 0x1ffu));
    if (mag >= 0x477ff000u)                                  /* >= 65520: inf */
        return (uint16_t)(sign | 0x7c00u);
    if (mag >= 0x38800000u) {                                /* normal binary16 */
        uint32_t h = ((mag >> 23) - 112u) << 10 | ((mag >> 13) & 0x3ffu);
        const uint32_t rest = mag & 0x1fffu;                 /* 13 dropped bits */
        if (rest > 0x1000u || (rest == 0x1000u && (h & 1u)))
            h += 1;                                          /* may carry into the exponent */
        return (uint16_t)(sign | h);
    }
    if (mag <= 0x33000000u)                                  /* <= 2^-25: rounds to zero */
        return sign;
    /* subnormal binary16: round |f| / 2^-24 to an integer, ties to even */
    const uint32_t full = (mag & 0x7fffffu) | 0x800000u;
    const int e = (int)(mag >> 23) - 127;                    /* -25 .. -15 */
    const int shift = -e - 1;                                /* 14 .. 24 */
    uint32_t m = full >> shift;
    const uint32_t rest = full & ((1u << shift) - 1u);
    const uint32_t half = 1u << (shift - 1);
    if (rest > half || (rest == half && (m & 1u)))
        m += 1;
    return (uint16_t)(sign | m);
}

/* ------------------------------------------------------------------------- */
/* Axis tables ("实现拆解" step 1).                                           */
/* cos_out and sin_out are row-major [length][dim/2].                        */
/* ------------------------------------------------------------------------- */

int oracle_axis_table(int64_t length, int64_t dim, double base,
                      float *cos_out, float *sin_out)
{
    if (length <= 0 || dim <= 0 || (dim % 2) != 0 || !(base > 0.0))
        return -1;
    const int64_t half = dim / 2;
    for (int64_t pos = 0; pos < length; ++pos) {
        for (int64_t j = 0; j < half; ++j) {
            double exponent = -(2.0 * (double)j) / (double)dim;
            double inv_freq = pow(base, exponent);
            double angle = (double)pos * inv_freq;
            cos_out[pos * half + j] = (float)cos(angle);
            sin_out[pos * half + j] = (float)sin(angle);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* One (even, odd) pair in the eager order ("关键源码片段", rotate_pair).      */
/* ------------------------------------------------------------------------- */

void oracle_rotate_pair_f32(float even, float odd, float c, float s,
                            float *out_even, float *out_odd)
{
    float even_cos = even * c;   /* each product rounded on its own */
    float odd_sin = odd * s;
    float even_sin = even * s;
    float odd_cos = odd * c;
    float y0 = even_cos - odd_sin; /* then one rounded subtract ... */
    float y1 = even_sin + odd_cos; /* ... and one rounded add        */
    *out_even = y0;
    *out_odd = y1;
}

/* ------------------------------------------------------------------------- */
/* The whole tensor. x and y are [B][T][H][W][heads][head_dim], contiguous,  */
/* the same memory as [B][T*H*W][heads][head_dim]. split = (d_T, d_H, d_W):  */
/* channels [0, d_T) use the T table at row t, [d_T, d_T+d_H) the H table at */
/* row h, the rest the W table at row w; inside a chunk, pair j is the       */
/* channels (2j, 2j+1) and reads table column j.                             */
/* ------------------------------------------------------------------------- */

static int check_shape(int64_t B, int64_t T, int64_t H, int64_t W,
                       int64_t heads, int64_t head_dim, const int32_t split[3])
{
    if (B <= 0 || T <= 0 || H <= 0 || W <= 0 || heads <= 0 || head_dim <= 0)
        return -1;
    for (int a = 0; a < 3; ++a)
        if (split[a] <= 0 || (split[a] % 2) != 0)
            return -1;
    if ((int64_t)split[0] + split[1] + split[2] != head_dim)
        return -1;
    return 0;
}

/* Rotate one head row (head_dim channels) of fp32 values in place. */
static void rotate_head_f32(float *v, int64_t t, int64_t h, int64_t w,
                            const int32_t split[3],
                            const float *const cos_tab[3],
                            const float *const sin_tab[3])
{
    const int64_t pos[3] = {t, h, w};
    int64_t chunk_start = 0;
    for (int axis = 0; axis < 3; ++axis) {
        const int64_t half = split[axis] / 2;
        const float *crow = cos_tab[axis] + pos[axis] * half;
        const float *srow = sin_tab[axis] + pos[axis] * half;
        for (int64_t j = 0; j < half; ++j) {
            const int64_t ch = chunk_start + 2 * j;
            float y0, y1;
            oracle_rotate_pair_f32(v[ch], v[ch + 1], crow[j], srow[j], &y0, &y1);
            v[ch] = y0;
            v[ch + 1] = y1;
        }
        chunk_start += split[axis];
    }
}

#define ORACLE_MAX_HEAD_DIM 4096

int oracle_rope3d_bf16(const uint16_t *x, uint16_t *y,
                       int64_t B, int64_t T, int64_t H, int64_t W,
                       int64_t heads, int64_t head_dim, const int32_t split[3],
                       const float *cos_t, const float *sin_t,
                       const float *cos_h, const float *sin_h,
                       const float *cos_w, const float *sin_w)
{
    if (check_shape(B, T, H, W, heads, head_dim, split) != 0 ||
        head_dim > ORACLE_MAX_HEAD_DIM)
        return -1;
    const float *const cos_tab[3] = {cos_t, cos_h, cos_w};
    const float *const sin_tab[3] = {sin_t, sin_h, sin_w};
    float v[ORACLE_MAX_HEAD_DIM];
    int64_t row = 0;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t h = 0; h < H; ++h)
                for (int64_t w = 0; w < W; ++w)
                    for (int64_t head = 0; head < heads; ++head, ++row) {
                        const uint16_t *src = x + row * head_dim;
                        uint16_t *dst = y + row * head_dim;
                        for (int64_t ch = 0; ch < head_dim; ++ch)
                            v[ch] = oracle_bf16_to_f32(src[ch]);
                        rotate_head_f32(v, t, h, w, split, cos_tab, sin_tab);
                        for (int64_t ch = 0; ch < head_dim; ++ch)
                            dst[ch] = oracle_f32_to_bf16(v[ch]);
                    }
    return 0;
}

int oracle_rope3d_f32(const float *x, float *y,
                      int64_t B, int64_t T, int64_t H, int64_t W,
                      int64_t heads, int64_t head_dim, const int32_t split[3],
                      const float *cos_t, const float *sin_t,
                      const float *cos_h, const float *sin_h,
                      const float *cos_w, const float *sin_w)
{
    if (check_shape(B, T, H, W, heads, head_dim, split) != 0 ||
        head_dim > ORACLE_MAX_HEAD_DIM)
        return -1;
    const float *const cos_tab[3] = {cos_t, cos_h, cos_w};
    const float *const sin_tab[3] = {sin_t, sin_h, sin_w};
    float v[ORACLE_MAX_HEAD_DIM];
    int64_t row = 0;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t h = 0; h < H; ++h)
                for (int64_t w = 0; w < W; ++w)
                    for (int64_t head = 0; head < heads; ++head, ++row) {
                        const float *src = x + row * head_dim;
                        float *dst = y + row * head_dim;
                        for (int64_t ch = 0; ch < head_dim; ++ch)
                            v[ch] = src[ch];
                        rotate_head_f32(v, t, h, w, split, cos_tab, sin_tab);
                        for (int64_t ch = 0; ch < head_dim; ++ch)
                            dst[ch] = v[ch];
                    }
    return 0;
}

int oracle_rope3d_f16(const uint16_t *x, uint16_t *y,
                      int64_t B, int64_t T, int64_t H, int64_t W,
                      int64_t heads, int64_t head_dim, const int32_t split[3],
                      const float *cos_t, const float *sin_t,
                      const float *cos_h, const float *sin_h,
                      const float *cos_w, const float *sin_w)
{
    if (check_shape(B, T, H, W, heads, head_dim, split) != 0 ||
        head_dim > ORACLE_MAX_HEAD_DIM)
        return -1;
    const float *const cos_tab[3] = {cos_t, cos_h, cos_w};
    const float *const sin_tab[3] = {sin_t, sin_h, sin_w};
    float v[ORACLE_MAX_HEAD_DIM];
    int64_t row = 0;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t h = 0; h < H; ++h)
                for (int64_t w = 0; w < W; ++w)
                    for (int64_t head = 0; head < heads; ++head, ++row) {
                        const uint16_t *src = x + row * head_dim;
                        uint16_t *dst = y + row * head_dim;
                        for (int64_t ch = 0; ch < head_dim; ++ch)
                            v[ch] = oracle_f16_to_f32(src[ch]);
                        rotate_head_f32(v, t, h, w, split, cos_tab, sin_tab);
                        for (int64_t ch = 0; ch < head_dim; ++ch)
                            dst[ch] = oracle_f32_to_f16(v[ch]);
                    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Sampled outputs: the element at each flat index of the output, computed   */
/* one at a time from the full input. Used where a full pass is too long.    */
/* ------------------------------------------------------------------------- */

/* Decode a flat element index into the grid position and channel, then
 * return the (even, odd) input pair, the table entry and which member of the
 * pair the index is. */
static int locate(int64_t idx, int64_t T, int64_t H, int64_t W,
                  int64_t heads, int64_t head_dim, const int32_t split[3],
                  const float *const cos_tab[3], const float *const sin_tab[3],
                  int64_t *pair_first, float *c, float *s, int *is_odd)
{
    const int64_t ch = idx % head_dim;
    const int64_t row = idx / head_dim;            /* (b, t, h, w, head) */
    const int64_t token = (row / heads) % (T * H * W);
    const int64_t t = token / (H * W);
    const int64_t h = (token / W) % H;
    const int64_t w = token % W;
    const int64_t pos[3] = {t, h, w};
    int64_t chunk_start = 0;
    for (int axis = 0; axis < 3; ++axis) {
        if (ch < chunk_start + split[axis]) {
            const int64_t j = (ch - chunk_start) / 2;
            const int64_t half = split[axis] / 2;
            *c = cos_tab[axis][pos[axis] * half + j];
            *s = sin_tab[axis][pos[axis] * half + j];
            *pair_first = row * head_dim + chunk_start + 2 * j;
            *is_odd = (int)((ch - chunk_start) % 2);
            return 0;
        }
        chunk_start += split[axis];
    }
    return -1;
}

int oracle_rope3d_bf16_at(const uint16_t *x, const int64_t *indices, int64_t n,
                          uint16_t *out,
                          int64_t B, int64_t T, int64_t H, int64_t W,
                          int64_t heads, int64_t head_dim, const int32_t split[3],
                          const float *cos_t, const float *sin_t,
                          const float *cos_h, const float *sin_h,
                          const float *cos_w, const float *sin_w)
{
    if (check_shape(B, T, H, W, heads, head_dim, split) != 0)
        return -1;
    const float *const cos_tab[3] = {cos_t, cos_h, cos_w};
    const float *const sin_tab[3] = {sin_t, sin_h, sin_w};
    const int64_t total = B * T * H * W * heads * head_dim;
    for (int64_t i = 0; i < n; ++i) {
        if (indices[i] < 0 || indices[i] >= total)
            return -1;
        int64_t first;
        float c, s, y0, y1;
        int odd;
        if (locate(indices[i], T, H, W, heads, head_dim, split, cos_tab,
                   sin_tab, &first, &c, &s, &odd) != 0)
            return -1;
        oracle_rotate_pair_f32(oracle_bf16_to_f32(x[first]),
                               oracle_bf16_to_f32(x[first + 1]), c, s, &y0, &y1);
        out[i] = oracle_f32_to_bf16(odd ? y1 : y0);
    }
    return 0;
}

int oracle_rope3d_f32_at(const float *x, const int64_t *indices, int64_t n,
                         float *out,
                         int64_t B, int64_t T, int64_t H, int64_t W,
                         int64_t heads, int64_t head_dim, const int32_t split[3],
                         const float *cos_t, const float *sin_t,
                         const float *cos_h, const float *sin_h,
                         const float *cos_w, const float *sin_w)
{
    if (check_shape(B, T, H, W, heads, head_dim, split) != 0)
        return -1;
    const float *const cos_tab[3] = {cos_t, cos_h, cos_w};
    const float *const sin_tab[3] = {sin_t, sin_h, sin_w};
    const int64_t total = B * T * H * W * heads * head_dim;
    for (int64_t i = 0; i < n; ++i) {
        if (indices[i] < 0 || indices[i] >= total)
            return -1;
        int64_t first;
        float c, s, y0, y1;
        int odd;
        if (locate(indices[i], T, H, W, heads, head_dim, split, cos_tab,
                   sin_tab, &first, &c, &s, &odd) != 0)
            return -1;
        oracle_rotate_pair_f32(x[first], x[first + 1], c, s, &y0, &y1);
        out[i] = odd ? y1 : y0;
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* NeoX-style RoPE of the Gemma3 text encoder (sglang PR #24660 review,      */
/* "关键源码片段", gemma_3.py _apply_rotary_pos_emb): the rows of a           */
/* cos_sin_cache [max_position][rotary_dim] = [cos | sin] are gathered by     */
/* token position, duplicated to the full rotary width and cast to the input  */
/* dtype; then q * cos + rotate_half(q) * sin in that dtype, where            */
/* rotate_half(x) = (-x2, x1) for the halves x1 = x[:d/2], x2 = x[d/2:].     */
/* Each tensor operation rounds to the input dtype: a product of two         */
/* 16-bit values is exact in float and rounded once; the sum of two 16-bit   */
/* values is rounded to float and then to the 16-bit type (the order a       */
/* PyTorch 16-bit add takes). rotary_dim is head_dim (the page passes        */
/* rotary_dim=head_dim).                                                     */
/* ------------------------------------------------------------------------- */

/* Cache rows in the page's layout: cos of p * base^(-2j/d) for j < d/2, then
 * the sines (standard RoPE angles; the page builds the cache with get_rope,
 * whose formula it does not print). */
int oracle_neox_cache(int64_t max_position, int64_t rotary_dim, double base, float *cache)
{
    if (max_position <= 0 || rotary_dim <= 0 || (rotary_dim % 2) != 0 || !(base > 0.0))
        return -1;
    const int64_t half = rotary_dim / 2;
    for (int64_t p = 0; p < max_position; ++p)
        for (int64_t j = 0; j < half; ++j) {
            double exponent = -(2.0 * (double)j) / (double)rotary_dim;
            double angle = (double)p * pow(base, exponent);
            cache[p * rotary_dim + j] = (float)cos(angle);
            cache[p * rotary_dim + half + j] = (float)sin(angle);
        }
    return 0;
}

/* One NeoX pair (x1 at channel j, x2 at channel j + d/2) in 16-bit storage:
 * c and s are already cast to the storage type. kind: 0 bf16, 2 fp16. */
static uint16_t to16(float f, int kind) { return kind == 0 ? oracle_f32_to_bf16(f) : oracle_f32_to_f16(f); }
static float from16(uint16_t h, int kind) { return kind == 0 ? oracle_bf16_to_f32(h) : oracle_f16_to_f32(h); }

void oracle_neox_pair16(uint16_t x1, uint16_t x2, uint16_t c, uint16_t s, int kind,
                        uint16_t *y1, uint16_t *y2)
{
    const float fx1 = from16(x1, kind), fx2 = from16(x2, kind);
    const float fc = from16(c, kind), fs = from16(s, kind);
    /* q * cos */
    const uint16_t x1c = to16(fx1 * fc, kind);
    const uint16_t x2c = to16(fx2 * fc, kind);
    /* rotate_half(q) * sin: (-x2) * sin for the first half, x1 * sin for the second */
    const float neg_x2 = -fx2;
    const uint16_t nx2s = to16(neg_x2 * fs, kind);
    const uint16_t x1s = to16(fx1 * fs, kind);
    /* the sum, rounded to float and then to the storage type */
    const float sum1 = from16(x1c, kind) + from16(nx2s, kind);
    const float sum2 = from16(x2c, kind) + from16(x1s, kind);
    *y1 = to16(sum1, kind);
    *y2 = to16(sum2, kind);
}

void oracle_neox_pair_f32(float x1, float x2, float c, float s, float *y1, float *y2)
{
    const float x1c = x1 * c;
    const float x2c = x2 * c;
    const float neg_x2 = -x2;
    const float nx2s = neg_x2 * s;
    const float x1s = x1 * s;
    *y1 = x1c + nx2s;
    *y2 = x2c + x1s;
}

/* x, y: [tokens][heads][head_dim] contiguous; kind 0 bf16 / 2 fp16 (uint16
 * bits) or 1 fp32. Positions outside [0, max_position) are rejected. */
int oracle_rope_neox(const void *x, void *y, int64_t tokens, int64_t heads, int64_t head_dim,
                     const int64_t *positions, const float *cache, int64_t max_position, int kind)
{
    if (tokens <= 0 || heads <= 0 || head_dim <= 0 || (head_dim % 2) != 0)
        return -1;
    const int64_t half = head_dim / 2;
    for (int64_t t = 0; t < tokens; ++t) {
        const int64_t p = positions[t];
        if (p < 0 || p >= max_position)
            return -1;
        const float *cs = cache + p * head_dim;
        for (int64_t h = 0; h < heads; ++h) {
            const int64_t row = (t * heads + h) * head_dim;
            for (int64_t j = 0; j < half; ++j) {
                if (kind == 1) {
                    const float *xf = (const float *)x;
                    float *yf = (float *)y;
                    oracle_neox_pair_f32(xf[row + j], xf[row + half + j], cs[j], cs[half + j],
                                         &yf[row + j], &yf[row + half + j]);
                } else {
                    const uint16_t *xh = (const uint16_t *)x;
                    uint16_t *yh = (uint16_t *)y;
                    const uint16_t c16 = to16(cs[j], kind);          /* cos.to(q.dtype) */
                    const uint16_t s16 = to16(cs[half + j], kind);   /* sin.to(q.dtype) */
                    oracle_neox_pair16(xh[row + j], xh[row + half + j], c16, s16, kind,
                                       &yh[row + j], &yh[row + half + j]);
                }
            }
        }
    }
    return 0;
}
