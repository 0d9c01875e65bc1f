/*
 * rope3d.h -- C ABI of the fused paired 3D rotary position embedding (RoPE)
 * for GB300 (sm_103a).
 *
 * What it computes (sglang PR #35698 review, "fused LTX-2.5 decoder 3D RoPE",
 * prhub.com.cn; sections "实现拆解" steps 1-4 and "关键源码片段"): before each
 * attention block of the LTX-2.5 diffusion video decoder, Q and K of shape
 * [B, T*H*W, heads, head_dim] (tokens row-major over the (T, H, W) grid) are
 * rotated pair by pair. head_dim is split into three chunks
 * split = (d_T, d_H, d_W); the chunk of axis X uses that axis's fp32 table
 * (cos_X, sin_X) of shape [L_X, d_X/2] at the row given by the token's grid
 * coordinate on X. Inside a chunk, pair j is channels (2j, 2j+1):
 *     y_even = RN(RN(even*cos) - RN(odd*sin))
 *     y_odd  = RN(RN(even*sin) + RN(odd*cos))
 * in float32, four separately rounded products and no fused multiply-add,
 * then a round-to-nearest-even cast back to the input dtype. Q and K share the
 * table lookups and are rotated in one kernel launch.
 *
 * Threading: every function may be called from any host thread; the table
 * cache and the verification gate are protected by one mutex.
 * Errors: every int-returning function returns ROPE3D_OK (0) or a negative
 * ROPE3D_ERR_* code; rope3d_status_string() names it. Nothing is written to
 * any output when a call fails its checks. No call ever falls back to a CPU
 * computation of the result.
 */
#ifndef ROPE3D_H
#define ROPE3D_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ROPE3D_ABI_VERSION 1

/* ---- status codes ------------------------------------------------------ */
#define ROPE3D_OK            0
#define ROPE3D_ERR_NULL     -1  /* a required pointer is NULL                     */
#define ROPE3D_ERR_SHAPE    -2  /* a size <= 0, head_dim != d_T+d_H+d_W, a chunk
                                   odd or <= 0, or a size beyond the limits below  */
#define ROPE3D_ERR_DTYPE    -3  /* dtype is not ROPE3D_BF16, ROPE3D_F32 or ROPE3D_F16 */
#define ROPE3D_ERR_ALIGN    -4  /* a Q/K/output pointer is not 4-byte aligned     */
#define ROPE3D_ERR_ALIAS    -5  /* an output overlaps an input or the other output */
#define ROPE3D_ERR_DEVICE   -6  /* a pointer is not memory of the expected kind on
                                   the current device (see each function)          */
#define ROPE3D_ERR_PARITY   -7  /* the verification gate found a mismatch for this
                                   configuration; it stays refused until
                                   rope3d_gate_reset()                            */
#define ROPE3D_ERR_CUDA     -8  /* a CUDA runtime call or kernel launch failed    */
#define ROPE3D_ERR_TABLES   -9  /* the table handle does not match (T, H, W, split) */
#define ROPE3D_ERR_NOMEM   -10  /* a device or host allocation failed             */
#define ROPE3D_ERR_ARG     -11  /* another argument is out of range               */
#define ROPE3D_ERR_SCRATCH -12  /* the tables do not fit the fixed table area of
                                   rope3d_apply_pair_noalloc (64 KiB)             */

/* ---- element types ----------------------------------------------------- */
#define ROPE3D_BF16 0   /* bfloat16 in and out                                */
#define ROPE3D_F32  1   /* float32 in and out (same steps, identity cast)     */
#define ROPE3D_F16  2   /* IEEE binary16 in and out (same steps, nearest-even
                           cast to binary16)                                  */

/* ---- limits -------------------------------------------------------------- */
#define ROPE3D_MAX_HEAD_DIM 4096   /* head_dim above this -> ROPE3D_ERR_SHAPE  */
#define ROPE3D_TABLE_CACHE_CAP 16  /* FIFO table cache size ("实现拆解" step 1) */

typedef struct rope3d_tables rope3d_tables;  /* opaque, refcounted */

/*
 * rope3d_build_tables -- the per-axis cos/sin tables of one (T, H, W) grid,
 * through the table cache ("实现拆解" step 1: _axis_tables(length, dim) and
 * _tables(); a module-level cache keyed on the grid, the split and the base,
 * capped at 16 entries with first-in-first-out eviction, shared by every
 * attention block).
 *
 * Table values: table X has [L_X][d_X/2] entries (L = T, H, W); entry
 * (p, j) is cos / sin of p * base^(-2j/d_X), evaluated in double precision
 * with the host C library and rounded once to float. (The pages give the
 * shape and inputs of the table, not its formula; this is standard per-axis
 * RoPE.)
 *
 *   T, H, W   grid extents, each in [1, 2^31)
 *   split     (d_T, d_H, d_W), each even and > 0; the sum is head_dim
 *   base      RoPE base, finite and > 0 (the decoder uses 10000)
 *   stream    cudaStream_t (NULL = legacy default stream) on which the upload
 *             of a newly built entry is ordered; later use on other streams is
 *             safe because the call waits for that upload before returning
 *   out       receives a handle that the caller owns one reference to
 *
 * A cache hit returns the existing entry (and does not refresh its age). When
 * a 17th entry is inserted the oldest is unlinked from the cache; its memory
 * is released when its last reference is released, so handles stay valid.
 * Release is stream-ordered and never waits for the device: every launch that
 * reads a handle's tables records an event on its stream, and a released
 * buffer is freed (cudaFreeAsync, on a stream of the library's own) once all
 * of those events have completed, checked on later calls into the cache
 * (rope3d_build_tables, rope3d_release_tables, rope3d_cache_clear,
 * rope3d_cache_retired). Launches into a capturing stream are not tracked: a
 * CUDA graph that holds such a launch reads the tables on every replay, so
 * keep a reference to the handle for as long as the graph may run.
 * Device memory: one buffer per entry from the device's stream-ordered
 * allocator (cudaMallocAsync on `stream`; cudaMalloc where it is unsupported).
 * Errors: NULL, SHAPE, ARG (bad base), NOMEM, CUDA.
 */
int rope3d_build_tables(int64_t T, int64_t H, int64_t W, const int32_t split[3],
                        double base, void *stream, rope3d_tables **out);

/* Drop one reference. Returns ERR_NULL for NULL. */
int rope3d_release_tables(rope3d_tables *tables);

/* Add one reference (for callers that share a handle). */
int rope3d_retain_tables(rope3d_tables *tables);

/*
 * rope3d_apply_pair -- rotate Q and K on the GPU in one kernel launch
 * ("实现拆解" steps 3-4: fused_ltx25_decoder_rope writes Q_out and K_out in a
 * single launch, after the preflight can_use_ltx25_decoder_rope and the
 * first-seen bit-exact gate).
 *
 *   q, k          device pointers, [B, T, H, W, heads, head_dim] contiguous
 *                 (the same memory as [B, T*H*W, heads, head_dim]), elements
 *                 of type dtype, 4-byte aligned, on the current device
 *   q_out, k_out  device pointers of the same shape and type, owned by the
 *                 caller; each must overlap neither input nor the other output
 *                 (q and k may overlap each other: they are only read)
 *   tables        a handle from rope3d_build_tables for the same T, H, W and
 *                 split
 *   dtype         ROPE3D_BF16, ROPE3D_F32 or ROPE3D_F16
 *   stream        cudaStream_t the kernel is launched on (NULL = default)
 *
 * The call is asynchronous on `stream`, except the first call for each
 * configuration (dtype, B, T, H, W, heads, head_dim, split, base) while the
 * gate is on (the default): that call waits for the kernel, copies Q, K and
 * the outputs back to the host, recomputes the result on the CPU in the
 * eager order and compares every element (equal bits; or both NaN). A match
 * marks the configuration verified; a mismatch marks it refused and returns
 * ROPE3D_ERR_PARITY now and on every later call (no fallback; the outputs of
 * the refused call hold the kernel's result). So make the first call of a
 * configuration outside CUDA graph capture, or turn the gate off.
 *
 * 16-byte-aligned pointers with head_dim and every chunk a multiple of 8 (bf16,
 * fp16) or 4 (fp32) elements take the 16-byte vector kernel; any other valid input
 * takes the per-pair kernel with the same arithmetic.
 * Errors: NULL, SHAPE, DTYPE, ALIGN, ALIAS, DEVICE (a pointer that is not
 * device or managed memory of the current device), TABLES, PARITY, CUDA.
 */
int rope3d_apply_pair(const void *q, const void *k, void *q_out, void *k_out,
                      const rope3d_tables *tables,
                      int64_t B, int64_t T, int64_t H, int64_t W,
                      int64_t heads, int64_t head_dim, const int32_t split[3],
                      int32_t dtype, void *stream);

/*
 * rope3d_apply_pair_strided -- rope3d_apply_pair for strided views, including
 * rotation in place. This extends the pages' kernel, whose preflight demands
 * contiguous Q and K ("关键源码片段", can_use_ltx25_decoder_rope: is_contiguous),
 * so that Q and K can be read straight out of a fused QKV projection buffer,
 * out of a crop of a larger grid, and written back in place, without the copy
 * that contiguity forces. Same arithmetic and tables.
 *
 *   q, k, q_out, k_out  device pointers to element (0, 0, 0, 0, 0, 0) of each
 *                       view of logical shape [B, T, H, W, heads, head_dim]
 *   *_strides           element strides of (batch, t, h, w, head), each >= 0;
 *                       channels are contiguous (stride 1). For 16-bit types
 *                       every stride must be even (pairs stay 4-byte aligned).
 *   other arguments     as for rope3d_apply_pair
 *
 * In place: q_out == q with the same strides (and/or k_out == k) is allowed.
 * Otherwise no element of an output may be an element of an input or of the
 * other output: views whose address ranges intersect are accepted only when
 * they have identical strides and provably disjoint elements (e.g. the Q, K
 * and V thirds of one fused buffer); an output view must not map two indices
 * to one element. Violations return ROPE3D_ERR_ALIAS.
 * The gate works as in rope3d_apply_pair; its first-call check gathers the
 * views into temporary contiguous device buffers (allocated and freed by
 * that call; the inputs are gathered before the kernel runs, so in-place
 * calls are checked too). Its key adds the four stride sets.
 * Errors: as rope3d_apply_pair; ALIGN also for odd strides of 16-bit types;
 * SHAPE for negative strides; NOMEM when the gate's buffers cannot be allocated.
 */
int rope3d_apply_pair_strided(const void *q, const void *k, void *q_out, void *k_out,
                              const rope3d_tables *tables,
                              int64_t B, int64_t T, int64_t H, int64_t W,
                              int64_t heads, int64_t head_dim, const int32_t split[3],
                              int32_t dtype,
                              const int64_t q_strides[5], const int64_t k_strides[5],
                              const int64_t q_out_strides[5], const int64_t k_out_strides[5],
                              void *stream);

/*
 * rope3d_preflight_strided -- the checks of rope3d_apply_pair_strided without
 * a launch; check_device = 0 skips the device-memory query (no GPU needed).
 */
int rope3d_preflight_strided(const void *q, const void *k, const void *q_out,
                             const void *k_out, const rope3d_tables *tables,
                             int64_t B, int64_t T, int64_t H, int64_t W,
                             int64_t heads, int64_t head_dim, const int32_t split[3],
                             int32_t dtype,
                             const int64_t q_strides[5], const int64_t k_strides[5],
                             const int64_t q_out_strides[5], const int64_t k_out_strides[5],
                             int32_t check_device);

/*
 * rope3d_patchify -- space-to-depth of the decoder's pixel/latent volume
 * (sglang PR #34471 review, "关键源码片段", _patchify of
 * ltx_2_5_diffusion_decoder.py): x of shape (B, C, F, H, W) becomes y of shape
 * (B, C*p*p, F, H/p, W/p) with channels packed as (channel, width offset,
 * height offset):  y[b, (c*p + pw)*p + ph, f, i, j] = x[b, c, f, i*p + ph, j*p + pw].
 * A bit-exact permutation: the element type only sets its size.
 *
 *   x, y        device pointers, contiguous, caller-owned, not overlapping,
 *               aligned to elem_bytes
 *   B, C, F, H, W   sizes of x; H and W multiples of p; B*C*F < 2^31,
 *               H*W <= 2^30
 *   p           patch size >= 1 (1, 2, 4 and 8 take the 16-byte vector kernel
 *               when W/p is a multiple of 16/elem_bytes and both pointers are
 *               16-byte aligned; other cases take an element kernel)
 *   elem_bytes  1, 2, 4 or 8
 *   stream      cudaStream_t; asynchronous
 * Errors: NULL, SHAPE, DTYPE (elem_bytes), ALIGN, ALIAS, DEVICE, CUDA.
 */
int rope3d_patchify(const void *x, void *y, int64_t B, int64_t C, int64_t F, int64_t H,
                    int64_t W, int64_t p, int32_t elem_bytes, void *stream);

/*
 * rope3d_unpatchify -- the exact inverse of rope3d_patchify (the page names
 * _unpatchify without code): y (B, C*p*p, F, H/p, W/p) back to x
 * (B, C, F, H, W). Arguments as rope3d_patchify, with B, C, F, H, W the sizes
 * of x.
 */
int rope3d_unpatchify(const void *y, void *x, int64_t B, int64_t C, int64_t F, int64_t H,
                      int64_t W, int64_t p, int32_t elem_bytes, void *stream);

/* The host-side checks of rope3d_patchify / rope3d_unpatchify (no GPU needed). */
int rope3d_patchify_check(const void *src, const void *dst, int64_t B, int64_t C, int64_t F,
                          int64_t H, int64_t W, int64_t p, int32_t elem_bytes);

/* Kernel of the last successful patchify call on this thread: 1 vector, 2 element. */
int rope3d_patchify_last_kernel(void);

/*
 * rope3d_apply_neox -- NeoX-style rotary embedding of the Gemma3 text encoder
 * (sglang PR #24660 review, "关键源码片段", gemma_3.py _apply_rotary_pos_emb):
 * for each token, row positions[t] of cos_sin_cache = [cos | sin] is cast to
 * the input dtype and applied to both halves of every head of Q and K:
 *     y = x * cos + rotate_half(x) * sin,  rotate_half(x) = (-x2, x1),
 * x1, x2 the halves of head_dim, each tensor operation rounded to the input
 * dtype (products rounded once; sums rounded to float, then to the dtype).
 *
 *   q, k          device, [tokens, q_heads, head_dim] / [tokens, k_heads,
 *                 head_dim] contiguous, 4-byte aligned
 *   q_out, k_out  device outputs of the same shapes; q_out == q and/or
 *                 k_out == k rotate in place; otherwise an output overlaps
 *                 no input. An output never overlaps the other input, the
 *                 other output, the positions, the cache or the counter.
 *   positions     device int64 [tokens], 8-byte aligned
 *   cos_sin_cache device fp32 [max_position][head_dim], 4-byte aligned (16 for
 *                 the vector kernel); rotary_dim is head_dim
 *   dtype         ROPE3D_BF16, ROPE3D_F16 or ROPE3D_F32
 *   invalid_count optional device int32: a position outside [0, max_position)
 *                 leaves its outputs unwritten and adds the number of skipped
 *                 work units (16-byte vectors or pairs) here; the caller zeroes
 *                 it. NULL: skipped silently.
 *   stream        cudaStream_t; asynchronous
 * The bit-exact gate does not run here. Errors: NULL, SHAPE (sizes <= 0, odd
 * head_dim, head_dim > ROPE3D_MAX_HEAD_DIM), DTYPE, ALIGN, ALIAS, DEVICE, CUDA.
 */
int rope3d_apply_neox(const void *q, const void *k, void *q_out, void *k_out,
                      const int64_t *positions, const float *cos_sin_cache,
                      int64_t max_position, int64_t tokens, int64_t q_heads, int64_t k_heads,
                      int64_t head_dim, int32_t dtype, int32_t *invalid_count, void *stream);

/* The host-side checks of rope3d_apply_neox, without a launch or device queries. */
int rope3d_neox_check(const void *q, const void *k, const void *q_out, const void *k_out,
                      const int64_t *positions, const float *cos_sin_cache,
                      int64_t max_position, int64_t tokens, int64_t q_heads, int64_t k_heads,
                      int64_t head_dim, int32_t dtype, const int32_t *invalid_count);

/*
 * rope3d_neox_cache_host -- fill a host cos_sin_cache [max_position][rotary_dim]
 * in the layout above: cos then sin of p * base^(-2j/rotary_dim), j < rotary_dim/2,
 * in double, rounded once to float (standard RoPE angles; the page builds the
 * cache with get_rope and does not print its formula).
 * Errors: NULL, SHAPE, ARG (base).
 */
int rope3d_neox_cache_host(int64_t max_position, int64_t rotary_dim, double base, float *cache);

/* Kernel of the last successful rope3d_apply_neox on this thread: 1 vector, 2 pair. */
int rope3d_neox_last_kernel(void);

/*
 * rope3d_na3d -- 3D neighbourhood attention with the RoPE fused into its
 * prologue. The decoder rotates Q and K before each attention block ("功能与动机")
 * and attends with NATTEN's 3D neighbourhood attention (sglang PR #34471
 * review, "关键源码片段", _na3d); rotating the Q and K tiles inside the
 * attention kernel removes the write and re-read of Q_out and K_out.
 * The rotation is rope3d_apply_pair's, bit for bit (bf16 operands); the
 * attention is the published neighbourhood attention: a query attends to the
 * k_t x k_h x k_w window centred on it, shifted inside the grid at borders,
 * with softmax(q.k / sqrt(head_dim)); bf16 tensor-core products with fp32
 * accumulation (see the test hooks below for the two kernels), fp32 softmax,
 * bf16 output.
 *
 *   q, k, v, out  device, bf16, [B, T, H, W, heads, 128] contiguous, 16-byte
 *                 aligned; out overlaps no input
 *   tables, split as rope3d_apply_pair (used when apply_rope != 0; every
 *                 chunk a multiple of 8; tables <= 48 KB)
 *   kernel_size   (k_t, k_h, k_w), odd, each no larger than its grid extent
 *   apply_rope    1: rotate Q and K first (fused), as
 *                 rope3d_na3d_rotate_once does, with K rotated into scratch
 *                 of K's size that the library takes from a per-device
 *                 memory pool in stream order (cudaMallocFromPoolAsync before
 *                 the two launches, cudaFreeAsync after them; the pool keeps
 *                 the memory for later calls until rope3d_cache_clear trims
 *                 it); 0: Q and K are used as given (the unfused path's
 *                 second kernel).
 *   stream        cudaStream_t; asynchronous
 * Limits: head_dim 128; T, H, W < 1024. The bit-exact gate does not run here.
 * Errors: NULL, SHAPE, ALIGN (16 bytes), ALIAS, TABLES, DEVICE, CUDA.
 */
int rope3d_na3d(const void *q, const void *k, const void *v, void *out,
                const rope3d_tables *tables, int64_t B, int64_t T, int64_t H, int64_t W,
                int64_t heads, int64_t head_dim, const int32_t split[3],
                const int32_t kernel_size[3], int32_t apply_rope, void *stream);

/*
 * rope3d_na3d_rotate_once -- rope3d_na3d with the RoPE applied, rotating
 * every element of Q and K exactly once. A first kernel rotates K into k_rot
 * (16-byte vectors, rope3d_apply_pair's arithmetic); the attention kernel
 * then rotates each Q tile while staging it (a query tile is read by one CTA
 * only) and reads the keys from k_rot. Q_out is never written, and no key is
 * rotated more than once. The result is bit-identical to rope3d_apply_pair
 * followed by rope3d_na3d with apply_rope = 0, and k_rot holds that path's
 * K_out.
 *
 *   q, k, v, out, tables, B, T, H, W, heads, head_dim, split, kernel_size,
 *   stream        as rope3d_na3d with apply_rope = 1
 *   k_rot         device, bf16, K's shape, 16-byte aligned, caller-owned;
 *                 receives the rotated K. k_rot == k rotates K in place;
 *                 otherwise k_rot overlaps no other argument. In either case
 *                 k_rot overlaps none of q, v and out (so q may share K's
 *                 memory only when K is not rotated in place).
 * Two kernels on `stream`, asynchronous; the second is launched with
 * programmatic stream serialization and waits for the first before it reads
 * K. Limits as rope3d_na3d. The bit-exact gate does not run here.
 * Errors: NULL, SHAPE, ALIGN (16 bytes), ALIAS, TABLES, DEVICE, CUDA.
 */
int rope3d_na3d_rotate_once(const void *q, const void *k, const void *v, void *k_rot,
                            void *out, const rope3d_tables *tables, int64_t B, int64_t T,
                            int64_t H, int64_t W, int64_t heads, int64_t head_dim,
                            const int32_t split[3], const int32_t kernel_size[3], void *stream);

/*
 * rope3d_na3d_preflight -- the checks of rope3d_na3d (k_rot NULL) or of
 * rope3d_na3d_rotate_once (k_rot given) without a launch: the status that
 * call would return before launching. apply_rope as for rope3d_na3d (implied
 * when k_rot is given). check_device = 0 skips the device queries (the
 * tables' device and the pointers' memory type), so the pointer, size,
 * window, alignment, overlap and table-key checks run without a GPU.
 */
int rope3d_na3d_preflight(const void *q, const void *k, const void *v, const void *k_rot,
                          const void *out, const rope3d_tables *tables, int64_t B, int64_t T,
                          int64_t H, int64_t W, int64_t heads, int64_t head_dim,
                          const int32_t split[3], const int32_t kernel_size[3],
                          int32_t apply_rope, int32_t check_device);

/*
 * Test hooks of the neighbourhood attention. Its attention has two kernels:
 * one on the fifth-generation tensor cores (tcgen05 MMAs with fp32
 * accumulators in tensor memory; 2 x 8 x 8 query blocks; it needs key-region
 * rows of at most 112 keys, i.e. min(W, kw + 7) <= 112), the default wherever
 * that holds, and one on the warp-level MMAs, for every other geometry. Both
 * are held to the same bound of the oracle, and all rotation modes of one
 * kernel give the same bits.
 *   rope3d_testing_na3d_kernel(which): 0 = the default, 1 = the tensor-core
 *     kernel where the geometry allows it (the same as 0), 2 = the warp-MMA
 *     kernel always. Errors: ARG.
 *   rope3d_testing_na3d_last_kernel(): the kernel of this thread's last
 *     attention launch: 1 tensor-core, 2 warp-MMA, 0 none yet.
 *   rope3d_testing_na3d_per_cta(on): 1 = rope3d_na3d with apply_rope = 1
 *     runs the kernel form that rotates Q and every K tile inside each CTA
 *     (no scratch; every key is rotated by each of the CTAs whose key region
 *     holds it, which measured slower than rotating K once); 0 = the default.
 *     Errors: ARG.
 *   rope3d_testing_na3d_wait_timeouts(count, reset): how many bounded waits
 *     of the tensor-core kernel on its MMA completions ran out (0 unless
 *     something is badly wrong; such a launch's output is not to be used);
 *     reset clears the count. Synchronises with the device. Errors: NULL, CUDA.
 */
int rope3d_testing_na3d_kernel(int32_t which);
int rope3d_testing_na3d_last_kernel(void);
int rope3d_testing_na3d_per_cta(int32_t on);
int rope3d_testing_na3d_wait_timeouts(int64_t *count, int32_t reset);

/*
 * rope3d_apply_pair_host -- the same rotation for HOST buffers: the library
 * streams Q and K to the GPU in token chunks, rotates each chunk with the same
 * kernel, and streams Q_out and K_out back, overlapping the two copy
 * directions with the kernel. Returns when the outputs are in host memory.
 *
 *   q, k, q_out, k_out  host pointers with the layout of rope3d_apply_pair;
 *                       pinned (page-locked) memory gives full copy speed,
 *                       pageable memory works but copies synchronously
 *   other arguments     as for rope3d_apply_pair; `stream` orders the work
 *                       after earlier work on it
 *
 * Scratch: device staging buffers owned by the library (allocated on first
 * use, reused and grown as needed, freed by rope3d_release_scratch()).
 * The gate applies as in rope3d_apply_pair, on the host buffers.
 * Errors: as rope3d_apply_pair; DEVICE when a pointer is device memory;
 * NOMEM when the staging buffers cannot be allocated.
 */
int rope3d_apply_pair_host(const void *q, const void *k, void *q_out, void *k_out,
                           const rope3d_tables *tables,
                           int64_t B, int64_t T, int64_t H, int64_t W,
                           int64_t heads, int64_t head_dim, const int32_t split[3],
                           int32_t dtype, void *stream);

/* Free the staging buffers of rope3d_apply_pair_host (waits for the device). */
int rope3d_release_scratch(void);

/*
 * rope3d_apply_pair_noalloc -- rope3d_apply_pair for callers that cannot
 * allocate device memory. This call has no counterpart in the pages: it
 * exists because rope3d_build_tables allocates the cached tables with
 * cudaMalloc, and some callers cannot call cudaMalloc (a process whose device
 * memory belongs to another allocator or a fixed budget, or a pipeline that
 * must not take cudaMalloc's implicit synchronisation). This call takes no
 * table handle: it computes the three axis tables on the host (the values of
 * rope3d_build_tables) and uploads them into a fixed 64 KiB table area in the
 * library's static device memory, then launches the same kernels. It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 *   q, k, q_out, k_out, B, T, H, W, heads, head_dim, split, dtype, stream
 *           as for rope3d_apply_pair (device pointers, caller-owned; the
 *           library cannot see the buffers' extents, so the caller must pass
 *           buffers of [B, T*H*W, heads, head_dim] elements of `dtype`)
 *   base    RoPE base, finite and > 0
 *
 * Limit: the tables, sum over X of L_X * d_X/2 entries of 8 bytes with each
 * axis rounded up to 4 entries, must fit 64 KiB (8192 entries); larger grids
 * return ROPE3D_ERR_SCRATCH before anything is copied or launched. The table
 * area belongs to every GPU that loads the library until the process exits.
 * The first call on each device looks up the area's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * The address is kept for the life of the process, so calls after a
 * cudaDeviceReset of that device are unsupported.
 * Every call shares the one area and leaves its tables there; nothing in it
 * has to start at zero, because each call writes every entry it reads. Calls
 * are serialised on the host, and calls on one stream are ordered, but calls
 * whose work overlaps on the GPU (different streams) race on the area.
 * The upload comes from pageable host memory, so the call waits for earlier
 * work on `stream` before returning; a stream in capture mode cannot record
 * that upload and is refused with ROPE3D_ERR_ARG before anything is enqueued.
 * The bit-exact gate does not run here.
 * Errors: as rope3d_apply_pair (without TABLES and PARITY), ARG (base, or a
 * capturing stream), SCRATCH.
 */
int rope3d_apply_pair_noalloc(const void *q, const void *k, void *q_out, void *k_out,
                              int64_t B, int64_t T, int64_t H, int64_t W,
                              int64_t heads, int64_t head_dim, const int32_t split[3],
                              double base, int32_t dtype, void *stream);

/*
 * rope3d_preflight -- the argument checks of rope3d_apply_pair without a
 * launch ("关键源码片段", can_use_ltx25_decoder_rope: sizes > 0,
 * head_dim == sum(split), every chunk even and > 0, 4-byte pointer alignment,
 * table shapes (T, d_T/2), (H, d_H/2), (W, d_W/2); plus the overlap check).
 * check_device = 0 skips the device-memory query, so the host-only checks can
 * run without a GPU. Returns the status rope3d_apply_pair would return before
 * launching.
 */
int rope3d_preflight(const void *q, const void *k, const void *q_out, const void *k_out,
                     const rope3d_tables *tables,
                     int64_t B, int64_t T, int64_t H, int64_t W,
                     int64_t heads, int64_t head_dim, const int32_t split[3],
                     int32_t dtype, int32_t check_device);

/*
 * rope3d_axis_table_host -- the host table builder alone: fills cos_out and
 * sin_out (each [length][dim/2] floats, caller-owned host memory) with the
 * values described under rope3d_build_tables. No GPU needed.
 * Errors: NULL, SHAPE (length <= 0, dim <= 0 or odd), ARG (base).
 */
int rope3d_axis_table_host(int64_t length, int64_t dim, double base,
                           float *cos_out, float *sin_out);

/*
 * rope3d_dit_freqs_host -- the RoPE frequency vector of the LTX DiT (sglang
 * PR #24660 review, "关键源码片段", ltx_2.py, the device-side frequency
 * generation that replaced _ltx2_rope_freq_grid_np):
 *     freqs[i] = float32( theta ** linspace(0, 1, n)[i] * pi / 2 ),
 *     n = dim / num_rope_elems (integer division),
 * every step in float64 when double_precision != 0, else in float32. How the
 * page combines the vector with the positions grid is elided there and is not
 * provided here. Readings of what the page leaves to the framework: linspace
 * value i is the nearest value of the precision to i / (n - 1) (n = 1 gives
 * 0); the power is correctly rounded in the precision (the float32 power is
 * the float64 power rounded once); pi is the nearest value of the precision;
 * each product is rounded once and the halving is exact.
 *
 *   dim, num_rope_elems  > 0 with 1 <= dim / num_rope_elems <= 2^24
 *   theta                finite and > 0
 *   out                  caller-owned host memory of dim / num_rope_elems floats
 * No GPU needed. Errors: NULL, SHAPE, ARG (theta).
 */
int rope3d_dit_freqs_host(int64_t dim, int64_t num_rope_elems, double theta,
                          int32_t double_precision, float *out);

/*
 * rope3d_tables_info -- the key of a handle: dims = (T, H, W), split, base.
 * Any output pointer may be NULL.
 */
int rope3d_tables_info(const rope3d_tables *tables, int64_t dims[3],
                       int32_t split[3], double *base);

/*
 * rope3d_tables_read -- copy axis `axis` (0 = T, 1 = H, 2 = W) of a handle
 * into caller-owned host arrays of [L_X][d_X/2] floats. from_device = 0 reads
 * the library's host copy; 1 reads back the device copy the kernel uses.
 * Errors: NULL, ARG (axis), CUDA.
 */
int rope3d_tables_read(const rope3d_tables *tables, int32_t axis, int32_t from_device,
                       float *cos_out, float *sin_out);

/* ---- table cache --------------------------------------------------------- */
/* Counters since the last rope3d_cache_clear(); any pointer may be NULL. */
int rope3d_cache_stats(int64_t *entries, int64_t *hits, int64_t *misses,
                       int64_t *evictions);
/* Unlink every entry (held handles stay valid), zero the counters, and return
 * the memory that rope3d_na3d's scratch pools keep to the device. */
int rope3d_cache_clear(void);
/*
 * Free the released table buffers whose last launches have completed;
 * *waiting (may be NULL) receives how many released buffers are still waiting
 * for launches in flight. Never waits for the device.
 */
int rope3d_cache_retired(int64_t *waiting);

/* ---- verification gate ("实现拆解" step 4: BitExactFusionGate) ------------ */
#define ROPE3D_GATE_OFF   0  /* never verify                                   */
#define ROPE3D_GATE_FIRST 1  /* verify the first call of each configuration    */
int rope3d_gate_set_mode(int32_t mode);
int rope3d_gate_get_mode(void);
/* Forget every verdict. */
int rope3d_gate_reset(void);
/*
 * Verdict for a configuration: 0 = not seen yet, 1 = verified, 2 = refused.
 * Returns the verdict (>= 0) or a negative error code.
 */
int rope3d_gate_verdict(int64_t B, int64_t T, int64_t H, int64_t W, int64_t heads,
                        int64_t head_dim, const int32_t split[3], double base,
                        int32_t dtype);
/*
 * Test hook for the gate's failure path: the next `count` verifications flip
 * one bit of the host copy of the kernel's output before comparing, so they
 * must refuse. Never touches device memory.
 */
int rope3d_testing_corrupt_gate(int32_t count);

/* ---- introspection ------------------------------------------------------- */
/*
 * Which kernel the last successful rope3d_apply_pair / _host launch used on
 * this thread: 1 = 16-byte vector kernel, 2 = per-pair kernel, 0 = none yet.
 * grid and block receive the launch shape of the last kernel (may be NULL).
 */
int rope3d_last_launch(int32_t *grid, int32_t *block);

/* Name of a status code (static storage). */
const char *rope3d_status_string(int status);

/* ROPE3D_ABI_VERSION of the built library. */
int rope3d_abi_version(void);

/*
 * Host-side check of the integer division used by the kernels' index decode:
 * returns n / d computed with the precomputed multiplier the kernels use
 * (valid for 1 <= d < 2^31 and 0 <= n < 2^31), or -1 for arguments out of range.
 */
int64_t rope3d_testing_fastdiv(int64_t n, int64_t d);

/*
 * Test hook: 1 makes the table cache keep its tables in host memory instead
 * of device memory, so the cache logic can be exercised without a GPU; the
 * GPU entry points then refuse those handles with ROPE3D_ERR_DEVICE. Only
 * allowed while the cache is empty. 0 restores device memory.
 */
int rope3d_testing_host_tables(int32_t on);

/*
 * Test hook: cap the work units (16-byte vectors or pairs) of one kernel
 * launch at n, so that small inputs exercise the split into several launches
 * that very large inputs take (rows never straddle two launches; a row larger
 * than n gets a launch of its own). Applies to the rotation kernels and to
 * the K pass of rope3d_na3d_rotate_once. 0 restores the default cap of 2^30.
 * Errors: ARG for n < 0 or n > 2^30.
 */
int rope3d_testing_max_units_per_launch(int64_t n);

/*
 * rope3d_debug_bounds -- the bounds checks of a debug build. A library built
 * with -DROPE3D_DEBUG_BOUNDS=1 (build(debug_bounds=True)) checks every index
 * its kernels compute (table entries, strided and permuted offsets, token
 * and key positions, shared-memory slots) before the access it guards; a
 * failed check adds one to an error count and skips the access, so the kernel
 * finishes. This takes the place of a memory checker where none can run.
 *   errors  out: failed checks since the last reset (0 in a normal build)
 *   reset   nonzero: clear the count after reading it
 * Returns 1 when the library was built with the checks, 0 when not.
 * Synchronises the device (debug builds). Errors: NULL, CUDA.
 */
int rope3d_debug_bounds(int64_t *errors, int32_t reset);

/*
 * Test hook of the debug build: the rotation kernels see every table n
 * entries shorter than it is (the memory stays valid), so their table-index
 * checks must fire and count; 0 restores. Errors: ARG in a normal build or
 * for n < 0.
 */
int rope3d_testing_debug_shrink_tables(int32_t n);

#ifdef __cplusplus
}
#endif
#endif /* ROPE3D_H */
