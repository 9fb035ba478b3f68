/*
 * na3d.h - C ABI of the GB300 (sm_103a) forward pass of 3-D neighborhood
 * attention (NA3D).
 *
 * The operation ("[Triton/Gluon] Add 3D neighborhood flash attention
 * (na3d_flash)", ROCm/aiter pull request 5230):
 *   - Motivation: the token at grid position (t,h,w) of a video latent
 *     attends only to its KT x KH x KW neighbours.
 *   - Technical Details, kernel bullets: windows shift inward at the grid
 *     borders so that every window holds exactly KT*KH*KW keys; the softmax
 *     runs online in log2 space.
 *   - Technical Details, launcher: inputs and output are (B, T, H, W, NH, HD)
 *     bfloat16, and q arrives already multiplied by head_dim^-0.5.
 *
 * On each axis of length N with odd window length K <= N, the query at i uses
 * keys [s, s+K) with s = min(max(i - K/2, 0), N - K) (integer division).
 * Scores are q.k accumulated in fp32, the softmax over the window runs in
 * fp32, the probabilities are rounded to bf16 for the P.V product (fp32
 * accumulation), and the output is rounded to bf16 (nearest even).
 *
 * The library allocates no memory and is safe to call from several host
 * threads at once. Its only state is a mutex-guarded cache of tiling plans
 * (keyed by grid and window sizes) and, per device, one word that records a
 * pipeline-wait timeout plus the small table of words through which
 * na3d_device_status takes it (see there).
 */
#ifndef NA3D_H
#define NA3D_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum na3d_status {
    NA3D_OK = 0,
    NA3D_ERR_NULL = 1,           /* a required pointer is NULL */
    NA3D_ERR_SHAPE = 2,          /* a size < 1, or a query box outside the grid */
    NA3D_ERR_KERNEL = 3,         /* a window length is even, < 1, or larger than its axis */
    NA3D_ERR_HEAD_DIM = 4,       /* HD is not a power of two >= 16 */
    NA3D_ERR_ALIGN = 5,          /* a tensor pointer is not 16-byte aligned */
    NA3D_ERR_ALIAS = 6,          /* out overlaps q, k or v */
    NA3D_ERR_OVERFLOW = 7,       /* a size overflows int64 or a TMA descriptor limit */
    NA3D_ERR_ARCH = 8,           /* the current device is not compute capability 10.3 */
    NA3D_ERR_CUDA = 9,           /* a CUDA runtime or driver call failed */
    NA3D_ERR_DEVICE_TIMEOUT = 10, /* a pipeline wait inside the kernel gave up */
    NA3D_ERR_UNSUPPORTED = 11    /* valid but not implemented (no current argument returns it) */
};

/*
 * na3d_fwd - out = NA3D(q, k, v) for one bf16 (B,T,H,W,NH,HD) problem.
 *
 * The operation of "[Triton/Gluon] Add 3D neighborhood flash attention
 * (na3d_flash)" (ROCm/aiter pull request 5230), Technical Details: the query
 * at (t,h,w) attends to the KT x KH x KW keys of its window, shifted inward at
 * the grid borders so that it always holds KT*KH*KW keys (the start rule is
 * stated at the top of this file); the launcher's convention that q arrives
 * already multiplied by head_dim^-0.5 and that inputs and output share the
 * (B,T,H,W,NH,HD) bf16 layout.
 *
 * q, k, v, out: DEVICE pointers to contiguous row-major bf16 tensors of shape
 *   (B, T, H, W, NH, HD) (HD fastest), each 16-byte aligned. The caller owns
 *   all four buffers; the library neither allocates nor frees memory.
 *   q must already be scaled by HD^-0.5: no scale is applied. q, k and v are
 *   read only and may alias one another; out must not overlap any of them.
 * B: batch size, T, H, W: grid sizes, NH: heads, all >= 1 (a size < 1,
 *   including an empty batch, returns NA3D_ERR_SHAPE).
 * HD: head dimension, a power of two >= 16, with NH*HD < 2^31 (else
 *   NA3D_ERR_OVERFLOW). Above 256 the output is computed in passes of 256
 *   columns that recompute the same scores (slower per column, same result).
 * KT, KH, KW: odd window lengths with 1 <= KT <= T, 1 <= KH <= H, 1 <= KW <= W.
 * stream: a cudaStream_t on the current device (NULL = legacy default stream).
 *
 * The call validates its arguments, encodes the TMA descriptors on the host
 * and enqueues one kernel on `stream`; it returns before the kernel runs. An
 * argument error returns its code before anything is enqueued (out is not
 * written). NA3D_ERR_CUDA reports a failed launch or descriptor encoding.
 * Faults inside the kernel surface through the stream as usual; a pipeline
 * wait that gives up is reported by na3d_device_status(). The launch may be
 * captured into a CUDA graph on `stream` (the tensor maps are passed by
 * value and the plan is chosen at capture time); replays read the buffers
 * the call was given. na3d_device_status synchronizes and cannot be captured.
 */
int na3d_fwd(const void* q, const void* k, const void* v, void* out,
             int64_t B, int64_t T, int64_t H, int64_t W, int64_t NH, int64_t HD,
             int64_t KT, int64_t KH, int64_t KW, void* stream);

/*
 * na3d_fwd_strided - na3d_fwd for inputs whose grid positions are not packed:
 * q, k and v each hold, for token p = ((b*T + t)*H + h)*W + w, its NH heads
 * of HD values at  base + p*token_stride + head*HD  (elements). This is the
 * layout of a fused QKV projection output [B,T,H,W,3,NH,HD]: token_stride =
 * 3*NH*HD, with q, k, v pointing at the three blocks of the first token, so
 * the projection output feeds the attention without a gather copy (the
 * copy the pages' benchmark pays: "[Triton/Gluon] Add 3D neighborhood flash
 * attention (na3d_flash)", Performance table, "times include the wrapper's
 * v.contiguous() staging copy").
 *
 * q_token_stride, k_token_stride, v_token_stride: >= NH*HD, in elements; a
 * stride times 2 bytes must be a multiple of 16. out stays contiguous
 * (B,T,H,W,NH,HD) and must not overlap the memory spanned by q, k or v.
 * All other arguments, the errors and the asynchrony are those of na3d_fwd;
 * a bad stride returns NA3D_ERR_SHAPE (too small) or NA3D_ERR_ALIGN.
 */
int na3d_fwd_strided(const void* q, const void* k, const void* v, void* out,
                     int64_t B, int64_t T, int64_t H, int64_t W, int64_t NH, int64_t HD,
                     int64_t KT, int64_t KH, int64_t KW, int64_t q_token_stride,
                     int64_t k_token_stride, int64_t v_token_stride, void* stream);

/*
 * na3d_fwd_region - queries on a box of the grid, keys and values on the whole
 * grid: out = NA3D(q, k, v) restricted to the grid positions (t0 + t, h0 + h,
 * w0 + w), 0 <= t < Tq, 0 <= h < Hq, 0 <= w < Wq. Every query keeps the window
 * it has in the whole grid (global coordinates, shifted inward at the grid's
 * borders, never at the box's), so the result equals the matching rows of
 * na3d_fwd on the whole grid. This generalises the test reference's
 * `w_offset` mode ("[Triton/Gluon] Add 3D neighborhood flash attention
 * (na3d_flash)", Technical Details, test file: q a W sub-slice, k and v the
 * full tensors, bounds in global W coordinates) to a box on all three axes:
 * tiles of a decoded video are computed with exact borders.
 *
 * q: (B, Tq, Hq, Wq, NH, HD) tokens with q_token_stride elements between
 *   consecutive positions of the box (heads packed).
 * k, v: (B, T, H, W, NH, HD), the whole grid, with k_token_stride and
 *   v_token_stride elements between consecutive grid positions.
 * out: contiguous (B, Tq, Hq, Wq, NH, HD); must not overlap the memory that
 *   q, k or v span.
 * t0, h0, w0 >= 0 and Tq, Hq, Wq >= 1 with t0 + Tq <= T, h0 + Hq <= H,
 *   w0 + Wq <= W; otherwise NA3D_ERR_SHAPE. Windows satisfy KT <= T,
 *   KH <= H, KW <= W (the box may be narrower than a window).
 * All other arguments, the errors and the asynchrony are those of
 * na3d_fwd_strided; na3d_fwd_strided is this call with the whole grid as the
 * box (t0 = h0 = w0 = 0, Tq = T, Hq = H, Wq = W).
 */
int na3d_fwd_region(const void* q, const void* k, const void* v, void* out,
                    int64_t B, int64_t T, int64_t H, int64_t W, int64_t NH, int64_t HD,
                    int64_t KT, int64_t KH, int64_t KW,
                    int64_t t0, int64_t h0, int64_t w0, int64_t Tq, int64_t Hq, int64_t Wq,
                    int64_t q_token_stride, int64_t k_token_stride, int64_t v_token_stride,
                    void* stream);

/*
 * na3d_qkv_proj - the fused QKV projection that feeds the attention:
 *   qkv[m][n] = bf16( s_n * ( sum_c x[m][c] * w[n][c] + bias[n] ) ),
 *   s_n = HD^-0.5 (rounded to fp32) for n < NH*HD (the q block), else 1,
 * with the sum and the bias added in fp32 and one rounding to bf16 (nearest
 * even). The decoder attention of "LTX-2.5 optimization: integrate faster
 * AITER NA3D flash attention for diffusion decoder" (xDiT pull request 773,
 * Summary; Notes) projects q, k and v with one concatenated weight and takes
 * q, k, v as views of the result; the attention wants q already scaled by
 * HD^-0.5 ("[Triton/Gluon] Add 3D neighborhood flash attention (na3d_flash)",
 * Technical Details, launcher). A row of qkv is [q heads | k heads | v heads],
 * i.e. (M, 3, NH, HD): pass qkv, qkv + NH*HD and qkv + 2*NH*HD (elements) to
 * na3d_fwd_strided with token strides 3*NH*HD, and M = B*T*H*W tokens in
 * (b, t, h, w) order.
 *
 * x: DEVICE pointer, bf16 (M, C) row-major (a token's C input channels).
 * w: DEVICE pointer, bf16 (3*NH*HD, C) row-major (one output feature per
 *   row, as a linear layer's weight), q rows first, then k, then v.
 * bias: DEVICE pointer, bf16 (3*NH*HD), or NULL for none.
 * qkv: DEVICE pointer, bf16 (M, 3*NH*HD) row-major; must not overlap x, w or
 *   bias. x, w and qkv are 16-byte aligned; C is a multiple of 8 (16-byte
 *   rows), else NA3D_ERR_ALIGN.
 * M >= 1 tokens, NH >= 1 heads, C >= 1 (else NA3D_ERR_SHAPE), HD a power
 *   of two >= 16.
 * Asynchronous on `stream`; errors as for na3d_fwd. na3d_device_status also
 * reports a pipeline wait of this kernel that gave up.
 */
int na3d_qkv_proj(const void* x, const void* w, const void* bias, void* qkv,
                  int64_t M, int64_t C, int64_t NH, int64_t HD, void* stream);

/*
 * na3d_selftest_withhold - a self-test of the kernel's failure detection:
 * na3d_fwd on contiguous tensors, except that CTA 0 does not issue the load
 * of its K chunk number `chunk` (0-based, in its own order). The score-tile
 * wait for that chunk runs out after about 2 s; the CTA then records the
 * timeout, drains its in-flight copies and MMAs, frees its tensor memory and
 * exits, and na3d_device_status() returns NA3D_ERR_DEVICE_TIMEOUT. out is
 * left partly unwritten. The stream and the device stay usable. Not for
 * production use. chunk < 0 returns NA3D_ERR_SHAPE; other arguments and
 * errors as na3d_fwd.
 */
int na3d_selftest_withhold(const void* q, const void* k, const void* v, void* out,
                           int64_t B, int64_t T, int64_t H, int64_t W, int64_t NH, int64_t HD,
                           int64_t KT, int64_t KH, int64_t KW, int64_t chunk, void* stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* na3d_status_string(int status);

/*
 * How na3d_fwd tiles one (batch, head) slice: queries are cut into bricks of
 * bt x bh x bw grid positions (at most 128 queries, one tile of the tensor
 * cores), and each brick streams the union of its queries' windows (its halo)
 * through shared memory in chunks of cr rows (consecutive h) of cw keys
 * (consecutive w) in one frame t. The scores of a chunk form one
 * 128 x n_mma tile (n_mma <= tile_cap).
 */
typedef struct na3d_plan_info {
    int32_t bt, bh, bw;           /* query brick */
    int32_t cw, cr;               /* chunk: cr rows of cw keys */
    int32_t n_mma;                /* score-tile width (cr*cw rounded up to 16) */
    int32_t hd_box;               /* head-dim columns per TMA box (HD or 64) */
    int32_t stages;               /* K/V shared-memory pipeline depth */
    int64_t bricks_per_slice;     /* bricks per (batch, head) slice */
    int64_t chunks_per_slice;     /* chunks per (batch, head) slice */
    int64_t smem_bytes;           /* dynamic shared memory per CTA */
    int32_t w_stride;             /* 8, 12, 14, 16 or 32: chunk rows padded to this many keys
                                     and the W window applied by the tensor core (12 and 14
                                     for HD 64 and 128 only); 1: every W window
                                     is the whole axis (KW == W), chunk rows are whole grid
                                     rows and the H window is applied by the tensor core;
                                     0: per-key masks */
    int32_t tile_cap;             /* score-tile capacity of the kernel instance: 128 (HD <= 64) or
                                     64 (HD >= 128), or 96 for the HD <= 64 instances whose score
                                     tiles are double-buffered (the next one is computed while
                                     the softmax works on the current one) */
} na3d_plan_info;

/*
 * na3d_plan - the tiling na3d_fwd would use for this problem, computed on the
 * host without touching a GPU. Arguments as for na3d_fwd; returns the same
 * argument-validation codes (without the pointer, alignment, alias and device
 * checks). `info` must not be NULL.
 */
int na3d_plan(int64_t T, int64_t H, int64_t W, int64_t NH, int64_t HD,
              int64_t KT, int64_t KH, int64_t KW, na3d_plan_info* info);

/*
 * na3d_device_status - after the work already enqueued on `stream`, takes
 * the current device's timeout flag and synchronizes `stream`. The flag is
 * set by any na3d kernel on the device whose pipeline wait gave up (a
 * deadlock guard: each wait inside the kernels is bounded, and a wait that
 * runs out records the flag, drains its in-flight copies and MMAs, frees its
 * tensor memory and returns, leaving part of its output unwritten).
 * "Takes" means read and cleared in one atomic step on the device: each
 * timeout is reported by exactly one call. The flag is per device, not per
 * launch: with several threads or streams launching on one device, the call
 * reports a timeout of any of their launches that completed before it.
 * Returns NA3D_ERR_DEVICE_TIMEOUT if the flag was set, NA3D_ERR_CUDA if the
 * enqueue or the synchronization fails, else NA3D_OK.
 */
int na3d_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* NA3D_H */
