/*
 * acnn.h -- C ABI of the GB300 (sm_103a) fused 2-D convolution library.
 *
 * Every entry point takes plain pointers and sizes, enqueues its work on the
 * caller's CUDA stream and returns an int status (ACNN_OK = 0).  Arguments are
 * validated on the host before anything is launched; a rejected call launches
 * nothing and returns an ACNN_ERR_* code.  No C++ exception crosses this ABI.
 *
 * Memory.  Every buffer is owned by the caller.  Pointers named "device" must
 * be device (or managed) memory of the current device; pointers named "host"
 * are host memory.  The library allocates no device memory on any call: the
 * one call that needs scratch space takes a caller-provided workspace whose
 * size acnn_conv2d_workspace_size() reports.  Outputs must not alias inputs.
 *
 * Asynchrony.  Calls return once the work is enqueued.  They neither
 * synchronise nor allocate, so they may be recorded into a CUDA graph with
 * stream capture (see the section runner at the end).
 *
 * Layouts.  Activations are NHWC (channels innermost, as in the inferencelayer
 * rtdetr_gpu.rs page) or NCHW (planes, as in the @framecast/rt rt.js page),
 * dense, with no padding between rows.  Conv weights are OHWI for NHWC
 * activations -- so that the GEMM reduction index k runs over (ky, kx, ci), the
 * order of rtdetr_gpu.rs IM2COL_SRC -- and OIHW for NCHW activations, the
 * [CO, CI, 3, 3] order of rt.js wgslConv.  Bias and PReLU alpha are always
 * fp32, as in rt.js wgslConv.  The companion ops index elements with 32 bits:
 * a tensor of 2^31 elements or more returns ACNN_ERR_TOO_LARGE.
 *
 * Alignment.  Device pointers must be 16-byte aligned (the tensor path reads
 * through TMA, which requires it); misaligned pointers return
 * ACNN_ERR_MISALIGNED.
 */
#ifndef ACNN_H_
#define ACNN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without the CUDA headers. NULL = legacy default stream. */
typedef struct CUstream_st* acnn_stream_t;

#define ACNN_VERSION 1

/* ---- status codes -------------------------------------------------------- */
enum {
    ACNN_OK = 0,
    ACNN_ERR_NULL_POINTER = 1,   /* a required pointer is NULL                   */
    ACNN_ERR_BAD_GEOMETRY = 2,   /* a size is <= 0, or the output would be empty  */
    ACNN_ERR_UNSUPPORTED = 3,    /* valid, but outside what this library covers   */
    ACNN_ERR_MISALIGNED = 4,     /* a device pointer is not 16-byte aligned       */
    ACNN_ERR_WORKSPACE = 5,      /* workspace NULL or smaller than required       */
    ACNN_ERR_ALIAS = 6,          /* the output overlaps an input                  */
    ACNN_ERR_BAD_ENUM = 7,       /* an enum argument is out of range              */
    ACNN_ERR_CUDA = 8,           /* a CUDA runtime/driver call failed             */
    ACNN_ERR_DEVICE_TIMEOUT = 9, /* a kernel's bounded pipeline wait expired      */
    ACNN_ERR_TOO_LARGE = 10      /* an index would overflow 32 bits               */
};

/* ---- enums --------------------------------------------------------------- */
typedef enum { ACNN_F32 = 0, ACNN_F16 = 1, ACNN_BF16 = 2 } acnn_dtype;
typedef enum { ACNN_NHWC = 0, ACNN_NCHW = 1 } acnn_layout;
/* Activations: relu(v) = max(v, 0) and silu(v) = v / (1 + exp(-v)) as in
 * rtdetr_gpu.rs ADDACT_SRC; prelu(v) = v >= 0 ? v : alpha[c] * v as in rt.js
 * wgslConv. */
typedef enum { ACNN_ACT_NONE = 0, ACNN_ACT_RELU = 1, ACNN_ACT_SILU = 2, ACNN_ACT_PRELU = 3 } acnn_act;
/* Residual: none; added before the activation, y = act(conv + res) (the
 * bottleneck's addact(relu) in rtdetr_gpu.rs); or after it, y = act(conv) + res
 * (rt.js wgslConv, dst = prelu(acc) + res). */
typedef enum { ACNN_RES_NONE = 0, ACNN_RES_ADD_THEN_ACT = 1, ACNN_RES_ACT_THEN_ADD = 2 } acnn_res;
typedef enum { ACNN_POOL_MAX = 0, ACNN_POOL_AVG = 1 } acnn_pool_kind;
typedef enum { ACNN_RESIZE_NEAREST = 0, ACNN_RESIZE_BILINEAR = 1 } acnn_resize_mode;

/* Geometry of one conv (or transposed conv) call.  n, h, w, c_in describe the
 * input; c_out the output channels; kh x kw the kernel; stride and pad are
 * the same along both axes.  dtype is the storage type of x, w, residual and
 * y; accumulation is always fp32. */
typedef struct {
    int n, h, w, c_in, c_out;
    int kh, kw, stride, pad;
    int layout; /* acnn_layout */
    int dtype;  /* acnn_dtype  */
} acnn_conv_desc;

/* ---- conv2d_fused ----------------------------------------------------------
 * y[n,oy,ox,co] = post(b[co] + sum_{ky,kx,ci} x[n, oy*s+ky-p, ox*s+kx-p, ci]
 *                                           * w[co,ky,kx,ci])
 * Taps outside the input read zero (rtdetr_gpu.rs IM2COL_SRC); the output
 * size is oh = (h + 2p - kh)/s + 1, ow likewise (rtdetr_gpu.rs RtDetrGpu::conv).
 * post = act for ACNN_RES_NONE; act(v + res) for ADD_THEN_ACT; act(v) + res for
 * ACT_THEN_ADD.  This is the conv of rtdetr_gpu.rs (im2col -> GEMM with the
 * bias and activation in the epilogue) and of rt.js wgslConv (PReLU, residual).
 *
 *   d          geometry (host pointer, read during the call only)
 *   x          device, input activations  [n,h,w,c_in] or [n,c_in,h,w]
 *   w          device, weights OHWI [c_out,kh,kw,c_in] (NHWC) or OIHW (NCHW)
 *   bias       device fp32 [c_out], or NULL for no bias
 *   alpha      device fp32 [c_out]; required iff act == ACNN_ACT_PRELU
 *   residual   device, same shape/layout/dtype as y; required iff res_mode != NONE
 *   y          device output [n,oh,ow,c_out] or [n,c_out,oh,ow]
 *   workspace  device scratch (contents clobbered), ws_bytes long.  Required:
 *              room for NHWC copies of x and w (NCHW calls on paths 1-2) or
 *              for the packed im2col matrix and weights (path 3).  Beyond
 *              that, up to acnn_conv2d_workspace_size(d) bytes let the
 *              tensor cores split K across more SMs (fewer bytes select fewer
 *              splits; NULL / 0 bytes is valid when nothing is required).
 * fp16/bf16 convs with c_out % 8 == 0 and c_out <= 4096 run on the tensor
 * cores: x is read by TMA (tiled for 1x1/s1/p0, im2col otherwise) when
 * c_in % 8 == 0 and the kernel is square; other such convs whose kh*kw*c_in is
 * at most 512 are first packed into an explicit im2col matrix in the
 * workspace.  Every other valid geometry (fp32 storage included) runs the
 * direct FFMA kernel.
 */
int acnn_conv2d_fused(const acnn_conv_desc* d, const void* x, const void* w,
                      const float* bias, const float* alpha, const void* residual,
                      int res_mode, int act, void* y, void* workspace, size_t ws_bytes,
                      acnn_stream_t stream);

/* conv2d_fused over the channel concatenation [x_a | x_b] without
 * materialising it (the concat of P1 CONCAT_SRC folded into the conv's
 * operand loads): d describes the conv on the concatenated input (c_in =
 * c_a + c_b channels); x_a is NHWC [n, h, w, c_a], x_b NHWC [n, h, w, c_b].
 * The result equals acnn_concat followed by acnn_conv2d_fused bit for bit
 * (the same operand values in the same k-block order).  Requires NHWC, fp16
 * or bf16, c_a a positive multiple of 64, c_b a positive multiple of 8 and a
 * geometry the tensor-core paths 1-2 take; else ACNN_ERR_UNSUPPORTED.  The
 * workspace is optional (split-K partial sums only); other arguments and
 * errors as acnn_conv2d_fused.
 */
int acnn_conv2d_fused_cat2(const acnn_conv_desc* d, const void* x_a, int c_a, const void* x_b,
                           const void* w, const float* bias, const float* alpha,
                           const void* residual, int res_mode, int act, void* y, void* workspace,
                           size_t ws_bytes, acnn_stream_t stream);

/* Output height and width of a conv with geometry d (host pointers). */
int acnn_conv2d_out_hw(const acnn_conv_desc* d, int* oh, int* ow);

/* Bytes of workspace for the fastest plan of geometry d: the staging copies
 * (required) plus split-K partial sums (optional). 0 when neither applies. */
size_t acnn_conv2d_workspace_size(const acnn_conv_desc* d);

/* Which kernel acnn_conv2d_fused would run for d: 0 = direct FFMA,
 * 1 = tcgen05 implicit GEMM with a tiled A load (1x1/s1/p0),
 * 2 = tcgen05 implicit GEMM with TMA im2col A loads,
 * 3 = explicit im2col pack, then the tcgen05 GEMM,
 * 4 = direct 3x3 kernel for fp16/bf16 inputs of 3, 6 or 7 channels (the input
 *     patch staged in shared memory, weights broadcast from shared memory or by
 *     warp shuffles); chosen only where path 3 cannot serve the geometry (path 3
 *     measured faster on the RGB stem and the 7-plane frame input) or when
 *     forced with acnn_conv2d_force_path;
 * negative = invalid. */
int acnn_conv2d_path(const acnn_conv_desc* d);

/* Tensor-core plan for d given ws_bytes of workspace: output pixels per tile
 * (*rows: 128/256), output channels per tile (*bn: 32/64/128/256) and K splits
 * (*splits, 1 = none; always 1 for NCHW, whose convs are never split).  Returns 0, or -1 when d does not take the tensor-core
 * path or ws_bytes is below the required staging (host pointers; the plan
 * depends on the current device's SM count). */
int acnn_conv2d_plan(const acnn_conv_desc* d, size_t ws_bytes, int* rows, int* bn, int* splits);

/* Tuning hook (the offline counterpart of rt.js's one-shot conv autotune,
 * tuneConvRB): force the tensor-core tile shape of every later conv call,
 * workspace query and plan query in this process -- bn output channels
 * (32/64/128/256) x rows output pixels (128/256) per tile, at most `splits`
 * K splits.  A shape the geometry has no kernel instantiation for is ignored
 * (the plan query reports what is used); splits are lowered until the split
 * units fit in one wave on the device and their partial sums in the
 * workspace.  bn = 0 restores the planner.  Process-wide, not per stream:
 * meant for tile sweeps (activation_cnn_gb300/tune.py), not for serving.
 * Returns ACNN_OK, or ACNN_ERR_BAD_GEOMETRY for values outside those sets. */
int acnn_conv2d_force_plan(int bn, int rows, int splits);

/* Tuning hook: force the direct tiny-C_in kernel (path = 4) for every later
 * conv whose geometry it serves (3, 6 or 7 input channels, 3x3, stride 1 or 2,
 * fp16/bf16), with its weights broadcast from shared memory (variant 0) or by
 * warp shuffles (variant 1); path = 0 restores the router.  Process-wide,
 * like acnn_conv2d_force_plan: for measuring one kernel against the other.
 * Returns ACNN_OK or ACNN_ERR_BAD_ENUM. */
int acnn_conv2d_force_path(int path, int variant);

/* ---- prepacked weights --------------------------------------------------------
 * The weights in the form the conv kernels read, made once (the pages convert
 * their weights once at start-up too), so that a call does not restage them:
 *   acnn_conv2d_prepacked_size(d)  bytes of the prepacked weight of geometry d
 *                                  (0 for an invalid d);
 *   acnn_conv2d_prepack(d, w, w_packed, stream)
 *                                  w (device, the layout acnn_conv2d_fused takes:
 *                                  OHWI for NHWC, OIHW for NCHW) -> w_packed
 *                                  (device, caller-owned, 16-byte aligned, no
 *                                  overlap with w): the packed [c_out][kp]
 *                                  matrix (K = kh*kw*c_in in (ky, kx, ci) order,
 *                                  zero-padded to kp) on path 3, OHWI on paths
 *                                  1-2, an unchanged copy on paths 0 and 4;
 *   acnn_conv2d_prepacked_workspace_size(d)
 *                                  the workspace of the prepacked call: the
 *                                  staged activation only, plus split-K sums;
 *   acnn_conv2d_fused_prepacked(...)
 *                                  acnn_conv2d_fused with w_packed in place of
 *                                  w: same arguments, results and errors.
 * A prepacked weight is valid for the geometry it was packed for only.
 */
size_t acnn_conv2d_prepacked_size(const acnn_conv_desc* d);
int acnn_conv2d_prepack(const acnn_conv_desc* d, const void* w, void* w_packed,
                        acnn_stream_t stream);
size_t acnn_conv2d_prepacked_workspace_size(const acnn_conv_desc* d);
int acnn_conv2d_fused_prepacked(const acnn_conv_desc* d, const void* x, const void* w_packed,
                                const float* bias, const float* alpha, const void* residual,
                                int res_mode, int act, void* y, void* workspace,
                                size_t ws_bytes, acnn_stream_t stream);

/* acnn_conv2d_fused_prepacked for an NCHW conv on the implicit-GEMM paths
 * (acnn_conv2d_path 1 or 2; y_nhwc also on path 3), with NHWC copies of its
 * activations, so that a chain of NCHW convs (rt.js run()'s conv stack) stages
 * each map once instead of per conv:
 *   x_nhwc  the input as NHWC [n][h][w][c_in] (device, 16-byte aligned), or
 *           NULL: staged from x in the workspace as acnn_conv2d_fused does.
 *           With x_nhwc the workspace needs no staging part (split-K sums only).
 *   y_nhwc  NHWC [n][oh][ow][c_out] (device, 16-byte aligned): the epilogue
 *           also writes y there -- the same values, bit for bit -- for the next
 *           conv's x_nhwc; NULL: none.
 * Neither may overlap another argument.  Returns ACNN_ERR_UNSUPPORTED when
 * d is NHWC or the path does not take the copies, otherwise the errors of
 * acnn_conv2d_fused_prepacked. */
int acnn_conv2d_fused_prepacked_staged(const acnn_conv_desc* d, const void* x,
                                       const void* x_nhwc, const void* w_packed,
                                       const float* bias, const float* alpha,
                                       const void* residual, int res_mode, int act, void* y,
                                       void* y_nhwc, void* workspace, size_t ws_bytes,
                                       acnn_stream_t stream);

/* ---- conv2d_fused without caller workspace ----------------------------------
 * No counterpart on the pages: an addition for callers that cannot allocate
 * device memory where they run a conv -- e.g. a plugin inside a framework
 * that owns all device memory and gives the plugin no allocator, or a
 * latency-critical loop in which cudaMalloc/cudaFree could synchronise the
 * device.  Same arguments, semantics and results as acnn_conv2d_fused, minus
 * the workspace: the scratch the NCHW tensor-core path needs is taken from a
 * static device array of ACNN_NOALLOC_SCRATCH_BYTES that the library holds on
 * every GPU that loads it, until the process exits.  Nothing is allocated or
 * freed (no cudaMalloc, cudaFree or allocating library call).
 *   - A call whose required scratch (the staging copies) exceeds
 *     ACNN_NOALLOC_SCRATCH_BYTES returns ACNN_ERR_WORKSPACE and launches nothing;
 *     optional split-K scratch is limited to what the array holds.
 *   - The first call on a device that needs scratch looks the array's device
 *     address up (cudaGetSymbolAddress) with that device current; make that
 *     first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents;
 *     nothing in it has to start at zero (each call overwrites what it reads).
 *     Calls whose kernels overlap on the GPU (other streams, other threads)
 *     race on it: serialise them.
 */
#define ACNN_NOALLOC_SCRATCH_BYTES (16u << 20)
int acnn_conv2d_fused_noalloc(const acnn_conv_desc* d, const void* x, const void* w,
                              const float* bias, const float* alpha, const void* residual,
                              int res_mode, int act, void* y, acnn_stream_t stream);

/* ---- conv with a pooled second output (cross-op fusion) --------------------
 * acnn_conv2d_fused_pool2: acnn_conv2d_fused of a 1x1/s1/p0 NHWC fp16/bf16
 * conv (C_in >= 64, even output height and width) that also writes
 * y_pool = the 2x2/s2 average pool of y (NHWC [n][oh/2][ow/2][c_out], same
 * dtype, caller-owned device buffer, 16-byte aligned, overlapping none of the
 * other buffers).  rtdetr_gpu.rs RtDetrGpu::encoder_maps runs AVGPOOL_SRC as a
 * kernel of its own on a stage's last bottleneck output, feeding the next
 * stage's shortcut; here the conv that writes that output also writes its
 * pooled map: each epilogue warp owns whole 2x2 windows (the conv's tiles are
 * rectangles of 16 x 8 or 8 x 16 pixels) and averages the four stored values
 * as the pool does, ((a + b) + c) + d in fp32 times 0.25 rounded once, so
 * y_pool equals acnn_pool2d(ACNN_POOL_AVG, 2, 2, 0) of y bit for bit.  No
 * workspace (no K split).  Returns ACNN_ERR_UNSUPPORTED for other geometries,
 * otherwise the errors of acnn_conv2d_fused; nothing is launched on error.
 */
int acnn_conv2d_fused_pool2(const acnn_conv_desc* d, const void* x, const void* w,
                            const float* bias, const float* alpha, const void* residual,
                            int res_mode, int act, void* y, void* y_pool, acnn_stream_t stream);

/* acnn_conv2d_fused_up2: acnn_conv2d_fused (x_b NULL; c_a ignored) or
 * acnn_conv2d_fused_cat2 (x_b non-NULL: channels [0, c_a) from x_a, the rest
 * from x_b) of an NHWC fp16/bf16 conv on the tensor-core paths that also
 * writes y_up = the nearest 2x upsample of y (NHWC [n][2 oh][2 ow][c_out],
 * same dtype, caller-owned device buffer, 16-byte aligned, overlapping none of
 * the other buffers).  rtdetr_gpu.rs RtDetrGpu::encoder_maps upsamples a
 * neck map with UPSAMPLE_SRC, a kernel of its own, right after the conv that
 * writes it; here that conv's epilogue writes each stored 16-byte piece of y
 * into the 2 x 2 block of y_up it maps to as well, so y_up equals
 * acnn_resize2d(ACNN_RESIZE_NEAREST, 2 oh, 2 ow) of y bit for bit.  Workspace
 * as acnn_conv2d_fused (split-K partial sums only).  Returns
 * ACNN_ERR_UNSUPPORTED for other geometries, ACNN_ERR_TOO_LARGE when y_up
 * would pass 2^31 - 1 pixels, otherwise the errors of acnn_conv2d_fused.
 */
int acnn_conv2d_fused_up2(const acnn_conv_desc* d, const void* x_a, int c_a, const void* x_b,
                          const void* w, const float* bias, const float* alpha,
                          const void* residual, int res_mode, int act, void* y, void* y_up,
                          void* workspace, size_t ws_bytes, acnn_stream_t stream);

/* ---- pool2d ----------------------------------------------------------------
 * MAX: y = max over the in-range taps of each k x k window at stride s, pad p
 *      (taps outside the input are skipped: -inf padding), rtdetr_gpu.rs
 *      MAXPOOL_SRC.  Bit-exact.
 * AVG: y = (sum of the k x k window) * (1/k^2), pad must be 0 (the 2x2/s2
 *      (a+b+c+d)*0.25 of rtdetr_gpu.rs AVGPOOL_SRC); accumulated in fp32.
 * x, y: device, layout/dtype as given; y has oh = (h + 2p - k)/s + 1 rows.
 */
int acnn_pool2d(int kind, int n, int h, int w, int c, int k, int stride, int pad,
                int layout, int dtype, const void* x, void* y, acnn_stream_t stream);

/* ---- resize2d --------------------------------------------------------------
 * NEAREST:  y[oy,ox] = x[floor(oy*h/oh), floor(ox*w/ow)]; the 2x case is
 *           rtdetr_gpu.rs UPSAMPLE_SRC.  Bit-exact (in_dtype must equal out_dtype).
 * BILINEAR: align_corners=false, src = (dst + 0.5)*(in/out) - 0.5, taps
 *           clamped to the image (rt.js wgslPrepQuarter, wgslFlowOut).
 * x: device [n,c,h,w]/[n,h,w,c] of in_dtype; y: device, oh x ow, out_dtype.
 */
int acnn_resize2d(int mode, int n, int c, int h, int w, int oh, int ow, int layout,
                  int in_dtype, int out_dtype, const void* x, void* y, acnn_stream_t stream);

/* ---- concat ----------------------------------------------------------------
 * Channel concat y = [a | b] (rtdetr_gpu.rs CONCAT_SRC): per pixel for NHWC,
 * per image plane block for NCHW.  a: device [.., c_a], b: device [.., c_b],
 * y: device [.., c_a + c_b], all of dtype.  Bit-exact.
 */
int acnn_concat(int n, int h, int w, int c_a, int c_b, int layout, int dtype,
                const void* a, const void* b, void* y, acnn_stream_t stream);

/* ---- deconv2d --------------------------------------------------------------
 * Transposed conv, rt.js wgslDeconv (gather form):
 *   y[co,oy,ox] = b[co] + sum over (ky,kx) with ty = oy + p - ky >= 0, even,
 *                 iy = ty/s < h (same along x) of sum_ci x[ci,iy,ix]*w[ci,co,ky,kx]
 * then act.  Only kh = kw = 4, stride 2, pad 1 is supported (oh = 2h).
 *   d      geometry; d->dtype is the type of x
 *   x      device input, d->layout
 *   w      device fp32 [c_in, c_out, 4, 4]   (fp32 as on the page)
 *   bias   device fp32 [c_out] or NULL; alpha as for conv2d_fused
 *   y      device output [n, c_out, 2h, 2w] (or NHWC) of out_dtype
 */
int acnn_deconv2d(const acnn_conv_desc* d, const void* x, const float* w, const float* bias,
                  const float* alpha, int act, int out_dtype, void* y, acnn_stream_t stream);

/* The deconv on the tensor cores, for fp16 with out_dtype fp16 and
 * c_in % 8 == 0 (its weights are rounded to fp16): regrouped as a 3x3/s1/p1 conv to 4 c_out output
 * channels (channel co * 4 + py * 2 + px of the conv's pixel (a, b) is the
 * deconv's output (co, 2a + py, 2b + px): rt.js wgslDeconv's gather form,
 * grouped by output parity), then a pixel shuffle.  The weights and bias are
 * regrouped (and the weights rounded to the storage type) in the workspace on
 * every call.
 *   acnn_deconv2d_workspace_size(d, out_dtype)  bytes of workspace, 0 when
 *                                  this form does not serve d;
 *   acnn_deconv2d_ws(...)          acnn_deconv2d's arguments plus the
 *                                  workspace (caller-owned device memory,
 *                                  16-byte aligned, overlapping no argument);
 *                                  with no or too small a workspace, or a
 *                                  geometry this form does not serve, it is
 *                                  acnn_deconv2d.  Same errors. */
size_t acnn_deconv2d_workspace_size(const acnn_conv_desc* d, int out_dtype);
int acnn_deconv2d_ws(const acnn_conv_desc* d, const void* x, const float* w, const float* bias,
                     const float* alpha, int act, int out_dtype, void* y, void* workspace,
                     size_t ws_bytes, acnn_stream_t stream);

/* ---- frame prep ------------------------------------------------------------
 * rt.js wgslPrepQuarter: two h x w RGBA8 frames (bytes R,G,B,A per pixel,
 * device) -> y = [7, h/4, w/4] NCHW of out_dtype (device): the planes B, G, R
 * of frame 0, then of frame 1, each a bilinear 1/4 downsample of byte/255,
 * then a plane filled with t.  h and w must be multiples of 4.
 */
int acnn_frame_prep_quarter(int h, int w, const uint8_t* rgba0, const uint8_t* rgba1, float t,
                            int out_dtype, void* y, acnn_stream_t stream);

/* ---- frame flow-out ----------------------------------------------------------
 * rt.js wgslFlowOut (the stage after the deconv of the frame stack), with
 * wgslPrepFull's full-resolution planes read straight from the frames.
 *   tmp8       device [5, h/8, w/8] NCHW of tmp8_dtype: flow of frame 0 (x, y),
 *              flow of frame 1 (x, y), mask logit
 *   rgba0/1    device h x w RGBA8 frames (bytes R, G, B, A per pixel)
 *   refine_res device [3, h/4, w/4] fp32 (planes B, G, R), the refine head's
 *              residual (rt.js tfact2, withRes), or NULL for none
 *   out_rgba   device h x w RGBA8 output
 * Per output pixel: the five planes upsampled x8 (bilinear, align_corners=
 * false, clamped taps), flows times 8, m = 1/(1+exp(-mask)); each frame's
 * B, G, R (byte/255) sampled bilinearly at (x, y) + its flow with clamped taps
 * (grid_sample border, align_corners=true); v = w0*m + w1*(1-m), plus, with a
 * residual, its x4 bilinear upsample (align_corners=false, clamped taps);
 * output bytes R, G, B = (uint)(clamp(v, 0, 1) * 255) (truncation), A = 255.
 * Computed in binary32 in one fixed order without fused multiply-adds; exp by
 * Cody-Waite reduction and a degree-7 Taylor polynomial.  h and w multiples of
 * 8; all pointers 16-byte aligned; out_rgba must not overlap an input.
 */
int acnn_frame_flow_out(int h, int w, const void* tmp8, int tmp8_dtype, const uint8_t* rgba0,
                        const uint8_t* rgba1, const float* refine_res, uint8_t* out_rgba,
                        acnn_stream_t stream);

/* ---- t-factored frame stack (rt.js tfact / tfact2) --------------------------
 * Refine prep, rt.js wgslRefinePrep: the refine head's input y = [11, h/4, w/4]
 * NCHW of out_dtype (device) from the same tmp8 and frames as the flow-out
 * stage.  For each quarter-resolution pixel (hx, hy), over the four pixels
 * (4 hx + i, 4 hy + j), i, j in {1, 2} (the centre 2x2 of its 4x4 block, the
 * taps of a 1/4 bilinear downsample with align_corners=false): the mean of
 * warped frame 0 (B, G, R), warped frame 1 (B, G, R) and the sigmoid mask,
 * then the mean of the four x8 flows (u0, v0, u1, v1) times 0.25 / 20.
 * Upsample and warp as in acnn_frame_flow_out; fp32 arithmetic, one rounding
 * to out_dtype on store.  h and w multiples of 8; pointers 16-byte aligned;
 * y must not overlap an input.
 */
int acnn_frame_refine_prep(int h, int w, const void* tmp8, int tmp8_dtype, const uint8_t* rgba0,
                           const uint8_t* rgba1, int out_dtype, void* y, acnn_stream_t stream);

/* Refine out, rt.js wgslRefineOut: y[co] = 2 sigmoid(b[co] + sum over ci, ky,
 * kx of x[ci][clamp(oy+ky-1)][clamp(ox+kx-1)] * w[co][ci][ky][kx]) - 1 for
 * co = 0..2 -- a 3x3 conv C -> 3 with replicate (clamped-index) padding.
 *   x  device [c, hh, hw] NCHW of dtype (16-byte aligned)
 *   w  device fp32 [3, c, 3, 3];  bias device fp32 [3]
 *   y  device fp32 [3, hh, hw] (16-byte aligned, no overlap with the inputs)
 * fp32 accumulation, in input-channel order.
 */
int acnn_frame_refine_out(int c, int hh, int hw, const void* x, int dtype, const float* w,
                          const float* bias, float* y, acnn_stream_t stream);

/* FiLM, rt.js wgslFilm with filmParams: the timestep MLP
 *   s[k] = b2[k] + sum_j w2[k][j] * max(0, w0[j] * t + b0[j]),  k < 2c,
 * evaluated on the device (the page runs it on the host), then
 *   y[ci][i] = x[ci][i] * (1 + s[ci]) + s[c + ci]   (i < n, one plane per channel)
 * with x, y device [c, n] of dtype (y may be x itself, else no overlap);
 * w0, b0 device fp32 [hn]; w2 device fp32 [2c, hn]; b2 device fp32 [2c];
 * c <= 65535.  One kernel on stream; fp32 arithmetic, one rounding to dtype
 * on store.
 */
int acnn_film(int c, long long n, int dtype, const void* x, float t, const float* w0,
              const float* b0, int hn, const float* w2, const float* b2, void* y,
              acnn_stream_t stream);

/* ---- status ------------------------------------------------------------------ */
/* Static string for a status code. */
const char* acnn_status_string(int status);

/* Synchronises stream, then returns and clears the device status word that
 * kernels set when a bounded pipeline wait expires (ACNN_OK if none did), or
 * ACNN_ERR_CUDA if a CUDA error is pending. */
int acnn_last_device_status(acnn_stream_t stream);

/* Debug knob for fault tests: the spin budget (in polls) of every bounded
 * device wait in later launches; 0 restores the default.  Host state only. */
int acnn_set_wait_budget(long long polls);

/* ---- section runner ---------------------------------------------------------
 * One CUDA graph per network section, the GPU form of rtdetr_gpu.rs's
 * Recorder (one submit per section) and rt.js's one command buffer per frame.
 * acnn_section_begin starts stream capture on stream; the ABI calls that
 * follow are recorded, not run; acnn_section_end ends the capture and returns
 * an instantiated executable graph in *exec (host handle owned by the caller,
 * released with acnn_section_destroy); acnn_section_launch replays it on a
 * stream.  Buffers recorded into a graph must outlive it.
 */
int acnn_section_begin(acnn_stream_t stream);
int acnn_section_end(acnn_stream_t stream, void** exec);
int acnn_section_launch(void* exec, acnn_stream_t stream);
int acnn_section_destroy(void* exec);

/* Number of SMs of the current device (host query, cached). */
int acnn_device_sm_count(void);

#ifdef __cplusplus
}
#endif

#endif /* ACNN_H_ */
