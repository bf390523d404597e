// common.cuh -- device helpers shared by the kernels of libacnn (sm_103a).
//
// Storage types, fp32 conversion, the fused epilogue (bias -> activation /
// residual -> down-cast) and launch-shape helpers.  Nothing here is shared
// with the oracle.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/acnn.h"

namespace acnn {

// ---------------------------------------------------------------- storage types
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

// fp32 -> storage type, round to nearest even (the reading used where the
// pages leave the f32 -> f16 store rounding open).
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// A vector of V storage elements moved as one aligned load/store.
template <typename T, int V> struct alignas(sizeof(T) * V) Vec {
    T v[V];
};

// ---------------------------------------------------------------- activations
// relu = max(v, 0) and silu = v / (1 + exp(-v)) as in rtdetr_gpu.rs ADDACT_SRC;
// prelu = v >= 0 ? v : alpha * v as in rt.js wgslConv.
__device__ __forceinline__ float apply_act(int act, float v, float alpha) {
    switch (act) {
    case ACNN_ACT_RELU: return fmaxf(v, 0.0f);
    case ACNN_ACT_SILU: return v / (1.0f + expf(-v));
    case ACNN_ACT_PRELU: return v >= 0.0f ? v : alpha * v;
    default: return v;
    }
}

// Epilogue of conv2d_fused on the bias-added accumulator v:
//   RES_NONE: act(v); ADD_THEN_ACT: act(v + r); ACT_THEN_ADD: act(v) + r.
__device__ __forceinline__ float epilogue(float v, int act, float alpha, int res_mode, float r) {
    if (res_mode == ACNN_RES_ADD_THEN_ACT) return apply_act(act, v + r, alpha);
    float a = apply_act(act, v, alpha);
    return res_mode == ACNN_RES_ACT_THEN_ADD ? a + r : a;
}

// Out-of-line copy of epilogue() for kernels whose epilogue is not hot: keeps
// one copy of the activation code instead of one per unrolled output.
static __device__ __noinline__ float epilogue_outlined(float v, int act, float alpha, int res_mode, float r) {
    return epilogue(v, act, alpha, res_mode, r);
}

// epilogue() with the SiLU (the one activation that needs expf) kept out of
// line: unrolled epilogues then carry one call instead of one expf each.
__device__ __forceinline__ float epilogue_fast(float v, int act, float alpha, int res_mode, float r) {
    if (act == ACNN_ACT_SILU) return epilogue_outlined(v, act, alpha, res_mode, r);
    return epilogue(v, act, alpha, res_mode, r);
}

__device__ __forceinline__ int64_t act_index(int layout, int C, int H, int W, int n, int c,
                                             int y, int x) {
    if (layout == ACNN_NHWC) return (((int64_t)n * H + y) * W + x) * C + c;
    return (((int64_t)n * C + c) * H + y) * W + x;
}

}  // namespace acnn

// ---------------------------------------------------------------- host helpers
// Launch helpers and per-TU launchers, declared here and defined in the .cu
// file that owns each kernel; the ABI layer (abi.cu) validates arguments
// before calling any of them.
namespace acnn {

struct ConvArgs {
    acnn_conv_desc d;
    int oh, ow;
    const void* x;
    const void* w;
    const float* bias;
    const float* alpha;
    const void* residual;
    int res_mode, act;
    void* y;
    int out_layout;  // layout y and residual are written/read in (may differ from d.layout)
    void* ws_part;         // split-K partial-sum workspace (256-byte aligned) or NULL
    size_t ws_part_bytes;  // its size: the planner uses at most this much
    // channel concat folded into the conv: x holds input channels [0, c_split)
    // and x2 channels [c_split, c_in), both NHWC (c_split = 0: x holds all)
    const void* x2 = nullptr;
    int c_split = 0;
    // A second output written by the conv's epilogue (NULL: none), NHWC:
    // y2_up = 0: [n][oh/2][ow/2][c_out], the 2x2/s2 average pool of y (1x1 convs);
    // y2_up = 1: [n][2 oh][2 ow][c_out], the nearest 2x upsample of y
    void* y2 = nullptr;
    int y2_up = 0;
    // NCHW convs on the tensor cores: an NHWC copy of x the caller already has
    // (the staging transpose is then skipped), and an NHWC copy of y to write
    // beside it (NULL: none)
    const void* x_nhwc = nullptr;
    void* y_nhwc = nullptr;
};

// Tile width and K split of the tensor-core conv for a geometry, given the
// bytes available for split-K partial sums (SIZE_MAX: as many as it wants).
struct IgemmPlan {
    int bn;             // output channels per tile: 32, 64, 128 or 256
    int ms;             // 128-pixel row blocks per tile: 1 or 2
    int splits;         // K splits (1 = none)
    int kb_per_split;   // k-blocks per split
    size_t part_bytes;  // fp32 partial-sum workspace the plan needs
    int bk;             // channels per k-block: 64, or 32 when C_in <= 32
};
IgemmPlan igemm_plan(const acnn_conv_desc& d, int oh, int ow, size_t part_budget);
// Force the tile shape of later plans (bn = 0 clears; see acnn_conv2d_force_plan).
void force_plan(int bn, int ms, int splits);

int sm_count();
int* device_status_ptr();         // device address of the status word
int ensure_smem_optin(const void* kernel, size_t bytes);  // per (kernel, device); ACNN_OK or ACNN_ERR_CUDA
long long wait_budget_polls();    // 0 = default (time-bounded)

cudaError_t launch_direct_conv(const ConvArgs& a, cudaStream_t s);
// Direct 3x3 conv for fp16/bf16 inputs of 3, 6 or 7 channels (conv_tiny.cu):
// whether it serves a geometry, and the launch (weights broadcast through
// shared memory, or by warp shuffles when weights_by_shuffle is set).
bool tiny_conv_ok(const acnn_conv_desc& d, int oh, int ow);
cudaError_t launch_tiny_conv(const ConvArgs& a, int weights_by_shuffle, cudaStream_t s);
// The weight-broadcast form of the tiny-C_in kernel by default (shared-memory
// broadcast: measured faster than the shuffle form on the frame input).
constexpr int kTinyWeightsByShuffle = 0;
// tensor-core path; returns ACNN_OK or an ACNN_ERR_* status
int launch_igemm_conv(const ConvArgs& a, cudaStream_t s);

cudaError_t launch_pool2d(int kind, int n, int h, int w, int c, int k, int stride, int pad,
                          int layout, int dtype, const void* x, void* y, cudaStream_t s);
cudaError_t launch_resize2d(int mode, int n, int c, int h, int w, int oh, int ow, int layout,
                            int in_dtype, int out_dtype, const void* x, void* y, cudaStream_t s);
cudaError_t launch_concat(int n, int h, int w, int ca, int cb, int layout, int dtype,
                          const void* a, const void* b, void* y, cudaStream_t s);
cudaError_t launch_deconv2d(const acnn_conv_desc& d, int oh, int ow, const void* x,
                            const float* w, const float* bias, const float* alpha, int act,
                            int out_dtype, void* y, cudaStream_t s);
cudaError_t launch_prep_quarter(int h, int w, const uint8_t* rgba0, const uint8_t* rgba1,
                                float t, int out_dtype, void* y, cudaStream_t s);
// flow-out stage of the frame stack (flow_out.cu)
cudaError_t launch_flow_out(int h, int w, const void* tmp8, int tmp8_dtype, const uint8_t* rgba0,
                            const uint8_t* rgba1, const float* res, uint8_t* out, cudaStream_t s);
// t-factored frame stack (flow_out.cu)
cudaError_t launch_refine_prep(int h, int w, const void* tmp8, int tmp8_dtype,
                               const uint8_t* rgba0, const uint8_t* rgba1, int out_dtype,
                               void* out, cudaStream_t s);
cudaError_t launch_refine_out(int c, int hh, int hw, const void* x, int dtype, const float* w,
                              const float* bias, float* y, cudaStream_t s);
cudaError_t launch_film(int c, int n, int dtype, const void* x, float t, const float* w0,
                        const float* b0, int hn, const float* w2, const float* b2, void* y,
                        cudaStream_t s);
// im2col pack of x into a [n*oh*ow, kp] matrix and of w into [c_out, kp] (2-byte types)
cudaError_t launch_im2col_pack(const acnn_conv_desc& d, int oh, int ow, int kp, const void* x,
                               void* a, const void* w, void* wp, cudaStream_t s);
// the packed weight operand [c_out, kp] alone (kp >= kh*kw*c_in, zero padded)
cudaError_t launch_weight_pack(const acnn_conv_desc& d, int kp, const void* w, void* wp,
                               cudaStream_t s);
// The 4x4/s2/p1 transposed conv on the tensor cores (memops.cu): its weights,
// bias and PReLU alpha regrouped for a 3x3/s1/p1 conv of 4 co (rounded up to
// co4) output channels, and the pixel shuffle of that conv's NHWC output into
// the deconv's output (fp16/bf16)
cudaError_t launch_deconv_gemm_weights(int dtype, const float* w, const float* bias,
                                       const float* alpha, void* wg, float* bg, float* ag, int ci,
                                       int co, int co4, cudaStream_t s);
cudaError_t launch_deconv_shuffle(int dtype, const void* ys, void* y, int layout, int n, int h,
                                  int w, int co, int co4, cudaStream_t s);
// NCHW -> NHWC activation transpose and OIHW -> OHWI weight transpose (2-byte types)
cudaError_t launch_nchw_to_nhwc(int n, int c, int hw, int elem_bytes, const void* x, void* y,
                                cudaStream_t s);

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialization, so its CTAs may start (and run
// their setup) while the previous kernel on the stream is still finishing;
// each kernel executes griddep_wait() before its first access to global
// memory, which returns once the previous kernel has completed and its writes
// are visible (immediately when there is no such kernel).
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel on the stream launch once every CTA of this grid has
// executed it (or exited).
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Resident blocks of `kernel` per SM at this block size (cached per kernel).
int occupancy_blocks(const void* kernel, int threads, size_t smem);

// Grid for a grid-stride kernel: enough blocks for the work, at most one wave
// of the blocks that can be resident at once (occupancy from the kernel's
// registers and shared memory), so no block waits for a second wave.
template <typename Kern>
inline int grid_occ(Kern kernel, long long work_items, int threads, size_t smem = 0) {
    long long want = (work_items + threads - 1) / threads;
    long long cap = (long long)sm_count() *
                    occupancy_blocks(reinterpret_cast<const void*>(kernel), threads, smem);
    if (want > cap) want = cap;
    return want < 1 ? 1 : (int)want;
}

inline int grid_for(long long work_items, int threads, int per_sm = 8) {
    long long want = (work_items + threads - 1) / threads;
    long long cap = (long long)sm_count() * per_sm;
    if (want > cap) want = cap;
    return want < 1 ? 1 : (int)want;
}

}  // namespace acnn
