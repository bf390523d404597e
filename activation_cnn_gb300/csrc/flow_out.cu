// flow_out.cu -- the flow-out stage of the frame stack ("@framecast/rt 1.0.0
// -- package/rt.js", wgslFlowOut, with wgslPrepFull's full-resolution planes
// read straight from the RGBA8 frames): from the 5-plane map the deconv
// leaves at 1/8 resolution (flow of frame 0, flow of frame 1, mask), per
// output pixel:
//   * the x8 bilinear upsample (align_corners=false) of the five planes, the
//     flows scaled by 8 and the mask through a sigmoid;
//   * a backward warp of each frame by its flow: bilinear over pixel
//     coordinates with clamped taps (grid_sample, border, align_corners=true);
//   * the blend w0 * m + w1 * (1 - m) and the RGBA8 pack, each channel
//     truncated from clamp(v, 0, 1) * 255, alpha 255.
// The page computes this in binary32 and truncates to bytes, so a float
// decides each output byte.  Every step is written with a round-to-nearest
// intrinsic (no fused multiply-adds) in one fixed order, and exp is computed
// by a named method (Cody-Waite reduction, degree-7 Taylor polynomial) rather
// than the library's, so that the result is a function of the inputs alone.
#include "common.cuh"

namespace acnn {

namespace {

// e^x: x = n ln2 + r with n = rint(x log2 e) and ln 2 split into a 15-bit head
// and a tail (Cody and Waite's reduction), e^r by the Taylor polynomial of
// degree 7 in Horner form (each step one correctly rounded fma), times 2^n.
__device__ __forceinline__ float flow_exp(float x) {
    const float log2e = 1.44269504088896341f;
    const float ln2_hi = 0.693145751953125f;
    const float ln2_lo = 1.42860682030941723e-6f;
    x = fminf(fmaxf(x, -87.0f), 88.0f);
    const float n = rintf(__fmul_rn(x, log2e));
    float r = __fsub_rn(x, __fmul_rn(n, ln2_hi));
    r = __fsub_rn(r, __fmul_rn(n, ln2_lo));
    float q = 1.0f / 5040.0f;
    q = __fmaf_rn(q, r, 1.0f / 720.0f);
    q = __fmaf_rn(q, r, 1.0f / 120.0f);
    q = __fmaf_rn(q, r, 1.0f / 24.0f);
    q = __fmaf_rn(q, r, 1.0f / 6.0f);
    q = __fmaf_rn(q, r, 0.5f);
    q = __fmaf_rn(q, r, 1.0f);
    q = __fmaf_rn(q, r, 1.0f);
    return ldexpf(q, (int)n);
}

// mix(a, b, f) = a * (1 - f) + b * f, three roundings
__device__ __forceinline__ float mixf(float a, float b, float f) {
    return __fadd_rn(__fmul_rn(a, __fsub_rn(1.0f, f)), __fmul_rn(b, f));
}

template <typename T> struct FlowIn {
    const T* t;
    int TH, TW;
    __device__ __forceinline__ float at(int c, int y, int x) const {
        return to_f32(t[((size_t)c * TH + y) * TW + x]);
    }
};

// bilinear of plane c at (sx, sy), taps clamped into the plane
template <typename T>
__device__ __forceinline__ float up(const FlowIn<T>& in, int c, float sx, float sy) {
    const float fx0 = floorf(sx), fy0 = floorf(sy);
    const float fx = __fsub_rn(sx, fx0), fy = __fsub_rn(sy, fy0);
    const int x0 = (int)fx0, y0 = (int)fy0;
    const int xa = min(max(x0, 0), in.TW - 1), xb = min(max(x0 + 1, 0), in.TW - 1);
    const int ya = min(max(y0, 0), in.TH - 1), yb = min(max(y0 + 1, 0), in.TH - 1);
    const float top = mixf(in.at(c, ya, xa), in.at(c, ya, xb), fx);
    const float bot = mixf(in.at(c, yb, xa), in.at(c, yb, xb), fx);
    return mixf(top, bot, fy);
}

// B, G, R of an RGBA8 frame at pixel-space (px, py), bilinear, clamped taps
__device__ __forceinline__ void warp_bgr(const uint32_t* __restrict__ f, int H, int W, float px,
                                         float py, float (&bgr)[3]) {
    const float fx0 = floorf(px), fy0 = floorf(py);
    const float fx = __fsub_rn(px, fx0), fy = __fsub_rn(py, fy0);
    // clamp in float first: a large flow can put the tap beyond the int range
    const int x0 = (int)fminf(fmaxf(fx0, -1.0f), (float)W);
    const int y0 = (int)fminf(fmaxf(fy0, -1.0f), (float)H);
    const int xa = min(max(x0, 0), W - 1), xb = min(max(x0 + 1, 0), W - 1);
    const int ya = min(max(y0, 0), H - 1), yb = min(max(y0 + 1, 0), H - 1);
    const uint32_t p00 = __ldg(f + (size_t)ya * W + xa), p01 = __ldg(f + (size_t)ya * W + xb);
    const uint32_t p10 = __ldg(f + (size_t)yb * W + xa), p11 = __ldg(f + (size_t)yb * W + xb);
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const int sh = 8 * (2 - k);  // B, G, R = bytes 2, 1, 0
        auto ch = [&](uint32_t p) { return __fdiv_rn(__uint2float_rn((p >> sh) & 255u), 255.0f); };
        bgr[k] = mixf(mixf(ch(p00), ch(p01), fx), mixf(ch(p10), ch(p11), fx), fy);
    }
}

template <typename T>
__global__ void __launch_bounds__(256) flow_out_kernel(const T* __restrict__ tmp8,
                                                       const uint32_t* __restrict__ f0,
                                                       const uint32_t* __restrict__ f1,
                                                       uint32_t* __restrict__ out, int H, int W) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const int x = blockIdx.x * blockDim.x + threadIdx.x;
    const int y = blockIdx.y * blockDim.y + threadIdx.y;
    if (x >= W || y >= H) return;
    const FlowIn<T> in{tmp8, H / 8, W / 8};
    const float sx = __fsub_rn(__fmul_rn(__fadd_rn((float)x, 0.5f), 0.125f), 0.5f);
    const float sy = __fsub_rn(__fmul_rn(__fadd_rn((float)y, 0.5f), 0.125f), 0.5f);
    const float u0 = __fmul_rn(up(in, 0, sx, sy), 8.0f), v0 = __fmul_rn(up(in, 1, sx, sy), 8.0f);
    const float u1 = __fmul_rn(up(in, 2, sx, sy), 8.0f), v1 = __fmul_rn(up(in, 3, sx, sy), 8.0f);
    const float m = __fdiv_rn(1.0f, __fadd_rn(1.0f, flow_exp(-up(in, 4, sx, sy))));
    float w0[3], w1[3];
    warp_bgr(f0, H, W, __fadd_rn((float)x, u0), __fadd_rn((float)y, v0), w0);
    warp_bgr(f1, H, W, __fadd_rn((float)x, u1), __fadd_rn((float)y, v1), w1);
    const float om = __fsub_rn(1.0f, m);
    uint32_t px = 255u << 24;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        float c = __fadd_rn(__fmul_rn(w0[k], m), __fmul_rn(w1[k], om));
        c = fminf(fmaxf(c, 0.0f), 1.0f);
        px |= __float2uint_rz(__fmul_rn(c, 255.0f)) << (8 * (2 - k));
    }
    out[(size_t)y * W + x] = px;
}

template <typename T>
cudaError_t flow_typed(int h, int w, const void* tmp8, const uint8_t* rgba0, const uint8_t* rgba1,
                       uint8_t* out, cudaStream_t s) {
    const dim3 block(32, 8), grid((w + 31) / 32, (h + 7) / 8);
    launch_pdl(flow_out_kernel<T>, grid, block, 0, s, static_cast<const T*>(tmp8),
               reinterpret_cast<const uint32_t*>(rgba0), reinterpret_cast<const uint32_t*>(rgba1),
               reinterpret_cast<uint32_t*>(out), h, w);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_flow_out(int h, int w, const void* tmp8, int tmp8_dtype, const uint8_t* rgba0,
                            const uint8_t* rgba1, uint8_t* out, cudaStream_t s) {
    switch (tmp8_dtype) {
    case ACNN_F32: return flow_typed<float>(h, w, tmp8, rgba0, rgba1, out, s);
    case ACNN_F16: return flow_typed<__half>(h, w, tmp8, rgba0, rgba1, out, s);
    default: return flow_typed<__nv_bfloat16>(h, w, tmp8, rgba0, rgba1, out, s);
    }
}

}  // namespace acnn
