// flow_out.cu -- the flow-out stage of the frame stack (and the t-factored
// stack's FiLM, refine prep and refine out, which share its arithmetic) ("@framecast/rt 1.0.0
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
// intrinsic (no fused multiply-adds) in the page's order; the mask's exp is
// CUDA's expf (the page's WGSL exp is a binary32 function of unstated
// rounding), so a byte can differ by one from another faithful binary32
// evaluation only where clamp(v, 0, 1) * 255 lies within a few ulp of an
// integer.
#include "common.cuh"

namespace acnn {

namespace {

// e^x for the mask's sigmoid: the CUDA math library's binary32 exp.
__device__ __forceinline__ float flow_exp(float x) { return expf(x); }

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

// byte / 255 for every byte value, correctly rounded (one division each),
// filled by the block before use: a shared-memory read per tap channel in
// place of a division
__device__ __forceinline__ void fill_unorm_lut(float* lut) {
    for (int i = threadIdx.y * blockDim.x + threadIdx.x; i < 256; i += blockDim.x * blockDim.y)
        lut[i] = __fdiv_rn(__uint2float_rn((unsigned)i), 255.0f);
    __syncthreads();
}

// B, G, R of an RGBA8 frame at pixel-space (px, py), bilinear, clamped taps
__device__ __forceinline__ void warp_bgr(const uint32_t* __restrict__ f, const float* lut, int H,
                                         int W, float px, float py, float (&bgr)[3]) {
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
        auto ch = [&](uint32_t p) { return lut[(p >> sh) & 255u]; };
        bgr[k] = mixf(mixf(ch(p00), ch(p01), fx), mixf(ch(p10), ch(p11), fx), fy);
    }
}

template <typename T>
__global__ void __launch_bounds__(256) flow_out_kernel(const T* __restrict__ tmp8,
                                                       const uint32_t* __restrict__ f0,
                                                       const uint32_t* __restrict__ f1,
                                                       const float* __restrict__ res,
                                                       uint32_t* __restrict__ out, int H, int W) {
    __shared__ float lut[256];
    fill_unorm_lut(lut);
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
    warp_bgr(f0, lut, H, W, __fadd_rn((float)x, u0), __fadd_rn((float)y, v0), w0);
    warp_bgr(f1, lut, H, W, __fadd_rn((float)x, u1), __fadd_rn((float)y, v1), w1);
    const float om = __fsub_rn(1.0f, m);
    // refine residual (t-factored stack): x4 bilinear upsample, added before the clamp
    float rv[3] = {0.0f, 0.0f, 0.0f};
    if (res) {
        const FlowIn<float> rin{res, H / 4, W / 4};
        const float rx = __fsub_rn(__fmul_rn(__fadd_rn((float)x, 0.5f), 0.25f), 0.5f);
        const float ry = __fsub_rn(__fmul_rn(__fadd_rn((float)y, 0.5f), 0.25f), 0.5f);
#pragma unroll
        for (int k = 0; k < 3; ++k) rv[k] = up(rin, k, rx, ry);
    }
    uint32_t px = 255u << 24;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        float c = __fadd_rn(__fmul_rn(w0[k], m), __fmul_rn(w1[k], om));
        if (res) c = __fadd_rn(c, rv[k]);
        c = fminf(fmaxf(c, 0.0f), 1.0f);
        px |= __float2uint_rz(__fmul_rn(c, 255.0f)) << (8 * (2 - k));
    }
    out[(size_t)y * W + x] = px;
}

template <typename T>
cudaError_t flow_typed(int h, int w, const void* tmp8, const uint8_t* rgba0, const uint8_t* rgba1,
                       const float* res, uint8_t* out, cudaStream_t s) {
    const dim3 block(32, 8), grid((w + 31) / 32, (h + 7) / 8);
    launch_pdl(flow_out_kernel<T>, grid, block, 0, s, static_cast<const T*>(tmp8),
               reinterpret_cast<const uint32_t*>(rgba0), reinterpret_cast<const uint32_t*>(rgba1),
               res, reinterpret_cast<uint32_t*>(out), h, w);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- t-factored stack
// Refine prep (rt.js wgslRefinePrep): per quarter-resolution pixel, the mean
// over the centre 2x2 of its 4x4 block of the warped frames (B, G, R each),
// the sigmoid mask and the x8 flows scaled by 0.25 / 20; 11 planes.  Same
// upsample / warp / exp steps as the flow-out stage; the values are stored
// (not truncated), so no byte decision rides on them.
template <typename T, typename To>
__global__ void __launch_bounds__(256) refine_prep_kernel(const T* __restrict__ tmp8,
                                                          const uint32_t* __restrict__ f0,
                                                          const uint32_t* __restrict__ f1,
                                                          To* __restrict__ out, int H, int W) {
    __shared__ float lut[256];
    fill_unorm_lut(lut);
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const int QH = H / 4, QW = W / 4;
    const int hx = blockIdx.x * blockDim.x + threadIdx.x;
    const int hy = blockIdx.y * blockDim.y + threadIdx.y;
    if (hx >= QW || hy >= QH) return;
    const FlowIn<T> in{tmp8, H / 8, W / 8};
    float acc[11];
#pragma unroll
    for (int k = 0; k < 11; ++k) acc[k] = 0.0f;
#pragma unroll
    for (int sy = 1; sy <= 2; ++sy)
#pragma unroll
        for (int sxp = 1; sxp <= 2; ++sxp) {
            const int X = 4 * hx + sxp, Y = 4 * hy + sy;
            const float gx = __fsub_rn(__fmul_rn(__fadd_rn((float)X, 0.5f), 0.125f), 0.5f);
            const float gy = __fsub_rn(__fmul_rn(__fadd_rn((float)Y, 0.5f), 0.125f), 0.5f);
            const float u0 = __fmul_rn(up(in, 0, gx, gy), 8.0f), v0 = __fmul_rn(up(in, 1, gx, gy), 8.0f);
            const float u1 = __fmul_rn(up(in, 2, gx, gy), 8.0f), v1 = __fmul_rn(up(in, 3, gx, gy), 8.0f);
            acc[6] += __fdiv_rn(1.0f, __fadd_rn(1.0f, flow_exp(-up(in, 4, gx, gy))));
            float w0[3], w1[3];
            warp_bgr(f0, lut, H, W, __fadd_rn((float)X, u0), __fadd_rn((float)Y, v0), w0);
            warp_bgr(f1, lut, H, W, __fadd_rn((float)X, u1), __fadd_rn((float)Y, v1), w1);
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                acc[k] += w0[k];
                acc[3 + k] += w1[k];
            }
            acc[7] += u0;
            acc[8] += v0;
            acc[9] += u1;
            acc[10] += v1;
        }
    const size_t P = (size_t)QH * QW, o = (size_t)hy * QW + hx;
#pragma unroll
    for (int k = 0; k < 7; ++k) out[k * P + o] = from_f32<To>(acc[k] * 0.25f);
#pragma unroll
    for (int k = 7; k < 11; ++k) out[k * P + o] = from_f32<To>(acc[k] * (0.25f * (0.25f / 20.0f)));
}

// Refine out (rt.js wgslRefineOut): conv3x3 C -> 3 with replicate (clamped)
// padding, fp32 weights [3][C][3][3], then 2 sigmoid(acc) - 1, fp32 output.
// One thread per output pixel; the weights of a block's channel chunk sit in
// shared memory.
template <typename T>
__global__ void __launch_bounds__(256) refine_out_kernel(const T* __restrict__ x,
                                                         const float* __restrict__ w,
                                                         const float* __restrict__ bias,
                                                         float* __restrict__ y, int C, int HH,
                                                         int HW) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    constexpr int kChunk = 64;  // input channels per shared-memory weight chunk
    __shared__ float sw[3][kChunk][9];
    const int ox = blockIdx.x * blockDim.x + threadIdx.x;
    const int oy = blockIdx.y * blockDim.y + threadIdx.y;
    const int tid = threadIdx.y * blockDim.x + threadIdx.x;
    float acc[3] = {bias[0], bias[1], bias[2]};
    const bool in = ox < HW && oy < HH;
    int ys[3], xs[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        ys[k] = min(max(oy + k - 1, 0), HH - 1);
        xs[k] = min(max(ox + k - 1, 0), HW - 1);
    }
    for (int c0 = 0; c0 < C; c0 += kChunk) {
        const int nc = min(kChunk, C - c0);
        __syncthreads();
        for (int i = tid; i < 3 * nc * 9; i += blockDim.x * blockDim.y) {
            const int co = i / (nc * 9), r = i - co * nc * 9, ci = r / 9, t = r - ci * 9;
            sw[co][ci][t] = w[((size_t)co * C + c0 + ci) * 9 + t];
        }
        __syncthreads();
        if (in) {
            for (int ci = 0; ci < nc; ++ci) {
                const T* pl = x + (size_t)(c0 + ci) * HH * HW;
#pragma unroll
                for (int ky = 0; ky < 3; ++ky)
#pragma unroll
                    for (int kx = 0; kx < 3; ++kx) {
                        const float v = to_f32(pl[(size_t)ys[ky] * HW + xs[kx]]);
#pragma unroll
                        for (int co = 0; co < 3; ++co) acc[co] = fmaf(v, sw[co][ci][ky * 3 + kx], acc[co]);
                    }
            }
        }
    }
    if (in) {
#pragma unroll
        for (int co = 0; co < 3; ++co)
            y[((size_t)co * HH + oy) * HW + ox] = 2.0f / (1.0f + expf(-acc[co])) - 1.0f;
    }
}

// FiLM (rt.js wgslFilm with filmParams): per channel c, the timestep MLP's two
// outputs s[c] = b2[c] + W2[c] relu(w0 t + b0) and s[C + c], then
// x' = x (1 + s[c]) + s[C + c] over the channel's plane.  Every block of
// channel c evaluates the two dot products itself (2 x hn multiply-adds, one
// warp), which costs less than a second launch.
template <typename T>
__global__ void __launch_bounds__(256) film_kernel(const T* __restrict__ x, float t,
                                                   const float* __restrict__ w0,
                                                   const float* __restrict__ b0, int hn,
                                                   const float* __restrict__ w2,
                                                   const float* __restrict__ b2,
                                                   T* __restrict__ y, int C, int N) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    __shared__ float ss[2];
    const int c = blockIdx.y;
    if (threadIdx.x < 32) {
        float a0 = 0.0f, a1 = 0.0f;
        for (int j = threadIdx.x; j < hn; j += 32) {
            const float hj = fmaxf(fmaf(w0[j], t, b0[j]), 0.0f);
            a0 = fmaf(w2[(size_t)c * hn + j], hj, a0);
            a1 = fmaf(w2[(size_t)(C + c) * hn + j], hj, a1);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            a0 += __shfl_xor_sync(0xffffffffu, a0, o);
            a1 += __shfl_xor_sync(0xffffffffu, a1, o);
        }
        if (threadIdx.x == 0) {
            ss[0] = 1.0f + (b2[c] + a0);
            ss[1] = b2[C + c] + a1;
        }
    }
    __syncthreads();
    const float scale = ss[0], shift = ss[1];
    const T* xp = x + (size_t)c * N;
    T* yp = y + (size_t)c * N;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < N; i += gridDim.x * blockDim.x)
        yp[i] = from_f32<T>(fmaf(to_f32(xp[i]), scale, shift));
}

}  // namespace

cudaError_t launch_flow_out(int h, int w, const void* tmp8, int tmp8_dtype, const uint8_t* rgba0,
                            const uint8_t* rgba1, const float* res, uint8_t* out, cudaStream_t s) {
    switch (tmp8_dtype) {
    case ACNN_F32: return flow_typed<float>(h, w, tmp8, rgba0, rgba1, res, out, s);
    case ACNN_F16: return flow_typed<__half>(h, w, tmp8, rgba0, rgba1, res, out, s);
    default: return flow_typed<__nv_bfloat16>(h, w, tmp8, rgba0, rgba1, res, out, s);
    }
}

namespace {
template <typename T, typename To>
cudaError_t refine_prep_typed(int h, int w, const void* tmp8, const uint8_t* rgba0,
                              const uint8_t* rgba1, void* out, cudaStream_t s) {
    const dim3 block(32, 8), grid((w / 4 + 31) / 32, (h / 4 + 7) / 8);
    launch_pdl(refine_prep_kernel<T, To>, grid, block, 0, s, static_cast<const T*>(tmp8),
               reinterpret_cast<const uint32_t*>(rgba0), reinterpret_cast<const uint32_t*>(rgba1),
               static_cast<To*>(out), h, w);
    return cudaGetLastError();
}
template <typename T>
cudaError_t refine_prep_in(int h, int w, const void* tmp8, const uint8_t* rgba0,
                           const uint8_t* rgba1, int out_dtype, void* out, cudaStream_t s) {
    switch (out_dtype) {
    case ACNN_F32: return refine_prep_typed<T, float>(h, w, tmp8, rgba0, rgba1, out, s);
    case ACNN_F16: return refine_prep_typed<T, __half>(h, w, tmp8, rgba0, rgba1, out, s);
    default: return refine_prep_typed<T, __nv_bfloat16>(h, w, tmp8, rgba0, rgba1, out, s);
    }
}
}  // namespace

cudaError_t launch_refine_prep(int h, int w, const void* tmp8, int tmp8_dtype,
                               const uint8_t* rgba0, const uint8_t* rgba1, int out_dtype,
                               void* out, cudaStream_t s) {
    switch (tmp8_dtype) {
    case ACNN_F32: return refine_prep_in<float>(h, w, tmp8, rgba0, rgba1, out_dtype, out, s);
    case ACNN_F16: return refine_prep_in<__half>(h, w, tmp8, rgba0, rgba1, out_dtype, out, s);
    default: return refine_prep_in<__nv_bfloat16>(h, w, tmp8, rgba0, rgba1, out_dtype, out, s);
    }
}

cudaError_t launch_refine_out(int c, int hh, int hw, const void* x, int dtype, const float* w,
                              const float* bias, float* y, cudaStream_t s) {
    const dim3 block(32, 8), grid((hw + 31) / 32, (hh + 7) / 8);
    switch (dtype) {
    case ACNN_F32:
        launch_pdl(refine_out_kernel<float>, grid, block, 0, s, static_cast<const float*>(x), w,
                   bias, y, c, hh, hw);
        break;
    case ACNN_F16:
        launch_pdl(refine_out_kernel<__half>, grid, block, 0, s, static_cast<const __half*>(x), w,
                   bias, y, c, hh, hw);
        break;
    default:
        launch_pdl(refine_out_kernel<__nv_bfloat16>, grid, block, 0, s,
                   static_cast<const __nv_bfloat16*>(x), w, bias, y, c, hh, hw);
        break;
    }
    return cudaGetLastError();
}

cudaError_t launch_film(int c, int n, int dtype, const void* x, float t, const float* w0,
                        const float* b0, int hn, const float* w2, const float* b2, void* y,
                        cudaStream_t s) {
    // about eight elements per thread: each block also evaluates its channel's
    // two MLP outputs, so fewer, longer blocks per channel
    const int bx = (n + 2047) / 2048 < 64 ? (n + 2047) / 2048 : 64;
    const dim3 grid(bx, c);
    switch (dtype) {
    case ACNN_F32:
        launch_pdl(film_kernel<float>, grid, dim3(256), 0, s, static_cast<const float*>(x), t, w0,
                   b0, hn, w2, b2, static_cast<float*>(y), c, n);
        break;
    case ACNN_F16:
        launch_pdl(film_kernel<__half>, grid, dim3(256), 0, s, static_cast<const __half*>(x), t,
                   w0, b0, hn, w2, b2, static_cast<__half*>(y), c, n);
        break;
    default:
        launch_pdl(film_kernel<__nv_bfloat16>, grid, dim3(256), 0, s,
                   static_cast<const __nv_bfloat16*>(x), t, w0, b0, hn, w2, b2,
                   static_cast<__nv_bfloat16*>(y), c, n);
        break;
    }
    return cudaGetLastError();
}

}  // namespace acnn
