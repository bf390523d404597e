// conv_direct.cu -- direct conv2d_fused on the FFMA pipes.
//
// Serves what the tensor-core path does not: fp32 storage (the fp32 stem),
// inputs with few channels (the 3-channel RGB stem, the 7-plane frame input),
// non-square kernels and channel counts TMA cannot address.
//
// Prior art: rt.js wgslConv / wgslConvRB stage a slab of input channels and
// their weights through workgroup memory and give each thread several output
// channels (and, in the register-blocked form, a 2x2 pixel patch).  Here a CTA
// of 256 threads computes a 16x16 output tile for 32 output channels; each
// thread holds 4 pixels (one column, rows 4 apart) x 8 channels = 32 fp32
// accumulators.  Per staged input channel and tap a thread reads 4 input
// values and 8 weights (two 16-byte broadcast loads: every lane of a warp
// reads the same 8 weights) and issues 32 FMAs.
//
// Accumulation per output: fp32 FMAs over the staged channel chunks, taps
// (ky, kx) within each channel; the fp32 bias is added to that sum in the
// epilogue, as a GEMM epilogue adds it; one rounding at the store.
#include "common.cuh"

namespace acnn {

namespace {

constexpr int kTH = 16, kTW = 16, kCOB = 32, kThreads = 256;
constexpr int kPxPerThread = 4, kCoPerThread = 8;

// One tap (ky, kx) of one staged input channel: 4 pixels x 8 output channels.
__device__ __forceinline__ void tap_fma(float (&acc)[kPxPerThread][kCoPerThread],
                                        const float* sin_c, const float* s_wt, int cg, int ty0,
                                        int tx, int S, int ky, int kx, int ITW) {
    const float4* wp = reinterpret_cast<const float4*>(s_wt + cg * kCoPerThread);
    const float4 w0 = wp[0], w1 = wp[1];
    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int j = 0; j < kPxPerThread; ++j) {
        const float xv = sin_c[((ty0 + 4 * j) * S + ky) * ITW + tx * S + kx];
#pragma unroll
        for (int c = 0; c < kCoPerThread; ++c) acc[j][c] = fmaf(xv, wv[c], acc[j][c]);
    }
}

template <typename T, int KH_, int KW_>
__global__ void __launch_bounds__(kThreads) direct_conv_kernel(
    const T* __restrict__ x, const T* __restrict__ w, const float* __restrict__ bias,
    const float* __restrict__ alpha, const T* __restrict__ res, T* __restrict__ y, int layout,
    int out_layout, int N, int H, int W, int C_in, int C_out, int kh_rt, int kw_rt, int S, int P,
    int OH, int OW, int act, int res_mode, int cic) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const int KH = KH_ > 0 ? KH_ : kh_rt;
    const int KW = KW_ > 0 ? KW_ : kw_rt;
    const int KK = KH * KW;
    const int ITH = (kTH - 1) * S + KH, ITW = (kTW - 1) * S + KW;

    extern __shared__ __align__(16) float smem[];
    float* s_in = smem;                                  // [cic][ITH][ITW]
    float* s_w = smem + ((cic * ITH * ITW + 3) & ~3);    // [cic][KK][kCOB], 16-byte aligned

    const int tiles_x = (OW + kTW - 1) / kTW;
    const int oy0 = (blockIdx.x / tiles_x) * kTH, ox0 = (blockIdx.x % tiles_x) * kTW;
    const int co0 = blockIdx.y * kCOB;
    const int n = blockIdx.z;
    const int tid = threadIdx.x;
    const int cg = tid >> 6, pg = tid & 63;
    const int tx = pg & 15, ty0 = pg >> 4;

    float acc[kPxPerThread][kCoPerThread];
#pragma unroll
    for (int j = 0; j < kPxPerThread; ++j)
#pragma unroll
        for (int c = 0; c < kCoPerThread; ++c) acc[j][c] = 0.0f;

    const int gy0 = oy0 * S - P, gx0 = ox0 * S - P;
    for (int ci0 = 0; ci0 < C_in; ci0 += cic) {
        const int nci = min(cic, C_in - ci0);
        __syncthreads();
        // stage the input halo tile of channels [ci0, ci0 + nci); taps outside
        // the image are zero (rtdetr_gpu.rs IM2COL_SRC)
        const int tile_elems = nci * ITH * ITW;
        // eight independent loads per thread in flight before any is stored
        constexpr int kBatch = 8;
        for (int base = tid; base < tile_elems; base += kThreads * kBatch) {
            float v[kBatch];
            int dst[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int idx = base + u * kThreads;
                v[u] = 0.0f;
                dst[u] = -1;
                if (idx < tile_elems) {
                    int ci, iy, ix;
                    if (layout == ACNN_NHWC) {
                        ci = idx % nci;
                        const int r = idx / nci;
                        ix = r % ITW;
                        iy = r / ITW;
                    } else {
                        ix = idx % ITW;
                        const int r = idx / ITW;
                        iy = r % ITH;
                        ci = r / ITH;
                    }
                    dst[u] = (ci * ITH + iy) * ITW + ix;
                    const int gy = gy0 + iy, gx = gx0 + ix;
                    if (gy >= 0 && gy < H && gx >= 0 && gx < W)
                        v[u] = to_f32(x[act_index(layout, C_in, H, W, n, ci0 + ci, gy, gx)]);
                }
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u)
                if (dst[u] >= 0) s_in[dst[u]] = v[u];
        }
        // stage the weights of those channels for kCOB output channels
        const int w_elems = nci * KK * kCOB;
        for (int idx = tid; idx < w_elems; idx += kThreads) {
            const int co = idx % kCOB;
            const int r = idx / kCOB;
            const int tap = r % KK, ci = r / KK;
            float v = 0.0f;
            if (co0 + co < C_out) {
                const int ky = tap / KW, kx = tap % KW;
                long long wi = layout == ACNN_NHWC
                                   ? (((long long)(co0 + co) * KH + ky) * KW + kx) * C_in + ci0 + ci
                                   : (((long long)(co0 + co) * C_in + ci0 + ci) * KH + ky) * KW + kx;
                v = to_f32(w[wi]);
            }
            s_w[idx] = v;
        }
        __syncthreads();

        for (int ci = 0; ci < nci; ++ci) {
            const float* sin_c = s_in + ci * ITH * ITW;
            if constexpr (KH_ > 0 && KW_ > 0) {
#pragma unroll
                for (int ky = 0; ky < KH_; ++ky)
#pragma unroll
                    for (int kx = 0; kx < KW_; ++kx)
                        tap_fma(acc, sin_c, s_w + (ci * KK + ky * KW_ + kx) * kCOB, cg, ty0, tx, S,
                                ky, kx, ITW);
            } else {
#pragma unroll 1
                for (int ky = 0; ky < KH; ++ky)
#pragma unroll 1
                    for (int kx = 0; kx < KW; ++kx)
                        tap_fma(acc, sin_c, s_w + (ci * KK + ky * KW + kx) * kCOB, cg, ty0, tx, S,
                                ky, kx, ITW);
            }
        }
    }

    // fused epilogue: bias -> act / residual -> storage type
    const int cb = co0 + cg * kCoPerThread;  // first of this thread's 8 output channels
    float bv[kCoPerThread], av[kCoPerThread];
#pragma unroll
    for (int c = 0; c < kCoPerThread; ++c) {
        const bool in = cb + c < C_out;
        bv[c] = (bias && in) ? bias[cb + c] : 0.0f;
        av[c] = (act == ACNN_ACT_PRELU && in) ? alpha[cb + c] : 0.0f;
    }
    // NHWC with 8 | C_out: the 8 channels are one aligned vector in memory
    const bool vec = out_layout == ACNN_NHWC && (C_out % kCoPerThread) == 0 && cb < C_out;
#pragma unroll
    for (int j = 0; j < kPxPerThread; ++j) {
        const int oy = oy0 + ty0 + 4 * j, ox = ox0 + tx;
        if (oy >= OH || ox >= OW) continue;
        if (vec) {
            // 16-byte vectors (the only alignment the ABI guarantees): 1 for 2-byte
            // types, 2 for fp32
            constexpr int V = 16 / sizeof(T);
            const long long oi = (((long long)n * OH + oy) * OW + ox) * C_out + cb;
#pragma unroll
            for (int h = 0; h < kCoPerThread; h += V) {
                Vec<T, V> rv, ov;
                if (res_mode != ACNN_RES_NONE) rv = *reinterpret_cast<const Vec<T, V>*>(res + oi + h);
#pragma unroll
                for (int c = 0; c < V; ++c) {
                    const float r = res_mode != ACNN_RES_NONE ? to_f32(rv.v[c]) : 0.0f;
                    ov.v[c] = from_f32<T>(
                        epilogue_fast(bv[h + c] + acc[j][h + c], act, av[h + c], res_mode, r));
                }
                *reinterpret_cast<Vec<T, V>*>(y + oi + h) = ov;
            }
            continue;
        }
#pragma unroll
        for (int c = 0; c < kCoPerThread; ++c) {
            const int co = cb + c;
            if (co >= C_out) continue;
            const long long oi = act_index(out_layout, C_out, OH, OW, n, co, oy, ox);
            const float r = res_mode != ACNN_RES_NONE ? to_f32(res[oi]) : 0.0f;
            y[oi] = from_f32<T>(epilogue_fast(bv[c] + acc[j][c], act, av[c], res_mode, r));
        }
    }
}

template <typename T, int KH_, int KW_>
cudaError_t launch_typed(const ConvArgs& a, cudaStream_t s) {
    const acnn_conv_desc& d = a.d;
    const int ITH = (kTH - 1) * d.stride + d.kh, ITW = (kTW - 1) * d.stride + d.kw;
    auto smem_for = [&](int c) {
        return (size_t)(((c * ITH * ITW + 3) & ~3) + c * d.kh * d.kw * kCOB) * sizeof(float);
    };
    if (smem_for(1) > 96 * 1024) return cudaErrorInvalidConfiguration;
    // stage as many input channels as fit in ~40 KB, so several CTAs share an SM
    int cic = d.c_in;
    while (cic > 1 && smem_for(cic) > 40 * 1024) --cic;
    const size_t smem = smem_for(cic);
    auto kern = direct_conv_kernel<T, KH_, KW_>;
    if (smem > 48 * 1024 &&
        ensure_smem_optin(reinterpret_cast<const void*>(kern), smem) != ACNN_OK)
        return cudaErrorInvalidValue;
    const int tiles = ((a.oh + kTH - 1) / kTH) * ((a.ow + kTW - 1) / kTW);
    dim3 grid(tiles, (d.c_out + kCOB - 1) / kCOB, d.n);
    launch_pdl(kern, grid, kThreads, smem, s, 
        static_cast<const T*>(a.x), static_cast<const T*>(a.w), a.bias, a.alpha,
        static_cast<const T*>(a.residual), static_cast<T*>(a.y), d.layout, a.out_layout, d.n,
        d.h, d.w, d.c_in, d.c_out, d.kh, d.kw, d.stride, d.pad, a.oh, a.ow, a.act, a.res_mode,
        cic);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dispatch(const ConvArgs& a, cudaStream_t s) {
    if (a.d.kh == 3 && a.d.kw == 3) return launch_typed<T, 3, 3>(a, s);
    if (a.d.kh == 1 && a.d.kw == 1) return launch_typed<T, 1, 1>(a, s);
    return launch_typed<T, 0, 0>(a, s);
}

}  // namespace

cudaError_t launch_direct_conv(const ConvArgs& a, cudaStream_t s) {
    switch (a.d.dtype) {
    case ACNN_F32: return launch_dispatch<float>(a, s);
    case ACNN_F16: return launch_dispatch<__half>(a, s);
    default: return launch_dispatch<__nv_bfloat16>(a, s);
    }
}

}  // namespace acnn
