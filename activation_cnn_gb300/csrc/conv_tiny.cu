// conv_tiny.cu -- direct 3x3 conv2d_fused for fp16/bf16 inputs with few
// channels: the RGB stem of the backbone (3 -> 32, stride 2, NHWC) and the
// first conv of the frame stack (7 or 6 planes -> 120, stride 2, NCHW).
//
// With C_in = 3..7 the reduction of one output is only 27..63 products, so a
// GEMM formulation either pads K to a tensor-core multiple or materialises an
// im2col matrix several times the size of the input.  Here the input is read
// once into shared memory and every product is an fp32 FMA.
//
// Prior art: rt.js wgslConv stages a slab of the input and its weights in
// workgroup memory and gives each invocation several output channels;
// wgslConvRBSg broadcasts the weights across a subgroup instead.  Both forms
// are here, chosen at compile time (WB):
//   * kWeightsSmem: the chunk's weights as fp32 in shared memory, read as
//     16-byte broadcast loads (the 8 weights a thread needs at one tap);
//   * kWeightsShfl: lane L of every warp holds the weights of output channel
//     co0 + L for all taps in registers, and each thread gathers its 8 with
//     warp shuffles (__shfl_sync) at every tap.
//
// A CTA of 256 threads (8 warps) computes an output tile of 8 rows x 32
// columns x 32 output channels.  Lane l of warp r owns output row oy0 + r,
// columns ox0 + 4 (l >> 2) .. + 3, channels co0 + 8 (l & 3) .. + 7: 32 fp32
// accumulators.  The input patch of the tile, (8 - 1) S + 3 rows x
// (32 - 1) S + 3 columns x C_in, is staged as fp32 with zeros outside the
// image; with stride 2 even and odd columns are stored apart so that the
// 8 distinct column groups of a warp fall in distinct banks.  Per input
// channel and kernel row a thread reads the 3S + 3 input values its 4 pixels
// need at the 3 horizontal taps once and issues 96 FMAs.
//
// Accumulation per output: fp32 FMAs in (ci, ky, kx) order; the fp32 bias
// is added to that sum in the epilogue, then residual / activation and one
// rounding to the storage type (as in the tensor-core epilogue).
#include "common.cuh"

namespace acnn {

namespace {

constexpr int kTinyThreads = 256;
constexpr int kTinyRows = 8;    // output rows per CTA (one per warp)
constexpr int kTinyCols = 32;   // output columns per CTA (4 per lane group of 4)
constexpr int kTinyCo = 32;     // output channels per CTA
constexpr int kWeightsSmem = 0, kWeightsShfl = 1;

// Patch geometry for stride S: rows and columns of input the tile reads, and
// the row pitch of one staged row (S = 2: two half rows of `half` floats).
template <int S> struct Patch {
    static constexpr int rows = (kTinyRows - 1) * S + 3;
    static constexpr int cols = (kTinyCols - 1) * S + 3;
    static constexpr int half = (cols + 1) / 2 + 1;  // odd pitch: even/odd halves
    static constexpr int pitch = S == 2 ? 2 * half : cols + 1;
    // staged position of column c within its row
    __device__ static constexpr int col(int c) { return S == 2 ? (c & 1) * half + (c >> 1) : c; }
};

// Occupancy: the shared-memory variant fits 64 registers (4 CTAs per SM, the
// latency of the staged loads hidden by 32 warps); the shuffle variant keeps
// C_in x 9 weights per lane and needs up to 128 (2 CTAs per SM).
template <int WB> struct TinyOcc { static constexpr int blocks = WB == 0 ? 3 : 2; };

template <typename T, int CIN, int S, int WB>
__global__ void __launch_bounds__(kTinyThreads, TinyOcc<WB>::blocks) tiny_conv3_kernel(
    const T* __restrict__ x, const T* __restrict__ w, const float* __restrict__ bias,
    const float* __restrict__ alpha, const T* __restrict__ res, T* __restrict__ y, int layout,
    int H, int W, int C_out, int P, int OH, int OW, int act, int res_mode) {
    using PT = Patch<S>;
    constexpr int KT = CIN * 9;                    // taps, (ci, ky, kx) order
    constexpr int NV = 3 * S + 3;                  // input values per (ci, ky) and thread
    __shared__ float s_in[CIN * PT::rows * PT::pitch];
    __shared__ __align__(16) float s_w[WB == kWeightsSmem ? KT * kTinyCo : 4];

    const int tiles_x = (OW + kTinyCols - 1) / kTinyCols;
    const int oy0 = (blockIdx.x / tiles_x) * kTinyRows, ox0 = (blockIdx.x % tiles_x) * kTinyCols;
    const int co0 = blockIdx.y * kTinyCo;
    const int n = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane & 3, px = lane >> 2;  // channel group, column group

    griddep_wait();  // every global read below may depend on the previous kernel
    // weights of this CTA's output channels (fp32); zero past C_out
    float wreg[WB == kWeightsShfl ? KT : 1];
    if constexpr (WB == kWeightsShfl) {
        const int co = co0 + lane;
#pragma unroll
        for (int t = 0; t < KT; ++t) {
            const int ci = t / 9, ky = (t % 9) / 3, kx = t % 3;
            wreg[t] = co < C_out
                          ? to_f32(w[layout == ACNN_NHWC ? ((long long)co * 9 + ky * 3 + kx) * CIN + ci
                                                         : ((long long)co * CIN + ci) * 9 + ky * 3 + kx])
                          : 0.0f;
        }
    }
    if constexpr (WB == kWeightsSmem) {
        for (int i = tid; i < KT * kTinyCo; i += kTinyThreads) {
            const int c = i % kTinyCo, t = i / kTinyCo, co = co0 + c;
            const int ci = t / 9, ky = (t % 9) / 3, kx = t % 3;
            s_w[i] = co < C_out
                         ? to_f32(w[layout == ACNN_NHWC ? ((long long)co * 9 + ky * 3 + kx) * CIN + ci
                                                        : ((long long)co * CIN + ci) * 9 + ky * 3 + kx])
                         : 0.0f;
        }
    }
    // stage the input patch (zero outside the image, rtdetr_gpu.rs IM2COL_SRC)
    const int gy0 = oy0 * S - P, gx0 = ox0 * S - P;
    constexpr int kElems = CIN * PT::rows * PT::cols;
    constexpr int kBatch = 8;  // independent loads in flight before any store
    for (int base = tid; base < kElems; base += kTinyThreads * kBatch) {
        float v[kBatch];
        int dst[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int idx = base + u * kTinyThreads;
            v[u] = 0.0f;
            dst[u] = -1;
            if (idx < kElems) {
                int ci, r, c;
                if (layout == ACNN_NHWC) {  // channels fastest: coalesced pixel runs
                    ci = idx % CIN;
                    const int q = idx / CIN;
                    c = q % PT::cols;
                    r = q / PT::cols;
                } else {  // columns fastest within a plane row
                    c = idx % PT::cols;
                    const int q = idx / PT::cols;
                    r = q % PT::rows;
                    ci = q / PT::rows;
                }
                dst[u] = (ci * PT::rows + r) * PT::pitch + PT::col(c);
                const int gy = gy0 + r, gx = gx0 + c;
                if (gy >= 0 && gy < H && gx >= 0 && gx < W)
                    v[u] = to_f32(x[layout == ACNN_NHWC
                                        ? (((long long)n * H + gy) * W + gx) * CIN + ci
                                        : (((long long)n * CIN + ci) * H + gy) * W + gx]);
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            if (dst[u] >= 0) s_in[dst[u]] = v[u];
    }
    __syncthreads();

    float acc[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[j][c] = 0.0f;

    const int r0 = warp * S;             // first patch row of this warp's output row
    const int c0 = 4 * px * S;           // first patch column of this lane's 4 pixels
#pragma unroll
    for (int ci = 0; ci < CIN; ++ci) {
#pragma unroll
        for (int ky = 0; ky < 3; ++ky) {
            const float* row = s_in + (ci * PT::rows + r0 + ky) * PT::pitch;
            float xv[NV];
#pragma unroll
            for (int i = 0; i < NV; ++i) xv[i] = row[PT::col(c0 + i)];
#pragma unroll
            for (int kx = 0; kx < 3; ++kx) {
                const int t = ci * 9 + ky * 3 + kx;
                float wv[8];
                if constexpr (WB == kWeightsSmem) {
                    const float4* wp = reinterpret_cast<const float4*>(s_w + t * kTinyCo + g * 8);
                    const float4 a = wp[0], b = wp[1];
                    wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
                    wv[4] = b.x; wv[5] = b.y; wv[6] = b.z; wv[7] = b.w;
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c) wv[c] = __shfl_sync(0xffffffffu, wreg[t], g * 8 + c);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float xj = xv[j * S + kx];
#pragma unroll
                    for (int c = 0; c < 8; ++c) acc[j][c] = fmaf(xj, wv[c], acc[j][c]);
                }
            }
        }
    }

    // fused epilogue: bias -> residual / activation -> storage type
    const int oy = oy0 + warp;
    const int cb = co0 + g * 8;
    if (oy >= OH || cb >= C_out) return;
    float bv[8], av[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const bool in = cb + c < C_out;
        bv[c] = (bias && in) ? bias[cb + c] : 0.0f;
        av[c] = (act == ACNN_ACT_PRELU && in) ? alpha[cb + c] : 0.0f;
    }
    const int oxb = ox0 + 4 * px;
    if (layout == ACNN_NHWC && C_out % 8 == 0) {
        // one 16-byte vector of 8 channels per pixel
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int ox = oxb + j;
            if (ox >= OW) break;
            const long long oi = (((long long)n * OH + oy) * OW + ox) * C_out + cb;
            Vec<T, 8> rv, ov;
            if (res_mode != ACNN_RES_NONE) rv = *reinterpret_cast<const Vec<T, 8>*>(res + oi);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float r = res_mode != ACNN_RES_NONE ? to_f32(rv.v[c]) : 0.0f;
                ov.v[c] = from_f32<T>(epilogue_fast(bv[c] + acc[j][c], act, av[c], res_mode, r));
            }
            *reinterpret_cast<Vec<T, 8>*>(y + oi) = ov;
        }
        return;
    }
    if (layout == ACNN_NCHW && OW % 4 == 0 && oxb < OW) {
        // the thread's 4 pixels are 4 consecutive values of each channel's row:
        // one 8-byte store per channel (OW % 4 == 0 keeps it aligned)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int co = cb + c;
            if (co >= C_out) break;
            const long long oi = (((long long)n * C_out + co) * OH + oy) * OW + oxb;
            Vec<T, 4> rv, ov;
            if (res_mode != ACNN_RES_NONE) rv = *reinterpret_cast<const Vec<T, 4>*>(res + oi);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float r = res_mode != ACNN_RES_NONE ? to_f32(rv.v[j]) : 0.0f;
                ov.v[j] = from_f32<T>(epilogue_fast(bv[c] + acc[j][c], act, av[c], res_mode, r));
            }
            *reinterpret_cast<Vec<T, 4>*>(y + oi) = ov;
        }
        return;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const int co = cb + c;
        if (co >= C_out) break;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int ox = oxb + j;
            if (ox >= OW) break;
            const long long oi = act_index(layout, C_out, OH, OW, n, co, oy, ox);
            const float r = res_mode != ACNN_RES_NONE ? to_f32(res[oi]) : 0.0f;
            y[oi] = from_f32<T>(epilogue_fast(bv[c] + acc[j][c], act, av[c], res_mode, r));
        }
    }
}

template <typename T, int CIN, int S>
cudaError_t launch_tiny_typed(const ConvArgs& a, int wb, cudaStream_t s) {
    const acnn_conv_desc& d = a.d;
    const int tiles = ((a.oh + kTinyRows - 1) / kTinyRows) * ((a.ow + kTinyCols - 1) / kTinyCols);
    dim3 grid((unsigned)tiles, (unsigned)((d.c_out + kTinyCo - 1) / kTinyCo), (unsigned)d.n);
    auto args = [&](auto kern) {
        launch_pdl(kern, grid, kTinyThreads, 0, s, static_cast<const T*>(a.x),
                   static_cast<const T*>(a.w), a.bias, a.alpha, static_cast<const T*>(a.residual),
                   static_cast<T*>(a.y), d.layout, d.h, d.w, d.c_out, d.pad, a.oh, a.ow, a.act,
                   a.res_mode);
    };
    if (wb == kWeightsShfl) args(tiny_conv3_kernel<T, CIN, S, kWeightsShfl>);
    else args(tiny_conv3_kernel<T, CIN, S, kWeightsSmem>);
    return cudaGetLastError();
}

template <typename T, int CIN>
cudaError_t launch_tiny_cin(const ConvArgs& a, int wb, cudaStream_t s) {
    return a.d.stride == 1 ? launch_tiny_typed<T, CIN, 1>(a, wb, s)
                           : launch_tiny_typed<T, CIN, 2>(a, wb, s);
}

template <typename T> cudaError_t launch_tiny_t(const ConvArgs& a, int wb, cudaStream_t s) {
    switch (a.d.c_in) {
    case 3: return launch_tiny_cin<T, 3>(a, wb, s);
    case 6: return launch_tiny_cin<T, 6>(a, wb, s);
    default: return launch_tiny_cin<T, 7>(a, wb, s);
    }
}

}  // namespace

bool tiny_conv_ok(const acnn_conv_desc& d, int oh, int ow) {
    if (d.dtype == ACNN_F32) return false;
    if (d.c_in != 3 && d.c_in != 6 && d.c_in != 7) return false;
    if (d.kh != 3 || d.kw != 3 || (d.stride != 1 && d.stride != 2) || d.pad > 2) return false;
    const long long tiles = (long long)((oh + kTinyRows - 1) / kTinyRows) *
                            ((ow + kTinyCols - 1) / kTinyCols);
    return tiles <= 0x7fffffffLL && d.n <= 65535 && (long long)d.n * d.h * d.w * d.c_in < (1ll << 40);
}

cudaError_t launch_tiny_conv(const ConvArgs& a, int weights_by_shuffle, cudaStream_t s) {
    const int wb = weights_by_shuffle ? kWeightsShfl : kWeightsSmem;
    return a.d.dtype == ACNN_BF16 ? launch_tiny_t<__nv_bfloat16>(a, wb, s)
                                  : launch_tiny_t<__half>(a, wb, s);
}

}  // namespace acnn
