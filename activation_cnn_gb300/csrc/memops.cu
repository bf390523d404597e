// memops.cu -- the memory-bound companion ops of the conv layer:
// max/avg pool, nearest/bilinear resize, channel concat, the RGBA8 frame
// prep, the 4x4/s2 transposed conv, and the NCHW -> NHWC transpose that
// feeds NCHW tensors to the tensor-core conv.
//
// NHWC kernels move 16 bytes per thread along the channel axis (8 bf16/fp16
// or 4 fp32 elements) when the channel count allows it; NCHW kernels walk the
// innermost (x) axis so that a warp touches consecutive addresses.  All use
// grid-stride loops over a grid sized in multiples of the SM count.
#include "common.cuh"

namespace acnn {

namespace {

constexpr int kThreads = 256;

// ----------------------------------------------------------------------------
// pooling: rtdetr_gpu.rs MAXPOOL_SRC (taps outside the input are skipped, so
// padding acts as -inf; the running max is replaced only by a strictly larger
// tap, in (dy, dx) order) and AVGPOOL_SRC ((a+b+c+d)*0.25 over a 2x2/s2 window;
// k x k windows generalise it as sum * (1/k^2)).
// ----------------------------------------------------------------------------
template <typename T, int V>
__global__ void __launch_bounds__(kThreads) pool_nhwc_kernel(
    const T* __restrict__ x, T* __restrict__ y, int kind, int N, int H, int W, int C, int OH,
    int OW, int K, int S, int P) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const int CV = C / V;
    const long long total = (long long)N * OH * OW * CV;
    const float inv = 1.0f / (float)(K * K);
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < (uint32_t)total;
         i += gridDim.x * blockDim.x) {
        int cv = (int)(i % CV);
        uint32_t p = i / CV;
        int ox = (int)(p % OW);
        p /= OW;
        int oy = (int)(p % OH);
        int n = (int)(p / OH);
        float acc[V];
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = kind == ACNN_POOL_MAX ? -INFINITY : 0.0f;
        for (int dy = 0; dy < K; ++dy) {
            int iy = oy * S + dy - P;
            if (iy < 0 || iy >= H) continue;
            for (int dx = 0; dx < K; ++dx) {
                int ix = ox * S + dx - P;
                if (ix < 0 || ix >= W) continue;
                Vec<T, V> t = *reinterpret_cast<const Vec<T, V>*>(
                    x + (((long long)n * H + iy) * W + ix) * C + (long long)cv * V);
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    float f = to_f32(t.v[v]);
                    if (kind == ACNN_POOL_MAX) {
                        if (f > acc[v]) acc[v] = f;
                    } else {
                        acc[v] += f;
                    }
                }
            }
        }
        Vec<T, V> o;
#pragma unroll
        for (int v = 0; v < V; ++v)
            o.v[v] = from_f32<T>(kind == ACNN_POOL_MAX ? acc[v] : acc[v] * inv);
        *reinterpret_cast<Vec<T, V>*>(y + (((long long)n * OH + oy) * OW + ox) * C +
                                      (long long)cv * V) = o;
    }
}

// 3x3/s2/p1 max-pool, NHWC (the stem's pool): all nine taps are loaded before
// any is compared (addresses clamped into the image, out-of-image taps then
// masked), so a thread keeps nine 16-byte loads in flight; the comparison
// order and the strictly-greater rule are those of the generic kernel.
template <typename T, int V>
__global__ void __launch_bounds__(kThreads) maxpool3s2_nhwc_kernel(
    const T* __restrict__ x, T* __restrict__ y, int N, int H, int W, int C, int OH, int OW) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const int CV = C / V;
    const long long total = (long long)N * OH * OW * CV;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < (uint32_t)total;
         i += gridDim.x * blockDim.x) {
        const int cv = (int)(i % CV);
        uint32_t p = i / CV;
        const int ox = (int)(p % OW);
        p /= OW;
        const int oy = (int)(p % OH);
        const int n = (int)(p / OH);
        const T* img = x + (long long)n * H * W * C + (long long)cv * V;
        Vec<T, V> t[9];
        bool ok[9];
#pragma unroll
        for (int dy = 0; dy < 3; ++dy)
#pragma unroll
            for (int dx = 0; dx < 3; ++dx) {
                const int iy = 2 * oy - 1 + dy, ix = 2 * ox - 1 + dx;
                ok[dy * 3 + dx] = iy >= 0 && iy < H && ix >= 0 && ix < W;
                const int iyc = min(max(iy, 0), H - 1), ixc = min(max(ix, 0), W - 1);
                t[dy * 3 + dx] = *reinterpret_cast<const Vec<T, V>*>(
                    img + ((long long)iyc * W + ixc) * C);
            }
        float best[V];
#pragma unroll
        for (int v = 0; v < V; ++v) best[v] = -INFINITY;
#pragma unroll
        for (int k = 0; k < 9; ++k)
            if (ok[k]) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const float f = to_f32(t[k].v[v]);
                    if (f > best[v]) best[v] = f;
                }
            }
        Vec<T, V> o;
#pragma unroll
        for (int v = 0; v < V; ++v) o.v[v] = from_f32<T>(best[v]);
        *reinterpret_cast<Vec<T, V>*>(y + (((long long)n * OH + oy) * OW + ox) * C +
                                      (long long)cv * V) = o;
    }
}

// Row-blocked NHWC kernels for the backbone's hot shapes.  Block (r, g) of the
// 2-D grid covers output row r = n*OH + oy and the g-th run of U*256 16-byte
// channel vectors of that row (vector j of the row: pixel j / CV, vector
// j % CV), so each thread computes its coordinates with one division and
// issues the loads of all its vectors before it stores any.

// 2x2/s2/p0 average pool: (a + b + c + d) * 0.25 in (dy, dx) order, as the
// generic kernel computes it.
template <typename T, int V, int U>
__global__ void __launch_bounds__(kThreads) avgpool2_rows_kernel(
    const T* __restrict__ x, T* __restrict__ y, int H, int W, int C, int OH, int OW) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const int CV = C / V;
    const int r = blockIdx.x, oy = r % OH, n = r / OH;
    const int row_vecs = OW * CV;
    const T* x0 = x + ((long long)n * H + 2 * oy) * W * C;
    const T* x1 = x0 + (long long)W * C;
    T* yr = y + (long long)r * OW * C;
    Vec<T, V> t[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int j = (blockIdx.y * U + u) * kThreads + threadIdx.x;
        if (j < row_vecs) {
            const int ox = j / CV, cv = j - ox * CV;
            const long long o = (long long)(2 * ox) * C + (long long)cv * V;
            t[u][0] = *reinterpret_cast<const Vec<T, V>*>(x0 + o);
            t[u][1] = *reinterpret_cast<const Vec<T, V>*>(x0 + o + C);
            t[u][2] = *reinterpret_cast<const Vec<T, V>*>(x1 + o);
            t[u][3] = *reinterpret_cast<const Vec<T, V>*>(x1 + o + C);
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int j = (blockIdx.y * U + u) * kThreads + threadIdx.x;
        if (j < row_vecs) {
            const int ox = j / CV, cv = j - ox * CV;
            Vec<T, V> o;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                float acc = 0.0f;
#pragma unroll
                for (int k = 0; k < 4; ++k) acc += to_f32(t[u][k].v[v]);
                o.v[v] = from_f32<T>(acc * 0.25f);
            }
            *reinterpret_cast<Vec<T, V>*>(yr + (long long)ox * C + (long long)cv * V) = o;
        }
    }
}

// 3x3/s2/p1 max pool, row-blocked: nine clamped loads per vector, then the
// out-of-image taps masked, strictly-greater replacement in (dy, dx) order.
template <typename T, int V>
__global__ void __launch_bounds__(kThreads) maxpool3s2_rows_kernel(
    const T* __restrict__ x, T* __restrict__ y, int H, int W, int C, int OH, int OW) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const int CV = C / V;
    const int r = blockIdx.x, oy = r % OH, n = r / OH;
    const int j = blockIdx.y * kThreads + threadIdx.x;
    if (j >= OW * CV) return;
    const int ox = j / CV, cv = j - ox * CV;
    const T* img = x + (long long)n * H * W * C + (long long)cv * V;
    Vec<T, V> t[9];
    bool ok[9];
#pragma unroll
    for (int dy = 0; dy < 3; ++dy)
#pragma unroll
        for (int dx = 0; dx < 3; ++dx) {
            const int iy = 2 * oy - 1 + dy, ix = 2 * ox - 1 + dx;
            ok[dy * 3 + dx] = iy >= 0 && iy < H && ix >= 0 && ix < W;
            const int iyc = min(max(iy, 0), H - 1), ixc = min(max(ix, 0), W - 1);
            t[dy * 3 + dx] = *reinterpret_cast<const Vec<T, V>*>(img + ((long long)iyc * W + ixc) * C);
        }
    float best[V];
#pragma unroll
    for (int v = 0; v < V; ++v) best[v] = -INFINITY;
#pragma unroll
    for (int k = 0; k < 9; ++k)
        if (ok[k]) {
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const float f = to_f32(t[k].v[v]);
                if (f > best[v]) best[v] = f;
            }
        }
    Vec<T, V> o;
#pragma unroll
    for (int v = 0; v < V; ++v) o.v[v] = from_f32<T>(best[v]);
    *reinterpret_cast<Vec<T, V>*>(y + ((long long)r * OW + ox) * C + (long long)cv * V) = o;
}

// Nearest 2x, row-blocked over input rows: one load, four stores per vector.
template <typename T, int V, int U>
__global__ void __launch_bounds__(kThreads) up2_rows_kernel(const T* __restrict__ x,
                                                            T* __restrict__ y, int H, int W,
                                                            int C) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const int CV = C / V;
    const int r = blockIdx.x, iy = r % H, n = r / H;
    const int OW = 2 * W;
    const T* xr = x + (long long)r * W * C;
    T* y0 = y + ((long long)n * 2 * H + 2 * iy) * OW * C;
    T* y1 = y0 + (long long)OW * C;
    Vec<T, V> t[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int j = (blockIdx.y * U + u) * kThreads + threadIdx.x;
        if (j < W * CV) t[u] = *reinterpret_cast<const Vec<T, V>*>(xr + (long long)j * V);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int j = (blockIdx.y * U + u) * kThreads + threadIdx.x;
        if (j < W * CV) {
            const int ix = j / CV, cv = j - ix * CV;
            const long long o = (long long)(2 * ix) * C + (long long)cv * V;
            *reinterpret_cast<Vec<T, V>*>(y0 + o) = t[u];
            *reinterpret_cast<Vec<T, V>*>(y0 + o + C) = t[u];
            *reinterpret_cast<Vec<T, V>*>(y1 + o) = t[u];
            *reinterpret_cast<Vec<T, V>*>(y1 + o + C) = t[u];
        }
    }
}

// Nearest 2x, NHWC: one thread per input pixel and 16-byte channel vector,
// one load and the four stores of its 2x2 output block.
template <typename T, int V>
__global__ void __launch_bounds__(kThreads) up2_nhwc_kernel(const T* __restrict__ x,
                                                            T* __restrict__ y, int N, int H,
                                                            int W, int C) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const int CV = C / V;
    const long long total = (long long)N * H * W * CV;
    const int OW = 2 * W;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < (uint32_t)total;
         i += gridDim.x * blockDim.x) {
        const int cv = (int)(i % CV);
        uint32_t p = i / CV;
        const int ix = (int)(p % W);
        p /= W;
        const int iy = (int)(p % H);
        const int n = (int)(p / H);
        const Vec<T, V> t = *reinterpret_cast<const Vec<T, V>*>(x + (long long)i * V);
        T* o = y + (((long long)n * 2 * H + 2 * iy) * OW + 2 * ix) * C + (long long)cv * V;
        *reinterpret_cast<Vec<T, V>*>(o) = t;
        *reinterpret_cast<Vec<T, V>*>(o + C) = t;
        *reinterpret_cast<Vec<T, V>*>(o + (long long)OW * C) = t;
        *reinterpret_cast<Vec<T, V>*>(o + (long long)OW * C + C) = t;
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) pool_nchw_kernel(
    const T* __restrict__ x, T* __restrict__ y, int kind, int N, int C, int H, int W, int OH,
    int OW, int K, int S, int P) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const long long total = (long long)N * C * OH * OW;
    const float inv = 1.0f / (float)(K * K);
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < (uint32_t)total;
         i += gridDim.x * blockDim.x) {
        int ox = (int)(i % OW);
        uint32_t p = i / OW;
        int oy = (int)(p % OH);
        const uint32_t nc = p / OH;
        const T* plane = x + (long long)nc * H * W;
        float acc = kind == ACNN_POOL_MAX ? -INFINITY : 0.0f;
        for (int dy = 0; dy < K; ++dy) {
            int iy = oy * S + dy - P;
            if (iy < 0 || iy >= H) continue;
            for (int dx = 0; dx < K; ++dx) {
                int ix = ox * S + dx - P;
                if (ix < 0 || ix >= W) continue;
                float f = to_f32(plane[(long long)iy * W + ix]);
                if (kind == ACNN_POOL_MAX) {
                    if (f > acc) acc = f;
                } else {
                    acc += f;
                }
            }
        }
        y[i] = from_f32<T>(kind == ACNN_POOL_MAX ? acc : acc * inv);
    }
}

// ----------------------------------------------------------------------------
// resize.  Nearest: source index floor(dst * in / out) (rtdetr_gpu.rs
// UPSAMPLE_SRC for 2x).  Bilinear, align_corners=false (rt.js wgslPrepQuarter,
// wgslFlowOut): src = (dst + 0.5) * (in/out) - 0.5, x0 = floor(src),
// f = src - x0, taps x0 and x0 + 1 clamped to the image,
// mix(mix(v00, v10, fx), mix(v01, v11, fx), fy).
// ----------------------------------------------------------------------------
struct BilinearTap {
    int a, b;
    float f;
};

__device__ __forceinline__ BilinearTap bilinear_tap(int dst, float scale, int in) {
    float src = ((float)dst + 0.5f) * scale - 0.5f;
    float fl = floorf(src);
    int i0 = (int)fl;
    BilinearTap t;
    t.f = src - fl;
    t.a = min(max(i0, 0), in - 1);
    t.b = min(max(i0 + 1, 0), in - 1);
    return t;
}

__device__ __forceinline__ float mixf(float a, float b, float t) { return a * (1.0f - t) + b * t; }

template <typename Ti, typename To, int V>
__global__ void __launch_bounds__(kThreads) resize_nhwc_kernel(
    const Ti* __restrict__ x, To* __restrict__ y, int mode, int N, int H, int W, int C, int OH,
    int OW, float sy, float sx) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const int CV = C / V;
    const long long total = (long long)N * OH * OW * CV;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < (uint32_t)total;
         i += gridDim.x * blockDim.x) {
        int cv = (int)(i % CV);
        uint32_t p = i / CV;
        int ox = (int)(p % OW);
        p /= OW;
        int oy = (int)(p % OH);
        int n = (int)(p / OH);
        const Ti* img = x + (long long)n * H * W * C + (long long)cv * V;
        Vec<To, V> o;
        if (mode == ACNN_RESIZE_NEAREST) {
            int iy = (int)(((long long)oy * H) / OH);
            int ix = (int)(((long long)ox * W) / OW);
            Vec<Ti, V> t = *reinterpret_cast<const Vec<Ti, V>*>(img + ((long long)iy * W + ix) * C);
#pragma unroll
            for (int v = 0; v < V; ++v) o.v[v] = from_f32<To>(to_f32(t.v[v]));
        } else {
            BilinearTap ty = bilinear_tap(oy, sy, H), tx = bilinear_tap(ox, sx, W);
            Vec<Ti, V> v00 = *reinterpret_cast<const Vec<Ti, V>*>(img + ((long long)ty.a * W + tx.a) * C);
            Vec<Ti, V> v10 = *reinterpret_cast<const Vec<Ti, V>*>(img + ((long long)ty.a * W + tx.b) * C);
            Vec<Ti, V> v01 = *reinterpret_cast<const Vec<Ti, V>*>(img + ((long long)ty.b * W + tx.a) * C);
            Vec<Ti, V> v11 = *reinterpret_cast<const Vec<Ti, V>*>(img + ((long long)ty.b * W + tx.b) * C);
#pragma unroll
            for (int v = 0; v < V; ++v) {
                float top = mixf(to_f32(v00.v[v]), to_f32(v10.v[v]), tx.f);
                float bot = mixf(to_f32(v01.v[v]), to_f32(v11.v[v]), tx.f);
                o.v[v] = from_f32<To>(mixf(top, bot, ty.f));
            }
        }
        *reinterpret_cast<Vec<To, V>*>(y + (((long long)n * OH + oy) * OW + ox) * C +
                                       (long long)cv * V) = o;
    }
}

template <typename Ti, typename To>
__global__ void __launch_bounds__(kThreads) resize_nchw_kernel(
    const Ti* __restrict__ x, To* __restrict__ y, int mode, int NC, int H, int W, int OH, int OW,
    float sy, float sx) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const long long total = (long long)NC * OH * OW;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < (uint32_t)total;
         i += gridDim.x * blockDim.x) {
        int ox = (int)(i % OW);
        uint32_t p = i / OW;
        int oy = (int)(p % OH);
        const uint32_t nc = p / OH;
        const Ti* plane = x + (long long)nc * H * W;
        float v;
        if (mode == ACNN_RESIZE_NEAREST) {
            int iy = (int)(((long long)oy * H) / OH);
            int ix = (int)(((long long)ox * W) / OW);
            v = to_f32(plane[(long long)iy * W + ix]);
        } else {
            BilinearTap ty = bilinear_tap(oy, sy, H), tx = bilinear_tap(ox, sx, W);
            float top = mixf(to_f32(plane[(long long)ty.a * W + tx.a]),
                             to_f32(plane[(long long)ty.a * W + tx.b]), tx.f);
            float bot = mixf(to_f32(plane[(long long)ty.b * W + tx.a]),
                             to_f32(plane[(long long)ty.b * W + tx.b]), tx.f);
            v = mixf(top, bot, ty.f);
        }
        y[i] = from_f32<To>(v);
    }
}

// NCHW resize, one block per output row (plane nc, row oy): the row's source
// rows and y weight are computed once, each thread produces V consecutive
// outputs of the row (its taps are L1 hits: a x8 upsample reads 2-3 source
// columns for 8 outputs) and writes them as one 16-byte vector.  Same
// arithmetic, in the same order, as resize_nchw_kernel.
template <typename Ti, typename To, int V>
__global__ void __launch_bounds__(kThreads) resize_nchw_rows_kernel(
    const Ti* __restrict__ x, To* __restrict__ y, int mode, int H, int W, int OH, int OW,
    float sy, float sx) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const long long r = blockIdx.x;  // nc * OH + oy
    const int oy = (int)(r % OH);
    const long long nc = r / OH;
    const int ox0 = (blockIdx.y * kThreads + threadIdx.x) * V;
    if (ox0 >= OW) return;
    const Ti* plane = x + nc * H * W;
    Vec<To, V> o;
    if (mode == ACNN_RESIZE_NEAREST) {
        const Ti* row = plane + (long long)(((long long)oy * H) / OH) * W;
#pragma unroll
        for (int v = 0; v < V; ++v)
            o.v[v] = from_f32<To>(to_f32(row[((long long)(ox0 + v) * W) / OW]));
    } else {
        const BilinearTap ty = bilinear_tap(oy, sy, H);
        const Ti* ra = plane + (long long)ty.a * W;
        const Ti* rb = plane + (long long)ty.b * W;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const BilinearTap tx = bilinear_tap(ox0 + v, sx, W);
            const float top = mixf(to_f32(ra[tx.a]), to_f32(ra[tx.b]), tx.f);
            const float bot = mixf(to_f32(rb[tx.a]), to_f32(rb[tx.b]), tx.f);
            o.v[v] = from_f32<To>(mixf(top, bot, ty.f));
        }
    }
    *reinterpret_cast<Vec<To, V>*>(y + r * OW + ox0) = o;
}

// NCHW bilinear upsample by 4 or more (the frame stack's x8 of the flow map),
// eight output rows per block: those rows read at most four source rows, so
// each thread interpolates its V columns along x on those source rows once
// (kept in registers) and every output is then one interpolation along y --
// the same operations, in the same order, as resize_nchw_kernel
// (mix(mix(v00, v10, fx), mix(v01, v11, fx), fy)), so the same bits.
constexpr int kUpRows = 8, kUpSpan = 4;

template <typename Ti, typename To, int V>
__global__ void __launch_bounds__(kThreads) resize_nchw_up_kernel(
    const Ti* __restrict__ x, To* __restrict__ y, int H, int W, int OH, int OW, float sy,
    float sx) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const int groups = (OH + kUpRows - 1) / kUpRows;
    const long long nc = blockIdx.x / groups;
    const int oy0 = (blockIdx.x % groups) * kUpRows;
    const int ox0 = (blockIdx.y * kThreads + threadIdx.x) * V;
    if (ox0 >= OW) return;
    const Ti* plane = x + nc * H * W;
    const int a0 = bilinear_tap(oy0, sy, H).a;  // first source row of the group
    // x-interpolated values of source rows a0 .. a0 + kUpSpan - 1 (clamped)
    float xi[kUpSpan][V];
    BilinearTap tx[V];
#pragma unroll
    for (int v = 0; v < V; ++v) tx[v] = bilinear_tap(ox0 + v, sx, W);
#pragma unroll
    for (int j = 0; j < kUpSpan; ++j) {
        const Ti* row = plane + (long long)min(a0 + j, H - 1) * W;
#pragma unroll
        for (int v = 0; v < V; ++v) xi[j][v] = mixf(to_f32(row[tx[v].a]), to_f32(row[tx[v].b]), tx[v].f);
    }
#pragma unroll 1
    for (int r = 0; r < kUpRows; ++r) {
        const int oy = oy0 + r;
        if (oy >= OH) break;
        const BilinearTap ty = bilinear_tap(oy, sy, H);
        const int ja = ty.a - a0, jb = ty.b - a0;  // in [0, kUpSpan) (checked on the host)
        Vec<To, V> o;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            float top = xi[0][v], bot = xi[0][v];
#pragma unroll
            for (int j = 1; j < kUpSpan; ++j) {
                if (ja == j) top = xi[j][v];
                if (jb == j) bot = xi[j][v];
            }
            o.v[v] = from_f32<To>(mixf(top, bot, ty.f));
        }
        *reinterpret_cast<Vec<To, V>*>(y + (nc * OH + oy) * OW + ox0) = o;
    }
}

// ----------------------------------------------------------------------------
// The 4x4/s2/p1 transposed conv as a 3x3/s1/p1 conv with four outputs per
// output channel, one per output parity (py, px): output (2a + py, 2b + px)
// of channel co takes input (a - 1 + dy, b - 1 + dx) through kernel tap
// (ky, kx) = (py + 3 - 2 dy, px + 3 - 2 dx) when both lie in [0, 3] (rt.js
// wgslDeconv's gather form, regrouped).  The conv's output channel
// co * 4 + py * 2 + px then holds output pixel (2a + py, 2b + px) of co at
// its pixel (a, b), and a pixel shuffle puts it in place.
// Weights: w (fp32 [CI][CO][4][4]) -> wg ([CO4][3][3][CI], storage type, OHWI
// for the NHWC conv), CO4 = 4 CO rounded up to 8 (extra channels zero); bias
// and PReLU alpha repeated four times ([CO4] fp32, zero past 4 CO).
template <typename T>
__global__ void __launch_bounds__(kThreads) deconv_gemm_weights_kernel(
    const float* __restrict__ w, const float* __restrict__ bias, const float* __restrict__ alpha,
    T* __restrict__ wg, float* __restrict__ bg, float* __restrict__ ag, int CI, int CO, int CO4) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const long long total = (long long)CO4 * 9 * CI;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int ci = (int)(i % CI);
        const long long q = i / CI;
        const int t = (int)(q % 9), o = (int)(q / 9);
        const int dy = t / 3, dx = t % 3;
        float v = 0.0f;
        if (o < 4 * CO) {
            const int co = o >> 2, py = (o >> 1) & 1, px = o & 1;
            const int ky = py + 3 - 2 * dy, kx = px + 3 - 2 * dx;
            if (ky >= 0 && ky < 4 && kx >= 0 && kx < 4)
                v = w[(((long long)ci * CO + co) * 4 + ky) * 4 + kx];
        }
        wg[i] = from_f32<T>(v);
    }
    for (int o = blockIdx.x * blockDim.x + threadIdx.x; o < CO4; o += gridDim.x * blockDim.x) {
        bg[o] = (bias && o < 4 * CO) ? bias[o >> 2] : 0.0f;
        ag[o] = (alpha && o < 4 * CO) ? alpha[o >> 2] : 0.0f;
    }
}

// Pixel shuffle: ys (NHWC [N][H][W][CO4]) -> y ([N][CO][2H][2W] or NHWC
// [N][2H][2W][CO]): y(co, 2a + py, 2b + px) = ys(a, b, co * 4 + py * 2 + px).
template <typename T>
__global__ void __launch_bounds__(kThreads) deconv_shuffle_kernel(
    const T* __restrict__ ys, T* __restrict__ y, int layout, int N, int H, int W, int CO, int CO4) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const int OH = 2 * H, OW = 2 * W;
    const long long total = (long long)N * CO * OH * OW;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        int n, co, oy, ox;
        if (layout == ACNN_NCHW) {  // consecutive threads: consecutive x of one plane
            ox = (int)(i % OW);
            long long q = i / OW;
            oy = (int)(q % OH);
            q /= OH;
            co = (int)(q % CO);
            n = (int)(q / CO);
        } else {  // consecutive threads: consecutive channels of one pixel
            co = (int)(i % CO);
            long long q = i / CO;
            ox = (int)(q % OW);
            q /= OW;
            oy = (int)(q % OH);
            n = (int)(q / OH);
        }
        const int a = oy >> 1, py = oy & 1, b = ox >> 1, px = ox & 1;
        y[i] = ys[(((long long)n * H + a) * W + b) * CO4 + co * 4 + py * 2 + px];
    }
}

// ----------------------------------------------------------------------------
// concat: rtdetr_gpu.rs CONCAT_SRC, y = [a | b] along channels.  NHWC: per
// pixel; NCHW: per image, the c_a planes of a then the c_b planes of b.  Both
// reduce to copying runs of `ra` elements from a and `rb` from b into
// consecutive runs of ra + rb elements of y.
// ----------------------------------------------------------------------------
template <typename T, int V>
__global__ void __launch_bounds__(kThreads) concat_kernel(
    const T* __restrict__ a, const T* __restrict__ b, T* __restrict__ y, long long runs,
    int ra, int rb) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    // four vectors per thread (one block-width apart), all loaded before any
    // is stored; one division per vector
    constexpr int U = 4;
    const uint32_t rv = (uint32_t)((ra + rb) / V);
    const uint32_t total = (uint32_t)(runs * rv);
    Vec<T, V> t[U];
    uint32_t run[U];
    int e[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint32_t i = (blockIdx.x * U + u) * blockDim.x + threadIdx.x;
        run[u] = i / rv;
        e[u] = (int)(i - run[u] * rv) * V;
        if (i < total) {
            const T* src = e[u] < ra ? a + (long long)run[u] * ra + e[u]
                                     : b + (long long)run[u] * rb + (e[u] - ra);
            t[u] = *reinterpret_cast<const Vec<T, V>*>(src);
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint32_t i = (blockIdx.x * U + u) * blockDim.x + threadIdx.x;
        if (i < total)
            *reinterpret_cast<Vec<T, V>*>(y + (long long)run[u] * (ra + rb) + e[u]) = t[u];
    }
}

// ----------------------------------------------------------------------------
// frame prep: rt.js wgslPrepQuarter.  unpack4x8unorm of each RGBA8 pixel gives
// r, g, b = bytes 0, 1, 2 over 255; the output planes are b, g, r of frame 0,
// b, g, r of frame 1 and a plane holding t, each colour plane bilinearly
// downsampled by 4 (src = (dst + 0.5) * 4 - 0.5, taps clamped).
// ----------------------------------------------------------------------------
template <typename To>
__global__ void __launch_bounds__(kThreads) prep_quarter_kernel(
    const uint32_t* __restrict__ f0, const uint32_t* __restrict__ f1, To* __restrict__ y, int H,
    int W, float t) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const int QH = H / 4, QW = W / 4;
    const long long P = (long long)QH * QW;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < (uint32_t)P;
         i += gridDim.x * blockDim.x) {
        int qx = (int)(i % QW), qy = (int)(i / QW);
        BilinearTap ty = bilinear_tap(qy, 4.0f, H), tx = bilinear_tap(qx, 4.0f, W);
#pragma unroll
        for (int f = 0; f < 2; ++f) {
            const uint32_t* fr = f == 0 ? f0 : f1;
            uint32_t p00 = fr[(long long)ty.a * W + tx.a], p10 = fr[(long long)ty.a * W + tx.b];
            uint32_t p01 = fr[(long long)ty.b * W + tx.a], p11 = fr[(long long)ty.b * W + tx.b];
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                int sh = 8 * (2 - k);  // plane k is byte 2 - k: b, g, r
                float top = mixf(((p00 >> sh) & 255u) / 255.0f, ((p10 >> sh) & 255u) / 255.0f, tx.f);
                float bot = mixf(((p01 >> sh) & 255u) / 255.0f, ((p11 >> sh) & 255u) / 255.0f, tx.f);
                y[(3 * f + k) * P + i] = from_f32<To>(mixf(top, bot, ty.f));
            }
        }
        y[6 * P + i] = from_f32<To>(t);
    }
}

// ----------------------------------------------------------------------------
// deconv: rt.js wgslDeconv in gather form.  One thread per output pixel and
// block of up to 8 output channels.  For output row oy the live taps are the
// ky with ty = oy + P - ky >= 0, ty % S == 0 and iy = ty / S < H; for 4x4/s2/p1
// that is two of the four ky (one parity class), so 4 of 16 taps are live.
// ----------------------------------------------------------------------------
constexpr int kDeconvCoBlock = 8;

// 4x4/s2/p1 transposed conv (the only geometry of the ABI), gather form
// restated per input pixel: output (2a + py, 2b + px) takes its taps from the
// 3x3 input neighbourhood of (a, b) -- rows a (ky = 1) and a - 1 (ky = 3) for
// py = 0, rows a + 1 (ky = 0) and a (ky = 2) for py = 1, the same along x --
// so one thread per input pixel accumulates the 2 x 2 outputs it owns.  A
// block covers 32 input pixels of one row and up to 8 output channels; its 8
// warps split C_in (warp g takes ci = g, g + 8, ...) and add their partial
// sums through shared memory in warp order.  Per channel a lane loads its own
// column of the three rows (issued one channel ahead of the arithmetic); the
// left and right columns come from the neighbouring lanes by shuffles, and
// lanes 0 and 31 load the two columns beyond the span.
// The weights of the block's output channels are staged in shared memory 64
// input channels at a time; a (ci, co) pair's 16 taps are four 16-byte
// broadcast reads.
constexpr int kDeconvWarps = 8;
constexpr int kDeconvChunk = 64;  // input channels per staged weight chunk

template <typename Ti, typename To>
__global__ void __launch_bounds__(32 * kDeconvWarps) deconv4s2_kernel(
    const Ti* __restrict__ x, const float* __restrict__ w, const float* __restrict__ bias,
    const float* __restrict__ alpha, To* __restrict__ y, int layout, int N, int CI, int CO, int H,
    int W, int act) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    constexpr int CB = kDeconvCoBlock;
    extern __shared__ float4 dsm[];  // weight chunk [ci][j][4] float4, then partial sums
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_x = (W + 31) / 32;
    const int a = (blockIdx.x / tiles_x) % H, n = (blockIdx.x / tiles_x) / H;
    const int b0 = (blockIdx.x % tiles_x) * 32;
    const int b = b0 + lane;
    const int co0 = blockIdx.y * CB;
    const int nco = min(CB, CO - co0);
    const int rs = 4 * nco + 1;
    float4* sw = dsm;                                            // kDeconvChunk * nco * 4
    float* red = reinterpret_cast<float*>(dsm + kDeconvChunk * nco * 4);  // [warp][lane][rs]
    // this lane's own column and its halo column (lanes 0 and 31 only)
    const int hxc = lane == 0 ? b0 - 1 : b0 + 32;
    const bool own_ok = b < W;
    const bool halo_ok = (lane == 0 || lane == 31) && hxc >= 0 && hxc < W;
    bool row_ok[3];
#pragma unroll
    for (int dy = 0; dy < 3; ++dy) row_ok[dy] = a - 1 + dy >= 0 && a - 1 + dy < H;
    // element strides: along a row, from one channel to the next, between rows
    const int64_t sx = layout == ACNN_NHWC ? CI : 1;
    const int64_t sc = layout == ACNN_NHWC ? 1 : (int64_t)H * W;
    const int64_t sy = layout == ACNN_NHWC ? (int64_t)W * CI : W;
    const Ti* xrow = x + act_index(layout, CI, H, W, n, 0, a - 1, 0);  // row a - 1, channel 0
    auto load = [&](int ci, float (&own)[3], float (&halo)[3]) {
#pragma unroll
        for (int dy = 0; dy < 3; ++dy) {
            const Ti* r = xrow + dy * sy + ci * sc;
            own[dy] = (row_ok[dy] && own_ok) ? to_f32(r[b * sx]) : 0.0f;
            halo[dy] = (row_ok[dy] && halo_ok) ? to_f32(r[hxc * sx]) : 0.0f;
        }
    };
    float acc[2][2][CB];
#pragma unroll
    for (int py = 0; py < 2; ++py)
#pragma unroll
        for (int px = 0; px < 2; ++px)
#pragma unroll
            for (int j = 0; j < CB; ++j) acc[py][px][j] = 0.0f;
    float own[3] = {0.0f, 0.0f, 0.0f}, halo[3] = {0.0f, 0.0f, 0.0f};
    if (warp < CI) load(warp, own, halo);
    for (int c0 = 0; c0 < CI; c0 += kDeconvChunk) {
        const int nc = min(kDeconvChunk, CI - c0);
        __syncthreads();  // the previous chunk is consumed
        for (int i = threadIdx.x; i < nc * nco * 4; i += 32 * kDeconvWarps) {
            const int cc = i / (nco * 4), r = i - cc * nco * 4;  // r = j * 4 + ky
            sw[i] = __ldg(reinterpret_cast<const float4*>(w + ((long long)(c0 + cc) * CO + co0) * 16) + r);
        }
        __syncthreads();
        for (int cc = warp; cc < nc; cc += kDeconvWarps) {
            const int ci = c0 + cc;
            float own_n[3] = {0.0f, 0.0f, 0.0f}, halo_n[3] = {0.0f, 0.0f, 0.0f};
            if (ci + kDeconvWarps < CI) load(ci + kDeconvWarps, own_n, halo_n);
            float nb[3][3];  // x at rows a-1..a+1, cols b-1..b+1 (zero outside)
#pragma unroll
            for (int dy = 0; dy < 3; ++dy) {
                const float left = __shfl_up_sync(0xffffffffu, own[dy], 1);
                const float right = __shfl_down_sync(0xffffffffu, own[dy], 1);
                nb[dy][0] = lane == 0 ? halo[dy] : left;
                nb[dy][1] = own[dy];
                nb[dy][2] = lane == 31 ? halo[dy] : right;
            }
            const float4* wc = sw + cc * nco * 4;
#pragma unroll
            for (int j = 0; j < CB; ++j) {
                if (j >= nco) break;
                float wt[4][4];  // [ky][kx]
#pragma unroll
                for (int ky = 0; ky < 4; ++ky) {
                    const float4 v = wc[j * 4 + ky];
                    wt[ky][0] = v.x, wt[ky][1] = v.y, wt[ky][2] = v.z, wt[ky][3] = v.w;
                }
#pragma unroll
                for (int py = 0; py < 2; ++py)
#pragma unroll
                    for (int px = 0; px < 2; ++px)
#pragma unroll
                        for (int ty = 0; ty < 2; ++ty)
#pragma unroll
                            for (int tx = 0; tx < 2; ++tx) {
                                // py = 0: (ky, row) = (1, a), (3, a-1); py = 1: (0, a+1), (2, a)
                                const int ky = py == 0 ? 1 + 2 * ty : 2 * ty;
                                const int dy = py == 0 ? 1 - ty : 2 - ty;
                                const int kx = px == 0 ? 1 + 2 * tx : 2 * tx;
                                const int dx = px == 0 ? 1 - tx : 2 - tx;
                                acc[py][px][j] = fmaf(nb[dy][dx], wt[ky][kx], acc[py][px][j]);
                            }
            }
#pragma unroll
            for (int dy = 0; dy < 3; ++dy) {
                own[dy] = own_n[dy];
                halo[dy] = halo_n[dy];
            }
        }
    }
    float* mine = red + ((size_t)warp * 32 + lane) * rs;
#pragma unroll
    for (int py = 0; py < 2; ++py)
#pragma unroll
        for (int px = 0; px < 2; ++px)
#pragma unroll
            for (int j = 0; j < CB; ++j)
                if (j < nco) mine[(py * 2 + px) * nco + j] = acc[py][px][j];
    __syncthreads();
    // 32 pixels x 4 outputs x nco channels, summed over the warps in order
    const int OH = 2 * H, OW = 2 * W;
    for (int i = threadIdx.x; i < 32 * 4 * nco; i += 32 * kDeconvWarps) {
        const int l = i / (4 * nco), r = i - l * 4 * nco;
        const int pp = r / nco, j = r - pp * nco;
        const int bb = b0 + l;
        if (bb >= W) continue;
        float v = bias ? bias[co0 + j] : 0.0f;
        for (int g = 0; g < kDeconvWarps; ++g) v += red[((size_t)g * 32 + l) * rs + r];
        const int oy = 2 * a + (pp >> 1), ox = 2 * bb + (pp & 1);
        const float al = (act == ACNN_ACT_PRELU) ? alpha[co0 + j] : 0.0f;
        y[act_index(layout, CO, OH, OW, n, co0 + j, oy, ox)] = from_f32<To>(apply_act(act, v, al));
    }
}

template <typename Ti, typename To>
__global__ void __launch_bounds__(kThreads) deconv_kernel(
    const Ti* __restrict__ x, const float* __restrict__ w, const float* __restrict__ bias,
    const float* __restrict__ alpha, To* __restrict__ y, int layout, int N, int CI, int CO,
    int H, int W, int OH, int OW, int K, int S, int P, int act) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const long long pix = (long long)N * OH * OW;
    const int co_blocks = (CO + kDeconvCoBlock - 1) / kDeconvCoBlock;
    const long long total = pix * co_blocks;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < (uint32_t)total;
         i += gridDim.x * blockDim.x) {
        int cb = (int)(i / (uint32_t)pix);
        uint32_t q = i - (uint32_t)cb * (uint32_t)pix;
        int ox = (int)(q % OW);
        q /= OW;
        int oy = (int)(q % OH);
        int n = (int)(q / OH);
        const int co0 = cb * kDeconvCoBlock;
        const int nco = min(kDeconvCoBlock, CO - co0);
        float acc[kDeconvCoBlock];
#pragma unroll
        for (int j = 0; j < kDeconvCoBlock; ++j)
            acc[j] = (bias && j < nco) ? bias[co0 + j] : 0.0f;
        for (int ky = 0; ky < K; ++ky) {
            int ty = oy + P - ky;
            if (ty < 0 || ty % S != 0) continue;
            int iy = ty / S;
            if (iy >= H) continue;
            for (int kx = 0; kx < K; ++kx) {
                int tx = ox + P - kx;
                if (tx < 0 || tx % S != 0) continue;
                int ix = tx / S;
                if (ix >= W) continue;
                for (int ci = 0; ci < CI; ++ci) {
                    float xv = to_f32(x[act_index(layout, CI, H, W, n, ci, iy, ix)]);
                    const float* wp = w + ((long long)ci * CO + co0) * K * K + ky * K + kx;
#pragma unroll
                    for (int j = 0; j < kDeconvCoBlock; ++j)
                        if (j < nco) acc[j] = fmaf(xv, __ldg(wp + (long long)j * K * K), acc[j]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kDeconvCoBlock; ++j)
            if (j < nco) {
                float al = (act == ACNN_ACT_PRELU) ? alpha[co0 + j] : 0.0f;
                y[act_index(layout, CO, OH, OW, n, co0 + j, oy, ox)] =
                    from_f32<To>(apply_act(act, acc[j], al));
            }
    }
}

// ----------------------------------------------------------------------------
// im2col pack for convs with few input channels (rtdetr_gpu.rs IM2COL_SRC:
// row m = output pixel, k = (ky, kx, ci), taps outside the input are zero),
// padded with zeros from K = kh*kw*C to Kp (a multiple of 8) so that rows are
// 16-byte aligned for the tensor-core GEMM.  Values are copied as raw 16-bit
// patterns.
// One block per (image, output row, segment of TP output pixels): the KH input
// rows the segment reads -- columns [ox0*S - P, ox0*S - P + RW) with
// RW = (TP - 1)*S + KW, every channel -- are staged in shared memory as
// [ky][px][c], zero outside the image, so that packed element k of output
// pixel px sits at staged offset px*S*C + (k / (KW*C))*RL + k % (KW*C)
// (RL = RW*C).  That offset minus px*S*C depends on k alone and is tabulated
// once per block; consecutive threads then write consecutive 16-byte chunks
// (8 k) of the segment's packed rows.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) im2col_pack_kernel(
    const uint16_t* __restrict__ x, uint16_t* __restrict__ a, int layout, int H, int W, int C,
    int KH, int KW, int S, int P, int OH, int OW, int Kp, int TP, int segs) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    extern __shared__ __align__(16) uint16_t st[];
    const int RW = (TP - 1) * S + KW;  // staged pixels per input row
    const int RL = RW * C;             // staged values per input row
    int* tab = reinterpret_cast<int*>(st + ((KH * RL + 1) & ~1));  // [Kp] staged offsets
    int b = blockIdx.x;
    const int seg = b % segs;
    b /= segs;
    const int oy = b % OH, n = b / OH;
    const int ox0 = seg * TP;
    const int np = min(TP, OW - ox0);
    const int ix0 = ox0 * S - P, iy0 = oy * S - P;
    const int K = KH * KW * C, KWC = KW * C;
    for (int k = threadIdx.x; k < Kp; k += blockDim.x)
        tab[k] = k < K ? (k / KWC) * RL + k % KWC : -1;
    // staged values [lo, hi) of a row lie inside the image (pixels 0..W-1)
    const int lo = max(0, -ix0) * C, hi = max(0, min(RW, W - ix0)) * C;
    for (int ky = 0; ky < KH; ++ky) {
        const int iy = iy0 + ky;
        uint16_t* row = st + ky * RL;
        if (iy < 0 || iy >= H) {
            for (int e = threadIdx.x; e < RL; e += blockDim.x) row[e] = 0;
        } else if (layout == ACNN_NHWC) {
            // the row's staged pixels are contiguous in an NHWC image; eight
            // loads per thread are issued before their stores
            const long long base = ((long long)n * H + iy) * W * C + (long long)ix0 * C;
            constexpr int U = 8;
            for (int e0 = threadIdx.x; e0 < RL; e0 += U * kThreads) {
                uint16_t v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int e = e0 + u * kThreads;
                    v[u] = (e >= lo && e < hi) ? x[base + e] : (uint16_t)0;
                }
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (e0 + u * kThreads < RL) row[e0 + u * kThreads] = v[u];
            }
        } else {
            // NCHW: one channel plane at a time, pixels fastest (coalesced)
            const long long plane = (long long)H * W;
            const uint16_t* xr = x + ((long long)n * C * H + iy) * W;
            for (int c = 0; c < C; ++c, xr += plane)
                for (int px = threadIdx.x; px < RW; px += blockDim.x) {
                    const int ix = ix0 + px;
                    row[px * C + c] = (ix >= 0 && ix < W) ? xr[ix] : (uint16_t)0;
                }
        }
    }
    __syncthreads();
    const int KG = Kp / 8;
    uint16_t* out = a + ((long long)(n * OH + oy) * OW + ox0) * Kp;
    if (blockDim.x % KG == 0) {
        // a thread's k-group g is the same on every iteration: its eight
        // staged offsets are read from the table once
        const int g = threadIdx.x % KG;
        int o8[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) o8[jj] = tab[g * 8 + jj];
        for (int px = threadIdx.x / KG; px < np; px += blockDim.x / KG) {
            const uint16_t* src = st + px * S * C;
            Vec<uint16_t, 8> v;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) v.v[jj] = o8[jj] >= 0 ? src[o8[jj]] : (uint16_t)0;
            *reinterpret_cast<Vec<uint16_t, 8>*>(out + (long long)px * Kp + g * 8) = v;
        }
    } else {
        for (int j = threadIdx.x; j < np * KG; j += blockDim.x) {
            const int px = j / KG, g = j - px * KG;
            const uint16_t* src = st + px * S * C;
            const int* t8 = tab + g * 8;
            Vec<uint16_t, 8> v;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int o = t8[jj];
                v.v[jj] = o >= 0 ? src[o] : (uint16_t)0;
            }
            *reinterpret_cast<Vec<uint16_t, 8>*>(out + (long long)px * Kp + g * 8) = v;
        }
    }
}

// Weights to the packed K order: wp[co][k], k = (ky, kx, ci), zero for k >= K;
// from OHWI (NHWC convs) or OIHW (NCHW convs).
__global__ void __launch_bounds__(kThreads) weight_pack_kernel(
    const uint16_t* __restrict__ w, uint16_t* __restrict__ wp, int layout, int C_out, int C,
    int KH, int KW, int Kp) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    const int K = KH * KW * C;
    const uint32_t total = (uint32_t)C_out * Kp;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += gridDim.x * blockDim.x) {
        const int co = (int)(i / Kp), k = (int)(i - (uint32_t)co * Kp);
        uint16_t val = 0;
        if (k < K) {
            const int tap = k / C, ci = k - tap * C;
            const int ky = tap / KW, kx = tap - ky * KW;
            val = layout == ACNN_NHWC ? w[(((long long)co * KH + ky) * KW + kx) * C + ci]
                                      : w[(((long long)co * C + ci) * KH + ky) * KW + kx];
        }
        wp[i] = val;
    }
}

// ----------------------------------------------------------------------------
// NCHW -> NHWC transpose of 16-bit elements through a 32x32 shared tile:
// per image, [C][HW] -> [HW][C].  Reads and writes are both coalesced.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) transpose_kernel(const uint16_t* __restrict__ x,
                                                         uint16_t* __restrict__ y, int C, int HW) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    __shared__ uint16_t tile[32][33];
    const int n = blockIdx.z;
    const int c0 = blockIdx.y * 32, p0 = blockIdx.x * 32;
    const uint16_t* xi = x + (long long)n * C * HW;
    uint16_t* yi = y + (long long)n * C * HW;
    int c = c0 + threadIdx.y, p = p0 + threadIdx.x;
    if (c < C && p < HW) tile[threadIdx.y][threadIdx.x] = xi[(long long)c * HW + p];
    __syncthreads();
    c = c0 + threadIdx.x;
    p = p0 + threadIdx.y;
    if (c < C && p < HW) yi[(long long)p * C + c] = tile[threadIdx.x][threadIdx.y];
}

// The same transpose for even C and HW through a 64 x 64 tile, 4-byte
// accesses: each warp reads 128-byte channel-row segments (2 pixels a lane)
// and writes 128-byte pixel-row segments (2 channels a lane).
__global__ void __launch_bounds__(256) transpose64_kernel(const uint16_t* __restrict__ x,
                                                          uint16_t* __restrict__ y, int C,
                                                          int HW) {
    griddep_wait();  // inputs may come from the previous kernel on the stream
    // [channel][pixel], 32 words a row; the 4-byte pixel pair w of row r is
    // stored at word w ^ (r / 2), so that both the row-wise writes (one row,
    // 32 words) and the column-wise reads (rows 2l and 2l + 1 for lane l, one
    // word each) touch 32 distinct banks
    __shared__ uint32_t tile[64][32];
    const int n = blockIdx.z;
    const int c0 = blockIdx.y * 64, p0 = blockIdx.x * 64;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint16_t* xi = x + (long long)n * C * HW;
    uint16_t* yi = y + (long long)n * C * HW;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int cc = warp * 8 + r, c = c0 + cc, p = p0 + 2 * lane;
        uint32_t v = 0;
        if (c < C && p < HW) v = *reinterpret_cast<const uint32_t*>(xi + (long long)c * HW + p);
        tile[cc][lane ^ ((cc >> 1) & 31)] = v;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int pp = warp * 8 + r, p = p0 + pp, c = c0 + 2 * lane;
        if (p < HW && c < C) {
            // rows 2 lane and 2 lane + 1 both carry the swizzle lane
            const int wd = (pp >> 1) ^ lane, sh = (pp & 1) * 16;
            const uint32_t v = ((tile[2 * lane][wd] >> sh) & 0xffffu) |
                               (((tile[2 * lane + 1][wd] >> sh) & 0xffffu) << 16);
            *reinterpret_cast<uint32_t*>(yi + (long long)p * C + c) = v;
        }
    }
}

template <typename T> int vec_for(int elems) {
    constexpr int V = 16 / sizeof(T);
    return elems % V == 0 ? V : 1;
}

template <typename T>
cudaError_t pool_typed(int kind, int n, int h, int w, int c, int k, int stride, int pad,
                       int layout, const void* x, void* y, cudaStream_t s) {
    int oh = (h + 2 * pad - k) / stride + 1, ow = (w + 2 * pad - k) / stride + 1;
    const T* xt = static_cast<const T*>(x);
    T* yt = static_cast<T*>(y);
    if (layout == ACNN_NHWC) {
        constexpr int V = 16 / sizeof(T);
        const long long rows = (long long)n * oh;
        const int row_vecs = c % V == 0 ? ow * (c / V) : 0;
        if (c % V == 0 && kind == ACNN_POOL_MAX && k == 3 && stride == 2 && pad == 1 &&
            rows <= 0x7fffffffLL && (row_vecs + kThreads - 1) / kThreads <= 65535) {
            dim3 g((unsigned)rows, (row_vecs + kThreads - 1) / kThreads);
            launch_pdl(maxpool3s2_rows_kernel<T, V>, g, kThreads, 0, s, xt, yt, h, w, c, oh, ow);
        } else if (c % V == 0 && kind == ACNN_POOL_AVG && k == 2 && stride == 2 && pad == 0 &&
                   rows <= 0x7fffffffLL && (row_vecs + 2 * kThreads - 1) / (2 * kThreads) <= 65535) {
            dim3 g((unsigned)rows, (row_vecs + 2 * kThreads - 1) / (2 * kThreads));
            launch_pdl(avgpool2_rows_kernel<T, V, 2>, g, kThreads, 0, s, xt, yt, h, w, c, oh, ow);
        } else if (c % V == 0 && kind == ACNN_POOL_MAX && k == 3 && stride == 2 && pad == 1) {
            long long work = (long long)n * oh * ow * (c / V);
            launch_pdl(maxpool3s2_nhwc_kernel<T, V>, grid_occ(maxpool3s2_nhwc_kernel<T, V>, work, kThreads), kThreads, 0, s, 
                xt, yt, n, h, w, c, oh, ow);
        } else if (c % V == 0) {
            long long work = (long long)n * oh * ow * (c / V);
            launch_pdl(pool_nhwc_kernel<T, V>, grid_occ(pool_nhwc_kernel<T, V>, work, kThreads), kThreads, 0, s, 
                xt, yt, kind, n, h, w, c, oh, ow, k, stride, pad);
        } else {
            long long work = (long long)n * oh * ow * c;
            launch_pdl(pool_nhwc_kernel<T, 1>, grid_occ(pool_nhwc_kernel<T, 1>, work, kThreads), kThreads, 0, s, 
                xt, yt, kind, n, h, w, c, oh, ow, k, stride, pad);
        }
    } else {
        long long work = (long long)n * c * oh * ow;
        launch_pdl(pool_nchw_kernel<T>, grid_occ(pool_nchw_kernel<T>, work, kThreads), kThreads, 0, s, 
            xt, yt, kind, n, c, h, w, oh, ow, k, stride, pad);
    }
    return cudaGetLastError();
}

template <typename Ti, typename To>
cudaError_t resize_typed(int mode, int n, int c, int h, int w, int oh, int ow, int layout,
                         const void* x, void* y, cudaStream_t s) {
    const Ti* xt = static_cast<const Ti*>(x);
    To* yt = static_cast<To*>(y);
    float sy = (float)h / (float)oh, sx = (float)w / (float)ow;
    if (layout == ACNN_NHWC) {
        constexpr int V = (16 / sizeof(Ti)) < (16 / sizeof(To)) ? (16 / sizeof(Ti)) : (16 / sizeof(To));
        if constexpr (sizeof(Ti) == sizeof(To)) {
            const long long in_rows = (long long)n * h;
            const int in_row_vecs = c % V == 0 ? w * (c / V) : 0;
            if (mode == ACNN_RESIZE_NEAREST && oh == 2 * h && ow == 2 * w && c % V == 0 &&
                in_rows <= 0x7fffffffLL && (in_row_vecs + 2 * kThreads - 1) / (2 * kThreads) <= 65535) {
                dim3 g((unsigned)in_rows, (in_row_vecs + 2 * kThreads - 1) / (2 * kThreads));
                launch_pdl(up2_rows_kernel<Ti, V, 2>, g, kThreads, 0, s, xt, reinterpret_cast<Ti*>(yt), h, w, c);
                return cudaGetLastError();
            }
            if (mode == ACNN_RESIZE_NEAREST && oh == 2 * h && ow == 2 * w && c % V == 0) {
                long long work = (long long)n * h * w * (c / V);
                launch_pdl(up2_nhwc_kernel<Ti, V>, grid_occ(up2_nhwc_kernel<Ti, V>, work, kThreads), kThreads, 0, s, 
                    xt, reinterpret_cast<Ti*>(yt), n, h, w, c);
                return cudaGetLastError();
            }
        }
        if (c % V == 0) {
            long long work = (long long)n * oh * ow * (c / V);
            launch_pdl(resize_nhwc_kernel<Ti, To, V>, grid_occ(resize_nhwc_kernel<Ti, To, V>, work, kThreads), kThreads, 0, s, 
                xt, yt, mode, n, h, w, c, oh, ow, sy, sx);
        } else {
            long long work = (long long)n * oh * ow * c;
            launch_pdl(resize_nhwc_kernel<Ti, To, 1>, grid_occ(resize_nhwc_kernel<Ti, To, 1>, work, kThreads), kThreads, 0, s, 
                xt, yt, mode, n, h, w, c, oh, ow, sy, sx);
        }
    } else {
        constexpr int VO = 16 / sizeof(To);
        const long long rows = (long long)n * c * oh;
        const int chunks = (ow / VO + kThreads - 1) / kThreads;
        const long long ublocks = (long long)n * c * ((oh + kUpRows - 1) / kUpRows);
        // eight output rows read at most kUpSpan source rows when the height
        // grows 4x or more: (8 - 1) / 4 + 2 = 3.75
        if (mode == ACNN_RESIZE_BILINEAR && oh >= 4 * h && ow % VO == 0 && ublocks <= 0x7fffffffLL &&
            chunks <= 65535) {
            launch_pdl(resize_nchw_up_kernel<Ti, To, VO>, dim3((unsigned)ublocks, chunks), kThreads, 0,
                       s, xt, yt, h, w, oh, ow, sy, sx);
        } else if (ow % VO == 0 && rows <= 0x7fffffffLL && chunks <= 65535) {
            // whole 16-byte output vectors per row (rows start aligned)
            launch_pdl(resize_nchw_rows_kernel<Ti, To, VO>, dim3((unsigned)rows, chunks), kThreads, 0,
                       s, xt, yt, mode, h, w, oh, ow, sy, sx);
        } else {
            long long work = (long long)n * c * oh * ow;
            launch_pdl(resize_nchw_kernel<Ti, To>, grid_occ(resize_nchw_kernel<Ti, To>, work, kThreads), kThreads, 0, s,
                xt, yt, mode, n * c, h, w, oh, ow, sy, sx);
        }
    }
    return cudaGetLastError();
}

template <typename To>
cudaError_t resize_from(int in_dtype, int mode, int n, int c, int h, int w, int oh, int ow,
                        int layout, const void* x, void* y, cudaStream_t s) {
    switch (in_dtype) {
    case ACNN_F32: return resize_typed<float, To>(mode, n, c, h, w, oh, ow, layout, x, y, s);
    case ACNN_F16: return resize_typed<__half, To>(mode, n, c, h, w, oh, ow, layout, x, y, s);
    default: return resize_typed<__nv_bfloat16, To>(mode, n, c, h, w, oh, ow, layout, x, y, s);
    }
}

template <typename T>
cudaError_t concat_typed(int n, int h, int w, int ca, int cb, int layout, const void* a,
                         const void* b, void* y, cudaStream_t s) {
    long long runs;
    long long ra, rb;
    if (layout == ACNN_NHWC) {
        runs = (long long)n * h * w;
        ra = ca;
        rb = cb;
    } else {
        runs = n;
        ra = (long long)ca * h * w;
        rb = (long long)cb * h * w;
    }
    constexpr int V = 16 / sizeof(T);
    const T* at = static_cast<const T*>(a);
    const T* bt = static_cast<const T*>(b);
    T* yt = static_cast<T*>(y);
    // one block per 4 x 256 vectors (the index stays below 2^32: the host checks it)
    auto blocks = [](long long work) { return (unsigned)((work + 4LL * kThreads - 1) / (4LL * kThreads)); };
    if (ra % V == 0 && rb % V == 0) {
        const long long work = runs * ((ra + rb) / V);
        launch_pdl(concat_kernel<T, V>, blocks(work), kThreads, 0, s, at, bt, yt, runs, (int)ra, (int)rb);
    } else {
        const long long work = runs * (ra + rb);
        launch_pdl(concat_kernel<T, 1>, blocks(work), kThreads, 0, s, at, bt, yt, runs, (int)ra, (int)rb);
    }
    return cudaGetLastError();
}

template <typename Ti, typename To>
cudaError_t deconv_typed(const acnn_conv_desc& d, int oh, int ow, const void* x, const float* w,
                         const float* bias, const float* alpha, int act, void* y,
                         cudaStream_t s) {
    if (d.kh == 4 && d.kw == 4 && d.stride == 2 && d.pad == 1) {
        const long long rows = (long long)d.n * d.h * ((d.w + 31) / 32);
        const int cob = (d.c_out + kDeconvCoBlock - 1) / kDeconvCoBlock;
        if (rows <= 0x7fffffffLL && cob <= 65535) {
            const int nco = d.c_out < kDeconvCoBlock ? d.c_out : kDeconvCoBlock;
            auto smem_for = [](int c) {  // weight chunk + partial sums
                return (size_t)kDeconvChunk * c * 64 +
                       (size_t)kDeconvWarps * 32 * (4 * c + 1) * sizeof(float);
            };
            const size_t smem = smem_for(nco);
            if (ensure_smem_optin(reinterpret_cast<const void*>(deconv4s2_kernel<Ti, To>),
                                  smem_for(kDeconvCoBlock)) != ACNN_OK)
                return cudaErrorInvalidValue;
            launch_pdl(deconv4s2_kernel<Ti, To>, dim3((unsigned)rows, cob), 32 * kDeconvWarps,
                       smem, s, static_cast<const Ti*>(x), w, bias, alpha, static_cast<To*>(y),
                       d.layout, d.n, d.c_in, d.c_out, d.h, d.w, act);
            return cudaGetLastError();
        }
    }
    long long work = (long long)d.n * oh * ow *
                     ((d.c_out + kDeconvCoBlock - 1) / kDeconvCoBlock);
    launch_pdl(deconv_kernel<Ti, To>, grid_occ(deconv_kernel<Ti, To>, work, kThreads), kThreads, 0, s, 
        static_cast<const Ti*>(x), w, bias, alpha, static_cast<To*>(y), d.layout, d.n, d.c_in,
        d.c_out, d.h, d.w, oh, ow, d.kh, d.stride, d.pad, act);
    return cudaGetLastError();
}

template <typename Ti>
cudaError_t deconv_from(int out_dtype, const acnn_conv_desc& d, int oh, int ow, const void* x,
                        const float* w, const float* bias, const float* alpha, int act, void* y,
                        cudaStream_t s) {
    switch (out_dtype) {
    case ACNN_F32: return deconv_typed<Ti, float>(d, oh, ow, x, w, bias, alpha, act, y, s);
    case ACNN_F16: return deconv_typed<Ti, __half>(d, oh, ow, x, w, bias, alpha, act, y, s);
    default: return deconv_typed<Ti, __nv_bfloat16>(d, oh, ow, x, w, bias, alpha, act, y, s);
    }
}

}  // namespace

cudaError_t launch_pool2d(int kind, int n, int h, int w, int c, int k, int stride, int pad,
                          int layout, int dtype, const void* x, void* y, cudaStream_t s) {
    switch (dtype) {
    case ACNN_F32: return pool_typed<float>(kind, n, h, w, c, k, stride, pad, layout, x, y, s);
    case ACNN_F16: return pool_typed<__half>(kind, n, h, w, c, k, stride, pad, layout, x, y, s);
    default: return pool_typed<__nv_bfloat16>(kind, n, h, w, c, k, stride, pad, layout, x, y, s);
    }
}

cudaError_t launch_resize2d(int mode, int n, int c, int h, int w, int oh, int ow, int layout,
                            int in_dtype, int out_dtype, const void* x, void* y, cudaStream_t s) {
    switch (out_dtype) {
    case ACNN_F32: return resize_from<float>(in_dtype, mode, n, c, h, w, oh, ow, layout, x, y, s);
    case ACNN_F16: return resize_from<__half>(in_dtype, mode, n, c, h, w, oh, ow, layout, x, y, s);
    default: return resize_from<__nv_bfloat16>(in_dtype, mode, n, c, h, w, oh, ow, layout, x, y, s);
    }
}

cudaError_t launch_concat(int n, int h, int w, int ca, int cb, int layout, int dtype,
                          const void* a, const void* b, void* y, cudaStream_t s) {
    if (dtype == ACNN_F32) return concat_typed<float>(n, h, w, ca, cb, layout, a, b, y, s);
    return concat_typed<uint16_t>(n, h, w, ca, cb, layout, a, b, y, s);  // 2-byte copy
}

cudaError_t launch_deconv2d(const acnn_conv_desc& d, int oh, int ow, const void* x,
                            const float* w, const float* bias, const float* alpha, int act,
                            int out_dtype, void* y, cudaStream_t s) {
    switch (d.dtype) {
    case ACNN_F32: return deconv_from<float>(out_dtype, d, oh, ow, x, w, bias, alpha, act, y, s);
    case ACNN_F16: return deconv_from<__half>(out_dtype, d, oh, ow, x, w, bias, alpha, act, y, s);
    default: return deconv_from<__nv_bfloat16>(out_dtype, d, oh, ow, x, w, bias, alpha, act, y, s);
    }
}

cudaError_t launch_prep_quarter(int h, int w, const uint8_t* rgba0, const uint8_t* rgba1,
                                float t, int out_dtype, void* y, cudaStream_t s) {
    long long work = (long long)(h / 4) * (w / 4);
    const uint32_t* f0 = reinterpret_cast<const uint32_t*>(rgba0);
    const uint32_t* f1 = reinterpret_cast<const uint32_t*>(rgba1);
    int g = grid_for(work, kThreads);
    switch (out_dtype) {
    case ACNN_F32:
        launch_pdl(prep_quarter_kernel<float>, g, kThreads, 0, s, f0, f1, static_cast<float*>(y), h, w, t);
        break;
    case ACNN_F16:
        launch_pdl(prep_quarter_kernel<__half>, g, kThreads, 0, s, f0, f1, static_cast<__half*>(y), h, w, t);
        break;
    default:
        launch_pdl(prep_quarter_kernel<__nv_bfloat16>, g, kThreads, 0, s, 
            f0, f1, static_cast<__nv_bfloat16*>(y), h, w, t);
        break;
    }
    return cudaGetLastError();
}

cudaError_t launch_im2col_pack(const acnn_conv_desc& d, int oh, int ow, int kp, const void* x,
                               void* a, const void* w, void* wp, cudaStream_t s) {
    // segment width: a whole output row, halved until the staged rows and the
    // offset table take at most 32 KB of shared memory (tp = 1 needs at most
    // 3 KB: K <= 512)
    auto staged = [&](int tp) {
        return (size_t)((d.kh * ((tp - 1) * d.stride + d.kw) * d.c_in + 1) & ~1) * 2 +
               (size_t)kp * 4;
    };
    int tp = ow;
    while (tp > 1 && staged(tp) > 32768) tp = (tp + 1) / 2;
    // and short enough that the launch has at least four blocks per SM (the
    // frame input: 136 output rows would otherwise give 136 blocks)
    while (tp > 16 && (long long)d.n * oh * ((ow + tp - 1) / tp) < 4LL * sm_count())
        tp = (tp + 1) / 2;
    const int segs = (ow + tp - 1) / tp;
    const long long blocks = (long long)d.n * oh * segs;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    launch_pdl(im2col_pack_kernel, (unsigned)blocks, kThreads, staged(tp), s, 
        static_cast<const uint16_t*>(x), static_cast<uint16_t*>(a), d.layout, d.h, d.w, d.c_in,
        d.kh, d.kw, d.stride, d.pad, oh, ow, kp, tp, segs);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !w) return e;  // no w: the weights are prepacked
    return launch_weight_pack(d, kp, w, wp, s);
}

cudaError_t launch_deconv_gemm_weights(int dtype, const float* w, const float* bias,
                                       const float* alpha, void* wg, float* bg, float* ag, int ci,
                                       int co, int co4, cudaStream_t s) {
    const long long work = (long long)co4 * 9 * ci;
    if (dtype == ACNN_BF16)
        launch_pdl(deconv_gemm_weights_kernel<__nv_bfloat16>,
                   grid_occ(deconv_gemm_weights_kernel<__nv_bfloat16>, work, kThreads), kThreads, 0, s,
                   w, bias, alpha, static_cast<__nv_bfloat16*>(wg), bg, ag, ci, co, co4);
    else
        launch_pdl(deconv_gemm_weights_kernel<__half>,
                   grid_occ(deconv_gemm_weights_kernel<__half>, work, kThreads), kThreads, 0, s, w,
                   bias, alpha, static_cast<__half*>(wg), bg, ag, ci, co, co4);
    return cudaGetLastError();
}

cudaError_t launch_deconv_shuffle(int dtype, const void* ys, void* y, int layout, int n, int h,
                                  int w, int co, int co4, cudaStream_t s) {
    const long long work = (long long)n * co * 4 * h * w;
    if (dtype == ACNN_BF16)
        launch_pdl(deconv_shuffle_kernel<__nv_bfloat16>,
                   grid_occ(deconv_shuffle_kernel<__nv_bfloat16>, work, kThreads), kThreads, 0, s,
                   static_cast<const __nv_bfloat16*>(ys), static_cast<__nv_bfloat16*>(y), layout, n, h,
                   w, co, co4);
    else
        launch_pdl(deconv_shuffle_kernel<__half>, grid_occ(deconv_shuffle_kernel<__half>, work, kThreads),
                   kThreads, 0, s, static_cast<const __half*>(ys), static_cast<__half*>(y), layout, n,
                   h, w, co, co4);
    return cudaGetLastError();
}

cudaError_t launch_weight_pack(const acnn_conv_desc& d, int kp, const void* w, void* wp,
                               cudaStream_t s) {
    launch_pdl(weight_pack_kernel, grid_occ(weight_pack_kernel, (long long)d.c_out * kp, kThreads), kThreads, 0, s,
        static_cast<const uint16_t*>(w), static_cast<uint16_t*>(wp), d.layout, d.c_out, d.c_in,
        d.kh, d.kw, kp);
    return cudaGetLastError();
}

cudaError_t launch_nchw_to_nhwc(int n, int c, int hw, int elem_bytes, const void* x, void* y,
                                cudaStream_t s) {
    if (elem_bytes != 2) return cudaErrorInvalidValue;
    if (c % 2 == 0 && hw % 2 == 0 && (hw + 63) / 64 <= 0x7fffffff && (c + 63) / 64 <= 65535 &&
        n <= 65535) {
        dim3 grid((hw + 63) / 64, (c + 63) / 64, n);
        launch_pdl(transpose64_kernel, grid, dim3(256), 0, s, static_cast<const uint16_t*>(x),
                   static_cast<uint16_t*>(y), c, hw);
        return cudaGetLastError();
    }
    dim3 grid((hw + 31) / 32, (c + 31) / 32, n), block(32, 32);
    launch_pdl(transpose_kernel, grid, block, 0, s, static_cast<const uint16_t*>(x),
                                            static_cast<uint16_t*>(y), c, hw);
    return cudaGetLastError();
}

}  // namespace acnn
