// abi.cu -- the extern "C" entry points of libacnn (include/acnn.h).
//
// Each entry point validates its arguments on the host, picks a kernel and
// enqueues it on the caller's stream.  A rejected call launches nothing.
// Device pointers are plain addresses owned by the caller; the library
// allocates no device memory.
#include <cuda_runtime.h>

#include <stdint.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "per_device.h"

namespace acnn {

// Status word the kernels set when a bounded pipeline wait expires.
__device__ int g_device_status = 0;

namespace {
std::atomic<long long> g_wait_budget{0};
constexpr int kMaxDevices = 64;
// Per-device values looked up once (static storage: zero until set).  Read
// with an acquire load; the first caller on a device fills them in.
std::atomic<int*> g_status_ptr[kMaxDevices];
std::atomic<int> g_sm_count[kMaxDevices];
std::mutex g_mu;

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    return dev;
}
}  // namespace

int sm_count() {
    const int dev = current_device();
    int n = g_sm_count[dev].load(std::memory_order_acquire);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
        g_sm_count[dev].store(n, std::memory_order_release);
    }
    return n;
}

// cudaFuncSetAttribute acts on the current device only, so the dynamic
// shared-memory opt-in of each kernel is recorded per (kernel, device): a
// process that drives several GPUs opts in on each before its first launch
// there.  Thread-safe; a larger request than the one recorded is set again.
int ensure_smem_optin(const void* kernel, size_t bytes) {
    static PerDeviceSizes done;
    const bool ok = done.ensure(kernel, current_device(), bytes, [&] {
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)bytes) == cudaSuccess;
    });
    return ok ? ACNN_OK : ACNN_ERR_CUDA;
}

int occupancy_blocks(const void* kernel, int threads, size_t smem) {
    struct Entry {
        const void* k;
        int threads;
        size_t smem;
        int dev;
        int blocks;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    const int dev = current_device();
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : cache)
        if (e.k == kernel && e.threads == threads && e.smem == smem && e.dev == dev) return e.blocks;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess ||
        n <= 0)
        n = 1;
    cache.push_back(Entry{kernel, threads, smem, dev, n});
    return n;
}

int* device_status_ptr() {
    const int dev = current_device();
    int* p = g_status_ptr[dev].load(std::memory_order_acquire);
    if (p) return p;
    std::lock_guard<std::mutex> lk(g_mu);
    p = g_status_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
        void* q = nullptr;
        if (cudaGetSymbolAddress(&q, g_device_status) != cudaSuccess) return nullptr;
        p = static_cast<int*>(q);
        g_status_ptr[dev].store(p, std::memory_order_release);
    }
    return p;
}

long long wait_budget_polls() { return g_wait_budget.load(); }

}  // namespace acnn

using namespace acnn;

namespace {

inline bool valid_dtype(int t) { return t == ACNN_F32 || t == ACNN_F16 || t == ACNN_BF16; }
inline bool valid_layout(int l) { return l == ACNN_NHWC || l == ACNN_NCHW; }
inline size_t elem_size(int t) { return t == ACNN_F32 ? 4 : 2; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

inline int status_of(cudaError_t e) { return e == cudaSuccess ? ACNN_OK : ACNN_ERR_CUDA; }

constexpr long long kIndexLimit = (1ll << 31) - 1;

// Geometry checks shared by conv and deconv descriptors.
int check_desc(const acnn_conv_desc* d) {
    if (!d) return ACNN_ERR_NULL_POINTER;
    if (!valid_dtype(d->dtype) || !valid_layout(d->layout)) return ACNN_ERR_BAD_ENUM;
    if (d->n <= 0 || d->h <= 0 || d->w <= 0 || d->c_in <= 0 || d->c_out <= 0 || d->kh <= 0 ||
        d->kw <= 0 || d->stride <= 0 || d->pad < 0)
        return ACNN_ERR_BAD_GEOMETRY;
    return ACNN_OK;
}

int conv_out(const acnn_conv_desc* d, int* oh, int* ow) {
    const long long h = ((long long)d->h + 2ll * d->pad - d->kh) / d->stride + 1;
    const long long w = ((long long)d->w + 2ll * d->pad - d->kw) / d->stride + 1;
    if ((long long)d->h + 2ll * d->pad < d->kh || (long long)d->w + 2ll * d->pad < d->kw || h <= 0 ||
        w <= 0)
        return ACNN_ERR_BAD_GEOMETRY;
    *oh = (int)h;
    *ow = (int)w;
    return ACNN_OK;
}

// The tensor-core path with TMA loads of x itself: fp16/bf16, TMA-addressable
// channel strides (16-byte multiples), output rows of whole 16-byte vectors,
// square kernels whose corner offsets fit the im2col descriptor, and 32-bit
// pixel indices.
// Largest C_out of the tensor-core paths: the NHWC epilogue keeps a copy of
// the bias and PReLU alpha of every column in shared memory.
constexpr int kTensorMaxCout = 4096;

bool tensor_path_ok(const acnn_conv_desc* d, int oh, int ow) {
    if (d->dtype == ACNN_F32) return false;
    if (d->c_in % 8 != 0 || d->c_out % 8 != 0) return false;
    if (d->c_out > kTensorMaxCout) return false;  // the epilogue's shared bias copy
    if (d->kh != d->kw || d->kh > 8 || d->stride > 8 || d->pad > 64) return false;
    if (d->pad - (d->kh - 1) < -128) return false;
    const long long m = (long long)d->n * oh * ow;
    const long long in = (long long)d->n * d->h * d->w;
    return m <= kIndexLimit && in <= kIndexLimit && (long long)d->c_out * oh * ow <= kIndexLimit;
}

// Padded reduction length of the packed path: K = kh*kw*c_in rounded up to 8.
int packed_k(const acnn_conv_desc* d) { return (d->kh * d->kw * d->c_in + 7) / 8 * 8; }

// The packed tensor-core path, for the convs TMA cannot address (few or odd
// input channels, non-square kernels): an explicit im2col matrix with
// K = kh*kw*c_in padded to a multiple of 8 is built in the workspace and
// multiplied on the tensor cores as a 1x1 conv.  Used while K stays small
// (at most 512), where the packed matrix costs little next to the output.
bool packed_path_ok(const acnn_conv_desc* d, int oh, int ow) {
    if (d->dtype == ACNN_F32 || d->c_out % 8 != 0 || tensor_path_ok(d, oh, ow)) return false;
    if (d->c_out > kTensorMaxCout) return false;
    const long long m = (long long)d->n * oh * ow;
    return packed_k(d) <= 512 && m * packed_k(d) <= kIndexLimit &&
           (long long)d->n * d->h * d->w * d->c_in <= kIndexLimit &&
           (long long)d->c_out * oh * ow <= kIndexLimit;
}

size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

// How a conv reaches the tensor cores: the path, the workspace it requires
// (staging copies: NHWC x and OHWI w for NCHW convs, or the packed im2col
// matrix and packed weights) and the geometry the GEMM kernel sees.
struct Route {
    int path;           // 0 direct, 1 tiled 1x1, 2 im2col, 3 packed
    size_t stage_x;     // bytes of the staged activation operand
    size_t stage_w;     // bytes of the staged weight operand
    acnn_conv_desc g;   // geometry of the tensor-core launch (NHWC)
};

// Path forced by acnn_conv2d_force_path (0: the router decides).
std::atomic<int> g_force_path{0};
std::atomic<int> g_tiny_shuffle{kTinyWeightsByShuffle};

Route route(const acnn_conv_desc* d, int oh, int ow) {
    Route r{0, 0, 0, *d};
    const size_t es = elem_size(d->dtype);
    if (tensor_path_ok(d, oh, ow)) {
        r.path = (d->kh == 1 && d->kw == 1 && d->stride == 1 && d->pad == 0) ? 1 : 2;
        if (d->layout == ACNN_NCHW) {
            r.stage_x = round256((size_t)d->n * d->h * d->w * d->c_in * es);
            r.stage_w = round256((size_t)d->c_out * d->kh * d->kw * d->c_in * es);
        }
        r.g.layout = ACNN_NHWC;
    } else if (tiny_conv_ok(*d, oh, ow) && (g_force_path.load() == 4 || !packed_path_ok(d, oh, ow))) {
        // direct kernel for 3/6/7 input channels (no staging): used where the
        // packed path cannot go, or when forced; the packed tensor-core path
        // measured faster on the RGB stem and the 7-plane frame input
        r.path = 4;
    } else if (packed_path_ok(d, oh, ow)) {
        const int kp = packed_k(d);
        r.path = 3;
        r.stage_x = round256((size_t)d->n * oh * ow * kp * es);
        r.stage_w = round256((size_t)d->c_out * kp * es);
        r.g = acnn_conv_desc{d->n, oh, ow, kp, d->c_out, 1, 1, 1, 0, ACNN_NHWC, d->dtype};
    }
    return r;
}

}  // namespace

extern "C" {

int acnn_conv2d_out_hw(const acnn_conv_desc* d, int* oh, int* ow) {
    if (!oh || !ow) return ACNN_ERR_NULL_POINTER;
    int st = check_desc(d);
    if (st != ACNN_OK) return st;
    return conv_out(d, oh, ow);
}

int acnn_conv2d_path(const acnn_conv_desc* d) {
    int oh, ow;
    if (check_desc(d) != ACNN_OK || conv_out(d, &oh, &ow) != ACNN_OK) return -1;
    return route(d, oh, ow).path;
}

size_t acnn_conv2d_workspace_size(const acnn_conv_desc* d) {
    int oh, ow;
    if (check_desc(d) != ACNN_OK || conv_out(d, &oh, &ow) != ACNN_OK) return 0;
    const Route r = route(d, oh, ow);
    if (r.path == 0 || r.path == 4) return 0;
    // NCHW-output convs are never split (no partial sums to hold)
    const size_t part = d->layout == ACNN_NHWC ? igemm_plan(r.g, oh, ow, SIZE_MAX).part_bytes : 0;
    return r.stage_x + r.stage_w + round256(part);
}

int acnn_conv2d_force_path(int path, int variant) {
    if (path != 0 && path != 4) return ACNN_ERR_BAD_ENUM;
    if (variant != 0 && variant != 1) return ACNN_ERR_BAD_ENUM;
    g_tiny_shuffle.store(path == 4 ? variant : kTinyWeightsByShuffle);
    g_force_path.store(path);
    return ACNN_OK;
}

int acnn_conv2d_force_plan(int bn, int rows, int splits) {
    if (bn == 0) {
        force_plan(0, 0, 0);
        return ACNN_OK;
    }
    if ((bn != 32 && bn != 64 && bn != 128 && bn != 256) || (rows != 128 && rows != 256) ||
        splits < 1 || splits > 64)
        return ACNN_ERR_BAD_GEOMETRY;
    force_plan(bn, rows / 128, splits);
    return ACNN_OK;
}

int acnn_conv2d_plan(const acnn_conv_desc* d, size_t ws_bytes, int* rows, int* bn,
                     int* splits) {
    int oh, ow;
    if (!rows || !bn || !splits || check_desc(d) != ACNN_OK || conv_out(d, &oh, &ow) != ACNN_OK)
        return -1;
    const Route r = route(d, oh, ow);
    if (r.path == 0 || r.path == 4 || ws_bytes < r.stage_x + r.stage_w) return -1;
    const size_t budget = d->layout == ACNN_NHWC ? ws_bytes - r.stage_x - r.stage_w : 0;
    const IgemmPlan pl = igemm_plan(r.g, oh, ow, budget);
    *rows = 128 * pl.ms;
    *bn = pl.bn;
    *splits = pl.splits;
    return 0;
}

namespace {

// Bytes of the weight operand as the conv kernels consume it (prepacked form):
// the packed [c_out, kp] matrix on the packed path, OHWI on the tensor-core
// paths, the caller's own layout on the direct path.
size_t prepacked_bytes(const acnn_conv_desc* d, const Route& r) {
    const size_t es = elem_size(d->dtype);
    if (r.path == 3) return (size_t)d->c_out * r.g.c_in * es;
    return (size_t)d->c_out * d->kh * d->kw * d->c_in * es;
}

int conv_fused_impl(const acnn_conv_desc* d, const void* x, const void* w, bool prepacked,
                    const float* bias, const float* alpha, const void* residual, int res_mode,
                    int act, void* y, void* workspace, size_t ws_bytes, acnn_stream_t stream,
                    const void* x_nhwc = nullptr, void* y_nhwc = nullptr) {
    int st = check_desc(d);
    if (st != ACNN_OK) return st;
    if (act < ACNN_ACT_NONE || act > ACNN_ACT_PRELU || res_mode < ACNN_RES_NONE ||
        res_mode > ACNN_RES_ACT_THEN_ADD)
        return ACNN_ERR_BAD_ENUM;
    if (!x || !w || !y) return ACNN_ERR_NULL_POINTER;
    if (act == ACNN_ACT_PRELU && !alpha) return ACNN_ERR_NULL_POINTER;
    if (res_mode != ACNN_RES_NONE && !residual) return ACNN_ERR_NULL_POINTER;
    int oh, ow;
    st = conv_out(d, &oh, &ow);
    if (st != ACNN_OK) return st;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (bias && !aligned16(bias)) ||
        (alpha && !aligned16(alpha)) || (residual && !aligned16(residual)) ||
        (workspace && !aligned16(workspace)))
        return ACNN_ERR_MISALIGNED;
    const size_t es = elem_size(d->dtype);
    const size_t xb = (size_t)d->n * d->h * d->w * d->c_in * es;
    const size_t wb = prepacked ? prepacked_bytes(d, route(d, oh, ow))
                                : (size_t)d->c_out * d->kh * d->kw * d->c_in * es;
    const size_t yb = (size_t)d->n * oh * ow * d->c_out * es;
    if (overlaps(y, yb, x, xb) || overlaps(y, yb, w, wb) ||
        (residual && res_mode != ACNN_RES_NONE && overlaps(y, yb, residual, yb)) ||
        (bias && overlaps(y, yb, bias, d->c_out * 4)) ||
        (alpha && act == ACNN_ACT_PRELU && overlaps(y, yb, alpha, d->c_out * 4)))
        return ACNN_ERR_ALIAS;
    if ((long long)d->n * oh * ow > kIndexLimit * 64) return ACNN_ERR_TOO_LARGE;

    ConvArgs a{};
    a.d = *d;
    a.oh = oh;
    a.ow = ow;
    a.x = x;
    a.w = w;
    a.bias = bias;
    a.alpha = act == ACNN_ACT_PRELU ? alpha : nullptr;
    a.residual = res_mode != ACNN_RES_NONE ? residual : nullptr;
    a.res_mode = res_mode;
    a.act = act;
    a.y = y;
    a.out_layout = d->layout;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    const Route r = route(d, oh, ow);
    // NHWC copies (NCHW convs on the implicit-GEMM paths only): an input copy
    // the caller staged already, an output copy to write beside y
    const bool nchw_tc = d->layout == ACNN_NCHW && (r.path == 1 || r.path == 2);
    if ((x_nhwc && !nchw_tc) || (y_nhwc && !(d->layout == ACNN_NCHW && r.path >= 1 && r.path <= 3)))
        return ACNN_ERR_UNSUPPORTED;
    if ((x_nhwc && !aligned16(x_nhwc)) || (y_nhwc && !aligned16(y_nhwc))) return ACNN_ERR_MISALIGNED;
    if (y_nhwc && (overlaps(y_nhwc, yb, y, yb) || overlaps(y_nhwc, yb, x, xb) ||
                   overlaps(y_nhwc, yb, w, wb) || (x_nhwc && overlaps(y_nhwc, yb, x_nhwc, xb)) ||
                   (residual && res_mode != ACNN_RES_NONE && overlaps(y_nhwc, yb, residual, yb))))
        return ACNN_ERR_ALIAS;
    if (x_nhwc && overlaps(y, yb, x_nhwc, xb)) return ACNN_ERR_ALIAS;
    a.y_nhwc = y_nhwc;
    if (r.path == 0) return status_of(launch_direct_conv(a, s));
    if (r.path == 4) return status_of(launch_tiny_conv(a, g_tiny_shuffle.load(), s));

    // Workspace: [staged x | staged w] (required for NCHW and packed convs; no
    // staged w with prepacked weights), then split-K partial sums (optional: a
    // smaller remainder selects fewer splits).
    const size_t stage_w = prepacked ? 0 : r.stage_w;
    const size_t stage = (x_nhwc ? 0 : r.stage_x) + stage_w;
    if (!workspace) ws_bytes = 0;
    if (ws_bytes < stage) return ACNN_ERR_WORKSPACE;
    if (ws_bytes > 0 &&
        (overlaps(workspace, ws_bytes, y, yb) || overlaps(workspace, ws_bytes, x, xb) ||
         overlaps(workspace, ws_bytes, w, wb) ||
         (a.residual && overlaps(workspace, ws_bytes, residual, yb)) ||
         (x_nhwc && overlaps(workspace, ws_bytes, x_nhwc, xb)) ||
         (y_nhwc && overlaps(workspace, ws_bytes, y_nhwc, yb))))
        return ACNN_ERR_ALIAS;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    a.ws_part = ws_bytes > stage ? ws + stage : nullptr;
    a.ws_part_bytes = ws_bytes - stage;
    cudaError_t e = cudaSuccess;
    if (r.path == 3) {
        // explicit im2col: [n*oh*ow, kp] and [c_out, kp], then a 1x1 GEMM whose
        // epilogue writes y in the caller's layout
        e = launch_im2col_pack(*d, oh, ow, r.g.c_in, x, ws, prepacked ? nullptr : w,
                               ws + r.stage_x, s);
        if (e != cudaSuccess) return ACNN_ERR_CUDA;
        a.d = r.g;
        a.x = ws;
        a.w = prepacked ? w : ws + r.stage_x;
        return launch_igemm_conv(a, s);
    }
    if (d->layout == ACNN_NHWC) return launch_igemm_conv(a, s);

    // NCHW on the TMA paths: NHWC copy of x (unless the caller has it) and
    // OHWI copy of w, then the implicit GEMM writing NCHW directly.
    const size_t xs = x_nhwc ? 0 : r.stage_x;
    if (!x_nhwc) {
        e = launch_nchw_to_nhwc(d->n, d->c_in, d->h * d->w, 2, x, ws, s);
        if (e != cudaSuccess) return ACNN_ERR_CUDA;
    }
    if (!prepacked) {
        e = launch_nchw_to_nhwc(d->c_out, d->c_in, d->kh * d->kw, 2, w, ws + xs, s);
        if (e != cudaSuccess) return ACNN_ERR_CUDA;
    }
    a.x = x_nhwc ? x_nhwc : ws;
    a.w = prepacked ? w : ws + xs;
    a.d.layout = ACNN_NHWC;
    a.out_layout = ACNN_NCHW;
    return launch_igemm_conv(a, s);
}

}  // namespace

int acnn_conv2d_fused(const acnn_conv_desc* d, const void* x, const void* w, const float* bias,
                      const float* alpha, const void* residual, int res_mode, int act, void* y,
                      void* workspace, size_t ws_bytes, acnn_stream_t stream) {
    return conv_fused_impl(d, x, w, false, bias, alpha, residual, res_mode, act, y, workspace,
                           ws_bytes, stream);
}

int acnn_conv2d_fused_prepacked(const acnn_conv_desc* d, const void* x, const void* w_packed,
                                const float* bias, const float* alpha, const void* residual,
                                int res_mode, int act, void* y, void* workspace,
                                size_t ws_bytes, acnn_stream_t stream) {
    return conv_fused_impl(d, x, w_packed, true, bias, alpha, residual, res_mode, act, y,
                           workspace, ws_bytes, stream);
}

int acnn_conv2d_fused_prepacked_staged(const acnn_conv_desc* d, const void* x,
                                       const void* x_nhwc, const void* w_packed,
                                       const float* bias, const float* alpha,
                                       const void* residual, int res_mode, int act, void* y,
                                       void* y_nhwc, void* workspace, size_t ws_bytes,
                                       acnn_stream_t stream) {
    if (!d) return ACNN_ERR_NULL_POINTER;
    if (d->layout != ACNN_NCHW && (x_nhwc || y_nhwc)) return ACNN_ERR_UNSUPPORTED;
    return conv_fused_impl(d, x, w_packed, true, bias, alpha, residual, res_mode, act, y, workspace,
                           ws_bytes, stream, x_nhwc, y_nhwc);
}

size_t acnn_conv2d_prepacked_size(const acnn_conv_desc* d) {
    int oh, ow;
    if (check_desc(d) != ACNN_OK || conv_out(d, &oh, &ow) != ACNN_OK) return 0;
    return prepacked_bytes(d, route(d, oh, ow));
}

size_t acnn_conv2d_prepacked_workspace_size(const acnn_conv_desc* d) {
    int oh, ow;
    if (check_desc(d) != ACNN_OK || conv_out(d, &oh, &ow) != ACNN_OK) return 0;
    const Route r = route(d, oh, ow);
    if (r.path == 0 || r.path == 4) return 0;
    const size_t part = d->layout == ACNN_NHWC ? igemm_plan(r.g, oh, ow, SIZE_MAX).part_bytes : 0;
    return r.stage_x + round256(part);
}

int acnn_conv2d_prepack(const acnn_conv_desc* d, const void* w, void* w_packed,
                        acnn_stream_t stream) {
    int st = check_desc(d);
    if (st != ACNN_OK) return st;
    int oh, ow;
    st = conv_out(d, &oh, &ow);
    if (st != ACNN_OK) return st;
    if (!w || !w_packed) return ACNN_ERR_NULL_POINTER;
    if (!aligned16(w) || !aligned16(w_packed)) return ACNN_ERR_MISALIGNED;
    const Route r = route(d, oh, ow);
    const size_t wb = (size_t)d->c_out * d->kh * d->kw * d->c_in * elem_size(d->dtype);
    if (overlaps(w_packed, prepacked_bytes(d, r), w, wb)) return ACNN_ERR_ALIAS;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (r.path == 3)
        e = launch_weight_pack(*d, r.g.c_in, w, w_packed, s);
    else if ((r.path == 1 || r.path == 2) && d->layout == ACNN_NCHW)
        e = launch_nchw_to_nhwc(d->c_out, d->c_in, d->kh * d->kw, 2, w, w_packed, s);
    else
        e = cudaMemcpyAsync(w_packed, w, wb, cudaMemcpyDeviceToDevice, s);
    return status_of(e);
}

int acnn_conv2d_fused_cat2(const acnn_conv_desc* d, const void* x_a, int c_a, const void* x_b,
                           const void* w, const float* bias, const float* alpha,
                           const void* residual, int res_mode, int act, void* y, void* workspace,
                           size_t ws_bytes, acnn_stream_t stream) {
    int st = check_desc(d);
    if (st != ACNN_OK) return st;
    if (act < ACNN_ACT_NONE || act > ACNN_ACT_PRELU || res_mode < ACNN_RES_NONE ||
        res_mode > ACNN_RES_ACT_THEN_ADD)
        return ACNN_ERR_BAD_ENUM;
    if (!x_a || !x_b || !w || !y) return ACNN_ERR_NULL_POINTER;
    if (act == ACNN_ACT_PRELU && !alpha) return ACNN_ERR_NULL_POINTER;
    if (res_mode != ACNN_RES_NONE && !residual) return ACNN_ERR_NULL_POINTER;
    const int c_b = d->c_in - c_a;
    if (d->layout != ACNN_NHWC || d->dtype == ACNN_F32 || c_a <= 0 || c_b <= 0 || c_a % 64 != 0 ||
        c_b % 8 != 0)
        return ACNN_ERR_UNSUPPORTED;
    int oh, ow;
    st = conv_out(d, &oh, &ow);
    if (st != ACNN_OK) return st;
    const Route r = route(d, oh, ow);
    if (r.path != 1 && r.path != 2) return ACNN_ERR_UNSUPPORTED;
    if (!aligned16(x_a) || !aligned16(x_b) || !aligned16(w) || !aligned16(y) ||
        (bias && !aligned16(bias)) || (alpha && !aligned16(alpha)) ||
        (residual && !aligned16(residual)) || (workspace && !aligned16(workspace)))
        return ACNN_ERR_MISALIGNED;
    const size_t es = elem_size(d->dtype);
    const size_t px = (size_t)d->n * d->h * d->w;
    const size_t xab = px * c_a * es, xbb = px * c_b * es;
    const size_t wb = (size_t)d->c_out * d->kh * d->kw * d->c_in * es;
    const size_t yb = (size_t)d->n * oh * ow * d->c_out * es;
    if (overlaps(y, yb, x_a, xab) || overlaps(y, yb, x_b, xbb) || overlaps(y, yb, w, wb) ||
        (residual && res_mode != ACNN_RES_NONE && overlaps(y, yb, residual, yb)) ||
        (bias && overlaps(y, yb, bias, d->c_out * 4)) ||
        (alpha && act == ACNN_ACT_PRELU && overlaps(y, yb, alpha, d->c_out * 4)))
        return ACNN_ERR_ALIAS;
    if (!workspace) ws_bytes = 0;
    if (ws_bytes > 0 &&
        (overlaps(workspace, ws_bytes, y, yb) || overlaps(workspace, ws_bytes, x_a, xab) ||
         overlaps(workspace, ws_bytes, x_b, xbb) || overlaps(workspace, ws_bytes, w, wb) ||
         (residual && res_mode != ACNN_RES_NONE && overlaps(workspace, ws_bytes, residual, yb))))
        return ACNN_ERR_ALIAS;
    ConvArgs a{};
    a.d = *d;
    a.oh = oh;
    a.ow = ow;
    a.x = x_a;
    a.x2 = x_b;
    a.c_split = c_a;
    a.w = w;
    a.bias = bias;
    a.alpha = act == ACNN_ACT_PRELU ? alpha : nullptr;
    a.residual = res_mode != ACNN_RES_NONE ? residual : nullptr;
    a.res_mode = res_mode;
    a.act = act;
    a.y = y;
    a.out_layout = ACNN_NHWC;
    a.ws_part = ws_bytes > 0 ? workspace : nullptr;  // NHWC: no staging, all for split-K
    a.ws_part_bytes = ws_bytes;
    return launch_igemm_conv(a, reinterpret_cast<cudaStream_t>(stream));
}

int acnn_conv2d_fused_pool2(const acnn_conv_desc* d, const void* x, const void* w,
                            const float* bias, const float* alpha, const void* residual,
                            int res_mode, int act, void* y, void* y_pool, acnn_stream_t stream) {
    int st = check_desc(d);
    if (st != ACNN_OK) return st;
    if (act < ACNN_ACT_NONE || act > ACNN_ACT_PRELU || res_mode < ACNN_RES_NONE ||
        res_mode > ACNN_RES_ACT_THEN_ADD)
        return ACNN_ERR_BAD_ENUM;
    if (!x || !w || !y || !y_pool) return ACNN_ERR_NULL_POINTER;
    if (act == ACNN_ACT_PRELU && !alpha) return ACNN_ERR_NULL_POINTER;
    if (res_mode != ACNN_RES_NONE && !residual) return ACNN_ERR_NULL_POINTER;
    int oh, ow;
    st = conv_out(d, &oh, &ow);
    if (st != ACNN_OK) return st;
    // a 1x1/s1/p0 NHWC 16-bit conv on the tiled tensor-core path, 64-channel
    // k-blocks, an even output map
    const Route r = route(d, oh, ow);
    if (r.path != 1 || d->layout != ACNN_NHWC || d->c_in < 64 || oh % 2 || ow % 2)
        return ACNN_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || !aligned16(y_pool) ||
        (bias && !aligned16(bias)) || (alpha && !aligned16(alpha)) ||
        (residual && !aligned16(residual)))
        return ACNN_ERR_MISALIGNED;
    const size_t es = elem_size(d->dtype);
    const size_t xb = (size_t)d->n * d->h * d->w * d->c_in * es;
    const size_t wb = (size_t)d->c_out * d->c_in * es;
    const size_t yb = (size_t)d->n * oh * ow * d->c_out * es;
    const size_t pb = yb / 4;
    const bool res = residual && res_mode != ACNN_RES_NONE;
    if (overlaps(y, yb, x, xb) || overlaps(y, yb, w, wb) || (res && overlaps(y, yb, residual, yb)) ||
        (bias && overlaps(y, yb, bias, d->c_out * 4)) ||
        (alpha && act == ACNN_ACT_PRELU && overlaps(y, yb, alpha, d->c_out * 4)) ||
        overlaps(y_pool, pb, y, yb) || overlaps(y_pool, pb, x, xb) || overlaps(y_pool, pb, w, wb) ||
        (res && overlaps(y_pool, pb, residual, yb)) ||
        (bias && overlaps(y_pool, pb, bias, d->c_out * 4)) ||
        (alpha && act == ACNN_ACT_PRELU && overlaps(y_pool, pb, alpha, d->c_out * 4)))
        return ACNN_ERR_ALIAS;
    ConvArgs a{};
    a.d = *d;
    a.oh = oh;
    a.ow = ow;
    a.x = x;
    a.w = w;
    a.bias = bias;
    a.alpha = act == ACNN_ACT_PRELU ? alpha : nullptr;
    a.residual = res ? residual : nullptr;
    a.res_mode = res_mode;
    a.act = act;
    a.y = y;
    a.y2 = y_pool;
    a.out_layout = ACNN_NHWC;
    return launch_igemm_conv(a, reinterpret_cast<cudaStream_t>(stream));
}

int acnn_conv2d_fused_up2(const acnn_conv_desc* d, const void* x_a, int c_a, const void* x_b,
                          const void* w, const float* bias, const float* alpha,
                          const void* residual, int res_mode, int act, void* y, void* y_up,
                          void* workspace, size_t ws_bytes, acnn_stream_t stream) {
    int st = check_desc(d);
    if (st != ACNN_OK) return st;
    if (act < ACNN_ACT_NONE || act > ACNN_ACT_PRELU || res_mode < ACNN_RES_NONE ||
        res_mode > ACNN_RES_ACT_THEN_ADD)
        return ACNN_ERR_BAD_ENUM;
    if (!x_a || !w || !y || !y_up) return ACNN_ERR_NULL_POINTER;
    if (act == ACNN_ACT_PRELU && !alpha) return ACNN_ERR_NULL_POINTER;
    if (res_mode != ACNN_RES_NONE && !residual) return ACNN_ERR_NULL_POINTER;
    // x_b NULL: x_a holds all c_in channels (c_a is ignored)
    const bool cat = x_b != nullptr;
    const int ca = cat ? c_a : d->c_in, cb = d->c_in - ca;
    if (d->layout != ACNN_NHWC || d->dtype == ACNN_F32) return ACNN_ERR_UNSUPPORTED;
    if (cat && (ca <= 0 || cb <= 0 || ca % 64 != 0 || cb % 8 != 0)) return ACNN_ERR_UNSUPPORTED;
    int oh, ow;
    st = conv_out(d, &oh, &ow);
    if (st != ACNN_OK) return st;
    const Route r = route(d, oh, ow);
    if (r.path != 1 && r.path != 2) return ACNN_ERR_UNSUPPORTED;
    if (4ll * d->n * oh * ow > kIndexLimit) return ACNN_ERR_TOO_LARGE;
    if (!aligned16(x_a) || (cat && !aligned16(x_b)) || !aligned16(w) || !aligned16(y) ||
        !aligned16(y_up) || (bias && !aligned16(bias)) || (alpha && !aligned16(alpha)) ||
        (residual && !aligned16(residual)) || (workspace && !aligned16(workspace)))
        return ACNN_ERR_MISALIGNED;
    const size_t es = elem_size(d->dtype);
    const size_t px = (size_t)d->n * d->h * d->w;
    const size_t xab = px * ca * es, xbb = px * cb * es;
    const size_t wb = (size_t)d->c_out * d->kh * d->kw * d->c_in * es;
    const size_t yb = (size_t)d->n * oh * ow * d->c_out * es;
    const size_t ub = 4 * yb;
    const bool res = residual && res_mode != ACNN_RES_NONE;
    auto hits = [&](const void* p, size_t n) {
        return overlaps(p, n, x_a, xab) || (cat && overlaps(p, n, x_b, xbb)) ||
               overlaps(p, n, w, wb) || (res && overlaps(p, n, residual, yb)) ||
               (bias && overlaps(p, n, bias, d->c_out * 4)) ||
               (alpha && act == ACNN_ACT_PRELU && overlaps(p, n, alpha, d->c_out * 4));
    };
    if (hits(y, yb) || hits(y_up, ub) || overlaps(y, yb, y_up, ub)) return ACNN_ERR_ALIAS;
    if (!workspace) ws_bytes = 0;
    if (ws_bytes > 0 && (hits(workspace, ws_bytes) || overlaps(workspace, ws_bytes, y, yb) ||
                         overlaps(workspace, ws_bytes, y_up, ub)))
        return ACNN_ERR_ALIAS;
    ConvArgs a{};
    a.d = *d;
    a.oh = oh;
    a.ow = ow;
    a.x = x_a;
    a.x2 = cat ? x_b : nullptr;
    a.c_split = cat ? ca : 0;
    a.w = w;
    a.bias = bias;
    a.alpha = act == ACNN_ACT_PRELU ? alpha : nullptr;
    a.residual = res ? residual : nullptr;
    a.res_mode = res_mode;
    a.act = act;
    a.y = y;
    a.y2 = y_up;
    a.y2_up = 1;
    a.out_layout = ACNN_NHWC;
    a.ws_part = ws_bytes > 0 ? workspace : nullptr;  // NHWC: no staging, all for split-K
    a.ws_part_bytes = ws_bytes;
    return launch_igemm_conv(a, reinterpret_cast<cudaStream_t>(stream));
}

int acnn_pool2d(int kind, int n, int h, int w, int c, int k, int stride, int pad, int layout,
                int dtype, const void* x, void* y, acnn_stream_t stream) {
    if (kind != ACNN_POOL_MAX && kind != ACNN_POOL_AVG) return ACNN_ERR_BAD_ENUM;
    if (!valid_dtype(dtype) || !valid_layout(layout)) return ACNN_ERR_BAD_ENUM;
    if (!x || !y) return ACNN_ERR_NULL_POINTER;
    if (n <= 0 || h <= 0 || w <= 0 || c <= 0 || k <= 0 || stride <= 0 || pad < 0)
        return ACNN_ERR_BAD_GEOMETRY;
    if (kind == ACNN_POOL_AVG && pad != 0) return ACNN_ERR_UNSUPPORTED;
    if (pad >= k) return ACNN_ERR_UNSUPPORTED;  // a window could hold no input tap
    if (h + 2 * pad < k || w + 2 * pad < k) return ACNN_ERR_BAD_GEOMETRY;
    const int oh = (h + 2 * pad - k) / stride + 1, ow = (w + 2 * pad - k) / stride + 1;
    if ((long long)n * h * w * c > kIndexLimit) return ACNN_ERR_TOO_LARGE;
    if (!aligned16(x) || !aligned16(y)) return ACNN_ERR_MISALIGNED;
    const size_t es = elem_size(dtype);
    if (overlaps(x, (size_t)n * h * w * c * es, y, (size_t)n * oh * ow * c * es))
        return ACNN_ERR_ALIAS;
    return status_of(launch_pool2d(kind, n, h, w, c, k, stride, pad, layout, dtype, x, y,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

int acnn_resize2d(int mode, int n, int c, int h, int w, int oh, int ow, int layout, int in_dtype,
                  int out_dtype, const void* x, void* y, acnn_stream_t stream) {
    if (mode != ACNN_RESIZE_NEAREST && mode != ACNN_RESIZE_BILINEAR) return ACNN_ERR_BAD_ENUM;
    if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype) || !valid_layout(layout))
        return ACNN_ERR_BAD_ENUM;
    if (!x || !y) return ACNN_ERR_NULL_POINTER;
    if (n <= 0 || c <= 0 || h <= 0 || w <= 0 || oh <= 0 || ow <= 0) return ACNN_ERR_BAD_GEOMETRY;
    if (mode == ACNN_RESIZE_NEAREST && in_dtype != out_dtype) return ACNN_ERR_UNSUPPORTED;
    if ((long long)n * c * oh * ow > kIndexLimit || (long long)n * c * h * w > kIndexLimit)
        return ACNN_ERR_TOO_LARGE;
    if (!aligned16(x) || !aligned16(y)) return ACNN_ERR_MISALIGNED;
    if (overlaps(x, (size_t)n * c * h * w * elem_size(in_dtype), y,
                 (size_t)n * c * oh * ow * elem_size(out_dtype)))
        return ACNN_ERR_ALIAS;
    return status_of(launch_resize2d(mode, n, c, h, w, oh, ow, layout, in_dtype, out_dtype, x, y,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int acnn_concat(int n, int h, int w, int c_a, int c_b, int layout, int dtype, const void* a,
                const void* b, void* y, acnn_stream_t stream) {
    if (!valid_dtype(dtype) || !valid_layout(layout)) return ACNN_ERR_BAD_ENUM;
    if (!a || !b || !y) return ACNN_ERR_NULL_POINTER;
    if (n <= 0 || h <= 0 || w <= 0 || c_a <= 0 || c_b <= 0) return ACNN_ERR_BAD_GEOMETRY;
    if (!aligned16(a) || !aligned16(b) || !aligned16(y)) return ACNN_ERR_MISALIGNED;
    const size_t es = elem_size(dtype), px = (size_t)n * h * w;
    if ((long long)n * (c_a + c_b) * h * w > kIndexLimit) return ACNN_ERR_TOO_LARGE;
    if (overlaps(y, px * (c_a + c_b) * es, a, px * c_a * es) ||
        overlaps(y, px * (c_a + c_b) * es, b, px * c_b * es))
        return ACNN_ERR_ALIAS;
    return status_of(launch_concat(n, h, w, c_a, c_b, layout, dtype, a, b, y,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

int acnn_deconv2d(const acnn_conv_desc* d, const void* x, const float* w, const float* bias,
                  const float* alpha, int act, int out_dtype, void* y, acnn_stream_t stream) {
    int st = check_desc(d);
    if (st != ACNN_OK) return st;
    if (act < ACNN_ACT_NONE || act > ACNN_ACT_PRELU || !valid_dtype(out_dtype))
        return ACNN_ERR_BAD_ENUM;
    if (!x || !w || !y) return ACNN_ERR_NULL_POINTER;
    if (act == ACNN_ACT_PRELU && !alpha) return ACNN_ERR_NULL_POINTER;
    if (d->kh != 4 || d->kw != 4 || d->stride != 2 || d->pad != 1) return ACNN_ERR_UNSUPPORTED;
    const int oh = (d->h - 1) * d->stride - 2 * d->pad + d->kh;
    const int ow = (d->w - 1) * d->stride - 2 * d->pad + d->kw;
    if ((long long)d->n * oh * ow * ((d->c_out + 7) / 8) > kIndexLimit ||
        (long long)d->n * d->c_in * d->h * d->w > kIndexLimit)
        return ACNN_ERR_TOO_LARGE;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (bias && !aligned16(bias)) ||
        (alpha && !aligned16(alpha)))
        return ACNN_ERR_MISALIGNED;
    const size_t yb = (size_t)d->n * d->c_out * oh * ow * elem_size(out_dtype);
    if (overlaps(y, yb, x, (size_t)d->n * d->c_in * d->h * d->w * elem_size(d->dtype)) ||
        overlaps(y, yb, w, (size_t)d->c_in * d->c_out * 16 * 4))
        return ACNN_ERR_ALIAS;
    return status_of(launch_deconv2d(*d, oh, ow, x, w, bias, act == ACNN_ACT_PRELU ? alpha : nullptr,
                                     act, out_dtype, y, reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
// The tensor-core form of the 4x4/s2/p1 deconv (a 3x3/s1/p1 conv to 4 c_out
// channels, then a pixel shuffle): whether it serves d, and its workspace
// [x staged NHWC (NCHW input only) | regrouped weights | bias | alpha | conv
// output], each 256-byte aligned; 0 when it does not serve d.
struct DeconvGemm {
    int co4;
    size_t x_stage, wg, bg, ag, ys, total;
};
DeconvGemm deconv_gemm_plan(const acnn_conv_desc* d, int out_dtype) {
    DeconvGemm g{};
    // fp16 only: the weights are rounded to the storage type, and bf16's 8-bit
    // significand moves an output by more than one unit of its storage there
    if (d->dtype != ACNN_F16 || out_dtype != d->dtype || d->c_in % 8 != 0) return g;
    if (d->kh != 4 || d->kw != 4 || d->stride != 2 || d->pad != 1) return g;
    const int co4 = (4 * d->c_out + 7) / 8 * 8;
    const acnn_conv_desc d3{d->n, d->h, d->w, d->c_in, co4, 3, 3, 1, 1, ACNN_NHWC, d->dtype};
    if (!tensor_path_ok(&d3, d->h, d->w)) return g;
    const size_t es = elem_size(d->dtype);
    g.co4 = co4;
    g.x_stage = d->layout == ACNN_NCHW ? round256((size_t)d->n * d->h * d->w * d->c_in * es) : 0;
    g.wg = round256((size_t)co4 * 9 * d->c_in * es);
    g.bg = round256((size_t)co4 * 4);
    g.ag = g.bg;
    g.ys = round256((size_t)d->n * d->h * d->w * co4 * es);
    g.total = g.x_stage + g.wg + g.bg + g.ag + g.ys;
    return g;
}
}  // namespace

size_t acnn_deconv2d_workspace_size(const acnn_conv_desc* d, int out_dtype) {
    if (check_desc(d) != ACNN_OK || !valid_dtype(out_dtype)) return 0;
    return deconv_gemm_plan(d, out_dtype).total;
}

int acnn_deconv2d_ws(const acnn_conv_desc* d, const void* x, const float* w, const float* bias,
                     const float* alpha, int act, int out_dtype, void* y, void* workspace,
                     size_t ws_bytes, acnn_stream_t stream) {
    const DeconvGemm g = deconv_gemm_plan(d, out_dtype);
    if (!workspace || g.total == 0 || ws_bytes < g.total)
        return acnn_deconv2d(d, x, w, bias, alpha, act, out_dtype, y, stream);
    // the same validation as the direct form, then the workspace
    int st = check_desc(d);
    if (st != ACNN_OK) return st;
    if (act < ACNN_ACT_NONE || act > ACNN_ACT_PRELU || !valid_dtype(out_dtype))
        return ACNN_ERR_BAD_ENUM;
    if (!x || !w || !y) return ACNN_ERR_NULL_POINTER;
    if (act == ACNN_ACT_PRELU && !alpha) return ACNN_ERR_NULL_POINTER;
    const int oh = 2 * d->h, ow = 2 * d->w;
    if ((long long)d->n * d->c_out * oh * ow > kIndexLimit ||
        (long long)d->n * d->c_in * d->h * d->w > kIndexLimit)
        return ACNN_ERR_TOO_LARGE;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || !aligned16(workspace) ||
        (bias && !aligned16(bias)) || (alpha && !aligned16(alpha)))
        return ACNN_ERR_MISALIGNED;
    const size_t es = elem_size(d->dtype);
    const size_t xb = (size_t)d->n * d->c_in * d->h * d->w * es;
    const size_t wb = (size_t)d->c_in * d->c_out * 16 * 4;
    const size_t yb = (size_t)d->n * d->c_out * oh * ow * es;
    if (overlaps(y, yb, x, xb) || overlaps(y, yb, w, wb) || overlaps(workspace, ws_bytes, x, xb) ||
        overlaps(workspace, ws_bytes, w, wb) || overlaps(workspace, ws_bytes, y, yb) ||
        (bias && overlaps(workspace, ws_bytes, bias, d->c_out * 4)) ||
        (alpha && overlaps(workspace, ws_bytes, alpha, d->c_out * 4)))
        return ACNN_ERR_ALIAS;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* x_nhwc = g.x_stage ? ws : const_cast<void*>(x);
    void* wg = ws + g.x_stage;
    float* bg = reinterpret_cast<float*>(ws + g.x_stage + g.wg);
    float* ag = reinterpret_cast<float*>(ws + g.x_stage + g.wg + g.bg);
    void* ys = ws + g.x_stage + g.wg + g.bg + g.ag;
    cudaError_t e = launch_deconv_gemm_weights(d->dtype, w, bias, act == ACNN_ACT_PRELU ? alpha : nullptr,
                                               wg, bg, ag, d->c_in, d->c_out, g.co4, s);
    if (e == cudaSuccess && g.x_stage)
        e = launch_nchw_to_nhwc(d->n, d->c_in, d->h * d->w, 2, x, x_nhwc, s);
    if (e != cudaSuccess) return ACNN_ERR_CUDA;
    ConvArgs a{};
    a.d = acnn_conv_desc{d->n, d->h, d->w, d->c_in, g.co4, 3, 3, 1, 1, ACNN_NHWC, d->dtype};
    a.oh = d->h;
    a.ow = d->w;
    a.x = x_nhwc;
    a.w = wg;
    a.bias = bg;
    a.alpha = act == ACNN_ACT_PRELU ? ag : nullptr;
    a.residual = nullptr;
    a.res_mode = ACNN_RES_NONE;
    a.act = act;
    a.y = ys;
    a.out_layout = ACNN_NHWC;
    st = launch_igemm_conv(a, s);
    if (st != ACNN_OK) return st;
    return status_of(launch_deconv_shuffle(d->dtype, ys, y, d->layout, d->n, d->h, d->w, d->c_out,
                                           g.co4, s));
}

int acnn_frame_prep_quarter(int h, int w, const uint8_t* rgba0, const uint8_t* rgba1, float t,
                            int out_dtype, void* y, acnn_stream_t stream) {
    if (!valid_dtype(out_dtype)) return ACNN_ERR_BAD_ENUM;
    if (!rgba0 || !rgba1 || !y) return ACNN_ERR_NULL_POINTER;
    if (h <= 0 || w <= 0 || h % 4 != 0 || w % 4 != 0) return ACNN_ERR_BAD_GEOMETRY;
    if ((long long)h * w > kIndexLimit) return ACNN_ERR_TOO_LARGE;
    if (!aligned16(rgba0) || !aligned16(rgba1) || !aligned16(y)) return ACNN_ERR_MISALIGNED;
    const size_t yb = (size_t)7 * (h / 4) * (w / 4) * elem_size(out_dtype);
    if (overlaps(y, yb, rgba0, (size_t)h * w * 4) || overlaps(y, yb, rgba1, (size_t)h * w * 4))
        return ACNN_ERR_ALIAS;
    return status_of(launch_prep_quarter(h, w, rgba0, rgba1, t, out_dtype, y,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

int acnn_frame_flow_out(int h, int w, const void* tmp8, int tmp8_dtype, const uint8_t* rgba0,
                        const uint8_t* rgba1, const float* refine_res, uint8_t* out_rgba,
                        acnn_stream_t stream) {
    if (!valid_dtype(tmp8_dtype)) return ACNN_ERR_BAD_ENUM;
    if (!tmp8 || !rgba0 || !rgba1 || !out_rgba) return ACNN_ERR_NULL_POINTER;
    if (h <= 0 || w <= 0 || h % 8 != 0 || w % 8 != 0) return ACNN_ERR_BAD_GEOMETRY;
    if ((long long)h * w > kIndexLimit) return ACNN_ERR_TOO_LARGE;
    if (!aligned16(tmp8) || !aligned16(rgba0) || !aligned16(rgba1) || !aligned16(out_rgba) ||
        (refine_res && !aligned16(refine_res)))
        return ACNN_ERR_MISALIGNED;
    const size_t fb = (size_t)h * w * 4;
    const size_t tb = (size_t)5 * (h / 8) * (w / 8) * elem_size(tmp8_dtype);
    const size_t rb = (size_t)3 * (h / 4) * (w / 4) * sizeof(float);
    if (overlaps(out_rgba, fb, rgba0, fb) || overlaps(out_rgba, fb, rgba1, fb) ||
        overlaps(out_rgba, fb, tmp8, tb) || (refine_res && overlaps(out_rgba, fb, refine_res, rb)))
        return ACNN_ERR_ALIAS;
    return status_of(launch_flow_out(h, w, tmp8, tmp8_dtype, rgba0, rgba1, refine_res, out_rgba,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int acnn_frame_refine_prep(int h, int w, const void* tmp8, int tmp8_dtype, const uint8_t* rgba0,
                           const uint8_t* rgba1, int out_dtype, void* y, acnn_stream_t stream) {
    if (!valid_dtype(tmp8_dtype) || !valid_dtype(out_dtype)) return ACNN_ERR_BAD_ENUM;
    if (!tmp8 || !rgba0 || !rgba1 || !y) return ACNN_ERR_NULL_POINTER;
    if (h <= 0 || w <= 0 || h % 8 != 0 || w % 8 != 0) return ACNN_ERR_BAD_GEOMETRY;
    if ((long long)h * w > kIndexLimit) return ACNN_ERR_TOO_LARGE;
    if (!aligned16(tmp8) || !aligned16(rgba0) || !aligned16(rgba1) || !aligned16(y))
        return ACNN_ERR_MISALIGNED;
    const size_t fb = (size_t)h * w * 4;
    const size_t tb = (size_t)5 * (h / 8) * (w / 8) * elem_size(tmp8_dtype);
    const size_t yb = (size_t)11 * (h / 4) * (w / 4) * elem_size(out_dtype);
    if (overlaps(y, yb, rgba0, fb) || overlaps(y, yb, rgba1, fb) || overlaps(y, yb, tmp8, tb))
        return ACNN_ERR_ALIAS;
    return status_of(launch_refine_prep(h, w, tmp8, tmp8_dtype, rgba0, rgba1, out_dtype, y,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int acnn_frame_refine_out(int c, int hh, int hw, const void* x, int dtype, const float* w,
                          const float* bias, float* y, acnn_stream_t stream) {
    if (!valid_dtype(dtype)) return ACNN_ERR_BAD_ENUM;
    if (!x || !w || !bias || !y) return ACNN_ERR_NULL_POINTER;
    if (c <= 0 || hh <= 0 || hw <= 0) return ACNN_ERR_BAD_GEOMETRY;
    if ((long long)c * hh * hw > kIndexLimit) return ACNN_ERR_TOO_LARGE;
    if (!aligned16(x) || !aligned16(y)) return ACNN_ERR_MISALIGNED;
    const size_t yb = (size_t)3 * hh * hw * sizeof(float);
    if (overlaps(y, yb, x, (size_t)c * hh * hw * elem_size(dtype)) ||
        overlaps(y, yb, w, (size_t)27 * c * sizeof(float)) || overlaps(y, yb, bias, 3 * sizeof(float)))
        return ACNN_ERR_ALIAS;
    return status_of(launch_refine_out(c, hh, hw, x, dtype, w, bias, y,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

int acnn_film(int c, long long n, int dtype, const void* x, float t, const float* w0,
              const float* b0, int hn, const float* w2, const float* b2, void* y,
              acnn_stream_t stream) {
    if (!valid_dtype(dtype)) return ACNN_ERR_BAD_ENUM;
    if (!x || !w0 || !b0 || !w2 || !b2 || !y) return ACNN_ERR_NULL_POINTER;
    if (c <= 0 || n <= 0 || hn <= 0) return ACNN_ERR_BAD_GEOMETRY;
    if (n > kIndexLimit || c > 65535 || (long long)c * n > kIndexLimit * 64) return ACNN_ERR_TOO_LARGE;
    const size_t xb = (size_t)c * n * elem_size(dtype);
    // y may be x itself (each element is read, then written, by one thread)
    if (y != x && overlaps(y, xb, x, xb)) return ACNN_ERR_ALIAS;
    return status_of(launch_film(c, (int)n, dtype, x, t, w0, b0, hn, w2, b2, y,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

const char* acnn_status_string(int status) {
    switch (status) {
    case ACNN_OK: return "ok";
    case ACNN_ERR_NULL_POINTER: return "a required pointer is NULL";
    case ACNN_ERR_BAD_GEOMETRY: return "invalid geometry (a size is not positive or the output is empty)";
    case ACNN_ERR_UNSUPPORTED: return "valid but unsupported geometry or mode";
    case ACNN_ERR_MISALIGNED: return "a device pointer is not 16-byte aligned";
    case ACNN_ERR_WORKSPACE: return "workspace missing or too small";
    case ACNN_ERR_ALIAS: return "the output overlaps an input";
    case ACNN_ERR_BAD_ENUM: return "an enum argument is out of range";
    case ACNN_ERR_CUDA: return "a CUDA call failed";
    case ACNN_ERR_DEVICE_TIMEOUT: return "a kernel's bounded pipeline wait expired";
    case ACNN_ERR_TOO_LARGE: return "an index would overflow 32 bits";
    default: return "unknown status";
    }
}

int acnn_last_device_status(acnn_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ACNN_ERR_CUDA;
    int* p = device_status_ptr();
    if (!p) return ACNN_ERR_CUDA;
    int v = 0;
    const int zero = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ACNN_ERR_CUDA;
    if (v != 0 && cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
        return ACNN_ERR_CUDA;
    return v;
}

int acnn_set_wait_budget(long long polls) {
    if (polls < 0) return ACNN_ERR_BAD_GEOMETRY;
    g_wait_budget.store(polls);
    return ACNN_OK;
}

int acnn_section_begin(acnn_stream_t stream) {
    return status_of(cudaStreamBeginCapture(reinterpret_cast<cudaStream_t>(stream),
                                            cudaStreamCaptureModeThreadLocal));
}

int acnn_section_end(acnn_stream_t stream, void** exec) {
    if (!exec) return ACNN_ERR_NULL_POINTER;
    *exec = nullptr;
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamEndCapture(reinterpret_cast<cudaStream_t>(stream), &g);
    if (e != cudaSuccess) return ACNN_ERR_CUDA;
    cudaGraphExec_t ge = nullptr;
    e = cudaGraphInstantiate(&ge, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return ACNN_ERR_CUDA;
    *exec = ge;
    return ACNN_OK;
}

int acnn_section_launch(void* exec, acnn_stream_t stream) {
    if (!exec) return ACNN_ERR_NULL_POINTER;
    return status_of(cudaGraphLaunch(static_cast<cudaGraphExec_t>(exec),
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int acnn_section_destroy(void* exec) {
    if (!exec) return ACNN_OK;
    return status_of(cudaGraphExecDestroy(static_cast<cudaGraphExec_t>(exec)));
}

int acnn_device_sm_count(void) { return sm_count(); }

}  // extern "C"

// ---------------------------------------------------------------------------
// acnn_conv2d_fused_noalloc: conv2d_fused for callers that cannot allocate.
//
// Some callers have no way to obtain device memory at the point where they
// run a conv: a plugin inside a host framework that owns every device
// allocation and hands the plugin no allocator, or a latency-critical loop
// where a cudaMalloc/cudaFree may synchronise the whole device.  For them the
// scratch that the NCHW tensor-core path needs (the NHWC copy of x and the
// OHWI copy of w) lives in the file-scope array below, sized once at
// ACNN_NOALLOC_SCRATCH_BYTES, which every GPU that loads the library holds
// until the process exits.
// ---------------------------------------------------------------------------
namespace {
__device__ __align__(256) uint8_t g_noalloc_scratch[ACNN_NOALLOC_SCRATCH_BYTES];
std::atomic<void*> g_noalloc_scratch_ptr[kMaxDevices];
std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device, looked up once
// per device with that device current (the host-side symbol is only a
// stand-in, never a device address); later calls take the cached address
// without locking.  NULL if the lookup fails.
void* noalloc_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    void* p = g_noalloc_scratch_ptr[dev].load(std::memory_order_acquire);
    if (p) return p;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    p = g_noalloc_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        g_noalloc_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    return p;
}
}  // namespace

extern "C" int acnn_conv2d_fused_noalloc(const acnn_conv_desc* d, const void* x, const void* w,
                                         const float* bias, const float* alpha,
                                         const void* residual, int res_mode, int act, void* y,
                                         acnn_stream_t stream) {
    int st = check_desc(d);
    if (st != ACNN_OK) return st;
    // The staging copies must fit; split-K partial sums use what is left
    // of the array (fewer splits when little is left).
    int oh, ow;
    st = conv_out(d, &oh, &ow);
    if (st != ACNN_OK) return st;
    const Route r = route(d, oh, ow);
    if (r.stage_x + r.stage_w > (size_t)ACNN_NOALLOC_SCRATCH_BYTES) return ACNN_ERR_WORKSPACE;
    const size_t want = acnn_conv2d_workspace_size(d);
    const size_t give = want < (size_t)ACNN_NOALLOC_SCRATCH_BYTES ? want
                                                                  : (size_t)ACNN_NOALLOC_SCRATCH_BYTES;
    void* ws = nullptr;
    if (give > 0) {
        ws = noalloc_scratch();
        if (!ws) return ACNN_ERR_CUDA;
    }
    return acnn_conv2d_fused(d, x, w, bias, alpha, residual, res_mode, act, y, ws, give, stream);
}
