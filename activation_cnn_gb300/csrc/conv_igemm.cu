// conv_igemm.cu -- NHWC implicit-GEMM conv2d_fused on the 5th-generation
// tensor cores (tcgen05 + TMEM), fed by TMA.
//
// GEMM view of the conv (rtdetr_gpu.rs RtDetrGpu::conv: im2col -> GEMM with
// the bias and activation in the epilogue): M = N*OH*OW output pixels,
// N_g = C_out, K = kh*kw*C_in in (ky, kx, ci) order.  Nothing is materialised:
//   * A (128 pixels x 64 channels per k-block) arrives by TMA -- a tiled box of
//     the [N*H*W, C_in] matrix for 1x1/s1/p0 convs (the NHWC map *is* the GEMM
//     operand, as the page notes), otherwise an im2col-mode box: 128
//     consecutive output pixels (wrapping rows and images), each read at the
//     tap offset (kx, ky), with the conv stride as the traversal stride and the
//     padding as the bounding box, out-of-image taps filled with zeros.
//   * B (BN output channels x 64 channels) is a tiled box of the OHWI weight
//     viewed as [C_out][kh*kw][C_in].
//   * Both land in shared memory in the 128-byte-swizzled K-major layout that
//     tcgen05.mma reads directly; a 64-channel k-block is one 128-byte row.
// Warp roles (448 threads, persistent, one CTA per SM):
//   warp 0  TMA producer (one lane) over a ring of operand stages in shared
//           memory (as deep as the shared memory left by the epilogue allows)
//   warp 1  TMEM allocator and MMA issuer (one lane): MS x 4 x (128 x BN x 16)
//           MMAs per k-block into an fp32 TMEM accumulator
//   warps 2-13 epilogue, three per TMEM lane quarter: tcgen05.ld 32 columns at
//           a time, + bias, activation, residual (before or after the
//           activation), down-cast, 16-byte stores through a shared-memory
//           slot; residual boxes stream in by cp.async several chunks ahead.
// Two TMEM accumulators alternate so the epilogue of one tile overlaps the
// MMAs of the next.  Every mbarrier wait is bounded: on expiry the kernel
// records ACNN_ERR_DEVICE_TIMEOUT in a device status word, raises a CTA-wide
// abort flag, drains its own in-flight copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace acnn {

namespace {

constexpr int BM = 128;             // output pixels per tile (TMEM lanes)
constexpr int kEpiGroups = 3;       // epilogue warps per TMEM lane quarter
constexpr int kEpiWarps = 4 * kEpiGroups;
constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer, MMA, epilogue warps
constexpr long long kTimeoutCycles = 8000000000ll;  // ~4 s per wait at 2 GHz
constexpr long long kDrainCycles = 400000000ll;     // ~0.2 s per drain wait

constexpr uint32_t kStageBytes = 32 * 64;  // epilogue slot: 32 rows x 32 channels x 2 B
constexpr int kMaxStages = 8;
constexpr int kMaxResDepth = 4;  // residual boxes in flight per epilogue warp
constexpr size_t kBarBytes = 512;
constexpr size_t kSmemMax = 232448;  // 227 KB of dynamic shared memory per CTA
// Shared memory besides the operand ring, the epilogue slots and the bias /
// PReLU-alpha copy (par_floats fp32 values).  The window must start 1024-byte
// aligned (the kernel checks): the swizzled operand tiles rely on it.
constexpr size_t kSmemFixed = kBarBytes;
static_assert((2 * kMaxStages + 6) * 8 + 12 <= kBarBytes, "barrier region too small");

// Tile of (128 * MS) output pixels x BN output channels, K in blocks of BK
// channels: MS row blocks of 128 share each B tile, so one pipeline step
// carries MS x BK/16 MMAs.  A k-block row is BK x 2 bytes: 128 B (BK = 64,
// 128-byte swizzle) or 64 B (BK = 32, 64-byte swizzle, for C_in <= 32).  The
// ring depth is chosen per launch from the shared memory left by the
// residual ring and, when the weights stay resident, by the weights.
template <int BN, int MS, int BK> struct Cfg {
    static constexpr uint32_t kABytes = BM * BK * 2;  // one 128-row block
    static constexpr uint32_t kAB = MS * kABytes;     // A bytes per stage
    static constexpr uint32_t kBBytes = BN * BK * 2;
    // halo rows (3x3, stride 1): one box of TM + 2 virtual pixels per kernel
    // row serves the three horizontal taps; the slot rounded up to 1024 bytes
    // so that every stage starts on a swizzle-atom boundary
    static constexpr uint32_t kAhTx = (BM * MS + 2) * BK * 2;
    static constexpr uint32_t kABh = (kAhTx + 1023u) / 1024u * 1024u;
    static constexpr uint32_t kTmemCols = 2 * MS * BN < 32 ? 32 : 2 * MS * BN;
    static_assert(kTmemCols <= 512, "TMEM holds 512 columns");
    static_assert(kSmemFixed + (size_t)kEpiWarps * kMaxResDepth * kStageBytes + 2 * (kAB + kBBytes) +
                          4096 * 4 * 2 <= kSmemMax,
                  "two stages, the deepest residual ring and the largest bias copy must fit");
};

struct Params {
    int M, C_out, taps, KW, kb_per_tap, num_kb;
    int num_m_tiles, num_n_tiles;
    int splits, kb_per_split;  // split-K: unit = tile * splits + split
    // split-K: fp32 partial tiles [tile][split][TM x BN] (chunk-blocked, see the
    // split-K epilogue) and one arrival counter per output tile (zeroed by the
    // host before the launch); NULL without a split
    float* part;
    unsigned* cnt;
    int OW, OHW, OH, S, P;
    // Halo rows (a_mode 2): output pixels are indexed on a virtual grid whose
    // rows are vw = OW + 2 wide (the two extra columns per row are computed
    // and discarded), M counts virtual pixels, and K runs over (kernel row,
    // channel block): num_kbh = 3 x kb_per_tap units of three taps each.
    // Without halo rows vw = OW.  vw_magic = floor((2^64 - 1) / vw) + 1 gives
    // v / vw as the high 64 bits of v * vw_magic (exact for v < 2^32).
    int vw;
    unsigned long long vw_magic;
    int num_kbh;
    // Rectangular tiles (a_mode 3, 1x1 convs with a pooled second output):
    // tile t = (n * rty + ty) * rtx + tx covers output rows ty * rh ... and
    // columns tx * rw ... of image n (rw = 2^rw_log2, rw * rh = 128), loaded as
    // one 4-D box; rtx_magic / rty_magic divide by rtx / rty as vw_magic does.
    int rw_log2, rh, rtx, rty;
    unsigned long long rtx_magic, rty_magic;
    void* y2;         // a_mode 3: NHWC [N][OH/2][OW/2][C_out], the 2x2/s2 average of y;
                      // y2_up: NHWC [N][2 OH][2 OW][C_out], the nearest 2x upsample of y
    int y2_up;
    void* y_nhwc;     // NCHW output: also an NHWC copy of y (the next conv's staged input), or NULL
    int a_mode;       // 0: tiled A (1x1/s1/p0); 1: im2col A; 2: im2col A with halo rows;
                      // 3: tiled A in rectangular tiles (1x1/s1/p0, pooled second output)
    int c_split;      // channels [c_split, C_in) come from the second A map (0: none)
    int out_layout;   // ACNN_NHWC or ACNN_NCHW for y and the residual
    int act, res_mode;
    const float* bias;
    const float* alpha;
    const void* res;
    void* y;
    int* status;
    long long budget;  // >0: give up a wait after this many polls; 0: after kTimeoutNs
    int stages;        // depth of the operand ring (2..kMaxStages)
    int res_depth;     // residual boxes in flight per epilogue warp (0: no residual)
    int b_resident;    // 1: all num_kb weight blocks loaded once, the ring carries A only
    int par_floats;    // NHWC epilogue: shared copy of bias [cpad] then alpha [cpad] (0: none)
    int ring_slots;    // 2 KB epilogue slots per epilogue warp (NHWC ring / NCHW transpose stage)
};

// Output pixel (row of the GEMM) v -> index of the real output pixel in
// [0, N*OH*OW), or -1 for a virtual column of a halo-row grid or a row past
// the end of the tile range.
// Rectangular tile: tile t -> (image, first row, first column).
// (A divisor of 1 has no 64-bit magic number: 2^64 wraps to 0.)
__device__ __forceinline__ void rect_tile(const Params& p, int t, int& n, int& y0, int& x0) {
    const int t2 = p.rtx == 1 ? t : (int)__umul64hi((unsigned long long)t, p.rtx_magic);  // t / rtx
    const int tx = t - t2 * p.rtx;
    n = p.rty == 1 ? t2 : (int)__umul64hi((unsigned long long)t2, p.rty_magic);  // t2 / rty
    y0 = (t2 - n * p.rty) * p.rh;
    x0 = tx << p.rw_log2;
}

__device__ __forceinline__ int real_pixel(const Params& p, int v) {
    if (v >= p.M) return -1;
    if (p.a_mode == 3) {
        int n, y0, x0;
        rect_tile(p, v >> 7, n, y0, x0);
        const int r = v & 127;
        const int oy = y0 + (r >> p.rw_log2), ox = x0 + (r & ((1 << p.rw_log2) - 1));
        return oy < p.OH && ox < p.OW ? (n * p.OH + oy) * p.OW + ox : -1;
    }
    if (p.a_mode != 2) return v;
    const int row = (int)__umul64hi((unsigned long long)v, p.vw_magic);  // v / vw
    const int j = v - row * p.vw;
    return j < p.OW ? row * p.OW + j : -1;
}

// The nearest 2x upsample of y as a second output: the 16-byte piece u of
// real output pixel m (row n * OH + oy, column ox) at channel col goes to the
// 2 x 2 block of pixels (2 oy + dy, 2 ox + dx), whose upsampled row index is
// 2 (n * OH + oy) + dy.
template <typename T>
__device__ __forceinline__ void store_up2(const Params& p, int m, int col, uint4 u) {
    const int row = m / p.OW, ox = m - row * p.OW;
    const long long W2 = 2ll * p.OW;
    T* up = static_cast<T*>(p.y2) + ((2ll * row) * W2 + 2 * ox) * p.C_out + col;
    *reinterpret_cast<uint4*>(up) = u;
    *reinterpret_cast<uint4*>(up + p.C_out) = u;
    *reinterpret_cast<uint4*>(up + W2 * p.C_out) = u;
    *reinterpret_cast<uint4*>(up + W2 * p.C_out + p.C_out) = u;
}

// Rows v0 .. v0 + 31 of one epilogue chunk -> real output pixels.  With
// rectangular tiles the tile's image and corner are decomposed once per chunk
// and a row then costs a shift and a mask; the other modes use real_pixel.
struct ChunkMap {
    int v0;
    int n, y0, x0, tr0;  // rectangular tiles: image, corner, first tile row of the chunk
};

__device__ __forceinline__ ChunkMap chunk_map(const Params& p, int v0) {
    ChunkMap c{v0, 0, 0, 0, 0};
    if (p.a_mode == 3 && v0 < p.M) {
        rect_tile(p, v0 >> 7, c.n, c.y0, c.x0);
        c.tr0 = v0 & 127;
    }
    return c;
}

__device__ __forceinline__ int map_row(const Params& p, const ChunkMap& c, int r) {
    if (p.a_mode != 3) return real_pixel(p, c.v0 + r);
    if (c.v0 >= p.M) return -1;
    const int tr = c.tr0 + r;
    const int oy = c.y0 + (tr >> p.rw_log2), ox = c.x0 + (tr & ((1 << p.rw_log2) - 1));
    return oy < p.OH && ox < p.OW ? (c.n * p.OH + oy) * p.OW + ox : -1;
}

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the same phase (returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Slow path of a bounded wait for the phase of `bar` with parity `parity`.
// Returns false if the CTA is aborting or this wait expired; on expiry it
// records the timeout in the device status word and raises the abort flag.
// Time is measured with the SM's cycle counter (cheap to read, unlike the
// global timer); kTimeoutCycles is ~4 s at the maximum SM clock.  With a poll
// budget (> 0) each poll is a non-blocking test, so the budget counts tests
// exactly (a try_wait may suspend the thread for a hardware-chosen time).
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag, long long budget,
                                             int* status) {
    long long t0 = -1;
    for (long long i = 1;; ++i) {
        if (budget > 0 ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
        bool expired = budget > 0 && i >= budget;
        if ((i & 255) == 0) {
            if (*abort_flag) return false;
            const long long now = clock64();
            if (t0 < 0) t0 = now;
            if (budget <= 0 && now - t0 > kTimeoutCycles) expired = true;
        }
        if (expired) {
            atomicCAS(status, 0, ACNN_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity,
                                           volatile int* abort_flag, const Params& p) {
    if (p.budget <= 0 && mbar_try_wait(bar, parity)) return true;
    return wait_phase_slow(bar, parity, abort_flag, p.budget, p.status);
}

// Bounded wait until the global counter *cnt reaches n (the splits of one
// output tile, run by CTAs that are all resident).  Returns false if the CTA
// is aborting or the wait expired (recorded like an mbarrier timeout).
__device__ __noinline__ bool wait_count(const unsigned* cnt, unsigned n, volatile int* abort_flag,
                                        const Params& p) {
    long long t0 = -1;
    for (long long i = 1;; ++i) {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
        if (v >= n) return true;
        bool expired = p.budget > 0 && i >= p.budget;
        if ((i & 255) == 0) {
            if (*abort_flag) return false;
            const long long now = clock64();
            if (t0 < 0) t0 = now;
            if (p.budget <= 0 && now - t0 > kTimeoutCycles) expired = true;
        }
        if (expired) {
            atomicCAS(p.status, 0, ACNN_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
        __nanosleep(64);
    }
}

// Time-bounded wait used only while draining after an abort.
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kDrainCycles) return;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// im2col load: coordinates {c, w, h, n} of the first pixel's window corner and
// the tap offsets {kx, ky} added to every pixel's position.
__device__ __forceinline__ void tma_load_im2col(uint32_t dst, const CUtensorMap* map,
                                                uint32_t bar, int c, int w, int h, int n,
                                                uint16_t off_w, uint16_t off_h) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.im2col.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2], {%7, %8};" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c), "r"(w), "r"(h), "r"(n),
        "h"(off_w), "h"(off_h)
        : "memory");
}

// 16-byte asynchronous global -> shared copy (L2 only); src_bytes = 0 writes
// zeros without reading.  Groups of copies are committed and waited on per
// thread.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until at most n (0..3, larger values act as 3) of this thread's
// committed groups are still pending.
__device__ __forceinline__ void cp_async_wait_newer(int n) {
    if (n <= 0) asm volatile("cp.async.wait_group 0;" ::: "memory");
    else if (n == 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
    else if (n == 2) asm volatile("cp.async.wait_group 2;" ::: "memory");
    else asm volatile("cp.async.wait_group 3;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// One lane of a converged warp (the lowest active one, the same lane on every
// call while all 32 are active) gets true.  The producer and MMA warps run
// their loops on all 32 lanes -- every wait, counter and coordinate warp-wide --
// and only the elected lane issues the TMA copies, MMAs and commits.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, 128 x N x 16, fp32 accumulate.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 op this thread issued so far completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one row per lane).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major operand whose rows are BK x 2
// bytes: BK = 64 -> 128-byte rows, 128-byte swizzle, 8-row core-matrix groups
// 1024 B apart; BK = 32 -> 64-byte rows, 64-byte swizzle, groups 512 B apart.
// Advancing the start address by 32 B steps K by 16 elements inside a row.
template <int BK> __device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    static_assert(BK == 64 || BK == 32, "k-block of 64 or 32 channels");
    constexpr uint64_t sbo = (uint64_t)BK * 2 * 8;
    constexpr uint64_t layout = BK == 64 ? 2 : 4;  // SWIZZLE_128B : SWIZZLE_64B
    return (uint64_t)((saddr & 0x3FFFFu) >> 4)  // start address >> 4
           | ((uint64_t)1 << 16)                // leading byte offset (unused here)
           | ((sbo >> 4) << 32)                 // stride byte offset: 8 rows
           | ((uint64_t)1 << 46)                // descriptor version (tcgen05)
           | (layout << 61);
}

// Descriptor of an operand that starts inside a swizzle atom (the halo-row A
// operand of horizontal tap kx starts kx rows into its stage): the tensor core
// takes the swizzle phase of each row from its absolute shared-memory address,
// the same address bits the TMA swizzled the rows by, so the plain descriptor
// at the shifted start is right (measured: also setting the matrix base offset
// field to the start's phase, bits 49-51, gives wrong sums).
template <int BK> __device__ __forceinline__ uint64_t smem_desc_at(uint32_t saddr) {
    return smem_desc<BK>(saddr);
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B both bf16 or
// both fp16, both K-major, N >> 3 and M >> 4 in their fields.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n, bool bf16) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

template <typename T> struct IsBf16 { static constexpr bool v = false; };
template <> struct IsBf16<__nv_bfloat16> { static constexpr bool v = true; };

// Two fp32 values -> two storage values (round to nearest even), lo at the lower address.
template <typename T> __device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <> __device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
template <> __device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
template <typename T> __device__ __forceinline__ void unpack2(uint32_t u, float& lo, float& hi);
template <> __device__ __forceinline__ void unpack2<__nv_bfloat16>(uint32_t u, float& lo, float& hi) {
    lo = __uint_as_float(u << 16);
    hi = __uint_as_float(u & 0xffff0000u);
}
template <> __device__ __forceinline__ void unpack2<__half>(uint32_t u, float& lo, float& hi) {
    __half2 h = *reinterpret_cast<__half2*>(&u);
    lo = __low2float(h);
    hi = __high2float(h);
}

// NCHW epilogue: the lane's 32 output channels (values v, channels ch0 ..,
// the first nj valid, nj a multiple of 8) of real pixel m also to the NHWC
// copy, as 16-byte pieces (the same rounding as the NCHW stores).
template <typename T>
__device__ __forceinline__ void store_nhwc_row(const Params& p, int m, int ch0, const float (&v)[32],
                                               int nj) {
    T* dst = static_cast<T*>(p.y_nhwc) + (long long)m * p.C_out + ch0;
#pragma unroll
    for (int k = 0; k < 4; ++k)
        if (8 * k < nj)
            *reinterpret_cast<uint4*>(dst + 8 * k) =
                make_uint4(pack2<T>(v[8 * k], v[8 * k + 1]), pack2<T>(v[8 * k + 2], v[8 * k + 3]),
                           pack2<T>(v[8 * k + 4], v[8 * k + 5]), pack2<T>(v[8 * k + 6], v[8 * k + 7]));
}

// Activation with the code fixed at compile time (no per-element branching).
// SiLU uses the fast exp and divide intrinsics: their error (a few fp32 ulp)
// is far below the fp16/bf16 storage rounding that follows.
template <int ACT> __device__ __forceinline__ float act_fixed(float v, float alpha) {
    if constexpr (ACT == ACNN_ACT_RELU) return fmaxf(v, 0.0f);
    else if constexpr (ACT == ACNN_ACT_SILU) return __fdividef(v, 1.0f + __expf(-v));
    else if constexpr (ACT == ACNN_ACT_PRELU) return v >= 0.0f ? v : alpha * v;
    else return v;
}

// The NHWC epilogue's form: the residual mode fixed at compile time (no
// residual term at all without one), the 32 biases and PReLU alphas of the
// chunk read from shared memory four at a time (bias[j], alpha[j]), the
// residual row read eight values at a time from its swizzled shared-memory
// row (16-byte piece j at rrow + ((j ^ swz) << 4)), and the result written
// over the accumulator values.
template <int ACT, int RES, typename T>
__device__ __forceinline__ void epi32_slot(float (&v)[32], const float* bias, const float* alpha,
                                           const uint8_t* rrow, uint32_t swz) {
#pragma unroll
    for (int j8 = 0; j8 < 4; ++j8) {
        float r[8];
        if constexpr (RES != ACNN_RES_NONE) {
            const uint4 u = *reinterpret_cast<const uint4*>(rrow + ((j8 ^ swz) << 4));
            unpack2<T>(u.x, r[0], r[1]);
            unpack2<T>(u.y, r[2], r[3]);
            unpack2<T>(u.z, r[4], r[5]);
            unpack2<T>(u.w, r[6], r[7]);
        }
#pragma unroll
        for (int j4 = 0; j4 < 8; j4 += 4) {
            const int j = j8 * 8 + j4;
            const float4 b4 = *reinterpret_cast<const float4*>(bias + j);
            float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if constexpr (ACT == ACNN_ACT_PRELU) a4 = *reinterpret_cast<const float4*>(alpha + j);
            const float bb[4] = {b4.x, b4.y, b4.z, b4.w};
            const float aa[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float x = v[j + k] + bb[k];
                if constexpr (RES == ACNN_RES_NONE) v[j + k] = act_fixed<ACT>(x, aa[k]);
                else if constexpr (RES == ACNN_RES_ADD_THEN_ACT)
                    v[j + k] = act_fixed<ACT>(x + r[j4 + k], aa[k]);
                else v[j + k] = act_fixed<ACT>(x, aa[k]) + r[j4 + k];
            }
        }
    }
}

template <int ACT, typename T>
__device__ __forceinline__ void epi32_slot_act(int res_mode, float (&v)[32], const float* bias,
                                               const float* alpha, const uint8_t* rrow,
                                               uint32_t swz) {
    if (res_mode == ACNN_RES_ADD_THEN_ACT)
        epi32_slot<ACT, ACNN_RES_ADD_THEN_ACT, T>(v, bias, alpha, rrow, swz);
    else if (res_mode == ACNN_RES_ACT_THEN_ADD)
        epi32_slot<ACT, ACNN_RES_ACT_THEN_ADD, T>(v, bias, alpha, rrow, swz);
    else epi32_slot<ACT, ACNN_RES_NONE, T>(v, bias, alpha, rrow, swz);
}

template <typename T>
__device__ __forceinline__ void epi32_slot_mode(int act, int res_mode, float (&v)[32],
                                                const float* bias, const float* alpha,
                                                const uint8_t* rrow, uint32_t swz) {
    switch (act) {  // both uniform across the CTA
    case ACNN_ACT_RELU: epi32_slot_act<ACNN_ACT_RELU, T>(res_mode, v, bias, alpha, rrow, swz); break;
    case ACNN_ACT_SILU: epi32_slot_act<ACNN_ACT_SILU, T>(res_mode, v, bias, alpha, rrow, swz); break;
    case ACNN_ACT_PRELU: epi32_slot_act<ACNN_ACT_PRELU, T>(res_mode, v, bias, alpha, rrow, swz); break;
    default: epi32_slot_act<ACNN_ACT_NONE, T>(res_mode, v, bias, alpha, rrow, swz); break;
    }
}

// ---------------------------------------------------------------- the kernel
template <int BN, int MS, int BK, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    igemm_conv_kernel(const __grid_constant__ CUtensorMap tmap_a,
                      const __grid_constant__ CUtensorMap tmap_a2,
                      const __grid_constant__ CUtensorMap tmap_b, const Params p) {
    using C = Cfg<BN, MS, BK>;
    constexpr int TM = BM * MS;  // output pixels per tile
    extern __shared__ uint8_t smem_raw[];
    // The swizzled tiles need a 1024-aligned window; the host sized the
    // allocation on that assumption.  A misaligned window is reported, not used.
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) atomicCAS(p.status, 0, ACNN_ERR_UNSUPPORTED);
        return;
    }
    const int S = p.stages;
    const bool bres = p.b_resident != 0;
    const bool halo = p.a_mode == 2;
    // per stage: A (one box; TM + 2 virtual pixels with halo rows) and, unless
    // the weights are resident, B (one tap's block; three with halo rows)
    const uint32_t a_slot = halo ? C::kABh : C::kAB;
    const uint32_t b_slot = halo ? 3u * C::kBBytes : C::kBBytes;
    uint8_t* sA = smem_raw;
    uint8_t* sB = sA + (size_t)S * a_slot;  // B ring (S slots) or all num_kb resident B blocks
    // epilogue slots: kEpiWarps x ring_slots x 2 KB, 1024-aligned
    uint8_t* sR = sB + (bres ? (size_t)p.num_kb * C::kBBytes : (size_t)S * b_slot);
    float* sP = reinterpret_cast<float*>(sR + (size_t)kEpiWarps * p.ring_slots * kStageBytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sP + p.par_floats);
    // bars: full[S], empty[S], tmem_full[2], tmem_empty[2], drain, weights
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * kMaxStages + 6);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
    const uint32_t wres_bar = bar0 + 8u * (2 * S + 5);  // resident weights landed

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), kEpiWarps);  // one arrival per epilogue warp
        }
        mbar_init(drain_bar, 1);
        mbar_init(wres_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tmap_a);
        if (p.c_split) prefetch_tmap(&tmap_a2);
        prefetch_tmap(&tmap_b);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    // everything above (barriers, TMEM, tensor-map prefetch) may overlap the
    // previous kernel on the stream; every global access below comes after it
    griddep_wait();

    // a work unit is one output tile and one K range (the whole K without split-K)
    const int num_tiles = p.num_m_tiles * p.num_n_tiles * p.splits;

    if (warp == 0) {
        {
            // ------------------------------------------------ TMA producer
            // (all 32 lanes walk the loop; the elected lane issues)
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = true;
            if (bres) {
                // every weight block of the (single) column tile, once
                if (elect_one()) {
                    mbar_arrive_expect_tx(wres_bar, (uint32_t)p.num_kb * C::kBBytes);
                    int tap = 0, c0 = 0;
                    for (int kb = 0; kb < p.num_kb; ++kb) {
                        tma_load_3d(smem_u32(sB + kb * C::kBBytes), &tmap_b, wres_bar, c0, tap, 0);
                        c0 += BK;
                        if (c0 >= p.kb_per_tap * BK) {
                            c0 = 0;
                            ++tap;
                        }
                    }
                }
                __syncwarp();
            }
            const uint32_t stage_tx =
                halo ? C::kAhTx + (bres ? 0u : 3u * C::kBBytes) : C::kAB + (bres ? 0u : C::kBBytes);
            const int num_k = halo ? p.num_kbh : p.num_kb;
            const int OHV = p.OHW / p.OW * p.vw;  // virtual pixels per image
            for (int unit = blockIdx.x; ok && unit < num_tiles; unit += gridDim.x) {
                const int tile = unit / p.splits, split = unit - tile * p.splits;
                const int m0 = (tile / p.num_n_tiles) * TM;
                const int n0 = (tile % p.num_n_tiles) * BN;
                const int kb0 = split * p.kb_per_split;
                const int kb1 = min(num_k, kb0 + p.kb_per_split);
                // window corner of the tile's first (virtual) output pixel
                const int img = m0 / OHV, r = m0 % OHV;
                const int wc = (r % p.vw) * p.S - p.P, hc = (r / p.vw) * p.S - p.P;
                // rectangular tile: image and corner of the 4-D box
                int rn = 0, ry0 = 0, rx0 = 0;
                if (p.a_mode == 3) rect_tile(p, m0 >> 7, rn, ry0, rx0);
                if (halo) {
                    // unit kb = (kernel row ky, channel block cb): one A box of
                    // TM + 2 virtual pixels at tap (0, ky), the B blocks of taps
                    // (ky, 0..2) unless resident
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!__all_sync(0xffffffffu,
                                        wait_phase(empty_bar(stage), phase ^ 1u, abort_flag, p))) {
                            ok = false;
                            break;
                        }
                        const int ky = kb / p.kb_per_tap, cb = kb - ky * p.kb_per_tap;
                        const int c0h = cb * BK;
                        const uint32_t fb = full_bar(stage);
                        const uint32_t a_dst = smem_u32(sA + (size_t)stage * a_slot);
                        const bool second = p.c_split && c0h >= p.c_split;
                        const CUtensorMap* am = second ? &tmap_a2 : &tmap_a;
                        const int ca = second ? c0h - p.c_split : c0h;
                        if (elect_one()) {
                            mbar_arrive_expect_tx(fb, stage_tx);
                            tma_load_im2col(a_dst, am, fb, ca, wc, hc, img, (uint16_t)0, (uint16_t)ky);
                            if (!bres)
                                for (int kx = 0; kx < 3; ++kx)
                                    tma_load_3d(smem_u32(sB + (size_t)stage * b_slot + kx * C::kBBytes),
                                                &tmap_b, fb, c0h, ky * 3 + kx, n0);
                        }
                        __syncwarp();
                        issued_mask |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    continue;
                }
                // (tap, channel block) of k-block kb0, then stepped without divisions
                int tap = kb0 / p.kb_per_tap;
                int c0 = (kb0 - tap * p.kb_per_tap) * BK;
                int ky = tap / p.KW, kx = tap - ky * p.KW;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!__all_sync(0xffffffffu,
                                    wait_phase(empty_bar(stage), phase ^ 1u, abort_flag, p))) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full_bar(stage);
                    const uint32_t a_dst = smem_u32(sA + (size_t)stage * a_slot);
                    // a folded concat: channel blocks from c_split on come from
                    // the second source (c_split is a multiple of BK)
                    const bool second = p.c_split && c0 >= p.c_split;
                    const CUtensorMap* am = second ? &tmap_a2 : &tmap_a;
                    const int ca = second ? c0 - p.c_split : c0;
                    if (elect_one()) {
                        mbar_arrive_expect_tx(fb, stage_tx);
                        if (p.a_mode == 0)
                            tma_load_2d(a_dst, am, fb, ca, m0);
                        else if (p.a_mode == 3)
                            tma_load_4d(a_dst, am, fb, ca, rx0, ry0, rn);
                        else
                            tma_load_im2col(a_dst, am, fb, ca, wc, hc, img, (uint16_t)kx,
                                            (uint16_t)ky);
                        if (!bres)
                            tma_load_3d(smem_u32(sB + (size_t)stage * b_slot), &tmap_b, fb, c0, tap,
                                        n0);
                    }
                    __syncwarp();
                    issued_mask |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    c0 += BK;
                    if (c0 >= p.kb_per_tap * BK) {
                        c0 = 0;
                        ++tap;
                        if (++kx == p.KW) {
                            kx = 0;
                            ++ky;
                        }
                    }
                }
            }
            if (!ok) {
                // let every copy this warp started land before the CTA exits
                for (int s = 0; s < S; ++s)
                    if (issued_mask & (1u << s)) wait_drain(full_bar(s), (issued_parity >> s) & 1u);
                if (bres) wait_drain(wres_bar, 0);
            }
        }
        __syncwarp();
        // this CTA's loads are all issued: the next kernel on the stream may
        // launch (its CTAs start as SMs free up and wait for this grid to end)
        griddep_launch_dependents();
    } else if (warp == 1) {
        {
            // ------------------------------------------------ MMA issuer
            // (all 32 lanes walk the loop; the elected lane -- lane 0 of the
            // converged warp every time -- issues the MMAs and their commits)
            constexpr uint32_t idesc = make_idesc(BM, BN, IsBf16<T>::v);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = !bres || __all_sync(0xffffffffu, wait_phase(wres_bar, 0, abort_flag, p));
            for (int unit = blockIdx.x; ok && unit < num_tiles; unit += gridDim.x) {
                const int split = unit % p.splits;
                const int kb0 = split * p.kb_per_split;
                const int kb1 = min(halo ? p.num_kbh : p.num_kb, kb0 + p.kb_per_split);
                if (!__all_sync(0xffffffffu,
                                wait_phase(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * MS * BN);
                if (halo) {
                    // unit kb = (ky, cb): horizontal tap kx reads the A box from
                    // row kx on (row block ms from row ms * 128 + kx), B tap (ky, kx)
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!__all_sync(0xffffffffu,
                                        wait_phase(full_bar(stage), phase, abort_flag, p))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const int ky = kb / p.kb_per_tap, cb = kb - ky * p.kb_per_tap;
                        const uint32_t a_base = smem_u32(sA + (size_t)stage * a_slot);
                        if (elect_one()) {
#pragma unroll
                            for (int kx = 0; kx < 3; ++kx) {
                                const uint32_t b_addr =
                                    bres ? smem_u32(sB + (size_t)((ky * 3 + kx) * p.kb_per_tap + cb) *
                                                             C::kBBytes)
                                         : smem_u32(sB + (size_t)stage * b_slot + kx * C::kBBytes);
                                const uint64_t bdesc = smem_desc<BK>(b_addr);
#pragma unroll
                                for (int ms = 0; ms < MS; ++ms) {
                                    const uint64_t adesc =
                                        smem_desc_at<BK>(a_base + (uint32_t)((ms * BM + kx) * BK * 2));
#pragma unroll
                                    for (int k = 0; k < BK / 16; ++k)
                                        mma_f16(d_tmem + (uint32_t)(ms * BN), adesc + 2u * k,
                                                bdesc + 2u * k, idesc,
                                                (kb != kb0 || kx != 0 || k != 0) ? 1u : 0u);
                                }
                            }
                            mma_commit(empty_bar(stage));  // frees the slot once these MMAs finish
                        }
                        __syncwarp();
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    if (elect_one()) mma_commit(tfull_bar(acc));
                    __syncwarp();
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1u;
                    continue;
                }
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!__all_sync(0xffffffffu, wait_phase(full_bar(stage), phase, abort_flag, p))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bdesc = smem_desc<BK>(smem_u32(
                        bres ? sB + (size_t)kb * C::kBBytes : sB + (size_t)stage * b_slot));
                    const uint64_t adesc0 = smem_desc<BK>(smem_u32(sA + (size_t)stage * a_slot));
                    if (elect_one()) {
#pragma unroll
                        for (int ms = 0; ms < MS; ++ms) {
                            // the row blocks of a stage lie kABytes apart (>> 4 in the descriptor)
                            const uint64_t adesc = adesc0 + (uint64_t)(ms * (C::kABytes >> 4));
#pragma unroll
                            for (int k = 0; k < BK / 16; ++k)
                                mma_f16(d_tmem + (uint32_t)(ms * BN), adesc + 2u * k,
                                        bdesc + 2u * k, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
                        }
                        mma_commit(empty_bar(stage));  // frees the slot once these MMAs finish
                    }
                    __syncwarp();
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (elect_one()) mma_commit(tfull_bar(acc));  // accumulator ready for the epilogue
                __syncwarp();
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok && lane == 0) {
                mma_commit(drain_bar);  // wait for every MMA this warp issued
                wait_drain(drain_bar, 0);
            }
        }
        __syncwarp();
    } else if (p.part) {
        // ---------------------------------------------------- epilogue warps, split-K
        // Every split of an output tile writes its raw fp32 accumulators to its
        // partial tile in the workspace and counts itself in on the tile's
        // counter; after all its units, a CTA waits for the tiles it touched
        // and finishes 1/S of each one's 32 x 32 blocks: the sum of all partial
        // tiles in split order (so the result does not depend on arrival
        // order), then the bias / residual / activation / store epilogue.
        // Partial tiles are chunk-blocked: the 32 x 32 block of
        // (row block ms, chunk ci, lane quarter q) holds lane l's columns
        // 4j..4j+3 at float offset (j * 32 + l) * 4, so each warp store or load
        // instruction moves 512 contiguous bytes.
        const int q = warp & 3;
        const int e = warp - 2;
        const int grp = e >> 2;
        const int S = p.splits;
        const T* res = static_cast<const T*>(p.res);
        T* y = static_cast<T*>(p.y);
        const bool prelu = p.act == ACNN_ACT_PRELU;
        const uint32_t swz = (uint32_t)((lane >> 1) & 3);
        const int crow = lane >> 2, cpiece = lane & 3;
        auto piece = [](int r, int j) { return r * 64 + ((j ^ ((r >> 1) & 3)) << 4); };
        uint8_t* slot = sR + (size_t)e * kStageBytes;  // one slot per warp (NHWC output)
        volatile int* met_flag = abort_flag + 1;  // all splits of the tile arrived
        const int cpad = prelu ? p.par_floats / 2 : p.par_floats;
        for (int i = threadIdx.x - 64; i < cpad; i += 32 * kEpiWarps) {
            sP[i] = (p.bias && i < p.C_out) ? __ldg(p.bias + i) : 0.f;
            if (prelu) sP[cpad + i] = i < p.C_out ? __ldg(p.alpha + i) : 0.f;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
        constexpr int kChunksPerTile = MS * (BN / 32);
        auto block_of = [&](int tile, int split, int ms, int ci) {
            return p.part +
                   ((((size_t)tile * S + split) * kChunksPerTile + ms * (BN / 32) + ci) * 4 + q) *
                       1024;
        };
        // Phase 1: every unit of this CTA -- MMAs, partial tile, count in.
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int unit = blockIdx.x; unit < num_tiles; unit += gridDim.x) {
            const int tile = unit / S, split = unit - tile * S;
            const int n0 = (tile % p.num_n_tiles) * BN;
            ok = __all_sync(0xffffffffu, wait_phase(tfull_bar(acc), acc_phase, abort_flag, p));
            if (!ok) break;
            tc_fence_after();
            const int nch = ((p.C_out - n0 < BN ? p.C_out - n0 : BN) + 31) >> 5;
            for (int i = grp; i < MS * nch; i += kEpiGroups) {
                const int ms = i / nch, ci = i - ms * nch;
                float v[32];
                tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) +
                              (uint32_t)(acc * MS * BN + ms * BN + ci * 32),
                          v);
                float* blk = block_of(tile, split, ms, ci);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<float4*>(blk + (j * 32 + lane) * 4) =
                        make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
            // every epilogue warp has written this split's partial tile
            asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
            if (e == 0 && lane == 0) {
                __threadfence();
                atomicAdd(p.cnt + tile, 1u);
            }
        }
        // Phase 2: for each of this CTA's units (t, sp), once all S splits of
        // tile t have counted in, finish the tile's 32 x 32 blocks
        // b = sp, sp + S, ...: the sum of every split's partial tile (read from
        // L2) in split order, then the epilogue.  No CTA waits before it has
        // written all its partial tiles and every CTA is resident (grid <= #SMs,
        // one CTA per SM), so the waits always end.
        for (int unit = blockIdx.x; ok && unit < num_tiles; unit += gridDim.x) {
            const int tile = unit / S, split = unit - tile * S;
            const int m0 = (tile / p.num_n_tiles) * TM;
            const int n0 = (tile % p.num_n_tiles) * BN;
            const int nch = ((p.C_out - n0 < BN ? p.C_out - n0 : BN) + 31) >> 5;
            if (e == 0 && lane == 0)
                *met_flag = wait_count(p.cnt + tile, (unsigned)S, abort_flag, p) ? 1 : 0;
            asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
            if (!*met_flag) break;
            __threadfence();  // the other splits' partial tiles are visible
            // finish one 32 x 32 block (row block ms, chunk ci, lane quarter qb)
            // of the tile from its split-order sum t
            auto finish = [&](int ms, int ci, int qb, float (&t)[32]) {
                const int c = ci * 32;
                const int row0 = m0 + ms * BM + qb * 32;
                if (p.out_layout == ACNN_NHWC) {
                    // residual row of this lane into its slot row, then the
                    // NHWC epilogue arithmetic and coalesced stores
                    const int mr = real_pixel(p, row0 + lane);
                    if (p.res_mode != ACNN_RES_NONE) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const bool in = mr >= 0 && n0 + c + j * 8 < p.C_out;
                            const T* src = res + (in ? (long long)mr * p.C_out + n0 + c + j * 8 : 0);
                            cp_async16(smem_u32(slot + lane * 64 + ((j ^ swz) << 4)), src, in ? 16u : 0u);
                        }
                        cp_async_commit();
                        cp_async_wait_newer(0);
                    }
                    epi32_slot_mode<T>(p.act, p.res_mode, t, sP + n0 + c, sP + cpad + n0 + c,
                                       slot + lane * 64, swz);
                    uint8_t* orow = slot + lane * 64;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<uint4*>(orow + ((j ^ swz) << 4)) = make_uint4(
                            pack2<T>(t[8 * j + 0], t[8 * j + 1]), pack2<T>(t[8 * j + 2], t[8 * j + 3]),
                            pack2<T>(t[8 * j + 4], t[8 * j + 5]), pack2<T>(t[8 * j + 6], t[8 * j + 7]));
                    __syncwarp();
                    const int col = n0 + c + cpiece * 8;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int rr = 8 * k + crow;
                        const uint4 u = *reinterpret_cast<const uint4*>(slot + piece(rr, cpiece));
                        const int mo = real_pixel(p, row0 + rr);
                        if (mo >= 0 && col < p.C_out) {
                            *reinterpret_cast<uint4*>(y + (long long)mo * p.C_out + col) = u;
                            if (p.y2_up) store_up2<T>(p, mo, col, u);
                        }
                    }
                    __syncwarp();  // the slot is read out before the next block reuses it
                } else {
                    const int mr = real_pixel(p, row0 + lane);
                    const bool valid = mr >= 0;
                    const int m = valid ? mr : 0;
                    const int img = m / p.OHW;
                    const long long base = (long long)img * p.C_out * p.OHW + (m - img * p.OHW);
                    const bool pre = p.res_mode == ACNN_RES_ADD_THEN_ACT;
                    const int nj = p.C_out - (n0 + c) < 32 ? p.C_out - (n0 + c) : 32;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (j >= nj) break;
                        const int ch = n0 + c + j;
                        const long long idx = base + (long long)ch * p.OHW;
                        const float rv =
                            (p.res_mode != ACNN_RES_NONE && valid) ? to_f32(res[idx]) : 0.f;
                        const float x = t[j] + sP[ch];
                        const float al = prelu ? sP[cpad + ch] : 0.f;
                        const float o = pre ? apply_act(p.act, x + rv, al) : apply_act(p.act, x, al) + rv;
                        if (valid) y[idx] = from_f32<T>(o);
                    }
                }
            };
            // add partial tile sp's values of this lane in block (ms, ci, qb)
            auto add_part = [&](float (&t)[32], int sp, int ms, int ci, int qb) {
                const float* blk = p.part +
                    ((((size_t)tile * S + sp) * kChunksPerTile + ms * (BN / 32) + ci) * 4 + qb) * 1024;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 u = __ldcg(reinterpret_cast<const float4*>(blk + (j * 32 + lane) * 4));
                    if (sp == 0) {
                        t[4 * j] = u.x; t[4 * j + 1] = u.y; t[4 * j + 2] = u.z; t[4 * j + 3] = u.w;
                    } else {
                        t[4 * j] += u.x; t[4 * j + 1] += u.y; t[4 * j + 2] += u.z; t[4 * j + 3] += u.w;
                    }
                }
            };
            const int nblk = MS * nch * 4;
            for (int b = split + S * e; b < nblk; b += S * kEpiWarps) {
                const int qb = b & 3, i = b >> 2;
                const int ms = i / nch, ci = i - ms * nch;
                float t[32];
                for (int sp = 0; sp < S; ++sp) add_part(t, sp, ms, ci, qb);
                finish(ms, ci, qb, t);
            }
            // every warp is done with this unit before the flag is reused
            asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
        }
        cp_async_wait_newer(0);
    } else if (p.out_layout == ACNN_NHWC) {
        // ---------------------------------------------------- epilogue warps, NHWC
        // Warp e (0..11) owns the 32 rows of its TMEM lane quarter (warp % 4)
        // and every third 32-channel chunk of each tile (group e / 4 picks
        // which), in (row block, channel) order.
        // Its chunks form one stream across tiles.  Each chunk uses one 2 KB
        // slot of the warp's ring in shared memory (32 rows x 64 B, 16-byte
        // pieces swizzled by row so that both row-wise and column-wise accesses
        // are free of bank conflicts):
        //   * with a residual, the ring has res_depth slots and the residual
        //     box of a chunk is copied in by cp.async up to res_depth chunks
        //     ahead (across tile boundaries), eight 64-byte rows per warp
        //     instruction;
        //   * the result of the chunk is written over its row of the slot, then
        //     read back eight rows per instruction and stored with 16-byte
        //     stores (rows >= M and channels >= C_out are skipped);
        //   * the bias and PReLU alpha come from a shared-memory copy.
        const int q = warp & 3;
        const int e = warp - 2;
        const int grp = e >> 2;
        const int RD = p.res_depth;  // 0 without a residual
        const int nnt = p.num_n_tiles;
        uint8_t* ring = sR + (size_t)e * (RD > 0 ? RD : 1) * kStageBytes;
        const T* res = static_cast<const T*>(p.res);
        T* y = static_cast<T*>(p.y);
        const bool prelu = p.act == ACNN_ACT_PRELU;
        const uint32_t swz = (uint32_t)((lane >> 1) & 3);  // swizzle of this lane's row
        const int crow = lane >> 2, cpiece = lane & 3;     // row-major copy pattern
        // byte offset of 16-byte piece j of row r inside a slot
        auto piece = [](int r, int j) { return r * 64 + ((j ^ ((r >> 1) & 3)) << 4); };
        // A cursor walks this warp's chunks: tile t (column tile nt = t % nnt),
        // row block ms, 32-channel chunk ci within the row block.
        const int nch_full = BN / 32;
        const int nch_last = ((p.C_out - (nnt - 1) * BN) + 31) >> 5;  // ragged last column tile
        struct Cursor {
            int t, nt, ms, ci;
        };
        auto settle = [&](Cursor& c) {  // carry ci into ms, then into the next tile
            while (c.t < num_tiles) {
                const int nch = c.nt == nnt - 1 ? nch_last : nch_full;
                while (c.ci >= nch) {
                    c.ci -= nch;
                    ++c.ms;
                }
                if (c.ms < MS) break;
                c.t += gridDim.x;
                c.nt = nnt == 1 ? 0 : c.t % nnt;
                c.ms = 0;
                c.ci = grp;
            }
        };
        // residual cursor
        Cursor rc{(int)blockIdx.x, nnt == 1 ? 0 : (int)blockIdx.x % nnt, 0, grp};
        settle(rc);
        int pend = 0, wb = 0, rb = 0;
        auto refill = [&]() {
            while (pend < RD && rc.t < num_tiles) {
                const int row0 = (nnt == 1 ? rc.t : rc.t / nnt) * TM + rc.ms * BM + q * 32;
                const int col = rc.nt * BN + rc.ci * 32 + cpiece * 8;
                const uint32_t sl = smem_u32(ring + wb * kStageBytes);
                const ChunkMap cm = chunk_map(p, row0);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = 8 * k + crow;
                    const int mr = map_row(p, cm, r);
                    const bool in = mr >= 0 && col < p.C_out;
                    const T* src = res + (in ? (long long)mr * p.C_out + col : 0);
                    cp_async16(sl + piece(r, cpiece), src, in ? 16u : 0u);
                }
                cp_async_commit();
                wb = wb + 1 == RD ? 0 : wb + 1;
                ++pend;
                rc.ci += kEpiGroups;
                settle(rc);
            }
        };
        // bias (and PReLU alpha) of every column, zero past C_out, copied once
        // into shared memory by the epilogue warps, which then sync among
        // themselves (named barrier 1)
        const int cpad = prelu ? p.par_floats / 2 : p.par_floats;
        for (int i = threadIdx.x - 64; i < cpad; i += 32 * kEpiWarps) {
            sP[i] = (p.bias && i < p.C_out) ? __ldg(p.bias + i) : 0.f;
            if (prelu) sP[cpad + i] = i < p.C_out ? __ldg(p.alpha + i) : 0.f;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
        refill();
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {  // splits == 1
            const int mt = nnt == 1 ? tile : tile / nnt;
            const int m0 = mt * TM;
            const int n0 = (tile - mt * nnt) * BN;
            const int nch = ((p.C_out - n0 < BN ? p.C_out - n0 : BN) + 31) >> 5;
            const int nchunks = MS * nch;  // chunk i: row block i / nch, channels (i % nch) * 32
            const bool ok = __all_sync(0xffffffffu, wait_phase(tfull_bar(acc), acc_phase, abort_flag, p));
            if (!ok) break;
            tc_fence_after();
            int ms = 0, ci = grp;
            for (int i = grp; i < nchunks; i += kEpiGroups) {
                while (ci >= nch) {
                    ci -= nch;
                    ++ms;
                }
                const int c = ci * 32;
                const int msc = ms;
                ci += kEpiGroups;
                const int row0 = m0 + ms * BM + q * 32;
                float v[32];
                tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) +
                              (uint32_t)(acc * MS * BN + msc * BN + c),
                          v);
                uint8_t* slot = ring + (RD > 0 ? rb : 0) * kStageBytes;
                if (RD > 0) {
                    // this chunk's box is the oldest in flight: let the newer
                    // pend - 1 stay pending, then see every lane's part of it
                    cp_async_wait_newer(pend - 1);
                    __syncwarp();
                    rb = rb + 1 == RD ? 0 : rb + 1;
                    --pend;
                }
                epi32_slot_mode<T>(p.act, RD > 0 ? p.res_mode : ACNN_RES_NONE, v, sP + n0 + c,
                                   sP + cpad + n0 + c, slot + lane * 64, swz);
                // this lane's row of results over its row of the slot
                uint8_t* orow = slot + lane * 64;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<uint4*>(orow + ((j ^ swz) << 4)) = make_uint4(
                        pack2<T>(v[8 * j + 0], v[8 * j + 1]), pack2<T>(v[8 * j + 2], v[8 * j + 3]),
                        pack2<T>(v[8 * j + 4], v[8 * j + 5]), pack2<T>(v[8 * j + 6], v[8 * j + 7]));
                __syncwarp();
                // eight rows per instruction out to y
                const int col = n0 + c + cpiece * 8;
                const ChunkMap cm = chunk_map(p, row0);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int rr = 8 * k + crow;
                    const uint4 u = *reinterpret_cast<const uint4*>(slot + piece(rr, cpiece));
                    const int mo = map_row(p, cm, rr);
                    if (mo >= 0 && col < p.C_out) {
                        *reinterpret_cast<uint4*>(y + (long long)mo * p.C_out + col) = u;
                        if (p.y2_up) store_up2<T>(p, mo, col, u);
                    }
                }
                if (p.y2 && !p.y2_up) {
                    // pooled second output (rectangular tiles): a chunk holds
                    // 32 / rw >= 2 whole tile rows, i.e. 8 whole 2x2 windows;
                    // lane l averages the 16-byte piece l & 3 (8 channels) of
                    // window l >> 2 from the window's four stored rows of the
                    // slot, as the 2x2/s2 average pool does:
                    // ((tl + tr) + bl) + br in fp32, times 0.25, rounded once
                    const int rw = 1 << p.rw_log2;
                    const int w = lane >> 2, j = lane & 3;
                    const int half = rw >> 1;  // windows per pair of pixel rows
                    const int rtl = (w / half) * 2 * rw + 2 * (w % half);  // top-left chunk row
                    const int tr = cm.tr0 + rtl;
                    const int oy = cm.y0 + (tr >> p.rw_log2), ox = cm.x0 + (tr & (rw - 1));
                    if (row0 < p.M && oy < p.OH && ox < p.OW && n0 + c + 8 * j < p.C_out) {
                        T* yp = static_cast<T*>(p.y2) +
                                ((long long)(cm.n * (p.OH >> 1) + (oy >> 1)) * (p.OW >> 1) +
                                 (ox >> 1)) * p.C_out +
                                n0 + c + 8 * j;
                        const int rows[4] = {rtl, rtl + 1, rtl + rw, rtl + rw + 1};
                        float acc[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint4 u = *reinterpret_cast<const uint4*>(slot + piece(rows[k], j));
                            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                float lo, hi;
                                unpack2<T>(w4[e], lo, hi);
                                acc[2 * e] = __fadd_rn(acc[2 * e], lo);
                                acc[2 * e + 1] = __fadd_rn(acc[2 * e + 1], hi);
                            }
                        }
                        *reinterpret_cast<uint4*>(yp) = make_uint4(
                            pack2<T>(__fmul_rn(acc[0], 0.25f), __fmul_rn(acc[1], 0.25f)),
                            pack2<T>(__fmul_rn(acc[2], 0.25f), __fmul_rn(acc[3], 0.25f)),
                            pack2<T>(__fmul_rn(acc[4], 0.25f), __fmul_rn(acc[5], 0.25f)),
                            pack2<T>(__fmul_rn(acc[6], 0.25f), __fmul_rn(acc[7], 0.25f)));
                    }
                }
                __syncwarp();  // the slot is read out before a refill overwrites it
                refill();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        cp_async_wait_newer(0);  // no copy into shared memory outlives the CTA
    } else {
        // ---------------------------------------------------- epilogue warps, NCHW
        // Same row/chunk split as above; lane l holds output pixel m0 + 32q + l.
        // A chunk whose 32 pixels lie in one image and start on an 8-pixel
        // boundary goes through the warp's shared-memory slot: its residual (if
        // any) comes in as 16-byte runs of 8 pixels of one channel and is read
        // back one pixel per lane; the result is written [channel][pixel] and
        // leaves as 16-byte runs (4 loads and 4 stores a lane instead of 32).
        // Other chunks take the per-element path: each of the 32 channel planes
        // read and written by 32 consecutive pixels.
        // Bias and alpha come from the shared copy.
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int grp = (warp - 2) >> 2;
        const int row = q * 32 + lane;
        const T* res = static_cast<const T*>(p.res);
        T* y = static_cast<T*>(p.y);
        const bool has_res = p.res_mode != ACNN_RES_NONE;
        const bool pre = p.res_mode == ACNN_RES_ADD_THEN_ACT;
        const bool prelu = p.act == ACNN_ACT_PRELU;
        const int cpad = prelu ? p.par_floats / 2 : p.par_floats;
        uint16_t* slot = reinterpret_cast<uint16_t*>(sR + (size_t)(warp - 2) * kStageBytes);
        const bool vec_ok = p.ring_slots > 0 && p.OHW % 8 == 0;
        for (int i = threadIdx.x - 64; i < cpad; i += 32 * kEpiWarps) {
            sP[i] = (p.bias && i < p.C_out) ? __ldg(p.bias + i) : 0.f;
            if (prelu) sP[cpad + i] = i < p.C_out ? __ldg(p.alpha + i) : 0.f;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kEpiWarps) : "memory");
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {  // splits == 1
            const int m0 = (tile / p.num_n_tiles) * TM;
            const int n0 = (tile % p.num_n_tiles) * BN;
            // every lane waits (acquiring the accumulator); the warp then agrees,
            // so the warp-collective TMEM loads below run converged or not at all
            const bool ok = __all_sync(0xffffffffu, wait_phase(tfull_bar(acc), acc_phase, abort_flag, p));
            if (!ok) break;
            tc_fence_after();
            const int nch = ((p.C_out - n0 < BN ? p.C_out - n0 : BN) + 31) >> 5;
            for (int i = grp; i < MS * nch; i += kEpiGroups) {
                const int ms = i / nch, c = (i - ms * nch) * 32;
                const int mr = real_pixel(p, m0 + ms * BM + row);
                const bool valid = mr >= 0;
                const int m = valid ? mr : 0;
                const int img = m / p.OHW;
                const long long base = (long long)img * p.C_out * p.OHW + (m - img * p.OHW);
                float v[32];
                tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) +
                              (uint32_t)(acc * MS * BN + ms * BN + c),
                          v);
                const int nj = p.C_out - (n0 + c) < 32 ? p.C_out - (n0 + c) : 32;
                // the chunk's 32 pixels: all in range, one image, 8-aligned start
                // (real pixels of the chunk's first and last rows: consecutive
                // when no virtual column of a halo-row grid lies between them)
                const int r0 = real_pixel(p, m0 + ms * BM + q * 32);
                const int r31 = real_pixel(p, m0 + ms * BM + q * 32 + 31);
                const int img0 = r0 / p.OHW;
                const bool vec = vec_ok && r0 >= 0 && r31 == r0 + 31 && r31 / p.OHW == img0 &&
                                 (r0 - img0 * p.OHW) % 8 == 0;
                if (vec) {
                    const long long base0 = (long long)img0 * p.C_out * p.OHW + (r0 - img0 * p.OHW);
                    if (has_res) {
                        // the chunk's residual, [channel][pixel] in the slot
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int piece = lane + 32 * k, j = piece >> 2, pb = piece & 3;
                            if (j < nj)
                                *reinterpret_cast<uint4*>(slot + j * 32 + pb * 8) =
                                    *reinterpret_cast<const uint4*>(
                                        res + base0 + (long long)(n0 + c + j) * p.OHW + pb * 8);
                        }
                        __syncwarp();
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int ch = n0 + c + j;  // < the padded bias copy
                        const float al = prelu ? sP[cpad + ch] : 0.f;
                        float o;
                        if (has_res) {
                            uint16_t rb = slot[j * 32 + lane];
                            const float rv = j < nj ? to_f32(*reinterpret_cast<const T*>(&rb)) : 0.f;
                            const float x = v[j] + sP[ch];
                            o = pre ? apply_act(p.act, x + rv, al) : apply_act(p.act, x, al) + rv;
                        } else {
                            o = apply_act(p.act, v[j] + sP[ch], al);
                        }
                        v[j] = o;
                    }
                    if (has_res) __syncwarp();  // every lane has its residual before the slot is reused
                    if (p.y_nhwc) store_nhwc_row<T>(p, r0 + lane, n0 + c, v, nj);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const T o = from_f32<T>(v[j]);
                        slot[j * 32 + lane] = *reinterpret_cast<const uint16_t*>(&o);
                    }
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int piece = lane + 32 * k, j = piece >> 2, pb = piece & 3;
                        if (j < nj) {
                            const uint4 u = *reinterpret_cast<const uint4*>(slot + j * 32 + pb * 8);
                            *reinterpret_cast<uint4*>(y + base0 + (long long)(n0 + c + j) * p.OHW +
                                                      pb * 8) = u;
                        }
                    }
                    __syncwarp();  // the slot is read out before the next chunk
                    continue;
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    if (j >= nj) break;
                    const int ch = n0 + c + j;
                    const long long idx = base + (long long)ch * p.OHW;
                    const float rv = (has_res && valid) ? to_f32(res[idx]) : 0.f;
                    const float x = v[j] + sP[ch];
                    const float al = prelu ? sP[cpad + ch] : 0.f;
                    const float o = pre ? apply_act(p.act, x + rv, al) : apply_act(p.act, x, al) + rv;
                    v[j] = o;
                    if (valid) y[idx] = from_f32<T>(o);
                }
                if (p.y_nhwc && valid) store_nhwc_row<T>(p, mr, n0 + c, v, nj);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
PFN_cuTensorMapEncodeIm2col_v12000 g_encode_im2col = nullptr;

bool load_encoders() {
    static std::once_flag once;
    static bool ok = false;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q1, q2;
        cudaError_t e1 = cudaGetDriverEntryPointByVersion(
            "cuTensorMapEncodeTiled", reinterpret_cast<void**>(&g_encode_tiled), 12000,
            cudaEnableDefault, &q1);
        cudaError_t e2 = cudaGetDriverEntryPointByVersion(
            "cuTensorMapEncodeIm2col", reinterpret_cast<void**>(&g_encode_im2col), 12000,
            cudaEnableDefault, &q2);
        ok = e1 == cudaSuccess && e2 == cudaSuccess && q1 == cudaDriverEntryPointSuccess &&
             q2 == cudaDriverEntryPointSuccess && g_encode_tiled && g_encode_im2col;
    });
    return ok;
}

struct Maps {
    CUtensorMap a, a2, b;
};

template <int BN, int MS, int BK, typename T>
int launch_bn(const ConvArgs& a, const Maps& m, Params prm, cudaStream_t s) {
    using C = Cfg<BN, MS, BK>;
    auto kern = igemm_conv_kernel<BN, MS, BK, T>;
    if (ensure_smem_optin(reinterpret_cast<const void*>(kern), kSmemMax) != ACNN_OK)
        return ACNN_ERR_CUDA;
    prm.num_n_tiles = (a.d.c_out + BN - 1) / BN;
    // Residual ring: deep (4 boxes per warp) when a tile has few k-blocks and
    // the epilogue's memory traffic dominates, else 3.
    const bool nhwc_res = prm.res_mode != ACNN_RES_NONE && prm.out_layout == ACNN_NHWC && !prm.part;
    const int rd = nhwc_res ? (prm.kb_per_split <= 2 ? kMaxResDepth : 3) : 0;
    // The operand ring takes the rest of shared memory (at most kMaxStages
    // deep).  With a single column tile the weights can instead stay resident
    // (loaded once per CTA), the ring then carrying A alone: chosen when that
    // still leaves a ring of 3 (or one as deep as without).
    const size_t b_all = (size_t)prm.num_kb * C::kBBytes;
    // shared bias / alpha copy for the NHWC epilogue: every column tile's
    // columns, so reads past C_out in a ragged last tile stay inside
    const bool nhwc_epi = prm.out_layout == ACNN_NHWC;
    prm.par_floats = prm.num_n_tiles * BN * (prm.act == ACNN_ACT_PRELU ? 2 : 1);
    const size_t par_bytes = (size_t)prm.par_floats * 4;
    // NHWC: the residual ring (split-K: rd = 0, one slot); NCHW: one slot, the
    // transposing stage of the vectorised stores
    prm.ring_slots = nhwc_epi ? (rd > 0 ? rd : 1) : 1;
    const size_t ring_bytes = (size_t)kEpiWarps * prm.ring_slots * kStageBytes;
    // bytes a stage holds: A, plus B unless resident (halo rows: the larger A
    // box and the three taps' B blocks)
    const bool halo = prm.a_mode == 2;
    const size_t a_slot = halo ? C::kABh : C::kAB;
    const size_t b_slot = halo ? 3 * (size_t)C::kBBytes : C::kBBytes;
    auto stages_for = [&](bool resident) -> int {
        if (kSmemFixed + ring_bytes + par_bytes > kSmemMax) return 0;
        size_t left = kSmemMax - kSmemFixed - ring_bytes - par_bytes;
        if (resident) {
            if (left < b_all) return 0;
            left -= b_all;
        }
        const size_t n = left / (a_slot + (resident ? 0 : b_slot));
        return n > (size_t)kMaxStages ? kMaxStages : (int)n;
    };
    const int s_ring = stages_for(false);
    const int s_res = prm.num_n_tiles == 1 ? stages_for(true) : 0;
    const bool resident = s_res >= 2 && s_res >= (s_ring < 3 ? s_ring : 3);
    prm.b_resident = resident ? 1 : 0;
    prm.stages = resident ? s_res : s_ring;
    prm.res_depth = rd;
    // fewer than two stages: C_out too large for the bias copy, or (halo rows)
    // a stage too large for the ring -- the caller retries without halo rows
    if (prm.stages < 2) return ACNN_ERR_UNSUPPORTED;
    const size_t smem = kSmemFixed + ring_bytes + par_bytes +
                        (size_t)prm.stages * (a_slot + (resident ? 0 : b_slot)) +
                        (resident ? b_all : 0);
    const int tiles = prm.num_m_tiles * prm.num_n_tiles * prm.splits;
    const int grid = tiles < sm_count() ? tiles : sm_count();
    // split-K relies on every CTA being resident: grid <= #SMs and one CTA per
    // SM (the shared memory allows no second)
    launch_pdl(kern, grid, kThreads, smem, s, m.a, m.a2, m.b, prm);
    return cudaGetLastError() == cudaSuccess ? ACNN_OK : ACNN_ERR_CUDA;
}

// The instantiated tile shapes: BK = 64 with (BN, MS) in {(256, 1), (128, 1),
// (128, 2), (64, 1), (64, 2)}; BK = 32 (C_in <= 32) with MS = 2 and BN in
// {128, 64, 32}.  igemm_plan picks only among these.
template <typename T>
int launch_typed(const ConvArgs& a, const IgemmPlan& pl, const Maps& m, const Params& prm,
                 cudaStream_t s) {
    if (pl.bk == 32) {
        if (pl.bn == 128) return launch_bn<128, 2, 32, T>(a, m, prm, s);
        if (pl.bn == 64) return launch_bn<64, 2, 32, T>(a, m, prm, s);
        return launch_bn<32, 2, 32, T>(a, m, prm, s);
    }
    if (pl.bn == 256) return launch_bn<256, 1, 64, T>(a, m, prm, s);
    if (pl.bn == 128) return pl.ms == 2 ? launch_bn<128, 2, 64, T>(a, m, prm, s)
                                        : launch_bn<128, 1, 64, T>(a, m, prm, s);
    return pl.ms == 2 ? launch_bn<64, 2, 64, T>(a, m, prm, s) : launch_bn<64, 1, 64, T>(a, m, prm, s);
}

}  // namespace

// Tile width and K split from a small cost model of one launch, in
// microseconds: every unit (tile x K range) streams its k-blocks at the
// slower of the producer's per-k-block issue cost (~0.3 us: the barrier wait,
// expect-tx and two TMA issues of one thread) and the MMA time of the block;
// units run in waves of one per SM; the layer cannot beat its HBM traffic;
// split-K adds a reduce launch that reads the fp32 partials and writes y.
// Tile shape forced by acnn_conv2d_force_plan (bn = 0: none), for plan sweeps.
namespace {
std::atomic<int> g_force_bn{0}, g_force_ms{0}, g_force_splits{0};

bool instantiated(int bk, int bn, int ms) {
    if (bk == 32) return ms == 2 && (bn == 128 || bn == 64 || bn == 32);
    return (bn == 256 && ms == 1) || ((bn == 128 || bn == 64) && (ms == 1 || ms == 2));
}
}  // namespace

void force_plan(int bn, int ms, int splits) {
    g_force_ms.store(ms);
    g_force_splits.store(splits);
    g_force_bn.store(bn);
}

IgemmPlan igemm_plan(const acnn_conv_desc& d, int oh, int ow, size_t part_budget) {
    {
        // a forced shape, when this geometry has an instantiation of it; the
        // split count is lowered until the split units fit in one wave and
        // their partial tiles in the budget
        const int fbn = g_force_bn.load(), fms = g_force_ms.load();
        const int bk = d.c_in <= 32 ? 32 : 64;
        if (fbn > 0 && instantiated(bk, fbn, fms)) {
            const long long M = (long long)d.n * oh * ow;
            const int num_kb = d.kh * d.kw * ((d.c_in + bk - 1) / bk);
            const long long tiles = ((M + BM * fms - 1) / (BM * fms)) * ((d.c_out + fbn - 1) / fbn);
            for (int sp = std::max(1, std::min(g_force_splits.load(), num_kb)); sp >= 1; --sp) {
                const int kbs = (num_kb + sp - 1) / sp;
                const int eff = (num_kb + kbs - 1) / kbs;
                const size_t tile_bytes = (size_t)BM * fms * fbn * sizeof(float);
                const size_t part = eff > 1 ? (((size_t)tiles * 4 + 255) & ~(size_t)255) +
                                                  (size_t)tiles * eff * tile_bytes
                                            : 0;
                if (eff == 1 || (part <= part_budget && tiles * eff <= sm_count()))
                    return IgemmPlan{fbn, fms, eff, kbs, part, bk};
            }
        }
    }
    const double kIssueUs = 0.30, kMmaUsPerMflop = 1.0 / 15.0, kHbmBytesPerUs = 6.0e6;
    const double kSplitUs = 1.5, kEpiUsPerChunk = 0.15;
    const double kL2GBsPerSm = 100.0, kL2Bytes = 96.0e6;
    const long long M = (long long)d.n * oh * ow;
    // 32-channel k-blocks when C_in <= 32: a 64-channel block would be half zeros
    const int bk = d.c_in <= 32 ? 32 : 64;
    const int num_kb = d.kh * d.kw * ((d.c_in + bk - 1) / bk);
    const int sms = sm_count();
    const double io_bytes = 2.0 * ((double)d.n * d.h * d.w * d.c_in + (double)M * d.c_out +
                                   (double)d.c_out * d.kh * d.kw * d.c_in);
    // defaults are instantiated shapes too (32-channel k-blocks come with MS = 2)
    const int ms0 = bk == 32 ? 2 : 1;
    IgemmPlan best{64, ms0, 1, num_kb, 0, bk}, best1{64, ms0, 1, num_kb, 0, bk};
    double best_cost = 1e30, best1_cost = 1e30;
    int bn0, bn_min;
    if (bk == 64) {
        bn0 = d.c_out >= 256 ? 256 : (d.c_out > 64 ? 128 : 64);
        bn_min = 64;
    } else {
        bn0 = d.c_out >= 128 ? 128 : (d.c_out > 32 ? 64 : 32);
        bn_min = 32;
    }
    for (int bn = bn0; bn >= bn_min; bn >>= 1) {
        for (int ms = 1; ms <= 2; ++ms) {
            if (bk == 32 && ms != 2) continue;   // instantiated: MS = 2 only
            if (bk == 64 && bn == 256 && ms != 1) continue;  // TMEM: 2 * ms * bn <= 512
            const long long mt = (M + BM * ms - 1) / (BM * ms);
            const long long tiles = mt * ((d.c_out + bn - 1) / bn);
            const double t_kb = fmax(kIssueUs, 2.0 * BM * ms * bn * bk * 1e-6 * kMmaUsPerMflop);
            for (int sp = 1; sp <= 16 && sp <= num_kb; ++sp) {
                const int kbs = (num_kb + sp - 1) / sp;
                const int eff = (num_kb + kbs - 1) / kbs;  // splits actually used
                if (eff != sp) continue;
                // split-K: tile counters + one fp32 partial tile per (tile, split)
                const size_t tile_bytes = (size_t)BM * ms * bn * sizeof(float);
                const size_t part = eff > 1 ? (((size_t)tiles * 4 + 255) & ~(size_t)255) +
                                                  (size_t)tiles * eff * tile_bytes
                                            : 0;
                if (part > part_budget) continue;
                const long long units = tiles * eff;
                // split only into one wave: with several units per CTA the extra
                // partial-tile traffic measured slower than no split
                if (eff > 1 && units > sms) continue;
                const long long waves = (units + sms - 1) / sms;
                double cost = waves * kbs * t_kb + ms * (bn / 64.0) * kEpiUsPerChunk * 2.0;
                cost = fmax(cost, io_bytes / kHbmBytesPerUs);
                // each split writes its partial tile and reads back one tile's
                // worth (its 1/S share of every split's partial, from L2 when the
                // partials fit there); a memset clears the counters
                if (eff > 1)
                    cost += kSplitUs + 2.0 * tile_bytes * 1e-6 / kL2GBsPerSm +
                            (part > kL2Bytes ? (double)part * 2.0 / kHbmBytesPerUs : 0.0);
                if (cost < best_cost * 0.97) {  // prefer wide, short tiles and no split on ties
                    best_cost = cost;
                    best = IgemmPlan{bn, ms, eff, kbs, part, bk};
                }
                if (eff == 1 && cost < best1_cost * 0.97) {
                    best1_cost = cost;
                    best1 = IgemmPlan{bn, ms, 1, kbs, 0, bk};
                }
            }
        }
    }
    // split only for a clear gain: the reduction adds latency the model only estimates
    return best.splits > 1 && best_cost > 0.85 * best1_cost ? best1 : best;
}

// Halo rows serve 3x3, stride 1, pad 1 convs on plans of at most 128 output
// channels per tile and no K split (the wider layers already run near the MMA
// rate); with 32-channel k-blocks (64-byte swizzle) too when kHaloBk32 holds.
constexpr bool kHaloBk32 = true;

bool halo_rows_ok(const acnn_conv_desc& d, int oh, int ow, const IgemmPlan& plan) {
    if (d.kh != 3 || d.kw != 3 || d.stride != 1 || d.pad != 1) return false;
    if (plan.splits != 1 || plan.bn > 128 || (plan.bk == 32 && !kHaloBk32)) return false;
    return (long long)d.n * oh * (ow + 2) <= 0x7fffffffLL;
}

int launch_igemm_conv(const ConvArgs& a, cudaStream_t s) {
    const acnn_conv_desc& d = a.d;
    if (!load_encoders()) return ACNN_ERR_CUDA;
    const int taps = d.kh * d.kw;
    const long long M = (long long)d.n * a.oh * a.ow;
    const CUtensorMapDataType dt =
        d.dtype == ACNN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const bool tiled = d.kh == 1 && d.kw == 1 && d.stride == 1 && d.pad == 0;
    // no K split for NCHW output: its split epilogue stores element by element,
    // while the unsplit one writes 16-byte runs
    IgemmPlan plan = igemm_plan(d, a.oh, a.ow,
                                a.ws_part && a.out_layout == ACNN_NHWC ? a.ws_part_bytes : 0);
    // A pooled second output (1x1/s1/p0 only): rectangular tiles of 128 pixels,
    // rw columns x 128 / rw rows with rw = 16 or 8, so that each epilogue warp's
    // 32 rows hold whole 2x2 windows; one 128-row block, no K split.
    const bool rect = a.y2 != nullptr && !a.y2_up;
    if (rect) {
        if (!tiled || plan.bk != 64 || a.out_layout != ACNN_NHWC || a.oh % 2 || a.ow % 2)
            return ACNN_ERR_UNSUPPORTED;
        plan.ms = 1;
        plan.splits = 1;
        plan.kb_per_split = d.kh * d.kw * ((d.c_in + 63) / 64);
        plan.part_bytes = 0;
    }
    const int rw = a.ow % 16 == 0 ? 16 : (a.ow % 8 == 0 ? 8 : 16);
    const int rh = 128 / rw;
    const int rtx = (a.ow + rw - 1) / rw, rty = (a.oh + rh - 1) / rh;
    const int bk = plan.bk;
    const CUtensorMapSwizzle swz = bk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const bool cat = a.x2 && a.c_split > 0;
    if (cat && a.c_split % bk != 0) return ACNN_ERR_UNSUPPORTED;  // a k-block must not straddle

    // first with halo rows where they apply, then (also when a halo-row stage
    // does not fit in shared memory) without
    for (int h = halo_rows_ok(d, a.oh, a.ow, plan) ? 1 : 0; h >= 0; --h) {
        const bool halo = h == 1;
        const int vw = halo ? a.ow + 2 : a.ow;  // row width of the (virtual) output grid
        const long long Mv = (long long)d.n * a.oh * vw;
        alignas(64) Maps maps;
        CUtensorMap& tb = maps.b;
        // the A operand's map over an NHWC tensor of `ch` channels (a folded
        // concat has two: channels [0, c_split) and [c_split, c_in))
        auto encode_a = [&](CUtensorMap* ta, const void* ptr, int ch) {
            if (rect) {
                // the NHWC map as {C, W, H, N}; a box is one rectangular tile
                cuuint64_t dims[4] = {(cuuint64_t)ch, (cuuint64_t)d.w, (cuuint64_t)d.h,
                                      (cuuint64_t)d.n};
                cuuint64_t strides[3] = {(cuuint64_t)ch * 2, (cuuint64_t)d.w * ch * 2,
                                         (cuuint64_t)d.h * d.w * ch * 2};
                cuuint32_t box[4] = {(cuuint32_t)bk, (cuuint32_t)rw, (cuuint32_t)rh, 1};
                cuuint32_t es[4] = {1, 1, 1, 1};
                return g_encode_tiled(ta, dt, 4, const_cast<void*>(ptr), dims, strides, box, es,
                                      CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            }
            if (tiled) {
                cuuint64_t dims[2] = {(cuuint64_t)ch, (cuuint64_t)M};
                cuuint64_t strides[1] = {(cuuint64_t)ch * 2};
                cuuint32_t box[2] = {(cuuint32_t)bk, (cuuint32_t)(BM * plan.ms)};
                cuuint32_t es[2] = {1, 1};
                return g_encode_tiled(ta, dt, 2, const_cast<void*>(ptr), dims, strides, box, es,
                                      CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            }
            cuuint64_t dims[4] = {(cuuint64_t)ch, (cuuint64_t)d.w, (cuuint64_t)d.h, (cuuint64_t)d.n};
            cuuint64_t strides[3] = {(cuuint64_t)ch * 2, (cuuint64_t)d.w * ch * 2,
                                     (cuuint64_t)d.h * d.w * ch * 2};
            // window corners range over [-pad, dim - 1 + pad - (k - 1)] (W then H);
            // with halo rows W runs two corners further (the two virtual columns
            // of each output row), and a box holds TM + 2 pixels
            int lower[2] = {-d.pad, -d.pad};
            int upper[2] = {halo ? d.pad : d.pad - (d.kw - 1), d.pad - (d.kh - 1)};
            cuuint32_t es[4] = {1, (cuuint32_t)d.stride, (cuuint32_t)d.stride, 1};
            return g_encode_im2col(ta, dt, 4, const_cast<void*>(ptr), dims, strides, lower, upper, bk,
                                   BM * plan.ms + (halo ? 2 : 0), es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                   swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        };
        CUresult r = encode_a(&maps.a, a.x, cat ? a.c_split : d.c_in);
        if (r == CUDA_SUCCESS) {
            if (cat) r = encode_a(&maps.a2, a.x2, d.c_in - a.c_split);
            else maps.a2 = maps.a;
        }
        if (r != CUDA_SUCCESS) return ACNN_ERR_CUDA;

        const int num_m_tiles = rect ? d.n * rty * rtx : (int)((Mv + BM * plan.ms - 1) / (BM * plan.ms));
        const int bn = plan.bn;
        {
            cuuint64_t dims[3] = {(cuuint64_t)d.c_in, (cuuint64_t)taps, (cuuint64_t)d.c_out};
            cuuint64_t strides[2] = {(cuuint64_t)d.c_in * 2, (cuuint64_t)taps * d.c_in * 2};
            cuuint32_t box[3] = {(cuuint32_t)bk, 1, (cuuint32_t)bn};
            cuuint32_t es[3] = {1, 1, 1};
            r = g_encode_tiled(&tb, dt, 3, const_cast<void*>(a.w), dims, strides, box, es,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        }
        if (r != CUDA_SUCCESS) return ACNN_ERR_CUDA;
        Params prm{};
        prm.M = rect ? num_m_tiles * BM : (int)Mv;
        prm.C_out = d.c_out;
        prm.taps = taps;
        prm.KW = d.kw;
        prm.kb_per_tap = (d.c_in + bk - 1) / bk;
        prm.num_kb = taps * prm.kb_per_tap;
        prm.num_kbh = halo ? d.kh * prm.kb_per_tap : 0;
        prm.num_m_tiles = num_m_tiles;
        prm.splits = plan.splits;
        prm.kb_per_split = halo ? prm.num_kbh : plan.kb_per_split;
        // split-K workspace: tile counters, then the partial tiles
        const int out_tiles = num_m_tiles * ((d.c_out + plan.bn - 1) / plan.bn);
        const size_t cnt_bytes = ((size_t)out_tiles * 4 + 255) & ~(size_t)255;
        prm.cnt = plan.splits > 1 ? static_cast<unsigned*>(a.ws_part) : nullptr;
        prm.part = plan.splits > 1
                       ? reinterpret_cast<float*>(static_cast<uint8_t*>(a.ws_part) + cnt_bytes)
                       : nullptr;
        if (plan.splits > 1 && cudaMemsetAsync(a.ws_part, 0, cnt_bytes, s) != cudaSuccess)
            return ACNN_ERR_CUDA;
        prm.OW = a.ow;
        prm.OH = a.oh;
        prm.OHW = a.oh * a.ow;
        prm.vw = vw;
        prm.vw_magic = ~0ull / (unsigned long long)vw + 1ull;
        prm.S = d.stride;
        prm.P = d.pad;
        prm.a_mode = rect ? 3 : (tiled ? 0 : (halo ? 2 : 1));
        prm.rw_log2 = rw == 16 ? 4 : 3;
        prm.rh = rh;
        prm.rtx = rtx;
        prm.rty = rty;
        prm.rtx_magic = ~0ull / (unsigned long long)rtx + 1ull;
        prm.rty_magic = ~0ull / (unsigned long long)rty + 1ull;
        prm.y2 = a.y2;
        prm.y2_up = a.y2_up;
        prm.y_nhwc = a.out_layout == ACNN_NCHW ? a.y_nhwc : nullptr;
        prm.c_split = cat ? a.c_split : 0;
        prm.out_layout = a.out_layout;
        prm.act = a.act;
        prm.res_mode = a.res_mode;
        prm.bias = a.bias;
        prm.alpha = a.alpha;
        prm.res = a.residual;
        prm.y = a.y;
        prm.status = device_status_ptr();
        prm.budget = wait_budget_polls();
        if (!prm.status) return ACNN_ERR_CUDA;
        const bool bf16 = d.dtype == ACNN_BF16;
        const int st = bf16 ? launch_typed<__nv_bfloat16>(a, plan, maps, prm, s)
                            : launch_typed<__half>(a, plan, maps, prm, s);
        if (halo && st == ACNN_ERR_UNSUPPORTED) continue;  // nothing launched: retry without
        return st;
    }
    return ACNN_ERR_UNSUPPORTED;
}

}  // namespace acnn
