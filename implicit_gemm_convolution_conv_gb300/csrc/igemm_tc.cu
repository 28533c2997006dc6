// Implicit-GEMM convolution on the 5th-generation tensor cores (tcgen05).
//
// GEMM view of the convolution sum (lpnh.cn/news/2745477 section 2.2; the
// Convolution3D extension of git.erdda.com/Tencent/ncnn/discussions/7001
// section 3.2):  M = output pixels of one (n, od) plane tile, N = output
// channels, K = taps x input channels. For each tap (kd, ky, kx) the A
// operand is the input shifted by that tap, which TMA fetches straight from a
// channels-last copy of x as a {64 ch, BW px, BH rows, 1 frame, 1 image} box:
// padding is TMA's out-of-bounds zero fill and the stride is TMA's element
// stride, so no im2col buffer exists. The B operand is the weight slab of the
// same tap, packed once as [tap][OC][C] (the page's "re-arrange weights at
// export time", sections 2.3 and 4.2).
//
// Persistent kernel, one CTA per SM, tiles handed out round-robin. Roles
// (192 threads): warp 0 lane 0 issues TMA loads into a STAGES-deep
// shared-memory ring; warp 1 owns TMEM and lane 0 issues tcgen05.mma (M=128,
// N=BN, K=16, fp32 accumulate) into one of two TMEM accumulators, so the MMAs
// of tile i+1 run while warps 2-5 drain tile i. The epilogue reads TMEM with
// tcgen05.ld (one output pixel per thread), adds the bias, applies ReLU,
// rounds to fp16/bf16, stages 32 output channels at a time in shared memory
// and writes them with TMA bulk-tensor stores into the NCHW/NCDHW output
// (plain coalesced stores when the output rows are not 16-byte aligned).
//
// Every wait on an mbarrier is bounded (SM cycle counter); on expiry the
// kernel records an error word, lets its own in-flight copies and MMAs land,
// frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "dev_common.cuh"
#include "internal.h"

namespace gbconv {

__device__ unsigned int g_device_error;   // bit 0: a bounded wait ran out
static std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(); }
void set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns); }

cudaError_t read_and_clear_device_error(unsigned int *code) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
}

namespace {

constexpr int kEpiWarps = 8;                      // warps 2..9, two per TMEM lane quadrant
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kGroupThreads = 128;                // one epilogue group = 4 warps = 128 lanes
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kMaxStages = 8;
constexpr int kBlockK = 64;                       // channels per stage: one 128-B row
constexpr uint32_t kAStageBytes = 128u * 128u;    // 128 pixel rows x 128 B
constexpr int kEpiChunk = 32;                     // output channels per staged store
constexpr uint32_t kStageOutBytes = 128u * kEpiChunk * 2u;   // 8 KB
// Epilogue used when the output is 16-byte aligned: 2 = vector stores, 1 = TMA stores.
constexpr int kEpiModeAligned = 2;

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait until the phase with the given parity has completed, for at most
// `limit` SM cycles; gives up early when another role raised the abort flag.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, long long limit,
                                             const volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (abort_flag && *abort_flag) return false;
        if (clock64() - t0 > limit) return false;
    }
}
__device__ __forceinline__ void raise_abort(volatile int *flag) {
    *flag = 1;
    atomicOr(&g_device_error, 1u);
}
__device__ __forceinline__ void epi_bar() {   // named barrier of all epilogue warps
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}
__device__ __forceinline__ void group_bar(int grp) {   // barrier of one epilogue group
    asm volatile("bar.sync %0, %1;" ::"r"(2 + grp), "n"(kGroupThreads) : "memory");
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *tm, uint32_t bar,
                                            int c0, int c1, int c2, int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *tm, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tma_store_5d(const CUtensorMap *tm, uint32_t src, int c0, int c1,
                                             int c2, int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::
            "l"(reinterpret_cast<uint64_t>(tm)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
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
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzle
// layout: rows of 64 16-bit elements (128 B), 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);   // start address
    d |= (uint64_t)1u << 16;                    // leading byte offset (unused here)
    d |= (uint64_t)(1024u >> 4) << 32;          // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1u << 46;                    // descriptor version for tcgen05
    d |= (uint64_t)2u << 61;                    // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, A/B fp16 or bf16,
// both K-major, shape M x N.
constexpr uint32_t make_idesc(int M, int N, bool bf16) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct TcArgs {
    const float *b;
    void *y;
    int OC, OD, OH, OW;
    int k, pad, pad_d, stride;
    int BW, BH, BN;
    int tiles_w, tiles_h, n_tiles;
    int num_tiles;
    int cblocks;
    int ksteps;
    int stages;
    int relu;
    int epi_mode;          // 0: direct element stores, 1: TMA tensor stores, 2: 16-byte stores
    uint32_t idesc;
    uint32_t tx_bytes;
    uint32_t tmem_cols;
    long long wait_limit_cycles;
};

struct TileCoord {
    int n, od, oh0, ow0, oc0;
};
__device__ __forceinline__ TileCoord tile_coord(const TcArgs &a, int t) {
    TileCoord c;
    const int nt = t % a.n_tiles;
    t /= a.n_tiles;
    const int tw = t % a.tiles_w; t /= a.tiles_w;
    const int th = t % a.tiles_h; t /= a.tiles_h;
    c.od = t % a.OD;
    c.n = t / a.OD;
    c.ow0 = tw * a.BW;
    c.oh0 = th * a.BH;
    c.oc0 = nt * a.BN;
    return c;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
igemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmY, const TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t b_stage = (uint32_t)a.BN * 128u;
    const uint32_t sA = base;
    const uint32_t sB = sA + (uint32_t)a.stages * kAStageBytes;
    const uint32_t sOut = sB + (uint32_t)a.stages * b_stage;          // 2 groups x 2 x 8 KB
    const uint32_t sBias = sOut + 4u * kStageOutBytes;                // 256 floats
    const uint32_t sBar = sBias + 1024u;
    const uint32_t full0 = sBar, empty0 = sBar + 8u * kMaxStages;
    const uint32_t tfull0 = sBar + 16u * kMaxStages, tempty0 = tfull0 + 16u;
    const uint32_t drain_bar = tempty0 + 16u;
    const uint32_t slot_addr = drain_bar + 8u;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem_raw + (slot_addr - raw));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_raw + (slot_addr + 4u - raw));
    volatile int *epi_fail = reinterpret_cast<volatile int *>(smem_raw + (slot_addr + 8u - raw));
    float *bias_s = reinterpret_cast<float *>(smem_raw + (sBias - raw));

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull0 + 8u * i, 1);
            mbar_init(tempty0 + 8u * i, kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        *epi_fail = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (a.epi_mode == 1) prefetch_tmap(&tmY);
    }
    if (warp == 1) {
        tmem_alloc(slot_addr, a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const long long limit = a.wait_limit_cycles;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- TMA producer
            // Ring position and tap counters advance incrementally: no integer
            // division on this single thread's per-k-step path.
            int s = 0;
            uint32_t ph = 0;
            int issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < a.num_tiles && ok; t += gridDim.x) {
                const TileCoord tc = tile_coord(a, t);
                const int x0 = tc.ow0 * a.stride - a.pad, y0 = tc.oh0 * a.stride - a.pad,
                          z0 = tc.od * a.stride - a.pad_d;
                int cb = 0, tap = 0, kx = 0, ky = 0, kz = 0;
                for (int it = 0; it < a.ksteps; ++it) {
                    const uint32_t fb = full0 + 8u * s;
                    if (!wait_bounded(empty0 + 8u * s, ph ^ 1u, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(fb, a.tx_bytes);
                    tma_load_5d(sA + (uint32_t)s * kAStageBytes, &tmA, fb, cb * kBlockK, x0 + kx,
                                y0 + ky, z0 + kz, tc.n);
                    tma_load_3d(sB + (uint32_t)s * b_stage, &tmB, fb, cb * kBlockK, tc.oc0, tap);
                    ++issued;
                    if (++cb == a.cblocks) {
                        cb = 0;
                        ++tap;
                        if (++kx == a.k) {
                            kx = 0;
                            if (++ky == a.k) { ky = 0; ++kz; }
                        }
                    }
                    if (++s == a.stages) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                raise_abort(abort_flag);
                // Let the copies already issued land before the CTA exits.
                const int first = issued > a.stages ? issued - a.stages : 0;
                for (int q = first; q < issued; ++q)
                    wait_bounded(full0 + 8u * (q % a.stages), (uint32_t)(q / a.stages) & 1u, limit,
                                 nullptr);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------ MMA issuer
            const uint64_t adesc0 = sw128_kmajor_desc(sA), bdesc0 = sw128_kmajor_desc(sB);
            const uint32_t a_step = kAStageBytes >> 4, b_step = b_stage >> 4;
            int s = 0;
            uint32_t ph = 0;
            int local = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < a.num_tiles && ok; t += gridDim.x, ++local) {
                const int acc = local & 1;
                const uint32_t use_ph = (uint32_t)(local >> 1) & 1u;
                if (!wait_bounded(tempty0 + 8u * acc, use_ph ^ 1u, limit, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * a.BN);
                uint64_t ad = adesc0, bd = bdesc0;
                for (int k = 0; k < s; ++k) { ad += a_step; bd += b_step; }
                for (int it = 0; it < a.ksteps; ++it) {
                    if (!wait_bounded(full0 + 8u * s, ph, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk)
                        tc_mma(d, ad + 2u * kk, bd + 2u * kk, a.idesc, (it | kk) != 0);
                    tc_commit(empty0 + 8u * s);
                    ad += a_step;
                    bd += b_step;
                    if (++s == a.stages) {
                        s = 0;
                        ph ^= 1u;
                        ad = adesc0;
                        bd = bdesc0;
                    }
                }
                if (ok) tc_commit(tfull0 + 8u * acc);
            }
            if (!ok) {
                raise_abort(abort_flag);
                tc_commit(drain_bar);
                wait_bounded(drain_bar, 0, limit, nullptr);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // Two groups of four warps; warp w reads TMEM lane quadrant w % 4, and
        // group g drains the 32-column chunks g, g+2, g+4, ...
        const int q = warp & 3;
        const int grp = (warp - 2) / 4;
        const int et = threadIdx.x - 64;      // 0..255
        const int gt = et & (kGroupThreads - 1);
        const int m = q * 32 + lane;          // accumulator row = tile pixel
        const int r = m / a.BW, c = m - r * a.BW;
        const int MT = a.BW * a.BH;
        const int64_t plane = (int64_t)a.OD * a.OH * a.OW;
        T *out_g = reinterpret_cast<T *>(smem_raw + (sOut - raw)) +
                   grp * 2 * (kStageOutBytes / sizeof(T));
        const uint32_t sOut_g = sOut + (uint32_t)grp * 2u * kStageOutBytes;
        const int nchunks = a.BN / kEpiChunk;
        int local = 0;
        int chunk_ctr = 0;
        for (int t = blockIdx.x; t < a.num_tiles; t += gridDim.x, ++local) {
            const TileCoord tc = tile_coord(a, t);
            const int acc = local & 1;
            int ok = 0;
            if (lane == 0)
                ok = wait_bounded(tfull0 + 8u * acc, (uint32_t)(local >> 1) & 1u, limit, abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok && lane == 0) *epi_fail = 1;
            // One decision for all epilogue warps (they share named barriers);
            // this barrier also orders the previous tile's bias reads.
            epi_bar();
            if (*epi_fail) {
                if (et == 0) raise_abort(abort_flag);
                break;
            }
            tc_fence_after();
            for (int j = et; j < a.BN; j += kEpiThreads) {
                const int oc = tc.oc0 + j;
                bias_s[j] = (a.b && oc < a.OC) ? __ldg(a.b + oc) : 0.0f;
            }
            epi_bar();
            const int oh = tc.oh0 + r, ow = tc.ow0 + c;
            const bool valid = m < MT && oh < a.OH && ow < a.OW;
            T *yp = static_cast<T *>(a.y) +
                    ((int64_t)tc.n * a.OC * a.OD + tc.od) * ((int64_t)a.OH * a.OW) +
                    (int64_t)oh * a.OW + ow;
            for (int ch = grp; ch < nchunks; ch += 2) {
                uint32_t v[32];
                tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * a.BN + ch * kEpiChunk), v);
                tmem_ld_wait();
                const float *bb = bias_s + ch * kEpiChunk;
                if (a.epi_mode == 0) {
                    if (valid) {
#pragma unroll
                        for (int j = 0; j < kEpiChunk; ++j) {
                            const int oc = tc.oc0 + ch * kEpiChunk + j;
                            if (oc < a.OC)
                                yp[(int64_t)oc * plane] =
                                    Storage<T>::from_float(epilogue(__uint_as_float(v[j]), bb[j], a.relu));
                        }
                    }
                } else {
                    const int buf = chunk_ctr & 1;
                    T *o = out_g + buf * (kStageOutBytes / sizeof(T));
                    if (a.epi_mode == 1) {
                        if (gt == 0) bulk_wait_read_1();   // the store that used `buf` has read it
                        group_bar(grp);
                    }
                    if (m < MT) {
#pragma unroll
                        for (int j = 0; j < kEpiChunk; ++j)
                            o[j * MT + m] = Storage<T>::from_float(epilogue(__uint_as_float(v[j]), bb[j], a.relu));
                    }
                    if (a.epi_mode == 1) {
                        fence_proxy_async_smem();
                        group_bar(grp);
                        if (gt == 0) {
                            tma_store_5d(&tmY, sOut_g + buf * kStageOutBytes, tc.ow0, tc.oh0, tc.od,
                                         tc.oc0 + ch * kEpiChunk, tc.n);
                            bulk_commit();
                        }
                    } else {
                        // 16-byte stores of 8 consecutive pixels of one channel.
                        group_bar(grp);
                        const int vpr = MT / 8;            // vectors per channel row
                        for (int vi = gt; vi < kEpiChunk * vpr; vi += kGroupThreads) {
                            const int j = vi / vpr, pv = (vi - j * vpr) * 8;
                            const int oc = tc.oc0 + ch * kEpiChunk + j;
                            const int rr = pv / a.BW, cc = pv - rr * a.BW;
                            if (oc < a.OC && tc.oh0 + rr < a.OH && tc.ow0 + cc < a.OW) {
                                T *dst = static_cast<T *>(a.y) +
                                         (((int64_t)tc.n * a.OC + oc) * a.OD + tc.od) * ((int64_t)a.OH * a.OW) +
                                         (int64_t)(tc.oh0 + rr) * a.OW + tc.ow0 + cc;
                                *reinterpret_cast<uint4 *>(dst) =
                                    *reinterpret_cast<const uint4 *>(o + j * MT + pv);
                            }
                        }
                    }
                    ++chunk_ctr;
                }
            }
            // All reads of this accumulator by this warp are done: hand it back.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8u * acc);
        }
        if (a.epi_mode == 1 && gt == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

// x [N][C][S] -> xc [N][S][Cp], zero in channels C..Cp-1 (S = D*H*W).
// 64 channels x 64 positions per CTA; 16-byte global loads and stores when
// x rows are 16-byte aligned (VEC), element loads otherwise.
template <typename T, bool VEC>
__global__ void __launch_bounds__(256)
to_channels_last_kernel(const T *__restrict__ x, T *__restrict__ xc, int C, int Cp, int64_t S) {
    __shared__ __align__(16) T tile[64][72];
    const int64_t s0 = (int64_t)blockIdx.x * 64;
    const int c0 = blockIdx.y * 64;
    const int n = blockIdx.z;
    const T *xn = x + (int64_t)n * C * S;
    T *xcn = xc + (int64_t)n * S * Cp;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int v = threadIdx.x + 256 * i;
        const int cl = v / 8, p = (v % 8) * 8;
        const int cc = c0 + cl;
        const int64_t s = s0 + p;
        if (VEC && cc < C && s + 8 <= S) {
            *reinterpret_cast<uint4 *>(&tile[cl][p]) =
                __ldg(reinterpret_cast<const uint4 *>(xn + (int64_t)cc * S + s));
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                tile[cl][p + j] = (cc < C && s + j < S) ? xn[(int64_t)cc * S + s + j] : T(0.0f);
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int v = threadIdx.x + 256 * i;
        const int pl = v % 64, cch = v / 64;          // lanes walk positions
        const int cc = c0 + cch * 8;
        const int64_t s = s0 + pl;
        if (s < S && cc < Cp) {
            alignas(16) T vals[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) vals[j] = tile[cch * 8 + j][pl];
            *reinterpret_cast<uint4 *>(xcn + s * Cp + cc) = *reinterpret_cast<const uint4 *>(vals);
        }
    }
}

// wp[tap][oc][cp] = w[oc][c][tap] for c < C, zero for C <= cp < Cp.
template <typename T>
__global__ void pack_tc_kernel(const T *__restrict__ w, T *__restrict__ wp, int OC, int C,
                               int Cp, int taps) {
    const int64_t total = (int64_t)taps * OC * Cp;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int cp = (int)(e % Cp);
        const int64_t r = e / Cp;
        const int oc = (int)(r % OC), tap = (int)(r / OC);
        wp[e] = cp < C ? w[((int64_t)oc * C + cp) * taps + tap] : T(0.0f);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// SM count and clock of the current device, looked up once per device.
struct DevInfo {
    int sms = 0;
    int clock_khz = 0;
};
cudaError_t dev_info(DevInfo *out) {
    static std::mutex mu;
    static DevInfo cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].sms == 0) {
        DevInfo d;
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.clock_khz, cudaDevAttrClockRate, dev);
        if (e != cudaSuccess) return e;
        cache[dev] = d;
    }
    *out = cache[dev];
    return cudaSuccess;
}

// Output-tile geometry: BH rows x BW columns of one (n, od) plane, BW*BH <= 128,
// boxes of at most 256 traversed elements per axis; BN a multiple of 32.
struct TileGeom {
    int BW, BH, BN, stages;
};

TileGeom choose_geom(const Problem &p) {
    TileGeom g{};
    const int bw_max = 256 / p.stride < 128 ? 256 / p.stride : 128;
    if (p.OW >= bw_max) {
        const int tiles = (p.OW + bw_max - 1) / bw_max;
        g.BW = (p.OW + tiles - 1) / tiles;
        // prefer 16-byte aligned column tiles (TMA-store epilogue)
        const int bw8 = (g.BW + 7) / 8 * 8;
        if (bw8 <= bw_max && (p.OW + bw8 - 1) / bw8 == tiles) g.BW = bw8;
        g.BH = 1;
    } else {
        g.BW = p.OW;
        int bh = 128 / p.OW;
        const int bh_max = 256 / p.stride;
        if (bh > bh_max) bh = bh_max;
        if (bh > p.OH) bh = p.OH;
        g.BH = bh < 1 ? 1 : bh;
    }
    int bn = (p.OC + 31) / 32 * 32;
    g.BN = bn > 256 ? 256 : bn;
    const int stage_bytes = (int)kAStageBytes + g.BN * 128;
    const int fixed = 1024 + 4 * (int)kStageOutBytes + 1024 + 256;
    int st = (227 * 1024 - fixed) / stage_bytes;
    g.stages = st > kMaxStages ? kMaxStages : st;
    return g;
}

size_t smem_bytes(const TileGeom &g) {
    return 1024 + (size_t)g.stages * (kAStageBytes + (size_t)g.BN * 128) + 4 * kStageOutBytes +
           1024 + 256;
}

uint32_t tmem_cols_for(int cols) {
    uint32_t c = 32;
    while (c < (uint32_t)cols) c <<= 1;
    return c;
}

template <typename T>
cudaError_t launch_tc_typed(const Problem &p, const void *xc, const void *wp, const float *b,
                            void *y, cudaStream_t s) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
    if (!encode) return cudaErrorInvalidValue;
    DevInfo info;
    cudaError_t e = dev_info(&info);
    if (e != cudaSuccess) return e;
    const TileGeom g = choose_geom(p);
    const int Cp = tc_cpad(p.C);
    const CUtensorMapDataType dt =
        p.dtype == GBCONV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;

    alignas(64) CUtensorMap tmA, tmB, tmY;
    {
        const cuuint64_t dims[5] = {(cuuint64_t)Cp, (cuuint64_t)p.W, (cuuint64_t)p.H,
                                    (cuuint64_t)p.D, (cuuint64_t)p.N};
        const cuuint64_t strides[4] = {(cuuint64_t)Cp * 2, (cuuint64_t)Cp * 2 * p.W,
                                       (cuuint64_t)Cp * 2 * p.W * p.H,
                                       (cuuint64_t)Cp * 2 * p.W * p.H * p.D};
        const cuuint32_t box[5] = {(cuuint32_t)kBlockK, (cuuint32_t)(g.BW * p.stride),
                                   (cuuint32_t)(g.BH * p.stride), 1, 1};
        const cuuint32_t es[5] = {1, (cuuint32_t)p.stride, (cuuint32_t)p.stride, 1, 1};
        if (encode(&tmA, dt, 5, const_cast<void *>(xc), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)Cp, (cuuint64_t)p.OC, (cuuint64_t)p.taps};
        const cuuint64_t strides[2] = {(cuuint64_t)Cp * 2, (cuuint64_t)Cp * 2 * p.OC};
        const cuuint32_t box[3] = {(cuuint32_t)kBlockK, (cuuint32_t)g.BN, 1};
        const cuuint32_t es[3] = {1, 1, 1};
        if (encode(&tmB, dt, 3, const_cast<void *>(wp), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // Epilogue store mode. 16-byte vector stores (mode 2) and TMA tensor
    // stores (mode 1) need 16-byte output rows, 16-byte column tiles and a
    // 16-byte aligned base; otherwise elements are stored one by one (mode 0).
    const bool aligned16 = (p.OW % 8 == 0) && (g.BW % 8 == 0) && (((uintptr_t)y % 16) == 0);
    int epi_mode = aligned16 ? kEpiModeAligned : 0;
    memset(&tmY, 0, sizeof(tmY));
    if (epi_mode == 1) {
        const cuuint64_t dims[5] = {(cuuint64_t)p.OW, (cuuint64_t)p.OH, (cuuint64_t)p.OD,
                                    (cuuint64_t)p.OC, (cuuint64_t)p.N};
        const cuuint64_t strides[4] = {(cuuint64_t)p.OW * 2, (cuuint64_t)p.OW * 2 * p.OH,
                                       (cuuint64_t)p.OW * 2 * p.OH * p.OD,
                                       (cuuint64_t)p.OW * 2 * p.OH * p.OD * p.OC};
        const cuuint32_t box[5] = {(cuuint32_t)g.BW, (cuuint32_t)g.BH, 1, (cuuint32_t)kEpiChunk, 1};
        const cuuint32_t es[5] = {1, 1, 1, 1, 1};
        if (encode(&tmY, dt, 5, y, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            epi_mode = 2;
    }

    TcArgs a{};
    a.b = b;
    a.y = y;
    a.OC = p.OC; a.OD = p.OD; a.OH = p.OH; a.OW = p.OW;
    a.k = p.k; a.pad = p.pad; a.pad_d = p.pad_d; a.stride = p.stride;
    a.BW = g.BW; a.BH = g.BH; a.BN = g.BN;
    a.tiles_w = (p.OW + g.BW - 1) / g.BW;
    a.tiles_h = (p.OH + g.BH - 1) / g.BH;
    a.n_tiles = (p.OC + g.BN - 1) / g.BN;
    const int64_t num_tiles = (int64_t)p.N * p.OD * a.tiles_h * a.tiles_w * a.n_tiles;
    a.num_tiles = (int)num_tiles;
    a.cblocks = (Cp + kBlockK - 1) / kBlockK;
    a.ksteps = p.taps * a.cblocks;
    a.stages = g.stages;
    a.relu = p.act == GBCONV_ACT_RELU;
    a.epi_mode = epi_mode;
    a.idesc = make_idesc(128, g.BN, p.dtype == GBCONV_BF16);
    a.tx_bytes = kAStageBytes / 128u * (uint32_t)(g.BW * g.BH) + (uint32_t)g.BN * 128u;
    a.tmem_cols = tmem_cols_for(2 * g.BN);
    const double cyc = (double)wait_limit_ns() * (double)info.clock_khz * 1e-6;
    a.wait_limit_cycles = cyc > 9.0e18 ? (long long)9e18 : (long long)cyc;

    const size_t smem = smem_bytes(g);
    auto kern = igemm_tc_kernel<T>;
    static std::atomic<uint64_t> attr_done{0};   // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (!(attr_done.load() >> (dev & 63) & 1ull)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        attr_done.fetch_or(1ull << (dev & 63));
    }
    const int grid = num_tiles < info.sms ? (int)num_tiles : info.sms;
    kern<<<grid, kThreads, smem, s>>>(tmA, tmB, tmY, a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_cl_typed(const Problem &p, const void *x, void *xc, cudaStream_t s) {
    const int Cp = tc_cpad(p.C);
    const int64_t S = p.in_vol;
    dim3 grid((unsigned)((S + 63) / 64), (unsigned)((Cp + 63) / 64), (unsigned)p.N);
    const bool vec = (S % 8 == 0) && ((uintptr_t)x % 16 == 0);
    if (vec)
        to_channels_last_kernel<T, true><<<grid, 256, 0, s>>>(static_cast<const T *>(x),
                                                              static_cast<T *>(xc), p.C, Cp, S);
    else
        to_channels_last_kernel<T, false><<<grid, 256, 0, s>>>(static_cast<const T *>(x),
                                                               static_cast<T *>(xc), p.C, Cp, S);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_pack_tc_typed(const Problem &p, const void *w, void *wp, cudaStream_t s) {
    const int64_t total = (int64_t)p.taps * p.OC * tc_cpad(p.C);
    const int blocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    pack_tc_kernel<T><<<blocks, 256, 0, s>>>(static_cast<const T *>(w), static_cast<T *>(wp), p.OC,
                                             p.C, tc_cpad(p.C), p.taps);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(const Problem &p) {
    if (p.dtype == GBCONV_F32) return false;
    const TileGeom g = choose_geom(p);
    const int64_t mtiles = (int64_t)p.N * p.OD * ((p.OH + g.BH - 1) / g.BH) *
                           ((p.OW + g.BW - 1) / g.BW) * ((p.OC + g.BN - 1) / g.BN);
    return g.BW * p.stride <= 256 && g.BH * p.stride <= 256 && mtiles < 0x7FFFFFFF &&
           g.stages >= 2 && p.N <= 65535;
}

cudaError_t launch_igemm_tc(const Problem &p, const void *xc, const void *wp, const float *b,
                            void *y, cudaStream_t s) {
    if (p.dtype == GBCONV_BF16) return launch_tc_typed<__nv_bfloat16>(p, xc, wp, b, y, s);
    return launch_tc_typed<__half>(p, xc, wp, b, y, s);
}

cudaError_t launch_to_channels_last(const Problem &p, const void *x, void *xc, cudaStream_t s) {
    if (p.dtype == GBCONV_BF16) return launch_cl_typed<__nv_bfloat16>(p, x, xc, s);
    return launch_cl_typed<__half>(p, x, xc, s);
}

cudaError_t launch_pack_tc(const Problem &p, const void *w, void *wp, cudaStream_t s) {
    if (p.dtype == GBCONV_BF16) return launch_pack_tc_typed<__nv_bfloat16>(p, w, wp, s);
    return launch_pack_tc_typed<__half>(p, w, wp, s);
}

}  // namespace gbconv
