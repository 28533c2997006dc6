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
// CTA roles (192 threads): warp 0 lane 0 issues TMA loads into a STAGES-deep
// shared-memory ring; warp 1 owns the TMEM accumulator and lane 0 issues
// tcgen05.mma (M=128, N=BN, K=16, fp32 accumulate in TMEM); warps 2-5 read the
// accumulator back with tcgen05.ld and run the fused epilogue (bias, ReLU,
// round to fp16/bf16) straight into the NCHW/NCDHW output, one TMEM lane (one
// output pixel) per thread so each store instruction of a warp writes 32
// consecutive pixels of one output channel.
//
// Every wait on an mbarrier is bounded (globaltimer); on expiry the kernel
// records an error word, lets its own in-flight copies and MMAs land, frees
// TMEM and returns.
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

constexpr int kThreads = 192;
constexpr int kMaxStages = 8;
constexpr int kBlockK = 64;                       // channels per stage: one 128-B row
constexpr uint32_t kAStageBytes = 128u * 128u;    // 128 pixel rows x 128 B

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
__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait until the phase with the given parity has completed, for at most
// `limit` ns; gives up early when another role has raised the abort flag.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit,
                                             const volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (abort_flag && *abort_flag) return false;
        if (globaltimer() - t0 > limit) return false;
    }
}
__device__ __forceinline__ void raise_abort(volatile int *flag) {
    *flag = 1;
    atomicOr(&g_device_error, 1u);
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
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
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
    int tiles_w, tiles_h;
    int cblocks;
    int ksteps;
    int stages;
    int relu;
    uint32_t idesc;
    uint32_t tx_bytes;
    uint32_t tmem_cols;
    uint64_t wait_limit_ns;
};

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
igemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sA = base;
    const uint32_t b_stage = (uint32_t)a.BN * 128u;
    const uint32_t sB = sA + (uint32_t)a.stages * kAStageBytes;
    const uint32_t sBar = sB + (uint32_t)a.stages * b_stage;
    auto full_bar = [&](int s) { return sBar + 8u * s; };
    auto empty_bar = [&](int s) { return sBar + 8u * (kMaxStages + s); };
    const uint32_t accum_bar = sBar + 16u * kMaxStages;
    const uint32_t drain_bar = accum_bar + 8u;
    const uint32_t slot_addr = accum_bar + 16u;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem_raw + (slot_addr - raw));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_raw + (slot_addr + 4u - raw));

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // Output tile of this CTA.
    int t = blockIdx.x;
    const int tw = t % a.tiles_w; t /= a.tiles_w;
    const int th = t % a.tiles_h; t /= a.tiles_h;
    const int od = t % a.OD;
    const int n = t / a.OD;
    const int ow0 = tw * a.BW, oh0 = th * a.BH;
    const int oc0 = blockIdx.y * a.BN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(accum_bar, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(slot_addr, a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t limit = a.wait_limit_ns;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- TMA producer
            int issued = 0;
            bool ok = true;
            for (int it = 0; it < a.ksteps; ++it) {
                const int s = it % a.stages;
                const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
                if (!wait_bounded(empty_bar(s), ph ^ 1u, limit, abort_flag)) {
                    ok = false;
                    break;
                }
                const int tap = it / a.cblocks, cb = it - tap * a.cblocks;
                const int kx = tap % a.k, ky = (tap / a.k) % a.k, kz = tap / (a.k * a.k);
                mbar_arrive_expect_tx(full_bar(s), a.tx_bytes);
                tma_load_5d(sA + s * kAStageBytes, &tmA, full_bar(s), cb * kBlockK,
                            ow0 * a.stride + kx - a.pad, oh0 * a.stride + ky - a.pad,
                            od * a.stride + kz - a.pad_d, n);
                tma_load_3d(sB + s * b_stage, &tmB, full_bar(s), cb * kBlockK, oc0, tap);
                issued = it + 1;
            }
            if (!ok) {
                raise_abort(abort_flag);
                // Let the copies already issued land before the CTA exits.
                const int first = issued > a.stages ? issued - a.stages : 0;
                for (int it = first; it < issued; ++it)
                    wait_bounded(full_bar(it % a.stages), (uint32_t)(it / a.stages) & 1u, limit,
                                 nullptr);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------ MMA issuer
            bool ok = true;
            for (int it = 0; it < a.ksteps; ++it) {
                const int s = it % a.stages;
                const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
                if (!wait_bounded(full_bar(s), ph, limit, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t ad = sw128_kmajor_desc(sA + s * kAStageBytes);
                const uint64_t bd = sw128_kmajor_desc(sB + s * b_stage);
#pragma unroll
                for (int kk = 0; kk < kBlockK / 16; ++kk)
                    tc_mma(tmem, ad + 2u * kk, bd + 2u * kk, a.idesc, (it | kk) != 0);
                tc_commit(empty_bar(s));
            }
            if (ok) {
                tc_commit(accum_bar);
            } else {
                raise_abort(abort_flag);
                tc_commit(drain_bar);
                wait_bounded(drain_bar, 0, limit, nullptr);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;               // TMEM lane quadrant of this warp
        int ok = 0;
        if (lane == 0) ok = wait_bounded(accum_bar, 0, limit, abort_flag) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            if (lane == 0) raise_abort(abort_flag);
        } else {
            tc_fence_after();
            const int m = q * 32 + lane;
            const int r = m / a.BW, c = m - r * a.BW;
            const int oh = oh0 + r, ow = ow0 + c;
            const bool valid = m < a.BW * a.BH && oh < a.OH && ow < a.OW;
            const int64_t plane = (int64_t)a.OD * a.OH * a.OW;
            T *y = static_cast<T *>(a.y) +
                   ((int64_t)n * a.OC * a.OD + od) * ((int64_t)a.OH * a.OW) +
                   (int64_t)oh * a.OW + ow;
            for (int j0 = 0; j0 < a.BN; j0 += 16) {
                uint32_t v[16];
                tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)j0, v);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int oc = oc0 + j0 + i;
                        if (oc < a.OC) {
                            const float bias = a.b ? __ldg(a.b + oc) : 0.0f;
                            y[(int64_t)oc * plane] =
                                Storage<T>::from_float(epilogue(__uint_as_float(v[i]), bias, a.relu));
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

// x [N][C][S] -> xc [N][S][Cp], zero in channels C..Cp-1 (S = D*H*W).
template <typename T>
__global__ void __launch_bounds__(256)
to_channels_last_kernel(const T *__restrict__ x, T *__restrict__ xc, int C, int Cp, int64_t S) {
    __shared__ T tile[64][65];
    const int64_t s0 = (int64_t)blockIdx.x * 64;
    const int c0 = blockIdx.y * 64;
    const int n = blockIdx.z;
    const T *xn = x + (int64_t)n * C * S;
    T *xcn = xc + (int64_t)n * S * Cp;
    {
        const int sl = threadIdx.x % 64, cb = threadIdx.x / 64;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int cl = cb + 4 * i;
            const int c = c0 + cl;
            const int64_t s = s0 + sl;
            tile[cl][sl] = (c < C && s < S) ? xn[(int64_t)c * S + s] : T(0.0f);
        }
    }
    __syncthreads();
    {
        const int cl = threadIdx.x % 64, sb = threadIdx.x / 64;
        const int c = c0 + cl;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int sl = sb + 4 * i;
            const int64_t s = s0 + sl;
            if (c < Cp && s < S) xcn[s * Cp + c] = tile[cl][sl];
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

// Output-tile geometry: BH rows x BW columns of one (n, od) plane, BW*BH <= 128,
// boxes of at most 256 traversed elements per axis.
struct TileGeom {
    int BW, BH, BN, stages;
};

TileGeom choose_geom(const Problem &p) {
    TileGeom g{};
    const int bw_max = 256 / p.stride < 128 ? 256 / p.stride : 128;
    if (p.OW >= bw_max) {
        const int tiles = (p.OW + bw_max - 1) / bw_max;
        g.BW = (p.OW + tiles - 1) / tiles;
        g.BH = 1;
    } else {
        g.BW = p.OW;
        int bh = 128 / p.OW;
        const int bh_max = 256 / p.stride;
        if (bh > bh_max) bh = bh_max;
        if (bh > p.OH) bh = p.OH;
        g.BH = bh < 1 ? 1 : bh;
    }
    int bn = (p.OC + 15) / 16 * 16;
    g.BN = bn > 256 ? 256 : bn;
    const int stage_bytes = (int)kAStageBytes + g.BN * 128;
    int st = (220 * 1024 - 2048) / stage_bytes;
    g.stages = st > kMaxStages ? kMaxStages : st;
    return g;
}

uint32_t tmem_cols_for(int bn) {
    uint32_t c = 32;
    while (c < (uint32_t)bn) c <<= 1;
    return c;
}

template <typename T>
cudaError_t launch_tc_typed(const Problem &p, const void *xc, const void *wp, const float *b,
                            void *y, cudaStream_t s) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
    if (!encode) return cudaErrorInvalidValue;
    const TileGeom g = choose_geom(p);
    const int Cp = tc_cpad(p.C);
    const CUtensorMapDataType dt =
        p.dtype == GBCONV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;

    alignas(64) CUtensorMap tmA, tmB;
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

    TcArgs a{};
    a.b = b;
    a.y = y;
    a.OC = p.OC; a.OD = p.OD; a.OH = p.OH; a.OW = p.OW;
    a.k = p.k; a.pad = p.pad; a.pad_d = p.pad_d; a.stride = p.stride;
    a.BW = g.BW; a.BH = g.BH; a.BN = g.BN;
    a.tiles_w = (p.OW + g.BW - 1) / g.BW;
    a.tiles_h = (p.OH + g.BH - 1) / g.BH;
    a.cblocks = (Cp + kBlockK - 1) / kBlockK;
    a.ksteps = p.taps * a.cblocks;
    a.stages = g.stages;
    a.relu = p.act == GBCONV_ACT_RELU;
    a.idesc = make_idesc(128, g.BN, p.dtype == GBCONV_BF16);
    a.tx_bytes = kAStageBytes / 128u * (uint32_t)(g.BW * g.BH) + (uint32_t)g.BN * 128u;
    a.tmem_cols = tmem_cols_for(g.BN);
    a.wait_limit_ns = wait_limit_ns();

    const size_t smem = 1024 + (size_t)g.stages * (kAStageBytes + (size_t)g.BN * 128) + 256;
    auto kern = igemm_tc_kernel<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t mtiles = (int64_t)p.N * p.OD * a.tiles_h * a.tiles_w;
    dim3 grid((unsigned)mtiles, (unsigned)((p.OC + g.BN - 1) / g.BN));
    kern<<<grid, kThreads, smem, s>>>(tmA, tmB, a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_cl_typed(const Problem &p, const void *x, void *xc, cudaStream_t s) {
    const int Cp = tc_cpad(p.C);
    const int64_t S = p.in_vol;
    dim3 grid((unsigned)((S + 63) / 64), (unsigned)((Cp + 63) / 64), (unsigned)p.N);
    to_channels_last_kernel<T><<<grid, 256, 0, s>>>(static_cast<const T *>(x), static_cast<T *>(xc),
                                                     p.C, Cp, S);
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
    if ((int64_t)p.N * p.in_vol > 0xFFFFFFFFll) return false;
    const TileGeom g = choose_geom(p);
    const int64_t mtiles = (int64_t)p.N * p.OD * ((p.OH + g.BH - 1) / g.BH) *
                           ((p.OW + g.BW - 1) / g.BW);
    return g.BW * p.stride <= 256 && g.BH * p.stride <= 256 && mtiles < 0x7FFFFFFF &&
           g.stages >= 2;
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
