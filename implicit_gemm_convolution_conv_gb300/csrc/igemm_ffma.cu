// Implicit-GEMM convolution on CUDA cores (exact fp32 FMA, any storage type).
//
// GEMM view of the convolution sum of lpnh.cn/news/2745477 section 2.2:
//   M = N * OD * OH * OW output pixels,  N_gemm = OC,  K = kvol * IC,
//   A[m][kk] = x at the input coordinate of output pixel m and tap/channel kk
//              (zero where that coordinate is padding),
//   B[kk][oc] = packed weights, row kk = tap * IC + ic,
//   y[n][oc][pixel] = epilogue(sum_kk A[m][kk] * B[kk][oc]).
// A is never materialised (no im2col buffer): each CTA gathers its A tile
// straight from the input into shared memory. The generic kernel takes the
// input and output element strides as arguments, so it reads and writes both
// NC(D)HW and channels-last N(D)HWC tensors; the packed-FMA variant below is
// NC(D)HW only. CTA tile BM x BN,
// K step BK, two shared-memory stages with the next stage prefetched into
// registers while the current one is multiplied; each thread accumulates an
// 8 x 8 register tile (two 4-wide pixel groups x two 4-wide channel groups).
#include "dev_common.cuh"
#include "internal.h"

namespace gbconv {
namespace {

constexpr int BM = 128, BN = 64, BK = 16, NT = 128;
static_assert(kFfmaOcAlign % BN == 0, "packed OC padding must cover the CTA tile");

struct FfmaArgs {
    const void *x;
    const void *wp;     // [taps][C][OCp]
    const float *b;
    void *y;
    int C, D, H, W, OC, OCp;
    int k, kd, stride, pad, pad_d;
    int OD, OH, OW;
    int64_t M, out_vol, in_hw;
    int K;              // taps * C
    int relu;
    // Element strides (generic kernel): x offset = n * xs_n + c * xs_c +
    // id * xs_d + ih * xs_h + iw * xs_w; y offset = n * ys_n + oc * ys_c +
    // pixel * ys_p, pixel = (od * OH + oh) * OW + ow.
    int64_t xs_n, xs_c, xs_d, xs_h, xs_w;
    int64_t ys_n, ys_c, ys_p;
    // split-K (fp32 cp.async kernel): CTA z of gridDim.z sums K steps
    // [ksteps z / splits, ksteps (z + 1) / splits) and stores the raw sums to
    // part[z][oc][m]; null: the CTA covers all of K and applies the epilogue.
    float *part;
    int splits;
};

template <typename T>
__global__ void __launch_bounds__(NT) igemm_ffma_kernel(const FfmaArgs a) {
    __shared__ __align__(16) float As[2][BK][BM];
    __shared__ __align__(16) float Bs[2][BK][BN];

    const T *x = static_cast<const T *>(a.x);
    const T *wp = static_cast<const T *>(a.wp);
    const int tid = threadIdx.x;
    const int64_t m0 = (int64_t)blockIdx.x * BM;
    const int n0 = blockIdx.y * BN;

    // This thread gathers A column `tid` (one output pixel) for every kk.
    const int64_t my_m = m0 + tid;
    const bool m_ok = my_m < a.M;
    int img = 0, od = 0, oh = 0, ow = 0;
    if (m_ok) {
        int64_t r = my_m;
        img = (int)(r / a.out_vol); r -= (int64_t)img * a.out_vol;
        od = (int)(r / ((int64_t)a.OH * a.OW)); r -= (int64_t)od * a.OH * a.OW;
        oh = (int)(r / a.OW); ow = (int)(r - (int64_t)oh * a.OW);
    }
    const int id0 = od * a.stride - a.pad_d, ih0 = oh * a.stride - a.pad,
              iw0 = ow * a.stride - a.pad;
    const T *x_img = x + (int64_t)img * a.xs_n;

    // B loader: row tid/8 of the stage, 8 consecutive output channels.
    const int b_row = tid / 8, b_col = (tid % 8) * 8;

    float a_reg[BK];
    float b_reg[8];

    auto gather = [&](int k0) {
        // (tap, c) of kk = k0; advanced incrementally across the BK rows.
        int tap = k0 / a.C, c = k0 - tap * a.C;
#pragma unroll
        for (int r = 0; r < BK; r++) {
            float v = 0.0f;
            if (m_ok && tap < a.kd * a.k * a.k) {
                const int kx = tap % a.k, ky = (tap / a.k) % a.k, kz = tap / (a.k * a.k);
                const int id = id0 + kz, ih = ih0 + ky, iw = iw0 + kx;
                if (id >= 0 && id < a.D && ih >= 0 && ih < a.H && iw >= 0 && iw < a.W)
                    v = Storage<T>::load(x_img + c * a.xs_c + id * a.xs_d + ih * a.xs_h + iw * a.xs_w);
            }
            a_reg[r] = v;
            if (++c == a.C) { c = 0; ++tap; }
        }
        const int kk = k0 + b_row;
#pragma unroll
        for (int j = 0; j < 8; j++)
            b_reg[j] = kk < a.K ? Storage<T>::load(wp + (int64_t)kk * a.OCp + n0 + b_col + j) : 0.0f;
    };
    auto stash = [&](int buf) {
#pragma unroll
        for (int r = 0; r < BK; r++) As[buf][r][tid] = a_reg[r];
        *reinterpret_cast<float4 *>(&Bs[buf][b_row][b_col]) =
            make_float4(b_reg[0], b_reg[1], b_reg[2], b_reg[3]);
        *reinterpret_cast<float4 *>(&Bs[buf][b_row][b_col + 4]) =
            make_float4(b_reg[4], b_reg[5], b_reg[6], b_reg[7]);
    };

    const int tm = tid % 16, tn = tid / 16;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
        for (int j = 0; j < 8; j++) acc[i][j] = 0.0f;

    const int ksteps = (a.K + BK - 1) / BK;
    gather(0);
    stash(0);
    __syncthreads();
    for (int ks = 0; ks < ksteps; ks++) {
        const int cur = ks & 1;
        if (ks + 1 < ksteps) gather((ks + 1) * BK);
#pragma unroll
        for (int kk = 0; kk < BK; kk++) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&As[cur][kk][tm * 4]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&As[cur][kk][64 + tm * 4]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[cur][kk][tn * 4]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[cur][kk][32 + tn * 4]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; i++)
#pragma unroll
                for (int j = 0; j < 8; j++) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        if (ks + 1 < ksteps) {
            stash(cur ^ 1);
            __syncthreads();
        }
    }

    T *y = static_cast<T *>(a.y);
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int64_t m = m0 + (i < 4 ? tm * 4 + i : 64 + tm * 4 + (i - 4));
        if (m >= a.M) continue;
        const int64_t im = m / a.out_vol, pix = m - im * a.out_vol;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const int oc = n0 + (j < 4 ? tn * 4 + j : 32 + tn * 4 + (j - 4));
            if (oc >= a.OC) continue;
            const float bias = a.b ? __ldg(a.b + oc) : 0.0f;
            y[im * a.ys_n + oc * a.ys_c + pix * a.ys_p] =
                Storage<T>::from_float(epilogue(acc[i][j], bias, a.relu));
        }
    }
}

// Packed-FMA variant for channel counts that are multiples of 16: every K
// step of 16 stays inside one tap, so the tap offset and the bounds of a
// pixel are resolved once per step, not per element. CTA tile 128 pixels x
// 128 channels, 256 threads, 8 x 8 outputs per thread accumulated as 8 x 4
// channel pairs with fma.rn.f32x2. The A tile is kept in shared memory as
// duplicated pairs {a, a} (the packed-FMA operand), written once per step
// from registers; the next step's A and B are loaded into registers while
// the current step is multiplied.
constexpr int WBM = 128, WBN = 128, WBK = 16, WNT = 256;
constexpr int kWideMinBlocks = 1;      // resident CTAs per SM the registers are sized for
static_assert(kFfmaOcAlign % WBN == 0, "packed OC padding must cover the CTA tile");

template <typename T>
__global__ void __launch_bounds__(WNT, kWideMinBlocks) igemm_ffma2_kernel(const FfmaArgs a) {
    extern __shared__ __align__(16) float smem_f[];
    float2 *As = reinterpret_cast<float2 *>(smem_f);                 // [2][WBK][WBM]
    float *Bs = smem_f + 2 * 2 * WBK * WBM;                            // [2][WBK][WBN]

    const T *x = static_cast<const T *>(a.x);
    const T *wp = static_cast<const T *>(a.wp);
    const int tid = threadIdx.x;
    const int64_t m0 = (int64_t)blockIdx.x * WBM;
    const int n0 = blockIdx.y * WBN;

    // A loader: pixel column tid % 128, k rows (tid / 128) + 2j, j < 8.
    const int a_col = tid % WBM, a_row0 = tid / WBM;
    const int64_t my_m = m0 + a_col;
    const bool m_ok = my_m < a.M;
    int img = 0, od = 0, oh = 0, ow = 0;
    if (m_ok) {
        int64_t r = my_m;
        img = (int)(r / a.out_vol); r -= (int64_t)img * a.out_vol;
        od = (int)(r / ((int64_t)a.OH * a.OW)); r -= (int64_t)od * a.OH * a.OW;
        oh = (int)(r / a.OW); ow = (int)(r - (int64_t)oh * a.OW);
    }
    const int id0 = od * a.stride - a.pad_d, ih0 = oh * a.stride - a.pad, iw0 = ow * a.stride - a.pad;
    const int64_t c_stride = (int64_t)a.D * a.in_hw;
    const T *x_img = x + (int64_t)img * a.C * c_stride;
    // B loader: row tid / 16, 8 consecutive channels from column (tid % 16) * 8.
    const int b_row = tid / 16, b_col = (tid % 16) * 8;

    float a_reg[8];
    float4 b_reg[2];
    auto gather = [&](int k0) {
        const int tap = k0 / a.C, c0 = k0 - tap * a.C;
        const int kx = tap % a.k, ky = (tap / a.k) % a.k, kz = tap / (a.k * a.k);
        const int id = id0 + kz, ih = ih0 + ky, iw = iw0 + kx;
        const bool ok = m_ok && id >= 0 && id < a.D && ih >= 0 && ih < a.H && iw >= 0 && iw < a.W;
        const T *src = x_img + (int64_t)(c0 + a_row0) * c_stride + (int64_t)id * a.in_hw +
                       (int64_t)ih * a.W + iw;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            a_reg[j] = ok ? Storage<T>::load(src + (int64_t)(2 * j) * c_stride) : 0.0f;
        const T *bsrc = wp + (int64_t)(k0 + b_row) * a.OCp + n0 + b_col;
        if (sizeof(T) == 4) {
            b_reg[0] = __ldg(reinterpret_cast<const float4 *>(bsrc));
            b_reg[1] = __ldg(reinterpret_cast<const float4 *>(bsrc) + 1);
        } else {
            float bv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) bv[j] = Storage<T>::load(bsrc + j);
            b_reg[0] = make_float4(bv[0], bv[1], bv[2], bv[3]);
            b_reg[1] = make_float4(bv[4], bv[5], bv[6], bv[7]);
        }
    };
    auto stash = [&](int buf) {
        float2 *Ab = As + buf * WBK * WBM;
#pragma unroll
        for (int j = 0; j < 8; ++j) Ab[(a_row0 + 2 * j) * WBM + a_col] = make_float2(a_reg[j], a_reg[j]);
        float *Bb = Bs + buf * WBK * WBN + b_row * WBN + b_col;
        *reinterpret_cast<float4 *>(Bb) = b_reg[0];
        *reinterpret_cast<float4 *>(Bb + 4) = b_reg[1];
    };

    // Thread tile: pixels {2tm, 2tm+1} + 32*i4 (i4 < 4) x channels 4tn + {0..3}
    // and 64 + 4tn + {0..3}.
    const int tm = tid % 16, tn = tid / 16;
    float2 acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

    const int ksteps = a.K / WBK;
    gather(0);
    stash(0);
    __syncthreads();
    for (int ks = 0; ks < ksteps; ++ks) {
        const int cur = ks & 1;
        if (ks + 1 < ksteps) gather((ks + 1) * WBK);
        const float2 *Ab = As + cur * WBK * WBM;
        const float *Bb = Bs + cur * WBK * WBN;
#pragma unroll
        for (int kk = 0; kk < WBK; ++kk) {
            float2 av[8];
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
                const float4 q = *reinterpret_cast<const float4 *>(&Ab[kk * WBM + 32 * i4 + 2 * tm]);
                av[2 * i4] = make_float2(q.x, q.y);
                av[2 * i4 + 1] = make_float2(q.z, q.w);
            }
            const float4 b0 = *reinterpret_cast<const float4 *>(&Bb[kk * WBN + 4 * tn]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&Bb[kk * WBN + 64 + 4 * tn]);
            const float2 bv[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                                  make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = __ffma2_rn(av[i], bv[j], acc[i][j]);
        }
        if (ks + 1 < ksteps) {
            // Buffer cur^1 was last read in the previous step, before the
            // barrier that ended it.
            stash(cur ^ 1);
            __syncthreads();
        }
    }

    T *y = static_cast<T *>(a.y);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t m = m0 + 32 * (i / 2) + 2 * tm + (i & 1);
        if (m >= a.M) continue;
        const int64_t im = m / a.out_vol, pix = m - im * a.out_vol;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int oc = n0 + (j < 2 ? 4 * tn + 2 * j + h : 64 + 4 * tn + 2 * (j - 2) + h);
                if (oc >= a.OC) continue;
                const float bias = a.b ? __ldg(a.b + oc) : 0.0f;
                const float v = h ? acc[i][j].y : acc[i][j].x;
                y[(im * a.OC + oc) * a.out_vol + pix] = Storage<T>::from_float(epilogue(v, bias, a.relu));
            }
        }
    }
}

// fp32 variant of the packed-FMA kernel (channel counts that are multiples
// of 16, NC(D)HW): the operand tiles go straight from global to shared
// memory with cp.async, four stages deep, so no thread stages them through
// registers and a thread needs at most 128 registers (several CTAs per SM).
// CTA tile 128 pixels x BN channels (BN 128 or 64), 2 * BN threads; a
// thread owns pixels 4 tm .. 4 tm + 3 and 64 + 4 tm .. + 3 (tm = tid % 16)
// and channels 4 tn .. 4 tn + 3 and BN / 2 + 4 tn .. + 3 (tn = tid / 16),
// accumulated as pixel pairs x channel with fma.rn.f32x2 (each weight is
// duplicated into a register pair). The A tile is [16 k][128 pixels]: each
// element is one 4-byte copy from x at the pixel's tap-shifted position,
// zero-filled at padding and past the last pixel (cp.async with a source
// size of 0); the B tile is [16 k][BN] straight from the packed weights
// [K][OCp] in 16-byte copies. (Copying each A element twice, so that the
// duplicated operand is A's and comes from shared memory, measured slower:
// the doubled A tile leaves fewer CTAs per SM.)
constexpr int CBM = 128, CBK = 16, CSTAGES = 4;

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, bool ok) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(ok ? 4 : 0) : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int BN>
__global__ void __launch_bounds__(2 * BN, BN == 128 ? 2 : 3) igemm_ffma_cp_kernel(const FfmaArgs a) {
    constexpr int NT = 2 * BN;
    constexpr int A_PER = CBK * CBM / NT;          // A elements a thread copies per stage
    constexpr int B_PER = CBK * BN / 4 / NT;        // 16-byte B chunks a thread copies per stage
    constexpr int STAGE_A = CBK * CBM, STAGE_B = CBK * BN;   // floats
    extern __shared__ __align__(16) float smem_f[];
    float *As = smem_f;                              // [CSTAGES][CBK][CBM]
    float *Bs = smem_f + CSTAGES * STAGE_A;          // [CSTAGES][CBK][BN]
    const uint32_t As_s = static_cast<uint32_t>(__cvta_generic_to_shared(As));
    const uint32_t Bs_s = static_cast<uint32_t>(__cvta_generic_to_shared(Bs));
    // programmatic dependent launch: the next kernel launches once every CTA
    // here has started; global memory only after the previous kernel is done
    pdl_launch_dependents();
    pdl_wait();

    const float *x = static_cast<const float *>(a.x);
    const float *wp = static_cast<const float *>(a.wp);
    const int tid = threadIdx.x;
    const int64_t m0 = (int64_t)blockIdx.x * CBM;
    const int n0 = blockIdx.y * BN;

    // A copier: pixel column tid % 128, k rows tid / 128 + (NT / 128) j.
    const int a_col = tid % CBM, a_row0 = tid / CBM;
    constexpr int A_ROW_STEP = NT / CBM;
    const int64_t my_m = m0 + a_col;
    const bool m_ok = my_m < a.M;
    int img = 0, od = 0, oh = 0, ow = 0;
    if (m_ok) {
        int64_t r = my_m;
        img = (int)(r / a.out_vol); r -= (int64_t)img * a.out_vol;
        od = (int)(r / ((int64_t)a.OH * a.OW)); r -= (int64_t)od * a.OH * a.OW;
        oh = (int)(r / a.OW); ow = (int)(r - (int64_t)oh * a.OW);
    }
    const int id0 = od * a.stride - a.pad_d, ih0 = oh * a.stride - a.pad, iw0 = ow * a.stride - a.pad;
    const int64_t c_stride = (int64_t)a.D * a.in_hw;
    const float *x_img = x + (int64_t)img * a.C * c_stride;

    auto load_stage = [&](int ks, int buf) {
        const int k0 = ks * CBK;
        const int tap = k0 / a.C, c0 = k0 - tap * a.C;
        const int kx = tap % a.k, ky = (tap / a.k) % a.k, kz = tap / (a.k * a.k);
        const int id = id0 + kz, ih = ih0 + ky, iw = iw0 + kx;
        const bool ok = m_ok && id >= 0 && id < a.D && ih >= 0 && ih < a.H && iw >= 0 && iw < a.W;
        // a padding element reads nothing (source size 0); its address stays inside x
        const float *src = ok ? x_img + (int64_t)(c0 + a_row0) * c_stride + (int64_t)id * a.in_hw +
                                    (int64_t)ih * a.W + iw
                              : x;
        const int64_t step = ok ? (int64_t)A_ROW_STEP * c_stride : 0;
        const uint32_t adst = As_s + (uint32_t)(buf * STAGE_A + a_row0 * CBM + a_col) * 4u;
#pragma unroll
        for (int j = 0; j < A_PER; ++j)
            cp_async4(adst + (uint32_t)(j * A_ROW_STEP * CBM) * 4u, src + j * step, ok);
        const uint32_t bdst = Bs_s + (uint32_t)(buf * STAGE_B) * 4u;
#pragma unroll
        for (int j = 0; j < B_PER; ++j) {
            const int q = tid + NT * j;                 // chunk: row q / (BN / 4), 4 channels
            const int row = q / (BN / 4), c4 = q % (BN / 4);
            cp_async16(bdst + (uint32_t)(row * BN + 4 * c4) * 4u, wp + (int64_t)(k0 + row) * a.OCp + n0 + 4 * c4);
        }
    };

    const int tm = tid % 16, tn = tid / 16;
    float2 acc[4][8];   // [pixel pair][channel]
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

    const int ksteps_all = a.K / CBK;
    const int z = blockIdx.z;
    const int ks_first = a.part ? (int)((int64_t)ksteps_all * z / a.splits) : 0;
    const int ksteps = a.part ? (int)((int64_t)ksteps_all * (z + 1) / a.splits) - ks_first : ksteps_all;
#pragma unroll
    for (int st = 0; st < CSTAGES - 1; ++st) {
        if (st < ksteps) load_stage(ks_first + st, st);
        cp_async_commit();
    }
    for (int ks = 0; ks < ksteps; ++ks) {
        // stage ks has landed (for every thread's copies after the barrier),
        // and every thread is done with the buffer the next load overwrites
        cp_async_wait<CSTAGES - 2>();
        __syncthreads();
        if (ks + CSTAGES - 1 < ksteps) load_stage(ks_first + ks + CSTAGES - 1, (ks + CSTAGES - 1) % CSTAGES);
        cp_async_commit();
        const float *Ab = As + (ks % CSTAGES) * STAGE_A;
        const float *Bb = Bs + (ks % CSTAGES) * STAGE_B;
#pragma unroll
        for (int kk = 0; kk < CBK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&Ab[kk * CBM + 4 * tm]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&Ab[kk * CBM + 64 + 4 * tm]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&Bb[kk * BN + 4 * tn]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&Bb[kk * BN + BN / 2 + 4 * tn]);
            const float2 av[4] = {make_float2(a0.x, a0.y), make_float2(a0.z, a0.w), make_float2(a1.x, a1.y),
                                  make_float2(a1.z, a1.w)};
            const float bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float2 bv = make_float2(bw[j], bw[j]);
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i][j] = __ffma2_rn(av[i], bv, acc[i][j]);
            }
        }
    }
    cp_async_wait<0>();

    if (a.part) {
        // raw partial sums, part[z][oc][m]: runs of 4 pixels as vectors
        // when M % 4 == 0 (the run then lies whole inside M)
        float *pz = a.part + (int64_t)z * a.OC * a.M;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int64_t m = m0 + 64 * r + 4 * tm;
            if (m >= a.M) continue;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int oc = n0 + (j < 4 ? 4 * tn + j : BN / 2 + 4 * tn + j - 4);
                if (oc >= a.OC) continue;
                float *dst = pz + (int64_t)oc * a.M + m;
                const float v[4] = {acc[2 * r][j].x, acc[2 * r][j].y, acc[2 * r + 1][j].x, acc[2 * r + 1][j].y};
                if ((a.M & 3) == 0) {
                    *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (m + e < a.M) dst[e] = v[e];
                }
            }
        }
        return;
    }

    // Epilogue: for each channel, the thread's two runs of 4 pixels; a run
    // inside one image's plane with y 16-byte aligned leaves as one vector.
    float *y = static_cast<float *>(a.y);
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int64_t m = m0 + 64 * r + 4 * tm;
        if (m >= a.M) continue;
        const int64_t im = m / a.out_vol, pix = m - im * a.out_vol;
        const bool vec = pix + 4 <= a.out_vol && m + 4 <= a.M && ((a.out_vol | pix) & 3) == 0 &&
                         ((uintptr_t)y & 15) == 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int oc = n0 + (j < 4 ? 4 * tn + j : BN / 2 + 4 * tn + j - 4);
            if (oc >= a.OC) continue;
            const float bias = a.b ? __ldg(a.b + oc) : 0.0f;
            const float v[4] = {acc[2 * r][j].x, acc[2 * r][j].y, acc[2 * r + 1][j].x, acc[2 * r + 1][j].y};
            if (vec) {
                *reinterpret_cast<float4 *>(y + (im * a.OC + oc) * a.out_vol + pix) =
                    make_float4(epilogue(v[0], bias, a.relu), epilogue(v[1], bias, a.relu),
                                epilogue(v[2], bias, a.relu), epilogue(v[3], bias, a.relu));
            } else {
                int64_t n = im, pp = pix;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (m + e < a.M) y[(n * a.OC + oc) * a.out_vol + pp] = epilogue(v[e], bias, a.relu);
                    if (++pp == a.out_vol) { pp = 0; ++n; }
                }
            }
        }
    }
}

// wp[(tap * C + c) * OCp + oc] = w[(oc * C + c) * taps + tap], zero-padded in
// oc. One CTA per (tap, c) row of the output; threads walk the channels.
template <typename T>
__global__ void pack_ffma_kernel(const T *__restrict__ w, T *__restrict__ wp,
                                 int OC, int C, int taps, int OCp) {
    pdl_launch_dependents();
    pdl_wait();   // wp may still be read by the previous call's GEMM
    const int row = blockIdx.x;                 // tap * C + c
    const int tap = row / C, c = row - tap * C;
    const T *src = w + (int64_t)c * taps + tap;
    T *dst = wp + (int64_t)row * OCp;
    for (int oc = threadIdx.x; oc < OCp; oc += blockDim.x)
        dst[oc] = oc < OC ? src[(int64_t)oc * C * taps] : T(0.0f);
}

// Split-K reduction: y = epilogue(sum over z of part[z][oc][m]), the
// slices added in order z = 0, 1, ... (the same result on every call). A
// thread takes 4 consecutive pixels of one channel.
__global__ void __launch_bounds__(256) ffma_split_reduce_kernel(const FfmaArgs a) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t mq = (a.M + 3) / 4;
    const int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (q >= mq * a.OC) return;
    const int oc = (int)(q / mq);
    const int64_t m = (q - (int64_t)oc * mq) * 4;
    const bool whole = (a.M & 3) == 0;
    float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int z = 0; z < a.splits; ++z) {
        const float *src = a.part + ((int64_t)z * a.OC + oc) * a.M + m;
        if (whole) {
            const float4 t = __ldg(reinterpret_cast<const float4 *>(src));
            v[0] += t.x; v[1] += t.y; v[2] += t.z; v[3] += t.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (m + e < a.M) v[e] += __ldg(src + e);
        }
    }
    const float bias = a.b ? __ldg(a.b + oc) : 0.0f;
    float *y = static_cast<float *>(a.y);
    const int64_t im = m / a.out_vol, pix = m - im * a.out_vol;
    if (m + 4 <= a.M && pix + 4 <= a.out_vol && ((a.out_vol | pix) & 3) == 0 && ((uintptr_t)y & 15) == 0) {
        *reinterpret_cast<float4 *>(y + (im * a.OC + oc) * a.out_vol + pix) =
            make_float4(epilogue(v[0], bias, a.relu), epilogue(v[1], bias, a.relu), epilogue(v[2], bias, a.relu),
                        epilogue(v[3], bias, a.relu));
    } else {
        int64_t n = im, pp = pix;
        for (int e = 0; e < 4 && m + e < a.M; ++e) {
            y[(n * a.OC + oc) * a.out_vol + pp] = epilogue(v[e], bias, a.relu);
            if (++pp == a.out_vol) { pp = 0; ++n; }
        }
    }
}

// fp32 cp.async kernel. With fewer 128 x 128 tiles than SMs and room for
// partial sums (slices > 1), K is split into S parts, S chosen to minimise
// the parts the busiest SM runs (ceil(tiles S / SMs) / S of a tile: for 120
// tiles on 152 SMs, S = 5 gives 0.8 against 1.0), then one reduction pass.
// Without a split: 128 x 128 tiles, or 128 x 64 when even those fill at
// most one wave (more, smaller CTAs).
cudaError_t launch_ffma_cp(FfmaArgs a, float *part, int slices, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t mt = (a.M + CBM - 1) / CBM;
    const int64_t tiles = mt * ((a.OC + 127) / 128);
    int split = 1;
    if (part && slices > 1 && tiles < sms) {
        double best = 1.0;
        for (int S = 2; S <= slices; ++S) {
            const double c = (double)((tiles * S + sms - 1) / sms) / S;
            if (c < best - 1e-9) {
                best = c;
                split = S;
            }
        }
        if (best > 0.9) split = 1;   // less than a tenth saved: not worth the reduction pass
    }
    a.part = split > 1 ? part : nullptr;
    a.splits = split;
    const bool wide = split > 1 || tiles * 2 > sms;
    const int bn = wide ? 128 : 64;
    const int smem = CSTAGES * (CBK * CBM + CBK * bn) * (int)sizeof(float);
    dim3 grid((unsigned)mt, (unsigned)((a.OC + bn - 1) / bn), (unsigned)split);
    if (log_enabled())
        log_line("igemm_ffma_cp_kernel grid=%ux%ux%u block=%d smem=%d tile=%dx%d stages=%d%s", grid.x, grid.y, grid.z,
                 2 * bn, smem, CBM, bn, CSTAGES, split > 1 ? " split_k (then ffma_split_reduce_kernel)" : "");
    if (wide) {
        e = cudaFuncSetAttribute(igemm_ffma_cp_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        e = launch_pdl(igemm_ffma_cp_kernel<128>, grid, dim3(256), smem, s, a);
    } else {
        e = cudaFuncSetAttribute(igemm_ffma_cp_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        e = launch_pdl(igemm_ffma_cp_kernel<64>, grid, dim3(128), smem, s, a);
    }
    if (e != cudaSuccess || split == 1) return e;
    const int64_t n = (a.M + 3) / 4 * a.OC;
    return launch_pdl(ffma_split_reduce_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, a);
}

template <typename T>
cudaError_t launch_ffma_typed(const FfmaArgs &a, bool cl, float *part, int slices, cudaStream_t s) {
    if constexpr (sizeof(T) == 4) {
        // 16-byte weight copies and 4-byte x copies need those alignments
        if (a.C % CBK == 0 && !cl && (uintptr_t)a.wp % 16 == 0 && (uintptr_t)a.x % 4 == 0)
            return launch_ffma_cp(a, part, slices, s);
    }
    if (a.C % WBK == 0 && !cl) {
        auto kern = igemm_ffma2_kernel<T>;
        const int smem = (2 * 2 * WBK * WBM + 2 * WBK * WBN) * (int)sizeof(float);
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        dim3 grid((unsigned)((a.M + WBM - 1) / WBM), (a.OC + WBN - 1) / WBN);
        if (log_enabled())
            log_line("igemm_ffma2_kernel grid=%ux%u block=%d smem=%d tile=%dx%d", grid.x, grid.y, WNT, smem, WBM, WBN);
        kern<<<grid, WNT, smem, s>>>(a);
        return cudaGetLastError();
    }
    dim3 grid((unsigned)((a.M + BM - 1) / BM), (a.OC + BN - 1) / BN);
    if (log_enabled())
        log_line("igemm_ffma_kernel grid=%ux%u block=%d tile=%dx%d%s", grid.x, grid.y, NT, BM, BN,
                 cl ? " channels_last" : "");
    igemm_ffma_kernel<T><<<grid, NT, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_pack_typed(const Problem &p, const void *w, void *wp, cudaStream_t s) {
    const int OCp = ffma_ocpad(p.OC);
    return launch_pdl(pack_ffma_kernel<T>, dim3((unsigned)(p.taps * p.C)), dim3(OCp < 256 ? OCp : 256), 0, s,
                      static_cast<const T *>(w), static_cast<T *>(wp), p.OC, p.C, p.taps, OCp);
}

}  // namespace

int ffma_split_slices(const Problem &p) {
    if (p.dtype != GBCONV_F32 || p.cl || p.C % CBK != 0) return 0;
    const int64_t M = (int64_t)p.N * p.out_vol;
    // Layers with at least 160 tiles of 128 x 128 already fill the SMs (152
    // on a GB300) and get no split, nor the room for one.
    if ((M + 127) / 128 * ((p.OC + 127) / 128) >= 160) return 0;
    const int ksteps = p.taps * p.C / CBK;
    int slices = ksteps / 2 < 8 ? ksteps / 2 : 8;
    const int64_t slice_bytes = (int64_t)p.OC * M * (int64_t)sizeof(float);
    while (slices > 1 && slices * slice_bytes > (64ll << 20)) --slices;
    return slices >= 2 ? slices : 0;
}

cudaError_t launch_igemm_ffma(const Problem &p, const void *x, const void *wp,
                              const float *b, void *y, float *part, int slices, cudaStream_t s) {
    FfmaArgs a{};
    a.x = x; a.wp = wp; a.b = b; a.y = y;
    a.C = p.C; a.D = p.D; a.H = p.H; a.W = p.W; a.OC = p.OC; a.OCp = ffma_ocpad(p.OC);
    a.k = p.k; a.kd = p.kd; a.stride = p.stride; a.pad = p.pad; a.pad_d = p.pad_d;
    a.OD = p.OD; a.OH = p.OH; a.OW = p.OW;
    a.M = (int64_t)p.N * p.out_vol; a.out_vol = p.out_vol;
    a.in_hw = (int64_t)p.H * p.W;
    a.K = p.taps * p.C;
    a.relu = p.act == GBCONV_ACT_RELU;
    const int64_t hw = (int64_t)p.H * p.W;
    a.xs_n = (int64_t)p.C * p.D * hw;
    a.ys_n = (int64_t)p.OC * p.out_vol;
    if (p.cl) {
        a.xs_c = 1; a.xs_w = p.C; a.xs_h = (int64_t)p.W * p.C; a.xs_d = hw * p.C;
        a.ys_c = 1; a.ys_p = p.OC;
    } else {
        a.xs_c = (int64_t)p.D * hw; a.xs_d = hw; a.xs_h = p.W; a.xs_w = 1;
        a.ys_c = p.out_vol; a.ys_p = 1;
    }
    switch (p.dtype) {
    case GBCONV_F32: return launch_ffma_typed<float>(a, p.cl, part, slices, s);
    case GBCONV_F16: return launch_ffma_typed<__half>(a, p.cl, nullptr, 0, s);
    default: return launch_ffma_typed<__nv_bfloat16>(a, p.cl, nullptr, 0, s);
    }
}

cudaError_t launch_pack_ffma(const Problem &p, const void *w, void *wp, cudaStream_t s) {
    switch (p.dtype) {
    case GBCONV_F32: return launch_pack_typed<float>(p, w, wp, s);
    case GBCONV_F16: return launch_pack_typed<__half>(p, w, wp, s);
    default: return launch_pack_typed<__nv_bfloat16>(p, w, wp, s);
    }
}

}  // namespace gbconv
