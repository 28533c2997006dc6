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

// wp[(tap * C + c) * OCp + oc] = w[(oc * C + c) * taps + tap], zero-padded in
// oc. One CTA per (tap, c) row of the output; threads walk the channels.
template <typename T>
__global__ void pack_ffma_kernel(const T *__restrict__ w, T *__restrict__ wp,
                                 int OC, int C, int taps, int OCp) {
    const int row = blockIdx.x;                 // tap * C + c
    const int tap = row / C, c = row - tap * C;
    const T *src = w + (int64_t)c * taps + tap;
    T *dst = wp + (int64_t)row * OCp;
    for (int oc = threadIdx.x; oc < OCp; oc += blockDim.x)
        dst[oc] = oc < OC ? src[(int64_t)oc * C * taps] : T(0.0f);
}

template <typename T>
cudaError_t launch_ffma_typed(const FfmaArgs &a, bool cl, cudaStream_t s) {
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
    pack_ffma_kernel<T><<<p.taps * p.C, OCp < 256 ? OCp : 256, 0, s>>>(
        static_cast<const T *>(w), static_cast<T *>(wp), p.OC, p.C, p.taps, OCp);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_igemm_ffma(const Problem &p, const void *x, const void *wp,
                              const float *b, void *y, cudaStream_t s) {
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
    case GBCONV_F32: return launch_ffma_typed<float>(a, p.cl, s);
    case GBCONV_F16: return launch_ffma_typed<__half>(a, p.cl, s);
    default: return launch_ffma_typed<__nv_bfloat16>(a, p.cl, s);
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
