// Direct convolution for layers with a small reduction depth (IC * kvol).
//
// Output-stationary, as the compute shader of lpnh.cn/news/2745477 section
// 2.2: each thread owns a fixed set of outputs and derives the input
// coordinates from them, so there are no write races and no atomics. Where
// the shader gives one output per invocation and re-reads x and w from
// memory for every tap, here a CTA stages the input halo of its output tile
// and the weight slab of its output-channel block in shared memory once, and
// each thread keeps a PX-pixel x OCT-channel register micro-tile, the GB300
// counterpart of the Convolution3D backend's "four output channels per
// invocation, weights packed by four" (git.erdda.com/Tencent/ncnn/
// discussions/7001, section 3.2; section 5.3 for the measured 2.91x).
//
// Thread layout: LANES = TW/PX threads along a row of the tile, OCG = OCB/OCT
// channel groups, TH rows; a thread's pixels are lane, lane+LANES, ... so
// consecutive lanes read consecutive shared-memory words (stride S) and write
// consecutive output columns.
#include "dev_common.cuh"
#include "internal.h"

namespace gbconv {
namespace {

struct DirectArgs {
    const void *x;
    const void *w;
    const float *b;
    void *y;
    int N, C, D, H, W, OC;
    int k, stride, pad, kd, pad_d;
    int OD, OH, OW;
    int relu;
    int oc_blocks;
};

template <int TH, int TW, int OCB, int PX, int OCT>
struct Tile {
    static constexpr int LANES = TW / PX;
    static constexpr int OCG = OCB / OCT;
    static constexpr int NT = LANES * OCG * TH;
    static_assert(TW % PX == 0 && OCB % OCT == 0, "tile");
    static_assert(NT % 32 == 0 && NT <= 1024, "threads");
};

__host__ __device__ constexpr int halo_extent(int tile, int k, int s) {
    return (tile - 1) * s + k;
}

// K, S > 0: compile-time kernel size / stride; 0: taken from the arguments.
template <typename T, int K, int S, int TH, int TW, int OCB, int PX, int OCT>
__global__ void __launch_bounds__(Tile<TH, TW, OCB, PX, OCT>::NT)
direct_conv_kernel(const DirectArgs a) {
    using TL = Tile<TH, TW, OCB, PX, OCT>;
    constexpr int LANES = TL::LANES, OCG = TL::OCG, NT = TL::NT;
    const int k = K ? K : a.k;
    const int s = S ? S : a.stride;
    const int IHT = halo_extent(TH, k, s);
    const int IWT = halo_extent(TW, k, s);
    const int CF = a.C * a.kd;                 // (channel, frame tap) pairs
    const int KK = k * k;

    extern __shared__ float smem[];
    pdl_wait();   // launched with programmatic dependent launch: global memory after the predecessor
    float *wsm = smem;                         // [CF * k * k][OCB]
    float *xs = smem + CF * KK * OCB;          // [CF][IHT][IWT]

    const T *x = static_cast<const T *>(a.x);
    const T *w = static_cast<const T *>(a.w);
    T *y = static_cast<T *>(a.y);

    int z = blockIdx.z;
    const int ocb = z % a.oc_blocks; z /= a.oc_blocks;
    const int od = z % a.OD;
    const int n = z / a.OD;
    const int oc0 = ocb * OCB;
    const int oh0 = blockIdx.y * TH, ow0 = blockIdx.x * TW;
    const int ih0 = oh0 * s - a.pad, iw0 = ow0 * s - a.pad;
    const int id0 = od * s - a.pad_d;

    // Weight slab for this channel block: wsm[t][o] = w[oc0 + o][t].
    const int tapsz = CF * KK;
    for (int e = threadIdx.x; e < tapsz * OCB; e += NT) {
        const int o = e / tapsz, t = e - o * tapsz;
        const int oc = oc0 + o;
        wsm[t * OCB + o] = oc < a.OC ? Storage<T>::load(w + (int64_t)oc * tapsz + t) : 0.0f;
    }
    // Input halo, zero outside the input (the padding).
    const int plane = IHT * IWT;
    for (int e = threadIdx.x; e < CF * plane; e += NT) {
        const int cf = e / plane, r = e - cf * plane;
        const int ih = r / IWT, iw = r - ih * IWT;
        const int c = cf / a.kd, dz = cf - c * a.kd;
        const int gd = id0 + dz, gh = ih0 + ih, gw = iw0 + iw;
        float v = 0.0f;
        if (gd >= 0 && gd < a.D && gh >= 0 && gh < a.H && gw >= 0 && gw < a.W)
            v = Storage<T>::load(x + (((int64_t)n * a.C + c) * a.D + gd) * ((int64_t)a.H * a.W) +
                                 (int64_t)gh * a.W + gw);
        xs[e] = v;
    }
    __syncthreads();

    const int lane = threadIdx.x % LANES;
    const int ocg = (threadIdx.x / LANES) % OCG;
    const int row = threadIdx.x / (LANES * OCG);

    float acc[PX][OCT];
#pragma unroll
    for (int j = 0; j < PX; j++)
#pragma unroll
        for (int o = 0; o < OCT; o++) acc[j][o] = 0.0f;

    for (int cf = 0; cf < CF; cf++) {
#pragma unroll
        for (int ky = 0; ky < (K ? K : 1); ky++) {
            // K == 0 (runtime k) runs this body once and loops inside.
            for (int kyr = 0; kyr < (K ? 1 : k); kyr++) {
                const int kyy = K ? ky : kyr;
                const float *xrow = xs + (cf * IHT + row * s + kyy) * IWT;
                const float *wrow = wsm + ((cf * k + kyy) * k) * OCB + ocg * OCT;
#pragma unroll
                for (int kx = 0; kx < (K ? K : 1); kx++) {
                    for (int kxr = 0; kxr < (K ? 1 : k); kxr++) {
                        const int kxx = K ? kx : kxr;
                        float xv[PX];
#pragma unroll
                        for (int j = 0; j < PX; j++) xv[j] = xrow[(lane + LANES * j) * s + kxx];
                        float wv[OCT];
                        const float4 *w4 = reinterpret_cast<const float4 *>(wrow + kxx * OCB);
#pragma unroll
                        for (int o4 = 0; o4 < OCT / 4; o4++) {
                            float4 t4 = w4[o4];
                            wv[4 * o4 + 0] = t4.x; wv[4 * o4 + 1] = t4.y;
                            wv[4 * o4 + 2] = t4.z; wv[4 * o4 + 3] = t4.w;
                        }
#pragma unroll
                        for (int j = 0; j < PX; j++)
#pragma unroll
                            for (int o = 0; o < OCT; o++) acc[j][o] = fmaf(xv[j], wv[o], acc[j][o]);
                    }
                }
            }
        }
    }

    const int oh = oh0 + row;
    if (oh >= a.OH) return;
#pragma unroll
    for (int o = 0; o < OCT; o++) {
        const int oc = oc0 + ocg * OCT + o;
        if (oc >= a.OC) break;
        const float bias = a.b ? __ldg(a.b + oc) : 0.0f;
        T *yrow = y + ((((int64_t)n * a.OC + oc) * a.OD + od) * a.OH + oh) * a.OW;
#pragma unroll
        for (int j = 0; j < PX; j++) {
            const int ow = ow0 + lane + LANES * j;
            if (ow < a.OW) yrow[ow] = Storage<T>::from_float(epilogue(acc[j][o], bias, a.relu));
        }
    }
}

template <int TH, int TW, int OCB, int PX, int OCT>
size_t direct_smem_bytes(const Problem &p) {
    const int iht = halo_extent(TH, p.k, p.stride), iwt = halo_extent(TW, p.k, p.stride);
    return sizeof(float) * ((size_t)p.C * p.kd * p.k * p.k * OCB +
                            (size_t)p.C * p.kd * iht * iwt);
}

constexpr size_t kDirectSmemLimit = 200 * 1024;

template <typename T, int K, int S, int TH, int TW, int OCB, int PX, int OCT>
cudaError_t launch_tile(const Problem &p, const DirectArgs &a0, cudaStream_t st) {
    using TL = Tile<TH, TW, OCB, PX, OCT>;
    DirectArgs a = a0;
    a.oc_blocks = (p.OC + OCB - 1) / OCB;
    const size_t smem = direct_smem_bytes<TH, TW, OCB, PX, OCT>(p);
    auto kern = direct_conv_kernel<T, K, S, TH, TW, OCB, PX, OCT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((p.OW + TW - 1) / TW, (p.OH + TH - 1) / TH,
              (unsigned)((int64_t)p.N * p.OD * a.oc_blocks));
    if (log_enabled())
        log_line("direct_conv_kernel grid=%ux%ux%u block=%d smem=%zu tile=%dx%d oc_block=%d", grid.x, grid.y,
                 grid.z, TL::NT, smem, TH, TW, OCB);
    return launch_pdl(kern, grid, dim3(TL::NT), smem, st, a);
}

// Tile shapes: "wide" for >= 16 output channels, "narrow" otherwise.
#define GB_WIDE 4, 64, 32, 4, 16
#define GB_NARROW 8, 32, 8, 2, 8

template <typename T>
cudaError_t launch_typed(const Problem &p, const DirectArgs &a, cudaStream_t st) {
    const bool wide = p.OC >= 16;
    if (p.k == 3 && p.stride == 1)
        return wide ? launch_tile<T, 3, 1, GB_WIDE>(p, a, st) : launch_tile<T, 3, 1, GB_NARROW>(p, a, st);
    if (p.k == 3 && p.stride == 2)
        return wide ? launch_tile<T, 3, 2, GB_WIDE>(p, a, st) : launch_tile<T, 3, 2, GB_NARROW>(p, a, st);
    return wide ? launch_tile<T, 0, 0, GB_WIDE>(p, a, st) : launch_tile<T, 0, 0, GB_NARROW>(p, a, st);
}

}  // namespace

bool direct_supported(const Problem &p) {
    const size_t wide = direct_smem_bytes<4, 64, 32, 4, 16>(p);
    const size_t narrow = direct_smem_bytes<8, 32, 8, 2, 8>(p);
    if ((p.OC >= 16 ? wide : narrow) > kDirectSmemLimit) return false;
    if (stem_supported(p)) return true;   // persistent kernel, 1-D grid
    // The tile kernel's grid z is images x frames x output-channel blocks
    // (32 channels wide, 8 narrow); CUDA caps it at 65535.
    const int ocb = p.OC >= 16 ? 32 : 8;
    return (int64_t)p.N * p.OD * ((p.OC + ocb - 1) / ocb) <= 65535;
}

cudaError_t launch_direct(const Problem &p, const void *x, const void *w,
                          const float *b, void *y, cudaStream_t s) {
    if (stem_supported(p)) return launch_direct_stem(p, x, w, b, y, s);
    DirectArgs a{};
    a.x = x; a.w = w; a.b = b; a.y = y;
    a.N = p.N; a.C = p.C; a.D = p.D; a.H = p.H; a.W = p.W; a.OC = p.OC;
    a.k = p.k; a.stride = p.stride; a.pad = p.pad; a.kd = p.kd; a.pad_d = p.pad_d;
    a.OD = p.OD; a.OH = p.OH; a.OW = p.OW;
    a.relu = p.act == GBCONV_ACT_RELU;
    switch (p.dtype) {
    case GBCONV_F32: return launch_typed<float>(p, a, s);
    case GBCONV_F16: return launch_typed<__half>(p, a, s);
    default: return launch_typed<__nv_bfloat16>(p, a, s);
    }
}

}  // namespace gbconv
