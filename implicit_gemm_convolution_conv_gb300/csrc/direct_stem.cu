// Direct convolution for few-channel 3x3 layers (detection stems): C <= 4,
// k = 3, stride 1 or 2, conv2d.
//
// The operation is the compute shader of lpnh.cn/news/2745477 section 2.2
// (output-stationary, input coordinates derived from the output coordinate,
// zero padding, bias, then ReLU fused into the write-back as in section 4.4).
// On GB300 this layer is bound by HBM (it writes 32 output values per input
// pixel read) with the FP32 pipes nearly as busy, so the kernel is organised to
// keep the FMA pipes fed while the stores stream out:
//  - persistent warps; each owns one 32-channel output block and a contiguous
//    run of warp tiles of 16 output pixels (one output row segment), walked
//    with incremental coordinates (no division on the per-tile path);
//  - each lane keeps P pixels x Q channels of accumulators (8 x 2) and the
//    Q x C x 9 weights of its channels in registers for the whole kernel (the
//    page-5 Convolution3D backend's "several output channels per invocation,
//    packed weights", git.erdda.com/Tencent/ncnn/discussions/7001 section
//    3.2); channel pairs accumulate with packed fp32 FMA (fma.rn.f32x2);
//  - the input halo of the tiles ahead streams into a per-warp shared-memory
//    ring with cp.async: 16-byte chunks aligned to 4 elements (zero-filled
//    outside the input, which is the padding) when rows are 16-byte aligned,
//    single elements otherwise;
//  - smem reads are 16-byte vectors shared by the lanes of a pixel group;
//    outputs leave as 16-byte stores of 4 consecutive pixels.
// With POOL (a 2x2, stride-2 max pool fused after bias and ReLU, as page 1
// section 4.4 fuses conv, ReLU and pooling into one shader) a warp tile is 2
// output rows x 8 pixels: the two lane halves hold the two rows of the same
// pixels and channels, one shuffle takes the row maximum and adjacent pixel
// pairs in registers the column maximum, and only the pooled quarter of the
// output is written.
#include "dev_common.cuh"
#include "internal.h"

namespace gbconv {
namespace {

constexpr int kTileOc = 32;                 // output channels per warp
constexpr int kWarps = 4;                   // warps per CTA
constexpr int kRing = 3;            // halo buffers per warp

template <int S, int TILE>
struct StemGeom {
    static constexpr int K = 3;
    static constexpr int kTilePx = TILE;             // output pixels per warp tile
    // A halo row covers input columns [ix0 - 4, ix0 - 4 + kRowPad), where ix0
    // = tw * 16 * S is the first input column of the tile before padding; the
    // tap at pixel i, column kx reads position 4 - pad + i*S + kx.
    static constexpr int kChunks = ((kTilePx - 1) * S + K + 2 + 3) / 4 + 1;   // 16-B chunks per row
    static constexpr int kRowPad = kChunks * 4;
};

struct StemArgs {
    const void *x;
    const void *w;
    const float *b;
    void *y;
    int N, H, W, OC, OH, OW, pad;
    int YH, YW;                             // stored output (pooled when POOL)
    int tile_rows;                          // OH, or YH with POOL
    int tiles_w, oc_blocks;
    int tiles_per_img;                      // tile_rows * tiles_w
    long long pix_tiles;                    // N * OH * tiles_w
    int warps_per_ocb;
    int relu;
    int vec_load;
    int vec_store;
};

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, int bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct TilePos {
    int n, oh, tw;
    __device__ __forceinline__ void advance(int tiles_w, int OH) {
        if (++tw == tiles_w) {
            tw = 0;
            if (++oh == OH) { oh = 0; ++n; }
        }
    }
};

template <typename T, int C, int S, int PAD, int P, int Q, int MINB, bool POOL>
__global__ void __launch_bounds__(kWarps * 32, MINB)
direct_stem_kernel(const StemArgs a) {
    // Lane tile: P consecutive pixels x Q output channels, the channels taken
    // as Q/2 packed pairs; a warp covers 32/Q channel groups x (P*Q/P) pixel
    // groups = P*Q pixels x 32 channels. With POOL the two pixel groups are
    // two output rows of the same P pixels.
    constexpr int QP = Q / 2;
    static_assert(Q % 2 == 0 && 32 % Q == 0, "lane tile");
    static_assert(!POOL || (Q == 2 && P % 4 == 0), "pooled tile: two rows of P pixels");
    using G = StemGeom<S, POOL ? P : P * Q>;
    constexpr int kTilePx = G::kTilePx;
    constexpr int K = 3;
    constexpr int kRowsPerC = POOL ? S + K : K;                 // halo rows per input channel
    constexpr int kRows = C * kRowsPerC;
    constexpr int kBuf = kRows * G::kRowPad;                    // floats per raw buffer
    constexpr int kTasks = (kRows * G::kChunks + 31) / 32;      // 16-byte chunks per lane
    __shared__ __align__(16) float halo[kWarps][kRing][kBuf];     // halo ring

    // Programmatic dependent launch: the grid is one resident wave, so the
    // next kernel in the stream may launch now; this one reads global memory
    // only once its predecessor has completed.
    pdl_launch_dependents();
    pdl_wait();
    const int wid = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int gw = blockIdx.x * kWarps + wid;
    const int ocb = gw % a.oc_blocks;
    const int slot = gw / a.oc_blocks;                          // index among warps of this block
    if (slot >= a.warps_per_ocb) return;
    // Contiguous run of pixel tiles [t0, t1) for this warp.
    const long long t0 = a.pix_tiles * slot / a.warps_per_ocb;
    const long long t1 = a.pix_tiles * (slot + 1) / a.warps_per_ocb;
    if (t0 >= t1) return;
    const int ntiles = (int)(t1 - t0);

    const int pg = lane / (32 / Q);          // pixel group: pixels P*pg .. P*pg+P-1
    const int og = lane % (32 / Q);          // channel group: channels Q*og .. Q*og+Q-1
    const T *x = static_cast<const T *>(a.x);
    const T *w = static_cast<const T *>(a.w);
    T *y = static_cast<T *>(a.y);
    const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(&halo[wid][0][0]));
    const long long HW = (long long)a.H * a.W;

    // This lane's share of a halo fill, fixed for every tile: chunk e of the
    // (row, 16-byte chunk) grid for e = lane, lane + 32, ...
    int t_dst[kTasks], t_ky[kTasks], t_col[kTasks];
    long long t_off[kTasks];
#pragma unroll
    for (int k = 0; k < kTasks; ++k) {
        const int e = lane + 32 * k;
        const int row = e / G::kChunks, ch = e - row * G::kChunks;
        const int c = row / kRowsPerC, ky = row - c * kRowsPerC;
        t_dst[k] = e < kRows * G::kChunks ? row * G::kRowPad + 4 * ch : -1;
        t_ky[k] = ky;
        t_col[k] = 4 * ch;
        t_off[k] = (long long)c * HW + (long long)ky * a.W + 4 * ch;
    }

    TilePos pf;                              // next tile to prefetch (oh: tile row)
    pf.n = (int)(t0 / a.tiles_per_img);
    {
        const int r = (int)(t0 - (long long)pf.n * a.tiles_per_img);
        pf.oh = r / a.tiles_w;
        pf.tw = r - pf.oh * a.tiles_w;
    }
    TilePos cur = pf;

    // Stage the halo of tile `p` into ring slot `slot_i` (zero outside x).
    auto prefetch = [&](const TilePos &p, int slot_i) {
        const int iy0 = (POOL ? 2 * p.oh : p.oh) * S - a.pad;
        const int cx0 = p.tw * kTilePx * S - 4;          // input column of position 0
        if (sizeof(T) == 4 && a.vec_load) {
            const T *base = x + (long long)p.n * C * HW + (long long)iy0 * a.W + cx0;
            const uint32_t dst0 = sbase + (uint32_t)(slot_i * kBuf) * 4u;
#pragma unroll
            for (int k = 0; k < kTasks; ++k) {
                if (t_dst[k] < 0) continue;
                const int iy = iy0 + t_ky[k], ix = cx0 + t_col[k];
                int bytes = 0;
                if ((unsigned)iy < (unsigned)a.H && (unsigned)ix < (unsigned)a.W)
                    bytes = min(4, a.W - ix) * 4;
                cp_async16(dst0 + (uint32_t)t_dst[k] * 4u, bytes ? base + t_off[k] : x, bytes);
            }
        } else {
            const uint32_t dst0 = sbase + (uint32_t)(slot_i * kBuf) * 4u;
            const T *xn = x + (long long)p.n * C * HW;
            for (int e = lane; e < kRows * G::kRowPad; e += 32) {
                const int row = e / G::kRowPad, col = e - row * G::kRowPad;
                const int c = row / kRowsPerC, ky = row - c * kRowsPerC;
                const int iy = iy0 + ky, ix = cx0 + col;
                const bool ok = iy >= 0 && iy < a.H && ix >= 0 && ix < a.W;
                const T *src = ok ? xn + (long long)c * HW + (long long)iy * a.W + ix : x;
                if (sizeof(T) == 4) {
                    cp_async4(dst0 + (uint32_t)(row * G::kRowPad + col) * 4u, src, ok ? 4 : 0);
                } else {
                    halo[wid][slot_i][row * G::kRowPad + col] = ok ? Storage<T>::to_float(*src) : 0.0f;
                }
            }
        }
        cp_async_commit();
    };

    // Weights of this lane's Q output channels as channel pairs, and biases.
    float2 wp[QP][C * 9];
    float2 bp[QP];
#pragma unroll
    for (int jp = 0; jp < QP; ++jp) {
        float bb[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int oc = ocb * kTileOc + og * Q + 2 * jp + h;
            bb[h] = (a.b && oc < a.OC) ? __ldg(a.b + oc) : 0.0f;
        }
        bp[jp] = make_float2(bb[0], bb[1]);
#pragma unroll
        for (int q = 0; q < C * 9; ++q) {
            float v[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int oc = ocb * kTileOc + og * Q + 2 * jp + h;
                v[h] = oc < a.OC ? Storage<T>::load(w + (long long)oc * C * 9 + q) : 0.0f;
            }
            wp[jp][q] = make_float2(v[0], v[1]);
        }
    }
    // Output pointers of this lane's first channel, advanced per tile.
    const long long plane = (long long)a.OH * a.OW;
    const int oc_base = ocb * kTileOc + og * Q;

    // Fill the ring, then: wait for tile i, compute it, refill its slot.
#pragma unroll
    for (int i = 0; i < kRing - 1; ++i) {
        if (i < ntiles) {
            prefetch(pf, i);
            pf.advance(a.tiles_w, a.tile_rows);
        } else {
            cp_async_commit();
        }
    }
    // A pixel group's taps start at position 4 - PAD + P*pg*S of a halo row:
    // read whole aligned float4 vectors and pick at fixed offsets.
    constexpr int kSpanP = (P - 1) * S + K;
    constexpr int kPairs = 4 - PAD + kSpanP;
    constexpr int kVec = (kPairs + 3) / 4;
    for (int i = 0; i < ntiles; ++i) {
        const int si = i % kRing;
        if (i + kRing - 1 < ntiles) {
            prefetch(pf, (i + kRing - 1) % kRing);
            pf.advance(a.tiles_w, a.tile_rows);
        } else {
            cp_async_commit();
        }
        cp_async_wait<kRing - 1>();
        __syncwarp();
        float2 acc[P][QP];
#pragma unroll
        for (int ii = 0; ii < P; ++ii)
#pragma unroll
            for (int jp = 0; jp < QP; ++jp) acc[ii][jp] = bp[jp];
        const float *hb = &halo[wid][si][0] + (POOL ? pg * S * G::kRowPad : pg * P * S);
#pragma unroll
        for (int c = 0; c < C; ++c) {
#pragma unroll
            for (int ky = 0; ky < K; ++ky) {
                // {x, x} operands of the packed FMA over channel pairs.
                float2 xp[4 * kVec];
                const float *row = hb + (c * kRowsPerC + ky) * G::kRowPad;
#pragma unroll
                for (int v = 0; v < kVec; ++v) {
                    const float4 q4 = *reinterpret_cast<const float4 *>(row + 4 * v);
                    xp[4 * v] = make_float2(q4.x, q4.x);
                    xp[4 * v + 1] = make_float2(q4.y, q4.y);
                    xp[4 * v + 2] = make_float2(q4.z, q4.z);
                    xp[4 * v + 3] = make_float2(q4.w, q4.w);
                }
                const float2 *xv = xp + (4 - PAD);
#pragma unroll
                for (int kx = 0; kx < K; ++kx)
#pragma unroll
                    for (int ii = 0; ii < P; ++ii)
#pragma unroll
                        for (int jp = 0; jp < QP; ++jp) {
                            const int q = (c * K + ky) * K + kx;
                            acc[ii][jp] = __ffma2_rn(xv[ii * S + kx], wp[jp][q], acc[ii][jp]);
                        }
            }
        }
        __syncwarp();                          // dup buffer is rewritten next tile

        if constexpr (!POOL) {
            const int owl = cur.tw * kTilePx + pg * P;
            T *y0 = y + ((long long)cur.n * a.OC + oc_base) * plane + (long long)cur.oh * a.OW + owl;
    #pragma unroll
            for (int j = 0; j < Q; ++j) {
                if (oc_base + j >= a.OC) break;
    #pragma unroll
                for (int i4 = 0; i4 < P; i4 += 4) {
                    const int ow0 = owl + i4;
                    float o[4];
    #pragma unroll
                    for (int ii = 0; ii < 4; ++ii) {
                        const float2 v = acc[i4 + ii][j >> 1];
                        const float r = (j & 1) ? v.y : v.x;
                        o[ii] = a.relu ? fmaxf(r, 0.0f) : r;
                    }
                    T *yr = y0 + j * plane + i4;
                    if (a.vec_store && ow0 + 3 < a.OW) {
                        if (sizeof(T) == 4) {
                            *reinterpret_cast<float4 *>(yr) = make_float4(o[0], o[1], o[2], o[3]);
                        } else {
                            alignas(8) T h[4];
    #pragma unroll
                            for (int ii = 0; ii < 4; ++ii) h[ii] = Storage<T>::from_float(o[ii]);
                            *reinterpret_cast<uint2 *>(yr) = *reinterpret_cast<const uint2 *>(h);
                        }
                    } else {
    #pragma unroll
                        for (int ii = 0; ii < 4; ++ii)
                            if (ow0 + ii < a.OW) yr[ii] = Storage<T>::from_float(o[ii]);
                    }
                }
            }
        } else {
            // Row maximum across the lane halves (rows 0 / 1), then the column
            // maximum over pixel pairs; lanes of row 0 store 4 pooled pixels.
            const int pw0 = cur.tw * (P / 2);                      // first pooled column
            const long long yplane = (long long)a.YH * a.YW;
            T *y0 = y + ((long long)cur.n * a.OC + oc_base) * yplane + (long long)cur.oh * a.YW + pw0;
#pragma unroll
            for (int j = 0; j < Q; ++j) {
                float pm[P / 2];
#pragma unroll
                for (int i = 0; i < P / 2; ++i) {
                    float m[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float2 v2 = acc[2 * i + h][j >> 1];
                        float v = (j & 1) ? v2.y : v2.x;
                        v = a.relu ? fmaxf(v, 0.0f) : v;
                        m[h] = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
                    }
                    pm[i] = fmaxf(m[0], m[1]);
                }
                if (pg != 0 || oc_base + j >= a.OC) continue;
                T *yr = y0 + j * yplane;
#pragma unroll
                for (int i4 = 0; i4 < P / 2; i4 += 4) {
                    if (a.vec_store && pw0 + i4 + 3 < a.YW) {
                        if (sizeof(T) == 4) {
                            *reinterpret_cast<float4 *>(yr + i4) = make_float4(pm[i4], pm[i4 + 1], pm[i4 + 2], pm[i4 + 3]);
                        } else {
                            alignas(8) T h[4];
#pragma unroll
                            for (int ii = 0; ii < 4; ++ii) h[ii] = Storage<T>::from_float(pm[i4 + ii]);
                            *reinterpret_cast<uint2 *>(yr + i4) = *reinterpret_cast<const uint2 *>(h);
                        }
                    } else {
#pragma unroll
                        for (int ii = 0; ii < 4; ++ii)
                            if (pw0 + i4 + ii < a.YW) yr[i4 + ii] = Storage<T>::from_float(pm[i4 + ii]);
                    }
                }
            }
        }
        cur.advance(a.tiles_w, a.tile_rows);
    }
    cp_async_wait<0>();
}

// The lane tile (pixels x channels), and the resident CTAs per SM the
// register budget is sized for.
constexpr int kStemP = 8;
constexpr int kStemQ = 2;
constexpr int kStemMinBlocks = 3;
constexpr int kStemTilePx = kStemP * kStemQ;

template <typename T, int C, int S, int PAD, bool POOL>
cudaError_t launch_stem_csp(const Problem &p, const StemArgs &a0, cudaStream_t s) {
    StemArgs a = a0;
    auto kern = direct_stem_kernel<T, C, S, PAD, kStemP, kStemQ, kStemMinBlocks, POOL>;
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * 32, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    // Resident warps, split evenly over the output-channel blocks; no more
    // warps per block than pixel tiles.
    long long warps = (long long)sms * per_sm * kWarps;
    long long per_ocb = warps / a.oc_blocks;
    if (per_ocb < 1) per_ocb = 1;
    if (per_ocb > a.pix_tiles) per_ocb = a.pix_tiles;
    a.warps_per_ocb = (int)per_ocb;
    const long long total_warps = per_ocb * a.oc_blocks;
    const int grid = (int)((total_warps + kWarps - 1) / kWarps);
    if (log_enabled())
        log_line("direct_stem_kernel grid=%d block=%d warps_per_oc_block=%d oc_blocks=%d pixel_tiles=%lld", grid,
                 kWarps * 32, a.warps_per_ocb, a.oc_blocks, (long long)a.pix_tiles);
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kWarps * 32), 0, s, a);
}

template <typename T, int C, int S, int PAD>
cudaError_t launch_stem_cs(const Problem &p, const StemArgs &a, cudaStream_t s) {
    return p.pool ? launch_stem_csp<T, C, S, PAD, true>(p, a, s) : launch_stem_csp<T, C, S, PAD, false>(p, a, s);
}

// Layers this small (at most 65,536 outputs, no pool) are bound by the
// dependent launch and one memory round trip, not by bandwidth or the FMA
// pipes: one thread per output element issues all of its loads at once (the
// C x 9 input values of its window, zero outside the input, and its C x 9
// weights), then the FMAs and one store, with no halo ring to fill first.
// The output index is NCHW order (ow fastest), so a warp's stores are
// consecutive pixels of one channel plane.
constexpr long long kTinyOutputs = 1 << 16;
template <typename T, int C, int S>
__global__ void __launch_bounds__(128) direct_tiny_kernel(const StemArgs a) {
    pdl_launch_dependents();
    pdl_wait();
    const long long total = (long long)a.N * a.OC * a.OH * a.OW;
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int ow = (int)(i % a.OW);
    long long r = i / a.OW;
    const int oh = (int)(r % a.OH);
    r /= a.OH;
    const int oc = (int)(r % a.OC);
    const int n = (int)(r / a.OC);
    const T *x = static_cast<const T *>(a.x) + (long long)n * C * a.H * a.W;
    const T *w = static_cast<const T *>(a.w) + (long long)oc * C * 9;
    float xv[C * 9], wv[C * 9];
#pragma unroll
    for (int c = 0; c < C; ++c)
#pragma unroll
        for (int ky = 0; ky < 3; ++ky)
#pragma unroll
            for (int kx = 0; kx < 3; ++kx) {
                const int t = (c * 3 + ky) * 3 + kx;
                const int ih = (int)oh * S - a.pad + ky, iw = (int)ow * S - a.pad + kx;
                xv[t] = (ih >= 0 && ih < a.H && iw >= 0 && iw < a.W)
                            ? Storage<T>::load(x + ((size_t)c * a.H + ih) * a.W + iw)
                            : 0.0f;
                wv[t] = Storage<T>::load(w + t);
            }
    const float bias = a.b ? __ldg(a.b + oc) : 0.0f;
    float acc = 0.0f;
#pragma unroll
    for (int t = 0; t < C * 9; ++t) acc = fmaf(xv[t], wv[t], acc);
    static_cast<T *>(a.y)[i] = Storage<T>::from_float(epilogue(acc, bias, a.relu));
}

template <typename T, int C>
cudaError_t launch_tiny_c(const Problem &p, const StemArgs &a, cudaStream_t s) {
    const long long total = (long long)p.N * p.OC * p.OH * p.OW;
    const dim3 grid((unsigned)((total + 127) / 128));
    if (log_enabled()) log_line("direct_tiny_kernel grid=%u block=128 outputs=%lld", grid.x, total);
    if (p.stride == 1) return launch_pdl(direct_tiny_kernel<T, C, 1>, grid, dim3(128), 0, s, a);
    return launch_pdl(direct_tiny_kernel<T, C, 2>, grid, dim3(128), 0, s, a);
}

template <typename T, int C>
cudaError_t launch_stem_c(const Problem &p, const StemArgs &a, cudaStream_t s) {
    if (!p.pool && (long long)p.N * p.OC * p.OH * p.OW <= kTinyOutputs) return launch_tiny_c<T, C>(p, a, s);
    if (p.pad == 0)
        return p.stride == 1 ? launch_stem_cs<T, C, 1, 0>(p, a, s) : launch_stem_cs<T, C, 2, 0>(p, a, s);
    return p.stride == 1 ? launch_stem_cs<T, C, 1, 1>(p, a, s) : launch_stem_cs<T, C, 2, 1>(p, a, s);
}

template <typename T>
cudaError_t launch_stem_t(const Problem &p, const StemArgs &a, cudaStream_t s) {
    switch (p.C) {
    case 1: return launch_stem_c<T, 1>(p, a, s);
    case 2: return launch_stem_c<T, 2>(p, a, s);
    case 3: return launch_stem_c<T, 3>(p, a, s);
    default: return launch_stem_c<T, 4>(p, a, s);
    }
}

}  // namespace

bool stem_supported(const Problem &p) {
    return p.ndim == 2 && p.C <= 4 && p.k == 3 && (p.stride == 1 || p.stride == 2) &&
           p.pad <= 1 && (int64_t)p.N * p.OH * ((p.OW + kStemTilePx - 1) / kStemTilePx) < (1ll << 40);
}

cudaError_t launch_direct_stem(const Problem &p, const void *x, const void *w, const float *b,
                               void *y, cudaStream_t s) {
    StemArgs a{};
    a.x = x; a.w = w; a.b = b; a.y = y;
    a.N = p.N; a.H = p.H; a.W = p.W; a.OC = p.OC; a.OH = p.OH; a.OW = p.OW; a.pad = p.pad;
    a.YH = p.YH; a.YW = p.YW;
    // Tiles: 16 pixels of one row, or (pooled) 2 rows x 8 pixels = 4 pooled pixels.
    a.tile_rows = p.pool ? p.YH : p.OH;
    a.tiles_w = p.pool ? (p.YW + kStemP / 2 - 1) / (kStemP / 2) : (p.OW + kStemTilePx - 1) / kStemTilePx;
    a.oc_blocks = (p.OC + kTileOc - 1) / kTileOc;
    a.tiles_per_img = a.tile_rows * a.tiles_w;
    a.pix_tiles = (long long)p.N * a.tiles_per_img;
    a.relu = p.act == GBCONV_ACT_RELU;
    const int e = p.elt;
    a.vec_load = (p.W % 4 == 0) && ((uintptr_t)x % 16 == 0);
    a.vec_store = (p.YW % 4 == 0) && ((uintptr_t)y % (4 * e) == 0);
    switch (p.dtype) {
    case GBCONV_F32: return launch_stem_t<float>(p, a, s);
    case GBCONV_F16: return launch_stem_t<__half>(p, a, s);
    default: return launch_stem_t<__nv_bfloat16>(p, a, s);
    }
}

}  // namespace gbconv
