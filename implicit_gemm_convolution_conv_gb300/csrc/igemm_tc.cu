// Implicit-GEMM convolution on the 5th-generation tensor cores (tcgen05).
//
// GEMM view of the convolution sum (lpnh.cn/news/2745477 section 2.2; the
// Convolution3D extension of git.erdda.com/Tencent/ncnn/discussions/7001
// section 3.2): M = 128 output channels, N = NP consecutive output pixels in
// (n, od, oh, ow) order (a tile may cross rows, frames and images), K = taps
// x input channels. The A operand is the weight slab of one tap, packed once
// as [tap][OC][C] (the page's "re-arrange weights at export time", sections
// 2.3 and 4.2). The B operand is the input shifted by that tap, which TMA
// fetches straight from a channels-last copy of x in im2col mode: one load
// brings NP pixel rows of one 128-byte channel block, each pixel read at its
// stride-spaced position plus the tap offset, with positions outside the
// input read as zero (the padding). No im2col buffer exists. Because a tile
// is any run of NP pixels, NP is chosen so that the tiles spread evenly over
// the SMs (for example 148 tiles of 224 pixels for a 128 x 128 x 256-channel
// layer, where whole-row tiles gave 128 tiles for 152 SMs).
//
// Persistent kernel, one CTA per SM, tiles handed out round-robin. Roles
// (320 threads): warp 0 lane 0 issues TMA loads into a STAGES-deep
// shared-memory ring; warp 1 owns TMEM and lane 0 issues tcgen05.mma (M=128,
// N=NP, K=16, fp32 accumulate) into one of two TMEM accumulators, so the MMAs
// of tile i+1 run while the epilogue drains tile i. The accumulator's TMEM
// lanes are output channels and its columns pixels, so each of the eight
// epilogue warps (two per lane quadrant, alternate 32-pixel chunks) reads 32
// consecutive pixels of one channel per thread with tcgen05.ld, adds the
// bias, applies ReLU, rounds to fp16/bf16 and writes 16-byte vectors
// into the output. A warp's 32 channels x 32 pixels go through a 2 KB
// staging tile in shared memory (64-byte swizzle) and leave as one TMA tensor
// store, [channel][pixel] for NCHW/NCDHW output and [pixel][channel] for
// channels-last output; two staging tiles per warp let a store drain while the
// next chunk is converted. (Stores from registers, 16-byte pixel vectors into
// 32 different channel planes per warp instruction, cost the video-VAE
// Convolution3D a tenth of its time.) Chunks that no single box can cover (a
// chunk folded over two rows of the tile and not clipped by the image edge,
// or an unaligned output) are stored from registers. For channels-last
// output, neighbouring lanes swap one value so that each lane holds two
// channels of one pixel.
//
// fp32 storage runs on the same kernel as three TF32 products. x and the
// packed weights carry a hi half (the value with its 13 low mantissa bits
// cleared, exact in TF32) and a lo half (the exact remainder) along the
// channel axis, and every 32-channel K block takes three MMA groups,
// w_hi x_hi + w_hi x_lo + w_lo x_hi (kind::tf32), leaving about 2^-20
// relative error per product: the split-product way to run fp32 GEMMs on
// TF32 units. A 128-byte K block holds 32 fp32 channels as it holds 64 f16
// ones, so the swizzle and descriptors are the same. A stage holds both
// halves of a K block, [w_hi | w_lo] (one box of a 4-D view of the packed
// weights) and [x_hi | x_lo] (one box of a 5-D view of x for conv2d, two
// boxes for conv3d): one thread issuing TMA gets about one box per 300
// cycles, so the three products share each stage's loads. fp32 outputs are
// staged in 128-byte rows (128-byte swizzle).
//
// Every wait on an mbarrier is bounded (SM cycle counter); on expiry the
// kernel records an error word, lets its own in-flight copies and MMAs land,
// frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "dev_common.cuh"
#include "internal.h"

namespace gbconv {
__device__ unsigned int g_device_error;   // bit 0: a bounded wait ran out
}
#include "tc_ptx.cuh"

namespace gbconv {
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

using namespace tc;

constexpr int kEpiWarps = 8;                      // warps 2..9, two per TMEM lane quadrant
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxStages = 8;
constexpr int kTileOc = 128;                      // MMA M: output channels per tile
constexpr uint32_t kWStageBytes = 128u * 128u;    // 128 channel rows x 128 B
constexpr int kColChunk = 32;                     // accumulator columns per tcgen05.ld
// Per storage type: channels per 128-byte K block, whether fp32 is split
// into TF32 hi/lo halves, and the epilogue's staging (a warp's 32 x 32
// outputs, two tiles per epilogue warp).
template <typename T>
struct TcElt {
    static constexpr int kBlk = 128 / (int)sizeof(T);
    static constexpr bool kSplit = sizeof(T) == 4;
    static constexpr uint32_t kChunkBytes = 32u * 32u * (uint32_t)sizeof(T);
    static constexpr uint32_t kStageBytes = (uint32_t)kEpiWarps * 2u * kChunkBytes;
};

struct TcArgs {
    const float *b;
    void *y;
    int OC, OD, OH, OW;
    int k, pad, pad_d, stride;
    long long out_vol;     // OD * OH * OW: pixels of one image's output
    long long P;           // N * out_vol: output pixels, in (n, od, oh, ow) order
    int NP;                // pixels per tile = MMA N (a multiple of 32)
    int oc_tiles;
    int num_tiles;
    int cblocks;
    int cs;                // fp32 split: channels of the hi half (the lo half starts there)
    uint32_t xlo_off;      // fp32 split: byte offset of the x_lo rows in a stage (NP * 128)
    int ksteps;
    int stages;
    int relu;
    int vec_store;         // NC(D)HW register stores as 16-byte vectors (out_vol % 8 == 0, y aligned)
    int cl;                // channels-last output [N][OD][OH][OW][OC]
    int pair_store;        // channels-last: 4-byte stores of channel pairs (OC even, y 4-byte aligned)
    int tma_store;         // staged chunks leave as TMA tensor stores (tmY valid)
    int single_tile;       // every CTA owns at most one tile: the staging tiles reuse the stage ring
    int prefetch;          // L2 prefetch before the dependency wait: 1 x (read in place), 2 packed weights too
    int in_w, in_h, in_d;  // input extents (prefetch starts are clamped into them)
    uint32_t idesc;
    uint32_t tx_bytes;
    uint32_t tmem_cols;
    long long wait_limit_cycles;
};

// A tile: NP consecutive output pixels from linear pixel p0 (any row, frame
// or image boundary inside it), times 128 output channels from oc0.
struct TileCoord {
    long long p0;
    int n, od, oh, ow, oc0;
};
// Tile t: output-channel block fastest (consecutive CTAs share the pixels,
// the weights of a block are read by every CTA), then the pixel runs.
__device__ __forceinline__ TileCoord tile_coord(const TcArgs &a, int t) {
    TileCoord c;
    const int ot = t % a.oc_tiles;
    c.p0 = (long long)(t / a.oc_tiles) * a.NP;
    c.oc0 = ot * kTileOc;
    const long long n = c.p0 / a.out_vol;
    long long r = c.p0 - n * a.out_vol;
    const long long plane = (long long)a.OH * a.OW;
    c.n = (int)n;
    c.od = (int)(r / plane);
    r -= (long long)c.od * plane;
    c.oh = (int)(r / a.OW);
    c.ow = (int)(r - (long long)c.oh * a.OW);
    return c;
}

// Accumulator orientation: TMEM lane = output channel, column = pixel of the
// tile, so an epilogue thread owns consecutive pixels of one output channel,
// which is how NCHW stores them.
template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
igemm_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                const __grid_constant__ CUtensorMap tmY, const TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    // A stage: weights (one 16 KB tile, or [w_hi | w_lo] for fp32), then the
    // pixels (NP rows of 128 B, or x_hi rows then x_lo rows for fp32).
    constexpr uint32_t w_stage = TcElt<T>::kSplit ? 2u * kWStageBytes : kWStageBytes;
    const uint32_t x_stage = (TcElt<T>::kSplit ? 2u : 1u) * (uint32_t)a.NP * 128u;
    const uint32_t sW = base;
    const uint32_t sX = sW + (uint32_t)a.stages * w_stage;
    // Epilogue staging (1024-aligned): its own region, or, when every CTA
    // owns one tile, the stage ring, which is idle once that tile's MMAs are
    // done (all its loads were consumed; none follow).
    const uint32_t ring_end = sX + (uint32_t)a.stages * x_stage;
    const uint32_t sY = a.single_tile ? sW : ring_end;
    const uint32_t sBar = a.single_tile ? ring_end : ring_end + TcElt<T>::kStageBytes;
    const uint32_t full0 = sBar, empty0 = sBar + 8u * kMaxStages;
    const uint32_t tfull0 = sBar + 16u * kMaxStages, tempty0 = tfull0 + 16u;
    const uint32_t drain_bar = tempty0 + 16u;
    const uint32_t slot_addr = drain_bar + 8u;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem_raw + (slot_addr - raw));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_raw + (slot_addr + 4u - raw));

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    pdl_launch_dependents();

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
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
        if (a.tma_store) prefetch_tmap(&tmY);
        // The first ring's worth of the first tile's boxes, for operands that
        // no kernel of this call writes, start towards L2 while the previous
        // kernel finishes (L2 is where the GPU's writes become coherent, so
        // the loads after the wait cannot see stale data). An x box is
        // prefetched at the traversal start its load uses, and only where
        // that start lies inside the tensor in every dimension. (An im2col
        // coordinate must lie in the traversal range [-pad, extent - 1 + pad
        // - (k - 1)] of each dimension; a start clamped to 0 leaves that range
        // when its upper end is negative, as for D = 1 with k = 5 and pad 2,
        // and such a copy ends the context with an illegal instruction.)
        if (!TcElt<T>::kSplit && a.prefetch && (int)blockIdx.x < a.num_tiles) {
            const TileCoord tc = tile_coord(a, blockIdx.x);
            const int x0 = tc.ow * a.stride - a.pad, y0 = tc.oh * a.stride - a.pad, z0 = tc.od * a.stride - a.pad_d;
            const bool x_inside = x0 >= 0 && y0 >= 0 && z0 >= 0;
            int cb = 0, kx = 0, ky = 0, kz = 0, tap = 0;
            for (int it = 0; it < a.stages && it < a.ksteps; ++it) {
                const int c0 = cb * TcElt<T>::kBlk;
                if (a.prefetch & 2) tma_prefetch_l2_3d(&tmW, c0, tc.oc0, tap);
                if ((a.prefetch & 1) && x_inside && x0 + kx < a.in_w && y0 + ky < a.in_h && z0 + kz < a.in_d)
                    tma_prefetch_l2_im2col_5d(&tmX, c0, x0, y0, z0, tc.n, (uint16_t)kx, (uint16_t)ky,
                                              (uint16_t)kz);
                if (++cb == a.cblocks) {
                    cb = 0;
                    ++tap;
                    if (++kx == a.k) {
                        kx = 0;
                        if (++ky == a.k) { ky = 0; ++kz; }
                    }
                }
            }
        }
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
    // Set-up above overlaps the previous kernel's tail; global memory below.
    pdl_wait();

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
                // traversal position of the tile's first pixel
                const int x0 = tc.ow * a.stride - a.pad, y0 = tc.oh * a.stride - a.pad,
                          z0 = tc.od * a.stride - a.pad_d;
                int cb = 0, tap = 0, kx = 0, ky = 0, kz = 0;
                for (int it = 0; it < a.ksteps; ++it) {
                    const uint32_t fb = full0 + 8u * s;
                    if (!wait_bounded(empty0 + 8u * s, ph ^ 1u, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int c0 = cb * TcElt<T>::kBlk;
                    const uint32_t dw = sW + (uint32_t)s * w_stage, dx = sX + (uint32_t)s * x_stage;
                    mbar_arrive_expect_tx(fb, a.tx_bytes);
                    if constexpr (TcElt<T>::kSplit) {
                        tma_load_4d(dw, &tmW, fb, c0, tc.oc0, 0, tap);              // [w_hi | w_lo]
                        tma_load_im2col_5d(dx, &tmX, fb, c0, x0, y0, z0, tc.n, (uint16_t)kx, (uint16_t)ky,
                                           (uint16_t)kz);                            // x_hi
                        tma_load_im2col_5d(dx + a.xlo_off, &tmX, fb, a.cs + c0, x0, y0, z0, tc.n, (uint16_t)kx,
                                           (uint16_t)ky, (uint16_t)kz);              // x_lo
                    } else {
                        tma_load_3d(dw, &tmW, fb, c0, tc.oc0, tap);
                        tma_load_im2col_5d(dx, &tmX, fb, c0, x0, y0, z0, tc.n, (uint16_t)kx, (uint16_t)ky,
                                           (uint16_t)kz);
                    }
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
            if (!ok) raise_abort(abort_flag);
            // Let the copies already issued land before the CTA exits (on the
            // normal path the MMA warp consumed them all; after an abort some
            // may still be in flight). Copy q completes phase q / stages of
            // its stage's barrier, the last phase issued on it.
            const int first = issued > a.stages ? issued - a.stages : 0;
            for (int q = first; q < issued; ++q)
                wait_bounded(full0 + 8u * (q % a.stages), (uint32_t)(q / a.stages) & 1u, kDrainLimitCycles,
                             nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------ MMA issuer
            const uint64_t wdesc0 = sw128_kmajor_desc(sW), xdesc0 = sw128_kmajor_desc(sX);
            const uint32_t w_step = w_stage >> 4, x_step = x_stage >> 4;
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
                const uint32_t d = tmem + (uint32_t)(acc * a.NP);
                uint64_t wd = wdesc0 + (uint64_t)s * w_step, xd = xdesc0 + (uint64_t)s * x_step;
                for (int it = 0; it < a.ksteps; ++it) {
                    if (!wait_bounded(full0 + 8u * s, ph, limit, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // Four MMAs of 32 bytes of K each (16 f16/bf16 or 8 tf32);
                    // fp32: three groups, w_hi x_hi, w_hi x_lo, w_lo x_hi.
                    if constexpr (TcElt<T>::kSplit) {
                        const uint64_t wlo = wd + (kWStageBytes >> 4), xlo = xd + (a.xlo_off >> 4);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            tc_mma_tf32(d, wd + 2u * kk, xd + 2u * kk, a.idesc, (it | kk) != 0);
                            tc_mma_tf32(d, wd + 2u * kk, xlo + 2u * kk, a.idesc, 1u);
                            tc_mma_tf32(d, wlo + 2u * kk, xd + 2u * kk, a.idesc, 1u);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma(d, wd + 2u * kk, xd + 2u * kk, a.idesc, (it | kk) != 0);
                    }
                    tc_commit(empty0 + 8u * s);
                    wd += w_step;
                    xd += x_step;
                    if (++s == a.stages) {
                        s = 0;
                        ph ^= 1u;
                        wd = wdesc0;
                        xd = xdesc0;
                    }
                }
                if (ok) tc_commit(tfull0 + 8u * acc);
            }
            if (!ok) raise_abort(abort_flag);
            // Every MMA this thread issued completes before TMEM is freed,
            // also when the epilogue gave up before reading the last
            // accumulator.
            tc_commit(drain_bar);
            wait_bounded(drain_bar, 0, kDrainLimitCycles, nullptr);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // Warp w reads TMEM lane quadrant w % 4 (32 output channels); the two
        // warps of a quadrant take alternate 32-pixel column chunks.
        const int q = warp & 3;
        const int grp = (warp - 2) / 4;
        const int nchunks = a.NP / kColChunk;
        const uint32_t ystage = sY + (uint32_t)(warp - 2) * 2u * TcElt<T>::kChunkBytes;
        int nst = 0;             // TMA stores this warp has issued
        int local = 0;
        const long long n_img = a.P / a.out_vol;
        for (int t = blockIdx.x; t < a.num_tiles; t += gridDim.x, ++local) {
            const TileCoord tc = tile_coord(a, t);
            // the tile's first pixel within image tc.n's planes
            const long long v_tile = tc.p0 - (long long)tc.n * a.out_vol;
            const int acc = local & 1;
            const int oc = tc.oc0 + q * 32 + lane;
            const bool oc_ok = oc < a.OC;
            // the bias load's latency passes while the accumulator fills
            const float bias = (a.b && oc_ok) ? __ldg(a.b + oc) : 0.0f;
            int ok = 0;
            if (lane == 0)
                ok = wait_bounded(tfull0 + 8u * acc, (uint32_t)(local >> 1) & 1u, limit, abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) raise_abort(abort_flag);
                break;
            }
            tc_fence_after();
            const bool odd = lane & 1;
            const int oc_even = oc - (odd ? 1 : 0);
            // One 32-pixel chunk, pixels pc .. pc + 31 of the (n, od, oh, ow)
            // order (those past P do not exist). NC(D)HW: pixel pc is element
            // v0 of image n0's plane of each channel; channels-last: row pc
            // of the [P][OC] matrix.
            auto store_chunk = [&](const uint32_t (&v)[32], int ch) {
                const long long pc = tc.p0 + (long long)ch * kColChunk;
                if (pc >= a.P) return;
                const int nv = a.P - pc < kColChunk ? (int)(a.P - pc) : kColChunk;
                // image n0 and plane position v0 of pixel pc, stepped from the
                // tile's start (no 64-bit division per chunk)
                long long n0 = tc.n, v0 = v_tile + (long long)ch * kColChunk;
                if (!a.cl)
                    while (v0 >= a.out_vol) {
                        v0 -= a.out_vol;
                        ++n0;
                    }
                const bool one_image = v0 + kColChunk <= a.out_vol || n0 + 1 == n_img;
                // One box: a channels-last chunk always; an NC(D)HW chunk that
                // lies in one image's planes (the tensor's end clips the last).
                if (a.tma_store && (a.cl || one_image)) {
                    const uint32_t buf = ystage + (uint32_t)(nst & 1) * TcElt<T>::kChunkBytes;
                    if (nst >= 2) {
                        // The store that last used this buffer has read it.
                        if (lane == 0) bulk_wait_read<1>();
                        __syncwarp();
                    }
                    if constexpr (TcElt<T>::kSplit) {
                        // fp32: rows of 128 B, 16-byte unit u of row r at unit
                        // u ^ (r & 7) (128-byte swizzle).
                        if (a.cl) {
                            // [pixel][channel]: this lane's channel in every pixel row.
#pragma unroll
                            for (int e = 0; e < kColChunk; ++e) {
                                const float val = epilogue(__uint_as_float(v[e]), bias, a.relu);
                                const uint32_t addr = buf + (uint32_t)e * 128u +
                                                      ((((uint32_t)lane >> 2) ^ (uint32_t)(e & 7)) << 4) +
                                                      ((uint32_t)lane & 3u) * 4u;
                                asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(val) : "memory");
                            }
                        } else {
                            // [channel][pixel]: this lane's row, 32 pixels.
#pragma unroll
                            for (int u = 0; u < 8; ++u) {
                                const uint32_t addr = buf + (uint32_t)lane * 128u +
                                                      (((uint32_t)u ^ ((uint32_t)lane & 7u)) << 4);
                                asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                                             "f"(epilogue(__uint_as_float(v[4 * u]), bias, a.relu)),
                                             "f"(epilogue(__uint_as_float(v[4 * u + 1]), bias, a.relu)),
                                             "f"(epilogue(__uint_as_float(v[4 * u + 2]), bias, a.relu)),
                                             "f"(epilogue(__uint_as_float(v[4 * u + 3]), bias, a.relu))
                                             : "memory");
                            }
                        }
                    } else {
                      if (a.cl) {
                        // [pixel][channel] rows of 64 B; 16-byte unit u of row e
                        // sits at unit u ^ ((e >> 1) & 3) (64-byte swizzle).
                        // All 16 exchanges first, then the stores: no store
                        // waits behind a shuffle's latency.
                        const uint32_t cb = (uint32_t)(lane & ~1) * 2u;      // byte of channel pair
                        uint32_t pk[kColChunk / 2];
#pragma unroll
                        for (int e = 0; e < kColChunk; e += 2) {
                            const float v0f = epilogue(__uint_as_float(v[e]), bias, a.relu);
                            const float v1f = epilogue(__uint_as_float(v[e + 1]), bias, a.relu);
                            const float got = __shfl_xor_sync(0xffffffffu, odd ? v0f : v1f, 1);
                            const typename Storage<T>::Pair pr = Storage<T>::pack2(odd ? got : v0f, odd ? v1f : got);
                            pk[e / 2] = *reinterpret_cast<const uint32_t *>(&pr);
                        }
#pragma unroll
                        for (int e = 0; e < kColChunk; e += 2) {
                            const int row = e + (odd ? 1 : 0);
                            const uint32_t addr = buf + (uint32_t)row * 64u +
                                                  ((((cb >> 4) ^ (uint32_t)((row >> 1) & 3)) << 4) | (cb & 15u));
                            asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(pk[e / 2]) : "memory");
                        }
                      } else {
                        // [channel][pixel] rows of 64 B: this lane's channel, 32 pixels.
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            typename Storage<T>::Pair h[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                h[e] = Storage<T>::pack2(epilogue(__uint_as_float(v[8 * u + 2 * e]), bias, a.relu),
                                                         epilogue(__uint_as_float(v[8 * u + 2 * e + 1]), bias, a.relu));
                            const uint32_t addr = buf + (uint32_t)lane * 64u +
                                                  (((uint32_t)u ^ (uint32_t)((lane >> 1) & 3)) << 4);
                            const uint4 hv = *reinterpret_cast<const uint4 *>(h);
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(hv.x), "r"(hv.y),
                                         "r"(hv.z), "r"(hv.w)
                                         : "memory");
                        }
                      }
                    }
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        const int chan = tc.oc0 + q * 32;
                        if (a.cl)
                            tma_store_2d(&tmY, buf, chan, (int)pc);
                        else
                            tma_store_3d(&tmY, buf, (int)v0, chan, (int)n0);
                        bulk_commit_group();
                    }
                    ++nst;
                    return;
                }
                if (a.cl) {
                    T *const yrow = static_cast<T *>(a.y) + pc * a.OC;     // pixel pc, channel 0
                    if (!TcElt<T>::kSplit && a.pair_store) {
                        // Even lanes keep pixel e, odd lanes pixel e + 1; each
                        // lane gets its partner's value of that pixel and
                        // stores the channel pair (oc_even, oc_even + 1).
                        const bool oc_pair_ok = oc_even < a.OC;
#pragma unroll
                        for (int e = 0; e < kColChunk; e += 2) {
                            const float v0f = epilogue(__uint_as_float(v[e]), bias, a.relu);
                            const float v1f = epilogue(__uint_as_float(v[e + 1]), bias, a.relu);
                            const float got = __shfl_xor_sync(0xffffffffu, odd ? v0f : v1f, 1);
                            const typename Storage<T>::Pair pr =
                                Storage<T>::pack2(odd ? got : v0f, odd ? v1f : got);
                            const int px = e + (odd ? 1 : 0);
                            if (oc_pair_ok && px < nv)
                                *reinterpret_cast<typename Storage<T>::Pair *>(yrow + (long long)px * a.OC + oc_even) = pr;
                        }
                    } else if (oc_ok) {
#pragma unroll
                        for (int e = 0; e < kColChunk; ++e)
                            if (e < nv)
                                yrow[(long long)e * a.OC + oc] =
                                    Storage<T>::from_float(epilogue(__uint_as_float(v[e]), bias, a.relu));
                    }
                    return;
                }
                if (!oc_ok) return;
                if (!TcElt<T>::kSplit && a.vec_store && nv == kColChunk && v0 + kColChunk <= a.out_vol) {
                    // 16-byte vectors of 8 consecutive pixels of one plane.
                    T *dst = static_cast<T *>(a.y) + ((long long)n0 * a.OC + oc) * a.out_vol + v0;
#pragma unroll
                    for (int i8 = 0; i8 < kColChunk / 8; ++i8) {
                        typename Storage<T>::Pair h[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            h[e] = Storage<T>::pack2(epilogue(__uint_as_float(v[8 * i8 + 2 * e]), bias, a.relu),
                                                     epilogue(__uint_as_float(v[8 * i8 + 2 * e + 1]), bias, a.relu));
                        *reinterpret_cast<uint4 *>(dst + 8 * i8) = *reinterpret_cast<const uint4 *>(h);
                    }
                } else {
                    // pixel by pixel, moving to the next image's plane at its end
                    long long n = n0, vv = v0;
#pragma unroll
                    for (int e = 0; e < kColChunk; ++e) {
                        if (e < nv)
                            static_cast<T *>(a.y)[(n * a.OC + oc) * a.out_vol + vv] =
                                Storage<T>::from_float(epilogue(__uint_as_float(v[e]), bias, a.relu));
                        if (++vv == a.out_vol) { vv = 0; ++n; }
                    }
                }
            };
            // Chunks grp, grp + 2, ...: the next chunk's TMEM load is in
            // flight while the current one is converted and stored. A CTA
            // with a single tile has nothing for its epilogue to hide under,
            // and there a TMEM load in flight slows the staging stores of the
            // chunk before it (measured on the 128 x 128 x 256-channel layer:
            // 1.76 against 1.57 us per epilogue), so it loads each chunk when
            // it needs it.
            const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * a.NP);
            uint32_t va[32], vb[32];
            int ch = grp;
            if (a.single_tile) {
                for (; ch < nchunks; ch += 2) {
                    tmem_ld32(tl + (uint32_t)(ch * kColChunk), va);
                    tmem_ld_wait();
                    store_chunk(va, ch);
                }
            }
            if (ch < nchunks) tmem_ld32(tl + (uint32_t)(ch * kColChunk), va);
            while (ch < nchunks) {
                tmem_ld_wait();
                if (ch + 2 < nchunks) tmem_ld32(tl + (uint32_t)((ch + 2) * kColChunk), vb);
                store_chunk(va, ch);
                ch += 2;
                if (ch >= nchunks) break;
                tmem_ld_wait();
                if (ch + 2 < nchunks) tmem_ld32(tl + (uint32_t)((ch + 2) * kColChunk), va);
                store_chunk(vb, ch);
                ch += 2;
            }
            tmem_ld_wait();
            // All reads of this accumulator by this warp are done: hand it back.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8u * acc);
        }
    }

    // The staging tiles must have been read before the CTA's shared memory
    // goes away; the stores' global writes complete with the grid.
    if (warp >= 2 && lane == 0) bulk_wait_read_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

// x [N][C][S] -> xc [N][S][Cp], zero in channels C..Cp-1 (S = D*H*W).
// A CTA moves 64 channels x 256 positions (32 KB of 16-bit values) through
// shared memory, all of its loads in flight at once (8 per thread): loads
// are 16-byte vectors along a channel's positions (32 lanes = 512 contiguous
// bytes), stores 16-byte vectors of 8 channels (8 lanes = one position's 128
// contiguous bytes). The shared tile keeps a channel's row of positions in
// 16-byte chunks whose index is XOR-ed with (channel / 8) % 8, so the column
// reads of the store phase hit 16 different banks per warp. With 16-byte
// rows (S % 8 == 0, x aligned) the loads are cp.async copies into the tile,
// which hold no registers: 32 registers a thread, 7 CTAs per SM (4 with the
// loads staged through registers; the video-VAE Convolution3D's 1,200
// blocks then took two full waves).
constexpr int kClC = 64, kClS = 256;
template <typename T, bool VEC>
__device__ __forceinline__ void to_channels_last_block(const T *__restrict__ x, T *__restrict__ xc, int C, int Cp,
                                                       int64_t S, int bx, int by, int bz, T (*tile)[kClS]) {
    const int64_t s0 = (int64_t)bx * kClS;
    const int c0 = by * kClC;
    const int n = bz;
    const T *xn = x + (int64_t)n * C * S;
    T *xcn = xc + (int64_t)n * S * Cp;
    constexpr int kIter = kClC * kClS / 8 / 256;
    if constexpr (VEC) {
        // 16-byte copies straight into the swizzled tile (S % 8 == 0 and x
        // 16-byte aligned: a vector is whole or past the tensor, where the
        // copy reads nothing and zero-fills); all of a thread's copies are in
        // flight at once and hold no registers.
        const uint32_t tbase = smem_u32(&tile[0][0]);
#pragma unroll
        for (int i = 0; i < kIter; ++i) {
            const int v = threadIdx.x + 256 * i;
            const int cl = v / (kClS / 8), p8 = v % (kClS / 8);
            const int cc = c0 + cl;
            const int64_t s = s0 + p8 * 8;
            const bool in = cc < C && s < S;
            const T *src = in ? xn + (int64_t)cc * S + s : xn;
            const uint32_t dst = tbase + (uint32_t)(cl * kClS + (p8 ^ ((cl >> 3) & 7)) * 8) * (uint32_t)sizeof(T);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(in ? 16 : 0)
                         : "memory");
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
        uint4 buf[kIter];
#pragma unroll
        for (int i = 0; i < kIter; ++i) {
            const int v = threadIdx.x + 256 * i;
            const int cl = v / (kClS / 8), p8 = v % (kClS / 8);
            const int cc = c0 + cl;
            const int64_t s = s0 + p8 * 8;
            alignas(16) T e[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) e[j] = (cc < C && s + j < S) ? xn[(int64_t)cc * S + s + j] : T(0.0f);
            buf[i] = *reinterpret_cast<const uint4 *>(e);
        }
#pragma unroll
        for (int i = 0; i < kIter; ++i) {
            const int v = threadIdx.x + 256 * i;
            const int cl = v / (kClS / 8), p8 = v % (kClS / 8);
            *reinterpret_cast<uint4 *>(&tile[cl][(p8 ^ ((cl >> 3) & 7)) * 8]) = buf[i];
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kIter; ++i) {
        const int v = threadIdx.x + 256 * i;
        const int cch = v % 8, pos = v / 8;
        const int cc = c0 + cch * 8;
        const int64_t s = s0 + pos;
        if (s < S && cc < Cp) {
            const int col = (((pos >> 3) ^ cch) << 3) | (pos & 7);
            alignas(16) T vals[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) vals[j] = tile[cch * 8 + j][col];
            *reinterpret_cast<uint4 *>(xcn + s * Cp + cc) = *reinterpret_cast<const uint4 *>(vals);
        }
    }
}
template <typename T, bool VEC>
__global__ void __launch_bounds__(256, 7)
to_channels_last_kernel(const T *__restrict__ x, T *__restrict__ xc, int C, int Cp, int64_t S) {
    __shared__ __align__(16) T tile[kClC][kClS];
    pdl_launch_dependents();   // the GEMM behind launches once every CTA here has started
    pdl_wait();                // global memory only once the previous kernel is complete
    to_channels_last_block<T, VEC>(x, xc, C, Cp, S, blockIdx.x, blockIdx.y, blockIdx.z, tile);
}

// wp[tap][oc][cp] = w[oc][c][tap] for c < C, zero for C <= cp < Cp. A CTA
// handles ocpb (1 to 8, at most 512 16-byte vectors' worth: pack_oc_block)
// output channels, 64 channels and up to 32 taps. When all taps
// fit and the block is whole, each output channel's part of w is one
// contiguous run of 64 * taps elements, read as 16-byte vectors; a thread
// issues all of its loads (at most 2) before it writes any to shared memory,
// so the CTA waits for one memory round trip. Other blocks read element by
// element in batches of 8 loads. Each (tap, output channel) pair's 64
// channels then leave as one 128-byte run of wp.
constexpr int kPkC = 64, kPkT = 32, kPkOc = 8;
// Output channels per pack block: the largest power of two up to 8 whose
// block is at most 512 vectors of 8 elements (two loads per thread).
inline int pack_oc_block(int taps) {
    const int tn = taps < kPkT ? taps : kPkT;
    int o = kPkOc;
    while (o > 1 && o * kPkC * tn / 8 > 512) o /= 2;
    return o;
}
template <typename T>
__device__ __forceinline__ void pack_tc_block(const T *__restrict__ w, T *__restrict__ wp, int OC, int C, int Cp,
                                              int taps, int ocpb, int bx, int by, int bz,
                                              T (*tile)[kPkC][kPkT + 1]) {
    static_assert(sizeof(T) == 2, "16-bit weights");
    const int oc0 = bx * ocpb, c0 = by * kPkC, t0 = bz * kPkT;
    const int tn = taps - t0 < kPkT ? taps - t0 : kPkT;
    const bool vec = t0 == 0 && tn == taps && c0 + kPkC <= C && oc0 + ocpb <= OC &&
                     ((int64_t)C * taps) % 8 == 0 && ((uintptr_t)w % 16) == 0;
    if (vec) {
        const int vpr = kPkC * taps / 8;                      // vectors per output channel's run
        // pack_oc_block keeps a block within 512 vectors: two per thread
        constexpr int kMaxV = 512 / 256;
        uint4 buf[kMaxV];
#pragma unroll
        for (int k = 0; k < kMaxV; ++k) {
            const int v = threadIdx.x + 256 * k;
            if (v < ocpb * vpr) {
                const int o = v / vpr, r = v - o * vpr;
                buf[k] = __ldg(reinterpret_cast<const uint4 *>(w + ((int64_t)(oc0 + o) * C + c0) * taps) + r);
            }
        }
#pragma unroll
        for (int k = 0; k < kMaxV; ++k) {
            const int v = threadIdx.x + 256 * k;
            if (v < ocpb * vpr) {
                const int o = v / vpr, r = v - o * vpr;
                const T *e = reinterpret_cast<const T *>(&buf[k]);
                int j = r * 8;
                int cl = j / taps, tl = j - cl * taps;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    tile[o][cl][tl] = e[q];
                    if (++tl == taps) { tl = 0; ++cl; }
                }
            }
        }
    } else {
        const int per_oc = kPkC * tn;
        for (int e0 = 0; e0 < ocpb * per_oc; e0 += 8 * 256) {
            T v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int e = e0 + 256 * k + threadIdx.x;
                const int o = e / per_oc, r = e - o * per_oc;
                const int cl = r / tn, tl = r - cl * tn;
                const int oc = oc0 + o, c = c0 + cl;
                v[k] = (e < ocpb * per_oc && oc < OC && c < C) ? w[((int64_t)oc * C + c) * taps + t0 + tl] : T(0.0f);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int e = e0 + 256 * k + threadIdx.x;
                if (e < ocpb * per_oc) {
                    const int o = e / per_oc, r = e - o * per_oc;
                    const int cl = r / tn, tl = r - cl * tn;
                    tile[o][cl][tl] = v[k];
                }
            }
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < tn * ocpb * kPkC; e += blockDim.x) {
        const int cl = e % kPkC, r = e / kPkC;
        const int o = r % ocpb, tl = r / ocpb;
        const int oc = oc0 + o, cp = c0 + cl;
        if (oc < OC && cp < Cp) wp[((int64_t)(t0 + tl) * OC + oc) * Cp + cp] = tile[o][cl][tl];
    }
}

// CTA b of a grid that holds npk CTAs of one pass and nlay of another, the
// pass with fewer CTAs first (measured: the other order leaves the smaller
// pass trailing the larger one). Sets *pack and returns the index within the
// pass.
__device__ __forceinline__ int prep_block_index(int b, int npk, int nlay, bool *pack) {
    if (npk <= nlay) {
        *pack = b < npk;
        return *pack ? b : b - npk;
    }
    *pack = b >= nlay;
    return *pack ? b - nlay : b;
}

// Both passes in front of the GEMM when the weights come as OIHW: npk CTAs
// do the weight-pack blocks (grid pkx x pky x pkz, x fastest) and nlay the
// layout blocks (grid clx x cly x N). The passes touch disjoint memory, so
// one grid runs them side by side and the GEMM waits on one launch.
template <typename T>
constexpr size_t prep_tile_bytes() {
    return sizeof(T) * kClC * kClS > sizeof(T) * kPkOc * kPkC * (kPkT + 1) ? sizeof(T) * kClC * kClS
                                                                          : sizeof(T) * kPkOc * kPkC * (kPkT + 1);
}
// MINB: resident CTAs per SM the registers are sized for. A grid that fits
// on the SMs at 4 CTAs each keeps 64 registers (the pack blocks' loads all in
// flight, no spills); a larger one (the video-VAE Convolution3D's 1,328
// blocks) runs 6 per SM, two waves instead of three (measured: its call
// 94.9 -> 90.5 us), at the cost of a few spilled registers in the pack blocks.
template <typename T, bool VEC, int MINB>
__global__ void __launch_bounds__(256, MINB)
prep_tc_kernel(const T *__restrict__ x, T *__restrict__ xc, int C, int Cp, int64_t S, int clx, int cly,
               const T *__restrict__ w, T *__restrict__ wp, int OC, int taps, int ocpb, int pkx, int pky, int npk,
               int nlay) {
    __shared__ __align__(16) unsigned char tile[prep_tile_bytes<T>()];
    pdl_launch_dependents();   // the GEMM behind launches once every CTA here has started
    pdl_wait();                // global memory only once the previous kernel is complete
    bool pack;
    const int q = prep_block_index(blockIdx.x, npk, nlay, &pack);
    if (pack)
        pack_tc_block<T>(w, wp, OC, C, Cp, taps, ocpb, q % pkx, (q / pkx) % pky, q / (pkx * pky),
                         reinterpret_cast<T (*)[kPkC][kPkT + 1]>(tile));
    else
        to_channels_last_block<T, VEC>(x, xc, C, Cp, S, q % clx, (q / clx) % cly, q / (clx * cly),
                                       reinterpret_cast<T (*)[kClS]>(tile));
}

// The weight pack for 16-bit data without shared memory: a grid of small
// CTAs (128 threads, at most 80 registers each), one of which fits on an SM
// next to a resident CTA of the tensor-core GEMM (the GEMM's shared memory
// stays within 226 KB for this). The grid can therefore launch behind the
// previous GEMM and wait at the dependency barrier on its SMs, and it lets
// the next GEMM launch and set up while it works. An item is one output
// channel oc, 64 channels and 8 taps: lane l takes channels 2l and 2l + 1,
// issues all 16 loads of its 8 taps (2-byte elements, the run of taps of
// each channel is contiguous in OIHW) before it stores, and writes
// wp[tap][oc][c .. c+1] as one 32-bit word per tap, so a warp writes each
// (tap, oc) row's 64 channels as 128 contiguous bytes; channels C .. Cp-1 are
// zeros.
constexpr int kPrThreads = 128;
template <typename T>
__global__ void __launch_bounds__(kPrThreads, 6)
pack_rt_kernel(const unsigned short *__restrict__ w, unsigned int *__restrict__ wp, int OC, int C, int Cp, int taps,
               long long items) {
    static_assert(sizeof(T) == 2, "16-bit weights");
    pdl_launch_dependents();   // the GEMM behind may launch and set up now
    pdl_wait();                // wp only once the previous kernel (which may read it) is complete
    const int lane = threadIdx.x & 31;
    const long long nw = (long long)gridDim.x * (kPrThreads / 32);
    const int pkb = (Cp + 63) / 64, pkt = (taps + 7) / 8;
    for (long long q = (long long)(threadIdx.x >> 5) * gridDim.x + blockIdx.x; q < items; q += nw) {
        const int oc = (int)(q / (pkb * pkt));
        const int rem = (int)(q - (long long)oc * pkb * pkt);
        const int c = (rem / pkt) * 64 + 2 * lane, t0 = (rem % pkt) * 8;
        if (c >= Cp) continue;
        const unsigned short *w0 = w + ((long long)oc * C + c) * taps;
        uint32_t pr[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int t = t0 + k;
            const uint32_t lo = (t < taps && c < C) ? (uint32_t)__ldg(w0 + t) : 0u;
            const uint32_t hi = (t < taps && c + 1 < C) ? (uint32_t)__ldg(w0 + taps + t) : 0u;
            pr[k] = lo | (hi << 16);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int t = t0 + k;
            if (t < taps) wp[(((long long)t * OC + oc) * Cp + c) / 2] = pr[k];
        }
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

PFN_cuTensorMapEncodeIm2col_v12000 get_encode_im2col() {
    static PFN_cuTensorMapEncodeIm2col_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeIm2col_v12000>(p);
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

// Tile geometry: NP consecutive output pixels (a multiple of 32, at most
// 256: the MMA's N) per tile, and the depth of the stage ring.
struct TileGeom {
    int NP, stages;
    bool single_tile;      // tiles <= SMs: the epilogue stages its outputs in the idle ring
};

uint32_t ystage_bytes(const Problem &p) {
    return p.dtype == GBCONV_F32 ? TcElt<float>::kStageBytes : TcElt<__half>::kStageBytes;
}

int64_t out_pixels(const Problem &p) { return (int64_t)p.N * p.out_vol; }

// Ring depth for NP pixels per tile (0 when two stages do not fit).
int stages_for(const Problem &p, int np, bool single) {
    const int split = p.dtype == GBCONV_F32 ? 2 : 1;
    const int stage_bytes = split * ((int)kWStageBytes + np * 128);
    const int fixed = 1024 + (single ? 0 : (int)ystage_bytes(p)) + 256;
    // 226 KB at most, so that a CTA of the small layout / pack grid (no
    // shared memory of its own) still fits on the SM next to this one
    int st = (226 * 1024 - fixed) / stage_bytes;
    if (st > kMaxStages) st = kMaxStages;
    // the epilogue's staging reuses the ring of a single-tile CTA
    if (single && (int64_t)st * stage_bytes < (int64_t)ystage_bytes(p)) return 0;
    return st >= 2 ? st : 0;
}

// Pixels per tile: tiles are runs of consecutive output pixels (TMA im2col
// loads cross rows, frames and images), so any multiple of 32 up to 256
// works. The choice minimises waves x (one MMA's cycles), with the measured
// f16 MMA time at M = 128 taken as max(N / 2, 32 + N / 4) cycles (full rate
// from N = 128; below that the shared-memory operand reads set it); ties go
// to larger tiles. Every MMA of a K step has this N, so the K loop length
// cancels out.
TileGeom choose_geom(const Problem &p, int sms) {
    TileGeom g{};
    const int64_t P = out_pixels(p);
    const int64_t oc_tiles = (p.OC + kTileOc - 1) / kTileOc;
    int64_t best_cost = -1;
    for (int np = 256; np >= 32; np -= 32) {
        const int64_t tiles = (P + np - 1) / np * oc_tiles;
        const bool single = tiles <= sms;
        const int st = stages_for(p, np, single);
        if (st == 0) continue;
        const int64_t waves = (tiles + sms - 1) / sms;
        const int64_t mma = np / 2 > 32 + np / 4 ? np / 2 : 32 + np / 4;
        const int64_t cost = waves * mma;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            g.NP = np;
            g.stages = st;
            g.single_tile = single;
        }
    }
    return g;
}

size_t smem_bytes(const TileGeom &g, const Problem &p) {
    const size_t split = p.dtype == GBCONV_F32 ? 2 : 1;
    return 1024 + (size_t)g.stages * split * (kWStageBytes + (size_t)g.NP * 128) +
           (g.single_tile ? 0 : ystage_bytes(p)) + 256;
}

uint32_t tmem_cols_for(int cols) {
    uint32_t c = 32;
    while (c < (uint32_t)cols) c <<= 1;
    return c;
}

// Pixel-box corners of the im2col traversal along W, H and D: positions run
// from -pad (front) to extent - 1 + pad_back - (k - 1), i.e. one per output
// coordinate at the conv stride. The 5-D form holds corners in [-16, 15].
struct Corners {
    int lo[3], hi[3];
    bool ok;
};
Corners im2col_corners(const Problem &p) {
    Corners c{};
    c.lo[0] = c.lo[1] = -p.pad;
    c.hi[0] = c.hi[1] = p.pad - (p.k - 1);
    c.lo[2] = -p.pad_d;
    c.hi[2] = p.pad_d_back - (p.kd - 1);
    c.ok = true;
    for (int i = 0; i < 3; ++i)
        if (c.lo[i] < -16 || c.lo[i] > 15 || c.hi[i] < -16 || c.hi[i] > 15) c.ok = false;
    return c;
}

template <typename T>
cudaError_t launch_tc_typed(const Problem &p, const void *xc, const void *wp, const float *b,
                            void *y, cudaStream_t s) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
    PFN_cuTensorMapEncodeIm2col_v12000 encode_im2col = get_encode_im2col();
    if (!encode || !encode_im2col) return cudaErrorInvalidValue;
    DevInfo info;
    cudaError_t e = dev_info(&info);
    if (e != cudaSuccess) return e;
    const TileGeom g = choose_geom(p, info.sms);
    if (g.NP == 0) return cudaErrorInvalidValue;
    constexpr bool split = TcElt<T>::kSplit;
    constexpr int blk = TcElt<T>::kBlk;
    constexpr cuuint64_t elt = sizeof(T);
    const int Cp = tc_row_channels(p);     // channels of a staged row (both halves for fp32)
    const CUtensorMapDataType dt = split ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                         : (p.dtype == GBCONV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    const int64_t P = out_pixels(p);

    alignas(64) CUtensorMap tmX, tmW, tmY;
    std::memset(&tmY, 0, sizeof(tmY));
    const int Cs = split ? tc_split_half(p.C) : 0;
    {
        // Channels-last input as {Cp, W, H, D, N}, read in im2col mode: a load
        // is NP consecutive output pixels x one 128-byte K block of channels,
        // each pixel taken at its stride-spaced position shifted by the tap;
        // taps reaching outside the input read zeros (the padding).
        const Corners c = im2col_corners(p);
        if (!c.ok) return cudaErrorInvalidValue;
        const cuuint64_t dims[5] = {(cuuint64_t)Cp, (cuuint64_t)p.W, (cuuint64_t)p.H,
                                    (cuuint64_t)p.D, (cuuint64_t)p.N};
        const cuuint64_t strides[4] = {(cuuint64_t)Cp * elt, (cuuint64_t)Cp * elt * p.W,
                                       (cuuint64_t)Cp * elt * p.W * p.H,
                                       (cuuint64_t)Cp * elt * p.W * p.H * p.D};
        const cuuint32_t es[5] = {1, (cuuint32_t)p.stride, (cuuint32_t)p.stride,
                                  (cuuint32_t)(p.ndim == 3 ? p.stride : 1), 1};
        if (encode_im2col(&tmX, dt, 5, const_cast<void *>(xc), dims, strides, c.lo, c.hi, (cuuint32_t)blk,
                          (cuuint32_t)g.NP, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    if (split) {
        // fp32 packed weights as {Cs, OC, 2, taps}: one box {32, 128, 2, 1}
        // lands as [w_hi | w_lo].
        const cuuint64_t dims[4] = {(cuuint64_t)Cs, (cuuint64_t)p.OC, 2, (cuuint64_t)p.taps};
        const cuuint64_t strides[3] = {(cuuint64_t)Cp * elt, (cuuint64_t)Cs * elt, (cuuint64_t)Cp * elt * p.OC};
        const cuuint32_t box[4] = {(cuuint32_t)blk, (cuuint32_t)kTileOc, 2, 1};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        if (encode(&tmW, dt, 4, const_cast<void *>(wp), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else {
        // Packed weights {Cp, OC, taps}; a box is one K block x 128 outputs.
        const cuuint64_t dims[3] = {(cuuint64_t)Cp, (cuuint64_t)p.OC, (cuuint64_t)p.taps};
        const cuuint64_t strides[2] = {(cuuint64_t)Cp * elt, (cuuint64_t)Cp * elt * p.OC};
        const cuuint32_t box[3] = {(cuuint32_t)blk, (cuuint32_t)kTileOc, 1};
        const cuuint32_t es[3] = {1, 1, 1};
        if (encode(&tmW, dt, 3, const_cast<void *>(wp), dims, strides, box, es,
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
    a.out_vol = p.out_vol;
    a.P = P;
    a.NP = g.NP;
    a.oc_tiles = (p.OC + kTileOc - 1) / kTileOc;
    const int64_t num_tiles = (P + g.NP - 1) / g.NP * a.oc_tiles;
    a.num_tiles = (int)num_tiles;
    a.cs = Cs;
    a.xlo_off = 128u * (uint32_t)g.NP;
    a.cblocks = split ? Cs / blk : (Cp + blk - 1) / blk;
    a.ksteps = p.taps * a.cblocks;
    a.stages = g.stages;
    a.relu = p.act == GBCONV_ACT_RELU;
    a.vec_store = !split && (p.out_vol % 8 == 0) && (((uintptr_t)y % 16) == 0);
    a.cl = p.cl;
    a.pair_store = !split && (p.OC % 2 == 0) && (((uintptr_t)y % 4) == 0);
    {
        // Output views for 32 x 32 TMA tensor stores (rows and base 16-byte
        // aligned; coordinates within int32): NC(D)HW as {out_vol, OC, N}
        // (a chunk's 32 pixels are consecutive in one image's channel
        // plane), channels-last as {OC, P} (32 consecutive pixel rows).
        const int a16 = 16 / (int)elt;
        const bool ok = ((uintptr_t)y % 16 == 0) &&
                        (p.cl ? (p.OC % a16 == 0 && P < 0x7FFFFFFF)
                              : (p.out_vol % a16 == 0 && p.out_vol < 0x7FFFFFFF));
        if (ok) {
            const CUtensorMapSwizzle sw = split ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
            if (p.cl) {
                const cuuint64_t dims[2] = {(cuuint64_t)p.OC, (cuuint64_t)P};
                const cuuint64_t strides[1] = {(cuuint64_t)p.OC * elt};
                const cuuint32_t box[2] = {32, 32};
                const cuuint32_t es[2] = {1, 1};
                a.tma_store = encode(&tmY, dt, 2, y, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
                              CUDA_SUCCESS;
            } else {
                const cuuint64_t dims[3] = {(cuuint64_t)p.out_vol, (cuuint64_t)p.OC, (cuuint64_t)p.N};
                const cuuint64_t strides[2] = {(cuuint64_t)p.out_vol * elt, (cuuint64_t)p.out_vol * p.OC * elt};
                const cuuint32_t box[3] = {32, 32, 1};
                const cuuint32_t es[3] = {1, 1, 1};
                a.tma_store = encode(&tmY, dt, 3, y, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
                              CUDA_SUCCESS;
            }
        }
    }
    a.idesc = split ? make_idesc_tf32(kTileOc, g.NP) : make_idesc(kTileOc, g.NP, p.dtype == GBCONV_BF16);
    // every load is NP pixel rows of 128 B (zero-filled outside the input)
    a.tx_bytes = (split ? 2u : 1u) * (kWStageBytes + 128u * (uint32_t)g.NP);
    a.tmem_cols = tmem_cols_for(2 * g.NP);
    const double cyc = (double)wait_limit_ns() * (double)info.clock_khz * 1e-6;
    a.wait_limit_cycles = cyc > 9.0e18 ? (long long)9e18 : (long long)cyc;

    a.single_tile = g.single_tile ? 1 : 0;
    // Only when x is read in place: behind the layout pass the weights alone
    // measured no faster.
    a.prefetch = tc_cl_direct(p) ? 1 | (p.w_layout == GBCONV_W_PACKED ? 2 : 0) : 0;
    a.in_w = p.W; a.in_h = p.H; a.in_d = p.D;
    const size_t smem = smem_bytes(g, p);
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
    if (log_enabled())
        log_line("igemm_tc_kernel<%s> grid=%d block=%d smem=%zu tiles=%lld pixels_per_tile=%d oc_tiles=%d "
                 "stages=%d ksteps=%d store=%s%s", split ? "tf32x3" : (p.dtype == GBCONV_BF16 ? "bf16" : "f16"),
                 grid, kThreads, smem, (long long)num_tiles, g.NP, a.oc_tiles, g.stages, a.ksteps,
                 a.tma_store ? "tma" : "registers", g.single_tile ? " staging_in_ring" : "");
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), smem, s, tmX, tmW, tmY, a);
}

#include "stem_tf32.cuh"

// fp32 on the tensor cores: x -> xs [N][S][2 Cs] with xs[..][c] = hi(x) and
// xs[..][Cs + c] = lo(x) = x - hi(x) for c < C, zero up to Cs (S = D*H*W).
// From NC(D)HW a CTA moves 32 channels x 256 positions through a padded
// shared tile (loads along positions, stores along channels); from
// channels-last x each thread splits one element in place of the copy.
constexpr int kSpC = 32, kSpS = 256;
template <bool VEC>
__device__ __forceinline__ void split_nchw_block(const float *__restrict__ x, float *__restrict__ xs, int C, int Cs,
                                                 int64_t S, int bx, int by, int bz, float (*tile)[kSpS + 1]) {
    const int64_t s0 = (int64_t)bx * kSpS;
    const int c0 = by * kSpC;
    const int n = bz;
    const float *xn = x + (int64_t)n * C * S;
    // Loads: 4 consecutive positions of one channel per thread (16-byte
    // vectors when S is a multiple of 4 and x 16-byte aligned), all of a
    // thread's loads in flight before any is stored.
    constexpr int kIter = kSpC * kSpS / 4 / 256;
    float4 buf[kIter];
#pragma unroll
    for (int i = 0; i < kIter; ++i) {
        const int e = threadIdx.x + 256 * i;
        const int cl = e / (kSpS / 4), sl = (e % (kSpS / 4)) * 4;
        const int c = c0 + cl;
        const int64_t sp = s0 + sl;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < C) {
            if (VEC && sp + 4 <= S) {
                v = __ldg(reinterpret_cast<const float4 *>(xn + (int64_t)c * S + sp));
            } else {
                if (sp < S) v.x = __ldg(xn + (int64_t)c * S + sp);
                if (sp + 1 < S) v.y = __ldg(xn + (int64_t)c * S + sp + 1);
                if (sp + 2 < S) v.z = __ldg(xn + (int64_t)c * S + sp + 2);
                if (sp + 3 < S) v.w = __ldg(xn + (int64_t)c * S + sp + 3);
            }
        }
        buf[i] = v;
    }
#pragma unroll
    for (int i = 0; i < kIter; ++i) {
        const int e = threadIdx.x + 256 * i;
        const int cl = e / (kSpS / 4), sl = (e % (kSpS / 4)) * 4;
        tile[cl][sl] = buf[i].x;
        tile[cl][sl + 1] = buf[i].y;
        tile[cl][sl + 2] = buf[i].z;
        tile[cl][sl + 3] = buf[i].w;
    }
    __syncthreads();
    // Stores: 4 consecutive channels of one position per thread, hi and lo
    // halves as two 16-byte vectors (Cs is a multiple of 32).
    float *xsn = xs + (int64_t)n * S * 2 * Cs;
#pragma unroll
    for (int i = 0; i < kIter; ++i) {
        const int e = threadIdx.x + 256 * i;
        const int sl = e / (kSpC / 4), cl = (e % (kSpC / 4)) * 4;
        const int64_t sp = s0 + sl;
        if (sp < S) {
            float4 h, l;
            tf32_split(tile[cl][sl], h.x, l.x);
            tf32_split(tile[cl + 1][sl], h.y, l.y);
            tf32_split(tile[cl + 2][sl], h.z, l.z);
            tf32_split(tile[cl + 3][sl], h.w, l.w);
            *reinterpret_cast<float4 *>(xsn + sp * 2 * Cs + c0 + cl) = h;
            *reinterpret_cast<float4 *>(xsn + sp * 2 * Cs + Cs + c0 + cl) = l;
        }
    }
}
// Element i = position * Cs + c of the split of channels-last x.
__device__ __forceinline__ void split_cl_elem(const float *__restrict__ x, float *__restrict__ xs, int C, int Cs,
                                              int64_t positions, int64_t i) {
    if (i >= positions * Cs) return;
    const int64_t sp = i / Cs;
    const int c = (int)(i - sp * Cs);
    float h = 0.0f, l = 0.0f;
    if (c < C) tf32_split(__ldg(x + sp * C + c), h, l);
    xs[sp * 2 * Cs + c] = h;
    xs[sp * 2 * Cs + Cs + c] = l;
}
// Element i = (tap * OC + oc) * Cs + c of w [OC][C][taps] -> wp [tap][OC][2 Cs]:
// the hi half, then the lo half.
__device__ __forceinline__ void pack_split_elem(const float *__restrict__ w, float *__restrict__ wp, int OC, int C,
                                                int Cs, int taps, int64_t i) {
    if (i >= (int64_t)taps * OC * Cs) return;
    const int c = (int)(i % Cs);
    const int64_t r = i / Cs;
    const int oc = (int)(r % OC), tap = (int)(r / OC);
    float h = 0.0f, l = 0.0f;
    if (c < C) tf32_split(__ldg(w + ((int64_t)oc * C + c) * taps + tap), h, l);
    wp[r * 2 * Cs + c] = h;
    wp[r * 2 * Cs + Cs + c] = l;
}
template <bool VEC>
__global__ void __launch_bounds__(256)
split_nchw_kernel(const float *__restrict__ x, float *__restrict__ xs, int C, int Cs, int64_t S) {
    __shared__ float tile[kSpC][kSpS + 1];
    pdl_launch_dependents();   // the GEMM behind launches once every CTA here has started
    pdl_wait();                // global memory only once the previous kernel is complete
    split_nchw_block<VEC>(x, xs, C, Cs, S, blockIdx.x, blockIdx.y, blockIdx.z, tile);
}
__global__ void __launch_bounds__(256)
split_cl_kernel(const float *__restrict__ x, float *__restrict__ xs, int C, int Cs, int64_t positions) {
    pdl_launch_dependents();   // the GEMM behind launches once every CTA here has started
    pdl_wait();                // global memory only once the previous kernel is complete
    split_cl_elem(x, xs, C, Cs, positions, (int64_t)blockIdx.x * blockDim.x + threadIdx.x);
}
__global__ void __launch_bounds__(256)
pack_split_kernel(const float *__restrict__ w, float *__restrict__ wp, int OC, int C, int Cs, int taps) {
    pdl_launch_dependents();   // the GEMM behind launches once every CTA here has started
    pdl_wait();                // global memory only once the previous kernel is complete
    pack_split_elem(w, wp, OC, C, Cs, taps, (int64_t)blockIdx.x * blockDim.x + threadIdx.x);
}
// The split-pack of OIHW weights and the split of x as one grid: npk CTAs
// pack 256 weight elements each, nsp split x (NC(D)HW blocks of a
// spx x spy x N grid, x fastest, or 256 channels-last elements each when
// XM == 0). XM: 0 channels-last x, 1 NC(D)HW, 2 NC(D)HW with 16-byte loads.
template <int XM>
__global__ void __launch_bounds__(256)
prep_split_kernel(const float *__restrict__ x, float *__restrict__ xs, int C, int Cs, int64_t S, int64_t positions,
                  int spx, int spy, const float *__restrict__ w, float *__restrict__ wp, int OC, int taps, int npk,
                  int nsp) {
    __shared__ float tile[kSpC][kSpS + 1];
    pdl_launch_dependents();   // the GEMM behind launches once every CTA here has started
    pdl_wait();                // global memory only once the previous kernel is complete
    bool pack;
    const int q = prep_block_index(blockIdx.x, npk, nsp, &pack);
    if (pack) {
        pack_split_elem(w, wp, OC, C, Cs, taps, (int64_t)q * 256 + threadIdx.x);
    } else {
        if (XM == 0)
            split_cl_elem(x, xs, C, Cs, positions, (int64_t)q * 256 + threadIdx.x);
        else
            split_nchw_block<XM == 2>(x, xs, C, Cs, S, q % spx, (q / spx) % spy, q / (spx * spy), tile);
    }
}

cudaError_t launch_split(const Problem &p, const void *x, void *xs, cudaStream_t s) {
    const int Cs = tc_split_half(p.C);
    const float *xf = static_cast<const float *>(x);
    float *xo = static_cast<float *>(xs);
    if (p.cl) {
        const int64_t n = (int64_t)p.N * p.in_vol * Cs;
        return launch_pdl(split_cl_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, xf, xo, p.C, Cs,
                          (int64_t)p.N * p.in_vol);
    } else {
        dim3 grid((unsigned)((p.in_vol + kSpS - 1) / kSpS), (unsigned)(Cs / kSpC), (unsigned)p.N);
        if (p.in_vol % 4 == 0 && (uintptr_t)xf % 16 == 0)
            return launch_pdl(split_nchw_kernel<true>, grid, dim3(256), 0, s, xf, xo, p.C, Cs, p.in_vol);
        return launch_pdl(split_nchw_kernel<false>, grid, dim3(256), 0, s, xf, xo, p.C, Cs, p.in_vol);
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_cl_typed(const Problem &p, const void *x, void *xc, cudaStream_t s) {
    const int Cp = tc_cpad(p.C);
    const int64_t S = p.in_vol;
    dim3 grid((unsigned)((S + kClS - 1) / kClS), (unsigned)((Cp + kClC - 1) / kClC), (unsigned)p.N);
    const bool vec = (S % 8 == 0) && ((uintptr_t)x % 16 == 0);
    if (vec)
        return launch_pdl(to_channels_last_kernel<T, true>, grid, dim3(256), 0, s, static_cast<const T *>(x),
                          static_cast<T *>(xc), p.C, Cp, S);
    else
        return launch_pdl(to_channels_last_kernel<T, false>, grid, dim3(256), 0, s, static_cast<const T *>(x),
                          static_cast<T *>(xc), p.C, Cp, S);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_pack_tc_typed(const Problem &p, const void *w, void *wp, cudaStream_t s) {
    DevInfo info;
    cudaError_t e = dev_info(&info);
    if (e != cudaSuccess) return e;
    const int Cp = tc_cpad(p.C);
    const long long items = (long long)p.OC * ((Cp + 63) / 64) * ((p.taps + 7) / 8);
    // four CTAs per SM, also when there are fewer items than warps (item q
    // goes to CTA q % grid, so the items spread over all SMs): the CTA beside
    // a resident GEMM CTA is joined by the others once that GEMM has left
    const long long grid = 4ll * info.sms;
    if (log_enabled()) log_line("pack_rt_kernel grid=%lld block=%d items=%lld", grid, kPrThreads, items);
    return launch_pdl(pack_rt_kernel<T>, dim3((unsigned)grid), dim3(kPrThreads), 0, s,
                      static_cast<const unsigned short *>(w), static_cast<unsigned int *>(wp), p.OC, p.C, Cp,
                      p.taps, items);
}

template <typename T>
cudaError_t launch_prep_tc_typed(const Problem &p, const void *w, void *wp, const void *x, void *xc, cudaStream_t s) {
    const int Cp = tc_cpad(p.C);
    const int64_t S = p.in_vol;
    const int64_t clx = (S + kClS - 1) / kClS, cly = (Cp + kClC - 1) / kClC;
    const int ocpb = pack_oc_block(p.taps);
    const int64_t pkx = (p.OC + ocpb - 1) / ocpb, pky = (Cp + kPkC - 1) / kPkC, pkz = (p.taps + kPkT - 1) / kPkT;
    const int64_t npk = pkx * pky * pkz, nlay = clx * cly * p.N;
    const int64_t total = npk + nlay;
    if (total > 0x7FFFFFFF) return cudaErrorNotSupported;   // caller falls back to two launches
    const bool vec = (S % 8 == 0) && ((uintptr_t)x % 16 == 0);
    DevInfo info;
    const cudaError_t e = dev_info(&info);
    if (e != cudaSuccess) return e;
    const bool big = total > 4ll * info.sms;
    auto kern = vec ? (big ? prep_tc_kernel<T, true, 6> : prep_tc_kernel<T, true, 4>)
                    : (big ? prep_tc_kernel<T, false, 6> : prep_tc_kernel<T, false, 4>);
    return launch_pdl(kern, dim3((unsigned)total), dim3(256), 0, s, static_cast<const T *>(x), static_cast<T *>(xc),
                      p.C, Cp, S, (int)clx, (int)cly, static_cast<const T *>(w), static_cast<T *>(wp), p.OC, p.taps,
                      ocpb, (int)pkx, (int)pky, (int)npk, (int)nlay);
}

cudaError_t launch_prep_split(const Problem &p, const void *w, void *wp, const void *x, void *xs, cudaStream_t s) {
    const int Cs = tc_split_half(p.C);
    const int64_t S = p.in_vol, positions = (int64_t)p.N * p.in_vol;
    const int64_t spx = (S + kSpS - 1) / kSpS, spy = Cs / kSpC;
    const int64_t nsp = p.cl ? (positions * Cs + 255) / 256 : spx * spy * p.N;
    const int64_t npk = ((int64_t)p.taps * p.OC * Cs + 255) / 256;
    const int64_t total = npk + nsp;
    if (total > 0x7FFFFFFF) return cudaErrorNotSupported;   // caller falls back to two launches
    const float *xf = static_cast<const float *>(x), *wf = static_cast<const float *>(w);
    float *xo = static_cast<float *>(xs), *wo = static_cast<float *>(wp);
    auto kern = p.cl ? prep_split_kernel<0>
                     : (S % 4 == 0 && (uintptr_t)xf % 16 == 0) ? prep_split_kernel<2> : prep_split_kernel<1>;
    return launch_pdl(kern, dim3((unsigned)total), dim3(256), 0, s, xf, xo, p.C, Cs, S, positions, (int)spx,
                      (int)spy, wf, wo, p.OC, p.taps, (int)npk, (int)nsp);
}

}  // namespace

bool tc_supported(const Problem &p) {
    // The SM count only shapes the tiling, not whether a tile fits.
    const TileGeom g = choose_geom(p, 152);
    if (g.NP == 0 || !im2col_corners(p).ok) return false;
    const int64_t tiles = (out_pixels(p) + g.NP - 1) / g.NP * ((p.OC + kTileOc - 1) / kTileOc);
    return tiles < 0x7FFFFFFF && out_pixels(p) < ((int64_t)1 << 40);
}

cudaError_t launch_igemm_tc(const Problem &p, const void *xc, const void *wp, const float *b,
                            void *y, cudaStream_t s) {
    if (p.dtype == GBCONV_F32) return launch_tc_typed<float>(p, xc, wp, b, y, s);
    if (p.dtype == GBCONV_BF16) return launch_tc_typed<__nv_bfloat16>(p, xc, wp, b, y, s);
    return launch_tc_typed<__half>(p, xc, wp, b, y, s);
}

bool stem_tc_supported(const Problem &p) {
    return p.ndim == 2 && p.dtype == GBCONV_F32 && p.k == 3 && p.C <= kStemMaxC && p.OC <= kStemMaxOC &&
           (int64_t)p.N * p.OH * p.OW <= kStemMaxPixels;
}

cudaError_t launch_stem_tc(const Problem &p, const void *x, const void *w, const float *b, void *y,
                           cudaStream_t s) {
    const float *xf = static_cast<const float *>(x), *wf = static_cast<const float *>(w);
    float *yf = static_cast<float *>(y);
    switch (p.C) {
    case 1: return launch_stem_tf32_c<1>(p, xf, wf, b, yf, s);
    case 2: return launch_stem_tf32_c<2>(p, xf, wf, b, yf, s);
    case 3: return launch_stem_tf32_c<3>(p, xf, wf, b, yf, s);
    default: return launch_stem_tf32_c<4>(p, xf, wf, b, yf, s);
    }
}

cudaError_t launch_to_channels_last(const Problem &p, const void *x, void *xc, cudaStream_t s) {
    if (p.dtype == GBCONV_F32) return launch_split(p, x, xc, s);
    if (p.dtype == GBCONV_BF16) return launch_cl_typed<__nv_bfloat16>(p, x, xc, s);
    return launch_cl_typed<__half>(p, x, xc, s);
}

cudaError_t launch_pack_tc(const Problem &p, const void *w, void *wp, cudaStream_t s) {
    if (p.dtype == GBCONV_F32) {
        const int Cs = tc_split_half(p.C);
        const int64_t n = (int64_t)p.taps * p.OC * Cs;
        return launch_pdl(pack_split_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s,
                          static_cast<const float *>(w), static_cast<float *>(wp), p.OC, p.C, Cs, p.taps);
    }
    if (p.dtype == GBCONV_BF16) return launch_pack_tc_typed<__nv_bfloat16>(p, w, wp, s);
    return launch_pack_tc_typed<__half>(p, w, wp, s);
}

cudaError_t launch_prep_tc(const Problem &p, const void *w, void *wp, const void *x, void *xc, cudaStream_t s) {
    cudaError_t e;
    if (p.dtype == GBCONV_F32) e = launch_prep_split(p, w, wp, x, xc, s);
    else if (p.dtype == GBCONV_BF16) e = launch_prep_tc_typed<__nv_bfloat16>(p, w, wp, x, xc, s);
    else e = launch_prep_tc_typed<__half>(p, w, wp, x, xc, s);
    if (e != cudaErrorNotSupported) return e;
    e = launch_pack_tc(p, w, wp, s);
    return e == cudaSuccess ? launch_to_channels_last(p, x, xc, s) : e;
}


}  // namespace gbconv
