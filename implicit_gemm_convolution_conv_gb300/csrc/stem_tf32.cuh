// fp32 convolution with a short reduction (C * 3 * 3 <= 36 taps: image
// stems) on the tcgen05 tensor cores, in TF32 with split operands.
//
// The operation is the output-stationary sum of lpnh.cn/news/2745477 section
// 2.2 (zero padding, bias, ReLU fused into the write-back as in section 4.4),
// cast as a GEMM per tile of 128 output pixels:
//   y[pixel][oc] = sum_t x[pixel][t] * w[oc][t],   t = (c, ky, kx), T = C * 9.
// Every fp32 value v is split as v = hi + lo: hi is v with its 13 low
// mantissa bits cleared (exactly representable in TF32) and lo = v - hi
// (exact in fp32; the MMA reads its top 19 bits). The splits are laid along
// K and N:
//   A[pixel][k] = [ x_hi | x_lo ]                      K = 2T (padded to 8)
//   B[n][k]     = [ w_hi | w_hi ]  for n <  OCP
//                 [ w_lo | w_lo ]  for n >= OCP        N = 2 * OCP
// so that one chain of K/8 MMAs leaves x.w_hi in TMEM column oc and x.w_lo in
// column OCP + oc; their sum is the fp32 product sum up to a relative error
// near 2^-20 per term (the TF32 reading of lo), far inside the fp32 parity
// tolerance (rel. L2 1e-5). Splitting fp32 products into TF32 pieces is the
// usual way to run fp32 GEMMs on TF32 units; carrying the pieces in K and N
// of one chain keeps the MMA count at K/8 (7 for three channels).
//
// GEMM orientation: M = 128 output pixels, N = 2 * OCP (OCP = OC rounded up
// to 16). A kernel that uses TMEM is resident once per SM, so one persistent
// CTA per SM runs G independent groups of 128 threads (up to 4, as shared
// memory and the 512 TMEM columns allow), each with its own pixel operand,
// accumulator and barriers; the groups overlap one another's loads, MMAs and
// stores. The weight operand is split once per CTA and shared. Thread i of a
// group owns pixel i of the group's tile: it splits its pixel's T taps into
// row i of A, one thread of the group issues the MMAs and commits to an
// mbarrier, and the thread then reads its own TMEM lane (row i of D), adds the
// two halves and the bias and applies ReLU.
//
// Where the pixel operand lives. At N <= 64 an MMA's time is set by the
// shared-memory bytes it reads, about 128 B per cycle: with A in shared memory
// a K-step of 8 reads (128 + N) rows x 32 B. When TMEM has room for every
// group's A next to its accumulator, a thread writes its A row into its own
// TMEM lane (tcgen05.st) and the MMAs read only B from shared memory; A then
// costs no shared-memory write either. Otherwise A is row i of a K-major,
// 128-byte-swizzled shared-memory tile.
//
// Two ways in and out of HBM:
// - TMA (input and output rows 16-byte aligned, stride <= 3): a tile is 2
//   output rows x 64 pixels. Its input halo (C x (s + 3) rows x 4-aligned
//   columns, zero filled outside the image: the padding) comes in as one TMA
//   box two tiles ahead of use, into a ring of two buffers per group; the
//   taps are read from shared memory. The results are staged as [oc][row]
//   [pixel] in the group's staging tile and leave as TMA tensor stores,
//   clipped at the image edges, which drain while the group builds its next
//   tile. (Storing from registers instead, one 128-byte warp store per
//   channel, measured twice as slow for this epilogue.)
// - Plain loads and stores otherwise: a tile is 128 consecutive pixels in
//   (n, oh, ow) order; each thread loads its taps from global memory (the
//   next tile's go out before the wait on the MMAs) and stores its pixel of
//   every channel (a warp writes 128 contiguous bytes per channel).

constexpr int kStemPxM = 128;                // pixels per tile (MMA M, TMEM lanes)
constexpr int kStemPxThreads = 128;          // threads per group
constexpr int kStemMaxOC = 128;              // MMA N = 2 * OCP <= 256
constexpr int kStemMaxC = 4;
constexpr int kStemMaxGroups = 4;
constexpr size_t kStemSmemLimit = 227 * 1024;
constexpr int kStemTileW = 64, kStemTileR = 2;   // TMA tiles: 2 output rows x 64 pixels
constexpr int kStemMaxTmaStride = 3;             // halo box width <= 256 columns
constexpr long long kStemMaxPixels = 1ll << 30;  // N * OH * OW: 32-bit tile and pixel indices

struct StemTcArgs {
    const float *x, *w, *b;
    float *y;
    int H, W, OC, OH, OW, pad, stride;
    int ocp;                   // OC rounded up to 16
    int ohw;                   // OH * OW
    int npix;                  // N * OH * OW
    int tiles;
    int tiles_w, tiles_h;      // TMA tiling: 64-pixel column blocks, row pairs
    int hd;                    // TMA: halo column of input column ow0 * s - pad (0..3)
    int hbw, hbh;              // TMA: halo box width (multiple of 4) and height
    uint32_t halo_box_bytes;   // TMA: C * hbh * hbw * 4
    uint32_t halo_bytes;       // one halo buffer, 128-byte aligned
    uint32_t region_bytes;     // per group: shared-memory pixel operand (A in shared memory) and,
                               // with TMA, the output staging tile
    uint32_t stage_off;        // TMA: the staging tile's offset within the region
    int ybox_c;                // TMA: channels per output box
    uint32_t idesc;
    uint32_t tmem_cols;        // all groups (a power of two)
    uint32_t group_cols;       // per group: accumulator, then (A in TMEM) the pixel operand
    uint32_t a_col;            // A in TMEM: its first column within the group's share
    int groups;                // 128-thread groups per CTA (1 to 4)
    int relu;
    long long wait_limit_cycles;
};

template <int C>
struct StemShape {
    static constexpr int T = C * 9;                   // taps
    static constexpr int KP = (2 * T + 7) / 8 * 8;    // K: hi and lo taps, MMA steps of 8
    static constexpr int KCH = (KP + 31) / 32;        // 128-byte chunks per operand row
};

__device__ __forceinline__ void tf32_split(float v, float &hi, float &lo) {
    hi = __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
    lo = v - hi;
}

// Row r of a K-major operand in the 128-byte swizzle layout: 16-byte unit u
// lies in chunk u / 8 (chunks `chunk_bytes` apart) at r * 128 + ((u % 8) ^
// (r % 8)) * 16.
template <int KP>
__device__ __forceinline__ void store_operand_row(uint32_t tile, uint32_t chunk_bytes, int r,
                                                  const float (&v)[KP]) {
#pragma unroll
    for (int u = 0; u < KP / 4; ++u) {
        const uint32_t off = (uint32_t)(u / 8) * chunk_bytes + (uint32_t)r * 128u +
                             (uint32_t)(((u & 7) ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(tile + off), "f"(v[4 * u]),
                     "f"(v[4 * u + 1]), "f"(v[4 * u + 2]), "f"(v[4 * u + 3])
                     : "memory");
    }
}

// 8 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float *v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                 "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// tcgen05.mma, kind::tf32, A read from TMEM (lane = row, K along columns).
__device__ __forceinline__ void tc_mma_tf32_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// This thread's row of the pixel operand from its pixel's taps: [hi | lo | 0
// pad], into its TMEM lane (ATM) or into row `row` of the shared-memory tile.
// The writes are complete (TMEM) or visible to the tensor core (shared
// memory) on return.
template <int C, bool ATM>
__device__ __forceinline__ void put_pixel_row(uint32_t sA, uint32_t tA_lane, int row, const float (&xv)[C * 9]) {
    using S = StemShape<C>;
    float v[S::KP];
#pragma unroll
    for (int t = 0; t < S::T; ++t) tf32_split(xv[t], v[t], v[S::T + t]);
#pragma unroll
    for (int t = 2 * S::T; t < S::KP; ++t) v[t] = 0.0f;
    if (ATM) {
#pragma unroll
        for (int s = 0; s < S::KP / 8; ++s) tmem_st8(tA_lane + 8u * s, v + 8 * s);
        tmem_st_wait();
    } else {
        store_operand_row<S::KP>(sA, 16384u, row, v);
        fence_proxy_async_shared();
    }
}

// The K/8 MMAs of one tile (one thread).
template <int KP, bool ATM>
__device__ __forceinline__ void stem_mmas(uint32_t tacc, uint32_t tA, uint32_t sA, uint32_t sB, uint32_t bchunk,
                                          uint32_t idesc) {
#pragma unroll
    for (int s = 0; s < KP / 8; ++s) {
        // K-step of 8 tf32: 8 TMEM columns, or 32 bytes = descriptor start address + 2.
        const uint64_t bd = sw128_kmajor_desc(sB + (uint32_t)(s / 4) * bchunk) + 2u * (s % 4);
        if (ATM) {
            tc_mma_tf32_ta(tacc, tA + 8u * s, bd, idesc, s > 0);
        } else {
            const uint64_t ad = sw128_kmajor_desc(sA + (uint32_t)(s / 4) * 16384u) + 2u * (s % 4);
            tc_mma_tf32(tacc, ad, bd, idesc, s > 0);
        }
    }
}

// Bounded wait by lane 0 of each warp, result shared with the warp. An
// expired wait raises the CTA's abort flag and sets the device error word;
// once the flag is up every later wait returns at once. The groups keep
// their control flow after an abort (their named barriers stay matched) but
// issue no further copy, MMA or store, so the drain at the end has at most
// one commit and one copy per halo buffer to wait for.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, long long limit, volatile int *abort_flag) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) {
        ok = wait_bounded(bar, parity, limit, abort_flag);
        if (!ok) raise_abort(abort_flag);
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// The pixel's T taps in (c, ky, kx) order from global memory, zero outside
// the input; pixel f of the (n, oh, ow) order, invalid past the last one.
template <int C>
__device__ __forceinline__ void stem_gather(const StemTcArgs &a, int f, float (&v)[C * 9]) {
    const bool valid = f < a.npix;
    const int n = valid ? f / a.ohw : 0;
    const int rem = valid ? f - n * a.ohw : 0;
    const int oh = rem / a.OW, ow = rem - oh * a.OW;
    const long long HW = (long long)a.H * a.W;
    const float *xn = a.x + (long long)n * C * HW;
    const int iy0 = oh * a.stride - a.pad, ix0 = ow * a.stride - a.pad;
#pragma unroll
    for (int c = 0; c < C; ++c)
#pragma unroll
        for (int ky = 0; ky < 3; ++ky) {
            const int iy = iy0 + ky;
            const bool row_ok = valid && (unsigned)iy < (unsigned)a.H;
            const float *xr = xn + c * HW + (long long)iy * a.W;
#pragma unroll
            for (int kx = 0; kx < 3; ++kx) {
                const int ix = ix0 + kx;
                v[(c * 3 + ky) * 3 + kx] = (row_ok && (unsigned)ix < (unsigned)a.W) ? __ldg(xr + ix) : 0.0f;
            }
        }
}

// TMA tile t: image, first output row, first output column.
struct StemTile {
    int n, oh0, ow0;
};
__device__ __forceinline__ StemTile stem_tile(const StemTcArgs &a, int t) {
    StemTile s;
    const int r = t / a.tiles_w;
    s.ow0 = (t - r * a.tiles_w) * kStemTileW;
    s.n = r / a.tiles_h;
    s.oh0 = (r - s.n * a.tiles_h) * kStemTileR;
    return s;
}
// The input halo of TMA tile t as one box: columns from ow0 * s - pad - hd
// (a multiple of 4), rows from oh0 * s - pad, all C channels of image n.
__device__ __forceinline__ void stem_load_halo(const CUtensorMap *tmX, const StemTcArgs &a, int t,
                                               uint32_t dst, uint32_t bar) {
    const StemTile s = stem_tile(a, t);
    mbar_arrive_expect_tx(bar, a.halo_box_bytes);
    tma_load_4d(dst, tmX, bar, s.ow0 * a.stride - a.pad - a.hd, s.oh0 * a.stride - a.pad, 0, s.n);
}

// The same box as an L2 prefetch, its start clamped to the image (a hint
// needs no zero fill; column 0 keeps the 16-byte alignment).
__device__ __forceinline__ void stem_prefetch_halo(const CUtensorMap *tmX, const StemTcArgs &a, int t) {
    const StemTile s = stem_tile(a, t);
    const int x0 = s.ow0 * a.stride - a.pad - a.hd, y0 = s.oh0 * a.stride - a.pad;
    tma_prefetch_l2_4d(tmX, x0 > 0 ? x0 : 0, y0 > 0 ? y0 : 0, 0, s.n);
}

// Bias, the two halves of the accumulator, ReLU; one store per output
// channel of this thread's pixel (y_px: its address in channel 0; the
// channel stride is OH * OW).
__device__ __forceinline__ void stem_epilogue(const StemTcArgs &a, uint32_t tlane, const float *sBias, float *y_px,
                                              bool valid) {
#pragma unroll 1
    for (int c0 = 0; c0 < a.ocp; c0 += 16) {
        uint32_t hv[16], lv[16];
        tmem_ld16(tlane + (uint32_t)c0, hv);
        tmem_ld16(tlane + (uint32_t)(a.ocp + c0), lv);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int oc = c0 + e;
                if (oc < a.OC)
                    y_px[(long long)oc * a.ohw] =
                        epilogue(__uint_as_float(hv[e]) + __uint_as_float(lv[e]), sBias[oc], a.relu);
            }
        }
    }
}

// This thread's T taps, pixel (r, j) of a TMA tile, from a halo buffer
// (shared memory, byte offset hoff from the dynamic shared-memory base).
template <int C>
__device__ __forceinline__ void stem_halo_taps(const StemTcArgs &a, const uint8_t *smem_raw, uint32_t hoff, int r,
                                               int j, bool pair_taps, float (&xv)[C * 9]) {
    const float *h = reinterpret_cast<const float *>(smem_raw + hoff);
    const int s = a.stride;
    if (pair_taps) {
        // Stride 2, odd hd: taps 1 and 2 of a row sit at an even column, so
        // one 8-byte load fetches both.
#pragma unroll
        for (int c = 0; c < C; ++c)
#pragma unroll
            for (int ky = 0; ky < 3; ++ky) {
                const float *hr = h + (c * a.hbh + r * 2 + ky) * a.hbw + j * 2 + a.hd;
                const float2 t12 = *reinterpret_cast<const float2 *>(hr + 1);
                xv[(c * 3 + ky) * 3] = hr[0];
                xv[(c * 3 + ky) * 3 + 1] = t12.x;
                xv[(c * 3 + ky) * 3 + 2] = t12.y;
            }
    } else {
#pragma unroll
        for (int c = 0; c < C; ++c)
#pragma unroll
            for (int ky = 0; ky < 3; ++ky) {
                const float *hr = h + (c * a.hbh + r * s + ky) * a.hbw + j * s + a.hd;
#pragma unroll
                for (int kx = 0; kx < 3; ++kx) xv[(c * 3 + ky) * 3 + kx] = hr[kx];
            }
    }
}

// Overlapped tile loop (TMA tiles, pixel operand in TMEM, OCP <= 32): the
// accumulator row fits in registers.
constexpr int kStemOvlMaxOcp = 32;

template <int C, bool TMA, bool ATM, bool OVL>
__global__ void __launch_bounds__(kStemPxThreads * kStemMaxGroups, 1)
stem_tf32_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                 const StemTcArgs a) {
    using S = StemShape<C>;
    constexpr int T = S::T, KP = S::KP, KCH = S::KCH;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int G = a.groups;
    const int nrows = 2 * a.ocp;                            // B rows = MMA N
    const uint32_t bchunk = (uint32_t)nrows * 128u;
    // Weight operand (KCH chunks of nrows x 128 B); per group its region
    // (shared-memory pixel operand, KCH chunks of 128 rows x 128 B, unless A
    // is in TMEM; with TMA the output staging tile, which shares the operand's
    // space when A is in shared memory); with TMA two halo buffers per group;
    // per group an MMA barrier and two halo barriers; the TMEM address; the
    // bias.
    const uint32_t sB = base;
    const uint32_t sR0 = sB + (uint32_t)KCH * bchunk;
    const uint32_t sH0 = sR0 + (uint32_t)G * a.region_bytes;
    const uint32_t sBar0 = (sH0 + (TMA ? 2u * (uint32_t)G * a.halo_bytes : 0u) + 7u) & ~7u;
    const uint32_t slot_addr = sBar0 + 24u * (uint32_t)G;
    float *sBias = reinterpret_cast<float *>(smem_raw + (((slot_addr + 4u + 15u) & ~15u) - raw));   // 16-byte aligned
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem_raw + (slot_addr - raw));
    // The abort flag sits in the 4 bytes after the TMEM address (sBias starts
    // at least 8 bytes after it).
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem_raw + (slot_addr + 4u - raw));

    const int tid = threadIdx.x;
    const int g = tid / kStemPxThreads, gtid = tid % kStemPxThreads;   // group, pixel row in the tile
    const int q = gtid / 32;                                // TMEM lane quadrant (warp id % 4)
    const uint32_t sA = sR0 + (uint32_t)g * a.region_bytes;
    const uint32_t barM = sBar0 + 24u * (uint32_t)g, barH = barM + 8u;   // halo barriers barH, barH + 8
    const uint32_t sHalo = sH0 + 2u * (uint32_t)g * a.halo_bytes;
    // The CTA's tiles are a contiguous range (5 or 6 of the 800 tiles of a
    // 640 x 640 stride-2 stem on 152 SMs), dealt round-robin to its groups.
    const int tend = (int)((long long)(blockIdx.x + 1) * a.tiles / gridDim.x);
    const int tstep = G;
    int tile = (int)((long long)blockIdx.x * a.tiles / gridDim.x) + g;
    const bool active = tile < tend;

    pdl_launch_dependents();
    // Kept by the group's thread 0: per halo buffer, 1 + the barrier phase
    // parity of a TMA load issued and not yet seen complete (0: none); and
    // the same for the group's last MMA commit. A copy or commit is issued
    // only after the previous one on its barrier was seen complete, so the
    // pending one is always its barrier's current phase.
    uint32_t halo_pending[2] = {0, 0};
    uint32_t mma_pending = 0;
    float xv[T];
    if (tid == 0) *abort_flag = 0;
    if (gtid == 0) {
        mbar_init(barM, 1);
        if (TMA) {
            mbar_init(barH, 1);
            mbar_init(barH + 8u, 1);
        }
        fence_mbar_init();
        if (TMA) {
            prefetch_tmap(&tmX);
            prefetch_tmap(&tmY);
            // The group's first two halos start towards L2 while the previous
            // kernel finishes; the loads after the wait below read them there.
            for (int k = 0; k < 2; ++k)
                if (tile + k * tstep < tend) stem_prefetch_halo(&tmX, a, tile + k * tstep);
        }
    }
    if (tid < 32) {
        tmem_alloc(slot_addr, a.tmem_cols);
        tmem_relinquish();
    }
    // Global memory from here on; the group's first loads go out before the
    // weight operand is built.
    pdl_wait();
    if (TMA && gtid == 0) {
        for (int k = 0; k < 2; ++k)
            if (tile + k * tstep < tend) {
                stem_load_halo(&tmX, a, tile + k * tstep, sHalo + (uint32_t)k * a.halo_bytes, barH + 8u * k);
                halo_pending[k] = 1u;
            }
    }
    if (!TMA && active) stem_gather<C>(a, tile * kStemPxM + gtid, xv);
    for (int o = tid; o < a.ocp; o += blockDim.x) sBias[o] = (a.b && o < a.OC) ? __ldg(a.b + o) : 0.0f;
    // Weight operand, element (r, kk) per thread in batches of 8 (all loads
    // of a batch in flight together): row r < OCP holds w_hi of channel r,
    // row OCP + oc holds w_lo of channel oc, both repeated for the x_hi and
    // x_lo halves of K; zero past 2T and for channels >= OC.
    constexpr int kWBatch = 8;
    for (int e0 = 0; e0 < nrows * KP; e0 += kWBatch * (int)blockDim.x) {
        float wv[kWBatch];
#pragma unroll
        for (int i = 0; i < kWBatch; ++i) {
            const int e = e0 + i * (int)blockDim.x + tid;
            const int r = e / KP, kk = e - r * KP;
            const int oc = r >= a.ocp ? r - a.ocp : r;
            const int t = kk < T ? kk : kk - T;
            wv[i] = (e < nrows * KP && kk < 2 * T && oc < a.OC) ? __ldg(a.w + oc * T + t) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < kWBatch; ++i) {
            const int e = e0 + i * (int)blockDim.x + tid;
            if (e >= nrows * KP) break;
            const int r = e / KP, kk = e - r * KP;
            float h, l;
            tf32_split(wv[i], h, l);
            const uint32_t off = (uint32_t)(kk / 32) * bchunk + (uint32_t)r * 128u +
                                 (uint32_t)((((kk & 31) >> 2) ^ (r & 7)) << 4) + (uint32_t)(kk & 3) * 4u;
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(sB + off), "f"(r >= a.ocp ? l : h) : "memory");
        }
    }
    fence_proxy_async_shared();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // This group's accumulator (its share of the columns) and, with A in
    // TMEM, its pixel operand; the lanes of quadrant q belong to this warp.
    const uint32_t tacc = *tmem_slot + (uint32_t)g * a.group_cols;
    const uint32_t tA = tacc + a.a_col;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;

    uint32_t mphase = 0;
    if constexpr (TMA && ATM && OVL) {
        // A group reads tile k's accumulator into registers, builds tile
        // k+1's operand and issues its MMAs, and only then stages and stores
        // tile k: the next tile's MMAs run under this tile's epilogue.
        const int r = gtid / kStemTileW, j = gtid % kStemTileW;    // this thread's pixel in the tile
        const bool pair_taps = a.stride == 2 && (a.hd & 1) && (a.hbw % 2 == 0);
        const uint32_t stage = sA + a.stage_off;
        const uint32_t stg = stage + (uint32_t)((r * kStemTileW + j) * 4);
        // The operand of this group's tile number kk, from halo buffer kk & 1.
        auto build = [&](int kk) {
            const int hb = kk & 1;
            const uint32_t hpar = (uint32_t)((kk >> 1) & 1);
            const bool landed = warp_wait(barH + 8u * hb, hpar, a.wait_limit_cycles, abort_flag);
            if (gtid == 0 && landed && halo_pending[hb] == 1u + hpar) halo_pending[hb] = 0;
            stem_halo_taps<C>(a, smem_raw, sHalo + (uint32_t)hb * a.halo_bytes - raw, r, j, pair_taps, xv);
            put_pixel_row<C, true>(sA, tA + lane_off, gtid, xv);
        };
        // After the group barrier that follows build(kk): the halo two tiles
        // ahead into the buffer just read, then tile t's MMAs (nothing new
        // once a wait has run out).
        auto issue = [&](int kk, int t) {
            if (gtid == 0 && !*abort_flag) {
                const int hb = kk & 1;
                const int ahead = t + 2 * tstep;
                if (ahead < tend) {
                    stem_load_halo(&tmX, a, ahead, sHalo + (uint32_t)hb * a.halo_bytes, barH + 8u * hb);
                    halo_pending[hb] = 1u + (uint32_t)(((kk + 2) >> 1) & 1);
                }
                stem_mmas<KP, true>(tacc, tA, sA, sB, bchunk, a.idesc);
                tc_commit(barM);
                mma_pending = 1u + mphase;
            }
        };
        if (active) {
            build(0);
            tc_fence_before();
            named_barrier(1 + g, kStemPxThreads);          // operand written, halo buffer 0 read
            tc_fence_after();
            issue(0, tile);
        }
        for (int k = 0; active; ++k) {
            const int next = tile + tstep;
            const bool has_next = next < tend;
            if (warp_wait(barM, mphase, a.wait_limit_cycles, abort_flag) && gtid == 0 && mma_pending == 1u + mphase)
                mma_pending = 0;
            mphase ^= 1u;
            tc_fence_after();
            float v[kStemOvlMaxOcp];
#pragma unroll
            for (int c0 = 0; c0 < kStemOvlMaxOcp; c0 += 16) {
                if (c0 < a.ocp) {
                    uint32_t hv[16], lv[16];
                    tmem_ld16(tacc + lane_off + (uint32_t)c0, hv);
                    tmem_ld16(tacc + lane_off + (uint32_t)(a.ocp + c0), lv);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        v[c0 + e] = epilogue(__uint_as_float(hv[e]) + __uint_as_float(lv[e]), sBias[c0 + e], a.relu);
                }
            }
            // Tile k's MMAs are done and its accumulator is in registers: the
            // operand and the accumulator are free for tile k+1.
            if (has_next) build(k + 1);
            // The previous tile's output stores have read the staging tile.
            if (gtid == 0) bulk_wait_read<0>();
            tc_fence_before();
            named_barrier(1 + g, kStemPxThreads);          // accumulator read, operand written, staging free
            tc_fence_after();
            if (has_next) issue(k + 1, next);
            // Tile k's outputs: staging tile [oc][row][pixel], then TMA stores.
#pragma unroll
            for (int oc = 0; oc < kStemOvlMaxOcp; ++oc)
                if (oc < a.ocp)
                    asm volatile("st.shared.f32 [%0], %1;" ::"r"(stg + (uint32_t)(oc * kStemTileR * kStemTileW * 4)),
                                 "f"(v[oc])
                                 : "memory");
            fence_proxy_async_shared();
            named_barrier(1 + g, kStemPxThreads);
            if (gtid == 0 && !*abort_flag) {
                const StemTile st = stem_tile(a, tile);
                const uint32_t box_bytes = (uint32_t)(a.ybox_c * kStemTileR * kStemTileW * 4);
                for (int c0 = 0, bi = 0; c0 < a.OC; c0 += a.ybox_c, ++bi)
                    tma_store_4d(&tmY, stage + (uint32_t)bi * box_bytes, st.ow0, st.oh0, c0, st.n);
                bulk_commit_group();
            }
            if (!has_next) break;
            tile = next;
        }
        if (gtid == 0) {
            bulk_wait_read_all();
            // After an abort a halo load may still be in flight: wait for it
            // to land (it is the current phase of its buffer's barrier).
            for (int k = 0; k < 2; ++k)
                if (halo_pending[k]) wait_bounded(barH + 8u * k, halo_pending[k] - 1u, kDrainLimitCycles, nullptr);
        }
    } else if (TMA) {
        const int r = gtid / kStemTileW, j = gtid % kStemTileW;    // this thread's pixel in the tile
        const int s = a.stride;
        const bool pair_taps = s == 2 && (a.hd & 1) && (a.hbw % 2 == 0);
        for (int k = 0; active; ++k) {
            const int hb = k & 1;
            const uint32_t hbuf = sHalo + (uint32_t)hb * a.halo_bytes;
            const uint32_t hpar = (uint32_t)((k >> 1) & 1);
            const bool landed = warp_wait(barH + 8u * hb, hpar, a.wait_limit_cycles, abort_flag);
            // (after an abort no load follows, and a wait for the other
            // parity may return at once without the pending load landing)
            if (gtid == 0 && landed && halo_pending[hb] == 1u + hpar) halo_pending[hb] = 0;
            {
                const float *h = reinterpret_cast<const float *>(smem_raw + (hbuf - raw));
                if (pair_taps) {
                    // Stride 2, odd hd: taps 1 and 2 of a row sit at an even
                    // column, so one 8-byte load fetches both.
#pragma unroll
                    for (int c = 0; c < C; ++c)
#pragma unroll
                        for (int ky = 0; ky < 3; ++ky) {
                            const float *hr = h + (c * a.hbh + r * 2 + ky) * a.hbw + j * 2 + a.hd;
                            const float2 t12 = *reinterpret_cast<const float2 *>(hr + 1);
                            xv[(c * 3 + ky) * 3] = hr[0];
                            xv[(c * 3 + ky) * 3 + 1] = t12.x;
                            xv[(c * 3 + ky) * 3 + 2] = t12.y;
                        }
                } else {
#pragma unroll
                    for (int c = 0; c < C; ++c)
#pragma unroll
                        for (int ky = 0; ky < 3; ++ky) {
                            const float *hr = h + (c * a.hbh + r * s + ky) * a.hbw + j * s + a.hd;
#pragma unroll
                            for (int kx = 0; kx < 3; ++kx) xv[(c * 3 + ky) * 3 + kx] = hr[kx];
                        }
                }
            }
            // The previous tile's output stores have read the staging tile
            // (which is the operand's space when A is in shared memory).
            if (!ATM && gtid == 0) bulk_wait_read<0>();
            if (!ATM) named_barrier(1 + g, kStemPxThreads);
            // The previous tile's MMAs, which read the operand, completed
            // before every thread of the group left its wait below.
            put_pixel_row<C, ATM>(sA, tA + lane_off, gtid, xv);
            if (ATM && gtid == 0) bulk_wait_read<0>();
            tc_fence_before();
            named_barrier(1 + g, kStemPxThreads);          // operand written, halo buffer hb read
            tc_fence_after();
            if (gtid == 0 && !*abort_flag) {
                const int ahead = tile + 2 * tstep;
                if (ahead < tend) {
                    stem_load_halo(&tmX, a, ahead, hbuf, barH + 8u * hb);
                    halo_pending[hb] = 1u + (uint32_t)(((k + 2) >> 1) & 1);
                }
                stem_mmas<KP, ATM>(tacc, tA, sA, sB, bchunk, a.idesc);
                tc_commit(barM);
                mma_pending = 1u + mphase;
            }
            if (warp_wait(barM, mphase, a.wait_limit_cycles, abort_flag) && gtid == 0 && mma_pending == 1u + mphase)
                mma_pending = 0;
            mphase ^= 1u;
            tc_fence_after();
            // Staging tile [oc][row][pixel].
            const uint32_t stage = sA + a.stage_off;
            const uint32_t stg = stage + (uint32_t)((r * kStemTileW + j) * 4);
#pragma unroll 1
            for (int c0 = 0; c0 < a.ocp; c0 += 16) {
                uint32_t hv[16], lv[16];
                tmem_ld16(tacc + lane_off + (uint32_t)c0, hv);
                tmem_ld16(tacc + lane_off + (uint32_t)(a.ocp + c0), lv);
                tmem_ld_wait();
                float bias[16];
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4)
                    *reinterpret_cast<float4 *>(&bias[4 * e4]) = reinterpret_cast<const float4 *>(sBias + c0)[e4];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int oc = c0 + e;
                    const float v = epilogue(__uint_as_float(hv[e]) + __uint_as_float(lv[e]), bias[e], a.relu);
                    asm volatile("st.shared.f32 [%0], %1;" ::"r"(stg + (uint32_t)(oc * kStemTileR * kStemTileW * 4)),
                                 "f"(v)
                                 : "memory");
                }
            }
            fence_proxy_async_shared();
            // TMEM reads complete before the group barrier that precedes the next MMAs.
            tc_fence_before();
            named_barrier(1 + g, kStemPxThreads);
            if (gtid == 0 && !*abort_flag) {
                const StemTile st = stem_tile(a, tile);
                const uint32_t box_bytes = (uint32_t)(a.ybox_c * kStemTileR * kStemTileW * 4);
                for (int c0 = 0, bi = 0; c0 < a.OC; c0 += a.ybox_c, ++bi)
                    tma_store_4d(&tmY, stage + (uint32_t)bi * box_bytes, st.ow0, st.oh0, c0, st.n);
                bulk_commit_group();
            }
            tile += tstep;
            if (tile >= tend) break;
        }
        if (gtid == 0) {
            // The stores must have read the staging tile before the CTA's
            // shared memory goes away; their global writes complete with the grid.
            bulk_wait_read_all();
            // After an abort a halo load may still be in flight: wait for it
            // to land (it is the current phase of its buffer's barrier).
            for (int k = 0; k < 2; ++k)
                if (halo_pending[k]) wait_bounded(barH + 8u * k, halo_pending[k] - 1u, kDrainLimitCycles, nullptr);
        }
    } else {
        while (active) {
            put_pixel_row<C, ATM>(sA, tA + lane_off, gtid, xv);
            tc_fence_before();
            named_barrier(1 + g, kStemPxThreads);
            tc_fence_after();
            if (gtid == 0 && !*abort_flag) {
                stem_mmas<KP, ATM>(tacc, tA, sA, sB, bchunk, a.idesc);
                tc_commit(barM);
                mma_pending = 1u + mphase;
            }
            const int f = tile * kStemPxM + gtid;
            const bool valid = f < a.npix;
            const int n = valid ? f / a.ohw : 0;
            float *y_px = a.y + (long long)n * a.OC * a.ohw + (valid ? f - n * a.ohw : 0);
            const int next = tile + tstep;
            if (next < tend) stem_gather<C>(a, next * kStemPxM + gtid, xv);   // in flight during the wait
            if (warp_wait(barM, mphase, a.wait_limit_cycles, abort_flag) && gtid == 0 && mma_pending == 1u + mphase)
                mma_pending = 0;
            mphase ^= 1u;
            tc_fence_after();
            stem_epilogue(a, tacc + lane_off, sBias, y_px, valid);
            tc_fence_before();
            if (next >= tend) break;
            tile = next;
        }
    }
    // After an abort the group's last commit may still be in flight: its
    // MMAs land before the TMEM is released.
    if (gtid == 0 && mma_pending) wait_bounded(barM, mma_pending - 1u, kDrainLimitCycles, nullptr);
    tc_fence_before();
    __syncthreads();
    if (tid < 32) {
        tc_fence_after();
        tmem_dealloc(*tmem_slot, a.tmem_cols);
    }
}

inline size_t stem_tc_smem_bytes(const StemTcArgs &a, int C, bool tma, int groups) {
    const int KP = (2 * C * 9 + 7) / 8 * 8, KCH = (KP + 31) / 32;
    return 1024 + (size_t)KCH * 2 * a.ocp * 128 + (size_t)groups * a.region_bytes +
           (tma ? 2 * (size_t)groups * a.halo_bytes : 0) + 8 + 24 * (size_t)groups + 32 + 4 * (size_t)a.ocp;
}

inline uint32_t round32(int v) { return (uint32_t)(v + 31) / 32u * 32u; }

template <int C>
cudaError_t launch_stem_tf32_c(const Problem &p, const float *x, const float *w, const float *b, float *y,
                               cudaStream_t s) {
    DevInfo info;
    cudaError_t e = dev_info(&info);
    if (e != cudaSuccess) return e;
    using S = StemShape<C>;
    StemTcArgs a{};
    a.x = x; a.w = w; a.b = b; a.y = y;
    a.H = p.H; a.W = p.W; a.OC = p.OC; a.OH = p.OH; a.OW = p.OW; a.pad = p.pad; a.stride = p.stride;
    a.ocp = (p.OC + 15) / 16 * 16;
    a.ohw = p.OH * p.OW;
    a.npix = p.N * a.ohw;
    a.idesc = make_idesc_tf32(kStemPxM, 2 * a.ocp);
    a.relu = p.act == GBCONV_ACT_RELU;
    const double cyc = (double)wait_limit_ns() * (double)info.clock_khz * 1e-6;
    a.wait_limit_cycles = cyc > 9.0e18 ? (long long)9e18 : (long long)cyc;
    const uint32_t operand_bytes = (uint32_t)S::KCH * 16384u;

    // TMA input and output: rows and bases 16-byte aligned, halo box within 256 columns.
    alignas(64) CUtensorMap tmX, tmY;
    std::memset(&tmX, 0, sizeof(tmX));
    std::memset(&tmY, 0, sizeof(tmY));
    bool tma = p.W % 4 == 0 && p.OW % 4 == 0 && (uintptr_t)x % 16 == 0 && (uintptr_t)y % 16 == 0 &&
               p.stride <= kStemMaxTmaStride;
    uint32_t stage_bytes = 0;
    if (tma) {
        a.hd = ((-p.pad) % 4 + 4) % 4;
        a.hbw = (a.hd + (kStemTileW - 1) * p.stride + 3 + 3) / 4 * 4;   // >= hd + 63 s + 3, a multiple of 4
        a.hbh = (kStemTileR - 1) * p.stride + 3;
        a.halo_box_bytes = (uint32_t)(C * a.hbh * a.hbw * 4);
        a.halo_bytes = (a.halo_box_bytes + 127u) & ~127u;
        a.tiles_w = (p.OW + kStemTileW - 1) / kStemTileW;
        a.tiles_h = (p.OH + kStemTileR - 1) / kStemTileR;
        a.tiles = p.N * a.tiles_h * a.tiles_w;
        a.ybox_c = a.ocp < 32 ? a.ocp : 32;
        // Output boxes cover roundup(OCP, ybox_c) staged channels.
        const int staged_c = (a.ocp + a.ybox_c - 1) / a.ybox_c * a.ybox_c;
        stage_bytes = (uint32_t)(staged_c * kStemTileR * kStemTileW * 4);
        PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
        const cuuint32_t es[4] = {1, 1, 1, 1};
        // x as {W, H, C, N}; a box is the halo of one tile.
        const cuuint64_t xd[4] = {(cuuint64_t)p.W, (cuuint64_t)p.H, (cuuint64_t)C, (cuuint64_t)p.N};
        const cuuint64_t xr = (cuuint64_t)p.W * 4;
        const cuuint64_t xs[3] = {xr, xr * p.H, xr * p.H * C};
        const cuuint32_t xb[4] = {(cuuint32_t)a.hbw, (cuuint32_t)a.hbh, (cuuint32_t)C, 1};
        // y as {OW, OH, OC, N}; a box is 64 pixels x 2 rows x ybox_c channels.
        const cuuint64_t yd[4] = {(cuuint64_t)p.OW, (cuuint64_t)p.OH, (cuuint64_t)p.OC, (cuuint64_t)p.N};
        const cuuint64_t yr = (cuuint64_t)p.OW * 4;
        const cuuint64_t ys[3] = {yr, yr * p.OH, yr * p.OH * p.OC};
        const cuuint32_t yb[4] = {(cuuint32_t)kStemTileW, (cuuint32_t)kStemTileR, (cuuint32_t)a.ybox_c, 1};
        tma = encode &&
              encode(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(x), xd, xs, xb, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
              encode(&tmY, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, y, yd, ys, yb, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    if (!tma) {
        a.halo_box_bytes = a.halo_bytes = 0;
        stage_bytes = 0;
        a.tiles = (a.npix + kStemPxM - 1) / kStemPxM;
    }
    // Per-group region: A in shared memory (operand_bytes, reused as the
    // staging tile once the MMAs are done) or A in TMEM (staging tile only).
    auto region_for = [&](bool atm) {
        return atm ? (stage_bytes + 1023u) & ~1023u : (operand_bytes > stage_bytes ? operand_bytes : stage_bytes);
    };

    // Groups per CTA: as many (up to 4) as shared memory and the SM's 512
    // TMEM columns allow, for A in shared memory and for A in TMEM; A goes to
    // TMEM when that keeps at least as many groups.
    const uint32_t acc_cols = round32(2 * a.ocp);
    auto groups_for = [&](bool atm) {
        StemTcArgs t = a;
        t.region_bytes = region_for(atm);
        const uint32_t gc = atm ? acc_cols + round32(S::KP) : acc_cols;
        int G = kStemMaxGroups;
        while (G > 0 && (stem_tc_smem_bytes(t, C, tma, G) > kStemSmemLimit || (uint32_t)G * gc > 512u)) --G;
        return G;
    };
    const int g_smem = groups_for(false), g_tmem = groups_for(true);
    const bool atm = g_tmem >= g_smem && g_tmem > 0;
    const int G = atm ? g_tmem : g_smem;
    if (G < 1) return cudaErrorInvalidValue;
    a.region_bytes = region_for(atm);
    a.stage_off = 0;
    a.groups = G;
    a.group_cols = atm ? acc_cols + round32(S::KP) : acc_cols;
    a.a_col = atm ? acc_cols : 0u;
    uint32_t cols = 32;
    while (cols < (uint32_t)G * a.group_cols) cols *= 2;
    a.tmem_cols = cols;
    const size_t smem = stem_tc_smem_bytes(a, C, tma, G);
    // Overlapped tile loop when the accumulator row fits in registers.
    const bool ovl = tma && atm && a.ocp <= kStemOvlMaxOcp;
    auto kern = tma ? (atm ? (ovl ? stem_tf32_kernel<C, true, true, true> : stem_tf32_kernel<C, true, true, false>)
                           : stem_tf32_kernel<C, true, false, false>)
                    : (atm ? stem_tf32_kernel<C, false, true, false> : stem_tf32_kernel<C, false, false, false>);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // One CTA per SM (a kernel that uses TMEM is resident once per SM).
    const int ctas = (a.tiles + G - 1) / G;
    const int grid = ctas < info.sms ? ctas : info.sms;
    if (log_enabled())
        log_line("stem_tf32_kernel<C=%d> grid=%d block=%d smem=%zu groups=%d tiles=%d operand=%s io=%s%s", C, grid,
                 kStemPxThreads * G, smem, G, a.tiles, atm ? "tmem" : "smem", tma ? "tma" : "plain",
                 ovl ? " overlapped" : "");
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kStemPxThreads * G), smem, s, tmX, tmY, a);
}
