// fp32 convolution with a short reduction (C * 3 * 3 <= 32 taps: image
// stems) on the tcgen05 tensor cores, each fp32 product carried by three
// TF32 products.
//
// The operation is the output-stationary sum of lpnh.cn/news/2745477 section
// 2.2 (zero padding, bias, ReLU fused into the write-back as in section 4.4),
// cast as a GEMM per 128-pixel tile: D[pixel][oc] = sum_k A[pixel][k] B[oc][k]
// with k = (c, ky, kx), K = C * 9 padded to 32 (one 128-byte row per pixel).
// Every fp32 value v is split as v = hi + lo with hi = v with its 13 low
// mantissa bits cleared (exactly representable in TF32) and lo = v - hi
// (exact in fp32; the MMA reads its top 19 bits). The tile accumulates
// x_hi*w_lo + x_lo*w_hi + x_hi*w_hi in fp32 in TMEM; the dropped x_lo*w_lo
// and the TF32 reading of lo leave a relative error near 2^-20 per product,
// far inside the fp32 parity tolerance (rel. L2 1e-5). This split-product
// scheme is the usual way to run fp32 GEMMs on TF32 units.
//
// On the CUDA cores this layer costs as much FP32 FMA time as HBM time, and
// the packed FMA needs a register move per input value; on the tensor cores
// the arithmetic is a few hundred cycles per tile and the kernel is left
// with its memory traffic: x read once (L1 absorbs the 2.25x tap overlap at
// stride 2) and y written once with warp-coalesced 128-byte stores.
//
// GEMM orientation: M = output channels (rows of the weight operand, padded
// with zero rows to 128), N = 256 pixels, K = 32. A tcgen05.mma costs the
// issuing thread tens of cycles whatever its size, so the tile is shaped for
// N = 256 (128 cycles of tensor work per instruction) rather than M = pixels
// with N = 32 output channels (16 cycles of work, issue-bound); the zero
// weight rows are the price.
//
// One persistent CTA per SM (kernels that use TMEM run one CTA per SM), 8
// warps. A tile = 256 pixels = 8 groups of 32 consecutive output pixels of
// one row, taken round-robin over the CTAs; thread i owns pixel i. Per tile:
// each thread splits its pixel's taps and writes row i of the hi and lo
// pixel operands (128-byte swizzle, two buffers); one thread issues the 12
// MMAs (3 products x 4 K-steps of 8) into one of two TMEM accumulators
// (256 columns each) and commits; the next tile's tap loads go out; then the
// previous tile's epilogue: warp w reads output channels 32*(w%4) .. (its
// TMEM lane quadrant) for 4 of the 8 pixel groups, adds the bias, applies
// ReLU, writes each 32-channel x 32-pixel block to a staging tile (128-byte
// swizzle) and issues a TMA tensor store (bulk, clipped at the output's
// edges). The 8 staging tiles are shared out among the warps that hold real
// channels, so a warp cycles through up to 4 of them without waiting for
// its previous store. The weight operand is split once per CTA.

constexpr int kStemTcPx = 256;               // pixels per tile (MMA N)
constexpr int kStemTcK = 32;                 // padded reduction (tf32 per 128-byte row)
constexpr int kStemTcM = 128;                // MMA M: output channels padded to 128
constexpr int kStemTcThreads = 256;
constexpr int kStemMaxOC = 128;

struct StemTcArgs {
    const float *x, *w, *b;
    float *y;
    int H, W, OC, OH, OW, pad, stride;
    int groups_w;              // 32-pixel groups per output row
    long long groups;          // N * OH * groups_w
    long long tiles;           // ceil(groups / 8)
    uint32_t idesc, tmem_cols;
    int relu;
    int tma_store;             // output rows 16-byte aligned: TMA tensor stores
    long long wait_limit_cycles;
};

__device__ __forceinline__ void tf32_split(float v, float &hi, float &lo) {
    hi = __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
    lo = v - hi;
}

// Row `r` of the hi and lo K-major 128-byte-swizzle tiles from 32 fp32
// values (8 chunks of 4 floats, chunk j at (j ^ (r & 7)) * 16).
__device__ __forceinline__ void store_split_row(uint32_t hi_tile, uint32_t lo_tile, int r,
                                                const float (&v)[kStemTcK]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) tf32_split(v[4 * j + e], h[e], l[e]);
        const uint32_t off = (uint32_t)r * 128u + (uint32_t)((j ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(hi_tile + off), "f"(h[0]), "f"(h[1]),
                     "f"(h[2]), "f"(h[3])
                     : "memory");
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(lo_tile + off), "f"(l[0]), "f"(l[1]),
                     "f"(l[2]), "f"(l[3])
                     : "memory");
    }
}

struct StemPix {
    int n, oh, ow0, ow;
    bool group_ok, valid;
};
// Pixel `lane` of group `grp` (0..7) of tile `tile`.
__device__ __forceinline__ StemPix stem_pixel(const StemTcArgs &a, long long tile, int grp, int lane) {
    StemPix p{0, 0, 0, 0, false, false};
    const long long g = tile * 8 + grp;
    if (tile < a.tiles && g < a.groups) {
        const int gw = (int)(g % a.groups_w);
        const long long t = g / a.groups_w;
        p.oh = (int)(t % a.OH);
        p.n = (int)(t / a.OH);
        p.ow0 = gw * 32;
        p.ow = p.ow0 + lane;
        p.group_ok = true;
        p.valid = p.ow < a.OW;
    }
    return p;
}

// The pixel's C*9 taps (zero outside the input and beyond C*9).
template <int C>
__device__ __forceinline__ void stem_gather(const StemTcArgs &a, const StemPix &p, float (&v)[kStemTcK]) {
    const long long HW = (long long)a.H * a.W;
    const float *xn = a.x + (long long)p.n * C * HW;
    const int iy0 = p.oh * a.stride - a.pad, ix0 = p.ow * a.stride - a.pad;
#pragma unroll
    for (int c = 0; c < C; ++c)
#pragma unroll
        for (int ky = 0; ky < 3; ++ky) {
            const int iy = iy0 + ky;
            const bool row_ok = p.valid && (unsigned)iy < (unsigned)a.H;
            const float *xr = xn + c * HW + (long long)iy * a.W;
#pragma unroll
            for (int kx = 0; kx < 3; ++kx) {
                const int ix = ix0 + kx;
                v[(c * 3 + ky) * 3 + kx] = (row_ok && (unsigned)ix < (unsigned)a.W) ? __ldg(xr + ix) : 0.0f;
            }
        }
#pragma unroll
    for (int q = C * 9; q < kStemTcK; ++q) v[q] = 0.0f;
}

template <int C>
__global__ void __launch_bounds__(kStemTcThreads, 1)
stem_tf32_kernel(const __grid_constant__ CUtensorMap tmY, const StemTcArgs a) {
    constexpr int KT = C * 9;                           // real taps
    static_assert(KT <= kStemTcK, "taps");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    // Weight operand hi / lo (128 rows each), pixel operand buffers 0 / 1
    // (hi 32 KB + lo 32 KB each), per-warp 4 KB output staging, bias, barriers.
    const uint32_t sWh = base, sWl = base + 16384u;
    const uint32_t sP = base + 32768u;
    const uint32_t sY = sP + 2u * 65536u;
    const uint32_t sBar = sY + 4096u * (kStemTcThreads / 32);
    const uint32_t slot_addr = sBar + 16u;
    float *sBias = reinterpret_cast<float *>(smem_raw + (slot_addr + 16u - raw));
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem_raw + (slot_addr - raw));

    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    if (tid == 0) {
        mbar_init(sBar, 1);
        mbar_init(sBar + 8u, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(slot_addr, a.tmem_cols);
        tmem_relinquish();
    }
    const long long tstep = gridDim.x;
    long long tile = blockIdx.x;

    // The first tile's tap loads go out before the weight operand is built.
    float xv[kStemTcK];
    stem_gather<C>(a, stem_pixel(a, tile, warp, lane), xv);
    for (int o = tid; o < kStemTcM; o += kStemTcThreads) {
        if (o < kStemMaxOC) sBias[o] = (a.b && o < a.OC) ? __ldg(a.b + o) : 0.0f;
        float wv[kStemTcK];
#pragma unroll
        for (int q = 0; q < kStemTcK; ++q)
            wv[q] = (o < a.OC && q < KT) ? __ldg(a.w + (long long)o * KT + q) : 0.0f;
        store_split_row(sWh, sWl, o, wv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int q4 = warp & 3;                     // TMEM lane quadrant: channels 32*q4 ..
    const int gh = warp >> 2;                    // pixel groups 4*gh .. 4*gh+3 in the epilogue
    const bool epi_warp = 32 * q4 < a.OC;
    // Staging tiles: epilogue warp e = gh * nq + q4 owns tiles [e*nbuf, e*nbuf + nbuf).
    const int nq = (a.OC + 31) / 32, nepi = 2 * nq;
    const int nbuf = nepi <= 2 ? 4 : (nepi <= 4 ? 2 : 1);
    const uint32_t ys0 = sY + 4096u * (uint32_t)((gh * nq + q4) * nbuf);
    int slot = 0;

    long long prev = -1;                         // tile whose epilogue is pending
    int i = 0;
    for (;; ++i) {
        const bool have = tile < a.tiles;
        const int bsel = i & 1;
        if (have) {
            // Pixel operands of this tile; buffer bsel was last read by the
            // MMAs of tile i-2, which every thread saw complete (iteration i-1).
            const uint32_t ph = sP + 65536u * bsel, pl = ph + 32768u;
            store_split_row(ph, pl, tid, xv);
            fence_proxy_async_shared();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (tid == 0) {
                const uint64_t wh = sw128_kmajor_desc(sWh), wl = sw128_kmajor_desc(sWl);
                const uint64_t xh = sw128_kmajor_desc(ph), xl = sw128_kmajor_desc(pl);
                const uint32_t d = tmem + (uint32_t)(bsel * kStemTcPx);
                // K-steps of 8 tf32 = 32 bytes = descriptor start + 2. Small
                // cross terms first, the hi x hi term last.
#pragma unroll
                for (int kk = 0; kk < kStemTcK / 8; ++kk) tc_mma_tf32(d, wh + 2u * kk, xl + 2u * kk, a.idesc, kk);
#pragma unroll
                for (int kk = 0; kk < kStemTcK / 8; ++kk) tc_mma_tf32(d, wl + 2u * kk, xh + 2u * kk, a.idesc, 1);
#pragma unroll
                for (int kk = 0; kk < kStemTcK / 8; ++kk) tc_mma_tf32(d, wh + 2u * kk, xh + 2u * kk, a.idesc, 1);
                tc_commit(sBar + 8u * bsel);
            }
            // The next tile's taps load while the tensor core works.
            if (tile + tstep < a.tiles) stem_gather<C>(a, stem_pixel(a, tile + tstep, warp, lane), xv);
        }
        if (prev >= 0) {
            // Epilogue of tile `prev` (buffer (i-1)&1): every warp sees its
            // MMAs complete (which also frees that pixel buffer).
            const int pb = (i - 1) & 1;
            int ok = 1;
            if (lane == 0) ok = wait_bounded(sBar + 8u * pb, (uint32_t)(((i - 1) >> 1) & 1), a.wait_limit_cycles, nullptr);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok && lane == 0) atomicOr(&g_device_error, 1u);
            tc_fence_after();
            if (epi_warp) {
                const int oc = 32 * q4 + lane;
                const float bias = sBias[oc];
#pragma unroll 1
                for (int gg = 0; gg < 4; ++gg) {
                    const int grp = 4 * gh + gg;
                    const StemPix p = stem_pixel(a, prev, grp, 0);
                    if (!p.group_ok) continue;
                    uint32_t v[32];
                    tmem_ld32(tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(pb * kStemTcPx + grp * 32), v);
                    tmem_ld_wait();
                    if (a.tma_store) {
                        const uint32_t ys = ys0 + 4096u * (uint32_t)slot;
                        if (++slot == nbuf) slot = 0;
                        // The store that last used this staging tile has read it.
                        if (lane == 0) {
                            if (nbuf == 4) bulk_wait_read<3>();
                            else if (nbuf == 2) bulk_wait_read<1>();
                            else bulk_wait_read<0>();
                        }
                        __syncwarp();
                        // Row `lane` (= channel) of a [32 ch][32 px] block, 128-byte swizzle.
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float r[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                r[e] = epilogue(__uint_as_float(v[4 * j + e]), bias, a.relu);
                            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(
                                             ys + (uint32_t)lane * 128u + (uint32_t)((j ^ (lane & 7)) << 4)),
                                         "f"(r[0]), "f"(r[1]), "f"(r[2]), "f"(r[3])
                                         : "memory");
                        }
                        fence_proxy_async_shared();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_4d(&tmY, ys, p.ow0, p.oh, 32 * q4, p.n);
                            bulk_commit_group();
                        }
                    } else if (oc < a.OC) {
                        const long long plane = (long long)a.OH * a.OW;
                        float *yp = a.y + ((long long)p.n * a.OC + oc) * plane + (long long)p.oh * a.OW + p.ow0;
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (p.ow0 + e < a.OW) yp[e] = epilogue(__uint_as_float(v[e]), bias, a.relu);
                    }
                }
            }
            tc_fence_before();                   // accumulator pb is rewritten two tiles on
        }
        if (!have) break;
        prev = tile;
        tile += tstep;
    }
    if (lane == 0) bulk_wait_all();

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

size_t stem_tc_smem_bytes() {
    return 1024 + 32768 + 2 * 65536 + 4096 * (kStemTcThreads / 32) + 16 + 16 + 4 * kStemMaxOC;
}

template <int C>
cudaError_t launch_stem_tf32_c(const Problem &p, const float *x, const float *w, const float *b, float *y,
                               cudaStream_t s) {
    DevInfo info;
    cudaError_t e = dev_info(&info);
    if (e != cudaSuccess) return e;
    StemTcArgs a{};
    a.x = x; a.w = w; a.b = b; a.y = y;
    a.H = p.H; a.W = p.W; a.OC = p.OC; a.OH = p.OH; a.OW = p.OW; a.pad = p.pad; a.stride = p.stride;
    a.groups_w = (p.OW + 31) / 32;
    a.groups = (long long)p.N * p.OH * a.groups_w;
    a.tiles = (a.groups + 7) / 8;
    a.idesc = make_idesc_tf32(kStemTcM, kStemTcPx);
    a.tmem_cols = 512;                           // two 256-column accumulators
    a.relu = p.act == GBCONV_ACT_RELU;
    const double cyc = (double)wait_limit_ns() * (double)info.clock_khz * 1e-6;
    a.wait_limit_cycles = cyc > 9.0e18 ? (long long)9e18 : (long long)cyc;

    alignas(64) CUtensorMap tmY;
    std::memset(&tmY, 0, sizeof(tmY));
    a.tma_store = (p.OW % 4 == 0) && ((uintptr_t)y % 16 == 0);
    if (a.tma_store) {
        PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
        // y as {OW, OH, OC, N}; a box is 32 pixels of one row x 32 channels,
        // staged with the 128-byte swizzle.
        const cuuint64_t dims[4] = {(cuuint64_t)p.OW, (cuuint64_t)p.OH, (cuuint64_t)p.OC, (cuuint64_t)p.N};
        const cuuint64_t row = (cuuint64_t)p.OW * 4;
        const cuuint64_t strides[3] = {row, row * p.OH, row * p.OH * p.OC};
        const cuuint32_t box[4] = {32, 1, 32, 1};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        if (!encode || encode(&tmY, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, y, dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_NONE,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            a.tma_store = 0;
    }
    const size_t smem = stem_tc_smem_bytes();
    auto kern = stem_tf32_kernel<C>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // One persistent CTA per SM.
    const long long grid = a.tiles < info.sms ? a.tiles : info.sms;
    kern<<<(unsigned)grid, kStemTcThreads, smem, s>>>(tmY, a);
    return cudaGetLastError();
}
