/*
 * Oracle for the forward convolution: the plain definition, in fp64.
 *
 * TEST INFRASTRUCTURE ONLY. This file, and everything under oracle/, is the
 * slow, obviously correct CPU statement of what the GPU library computes. It
 * shares no code with the CUDA path. Only the tests, the smoke check and the
 * bench's CPU-baseline leg may load it; the library never does.
 *
 * What it computes (lpnh.cn/news/2745477, PP-OCR on Vulkan compute shaders,
 * section 2.2 "compute shader and SPIR-V"): every output element (ox, oy, oc)
 * sums input x weight over every input channel ic and every kernel tap
 * (ky, kx), where the input coordinate is derived from the output coordinate
 * as  iy = oy*stride - pad + ky,  ix = ox*stride - pad + kx;  taps that fall
 * outside the input are skipped (zero padding). The bias of the output channel
 * is added last. Input is channel-major (NCHW), weights are [oc][ic][ky][kx]
 * (OIHW). There is no kernel flip: this is cross-correlation.
 *
 * The same page, section 4.4 (tuning log), fuses ReLU into the write-back;
 * here ReLU is max(v, 0) applied after the bias when `relu` is non-zero.
 *
 * Convolution3D (git.erdda.com/Tencent/ncnn/discussions/7001, "SeedVR2 NCNN
 * Vulkan", section 3.2 "six custom layers") is the same sum with one more
 * spatial axis: time/depth, with the same kernel size and stride. The frame
 * axis has its own padding, pd0 zero frames before the first input frame and
 * pd1 after the last: pd0 = pd1 = pad for the symmetric case; the video VAE's
 * causal Convolution3D (same page, section 3.3) pads only the front, with
 * k-1 frames (an output frame then reads its own and earlier frames), and a
 * chunk that carries the previous chunk's frames is not padded at all.
 * The input frame of tap kd is  id = od*stride - pd0 + kd, and the number of
 * output frames is floor((D + pd0 + pd1 - k)/stride) + 1.
 *
 * Readings where the page is silent: a batch axis N is added in front (batch
 * stride C*H*W); the output size is floor((H + 2*pad - k)/stride) + 1 per
 * axis; every value is widened to double before use and the sum is kept in
 * double and never rounded. A NULL bias means no bias.
 *
 * Accumulation order: ic outermost, then the taps in row-major order, exactly
 * as the page's loop nest; one scalar double accumulator per output.
 */
#include <stddef.h>
#include <stdint.h>

static int64_t out_extent2(int64_t in, int k, int p0, int p1, int stride)
{
    int64_t span = in + (int64_t)p0 + p1 - k;
    if (span < 0)
        return 0;
    return span / stride + 1;
}

static int64_t out_extent(int64_t in, int k, int pad, int stride)
{
    int64_t span = in + 2 * (int64_t)pad - k;
    if (span < 0 || stride <= 0)
        return -1;
    return span / stride + 1;
}

/* One output element of the 2D convolution, y[n][oc][oy][ox]. */
static double conv2d_one(int C, int H, int W, int k, int pad, int stride,
                         int relu, const double *x, const double *w,
                         const double *b, int64_t n, int64_t oc, int64_t oy,
                         int64_t ox)
{
    double acc = 0.0;
    for (int64_t ic = 0; ic < C; ic++) {
        for (int64_t ky = 0; ky < k; ky++) {
            int64_t iy = oy * stride - pad + ky;
            if (iy < 0 || iy >= H)
                continue;
            for (int64_t kx = 0; kx < k; kx++) {
                int64_t ix = ox * stride - pad + kx;
                if (ix < 0 || ix >= W)
                    continue;
                double xv = x[((n * C + ic) * H + iy) * W + ix];
                double wv = w[((oc * C + ic) * k + ky) * k + kx];
                acc += xv * wv;
            }
        }
    }
    if (b)
        acc += b[oc];
    if (relu && acc < 0.0)
        acc = 0.0;
    return acc;
}

/* One output element of the 3D convolution, y[n][oc][od][oy][ox]. */
static double conv3d_one(int C, int D, int H, int W, int k, int pad, int pd0,
                         int stride, int relu, const double *x,
                         const double *w, const double *b, int64_t n,
                         int64_t oc, int64_t od, int64_t oy, int64_t ox)
{
    double acc = 0.0;
    for (int64_t ic = 0; ic < C; ic++) {
        for (int64_t kd = 0; kd < k; kd++) {
            int64_t id = od * stride - pd0 + kd;
            if (id < 0 || id >= D)
                continue;
            for (int64_t ky = 0; ky < k; ky++) {
                int64_t iy = oy * stride - pad + ky;
                if (iy < 0 || iy >= H)
                    continue;
                for (int64_t kx = 0; kx < k; kx++) {
                    int64_t ix = ox * stride - pad + kx;
                    if (ix < 0 || ix >= W)
                        continue;
                    double xv = x[(((n * C + ic) * D + id) * H + iy) * W + ix];
                    double wv = w[(((oc * C + ic) * k + kd) * k + ky) * k + kx];
                    acc += xv * wv;
                }
            }
        }
    }
    if (b)
        acc += b[oc];
    if (relu && acc < 0.0)
        acc = 0.0;
    return acc;
}

/*
 * Full 2D convolution. x: [N][C][H][W], w: [OC][C][k][k], b: [OC] or NULL,
 * y: [N][OC][OH][OW], all double. Returns 0, or -1 on an invalid shape.
 */
int oracle_conv2d(int N, int C, int H, int W, int OC, int k, int pad,
                  int stride, int relu, const double *x, const double *w,
                  const double *b, double *y)
{
    int64_t OH = out_extent(H, k, pad, stride);
    int64_t OW = out_extent(W, k, pad, stride);
    if (N <= 0 || C <= 0 || OC <= 0 || k <= 0 || pad < 0 || OH <= 0 ||
        OW <= 0)
        return -1;
    int64_t rows = (int64_t)N * OC * OH;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        int64_t oy = r % OH;
        int64_t oc = (r / OH) % OC;
        int64_t n = r / (OH * OC);
        for (int64_t ox = 0; ox < OW; ox++)
            y[r * OW + ox] = conv2d_one(C, H, W, k, pad, stride, relu, x, w,
                                        b, n, oc, oy, ox);
    }
    return 0;
}

/*
 * Full 3D convolution. x: [N][C][D][H][W], w: [OC][C][k][k][k],
 * y: [N][OC][OD][OH][OW]. pd0 / pd1: zero frames before / after the input
 * frames. Returns 0, or -1 on an invalid shape.
 */
int oracle_conv3d(int N, int C, int D, int H, int W, int OC, int k, int pad,
                  int pd0, int pd1, int stride, int relu, const double *x,
                  const double *w, const double *b, double *y)
{
    int64_t OD = out_extent2(D, k, pd0, pd1, stride);
    int64_t OH = out_extent(H, k, pad, stride);
    int64_t OW = out_extent(W, k, pad, stride);
    if (N <= 0 || C <= 0 || OC <= 0 || k <= 0 || pad < 0 || pd0 < 0 ||
        pd1 < 0 || OD <= 0 || OH <= 0 || OW <= 0)
        return -1;
    int64_t rows = (int64_t)N * OC * OD * OH;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        int64_t oy = r % OH;
        int64_t od = (r / OH) % OD;
        int64_t oc = (r / (OH * OD)) % OC;
        int64_t n = r / (OH * OD * OC);
        for (int64_t ox = 0; ox < OW; ox++)
            y[r * OW + ox] = conv3d_one(C, D, H, W, k, pad, pd0, stride, relu,
                                        x, w, b, n, oc, od, oy, ox);
    }
    return 0;
}

/*
 * Selected outputs of the 2D convolution: out[i] = y.flat[idx[i]] where y is
 * the [N][OC][OH][OW] result of oracle_conv2d. Returns 0, -1 on an invalid
 * shape, -2 on an index outside y.
 */
int oracle_conv2d_at(int N, int C, int H, int W, int OC, int k, int pad,
                     int stride, int relu, const double *x, const double *w,
                     const double *b, const int64_t *idx, int64_t count,
                     double *out)
{
    int64_t OH = out_extent(H, k, pad, stride);
    int64_t OW = out_extent(W, k, pad, stride);
    if (N <= 0 || C <= 0 || OC <= 0 || k <= 0 || pad < 0 || OH <= 0 ||
        OW <= 0)
        return -1;
    int64_t total = (int64_t)N * OC * OH * OW;
    for (int64_t i = 0; i < count; i++)
        if (idx[i] < 0 || idx[i] >= total)
            return -2;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; i++) {
        int64_t f = idx[i];
        int64_t ox = f % OW;
        int64_t oy = (f / OW) % OH;
        int64_t oc = (f / (OW * OH)) % OC;
        int64_t n = f / (OW * OH * OC);
        out[i] = conv2d_one(C, H, W, k, pad, stride, relu, x, w, b, n, oc, oy,
                            ox);
    }
    return 0;
}

/* Selected outputs of the 3D convolution (flat indices into NCDHW y). */
int oracle_conv3d_at(int N, int C, int D, int H, int W, int OC, int k, int pad,
                     int pd0, int pd1, int stride, int relu, const double *x,
                     const double *w, const double *b, const int64_t *idx,
                     int64_t count, double *out)
{
    int64_t OD = out_extent2(D, k, pd0, pd1, stride);
    int64_t OH = out_extent(H, k, pad, stride);
    int64_t OW = out_extent(W, k, pad, stride);
    if (N <= 0 || C <= 0 || OC <= 0 || k <= 0 || pad < 0 || pd0 < 0 ||
        pd1 < 0 || OD <= 0 || OH <= 0 || OW <= 0)
        return -1;
    int64_t total = (int64_t)N * OC * OD * OH * OW;
    for (int64_t i = 0; i < count; i++)
        if (idx[i] < 0 || idx[i] >= total)
            return -2;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; i++) {
        int64_t f = idx[i];
        int64_t ox = f % OW;
        int64_t oy = (f / OW) % OH;
        int64_t od = (f / (OW * OH)) % OD;
        int64_t oc = (f / (OW * OH * OD)) % OC;
        int64_t n = f / (OW * OH * OD * OC);
        out[i] = conv3d_one(C, D, H, W, k, pad, pd0, stride, relu, x, w, b, n,
                            oc, od, oy, ox);
    }
    return 0;
}

/* Number of OpenMP threads the oracle runs on (1 without OpenMP). */
int oracle_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
