/*
 * A plain C caller of the gbconv C ABI (include/gbconv.h): no Python, no
 * torch. Device memory comes from cudaMalloc, the stream is the default
 * stream, and every result is compared with the fp64 test oracle
 * (oracle/conv_ref.c, liboracle.so), which computes the plain definition of
 * the convolution (lpnh.cn/news/2745477, section 2.2).
 *
 * Cases (AUTO kernel choice, OIHW weights packed inside the call):
 *   1. fp32 image stem, 3 -> 32 channels, 3x3, stride 2, ReLU
 *   2. fp32 wide layer, 40 -> 72 channels, 3x3, stride 1 (three TF32 products)
 *   3. bf16 conv3d, 24 -> 16 channels, 3x3x3, causal frames
 * Tolerances: fp32 relative L2 <= 1e-5 and max abs <= 1e-4; bf16 NRMSE
 * <= 2.5e-3 against the unrounded result.
 *
 * Without a supported GPU it checks the validation path instead: a valid
 * call returns GBCONV_ERR_UNSUPPORTED_DEVICE and a malformed one its own code.
 * Exit status 0 on success.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "gbconv.h"

int oracle_conv2d(int N, int C, int H, int W, int OC, int k, int pad, int stride, int relu, const double *x,
                  const double *w, const double *b, double *y);
int oracle_conv3d(int N, int C, int D, int H, int W, int OC, int k, int pad, int pd0, int pd1, int stride,
                  int relu, const double *x, const double *w, const double *b, double *y);

static uint64_t g_state = 0x9E3779B97F4A7C15ull;
static double urand(void) { /* U[-1, 1) from a 64-bit LCG (Knuth's MMIX constants) */
    g_state = g_state * 6364136223846793005ull + 1442695040888963407ull;
    return (double)(g_state >> 11) * (1.0 / 9007199254740992.0) * 2.0 - 1.0;
}

/* float -> bfloat16 bits, round to nearest even; and back (exact). */
static uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
static double from_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

struct Case {
    const char *name;
    int ndim, N, C, D, H, W, OC, k, pad, stride, relu, dtype, causal;
};

static int check(cudaError_t e, const char *what) {
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

static int run_case(const struct Case *c) {
    const int kd = c->ndim == 3 ? c->k : 1;
    const int pd0 = c->ndim == 3 ? (c->causal ? c->k - 1 : c->pad) : 0;
    const int pd1 = c->ndim == 3 ? (c->causal ? 0 : c->pad) : 0;
    const int OD = c->ndim == 3 ? (c->D + pd0 + pd1 - c->k) / c->stride + 1 : 1;
    const int OH = (c->H + 2 * c->pad - c->k) / c->stride + 1;
    const int OW = (c->W + 2 * c->pad - c->k) / c->stride + 1;
    const size_t nx = (size_t)c->N * c->C * c->D * c->H * c->W;
    const size_t nw = (size_t)c->OC * c->C * kd * c->k * c->k;
    const size_t ny = (size_t)c->N * c->OC * OD * OH * OW;
    const size_t elt = c->dtype == GBCONV_F32 ? 4 : 2;

    double *xd = malloc(nx * sizeof(double)), *wd = malloc(nw * sizeof(double));
    double *bd = malloc((size_t)c->OC * sizeof(double)), *yref = malloc(ny * sizeof(double));
    void *xh = malloc(nx * elt), *wh = malloc(nw * elt), *yh = malloc(ny * elt);
    float *bh = malloc((size_t)c->OC * sizeof(float));
    const double wscale = sqrt(2.0 / (double)(c->C * kd * c->k * c->k));
    for (size_t i = 0; i < nx + nw; ++i) {
        const int is_x = i < nx;
        const float f = (float)(urand() * (is_x ? 1.0 : wscale));
        double v;
        if (c->dtype == GBCONV_F32) {
            v = f;
            ((float *)(is_x ? xh : wh))[is_x ? i : i - nx] = f;
        } else {
            const uint16_t h = to_bf16(f);
            v = from_bf16(h);
            ((uint16_t *)(is_x ? xh : wh))[is_x ? i : i - nx] = h;
        }
        if (is_x) xd[i] = v; else wd[i - nx] = v;
    }
    for (int o = 0; o < c->OC; ++o) {
        bh[o] = (float)(urand() * 0.1);
        bd[o] = bh[o];
    }

    gbconv_desc d;
    memset(&d, 0, sizeof d);
    d.N = c->N; d.C = c->C; d.D = c->D; d.H = c->H; d.W = c->W;
    d.OC = c->OC; d.k = c->k; d.pad = c->pad; d.stride = c->stride;
    d.dtype = c->dtype; d.act = c->relu ? GBCONV_ACT_RELU : GBCONV_ACT_NONE;
    d.w_layout = GBCONV_W_OIHW; d.algo = GBCONV_ALGO_AUTO;
    d.flags = c->causal ? GBCONV_TPAD_CAUSAL : 0;
    size_t ws = 0;
    int algo = 0, fail = 0;
    if (gbconv_workspace_size(&d, c->ndim, &ws) != GBCONV_OK || gbconv_select_algo(&d, c->ndim, &algo) != GBCONV_OK) {
        fprintf(stderr, "%s: descriptor rejected\n", c->name);
        return 1;
    }
    void *xg = NULL, *wg = NULL, *yg = NULL, *wsg = NULL;
    float *bg = NULL;
    fail |= check(cudaMalloc(&xg, nx * elt), "cudaMalloc x");
    fail |= check(cudaMalloc(&wg, nw * elt), "cudaMalloc w");
    fail |= check(cudaMalloc((void **)&bg, (size_t)c->OC * 4), "cudaMalloc b");
    fail |= check(cudaMalloc(&yg, ny * elt), "cudaMalloc y");
    if (ws) fail |= check(cudaMalloc(&wsg, ws), "cudaMalloc workspace");
    if (fail) return 1;
    d.workspace = wsg;
    d.workspace_bytes = ws;
    fail |= check(cudaMemcpy(xg, xh, nx * elt, cudaMemcpyHostToDevice), "copy x");
    fail |= check(cudaMemcpy(wg, wh, nw * elt, cudaMemcpyHostToDevice), "copy w");
    fail |= check(cudaMemcpy(bg, bh, (size_t)c->OC * 4, cudaMemcpyHostToDevice), "copy b");
    const gbconv_status st = c->ndim == 3 ? gbconv_conv3d_fwd(&d, xg, wg, bg, yg, 0)
                                          : gbconv_conv2d_fwd(&d, xg, wg, bg, yg, 0);
    if (st != GBCONV_OK) {
        fprintf(stderr, "%s: %s\n", c->name, gbconv_status_string(st));
        return 1;
    }
    if (gbconv_check_device_error(0) != GBCONV_OK) {
        fprintf(stderr, "%s: device error\n", c->name);
        return 1;
    }
    fail |= check(cudaMemcpy(yh, yg, ny * elt, cudaMemcpyDeviceToHost), "copy y");
    cudaFree(xg); cudaFree(wg); cudaFree(bg); cudaFree(yg);
    if (wsg) cudaFree(wsg);
    if (fail) return 1;

    if (c->ndim == 3)
        oracle_conv3d(c->N, c->C, c->D, c->H, c->W, c->OC, c->k, c->pad, pd0, pd1, c->stride, c->relu, xd, wd,
                      bd, yref);
    else
        oracle_conv2d(c->N, c->C, c->H, c->W, c->OC, c->k, c->pad, c->stride, c->relu, xd, wd, bd, yref);
    double e2 = 0.0, r2 = 0.0, emax = 0.0;
    for (size_t i = 0; i < ny; ++i) {
        const double y = c->dtype == GBCONV_F32 ? (double)((float *)yh)[i] : from_bf16(((uint16_t *)yh)[i]);
        const double e = fabs(y - yref[i]);
        e2 += e * e;
        r2 += yref[i] * yref[i];
        if (e > emax || e != e) emax = e;
    }
    const double rel = sqrt(e2 / (r2 > 0 ? r2 : 1e-300));
    const int ok = c->dtype == GBCONV_F32 ? (rel <= 1e-5 && emax <= 1e-4) : (rel <= 2.5e-3);
    printf("%-40s algo %-10s rel_l2 %.3e max_abs %.3e %s\n", c->name, gbconv_algo_name(algo), rel, emax,
           ok ? "ok" : "FAIL");
    free(xd); free(wd); free(bd); free(yref); free(xh); free(wh); free(yh); free(bh);
    return ok ? 0 : 1;
}

int main(void) {
    if (!gbconv_device_supported(0)) {
        /* Validation only: a valid call reaches the device check, a bad one
           is rejected before it (fake, aligned pointers; nothing is read). */
        gbconv_desc d;
        memset(&d, 0, sizeof d);
        d.N = 1; d.C = 3; d.D = 1; d.H = 32; d.W = 32; d.OC = 8; d.k = 3; d.pad = 1; d.stride = 1;
        void *p = (void *)(uintptr_t)(1u << 20);
        const gbconv_status a = gbconv_conv2d_fwd(&d, p, (char *)p + (1 << 16), NULL, (char *)p + (1 << 18), 0);
        d.act = 7;
        const gbconv_status b = gbconv_conv2d_fwd(&d, p, (char *)p + (1 << 16), NULL, (char *)p + (1 << 18), 0);
        printf("no supported GPU: valid call -> %s, bad activation -> %s\n", gbconv_status_string(a),
               gbconv_status_string(b));
        return (a == GBCONV_ERR_UNSUPPORTED_DEVICE && b == GBCONV_ERR_ACT) ? 0 : 1;
    }
    const struct Case cases[] = {
        {"conv2d f32 stem 1x3x96x128 -> 32, s2, relu", 2, 1, 3, 1, 96, 128, 32, 3, 1, 2, 1, GBCONV_F32, 0},
        {"conv2d f32 2x40x20x36 -> 72", 2, 2, 40, 1, 20, 36, 72, 3, 1, 1, 0, GBCONV_F32, 0},
        {"conv3d bf16 1x24x5x12x40 -> 16, causal", 3, 1, 24, 5, 12, 40, 16, 3, 1, 1, 1, GBCONV_BF16, 1},
    };
    int fails = 0;
    for (size_t i = 0; i < sizeof cases / sizeof cases[0]; ++i) fails += run_case(&cases[i]);
    return fails ? 1 : 0;
}
